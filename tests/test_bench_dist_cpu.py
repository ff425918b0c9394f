"""Multi-rank host logic of bench.py on CPU: two gloo ranks.  The reported
step time is the max over ranks; the heads are partitioned over the ranks
(weak: rank r owns head block r of an N*H-head job; strong: the workload's
heads are split), the ranges tile the heads exactly, and the ranks' unmasked
FLOPs add up to the job's."""

import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (world, rank, rank)
    my_ms = [3.0, 5.5][rank]
    got = bench.reduce_max(my_ms, world)
    bench.barrier(world)
    results[rank] = got
    dist.destroy_process_group()


def _partition_worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench
    from block_sparse_masked_build_gb300 import workloads as wl

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    out = {}
    for name in ("cfg2_causal_s2048_d128", "cfg3_packed_s8192_d128"):
        w = wl.WORKLOADS[name]
        seg = wl.make_segment_ids(w)
        for strong in (False, True):
            wr, h0, h1, Hg = bench.rank_workload(w, world, rank, strong)
            f = bench.workload_flops(wr, seg) if wr.H > 0 else 0
            t = torch.tensor([f], dtype=torch.float64)
            dist.all_reduce(t)  # sum over ranks
            out[(name, strong)] = (h0, h1, Hg, wr.H, wr.seed, int(t.item()))
    results[rank] = out
    dist.destroy_process_group()


def test_two_rank_head_partition():
    sys.path.insert(0, ROOT)
    import bench
    from block_sparse_masked_build_gb300 import workloads as wl

    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    procs = [ctx.Process(target=_partition_worker,
                         args=(r, world, port, results))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    res = dict(results)
    for name in ("cfg2_causal_s2048_d128", "cfg3_packed_s8192_d128"):
        w = wl.WORKLOADS[name]
        full = bench.workload_flops(w, wl.make_segment_ids(w))
        for strong in (False, True):
            ranges = sorted((res[r][(name, strong)][:2]) for r in range(world))
            Hg = res[0][(name, strong)][2]
            assert Hg == (w.H if strong else world * w.H)
            # the ranks' head ranges tile [0, Hg) with no gap or overlap
            assert ranges[0][0] == 0 and ranges[-1][1] == Hg
            assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
            # each rank holds exactly its heads
            for r in range(world):
                h0, h1, _, nh, seed, _ = res[r][(name, strong)]
                assert nh == h1 - h0
                if not strong:  # own draw per head block; block 0 = N=1
                    assert seed == bench.rank_seed(w, r)
                    assert (seed == w.seed) == (r == 0)
            total = res[0][(name, strong)][5]
            assert total == res[1][(name, strong)][5]
            assert total == (full if strong else world * full)


def test_head_partition_groups_and_uneven_sizes():
    sys.path.insert(0, ROOT)
    import bench

    for H, world, group in [(16, 3, 1), (12, 5, 2), (8, 8, 4), (3, 4, 1)]:
        spans = [bench.head_partition(H, world, r, group) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == H
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 == b0
        for h0, h1 in spans:
            assert h0 % group == 0 and h1 % group == 0 and h1 >= h0
        sizes = [h1 - h0 for h0, h1 in spans]
        assert max(sizes) - min(sizes) <= group


def test_two_rank_max_reduction():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, results))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(results) == {0: 5.5, 1: 5.5}


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max(1.25, 1) == 1.25
    a = bench.parse_args([])
    assert a.gpus == 1 and a.impl == "ours"
    assert a.workload == "cfg3_packed_s8192_d128"


def test_reference_arm_json_contract():
    # the oracle arm on CPU, on the small causal workload: one JSON line
    # with the contract's keys and a positive throughput
    sys.path.insert(0, ROOT)
    import json
    import bench
    from block_sparse_masked_build_gb300 import workloads as wl

    args = bench.parse_args(["--impl", "reference", "--steps", "2",
                             "--warmup", "1", "--workload",
                             "cfg1_causal_s256_d64"])
    line = bench.run_reference(args, wl.WORKLOADS[args.workload])
    json.dumps(line)
    for key in ("metric", "value", "unit", "impl", "steps", "warmup",
                "ms_per_step", "higher_is_better", "config", "cpu_baseline",
                "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["steps"] == 2 and line["warmup"] == 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["config"]["workload"] == "cfg1_causal_s256_d64"


def test_flop_counts_of_every_workload_are_positive():
    # the bench's FLOP denominators, including the band and arbitrary-mask
    # diagnostics, from the closed-form counter
    sys.path.insert(0, ROOT)
    import bench
    from block_sparse_masked_build_gb300 import workloads as wl

    for name, w in wl.WORKLOADS.items():
        if w.S > 8192:
            continue  # the long local-window count takes longer; pinned elsewhere
        f = bench.workload_flops(w, wl.make_segment_ids(w))
        assert f > 0, name


def test_recorded_traffic_lines_are_well_formed():
    # every TRAFFIC_JSON line of the ncu summaries names a bench workload and
    # a per-launch DRAM figure within a plausible multiple of that
    # workload's algorithmic bytes; the roofline takes a line only when its
    # source hash is the current forward sources' hash
    sys.path.insert(0, ROOT)
    import json
    import re
    import bench
    from block_sparse_masked_build_gb300 import workloads as wl

    prof = os.path.join(ROOT, "profiles")
    seen = 0
    for name in sorted(os.listdir(prof)):
        with open(os.path.join(prof, name)) as f:
            for line in f:
                m = re.match(r"\s*TRAFFIC_JSON:\s*(\{.*\})\s*$", line)
                if not m:
                    continue
                d = json.loads(m.group(1))
                assert set(d) == {"src", "workload", "dram_bytes_per_launch"}
                assert re.fullmatch(r"[0-9a-f]{16}", d["src"])
                w = wl.WORKLOADS[d["workload"]]
                algo = bench.algorithmic_bytes(w)
                assert 0.5 * algo < d["dram_bytes_per_launch"] < 5 * algo
                got = bench.recorded_traffic(d["workload"])
                if d["src"] == bench.fwd_source_hash():
                    assert got == float(d["dram_bytes_per_launch"])
                seen += 1
    assert seen >= 1
