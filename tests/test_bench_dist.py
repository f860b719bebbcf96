"""bench.py's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

Under torchrun each rank runs its own replica of the workload; the timing is the maximum over ranks, and the
reference arm runs on rank 0 alone.  These tests exercise that logic without a GPU.
"""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, _ = bench._dist()
    assert (ws, r) == (world, rank)
    bench._init_pg(ws, "gloo")
    bench.barrier(ws)
    got = bench.max_over_ranks(10.0 + rank, ws)
    # the reference arm runs on rank 0 only: other ranks return at once, before touching any workload
    rc = 0 if rank == 0 else bench.run_reference(type("A", (), {"workload": 1, "steps": 1, "warmup": 3})())
    import torch.distributed as dist
    dist.destroy_process_group()
    out.put((rank, got, rc))


def test_max_over_ranks_barrier_and_rank0_only_reference():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=5) for _ in range(world))
    assert [g for _, g, _ in res] == [11.0, 11.0]
    assert [rc for _, _, rc in res] == [0, 0]


def test_traffic_record_follows_the_code_not_the_comments():
    # a recorded ncu traffic figure stays valid through an edit of the comments and goes stale with the code
    sys.path.insert(0, ROOT)
    import bench
    src = "// header\n__global__ void k(float* p) {  /* note */\n    p[0] = 1.f;   // store\n}\n"
    assert bench._code_only(src) == bench._code_only(src.replace("// store", "// the store, reworded\n//"))
    assert bench._code_only(src) != bench._code_only(src.replace("1.f", "2.f"))
    assert "header" not in bench._code_only(src) and "note" not in bench._code_only(src)
    for kind in bench.TRAFFIC_SOURCES:
        assert len(bench.sources_sha256(kind)) == 64


def test_roofline_counts_of_the_headline_workloads():
    # the algorithmic bytes and flops the bench divides by time, against the figures worked out by hand:
    # prefill, the survey's count (o in bf16): 262,144 token-heads x (3 x 256 B bf16 q, k, v + 256 B o + 4 B g + 4 B
    # beta) plus 64 states of 64 KiB read and written, 278,921,216 B; with o counted as the fp32 the call writes,
    # 512 B of o per token-head; backward: per chunk-head of 16 rows, 3 C^2 d_k (Q K^T, K K^T, the dQ / dK pair
    # sums) + 8 C d_k d_v (Z, the state update, dDelta, the state gradient x 2, the three state products) +
    # 2.5 C^2 d_v (the two solves, P^T dO, dP and dA) multiply-adds over 16,384 chunk-heads
    sys.path.insert(0, ROOT)
    import bench
    from gated_delta_rule_gdn_gb300 import workloads as W
    assert bench._alg_bytes(W.config(1)) == 262_144 * 1032 + 64 * 2 * 65_536 == 278_921_216
    assert bench._alg_bytes(W.config(1), 4) == 262_144 * 1288 + 64 * 2 * 65_536 == 346_030_080
    # KDA: the per-channel gate adds 4 (d_k - 1) B per token-head; no initial state, so the state is written only
    assert bench._alg_bytes(W.config(3)) == 524_288 * (1032 + 4 * 127) + 64 * 65_536 == 811_597_824
    # head size 256: 131,072 token-heads x (3 x 512 B q, k, v + 512 B o + 8 B g, beta) plus 32 states of 256 KiB
    # read and written
    assert bench._alg_bytes(W.HEAD256) == 131_072 * 2056 + 32 * 2 * 262_144 == 286_261_248
    # the fp32 tiny case: 64 token-heads x (3 x 64 B + 64 B o + 8 B) plus one 1 KiB state, written only
    assert bench._alg_bytes(W.config(0), 4) == 64 * 264 + 1024 == 17_920
    macs = 3 * 16 * 16 * 128 + 8 * 16 * 128 * 128 + 5 * 16 * 16 * 128 // 2
    assert macs == 2_277_376
    assert bench._bwd_flops(W.config(1), 16) == 2 * macs * 16_384 == 74_625_056_768


def test_reference_arm_on_the_tiny_and_head256_workloads(capsys):
    # the reference arm samples up to four heads, so a one-head workload runs too; the head-256 workload maps to
    # its own shape
    sys.path.insert(0, ROOT)
    import json
    import bench
    assert bench.main(["--impl", "reference", "--workload", "0", "--steps", "1", "--warmup", "3"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["config"]["workload"] == "gdn_tiny_b1_t64_h1_d16_c16_f32"
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    w = bench._chunk_workload(8)
    assert (w.dk, w.dv, w.H, w.B, w.T) == (256, 256, 8, 4, 4096)
    assert bench._traffic_kind(w.name) == "chunk_gdn_d256"
    assert bench._traffic_kind(bench._chunk_workload(0).name) == "chunk_generic"
