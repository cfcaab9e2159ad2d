"""Host-side logic of bench.py: the algorithmic byte and flop counts of the
roofline against their closed forms, the shortened-workload option, the
reference arm on non-zero ranks, and the multi-rank path (barrier, the
slowest rank's time, the whole-job rate) as two gloo ranks on the CPU."""
import argparse
import os
import socket

import torch.multiprocessing as mp

import bench
import workloads as wl


def test_algorithmic_counts_of_the_five_workloads():
    # bytes: read q, k, v and write out once, (2 D + 2 Dv) elements per token-head
    assert bench.alg_bytes(wl.LONG_65536) == 16 * 65536 * (2 * 128 + 2 * 128) * 2
    assert bench.alg_bytes(wl.TINY_F32) == 64 * (2 * 16 + 2 * 16) * 4
    # flops per token-head: 4 P Dv (S update, readout) + 3 P (z, denominator) + Dv (divide)
    assert bench.alg_flops(wl.LONG_65536) == 16 * 65536 * (4 * 128 * 128 + 3 * 128 + 128)
    # random features add the projection and the exponent arguments: 4 m D + 2 D + 2 m
    p = wl.PRF_16384
    per = 4 * 256 * 64 + 3 * 256 + 64 + 4 * 256 * 64 + 2 * 64 + 2 * 256
    assert bench.alg_flops(p) == 2 * 8 * 16384 * per
    # the long workload is HBM-bound against any B300-class ridge point
    assert bench.alg_flops(wl.LONG_65536) / bench.alg_bytes(wl.LONG_65536) < 100


def test_seq_len_option_shortens_the_named_workload():
    a = argparse.Namespace(workload=wl.LONG_65536.name, seq_len=16384)
    w = bench.workload_of(a)
    assert (w.B, w.H, w.N, w.D, w.Dv) == (1, 16, 16384, 128, 128)
    assert w.name == "causal_B1_H16_N16384_D128_bf16"
    a.seq_len = 0
    assert bench.workload_of(a) == wl.LONG_65536


def test_reference_arm_is_silent_on_other_ranks(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    a = argparse.Namespace(workload=wl.LONG_65536.name, seq_len=0, steps=1, warmup=3)
    assert bench.run_reference(a) is None
    assert capsys.readouterr().out == ""


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench as b

    w, r, _ = b.dist_setup()
    b.barrier(w)
    t_ms = 10.0 + 5.0 * r                # rank 1 is the slower one
    slowest = b.max_over_ranks(t_ms, w)
    q.put((r, w, slowest, b.job_rate(1000.0, 4, w, slowest)))
    b.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_rate():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    for _, ws, slowest, rate in got:
        assert ws == 2
        assert slowest == 15.0
        # both ranks' units over the slowest rank's time
        assert abs(rate - 1000.0 * 4 * 2 / 0.015) < 1e-6 * rate


def test_oracle_sample_gives_every_thread_a_head():
    for w in wl.WORKLOADS.values():
        for cores in (1, 8, 16, 64):
            h, n = bench.oracle_sample(w, 2.0, cores)
            assert min(w.B * w.H, cores) <= h <= w.B * w.H
            assert 1 <= n <= w.N
    # a large budget takes the whole workload
    assert bench.oracle_sample(wl.IMAGE_3072, 1e9, 8) == (32, 3072)


def test_reference_arm_times_whole_steps_of_the_tiny_workload(monkeypatch, capsys):
    import json

    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    a = argparse.Namespace(workload=wl.TINY_F32.name, seq_len=0, steps=4, warmup=3)
    bench.run_reference(a)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"]["step"] == "one oracle call over the whole workload"
    # value and ms_per_step describe the same timed steps
    tokens = wl.TINY_F32.B * wl.TINY_F32.N
    assert abs(line["value"] * line["ms_per_step"] / 1e3 - tokens) < 1e-6 * tokens
    assert line["cpu_baseline"]["cores"] == 1   # one head: one thread has work


def test_rpe_sample_bias_rows_match_the_head_and_offsets():
    import numpy as np
    import torch

    w = wl.small(B=2, H=3, N=10, D=4, Dv=4)
    b = torch.arange(3 * 19, dtype=torch.float32).reshape(3, 19)
    got = bench.np64_bias(b, 4, 6, w)   # heads 0..3 -> rows 0, 1, 2, 0; offsets |t| < 6
    assert got.shape == (4, 11)
    assert np.array_equal(got[3], b[0, 4:15].double().numpy())
    # offset 0 of the sample sits in its middle, as in the full row
    assert got[1, 5] == b[1, 9]
