"""The benchmark's multi-process path (replicas, no data-path collective), on CPU.

Under torchrun every rank runs its own decode batch on its own GPU; the only
collectives are the barrier around the timed region and the max over ranks of
the timed durations. Here two gloo ranks on 127.0.0.1 stand in for the GPUs:
each reports its own duration, both must see the largest, and the job's rate
counts every rank's tokens over that slowest time. Ranks other than 0 of the
reference arm exit without work or output.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, durations, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        dist.barrier()
        slowest = bench.max_over_ranks(durations[rank], dist, "cpu")
        out[rank] = (slowest, bench.job_rate(ws, 32, 10, slowest))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_with_two_gloo_ranks():
    world, port = 2, _free_port()
    durations = [0.5, 0.8]
    with mp.get_context("spawn").Manager() as m:  # no fork of this (threaded) process
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, durations, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    slowest, rate = res[0]
    assert slowest == 0.8
    assert rate == pytest.approx(world * 32 * 10 / 0.8)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, None, "cpu") == 1.25
    assert bench.job_rate(1, 32, 100, 2.0) == 1600.0


def test_reference_arm_other_ranks_exit_without_output():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_roofline_bound_follows_the_ridge_point():
    """Below the ridge (peak flops / peak bytes) the bound is HBM, above it the tensor pipe;
    the fraction is the achieved rate over that peak."""
    sys.path.insert(0, ROOT)
    import bench
    hbm, tf = 6775.6, 1946.8  # ridge ~287 flop/B
    one = bench.roofline_bound(flops=234e6 * 1000, nbytes=1e9, us=200.0, hbm_gbs=hbm, tflops=tf)
    assert one["bound"] == "hbm" and one["unit"] == "GB/s"
    assert one["achieved"] == pytest.approx(5000.0) and one["frac"] == pytest.approx(5000.0 / hbm)
    two = bench.roofline_bound(flops=468e9, nbytes=1e9, us=400.0, hbm_gbs=hbm, tflops=tf)
    assert two["bound"] == "tensor" and two["unit"] == "TFLOP/s"
    assert two["achieved"] == pytest.approx(1170.0) and two["frac"] == pytest.approx(1170.0 / tf)
    assert two["flop_per_byte"] == pytest.approx(468.0)


def test_decode_plus_combine_counts_the_merge_output():
    """The decode unit's bytes: the decode kernel's algorithmic bytes plus the merged u (bf16)
    and lse (fp32) the combine writes; at 32 x 4096, 155,721,856 + 32*128*(1024+4)."""
    import bench
    import mla_inputs as mi
    inp = mi.make_inputs(B=2, H=4, n_q=1, seq_lens=[5, 7], seed=1)
    dec_bytes, _ = bench.decode_alg(inp)
    line = bench.decode_combine_line(30.0, 5.0, dec_bytes, inp, hbm=1000.0)
    assert line["alg_bytes"] == dec_bytes + 2 * 4 * (512 * 2 + 4)
    assert abs(line["us"] - 35.0) < 1e-12
    assert abs(line["frac"] - line["alg_bytes"] / 35e-6 / 1e9 / 1000.0) < 1e-12
    assert 155_721_856 + 32 * 128 * 1028 == 159_932_544  # the 32 x 4096 decode unit
