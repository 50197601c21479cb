"""The FP8 (e4m3, per-channel scales) latent cache on the GPU (GPU only).

Parity is against the oracle run on the DEQUANTISED latents (oracle.absorbed_fp8_f64:
scale[d] * e4m3(code), then the exact fp64 absorbed loops), at the tolerances of every
parity test. The quantiser kernel is integer work and must give the generator's codes
bit for bit. A separate test bounds how far the FP8 path's results move from the bf16
path's: rounding to e4m3 (3 mantissa bits, nearest) leaves each latent within 2^-4 of
its value relative, uniformly spread, i.e. 2^-5 on average; u, a weighted mean of the
latents, inherits that relative size, so its mean relative change is bounded here by
2^-4 (Huny's Dev Blog section 6 item 4: FP8 with per-channel scales; ailab.paldyn.com
"MQA와 GQA": FP8 usually costs little quality).
"""
import numpy as np
import pytest

import mla_inputs as mi
import oracle
from tests.helpers import assert_close, dev_bf16_to_f64, dev_to_bits, device_inputs, errors

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    import mla_latent_kv_paged_gb300 as m
    m.build()
    return m


def fp8_device(inp, pg, mla):
    """Device tensors of the bf16 inputs plus the FP8 cache (quantised on the host by the
    generator) and its scales; returns (d, pg8, codes_logical)."""
    import torch
    d = device_inputs(inp, pg)
    pg8 = mi.make_paged_fp8(inp, pg)
    d["cache8"] = torch.from_numpy(pg8.cache).cuda()
    d["scales"] = torch.from_numpy(pg8.scales).cuda()
    codes = mi.quantize_fp8(np.concatenate([inp.c, inp.kr], axis=1), pg8.scales)
    return d, pg8, codes


def run_fp8(mla, inp, d, num_splits=None, planned=False):
    import torch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_abs = mla.absorb_q(d["q_nope"], d["q_rope"], d["w_uk"])
    B, max_pages = d["block_table"].shape
    if planned:
        ws, g = mla.decode_plan(d["seq_lens"], n_q=inp.n_q, H=inp.H, max_pages=max_pages,
                                num_pages=d["cache8"].shape[0], num_splits=num_splits, err_word=err)
        mla.decode_paged_fp8(q_abs, d["cache8"], d["scales"], d["block_table"], d["seq_lens"], n_q=inp.n_q,
                             num_splits=g, workspace=ws, err_word=err, planned=True)
    else:
        ws, g = mla.decode_paged_fp8(q_abs, d["cache8"], d["scales"], d["block_table"], d["seq_lens"],
                                     n_q=inp.n_q, num_splits=num_splits, err_word=err)
    u, lse = mla.combine(ws, B=inp.B, n_q=inp.n_q, H=inp.H, num_splits=g)
    out = mla.out_proj(u, d["w_uv"])
    torch.cuda.synchronize()
    return dict(u=u, lse=lse, out=out, err=int(err.item()))


def compare_fp8(inp, codes, scales, r):
    ref = oracle.absorbed_fp8_f64(inp, codes, scales)
    T, H = inp.B * inp.n_q, inp.H
    assert_close(dev_bf16_to_f64(r["u"]).reshape(T * H, 512), ref["u"], "u")
    assert_close(r["lse"].double().cpu().numpy().reshape(T * H), ref["lse"], "lse")
    assert_close(dev_bf16_to_f64(r["out"]).reshape(T * H, 128), ref["out"], "out")


def test_quantiser_kernel_matches_the_generator_bit_for_bit(mla):
    import torch
    rng = np.random.default_rng(21)
    n = 3000
    x = rng.standard_normal((n, 576)).astype(np.float32) * rng.choice([1e-3, 1.0, 30.0], size=(n, 1)).astype(np.float32)
    x[0, :8] = [0.0, -0.0, 1e-30, -1e-30, 447.9, -1000.0, 2.0 ** -9, 3.0 * 2.0 ** -11]
    bits = mi.f32_to_bf16(x)
    scales = rng.uniform(0.01, 2.0, size=576).astype(np.float32)
    ref = mi.quantize_fp8(bits, scales)
    got = mla.quantize_fp8(torch.from_numpy(bits.view(np.int16)).cuda(), torch.from_numpy(scales).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), ref)


def test_fp8_tiny_workload_all_rows(mla):
    inp = mi.workload_inputs(1)
    pg = mi.make_paged(inp, spare_pages=4)
    d, pg8, codes = fp8_device(inp, pg, mla)
    r = run_fp8(mla, inp, d)
    assert r["err"] == 0
    compare_fp8(inp, codes, pg8.scales, r)


@pytest.mark.parametrize("splits", [1, 3, 64])
def test_fp8_ragged_multitoken_all_rows(mla, splits):
    """Partial last pages (NaN-coded slack rows), a 2-token sequence, causal pairs, any split count."""
    inp = mi.make_inputs(B=5, H=128, n_q=2, seq_lens=[2, 64, 65, 300, 1000], seed=41)
    pg = mi.make_paged(inp, spare_pages=3)
    d, pg8, codes = fp8_device(inp, pg, mla)
    r = run_fp8(mla, inp, d, num_splits=splits)
    assert r["err"] == 0
    compare_fp8(inp, codes, pg8.scales, r)


@pytest.mark.parametrize("H", [16, 100])
def test_fp8_fewer_heads_planned(mla, H):
    inp = mi.make_inputs(B=3, H=H, n_q=1, seq_lens=[130, 64, 7], seed=43 + H)
    pg = mi.make_paged(inp)
    d, pg8, codes = fp8_device(inp, pg, mla)
    r = run_fp8(mla, inp, d, num_splits=4, planned=True)
    assert r["err"] == 0
    compare_fp8(inp, codes, pg8.scales, r)


def test_fp8_page_permutation_is_bit_exact(mla):
    inp = mi.make_inputs(B=4, H=128, n_q=1, seq_lens=[500, 64, 1, 257], seed=47)
    rs = []
    for perm, spare in [(1, 2), (2, 9)]:
        pg = mi.make_paged(inp, perm_seed=perm, spare_pages=spare)
        d, pg8, codes = fp8_device(inp, pg, mla)
        rs.append(run_fp8(mla, inp, d))
    for k in ("u", "out"):
        assert np.array_equal(dev_to_bits(rs[0][k]), dev_to_bits(rs[1][k])), k
    assert np.array_equal(rs[0]["lse"].cpu().numpy().view(np.uint32), rs[1]["lse"].cpu().numpy().view(np.uint32))


def test_fp8_rising_scores_all_rows(mla):
    """Large, rising scores (the lazy rescale and large exchanged partials) on the FP8 path."""
    base = mi.make_inputs(B=3, H=128, n_q=1, seq_lens=[700, 1500, 130], seed=92)
    inp = mi.with_rising_scores(base, col=40, kind="ramp")
    pg = mi.make_paged(inp, spare_pages=3)
    d, pg8, codes = fp8_device(inp, pg, mla)
    r = run_fp8(mla, inp, d, num_splits=4)
    assert r["err"] == 0
    compare_fp8(inp, codes, pg8.scales, r)


def test_fp8_full_size_workload_all_rows(mla):
    """32 x 4096 (the benchmark's FP8 side line) in its launch configuration, every row."""
    inp = mi.workload_inputs(2)
    pg = mi.make_paged(inp, spare_pages=mi.WORKLOADS[2].spare_pages)
    d, pg8, codes = fp8_device(inp, pg, mla)
    r = run_fp8(mla, inp, d)
    assert r["err"] == 0
    compare_fp8(inp, codes, pg8.scales, r)


def test_fp8_moves_results_within_the_e4m3_bound_of_the_bf16_path(mla):
    """The FP8 cache's results against the bf16 cache's on the same inputs (both on the GPU):
    mean relative change of u and out at most 2^-4, and of lse (absolute, mean) at most 2^-4."""
    import torch
    inp = mi.make_inputs(B=4, H=128, n_q=1, seq_lens=[4096, 700, 1500, 130], seed=96)
    pg = mi.make_paged(inp, spare_pages=3)
    d, pg8, codes = fp8_device(inp, pg, mla)
    r8 = run_fp8(mla, inp, d)
    r16 = mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], d["cache"], d["block_table"],
                          d["seq_lens"], n_q=1)
    torch.cuda.synchronize()
    _, mr_u = errors(dev_bf16_to_f64(r8["u"]), dev_bf16_to_f64(r16["u"]))
    _, mr_out = errors(dev_bf16_to_f64(r8["out"]), dev_bf16_to_f64(r16["out"]))
    lse_diff = np.abs(r8["lse"].double().cpu().numpy() - r16["lse"].double().cpu().numpy()).mean()
    assert mr_u <= 2.0 ** -4 and mr_out <= 2.0 ** -4 and lse_diff <= 2.0 ** -4, (mr_u, mr_out, lse_diff)
    # and it is a real change (the FP8 path does not read the bf16 cache)
    assert mr_u > 2.0 ** -9


def test_step_and_captured_step_on_the_fp8_cache(mla):
    """decode_step and CapturedStep take the FP8 cache with its scales: the bits of the
    explicit FP8 path (plan, absorb, FP8 decode, merge, up-projection), and the oracle on
    the dequantised codes."""
    import torch
    inp = mi.make_inputs(B=4, H=128, n_q=2, seq_lens=[3, 130, 700, 64], seed=57)
    pg = mi.make_paged(inp, spare_pages=2)
    d, pg8, codes = fp8_device(inp, pg, mla)
    cache8 = torch.from_numpy(pg8.cache).cuda()
    scales = torch.from_numpy(pg8.scales).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], cache8, d["block_table"], d["seq_lens"],
                        n_q=2, num_splits=7, err_word=err, fp8_scales=scales)
    q_abs = mla.absorb_q(d["q_nope"], d["q_rope"], d["w_uk"])
    ws, g = mla.decode_paged_fp8(q_abs, cache8, scales, d["block_table"], d["seq_lens"], n_q=2, num_splits=7,
                                 err_word=err)
    u, lse = mla.combine(ws, B=4, n_q=2, H=128, num_splits=g)
    out = mla.out_proj(u, d["w_uv"])
    step = mla.CapturedStep(d["w_uk"], d["w_uv"], cache8, d["block_table"], d["seq_lens"], n_q=2, num_splits=7,
                            err_word=err, fp8_scales=scales)
    rc = step(d["q_nope"], d["q_rope"])
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for k, ref in (("u", u), ("out", out)):
        assert np.array_equal(dev_to_bits(r[k]), dev_to_bits(ref)), k
        assert np.array_equal(dev_to_bits(rc[k]), dev_to_bits(ref)), k
    assert np.array_equal(r["lse"].cpu().numpy().view(np.uint32), lse.cpu().numpy().view(np.uint32))
    o = oracle.absorbed_fp8_f64(inp, codes, pg8.scales)
    T, H = inp.B * inp.n_q, inp.H
    assert_close(dev_bf16_to_f64(r["out"]).reshape(T * H, 128), o["out"], "out")
    with pytest.raises(ValueError):
        mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], cache8, d["block_table"], d["seq_lens"],
                        n_q=2)


def test_fp8_steps_back_to_back_on_one_workspace_and_host_io(mla):
    """FP8 steps with alternating lengths enqueued back to back on one workspace give the bits
    of each step run alone; the host-I/O graph on the FP8 cache gives the eager step's bits."""
    import torch
    inps = [mi.make_inputs(B=8, H=128, n_q=1, seq_lens=lens, seed=60 + i)
            for i, lens in enumerate([[2048] * 8, [64, 3000, 1, 700, 2000, 130, 1500, 900]])]
    pgs = [mi.make_paged(x, spare_pages=2) for x in inps]
    ds = [fp8_device(x, pg, mla)[0] for x, pg in zip(inps, pgs)]

    def step(d, bufs=None):
        return mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], d["cache8"], d["block_table"],
                               d["seq_lens"], n_q=1, num_splits=20, bufs=bufs, fp8_scales=d["scales"])

    refs = []
    for d in ds:
        refs.append(step(d))
        torch.cuda.synchronize()
    ws = torch.zeros(mla.workspace_bytes(8, 1, 128, 20), dtype=torch.uint8, device="cuda")
    outs = [(i, step(d, {"workspace": ws})) for rep in range(3) for i, d in enumerate(ds)]
    torch.cuda.synchronize()
    for i, r in outs:
        for k in ("u", "out"):
            assert np.array_equal(dev_to_bits(r[k]), dev_to_bits(refs[i][k])), (i, k)
    d = ds[1]
    cap = mla.CapturedStep(d["w_uk"], d["w_uv"], d["cache8"], d["block_table"], d["seq_lens"], n_q=1,
                           num_splits=20, host_io=True, fp8_scales=d["scales"])
    cap.host["q_nope"].copy_(d["q_nope"].cpu())
    cap.host["q_rope"].copy_(d["q_rope"].cpu())
    cap.replay_host()
    torch.cuda.synchronize()
    assert torch.equal(cap.host["out"].view(torch.int16), refs[1]["out"].cpu().view(torch.int16))
    assert torch.equal(cap.host["lse"], refs[1]["lse"].cpu())
