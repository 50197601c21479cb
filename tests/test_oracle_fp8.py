"""Pins of the oracle's FP8 latent-cache path (CPU only).

The FP8 cache keeps each latent row as e4m3 codes with one float32 scale per
column (Huny's Dev Blog "MLA 아키텍처 해부", section 6 item 4: FP8 on the latent
needs per-channel or per-block scales; ailab.paldyn.com "MQA와 GQA", KV-cache
quantisation: outlier channels are why K is scaled per channel). The oracle's
decode of the codes, its dequantisation and its absorbed path on dequantised
latents are pinned here to a library decoder, to e4m3's rounding bound, and to
the already pinned bf16 absorbed path.
"""
import math

import numpy as np
import pytest

import mla_inputs as mi
import oracle


def test_e4m3_decode_matches_the_library_type_for_every_code():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_decode_special_values():
    v = oracle.e4m3_decode(np.array([0x00, 0x80, 0x38, 0xB8, 0x7E, 0x01, 0x08, 0x07, 0x3F], dtype=np.uint8))
    assert v[0] == 0.0 and v[1] == 0.0 and math.copysign(1, v[1]) < 0
    assert v[2] == 1.0 and v[3] == -1.0          # exponent field 7 = bias
    assert v[4] == 448.0                          # 2^8 * 1.75, the largest finite value
    assert v[5] == 2.0 ** -9                      # smallest subnormal
    assert v[6] == 2.0 ** -6                      # smallest normal
    assert v[7] == 7 * 2.0 ** -9                  # largest subnormal
    assert v[8] == 1.875                          # 1 + 7/8
    # codes 0..126 are strictly increasing
    assert (np.diff(oracle.e4m3_decode(np.arange(127, dtype=np.uint8))) > 0).all()


def test_quantiser_round_trip_within_half_a_quantum():
    """dequant(quant(x)) - x is at most half of e4m3's spacing at |x| (2^-4 relative in the
    normal range, s * 2^-10 absolute below it), with the per-channel scales' definition."""
    inp = mi.make_inputs(B=2, H=4, n_q=1, seq_lens=[300, 77], seed=3)
    s = mi.fp8_channel_scales(inp)
    rows = np.concatenate([inp.c, inp.kr], axis=1)
    x = mi.bf16_to_f32(rows).astype(np.float64)
    # each column's largest magnitude maps to the largest code
    amax = np.abs(x).max(axis=0)
    assert np.allclose(amax / s, 448.0, rtol=1e-6)
    deq = oracle.dequant_fp8_f64(mi.quantize_fp8(rows, s), s)
    y = x / s  # the value each code approximates, in units of the scale
    half_q = np.where(np.abs(y) >= 2.0 ** -6, np.abs(y) * 2.0 ** -4, 2.0 ** -10)
    assert (np.abs(deq / s - y) <= half_q * (1 + 1e-6) + 1e-12).all()
    # and the codes are round-to-nearest: the error exceeds a third of a quantum somewhere
    assert (np.abs(deq / s - y) > half_q / 3).any()


def test_quantiser_matches_the_library_conversion():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(50000) * 60, rng.standard_normal(50000) * 0.003]).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mi.f32_to_e4m3(x), ref)
    assert mi.f32_to_e4m3(np.array([1000.0, -1e6], np.float32)).tolist() == [0x7E, 0xFE]  # saturated


@pytest.mark.parametrize("n_q", [1, 2])
def test_fp8_path_equals_bf16_path_on_exact_values(n_q):
    """With scale 1 and latents that are e4m3 values (all exact in bf16), the FP8 oracle
    and the bf16 oracle run the same arithmetic on the same numbers: identical bits."""
    base = mi.make_inputs(B=3, H=8, n_q=n_q, seq_lens=[40, 129, 3], seed=5 + n_q)
    rng = np.random.default_rng(17)
    codes = rng.integers(0, 0x40, size=(base.total_tokens, 576)).astype(np.uint8)  # |v| <= 1.875
    codes |= (rng.integers(0, 2, size=codes.shape) << 7).astype(np.uint8)
    vals = oracle.e4m3_decode(codes)
    bits = mi.f32_to_bf16(vals.astype(np.float32))
    assert np.array_equal(mi.bf16_to_f32(bits).astype(np.float64), vals)
    import dataclasses
    inp = dataclasses.replace(base, c=bits[:, :512].copy(), kr=bits[:, 512:].copy())
    a = oracle.absorbed_f64(inp)
    f = oracle.absorbed_fp8_f64(inp, codes, np.ones(576, np.float32))
    for k in ("q_abs", "u", "lse", "out"):
        assert np.array_equal(a[k], f[k]), k


def test_fp8_scales_enter_both_score_and_value():
    """Doubling every scale doubles the dequantised latents: in a one-token context u is the
    dequantised row itself and doubles, and the log-sum-exp is the token's score, which
    doubles (both the latent and the positional term scale)."""
    inp = mi.make_inputs(B=1, H=4, n_q=1, seq_lens=[1], seed=9)
    rows = np.concatenate([inp.c, inp.kr], axis=1)
    s = mi.fp8_channel_scales(inp)
    codes = mi.quantize_fp8(rows, s)
    r1 = oracle.absorbed_fp8_f64(inp, codes, s)
    r2 = oracle.absorbed_fp8_f64(inp, codes, 2 * s)
    deq = oracle.dequant_fp8_f64(codes, s)
    assert np.array_equal(r1["u"], np.repeat(deq[:, :512], 4, axis=0))
    assert np.array_equal(r2["u"], 2 * r1["u"])
    assert np.array_equal(r2["lse"], 2 * r1["lse"])
