"""GPU tests of the merged value/output projection (mla_merge_w_comb, mla_out_comb).

W_comb = W_UV W_O per head and the layer output u W_comb summed over heads
(Huny's Dev Blog "MLA 아키텍처 해부" section 3, item 2) are compared with the
fp64 oracle on the same bf16 inputs. The merge is one bf16 rounding of an fp32
sum over d_v = 128 terms: bound 2^-8 relative. The output sums H * 512 products
in fp32 partials (split across CTAs, added in a fixed order) and is rounded to
bf16 once: bound 2^-8 relative plus an absolute term of 2^-16 times the sum of
the products' magnitudes (fp32 accumulation). At DeepSeek-V3 width (d_model
7168, 128 heads) the merged weight is checked on sampled output columns, whose
rows the oracle merges alone.
"""
import math

import numpy as np
import pytest

import mla_inputs as mi
import oracle
from tests.helpers import assert_close, dev_bf16_to_f64, dev_to_bits, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    import mla_latent_kv_paged_gb300 as m
    m.build()
    return m


def _w_uv(H, seed):
    rng = np.random.default_rng(seed)
    return mi.f32_to_bf16((rng.standard_normal((H, 128, 512)) / math.sqrt(512)).astype(np.float32))


def _u(T, H, seed):
    # u is a convex combination of N(0,1) latents: smaller than 1 in magnitude
    rng = np.random.default_rng(seed)
    return mi.f32_to_bf16((rng.standard_normal((T, H, 512)) * 0.3).astype(np.float32))


def _bound(u_bits, w, ref):
    """2^-8 relative + 2^-16 x sum_k |u_k w_k| per output (fp32 accumulation over H * 512 terms)."""
    mag = np.abs(mi.bf16_to_f32(u_bits).astype(np.float64)).reshape(u_bits.shape[0], -1) @ \
        np.abs(w.reshape(w.shape[0], -1)).T
    return np.abs(ref) * 2.0 ** -8 + mag * 2.0 ** -16


@pytest.mark.parametrize("H,d_model", [(4, 128), (16, 384), (128, 256)])
def test_merge_matches_the_oracle(mla, H, d_model):
    import torch
    w_uv = _w_uv(H, H)
    w_o = mi.output_projection(d_model, H, seed=d_model)
    got = dev_bf16_to_f64(mla.merge_w_comb(to_dev_bf16(w_uv), to_dev_bf16(w_o)))
    torch.cuda.synchronize()
    ref = oracle.merge_w_comb_f64(w_uv, w_o)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-7), np.abs(got - ref).max()


@pytest.mark.parametrize("T,H,d_model", [(1, 4, 128), (32, 16, 512), (33, 8, 256), (130, 2, 384), (32, 128, 256)])
def test_out_comb_matches_the_oracle(mla, T, H, d_model):
    """The same bf16 W_comb (the oracle's merge, rounded) on both sides; row tiles of 32,
    64 and 128 with ragged tails, one to sixteen splits of the reduction."""
    import torch
    u = _u(T, H, T + H)
    w = mi.f32_to_bf16(oracle.merge_w_comb_f64(_w_uv(H, 3), mi.output_projection(d_model, H, 4)).astype(np.float32))
    got = dev_bf16_to_f64(mla.out_comb(to_dev_bf16(u), to_dev_bf16(w)))
    torch.cuda.synchronize()
    wf = mi.bf16_to_f32(w).astype(np.float64)
    ref = oracle.out_comb_f64(u, w)
    assert got.shape == (T, d_model)
    assert np.all(np.abs(got - ref) <= _bound(u, wf, ref)), np.abs(got - ref).max()


def test_merged_output_at_v3_width_on_sampled_columns(mla):
    """d_model 7168, 128 heads, 32 rows (the benchmark's shape): GPU merge and GPU output,
    against the oracle's exact merged output (no rounding of W_comb) on 24 sampled output
    columns, within the decode tolerance (max-abs 2e-2, mean-rel 5e-3); the same call twice
    gives the same bits."""
    import torch
    T, H, d_model = 32, 128, 7168
    u = _u(T, H, 41)
    w_uv = _w_uv(H, 42)
    w_o = mi.output_projection(d_model, H, 43)
    w_comb = mla.merge_w_comb(to_dev_bf16(w_uv), to_dev_bf16(w_o))
    d_u = to_dev_bf16(u)
    out = mla.out_comb(d_u, w_comb)
    out2 = mla.out_comb(d_u, w_comb)
    torch.cuda.synchronize()
    cols = np.random.default_rng(44).choice(d_model, 24, replace=False)
    cols[:2] = [0, d_model - 1]
    ref = oracle.out_comb_f64(u, oracle.merge_w_comb_f64(w_uv, w_o[cols]))
    assert_close(dev_bf16_to_f64(out)[:, cols], ref, "merged output, sampled columns")
    # the merged weight's sampled rows, elementwise
    wc = dev_bf16_to_f64(w_comb)[cols]
    wref = oracle.merge_w_comb_f64(w_uv, w_o[cols])
    assert np.all(np.abs(wc - wref) <= np.abs(wref) * 2.0 ** -8 + 1e-7)
    assert np.array_equal(dev_to_bits(out), dev_to_bits(out2))
