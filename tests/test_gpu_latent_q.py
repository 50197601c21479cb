"""GPU tests of the query-side absorption (mla_merge_w_kq, mla_absorb_q_latent).

The merged weight W_KQ = W_UK^T W_UQ per head and the absorbed query taken
straight from the compressed query latent (ingu627.github.io "Multi-Head Latent
Attention (MLA)" section 2.2, S = C_KV^T W_KQ C_Q) are compared element by
element with the fp64 oracle on the same bf16 inputs: each output is one bf16
rounding of an fp32 sum, so the bound is 2^-8 relative plus a small absolute
term for fp32 accumulation. The positional columns are a copy and must match
bit for bit. The whole merged path is also held to the decode tolerance
against the unmerged two-step query computed exactly.
"""
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


def _w_uk(H, seed):
    rng = np.random.default_rng(seed)
    return mi.f32_to_bf16((rng.standard_normal((H, 128, 512)) / np.sqrt(512)).astype(np.float32))


def _q_rope(T, H, seed):
    rng = np.random.default_rng(seed)
    return mi.f32_to_bf16(rng.standard_normal((T, H, 64)).astype(np.float32))


@pytest.mark.parametrize("d_q,H", [(64, 128), (192, 8), (1536, 16), (1600, 3)])
def test_merge_matches_the_oracle(mla, d_q, H):
    import torch
    _, w_uq = mi.latent_query_inputs(1, H, d_q, seed=d_q + H)
    w_uk = _w_uk(H, 7)
    got = dev_bf16_to_f64(mla.merge_w_kq(to_dev_bf16(w_uq), to_dev_bf16(w_uk)))
    torch.cuda.synchronize()
    ref = oracle.merge_w_kq_f64(w_uq, w_uk)
    assert got.shape == ref.shape
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6), np.abs(got - ref).max()


@pytest.mark.parametrize("T,H,d_q", [(1, 4, 64), (32, 128, 1536), (100, 8, 512), (130, 4, 1536), (33, 2, 128)])
def test_latent_query_matches_the_oracle(mla, T, H, d_q):
    """The same bf16 W_KQ (the oracle's merge, rounded) on both sides."""
    import torch
    c_q, w_uq = mi.latent_query_inputs(T, H, d_q, seed=3 * T + d_q)
    w_kq = mi.f32_to_bf16(oracle.merge_w_kq_f64(w_uq, _w_uk(H, 8)).astype(np.float32))
    q_rope = _q_rope(T, H, 9)
    q_abs = mla.absorb_q_latent(to_dev_bf16(c_q), to_dev_bf16(q_rope), to_dev_bf16(w_kq))
    torch.cuda.synchronize()
    ref = oracle.absorb_latent_f64(c_q, w_kq, q_rope)
    got = dev_bf16_to_f64(q_abs)
    assert np.all(np.abs(got[..., :512] - ref[..., :512]) <= np.abs(ref[..., :512]) * 2.0 ** -8 + 1e-4), \
        np.abs(got - ref).max()
    assert np.array_equal(dev_to_bits(q_abs)[..., 512:], q_rope)


def test_merged_path_matches_the_two_step_query(mla):
    """GPU merge then GPU latent query, against the exact unmerged query
    (c_q W_UQ) W_UK of the oracle, at the benchmark's shape (32 rows, 128 heads,
    d_q 1536), within the decode tolerance (max-abs 2e-2, mean-rel 5e-3)."""
    import torch
    T, H, d_q = 32, 128, 1536
    c_q, w_uq = mi.latent_query_inputs(T, H, d_q, seed=77)
    w_uk = _w_uk(H, 78)
    q_rope = _q_rope(T, H, 79)
    w_kq = mla.merge_w_kq(to_dev_bf16(w_uq), to_dev_bf16(w_uk))
    got = dev_bf16_to_f64(mla.absorb_q_latent(to_dev_bf16(c_q), to_dev_bf16(q_rope), w_kq))
    torch.cuda.synchronize()
    ref = oracle.absorb_latent_f64(c_q, oracle.merge_w_kq_f64(w_uq, w_uk), q_rope)
    assert_close(got, ref, "merged query path")
    # the positional columns are a copy
    assert_close(got[..., 512:], ref[..., 512:], "positional columns", max_abs=0.0, mean_rel=0.0)


def test_latent_query_is_reproducible(mla):
    import torch
    T, H, d_q = 32, 16, 1536
    c_q, w_uq = mi.latent_query_inputs(T, H, d_q, seed=5)
    w_kq = mla.merge_w_kq(to_dev_bf16(w_uq), to_dev_bf16(_w_uk(H, 6)))
    a = mla.absorb_q_latent(to_dev_bf16(c_q), to_dev_bf16(_q_rope(T, H, 7)), w_kq)
    b = mla.absorb_q_latent(to_dev_bf16(c_q), to_dev_bf16(_q_rope(T, H, 7)), w_kq)
    torch.cuda.synchronize()
    assert np.array_equal(dev_to_bits(a), dev_to_bits(b))
