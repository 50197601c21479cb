"""GPU tests of the cache-append step (mla_append_kv) against the oracle.

The new tokens' rows, c = h W^DKV and k^R = RoPE(h W^KR) (Huny's Dev Blog "MLA
아키텍처 해부" sections 1.2 and 2.2), are compared element by element with the
fp64 oracle: each is a bf16 rounding of an fp32 sum, so the bound is one bf16
rounding (2^-8 relative) plus 1e-3 absolute for fp32 accumulation over
d_model. Every other byte of the cache must be unchanged, and repeated calls
give identical bits. The last test runs the pages' case 5 (section 5): tokens
appended one by one on the GPU and decoded after each, against the oracle on
the same growing context.
"""
import math

import numpy as np
import pytest

import mla_inputs as mi
import oracle
from tests.helpers import assert_close, dev_bf16_to_f64, dev_to_bits, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    import mla_latent_kv_paged_gb300 as m
    m.build()
    return m


def _weights(d_model, seed):
    rng = np.random.default_rng(seed)
    return mi.f32_to_bf16((rng.standard_normal((576, d_model)) / math.sqrt(d_model)).astype(np.float32))


def _hidden(T, d_model, seed):
    rng = np.random.default_rng(seed)
    return mi.f32_to_bf16(rng.standard_normal((T, d_model)).astype(np.float32))


def _rows(bits_cache, block_table, seq_lens, n_q):
    """The new rows (b, j) as read back from a cache of bf16 bits [pages, 64, 576]."""
    out = []
    for b, L in enumerate(seq_lens):
        for j in range(n_q):
            pos = int(L) - n_q + j
            out.append(bits_cache[block_table[b][pos // 64], pos % 64])
    return np.stack(out)


@pytest.mark.parametrize("n_q,d_model,lens", [
    (1, 512, [1, 64, 65, 200]),
    (2, 7168, [2, 64, 129, 300]),
    (1, 7168, [4096] * 32),      # the benchmark's batch at DeepSeek-V3 width
    (2, 1024, list(range(2, 300, 3))),  # 100 sequences: two row tiles
])
def test_append_writes_the_oracle_rows(mla, n_q, d_model, lens):
    import torch
    B = len(lens)
    inp = mi.make_inputs(B=B, H=8, n_q=n_q, seq_lens=lens, seed=11 + d_model)
    pg = mi.make_paged(inp, spare_pages=4)
    h = _hidden(B * n_q, d_model, 5)
    w = _weights(d_model, 6)
    cache = to_dev_bf16(pg.cache)
    before = dev_to_bits(cache)
    bt, sl = to_dev_i32(pg.block_table), to_dev_i32(inp.seq_lens)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = mla.append_kv(to_dev_bf16(h), to_dev_bf16(w), cache, bt, sl, n_q=n_q, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    after = dev_to_bits(cache)
    pos = np.array([int(L) - n_q + j for L in inp.seq_lens for j in range(n_q)], dtype=np.int64)
    ref = oracle.append_f64(h, w, pos)
    got = mi.bf16_to_f32(_rows(after, pg.block_table, inp.seq_lens, n_q)).astype(np.float64)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-3), np.abs(got - ref).max()
    # nothing else changed (slack rows and spare pages keep their NaN poison)
    mask = np.ones(after.shape[:2], dtype=bool)
    for b, L in enumerate(inp.seq_lens):
        for j in range(n_q):
            p = int(L) - n_q + j
            mask[pg.block_table[b][p // 64], p % 64] = False
    assert np.array_equal(after[mask], before[mask])
    # the same bits again with the returned (zeroed-again) workspace
    cache2 = to_dev_bf16(pg.cache)
    mla.append_kv(to_dev_bf16(h), to_dev_bf16(w), cache2, bt, sl, n_q=n_q, workspace=ws, err_word=err)
    torch.cuda.synchronize()
    assert np.array_equal(dev_to_bits(cache2), after)


def test_append_then_decode_matches_the_oracle(mla):
    """Huny section 5 case 5 on the GPU: four decode steps, each appending its token's row
    with mla_append_kv and decoding the grown context; the oracle gets the same contexts with
    its own appended rows."""
    import dataclasses
    import torch
    B, H, d_model = 3, 16, 512
    lens0 = np.array([63, 64, 130])
    base = mi.make_inputs(B=B, H=H, n_q=1, seq_lens=lens0 + 4, seed=91)  # room for four new tokens
    pg = mi.make_paged(base, spare_pages=4)
    cache = to_dev_bf16(pg.cache)
    bt = to_dev_i32(pg.block_table)
    w = _weights(d_model, 92)
    d_w = to_dev_bf16(w)
    # logical rows on the host: the first lens0[b] rows of each sequence, then the appended ones
    c_rows = [base.c[base.seq_off[b]:base.seq_off[b] + lens0[b]].copy() for b in range(B)]
    kr_rows = [base.kr[base.seq_off[b]:base.seq_off[b] + lens0[b]].copy() for b in range(B)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = None
    for step in range(4):
        L = lens0 + step + 1
        sl = to_dev_i32(L)
        h = _hidden(B, d_model, 93 + step)
        ws = mla.append_kv(to_dev_bf16(h), d_w, cache, bt, sl, n_q=1, workspace=ws, err_word=err)
        new = mi.f32_to_bf16(oracle.append_f64(h, w, L - 1).astype(np.float32))
        for b in range(B):
            c_rows[b] = np.vstack([c_rows[b], new[b:b + 1, :512]])
            kr_rows[b] = np.vstack([kr_rows[b], new[b:b + 1, 512:]])
        rng = np.random.default_rng(200 + step)
        q_nope = mi.f32_to_bf16(rng.standard_normal((B, 1, H, 128)).astype(np.float32))
        q_rope = mi.f32_to_bf16(rng.standard_normal((B, 1, H, 64)).astype(np.float32))
        inp = dataclasses.replace(base, seq_lens=L.astype(np.int32),
                                  seq_off=np.concatenate([[0], np.cumsum(L)]).astype(np.int64),
                                  c=np.vstack(c_rows), kr=np.vstack(kr_rows), q_nope=q_nope, q_rope=q_rope)
        r = mla.decode_step(to_dev_bf16(q_nope.reshape(B, H, 128)), to_dev_bf16(q_rope.reshape(B, H, 64)),
                            to_dev_bf16(base.w_uk), to_dev_bf16(base.w_uv), cache, bt, sl, n_q=1, err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ref = oracle.absorbed_f64(inp)
        assert_close(dev_bf16_to_f64(r["out"]).reshape(-1, 128), ref["out"], f"out step {step}")
        assert_close(r["lse"].double().cpu().numpy().reshape(-1), ref["lse"], f"lse step {step}")
