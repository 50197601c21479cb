"""Pages of 128 tokens (GPU only).

The Huny's Dev Blog page "MLA 아키텍처 해부" (section 6, item 2) sets MLA's
cache pages at 64 to 128 tokens. The kernels read the cache in tiles of 64
tokens, two to a page of 128: the split plan counts tiles, the decode kernel
finds a tile's page through the block table and its rows at offset
64 * (tile % 2) inside it, and the append kernel writes row pos % 128 of page
pos / 128. Parity is against the oracle at the tolerances of every parity
test; a cache laid out in pages of 128 must give the bits of the same tokens
laid out in pages of 64, because the kernels see the same tiles in the same
order either way.
"""
import math

import numpy as np
import pytest

import mla_inputs as mi
import oracle
from tests.helpers import (assert_close, dev_bf16_to_f64, dev_to_bits, device_inputs, plan_mirror, to_dev_bf16,
                           to_dev_i32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    import mla_latent_kv_paged_gb300 as m
    m.build()
    return m


def run_step(mla, inp, pg, num_splits=None):
    import torch
    d = device_inputs(inp, pg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], d["cache"], d["block_table"],
                        d["seq_lens"], n_q=inp.n_q, num_splits=num_splits, err_word=err)
    torch.cuda.synchronize()
    r["err"] = int(err.item())
    return r


def compare_full(inp, r):
    ref = oracle.absorbed_f64(inp)
    T, H = inp.B * inp.n_q, inp.H
    assert_close(dev_bf16_to_f64(r["u"]).reshape(T * H, 512), ref["u"], "u")
    assert_close(r["lse"].double().cpu().numpy().reshape(T * H), ref["lse"], "lse")
    assert_close(dev_bf16_to_f64(r["out"]).reshape(T * H, 128), ref["out"], "out")


@pytest.mark.parametrize("splits", [1, 3, 7, 64])
def test_ragged_multitoken_all_rows(mla, splits):
    """Contexts ending in either tile of their last page (64 | 65 | 127 | 128 | 129), a
    2-token sequence, causal pairs; with 64 splits most ranges start or end inside a page."""
    inp = mi.make_inputs(B=7, H=128, n_q=2, seq_lens=[2, 64, 65, 127, 128, 129, 1000], seed=141)
    pg = mi.make_paged(inp, spare_pages=3, page=128)
    assert pg.cache.shape[1] == 128
    r = run_step(mla, inp, pg, num_splits=splits)
    assert r["err"] == 0
    compare_full(inp, r)


@pytest.mark.parametrize("splits", [2, 76])
def test_same_bits_as_pages_of_64(mla, splits):
    inp = mi.make_inputs(B=5, H=128, n_q=1, seq_lens=[500, 64, 1, 257, 2000], seed=147)
    r64 = run_step(mla, inp, mi.make_paged(inp, perm_seed=1, spare_pages=2, page=64), num_splits=splits)
    r128 = run_step(mla, inp, mi.make_paged(inp, perm_seed=2, spare_pages=5, page=128), num_splits=splits)
    assert r64["err"] == 0 and r128["err"] == 0
    for k in ("u", "out", "q_abs"):
        assert np.array_equal(dev_to_bits(r64[k]), dev_to_bits(r128[k])), k
    assert np.array_equal(r64["lse"].cpu().numpy().view(np.uint32), r128["lse"].cpu().numpy().view(np.uint32))


def test_plan_counts_tiles_and_clamps_to_the_table(mla):
    """The plan's items are 64-token tile ranges; a context longer than max_pages * 128
    is clamped to it and reported (MLA_ERR_BOUNDS), the rest of the batch unaffected."""
    import torch
    inp = mi.make_inputs(B=6, H=16, n_q=1, seq_lens=[1, 65, 130, 64, 1000, 63], seed=149)
    pg = mi.make_paged(inp, page=128)
    G = 5
    ws, g = mla.decode_plan(to_dev_i32(inp.seq_lens), n_q=1, H=16, max_pages=pg.max_pages,
                            num_pages=pg.num_pages, num_splits=G, page_size=128)
    torch.cuda.synchronize()
    host = ws.cpu().numpy()
    B, I = inp.B, G + inp.B

    def i32(off, n):
        return host[off:off + 4 * n].view(np.int32)

    offs, off = [], 0
    for nbytes in [64 * 4, (G + 1) * 4, (B + 1) * 4, B * 4, I * 4, I * 4, I * 4]:
        offs.append(off)
        off = (off + nbytes + 255) // 256 * 256
    pl = plan_mirror(inp.seq_lens, 1, pg.max_pages, G, page=128)
    n = len(pl["items"])
    assert list(i32(offs[0], 3)) == [n, pl["Ge"], pl["total"]]
    assert pl["total"] == sum((L + 63) // 64 for L in inp.seq_lens)  # tiles, not pages
    assert np.array_equal(i32(offs[1], G + 1), pl["range_item"])
    assert np.array_equal(i32(offs[2], B + 1), pl["seq_item"])
    for k in range(3):
        assert np.array_equal(i32(offs[4 + k], n), pl["items"][:, k])
    # a context past the table's reach: 1000 tokens with max_pages 8 (1024 tokens) fits,
    # 1100 does not
    lens = inp.seq_lens.copy()
    lens[4] = 1100
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws2, _ = mla.decode_plan(to_dev_i32(lens), n_q=1, H=16, max_pages=pg.max_pages, num_pages=pg.num_pages,
                             num_splits=G, page_size=128, err_word=err)
    torch.cuda.synchronize()
    assert pg.max_pages * 128 == 1024
    assert int(err.item()) == 6  # MLA_ERR_BOUNDS
    assert ws2.cpu().numpy()[offs[3] + 16:offs[3] + 20].view(np.int32)[0] == 1024


def test_fp8_cache_in_pages_of_128(mla):
    import torch
    inp = mi.make_inputs(B=5, H=128, n_q=2, seq_lens=[2, 127, 129, 300, 1000], seed=151)
    pg = mi.make_paged(inp, spare_pages=3, page=128)
    pg8 = mi.make_paged_fp8(inp, pg)
    d = device_inputs(inp, pg)
    cache8 = torch.from_numpy(pg8.cache).cuda()
    scales = torch.from_numpy(pg8.scales).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_abs = mla.absorb_q(d["q_nope"], d["q_rope"], d["w_uk"])
    ws, g = mla.decode_paged_fp8(q_abs, cache8, scales, d["block_table"], d["seq_lens"], n_q=inp.n_q,
                                 num_splits=5, err_word=err)
    u, lse = mla.combine(ws, B=inp.B, n_q=inp.n_q, H=inp.H, num_splits=g)
    out = mla.out_proj(u, d["w_uv"])
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    codes = mi.quantize_fp8(np.concatenate([inp.c, inp.kr], axis=1), pg8.scales)
    ref = oracle.absorbed_fp8_f64(inp, codes, pg8.scales)
    T, H = inp.B * inp.n_q, inp.H
    assert_close(dev_bf16_to_f64(u).reshape(T * H, 512), ref["u"], "u")
    assert_close(lse.double().cpu().numpy().reshape(T * H), ref["lse"], "lse")
    assert_close(dev_bf16_to_f64(out).reshape(T * H, 128), ref["out"], "out")


def test_append_writes_row_pos_mod_128(mla):
    """mla_append_kv with pages of 128: row pos % 128 of page block_table[b][pos / 128]
    holds the oracle's row; every other byte of the cache is unchanged."""
    import torch
    lens = [1, 64, 65, 128, 129, 200, 256]
    n_q, d_model = 1, 512
    inp = mi.make_inputs(B=len(lens), H=8, n_q=n_q, seq_lens=lens, seed=155)
    pg = mi.make_paged(inp, spare_pages=2, page=128)
    rng = np.random.default_rng(156)
    h = mi.f32_to_bf16(rng.standard_normal((len(lens), d_model)).astype(np.float32))
    w = mi.f32_to_bf16((rng.standard_normal((576, d_model)) / math.sqrt(d_model)).astype(np.float32))
    cache = to_dev_bf16(pg.cache)
    before = dev_to_bits(cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.append_kv(to_dev_bf16(h), to_dev_bf16(w), cache, to_dev_i32(pg.block_table), to_dev_i32(inp.seq_lens),
                  n_q=n_q, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    after = dev_to_bits(cache)
    pos = np.array(lens, dtype=np.int64) - 1
    ref = oracle.append_f64(h, w, pos)
    got = np.stack([after[pg.block_table[b][p // 128], p % 128] for b, p in enumerate(pos)])
    got = mi.bf16_to_f32(got).astype(np.float64)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-3), np.abs(got - ref).max()
    mask = np.ones(after.shape[:2], dtype=bool)
    for b, p in enumerate(pos):
        mask[pg.block_table[b][p // 128], p % 128] = False
    assert np.array_equal(after[mask], before[mask])


def test_maximum_batch_in_pages_of_128(mla):
    """4096 short contexts in pages of 128 (the block plan kernel, tiles at both offsets of a
    page), and splits beyond the number of tiles (empty ranges)."""
    lens = np.random.default_rng(128).integers(1, 260, size=4096)
    lens[:4] = [1, 64, 65, 129]
    inp = mi.make_inputs(B=4096, H=8, n_q=1, seq_lens=list(lens), seed=128)
    pg = mi.make_paged(inp, spare_pages=2, page=128)
    for splits in (None, 9000):
        r = run_step(mla, inp, pg, num_splits=splits)
        assert r["err"] == 0
        compare_full(inp, r)

