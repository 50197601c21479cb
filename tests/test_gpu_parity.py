"""Parity of the CUDA path with the CPU oracle, through the C ABI (GPU only).

Floating-point results must agree with the oracle within max |err| <= 2e-2 and
sum|err| / sum|ref| <= 5e-3 (bf16 inputs, fp32 accumulation); integer and
indexing work (the split plan, page gathers, error words) must be bit-exact.
"""
import math

import numpy as np
import pytest

import mla_inputs as mi
import oracle
from tests.helpers import (assert_close, dev_bf16_to_f64, dev_to_bits, device_inputs, plan_mirror,
                           to_dev_bf16, to_dev_i32)

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(192.0)


@pytest.fixture(scope="module")
def mla():
    import mla_latent_kv_paged_gb300 as m
    m.build()
    return m


def run_step(mla, inp, pg, num_splits=None, err=None):
    import torch
    d = device_inputs(inp, pg)
    if err is None:
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], d["cache"], d["block_table"],
                        d["seq_lens"], n_q=inp.n_q, num_splits=num_splits, err_word=err)
    torch.cuda.synchronize()
    r["err"] = int(err.item())
    return r


def compare_full(inp, r, rows=None):
    ref = oracle.absorbed_f64(inp, rows)
    T, H = inp.B * inp.n_q, inp.H
    sel = slice(None) if rows is None else rows
    u = dev_bf16_to_f64(r["u"]).reshape(T * H, 512)[sel]
    out = dev_bf16_to_f64(r["out"]).reshape(T * H, 128)[sel]
    lse = r["lse"].double().cpu().numpy().reshape(T * H)[sel]
    assert_close(u, ref["u"], "u")
    assert_close(lse, ref["lse"], "lse")
    return assert_close(out, ref["out"], "out")


# ------------------------------------------------------------------ single steps
@pytest.mark.parametrize("T,H", [(2, 16), (37, 128), (128, 128), (3, 5)])
def test_absorb_q(mla, T, H):
    rng = np.random.default_rng(T * 1000 + H)
    qn = mi.f32_to_bf16(rng.standard_normal((T, H, 128), dtype=np.float32))
    qr = mi.f32_to_bf16(rng.standard_normal((T, H, 64), dtype=np.float32))
    wk = mi.f32_to_bf16(rng.standard_normal((H, 128, 512), dtype=np.float32) / np.float32(math.sqrt(512)))
    ref = oracle.absorb_q_f64(qn, qr, wk)
    q_abs = mla.absorb_q(to_dev_bf16(qn), to_dev_bf16(qr), to_dev_bf16(wk))
    got_bits = dev_to_bits(q_abs)
    assert np.array_equal(got_bits[..., 512:], qr)  # the rotated query is copied bit for bit
    got = mi.bf16_to_f32(got_bits[..., :512]).astype(np.float64)
    # one bf16 rounding of an fp32 sum: within 2^-8 relative plus fp32 noise
    assert (np.abs(got - ref[..., :512]) <= np.abs(ref[..., :512]) * 2.0 ** -8 + 1e-5).all()


@pytest.mark.parametrize("T,H", [(2, 16), (37, 128), (128, 128), (3, 5)])
def test_out_proj(mla, T, H):
    rng = np.random.default_rng(T * 7 + H)
    u = mi.f32_to_bf16(rng.standard_normal((T, H, 512), dtype=np.float32) * np.float32(0.1))
    wv = mi.f32_to_bf16(rng.standard_normal((H, 128, 512), dtype=np.float32) / np.float32(math.sqrt(512)))
    ref = oracle.out_proj_f64(u, wv)
    out = dev_bf16_to_f64(mla.out_proj(to_dev_bf16(u), to_dev_bf16(wv)))
    assert (np.abs(out - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-5).all()


def test_captured_step_replays_equal_eager_steps(mla):
    """CapturedStep gives the eager step's bits, and sees in-place changes of seq_lens / block_table."""
    import torch
    inp = mi.make_inputs(B=3, H=128, n_q=2, seq_lens=[70, 300, 129], seed=77)
    pg = mi.make_paged(inp, spare_pages=8)
    d = device_inputs(inp, pg)
    step = mla.CapturedStep(d["w_uk"], d["w_uv"], d["cache"], d["block_table"], d["seq_lens"], n_q=2, num_splits=5)
    r = step(d["q_nope"], d["q_rope"])
    e = mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], d["cache"], d["block_table"],
                        d["seq_lens"], n_q=2, num_splits=5)
    torch.cuda.synchronize()
    for k in ("u", "out"):
        assert torch.equal(r[k].view(torch.int16), e[k].view(torch.int16)), k
    assert torch.equal(r["lse"], e["lse"])
    compare_full(inp, r)
    # shorter contexts and another page order, written in place: the replay follows them
    inp2 = mi.make_inputs(B=3, H=128, n_q=2, seq_lens=[66, 200, 64], seed=78)
    pg2 = mi.make_paged(inp2, perm_seed=5, spare_pages=8, max_pages=pg.max_pages)
    d2 = device_inputs(inp2, pg2)
    d["cache"][: d2["cache"].shape[0]].copy_(d2["cache"])
    d["w_uk"].copy_(d2["w_uk"])  # the step keeps pointers to the weights as well
    d["w_uv"].copy_(d2["w_uv"])
    d["block_table"].copy_(d2["block_table"])
    d["seq_lens"].copy_(d2["seq_lens"])
    r2 = step(d2["q_nope"], d2["q_rope"])
    torch.cuda.synchronize()
    compare_full(inp2, r2)


def test_captured_step_host_io_copies_inside_the_graph(mla):
    """host_io=True: inputs from pinned host buffers, results back to them, in one replay;
    the same bits as the eager step, and new host inputs are picked up by the next replay."""
    import torch
    inp = mi.make_inputs(B=3, H=128, n_q=1, seq_lens=[70, 300, 129], seed=79)
    pg = mi.make_paged(inp, spare_pages=8)
    d = device_inputs(inp, pg)
    step = mla.CapturedStep(d["w_uk"], d["w_uv"], d["cache"], d["block_table"], d["seq_lens"], n_q=1,
                            num_splits=5, host_io=True)
    h = step.host
    h["q_nope"].copy_(d["q_nope"].cpu())
    h["q_rope"].copy_(d["q_rope"].cpu())
    step.replay_host()
    torch.cuda.synchronize()
    e = mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], d["cache"], d["block_table"],
                        d["seq_lens"], n_q=1, num_splits=5)
    torch.cuda.synchronize()
    assert torch.equal(h["out"].view(torch.int16), e["out"].cpu().view(torch.int16))
    assert torch.equal(h["lse"], e["lse"].cpu())
    # a shorter context for sequence 1 (its first 200 rows), written into the host buffer only
    import dataclasses
    L = inp.seq_lens.copy()
    L[1] = 200
    off = inp.seq_off
    keep = np.concatenate([np.arange(off[0], off[1]), np.arange(off[1], off[1] + 200), np.arange(off[2], off[3])])
    inp2 = dataclasses.replace(inp, seq_lens=L.astype(np.int32),
                               seq_off=np.concatenate([[0], np.cumsum(L)]).astype(np.int64),
                               c=inp.c[keep], kr=inp.kr[keep])
    h["seq_lens"].copy_(torch.from_numpy(inp2.seq_lens))
    step.replay_host()
    torch.cuda.synchronize()
    ref = oracle.absorbed_f64(inp2)
    assert_close(dev_bf16_to_f64(h["out"]).reshape(-1, 128), ref["out"], "out")
    assert_close(h["lse"].double().numpy().reshape(-1), ref["lse"], "lse")


def test_combine_alone_merges_oracle_partials(mla):
    """Feed oracle partials through the documented workspace layout into mla_combine."""
    import torch
    inp = mi.make_inputs(B=3, H=8, n_q=2, seq_lens=[70, 300, 129], seed=31)
    G = 4
    pl = plan_mirror(inp.seq_lens, inp.n_q, 8, G)
    ws = torch.zeros(mla.workspace_bytes(inp.B, inp.n_q, inp.H, G), dtype=torch.uint8, device="cuda")
    # fill seq_item and the partials at the documented offsets
    I = G + inp.B
    offs, off = [], 0
    for nbytes in [64 * 4, (G + 1) * 4, (inp.B + 1) * 4, inp.B * 4, I * 4, I * 4, I * 4,
                   I * inp.n_q * inp.H * 4, I * inp.n_q * inp.H * 512 * 2]:
        offs.append(off)
        off = (off + nbytes + 255) // 256 * 256
    host = np.zeros(ws.numel(), dtype=np.uint8)
    host[offs[2]:offs[2] + (inp.B + 1) * 4] = pl["seq_item"].astype(np.int32).view(np.uint8)
    lse_part = np.full((I, inp.n_q, inp.H), -np.inf, dtype=np.float32)
    o_part = np.zeros((I, inp.n_q, 64, inp.H, 8), dtype=np.float16)  # [c/8][h][c%8]
    rows = np.arange(inp.B * inp.n_q * inp.H)
    for k, (b, p0, p1) in enumerate(pl["items"]):
        part = oracle.split_partials_f64(inp, [[p0 * 64, p1 * 64]], rows)
        for j in range(inp.n_q):
            r = (b * inp.n_q + j) * inp.H + np.arange(inp.H)
            lse_part[k, j] = part["lse"][r, 0]
            o_part[k, j] = part["u"][r, 0].reshape(inp.H, 64, 8).transpose(1, 0, 2)
    host[offs[7]:offs[7] + lse_part.nbytes] = lse_part.view(np.uint8).ravel()
    host[offs[8]:offs[8] + o_part.nbytes] = o_part.view(np.uint8).ravel()
    ws.copy_(torch.from_numpy(host))
    u, lse = mla.combine(ws, B=inp.B, n_q=inp.n_q, H=inp.H, num_splits=G)
    torch.cuda.synchronize()
    ref = oracle.absorbed_f64(inp)
    assert_close(dev_bf16_to_f64(u).reshape(-1, 512), ref["u"], "u", max_abs=1e-2, mean_rel=3e-3)
    assert np.abs(lse.double().cpu().numpy().ravel() - ref["lse"]).max() <= 1e-5


# ------------------------------------------------------------------ the decode path
def test_tiny_workload_all_rows(mla):
    inp = mi.workload_inputs(1)
    pg = mi.make_paged(inp, spare_pages=4)
    r = run_step(mla, inp, pg)
    assert r["err"] == 0
    compare_full(inp, r)


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 64])
def test_ragged_multitoken_all_rows(mla, splits):
    """Several pages, partial last pages, a 1-token sequence, causal pairs, any split count."""
    inp = mi.make_inputs(B=5, H=128, n_q=2, seq_lens=[2, 64, 65, 300, 1000], seed=41)
    pg = mi.make_paged(inp, spare_pages=3)
    r = run_step(mla, inp, pg, num_splits=splits)
    assert r["err"] == 0
    compare_full(inp, r)


@pytest.mark.parametrize("H", [1, 16, 100])
def test_fewer_heads(mla, H):
    inp = mi.make_inputs(B=3, H=H, n_q=1, seq_lens=[130, 64, 7], seed=43 + H)
    pg = mi.make_paged(inp)
    r = run_step(mla, inp, pg, num_splits=4)
    assert r["err"] == 0
    compare_full(inp, r)


def test_full_step_matches_explicit_path(mla):
    """Multi-token decode against the oracle's explicit (non-absorbed) K, V path."""
    inp = mi.make_inputs(B=2, H=128, n_q=2, seq_lens=[333, 129], seed=45)
    pg = mi.make_paged(inp)
    r = run_step(mla, inp, pg)
    e = oracle.explicit_f64(inp)
    out = dev_bf16_to_f64(r["out"]).reshape(-1, 128)
    assert_close(out, e["out"], "out vs explicit")


def test_page_permutation_is_bit_exact(mla):
    """The same logical cache in two different page layouts gives identical bits."""
    inp = mi.make_inputs(B=4, H=128, n_q=1, seq_lens=[500, 64, 1, 257], seed=47)
    r1 = run_step(mla, inp, mi.make_paged(inp, perm_seed=1, spare_pages=2))
    r2 = run_step(mla, inp, mi.make_paged(inp, perm_seed=2, spare_pages=9))
    for k in ["u", "out", "q_abs"]:
        assert np.array_equal(dev_to_bits(r1[k]), dev_to_bits(r2[k])), k
    assert np.array_equal(r1["lse"].cpu().numpy().view(np.uint32), r2["lse"].cpu().numpy().view(np.uint32))


def test_plan_is_bit_exact(mla):
    import torch
    inp = mi.make_inputs(B=6, H=16, n_q=1, seq_lens=[1, 65, 130, 64, 1000, 63], seed=49)
    pg = mi.make_paged(inp)
    G = 5
    r = run_step(mla, inp, pg, num_splits=G)
    ws = r["workspace"].cpu().numpy()
    B = inp.B
    I = G + B

    def i32(off, n):
        return ws[off:off + 4 * n].view(np.int32)

    offs, off = [], 0
    for nbytes in [64 * 4, (G + 1) * 4, (B + 1) * 4, B * 4, I * 4, I * 4, I * 4]:
        offs.append(off)
        off = (off + nbytes + 255) // 256 * 256
    pl = plan_mirror(inp.seq_lens, 1, pg.max_pages, G)
    n = len(pl["items"])
    hdr = i32(offs[0], 3)
    assert list(hdr) == [n, pl["Ge"], pl["total"]]
    assert np.array_equal(i32(offs[1], G + 1), pl["range_item"])
    assert np.array_equal(i32(offs[2], B + 1), pl["seq_item"])
    assert np.array_equal(i32(offs[3], B), inp.seq_lens)
    assert np.array_equal(i32(offs[4], n), pl["items"][:, 0])
    assert np.array_equal(i32(offs[5], n), pl["items"][:, 1])
    assert np.array_equal(i32(offs[6], n), pl["items"][:, 2])
    # the range descriptions at the end of the workspace: each range's first piece
    off_lse = off  # after item_tile1: lse_part, o_part, then range_desc
    off_o = (off_lse + I * inp.n_q * inp.H * 4 + 255) // 256 * 256
    off_rd = (off_o + I * inp.n_q * inp.H * 512 * 2 + 255) // 256 * 256
    desc = ws[off_rd:off_rd + 16 * (G + 1)].view(np.int32).reshape(G + 1, 4)
    for p in range(G + 1):
        r = int(pl["range_item"][p])
        want = [r, -1, 0, 0] if r >= n else [r, *(int(x) for x in pl["items"][r])]
        assert list(desc[p]) == want, (p, list(desc[p]), want)


@pytest.mark.parametrize("splits", [None, 7000])
def test_maximum_batch_short_contexts(mla, splits):
    """B = MLA_MAX_BATCH sequences of 1..130 tokens (one-token contexts included); 7000 splits is
    more ranges than pages, so some ranges are empty and every other range holds one page."""
    lens = np.random.default_rng(4096).integers(1, 131, size=4096)
    lens[:3] = [1, 64, 65]
    inp = mi.make_inputs(B=4096, H=8, n_q=1, seq_lens=list(lens), seed=4096)
    pg = mi.make_paged(inp, spare_pages=2)
    r = run_step(mla, inp, pg, num_splits=splits)
    assert r["err"] == 0
    compare_full(inp, r)
    if splits is not None:
        G, B = splits, inp.B
        ws = r["workspace"].cpu().numpy()
        offs, off = [], 0
        for nbytes in [64 * 4, (G + 1) * 4, (B + 1) * 4]:
            offs.append(off)
            off = (off + nbytes + 255) // 256 * 256
        pl = plan_mirror(inp.seq_lens, 1, pg.max_pages, G)
        assert np.array_equal(ws[offs[1]:offs[1] + 4 * (G + 1)].view(np.int32), pl["range_item"])
        assert np.array_equal(ws[offs[2]:offs[2] + 4 * (B + 1)].view(np.int32), pl["seq_item"])


def test_incremental_decode_matches_fresh(mla):
    """Huny section 5 case 5: 8 prefill tokens, then 4 decode steps each appending
    one latent; every step matches the oracle at that length, and decoding a
    cache that already holds later tokens in its slack gives the same bits."""
    import torch
    full = mi.make_inputs(B=1, H=128, n_q=1, seq_lens=[12], seed=51)
    pg_full = mi.make_paged(full, spare_pages=0)
    d = device_inputs(full, pg_full)
    for L in range(8, 13):
        sub = mi.Inputs(B=1, H=128, n_q=1, seq_lens=np.array([L], np.int32),
                        seq_off=np.array([0, L]), c=full.c[:L], kr=full.kr[:L], q_nope=full.q_nope,
                        q_rope=full.q_rope, w_uk=full.w_uk, w_uv=full.w_uv)
        pg_sub = mi.make_paged(sub, spare_pages=0)
        r_fresh = run_step(mla, sub, pg_sub)
        compare_full(sub, r_fresh)
        sl = torch.tensor([L], dtype=torch.int32, device="cuda")
        r_grown = mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], d["cache"],
                                  d["block_table"], sl, n_q=1)
        torch.cuda.synchronize()
        for k in ["u", "out"]:
            assert np.array_equal(dev_to_bits(r_fresh[k]), dev_to_bits(r_grown[k])), (L, k)


def test_back_to_back_steps_share_one_workspace(mla):
    """Steps enqueued back to back on one workspace with other lengths each time (so other
    plans): the next step's plan is written while the kernel before it still runs, which
    must not be while the previous step's decode kernel or merge still read the plan.
    Each step is compared bit for bit with the same step run alone."""
    import torch
    H = 128
    inps = [mi.make_inputs(B=8, H=H, n_q=1, seq_lens=lens, seed=90 + i)
            for i, lens in enumerate([[4096] * 8, [64, 5000, 1, 700, 3000, 130, 2000, 900]])]
    pgs = [mi.make_paged(x, spare_pages=2) for x in inps]
    ds = [device_inputs(x, pg) for x, pg in zip(inps, pgs)]
    refs = []
    for d in ds:
        refs.append(mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], d["cache"], d["block_table"],
                                    d["seq_lens"], n_q=1, num_splits=20))
        torch.cuda.synchronize()
    ws = torch.zeros(mla.workspace_bytes(8, 1, H, 20), dtype=torch.uint8, device="cuda")
    outs = []
    for rep in range(4):
        for i, d in enumerate(ds):
            outs.append((i, mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], d["cache"],
                                            d["block_table"], d["seq_lens"], n_q=1, num_splits=20,
                                            bufs={"workspace": ws})))
    torch.cuda.synchronize()
    for i, r in outs:
        for k in ("u", "out"):
            assert np.array_equal(dev_to_bits(r[k]), dev_to_bits(refs[i][k])), (i, k)
        assert np.array_equal(r["lse"].cpu().numpy().view(np.uint32), refs[i]["lse"].cpu().numpy().view(np.uint32))


def test_device_errors_are_reported_without_faulting(mla):
    import torch
    inp = mi.make_inputs(B=2, H=16, n_q=1, seq_lens=[100, 70], seed=53)
    pg = mi.make_paged(inp)
    d = device_inputs(inp, pg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # context longer than the block table row
    sl = torch.tensor([100, 64 * pg.max_pages + 5], dtype=torch.int32, device="cuda")
    mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], d["cache"], d["block_table"], sl,
                    n_q=1, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 6
    # a page id outside the pool
    err.zero_()
    bt = d["block_table"].clone()
    bt[0, 0] = pg.num_pages + 3
    mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], d["cache"], bt, d["seq_lens"],
                    n_q=1, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 6
    # latents beyond the fp16 range of the split partials (|c| = 2^17): the
    # normalised partial of a range is a convex combination of them
    err.zero_()
    big = d["cache"].clone()
    big[..., :512] = 131072.0
    mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], big, d["block_table"], d["seq_lens"],
                    n_q=1, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 7
    # the context still works afterwards
    r = run_step(mla, inp, pg)
    assert r["err"] == 0
    compare_full(inp, r)


# ------------------------------------------------------------------ full-size workloads
SAMPLE = 24


def sampled_rows(inp, n=SAMPLE, seed=0):
    rng = np.random.default_rng(seed)
    total = inp.B * inp.n_q * inp.H
    rows = rng.choice(total, size=min(n, total), replace=False)
    # always include the first and last rows (first/last sequence, head 0 / H-1)
    return np.unique(np.concatenate([rows, [0, total - 1]])).astype(np.int64)


@pytest.mark.parametrize("index", [2, 3, 4, 5])
def test_full_size_workload_all_rows(mla, index):
    """Full-size workloads in the benchmark's launch configuration (default split
    count), every row (sequence, query, head) compared with the fp64 absorbed
    oracle; the explicit (non-absorbed) oracle, ~60 times costlier, on sampled rows
    of the two-token workload."""
    inp = mi.workload_inputs(index)
    pg = mi.make_paged(inp, spare_pages=mi.WORKLOADS[index].spare_pages)
    r = run_step(mla, inp, pg)
    assert r["err"] == 0
    compare_full(inp, r)
    if index == 5:
        rows = sampled_rows(inp, seed=index)[:4]
        e = oracle.explicit_f64(inp, rows)
        out = dev_bf16_to_f64(r["out"]).reshape(-1, 128)[rows]
        assert_close(out, e["out"], "out vs explicit")


@pytest.mark.parametrize("case", ["tiny", "ragged_multitoken", "many_short"])
def test_planned_decode_equals_decode_paged(mla, case):
    """mla_decode_plan (enqueued before mla_absorb_q) then mla_decode_paged_planned gives the
    workspace plan and the merged u, lse of mla_decode_paged bit for bit."""
    import torch
    splits = None
    if case == "tiny":
        inp = mi.workload_inputs(1)
    elif case == "ragged_multitoken":
        inp = mi.make_inputs(B=9, H=16, n_q=2, seq_lens=[2, 3, 64, 65, 129, 500, 1000, 77, 4000], seed=5)
        splits = 7
    else:
        lens = np.random.default_rng(7).integers(1, 131, size=1000)
        inp = mi.make_inputs(B=1000, H=8, n_q=1, seq_lens=list(lens), seed=7)
    pg = mi.make_paged(inp, spare_pages=2)
    d = device_inputs(inp, pg)
    B, H = inp.B, inp.H
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_abs = mla.absorb_q(d["q_nope"], d["q_rope"], d["w_uk"])
    ws1, g = mla.decode_paged(q_abs, d["cache"], d["block_table"], d["seq_lens"], n_q=inp.n_q,
                              num_splits=splits, err_word=err)
    u1, lse1 = mla.combine(ws1, B=B, n_q=inp.n_q, H=H, num_splits=g)
    ws2, g2 = mla.decode_plan(d["seq_lens"], n_q=inp.n_q, H=H, max_pages=pg.max_pages, num_pages=pg.num_pages,
                              num_splits=g, err_word=err)
    q2 = mla.absorb_q(d["q_nope"], d["q_rope"], d["w_uk"])
    mla.decode_paged(q2, d["cache"], d["block_table"], d["seq_lens"], n_q=inp.n_q, num_splits=g2, workspace=ws2,
                     err_word=err, planned=True)
    u2, lse2 = mla.combine(ws2, B=B, n_q=inp.n_q, H=H, num_splits=g2)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and g2 == g
    assert np.array_equal(ws1[:12].cpu().numpy(), ws2[:12].cpu().numpy())  # pieces, used splits, pages
    assert np.array_equal(dev_to_bits(u1), dev_to_bits(u2))
    assert np.array_equal(lse1.cpu().numpy().view(np.uint32), lse2.cpu().numpy().view(np.uint32))


def test_outputs_stay_inside_their_buffers(mla):
    """Red zones: every output and the workspace sit between guard bytes that must come
    back untouched, and no input (cache, tables, queries, weights) changes."""
    import torch
    inp = mi.make_inputs(B=5, H=128, n_q=2, seq_lens=[2, 64, 65, 300, 1000], seed=55)
    pg = mi.make_paged(inp, spare_pages=3)
    d = device_inputs(inp, pg)
    before = {k: v.clone() for k, v in d.items()}
    T, H, G = inp.B * inp.n_q, inp.H, 7
    GUARD = 4096

    def guarded(nbytes, dtype, shape):
        raw = torch.full((nbytes + 2 * GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
        return raw, raw[GUARD:GUARD + nbytes].view(dtype).view(shape)

    es = lambda dt: torch.tensor([], dtype=dt).element_size()  # noqa: E731
    raws, bufs = {}, {}
    for name, dt, shape in [("q_abs", torch.bfloat16, (T, H, 576)), ("u", torch.bfloat16, (T, H, 512)),
                            ("lse", torch.float32, (T, H)), ("out", torch.bfloat16, (T, H, 128))]:
        raws[name], bufs[name] = guarded(int(np.prod(shape)) * es(dt), dt, shape)
    wsb = mla.workspace_bytes(inp.B, inp.n_q, H, G)
    raws["workspace"], bufs["workspace"] = guarded(wsb, torch.uint8, (wsb,))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = mla.decode_step(d["q_nope"], d["q_rope"], d["w_uk"], d["w_uv"], d["cache"], d["block_table"],
                        d["seq_lens"], n_q=inp.n_q, num_splits=G, bufs=bufs, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for name, raw in raws.items():
        assert (raw[:GUARD] == 0xA5).all() and (raw[-GUARD:] == 0xA5).all(), name
    for k, v in d.items():
        assert torch.equal(v.view(torch.uint8) if v.dtype != torch.int32 else v,
                           before[k].view(torch.uint8) if v.dtype != torch.int32 else before[k]), k
    r["err"] = 0
    compare_full(inp, r)


def plan_arrays(ws, B, G):
    """The plan part of a decode workspace (host bytes) as numpy arrays, at the documented offsets."""
    I = G + B
    offs, off = [], 0
    for nbytes in [64 * 4, (G + 1) * 4, (B + 1) * 4, B * 4, I * 4, I * 4, I * 4]:
        offs.append(off)
        off = (off + nbytes + 255) // 256 * 256
    return offs, off


PLAN_CASES = [
    # (seq_lens, n_q, splits): one warp plans up to 32 sequences, a block beyond
    ([1], 1, 1), ([1], 1, 5), ([64, 65], 1, 1), ([64, 65], 1, 3), ([4096] * 32, 1, 76),
    ([4096] * 32, 1, 64), ([1, 2, 3] * 10 + [700, 9000], 1, 76), ([63, 64, 65, 127, 128, 129] * 5, 2, 17),
    (list(range(2, 66, 2)), 2, 200), ([300] * 33, 1, 76), ([5000, 1, 1, 1] * 10, 1, 7),
]


@pytest.mark.parametrize("lens,n_q,G", PLAN_CASES)
def test_plan_kernels_match_the_mirror(mla, lens, n_q, G):
    """Both plan kernels (a warp for at most 32 sequences, a block beyond) against the Python
    statement of the plan, every array bit for bit, including the range descriptions."""
    import torch
    B = len(lens)
    max_pages = max((L + 63) // 64 for L in lens)
    ws, g = mla.decode_plan(to_dev_i32(np.array(lens, dtype=np.int32)), n_q=n_q, H=8, max_pages=max_pages,
                            num_pages=B * max_pages, num_splits=G)
    torch.cuda.synchronize()
    host = ws.cpu().numpy()
    offs, off_lse = plan_arrays(host, B, G)
    I = G + B

    def i32(o, n):
        return host[o:o + 4 * n].view(np.int32)

    pl = plan_mirror(lens, n_q, max_pages, G)
    n = len(pl["items"])
    assert list(i32(offs[0], 3)) == [n, pl["Ge"], pl["total"]]
    assert np.array_equal(i32(offs[1], G + 1), pl["range_item"])
    assert np.array_equal(i32(offs[2], B + 1), pl["seq_item"])
    assert np.array_equal(i32(offs[3], B), np.clip(lens, n_q, None))
    for k in range(3):
        assert np.array_equal(i32(offs[4 + k], n), pl["items"][:, k])
    off_o = (off_lse + I * n_q * 8 * 4 + 255) // 256 * 256
    off_rd = (off_o + I * n_q * 8 * 512 * 2 + 255) // 256 * 256
    desc = host[off_rd:off_rd + 16 * (G + 1)].view(np.int32).reshape(G + 1, 4)
    for p in range(G + 1):
        r = int(pl["range_item"][p])
        want = [r, -1, 0, 0] if r >= n else [r, *(int(x) for x in pl["items"][r])]
        assert list(desc[p]) == want, (p, list(desc[p]), want)
