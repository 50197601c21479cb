"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties the oracle to something it does not compute itself: the
explicit (non-absorbed) path the pages prove equal (Huny's Dev Blog "MLA
아키텍처 해부", section 3 and section 5 case 4), torch's textbook
scaled-dot-product attention on explicitly reconstructed keys and values,
closed forms (one token, zero query), numpy reductions, and the rank bound of
section 5 case 2. ``test_planted_mistakes_are_caught`` shows that each of five
plausible mistakes planted in the oracle fails these pins.
"""
import math

import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle

SCALE = 1.0 / math.sqrt(128 + 64)


def f64(bits):
    return mi.bf16_to_f32(bits).astype(np.float64)


def sdpa_reference(inp, scale=SCALE):
    """Textbook attention via torch SDPA on explicit K = c W_UK^T, V = c W_UV^T (fp64)."""
    H, n_q = inp.H, inp.n_q
    wk = torch.from_numpy(f64(inp.w_uk))  # [H, d_nope, d_c]
    wv = torch.from_numpy(f64(inp.w_uv))  # [H, d_v, d_c]
    qn = torch.from_numpy(f64(inp.q_nope))
    qr = torch.from_numpy(f64(inp.q_rope))
    outs, lses = [], []
    for b in range(inp.B):
        s0, s1 = int(inp.seq_off[b]), int(inp.seq_off[b + 1])
        L = s1 - s0
        cb = torch.from_numpy(f64(inp.c[s0:s1]))
        kb = torch.from_numpy(f64(inp.kr[s0:s1]))
        K = torch.einsum("sc,hic->hsi", cb, wk)                       # [H, L, d_nope]
        key = torch.cat([K, kb.expand(H, L, kb.shape[1])], dim=-1)    # [H, L, 192]
        V = torch.einsum("sc,hic->hsi", cb, wv)                       # [H, L, d_v]
        q = torch.cat([qn[b], qr[b]], dim=-1).permute(1, 0, 2)        # [H, n_q, 192]
        allowed = torch.arange(L)[None, :] <= (L - n_q + torch.arange(n_q))[:, None]  # [n_q, L]
        o = torch.nn.functional.scaled_dot_product_attention(
            q[None], key[None], V[None], attn_mask=allowed, scale=scale)[0]           # [H, n_q, d_v]
        logits = torch.einsum("hjd,hsd->hjs", q, key) * scale
        lse = torch.logsumexp(logits.masked_fill(~allowed, float("-inf")), dim=-1)    # [H, n_q]
        outs.append(o.permute(1, 0, 2))
        lses.append(lse.permute(1, 0))
    out = torch.stack(outs).reshape(-1, wv.shape[1]).numpy()
    lse = torch.stack(lses).reshape(-1).numpy()
    return out, lse


@pytest.fixture(scope="module")
def tiny():
    return mi.workload_inputs(1)


@pytest.fixture(scope="module")
def multitok():
    # ragged contexts, two causal queries, several pages, a one-token-past-page tail
    return mi.make_inputs(B=3, H=4, n_q=2, seq_lens=[5, 64, 130], seed=7)


def test_absorbed_equals_explicit_tiny(tiny):
    """Huny section 5 case 4: absorbed and explicit agree; the pages print ~1e-15."""
    a = oracle.absorbed_f64(tiny)
    e = oracle.explicit_f64(tiny)
    assert np.abs(a["out"] - e["out"]).max() <= 1e-10
    assert np.abs(a["lse"] - e["lse"]).max() <= 1e-10


def test_absorbed_equals_explicit_logits_and_probs(multitok):
    n_max = int(multitok.seq_lens.max())
    e = oracle.explicit_f64(multitok, max_tokens=n_max)
    for row in range(multitok.B * multitok.n_q * multitok.H):
        a = oracle.absorbed_probs_f64(multitok, row)
        n = len(a["logits"])
        assert np.abs(a["logits"] - e["logits"][row, :n]).max() <= 1e-10
        assert np.abs(a["probs"] - e["probs"][row, :n]).max() <= 1e-10
        assert np.all(e["probs"][row, n:] == 0.0)


@pytest.mark.parametrize("case", ["tiny", "multitok"])
def test_oracle_matches_torch_sdpa(case, request):
    """The oracle's result equals torch's textbook attention on explicit K, V."""
    inp = request.getfixturevalue(case)
    ref_out, ref_lse = sdpa_reference(inp)
    a = oracle.absorbed_f64(inp)
    e = oracle.explicit_f64(inp)
    assert np.abs(a["out"] - ref_out).max() <= 1e-10
    assert np.abs(e["out"] - ref_out).max() <= 1e-10
    assert np.abs(a["lse"] - ref_lse).max() <= 1e-10


def test_score_split_equals_concatenated_dot(multitok):
    """Huny section 2.2 and section 5 case 3: q.k = q^C.k^C + q^R.k^R."""
    row = 2 * multitok.H + 3  # b=1, j=0, h=3
    b, j, h = 1, 0, 3
    a = oracle.absorbed_probs_f64(multitok, row)
    s0 = int(multitok.seq_off[b])
    n = len(a["logits"])
    K = oracle.explicit_keys_f64(multitok.c[s0:s0 + n], multitok.w_uk, h)      # [n, 128]
    qn = f64(multitok.q_nope[b, j, h])
    qr = f64(multitok.q_rope[b, j, h])
    kr = f64(multitok.kr[s0:s0 + n])
    concat = np.concatenate([K, kr], axis=1) @ np.concatenate([qn, qr])
    assert np.abs(a["content"] - K @ qn).max() <= 1e-12 * max(1.0, np.abs(K @ qn).max())
    assert np.abs(a["pos"] - kr @ qr).max() <= 1e-12 * max(1.0, np.abs(kr @ qr).max())
    assert np.abs((a["content"] + a["pos"]) - concat).max() <= 1e-11


@pytest.mark.parametrize("L", [1, 2, 3, 64, 65])
def test_softmax_rows_sum_to_one(L):
    """ikmyungterran guide section 1.4: the softmax weights of a row sum to 1."""
    inp = mi.make_inputs(B=1, H=2, n_q=1, seq_lens=[L], seed=100 + L)
    e = oracle.explicit_f64(inp, max_tokens=L)
    assert np.abs(e["probs"].sum(axis=1) - 1.0).max() <= 1e-12
    assert (e["probs"] >= 0).all()
    for row in range(2):
        a = oracle.absorbed_probs_f64(inp, row)
        assert abs(a["probs"].sum() - 1.0) <= 1e-12


def test_single_token_context_returns_its_latent():
    """One cached token: the weight is exactly 1, so u is that latent."""
    inp = mi.make_inputs(B=2, H=3, n_q=1, seq_lens=[1, 1], seed=3)
    a = oracle.absorbed_f64(inp)
    for b in range(2):
        for h in range(3):
            r = b * 3 + h
            c0 = f64(inp.c[inp.seq_off[b]])
            assert np.array_equal(a["u"][r], c0)
            z0 = (a["q_abs"][r] @ np.concatenate([c0, f64(inp.kr[inp.seq_off[b]])])) * SCALE
            assert abs(a["lse"][r] - z0) <= 1e-12 * max(1.0, abs(z0))
            ref = f64(inp.w_uv[h]) @ c0
            assert np.abs(a["out"][r] - ref).max() <= 1e-12


def test_zero_query_averages_the_latents():
    """q = 0 gives uniform weights: u = mean of the attended latents, lse = ln n."""
    inp = mi.make_inputs(B=2, H=2, n_q=2, seq_lens=[7, 70], seed=5)
    inp.q_nope[...] = 0
    inp.q_rope[...] = 0
    a = oracle.absorbed_f64(inp)
    for b in range(2):
        for j in range(2):
            n = int(inp.seq_lens[b]) - 2 + j + 1
            mean = f64(inp.c[inp.seq_off[b]: inp.seq_off[b] + n]).mean(axis=0)
            for h in range(2):
                r = (b * 2 + j) * 2 + h
                assert np.abs(a["u"][r] - mean).max() <= 1e-12
                assert abs(a["lse"][r] - math.log(n)) <= 1e-12


def test_identity_absorption_is_single_head_attention():
    """W_UK = [I_128 | 0]: the absorbed query is q^C padded with zeros, so the
    result is textbook attention with keys [c[:, :128] ; k^R] and values W_UV c."""
    inp = mi.make_inputs(B=1, H=1, n_q=1, seq_lens=[97], seed=11)
    w = np.zeros((1, 128, 512), dtype=np.uint16)
    w[0, np.arange(128), np.arange(128)] = 0x3F80  # bf16 1.0
    inp.w_uk = w
    a = oracle.absorbed_f64(inp)
    c = torch.from_numpy(f64(inp.c))
    key = torch.cat([c[:, :128], torch.from_numpy(f64(inp.kr))], dim=1)
    V = c @ torch.from_numpy(f64(inp.w_uv[0])).T
    q = torch.cat([torch.from_numpy(f64(inp.q_nope[0, 0, 0])), torch.from_numpy(f64(inp.q_rope[0, 0, 0]))])
    o = torch.nn.functional.scaled_dot_product_attention(q[None, None], key[None], V[None], scale=SCALE)[0, 0]
    assert np.abs(a["q_abs"][0, :128] - f64(inp.q_nope[0, 0, 0])).max() == 0.0
    assert np.abs(a["q_abs"][0, 128:512]).max() == 0.0
    assert np.abs(a["out"][0] - o.numpy()).max() <= 1e-10


def test_reconstructed_keys_have_rank_at_most_d_c():
    """Huny section 5 case 2 (d_c = 16 here): K = C W_UK^T has rank <= d_c."""
    rng = np.random.default_rng(21)
    c = mi.f32_to_bf16(rng.standard_normal((128, 16), dtype=np.float32))
    w = mi.f32_to_bf16(rng.standard_normal((2, 64, 16), dtype=np.float32))
    for h in range(2):
        K = oracle.explicit_keys_f64(c, w, h)
        assert K.shape == (128, 64)
        assert np.abs(K - f64(c) @ f64(w[h]).T).max() <= 1e-12
        assert np.linalg.matrix_rank(K) == 16


def test_split_pieces_merge_to_the_unsplit_result(multitok):
    """Log-sum-exp merge of per-range partials reproduces the whole softmax."""
    rows = np.arange(multitok.B * multitok.n_q * multitok.H)
    full = oracle.absorbed_f64(multitok)
    one = oracle.split_partials_f64(multitok, [[0, 1 << 30]], rows)
    assert np.abs(one["u"][:, 0] - full["u"]).max() <= 1e-12
    assert np.abs(one["lse"][:, 0] - full["lse"]).max() <= 1e-12
    pieces = [[0, 3], [3, 64], [64, 129], [129, 200], [500, 600]]
    parts = oracle.split_partials_f64(multitok, pieces, rows)
    assert np.isneginf(parts["lse"][:, 4]).all() and (parts["u"][:, 4] == 0).all()
    merged = oracle.combine_f64(parts["u"], parts["lse"])
    assert np.abs(merged["u"] - full["u"]).max() <= 1e-12
    assert np.abs(merged["lse"] - full["lse"]).max() <= 1e-12


def test_fp32_variant_tracks_fp64(tiny):
    a = oracle.absorbed_f64(tiny)
    f = oracle.absorbed_f32(tiny)
    assert np.abs(f["out"] - a["out"]).max() <= 1e-4 * max(1.0, np.abs(a["out"]).max())
    assert np.abs(f["lse"] - a["lse"]).max() <= 1e-4


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5])
def test_planted_mistakes_are_caught(mutant, multitok):
    """A copy of the oracle with one planted mistake must fail the SDPA pin."""
    ref_out, ref_lse = sdpa_reference(multitok)
    bad = oracle.mutant_absorbed_f64(mutant, multitok)
    err = max(np.abs(bad["out"] - ref_out).max(), np.abs(bad["lse"] - ref_lse).max())
    assert err > 1e-6, f"mutant {mutant} slipped through (err {err:g})"


def test_single_step_functions(tiny):
    """The absorption and up-projection steps alone agree with numpy matmuls and
    with the corresponding parts of the whole absorbed path."""
    T = tiny.B * tiny.n_q
    qn = tiny.q_nope.reshape(T, tiny.H, -1)
    qr = tiny.q_rope.reshape(T, tiny.H, -1)
    qa = oracle.absorb_q_f64(qn, qr, tiny.w_uk)
    ref = np.einsum("thi,hic->thc", f64(qn), f64(tiny.w_uk))
    assert np.abs(qa[..., :512] - ref).max() <= 1e-11
    assert np.array_equal(qa[..., 512:], f64(qr))
    full = oracle.absorbed_f64(tiny)
    assert np.abs(qa.reshape(-1, 576) - full["q_abs"]).max() <= 1e-12
    rng = np.random.default_rng(8)
    u = mi.f32_to_bf16(rng.standard_normal((T, tiny.H, 512), dtype=np.float32))
    o = oracle.out_proj_f64(u, tiny.w_uv)
    assert np.abs(o - np.einsum("hvc,thc->thv", f64(tiny.w_uv), f64(u))).max() <= 1e-11
    # W_UV applied to the absorbed path's own u reproduces its out
    o_full = np.einsum("hvc,thc->thv", f64(tiny.w_uv), full["u"].reshape(T, tiny.H, 512))
    assert np.abs(o_full.reshape(-1, 128) - full["out"]).max() <= 1e-11


# ------------------------------------------------------------------ cache append
def _append_case(T=5, d_model=96, seed=3):
    rng = np.random.default_rng(seed)
    h = mi.f32_to_bf16(rng.standard_normal((T, d_model)).astype(np.float32))
    w = mi.f32_to_bf16((rng.standard_normal((576, d_model)) / math.sqrt(d_model)).astype(np.float32))
    pos = np.array([0, 1, 63, 64, 131071][:T], dtype=np.int64)
    return h, w, pos


def test_append_latent_part_is_the_plain_projection():
    """Huny section 1.2: c_t = h_t W^DKV, checked against numpy's matmul."""
    h, w, pos = _append_case()
    r = oracle.append_f64(h, w, pos)
    assert np.abs(r[:, :512] - f64(h) @ f64(w[:512]).T).max() < 1e-12


def test_append_positional_part_matches_the_generator_rotation():
    """Section 2.2: k^R_t = RoPE(h_t W^KR), against the input generator's own rotation code."""
    h, w, pos = _append_case()
    r = oracle.append_f64(h, w, pos)
    k = f64(h) @ f64(w[512:]).T
    assert np.abs(r[:, 512:] - mi.rope_rotate(k, pos)).max() < 1e-10
    # position 0 is the identity rotation
    assert np.array_equal(r[0, 512:], k[0])


def test_append_identity_weights_and_rotation_properties():
    """W = I (d_model = 576): the row is h with its last 64 values rotated; the rotation keeps
    every pair's norm, and the dot of two rotated vectors depends only on the position gap."""
    rng = np.random.default_rng(5)
    T = 4
    h = mi.f32_to_bf16(rng.standard_normal((T, 576)).astype(np.float32))
    eye = mi.f32_to_bf16(np.eye(576, dtype=np.float32))
    pos = np.array([3, 10, 1000, 1007], dtype=np.int64)
    r = oracle.append_f64(h, eye, pos)
    assert np.array_equal(r[:, :512], f64(h)[:, :512])
    x = f64(h)[:, 512:]
    pairs_in = x[:, 0::2] ** 2 + x[:, 1::2] ** 2
    pairs_out = r[:, 512::2] ** 2 + r[:, 513::2] ** 2
    assert np.abs(pairs_in - pairs_out).max() < 1e-12 * max(1.0, pairs_in.max())
    # same inputs at positions (3, 10) and (1000, 1007): the same gap of 7, the same dot
    same = np.vstack([x[0], x[1], x[0], x[1]])
    h2 = np.hstack([f64(h)[:, :512], same])
    r2 = oracle.append_f64(mi.f32_to_bf16(h2.astype(np.float32)), eye, pos)
    d1 = r2[0, 512:] @ r2[1, 512:]
    d2 = r2[2, 512:] @ r2[3, 512:]
    assert abs(d1 - d2) < 1e-9 * max(1.0, abs(d1))


# ------------------------------------------------------------------ query-side absorption
def _latent_case(T=3, H=4, d_q=96, seed=9):
    c_q, w_uq = mi.latent_query_inputs(T, H, d_q, seed)
    rng = np.random.default_rng(seed + 1)
    w_uk = mi.f32_to_bf16((rng.standard_normal((H, 128, 512)) / math.sqrt(512)).astype(np.float32))
    q_rope = mi.f32_to_bf16(rng.standard_normal((T, H, 64)).astype(np.float32))
    return c_q, w_uq, w_uk, q_rope


def test_merged_weight_is_the_per_head_product():
    """ingu627 "Multi-Head Latent Attention (MLA)" section 2.2, W_KQ = W_UK^T W_UQ per head,
    against numpy's einsum; with W_UQ the identity (d_q = d_nope) the merge returns W_UK."""
    _, w_uq, w_uk, _ = _latent_case()
    m = oracle.merge_w_kq_f64(w_uq, w_uk)
    assert np.abs(m - np.einsum("khi,hic->khc", f64(w_uq), f64(w_uk))).max() < 1e-12
    H = w_uk.shape[0]
    eye = np.zeros((128, H, 128), dtype=np.float32)
    for h in range(H):
        eye[:, h, :] = np.eye(128, dtype=np.float32)
    m = oracle.merge_w_kq_f64(mi.f32_to_bf16(eye), w_uk)
    assert np.array_equal(m, f64(w_uk).transpose(1, 0, 2))


def test_latent_query_equals_the_two_step_query():
    """Associativity: the absorbed query through the merged weight equals c_q W_UQ (the
    no-RoPE query) followed by the absorption step of the unmerged path."""
    c_q, w_uq, w_uk, q_rope = _latent_case()
    qa = oracle.absorb_latent_f64(c_q, oracle.merge_w_kq_f64(w_uq, w_uk), q_rope)
    q_nope = np.einsum("tk,khi->thi", f64(c_q), f64(w_uq))
    two_step = np.einsum("thi,hic->thc", q_nope, f64(w_uk))
    assert np.abs(qa[..., :512] - two_step).max() < 1e-12 * max(1.0, np.abs(two_step).max())
    assert np.array_equal(qa[..., 512:], f64(q_rope))
    # the same through the oracle's own absorption step, when q_nope is bf16-exact:
    # one-hot compressed queries pick rows of W_UQ, which are bf16 values
    T, d_q = c_q.shape
    one_hot = np.zeros((T, d_q), dtype=np.float32)
    ks = [0, d_q // 2, d_q - 1]
    for t in range(T):
        one_hot[t, ks[t]] = 1.0
    oh = mi.f32_to_bf16(one_hot)
    qa1 = oracle.absorb_latent_f64(oh, oracle.merge_w_kq_f64(w_uq, w_uk), q_rope)
    ref = oracle.absorb_q_f64(np.stack([w_uq[k] for k in ks]), q_rope, w_uk)
    assert np.abs(qa1 - ref).max() < 1e-12
    zero = oracle.absorb_latent_f64(np.zeros_like(c_q), oracle.merge_w_kq_f64(w_uq, w_uk), q_rope)
    assert not zero[..., :512].any() and np.array_equal(zero[..., 512:], f64(q_rope))


def test_merged_scores_equal_the_explicit_keys_scores():
    """S = C_KV^T (W_UK^T W_UQ) C_Q: the latent scores of the merged query equal the
    scores of the explicitly reconstructed keys against the decompressed query."""
    c_q, w_uq, w_uk, q_rope = _latent_case(T=2)
    rng = np.random.default_rng(33)
    c = mi.f32_to_bf16(rng.standard_normal((40, 512)).astype(np.float32))
    qa = oracle.absorb_latent_f64(c_q, oracle.merge_w_kq_f64(w_uq, w_uk), q_rope)
    q_nope = np.einsum("tk,khi->thi", f64(c_q), f64(w_uq))
    for h in range(w_uk.shape[0]):
        K = oracle.explicit_keys_f64(c, w_uk, h)  # [tokens][d_nope]
        s_explicit = q_nope[:, h, :] @ K.T
        s_latent = qa[:, h, :512] @ f64(c).T
        assert np.abs(s_latent - s_explicit).max() < 1e-11 * max(1.0, np.abs(s_explicit).max())


# ------------------------------------------------------------------ merged output projection
def _comb_case(T=3, H=4, d_model=80, seed=13):
    rng = np.random.default_rng(seed)
    u = mi.f32_to_bf16((rng.standard_normal((T, H, 512)) * 0.3).astype(np.float32))
    w_uv = mi.f32_to_bf16((rng.standard_normal((H, 128, 512)) / math.sqrt(512)).astype(np.float32))
    w_o = mi.output_projection(d_model, H, seed + 1)
    return u, w_uv, w_o


def test_merged_output_weight_is_the_per_head_product():
    """Huny section 3 item 2, W_i,comb = W_i^UV W_i^O, against numpy's einsum; an identity
    output projection (d_model = H * d_v) gives W_UV itself."""
    u, w_uv, w_o = _comb_case()
    m = oracle.merge_w_comb_f64(w_uv, w_o)
    assert np.abs(m - np.einsum("nhv,hvc->nhc", f64(w_o), f64(w_uv))).max() < 1e-12
    H = w_uv.shape[0]
    eye = np.eye(H * 128, dtype=np.float32).reshape(H * 128, H, 128)
    m = oracle.merge_w_comb_f64(w_uv, mi.f32_to_bf16(eye))
    assert np.array_equal(m.reshape(H, 128, H, 512)[np.arange(H), :, np.arange(H)], f64(w_uv))


def test_merged_output_equals_out_proj_then_output_projection():
    """Associativity: u W_comb summed over heads equals the unmerged route, the per-head
    up-projection (the oracle's out_proj) followed by the output projection."""
    u, w_uv, w_o = _comb_case()
    got = oracle.out_comb_f64(u, oracle.merge_w_comb_f64(w_uv, w_o))
    heads = oracle.out_proj_f64(u, w_uv)  # [T][H][d_v]
    ref = np.einsum("thv,nhv->tn", heads, f64(w_o))
    assert np.abs(got - ref).max() < 1e-12 * max(1.0, np.abs(ref).max())
    # identity output projection: the heads side by side
    H = w_uv.shape[0]
    eye = mi.f32_to_bf16(np.eye(H * 128, dtype=np.float32).reshape(H * 128, H, 128))
    side = oracle.out_comb_f64(u, oracle.merge_w_comb_f64(w_uv, eye))
    assert np.abs(side - heads.reshape(u.shape[0], -1)).max() < 1e-12
