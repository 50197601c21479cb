"""The allocation-free decode entry point (GPU only; collected last on purpose).

mla_decode_noalloc serves callers that cannot hand the library a workspace:
it keeps the split plan and partial results in a fixed array inside the
library. Called twice in a row through the C ABI, it must give u and lse that
match the CPU oracle within the tolerances of the other parity tests, and the
same values as mla_decode_paged + mla_combine with a caller-provided workspace;
a request too large for the array must be refused before any launch.
"""
import ctypes

import numpy as np
import pytest

import mla_inputs as mi
import oracle
from tests.helpers import MAX_ABS, MEAN_REL, assert_close, dev_bf16_to_f64, dev_to_bits, device_inputs

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    import torch

    import mla_latent_kv_paged_gb300 as mla
    mla.build()
    lib = mla.lib()
    cases = [dict(B=6, n_q=1, lens=[100, 64, 1, 700, 130, 2000], seed=61, G=7),
             dict(B=3, n_q=2, lens=[5, 300, 64], seed=62, G=4)]
    for case in cases:  # two calls in a row on the shared scratch
        inp = mi.make_inputs(B=case["B"], H=128, n_q=case["n_q"], seq_lens=case["lens"], seed=case["seed"])
        pg = mi.make_paged(inp, spare_pages=3)
        d = device_inputs(inp, pg)
        q_abs = mla.absorb_q(d["q_nope"], d["q_rope"], d["w_uk"])
        ws, G = mla.decode_paged(q_abs, d["cache"], d["block_table"], d["seq_lens"], n_q=inp.n_q,
                                 num_splits=case["G"])
        u_ref, lse_ref = mla.combine(ws, B=inp.B, n_q=inp.n_q, H=inp.H, num_splits=G)
        u = torch.full_like(u_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        st = lib.mla_decode_noalloc(
            ctypes.c_void_p(q_abs.data_ptr()), ctypes.c_void_p(d["cache"].data_ptr()),
            ctypes.c_void_p(d["block_table"].data_ptr()), ctypes.c_void_p(d["seq_lens"].data_ptr()),
            inp.B, inp.n_q, inp.H, pg.num_pages, 64, pg.max_pages, ctypes.c_float(mla.DEFAULT_SCALE), G,
            ctypes.c_void_p(u.data_ptr()), ctypes.c_void_p(lse.data_ptr()), ctypes.c_void_p(err.data_ptr()),
            stream)
        assert st == 0, mla.STATUS.get(st, st)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        ref = oracle.absorbed_f64(inp)
        T, H = inp.B * inp.n_q, inp.H
        assert_close(dev_bf16_to_f64(u).reshape(T * H, 512), ref["u"], "u vs oracle", MAX_ABS, MEAN_REL)
        assert_close(lse.double().cpu().numpy().reshape(T * H), ref["lse"], "lse vs oracle", MAX_ABS, MEAN_REL)
        assert_close(dev_bf16_to_f64(u), dev_bf16_to_f64(u_ref), "u", MAX_ABS, MEAN_REL)
        assert_close(lse.double().cpu().numpy(), lse_ref.double().cpu().numpy(), "lse", MAX_ABS, MEAN_REL)


def test_noalloc_refuses_requests_beyond_its_array():
    import torch

    import mla_latent_kv_paged_gb300 as mla
    lib = mla.lib()
    cap = lib.mla_decode_noalloc_max_bytes()
    B, n_q, H, G = 4096, 2, 128, 76
    assert lib.mla_decode_workspace_bytes(B, n_q, H, G) > cap
    x = torch.zeros(64, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(x.data_ptr())
    st = lib.mla_decode_noalloc(p, p, p, p, B, n_q, H, 8, 64, 4, ctypes.c_float(0.07), G, p, p, None, None)
    assert st == 3  # MLA_ERR_WORKSPACE_TOO_SMALL, nothing launched


def test_noalloc_back_to_back_calls_with_different_lengths():
    """Calls enqueued back to back share the library's array: the second call's plan (other
    lengths, so other pieces) must not overwrite the array while the first call's merge still
    reads it. Each call is compared bit for bit with the workspace entry point."""
    import torch

    import mla_latent_kv_paged_gb300 as mla
    mla.build()
    H = 128
    inps = [mi.make_inputs(B=8, H=H, n_q=1, seq_lens=lens, seed=70 + i)
            for i, lens in enumerate([[4096] * 8, [64, 5000, 1, 700, 3000, 130, 2000, 900]])]
    pgs = [mi.make_paged(x, spare_pages=2) for x in inps]
    ds = [device_inputs(x, pg) for x, pg in zip(inps, pgs)]
    q_abs = [mla.absorb_q(d["q_nope"], d["q_rope"], d["w_uk"]) for d in ds]
    refs = []
    for i, d in enumerate(ds):
        ws, G = mla.decode_paged(q_abs[i], d["cache"], d["block_table"], d["seq_lens"], n_q=1, num_splits=20)
        refs.append(mla.combine(ws, B=8, n_q=1, H=H, num_splits=G))
    torch.cuda.synchronize()
    outs = []
    for rep in range(4):  # the two calls back to back, several times
        for i, d in enumerate(ds):
            u = torch.empty((8, H, 512), dtype=torch.bfloat16, device="cuda")
            lse = torch.empty((8, H), dtype=torch.float32, device="cuda")
            outs.append((i, mla.decode_noalloc(q_abs[i], d["cache"], d["block_table"], d["seq_lens"], n_q=1,
                                               u=u, lse=lse, num_splits=20)))
    torch.cuda.synchronize()
    for i, (u, lse) in outs:
        assert np.array_equal(dev_to_bits(u), dev_to_bits(refs[i][0]))
        assert np.array_equal(lse.cpu().numpy().view(np.uint32), refs[i][1].cpu().numpy().view(np.uint32))


def test_noalloc_in_pages_of_128():
    import torch

    import mla_latent_kv_paged_gb300 as mla
    mla.build()
    inp = mi.make_inputs(B=4, H=128, n_q=2, seq_lens=[3, 127, 129, 700], seed=171)
    pg = mi.make_paged(inp, spare_pages=2, page=128)
    d = device_inputs(inp, pg)
    q_abs = mla.absorb_q(d["q_nope"], d["q_rope"], d["w_uk"])
    T, H = inp.B * inp.n_q, inp.H
    u = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.decode_noalloc(q_abs, d["cache"], d["block_table"], d["seq_lens"], n_q=inp.n_q, num_splits=5, u=u,
                       lse=lse, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.absorbed_f64(inp)
    assert_close(dev_bf16_to_f64(u).reshape(T * H, 512), ref["u"], "u")
    assert_close(lse.double().cpu().numpy().reshape(T * H), ref["lse"], "lse")
