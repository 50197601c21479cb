"""A bounded wait of the decode kernel gives up, reports it, and leaves the context usable (GPU only).

Every wait of the decode kernel on an mbarrier is bounded; when one runs out
the kernel records MLA_ERR_TIMEOUT in err_word, lets every other wait of the
CTA return at once, frees its tensor memory and finishes. The test build of the
library (include/mla_debug.h) can keep the producer warp from loading anything
and shorten the limit to about a millisecond: nothing then completes the
consumers' barriers, the waits run out, and the call must return with the
error recorded. A normal call afterwards, in the same context, must match the
oracle. No fault, trap or hang is involved: the waits end by their limit.
"""
import numpy as np
import pytest

import mla_inputs as mi
import oracle
from tests.helpers import abi_step, assert_close, dev_bf16_to_f64, device_inputs

pytestmark = pytest.mark.gpu

MLA_ERR_TIMEOUT = 5


def test_wait_runs_out_then_context_recovers():
    import torch

    import mla_latent_kv_paged_gb300 as mla
    dbg = mla.debug_lib()
    inp = mi.make_inputs(B=2, H=128, n_q=1, seq_lens=[300, 130], seed=97)
    pg = mi.make_paged(inp, spare_pages=2)
    d = device_inputs(inp, pg)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert dbg.mla_debug_reset() == 0
    try:
        assert dbg.mla_debug_set_wait_limit(2_000_000) == 0  # about 1 ms of SM cycles
        assert dbg.mla_debug_set_skip_producer(1) == 0
        abi_step(dbg, d, inp, pg, num_splits=2, err=err)
        torch.cuda.synchronize()  # returns: every wait ended by its limit
        assert int(err.item()) == MLA_ERR_TIMEOUT
    finally:
        assert dbg.mla_debug_reset() == 0
    err.zero_()
    r = abi_step(dbg, d, inp, pg, num_splits=2, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.absorbed_f64(inp)
    T, H = inp.B * inp.n_q, inp.H
    assert_close(dev_bf16_to_f64(r["u"]).reshape(T * H, 512), ref["u"], "u")
    assert_close(dev_bf16_to_f64(r["out"]).reshape(T * H, 128), ref["out"], "out")
    assert np.isfinite(r["lse"].cpu().numpy()).all()


def test_fp8_wait_runs_out_then_context_recovers():
    """The same on the FP8 cache (its own rings of code and operand slots)."""
    import ctypes
    import math

    import torch

    import mla_latent_kv_paged_gb300 as mla
    dbg = mla.debug_lib()
    inp = mi.make_inputs(B=2, H=128, n_q=1, seq_lens=[300, 130], seed=98)
    pg = mi.make_paged(inp, spare_pages=2)
    pg8 = mi.make_paged_fp8(inp, pg)
    d = device_inputs(inp, pg)
    cache8 = torch.from_numpy(pg8.cache).cuda()
    scales = torch.from_numpy(pg8.scales).cuda()
    T, H, G = inp.B * inp.n_q, inp.H, 2
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None  # noqa: E731
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    q_abs = torch.empty((T, H, 576), dtype=torch.bfloat16, device="cuda")
    assert dbg.mla_absorb_q(p(d["q_nope"]), p(d["q_rope"]), p(d["w_uk"]), p(q_abs), T, H, 128, 64, 512, s) == 0
    ws = torch.empty(int(dbg.mla_decode_workspace_bytes(inp.B, 1, H, G)), dtype=torch.uint8, device="cuda")
    u = torch.empty((T, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def decode():
        st = dbg.mla_decode_paged_fp8(p(q_abs), p(cache8), p(scales), p(d["block_table"]), p(d["seq_lens"]),
                                      inp.B, 1, H, pg.num_pages, 64, pg.max_pages,
                                      ctypes.c_float(1.0 / math.sqrt(192.0)), G, p(ws), ws.numel(), p(err), s)
        assert st == 0
        assert dbg.mla_combine(p(ws), inp.B, 1, H, G, p(u), p(lse), s) == 0

    assert dbg.mla_debug_reset() == 0
    try:
        assert dbg.mla_debug_set_wait_limit(2_000_000) == 0
        assert dbg.mla_debug_set_skip_producer(1) == 0
        decode()
        torch.cuda.synchronize()
        assert int(err.item()) == MLA_ERR_TIMEOUT
    finally:
        assert dbg.mla_debug_reset() == 0
    err.zero_()
    decode()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    codes = mi.quantize_fp8(np.concatenate([inp.c, inp.kr], axis=1), pg8.scales)
    ref = oracle.absorbed_fp8_f64(inp, codes, pg8.scales)
    assert_close(dev_bf16_to_f64(u).reshape(T * H, 512), ref["u"], "u")
    assert_close(lse.double().cpu().numpy().reshape(-1), ref["lse"], "lse")
