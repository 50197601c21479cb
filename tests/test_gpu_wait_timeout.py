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
