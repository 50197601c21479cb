"""A step's host I/O (GPU only). mla_copy16, the kernel copy: bytes from pinned host
memory to the device and back, device to device, bit for bit; pageable host memory is
refused before any launch. Integer work: exact. mla_out_proj and mla_combine writing
their outputs into pinned host memory: the bits they write into device memory."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mla():
    import mla_latent_kv_paged_gb300 as m
    m.build()
    return m


@pytest.mark.parametrize("nbytes", [16, 4096 + 48, 1_581_184, 10 * 1024 * 1024 + 16 * 7])
def test_round_trip_through_pinned_host_memory(mla, nbytes):
    import torch
    rng = np.random.default_rng(nbytes)
    data = torch.from_numpy(rng.integers(0, 256, size=nbytes, dtype=np.uint8))
    host_in = data.clone().pin_memory()
    dev = torch.full((nbytes,), 7, dtype=torch.uint8, device="cuda")
    mla.copy16(host_in, dev)
    dev2 = torch.empty_like(dev)
    mla.copy16(dev, dev2)
    host_out = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    mla.copy16(dev2, host_out)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), data)
    assert torch.equal(host_out, data)


def test_offset_inside_a_pinned_allocation(mla):
    """A view that starts inside a pinned allocation maps to the same offset on the device."""
    import torch
    base = torch.arange(4096, dtype=torch.int32).pin_memory()
    dev = torch.zeros(1024, dtype=torch.int32, device="cuda")
    mla.copy16(base[512:1536], dev)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), torch.arange(512, 1536, dtype=torch.int32))


def test_pageable_host_memory_is_refused(mla):
    import torch
    pageable = torch.zeros(4096, dtype=torch.uint8)
    dev = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    with pytest.raises(mla.MlaError):
        mla.copy16(pageable, dev)


def _proj_inputs(T, H, seed):
    import torch
    g = torch.Generator().manual_seed(seed)
    u = (torch.randn((T, H, 512), generator=g) * 0.5).to(torch.bfloat16).cuda()
    w_uv = (torch.randn((H, 128, 512), generator=g) / 512 ** 0.5).to(torch.bfloat16).cuda()
    return u, w_uv


@pytest.mark.parametrize("T", [1, 32, 77])
def test_out_proj_writes_pinned_host_memory(mla, T):
    """out in pinned host memory (a view at an offset inside its allocation): the bits
    out_proj writes into device memory."""
    import torch
    H = 128
    u, w_uv = _proj_inputs(T, H, 500 + T)
    dev_out = mla.out_proj(u, w_uv)
    pinned = torch.full((T * H * 128 + 64,), -1, dtype=torch.int16).pin_memory()
    host_out = pinned[64:].view(torch.bfloat16).view(T, H, 128)
    mla.out_proj(u, w_uv, host_out)
    torch.cuda.synchronize()
    assert torch.equal(host_out.view(torch.int16), dev_out.cpu().view(torch.int16))
    assert torch.equal(pinned[:64], torch.full((64,), -1, dtype=torch.int16))


def test_out_proj_refuses_pageable_host_memory(mla):
    import torch
    u, w_uv = _proj_inputs(4, 8, 7)
    with pytest.raises(mla.MlaError):
        mla.out_proj(u, w_uv, torch.zeros((4, 8, 128), dtype=torch.bfloat16))


def test_combine_writes_lse_into_pinned_host_memory(mla):
    import torch
    import mla_inputs as mi
    from tests.helpers import device_inputs
    inp = mi.make_inputs(B=3, H=128, n_q=2, seq_lens=[70, 300, 129], seed=83)
    pg = mi.make_paged(inp, spare_pages=4)
    d = device_inputs(inp, pg)
    q_abs = mla.absorb_q(d["q_nope"], d["q_rope"], d["w_uk"])
    ws, g = mla.decode_paged(q_abs, d["cache"], d["block_table"], d["seq_lens"], n_q=2, num_splits=5)
    u_dev, lse_dev = mla.combine(ws, B=3, n_q=2, H=128, num_splits=g)
    lse_host = torch.zeros((6, 128), dtype=torch.float32).pin_memory()
    u2, _ = mla.combine(ws, B=3, n_q=2, H=128, num_splits=g, lse=lse_host)
    torch.cuda.synchronize()
    assert torch.equal(lse_host.view(torch.int32), lse_dev.cpu().view(torch.int32))
    assert torch.equal(u2.view(torch.int16), u_dev.view(torch.int16))
    with pytest.raises(mla.MlaError):
        mla.combine(ws, B=3, n_q=2, H=128, num_splits=g, lse=torch.zeros((6, 128), dtype=torch.float32))
