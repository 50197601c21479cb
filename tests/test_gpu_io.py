"""mla_copy16, the kernel copy of a step's host I/O (GPU only): bytes from pinned host
memory to the device and back, device to device, bit for bit; pageable host memory is
refused before any launch. Integer work: exact."""
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
