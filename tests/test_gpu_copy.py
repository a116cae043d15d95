"""qspec_copy on the GPU: pinned host to device, device to pinned host, device to device, offsets
inside a pinned allocation, ordering after the kernel that writes its source, and the refusal of
pageable host memory."""
import pytest
import torch

from gpu_util import DEV, lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return lib()


def _bytes(n, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g)


@pytest.mark.parametrize("n", [16, 4096, 57344 + 16, 1796864])
def test_host_to_device_and_back(q, n):
    src = _bytes(n, n).pin_memory()
    dev = torch.zeros(n, dtype=torch.uint8, device=DEV)
    q.qspec_copy(dev, src)
    back = torch.zeros(n, dtype=torch.uint8).pin_memory()
    q.qspec_copy(back, dev)
    q.qspec_check_status()
    assert torch.equal(dev.cpu(), src)
    assert torch.equal(back, src)


def test_device_to_device_and_views(q):
    a = _bytes(1 << 20, 3).to(DEV)
    b = torch.zeros_like(a)
    q.qspec_copy(b, a)
    # a view 48 bytes into a pinned allocation, and a view into a device buffer
    host = _bytes(8192, 4).pin_memory()
    d2 = torch.zeros(8192, dtype=torch.uint8, device=DEV)
    q.qspec_copy(d2[256:256 + 4096], host[48:48 + 4096])
    q.qspec_check_status()
    assert torch.equal(b, a)
    assert torch.equal(d2[256:256 + 4096].cpu(), host[48:48 + 4096])
    assert int(d2[:256].sum()) == 0 and int(d2[256 + 4096:].sum()) == 0


def test_reads_device_source_after_the_writer(q):
    # the source is written by the kernel just before in the stream; the copy reads it only after
    # that kernel has finished
    for i in range(20):
        x = torch.empty(1 << 16, dtype=torch.int32, device=DEV)
        x.fill_(i + 1)
        out = torch.zeros(1 << 16, dtype=torch.int32).pin_memory()
        q.qspec_copy(out, x)
        q.qspec_check_status()
        assert bool((out == i + 1).all())


def test_pageable_host_memory_is_refused(q):
    src = _bytes(4096, 5)  # not pinned
    dev = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    with pytest.raises(ValueError):
        q.qspec_copy(dev, src)  # the binding refuses it
    with pytest.raises(q.QSpecError) as e:  # and so does the library itself
        q._check("qspec_copy", q.load().qspec_copy(dev.data_ptr(), src.data_ptr(), 4096, None))
    assert q.STATUS[e.value.code] == "QSPEC_ERR_INVALID_ARG"
