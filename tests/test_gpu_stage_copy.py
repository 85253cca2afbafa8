"""The staging copy (pkv_stage_copy): host -> device from a pinned buffer, device -> host
into one, and device -> device, byte for byte, at sizes from one 16-byte word to more than
a wave of threads, and in order with the kernels around it on the stream."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_17_gb300 as m

    return m


def _bytes(n, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g)


@pytest.mark.parametrize("n", [16, 4096, 873472, 536576, 16 * 152 * 1024 + 48])
def test_host_to_device_to_host(pkv, n):
    src = _bytes(n, n).pin_memory()
    dev = torch.full((n,), 7, dtype=torch.uint8, device="cuda")
    pkv.stage_copy(dev, src)
    back = torch.zeros(n, dtype=torch.uint8).pin_memory()
    pkv.stage_copy(back, dev)
    torch.cuda.synchronize()
    assert torch.equal(dev.cpu(), src)
    assert torch.equal(back, src)


def test_device_to_device_and_stream_order(pkv):
    """A torch kernel writes the source, the copy follows it, a torch kernel reads the copy:
    the copy sees the first and is seen by the second."""
    n = 1 << 20
    a = torch.empty(n // 4, dtype=torch.float32, device="cuda")
    b = torch.empty_like(a)
    for it in range(5):
        a.fill_(float(it + 1))
        pkv.stage_copy(b, a)
        s = float(b.sum())
        assert s == float(it + 1) * (n // 4)


def test_refusals(pkv):
    h = torch.zeros(64, dtype=torch.uint8)  # not pinned
    d = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        pkv.stage_copy(d, h)
    with pytest.raises(ValueError):
        pkv.stage_copy(d, torch.zeros(48, dtype=torch.uint8, device="cuda"))
    with pytest.raises(pkv.PkvError):
        pkv.stage_copy(d[:24], torch.zeros(24, dtype=torch.uint8, device="cuda"))


def test_ordinary_host_memory_is_refused(pkv):
    """Host memory that is not page-locked is refused on the host (no kernel runs)."""
    import ctypes

    import numpy as np

    host = np.zeros(4096, dtype=np.uint8)  # ordinary, unregistered host memory
    base = host.ctypes.data
    ptr = (base + 15) // 16 * 16
    d = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    st = pkv.lib.pkv_stage_copy(d.data_ptr(), ctypes.c_void_p(ptr), 1024, None)
    assert st == pkv.PKV_ERR_INVALID_ARG and "page-locked" in pkv.lib.pkv_last_error().decode()
    st = pkv.lib.pkv_stage_copy(ctypes.c_void_p(ptr), d.data_ptr(), 1024, None)
    assert st == pkv.PKV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert pkv.check_device_status() == 0

