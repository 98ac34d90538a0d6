"""Pinned host buffers passed straight to the C ABI: the kernels read and
write host memory in place (mapped at the same address on the device) and
give the same bits as with device buffers; unpinned host memory is refused."""
import ctypes

import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe
from synth import normal, randint, to_bf16, uniform

pytestmark = pytest.mark.gpu


def _pin(t):
    return t.cpu().pin_memory()


def test_ops_on_pinned_host_buffers_match_device():
    x = torch.from_numpy(to_bf16(normal(5, "zc.x", (64, 4096), 0.0, 1.0)).view(np.int16)).view(torch.bfloat16)
    r = torch.from_numpy(to_bf16(normal(5, "zc.r", (64, 4096), 0.0, 1.0)).view(np.int16)).view(torch.bfloat16)
    w = torch.from_numpy(to_bf16(uniform(5, "zc.w", (4096,), 0.5, 1.5)).view(np.int16)).view(torch.bfloat16)
    xd, rd, wd = x.cuda(), r.cuda(), w.cuda()
    y_dev, h_dev = gbe.add_rmsnorm(xd, rd, wd, 1e-5)
    xh, rh = _pin(x), _pin(r)
    yh, hh = torch.empty_like(xh).pin_memory(), torch.empty_like(xh).pin_memory()
    gbe.gbe_add_rmsnorm(xh, rh, wd, yh, hh, 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(yh.view(torch.int16), y_dev.cpu().view(torch.int16))
    assert torch.equal(hh.view(torch.int16), h_dev.cpu().view(torch.int16))
    # silu-mul, argmax and rope with host inputs and outputs
    g = _pin(x)
    ys = torch.empty_like(g).pin_memory()
    gbe.gbe_silu_mul(g, rh, ys)
    am = torch.empty(64, dtype=torch.int32).pin_memory()
    gbe.gbe_argmax(xh, am)
    q = _pin(x.view(64, 32, 128))
    qo = torch.empty_like(q).pin_memory()
    pos = _pin(torch.from_numpy(randint(5, "zc.pos", (64,), 0, 8192)))
    om = (500000.0 ** (-2.0 * torch.arange(64, dtype=torch.float64) / 128)).float().cuda()
    gbe.gbe_rope(q, qo, pos, om, 128, 1.0, 0)
    torch.cuda.synchronize()
    assert torch.equal(ys.view(torch.int16), gbe.silu_mul(xd, rd).cpu().view(torch.int16))
    assert torch.equal(am, gbe.argmax(xd).cpu())
    assert torch.equal(qo.view(torch.int16),
                       gbe.rope(xd.view(64, 32, 128), pos.cuda(), om, 128).cpu().view(torch.int16))


def test_unpinned_host_memory_is_refused():
    L = gbe.lib()
    a = torch.ones(1000)  # pageable host memory
    y = torch.zeros(1000, device="cuda")
    st = L.gbe_add(a.data_ptr(), y.data_ptr(), y.data_ptr(), 1000, 0, torch.cuda.current_stream().cuda_stream)
    assert st == 10
    with pytest.raises(ValueError):
        gbe.gbe_add(a, y, y)


def _pinned_allocation_end(ptr: int) -> int:
    """End address of the pinned host allocation that holds `ptr` (torch's
    pinned allocator rounds blocks up, so a tensor may end before it)."""
    cu = ctypes.CDLL("libcuda.so.1")
    start, size = ctypes.c_uint64(0), ctypes.c_size_t(0)
    assert cu.cuPointerGetAttribute(ctypes.byref(start), 11, ctypes.c_uint64(ptr)) == 0  # RANGE_START_ADDR
    assert cu.cuPointerGetAttribute(ctypes.byref(size), 12, ctypes.c_uint64(ptr)) == 0   # RANGE_SIZE
    return start.value + size.value


def test_pinned_extent_past_allocation_is_refused():
    """Pinned host memory is held to the end of its allocation like device
    memory: a row reaching exactly to the end is accepted, one element more
    is refused on the host and nothing runs (the output keeps its value)."""
    L = gbe.lib()
    s = torch.cuda.current_stream().cuda_stream
    h = torch.ones(1024, dtype=torch.float32).pin_memory()
    out = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    n_fit = (_pinned_allocation_end(h.data_ptr()) - h.data_ptr()) // 4
    assert 1024 <= n_fit < (1 << 31)
    assert L.gbe_argmax(h.data_ptr(), out.data_ptr(), 1, n_fit, 0, s) == 0
    torch.cuda.synchronize()
    out.fill_(7)
    assert L.gbe_argmax(h.data_ptr(), out.data_ptr(), 1, n_fit + 1, 0, s) == 10
    torch.cuda.synchronize()
    assert int(out.item()) == 7
