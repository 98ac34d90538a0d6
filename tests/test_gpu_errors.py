"""Host-side refusals with a GPU present: bad pointers, partial overlaps and
extents past an allocation return an error status and enqueue nothing (the
output buffer keeps its contents)."""
import ctypes

import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe

pytestmark = pytest.mark.gpu


def _stream():
    return torch.cuda.current_stream().cuda_stream


def test_host_pointer_is_refused():
    L = gbe.lib()
    host = np.ones(1024, np.float32)
    dev = torch.ones(1024, device="cuda")
    y = torch.full((1024,), 7.0, device="cuda")
    st = L.gbe_add(host.ctypes.data, dev.data_ptr(), y.data_ptr(), 1024, 0, _stream())
    assert st == 10
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


def _allocation_end(ptr: int) -> int:
    """End address of the driver allocation that holds `ptr` (torch's caching
    allocator hands out pieces of larger segments)."""
    cu = ctypes.CDLL("libcuda.so.1")
    base, size = ctypes.c_uint64(0), ctypes.c_size_t(0)
    assert cu.cuMemGetAddressRange_v2(ctypes.byref(base), ctypes.byref(size), ctypes.c_uint64(ptr)) == 0
    return base.value + size.value


def test_extent_past_allocation_is_refused():
    L = gbe.lib()
    out = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    torch.cuda.empty_cache()  # so x starts a fresh segment of its own
    x = torch.ones(1 << 20, device="cuda")
    end = _allocation_end(x.data_ptr())
    n_fit = (end - x.data_ptr()) // 4
    # one row reaching exactly to the end of the allocation is accepted ...
    assert L.gbe_argmax(x.data_ptr(), out.data_ptr(), 1, n_fit, 0, _stream()) == 0
    torch.cuda.synchronize()
    out.fill_(7)
    # ... one element more is refused and nothing runs: GBE_ERR_POINTER, or
    # GBE_ERR_ALIAS (checked first) when the output happens to sit right
    # after x's allocation, inside the extent asked for
    past = L.gbe_argmax(x.data_ptr(), out.data_ptr(), 1, n_fit + 1, 0, _stream())
    assert past == (8 if out.data_ptr() == end else 10)
    torch.cuda.synchronize()
    assert int(out.item()) == 7


def test_partial_overlap_is_refused():
    L = gbe.lib()
    buf = torch.ones(2048, device="cuda")
    w = torch.ones(64, device="cuda")
    x = buf[:1024]
    y = buf[512:1536]
    assert L.gbe_rmsnorm(x.data_ptr(), w.data_ptr(), y.data_ptr(), 16, 64, 1e-5, 0, _stream()) == 8
    # y overlapping the gain is refused too
    big = torch.ones(1024 + 64, device="cuda")
    assert L.gbe_rmsnorm(big[64:].data_ptr(), big.data_ptr(), big[:1024].data_ptr(), 16, 64, 1e-5, 0,
                         _stream()) == 8
    # exact aliases that the op allows are accepted
    assert L.gbe_rmsnorm(x.data_ptr(), w.data_ptr(), x.data_ptr(), 16, 64, 1e-5, 0, _stream()) == 0


def test_misaligned_and_null_pointers_are_refused():
    L = gbe.lib()
    a = torch.ones(100, device="cuda")
    base = a.data_ptr()
    assert L.gbe_add(base + 2, base, base, 10, 0, _stream()) == 9
    assert L.gbe_add(None, base, base, 10, 0, _stream()) == 1
    bf = torch.ones(100, dtype=torch.bfloat16, device="cuda")
    assert L.gbe_add(bf.data_ptr() + 1, bf.data_ptr(), bf.data_ptr(), 10, 1, _stream()) == 9


def test_binding_raises_with_status():
    x = torch.ones(4, 8, device="cuda")
    with pytest.raises(gbe.GbeError) as e:
        gbe.gbe_rmsnorm(x, torch.ones(8, device="cuda"), x, -1.0)
    assert e.value.status == 5
    with pytest.raises(gbe.GbeError) as e:
        gbe.argmax(torch.ones(3, 0, device="cuda"))
    assert e.value.status == 7
