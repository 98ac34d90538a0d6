"""Pinned host buffers passed straight to the C ABI: the kernels read and
write host memory in place (mapped at the same address on the device) and
give the same bits as with device buffers; unpinned host memory is refused."""
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
