"""The ops inside CUDA graphs and on side streams, as a decode loop runs
them: a chain captured once (the host checks run at capture) and replayed
gives the eager chain's bits, replays read the buffers' current contents,
and calls on a non-default stream order correctly against that stream."""
import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe
from gpu_util import bits
from synth import normal, randint, to_bf16, units
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _decode_inputs(seed):
    T, d, ffn, V = 64, 4096, 14336, 128256
    dev = "cuda"
    t = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    x = t(to_bf16(normal(seed, "g.x", (T, d), 0.0, 1.0)))
    res = t(to_bf16(normal(seed, "g.r", (T, d), 0.0, 1.0)))
    w = t(to_bf16(normal(seed, "g.w", (d,), 1.0, 0.1)))
    q = t(to_bf16(normal(seed, "g.q", (T, 32, 128), 0.0, 1.0)))
    k = t(to_bf16(normal(seed, "g.k", (T, 8, 128), 0.0, 1.0)))
    pos = torch.from_numpy(randint(seed, "g.pos", (T,), 0, 8192)).to(dev)
    om = torch.from_numpy(W.inv_freq(500000.0, 128, 64)).to(dev)
    gate = t(to_bf16(normal(seed, "g.gate", (T, ffn), 0.0, 2.0)))
    up = t(to_bf16(normal(seed, "g.up", (T, ffn), 0.0, 2.0)))
    logits = t(to_bf16(normal(seed, "g.l", (T, V), 0.0, 4.0)))
    u = torch.from_numpy(units(seed, "g.u", T).astype(np.float32)).to(dev)
    return dict(x=x, res=res, w=w, q=q, k=k, pos=pos, om=om, gate=gate, up=up, logits=logits, u=u)


def _chain(b, o):
    gbe.gbe_add_rmsnorm(b["x"], b["res"], b["w"], o["y"], o["h"], 1e-5)
    gbe.gbe_rope_qk(b["q"], o["q"], b["k"], o["k"], b["pos"], b["om"], 128, 1.0, 0)
    gbe.gbe_silu_mul(b["gate"], b["up"], o["s"])
    gbe.gbe_argmax(b["logits"], o["am"])
    gbe.gbe_sample(b["logits"], b["u"], o["tp"], "top_p", temperature=0.7, p=0.9)
    gbe.gbe_sample(b["logits"], b["u"], o["tk"], "top_k", temperature=0.7, top_k=50)


def _outputs(b):
    T = b["x"].shape[0]
    return dict(y=torch.empty_like(b["x"]), h=torch.empty_like(b["x"]), q=torch.empty_like(b["q"]),
                k=torch.empty_like(b["k"]), s=torch.empty_like(b["gate"]),
                am=torch.empty(T, dtype=torch.int32, device="cuda"),
                tp=torch.empty(T, dtype=torch.int32, device="cuda"),
                tk=torch.empty(T, dtype=torch.int32, device="cuda"))


def _snapshot(o):
    return {k: bits(v).copy() for k, v in o.items()}


def test_graph_replay_equals_eager():
    b = _decode_inputs(41)
    eager = _outputs(b)
    _chain(b, eager)
    torch.cuda.synchronize()
    want = _snapshot(eager)

    o = _outputs(b)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _chain(b, o)  # warm-up on the capture stream
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        _chain(b, o)
    for v in o.values():
        v.zero_()
    g.replay()
    torch.cuda.synchronize()
    got = _snapshot(o)
    for name in want:
        assert np.array_equal(got[name], want[name]), name

    # a replay reads the inputs' current contents
    b2 = _decode_inputs(42)
    for key in b:
        b[key].copy_(b2[key])
    g.replay()
    torch.cuda.synchronize()
    eager2 = _outputs(b2)
    _chain(b2, eager2)
    torch.cuda.synchronize()
    for name, v in _snapshot(eager2).items():
        assert np.array_equal(_snapshot(o)[name], v), name


def test_side_stream_orders_after_its_producer():
    """A producer and the op on one side stream: the op sees the producer's
    data (stream order), not the buffer's old contents."""
    b = _decode_inputs(43)
    side = torch.cuda.Stream()
    x = torch.zeros_like(b["x"])
    y = torch.empty_like(x)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        torch.cuda._sleep(1_000_000)  # keep the stream busy so a misordered op would read zeros
        x.copy_(b["x"])
        gbe.gbe_rmsnorm(x, b["w"], y, 1e-5)
    torch.cuda.synchronize()
    want = gbe.rmsnorm(b["x"], b["w"], 1e-5)
    assert np.array_equal(bits(y), bits(want))
