"""The parity report: for every op of every workload, at full size, the
largest observed error of the CUDA path against the oracle as a fraction of
its bar (a ratio <= 1 passes), and for the exact ops the count of
differing results (0 passes).

Bars (as in gpu_util): RMSNorm y, SiLU-mul and add+RMSNorm y:
|y - y_oracle| <= rtol |y_oracle| + 1e-30; RoPE: per pair
|y - y_oracle| <= rtol mu |(a, b)|; rtol 1e-5 (f32) / 1e-2 (bf16).  Exact:
argmax, embedding, add, the h of add+RMSNorm (against the oracle's
storage rounding).

The test prints one JSON line (seen with -s) and asserts every ratio."""
import json

import numpy as np
import pytest
import torch

import elementwise_row_rmsnorm_gb300 as gbe
import oracle
from gpu_util import RTOL, bits, to_dev, to_f32, widen
from synth import workloads as W

pytestmark = pytest.mark.gpu


def _rel_ratio(got, want, dtype):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    fin = np.isfinite(want)
    if not fin.any():
        return 0.0
    return float(np.max(np.abs(got[fin] - want[fin]) / (RTOL[dtype] * np.abs(want[fin]) + 1e-30)))


def _rope_ratio(got, want, x, r, mu, layout, dtype):
    got, want, x = (np.asarray(a, np.float64) for a in (got, want, x))
    i = np.arange(r // 2)
    ia, ib = (i, i + r // 2) if layout == 0 else (2 * i, 2 * i + 1)
    tol = RTOL[dtype] * abs(mu) * np.hypot(x[..., ia], x[..., ib]) + 1e-30
    return float(max(np.max(np.abs(got[..., ia] - want[..., ia]) / tol),
                     np.max(np.abs(got[..., ib] - want[..., ib]) / tol)))


def _exact(got_bits, want_f32, dtype):
    want = oracle.get().bf16_round(want_f32) if dtype == "bf16" else want_f32.view(np.uint32)
    return int(np.count_nonzero(got_bits != want))


def _report(workload):
    o = oracle.get()
    res = {}
    for name, build in W.cases(workload).items():
        a, p = build()
        dt = p.get("dtype", "f32")
        if name == "rmsnorm":
            y = gbe.rmsnorm(to_dev(a["x"]), to_dev(a["w"]), p["eps"])
            res[name] = _rel_ratio(to_f32(y), o.rmsnorm(widen(a["x"]), widen(a["w"]), p["eps"]), dt)
        elif name == "add_rmsnorm":
            y, h = gbe.add_rmsnorm(to_dev(a["x"]), to_dev(a["residual"]), to_dev(a["w"]), p["eps"])
            yo, ho = o.add_rmsnorm(widen(a["x"]), widen(a["residual"]), widen(a["w"]), p["eps"],
                                   h_bf16=(dt == "bf16"))
            res[name] = _rel_ratio(to_f32(y), yo, dt)
            res[name + ".h_mismatches"] = _exact(bits(h), ho, dt)
        elif name.startswith("rope"):
            xd = to_dev(a["x"])
            pos, om = to_dev(a["pos"]), to_dev(a["inv_freq"])
            y = gbe.rope(xd, pos, om, p["r"], p["mu"], p["layout"], in_place=p.get("in_place", False))
            want = o.rope(widen(a["x"]), a["pos"], a["inv_freq"], p["r"], p["mu"], p["layout"])
            res[name] = _rope_ratio(to_f32(y), want, widen(a["x"]), p["r"], p["mu"], p["layout"], dt)
        elif name == "silu_mul":
            y = gbe.silu_mul(to_dev(a["gate"]), to_dev(a["up"]))
            res[name] = _rel_ratio(to_f32(y), o.silu_mul(widen(a["gate"]), widen(a["up"])), dt)
        elif name == "embedding":
            out = gbe.embedding(to_dev(a["table"]), to_dev(a["ids"]))
            res[name + "_mismatches"] = _exact(bits(out), o.embedding(widen(a["table"]), a["ids"]), dt)
        elif name == "add":
            y = gbe.add(to_dev(a["a"]), to_dev(a["b"]))
            res[name + "_mismatches"] = _exact(bits(y), o.add(widen(a["a"]), widen(a["b"])), dt)
        elif name == "argmax":
            got = gbe.argmax(to_dev(a["x"])).cpu().numpy()
            res[name + "_mismatches"] = int(np.count_nonzero(got != o.argmax(widen(a["x"]))))
        del a
        torch.cuda.empty_cache()
    return res


@pytest.mark.parametrize("workload", W.ALL)
def test_parity_report(workload):
    res = _report(workload)
    print(json.dumps({"workload": workload, **{k: round(v, 4) if isinstance(v, float) else v
                                               for k, v in res.items()}}))
    for k, v in res.items():
        if k.endswith("mismatches"):
            assert v == 0, (workload, k, v)
        else:
            assert v <= 1.0, (workload, k, v)
