"""Host-side logic of bench.py (no GPU): the batch sweep's slicing and byte
counts, the extra inputs built only when asked for, and the per-op DRAM
traffic file and its lookup keyed by the kernels' source hashes."""
import numpy as np

import bench
from synth import workloads as W


def test_batch_sweep_slices_the_first_rows():
    data = bench.build_workload_inputs(W.WIDE)
    sweep = bench.batch_sweep(data)
    full_argmax, _ = bench.op_bytes("argmax", *data["argmax"])
    rows = data["argmax"][1]["rows"]
    bs = sorted(int(k.split("@")[1]) for k in sweep if k.startswith("argmax@"))
    assert bs[0] == 1 and bs[-1] == rows and all(b2 == 2 * b1 for b1, b2 in zip(bs[:-2], bs[1:-1]))
    for key, (arrays, params) in sweep.items():
        op, b = key.split("@")
        b = int(b)
        assert params["rows"] == b
        assert arrays["x"].shape[0] == b
        assert np.shares_memory(arrays["x"], data[op][0]["x"]), "a view of the first rows, not a copy"
        if op == "rmsnorm":
            assert arrays["w"] is data[op][0]["w"], "per-column weights are not sliced"
        nb, r = bench.op_bytes(op, arrays, params)
        assert r == b
    nb1024, _ = bench.op_bytes("argmax", *sweep[f"argmax@{rows}"])
    assert nb1024 == full_argmax


def test_extra_inputs_only_when_asked_for():
    few = bench.build_extra_inputs(64, ops=("layernorm", "rope_multi"))
    assert sorted(few) == ["layernorm", "rope_multi"]
    assert few["layernorm"][0]["x"].shape[0] == 64
    with_sampling = bench.build_extra_inputs(64, ops=("sample_top_p",))
    assert sorted(with_sampling) == ["sample_top_p"]
    assert with_sampling["sample_top_p"][0]["x"].shape == (64, 128256)


def test_dram_traffic_file_and_lookup():
    # profiles/dram_traffic.txt: one line per op of the step (bytes per
    # launch, the hash of the kernel sources it was taken on); the dominant
    # kernel (argmax over [8192, 128256] bf16, read once) within 1 % of its
    # algorithmic bytes.  The lookup gives that figure while the hash matches
    # the sources, and null once they have changed.
    import os
    path = os.path.join(os.path.dirname(bench.__file__), "profiles", "dram_traffic.txt")
    rows = {}
    for line in open(path):
        if line.strip() and not line.startswith("#"):
            op, nbytes, h = line.split()
            rows[op] = (int(nbytes), h)
    for op, _ in bench.STEP:
        assert op in rows and rows[op][0] > 0 and len(rows[op][1]) == 16, op
        got = bench.dram_traffic(op)
        assert got in (None, rows[op][0]), op
        assert (got is not None) == (rows[op][1] == bench.sources_hash(op)), op
    algorithmic = 8192 * 128256 * 2 + 8192 * 4
    assert abs(rows["argmax"][0] - algorithmic) <= 0.01 * algorithmic
