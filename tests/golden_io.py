"""Reader of the text fixtures under tests/golden/ (values the pages print)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            parts = val.split()
            if key == "op":
                out[key] = val
            elif len(parts) == 1 and key in ("layout", "pos", "r", "index"):
                out[key] = int(parts[0])
            elif len(parts) == 1 and key in ("eps", "mu"):
                out[key] = float(parts[0])
            else:
                out[key] = np.array([float(p) for p in parts], dtype=np.float64)
    return out


def printed_close(got, printed, decimals: int) -> bool:
    """True when `got` (an f32 result) agrees with a value the page printed to
    `decimals` places: within one unit of the last printed place (the page
    rounds its own intermediate steps to that many places, so half a unit is
    not always enough) plus two f32 ulps of the value (the f32 steps round
    too)."""
    got = np.asarray(got, dtype=np.float64)
    tol = 10.0 ** (-decimals) + 2.0 * 2.0 ** -23 * np.abs(printed)
    return bool(np.all(np.abs(got - printed) <= tol))
