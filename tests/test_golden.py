"""The oracle and the seeded generator still reproduce the stored tiny-workload fixture."""
import os

import numpy as np

import oracle
from gated_deltanet_linear_delta_gb300 import inputs

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load():
    rec = {"out": [], "state": []}
    with open(os.path.join(HERE, "tiny_fp32.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            if parts[0] in ("out_rms", "state_fro"):
                rec[parts[0]] = float(parts[1])
            else:
                rec[parts[0]].append((tuple(int(x) for x in parts[1:-1]), float(parts[-1])))
    return rec


def test_tiny_fp32_fixture():
    rec = _load()
    b = inputs.tiny_fp32(seed=0)
    for fn in (lambda: oracle.gdn_sequential(b.q, b.k, b.v, b.g, b.b, None, B=1),
               lambda: oracle.gdn_chunked(b.q, b.k, b.v, b.g, b.b, None, B=1, chunk=16)):
        out, st = fn()
        np.testing.assert_allclose(np.sqrt(np.mean(out ** 2)), rec["out_rms"], rtol=1e-12)
        np.testing.assert_allclose(np.linalg.norm(st), rec["state_fro"], rtol=1e-12)
        for idx, val in rec["out"]:
            np.testing.assert_allclose(out[idx], val, rtol=1e-10, atol=1e-13)
        for idx, val in rec["state"]:
            np.testing.assert_allclose(st[idx], val, rtol=1e-10, atol=1e-13)
