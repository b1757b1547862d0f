"""Write the golden fixtures under tests/golden/ from the fp64 oracle.

The pages print no worked example of the gated delta rule, so these fixtures
are not the pages' numbers: they are the oracle's own results on the seeded
tiny fp32 workload (B=1, T=64, Hk=Hv=2, dk=dv=32, chunk 16, seed 0), kept to
catch any later drift of the oracle or of the input generator. They are
written by this script only, which calls nothing but ``oracle`` and the seeded
input generator.

    python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from gated_deltanet_linear_delta_gb300 import inputs  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def sample_index(shape, n, seed):
    r = np.random.default_rng(seed)
    return [tuple(int(r.integers(0, s)) for s in shape) for _ in range(n)]


def main():
    b = inputs.tiny_fp32(seed=0)
    out, st = oracle.gdn_sequential(b.q, b.k, b.v, b.g, b.b, None, B=1)
    lines = ["# tiny fp32 workload: B=1 T=64 Hk=Hv=2 dk=dv=32 chunk=16 seed=0, zero initial state",
             "# written by tests/golden/make_golden.py from the fp64 oracle (token scan)",
             f"out_rms {np.sqrt(np.mean(out ** 2)):.17e}",
             f"state_fro {np.linalg.norm(st):.17e}"]
    for idx in sample_index(out.shape, 24, 1):
        lines.append("out " + " ".join(map(str, idx)) + f" {out[idx]:.17e}")
    for idx in sample_index(st.shape, 24, 2):
        lines.append("state " + " ".join(map(str, idx)) + f" {st[idx]:.17e}")
    with open(os.path.join(HERE, "tiny_fp32.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
