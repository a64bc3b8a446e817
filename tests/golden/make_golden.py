"""Writes tests/golden/tiny_fp32_oracle.json: the float64 oracle's exact-solve output
for every row of the tiny fp32 workload (B=1, H=1, n=64, d=16, seed 0).

Calls only the oracle and the seeded input generator.  The stored values guard the
generator and the oracle against silent drift (platform, numpy version); they are
not used as expected values for the CUDA path, which is always compared with the
oracle run in the same process.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from local_linear_attention_flashlla_gb300.inputs import workload, make_inputs  # noqa: E402
from oracle.lla_ref import lla_ref  # noqa: E402


def main():
    w = workload("tiny_fp32")
    q, k, v = (t.double().numpy() for t in make_inputs(w))
    out, rho, den = lla_ref(q, k, v, w.tau, w.lam)
    doc = {"workload": "tiny_fp32", "tau": w.tau, "lambda": w.lam,
           "q_checksum": float(q.sum()), "k_checksum": float(k.sum()), "v_checksum": float(v.sum()),
           "out": out.tolist(), "rho": rho.tolist(), "denom": den.tolist()}
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_fp32_oracle.json"), "w") as f:
        json.dump(doc, f)


if __name__ == "__main__":
    main()
