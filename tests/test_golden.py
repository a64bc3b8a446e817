"""The seeded generator and the oracle reproduce the stored tiny-workload fixture."""
import json
import os

import numpy as np

from local_linear_attention_flashlla_gb300.inputs import workload, make_inputs
from oracle.lla_ref import lla_ref

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_fp32_fixture_reproduces():
    with open(os.path.join(HERE, "golden", "tiny_fp32_oracle.json")) as f:
        doc = json.load(f)
    w = workload("tiny_fp32")
    q, k, v = (t.double().numpy() for t in make_inputs(w))
    assert abs(q.sum() - doc["q_checksum"]) < 1e-9
    assert abs(k.sum() - doc["k_checksum"]) < 1e-9
    assert abs(v.sum() - doc["v_checksum"]) < 1e-9
    out, rho, den = lla_ref(q, k, v, w.tau, w.lam)
    assert np.abs(out - np.array(doc["out"])).max() < 1e-12
    assert np.abs(rho - np.array(doc["rho"])).max() < 1e-12
    assert np.abs(den - np.array(doc["denom"])).max() < 1e-12
