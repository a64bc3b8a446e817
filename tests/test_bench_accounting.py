"""bench.py's accounting, on CPU: the FLOP and byte counts the roofline divides, and the committed
DRAM traffic it reports.

* useful forward FLOPs = (4 + 3T) passes x 2d per causal pair, the formula the workload's metric
  is quoted with; the tensor path executes 7 + 3T passes (the max sweep, the output sweep's rho.k
  and the product of rho's fp16 remainder), the fp32 path 6 + 3T;
* a causal pair count of n(n+1)/2 per (b, h), checked by brute force on a tiny n;
* decode method bytes = K in each of the T + 2 passes plus V once, plus q and the outputs;
* the committed traffic is returned only for the exact kernel sources it was captured on, and
  scales with the batch (independent slices); any other shape change gives none.
"""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from local_linear_attention_flashlla_gb300.inputs import workload  # noqa: E402


def test_causal_pair_count_by_brute_force():
    w = workload("lm_bf16", B=2, H=3, n=7, d=16)
    pairs = sum(1 for _ in range(w.B * w.H) for i in range(w.n) for j in range(i + 1))
    assert bench.useful_flops(w, 0) == 4 * 2 * w.d * pairs


@pytest.mark.parametrize("T", [0, 1, 16])
def test_forward_flop_formulas(T):
    w = workload("lm_bf16")
    pairs = w.n * (w.n + 1) / 2 * w.B * w.H
    assert bench.useful_flops(w, T) == (4 + 3 * T) * 2 * w.d * pairs
    assert bench.executed_flops(w, T, 1) == (7 + 3 * T) * 2 * w.d * pairs      # tensor path
    assert bench.executed_flops(w, T, 2) == (6 + 3 * T) * 2 * w.d * pairs      # fp32 path


def test_lm_workload_useful_flops_per_call():
    # 8 x 16 heads, n = 4096, d = 128, T = 16: 52 passes x 256 flops x 8 390 656 pairs x 128 heads
    w = workload("lm_bf16")
    assert bench.useful_flops(w, 16) == pytest.approx(1.430e13, rel=1e-3)


def test_decode_bytes():
    w = workload("decode_bf16")
    T = w.cg_max_iters
    comp, method = bench.decode_bytes(w, T, moment=False)
    kv = w.B * w.H * w.n * w.d * 2
    assert method >= (T + 2) * kv + kv
    assert comp >= 2 * kv and comp < method
    # the moment form reads K twice and V once
    comp_m, method_m = bench.decode_bytes(w, T, moment=True)
    assert comp_m == comp and method_m == comp + kv
    assert comp - 2 * kv == w.B * w.H * (w.d * (2 + 2 + 4) + 4)


def test_decode_form_accounting_follows_the_auto_rule():
    lim = 52952
    w = workload("decode_bf16")
    assert bench.decode_uses_moment_form(w, "auto", lim)                       # n = 4096
    assert not bench.decode_uses_moment_form(w.with_(n=32768), "auto", lim)   # a CUDA-core form
    assert bench.decode_uses_moment_form(w.with_(n=60000), "auto", lim)       # past their limit
    assert not bench.decode_uses_moment_form(w.with_(dtype="fp32"), "auto", lim)
    assert not bench.decode_uses_moment_form(w.with_(d=64), "auto", lim)
    assert bench.decode_uses_moment_form(w.with_(n=32768), "moment", lim)
    assert not bench.decode_uses_moment_form(w, "stream", lim)


def test_traffic_is_tied_to_the_sources_and_scales_with_the_batch(tmp_path, monkeypatch):
    w = workload("lm_bf16")
    doc = {"lla_tc_kernel:lm_bf16": {"source_hash": bench.kernel_source_hash("lla_tc_kernel"),
                                     "dram_bytes_per_launch": 800}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(doc))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the sources are read from the real tree, the summary from the temporary one
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: doc["lla_tc_kernel:lm_bf16"]["source_hash"])
    assert bench.load_traffic("lla_tc_kernel", w) == 800
    assert bench.load_traffic("lla_tc_kernel", w.with_(B=2)) == 200
    assert bench.load_traffic("lla_tc_kernel", w.with_(n=2048)) is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "0" * 16)
    assert bench.load_traffic("lla_tc_kernel", w) is None


def test_tolerance_mode_flops_by_brute_force():
    """Tolerance mode: each query tile runs as many CG sweeps as its slowest query; the useful
    count sums (4 + 3 T_t) passes of 2d over each tile's causal pairs, checked pair by pair on a
    ragged shape for both tile sizes."""
    import numpy as np
    w = workload("lm_bf16", B=2, H=2, n=75, d=16)
    rng = np.random.default_rng(3)
    its = rng.integers(0, 9, size=(w.B, w.H, w.n))
    for path, rows in ((1, 128), (2, 32)):
        useful = executed = 0
        for b in range(w.B):
            for h in range(w.H):
                for i in range(w.n):
                    t = i // rows
                    T = its[b, h, t * rows:(t + 1) * rows].max()
                    a = 8 if path == 1 else 6
                    bb = 5 if path == 1 else 3
                    useful += (4 + 3 * T) * 2 * w.d * (i + 1)
                    executed += (a + bb * T) * 2 * w.d * (i + 1)
        u, e, t_mean, t_pw = bench.tolerance_flops(w, its, path, precise=True)
        assert u == useful and e == executed
        T_tile, pairs = bench.tile_iterations(its, rows)
        assert t_mean == T_tile.mean() and pairs.sum() == w.n * (w.n + 1) / 2
        # a uniform count reduces to the fixed-cap formula
        u1, _, _, t1 = bench.tolerance_flops(w, np.full_like(its, 5), path, precise=True)
        assert u1 == bench.useful_flops(w, 5) and t1 == 5.0


def test_iteration_histogram_counts_every_query():
    import numpy as np
    its = np.array([[[0, 3, 3, 64]]])
    assert bench.iteration_histogram(its) == {"0": 1, "3": 2, "64": 1}
