"""Benchmark of the causal LLA forward pass (one JSON line on stdout, rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--op lla|parallax|decode|backward] [--workload lm_bf16] [--batch B]
                    [--path auto|tensor|fp32] [--no-cpu-baseline] [--no-e2e]

A step is one lla_forward call over the whole workload (all heads, all queries):
max sweep, moment sweep, CG sweeps and output sweep.  Inputs are seeded synthetic
tensors already resident in HBM; L2 is flushed (a 512 MiB write) before every timed
step, outside the timed interval.  Timing uses CUDA events on the launching stream.

N > 1 (torchrun): every rank runs the same workload on its own GPU with its own seed
(weak scaling; heads are independent, there is no collective on the data path);
value = tokens of all ranks / max over ranks of the timed seconds.

--impl reference times the float64 CPU oracle (the only reference this project has)
on a bounded sample of the workload's rows on rank 0 and extrapolates to the workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal LLA fwd tokens/s & TFLOP/s at d=128 bf16; fraction of BF16 tensor peak"
METRIC_DECODE = "LLA decode step tokens/s (one token per sequence) and HBM GB/s at d=128 bf16; fraction of HBM peak"
METRIC_PARALLAX = "causal Parallax-form fwd (caller probe) tokens/s & TFLOP/s at d=128 bf16; fraction of BF16 tensor peak"
METRIC_BACKWARD = "causal LLA backward (dq, dk, dv) tokens/s & TFLOP/s at d=128, bf16 inputs; fraction of BF16 tensor peak"


def useful_flops(w, T):
    """(2 + 3T + 2) causal GEMM passes of 2d flops per pair (moment, CG, output)."""
    pairs = w.n * (w.n + 1) / 2 * w.B * w.H
    return (4 + 3 * T) * 2 * w.d * pairs


def executed_flops(w, T, path):
    """Adds the logits-only max sweep and the output sweep's rho.k product; on the tensor path
    (path 1) also the product of rho's fp16 remainder (R_lo) in the output sweep."""
    pairs = w.n * (w.n + 1) / 2 * w.B * w.H
    return ((7 if path == 1 else 6) + 3 * T) * 2 * w.d * pairs


# query rows per tile of each path (tensor path 1, fp32 path 2): a tile runs CG sweeps until its
# last query stops, so in tolerance mode the work follows each tile's largest iteration count
TILE_ROWS = {1: 128, 2: 32}


def tile_iterations(its, tile_rows):
    """Per query tile: the iterations it executed (the most any of its queries ran), and its causal
    pair count.  its: int array [B, H, n].  Returns (T_tile [B, H, nt], pairs [nt])."""
    import numpy as np
    B, H, n = its.shape
    nt = (n + tile_rows - 1) // tile_rows
    pad = np.zeros((B, H, nt * tile_rows), dtype=np.int64)
    pad[:, :, :n] = its
    T_tile = pad.reshape(B, H, nt, tile_rows).max(axis=-1)
    i1 = np.arange(1, nt * tile_rows + 1, dtype=np.float64)
    i1[n:] = 0.0
    pairs = i1.reshape(nt, tile_rows).sum(axis=-1)
    return T_tile, pairs


def tolerance_flops(w, its, path, precise):
    """Tolerance mode: useful FLOPs sum (4 + 3 T_t) passes of 2d over each tile t's causal pairs,
    T_t the iterations tile t executed; executed FLOPs add the max sweep and the output sweep's
    rho.k product (fp32 path: 6 + 3 T_t), the tensor path's R_lo product (7 + 3 T_t), and in its
    precise form the hi + lo halves of the moment and CG coefficients and of the CG direction
    (8 + 5 T_t).  Returns (useful, executed, T tile mean, T pair-weighted mean)."""
    import numpy as np
    T_tile, pairs = tile_iterations(its, TILE_ROWS[path])
    p = np.broadcast_to(pairs, T_tile.shape)
    useful = float(((4 + 3 * T_tile) * p).sum()) * 2 * w.d
    a, b = (8, 5) if (path == 1 and precise) else ((7, 3) if path == 1 else (6, 3))
    executed = float(((a + b * T_tile) * p).sum()) * 2 * w.d
    return useful, executed, float(T_tile.mean()), float((T_tile * p).sum() / p.sum())


def iteration_histogram(its):
    """Per-query CG iteration counts as {iterations: queries}, nonzero bins only."""
    import numpy as np
    h = np.bincount(np.asarray(its).ravel())
    return {str(k): int(c) for k, c in enumerate(h) if c}


def parallax_useful_flops(w):
    """Parallax form: q.k, the weighted key mean, probe.k and the value product: 4 passes of 2d."""
    return 4 * 2 * w.d * (w.n * (w.n + 1) / 2 * w.B * w.H)


def parallax_executed_flops(w, tensor):
    """Adds the max sweep's q.k, the recomputed q.k of the moment and output sweeps and, on the
    tensor path, the probe's lo-part product."""
    return (7 if tensor else 6) * 2 * w.d * (w.n * (w.n + 1) / 2 * w.B * w.H)


def backward_useful_flops(w, T):
    """(11 + 2T) causal passes of 2d flops per pair: q.k, g.v, the two moment sums, T CG
    iterations of (p.k, accumulate), rho'.k and y.k, and the dq, dk (three terms) and dv sums."""
    return (11 + 2 * T) * 2 * w.d * (w.n * (w.n + 1) / 2 * w.B * w.H)


def backward_executed_flops(w, T, tensor=False):
    """As the kernels run them, in passes of 2d flops per causal pair.  fp32 path: the stats kernel
    (q.k in the max sweep, q.k, g.v and the two moment sums, 3 per CG iteration: 5 + 3T), the dq
    kernel (q.k, rho'.k, y.k, g.v, dq: 5) and the key-major kernel (the same four dots, dk's three
    terms, dv: 8).  Tensor path: the stats kernel (S in the max sweep; S, H and the hi + lo weight
    products in the moment and TBAR sweeps; S, the hi + lo direction and coefficient products per
    CG iteration: 9 + 5T), the dq kernel (S, H and the hi + lo rho'.k and y.k products, the hi + lo
    ds.k sum: 8) and the dk/dv kernel (the same six products, hi + lo coefficients against q, g and
    the hi + lo y and rho': 18)."""
    rest = 26 if tensor else 13
    stats = (9 + 5 * T) if tensor else (5 + 3 * T)
    return (stats + rest) * 2 * w.d * (w.n * (w.n + 1) / 2 * w.B * w.H)


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0}, "fallback"


def fp32_alu_peak_tflops(sm_mhz):
    """152 SMs x 128 fp32 lanes x 2 flops (FMA) per clock."""
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows for j in range(4) if r[5 + j].lower() == "active"})
        loaded = [s for s in sm if s > 0.5 * (max(sm) if sm else 1)]
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# the sources each captured kernel is compiled from (its traffic figure is void once any changes)
KERNEL_SOURCES = {
    "lla_tc_kernel": ("lla_tensor.cu", "tc_ptx.cuh", "tc_host.h", "lla_internal.h"),
    "lla_tc_kernel_bwd": ("lla_tensor.cu", "tc_ptx.cuh", "tc_host.h", "lla_internal.h"),
    "lla_simt_kernel": ("lla_simt.cu", "lla_internal.h"),
    "lla_decode_kernel": ("lla_decode.cu", "lla_internal.h"),
    "lla_decode_mom_kernel": ("lla_decode_tc.cu", "tc_ptx.cuh", "tc_host.h", "lla_internal.h"),
    "lla_bwd_stats_kernel": ("lla_backward.cu", "lla_internal.h"),
    "lla_bwd_dq_key_kernels": ("lla_backward.cu", "lla_internal.h"),
}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "local_linear_attention_flashlla_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def load_traffic(kernel, w):
    """DRAM bytes per launch from the committed ncu summary, if taken on this exact source.

    The summary holds the bytes of the named workload at its default batch; the (b, h) slices are
    independent, so a run at another batch B scales them by B / default B.  Any other change to
    the workload's shape gives None."""
    from local_linear_attention_flashlla_gb300.inputs import workload
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            doc = json.load(f)
    except (OSError, ValueError):
        return None
    ent = doc.get(f"{kernel}:{w.name}")
    if not ent or kernel not in KERNEL_SOURCES or ent.get("source_hash") != kernel_source_hash(kernel):
        return None
    base = workload(w.name)
    if w.with_(B=base.B) != base:
        return None
    return int(round(ent.get("dram_bytes_per_launch") * w.B / base.B))


# ----------------------------------------------------------------------------- CPU oracle timing

def _oracle_row(op, q, k, v, extra, tau, lam, b, h, i):
    """One oracle row: extra is the probe (parallax) or the output cotangent (backward)."""
    from oracle.lla_ref import lla_row, lla_row_grad, parallax_row
    if op == "parallax":
        return parallax_row(q[b, h, i], k[b, h, : i + 1], v[b, h, : i + 1], extra[b, h, i], tau)
    if op == "backward":
        return lla_row_grad(q[b, h, i], k[b, h, : i + 1], v[b, h, : i + 1], extra[b, h, i], tau, lam)
    return lla_row(q[b, h, i], k[b, h, : i + 1], v[b, h, : i + 1], tau, lam)


_POOL_JOB = None


def _pool_init(job):
    """Pool initializer: the sampled inputs reach each worker once, when it starts (not timed)."""
    global _POOL_JOB
    _POOL_JOB = job
    import oracle.lla_ref  # noqa: F401


def _pool_warm(_):
    """Wait until a worker has started; the short sleep spreads the warm-up tasks over all of them."""
    time.sleep(0.2)
    return os.getpid()


def _oracle_rows_worker(rows):
    """Time each row; also the worker's wall-clock start and end of its row loop (comparable across
    the processes of one host), so the caller measures the span in which the rows actually ran."""
    op, q, k, v, probe, tau, lam = _POOL_JOB
    out = []
    start = time.time()
    for (b, h, i) in rows:
        t0 = time.perf_counter()
        _oracle_row(op, q, k, v, probe, tau, lam, b, h, i)
        out.append((i, time.perf_counter() - t0))
    return out, start, time.time()


def cpu_oracle_throughput(w, qkv, budget_s=8.0, seed=123, op="lla", probe=None):
    """Time the oracle on a bounded random sample of rows on all host cores; extrapolate.

    Per-row cost is fitted as a + b (i + 1) (the dense Sigma build is (i+1) d^2) and
    integrated over every (b, h, i) of the workload.
    """
    import multiprocessing as mp

    import numpy as np

    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(seed)
    # a row's cost depends on its position i, not on its (b, h): sample the rows of two random heads,
    # so each worker receives a few MB of inputs instead of the whole workload
    heads = [(int(rng.integers(w.B)), int(rng.integers(w.H))) for _ in range(2)]
    sel = lambda t: np.stack([t[b, h] for b, h in heads])[:, None].astype(np.float64)
    q, k, v = (sel(t.double().numpy()) for t in qkv)
    pr = None if probe is None else sel(probe.double().numpy())
    # calibrate: one row at the mean causal length (after a first call that pays the imports)
    i_mid = w.n // 2
    _oracle_row(op, q, k, v, pr, w.tau, w.lam, 0, 0, min(i_mid, 7))
    t0 = time.perf_counter()
    _oracle_row(op, q, k, v, pr, w.tau, w.lam, 0, 0, i_mid)
    per_row = max(time.perf_counter() - t0, 1e-4)
    n_rows = int(max(cores * 2, min(200000, budget_s * cores / per_row)))
    rows = [(int(rng.integers(len(heads))), 0, int(rng.integers(w.n))) for _ in range(n_rows)]
    chunks = [rows[c::cores] for c in range(cores)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores, initializer=_pool_init, initargs=((op, q, k, v, pr, w.tau, w.lam),)) as pool:
        pool.map(_pool_warm, range(cores), chunksize=1)       # every worker started, inputs received
        t0 = time.perf_counter()
        res = pool.map(_oracle_rows_worker, chunks, chunksize=1)
        wall = time.perf_counter() - t0
    pts = [p for r, _, _ in res for p in r]
    i_arr = np.array([p[0] + 1 for p in pts], dtype=np.float64)
    t_arr = np.array([p[1] for p in pts])
    A = np.stack([np.ones_like(i_arr), i_arr], axis=1)
    (a, b), *_ = np.linalg.lstsq(A, t_arr, rcond=None)
    a, b = max(a, 0.0), max(b, 1e-12)
    total_single = w.B * w.H * (w.n * a + b * w.n * (w.n + 1) / 2)
    # parallel efficiency over the span in which the workers' row loops ran (from the first start to
    # the last end): it counts contention and imbalance, not the pool's start-up
    span = max(e for _, _, e in res) - min(st for _, st, _ in res)
    eff = min(1.0, t_arr.sum() / (cores * span))
    est_wall = total_single / (cores * eff)
    tokens = w.B * w.n
    return {"value": tokens / est_wall, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": (f"{len(pts)} random rows i of two random (b,h) heads of {w.name} "
                       + ("in the Parallax form (float64, explicit Sigma_KV)" if op == "parallax" else
                          "differentiated exactly (float64, dense Sigma, Cholesky, adjoint solve)" if op == "backward"
                          else "solved exactly (float64, dense Sigma, Cholesky)")
                       + f" in {wall:.1f} s wall on {cores} processes ({eff:.2f} parallel efficiency over the "
                       f"rows' span); per-row cost a+b(i+1) fitted and integrated over all {w.B * w.H * w.n} "
                       f"rows: est. {est_wall:.0f} s per step"),
            "est_seconds_per_step": est_wall}


# ----------------------------------------------------------------------------- main

def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="lm_bf16")
    ap.add_argument("--path", choices=["auto", "tensor", "fp32"], default="auto")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--op", choices=["lla", "parallax", "decode", "backward"], default="lla",
                    help="lla: the LLA forward (default); parallax: the Parallax form with a synthetic probe; "
                         "decode: one decode step (use --workload decode_bf16); backward: dq, dk, dv of the forward")
    ap.add_argument("--decode-form", choices=["auto", "moment", "stream", "cluster"], default="auto",
                    help="decode: the form (auto = moment for bf16 caches at d=128)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch B (a smaller case for profiler captures)")
    ap.add_argument("--lam", type=float, default=None,
                    help="override the workload's lambda (illcond_bf16 is quoted at 1e-3, 1e-1 and 1e6)")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def ranks_max(value, device):
    """The largest of a float over the ranks (the slowest rank's time); the value itself with one
    process.  device: where the reduction tensor lives (a CUDA device under NCCL, "cpu" under gloo)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, units_per_rank_step, steps, total_ms):
    """Whole-job units per second: every rank processes units_per_rank_step per step (weak scaling),
    timed by the slowest rank's total_ms."""
    return world * units_per_rank_step * steps / (total_ms / 1e3)


def rank_workload(w, rank):
    """Each rank draws its own inputs (seed + rank) for the same workload shape."""
    return w.with_(seed=w.seed + rank)


def run_reference(args, world, rank):
    if rank != 0:
        return
    if args.op == "decode":
        run_reference_decode(args)
        return
    from local_linear_attention_flashlla_gb300.inputs import make_cotangent, make_inputs, make_probe, workload
    w = workload(args.workload) if args.batch is None else workload(args.workload, B=args.batch)
    qkv = make_inputs(w)
    parallax = args.op == "parallax"
    backward = args.op == "backward"
    extra = make_probe(w) if parallax else make_cotangent(w) if backward else None
    steps = []
    cb = None
    for s in range(args.warmup + args.steps):
        cb = cpu_oracle_throughput(w, qkv, budget_s=2.0, seed=1000 + s, op=args.op, probe=extra)
        if s >= args.warmup:
            steps.append(cb["est_seconds_per_step"])
    sec = statistics.mean(steps)
    value = w.B * w.n / sec
    T = w.cg_max_iters
    metric = METRIC_PARALLAX if parallax else METRIC_BACKWARD if backward else METRIC
    flops = parallax_useful_flops(w) if parallax else backward_useful_flops(w, T) if backward else useful_flops(w, T)
    line = {"impl": "reference", "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w.name} B={w.B} H={w.H} n={w.n} d={w.d} tau={w.tau:.5g} lambda={w.lam} "
                                   f"cg_iters={T} cg_tol={w.cg_tol}", "l2": "n/a (CPU)"},
            "tflops": flops / sec / 1e12,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cb["cores"], "kind": "oracle",
                             "sample": cb["sample"]},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def decode_uses_moment_form(w, form, max_n):
    """Whether the decode call runs the moment form: asked for by name, or AUTO's choice (include/lla.h:
    bf16 caches at d = 128 with n <= 16384, or n past max_n, the CUDA-core forms' limit)."""
    if form == "moment":
        return True
    return form == "auto" and w.dtype == "bf16" and w.d == 128 and (w.n <= 16384 or w.n > max_n)


def decode_bytes(w, T, moment):
    """(compulsory, method) HBM bytes of one decode step.  Compulsory: the caches, q and the
    outputs once.  Method: the moment form reads K twice (the logits' maximum and kbar, then the
    centred moments) and V once; the CUDA-core forms read K in each of the T + 2 passes (moments,
    T CG iterations, output) and V once, as the three-phase algorithm reads them when the cache
    does not stay on chip."""
    e = 2 if w.dtype == "bf16" else 4
    heads = w.B * w.H
    cache = heads * w.n * w.d * e
    small = heads * w.d * (e + e + 4) + heads * 4          # q, out, rho, denom
    comp = 2 * cache + small
    return comp, comp + cache if moment else (T + 2) * cache + cache + small


def _decode_oracle_worker(rows):
    q, k, v, tau, lam = _POOL_JOB
    from oracle.lla_ref import lla_row
    out = []
    start = time.time()
    for (b, h) in rows:
        t0 = time.perf_counter()
        lla_row(q[b, h], k[b, h], v[b, h], tau, lam)
        out.append(time.perf_counter() - t0)
    return out, start, time.time()


def decode_cpu_baseline(w, qd, k, v, budget_s=12.0, seed=7):
    """The oracle (exact solve) on a bounded random sample of (b, h) decode rows, all host cores."""
    import multiprocessing as mp

    import numpy as np
    from oracle.lla_ref import lla_row
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    cores = os.cpu_count() or 1
    rng = np.random.default_rng(seed)
    # every decode row costs the same (the whole cache): time rows of two random heads, so each
    # worker receives a few MB of inputs instead of the whole cache
    heads = [(int(rng.integers(w.B)), int(rng.integers(w.H))) for _ in range(2)]
    qn, kn, vn = (np.stack([t[b, h].double().numpy() for b, h in heads])[:, None] for t in (qd, k, v))
    lla_row(qn[0, 0], kn[0, 0][:8], vn[0, 0][:8], w.tau, w.lam)   # a first, short call pays the imports
    t0 = time.perf_counter()
    lla_row(qn[0, 0], kn[0, 0], vn[0, 0], w.tau, w.lam)
    per = max(time.perf_counter() - t0, 1e-4)
    count = int(max(cores, min(100000, budget_s * cores / per)))
    rows = [(int(rng.integers(len(heads))), 0) for _ in range(count)]
    with mp.get_context("spawn").Pool(cores, initializer=_pool_init, initargs=((qn, kn, vn, w.tau, w.lam),)) as pool:
        pool.map(_pool_warm, range(cores), chunksize=1)       # every worker started, inputs received
        t0 = time.perf_counter()
        res = pool.map(_decode_oracle_worker, [rows[c::cores] for c in range(cores)], chunksize=1)
        wall = time.perf_counter() - t0
    times = [x for r, _, _ in res for x in r]
    # parallel efficiency over the span of the workers' row loops, as in cpu_oracle_throughput
    span = max(e for _, _, e in res) - min(st for _, st, _ in res)
    eff = min(1.0, sum(times) / (cores * span))
    est = w.B * w.H * (sum(times) / len(times)) / (cores * eff)
    return {"value": w.B / est, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": (f"{len(times)} decode rows of two random (b,h) heads of {w.name} solved exactly (float64, dense Sigma, "
                       f"Cholesky) in {wall:.1f} s wall on {cores} processes ({eff:.2f} parallel efficiency over "
                       f"the rows' span); mean per-row cost times B*H = "
                       f"{w.B * w.H} rows: est. {est:.1f} s per step")}


def run_reference_decode(args):
    """The oracle as the reference arm of the decode step: bounded samples of (b, h) rows."""
    from local_linear_attention_flashlla_gb300.inputs import make_inputs, workload
    name = args.workload if args.workload != "lm_bf16" else "decode_bf16"
    w = workload(name) if args.batch is None else workload(name, B=args.batch)
    q, k, v = make_inputs(w)
    qd = q[:, :, w.n - 1].contiguous()
    secs, cb = [], None
    for s_ in range(args.warmup + args.steps):
        cb = decode_cpu_baseline(w, qd, k, v, budget_s=2.0, seed=2000 + s_)
        if s_ >= args.warmup:
            secs.append(w.B / cb["value"])
    sec = statistics.mean(secs)
    value = w.B / sec
    line = {"impl": "reference", "metric": METRIC_DECODE, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w.name} B={w.B} H={w.H} cache n={w.n} d={w.d} tau={w.tau:.5g} lambda={w.lam} "
                                   f"cg_iters={w.cg_max_iters} cg_tol={w.cg_tol}", "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cb["cores"], "kind": "oracle",
                             "sample": cb["sample"]},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def run_decode(args, world, rank, local):
    import torch

    import local_linear_attention_flashlla_gb300 as lla
    from local_linear_attention_flashlla_gb300.inputs import make_inputs, workload

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    name = args.workload if args.workload != "lm_bf16" else "decode_bf16"
    w = workload(name) if args.batch is None else workload(name, B=args.batch)
    q, k, v = make_inputs(rank_workload(w, rank))
    qd_host = q[:, :, w.n - 1].contiguous()
    qd, kc, vc = qd_host.to(dev), k.to(dev), v.to(dev)
    del q
    out = torch.empty_like(qd)
    rho = torch.empty(qd.shape, dtype=torch.float32, device=dev)
    den = torch.empty(qd.shape[:2], dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    T = w.cg_max_iters

    form = {"auto": lla.LLA_DECODE_AUTO, "moment": lla.LLA_DECODE_MOMENT, "stream": lla.LLA_DECODE_STREAM,
            "cluster": lla.LLA_DECODE_CLUSTER}[args.decode_form]
    moment = decode_uses_moment_form(w, args.decode_form, lla.lla_decode_max_n(w.d))
    kname = "lla_decode_mom_kernel" if moment else "lla_decode_kernel"

    def step(qq=qd):
        lla.decode(qq, kc, vc, w.n, w.tau, w.lam, T, w.cg_tol, out=out, rho=rho, denom=den, form=form)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    lla.lla_sync_status()
    lla.lla_profile_enable(True)
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    times, main_times = [], []
    for _ in range(args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
        main_times.append(lla.lla_profile_read()[0])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    lla.lla_profile_enable(False)
    lla.lla_sync_status()
    total_ms = sum(times)
    total_ms = ranks_max(total_ms, dev)
    ms_per_step = total_ms / args.steps
    value = job_throughput(world, w.B, args.steps, total_ms)
    comp, method = decode_bytes(w, T, moment)
    kern_ms = sum(main_times) / len(main_times)
    peaks, peak_kind = load_peaks()
    hbm = peaks.get("hbm_gbs", 6800.0)
    achieved = method / (kern_ms / 1e3) / 1e9

    e2e = None
    if not args.no_e2e:
        hq = qd_host.pin_memory()
        ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hr = torch.empty(rho.shape, dtype=rho.dtype).pin_memory()
        hd = torch.empty(den.shape, dtype=den.dtype).pin_memory()
        dq = torch.empty_like(qd)
        e2e_ms = []
        for it in range(args.warmup + args.steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dq.copy_(hq, non_blocking=True)          # the new token's query; the cache stays resident
            step(dq)
            ho.copy_(out, non_blocking=True)
            hr.copy_(rho, non_blocking=True)
            hd.copy_(den, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            if it >= args.warmup:
                e2e_ms.append(e0.elapsed_time(e1))
        tot = sum(e2e_ms)
        tot = ranks_max(tot, dev)
        e2e = {"value": job_throughput(world, w.B, len(e2e_ms), tot), "unit": "tokens/s",
               "h2d_bytes_per_step": hq.numel() * hq.element_size(),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in (ho, hr, hd))}

    line = {"metric": METRIC_DECODE, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": ("bf16 in, bf16 products (w k as three terms), f32 accumulate and CG" if moment else
                      "bf16 in, f32 compute") if w.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": f"{w.name} B={w.B} H={w.H} cache n={w.n} d={w.d} tau={w.tau:.5g} lambda={w.lam} "
                                   f"cg_iters={T} cg_tol={w.cg_tol}", "l2": "flushed before every step (512 MiB write)",
                       "inputs": f"{w.dtype} caches resident in HBM"},
            "hbm_gbs": method / (ms_per_step / 1e3) / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": load_traffic(kname, w),
                         "peak_source": f"{peak_kind} copy bandwidth",
                         "bytes_counted": (f"method bytes {method} per step: K twice, V once, q and outputs once "
                                           f"(compulsory: {comp})") if moment else
                                          (f"method bytes {method} per step: K in each of T+2 passes, V once, q and "
                                           f"outputs once (compulsory: {comp})")},
            "clocks": clocks, "e2e": e2e, "gpu_launches": args.steps,
            "decode_form": "moment" if moment else args.decode_form,
            "dominant_kernel": {"name": kname, "ms_per_launch": kern_ms, "share_of_step": kern_ms / ms_per_step},
            "cg_iters_counted": T}
    if moment:
        # the products D += A^T [K | V] with A carried as three bf16 terms: 3 x 2 x d x 2d per key
        flops = 3 * 2 * w.d * 2 * w.d * w.n * w.B * w.H
        line["tensor_pipe"] = {"tflops": flops / (kern_ms / 1e3) / 1e12, "of_bf16_peak":
                               flops / (kern_ms / 1e3) / 1e12 / peaks.get("bf16_tflops", 1935.5),
                               "flops_counted": "3 bf16 terms x 2 x d x 2d per cached key (the issued products)"}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = decode_cpu_baseline(w, qd_host, k, v)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_backward(args, world, rank, local):
    """One step = one lla_backward call over the whole workload: dq, dk, dv of sum(dout * out)
    with q, k, v, dout and the forward's rho, denom resident in HBM (the forward runs once,
    untimed, before the loop: its outputs are the backward's inputs)."""
    import torch

    import local_linear_attention_flashlla_gb300 as lla
    from local_linear_attention_flashlla_gb300.inputs import make_cotangent, make_inputs, workload

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workload(args.workload) if args.batch is None else workload(args.workload, B=args.batch)
    wr = rank_workload(w, rank)
    qkv_host = make_inputs(wr)
    g_host = make_cotangent(wr)
    q, k, v = (t.to(dev) for t in qkv_host)
    g = g_host.to(dev)
    T = w.cg_max_iters
    path = {"auto": lla.LLA_PATH_AUTO, "tensor": lla.LLA_PATH_TENSOR, "fp32": lla.LLA_PATH_FP32}[args.path]
    dtype_code = lla.LLA_DTYPE_BF16 if w.dtype == "bf16" else lla.LLA_DTYPE_FP32
    rpath = lla.lla_resolve_path(dtype_code, path, w.d)
    _, rho, den = lla.forward(q, k, v, w.tau, w.lam, T, w.cg_tol)
    grads = [torch.empty(q.shape, dtype=torch.float32, device=dev) for _ in range(3)]
    ws = torch.empty(lla.lla_backward_workspace_size(dtype_code, path, w.B, w.H, w.n, w.d), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(qq=q, kk=k, vv=v, rr=rho, dd=den, gg=g):
        lla.backward(qq, kk, vv, rr, dd, gg, w.tau, w.lam, T, w.cg_tol, path=path, dq=grads[0], dk=grads[1],
                     dv=grads[2], workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    lla.lla_sync_status()
    lla.lla_profile_enable(True)
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    times, main_times = [], []
    for _ in range(args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
        main_times.append(lla.lla_profile_read())
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    lla.lla_profile_enable(False)
    lla.lla_sync_status()
    total_ms = sum(times)
    total_ms = ranks_max(total_ms, dev)
    ms_per_step = total_ms / args.steps
    tokens = w.B * w.n
    value = job_throughput(world, tokens, args.steps, total_ms)
    flops = backward_useful_flops(w, T)
    q_ms = sum(m for m, _ in main_times) / len(main_times)          # stats kernel (moments and adjoint CG)
    call_ms = sum(t_ for _, t_ in main_times) / len(main_times)     # the whole call
    k_ms = max(call_ms - q_ms, 1e-9)                                 # dq and dk/dv stages (tensor path: with their prep)
    pairs_flops = 2 * w.d * (w.n * (w.n + 1) / 2 * w.B * w.H)
    q_flops = (4 + 2 * T) * pairs_flops      # the stats stage's useful share: q.k, g.v, two moment sums, CG
    k_flops = 7 * pairs_flops                # the rest: rho'.k, y.k, dq; dk (three terms) and dv
    peaks, peak_kind = load_peaks()
    alu_peak = fp32_alu_peak_tflops(peaks.get("sm_max_mhz", 2070.0))
    stats_tensor = rpath == lla.LLA_PATH_TENSOR
    if stats_tensor:
        stats_peak, stats_bound, stats_src = peaks["bf16_tflops"], "tensor", f"{peak_kind} bf16 burst"
    else:
        stats_peak, stats_bound, stats_src = alu_peak, "alu", "derived: 152 SMs x 128 fp32 FMA lanes x 2 flops x max SM clock"
    stats_roof = {"bound": stats_bound, "achieved": q_flops / (q_ms / 1e3) / 1e12, "peak": stats_peak,
                  "unit": "TFLOP/s", "frac": q_flops / (q_ms / 1e3) / 1e12 / stats_peak,
                  "traffic": load_traffic("lla_tc_kernel_bwd" if stats_tensor else "lla_bwd_stats_kernel", w),
                  "peak_source": stats_src,
                  "flops_counted": "stats stage, useful (4+2T) passes x 2d per causal pair"
                                   + ("; executed on tensor cores: (9+5T) passes (hi + lo operands)" if stats_tensor else "")}
    rest_peak = peaks["bf16_tflops"] if stats_tensor else alu_peak
    rest_roof = {"bound": "tensor" if stats_tensor else "alu", "achieved": k_flops / (k_ms / 1e3) / 1e12,
                 "peak": rest_peak, "unit": "TFLOP/s", "frac": k_flops / (k_ms / 1e3) / 1e12 / rest_peak,
                 "traffic": None,
                 "peak_source": f"{peak_kind} bf16 burst" if stats_tensor else
                 "derived: 152 SMs x 128 fp32 FMA lanes x 2 flops x max SM clock",
                 "flops_counted": "dq and dk/dv stages, useful 7 passes x 2d per causal pair"
                                  + ("; executed on tensor cores: 26 passes (hi + lo operands)" if stats_tensor else "")}
    stats_name = "lla_tc_kernel<128,bwd>" if stats_tensor else "lla_bwd_stats_kernel"
    rest_name = ("lla_bwd_dq_tc_kernel + lla_bwd_kv_tc_kernel (+ prep)" if stats_tensor
                 else "lla_bwd_dq_kernel + lla_bwd_key_kernel")
    dominant_is_stats = q_ms >= k_ms
    roof = stats_roof if dominant_is_stats else rest_roof

    # end to end through the C-ABI host-buffer call (lla_backward_host: chunked copies in and out
    # overlapped with the compute), from and into pinned host buffers
    e2e = None
    if not args.no_e2e:
        hin = [t.pin_memory() for t in (*qkv_host, g_host)] + [rho.cpu().pin_memory(), den.cpu().pin_memory()]
        hout = [torch.empty(q.shape, dtype=torch.float32).pin_memory() for _ in range(3)]
        dtype_c = lla.LLA_DTYPE_BF16 if q.dtype == torch.bfloat16 else lla.LLA_DTYPE_FP32
        hbuf = torch.empty(lla.lla_backward_host_buffer_size(dtype_c, path, w.B, w.H, w.n, w.d, 0),
                           dtype=torch.uint8, device=dev)
        e2e_ms = []
        for it in range(args.warmup + args.steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            lla.backward_host(hin[0], hin[1], hin[2], hin[4], hin[5], hin[3], w.tau, w.lam, T, w.cg_tol, path=path,
                              dq=hout[0], dk=hout[1], dv=hout[2], device_buffer=hbuf)
            e1.record(stream)
            e1.synchronize()
            if it >= args.warmup:
                e2e_ms.append(e0.elapsed_time(e1))
        tot = sum(e2e_ms)
        tot = ranks_max(tot, dev)
        e2e = {"value": job_throughput(world, tokens, len(e2e_ms), tot), "unit": "tokens/s",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hin),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in hout)}

    line = {"metric": METRIC_BACKWARD, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16 hi+lo / f32" if stats_tensor else "f32", "data": "synthetic",
            "config": {"workload": f"{w.name} B={w.B} H={w.H} n={w.n} d={w.d} tau={w.tau:.5g} lambda={w.lam} "
                                   f"cg_iters={T} cg_tol={w.cg_tol} (forward and adjoint)",
                       "l2": "flushed before every step (512 MiB write)",
                       "inputs": f"{w.dtype} q,k,v,dout and the forward's fp32 rho, denom resident in HBM"},
            "tflops": world * flops * args.steps / (total_ms / 1e3) / 1e12,
            "tflops_executed": world * backward_executed_flops(w, T, stats_tensor) * args.steps / (total_ms / 1e3) / 1e12,
            "roofline": roof, "clocks": clocks, "e2e": e2e,
            "gpu_launches": (7 if stats_tensor else 3) * args.steps,
            "dominant_kernel": {"name": stats_name if dominant_is_stats else rest_name,
                                "ms_per_launch": q_ms if dominant_is_stats else k_ms,
                                "share_of_step": (q_ms if dominant_is_stats else k_ms) / ms_per_step},
            "stages": {"stats": {"kernel": stats_name, "ms": q_ms, "roofline": stats_roof},
                       "dq_dk_dv": {"kernels": rest_name, "ms": k_ms, "roofline": rest_roof}},
            "path": "tensor (tcgen05 stats, dq, dk/dv)" if stats_tensor else "fp32",
            "cg_iters_counted": T}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_throughput(w, qkv_host, op="backward", probe=g_host)
        line["cpu_baseline"].pop("est_seconds_per_step", None)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


class _StreamOrderedPool:
    """High-water mark of the device's current stream-ordered pool (the one cudaMallocAsync, and
    so lla_forward's workspace, draws from), through the CUDA driver API."""
    USED_MEM_HIGH = 8                      # CUmemPool_attribute

    def __init__(self, device_index):
        import ctypes
        self.ct = ctypes
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        self.pool = ctypes.c_void_p()
        if self.cu.cuDeviceGet(ctypes.byref(dev), device_index) or \
                self.cu.cuDeviceGetMemPool(ctypes.byref(self.pool), dev):
            raise OSError("cannot query the device's memory pool")

    def reset(self):
        zero = self.ct.c_uint64(0)
        self.cu.cuMemPoolSetAttribute(self.pool, self.USED_MEM_HIGH, self.ct.byref(zero))

    def high(self):
        val = self.ct.c_uint64()
        self.cu.cuMemPoolGetAttribute(self.pool, self.USED_MEM_HIGH, self.ct.byref(val))
        return int(val.value)


def memory_and_n_scaling(lla, w, path, dev, peak_tflops, flush, ns=(4096, 8192, 16384, 32768), steps=3):
    """Device memory of one lla_forward call and its time at n in ns (H, B and d of w).

    Memory: the caller's tensors (q, k, v in; out, rho, denom out: torch's peak allocation while
    they exist) plus the workspace the call takes from the stream-ordered pool (the pool's high-water
    mark during the call, workspace not supplied): peak device bytes, and per element of q.
    Time: CUDA events around each call after a warm-up, L2 flushed before each (as the headline)."""
    import torch
    from local_linear_attention_flashlla_gb300.inputs import make_inputs
    pool = _StreamOrderedPool(dev.index if dev.index is not None else 0)
    mem, series = None, []
    for n in ns:
        wn = w.with_(n=n)
        qkv_host = make_inputs(wn)
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats(dev)
        base = torch.cuda.memory_allocated(dev)
        q, k, v = (t.to(dev) for t in qkv_host)
        out = torch.empty_like(q)
        rho = torch.empty(q.shape, dtype=torch.float32, device=dev)
        den = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        lla.forward(q, k, v, wn.tau, wn.lam, wn.cg_max_iters, wn.cg_tol, path=path, out=out, rho=rho, denom=den)
        torch.cuda.synchronize()
        pool.reset()
        lla.forward(q, k, v, wn.tau, wn.lam, wn.cg_max_iters, wn.cg_tol, path=path, out=out, rho=rho, denom=den)
        torch.cuda.synchronize()
        pool_bytes = pool.high()
        tensor_bytes = torch.cuda.max_memory_allocated(dev) - base
        elems = wn.B * wn.H * wn.n * wn.d
        times = []
        for _ in range(steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            lla.forward(q, k, v, wn.tau, wn.lam, wn.cg_max_iters, wn.cg_tol, path=path, out=out, rho=rho, denom=den)
            e1.record()
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        ms = statistics.median(times)
        tf = useful_flops(wn, wn.cg_max_iters) / (ms / 1e3) / 1e12
        series.append({"n": n, "ms": ms, "tflops": tf, "frac": tf / peak_tflops,
                       "peak_device_bytes": tensor_bytes + pool_bytes, "bytes_per_element": (tensor_bytes + pool_bytes) / elems})
        if n == w.n:
            mem = {"n": n, "caller_tensor_bytes": tensor_bytes, "workspace_pool_bytes": pool_bytes,
                   "peak_device_bytes": tensor_bytes + pool_bytes,
                   "bytes_per_element": (tensor_bytes + pool_bytes) / elems,
                   "lla_workspace_size": lla.lla_workspace_size(lla.LLA_DTYPE_BF16, path, wn.B, wn.H, wn.n, wn.d),
                   "how": "torch peak allocation of q,k,v,out,rho,denom + the stream-ordered pool's high-water mark "
                          "during one lla_forward call that takes its workspace from the pool"}
        del q, k, v, out, rho, den
        torch.cuda.empty_cache()
    t_last = series[-1]["ms"] / series[-1]["n"] ** 2
    for e in series:
        e["ms_over_n2_rel_to_largest"] = (e["ms"] / e["n"] ** 2) / t_last
    return mem, series


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.op == "decode":
        run_decode(args, world, rank, local)
        return
    if args.op == "backward":
        run_backward(args, world, rank, local)
        return
    import numpy as np
    import torch

    import local_linear_attention_flashlla_gb300 as lla
    from local_linear_attention_flashlla_gb300.inputs import make_inputs, make_probe, workload

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workload(args.workload) if args.batch is None else workload(args.workload, B=args.batch)
    if args.lam is not None:
        w = w.with_(lam=args.lam)
    path = {"auto": lla.LLA_PATH_AUTO, "tensor": lla.LLA_PATH_TENSOR, "fp32": lla.LLA_PATH_FP32}[args.path]
    dtype_code = lla.LLA_DTYPE_BF16 if w.dtype == "bf16" else lla.LLA_DTYPE_FP32
    rpath = lla.lla_resolve_path(dtype_code, path, w.d)
    qkv_host = make_inputs(rank_workload(w, rank))
    q, k, v = (t.to(dev) for t in qkv_host)
    parallax = args.op == "parallax"
    probe_host = make_probe(rank_workload(w, rank)) if parallax else None
    probe = probe_host.to(dev) if parallax else None
    out = torch.empty_like(q)
    rho = torch.empty(q.shape, dtype=torch.float32, device=dev)
    den = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    ws_bytes = lla.lla_workspace_size(dtype_code, path, w.B, w.H, w.n, w.d)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        if parallax:
            lla.parallax_forward(q, k, v, probe, w.tau, path=path, out=out, workspace=ws if ws_bytes else None)
        else:
            lla.forward(q, k, v, w.tau, w.lam, w.cg_max_iters, w.cg_tol, path=path, out=out, rho=rho, denom=den,
                        workspace=ws if ws_bytes else None)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    lla.lla_sync_status()

    lla.lla_profile_enable(True)      # events around the dominant kernel of every call
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    times, main_times = [], []
    for _ in range(args.steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
        main_times.append(lla.lla_profile_read()[0])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    lla.lla_profile_enable(False)
    lla.lla_sync_status()
    total_ms = sum(times)
    total_ms = ranks_max(total_ms, dev)
    ms_per_step = total_ms / args.steps
    tokens = w.B * w.n
    value = job_throughput(world, tokens, args.steps, total_ms)
    T = w.cg_max_iters if (w.cg_tol == 0 or parallax) else None
    iters_info = None
    if T is None:   # tolerance-driven: count the iterations each query tile executed
        _, _, _, its = lla.forward(q, k, v, w.tau, w.lam, w.cg_max_iters, w.cg_tol, path=path, return_iters=True)
        its = its.cpu().numpy()
        flops, flops_exec, T_mean, T_pw = tolerance_flops(w, its, rpath, precise=True)
        T = T_pw
        iters_info = {"tile_rows": TILE_ROWS[rpath], "tile_mean": T_mean, "pair_weighted_tile_mean": T_pw,
                      "query_mean": float(its.mean()), "query_max": int(its.max()),
                      "query_histogram": iteration_histogram(its)}
    else:
        flops = parallax_useful_flops(w) if parallax else useful_flops(w, T)
        flops_exec = (parallax_executed_flops(w, rpath == lla.LLA_PATH_TENSOR) if parallax else
                      executed_flops(w, T, rpath))
    tflops = world * flops * args.steps / (total_ms / 1e3) / 1e12

    # end to end through the public API from pinned host buffers: the LLA forward through the C-ABI
    # host-buffer call (lla_forward_host: chunked copies in and out overlapped with the compute);
    # the Parallax form, which has no host-buffer call, as copy in, device call, copy out
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (t.pin_memory() for t in qkv_host)
        hp = probe_host.pin_memory() if parallax else None
        ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hr = torch.empty(rho.shape, dtype=rho.dtype).pin_memory()
        hd = torch.empty(den.shape, dtype=den.dtype).pin_memory()
        if parallax:
            dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
            dp = torch.empty_like(probe)
        else:
            dtype_c = lla.LLA_DTYPE_BF16 if q.dtype == torch.bfloat16 else lla.LLA_DTYPE_FP32
            hbuf = torch.empty(lla.lla_forward_host_buffer_size(dtype_c, path, w.B, w.H, w.n, w.d, 0),
                               dtype=torch.uint8, device=dev)
        e2e_ms = []
        for it in range(args.warmup + args.steps):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if parallax:
                dq.copy_(hq, non_blocking=True)
                dk.copy_(hk, non_blocking=True)
                dv.copy_(hv, non_blocking=True)
                dp.copy_(hp, non_blocking=True)
                lla.parallax_forward(dq, dk, dv, dp, w.tau, path=path, out=out, workspace=ws if ws_bytes else None)
                ho.copy_(out, non_blocking=True)
            else:
                lla.forward_host(hq, hk, hv, w.tau, w.lam, w.cg_max_iters, w.cg_tol, path=path, out=ho, rho=hr,
                                 denom=hd, device_buffer=hbuf)
            e1.record(stream)
            e1.synchronize()
            if it >= args.warmup:
                e2e_ms.append(e0.elapsed_time(e1))
        tot = sum(e2e_ms)
        tot = ranks_max(tot, dev)
        e2e = {"value": job_throughput(world, tokens, len(e2e_ms), tot), "unit": "tokens/s",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (hq, hk, hv) + ((hp,) if parallax else ())),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in ((ho,) if parallax else (ho, hr, hd)))}

    peaks, peak_kind = load_peaks()
    # fp32 path: one kernel per step; tensor path: max|x| pre-pass, fp16 conversion, fused sweep kernel
    # (the precise and Parallax forms launch the fused kernel twice: without MAX sweeps, then again
    # for the tiles the first launch marked)
    launches_per_step = 1 if rpath == lla.LLA_PATH_FP32 else (4 if (parallax or w.cg_tol > 0) else 3)
    kern_name = "lla_simt_kernel" if rpath == lla.LLA_PATH_FP32 else "lla_tc_kernel"
    dominant_ms = sum(main_times) / len(main_times)
    achieved = flops / (dominant_ms / 1e3) / 1e12
    if rpath == lla.LLA_PATH_FP32:
        peak = fp32_alu_peak_tflops(peaks.get("sm_max_mhz", 2070.0))
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": load_traffic(kern_name, w),
                "peak_source": "derived: 152 SMs x 128 fp32 FMA lanes x 2 flops x max SM clock",
                "flops_counted": "useful (4+3T) passes x 2d per causal pair"}
        dtype = "bf16 in, f32 compute" if w.dtype == "bf16" else "f32"
    else:
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": None if parallax else load_traffic(kern_name, w), "peak_source": f"{peak_kind} bf16 burst",
                "flops_counted": ("useful 4 passes (q.k, weighted key mean, probe.k, values) x 2d per causal pair"
                                  if parallax else "useful (4+3T) passes x 2d per causal pair")}
        dtype = "bf16 in, f16 MMA operands (exact), f32 accumulate and CG state"

    line = {"metric": METRIC_PARALLAX if parallax else METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": {"workload": f"{w.name} B={w.B} H={w.H} n={w.n} d={w.d} tau={w.tau:.5g} lambda={w.lam} "
                                   f"cg_iters={w.cg_max_iters} cg_tol={w.cg_tol}",
                       "path": {1: "tensor", 2: "fp32"}[rpath], "l2": "flushed before every step (512 MiB write)",
                       "inputs": "bf16 q,k,v resident in HBM" if w.dtype == "bf16" else "fp32 q,k,v in HBM"},
            "tflops": tflops,
            "tflops_executed": world * flops_exec * args.steps / (total_ms / 1e3) / 1e12,
            "roofline": roof, "clocks": clocks, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "dominant_kernel": {"name": kern_name, "ms_per_launch": dominant_ms,
                                "share_of_step": dominant_ms / ms_per_step},
            "cg_iters_counted": None if parallax else T}
    if iters_info is not None:
        line["cg_iterations"] = iters_info
        line["roofline"]["flops_counted"] = ("useful (4+3T_t) passes x 2d over each query tile's causal pairs, "
                                             "T_t the iterations that tile executed")
    if w.name == "long_bf16" and world == 1 and not parallax:
        line["memory"], line["n_scaling"] = memory_and_n_scaling(lla, w, path, dev, peak, flush)
    if parallax:
        line["config"]["workload"] = f"{w.name} B={w.B} H={w.H} n={w.n} d={w.d} tau={w.tau:.5g} (Parallax form, probe)"
        line["config"]["probe"] = "seeded RMS-normalised Gaussian rows / sqrt(d), fp32"
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_throughput(w, qkv_host, op=args.op, probe=probe_host)
        line["cpu_baseline"].pop("est_seconds_per_step", None)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
