"""Shared helpers for the GPU parity tests: run the CUDA path, run the oracle on the
same inputs, and compare with the error metrics stated in the tests.

Metrics (per compared row, then the max over rows):
* out:   max_e |out - ref| / RMS(v), RMS over the whole v tensor;
* rho:   max_e |rho - ref| / RMS(ref rho over the compared rows);
* denom: |denom - ref| / ref.
"""
import math

import numpy as np
import torch

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300.inputs import make_inputs, sample_rows
from oracle.lla_ref import lla_ref, softmax_ref


def run_gpu(w, path, lam=None, tol=None, iters=None, return_iters=True, inputs=None):
    q, k, v = make_inputs(w) if inputs is None else inputs
    dev = torch.device("cuda:0")
    res = lla.forward(q.to(dev), k.to(dev), v.to(dev), w.tau, w.lam if lam is None else lam,
                      w.cg_max_iters if iters is None else iters, w.cg_tol if tol is None else tol,
                      path=path, return_iters=return_iters)
    torch.cuda.synchronize()
    lla.lla_sync_status()
    host = [t.cpu() for t in res]
    return (q, k, v), host


def pick(arr, rows):
    a = arr.double().numpy() if isinstance(arr, torch.Tensor) else arr
    return np.array([a[b, h, i] for b, h, i in rows])


def oracle_rows(qkv, w, rows, lam=None, iters=None, tol=None):
    qn, kn, vn = (t.double().numpy() for t in qkv)
    lam = w.lam if lam is None else lam
    T = w.cg_max_iters if iters is None else iters
    tol = w.cg_tol if tol is None else tol
    exact = lla_ref(qn, kn, vn, w.tau, lam, rows=rows)
    cg = lla_ref(qn, kn, vn, w.tau, lam, rows=rows, deflated=(T, tol))
    return exact, cg, math.sqrt(float(np.mean(vn ** 2)))


def errors(g_out, g_rho, g_den, ref, rms_v):
    r_out, r_rho, r_den = ref
    e_out = np.abs(g_out - r_out).max(axis=1) / rms_v
    rms_rho = math.sqrt(float(np.mean(r_rho ** 2))) or 1.0
    e_rho = np.abs(g_rho - r_rho).max(axis=1) / rms_rho
    e_den = np.abs(g_den - r_den) / np.abs(r_den)
    return e_out, e_rho, e_den


def all_rows(w):
    return [(b, h, i) for b in range(w.B) for h in range(w.H) for i in range(w.n)]


def rows_for(w, count):
    return sample_rows(w, count) if w.B * w.H * w.n > count else all_rows(w)


def softmax_rows(qkv, w, rows):
    qn, kn, vn = (t.double().numpy() for t in qkv)
    return softmax_ref(qn, kn, vn, w.tau, rows=rows)
