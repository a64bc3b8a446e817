"""The C-ABI library builds, loads, exports every symbol include/lla.h declares, and
rejects bad arguments on the host (no GPU needed: nothing is launched)."""
import ctypes
import os
import re

import pytest

import local_linear_attention_flashlla_gb300 as lla
from local_linear_attention_flashlla_gb300 import build as lla_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(lla.library_path()):
        lla_build.build()
    return lla.load_library()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "lla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lla_[a-z_]+)\s*\(", text)))


def test_header_declares_the_bound_entry_points():
    assert _declared_functions() == sorted(lla.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert lib.lla_version() == 10000


def _call_ex(lib, **kw):
    a = dict(dtype=0, path=0, q=16, k=32, v=48, out=64, rho=80, den=96, it=None, B=1, H=1, n=8, d=64,
             tau=0.1, lam=1.0, T=4, tol=0.0, ws=None, wsb=0, stream=None)
    a.update(kw)
    return lib.lla_forward_ex(a["dtype"], a["path"], a["q"], a["k"], a["v"], a["out"], a["rho"], a["den"], a["it"],
                              a["B"], a["H"], a["n"], a["d"], a["tau"], a["lam"], a["T"], a["tol"], a["ws"], a["wsb"],
                              a["stream"])


@pytest.mark.parametrize("bad", [
    dict(q=None), dict(out=None), dict(rho=None), dict(den=None), dict(q=17), dict(B=0), dict(n=0), dict(H=-1),
    dict(B=65536), dict(B=256, H=256),
    dict(d=48), dict(d=256), dict(tau=0.0), dict(tau=-1.0), dict(tau=float("nan")), dict(lam=0.0),
    dict(lam=float("inf")), dict(T=0), dict(T=5000), dict(tol=-1.0), dict(dtype=7), dict(path=9),
])
def test_invalid_arguments_rejected_before_launch(lib, bad):
    assert _call_ex(lib, **bad) == lla.LLA_ERR_INVALID_ARG
    assert lib.lla_last_error().decode()


def test_tensor_path_needs_bf16_and_supported_dim(lib):
    assert _call_ex(lib, dtype=1, path=lla.LLA_PATH_TENSOR) == lla.LLA_ERR_UNSUPPORTED
    assert _call_ex(lib, d=32, path=lla.LLA_PATH_TENSOR) == lla.LLA_ERR_UNSUPPORTED


def test_path_resolution_and_workspace_size(lib):
    assert lib.lla_resolve_path(lla.LLA_DTYPE_FP32, lla.LLA_PATH_AUTO, 128) == lla.LLA_PATH_FP32
    assert lib.lla_resolve_path(lla.LLA_DTYPE_BF16, lla.LLA_PATH_AUTO, 128) == lla.LLA_PATH_TENSOR
    assert lib.lla_resolve_path(lla.LLA_DTYPE_BF16, lla.LLA_PATH_AUTO, 64) == lla.LLA_PATH_TENSOR
    assert lib.lla_resolve_path(lla.LLA_DTYPE_BF16, lla.LLA_PATH_AUTO, 32) == lla.LLA_PATH_FP32
    assert lib.lla_resolve_path(lla.LLA_DTYPE_BF16, lla.LLA_PATH_FP32, 128) == lla.LLA_PATH_FP32
    assert lib.lla_workspace_size(lla.LLA_DTYPE_FP32, lla.LLA_PATH_AUTO, 2, 2, 64, 64) == 0
    assert lib.lla_workspace_size(lla.LLA_DTYPE_BF16, lla.LLA_PATH_TENSOR, 2, 2, 64, 64) > 0


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 1, 4, 16)
    with pytest.raises(lla.LLAError):
        lla.forward(x, x, x, 0.25, 0.1, 4)


def _call_parallax(lib, **kw):
    a = dict(dtype=0, path=0, q=16, k=32, v=48, probe=80, out=64, B=1, H=1, n=8, d=64, tau=0.1, ws=None, wsb=0,
             stream=None)
    a.update(kw)
    return lib.lla_parallax_forward(a["dtype"], a["path"], a["q"], a["k"], a["v"], a["probe"], a["out"], a["B"],
                                    a["H"], a["n"], a["d"], a["tau"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("bad", [
    dict(q=None), dict(probe=None), dict(out=None), dict(probe=20), dict(B=0), dict(n=0), dict(d=48), dict(B=65536),
    dict(tau=0.0), dict(tau=float("nan")), dict(dtype=5), dict(path=-1),
])
def test_parallax_invalid_arguments_rejected_before_launch(lib, bad):
    assert _call_parallax(lib, **bad) == lla.LLA_ERR_INVALID_ARG
    assert lib.lla_last_error().decode()


def test_parallax_tensor_path_needs_bf16_and_supported_dim(lib):
    assert _call_parallax(lib, dtype=1, path=lla.LLA_PATH_TENSOR) == lla.LLA_ERR_UNSUPPORTED
    assert _call_parallax(lib, d=16, path=lla.LLA_PATH_TENSOR) == lla.LLA_ERR_UNSUPPORTED


def test_parallax_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 1, 4, 16)
    with pytest.raises(lla.LLAError):
        lla.parallax_forward(x, x, x, x, 0.25)


def _call_decode(lib, **kw):
    a = dict(dtype=0, q=16, k=32, v=48, out=64, rho=80, den=96, it=None, B=1, H=1, n=8, n_cap=8, d=64, tau=0.1,
             lam=1.0, T=4, tol=0.0, stream=None)
    a.update(kw)
    return lib.lla_decode(a["dtype"], a["q"], a["k"], a["v"], a["out"], a["rho"], a["den"], a["it"], a["B"], a["H"],
                          a["n"], a["n_cap"], a["d"], a["tau"], a["lam"], a["T"], a["tol"], a["stream"])


@pytest.mark.parametrize("bad", [
    dict(q=None), dict(k=None), dict(rho=None), dict(den=None), dict(v=40), dict(B=0), dict(n=0), dict(n_cap=7),
    dict(d=48), dict(tau=0.0), dict(lam=-1.0), dict(T=0), dict(tol=float("nan")), dict(dtype=3),
])
def test_decode_invalid_arguments_rejected_before_launch(lib, bad):
    assert _call_decode(lib, **bad) == lla.LLA_ERR_INVALID_ARG
    assert lib.lla_last_error().decode()


def _call_decode_ex(lib, form, **kw):
    a = dict(dtype=0, q=16, k=32, v=48, out=64, rho=80, den=96, it=None, B=1, H=1, n=8, n_cap=8, d=64, tau=0.1,
             lam=1.0, T=4, tol=0.0, stream=None)
    a.update(kw)
    return lib.lla_decode_ex(form, a["dtype"], a["q"], a["k"], a["v"], a["out"], a["rho"], a["den"], a["it"], a["B"],
                             a["H"], a["n"], a["n_cap"], a["d"], a["tau"], a["lam"], a["T"], a["tol"], a["stream"])


def test_decode_cache_length_limit(lib):
    """The CUDA-core forms keep a head's n weights in shared memory (the moment form, which AUTO
    takes for bf16 caches at d = 128, has no such limit and is not called here: it needs a GPU)."""
    for d in (16, 32, 64, 128):
        m = lib.lla_decode_max_n(d)
        assert 32768 <= m < 60000
        assert _call_decode(lib, dtype=1, d=d, n=m + 1, n_cap=m + 1) == lla.LLA_ERR_UNSUPPORTED
        assert _call_decode_ex(lib, lla.LLA_DECODE_STREAM, d=d, n=m + 1, n_cap=m + 1) == lla.LLA_ERR_UNSUPPORTED
    assert lib.lla_decode_max_n(48) == 0


@pytest.mark.parametrize("form,kw,status", [
    (lla.LLA_DECODE_MOMENT, dict(dtype=1, d=128), lla.LLA_ERR_UNSUPPORTED),      # fp32 caches
    (lla.LLA_DECODE_MOMENT, dict(d=64), lla.LLA_ERR_UNSUPPORTED),                # d != 128
    (lla.LLA_DECODE_CLUSTER, dict(d=128, n=40000, n_cap=40000), lla.LLA_ERR_UNSUPPORTED),   # an eighth too long
    (7, dict(), lla.LLA_ERR_INVALID_ARG),
    (-1, dict(), lla.LLA_ERR_INVALID_ARG),
    (lla.LLA_DECODE_MOMENT, dict(d=128, B=0), lla.LLA_ERR_INVALID_ARG),
])
def test_decode_form_rejected_before_launch(lib, form, kw, status):
    assert _call_decode_ex(lib, form, **kw) == status
    assert lib.lla_last_error().decode()


def _call_backward(lib, **kw):
    a = dict(dtype=0, path=0, q=16, k=32, v=48, rho=64, den=80, dout=96, dq=112, dk=128, dv=144, it=None, B=1, H=1,
             n=8, d=64, tau=0.1, lam=1.0, T=4, tol=0.0, ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.lla_backward(a["dtype"], a["path"], a["q"], a["k"], a["v"], a["rho"], a["den"], a["dout"], a["dq"],
                            a["dk"], a["dv"], a["it"], a["B"], a["H"], a["n"], a["d"], a["tau"], a["lam"], a["T"],
                            a["tol"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("bad", [
    dict(q=None), dict(rho=None), dict(den=None), dict(dout=None), dict(dq=None), dict(dk=None), dict(dv=None),
    dict(dv=40), dict(B=0), dict(n=0), dict(H=70000), dict(d=48), dict(tau=0.0), dict(lam=-1.0), dict(T=0),
    dict(tol=float("nan")), dict(dtype=3), dict(path=7), dict(ws=4096, ws_bytes=16),
    dict(ws=4096 + 16, ws_bytes=1 << 20),
])
def test_backward_invalid_arguments_rejected_before_launch(lib, bad):
    assert _call_backward(lib, **bad) == lla.LLA_ERR_INVALID_ARG
    assert lib.lla_last_error().decode()


def test_backward_tensor_path_needs_bf16_and_supported_dim(lib):
    assert _call_backward(lib, dtype=1, path=lla.LLA_PATH_TENSOR) == lla.LLA_ERR_UNSUPPORTED
    assert _call_backward(lib, d=32, path=lla.LLA_PATH_TENSOR) == lla.LLA_ERR_UNSUPPORTED


def test_backward_workspace_size(lib):
    fp32 = lla.LLA_PATH_FP32
    # fp32 path: one 32-byte record and one fp32 d-vector per query, each part rounded up to 256 bytes
    assert lib.lla_backward_workspace_size(0, fp32, 2, 3, 100, 64) == 19200 + 153600
    assert lib.lla_backward_workspace_size(1, fp32, 1, 1, 1, 16) == 256 + 256
    assert lib.lla_backward_workspace_size(0, fp32, 0, 1, 1, 16) == 0
    # tensor path (bf16, d = 64 resolves to it): the records, the forward kernel's scratch and dout in fp16,
    # then the dk/dv stage's scratch: a 256-byte header, rho' and y as fp16 hi + lo, two words per key
    recs = 19200 + 153600
    fwd = lib.lla_workspace_size(0, lla.LLA_PATH_TENSOR, 2, 3, 100, 64)
    half = ((2 * 3 * 100 * 64 * 2 + 255) // 256) * 256
    kmax = ((2 * 3 * 100 * 8 + 255) // 256) * 256
    assert lib.lla_backward_workspace_size(0, lla.LLA_PATH_AUTO, 2, 3, 100, 64) == recs + fwd + half + 256 + 4 * half + kmax


def test_backward_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 1, 4, 16)
    with pytest.raises(lla.LLAError):
        lla.backward(x, x, x, x, torch.zeros(1, 1, 4), x, 0.25, 1.0, 4)


def _call_host(lib, **kw):
    a = dict(dtype=0, path=0, q=16, k=32, v=48, out=64, rho=80, den=96, it=None, B=1, H=1, n=8, d=64,
             tau=0.1, lam=1.0, T=4, tol=0.0, chunk=0, buf=None, bufb=0, stream=None)
    a.update(kw)
    return lib.lla_forward_host(a["dtype"], a["path"], a["q"], a["k"], a["v"], a["out"], a["rho"], a["den"],
                                a["it"], a["B"], a["H"], a["n"], a["d"], a["tau"], a["lam"], a["T"], a["tol"],
                                a["chunk"], a["buf"], a["bufb"], a["stream"])


@pytest.mark.parametrize("bad", [
    dict(q=None), dict(v=None), dict(out=None), dict(rho=None), dict(den=None), dict(B=0), dict(n=0), dict(d=48),
    dict(tau=0.0), dict(lam=float("nan")), dict(T=0), dict(tol=-1.0), dict(dtype=7), dict(path=9), dict(chunk=-1),
    dict(buf=256, bufb=16), dict(buf=257, bufb=1 << 40),
])
def test_host_forward_invalid_arguments_rejected_before_launch(lib, bad):
    assert _call_host(lib, **bad) == lla.LLA_ERR_INVALID_ARG
    assert lib.lla_last_error().decode()


def test_host_forward_tensor_path_needs_bf16_and_supported_dim(lib):
    assert _call_host(lib, dtype=1, path=lla.LLA_PATH_TENSOR) == lla.LLA_ERR_UNSUPPORTED
    assert _call_host(lib, d=32, path=lla.LLA_PATH_TENSOR) == lla.LLA_ERR_UNSUPPORTED


def test_host_forward_buffer_size(lib):
    """Two halves, each holding one chunk's q, k, v, out, rho, denom, cg_iters (each rounded up to
    256 bytes) and, on the tensor path, the chunk's workspace."""
    def a256(x):
        return (x + 255) & ~255

    def expect(dtype, path, C, n, d):
        es = 2 if dtype == lla.LLA_DTYPE_BF16 else 4
        ws = lib.lla_workspace_size(dtype, path, C, 1, n, d)
        return 2 * (4 * a256(C * n * d * es) + a256(C * n * d * 4) + 2 * a256(C * n * 4) + a256(ws))

    bf, f32, ten, fp = lla.LLA_DTYPE_BF16, lla.LLA_DTYPE_FP32, lla.LLA_PATH_TENSOR, lla.LLA_PATH_FP32
    # automatic chunk: about eight chunks of the B*H slices (8 slices -> 1, 128 -> 16, 3 -> 1)
    assert lib.lla_forward_host_buffer_size(bf, ten, 2, 4, 300, 64, 0) == expect(bf, ten, 1, 300, 64)
    assert lib.lla_forward_host_buffer_size(bf, ten, 8, 16, 256, 128, 0) == expect(bf, ten, 16, 256, 128)
    assert lib.lla_forward_host_buffer_size(f32, fp, 1, 3, 100, 32, 0) == expect(f32, fp, 1, 100, 32)
    # explicit chunk, clamped to the slice count
    assert lib.lla_forward_host_buffer_size(bf, ten, 2, 4, 300, 64, 3) == expect(bf, ten, 3, 300, 64)
    assert lib.lla_forward_host_buffer_size(bf, ten, 2, 4, 300, 64, 50) == expect(bf, ten, 8, 300, 64)
    assert lib.lla_forward_host_buffer_size(bf, ten, 2, 4, 300, 64, -1) == 0
    assert lib.lla_forward_host_buffer_size(bf, ten, 2, 4, 300, 48, 0) == 0


def test_host_binding_refuses_non_contiguous_inputs():
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 1, 8, 32)[..., ::2]
    with pytest.raises(lla.LLAError):
        lla.forward_host(x, x, x, 0.25, 0.1, 4)


def _call_bwd_host(lib, **kw):
    a = dict(dtype=0, path=0, q=16, k=32, v=48, rho=64, den=80, g=96, dq=112, dk=128, dv=144, it=None, B=1, H=1, n=8,
             d=64, tau=0.1, lam=1.0, T=4, tol=0.0, chunk=0, buf=None, bufb=0, stream=None)
    a.update(kw)
    return lib.lla_backward_host(a["dtype"], a["path"], a["q"], a["k"], a["v"], a["rho"], a["den"], a["g"], a["dq"],
                                 a["dk"], a["dv"], a["it"], a["B"], a["H"], a["n"], a["d"], a["tau"], a["lam"], a["T"],
                                 a["tol"], a["chunk"], a["buf"], a["bufb"], a["stream"])


@pytest.mark.parametrize("bad", [
    dict(q=None), dict(g=None), dict(rho=None), dict(den=None), dict(dq=None), dict(dv=None), dict(B=0), dict(n=0),
    dict(B=70000), dict(d=48), dict(tau=0.0), dict(lam=float("nan")), dict(T=0), dict(tol=-1.0), dict(dtype=7),
    dict(path=9), dict(chunk=-1), dict(buf=256, bufb=16), dict(buf=257, bufb=1 << 40),
])
def test_backward_host_invalid_arguments_rejected_before_launch(lib, bad):
    assert _call_bwd_host(lib, **bad) == lla.LLA_ERR_INVALID_ARG
    assert lib.lla_last_error().decode()


def test_backward_host_buffer_size(lib):
    """Two halves, each holding one chunk's q, k, v, dout, rho, dq, dk, dv, denom, cg_iters (each
    rounded up to 256 bytes) and the chunk's backward workspace."""
    def a256(x):
        return (x + 255) & ~255

    def expect(dtype, path, C, n, d):
        es = 2 if dtype == lla.LLA_DTYPE_BF16 else 4
        ws = lib.lla_backward_workspace_size(dtype, path, C, 1, n, d)
        return 2 * (4 * a256(C * n * d * es) + 4 * a256(C * n * d * 4) + 2 * a256(C * n * 4) + a256(ws))

    bf, f32, ten, fp = lla.LLA_DTYPE_BF16, lla.LLA_DTYPE_FP32, lla.LLA_PATH_TENSOR, lla.LLA_PATH_FP32
    assert lib.lla_backward_host_buffer_size(bf, ten, 8, 16, 256, 128, 0) == expect(bf, ten, 16, 256, 128)
    assert lib.lla_backward_host_buffer_size(f32, fp, 1, 3, 100, 32, 0) == expect(f32, fp, 1, 100, 32)
    assert lib.lla_backward_host_buffer_size(bf, ten, 2, 4, 300, 64, 3) == expect(bf, ten, 3, 300, 64)
    assert lib.lla_backward_host_buffer_size(bf, ten, 2, 4, 300, 64, -1) == 0
