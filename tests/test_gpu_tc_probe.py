"""tcgen05 descriptor/TMA/TMEM helpers checked on single 128x128x128 fp16 products
against torch fp32 matmul (the helpers the LLA tensor kernel is built from)."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

from tc_probe import build_probe


@pytest.fixture(scope="module")
def probe_lib():
    """The probe library, compiled for sm_103a on first use (a test fixture, not part of liblla)."""
    return ctypes.CDLL(build_probe.build())


def test_umma_descriptors_match_matmul(lla_gpu, probe_lib):
    lib = probe_lib
    lib.lla_probe_umma.restype = ctypes.c_int
    lib.lla_probe_umma.argtypes = [ctypes.c_void_p] * 6
    g = torch.Generator().manual_seed(0)
    dev = torch.device("cuda:0")
    A, B, B2 = (torch.randint(-8, 9, (128, 128), generator=g).to(torch.float16).to(dev) / 4 for _ in range(3))
    D = [torch.full((128, 128), float("nan"), device=dev) for _ in range(3)]
    rc = lib.lla_probe_umma(A.data_ptr(), B.data_ptr(), B2.data_ptr(), *(d.data_ptr() for d in D))
    torch.cuda.synchronize()
    assert rc == 0, rc
    Af, Bf, B2f = A.float(), B.float(), B2.float()
    want = [Af @ Bf.T, Af @ B2f, Af @ Bf.T]
    names = ["SS K-major (TMA A)", "TS MN-major B", "SS K-major (thread-written A)"]
    msgs = []
    for name, d, w in zip(names, D, want):
        err = (d - w).abs().max().item()
        if not err <= 1e-3:
            alt = {"A B2^T": (Af @ B2f.T), "A^T B": Af.T @ Bf, "(A B^T)^T": (Af @ Bf.T).T}
            close = [k for k, v in alt.items() if (d - v).abs().max().item() < 1e-3]
            msgs.append(f"{name}: max err {err} (matches {close})")
    assert not msgs, "; ".join(msgs)


def test_umma_mn_major_bf16_moment_product(lla_gpu, probe_lib):
    """The decode moment product's form: D[128 x 256] = At^T [K | V] with bf16 operands, A written
    by threads and B loaded by TMA, both MN-major (64-row boxes at an 8 KB stride), N = 256."""
    lib = probe_lib
    lib.lla_probe_umma_mn.restype = ctypes.c_int
    lib.lla_probe_umma_mn.argtypes = [ctypes.c_void_p] * 4
    g = torch.Generator().manual_seed(1)
    dev = torch.device("cuda:0")
    At, K, V = (torch.randint(-8, 9, (64, 128), generator=g).to(torch.bfloat16).to(dev) / 4 for _ in range(3))
    D = torch.full((128, 256), float("nan"), device=dev)
    rc = lib.lla_probe_umma_mn(At.data_ptr(), K.data_ptr(), V.data_ptr(), D.data_ptr())
    torch.cuda.synchronize()
    assert rc == 0, rc
    want = At.float().T @ torch.cat([K.float(), V.float()], dim=1)
    err = (D - want).abs().max().item()
    assert err <= 1e-3, f"MN-major bf16 product: max err {err}"
