"""Build the test-only tcgen05 probe library (liblla_probe.so) next to this file.

The probe checks the UMMA descriptor encodings and the TMA/TMEM helpers of the tensor kernels on
single 128x128x128 fp16 products.  It is a test fixture, not part of the library: it includes the
package's device helpers (csrc/tc_ptx.cuh, csrc/tc_host.h) and is compiled for sm_103a on demand
by the test that uses it.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
CSRC = os.path.join(ROOT, "local_linear_attention_flashlla_gb300", "csrc")
OUT = os.path.join(HERE, "_build", "liblla_probe.so")


def build():
    """Compile lla_probe.cu into _build/liblla_probe.so; returns its path."""
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    from local_linear_attention_flashlla_gb300.build import ARCH, nvcc_path
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    tmp = OUT + ".tmp"
    cmd = [nvcc_path(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + CSRC, "-I" + HERE,
           "-shared", os.path.join(HERE, "lla_probe.cu"), "-o", tmp, "-lcudart"]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("probe build failed (%d):\n%s" % (r.returncode, r.stdout))
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build())
