"""The FMA-pipe 2^x of the prefill softmax (csrc/pkv_exp2.cuh): cubic minimax
polynomial after reduction to the nearest integer.

CPU: the header's coefficients, evaluated in float64 on [-1/2, 1/2], keep the relative
error the header states (7.5e-5), and the error equioscillates (the minimax property).
GPU: the device function against CUDA's exp2f over the whole range the softmax uses,
including the clamp below -125 and NaN.
"""

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_decode_mapping_gb300", "csrc")
HEADER = os.path.join(CSRC, "pkv_exp2.cuh")
BOUND = 7.5e-5


def coefficients():
    text = open(HEADER).read()
    cs = [float.fromhex(re.search(rf"kExp2C{i} = (0x[0-9a-fA-F.p+-]+)f;", text).group(1))
          for i in range(4)]
    return np.array(cs, dtype=np.float32).astype(np.float64)


def test_polynomial_error_bound_and_equioscillation():
    c = coefficients()
    f = np.linspace(-0.5, 0.5, 400001)
    rel = (((c[3] * f + c[2]) * f + c[1]) * f + c[0]) / np.exp2(f) - 1.0
    assert np.abs(rel).max() <= BOUND
    # minimax of degree 3: the error alternates sign at 5 extrema of equal size
    ext = [np.abs(rel[(f >= lo) & (f <= hi)]).max()
           for lo, hi in ((-0.5, -0.45), (-0.35, -0.1), (-0.1, 0.2), (0.2, 0.45), (0.45, 0.5))]
    assert max(ext) / min(ext) < 1.05, ext


@pytest.mark.gpu
def test_device_exp2_fma_against_exp2f(tmp_path):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    so = tmp_path / "exp2_probe.so"
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                    "-Xcompiler", "-fPIC", "-I", CSRC, os.path.join(ROOT, "tests", "exp2_probe.cu"),
                    "-o", str(so)], check=True)
    lib = ctypes.CDLL(str(so))
    lib.exp2_probe.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int]
    x = torch.cat([torch.linspace(-125.0, 126.0, 2_000_001), torch.linspace(-8.0, 8.0, 1_000_001),
                   torch.tensor([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 126.9, -124.99])]).cuda()
    poly, ref = torch.empty_like(x), torch.empty_like(x)
    assert lib.exp2_probe(x.data_ptr(), poly.data_ptr(), ref.data_ptr(), x.numel()) == 0
    rel = (poly.double() / ref.double() - 1.0).abs()
    assert float(rel.max()) <= BOUND + 2.0 ** -22, float(rel.max())
    # below the clamp, and NaN: 2^-125 (a normal float), never a NaN or a wrapped exponent
    lo = torch.tensor([-126.0, -200.0, -1e30, float("-inf"), float("nan")]).cuda()
    out_p, out_r = torch.empty_like(lo), torch.empty_like(lo)
    assert lib.exp2_probe(lo.data_ptr(), out_p.data_ptr(), out_r.data_ptr(), lo.numel()) == 0
    want = torch.full_like(lo, 2.0 ** -125)
    assert torch.allclose(out_p, want, rtol=BOUND, atol=0.0), out_p
