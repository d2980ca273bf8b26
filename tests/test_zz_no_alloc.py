"""paged_decode_attention_noalloc against paged_decode_attention, through the C ABI.

The allocation-free entry point exists for callers that cannot allocate device
memory themselves -- frameworks or plugins that own all device memory, or
latency-critical loops where an allocation (which may synchronise the device) is
not allowed -- and so cannot hand paged_decode_attention the workspace its split
plan needs.  It runs the same kernels with that workspace in a fixed array inside
the library.  Here it must give the same output as the ordinary entry point (with
a caller workspace), within the tolerance the other GPU tests use, on two calls in
a row (the second call finds the first call's leftovers in the shared array).

This file is named to be collected last, so that a run stopping at the first
failure has run every other test before it; it also passes on its own.
"""

import ctypes

import pytest
import torch

from paged_kv_decode_mapping_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 2.0 ** -8


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_mapping_gb300 import build

    build.build()
    from paged_kv_decode_mapping_gb300 import binding

    return binding


def _noalloc(B, out, g):
    d = B.cache_desc(g["k_cache"])
    Bn, Hq, _ = g["q"].shape
    return B.lib().paged_decode_attention_noalloc(
        out.data_ptr(), g["q"].data_ptr(), g["k_cache"].data_ptr(), g["v_cache"].data_ptr(),
        g["block_tables"].data_ptr(), g["block_tables"].shape[1], g["context_lens"].data_ptr(),
        g["max_context_len"], Bn, Hq, ctypes.byref(d), g["scale"],
        torch.cuda.current_stream().cuda_stream)


def _with_workspace(B, g):
    out = torch.empty_like(g["q"])
    Bn, Hq, D = g["q"].shape
    need = B.paged_decode_workspace_size(Bn, Hq, g["k_cache"].shape[1], D, g["max_context_len"])
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
    B.paged_decode_attention(out, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                             g["context_lens"], g["max_context_len"], g["scale"], workspace=ws)
    return out, need


def test_noalloc_matches_workspace_entry_point_twice(B):
    cases = [
        W.small_workload(B=4, Hq=24, Hkv=8, D=128, BS=32, lens=(4096, 3000, 17, 2500), seed=41,
                         write="none"),
        W.small_workload(B=6, Hq=32, Hkv=8, D=64, BS=16, lens=(2048, 1, 700, 2047, 300, 1500),
                         seed=42, write="none"),
    ]
    for w in cases:  # two calls in a row on the shared scratch array
        inp = W.make_inputs(w, poison=True)
        g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
        ref, need = _with_workspace(B, g)
        assert 0 < need <= B.NOALLOC_SCRATCH_BYTES  # the decode really uses the scratch
        out = torch.full_like(g["q"], float("nan"))
        rc = _noalloc(B, out, g)
        assert rc == 0, B.pkv_last_error()
        torch.cuda.synchronize()
        got, want = out.cpu().double(), ref.cpu().double()
        assert torch.isfinite(got).all()
        err = (got - want).abs()
        assert bool((err <= ATOL + RTOL * want.abs()).all()), float(err.max())
    assert B.pkv_device_errors(clear=True) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(B):
    # a plan whose partition workspace exceeds the fixed array is refused up front
    # (one completion counter per (sequence, kv head): 65535 x 256 of them is 64 MiB)
    Bn, Hq, Hkv, D, L, BS = 65535, 256, 256, 64, 64, 64
    need = B.paged_decode_workspace_size(Bn, Hq, Hkv, D, L)
    assert need > B.NOALLOC_SCRATCH_BYTES
    d = B.pkv_cache_desc(16, BS, Hkv, D)
    fake = ctypes.c_void_p(1 << 20)
    rc = B.lib().paged_decode_attention_noalloc(fake, fake, fake, fake, fake, L // BS, fake, L, Bn,
                                                Hq, ctypes.byref(d), 0.1, None)
    assert rc == -4 and "scratch" in B.pkv_last_error()
