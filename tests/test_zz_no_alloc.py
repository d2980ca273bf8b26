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


def _cudart():
    # the CUDA runtime libpkv.so is linked against (already loaded, found by its soname)
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            return ctypes.CDLL(name)
        except OSError:
            continue
    pytest.skip("libcudart not loadable by name")


def _captured_nodes(rt, stream, fn) -> int:
    """Runs fn() while `stream` is being captured into a CUDA graph (relaxed mode) and
    returns how many nodes the graph got.  Nothing captured is ever launched."""
    assert rt.cudaStreamBeginCapture(ctypes.c_void_p(stream.cuda_stream), 2) == 0
    try:
        fn()
    finally:
        graph = ctypes.c_void_p()
        assert rt.cudaStreamEndCapture(ctypes.c_void_p(stream.cuda_stream), ctypes.byref(graph)) == 0
    n = ctypes.c_size_t(0)
    assert rt.cudaGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    assert rt.cudaGraphDestroy(graph) == 0
    return int(n.value)


def test_noalloc_refused_calls_enqueue_nothing(B):
    """Arguments the launcher cannot plan (head_dim 96, a query group over 8) with
    65535 x 256 (sequence, kv head) units -- enough counters that clearing them would
    overrun the fixed array twice over -- are refused before anything reaches the
    stream: captured on a side stream, the refused calls add no node to the graph,
    while an accepted call adds its clear and its kernel."""
    rt = _cudart()
    w = W.small_workload(B=2, Hq=8, Hkv=2, D=64, BS=16, lens=(900, 40), seed=44, write="none")
    g = {k: (v.cuda() if isinstance(v, torch.Tensor) else v)
         for k, v in W.make_inputs(w).items()}
    out = torch.empty_like(g["q"])
    assert _noalloc(B, out, g) == 0  # first call on this device: set-up outside capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    fake = ctypes.c_void_p(1 << 20)

    def refused():
        for hkv, d in ((256, 96), (16, 64)):
            desc = B.pkv_cache_desc(16, 16, hkv, d)
            rc = B.lib().paged_decode_attention_noalloc(fake, fake, fake, fake, fake, 4, fake, 64,
                                                        65535, 256, ctypes.byref(desc), 0.1,
                                                        ctypes.c_void_p(s.cuda_stream))
            assert rc == -3, (hkv, d, rc)

    def accepted():
        d = B.cache_desc(g["k_cache"])
        rc = B.lib().paged_decode_attention_noalloc(
            out.data_ptr(), g["q"].data_ptr(), g["k_cache"].data_ptr(), g["v_cache"].data_ptr(),
            g["block_tables"].data_ptr(), g["block_tables"].shape[1], g["context_lens"].data_ptr(),
            g["max_context_len"], 2, 8, ctypes.byref(d), g["scale"], ctypes.c_void_p(s.cuda_stream))
        assert rc == 0, B.pkv_last_error()

    assert _captured_nodes(rt, s, refused) == 0
    assert _captured_nodes(rt, s, accepted) >= 2
    torch.cuda.synchronize()
    assert B.pkv_device_errors(clear=True) == 0
