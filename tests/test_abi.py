"""The C ABI without a GPU: the library loads, exports every declared symbol, and
rejects bad arguments on the host before touching the device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "paged_kv.h")


@pytest.fixture(scope="module")
def B():
    from paged_kv_decode_mapping_gb300 import build

    build.build()
    from paged_kv_decode_mapping_gb300 import binding

    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("paged_kv_write", "paged_decode_attention", "paged_decode_split",
              "paged_decode_combine", "paged_decode_plan", "paged_decode_workspace_size",
              "paged_decode_split_workspace_size", "pkv_device_errors", "pkv_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(B):
    lib = B.lib()
    for n in declared_functions():
        assert hasattr(lib, n), f"libpkv.so does not export {n}"


def test_library_exports_nothing_else(B):
    out = os.popen(f"nm -D --defined-only {B.LIB_PATH}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(declared_functions()), exported ^ set(declared_functions())


FAKE = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced by the host checks


def _desc(B, nb=64, bs=16, hkv=2, d=64):
    return B.pkv_cache_desc(nb, bs, hkv, d)


def _attn(B, desc, hq=8, max_len=100, max_blocks=8, ws=None, ws_bytes=0, out=FAKE):
    return B.lib().paged_decode_attention(out, FAKE, FAKE, FAKE, FAKE, max_blocks, FAKE, max_len, 2,
                                          hq, ctypes.byref(desc), 0.125, ws, ws_bytes, None)


def test_attention_argument_errors(B):
    lib = B.lib()
    assert _attn(B, _desc(B, d=96)) == -3 and "head_dim" in B.pkv_last_error()
    assert _attn(B, _desc(B, bs=12)) == -3
    assert _attn(B, _desc(B, bs=512)) == -3
    assert _attn(B, _desc(B), hq=7) == -2          # not a multiple of num_kv_heads
    assert _attn(B, _desc(B, hkv=1), hq=16) == -3  # group of 16 > 8
    assert _attn(B, _desc(B), max_len=200) == -2   # over max_blocks * block_size
    assert _attn(B, _desc(B, nb=0)) == -2
    assert _attn(B, _desc(B), out=None) == -1
    assert _attn(B, _desc(B), out=ctypes.c_void_p((1 << 20) + 2)) == -5
    assert lib.paged_decode_attention(FAKE, ctypes.c_void_p((1 << 20) + 4), FAKE, FAKE, FAKE, 8,
                                      FAKE, 100, 2, 8, ctypes.byref(_desc(B)), 0.1, None, 0, None) == -5
    assert lib.paged_decode_attention(FAKE, FAKE, FAKE, FAKE, FAKE, 8, FAKE, 100, 2, 8, None, 0.1,
                                      None, 0, None) == -1
    # a split plan without enough workspace is refused before any launch
    assert _attn(B, _desc(B, hkv=1), hq=8, max_len=4096, max_blocks=256) == -4
    assert "workspace" in B.pkv_last_error()


def test_split_and_combine_argument_errors(B):
    lib = B.lib()
    d = _desc(B)
    args = (FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, FAKE, 100, 2, 8, ctypes.byref(d), 0.1)
    assert lib.paged_decode_split(*args, 100, None) == -2  # not a multiple of 64
    assert lib.paged_decode_split(*args, 0, None) == -2
    assert lib.paged_decode_split(None, FAKE, *args[2:], 64, None) == -1
    assert lib.paged_decode_combine(FAKE, FAKE, FAKE, FAKE, 100, 2, 8, 80, 64, None) == -3
    assert lib.paged_decode_combine(FAKE, FAKE, FAKE, FAKE, 100, 2, 8, 64, 0, None) == -2
    assert lib.paged_decode_combine(FAKE, None, FAKE, FAKE, 100, 2, 8, 64, 64, None) == -1


def test_write_argument_errors(B):
    lib = B.lib()
    d = _desc(B, d=60)
    assert lib.paged_kv_write(FAKE, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(d), None) == -3
    d = _desc(B)
    assert lib.paged_kv_write(FAKE, FAKE, FAKE, -1, FAKE, FAKE, ctypes.byref(d), None) == -2
    assert lib.paged_kv_write(None, FAKE, FAKE, 4, FAKE, FAKE, ctypes.byref(d), None) == -1
    assert lib.paged_kv_write(FAKE, FAKE, ctypes.c_void_p((1 << 20) + 4), 4, FAKE, FAKE,
                              ctypes.byref(d), None) == -5
    assert lib.paged_kv_write(FAKE, FAKE, FAKE, 4, FAKE, FAKE, None, None) == -1
    # zero tokens is a no-op that succeeds without a device
    assert lib.paged_kv_write(None, None, None, 0, None, None, ctypes.byref(d), None) == 0


def test_rope_step_argument_errors(B):
    lib = B.lib()
    d = _desc(B)

    def call(rotary_dim=64, positions=FAKE, cos_sin=FAKE, desc=d, out=FAKE):
        # out, q, k, v, slots, positions, cos_sin, max_position, rotary_dim, neox,
        # k_cache, v_cache, tables, max_blocks, lens, max_len, num_seqs, hq, desc, scale,
        # workspace, bytes, stream
        return lib.paged_decode_step_rope(out, FAKE, FAKE, FAKE, FAKE, positions, cos_sin, 128,
                                          rotary_dim, 1, FAKE, FAKE, FAKE, 8, FAKE, 100, 2, 8,
                                          ctypes.byref(desc), 0.125, None, 0, None)

    assert call(rotary_dim=24) == -3 and "rotary_dim" in B.pkv_last_error()
    assert call(rotary_dim=128) == -3                   # more than head_dim
    assert call(positions=None) == -1
    assert call(cos_sin=None) == -1
    assert call(cos_sin=ctypes.c_void_p((1 << 20) + 4)) == -5
    assert call(desc=_desc(B, d=96)) == -3
    assert call(out=None) == -1


def test_prefill_argument_errors(B):
    lib = B.lib()
    d = _desc(B)

    def call(out=FAKE, qs=FAKE, max_len=100, max_q=16, desc=d):
        return lib.paged_prefill_attention(out, FAKE, FAKE, FAKE, FAKE, 8, FAKE, max_len, qs, max_q,
                                           2, 8, ctypes.byref(desc), 0.125, None)

    assert call(max_q=101) == -2                          # more queries than context
    assert call(qs=None) == -1
    assert call(out=None) == -1
    assert call(out=ctypes.c_void_p((1 << 20) + 8)) == -5  # 8-byte aligned: not enough
    assert call(desc=_desc(B, d=96)) == -3
    assert call(max_q=0) == 0                             # nothing to do


def test_empty_batch_is_a_no_op(B):
    lib = B.lib()
    d = _desc(B)
    assert lib.paged_decode_attention(None, None, None, None, None, 8, None, 0, 0, 8,
                                      ctypes.byref(d), 0.1, None, 0, None) == 0


def test_noalloc_refuses_bad_arguments_before_any_device_work(B):
    """The allocation-free decode runs every host check before it touches its fixed
    scratch array.  Shapes the launcher cannot plan (workspace size 0) used to slip past
    the size check into a clear of num_seqs * num_kv_heads counters; with 65535 x 256
    of them that clear alone would be 64 MiB, twice the array.  Each must come back
    with an error on the host (no GPU here: any device work would fail differently)."""
    lib = B.lib()

    def call(desc, hq, n=65535, max_len=64, max_blocks=4, out=FAKE, q=FAKE):
        return lib.paged_decode_attention_noalloc(out, q, FAKE, FAKE, FAKE, max_blocks, FAKE,
                                                  max_len, n, hq, ctypes.byref(desc), 0.1, None)

    assert B.paged_decode_workspace_size(65535, 256, 256, 96, 64) == 0
    assert call(_desc(B, hkv=256, d=96), 256) == -3 and "head_dim" in B.pkv_last_error()
    assert call(_desc(B, hkv=16), 256) == -3 and "group" in B.pkv_last_error()   # group 16
    assert call(_desc(B, hkv=3), 256) == -2                                        # 256 % 3
    assert call(_desc(B, hkv=8), 64, n=70000) in (-3, -4)                          # > 65535 sequences
    assert call(_desc(B, hkv=2), 8, n=2, out=None) == -1
    assert call(_desc(B, hkv=2), 8, n=2, q=ctypes.c_void_p((1 << 20) + 4)) == -5
    assert call(_desc(B, hkv=2), 8, n=2, max_len=100) == -2                       # over the table
    assert call(_desc(B, hkv=2), 8, n=0, out=None, q=None) == 0                   # nothing to do


def test_ctas_per_sm_rejects_unknown_shapes_without_a_device(B):
    """pkv_decode_ctas_per_sm refuses a head_dim or an arrangement it has no kernel for,
    on the host, before asking the CUDA runtime anything."""
    lib = B.lib()
    assert lib.pkv_decode_ctas_per_sm(96, B.PATH_PERSISTENT) == -3
    assert lib.pkv_decode_ctas_per_sm(64, 7) == -3
    assert lib.pkv_decode_ctas_per_sm(128, 0) == -3


def test_pinned_host_tensors_are_accepted_only_where_documented(B):
    """The binding lets pinned host tensors through for the per-step decode arguments and
    nowhere else (the caches stay device memory); pageable host tensors are refused."""
    import torch

    q = torch.zeros(2, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="pinned host memory"):
        B._need(q, "q", torch.bfloat16, 3, True)  # pageable
    with pytest.raises(ValueError, match="must be a CUDA tensor$"):
        B._need(q, "k_cache", torch.bfloat16, 3)
