"""Thin ctypes binding of libpkv.so: argument marshalling only.

Every function has the name of the C entry point it calls (``include/paged_kv.h``),
takes torch CUDA tensors, checks their dtypes/shapes/contiguity, and passes raw
device pointers, sizes and the current CUDA stream.  All computation happens in
the library's kernels; there is no fallback.  Importing this module raises if
``libpkv.so`` has not been built.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpkv.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(LIB_PATH)

PKV_OK = 0
ERRORS = {-1: "PKV_ERR_NULL", -2: "PKV_ERR_SHAPE", -3: "PKV_ERR_UNSUPPORTED",
          -4: "PKV_ERR_WORKSPACE", -5: "PKV_ERR_ALIGN", -6: "PKV_ERR_CUDA", -7: "PKV_ERR_DEVICE",
          -8: "PKV_ERR_NOSPACE"}
DEVERR = {1: "BLOCK_ID", 2: "SLOT", 4: "CONTEXT_LEN", 8: "TIMEOUT", 16: "POSITION"}


class PkvError(RuntimeError):
    def __init__(self, code: int, where: str):
        msg = _lib.pkv_last_error().decode(errors="replace")
        super().__init__(f"{where}: {ERRORS.get(code, code)}: {msg}")
        self.code = code


class pkv_cache_desc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


_P = ctypes.c_void_p
_i32, _i64, _f32, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_D = ctypes.POINTER(pkv_cache_desc)

_lib.paged_kv_write.argtypes = [_P, _P, _P, _i64, _P, _P, _D, _P]
_lib.paged_kv_write.restype = ctypes.c_int
_lib.paged_kv_write_rope.argtypes = [_P, _P, _P, _i32, _P, _P, _i64, _P, _i64, _i32, _i32, _P, _P,
                                     _D, _P]
_lib.paged_kv_write_rope.restype = ctypes.c_int
_lib.paged_decode_plan.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
_lib.paged_decode_plan.restype = _i32
_lib.paged_decode_path.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
_lib.paged_decode_path.restype = _i32
_lib.pkv_set_decode_consumer.argtypes = [_i32]
_lib.pkv_set_decode_consumer.restype = _i32
_lib.pkv_decode_ctas_per_sm.argtypes = [_i32, _i32]
_lib.pkv_decode_ctas_per_sm.restype = _i32
_lib.paged_decode_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32]
_lib.paged_decode_workspace_size.restype = _sz
_lib.paged_decode_split_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32]
_lib.paged_decode_split_workspace_size.restype = _sz
_lib.paged_decode_attention.argtypes = [_P, _P, _P, _P, _P, _i32, _P, _i32, _i32, _i32, _D, _f32,
                                        _P, _sz, _P]
_lib.paged_decode_attention.restype = ctypes.c_int
_lib.paged_decode_step.argtypes = [_P, _P, _P, _P, _P, _i64, _P, _P, _P, _i32, _P, _i32, _i32,
                                   _i32, _D, _f32, _P, _sz, _P]
_lib.paged_decode_step.restype = ctypes.c_int
_lib.paged_decode_step_rope.argtypes = [_P, _P, _P, _P, _P, _P, _P, _i64, _i32, _i32, _P, _P, _P,
                                        _i32, _P, _i32, _i32, _i32, _D, _f32, _P, _sz, _P]
_lib.paged_decode_step_rope.restype = ctypes.c_int
_lib.paged_prefill_attention.argtypes = [_P, _P, _P, _P, _P, _i32, _P, _i32, _P, _i32, _i32, _i32,
                                         _D, _f32, _P]
_lib.paged_prefill_attention.restype = ctypes.c_int
_lib.paged_decode_split.argtypes = [_P, _P, _P, _P, _P, _P, _i32, _P, _i32, _i32, _i32, _D, _f32,
                                    _i32, _P]
_lib.paged_decode_split.restype = ctypes.c_int
_lib.paged_decode_combine.argtypes = [_P, _P, _P, _P, _i32, _i32, _i32, _i32, _i32, _P]
_lib.paged_decode_combine.restype = ctypes.c_int
_lib.paged_decode_attention_noalloc.argtypes = [_P, _P, _P, _P, _P, _i32, _P, _i32, _i32, _i32,
                                                _D, _f32, _P]
_lib.paged_decode_attention_noalloc.restype = ctypes.c_int
NOALLOC_SCRATCH_BYTES = 32 << 20  # PKV_NOALLOC_SCRATCH_BYTES in include/paged_kv.h
_lib.pkv_bm_create.argtypes = [_i64, _i32]
_lib.pkv_bm_create.restype = _P
_lib.pkv_bm_destroy.argtypes = [_P]
_lib.pkv_bm_destroy.restype = None
_lib.pkv_bm_num_free_blocks.argtypes = [_P]
_lib.pkv_bm_num_free_blocks.restype = _i64
_lib.pkv_bm_add_sequence.argtypes = [_P, _i64, _i64]
_lib.pkv_bm_add_sequence.restype = ctypes.c_int
_lib.pkv_bm_append_slots.argtypes = [_P, _P, _i32, _P]
_lib.pkv_bm_append_slots.restype = ctypes.c_int
_lib.pkv_bm_free_sequence.argtypes = [_P, _i64]
_lib.pkv_bm_free_sequence.restype = ctypes.c_int
_lib.pkv_bm_preempt_lifo.argtypes = [_P, ctypes.POINTER(ctypes.c_int64)]
_lib.pkv_bm_preempt_lifo.restype = ctypes.c_int
_lib.pkv_bm_block_tables.argtypes = [_P, _P, _i32, _i32, _P, _P]
_lib.pkv_bm_block_tables.restype = ctypes.c_int
_lib.pkv_device_errors.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
_lib.pkv_device_errors.restype = ctypes.c_int
_lib.pkv_last_error.argtypes = []
_lib.pkv_last_error.restype = ctypes.c_char_p


def lib() -> ctypes.CDLL:
    return _lib


def _check(rc: int, where: str):
    if rc != PKV_OK:
        raise PkvError(rc, where)


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype, ndim: int, host_ok: bool = False):
    """host_ok: a page-locked CPU tensor is accepted too (the kernels address it directly)."""
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got shape {tuple(t.shape)}")
    if not t.is_cuda and not (host_ok and t.is_pinned()):
        raise ValueError(f"{name}: must be a CUDA tensor" + (" or pinned host memory" if host_ok else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def cache_desc(k_cache: torch.Tensor) -> pkv_cache_desc:
    NB, Hkv, BS, D = k_cache.shape
    return pkv_cache_desc(NB, BS, Hkv, D)


def paged_kv_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor, stream=None) -> None:
    """k/v [T, Hkv, D] bf16 are copied into k_cache/v_cache [NB, Hkv, BS, D] at their slots
    (k, v and slot_mapping may be pinned host tensors)."""
    _need(k, "k", torch.bfloat16, 3, True)
    _need(v, "v", torch.bfloat16, 3, True)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, True)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    if k.shape != v.shape or k_cache.shape != v_cache.shape:
        raise ValueError("k/v or k_cache/v_cache shapes differ")
    if k.shape[0] != slot_mapping.shape[0] or tuple(k.shape[1:]) != (k_cache.shape[1], k_cache.shape[3]):
        raise ValueError("k [T, Hkv, D] does not match slot_mapping [T] / cache [NB, Hkv, BS, D]")
    d = cache_desc(k_cache)
    _check(_lib.paged_kv_write(_ptr(k), _ptr(v), _ptr(slot_mapping), k.shape[0], _ptr(k_cache),
                               _ptr(v_cache), ctypes.byref(d), _stream(stream)), "paged_kv_write")


def paged_kv_write_rope(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                        positions: torch.Tensor, cos_sin: torch.Tensor, k_cache: torch.Tensor,
                        v_cache: torch.Tensor, q: Optional[torch.Tensor] = None,
                        rotary_dim: Optional[int] = None, neox_style: bool = True,
                        stream=None) -> None:
    """RoPE of k (and q, in place) at `positions`, then the slot write of k and v."""
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(positions, "positions", torch.int64, 1)
    _need(cos_sin, "cos_sin", torch.float32, 2)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    if q is not None:
        _need(q, "q", torch.bfloat16, 3)
        if q.shape[0] != k.shape[0] or q.shape[2] != k.shape[2]:
            raise ValueError("q must be [T, Hq, D] with k's T and D")
    r = k.shape[2] if rotary_dim is None else int(rotary_dim)
    if cos_sin.shape[1] != r:
        raise ValueError("cos_sin must be [max_position, rotary_dim]")
    if not (k.shape[0] == slot_mapping.shape[0] == positions.shape[0]):
        raise ValueError("k, slot_mapping and positions must have the same number of tokens")
    d = cache_desc(k_cache)
    _check(_lib.paged_kv_write_rope(_ptr(k), _ptr(v), _ptr(q), 0 if q is None else q.shape[1],
                                    _ptr(slot_mapping), _ptr(positions), k.shape[0], _ptr(cos_sin),
                                    cos_sin.shape[0], r, 1 if neox_style else 0, _ptr(k_cache),
                                    _ptr(v_cache), ctypes.byref(d), _stream(stream)),
           "paged_kv_write_rope")


PATH_PARTITIONS, PATH_CLUSTER, PATH_PERSISTENT = 1, 2, 3
CONSUMER_TENSOR, CONSUMER_FMA = 0, 1


def pkv_set_decode_consumer(consumer: int) -> int:
    """Selects the consumer warps' arithmetic of the partition decode kernel (CONSUMER_*);
    returns the previous one."""
    rc = int(_lib.pkv_set_decode_consumer(consumer))
    if rc < 0:
        _check(rc, "pkv_set_decode_consumer")
    return rc


def pkv_decode_ctas_per_sm(head_dim: int, path: int) -> int:
    """CTAs per SM of the decode kernel of `path` (PATH_*) on the current device."""
    n = int(_lib.pkv_decode_ctas_per_sm(head_dim, path))
    if n < 0:
        _check(n, "pkv_decode_ctas_per_sm")
    return n


def paged_decode_path(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                      max_context_len: int, num_sms: int = 0) -> int:
    """Kernel arrangement paged_decode_attention launches for these sizes (PATH_*; 0 if none)."""
    return int(_lib.paged_decode_path(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      max_context_len, num_sms))


def paged_decode_plan(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                      max_context_len: int, num_sms: int = 0) -> int:
    """Partition size (tokens) paged_decode_attention cuts each (sequence, kv head) into."""
    return int(_lib.paged_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      max_context_len, num_sms))


def paged_decode_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                                max_context_len: int) -> int:
    return int(_lib.paged_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                max_context_len))


def paged_decode_split_workspace_size(num_seqs: int, num_q_heads: int, head_dim: int,
                                      max_context_len: int, partition_tokens: int) -> int:
    return int(_lib.paged_decode_split_workspace_size(num_seqs, num_q_heads, head_dim,
                                                      max_context_len, partition_tokens))


def _decode_checks(q, k_cache, v_cache, block_tables, context_lens, host_ok=False):
    _need(q, "q", torch.bfloat16, 3, host_ok)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2, host_ok)
    _need(context_lens, "context_lens", torch.int32, 1, host_ok)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    B = q.shape[0]
    if block_tables.shape[0] != B or context_lens.shape[0] != B or q.shape[2] != k_cache.shape[3]:
        raise ValueError("q [B, Hq, D], block_tables [B, M], context_lens [B], cache [NB, Hkv, BS, D] disagree")


def paged_decode_attention(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                           v_cache: torch.Tensor, block_tables: torch.Tensor,
                           context_lens: torch.Tensor, max_context_len: int, scale: float,
                           workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """out [B, Hq, D] bf16 = paged GQA decode attention (split + combine when the plan says so).

    ``workspace`` (uint8, CUDA, zero-filled before its first use) may be omitted; then a
    zeroed buffer of ``paged_decode_workspace_size`` bytes is taken from torch's allocator.
    out, q, block_tables and context_lens may be pinned host tensors (read and written
    by the kernels over the host link).
    """
    _decode_checks(q, k_cache, v_cache, block_tables, context_lens, host_ok=True)
    _need(out, "out", torch.bfloat16, 3, True)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    B, Hq, D = q.shape
    need = paged_decode_workspace_size(B, Hq, k_cache.shape[1], D, max_context_len)
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=k_cache.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    d = cache_desc(k_cache)
    _check(_lib.paged_decode_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(block_tables), block_tables.shape[1],
                                       _ptr(context_lens), int(max_context_len), B, Hq,
                                       ctypes.byref(d), float(scale), _ptr(workspace), ws_bytes,
                                       _stream(stream)), "paged_decode_attention")


def paged_decode_step(out: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                      slot_mapping: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor,
                      max_context_len: int, scale: float, workspace: Optional[torch.Tensor] = None,
                      stream=None) -> None:
    """One decode step: the slot write of k/v, then attention over the updated caches.
    out, q, k, v, slot_mapping, block_tables and context_lens may be pinned host tensors:
    the kernels then read and write them over the host link (no copies)."""
    _decode_checks(q, k_cache, v_cache, block_tables, context_lens, host_ok=True)
    _need(out, "out", torch.bfloat16, 3, True)
    _need(k, "k", torch.bfloat16, 3, True)
    _need(v, "v", torch.bfloat16, 3, True)
    _need(slot_mapping, "slot_mapping", torch.int64, 1, True)
    if out.shape != q.shape or k.shape != v.shape or k.shape[0] != slot_mapping.shape[0]:
        raise ValueError("out/q, k/v or slot_mapping shapes disagree")
    B, Hq, D = q.shape
    need = paged_decode_workspace_size(B, Hq, k_cache.shape[1], D, max_context_len)
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=k_cache.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    d = cache_desc(k_cache)
    _check(_lib.paged_decode_step(_ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(slot_mapping),
                                  k.shape[0], _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                  block_tables.shape[1], _ptr(context_lens), int(max_context_len),
                                  B, Hq, ctypes.byref(d), float(scale), _ptr(workspace), ws_bytes,
                                  _stream(stream)), "paged_decode_step")


def paged_decode_step_rope(out: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                           slot_mapping: torch.Tensor, positions: torch.Tensor,
                           cos_sin: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                           block_tables: torch.Tensor, context_lens: torch.Tensor,
                           max_context_len: int, scale: float, rotary_dim: Optional[int] = None,
                           neox_style: bool = True, workspace: Optional[torch.Tensor] = None,
                           stream=None) -> None:
    """One decode step with RoPE: rotate q (in place) and k at `positions`, write k/v at
    their slots, then attention over the updated caches.  Token b is sequence b's."""
    _decode_checks(q, k_cache, v_cache, block_tables, context_lens)
    _need(out, "out", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 3)
    _need(v, "v", torch.bfloat16, 3)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(positions, "positions", torch.int64, 1)
    _need(cos_sin, "cos_sin", torch.float32, 2)
    B, Hq, D = q.shape
    if out.shape != q.shape or k.shape != v.shape or k.shape[0] != B or k.shape[2] != D:
        raise ValueError("out/q, k/v shapes disagree (one new token per sequence)")
    if not (slot_mapping.shape[0] == positions.shape[0] == B):
        raise ValueError("slot_mapping and positions need one entry per sequence")
    r = D if rotary_dim is None else int(rotary_dim)
    if cos_sin.shape[1] != r:
        raise ValueError("cos_sin must be [max_position, rotary_dim]")
    need = paged_decode_workspace_size(B, Hq, k_cache.shape[1], D, max_context_len)
    if workspace is None and need > 0:
        workspace = torch.zeros(need, dtype=torch.uint8, device=k_cache.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    d = cache_desc(k_cache)
    _check(_lib.paged_decode_step_rope(_ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(slot_mapping),
                                       _ptr(positions), _ptr(cos_sin), cos_sin.shape[0], r,
                                       1 if neox_style else 0, _ptr(k_cache), _ptr(v_cache),
                                       _ptr(block_tables), block_tables.shape[1],
                                       _ptr(context_lens), int(max_context_len), B, Hq,
                                       ctypes.byref(d), float(scale), _ptr(workspace), ws_bytes,
                                       _stream(stream)), "paged_decode_step_rope")


def paged_prefill_attention(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                            v_cache: torch.Tensor, block_tables: torch.Tensor,
                            context_lens: torch.Tensor, max_context_len: int,
                            query_start: torch.Tensor, max_query_len: int, scale: float,
                            stream=None) -> None:
    """Causal attention of each sequence's last n_b cached tokens (packed q [Nq, Hq, D])."""
    _need(q, "q", torch.bfloat16, 3)
    _need(out, "out", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(query_start, "query_start", torch.int32, 1)
    B = context_lens.shape[0]
    if out.shape != q.shape or query_start.shape[0] != B + 1 or block_tables.shape[0] != B:
        raise ValueError("out/q, query_start [B+1] or block_tables [B, M] disagree")
    d = cache_desc(k_cache)
    _check(_lib.paged_prefill_attention(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(block_tables), block_tables.shape[1],
                                        _ptr(context_lens), int(max_context_len),
                                        _ptr(query_start), int(max_query_len), B, q.shape[1],
                                        ctypes.byref(d), float(scale), _stream(stream)),
           "paged_prefill_attention")


def paged_decode_attention_noalloc(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                   v_cache: torch.Tensor, block_tables: torch.Tensor,
                                   context_lens: torch.Tensor, max_context_len: int, scale: float,
                                   stream=None) -> None:
    """paged_decode_attention without a workspace: the library's fixed scratch array is used."""
    _decode_checks(q, k_cache, v_cache, block_tables, context_lens)
    _need(out, "out", torch.bfloat16, 3)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    B, Hq, D = q.shape
    d = cache_desc(k_cache)
    _check(_lib.paged_decode_attention_noalloc(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                               _ptr(block_tables), block_tables.shape[1],
                                               _ptr(context_lens), int(max_context_len), B, Hq,
                                               ctypes.byref(d), float(scale), _stream(stream)),
           "paged_decode_attention_noalloc")


def paged_decode_split(o_part: torch.Tensor, lse_part: torch.Tensor, q: torch.Tensor,
                       k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                       context_lens: torch.Tensor, max_context_len: int, scale: float,
                       partition_tokens: int, stream=None) -> None:
    """o_part [B, Hq, n, D] fp32 and lse_part [B, Hq, n] fp32 for n = ceil(max_len / P)."""
    _decode_checks(q, k_cache, v_cache, block_tables, context_lens)
    _need(o_part, "o_part", torch.float32, 4)
    _need(lse_part, "lse_part", torch.float32, 3)
    B, Hq, D = q.shape
    n = -(-int(max_context_len) // int(partition_tokens)) if partition_tokens > 0 else 0
    if tuple(o_part.shape) != (B, Hq, n, D) or tuple(lse_part.shape) != (B, Hq, n):
        raise ValueError(f"o_part must be {(B, Hq, n, D)} and lse_part {(B, Hq, n)}")
    d = cache_desc(k_cache)
    _check(_lib.paged_decode_split(_ptr(o_part), _ptr(lse_part), _ptr(q), _ptr(k_cache),
                                   _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                                   _ptr(context_lens), int(max_context_len), B, Hq,
                                   ctypes.byref(d), float(scale), int(partition_tokens),
                                   _stream(stream)), "paged_decode_split")


def paged_decode_combine(out: torch.Tensor, o_part: torch.Tensor, lse_part: torch.Tensor,
                         context_lens: torch.Tensor, max_context_len: int, partition_tokens: int,
                         stream=None) -> None:
    _need(out, "out", torch.bfloat16, 3)
    _need(o_part, "o_part", torch.float32, 4)
    _need(lse_part, "lse_part", torch.float32, 3)
    _need(context_lens, "context_lens", torch.int32, 1)
    B, Hq, D = out.shape
    _check(_lib.paged_decode_combine(_ptr(out), _ptr(o_part), _ptr(lse_part), _ptr(context_lens),
                                     int(max_context_len), B, Hq, D, int(partition_tokens),
                                     _stream(stream)), "paged_decode_combine")


def pkv_device_errors(clear: bool = True) -> int:
    """Synchronises the device and returns the device error bits (PKV_DEVERR_*)."""
    f = ctypes.c_uint32(0)
    _check(_lib.pkv_device_errors(ctypes.byref(f), 1 if clear else 0), "pkv_device_errors")
    return int(f.value)


def pkv_last_error() -> str:
    return _lib.pkv_last_error().decode(errors="replace")


class BlockManager:
    """The library's host block allocator (pkv_bm_*): block tables and slot mappings."""

    def __init__(self, num_blocks: int, block_size: int):
        self._h = _lib.pkv_bm_create(int(num_blocks), int(block_size))
        if not self._h:
            raise PkvError(-2, "pkv_bm_create")
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            _lib.pkv_bm_destroy(h)

    @property
    def num_free_blocks(self) -> int:
        n = int(_lib.pkv_bm_num_free_blocks(self._h))
        if n < 0:
            raise PkvError(n, "pkv_bm_num_free_blocks")
        return n

    def add_sequence(self, seq_id: int, num_tokens: int) -> None:
        _check(_lib.pkv_bm_add_sequence(self._h, int(seq_id), int(num_tokens)), "pkv_bm_add_sequence")

    def append_slots(self, seq_ids) -> torch.Tensor:
        ids = torch.as_tensor(list(seq_ids), dtype=torch.int64).contiguous()
        out = torch.empty(len(ids), dtype=torch.int64)
        _check(_lib.pkv_bm_append_slots(self._h, ids.data_ptr(), len(ids), out.data_ptr()),
               "pkv_bm_append_slots")
        return out

    def free_sequence(self, seq_id: int) -> None:
        _check(_lib.pkv_bm_free_sequence(self._h, int(seq_id)), "pkv_bm_free_sequence")

    def preempt_lifo(self) -> int:
        v = ctypes.c_int64(0)
        _check(_lib.pkv_bm_preempt_lifo(self._h, ctypes.byref(v)), "pkv_bm_preempt_lifo")
        return int(v.value)

    def block_tables(self, seq_ids, max_blocks_per_seq: int):
        ids = torch.as_tensor(list(seq_ids), dtype=torch.int64).contiguous()
        tables = torch.empty(len(ids), int(max_blocks_per_seq), dtype=torch.int32)
        lens = torch.empty(len(ids), dtype=torch.int32)
        _check(_lib.pkv_bm_block_tables(self._h, ids.data_ptr(), len(ids), int(max_blocks_per_seq),
                                        tables.data_ptr(), lens.data_ptr()), "pkv_bm_block_tables")
        return tables, lens
