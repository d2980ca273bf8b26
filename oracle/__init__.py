"""CPU oracle for paged-KV decode -- TEST INFRASTRUCTURE ONLY.

A thin ctypes wrapper over ``oracle.c`` (plain fp64 C).  Only the tests, the smoke
check and the benchmark's CPU-baseline leg use it; the library's product path
never imports it.  Inputs are torch CPU tensors (bf16 tensors are passed as their
raw 16-bit patterns); outputs are float64 tensors.

Each function states the definition it follows in ``oracle.c``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()


def build(src: str = _SRC, out: str = _LIB, extra_flags: tuple = ()) -> str:
    """Compile ``oracle.c`` with gcc into a shared library (OpenMP over rows)."""
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp",
           *extra_flags, src, "-o",
           out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _stale(lib: str, src: str) -> bool:
    return not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src)


class Oracle:
    """Bindings to one compiled oracle library (the real one, or a test's variant)."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        L = ctypes.CDLL(lib_path)
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = dbl
        L.oracle_double_to_bf16.argtypes = [dbl]
        L.oracle_double_to_bf16.restype = ctypes.c_uint16
        L.oracle_kv_write.argtypes = [P, P, P, i64, P, P, i64, i32, i32, i32]
        L.oracle_kv_write.restype = ctypes.c_int
        L.oracle_decode_rows.argtypes = [P, P, i32, P, P, P, P, i32, P, i32, i32, i32, i64, i32,
                                         i32, dbl, i32]
        L.oracle_decode_rows.restype = ctypes.c_int
        L.oracle_decode_attention.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i64, i32, i32,
                                              dbl, i32]
        L.oracle_decode_attention.restype = ctypes.c_int
        L.oracle_decode_partitions.argtypes = [P, P, i32, i32, i32, i32, P, P, P, P, i32, P, i32,
                                               i32, i32, i64, i32, i32, dbl]
        L.oracle_decode_partitions.restype = ctypes.c_int
        L.oracle_lse_combine.argtypes = [P, P, P, i32, i32]
        L.oracle_lse_combine.restype = ctypes.c_int
        L.oracle_kv_write_rope.argtypes = [P, P, P, i32, P, P, i64, P, i64, i32, i32, P, P, i64,
                                           i32, i32, i32]
        L.oracle_kv_write_rope.restype = ctypes.c_int
        L.oracle_prefill_attention.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32, i64, i32,
                                               i32, dbl, i32]
        L.oracle_prefill_attention.restype = ctypes.c_int
        self._L = L

    # -- helpers -------------------------------------------------------------
    @staticmethod
    def _u16(t: torch.Tensor) -> np.ndarray:
        assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
        return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy().view(np.uint16))

    @staticmethod
    def _arr(t, dtype) -> np.ndarray:
        if isinstance(t, torch.Tensor):
            t = t.cpu().numpy()
        return np.ascontiguousarray(np.asarray(t, dtype=dtype))

    @staticmethod
    def _p(a: np.ndarray):
        return a.ctypes.data_as(ctypes.c_void_p)

    @staticmethod
    def _check(rc: int, what: str):
        if rc != 0:
            raise RuntimeError(f"oracle {what} failed with code {rc}")

    # -- bf16 conversions -----------------------------------------------------
    def bf16_to_double(self, bits: int) -> float:
        return self._L.oracle_bf16_to_double(int(bits) & 0xFFFF)

    def double_to_bf16(self, x: float) -> int:
        return int(self._L.oracle_double_to_bf16(float(x)))

    # -- the slot-mapping write ---------------------------------------------
    def kv_write(self, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                 k_cache: torch.Tensor, v_cache: torch.Tensor):
        """Returns new (k_cache, v_cache) bf16 tensors after writing k/v at their slots."""
        NB, Hkv, BS, D = k_cache.shape
        kc, vc = self._u16(k_cache).copy(), self._u16(v_cache).copy()
        ka, va = self._u16(k), self._u16(v)
        sl = self._arr(slot_mapping, np.int64)
        rc = self._L.oracle_kv_write(self._p(ka), self._p(va), self._p(sl), len(sl), self._p(kc),
                                     self._p(vc), NB, Hkv, BS, D)
        self._check(rc, "kv_write")
        to_t = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).reshape(NB, Hkv, BS, D)
        return to_t(kc), to_t(vc)

    def kv_write_rope(self, k, v, slot_mapping, positions, cos_sin, k_cache, v_cache, q=None,
                      rotary_dim=None, neox_style=True):
        """Rotary embedding of k (and q) at `positions` (fp32 table cos_sin [max_pos, r]),
        then the slot write.  Returns (k_cache, v_cache, q) as new bf16 tensors."""
        NB, Hkv, BS, D = k_cache.shape
        r = D if rotary_dim is None else int(rotary_dim)
        kc, vc = self._u16(k_cache).copy(), self._u16(v_cache).copy()
        ka, va = self._u16(k), self._u16(v)
        qa = self._u16(q).copy() if q is not None else None
        Hq = q.shape[1] if q is not None else 0
        sl = self._arr(slot_mapping, np.int64)
        po = self._arr(positions, np.int64)
        cs = self._arr(cos_sin, np.float32)
        rc = self._L.oracle_kv_write_rope(self._p(ka), self._p(va),
                                          self._p(qa) if qa is not None else None, Hq,
                                          self._p(sl), self._p(po), len(sl), self._p(cs),
                                          cs.shape[0], r, 1 if neox_style else 0, self._p(kc),
                                          self._p(vc), NB, Hkv, BS, D)
        self._check(rc, "kv_write_rope")
        to_t = lambda a, shape: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).reshape(shape)
        qo = to_t(qa, tuple(q.shape)) if q is not None else None
        return to_t(kc, (NB, Hkv, BS, D)), to_t(vc, (NB, Hkv, BS, D)), qo

    # -- decode attention -----------------------------------------------------
    def decode(self, q, k_cache, v_cache, block_tables, context_lens, scale: float,
               rows: Optional[torch.Tensor] = None, num_threads: int = 0) -> torch.Tensor:
        """fp64 attention output: [B, Hq, D], or [len(rows), D] for (b, h) rows."""
        B, Hq, D = q.shape
        NB, Hkv, BS, D2 = k_cache.shape
        assert D == D2
        qa, ka, va = self._u16(q), self._u16(k_cache), self._u16(v_cache)
        bt = self._arr(block_tables, np.int32)
        cl = self._arr(context_lens, np.int32)
        maxb = bt.shape[1] if bt.ndim == 2 else 1
        if rows is None:
            out = np.zeros((B, Hq, D), dtype=np.float64)
            rc = self._L.oracle_decode_attention(self._p(out), self._p(qa), self._p(ka),
                                                 self._p(va), self._p(bt), maxb, self._p(cl), B,
                                                 Hq, Hkv, NB, BS, D, float(scale), num_threads)
        else:
            rw = self._arr(rows, np.int32).reshape(-1, 2)
            out = np.zeros((rw.shape[0], D), dtype=np.float64)
            rc = self._L.oracle_decode_rows(self._p(out), self._p(rw), rw.shape[0], self._p(qa),
                                            self._p(ka), self._p(va), self._p(bt), maxb,
                                            self._p(cl), B, Hq, Hkv, NB, BS, D, float(scale),
                                            num_threads)
        self._check(rc, "decode")
        return torch.from_numpy(out)

    def prefill(self, q, k_cache, v_cache, block_tables, context_lens, query_start,
                scale: float, num_threads: int = 0) -> torch.Tensor:
        """fp64 causal attention of each sequence's last n_b tokens (packed q [Nq, Hq, D])."""
        Nq, Hq, D = q.shape
        NB, Hkv, BS, _ = k_cache.shape
        qa, ka, va = self._u16(q), self._u16(k_cache), self._u16(v_cache)
        bt = self._arr(block_tables, np.int32)
        cl = self._arr(context_lens, np.int32)
        qs = self._arr(query_start, np.int32)
        out = np.zeros((Nq, Hq, D), dtype=np.float64)
        rc = self._L.oracle_prefill_attention(self._p(out), self._p(qa), self._p(ka), self._p(va),
                                              self._p(bt), bt.shape[1], self._p(cl), self._p(qs),
                                              len(cl), Hq, Hkv, NB, BS, D, float(scale),
                                              num_threads)
        self._check(rc, "prefill")
        return torch.from_numpy(out)

    def decode_partitions(self, b: int, h: int, num_parts: int, partition_tokens: int, q,
                          k_cache, v_cache, block_tables, context_lens, scale: float):
        """Per token range [r*P, (r+1)*P): (o [num_parts, D] fp64, lse [num_parts] fp64)."""
        B, Hq, D = q.shape
        NB, Hkv, BS, _ = k_cache.shape
        qa, ka, va = self._u16(q), self._u16(k_cache), self._u16(v_cache)
        bt = self._arr(block_tables, np.int32)
        cl = self._arr(context_lens, np.int32)
        o = np.zeros((max(num_parts, 1), D), dtype=np.float64)
        lse = np.zeros(max(num_parts, 1), dtype=np.float64)
        rc = self._L.oracle_decode_partitions(self._p(o), self._p(lse), num_parts,
                                              partition_tokens, b, h, self._p(qa), self._p(ka),
                                              self._p(va), self._p(bt), bt.shape[1], self._p(cl),
                                              B, Hq, Hkv, NB, BS, D, float(scale))
        self._check(rc, "decode_partitions")
        return torch.from_numpy(o[:num_parts]), torch.from_numpy(lse[:num_parts])

    def lse_combine(self, o_part: torch.Tensor, lse_part: torch.Tensor) -> torch.Tensor:
        o = self._arr(o_part, np.float64)
        lse = self._arr(lse_part, np.float64)
        n, D = o.shape
        out = np.zeros(D, dtype=np.float64)
        rc = self._L.oracle_lse_combine(self._p(out), self._p(o), self._p(lse), n, D)
        self._check(rc, "lse_combine")
        return torch.from_numpy(out)

    # -- one whole decode step: write, then attend ---------------------------
    def step(self, inp: dict, num_threads: int = 0):
        """KV write of this step's tokens, then attention over the updated cache."""
        kc, vc = self.kv_write(inp["k_new"], inp["v_new"], inp["slot_mapping"], inp["k_cache"],
                               inp["v_cache"])
        out = self.decode(inp["q"], kc, vc, inp["block_tables"], inp["context_lens"],
                          inp["scale"], num_threads=num_threads)
        return out, kc, vc


_default: Optional[Oracle] = None


def get() -> Oracle:
    """The oracle compiled from ``oracle.c`` (rebuilt when the source is newer)."""
    global _default
    with _lock:
        if _default is None:
            if _stale(_LIB, _SRC):
                build()
            _default = Oracle(_LIB)
    return _default
