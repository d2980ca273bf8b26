"""Seeded synthetic inputs for paged-KV decode.

This module only draws inputs: sequence lengths, a shuffled physical block pool,
per-sequence block tables, the slot mapping of the tokens written this step, and
N(0, 1) bf16 tensors.  It holds none of the attention or KV-write arithmetic, so
both the CUDA path and the CPU oracle can take their inputs from it.

Shapes follow the layout the library uses:

* ``q``            bf16 ``[B, Hq, D]``
* ``k_cache``      bf16 ``[NB, Hkv, BS, D]`` (``v_cache`` alike)
* ``block_tables`` int32 ``[B, max_blocks_per_seq]`` (unused entries are -1)
* ``context_lens`` int32 ``[B]`` (the lengths *after* this step's write)
* ``k_new``/``v_new`` bf16 ``[T, Hkv, D]`` and ``slot_mapping`` int64 ``[T]``

Recipe (fixed order of draws from one ``torch.Generator`` seeded with the case's
seed): context lengths, the pool permutation, ``q``, ``k_cache``, ``v_cache``,
``k_new``, ``v_new``.  Every float tensor is drawn as float32 N(0, 1) and rounded
to bf16 (round to nearest even).  Sequence ``b`` owns consecutive entries of one
random permutation of the pool, so its logical blocks are scattered over the pool
(the "scattered blocks" setting of the mini-vLLM page's paged-attention test).
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode step: sizes and how lengths / pool / writes are drawn."""

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    BS: int
    lens: str  # "fixed", "uniform", "lognormal", "explicit"
    L: int = 0  # fixed length
    L_lo: int = 0  # uniform / clip lower bound
    L_hi: int = 0  # uniform / clip upper bound
    median: float = 0.0  # lognormal median
    sigma: float = 1.0  # lognormal sigma
    pool_blocks: int = 0  # 0: ceil(pool_factor * blocks in use)
    pool_factor: float = 1.25
    write: str = "last"  # "last": one token per sequence at position L_b-1; "slot128"; "none"
    partition_tokens: int = 0  # 0: the launcher picks
    seed: int = 0
    explicit_lens: Optional[Sequence[int]] = None

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


# The five workloads of the benchmark table.  Seeds are 1000 + workload number.
WORKLOADS = {
    1: Workload("decode B=1 ctx=128 Hq=32 Hkv=8 D=64 BS=16", B=1, Hq=32, Hkv=8, D=64, BS=16,
                lens="fixed", L=128, pool_blocks=64, write="slot128", seed=1001),
    2: Workload("decode B=16 ctx=2048 Hq=32 Hkv=8 D=64 BS=16", B=16, Hq=32, Hkv=8, D=64, BS=16,
                lens="fixed", L=2048, pool_blocks=2560, write="last", seed=1002),
    3: Workload("decode B=64 ctx~U[128,4096] Hq=24 Hkv=8 D=128 BS=16", B=64, Hq=24, Hkv=8, D=128,
                BS=16, lens="uniform", L_lo=128, L_hi=4096, pool_factor=1.25, write="last",
                seed=1003),
    4: Workload("continuous-batching B=256 ctx~lognormal(med 512)[16,8192] Hq=32 Hkv=4 D=64 BS=16",
                B=256, Hq=32, Hkv=4, D=64, BS=16, lens="lognormal", median=512.0, sigma=1.0,
                L_lo=16, L_hi=8192, pool_factor=1.25, write="last", seed=1004),
    5: Workload("long-context split-K B=4 ctx=32768 Hq=24 Hkv=8 D=128 BS=32 P=512", B=4, Hq=24,
                Hkv=8, D=128, BS=32, lens="fixed", L=32768, pool_blocks=5120, write="last",
                partition_tokens=512, seed=1005),
}


def small_workload(B=2, Hq=8, Hkv=2, D=64, BS=16, lens=(37, 100), pool_factor=1.5, seed=7,
                   write="last", partition_tokens=0, name="small") -> Workload:
    """A small case with explicit lengths (for tests that the oracle finishes in seconds)."""
    return Workload(name, B=B, Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens="explicit",
                    explicit_lens=tuple(int(x) for x in lens), pool_factor=pool_factor,
                    write=write, partition_tokens=partition_tokens, seed=seed)


def _draw_lens(w: Workload, g: torch.Generator) -> torch.Tensor:
    if w.lens == "fixed":
        return torch.full((w.B,), w.L, dtype=torch.int64)
    if w.lens == "uniform":
        return torch.randint(w.L_lo, w.L_hi + 1, (w.B,), generator=g, dtype=torch.int64)
    if w.lens == "lognormal":
        x = torch.empty(w.B, dtype=torch.float64).log_normal_(math.log(w.median), w.sigma,
                                                              generator=g)
        return x.round().clamp(w.L_lo, w.L_hi).to(torch.int64)
    if w.lens == "explicit":
        assert w.explicit_lens is not None and len(w.explicit_lens) == w.B
        return torch.tensor(list(w.explicit_lens), dtype=torch.int64)
    raise ValueError(w.lens)


def _randn_bf16(shape, g: torch.Generator) -> torch.Tensor:
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def make_inputs(w: Workload, poison: bool = False, seed: Optional[int] = None) -> dict:
    """Draw every input of one decode step on the CPU (deterministic for a given seed).

    ``poison=True`` fills every cache slot that no sequence reads (slots past
    ``L_b`` in a sequence's last block and blocks nobody owns) with NaN, so a
    kernel that touches them shows it.
    """
    g = torch.Generator(device="cpu").manual_seed(w.seed if seed is None else seed)
    lens = _draw_lens(w, g)
    nblk = (lens + w.BS - 1) // w.BS
    used = int(nblk.sum())
    NB = w.pool_blocks if w.pool_blocks else int(math.ceil(w.pool_factor * used))
    NB = max(NB, used, 1)
    perm = torch.randperm(NB, generator=g)
    maxb = max(int(nblk.max()) if w.B else 0, 1)
    tables = torch.full((w.B, maxb), -1, dtype=torch.int32)
    off = 0
    for b in range(w.B):
        n = int(nblk[b])
        tables[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    q = _randn_bf16((w.B, w.Hq, w.D), g)
    k_cache = _randn_bf16((NB, w.Hkv, w.BS, w.D), g)
    v_cache = _randn_bf16((NB, w.Hkv, w.BS, w.D), g)

    if w.write == "last":
        T = w.B
        slots = torch.empty(T, dtype=torch.int64)
        for b in range(w.B):
            pos = int(lens[b]) - 1
            if pos < 0:
                slots[b] = -1
            else:
                slots[b] = int(tables[b, pos // w.BS]) * w.BS + pos % w.BS
    elif w.write == "slot128":
        T = 1
        slots = torch.tensor([128], dtype=torch.int64)
    elif w.write == "none":
        T = 0
        slots = torch.empty(0, dtype=torch.int64)
    else:
        raise ValueError(w.write)
    k_new = _randn_bf16((T, w.Hkv, w.D), g)
    v_new = _randn_bf16((T, w.Hkv, w.D), g)

    if poison:
        live = torch.zeros(NB, w.BS, dtype=torch.bool)
        for b in range(w.B):
            for t in range(0, int(lens[b]), w.BS):
                n = min(w.BS, int(lens[b]) - t)
                live[int(tables[b, t // w.BS]), :n] = True
        dead = ~live
        nan = torch.tensor(float("nan"), dtype=torch.bfloat16)
        k_cache.masked_fill_(dead[:, None, :, None], nan)
        v_cache.masked_fill_(dead[:, None, :, None], nan)

    P = w.partition_tokens
    return dict(
        workload=w, q=q, k_cache=k_cache, v_cache=v_cache, block_tables=tables,
        context_lens=lens.to(torch.int32), max_context_len=int(lens.max()) if w.B else 0,
        k_new=k_new, v_new=v_new, slot_mapping=slots, scale=1.0 / math.sqrt(w.D),
        num_blocks=NB, partition_tokens=P,
    )


def shard_range(n: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous share ``[lo, hi)`` of ``n`` independent sequences for ``rank`` of ``world``."""
    base, rem = divmod(n, world)
    lo = rank * base + min(rank, rem)
    return lo, lo + base + (1 if rank < rem else 0)
