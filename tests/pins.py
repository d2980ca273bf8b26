"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when the
oracle disagrees with what the pages or the mathematics fix:

* a library routine (torch fp64 ``scaled_dot_product_attention``, torch's
  float32 -> bf16 conversion),
* closed forms (context length 1 returns V; identical keys or a zero scale return
  the mean of V; two tokens give a sigmoid mix),
* invariants (paged == dense on scattered blocks -- the mini-vLLM README's M4
  test; any permutation of the physical pool leaves the output unchanged,
  enumerated exhaustively on a tiny pool; cached decode == recompute -- the
  llm-stack KV-cache gate; NaN in slots nobody owns changes nothing),
* the flash-decoding algebra (merging per-range log-sum-exp results equals the
  unsplit softmax, for every split).

The same functions run against deliberately broken oracle builds, each of which
must fail at least one pin.
"""

from __future__ import annotations

import itertools
import math

import torch
import torch.nn.functional as F

from paged_kv_decode_mapping_gb300 import workloads as W


def _case(B=3, Hq=8, Hkv=2, D=16, BS=4, lens=(1, 7, 13), seed=11, pool_factor=1.5, write="last"):
    w = W.small_workload(B=B, Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=lens, seed=seed,
                         pool_factor=pool_factor, write=write)
    return W.make_inputs(w)


def _gather(cache: torch.Tensor, table_row: torch.Tensor, L: int, g: int) -> torch.Tensor:
    """Dense [L, D] rows of kv head g via torch advanced indexing."""
    BS = cache.shape[2]
    t = torch.arange(L)
    phys = table_row.long()[t // BS]
    return cache[phys, g, t % BS, :].double()


def _sdpa_reference(inp) -> torch.Tensor:
    """torch fp64 SDPA (not causal) per sequence on gathered K/V, GQA via repeat_interleave."""
    q, kc, vc = inp["q"], inp["k_cache"], inp["v_cache"]
    B, Hq, D = q.shape
    Hkv = kc.shape[1]
    G = Hq // Hkv
    out = torch.zeros(B, Hq, D, dtype=torch.float64)
    for b in range(B):
        L = int(inp["context_lens"][b])
        if L == 0:
            continue
        K = torch.stack([_gather(kc, inp["block_tables"][b], L, g) for g in range(Hkv)])
        V = torch.stack([_gather(vc, inp["block_tables"][b], L, g) for g in range(Hkv)])
        K = K.repeat_interleave(G, dim=0)[None]  # [1, Hq, L, D]
        V = V.repeat_interleave(G, dim=0)[None]
        qq = q[b].double()[None, :, None, :]  # [1, Hq, 1, D]
        o = F.scaled_dot_product_attention(qq, K, V, is_causal=False, scale=inp["scale"])
        out[b] = o[0, :, 0, :]
    return out


def _decode(o, inp, **kw):
    return o.decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                    inp["context_lens"], inp["scale"], **kw)


# --------------------------------------------------------------------------- bf16
def pin_bf16_widening(o):
    """bf16 -> double equals torch's exact bf16 -> float64 for all 65536 patterns."""
    bits = torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).double()
    for i in range(0, 65536, 257):  # a spread-out sample through ctypes, all sign/exponent mixes
        got = o.bf16_to_double(int(bits[i]) & 0xFFFF)
        r = float(ref[i])
        assert (math.isnan(got) and math.isnan(r)) or got == r, (i, got, r)


def pin_bf16_rounding(o):
    """double -> bf16 (RNE) equals torch's float32 -> bf16 on float32 inputs, incl. ties."""
    g = torch.Generator().manual_seed(5)
    xs = torch.cat([
        torch.randn(3000, generator=g) * torch.exp2(torch.randint(-30, 30, (3000,), generator=g).float()),
        # exact ties: a bf16 value plus half an ulp (both parities of the last kept bit)
        (torch.arange(1, 300, dtype=torch.int32) << 16 | 0x8000).view(torch.float32),
        (torch.arange(0x3F80, 0x3FF0, dtype=torch.int32) << 16 | 0x8000).view(torch.float32),
        torch.tensor([0.0, -0.0, 1e-40, -1e-40, 3.0e38, 65504.0, 1.0 / 3.0]),
    ])
    ref = xs.to(torch.bfloat16).view(torch.int16)
    for x, r in zip(xs.tolist(), ref.tolist()):
        got = o.double_to_bf16(x)
        assert got == (r & 0xFFFF), (x, hex(got), hex(r & 0xFFFF))


# ------------------------------------------------------------------------- write
def pin_write(o):
    """Written slots hold exactly the input bits; every other byte is unchanged;
    negative slots are skipped; slot 0 and a slot in the last block are honoured."""
    inp = _case(B=2, Hq=4, Hkv=2, D=8, BS=4, lens=(6, 9), write="none")
    NB = inp["num_blocks"]
    g = torch.Generator().manual_seed(3)
    slots = torch.tensor([0, -1, NB * 4 - 1, 5, 17], dtype=torch.int64)
    k = torch.randn(len(slots), 2, 8, generator=g).to(torch.bfloat16)
    v = torch.randn(len(slots), 2, 8, generator=g).to(torch.bfloat16)
    kc, vc = o.kv_write(k, v, slots, inp["k_cache"], inp["v_cache"])
    ek, ev = inp["k_cache"].clone(), inp["v_cache"].clone()
    for i, s in enumerate(slots.tolist()):
        if s >= 0:
            ek[s // 4, :, s % 4, :] = k[i]
            ev[s // 4, :, s % 4, :] = v[i]
    assert torch.equal(kc.view(torch.int16), ek.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), ev.view(torch.int16))


# --------------------------------------------------------------------- attention
def pin_sdpa(o):
    """Oracle == torch fp64 SDPA (non-causal) on the gathered copy, GQA and MHA."""
    for kw in (dict(), dict(Hq=4, Hkv=4, lens=(3, 16, 9)), dict(Hq=6, Hkv=2, D=8, BS=2,
                                                                 lens=(5, 1, 12))):
        inp = _case(**kw)
        got = _decode(o, inp)
        ref = _sdpa_reference(inp)
        assert torch.allclose(got, ref, atol=1e-12, rtol=1e-12), (got - ref).abs().max()


def pin_paged_equals_dense(o):
    """Scattered blocks give the same output as one contiguous, in-order copy."""
    inp = _case(lens=(5, 11, 16))
    B, BS = 3, 4
    Hkv, D = inp["k_cache"].shape[1], inp["k_cache"].shape[3]
    nblk = [(int(L) + BS - 1) // BS for L in inp["context_lens"]]
    NB = sum(nblk)
    kd = torch.zeros(NB, Hkv, BS, D, dtype=torch.bfloat16)
    vd = torch.zeros_like(kd)
    tables = torch.zeros(B, max(nblk), dtype=torch.int32)
    nxt = 0
    for b in range(B):
        L = int(inp["context_lens"][b])
        for t in range(L):
            blk, off = nxt + t // BS, t % BS
            src = int(inp["block_tables"][b, t // BS])
            kd[blk, :, off] = inp["k_cache"][src, :, t % BS]
            vd[blk, :, off] = inp["v_cache"][src, :, t % BS]
        tables[b, :nblk[b]] = torch.arange(nxt, nxt + nblk[b], dtype=torch.int32)
        nxt += nblk[b]
    dense = dict(inp, k_cache=kd, v_cache=vd, block_tables=tables)
    assert torch.equal(_decode(o, inp), _decode(o, dense))


def pin_pool_permutations(o):
    """Brute force: every permutation of a 6-block pool (rewrite pool + tables) leaves
    the output bit-identical."""
    inp = _case(B=2, Hq=4, Hkv=2, D=4, BS=2, lens=(5, 3), pool_factor=1.2)
    NB = inp["k_cache"].shape[0]
    assert NB == 6
    ref = _decode(o, inp)
    tab = inp["block_tables"]
    for perm in itertools.permutations(range(NB)):
        p = torch.tensor(perm)
        kc = torch.empty_like(inp["k_cache"])
        vc = torch.empty_like(inp["v_cache"])
        kc[p] = inp["k_cache"]
        vc[p] = inp["v_cache"]
        nt = torch.where(tab >= 0, p[tab.clamp(min=0).long()].to(torch.int32), tab)
        got = _decode(o, dict(inp, k_cache=kc, v_cache=vc, block_tables=nt))
        assert torch.equal(got, ref), perm


def pin_length_one(o):
    """Context length 1: the output is the single cached V row, exactly."""
    inp = _case(lens=(1, 1, 1))
    got = _decode(o, inp)
    G = inp["q"].shape[1] // inp["k_cache"].shape[1]
    for b in range(3):
        phys = int(inp["block_tables"][b, 0])
        for h in range(inp["q"].shape[1]):
            assert torch.equal(got[b, h], inp["v_cache"][phys, h // G, 0].double()), (b, h)


def pin_identical_keys_and_zero_scale(o):
    """All keys equal, or scale 0: uniform weights, so the output is the mean of V."""
    inp = _case(lens=(4, 9, 13))
    kc = inp["k_cache"].clone()
    kc[:] = kc[0, :, :1, :]  # one key row repeated everywhere (per kv head)
    for case in (dict(inp, k_cache=kc), dict(inp, scale=0.0)):
        got = _decode(o, case)
        G = inp["q"].shape[1] // inp["k_cache"].shape[1]
        for b in range(3):
            L = int(inp["context_lens"][b])
            for h in range(inp["q"].shape[1]):
                Vd = _gather(inp["v_cache"], inp["block_tables"][b], L, h // G)
                assert torch.allclose(got[b, h], Vd.mean(0), atol=1e-13), (b, h)


def pin_two_tokens(o):
    """Two tokens: out = sigmoid(s1 - s2) v1 + sigmoid(s2 - s1) v2."""
    inp = _case(lens=(2, 2, 2))
    got = _decode(o, inp)
    G = inp["q"].shape[1] // inp["k_cache"].shape[1]
    for b in range(3):
        for h in range(inp["q"].shape[1]):
            K = _gather(inp["k_cache"], inp["block_tables"][b], 2, h // G)
            V = _gather(inp["v_cache"], inp["block_tables"][b], 2, h // G)
            qd = inp["q"][b, h].double()
            s1, s2 = inp["scale"] * float(qd @ K[0]), inp["scale"] * float(qd @ K[1])
            sig = 1.0 / (1.0 + math.exp(-(s1 - s2)))
            ref = sig * V[0] + (1.0 - sig) * V[1]
            assert torch.allclose(got[b, h], ref, atol=1e-13), (b, h)


def pin_context_zero(o):
    """An empty context gives a zero output (no NaN)."""
    inp = _case(lens=(0, 5, 0))
    got = _decode(o, inp)
    assert torch.equal(got[0], torch.zeros_like(got[0])) and torch.equal(got[2], torch.zeros_like(got[2]))
    assert torch.isfinite(got).all()


def pin_nan_poison(o):
    """NaN in every slot no sequence owns leaves the output finite and unchanged."""
    w = W.small_workload(B=3, Hq=8, Hkv=2, D=16, BS=4, lens=(3, 10, 13), seed=11)
    clean = W.make_inputs(w)
    dirty = W.make_inputs(w, poison=True)
    assert torch.isnan(dirty["k_cache"].float()).any()
    a, b = _decode(o, clean), _decode(o, dirty)
    assert torch.isfinite(b).all() and torch.equal(a, b)


def pin_partitions(o):
    """Flash-decoding algebra: merging the per-range (o, lse) of any split equals the
    unsplit output; one range is the identity; ranges past the end weigh nothing."""
    inp = _case(lens=(1, 7, 13))
    full = _decode(o, inp)
    for b in range(3):
        L = int(inp["context_lens"][b])
        for h in (0, 3, 7):
            for P in (1, 2, 3, 5, 13, 64):
                n = (L + P - 1) // P + 1  # one extra, empty range
                op, lse = o.decode_partitions(b, h, n, P, inp["q"], inp["k_cache"],
                                              inp["v_cache"], inp["block_tables"],
                                              inp["context_lens"], inp["scale"])
                assert lse[-1] == -math.inf and torch.equal(op[-1], torch.zeros_like(op[-1]))
                got = o.lse_combine(op, lse)
                assert torch.allclose(got, full[b, h], atol=1e-13), (b, h, P)
            # lse of the whole range is the log of the softmax normaliser of the scaled scores
            op, lse = o.decode_partitions(b, h, 1, 10_000, inp["q"], inp["k_cache"],
                                          inp["v_cache"], inp["block_tables"],
                                          inp["context_lens"], inp["scale"])
            G = inp["q"].shape[1] // inp["k_cache"].shape[1]
            K = _gather(inp["k_cache"], inp["block_tables"][b], L, h // G)
            s = inp["scale"] * (K @ inp["q"][b, h].double())
            assert abs(float(lse[0]) - float(torch.logsumexp(s, 0))) < 1e-12
            assert torch.allclose(o.lse_combine(op, lse), op[0], atol=1e-15)


def pin_cached_equals_recompute(o):
    """Writing a sequence's K/V one token per step through the slot mapping, then
    decoding, equals attention recomputed over all tokens at once."""
    BS, Hkv, D, Hq = 4, 2, 8, 4
    L = 11
    g = torch.Generator().manual_seed(9)
    Kall = torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16)
    Vall = torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16)
    q = torch.randn(1, Hq, D, generator=g).to(torch.bfloat16)
    NB = 5
    table = torch.tensor([[3, 0, 4]], dtype=torch.int32)
    kc = torch.zeros(NB, Hkv, BS, D, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    for t in range(L):
        slot = int(table[0, t // BS]) * BS + t % BS
        kc, vc = o.kv_write(Kall[t:t + 1], Vall[t:t + 1], torch.tensor([slot]), kc, vc)
    got = o.decode(q, kc, vc, table, torch.tensor([L], dtype=torch.int32), 0.5)
    K = Kall.double().permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)[None]
    V = Vall.double().permute(1, 0, 2).repeat_interleave(Hq // Hkv, 0)[None]
    ref = F.scaled_dot_product_attention(q.double()[:, :, None, :], K, V, scale=0.5)[:, :, 0]
    assert torch.allclose(got, ref, atol=1e-12)


# ------------------------------------------------------------------ RoPE write
def rope_table(max_pos, rotary_dim, base=10000.0, dtype=torch.float64):
    """cos/sin table [max_pos, r]: angle(pos, i) = pos * base^(-2i/r), cos first then sin."""
    half = rotary_dim // 2
    inv = base ** (-torch.arange(half, dtype=torch.float64) * 2.0 / rotary_dim)
    ang = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv[None, :]
    return torch.cat([ang.cos(), ang.sin()], dim=1).to(dtype)


def _rope_case(T=5, Hkv=2, Hq=4, D=16, seed=2):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    q = torch.randn(T, Hq, D, generator=g).to(torch.bfloat16)
    kc = torch.zeros(4, Hkv, 4, D, dtype=torch.bfloat16)
    return k, v, q, kc


def pin_rope_zero_angle_is_identity(o):
    """Rotation by angle 0 (cos 1, sin 0) leaves k and q bit-identical."""
    k, v, q, kc = _rope_case()
    cs = torch.cat([torch.ones(1, 8), torch.zeros(1, 8)], dim=1).float()
    slots = torch.arange(5, dtype=torch.int64)
    kr, vr, qr = o.kv_write_rope(k, v, slots, torch.zeros(5, dtype=torch.int64), cs, kc, kc, q=q)
    ek, ev = o.kv_write(k, v, slots, kc, kc)
    assert torch.equal(kr.view(torch.int16), ek.view(torch.int16))
    assert torch.equal(vr.view(torch.int16), ev.view(torch.int16))
    assert torch.equal(qr.view(torch.int16), q.view(torch.int16))


def _rope_exact(x: torch.Tensor, cs: torch.Tensor, pos: torch.Tensor) -> torch.Tensor:
    """Rotate-half pairs (i, i + D/2) of x [T, H, D] as the complex product
    (x_i + i x_{i+D/2}) e^{i angle(pos, i)} in complex128, angle from the table cs."""
    half = x.shape[-1] // 2
    xd = x.double()
    z = torch.complex(xd[..., :half], xd[..., half:])
    c = cs.double()[pos][:, None, :half]
    s = cs.double()[pos][:, None, half:]
    zr = z * torch.complex(c, s)
    return torch.cat([zr.real, zr.imag], dim=-1)


def _within_bf16_rounding(y: torch.Tensor, exact: torch.Tensor, x: torch.Tensor) -> bool:
    err = (y.double() - exact).abs()
    return bool((err <= 2.0 ** -8 * exact.abs() + 1e-6 * (1 + x.double().abs())).all())


def pin_rope_is_complex_rotation(o):
    """Each pair (x1, x2) becomes (x1 + i x2) * e^{i angle}, computed independently in
    complex128; the oracle's fp32-then-bf16 result is within bf16 rounding of it.  Both
    the query rotated in place and the keys as they land in the cache (each token at
    its own nonzero position, every kv head), since the cache must hold keys rotated at
    their absolute positions."""
    k, v, q, kc = _rope_case(T=6, D=32)
    cs = rope_table(50, 32).float()
    pos = torch.tensor([3, 1, 7, 13, 31, 49], dtype=torch.int64)
    slots = torch.tensor([5, 0, 15, 8, 2, 11], dtype=torch.int64)  # in a 4-block x 4-slot pool
    kc_out, vc_out, qr = o.kv_write_rope(k, v, slots, pos, cs, kc, kc, q=q)
    assert _within_bf16_rounding(qr, _rope_exact(q, cs, pos), q), "q"
    kr = torch.stack([kc_out[int(sl) // 4, :, int(sl) % 4, :] for sl in slots])  # [T, Hkv, D]
    vr = torch.stack([vc_out[int(sl) // 4, :, int(sl) % 4, :] for sl in slots])
    assert _within_bf16_rounding(kr, _rope_exact(k, cs, pos), k), "k in the cache"
    assert torch.equal(vr.view(torch.int16), v.view(torch.int16)), "v is copied, not rotated"


def pin_rope_pairing_permutation(o):
    """Interleaved pairs (2i, 2i+1) are the rotate-half pairs (i, i + r/2) of the vector
    with its even coordinates first and odd ones after (the pairing permutation)."""
    k, v, q, kc = _rope_case(T=4, D=16)
    cs = rope_table(20, 16).float()
    pos = torch.tensor([3, 5, 11, 19], dtype=torch.int64)
    perm = torch.cat([torch.arange(0, 16, 2), torch.arange(1, 16, 2)])
    inv = torch.argsort(perm)
    none = torch.full((4,), -1, dtype=torch.int64)
    _, _, qi = o.kv_write_rope(k, v, none, pos, cs, kc, kc, q=q, neox_style=False)
    _, _, qn = o.kv_write_rope(k, v, none, pos, cs, kc, kc, q=q[..., perm].contiguous(), neox_style=True)
    assert torch.equal(qi.view(torch.int16), qn[..., inv].contiguous().view(torch.int16))


def pin_rope_relative_position(o):
    """<R(m) q, R(n) k> depends only on m - n (up to bf16 rounding of the rotated vectors):
    q rotated in place at m, k rotated through the write at n and read back from the
    cache slot it was written to."""
    k, v, q, kc = _rope_case(T=1, Hkv=1, Hq=1, D=64, seed=4)
    cs = rope_table(200, 64).float()
    none = torch.full((1,), -1, dtype=torch.int64)
    slot = torch.tensor([6], dtype=torch.int64)

    def rot_q(p):
        _, _, y = o.kv_write_rope(k, v, none, torch.tensor([p]), cs, kc[:, :1], kc[:, :1], q=q)
        return y.double().flatten()

    def rot_k(p):
        kc1, _, _ = o.kv_write_rope(k, v, slot, torch.tensor([p]), cs, kc[:, :1], kc[:, :1])
        return kc1[1, 0, 2].double()  # slot 6 = block 1, offset 2

    base = float(rot_q(40) @ rot_k(25))
    assert abs(base - float(q.double().flatten() @ k.double().flatten())) > 1e-3  # rotation matters
    for d in (0, 17, 100, 150):
        other = float(rot_q(40 + d) @ rot_k(25 + d))
        assert abs(other - base) < 0.05 * (1 + abs(base)), (d, other, base)
    # and a different offset m - n gives a different product
    assert abs(float(rot_q(40) @ rot_k(29)) - base) > 1e-3


def pin_rope_partial_rotary(o):
    """Coordinates at or past rotary_dim are copied unchanged; the rest match a full
    rotation of the first rotary_dim coordinates."""
    k, v, q, kc = _rope_case(T=3, D=32)
    cs = rope_table(10, 16).float()
    pos = torch.tensor([1, 4, 9], dtype=torch.int64)
    none = torch.full((3,), -1, dtype=torch.int64)
    _, _, qp = o.kv_write_rope(k, v, none, pos, cs, kc, kc, q=q, rotary_dim=16)
    assert torch.equal(qp[..., 16:].contiguous().view(torch.int16), q[..., 16:].contiguous().view(torch.int16))
    kc16 = torch.zeros(4, 2, 4, 16, dtype=torch.bfloat16)
    _, _, qf = o.kv_write_rope(k[..., :16].contiguous(), v[..., :16].contiguous(), none, pos, cs,
                               kc16, kc16, q=q[..., :16].contiguous())
    assert torch.equal(qp[..., :16].contiguous().view(torch.int16), qf.view(torch.int16))


# ---------------------------------------------------------------- paged prefill
def _prefill_case(lens=(9, 23, 4), chunks=(9, 5, 1), Hq=8, Hkv=2, D=16, BS=4, seed=3):
    inp = _case(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=lens, seed=seed, write="none")
    g = torch.Generator().manual_seed(seed + 1)
    qs = torch.tensor([0] + list(itertools.accumulate(chunks)), dtype=torch.int32)
    q = torch.randn(int(qs[-1]), Hq, D, generator=g).to(torch.bfloat16)
    return inp, q, qs


def pin_prefill_matches_sdpa_with_causal_mask(o):
    """Chunked prefill == torch fp64 SDPA over the gathered keys with the mask t <= p
    (is_causal=True when the chunk is the whole context)."""
    for lens, chunks in (((9, 23, 4), (9, 5, 1)), ((16, 7), (16, 7))):
        inp, q, qs = _prefill_case(lens, chunks)
        got = o.prefill(q, inp["k_cache"], inp["v_cache"], inp["block_tables"], inp["context_lens"],
                        qs, inp["scale"])
        Hq, Hkv = q.shape[1], inp["k_cache"].shape[1]
        for b, (L, n) in enumerate(zip(lens, chunks)):
            K = torch.stack([_gather(inp["k_cache"], inp["block_tables"][b], L, g) for g in range(Hkv)])
            V = torch.stack([_gather(inp["v_cache"], inp["block_tables"][b], L, g) for g in range(Hkv)])
            K, V = K.repeat_interleave(Hq // Hkv, 0)[None], V.repeat_interleave(Hq // Hkv, 0)[None]
            qq = q[int(qs[b]):int(qs[b + 1])].double().permute(1, 0, 2)[None]  # [1, Hq, n, D]
            if n == L:
                ref = F.scaled_dot_product_attention(qq, K, V, is_causal=True, scale=inp["scale"])
            else:
                pos = torch.arange(L - n, L)[:, None]
                mask = torch.arange(L)[None, :] <= pos
                ref = F.scaled_dot_product_attention(qq, K, V, attn_mask=mask, scale=inp["scale"])
            assert torch.allclose(got[int(qs[b]):int(qs[b + 1])], ref[0].permute(1, 0, 2), atol=1e-12)


def pin_prefill_last_token_is_decode(o):
    """The last query of each chunk sees every cached key: it equals decode attention."""
    inp, q, qs = _prefill_case()
    got = o.prefill(q, inp["k_cache"], inp["v_cache"], inp["block_tables"], inp["context_lens"],
                    qs, inp["scale"])
    last = q[(qs[1:] - 1).long()]
    dec = o.decode(last, inp["k_cache"], inp["v_cache"], inp["block_tables"], inp["context_lens"],
                   inp["scale"])
    assert torch.equal(got[(qs[1:] - 1).long()], dec)


ALL_PINS = [
    pin_bf16_widening, pin_bf16_rounding, pin_write, pin_sdpa, pin_paged_equals_dense,
    pin_pool_permutations, pin_length_one, pin_identical_keys_and_zero_scale, pin_two_tokens,
    pin_context_zero, pin_nan_poison, pin_partitions, pin_cached_equals_recompute,
    pin_rope_zero_angle_is_identity, pin_rope_is_complex_rotation, pin_rope_pairing_permutation,
    pin_rope_relative_position, pin_rope_partial_rotary,
    pin_prefill_matches_sdpa_with_causal_mask, pin_prefill_last_token_is_decode,
]
