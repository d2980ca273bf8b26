"""CUDA path vs the CPU oracle, through the C ABI.

Bar: the KV write is bit-exact (the whole pool is compared, so no other byte may
change); attention is within |gpu - oracle| <= 1e-2 elementwise wherever
|oracle| <= 2.56, and within 1e-2 + 2^-8 |oracle| elsewhere.  The 1e-2 absolute
bound is the stated target; the 2^-8 |oracle| term is the bf16 output's own
half-ulp, which only exceeds 1e-2 where |out| > 2.56 (a bf16 value can be no
closer than that to the fp64 result).  Attention inputs carry NaN in every slot no
sequence owns, so reading one shows up.
"""

import dataclasses
import math

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

    binding.pkv_device_errors(clear=True)
    return binding


def dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


ABS_ONLY_BELOW = 2.56  # |oracle| at which the bf16 half-ulp term reaches 1e-2


def check_attention(got: torch.Tensor, ref: torch.Tensor, tag: str,
                    abs_only_below: float = ABS_ONLY_BELOW) -> float:
    got = got.cpu().double()
    assert torch.isfinite(got).all(), f"{tag}: non-finite output"
    err = (got - ref).abs()
    # every element: the absolute target where the output is small enough for a bf16
    # value to reach it, the target plus the output's own half-ulp elsewhere
    bound = torch.where(ref.abs() <= abs_only_below, torch.full_like(ref, ATOL),
                        ATOL + RTOL * ref.abs())
    bad = err > bound
    assert not bool(bad.any()), (f"{tag}: {int(bad.sum())} outputs out of tolerance, max |diff| "
                                 f"{err.max():.3e}")
    return float(err.max())


def step(B, g):
    """One decode step as the benchmark runs it: slot write, then attention (launcher's plan)."""
    B.paged_kv_write(g["k_new"], g["v_new"], g["slot_mapping"], g["k_cache"], g["v_cache"])
    out = torch.empty_like(g["q"])
    B.paged_decode_attention(out, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                             g["context_lens"], g["max_context_len"], g["scale"])
    return out


def assert_no_device_errors(B):
    flags = B.pkv_device_errors(clear=True)
    assert flags == 0, f"device error bits {flags:#x}"


# --------------------------------------------------------------- full workloads
@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_workload_step_matches_oracle(B, oracle, wid):
    w = W.WORKLOADS[wid]
    inp = W.make_inputs(w, poison=True)
    g = dev(inp)
    out = step(B, g)
    torch.cuda.synchronize()
    assert_no_device_errors(B)
    ref, kc_ref, vc_ref = oracle.step(inp)
    # KV write: every byte of both pools
    assert torch.equal(g["k_cache"].cpu().view(torch.int16), kc_ref.view(torch.int16))
    assert torch.equal(g["v_cache"].cpu().view(torch.int16), vc_ref.view(torch.int16))
    check_attention(out, ref, w.name)


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_workload_fused_step_entry_point(B, oracle, wid):
    """paged_decode_step (write, then attention launched as a programmatic dependent of
    the write) gives the same cache bytes and outputs as the oracle."""
    w = W.WORKLOADS[wid]
    inp = W.make_inputs(w, poison=True)
    g = dev(inp)
    out = torch.empty_like(g["q"])
    for _ in range(2):  # the second step rewrites the same slots: same result
        B.paged_decode_step(out, g["q"], g["k_new"], g["v_new"], g["slot_mapping"], g["k_cache"],
                            g["v_cache"], g["block_tables"], g["context_lens"],
                            g["max_context_len"], g["scale"])
    torch.cuda.synchronize()
    assert_no_device_errors(B)
    ref, kc_ref, vc_ref = oracle.step(inp)
    assert torch.equal(g["k_cache"].cpu().view(torch.int16), kc_ref.view(torch.int16))
    assert torch.equal(g["v_cache"].cpu().view(torch.int16), vc_ref.view(torch.int16))
    check_attention(out, ref, w.name + " (paged_decode_step)")


@pytest.mark.parametrize("D,Hq,Hkv,lens,path", [
    (64, 8, 2, (1500, 700), "cluster"),
    (128, 24, 8, (5000, 4100, 300, 9000), "partitions"),
    (64, 4, 4, (100, 37), "partitions"),
])
def test_step_writes_inside_the_range(B, oracle, D, Hq, Hkv, lens, path):
    """paged_decode_step whose slots land inside the sequences' ranges, not only at their
    ends (a block read by the first chunk of a partition, a block in the middle): the
    decode reads blocks the write does not touch before that grid finishes, and must
    read the touched ones after it."""
    w = W.small_workload(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, BS=16, lens=lens, seed=81 + D,
                         write="none")
    inp = W.make_inputs(w, poison=True)
    want = {"cluster": B.PATH_CLUSTER, "partitions": B.PATH_PARTITIONS}[path]
    assert B.paged_decode_path(w.B, Hq, Hkv, D, inp["max_context_len"]) == want
    tb = inp["block_tables"]
    slot = lambda b, t: int(tb[b, t // 16]) * 16 + t % 16
    slots = [slot(0, 5), slot(0, lens[0] // 2), slot(1, lens[1] - 1), -1, slot(0, lens[0] - 1)]
    gen = torch.Generator().manual_seed(82)
    T = len(slots)
    kn = torch.randn(T, Hkv, D, generator=gen).to(torch.bfloat16)
    vn = torch.randn(T, Hkv, D, generator=gen).to(torch.bfloat16)
    sm = torch.tensor(slots, dtype=torch.int64)
    kc, vc = oracle.kv_write(kn, vn, sm, inp["k_cache"], inp["v_cache"])
    ref = oracle.decode(inp["q"], kc, vc, tb, inp["context_lens"], inp["scale"])
    g = dev(inp)
    out = torch.empty_like(g["q"])
    B.paged_decode_step(out, g["q"], kn.cuda(), vn.cuda(), sm.cuda(), g["k_cache"], g["v_cache"],
                        g["block_tables"], g["context_lens"], g["max_context_len"], g["scale"])
    torch.cuda.synchronize()
    assert_no_device_errors(B)
    assert torch.equal(g["k_cache"].cpu().view(torch.int16), kc.view(torch.int16))
    check_attention(out, ref, f"writes inside the range ({path})")


@pytest.mark.parametrize("wid", [2, 5])
def test_workload_explicit_partition(B, oracle, wid):
    """The workload's own partition size (512 tokens for the long-context case) through the
    explicit split + combine entry points."""
    w = W.WORKLOADS[wid]
    inp = W.make_inputs(dataclasses.replace(w, write="none"), poison=True)
    g = dev(inp)
    P = 512
    n = math.ceil(inp["max_context_len"] / P)
    Bn, Hq, D = inp["q"].shape
    o_part = torch.empty(Bn, Hq, n, D, device="cuda")
    lse = torch.empty(Bn, Hq, n, device="cuda")
    B.paged_decode_split(o_part, lse, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                         g["context_lens"], inp["max_context_len"], inp["scale"], P)
    out = torch.empty_like(g["q"])
    B.paged_decode_combine(out, o_part, lse, g["context_lens"], inp["max_context_len"], P)
    torch.cuda.synchronize()
    assert_no_device_errors(B)
    ref = oracle.decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                        inp["context_lens"], inp["scale"])
    check_attention(out, ref, w.name)
    # sampled partials against the oracle's per-range results
    for (b, h) in [(0, 0), (Bn - 1, Hq - 1), (Bn // 2, Hq // 3)]:
        ro, rl = oracle.decode_partitions(b, h, n, P, inp["q"], inp["k_cache"], inp["v_cache"],
                                          inp["block_tables"], inp["context_lens"], inp["scale"])
        assert torch.allclose(o_part[b, h].cpu().double(), ro, atol=2e-3), (b, h)
        assert torch.allclose(lse[b, h].cpu().double(), rl, atol=2e-3, rtol=1e-5), (b, h)


# ------------------------------------------------------------------ small grid
GRID = []
for D in (64, 128):
    for BS in (8, 16, 32, 128):
        for (Hq, Hkv) in ((2, 2), (8, 2), (16, 2)):
            GRID.append((D, BS, Hq, Hkv))
GRID += [(128, 16, 24, 8), (64, 16, 32, 8), (64, 32, 6, 2), (128, 32, 10, 2), (64, 256, 14, 2),
         (64, 64, 4, 4)]


@pytest.mark.parametrize("D,BS,Hq,Hkv", GRID)
def test_small_cases(B, oracle, D, BS, Hq, Hkv):
    lens = (1, 15, 16, 17, 63, 64, 65, 130, 700, 1025)
    w = W.small_workload(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=lens, seed=D + BS + Hq)
    inp = W.make_inputs(w, poison=True)
    g = dev(inp)
    out = step(B, g)
    ref, kc_ref, vc_ref = oracle.step(inp)
    assert torch.equal(g["k_cache"].cpu().view(torch.int16), kc_ref.view(torch.int16))
    check_attention(out, ref, f"auto plan D={D} BS={BS} G={Hq // Hkv}")
    # every explicit partition size over the same (updated) cache
    for P in (64, 128, 320, 1088):
        n = math.ceil(inp["max_context_len"] / P)
        o_part = torch.empty(w.B, Hq, n, D, device="cuda")
        lse = torch.empty(w.B, Hq, n, device="cuda")
        B.paged_decode_split(o_part, lse, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                             g["context_lens"], inp["max_context_len"], inp["scale"], P)
        o2 = torch.empty_like(g["q"])
        B.paged_decode_combine(o2, o_part, lse, g["context_lens"], inp["max_context_len"], P)
        check_attention(o2, ref, f"P={P} D={D} BS={BS} G={Hq // Hkv}")
    assert_no_device_errors(B)


# Few (sequence, kv head) units: the plan gives P = 512 here, so a unit has
# ceil(max_len / 512) partitions.  2..8 of them form one thread-block cluster that merges
# through distributed shared memory; 9 or more merge through global memory.
CLUSTER_CASES = [
    # D, BS, Hq, Hkv, lens, partitions
    (64, 16, 8, 1, (4096,), 8),                      # the largest cluster
    (64, 16, 8, 1, (4097,), 9),                      # one more: global-memory merge
    (128, 32, 8, 1, (1025, 0, 1, 512, 513), 3),      # empty contexts and empty partitions
    (64, 16, 32, 4, (2048, 1500, 3), 4),             # G = 8: two heads per CTA
    (64, 16, 8, 1, (1000, 20), 2),                   # G = 8: four heads per CTA
    (128, 16, 6, 2, (900, 1800), 4),                 # G = 3, head_dim 128
    (64, 8, 2, 2, (600,), 2),                        # G = 1, two partitions
]


@pytest.mark.parametrize("D,BS,Hq,Hkv,lens,parts", CLUSTER_CASES)
def test_cluster_merge_shapes(B, oracle, D, BS, Hq, Hkv, lens, parts):
    w = W.small_workload(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=lens, seed=31 + D + Hq)
    inp = W.make_inputs(w, poison=True)
    P = B.paged_decode_plan(w.B, Hq, Hkv, D, inp["max_context_len"])
    assert math.ceil(inp["max_context_len"] / P) == parts
    assert B.paged_decode_path(w.B, Hq, Hkv, D, inp["max_context_len"]) == (
        B.PATH_CLUSTER if parts <= 8 else B.PATH_PARTITIONS)
    g = dev(inp)
    out = step(B, g)
    ref, kc_ref, _ = oracle.step(inp)
    assert torch.equal(g["k_cache"].cpu().view(torch.int16), kc_ref.view(torch.int16))
    check_attention(out, ref, f"{parts} partitions D={D} G={Hq // Hkv}")
    o = out.cpu()
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.equal(o[b], torch.zeros_like(o[b]))
    assert_no_device_errors(B)


def _lens(n, lo, hi, seed, extra=()):
    g = torch.Generator().manual_seed(seed)
    x = torch.randint(lo, hi + 1, (n,), generator=g).tolist()
    for i, v in enumerate(extra):
        x[(7 * i + 3) % n] = v
    return tuple(int(v) for v in x)


# Many (sequence, kv head) units -- at least one wave of CTAs -- take the persistent
# kernel (at most 1024 sequences); the batch over 1024 takes the grid kernel.  The
# kernel's work order has two forms: where the single-partition items fill a wave of
# CTAs (456 at D=64, 304 at D=128 on 152 SMs), the last partitions of multi-partition
# sequences follow the full partitions (the last two cases); otherwise they are sorted
# in by size.
PERSIST_CASES = [
    # D, BS, Hq, Hkv, lens
    (64, 16, 16, 4, _lens(120, 0, 3000, 1, (0, 1, 63, 64, 1024, 1025, 2048, 3000, 0))),
    (128, 32, 24, 8, _lens(40, 0, 5000, 2, (0, 4096, 1, 2049))),
    (64, 8, 8, 1, _lens(460, 1, 700, 3, (512, 513))),
    (64, 256, 4, 4, _lens(116, 1, 2100, 4, (1024, 2048, 1))),
    (64, 16, 2, 1, _lens(1100, 1, 300, 5)),
    (64, 16, 8, 1, tuple(3000 if b == 17 else 0 for b in range(500))),
    (64, 16, 8, 1, _lens(600, 1, 600, 6, tuple(range(1600, 5000, 120)) + (0, 1536, 1537))),
    (128, 16, 16, 2, _lens(205, 1, 500, 7, (2000, 3100, 4700, 1537, 1536, 0))),
    (64, 16, 32, 4, _lens(300, 1, 4000, 9)),       # many multi-partition sequences, T > 0
    (128, 16, 24, 8, _lens(60, 1, 6000, 10)),      # ... and T = 0
]


@pytest.mark.parametrize("D,BS,Hq,Hkv,lens", PERSIST_CASES)
def test_many_units_decode(B, oracle, D, BS, Hq, Hkv, lens):
    w = W.small_workload(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=lens, seed=41 + D + Hq,
                         write="none")
    inp = W.make_inputs(w, poison=True)
    path = B.paged_decode_path(w.B, Hq, Hkv, D, inp["max_context_len"])
    assert path == (B.PATH_PERSISTENT if w.B <= 1024 else B.PATH_PARTITIONS)
    g = dev(inp)
    ref = oracle.decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                        inp["context_lens"], inp["scale"])
    nbytes = B.paged_decode_workspace_size(w.B, Hq, Hkv, D, inp["max_context_len"])
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for call in range(3):  # the item counter and merge counters are reset by each call
        out = torch.full_like(g["q"], float("nan"))
        B.paged_decode_attention(out, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                                 g["context_lens"], inp["max_context_len"], inp["scale"],
                                 workspace=ws)
        check_attention(out, ref, f"call {call} D={D} BS={BS} G={Hq // Hkv} B={w.B}")
        torch.cuda.synchronize()
        head = ws[:w.B * Hkv * 4 + 8].view(torch.int32)
        assert int(head.abs().sum()) == 0, "counters not back at zero"
    o = out.cpu()
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.equal(o[b], torch.zeros_like(o[b]))
    assert_no_device_errors(B)


def test_very_long_contexts(B, oracle):
    """131072 and 70001 tokens: the plan cuts each (sequence, kv head) into well over a
    hundred partitions merged by the last one through global memory (the merge folds them
    8 at a time), and a chunked prefill of the last 512 tokens walks ~1000 key blocks of
    128 per tile."""
    import itertools
    lens = (131072, 70001)
    w = W.small_workload(B=2, Hq=8, Hkv=1, D=128, BS=32, lens=lens, seed=95, write="last")
    inp = W.make_inputs(w, poison=True)
    P = B.paged_decode_plan(2, 8, 1, 128, inp["max_context_len"])
    assert math.ceil(inp["max_context_len"] / P) > 100
    assert B.paged_decode_path(2, 8, 1, 128, inp["max_context_len"]) == B.PATH_PARTITIONS
    g = dev(inp)
    out = step(B, g)
    ref, kc_ref, vc_ref = oracle.step(inp)
    assert torch.equal(g["k_cache"].cpu().view(torch.int16), kc_ref.view(torch.int16))
    check_attention(out, ref, "131072 tokens")
    # chunked prefill over the updated cache, sampled rows
    chunks = (512, 512)
    qs = torch.tensor([0] + list(itertools.accumulate(chunks)), dtype=torch.int32)
    q = torch.randn(1024, 8, 128, generator=torch.Generator().manual_seed(96)).to(torch.bfloat16)
    po = torch.full((1024, 8, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.paged_prefill_attention(po, q.cuda(), g["k_cache"], g["v_cache"], g["block_tables"],
                              g["context_lens"], inp["max_context_len"], qs.cuda(), 512, inp["scale"])
    got = po.cpu()
    assert torch.isfinite(got.float()).all()
    for b in (0, 1):
        rows = slice(int(qs[b + 1]) - 4, int(qs[b + 1]))
        pref = oracle.prefill(q[rows], kc_ref, vc_ref, inp["block_tables"][b:b + 1],
                              inp["context_lens"][b:b + 1], torch.tensor([0, 4], dtype=torch.int32),
                              inp["scale"])
        check_attention(got[rows], pref, f"prefill at {lens[b]} tokens")
    assert_no_device_errors(B)


def test_large_ragged_batch(B, oracle):
    """Many (sequence, kv head) units with ragged contexts up to 512."""
    lens = tuple(int(x) for x in torch.randint(1, 513, (160,), generator=torch.Generator().manual_seed(4)))
    w = W.small_workload(B=160, Hq=16, Hkv=4, D=64, BS=16, lens=lens, seed=5)
    inp = W.make_inputs(w, poison=True)
    g = dev(inp)
    out = step(B, g)
    ref, _, _ = oracle.step(inp)
    check_attention(out, ref, "ragged B=160")
    assert_no_device_errors(B)


def test_split_partials_match_oracle(B, oracle):
    w = W.small_workload(B=3, Hq=12, Hkv=4, D=128, BS=16, lens=(5, 300, 1000), seed=8, write="none")
    inp = W.make_inputs(w, poison=True)
    g = dev(inp)
    P = 128
    n = math.ceil(1000 / P)
    o_part = torch.full((3, 12, n, 128), float("nan"), device="cuda")
    lse = torch.full((3, 12, n), float("nan"), device="cuda")
    B.paged_decode_split(o_part, lse, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                         g["context_lens"], 1000, inp["scale"], P)
    for b in range(3):
        L = int(inp["context_lens"][b])
        for h in range(12):
            ro, rl = oracle.decode_partitions(b, h, n, P, inp["q"], inp["k_cache"], inp["v_cache"],
                                              inp["block_tables"], inp["context_lens"], inp["scale"])
            k = math.ceil(L / P)
            assert torch.allclose(o_part[b, h, :k].cpu().double(), ro[:k], atol=2e-3), (b, h)
            assert torch.allclose(lse[b, h, :k].cpu().double(), rl[:k], atol=2e-3, rtol=1e-5), (b, h)
            assert torch.isnan(lse[b, h, k:].cpu()).all(), "empty ranges must not be written"
    assert_no_device_errors(B)


def test_combine_alone(B, oracle):
    """The combine kernel on partials computed by the oracle."""
    w = W.small_workload(B=2, Hq=4, Hkv=2, D=64, BS=16, lens=(900, 1), seed=9, write="none")
    inp = W.make_inputs(w)
    P = 64
    n = math.ceil(900 / P)
    o_part = torch.zeros(2, 4, n, 64, dtype=torch.float64)
    lse = torch.zeros(2, 4, n, dtype=torch.float64)
    for b in range(2):
        for h in range(4):
            o_part[b, h], lse[b, h] = oracle.decode_partitions(
                b, h, n, P, inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                inp["context_lens"], inp["scale"])
    out = torch.empty(2, 4, 64, dtype=torch.bfloat16, device="cuda")
    B.paged_decode_combine(out, o_part.float().cuda(), lse.float().cuda(),
                           inp["context_lens"].cuda(), 900, P)
    ref = torch.stack([torch.stack([oracle.lse_combine(o_part[b, h, :math.ceil(int(inp['context_lens'][b]) / P)],
                                                       lse[b, h, :math.ceil(int(inp['context_lens'][b]) / P)])
                                    for h in range(4)]) for b in range(2)])
    check_attention(out, ref, "combine")


# ------------------------------------------------------------------ edge cases
def test_empty_and_length_one(B, oracle):
    w = W.small_workload(B=4, Hq=8, Hkv=2, D=64, BS=16, lens=(0, 1, 0, 1), seed=12, write="none")
    inp = W.make_inputs(w, poison=True)
    g = dev(inp)
    out = step(B, g)
    o = out.cpu()
    assert torch.equal(o[0], torch.zeros_like(o[0])) and torch.equal(o[2], torch.zeros_like(o[2]))
    for b in (1, 3):  # one token: the output is that V row, bit for bit
        phys = int(inp["block_tables"][b, 0])
        for h in range(8):
            assert torch.equal(o[b, h].view(torch.int16), inp["v_cache"][phys, h // 4, 0].view(torch.int16))
    # split path with empty sequences: combine writes zeros
    o_part = torch.empty(4, 8, 1, 64, device="cuda")
    lse = torch.empty(4, 8, 1, device="cuda")
    B.paged_decode_split(o_part, lse, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                         g["context_lens"], 1, inp["scale"], 64)
    o2 = torch.full_like(g["q"], float("nan"))
    B.paged_decode_combine(o2, o_part, lse, g["context_lens"], 1, 64)
    assert torch.equal(o2.cpu().view(torch.int16), o.view(torch.int16))
    assert_no_device_errors(B)


def test_identical_keys_give_mean_of_v(B, oracle):
    w = W.small_workload(B=2, Hq=8, Hkv=2, D=128, BS=32, lens=(333, 1200), seed=13, write="none")
    inp = W.make_inputs(w)
    inp["k_cache"][:] = inp["k_cache"][0, :, :1, :]
    g = dev(inp)
    out = step(B, g)
    ref = oracle.decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                        inp["context_lens"], inp["scale"])
    check_attention(out, ref, "identical keys")
    assert float(ref.abs().max()) < 0.5  # a mean of hundreds of N(0,1) values


def test_pool_permutation_invariance(B):
    """Moving the physical blocks (and rewriting the tables) changes no output bit."""
    w = W.small_workload(B=3, Hq=24, Hkv=8, D=128, BS=16, lens=(100, 517, 2000), seed=14, write="none")
    inp = W.make_inputs(w)
    g = dev(inp)
    out1 = step(B, g)
    NB = inp["num_blocks"]
    p = torch.randperm(NB, generator=torch.Generator().manual_seed(1))
    kc = torch.empty_like(inp["k_cache"])
    vc = torch.empty_like(inp["v_cache"])
    kc[p] = inp["k_cache"]
    vc[p] = inp["v_cache"]
    tab = inp["block_tables"]
    nt = torch.where(tab >= 0, p[tab.clamp(min=0).long()].to(torch.int32), tab)
    g2 = dev(dict(inp, k_cache=kc, v_cache=vc, block_tables=nt))
    out2 = step(B, g2)
    assert torch.equal(out1.cpu().view(torch.int16), out2.cpu().view(torch.int16))


def test_cached_decode_equals_recompute(B, oracle):
    """Appending one token per step through the slot write, then decoding, equals the
    oracle over the finished cache (the llm-stack KV-cache gate, on the GPU path)."""
    w = W.small_workload(B=2, Hq=8, Hkv=2, D=64, BS=16, lens=(40, 90), seed=15, write="none")
    inp = W.make_inputs(w)
    gen = torch.Generator().manual_seed(2)
    steps = 24
    g = dev(inp)
    lens = inp["context_lens"].clone() - steps
    for s in range(steps):
        kn = torch.randn(2, 2, 64, generator=gen).to(torch.bfloat16)
        vn = torch.randn(2, 2, 64, generator=gen).to(torch.bfloat16)
        slots = torch.tensor([int(inp["block_tables"][b, int(lens[b]) // 16]) * 16 + int(lens[b]) % 16
                              for b in range(2)], dtype=torch.int64)
        inp["k_cache"], inp["v_cache"] = oracle.kv_write(kn, vn, slots, inp["k_cache"], inp["v_cache"])
        B.paged_kv_write(kn.cuda(), vn.cuda(), slots.cuda(), g["k_cache"], g["v_cache"])
        lens += 1
        out = torch.empty_like(g["q"])
        B.paged_decode_attention(out, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                                 lens.to(torch.int32).cuda(), int(lens.max()), inp["scale"])
        ref = oracle.decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                            lens.to(torch.int32), inp["scale"])
        check_attention(out, ref, f"step {s}")
    assert torch.equal(g["k_cache"].cpu().view(torch.int16), inp["k_cache"].view(torch.int16))


def test_write_skips_negative_slots_and_keeps_other_bytes(B, oracle):
    w = W.small_workload(B=2, Hq=4, Hkv=4, D=128, BS=8, lens=(9, 30), seed=16, write="none")
    inp = W.make_inputs(w)
    NB = inp["num_blocks"]
    slots = torch.tensor([0, -1, 7, NB * 8 - 1, -5, 13], dtype=torch.int64)
    gen = torch.Generator().manual_seed(3)
    kn = torch.randn(6, 4, 128, generator=gen).to(torch.bfloat16)
    vn = torch.randn(6, 4, 128, generator=gen).to(torch.bfloat16)
    kc, vc = inp["k_cache"].cuda(), inp["v_cache"].cuda()
    B.paged_kv_write(kn.cuda(), vn.cuda(), slots.cuda(), kc, vc)
    ek, ev = oracle.kv_write(kn, vn, slots, inp["k_cache"], inp["v_cache"])
    assert torch.equal(kc.cpu().view(torch.int16), ek.view(torch.int16))
    assert torch.equal(vc.cpu().view(torch.int16), ev.view(torch.int16))
    assert_no_device_errors(B)


def test_non_default_stream(B, oracle):
    w = W.small_workload(B=2, Hq=8, Hkv=2, D=64, BS=16, lens=(700, 50), seed=17)
    inp = W.make_inputs(w, poison=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = dev(inp)
        out = step(B, g)
    s.synchronize()
    ref, _, _ = oracle.step(inp)
    check_attention(out, ref, "side stream")


# --------------------------------------------------------------- device errors
def test_device_error_bits(B):
    """Out-of-range block ids, slots and lengths are caught by the kernels' own bounds
    checks: they raise a bit, never read or write outside the buffers."""
    w = W.small_workload(B=2, Hq=8, Hkv=2, D=64, BS=16, lens=(40, 90), seed=18, write="none")
    inp = W.make_inputs(w)
    g = dev(inp)
    B.pkv_device_errors(clear=True)
    bad_tab = g["block_tables"].clone()
    bad_tab[1, 2] = inp["num_blocks"] + 5
    out = torch.empty_like(g["q"])
    B.paged_decode_attention(out, g["q"], g["k_cache"], g["v_cache"], bad_tab, g["context_lens"],
                             90, inp["scale"])
    assert B.pkv_device_errors(clear=True) & 1
    slots = torch.tensor([inp["num_blocks"] * 16 + 3], dtype=torch.int64, device="cuda")
    kn = torch.zeros(1, 2, 64, dtype=torch.bfloat16, device="cuda")
    before = g["k_cache"].clone()
    B.paged_kv_write(kn, kn, slots, g["k_cache"], g["v_cache"])
    assert B.pkv_device_errors(clear=True) & 2
    assert torch.equal(before.view(torch.int16), g["k_cache"].view(torch.int16))
    lens = g["context_lens"].clone()
    lens[0] = 1000  # past the table's capacity: clamped
    B.paged_decode_attention(out, g["q"], g["k_cache"], g["v_cache"], g["block_tables"], lens,
                             90, inp["scale"])
    assert B.pkv_device_errors(clear=True) & 4
    assert B.pkv_device_errors(clear=True) == 0
    # a prefill whose max_query_len understates a sequence's query count: flagged
    qs = torch.tensor([0, 80, 90], dtype=torch.int32, device="cuda")
    qp = torch.zeros(90, 8, 64, dtype=torch.bfloat16, device="cuda")
    po = torch.empty_like(qp)
    B.paged_prefill_attention(po, qp, g["k_cache"], g["v_cache"], g["block_tables"],
                              g["context_lens"], 90, qs, 10, inp["scale"])
    assert B.pkv_device_errors(clear=True) & 4
    assert B.pkv_device_errors(clear=True) == 0


# ------------------------------------------------------- block-manager driven steps
def test_block_manager_driven_decode_steps(B, oracle):
    """Decode steps whose block tables and slot mappings come from the host block
    manager: prompts written through its slots, one appended token per step, a finished
    sequence freed and a new one admitted into the reused blocks, a LIFO preemption.
    Caches and outputs match the oracle at every step."""
    BS, Hkv, D, Hq, NB = 16, 2, 64, 8, 48
    gen = torch.Generator().manual_seed(21)
    rnd = lambda *s: torch.randn(*s, generator=gen).to(torch.bfloat16)
    kc, vc = rnd(NB, Hkv, BS, D), rnd(NB, Hkv, BS, D)
    kg, vg = kc.cuda(), vc.cuda()
    bm = B.BlockManager(NB, BS)

    def write(ids):
        nonlocal kc, vc
        slots = bm.append_slots(ids)
        kn, vn = rnd(len(ids), Hkv, D), rnd(len(ids), Hkv, D)
        kc, vc = oracle.kv_write(kn, vn, slots, kc, vc)
        return kn, vn, slots

    def admit(s, n):
        bm.add_sequence(s, 0)
        kn, vn, slots = write([s] * n)
        B.paged_kv_write(kn.cuda(), vn.cuda(), slots.cuda(), kg, vg)

    for s, n in ((1, 37), (2, 100), (3, 5)):
        admit(s, n)
    active = [1, 2, 3]
    for step in range(6):
        if step == 2:
            bm.free_sequence(2)
            active.remove(2)
            admit(4, 60)
            active.append(4)
        if step == 4:
            assert bm.preempt_lifo() == 4
            active.remove(4)
        kn, vn, slots = write(active)
        tables, lens = bm.block_tables(active, NB)
        q = rnd(len(active), Hq, D)
        out = torch.empty(len(active), Hq, D, dtype=torch.bfloat16, device="cuda")
        B.paged_decode_step(out, q.cuda(), kn.cuda(), vn.cuda(), slots.cuda(), kg, vg,
                            tables.cuda(), lens.cuda(), int(lens.max()), 0.125)
        ref = oracle.decode(q, kc, vc, tables, lens, 0.125)
        check_attention(out, ref, f"manager step {step}")
        assert torch.equal(kg.cpu().view(torch.int16), kc.view(torch.int16))
        assert torch.equal(vg.cpu().view(torch.int16), vc.view(torch.int16))
    assert_no_device_errors(B)



@pytest.mark.parametrize("zero_copy", [False, True])
def test_whole_step_graph_replay(B, oracle, zero_copy):
    """The whole decode step -- one host-to-device copy of the step's inputs from pinned
    memory, paged_decode_step, the device-to-host copy of the output -- captured once
    as a CUDA graph and replayed for several steps, the host buffers refilled between
    replays (one new token per sequence per step).  Every replay's output matches the
    oracle, the caches match bit for bit, and the merge counters stay consistent across
    replays (the lengths need several partitions).  zero_copy: no copies; the kernels
    read the inputs from, and write the output to, the pinned host buffers."""
    Bn, Hq, Hkv, D, BS, steps = 3, 8, 2, 64, 16, 5
    w = W.small_workload(B=Bn, Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=(1300, 700, 1517), seed=23,
                         write="none")
    inp = W.make_inputs(w)
    final = inp["context_lens"].clone()
    max_len = int(final.max())
    assert B.paged_decode_plan(Bn, Hq, Hkv, D, max_len) < max_len  # several partitions
    kg, vg = inp["k_cache"].cuda(), inp["v_cache"].cuda()
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    shapes = {"q": ((Bn, Hq, D), torch.bfloat16), "k_new": ((Bn, Hkv, D), torch.bfloat16),
              "v_new": ((Bn, Hkv, D), torch.bfloat16), "slot_mapping": ((Bn,), torch.int64),
              "block_tables": (tuple(inp["block_tables"].shape), torch.int32),
              "context_lens": ((Bn,), torch.int32)}
    host = {k: torch.zeros(*shp, dtype=dt).pin_memory() for k, (shp, dt) in shapes.items()}
    devb = {k: torch.zeros(*shp, dtype=dt, device="cuda") for k, (shp, dt) in shapes.items()}
    out = torch.empty(Bn, Hq, D, dtype=torch.bfloat16, device="cuda")
    out_h = torch.empty(Bn, Hq, D, dtype=torch.bfloat16).pin_memory()
    ws = torch.zeros(B.paged_decode_workspace_size(Bn, Hq, Hkv, D, max_len), dtype=torch.uint8,
                     device="cuda")

    def body():
        if zero_copy:
            B.paged_decode_step(out_h, host["q"], host["k_new"], host["v_new"],
                                host["slot_mapping"], kg, vg, host["block_tables"],
                                host["context_lens"], max_len, inp["scale"], workspace=ws)
            return
        for k in names:
            devb[k].copy_(host[k], non_blocking=True)
        B.paged_decode_step(out, devb["q"], devb["k_new"], devb["v_new"], devb["slot_mapping"],
                            kg, vg, devb["block_tables"], devb["context_lens"], max_len,
                            inp["scale"], workspace=ws)
        out_h.copy_(out, non_blocking=True)

    gen = torch.Generator().manual_seed(5)
    rnd = lambda *s: torch.randn(*s, generator=gen).to(torch.bfloat16)
    kc, vc = inp["k_cache"], inp["v_cache"]
    lens = final - steps
    stream = torch.cuda.Stream()
    graph = None
    for s in range(steps + 1):
        lens = lens + 1 if s > 0 else lens
        slots = torch.tensor([int(inp["block_tables"][b, (int(lens[b]) - 1) // BS]) * BS
                              + (int(lens[b]) - 1) % BS for b in range(Bn)], dtype=torch.int64)
        fill = {"q": rnd(Bn, Hq, D), "k_new": rnd(Bn, Hkv, D), "v_new": rnd(Bn, Hkv, D),
                "slot_mapping": slots, "block_tables": inp["block_tables"],
                "context_lens": lens.to(torch.int32)}
        for k in names:
            host[k].copy_(fill[k])
        kc, vc = oracle.kv_write(fill["k_new"], fill["v_new"], slots, kc, vc)
        if s == 0:   # the first step runs eagerly (warm-up), then the graph is captured
            with torch.cuda.stream(stream):
                body()
            stream.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                body()
        else:
            with torch.cuda.stream(stream):
                graph.replay()
            stream.synchronize()
        ref = oracle.decode(fill["q"], kc, vc, inp["block_tables"], lens.to(torch.int32),
                            inp["scale"])
        check_attention(out_h.clone(), ref, f"graph step {s}")
    assert torch.equal(kg.cpu().view(torch.int16), kc.view(torch.int16))
    assert torch.equal(vg.cpu().view(torch.int16), vc.view(torch.int16))
    assert int(ws[:Bn * Hkv * 4].view(torch.int32).abs().sum()) == 0  # counters back at zero
    assert_no_device_errors(B)


# ---------------------------------------------------------------- fused RoPE write
from pins import rope_table  # noqa: E402


@pytest.mark.parametrize("D,r,neox,Hq,Hkv", [(64, 64, True, 8, 2), (128, 128, True, 24, 8),
                                             (128, 128, False, 12, 4), (64, 32, True, 4, 4),
                                             (128, 64, False, 16, 2), (64, 16, True, 8, 1)])
def test_rope_write_bit_exact(B, oracle, D, r, neox, Hq, Hkv):
    T, BS, NB, maxpos = 37, 16, 20, 5000
    gen = torch.Generator().manual_seed(D + r + Hq)
    rnd = lambda *s: torch.randn(*s, generator=gen).to(torch.bfloat16)
    k, v, q = rnd(T, Hkv, D), rnd(T, Hkv, D), rnd(T, Hq, D)
    kc, vc = rnd(NB, Hkv, BS, D), rnd(NB, Hkv, BS, D)
    slots = torch.randperm(NB * BS, generator=gen)[:T].to(torch.int64)
    slots[3] = -1
    pos = torch.randint(0, maxpos, (T,), generator=gen, dtype=torch.int64)
    cs = rope_table(maxpos, r, base=500000.0).float()
    ek, ev, eq = oracle.kv_write_rope(k, v, slots, pos, cs, kc, vc, q=q, rotary_dim=r, neox_style=neox)
    kg, vg, qg = kc.cuda(), vc.cuda(), q.cuda()
    B.paged_kv_write_rope(k.cuda(), v.cuda(), slots.cuda(), pos.cuda(), cs.cuda(), kg, vg, q=qg,
                          rotary_dim=r, neox_style=neox)
    torch.cuda.synchronize()
    assert torch.equal(kg.cpu().view(torch.int16), ek.view(torch.int16))
    assert torch.equal(vg.cpu().view(torch.int16), ev.view(torch.int16))
    assert torch.equal(qg.cpu().view(torch.int16), eq.view(torch.int16))
    assert_no_device_errors(B)


def test_rope_write_then_decode(B, oracle):
    """One decode step with RoPE: rotate the step's q and new k at position L-1, write, attend."""
    w = W.small_workload(B=4, Hq=32, Hkv=8, D=128, BS=16, lens=(1, 200, 513, 1300), seed=33)
    inp = W.make_inputs(w, poison=True)
    pos = (inp["context_lens"].long() - 1).clamp(min=0)
    cs = rope_table(2048, 128).float()
    kc, vc, qr = oracle.kv_write_rope(inp["k_new"], inp["v_new"], inp["slot_mapping"], pos, cs,
                                      inp["k_cache"], inp["v_cache"], q=inp["q"])
    ref = oracle.decode(qr, kc, vc, inp["block_tables"], inp["context_lens"], inp["scale"])
    g = dev(inp)
    B.paged_kv_write_rope(g["k_new"], g["v_new"], g["slot_mapping"], pos.cuda(), cs.cuda(),
                          g["k_cache"], g["v_cache"], q=g["q"])
    out = torch.empty_like(g["q"])
    B.paged_decode_attention(out, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                             g["context_lens"], g["max_context_len"], g["scale"])
    check_attention(out, ref, "rope + decode")
    assert torch.equal(g["q"].cpu().view(torch.int16), qr.view(torch.int16))


STEP_ROPE_CASES = [
    # D, BS, Hq, Hkv, lens, rotary_dim, neox, path
    (64, 16, 8, 2, (37, 100, 5), 64, True, "partitions"),
    (128, 16, 8, 2, (1500, 700), 128, False, "cluster"),
    (64, 16, 16, 4, _lens(120, 1, 3000, 6, (1, 1536, 1537)), 32, True, "persistent"),
    (128, 32, 24, 8, _lens(40, 1, 4000, 7), 64, False, "persistent"),
]


@pytest.mark.parametrize("D,BS,Hq,Hkv,lens,r,neox,path", STEP_ROPE_CASES)
def test_decode_step_rope(B, oracle, D, BS, Hq, Hkv, lens, r, neox, path):
    """paged_decode_step_rope: q rotated in place and k rotated and written bit for bit
    like the oracle; the attention (a programmatic dependent that reads q after the
    rotary write) within tolerance of the oracle over the rotated q and caches."""
    w = W.small_workload(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=lens, seed=51 + D + r)
    inp = W.make_inputs(w, poison=True)
    want = {"partitions": B.PATH_PARTITIONS, "cluster": B.PATH_CLUSTER,
            "persistent": B.PATH_PERSISTENT}[path]
    assert B.paged_decode_path(w.B, Hq, Hkv, D, inp["max_context_len"]) == want
    pos = (inp["context_lens"].long() - 1).clamp(min=0)
    cs = rope_table(inp["max_context_len"] + 1, r).float()
    kc, vc, qr = oracle.kv_write_rope(inp["k_new"], inp["v_new"], inp["slot_mapping"], pos, cs,
                                      inp["k_cache"], inp["v_cache"], q=inp["q"], rotary_dim=r,
                                      neox_style=neox)
    ref = oracle.decode(qr, kc, vc, inp["block_tables"], inp["context_lens"], inp["scale"])
    g = dev(inp)
    out = torch.empty_like(g["q"])
    B.paged_decode_step_rope(out, g["q"], g["k_new"], g["v_new"], g["slot_mapping"], pos.cuda(),
                             cs.cuda(), g["k_cache"], g["v_cache"], g["block_tables"],
                             g["context_lens"], g["max_context_len"], g["scale"], rotary_dim=r,
                             neox_style=neox)
    check_attention(out, ref, f"rope step {path} D={D} r={r}")
    assert torch.equal(g["q"].cpu().view(torch.int16), qr.view(torch.int16))
    assert torch.equal(g["k_cache"].cpu().view(torch.int16), kc.view(torch.int16))
    assert torch.equal(g["v_cache"].cpu().view(torch.int16), vc.view(torch.int16))
    assert_no_device_errors(B)


def test_rope_position_out_of_range_is_flagged(B):
    k = torch.zeros(2, 1, 64, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 1, 16, 64, dtype=torch.bfloat16, device="cuda")
    cs = rope_table(8, 64).float().cuda()
    B.pkv_device_errors(clear=True)
    B.paged_kv_write_rope(k, k, torch.tensor([0, 1], device="cuda"), torch.tensor([3, 8], device="cuda"),
                          cs, kc, kc.clone())
    assert B.pkv_device_errors(clear=True) == 16


# ------------------------------------------------------------------ paged prefill
PREFILL = [
    # D, BS, Hq, Hkv, lens, chunks
    (64, 16, 8, 2, (37, 100, 1, 300), (37, 20, 1, 300)),
    (128, 16, 24, 8, (513, 64, 1000), (513, 64, 7)),
    (128, 32, 12, 4, (65, 130), (1, 130)),
    (64, 8, 4, 4, (200, 31, 17), (50, 31, 16)),
    (64, 128, 16, 2, (700, 2), (120, 2)),
    (128, 16, 8, 1, (90, 90), (90, 45)),
]


@pytest.mark.parametrize("D,BS,Hq,Hkv,lens,chunks", PREFILL)
def test_prefill_matches_oracle(B, oracle, D, BS, Hq, Hkv, lens, chunks):
    import itertools
    w = W.small_workload(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=lens, seed=D + BS + Hq,
                         write="none")
    inp = W.make_inputs(w, poison=True)
    gen = torch.Generator().manual_seed(len(lens))
    qs = torch.tensor([0] + list(itertools.accumulate(chunks)), dtype=torch.int32)
    q = torch.randn(int(qs[-1]), Hq, D, generator=gen).to(torch.bfloat16)
    ref = oracle.prefill(q, inp["k_cache"], inp["v_cache"], inp["block_tables"], inp["context_lens"],
                         qs, inp["scale"])
    g = dev(inp)
    out = torch.full((int(qs[-1]), Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.paged_prefill_attention(out, q.cuda(), g["k_cache"], g["v_cache"], g["block_tables"],
                              g["context_lens"], inp["max_context_len"], qs.cuda(), max(chunks),
                              inp["scale"])
    check_attention(out, ref, f"prefill D={D} BS={BS} G={Hq // Hkv}")
    assert_no_device_errors(B)


@pytest.mark.parametrize("D,BS,Hq,Hkv", [(128, 32, 8, 2), (64, 16, 12, 4)])
def test_prefill_wide_scores_and_full_tiles(B, oracle, D, BS, Hq, Hkv):
    """Scores spread wide (scale 1): a row's running max often jumps by more than 2^8,
    so the rescale of O in TMEM runs.  Several full 128-row tiles per (sequence, kv
    head), causal diagonals inside key blocks, and a ragged last block."""
    import itertools
    lens, chunks = (1100, 400, 129), (260, 400, 3)
    w = W.small_workload(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=lens, seed=61 + D,
                         write="none")
    inp = W.make_inputs(w, poison=True)
    gen = torch.Generator().manual_seed(62)
    qs = torch.tensor([0] + list(itertools.accumulate(chunks)), dtype=torch.int32)
    q = torch.randn(int(qs[-1]), Hq, D, generator=gen).to(torch.bfloat16)
    ref = oracle.prefill(q, inp["k_cache"], inp["v_cache"], inp["block_tables"], inp["context_lens"],
                         qs, 1.0)
    g = dev(inp)
    out = torch.full((int(qs[-1]), Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.paged_prefill_attention(out, q.cuda(), g["k_cache"], g["v_cache"], g["block_tables"],
                              g["context_lens"], inp["max_context_len"], qs.cuda(), max(chunks), 1.0)
    check_attention(out, ref, f"prefill scale 1 D={D} G={Hq // Hkv}")
    assert_no_device_errors(B)


@pytest.mark.parametrize("wid", [2, 3, 4, 5])
def test_workload_prefill_every_row(B, oracle, wid):
    """Prefill of the last min(L, 512) tokens of every sequence at the workload's full size
    (the configuration bench.py --kernel prefill times), every query row of every head
    against the oracle (threads over (sequence, kv head) pairs): the causal diagonal of
    every 128-row tile, the ragged last tiles and the ragged last key blocks included."""
    import itertools
    w = W.WORKLOADS[wid]
    inp = W.make_inputs(w, poison=True)
    Bn, Hq, D = inp["q"].shape
    lens = inp["context_lens"].long()
    chunks = torch.clamp(lens, max=512)
    qs = torch.tensor([0] + list(itertools.accumulate(chunks.tolist())), dtype=torch.int32)
    gen = torch.Generator().manual_seed(70 + wid)
    q = torch.randn(int(qs[-1]), Hq, D, generator=gen).to(torch.bfloat16)
    g = dev(inp)
    out = torch.full((int(qs[-1]), Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.paged_prefill_attention(out, q.cuda(), g["k_cache"], g["v_cache"], g["block_tables"],
                              g["context_lens"], inp["max_context_len"], qs.cuda(),
                              int(chunks.max()), inp["scale"])
    torch.cuda.synchronize()
    assert_no_device_errors(B)
    got = out.cpu()
    del g, out
    ref = oracle.prefill(q, inp["k_cache"], inp["v_cache"], inp["block_tables"],
                         inp["context_lens"], qs, inp["scale"])
    check_attention(got, ref, f"{w.name} prefill, all {int(qs[-1])} query rows")


@pytest.mark.parametrize("wid", [2, 3, 4, 5])
def test_workload_decode_step_rope(B, oracle, wid):
    """paged_decode_step_rope at the workload's full size (bench.py --kernel rope_step):
    q and both caches bit for bit, every output within tolerance."""
    w = W.WORKLOADS[wid]
    inp = W.make_inputs(w, poison=True)
    D = inp["q"].shape[2]
    pos = (inp["context_lens"].long() - 1).clamp(min=0)
    cs = rope_table(inp["max_context_len"] + 1, D).float()
    kc, vc, qr = oracle.kv_write_rope(inp["k_new"], inp["v_new"], inp["slot_mapping"], pos, cs,
                                      inp["k_cache"], inp["v_cache"], q=inp["q"])
    ref = oracle.decode(qr, kc, vc, inp["block_tables"], inp["context_lens"], inp["scale"])
    g = dev(inp)
    out = torch.empty_like(g["q"])
    B.paged_decode_step_rope(out, g["q"], g["k_new"], g["v_new"], g["slot_mapping"], pos.cuda(),
                             cs.cuda(), g["k_cache"], g["v_cache"], g["block_tables"],
                             g["context_lens"], g["max_context_len"], g["scale"])
    torch.cuda.synchronize()
    assert_no_device_errors(B)
    assert torch.equal(g["q"].cpu().view(torch.int16), qr.view(torch.int16))
    assert torch.equal(g["k_cache"].cpu().view(torch.int16), kc.view(torch.int16))
    assert torch.equal(g["v_cache"].cpu().view(torch.int16), vc.view(torch.int16))
    check_attention(out, ref, f"{w.name} rope step")


@pytest.mark.parametrize("D,BS", [(64, 16), (128, 32)])
@pytest.mark.parametrize("wide", [False, True])
def test_prefill_two_tiles_ragged(B, oracle, D, BS, wide):
    """Enough (sequence, kv head) units (40 x 8 = 320 >= two waves on 152 SMs) that the
    launcher gives each CTA two 128-row query tiles: ragged lengths, chunk sizes from one
    token to the whole sequence, tiles whose second half is empty.  With `wide`, scale 1
    spreads the scores so that rows' maxima jump between key blocks and the rescale of O
    in TMEM runs (at head_dim 64 it also rescales the row-sum column that the tensor core
    accumulates)."""
    import itertools
    gen = torch.Generator().manual_seed(90 + D)
    lens = [int(x) for x in torch.randint(1, 261, (40,), generator=gen)]
    chunks = [max(1, int(torch.randint(0, L + 1, (1,), generator=gen))) for L in lens]
    chunks[0], chunks[1] = lens[0], 1
    w = W.small_workload(B=40, Hq=16, Hkv=8, D=D, BS=BS, lens=tuple(lens), seed=91 + D, write="none")
    inp = W.make_inputs(w, poison=True)
    qs = torch.tensor([0] + list(itertools.accumulate(chunks)), dtype=torch.int32)
    q = torch.randn(int(qs[-1]), 16, D, generator=gen).to(torch.bfloat16)
    scale = 1.0 if wide else inp["scale"]
    ref = oracle.prefill(q, inp["k_cache"], inp["v_cache"], inp["block_tables"], inp["context_lens"],
                         qs, scale)
    g = dev(inp)
    out = torch.full((int(qs[-1]), 16, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.paged_prefill_attention(out, q.cuda(), g["k_cache"], g["v_cache"], g["block_tables"],
                              g["context_lens"], inp["max_context_len"], qs.cuda(), max(chunks),
                              scale)
    # At scale 1 the scores spread over tens of units (base 2), the lazy reference max is
    # often stale by up to 2^8, and each weight enters P.V as one bf16 value (2^-9
    # relative).  Those weights' rounding then adds up to another 2^-9 |out| on top of the
    # output's own bf16 half-ulp, so here the 2^-8 |oracle| term applies to every element
    # (measured at head_dim 128: 2 of 5.5 M outputs between 1e-2 and 1.6e-2).
    check_attention(out, ref, f"two-tile prefill D={D} BS={BS} scale={scale}",
                    abs_only_below=0.0 if wide else ABS_ONLY_BELOW)
    assert_no_device_errors(B)


def test_prefill_single_token_chunks_equal_decode(B, oracle):
    """A chunk of one token per sequence is a decode step."""
    w = W.small_workload(B=3, Hq=32, Hkv=8, D=64, BS=16, lens=(5, 900, 2048), seed=51, write="none")
    inp = W.make_inputs(w, poison=True)
    g = dev(inp)
    qs = torch.arange(4, dtype=torch.int32).cuda()
    out = torch.empty_like(g["q"])
    B.paged_prefill_attention(out, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                              g["context_lens"], inp["max_context_len"], qs, 1, inp["scale"])
    dec = torch.empty_like(g["q"])
    B.paged_decode_attention(dec, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                             g["context_lens"], inp["max_context_len"], inp["scale"])
    ref = oracle.decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                        inp["context_lens"], inp["scale"])
    check_attention(out, ref, "prefill n=1")
    check_attention(dec, ref, "decode")


# ------------------------------------------------- CUDA-core form of the consumer warps
@pytest.fixture
def fma_consumer(B):
    prev = B.pkv_set_decode_consumer(B.CONSUMER_FMA)
    yield
    B.pkv_set_decode_consumer(prev)


@pytest.mark.parametrize("D,BS,Hq,Hkv", [(64, 16, 8, 2), (128, 16, 24, 8), (64, 32, 32, 4),
                                         (128, 32, 16, 2), (64, 16, 4, 4), (128, 8, 8, 8)])
def test_fma_consumer_small_cases(B, oracle, fma_consumer, D, BS, Hq, Hkv):
    """The CUDA-core consumer (fp32 FMAs, shuffles) against the oracle: the launcher's
    plan (cluster or partition path), then explicit partitions through split + combine;
    ragged lengths, partial 16-key groups, G from 1 to 8."""
    lens = (1, 15, 16, 17, 63, 64, 65, 130, 700, 1025)
    w = W.small_workload(B=len(lens), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=lens, seed=7 * D + BS + Hq)
    inp = W.make_inputs(w, poison=True)
    assert B.paged_decode_path(w.B, Hq, Hkv, D, inp["max_context_len"]) in (B.PATH_CLUSTER,
                                                                            B.PATH_PARTITIONS)
    g = dev(inp)
    out = step(B, g)
    ref, kc_ref, vc_ref = oracle.step(inp)
    check_attention(out, ref, f"fma consumer D={D} BS={BS} G={Hq // Hkv}")
    for P in (64, 320):
        n = math.ceil(inp["max_context_len"] / P)
        o_part = torch.empty(w.B, Hq, n, D, device="cuda")
        lse = torch.empty(w.B, Hq, n, device="cuda")
        B.paged_decode_split(o_part, lse, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                             g["context_lens"], inp["max_context_len"], inp["scale"], P)
        o2 = torch.empty_like(g["q"])
        B.paged_decode_combine(o2, o_part, lse, g["context_lens"], inp["max_context_len"], P)
        check_attention(o2, ref, f"fma consumer P={P} D={D} G={Hq // Hkv}")
    assert_no_device_errors(B)


@pytest.mark.parametrize("wid,P", [(1, 0), (2, 0), (5, 0), (3, 1024), (4, 1024)])
def test_fma_consumer_workloads(B, oracle, fma_consumer, wid, P):
    """Full workloads with the CUDA-core consumer, in the configuration bench.py times it:
    the fused step on the partition kernel's paths (workloads 1, 2, 5), and split +
    combine at P = 1024 where the fused step takes the persistent kernel (3, 4)."""
    w = W.WORKLOADS[wid]
    inp = W.make_inputs(w, poison=True)
    g = dev(inp)
    ref, kc_ref, vc_ref = oracle.step(inp)
    if P == 0:
        out = step(B, g)
    else:
        B.paged_kv_write(g["k_new"], g["v_new"], g["slot_mapping"], g["k_cache"], g["v_cache"])
        Bn, Hq, D = inp["q"].shape
        n = math.ceil(inp["max_context_len"] / P)
        o_part = torch.empty(Bn, Hq, n, D, device="cuda")
        lse = torch.empty(Bn, Hq, n, device="cuda")
        B.paged_decode_split(o_part, lse, g["q"], g["k_cache"], g["v_cache"], g["block_tables"],
                             g["context_lens"], inp["max_context_len"], inp["scale"], P)
        out = torch.empty_like(g["q"])
        B.paged_decode_combine(out, o_part, lse, g["context_lens"], inp["max_context_len"], P)
    torch.cuda.synchronize()
    assert_no_device_errors(B)
    check_attention(out, ref, f"{w.name} (fma consumer)")


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("path", ["partitions", "persistent"])
def test_decode_kernels_fit_the_planned_ctas_per_sm(B, D, path):
    """The launcher sizes grids for 3 decode CTAs per SM at head_dim 64 and 2 at 128; a
    kernel whose registers or shared memory no longer allow that would run a second wave
    of CTAs.  Checked against the CUDA runtime's occupancy for the built kernels, both
    consumer forms of the partition kernel included."""
    want = 3 if D == 64 else 2
    p = B.PATH_PERSISTENT if path == "persistent" else B.PATH_PARTITIONS
    assert B.pkv_decode_ctas_per_sm(D, p) == want
    if path == "partitions":
        prev = B.pkv_set_decode_consumer(B.CONSUMER_FMA)
        try:
            assert B.pkv_decode_ctas_per_sm(D, p) == want
        finally:
            B.pkv_set_decode_consumer(prev)


@pytest.mark.parametrize("wid", [2, 3, 4])
def test_decode_step_zero_copy_matches_device_inputs(B, wid):
    """paged_decode_step with the step's inputs and output in pinned host memory (the
    kernels read and write them over the host link) gives bit for bit the output and the
    caches of the same step on device copies, on the cluster (2) and persistent (3, 4)
    arrangements."""
    w = W.WORKLOADS[wid]
    inp = W.make_inputs(w)
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    host = {k: inp[k].contiguous().pin_memory() for k in names}
    dev = {k: inp[k].cuda() for k in names}
    outs, caches = [], []
    for src in (dev, host):
        kc, vc = inp["k_cache"].cuda(), inp["v_cache"].cuda()
        out = (torch.empty(inp["q"].shape, dtype=torch.bfloat16, device="cuda") if src is dev
               else torch.empty(inp["q"].shape, dtype=torch.bfloat16).pin_memory())
        B.paged_decode_step(out, src["q"], src["k_new"], src["v_new"], src["slot_mapping"], kc, vc,
                            src["block_tables"], src["context_lens"], inp["max_context_len"],
                            inp["scale"])
        torch.cuda.synchronize()
        outs.append(out.cpu())
        caches.append((kc.cpu(), vc.cpu()))
        del kc, vc
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(caches[0][0].view(torch.int16), caches[1][0].view(torch.int16))
    assert torch.equal(caches[0][1].view(torch.int16), caches[1][1].view(torch.int16))
    assert_no_device_errors(B)


@pytest.mark.parametrize("wid", [1, 2, 5])
def test_decode_attention_and_write_zero_copy(B, wid):
    """paged_kv_write and paged_decode_attention with their per-step arguments in pinned
    host memory (workload 1: one partition; 2: cluster merge; 5: ticket merge) give bit
    for bit the caches and output of the same calls on device copies."""
    w = W.WORKLOADS[wid]
    inp = W.make_inputs(w)
    results = []
    for host in (False, True):
        put = (lambda t: t.contiguous().pin_memory()) if host else (lambda t: t.cuda())
        kc, vc = inp["k_cache"].cuda(), inp["v_cache"].cuda()
        B.paged_kv_write(put(inp["k_new"]), put(inp["v_new"]), put(inp["slot_mapping"]), kc, vc)
        out = put(torch.empty(inp["q"].shape, dtype=torch.bfloat16))
        B.paged_decode_attention(out, put(inp["q"]), kc, vc, put(inp["block_tables"]),
                                 put(inp["context_lens"]), inp["max_context_len"], inp["scale"])
        torch.cuda.synchronize()
        results.append((out.cpu().view(torch.int16), kc.cpu().view(torch.int16),
                        vc.cpu().view(torch.int16)))
        del kc, vc
    for a, b in zip(*results):
        assert torch.equal(a, b)
    assert_no_device_errors(B)
