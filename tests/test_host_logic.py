"""Host-side logic without a GPU: the split plan, workspace sizing, the seeded
input recipe, and the per-rank sharding of independent sequences."""

import math

import pytest
import torch

from paged_kv_decode_mapping_gb300 import workloads as W


@pytest.fixture(scope="module")
def B():
    from paged_kv_decode_mapping_gb300 import build

    build.build()
    from paged_kv_decode_mapping_gb300 import binding

    return binding


def test_plan_picks_partitions_from_context_length(B):
    """Few (sequence, kv head) units: about one wave of long partitions (3 CTAs/SM at
    head_dim 64, 2 at 128); many units: 1024 tokens; never below min(context, 512)."""
    sms = 152
    assert B.paged_decode_plan(1, 32, 8, 64, 128, sms) == 128          # short: one partition
    assert B.paged_decode_plan(16, 32, 8, 64, 2048, sms) == 704        # 128 units x 3 = 384 CTAs
    assert B.paged_decode_plan(4, 24, 8, 128, 32768, sms) == 3648      # 32 units x 9 = 288 CTAs
    assert B.paged_decode_plan(64, 24, 8, 128, 4096, sms) == 1536      # 512 units >= 304 slots
    assert B.paged_decode_plan(256, 32, 4, 64, 8192, sms) == 1536      # persistent work items
    assert B.paged_decode_plan(2048, 8, 1, 64, 8192, sms) == 1024      # > 1024 sequences
    assert B.paged_decode_plan(256, 32, 4, 64, 300, sms) == 320        # short contexts stay whole
    assert B.paged_decode_plan(1, 8, 8, 64, 1, sms) == 64
    assert B.paged_decode_plan(0, 8, 8, 64, 4096, sms) == 0
    assert B.paged_decode_plan(2, 8, 8, 96, 4096, sms) == 0            # unsupported head_dim
    assert B.paged_decode_plan(2, 8, 1, 64, 4096, sms) == 512          # group 8: the largest built
    assert B.paged_decode_plan(2, 16, 1, 64, 4096, sms) == 0           # group 16: not built
    for b, hq, h, d, L in [(1, 1, 1, 64, 100_000), (3, 12, 4, 128, 5000), (1000, 8, 8, 64, 600)]:
        P = B.paged_decode_plan(b, hq, h, d, L, sms)
        assert P % 64 == 0 and P >= min(512, -(-L // 64) * 64)


def test_path_follows_the_plan(B):
    sms = 152
    P = lambda *a: B.paged_decode_path(*a, sms)
    assert P(1, 32, 8, 64, 128) == B.PATH_PARTITIONS          # one partition: nothing to merge
    assert P(16, 32, 8, 64, 2048) == B.PATH_CLUSTER           # 3 partitions per unit, one wave
    assert P(4, 24, 8, 128, 32768) == B.PATH_PARTITIONS       # 9 partitions: above the cluster limit
    assert P(1, 8, 1, 64, 4096) == B.PATH_CLUSTER             # 8 partitions: the largest cluster
    assert P(1, 8, 1, 64, 4097) == B.PATH_PARTITIONS
    assert P(64, 24, 8, 128, 4096) == B.PATH_PERSISTENT       # 512 units >= 304 slots
    assert P(256, 32, 4, 64, 8192) == B.PATH_PERSISTENT
    assert P(2048, 8, 1, 64, 8192) == B.PATH_PARTITIONS       # more sequences than its tables hold
    assert P(400, 8, 1, 64, 4096) == B.PATH_PARTITIONS        # 400 units < 456 slots: whole
    assert P(200, 8, 1, 64, 4096) == B.PATH_CLUSTER           # 2 partitions each, 400 CTAs
    # the persistent kernel's work order has at most 64 categories: R - 1 full-partition
    # levels + 24 + 2 last-partition sizes at P = 1536, so contexts up to 39 * 1536
    assert P(600, 8, 1, 64, 59904) == B.PATH_PERSISTENT
    assert P(600, 8, 1, 64, 59905) == B.PATH_PARTITIONS
    assert P(0, 8, 1, 64, 4096) == 0
    assert P(2, 16, 1, 64, 4096) == 0                         # unsupported group


def test_workspace_sizes(B):
    # o_part [B, Hq, n, D] fp32 + lse_part [B, Hq, n] fp32, each padded to 256 bytes
    n = math.ceil(32768 / 512)
    rows = 4 * 24 * n
    expect = -(-rows * 128 * 4 // 256) * 256 + -(-rows * 4 // 256) * 256
    assert B.paged_decode_split_workspace_size(4, 24, 128, 32768, 512) == expect
    assert B.paged_decode_split_workspace_size(4, 24, 128, 0, 512) == 0
    assert B.paged_decode_split_workspace_size(4, 24, 128, 100, 0) == 0
    # paged_decode_attention: counters [B*Hkv] u32 and two scheduling words, then the
    # split layout for the planned P
    up = lambda x: -(-x // 256) * 256
    for (b, hkv) in ((4, 8), (64, 8), (1, 8)):
        P = B.paged_decode_plan(b, 24, hkv, 128, 32768)
        assert B.paged_decode_workspace_size(b, 24, hkv, 128, 32768) == (
            up(b * hkv * 4 + 8) + B.paged_decode_split_workspace_size(b, 24, 128, 32768, P))


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_workload_recipe(wid):
    w = W.WORKLOADS[wid]
    if wid in (3, 5):  # big pools: check the drawn metadata on a copy with a tiny head dim
        import dataclasses
        w = dataclasses.replace(w, D=8)
    inp = W.make_inputs(w)
    lens = inp["context_lens"]
    assert inp["q"].shape == (w.B, w.Hq, w.D) and inp["q"].dtype == torch.bfloat16
    assert inp["k_cache"].shape == (inp["num_blocks"], w.Hkv, w.BS, w.D)
    if w.lens == "fixed":
        assert (lens == w.L).all()
    if w.lens == "uniform":
        assert lens.min() >= w.L_lo and lens.max() <= w.L_hi
    if w.lens == "lognormal":
        assert lens.min() >= w.L_lo and lens.max() <= w.L_hi
        assert 300 < float(lens.double().median()) < 800
    nblk = (lens + w.BS - 1) // w.BS
    used = torch.cat([inp["block_tables"][b, :int(nblk[b])] for b in range(w.B)])
    assert len(set(used.tolist())) == len(used), "a physical block is owned twice"
    assert used.min() >= 0 and used.max() < inp["num_blocks"]
    if w.pool_blocks:
        assert inp["num_blocks"] == w.pool_blocks
    else:
        assert inp["num_blocks"] == math.ceil(w.pool_factor * int(nblk.sum()))
    if w.write == "last":
        for b in range(w.B):
            pos = int(lens[b]) - 1
            assert int(inp["slot_mapping"][b]) == int(inp["block_tables"][b, pos // w.BS]) * w.BS + pos % w.BS
    # deterministic: the same seed draws the same inputs
    again = W.make_inputs(w)
    assert torch.equal(again["q"].view(torch.int16), inp["q"].view(torch.int16))
    assert torch.equal(again["block_tables"], inp["block_tables"])


def test_poison_marks_only_unowned_slots():
    w = W.small_workload(B=2, Hq=4, Hkv=2, D=8, BS=4, lens=(5, 3), seed=1)
    inp = W.make_inputs(w, poison=True)
    kc = inp["k_cache"].float()
    for b, L in enumerate(inp["context_lens"].tolist()):
        for t in range(L):
            assert torch.isfinite(kc[int(inp["block_tables"][b, t // 4]), :, t % 4]).all()
    assert int(torch.isnan(kc[:, 0, :, 0]).sum()) == inp["num_blocks"] * 4 - 8


def test_shard_range_partitions_sequences():
    for n in (0, 1, 5, 16, 257):
        for world in (1, 2, 3, 8):
            seen = []
            for r in range(world):
                lo, hi = W.shard_range(n, r, world)
                seen.extend(range(lo, hi))
            assert seen == list(range(n))
