"""The host block manager (pkv_bm_*) against the reference model, on the CPU.

Random admit / append / free / preempt sequences drive both; after every operation they
must agree on every quantity the pages fix (success or no-space, lengths, blocks per
sequence, free blocks, the LIFO victim), and the manager's state must be valid: no block
owned twice, every table exactly ceil(length / block_size) long, and every slot it
handed out equal to table[pos // block_size] * block_size + pos % block_size.
"""

import random

import pytest
import torch

from oracle.block_manager import BlockManagerModel, NoSpace


@pytest.fixture(scope="module")
def B():
    from paged_kv_decode_mapping_gb300 import build

    build.build()
    from paged_kv_decode_mapping_gb300 import binding

    return binding


def check_state(B, bm, model, slots_seen):
    ids = sorted(model.lens)
    maxb = max([model.blocks_of(s) for s in ids] + [1])
    tables, lens = bm.block_tables(ids, maxb)
    owned = []
    for i, s in enumerate(ids):
        assert int(lens[i]) == model.lens[s]
        n = model.blocks_of(s)
        row = tables[i].tolist()
        assert all(x >= 0 for x in row[:n]) and all(x == -1 for x in row[n:])
        owned += row[:n]
        for pos, slot in slots_seen.get(s, {}).items():
            assert slot == row[pos // bm.block_size] * bm.block_size + pos % bm.block_size
    assert len(owned) == len(set(owned)), "a block is owned twice"
    assert all(0 <= x < bm.num_blocks for x in owned)
    assert bm.num_free_blocks == model.num_free == bm.num_blocks - len(owned)


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_the_model(B, seed):
    rng = random.Random(seed)
    NB, BS = rng.choice([(8, 4), (16, 2), (40, 16), (5, 1)])
    bm, model = B.BlockManager(NB, BS), BlockManagerModel(NB, BS)
    slots_seen = {}
    next_id = 100
    for _ in range(300):
        op = rng.random()
        if op < 0.3:
            n = rng.randint(0, 3 * BS)
            try:
                model.add(next_id, n)
                ok = True
            except NoSpace:
                ok = False
            if ok:
                bm.add_sequence(next_id, n)
            else:
                with pytest.raises(B.PkvError) as e:
                    bm.add_sequence(next_id, n)
                assert e.value.code == -8
            next_id += 1
        elif op < 0.75 and model.lens:
            ids = [rng.choice(sorted(model.lens)) for _ in range(rng.randint(1, 4))]
            before = dict(model.lens)
            try:
                model.append(ids)
                ok = True
            except NoSpace:
                ok = False
            if ok:
                slots = bm.append_slots(ids).tolist()
                count = {}
                for s, slot in zip(ids, slots):
                    pos = before[s] + count.get(s, 0)
                    count[s] = count.get(s, 0) + 1
                    slots_seen.setdefault(s, {})[pos] = slot
            else:
                with pytest.raises(B.PkvError) as e:
                    bm.append_slots(ids)
                assert e.value.code == -8
        elif op < 0.9 and model.lens:
            s = rng.choice(sorted(model.lens))
            model.free(s)
            bm.free_sequence(s)
            slots_seen.pop(s, None)
        elif model.lens:
            v = model.preempt_lifo()
            assert bm.preempt_lifo() == v
            slots_seen.pop(v, None)
        check_state(B, bm, model, slots_seen)


def test_fresh_pool_and_errors(B):
    bm = B.BlockManager(4, 16)
    assert bm.num_free_blocks == 4
    bm.add_sequence(1, 17)  # two blocks
    assert bm.num_free_blocks == 2
    t, l = bm.block_tables([1], 4)
    assert t[0, :2].tolist() == [0, 1] and t[0, 2:].tolist() == [-1, -1] and int(l[0]) == 17
    assert bm.append_slots([1]).tolist() == [1 * 16 + 1]   # position 17 lives in block 1
    with pytest.raises(B.PkvError):
        bm.add_sequence(1, 3)                                 # already present
    with pytest.raises(B.PkvError):
        bm.append_slots([7])                                  # unknown sequence
    with pytest.raises(B.PkvError) as e:
        bm.add_sequence(2, 64)                                # 4 blocks, 2 free
    assert e.value.code == -8 and bm.num_free_blocks == 2     # nothing changed
    bm.add_sequence(3, 0)                                     # an empty sequence owns nothing
    assert bm.append_slots([3]).tolist() == [2 * 16]          # its first token takes a block
    assert bm.preempt_lifo() == 3 and bm.num_free_blocks == 2
    bm.free_sequence(1)
    assert bm.num_free_blocks == 4
    with pytest.raises(B.PkvError):
        bm.preempt_lifo()
