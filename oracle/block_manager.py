"""Reference model of the KV block manager -- TEST INFRASTRUCTURE ONLY.

Plain Python following the pages' description:

* "mini-vLLM" LLM-Inference-Engine README, paged KV-cache paragraph and M4 row: a fixed
  pool of physical blocks, each holding block_size token slots; a per-sequence block
  table maps logical positions to physical blocks; under memory pressure the most
  recently admitted sequence is preempted (LIFO).
* "vLLM-Style Llama Inference Engine", How it works: the scheduler allocates blocks,
  finished requests release them.

Which free block is handed out is not fixed by the pages, so the model tracks only what
is: how many blocks each sequence owns (ceil(length / block_size)), how many are free,
whether a request fits, and which sequence LIFO preemption picks.
"""

from __future__ import annotations

import math


class NoSpace(Exception):
    pass


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int):
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.lens: dict[int, int] = {}
        self.admitted: list[int] = []  # admission order, oldest first

    def blocks_of(self, seq_id: int) -> int:
        return math.ceil(self.lens[seq_id] / self.block_size)

    @property
    def num_free(self) -> int:
        return self.num_blocks - sum(self.blocks_of(s) for s in self.lens)

    def add(self, seq_id: int, num_tokens: int) -> None:
        if seq_id in self.lens:
            raise KeyError(seq_id)
        if math.ceil(num_tokens / self.block_size) > self.num_free:
            raise NoSpace()
        self.lens[seq_id] = num_tokens
        self.admitted.append(seq_id)

    def append(self, seq_ids) -> None:
        new = {}
        for s in seq_ids:
            if s not in self.lens:
                raise KeyError(s)
            new[s] = new.get(s, 0) + 1
        need = sum(math.ceil((self.lens[s] + k) / self.block_size) - self.blocks_of(s)
                   for s, k in new.items())
        if need > self.num_free:
            raise NoSpace()
        for s, k in new.items():
            self.lens[s] += k

    def free(self, seq_id: int) -> None:
        del self.lens[seq_id]
        self.admitted.remove(seq_id)

    def preempt_lifo(self) -> int:
        if not self.admitted:
            raise NoSpace()
        victim = self.admitted[-1]
        self.free(victim)
        return victim
