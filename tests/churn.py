"""Dynamic request traffic for the churn tests: requests arrive (Poisson),
are admitted into free slots when the pool can hold their prompt and their
growth, generate a drawn number of tokens (one generation step and one
attention call with score update per tick) and are freed when done, so that
the free list's start and end counters wrap the pool many times (DiffKV,
Memory management: circular free page list; Evaluation: dynamic workloads).

The generator holds no compaction arithmetic: it only decides which
operations run, from the pool's free-page count."""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class Churn:
    seed: int
    max_requests: int
    n_kv_heads: int
    t_hi: int
    slack: int = 1
    tiers: int = 2                                 # precision tiers of the pool (3 with mid)
    prompt_lens: tuple = (100, 700)
    gen_lens: tuple = (5, 40)
    rate: float = 0.35
    queue: list = field(default_factory=list)
    active: dict = field(default_factory=dict)     # slot -> [generated, target, prompt length]
    n_arrived: int = 0

    def __post_init__(self):
        self.rng = np.random.default_rng([self.seed, 0xC4E2])

    def _growth_pages(self, gen: int) -> int:
        # pages a request may still take while it generates `gen` tokens:
        # a new page per tier at most every t_hi tokens, plus one each
        return self.tiers * self.n_kv_heads * (gen // self.t_hi + 2)

    def tick(self, free_pages: int) -> list:
        """Operations of one tick, in order: ("prompt", slot, n0, seed),
        ("decode", slots), ("attend", slots), ("free", slot)."""
        ops = []
        for _ in range(int(self.rng.poisson(self.rate))):
            n0 = int(self.rng.integers(self.prompt_lens[0], self.prompt_lens[1] + 1))
            gen = int(self.rng.integers(self.gen_lens[0], self.gen_lens[1] + 1))
            self.queue.append((n0, gen))
        budget = free_pages - sum(self._growth_pages(t - g) for g, t, _ in self.active.values())
        while self.queue:
            free_slots = [s for s in range(self.max_requests) if s not in self.active]
            n0, gen = self.queue[0]
            grant = self.n_kv_heads * (-(-n0 // self.t_hi) + self.slack)
            if not free_slots or budget < grant + self._growth_pages(gen):
                break
            self.queue.pop(0)
            slot = int(self.rng.choice(free_slots))
            budget -= grant + self._growth_pages(gen)
            self.active[slot] = [0, gen, n0]
            ops.append(("prompt", slot, n0, self.seed * 100003 + self.n_arrived))
            self.n_arrived += 1
        if self.active:
            slots = sorted(self.active)
            ops.append(("decode", slots))
            ops.append(("attend", slots))
            for s in slots:
                self.active[s][0] += 1
        for s in sorted(self.active):
            g, t, _ = self.active[s]
            if g >= t:
                ops.append(("free", s))
                del self.active[s]
        return ops
