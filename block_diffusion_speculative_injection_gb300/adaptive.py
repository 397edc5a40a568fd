"""Block size per step from the recent acceptance lengths.

The pages train the drafter with a large block that carries over to smaller
inference blocks (Deep Research Report, "Key points": training innovations)
and list adaptive block sizes as a future direction ("Discussion and open
problems"), without a rule.  This policy takes the plainest one: a block of
B slots can accept at most B - 1 draft tokens, so size the next block to the
recent acceptance plus the anchor plus a little slack,

    ema <- decay * ema + (1 - decay) * mean(accepted lengths of the step)
    B   =  clamp(ceil(ema) + 1 + slack, b_min, b_max)

starting from ema = b_max - 1 (the configured block).  When a block is
accepted whole, ema reaches B - 1 and the next block grows by `slack`.

At one sequence the target pass streams weights and costs the same at any B,
so a smaller block saves nothing there; the saving is in verify rows
(batch x B) once the pass is compute-bound at larger batches.  Greedy
decoding emits the same tokens whatever B is (the method is lossless), which
is what the GPU tests check.
"""
from __future__ import annotations

import math
from typing import Sequence


class AdaptiveBlock:
    def __init__(self, b_max: int, b_min: int = 2, decay: float = 0.5, slack: int = 2):
        if not 1 <= b_min <= b_max:
            raise ValueError("need 1 <= b_min <= b_max")
        if not 0.0 <= decay < 1.0:
            raise ValueError("decay must be in [0, 1)")
        if slack < 0:
            raise ValueError("slack must be >= 0")
        self.b_max, self.b_min, self.decay, self.slack = b_max, b_min, decay, slack
        self.ema = float(b_max - 1)

    def next_block(self) -> int:
        b = math.ceil(self.ema - 1e-9) + 1 + self.slack
        return int(min(self.b_max, max(self.b_min, b)))

    def update(self, accepted: Sequence[int]) -> None:
        """accepted: the accepted draft-token counts of the step's sequences."""
        if len(accepted) == 0:
            return
        mean = sum(int(a) for a in accepted) / len(accepted)
        self.ema = self.decay * self.ema + (1.0 - self.decay) * mean
