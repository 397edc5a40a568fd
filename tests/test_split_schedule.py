"""Host logic of the split drafter / verifier pipeline, on the CPU.

The two sides are replaced by fakes around a toy target (the next token is
a fixed function of the current token and its position) and a toy drafter
that is right except at every third position.  The pipeline must then give
the target's own greedy tokens (lossless) for any group count, the
drafter's committed lengths must follow the verifier's, and the rows it is
handed for injection must cover every position of every sequence exactly
once, in order.
"""
from types import SimpleNamespace

import numpy as np
import pytest
import torch

from block_diffusion_speculative_injection_gb300.split import Handoff, SplitDFlash

V = 97


def target(tok: int, pos: int) -> int:
    return (tok * 31 + pos * 7 + 3) % V


class FakeVerifier:
    def __init__(self, max_rows):
        self.device = torch.device("cpu")
        self.eng = SimpleNamespace(max_rows=max_rows)
        self.len, self.last = {}, {}

    def reset(self, s):
        self.len[s], self.last[s] = 0, None

    def prefill_chunk(self, sid, toks):
        s, n, p0 = int(sid[0]), toks.numel(), self.len[int(sid[0])]
        self.len[s] += n
        self.last[s] = int(toks[-1])
        anchor = target(self.last[s], self.len[s] - 1)
        h = Handoff(torch.zeros(n, 1, 1), torch.full((n,), s, dtype=torch.int32),
                    torch.arange(p0, p0 + n, dtype=torch.int32), torch.tensor([n], dtype=torch.int32))
        return torch.tensor([anchor], dtype=torch.int32), h

    def verify_block(self, sid, block):
        b, B = block.shape
        acc, nxt = torch.empty(b, dtype=torch.int32), torch.empty(b, dtype=torch.int32)
        emitted = torch.full((b, B), -1, dtype=torch.int32)
        argmax = torch.empty(b, B, dtype=torch.int32)
        rs, rp = [], []
        for k in range(b):
            s, P = int(sid[k]), self.len[int(sid[k])]
            am = [target(int(block[k, j]), P + j) for j in range(B)]
            argmax[k] = torch.tensor(am)
            a = 0
            while a < B - 1 and int(block[k, a + 1]) == am[a]:
                a += 1
            emitted[k, :a] = block[k, 1:a + 1]
            emitted[k, a] = am[a]
            acc[k], nxt[k] = a, am[a]
            self.len[s] += a + 1
            rs += [s if j <= a else -1 for j in range(B)]
            rp += [P + j for j in range(B)]
        h = Handoff(torch.zeros(b * B, 1, 1), torch.tensor(rs, dtype=torch.int32),
                    torch.tensor(rp, dtype=torch.int32), acc + 1)
        return acc, nxt, emitted, argmax, h


class FakeDrafter:
    def __init__(self, B):
        self.device = torch.device("cpu")
        self.B = B
        self.len, self.injected = {}, {}

    def reset(self, s):
        self.len[s], self.injected[s] = 0, []

    def absorb(self, sid, h):
        for r in range(h.row_seq.numel()):
            s = int(h.row_seq[r])
            if s >= 0:
                self.injected[s].append(int(h.row_pos[r]))
        for k in range(sid.numel()):
            self.len[int(sid[k])] += int(h.counts[k])

    def draft(self, sid, anchors):
        b = sid.numel()
        block = torch.empty(b, self.B, dtype=torch.int32)
        for k in range(b):
            P = self.len[int(sid[k])]
            block[k, 0] = int(anchors[k])
            for j in range(1, self.B):
                t = target(int(block[k, j - 1]), P + j - 1)
                block[k, j] = t if (P + j) % 3 else (t + 1) % V
        return block


def ar_tokens(prompt, n):
    toks, pos = [int(prompt[-1])], len(prompt) - 1
    out = []
    for _ in range(n):
        t = target(toks[-1], pos)
        out.append(t)
        toks.append(t)
        pos += 1
    return out


def make(B, max_rows):
    sp = SplitDFlash.__new__(SplitDFlash)
    sp.B = B
    sp.verifier, sp.drafter = FakeVerifier(max_rows), FakeDrafter(B)
    sp.vdev = sp.ddev = torch.device("cpu")
    return sp


@pytest.mark.parametrize("groups", [1, 2, 3])
def test_pipeline_is_lossless_and_keeps_both_sides_in_step(groups):
    rng = np.random.default_rng(3)
    prompts = [rng.integers(0, V, size=n).astype(np.int32) for n in (40, 7, 25, 61, 12)]
    sp = make(B=8, max_rows=16)  # prompts longer than 16 rows go in chunks
    n = 30
    out = sp.generate(prompts, n, groups=groups)
    assert out == [ar_tokens(p, n) for p in prompts]
    for s, p in enumerate(prompts):
        L = sp.verifier.len[s]
        assert sp.drafter.len[s] == L
        assert sp.drafter.injected[s] == list(range(L))  # every position once, in order
        assert L >= len(p) + n - 1  # the newest token is the next anchor, not yet committed
