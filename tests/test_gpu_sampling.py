"""Temperature-1 drafting and acceptance through the C ABI against the oracle.

dflash_sample_rows draws the draft tokens of every block slot; the draws are
compared with oracle.sampling.sample_row.  dflash_spec_accept_sampled is then
fed the oracle's draft tokens (so one near-tie draw cannot change the rest)
and its accept length and emitted token are compared with
oracle.sampling.spec_accept.

Both sides take the same decisions from the same fp32 logits and uniforms;
the GPU sums in fp32 and the oracle in fp64, so a decision that lies within
fp32 rounding of a tie may go either way.  Such positions are exempt from
equality (relative band 1e-5), and the GPU's choice must still be valid: an
exempt accept test may pass or fail; an exempt draw must name a token whose
cumulative-weight interval lies within the band of the oracle's target.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from oracle.sampling import sample_row, softmax, spec_accept

pytestmark = pytest.mark.gpu

BAND = 1e-5


def _draw_ok(w, u, got, want):
    """got is the oracle's token, or a neighbour within the rounding band."""
    if got == want:
        return True
    if not 0 <= got < len(w):
        return False
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    t = float(u) * c[-1]
    lo = c[got - 1] if got > 0 else 0.0
    return w[got] > 0 and lo - BAND * c[-1] <= t <= c[got] + BAND * c[-1]


def _gpu_sample(logits2d, u):
    from block_diffusion_speculative_injection_gb300 import capi
    rows, V = logits2d.shape
    x = torch.from_numpy(np.ascontiguousarray(logits2d)).cuda()
    uu = torch.from_numpy(np.ascontiguousarray(u, dtype=np.float32)).cuda()
    out = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(capi.dflash_sample_workspace(rows, V), dtype=torch.uint8, device="cuda")
    capi.dflash_sample_rows(rows, V, x, uu, out, ws)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("rows,V", [(1, 1), (7, 1000), (40, 4096), (33, 4097), (64, 151936)])
def test_sample_rows_matches_oracle(rows, V):
    d, _, u, _, _ = wl.sampling_inputs(1, rows, V)
    logits = d[0]
    got = _gpu_sample(logits, u[0])
    for r in range(rows):
        want = sample_row(logits[r], float(u[0, r]))
        assert _draw_ok(softmax(logits[r]), u[0, r], int(got[r]), want), (r, got[r], want)


def test_sample_rows_masked_and_peaked():
    V = 5000
    logits = np.full((3, V), -np.inf, dtype=np.float32)
    logits[0, 4321] = 0.0                         # one token with all the mass
    logits[1, [7, 4099]] = 0.0                    # two tokens, in different chunks
    logits[2] = np.linspace(-30, 30, V, dtype=np.float32)  # mass piled at the end
    got = _gpu_sample(logits, np.array([0.999, 0.75, 0.0], dtype=np.float32))
    assert got[0] == 4321 and got[1] == 4099
    w = softmax(logits[2])
    assert _draw_ok(w, 0.0, int(got[2]), int(np.searchsorted(np.cumsum(w), 0.0, side="right")))


def _run_accept(batch, block, V, agreement):
    from block_diffusion_speculative_injection_gb300 import capi
    dl, tl, ud, ua, ur = wl.sampling_inputs(batch, block, V, agreement=agreement)
    # the oracle's draft tokens d_j ~ p_j
    tokens = np.zeros((batch, block), dtype=np.int32)
    for b in range(batch):
        for j in range(1, block):
            tokens[b, j] = sample_row(dl[b, j], float(ud[b, j]))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    acc = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    em = torch.full((batch,), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(capi.dflash_spec_accept_workspace(batch, block, V), dtype=torch.uint8,
                     device="cuda")
    capi.dflash_spec_accept_sampled(batch, block, V, t(dl[:, 1:]), t(tl), t(tokens), t(ua), t(ur), acc, em, ws)
    torch.cuda.synchronize()
    return dl, tl, tokens, ua, ur, acc.cpu().numpy(), em.cpu().numpy()


def _check_accept(dl, tl, tokens, ua, ur, acc, em):
    batch, block, V = tl.shape
    n_exact = 0
    for b in range(batch):
        a_want, em_want = spec_accept(dl[b], tl[b], tokens[b], ua[b], float(ur[b]))
        p, q = softmax(dl[b]), softmax(tl[b])
        # accept tests near a tie are exempt: the GPU's length must still be a
        # length the rule allows with each exempt test taken either way
        tests = []
        for j in range(1, block):
            d = tokens[b, j]
            lhs, rhs = float(ua[b, j]) * p[j, d], q[j - 1, d]
            tests.append((lhs < rhs, abs(lhs - rhs) <= BAND * max(lhs, rhs)))
        a = int(acc[b])
        assert 0 <= a <= block - 1
        assert all(ok or tie for ok, tie in tests[:a]), (b, a, a_want)
        if a < block - 1:
            ok, tie = tests[a]
            assert (not ok) or tie, (b, a, a_want)
        if a == a_want:
            w = np.maximum(q[a] - p[a + 1], 0.0) if a < block - 1 else q[block - 1]
            if w.sum() == 0:
                w = q[a]
            assert _draw_ok(w, ur[b], int(em[b]), em_want), (b, int(em[b]), em_want)
            n_exact += 1
    return n_exact


@pytest.mark.parametrize("batch,block,V,agreement", [
    (1, 16, 1000, 0.9), (8, 16, 1000, 0.99), (32, 16, 4097, 0.95), (4, 16, 151936, 0.95),
    (3, 1, 2000, 0.9), (5, 4, 151936, 0.999)])
def test_spec_accept_matches_oracle(batch, block, V, agreement):
    res = _run_accept(batch, block, V, agreement)
    n_exact = _check_accept(*res)
    assert n_exact >= batch - 1  # all but a rare tie agree on the accept length
    acc = res[5]
    if agreement >= 0.99 and block > 1:
        assert acc.max() >= 1  # the agreeing cases do accept draft tokens


def test_spec_accept_identical_distributions_accept_all():
    from block_diffusion_speculative_injection_gb300 import capi
    batch, block, V = 6, 16, 3000
    dl, _, ud, ua, ur = wl.sampling_inputs(batch, block, V)
    tl = np.concatenate([dl[:, 1:], dl[:, :1]], axis=1)  # q_{j-1} = p_j exactly
    tokens = np.zeros((batch, block), dtype=np.int32)
    for b in range(batch):
        for j in range(1, block):
            tokens[b, j] = sample_row(dl[b, j], float(ud[b, j]))
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    acc = torch.zeros(batch, dtype=torch.int32, device="cuda")
    em = torch.zeros(batch, dtype=torch.int32, device="cuda")
    ws = torch.empty(capi.dflash_spec_accept_workspace(batch, block, V), dtype=torch.uint8, device="cuda")
    capi.dflash_spec_accept_sampled(batch, block, V, t(dl[:, 1:]), t(tl), t(tokens), t(ua), t(ur), acc, em, ws)
    torch.cuda.synchronize()
    assert (acc.cpu().numpy() == block - 1).all()


def test_invalid_arguments_are_refused():
    from block_diffusion_speculative_injection_gb300 import capi
    assert capi.dflash_sample_workspace(0, 10) == -1
    assert capi.dflash_spec_accept_workspace(1, 33, 10) == -1
    assert capi.dflash_spec_accept_workspace(1, 16, 600000) == -1
    x = torch.zeros(2, 10, device="cuda")
    u = torch.zeros(2, device="cuda")
    out = torch.zeros(2, dtype=torch.int32, device="cuda")
    small = torch.empty(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(capi.DFlashError) as e:
        capi.dflash_sample_rows(2, 10, x, u, out, small)
    assert e.value.status == 1
