"""Pins of the temperature-1 acceptance oracle (oracle/sampling.py).

* the draw: inverse CDF equals numpy's searchsorted over the cumulative sum;
* the rule as a whole is lossless: integrating the oracle over grids of its
  uniforms gives, for the token at the first drafted position, exactly the
  target distribution q_0 (and q_1 for the bonus after an acceptance) --
  the property the reading was chosen for, which a wrong inequality, a
  missing residual or a residual of the wrong sign fails;
* limiting cases: identical draft and target distributions accept every
  token; a draft token the target gives zero mass is always rejected and the
  residual is the target distribution itself;
* hand-derived cases in tests/golden/sampling_cases.txt.
"""
import os

import numpy as np
import pytest

from oracle.sampling import draft_tokens, inverse_cdf, sample_row, softmax, spec_accept

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sampling_cases.txt")


def test_inverse_cdf_matches_searchsorted():
    rng = np.random.default_rng(11)
    for _ in range(200):
        w = rng.random(rng.integers(1, 40)) * (rng.random() < 0.5 or 1.0)
        w[rng.random(w.shape) < 0.3] = 0.0
        if w.sum() == 0:
            w[0] = 1.0
        u = rng.random()
        ref = int(np.searchsorted(np.cumsum(w), u * w.sum(), side="right"))
        assert inverse_cdf(w, u) == ref


def test_sample_row_is_softmax_draw():
    x = np.log(np.array([0.1, 0.2, 0.3, 0.4]))
    assert [sample_row(x, u) for u in (0.05, 0.15, 0.35, 0.65, 0.95)] == [0, 1, 2, 3, 3]


def _grid(n):
    return (np.arange(n) + 0.5) / n


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_rule_is_lossless(seed):
    rng = np.random.default_rng(seed)
    V, N = 5, 4000
    dl = rng.normal(0, 1.5, (2, V))
    tl = rng.normal(0, 1.5, (2, V))
    p, q = softmax(dl), softmax(tl)
    first = np.zeros(V)  # distribution of the token at block position 1
    acc_mass = 0.0
    for d in range(V):
        toks = [0, d]
        # accept test integrated over u_accept; the draw after a rejection
        # depends on u_resample alone, so it is integrated on its own
        acc = np.mean([spec_accept(dl, tl, toks, [0.0, u], 0.5)[0] == 1 for u in _grid(N)])
        first[d] += p[1, d] * acc
        acc_mass += p[1, d] * acc
        if acc < 1.0:
            for ur in _grid(N):
                a, em = spec_accept(dl, tl, toks, [0.0, 1.0 - 1e-12], ur)
                assert a == 0
                first[em] += p[1, d] * (1.0 - acc) / N
    second = np.zeros(V)  # the bonus after d_1 is accepted: q_1
    for ur in _grid(N):
        second[spec_accept(dl, tl, [0, int(np.argmax(q[0] / p[1]))], [0.0, 0.0], ur)[1]] += 1.0 / N
    assert np.abs(first - q[0]).max() < 2e-3
    assert np.abs(second - q[1]).max() < 2e-3
    # acceptance probability = sum_x min(p, q)
    assert abs(acc_mass - np.minimum(p[1], q[0]).sum()) < 2e-3


def test_identical_distributions_accept_everything():
    rng = np.random.default_rng(5)
    B, V = 6, 9
    logits = rng.normal(0, 2, (B, V))
    tl = np.vstack([logits[1:], rng.normal(0, 2, (1, V))])  # q_{j-1} = p_j
    for trial in range(50):
        u = rng.random(B)
        toks = np.concatenate([[0], draft_tokens(logits, rng.random(B))[1:]])
        a, _ = spec_accept(logits, tl, toks, u, rng.random())
        assert a == B - 1


def test_zero_target_mass_rejects_and_resamples_target():
    V = 6
    z = -np.inf
    dl = np.array([[0, 0, 0, 0, 0, 0], [np.log(0.5), np.log(0.5), z, z, z, z]])
    tl = np.array([[z, z, np.log(0.25), np.log(0.25), np.log(0.25), np.log(0.25)], [0, 0, 0, 0, 0, 0]])
    for u in (0.0, 0.5, 0.999):
        for ur, want in ((0.1, 2), (0.3, 3), (0.6, 4), (0.9, 5)):
            a, em = spec_accept(dl, tl, [0, 1], [0.0, u], ur)
            assert (a, em) == (0, want)


def _parse_rows(field):
    return np.array([[float(x) for x in r.split()] for r in field.split(";")])


def test_golden_cases():
    n = 0
    with open(GOLDEN) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            cols = [c.strip() for c in line.split("|")]
            p = _parse_rows(cols[0])
            q = _parse_rows(cols[1])
            d = [int(x) for x in cols[2].split()]
            u = [float(x) for x in cols[3].split()]
            ures, a_want, em_want = float(cols[4]), int(cols[5]), int(cols[6])
            B = q.shape[0]
            dl = np.vstack([np.zeros((1, p.shape[1])), np.log(p)])
            a, em = spec_accept(dl, np.log(q), [0] + d, [0.0] + u, ures)
            assert (a, em) == (a_want, em_want), line
            assert dl.shape[0] == B
            n += 1
    assert n == 7
