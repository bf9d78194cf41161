"""Expected tokens per round (speculative-decoding explainer, section "一轮能赚多少：接受率的算术").

q is uniform on tokens 0-3 and p = beta*q + (1-beta)*uniform on tokens 4-7, so that
sum min(p, q) = beta for every row. With gamma = K drafts the mean of a+1 must match
(1 - beta^(gamma+1)) / (1 - beta), whose two-decimal values are printed on the page; a is
geometric truncated at gamma, and every resample lands uniformly on 4-7.
"""

import math

import numpy as np
import pytest
from scipy import stats

import oracle
from conftest import read_table

N = 1_000_000
TABLE = [(float(b), int(g), float(v)) for b, g, v in read_table("expected_tokens_table.txt")]


def closed_form(beta, gamma):
    return (1 - beta ** (gamma + 1)) / (1 - beta)


@pytest.mark.parametrize("beta,gamma,printed", TABLE)
def test_expected_tokens(beta, gamma, printed):
    assert round(closed_form(beta, gamma), 2) == printed
    V = 8
    q = np.array([0.25] * 4 + [0.0] * 4, np.float32)
    p = np.array([beta * 0.25] * 4 + [(1 - beta) * 0.25] * 4, np.float32)
    rng = np.random.default_rng(int(beta * 100) + gamma)
    drafts = rng.integers(0, 4, size=(N, gamma), dtype=np.int32)
    # every row of every request is the same (p, q): row stride 0
    res = oracle.verify_probs_strided(N, gamma, V, p, 0, q, 0, drafts, seed=gamma)
    a = res["num_accepted"].astype(np.int64)
    tokens = a + 1
    mean = tokens.mean()
    se = tokens.std() / math.sqrt(N)
    assert abs(mean - closed_form(beta, gamma)) < 4 * se, (mean, closed_form(beta, gamma), se)
    # law of a: P(a = j) = beta^j (1 - beta) for j < gamma, beta^gamma for j = gamma
    law = np.array([beta ** j * (1 - beta) for j in range(gamma)] + [beta ** gamma])
    counts = np.bincount(a, minlength=gamma + 1)
    stat = ((counts - N * law) ** 2 / (N * law)).sum()
    assert stat < stats.chi2.ppf(1 - 1e-3, gamma), stat
    # resampled tokens are uniform on 4..7
    toks = res["out_tokens"]
    rej = a < gamma
    b = toks[np.nonzero(rej)[0], a[rej]]
    assert np.all((b >= 4) & (b <= 7))
    cb = np.bincount(b - 4, minlength=4)
    stat_b = ((cb - cb.sum() / 4) ** 2 / (cb.sum() / 4)).sum()
    assert stat_b < stats.chi2.ppf(1 - 1e-3, 3), stat_b
    # accepted tokens are the drafts themselves
    for j in range(gamma):
        sel = a > j
        assert np.array_equal(toks[sel, j], drafts[sel, j])
