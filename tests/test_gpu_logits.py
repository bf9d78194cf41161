"""GPU parity of sd_verify on bf16 logit rows (fused temperature softmax) against the oracle's
double-precision evaluation.

Tolerances: p/q at the drafts within 2e-6 absolute of the double values; a token or accept
decision may differ from the oracle only where the oracle's own decision margin is below 1e-5
(accept: |P - uQ| / max(P, uQ); race: (k1 - k2) / k1 of its top two keys), each such divergence
counted, and the count under 1e-4 of the B*(K+1) verify positions. Greedy requests (T = 0) work
on the raw logits and must match exactly.
"""

import numpy as np
import pytest
import torch

import verify_draft_prep_gb300 as sd  # noqa: F401
from devrun import oracle_verify_rows, run_verify

pytestmark = pytest.mark.gpu

P_TOL = 2e-6
MARGIN = 1e-5
RATE = 1e-4


def compare_logits(got, want, K, req_ids=None):
    """Returns the number of tolerated divergences; raises on any other difference."""
    sel = slice(None) if req_ids is None else np.asarray(req_ids)
    ga, wa = got["num_accepted"][sel], want["num_accepted"]
    gt, wt = got["out_tokens"][sel], want["out_tokens"]
    gp, gq = got["p_at_draft"][sel], got["q_at_draft"][sel]
    wp, wq = want["p_at_draft"], want["q_at_draft"]
    diverged = 0
    for i in range(len(wa)):
        a_g, a_w = int(ga[i]), int(wa[i])
        if a_g != a_w:
            j = min(a_g, a_w)  # the first accept decision that differs
            m = want["accept_margin"][i, j]
            assert 0 <= m < MARGIN, (i, a_g, a_w, m)
            diverged += 1
            continue
        if not np.array_equal(gt[i], wt[i]):
            assert want["race_margin"][i] < MARGIN, (i, gt[i], wt[i], want["race_margin"][i])
            diverged += 1
        ex = min(a_w, K - 1) + 1  # examined drafts
        assert np.all(np.abs(gp[i, :ex] - wp[i, :ex]) <= P_TOL), (i, gp[i, :ex], wp[i, :ex])
        assert np.all(np.abs(gq[i, :ex] - wq[i, :ex]) <= P_TOL), (i, gq[i, :ex], wq[i, :ex])
        assert np.all(gp[i, ex:] == -1.0) and np.all(wp[i, ex:] == -1.0)
    return diverged


def logit_case(rng, B, K, V, sigma=0.5, tlo=0.5, thi=1.2, greedy_frac=0.0):
    lt = torch.from_numpy(2.0 * rng.standard_normal((B * (K + 1), V)).astype(np.float32))
    lt = lt.to(torch.bfloat16)
    ld = (lt.view(B, K + 1, V)[:, :K].float()
          + sigma * torch.from_numpy(rng.standard_normal((B, K, V)).astype(np.float32)))
    ld = ld.to(torch.bfloat16).view(B * K, V)
    T = torch.from_numpy(rng.uniform(tlo, thi, B).astype(np.float32))
    g = torch.from_numpy(rng.random(B) < greedy_frac)
    T[g] = 0.0
    q = torch.softmax(ld.float().view(B, K, V) / torch.where(T > 0, T, 1.0).view(B, 1, 1), -1)
    d = torch.multinomial(q.view(B * K, V), 1,
                          generator=torch.Generator().manual_seed(int(rng.integers(1 << 30))))
    d = d.view(B, K).to(torch.int32)
    am = lt.view(B, K + 1, V).float().argmax(-1)
    for b in torch.nonzero(g).flatten().tolist():
        m = int(rng.integers(0, K + 1))
        d[b, :m] = am[b, :m].to(torch.int32)
    return lt, ld, d, T


@pytest.mark.parametrize("B,K,V,greedy,seed", [
    (8, 4, 1024, 0.0, 0),
    (24, 5, 50001, 0.25, 1),
    (12, 8, 201088, 0.2, 2),
    (40, 3, 777, 0.5, 3),
    (200, 3, 50001, 0.2, 4),  # enough requests for clusters of 4 CTAs (B * 4 CTAs fill a wave)
    (192, 16, 40009, 0.1, 5),  # K = SD_K_MAX with clusters of 4
])
def test_logits_within_tolerance(B, K, V, greedy, seed):
    rng = np.random.default_rng(200 + seed)
    lt, ld, d, T = logit_case(rng, B, K, V, greedy_frac=greedy)
    got = run_verify(lt.cuda(), ld.cuda(), d.cuda(), T.cuda(), seed=seed)
    want = oracle_verify_rows(lt, ld, d, T, seed=seed)
    div = compare_logits(got, want, K)
    assert div <= RATE * B * (K + 1)
    assert got["err"] == want["err"]
    # greedy requests are exact
    g = (T == 0).numpy()
    assert np.array_equal(got["out_tokens"][g], want["out_tokens"][g])
    assert np.array_equal(got["p_at_draft"][g], want["p_at_draft"][g])
