"""Pins of the oracle's drafter-side sampling (reading R13: the drafter's K output rows per request
are sampled by the exponential race with the Philox tag-2 stream; temperature 0 takes the argmax).

What the mathematics fixes: the race argmax_x q(x)/E_x with E_x ~ Exp(1) independent draws x
with probability q(x) / sum q (exponential-race / Gumbel-max identity), so over many requests the
drafts follow q (fp32 rows) or softmax(l / T) (logit rows): chi-square at alpha = 1e-3 against
those laws. A missing temperature, a softmax on the wrong scale, a race on 1 - q, a key with E in
the numerator or a stream shared across the K rows each fail one of the tests below.
"""

import numpy as np
from scipy import stats

import oracle

ALPHA = 1e-3
Q0 = np.array([0.30, 0.05, 0.15, 0.02, 0.20, 0.08, 0.12, 0.08], np.float32)
Q1 = np.array([0.05, 0.05, 0.40, 0.10, 0.10, 0.05, 0.05, 0.20], np.float32)
L0 = np.array([1.5, -0.5, 0.25, 2.0, -1.0, 0.0, 0.75, -2.0], np.float32)


def _chi2_ok(counts, prob):
    n = counts.sum()
    e = prob.astype(np.float64) / prob.astype(np.float64).sum() * n
    stat = ((counts - e) ** 2 / e).sum()
    return stat < stats.chi2.ppf(1 - ALPHA, len(counts) - 1), stat


def _bf16_bits(x):
    b = np.asarray(x, np.float32).view(np.uint32)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def test_fp32_rows_follow_q_per_row():
    N = 200_000
    q = np.ascontiguousarray(np.broadcast_to(np.stack([Q0, Q1]), (N, 2, 8)))
    res = oracle.draft_sample_probs(q, seed=21)
    assert res["err"] == 0
    for k, qk in enumerate((Q0, Q1)):
        ok, stat = _chi2_ok(np.bincount(res["drafts"][:, k], minlength=8), qk)
        assert ok, (k, stat)
    # the two rows of a request draw from different counters: their draws are independent
    joint = np.bincount(res["drafts"][:, 0] * 8 + res["drafts"][:, 1], minlength=64)
    ok, stat = _chi2_ok(joint, np.outer(Q0, Q1).ravel())
    assert ok, stat


def test_logit_rows_follow_softmax_at_temperature():
    N = 200_000
    for T in (0.6, 1.3):
        lb = np.ascontiguousarray(np.broadcast_to(_bf16_bits(L0), (N, 1, 8)))
        temp = np.full(N, T, np.float32)
        res = oracle.draft_sample_logits(lb, temperature=temp, seed=33)
        lv = lb[0, 0].astype(np.uint32) << 16
        law = np.exp(lv.view(np.float32).astype(np.float64) / T)
        ok, stat = _chi2_ok(np.bincount(res["drafts"][:, 0], minlength=8), law / law.sum())
        assert ok, (T, stat)


def test_temperature_zero_takes_the_argmax_lowest_index_on_ties():
    q = np.array([[[0.1, 0.3, 0.3, 0.2, 0.1]]], np.float32)
    res = oracle.draft_sample_probs(q, temperature=np.zeros(1, np.float32), seed=5)
    assert res["drafts"][0, 0] == 1
    lb = _bf16_bits(np.array([[[0.5, 2.0, -1.0, 2.0]]], np.float32))
    res = oracle.draft_sample_logits(lb, temperature=np.zeros(1, np.float32), seed=5)
    assert res["drafts"][0, 0] == 1


def test_zero_row_gives_token_zero_and_the_error_bit():
    q = np.zeros((2, 1, 6), np.float32)
    q[1, 0, 4] = 1.0
    res = oracle.draft_sample_probs(q, seed=9)
    assert res["drafts"][0, 0] == 0 and res["drafts"][1, 0] == 4
    assert res["err"] & oracle.ERR_ZERO_ROW


def test_stream_differs_from_the_verify_race():
    # the same row raced in the verify stream (tag 1) and in the drafter stream (tag 2): the two
    # winners agree only as often as two independent draws from q do (sum q^2), not always
    n = 4000
    agree = 0
    for r in range(n):
        q = Q0.copy()
        verify_winner = oracle.race_row(q, None, seed=17, r=r, j=0)[0]
        sample = oracle.draft_sample_probs(q[None, None, :], seed=17, req_ids=np.array([r]))
        agree += int(sample["drafts"][0, 0] == verify_winner)
    p_agree = float((Q0.astype(np.float64) ** 2).sum())
    assert abs(agree / n - p_agree) < 5 * np.sqrt(p_agree * (1 - p_agree) / n)
    assert oracle.race_E(17, 3, 1, 6, tag=2) != oracle.race_E(17, 3, 1, 6)


def test_request_ids_reproduce_the_batch():
    rng = np.random.default_rng(6)
    q = rng.random((12, 3, 50)).astype(np.float32)
    full = oracle.draft_sample_probs(q, seed=8)
    part = oracle.draft_sample_probs(q[5:9], seed=8, req_ids=np.arange(5, 9))
    assert np.array_equal(part["drafts"], full["drafts"][5:9])
