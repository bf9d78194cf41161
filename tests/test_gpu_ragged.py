"""GPU parity of sd_verify_ragged (a draft count per request, packed rows) against the oracle:
every integer output and P/Q bit-exact on fp32 rows (cluster kernel, and the race kernel when
every request samples), the logit tolerances of test_gpu_logits on bf16 rows, requests without
drafts, and counts outside [0, K_max] (clamped, error bit)."""

import numpy as np
import pytest
import torch

import oracle
import verify_draft_prep_gb300 as sd
from devrun import assert_verify_equal, to_dev
from test_gpu_logits import MARGIN, P_TOL, RATE

pytestmark = pytest.mark.gpu


def ragged_case(rng, B, K_max, V, greedy_frac=0.0, zero_frac=0.15):
    ks = rng.integers(1, K_max + 1, B)
    ks[rng.random(B) < zero_frac] = 0
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    n = int(cu[-1])
    lt = 2.0 * rng.standard_normal((n + B, V))
    p = np.exp(lt - lt.max(-1, keepdims=True))
    p = (p / p.sum(-1, keepdims=True)).astype(np.float32)
    q = np.empty((n, V), np.float32)
    d = np.empty(n, np.int32)
    for r in range(B):
        for j in range(int(ks[r])):
            lq = lt[cu[r] + r + j] + 0.6 * rng.standard_normal(V)
            qq = np.exp(lq - lq.max())
            qq /= qq.sum()
            q[cu[r] + j] = qq
            d[cu[r] + j] = rng.choice(V, p=qq)
    T = np.ones(B, np.float32)
    g = rng.random(B) < greedy_frac
    T[g] = 0.0
    for r in np.nonzero(g)[0]:
        for j in range(int(ks[r])):
            d[cu[r] + j] = q[cu[r] + j].argmax() if rng.random() < 0.5 else p[cu[r] + r + j].argmax()
    return p, q, d, cu, T


def run_ragged(target, draft, drafts, cu, K_max, temperature=None, seed=0):
    B = len(cu) - 1
    dev = target.device
    out = dict(out_tokens=torch.full((B, K_max + 1), -7, dtype=torch.int32, device=dev),
               num_accepted=torch.full((B,), -7, dtype=torch.int32, device=dev),
               p_at_draft=torch.full((B, K_max), -7.0, device=dev),
               q_at_draft=torch.full((B, K_max), -7.0, device=dev),
               err=torch.zeros(1, dtype=torch.int32, device=dev))
    sd.sd_verify_ragged(target, draft, drafts, cu, out["out_tokens"], out["num_accepted"],
                        temperature=temperature, seed=seed, p_at_draft=out["p_at_draft"],
                        q_at_draft=out["q_at_draft"], err=out["err"])
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["err"] = int(res["err"][0])
    return res


@pytest.mark.parametrize("B,K_max,V,greedy,temp,seed", [
    (7, 4, 1001, 0.3, True, 1),        # cluster kernel, mixed greedy, ragged tail
    (20, 8, 20011, 0.0, True, 2),
    (200, 6, 20000, 0.0, False, 3),    # every request samples: the race kernel
    (33, 16, 4099, 0.5, True, 4),      # K_max = SD_K_MAX
])
def test_probability_rows_bit_exact(B, K_max, V, greedy, temp, seed):
    rng = np.random.default_rng(700 + seed)
    p, q, d, cu, T = ragged_case(rng, B, K_max, V, greedy_frac=greedy)
    draft = to_dev(q) if q.shape[0] else torch.zeros(0, V).cuda()
    got = run_ragged(to_dev(p), draft, to_dev(d), to_dev(cu), K_max,
                     to_dev(T) if temp else None, seed=seed)
    want = oracle.verify_ragged(p, q, d, cu, K_max, temperature=T if temp else None, seed=seed)
    assert_verify_equal(got, want)


@pytest.mark.parametrize("B,V,seed", [
    (16, 30011, 77),
    (200, 40009, 78),  # enough requests for clusters of 4 CTAs per request
])
def test_logit_rows_within_tolerance(B, V, seed):
    rng = np.random.default_rng(seed)
    K_max = 6
    ks = rng.integers(0, K_max + 1, B)
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    n = int(cu[-1])
    lt = torch.from_numpy(2.0 * rng.standard_normal((n + B, V)).astype(np.float32)).to(
        torch.bfloat16)
    ld = torch.empty(n, V, dtype=torch.bfloat16)
    for r in range(B):
        for j in range(int(ks[r])):
            row = lt[cu[r] + r + j].float() + 0.5 * torch.from_numpy(
                rng.standard_normal(V).astype(np.float32))
            ld[cu[r] + j] = row.to(torch.bfloat16)
    T = torch.from_numpy(rng.uniform(0.5, 1.2, B).astype(np.float32))
    d = torch.empty(n, dtype=torch.int32)
    for r in range(B):
        for j in range(int(ks[r])):
            pr = torch.softmax(ld[cu[r] + j].float() / T[r], -1).numpy().astype(np.float64)
            d[cu[r] + j] = int(rng.choice(V, p=pr / pr.sum()))
    got = run_ragged(lt.cuda(), ld.cuda(), d.cuda(), to_dev(cu), K_max, T.cuda(), seed=9)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    want = oracle.verify_ragged(bits(lt), bits(ld), d.numpy(), cu, K_max, temperature=T.numpy(),
                                seed=9, logits=True)
    diverged = 0
    for i in range(B):
        if got["num_accepted"][i] != want["num_accepted"][i]:
            j = min(got["num_accepted"][i], want["num_accepted"][i])
            assert 0 <= want["accept_margin"][i, j] < MARGIN
            diverged += 1
            continue
        if not np.array_equal(got["out_tokens"][i], want["out_tokens"][i]):
            assert want["race_margin"][i] < MARGIN
            diverged += 1
        ex = min(int(want["num_accepted"][i]), int(ks[i]) - 1) + 1 if ks[i] else 0
        assert np.all(np.abs(got["p_at_draft"][i, :ex] - want["p_at_draft"][i, :ex]) <= P_TOL)
        assert np.all(np.abs(got["q_at_draft"][i, :ex] - want["q_at_draft"][i, :ex]) <= P_TOL)
        assert np.all(got["p_at_draft"][i, ex:] == -1.0)
    assert diverged <= max(1, int(RATE * B * (K_max + 1)))


def test_counts_outside_the_range_are_clamped_and_flagged():
    rng = np.random.default_rng(5)
    B, K_max, V = 3, 2, 500
    p, q, d, cu, _ = ragged_case(rng, B, K_max, V, zero_frac=0.0)
    bad = cu.copy()
    bad[2] = bad[1] + 5          # request 1 claims 5 > K_max drafts, request 2 then a negative count
    # the rows the clamped counts address stay inside these arrays (padded by 16 rows)
    pp = np.concatenate([p, np.zeros((16, V), np.float32)])
    qp = np.concatenate([q, np.zeros((16, V), np.float32)])
    dp = np.concatenate([d, np.zeros(16, np.int32)])
    got = run_ragged(to_dev(pp), to_dev(qp), to_dev(dp), to_dev(bad), K_max, None, seed=1)
    assert got["err"] & sd.SD_ERR_DRAFT_COUNT
    # request 0 is untouched by the bad count
    want = oracle.verify_ragged(p, q, d, cu, K_max, seed=1)
    assert np.array_equal(got["out_tokens"][0], want["out_tokens"][0])
    assert got["num_accepted"][1] <= K_max
