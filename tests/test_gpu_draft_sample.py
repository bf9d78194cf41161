"""GPU parity of sd_draft_sample (drafter-side sampling of the next drafts, tag-2 Philox stream)
against the oracle.

fp32 probability rows: every draft and the error bits bit-exact (the keys are the same fp32
divisions on both sides). bf16 logit rows: the kernel's softmax is fp32 with hardware
exponentials, the oracle's double, so a draft may differ only where the oracle's own race margin
(k1 - k2) / k1 is below 1e-5, each such divergence counted and the count under 1e-4 of the rows
(at least one allowed); temperature-0 rows work on the raw logits and must match exactly.
"""

import numpy as np
import pytest
import torch

import oracle
import verify_draft_prep_gb300 as sd
import workloads
from devrun import random_probs_case, to_dev

pytestmark = pytest.mark.gpu

MARGIN = 1e-5
RATE = 1e-4


def run_sample(rows, B, K, temperature=None, seed=0, request_base=0):
    dev = rows.device
    drafts = torch.full((B, K), -7, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sd.sd_draft_sample(rows, drafts, temperature=temperature, seed=seed,
                       request_base=request_base, err=err)
    torch.cuda.synchronize()
    return drafts.cpu().numpy(), int(err.item())


def oracle_probs(rows, B, K, temperature=None, seed=0, req_ids=None):
    V = rows.shape[1]
    q = rows.float().cpu().numpy().reshape(B, K, V)
    T = None if temperature is None else temperature.cpu().numpy()
    return oracle.draft_sample_probs(q, temperature=T, seed=seed, req_ids=req_ids)


def oracle_logits(rows, B, K, temperature=None, seed=0):
    V = rows.shape[1]
    bits = rows.cpu().contiguous().view(torch.int16).numpy().view(np.uint16).reshape(B, K, V)
    T = None if temperature is None else temperature.cpu().numpy()
    return oracle.draft_sample_logits(bits, temperature=T, seed=seed)


@pytest.mark.parametrize("B,K,V,greedy,seed", [
    (1, 4, 1024, 0.0, 0),
    (7, 3, 1001, 0.3, 1),          # ragged tail
    (16, 5, 4099, 0.5, 2),
    (9, 16, 70001, 0.4, 3),        # K = SD_K_MAX, cluster of 8, ragged
    (33, 2, 20000, 0.25, 4),
    (64, 1, 8, 0.2, 5),            # tiny vocabulary
    (5, 2, 1, 0.4, 6),             # V = 1
])
def test_probability_rows_bit_exact(B, K, V, greedy, seed):
    rng = np.random.default_rng(500 + seed)
    _, q, _, T = random_probs_case(rng, B, K, V, sigma=0.7, greedy_frac=greedy)
    rows, temp = to_dev(q), to_dev(T)
    got, gerr = run_sample(rows, B, K, temp, seed=seed * 31 + 7)
    want = oracle_probs(rows, B, K, temp, seed=seed * 31 + 7)
    assert np.array_equal(got, want["drafts"])
    assert gerr == want["err"]


def test_unaligned_rows_zero_rows_and_no_temperature():
    rng = np.random.default_rng(17)
    B, K, V, ld = 6, 3, 5003, 5005
    _, q, _, _ = random_probs_case(rng, B, K, V)
    q3 = q.reshape(B, K, V)
    q3[1, 2] = 0.0                    # no positive entry: draft 0 and the error bit
    q3[2, 0, :] = 0.0
    q3[2, 0, 4321] = 1.0              # one-hot row
    buf = torch.zeros(B * K, ld)
    buf[:, 1:V + 1] = torch.from_numpy(q3.reshape(B * K, V))
    rows = buf.cuda()[:, 1:V + 1]     # row starts not 16-byte aligned: scalar loads
    got, gerr = run_sample(rows, B, K, None, seed=3)
    want = oracle_probs(torch.from_numpy(q3.reshape(B * K, V)), B, K, None, seed=3)
    assert np.array_equal(got, want["drafts"])
    assert got[2, 0] == 4321 and got[1, 2] == 0
    assert gerr == want["err"] and gerr & sd.SD_ERR_ZERO_ROW


def test_request_base_shards_reproduce_the_batch():
    rng = np.random.default_rng(23)
    B, K, V = 10, 4, 30011
    _, q, _, _ = random_probs_case(rng, B, K, V)
    rows = to_dev(q)
    whole, _ = run_sample(rows, B, K, None, seed=9)
    lo, _ = run_sample(rows[:3 * K], 3, K, None, seed=9)
    hi, _ = run_sample(rows[3 * K:], B - 3, K, None, seed=9, request_base=3)
    assert np.array_equal(np.concatenate([lo, hi]), whole)
    want = oracle_probs(rows[3 * K:], B - 3, K, None, seed=9, req_ids=np.arange(3, B))
    assert np.array_equal(hi, want["drafts"])


def test_logit_rows_within_margin():
    rng = np.random.default_rng(31)
    B, K, V = 24, 4, 50021
    lt = torch.from_numpy(2.0 * rng.standard_normal((B * K, V)).astype(np.float32))
    rows = lt.to(torch.bfloat16).cuda()
    T = torch.from_numpy(rng.uniform(0.5, 1.2, B).astype(np.float32))
    T[::5] = 0.0                      # some greedy requests
    got, gerr = run_sample(rows, B, K, T.cuda(), seed=12)
    want = oracle_logits(rows, B, K, T, seed=12)
    diverged = 0
    for i in range(B):
        for k in range(K):
            if got[i, k] != want["drafts"][i, k]:
                assert float(T[i]) != 0.0, (i, k)
                assert want["margin"][i, k] < MARGIN, (i, k, want["margin"][i, k])
                diverged += 1
    assert diverged <= max(1, int(RATE * B * K))
    assert gerr == want["err"]


@pytest.mark.parametrize("name,B", [("b64", 64), ("b1024lg", 48)])
def test_config_draft_rows(name, B):
    # the configs' draft rows stand in for the drafter's outputs at new_token_idx
    w = workloads.make(name, device="cuda", B=B)
    T = None if w.kind == "probs" else w.temperature
    got, gerr = run_sample(w.draft, w.B, w.K, T, seed=77)
    if w.kind == "probs":
        want = oracle_probs(w.draft, w.B, w.K, None, seed=77)
        assert np.array_equal(got, want["drafts"])
    else:
        want = oracle_logits(w.draft, w.B, w.K, w.temperature, seed=77)
        bad = got != want["drafts"]
        assert np.all(want["margin"][bad] < MARGIN)
        assert bad.sum() <= max(1, int(RATE * w.B * w.K))
    assert gerr == want["err"]
