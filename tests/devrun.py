"""Helpers for the GPU parity tests: run the library through its Python binding on device
tensors, run the oracle on host copies of the same inputs, compare."""

import numpy as np
import torch

import oracle
import verify_draft_prep_gb300 as sd

DEV = "cuda"


def to_dev(a, dtype=None):
    t = torch.as_tensor(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(DEV)


def run_verify(target, draft, drafts, temperature=None, seed=0, request_base=0):
    """target [B*(K+1), V], draft [B*K, V] device tensors (fp32 or bf16)."""
    B, K = drafts.shape
    dev = target.device
    out = dict(out_tokens=torch.full((B, K + 1), -7, dtype=torch.int32, device=dev),
               num_accepted=torch.full((B,), -7, dtype=torch.int32, device=dev),
               p_at_draft=torch.full((B, K), -7.0, device=dev),
               q_at_draft=torch.full((B, K), -7.0, device=dev),
               err=torch.zeros(1, dtype=torch.int32, device=dev))
    sd.sd_verify(target, draft, drafts, out["out_tokens"], out["num_accepted"],
                 temperature=temperature, seed=seed, p_at_draft=out["p_at_draft"],
                 q_at_draft=out["q_at_draft"], err=out["err"], request_base=request_base)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    res["err"] = int(res["err"][0])
    return res


def oracle_verify_rows(target, draft, drafts, temperature=None, seed=0, req_ids=None):
    """Oracle on host copies; target [B*(K+1), V] / draft [B*K, V] (torch, any device)."""
    B, K = drafts.shape
    drafts_h = drafts.cpu().numpy()
    temp_h = None if temperature is None else temperature.cpu().numpy()
    if req_ids is not None:
        idx = torch.as_tensor(req_ids, dtype=torch.long, device=target.device)
        t3 = target.view(B, K + 1, -1)[idx]
        d3 = draft.view(B, K, -1)[idx]
        drafts_h = drafts_h[np.asarray(req_ids)]
        temp_h = None if temp_h is None else temp_h[np.asarray(req_ids)]
        rid = np.asarray(req_ids, np.int32)
    else:
        t3 = target.view(B, K + 1, -1)
        d3 = draft.view(B, K, -1)
        rid = None
    if target.dtype == torch.float32:
        return oracle.verify_probs(t3.cpu().numpy(), d3.cpu().numpy(), drafts_h,
                                   temperature=temp_h, seed=seed, req_ids=rid)
    tb = t3.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    db = d3.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return oracle.verify_logits(tb, db, drafts_h, temperature=temp_h, seed=seed, req_ids=rid,
                                margins=True)


def assert_verify_equal(got, want, req_ids=None, check_err=True):
    sel = slice(None) if req_ids is None else np.asarray(req_ids)
    for k in ("num_accepted", "out_tokens"):
        g = got[k][sel]
        if not np.array_equal(g, want[k]):
            bad = np.nonzero((g != want[k]).reshape(len(g), -1).any(axis=1))[0]
            raise AssertionError(f"{k} differs on {bad.size} requests, first {bad[:8]}: "
                                 f"gpu {g[bad[:3]]} oracle {want[k][bad[:3]]}")
    for k in ("p_at_draft", "q_at_draft"):
        g = got[k][sel]
        assert np.array_equal(g.view(np.uint32), want[k].view(np.uint32)), k
    if check_err:
        assert got["err"] == want["err"], (got["err"], want["err"])


def random_probs_case(rng, B, K, V, sigma=0.5, greedy_frac=0.0, zero_frac=0.0):
    """Host numpy case: target [B*(K+1), V], draft [B*K, V], drafts [B, K], temperature [B]."""
    l = 2.0 * rng.standard_normal((B, K + 1, V))
    p = np.exp(l - l.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    lq = l[:, :K] + sigma * rng.standard_normal((B, K, V))
    q = np.exp(lq - lq.max(-1, keepdims=True))
    q /= q.sum(-1, keepdims=True)
    p = p.astype(np.float32)
    q = q.astype(np.float32)
    if zero_frac:
        p[rng.random(p.shape) < zero_frac] = 0
        q[rng.random(q.shape) < zero_frac] = 0
    drafts = np.empty((B, K), np.int32)
    for b in range(B):
        for j in range(K):
            qq = q[b, j].astype(np.float64)
            s = qq.sum()
            drafts[b, j] = rng.choice(V, p=qq / s) if s > 0 else rng.integers(0, V)
    temp = np.ones(B, np.float32)
    g = rng.random(B) < greedy_frac
    temp[g] = 0.0
    for b in np.nonzero(g)[0]:
        drafts[b] = q[b].argmax(-1)
        # make some greedy drafts match the target's argmax
        m = rng.integers(0, K + 1)
        drafts[b, :m] = p[b, :m].argmax(-1)
    return (p.reshape(B * (K + 1), V), q.reshape(B * K, V), drafts, temp)
