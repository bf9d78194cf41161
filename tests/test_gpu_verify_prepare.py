"""GPU parity of sd_verify_prepare (verify and the drafter-batch rebuild in one call): every
output bit for bit what sd_verify then sd_pdraft_prepare write on the same inputs, on the fused
one-launch path (all-sampled probability batches that fit one wave) and on the two-kernel path;
the workspace is left zeroed; error bits agree; the rebuild matches the oracle."""

import numpy as np
import pytest
import torch

import oracle
import verify_draft_prep_gb300 as sd
import workloads

pytestmark = pytest.mark.gpu

REBUILD = ("input_ids", "positions", "slot_mapping", "hidden_map", "is_masked", "is_rejected",
           "start_loc", "new_token_idx", "total_out")


def outputs(w, cap):
    B, K, dev = w.B, w.K, "cuda"
    o = dict(out_tokens=torch.full((B, K + 1), 77, dtype=torch.int32, device=dev),
             num_accepted=torch.full((B,), 77, dtype=torch.int32, device=dev),
             p_at_draft=torch.full((B, K), 77.0, device=dev),
             q_at_draft=torch.full((B, K), 77.0, device=dev),
             input_ids=torch.full((cap,), 77, dtype=torch.int32, device=dev),
             positions=torch.full((cap,), 77, dtype=torch.int32, device=dev),
             slot_mapping=torch.full((cap,), 77, dtype=torch.int32, device=dev),
             hidden_map=torch.full((cap,), 77, dtype=torch.int32, device=dev),
             is_masked=torch.full((cap,), 77, dtype=torch.uint8, device=dev),
             is_rejected=torch.full((B, K + 1), 77, dtype=torch.uint8, device=dev),
             start_loc=torch.full((B + 1,), 77, dtype=torch.int32, device=dev),
             new_token_idx=torch.full((B, K), 77, dtype=torch.int32, device=dev),
             total_out=torch.full((1,), 77, dtype=torch.int32, device=dev),
             out_hidden=torch.full((cap, w.H), 7.0, device=dev).to(torch.bfloat16),
             err=torch.zeros(1, dtype=torch.int32, device=dev))
    return o


def run_fused(w, T, cap, ws, hidden=None, table=None):
    o = outputs(w, cap)
    hidden = w.hidden if hidden is None else hidden
    table = w.block_table if table is None else table
    sd.sd_verify_prepare(w.target, w.draft, w.drafts, o["out_tokens"], o["num_accepted"], w.pos0,
                         table, w.block_size, w.mask_token_id, o["input_ids"], o["positions"],
                         o["slot_mapping"], o["hidden_map"], o["is_masked"], o["is_rejected"],
                         o["start_loc"], o["new_token_idx"], o["total_out"], hidden, w.h_shared,
                         o["out_hidden"], temperature=T, seed=w.seed, p_at_draft=o["p_at_draft"],
                         q_at_draft=o["q_at_draft"], err=o["err"], workspace_buf=ws)
    torch.cuda.synchronize()
    return o


def run_separate(w, T, cap, hidden=None, table=None):
    o = outputs(w, cap)
    hidden = w.hidden if hidden is None else hidden
    table = w.block_table if table is None else table
    sd.sd_verify(w.target, w.draft, w.drafts, o["out_tokens"], o["num_accepted"], temperature=T,
                 seed=w.seed, p_at_draft=o["p_at_draft"], q_at_draft=o["q_at_draft"],
                 err=o["err"])
    sd.sd_pdraft_prepare(o["out_tokens"], o["num_accepted"], w.pos0, table, w.block_size,
                         w.mask_token_id, o["input_ids"], o["positions"], o["slot_mapping"],
                         o["hidden_map"], o["is_masked"], o["is_rejected"], o["start_loc"],
                         o["new_token_idx"], o["total_out"], hidden, w.h_shared, o["out_hidden"],
                         err=o["err"])
    torch.cuda.synchronize()
    return o


def assert_same(a, b):
    for k, v in a.items():
        x, y = v, b[k]
        if v.dtype == torch.bfloat16:
            x, y = v.view(torch.int16), b[k].view(torch.int16)
        assert torch.equal(x, y), k


def new_ws(B):
    n = sd.load().sd_verify_prepare_workspace_bytes(B)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("name,B,temp,kernels", [
    ("b64", 64, False, 1),      # the benchmark's workload: one launch
    ("b64", 16, False, 1),      # more CTAs per request
    ("small", 1, False, 1),     # one CTA
    ("b64", 64, True, 2),       # per-request temperatures: verify kernel, then rebuild kernel
    ("b256mix", 32, True, 2),   # greedy requests among them
    ("b512rag", 200, False, 2),  # two waves: the race kernel, then the rebuild kernel
    ("small", 192, False, 1),   # the largest batch the single launch takes
    ("small", 193, False, 2),   # one more request: two kernels
])
def test_same_bytes_as_the_two_calls(name, B, temp, kernels):
    w = workloads.make(name, device="cuda", B=B)
    T = w.temperature if temp else None
    assert sd.sd_verify_prepare_kernels(w.B, w.K, w.V, sd.SD_F32_PROBS, temp) == kernels
    ws = new_ws(w.B)
    want = run_separate(w, T, w.capacity)
    for _ in range(2):  # the workspace comes back zeroed and serves the next call
        got = run_fused(w, T, w.capacity, ws)
        assert_same(got, want)
        assert int(ws.count_nonzero()) == 0
    assert int(got["err"].item()) == 0


def test_rebuild_matches_the_oracle():
    w = workloads.make("b64", device="cuda", B=24)
    got = run_fused(w, None, w.capacity, new_ws(w.B))
    toks, acc = got["out_tokens"].cpu().numpy(), got["num_accepted"].cpu().numpy()
    e = oracle.pdraft_expand(toks, acc, w.pos0.cpu().numpy(), w.block_table.cpu().numpy(),
                             w.block_size, w.mask_token_id)
    for k in REBUILD:
        assert np.array_equal(got[k].cpu().numpy(), e[k]), k
    bits = lambda t: t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    init = torch.full((w.capacity, w.H), 7.0).to(torch.bfloat16)
    want, gerr = oracle.hidden_gather(int(e["total_out"][0]), e["hidden_map"], bits(w.hidden),
                                      bits(w.h_shared), out_init=bits(init))
    assert gerr == 0 and e["err"] == 0
    assert np.array_equal(bits(got["out_hidden"]), want)


def test_error_paths_match_the_two_calls():
    w = workloads.make("b64", device="cuda", B=32)
    table = w.block_table.clone()
    table[3, :] = -1                      # request 3's slots miss the table
    n_in = w.B * (w.K + 1) - 5            # the last request's late hidden rows are missing
    hidden = w.hidden[:n_in]
    cap = w.B * w.K                       # too small for every outcome
    for T in (None, w.temperature):
        want = run_separate(w, T, cap, hidden=hidden, table=table)
        got = run_fused(w, T, cap, new_ws(w.B), hidden=hidden, table=table)
        assert_same(got, want)
        err = int(got["err"].item())
        assert err & sd.SD_ERR_BLOCK_TABLE and err & sd.SD_ERR_TOTAL_RANGE


@pytest.mark.parametrize("B,greedy_every", [(48, 0), (40, 3), (1024, 0)])
def test_logit_rows_same_bytes_as_the_two_calls(B, greedy_every):
    # logit rows: the verify kernel (softmax statistics, decisions and races), then the rebuild
    # kernel; every output, greedy requests among them, against the two calls
    w = workloads.make("b1024lg", device="cuda", B=B)
    T = w.temperature.clone()
    if greedy_every:
        T[::greedy_every] = 0.0
    assert sd.sd_verify_prepare_kernels(w.B, w.K, w.V, sd.SD_BF16_LOGITS, True) == 2
    ws = new_ws(w.B)
    want = run_separate(w, T, w.capacity)
    for _ in range(2):  # the workspace comes back zeroed and serves the next call
        got = run_fused(w, T, w.capacity, ws)
        assert_same(got, want)
        assert int(ws.count_nonzero()) == 0
    assert int(got["err"].item()) == 0
    assert int((got["input_ids"] == -1).sum()) == w.capacity - int(got["total_out"].item())


def test_logit_rows_error_paths_match_the_two_calls():
    w = workloads.make("b1024lg", device="cuda", B=24)
    table = w.block_table.clone()
    table[5, :] = -1                      # request 5's slots miss the table
    n_in = w.B * (w.K + 1) - 7            # the last request's late hidden rows are missing
    hidden = w.hidden[:n_in]
    cap = w.B * w.K                       # too small for every outcome
    want = run_separate(w, w.temperature, cap, hidden=hidden, table=table)
    got = run_fused(w, w.temperature, cap, new_ws(w.B), hidden=hidden, table=table)
    assert_same(got, want)
    err = int(got["err"].item())
    assert err & sd.SD_ERR_BLOCK_TABLE and err & sd.SD_ERR_TOTAL_RANGE


def test_out_of_range_drafts_match_the_two_calls():
    # a draft token outside [0, V) is rejected with SD_ERR_TOKEN_RANGE; on the single launch the
    # rebuild CTA, which recomputes the decisions, raises it
    w = workloads.make("b64", device="cuda", B=16)
    w.drafts = w.drafts.clone()
    w.drafts[2, 0] = w.V            # request 2: its first draft is out of range
    w.drafts[5, 3] = -4             # request 5: its fourth
    assert sd.sd_verify_prepare_kernels(w.B, w.K, w.V, sd.SD_F32_PROBS, False) == 1
    want = run_separate(w, None, w.capacity)
    got = run_fused(w, None, w.capacity, new_ws(w.B))
    assert_same(got, want)
    assert int(got["err"].item()) & sd.SD_ERR_TOKEN_RANGE
    assert int(got["num_accepted"][2]) == 0


def test_unaligned_rows_and_ragged_vocabulary():
    # rows that do not start on 16-byte boundaries (scalar loads) and a vocabulary that is not a
    # multiple of the 4-entry unit: the single launch's race tails, against the two calls
    rng = np.random.default_rng(11)
    B, K, V, H = 24, 3, 5003, 40
    w = workloads.make("small", device="cuda", B=B)
    lt = 2.0 * rng.standard_normal((B * (K + 1), V))
    p = np.exp(lt - lt.max(-1, keepdims=True))
    p = (p / p.sum(-1, keepdims=True)).astype(np.float32)
    lq = lt[np.arange(B * (K + 1)).reshape(B, K + 1)[:, :K].reshape(-1)] + 0.5 * rng.standard_normal((B * K, V))
    q = np.exp(lq - lq.max(-1, keepdims=True))
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    q64 = q.astype(np.float64)
    d = np.array([rng.choice(V, p=q64[i] / q64[i].sum()) for i in range(B * K)],
                 np.int32).reshape(B, K)
    ld = V + 1                                      # odd row stride: no 16-byte rows
    tbuf = torch.zeros(B * (K + 1), ld, device="cuda")
    dbuf = torch.zeros(B * K, ld, device="cuda")
    tbuf[:, :V] = torch.from_numpy(p).cuda()
    dbuf[:, :V] = torch.from_numpy(q).cuda()
    w.target, w.draft = tbuf[:, :V], dbuf[:, :V]
    w.drafts = torch.from_numpy(d).cuda()
    w.K, w.V, w.H = K, V, H
    w.hidden = torch.from_numpy(rng.standard_normal((B * (K + 1), H)).astype(np.float32)).to(
        torch.bfloat16).cuda()
    w.h_shared = torch.from_numpy(rng.standard_normal(H).astype(np.float32)).to(torch.bfloat16).cuda()
    w.mask_token_id = V
    assert sd.sd_verify_prepare_kernels(B, K, V, sd.SD_F32_PROBS, False) == 1
    want = run_separate(w, None, w.capacity)
    got = run_fused(w, None, w.capacity, new_ws(B))
    assert_same(got, want)
    assert int(got["err"].item()) == 0
    ref = oracle.verify_probs(p.reshape(B, K + 1, V), q.reshape(B, K, V), d, seed=w.seed)
    assert np.array_equal(got["out_tokens"].cpu().numpy(), ref["out_tokens"])


@pytest.mark.parametrize("withhold", [0, 37, 63])
def test_bounded_wait_runs_out_cleanly(withhold):
    # The single launch's one wait: the CTA completing a request's race row polls for the first
    # drafter slot the request's rebuild CTA publishes. The diagnostic entry holds one request's
    # publication back until that wait has run out (500 us of the GPU clock): the call must raise
    # SD_ERR_WAIT, leave only that request's final drafter token unwritten, leave the workspace
    # zeroed, and the next call must be whole again. Nothing faults, traps or hangs.
    w = workloads.make("b64", device="cuda")
    assert sd.sd_verify_prepare_kernels(w.B, w.K, w.V, sd.SD_F32_PROBS, False) == 1
    cap = w.capacity
    ws = new_ws(w.B)
    want = run_separate(w, None, cap)
    o = outputs(w, cap)
    sd.sd_verify_prepare(w.target, w.draft, w.drafts, o["out_tokens"], o["num_accepted"], w.pos0,
                         w.block_table, w.block_size, w.mask_token_id, o["input_ids"],
                         o["positions"], o["slot_mapping"], o["hidden_map"], o["is_masked"],
                         o["is_rejected"], o["start_loc"], o["new_token_idx"], o["total_out"],
                         w.hidden, w.h_shared, o["out_hidden"], seed=w.seed,
                         p_at_draft=o["p_at_draft"], q_at_draft=o["q_at_draft"], err=o["err"],
                         workspace_buf=ws, diag_withhold=(withhold, 500))
    torch.cuda.synchronize()
    assert int(o["err"].item()) == sd.SD_ERR_WAIT
    assert int(ws.count_nonzero()) == 0
    g = int(want["start_loc"][withhold]) + int(want["num_accepted"][withhold])
    ids = want["input_ids"].clone()
    ids[g] = 77  # the prefill: the withheld request's final token is not written
    assert torch.equal(o["input_ids"], ids)
    for k in o:
        if k not in ("input_ids", "err"):
            x, y = o[k], want[k]
            if x.dtype == torch.bfloat16:
                x, y = x.view(torch.int16), y.view(torch.int16)
            assert torch.equal(x, y), k
    got = run_fused(w, None, cap, ws)
    assert_same(got, want)
    assert int(ws.count_nonzero()) == 0


def test_withheld_diagnostic_without_a_wait():
    # batches that take two kernels have no wait: the diagnostic entry then writes what
    # sd_verify_prepare writes, with no error
    w = workloads.make("b64", device="cuda", B=16)
    T = w.temperature
    assert sd.sd_verify_prepare_kernels(w.B, w.K, w.V, sd.SD_F32_PROBS, True) == 2
    want = run_separate(w, T, w.capacity)
    o = outputs(w, w.capacity)
    sd.sd_verify_prepare(w.target, w.draft, w.drafts, o["out_tokens"], o["num_accepted"], w.pos0,
                         w.block_table, w.block_size, w.mask_token_id, o["input_ids"],
                         o["positions"], o["slot_mapping"], o["hidden_map"], o["is_masked"],
                         o["is_rejected"], o["start_loc"], o["new_token_idx"], o["total_out"],
                         w.hidden, w.h_shared, o["out_hidden"], temperature=T, seed=w.seed,
                         p_at_draft=o["p_at_draft"], q_at_draft=o["q_at_draft"], err=o["err"],
                         workspace_buf=new_ws(w.B), diag_withhold=(3, 500))
    torch.cuda.synchronize()
    assert_same(o, want)
