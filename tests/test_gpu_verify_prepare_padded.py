"""GPU parity of sd_verify_prepare_padded (verify and the padded drafter-batch rebuild in one call):
every output bit for bit what sd_verify then sd_pdraft_prepare_padded write on the same inputs, on
the single launch (all-sampled probability batches of one wave, where each rebuild CTA recomputes
its own request's decisions and the race writes the final token at its fixed row) and on the
two-kernel path; the workspace is left zeroed; error bits agree; the rows match the oracle."""

import numpy as np
import pytest
import torch

import oracle
import verify_draft_prep_gb300 as sd
import workloads

pytestmark = pytest.mark.gpu

PADDED = ("input_ids", "positions", "slot_mapping", "hidden_map", "is_masked", "rejected",
          "scatter_map", "new_token_idx")


def outputs(w):
    B, K, dev = w.B, w.K, "cuda"
    n = B * 2 * K
    i32 = lambda *s: torch.full(s, 77, dtype=torch.int32, device=dev)  # noqa: E731
    u8 = lambda *s: torch.full(s, 77, dtype=torch.uint8, device=dev)  # noqa: E731
    return dict(out_tokens=i32(B, K + 1), num_accepted=i32(B),
                p_at_draft=torch.full((B, K), 77.0, device=dev),
                q_at_draft=torch.full((B, K), 77.0, device=dev),
                input_ids=i32(n), positions=i32(n), slot_mapping=i32(n), hidden_map=i32(n),
                is_masked=u8(n), rejected=u8(n), scatter_map=i32(B * (K + 1)),
                new_token_idx=i32(B, K),
                out_hidden=torch.full((n, w.H), 7.0, device=dev).to(torch.bfloat16),
                err=torch.zeros(1, dtype=torch.int32, device=dev))


def run_one_call(w, T, ws, hidden=None, table=None):
    o = outputs(w)
    hidden = w.hidden if hidden is None else hidden
    table = w.block_table if table is None else table
    sd.sd_verify_prepare_padded(
        w.target, w.draft, w.drafts, o["out_tokens"], o["num_accepted"], w.pos0, table,
        w.block_size, w.mask_token_id, o["input_ids"], o["positions"], o["slot_mapping"],
        o["hidden_map"], o["is_masked"], o["rejected"], o["scatter_map"], o["new_token_idx"],
        target_hidden=hidden, h_shared=w.h_shared, out_hidden=o["out_hidden"], temperature=T,
        seed=w.seed, p_at_draft=o["p_at_draft"], q_at_draft=o["q_at_draft"], err=o["err"],
        workspace_buf=ws)
    torch.cuda.synchronize()
    return o


def run_two_calls(w, T, hidden=None, table=None):
    o = outputs(w)
    hidden = w.hidden if hidden is None else hidden
    table = w.block_table if table is None else table
    sd.sd_verify(w.target, w.draft, w.drafts, o["out_tokens"], o["num_accepted"], temperature=T,
                 seed=w.seed, p_at_draft=o["p_at_draft"], q_at_draft=o["q_at_draft"],
                 err=o["err"])
    sd.sd_pdraft_prepare_padded(o["out_tokens"], o["num_accepted"], w.pos0, table, w.block_size,
                                w.mask_token_id, o["input_ids"], o["positions"],
                                o["slot_mapping"], o["hidden_map"], o["is_masked"],
                                o["rejected"], o["scatter_map"], o["new_token_idx"],
                                target_hidden=hidden, h_shared=w.h_shared,
                                out_hidden=o["out_hidden"], err=o["err"])
    torch.cuda.synchronize()
    return o


def assert_same(a, b):
    for k, v in a.items():
        x, y = v, b[k]
        if v.dtype == torch.bfloat16:
            x, y = v.view(torch.int16), b[k].view(torch.int16)
        assert torch.equal(x, y), k


def new_ws(w, dtype=sd.SD_F32_PROBS):
    n = sd.load().sd_verify_workspace_bytes(w.B, w.K, w.V, dtype)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("name,B,temp,kernels", [
    ("b64", 64, False, 1),       # the benchmark's all-sampled batch: one launch
    ("b64", 16, False, 1),       # more race CTAs per request
    ("small", 1, False, 1),      # one request
    ("small", 192, False, 1),    # the largest batch the single launch takes
    ("small", 193, False, 2),    # one more: the verify kernel, then the padded rebuild kernel
    ("b64", 64, True, 2),        # per-request temperatures
    ("b256mix", 32, True, 2),    # greedy requests among them
    ("b512rag", 200, False, 2),  # two waves: the race kernel, then the rebuild kernel
    ("b1024lg", 24, True, 2),    # logit rows, clusters of 8
    ("b1024lg", 192, True, 2),   # logit rows, clusters of 4
])
def test_same_bytes_as_the_two_calls(name, B, temp, kernels):
    w = workloads.make(name, device="cuda", B=B)
    T = w.temperature if temp else None
    dtype = sd.SD_BF16_LOGITS if w.kind == "logits" else sd.SD_F32_PROBS
    assert sd.sd_verify_prepare_kernels(w.B, w.K, w.V, dtype, temp) == kernels
    ws = new_ws(w, dtype)
    want = run_two_calls(w, T)
    for _ in range(2):  # the workspace comes back zeroed and serves the next call
        got = run_one_call(w, T, ws)
        assert_same(got, want)
        assert int(ws.count_nonzero()) == 0
    assert int(got["err"].item()) == 0


@pytest.mark.parametrize("name,B,temp", [
    ("b64", 24, False),      # the single launch of rebuild CTAs and race CTAs
    ("b256mix", 32, True),   # verify kernel then the padded rebuild kernel
    ("b1024lg", 24, True),   # the same on logit rows
])
def test_rows_match_the_oracle(name, B, temp):
    w = workloads.make(name, device="cuda", B=B)
    dtype = sd.SD_BF16_LOGITS if w.kind == "logits" else sd.SD_F32_PROBS
    got = run_one_call(w, w.temperature if temp else None, new_ws(w, dtype))
    bits = lambda t: t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    want = oracle.pdraft_prepare_padded(got["out_tokens"].cpu().numpy(),
                                        got["num_accepted"].cpu().numpy(), w.pos0.cpu().numpy(),
                                        w.block_table.cpu().numpy(), w.block_size,
                                        w.mask_token_id, bits(w.hidden), bits(w.h_shared))
    for k in PADDED:
        assert np.array_equal(got[k].cpu().numpy().reshape(-1), want[k].reshape(-1)), k
    assert np.array_equal(bits(got["out_hidden"]).reshape(-1), want["out_hidden"].reshape(-1))
    assert want["err"] == 0


@pytest.mark.parametrize("name", ["b64", "b1024lg"])
def test_error_paths_match_the_two_calls(name):
    w = workloads.make(name, device="cuda", B=32)
    dtype = sd.SD_BF16_LOGITS if w.kind == "logits" else sd.SD_F32_PROBS
    table = w.block_table.clone()
    table[3, :] = -1                      # request 3's live slots miss the table
    n_in = w.B * (w.K + 1) - 5            # the last request's late hidden rows are missing
    hidden = w.hidden[:n_in]
    w.drafts = w.drafts.clone()
    w.drafts[6, 0] = w.V                  # request 6: its first draft is out of range
    for T in (None, w.temperature):
        want = run_two_calls(w, T, hidden=hidden, table=table)
        got = run_one_call(w, T, new_ws(w, dtype), hidden=hidden, table=table)
        assert_same(got, want)
        err = int(got["err"].item())
        assert err & sd.SD_ERR_BLOCK_TABLE and err & sd.SD_ERR_TOKEN_RANGE
        assert int(got["num_accepted"][6]) == 0
