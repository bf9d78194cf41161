"""GPU parity on the five named workloads at full size, in the launch configuration the
benchmark times (verify -> expand -> gather on one stream). The oracle checks every request of
every configuration. The larger ones go to the oracle in chunks of requests (verify is
independent per request, and the oracle takes the request index for its Philox counters), so
that only one chunk's rows are on the host at a time. Expand and gather are then checked
bit-exact on the GPU's own verify outputs."""

import numpy as np
import pytest
import torch

import oracle
import verify_draft_prep_gb300 as sd
import workloads
from devrun import assert_verify_equal, oracle_verify_rows
from test_gpu_logits import MARGIN, RATE, compare_logits  # noqa: F401

pytestmark = pytest.mark.gpu


def run_step(w):
    B, K, dev = w.B, w.K, "cuda"
    cap = w.capacity
    o = dict(out_tokens=torch.empty(B, K + 1, dtype=torch.int32, device=dev),
             num_accepted=torch.empty(B, dtype=torch.int32, device=dev),
             p_at_draft=torch.empty(B, K, device=dev), q_at_draft=torch.empty(B, K, device=dev),
             input_ids=torch.empty(cap, dtype=torch.int32, device=dev),
             positions=torch.empty(cap, dtype=torch.int32, device=dev),
             slot_mapping=torch.empty(cap, dtype=torch.int32, device=dev),
             hidden_map=torch.empty(cap, dtype=torch.int32, device=dev),
             is_masked=torch.empty(cap, dtype=torch.uint8, device=dev),
             is_rejected=torch.empty(B, K + 1, dtype=torch.uint8, device=dev),
             start_loc=torch.empty(B + 1, dtype=torch.int32, device=dev),
             new_token_idx=torch.empty(B, K, dtype=torch.int32, device=dev),
             total_out=torch.empty(1, dtype=torch.int32, device=dev),
             out_hidden=torch.full((cap, w.H), 7.0, device=dev).to(torch.bfloat16),
             err=torch.zeros(1, dtype=torch.int32, device=dev))
    sd.sd_verify(w.target, w.draft, w.drafts, o["out_tokens"], o["num_accepted"],
                 temperature=w.temperature, seed=w.seed, p_at_draft=o["p_at_draft"],
                 q_at_draft=o["q_at_draft"], err=o["err"])
    sd.sd_pdraft_expand(o["out_tokens"], o["num_accepted"], w.pos0, w.block_table, w.block_size,
                        w.mask_token_id, o["input_ids"], o["positions"], o["slot_mapping"],
                        o["hidden_map"], o["is_masked"], o["is_rejected"], o["start_loc"],
                        o["new_token_idx"], o["total_out"], err=o["err"])
    sd.sd_hidden_gather(o["total_out"], o["hidden_map"], w.hidden, w.h_shared, o["out_hidden"],
                        err=o["err"])
    # the fused rebuild (the benchmark's path) must write the same bytes
    p = {k: torch.full_like(o[k], 77) for k in ("input_ids", "positions", "slot_mapping",
                                                  "hidden_map", "is_masked", "is_rejected",
                                                  "start_loc", "new_token_idx", "total_out")}
    p_hidden = torch.full((cap, w.H), 7.0, device=dev).to(torch.bfloat16)
    sd.sd_pdraft_prepare(o["out_tokens"], o["num_accepted"], w.pos0, w.block_table, w.block_size,
                         w.mask_token_id, p["input_ids"], p["positions"], p["slot_mapping"],
                         p["hidden_map"], p["is_masked"], p["is_rejected"], p["start_loc"],
                         p["new_token_idx"], p["total_out"], w.hidden, w.h_shared, p_hidden,
                         err=o["err"])
    torch.cuda.synchronize()
    for k, v in p.items():
        assert torch.equal(v, o[k]), k
    assert torch.equal(p_hidden.view(torch.int16), o["out_hidden"].view(torch.int16))
    res = {k: v.cpu() for k, v in o.items()}
    res = {k: (v.numpy() if v.dtype != torch.bfloat16 else v) for k, v in res.items()}
    res["err"] = int(res["err"][0])
    return res


def check_prep(w, res):
    e = oracle.pdraft_expand(res["out_tokens"], res["num_accepted"], w.pos0.cpu().numpy(),
                             w.block_table.cpu().numpy(), w.block_size, w.mask_token_id)
    for k in ("input_ids", "positions", "slot_mapping", "hidden_map", "is_masked", "is_rejected",
              "start_loc", "new_token_idx", "total_out"):
        assert np.array_equal(res[k], e[k]), k
    assert e["err"] == 0
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    init = torch.full((w.capacity, w.H), 7.0).to(torch.bfloat16)
    want, gerr = oracle.hidden_gather(int(e["total_out"][0]), e["hidden_map"], bits(w.hidden.cpu()),
                                      bits(w.h_shared.cpu()), out_init=bits(init))
    assert gerr == 0
    assert np.array_equal(bits(res["out_hidden"]), want)


def oracle_all_requests(w, chunk):
    """The oracle on every request of the batch, `chunk` requests at a time (each chunk's rows
    are copied to the host on their own; the request indices keep the Philox counters)."""
    parts, err = [], 0
    for c0 in range(0, w.B, chunk):
        req = np.arange(c0, min(w.B, c0 + chunk), dtype=np.int32)
        res = oracle_verify_rows(w.target, w.draft, w.drafts, w.temperature, seed=w.seed,
                                 req_ids=req)
        err |= res.pop("err")
        parts.append(res)
    want = {k: np.concatenate([p[k] for p in parts]) for k in parts[0]}
    want["err"] = err
    return want


@pytest.mark.parametrize("name,null_temp", [("small", False), ("b64", False), ("b64", True),
                                            ("b256mix", False), ("b512rag", False),
                                            ("b512rag", True)])
def test_probs_config_full_size(name, null_temp):
    w = workloads.make(name, device="cuda")
    if null_temp:  # every request samples at T = 1: the same results through the NULL path
        assert bool((w.temperature == 1).all())
        w.temperature = None
    res = run_step(w)
    want = oracle_all_requests(w, chunk=128)
    got = {k: res[k] for k in ("out_tokens", "num_accepted", "p_at_draft", "q_at_draft")}
    got["err"] = res["err"]
    assert_verify_equal(got, want)
    check_prep(w, res)
    a = res["num_accepted"]
    print(f"{name}: all {w.B} requests bit-exact; mean accepted {a.mean():.3f}, "
          f"histogram {np.bincount(a, minlength=w.K + 1)}")


def test_logits_config_full_size():
    w = workloads.make("b1024lg", device="cuda")
    res = run_step(w)
    want = oracle_all_requests(w, chunk=128)
    got = {k: res[k] for k in ("out_tokens", "num_accepted", "p_at_draft", "q_at_draft")}
    div = compare_logits(got, want, w.K)
    positions = w.B * (w.K + 1)
    print(f"b1024lg: all {w.B} requests; {div} tolerated divergences at margins below {MARGIN} "
          f"over {positions} positions (limit {RATE * positions:.2f})")
    assert div <= RATE * positions
    assert res["err"] == 0 and want["err"] == 0
    check_prep(w, res)
