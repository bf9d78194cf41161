"""GPU parity of sd_pdraft_prepare_padded (fixed rows of 2K drafter slots, rejected leftovers on
PADDING_SLOT_ID, scatter-form hidden map) against the oracle: every output element and every
hidden byte bit-exact, error bits equal."""

import json

import numpy as np
import pytest
import torch

import oracle
import verify_draft_prep_gb300 as sd
import workloads
from conftest import golden_path

pytestmark = pytest.mark.gpu

KEYS = ("input_ids", "positions", "slot_mapping", "hidden_map", "is_masked", "rejected",
        "scatter_map", "new_token_idx")


def _i32(a):
    return torch.as_tensor(np.ascontiguousarray(a, np.int32)).cuda()


def run_padded(out_tokens, num_acc, pos0, table, bs, mask_id, hidden=None, h_shared=None):
    B, K1 = out_tokens.shape
    K = K1 - 1
    n = B * 2 * K
    dev = "cuda"
    o = dict(input_ids=torch.full((n,), 555, dtype=torch.int32, device=dev),
             positions=torch.full((n,), 555, dtype=torch.int32, device=dev),
             slot_mapping=torch.full((n,), 555, dtype=torch.int32, device=dev),
             hidden_map=torch.full((n,), 555, dtype=torch.int32, device=dev),
             is_masked=torch.full((n,), 9, dtype=torch.uint8, device=dev),
             rejected=torch.full((n,), 9, dtype=torch.uint8, device=dev),
             scatter_map=torch.full((B * K1,), 555, dtype=torch.int32, device=dev),
             new_token_idx=torch.full((B, K), 555, dtype=torch.int32, device=dev))
    out_hidden = None
    if hidden is not None:
        out_hidden = torch.full((n, hidden.shape[1]), 7, dtype=torch.int16, device=dev).view(
            torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sd.sd_pdraft_prepare_padded(_i32(out_tokens), _i32(num_acc), _i32(pos0), _i32(table), bs,
                                mask_id, o["input_ids"], o["positions"], o["slot_mapping"],
                                o["hidden_map"], o["is_masked"], o["rejected"], o["scatter_map"],
                                o["new_token_idx"], target_hidden=hidden, h_shared=h_shared,
                                out_hidden=out_hidden, err=err)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in o.items()}
    if out_hidden is not None:
        res["out_hidden"] = out_hidden.view(torch.int16).cpu().numpy().view(np.uint16)
    res["err"] = int(err.item())
    return res


def bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def test_hand_example_on_gpu():
    g = json.load(open(golden_path("padded_hand_example.json")))
    B, K = len(g["num_accepted"]), g["K"]
    rng = np.random.default_rng(1)
    hid = torch.from_numpy(rng.standard_normal((B * (K + 1), 8)).astype(np.float32)).to(
        torch.bfloat16).cuda()
    hs = torch.from_numpy(rng.standard_normal(8).astype(np.float32)).to(torch.bfloat16).cuda()
    got = run_padded(np.array(g["out_tokens"]), g["num_accepted"], g["pos0"],
                     np.array(g["block_table"]), g["block_size"], g["mask_token_id"], hid, hs)
    for k, v in g["expected"].items():
        assert np.array_equal(np.ravel(got[k]), np.ravel(v)), k
    hb, sb = bits(hid), bits(hs)
    for i, m in enumerate(g["expected"]["hidden_map"]):
        assert np.array_equal(got["out_hidden"][i], hb[m] if m >= 0 else sb), i
    assert got["err"] == 0


@pytest.mark.parametrize("name,B", [("small", 1), ("b64", 64), ("b1024lg", 1024)])
def test_config_rebuild_bit_exact(name, B):
    w = workloads.make(name, device="cuda", B=B)
    rng = np.random.default_rng(B)
    K = w.K
    a = rng.integers(0, K + 1, w.B).astype(np.int32)
    toks = rng.integers(0, w.V, (w.B, K + 1)).astype(np.int32)
    for r in range(w.B):
        toks[r, a[r] + 1:] = -1
    got = run_padded(toks, a, w.pos0.cpu().numpy(), w.block_table.cpu().numpy(), w.block_size,
                     w.mask_token_id, w.hidden, w.h_shared)
    want = oracle.pdraft_prepare_padded(toks, a, w.pos0.cpu().numpy(),
                                        w.block_table.cpu().numpy(), w.block_size,
                                        w.mask_token_id, bits(w.hidden), bits(w.h_shared))
    for k in KEYS + ("out_hidden",):
        assert np.array_equal(got[k].reshape(-1), want[k].reshape(-1)), k
    assert got["err"] == want["err"] == 0


def test_errors_and_metadata_only():
    toks = np.array([[5, 6, 7], [8, 9, 10]], np.int32)
    a = np.array([3, -1], np.int32)
    pos0 = np.array([0, 100], np.int32)
    table = np.array([[0, 1], [2, 3]], np.int32)
    got = run_padded(toks, a, pos0, table, 16, 99)           # no hidden states: metadata only
    rng = np.random.default_rng(2)
    want = oracle.pdraft_prepare_padded(toks, a, pos0, table, 16, 99,
                                        rng.integers(0, 9, (6, 2), dtype=np.uint16),
                                        np.zeros(2, np.uint16))
    for k in KEYS:
        assert np.array_equal(got[k].reshape(-1), want[k].reshape(-1)), k
    assert got["err"] == want["err"]
    assert got["err"] & sd.SD_ERR_NUM_ACCEPTED and got["err"] & sd.SD_ERR_BLOCK_TABLE


def test_after_verify_in_stream_order():
    # the rebuild reads sd_verify's outputs on the same stream (a programmatic dependent launch)
    w = workloads.make("b64", device="cuda", B=16)
    B, K = w.B, w.K
    out_tokens = torch.empty(B, K + 1, dtype=torch.int32, device="cuda")
    num_acc = torch.empty(B, dtype=torch.int32, device="cuda")
    sd.sd_verify(w.target, w.draft, w.drafts, out_tokens, num_acc, temperature=w.temperature,
                 seed=w.seed)
    n = B * 2 * K
    o = {k: torch.empty(n, dtype=torch.int32, device="cuda")
         for k in ("input_ids", "positions", "slot_mapping", "hidden_map")}
    m8 = {k: torch.empty(n, dtype=torch.uint8, device="cuda") for k in ("is_masked", "rejected")}
    sm = torch.empty(B * (K + 1), dtype=torch.int32, device="cuda")
    nti = torch.empty(B, K, dtype=torch.int32, device="cuda")
    sd.sd_pdraft_prepare_padded(out_tokens, num_acc, w.pos0, w.block_table, w.block_size,
                                w.mask_token_id, o["input_ids"], o["positions"],
                                o["slot_mapping"], o["hidden_map"], m8["is_masked"],
                                m8["rejected"], sm, nti)
    torch.cuda.synchronize()
    want = oracle.pdraft_prepare_padded(out_tokens.cpu().numpy(), num_acc.cpu().numpy(),
                                        w.pos0.cpu().numpy(), w.block_table.cpu().numpy(),
                                        w.block_size, w.mask_token_id,
                                        np.zeros((B * (K + 1), 1), np.uint16),
                                        np.zeros(1, np.uint16))
    assert np.array_equal(o["input_ids"].cpu().numpy(), want["input_ids"])
    assert np.array_equal(nti.cpu().numpy(), want["new_token_idx"])
    assert np.array_equal(sm.cpu().numpy(), want["scatter_map"])
