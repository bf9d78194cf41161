"""GPU parity of sd_pdraft_prepare_ragged (the rebuild with a draft count per request) against
the oracle: a hand-worked example, random batches with hidden states, and the whole ragged step
(sd_verify_ragged, then the ragged rebuild) against the oracle's ragged verify and rebuild."""

import json

import numpy as np
import pytest
import torch

import oracle
import verify_draft_prep_gb300 as sd
from conftest import golden_path
from devrun import to_dev
from test_gpu_ragged import ragged_case

pytestmark = pytest.mark.gpu

KEYS = ("input_ids", "positions", "slot_mapping", "hidden_map", "is_masked", "is_rejected",
        "start_loc", "new_token_idx", "total_out")


def _i32(a):
    return torch.as_tensor(np.ascontiguousarray(a, np.int32)).cuda()


def bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run_prepare_ragged(out_tokens, num_acc, cu, pos0, table, bs, mask_id, hidden, h_shared):
    B, K1 = out_tokens.shape
    K = K1 - 1
    cap = B * 2 * K
    dev = "cuda"
    fill = lambda shape, v, dt=torch.int32: torch.full(shape, v, dtype=dt, device=dev)  # noqa
    o = dict(input_ids=fill((cap,), 555), positions=fill((cap,), 555),
             slot_mapping=fill((cap,), 555), hidden_map=fill((cap,), 555),
             is_masked=fill((cap,), 9, torch.uint8), is_rejected=fill((B, K + 1), 9, torch.uint8),
             start_loc=fill((B + 1,), 555), new_token_idx=fill((B, K), 555),
             total_out=fill((1,), 555))
    out_hidden = torch.zeros(cap, hidden.shape[1], dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ot = out_tokens if torch.is_tensor(out_tokens) else _i32(out_tokens)
    na = num_acc if torch.is_tensor(num_acc) else _i32(num_acc)
    sd.sd_pdraft_prepare_ragged(ot, na, _i32(cu), _i32(pos0), _i32(table), bs, mask_id,
                                o["input_ids"], o["positions"], o["slot_mapping"],
                                o["hidden_map"], o["is_masked"], o["is_rejected"],
                                o["start_loc"], o["new_token_idx"], o["total_out"], hidden,
                                h_shared, out_hidden, err=err)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in o.items()}
    res["out_hidden"] = bits(out_hidden)
    res["err"] = int(err.item())
    return res


def test_hand_example_on_gpu():
    g = json.load(open(golden_path("expand_ragged_hand_example.json")))
    rng = np.random.default_rng(2)
    n_rows = g["cu_drafts"][-1] + len(g["num_accepted"])
    hid = torch.from_numpy(rng.standard_normal((n_rows, 8)).astype(np.float32)).to(
        torch.bfloat16).cuda()
    hs = torch.from_numpy(rng.standard_normal(8).astype(np.float32)).to(torch.bfloat16).cuda()
    got = run_prepare_ragged(np.array(g["out_tokens"]), g["num_accepted"], g["cu_drafts"],
                             g["pos0"], np.array(g["block_table"]), g["block_size"],
                             g["mask_token_id"], hid, hs)
    for k, v in g["expected"].items():
        assert np.array_equal(np.ravel(got[k]), np.ravel(v)), k
    hb, sb = bits(hid), bits(hs)
    for i, m in enumerate(g["expected"]["hidden_map"][:g["expected"]["total_out"]]):
        assert np.array_equal(got["out_hidden"][i], hb[m] if m >= 0 else sb), i
    assert got["err"] == 0


def test_ragged_step_end_to_end():
    rng = np.random.default_rng(41)
    B, K_max, V, H, bs = 48, 6, 20011, 256, 16
    p, q, d, cu, T = ragged_case(rng, B, K_max, V, greedy_frac=0.3)
    pos0 = rng.integers(0, 2000, B).astype(np.int32)
    width = (int(pos0.max()) + 2 * K_max) // bs + 1
    table = rng.permutation(B * width).astype(np.int32).reshape(B, width)
    hid = torch.from_numpy(rng.standard_normal((int(cu[-1]) + B, H)).astype(np.float32)).to(
        torch.bfloat16).cuda()
    hs = torch.from_numpy(rng.standard_normal(H).astype(np.float32)).to(torch.bfloat16).cuda()
    out_tokens = torch.empty(B, K_max + 1, dtype=torch.int32, device="cuda")
    num_acc = torch.empty(B, dtype=torch.int32, device="cuda")
    sd.sd_verify_ragged(to_dev(p), to_dev(q), to_dev(d), to_dev(cu), out_tokens, num_acc,
                        temperature=to_dev(T), seed=17)
    got = run_prepare_ragged(out_tokens, num_acc, cu, pos0, table, bs, 10**6, hid, hs)
    ver = oracle.verify_ragged(p, q, d, cu, K_max, temperature=T, seed=17)
    assert np.array_equal(out_tokens.cpu().numpy(), ver["out_tokens"])
    want = oracle.pdraft_expand(ver["out_tokens"], ver["num_accepted"], pos0, table, bs, 10**6,
                                cu=cu)
    for k in KEYS:
        assert np.array_equal(got[k].reshape(-1), want[k].reshape(-1)), k
    tot = int(want["total_out"][0])
    gh, _ = oracle.hidden_gather(tot, want["hidden_map"], bits(hid), bits(hs))
    assert np.array_equal(got["out_hidden"][:tot], gh[:tot])
    assert got["err"] == want["err"] == 0


@pytest.mark.parametrize("B,K_max,V,greedy,temp,kernels", [
    (48, 6, 20011, 0.0, False, 1),   # every request samples: the single launch
    (40, 16, 4099, 0.0, False, 1),   # K_max = SD_K_MAX, counts 0..16
    (48, 6, 20011, 0.3, True, 2),    # greedy requests among them: two kernels
])
def test_one_call_ragged_step(B, K_max, V, greedy, temp, kernels):
    # sd_verify_prepare_ragged writes what sd_verify_ragged then sd_pdraft_prepare_ragged write,
    # byte for byte, and the oracle's ragged verify and rebuild
    rng = np.random.default_rng(300 + B + K_max)
    p, q, d, cu, T = ragged_case(rng, B, K_max, V, greedy_frac=greedy)
    H, bs = 64, 16
    pos0 = rng.integers(0, 2000, B).astype(np.int32)
    width = (int(pos0.max()) + 2 * K_max) // bs + 1
    table = rng.permutation(B * width).astype(np.int32).reshape(B, width)
    hid = torch.from_numpy(rng.standard_normal((int(cu[-1]) + B, H)).astype(np.float32)).to(
        torch.bfloat16).cuda()
    hs = torch.from_numpy(rng.standard_normal(H).astype(np.float32)).to(torch.bfloat16).cuda()
    Tt = to_dev(T) if temp else None
    assert sd.sd_verify_prepare_kernels(B, K_max, V, sd.SD_F32_PROBS, temp) == kernels
    cap = B * 2 * K_max

    def outs():
        fill = lambda shape, v, dt=torch.int32: torch.full(shape, v, dtype=dt, device="cuda")  # noqa
        return dict(out_tokens=fill((B, K_max + 1), 77), num_accepted=fill((B,), 77),
                    p_at=fill((B, K_max), 77.0, torch.float32),
                    q_at=fill((B, K_max), 77.0, torch.float32),
                    input_ids=fill((cap,), 77), positions=fill((cap,), 77),
                    slot_mapping=fill((cap,), 77), hidden_map=fill((cap,), 77),
                    is_masked=fill((cap,), 7, torch.uint8),
                    is_rejected=fill((B, K_max + 1), 7, torch.uint8),
                    start_loc=fill((B + 1,), 77), new_token_idx=fill((B, K_max), 77),
                    total_out=fill((1,), 77),
                    out_hidden=torch.zeros(cap, H, dtype=torch.bfloat16, device="cuda"),
                    err=fill((1,), 0))

    a, b = outs(), outs()
    args = (to_dev(p), to_dev(q), to_dev(d), to_dev(cu))
    sd.sd_verify_ragged(*args, a["out_tokens"], a["num_accepted"], temperature=Tt, seed=23,
                        p_at_draft=a["p_at"], q_at_draft=a["q_at"], err=a["err"])
    sd.sd_pdraft_prepare_ragged(a["out_tokens"], a["num_accepted"], args[3], _i32(pos0),
                                _i32(table), bs, 10**6, a["input_ids"], a["positions"],
                                a["slot_mapping"], a["hidden_map"], a["is_masked"],
                                a["is_rejected"], a["start_loc"], a["new_token_idx"],
                                a["total_out"], hid, hs, a["out_hidden"], err=a["err"])
    ws = torch.zeros(sd.load().sd_verify_prepare_workspace_bytes(B), dtype=torch.uint8,
                     device="cuda")
    sd.sd_verify_prepare_ragged(*args, b["out_tokens"], b["num_accepted"], _i32(pos0),
                                _i32(table), bs, 10**6, b["input_ids"], b["positions"],
                                b["slot_mapping"], b["hidden_map"], b["is_masked"],
                                b["is_rejected"], b["start_loc"], b["new_token_idx"],
                                b["total_out"], hid, hs, b["out_hidden"], temperature=Tt,
                                seed=23, p_at_draft=b["p_at"], q_at_draft=b["q_at"],
                                err=b["err"], workspace_buf=ws)
    torch.cuda.synchronize()
    for k in a:
        x, y = a[k], b[k]
        if x.dtype == torch.bfloat16:
            x, y = x.view(torch.int16), y.view(torch.int16)
        assert torch.equal(x, y), k
    assert int(ws.count_nonzero()) == 0 and int(b["err"].item()) == 0
    ver = oracle.verify_ragged(p, q, d, cu, K_max, temperature=T if temp else None, seed=23)
    assert np.array_equal(b["out_tokens"].cpu().numpy(), ver["out_tokens"])
    want = oracle.pdraft_expand(ver["out_tokens"], ver["num_accepted"], pos0, table, bs, 10**6,
                                cu=cu)
    for k in KEYS:
        assert np.array_equal(b[k].cpu().numpy().reshape(-1), want[k].reshape(-1)), k
