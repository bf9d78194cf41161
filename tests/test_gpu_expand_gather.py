"""GPU parity of sd_pdraft_expand and sd_hidden_gather against the oracle: every output element
bit-exact (ids, positions, slots, maps, masks, start indices, new-token indices, total), every
gathered hidden byte exact, rows past total_out untouched, error bits equal."""

import json

import numpy as np
import pytest
import torch

import oracle
import verify_draft_prep_gb300 as sd
from conftest import golden_path

pytestmark = pytest.mark.gpu

KEYS = ("input_ids", "positions", "slot_mapping", "hidden_map", "is_masked", "is_rejected",
        "start_loc", "new_token_idx", "total_out")


def run_expand(out_tokens, num_acc, pos0, table, bs, mask_id, capacity=None):
    B, K1 = out_tokens.shape
    K = K1 - 1
    cap = B * 2 * K if capacity is None else capacity
    dev = "cuda"
    o = dict(input_ids=torch.full((cap,), 555, dtype=torch.int32, device=dev),
             positions=torch.full((cap,), 555, dtype=torch.int32, device=dev),
             slot_mapping=torch.full((cap,), 555, dtype=torch.int32, device=dev),
             hidden_map=torch.full((cap,), 555, dtype=torch.int32, device=dev),
             is_masked=torch.full((cap,), 9, dtype=torch.uint8, device=dev),
             is_rejected=torch.full((B, K + 1), 9, dtype=torch.uint8, device=dev),
             start_loc=torch.full((B + 1,), 555, dtype=torch.int32, device=dev),
             new_token_idx=torch.full((B, K), 555, dtype=torch.int32, device=dev),
             total_out=torch.full((1,), 555, dtype=torch.int32, device=dev))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a, np.int32)).cuda()  # noqa: E731
    sd.sd_pdraft_expand(t(out_tokens), t(num_acc), t(pos0), t(table), bs, mask_id,
                        o["input_ids"], o["positions"], o["slot_mapping"], o["hidden_map"],
                        o["is_masked"], o["is_rejected"], o["start_loc"], o["new_token_idx"],
                        o["total_out"], err=err)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in o.items()}
    res["err"] = int(err.item())
    return res


def check_expand(got, want):
    for k in KEYS:
        assert np.array_equal(got[k], want[k]), k
    assert got["err"] == want["err"]


def test_hand_example_on_gpu():
    g = json.load(open(golden_path("expand_hand_example.json")))
    got = run_expand(np.array(g["out_tokens"]), g["num_accepted"], g["pos0"],
                     np.array(g["block_table"]), g["block_size"], g["mask_token_id"])
    for k, v in g["expected"].items():
        assert np.array_equal(np.ravel(got[k]), np.ravel(v)), k


def _random(rng, B, K, bs=16):
    a = rng.integers(0, K + 1, B).astype(np.int32)
    out_tokens = np.full((B, K + 1), -1, np.int32)
    for r in range(B):
        out_tokens[r, : a[r] + 1] = rng.integers(0, 200000, a[r] + 1)
    pos0 = rng.integers(0, 32000, B).astype(np.int32)
    need = (pos0 + 2 * K) // bs + 1
    table = np.full((B, int(need.max())), -1, np.int32)
    perm = rng.permutation(int(need.sum())).astype(np.int32)
    off = 0
    for r in range(B):
        table[r, : need[r]] = perm[off: off + need[r]]
        off += need[r]
    return out_tokens, a, pos0, table


@pytest.mark.parametrize("B,K", [(1, 1), (3, 4), (64, 5), (255, 7), (256, 7), (257, 8),
                                 (1024, 8), (3000, 16)])
def test_expand_random_bit_exact(B, K):
    rng = np.random.default_rng(B * 31 + K)
    out_tokens, a, pos0, table = _random(rng, B, K)
    got = run_expand(out_tokens, a, pos0, table, 16, 201088)
    want = oracle.pdraft_expand(out_tokens, a, pos0, table, 16, 201088)
    check_expand(got, want)


def test_expand_errors_and_small_capacity():
    rng = np.random.default_rng(5)
    out_tokens, a, pos0, table = _random(rng, 300, 4)
    a[7] = 9            # out of range: clamped
    a[8] = -2
    table[10, :] = -1   # block-table misses
    pos0[11] = -40      # negative positions
    got = run_expand(out_tokens, a, pos0, table, 16, 5)
    want = oracle.pdraft_expand(out_tokens, a, pos0, table, 16, 5)
    assert want["err"] == (oracle.ERR_NUM_ACCEPTED | oracle.ERR_BLOCK_TABLE)
    check_expand(got, want)
    cap = 1000  # smaller than the total: truncated with an error bit
    got = run_expand(out_tokens, a, pos0, table, 16, 5, capacity=cap)
    want = oracle.pdraft_expand(out_tokens, a, pos0, table, 16, 5, capacity=cap)
    assert want["err"] & oracle.ERR_TOTAL_RANGE
    check_expand(got, want)


def test_expand_empty_batch():
    got = run_expand(np.zeros((0, 3), np.int32), np.zeros(0, np.int32), np.zeros(0, np.int32),
                     np.zeros((0, 1), np.int32), 16, 1, capacity=6)
    assert got["total_out"][0] == 0 and list(got["start_loc"]) == [0]
    assert list(got["input_ids"]) == [-1] * 6 and list(got["slot_mapping"]) == [-1] * 6


def run_gather(total, hmap, target, h_shared, cap, out_init):
    out = out_init.clone().cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sd.sd_hidden_gather(torch.tensor([total], dtype=torch.int32).cuda(),
                        torch.as_tensor(hmap).cuda(), target.cuda(), h_shared.cuda(), out,
                        err=err)
    torch.cuda.synchronize()
    return out.cpu(), int(err.item())


@pytest.mark.parametrize("B,K,H", [(1, 4, 64), (64, 5, 2880), (37, 7, 2048), (9, 3, 100),
                                   (5, 2, 13)])
def test_gather_bit_exact(B, K, H):
    rng = np.random.default_rng(H + B)
    out_tokens, a, pos0, table = _random(rng, B, K)
    e = oracle.pdraft_expand(out_tokens, a, pos0, table, 16, 9)
    total = int(e["total_out"][0])
    cap = B * 2 * K
    target = torch.randn(B * (K + 1), H).to(torch.bfloat16)
    h_shared = torch.randn(H).to(torch.bfloat16)
    init = torch.full((cap, H), 3.0).to(torch.bfloat16)
    got, err = run_gather(total, e["hidden_map"], target, h_shared, cap, init)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    want, werr = oracle.hidden_gather(total, e["hidden_map"], bits(target), bits(h_shared),
                                      out_init=bits(init))
    assert err == werr == 0
    assert np.array_equal(bits(got), want)


def test_gather_strided_and_map_errors():
    H, n_in, cap = 24, 10, 8
    base = torch.randn(n_in, 40).to(torch.bfloat16).cuda()
    target = base[:, 3:3 + H]  # row stride 40, offset 3 elements: scalar path
    h_shared = torch.randn(H).to(torch.bfloat16)
    hmap = np.array([0, 9, -1, 12, 4, -1, 2, 2], np.int32)
    init = torch.zeros(cap, H).to(torch.bfloat16)
    got, err = run_gather(7, hmap, target, h_shared, cap, init)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    want, werr = oracle.hidden_gather(7, hmap, bits(target.cpu()), bits(h_shared),
                                      out_init=bits(init))
    assert err == werr == oracle.ERR_MAP_RANGE
    assert np.array_equal(bits(got), want)


def run_prepare(out_tokens, num_acc, pos0, table, bs, mask_id, target, h_shared, out_init,
                capacity=None, after_verify=False):
    """sd_pdraft_prepare (expand + gather in one launch); returns expand outputs and hidden."""
    B, K1 = out_tokens.shape
    K = K1 - 1
    cap = B * 2 * K if capacity is None else capacity
    dev = "cuda"
    o = dict(input_ids=torch.full((cap,), 555, dtype=torch.int32, device=dev),
             positions=torch.full((cap,), 555, dtype=torch.int32, device=dev),
             slot_mapping=torch.full((cap,), 555, dtype=torch.int32, device=dev),
             hidden_map=torch.full((cap,), 555, dtype=torch.int32, device=dev),
             is_masked=torch.full((cap,), 9, dtype=torch.uint8, device=dev),
             is_rejected=torch.full((B, K + 1), 9, dtype=torch.uint8, device=dev),
             start_loc=torch.full((B + 1,), 555, dtype=torch.int32, device=dev),
             new_token_idx=torch.full((B, K), 555, dtype=torch.int32, device=dev),
             total_out=torch.full((1,), 555, dtype=torch.int32, device=dev))
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = out_init.clone().cuda()
    t = lambda a: torch.as_tensor(np.ascontiguousarray(a, np.int32)).cuda()  # noqa: E731
    sd.sd_pdraft_prepare(t(out_tokens), t(num_acc), t(pos0), t(table), bs, mask_id,
                         o["input_ids"], o["positions"], o["slot_mapping"], o["hidden_map"],
                         o["is_masked"], o["is_rejected"], o["start_loc"], o["new_token_idx"],
                         o["total_out"], target.cuda(), h_shared.cuda(), out, err=err)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in o.items()}
    res["err"] = int(err.item())
    return res, out.cpu()


@pytest.mark.parametrize("B,K,H", [(1, 4, 64), (64, 5, 2880), (256, 7, 2048), (300, 8, 2880),
                                   (1024, 8, 2880), (9, 3, 100), (5, 2, 13), (3000, 16, 64)])
def test_prepare_bit_exact(B, K, H):
    rng = np.random.default_rng(B + 7 * K + H)
    out_tokens, a, pos0, table = _random(rng, B, K)
    cap = B * 2 * K
    target = torch.randn(B * (K + 1), H).to(torch.bfloat16)
    h_shared = torch.randn(H).to(torch.bfloat16)
    init = torch.full((cap, H), 3.0).to(torch.bfloat16)
    got, hid = run_prepare(out_tokens, a, pos0, table, 16, 201088, target, h_shared, init)
    want = oracle.pdraft_expand(out_tokens, a, pos0, table, 16, 201088)
    check_expand(got, want)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    wh, werr = oracle.hidden_gather(int(want["total_out"][0]), want["hidden_map"], bits(target),
                                    bits(h_shared), out_init=bits(init))
    assert werr == 0
    assert np.array_equal(bits(hid), wh)


def test_prepare_errors_and_truncation():
    rng = np.random.default_rng(77)
    B, K, H = 300, 4, 24
    out_tokens, a, pos0, table = _random(rng, B, K)
    a[7] = 9
    table[10, :] = -1
    pos0[11] = -40
    target = torch.randn(B * (K + 1), H).to(torch.bfloat16)
    h_shared = torch.randn(H).to(torch.bfloat16)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    for cap in (B * 2 * K, 1000, 0):
        init = torch.full((cap, H), 3.0).to(torch.bfloat16)
        got, hid = run_prepare(out_tokens, a, pos0, table, 16, 5, target, h_shared, init,
                               capacity=cap)
        want = oracle.pdraft_expand(out_tokens, a, pos0, table, 16, 5, capacity=cap)
        check_expand(got, want)
        wh, _ = oracle.hidden_gather(min(int(want["total_out"][0]), cap), want["hidden_map"],
                                     bits(target), bits(h_shared), capacity=cap,
                                     out_init=bits(init))
        assert np.array_equal(bits(hid), wh)
