"""Pins for the draft-batch rebuild and the hidden-state gather (P-EAGLE blog, sections
"核心方法", "并行草稿生成的挑战", "Triton Kernel", "Hidden State 管理").

Expand: a hand-worked three-request example (tests/golden/expand_hand_example.json), start
indices against torch.cumsum, and the error paths. Gather: against the page's own formulation --
scatter the target rows to their drafter slots, then torch.where(mask, h_shared, hidden) --
byte for byte.
"""

import json

import numpy as np
import torch

import oracle
from conftest import golden_path


def test_expand_hand_example():
    g = json.load(open(golden_path("expand_hand_example.json")))
    o = oracle.pdraft_expand(g["out_tokens"], g["num_accepted"], g["pos0"], g["block_table"],
                             g["block_size"], g["mask_token_id"])
    exp = g["expected"]
    assert o["err"] == 0
    assert int(o["total_out"][0]) == exp["total_out"]
    for k in ("start_loc", "input_ids", "positions", "slot_mapping", "hidden_map", "is_masked",
              "is_rejected", "new_token_idx"):
        assert np.array_equal(o[k], np.array(exp[k])), k


def _random_expand_inputs(rng, B, K, bs=16):
    a = rng.integers(0, K + 1, B).astype(np.int32)
    out_tokens = np.full((B, K + 1), -1, np.int32)
    for r in range(B):
        out_tokens[r, : a[r] + 1] = rng.integers(0, 1000, a[r] + 1)
    pos0 = rng.integers(0, 300, B).astype(np.int32)
    need = (pos0 + 2 * K) // bs + 1
    width = int(need.max())
    perm = rng.permutation(int(need.sum())).astype(np.int32)
    table = np.full((B, width), -1, np.int32)
    off = 0
    for r in range(B):
        table[r, : need[r]] = perm[off: off + need[r]]
        off += need[r]
    return out_tokens, a, pos0, table


def test_expand_start_loc_is_exclusive_cumsum_and_rows_are_consistent():
    rng = np.random.default_rng(13)
    for B, K in [(1, 1), (7, 3), (64, 5), (33, 8), (5, 16)]:
        out_tokens, a, pos0, table = _random_expand_inputs(rng, B, K)
        o = oracle.pdraft_expand(out_tokens, a, pos0, table, 16, 4242)
        L = torch.from_numpy(a.astype(np.int64) + K)
        want = torch.cat([torch.zeros(1, dtype=torch.int64), torch.cumsum(L, 0)]).numpy()
        assert np.array_equal(o["start_loc"], want)
        assert o["total_out"][0] == want[-1]
        assert o["err"] == 0
        # every drafter slot maps to a KV slot inside its request's own blocks
        for r in range(B):
            s = o["start_loc"][r]
            slots = o["slot_mapping"][s: s + a[r] + K]
            blocks = set((table[r][table[r] >= 0]).tolist())
            assert all(int(x) // 16 in blocks for x in slots)
            assert len(set(slots.tolist())) == len(slots)  # no two slots collide
            assert np.all(o["hidden_map"][s: s + a[r] + 1] == r * (K + 1) + np.arange(a[r] + 1))
            assert np.all(o["input_ids"][s + a[r] + 1: s + a[r] + K] == 4242)


def test_expand_error_paths():
    K = 2
    out_tokens = np.array([[1, 2, -1], [3, -1, -1]], np.int32)
    pos0 = np.array([14, 5], np.int32)
    table = np.array([[4, -1], [6, -1]], np.int32)  # request 0 needs block 1 (positions 16+)
    o = oracle.pdraft_expand(out_tokens, [1, 0], pos0, table, 16, 99)
    assert o["err"] & oracle.ERR_BLOCK_TABLE
    s = o["slot_mapping"][:3]
    assert list(s) == [4 * 16 + 15, -1, -1]
    o = oracle.pdraft_expand(out_tokens, [5, 0], pos0, table, 16, 99)
    assert o["err"] & oracle.ERR_NUM_ACCEPTED  # clamped to K
    o = oracle.pdraft_expand(np.zeros((0, 3), np.int32), np.zeros(0, np.int32),
                             np.zeros(0, np.int32), np.zeros((0, 1), np.int32), 16, 99)
    assert o["total_out"][0] == 0 and list(o["start_loc"]) == [0]


def test_gather_matches_page_scatter_where():
    rng = np.random.default_rng(14)
    B, K, H = 9, 4, 40
    out_tokens, a, pos0, table = _random_expand_inputs(rng, B, K)
    e = oracle.pdraft_expand(out_tokens, a, pos0, table, 16, 7)
    total = int(e["total_out"][0])
    cap = B * 2 * K
    target = torch.randn(B * (K + 1), H).to(torch.bfloat16)
    h_shared = torch.randn(H).to(torch.bfloat16)
    tbits = target.view(torch.int16).numpy().view(np.uint16)
    hbits = h_shared.view(torch.int16).numpy().view(np.uint16)
    sentinel = np.full((cap, H), 0xABCD, np.uint16)
    got, err = oracle.hidden_gather(total, e["hidden_map"], tbits, hbits, out_init=sentinel)
    assert err == 0
    # the page's form: scatter target rows to their drafter slots, then where(mask, h_shared, .)
    hidden = torch.from_numpy(sentinel.view(np.int16).copy()).view(torch.bfloat16)
    m = torch.from_numpy(e["hidden_map"][:total].astype(np.int64))
    dest = torch.nonzero(m >= 0).squeeze(1)
    out_hidden_state_mapping = torch.full((B * (K + 1),), -1, dtype=torch.int64)
    out_hidden_state_mapping[m[dest]] = dest
    src_rows = torch.nonzero(out_hidden_state_mapping >= 0).squeeze(1)
    hidden[out_hidden_state_mapping[src_rows]] = target[src_rows]
    mask = torch.from_numpy(e["is_masked"][:total].astype(bool))
    hidden[:total] = torch.where(mask.unsqueeze(1), h_shared, hidden[:total])
    want = hidden.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    assert np.all(got[total:] == 0xABCD)  # rows past total_out untouched


def test_gather_map_out_of_range_flags():
    th = np.arange(12, dtype=np.uint16).reshape(3, 4)
    hs = np.full(4, 9, np.uint16)
    got, err = oracle.hidden_gather(2, np.array([1, 5], np.int32), th, hs)
    assert err & oracle.ERR_MAP_RANGE
    assert list(got[0]) == [4, 5, 6, 7] and list(got[1]) == [9, 9, 9, 9]
