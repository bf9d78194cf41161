"""Pins of the oracle's padded drafter batch (reading R14 of the P-EAGLE blog's rebuild: fixed rows
of 2K slots per request, rejected leftovers on PADDING_SLOT_ID = -1, scatter-form hidden map).

A hand-worked example (tests/golden/padded_hand_example.json), then invariants against the
packed layout's own oracle function: the live slots of each padded row are exactly that
request's packed slots, the padding count is K - a_r, and the scatter map and the gather map
describe the same hidden-state copies.
"""

import json

import numpy as np

import oracle
from conftest import golden_path


def _bits(rng, shape):
    return rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)


def test_hand_example():
    g = json.load(open(golden_path("padded_hand_example.json")))
    B, K = len(g["num_accepted"]), g["K"]
    rng = np.random.default_rng(0)
    H = 4
    th = _bits(rng, (B * (K + 1), H))
    hs = _bits(rng, (H,))
    o = oracle.pdraft_prepare_padded(np.array(g["out_tokens"]), np.array(g["num_accepted"]),
                                     np.array(g["pos0"]), np.array(g["block_table"]),
                                     g["block_size"], g["mask_token_id"], th, hs)
    for k, v in g["expected"].items():
        assert np.array_equal(o[k].reshape(-1), np.array(v).reshape(-1)), k
    assert o["err"] == 0
    for i, m in enumerate(g["expected"]["hidden_map"]):
        assert np.array_equal(o["out_hidden"][i], th[m] if m >= 0 else hs), i


def test_live_slots_are_the_packed_layout():
    rng = np.random.default_rng(3)
    B, K, bs = 40, 5, 16
    a = rng.integers(0, K + 1, B).astype(np.int32)
    toks = rng.integers(0, 1000, (B, K + 1)).astype(np.int32)
    pos0 = rng.integers(0, 500, B).astype(np.int32)
    width = (int(pos0.max()) + 2 * K) // bs + 1
    table = rng.permutation(B * width).astype(np.int32).reshape(B, width)
    H = 8
    th = _bits(rng, (B * (K + 1), H))
    hs = _bits(rng, (H,))
    pad = oracle.pdraft_prepare_padded(toks, a, pos0, table, bs, 1000, th, hs)
    pk = oracle.pdraft_expand(toks, a, pos0, table, bs, 1000)
    W = 2 * K
    for r in range(B):
        L = int(a[r]) + K
        s0 = int(pk["start_loc"][r])
        for key in ("input_ids", "positions", "slot_mapping", "hidden_map", "is_masked"):
            assert np.array_equal(pad[key][r * W:r * W + L], pk[key][s0:s0 + L]), (r, key)
        assert pad["rejected"][r * W:(r + 1) * W].sum() == K - a[r]
        assert np.all(pad["slot_mapping"][r * W + L:(r + 1) * W] == -1)
        assert np.array_equal(pad["new_token_idx"][r] - r * W,
                              pk["new_token_idx"][r] - s0)
    # scatter and gather describe the same copies
    for t in range(B * (K + 1)):
        d = pad["scatter_map"][t]
        if d >= 0:
            assert pad["hidden_map"][d] == t
            assert np.array_equal(pad["out_hidden"][d], th[t])
    gathered = pad["hidden_map"] >= 0
    assert gathered.sum() == (pad["scatter_map"] >= 0).sum()
    assert np.all(pad["out_hidden"][~gathered] == hs)
    assert pad["err"] == 0


def test_errors_clamp_and_flag():
    rng = np.random.default_rng(4)
    B, K = 2, 2
    toks = np.array([[5, 6, 7], [8, 9, 10]], np.int32)
    a = np.array([3, -1], np.int32)             # outside [0, K]: clamped, flagged
    pos0 = np.array([0, 100], np.int32)
    table = np.array([[0, 1], [2, 3]], np.int32)  # request 1's positions are past its table
    th = _bits(rng, (B * (K + 1), 2))
    hs = _bits(rng, (2,))
    o = oracle.pdraft_prepare_padded(toks, a, pos0, table, 16, 99, th, hs)
    assert o["err"] & oracle.ERR_NUM_ACCEPTED and o["err"] & oracle.ERR_BLOCK_TABLE
    assert list(o["input_ids"][:4]) == [5, 6, 7, 99]     # a clamped to K = 2
    assert list(o["input_ids"][4:]) == [8, 99, 99, 99]   # a clamped to 0
    assert list(o["slot_mapping"][4:]) == [-1, -1, -1, -1]
