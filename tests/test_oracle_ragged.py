"""Pins of the oracle's per-request draft counts (sd_verify_ragged's definition: each request is
verified on its own with K = K_r; K_r = 0 samples the bonus token from p_0 alone).

The ragged composition reuses the pinned batch oracle, so these pin what it adds: the packing of
the rows (a uniform count must give the batch oracle's results), the request index each request
keeps in the Philox counters, and the K_r = 0 case against the single-row race.
"""

import numpy as np

import oracle
from devrun import random_probs_case


def _pack(p, q, d, B, K):
    V = p.shape[-1]
    return (p.reshape(B * (K + 1), V), q.reshape(B * K, V), d.reshape(B * K),
            np.arange(B + 1, dtype=np.int32) * K)


def test_uniform_counts_reproduce_the_batch():
    rng = np.random.default_rng(8)
    B, K, V = 9, 4, 300
    p, q, d, T = random_probs_case(rng, B, K, V, greedy_frac=0.3)
    tp, tq, td, cu = _pack(p, q, d, B, K)
    rag = oracle.verify_ragged(tp, tq, td, cu, K, temperature=T, seed=5)
    full = oracle.verify_probs(p.reshape(B, K + 1, V), q.reshape(B, K, V), d, temperature=T,
                               seed=5)
    for k in ("out_tokens", "num_accepted", "p_at_draft", "q_at_draft"):
        assert np.array_equal(rag[k], full[k]), k
    assert rag["err"] == full["err"]


def test_mixed_counts_keep_each_request_index():
    rng = np.random.default_rng(9)
    B, K_max, V = 12, 5, 200
    ks = rng.integers(0, K_max + 1, B)
    cu = np.concatenate([[0], np.cumsum(ks)]).astype(np.int32)
    tp = rng.random((int(cu[-1]) + B, V)).astype(np.float32)
    tq = rng.random((int(cu[-1]), V)).astype(np.float32)
    td = rng.integers(0, V, int(cu[-1])).astype(np.int32)
    rag = oracle.verify_ragged(tp, tq, td, cu, K_max, seed=3)
    for r in range(B):
        k = int(ks[r])
        t = tp[cu[r] + r: cu[r] + r + k + 1][None]
        res = oracle.verify_probs(t, tq[cu[r]: cu[r] + k][None].reshape(1, k, V),
                                  td[cu[r]: cu[r] + k][None].reshape(1, k), seed=3,
                                  req_ids=np.array([r], np.int32))
        assert np.array_equal(rag["out_tokens"][r, :k + 1], res["out_tokens"][0]), r
        assert np.all(rag["out_tokens"][r, k + 1:] == -1)
        assert rag["num_accepted"][r] == res["num_accepted"][0]


def test_zero_drafts_sample_the_bonus_from_p0():
    rng = np.random.default_rng(10)
    V = 64
    p0 = rng.random((3, V)).astype(np.float32)
    cu = np.zeros(4, np.int32)                           # three requests, no drafts
    rag = oracle.verify_ragged(p0, np.zeros((0, V), np.float32), np.zeros(0, np.int32), cu, 2,
                               seed=44)
    for r in range(3):
        x, _ = oracle.race_row(p0[r], None, seed=44, r=r, j=0)
        assert rag["out_tokens"][r, 0] == x and rag["num_accepted"][r] == 0
        assert list(rag["out_tokens"][r, 1:]) == [-1, -1]


def test_rebuild_with_per_request_counts_hand_example():
    import json

    from conftest import golden_path

    g = json.load(open(golden_path("expand_ragged_hand_example.json")))
    o = oracle.pdraft_expand(np.array(g["out_tokens"]), np.array(g["num_accepted"]),
                             np.array(g["pos0"]), np.array(g["block_table"]), g["block_size"],
                             g["mask_token_id"], cu=np.array(g["cu_drafts"]))
    for k, v in g["expected"].items():
        assert np.array_equal(np.ravel(o[k]), np.ravel(v)), k
    assert o["err"] == 0


def test_rebuild_uniform_counts_reproduce_the_batch_layout():
    rng = np.random.default_rng(12)
    B, K, bs = 20, 4, 16
    a = rng.integers(0, K + 1, B).astype(np.int32)
    toks = rng.integers(0, 500, (B, K + 1)).astype(np.int32)
    pos0 = rng.integers(0, 300, B).astype(np.int32)
    width = (int(pos0.max()) + 2 * K) // bs + 1
    table = rng.permutation(B * width).astype(np.int32).reshape(B, width)
    full = oracle.pdraft_expand(toks, a, pos0, table, bs, 500)
    rag = oracle.pdraft_expand(toks, a, pos0, table, bs, 500,
                               cu=np.arange(B + 1, dtype=np.int32) * K)
    for k in ("input_ids", "positions", "slot_mapping", "hidden_map", "is_masked",
              "is_rejected", "start_loc", "new_token_idx", "total_out"):
        assert np.array_equal(full[k], rag[k]), k


def test_rebuild_count_out_of_range_is_clamped_and_flagged():
    toks = np.array([[5, 6, 7], [8, 9, 10]], np.int32)
    o = oracle.pdraft_expand(toks, np.array([1, 0], np.int32), np.array([0, 0], np.int32),
                             np.array([[0, 1], [2, 3]], np.int32), 16, 99,
                             cu=np.array([0, 5, 5], np.int32))  # request 0 claims 5 > K = 2
    assert o["err"] & oracle.ERR_DRAFT_COUNT
    assert int(o["total_out"][0]) == (1 + 2) + (0 + 0)
