"""The N > 1 path on the host: two gloo ranks on CPU split one batch by request.

Each rank verifies its contiguous shard with the Philox request index offset by its shard start
(the request_base argument of sd_verify), then rebuilds its own draft batch. Gathered in rank
order, the shards must reproduce the one-rank run of the whole batch exactly: the verify outputs
bit for bit, and the rebuild after shifting each shard's row indices by the rows and hidden-state
rows of the shards before it. The oracle stands in for the device kernels (no GPU here); the
sharding arithmetic, the all-gather of shard sizes and the max-over-ranks timing are the library's
own host code. Ragged shards (sizes not fixed in advance) take their request_base from the
all-gather."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from devrun import random_probs_case
from verify_draft_prep_gb300 import shard

B, K, V, BLOCK = 7, 3, 64, 16
SEED = 0xC0FFEE


def _case():
    rng = np.random.default_rng(123)
    t, d, drafts, temp = random_probs_case(rng, B, K, V, greedy_frac=0.3)
    t3 = t.reshape(B, K + 1, V)
    d3 = d.reshape(B, K, V)
    pos0 = rng.integers(20, 200, B).astype(np.int32)
    need = (pos0 + 2 * K) // BLOCK + 1
    table = np.full((B, int(need.max())), -1, np.int32)
    perm = rng.permutation(int(need.sum())).astype(np.int32)
    o = 0
    for r in range(B):
        table[r, :need[r]] = perm[o:o + need[r]]
        o += need[r]
    return t3, d3, drafts, temp, pos0, table


def _run(t3, d3, drafts, temp, pos0, table, base):
    n = drafts.shape[0]
    ver = oracle.verify_probs(t3, d3, drafts, temperature=temp, seed=SEED,
                              req_ids=np.arange(base, base + n, dtype=np.int32))
    exp = oracle.pdraft_expand(ver["out_tokens"], ver["num_accepted"], pos0, table, BLOCK, V)
    return ver, exp


def _gather_rows(x, world):
    """All-gather a variable-length int64 array, concatenated in rank order."""
    x = torch.as_tensor(np.ascontiguousarray(x), dtype=torch.int64).reshape(-1)
    n = torch.tensor([x.numel()], dtype=torch.int64)
    ns = [torch.zeros_like(n) for _ in range(world)]
    dist.all_gather(ns, n)
    m = max(int(v.item()) for v in ns)
    pad = torch.zeros(m, dtype=torch.int64)
    pad[:x.numel()] = x
    got = [torch.zeros_like(pad) for _ in range(world)]
    dist.all_gather(got, pad)
    return np.concatenate([g[:int(c.item())].numpy() for g, c in zip(got, ns)])


def _worker(rank, world, port, ragged):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t3, d3, drafts, temp, pos0, table = _case()
        if ragged:  # sizes chosen by the caller, not by shard_bounds: the bases come from counts
            counts = [2, B - 2]
            start = sum(counts[:rank])
            count = counts[rank]
            base, total = shard.request_base(count)
            assert (base, total) == (start, B)
        else:
            start, count = shard.shard_bounds(B, world, rank)
            base = start
        sl = slice(start, start + count)
        ver, exp = _run(t3[sl], d3[sl], drafts[sl], temp[sl], pos0[sl], table[sl], base)
        tot = int(exp["total_out"][0])
        # rows and target hidden-state rows held by the ranks before this one
        rows_before = shard.request_base(tot)[0]
        hidden_before = base * (K + 1)
        hm = exp["hidden_map"][:tot].astype(np.int64)
        hm[hm >= 0] += hidden_before
        g = {k: _gather_rows(ver[k], world) for k in ("out_tokens", "num_accepted")}
        g["p_at_draft"] = _gather_rows(ver["p_at_draft"].view(np.int32), world)
        for k in ("input_ids", "positions", "slot_mapping", "is_masked"):
            g[k] = _gather_rows(exp[k][:tot], world)
        g["hidden_map"] = _gather_rows(hm, world)
        g["start_loc"] = _gather_rows(exp["start_loc"][:-1].astype(np.int64) + rows_before, world)
        g["total"] = _gather_rows(np.array([tot]), world).sum()
        # whole-job timing: every rank reports its own duration, the job takes the maximum
        t = torch.tensor([10.0 + rank])
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        rate = shard.whole_job_rate(count, world, float(t.item()))
        if rank == 0:
            ver1, exp1 = _run(t3, d3, drafts, temp, pos0, table, 0)
            tot1 = int(exp1["total_out"][0])
            assert np.array_equal(g["out_tokens"], ver1["out_tokens"].reshape(-1))
            assert np.array_equal(g["num_accepted"], ver1["num_accepted"])
            assert np.array_equal(g["p_at_draft"], ver1["p_at_draft"].view(np.int32).reshape(-1))
            assert g["total"] == tot1
            for k in ("input_ids", "positions", "slot_mapping", "is_masked", "hidden_map"):
                assert np.array_equal(g[k], exp1[k][:tot1]), k
            assert np.array_equal(g["start_loc"], exp1["start_loc"][:-1])
            assert float(t.item()) == 10.0 + world - 1
            assert rate == pytest.approx(world * count / ((10.0 + world - 1) / 1e3))
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("ragged", [False, True])
def test_two_rank_shards_reproduce_one_rank(ragged):
    oracle.build()
    mp.spawn(_worker, args=(2, _free_port(), ragged), nprocs=2, join=True)


def test_shard_bounds_cover_the_batch():
    for batch in (0, 1, 7, 64, 1023):
        for world in (1, 2, 3, 8):
            spans = [shard.shard_bounds(batch, world, r) for r in range(world)]
            assert spans[0][0] == 0
            assert all(a[0] + a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert sum(c for _, c in spans) == batch
            assert max(c for _, c in spans) - min(c for _, c in spans) <= 1
    with pytest.raises(ValueError):
        shard.shard_bounds(4, 2, 2)


def test_request_base_without_a_process_group():
    assert shard.request_base(5) == (0, 5)
