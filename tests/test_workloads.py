"""Host-side checks of the seeded synthetic inputs (shapes, structure, determinism)."""

import torch

import workloads


def test_small_workload_shapes_and_structure():
    w = workloads.make("small")
    B, K, V, H = w.B, w.K, w.V, w.H
    assert (B, K, V, H) == (1, 4, 1024, 64)
    assert w.target.shape == (B * (K + 1), V) and w.target.dtype == torch.float32
    assert w.draft.shape == (B * K, V)
    assert torch.allclose(w.target.sum(-1), torch.ones(B * (K + 1)), atol=1e-5)
    assert w.drafts.dtype == torch.int32 and int(w.drafts.max()) < V
    assert int(w.pos0[0]) == 37
    assert w.block_table.shape == (1, 3)  # floor((37 + 8) / 16) + 1 blocks
    assert w.hidden.shape == (B * (K + 1), H) and w.hidden.dtype == torch.bfloat16
    assert w.mask_token_id == V


def test_block_tables_cover_every_drafter_position():
    g = torch.Generator().manual_seed(3)
    pos0 = torch.randint(0, 5000, (40,), generator=g)
    K = 8
    t = workloads.block_tables(pos0, K, 16, g, "cpu")
    need = (pos0 + 2 * K) // 16 + 1
    used = t[t >= 0]
    assert used.numel() == int(need.sum())
    assert torch.equal(torch.sort(used).values, torch.arange(int(need.sum()), dtype=torch.int32))
    for r in range(40):
        assert torch.all(t[r, : need[r]] >= 0) and torch.all(t[r, need[r]:] == -1)


def test_generation_is_deterministic_and_greedy_drafts_are_argmax():
    a = workloads.make("b256mix", B=6)
    b = workloads.make("b256mix", B=6)
    assert torch.equal(a.target, b.target) and torch.equal(a.drafts, b.drafts)
    assert torch.equal(a.temperature, torch.tensor([0.0, 1.0] * 3))
    q = a.draft.view(6, a.K, a.V)
    for r in (0, 2, 4):
        assert torch.equal(a.drafts[r].long(), q[r].argmax(-1))


def test_logits_workload():
    w = workloads.make("b1024lg", B=3)
    assert w.target.dtype == torch.bfloat16 and w.kind == "logits"
    assert torch.all((w.temperature >= 0.5) & (w.temperature <= 1.2))
