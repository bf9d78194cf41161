"""Seeded synthetic inputs for the verify step and the P-EAGLE draft-batch rebuild.

This module is shared by the tests, the benchmark and the smoke check. It generates input data
only (target/draft probability or logit rows, drafts, temperatures, positions, block tables,
hidden states); it holds none of the method's own arithmetic, and it imports neither the oracle
nor the CUDA library.

The five named workloads stand in for the chat and code benchmarks the P-EAGLE blog evaluates on
(MT-Bench, HumanEval, SPEED-Bench; UltraChat sequence lengths), which are not available here:

  small    B=1,    K=4, V=1024,   fp32 probs, sigma 0.5, H=64,   context 37
  b64      B=64,   K=5, V=201088, fp32 probs, sigma 0.5, H=2880, context U[512, 8192]
  b256mix  B=256,  K=7, V=151936, fp32 probs, sigma 0.2, H=2048, context U[1000, 16000],
           even requests greedy (temperature 0, drafts = argmax q), odd requests temperature 1
  b512rag  B=512,  K=8, V=201088, fp32 probs, sigma_r ~ U[0.1, 1.5], H=2880,
           context log-uniform [128, 32000]
  b1024lg  B=1024, K=8, V=201088, bf16 logits, target N(0, 2^2), draft = target + N(0, 0.5^2),
           temperature_r ~ U[0.5, 1.2], H=2880, context U[2000, 10800]

Probability rows: per request and row, logits l ~ N(0, 2^2); p_j = softmax(l_j); the draft rows
are q_j = softmax(l_j + N(0, sigma^2)); drafts d_{j+1} ~ q_j. Block size 16; request r needs
floor((pos0_r + 2K) / 16) + 1 blocks, whose physical ids are consecutive slices of one random
permutation; unused table entries are -1. MASK id = V. Philox seed 0.
"""

from __future__ import annotations

import dataclasses
import math

import torch

BLOCK_SIZE = 16

CONFIGS = [
    dict(name="small", B=1, K=4, V=1024, H=64, kind="probs", sigma=0.5, ctx=("fixed", 37)),
    dict(name="b64", B=64, K=5, V=201088, H=2880, kind="probs", sigma=0.5, ctx=("uniform", 512, 8192)),
    dict(name="b256mix", B=256, K=7, V=151936, H=2048, kind="probs", sigma=0.2,
         ctx=("uniform", 1000, 16000), greedy="even"),
    dict(name="b512rag", B=512, K=8, V=201088, H=2880, kind="probs", sigma=("uniform", 0.1, 1.5),
         ctx=("loguniform", 128, 32000)),
    dict(name="b1024lg", B=1024, K=8, V=201088, H=2880, kind="logits", sigma=0.5,
         temp=("uniform", 0.5, 1.2), ctx=("uniform", 2000, 10800)),
]


def config_label(cfg: dict) -> str:
    kind = "fp32 probs" if cfg["kind"] == "probs" else "bf16 logits"
    return f"{cfg['name']}: B={cfg['B']} K={cfg['K']} V={cfg['V']} {kind} H={cfg['H']}"


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    K: int
    V: int
    H: int
    kind: str                    # "probs" (fp32) or "logits" (bf16)
    target: torch.Tensor         # [B*(K+1), V] rows p_0..p_K of each request
    draft: torch.Tensor          # [B*K, V] rows q_0..q_{K-1}
    drafts: torch.Tensor         # [B, K] int32, d_1..d_K
    temperature: torch.Tensor    # [B] float32
    pos0: torch.Tensor           # [B] int32, position of verify slot 0
    block_table: torch.Tensor    # [B, max_blocks] int32, -1 where unused
    block_size: int
    hidden: torch.Tensor         # [B*(K+1), H] bf16 target hidden states
    h_shared: torch.Tensor       # [H] bf16
    mask_token_id: int
    seed: int

    @property
    def capacity(self) -> int:
        return self.B * 2 * self.K


def _draw(spec, n, gen, device):
    if isinstance(spec, (int, float)):
        return torch.full((n,), float(spec), device=device)
    kind = spec[0]
    u = torch.rand(n, generator=gen, device=device, dtype=torch.float64)
    if kind == "uniform":
        return spec[1] + (spec[2] - spec[1]) * u
    if kind == "loguniform":
        return torch.exp(math.log(spec[1]) + (math.log(spec[2]) - math.log(spec[1])) * u)
    raise ValueError(spec)


def _contexts(spec, B, gen, device):
    if spec[0] == "fixed":
        return torch.full((B,), spec[1], dtype=torch.int64, device=device)
    return torch.floor(_draw(spec, B, gen, device)).to(torch.int64)


def block_tables(pos0: torch.Tensor, K: int, block_size: int, gen, device):
    """Shuffled paged-KV block tables covering positions up to pos0 + 2K."""
    need = (pos0 + 2 * K) // block_size + 1
    total = int(need.sum())
    perm = torch.randperm(total, generator=gen, device=device).to(torch.int32)
    width = int(need.max())
    B = pos0.shape[0]
    table = torch.full((B, width), -1, dtype=torch.int32, device=device)
    col = torch.arange(width, device=device).unsqueeze(0)
    mask = col < need.unsqueeze(1)
    table[mask] = perm
    return table


def make_probs_rows(B, K, V, sigma, gen, device, greedy_mask=None, chunk=32):
    """fp32 probability rows: target [B*(K+1), V], draft [B*K, V], drafts [B, K]."""
    target = torch.empty(B * (K + 1), V, dtype=torch.float32, device=device)
    draft = torch.empty(B * K, V, dtype=torch.float32, device=device)
    drafts = torch.empty(B, K, dtype=torch.int32, device=device)
    for r0 in range(0, B, chunk):
        r1 = min(B, r0 + chunk)
        n = r1 - r0
        l = 2.0 * torch.randn(n, K + 1, V, generator=gen, device=device)
        s = sigma[r0:r1].to(torch.float32).view(n, 1, 1)
        ld = l[:, :K] + s * torch.randn(n, K, V, generator=gen, device=device)
        target[r0 * (K + 1):r1 * (K + 1)] = torch.softmax(l, dim=-1).view(n * (K + 1), V)
        q = torch.softmax(ld, dim=-1).view(n * K, V)
        draft[r0 * K:r1 * K] = q
        d = torch.multinomial(q, 1, generator=gen).view(n, K)
        if greedy_mask is not None:
            g = greedy_mask[r0:r1]
            if bool(g.any()):
                d[g] = q.view(n, K, V).argmax(dim=-1)[g]
        drafts[r0:r1] = d.to(torch.int32)
        del l, ld, q
    return target, draft, drafts


def make_logit_rows(B, K, V, sigma, temperature, gen, device, chunk=32):
    """bf16 logit rows: target [B*(K+1), V], draft [B*K, V]; drafts ~ softmax(l^d / T)."""
    target = torch.empty(B * (K + 1), V, dtype=torch.bfloat16, device=device)
    draft = torch.empty(B * K, V, dtype=torch.bfloat16, device=device)
    drafts = torch.empty(B, K, dtype=torch.int32, device=device)
    for r0 in range(0, B, chunk):
        r1 = min(B, r0 + chunk)
        n = r1 - r0
        lt = (2.0 * torch.randn(n, K + 1, V, generator=gen, device=device)).to(torch.bfloat16)
        ld = (lt[:, :K].float() + sigma * torch.randn(n, K, V, generator=gen, device=device)
              ).to(torch.bfloat16)
        target[r0 * (K + 1):r1 * (K + 1)] = lt.view(n * (K + 1), V)
        draft[r0 * K:r1 * K] = ld.view(n * K, V)
        T = temperature[r0:r1].view(n, 1, 1)
        q = torch.softmax(ld.float() / T, dim=-1).view(n * K, V)
        drafts[r0:r1] = torch.multinomial(q, 1, generator=gen).view(n, K).to(torch.int32)
        del lt, ld, q
    return target, draft, drafts


def make(index_or_name, device="cpu", B: int | None = None, seed: int = 0,
         gen_seed: int | None = None) -> Workload:
    """Build a named workload. ``B`` overrides the batch size (for small test versions)."""
    if isinstance(index_or_name, str):
        idx = [c["name"] for c in CONFIGS].index(index_or_name)
    else:
        idx = int(index_or_name)
    cfg = CONFIGS[idx]
    B = cfg["B"] if B is None else B
    K, V, H = cfg["K"], cfg["V"], cfg["H"]
    gen = torch.Generator(device=device)
    gen.manual_seed(1000 + idx if gen_seed is None else gen_seed)
    ctx = _contexts(cfg["ctx"], B, gen, device)
    temp_spec = cfg.get("temp", 1.0)
    temperature = _draw(temp_spec, B, gen, device).to(torch.float32)
    greedy_mask = None
    if cfg.get("greedy") == "even":
        greedy_mask = (torch.arange(B, device=device) % 2) == 0
        temperature[greedy_mask] = 0.0
    sigma = _draw(cfg["sigma"], B, gen, device)
    if cfg["kind"] == "probs":
        target, draft, drafts = make_probs_rows(B, K, V, sigma, gen, device, greedy_mask)
    else:
        target, draft, drafts = make_logit_rows(B, K, V, cfg["sigma"], temperature, gen, device)
    pos0 = ctx.to(torch.int32)
    table = block_tables(ctx, K, BLOCK_SIZE, gen, device)
    hidden = torch.randn(B * (K + 1), H, generator=gen, device=device).to(torch.bfloat16)
    h_shared = torch.randn(H, generator=gen, device=device).to(torch.bfloat16)
    return Workload(name=cfg["name"], B=B, K=K, V=V, H=H, kind=cfg["kind"], target=target,
                    draft=draft, drafts=drafts, temperature=temperature, pos0=pos0,
                    block_table=table, block_size=BLOCK_SIZE, hidden=hidden, h_shared=h_shared,
                    mask_token_id=V, seed=seed)


def bf16_bits(t: torch.Tensor):
    """The raw 16-bit patterns of a bf16 tensor, as a numpy uint16 array (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
