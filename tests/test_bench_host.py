"""Host logic of bench.py (no GPU): the algorithmic byte model the roofline divides by, checked
against per-request counts written out for a tiny batch, and the launch-count bookkeeping."""

import numpy as np
import torch

import bench
import workloads


def _tiny(kind="probs", greedy=()):
    w = workloads.make("small", device="cpu", B=4)
    w.kind = kind
    T = torch.ones(w.B)
    for r in greedy:
        T[r] = 0.0
    w.temperature = T
    return w


def test_probability_model_counts_rows_per_request():
    w = _tiny(greedy=(3,))
    K, V, H = w.K, w.V, w.H
    a = np.array([0, 2, K, 1])              # request 3 is greedy
    verify, expand, gather, verify_read = bench.algorithmic_bytes(w, a)
    scalars = 4 * K + 4 * (K + 2) + 4
    want = 0
    for r, ar in enumerate(a):
        if r == 3:                          # greedy: rows 0..a_r of p, no gathers
            want += (ar + 1) * 4 * V + scalars
        else:                               # sampled: 32-byte gathers of P and Q up to the
            rows = 2 if ar < K else 1       # rejection, then p and q (or p alone) once
            want += rows * 4 * V + 2 * 32 * min(ar + 1, K) + scalars
    assert verify == want == verify_read
    # rebuild: accepted hidden rows in, a_r + K drafter rows out, h_shared once
    assert gather == int(((a + 1) * 2 * H + (a + K) * 2 * H).sum()) + 2 * H
    assert expand > 0


def test_logit_model_counts_every_row():
    w = _tiny(kind="logits")
    K, V = w.K, w.V
    a = np.array([0, 1, K, 2])
    verify, _, _, verify_read = bench.algorithmic_bytes(w, a)
    scalars = 4 * K + 4 * (K + 2) + 4
    assert verify == w.B * ((2 * K + 1) * 2 * V + scalars)
    rows_read = (a + 1) + np.minimum(a + 1, K)
    assert verify_read == int((rows_read * 2 * V + scalars).sum())
    assert verify_read < verify


def test_traffic_table_names_known_configs():
    names = {c["name"] for c in workloads.CONFIGS}
    for (cfg, h), (bytes_, note) in bench.MEASURED_TRAFFIC.items():
        assert cfg in names and len(h) == 16 and bytes_ > 0 and "ncu" in note
