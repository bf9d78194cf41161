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


def test_oracle_samples_hold_the_requests_they_count():
    # a timed oracle pass over a prefix of the batch must verify exactly the requests it counts
    w = workloads.make("small", device="cpu", B=12)
    hc = bench.host_copy(w)
    s = bench.first_requests(hc, 5)
    assert s["B"] == 5
    for k in ("target", "draft", "drafts", "temperature", "pos0", "block_table"):
        assert s[k].shape[0] == 5, k
    assert s["hidden"].shape[0] == 5 * (w.K + 1)
    # a prefix of a prefix is taken from the whole batch's arrays, not a stale sample
    s2 = bench.first_requests(hc, 9)
    assert s2["target"].shape[0] == 9 and np.array_equal(s2["target"][:5], s["target"])
    v, passes, el = bench.oracle_rate(s, 1, 0.01)
    assert passes >= 1 and abs(v - 5 * passes / el) <= 1e-9 * v
    sz = bench.sized_sample(hc, 2, 0.05)
    assert 1 <= sz["B"] <= 12 and sz["target"].shape[0] == sz["B"]


def test_reference_arm_prints_the_timed_arms_config(capsys):
    import argparse
    import json

    args = argparse.Namespace(config="small", steps=2, warmup=1, sets=0, batch=0)
    bench.run_reference(args, 1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    cfg = [c for c in workloads.CONFIGS if c["name"] == "small"][0]
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "requests/s"
    assert line["config"]["workload"] == bench.config_dict(cfg, 1, 4, 0.0, 1, 0)["workload"]
    assert set(line["config"]) == set(bench.config_dict(cfg, 1, 4, 0.0, 1, 0))
    assert line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1


def test_philox_peak_from_unit_counts():
    # 152 SMs x clock x 64 multiply lanes, 40 lane operations (20 64-bit products) per block
    assert abs(bench.philox_peak() - 152 * 2070e6 * 64 / 40) / bench.philox_peak() < 0.05


def test_sampler_roofline_binds_on_the_longer_bound():
    import types
    peak = 6753.8
    # bf16 rows of 2e5 entries: one Philox block per 4 entries outweighs 2 bytes per entry
    w = types.SimpleNamespace(B=1024, K=8, V=201088)
    by = w.B * w.K * w.V * 2
    r = bench.sample_roofline(w, 1.2, by, peak)
    assert r["bound"] == "alu" and r["frac"] == r["alu"]["frac"]
    blocks = w.B * w.K * ((w.V + 3) // 4)
    assert r["alu"]["philox_blocks_per_launch"] == blocks
    assert abs(r["alu"]["frac"] - blocks / 1.2e-3 / bench.philox_peak()) < 1e-12
    assert abs(r["hbm_frac"] - by / 1.2e-3 / 1e9 / peak) < 1e-12
    # fp32 rows: 4 bytes per entry at the copy bandwidth take longer than the Philox work
    w = types.SimpleNamespace(B=64, K=5, V=201088)
    r = bench.sample_roofline(w, 0.075, w.B * w.K * w.V * 4, peak)
    assert r["bound"] == "hbm" and r["frac"] == r["hbm_frac"]
