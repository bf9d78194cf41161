"""GPU: the device Philox stream and race variates against the oracle, and the exhaustive error
bound of the race filter's fast -log approximation."""

import math

import numpy as np
import pytest
import torch

import oracle
import verify_draft_prep_gb300 as sd

pytestmark = pytest.mark.gpu


def test_device_philox_matches_oracle():
    rng = np.random.default_rng(0)
    n = 4096
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    ctr[:3] = [[0, 0, 0, 0], [0xFFFFFFFF] * 4, [0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344]]
    for seed in (0, 0xFFFFFFFFFFFFFFFF, 0x299F31D0A4093822, 12345):
        c = torch.from_numpy(ctr.view(np.int32)).cuda()
        out = torch.zeros_like(c)
        sd.sd_philox_words(c, seed, out)
        got = out.cpu().numpy().view(np.uint32)
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for i in range(0, n, 97):
            assert list(got[i]) == list(oracle.philox4x32_10(ctr[i], key)), (seed, i)


def test_device_race_E_matches_oracle():
    # same seed/counter words -> same E: device double log vs the host libm log, both rounded
    # to fp32. They may differ only where the double result sits on an fp32 rounding boundary.
    rng = np.random.default_rng(1)
    w = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    w[:6] = [0, 1, 2**31, 0xFF000000, 0xFFFFFFFE, 0xFFFFFFFF]
    t = torch.from_numpy(w.view(np.int32)).cuda()
    E = torch.zeros(w.size, dtype=torch.float32, device="cuda")
    sd.sd_race_E(t, E)
    got = E.cpu().numpy()
    want = np.array([-math.log((int(v) + 0.5) / 2**32) for v in w]).astype(np.float32)  # libm
    mismatch = np.nonzero(got != want)[0]
    assert mismatch.size == 0, (mismatch[:5], got[mismatch[:5]], want[mismatch[:5]])
    # spot-check against the oracle's own function on the race counter layout
    for x in range(0, 4000, 37):
        words = oracle.philox4x32_10([x >> 2, 3, 5, 1], [7, 0])
        wt = torch.tensor([int(words[x & 3])], dtype=torch.int64).to(torch.int32).cuda()
        e1 = torch.zeros(1, device="cuda")
        sd.sd_race_E(wt, e1)
        assert e1.item() == oracle.race_E(7, 5, 3, x)


def test_race_filter_approximation_bound_exhaustive():
    # every one of the 2^32 words. The race keeps every unit whose approximate maximum is within
    # a relative band of 2^-7 of the CTA's; that is exact as long as twice the approximation's
    # worst error stays below the band, asserted here with a further factor 4 of margin.
    out = torch.zeros(1, dtype=torch.float32, device="cuda")
    sd.sd_race_E_approx_error(0, 1 << 32, out)
    torch.cuda.synchronize()
    worst = out.item()
    print(f"worst relative error of the race filter's 1/E approximation: {worst:.3e}")
    assert 0 < worst <= 2.0**-10


def test_pair_evaluated_E_is_the_double_path_on_every_word():
    # The kernels form E from pairs of fp32 and take the double log only where the pair's value
    # lies within 2^-36 of an fp32 rounding boundary; over all 2^32 words that must give the
    # double path's value bit for bit, with the double path taken rarely (about 1 word in 2900).
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    sd.sd_race_E_check(0, 1 << 32, counts)
    torch.cuda.synchronize()
    mismatches, near = (int(v) for v in counts.cpu())
    print(f"pair-evaluated E: {mismatches} mismatches, {near} words on the double path")
    assert mismatches == 0
    assert 0 < near < (1 << 32) // 1000
