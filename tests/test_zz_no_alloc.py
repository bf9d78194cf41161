"""GPU: sd_verify_noalloc, the verify entry point for callers that cannot allocate device memory
(for instance a plugin that is handed only its input and output buffers by a host runtime that
owns every allocation). Its merge slots live in a fixed device array inside the library instead
of a caller-provided workspace. Called here through the C ABI with ctypes, twice in a row, and
compared with sd_verify's results on the same inputs: every output must match exactly, up to
the largest batch the fixed array holds.

This file is collected last so that a run stopping at its first failure has already run every
other test; it also passes alone in a fresh process."""

import ctypes

import numpy as np
import pytest
import torch

import verify_draft_prep_gb300 as sd
import workloads

pytestmark = pytest.mark.gpu


def _outputs(B, K):
    z = lambda *shape: torch.full(shape, -7, dtype=torch.int32, device="cuda")  # noqa: E731
    return dict(out_tokens=z(B, K + 1), num_accepted=z(B), err=torch.zeros(1, dtype=torch.int32,
                                                                          device="cuda"),
                p_at=torch.full((B, K), -7.0, device="cuda"),
                q_at=torch.full((B, K), -7.0, device="cuda"))


def _noalloc_call(lib, w, o, dtype):
    B, K, V = w.B, w.K, w.V
    stream = torch.cuda.current_stream().cuda_stream
    temp = None if w.temperature is None else w.temperature.data_ptr()
    return lib.sd_verify_noalloc(B, K, V, dtype, w.target.data_ptr(), w.target.stride(0),
                                 w.draft.data_ptr(), w.draft.stride(0), w.drafts.data_ptr(),
                                 temp, w.seed, 0, o["out_tokens"].data_ptr(),
                                 o["num_accepted"].data_ptr(), o["p_at"].data_ptr(),
                                 o["q_at"].data_ptr(), o["err"].data_ptr(), stream)


def _check_against_workspace_entry_point(lib, w, dtype):
    ref = _outputs(w.B, w.K)
    sd.sd_verify(w.target, w.draft, w.drafts, ref["out_tokens"], ref["num_accepted"],
                 temperature=w.temperature, seed=w.seed, p_at_draft=ref["p_at"],
                 q_at_draft=ref["q_at"], err=ref["err"])
    torch.cuda.synchronize()
    for call in range(2):  # the shared scratch must serve consecutive calls
        o = _outputs(w.B, w.K)
        assert _noalloc_call(lib, w, o, dtype) == 0
        torch.cuda.synchronize()
        for k in ("out_tokens", "num_accepted", "err"):
            assert torch.equal(o[k], ref[k]), (call, k)
        for k in ("p_at", "q_at"):
            assert torch.equal(o[k].view(torch.int32), ref[k].view(torch.int32)), (call, k)


@pytest.mark.parametrize("name,B,dtype", [("b64", 64, sd.SD_F32_PROBS),
                                          ("b256mix", 40, sd.SD_F32_PROBS),
                                          ("b1024lg", 24, sd.SD_BF16_LOGITS)])
def test_noalloc_matches_workspace_entry_point(name, B, dtype):
    sd.build()
    lib = sd.load()
    w = workloads.make(name, device="cuda", B=B)
    _check_against_workspace_entry_point(lib, w, dtype)


@pytest.mark.parametrize("V,K", [(1024, 4), (16384, 2)])
def test_noalloc_at_its_largest_batch(V, K):
    # B = SD_VERIFY_NOALLOC_MAX_B, every request sampled at T = 1 (temperature NULL), so every
    # request merges its race through its slot and the whole fixed array is used: with V = 1024
    # one CTA per request, with V = 16384 the kernel that spreads every race row over all SMs.
    sd.build()
    lib = sd.load()
    B = sd.SD_VERIFY_NOALLOC_MAX_B
    g = torch.Generator(device="cuda").manual_seed(4242 + V)
    lt = 2.0 * torch.randn(B, K + 1, V, generator=g, device="cuda")
    lq = lt[:, :K] + 0.5 * torch.randn(B, K, V, generator=g, device="cuda")
    q = torch.softmax(lq, -1).reshape(B * K, V)
    w = workloads.make("small", device="cuda", B=1)
    w.B, w.K, w.V = B, K, V
    w.target = torch.softmax(lt, -1).reshape(B * (K + 1), V)
    w.draft = q
    w.drafts = torch.multinomial(q, 1, generator=g).view(B, K).to(torch.int32)
    w.temperature = None
    _check_against_workspace_entry_point(lib, w, sd.SD_F32_PROBS)


def test_noalloc_rejects_batches_beyond_its_scratch():
    sd.build()
    lib = sd.load()
    B = sd.SD_VERIFY_NOALLOC_MAX_B + 1
    P = None
    rc = lib.sd_verify_noalloc(B, 2, 10, sd.SD_F32_PROBS, P, 10, P, 10, P, P, 0, 0, P, P, P, P,
                               P, P)
    assert rc == -7
    assert b"SD_VERIFY_NOALLOC_MAX_B" in lib.sd_status_string(rc)
    assert lib.sd_verify_noalloc(0, 2, 10, sd.SD_F32_PROBS, P, 10, P, 10, P, P, 0, 0, P, P, P, P,
                                 P, P) == 0
    _ = ctypes  # the entry point is called through the C ABI above
    assert np.int32(rc) == -7
