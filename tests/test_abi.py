"""The C-ABI library loads and exports every entry point include/sd.h declares; host-side
argument checks answer before any device work (so they run on a machine without a GPU)."""

import ctypes
import os
import re

import pytest

import verify_draft_prep_gb300 as sd
from conftest import ROOT


def _declared():
    text = open(os.path.join(ROOT, "include", "sd.h")).read()
    return sorted(set(re.findall(r"^SD_API\s+[\w\s\*]+?\b(sd_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    sd.build()
    return sd.load()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"sd_verify", "sd_pdraft_expand", "sd_hidden_gather"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(names) == sorted(sd.EXPORTED)
    assert lib.sd_version() == 100


def test_internal_symbols_are_hidden(lib):
    raw = ctypes.CDLL(sd.LIB_PATH)
    for n in ("sd_verify_launch", "sd_expand_launch", "sd_gather_launch"):
        with pytest.raises(AttributeError):
            getattr(raw, n)


def test_host_argument_checks(lib):
    P = None
    # K out of range, V < 1, ld < V, bad dtype
    assert lib.sd_verify(1, 0, 10, 0, P, 10, P, 10, P, P, 0, 0, P, P, P, P, P, 0, P, P) == -2
    assert lib.sd_verify(1, 17, 10, 0, P, 10, P, 10, P, P, 0, 0, P, P, P, P, P, 0, P, P) == -2
    assert lib.sd_verify(1, 2, 0, 0, P, 10, P, 10, P, P, 0, 0, P, P, P, P, P, 0, P, P) == -2
    assert lib.sd_verify(1, 2, 10, 0, P, 9, P, 10, P, P, 0, 0, P, P, P, P, P, 0, P, P) == -2
    assert lib.sd_verify(1, 2, 10, 7, P, 10, P, 10, P, P, 0, 0, P, P, P, P, P, 0, P, P) == -3
    # null rows
    assert lib.sd_verify(1, 2, 10, 0, P, 10, P, 10, P, P, 0, 0, P, P, P, P, P, 0, P, P) == -1
    # a workspace smaller than sd_verify_workspace_bytes is refused
    assert lib.sd_verify_workspace_bytes(64, 5, 201088, 0) == 64 * 16
    assert lib.sd_verify(4, 2, 10, 0, 16, 10, 16, 10, 16, P, 0, 0, 16, 16, P, P, 16, 63, P, P) == -2
    # request_base + B beyond the 32-bit Philox request index
    assert lib.sd_verify(4, 2, 10, 0, 16, 10, 16, 10, 16, P, 0, 2**32 - 3, 16, 16, P, P, 16, 64, P,
                         P) == -2
    # the launch-count query checks its arguments before it looks at the device
    assert lib.sd_verify_kernels(4, 10, 7, 0) == -3
    assert lib.sd_verify_kernels(-1, 10, 0, 0) == -2
    assert lib.sd_verify_kernels(0, 10, 0, 0) == 0
    # an empty batch is a no-op
    assert lib.sd_verify(0, 2, 10, 0, P, 10, P, 10, P, P, 0, 0, P, P, P, P, P, 0, P, P) == 0
    # drafter-side sampling: K range, ld < V, dtype, request_base overflow, null rows, empty batch
    assert lib.sd_draft_sample(2, 0, 10, 0, 16, 10, P, 0, 0, 16, P, P) == -2
    assert lib.sd_draft_sample(2, 17, 10, 0, 16, 10, P, 0, 0, 16, P, P) == -2
    assert lib.sd_draft_sample(2, 3, 10, 0, 16, 9, P, 0, 0, 16, P, P) == -2
    assert lib.sd_draft_sample(2, 3, 10, 5, 16, 10, P, 0, 0, 16, P, P) == -3
    assert lib.sd_draft_sample(2, 3, 10, 0, 16, 10, P, 0, 2**32 - 1, 16, P, P) == -2
    assert lib.sd_draft_sample(2, 3, 10, 0, P, 10, P, 0, 0, 16, P, P) == -1
    assert lib.sd_draft_sample(0, 3, 10, 0, P, 10, P, 0, 0, P, P, P) == 0
    # ragged rebuild: the prefix of counts is required
    assert lib.sd_pdraft_prepare_ragged(1, 2, 16, 16, P, 16, 16, 1, 16, 0, 4, *([16] * 9), 8,
                                        16, 8, 1, 16, 16, 8, P, P) == -1
    # padded rebuild: K range, null outputs, empty batch
    assert lib.sd_pdraft_prepare_padded(1, 0, *([P] * 4), 1, 16, 0, *([P] * 8), 8, P, 8, 0, P, P,
                                        8, P, P) == -2
    assert lib.sd_pdraft_prepare_padded(1, 2, *([P] * 4), 1, 16, 0, *([P] * 8), 8, P, 8, 0, P, P,
                                        8, P, P) == -1
    assert lib.sd_pdraft_prepare_padded(0, 2, *([P] * 4), 1, 16, 0, *([P] * 8), 8, P, 8, 0, P, P,
                                        8, P, P) == 0
    # expand: block size 0, null outputs
    assert lib.sd_pdraft_expand(1, 2, P, P, P, P, 1, 0, 0, 4, *([P] * 11)) == -2
    assert lib.sd_pdraft_expand(1, 2, P, P, P, P, 1, 16, 0, 4, *([P] * 11)) == -1
    # gather: H < 1, ld < H, odd (misaligned) bf16 pointer
    assert lib.sd_hidden_gather(4, 0, P, P, P, 8, 1, P, P, 8, P, P) == -2
    assert lib.sd_hidden_gather(4, 8, P, P, P, 7, 1, P, P, 8, P, P) == -2
    one = ctypes.c_int32(0)
    assert lib.sd_hidden_gather(4, 8, ctypes.addressof(one), 16, 17, 8, 1, 32, 64, 8, P, P) == -4
    assert lib.sd_status_string(-4).decode().startswith("a pointer")


def _vp_args(B=4, K=2, V=10, ws_bytes=80, P=16, **over):
    """sd_verify_prepare's 42 arguments with every pointer set to a dummy non-null value."""
    a = dict(B=B, K=K, V=V, dtype=0, target=P, ld_t=V, draft=P, ld_d=V, drafts=P, temperature=None,
             seed=0, request_base=0, out_tokens=P, num_accepted=P, p_at=None, q_at=None, pos0=P,
             block_table=P, max_blocks=4, block_size=16, mask_id=V, capacity=B * 2 * K,
             input_ids=P, positions=P, slot_mapping=P, hidden_map=P, is_masked=P, is_rejected=P,
             start_loc=P, new_token_idx=P, total_out=P, H=8, target_hidden=P, ld_in=8,
             n_in_rows=B * (K + 1), h_shared=P, out_hidden=P, ld_out=8, workspace=P,
             ws_bytes=ws_bytes, err=None, stream=None)
    a.update(over)
    return list(a.values())


def test_verify_prepare_host_checks(lib):
    assert lib.sd_verify_prepare_workspace_bytes(64) == 64 * 16
    assert lib.sd_verify_prepare_workspace_bytes(0) == 0
    assert lib.sd_verify_prepare(*_vp_args(K=0)) == -2
    assert lib.sd_verify_prepare(*_vp_args(dtype=5)) == -3
    assert lib.sd_verify_prepare(*_vp_args(ws_bytes=63)) == -2        # B*16 needed
    assert lib.sd_verify_prepare(*_vp_args(H=0)) == -2
    assert lib.sd_verify_prepare(*_vp_args(h_shared=None)) == -1
    assert lib.sd_verify_prepare(*_vp_args(start_loc=None)) == -1
    assert lib.sd_verify_prepare(*_vp_args(target=None)) == -1
    assert lib.sd_verify_prepare(*_vp_args(workspace=24, ws_bytes=96)) == -4  # 16-byte aligned
    assert lib.sd_verify_prepare_kernels(4, 2, 10, 7, 0) == -3
    assert lib.sd_verify_prepare_kernels(4, 0, 10, 0, 0) == -2
    assert lib.sd_verify_prepare_kernels(0, 2, 10, 0, 0) == 0


def test_error_bits_match_the_header():
    # every SD_ERR_* bit of include/sd.h has the same value in the Python package, and no two
    # bits share a value
    text = open(os.path.join(ROOT, "include", "sd.h")).read()
    bits = dict((n, int(v)) for n, v in re.findall(r"#define (SD_ERR_\w+) (\d+)", text))
    assert bits and len(set(bits.values())) == len(bits)
    for name, value in bits.items():
        assert getattr(sd, name) == value, name
        assert value & (value - 1) == 0, name  # a single bit


def test_constants_match_the_header():
    text = open(os.path.join(ROOT, "include", "sd.h")).read()
    for name in ("SD_F32_PROBS", "SD_BF16_LOGITS", "SD_K_MAX", "SD_VERIFY_NOALLOC_MAX_B"):
        m = re.search(r"#define %s (\d+)" % name, text)
        assert m and getattr(sd, name) == int(m.group(1)), name
    # every status code has its own text
    codes = [int(v) for v in re.findall(r"#define SD_E_\w+ \((-\d+)\)", text)]
    texts = {sd.load().sd_status_string(c) for c in codes + [0]}
    assert len(texts) == len(codes) + 1
