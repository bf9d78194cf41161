"""Python binding of libsd_gb300 (speculative-decoding verify + P-EAGLE draft-batch rebuild).

Argument marshalling only: every call forwards raw device pointers, sizes and the current CUDA
stream of the tensors' device to the C ABI declared in include/sd.h; all arithmetic runs in the
library's sm_103a kernels. There is no fallback: if the shared library is missing or fails to
load, every call raises.

Build the library with ``verify_draft_prep_gb300.build()`` (nvcc, sm_103a).
"""

from __future__ import annotations

import ctypes
import os
import threading

from ._build import LIB as LIB_PATH
from ._build import build

SD_F32_PROBS = 0
SD_BF16_LOGITS = 1
SD_K_MAX = 16
SD_VERIFY_NOALLOC_MAX_B = 4096

SD_ERR_TOKEN_RANGE = 1
SD_ERR_BLOCK_TABLE = 2
SD_ERR_NUM_ACCEPTED = 4
SD_ERR_MAP_RANGE = 8
SD_ERR_ZERO_ROW = 16
SD_ERR_TOTAL_RANGE = 32
SD_ERR_WAIT = 64
SD_ERR_DRAFT_COUNT = 128

EXPORTED = ["sd_verify", "sd_verify_workspace_bytes", "sd_verify_kernels",
            "sd_verify_noalloc", "sd_draft_sample", "sd_pdraft_prepare_padded",
            "sd_verify_ragged", "sd_pdraft_prepare_ragged", "sd_pdraft_expand", "sd_pdraft_prepare", "sd_hidden_gather", "sd_philox_words", "sd_race_E",
            "sd_race_E_approx_error", "sd_race_E_check", "sd_status_string", "sd_version",
            "sd_verify_prepare", "sd_verify_prepare_workspace_bytes", "sd_verify_prepare_kernels",
            "sd_verify_prepare_ragged", "sd_diag_verify_prepare_withheld",
            "sd_verify_prepare_padded"]

_lock = threading.Lock()
_lib = None


class SDError(RuntimeError):
    pass


def load():
    """Load libsd_gb300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise SDError(f"{LIB_PATH} is missing: build it with verify_draft_prep_gb300.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P, i32, i64, u32, u64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_long, ctypes.c_uint32,
                                 ctypes.c_uint64)
        lib.sd_verify.argtypes = [i32, i32, i32, i32, P, i64, P, i64, P, P, u64, u32, P, P, P,
                                  P, P, ctypes.c_size_t, P, P]
        lib.sd_verify.restype = i32
        lib.sd_verify_ragged.argtypes = [i32, i32, i32, i32, P, i64, P, i64, P, P, P, u64, u32, P,
                                         P, P, P, P, ctypes.c_size_t, P, P]
        lib.sd_verify_ragged.restype = i32
        lib.sd_verify_noalloc.argtypes = [i32, i32, i32, i32, P, i64, P, i64, P, P, u64, u32, P,
                                          P, P, P, P, P]
        lib.sd_verify_noalloc.restype = i32
        lib.sd_verify_workspace_bytes.argtypes = [i32, i32, i32, i32]
        lib.sd_verify_workspace_bytes.restype = ctypes.c_size_t
        lib.sd_draft_sample.argtypes = [i32, i32, i32, i32, P, i64, P, u64, u32, P, P, P]
        lib.sd_draft_sample.restype = i32
        lib.sd_verify_kernels.argtypes = [i32, i32, i32, i32]
        lib.sd_verify_kernels.restype = i32
        lib.sd_verify_prepare.argtypes = [i32, i32, i32, i32, P, i64, P, i64, P, P, u64, u32, P,
                                          P, P, P, P, P, i32, i32, ctypes.c_int32, i32, P, P, P,
                                          P, P, P, P, P, P, i32, P, i64, i32, P, P, i64, P,
                                          ctypes.c_size_t, P, P]
        lib.sd_verify_prepare.restype = i32
        lib.sd_diag_verify_prepare_withheld.argtypes = [i32, u32] + lib.sd_verify_prepare.argtypes
        lib.sd_diag_verify_prepare_withheld.restype = i32
        lib.sd_verify_prepare_ragged.argtypes = [i32, i32, i32, i32, P, i64, P, i64, P, P, P, u64,
                                                 u32, P, P, P, P, P, P, i32, i32, ctypes.c_int32,
                                                 i32, P, P, P, P, P, P, P, P, P, i32, P, i64, i32,
                                                 P, P, i64, P, ctypes.c_size_t, P, P]
        lib.sd_verify_prepare_ragged.restype = i32
        lib.sd_verify_prepare_workspace_bytes.argtypes = [i32]
        lib.sd_verify_prepare_workspace_bytes.restype = ctypes.c_size_t
        lib.sd_verify_prepare_kernels.argtypes = [i32, i32, i32, i32, i32]
        lib.sd_verify_prepare_kernels.restype = i32
        lib.sd_pdraft_expand.argtypes = [i32, i32, P, P, P, P, i32, i32, ctypes.c_int32, i32,
                                         P, P, P, P, P, P, P, P, P, P, P]
        lib.sd_pdraft_expand.restype = i32
        lib.sd_pdraft_prepare.argtypes = [i32, i32, P, P, P, P, i32, i32, ctypes.c_int32, i32,
                                          P, P, P, P, P, P, P, P, P, i32, P, i64, i32, P, P, i64,
                                          P, P]
        lib.sd_pdraft_prepare.restype = i32
        lib.sd_pdraft_prepare_ragged.argtypes = [i32, i32, P, P, P, P, P, i32, i32,
                                                 ctypes.c_int32, i32, P, P, P, P, P, P, P, P, P,
                                                 i32, P, i64, i32, P, P, i64, P, P]
        lib.sd_pdraft_prepare_ragged.restype = i32
        lib.sd_pdraft_prepare_padded.argtypes = [i32, i32, P, P, P, P, i32, i32, ctypes.c_int32,
                                                 P, P, P, P, P, P, P, P, i32, P, i64, i32, P, P,
                                                 i64, P, P]
        lib.sd_pdraft_prepare_padded.restype = i32
        lib.sd_verify_prepare_padded.argtypes = [i32, i32, i32, i32, P, i64, P, i64, P, P, u64,
                                                 u32, P, P, P, P, P, P, i32, i32, ctypes.c_int32,
                                                 P, P, P, P, P, P, P, P, i32, P, i64, i32, P, P,
                                                 i64, P, ctypes.c_size_t, P, P]
        lib.sd_verify_prepare_padded.restype = i32
        lib.sd_hidden_gather.argtypes = [i32, i32, P, P, P, i64, i32, P, P, i64, P, P]
        lib.sd_hidden_gather.restype = i32
        lib.sd_philox_words.argtypes = [i32, P, u64, P, P]
        lib.sd_philox_words.restype = i32
        lib.sd_race_E.argtypes = [i32, P, P, P]
        lib.sd_race_E.restype = i32
        lib.sd_race_E_approx_error.argtypes = [u32, u64, P, P]
        lib.sd_race_E_approx_error.restype = i32
        lib.sd_race_E_check.argtypes = [u32, u64, P, P]
        lib.sd_race_E_check.restype = i32
        lib.sd_status_string.argtypes = [i32]
        lib.sd_status_string.restype = ctypes.c_char_p
        lib.sd_version.argtypes = []
        lib.sd_version.restype = i32
        _lib = lib
        return lib


def _check(rc: int, what: str):
    if rc != 0:
        msg = load().sd_status_string(rc).decode()
        raise SDError(f"{what} failed: {msg} ({rc})")


def _ptr(t):
    """Device pointer of a tensor on the GPU, or of a pinned host tensor (page-locked host memory
    is addressable by the GPU: the kernels then read it over the host link)."""
    if t is None:
        return None
    if not (t.is_cuda or t.is_pinned()):
        raise SDError("tensors passed to libsd_gb300 must live on the GPU or in pinned memory")
    return t.data_ptr()


def _device(t):
    """The tensor's GPU, or the current GPU for a pinned host tensor."""
    import torch

    return t.device if t.is_cuda else torch.device("cuda", torch.cuda.current_device())


def _stream(t, stream):
    import torch

    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    # a pinned host tensor has no device of its own: the current device's stream
    return torch.cuda.current_stream(_device(t)).cuda_stream


def _row_stride(t):
    if t.dim() != 2 or t.stride(1) != 1:
        raise SDError("row arrays must be 2-D with contiguous rows")
    return t.stride(0)


_workspaces = {}


def workspace(device, B, K, V, dtype):
    """A zeroed verify workspace for this device, shared by calls that pass none (calls on
    concurrent streams must pass their own)."""
    import torch

    need = load().sd_verify_workspace_bytes(B, K, V, dtype)
    key = torch.device(device)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=key)
        _workspaces[key] = ws
    return ws


def sd_verify(target, draft, drafts, out_tokens, num_accepted, temperature=None, seed=0,
              p_at_draft=None, q_at_draft=None, err=None, stream=None, workspace_buf=None,
              request_base=0):
    """Verify K drafts per request (see include/sd.h).

    target: [B*(K+1), V] float32 probabilities or bfloat16 logits; draft: [B*K, V] same dtype;
    drafts: [B, K] int32; out_tokens: [B, K+1] int32; num_accepted: [B] int32;
    temperature: [B] float32 or None; p_at_draft / q_at_draft: [B, K] float32 or None;
    err: [1] int32 or None; workspace_buf: zeroed uint8 device tensor of at least
    sd_verify_workspace_bytes bytes, or None for this device's shared one; request_base: the
    global request index of local request 0 (a shard of a larger batch).
    """
    import torch

    B, K = drafts.shape
    V = target.shape[1]
    if target.dtype == torch.float32:
        dtype = SD_F32_PROBS
    elif target.dtype == torch.bfloat16:
        dtype = SD_BF16_LOGITS
    else:
        raise SDError("target must be float32 probabilities or bfloat16 logits")
    if draft.dtype != target.dtype or draft.shape[1] != V:
        raise SDError("draft must match target's dtype and vocabulary")
    if target.shape[0] != B * (K + 1) or draft.shape[0] != B * K:
        raise SDError("row counts must be B*(K+1) (target) and B*K (draft)")
    ws = workspace_buf if workspace_buf is not None else workspace(_device(target), B, K, V,
                                                                   dtype)
    rc = load().sd_verify(B, K, V, dtype, _ptr(target), _row_stride(target), _ptr(draft),
                          _row_stride(draft), _ptr(drafts), _ptr(temperature), seed,
                          request_base, _ptr(out_tokens), _ptr(num_accepted), _ptr(p_at_draft),
                          _ptr(q_at_draft), _ptr(ws), ws.numel(), _ptr(err),
                          _stream(target, stream))
    _check(rc, "sd_verify")


def sd_verify_prepare(target, draft, drafts, out_tokens, num_accepted, pos0, block_table,
                      block_size, mask_token_id, input_ids, positions, slot_mapping, hidden_map,
                      is_masked, is_rejected, start_loc, new_token_idx, total_out, target_hidden,
                      h_shared, out_hidden, temperature=None, seed=0, p_at_draft=None,
                      q_at_draft=None, err=None, stream=None, workspace_buf=None,
                      request_base=0, diag_withhold=None):
    """sd_verify then sd_pdraft_prepare on its outputs, in one call (see include/sd.h): arguments
    as for the two calls; workspace_buf: zeroed uint8 device tensor of at least
    sd_verify_prepare_workspace_bytes(B) bytes, or None for this device's shared one.
    diag_withhold: test support, (request, wait_us) for sd_diag_verify_prepare_withheld."""
    import torch

    B, K = drafts.shape
    V = target.shape[1]
    if target.dtype == torch.float32:
        dtype = SD_F32_PROBS
    elif target.dtype == torch.bfloat16:
        dtype = SD_BF16_LOGITS
    else:
        raise SDError("target must be float32 probabilities or bfloat16 logits")
    if draft.dtype != target.dtype or draft.shape[1] != V:
        raise SDError("draft must match target's dtype and vocabulary")
    if target.shape[0] != B * (K + 1) or draft.shape[0] != B * K:
        raise SDError("row counts must be B*(K+1) (target) and B*K (draft)")
    cap, H = out_hidden.shape
    if input_ids.shape[0] != cap:
        raise SDError("out_hidden must have one row per drafter slot")
    ws = workspace_buf if workspace_buf is not None else workspace(_device(target), B, K, V,
                                                                   dtype)
    lib = load()
    fn, pre = lib.sd_verify_prepare, ()
    if diag_withhold is not None:
        fn, pre = lib.sd_diag_verify_prepare_withheld, tuple(diag_withhold)
    rc = fn(
        *pre, B, K, V, dtype, _ptr(target), _row_stride(target), _ptr(draft), _row_stride(draft),
        _ptr(drafts), _ptr(temperature), seed, request_base, _ptr(out_tokens),
        _ptr(num_accepted), _ptr(p_at_draft), _ptr(q_at_draft), _ptr(pos0), _ptr(block_table),
        block_table.shape[1], block_size, mask_token_id, cap, _ptr(input_ids), _ptr(positions),
        _ptr(slot_mapping), _ptr(hidden_map), _ptr(is_masked), _ptr(is_rejected),
        _ptr(start_loc), _ptr(new_token_idx), _ptr(total_out), H, _ptr(target_hidden),
        _row_stride(target_hidden), target_hidden.shape[0], _ptr(h_shared), _ptr(out_hidden),
        _row_stride(out_hidden), _ptr(ws), ws.numel(), _ptr(err), _stream(target, stream))
    _check(rc, "sd_verify_prepare")


def sd_verify_prepare_ragged(target, draft, drafts, cu_drafts, out_tokens, num_accepted, pos0,
                             block_table, block_size, mask_token_id, input_ids, positions,
                             slot_mapping, hidden_map, is_masked, is_rejected, start_loc,
                             new_token_idx, total_out, target_hidden, h_shared, out_hidden,
                             temperature=None, seed=0, p_at_draft=None, q_at_draft=None, err=None,
                             stream=None, workspace_buf=None, request_base=0):
    """sd_verify_ragged then sd_pdraft_prepare_ragged on its outputs, in one call (see
    include/sd.h); shapes as for the two calls (out_tokens [B, K_max+1])."""
    import torch

    B, K1 = out_tokens.shape
    V = target.shape[1]
    if target.dtype == torch.float32:
        dtype = SD_F32_PROBS
    elif target.dtype == torch.bfloat16:
        dtype = SD_BF16_LOGITS
    else:
        raise SDError("target must be float32 probabilities or bfloat16 logits")
    if draft.dtype != target.dtype or cu_drafts.shape[0] != B + 1:
        raise SDError("draft must match target; cu_drafts needs B+1 entries")
    cap, H = out_hidden.shape
    if input_ids.shape[0] != cap:
        raise SDError("out_hidden must have one row per drafter slot")
    ws = workspace_buf if workspace_buf is not None else workspace(_device(target), B, K1 - 1, V,
                                                                   dtype)
    rc = load().sd_verify_prepare_ragged(
        B, K1 - 1, V, dtype, _ptr(target), _row_stride(target), _ptr(draft),
        _row_stride(draft) if draft.shape[0] else V, _ptr(drafts), _ptr(cu_drafts),
        _ptr(temperature), seed, request_base, _ptr(out_tokens), _ptr(num_accepted),
        _ptr(p_at_draft), _ptr(q_at_draft), _ptr(pos0), _ptr(block_table), block_table.shape[1],
        block_size, mask_token_id, cap, _ptr(input_ids), _ptr(positions), _ptr(slot_mapping),
        _ptr(hidden_map), _ptr(is_masked), _ptr(is_rejected), _ptr(start_loc),
        _ptr(new_token_idx), _ptr(total_out), H, _ptr(target_hidden),
        _row_stride(target_hidden), target_hidden.shape[0], _ptr(h_shared), _ptr(out_hidden),
        _row_stride(out_hidden), _ptr(ws), ws.numel(), _ptr(err), _stream(target, stream))
    _check(rc, "sd_verify_prepare_ragged")


def sd_verify_prepare_kernels(B, K, V, dtype, has_temperature):
    """Kernels one sd_verify_prepare call launches (0, 1 or 2)."""
    n = load().sd_verify_prepare_kernels(B, K, V, dtype, int(bool(has_temperature)))
    if n < 0:
        _check(n, "sd_verify_prepare_kernels")
    return n


def sd_verify_ragged(target, draft, drafts, cu_drafts, out_tokens, num_accepted, temperature=None,
                     seed=0, p_at_draft=None, q_at_draft=None, err=None, stream=None,
                     workspace_buf=None, request_base=0):
    """Verify with a draft count per request (see include/sd.h).

    cu_drafts: [B+1] int32 exclusive prefix of the counts; target: [cu[B] + B, V] rows;
    draft: [cu[B], V]; drafts: [cu[B]] int32; out_tokens: [B, K_max+1]; p/q_at: [B, K_max].
    """
    import torch

    B, K1 = out_tokens.shape
    V = target.shape[1]
    if target.dtype == torch.float32:
        dtype = SD_F32_PROBS
    elif target.dtype == torch.bfloat16:
        dtype = SD_BF16_LOGITS
    else:
        raise SDError("target must be float32 probabilities or bfloat16 logits")
    if draft.dtype != target.dtype or cu_drafts.shape[0] != B + 1:
        raise SDError("draft must match target; cu_drafts needs B+1 entries")
    ws = workspace_buf if workspace_buf is not None else workspace(_device(target), B, K1 - 1, V,
                                                                   dtype)
    rc = load().sd_verify_ragged(B, K1 - 1, V, dtype, _ptr(target), _row_stride(target),
                                 _ptr(draft), _row_stride(draft) if draft.shape[0] else V,
                                 _ptr(drafts), _ptr(cu_drafts), _ptr(temperature), seed,
                                 request_base, _ptr(out_tokens), _ptr(num_accepted),
                                 _ptr(p_at_draft), _ptr(q_at_draft), _ptr(ws), ws.numel(),
                                 _ptr(err), _stream(target, stream))
    _check(rc, "sd_verify_ragged")


def sd_verify_kernels(B, V, dtype, has_temperature):
    """How many kernels one sd_verify call with these sizes launches on the current device."""
    n = load().sd_verify_kernels(B, V, dtype, int(bool(has_temperature)))
    if n < 0:
        raise SDError(f"sd_verify_kernels: {load().sd_status_string(n).decode()}")
    return n


def sd_draft_sample(rows, drafts, temperature=None, seed=0, request_base=0, err=None,
                    stream=None):
    """Sample the drafter's K new drafts per request (see include/sd.h).

    rows: [B*K, V] float32 probabilities or bfloat16 logits; drafts: [B, K] int32 (output);
    temperature: [B] float32 or None; request_base: global request index of local request 0.
    """
    import torch

    B, K = drafts.shape
    V = rows.shape[1]
    if rows.dtype == torch.float32:
        dtype = SD_F32_PROBS
    elif rows.dtype == torch.bfloat16:
        dtype = SD_BF16_LOGITS
    else:
        raise SDError("rows must be float32 probabilities or bfloat16 logits")
    if rows.shape[0] != B * K:
        raise SDError("rows must hold B*K rows")
    rc = load().sd_draft_sample(B, K, V, dtype, _ptr(rows), _row_stride(rows), _ptr(temperature),
                                seed, request_base, _ptr(drafts), _ptr(err), _stream(rows, stream))
    _check(rc, "sd_draft_sample")


def sd_pdraft_expand(out_tokens, num_accepted, pos0, block_table, block_size, mask_token_id,
                     input_ids, positions, slot_mapping, hidden_map, is_masked, is_rejected,
                     start_loc, new_token_idx, total_out, err=None, stream=None):
    """Rebuild the drafter batch (see include/sd.h). Outputs have `capacity` = len(input_ids)."""
    B, K1 = out_tokens.shape
    rc = load().sd_pdraft_expand(
        B, K1 - 1, _ptr(out_tokens), _ptr(num_accepted), _ptr(pos0), _ptr(block_table),
        block_table.shape[1], block_size, mask_token_id, input_ids.shape[0], _ptr(input_ids),
        _ptr(positions), _ptr(slot_mapping), _ptr(hidden_map), _ptr(is_masked),
        _ptr(is_rejected), _ptr(start_loc), _ptr(new_token_idx), _ptr(total_out), _ptr(err),
        _stream(start_loc, stream))
    _check(rc, "sd_pdraft_expand")


def sd_pdraft_prepare(out_tokens, num_accepted, pos0, block_table, block_size, mask_token_id,
                      input_ids, positions, slot_mapping, hidden_map, is_masked, is_rejected,
                      start_loc, new_token_idx, total_out, target_hidden, h_shared, out_hidden,
                      err=None, stream=None):
    """sd_pdraft_expand and the hidden-state gather in one launch (see include/sd.h)."""
    B, K1 = out_tokens.shape
    cap, H = out_hidden.shape
    if input_ids.shape[0] != cap:
        raise SDError("out_hidden must have one row per drafter slot")
    rc = load().sd_pdraft_prepare(
        B, K1 - 1, _ptr(out_tokens), _ptr(num_accepted), _ptr(pos0), _ptr(block_table),
        block_table.shape[1], block_size, mask_token_id, cap, _ptr(input_ids), _ptr(positions),
        _ptr(slot_mapping), _ptr(hidden_map), _ptr(is_masked), _ptr(is_rejected),
        _ptr(start_loc), _ptr(new_token_idx), _ptr(total_out), H, _ptr(target_hidden),
        _row_stride(target_hidden), target_hidden.shape[0], _ptr(h_shared), _ptr(out_hidden),
        _row_stride(out_hidden), _ptr(err), _stream(start_loc, stream))
    _check(rc, "sd_pdraft_prepare")


def sd_pdraft_prepare_ragged(out_tokens, num_accepted, cu_drafts, pos0, block_table, block_size,
                             mask_token_id, input_ids, positions, slot_mapping, hidden_map,
                             is_masked, is_rejected, start_loc, new_token_idx, total_out,
                             target_hidden, h_shared, out_hidden, err=None, stream=None):
    """sd_pdraft_prepare with a draft count per request (see include/sd.h)."""
    B, K1 = out_tokens.shape
    cap, H = out_hidden.shape
    if input_ids.shape[0] != cap or cu_drafts.shape[0] != B + 1:
        raise SDError("out_hidden needs one row per drafter slot, cu_drafts B+1 entries")
    rc = load().sd_pdraft_prepare_ragged(
        B, K1 - 1, _ptr(out_tokens), _ptr(num_accepted), _ptr(cu_drafts), _ptr(pos0),
        _ptr(block_table), block_table.shape[1], block_size, mask_token_id, cap, _ptr(input_ids),
        _ptr(positions), _ptr(slot_mapping), _ptr(hidden_map), _ptr(is_masked),
        _ptr(is_rejected), _ptr(start_loc), _ptr(new_token_idx), _ptr(total_out), H,
        _ptr(target_hidden), _row_stride(target_hidden), target_hidden.shape[0], _ptr(h_shared),
        _ptr(out_hidden), _row_stride(out_hidden), _ptr(err), _stream(start_loc, stream))
    _check(rc, "sd_pdraft_prepare_ragged")


def sd_pdraft_prepare_padded(out_tokens, num_accepted, pos0, block_table, block_size,
                             mask_token_id, input_ids, positions, slot_mapping, hidden_map,
                             is_masked, rejected, scatter_map, new_token_idx, target_hidden=None,
                             h_shared=None, out_hidden=None, err=None, stream=None):
    """The drafter batch in fixed rows of 2K slots per request (see include/sd.h); outputs have
    B*2K entries (out_hidden [B*2K, H] bf16, or None for the metadata alone)."""
    B, K1 = out_tokens.shape
    K = K1 - 1
    if input_ids.shape[0] != B * 2 * K:
        raise SDError("padded outputs have B*2K entries")
    H = out_hidden.shape[1] if out_hidden is not None else 1
    n_in = target_hidden.shape[0] if target_hidden is not None else 0
    rc = load().sd_pdraft_prepare_padded(
        B, K, _ptr(out_tokens), _ptr(num_accepted), _ptr(pos0), _ptr(block_table),
        block_table.shape[1], block_size, mask_token_id, _ptr(input_ids), _ptr(positions),
        _ptr(slot_mapping), _ptr(hidden_map), _ptr(is_masked), _ptr(rejected),
        _ptr(scatter_map), _ptr(new_token_idx), H, _ptr(target_hidden),
        _row_stride(target_hidden) if target_hidden is not None else H, n_in, _ptr(h_shared),
        _ptr(out_hidden), _row_stride(out_hidden) if out_hidden is not None else H, _ptr(err),
        _stream(input_ids, stream))
    _check(rc, "sd_pdraft_prepare_padded")


def sd_verify_prepare_padded(target, draft, drafts, out_tokens, num_accepted, pos0, block_table,
                             block_size, mask_token_id, input_ids, positions, slot_mapping,
                             hidden_map, is_masked, rejected, scatter_map, new_token_idx,
                             target_hidden=None, h_shared=None, out_hidden=None, temperature=None,
                             seed=0, p_at_draft=None, q_at_draft=None, err=None, stream=None,
                             workspace_buf=None, request_base=0):
    """sd_verify then sd_pdraft_prepare_padded on its outputs, in one call (see include/sd.h):
    arguments as for the two calls; workspace_buf as for sd_verify."""
    import torch

    B, K = drafts.shape
    V = target.shape[1]
    if target.dtype == torch.float32:
        dtype = SD_F32_PROBS
    elif target.dtype == torch.bfloat16:
        dtype = SD_BF16_LOGITS
    else:
        raise SDError("target must be float32 probabilities or bfloat16 logits")
    if draft.dtype != target.dtype or draft.shape[1] != V:
        raise SDError("draft must match target's dtype and vocabulary")
    if target.shape[0] != B * (K + 1) or draft.shape[0] != B * K:
        raise SDError("row counts must be B*(K+1) (target) and B*K (draft)")
    if input_ids.shape[0] != B * 2 * K:
        raise SDError("padded outputs have B*2K entries")
    H = out_hidden.shape[1] if out_hidden is not None else 1
    n_in = target_hidden.shape[0] if target_hidden is not None else 0
    ws = workspace_buf if workspace_buf is not None else workspace(_device(target), B, K, V,
                                                                   dtype)
    rc = load().sd_verify_prepare_padded(
        B, K, V, dtype, _ptr(target), _row_stride(target), _ptr(draft), _row_stride(draft),
        _ptr(drafts), _ptr(temperature), seed, request_base, _ptr(out_tokens),
        _ptr(num_accepted), _ptr(p_at_draft), _ptr(q_at_draft), _ptr(pos0), _ptr(block_table),
        block_table.shape[1], block_size, mask_token_id, _ptr(input_ids), _ptr(positions),
        _ptr(slot_mapping), _ptr(hidden_map), _ptr(is_masked), _ptr(rejected), _ptr(scatter_map),
        _ptr(new_token_idx), H, _ptr(target_hidden),
        _row_stride(target_hidden) if target_hidden is not None else H, n_in, _ptr(h_shared),
        _ptr(out_hidden), _row_stride(out_hidden) if out_hidden is not None else H, _ptr(ws),
        ws.numel(), _ptr(err), _stream(target, stream))
    _check(rc, "sd_verify_prepare_padded")


def sd_hidden_gather(total_out, hidden_map, target_hidden, h_shared, out_hidden, err=None,
                     stream=None):
    """Gather drafter hidden states (see include/sd.h). bf16 rows."""
    cap, H = out_hidden.shape
    rc = load().sd_hidden_gather(cap, H, _ptr(total_out), _ptr(hidden_map), _ptr(target_hidden),
                                 _row_stride(target_hidden), target_hidden.shape[0],
                                 _ptr(h_shared), _ptr(out_hidden), _row_stride(out_hidden),
                                 _ptr(err), _stream(out_hidden, stream))
    _check(rc, "sd_hidden_gather")


def sd_philox_words(ctr, seed, out, stream=None):
    rc = load().sd_philox_words(ctr.shape[0], _ptr(ctr), seed, _ptr(out), _stream(ctr, stream))
    _check(rc, "sd_philox_words")


def sd_race_E(w, E, stream=None):
    rc = load().sd_race_E(w.shape[0], _ptr(w), _ptr(E), _stream(w, stream))
    _check(rc, "sd_race_E")


def sd_race_E_approx_error(w_begin, count, max_rel, stream=None):
    rc = load().sd_race_E_approx_error(w_begin, count, _ptr(max_rel), _stream(max_rel, stream))
    _check(rc, "sd_race_E_approx_error")


def sd_race_E_check(w_begin, count, counts, stream=None):
    """counts: int64 CUDA tensor [2], zeroed: (words differing from the double path, words that
    took the double path) over [w_begin, w_begin + count)."""
    rc = load().sd_race_E_check(w_begin, count, _ptr(counts), _stream(counts, stream))
    _check(rc, "sd_race_E_check")
