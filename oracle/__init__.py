"""Plain CPU oracle for the verify step and the P-EAGLE draft-batch rebuild.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` are the only callers. The product library never imports this package, and this
package never imports the product library: the two share only the seeded input generators in
``workloads``.

The arithmetic lives in ``sd_oracle.cpp`` (plain C++17, compiled without FMA contraction or
fast-math). This module compiles it with gcc and wraps it with ctypes over numpy arrays.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sd_oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libsd_oracle.so")
_lock = threading.Lock()
_lib = None

ERR_TOKEN_RANGE = 1
ERR_BLOCK_TABLE = 2
ERR_NUM_ACCEPTED = 4
ERR_MAP_RANGE = 8
ERR_ZERO_ROW = 16
ERR_TOTAL_RANGE = 32
ERR_DRAFT_COUNT = 128


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libsd_oracle.so`` (gcc, no GPU needed)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", "-Wall", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        override = os.environ.get("SD_ORACLE_LIB")  # a separately built copy (mutation tests)
        lib = ctypes.CDLL(override if override else build())
        P = ctypes.c_void_p
        i32, i64, u32, u64 = ctypes.c_int, ctypes.c_long, ctypes.c_uint32, ctypes.c_uint64
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_accept_uniform.argtypes = [u64, u32, u32]
        lib.oracle_accept_uniform.restype = ctypes.c_double
        lib.oracle_race_E.argtypes = [u64, u32, u32, u32]
        lib.oracle_race_E.restype = ctypes.c_float
        lib.oracle_race_E_tag.argtypes = [u64, u32, u32, u32, u32]
        lib.oracle_race_E_tag.restype = ctypes.c_float
        sample_args = [i32, i32, i32, P, i64, P, u64, P, P, P, P, i32]
        lib.oracle_draft_sample_probs.argtypes = sample_args
        lib.oracle_draft_sample_probs.restype = i32
        lib.oracle_draft_sample_logits.argtypes = sample_args
        lib.oracle_draft_sample_logits.restype = i32
        lib.oracle_race_row_f32.argtypes = [P, P, i32, i32, u64, u32, u32, P]
        lib.oracle_race_row_f32.restype = i32
        verify_args = [i32, i32, i32, P, i64, P, i64, P, P, u64, P, P, P, P, P, P, P, P, i32]
        lib.oracle_verify_probs.argtypes = verify_args
        lib.oracle_verify_probs.restype = i32
        lib.oracle_verify_logits.argtypes = verify_args
        lib.oracle_verify_logits.restype = i32
        lib.oracle_pdraft_expand.argtypes = [i32, i32, P, P, P, P, i32, i32, ctypes.c_int32,
                                             i32, P, P, P, P, P, P, P, P, P, P, P]
        lib.oracle_pdraft_expand.restype = i32
        lib.oracle_pdraft_prepare_padded.argtypes = [i32, i32, P, P, P, P, i32, i32,
                                                     ctypes.c_int32, P, P, P, P, P, P, P, P,
                                                     i32, P, i64, i32, P, P, i64, P]
        lib.oracle_pdraft_prepare_padded.restype = i32
        lib.oracle_hidden_gather.argtypes = [i32, i32, P, P, P, i64, i32, P, P, i64, P]
        lib.oracle_hidden_gather.restype = i32
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def philox4x32_10(ctr, key):
    """Philox4x32-10 of one 4-word counter under a 2-word key (Salmon et al., SC'11)."""
    c = _c(ctr, np.uint32)
    k = _c(key, np.uint32)
    out = np.zeros(4, np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def accept_uniform(seed: int, r: int, j: int) -> float:
    return _load().oracle_accept_uniform(seed, r, j)


def race_E(seed: int, r: int, j: int, x: int, tag: int = 1) -> float:
    if tag == 1:
        return _load().oracle_race_E(seed, r, j, x)
    return _load().oracle_race_E_tag(seed, r, j, x, tag)


def race_row(p, q, seed, r, j):
    """Exponential race on one fp32 row: returns (token or -1 when no key is positive, margin)."""
    p = _c(p, np.float32)
    qq = None if q is None else _c(q, np.float32)
    m = ctypes.c_double(0.0)
    x = _load().oracle_race_row_f32(_ptr(p), _ptr(qq), 0 if q is None else 1, p.shape[-1],
                                    seed, r, j, ctypes.byref(m))
    return x, m.value


def _verify(fn, B, K, V, target, ld_t, draft, ld_d, drafts, temperature, seed, req_ids,
            nthreads, margins):
    out_tokens = np.zeros((B, K + 1), np.int32)
    num_acc = np.zeros(B, np.int32)
    p_at = np.zeros((B, K), np.float32)
    q_at = np.zeros((B, K), np.float32)
    acc_m = np.zeros((B, K), np.float64) if margins else None
    race_m = np.zeros(B, np.float64) if margins else None
    err = np.zeros(1, np.int32)
    drafts = _c(drafts, np.int32)
    temp = None if temperature is None else _c(temperature, np.float32)
    rid = None if req_ids is None else _c(req_ids, np.int32)
    rc = fn(B, K, V, _ptr(target), ld_t, _ptr(draft), ld_d, _ptr(drafts), _ptr(temp), seed,
            _ptr(rid), _ptr(out_tokens), _ptr(num_acc), _ptr(p_at), _ptr(q_at), _ptr(acc_m),
            _ptr(race_m), _ptr(err), nthreads)
    if rc != 0:
        raise ValueError(f"oracle verify rejected its arguments (rc={rc})")
    res = dict(out_tokens=out_tokens, num_accepted=num_acc, p_at_draft=p_at, q_at_draft=q_at,
               err=int(err[0]))
    if margins:
        res["accept_margin"] = acc_m
        res["race_margin"] = race_m
    return res


def verify_probs(target, draft, drafts, temperature=None, seed=0, req_ids=None, nthreads=0,
                 margins=False):
    """Verify B requests on fp32 probability rows.

    target: [B, K+1, V] float32 (p_0..p_K); draft: [B, K, V] float32 (q_0..q_{K-1});
    drafts: [B, K] int32 (d_1..d_K). Returns a dict of numpy arrays.
    """
    target = _c(target, np.float32)
    draft = _c(draft, np.float32)
    B, K1, V = target.shape
    return _verify(_load().oracle_verify_probs, B, K1 - 1, V, target, V, draft, V, drafts,
                   temperature, seed, req_ids, nthreads, margins)


def verify_probs_strided(B, K, V, target, ld_t, draft, ld_d, drafts, temperature=None, seed=0,
                         req_ids=None, nthreads=0, margins=False):
    """As ``verify_probs`` on raw 2-D row arrays with explicit row strides (0 = one shared row)."""
    target = _c(target, np.float32)
    draft = _c(draft, np.float32)
    return _verify(_load().oracle_verify_probs, B, K, V, target, ld_t, draft, ld_d, drafts,
                   temperature, seed, req_ids, nthreads, margins)


def verify_logits(target_bits, draft_bits, drafts, temperature=None, seed=0, req_ids=None,
                  nthreads=0, margins=True):
    """Verify on bf16 logits given as uint16 bit patterns: target [B, K+1, V], draft [B, K, V]."""
    target_bits = _c(target_bits, np.uint16)
    draft_bits = _c(draft_bits, np.uint16)
    B, K1, V = target_bits.shape
    return _verify(_load().oracle_verify_logits, B, K1 - 1, V, target_bits, V, draft_bits, V,
                   drafts, temperature, seed, req_ids, nthreads, margins)


def _draft_sample(fn, rows, B, K, temperature, seed, req_ids, nthreads):
    V = rows.shape[-1]
    drafts = np.zeros((B, K), np.int32)
    margin = np.zeros((B, K), np.float64)
    err = np.zeros(1, np.int32)
    temp = None if temperature is None else _c(temperature, np.float32)
    rid = None if req_ids is None else _c(req_ids, np.int32)
    rc = fn(B, K, V, _ptr(rows), V, _ptr(temp), seed, _ptr(rid), _ptr(drafts), _ptr(margin),
            _ptr(err), nthreads)
    if rc != 0:
        raise ValueError(f"oracle draft sampling rejected its arguments (rc={rc})")
    return dict(drafts=drafts, margin=margin, err=int(err[0]))


def draft_sample_probs(q, temperature=None, seed=0, req_ids=None, nthreads=0):
    """Drafter-side sampling on fp32 rows q [B, K, V] (reading R13)."""
    q = _c(q, np.float32)
    B, K, _ = q.shape
    return _draft_sample(_load().oracle_draft_sample_probs, q, B, K, temperature, seed, req_ids,
                         nthreads)


def draft_sample_logits(logit_bits, temperature=None, seed=0, req_ids=None, nthreads=0):
    """Drafter-side sampling on bf16 logit rows [B, K, V] given as uint16 bit patterns."""
    lb = _c(logit_bits, np.uint16)
    B, K, _ = lb.shape
    return _draft_sample(_load().oracle_draft_sample_logits, lb, B, K, temperature, seed,
                         req_ids, nthreads)


def verify_ragged(target, draft, drafts, cu, K_max, temperature=None, seed=0, logits=False,
                  req_base=0, nthreads=0):
    """Verify with a draft count per request: request r has K_r = cu[r+1] - cu[r] drafts, target
    rows cu[r] + r .. cu[r] + r + K_r, draft rows and tokens cu[r] .. cu[r] + K_r - 1. Each
    request is verified on its own, by the batch oracle with K = K_r and its own request index
    (requests with equal K_r in one call). Outputs are padded to K_max like the library's."""
    cu = np.asarray(cu, np.int64)
    B = len(cu) - 1
    ks = cu[1:] - cu[:-1]
    out = dict(out_tokens=np.full((B, K_max + 1), -1, np.int32),
               num_accepted=np.zeros(B, np.int32),
               p_at_draft=np.full((B, K_max), -1.0, np.float32),
               q_at_draft=np.full((B, K_max), -1.0, np.float32),
               accept_margin=np.full((B, K_max), -1.0), race_margin=np.zeros(B), err=0)
    temp = None if temperature is None else np.asarray(temperature, np.float32)
    for k in sorted(set(ks.tolist())):
        idx = np.nonzero(ks == k)[0]
        t = np.stack([target[cu[r] + r: cu[r] + r + k + 1] for r in idx])
        d = (np.stack([draft[cu[r]: cu[r] + k] for r in idx]) if k > 0
             else np.zeros((len(idx), 0, target.shape[1]), target.dtype))
        dr = (np.stack([drafts[cu[r]: cu[r] + k] for r in idx]) if k > 0
              else np.zeros((len(idx), 0), np.int32))
        T = None if temp is None else temp[idx]
        rid = (idx + req_base).astype(np.int32)
        if logits:
            res = verify_logits(t, d, dr, temperature=T, seed=seed, req_ids=rid,
                                nthreads=nthreads, margins=True)
        else:
            res = verify_probs(t, d, dr, temperature=T, seed=seed, req_ids=rid,
                               nthreads=nthreads)
        out["out_tokens"][idx, :k + 1] = res["out_tokens"]
        out["num_accepted"][idx] = res["num_accepted"]
        out["p_at_draft"][idx, :k] = res["p_at_draft"]
        out["q_at_draft"][idx, :k] = res["q_at_draft"]
        if logits:
            out["accept_margin"][idx, :k] = res["accept_margin"]
            out["race_margin"][idx] = res["race_margin"]
        out["err"] |= res["err"]
    return out


def pdraft_expand(out_tokens, num_accepted, pos0, block_table, block_size, mask_token_id,
                  capacity=None, cu=None):
    """Drafter-batch rebuild; cu (optional [B+1]): per-request draft counts (reading R17)."""
    out_tokens = _c(out_tokens, np.int32)
    num_accepted = _c(num_accepted, np.int32)
    pos0 = _c(pos0, np.int32)
    block_table = _c(block_table, np.int32)
    B, K1 = out_tokens.shape
    K = K1 - 1
    cap = B * 2 * K if capacity is None else capacity
    o = dict(input_ids=np.zeros(cap, np.int32), positions=np.zeros(cap, np.int32),
             slot_mapping=np.zeros(cap, np.int32), hidden_map=np.zeros(cap, np.int32),
             is_masked=np.zeros(cap, np.uint8), is_rejected=np.zeros((B, K + 1), np.uint8),
             start_loc=np.zeros(B + 1, np.int32), new_token_idx=np.zeros((B, K), np.int32),
             total_out=np.zeros(1, np.int32))
    err = np.zeros(1, np.int32)
    rc = _load().oracle_pdraft_expand(
        B, K, _ptr(out_tokens), _ptr(num_accepted), _ptr(pos0), _ptr(block_table),
        block_table.shape[1] if block_table.ndim == 2 else 0, block_size, mask_token_id, cap,
        _ptr(o["input_ids"]), _ptr(o["positions"]), _ptr(o["slot_mapping"]),
        _ptr(o["hidden_map"]), _ptr(o["is_masked"]), _ptr(o["is_rejected"]),
        _ptr(o["start_loc"]), _ptr(o["new_token_idx"]), _ptr(o["total_out"]), _ptr(err),
        _ptr(None if cu is None else _c(cu, np.int32)))
    if rc != 0:
        raise ValueError(f"oracle expand rejected its arguments (rc={rc})")
    o["err"] = int(err[0])
    return o


def pdraft_prepare_padded(out_tokens, num_accepted, pos0, block_table, block_size, mask_token_id,
                          target_hidden_bits, h_shared_bits):
    """Padded drafter batch (reading R14): B rows of 2K slots, every output row written."""
    out_tokens = _c(out_tokens, np.int32)
    num_accepted = _c(num_accepted, np.int32)
    pos0 = _c(pos0, np.int32)
    block_table = _c(block_table, np.int32)
    th = _c(target_hidden_bits, np.uint16)
    hs = _c(h_shared_bits, np.uint16)
    B, K1 = out_tokens.shape
    K = K1 - 1
    n = B * 2 * K
    H = hs.shape[-1]
    o = dict(input_ids=np.zeros(n, np.int32), positions=np.zeros(n, np.int32),
             slot_mapping=np.zeros(n, np.int32), hidden_map=np.zeros(n, np.int32),
             is_masked=np.zeros(n, np.uint8), rejected=np.zeros(n, np.uint8),
             scatter_map=np.zeros(B * K1, np.int32), new_token_idx=np.zeros((B, K), np.int32),
             out_hidden=np.zeros((n, H), np.uint16))
    err = np.zeros(1, np.int32)
    rc = _load().oracle_pdraft_prepare_padded(
        B, K, _ptr(out_tokens), _ptr(num_accepted), _ptr(pos0), _ptr(block_table),
        block_table.shape[1] if block_table.ndim == 2 else 0, block_size, mask_token_id,
        _ptr(o["input_ids"]), _ptr(o["positions"]), _ptr(o["slot_mapping"]),
        _ptr(o["hidden_map"]), _ptr(o["is_masked"]), _ptr(o["rejected"]), _ptr(o["scatter_map"]),
        _ptr(o["new_token_idx"]), H, _ptr(th), H, th.shape[0], _ptr(hs), _ptr(o["out_hidden"]), H,
        _ptr(err))
    if rc != 0:
        raise ValueError(f"oracle padded rebuild rejected its arguments (rc={rc})")
    o["err"] = int(err[0])
    return o


def hidden_gather(total_out, hidden_map, target_hidden_bits, h_shared_bits, capacity=None,
                  out_init=None):
    """Gather bf16 rows (given as uint16 bit patterns)."""
    hidden_map = _c(hidden_map, np.int32)
    th = _c(target_hidden_bits, np.uint16)
    hs = _c(h_shared_bits, np.uint16)
    H = hs.shape[-1]
    cap = hidden_map.shape[0] if capacity is None else capacity
    out = (np.zeros((cap, H), np.uint16) if out_init is None
           else np.array(out_init, dtype=np.uint16, copy=True))
    tot = np.array([total_out], np.int32)
    err = np.zeros(1, np.int32)
    rc = _load().oracle_hidden_gather(cap, H, _ptr(tot), _ptr(hidden_map), _ptr(th), H,
                                      th.shape[0], _ptr(hs), _ptr(out), H, _ptr(err))
    if rc != 0:
        raise ValueError(f"oracle gather rejected its arguments (rc={rc})")
    return out, int(err[0])
