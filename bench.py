"""Benchmark: one decoding step's verify + draft-batch rebuild on one GB300 (or N replicas).

A step is sd_verify followed by sd_pdraft_prepare (the draft-batch rebuild and the hidden-state
gather, launched as a programmatic dependent of verify) on one batch of synthetic inputs already
resident in HBM. W warm-up steps, then exactly K timed steps replayed from CUDA graphs that rotate
over several input sets (whose rows together exceed the 129 MB L2). Prints one JSON line
(rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config b1024lg] [--impl gb300|reference]

The timed workload is b1024lg (B=1024, K=8, V=201088 bf16 logits, the largest configuration);
b64, b256mix and b512rag are then timed the same way in the same process and reported under
"configs". --impl reference times the plain CPU oracle (the baseline this library is checked
against) on the host cores for the same workload, inputs and metric.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify+draft-prep requests/s at 1 GB300; achieved HBM GB/s vs roofline"
L2_BYTES = 129 * 1024 * 1024

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the verify kernel, from one ncu
# capture, keyed by workload and by the hash of the kernel source it was taken on (the number is
# reported only while the source is unchanged).
# Captures of a reduced batch are scaled to the full batch by the units processed (the kernels'
# traffic grows in proportion to the requests).
MEASURED_TRAFFIC = {
    ("b64", "c8fd3a12768eb5f3"): (90.784256e6, "ncu --set full, one fused launch of the full "
                                               "batch (one input set)"),
    ("b256mix", "c8fd3a12768eb5f3"): (432.580096e6, "ncu --set full at B=128, scaled x2"),
    ("b512rag", "c8fd3a12768eb5f3"): (784.234496e6, "ncu --set full at B=192, scaled x512/192"),
    ("b1024lg", "c8fd3a12768eb5f3"): (3670.736896e6, "ncu --set full at B=192, scaled x1024/192"),
}


def _src_hash():
    h = hashlib.sha256()
    for f in ("sd_verify.cu", "sd_common.cuh", "sd_rebuild.cuh"):
        with open(os.path.join(ROOT, "verify_draft_prep_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def philox_peak():
    """Philox4x32-10 blocks per second the GPU's integer multipliers allow, from unit counts and
    the clock: each block takes 20 32x32->64-bit products (two per round), each product two
    operations of an SM's 64 integer-multiply lanes per clock; 152 SMs at the maximum SM clock
    (MEASURED_PEAKS.json, else 2070 MHz)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f)["sm_max_mhz"])
    except Exception:
        mhz = 2070.0
    return 152 * mhz * 1e6 * 64 / (20 * 2)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def algorithmic_bytes(w, a):
    """Bytes the method must move per step, from the accepted counts a (numpy [B]): verify (the
    roofline's model), expand, gather, and verify counting only the rows the kernel must read.

    Probability rows use the minimum-bytes model: the scalar gathers of the accept scan plus one p
    and one q row at the first rejection (only p when every draft is accepted), or the a_r + 1
    rows a greedy request scans. Logit rows use the full-row model (every target and draft row of
    the request, 2K + 1 rows), the roofline stated for the fused-softmax variant; the kernel
    itself reads rows lazily (rows 0..a_r of both, and never the rows after the first
    rejection), which the fourth figure counts."""
    import torch

    B, K, V, H = w.B, w.K, w.V, w.H
    T = w.temperature.cpu().numpy()
    greedy = T == 0
    esz = 4 if w.kind == "probs" else 2
    a = a.astype(np.int64)
    scalars = 4 * K + 4 * (K + 2) + 4  # drafts, out_tokens + num_accepted, temperature
    if w.kind == "probs":
        rows = np.where(greedy, a + 1, np.where(a < K, 2, 1))
        gathers = np.where(greedy, 0, 2 * 32 * np.minimum(a + 1, K))
        verify = verify_read = int((rows * esz * V + gathers + scalars).sum())
    else:
        verify = int(B * ((2 * K + 1) * esz * V + scalars))
        rows_read = np.where(greedy, a + 1, (a + 1) + np.minimum(a + 1, K))
        verify_read = int((rows_read * esz * V + scalars).sum())
    blocks = (2 * K) // w.block_size + 2
    expand = int((4 * (K + 4) + 4 * blocks + (a + K) * 17 + (K + 1) + 4 * K).sum())
    gather = int(((a + 1) * 2 * H + (a + K) * 2 * H).sum()) + 2 * H
    del torch
    return verify, expand, gather, verify_read


def sample_roofline(w, avg_ms, sample_bytes, peak):
    """The drafter-side sampler against both of its bounds: HBM (every row read once) and the
    integer multipliers (one Philox4x32-10 block per 4 entries of every sampled row, the race's
    variates). The binding one is the bound whose time is longer."""
    rows = w.B * w.K
    blocks = rows * ((w.V + 3) // 4)
    pk_alu = philox_peak()
    t_hbm, t_alu = sample_bytes / (peak * 1e9), blocks / pk_alu
    hbm = {"achieved_GBps": sample_bytes / (avg_ms * 1e-3) / 1e9,
           "frac": sample_bytes / (avg_ms * 1e-3) / 1e9 / peak}
    alu = {"philox_blocks_per_launch": blocks,
           "achieved_blocks_per_s": blocks / (avg_ms * 1e-3), "peak_blocks_per_s": pk_alu,
           "frac": blocks / (avg_ms * 1e-3) / pk_alu,
           "peak_source": "unit counts: 152 SMs x max SM clock x 64 multiply lanes / 40 lane "
                          "operations per block"}
    bound = "alu" if t_alu > t_hbm else "hbm"
    return {"kernel": "sd_draft_sample", "us": avg_ms * 1e3, "bound": bound,
            "frac": (alu if bound == "alu" else hbm)["frac"], "bytes_per_launch": sample_bytes,
            "achieved_GBps": hbm["achieved_GBps"], "hbm_frac": hbm["frac"], "alu": alu}


def make_set(cfg_name, s, device, rank, batch=None):
    """Input set s of a workload on this rank (set 0 is also what the oracle baselines time)."""
    import workloads

    idx = [c["name"] for c in workloads.CONFIGS].index(cfg_name)
    return workloads.make(idx, device=device, gen_seed=1000 + idx + 101 * s + 7919 * rank,
                          B=batch)


def alloc_outputs(w, device):
    import torch

    B, K, cap = w.B, w.K, w.capacity
    i32 = dict(dtype=torch.int32, device=device)
    return dict(out_tokens=torch.empty(B, K + 1, **i32), num_accepted=torch.empty(B, **i32),
                next_drafts=torch.empty(B, K, **i32),
                pad_ids=torch.empty(B * 2 * K, **i32), pad_pos=torch.empty(B * 2 * K, **i32),
                pad_slot=torch.empty(B * 2 * K, **i32), pad_map=torch.empty(B * 2 * K, **i32),
                pad_masked=torch.empty(B * 2 * K, dtype=torch.uint8, device=device),
                pad_rej=torch.empty(B * 2 * K, dtype=torch.uint8, device=device),
                pad_scatter=torch.empty(B * (K + 1), **i32), pad_nti=torch.empty(B, K, **i32),
                pad_hidden=torch.empty(B * 2 * K, w.H, dtype=torch.bfloat16, device=device),
                input_ids=torch.empty(cap, **i32), positions=torch.empty(cap, **i32),
                slot_mapping=torch.empty(cap, **i32), hidden_map=torch.empty(cap, **i32),
                is_masked=torch.empty(cap, dtype=torch.uint8, device=device),
                is_rejected=torch.empty(B, K + 1, dtype=torch.uint8, device=device),
                start_loc=torch.empty(B + 1, **i32), new_token_idx=torch.empty(B, K, **i32),
                total_out=torch.empty(1, **i32),
                out_hidden=torch.empty(cap, w.H, dtype=torch.bfloat16, device=device),
                err=torch.zeros(1, **i32),
                ws=torch.zeros(max(16, 16 * B), dtype=torch.uint8, device=device))


def temperatures(w):
    """The workload's temperatures, or None when every request samples at T = 1 (the library
    then needs no per-request temperature and launches only its sampling kernel)."""
    if not hasattr(w, "_temp_arg"):
        w._temp_arg = None if bool((w.temperature == 1.0).all()) else w.temperature
    return w._temp_arg


def launch_step(sd, w, o, stream=None):
    """One step through sd_verify_prepare: verify and the draft-batch rebuild + hidden gather in
    one launch when every request samples on probability rows and the batch fits one wave, else
    the verify kernel and the rebuild kernel (its programmatic dependent)."""
    sd.sd_verify_prepare(w.target, w.draft, w.drafts, o["out_tokens"], o["num_accepted"], w.pos0,
                         w.block_table, w.block_size, w.mask_token_id, o["input_ids"],
                         o["positions"], o["slot_mapping"], o["hidden_map"], o["is_masked"],
                         o["is_rejected"], o["start_loc"], o["new_token_idx"], o["total_out"],
                         w.hidden, w.h_shared, o["out_hidden"], temperature=temperatures(w),
                         seed=w.seed, err=o["err"], stream=stream, workspace_buf=o["ws"],
                         request_base=getattr(w, "request_base", 0))


def launch_prepare(sd, w, o, stream=None):
    sd.sd_pdraft_prepare(o["out_tokens"], o["num_accepted"], w.pos0, w.block_table, w.block_size,
                         w.mask_token_id, o["input_ids"], o["positions"], o["slot_mapping"],
                         o["hidden_map"], o["is_masked"], o["is_rejected"], o["start_loc"],
                         o["new_token_idx"], o["total_out"], w.hidden, w.h_shared,
                         o["out_hidden"], err=o["err"], stream=stream)


def launch_verify(sd, w, o, stream=None):
    # request_base: this rank's shard starts at request rank * B of the job's global batch
    sd.sd_verify(w.target, w.draft, w.drafts, o["out_tokens"], o["num_accepted"],
                 temperature=temperatures(w), seed=w.seed, err=o["err"], stream=stream,
                 workspace_buf=o["ws"], request_base=getattr(w, "request_base", 0))


def launch_draft_sample(sd, w, o, stream=None):
    # the config's draft rows stand in for the drafter's outputs at new_token_idx
    sd.sd_draft_sample(w.draft, o["next_drafts"], temperature=temperatures(w), seed=w.seed + 1,
                       request_base=getattr(w, "request_base", 0), err=o["err"], stream=stream)


def launch_prepare_padded(sd, w, o, stream=None):
    sd.sd_pdraft_prepare_padded(o["out_tokens"], o["num_accepted"], w.pos0, w.block_table,
                                w.block_size, w.mask_token_id, o["pad_ids"], o["pad_pos"],
                                o["pad_slot"], o["pad_map"], o["pad_masked"], o["pad_rej"],
                                o["pad_scatter"], o["pad_nti"], target_hidden=w.hidden,
                                h_shared=w.h_shared, out_hidden=o["pad_hidden"], err=o["err"],
                                stream=stream)


def launch_verify_prepare_padded(sd, w, o, stream=None):
    """The step with the padded drafter batch in one call (one launch for an all-sampled batch
    of one wave)."""
    sd.sd_verify_prepare_padded(w.target, w.draft, w.drafts, o["out_tokens"], o["num_accepted"],
                                w.pos0, w.block_table, w.block_size, w.mask_token_id,
                                o["pad_ids"], o["pad_pos"], o["pad_slot"], o["pad_map"],
                                o["pad_masked"], o["pad_rej"], o["pad_scatter"], o["pad_nti"],
                                target_hidden=w.hidden, h_shared=w.h_shared,
                                out_hidden=o["pad_hidden"], temperature=temperatures(w),
                                seed=w.seed, err=o["err"], stream=stream, workspace_buf=o["ws"],
                                request_base=getattr(w, "request_base", 0))


def time_graph(fn, sets, outs, stream, K):
    """Average duration (ms) of K launches of `fn`, rotating over the input sets, replayed
    from one CUDA graph."""
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for s in range(K):
                fn(sets[s % len(sets)], outs[s % len(sets)], stream)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record(stream)
        g.replay()
        b.record(stream)
    stream.synchronize()
    return a.elapsed_time(b) / K


def oracle_pass(hc, nthreads):
    """One pass of the oracle over every request of the host copy hc: verify, expand, gather."""
    import oracle

    if hc["kind"] == "probs":
        res = oracle.verify_probs(hc["target"], hc["draft"], hc["drafts"],
                                  temperature=hc["temperature"], seed=0, nthreads=nthreads)
    else:
        res = oracle.verify_logits(hc["target"], hc["draft"], hc["drafts"],
                                   temperature=hc["temperature"], seed=0, nthreads=nthreads,
                                   margins=False)
    e = oracle.pdraft_expand(res["out_tokens"], res["num_accepted"], hc["pos0"],
                             hc["block_table"], hc["block_size"], hc["mask"])
    oracle.hidden_gather(int(e["total_out"][0]), e["hidden_map"], hc["hidden"], hc["h_shared"])


def first_requests(hc, n):
    """The first n requests of a host copy (a bounded sample of the batch)."""
    K = hc["K"]
    out = dict(hc)
    for k in ("target", "draft", "drafts", "temperature", "pos0", "block_table"):
        out[k] = hc[k][:n]
    out["hidden"] = hc["hidden"][:n * (K + 1)]
    out["B"] = n
    return out


def oracle_rate(hc, nthreads, budget_s, max_passes=100000):
    """Requests/s of the oracle (as it stands) on hc: whole passes until budget_s has elapsed."""
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle_pass(hc, nthreads)
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s or passes >= max_passes:
            return hc["B"] * passes / el, passes, el


def sized_sample(hc, nthreads, seconds):
    """The largest prefix of the batch whose oracle pass takes about `seconds` (measured on a
    probe of a few requests per thread), at least one request."""
    n = min(hc["B"], max(1, 2 * max(1, nthreads)))
    probe = first_requests(hc, n)
    t0 = time.perf_counter()
    oracle_pass(probe, nthreads)
    per_pass = time.perf_counter() - t0
    # requests are spread over the threads: a pass of m requests takes ~ceil(m/threads) rounds
    per_round = per_pass / max(1, -(-n // max(1, nthreads)))
    m = int(seconds / max(per_round, 1e-9)) * max(1, nthreads)
    return first_requests(hc, max(1, min(hc["B"], m)))


def run_cpu_baseline(hc, budget_s=10.0, single_s=4.0):
    """The oracle (as it stands) on this process's host cores, on the same inputs as the GPU
    (set 0 of the timed workload): all cores over whole passes of the batch, then one thread on
    a bounded prefix of it."""
    cores = len(os.sched_getaffinity(0))
    sample = sized_sample(hc, cores, budget_s / 2) if hc["B"] > 1 else hc
    v, passes, el = oracle_rate(sample, cores, budget_s)
    one = sized_sample(hc, 1, single_s / 2)
    v1, passes1, el1 = oracle_rate(one, 1, single_s)
    return {"value": v, "unit": "requests/s", "cores": cores, "kind": "oracle",
            "sample": f"{passes} passes over the first {sample['B']} of the batch's {hc['B']} "
                      f"requests (set 0 of the timed inputs; verify + expand + gather) on "
                      f"{cores} threads, {el:.1f} s",
            "single_thread": {"value": v1, "unit": "requests/s", "cores": 1,
                              "sample": f"{passes1} passes over the first {one['B']} requests on "
                                        f"one thread, {el1:.1f} s"}}


def host_copy(w):
    import torch

    B, K, V = w.B, w.K, w.V
    bits = lambda t: t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    if w.kind == "probs":
        tgt = w.target.view(B, K + 1, V).cpu().numpy()
        dft = w.draft.view(B, K, V).cpu().numpy()
    else:
        tgt = bits(w.target).reshape(B, K + 1, V)
        dft = bits(w.draft).reshape(B, K, V)
    return dict(B=B, K=K, V=V, kind=w.kind, target=tgt, draft=dft,
                drafts=w.drafts.cpu().numpy(), temperature=w.temperature.cpu().numpy(),
                pos0=w.pos0.cpu().numpy(), block_table=w.block_table.cpu().numpy(),
                block_size=w.block_size, mask=w.mask_token_id, hidden=bits(w.hidden),
                h_shared=bits(w.h_shared))


# The configurations measured besides the timed one (every configuration of the bar on one
# record); the launch-bound one-request case is a parity case only.
EXTRA_CONFIGS = ("b64", "b256mix", "b512rag")


def config_dict(cfg, B, nsets, rows_gb, world, batch):
    import workloads

    return {"workload": workloads.config_label(cfg) + (
                f" [reduced to B={B} for profiling]" if batch else ""),
            "B": B, "K": cfg["K"], "V": cfg["V"], "H": cfg["H"],
            "l2": f"{nsets} rotating input sets (rows of all sets {rows_gb:.1f} GB > 129 MB L2; "
                  f"a set recurs after {nsets - 1} others)",
            "timing": "CUDA graphs of the timed steps, one sd_verify_prepare call each (one "
                      "launch when the batch is all-sampled and fits one wave, else verify then "
                      "the rebuild as its programmatic dependent); the dominant kernel alone in "
                      "a second graph for the roofline",
            "parallelism": f"dp{world}: request shards of {B} per GPU"}


def n_sets(cfg):
    return 4 if cfg["B"] * cfg["V"] < 64 * 201088 * 2 else 2


def measure(name, args, sd, device, rank, world, steps, keep_set0=False):
    """Time `steps` steps of one workload (W warm-up steps first) and its kernels; returns the
    figures (and set 0 when keep_set0, for the end-to-end and oracle legs)."""
    import torch
    import torch.distributed as dist

    import workloads
    from verify_draft_prep_gb300 import shard

    cfg = [c for c in workloads.CONFIGS if c["name"] == name][0]
    batch = args.batch or None
    nsets = args.sets or n_sets(cfg)
    sets = [make_set(name, s, device, rank, batch) for s in range(nsets)]
    outs = [alloc_outputs(w, device) for w in sets]
    for w in sets:
        temperatures(w)  # decided before any graph capture (it reads the device)
        # each rank holds its own shard of the job's batch: requests rank*B .. rank*B + B - 1 in
        # the Philox counters (weak scaling, no exchange on the data path)
        w.request_base = shard.request_base(w.B)[0] if world > 1 else 0

    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            launch_step(sd, sets[i % nsets], outs[i % nsets], stream)
    stream.synchronize()

    # the timed steps are replayed from CUDA graphs of up to CHUNK steps (a graph of K % CHUNK
    # steps makes up the rest, so exactly K steps run); the timed region is bracketed by two
    # events (per-step events only with --step-events)
    K = steps
    CHUNK = min(K, 200)

    def capture(n, with_events):
        evs_ = None
        if with_events:
            try:
                evs_ = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n + 1)]
            except TypeError:
                evs_ = None
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for s in range(n):
                    if evs_:
                        evs_[s].record(stream)
                    launch_step(sd, sets[s % nsets], outs[s % nsets], stream)
                if evs_:
                    evs_[n].record(stream)
        with torch.cuda.stream(stream):
            g.replay()  # one untimed replay (graph upload)
        stream.synchronize()
        return g, evs_

    graph, evs = capture(CHUNK, args.step_events)
    full, rest = divmod(K, CHUNK)
    graph_rest = capture(rest, False)[0] if rest else None

    clocks = ClockSampler(int(str(device).split(":")[-1]))
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):  # graphs replay on the current stream
        start.record(stream)
        for _ in range(full):
            graph.replay()
        if graph_rest is not None:
            graph_rest.replay()
        end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    total_ms = start.elapsed_time(end)
    # bytes per step from each set's accepted counts (every set has run by now: the graphs
    # rotate over all of them; the same inputs give the same counts on every run)
    per_set = []
    for w, o in zip(sets, outs):
        a = o["num_accepted"].cpu().numpy()
        per_set.append(algorithmic_bytes(w, a)[:3] + (a, algorithmic_bytes(w, a)[3]))
    errs = [int(o["err"].item()) for o in outs]
    step_ms = [evs[s].elapsed_time(evs[s + 1]) for s in range(CHUNK)] if evs else []
    # the dominant kernel alone, CHUNK launches in a graph of its own, right after the timed
    # region: the fused step kernel when the step is one launch, else the verify kernel
    dt_code = 0 if cfg["kind"] == "probs" else 1
    has_t = temperatures(sets[0]) is not None
    step_kernels = sd.sd_verify_prepare_kernels(sets[0].B, sets[0].K, sets[0].V, dt_code, has_t)
    fused = step_kernels == 1
    avg_f = time_graph(lambda w, o, st: launch_step(sd, w, o, st), sets, outs, stream,
                       CHUNK) if fused else None
    avg_v = time_graph(lambda w, o, st: launch_verify(sd, w, o, st), sets, outs, stream, CHUNK)
    avg_p = time_graph(lambda w, o, st: launch_prepare(sd, w, o, st), sets, outs, stream, CHUNK)
    # the padded form of the rebuild (fixed 2K-slot rows), timed alone after the same verify
    avg_pp = time_graph(lambda w, o, st: launch_prepare_padded(sd, w, o, st), sets, outs, stream,
                        CHUNK)
    # ... and the whole step with the padded batch through the one call, against the same step
    # as the two calls (sd_verify, then sd_pdraft_prepare_padded) back to back
    avg_vpp = time_graph(lambda w, o, st: launch_verify_prepare_padded(sd, w, o, st), sets, outs,
                         stream, CHUNK)
    avg_v2p = time_graph(lambda w, o, st: (launch_verify(sd, w, o, st),
                                           launch_prepare_padded(sd, w, o, st)), sets, outs,
                         stream, CHUNK)
    # the next row of the method: drafter-side sampling of the K new drafts, timed alone
    avg_s = time_graph(lambda w, o, st: launch_draft_sample(sd, w, o, st), sets, outs, stream,
                       CHUNK)
    if world > 1:
        t = torch.tensor([total_ms], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())

    B = sets[0].B
    ms_per_step = total_ms / K
    value = shard.whole_job_rate(B * K, world, total_ms)
    bytes_v = float(np.mean([per_set[s % nsets][0] for s in range(CHUNK)]))
    bytes_read = float(np.mean([per_set[s % nsets][4] for s in range(CHUNK)]))
    # the rebuild's and the gather's bytes, and the step's: verify counted by the rows it must read
    bytes_rest = float(np.mean([sum(per_set[s % nsets][1:3]) for s in range(CHUNK)]))
    bytes_all = bytes_read + bytes_rest
    peak, peak_kind = _peaks()
    # roofline of the dominant kernel: the fused step kernel moves the verify's, the expand's and
    # the gather's bytes; the verify kernel alone the rows it must read (for probability rows the
    # minimum-bytes model; for logit rows the rows up to the first rejection, the least any exact
    # verify reads; the full-row model of every logit row is reported beside it)
    bytes_dom = bytes_all if fused else bytes_read
    avg_dom = avg_f if fused else avg_v
    achieved = bytes_dom / (avg_dom * 1e-3) / 1e9
    traffic, traffic_note = (None, "no capture of the current kernel source")
    if not args.batch and (name, _src_hash()) in MEASURED_TRAFFIC:
        traffic, traffic_note = MEASURED_TRAFFIC[(name, _src_hash())]
    a_all = np.concatenate([p[3] for p in per_set])
    w0s = sets[0]
    sample_bytes = w0s.B * w0s.K * w0s.V * w0s.draft.element_size() + w0s.B * w0s.K * 4 + w0s.B * 4
    pad_bytes = float(np.mean([
        int(((per_set[s % nsets][3] + 1) * 2 * w0s.H).sum()) + w0s.B * 2 * w0s.K * (2 * w0s.H + 18)
        + w0s.B * (w0s.K + 1) * 4 + w0s.B * w0s.K * 4 for s in range(CHUNK)]))
    rows_gb = nsets * w0s.target.numel() * w0s.target.element_size() / 1e9
    logits = cfg["kind"] != "probs"
    roofline = {
        "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
        "frac": achieved / peak, "traffic": traffic, "traffic_source": traffic_note,
        "kernel": "sd_verify_prepare (verify and rebuild in one launch)" if fused else "sd_verify",
        "kernel_us": avg_dom * 1e3, "peak_source": peak_kind,
        "algorithmic_bytes_per_launch": bytes_dom,
        "bytes_model": ("minimum bytes (scalar gathers + one p and one q row per sampled request, "
                        "a_r + 1 rows per greedy one)" if not logits else
                        "rows up to the first rejection (a_r + 1 target and min(a_r + 1, K) draft "
                        "logit rows per request) + scalars")
        + ("; plus the rebuild's slots and hidden rows" if fused else ""),
        "verify_alone": {"us": avg_v * 1e3, "bytes": bytes_read,
                         "frac": bytes_read / (avg_v * 1e-3) / 1e9 / peak},
        # the verify kernel against the bytes it must read (rows up to the first rejection):
        # its own efficiency, whatever the roofline model of the variant
        "frac_rows_read": (bytes_read / (avg_v * 1e-3) / 1e9) / peak,
        "rows_read_bytes": bytes_read,
        "step_frac": (bytes_all / (ms_per_step * 1e-3) / 1e9) / peak,
    }
    if logits:
        # the full-row model (every target and draft logit row of every request, 2K + 1 rows):
        # bytes no lazy verify reads, so this fraction can exceed 1
        roofline["full_row"] = {"bytes": bytes_v, "frac": bytes_v / (avg_v * 1e-3) / 1e9 / peak,
                                "step_frac": (bytes_v + bytes_rest)
                                / (ms_per_step * 1e-3) / 1e9 / peak}
    res = {
        "cfg": cfg, "B": B, "steps": K, "value": value, "ms_per_step": ms_per_step,
        "launches": step_kernels, "clocks": clk, "roofline": roofline,
        "config": config_dict(cfg, B, nsets, rows_gb, world, batch),
        "dtype": "f32" if not logits else "bf16",
        "draft_sample": dict(sample_roofline(w0s, avg_s, sample_bytes, peak),
                             rows=f"B*K = {w0s.B * w0s.K} rows of V = {w0s.V}, each read once "
                                  "from HBM"),
        "prepare_padded": {"kernel": "sd_pdraft_prepare_padded", "us": avg_pp * 1e3,
                           "bytes_per_launch": pad_bytes,
                           "achieved_GBps": pad_bytes / (avg_pp * 1e-3) / 1e9,
                           "frac": pad_bytes / (avg_pp * 1e-3) / 1e9 / peak,
                           "rows": f"B*2K = {w0s.B * 2 * w0s.K} drafter rows, every one written "
                                   "(hidden states read for the a_r + 1 target rows of each "
                                   "request)",
                           # the step with this batch in one call (sd_verify_prepare_padded):
                           # the verify's bytes and the padded rebuild's
                           "step_one_call": {
                               "us": avg_vpp * 1e3,
                               "two_calls_us": avg_v2p * 1e3,
                               "each_alone_us": (avg_v + avg_pp) * 1e3,
                               "launches": sd.sd_verify_prepare_kernels(
                                   w0s.B, w0s.K, w0s.V, dt_code, has_t),
                               "frac": (bytes_read + pad_bytes) / (avg_vpp * 1e-3) / 1e9 / peak}},
        "info": {"verify_ms": avg_v, "prepare_ms": avg_p,
                 "step_ms_median": float(np.median(step_ms)) if step_ms else None,
                 "step_bytes": bytes_all,
                 "step_GBps": bytes_all / (ms_per_step * 1e-3) / 1e9,
                 "mean_accepted": float(a_all.mean()), "err": errs},
    }
    if keep_set0:
        res["set0"] = sets[0]
    del sets, outs, graph, graph_rest
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def summary(r, cpu=None):
    """The figures of one configuration in the record's per-configuration table."""
    rf = r["roofline"]
    out = {"workload": r["config"]["workload"], "value": r["value"], "unit": "requests/s",
           "ms_per_step": r["ms_per_step"], "steps": r["steps"],
           "gpu_launches": r["launches"] * r["steps"],
           "kernel": rf["kernel"], "kernel_us": rf["kernel_us"], "frac": rf["frac"],
           "frac_rows_read": rf["frac_rows_read"], "step_frac": rf["step_frac"],
           "verify_alone": rf["verify_alone"], "traffic": rf["traffic"],
           "algorithmic_bytes_per_launch": rf["algorithmic_bytes_per_launch"],
           "bytes_model": rf["bytes_model"], "clocks": r["clocks"],
           "mean_accepted": r["info"]["mean_accepted"], "err": r["info"]["err"],
           "draft_sample": r["draft_sample"], "prepare_padded": r["prepare_padded"]}
    if cpu is not None:
        out["cpu_baseline"] = cpu
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="b1024lg")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--sets", type=int, default=0, help="input sets to rotate (0: auto)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="time only --config (not the other configurations)")
    ap.add_argument("--batch", type=int, default=0,
                    help="profiling aid: the config's shapes with this many requests (0: as "
                         "configured); a line with a reduced batch is not the config's number")
    ap.add_argument("--step-events", action="store_true",
                    help="record an event at every step boundary (per-step times; the event "
                         "nodes break the programmatic launch edge between steps)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if args.impl == "gb300" else "gloo")

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, world)
        if world > 1:
            dist.destroy_process_group()
        return

    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    import verify_draft_prep_gb300 as sd

    sd.load()

    main_res = measure(args.config, args, sd, device, rank, world, args.steps, keep_set0=True)
    w0 = main_res.pop("set0")
    # end to end through the public API: pinned host inputs -> device, step, results -> host
    e2e = run_e2e(sd, w0, device, args.e2e_steps)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline(host_copy(w0))
    del w0
    torch.cuda.empty_cache()

    # the other configurations of the bar, each timed the same way in this process
    extras = {}
    if not args.no_extra and not args.batch:
        for name in EXTRA_CONFIGS:
            if name == args.config:
                continue
            r = measure(name, args, sd, device, rank, world, args.steps, keep_set0=rank == 0
                        and not args.no_cpu_baseline)
            c = None
            if "set0" in r:
                c = run_cpu_baseline(host_copy(r.pop("set0")), budget_s=3.0, single_s=1.5)
                torch.cuda.empty_cache()
            extras[name] = summary(r, c)

    print(json.dumps({"info": main_res["info"]}), file=sys.stderr)
    if rank == 0:
        K = args.steps
        line = {
            "metric": METRIC, "value": main_res["value"], "unit": "requests/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": main_res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": main_res["dtype"], "data": "synthetic", "config": main_res["config"],
            "roofline": main_res["roofline"], "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": main_res["launches"] * K, "clocks": main_res["clocks"],
            "draft_sample": main_res["draft_sample"],
            "prepare_padded": main_res["prepare_padded"],
            "configs": extras,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_e2e(sd, w, device, steps):
    """Same metric through the public API with host buffers: each step copies its inputs from
    pinned host memory, runs the three calls, and reads every result back."""
    import torch

    ins = {k: getattr(w, k) for k in ("target", "draft", "drafts", "temperature", "pos0",
                                      "block_table", "hidden", "h_shared")}
    host = {k: v.cpu().pin_memory() for k, v in ins.items()}
    dev = {k: torch.empty_like(v) for k, v in ins.items()}
    o = alloc_outputs(w, device)
    res_keys = ("out_tokens", "num_accepted", "input_ids", "positions", "slot_mapping",
                "hidden_map", "is_masked", "is_rejected", "start_loc", "new_token_idx",
                "total_out", "out_hidden")
    back = {k: torch.empty(o[k].shape, dtype=o[k].dtype, pin_memory=True) for k in res_keys}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in back.values())

    class W:
        pass

    wd = W()
    for k, v in vars(w).items():
        setattr(wd, k, v)
    for k, v in dev.items():
        setattr(wd, k, v)
    if getattr(w, "_temp_arg", None) is not None:
        wd._temp_arg = dev["temperature"]  # the copy made inside each step, not set 0's tensor
    stream = torch.cuda.Stream(device)
    # host->device copies spread over several streams (several copy engines on the host link):
    # the large row arrays in row chunks, round-robin; the step's kernels wait for all of them,
    # and a step's copies wait for the previous step's kernels (no overlap across steps)
    copy_streams = [torch.cuda.Stream(device) for _ in range(4)]
    pieces = []
    for k in ins:
        h, d = host[k], dev[k]
        n = max(1, min(8, h.shape[0] // 64)) if h.dim() == 2 else 1
        step_rows = (h.shape[0] + n - 1) // n if h.dim() == 2 else None
        for c in range(n):
            if step_rows is None:
                pieces.append((h, d))
            else:
                pieces.append((h[c * step_rows:(c + 1) * step_rows],
                               d[c * step_rows:(c + 1) * step_rows]))
    done = torch.cuda.Event()
    done.record(stream)

    def step():
        evs = []
        for i, cs in enumerate(copy_streams):
            cs.wait_event(done)
            with torch.cuda.stream(cs):
                for hp, dp in pieces[i::len(copy_streams)]:
                    dp.copy_(hp, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(cs)
            evs.append(ev)
        for ev in evs:
            stream.wait_event(ev)
        launch_step(sd, wd, o, stream)
        for k in res_keys:
            back[k].copy_(o[k], non_blocking=True)
        done.record(stream)

    with torch.cuda.stream(stream):
        for _ in range(2):
            step()
        stream.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        done.record(stream)  # the first timed step's copies start after s
        for _ in range(steps):
            step()
        e.record(stream)
        stream.synchronize()
    ms = s.elapsed_time(e) / steps

    # The same calls given the pinned host arrays themselves: the kernels read over the host link
    # only what the step needs (the rows up to the first rejection, the accepted hidden rows)
    wz = W()
    for k, v in vars(w).items():
        setattr(wz, k, v)
    for k, v in host.items():
        setattr(wz, k, v)
    if getattr(w, "_temp_arg", None) is not None:
        wz._temp_arg = host["temperature"]

    def step_zero_copy():
        launch_step(sd, wz, o, stream)
        for k in res_keys:
            back[k].copy_(o[k], non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(2):
            step_zero_copy()
        stream.synchronize()
        sz, ez = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sz.record(stream)
        for _ in range(steps):
            step_zero_copy()
        ez.record(stream)
        stream.synchronize()
    ms_zc = sz.elapsed_time(ez) / steps
    a = o["num_accepted"].cpu().numpy()
    rows_read = algorithmic_bytes(w, a)[3] + int(((a.astype(np.int64) + 1) * 2 * w.H).sum())
    world = 1
    import torch.distributed as dist

    if dist.is_initialized():  # the job's rate: every rank's requests over the slowest rank
        world = dist.get_world_size()
        t = torch.tensor([ms, ms_zc], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms, ms_zc = float(t[0].item()), float(t[1].item())
    return {"value": world * w.B / (ms * 1e-3), "unit": "requests/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
            "zero_copy": {"value": world * w.B / (ms_zc * 1e-3), "unit": "requests/s",
                          "ms_per_step": ms_zc, "host_bytes_read_per_step": rows_read,
                          "d2h_bytes_per_step": d2h,
                          "how": "the same public calls given the pinned host input arrays; the "
                                 "kernels read over the host link only the rows the step needs"}}


def run_reference(args, world):
    """The oracle on the host cores: the same workload, inputs (set 0 of the timed workload, made
    by the same generator on the GPU when there is one), metric and unit as the timed arm. Each
    step is one oracle pass over a bounded prefix of the batch, sized so that the warm-up and
    timed steps take about two minutes at most."""
    import torch

    import workloads

    cfg = [c for c in workloads.CONFIGS if c["name"] == args.config][0]
    device = "cuda:0" if torch.cuda.is_available() else "cpu"
    w = make_set(args.config, 0, device, 0, args.batch or None)
    hc = host_copy(w)
    B, nsets = w.B, args.sets or n_sets(cfg)
    rows_gb = nsets * w.target.numel() * w.target.element_size() / 1e9
    del w
    cores = len(os.sched_getaffinity(0))
    hs = sized_sample(hc, cores, 100.0 / max(1, args.steps + args.warmup))
    Bs = hs["B"]
    for _ in range(args.warmup):
        oracle_pass(hs, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_pass(hs, cores)
    el = time.perf_counter() - t0
    value = Bs * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "requests/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if cfg["kind"] == "probs" else "bf16",
        "data": "synthetic", "config": config_dict(cfg, B, nsets, rows_gb, world, args.batch),
        "cpu_baseline": {"value": value, "unit": "requests/s", "cores": cores, "kind": "oracle",
                         "sample": f"every step verifies and rebuilds the first {Bs} of the "
                                   f"batch's {B} requests (set 0 of the timed inputs) on "
                                   f"{cores} threads"},
        "e2e": {"value": value, "unit": "requests/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
