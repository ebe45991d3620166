"""Benchmark of the indexer -> Top-K -> sparse-attention decode step.

Default workload: decode, batch 64, context 8192 (indexer 64 heads x 128 with
FP8 keys, Top-K 2048, attention 128 heads over a 576-dim bf16 latent row),
synthetic seeded inputs resident in HBM.  One step is one pass of the whole
path over the batch: indexer scores, Top-K selection, sparse attention.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl si|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own batch
(requests are independent: weak scaling, no collective on the data path; the
only collectives are the timing barrier and a max over ranks).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("decode queries/s + achieved HBM GB/s (% of 8 TB/s); "
          "prefill indexer TFLOP/s (% peak)")
NOMINAL_HBM_GBS = 8000.0
L2_FLUSH_BYTES = 512 << 20   # > 129 MB L2


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p["bf16_tflops_sustained"]), "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "src": "fallback"}


# ---------------------------------------------------------------- bytes/flops

def algorithmic_bytes(wl, out_bytes=2):
    """Bytes the method must move per step, by kernel, and its FLOPs.

    Keys and latent rows are counted once per sequence (the rows of a
    prefill chunk share their sequence's cache; a decode row is the only row
    of its request): a sequence's queries need its keys 0 .. max pos and at
    most that many selected latent rows.
    indexer: those keys (e4m3 row + fp32 scale), each row's indexer heads
             (bf16) and weights (fp32), and the fp32 scores written.
    topk:    the scores read, the indices written.
    attn:    the selected latent rows (bf16), the query heads (bf16), the
             output (`out_bytes` per element) and the indices read."""
    import numpy as np
    pos = wl.q_pos.astype("int64")
    n_keys_rows = int((pos + 1).sum())                         # scores per row
    sel = np.minimum(wl.K, pos + 1)
    n_sel_rows = int(sel.sum())                                # gathers per row
    keys_seq = np.zeros(wl.n_seq, dtype=np.int64)
    sel_seq = np.zeros(wl.n_seq, dtype=np.int64)
    np.maximum.at(keys_seq, wl.q_seq, pos + 1)
    np.add.at(sel_seq, wl.q_seq, sel)
    n_keys = int(keys_seq.sum())
    n_sel = int(np.minimum(sel_seq, keys_seq).sum())
    esz = {"bf16": 2, "e4m3": 1, "e2m1": 0.5}.get(wl.kv_dtype, 4)
    kv_scale_b = 0 if getattr(wl, "kv_scale", None) is None else wl.kv_scale.shape[-1] * 4
    kesz = 1 if wl.k_idx_dtype in ("e4m3", "mxe4m3") else 4
    # per key: one fp32 scale (e4m3 keys) or one E8M0 byte per 32 entries (MXFP8)
    ksc = 0 if wl.k_scale is None else \
        wl.k_scale.dtype.itemsize * (wl.k_scale.shape[-1] if wl.k_scale.ndim == 3 else 1)
    idx_b = n_keys * (wl.Di * kesz + ksc) \
        + wl.n_q * (wl.Hi * wl.Di * 2 + wl.Hi * 4) + n_keys_rows * 4
    topk_b = n_keys_rows * 4 + wl.n_q * wl.K * 4
    qesz = 2 if (getattr(wl, "attn_q_dtype", "") or wl.kv_dtype) == "bf16" else 4
    attn_b = n_sel * int(wl.Dqk * esz + kv_scale_b) + wl.n_q * wl.Hq * wl.Dqk * qesz \
        + wl.n_q * wl.Hq * wl.Dv * out_bytes \
        + wl.n_q * wl.K * 4
    flops_idx = 2 * n_keys_rows * wl.Hi * wl.Di
    flops_attn = 2 * n_sel_rows * wl.Hq * (wl.Dqk + wl.Dv)
    return {"indexer": idx_b, "topk": topk_b, "attn": attn_b,
            "flops_indexer": flops_idx, "flops_attn": flops_attn}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            # the raw samples; SI_CLOCK_LOG_DIR keeps them somewhere other than the
            # temporary directory
            d = os.environ.get("SI_CLOCK_LOG_DIR") or tempfile.gettempdir()
            os.makedirs(d, exist_ok=True)
            self.path = os.path.join(d, f"si_clocks_{os.getpid()}.csv")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- helpers

def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(workload: str, rank: int) -> int:
    """Each rank runs its own independent batch of the same shapes: the
    configuration's seed offset by 1000 x rank."""
    import synth
    return synth.CONFIGS[workload]["seed"] + 1000 * rank


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's figure (a MAX all-reduce: with the timing barrier,
    the only collective of the benchmark)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, n_q: int, ms_per_step: float) -> float:
    """Queries per second of the whole job: every rank's rows over the
    slowest rank's step time."""
    return world * n_q / (ms_per_step / 1e3)


# Workload names of the committed ncu captures (profiles/*.md).
PROFILE_WORKLOAD = {"c1": "decode b64 ctx8192", "c3": "decode b16 ctx131072",
                    "c1:kv8": "decode b64 ctx8192 fp8 kv", "c1:kv4": "decode b64 ctx8192 fp4 kv",
                    "c1:mx": "decode b64 ctx8192 mxfp8 indexer",
                    "c4": "mixed 28 decode + 4 chunks"}
# The step whose operand format each variant changes; the other kernels of a
# variant run as on the plain workload.
VARIANT_KERNEL = {":kv8": "attn", ":kv4": "attn", ":mx": "indexer"}


def code_sha(text: str) -> str:
    """sha256 (first 16 hex digits) of a CUDA source with its comments and
    blank lines removed: an edit of comments alone keeps a capture's counters
    valid, any change of code does not."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def _kernel_traffic(kernel: str, source: str, workload: str):
    """DRAM bytes per launch from the committed ncu capture of this kernel on
    this workload, if the kernel's source code is unchanged since the
    counters were taken; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(f"{kernel}@{PROFILE_WORKLOAD.get(workload, workload)}")
        with open(os.path.join(ROOT, "indexer_driven_top_gb300", "csrc", source)) as f:
            sha = code_sha(f.read())
        if rec and rec.get("source_sha") == sha:
            return rec.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def _topk_kernel(wl, sms=152):
    """The Top-K kernel the library picks for this batch (the rule in
    si_topk.cu's launcher): clusters for long rows in a small batch, one CTA
    per row with its keys in shared memory for many rows of 8193..16384,
    else one CTA per row from registers or streaming."""
    longest = getattr(wl, "max_ctx", 0)
    C = -(-longest // 32768)
    if longest > 16384 and C <= 8 and wl.n_q * C <= 2 * sms:
        return "k_topk_cluster"
    if 8192 < longest <= 16384 and wl.n_q > sms:
        return "k_topk_cluster"
    return "k_topk_rows"


def _kernel_of(wl):
    """The CUDA kernel (and its source file) each step of the path runs for
    this workload: the tensor-core kernels where their shape conditions hold
    (64 x 128 indexer with bf16 q and e4m3 keys; 128 heads x 576 latent rows
    in bf16, FP8 or FP4), the generic ones otherwise."""
    tc_ix = wl.Hi == 64 and wl.Di == 128 and (
        (wl.q_idx_dtype in ("bf16", "e4m3") and wl.k_idx_dtype == "e4m3")
        or (wl.q_idx_dtype in ("bf16", "mxe4m3") and wl.k_idx_dtype == "mxe4m3"))
    tc_at = (wl.Hq == 128 and wl.Dqk == 576 and wl.Dv == 512
             and wl.kv_dtype in ("bf16", "e4m3", "e2m1"))
    prefill = tc_ix and wl.n_seq == 1 and wl.n_q >= 64
    # a planned mixed batch sends each run of >= 64 rows of one sequence (a
    # prefill chunk) to the prefill kernel, the other rows to the decode one
    import numpy as np
    q_seq = np.asarray(getattr(wl, "q_seq", np.zeros(0, np.int32)))
    cuts = np.flatnonzero(np.diff(q_seq)) + 1
    runs = np.diff(np.concatenate([[0], cuts, [len(q_seq)]]))
    chunks = tc_ix and not prefill and bool((runs >= 64).any())
    return {"indexer": ("k_indexer_prefill", "si_indexer_prefill.cu") if prefill
            else ("k_indexer_prefill + k_indexer_tc", "si_indexer_prefill.cu") if chunks
            else ("k_indexer_tc", "si_indexer_tc.cu") if tc_ix
            else ("k_indexer_generic", "si_generic.cu"),
            "topk": (_topk_kernel(wl), "si_topk.cu"),
            "attn": ("k_attn_tc", "si_attn_tc.cu") if tc_at
            else ("k_attn_generic", "si_generic.cu")}


def roofline_of(kernel, wl, algo, ms, peaks, long_step, variant=""):
    """Roofline of one kernel of the step: its algorithmic bytes and FLOPs over
    its measured time, against the measured HBM copy bandwidth and the dense
    tensor peak of its operand type (the indexer multiplies FP8 operands: the
    measured bf16 peak x the nominal FP8/bf16 ratio of 2).  The bound reported
    is the one the kernel is closer to; a kernel timed inside a step longer
    than a millisecond is held to the sustained tensor figure."""
    name, src = _kernel_of(wl)[kernel]
    nbytes = algo[kernel]
    flops = algo.get("flops_" + {"indexer": "indexer", "attn": "attn"}.get(kernel, ""), 0)
    gbs = nbytes / (ms / 1e3) / 1e9
    tf_peak = peaks["bf16_tflops_sustained" if long_step else "bf16_tflops"]
    if kernel == "indexer":
        tf_peak *= 2.0
    tfs = flops / (ms / 1e3) / 1e12 if flops else 0.0
    hbm = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
           "frac": gbs / peaks["hbm_gbs"], "peak_src": peaks["src"] + " (hbm_gbs, copy)"}
    ten = {"bound": "tensor", "achieved": tfs, "peak": tf_peak, "unit": "TFLOP/s",
           "frac": tfs / tf_peak,
           "peak_src": peaks["src"] + (" (bf16_tflops_sustained" if long_step else " (bf16_tflops")
                       + (" x 2 for FP8)" if kernel == "indexer" else ")")}
    roof = dict(ten if ten["frac"] > hbm["frac"] else hbm)
    roof.update({"kernel": name,
                 "traffic": _kernel_traffic(
                     name, src, wl.name + (variant if VARIANT_KERNEL.get(variant) == kernel else ""))
                 if roof["bound"] == "hbm" else None,
                 "algorithmic_bytes_per_launch": nbytes, "algorithmic_flop_per_launch": flops,
                 "ms_per_launch": ms,
                 "other_bound": {k: (ten if roof["bound"] == "hbm" else hbm)[k]
                                 for k in ("bound", "achieved", "peak", "unit", "frac")}})
    return roof


def workload_record(si, dev, name, steps, warmup, variant="", **over):
    """One of the other configurations, timed the same way as the headline
    step (three calls per step, L2 flushed before every step): queries/s, the
    step's algorithmic bytes over its time, per-kernel times and the roofline
    of the dominant kernel.  `over` are generator options (e.g. idx_mx)."""
    import torch
    import synth
    wl = synth.make(name, **over)
    dw = si.upload(wl, dev)
    b, ix, at, K = dw.batch, dw.indexer, dw.attention, dw.k_top
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, b, ix, at, K), dev)
    scores = torch.empty((wl.n_q, b.max_ctx), dtype=torch.float32, device=dev)
    idx = torch.empty((wl.n_q, K), dtype=torch.int32, device=dev)
    out = torch.empty((wl.n_q, wl.Hq, wl.Dv), dtype=getattr(torch, OUT_DTYPE), device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev):
        ev[0].record(stream)
        si.indexer_scores(b, ix, scores, ws, stream)
        ev[1].record(stream)
        si.topk(b, scores, K, idx, ws, stream)
        ev[2].record(stream)
        si.sparse_attn(b, at, idx, K, out, ws, stream=stream)
        ev[3].record(stream)

    n = max(3, min(steps, 20))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    for _ in range(max(3, warmup)):
        step(evs[0])
    for i in range(n):
        flush.fill_(i & 0xFF)
        step(evs[i])
    torch.cuda.synchronize(dev)
    assert si.workspace_status(ws, stream) == 0
    kms = {"indexer": sum(e[0].elapsed_time(e[1]) for e in evs) / n,
           "topk": sum(e[1].elapsed_time(e[2]) for e in evs) / n,
           "attn": sum(e[2].elapsed_time(e[3]) for e in evs) / n}
    ms = sum(e[0].elapsed_time(e[3]) for e in evs) / n
    peaks = _peaks()
    algo = algorithmic_bytes(wl, OUT_BYTES)
    total = algo["indexer"] + algo["topk"] + algo["attn"]
    gbs = total / (ms / 1e3) / 1e9
    dom = max(kms, key=kms.get)
    rec = {"workload": _workload_name(wl), "queries_per_s": wl.n_q / (ms / 1e3),
           "ms_per_step": ms, "steps": n,
           "hbm": {"algorithmic_bytes_per_step": total, "achieved_gbs": gbs,
                   "frac_of_8tbs": gbs / NOMINAL_HBM_GBS, "frac_of_measured": gbs / peaks["hbm_gbs"]},
           "kernels_ms": kms, "kernels": {k: v[0] for k, v in _kernel_of(wl).items()},
           "roofline": roofline_of(dom, wl, algo, kms[dom], peaks, ms > 1.0, variant),
           "indexer_roofline": roofline_of("indexer", wl, algo, kms["indexer"], peaks, ms > 1.0,
                                           variant),
           "l2": "flushed between steps (512 MiB write)"}
    if over:
        rec["options"] = over
    del dw, ws, scores, idx, out, flush
    torch.cuda.empty_cache()
    return rec


def cpu_baseline(wl, rows, threads):
    """The CPU oracle, as it stands, on a bounded sample of query rows."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    oracle.run(wl, rows=rows, threads=threads)
    dt = time.perf_counter() - t0
    return {"value": len(rows) / dt, "unit": "queries/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(rows)} of {wl.n_q} decode rows of workload {wl.name}, "
                      f"full indexer + Top-K + attention per row, {dt:.1f} s"}


def _threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- reference

def run_reference(args):
    """Reference arm: the CPU oracle timed on the host cores."""
    import synth
    wl = synth.make(args.workload)
    threads = _threads()
    rows_per_step = max(threads, 16)
    rows = [i % wl.n_q for i in range(rows_per_step)]
    import oracle
    oracle.build()
    for _ in range(args.warmup):
        oracle.run(wl, rows=rows[:threads], threads=threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.run(wl, rows=rows, threads=threads)
        times.append(time.perf_counter() - t0)
    per_q = sum(times) / (args.steps * len(rows))
    value = 1.0 / per_q
    # ms_per_step is the time of one timed step as it ran: `rows` query rows
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": _workload_name(wl), "rows_per_timed_step": len(rows)},
        "cpu_baseline": {"value": value, "unit": "queries/s", "cores": threads, "kind": "oracle",
                         "sample": f"{len(rows)} decode rows per step of {wl.n_q}"},
        "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


PREFILL_STRIP_ROWS = 1024  # 1024 rows x 16384 positions x 4 B = 64 MiB: the strip stays in L2


def _prefill_once(si, dev, steps, mode):
    """The 16384-token causal prefill's indexer, run as the fused path runs it:
    strips of PREFILL_STRIP_ROWS rows, each scored into a strip buffer that
    stays in L2 and then consumed by the Top-K.  Returns (causal pairs,
    algorithmic FLOPs, indexer ms per prefill: the sum over the strips of the
    indexer launches' event-timed durations, ms of the whole strip loop).
    mode: "bf16" (the configuration: bf16 query, e4m3 keys + fp32 scale),
    "e4m3" (query stored e4m3 + fp32 scale per (row, head)) or "mx" (MXFP8
    keys, the bf16 query converted to MXFP8 inside the kernel)."""
    import torch
    import indexer_driven_top_gb300 as si_mod
    import synth
    wl = synth.make("c2", Hq=1, Dqk=64, Dv=64, q_idx_fp8=mode == "e4m3", idx_mx=mode == "mx")
    dw = si.upload(wl, dev)
    b, ix, K = dw.batch, dw.indexer, dw.k_top
    ld = b.max_ctx
    R = PREFILL_STRIP_ROWS
    strip = torch.empty((R, ld), dtype=torch.float32, device=dev)
    idx = torch.empty((wl.n_q, K), dtype=torch.int32, device=dev)
    ws = si.alloc_workspace(si.workspace_size(si.OP_TOPK, b, ix, None, K), dev)
    stream = torch.cuda.current_stream(dev)
    strips = []
    for r0 in range(0, wl.n_q, R):
        r1 = min(wl.n_q, r0 + R)
        sb = si_mod.Batch(b.block_table, b.ctx_len, b.q_seq[r0:r1], b.q_pos[r0:r1], b.page_size,
                          b.max_ctx, b.n_blocks, host_q_seq=wl.q_seq[r0:r1])
        six = si_mod.Indexer(ix.q[r0:r1], ix.q_dtype, ix.w[r0:r1], ix.k,
                             None if ix.q_scale is None else ix.q_scale[r0:r1])
        strips.append((sb, six, strip[: r1 - r0], idx[r0:r1]))

    def run(ev=None):
        for i, (sb, six, sc, ib) in enumerate(strips):
            if ev:
                ev[2 * i].record(stream)
            si.indexer_scores(sb, six, sc, ws, stream)
            if ev:
                ev[2 * i + 1].record(stream)
            si.topk(sb, sc, K, ib, ws, stream)

    for _ in range(2):
        run()
    torch.cuda.synchronize(dev)
    n = max(3, min(steps, 10))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(strips))] for _ in range(n)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(n):
        run(evs[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    assert si.workspace_status(ws, stream) == 0
    ms = sum(e[2 * i].elapsed_time(e[2 * i + 1]) for e in evs for i in range(len(strips))) / n
    ms_loop = t0.elapsed_time(t1) / n
    # the same work as one call of section 4.1's fused operator (si_indexer_topk:
    # the strips inside the call, each after the first overlapping the
    # previous Top-K's end); its selection must equal the strip loop's
    ws_sel = si.alloc_workspace(si.workspace_size(si.OP_SELECT, b, ix, None, K), dev)
    idx_sel = torch.empty_like(idx)
    for _ in range(2):
        si.indexer_topk(b, ix, K, idx_sel, ws_sel, stream)
    torch.cuda.synchronize(dev)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(n):
        si.indexer_topk(b, ix, K, idx_sel, ws_sel, stream)
    f1.record(stream)
    torch.cuda.synchronize(dev)
    assert si.workspace_status(ws_sel, stream) == 0 and torch.equal(idx_sel, idx)
    ms_fused = f0.elapsed_time(f1) / n
    pairs = int((wl.q_pos.astype("int64") + 1).sum())
    flops = 2.0 * wl.Hi * wl.Di * pairs
    del dw, strip, idx, ws, strips, ws_sel, idx_sel
    torch.cuda.empty_cache()
    return pairs, flops, ms, ms_loop, ms_fused


E2E_REPLICAS = 3
# The attention output is written in bf16, the activation type the output
# projection consumes (fp32 accumulation inside the kernel); the parity tests
# check both fp32 and bf16 outputs.
OUT_DTYPE = "bfloat16"
OUT_BYTES = 2


def e2e_pipelined(si, wl, dw, h_qidx, h_w, h_q, args, dev):
    """End-to-end decode throughput as a serving loop would run it: every step
    copies its query inputs (q_idx, w, q) from pinned host memory, runs
    si_fused_decode and copies out and idx back to pinned host memory.  The
    three stages run on their own streams so that step i's copies overlap
    steps i - 1 and i + 1; events order each replica's buffers (inputs are
    not overwritten before the call that reads them has finished, outputs
    not before they were copied out).  Steps go round E2E_REPLICAS device
    replicas of the workload, so the caches a step reads were last touched
    two steps earlier (at least 2 x 220 MB of other traffic through the
    129 MB L2).  Returns ms per step: device time from the first input copy
    to the last result copy, divided by the step count."""
    import torch
    R = E2E_REPLICAS
    reps = [dw] + [si.upload(wl, dev) for _ in range(R - 1)]
    n_q, K = wl.n_q, dw.k_top
    outs = [torch.empty((n_q, wl.Hq, wl.Dv), dtype=getattr(torch, OUT_DTYPE), device=dev)
            for _ in range(R)]
    idxs = [torch.empty((n_q, K), dtype=torch.int32, device=dev) for _ in range(R)]
    h_outs = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    h_idxs = [torch.empty(i.shape, dtype=i.dtype).pin_memory() for i in idxs]
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, dw.batch, dw.indexer, dw.attention, K),
                            dev)
    s_in, s_c, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(R)]
    ev_c = [torch.cuda.Event() for _ in range(R)]
    ev_out = [torch.cuda.Event() for _ in range(R)]

    def step(i):
        j = i % R
        d = reps[j]
        if i >= R:
            s_in.wait_event(ev_c[j])          # call i - R has read replica j's inputs
        with torch.cuda.stream(s_in):
            d.indexer.q.copy_(h_qidx, non_blocking=True)
            d.indexer.w.copy_(h_w, non_blocking=True)
            d.attention.q.copy_(h_q, non_blocking=True)
        ev_in[j].record(s_in)
        s_c.wait_event(ev_in[j])
        if i >= R:
            s_c.wait_event(ev_out[j])         # results of step i - R copied out
        si.fused_decode(d.batch, d.indexer, d.attention, K, idxs[j], outs[j], ws, stream=s_c)
        ev_c[j].record(s_c)
        s_out.wait_event(ev_c[j])
        with torch.cuda.stream(s_out):
            h_outs[j].copy_(outs[j], non_blocking=True)
            h_idxs[j].copy_(idxs[j], non_blocking=True)
        ev_out[j].record(s_out)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(args.steps):
        step(i)
    s_in.wait_stream(s_out)
    t1.record(s_in)
    torch.cuda.synchronize(dev)
    assert si.workspace_status(ws, s_c) == 0
    assert torch.equal(idxs[0].cpu(), h_idxs[0])
    return t0.elapsed_time(t1) / args.steps


def prefill_indexer(si, dev, steps):
    """Indexer throughput on the 16384-token causal prefill (every row scores
    all earlier positions): algorithmic TFLOP/s = 2 * Hi * Di * causal pairs /
    indexer time, the indexer run strip by strip as the fused path runs it
    (each 64 MiB score strip stays in L2 for the Top-K that follows).  The
    attention operands of that workload are not needed, so they are generated
    at a token size (the indexer inputs are drawn first and do not change).
    Headline: the configuration's bf16 query, exact, which the tensor core
    runs as two e4m3 terms (twice the algorithmic FP8 work).  Also timed, as a
    labelled option: the query quantised to e4m3 with one fp32 scale per
    (row, head), as the indexer prolog of section 4.3 quantises it (the oracle
    scores those same bytes)."""
    peaks = _peaks()
    fp8_peak = 2.0 * peaks["bf16_tflops"]   # measured bf16 burst x nominal fp8/bf16 ratio (2)
    pairs, flops, ms, ms_loop, ms_fused = _prefill_once(si, dev, steps, "bf16")
    tflops = flops / (ms / 1e3) / 1e12
    _, _, ms8, ms8_loop, ms8_fused = _prefill_once(si, dev, steps, "e4m3")
    tflops8 = flops / (ms8 / 1e3) / 1e12
    _, _, msx, msx_loop, msx_fused = _prefill_once(si, dev, steps, "mx")
    tflopsx = flops / (msx / 1e3) / 1e12
    return {"workload": "causal prefill 16384 tokens, indexer 64x128, e4m3 keys + fp32 scale, "
                        "bf16 query",
            "kernel": "k_indexer_prefill",
            "timing": f"strips of {PREFILL_STRIP_ROWS} rows (64 MiB of scores, L2-resident), "
                      "indexer then Top-K per strip; indexer launches event-timed and summed; "
                      "ms_indexer_topk_call: the same prefill as one si_indexer_topk call",
            "causal_pairs": pairs, "algorithmic_tflop": flops / 1e12, "ms_per_prefill": ms,
            "tflops": tflops, "fp8_peak_tflops": fp8_peak,
            "peak_src": peaks["src"] + " (bf16 burst x 2)",
            "frac_of_fp8_peak": tflops / fp8_peak,
            "ms_strip_loop_with_topk": ms_loop,
            "ms_indexer_topk_call": ms_fused,
            "option_e4m3_query": {"ms_per_prefill": ms8, "tflops": tflops8,
                                  "frac_of_fp8_peak": tflops8 / fp8_peak,
                                  "ms_strip_loop_with_topk": ms8_loop,
                                  "ms_indexer_topk_call": ms8_fused,
                                  "note": "query quantised to e4m3 + fp32 scale per (row, head); "
                                          "not the configuration's query format"},
            "option_mxfp8": {"ms_per_prefill": msx, "tflops": tflopsx,
                             "frac_of_fp8_peak": tflopsx / fp8_peak,
                             "ms_strip_loop_with_topk": msx_loop,
                             "ms_indexer_topk_call": msx_fused,
                             "note": "section 5.1's MXFP8 indexer: keys in groups of 32 with E8M0 "
                                     "scales, the bf16 query converted to MXFP8 inside the kernel "
                                     "(block-scaled UMMA, three rows per 192-wide block)"}}


def mxfp8_conversion(si, dev, steps):
    """si_quant_mxfp8 (section 4.3's per-group quantisation of the indexer
    query, in section 5.1's MXFP8 format) on the 16384-token prefill's query:
    16384 rows x 64 heads x 128 bf16 entries (268 MB, larger than L2, so no
    flush is needed between calls).  Algorithmic bytes: 2 read + 1 + 1/32
    written per entry, over the event-timed call, against the measured HBM
    copy bandwidth.  The values are seeded N(0, 1/128) draws made on the
    device (the conversion is checked bit for bit against the oracle by the
    tests, not here)."""
    import torch
    rows, dim = 16384 * 64, 128
    g = torch.Generator(device=dev)
    g.manual_seed(2)
    x = (torch.randn((rows, dim), generator=g, device=dev) / dim ** 0.5).to(torch.bfloat16)
    codes = torch.empty((rows, dim), dtype=torch.uint8, device=dev)
    scales = torch.empty((rows, dim // 32), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        si.quant_mxfp8(x, codes, scales, stream)
    torch.cuda.synchronize(dev)
    n = max(10, min(steps, 50))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for e0, e1 in evs:
        e0.record(stream)
        si.quant_mxfp8(x, codes, scales, stream)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)
    nbytes = rows * dim * 3 + rows * dim // 32
    gbs = nbytes / (ms / 1e3) / 1e9
    peaks = _peaks()
    del x, codes, scales
    torch.cuda.empty_cache()
    return {"workload": "16384 x 64 x 128 bf16 indexer query rows (causal prefill 16384)",
            "kernel": "k_quant_mxfp8", "call": "si_quant_mxfp8", "ms_per_call": ms,
            "algorithmic_bytes": nbytes, "achieved_gbs": gbs,
            "frac_of_measured_hbm": gbs / peaks["hbm_gbs"],
            "l2": "input 268 MB, larger than L2"}


def candidate_selection(si, dev, steps, n_cand=16384):
    """Candidate-restricted selection (the vLLM article on DeepSeek-V4.1,
    "Kernels": indexer logits over a fixed candidate set per query) on the
    long-context decode workload (16 rows x 131072 positions, 1 % planted
    keys) with n_cand seeded candidates per row, timed beside the
    full-context indexer + Top-K of the same rows.  The attention operands
    are not needed and are generated at a token size (the indexer inputs are
    drawn first and do not change).  L2 is flushed before every timed call.
    Algorithmic bytes of the candidate call: per candidate its list entry
    (4 B), key row (e4m3) and scale (4 B) and its score (4 B); per row the
    indexer query (bf16), the head weights and the K output indices."""
    import torch
    import synth
    wl = synth.make("c3", Hq=1, Dqk=64, Dv=64)
    cand = synth.candidates(wl, n_cand, seed=31)
    dw = si.upload(wl, dev)
    b, ix, K = dw.batch, dw.indexer, dw.k_top
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    ws_full = si.alloc_workspace(si.workspace_size(si.OP_TOPK, b, ix, None, K), dev)
    scores = torch.empty((wl.n_q, b.max_ctx), dtype=torch.float32, device=dev)
    idx = torch.empty((wl.n_q, K), dtype=torch.int32, device=dev)
    c = torch.from_numpy(cand).to(dev)
    ws_c = si.alloc_workspace(si.workspace_size_cand(b, ix, n_cand), dev)
    idx_c = torch.empty((wl.n_q, K), dtype=torch.int32, device=dev)

    def full():
        si.indexer_scores(b, ix, scores, ws_full, stream)
        si.topk(b, scores, K, idx, ws_full, stream)

    def restricted():
        si.indexer_topk_cand(b, ix, c, K, idx_c, ws_c, stream=stream)

    def timed(fn):
        for _ in range(3):
            fn()
        n = max(5, min(steps, 50))
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
        for i in range(n):
            flush.zero_()
            ev[2 * i].record(stream)
            fn()
            ev[2 * i + 1].record(stream)
        torch.cuda.synchronize(dev)
        return sum(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(n)) / n

    ms_full, ms_c = timed(full), timed(restricted)
    assert si.workspace_status(ws_c, stream) == 0 and si.workspace_status(ws_full, stream) == 0
    key_bytes = wl.Di + 4
    nbytes = (wl.n_q * n_cand * (4 + key_bytes + 4)
              + wl.n_q * (wl.Hi * wl.Di * 2 + wl.Hi * 4 + K * 4))
    peaks = _peaks()
    gbs = nbytes / (ms_c / 1e3) / 1e9
    return {"workload": "decode batch 16 x context 131072 (1% planted keys), "
                        f"{n_cand} candidates per row, indexer 64x128 fp8, top-k {K}",
            "call": "si_indexer_topk_cand (indexer gathering the candidate keys, top-k writing positions)",
            "ms_per_call": ms_c, "queries_per_s": wl.n_q / (ms_c / 1e3),
            "algorithmic_bytes": nbytes, "achieved_gbs": gbs,
            "frac_of_measured_hbm": gbs / peaks["hbm_gbs"],
            "full_context": {"call": "si_indexer_scores + si_topk over all 131072 positions",
                             "ms_per_call": ms_full},
            "speedup_vs_full_context": ms_full / ms_c,
            "indexer_dram_bytes_per_launch": _kernel_traffic(
                "k_indexer_tc", "si_indexer_tc.cu", "candidates b16 16384"),
            "l2": "flushed before every timed call (512 MiB write)"}


def _workload_name(wl):
    names = {
        "c1": "decode batch 64 x context 8192, indexer 64x128 fp8, top-k 2048, MLA 128x576 bf16",
        "c2": "causal prefill 16384 tokens, indexer 64x128 fp8, top-k 2048, MLA 128x576 bf16",
        "c3": "decode batch 16 x context 131072 (1% planted keys), indexer 64x128 fp8, top-k 2048, "
              "MLA 128x576 bf16",
        "c4": "mixed batch: 28 decode rows + 4 prefill chunks of 2048 over contexts 1K-64K, "
              "indexer 64x128 fp8, top-k 2048, MLA 128x576 bf16",
    }
    name = names.get(wl.name, wl.name)
    # the indexer and cache formats the workload was generated with
    if wl.k_idx_dtype == "mxe4m3":
        name = name.replace("indexer 64x128 fp8", "indexer 64x128 MXFP8 keys, "
                            + ("MXFP8" if wl.q_idx_dtype == "mxe4m3" else wl.q_idx_dtype) + " query")
    if wl.kv_dtype in ("e4m3", "e2m1"):
        name = name.replace("MLA 128x576 bf16", "MLA 128x576 "
                            + {"e4m3": "FP8", "e2m1": "FP4"}[wl.kv_dtype] + " latent cache")
    return name


# ---------------------------------------------------------------- main arm

def run_si(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import indexer_driven_top_gb300 as si
    import synth

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    wl = synth.make(args.workload, seed=rank_seed(args.workload, rank),
                    **({"kv_fp8": True} if args.kv_fp8 else {}),
                    **({"kv_fp4": True} if args.kv_fp4 else {}),
                    **({"idx_mx": True} if args.idx_mx else {}))
    dw = si.upload(wl, dev)
    b, ix, at, K = dw.batch, dw.indexer, dw.attention, dw.k_top
    n_q = wl.n_q
    ld = b.max_ctx
    ws = si.alloc_workspace(si.workspace_size(si.OP_FUSED, b, ix, at, K), dev)
    scores = torch.empty((n_q, ld), dtype=torch.float32, device=dev)
    idx = torch.empty((n_q, K), dtype=torch.int32, device=dev)
    out = torch.empty((n_q, wl.Hq, wl.Dv), dtype=getattr(torch, OUT_DTYPE), device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        """The per-kernel pass: the three calls one by one."""
        if ev:
            ev[0].record(stream)
        si.indexer_scores(b, ix, scores, ws, stream)
        if ev:
            ev[1].record(stream)
        si.topk(b, scores, K, idx, ws, stream)
        if ev:
            ev[2].record(stream)
        si.sparse_attn(b, at, idx, K, out, ws, stream=stream)
        if ev:
            ev[3].record(stream)

    ws_step = si.alloc_workspace(si.workspace_size(si.OP_FUSED, b, ix, at, K), dev)

    def fused_step():
        """The timed step: the whole path in one call on resident inputs."""
        si.fused_decode(b, ix, at, K, idx, out, ws_step, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
        fused_step()
    torch.cuda.synchronize(dev)
    assert si.workspace_status(ws, stream) == 0
    assert si.workspace_status(ws_step, stream) == 0

    # Timed passes over K steps each, L2 flushed before every step.  The step
    # pass times si_fused_decode, the whole path in one call (scores, Top-K --
    # inside the indexer where the fused selection applies -- and attention),
    # bracketed by two events; it gives `value`.  The kernel pass runs the
    # three entry points one by one with an event between the launches for
    # the per-kernel breakdown and the roofline; the select pass times
    # si_indexer_topk (scores + Top-K as one operator) alone.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = si.launch_count()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)            # evict the previous step's data from L2
        sevs[i][0].record(stream)
        fused_step()
        sevs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    launches = si.launch_count() - launches0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        step(evs[i])
    torch.cuda.synchronize(dev)
    assert si.workspace_status(ws, stream) == 0

    assert si.workspace_status(ws_step, stream) == 0
    t_k = {"indexer": [e[0].elapsed_time(e[1]) for e in evs],
           "topk": [e[1].elapsed_time(e[2]) for e in evs],
           "attn": [e[2].elapsed_time(e[3]) for e in evs]}
    # select pass: scores + Top-K as one operator (si_indexer_topk)
    ws_s = si.alloc_workspace(si.workspace_size(si.OP_SELECT, b, ix, None, K), dev)
    si.indexer_topk(b, ix, K, idx, ws_s, stream)
    selv = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        selv[i][0].record(stream)
        si.indexer_topk(b, ix, K, idx, ws_s, stream)
        selv[i][1].record(stream)
    torch.cuda.synchronize(dev)
    assert si.workspace_status(ws_s, stream) == 0
    sel_ms = sum(e[0].elapsed_time(e[1]) for e in selv) / args.steps
    del ws_s
    ms = sum(e[0].elapsed_time(e[1]) for e in sevs) / args.steps
    ms_max = max_over_ranks(ms, world, dev)
    value = whole_job_rate(world, n_q, ms_max)
    e2e = None
    if not args.no_e2e:
        # ---- end to end: host (pinned) buffers in and out, through the fused call
        h_qidx = torch.from_numpy(wl.q_idx).view(torch.bfloat16).pin_memory()
        h_w = torch.from_numpy(wl.w).pin_memory()
        h_q = torch.from_numpy(wl.q).view(torch.bfloat16).pin_memory()
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_idx = torch.empty(idx.shape, dtype=idx.dtype).pin_memory()
        ws_f = si.alloc_workspace(si.workspace_size(si.OP_FUSED, b, ix, at, K), dev)
        e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]

        def e2e_step(ev=None):
            if ev:
                ev[0].record(stream)
            ix.q.copy_(h_qidx, non_blocking=True)
            ix.w.copy_(h_w, non_blocking=True)
            at.q.copy_(h_q, non_blocking=True)
            si.fused_decode(b, ix, at, K, idx, out, ws_f, stream=stream)
            h_out.copy_(out, non_blocking=True)
            h_idx.copy_(idx, non_blocking=True)
            if ev:
                ev[1].record(stream)

        for _ in range(max(3, args.warmup)):
            e2e_step()
        torch.cuda.synchronize(dev)
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            e2e_step(e2e_ev[i])
        torch.cuda.synchronize(dev)
        assert si.workspace_status(ws_f, stream) == 0
        e2e_ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in e2e_ev) / args.steps, world,
                                dev)
        h2d = h_qidx.numel() * 2 + h_w.numel() * 4 + h_q.numel() * 2
        d2h = h_out.numel() * h_out.element_size() + h_idx.numel() * 4
        del ws_f
        e2e_pipe_ms = max_over_ranks(e2e_pipelined(si, wl, dw, h_qidx, h_w, h_q, args, dev),
                                     world, dev)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    if not args.no_e2e:
        e2e = {"value": whole_job_rate(world, n_q, e2e_pipe_ms), "unit": "queries/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_pipe_ms,
               "call": "si_fused_decode with pinned host inputs/outputs",
               "timing": f"first input copy to last result copy over {args.steps} steps; "
                         f"copies in, fused call and copies out overlap across steps on three "
                         f"streams; {E2E_REPLICAS} device replicas of the resident caches "
                         f"taken in turn so that consecutive steps share no cached data",
               "serial": {"value": whole_job_rate(world, n_q, e2e_ms), "ms_per_step": e2e_ms,
                          "timing": "each step alone: copies in, fused call, copies out, "
                                    "L2 flushed between steps"}}

    # ---- roofline of the dominant kernel
    peaks = _peaks()
    algo = algorithmic_bytes(wl, OUT_BYTES)
    mean_k = {k: sum(v) / len(v) for k, v in t_k.items()}
    dom = max(mean_k, key=mean_k.get)
    roof = roofline_of(dom, wl, algo, mean_k[dom], peaks, ms > 1.0,
                       ":kv8" if args.kv_fp8 else ":kv4" if args.kv_fp4 else
                       ":mx" if args.idx_mx else "")
    total_bytes = algo["indexer"] + algo["topk"] + algo["attn"]
    step_gbs = total_bytes / (ms / 1e3) / 1e9

    prefill = None if args.no_prefill else prefill_indexer(si, dev, args.steps)
    others = {}
    if (not args.no_other_workloads and args.workload == "c1" and
            not (args.kv_fp8 or args.kv_fp4 or args.idx_mx)):
        del dw, ws, ws_step, scores, idx, out, flush
        torch.cuda.empty_cache()
        others = {"long_context": workload_record(si, dev, "c3", args.steps, args.warmup),
                  "mixed": workload_record(si, dev, "c4", args.steps, args.warmup),
                  "mxfp8_indexer": workload_record(si, dev, "c1", args.steps, args.warmup,
                                                   variant=":mx", idx_mx=True),
                  "mxfp8_conversion": mxfp8_conversion(si, dev, args.steps)}

    cpu = None
    if not args.no_cpu_baseline:
        threads = _threads()
        cpu = cpu_baseline(wl, list(range(n_q)), threads)

    line = {
        "metric": METRIC, "value": value, "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": _workload_name(wl), "batch": n_q, "context": ld, "top_k": K,
                   "indexer": (f"{wl.Hi}x{wl.Di} MXFP8 keys (groups of 32, E8M0 scales), bf16 q "
                               "converted to MXFP8 on the device" if args.idx_mx else
                               f"{wl.Hi}x{wl.Di} e4m3 keys + fp32 scale, bf16 q"),
                   "attention": f"{wl.Hq} heads x {wl.Dqk} (v {wl.Dv}) "
                                f"{'e4m3 cache + fp32 scale per 128-entry tile, bf16 q' if args.kv_fp8 else 'e2m1 cache + fp32 scale per 16-entry block, bf16 q' if args.kv_fp4 else 'bf16'}, "
                                f"fp32 accumulate, {OUT_DTYPE} out",
                   "page": wl.page, "l2": "flushed between steps (512 MiB write)",
                   "step": "si_fused_decode (scores, Top-K, attention in one call) on "
                           "resident inputs; kernels_ms from the three calls one by one",
                   "parallelism": f"dp{world} (independent requests per rank)"},
        "hbm": {"algorithmic_bytes_per_step": total_bytes, "achieved_gbs": step_gbs,
                "frac_of_8tbs": step_gbs / NOMINAL_HBM_GBS,
                "frac_of_measured": step_gbs / peaks["hbm_gbs"]},
        "kernels_ms": mean_k,
        "indexer_topk_ms": sel_ms,
        "kernels": {k: v[0] for k, v in _kernel_of(wl).items()},
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": int(launches),
        "roofline": roof,
        "cpu_baseline": cpu,
        "prefill_indexer": prefill,
        **others,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["si", "reference"], default="si")
    ap.add_argument("--workload", default="c1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end legs")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the long-context and mixed-batch records of the default line")
    ap.add_argument("--idx-mx", action="store_true",
                    help="indexer keys in MXFP8 (groups of 32, E8M0 scales); the bf16 query is "
                         "converted on the device")
    ap.add_argument("--kv-fp4", action="store_true",
                    help="store the latent KV cache in FP4 e2m1 (one scale per row and 16-entry "
                         "block, the NVFP4 block)")
    ap.add_argument("--kv-fp8", action="store_true",
                    help="store the latent KV cache in FP8 (one scale per row and 128-entry tile)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the prefill indexer (both query formats) and print its record")
    ap.add_argument("--cand-only", action="store_true",
                    help="time only candidate-restricted selection (16 x 131072, 16384 candidates "
                         "per row) beside the full-context indexer + Top-K, and print its record")
    args = ap.parse_args()
    if args.cand_only:
        import torch
        import indexer_driven_top_gb300 as si
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps({"candidate_selection": candidate_selection(si, dev, args.steps)}),
              flush=True)
        return
    if args.prefill_only:
        import torch
        import indexer_driven_top_gb300 as si
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps({"prefill_indexer": prefill_indexer(si, dev, args.steps)}), flush=True)
        return
    if args.impl == "reference":
        world, rank, _ = _dist()
        if rank == 0:
            run_reference(args)
        return
    run_si(args)


if __name__ == "__main__":
    main()
