#!/usr/bin/env python3
"""Throughput of the KPool DSA step (one DSA layer: compress + score + top-k +
sparse MLA) on B300, with the roofline of its dominant kernel and the fp64
oracle timed on the host cores beside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kpool|reference]
                    [--workload decode|ragged|prefill|long]

Prints ONE JSON line (rank 0).  Timing: every step is a CUDA-graph replay of
kp_dsa_forward bracketed by CUDA events on the launching stream; a 256 MB read
flushes L2 between steps, outside the events.  Under torchrun each rank runs
its own batch (weak scaling over independent sequences, no collective on the
data path); value = all ranks' query tokens / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import kpool_inputs as KI  # noqa: E402
from dsa_indexer_sparse_kpool_b300 import replicas  # noqa: E402

METRIC = {"decode": "DSA decode tokens/s per B300", "ragged": "DSA decode tokens/s per B300",
          "long": "DSA decode tokens/s per B300", "prefill": "DSA prefill tokens/s per B300"}
DESCR = {
    "decode": "decode: 32 seqs x ctx 32768, 1 query each, top-k 2048 tokens (512 pools + tail), "
              "indexer 32x128, MLA 64 heads x 576 latent, bf16",
    "ragged": "ragged decode + MTP: 8 seqs, ctx U[65537,131071] (not multiples of 4), 2 queries each, top-k 2048",
    "prefill": "chunked causal prefill: 1 seq, 4096 new queries on 61440 cached (ctx 65536), top-k 2048",
    "long": "long-context decode: 1 seq, ctx 1,048,575, 4 queries, top-k 2048",
}
STAGES = ("kpool_compress", "indexer_score", "topk_select", "sparse_mla_attend")
FUSED_STAGES = ("kpool_compress", "indexer_score_select", "sparse_mla_attend")
KERNEL_FILES = {   # each stage's kernel source and the headers it includes
    "kpool_compress": ("compress.cu", "score_plan.cuh", "kp_common.cuh"),
    "indexer_score": ("score.cu", "score_plan.cuh", "kp_common.cuh"),
    "topk_select": ("topk.cu", "topk_select.cuh", "kp_common.cuh"),
    "indexer_score_select": ("score_select.cu", "topk_select.cuh", "score_plan.cuh", "kp_common.cuh"),
    "sparse_mla_attend": ("attend.cu", "kp_common.cuh"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="kpool", choices=["kpool", "reference"])
    ap.add_argument("--workload", default="decode", choices=["decode", "ragged", "prefill", "long"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--select", default="auto", choices=["auto", "staged", "fused"],
                    help="how the step scores and selects (fused: one kernel, scores kept on chip)")
    ap.add_argument("--share-mtp", action="store_true",
                    help="each sequence's later queries attend its first query's selection (shared selection)")
    ap.add_argument("--paged", type=int, default=0, metavar="TOKENS",
                    help="page the caches in pages of TOKENS positions (block table, shuffled pages)")
    return ap.parse_args()


# ------------------------------------------------------------------ workload facts

def workload(name: str, rank: int) -> KI.Workload:
    spec = KI.named(name)
    spec.seed = replicas.rank_seed(spec.seed, rank)   # each rank its own independent batch
    return KI.make(spec)


def algorithmic_bytes(wl: KI.Workload):
    """Bytes the method must move per step, by stage: pooled keys once per
    sequence plus q and w (score); 1024 B per attended latent row (each row of a
    sequence counted at most once) plus q_lat, out and lse per query (attend);
    new key and gate rows plus new pooled rows (compress)."""
    kp = wl.spec.kpool
    K = wl.k_pools
    nf = (wl.q_pos.astype(np.int64) + 1) // kp
    tail = (wl.q_pos.astype(np.int64) + 1) - nf * kp
    n_tok = np.minimum(nf, K) * kp + tail
    # pooled keys once per sequence (the largest n_full among its queries), q and w
    per_seq = {}
    for q in range(wl.NQ):
        b = int(wl.q_seq[q])
        per_seq[b] = max(per_seq.get(b, 0), int(nf[q]))
    score = sum(per_seq.values()) * 128 * 2 + wl.NQ * (32 * 128 * 2 + 32 * 4)
    # latent rows: each query's gathered rows, but never more than the sequence
    # holds (the queries of a prefill chunk share one cache)
    tok_per_seq = {}
    for q in range(wl.NQ):
        b = int(wl.q_seq[q])
        tok_per_seq[b] = tok_per_seq.get(b, 0) + int(n_tok[q])
    rows = sum(min(v, int(wl.lens[b])) for b, v in tok_per_seq.items())
    attend = rows * 512 * 2 + wl.NQ * 64 * (512 * 2 + 512 * 2 + 4)
    n_new = int((wl.lens - wl.prev_len).sum())
    new_pools = int(sum(int(L) // kp - int(P) // kp for L, P in zip(wl.lens, wl.prev_len)))
    compress = n_new * 2 * 128 * 2 + new_pools * 128 * 2
    return {"kpool_compress": compress, "indexer_score": score, "topk_select": 0,
            "sparse_mla_attend": attend}, int(n_tok.sum())


def kernel_bytes(wl: KI.Workload, alg: dict) -> dict:
    """Bytes each kernel must move per launch.  The step's count leaves out the
    fp32 scores (an intermediate of the step); the top-k kernel on its own reads
    every visible pool's score once (4 B) and writes its selection (K + 1
    words per query).  The fused score-and-select keeps the scores on chip and
    moves the scorer's bytes plus the selection."""
    nf = (wl.q_pos.astype(np.int64) + 1) // wl.spec.kpool
    sel = wl.NQ * (wl.k_pools + 1) * 4
    kb = dict(alg)
    kb["topk_select"] = int(nf.sum()) * 4 + sel
    kb["indexer_score_select"] = alg["indexer_score"] + sel
    return kb


def algorithmic_flops(wl: KI.Workload):
    """Tensor-core flops the method must do per step, by stage: scores over each
    query's visible pools (32 heads x 128 dims), and Q.K plus P.V over each
    query's attended tokens (64 heads x 512 latent columns)."""
    kp = wl.spec.kpool
    nf = (wl.q_pos.astype(np.int64) + 1) // kp
    tail = (wl.q_pos.astype(np.int64) + 1) - nf * kp
    n_tok = np.minimum(nf, wl.k_pools) * kp + tail
    return {"kpool_compress": 0, "indexer_score": int(nf.sum()) * 32 * 128 * 2, "topk_select": 0,
            "sparse_mla_attend": int(n_tok.sum()) * 64 * 512 * 2 * 2}


def measured_peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    return 6400.0, 1800.0, 1400.0, "fallback"


def code_of(src: str) -> str:
    """C++/CUDA source without its comments and with runs of white space
    collapsed: what a traffic figure depends on.  (String literals in these
    sources hold no comment markers.)"""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def kernel_source_hash(stage: str) -> str:
    """Hash of the code of the stage's kernel source and its headers (comments
    and layout ignored): a traffic figure is used only while the code it was
    captured on is unchanged."""
    h = hashlib.sha256()
    for f in KERNEL_FILES[stage]:
        h.update(code_of(open(os.path.join(ROOT, "dsa_indexer_sparse_kpool_b300", "csrc", f)).read()).encode())
    return h.hexdigest()[:16]


def kernel_traffic(stage: str, workload_name: str):
    """ncu DRAM bytes per launch of this stage's kernel on this workload
    (profiles/ncu_traffic.txt), if that capture was taken on the current kernel
    source; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    sha = kernel_source_hash(stage)
    for line in open(p):
        f = line.split()
        # stage kernel workload bytes_per_launch ... source_sha
        if len(f) >= 5 and not line.startswith("#") and f[0] == stage and f[2] == workload_name and f[-1] == sha:
            return int(f[3])
    return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """SM clock and throttle reasons sampled through NVML every millisecond in
    a background thread (reads only; no setting of the GPU is changed), so
    that even a timed region of a few milliseconds holds samples.  Each sample
    is stamped with time.monotonic(); `window(t0, t1)` summarises the samples
    inside [t0, t1]."""
    REASONS = (("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20), ("hw_thermal_slowdown", 0x40),
               ("hw_power_brake_slowdown", 0x80), ("sw_power_cap", 0x4))

    def __init__(self, device_index: int):
        import threading
        self.samples = []
        self.error = None
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._run, args=(device_index,), daemon=True)

    def _run(self, device_index):
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")        # the driver's NVML, read-only queries

            def ok(r, what):
                if r != 0:
                    raise RuntimeError(f"{what} returned {r}")
            ok(nv.nvmlInit_v2(), "nvmlInit_v2")
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            h = ctypes.c_void_p()
            ok(nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)), "nvmlDeviceGetHandleByUUID")
            clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
            sm_clock = 1                                   # NVML_CLOCK_SM
            ok(nv.nvmlDeviceGetMaxClockInfo(h, sm_clock, ctypes.byref(mx)), "nvmlDeviceGetMaxClockInfo")
            reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            while not self._stop.is_set():
                ok(nv.nvmlDeviceGetClockInfo(h, sm_clock, ctypes.byref(clk)), "nvmlDeviceGetClockInfo")
                ok(reasons(h, ctypes.byref(rs)), "clock event reasons")
                self.samples.append((time.monotonic(), clk.value, mx.value, rs.value))
                time.sleep(0.001)
            nv.nvmlShutdown()
        except Exception as e:  # no NVML: report that, never guess
            self.error = f"{type(e).__name__}: {e}"

    def start(self):
        self._thread.start()
        t0 = time.monotonic()
        while not self.samples and self.error is None and time.monotonic() - t0 < 5.0:
            time.sleep(0.005)

    def stop(self):
        self._stop.set()
        self._thread.join(timeout=5)

    def window(self, t0: float, t1: float):
        if self.error is not None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable: " + self.error], "samples": 0}
        sel = [x for x in self.samples if t0 <= x[0] <= t1]
        reasons = set()
        for _, _, _, rs in sel:
            for name, bit in self.REASONS:
                if rs & bit:
                    reasons.add(name)
        sm = [x[1] for x in sel]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(x[2] for x in sel) if sel else None,
                "sm_mhz_min": min(sm) if sm else None, "reasons": sorted(reasons), "samples": len(sel),
                "source": "NVML, 1 ms period"}


# ------------------------------------------------------------------ CPU oracle baseline

def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


class OracleStep:
    """The fp64 oracle doing this workload's step for a batch of queries:
    compress of the pools the step's new tokens complete, scores over all
    visible pools, top-k, attention.  The pooled caches of the sequences as they
    were before the step are built once in the constructor (cache state, not
    step work)."""

    def __init__(self, wl: KI.Workload, threads: int):
        import oracle
        self.oracle, self.wl, self.threads, kp = oracle, wl, threads, wl.spec.kpool
        pooled, self.pool_off, off = [], np.zeros(wl.B, np.int64), 0
        for b in range(wl.B):
            a, e = int(wl.tok_off[b]), int(wl.tok_off[b] + wl.prev_len[b])
            p, _ = oracle.kpool_compress(KI.bits(wl.keys[a:e]), KI.bits(wl.gates[a:e]), KI.bits(wl.ape), kp)
            full = np.zeros((int(wl.lens[b]) // kp + 1, 128), np.uint16)
            full[:p.shape[0]] = p
            pooled.append(full)
            self.pool_off[b] = off
            off += full.shape[0]
        self.pooled = np.concatenate(pooled)
        self.lat = KI.bits(wl.latent)
        self.keys, self.gates, self.ape = KI.bits(wl.keys), KI.bits(wl.gates), KI.bits(wl.ape)
        self.q_idx, self.q_lat, self.w = KI.bits(wl.q_idx), KI.bits(wl.q_lat), wl.w.numpy()

    def run(self, queries) -> int:
        wl, kp, o = self.wl, self.wl.spec.kpool, self.oracle
        bq = np.asarray(queries)
        for b in sorted({int(wl.q_seq[q]) for q in bq}):
            p0, p1 = int(wl.prev_len[b]) // kp, int(wl.lens[b]) // kp
            if p1 > p0:
                a, e = int(wl.tok_off[b]) + p0 * kp, int(wl.tok_off[b]) + p1 * kp
                newp, _ = o.kpool_compress(self.keys[a:e], self.gates[a:e], self.ape, kp)
                self.pooled[self.pool_off[b] + p0: self.pool_off[b] + p1] = newp
        o.dsa_queries(wl.q_seq[bq], wl.q_pos[bq], self.pool_off, wl.tok_off, kp, wl.k_pools, 1, self.q_idx[bq],
                      self.w[bq], self.pooled, self.q_lat[bq], self.lat, wl.spec.sm_scale, threads=self.threads)
        return len(bq)

    def batches(self):
        qs = list(range(self.wl.NQ))
        while True:
            for i in range(0, len(qs), self.threads):
                yield qs[i:i + self.threads]

    def rate(self, seconds: float):
        """Query tokens per second over whole batches until `seconds` have passed."""
        done, t0, it = 0, time.perf_counter(), self.batches()
        while True:
            done += self.run(next(it))
            if time.perf_counter() - t0 >= seconds:
                break
        wall = time.perf_counter() - t0
        return done / wall, done, wall


# ------------------------------------------------------------------ reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = workload(args.workload, 0)
    threads = os.cpu_count() or 1
    ob = OracleStep(wl, threads)
    it = ob.batches()
    t0 = time.perf_counter()
    ob.run(next(it))                              # calibration: one batch
    per_step = time.perf_counter() - t0
    steps = max(1, min(args.steps, int(120.0 / max(per_step, 1e-6))))
    for _ in range(min(args.warmup, 2)):
        ob.run(next(it))
    t0 = time.perf_counter()
    n = 0
    for _ in range(steps):
        n += ob.run(next(it))
    wall = time.perf_counter() - t0
    val = n / wall
    line = {"impl": "reference", "metric": METRIC[args.workload], "value": val, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": steps, "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": wall / steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": DESCR[args.workload], "queries_per_step": min(threads, wl.NQ)},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": f"each step = {min(threads, wl.NQ)} whole queries of the workload (compress "
                                       f"of the step's new pools, scores, top-k, attention), OpenMP over queries; "
                                       f"steps capped so the run ends in about 2 minutes"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm

def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch.distributed as dist
    from dsa_indexer_sparse_kpool_b300 import Config
    from dsa_indexer_sparse_kpool_b300 import build as kbuild
    from dsa_indexer_sparse_kpool_b300.session import build_session, build_step

    kbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    wl = workload(args.workload, rank)
    from dsa_indexer_sparse_kpool_b300 import SELECT_AUTO, SELECT_STAGED, SELECT_FUSED
    mode = {"auto": SELECT_AUTO, "staged": SELECT_STAGED, "fused": SELECT_FUSED}[args.select]
    cfg = Config(topk_tokens=wl.spec.topk_tokens, sm_scale=wl.spec.sm_scale, select_mode=mode)
    sess = build_session(cfg, wl.lens.tolist(), wl.prev_len.tolist(), wl.tok_off.tolist(), wl.pool_off.tolist(),
                         wl.pool_rows, wl.latent, wl.keys, wl.gates, wl.ape, device=dev,
                         page_tokens=args.paged or None)
    step = build_step(sess, wl.lens.tolist(), wl.prev_len.tolist(), wl.tok_off.tolist(), wl.keys, wl.gates,
                      wl.q_seq, wl.q_pos, wl.q_idx, wl.w, wl.q_lat)
    NQ = wl.NQ
    if args.share_mtp:   # the MTP verification queries take their sequence's first query's selection
        first = {}
        share = []
        for q in range(NQ):
            b = int(wl.q_seq[q])
            if b in first:
                share.append(first[b])
            else:
                first[b] = q
                share.append(-1)
        step.set_share(share)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(256 << 18, dtype=torch.float32, device=dev).fill_(1.0)   # 256 MB > 126 MB L2

    def flush_l2():
        flush.sum()

    with torch.cuda.stream(stream):
        for _ in range(3):                      # eager warm-up (lazy init outside capture)
            step.run()
        torch.cuda.synchronize()
        assert int(sess.status.item()) == 0, "device status set during warm-up"
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step.run()
        fused = step.fused()
        stages = FUSED_STAGES if fused else STAGES
        calls, _ = step.stage_calls(fused=fused)
        for c in calls:
            c()
        stage_graphs = []
        for c in calls:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                c()
            stage_graphs.append(g)
        torch.cuda.synchronize()

        def barrier():
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()

        # ---- headline: K replays of the whole step
        sampler = ClockSampler(local)
        sampler.start()
        for _ in range(args.warmup):
            flush_l2()
            graph.replay()
        barrier()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        th0 = time.monotonic()
        for i in range(args.steps):
            flush_l2()
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        barrier()
        th1 = time.monotonic()
        step_ms = [a.elapsed_time(b) for a, b in ev]
        total_ms = float(sum(step_ms))

        # ---- per-stage breakdown (one graph per stage, events between)
        ks = max(1, min(args.steps, 500))
        sev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(ks)]
        for i in range(ks):
            flush_l2()
            sev[i][0].record(stream)
            for j, g in enumerate(stage_graphs):
                g.replay()
                sev[i][j + 1].record(stream)
        barrier()
        stage_ms = {stages[j]: float(np.mean([sev[i][j].elapsed_time(sev[i][j + 1]) for i in range(ks)]))
                    for j in range(len(stages))}

        # ---- end to end: pinned host inputs -> step -> host outputs, every step.
        # The step's inputs and outputs are packed into one device buffer each
        # (Step.pack_io), so each direction is one copy from / to pinned memory,
        # and the step is captured again on the packed tensors.
        keep_alive = (step.q_idx, step.w, step.q_lat, step.keys, step.gates, step.prev_len, step.new_off,
                      step.queries, step.out, step.lse)  # the headline graph's tensors
        in_buf, out_buf = step.pack_io()
        h_in = torch.empty(in_buf.numel(), dtype=torch.uint8).pin_memory()
        h_in.copy_(in_buf)
        h_out = torch.empty(out_buf.numel(), dtype=torch.uint8).pin_memory()
        h2d = in_buf.numel()
        d2h = out_buf.numel()
        # Step.run_host: the inputs from pinned memory (q_lat on a second
        # stream, overlapping compression, scoring and selection), the step,
        # out and lse back to pinned memory; captured as one graph.
        step.run_host(h_in, h_out)
        torch.cuda.synchronize()
        graph_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_e2e, stream=stream):
            step.run_host(h_in, h_out)
        ke = max(1, min(args.steps, 1000))
        eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(ke)]
        for i in range(ke):
            flush_l2()
            eev[i][0].record(stream)
            graph_e2e.replay()
            eev[i][1].record(stream)
        barrier()
        t_all1 = time.monotonic()
        sampler.stop()
        del keep_alive
        e2e_ms = float(np.mean([a.elapsed_time(b) for a, b in eev]))
        status = int(sess.status.item())
        clocks = sampler.window(th0, th1)
        clocks["window"] = "headline timed region"
        if clocks["samples"] < 3:      # a very short headline region: every timed phase
            clocks = sampler.window(th0, t_all1)
            clocks["window"] = "all timed phases (headline, per-stage, end-to-end)"

    # ---- aggregate over ranks (max of the ranks' times)
    total_ms, e2e_ms = replicas.max_over_ranks([total_ms, e2e_ms], device=dev)
    t_step = total_ms / args.steps
    t_e2e = e2e_ms
    value = replicas.job_rate(NQ, world, t_step * 1e-3)
    e2e_value = replicas.job_rate(NQ, world, t_e2e * 1e-3)

    if rank == 0:
        alg, n_tok = algorithmic_bytes(wl)
        flops = algorithmic_flops(wl)
        if fused:   # one kernel does the scoring's work and the selection's
            alg["indexer_score_select"] = alg["indexer_score"] + alg["topk_select"]
            flops["indexer_score_select"] = flops["indexer_score"] + flops["topk_select"]
        hbm, bf16, bf16_sus, src = measured_peaks()
        # Every stage against its bound: tensor when its flops take longer at
        # the bf16 peak than its bytes at the HBM peak, else HBM (the kernel's
        # own bytes: top-k counts the score rows it reads).  The per-stage
        # graphs run ks launches back to back, under a second: the burst bf16
        # peak applies.
        kbytes = kernel_bytes(wl, alg)
        stage_roof = {}
        for st in stages:
            t = stage_ms[st] * 1e-3
            tpeak = bf16 if t * ks < 1.0 else bf16_sus
            tr = kernel_traffic(st, args.workload)
            if flops[st] > 0 and flops[st] / (tpeak * 1e12) > kbytes[st] / (hbm * 1e9):
                ach = flops[st] / t / 1e12
                stage_roof[st] = {"bound": "tensor", "achieved": ach, "peak": tpeak, "unit": "TFLOP/s",
                                  "frac": ach / tpeak,
                                  "peak_source": src + (" bf16 burst" if tpeak == bf16 else " bf16 sustained"),
                                  "traffic": tr, "algorithmic_flops": flops[st], "algorithmic_bytes": kbytes[st],
                                  "avg_launch_ms": stage_ms[st]}
            else:
                ach = kbytes[st] / t / 1e9
                stage_roof[st] = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                                  "peak_source": src + " HBM copy", "traffic": tr, "algorithmic_bytes": kbytes[st],
                                  "avg_launch_ms": stage_ms[st]}
        dominant = max(stages, key=lambda st: stage_ms[st])
        roof = dict(stage_roof[dominant], kernel=dominant)
        step_bytes = sum(alg[st] for st in stages)
        cpu = None
        if not args.no_cpu_baseline:
            threads = os.cpu_count() or 1
            rate, done, wall = OracleStep(wl, threads).rate(args.cpu_seconds)
            rate1, done1, wall1 = OracleStep(wl, 1).rate(max(1.0, args.cpu_seconds / 3))
            cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                   "cpu_model": cpu_model(),
                   "sample": f"{done} whole queries of this workload in {wall:.1f} s (compress of the step's new "
                             f"pools, scores over all visible pools, top-k, attention), OpenMP over queries",
                   "single_thread": {"value": rate1, "unit": "tokens/s", "cores": 1,
                                     "sample": f"{done1} whole queries in {wall1:.1f} s on one thread"}}
        line = {
            "metric": METRIC[args.workload], "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": DESCR[args.workload], "batch": wl.B, "queries": NQ,
                       "ctx": int(wl.lens.max()), "topk_tokens": wl.spec.topk_tokens,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "caches": f"paged, {args.paged}-token pages (block table)" if args.paged else "contiguous",
                       "select": ("fused: scores and top-k in one kernel, no score matrix" if fused else
                                  "staged: score matrix in the workspace, then top-k")
                                 + ("; later queries of a sequence share its first query's selection"
                                    if args.share_mtp else ""),
                       "l2": "flushed between timed steps (256 MB read)", "timing": "CUDA-graph replay, events"},
            "roofline": roof,
            "stage_roofline": stage_roof,
            "step_roofline": {"algorithmic_bytes": step_bytes, "achieved_GBps": step_bytes / (t_step * 1e-3) / 1e9,
                              "frac": step_bytes / (t_step * 1e-3) / 1e9 / hbm},
            "stage_ms": stage_ms,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "path": "Step.run_host from pinned memory: q_lat crosses on a second stream while compress, "
                            "score and top-k run; batches of at least 512 queries then pipeline chunks of 256 "
                            "(q_lat in, attention, out and lse back)"},
            "gpu_launches": step.launches_per_step() * args.steps,
            "clocks": clocks,
            "device_status": status,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
