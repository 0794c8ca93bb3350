"""Throughput of the dense steps either side of the DSA step on one GPU, each
library call beside the same products through torch (cuBLAS), on random
weights of the GLM-5.3-Flash widths.

    python -m dsa_indexer_sparse_kpool_b300.bench_dense [--tokens 32 4096] [--reps 50]

Prints one JSON line per (call, token count): the call's median time over
``reps`` launches (CUDA events on the launching stream, L2 flushed before
every launch), cuBLAS's median for the same products, the algorithmic flops
and bytes (operands read once, outputs written once), and the fraction of the
bound that applies (bf16 tensor peak when the flops take longer at that peak
than the bytes at the HBM peak, else HBM), against the measured peaks in
MEASURED_PEAKS.json when present.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics

import torch

import dsa_indexer_sparse_kpool_b300 as kp
import kpool_inputs as KI

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6400.0, 1800.0, "fallback"


def timed(fn, reps, flush):
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    for a, b in ev:
        flush.sum()
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def cases(T: int, pj: KI.Projections):
    """(name, library call, torch call, flops, bytes) for T tokens."""
    d = {k: getattr(pj, k).cuda() for k in ("hidden", "q_lora", "q_nope", "out_lat", "w_iq", "w_ik", "w_ig", "w_iw",
                                            "w_uk", "w_uv", "w_o")}
    bf, f32 = torch.bfloat16, torch.float32
    q_idx = torch.empty(T, 32, 128, dtype=bf, device="cuda")
    keys = torch.empty(T, 128, dtype=bf, device="cuda")
    gates = torch.empty(T, 128, dtype=bf, device="cuda")
    w = torch.empty(T, 32, dtype=f32, device="cuda")
    q_lat = torch.zeros(T, 64, 576, dtype=bf, device="cuda")
    o = torch.empty(T, 64, 256, dtype=bf, device="cuda")
    hid = torch.empty(T, 4096, dtype=bf, device="cuda")
    w_kgw = torch.cat([d["w_ik"], d["w_ig"], d["w_iw"]])           # torch: one product for keys, gates, w

    def proj_lib():
        kp.kp_indexer_project(d["hidden"], d["q_lora"], d["w_iq"], d["w_ik"], d["w_ig"], d["w_iw"], q_idx, keys,
                              gates, w)

    def proj_torch():
        torch.matmul(d["q_lora"], d["w_iq"].t())
        torch.matmul(d["hidden"], w_kgw.t())

    def absq_lib():
        kp.kp_mla_absorb_q(d["q_nope"], d["w_uk"], q_lat)

    def absq_torch():
        torch.bmm(d["q_nope"].transpose(0, 1), d["w_uk"].transpose(1, 2))

    def abso_lib():
        kp.kp_mla_absorb_out(d["out_lat"], d["w_uv"], d["w_o"], o, hid)

    def abso_torch():
        oo = torch.bmm(d["out_lat"].transpose(0, 1), d["w_uv"].transpose(1, 2))      # [64][T][256]
        torch.matmul(oo.transpose(0, 1).reshape(T, 64 * 256), d["w_o"].t())

    proj_flops = 2 * T * (4096 * 1536 + (128 + 128 + 32) * 4096)
    proj_bytes = 2 * (4096 * 1536 + 288 * 4096) + 2 * T * (4096 + 1536) + T * (2 * 4096 + 2 * 256 + 4 * 32)
    absq_flops = 2 * T * 64 * 512 * 256
    absq_bytes = 2 * 64 * 512 * 256 + 2 * T * 64 * 256 + 2 * T * 64 * 512
    abso_flops = 2 * T * 64 * 256 * 512 + 2 * T * 4096 * 16384
    abso_bytes = 2 * (64 * 256 * 512 + 4096 * 16384) + 2 * T * 64 * 512 + 2 * T * 64 * 256 * 2 + 2 * T * 4096
    return [("kp_indexer_project", proj_lib, proj_torch, proj_flops, proj_bytes),
            ("kp_mla_absorb_q", absq_lib, absq_torch, absq_flops, absq_bytes),
            ("kp_mla_absorb_out", abso_lib, abso_torch, abso_flops, abso_bytes)]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--tokens", type=int, nargs="+", default=[32, 4096])
    ap.add_argument("--reps", type=int, default=50)
    args = ap.parse_args()
    hbm, bf16, src = peaks()
    flush = torch.empty(256 << 18, dtype=torch.float32, device="cuda").fill_(1.0)   # 256 MB > L2
    for T in args.tokens:
        pj = KI.make_projections(T, seed=11)
        for name, lib_fn, torch_fn, flops, nbytes in cases(T, pj):
            t_lib = timed(lib_fn, args.reps, flush)
            t_ref = timed(torch_fn, args.reps, flush)
            tensor = flops / (bf16 * 1e12) > nbytes / (hbm * 1e9)
            ach = flops / (t_lib * 1e-3) / 1e12 if tensor else nbytes / (t_lib * 1e-3) / 1e9
            peak = bf16 if tensor else hbm
            print(json.dumps({
                "call": name, "tokens": T, "ms": t_lib, "cublas_ms": t_ref, "vs_cublas": t_ref / t_lib,
                "flops": flops, "bytes": nbytes,
                "roofline": {"bound": "tensor" if tensor else "hbm", "achieved": ach, "peak": peak,
                             "unit": "TFLOP/s" if tensor else "GB/s", "frac": ach / peak,
                             "peak_source": src + (" bf16 burst" if tensor else " HBM copy")},
                "l2": "flushed before every launch"}), flush=True)


if __name__ == "__main__":
    main()
