#!/usr/bin/env python
"""Throughput bench of the MX-scaled FP8 wo_a path on GB300.

One step = the wo_a forward of one 8K-token prefill chunk: fused inverse
RoPE + group-128 quantisation of x [8192, 8, 4096] (BF16) followed by the
block-scaled batched GEMM against W [8, 1024, 4096] (E4M3 + E8M0 scales),
output [8192, 8, 1024] BF16.  Inputs are resident in HBM; the weight set
rotates over 8 distinct sets (256 MiB) and x alone is 512 MiB, so every
step streams operands larger than the 129 MB L2.

The JSON line reports tokens/s over exactly --steps steps (CUDA events on
the launching stream, barrier + synchronize on both sides, max over ranks),
the end-to-end figure through the public API with pinned host buffers, the
roofline of the dominant kernel (the GEMM, against the dense FP8 tensor
peak), secondary workloads (decode latency per layer, the unaligned-K
linear, the dequantiser, the 100K-token stream), the CPU oracle timed on a
bounded sample, and the SM clocks sampled during the timed region.

--impl reference times the CPU oracle (the reference arm)
on bounded samples of the same workload.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

if "--impl" in sys.argv and "reference" in sys.argv:
    # The oracle arm runs single-threaded so that `cores` is exact.
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

T_PREFILL, G, D, N, R = 8192, 8, 4096, 1024, 64
KG = D // 128
N_WSETS = 8
METRIC = "wo_a FP8 path tokens/s @8K prefill"
UNIT = "tokens/s"
L2_BYTES = 129 * 1024 * 1024


def gemm_flops(T):
    return 2.0 * T * G * N * D


def quant_bytes(T):
    # x read, codes + scale bytes written, position read, cos+sin rows read
    return T * (2 * G * D + G * D + G * KG + 8 + 2 * (R // 2) * 2)


def gemm_bytes(T):
    # weight codes + raw scale bytes, activation codes + scale bytes, BF16 output
    return G * N * D + G * N * KG + T * G * (D + KG) + 2 * T * G * N


def wo_a_bytes(T):
    # the whole projection in one launch: x read, positions and cos/sin rows read,
    # weight codes + raw scale bytes read, BF16 output written (the activation
    # codes never need to leave the chip)
    return T * (2 * G * D + 8 + 2 * (R // 2) * 2) + G * N * D + G * N * KG + 2 * T * G * N


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def measured_traffic(key):
    """DRAM bytes per launch from the committed ncu capture, or None when the
    kernel source has changed since that capture."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = dict(p.split("=", 1) for p in line.split()[1:] if "=" in p)
            if line.split() and line.split()[0] == key:
                src = os.path.join(ROOT, parts["source"])
                with open(src, "rb") as g:
                    if hashlib.sha256(g.read()).hexdigest()[:16] != parts["sha256_16"]:
                        return None
                return int(parts["bytes"])
    return None


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        top = max(sm) if sm else None
        loaded = [v for v in sm if top and v >= 0.5 * top] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": num(rows[0][2]), "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ------------------------------------------------------------- GPU helpers
def make_weights(mxq, n_sets, seed, device):
    """Distinct weight sets: FP32 N(0, 0.02) quantised per row in groups of 128
    by the library's own quantiser (R = 0), scales prepared for the GEMM."""
    import workloads as W

    sets = []
    for i in range(n_sets):
        wf = W.f32_normal_cuda((G * N, 1, D), seed=seed + i, std=0.02, device=device)
        wq, ws = mxq.mxq_inv_rope_group_quant(wf.to(torch.bfloat16), R=0)
        wq = wq.view(G, N, D)
        ws = ws.view(G, N, KG)
        sets.append((wq, mxq.mxq_prepare_weight_scales(ws, D), ws))
        del wf
    return sets


def time_graph(fn, reps, warm=3):
    """Capture fn() into a CUDA graph, replay it `reps` times; ms per replay."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(warm):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def rope_tables(max_pos, device):
    import workloads as W

    c, s = W.rope_cache(max_pos, R)
    return c.to(device), s.to(device)


def secondary(mxq, device, peaks):
    import workloads as W

    out = {}
    hbm = peaks["hbm_gbs"]
    cos, sin = rope_tables(32768, device)
    # wo_a decode: 61 layers with distinct weights (2 GB, far above L2) in one graph.
    layers = 61
    wsets = make_weights(mxq, layers, seed=5000, device=device)
    dec = {}
    for T in W.DECODE_T:
        x = W.bf16_normal_cuda((T, G, D), seed=6000 + T, device=device)
        pos = W.positions_uniform_cuda(T, seed=6100 + T, max_pos=32768, device=device)
        q = torch.empty((T, G, D), dtype=torch.uint8, device=device)
        sc = torch.empty((T, G, KG), dtype=torch.uint8, device=device)
        o = torch.empty((T, G, N), dtype=torch.bfloat16, device=device)

        need = mxq.mxq_wo_a_workspace_bytes(T, G, D, N)
        wo_ws = torch.empty(need, dtype=torch.uint8, device=device) if need else None

        def layer_stack():  # the product path: mxq_wo_a, one call per layer
            for wq, wsf, _ in wsets:
                mxq.wo_a(x, pos, cos, sin, wq, wsf, R=R, out=o, ws=wo_ws)

        def two_kernel_stack():  # quantiser + GEMM as two launches, for comparison
            for wq, wsf, _ in wsets:
                mxq.mxq_inv_rope_group_quant(x, pos, cos, sin, R, q=q, sc=sc)
                mxq.mxq_bmm_a8w8(q, sc, wq, wsf, out=o)

        ms = time_graph(layer_stack, 20)
        ms2 = time_graph(two_kernel_stack, 20)
        us = ms * 1e3 / layers
        us2 = ms2 * 1e3 / layers
        # algorithmic bytes of the fused layer: weights + scales, x, positions, cos/sin, output
        byt = G * N * D + G * N * KG + T * (2 * G * D + 8 + 2 * (R // 2) * 2) + 2 * T * G * N
        dec[str(T)] = {"us_per_layer": round(us, 2), "hbm_frac": round(byt / (us * 1e-6) / 1e9 / hbm, 3),
                       "gbs": round(byt / (us * 1e-6) / 1e9, 1),
                       "two_kernel_us_per_layer": round(us2, 2)}
    out["decode_wo_a"] = {"workload": "x [T,8,4096], W [8,1024,4096], 61 distinct layers in one CUDA graph; "
                                      "mxq_wo_a per layer (one fused launch for T <= 32, quantiser + GEMM above)",
                          "per_T": dec}
    del wsets
    torch.cuda.empty_cache()

    # Unaligned-K MXFP8 linear and the dequantiser: N=5120, K in {576, 288, 2304},
    # enough distinct weight sets per K that one pass streams more than 3 x L2
    # (codes + prepared scales), so no call finds its weight in L2.
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    lin = {}
    for K in W.LINEAR_K:
        kg = (K + 127) // 128
        per_set = W.LINEAR_N * K + mxq.mxq_weight_scale_bytes(1, W.LINEAR_N, K)
        n_sets = max(40, -(-3 * l2 // per_set) + 1)
        sets = []
        for i in range(n_sets):
            wf = W.f32_normal_cuda((W.LINEAR_N, 1, K), seed=7000 + 50 * K + i, std=0.02, device=device)
            wq, ws = mxq.mxq_inv_rope_group_quant(wf.to(torch.bfloat16), R=0)
            sets.append((wq.view(W.LINEAR_N, K), ws.view(1, W.LINEAR_N, kg),
                         mxq.mxq_prepare_weight_scales(ws.view(1, W.LINEAR_N, kg), K)))
        res = {}
        for M in W.LINEAR_M:
            x = W.bf16_normal_cuda((M, K), seed=7100 + M, device=device)
            o = torch.empty((M, W.LINEAR_N), dtype=torch.bfloat16, device=device)
            need = mxq.mxq_linear_workspace_bytes(M, W.LINEAR_N, K)
            ws_buf = torch.empty(need, dtype=torch.uint8, device=device) if need else None

            def lin_stack():
                for wq, _, wsf in sets:
                    mxq.mxq_linear(x, wq, wsf, out=o, ws=ws_buf)

            us = time_graph(lin_stack, 20) * 1e3 / len(sets)
            byt = W.LINEAR_N * K + W.LINEAR_N * kg + 2 * M * K + 2 * M * W.LINEAR_N  # fused: x read once
            res[f"M{M}"] = {"us": round(us, 2), "gbs": round(byt / (us * 1e-6) / 1e9, 1),
                            "hbm_frac": round(byt / (us * 1e-6) / 1e9 / hbm, 3)}
        res["weight_sets"] = n_sets
        res["weight_bytes_per_pass"] = n_sets * per_set
        deq_out = torch.empty((1, W.LINEAR_N, K), dtype=torch.bfloat16, device=device)

        def deq_stack():
            for wq, ws, _ in sets:
                mxq.mxq_dequant_bf16(wq.view(1, W.LINEAR_N, K), ws, out=deq_out)

        us = time_graph(deq_stack, 20) * 1e3 / len(sets)
        byt = 3 * W.LINEAR_N * K + W.LINEAR_N * kg
        res["dequant"] = {"us": round(us, 2), "gbs": round(byt / (us * 1e-6) / 1e9, 1),
                          "hbm_frac": round(byt / (us * 1e-6) / 1e9 / hbm, 3)}
        lin[str(K)] = res
        del sets
    out["linear_unaligned_k"] = {"workload": "N=5120, distinct weight sets per K streaming > 3 x L2 "
                                             "per pass, CUDA graph", "l2_bytes": l2, "per_K": lin}
    torch.cuda.empty_cache()
    return out


def kv_insert_bench(mxq, device, peaks):
    """Forward RoPE + KV-cache insert (E4M3 cache, per-tensor scale): a prefill
    chunk q [8192, 64, 512] / kv [8192, 512] (query out of place and in place),
    and decode T = 1 / 8 / 64 over 61 layers with distinct caches in one CUDA
    graph."""
    import workloads as W

    H, Dh, Rk = 64, 512, 64
    hbm = peaks["hbm_gbs"]
    cos, sin = rope_tables(65536, device)
    scale = torch.tensor([0.0371], dtype=torch.float32, device=device)
    out = {}
    T = 8192
    q = W.bf16_normal_cuda((T, H, Dh), seed=8100, device=device)
    kv = W.bf16_normal_cuda((T, Dh), seed=8101, std=4.0, device=device)
    pos = torch.arange(32768, 32768 + T, dtype=torch.int64, device=device)
    slots = torch.randperm(4 * T, device=device)[:T].to(torch.int64)
    cache = torch.zeros((4 * T, Dh), dtype=torch.uint8, device=device)
    q_out = torch.empty_like(q)
    side = T * (2 * Dh + Dh + 8 + 8 + 2 * Rk)  # kv read, cache row written, pos, slot, cos/sin
    for name, qo, byt in (("prefill_out_of_place", q_out, 2 * (2 * T * H * Dh) + side),
                          ("prefill_in_place", q, 2 * (2 * T * H * Rk) + side)):
        for _ in range(5):
            mxq.mxq_rope_kv_insert(q, kv, pos, cos, sin, Rk, slots, cache, scale=scale, q_out=qo)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 20
        a.record()
        for _ in range(reps):
            mxq.mxq_rope_kv_insert(q, kv, pos, cos, sin, Rk, slots, cache, scale=scale, q_out=qo)
        b.record()
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / reps
        out[name] = {"us": round(us, 2), "algorithmic_bytes": byt, "gbs": round(byt / (us * 1e-6) / 1e9, 1),
                     "hbm_frac": round(byt / (us * 1e-6) / 1e9 / hbm, 3)}
    out["prefill_out_of_place"]["traffic"] = measured_traffic("rope_kv_insert_prefill_8k")
    del q, kv, q_out, cache
    torch.cuda.empty_cache()
    dec = {}
    layers = 61
    for T in (1, 8, 64):
        q = W.bf16_normal_cuda((T, H, Dh), seed=8200 + T, device=device)
        kv = W.bf16_normal_cuda((T, Dh), seed=8300 + T, std=4.0, device=device)
        pos = W.positions_uniform_cuda(T, seed=8400 + T, max_pos=65536, device=device)
        slots = torch.arange(T, dtype=torch.int64, device=device) * 7
        caches = [torch.zeros((8 * T, Dh), dtype=torch.uint8, device=device) for _ in range(layers)]
        q_out = torch.empty_like(q)

        def stack():
            for c in caches:
                mxq.mxq_rope_kv_insert(q, kv, pos, cos, sin, Rk, slots, c, scale=scale, q_out=q_out)

        us = time_graph(stack, 20) * 1e3 / layers
        byt = 2 * (2 * T * H * Dh) + T * (2 * Dh + Dh + 8 + 8 + 2 * Rk)
        dec[str(T)] = {"us_per_layer": round(us, 2), "gbs": round(byt / (us * 1e-6) / 1e9, 1)}
    out["decode"] = dec
    out["workload"] = ("q [T,64,512] bf16, kv [T,512] bf16, R=64, E4M3 cache with per-tensor scale; "
                       "prefill T=8192 at positions 32768.., decode 61 layers in one CUDA graph")
    return out


def stream_100k(mxq, device):
    """100,000-token prefill stream (12 x 8192 + 1696) through 61 wo_a layers."""
    import workloads as W

    cos, sin = rope_tables(100000, device)
    wsets = make_weights(mxq, W.STREAM_LAYERS, seed=9000, device=device)
    chunks, start = [], 0
    for i, T in enumerate(W.STREAM_CHUNKS):
        x = W.bf16_normal_cuda((T, G, D), seed=9500 + i, device=device)
        pos = torch.arange(start, start + T, dtype=torch.int64, device=device)
        chunks.append((x, pos))
        start += T
    o = torch.empty((8192, G, N), dtype=torch.bfloat16, device=device)
    ws = torch.empty(mxq.mxq_wo_a_workspace_bytes(8192, G, D, N), dtype=torch.uint8, device=device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(chunks) + 1)]

    def run():  # mxq_wo_a per (chunk, layer): one launch each
        for ci, (x, pos) in enumerate(chunks):
            ev[ci].record()
            T = x.shape[0]
            for wq, wsf, _ in wsets:
                mxq.wo_a(x, pos, cos, sin, wq, wsf, R=R, out=o[:T], ws=ws)
        ev[-1].record()

    run()
    torch.cuda.synchronize()
    run()
    torch.cuda.synchronize()
    per_chunk = [ev[i].elapsed_time(ev[i + 1]) for i in range(len(chunks))]
    total = ev[0].elapsed_time(ev[-1])
    del wsets, chunks
    torch.cuda.empty_cache()
    return {"workload": "12x8192 + 1696 tokens, positions 0..99999, 61 distinct layers",
            "tokens_per_s": round(100000 / (total * 1e-3), 1), "total_ms": round(total, 3),
            "chunk8192_ms_median": round(statistics.median(per_chunk[:-1]), 3),
            "chunk1696_ms": round(per_chunk[-1], 3)}


# ----------------------------------------------------------- CPU oracle leg
def oracle_sample_run(tokens, seed):
    """One oracle pass (quantiser + fp64 GEMM) over `tokens` tokens of the 8K
    chunk workload; returns elapsed seconds."""
    import workloads as W
    from oracle import mx_oracle as O

    x = W.bf16_normal((tokens, G, D), seed=seed, outlier_frac=0.01)
    pos = W.positions_arange(seed % 4096, tokens).numpy()
    cos, sin = _oracle_tables()
    w_codes, w_scales = _oracle_weights()
    t0 = time.perf_counter()
    a, sa = O.inv_rope_group_quant(W.bf16_bits(x), pos, cos, sin, R)
    O.bmm_a8w8_ref(a, sa, w_codes, w_scales)
    return time.perf_counter() - t0


_cache = {}


def _oracle_tables():
    import workloads as W

    if "cs" not in _cache:
        c, s = W.rope_cache(8192, R)
        _cache["cs"] = (W.bf16_bits(c), W.bf16_bits(s))
    return _cache["cs"]


def _oracle_weights():
    import workloads as W
    from oracle import mx_oracle as O

    if "w" not in _cache:
        wf = W.f32_normal((G, N, D), seed=3, std=0.02).numpy()
        _cache["w"] = O.group_quant_rows(wf)
    return _cache["w"]


def _oracle_subprocess(code, threads):
    """Runs oracle timing code in a fresh interpreter whose BLAS and OpenMP use
    exactly `threads` threads (the thread count must be fixed before numpy
    loads); returns its last output line as JSON, or None."""
    n = str(threads)
    env = dict(os.environ, OPENBLAS_NUM_THREADS=n, OMP_NUM_THREADS=n, MKL_NUM_THREADS=n)
    r = subprocess.run([sys.executable, "-c", code], env=env, stdout=subprocess.PIPE,
                       stderr=subprocess.PIPE, text=True, timeout=900)
    if r.returncode != 0:
        return None
    return json.loads(r.stdout.strip().splitlines()[-1])


def _oracle_budget_code(budget_s):
    return ("import sys,json,time; sys.path.insert(0, %r); import bench\n"
            "bench._oracle_weights(); bench._oracle_tables()\n"
            "tok, el, i = 0, 0.0, 0\n"
            "while el < %f:\n"
            "    el += bench.oracle_sample_run(16, 100 + i); tok += 16; i += 1\n"
            "print(json.dumps({'tokens': tok, 'seconds': el}))\n") % (ROOT, budget_s)


def cpu_baseline(budget_s=12.0):
    """Oracle throughput on the host cores on bounded samples: one thread (the
    reported value), and every core (BLAS threads = the core count) beside it."""
    d = _oracle_subprocess(_oracle_budget_code(budget_s), 1)
    if d is None:
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": "failed"}
    line = {"value": round(d["tokens"] / d["seconds"], 3), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{d['tokens']} tokens of the 8K chunk in batches of 16 (x [16,8,4096] -> "
                      f"quantiser + fp64 GEMM against W [8,1024,4096]), {d['seconds']:.1f} s, "
                      f"one thread"}
    ncores = os.cpu_count() or 1
    da = _oracle_subprocess(_oracle_budget_code(budget_s * 0.5), ncores)
    if da is not None:
        line["all_cores"] = {"value": round(da["tokens"] / da["seconds"], 3), "unit": UNIT,
                             "cores": ncores,
                             "sample": f"{da['tokens']} tokens, {da['seconds']:.1f} s, BLAS on "
                                       f"{ncores} threads (the quantiser part is single-threaded numpy)"}
    return line


# ---------------------------------------------------------- multi-rank glue
def rank_env():
    """(world size, rank, local rank) as torchrun sets them; one process = 1."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value, device=None):
    """The largest `value` over all ranks: a job's step time is its slowest
    rank's.  Identity outside a process group of more than one rank."""
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    on = device if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=on)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, units_per_rank, ms_step):
    """Whole-job rate: every rank processes its own units (weak scaling, no
    exchange) and the job takes as long as its slowest rank."""
    return world * units_per_rank / (ms_step * 1e-3)


def prefill_config(world):
    """The headline workload, as both arms report it."""
    return {"workload": "wo_a prefill chunk: x [8192,8,4096] bf16 (1% x50 outliers), "
                        "positions 0..8191, R=64 -> inverse RoPE + group-128 quant -> "
                        "block-scaled bmm with W [8,1024,4096] e4m3+e8m0 -> [8192,8,1024] bf16",
            "weight_sets": N_WSETS,
            "l2": "inputs larger than L2 (x 512 MiB; 8 rotating weight sets 256 MiB)",
            "parallelism": f"replicas x{world}, one 8K chunk per GPU"}


def run_reference(args, rank):
    if rank != 0:
        return
    per_step = 16
    # The oracle runs in a fresh interpreter pinned to one thread (this
    # process's numpy has already chosen its BLAS thread count).
    code = ("import sys,json; sys.path.insert(0, %r); import bench\n"
            "bench._oracle_weights(); bench._oracle_tables()\n"
            "for i in range(%d): bench.oracle_sample_run(%d, 10 + i)\n"
            "el = sum(bench.oracle_sample_run(%d, 1000 + i) for i in range(%d))\n"
            "print(json.dumps({'seconds': el}))\n") % (ROOT, args.warmup, per_step, per_step,
                                                        args.steps)
    d = _oracle_subprocess(code, 1)
    if d is None:
        print(json.dumps({"impl": "reference", "unavailable": "the oracle run failed"}), flush=True)
        return
    el = d["seconds"]
    value = per_step * args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": prefill_config(1),
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"each step the oracle (quantiser + fp64 GEMM) on {per_step} "
                                       "tokens of the 8K chunk, one thread"},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def single_workload(mxq, device, peaks, args):
    """Eager run of one secondary workload (decode layer or MXFP8 linear over 24
    distinct weight sets, or the KV insert over 4 caches): --warmup passes,
    then --steps timed calls."""
    import workloads as W

    n_sets = 24
    if args.workload == "decode":
        T = args.tokens
        wsets = make_weights(mxq, n_sets, seed=5000, device=device)
        cos, sin = rope_tables(32768, device)
        x = W.bf16_normal_cuda((T, G, D), seed=6000 + T, device=device)
        pos = W.positions_uniform_cuda(T, seed=6100 + T, max_pos=32768, device=device)
        o = torch.empty((T, G, N), dtype=torch.bfloat16, device=device)
        need = mxq.mxq_wo_a_workspace_bytes(T, G, D, N)
        ws = torch.empty(need, dtype=torch.uint8, device=device) if need else None

        def call(i):
            wq, wsf, _ = wsets[i % n_sets]
            mxq.wo_a(x, pos, cos, sin, wq, wsf, R=R, out=o, ws=ws)

        byt = G * N * D + G * N * KG + T * (2 * G * D + 8 + 2 * (R // 2) * 2) + 2 * T * G * N
        desc = f"wo_a decode x [{T},8,4096] -> [{T},8,1024], W [8,1024,4096], {n_sets} weight sets"
    elif args.workload == "kv":
        T, Hq, Dh, Rk = args.tokens, 64, 512, 64
        q = W.bf16_normal_cuda((T, Hq, Dh), seed=8100, device=device)
        kv = W.bf16_normal_cuda((T, Dh), seed=8101, std=4.0, device=device)
        pos = torch.arange(32768, 32768 + T, dtype=torch.int64, device=device)
        cos, sin = rope_tables(32768 + T, device)
        slots = torch.randperm(4 * T, device=device)[:T].to(torch.int64)
        caches = [torch.zeros((4 * T, Dh), dtype=torch.uint8, device=device) for _ in range(4)]
        scale = torch.tensor([0.0371], dtype=torch.float32, device=device)
        q_out = torch.empty_like(q)

        def call(i):
            mxq.mxq_rope_kv_insert(q, kv, pos, cos, sin, Rk, slots, caches[i % 4], scale=scale, q_out=q_out)

        byt = 2 * (2 * T * Hq * Dh) + T * (2 * Dh + Dh + 8 + 8 + 2 * Rk)
        desc = f"forward RoPE + E4M3 KV insert, q [{T},64,512] out of place, kv [{T},512]"
    else:
        M, K, Nl = args.tokens, args.k, W.LINEAR_N
        kg = (K + 127) // 128
        sets = []
        for i in range(n_sets):
            wf = W.f32_normal_cuda((Nl, 1, K), seed=7000 + i, std=0.02, device=device)
            wq, wsc = mxq.mxq_inv_rope_group_quant(wf.to(torch.bfloat16), R=0)
            sets.append((wq.view(Nl, K), mxq.mxq_prepare_weight_scales(wsc.view(1, Nl, kg), K)))
        x = W.bf16_normal_cuda((M, K), seed=7100 + M, device=device)
        o = torch.empty((M, Nl), dtype=torch.bfloat16, device=device)
        need = mxq.mxq_linear_workspace_bytes(M, Nl, K)
        ws = torch.empty(need, dtype=torch.uint8, device=device) if need else None

        def call(i):
            wq, wsf = sets[i % n_sets]
            mxq.mxq_linear(x, wq, wsf, out=o, ws=ws)

        byt = Nl * K + Nl * kg + 2 * M * K + 2 * M * Nl
        desc = f"MXFP8 linear x [{M},{K}] -> [{M},{Nl}], {n_sets} weight sets"
    for i in range(max(args.warmup, 1) * n_sets):
        call(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(args.steps):
        call(i)
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / args.steps
    if mxq.mxq_watchdog_read() != 0:
        raise SystemExit("a bounded wait inside a kernel ran out")
    return {"workload": args.workload, "config": desc, "steps": args.steps, "us_per_call": round(us, 3),
            "gbs": round(byt / (us * 1e-6) / 1e9, 1),
            "hbm_frac": round(byt / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4), "timing": "eager, back to back"}


# ------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--workload", choices=["prefill", "decode", "linear", "kv"], default="prefill",
                    help="prefill (default, the headline); decode / linear / kv: a short eager run "
                         "of that workload alone (for profiling), its own JSON line")
    ap.add_argument("--tokens", type=int, default=1, help="T (decode, kv) or M (linear)")
    ap.add_argument("--k", type=int, default=576, help="K of the linear workload")
    args = ap.parse_args()

    world, rank, local_rank = rank_env()
    if args.impl == "reference":
        return run_reference(args, rank)

    import torch.distributed as dist

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    def barrier():
        if world > 1:
            dist.barrier()

    from mxfp8_block_scaled_inv_gb300 import build as B

    if rank == 0:
        B.build()
    barrier()
    import mxfp8_block_scaled_inv_gb300 as mxq
    import workloads as W

    mxq.lib()
    peaks = load_peaks()
    torch.manual_seed(0)
    if args.workload != "prefill":
        if rank == 0:
            print(json.dumps(single_workload(mxq, device, peaks, args)), flush=True)
        return

    # Inputs resident in HBM.  Each rank owns its own chunk (weak scaling, no exchange).
    x = W.bf16_normal_cuda((T_PREFILL, G, D), seed=400 + rank, outlier_frac=0.01, device=device)
    pos = torch.arange(0, T_PREFILL, dtype=torch.int64, device=device)
    cos, sin = rope_tables(T_PREFILL, device)
    wsets = make_weights(mxq, N_WSETS, seed=100, device=device)
    q = torch.empty((T_PREFILL, G, D), dtype=torch.uint8, device=device)
    sc = torch.empty((T_PREFILL, G, KG), dtype=torch.uint8, device=device)
    out = torch.empty((T_PREFILL, G, N), dtype=torch.bfloat16, device=device)
    wo_ws = torch.empty(mxq.mxq_wo_a_workspace_bytes(T_PREFILL, G, D, N), dtype=torch.uint8,
                        device=device)
    stream = torch.cuda.current_stream()

    def step(i, evs=None):
        # One library call: the quantising CTA-pair GEMM (one kernel, after a
        # clear of its job counters).
        wq, wsf, _ = wsets[i % N_WSETS]
        if evs is not None:
            evs[0].record(stream)
        mxq.wo_a(x, pos, cos, sin, wq, wsf, R=R, out=out, ws=wo_ws, stream=stream)
        if evs is not None:
            evs[1].record(stream)

    def two_kernel_step(i, evs=None):
        # The same projection as quantiser + GEMM (two kernels), for comparison.
        wq, wsf, _ = wsets[i % N_WSETS]
        if evs is not None:
            evs[0].record(stream)
        mxq.mxq_inv_rope_group_quant(x, pos, cos, sin, R, q=q, sc=sc, stream=stream)
        if evs is not None:
            evs[1].record(stream)
        mxq.mxq_bmm_a8w8(q, sc, wq, wsf, out=out, stream=stream)
        if evs is not None:
            evs[2].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    barrier()

    clocks = ClockSampler(local_rank)
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    t_host1 = time.time()
    clocks.stop()
    clk = clocks.summary(t_host0, t_host1)

    ms_total = start.elapsed_time(end)
    ms_step = ms_total / args.steps
    # A step is one launch of the quantising GEMM, so its kernel time is the
    # step time (launches back to back, as in use).  For comparison, the same
    # launch bracketed by CUDA events one at a time, over at least 50 launches
    # (the events break the overlap of consecutive launches, so this reads a
    # little longer).
    n_br = max(50, min(args.steps, 100))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_br)]
    for i, e in enumerate(evs):
        step(i, e)
    torch.cuda.synchronize()
    t_bracketed = sum(e[0].elapsed_time(e[1]) for e in evs) / n_br
    t_fused = ms_step
    ms_step = max_over_ranks(ms_step, device)
    value = job_throughput(world, T_PREFILL, ms_step)

    # The same projection as quantiser + GEMM (two kernels), for comparison:
    # steps back to back for the step time, then bracketed ones for the
    # per-kernel times and rooflines.
    n_two = max(10, min(args.steps, 50))
    for i in range(args.warmup):
        two_kernel_step(i)
    torch.cuda.synchronize()
    a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a2.record(stream)
    for i in range(n_two):
        two_kernel_step(i)
    b2.record(stream)
    evs2 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(50)]
    for i, e in enumerate(evs2):
        two_kernel_step(i, e)
    torch.cuda.synchronize()
    ms_two = a2.elapsed_time(b2) / n_two
    t_quant = sum(e[0].elapsed_time(e[1]) for e in evs2) / len(evs2)
    t_gemm = sum(e[1].elapsed_time(e[2]) for e in evs2) / len(evs2)

    # End to end through the public API: pinned host x -> device, wo_a, output
    # -> host, every step.  The steps are pipelined on three streams (copy
    # in, compute, copy out) with double-buffered device buffers, so the host
    # link carries step i+1's input while step i computes and its output
    # returns; the timed region runs from the first input copy to the last
    # output copy.
    x_host = x.cpu().pin_memory()
    pos_host = pos.cpu().pin_memory()
    out_host = torch.empty((T_PREFILL, G, N), dtype=torch.bfloat16).pin_memory()
    x_dev = [torch.empty_like(x) for _ in range(2)]
    pos_dev = [torch.empty_like(pos) for _ in range(2)]
    out_dev = [torch.empty((T_PREFILL, G, N), dtype=torch.bfloat16, device=device)
               for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 20))
    s_in, s_comp, s_out = (torch.cuda.Stream(device=device) for _ in range(3))

    def e2e_run(nsteps, first=0):
        read_done = [None, None]  # compute finished reading x_dev[b]
        sent_done = [None, None]  # out_dev[b] copied to the host
        last = None
        for i in range(first, first + nsteps):
            bb = i % 2
            wq, wsf, _ = wsets[i % N_WSETS]
            with torch.cuda.stream(s_in):
                if read_done[bb] is not None:
                    s_in.wait_event(read_done[bb])
                x_dev[bb].copy_(x_host, non_blocking=True)
                pos_dev[bb].copy_(pos_host, non_blocking=True)
                e_in = torch.cuda.Event()
                e_in.record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(e_in)
                if sent_done[bb] is not None:
                    s_comp.wait_event(sent_done[bb])
                mxq.wo_a(x_dev[bb], pos_dev[bb], cos, sin, wq, wsf, R=R, out=out_dev[bb], ws=wo_ws,
                         stream=s_comp)
                e_c = torch.cuda.Event()
                e_c.record(s_comp)
                read_done[bb] = e_c
            with torch.cuda.stream(s_out):
                s_out.wait_event(e_c)
                out_host.copy_(out_dev[bb], non_blocking=True)
                e_o = torch.cuda.Event()
                e_o.record(s_out)
                sent_done[bb] = e_o
                last = e_o
        return last

    e2e_run(3)
    torch.cuda.synchronize()
    barrier()
    a = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    last = e2e_run(e2e_steps, first=3)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s_out):
        s_out.wait_event(last)
        b.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(b) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, device)
    e2e_value = job_throughput(world, T_PREFILL, e2e_ms)
    h2d = x_host.numel() * 2 + pos_host.numel() * 8
    d2h = out_host.numel() * 2
    del x_host, out_host

    # The launches are sub-millisecond and timed in a run of a few seconds:
    # the burst peak applies (dense FP8 = 2 x dense BF16, the nominal ratio).
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    fused_tflops = gemm_flops(T_PREFILL) / (t_fused * 1e-3) / 1e12
    gemm_tflops = gemm_flops(T_PREFILL) / (t_gemm * 1e-3) / 1e12
    quant_gbs = quant_bytes(T_PREFILL) / (t_quant * 1e-3) / 1e9

    traffic = measured_traffic("wo_a_prefill_8k")
    sec = {}
    if not args.no_secondary and rank == 0:
        sec = secondary(mxq, device, peaks)
        sec["stream_100k"] = stream_100k(mxq, device)
        sec["rope_kv_insert"] = kv_insert_bench(mxq, device, peaks)
    if mxq.mxq_watchdog_read() != 0:
        raise SystemExit("a bounded wait inside a kernel ran out; numbers are not valid")

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic",
            "config": prefill_config(world),
            "gpu_launches": args.steps,
            "breakdown_ms": {"wo_a_one_launch": round(t_fused, 5),
                             "wo_a_one_launch_bracketed": round(t_bracketed, 5),
                             "bracketed_launches": n_br},
            "roofline": {"bound": "tensor",
                         "kernel": "bmm_a8w8 quantising CTA-pair form (the whole wo_a chunk, one launch)",
                         "achieved": round(fused_tflops, 1), "peak": round(fp8_peak, 1),
                         "unit": "TFLOP/s", "frac": round(fused_tflops / fp8_peak, 4),
                         "traffic": traffic,
                         "algorithmic_bytes": wo_a_bytes(T_PREFILL),
                         "traffic_over_algorithmic": (round(traffic / wo_a_bytes(T_PREFILL), 3)
                                                      if traffic else None),
                         "kernel_ms": round(t_fused, 5),
                         "peak_source": f"{peaks['source']}: 2 x burst bf16 "
                                        f"{peaks['bf16_tflops']} TFLOP/s (fp8/bf16 nominal 4.5/2.25)"},
            "two_kernel": {
                "what": "the same chunk as quantiser + GEMM (two launches)",
                "ms_per_step": round(ms_two, 5),
                "value": round(T_PREFILL / (ms_two * 1e-3), 1),
                "breakdown_ms": {"quant": round(t_quant, 5), "gemm": round(t_gemm, 5)},
                "gemm_roofline": {"bound": "tensor", "achieved": round(gemm_tflops, 1),
                                  "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                                  "frac": round(gemm_tflops / fp8_peak, 4),
                                  "traffic": measured_traffic("bmm_a8w8_prefill_8k")},
                "quantiser_roofline": {"bound": "hbm", "achieved": round(quant_gbs, 1),
                                       "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                       "frac": round(quant_gbs / peaks["hbm_gbs"], 4),
                                       "traffic": measured_traffic("inv_rope_group_quant_prefill_8k")}},
            "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                    "schedule": "mxq_wo_a per step; copy-in, compute and copy-out on three "
                                "streams, double-buffered device buffers"},
            "clocks": clk,
            "secondary": sec,
        }
        if not args.no_cpu and world == 1:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    barrier()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
