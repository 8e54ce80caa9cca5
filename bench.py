#!/usr/bin/env python
"""Benchmark: the fused GEMM-epilogue chain of a LLaMA-3-1B-shaped block on one GB300.

Workload (one step, all on one GPU, bf16 in / fp32 accumulate / bf16 out):
    M = 16384 tokens, hidden H = 2048, FFN F = 8192, synthetic seeded inputs.
    G1      h = O W_o^T + R, partial sums of squares of h, u = h * g
            (GEMM + residual + partial RMS + RMSNorm-gain broadcast epilogue)
    reduce  r = 1 / sqrt(sum partials / H + eps)      (the light row reduce)
    G2      a = silu(G) U, [G | U] = r (u W_gu^T)     (deferred-r GEMM + SwiGLU epilogue)
    G3      Y = a W_d^T + h                            (GEMM + residual epilogue)
"CODA: new research optimizes Transformer training with GEMM-epilogue programming"
(kucoin.com news flash), sections "El epílogo esconde un tesoro" and "Resultados del
experimento" (LLaMA-style 16K-token batches).

Prints ONE JSON line (rank 0).  `value` is tokens/s over all ranks (each rank runs its own
16384-token replica: the forward rows are independent, so there is no collective in the
data path).  `--impl reference` times the fp64 CPU oracle instead (the slow reference arm).
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused GEMM-epilogue chain TFLOP/s & tokens/s at 16K tokens; % of roofline"
M_TOK, HID, FFN, EPS = 16384, 2048, 8192, 1e-6
WORKLOAD = "LLaMA-3-1B-shaped block forward: attn-out GEMM+residual+partial RMS+gain broadcast -> row reduce " \
           "-> deferred-r gate/up GEMM+SwiGLU -> down GEMM+residual; M=16384 tokens, H=2048, F=8192, bf16"
FLOP = {"G1": 2 * M_TOK * HID * HID, "G2": 2 * M_TOK * 2 * FFN * HID, "G3": 2 * M_TOK * HID * FFN}
CHAIN_FLOP = sum(FLOP.values())
MB = 1e6
# compulsory bytes: each operand read once, each output written once (bf16 = 2 B, fp32 = 4 B)
BYTES = {
    "G1": 2 * (M_TOK * HID * 4 + HID * HID) + 4 * M_TOK * (HID // 256) + 4 * HID,
    "reduce": 4 * (M_TOK * (HID // 256) + M_TOK),
    "G2": 2 * (M_TOK * HID + 2 * FFN * HID + M_TOK * FFN) + 4 * M_TOK,
    "G3": 2 * (M_TOK * FFN + HID * FFN + 2 * M_TOK * HID),
}
CHAIN_BYTES = sum(BYTES.values())
LAUNCHES_PER_STEP = 4     # G1, reduce, G2, G3
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = ["gemm_epilogue_transformer_tcgen05_gb300/csrc/coda_gemm.cuh",
                  "gemm_epilogue_transformer_tcgen05_gb300/csrc/coda_ptx.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_G2_block_forward.md")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["coda", "reference"], default="coda")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-compare", action="store_true", help="skip the torch eager comparator and error check")
    p.add_argument("--no-others", action="store_true", help="skip the backward / QKV / fp8 chain measurements")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    p.add_argument("--no-layers", action="store_true", help="skip the full decoder-layer measurements")
    p.add_argument("--traffic-pass", action="store_true",
                   help="run only the fused chain twice, then the torch eager chain twice (a short program "
                        "for a per-kernel DRAM-bytes capture); prints one JSON line naming the launches")
    p.add_argument("--nvfp4-pass", action="store_true",
                   help="run only the NVFP4 MLP (H 4096, F 14336): quantise X, then the chain twice (a short "
                        "program for a per-kernel capture)")
    p.add_argument("--fp8-pass", action="store_true",
                   help="run only the FP8 MLP (H 4096, F 14336): the chain once for the delayed s_a, then twice "
                        "(a short program for a per-kernel capture)")
    p.add_argument("--nvfp4-bwd-pass", action="store_true",
                   help="run only the NVFP4 MLP backward (H 4096, F 14336) twice, after its weight preparation "
                        "(a short program for a per-kernel capture)")
    p.add_argument("--row-rms-pass", action="store_true",
                   help="run only the full-row RMS of a [16384, 8192] bf16 tensor, five times (a short program for "
                        "a per-kernel DRAM-bytes capture of the bandwidth-bound reduce)")
    p.add_argument("--tokens", type=int, default=M_TOK,
                   help="token count of --traffic-pass / --nvfp4-pass / --fp8-pass / --nvfp4-bwd-pass")
    p.add_argument("--compile-compare", action="store_true",
                   help="also time torch.compile of the unfused comparators (compiles on first use)")
    return p.parse_args()


# ------------------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sus=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


# a timed region shorter than this runs at the clocks of a burst, above the power-capped
# clocks of a seconds-long loop: its fractions are taken of the burst peak
SUSTAINED_REGION_S = 2.0


CAPPED_CLOCK_FRAC = 0.9   # a median SM clock below this share of the maximum: power-capped run


def tensor_peak(pk, region_s, sm_mhz=None, sm_max_mhz=None):
    """(peak TFLOP/s, kind) of the bf16 tensor roofline for a timed region of region_s seconds:
    the measured burst figure for a short region at full clocks; the sustained one (measured
    under the power cap) for a long region, or wherever the SM clocks sampled during the region
    show the cap (median below CAPPED_CLOCK_FRAC of the maximum)."""
    if sm_mhz and sm_max_mhz and sm_mhz < CAPPED_CLOCK_FRAC * sm_max_mhz:
        return pk["bf16_sus"], (f"bf16 sustained, of {pk['source']} (median SM clock {sm_mhz:.0f} of "
                                f"{sm_max_mhz:.0f} MHz during the {region_s:.3f} s region: power-capped)")
    if region_s < SUSTAINED_REGION_S:
        return pk["bf16"], f"bf16 burst, of {pk['source']} (timed region {region_s:.3f} s < {SUSTAINED_REGION_S} s)"
    return pk["bf16_sus"], f"bf16 sustained, of {pk['source']} (timed region {region_s:.3f} s)"


def lib_peak(entry, fallback):
    """Highest measured rate of a library GEMM (burst or sustained), the ceiling a kernel of the
    same dtype is held to; `fallback` where the library run failed."""
    vals = [entry.get(k) for k in ("burst_tflops", "sustained_tflops") if entry.get(k)]
    return max(vals) if vals else fallback


def kernel_hash():
    """Hash of the kernel sources' code: comments and blank space are left out, so a change
    to the comments alone keeps a recorded traffic figure valid."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            txt = f.read()
        txt = re.sub(r"/\*.*?\*/", " ", txt, flags=re.S)
        txt = re.sub(r"//[^\n]*", " ", txt)
        h.update(" ".join(txt.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes (read + write) per launch of G2 from the committed ncu summary, or None when
    the summary is missing or the kernel sources changed after the counters were taken (the
    summary records the hash of the kernel sources it was measured with)."""
    try:
        with open(TRAFFIC_FILE) as f:
            txt = f.read()
        h = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", txt).group(1)
        b = float(re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt).group(1))
        return b if h == kernel_hash() else None
    except Exception:
        return None


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


class ClockSampler:
    """nvidia-smi samples (every 100 ms) while the timed region runs."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_id):
        self.dev_id = dev_id
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev_id}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def mark(self, begin):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sel = [r for t, r in self.rows if self.t0 and self.t1 and self.t0 - 0.05 <= t <= self.t1 + 0.05]
        if len(sel) < 3:
            sel = [r for _, r in self.rows]
        sm, smax, reasons = [], [], set()
        for r in sel:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def nvsmi_id(torch):
    try:
        p = torch.cuda.get_device_properties(torch.cuda.current_device())
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0]
        return vis if vis.isdigit() else "0"


# ------------------------------------------------------------------- distributed
def max_over_ranks(ms, dist, device="cuda"):
    """The slowest rank's time (every rank gets it); `dist` None means a single rank."""
    if dist is None:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tokens_per_s(world, tokens_per_rank, ms):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms * 1e-3)

def dist_init(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and world > 1:
        print(f"warning: WORLD_SIZE={world} but --gpus={args.gpus}", file=sys.stderr)
    return world, rank, local


# --------------------------------------------------------------- the CPU oracle arm
def oracle_sample_rate(target_s):
    """Times the fp64 oracle's plain block forward on a bounded sample of token rows of
    the same workload; tokens/s = rows / seconds (forward rows are independent)."""
    import numpy as np

    import coda_synth as S
    import oracle as O
    inp = S.block_inputs(M_TOK, HID, FFN, seed=0)
    x = {k: inp[k].to(__import__("torch").float64).numpy() for k in ("O", "R", "W_o", "W_gu", "W_d", "g")}
    rows = 64
    t0 = time.perf_counter()
    O.block_forward(x["O"][:rows], x["R"][:rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], EPS)
    dt = time.perf_counter() - t0
    rows = int(min(M_TOK, max(rows, rows * target_s / max(dt, 1e-3))))
    rows = max(64, (rows // 64) * 64)
    t0 = time.perf_counter()
    O.block_forward(x["O"][:rows], x["R"][:rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], EPS)
    dt = time.perf_counter() - t0
    del np
    return rows / dt, rows, dt


def workload_config(world):
    """The `config` of both arms' JSON lines: the same workload, named by what it is."""
    return {"workload": WORKLOAD, "tokens": M_TOK, "hidden": HID, "ffn": FFN,
            "l2": f"inputs larger than L2: {CHAIN_BYTES / MB:.0f} MB compulsory traffic per step "
                  f"vs {L2_BYTES / MB:.0f} MB L2; no flush",
            "parallelism": f"replicas x{world} (no data-path collective)"}


# the reference arm's whole run (warm-up and timed steps) is kept within this many seconds
REFERENCE_BUDGET_S = 240.0


def reference_rows(rate, steps, warmup, budget_s=REFERENCE_BUDGET_S):
    """Token rows per step of the reference arm: the whole batch when every step of the run
    fits the budget at the measured rate (tokens/s), else the largest multiple of 64 that does."""
    per_step = budget_s / max(1, steps + warmup)
    if M_TOK / rate <= per_step:
        return M_TOK
    return max(64, int(rate * per_step) // 64 * 64)


def run_reference(args, world, rank):
    if rank != 0:
        return
    steps = max(1, args.steps)
    rate, _, _ = oracle_sample_rate(2.0)
    rows = reference_rows(rate, steps, args.warmup)
    times = []
    import coda_synth as S
    import oracle as O
    import torch
    inp = S.block_inputs(M_TOK, HID, FFN, seed=0)
    x = {k: inp[k].to(torch.float64).numpy() for k in ("O", "R", "W_o", "W_gu", "W_d", "g")}
    for i in range(args.warmup + steps):
        t0 = time.perf_counter()
        O.block_forward(x["O"][:rows], x["R"][:rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], EPS)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    value = rows / t
    ms_full = M_TOK / value * 1e3
    cores = cpu_cores()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms_full, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(world),
        "tflops": CHAIN_FLOP / (ms_full * 1e-3) / 1e12,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows} of {M_TOK} token rows per step (fp64 numpy oracle, plain unfused chain; "
                                   f"rows are independent)", "rows_per_step": rows},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- the GPU arm
def traffic_pass(args):
    """The fused block forward (coda_block_forward: G1, reduce, G2, G3) twice, then the same
    block as torch eager ops twice, with nothing else on the device: under a per-kernel
    counter capture the second pass of each is the warm, steady-state one."""
    import torch

    import coda_synth as S
    from gemm_epilogue_transformer_tcgen05_gb300 import coda as C

    C.lib()
    BF = torch.bfloat16
    M, H, F = args.tokens, HID, FFN
    d = S.block_inputs(M, H, F, seed=0, device="cuda")
    h, u, Y = (torch.empty((M, H), dtype=BF, device="cuda") for _ in range(3))
    r = torch.empty((M,), device="cuda")
    a = torch.empty((M, F), dtype=BF, device="cuda")
    ws = torch.empty((C.coda_workspace_size(C.WS_BLOCK_FWD, M, H, F) // 4,), device="cuda")
    for _ in range(2):
        C.coda_block_forward(d["O"], d["R"], d["W_o"], d["W_gu"], d["W_d"], EPS, h, r, a, Y, ws, g=d["g"], u=u)
    torch.cuda.synchronize()
    for _ in range(2):
        Yt = unfused_chain(torch, d, F)
    torch.cuda.synchronize()
    st, site = C.coda_get_device_status()
    if st != C.OK:
        raise RuntimeError(f"device status {st} (site {site})")
    print(json.dumps({"traffic_pass": {"tokens": M, "hidden": H, "ffn": F,
                                       "order": "fused chain x2 (G1, reduce, G2, G3), then torch eager chain x2",
                                       "normwise_diff": float((Y.float() - Yt.float()).abs().max()
                                                              / Yt.float().abs().max())}}), flush=True)


def nvfp4_pass(args):
    """The NVFP4 MLP at the LLaMA-3-8B width: weight and X quantisation (three quantiser
    launches), then the chain twice (row RMS, gate/up GEMM, down GEMM each time), nothing else
    on the device: under a per-kernel capture the second chain is the warm one."""
    import torch

    import coda_synth as S
    from gemm_epilogue_transformer_tcgen05_gb300 import coda as C

    C.lib()
    M, H, F = args.tokens, 4096, 14336
    ni = S.nvfp4_mlp_inputs(M, H, F, seed=0, device="cuda")
    sc = lambda t: float(t.abs().max()) / (6 * 448)
    X, W, Wd = C.Nvfp4.empty(M, H, sc(ni["h"])), C.Nvfp4.empty(2 * F, H, sc(ni["W_gu"])), C.Nvfp4.empty(H, F, sc(ni["W_d"]))
    C.coda_quantize_nvfp4(ni["W_gu"], W)
    C.coda_quantize_nvfp4(ni["W_d"], Wd)
    C.coda_quantize_nvfp4(ni["h"], X)
    r, amax = torch.empty((M,), device="cuda"), torch.empty((1,), device="cuda")
    a = C.Nvfp4.empty(M, F, 1.0)
    Y = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    P = torch.empty((H // 256, M), device="cuda")
    for i in range(2):
        C.coda_mlp_nvfp4(ni["h"], X, W, Wd, EPS, r, a, amax, Y, P)
        if i == 0:
            torch.cuda.synchronize()
            a.s = float(amax.item()) / (6 * 448)
    torch.cuda.synchronize()
    st, site = C.coda_get_device_status()
    if st != C.OK:
        raise RuntimeError(f"device status {st} (site {site})")
    print(json.dumps({"nvfp4_pass": {"tokens": M, "hidden": H, "ffn": F,
                                     "order": "quantise W_gu, W_d, X; chain x2 (row RMS, gate/up GEMM, down GEMM)",
                                     "Y_rms": float(Y.float().pow(2).mean().sqrt())}}), flush=True)


def fp8_pass(args):
    """The FP8 MLP at the LLaMA-3-8B width (row RMS, gate/up e4m3 GEMM + r + SwiGLU + e4m3
    requantisation + amax, down e4m3 GEMM + residual + partials): once to take the delayed s_a
    from its amax, then twice, nothing else on the device."""
    import torch

    import coda_synth as S
    from gemm_epilogue_transformer_tcgen05_gb300 import coda as C

    C.lib()
    M, H, F = args.tokens, 4096, 14336
    fi = S.fp8_mlp_inputs(M, H, F, seed=0)
    h, X, W, Wd = (fi[k].to("cuda").contiguous() for k in ("h", "Xq", "Wq", "Wdq"))
    r, amax = torch.empty((M,), device="cuda"), torch.empty((1,), device="cuda")
    aq = torch.empty((M, F), dtype=torch.uint8, device="cuda")
    Y = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    P = torch.empty((H // 256, M), device="cuda")
    s_a = 1.0
    for i in range(3):
        C.coda_mlp_fp8(h, X, W, Wd, fi["s_x"], fi["s_w"], fi["s_wd"], s_a, EPS, r, aq, amax, Y, P)
        if i == 0:
            torch.cuda.synchronize()
            s_a = float(amax.item()) / 448.0
    torch.cuda.synchronize()
    st, site = C.coda_get_device_status()
    if st != C.OK:
        raise RuntimeError(f"device status {st} (site {site})")
    print(json.dumps({"fp8_pass": {"tokens": M, "hidden": H, "ffn": F,
                                   "order": "chain x3 (row RMS, gate/up GEMM, down GEMM); the first sets s_a",
                                   "Y_rms": float(Y.float().pow(2).mean().sqrt())}}), flush=True)


def row_rms_pass(args):
    """The full-row RMS (coda_row_rms) of a [16384, 8192] bf16 tensor (268 MB read, 64 KB
    written) five times back to back, with nothing else on the device."""
    import torch

    from gemm_epilogue_transformer_tcgen05_gb300 import coda as C

    C.lib()
    X = torch.randn((M_TOK, 8192), device="cuda", generator=torch.Generator(device="cuda").manual_seed(5))
    X = X.to(torch.bfloat16)
    r = torch.empty((M_TOK,), device="cuda")
    for _ in range(5):
        C.coda_row_rms(X, EPS, r)
    torch.cuda.synchronize()
    print(json.dumps({"row_rms_pass": {"rows": M_TOK, "cols": 8192, "launches": 5,
                                       "bytes_per_launch": 2 * M_TOK * 8192 + 4 * M_TOK,
                                       "r_mean": float(r.mean())}}), flush=True)


def run_coda(args, world, rank, local):
    import numpy as np
    import torch

    import coda_synth as S
    from gemm_epilogue_transformer_tcgen05_gb300 import coda as C

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    C.lib()
    BF = torch.bfloat16
    M, H, F = M_TOK, HID, FFN
    inp = S.block_inputs(M, H, F, seed=rank)
    d = {k: inp[k].to("cuda").contiguous() for k in ("O", "R", "W_o", "W_gu", "W_d", "g")}
    h = torch.empty((M, H), dtype=BF, device="cuda")
    u = torch.empty((M, H), dtype=BF, device="cuda")
    r = torch.empty((M,), device="cuda")
    a = torch.empty((M, F), dtype=BF, device="cuda")
    Y = torch.empty((M, H), dtype=BF, device="cuda")
    P = torch.empty((H // 256, M), device="cuda")
    stream = torch.cuda.current_stream()

    def step(ev=None):
        # the chain as its four C-ABI launches (coda_block_forward with the gain broadcast
        # issues exactly these, in this order); events bracket the dominant GEMM
        C.coda_gemm_epilogue(d["O"], d["W_o"], [C.OP_ADD_SIDE, C.OP_ROW_SUMSQ_PARTIAL, C.OP_STORE_COL_SCALED], h,
                             residual=d["R"], row_partials=P, col_scale=d["g"], store_aux=u, stream=stream)
        C.coda_rms_partial_reduce(P, M, H, EPS, r, stream=stream)
        if ev is not None:
            ev[0].record(stream)
        C.coda_gemm_epilogue(u, d["W_gu"], [C.OP_ROW_SCALE, C.OP_SWIGLU], a, row_scale=r, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        C.coda_gemm_epilogue(a, d["W_d"], [C.OP_ADD_SIDE], Y, residual=h, stream=stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    st, site = C.coda_get_device_status(stream)
    if st != C.OK:
        raise RuntimeError(f"device status {st} (site {site}) during warm-up")

    sampler = ClockSampler(nvsmi_id(torch)) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    if sampler:
        sampler.mark(True)
    t_start.record(stream)
    for i in range(args.steps):
        step()
    t_end.record(stream)
    barrier()
    if sampler:
        sampler.mark(False)
    ms = t_start.elapsed_time(t_end)
    # G2's launches are timed in the next region, of the same steps: an event recorded between
    # two launches separates them (the next launch no longer overlaps the previous kernel's
    # tail), which cost the step 1.2% when the events sat in the region above
    for i in range(args.steps):
        step(evs[i])
    torch.cuda.synchronize()
    g2_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs)
    st, site = C.coda_get_device_status(stream)
    if st != C.OK:
        raise RuntimeError(f"device status {st} (site {site}) in the timed region")
    ms = max_over_ranks(ms, dist)
    if sampler:
        time.sleep(0.15)
        sampler.stop()
    ms_step = ms / args.steps
    value = aggregate_tokens_per_s(world, M, ms_step)

    # ---- end to end through the public chain call, host buffers (pinned) both ways.
    # Each step copies its inputs O, R from pinned host memory and its result Y back; the
    # copies of neighbouring steps run on two copy streams under the compute of this step
    # (two device slots for O, R, Y), the way a stream of batches would be served.
    e2e = None
    if not args.no_e2e:
        O_h = inp["O"].pin_memory()
        R_h = inp["R"].pin_memory()
        Y_h = [torch.empty((M, H), dtype=BF).pin_memory() for _ in range(2)]
        ws = torch.empty((C.coda_workspace_size(C.WS_BLOCK_FWD, M, H, F) // 4,), device="cuda")
        O_d = [torch.empty_like(d["O"]) for _ in range(2)]
        R_d = [torch.empty_like(d["R"]) for _ in range(2)]
        Y_d = [torch.empty_like(Y) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        for e_ in ev_done + ev_out:
            e_.record(stream)

        def e2e_step(i):
            k = i % 2
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_done[k])            # the step that used this slot has finished
                O_d[k].copy_(O_h, non_blocking=True)
                R_d[k].copy_(R_h, non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            stream.wait_event(ev_out[k])              # Y_d[k] of step i-2 has been read back
            C.coda_block_forward(O_d[k], R_d[k], d["W_o"], d["W_gu"], d["W_d"], EPS, h, r, a, Y_d[k], ws, g=d["g"],
                                 u=u, stream=stream)
            ev_done[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[k])
                Y_h[k].copy_(Y_d[k], non_blocking=True)
                ev_out[k].record(s_out)

        # at least 50 steps, so that the one copy of each kind that nothing overlaps (the first
        # step's inputs, the last step's result) weighs little against the steady state
        n_e2e = max(4, min(max(args.steps, 50), 100))
        for i in range(4):
            e2e_step(i)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n_e2e):
            e2e_step(i)
        s_out.synchronize()
        stream.wait_stream(s_out)
        e1.record(stream)
        barrier()
        ems = max_over_ranks(e0.elapsed_time(e1) / n_e2e, dist)
        e2e = {"value": aggregate_tokens_per_s(world, M, ems), "unit": "tokens/s", "ms_per_step": ems, "steps": n_e2e,
               "h2d_bytes_per_step": O_h.numel() * 2 + R_h.numel() * 2, "d2h_bytes_per_step": Y_h[0].numel() * 2,
               "pipelined": "copies of neighbouring steps overlap this step's compute (2 slots, 2 copy streams)"}

    # ---- the same chain captured once in a CUDA graph and replayed (host launch work gone)
    graph_ms = None
    if rank == 0:
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        with torch.cuda.stream(gs):
            step_on = lambda: (C.coda_gemm_epilogue(d["O"], d["W_o"], [C.OP_ADD_SIDE, C.OP_ROW_SUMSQ_PARTIAL,
                                                                        C.OP_STORE_COL_SCALED], h, residual=d["R"],
                                                    row_partials=P, col_scale=d["g"], store_aux=u, stream=gs),
                               C.coda_rms_partial_reduce(P, M, H, EPS, r, stream=gs),
                               C.coda_gemm_epilogue(u, d["W_gu"], [C.OP_ROW_SCALE, C.OP_SWIGLU], a, row_scale=r,
                                                    stream=gs),
                               C.coda_gemm_epilogue(a, d["W_d"], [C.OP_ADD_SIDE], Y, residual=h, stream=gs))
            step_on()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for _ in range(10):
                step_on()
        n_rep = max(3, min(args.steps // 10, 50))
        with torch.cuda.stream(gs):           # replay() launches on the current stream
            for _ in range(2):
                graph.replay()
            torch.cuda.synchronize()
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(gs)
            for _ in range(n_rep):
                graph.replay()
            g1.record(gs)
        torch.cuda.synchronize()
        graph_ms = g0.elapsed_time(g1) / (10 * n_rep)
        del graph

    # ---- the same chain with L2 cold before every step (the timed line above is warm:
    # back to back, as in training)
    cold_ms = cold_l2(torch, step, stream, max(5, min(args.steps, 50))) if rank == 0 else None

    # ---- per-kernel device times: a separate short run with events between the four launches
    # (kept out of the timed region, where extra events could hold back the launch overlap)
    per_kernel = None
    if rank == 0:
        n_k = max(5, min(args.steps, 100))
        kev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(n_k)]
        calls = [lambda: C.coda_gemm_epilogue(d["O"], d["W_o"], [C.OP_ADD_SIDE, C.OP_ROW_SUMSQ_PARTIAL,
                                                                 C.OP_STORE_COL_SCALED], h, residual=d["R"],
                                              row_partials=P, col_scale=d["g"], store_aux=u, stream=stream),
                 lambda: C.coda_rms_partial_reduce(P, M, H, EPS, r, stream=stream),
                 lambda: C.coda_gemm_epilogue(u, d["W_gu"], [C.OP_ROW_SCALE, C.OP_SWIGLU], a, row_scale=r,
                                              stream=stream),
                 lambda: C.coda_gemm_epilogue(a, d["W_d"], [C.OP_ADD_SIDE], Y, residual=h, stream=stream)]
        for i in range(3 + n_k):
            for j, call in enumerate(calls):
                if i >= 3:
                    kev[i - 3][j].record(stream)
                call()
            if i >= 3:
                kev[i - 3][4].record(stream)
        torch.cuda.synchronize()
        pk_ = peaks()
        per_kernel = {}
        for j, name in enumerate(("G1", "reduce", "G2", "G3")):
            k_ms = statistics.mean(e[j].elapsed_time(e[j + 1]) for e in kev)
            entry = {"ms": k_ms, "algorithmic_bytes": BYTES[name]}
            if name in FLOP:
                entry.update(tflops=FLOP[name] / (k_ms * 1e-3) / 1e12,
                             frac_of_burst=FLOP[name] / (k_ms * 1e-3) / 1e12 / pk_["bf16"],
                             frac_of_sustained=FLOP[name] / (k_ms * 1e-3) / 1e12 / pk_["bf16_sus"])
            else:
                entry.update(gbs=BYTES[name] / (k_ms * 1e-3) / 1e9, bound="launch latency")
            per_kernel[name] = entry

    # ---- the other chains of the hot path, device-timed the same way (fewer steps)
    others = None
    if not args.no_others and rank == 0:
        others = other_workloads(torch, C, S, args, stream)
        if not args.no_layers:
            others.update(layer_workloads(torch, C, S, args, stream))

    # ---- comparator: the same chain unfused in torch eager (cuBLAS GEMMs), and errors
    compare = None
    if not args.no_compare and rank == 0:
        compare = unfused_compare(torch, d, {"h": h, "r": r, "a": a, "Y": Y}, inp, stream, args)
        compare["backward"] = backward_compare(torch, C, S, stream)

    # ---- the library e4m3 / NVFP4 peaks, once nothing is left to time (their sustained loops
    # leave the GPU at its power cap for a while)
    if others is not None:
        finish_lib_peaks(torch, others, peaks())

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    pk = peaks()
    g2_tflops = FLOP["G2"] / (g2_ms * 1e-3) / 1e12
    traffic = recorded_traffic()
    clocks = sampler.summary() if sampler else None
    peak, peak_kind = tensor_peak(pk, ms / 1e3, clocks.get("sm_mhz") if clocks else None,
                                  clocks.get("sm_max_mhz") if clocks else None)
    chain_roof = lambda tf: max(CHAIN_FLOP / (tf * 1e12), CHAIN_BYTES / (pk["hbm"] * 1e9)) * 1e3
    chain_roof_ms = chain_roof(peak)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(world),
        "tflops": CHAIN_FLOP / (ms_step * 1e-3) / 1e12,
        "chain_roofline": {"ms": chain_roof_ms, "frac": chain_roof_ms / ms_step, "peak_tflops": peak,
                           "peak_kind": peak_kind, "frac_of_burst": chain_roof(pk["bf16"]) / ms_step,
                           "frac_of_sustained": chain_roof(pk["bf16_sus"]) / ms_step},
        "roofline": {"kernel": "G2 gate/up GEMM + deferred r + SwiGLU (gemm_epilogue_kernel, EPI_SWIGLU)",
                     "bound": "tensor", "achieved": g2_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": g2_tflops / peak, "traffic": traffic, "peak_kind": peak_kind,
                     "frac_of_burst": g2_tflops / pk["bf16"], "frac_of_sustained": g2_tflops / pk["bf16_sus"],
                     "sm_mhz_median": clocks["sm_mhz"] if clocks else None, "ms_per_launch": g2_ms,
                     "launch_timing": "CUDA events around each G2 launch in a second region of the same "
                                      f"{args.steps} steps, right after the timed one (events between the "
                                      "launches cost the step about 1.2%, so the timed region has none)",
                     "algorithmic_bytes": BYTES["G2"], "flop_per_launch": FLOP["G2"]},
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": clocks,
    }
    if e2e:
        line["e2e"] = e2e
    if cold_ms:
        line["cold_l2"] = {"ms_per_step": cold_ms, "tokens_per_s": M / (cold_ms * 1e-3),
                           "chain_roofline_frac": chain_roof_ms / cold_ms,
                           "note": "1 GiB scratch write before every step, outside the timed events; median"}
    if graph_ms:
        line["cuda_graph"] = {"ms_per_step": graph_ms, "tokens_per_s": M / (graph_ms * 1e-3),
                              "note": "10 steps captured once in a CUDA graph, replayed"}
    if per_kernel:
        line["per_kernel"] = dict(per_kernel, note="events between the four launches in a separate run of the "
                                                   "same chain; TFLOP/s against the measured bf16 peaks")
    if others:
        line["other_workloads"] = others
    if compare:
        line["compare"] = compare
    if not args.no_cpu_baseline:
        rate, rows, dt = oracle_sample_rate(args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": f"{rows} of {M} token rows, {dt:.1f} s (fp64 numpy oracle, plain "
                                          f"unfused chain; rows are independent)"}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    del np


def _time(torch, fn, stream, steps, warmup=3, settle_s=0.1):
    # A short idle first: the timed regions are short and held to the burst peaks, and the
    # power limiter would otherwise carry the previous (seconds-long, power-capped) workload's
    # state into this one.  The warm-up steps still run before the timing starts.
    torch.cuda.synchronize()
    time.sleep(settle_s)
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def cold_l2(torch, fn, stream, n, warmup=3):
    """Median device time of fn with L2 cold: a 1 GiB scratch write (eight times L2) runs
    before every repetition, outside the events that time fn."""
    scratch = torch.empty((1 << 30,), dtype=torch.uint8, device="cuda")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(warmup + n):
        scratch.zero_()
        if i >= warmup:
            evs[i - warmup][0].record(stream)
        fn()
        if i >= warmup:
            evs[i - warmup][1].record(stream)
    torch.cuda.synchronize()
    del scratch
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)


def fp8_peak(torch, seconds=2.0):
    """Dense e4m3 GEMM throughput of the vendor library (torch._scaled_mm, per-tensor scales,
    bf16 out) at 8192^3, measured the way the bf16 peaks were: the best of 10 single launches
    (burst) and back to back for a few seconds (sustained).  A roofline denominator only."""
    n = 8192
    gen = torch.Generator(device="cuda").manual_seed(3)
    a = torch.randn((n, n), device="cuda", generator=gen).to(torch.float8_e4m3fn)
    b = torch.randn((n, n), device="cuda", generator=gen).to(torch.float8_e4m3fn)
    one = torch.ones((), device="cuda")

    def f():
        return torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

    for _ in range(5):
        f()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(10):
        e0.record()
        f()
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    flop = 2.0 * n ** 3
    reps = max(10, int(seconds * 1e3 / best))
    e0.record()
    for _ in range(reps):
        f()
    e1.record()
    torch.cuda.synchronize()
    sus = flop * reps / (e0.elapsed_time(e1) * 1e-3) / 1e12
    return {"burst_tflops": flop / (best * 1e-3) / 1e12, "sustained_tflops": sus, "reps_sustained": reps,
            "how": "torch._scaled_mm e4m3 x e4m3 -> bf16, 8192^3, per-tensor scales: best of 10 (burst); "
                   f"{reps} back to back (sustained)"}


def fp4_peak(torch, fp8_sustained, seconds=2.0):
    """Dense NVFP4 GEMM throughput of the vendor library (torch._scaled_mm on e2m1 operands
    with e4m3 block scales, bf16 out) at 8192^3, burst and sustained as for fp8.  Where this
    torch cannot run it, the nominal ratio (13.5 / 4.5 PFLOP/s = 3x the measured e4m3 peak)
    stands in, and the entry says so."""
    n = 8192
    try:
        gen = torch.Generator(device="cuda").manual_seed(4)
        a = torch.randint(0, 256, (n, n // 2), dtype=torch.uint8, device="cuda", generator=gen)
        b = torch.randint(0, 256, (n, n // 2), dtype=torch.uint8, device="cuda", generator=gen)
        a, b = a.view(torch.float4_e2m1fn_x2), b.view(torch.float4_e2m1fn_x2)
        sa = torch.full((n, n // 16), 0x38, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
        sb = torch.full((n, n // 16), 0x38, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)

        def f():
            return torch._scaled_mm(a, b.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16)

        for _ in range(5):
            f()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        best = float("inf")
        for _ in range(10):
            e0.record()
            f()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        flop = 2.0 * n ** 3
        reps = max(10, int(seconds * 1e3 / best))
        e0.record()
        for _ in range(reps):
            f()
        e1.record()
        torch.cuda.synchronize()
        sus = flop * reps / (e0.elapsed_time(e1) * 1e-3) / 1e12
        return {"burst_tflops": flop / (best * 1e-3) / 1e12, "sustained_tflops": sus, "reps_sustained": reps,
                "how": "torch._scaled_mm NVFP4 (e2m1, e4m3 block scales) -> bf16, 8192^3: best of 10 (burst); "
                       f"{reps} back to back (sustained)"}
    except Exception as ex:
        return {"sustained_tflops_nominal_ratio": 3.0 * fp8_sustained,
                "error": f"{type(ex).__name__}: {ex}"[:200],
                "how": "library NVFP4 GEMM unavailable here: 3x the measured e4m3 sustained peak (nominal ratio)"}


def finish_lib_peaks(torch, out, pk):
    """The library e4m3 and NVFP4 GEMM rates (the denominators of those chains' rooflines),
    measured once every workload has been timed, and the rooflines that wait for them."""
    deferred = out.pop("_deferred", [])
    try:
        out["fp8_peak"] = fp8_peak(torch)
    except Exception as ex:                       # a torch without e4m3 GEMMs: keep the nominal ratio
        out["fp8_peak"] = {"error": f"{type(ex).__name__}: {ex}"[:200]}
    if "sustained_tflops" in out["fp8_peak"]:
        peak8 = lib_peak(out["fp8_peak"], 2 * pk["bf16"])
        note8 = "e4m3 library GEMM measured after every workload, the higher of burst and sustained"
    else:
        peak8 = 2 * pk["bf16"]
        note8 = "fp8 peak taken as 2x the measured bf16 burst peak (nominal ratio)"
    out["fp4_peak"] = fp4_peak(torch, peak8)
    peak4 = lib_peak(out["fp4_peak"], out["fp4_peak"].get("sustained_tflops_nominal_ratio"))
    for v in out.get("mlp_nvfp4_N4", {}).get("per_gemm", {}).values():
        v["frac_of_peak"] = v["tflops"] / peak4
    for kind, entry, fl, by in deferred:
        peak = peak8 if kind == "fp8" else peak4
        roof = max(fl / (peak * 1e12), by / (pk["hbm"] * 1e9)) * 1e3
        entry.update({"roofline_ms": roof, "roofline_frac": roof / entry["ms"], "peak_tflops": peak})
        if kind == "fp8":
            entry["peak_note"] = note8


def other_workloads(torch, C, S, args, stream):
    """Device time of the other chains at their full sizes (16384 tokens): the block backward
    (C2), QKV + RoPE (C3), the fp8 and NVFP4 MLPs (C4, N4), the hidden-size sweep (N3) and the
    LM head with cross-entropy (N1), with TFLOP/s and the fraction of their rooflines.  Each is
    timed over a short region (well under a second), so the tensor peaks are the burst ones:
    the measured bf16 burst figure, and the higher of the burst and sustained rates of the
    library's e4m3 and NVFP4 GEMMs measured in the same run."""
    BF = torch.bfloat16
    pk = peaks()
    steps = max(5, min(args.steps, 50))
    out = {}
    # The e4m3 and NVFP4 rooflines are held to the library GEMMs' measured rates, taken at the
    # end of this section: their seconds-long sustained loops leave the GPU at its power cap for
    # a while, which would slow whatever were timed right after them.  Until then each entry
    # keeps its FLOP and byte counts here.
    deferred = []   # (dtype, entry, flop, bytes)
    # the light row reduce in its full-row form, where bandwidth can be seen: r of a
    # [16384, 8192] bf16 tensor (268 MB read), back to back
    Xr = torch.randn((M_TOK, 8192), device="cuda", generator=torch.Generator(device="cuda").manual_seed(5)).to(BF)
    rr = torch.empty((M_TOK,), device="cuda")
    ms = _time(torch, lambda: C.coda_row_rms(Xr, EPS, rr, stream=stream), stream, 50)
    byt = 2 * M_TOK * 8192 + 4 * M_TOK
    out["row_rms_full_row_M16384_N8192"] = {"ms": ms, "gbs": byt / (ms * 1e-3) / 1e9, "bytes": byt,
                                             "frac_of_hbm": byt / (ms * 1e-3) / 1e9 / pk["hbm"],
                                             "frac_of_nominal_7900": byt / (ms * 1e-3) / 1e9 / 7900.0,
                                             "peak_kind": f"HBM copy, {pk['source']}"}
    del Xr, rr
    # C2: block backward (after a training-mode forward that saves Z)
    M, H, F = M_TOK, HID, FFN
    inp = S.block_inputs(M, H, F, seed=0, with_grad=True)
    d = {k: inp[k].to("cuda").contiguous() for k in ("O", "R", "W_o", "W_gu", "W_d", "g", "dY")}
    h = torch.empty((M, H), dtype=BF, device="cuda")
    u = torch.empty((M, H), dtype=BF, device="cuda")
    r = torch.empty((M,), device="cuda")
    a = torch.empty((M, F), dtype=BF, device="cuda")
    Y = torch.empty((M, H), dtype=BF, device="cuda")
    Z = torch.empty((M, 2 * F), dtype=BF, device="cuda")
    wsf = torch.empty((C.coda_workspace_size(C.WS_BLOCK_FWD, M, H, F) // 4,), device="cuda")
    C.coda_block_forward(d["O"], d["R"], d["W_o"], d["W_gu"], d["W_d"], EPS, h, r, a, Y, wsf, Z=Z, g=d["g"], u=u,
                         stream=stream)
    e = torch.empty((M, 2 * F), dtype=BF, device="cuda")
    dh = torch.empty((M, H), dtype=BF, device="cuda")
    dO = torch.empty((M, H), dtype=BF, device="cuda")
    dW_o = torch.empty((H, H), device="cuda")
    dW_gu = torch.empty((2 * F, H), device="cuda")
    dW_d = torch.empty((H, F), device="cuda")
    dg = torch.empty((H,), device="cuda")
    c = torch.empty((M,), device="cuda")
    wsb = torch.empty((C.coda_workspace_size(C.WS_BLOCK_BWD, M, H, F) // 4,), device="cuda")
    bwd = lambda: C.coda_block_backward(d["O"], d["W_o"], d["W_gu"], d["W_d"], d["g"], h, r, Z, a, d["dY"], e, dh,
                                        dO, dW_o, dW_gu, dW_d, dg, c, wsb, stream=stream)
    ms = _time(torch, bwd, stream, steps)
    flop = 2 * (2 * M * F * H + 2 * M * 2 * F * H + 2 * M * H * H)
    byt = 2 * (M * H * 3 + H * F + 2 * M * F * 2) + 4 * H * F + 2 * (2 * M * F + 2 * F * H + 3 * M * H) + \
        4 * 2 * F * H + 2 * (M * H * 3 + H * H) + 4 * H * H
    roof = max(flop / (pk["bf16"] * 1e12), byt / (pk["hbm"] * 1e9)) * 1e3
    out["block_backward_C2"] = {"ms": ms, "tflops": flop / (ms * 1e-3) / 1e12, "roofline_ms": roof,
                                "roofline_frac": roof / ms, "tokens_per_s": M / (ms * 1e-3), "launches": 8}
    fwd_train = lambda: C.coda_block_forward(d["O"], d["R"], d["W_o"], d["W_gu"], d["W_d"], EPS, h, r, a, Y, wsf,
                                             Z=Z, g=d["g"], u=u, stream=stream)
    ms_f = _time(torch, fwd_train, stream, steps)
    out["block_forward_train_mode"] = {"ms": ms_f, "tokens_per_s": M / (ms_f * 1e-3),
                                       "note": "G1 (+ u = h g), reduce, G2 saving Z = [G|U], G3"}
    # the other way to apply the RMSNorm gain: folded into W_gu once per weight update, so that
    # G1 stores only h and the gate/up GEMM reads h
    Wf = torch.empty_like(d["W_gu"])
    fold = lambda: C.coda_fold_gain(d["W_gu"], d["g"], Wf, stream=stream)
    fold()
    fwd_fold = lambda: C.coda_block_forward(d["O"], d["R"], d["W_o"], Wf, d["W_d"], EPS, h, r, a, Y, wsf,
                                            stream=stream)
    fwd_bc = lambda: C.coda_block_forward(d["O"], d["R"], d["W_o"], d["W_gu"], d["W_d"], EPS, h, r, a, Y, wsf,
                                          g=d["g"], u=u, stream=stream)
    ms_bc = _time(torch, fwd_bc, stream, steps)        # the headline chain, timed again beside it
    ms_ff = _time(torch, fwd_fold, stream, steps)
    ms_fold = _time(torch, fold, stream, steps)
    out["block_forward_folded_gain"] = {"ms": ms_ff, "tokens_per_s": M / (ms_ff * 1e-3), "fold_ms": ms_fold,
                                        "plus_fold_ms": ms_ff + ms_fold, "broadcast_ms_same_section": ms_bc,
                                        "note": "C1 with W_gu' = W_gu diag(g) folded beforehand (timed on its own): "
                                                "G1 stores h only, G2 reads h; the headline broadcasts g instead "
                                                "(broadcast_ms_same_section: the headline chain timed just before, "
                                                "under the same clocks)"}
    del Wf
    del d, h, u, r, a, Y, Z, e, dh, dO, dW_o, dW_gu, dW_d, dg, c, wsb, wsf
    torch.cuda.empty_cache()
    # C3: QKV projection + deferred r + RoPE (r from a full-row pass over h)
    N, hd, seq = 3072, 64, 1024
    qi = S.qkv_inputs(M, H, N, seed=0)
    hq, Wq_, gq = (qi[k].to("cuda").contiguous() for k in ("h", "W_qkv", "g"))
    Wqf = torch.empty_like(Wq_)
    cos = torch.empty((seq, hd // 2), device="cuda")
    sin = torch.empty_like(cos)
    C.coda_rope_table(seq, hd, 500000.0, cos, sin, stream=stream)
    rq = torch.empty((M,), device="cuda")
    oq = torch.empty((M, N), dtype=BF, device="cuda")

    fold = lambda: C.coda_fold_gain(Wq_, gq, Wqf, stream=stream)   # the gain onto W_qkv
    fold()                                            # once per weight update
    qkv = lambda: C.coda_qkv_rope(hq, Wqf, EPS, seq, hd, 2560, cos, sin, rq, oq, stream=stream)
    ms = _time(torch, qkv, stream, steps)
    ms_fold = _time(torch, fold, stream, steps)
    flop = 2 * M * N * H
    byt = 2 * (M * H * 2 + N * H + M * N) + 4 * M
    roof = max(flop / (pk["bf16"] * 1e12), byt / (pk["hbm"] * 1e9)) * 1e3
    out["qkv_rope_C3"] = {"ms": ms, "tflops": flop / (ms * 1e-3) / 1e12, "roofline_ms": roof,
                          "roofline_frac": roof / ms, "tokens_per_s": M / (ms * 1e-3), "launches": 2,
                          "fold_ms": ms_fold, "plus_fold_ms": ms + ms_fold,
                          "note": "row RMS of h (one pass) + QKV GEMM with r and RoPE epilogue; the gain fold "
                                  "onto W_qkv runs once per weight update and is timed on its own (fold_ms)"}
    # N2: its backward (RoPE transposed + attention-input RMSNorm backward + dW)
    dq = torch.randn((M, N), generator=torch.Generator(device="cuda").manual_seed(7), device="cuda").to(BF)
    eq = torch.empty((M, N), dtype=BF, device="cuda")
    dhq = torch.empty((M, H), dtype=BF, device="cuda")
    dWq = torch.empty((N, H), device="cuda")
    dgq, cq = torch.empty((H,), device="cuda"), torch.empty((M,), device="cuda")
    wsq = torch.empty((((M + 31) // 32) * H,), device="cuda")
    qb = lambda: C.coda_qkv_rope_backward(hq, gq, Wq_, rq, oq, dq, seq, hd, 2560, cos, sin, eq, dhq, dWq, dgq, cq,
                                          wsq, stream=stream)
    ms = _time(torch, qb, stream, steps)
    flop = 2 * (2 * M * N * H)
    byt = 2 * (M * N * 3 + M * N * 2 + N * H * 2 + M * H * 3) + 4 * N * H
    roof = max(flop / (pk["bf16"] * 1e12), byt / (pk["hbm"] * 1e9)) * 1e3
    # per kernel: the two GEMMs at the tensor peak plus the RoPE-backward pass (dout and out read,
    # e written) at the HBM peak
    roof_k = (flop / (pk["bf16"] * 1e12) + (2 * 3 * M * N + 4 * 2 * M) / (pk["hbm"] * 1e9)) * 1e3
    out["qkv_rope_backward_N2"] = {"ms": ms, "tflops": flop / (ms * 1e-3) / 1e12, "roofline_ms": roof,
                                   "roofline_frac": roof / ms, "kernel_sum_roofline_ms": roof_k,
                                   "kernel_sum_roofline_frac": roof_k / ms,
                                   "tokens_per_s": M / (ms * 1e-3), "launches": 4,
                                   "note": "RoPE backward + row scale pass, dh GEMM + RMSNorm-bwd epilogue, dg "
                                           "column reduce, dW GEMM"}
    del hq, Wq_, gq, Wqf, oq, dq, eq, dhq, dWq, wsq
    torch.cuda.empty_cache()
    # C4: fp8 MLP
    H8, F8 = 4096, 14336
    fi = S.fp8_mlp_inputs(M, H8, F8, seed=0)
    h8, X8, W8, Wd8 = (fi[k].to("cuda").contiguous() for k in ("h", "Xq", "Wq", "Wdq"))
    r8 = torch.empty((M,), device="cuda")
    aq = torch.empty((M, F8), dtype=torch.uint8, device="cuda")
    am = torch.empty((1,), device="cuda")
    Y8 = torch.empty((M, H8), dtype=BF, device="cuda")
    P8 = torch.empty((H8 // 256, M), device="cuda")
    s_a = 1.0
    run8 = lambda: C.coda_mlp_fp8(h8, X8, W8, Wd8, fi["s_x"], fi["s_w"], fi["s_wd"], s_a, EPS, r8, aq, am, Y8, P8,
                                  stream=stream)
    run8()
    torch.cuda.synchronize()
    s_a = float(am.item()) / 448.0                     # delayed scaling from the previous pass
    ms = _time(torch, run8, stream, steps)
    flop = 2 * M * 2 * F8 * H8 + 2 * M * H8 * F8
    byt = (M * H8 + 2 * F8 * H8 + M * F8) + (M * F8 + H8 * F8) + 2 * (M * H8 * 3) + 4 * M * (H8 // 256 + 1)
    out["mlp_fp8_C4"] = {"ms": ms, "tflops": flop / (ms * 1e-3) / 1e12, "tokens_per_s": M / (ms * 1e-3),
                         "launches": 3, "frac_of_2x_bf16": flop / (ms * 1e-3) / 1e12 / (2 * pk["bf16"])}
    deferred.append(("fp8", out["mlp_fp8_C4"], flop, byt))
    # N4: its backward on e4m3 operands, after a training-mode forward that saves Z = [G | U]
    Z8 = torch.empty((M, 2 * F8), dtype=BF, device="cuda")
    fwd8 = lambda: C.coda_mlp_fp8(h8, X8, W8, Wd8, fi["s_x"], fi["s_w"], fi["s_wd"], s_a, EPS, r8, aq, am, Y8, P8,
                                  Z=Z8, stream=stream)
    ms_fz = _time(torch, fwd8, stream, steps)
    dY8 = torch.randn((M, H8), generator=torch.Generator(device="cuda").manual_seed(9), device="cuda").to(BF)
    s_dy = float(dY8.abs().max()) / 448.0
    U8 = torch.uint8
    dYq8 = torch.empty((M, H8), dtype=U8, device="cuda")
    eq8 = torch.empty((M, 2 * F8), dtype=U8, device="cuda")
    am_dy, am_e = torch.empty((1,), device="cuda"), torch.empty((1,), device="cuda")
    c8 = torch.empty((M,), device="cuda")
    dh8 = torch.empty((M, H8), dtype=BF, device="cuda")
    dWd8, dW8 = torch.empty((H8, F8), device="cuda"), torch.empty((2 * F8, H8), device="cuda")
    ws8 = torch.empty((C.coda_workspace_size(C.WS_MLP_FP8_BWD, M, H8, F8) // 4,), device="cuda")
    s_e = [1.0]
    bwd8 = lambda: C.coda_mlp_fp8_backward(h8, X8, W8, Wd8, Z8, aq, r8, dY8, fi["s_x"], fi["s_w"], fi["s_wd"], s_a,
                                           s_dy, s_e[0], dYq8, am_dy, eq8, am_e, c8, dh8, dWd8, dW8, ws8,
                                           stream=stream)
    bwd8()
    torch.cuda.synchronize()
    s_e[0] = float(am_e.item()) / 448.0               # delayed scaling from the previous pass
    ms = _time(torch, bwd8, stream, steps)
    flop = 12 * M * H8 * F8                            # dA, dW_d: 2MHF each; dh, dW: 4MHF each
    byt = 3 * M * H8 + (M * H8 + H8 * F8 + 4 * M * F8 + 2 * M * F8) + (M * H8 + M * F8 + 4 * H8 * F8) + \
        (2 * M * F8 + 2 * F8 * H8 + 6 * M * H8) + (2 * M * F8 + M * H8 + 8 * F8 * H8)
    out["mlp_fp8_backward_N4"] = {"ms": ms, "tflops": flop / (ms * 1e-3) / 1e12, "tokens_per_s": M / (ms * 1e-3),
                                  "launches": 6, "train_forward_ms": ms_fz,
                                  "note": "quantise dY, dA GEMM + SwiGLU-bwd (e4m3 e), row reduce, dW_d, "
                                          "dh GEMM + RMSNorm-bwd combine, dW; e4m3 operands, MN-major where "
                                          "transposed"}
    deferred.append(("fp8", out["mlp_fp8_backward_N4"], flop, byt))
    del h8, X8, W8, Wd8, aq, Y8, P8, Z8, dY8, dYq8, eq8, dh8, dWd8, dW8, ws8
    torch.cuda.empty_cache()
    # N4: the same MLP with NVFP4 operands (e2m1 codes, e4m3 block scales per 16 K elements)
    ni = S.nvfp4_mlp_inputs(M, H8, F8, seed=0, device="cuda")
    h4 = ni["h"]
    amax4 = lambda t: float(t.abs().max()) / (6 * 448)
    X4 = C.Nvfp4.empty(M, H8, amax4(h4))
    W4 = C.Nvfp4.empty(2 * F8, H8, amax4(ni["W_gu"]))
    Wd4 = C.Nvfp4.empty(H8, F8, amax4(ni["W_d"]))
    C.coda_quantize_nvfp4(ni["W_gu"], W4, stream=stream)   # weight preparation
    C.coda_quantize_nvfp4(ni["W_d"], Wd4, stream=stream)
    quant_x = lambda: C.coda_quantize_nvfp4(h4, X4, stream=stream)
    quant_x()
    del ni
    r4 = torch.empty((M,), device="cuda")
    am4 = torch.empty((1,), device="cuda")
    Y4 = torch.empty((M, H8), dtype=BF, device="cuda")
    P4 = torch.empty((H8 // 256, M), device="cuda")
    a4 = C.Nvfp4.empty(M, F8, 1.0)
    run4 = lambda: C.coda_mlp_nvfp4(h4, X4, W4, Wd4, EPS, r4, a4, am4, Y4, P4, stream=stream)
    run4()
    torch.cuda.synchronize()
    a4.s = float(am4.item()) / (6 * 448)              # delayed scaling from the previous pass
    ms = _time(torch, run4, stream, steps)
    flop = 2 * M * 2 * F8 * H8 + 2 * M * H8 * F8
    sfb = lambda R, K: (R * K) // 16                    # block-scale bytes
    byt = (M * H8 // 2 + sfb(M, H8) + F8 * H8 + sfb(2 * F8, H8) + M * F8 // 2 + sfb(M, F8)) + \
        (M * F8 // 2 + sfb(M, F8) + H8 * F8 // 2 + sfb(H8, F8)) + 2 * (M * H8 * 3) + 4 * M * (H8 // 256 + 1)
    ms_q = _time(torch, quant_x, stream, steps)
    byt_q = 2 * M * H8 + M * H8 // 2 + sfb(M, H8)
    # the chain's two GEMMs launched on their own through the public GEMM call, with its arguments
    gate_up = lambda: C.coda_gemm_epilogue(X4, W4, [C.OP_TENSOR_SCALE, C.OP_ROW_SCALE, C.OP_SWIGLU, C.OP_AMAX], a4,
                                           row_scale=r4, tensor_scale=X4.s * W4.s, amax=am4, stream=stream)
    down = lambda: C.coda_gemm_epilogue(a4, Wd4, [C.OP_TENSOR_SCALE, C.OP_ADD_SIDE, C.OP_ROW_SUMSQ_PARTIAL], Y4,
                                        residual=h4, tensor_scale=a4.s * Wd4.s, row_partials=P4, stream=stream)
    per_gemm = {}
    for name, fn, fl in (("gate_up_swiglu_nvfp4_out", gate_up, 2 * M * 2 * F8 * H8),
                         ("down_residual", down, 2 * M * H8 * F8)):
        g_ms = _time(torch, fn, stream, steps)
        per_gemm[name] = {"ms": g_ms, "tflops": fl / (g_ms * 1e-3) / 1e12}
    nv4 = {"ms": ms, "tflops": flop / (ms * 1e-3) / 1e12, "tokens_per_s": M / (ms * 1e-3), "launches": 3,
           "vs_fp8_chain": out["mlp_fp8_C4"]["ms"] / ms,
           "quantize_x_ms": ms_q, "quantize_x_gbs": byt_q / (ms_q * 1e-3) / 1e9,
           "quantize_x_frac_of_hbm": byt_q / (ms_q * 1e-3) / 1e9 / pk["hbm"],
           "per_gemm": per_gemm,
           "note": "row RMS, gate/up GEMM + r + SwiGLU + NVFP4 quantisation of a (codes, block scales, amax), "
                   "down GEMM + residual + partials; X quantised beforehand (quantize_x_ms, the pass a previous "
                   "layer's epilogue would fold in)"}
    del h4, X4, W4, Wd4, Y4, P4, a4
    torch.cuda.empty_cache()
    # N4: the NVFP4 MLP backward (each GEMM's operands quantised along its own K)
    nvb = nvfp4_backward_workload(torch, C, S, steps, pk)
    out["mlp_nvfp4_N4"] = nv4
    out["mlp_nvfp4_backward_N4"] = nvb
    deferred.append(("fp4", nv4, flop, byt))
    deferred.append(("fp4", nvb, nvb.pop("flop"), nvb["bytes"]))
    # N3: the block forward at the 7B and 70B LLaMA-3 hidden sizes, beside torch eager
    for name, Hs, Fs in (("block_forward_7B_H4096_F14336", 4096, 14336), ("block_forward_70B_H8192_F28672", 8192,
                                                                           28672)):
        bi = S.block_inputs(M, Hs, Fs, seed=0, device="cuda")
        hs, us, Ys = (torch.empty((M, Hs), dtype=BF, device="cuda") for _ in range(3))
        rs_ = torch.empty((M,), device="cuda")
        as_ = torch.empty((M, Fs), dtype=BF, device="cuda")
        wss = torch.empty((C.coda_workspace_size(C.WS_BLOCK_FWD, M, Hs, Fs) // 4,), device="cuda")
        run = lambda: C.coda_block_forward(bi["O"], bi["R"], bi["W_o"], bi["W_gu"], bi["W_d"], EPS, hs, rs_, as_, Ys,
                                           wss, g=bi["g"], u=us, stream=stream)
        ms = _time(torch, run, stream, max(3, min(args.steps, 20)))
        flop = 2 * M * Hs * Hs + 2 * M * 2 * Fs * Hs + 2 * M * Hs * Fs
        byt = 2 * (M * Hs * 4 + Hs * Hs) + 2 * (M * Hs + 2 * Fs * Hs + M * Fs) + 2 * (M * Fs + Hs * Fs + 2 * M * Hs)
        roof = max(flop / (pk["bf16"] * 1e12), byt / (pk["hbm"] * 1e9)) * 1e3
        t_ms = _time(torch, lambda: unfused_chain(torch, bi, Fs), stream, max(3, min(args.steps, 10)))
        out[name] = {"ms": ms, "tflops": flop / (ms * 1e-3) / 1e12, "roofline_ms": roof, "roofline_frac": roof / ms,
                     "tokens_per_s": M / (ms * 1e-3), "launches": 4, "unfused_torch_eager_ms": t_ms,
                     "speedup_vs_unfused": t_ms / ms}
        if args.compile_compare:
            out[name].update(compiled_time(torch, lambda: unfused_chain(torch, bi, Fs), stream,
                                           max(3, min(args.steps, 10)), ms))
        del bi, hs, us, Ys, as_, wss
        torch.cuda.empty_cache()
    # N1: final RMSNorm + LM head + cross-entropy (vocabulary 128256), forward and backward
    V = 128256
    li = S.lm_head_inputs(M, H, V, seed=0)
    hl, gl, Wv, tg = (li[k].to("cuda").contiguous() for k in ("h", "g", "W_v", "targets"))
    ul = torch.empty((M, H), dtype=BF, device="cuda")
    rl, lse, loss, mean = (torch.empty((n,), device="cuda") for n in (M, M, M, 1))
    wsx = torch.empty((C.coda_workspace_size(C.WS_XENT_FWD, M, H, V) // 4,), device="cuda")
    fx = lambda: C.coda_lm_head_xent_forward(hl, gl, Wv, tg, EPS, ul, rl, lse, loss, mean, wsx, stream=stream)
    steps_x = max(3, min(args.steps, 20))
    ms_f = _time(torch, fx, stream, steps_x)
    el = torch.empty((M, V), dtype=BF, device="cuda")
    dhl = torch.empty((M, H), dtype=BF, device="cuda")
    dWv = torch.empty((V, H), device="cuda")
    dgl, cl = torch.empty((H,), device="cuda"), torch.empty((M,), device="cuda")
    wsb = torch.empty((C.coda_workspace_size(C.WS_XENT_BWD, M, H, V) // 4,), device="cuda")
    bx = lambda: C.coda_lm_head_xent_backward(hl, gl, Wv, tg, ul, rl, lse, 1.0, el, dhl, dWv, dgl, cl, wsb,
                                              stream=stream)
    ms_b = _time(torch, bx, stream, steps_x)
    flop = 2 * M * V * H
    byt_f = 2 * (M * H * 2 + V * H) + 4 * M * (2 * ((V + 255) // 256) + 5)
    byt_b = 2 * (V * H * 3 + M * V * 3 + M * H * 3) + 4 * V * H
    for name, ms, fl, by, nl in (("lm_head_xent_forward_N1", ms_f, flop, byt_f, 3),
                                 ("lm_head_xent_backward_N1", ms_b, 3 * flop, byt_b, 5)):
        roof = max(fl / (pk["bf16"] * 1e12), by / (pk["hbm"] * 1e9)) * 1e3
        out[name] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "roofline_ms": roof, "roofline_frac": roof / ms,
                     "tokens_per_s": M / (ms * 1e-3), "launches": nl, "vocab": V}
    del hl, gl, Wv, tg, ul, el, dhl, dWv, wsb, wsx
    torch.cuda.empty_cache()
    out["_deferred"] = deferred   # finished by finish_lib_peaks once nothing else is left to time
    return out


def nvfp4_backward_workload(torch, C, S, steps, pk, M=M_TOK, H=4096, F=14336, peak4=None):
    """Device time of the NVFP4 MLP backward at the LLaMA-3-8B MLP shape: 9 launches (dY
    quantised along rows and columns in one pass, the dA GEMM with the SwiGLU-backward epilogue,
    the row reduce, e along rows and columns in one pass, silu(G) U and h along columns, the
    dW_d, dh and dW GEMMs).
    The weights' transposed quantisation is weight preparation, outside the timing."""
    t = S.nvfp4_mlp_bwd_inputs(M, H, F, seed=0, device="cuda")
    sc = lambda x: float(x.abs().max()) / (6 * 448)
    W_guT, W_dT = C.Nvfp4.empty(H, 2 * F, sc(t["W_gu"])), C.Nvfp4.empty(F, H, sc(t["W_d"]))
    C.coda_quantize_nvfp4_t(t["W_gu"], W_guT)
    C.coda_quantize_nvfp4_t(t["W_d"], W_dT)
    nv = lambda R, K: C.Nvfp4.empty(R, K)
    bufs = dict(dY_r=nv(M, H), dY_c=nv(H, M), e=torch.empty((M, 2 * F), dtype=torch.bfloat16, device="cuda"),
                e_r=nv(M, 2 * F), e_c=nv(2 * F, M), a_c=nv(F, M), x_c=nv(H, M),
                amax_dy=torch.empty((1,), device="cuda"), amax_e=torch.empty((1,), device="cuda"),
                c=torch.empty((M,), device="cuda"), dh=torch.empty((M, H), dtype=torch.bfloat16, device="cuda"),
                dW_d=torch.empty((H, F), device="cuda"), dW=torch.empty((2 * F, H), device="cuda"))
    ws = torch.empty((C.coda_workspace_size(C.WS_MLP_NVFP4_BWD, M, H, F) // 4,), device="cuda")
    G, U = t["Z"][:, :F].float(), t["Z"][:, F:].float()
    s_a = float((torch.nn.functional.silu(G) * U).abs().max()) / (6 * 448)
    del G, U
    s_dy, s_x = sc(t["dY"]), sc(t["h"])
    s_e = [1.0]
    b = bufs
    run = lambda: C.coda_mlp_nvfp4_backward(t["h"], W_guT, W_dT, t["Z"], t["r"], t["dY"], s_x, s_a, s_dy, s_e[0],
                                            b["dY_r"], b["dY_c"], b["e"], b["e_r"], b["e_c"], b["a_c"], b["x_c"],
                                            b["amax_dy"], b["amax_e"], b["c"], b["dh"], b["dW_d"], b["dW"], ws)
    run()
    torch.cuda.synchronize()
    s_e[0] = float(b["amax_e"].item()) / (6 * 448)      # delayed scaling from the previous pass
    ms = _time(torch, run, torch.cuda.current_stream(), steps)
    flop = 12 * M * H * F                                # dA, dW_d: 2MHF each; dh, dW: 4MHF each
    n4 = lambda R, K: R * K // 2 + R * K // 16           # NVFP4 codes + block scales
    byt = (2 * M * H + 2 * n4(M, H)) + (n4(M, H) + n4(F, H) + 2 * 2 * M * F + 2 * 2 * M * F + 4 * M) + \
        (2 * 2 * M * F + 2 * n4(M, 2 * F)) + (2 * 2 * M * F + n4(F, M)) + (2 * M * H + n4(H, M)) + \
        (n4(H, M) + n4(F, M) + 4 * H * F) + (n4(M, 2 * F) + n4(H, 2 * F) + 2 * 3 * M * H + 4 * M) + \
        (n4(2 * F, M) + n4(H, M) + 4 * 2 * F * H)
    res = {"ms": ms, "tflops": flop / (ms * 1e-3) / 1e12, "tokens_per_s": M / (ms * 1e-3), "launches": 9,
           "bytes": byt, "flop": flop,
           "note": "quantise dY (rows and columns, one pass), dA GEMM + SwiGLU-bwd (bf16 e), row reduce, quantise e "
                   "(rows and columns, one pass), silu(G) U and h (columns), dW_d, dh GEMM + RMSNorm-bwd combine, dW; "
                   "NVFP4 operands blocked along each GEMM's K"}
    if peak4:
        roof = max(flop / (peak4 * 1e12), byt / (pk["hbm"] * 1e9)) * 1e3
        res.update({"roofline_ms": roof, "roofline_frac": roof / ms, "peak_tflops": peak4})
    del t, bufs, ws
    torch.cuda.empty_cache()
    return res


def compiled_time(torch, fn, stream, steps, ms_coda):
    """Device time of torch.compile(fn) (compiled on its first calls, outside the timing)."""
    try:
        cf = torch.compile(fn)
        t = _time(torch, cf, stream, steps, warmup=3)
        return {"torch_compile_ms": t, "speedup_vs_torch_compile": t / ms_coda}
    except Exception as ex:
        return {"torch_compile_error": f"{type(ex).__name__}: {ex}"[:200]}


LAYERS = (("layer_1B_H2048_F8192", 2048, 8192, 32, 8, 64),
          ("layer_7B_H4096_F14336", 4096, 14336, 32, 8, 128),
          ("layer_70B_H8192_F28672", 8192, 28672, 64, 8, 128))


def layer_workloads(torch, C, S, args, stream):
    """A whole LLaMA-style decoder layer forward at 16384 tokens (16 sequences of 1024):
    attention-input RMSNorm + QKV + RoPE, causal attention with grouped KV heads, output
    projection + residual, MLP RMSNorm + gate/up + SwiGLU + down + residual.  Attention is
    the library's (torch scaled_dot_product_attention) on both sides; everything else is
    either the fused chain (coda_fold_gain + coda_qkv_rope, then coda_block_forward) or
    torch eager ops with cuBLAS GEMMs.  Device time per layer, both sides, and attention
    alone."""
    BF = torch.bfloat16
    Fn = torch.nn.functional
    M, seq = M_TOK, 1024
    B = M // seq
    steps = max(3, min(args.steps, 10))
    out = {}
    for name, H, F, nq, nkv, hd in LAYERS:
        li = S.layer_inputs(M, H, F, nq, nkv, hd, seed=0, device="cuda")
        x, g1, Wqkv, W_o, g2, W_gu, W_d = (li[k] for k in ("x", "g_attn", "W_qkv", "W_o", "g_mlp", "W_gu", "W_d"))
        nqk = (nq + nkv) * hd
        cos = torch.empty((seq, hd // 2), device="cuda")
        sin = torch.empty_like(cos)
        C.coda_rope_table(seq, hd, 500000.0, cos, sin, stream=stream)
        Wqf = torch.empty_like(Wqkv)
        r1 = torch.empty((M,), device="cuda")
        qkv = torch.empty((M, Wqkv.shape[0]), dtype=BF, device="cuda")
        h, u, Y = (torch.empty((M, H), dtype=BF, device="cuda") for _ in range(3))
        r2 = torch.empty((M,), device="cuda")
        a = torch.empty((M, F), dtype=BF, device="cuda")
        ws = torch.empty((C.coda_workspace_size(C.WS_BLOCK_FWD, M, H, F) // 4,), device="cuda")

        def attention(t):
            q = t[:, :nq * hd].view(B, seq, nq, hd).transpose(1, 2)
            k = t[:, nq * hd:nqk].view(B, seq, nkv, hd).transpose(1, 2)
            v = t[:, nqk:].view(B, seq, nkv, hd).transpose(1, 2)
            o = Fn.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True)
            return o.transpose(1, 2).reshape(M, nq * hd)

        def ours():
            C.coda_fold_gain(Wqkv, g1, Wqf, stream=stream)
            C.coda_qkv_rope(x, Wqf, EPS, seq, hd, nqk, cos, sin, r1, qkv, stream=stream)
            o = attention(qkv)
            C.coda_block_forward(o, x, W_o, W_gu, W_d, EPS, h, r2, a, Y, ws, g=g2, u=u, stream=stream)
            return Y

        def rope_t(t, nh):
            tf = t.float().view(B, seq, nh, hd // 2, 2)
            c, s_ = cos.view(1, seq, 1, hd // 2), sin.view(1, seq, 1, hd // 2)
            x0, x1 = tf[..., 0], tf[..., 1]
            return torch.stack((x0 * c - x1 * s_, x0 * s_ + x1 * c), -1).view(M, nh * hd).to(BF)

        def torch_layer():
            xf = x.float()
            xn = (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + EPS)).to(BF) * g1.to(BF)
            t = Fn.linear(xn, Wqkv)
            t = torch.cat((rope_t(t[:, :nq * hd], nq), rope_t(t[:, nq * hd:nqk], nkv), t[:, nqk:]), 1)
            o = attention(t)
            return unfused_chain(torch, {"O": o, "R": x, "W_o": W_o, "g": g2, "W_gu": W_gu, "W_d": W_d}, F)

        ms = _time(torch, ours, stream, steps)
        t_ms = _time(torch, torch_layer, stream, steps)
        att_ms = _time(torch, lambda: attention(qkv), stream, steps)
        Yc = ours().float()
        Yt = torch_layer().float()
        torch.cuda.synchronize()
        diff = float((Yc - Yt).abs().max() / Yt.abs().max())
        out[name] = {"ms": ms, "torch_eager_ms": t_ms, "speedup_vs_torch_eager": t_ms / ms,
                     "attention_ms": att_ms, "non_attention_speedup": (t_ms - att_ms) / (ms - att_ms),
                     "tokens_per_s": M / (ms * 1e-3), "normwise_diff_vs_torch_eager": diff,
                     "heads": f"{nq} query / {nkv} key-value heads of {hd}"}
        if args.compile_compare:
            out[name].update(compiled_time(torch, torch_layer, stream, steps, ms))
        del li, x, g1, Wqkv, W_o, g2, W_gu, W_d, Wqf, qkv, h, u, Y, a, ws, Yc, Yt
        torch.cuda.empty_cache()
    return out


def unfused_chain(torch, d, F, parts=False):
    """The same block forward as separate torch eager ops (cuBLAS GEMMs, then residual add,
    RMSNorm, SwiGLU, residual add as their own kernels): the comparator the pages measure
    against.  With parts=True also returns its intermediates h, r, a."""
    F_ = torch.nn.functional
    hh = F_.linear(d["O"], d["W_o"]) + d["R"]
    var = hh.float().pow(2).mean(-1, keepdim=True)
    rs = torch.rsqrt(var + EPS)
    y = (hh.float() * rs).to(torch.bfloat16) * d["g"].to(torch.bfloat16)
    z = F_.linear(y, d["W_gu"])
    act = F_.silu(z[:, :F]) * z[:, F:]
    out = F_.linear(act, d["W_d"]) + hh
    return (out, {"h": hh, "r": rs[:, 0], "a": act, "Y": out}) if parts else out


def unfused_compare(torch, d, fused, inp, stream, args):
    """torch eager bf16 chain of the same block (separate GEMM / add / RMSNorm / SwiGLU
    kernels, cuBLAS GEMMs): its time, and the max relative error (RMS floor) of h, r, a and Y
    of both chains against the fp64 oracle's plain chain on 256 sampled rows.  `fused` holds
    the fused chain's h, r, a, Y from its last step.  a is the product of two bf16-rounded
    GEMM results in both chains, so its error carries the bf16 storage of h (or u = h g) and
    of the GEMM inputs, whichever chain computes it."""
    import numpy as np

    import oracle as O

    def chain():
        return unfused_chain(torch, d, FFN)

    for _ in range(3):
        Yt = chain()
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        Yt = chain()
    e1.record()
    torch.cuda.synchronize()
    t_ms = e0.elapsed_time(e1) / n
    _, tparts = unfused_chain(torch, d, FFN, parts=True)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(0).choice(M_TOK, size=256, replace=False))
    x = {k: inp[k].to(torch.float64).numpy() for k in ("O", "R", "W_o", "W_gu", "W_d", "g")}
    ref = O.block_forward(x["O"][rows], x["R"][rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], EPS)
    rows_t = torch.from_numpy(rows).cuda()
    pick = lambda t: t.index_select(0, rows_t).double().cpu().numpy()
    errs = {}
    for name in ("h", "r", "a", "Y"):
        errs[name] = {"fused": O.max_rel_err(pick(fused[name]), ref[name]),
                      "unfused_torch": O.max_rel_err(pick(tparts[name]), ref[name])}
    return {"unfused_torch_eager_ms_per_step": t_ms, "unfused_tokens_per_s": M_TOK / (t_ms * 1e-3),
            "max_rel_err_fused_vs_oracle": errs["Y"]["fused"],
            "max_rel_err_unfused_torch_vs_oracle": errs["Y"]["unfused_torch"],
            "max_rel_err_vs_oracle": errs, "error_rows": 256,
            "error_metric": "max_i |x_i - ref_i| / max(|ref_i|, rms(ref)) against the fp64 oracle's plain chain"}


def backward_compare(torch, C, S, stream):
    """The block backward's row outputs (dh = dR, dO, and e) against the fp64 oracle on 256
    sampled rows: the fused chain (training-mode forward, then coda_block_backward) and torch
    autograd through the unfused bf16 chain.  The weight gradients sum over every row; the
    tests check them (on exact inputs at full size)."""
    import numpy as np

    import oracle as O
    M, H, F = M_TOK, HID, FFN
    BF = torch.bfloat16
    inp = S.block_inputs(M, H, F, seed=0, with_grad=True)
    d = {k: inp[k].to("cuda").contiguous() for k in ("O", "R", "W_o", "W_gu", "W_d", "g", "dY")}
    h, u, a, Y = (torch.empty((M, n), dtype=BF, device="cuda") for n in (H, H, F, H))
    r = torch.empty((M,), device="cuda")
    Z = torch.empty((M, 2 * F), dtype=BF, device="cuda")
    wsf = torch.empty((C.coda_workspace_size(C.WS_BLOCK_FWD, M, H, F) // 4,), device="cuda")
    C.coda_block_forward(d["O"], d["R"], d["W_o"], d["W_gu"], d["W_d"], EPS, h, r, a, Y, wsf, Z=Z, g=d["g"], u=u,
                         stream=stream)
    e = torch.empty((M, 2 * F), dtype=BF, device="cuda")
    dh, dO = torch.empty((M, H), dtype=BF, device="cuda"), torch.empty((M, H), dtype=BF, device="cuda")
    dW_o, dW_gu, dW_d = (torch.empty(s, device="cuda") for s in ((H, H), (2 * F, H), (H, F)))
    dg, c = torch.empty((H,), device="cuda"), torch.empty((M,), device="cuda")
    wsb = torch.empty((C.coda_workspace_size(C.WS_BLOCK_BWD, M, H, F) // 4,), device="cuda")
    C.coda_block_backward(d["O"], d["W_o"], d["W_gu"], d["W_d"], d["g"], h, r, Z, a, d["dY"], e, dh, dO, dW_o,
                          dW_gu, dW_d, dg, c, wsb, stream=stream)
    torch.cuda.synchronize()
    leaf = {k: d[k].clone().requires_grad_(k in ("O", "R")) for k in ("O", "R", "W_o", "W_gu", "W_d", "g")}
    unfused_chain(torch, leaf, F).backward(d["dY"])
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(1).choice(M, size=256, replace=False))
    x = {k: inp[k].to(torch.float64).numpy() for k in ("O", "R", "W_o", "W_gu", "W_d", "g", "dY")}
    f = O.block_forward(x["O"][rows], x["R"][rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], EPS)
    b = O.block_backward_fused(f, x["O"][rows], x["W_o"], x["g"], x["W_gu"], x["W_d"], x["dY"][rows])
    rows_t = torch.from_numpy(rows).cuda()
    pick = lambda t: t.detach().index_select(0, rows_t).double().cpu().numpy()
    errs = {"dh": {"fused": O.max_rel_err(pick(dh), b["dh"]), "unfused_torch": O.max_rel_err(pick(leaf["R"].grad), b["dh"])},
            "dO": {"fused": O.max_rel_err(pick(dO), b["dO"]), "unfused_torch": O.max_rel_err(pick(leaf["O"].grad), b["dO"])},
            "e": {"fused": O.max_rel_err(pick(e), b["e"])}}
    return {"max_rel_err_vs_oracle": errs, "error_rows": 256,
            "note": "row outputs of the block backward; e = r [dG | dU] exists in the fused chain only"}


def main():
    args = parse()
    world, rank, local = dist_init(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.traffic_pass or args.nvfp4_pass or args.row_rms_pass or args.nvfp4_bwd_pass or args.fp8_pass:
        if rank == 0:
            if args.traffic_pass:
                traffic_pass(args)
            elif args.nvfp4_pass:
                nvfp4_pass(args)
            elif args.fp8_pass:
                fp8_pass(args)
            elif args.nvfp4_bwd_pass:
                import torch

                import coda_synth as S
                from gemm_epilogue_transformer_tcgen05_gb300 import coda as C
                C.lib()
                res = nvfp4_backward_workload(torch, C, S, 1, peaks(), M=args.tokens)
                print(json.dumps({"nvfp4_bwd_pass": {"tokens": args.tokens, "hidden": 4096, "ffn": 14336,
                                                     "order": "weight prep (2 launches), backward (warm-up "
                                                              "with s_e = 1), then 3 warm-up + 1 timed",
                                                     "ms": res["ms"]}}), flush=True)
            else:
                row_rms_pass(args)
        return
    run_coda(args, world, rank, local)


if __name__ == "__main__":
    main()
