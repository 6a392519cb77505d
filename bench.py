"""Benchmark of the weight-only quantized decode GEMV on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--m M]

One JSON line on rank 0 (stdout); everything else goes to stderr.

Default workload ("cbk4_7b_stack"): the projection stack of a 32-layer 7B
decoder -- per layer q/k/v/o 4096x4096, gate/up 11008x4096, down 4096x11008
(224 projections, 4-bit scalar codebook, 16 fp16 centroids each) plus a
32000x4096 LM head with an 8-bit codebook (256 centroids) -- at M = 1.  The
projections that share their input run as one stacked handle each (q|k|v and
gate|up), so one step is one token of 129 GEMV calls, replayed as CUDA
graphs.  The stack is 3.37 GB of packed weights, far larger than L2, so no
flush is needed.
Inputs are synthetic and seeded (see bit_weight_only_gb300/inputs.py).

The metric is the achieved weight-stream bandwidth: algorithmic bytes
(packed weights + codebooks/scales + x + y) per step / device time per step.

--impl reference times the CPU oracle (fp64, plain C, this repository's
test reference) on a bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Quantized decode GEMV achieved HBM GB/s & % of GB300 peak, M=1..16"
UNIT = "GB/s"


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


def hbm_peak():
    p = measured_peaks()
    if p and p.get("hbm_gbs"):
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _code_only(text: str) -> str:
    """C/C++ source without its comments and with whitespace runs collapsed
    (string and character literals kept as they are)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


# The sources of the kernels that stream each format at M = 1 (the kernel,
# its format's decode, the shared device helpers and launch code), whose
# code keys the stored DRAM-traffic captures: a change to any other kernel
# leaves them valid.  M > 1 adds the tensor-core kernels' sources.
KERNEL_SOURCES = {
    "cbk4": ["gemv_kernel.cuh", "rowgroup_kernel.cuh", "fmt_cbk.cuh", "device_common.cuh", "launch_table.cuh",
             "formats.h", "fmt_cbk4.cu", "fmt_cbk8.cu"],
    "cbk8": ["gemv_kernel.cuh", "rowgroup_kernel.cuh", "fmt_cbk.cuh", "device_common.cuh", "launch_table.cuh",
             "formats.h", "fmt_cbk8.cu"],
    "q4_0": ["gemv_kernel.cuh", "fmt_fields.cuh", "device_common.cuh", "launch_table.cuh", "formats.h", "fmt_q4_0.cu"],
    "pq2_0": ["gemv_kernel.cuh", "fmt_fields.cuh", "device_common.cuh", "launch_table.cuh", "formats.h", "fmt_pq2.cu"],
    "aqlm_2x8": ["gemv_kernel.cuh", "device_common.cuh", "formats.h", "fmt_aqlm.cu"],
    "cbk4_row": ["gemv_kernel.cuh", "fmt_cbk.cuh", "device_common.cuh", "launch_table.cuh", "formats.h",
                 "fmt_cbk4row.cu"],
    "aqlm_1x16": ["gemv_kernel.cuh", "device_common.cuh", "formats.h", "fmt_aqlm1x16.cu"],
}
KERNEL_SOURCES_MMA = ["mma_kernel.cuh", "tc5_kernel.cuh", "fmt_aqlm_mma.cu"]


def kernel_source_hash(fmt: str | None = None, M: int = 1) -> str:
    """Hash of the code (comments and layout ignored) of the sources behind
    format fmt's kernels at M rows (all of csrc when fmt has no list), which
    keys the stored DRAM-traffic captures."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_weight_only_gb300", "csrc")
    files = KERNEL_SOURCES.get(fmt)
    files = (files + (KERNEL_SOURCES_MMA if M > 1 else [])) if files else sorted(os.listdir(csrc))
    for f in files:
        h.update(f.encode())
        h.update(_code_only(open(os.path.join(csrc, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


# ----------------------------------------------------------- workloads ----

LLAMA7B = [("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096), ("o", 4096, 4096),
           ("gate", 11008, 4096), ("up", 11008, 4096), ("down", 4096, 11008)]


LLAMA70B_AQLM = [("gate", 28672, 8192), ("up", 28672, 8192), ("down", 8192, 28672),
                 ("q", 8192, 8192), ("o", 8192, 8192)]


def cbk4_stack_specs(layers=32, stacked=True, head=True, glu=False):
    """The 7B projection stack.  stacked: q|k|v and gate|up, which share
    their input, run as one stacked handle each (4 GEMV calls per layer);
    glu: gate|up as a fused SiLU(gate)*up handle instead (output 11008)."""
    specs = []
    for layer in range(layers):
        if stacked:
            specs += [("cbk4", f"L{layer}.qkv", [4096, 4096, 4096], 4096),
                      ("cbk4", f"L{layer}.o", 4096, 4096),
                      ("cbk4_glu", f"L{layer}.gate_up", 11008, 4096) if glu else
                      ("cbk4", f"L{layer}.gate_up", [11008, 11008], 4096),
                      ("cbk4", f"L{layer}.down", 4096, 11008)]
        else:
            for name, N, K in LLAMA7B:
                specs.append(("cbk4", f"L{layer}.{name}", N, K))
    if head:
        specs.append(("cbk8", "lm_head", 32000, 4096))
    return specs


def total_rows(N):
    return sum(N) if isinstance(N, (list, tuple)) else N


WORKLOADS = {
    # name: (specs, dominant format, description)
    "cbk4_7b_stack": (lambda: cbk4_stack_specs(), "cbk4",
                      "7B decoder projection stack, 224 CBK4 projections (q|k|v and gate|up stacked: "
                      "128 calls) + CBK8 LM head 32000x4096"),
    "cbk4_7b_layer": (lambda: cbk4_stack_specs(layers=1, head=False), "cbk4",
                      "one layer of the 7B CBK4 projection stack: q|k|v 12288x4096, o 4096x4096, gate|up "
                      "22016x4096, down 4096x11008 (the stack's four call shapes; the small case for "
                      "DRAM-traffic captures)"),
    "cbk4_7b_stack_glu": (lambda: cbk4_stack_specs(glu=True), "cbk4",
                          "7B decoder projection stack, 224 CBK4 projections as 128 calls (q|k|v stacked, "
                          "gate|up fused: SiLU(gate)*up stored) + CBK8 LM head 32000x4096"),
    "cbk4_7b_stack_unfused": (lambda: cbk4_stack_specs(stacked=False), "cbk4",
                              "7B decoder projection stack, 224 CBK4 calls + CBK8 LM head 32000x4096"),
    "q4_0_4096": (lambda: [("q4_0", "q4_0", 4096, 4096)], "q4_0", "Q4_0 GEMV 4096x4096"),
    "q4_0_down": (lambda: [("q4_0", "down", 8192, 28672)], "q4_0", "Q4_0 down 8192x28672"),
    "pq2_5120": (lambda: [("pq2_0", "gate_up", 34816, 5120), ("pq2_0", "down", 5120, 17408)],
                 "pq2_0", "PQ2_0 gate+up 34816x5120 and down 5120x17408"),
    "pq2_down": (lambda: [("pq2_0", "down", 8192, 28672)], "pq2_0", "PQ2_0 down 8192x28672"),
    "cbk4_down": (lambda: [("cbk4", "down", 8192, 28672)], "cbk4", "CBK4 down 8192x28672"),
    "cbk8_head": (lambda: [("cbk8", "lm_head", 32000, 4096)], "cbk8", "CBK8 LM head 32000x4096"),
    "cbk4_4096": (lambda: [("cbk4", "q", 4096, 4096)], "cbk4", "CBK4 7B attention projection 4096x4096"),
    "cbk4_gate": (lambda: [("cbk4", "gate", 11008, 4096)], "cbk4", "CBK4 7B gate projection 11008x4096"),
    "aqlm_70b_layer": (lambda: [("aqlm_2x8", n, N, K) for n, N, K in LLAMA70B_AQLM], "aqlm_2x8",
                       "70B-shaped AQLM 2x8 layer: gate, up 28672x8192, down 8192x28672, q, o 8192x8192"),
    "aqlm_70b_layer_stacked": (lambda: [("aqlm_2x8", "gate_up", [28672, 28672], 8192)] +
                               [("aqlm_2x8", n, N, K) for n, N, K in LLAMA70B_AQLM[2:]], "aqlm_2x8",
                               "70B-shaped AQLM 2x8 layer with gate|up stacked (one call, a codebook pair "
                               "each): gate|up 57344x8192, down 8192x28672, q, o 8192x8192"),
    "aqlm_down": (lambda: [("aqlm_2x8", "down", 8192, 28672)], "aqlm_2x8", "AQLM 2x8 down 8192x28672"),
    "aqlm1x16_70b_layer": (lambda: [("aqlm_1x16", n, N, K) for n, N, K in LLAMA70B_AQLM], "aqlm_1x16",
                           "70B-shaped AQLM 1x16 layer: gate, up 28672x8192, down 8192x28672, q, o 8192x8192"),
    "aqlm1x16_down": (lambda: [("aqlm_1x16", "down", 8192, 28672)], "aqlm_1x16", "AQLM 1x16 down 8192x28672"),
    "cbk4row_7b_layer": (lambda: [("cbk4_row", n, N, K) for n, N, K in LLAMA7B], "cbk4_row",
                         "7B decoder layer, CBK4 with per-row fp32 codebooks: q, k, v, o 4096x4096, "
                         "gate, up 11008x4096, down 4096x11008"),
    "cbk4row_down": (lambda: [("cbk4_row", "down", 8192, 28672)], "cbk4_row",
                     "CBK4 with per-row fp32 codebooks, down 8192x28672"),
    "cbk8row_head": (lambda: [("cbk8_row", "lm_head", 32000, 4096)], "cbk8_row",
                     "CBK8 LM head 32000x4096 with per-row fp32 codebooks (256 per row)"),
    "pq2_5120_glu": (lambda: [("pq2_0_glu", "gate_up", 17408, 5120), ("pq2_0", "down", 5120, 17408)], "pq2_0_glu",
                     "PQ2_0 MLP of the 5120/17408 model: gate and up 17408x5120 with SiLU(gate)*up fused "
                     "(one launch), then down 5120x17408"),
}


def canonical_extra_bytes(fmt, N):
    return {"q4_0": 0, "pq2_0": 0, "cbk4": 32, "cbk8": 512, "aqlm_2x8": 2 * N + 8192,
            "aqlm_1x16": 2 * N + 65536 * 8 * 2, "cbk4_row": 64 * N, "cbk8_row": 1024 * N}[fmt]


def stacked_extra_bytes(fmt, segs):
    """Codebooks and scales of a stacked handle's canonical inputs: those of
    its segments as separate matrices (a codebook, or AQLM's pair, per
    segment; one scale per row)."""
    return sum(canonical_extra_bytes(fmt, n) for n in segs)


def build_handles(specs, M, device, seed=0):
    """Create one handle per projection from device-drawn canonical inputs."""
    import torch
    from bit_weight_only_gb300 import inputs, qgemv
    ops = []
    # all activations in one buffer and all outputs in another, so the end to
    # end run moves one input copy and one output copy per step
    x_all = torch.empty(sum(M * K for _, _, _, K in specs), dtype=torch.float16, device=device)
    y_all = torch.empty(sum(M * total_rows(N) for _, _, N, _ in specs), dtype=torch.float32, device=device)
    xo = yo = 0
    c16 = inputs.cbk_centroids(16)
    c256 = inputs.cbk_centroids(256)
    p16, p256 = inputs.cbk_cell_probs(c16), inputs.cbk_cell_probs(c256)
    for fmt, name, N, K in specs:
        tag = f"bench/{name}"
        scales = cb = None
        if isinstance(N, (list, tuple)):   # stacked projections, one codebook each
            segs = list(N)
            if fmt == "cbk4":
                packed = torch.cat([inputs.cbk_packed_cuda(f"{tag}/{s}", n, K, 4, p16, device, seed)
                                    for s, n in enumerate(segs)])
                h = qgemv.QGemv.stacked(fmt, segs, K, packed, None, np.concatenate([c16] * len(segs)))
            elif fmt == "aqlm_2x8":  # codes, scales and a codebook pair per segment
                parts = [inputs.aqlm_inputs_cuda(f"{tag}/{s}", n, K, device=device, seed=seed)
                         for s, n in enumerate(segs)]
                packed = torch.cat([q[0] for q in parts])
                h = qgemv.QGemv.stacked(fmt, segs, K, packed, torch.cat([q[1] for q in parts]),
                                        torch.cat([q[2] for q in parts]))
                del parts
            else:
                raise ValueError(fmt)
            N = sum(segs)
            nbytes = qgemv.qgemv_packed_bytes(fmt, N, K) + stacked_extra_bytes(fmt, segs) + 2 * M * K + 4 * M * N
            del packed
            x = x_all[xo:xo + M * K].view(M, K)
            x.copy_(inputs.x_fp16_cuda(f"{tag}/x", M, K, device=device, seed=seed))
            y = y_all[yo:yo + M * N].view(M, N)
            xo += M * K
            yo += M * N
            ops.append({"fmt": fmt, "name": name, "N": N, "K": K, "h": h, "x": x, "y": y, "bytes": nbytes})
            continue
        if fmt == "cbk4_glu":  # gate and up in one handle (a codebook each), output SiLU(gate) * up
            pg = inputs.cbk_packed_cuda(f"{tag}/gate", N, K, 4, p16, device, seed)
            pu = inputs.cbk_packed_cuda(f"{tag}/up", N, K, 4, p16, device, seed)
            h = qgemv.QGemv.glu("cbk4", N, K, pg, pu, c16, c16)
            del pg, pu
            x = x_all[xo:xo + M * K].view(M, K)
            x.copy_(inputs.x_fp16_cuda(f"{tag}/x", M, K, device=device, seed=seed))
            y = y_all[yo:yo + M * N].view(M, N)
            xo += M * K
            yo += M * N
            nbytes = 2 * (qgemv.qgemv_packed_bytes("cbk4", N, K) + canonical_extra_bytes("cbk4", N)) + 2 * M * K + 4 * M * N
            ops.append({"fmt": fmt, "name": name, "N": N, "K": K, "h": h, "x": x, "y": y, "bytes": nbytes})
            continue
        if fmt == "pq2_0_glu":  # gate and up in one handle, output SiLU(gate) * up
            pg = inputs.pq2_packed_cuda(f"{tag}/gate", N, K, device=device, seed=seed)
            pu = inputs.pq2_packed_cuda(f"{tag}/up", N, K, device=device, seed=seed)
            h = qgemv.QGemv.glu("pq2_0", N, K, pg, pu)
            del pg, pu
            x = x_all[xo:xo + M * K].view(M, K)
            x.copy_(inputs.x_fp16_cuda(f"{tag}/x", M, K, device=device, seed=seed))
            y = y_all[yo:yo + M * N].view(M, N)
            xo += M * K
            yo += M * N
            nbytes = 2 * qgemv.qgemv_packed_bytes("pq2_0", N, K) + 2 * M * K + 4 * M * N
            ops.append({"fmt": fmt, "name": name, "N": N, "K": K, "h": h, "x": x, "y": y, "bytes": nbytes})
            continue
        if fmt == "cbk4":
            packed = inputs.cbk_packed_cuda(tag, N, K, 4, p16, device, seed)
            cb = c16
        elif fmt == "cbk8":
            packed = inputs.cbk_packed_cuda(tag, N, K, 8, p256, device, seed)
            cb = c256
        elif fmt == "pq2_0":
            packed = inputs.pq2_packed_cuda(tag, N, K, device=device, seed=seed)
        elif fmt == "q4_0":
            w = inputs.w_fp32_cuda(tag, N, K, device=device, seed=seed)
            packed = qgemv.quantize_q4_0(w)
            del w
        elif fmt == "aqlm_2x8":
            packed, scales, cb = inputs.aqlm_inputs_cuda(tag, N, K, device=device, seed=seed)
        elif fmt == "aqlm_1x16":
            packed, scales, cb = inputs.aqlm_1x16_inputs_cuda(tag, N, K, device=device, seed=seed)
        elif fmt == "cbk4_row":
            packed = inputs.cbk_packed_cuda(tag, N, K, 4, p16, device, seed)
            cb = inputs.cbk_row_codebooks(inputs.rng(f"{tag}/cb", seed), N)
        elif fmt == "cbk8_row":
            packed = inputs.cbk_packed_cuda(tag, N, K, 8, p256, device, seed)
            cb = inputs.cbk_row_codebooks(inputs.rng(f"{tag}/cb", seed), N, L=256)
        else:
            raise ValueError(fmt)
        h = qgemv.QGemv(fmt, N, K, packed, scales, cb)
        del packed
        x = x_all[xo:xo + M * K].view(M, K)
        x.copy_(inputs.x_fp16_cuda(f"{tag}/x", M, K, device=device, seed=seed))
        y = y_all[yo:yo + M * N].view(M, N)
        xo += M * K
        yo += M * N
        nbytes = qgemv.qgemv_packed_bytes(fmt, N, K) + canonical_extra_bytes(fmt, N) + 2 * M * K + 4 * M * N
        ops.append({"fmt": fmt, "name": name, "N": N, "K": K, "h": h, "x": x, "y": y,
                    "bytes": nbytes})
    torch.cuda.synchronize()
    return ops, x_all, y_all


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"qgemv_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "0x1", "1"):
                    reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------- our arm ------

def x_int8_launches(M, prepared=False):
    """Launches of one PQ2_0 INT8-path call: up to three rows, the CUDA-core
    kernel (four, two, then one rows per launch); four or more, the
    activation prologue then the tensor-core kernel (on prepared activations
    the tensor-core kernel alone)."""
    if M < 4:
        return M // 2 + M % 2
    return 1 if prepared else 2


def max_over_ranks(values, world, device):
    """Each value's maximum over the ranks (the slowest rank sets the job's
    time); the values themselves on one rank."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def run_ours(args, rank, world, device):
    import torch
    from bit_weight_only_gb300 import build, qgemv
    build.build()            # compiles only if sources changed
    qgemv.load()             # fails loudly without the library

    specs_fn, dominant, desc = WORKLOADS[args.workload]
    M = args.m
    t_setup = time.time()
    specs = specs_fn()
    # A step must read its weights from HBM: a workload smaller than three L2s
    # gets that many independent copies (own weights, x and y) and a step
    # runs all of them back to back, so no copy is still in L2 when its turn
    # comes round again.
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    one_copy = sum(qgemv.qgemv_packed_bytes(f[:-4] if f.endswith("_glu") else f, total_rows(N), K)
                   * (2 if f.endswith("_glu") else 1) for f, _, N, K in specs)
    R = 1 if one_copy >= 3 * l2 else -(-3 * l2 // one_copy)
    copies = [build_handles(specs, M, device, seed=r) for r in range(R)]
    ops = [o for c_ops, _, _ in copies for o in c_ops]
    if args.x_int8:  # PQ2_0 integer path: INT8 activations per group of 128
        for o in ops:
            if o["fmt"] == "pq2_0":
                o["h"].set_x_int8(True)
                o["x_int8"] = True
                if args.prepared is not None:  # the prologue (Hadamard mixing, codes) then the GEMV
                    M_, K_ = o["x"].shape
                    o["xq"] = torch.empty(qgemv.qgemv_xq_bytes(M_, K_), dtype=torch.uint8, device=device)
                    o["signs"] = (torch.randint(0, 2, (K_,), device=device, dtype=torch.int8) * 2 - 1
                                  if args.prepared else None)
    log(f"[bench] rank {rank}: {len(specs)} GEMVs x {R} copies ready in {time.time() - t_setup:.1f}s")

    step_bytes = sum(o["bytes"] for o in ops)
    # the dominant format's calls (with its fused gate|up handles, if any)
    in_dom = lambda o: o["fmt"] in (dominant, dominant + "_glu")
    dom = [o for o in ops if in_dom(o)]
    rest = [o for o in ops if not in_dom(o)]
    dom_bytes = sum(o["bytes"] for o in dom)

    stream = torch.cuda.Stream(device=device)
    graphs = []  # the dominant format's GEMVs, then the rest (or None)
    for group in (dom, rest):
        if not group:
            graphs.append(None)
            continue
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for o in group:
                cs = torch.cuda.current_stream()
                if "xq" in o:
                    M_, K_ = o["x"].shape
                    qgemv.qgemv_prepare_x_int8(o["x"].data_ptr(), M_, K_,
                                               None if o["signs"] is None else o["signs"].data_ptr(),
                                               args.prepared, o["xq"].data_ptr(), cs)
                    o["h"].run_xq(o["xq"], M_, o["y"], stream=cs)
                else:
                    o["h"].run(o["x"], o["y"], stream=cs)
        graphs.append(g)
    g_dom, g_rest = graphs

    def step():
        g_dom.replay()
        if g_rest is not None:
            g_rest.replay()

    def check_status():
        for o in ops:
            o["h"].status()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    check_status()

    if world > 1:
        torch.distributed.barrier()
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for k in range(K):
            ev[k][0].record(stream)
            g_dom.replay()
            ev[k][1].record(stream)
            if g_rest is not None:
                g_rest.replay()
        end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    total_ms = start.elapsed_time(end)
    dom_ms = sum(a.elapsed_time(b) for a, b in ev)
    check_status()

    # End to end: every step copies all activations in from pinned host
    # memory, runs the same API calls (graph-replayed) and reads the last
    # GEMV's output (the LM head logits for the stack) back to pinned host
    # memory, then synchronizes, as a decode loop that needs its logits would.
    x_dev = [c_x for _, c_x, _ in copies]
    x_host = [t.to("cpu").pin_memory() for t in x_dev]
    y_last = ops[-1]["y"]
    y_host = torch.empty_like(y_last, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in x_host)
    d2h = y_host.numel() * y_host.element_size()
    K_e2e = max(1, min(K, 500))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(K_e2e):
            for d, h in zip(x_dev, x_host):
                d.copy_(h, non_blocking=True)
            step()
            y_host.copy_(y_last, non_blocking=True)
            stream.synchronize()
    e2e_s = time.perf_counter() - t0

    total_ms, dom_ms, e2e_s = max_over_ranks([total_ms, dom_ms, e2e_s], world, device)
    if rank != 0:
        return None

    ms_step = total_ms / K
    value = world * step_bytes / (ms_step * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    dom_launches = len(dom)
    dom_achieved = dom_bytes / (dom_ms / K * 1e-3) / 1e9
    traffic = None
    prof = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(prof):
        try:
            pj = json.load(open(prof))
            entry = pj.get((args.workload if M == 1 else f"{args.workload}/M={M}")
                           + ("/x_int8" if args.x_int8 else ""))
            if entry and entry.get("kernel_source_hash") == kernel_source_hash(entry.get("format"), M):
                traffic = entry.get("dram_bytes_per_launch")
        except Exception:
            traffic = None
    e2e_value = world * step_bytes * K_e2e / e2e_s / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8xint2->int32, f32" if args.x_int8 else "f32",
        "data": "synthetic",
        "config": {"workload": args.workload,
                   "description": desc + (", INT8 activations" if args.x_int8 else "")
                   + ("" if args.prepared is None else
                      ", prepared by qgemv_prepare_x_int8" + (" with Hadamard mixing (1024)" if args.prepared else "")),
                   "M": M, "x_int8": bool(args.x_int8), "prepared_x": args.prepared,
                   "gemvs_per_step": len(ops), "bytes_per_step": step_bytes,
                   "l2": (f"weights larger than 3x L2 ({l2 >> 20} MiB): no flush needed" if R == 1 else
                          f"weights rotate through {R} copies ({R * one_copy / 1e6:.0f} MB > 3x L2 of {l2 >> 20} MiB)"),
                   "parallelism": f"replicas{world}", "peak_hbm_gbs": peak,
                   "frac_of_peak": round(value / world / peak, 4)},
        "roofline": {"bound": "hbm",
                     "kernel": (("wstream_kernel<FmtPQ2I8, MB>, MB = 2, 1 rows per launch" if M < 4 else
                                 f"wstream_mma_kernel<FmtPQ2Q8, NB={1 if M <= 8 else 2}> (f16 MMA on INT8 codes)")
                                if args.x_int8
                                else "aqlm1x16_kernel (codebook entries gathered from L2: a 32-byte sector "
                                     "per group of 8 weights bounds it before HBM does)" if dominant == "aqlm_1x16"
                                else "wstream_kernel<FmtCBK4R, MB>, MB = 8, 2, 1 activation rows per launch"
                                if dominant == "cbk4_row"
                                else "rowcb8_kernel<MB> (one warp per row, its codebook in shared memory)"
                                if dominant == "cbk8_row"
                                else "wstream_kernel<FmtPQ2, 1, GLU> (gate and up interleaved, SiLU(gate)*up stored)"
                                if dominant == "pq2_0_glu"
                                else f"aqlm_table_kernel<MB={M}>" if dominant == "aqlm_2x8" and M <= 2
                                else (f"wstream_kernel<{dominant}, M=1>"
                                      + (" and rowgroup_stream_kernel (matrices of at most one 32-row group per SM)"
                                         if dominant in ("cbk4", "cbk8") else "")) if M == 1
                                else f"wstream_mma_kernel<{dominant}, NB={1 if M <= 8 else 2}>"),
                     "achieved": round(dom_achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(dom_achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": traffic,
                     "bytes_per_launch": dom_bytes / max(1, dom_launches),
                     "avg_launch_us": round(dom_ms / K / max(1, dom_launches) * 1e3, 3)},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": K_e2e},
        # one launch per GEMV (AQLM: one table pass for M <= 2, else the
        # tensor-core kernel; the fused SiLU(gate)*up one for every M); the
        # INT8 path with several rows adds its activation prologue; CBK4_ROW
        # launches once per 8, 2 or 1 rows
        "gpu_launches": sum((x_int8_launches(M, "xq" in o) + (1 if "xq" in o else 0)) if o.get("x_int8") else
                            (M // 8 + (M % 8) // 2 + M % 2) if o["fmt"] == "cbk4_row" else
                            1 for o in ops) * K,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args.workload, M, budget_s=args.cpu_seconds, x_int8=args.x_int8,
                                            prepared=args.prepared)
    return line


# ---------------------------------------------------- oracle (CPU) arm ----

def oracle_sample(workload, M, rows, seed=0):
    """Host inputs for `rows` rows of the workload's first dominant matrix."""
    from bit_weight_only_gb300 import inputs
    specs_fn, dominant, _ = WORKLOADS[workload]
    fmt, name, N, K = next(s for s in specs_fn() if s[0] == dominant)
    rows = min(rows, total_rows(N))
    g = inputs.rng(f"cpu/{name}", seed)
    scales = cb = None
    if fmt == "cbk4":
        cb = inputs.cbk_centroids(16)
        packed = inputs.cbk_packed(g, rows, K, 4, inputs.cbk_cell_probs(cb))
    elif fmt == "cbk8":
        cb = inputs.cbk_centroids(256)
        packed = inputs.cbk_packed(g, rows, K, 8, inputs.cbk_cell_probs(cb))
    elif fmt == "pq2_0":
        packed = inputs.pq2_packed(g, rows, K)
    elif fmt == "pq2_0_glu":  # (gate, up)
        packed = (inputs.pq2_packed(g, rows, K), inputs.pq2_packed(g, rows, K))
    elif fmt == "q4_0":
        packed = inputs.q4_0_random_blocks(g, rows, K)
    elif fmt == "aqlm_1x16":
        packed, scales, cb = inputs.aqlm_1x16_inputs(g, rows, K)
    elif fmt == "cbk4_row":
        packed = inputs.cbk_packed(g, rows, K, 4, inputs.cbk_cell_probs(inputs.cbk_centroids(16)))
        cb = inputs.cbk_row_codebooks(g, rows)
    elif fmt == "cbk8_row":
        packed = inputs.cbk_packed(g, rows, K, 8, inputs.cbk_cell_probs(inputs.cbk_centroids(256)))
        cb = inputs.cbk_row_codebooks(g, rows, L=256)
    else:
        packed, scales, cb = inputs.aqlm_inputs(g, rows, K)
    x = inputs.x_fp16(inputs.rng("cpu/x", seed), M, K)
    pbytes = sum(a.nbytes for a in packed) if isinstance(packed, tuple) else packed.nbytes
    nbytes = (pbytes + (0 if scales is None else scales.nbytes)
              + (0 if cb is None else cb.nbytes) + x.nbytes + 4 * M * rows)
    return fmt, name, rows, K, packed, scales, cb, x, nbytes


def time_oracle(workload, M, rows, threads, reps=1, x_int8=False, prepared=None):
    import oracle
    fmt, name, rows, K, packed, scales, cb, x, nbytes = oracle_sample(workload, M, rows)
    int8 = x_int8 and fmt == "pq2_0"
    signs = np.random.default_rng(0).choice([-1, 1], size=K).astype(np.int8) if prepared else None
    t0 = time.perf_counter()
    for _ in range(reps):
        if fmt == "pq2_0_glu":
            oracle.gemv_glu("pq2_0", rows, K, packed[0], packed[1], x, nthreads=threads)
        elif int8 and prepared is not None:
            q, a = oracle.prepare_x_int8(x, prepared, signs)
            oracle.gemv_pq2_int8_q(rows, K, packed, q, a, nthreads=threads)
        elif int8:
            oracle.gemv_pq2_int8(rows, K, packed, x, nthreads=threads)
        else:
            oracle.gemv(fmt, rows, K, packed, scales, cb, x, nthreads=threads)
    dt = time.perf_counter() - t0
    return dt, nbytes * reps, (f"{reps} x {rows} rows of {name} ({fmt}{', INT8 activations' if int8 else ''}, "
                               f"K={K}), M={M}")


def cpu_baseline(workload, M, budget_s=15.0, x_int8=False, prepared=None):
    """The oracle as it stands on the host cores, on a bounded sample (about
    budget_s seconds of work: repeated passes over rows of the workload's
    first matrix)."""
    threads = os.cpu_count() or 1
    rows, reps = 256, 1
    dt, nbytes, desc = time_oracle(workload, M, rows, threads, reps, x_int8, prepared)
    while dt < budget_s / 2:
        if rows < 4096:
            rows *= 4
        else:
            reps = max(reps * 2, int(reps * budget_s / max(dt, 1e-3) * 0.6))
        dt, nbytes, desc = time_oracle(workload, M, rows, threads, reps, x_int8, prepared)
    return {"value": round(nbytes / dt / 1e9, 4), "unit": UNIT, "cores": threads,
            "kind": "oracle", "sample": desc, "seconds": round(dt, 3)}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    threads = os.cpu_count() or 1
    total_budget = args.cpu_seconds * 4
    per_step = max(0.05, total_budget / max(1, args.steps + args.warmup))
    rows = 64
    i8, pr = args.x_int8, args.prepared
    dt, nbytes, desc = time_oracle(args.workload, args.m, rows, threads, x_int8=i8, prepared=pr)
    while dt < per_step / 2 and rows < 65536:
        rows *= 2
        dt, nbytes, desc = time_oracle(args.workload, args.m, rows, threads, x_int8=i8, prepared=pr)
    for _ in range(args.warmup):
        time_oracle(args.workload, args.m, rows, threads, x_int8=i8, prepared=pr)
    times = []
    for _ in range(args.steps):
        dt, nbytes, desc = time_oracle(args.workload, args.m, rows, threads, x_int8=i8, prepared=pr)
        times.append(dt)
    tot = sum(times)
    value = nbytes * len(times) / tot / 1e9
    specs_fn, dominant, wdesc = WORKLOADS[args.workload]
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / len(times) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "description": wdesc + (", INT8 activations" if i8 else ""),
                   "M": args.m, "x_int8": bool(i8), "prepared_x": pr, "parallelism": f"replicas{world}"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ main --

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="cbk4_7b_stack")
    ap.add_argument("--m", type=int, default=1)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--x-int8", action="store_true",
                    help="PQ2_0 workloads: INT8 activations (the integer path, lossy by design)")
    ap.add_argument("--prepared", type=int, choices=[0, 1024], default=None,
                    help="with --x-int8: run the activation prologue (qgemv_prepare_x_int8, Hadamard "
                         "block 0 or 1024) and the GEMV on its codes (qgemv_run_xq) in every step")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.x_int8 and WORKLOADS[args.workload][1] != "pq2_0":
        ap.error("--x-int8 needs a PQ2_0 workload")
    if args.prepared is not None and not args.x_int8:
        ap.error("--prepared needs --x-int8")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    line = run_ours(args, rank, world, device)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
