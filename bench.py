"""Benchmark of the FP8 W8A8 rollout hot path on GB300.

One step = one pass of every hot-path operation over one batch of synthetic
input, with all inputs resident in HBM:

  1. weight sync: 128x128 blockwise E4M3 quantization of all 36 Qwen3-8B
     layers (qkv [6144,4096], o [4096,4096], gate_up [24576,4096],
     down [4096,12288]; 6.95e9 weights) -- one batched launch;
  2. Qwen3-8B prefill linears at M = 8192 tokens: 1x128 activation
     quantization, then the blockwise FP8 GEMM, for each of the 4 linears
     (weights from step 1, layer 0);
  3. one Qwen3-30B-A3B MoE layer: 4096 tokens routed top-8 over 128 experts;
     activation quantization straight into the 32768 routed rows (the
     gather fused into the quantizer), grouped gate_up GEMM, quantization of
     the [32768, 768] down input, grouped down GEMM;
  4. KV-cache recalibration: per-tensor amax + E4M3 quantization of K and V,
     each [32, 8192, 8, 128];
  5. decode-sized Qwen3-8B linears at M = 64 and at M = 256 tokens: for each
     of the 36 layers and each of its 4 linears, the W8A8 linear from BF16
     activations (1x128 activation quantization, then the blockwise FP8 GEMM
     with the layer's weights from step 1, chained as programmatic
     dependents).  6.3 GB of FP8 weights per pass,
     so every pass streams them from HBM; each pass is one CUDA-graph replay,
     the linears marked as reading static weights.

Metric: each phase is measured against its roofline time
t_roof = max(flops / peak_fp8, bytes / peak_hbm) with algorithmic bytes and
flops; `value` = 100 * (roofline time of the work all ranks did) / (wall time
of the slowest rank), i.e. percent of one GB300's roofline, summed over GPUs.
The two named sub-metrics (GEMM TFLOP/s, quantizer GB/s) are reported too.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "blockwise-FP8 GEMM TFLOP/s and FP8 quantize GB/s, as % of GB300 roofline"
UNIT = "% of GB300 roofline (sum over GPUs)"
WORKLOAD = ("qwen3-8b weight sync (36 layers, 128x128 blockwise E4M3) + qwen3-8b W8A8 linears "
            "at M=8192 + qwen3-30b-a3b MoE layer (4096 tok, 128 experts, top-8) + FP8 KV "
            "recalibration K,V [32,8192,8,128] + qwen3-8b W8A8 decode linears at M=64 and "
            "M=256 over all 36 layers")
DECODE_MS = (64, 256)

# ------------------------------------------------------------------ peaks

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio, 4.5 / 2.25 PFLOP/s
NOMINAL_FP8_TFLOPS = 4500.0


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


# ------------------------------------------------------- algorithmic work

def cdiv(a, b):
    return (a + b - 1) // b


def work_model():
    """(name, flops, bytes) per phase of one step, from the shapes alone."""
    from w8a8_gemm_rl_gb300 import synth
    ph = []
    # 1. weight sync
    elems = 0
    blocks = 0
    for n, k in synth.QWEN3_8B_LINEARS.values():
        elems += n * k * synth.QWEN3_8B_LAYERS
        blocks += cdiv(n, 128) * cdiv(k, 128) * synth.QWEN3_8B_LAYERS
    ph.append(("weight_quant", 0, 3 * elems + 4 * blocks))
    # 2. linears at M = 8192
    M = 8192
    aq_bytes = gemm_flops = gemm_bytes = 0
    for n, k in synth.QWEN3_8B_LINEARS.values():
        aq_bytes += 3 * M * k + 4 * M * cdiv(k, 128)
        gemm_flops += 2 * M * n * k
        gemm_bytes += M * k + n * k + 4 * (M * cdiv(k, 128) + cdiv(n, 128) * cdiv(k, 128)) + 2 * M * n
    ph.append(("act_quant_linears", 0, aq_bytes))
    ph.append(("gemm_linears", gemm_flops, gemm_bytes))
    # 3. MoE layer
    T, H, E, I, K8 = synth.MOE_TOKENS, synth.MOE_HIDDEN, synth.MOE_EXPERTS, synth.MOE_INTER, synth.MOE_TOPK
    R = T * K8
    moe_q = 3 * T * H + 4 * T * cdiv(H, 128) + 3 * R * I + 4 * R * cdiv(I, 128)
    gu_f = 2 * R * (2 * I) * H
    gu_b = E * 2 * I * H + 4 * E * cdiv(2 * I, 128) * cdiv(H, 128) + T * H + 4 * T * cdiv(H, 128) + 4 * R + 2 * R * 2 * I
    dn_f = 2 * R * H * I
    dn_b = E * H * I + 4 * E * cdiv(H, 128) * cdiv(I, 128) + R * I + 4 * R * cdiv(I, 128) + 2 * R * H
    ph.append(("act_quant_moe", 0, moe_q))
    ph.append(("grouped_gemm_moe", gu_f + dn_f, gu_b + dn_b))
    # 4. KV recalibration: amax pass (2 B/elem) then code pass (2 + 1 B/elem), K and V
    kv = int(np.prod(synth.KV_SHAPE))
    ph.append(("kv_quant", 0, 2 * 5 * kv))
    # 5. decode linears: every layer's 4 linears at M tokens, act quant + GEMM
    for M in DECODE_MS:
        f = b = 0
        for n, k in synth.QWEN3_8B_LINEARS.values():
            f += 2 * M * n * k
            b += 3 * M * k + 4 * M * cdiv(k, 128)  # act quant
            b += M * k + n * k + 4 * (M * cdiv(k, 128) + cdiv(n, 128) * cdiv(k, 128)) + 2 * M * n
        ph.append((f"decode_m{M}", f * synth.QWEN3_8B_LAYERS, b * synth.QWEN3_8B_LAYERS))
    return ph


def fp8_peak_tflops(peaks):
    """Dense FP8 tensor peak: the measured BF16 burst peak (a cuBLAS GEMM
    timed alone) x the nominal FP8/BF16 ratio.  The step is milliseconds
    long, so the burst figure applies rather than the sustained one."""
    return FP8_OVER_BF16 * peaks["bf16_tflops"]


def t_roof(flops, nbytes, peaks):
    return max(flops / (fp8_peak_tflops(peaks) * 1e12), nbytes / (peaks["hbm_gbs"] * 1e9))


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples during the timed region (read-only queries)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- our arm

class Workload:
    """Device-resident inputs and outputs of one step."""

    def __init__(self, dev, seed_base=0):
        from w8a8_gemm_rl_gb300 import synth
        self.synth = synth
        S = seed_base
        L = synth.QWEN3_8B_LAYERS
        self.w = []
        for l in range(L):
            for j, (n, k) in enumerate(synth.QWEN3_8B_LINEARS.values()):
                self.w.append(synth.weights(n, k, seed=S + 1000 * l + j, device=dev))
        self.wout = [(torch.empty(w.shape, dtype=torch.uint8, device=dev),
                      torch.empty((cdiv(w.shape[0], 128), cdiv(w.shape[1], 128)), dtype=torch.float32, device=dev))
                     for w in self.w]
        M = 8192
        self.lin = []
        for j, (n, k) in enumerate(synth.QWEN3_8B_LINEARS.values()):
            x = synth.activations(M, k, seed=S + 50 + j, device=dev)
            self.lin.append(dict(x=x, xq=torch.empty((M, k), dtype=torch.uint8, device=dev),
                                 xs=torch.empty((M, cdiv(k, 128)), dtype=torch.float32, device=dev),
                                 wq=self.wout[j][0], ws=self.wout[j][1],
                                 y=torch.empty((M, n), dtype=torch.bfloat16, device=dev)))
        T, H, E, I, K8 = synth.MOE_TOKENS, synth.MOE_HIDDEN, synth.MOE_EXPERTS, synth.MOE_INTER, synth.MOE_TOPK
        r = synth.moe_routing(T, E, K8, seed=S + 60, device="cpu")
        self.total = T * K8
        self.row_idx = r.row_idx.to(dev)
        self.off = r.group_offsets.to(dev)
        self.moe_x = synth.activations(T, H, seed=S + 61, device=dev)
        self.moe_d = synth.activations(self.total, I, seed=S + 62, device=dev)
        # expert weights, blockwise FP8 (quantized once here: the MoE phase
        # measures the grouped GEMMs; weight quantization is phase 1)
        import w8a8_gemm_rl_gb300 as W
        self.gu_q = torch.empty((E, 2 * I, H), dtype=torch.uint8, device=dev)
        self.gu_s = torch.empty((E, cdiv(2 * I, 128), cdiv(H, 128)), dtype=torch.float32, device=dev)
        self.dn_q = torch.empty((E, H, I), dtype=torch.uint8, device=dev)
        self.dn_s = torch.empty((E, cdiv(H, 128), cdiv(I, 128)), dtype=torch.float32, device=dev)
        gu = synth.weights(E * 2 * I, H, seed=S + 63, device=dev)
        dn = synth.weights(E * H, I, seed=S + 64, device=dev)
        for e in range(E):
            W.quantize_weight_blockwise(gu[e * 2 * I:(e + 1) * 2 * I], self.gu_q[e], self.gu_s[e])
            W.quantize_weight_blockwise(dn[e * H:(e + 1) * H], self.dn_q[e], self.dn_s[e])
        del gu, dn
        # the gate_up input, quantized directly in routed (expert-sorted) order
        self.mx_q = torch.empty((self.total, H), dtype=torch.uint8, device=dev)
        self.mx_s = torch.empty((self.total, cdiv(H, 128)), dtype=torch.float32, device=dev)
        self.md_q = torch.empty((self.total, I), dtype=torch.uint8, device=dev)
        self.md_s = torch.empty((self.total, cdiv(I, 128)), dtype=torch.float32, device=dev)
        self.y_gu = torch.empty((self.total, 2 * I), dtype=torch.bfloat16, device=dev)
        self.y_dn = torch.empty((self.total, H), dtype=torch.bfloat16, device=dev)
        self.kv = [synth.kv_cache(seed=S + 70 + i, device=dev) for i in range(2)]
        self.kv_q = [torch.empty(t.shape, dtype=torch.uint8, device=dev) for t in self.kv]
        self.kv_s = [torch.empty(1, dtype=torch.float32, device=dev) for _ in self.kv]
        self.kv_a = [torch.empty(1, dtype=torch.float32, device=dev) for _ in self.kv]
        # decode linears: one activation per (M, linear), shared by the layers
        self.dec = {}
        for M in DECODE_MS:
            rows = []
            for j, (n, k) in enumerate(synth.QWEN3_8B_LINEARS.values()):
                rows.append(dict(x=synth.activations(M, k, seed=S + 80 + 10 * j + M, device=dev),
                                 xq=torch.empty((M, k), dtype=torch.uint8, device=dev),
                                 xs=torch.empty((M, cdiv(k, 128)), dtype=torch.float32, device=dev),
                                 y=torch.empty((M, n), dtype=torch.bfloat16, device=dev)))
            self.dec[M] = rows
        self.graphs = {}
        torch.cuda.synchronize()

    def decode_pass(self, W, M):
        """All 36 layers' 4 linears at M tokens, each the W8A8 linear from
        BF16 activations (w8a8_linear): the activation quantizer, then the
        GEMM, chained as programmatic dependents."""
        nlin = len(self.synth.QWEN3_8B_LINEARS)
        for l in range(self.synth.QWEN3_8B_LAYERS):
            for j, d in enumerate(self.dec[M]):
                wq, ws = self.wout[nlin * l + j]
                W.w8a8_linear(d["x"], wq, ws, d["y"], d["xq"], d["xs"], static_weights=True)

    def capture_decode(self, W):
        """One CUDA graph per decode pass (captured once, replayed per step)."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for M in DECODE_MS:
                self.decode_pass(W, M)
            torch.cuda.synchronize()
            for M in DECODE_MS:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    self.decode_pass(W, M)
                self.graphs[M] = g
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()

    def input_tensors(self):
        return ([*self.w] + [d["x"] for d in self.lin] + [self.moe_x, self.moe_d, self.row_idx, self.off]
                + list(self.kv) + [d["x"] for M in DECODE_MS for d in self.dec[M]])

    def output_tensors(self):
        outs = []
        for q, s in self.wout:
            outs += [q, s]
        for d in self.lin:
            outs += [d["y"]]
        outs += [self.y_gu, self.y_dn]
        outs += self.kv_q + self.kv_s + self.kv_a
        outs += [d["y"] for M in DECODE_MS for d in self.dec[M]]
        return outs


# weight batch (144 matrices), 4 x (act quant + GEMM), MoE 4, KV 2 x 2, and
# per decode pass 36 layers x 4 linears x (act quant + GEMM)
LAUNCHES_PER_STEP = 1 + 4 * 2 + 4 + 2 * 2 + len(DECODE_MS) * 36 * 4 * 2


def run_step(W, wl, events=None, skip_weights=False):
    """Queue one step on the current stream; events (if given) bracket phases.
    skip_weights: the weight sync was queued by the caller (in slices)."""
    def mark(i):
        if events is not None:
            events[i].record()
    mark(0)
    if not skip_weights:
        W.quantize_weight_blockwise_batched(wl.w, wl.wout)
    mark(1)
    for d in wl.lin:
        W.quantize_act_per_token_group(d["x"], d["xq"], d["xs"])
    mark(2)
    for d in wl.lin:
        W.fp8_block_gemm(d["xq"], d["xs"], d["wq"], d["ws"], d["y"])
    mark(3)
    # the routed-row gather rides on the activation quantizer, so the
    # grouped GEMMs read contiguous rows (the same result as quantizing x and
    # gathering inside the GEMM: quantization works per row)
    W.quantize_act_per_token_group_gather(wl.moe_x, wl.row_idx, wl.mx_q, wl.mx_s)
    W.quantize_act_per_token_group(wl.moe_d, wl.md_q, wl.md_s)
    mark(4)
    W.fp8_grouped_gemm(wl.mx_q, wl.mx_s, None, wl.off, wl.total, wl.gu_q, wl.gu_s, wl.y_gu)
    W.fp8_grouped_gemm(wl.md_q, wl.md_s, None, wl.off, wl.total, wl.dn_q, wl.dn_s, wl.y_dn)
    mark(5)
    for i in range(2):
        W.kv_amax_quantize(wl.kv[i], wl.kv_q[i], wl.kv_s[i], wl.kv_a[i])
    mark(6)
    for i, M in enumerate(DECODE_MS):
        wl.graphs[M].replay()
        mark(7 + i)


PHASE_ORDER = ["weight_quant", "act_quant_linears", "gemm_linears", "act_quant_moe", "grouped_gemm_moe",
               "kv_quant"] + [f"decode_m{M}" for M in DECODE_MS]


def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# DRAM bytes (read + written) of one launch of the batched weight quantizer
# (144 matrices), from an ncu capture of the same kernel on one Qwen3-8B
# layer's 4 matrices, repeated launches with ncu's cache control off (so a
# launch's writes include the codes the previous one left dirty in L2, and
# a read-only flush after the last launch shows what it left), scaled by the
# 36 layers (traffic grows with the elements).  Keyed by a hash of the
# kernel's sources: any change to them makes the figure stale, and it is
# then reported as null.
WEIGHT_QUANT_SOURCES = ("quant.cu", "common.cuh", "ptx.cuh", "tmap.h")
WEIGHT_QUANT_TRAFFIC = {
    # profiles/weight_quant_batched_qwen3_8b_layer.md: 36 x (385.9 + 192.3) MB
    "831b98e3d9eef423": 36 * (385895168 + 192344832),
}


def weight_quant_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in WEIGHT_QUANT_SOURCES:
        with open(os.path.join(ROOT, "w8a8_gemm_rl_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def weight_quant_traffic(args):
    if args.traffic is not None:
        return args.traffic
    return WEIGHT_QUANT_TRAFFIC.get(weight_quant_source_hash())


def job_value(ms_total_local, steps, roof_step_s, world):
    """Whole-job result of a timed region: the slowest rank's wall time
    (max over ranks) and `value` = 100 * (roofline time of the work all
    ranks did) / that wall time.  Every rank gets the same numbers."""
    ms_total = max_over_ranks(ms_total_local, world)
    ms_step = ms_total / steps
    value = 100.0 * world * roof_step_s / (ms_step * 1e-3)
    return ms_total, ms_step, value


# ------------------------------------------------------------ CPU baseline
#
# The CPU oracle as it stands, on a fixed, bounded sample of the step's
# phases.  The sample is a number of identical-sized units; a unit holds a
# strip of each phase's work (below), and the units are spread over one
# process per host core (spawned, so no process is forked after the GPU is
# in use).  The same sample is timed by --impl reference.

CPU_UNIT_PARTS = (
    "weight quant 256x4096 (o projection strip)",
    "act quant 256x4096",
    "dense GEMM 1024 outputs of the qkv linear (K=4096)",
    "grouped GEMM 512 outputs of the MoE gate_up (K=2048)",
    "KV amax + quant 262144 elements",
)
_CPU_UNIT = None


def _cpu_unit_init():
    """Inputs of the CPU sample's units, generated once per process."""
    global _CPU_UNIT
    import oracle as O
    from w8a8_gemm_rl_gb300 import synth
    O.lib()
    w = synth.bf16_bits(synth.weights(4096, 4096, seed=1))
    x = synth.bf16_bits(synth.activations(1024, 4096, seed=2))
    xq, xs = O.quantize_act_per_token_group(x[:64])
    wq, ws = O.quantize_weight_blockwise(w[:256])
    gx = synth.bf16_bits(synth.activations(64, 2048, seed=4))
    gw = synth.bf16_bits(synth.weights(256, 2048, seed=5))
    gxq, gxs = O.quantize_act_per_token_group(gx)
    gwq, gws = O.quantize_weight_blockwise(gw)
    kv = synth.bf16_bits(synth.kv_cache(seed=3, shape=(1, 256, 8, 128)))
    _CPU_UNIT = dict(w=w, x=x, g=(xq, xs, wq, ws), gg=(gxq, gxs, gwq, gws), kv=kv)


def _cpu_unit_run(i):
    """One unit of the CPU sample (index i picks the strips); returns its
    wall time in seconds."""
    import oracle as O
    if _CPU_UNIT is None:
        _cpu_unit_init()
    u = _CPU_UNIT
    rng = np.random.default_rng(i)
    t0 = time.perf_counter()
    r = 256 * (i % 16)
    O.quantize_weight_blockwise(u["w"][r:r + 256])
    r = 256 * (i % 4)
    O.quantize_act_per_token_group(u["x"][r:r + 256])
    O.block_gemm_entries(*u["g"], rng.integers(0, 64, 1024), rng.integers(0, 256, 1024))
    O.block_gemm_entries(*u["gg"], rng.integers(0, 64, 512), rng.integers(0, 256, 512))
    O.kv_amax_quantize(u["kv"])
    return time.perf_counter() - t0


def cpu_unit_roofline_s(peaks):
    """GB300 roofline time of one unit's work (same accounting as the step)."""
    return (t_roof(0, 3 * 256 * 4096 + 4 * 2 * 32, peaks)
            + t_roof(0, 3 * 256 * 4096 + 4 * 256 * 32, peaks)
            + t_roof(2 * 1024 * 4096, 0, peaks)
            + t_roof(2 * 512 * 2048, 0, peaks)
            + t_roof(0, 5 * 256 * 8 * 128, peaks))


def host_cpu_info():
    """(logical cores usable by this process, CPU model string)."""
    try:
        cores = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        cores = os.cpu_count() or 1
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith("model name"):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    if model is None:
        import platform
        model = platform.machine()
    return cores, model


class CpuSample:
    """The CPU oracle on a fixed sample of `units_per_core` units per host
    core, timed on all cores (one spawned process each) and on one core."""

    def __init__(self, units_per_core=4):
        import multiprocessing as mp
        self.cores, self.model = host_cpu_info()
        self.units = units_per_core * self.cores
        self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_cpu_unit_init)
        # every worker has built its inputs before anything is timed
        self.pool.map(_cpu_unit_run, range(self.cores), chunksize=1)
        _cpu_unit_init()

    def run_all_cores(self):
        t0 = time.perf_counter()
        self.pool.map(_cpu_unit_run, range(self.units), chunksize=1)
        return time.perf_counter() - t0

    def run_one_core(self, units=2):
        return sum(_cpu_unit_run(i) for i in range(units)) / units

    def close(self):
        self.pool.close()
        self.pool.join()

    def describe(self):
        return (f"{self.units} units ({self.cores} cores x {self.units // self.cores}); "
                f"a unit = " + "; ".join(CPU_UNIT_PARTS))


def cpu_baseline_oracle(reps=1):
    """The CPU oracle on the fixed sample: percent of one GB300's roofline
    that the host's cores reach, with the single-core figure beside it."""
    peaks = load_peaks()
    smp = CpuSample()
    try:
        unit_roof = cpu_unit_roofline_s(peaks)
        wall = min(smp.run_all_cores() for _ in range(reps))
        one = smp.run_one_core()
    finally:
        smp.close()
    value = 100.0 * smp.units * unit_roof / wall
    info = {"kind": "oracle", "cores": smp.cores, "cpu_model": smp.model,
            "seconds": round(wall, 2), "cpu_seconds": round(wall * smp.cores, 1),
            "value_1core": round(100.0 * unit_roof / one, 6),
            "sample": smp.describe() + " (C oracle as it stands, one process per core)"}
    return value, info


def bench_ours(args):
    rank, world, local = dist_setup(args.gpus)
    import w8a8_gemm_rl_gb300 as W
    from w8a8_gemm_rl_gb300 import _build
    if rank == 0 or not os.path.exists(W.LIB_PATH):
        _build.build()
    barrier(world)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    wl = Workload(dev, seed_base=0)
    stream = torch.cuda.current_stream()
    W.quantize_weight_blockwise_batched(wl.w, wl.wout)  # the decode passes read these codes
    wl.capture_decode(W)
    for _ in range(args.warmup):
        run_step(W, wl)
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    # timed region: K steps, phase events in every step
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(PHASE_ORDER) + 1)]
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for s in range(args.steps):
        run_step(W, wl, ev[s])
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms_total_local = start.elapsed_time(end)
    phase_ms = {name: 0.0 for name in PHASE_ORDER}
    for s in range(args.steps):
        for i, name in enumerate(PHASE_ORDER):
            phase_ms[name] += ev[s][i].elapsed_time(ev[s][i + 1]) / args.steps
    assert W.consume_device_error() == 0

    model = {name: (f, b) for name, f, b in work_model()}
    roof_step = sum(t_roof(f, b, peaks) for f, b in model.values())
    ms_total, ms_step, value = job_value(ms_total_local, args.steps, roof_step, world)
    phases = {}
    for name in PHASE_ORDER:
        f, b = model[name]
        t = phase_ms[name] * 1e-3
        d = {"ms": round(phase_ms[name], 4), "pct_roofline": round(100 * t_roof(f, b, peaks) / t, 2)}
        if f:
            d["tflops"] = round(f / t / 1e12, 1)
        d["gbs"] = round(b / t / 1e9, 1)
        phases[name] = d
    q_bytes = sum(model[n][1] for n in PHASE_ORDER if "quant" in n)
    q_ms = sum(phase_ms[n] for n in PHASE_ORDER if "quant" in n)
    g_flops = sum(model[n][0] for n in PHASE_ORDER if "gemm" in n)
    g_ms = sum(phase_ms[n] for n in PHASE_ORDER if "gemm" in n)
    # dominant kernel: the batched weight quantizer (one launch per step)
    dom = "weight_quant"
    dom_t = phase_ms[dom] * 1e-3
    achieved = model[dom][1] / dom_t / 1e9
    roofline = {"kernel": "weight_quant_kernel (batched, 1 launch = 144 matrices)", "bound": "hbm",
                "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"],
                "traffic": weight_quant_traffic(args)}
    gemm_roof = {"kernel": "fp8_gemm_kernel<DENSE> (4 launches, M=8192)", "bound": "tensor",
                 "achieved": round(model["gemm_linears"][0] / (phase_ms["gemm_linears"] * 1e-3) / 1e12, 1),
                 "peak": round(fp8_peak_tflops(peaks), 1), "unit": "TFLOP/s",
                 "peak_note": "measured bf16 burst x 2 (nominal fp8/bf16 ratio)",
                 "peak_nominal": NOMINAL_FP8_TFLOPS,
                 "peak_nominal_note": "GB300 dense FP8, vendor figure"}
    gemm_roof["frac"] = round(gemm_roof["achieved"] / gemm_roof["peak"], 4)
    gemm_roof["frac_nominal"] = round(gemm_roof["achieved"] / NOMINAL_FP8_TFLOPS, 4)
    decode_gemm = measure_decode_gemm_only(W, wl, peaks)

    next_rows = None if args.no_next_rows else measure_next_rows(W, wl, peaks)
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(W, wl, args, roof_step, world)
    cpu = None
    if rank == 0 and world >= 1 and not args.no_cpu_baseline and world == 1:
        v, info = cpu_baseline_oracle()
        cpu = dict(info, value=round(v, 4), unit=UNIT)
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded; shapes and distributions of the Qwen3-8B / Qwen3-30B-A3B workloads)",
        "config": {"workload": WORKLOAD, "l2": "inputs larger than L2 (~30 GB streamed per step)",
                   "parallelism": f"replica per GPU x{world} (no data-path collective)"},
        "quant_gbs": round(q_bytes / (q_ms * 1e-3) / 1e9 * world, 1),
        "gemm_tflops": round(g_flops / (g_ms * 1e-3) / 1e12 * world, 1),
        "phases": phases, "roofline": roofline, "gemm_roofline": gemm_roof,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": clk, "peaks": peaks, "next_rows": next_rows, "decode_gemm_only": decode_gemm,
    }
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measure_decode_gemm_only(W, wl, peaks, reps=5):
    """The decode passes' GEMMs alone (activations quantized once before):
    one CUDA graph per M of the 144 GEMMs, timed after the timed region, on
    the GEMMs' own roofline (weight, activation and output bytes)."""
    from w8a8_gemm_rl_gb300 import synth
    out = {}
    nlin = len(synth.QWEN3_8B_LINEARS)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    for M in DECODE_MS:
        for d in wl.dec[M]:
            W.quantize_act_per_token_group(d["x"], d["xq"], d["xs"])

        def gemms():
            for l in range(synth.QWEN3_8B_LAYERS):
                for j, d in enumerate(wl.dec[M]):
                    wq, ws = wl.wout[nlin * l + j]
                    W.fp8_block_gemm(d["xq"], d["xs"], wq, ws, d["y"], static_weights=True)
        with torch.cuda.stream(side):
            gemms()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                gemms()
        torch.cuda.current_stream().wait_stream(side)
        g.replay()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(reps):
            g.replay()
        t1.record()
        torch.cuda.synchronize()
        sec = t0.elapsed_time(t1) * 1e-3 / reps
        per = {}
        f = b = 0
        for name, (n, k) in synth.QWEN3_8B_LINEARS.items():
            fl = 2 * M * n * k
            by = M * k + n * k + 4 * (M * cdiv(k, 128) + cdiv(n, 128) * cdiv(k, 128)) + 2 * M * n
            f += fl
            b += by
            per[name] = round(1e6 * t_roof(fl, by, peaks), 2)
        f *= synth.QWEN3_8B_LAYERS
        b *= synth.QWEN3_8B_LAYERS
        out[f"m{M}"] = {"workload": f"36 layers x 4 linears at M={M}, one graph of 144 GEMMs",
                        "ms": round(sec * 1e3, 4), "us_per_gemm": round(sec * 1e6 / 144, 2),
                        "pct_roofline": round(100 * t_roof(f, b, peaks) / sec, 2),
                        "gbs": round(b / sec / 1e9, 1), "roofline_us_per_linear": per}
        if M <= 128:
            # the same decode pass with each linear as ONE kernel (the
            # quantization fused into the GEMM) instead of quantizer + GEMM
            def single():
                for l in range(synth.QWEN3_8B_LAYERS):
                    for j, d in enumerate(wl.dec[M]):
                        wq, ws = wl.wout[nlin * l + j]
                        W.w8a8_linear(d["x"], wq, ws, d["y"], static_weights=True, single_kernel=True)
            with torch.cuda.stream(side):
                single()
                torch.cuda.synchronize()
                g1 = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g1, stream=side):
                    single()
            torch.cuda.current_stream().wait_stream(side)
            g1.replay()
            torch.cuda.synchronize()
            t0.record()
            for _ in range(reps):
                g1.replay()
            t1.record()
            torch.cuda.synchronize()
            out[f"m{M}"]["single_kernel_linear_ms"] = round(t0.elapsed_time(t1) / reps, 4)
            out[f"m{M}"]["single_kernel_note"] = (
                "the decode pass with each linear as one kernel quantizing its own token rows "
                "(every 128-column weight tile repeats the quantization); the phase runs "
                "quantizer + GEMM instead")
    assert W.consume_device_error() == 0
    return out


def measure_next_rows(W, wl, peaks, reps=3):
    """Rows past the hot path, each on its own kernel roofline (HBM): the
    power-of-two-scale weight quantizer, the dequantizer (fake quant) over
    every weight matrix of the model from its 128x128-block codes, and the
    quantization-error report over the same matrices (128x128 report
    blocks) -- each one batched launch over all 144 matrices, inputs (20 GB)
    far larger than L2 -- and the decode attention over the step's FP8 KV
    cache; CUDA events around each sweep."""
    out = {}
    elems = sum(w.numel() for w in wl.w)
    blocks = sum(cdiv(w.shape[0], 128) * cdiv(w.shape[1], 128) for w in wl.w)
    dev = wl.w[0].device
    yall = torch.empty(elems, dtype=torch.bfloat16, device=dev)
    sall = torch.empty(blocks * 3, dtype=torch.float64, device=dev)
    ys, sts = [], []
    eo = bo = 0
    for w in wl.w:
        n, k = w.shape
        ys.append(yall[eo:eo + n * k].view(n, k))
        nb = cdiv(n, 128) * cdiv(k, 128)
        sts.append(sall[bo:bo + 3 * nb].view(cdiv(n, 128), cdiv(k, 128), 3))
        eo += n * k
        bo += 3 * nb
    qs = [q for q, _ in wl.wout]
    ss = [sc for _, sc in wl.wout]

    def sweep(kind):
        if kind == "dequant":
            W.dequantize_blockwise_batched(qs, ss, ys)
        else:
            W.quant_error_report_batched(wl.w, qs, ss, sts)

    # power-of-two scales: the same weight sync as the step, one batched launch
    def pow2_sweep():
        W.quantize_weight_blockwise_batched(wl.w, wl.wout, pow2=True)
    pow2_sweep()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(reps):
        pow2_sweep()
    t1.record()
    torch.cuda.synchronize()
    sec = t0.elapsed_time(t1) * 1e-3 / reps
    nb = 3 * elems + 4 * blocks
    out["quantize_weight_blockwise_batched_pow2"] = {
        "workload": "all 144 Qwen3-8B weight matrices, 128x128 blocks, 1 batched launch",
        "ms": round(sec * 1e3, 3), "gbs": round(nb / sec / 1e9, 1),
        "pct_roofline": round(100 * nb / sec / 1e9 / peaks["hbm_gbs"], 2), "bytes_per_sweep": nb}
    # decode attention: one query token per sequence (32 query heads) over
    # the step's FP8 KV cache [32, 8192, 8, 128], every token attended
    kq, vq = wl.kv_q
    B, S, Hkv, D = kq.shape
    g = torch.Generator(device=kq.device)
    g.manual_seed(90)
    qa = torch.randint(0, 126, (B, 4 * Hkv, D), dtype=torch.uint8, device=kq.device, generator=g)
    qsc = torch.full((1,), 0.01, dtype=torch.float32, device=kq.device)
    lens = torch.full((B,), S, dtype=torch.int32, device=kq.device)
    att = W.fp8_decode_attention(qa, qsc, kq, wl.kv_s[0], vq, wl.kv_s[1], lens)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(10):
        W.fp8_decode_attention(qa, qsc, kq, wl.kv_s[0], vq, wl.kv_s[1], lens, out=att)
    t1.record()
    torch.cuda.synchronize()
    sec = t0.elapsed_time(t1) * 1e-3 / 10
    nb = 2 * kq.numel() + qa.numel() + 2 * att.numel() + 4 * B
    out["fp8_decode_attention"] = {
        "workload": "32 sequences x 8192 tokens, 32 query heads over 8 KV heads, head dim 128",
        "us": round(sec * 1e6, 1), "gbs": round(nb / sec / 1e9, 1),
        "pct_roofline": round(100 * nb / sec / 1e9 / peaks["hbm_gbs"], 2), "bytes_per_call": nb}
    out["fp8_prefill_attention"] = measure_prefill_attention(W, peaks)
    out["fp8_block_gemm_pow2"] = measure_pow2_gemm(W, wl, peaks, reps)
    out["config1_single_linear"] = measure_single_linear(W, peaks)
    W.quantize_weight_blockwise_batched(wl.w, wl.wout)
    for kind, nbytes in (("dequant", 3 * elems + 4 * blocks),
                         ("quant_error_report", 3 * elems + 4 * blocks + 24 * blocks)):
        sweep(kind)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(reps):
            sweep(kind)
        t1.record()
        torch.cuda.synchronize()
        sec = t0.elapsed_time(t1) * 1e-3 / reps
        name = "dequantize_blockwise_batched" if kind == "dequant" else "quant_error_report_batched"
        out[name] = {"workload": "all 144 Qwen3-8B weight matrices, 128x128 blocks, 1 batched launch",
                     "ms": round(sec * 1e3, 3), "gbs": round(nbytes / sec / 1e9, 1),
                     "pct_roofline": round(100 * nbytes / sec / 1e9 / peaks["hbm_gbs"], 2),
                     "bytes_per_sweep": nbytes}
    del yall, sall
    assert W.consume_device_error() == 0
    return out


def prefill_attention_flops(B, S, Hq, D=128):
    """Causal attention: query token i meets keys 0..i, 2 D FLOPs each for
    Q K^T and for P V."""
    return 4 * D * Hq * B * S * (S + 1) // 2


def measure_prefill_attention(W, peaks, reps=10):
    """Causal prefill attention for a rollout prompt batch on Qwen3-8B's
    attention shape: 4 sequences x 2048 tokens, 32 query heads over 8 KV
    heads, head dim 128; Q, K, V per-tensor-quantized N(0, 1) activations.
    Tensor work (Q K^T on E4M3, P V in f16 with the weights in two parts),
    against the FP8 peak."""
    from w8a8_gemm_rl_gb300 import synth
    B, S, Hq, Hkv = 4, 2048, 32, 8
    x = [synth.activations(B * S * h, 128, seed=95 + i, device="cuda").reshape(B, S, h, 128)
         for i, h in enumerate((Hq, Hkv, Hkv))]
    qkv = [W.kv_amax_quantize(t) for t in x]
    args = (qkv[0][0], qkv[0][1], qkv[1][0], qkv[1][1], qkv[2][0], qkv[2][1])
    att = W.fp8_prefill_attention(*args)
    for _ in range(3):
        W.fp8_prefill_attention(*args, out=att)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(reps):
        W.fp8_prefill_attention(*args, out=att)
    t1.record()
    torch.cuda.synchronize()
    assert W.consume_device_error() == 0
    sec = t0.elapsed_time(t1) * 1e-3 / reps
    f = prefill_attention_flops(B, S, Hq)
    tf = f / sec / 1e12
    return {"workload": "4 sequences x 2048 tokens, causal, 32 query heads over 8 KV heads, "
                        "head dim 128", "us": round(sec * 1e6, 1), "tflops": round(tf, 1),
            "pct_roofline": round(100 * tf / fp8_peak_tflops(peaks), 2), "flops_per_call": f,
            "note": "tcgen05 path: E4M3 Q K^T and two-part f16 P V into tensor memory, "
                    "persistent CTAs over 128-token query blocks"}


def single_linear_work():
    """Algorithmic work of one W8A8 linear of X [128, 512] and W [256, 512]
    (both quantized, then the GEMM): FLOPs and bytes."""
    m, n, k = 128, 256, 512
    q_x = 2 * m * k + m * k + 4 * m * cdiv(k, 128)
    q_w = 2 * n * k + n * k + 4 * cdiv(n, 128) * cdiv(k, 128)
    g = m * k + n * k + 4 * (m * cdiv(k, 128) + cdiv(n, 128) * cdiv(k, 128)) + 2 * m * n
    return 2 * m * n * k, q_x + q_w + g


def measure_single_linear(W, peaks, reps=200):
    """One W8A8 linear at the smallest configuration the pages give, X
    [128, 512] ~ N(0,1) with 0.1% x50 outliers and W [256, 512] ~ N(0, 0.02)
    (seeds 0 and 1): quantize W, quantize X, then the GEMM, as three eager
    launches and as one CUDA-graph replay, and w8a8_linear (one kernel that
    quantizes X on the way into the GEMM, W already quantized).  Latency-bound: microseconds per call
    are the figure; the roofline share is nominal."""
    from w8a8_gemm_rl_gb300 import synth
    m, n, k = 128, 256, 512
    x = synth.activations(m, k, seed=0, device="cuda")
    w = synth.weights(n, k, seed=1, device="cuda")
    xq = torch.empty((m, k), dtype=torch.uint8, device="cuda")
    xs = torch.empty((m, cdiv(k, 128)), dtype=torch.float32, device="cuda")
    wq = torch.empty((n, k), dtype=torch.uint8, device="cuda")
    ws = torch.empty((cdiv(n, 128), cdiv(k, 128)), dtype=torch.float32, device="cuda")
    y = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")

    def three():
        W.quantize_weight_blockwise(w, wq, ws)
        W.quantize_act_per_token_group(x, xq, xs)
        W.fp8_block_gemm(xq, xs, wq, ws, y)

    def linear():
        W.w8a8_linear(x, wq, ws, y)

    def timed(fn):
        for _ in range(10):
            fn()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(reps):
            fn()
        t1.record()
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) * 1e3 / reps

    us_eager = timed(three)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        three()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            three()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    us_graph = timed(graph.replay)
    us_linear = timed(linear)
    assert W.consume_device_error() == 0
    f, b = single_linear_work()
    troof_us = t_roof(f, b, peaks) * 1e6
    return {"workload": "X [128, 512] and W [256, 512], both quantized (1x128, 128x128) then the GEMM",
            "us_three_launches": round(us_eager, 2), "us_graph": round(us_graph, 2),
            "us_w8a8_linear": round(us_linear, 2), "troof_us": round(troof_us, 3),
            "pct_roofline_graph": round(100 * troof_us / us_graph, 2),
            "note": "launch- and latency-bound: the microseconds are the figure"}


def measure_pow2_gemm(W, wl, peaks, reps=3):
    """The power-of-two-scale GEMM (block-scaled MMA) on the four Qwen3-8B
    linears at M=8192, operands quantized with power-of-two scales, timed
    beside the FP32-scale GEMM on the same codes and scales (both compute
    the same product; only the scaling hardware differs)."""
    ops = []
    for j, d in enumerate(wl.lin):
        m, k = d["x"].shape
        xq, xs = W.quantize_act_per_token_group(d["x"], pow2=True)
        wq, ws = W.quantize_weight_blockwise(wl.w[j], pow2=True)
        ops.append((xq, xs, wq, ws, torch.empty_like(d["y"])))
    flops = sum(2 * o[0].shape[0] * o[0].shape[1] * o[2].shape[0] for o in ops)
    res = {"workload": "Qwen3-8B qkv/o/gate_up/down linears at M=8192, power-of-two scales, 4 launches"}
    for name, fn in (("pow2", W.fp8_block_gemm_pow2), ("fp32_scale_kernel", W.fp8_block_gemm)):
        for o in ops:
            fn(*o[:4], y=o[4])
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(reps):
            for o in ops:
                fn(*o[:4], y=o[4])
        t1.record()
        torch.cuda.synchronize()
        sec = t0.elapsed_time(t1) * 1e-3 / reps
        tf = flops / sec / 1e12
        res[name] = {"ms": round(sec * 1e3, 3), "tflops": round(tf, 1),
                     "frac": round(tf / fp8_peak_tflops(peaks), 4)}
    res["peak_tflops"] = round(fp8_peak_tflops(peaks), 1)
    res["peak_note"] = "measured bf16 burst x 2 (nominal fp8/bf16 ratio)"
    assert W.consume_device_error() == 0
    del ops
    return res


def measure_e2e(W, wl, args, roof_step, world, chunks=8, in_streams=1):
    """Same step through the public API with HOST inputs/outputs: every step
    copies its inputs from pinned host memory and its results back.

    The copies run on their own streams (in_streams for host->device, whose
    transfers run concurrently, and one for device->host) and overlap the
    compute: the weight sync goes in `chunks` slices (host->device of slice
    c+1 while slice c is quantized and slice c-1's codes go back), the other
    inputs follow the weights in, and each result leaves as soon as its
    phase ends.  Consecutive steps overlap too: a slice's device buffers
    are refilled only after the previous step has read them (events)."""
    nw = len(wl.w)
    bounds = [nw * c // chunks for c in range(chunks + 1)]
    w_in = list(wl.w)
    w_out = [t for q, s in wl.wout for t in (q, s)]
    rest_in = [t for t in wl.input_tensors() if all(t is not w for w in w_in)]
    rest_out = [t for t in wl.output_tensors() if all(t is not o for o in w_out)]

    def pinned(ts):
        return [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ts]

    h_w_in, h_w_out, h_rest_in, h_rest_out = pinned(w_in), pinned(w_out), pinned(rest_in), pinned(rest_out)
    for h, t in zip(h_w_in + h_rest_in, w_in + rest_in):
        h.copy_(t)
    torch.cuda.synchronize()
    bi = sum(t.numel() * t.element_size() for t in w_in + rest_in)
    bo = sum(t.numel() * t.element_size() for t in w_out + rest_out)
    comp = torch.cuda.current_stream()
    s_ins = [torch.cuda.Stream() for _ in range(in_streams)]
    s_out = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    steps = max(2, min(args.steps, 5))
    for rep in range(2):  # one untimed pass, then the timed one
        barrier(world)
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(comp)
        for si in s_ins:
            si.wait_stream(comp)
        s_out.wait_stream(comp)
        read_done = [None] * chunks  # quant of slice c finished reading its weights
        sent = [None] * chunks       # slice c's codes are back on the host
        rest_read = rest_sent = None
        for _ in range(steps):
            w_ready = []
            for c in range(chunks):
                s_in = s_ins[c % in_streams]
                if read_done[c] is not None:
                    s_in.wait_event(read_done[c])
                with torch.cuda.stream(s_in):
                    for i in range(bounds[c], bounds[c + 1]):
                        w_in[i].copy_(h_w_in[i], non_blocking=True)
                e = ev(); e.record(s_in); w_ready.append(e)
            s_in = s_ins[chunks % in_streams]
            if rest_read is not None:
                s_in.wait_event(rest_read)
            with torch.cuda.stream(s_in):
                for h, t in zip(h_rest_in, rest_in):
                    t.copy_(h, non_blocking=True)
            rest_ready = ev(); rest_ready.record(s_in)
            for c in range(chunks):
                comp.wait_event(w_ready[c])
                if sent[c] is not None:
                    comp.wait_event(sent[c])
                lo, hi = bounds[c], bounds[c + 1]
                W.quantize_weight_blockwise_batched(w_in[lo:hi], wl.wout[lo:hi])
                e = ev(); e.record(comp); read_done[c] = e
                s_out.wait_event(e)
                with torch.cuda.stream(s_out):
                    for i in range(2 * lo, 2 * hi):
                        h_w_out[i].copy_(w_out[i], non_blocking=True)
                e2 = ev(); e2.record(s_out); sent[c] = e2
            comp.wait_event(rest_ready)
            if rest_sent is not None:
                comp.wait_event(rest_sent)
            run_step(W, wl, skip_weights=True)
            rest_read = ev(); rest_read.record(comp)
            s_out.wait_event(rest_read)
            with torch.cuda.stream(s_out):
                for h, t in zip(h_rest_out, rest_out):
                    h.copy_(t, non_blocking=True)
            rest_sent = ev(); rest_sent.record(s_out)
        comp.wait_stream(s_out)
        for si in s_ins:
            comp.wait_stream(si)
        end.record(comp)
        torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end) / steps, world)
    return {"value": round(100.0 * world * roof_step / (ms * 1e-3), 3), "unit": UNIT,
            "ms_per_step": round(ms, 3), "steps": steps, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo,
            "overlap": f"{in_streams} host->device streams and 1 device->host stream beside the "
                       f"compute; weight sync in {chunks} slices"}


# -------------------------------------------------------- reference arm

def bench_reference(args):
    """The oracle timed on the host cores, on the same fixed sample as
    cpu_baseline per step (the reference arm of this metric)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    peaks = load_peaks()
    smp = CpuSample()
    try:
        unit_roof = cpu_unit_roofline_s(peaks)
        for _ in range(args.warmup):
            smp.run_all_cores()
        walls = [smp.run_all_cores() for _ in range(args.steps)]
        one = smp.run_one_core()
    finally:
        smp.close()
    wall = float(np.sum(walls))
    value = 100.0 * smp.units * unit_roof * len(walls) / wall
    info = {"kind": "oracle", "cores": smp.cores, "cpu_model": smp.model,
            "value_1core": round(100.0 * unit_roof / one, 6),
            "sample": smp.describe() + " (C oracle as it stands, one process per core)"}
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT,
           "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1000 * wall / max(args.steps, 1), 1), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
           "config": {"workload": WORKLOAD, "sample": info["sample"]},
           "cpu_baseline": dict(info, value=round(value, 5), unit=UNIT),
           "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip the measurements of the rows past the hot path")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per launch of the dominant kernel, if measured for the current sources")
    args = ap.parse_args()
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
