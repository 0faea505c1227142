"""Benchmark of the W4A16 hot path on the workloads' model shapes (synthetic, seeded).

One step is one pass of the whole hot path over every workload (per layer the
weights are held as four row blocks: q|k|v, o, gate|up, down, i.e. the 7
projections with the blocks that share an input stored contiguously):
  single   - one 896 x 896 GEMV at M = 1 (Qwen2.5-0.5B q_proj), repeated on
             the same weight (L2-resident, "warm") and over 600 distinct
             copies (271 MB, more than twice the 129 MB L2, "rotated"); and
             the 1000 x 896 GEMV fused with top-5 selection over 600 copies;
  0.6B     - one Qwen3-0.6B decode token at M = 1: 28 layers x 4 blocks as
             one dependent projection list, then the lm_head GEMV with
             greedy argmax;
  decode   - one Qwen2.5-3B token at M = 1: the 144 projection GEMVs in layer
             order as one w4_gemv_seq list (a persistent launch per 96
             operations; every operation waits until all earlier ones are
             complete, as a dependent chain of projections would), then the
             lm_head GEMV fused with top-50 selection;
  batched  - the 3B projection set at M = 2, 4, 8, 16 activation rows (one
             w4_gemv per block, each streaming its weights while the previous
             kernel finishes), then per-row greedy argmax over the lm_head;
  kernels  - the lm_head GEMV + top-50 alone (8 calls back to back over two
             distinct weights), and the 36 gate|up GEMVs (2048 -> 22016)
             back to back: per-kernel decode bandwidth;
  sym128   - the 3B decode token again in the symmetric group-128 format
             (scale only, w = scale * (q - 8));
  prefill  - w4_dequant_f16 of all 144 3B weight blocks into the transposed
             half scratch, then f16_gemm for each block at M = 128, 512, 1570
             and 4096 tokens; and M = 128 through w4_gemm (dequantisation
             inside the tensor-core GEMM).
Each part is a CUDA graph replayed on one stream; CUDA events time each part.
The headline `value` is the 3B decode-token bandwidth (algorithmic bytes of
the token's weights / decode time), the first quantity of the metric; the
other quantities are reported under `parts`.  `e2e` runs the decode token
through the public API every step (projection list + lm_head calls, pinned
host activations copied in, the top-50 copied out).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       python bench.py --profile gemv|gemv16|gemm|gemm_all|dequant|lmhead|seq|seq_nowait|w4gemm|w4gemm_down
           (cases for ncu)
Under torchrun (N > 1) every rank runs an independent replica (the path has no
exchange step) and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
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

import synth  # noqa: E402

METRIC = "W4A16 decode GEMV GB/s (% HBM peak); prefill TFLOP/s; 3B-shape decode tok/s"
LAYERS = synth.QWEN25_3B_LAYERS
PROJ = synth.QWEN25_3B
LM_K, LM_N = synth.QWEN25_3B_LM_HEAD
PREFILL_MS = (128, 512, 1570, 4096)
PREFILL_M = 1570
SMALL_M = 128
BATCH_MS = (2, 4, 8, 16)
BATCH_M = 16
TOPK = 50
ROT_COPIES = 600       # distinct single-GEMV weights per rotation (> 2x L2 of bytes)
LM_REPS = 8            # lm_head calls per replay of the lm_head part
WARM_REPS = 200
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Datasheet peaks of one GB300: HBM3e 8 TB/s; dense FP16/BF16 tensor 2.25
# PFLOP/s (NVIDIA's HGX B300 figure, 36 PFLOPS FP16/BF16 per 8 GPUs, is with
# 2:4 sparsity; dense is half of it per GPU).
SPEC_PEAKS = {"hbm_gbs": 8000.0, "fp16_dense_tflops": 2250.0}
SPEC_SOURCE = ("GB300 datasheet: HBM3e 8 TB/s; dense FP16/BF16 tensor 2.25 PFLOP/s "
               "(HGX B300: 36 PFLOPS per 8 GPUs with 2:4 sparsity)")


def weight_bytes(N, K):
    return N * K // 2 + 2 * 2 * N * (K // 64)   # codes + fp16 scale + fp16 bias


def weight_bytes_sym128(N, K):
    return N * K // 2 + 2 * N * (K // 128)      # codes + fp16 scale


DECODE_BYTES = LAYERS * sum(weight_bytes(N, K) for _, K, N in PROJ) + weight_bytes(LM_N, LM_K)
DECODE_BYTES_SYM128 = LAYERS * sum(weight_bytes_sym128(N, K) for _, K, N in PROJ) + weight_bytes_sym128(LM_N, LM_K)
PROJ_WEIGHTS = LAYERS * sum(N * K for _, K, N in PROJ)
PREFILL_FLOPS = 2.0 * PREFILL_M * PROJ_WEIGHTS
SMALL_FLOPS = 2.0 * SMALL_M * PROJ_WEIGHTS
DEQUANT_BYTES = LAYERS * sum(weight_bytes(N, K) + 2 * N * K for _, K, N in PROJ)
L06, PROJ06 = synth.QWEN3_06B_LAYERS, synth.QWEN3_06B
LM06_K, LM06_N = synth.QWEN3_06B_LM_HEAD
DECODE06_BYTES = L06 * sum(weight_bytes(N, K) for _, K, N in PROJ06) + weight_bytes(LM06_N, LM06_K)
SINGLE_N, SINGLE_K = 896, 896            # Qwen2.5-0.5B q_proj
SEL_N, SEL_K, SEL_TOPK = 1000, 896, 5    # the same call with top-5 over 1000 rows
SINGLE_BYTES = weight_bytes(SINGLE_N, SINGLE_K) + 2 * SINGLE_K + 2 * SINGLE_N   # weights + x + y
SEL_BYTES = weight_bytes(SEL_N, SEL_K) + 2 * SEL_K

CONFIG = {
    "workload": ("qwen2.5-0.5b q_proj GEMV 896x896 M=1 (warm and rotated over 271 MB) + 1000x896 top-5; "
                 "qwen3-0.6b decode token M=1 (28 layers as a dependent projection list + lm_head argmax); "
                 "qwen2.5-3b decode token M=1 (36 layers x [qkv, o, gate_up, down] as one dependent projection "
                 "list + lm_head top-50; headline); 3b batched decode M=2/4/8/16 (+ per-row argmax); "
                 "3b prefill dequant-once + f16 GEMM at M=128/512/1570/4096 and w4_gemm at M=128; 3b decode "
                 "token in the symmetric group-128 format (parts)"),
    "model": "Qwen2.5-3B-shaped projections x36 + lm_head 2048->151936 (headline); Qwen3-0.6B and "
             "Qwen2.5-0.5B shapes in parts",
    "global_batch": 1, "seq_len": PREFILL_M,
    "l2": "inputs larger than L2 (1.74 GB of weights per 3B decode pass, 5.5 GB scratch; single GEMVs rotated "
          "over 600 copies), except the part marked warm",
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def peak_value(peaks, *keys):
    for k in keys:
        v = peaks.get(k)
        if isinstance(v, (int, float)):
            return float(v)
        if isinstance(v, dict):
            for kk in ("value", "gbs", "tflops"):
                if isinstance(v.get(kk), (int, float)):
                    return float(v[kk])
    return None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
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
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm

# The projections of one layer as the engine stores them: q, k, v as one row
# block (they read the same activations), gate and up as one row block.  The
# bytes and the arithmetic are those of the separate projections.
FUSED = [("qkv", 2048, 2048 + 256 + 256, ("q", "k", "v")), ("o", 2048, 2048, ("o",)),
         ("gate_up", 2048, 2 * 11008, ("gate", "up")), ("down", 11008, 2048, ("down",))]
FUSED06 = [("qkv", 1024, 2048 + 1024 + 1024, ("q", "k", "v")), ("o", 2048, 1024, ("o",)),
           ("gate_up", 1024, 2 * 3072, ("gate", "up")), ("down", 3072, 1024, ("down",))]
SRC = {"qkv": "attn", "o": "o", "gate_up": "mlp", "down": "down"}
PROJ_SRC = {"q": "attn", "k": "attn", "v": "attn", "o": "o", "gate": "mlp", "up": "mlp", "down": "down"}


class Model:
    """Device-resident synthetic weights: the Qwen2.5-3B projection set +
    lm_head (affine group 64, and symmetric group 128), the Qwen3-0.6B set +
    lm_head, and the rotated single-GEMV copies."""

    def __init__(self, torch, w4, dev):
        self.torch, self.w4, self.dev = torch, w4, dev
        t0 = time.time()
        self.layers = self._blocks(PROJ, FUSED, LAYERS, 1000, sym=False)
        qw, s, b = synth.make_linear(99, LM_N, LM_K)
        self.lm = (self._up(qw.view(np.int32)), self._up(s), self._up(b), LM_N, LM_K)
        # A second lm_head weight: the lm_head part alternates the two, so that
        # no call finds its 175 MB in the 129 MB L2.
        qw, s, b = synth.make_linear(96, LM_N, LM_K)
        self.lm_b = (self._up(qw.view(np.int32)), self._up(s), self._up(b), LM_N, LM_K)
        # The same shapes in the symmetric group-128 format (scales only).
        self.layers_s128 = self._blocks(PROJ, FUSED, LAYERS, 5000, sym=True)
        qw, s, _ = synth.make_linear_sym(98, LM_N, LM_K, 128)
        self.lm_s128 = (self._up(qw.view(np.int32)), self._up(s), None, LM_N, LM_K)
        # Qwen3-0.6B.
        self.layers06 = self._blocks(PROJ06, FUSED06, L06, 3000, sym=False)
        qw, s, b = synth.make_linear(97, LM06_N, LM06_K)
        self.lm06 = (self._up(qw.view(np.int32)), self._up(s), self._up(b), LM06_N, LM06_K)
        # Single-GEMV weights: copy 0 is the seed-0 weight; the others rotate.
        self.single = [self._linear(0 + i, SINGLE_N, SINGLE_K) for i in range(ROT_COPIES)]
        self.sel = [self._linear(20000 + i, SEL_N, SEL_K) for i in range(ROT_COPIES)]
        self.setup_s = time.time() - t0

    def _linear(self, seed, N, K):
        qw, s, b = synth.make_linear(seed, N, K)
        return self._up(qw.view(np.int32)), self._up(s), self._up(b)

    def _blocks(self, proj, fused, layers, base, sym):
        seeds = {name: p for p, (name, _, _) in enumerate(proj)}
        rows = {name: n for name, _, n in proj}
        out = []
        for l in range(layers):
            blocks = {}
            for name, K, N, parts in fused:
                if sym:
                    mats = [synth.make_linear_sym(synth.layer_seed(base, l, seeds[q]), rows[q], K, 128)
                            for q in parts]
                    qw = np.concatenate([m[0] for m in mats])
                    s = np.concatenate([m[1] for m in mats])
                    blocks[name] = (self._up(qw.view(np.int32)), self._up(s), None, N, K)
                else:
                    mats = [synth.make_linear(synth.layer_seed(base, l, seeds[q]), rows[q], K) for q in parts]
                    qw, s, b = (np.concatenate([m[i] for m in mats]) for i in range(3))
                    blocks[name] = (self._up(qw.view(np.int32)), self._up(s), self._up(b), N, K)
            out.append(blocks)
        return out

    def _up(self, a):
        return self.torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)


def x_inputs(torch, dev, M, seed, dims=(2048, 2048, 2048, 11008, LM_K)):
    """Activations per block: attn (q,k,v), o, mlp (gate, up), down, lm_head."""
    names = ("attn", "o", "mlp", "down", "lm")
    return {n: torch.from_numpy(synth.make_x(seed + 100 * i, M, K)).to(dev) for i, (n, K) in enumerate(zip(names, dims))}


def run_ours(args, rank, world):
    import torch

    import int4_weight_only_affine_gb300 as w4

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    model = Model(torch, w4, dev)
    stream = torch.cuda.Stream(dev)
    ov = w4.OVERLAP_PREVIOUS  # weights are constant: stream them while the previous kernel finishes

    def new(shape, dtype=torch.float16):
        return torch.empty(shape, dtype=dtype, device=dev)

    # ---- decode buffers ----
    xs = {M: x_inputs(torch, dev, M, 10 if M == 1 else 20 + M) for M in (1,) + BATCH_MS}
    ys = {M: {n: new((M, N)) for n, K, N, _ in FUSED} for M in (1,) + BATCH_MS}
    idx1, val1 = new((1, TOPK), torch.int32), new((1, TOPK), torch.float32)
    sel_b = {M: (new((M, 1), torch.int32), new((M, 1), torch.float32),
                 new(w4.lm_head_workspace_bytes(M, LM_N, 1), torch.uint8)) for M in BATCH_MS}
    ws1 = new(w4.lm_head_workspace_bytes(1, LM_N, TOPK), torch.uint8)
    ys_gu = new((1, 2 * 11008))
    # ---- 0.6B decode buffers ----
    xs06 = x_inputs(torch, dev, 1, 30, dims=(1024, 2048, 1024, 3072, LM06_K))
    ys06 = {n: new((1, N)) for n, K, N, _ in FUSED06}
    idx06, val06 = new((1, 1), torch.int32), new((1, 1), torch.float32)
    ws06 = new(w4.lm_head_workspace_bytes(1, LM06_N, 1), torch.uint8)
    # ---- single GEMV (config 0) ----
    x896 = torch.from_numpy(synth.make_x(0, 1, SINGLE_K)).to(dev)
    y896 = new((1, SINGLE_N))
    idx5, val5 = new((1, SEL_TOPK), torch.int32), new((1, SEL_TOPK), torch.float32)
    ws5 = new(w4.lm_head_workspace_bytes(1, SEL_N, SEL_TOPK), torch.uint8)
    # ---- prefill buffers: one transposed scratch per weight block; x/y per kind at the largest M ----
    scratch = [{n: new((K, N)) for n, K, N, _ in FUSED} for _ in range(LAYERS)]
    MX = max(PREFILL_MS)
    xp = {k: (torch.randn((MX, K), device=dev)).half() for k, K in
          (("attn", 2048), ("o", 2048), ("mlp", 2048), ("down", 11008))}
    yp = {n: new((MX, N)) for n, K, N, _ in FUSED}
    ws_gemm = w4.w4_gemm_workspace(SMALL_M, max(N for _, _, N, _ in FUSED), max(K for _, K, _, _ in FUSED),
                                   dev)  # zero-filled once; its tile counters reset themselves

    # A second form of the decode token's dependency: each projection reads
    # (a prefix of) the previous one's output -- q|k|v <- down of the layer
    # before, o <- the q part, gate|up <- o, down <- the gate part (the
    # attention, norm and activation between them are not GEMVs and are left
    # out) -- and the lm_head reads the last down output; the list kernel
    # hands each output on through its tagged exchange.  (The random weights
    # make these values overflow to inf / NaN after a few layers; that
    # changes no kernel's work or timing.)
    def seq_chain(layers, fused, x0, y, group=None):
        ops = []
        prev = x0
        for l in range(len(layers)):
            for name, K, _, _ in fused:
                qw, s, b, N, K = layers[l][name]
                x = prev.view(-1)[:K].view(1, K) if ops else prev
                op = (x, qw, s, b, y[name], len(ops) > 0)
                ops.append(op + ((group,) if group else ()))
                prev = y[name]
        return w4.GemvList(ops)

    # The headline form: external activations, every operation waiting
    # (completion counter) until all earlier ones are complete.
    def seq_barriers(layers, fused, x, y):
        ops = []
        for l in range(len(layers)):
            for name, _, _, _ in fused:
                qw, s, b, N, K = layers[l][name]
                ops.append((x[SRC[name]], qw, s, b, y[name], len(ops) > 0))
        return w4.GemvList(ops)

    def seq_barriers_g(layers, fused, x, y, group):
        ops = []
        for l in range(len(layers)):
            for name, _, _, _ in fused:
                qw, s, b, N, K = layers[l][name]
                ops.append((x[SRC[name]], qw, s, b, y[name], len(ops) > 0, group))
        return w4.GemvList(ops)

    seq3b = seq_barriers(model.layers, FUSED, xs[1], ys[1])
    # Diagnostic: the same 144 projections with no dependency between them
    # (no operation waits), separating the list's own rate from its waits.
    seq3b_free = w4.GemvList([op[:5] + (False,) for op in seq3b.ops])
    seq3b_free_ws = seq3b_free.workspace()
    seq3b_ws = seq3b.workspace()          # zero-filled once; its counters reset themselves
    seq3b_chain = seq_chain(model.layers, FUSED, xs[1]["attn"], ys[1])
    seq3b_chain_ws = seq3b_chain.workspace()
    seq_s128 = seq_barriers_g(model.layers_s128, FUSED, xs[1], ys[1], 128)
    seq_s128_ws = seq_s128.workspace()
    seq06 = seq_barriers(model.layers06, FUSED06, xs06, ys06)
    seq06_ws = seq06.workspace()

    # Batched decode at M = 2 and 4 as projection lists too (the activations
    # of the 11008-wide down projection fit in shared memory up to M = 4).
    seq_b = {M: seq_barriers(model.layers, FUSED, xs[M], ys[M]) for M in (2, 4)}
    seq_b_ws = {M: seq_b[M].workspace() for M in (2, 4)}

    def batched_list(M):
        def run():
            seq_b[M].run(seq_b_ws[M], stream)
            qw, s, b, N, K = model.lm
            idx, val, ws = sel_b[M]
            w4.lm_head_argmax_topk(xs[M]["lm"], qw, s, b, k=1, idx=idx, val=val, workspace=ws, stream=stream,
                                   flags=ov)
        return run

    def decode_seq():
        seq3b.run(seq3b_ws, stream)
        qw, s, b, N, K = model.lm
        w4.lm_head_argmax_topk(xs[1]["lm"], qw, s, b, k=TOPK, idx=idx1, val=val1, workspace=ws1, stream=stream,
                               flags=ov)

    def decode_seq_free():
        seq3b_free.run(seq3b_free_ws, stream)
        qw, s, b, N, K = model.lm
        w4.lm_head_argmax_topk(xs[1]["lm"], qw, s, b, k=TOPK, idx=idx1, val=val1, workspace=ws1, stream=stream,
                               flags=ov)

    def decode_seq_chain():
        seq3b_chain.run(seq3b_chain_ws, stream)
        qw, s, b, N, K = model.lm
        w4.lm_head_argmax_topk(ys[1]["down"], qw, s, b, k=TOPK, idx=idx1, val=val1, workspace=ws1, stream=stream,
                               flags=ov)

    def decode_seq_s128():
        seq_s128.run(seq_s128_ws, stream)
        qw, s, b, N, K = model.lm_s128
        w4.lm_head_argmax_topk(xs[1]["lm"], qw, s, None, k=TOPK, idx=idx1, val=val1, workspace=ws1,
                               stream=stream, flags=ov, group=128)

    def decode06():
        seq06.run(seq06_ws, stream)
        qw, s, b, N, K = model.lm06
        w4.lm_head_argmax_topk(xs06["lm"], qw, s, b, k=1, idx=idx06, val=val06, workspace=ws06, stream=stream,
                               flags=ov)

    def single_warm():
        qw, s, b = model.single[0]
        for _ in range(WARM_REPS):
            w4.w4_gemv(x896, qw, s, b, y=y896, stream=stream, flags=ov)

    def single_rot():
        for qw, s, b in model.single:
            w4.w4_gemv(x896, qw, s, b, y=y896, stream=stream, flags=ov)

    def sel_rot():
        for qw, s, b in model.sel:
            w4.lm_head_argmax_topk(x896, qw, s, b, k=SEL_TOPK, idx=idx5, val=val5, workspace=ws5, stream=stream,
                                   flags=ov)

    def w4gemm_small():
        first = True
        for l in range(LAYERS):
            for name, _, N, _ in FUSED:
                qw, s, b, N, K = model.layers[l][name]
                w4.w4_gemm(xp[SRC[name]][:SMALL_M], qw, s, b, y=yp[name][:SMALL_M], workspace=ws_gemm,
                           stream=stream, flags=0 if first else ov)
                first = False

    def gemm_at(M):
        def run():
            first = True
            for l in range(LAYERS):
                for name, _, _, _ in FUSED:
                    # After the first GEMM every scratch is long complete: fetch the
                    # weights early and wait for the previous GEMM only for x and y.
                    w4.f16_gemm(xp[SRC[name]][:M], scratch[l][name], y=yp[name][:M], stream=stream,
                                flags=0 if first else ov)
                    first = False
        return run

    def lm_only():
        for i in range(LM_REPS):
            qw, s, b, N, K = (model.lm, model.lm_b)[i % 2]
            w4.lm_head_argmax_topk(xs[1]["lm"], qw, s, b, k=TOPK, idx=idx1, val=val1, workspace=ws1, stream=stream,
                                   flags=ov)

    def gate_up_only():
        for l in range(LAYERS):
            qw, s, b, N, K = model.layers[l]["gate_up"]
            w4.w4_gemv(xs[1]["mlp"], qw, s, b, y=ys_gu, stream=stream, flags=ov)

    def batched(M):
        def run():
            for l in range(LAYERS):
                for name, _, _, _ in FUSED:
                    qw, s, b, N, K = model.layers[l][name]
                    w4.w4_gemv(xs[M][SRC[name]], qw, s, b, y=ys[M][name], stream=stream, flags=ov)
            qw, s, b, N, K = model.lm
            idx, val, ws = sel_b[M]
            w4.lm_head_argmax_topk(xs[M]["lm"], qw, s, b, k=1, idx=idx, val=val, workspace=ws, stream=stream,
                                   flags=ov)
        return run

    def dequant_all():
        for l in range(LAYERS):
            for name, _, _, _ in FUSED:
                qw, s, b, N, K = model.layers[l][name]
                # distinct weights into distinct scratch buffers: independent calls
                w4.w4_dequant_f16(qw, s, b, w16=scratch[l][name], stream=stream, flags=ov)

    parts = {
        "dequant": dequant_all,
        "gemm": gemm_at(PREFILL_M),
        "gemm_m512": gemm_at(512),
        "gemm_m4096": gemm_at(4096),
        "decode_m1": decode_seq,
        "decode_m1_chain": decode_seq_chain,
        "decode_m1_nowait": decode_seq_free,
        **{f"decode_m{M}": batched(M) for M in BATCH_MS},
        **{f"decode_m{M}_list": batched_list(M) for M in (2, 4)},
        "lm_head_m1": lm_only,
        "gate_up_m1": gate_up_only,
        "decode_m1_s128": decode_seq_s128,
        "decode06_m1": decode06,
        "single_warm": single_warm,
        "single_rot": single_rot,
        "sel5_rot": sel_rot,
        "w4gemm_m128": w4gemm_small,
        "gemm_m128": gemm_at(SMALL_M),
    }
    nb = LAYERS * len(FUSED)
    n_seq = (nb + 95) // 96
    n_seq06 = (L06 * len(FUSED06) + 95) // 96
    launches = {"dequant": nb, "gemm": nb, "gemm_m512": nb, "gemm_m4096": nb, "decode_m1": n_seq + 2,
                **{f"decode_m{M}": nb + 2 for M in BATCH_MS},
                **{f"decode_m{M}_list": n_seq + 2 for M in (2, 4)}, "lm_head_m1": 2 * LM_REPS, "gate_up_m1": LAYERS,
                "decode_m1_s128": n_seq + 2, "decode_m1_chain": n_seq + 2, "decode_m1_nowait": n_seq + 2, "decode06_m1": n_seq06 + 2, "single_warm": WARM_REPS,
                "single_rot": ROT_COPIES, "sel5_rot": 2 * ROT_COPIES, "w4gemm_m128": nb, "gemm_m128": nb}
    # eager warm-up (sets kernel attributes), then capture one graph per part
    with torch.cuda.stream(stream):
        for f in parts.values():
            f()
    stream.synchronize()
    graphs = {}
    for name, f in parts.items():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            f()
        graphs[name] = g
    torch.cuda.synchronize()
    if w4.device_status() != 0:
        raise RuntimeError("device-side wait expired during warm-up")

    order = list(parts)
    ev = {n: [] for n in order}

    def step(record):
        for n in order:
            if record:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            graphs[n].replay()
            if record:
                e1.record(stream)
                ev[n].append((e0, e1))

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(False)
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(dev.index)
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for _ in range(args.steps):
            step(True)
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    if w4.device_status() != 0:
        raise RuntimeError("device-side wait expired in the timed region")

    total_ms = t_start.elapsed_time(t_end) / args.steps
    part_ms = {n: statistics.median([a.elapsed_time(b) for a, b in ev[n]]) for n in order}
    part_mean = {n: sum(a.elapsed_time(b) for a, b in ev[n]) / args.steps for n in order}
    total_ms = max_over_ranks(total_ms, world)

    # ---- e2e: the decode token through the public API with host buffers ----
    # Every step: pinned host activations copied in, the projection list and
    # the lm_head call issued through the binding (C ABI), the top-50 copied
    # out, and the stream synchronised; timed on the host clock.
    e2e_in = xs[1]                      # every projection's activations and the lm_head's
    host_x = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in e2e_in.items()}
    for k, v in e2e_in.items():
        host_x[k].copy_(v.cpu())
    host_idx = torch.empty((1, TOPK), dtype=torch.int32, pin_memory=True)
    host_val = torch.empty((1, TOPK), dtype=torch.float32, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host_x.values())
    d2h = host_idx.numel() * 4 + host_val.numel() * 4

    def e2e_loop(issue):
        times = []
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                for k, v in host_x.items():
                    e2e_in[k].copy_(v, non_blocking=True)
                issue()
                host_idx.copy_(idx1, non_blocking=True)
                host_val.copy_(val1, non_blocking=True)
                stream.synchronize()
                if i >= args.warmup:
                    times.append(time.perf_counter() - t0)
        return max_over_ranks(statistics.median(times), world)

    e2e_s = e2e_loop(decode_seq)                          # API calls every step
    e2e_graph_s = e2e_loop(graphs["decode_m1"].replay)    # the same work replayed as a CUDA graph
    if w4.device_status() != 0:
        raise RuntimeError("device-side wait expired in the end-to-end runs")

    part_ms = {n: max_over_ranks(v, world) for n, v in part_ms.items()}
    res = {
        "total_ms": total_ms, "part_ms": part_ms, "part_mean_ms": part_mean, "decode_ms": part_ms["decode_m1"],
        "e2e_s": e2e_s, "e2e_graph_s": e2e_graph_s, "h2d": h2d, "d2h": d2h, "clocks": clk,
        "setup_s": model.setup_s, "launches_per_step": sum(launches.values()), "launches": launches,
    }
    return res


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    """The maximum of v over the ranks (NCCL needs a device tensor, gloo a host one)."""
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- oracle arm

def oracle_decode_sample(budget_s, threads):
    """Time the CPU oracle GEMV over the decode projections in layer order
    until `budget_s` has elapsed; returns (bytes processed, seconds, sample text)."""
    import oracle
    x = {k: synth.make_x(10 + off, 1, K) for k, off, K in
         (("attn", 0, 2048), ("o", 100, 2048), ("mlp", 200, 2048), ("down", 300, 11008))}
    done_bytes, t_used, n_mats = 0, 0.0, 0
    for l in range(LAYERS):
        for p, (name, K, N) in enumerate(PROJ):
            qw, s, b = synth.make_linear(synth.layer_seed(1000, l, p), N, K)
            t0 = time.perf_counter()
            oracle.gemv(x[PROJ_SRC[name]], qw, s, b, N, K, threads=threads)
            t_used += time.perf_counter() - t0
            done_bytes += weight_bytes(N, K)
            n_mats += 1
            if t_used >= budget_s:
                return done_bytes, t_used, f"first {n_mats} projection GEMVs (M=1) of the 3B decode order"
    return done_bytes, t_used, f"all {n_mats} projection GEMVs (M=1) of the 3B decode order"


def cpu_baseline(budget_s=12.0):
    threads = os.cpu_count() or 1
    nb, t, sample = oracle_decode_sample(budget_s, threads)
    return {"value": nb / t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": sample + f" ({nb / 1e6:.1f} MB of int4 weights, {t:.1f} s)"}


# ---------------------------------------------------------------- profiling cases

def profile_case(which, iters=3):
    import torch

    import int4_weight_only_affine_gb300 as w4
    dev = torch.device("cuda:0")
    if which in ("gemv", "gemv16", "dequant"):
        K, N = 2048, 22016   # gate and up projections stored as one matrix
        qw, s, b = synth.make_linear(1, N, K)
        a = [torch.from_numpy(t).to(dev) for t in (qw.view(np.int32), s, b)]
        x = torch.from_numpy(synth.make_x(2, 16 if which == "gemv16" else 1, K)).to(dev)
        for _ in range(iters):
            if which == "dequant":
                w4.w4_dequant_f16(*a)
            else:
                w4.w4_gemv(x, *a)
    elif which == "gemm_all":
        # f16_gemm at M = 1570 over the 144 Qwen2.5-3B blocks, once (after a
        # warm-up pass): the launches whose DRAM traffic the bench reports.
        seeds = {name: p for p, (name, _, _) in enumerate(PROJ)}
        rows = {name: n for name, _, n in PROJ}
        xp = {K: torch.randn((PREFILL_M, K), device=dev).half() for K in (2048, 11008)}
        blocks = []
        for l in range(LAYERS):
            for name, K, N, parts in FUSED:
                mats = [synth.make_linear(synth.layer_seed(1000, l, seeds[q]), rows[q], K) for q in parts]
                qw = np.concatenate([m[0] for m in mats]).view(np.int32)
                s, b = (np.concatenate([m[i] for m in mats]) for i in (1, 2))
                blocks.append((w4.w4_dequant_f16(*[torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in (qw, s, b)]),
                               K, N))
        y = torch.empty((PREFILL_M, 2 * 11008), dtype=torch.float16, device=dev)
        for _ in range(2):
            for w16, K, N in blocks:
                w4.f16_gemm(xp[K], w16, y=y.view(-1)[:PREFILL_M * N].view(PREFILL_M, N))
    elif which == "lmhead":
        qw, s, b = synth.make_linear(1, LM_N, LM_K)
        a = [torch.from_numpy(t).to(dev) for t in (qw.view(np.int32), s, b)]
        x = torch.from_numpy(synth.make_x(2, 1, LM_K)).to(dev)
        for _ in range(iters):
            w4.lm_head_argmax_topk(x, *a, k=TOPK)
    elif which == "seq":
        # two layers' blocks as one dependent projection list (M = 1)
        ops = []
        seeds = {name: p for p, (name, _, _) in enumerate(PROJ)}
        rows = {name: n for name, _, n in PROJ}
        for l in range(2):
            for name, K, N, parts in FUSED:
                mats = [synth.make_linear(synth.layer_seed(1000, l, seeds[q]), rows[q], K) for q in parts]
                qw, s, b = (np.concatenate([m[i] for m in mats]) for i in range(3))
                x = torch.from_numpy(synth.make_x(10 + len(ops), 1, K)).to(dev)
                y = torch.empty((1, N), dtype=torch.float16, device=dev)
                ops.append((x, *[torch.from_numpy(np.ascontiguousarray(t)).to(dev) for t in (qw.view(np.int32), s, b)],
                            y, len(ops) > 0))
        ws = w4.seq_workspace(ops)
        for _ in range(iters):
            w4.w4_gemv_seq(ops, workspace=ws)
    elif which == "seq_nowait":
        # eight independent gate|up operations (2048 -> 22016) as one list,
        # no waits: the list kernel's consumer rate apart from dependencies
        K, N = 2048, 22016
        x = torch.from_numpy(synth.make_x(3, 1, K)).to(dev)
        y = torch.empty((1, N), dtype=torch.float16, device=dev)
        ops = []
        for i in range(8):
            qw, s, b = synth.make_linear(1000 + 7 * i + 2, N, K)
            ops.append((x, *[torch.from_numpy(np.ascontiguousarray(t)).to(dev) for t in (qw.view(np.int32), s, b)],
                        y, False))
        gl = w4.GemvList(ops)
        ws = gl.workspace()
        for _ in range(iters + 1):
            gl.run(ws)
    elif which in ("w4gemm", "w4gemm_down"):
        # the fused int4 GEMM at M = 128 on the gate|up block (2048 -> 22016)
        # or the down block (11008 -> 2048)
        K, N, M = (2048, 22016, 128) if which == "w4gemm" else (11008, 2048, 128)
        qw, s, b = synth.make_linear(1, N, K)
        a = [torch.from_numpy(t).to(dev) for t in (qw.view(np.int32), s, b)]
        x = torch.from_numpy(synth.make_x(2, M, K)).to(dev)
        ws = w4.w4_gemm_workspace(M, N, K, dev)
        for _ in range(iters + 1):
            w4.w4_gemm(x, *a, workspace=ws)
    elif which == "gemm":
        x = torch.randn((PREFILL_M, 2048), device=dev).half()
        w = (0.05 * torch.randn((2048, 11008), device=dev)).half()
        for _ in range(iters):
            w4.f16_gemm(x, w)
    torch.cuda.synchronize()
    assert w4.device_status() == 0
    print(json.dumps({"profile": which, "iters": iters}))


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--profile", default=None,
                    choices=["gemv", "gemv16", "gemm", "gemm_all", "dequant", "lmhead", "seq", "seq_nowait",
                             "w4gemm", "w4gemm_down"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.profile:
        profile_case(args.profile)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    peaks, peak_src = load_peaks()
    hbm = peak_value(peaks, "hbm_gbs", "hbm") or FALLBACK_PEAKS["hbm_gbs"]
    tflops = peak_value(peaks, "bf16_tflops", "bf16") or FALLBACK_PEAKS["bf16_tflops"]

    if args.impl == "reference":
        # The reference arm is the CPU oracle; under torchrun only rank 0 works.
        if rank != 0:
            return
        per_step = []
        threads = os.cpu_count() or 1
        for i in range(args.warmup + args.steps):
            nb, t, sample = oracle_decode_sample(8.0 / max(1, args.steps), threads)
            if i >= args.warmup:
                per_step.append((nb, t))
        nb = sum(p[0] for p in per_step)
        t = sum(p[1] for p in per_step)
        v = nb / t / 1e9
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": {**CONFIG, "parallelism": "cpu"},
                "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                                 "sample": sample + " (bounded per step; the headline quantity: int4 weight bytes "
                                                    "of the 3B decode projections per second)"},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    r = run_ours(args, rank, world)
    if rank != 0:
        return
    print(json.dumps(report(args, r, world, peaks, peak_src, hbm, tflops)))


def f16_gemm_source_hash():
    """sha256/16 of the f16_gemm kernels' source: gemm.cu up to its w4_gemm section."""
    import hashlib
    src = open(os.path.join(ROOT, "int4_weight_only_affine_gb300", "csrc", "gemm.cu")).read()
    cut = src.find("// w4_gemm: the int4 GEMM")
    return hashlib.sha256(src[:cut if cut >= 0 else len(src)].encode()).hexdigest()[:16]


def gemm_traffic():
    """DRAM bytes per f16_gemm launch at M = 1570 (average over the 144 blocks)
    from the committed ncu summary, if it was taken on the current f16_gemm
    source (None otherwise: the counters would describe another kernel)."""
    path = os.path.join(ROOT, "profiles", "gemm_f16_m1570_all_blocks.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("f16_gemm source sha256/16") != f16_gemm_source_hash():
        return None
    try:
        return float(vals["DRAM bytes per launch"])
    except (KeyError, ValueError):
        return None


def report(args, r, world, peaks, peak_src, hbm, tflops):
    pm = r["part_ms"]
    spec_hbm, spec_tf = SPEC_PEAKS["hbm_gbs"], SPEC_PEAKS["fp16_dense_tflops"]

    def gbs(nbytes, ms):
        return nbytes / (ms / 1e3) / 1e9

    def hbm_part(nbytes, ms, **extra):
        v = gbs(nbytes, ms)
        return {"ms": ms, "GB_s": v, "frac_hbm": v / hbm, "frac_hbm_spec": v / spec_hbm, **extra}

    def gemm_part(M, ms, **extra):
        tf = 2.0 * M * PROJ_WEIGHTS / (ms / 1e3) / 1e12
        return {"ms": ms, "M": M, "TFLOP_s": tf, "frac_tensor": tf / tflops, "frac_tensor_spec": tf / spec_tf,
                **extra}

    decode_gbs = gbs(DECODE_BYTES, pm["decode_m1"])
    gemm_tflops = PREFILL_FLOPS / (pm["gemm"] / 1e3) / 1e12
    lm_gbs = gbs(weight_bytes(LM_N, LM_K), pm["lm_head_m1"] / LM_REPS)
    proj_bytes = LAYERS * sum(weight_bytes(N, K) for _, K, N in PROJ)
    two_ms = pm["dequant"] + pm["gemm_m128"]
    parts = {
        "single_gemv_896_m1_warm": hbm_part(SINGLE_BYTES, pm["single_warm"] / WARM_REPS,
                                            note=f"{WARM_REPS} launches on one L2-resident weight; ms per launch"),
        "single_gemv_896_m1_rotated": hbm_part(SINGLE_BYTES, pm["single_rot"] / ROT_COPIES,
                                               note=f"{ROT_COPIES} distinct weights (271 MB); ms per launch"),
        "topk5_1000x896_m1_rotated": hbm_part(SEL_BYTES, pm["sel5_rot"] / ROT_COPIES,
                                              note=f"lm_head_argmax_topk k=5 over {ROT_COPIES} distinct weights; "
                                                   "ms per call"),
        "decode06_m1": hbm_part(DECODE06_BYTES, pm["decode06_m1"], tok_s=1e3 / pm["decode06_m1"],
                                note="Qwen3-0.6B token: 112 dependent GEMVs (28 x 4 blocks) + lm_head argmax"),
        "decode_m1": hbm_part(DECODE_BYTES, pm["decode_m1"], tok_s=1e3 / pm["decode_m1"],
                              note="every operation waits (completion counter) until all earlier ones are "
                                   "complete; + lm_head top-50"),
        "decode_m1_chain": hbm_part(DECODE_BYTES, pm["decode_m1_chain"], tok_s=1e3 / pm["decode_m1_chain"],
                                    note="each operation reads (a prefix of) the previous output through the "
                                         "tagged exchange; lm_head reads the last output"),
        "decode_m1_nowait": hbm_part(DECODE_BYTES, pm["decode_m1_nowait"],
                                     note="diagnostic, not a decode token: the same 144 projections as one list "
                                          "with no waits (no dependencies) + lm_head top-50"),
        **{f"decode_m{M}": hbm_part(DECODE_BYTES, pm[f"decode_m{M}"], tok_s=M * 1e3 / pm[f"decode_m{M}"],
                                    gemv_tflop_s=2.0 * M * (PROJ_WEIGHTS + LM_N * LM_K) / (pm[f"decode_m{M}"] / 1e3)
                                    / 1e12) for M in BATCH_MS},
        **{f"decode_m{M}_list": hbm_part(DECODE_BYTES, pm[f"decode_m{M}_list"], tok_s=M * 1e3 / pm[f"decode_m{M}_list"],
                                         note="the M-row token as one projection list (each operation waiting on "
                                              "the completion counter) + per-row argmax")
           for M in (2, 4)},
        "dequant": hbm_part(DEQUANT_BYTES, pm["dequant"]),
        "gemm_m128": gemm_part(128, pm["gemm_m128"]),
        "gemm_m512": gemm_part(512, pm["gemm_m512"]),
        "gemm_m1570": gemm_part(PREFILL_M, pm["gemm"]),
        "gemm_m4096": gemm_part(4096, pm["gemm_m4096"]),
        "lm_head_m1_top50": hbm_part(weight_bytes(LM_N, LM_K), pm["lm_head_m1"] / LM_REPS,
                                     note=f"{LM_REPS} calls back to back alternating two distinct 175 MB weights "
                                          "(each call pass 1 + pass 2); ms per call"),
        "gemv_gate_up_m1_x36": hbm_part(LAYERS * weight_bytes(2 * 11008, 2048), pm["gate_up_m1"]),
        "decode_m1_sym128": hbm_part(DECODE_BYTES_SYM128, pm["decode_m1_s128"], tok_s=1e3 / pm["decode_m1_s128"],
                                     format="symmetric int4, group 128 (scale only), same shapes"),
        "prefill_m128_w4gemm": gemm_part(SMALL_M, pm["w4gemm_m128"],
                                         weight_GB_s=gbs(proj_bytes, pm["w4gemm_m128"])),
        "prefill_m128_dequant_then_gemm": {"ms": two_ms, "TFLOP_s": SMALL_FLOPS / (two_ms / 1e3) / 1e12,
                                           "gemm_ms": pm["gemm_m128"]},
    }
    for M in PREFILL_MS:   # dequant-once + GEMM, the prefill as the pages describe it
        key = "gemm" if M == PREFILL_M else f"gemm_m{M}"
        t = pm["dequant"] + pm[key]
        parts[f"prefill_m{M}_dequant_then_gemm"] = {"ms": t, "TFLOP_s": 2.0 * M * PROJ_WEIGHTS / (t / 1e3) / 1e12}
    line = {
        "metric": METRIC,
        "value": decode_gbs * world,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": r["total_ms"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {**CONFIG, "parallelism": f"replicas{world}"},
        "parts": parts,
        "roofline": {"bound": "tensor", "kernel": "f16_gemm (tcgen05), M = 1570, average over the 144 blocks",
                     "achieved": gemm_tflops, "peak": tflops, "unit": "TFLOP/s", "frac": gemm_tflops / tflops,
                     "traffic": gemm_traffic(), "frac_spec": gemm_tflops / spec_tf, "peak_spec": spec_tf,
                     "frac_sustained": gemm_tflops / (peak_value(peaks, "bf16_tflops_sustained") or tflops),
                     "peak_source": f"{peak_src} bf16 dense burst (fp16 dense taken equal); spec: {SPEC_SOURCE}"},
        "roofline_decode": {"bound": "hbm", "kernel": "w4_gemv_seq + lm_head (3B decode token, dependent chain)",
                            "achieved": decode_gbs, "peak": hbm, "unit": "GB/s", "frac": decode_gbs / hbm,
                            "traffic": None, "frac_spec": decode_gbs / spec_hbm, "peak_spec": spec_hbm,
                            "peak_source": f"{peak_src} HBM copy; spec: {SPEC_SOURCE}"},
        "roofline_gemv": {"bound": "hbm", "kernel": "lm_head GEMV 2048->151936 + top-50 (largest decode GEMV)",
                          "achieved": lm_gbs, "peak": hbm, "unit": "GB/s", "frac": lm_gbs / hbm,
                          "traffic": None, "frac_spec": lm_gbs / spec_hbm, "peak_spec": spec_hbm,
                          "peak_source": f"{peak_src} HBM copy; spec: {SPEC_SOURCE}"},
        "e2e": {"value": DECODE_BYTES / r["e2e_s"] / 1e9 * world, "unit": "GB/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "ms_per_token": 1e3 * r["e2e_s"],
                "note": "3B decode token through the public API every step (GemvList.run = w4_gemv_seq, "
                        "lm_head_argmax_topk): pinned H2D activations, D2H top-50, stream synchronised"},
        "e2e_graph": {"value": DECODE_BYTES / r["e2e_graph_s"] / 1e9 * world, "unit": "GB/s",
                      "ms_per_token": 1e3 * r["e2e_graph_s"],
                      "note": "the same token with the kernels replayed as a CUDA graph"},
        "gpu_launches": r["launches_per_step"] * args.steps,
        "clocks": r["clocks"],
        "setup_s": r["setup_s"],
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline()
    return line


if __name__ == "__main__":
    main()
