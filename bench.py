#!/usr/bin/env python
"""Benchmark of one QSPEC decoding round on the GB300 path.

Workload (default): a Llama-3-8B-shaped model -- 32 layers, each with its
seven linears stacked as qkv (4096 -> 6144), o (4096 -> 4096), gate/up
(4096 -> 28672) and down (14336 -> 4096), plus the 4096 x 128256 LM head --
with random INT4 weights (codes U{0..15}, fp16 scales U(0.005, 0.02), zero
points U{0..15}, group 128), batch B = 1, gamma = 4 drafts.  One step is one
round of the hot path:
  gamma draft passes: per layer and linear, INT4 activation quantisation and
      the W4A4 linear at M = B; then the W4A4 LM head;
  one verify pass: every linear and the LM head in W4A16 at M = B (gamma + 1);
  sampled verification of the gamma drafts over the 128256-token vocabulary;
  the KV overwrite of the accepted rows in a 32-layer x 8-head x 4096 x 128
  bf16 cache.
Activations are bf16 N(0, 1) with 1 % outlier channels x20; target logits
N(0, 3^2), draft logits = target + N(0, 0.5^2); drafts drawn from the draft
rows.  Attention, norms and embeddings are not on this path and are not run;
the verification reads its synthetic logits.  Weights (3.9 GB) exceed L2, so
no flush is needed between steps.

value    accepted tokens per second, sum_b (A_b + 1) / step time, with every
         input resident in HBM (CUDA graphs, CUDA events around K steps).
e2e      the same through host buffers: per step, pinned host -> device copy
         of that step's inputs, the round, device -> host read of its tokens.
roofline the dominant kernel (the W4A4 small-M linear), its algorithmic bytes
         over its CUDA-event time, against the measured HBM copy bandwidth.

--impl reference runs the CPU oracle (plain C, all host cores) on a bounded
sample of the same round each step and extrapolates the round time.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from quantized_speculative_decoding_shared_gb300 import synthetic as syn  # noqa: E402
from quantized_speculative_decoding_shared_gb300.round import QspecRound  # noqa: E402

GROUP = 128
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# dense tcgen05 kind::f8f6f4 (E4M3) rate measured on this GPU with a
# shared-memory-operand MMA loop (M = 128, N = 256, K = 32, one CTA per SM,
# CUDA events): 128 cycles per MMA, 4821.8 TFLOP/s
E4M3_PROBE_TFLOPS = 4821.8

# draft-logit noise of the Qwen2.5-7B workloads: mean acceptance 0.60 per
# draft position on the oracle (tests/golden/calibrate_q_noise.py)
QWEN_Q_NOISE = json.load(open(os.path.join(ROOT, "tests", "golden", "qwen_q_noise.json")))["q_noise"]

WORKLOADS = {
    # Llama-3-8B decode at batch 1: W4A4 draft at M = 1, W4A16 verify at M = 5
    "llama3-8b-decode-b1-g4": dict(shape=syn.LLAMA3_8B, B=1, gamma=4, outliers=0.01,
                                   T=4096, p_std=3.0, q_noise=0.5, seed=1),
    # Llama-3-8B at batch 16: W4A16 verify at M = 80 (with the LM head), verification
    # over 16 x 5 x 128256 logits, KV overwrite on the 32-layer cache
    "llama3-8b-b16-g4": dict(shape=syn.LLAMA3_8B, B=16, gamma=4, outliers=0.0,
                             T=4096, p_std=3.0, q_noise=0.5, seed=2),
    # Qwen2.5-7B at batch 32, gamma 2 / 4 / 8 (W4A4 at M = 32, W4A16 at M = 96 / 160 / 288)
    "qwen2.5-7b-b32-g2": dict(shape=syn.QWEN25_7B, B=32, gamma=2, outliers=0.0,
                              T=4096, p_std=3.0, q_noise=QWEN_Q_NOISE, seed=3),
    "qwen2.5-7b-b32-g4": dict(shape=syn.QWEN25_7B, B=32, gamma=4, outliers=0.0,
                              T=4096, p_std=3.0, q_noise=QWEN_Q_NOISE, seed=3),
    "qwen2.5-7b-b32-g8": dict(shape=syn.QWEN25_7B, B=32, gamma=8, outliers=0.0,
                              T=4096, p_std=3.0, q_noise=QWEN_Q_NOISE, seed=3),
}
PREFILL = "llama3-8b-prefill-m4096"
DEFAULT_WORKLOAD = "llama3-8b-decode-b1-g4"


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + [PREFILL],
                    default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the short timed runs of the other workloads (single-GPU default run)")
    ap.add_argument("--rounds", type=int, default=16, help="distinct captured rounds (RNG round ids)")
    ap.add_argument("--profile-case", choices=["w4a4_m1", "w4a16_m5", "w4a16_m80", "quant", "verify_sample",
                                               "verify_greedy", "kv", "fp8_m5", "w4a4_m4096", "w4a4_m32",
                                              "w4a4_m16_down", "w4a4_m16", "w4a4_m16_gateup", "draft_sample"],
                    help="run one kernel a few times on a single LM-head-sized case (for ncu)")
    ap.add_argument("--profile-reps", type=int, default=3)
    return ap.parse_args()


def profile_case(name, reps):
    """One kernel on one case larger than L2 (the 128256 x 4096 LM head: 263 MB
    of packed weights), launched `reps` times; prints nothing measured."""
    from quantized_speculative_decoding_shared_gb300 import binding as q
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    N, K = 128256, 4096
    if name in ("w4a4_m1", "w4a16_m5", "w4a16_m80", "quant"):
        codes, s, z = syn.weights(N, K, 5, device=dev)
        packed, sz = q.pack_weights(codes, s, z)
        del codes
        M = {"w4a16_m5": 5, "w4a16_m80": 80}.get(name, 1)
        x = syn.activations(M, K, 6, device=dev, outlier_frac=0.01)
        xq, sx, qs = q.quant_act_int4(x)
        for _ in range(reps):
            if name == "w4a4_m1":
                q.linear_w4a4_bf16(x, packed, sz)
            elif name in ("w4a16_m5", "w4a16_m80"):
                q.linear_w4a16(x, packed, sz)
            else:
                q.quant_act_int4(syn.activations(4096, 14336, 7, device=dev))
    elif name == "fp8_m5":
        # the Q8 (FP8) verify linear on the 128256 x 4096 LM head at M = 5
        g = torch.Generator(device=dev).manual_seed(5)
        w16 = (torch.randn((N, K), generator=g, device=dev) * 0.02).to(torch.float16)
        w8, s8 = q.quant_weights_fp8(w16)
        del w16
        xq, sa = q.quant_act_fp8(syn.activations(5, K, 6, device=dev, outlier_frac=0.01))
        for _ in range(reps):
            q.linear_fp8(xq, sa, w8, s8)
    elif name == "w4a4_m4096":
        # W4A4 at M = 4096 through the stacked gate/up projection (4096 -> 28672)
        codes, s, z = syn.weights(28672, 4096, 40, device=dev)
        packed, sz = q.pack_weights(codes, s, z)
        del codes
        xq, sx, qs = q.quant_act_int4(syn.activations(4096, 4096, 50, device=dev))
        for _ in range(reps):
            q.linear_w4a4(xq, sx, qs, packed, sz)
    elif name in ("w4a4_m32", "w4a4_m16_down", "w4a4_m16", "w4a4_m16_gateup"):
        # the decode-batch W4A4 tensor-core kernel: the LM head at 32 tokens,
        # the 4096 x 14336 down projection at 16 (groups split over 4-CTA
        # clusters), or the 28672 x 4096 gate/up projection at 16 (one CTA per
        # 128-channel tile); the tensor-memory GEMV on the LM head at 16 tokens
        M, Nn, Kk = {"w4a4_m32": (32, N, K), "w4a4_m16_down": (16, 4096, 14336), "w4a4_m16": (16, N, K),
                     "w4a4_m16_gateup": (16, 28672, 4096)}[name]
        codes, s, z = syn.weights(Nn, Kk, 41, device=dev)
        packed, sz = q.pack_weights(codes, s, z)
        del codes
        xq, sx, qs = q.quant_act_int4(syn.activations(M, Kk, 51, device=dev))
        for _ in range(reps):
            q.linear_w4a4(xq, sx, qs, packed, sz)
    elif name == "draft_sample":
        # one draft position's logits, 16 x 128256 (4 MB: the real size, in L2)
        Qd = syn.logits_noisy_draft(16, 1, 128256, 98, device=dev)[1][:, 0, :].contiguous()
        ws = q.draft_workspace(16, 128256, dev)
        for r in range(reps):
            q.draft_sample(Qd, 5, r, 1, workspace=ws)
    elif name in ("verify_sample", "verify_greedy"):
        P, Q, d = syn.logits_noisy_draft(256, 4, 128256, 4, device=dev)
        ws = q.verify_workspace(256, 4, 128256, dev)
        for r in range(reps):
            if name == "verify_sample":
                q.verify_sample(P, Q, d, 1, r, workspace=ws)
            else:
                q.verify_greedy(P, d, workspace=ws)
    else:
        kc, vc = syn.kv_cache(32, 16, 8, 4096, 128, 2, device=dev)
        kn, vn = syn.kv_new(32, 16, 4, 8, 128, 3, device=dev)
        base = syn.base_positions(16, 4096, 4, 2, device=dev)
        nacc = torch.full((16,), 4, dtype=torch.int32, device=dev)
        for _ in range(reps):
            q.kv_overwrite(kc, vc, kn, vn, base, nacc)
    torch.cuda.synchronize()
    print("profile case %s: %d launches done" % (name, reps))


# ---------------------------------------------------------------------------
# algorithmic bytes (per launch) of the HBM-bound steps
# ---------------------------------------------------------------------------
def bytes_w4a16(M, N, K):
    return K * N // 2 + 4 * N * K // GROUP + 2 * M * K + 2 * M * N


def bytes_w4a4(M, N, K):
    return K * N // 2 + 4 * N * K // GROUP + M * K // 2 + 8 * M * K // GROUP + 2 * M * N


def bytes_w4a4_bf16(M, N, K):
    """The draft call with the quantiser inside: bf16 activations read, the
    quantised activations (xq, sx, qs) written once."""
    return K * N // 2 + 4 * N * K // GROUP + 2 * M * K + M * K // 2 + 8 * M * K // GROUP + 2 * M * N


def bytes_quant(M, K):
    return 2 * M * K + M * K // 2 + 8 * M * K // GROUP


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def _code_only(text):
    """C/C++ source without comments and with whitespace collapsed: what the
    compiler sees, so that editing a comment keeps a record valid."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(name):
    """The kernel's source file with the library headers it compiles in
    (code only: comments and whitespace do not count)."""
    d = os.path.join(ROOT, "quantized_speculative_decoding_shared_gb300", "csrc")
    h = hashlib.sha256()
    for f in (name, "qspec_device.cuh", "qspec_host.h"):
        h.update(_code_only(open(os.path.join(d, f)).read()).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def recorded_traffic(kernel_file):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current source of the kernel; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        d = json.load(open(p))
        e = d[kernel_file]
        if e.get("source_sha256_16") == kernel_source_hash(kernel_file):
            return e
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            t = [v.strip() for v in line.split(",")]
            if len(t) >= 9:
                rows.append(t)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# the round on the GPU
# ---------------------------------------------------------------------------
class GpuRound(QspecRound):
    """The library's round harness on a bench workload, plus the algorithmic
    bytes of its passes (for the roofline)."""

    def __init__(self, wl, dev):
        super().__init__(wl["shape"], wl["B"], wl["gamma"], wl["T"], wl["seed"], dev,
                         outliers=wl["outliers"], p_std=wl["p_std"], q_noise=wl["q_noise"])

    def draft_linears_only(self, j=0):
        self.draft_linears(j)

    def verify_linears_only(self):
        self.verify_linears()

    def bytes_draft_linears(self):
        b = sum(bytes_w4a4_bf16(self.B, N, K) for _, N, K in self.linears) * self.L
        return b + bytes_w4a4_bf16(self.B, self.V, self.hidden)

    def bytes_verify_linears(self):
        Mv = self.B * (self.gamma + 1)
        b = sum(bytes_w4a16(Mv, N, K) for _, N, K in self.linears) * self.L
        return b + bytes_w4a16(Mv, self.V, self.hidden)


def aggregate_over_ranks(seconds, tokens, device):
    """Whole-job figures over the ranks of a weak-scaling run: the slowest
    rank's time and the tokens of all ranks.  One rank: unchanged."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(seconds), int(tokens)
    t = torch.tensor([float(seconds), float(tokens)], dtype=torch.float64, device=device)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(mx[0]), int(round(float(t[1])))


def row_kernels(dev, stream, reps=5, calls=10):
    """Every hot-path row timed on its own at a representative size (CUDA
    graph replays of `calls` back-to-back calls, CUDA events; per call, so the
    graph launch is spread over the calls as in a longer pipeline):
    algorithmic bytes per call, GB/s, fraction of the measured HBM
    bandwidth."""
    from quantized_speculative_decoding_shared_gb300 import binding as q
    peak, _ = measured_peaks()
    out = {}

    def rec(name, fn, nbytes, note):
        fn()
        torch.cuda.synchronize()

        def many():
            for _ in range(calls):
                fn()
        g = capture(many, stream)
        t = time_graph(g, reps, stream) / calls
        out[name] = {"case": note, "us": round(t * 1e3, 2), "bytes": int(nbytes),
                     "GB/s": round(nbytes / (t / 1e3) / 1e9, 1),
                     "frac_hbm": round(nbytes / (t / 1e3) / 1e9 / peak, 4)}
        del g

    N, K = 128256, 4096
    codes, s_, z_ = syn.weights(N, K, 91, device=dev)
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
    sz = torch.empty((N, K // GROUP), dtype=torch.int32, device=dev)
    rec("a1_pack", lambda: q.qspec_pack_weights(codes, s_, z_, N, K, packed, sz),
        N * K + 4 * N * K // GROUP + N * K // 2 + 4 * N * K // GROUP, "128256 x 4096 (LM head)")
    del codes, s_, z_, packed, sz
    M, K = 4096, 14336
    x = syn.activations(M, K, 92, device=dev)
    xq = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    sx = torch.empty((M, K // GROUP), dtype=torch.float32, device=dev)
    qs = torch.empty((M, K // GROUP), dtype=torch.int32, device=dev)
    rec("a2_quant_act_int4", lambda: q.qspec_quant_act_int4(x, M, K, K, xq, sx, qs),
        bytes_quant(M, K), "4096 x 14336")
    del x, xq, sx, qs
    B, g, V = 16, 4, 128256
    P, Q, d = syn.logits_noisy_draft(B, g, V, 93, device=dev)
    ws = q.verify_workspace(256, g, V, dev)
    n_acc = torch.empty(256, dtype=torch.int32, device=dev)
    o = torch.empty((256, g + 1), dtype=torch.int32, device=dev)
    rec("a5_verify_greedy", lambda: q.qspec_verify_greedy(P, d, B, g, V, n_acc, o, ws, ws.numel()),
        2 * B * (g + 1) * V, "B 16, gamma 4, V 128256")
    del P, Q, d
    B = 256
    P, Q, d = syn.logits_noisy_draft(B, g, V, 94, device=dev)
    rec("a6_verify_sample", lambda: q.qspec_verify_sample(P, Q, d, B, g, V, 5, 0, n_acc, o, ws, ws.numel()),
        2 * B * (2 * g + 1) * V, "B 256, gamma 4, V 128256")
    del P, Q, d, ws
    B = 16
    Qd = syn.logits_noisy_draft(B, 1, V, 98, device=dev)[1][:, 0, :].contiguous()
    dws = q.draft_workspace(B, V, dev)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    conf = torch.empty(B, dtype=torch.float32, device=dev)
    ent = torch.empty(B, dtype=torch.float32, device=dev)
    rec("next_draft_sample", lambda: q.qspec_draft_sample(Qd, B, V, 5, 0, 1, tok, conf, ent, dws, dws.numel()),
        2 * B * V, "B 16, V 128256, one draft position: token, confidence, entropy")
    del Qd, dws
    L, B, H, T, D = 32, 16, 8, 4096, 128
    kc, vc = syn.kv_cache(L, B, H, T, D, 95, device=dev)
    kn, vn = syn.kv_new(L, B, g, H, D, 96, device=dev)
    base = syn.base_positions(B, T, g, 97, device=dev)
    na = torch.full((B,), g, dtype=torch.int32, device=dev)
    rec("a7_kv_overwrite", lambda: q.qspec_kv_overwrite(kc, vc, kn, vn, base, na, L, B, H, T, D, g),
        2 * 2 * 2 * L * B * (g + 1) * H * D, "32 layers x 16 seq x 8 heads x 4096 x 128, all 4 drafts accepted")
    del kc, vc, kn, vn
    torch.cuda.synchronize()
    return out


def targets(rnd_obj, dev, stream, reps=5):
    """The two explicit performance targets, measured in the same run:
    W4A16 verify linears at M <= 64 (and 80) against HBM, the W4A4 draft
    linears at decode M against HBM, and the W4A4 prefill GEMM at M = 4096
    against the E4M3 tensor peak.  The linears are one Llama-3-8B layer's
    (q/k/v, o, gate/up, down) plus the LM head, 390 MB of packed weights, so
    every replay streams from HBM (larger than L2); CUDA-graph replays of one
    call per linear, CUDA events on the launching stream."""
    from quantized_speculative_decoding_shared_gb300 import binding as q
    peak, kind = measured_peaks()
    linears = [(name, N, K, rnd_obj.w[0][name]) for name, N, K in rnd_obj.linears]
    linears.append(("lm_head", rnd_obj.V, rnd_obj.hidden, rnd_obj.lm))
    out = {"peak_hbm_GBs": peak, "peak_source": kind,
           "shapes": "Llama-3-8B layer (qkv 4096->6144, o 4096->4096, gate/up 4096->28672, down 14336->4096) "
                     "+ LM head 4096->128256"}

    def run(fn_list, nbytes):
        for f in fn_list:
            f()
        torch.cuda.synchronize()

        def all_calls():
            for f in fn_list:
                f()
        g = capture(all_calls, stream)
        t = time_graph(g, reps, stream)
        del g
        return t, nbytes / (t / 1e3) / 1e9

    w16 = {}
    for M in (5, 16, 32, 64, 80):
        fns, nbytes = [], 0
        for j, (name, N, K, pk) in enumerate(linears):
            x = syn.activations(M, K, 200 + j, device=dev, outlier_frac=0.01)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            fns.append(lambda x=x, y=y, pk=pk, N=N, K=K, M=M: q.qspec_linear_w4a16(x, K, pk[0], pk[1], M, N, K,
                                                                                   y, N))
            nbytes += bytes_w4a16(M, N, K)
        t, gbs = run(fns, nbytes)
        w16["M%d" % M] = {"ms": round(t, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peak, 4)}
    out["w4a16_verify"] = dict(w16, target="frac_hbm >= 0.70 for M <= 64")
    w4 = {}
    for M in (1, 16, 32):
        fns, nbytes = [], 0
        for j, (name, N, K, pk) in enumerate(linears):
            x = syn.activations(M, K, 300 + j, device=dev, outlier_frac=0.01)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            xq = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
            sx = torch.empty((M, K // GROUP), dtype=torch.float32, device=dev)
            qs = torch.empty((M, K // GROUP), dtype=torch.int32, device=dev)
            fns.append(lambda x=x, y=y, pk=pk, N=N, K=K, M=M, xq=xq, sx=sx, qs=qs:
                       q.qspec_linear_w4a4_bf16(x, K, pk[0], pk[1], M, N, K, y, N, xq, sx, qs))
            nbytes += bytes_w4a4_bf16(M, N, K)
        t, gbs = run(fns, nbytes)
        w4["M%d" % M] = {"ms": round(t, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peak, 4)}
    out["w4a4_draft"] = w4
    # SpecQuant Q8 verify: FP8 weights derived from an FP16 parent of the same
    # shapes, per-token E4M3 activations, the FP8 linear (two calls per linear)
    q8 = {}
    fp8w = []
    for j, (name, N, K, _) in enumerate(linears):
        g = torch.Generator(device=dev).manual_seed(500 + j)
        w16 = (torch.randn((N, K), generator=g, device=dev) * 0.02).to(torch.float16)
        fp8w.append((name, N, K) + q.quant_weights_fp8(w16))
        del w16
    for M in (5, 80):
        fns, nbytes = [], 0
        for j, (name, N, K, w8, s8) in enumerate(fp8w):
            x = syn.activations(M, K, 600 + j, device=dev, outlier_frac=0.01)
            xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
            sa = torch.empty(M, dtype=torch.float32, device=dev)
            y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            fns.append(lambda x=x, xq=xq, sa=sa, K=K, M=M: q.qspec_quant_act_fp8(x, M, K, K, xq, sa))
            fns.append(lambda xq=xq, sa=sa, w8=w8, s8=s8, y=y, N=N, K=K, M=M:
                       q.qspec_linear_fp8(xq, sa, w8, s8, M, N, K, y, N))
            nbytes += N * K + 4 * N + 2 * M * K + M * K + 4 * M + M * K + 2 * M * N
        t, gbs = run(fns, nbytes)
        q8["M%d" % M] = {"ms": round(t, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peak, 4)}
    del fp8w
    out["q8_fp8_verify"] = dict(q8, bytes="E4M3 weights 1 byte each + scales; activations quantised per call")
    # prefill: M = 4096 through gate/up and down
    M = 4096
    bf16, bkind = measured_bf16_tflops()
    e4m3 = 2.0 * bf16
    fns4, fns16, flops = [], [], 0
    for j, (name, N, K, pk) in enumerate(linears):
        if name not in ("gate_up_proj", "down_proj"):
            continue
        x = syn.activations(M, K, 400 + j, device=dev)
        xq, sx, qs = q.quant_act_int4(x)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fns4.append(lambda xq=xq, sx=sx, qs=qs, pk=pk, y=y, N=N, K=K:
                    q.qspec_linear_w4a4(xq, sx, qs, pk[0], pk[1], M, N, K, y, N))
        fns16.append(lambda x=x, pk=pk, y=y, N=N, K=K: q.qspec_linear_w4a16(x, K, pk[0], pk[1], M, N, K, y, N))
        flops += 2 * M * N * K
    t4, _ = run(fns4, 0)
    t16, _ = run(fns16, 0)
    tops = flops / (t4 / 1e3) / 1e12
    tf16 = flops / (t16 / 1e3) / 1e12
    out["w4a4_prefill_m4096"] = {
        "ms": round(t4, 4), "TOPS": round(tops, 1),
        "peak_e4m3_TFLOPs": round(e4m3, 1),
        "peak_source": "%s bf16 dense burst x 2 (the nominal e4m3 / bf16 ratio)" % bkind,
        "frac": round(tops / e4m3, 4),
        "frac_of_e4m3_probe": round(tops / E4M3_PROBE_TFLOPS, 4),
        "target": "frac >= 0.50"}
    out["w4a16_prefill_m4096"] = {"ms": round(t16, 4), "TFLOPs": round(tf16, 1), "peak_bf16_TFLOPs": bf16,
                                  "frac": round(tf16 / bf16, 4)}
    torch.cuda.synchronize()
    return out


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def time_graph(g, reps, stream):
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        torch.cuda.synchronize()
        s.record(stream)
        for _ in range(reps):
            g.replay()
        e.record(stream)
    e.synchronize()
    return s.elapsed_time(e) / reps


# ---------------------------------------------------------------------------
# CPU oracle: a bounded sample of the same round, extrapolated
# ---------------------------------------------------------------------------
class OracleRound:
    """One layer of each pass, an LM-head row slice and the full verification
    are run by the oracle; the round time is extrapolated to all layers and
    rows (layers are identical in shape, rows of a linear are independent)."""

    def __init__(self, wl, lm_rows=2048):
        import oracle
        self.o = oracle
        self.wl = wl
        sh = wl["shape"]
        self.B, self.gamma, self.L, self.V = wl["B"], wl["gamma"], sh["layers"], sh["vocab"]
        self.hidden = sh["hidden"]
        self.linears = syn.fused_layer_linears(sh)
        self.lm_rows = lm_rows
        seed = wl["seed"]
        self.packs = {}
        for j, (name, N, K) in enumerate(self.linears):
            codes, s, z = syn.weights(N, K, seed * 100003 + j)
            st, p, szz = oracle.pack_weights(codes.numpy(), syn.bits16(s), syn.bits16(z))
            self.packs[name] = (p, szz)
        codes, s, z = syn.weights(lm_rows, self.hidden, seed * 100003 + 7777)
        st, p, szz = oracle.pack_weights(codes.numpy(), syn.bits16(s), syn.bits16(z))
        self.lm = (p, szz)
        Mv = self.B * (self.gamma + 1)
        self.xd = {n: syn.bits16(syn.activations(self.B, K, seed * 7 + j, outlier_frac=wl["outliers"]))
                   for j, (n, _, K) in enumerate(self.linears)}
        self.xv = {n: syn.bits16(syn.activations(Mv, K, seed * 11 + j, outlier_frac=wl["outliers"]))
                   for j, (n, _, K) in enumerate(self.linears)}
        self.xd_lm = syn.bits16(syn.activations(self.B, self.hidden, seed * 13))
        self.xv_lm = syn.bits16(syn.activations(Mv, self.hidden, seed * 17))
        P, Q, d = syn.logits_noisy_draft(self.B, self.gamma, self.V, seed * 19,
                                         p_std=wl["p_std"], q_noise=wl["q_noise"])
        self.P, self.Q, self.d = syn.bits16(P), syn.bits16(Q), d.numpy()
        H, D, T = sh["kv_heads"], sh["head_dim"], wl["T"]
        kc, vc = syn.kv_cache(1, self.B, H, T, D, seed * 23)
        kn, vn = syn.kv_new(1, self.B, self.gamma, H, D, seed * 29)
        self.kc, self.vc = syn.bits16(kc).copy(), syn.bits16(vc).copy()
        self.kn, self.vn = syn.bits16(kn), syn.bits16(vn)
        self.base = syn.base_positions(self.B, T, self.gamma, seed * 31).numpy()

    def step(self, rnd):
        o, t0 = self.o, time.perf_counter
        a = t0()
        for name, N, K in self.linears:                       # one layer, one draft step
            st, xq, sx, qs = o.quant_act_int4(self.xd[name])
            o.linear_w4a4(xq, sx, *self.packs[name])
        b = t0()
        st, xq, sx, qs = o.quant_act_int4(self.xd_lm)
        o.linear_w4a4(xq, sx, *self.lm)                       # LM-head row slice
        c = t0()
        for name, N, K in self.linears:                       # one layer, verify pass
            o.linear_w4a16(self.xv[name], *self.packs[name])
        d = t0()
        o.linear_w4a16(self.xv_lm, *self.lm)
        e = t0()
        st, n_acc, out = o.verify_sample(self.P, self.Q, self.d, 1234, rnd)
        f = t0()
        o.kv_overwrite(self.kc, self.vc, self.kn, self.vn, self.base, n_acc, self.gamma)
        g = t0()
        scale = self.V / self.lm_rows
        t_round = (self.gamma * (self.L * (b - a) + (c - b) * scale) + self.L * (d - c)
                   + (e - d) * scale + (f - e) + self.L * (g - f))
        sampled = (b - a) + (c - b) + (d - c) + (e - d) + (f - e) + (g - f)
        return int((n_acc + 1).sum()), t_round, sampled


def cpu_model():
    """The host CPU's model string, from /proc/cpuinfo (or lscpu)."""
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(wl, steps=3):
    """The oracle on the host cores (all of them, then one thread) on a
    bounded sample of the round, extrapolated to the whole round."""
    import oracle
    orc = OracleRound(wl)
    orc.step(0)
    tok = tsum = sampled = 0.0
    for r in range(steps):
        k, t, s = orc.step(r)
        tok, tsum, sampled = tok + k, tsum + t, sampled + s
    cores = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        k1, t1, s1 = orc.step(steps)
    finally:
        oracle.set_num_threads(cores)
    return {"value": tok / tsum, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(), "single_thread_value": k1 / t1,
            "sample": ("%d rounds; per round 1 of %d layers (draft and verify linears), LM head "
                       "%d of %d rows, full verification and 1-layer KV overwrite, extrapolated "
                       "to the full round; %.1f s of oracle time measured on %d threads, then one "
                       "round on 1 thread (%.1f s)"
                       % (steps, orc.L, orc.lm_rows, orc.V, sampled, cores, s1))}


# ---------------------------------------------------------------------------
def prefill_numbers(dev, steps, warmup):
    """M = 4096 tokens through Llama-3-8B gate/up (4096 -> 14336, stacked as
    28672) and down (14336 -> 4096): W4A4 on the tensor cores (TOPS, exact
    integer products) and W4A16 (bf16 tensor cores); plus batch-256 sampled
    verification over 128256 tokens at gamma 4. Returns the timings."""
    from quantized_speculative_decoding_shared_gb300 import binding as q
    M = 4096
    shapes = [("gate_up_proj", 28672, 4096), ("down_proj", 4096, 14336)]
    mats = {}
    for j, (name, N, K) in enumerate(shapes):
        codes, s_, z_ = syn.weights(N, K, 40 + j, device=dev)
        mats[name] = q.pack_weights(codes, s_, z_)
        del codes
    xs = {name: syn.activations(M, K, 50 + j, device=dev) for j, (name, N, K) in enumerate(shapes)}
    qx = {name: q.quant_act_int4(xs[name]) for name, _, _ in shapes}
    ys = {name: torch.empty((M, N), dtype=torch.bfloat16, device=dev) for name, N, _ in shapes}
    stream = torch.cuda.Stream(device=dev)

    def run4():
        for name, N, K in shapes:
            xq, sx, qs = qx[name]
            q.linear_w4a4(xq, sx, qs, *mats[name], out=ys[name])

    def run16():
        for name, N, K in shapes:
            q.linear_w4a16(xs[name], *mats[name], out=ys[name])

    with torch.cuda.stream(stream):
        run4(); run16()
    torch.cuda.synchronize()
    flops = sum(2 * M * N * K for _, N, K in shapes)
    g4, g16 = capture(run4, stream), capture(run16, stream)
    for _ in range(warmup):
        time_graph(g4, 1, stream)
    clocks = ClockSampler(dev.index)
    clocks.start()
    t4 = time_graph(g4, steps, stream)
    t16 = time_graph(g16, steps, stream)
    clk = clocks.stop()
    P, Q, d = syn.logits_noisy_draft(256, 4, 128256, 4, device=dev)
    ws = q.verify_workspace(256, 4, 128256, dev)
    gv = capture(lambda: q.verify_sample(P, Q, d, 1, 0, workspace=ws), stream)
    tv = time_graph(gv, steps, stream)
    vbytes = 2 * 256 * 9 * 128256
    peak_hbm, _ = measured_peaks()
    return {"M": M, "shapes": shapes, "w4a4_TOPS": round(flops / (t4 / 1e3) / 1e12, 2),
            "w4a4_ms": round(t4, 4),
            "w4a16_TFLOPS": round(flops / (t16 / 1e3) / 1e12, 2), "w4a16_ms": round(t16, 4),
            "verify_b256_g4": {"ms": round(tv, 4), "GB/s": round(vbytes / (tv / 1e3) / 1e9, 1),
                               "frac_hbm": round(vbytes / (tv / 1e3) / 1e9 / peak_hbm, 4)},
            "clocks": clk}


def prefill_bench(args):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    r = prefill_numbers(dev, args.steps, args.warmup)
    line = {"metric": "W4A4 INT TOPS (M = 4096)", "value": r["w4a4_TOPS"],
            "unit": "TOPS", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": r["w4a4_ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int4 x int4 -> exact (e4m3 tensor operands, fp32 = exact int)",
            "data": "synthetic", "config": {"workload": PREFILL, "M": r["M"], "shapes": r["shapes"]},
            "w4a16": {"TFLOPS": r["w4a16_TFLOPS"], "ms": r["w4a16_ms"]},
            "verify_b256_g4": r["verify_b256_g4"], "clocks": r["clocks"]}
    print(json.dumps(line))


def timed_rounds(rnd_obj, stream, R, warmup, steps, barrier=lambda: None, clocks=None):
    """Eager round (status check), R captured round graphs, W warm-up replays,
    then K timed replays with CUDA events on the launching stream. Returns
    (graphs, launches per round, device ms, accepted tokens, clock record)."""
    from quantized_speculative_decoding_shared_gb300 import binding as qb
    acc_log = torch.zeros((R, rnd_obj.B), dtype=torch.int32, device=rnd_obj.dev)
    # eager round first: sets kernel attributes outside capture, checks status
    with torch.cuda.stream(stream):
        rnd_obj.run(0)
    torch.cuda.synchronize()
    if int(rnd_obj.status.item()) != 0:
        raise RuntimeError("device status %d after the eager round" % int(rnd_obj.status.item()))
    # the library's own count of the kernels one round launches (read around
    # the capture of the first round's graph)
    n_before = qb.qspec_kernel_launches()
    graphs = [capture(lambda: rnd_obj.run(0, acc_log[0]), stream)]
    launches_per_round = qb.qspec_kernel_launches() - n_before
    graphs += [capture(lambda r=r: rnd_obj.run(r, acc_log[r]), stream) for r in range(1, R)]
    with torch.cuda.stream(stream):
        # setup: the first launch of a captured graph also uploads it, so
        # every graph is launched once before the warm-up steps
        for gr in graphs:
            gr.replay()
        for i in range(warmup):
            graphs[i % R].replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(steps):
            graphs[i % R].replay()
        ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    barrier()
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop() if clocks is not None else None
    acc = acc_log.cpu().numpy()
    tokens = int(sum((acc[i % R] + 1).sum() for i in range(steps)))
    if int(rnd_obj.status.item()) != 0:
        raise RuntimeError("device status %d" % int(rnd_obj.status.item()))
    return graphs, launches_per_round, ms, tokens, clk


def other_workloads(names, dev, steps=10, warmup=3, R=4):
    """Short timed runs of the other decode workloads (one at a time, memory
    released in between) and of the M = 4096 prefill linears, so that one
    default run carries a device-timed figure for every configuration."""
    out = {}
    stream = torch.cuda.Stream(device=dev)
    for name in names:
        wl = WORKLOADS[name]
        rnd_obj = GpuRound(wl, dev)
        clocks = ClockSampler(dev.index)
        graphs, lpr, ms, tokens, clk = timed_rounds(rnd_obj, stream, R, warmup, steps,
                                                    clocks=clocks)
        t4 = time_graph(capture(rnd_obj.draft_linears_only, stream), 5, stream)
        t16 = time_graph(capture(rnd_obj.verify_linears_only, stream), 5, stream)
        out[name] = {"value": round(tokens / (ms / 1e3), 2), "unit": "tokens/s",
                     "steps": steps, "warmup": warmup, "ms_per_step": round(ms / steps, 4),
                     "tokens_per_step": tokens / steps, "batch": wl["B"], "gamma": wl["gamma"],
                     "gpu_launches": lpr * steps,
                     "draft_step_linears_ms": round(t4, 4), "M_draft": wl["B"],
                     "verify_pass_linears_ms": round(t16, 4),
                     "M_verify": wl["B"] * (wl["gamma"] + 1),
                     "clocks": {k: clk.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")}}
        del graphs, rnd_obj
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    r = prefill_numbers(dev, steps, warmup)
    clk = r.pop("clocks")
    r["clocks"] = {k: clk.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")}
    out[PREFILL] = r
    torch.cuda.empty_cache()
    return out


def main():
    args = parse_args()
    if args.profile_case:
        profile_case(args.profile_case, args.profile_reps)
        return
    if args.workload == PREFILL:
        prefill_bench(args)
        return
    wl = WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    sh = wl["shape"]
    cfg = {"workload": args.workload, "model_shape": "%d layers, %d hidden, %d vocab" % (
           sh["layers"], sh["hidden"], sh["vocab"]), "batch": wl["B"], "gamma": wl["gamma"],
           "l2": "inputs larger than L2 (every step reads all packed weights, ~4 GB)",
           "parallelism": "replicas x%d" % args.gpus}

    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        orc = OracleRound(wl)
        for r in range(args.warmup):
            orc.step(r)
        tok = tsum = sampled = 0.0
        for r in range(args.steps):
            k, t, s = orc.step(args.warmup + r)
            tok, tsum, sampled = tok + k, tsum + t, sampled + s
        v = tok / tsum
        line = {"impl": "reference", "metric": "accepted tokens/s", "value": v, "unit": "tokens/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * tsum / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "int4 weights; u64/u128 sums",
                "data": "synthetic", "config": cfg,
                "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": oracle.num_threads(),
                                 "kind": "oracle", "cpu_model": cpu_model(),
                                 "sample": "per step 1 of %d layers, LM head %d of %d rows, full "
                                           "verification; %.1f s of oracle time in total"
                                           % (orc.L, orc.lm_rows, orc.V, sampled)},
                "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from quantized_speculative_decoding_shared_gb300 import build as qbuild
    if not os.path.exists(os.path.join(ROOT, "quantized_speculative_decoding_shared_gb300", "_lib",
                                       "libqspec.so")):
        qbuild.build()
    rnd_obj = GpuRound(wl, dev)
    stream = torch.cuda.Stream(device=dev)
    R = max(1, args.rounds)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    graphs, launches_per_round, ms, tokens, clk = timed_rounds(
        rnd_obj, stream, R, args.warmup, args.steps, barrier, ClockSampler(local))
    sec, tokens = aggregate_over_ranks(ms / 1e3, tokens, dev)
    ms = sec * 1e3
    value = tokens / sec

    # dominant kernel: one draft step's W4A4 linears, graph-replayed alone
    g4 = capture(rnd_obj.draft_linears_only, stream)
    g16 = capture(rnd_obj.verify_linears_only, stream)
    reps = 10
    t4 = time_graph(g4, reps, stream)
    t16 = time_graph(g16, reps, stream)
    n4 = rnd_obj.L * len(rnd_obj.linears) + 1
    peak, peak_kind = measured_peaks()
    ach4 = rnd_obj.bytes_draft_linears() / (t4 / 1e3) / 1e9
    ach16 = rnd_obj.bytes_verify_linears() / (t16 / 1e3) / 1e9
    one_token = wl["B"] == 1
    traffic = recorded_traffic("w4a4_dp4a.cu") if one_token else None
    roofline = {"bound": "hbm",
                "kernel": ("w4a4_dp4a_gemv_kernel (W4A4 linear, M = 1)" if one_token
                           else "W4A4 linears, M = %d" % wl["B"]),
                "achieved": round(ach4, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach4 / peak, 4), "peak_source": peak_kind,
                "bytes_per_launch": rnd_obj.bytes_draft_linears() / n4,
                "launch_us": 1e3 * t4 / n4,
                # ncu DRAM bytes of one captured launch (the LM head at this M),
                # scaled by algorithmic bytes to the average launch above
                "traffic": (round(traffic["dram_bytes_per_algorithmic_byte"] *
                                  rnd_obj.bytes_draft_linears() / n4)
                            if traffic else None)}

    # e2e: host buffers, copies inside the timed region
    host_in = [t.cpu().pin_memory() for t in rnd_obj.host_inputs()]
    dev_in = rnd_obj.host_inputs()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    out_host = torch.empty_like(rnd_obj.out, device="cpu").pin_memory()
    nacc_host = torch.empty_like(rnd_obj.n_acc, device="cpu").pin_memory()
    d2h = out_host.numel() * 4 + nacc_host.numel() * 4
    e2e_tokens = 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            for hsrc, ddst in zip(host_in, dev_in):
                ddst.copy_(hsrc, non_blocking=True)
            graphs[i % R].replay()
            out_host.copy_(rnd_obj.out, non_blocking=True)
            nacc_host.copy_(rnd_obj.n_acc, non_blocking=True)
            stream.synchronize()
            e2e_tokens += int((nacc_host + 1).sum())
    t_e2e = time.perf_counter() - t0
    t_e2e, e2e_tokens = aggregate_over_ranks(t_e2e, e2e_tokens, dev)

    if rank != 0:
        return
    line = {"metric": "accepted tokens/s", "value": round(value, 2), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int4 w; int32 acc (W4A4) / bf16 x "
            "fp32 acc (W4A16); u64/u128 integer verification", "data": "synthetic",
            "config": cfg, "tokens_per_step": tokens / args.steps / world,
            "e2e": {"value": round(e2e_tokens / t_e2e, 2), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "roofline": roofline,
            "kernels": {"w4a4_draft_linears": {"GB/s": round(ach4, 1), "frac_hbm": round(ach4 / peak, 4),
                                               "ms_per_draft_step": round(t4, 4), "M": wl["B"]},
                        "w4a16_verify_linears": {"GB/s": round(ach16, 1),
                                                 "frac_hbm": round(ach16 / peak, 4),
                                                 "ms_per_verify_pass": round(t16, 4),
                                                 "M": wl["B"] * (wl["gamma"] + 1)}},
            "rows": row_kernels(dev, stream),
            "targets": targets(rnd_obj, dev, stream),
            "gpu_launches": launches_per_round * args.steps,
            "clocks": clk}
    if world == 1 and args.workload == DEFAULT_WORKLOAD and not args.no_workloads:
        del graphs, g4, g16, rnd_obj, dev_in
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        line["workloads"] = other_workloads([n for n in WORKLOADS if n != args.workload], dev)
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    print(json.dumps(line))


if __name__ == "__main__":
    main()
