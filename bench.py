"""Benchmark of the Q4_K x Q8_1 decode hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl rz|reference]
                    [--workload stack|gemv] [--batch M] [--position P]

Workloads (synthetic, seeded; rz_synth):
  stack  one decode step of the 32-layer Llama-7B-shaped Q4_K stack (hidden 4096,
         intermediate 11008, 32 heads, head_dim 128, f32 KV cache at position P,
         M tokens) plus output RMSNorm and the Q4_0 LM head 32000 x 4096.
  gemv   one Q4_K x Q8_1 GEMV 4096 x 14336 (M tokens), weights rotated through
         copies larger than twice the L2.

One JSON line on stdout (rank 0).  `value` is the achieved HBM bandwidth of the
whole step: algorithmic bytes (quantised weights + activations + KV cache read
+ outputs) / device time, summed over ranks.  Multi-GPU runs are independent
replicas (the path has no exchange step): `scaling` is weak.
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

import numpy as np  # noqa: E402

import rz_synth as S  # noqa: E402

METRIC = "Q4_K×Q8_1 GEMV achieved HBM GB/s (% of GB300 peak); decode tokens/s/layer stack"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


# ----------------------------------------------------------------------------- helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak() -> float:
    """Dense 16-bit tensor peak in TFLOP/s: the measured bf16 burst figure (f16
    runs at the same rate), else the fallback 1900."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def profile_traffic(kernel_file: str, workload: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on the
    current source of the kernel (sha256 of the .cu file), else None."""
    src = os.path.join(ROOT, "quantized_q4_q8_gb300", "csrc", kernel_file)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for fn in sorted(os.listdir(os.path.join(ROOT, "profiles"))) if os.path.isdir(
            os.path.join(ROOT, "profiles")) else []:
        if not fn.endswith((".md", ".txt")):
            continue
        txt = open(os.path.join(ROOT, "profiles", fn)).read()
        m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", txt)
        m_wl = re.search(r"workload:\s*(\S+)", txt)
        m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", txt)
        if m_sha and m_tr and m_wl and m_sha.group(1) == sha and m_wl.group(1) == workload:
            return int(m_tr.group(1))
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
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
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if _cuda_ok() else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def _cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, v: float, device) -> float:
    if pg is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- workloads
def gemv_bytes(out_dim: int, in_dim: int, m: int) -> int:
    """Algorithmic bytes of one Q4_K x Q8_1 GEMV: quantised weights + Q8_1
    activations (1.25 B per value) + f32 outputs."""
    return out_dim * (in_dim // 256) * S.Q4K_BYTES + m * in_dim * 5 // 4 + m * out_dim * 4


def time_graph(graph, stream, reps: int) -> float:
    """ms per replay of a captured graph, CUDA events on the launching stream."""
    import torch
    graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def capture(fn, stream):
    """fn() once eagerly (kernel attributes), then captured into a CUDA graph."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


def measure_gemv(rz, out_dim: int, in_dim: int, m: int, dev, stream, launches: int = 64,
                 reps: int = 30):
    """One Q4_K x Q8_1 GEMV shape timed as back-to-back launches in a CUDA graph, the
    weights rotated through distinct copies larger than twice the L2 together (no
    launch finds its weights in L2).  Returns us per launch, GB/s, copies."""
    import torch
    wbytes = out_dim * (in_dim // 256) * S.Q4K_BYTES
    ncopies = max(2, int(np.ceil(2 * L2_BYTES / wbytes)) + 1)
    w0 = S.q4k_weight_device(f"sweep.{out_dim}.{in_dim}", out_dim, in_dim, dev)
    ws = [w0] + [w0.clone() for _ in range(ncopies - 1)]
    x = torch.randn((m, in_dim), device=dev, generator=S.torch_gen(f"sweep.x.{in_dim}.{m}", dev))
    q8 = rz.q8_1_quantize(x)
    y = torch.empty((m, out_dim), dtype=torch.float32, device=dev)

    def launch():
        for i in range(launches):
            rz.rz_q4k_q8_gemv(ws[i % ncopies], q8, y, m, out_dim, in_dim, stream=stream)

    g = capture(launch, stream)
    ms = time_graph(g, stream, reps) / launches
    del g, ws
    us = ms * 1e3
    return {"us": round(us, 3), "gbs": round(gemv_bytes(out_dim, in_dim, m) / (ms * 1e-3) / 1e9, 1),
            "weight_copies": ncopies}


def measure_gemm(rz, out_dim: int, in_dim: int, m: int, dev, stream, launches: int = 8, reps: int = 10):
    """The many-token tensor-core product (rz_q4k_q8_gemm: operand packing + the
    tcgen05 GEMM) for one shape, timed like measure_gemv.  Returns us per call and
    TFLOP/s of the integer-dot work (2 m out in) and of what the tensor cores
    execute (9/8 of it: the min-term product)."""
    import torch
    wbytes = out_dim * (in_dim // 256) * S.Q4K_BYTES
    ncopies = max(2, int(np.ceil(2 * L2_BYTES / wbytes)) + 1)
    w0 = S.q4k_weight_device(f"sweep.{out_dim}.{in_dim}", out_dim, in_dim, dev)
    ws = [w0] + [w0.clone() for _ in range(ncopies - 1)]
    x = torch.randn((m, in_dim), device=dev, generator=S.torch_gen(f"gemm.x.{in_dim}.{m}", dev))
    q8 = rz.q8_1_quantize(x)
    y = torch.empty((m, out_dim), dtype=torch.float32, device=dev)
    wsb = rz.q4k_q8_gemm_workspace_bytes(m, in_dim)
    work = torch.empty(wsb, dtype=torch.uint8, device=dev)

    def launch():
        for i in range(launches):
            rz.rz_q4k_q8_gemm(ws[i % ncopies], q8, y, out_dim, m, out_dim, in_dim, work, wsb, stream=stream)

    g = capture(launch, stream)
    ms = time_graph(g, stream, reps) / launches
    del g, ws
    flops = 2.0 * m * out_dim * in_dim
    return {"us": round(ms * 1e3, 2), "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
            "tensor_tflops": round(1.125 * flops / (ms * 1e-3) / 1e12, 1), "weight_copies": ncopies}


class GemvWorkload:
    """Q4_K x Q8_1 GEMV, out 4096 x in 14336 (the largest shape of the Llama sweep),
    launched back to back over weight copies larger than twice the L2."""
    out_dim, in_dim = 4096, 14336
    kernel_file = "gemv_q4k.cu"
    launches = 64

    def __init__(self, m: int):
        self.m = m
        self.name = f"q4k_q8_gemv_{self.out_dim}x{self.in_dim}_m{m}"

    def setup(self, dev):
        import torch
        import quantized_q4_q8_gb300 as rz
        self.rz = rz
        self.wbytes = self.out_dim * (self.in_dim // 256) * S.Q4K_BYTES
        self.ncopies = max(2, int(np.ceil(2 * L2_BYTES / self.wbytes)) + 1)
        w0 = S.q4k_weight_device(f"sweep.{self.out_dim}.{self.in_dim}", self.out_dim, self.in_dim, dev)
        self.ws = [w0] + [w0.clone() for _ in range(self.ncopies - 1)]
        self.x = torch.randn((self.m, self.in_dim), device=dev,
                             generator=S.torch_gen(f"sweep.x.{self.in_dim}.{self.m}", dev))
        self.q8 = rz.q8_1_quantize(self.x)
        self.y = torch.empty((self.m, self.out_dim), dtype=torch.float32, device=dev)
        self.graph = None
        # pinned host buffers for the end-to-end leg
        self.x_pin = self.x.cpu().pin_memory()
        self.y_pin = torch.empty((self.m, self.out_dim), dtype=torch.float32).pin_memory()

    def bytes_per_step(self):
        return self.launches * gemv_bytes(self.out_dim, self.in_dim, self.m)

    def launches_per_step(self):
        return self.launches

    def _launch(self, stream):
        for i in range(self.launches):
            self.rz.rz_q4k_q8_gemv(self.ws[i % self.ncopies], self.q8, self.y, self.m, self.out_dim,
                                   self.in_dim, stream=stream)

    def step(self, stream):
        if self.graph is None:
            self.graph = capture(lambda: self._launch(stream), stream)
        self.graph.replay()

    def e2e_step(self, stream):
        """host x -> device, quantise, the GEMVs, device y -> host (through the C ABI)."""
        self.x.copy_(self.x_pin, non_blocking=True)
        self.rz.rz_q8_1_quantize(self.x, self.q8, self.m, self.in_dim, stream=stream)
        self.graph.replay()
        self.y_pin.copy_(self.y, non_blocking=True)

    def e2e_bytes(self):
        return self.m * self.in_dim * 4, self.m * self.out_dim * 4

    def e2e_launches(self):
        return self.launches + 1

    def dominant(self):
        return {"kernel": "q4k_gemv_kernel", "bytes_per_launch": gemv_bytes(self.out_dim, self.in_dim, self.m),
                "launches_per_step": self.launches}

    def dominant_time(self, stream):
        return None

    def cpu_sample(self, min_seconds: float = 0.0):
        """The oracle on the same GEMV (all rows), repeated until min_seconds."""
        import oracle
        cores = oracle.use_all_cores(True)
        w = S.q4k_weight(f"sweep.{self.out_dim}.{self.in_dim}", self.out_dim, self.in_dim)
        x8 = oracle.q8_1_quantize(S.normal(f"sweep.x.{self.in_dim}.{self.m}", (self.m, self.in_dim)))
        reps, t_total = 0, 0.0
        while reps == 0 or t_total < min_seconds:
            t0 = time.perf_counter()
            oracle.q4k_q8_gemv(w, x8, self.m, self.out_dim, self.in_dim)
            t_total += time.perf_counter() - t0
            reps += 1
        dt = t_total / reps
        return {"value": gemv_bytes(self.out_dim, self.in_dim, self.m) / dt / 1e9, "unit": "GB/s",
                "cores": cores, "kind": "oracle",
                "sample": f"the whole {self.out_dim}x{self.in_dim} GEMV (m={self.m}) x {reps}, C oracle "
                          f"on {cores} host threads (rows split over threads), {dt:.3f} s each"}

    def config(self):
        return {"workload": self.name, "out_dim": self.out_dim, "in_dim": self.in_dim,
                "batch_tokens": self.m, "launches_per_step": self.launches,
                "weight_copies": self.ncopies,
                "l2": "weights rotated through copies > 2x L2"}

    def config_ref(self):
        return {"workload": self.name, "out_dim": self.out_dim, "in_dim": self.in_dim,
                "batch_tokens": self.m}

    def cpu_baseline(self):
        return self.cpu_sample(min_seconds=10.0)


class StackWorkload:
    """One decode step of the 32-layer Llama-7B-shaped Q4_K stack + Q4_0 LM head."""
    vocab = S.LLAMA_VOCAB
    max_seq = S.LLAMA_MAX_SEQ
    kernel_file = "gemv_q4k.cu"

    def __init__(self, m: int, position: int, n_layers: int = S.LLAMA_LAYERS):
        self.m = m
        self.position = position
        self.n_layers = n_layers
        self.shape = S.LLAMA7B
        # from four tokens on the step's GEMVs run on the tensor cores (mma.sync)
        self.gemv_kernel = "q4k_gemv_mma_kernel" if m >= 4 else "q4k_gemv_kernel"
        self.kernel_file = "gemv_q4k_mma.cu" if m >= 4 else "gemv_q4k.cu"
        self.name = f"llama7b_q4k_decode_stack_l{self.n_layers}_m{m}_pos{position}"

    # ---- algorithmic bytes of one step
    def weight_bytes(self):
        sh = self.shape
        return self.n_layers * (sh.weight_bytes() + 2 * sh.hidden * 4) + sh.hidden * 4 + \
            self.vocab * (sh.hidden // 32) * S.Q4_0_BYTES

    def bytes_per_step(self):
        sh, m, p = self.shape, self.m, self.position
        act = 0
        for o, i in sh.weight_shapes().values():          # Q8_1 in, f32 out per GEMV
            act += m * i * 5 // 4 + m * o * 4
        kv = m * (p + 1) * sh.kv_dim * 4 * 2 + m * sh.kv_dim * 4 * 2   # read rows 0..p, write row p
        per_layer = act + kv + 2 * m * sh.hidden_pad * 4                # layer input and output
        head = m * sh.hidden * 4 + m * self.vocab * 4
        return self.weight_bytes() + self.n_layers * per_layer + head

    def fused_gemv_bytes(self):
        """Algorithmic bytes of the step's four GEMV launches per layer, as they run
        in the step: Q|K|V (f32 input normalised and quantised inside, gamma), O
        (Q8_1 input, residual), gate/up (f32 input, gamma, h out), down (f32 h in,
        residual)."""
        sh, m = self.shape, self.m
        W = {nm: o * (i // 256) * S.Q4K_BYTES for nm, (o, i) in sh.weight_shapes().items()}
        hp, q, kv, inter = sh.hidden_pad, sh.q_dim, sh.kv_dim, sh.inter
        # input of the norm-fed GEMVs: the f32 row and gamma (normalised inside), or
        # from four tokens on the Q8_1 written by the separate norm / quantise launch
        x_in = m * hp * 4 + sh.hidden * 4 if m < 4 else m * hp * 5 // 4
        h_in = m * inter * 4 if m < 4 else m * inter * 5 // 4
        qkv = W["wq"] + W["wk"] + W["wv"] + x_in + m * (q + 2 * kv) * 4
        o = W["wo"] + m * sh.q_pad * 5 // 4 + 2 * m * hp * 4
        gu = W["wgate"] + W["wup"] + x_in + m * inter * 4
        dn = W["wdown"] + h_in + 2 * m * hp * 4
        return self.n_layers * (qkv + o + gu + dn)

    def head_bytes(self):
        sh, m = self.shape, self.m
        return self.vocab * (sh.hidden // 32) * S.Q4_0_BYTES + sh.hidden * 4 + m * sh.hidden * 4 + \
            m * self.vocab * 4

    def launches_per_step(self):
        # the library's own count: RoPE table + the launches of every layer + output
        # norm + LM head
        return self.stack.launches(self.m, with_head=True)

    def setup(self, dev):
        import torch
        import quantized_q4_q8_gb300 as rz
        self.rz = rz
        sh = self.shape
        self.dls = []
        for i in range(self.n_layers):
            w = S.layer_device(sh, f"stack.l{i}", dev)
            self.dls.append(rz.DeviceLayer(w, sh.hidden, sh.hidden_pad, sh.n_heads, sh.n_kv_heads,
                                           sh.head_dim, sh.inter, sh.eps, sh.rope_theta,
                                           sh.rope_mode))
        self.kvs = [rz.DeviceKV(*S.kv_prefill_device(sh, f"stack.kv{i}", self.max_seq,
                                                     self.position, self.m, dev))
                    for i in range(self.n_layers)]
        g = S.torch_gen("stack.out_gamma", dev)
        self.out_gamma = torch.rand(sh.hidden, device=dev, generator=g) + 0.5
        self.lm = S.q4_0_weight_device("stack.lm_head", self.vocab, sh.hidden, dev)
        self.stack = rz.DeviceStack(self.dls, self.kvs, self.out_gamma, self.lm, self.vocab)
        self.x = torch.zeros((self.m, sh.hidden_pad), dtype=torch.float32, device=dev)
        self.x[:, :sh.hidden] = torch.randn((self.m, sh.hidden), device=dev,
                                            generator=S.torch_gen("stack.x", dev))
        self.ws = rz.workspace(self.stack.workspace_bytes(self.m), dev)
        self.hid = torch.empty((self.m, sh.hidden_pad), dtype=torch.float32, device=dev)
        self.logits = torch.empty((self.m, self.vocab), dtype=torch.float32, device=dev)
        self.x_pin = self.x.cpu().pin_memory()
        self.logits_pin = torch.empty((self.m, self.vocab), dtype=torch.float32).pin_memory()
        self.graph = None
        self.gemv_graph = None

    def _launch(self, stream):
        self.rz.rz_decode_stack(self.x, self.stack, None, self.position, self.m, self.hid,
                                self.logits, self.ws, stream=stream)

    def step(self, stream):
        if self.graph is None:
            self.graph = capture(lambda: self._launch(stream), stream)
        self.graph.replay()

    def e2e_step(self, stream):
        """host hidden -> device, the whole stack, device logits -> host."""
        self.x.copy_(self.x_pin, non_blocking=True)
        self.graph.replay()
        self.logits_pin.copy_(self.logits, non_blocking=True)

    def e2e_bytes(self):
        return self.m * self.shape.hidden_pad * 4, self.m * self.vocab * 4

    def e2e_launches(self):
        return self.launches_per_step()

    def dominant(self):
        n = self.n_layers * 4
        return {"kernel": self.gemv_kernel, "bytes_per_launch": self.fused_gemv_bytes() / n,
                "launches_per_step": n,
                "what": ("the step's own four GEMV launches per layer (Q|K|V with the RMSNorm/Q8_1 "
                         "prologue, O + residual, gate/up with the norm prologue and SiLU*up, down "
                         "with the Q8_1 prologue + residual), all layers back to back in one graph"
                         if self.m < 4 else
                         "the step's own four GEMV launches per layer (Q|K|V, O + residual, gate/up with "
                         "SiLU*up, down + residual) and the separate RMSNorm / Q8_1 launches that feed "
                         "them at this batch, all layers back to back in one graph; the time of those "
                         "small launches is counted into the GEMVs'")}

    def dominant_time(self, stream, reps=20):
        """Average launch duration of the dominant kernel inside the step: the four
        GEMV launches of every layer, with the same fused prologues and epilogues the
        step runs (rz_rmsnorm_q4k_gemv, rz_q4k_q8_gemv_ex with a residual,
        rz_swiglu_ffn), replayed back to back as one CUDA graph (CUDA events on the
        stream).  The attention, the RoPE table and the LM head are left out."""
        import torch
        rz, sh, m, dev = self.rz, self.shape, self.m, self.x.device
        if self.gemv_graph is None:
            self.g_in = self.x
            self.g_qkv = torch.empty((m, sh.q_dim + 2 * sh.kv_dim), dtype=torch.float32, device=dev)
            self.g_a8 = rz.q8_1_quantize(torch.randn((m, sh.q_pad), device=dev,
                                                      generator=S.torch_gen("dom.att", dev)))
            self.g_res = torch.empty((m, sh.hidden_pad), dtype=torch.float32, device=dev)
            self.g_out = torch.empty((m, sh.hidden_pad), dtype=torch.float32, device=dev)
            self.g_ws = rz.workspace(rz.swiglu_ffn_workspace_bytes(m, sh.hidden_pad, sh.inter), dev)

            # from four tokens on the step quantises the normed input in a separate
            # launch and feeds the GEMV Q8_1 (each CTA would stage the tokens one
            # after another); the graph does what the step does
            separate = m >= 4
            self.g_x8 = torch.empty(rz.q8_1_size(m, sh.hidden_pad), dtype=torch.uint8, device=dev)

            def launch():
                for dl in self.dls:
                    t = dl.t
                    if separate:
                        rz.rz_rmsnorm(self.g_in, t["attn_gamma"], None, self.g_x8, m, sh.hidden, sh.hidden_pad,
                                      sh.eps, stream=stream)
                        rz.rz_q4k_q8_gemv_multi(self.g_x8, [t["wq"], t["wk"], t["wv"]],
                                                [sh.q_dim, sh.kv_dim, sh.kv_dim], None, self.g_qkv,
                                                sh.q_dim + 2 * sh.kv_dim, m, sh.hidden_pad, stream=stream)
                    else:
                        rz.rz_rmsnorm_q4k_gemv(self.g_in, sh.hidden_pad, t["attn_gamma"], sh.hidden, sh.eps,
                                               [t["wq"], t["wk"], t["wv"]], [sh.q_dim, sh.kv_dim, sh.kv_dim],
                                               None, self.g_qkv, sh.q_dim + 2 * sh.kv_dim, m, sh.hidden_pad,
                                               stream=stream)
                    rz.rz_q4k_q8_gemv_ex(t["wo"], self.g_a8, None, self.g_in, self.g_res, sh.hidden_pad, m,
                                         sh.hidden, sh.q_pad, stream=stream)
                    rz.swiglu_ffn(self.g_res, t["ffn_gamma"], t["wgate"], t["wup"], t["wdown"], sh.hidden,
                                  sh.hidden_pad, sh.inter, sh.eps, out=self.g_out, ws=self.g_ws,
                                  stream=stream)

            self.gemv_graph = capture(launch, stream)
        return time_graph(self.gemv_graph, stream, reps) / self.dominant()["launches_per_step"]

    def cpu_sample(self, n_sample_layers: int = 1):
        """The oracle on n_sample_layers layers of the same shape plus the LM head, one
        token, timed on this host; the step time is extrapolated from the mean layer time."""
        import oracle
        cores = oracle.use_all_cores(True)
        sh = self.shape
        kc, vc = S.kv_prefill(sh, "cpu.kv", self.position + 1, self.position, 1)
        x = S.hidden_input("cpu.x", 1, sh.hidden, sh.hidden_pad)[0]
        t_layers = []
        for li in range(n_sample_layers):
            L = S.layer(sh, f"cpu.l{li}")
            ol = oracle.LayerWeights(**L.w, attn_gamma=L.attn_gamma, ffn_gamma=L.ffn_gamma,
                                     hidden=sh.hidden, hidden_pad=sh.hidden_pad,
                                     n_heads=sh.n_heads, n_kv_heads=sh.n_kv_heads,
                                     head_dim=sh.head_dim, inter=sh.inter, eps=sh.eps,
                                     rope_theta=sh.rope_theta, rope_mode=sh.rope_mode)
            t0 = time.perf_counter()
            x = oracle.decode_layer(x, ol, kc[0], vc[0], self.position)
            t_layers.append(time.perf_counter() - t0)
        lm = S.q4_0_weight("cpu.lm", self.vocab, sh.hidden)
        t0 = time.perf_counter()
        oracle.q4_0_gemv(lm, x[:sh.hidden], self.vocab, sh.hidden)
        t_head = time.perf_counter() - t0
        t_layer = sum(t_layers) / len(t_layers)
        t_step = (self.n_layers * t_layer + t_head) * self.m
        one_token = StackWorkload(1, self.position, self.n_layers)
        return {"value": one_token.bytes_per_step() * self.m / t_step / 1e9, "unit": "GB/s",
                "cores": cores, "kind": "oracle",
                "tokens_per_s": self.m / t_step,
                "sample": f"{n_sample_layers} of {self.n_layers} layers (C oracle on {cores} host "
                          f"threads, rows and heads split over threads; mean {t_layer:.3f} s per layer) "
                          f"+ the Q4_0 LM head ({t_head:.3f} s), one token at position {self.position}; "
                          f"step time extrapolated as {self.n_layers} x layer + head per token"}

    def cpu_baseline(self):
        return self.cpu_sample(n_sample_layers=8)

    def config_ref(self):
        return {"workload": self.name, "layers": self.n_layers, "hidden": self.shape.hidden,
                "intermediate": self.shape.inter, "heads": self.shape.n_heads,
                "kv_heads": self.shape.n_kv_heads, "head_dim": self.shape.head_dim,
                "vocab": self.vocab, "batch_tokens": self.m, "position": self.position,
                "max_seq": self.max_seq,
                "weights_bytes": self.weight_bytes(),
                "l2": "inputs larger than L2 (3.7 GB of weights per step)"}

    def config(self):
        c = self.config_ref()
        c["launch"] = "one CUDA graph per step (PDL edges between kernels)"
        return c


WORKLOADS = {"gemv": GemvWorkload, "stack": StackWorkload}


def make_workload(args):
    if args.workload == "gemv":
        return GemvWorkload(args.batch)
    return StackWorkload(args.batch, args.position, args.layers)


# ----------------------------------------------------------------------------- arms
# GEMV shapes reported beside every stack run: the target shape of the Llama sweep
# at one token, and the widest batched-decode GEMV at 16 tokens.
SUBRECORD_GEMVS = [(4096, 14336, 1), (14336, 4096, 16)]
# The many-token (prefill) product on the tensor cores: a 512-token prompt
# against the widest Llama-sweep shapes.
SUBRECORD_GEMMS = [(4096, 14336, 512), (14336, 4096, 512)]
MIN_TIMED_S = 1.0


def run_timed_blocks(wl, stream, steps, pg, dev):
    """Blocks of exactly `steps` steps, each bracketed by a barrier and a device
    synchronisation and timed with CUDA events on the launching stream, repeated
    until the blocks add up to MIN_TIMED_S (so that the clock record covers a
    steady stretch).  Returns the median block's ms per step (max over ranks) and
    the number of blocks."""
    import torch
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    per_step, total_s = [], 0.0
    while True:
        barrier(pg)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                wl.step(stream)
            e1.record(stream)
        torch.cuda.synchronize()
        barrier(pg)
        ms = e0.elapsed_time(e1)
        per_step.append(ms / steps)
        total_s += ms * 1e-3
        # every rank runs the same number of blocks: the decision is rank 0's
        done = total_s >= MIN_TIMED_S or len(per_step) >= 10000
        if pg is not None:
            t = torch.tensor([1.0 if done else 0.0], device=dev)
            pg.broadcast(t, 0)
            done = bool(t.item())
        if done:
            break
    return max_over_ranks(pg, statistics.median(per_step), dev), len(per_step)


def run_rz(args, world, rank, local, pg):
    import torch
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    import quantized_q4_q8_gb300 as rz
    rz.load()
    wl = make_workload(args)
    wl.setup(dev)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_line = wl.cpu_baseline()   # before any timing: the host is idle here
    else:
        cpu_line = None
    stream = torch.cuda.Stream(device=dev)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            wl.step(stream)
    torch.cuda.synchronize()
    st, code = rz.check_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error word after warm-up: 0x{code:x}")

    # ---- device-timed region
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else local)
    barrier(pg)
    torch.cuda.synchronize()
    if rank == 0:
        clocks.start()
        time.sleep(0.3)
    ms, blocks = run_timed_blocks(wl, stream, args.steps, pg, dev)
    clk = clocks.stop() if rank == 0 else None

    # ---- dominant kernel: average launch duration over back-to-back launches
    dom = wl.dominant()
    dom_ms = wl.dominant_time(stream)
    if dom_ms is None:   # the step is back-to-back launches of the dominant kernel
        dom_ms = ms / dom["launches_per_step"]

    # ---- end to end through the C ABI with host buffers
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            wl.e2e_step(stream)
    torch.cuda.synchronize()
    barrier(pg)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            wl.e2e_step(stream)
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    e2e_ms = max_over_ranks(pg, e0.elapsed_time(e1) / args.steps, dev)

    # ---- the GEMV shapes of the metric, reported beside the step
    peak, peak_kind = measured_peaks()
    gemvs = {}
    if not args.no_subrecords:
        for o, i, m in SUBRECORD_GEMVS:
            r = measure_gemv(rz, o, i, m, dev, stream)
            r["frac"] = round(r["gbs"] / peak, 4)
            gemvs[f"{o}x{i}_m{m}"] = r
    gemms = {}
    if not args.no_subrecords:
        tc_peak = measured_tensor_peak()
        for o, i, m in SUBRECORD_GEMMS:
            r = measure_gemm(rz, o, i, m, dev, stream)
            r["frac_of_f16_tensor_peak"] = round(r["tensor_tflops"] / tc_peak, 4)
            gemms[f"{o}x{i}_m{m}"] = r
    st, code = rz.check_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error word after timing: 0x{code:x}")

    bytes_step = wl.bytes_per_step()
    value = world * bytes_step / (ms * 1e-3) / 1e9
    achieved = dom["bytes_per_launch"] / (dom_ms * 1e-3) / 1e9
    traffic = profile_traffic(wl.kernel_file, wl.name)
    cfg = wl.config()
    cfg["timed_blocks"] = blocks
    cfg["timed_region"] = (f"{blocks} blocks of {args.steps} steps (median block), at least "
                           f"{MIN_TIMED_S:g} s in total")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "q4k_x_q8_1_int8dot_f32",
        "data": "synthetic (seeded, distributions of the workload definition)",
        "config": cfg,
        "pct_of_peak": round(100 * value / world / peak, 2),
        "tokens_per_s": round(world * wl.m / (ms * 1e-3), 2),
        "tokens_per_s_per_layer_stack": round(world * wl.m / (ms * 1e-3), 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": dom["kernel"], "launch_us": round(dom_ms * 1e3, 3),
                     "bytes_per_launch": int(dom["bytes_per_launch"]),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s"},
        "gemv": gemvs,
        "prefill_gemm": gemms,
        "e2e": {"value": round(world * bytes_step / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": wl.e2e_bytes()[0], "d2h_bytes_per_step": wl.e2e_bytes()[1],
                "ms_per_step": round(e2e_ms, 5)},
        "gpu_launches": blocks * args.steps * wl.launches_per_step(),
        "clocks": clk,
    }
    if "what" in dom:
        line["roofline"]["what"] = dom["what"]
    if cpu_line is not None:
        line["cpu_baseline"] = cpu_line
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, world, rank):
    """The oracle timed on the host cores on a bounded sample of the same workload."""
    if rank != 0:
        return
    wl = make_workload(args)
    samples = []
    for _ in range(args.steps):
        samples.append(wl.cpu_sample())
    v = statistics.median(s["value"] for s in samples)
    cb = dict(samples[0])
    cb["value"] = v
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": cb["unit"],
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 oracle", "data": "synthetic", "config": wl.config_ref(),
        "cpu_baseline": cb,
        "e2e": {"value": round(v, 4), "unit": cb["unit"], "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="steps per timed block (default: 200 for the stack, 50 for the GEMV)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="rz", choices=["rz", "reference"])
    ap.add_argument("--workload", default="stack", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-subrecords", action="store_true",
                    help="skip the GEMV shapes reported beside the step")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--position", type=int, default=1024)
    ap.add_argument("--layers", type=int, default=S.LLAMA_LAYERS,
                    help="layers of the stack (32 for the benchmark; fewer for small profiles)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.steps is None:
        args.steps = 200 if args.workload == "stack" else 50
        if args.impl == "reference":
            args.steps = 3
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only; other ranks have no work
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    world, rank, local, pg = dist_setup(args.gpus)
    run_rz(args, world, rank, local, pg)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
