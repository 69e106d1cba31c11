"""Benchmark of the filtered decoder-block backward on one GB300.

Workload: one TinyLlama-1.1B-shaped block (d_model 2048, 32 query / 4 kv heads
of 64, SwiGLU 5632, RMSNorm, RoPE base 10000), batch 4 x 2048 tokens, causal;
40% of each sequence filtered by the lowest Gumbel(0,1) scores; weights
N(0, 0.02), block input and upstream gradient N(0, 1); all synthetic and
seeded.  A step is the whole hot path: compaction of the keep-mask, gather of
the kept rows, the dimension-reduced GEMMs, the filtered attention backward,
the norm / activation / RoPE backward and the scatter of dx.

Prints one JSON line (rank 0).  The headline numbers are the TinyLlama-shaped
block's; "configs" adds the same filtered / unfiltered timing for the
Qwen2.5-shaped block, the Phi-1.5-shaped block at 0/20/40/60% filtered (span
masks) and the 22-block TinyLlama-shaped stack with its LM head
(`--headline-only` skips them); "forward" times the library's dense forward of
the headline block (collider_layer_fwd, which also writes every saved set the
bench uses).  `--impl reference` times the fp64 CPU oracle on the host cores
instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "filtered-backward tokens/s, TFLOP/s vs bf16 TC peak, speedup vs unfiltered"
WORKLOAD = "tinyllama_layer"
SAVED = "lean"   # --saved


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--headline-only", action="store_true",
                   help="time only the headline block (skip the other block shapes and the stack)")
    p.add_argument("--workload", default=WORKLOAD, choices=sorted(k for k in workloads.WORKLOADS if k.endswith("_layer")),
                   help="block shape for --case gemm / attn")
    p.add_argument("--saved", default="lean", choices=["lean", "full"],
                   help="saved set the filtered backward is given (Llama-style blocks): lean leaves out "
                        "a, b and s, which it recomputes for the kept rows; full passes them")
    p.add_argument("--case", default="layer", choices=["layer", "gemm", "attn", "timeline"],
                   help="layer: the benchmark; gemm / attn: one kernel family on a small input "
                        "(larger than L2) for profiler captures; timeline: every launch of one "
                        "filtered block step of --workload on its stream, with start and end times")
    return p.parse_args()


def config_dict(s, l2):
    return {"workload": f"{WORKLOAD}: TinyLlama-1.1B-shaped decoder block backward, batch {s.B} x seq {s.T}, "
                        f"d_model {s.D}, heads {s.H}/{s.Hkv}x{s.dh}, SwiGLU {s.F}, "
                        f"{int(s.f * 100)}% tokens filtered per sequence (Gumbel scores)",
            "global_batch": s.B, "seq_len": s.T, "filtered_fraction": s.f, "parallelism": "replicas",
            "saved_set": ("lean: a, b, s recomputed for the kept rows" if SAVED == "lean" and s.arch == "llama"
                          else "full"),
            "l2": l2}


# ---------------------------------------------------------------------------
GEMM_PROFILE = os.path.join(ROOT, "profiles", "tc_gemm_2sm_tinyllama_case.md")
GEMM_SOURCE = os.path.join(ROOT, "sparse_backward_gemm_gb300", "csrc", "gemm_tc.cu")


def gemm_traffic():
    """DRAM bytes (read + write) of one step's GEMM launches, from the committed ncu summary,
    as long as the GEMM source is still the one profiled; else None."""
    try:
        text = open(GEMM_PROFILE).read()
        want = re.search(r"gemm_tc\.cu sha256: ([0-9a-f]+)", text).group(1)
        nbytes = int(re.search(r"traffic_bytes_per_step: (\d+)", text).group(1))
        with open(GEMM_SOURCE, "rb") as f:
            have = hashlib.sha256(f.read()).hexdigest()
    except (OSError, AttributeError, ValueError):
        return None
    return nbytes if have.startswith(want) else None


# ---------------------------------------------------------------------------
# algorithmic work (counted over kept tokens only)
def gemm_flops(s, nk):
    p_lin = s.D * s.Nqkv + s.H * s.dh * s.D + s.D * s.Nup + s.F * s.D
    return 4.0 * nk * p_lin


def attn_flops(s, kept_per_seq):
    return 10.0 * s.dh * s.H * sum(m * (m + 1) / 2 for m in kept_per_seq)


# ---------------------------------------------------------------------------
# synthetic saved activations: the library's own dense forward on the GPU
# (input preparation, outside the backward's timed region)
def layer_desc(cl, s):
    return cl.LayerDesc(arch=cl.ARCH_LLAMA if s.arch == "llama" else cl.ARCH_PHI, B=s.B, T=s.T, D=s.D, H=s.H,
                        Hkv=s.Hkv, dh=s.dh, F=s.F, rotary_dim=s.rotary_dim, rope_base=s.rope_base,
                        norm=cl.NORM_RMS if s.norm == "rms" else cl.NORM_LAYER, eps=s.eps,
                        act=cl.ACT_SWIGLU if s.act == "swiglu" else cl.ACT_GELU_TANH, qkv_bias=int(s.qkv_bias),
                        out_bias=int(s.out_bias), mlp_bias=int(s.mlp_bias))


def grad_buffers(s, dev):
    """f32 weight-gradient buffers of one block (the bias / beta ones where the shape has them)."""
    import torch
    shapes = dict(dnorm1_w=(s.D,), dw_qkv=(s.D, s.Nqkv), dw_o=(s.H * s.dh, s.D), dw_up=(s.D, s.Nup),
                  dw_down=(s.F, s.D))
    if s.norm == "ln":
        shapes["dnorm1_b"] = (s.D,)
    if s.arch == "llama":
        shapes["dnorm2_w"] = (s.D,)
    if s.qkv_bias:
        shapes["db_qkv"] = (s.Nqkv,)
    if s.out_bias:
        shapes["db_o"] = (s.D,)
    if s.mlp_bias:
        shapes["db_up"] = (s.Nup,)
        shapes["db_down"] = (s.D,)
    return {k: torch.empty(v, dtype=torch.float32, device=dev) for k, v in shapes.items()}


class NativeForward:
    """The library's dense forward of one block (collider_layer_fwd): parameter
    struct, the saved-set buffers it writes, y and its workspace."""

    def __init__(self, cl, s, W, desc, dev):
        import torch
        self.cl, self.s, self.desc = cl, s, desc
        g = lambda k: W[k].data_ptr() if k in W else None
        self.params = cl.LayerParams(**{k: g(k) for k in ("norm1_w", "norm1_b", "w_qkv", "b_qkv", "w_o", "b_o",
                                                          "norm2_w", "w_up", "b_up", "w_down", "b_down")})
        bf = lambda *shp: torch.empty(shp, dtype=torch.bfloat16, device=dev)
        f32 = lambda *shp: torch.empty(shp, dtype=torch.float32, device=dev)
        t = dict(a=bf(s.M, s.D), rstd1=f32(s.M), qkv=bf(s.M, s.Nqkv), o=bf(s.M, s.H * s.dh),
                 lse=f32(s.B, s.H, s.T), up=bf(s.M, s.Nup))
        if s.arch == "llama":
            t.update(h=bf(s.M, s.D), b=bf(s.M, s.D), rstd2=f32(s.M), s=bf(s.M, s.F))
        else:
            t["mean1"] = f32(s.M)
        self.t = t
        self.acts = cl.LayerActs(**{k: v.data_ptr() for k, v in t.items()})
        self.y = bf(s.M, s.D)
        self.ws = torch.empty(cl.collider_layer_fwd_workspace_size(desc), dtype=torch.uint8, device=dev)

    def run(self, x, stream=None):
        self.cl.collider_layer_fwd(self.desc, self.params, x, self.y, self.acts, self.ws, stream)

    def saved(self, x) -> dict:
        return dict(x=x, **self.t)


class Block:
    """One block's synthetic inputs, saved activations (written by the library's
    own dense forward), gradient buffers and workspace on the GPU; step() runs
    compaction + the layer backward."""

    def __init__(self, cl, s, dev):
        import torch
        self.cl, self.s = cl, s
        wn = workloads.layer_weights(s)
        tn = workloads.layer_inputs(s)
        self.keep_np = tn["keep"]
        self.W = {k: torch.from_numpy(v).to(dev).bfloat16() for k, v in wn.items()}
        x = torch.from_numpy(tn["x"]).to(dev).bfloat16()
        self.x = x
        self.dout = torch.from_numpy(tn["dout"]).to(dev).bfloat16()
        # "unfiltered" is the dense backward: the library's NULL-index call,
        # which reads FULL rows in place (no compaction, gather or scatter)
        self.masks = {"filtered": torch.from_numpy(tn["keep"]).to(dev), "unfiltered": None}
        self.desc = layer_desc(cl, s)
        self.fwd = NativeForward(cl, s, self.W, self.desc, dev)
        self.fwd.run(x)
        self.saved = self.fwd.saved(x)
        self.weights = cl.LayerWeights(**{k: self.W[k].data_ptr() for k in
                                          ("norm1_w", "w_qkv", "w_o", "norm2_w", "w_up", "w_down") if k in self.W})
        self.sv = cl.LayerSaved(**{k: v.data_ptr() for k, v in self.saved.items()})
        # what the filtered backward is given: without a, b and s (Llama-style
        # blocks; recomputed for the kept rows) unless --saved full
        lean = SAVED == "lean" and s.arch == "llama"
        self.saved_filtered = {k: v for k, v in self.saved.items() if not (lean and k in ("a", "b", "s"))}
        self.sv_filtered = cl.LayerSaved(**{k: v.data_ptr() for k, v in self.saved_filtered.items()})
        self.G = grad_buffers(s, dev)
        self.dx = torch.empty(s.M, s.D, dtype=torch.bfloat16, device=dev)
        self.grads = cl.LayerGrads(dx=self.dx.data_ptr(), **{k: v.data_ptr() for k, v in self.G.items()})
        self.ws = torch.empty(cl.collider_layer_workspace_size(self.desc), dtype=torch.uint8, device=dev)
        self.idx = torch.empty(s.M, dtype=torch.int32, device=dev)
        self.cu = torch.empty(s.B + 1, dtype=torch.int32, device=dev)
        self.nk = torch.empty(1, dtype=torch.int32, device=dev)

    def step(self, mask, stream, sv=None, dout=None):
        """mask None: the unfiltered dense backward (no compaction, NULL index)."""
        cl, s = self.cl, self.s
        index = (None, None, None)
        if mask is not None:
            cl.collider_compact(mask, s.B, s.T, self.idx, self.cu, self.nk, None, stream)
            index = (self.idx, self.cu, self.nk)
        if sv is None:
            sv = self.sv if mask is None else self.sv_filtered
        cl.collider_layer_bwd(self.desc, self.weights, sv, self.dout if dout is None else dout, cl.ROWS_FULL,
                              *index, self.grads, cl.ROWS_FULL, self.ws, stream)


class Stack:
    """The 22-block stack: inputs and saved activations of every block (the
    library's dense forward, block by block), LM head and embedding; step() runs
    compaction + collider_stack_bwd."""

    def __init__(self, cl, st, dev):
        import torch
        self.cl, self.st = cl, st
        ls = st.layer
        t = workloads.stack_tensors(st)
        self.keep_np = t["keep"]
        self.mask = torch.from_numpy(t["keep"]).to(dev)
        self.mask_all = None   # the unfiltered dense backward: the NULL-index call
        E = torch.from_numpy(t["E"]).to(dev).bfloat16()
        ids = torch.from_numpy(t["ids"].astype(np.int64)).to(dev)
        x = E[ids]
        self.saved, self.Ws = [], []
        self.desc = layer_desc(cl, ls)
        with torch.no_grad():
            for w in t["layers"]:
                W = {k: torch.from_numpy(v).to(dev).bfloat16() for k, v in w.items()}
                fw = NativeForward(cl, ls, W, self.desc, dev)
                fw.run(x)
                self.saved.append(fw.saved(x))
                self.Ws.append(W)
                x = fw.y
                fw.ws = None   # the workspace is not kept per block
            xf = x.float()
            self.rstdf = torch.rsqrt(xf.pow(2).mean(-1) + ls.eps)
            self.nf = torch.from_numpy(t["normf_w"]).to(dev).bfloat16()
            self.y = (xf * self.rstdf[:, None] * self.nf.float()).bfloat16()
            self.wlm = torch.from_numpy(t["w_lm"]).to(dev).bfloat16()
            self.z = (self.y @ self.wlm).bfloat16()
        self.xL = x
        L = st.L
        self.Wc = (cl.LayerWeights * L)(*[cl.LayerWeights(**{k: W[k].data_ptr() for k in
                                                              ("norm1_w", "w_qkv", "w_o", "norm2_w", "w_up", "w_down")})
                                          for W in self.Ws])
        self.Sc = (cl.LayerSaved * L)(*[cl.LayerSaved(**{k: v.data_ptr() for k, v in sv.items()}) for sv in self.saved])
        # the filtered call's saved sets: without a, b and s unless --saved full
        lean = SAVED == "lean"
        self.Sc_filtered = (cl.LayerSaved * L)(*[cl.LayerSaved(**{k: v.data_ptr() for k, v in sv.items()
                                                                  if not (lean and k in ("a", "b", "s"))})
                                                 for sv in self.saved])
        self.G = [grad_buffers(ls, dev) for _ in range(L)]
        self.Gc = (cl.LayerGrads * L)(*[cl.LayerGrads(dx=None, **{k: v.data_ptr() for k, v in g.items()})
                                        for g in self.G])
        self.targets = torch.from_numpy(t["targets"]).to(dev)
        self.ids = torch.from_numpy(t["ids"]).to(dev)
        self.dnf = torch.empty(ls.D, device=dev)
        self.dlm = torch.empty(ls.D, st.V, device=dev)
        self.dE = torch.empty(st.V, ls.D, device=dev)
        self.ws = torch.empty(cl.collider_stack_workspace_size(self.desc, L, st.V), dtype=torch.uint8, device=dev)
        self.idx = torch.empty(ls.M, dtype=torch.int32, device=dev)
        self.cu = torch.empty(ls.B + 1, dtype=torch.int32, device=dev)
        self.nk = torch.empty(1, dtype=torch.int32, device=dev)

    def step(self, mask, stream):
        """mask None: the unfiltered dense backward (no compaction, NULL index)."""
        cl, st = self.cl, self.st
        ls = st.layer
        index = (None, None, None)
        if mask is not None:
            cl.collider_compact(mask, ls.B, ls.T, self.idx, self.cu, self.nk, None, stream)
            index = (self.idx, self.cu, self.nk)
        cl.collider_stack_bwd(self.desc, st.L, st.V, self.Wc, self.Sc if mask is None else self.Sc_filtered,
                              self.z, self.targets, self.ids, self.y,
                              self.xL, self.rstdf, self.nf, self.wlm, *index, self.Gc, self.dnf,
                              self.dlm, self.dE, self.ws, stream)


# ---------------------------------------------------------------------------
class Clocks:
    """nvidia-smi samples during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.p = None
        # raw samples (the JSON line carries their summary); COLLIDER_CLOCKS_DIR keeps them
        self.path = os.path.join(os.environ.get("COLLIDER_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"collider_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.p = None
        return self

    def __exit__(self, *a):
        if self.p is not None:
            self.p.terminate()
            self.p.wait(timeout=10)
            self.f.close()

    def summary(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": float(np.median(loaded)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(vals, device):
    """Element-wise max over all ranks (the slowest replica sets the job time);
    identity outside a multi-rank run."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in vals]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def profile_pass(cl, step_fn, steps, warmup, flush, n_kept):
    """Per-launch event times of `steps` steps, every launch on one stream
    (the library's profiler; the weight-gradient side stream is off so no
    kernel shares the GPU with another).  Returns per-kernel [launches, ms]
    summed over the steps, the GEMM launches' algorithmic FLOPs and time, and
    a per-shape GEMM table (ms per step)."""
    import torch
    os.environ["COLLIDER_SIDE_STREAM"] = "0"
    try:
        for _ in range(warmup):
            step_fn()
        cl.collider_profile_enable(1)
        for _ in range(steps):
            flush.fill_(1)
            step_fn()
        torch.cuda.synchronize()
        cl.collider_profile_enable(0)
    finally:
        os.environ["COLLIDER_SIDE_STREAM"] = "1"
    per, shapes = {}, {}
    gemm_ms, gemm_fl = 0.0, 0.0
    for i in range(cl.collider_profile_count()):
        name, (m, n, k, dyn), ms = cl.collider_profile_get(i)
        d = per.setdefault(name, [0, 0.0])
        d[0] += 1
        d[1] += ms
        if name == "tc_gemm":
            mm = n_kept if dyn == 1 else m
            kk = n_kept if dyn == 2 else k
            gemm_ms += ms
            gemm_fl += 2.0 * mm * n * kk
            key = f"{mm}x{n}x{kk}" + ("" if dyn != 2 else " (dW)")
            e = shapes.setdefault(key, [0.0, 2.0 * mm * n * kk])
            e[0] += ms / steps
    return per, gemm_ms, gemm_fl, shapes


def attn_roofline(per, steps, fl_per_step, peak, src):
    """The attention backward's main pass (and with its D' pre-pass) against
    the bf16 tensor peak: 5-unit algorithmic FLOPs over event time."""
    main = per.get("attn_main_tc", [0, 0.0])[1] / steps
    pre = per.get("attn_dprep_tc", [0, 0.0])[1] / steps
    if main <= 0:
        return None
    a_main = fl_per_step / (main * 1e-3) / 1e12
    a_both = fl_per_step / ((main + pre) * 1e-3) / 1e12
    return {"bound": "tensor", "kernel": "attn_main_tc (tcgen05 filtered attention backward, main pass)",
            "achieved": a_main, "peak": peak, "unit": "TFLOP/s", "frac": a_main / peak,
            "peak_source": f"bf16_tflops ({src})", "traffic": None,
            "ms_per_step": main, "prepass_ms_per_step": pre,
            "frac_with_prepass": a_both / peak,
            "flops": "5 matmul units over the kept causal pairs: 10*dh*H*sum_b m_b(m_b+1)/2 per step"}


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ---------------------------------------------------------------------------
def cpu_baseline(s, budget_s=20.0):
    """The fp64 oracle, as it stands, on one sequence of the workload."""
    from oracle import block as ob
    one = s.with_(B=1)
    w = workloads.layer_weights(s)
    t = workloads.layer_inputs(s)
    T = s.T
    x, dout, keep = t["x"][:T], t["dout"][:T], t["keep"][:1]
    _, saved = ob.block_forward(x, w, one, round_saved=True)
    t0 = time.perf_counter()
    ob.block_backward(dout, saved, w, one, keep)
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    return {"value": T / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"1 of {s.B} sequences ({T} tokens, {int(keep.sum())} kept), fp64 numpy, "
                      f"backward only, {dt:.1f} s"}


def run_reference(args):
    s = workloads.WORKLOADS[WORKLOAD]
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    times = []
    cb = None
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(s)
        if i >= args.warmup:
            times.append(s.T / r["value"])
            cb = r
    sec = float(np.mean(times))
    val = s.T / sec
    cb = dict(cb, value=val)
    print(json.dumps({"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
                      "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                      "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
                      "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                      "config": config_dict(s, "n/a (CPU)"), "cpu_baseline": cb,
                      "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                              "d2h_bytes_per_step": 0}}))


# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist
    import sparse_backward_gemm_gb300 as cl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    s = workloads.WORKLOADS[WORKLOAD]
    M = s.M

    # ---- inputs (seeded, synthetic), saved activations by the library's forward ----
    blk = Block(cl, s, dev)
    tn = {"keep": blk.keep_np}
    W, saved, dout, masks, G, dx = blk.W, blk.saved, blk.dout, blk.masks, blk.G, blk.dx
    desc, weights, grads, ws, idx, cu, nk = blk.desc, blk.weights, blk.grads, blk.ws, blk.idx, blk.cu, blk.nk
    torch.cuda.synchronize()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(mask):
        blk.step(mask, stream)

    def timed(mask, K, Wm, step_fn=None):
        step_fn = step_fn or step
        for _ in range(Wm):
            step_fn(mask)
        cl.collider_check(stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        cl.collider_launch_count(1)
        for e0, e1 in ev:
            flush.fill_(1)   # evict L2 between steps
            e0.record(stream)
            step_fn(mask)
            e1.record(stream)
        torch.cuda.synchronize()
        launches = cl.collider_launch_count(1)
        if world > 1:
            dist.barrier()
        cl.collider_check(stream)
        ms = [a.elapsed_time(b) for a, b in ev]
        return float(np.mean(ms)), launches

    # ---- main timed region (filtered) with clock sampling ----------------
    with Clocks(local) as clk:
        ms_f, launches = timed(masks["filtered"], args.steps, args.warmup)
    clocks = clk.summary()
    ms_u, _ = timed(masks["unfiltered"], args.steps, args.warmup)
    ms_f, ms_u = max_over_ranks([ms_f, ms_u], dev)

    # ---- per-kernel times from the library profiler (separate pass) ------
    # The weight-gradient GEMMs normally overlap the rest of the step on a
    # second stream; for per-kernel durations (the roofline) this pass runs
    # every launch on one stream, so no kernel shares the GPU with another.
    n_kept = int(tn["keep"].sum())
    kept_per_seq = tn["keep"].sum(axis=1).tolist()
    per, gemm_ms, gemm_fl, gemm_shapes = profile_pass(cl, lambda: step(masks["filtered"]), args.steps,
                                                      args.warmup, flush, n_kept)
    peaks, src = measured_peaks()
    achieved = gemm_fl / (gemm_ms * 1e-3) / 1e12 if gemm_ms > 0 else 0.0
    step_ms_prof = sum(v[1] for v in per.values()) / args.steps

    # ---- end to end through the C ABI with host buffers ------------------
    # Every step copies its inputs (the saved set the filtered call is given,
    # dOut, keep-mask) from pinned host memory and its outputs (weight
    # gradients, dx) back.  The
    # copies are pipelined the way a training loop prefetches: the inputs of
    # step i+1 go up on a copy stream while step i computes (two device input
    # sets), and step i's outputs come down on a third stream while step i+1
    # computes (two device output sets).  All copies sit inside the timed region.
    host_in = {k: v.cpu().pin_memory() for k, v in blk.saved_filtered.items()}
    host_dout = dout.cpu().pin_memory()
    host_mask = masks["filtered"].cpu().pin_memory()
    host_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in G.items()}
    host_dx = torch.empty(dx.shape, dtype=dx.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host_in.values()) + host_dout.numel() * 2 + host_mask.numel()
    d2h = sum(v.numel() * 4 for v in G.values()) + dx.numel() * 2
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    sets = []
    for _ in range(2):
        din = {k: torch.empty_like(v) for k, v in blk.saved_filtered.items()}
        dgr = {k: torch.empty_like(v) for k, v in G.items()}
        ddx = torch.empty_like(dx)
        sets.append(dict(
            din=din, dout=torch.empty_like(dout), mask=torch.empty_like(masks["filtered"]), G=dgr, dx=ddx,
            sv=cl.LayerSaved(**{k: din[k].data_ptr() for k in din}),
            grads=cl.LayerGrads(dx=ddx.data_ptr(), **{k: v.data_ptr() for k, v in dgr.items()}),
            loaded=torch.cuda.Event(), computed=torch.cuda.Event(), drained=torch.cuda.Event()))

    def e2e_run(n):
        up.wait_stream(stream)     # nothing of this run starts before the work already on the stream
        down.wait_stream(stream)

        def upload(i):
            b_ = sets[i % 2]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(b_["computed"])      # step i-2 is done reading this set
                for k in host_in:
                    b_["din"][k].copy_(host_in[k], non_blocking=True)
                b_["dout"].copy_(host_dout, non_blocking=True)
                b_["mask"].copy_(host_mask, non_blocking=True)
                b_["loaded"].record(up)
        upload(0)
        for i in range(n):
            b_ = sets[i % 2]
            if i + 1 < n:
                upload(i + 1)
            stream.wait_event(b_["loaded"])
            if i >= 2:
                stream.wait_event(b_["drained"])                  # outputs of step i-2 are on the host
            cl.collider_compact(b_["mask"], s.B, s.T, idx, cu, nk, None, stream)
            cl.collider_layer_bwd(desc, weights, b_["sv"], b_["dout"], cl.ROWS_FULL, idx, cu, nk, b_["grads"],
                                  cl.ROWS_FULL, ws, stream)
            b_["computed"].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(b_["computed"])
                for k in host_out:
                    host_out[k].copy_(b_["G"][k], non_blocking=True)
                host_dx.copy_(b_["dx"], non_blocking=True)
                b_["drained"].record(down)
        stream.wait_stream(down)
        stream.wait_stream(up)

    e2e_run(args.warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    e2e_ms = max_over_ranks([e2e_ms], dev)[0]

    # ---- the library's own dense forward of the same block ----------------
    # (collider_layer_fwd: the producer of the saved set; not part of the
    # filtered backward's step, reported beside it)
    fwd_run = lambda st_: blk.fwd.run(blk.x, st_)
    ms_fwd, fwd_launches = timed(masks["filtered"], args.steps, args.warmup, lambda m: fwd_run(stream))
    ms_fwd = max_over_ranks([ms_fwd], dev)[0]
    cl.collider_profile_enable(1)
    for _ in range(args.steps):
        flush.fill_(1)
        fwd_run(stream)
    torch.cuda.synchronize()
    cl.collider_profile_enable(0)
    fwd_per, fwd_gemm_ms, fwd_gemm_fl = {}, 0.0, 0.0
    for i in range(cl.collider_profile_count()):
        name, (m, n, k, dyn), ms = cl.collider_profile_get(i)
        fwd_per[name] = fwd_per.get(name, 0.0) + ms / args.steps
        if name == "tc_gemm":
            fwd_gemm_ms += ms / args.steps
            fwd_gemm_fl += 2.0 * m * n * k
    forward = {"ms_per_step": ms_fwd, "tokens_per_s": s.M * world / (ms_fwd * 1e-3), "gpu_launches": fwd_launches,
               "gemm_tflops": fwd_gemm_fl / args.steps / (fwd_gemm_ms * 1e-3) / 1e12 if fwd_gemm_ms > 0 else None,
               "kernels_ms_per_step": {k: round(v, 4) for k, v in sorted(fwd_per.items())}}

    # ---- the other block shapes and the 22-block stack (filtered vs unfiltered) ----
    configs = {}
    if not args.headline_only:
        runs = [("qwen25_layer", workloads.WORKLOADS["qwen25_layer"])]
        runs += [(f"phi15_layer f={f}", workloads.WORKLOADS["phi15_layer"].with_(f=f)) for f in (0.0, 0.2, 0.4, 0.6)]
        del blk
        torch.cuda.empty_cache()
        for label, shp in runs:
            b2 = Block(cl, shp, dev)
            ms2f, _ = timed(b2.masks["filtered"], args.steps, args.warmup, lambda m: b2.step(m, stream))
            ms2u, _ = timed(b2.masks["unfiltered"], args.steps, args.warmup, lambda m: b2.step(m, stream))
            ms2f, ms2u = max_over_ranks([ms2f, ms2u], dev)
            nk2 = int(b2.keep_np.sum())
            p2, g2_ms, g2_fl, _ = profile_pass(cl, lambda: b2.step(b2.masks["filtered"], stream), 3, 1, flush, nk2)
            configs[label] = {"tokens_per_s": shp.M * world / (ms2f * 1e-3), "ms_per_step": ms2f,
                              "unfiltered_ms_per_step": ms2u, "speedup_vs_unfiltered": ms2u / ms2f,
                              "kept_tokens": nk2, "tokens": shp.M,
                              "gemm_frac": (g2_fl / (g2_ms * 1e-3) / 1e12) / peaks["bf16_tflops"] if g2_ms > 0 else None,
                              "attention": attn_roofline(p2, 3, attn_flops(shp, b2.keep_np.sum(axis=1).tolist()),
                                                         peaks["bf16_tflops"], src),
                              "kernels_ms_per_step": {k: round(v[1] / 3, 4) for k, v in sorted(p2.items())}}
            del b2
            torch.cuda.empty_cache()
        st = workloads.WORKLOADS["tinyllama_stack"]
        stk = Stack(cl, st, dev)
        K2 = max(10, args.steps // 2)
        ms3f, _ = timed(stk.mask, K2, args.warmup, lambda m: stk.step(m, stream))
        ms3u, _ = timed(stk.mask_all, K2, args.warmup, lambda m: stk.step(m, stream))
        ms3f, ms3u = max_over_ranks([ms3f, ms3u], dev)
        # serialised profiler pass over the whole stack: GEMM and attention
        # fractions of the largest workload
        nk3 = int(stk.keep_np.sum())
        sp, sg_ms, sg_fl, sg_shapes = profile_pass(cl, lambda: stk.step(stk.mask, stream), 3, 1, flush, nk3)
        s_att = attn_roofline(sp, 3, st.L * attn_flops(st.layer, stk.keep_np.sum(axis=1).tolist()),
                              peaks["bf16_tflops"], src)
        s_ach = sg_fl / (sg_ms * 1e-3) / 1e12 if sg_ms > 0 else 0.0
        configs["tinyllama_stack (22 blocks + LM head)"] = {
            "tokens_per_s": st.layer.M * world / (ms3f * 1e-3), "ms_per_step": ms3f, "unfiltered_ms_per_step": ms3u,
            "speedup_vs_unfiltered": ms3u / ms3f, "kept_tokens": nk3, "tokens": st.layer.M,
            "steps": K2,
            "roofline": {
                "gemm": {"bound": "tensor", "kernel": "tc_gemm (all launches of a step: 22 blocks + LM head)",
                         "achieved": s_ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": s_ach / peaks["bf16_tflops"], "ms_per_step": sg_ms / 3,
                         "launches_per_step": sp.get("tc_gemm", [0, 0])[0] // 3},
                "attention": s_att,
                "step_ms_serialised": sum(v[1] for v in sp.values()) / 3,
                "kernels_ms_per_step": {k: round(v[1] / 3, 4) for k, v in sorted(sp.items())},
                "timing": "per-launch CUDA events, every launch on one stream (serialised pass, 3 steps)"}}
        del stk
        torch.cuda.empty_cache()

    if rank == 0:
        tokens = s.M * world
        line = {
            "metric": METRIC, "value": tokens / (ms_f * 1e-3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_f, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_dict(s, "flushed: 256 MB device write before every timed step, outside its events"),
            "kept_tokens": n_kept,
            "tflops": (gemm_flops(s, n_kept) + attn_flops(s, kept_per_seq)) / (ms_f * 1e-3) / 1e12,
            "unfiltered_ms_per_step": ms_u, "speedup_vs_unfiltered": ms_u / ms_f,
            "roofline": {"bound": "tensor", "kernel": "tc_gemm (tcgen05 bf16 GEMM, all launches of a step)",
                         "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["bf16_tflops"], "peak_source": f"bf16_tflops ({src})",
                         "traffic": gemm_traffic(), "traffic_unit": "bytes per step (8 launches), ncu cold-cache",
                         "gemm_ms_per_step": gemm_ms / args.steps,
                         "timing": "per-launch CUDA events, every launch on one stream (serialised pass)",
                         "step_ms_serialised": step_ms_prof,
                         "attention": attn_roofline(per, args.steps, attn_flops(s, kept_per_seq),
                                                    peaks["bf16_tflops"], src),
                         "speedup_vs_unfiltered": ms_u / ms_f, "unfiltered_ms_per_step": ms_u,
                         "stack": (configs.get("tinyllama_stack (22 blocks + LM head)") or {}).get("roofline")},
            "kernels_ms_per_step": {k: round(v[1] / args.steps, 4) for k, v in sorted(per.items())},
            "gemms": {k: {"ms": round(v[0], 4), "tflops": round(v[1] / (v[0] * 1e-3) / 1e12, 1)}
                      for k, v in gemm_shapes.items()},
            "gpu_launches": launches,
            "configs": configs,
            "forward": forward,
            "clocks": clocks,
            "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(s)
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_case(args):
    """One kernel family alone, for profiler captures: prints per-launch times."""
    import torch
    import sparse_backward_gemm_gb300 as cl
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    s = workloads.WORKLOADS[args.workload]
    keep = workloads.keep_mask(s.B, s.T, s.f, s.mask, s.seed_base)
    mask = torch.from_numpy(keep).to(dev)
    M = s.M
    idx = torch.empty(M, dtype=torch.int32, device=dev)
    cu = torch.empty(s.B + 1, dtype=torch.int32, device=dev)
    nk = torch.empty(1, dtype=torch.int32, device=dev)
    cl.collider_compact(mask, s.B, s.T, idx, cu, nk)
    g = torch.Generator(device=dev).manual_seed(1)
    rnd = lambda *shape: torch.randn(*shape, device=dev, generator=g).bfloat16()
    if args.case == "gemm":
        # MLP down-projection of the workload: dX [Mk, F] and dW [F, D] over the kept rows
        K, N = s.F, s.D
        X, W, dY = rnd(M, K), (rnd(K, N) * 0.02).bfloat16(), rnd(M, N)
        dX = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        dW = torch.empty(K, N, dtype=torch.float32, device=dev)
        ws = torch.empty(cl.collider_linear_workspace_size(cl.BF16, M, K, N), dtype=torch.uint8, device=dev)
        call = lambda: cl.collider_linear_bwd(cl.BF16, M, K, N, X, cl.ROWS_FULL, W, dY, cl.ROWS_FULL, idx, nk, dX,
                                              cl.ROWS_COMPACT, dW, None, ws)
        flops = {"tc_gemm": 4.0 * int(keep.sum()) * K * N}   # dX and dW
    else:
        H, Hkv, dh = s.H, s.Hkv, s.dh
        Q, Kt, V, dO = rnd(M, H * dh), rnd(M, Hkv * dh), rnd(M, Hkv * dh), rnd(M, H * dh)
        lse = (torch.rand(s.B, s.H, s.T, device=dev, generator=g) * 4 + 2).float()
        out = [torch.empty(M, n * dh, dtype=torch.bfloat16, device=dev) for n in (H, Hkv, Hkv)]
        ws = torch.empty(cl.collider_attn_workspace_size(s.B, s.T, H, Hkv, dh), dtype=torch.uint8, device=dev)
        call = lambda: cl.collider_attn_bwd(s.B, s.T, H, Hkv, dh, 1, dh ** -0.5, dh, s.rope_base, Q, Kt, V, None,
                                            dO, H * dh, Hkv * dh, H * dh, cl.ROWS_FULL, lse, idx, cu, nk, *out,
                                            cl.ROWS_COMPACT, ws)
        flops = {"attn_main": attn_flops(s, keep.sum(axis=1).tolist())}
    for _ in range(args.warmup):
        call()
    cl.collider_check()
    cl.collider_profile_enable(1)
    for _ in range(args.steps):
        call()
    torch.cuda.synchronize()
    cl.collider_profile_enable(0)
    cl.collider_check()
    per = {}
    for i in range(cl.collider_profile_count()):
        name, _, ms = cl.collider_profile_get(i)
        per.setdefault(name, []).append(ms)
    res = {k: {"launches_per_call": len(v) // args.steps, "ms_per_call": sum(v) / args.steps} for k, v in per.items()}
    for k, fl in flops.items():
        if k in res:
            res[k]["tflops"] = fl / (res[k]["ms_per_call"] * 1e-3) / 1e12
    print(json.dumps({"case": args.case, "kernels": res}))


def run_timeline(args):
    """One filtered block step as it runs (weight-gradient side stream and all):
    each launch's stream, the time its launch reached the head of that stream,
    its end, and its duration, from the library's per-launch events.  The
    events recorded between launches can keep a kernel from being launched
    before the one ahead of it has completed, so the step runs a little longer
    than in the timed region."""
    import torch
    import sparse_backward_gemm_gb300 as cl
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(0)
    s = workloads.WORKLOADS[args.workload]
    blk = Block(cl, s, dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        blk.step(blk.masks["filtered"], stream)
    cl.collider_check(stream)
    for rep in range(args.steps):
        flush.fill_(1)
        torch.cuda.synchronize()
        cl.collider_profile_enable(1)
        blk.step(blk.masks["filtered"], stream)
        torch.cuda.synchronize()
        cl.collider_profile_enable(0)
        print(f"# {args.workload}, step {rep}: launch, stream, kernel, M x N x K (GEMMs), start us, end us, us")
        for i in range(cl.collider_profile_count()):
            name, (m, n, k, dyn), ms = cl.collider_profile_get(i)
            t0, t1, si = cl.collider_profile_get_span(i)
            shape = f"{m}x{n}x{k}" if name == "tc_gemm" else "-"
            print(f"{i:3d} {si} {name:16s} {shape:18s} {t0 * 1e3:8.1f} {t1 * 1e3:8.1f} {ms * 1e3:7.1f}")
    cl.collider_check(stream)


if __name__ == "__main__":
    a = parse()
    SAVED = a.saved
    if a.impl == "reference":
        run_reference(a)
    elif a.case == "timeline":
        run_timeline(a)
    elif a.case != "layer":
        run_case(a)
    else:
        run_ours(a)
