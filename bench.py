"""Benchmark of the CPR Gated DeltaNet hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload prefill]
                    [--impl ours|reference]

Prints ONE JSON line (rank 0).  The headline workload (default) is the
Prefill configuration: B=4 sequences x T=4096 tokens, H=16 heads,
d_k=d_v=128, C=64, bf16 q/k/v, fp32 gates/state/accumulation/output; a step
is one trainer-forward call (cpr_gdn_fwd: outputs o and the final state).
Other workloads: trainer (B=8 fwd+bwd), decode (64 sequences prefilled with
2048 tokens, one decode step per step), varlen (48 packed sequences of
U[128, 8192] tokens, fwd+bwd).  Inputs are seeded synthetic tensors
(infer_consistent_linear_gb300.synth), generated on the host and copied to
the device before timing; every workload's working set exceeds the 129 MB L2.

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent sequences: weak scaling, no data-path collective); timing is the
max over ranks between barriers.

--impl reference times the CPU oracle (fp64 recurrence, the method's
definition) on a bounded sample of the same workload on the host cores.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "CPR-GDN fwd/fwd+bwd tokens/s + decode µs/step; % of roofline; bitwise-exact flag"
MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")

WORKLOADS = {
    "prefill": dict(desc="Prefill: B=4, H=16, T=4096, d_k=d_v=128, C=64, bf16 in, fp32 out/state; "
                         "forward output and final state", lens=[4096] * 4, H=16, d=128, op="fwd"),
    "trainer": dict(desc="Trainer fwd+bwd: B=8, H=16, T=4096, d_k=d_v=128, C=64, bf16; dO ~ N(0,1)",
                    lens=[4096] * 8, H=16, d=128, op="fwdbwd"),
    "decode": dict(desc="Decode: 64 sequences prefilled with 2048 tokens, one token per sequence per "
                        "step, H=32, d_k=d_v=128, C=64, bf16", lens=[2048] * 64, H=32, d=128,
                   op="decode"),
    "varlen": dict(desc="Varlen fwd+bwd: 48 packed sequences, lengths ~ U[128, 8192] (seed 0), H=16, "
                        "d_k=d_v=128, C=64, bf16", lens=None, H=16, d=128, op="fwdbwd"),
}
C = 64


def peaks():
    try:
        with open(MEASURED_PEAKS) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    sm_max_mhz=float(p.get("sm_max_mhz", 2070.0)), source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, sm_max_mhz=2070.0, source="fallback")


def workload_lens(name):
    w = WORKLOADS[name]
    if w["lens"] is not None:
        return list(w["lens"])
    from infer_consistent_linear_gb300.synth import varlen_lengths
    return varlen_lengths(48, 128, 8192, seed=0)


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in self.rows if num(r[1])]
        mx = [num(r[2]) for r in self.rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(self.rows)}


# ------------------------------------------------------- algorithmic work
def algo_fwd_bytes_per_head_token(d, io_bytes=2, out_bytes=4):
    # q, k, v in; g, beta in (fp32); o out
    return 3 * d * io_bytes + 8 + d * out_bytes


def algo_bwd_bytes_per_head_token(d, io_bytes=2, out_bytes=4):
    # reads q, k, v, g, beta, dO (fp32); writes dq, dk, dv (fp32), dg, dbeta
    return 3 * d * io_bytes + 8 + d * 4 + 3 * d * out_bytes + 8


def algo_fwd_flops_per_chunk(d, Cc=C):
    # dense intra-chunk contractions: K K^T, Q K^T, T (I+A)-apply to K and V,
    # W'H, Q H, P Delta, K^T Delta  (3 C^2 d_k + 2 C^2 d_v + 3 C d_k d_v MACs)
    return 2 * (3 * Cc * Cc * d + 2 * Cc * Cc * d + 3 * Cc * d * d)


def algo_bwd_flops_per_chunk(d, Cc=C):
    # 14 C^2 d + 8 C d^2 + 2 C^3 MACs per chunk (the planned schedule incl. recompute)
    return 2 * (14 * Cc * Cc * d + 8 * Cc * d * d + 2 * Cc ** 3)


DECODE_ALGO_BYTES_PER_SEQ_HEAD = 84_492  # H_n read + amortised commit + token io + buffered rows


def simt_kernel_flops_per_chunk(name, d, Cc=C):
    """fp32 FMA work each SIMT kernel performs per (chunk, head) (x2 FLOP)."""
    pa, pp = Cc * (Cc - 1) // 2, Cc * (Cc + 1) // 2
    t_fma = Cc * (Cc - 1) * (Cc + 1) // 6
    if name == "cpr_prep":
        return 2 * ((pa + pp) * d + t_fma + pp * 2 * d)
    if name == "cpr_state_fwd":
        return 2 * (3 * Cc * d * d + pp * d)
    if name == "cpr_state_bwd":
        return 2 * ((pp + Cc * d) * d + pp * d + 2 * Cc * d * d)
    if name == "cpr_grad_chunk":
        return 2 * (9 * Cc * d * d + 6 * pp * d + 2 * Cc * Cc * d)
    return None


def chunk_count(lens):
    return sum((L + C - 1) // C for L in lens)


# ------------------------------------------------------------ our arm
class OurStep:
    """Device-resident inputs, outputs and workspaces for one workload."""

    def __init__(self, name, dev, n_decode_steps=0):
        import infer_consistent_linear_gb300 as cpr
        from infer_consistent_linear_gb300.synth import make_inputs
        self.cpr = cpr
        self.name = name
        self.w = WORKLOADS[name]
        self.lens = workload_lens(name)
        self.H, self.d, self.op = self.w["H"], self.w["d"], self.w["op"]
        H, d = self.H, self.d
        self.c = cpr.default_contract(torch.bfloat16, d)
        self.dig = cpr.contract_digest(self.c)
        self.dev = dev
        if self.op == "decode":
            full = [L + n_decode_steps for L in self.lens]
            x = make_inputs(full, H, d, d, io_dtype=torch.bfloat16, seed=0)
            self.x_host = x
            xd = x.to(dev)
            cu = x.cu_seqlens.tolist()
            n_seq = len(self.lens)
            sel = torch.cat([torch.arange(cu[b], cu[b] + self.lens[b]) for b in range(n_seq)])
            cu_pre = torch.tensor([0] + torch.cumsum(torch.tensor(self.lens), 0).tolist(),
                                  dtype=torch.int32)
            _, _, self.cache = cpr.cpr_gdn_prefill(
                xd.q[sel.to(dev)], xd.k[sel.to(dev)], xd.v[sel.to(dev)], xd.g[sel.to(dev)],
                xd.beta[sel.to(dev)], cu_pre.to(dev), contract=self.c, digest=self.dig,
                want_final=False)
            # per-step token batches [n_seq, H, d], laid out step-major
            idx = torch.tensor([[cu[b] + self.lens[b] + t for b in range(n_seq)]
                                for t in range(n_decode_steps)]).reshape(-1).to(dev)
            self.tok = [t.index_select(0, idx).view(n_decode_steps, n_seq, *t.shape[1:]).contiguous()
                        for t in (xd.q, xd.k, xd.v, xd.g, xd.beta)]
            self.o_steps = torch.empty(n_decode_steps, n_seq, H, d, device=dev)
            self.xd_full = xd
            self.t = 0
            torch.cuda.synchronize()
            return
        x = make_inputs(self.lens, H, d, d, io_dtype=torch.bfloat16, seed=0,
                        with_grad=(self.op == "fwdbwd"))
        self.x_host = x
        self.xd = x.to(dev)
        n_tok, n_seq = sum(self.lens), len(self.lens)
        self.o = torch.empty(n_tok, H, d, device=dev)
        self.fin = torch.empty(n_seq, H, d, d, device=dev)
        self.ws = torch.empty(cpr.workspace_bytes(self.c, cpr.CPR_OP_FWD, n_seq, n_tok, H),
                              dtype=torch.uint8, device=dev)
        if self.op == "fwdbwd":
            self.wsb = torch.empty(cpr.workspace_bytes(self.c, cpr.CPR_OP_BWD, n_seq, n_tok, H),
                                   dtype=torch.uint8, device=dev)
            self.gouts = dict(dq=torch.empty(n_tok, H, d, device=dev),
                              dk=torch.empty(n_tok, H, d, device=dev),
                              dv=torch.empty(n_tok, H, d, device=dev),
                              dg=torch.empty(n_tok, H, device=dev),
                              dbeta=torch.empty(n_tok, H, device=dev),
                              dh0=torch.empty(n_seq, H, d, d, device=dev))
        torch.cuda.synchronize()

    def run(self, xd=None):
        cpr = self.cpr
        if self.op == "decode":
            t = self.t
            q, k, v, g, b = (x[t] for x in self.tok)
            cpr.cpr_gdn_decode_step(q, k, v, g, b, self.cache, contract=self.c, digest=self.dig,
                                    out=self.o_steps[t])
            self.t += 1
            return
        x = xd if xd is not None else self.xd
        cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, contract=self.c, digest=self.dig,
                        out=self.o, final=self.fin, workspace=self.ws)
        if self.op == "fwdbwd":
            cpr.cpr_gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, contract=self.c,
                            digest=self.dig, workspace=self.wsb, outs=self.gouts)

    def tokens_per_step(self):
        return len(self.lens) if self.op == "decode" else sum(self.lens)

    def algo(self):
        """(bytes, flops) of the method per step (path roofline)."""
        d, H = self.d, self.H
        if self.op == "decode":
            return DECODE_ALGO_BYTES_PER_SEQ_HEAD * len(self.lens) * H, 0
        ht = sum(self.lens) * H
        nch = chunk_count(self.lens) * H
        byt = ht * algo_fwd_bytes_per_head_token(d) + len(self.lens) * H * d * d * 4
        fl = nch * algo_fwd_flops_per_chunk(d)
        if self.op == "fwdbwd":
            byt += ht * algo_bwd_bytes_per_head_token(d) + len(self.lens) * H * d * d * 4
            fl += nch * algo_bwd_flops_per_chunk(d)
        return byt, fl

    def kernel_units(self, kname):
        """Units (chunk-heads, or (seq, head) pairs for decode) one launch processes."""
        if kname == "cpr_decode":
            return len(self.lens) * self.H
        return chunk_count(self.lens) * self.H


# ------------------------------------------------------------ distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ timing
def time_device(step, K, W, world, profile=False):
    """W untimed warm-up steps, then K steps between barriers; CUDA events on
    the launching stream.  Returns (ms_per_step max over ranks, per-kernel
    profile or None)."""
    cpr = step.cpr
    for _ in range(W):
        step.run()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if profile:
        cpr.profile_begin()
    s.record(stream)
    for _ in range(K):
        step.run()
    e.record(stream)
    torch.cuda.synchronize()
    prof = cpr.profile_end() if profile else None
    barrier(world)
    ms = s.elapsed_time(e) / K
    return max_over_ranks(ms, world), prof


def time_e2e(step, K, W, world):
    """Same step through the public API with pinned host buffers: every step
    copies its inputs host->device and its results device->host inside the
    timed region.  Returns (ms_per_step, h2d_bytes, d2h_bytes)."""
    dev_bufs, host_in, host_out, dev_out = [], [], [], []
    if step.op == "decode":
        n = len(step.tok[0])
        ins = [t for t in step.tok]                       # [n_steps, n_seq, ...]
        host_in = [t.cpu().pin_memory() for t in ins]
        dev_bufs = [torch.empty_like(t[0]) for t in ins]
        out_host = torch.empty_like(step.o_steps[0], device="cpu").pin_memory()
        total = min(n, W + K)
    else:
        x = step.xd
        names = ["q", "k", "v", "g", "beta", "cu_seqlens"] + (["dO"] if step.op == "fwdbwd" else [])
        srcs = [getattr(step.x_host, nm) for nm in names]
        host_in = [t.contiguous().pin_memory() for t in srcs]
        dev_bufs = [torch.empty_like(getattr(x, nm)) for nm in names]
        dev_out = [step.o, step.fin] + ([step.gouts[k] for k in ("dq", "dk", "dv", "dg", "dbeta", "dh0")]
                                        if step.op == "fwdbwd" else [])
        host_out = [torch.empty_like(t, device="cpu").pin_memory() for t in dev_out]
    h2d = sum(t[0].numel() * t.element_size() if step.op == "decode" else t.numel() * t.element_size()
              for t in host_in)
    stream = torch.cuda.current_stream()

    def one(i):
        if step.op == "decode":
            for hb, db in zip(host_in, dev_bufs):
                db.copy_(hb[i], non_blocking=True)
            q, k, v, g, b = dev_bufs
            step.cpr.cpr_gdn_decode_step(q, k, v, g, b, step.cache, contract=step.c,
                                         digest=step.dig, out=step.o_steps[i])
            out_host.copy_(step.o_steps[i], non_blocking=True)
        else:
            for hb, db in zip(host_in, dev_bufs):
                db.copy_(hb, non_blocking=True)
            from infer_consistent_linear_gb300.synth import GdnInputs
            d = dict(zip(["q", "k", "v", "g", "beta", "cu_seqlens", "dO"], dev_bufs))
            xin = GdnInputs(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], None, d.get("dO"))
            step.run(xin)
            for ho, do in zip(host_out, dev_out):
                ho.copy_(do, non_blocking=True)

    if step.op == "decode":
        # replay from a fresh copy of the cache so positions line up
        step.t = 0
        blob0 = step.cache.blob.clone()
        for i in range(min(W, total)):
            one(i)
        torch.cuda.synchronize()
        step.cache.blob.copy_(blob0)
        K = min(K, total)
        start = 0
    else:
        for i in range(W):
            one(i)
        start = 0
    torch.cuda.synchronize()
    barrier(world)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for i in range(K):
        one(start + i)
    e.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    d2h = (out_host.numel() * out_host.element_size() if step.op == "decode"
           else sum(t.numel() * t.element_size() for t in host_out))
    return max_over_ranks(s.elapsed_time(e) / K, world), int(h2d), int(d2h)

# CPR_BENCH_PART4
