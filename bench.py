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


N_SEQ_OVERRIDE = None   # --n-seq: first n sequences only (small cases for profiler captures)


def workload_lens(name):
    w = WORKLOADS[name]
    if w["lens"] is not None:
        lens = list(w["lens"])
    else:
        from infer_consistent_linear_gb300.synth import varlen_lengths
        lens = varlen_lengths(48, 128, 8192, seed=0)
    return lens[:N_SEQ_OVERRIDE] if N_SEQ_OVERRIDE else lens


# ---------------------------------------------------------------- clocks
class _Nvml:
    """Read-only NVML queries through the driver's library (ctypes): the SM clock, its
    maximum and the active clock-event (throttle) reasons of one device."""
    SM = 1   # NVML_CLOCK_SM
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40}

    def __init__(self, index):
        import ctypes
        self.c = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        rc = -1
        try:   # the same physical GPU as torch's device `index` (NVML may number GPUs otherwise)
            uuid = "GPU-" + str(torch.cuda.get_device_properties(index).uuid)
            rc = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h))
        except Exception:
            rc = -1
        if rc != 0 and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM, ctypes.byref(mx)) == 0 \
            else None

    def sample(self):
        c = self.c
        mhz, rs = c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, c.byref(mhz)) != 0:
            return None
        bits = rs.value if self.reasons_fn(self.h, c.byref(rs)) == 0 else 0
        return float(mhz.value), [n for n, b in self.BITS.items() if bits & b]


def gpu_local_cpus(index):
    """The host CPUs NVML names as nearest the GPU that torch calls `index` (read-only
    query), intersected with the CPUs this process may run on; None when unknown."""
    try:
        import ctypes
        n = _Nvml(index)
        words = ((os.cpu_count() or 64) + 63) // 64
        mask = (ctypes.c_ulong * words)()
        if n.lib.nvmlDeviceGetCpuAffinity(n.h, ctypes.c_uint(words), mask) != 0:
            return None
        near = {w * 64 + b for w in range(words) for b in range(64) if (mask[w] >> b) & 1}
        sel = near & os.sched_getaffinity(0)
        return sel or None
    except Exception:
        return None


class ClockSampler:
    """Samples SM clocks and throttle reasons while running: NVML every millisecond when the
    driver's library loads (a timed region can be a few milliseconds), else nvidia-smi every
    200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.rows = []       # nvidia-smi rows
        self.fast = []       # (mhz, [reasons]) from NVML
        self.nvml = None
        self.proc = None
        self.thread = None
        self.running = False

    def start(self):
        try:
            self.nvml = _Nvml(self.dev)
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            self.running = True
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
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

    def _poll(self):
        while self.running:
            s = self.nvml.sample()
            if s is not None:
                self.fast.append(s)
            time.sleep(0.001)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        self.running = False
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        if self.fast:
            sm = [m for m, _ in self.fast]
            reasons = sorted({r for _, rs in self.fast for r in rs})
            return {"sm_mhz": statistics.median(sm), "sm_max_mhz": self.nvml.max_mhz, "reasons": reasons,
                    "samples": len(self.fast), "source": "NVML, 1 ms"}

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
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(self.rows),
                "source": "nvidia-smi, 200 ms"}


# ------------------------------------------------------- algorithmic work
def algo_fwd_bytes_per_head_token(d, io_bytes=2, out_bytes=4):
    # q, k, v in; g, beta in (fp32); o out
    return 3 * d * io_bytes + 8 + d * out_bytes


def algo_bwd_bytes_per_head_token(d, io_bytes=2, out_bytes=4):
    # reads q, k, v, g, beta, dO; writes dq, dk, dv, dg, dbeta (dO and the three gradients
    # at out_bytes: 1,808 B with bf16, 2,832 B with the fp32 this build reads and writes)
    return 3 * d * io_bytes + 8 + d * out_bytes + 3 * d * out_bytes + 8


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


def tc_kernel_flops_per_chunk(name, d, Cc=C):
    """Algorithmic dense-contraction FLOPs each tensor-core kernel carries per
    (chunk, head): prep K K^T, Q K^T, T-applied K and V (4 C^2 d MACs); state
    W'H, QH, K^T Delta (3 C d^2) and P Delta (C^2 d).  The hi/lo split passes
    the kernels issue on top of these are not counted."""
    if name == "cpr_tc_prep":
        return 2 * 4 * Cc * Cc * d
    if name == "cpr_tc_state":
        return 2 * (3 * Cc * d * d + Cc * Cc * d)
    if name == "cpr_tc_state_bwd":   # P^T dO, T^T dDelta (C^2 d); K dH', Q^T dO, K^T dR (C d^2)
        return 2 * (2 * Cc * Cc * d + 3 * Cc * d * d)
    if name == "cpr_tc_grad":        # [Q;K]K^T, [dO;dR]Delta^T, G1 K, G1^T Q, M2 K; [dO;dR]H^T, Delta dH'^T
        return 2 * (7 * Cc * Cc * d + 3 * Cc * d * d)
    return None


def tc_kernel_bytes(name, lens, H, d, io_bytes=2, out_bytes=4):
    """The method's algorithmic bytes (inputs read, results written) each tensor-core
    kernel is charged with, so that the kernels of a step add up to the path's figure:
    prep reads q, k, v, g, beta; the state pass writes o and the final states; the
    reverse state pass reads dO and writes dh0; the gradient kernel reads q, k, v, g,
    beta again and writes dq, dk, dv, dg, dbeta.  Workspace tiles are not algorithmic."""
    ht = sum(lens) * H
    states = len(lens) * H * d * d * 4
    if name == "cpr_tc_prep":
        return ht * (3 * d * io_bytes + 8)
    if name == "cpr_tc_state":
        return ht * d * out_bytes + states
    if name == "cpr_tc_state_bwd":
        return ht * d * 4 + states
    if name == "cpr_tc_grad":
        return ht * (3 * d * io_bytes + 8 + 3 * d * out_bytes + 8)
    return None


def chunk_count(lens):
    return sum((L + C - 1) // C for L in lens)


# ------------------------------------------------------------ our arm
class OurStep:
    """Device-resident inputs, outputs and workspaces for one workload."""

    def __init__(self, name, dev, n_decode_steps=0, policy="tc"):
        import infer_consistent_linear_gb300 as cpr
        from infer_consistent_linear_gb300.synth import make_inputs
        self.cpr = cpr
        self.name = name
        self.w = WORKLOADS[name]
        self.lens = workload_lens(name)
        self.H, self.d, self.op = self.w["H"], self.w["d"], self.w["op"]
        H, d = self.H, self.d
        if policy == "tc":
            self.c = cpr.default_contract(torch.bfloat16, d, dv_splits=2,
                                          operand_policy=cpr.CPR_POLICY_TC_BF16X3)
        else:
            self.c = cpr.simt_contract(torch.bfloat16, d)
        self.dig = cpr.contract_digest(self.c)
        self.saved = policy == "tc"
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
            self.blob0 = self.cache.blob.clone()   # cache right after the prefill
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

    def run(self, xd=None, outs=None):
        """One step; `xd` / `outs` replace the step's own device inputs / outputs (outs: o,
        final, then dq, dk, dv, dg, dbeta, dh0 for the trainer)."""
        cpr = self.cpr
        if self.op == "decode":
            t = self.t
            q, k, v, g, b = (x[t] for x in self.tok)
            cpr.cpr_gdn_decode_step(q, k, v, g, b, self.cache, contract=self.c, digest=self.dig,
                                    out=self.o_steps[t])
            self.t += 1
            return
        x = xd if xd is not None else self.xd
        o, fin = (outs[0], outs[1]) if outs is not None else (self.o, self.fin)
        gouts = (dict(zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), outs[2:]))
                 if outs is not None and self.op == "fwdbwd" else getattr(self, "gouts", None))
        # the trainer step: a training forward that keeps its tiles for the backward
        # (tensor-core contract), or forward + backward-with-recompute (SIMT contract)
        train = self.op == "fwdbwd" and self.saved
        cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, contract=self.c, digest=self.dig,
                        out=o, final=fin, workspace=self.wsb if train else self.ws,
                        train=train)
        if self.op == "fwdbwd":
            cpr.cpr_gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, contract=self.c,
                            digest=self.dig, workspace=self.wsb, outs=gouts, saved=train)

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
        if kname in ("cpr_decode", "cpr_tc_decode"):
            return len(self.lens) * self.H
        return chunk_count(self.lens) * self.H


# ------------------------------------------------------------ distributed
def dist_setup():
    """One process per GPU (torchrun env).  The ranks are independent replicas:
    they exchange only the barrier around the timed region and the max of the
    per-rank times (NCCL on GPUs, gloo on a host without one)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
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
    """Same step through the public API with pinned host buffers: every step copies its
    inputs host->device and its results device->host inside the timed region.  The copies
    run on their own streams with two sets of device buffers, so that step i + 1's upload
    and step i - 1's download overlap step i's kernels, as a serving loop would run them.
    The host side runs on the CPUs nearest the GPU, as a serving process would be placed,
    so that the pinned buffers (first touched here) live in that CPU's memory; the process's
    CPU set is restored afterwards.  Returns (ms_per_step, h2d_bytes, d2h_bytes, cpus)."""
    allowed = os.sched_getaffinity(0)
    near = gpu_local_cpus(torch.cuda.current_device())
    if near and near != allowed:
        os.sched_setaffinity(0, near)
    try:
        r = _time_e2e(step, K, W, world)
    finally:
        os.sched_setaffinity(0, allowed)
    return r + (len(near) if near else None,)


def _time_e2e(step, K, W, world):
    cs = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    if step.op == "decode":
        n_steps = len(step.tok[0])
        host_in = [t.cpu().pin_memory() for t in step.tok]          # [n_steps, n_seq, ...]
        dev_in = [[torch.empty_like(t[0]) for t in step.tok] for _ in range(2)]
        dev_out = [[torch.empty_like(step.o_steps[0])] for _ in range(2)]
        host_in_of = lambda i: [t[i] for t in host_in]
        total = min(n_steps, W + K)
    else:
        names = ["q", "k", "v", "g", "beta", "cu_seqlens"] + (["dO"] if step.op == "fwdbwd" else [])
        srcs = [getattr(step.x_host, nm).contiguous().pin_memory() for nm in names]
        dev_in = [[torch.empty_like(getattr(step.xd, nm)) for nm in names] for _ in range(2)]
        outs0 = [step.o, step.fin] + ([step.gouts[k] for k in ("dq", "dk", "dv", "dg", "dbeta", "dh0")]
                                      if step.op == "fwdbwd" else [])
        dev_out = [outs0] + [[torch.empty_like(t) for t in outs0]]
        host_in_of = lambda i: srcs
        total = W + K
    host_out = [[torch.empty_like(t, device="cpu").pin_memory() for t in dev_out[0]] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in_of(0))
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    ev_up = [torch.cuda.Event() for _ in range(2)]     # buffer b's inputs have landed
    ev_done = [torch.cuda.Event() for _ in range(2)]   # the kernels reading/writing buffer b are done
    ev_down = [torch.cuda.Event() for _ in range(2)]   # buffer b's results have left

    def one(i):
        b = i % 2
        with torch.cuda.stream(up):
            up.wait_event(ev_done[b])          # step i - 2 no longer reads these inputs
            for hb, db in zip(host_in_of(i), dev_in[b]):
                db.copy_(hb, non_blocking=True)
            ev_up[b].record(up)
        cs.wait_event(ev_up[b])
        cs.wait_event(ev_down[b])              # step i - 2's results are on the host
        if step.op == "decode":
            q, k, v, g, bt = dev_in[b]
            step.cpr.cpr_gdn_decode_step(q, k, v, g, bt, step.cache, contract=step.c, digest=step.dig,
                                         out=dev_out[b][0])
        else:
            from infer_consistent_linear_gb300.synth import GdnInputs
            d = dict(zip(["q", "k", "v", "g", "beta", "cu_seqlens", "dO"], dev_in[b]))
            step.run(GdnInputs(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], None, d.get("dO")),
                     outs=dev_out[b])
        ev_done[b].record(cs)
        with torch.cuda.stream(down):
            down.wait_event(ev_done[b])
            for ho, do in zip(host_out[b], dev_out[b]):
                ho.copy_(do, non_blocking=True)
            ev_down[b].record(down)

    if step.op == "decode":
        step.cache.blob.copy_(step.blob0)      # replay the same tokens from the post-prefill cache
        Wd = min(W, total)
        K = min(K, total - Wd)
    else:
        Wd = W
    for i in range(Wd):
        one(i)
    torch.cuda.synchronize()
    barrier(world)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(cs)
    up.wait_event(s)
    down.wait_event(s)
    for i in range(K):
        one(Wd + i)
    cs.wait_event(ev_down[0])
    cs.wait_event(ev_down[1])
    e.record(cs)
    torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(s.elapsed_time(e) / K, world), int(h2d), int(d2h)


# ------------------------------------------------------------ roofline
def load_traffic():
    try:
        with open(TRAFFIC_FILE) as f:
            return json.load(f)
    except Exception:
        return {}


# the sources each tensor-core kernel's DRAM traffic depends on: the shared forward
# headers and launchers, plus its own header
_TC_SRC_BASE = ("common.cuh", "simt_fwd.cuh", "tc_common.cuh", "tc_fwd.cuh", "tc_launch.cu", "tc_launch.h")
_TC_SRC_OWN = {"cpr_tc_decode": ("tc_decode.cuh",), "cpr_tc_state_bwd": ("tc_bwd.cuh",),
               "cpr_tc_grad": ("tc_bwd.cuh",)}


def kernel_src_sha(name):
    """Hash of the sources kernel `name` is built from, which its stored ncu traffic
    figures belong to: a change to another kernel's header leaves them valid."""
    import hashlib
    csrc = os.path.join(ROOT, "infer_consistent_linear_gb300", "csrc")
    h = hashlib.sha256()
    for s in sorted(_TC_SRC_BASE + _TC_SRC_OWN.get(name, ())):
        with open(os.path.join(csrc, s), "rb") as f:
            h.update(s.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def step_bytes(step, out_bytes):
    """The method's algorithmic bytes of one step, with o (and for the backward dq, dk, dv)
    counted at `out_bytes` per element: q, k, v, g, beta in, o out, the final states; the
    backward reads them and dO again and writes the gradients and dh0."""
    d, H = step.d, step.H
    ht = sum(step.lens) * H
    states = len(step.lens) * H * d * d * 4
    byt = ht * algo_fwd_bytes_per_head_token(d, out_bytes=out_bytes) + states
    if step.op == "fwdbwd":
        byt += ht * algo_bwd_bytes_per_head_token(d, out_bytes=out_bytes) + states
    return byt


def roofline_for(step, prof, pk):
    """Roofline of the dominant kernel (largest share of device time).  `achieved` and
    `frac` charge the launch with ALL of the step's algorithmic bytes (the method's
    per-head-token figure with a bf16 o, times the head-tokens one launch covers, plus the
    states) over the kernel's average launch time; `frac_fp32_out` is the same with the
    fp32 o (and gradients) this build writes; `frac_kernel_share` charges the kernel only
    its own share of those bytes (what it reads or writes of the method's tensors)."""
    if not prof:
        return None
    name, (launches, total_ms) = max(prof.items(), key=lambda kv: kv[1][1])
    avg_s = total_ms / launches / 1e3
    units = step.kernel_units(name)
    traffic = None
    tr = load_traffic().get(f"{name}/{step.name}")
    # (stored for the full workload: a run on part of it, --n-seq, has none)
    if tr and tr.get("kernel_src_sha") == kernel_src_sha(name) and not N_SEQ_OVERRIDE:
        traffic = tr.get("bytes_per_launch")
    tfl = tc_kernel_flops_per_chunk(name, step.d)
    if tfl is not None:
        flops = tfl * units
        share = tc_kernel_bytes(name, step.lens, step.H, step.d)
        byt16, byt32 = step_bytes(step, 2), step_bytes(step, 4)
        ach = byt16 / avg_s / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4), "traffic": traffic,
                "traffic_gbs": round(traffic / avg_s / 1e9, 1) if traffic else None,
                "avg_launch_us": round(avg_s * 1e6, 2), "algo_bytes_per_launch": byt16,
                "bytes_rule": "all of the step's algorithmic bytes, o counted in bf16 (1,032 B per "
                              "head-token forward) plus the states, over this kernel's launch time",
                "frac_fp32_out": round(byt32 / avg_s / 1e9 / pk["hbm_gbs"], 4),
                "algo_bytes_fp32_out": byt32,
                "frac_kernel_share": round(share / avg_s / 1e9 / pk["hbm_gbs"], 4),
                "kernel_share_bytes": share,
                "tensor_frac": round(flops / avg_s / 1e12 / pk["bf16_tflops"], 4),
                "algo_flops_per_launch": flops,
                "peak_source": "measured copy bandwidth (of measured)"}
    if name in ("cpr_decode", "cpr_tc_decode"):
        byt = DECODE_ALGO_BYTES_PER_SEQ_HEAD * units
        ach = byt / avg_s / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4), "traffic": traffic,
                "traffic_gbs": round(traffic / avg_s / 1e9, 1) if traffic else None,
                "avg_launch_us": round(avg_s * 1e6, 2), "algo_bytes_per_launch": byt}
    fl = simt_kernel_flops_per_chunk(name, step.d)
    if fl is None:
        return None
    flops = fl * units
    alu_peak = 152 * 128 * 2 * pk["sm_max_mhz"] * 1e6 / 1e12  # fp32 FMA lanes x clock
    ach = flops / avg_s / 1e12
    return {"kernel": name, "bound": "alu", "achieved": round(ach, 3), "peak": round(alu_peak, 2),
            "unit": "TFLOP/s", "frac": round(ach / alu_peak, 4), "traffic": traffic,
            "avg_launch_us": round(avg_s * 1e6, 2), "algo_flops_per_launch": flops,
            "peak_source": "152 SMs x 128 fp32 lanes x 2 FLOP x max SM clock"}


def path_roofline(step, ms, pk):
    """The method's roofline for the whole step: the slower of its bytes at
    HBM bandwidth and its dense-contraction FLOPs at the bf16 tensor peak.  `frac`
    counts o in bf16 (the method's byte figure), `frac_fp32_out` in fp32."""
    byt, fl = step.algo()
    t_mma = fl / (pk["bf16_tflops"] * 1e12)
    res = {"measured_us": round(ms * 1e3, 2), "algo_flops": int(fl), "peaks": pk["source"]}
    if step.op == "decode":
        t_hbm = byt / (pk["hbm_gbs"] * 1e9)
        t = max(t_hbm, t_mma)
        return {**res, "bound": "hbm", "roofline_us": round(t * 1e6, 2), "frac": round(t / (ms / 1e3), 4),
                "algo_bytes": int(byt)}
    b16, b32 = step_bytes(step, 2), step_bytes(step, 4)
    t16, t32 = max(b16 / (pk["hbm_gbs"] * 1e9), t_mma), max(b32 / (pk["hbm_gbs"] * 1e9), t_mma)
    return {**res, "bound": "hbm" if b16 / (pk["hbm_gbs"] * 1e9) >= t_mma else "tensor",
            "roofline_us": round(t16 * 1e6, 2), "frac": round(t16 / (ms / 1e3), 4), "algo_bytes": int(b16),
            "roofline_us_fp32_out": round(t32 * 1e6, 2), "frac_fp32_out": round(t32 / (ms / 1e3), 4),
            "algo_bytes_fp32_out": int(b32)}


# ------------------------------------------------------------ CPU oracle
def cpu_sample(name, n_steps_hint=1):
    """Oracle run on a bounded sample of the workload; returns (units, seconds, desc, cores)."""
    import oracle
    from infer_consistent_linear_gb300.synth import make_inputs
    oracle.build()
    cores = oracle.default_threads()
    w = WORKLOADS[name]
    H, d = w["H"], w["d"]
    if w["op"] == "decode":
        # one decode step for every (sequence, head): one token from a full state
        n_seq = len(workload_lens(name))
        x = make_inputs([1] * n_seq, H, d, d, io_dtype=torch.bfloat16, seed=0, h0_std=0.1)
        t0 = time.perf_counter()
        oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0)
        dt = time.perf_counter() - t0
        return 1, dt, f"one decode step: {n_seq} sequences x {H} heads, fp64 recurrence", cores
    lens = workload_lens(name)
    if w["op"] == "fwd":
        sample = lens[:2]
    else:
        sample = lens[:1]
    x = make_inputs(sample, H, d, d, io_dtype=torch.bfloat16, seed=0, with_grad=(w["op"] == "fwdbwd"))
    t0 = time.perf_counter()
    oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens)
    if w["op"] == "fwdbwd":
        oracle.gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO)
    dt = time.perf_counter() - t0
    return sum(sample), dt, (f"{len(sample)} of {len(lens)} sequences ({sum(sample)} tokens) x {H} "
                             f"heads, fp64 {'fwd+bwd' if w['op'] == 'fwdbwd' else 'fwd'}"), cores


def unit_of(name):
    return ("us/step", False) if WORKLOADS[name]["op"] == "decode" else ("tokens/s", True)


def value_of(name, ms, tokens_per_step, world):
    if WORKLOADS[name]["op"] == "decode":
        return round(ms * 1e3, 3)
    return round(world * tokens_per_step / (ms / 1e3), 1)


def run_reference(args, rank, world):
    if rank != 0:
        return
    name = args.workload
    unit, hib = unit_of(name)
    times, units = [], 0
    desc = cores = None
    for i in range(args.warmup + args.steps):
        u, dt, desc, cores = cpu_sample(name)
        if i >= args.warmup:
            times.append(dt)
            units += u
    total = sum(times)
    if WORKLOADS[name]["op"] == "decode":
        value = round(total / len(times) * 1e6, 3)
    else:
        value = round(units / total, 1)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / len(times) * 1e3, 3),
            "higher_is_better": hib, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOADS[name]["desc"], "sample": desc},
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


BAD_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


def measure(step, K, W, world, local):
    """Device-timed region with clock sampling; re-measured once if the clock
    record shows a hardware/thermal slowdown."""
    for attempt in range(2):
        clocks = ClockSampler(local)
        clocks.start()
        ms, prof = time_device(step, K, W, world, profile=True)
        clocks.stop()
        ck = clocks.summary()
        if not (set(ck["reasons"]) & BAD_REASONS):
            break
        if step.op == "decode":
            break  # tokens are consumed; keep the record and report it
    ck["attempts"] = attempt + 1
    return ms, prof, ck


def kernel_table(prof, ms_total):
    tot = sum(v[1] for v in prof.values()) or 1.0
    return {k: {"launches": n, "avg_us": round(t / n * 1e3, 2), "share": round(t / tot, 4)}
            for k, (n, t) in prof.items()}


def decode_bitwise(step, n_done):
    """Decode outputs vs a one-shot forward over the full sequences (bits)."""
    cpr = step.cpr
    xd = step.xd_full
    o_full, _ = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, contract=step.c,
                                digest=step.dig, want_final=False)
    cu = xd.cu_seqlens.tolist()
    idx = torch.tensor([[cu[b] + step.lens[b] + t for b in range(len(step.lens))]
                        for t in range(n_done)], device=o_full.device).reshape(-1)
    ref = o_full.index_select(0, idx).view_as(step.o_steps[:n_done])
    return bool(torch.equal(ref.view(torch.int32), step.o_steps[:n_done].contiguous().view(torch.int32)))


def decode_step_stats(step, K, W):
    """The Decode workload's steps again, from the cache right after the prefill: first
    each step timed on its own (events between steps), for the median; then the same W + K
    steps with the last K captured once as a CUDA graph through the public API and
    replayed, timed as a whole.  The replayed outputs are compared bit for bit with the
    eager ones."""
    res = {}
    step.cache.blob.copy_(step.blob0)
    step.t = 0
    for _ in range(W):
        step.run()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    ev[0].record()
    for i in range(K):
        step.run()
        ev[i + 1].record()
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(K)]
    res.update(us_per_step_median=round(statistics.median(per), 3), us_per_step_min=round(min(per), 3),
               us_per_step_max=round(max(per), 3))
    eager = step.o_steps[W:W + K].clone()
    try:
        step.cache.blob.copy_(step.blob0)
        step.t = 0
        for _ in range(W):
            step.run()
        torch.cuda.synchronize()
        snap = step.cache.blob.clone()
        step.o_steps[W:W + K].zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(K):
                step.run()
        torch.cuda.synchronize()
        step.cache.blob.copy_(snap)      # capturing ran nothing; replay from the same cache
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        g.replay()
        e.record()
        torch.cuda.synchronize()
        res["us_per_step_graph"] = round(s.elapsed_time(e) * 1e3 / K, 3)
        res["graph_bitwise_equal_to_eager"] = bool(torch.equal(
            eager.view(torch.int32), step.o_steps[W:W + K].contiguous().view(torch.int32)))
        del g
    except Exception as exc:   # reported, not fatal to the bench line
        res["graph_error"] = f"{type(exc).__name__}: {exc}"
    return res


def secondary(name, dev, world, local, steps, warmup, pk, policy):
    n_dec = steps + warmup if WORKLOADS[name]["op"] == "decode" else 0
    st = OurStep(name, dev, n_decode_steps=n_dec, policy=policy)
    ms, prof = time_device(st, steps, warmup, world, profile=True)
    unit, hib = unit_of(name)
    res = {"workload": WORKLOADS[name]["desc"], "value": value_of(name, ms, st.tokens_per_step(), world),
           "unit": unit, "higher_is_better": hib, "ms_per_step": round(ms, 4), "steps": steps,
           "path_roofline": path_roofline(st, ms, pk), "roofline": roofline_for(st, prof, pk),
           "kernels": kernel_table(prof, ms)}
    if WORKLOADS[name]["op"] == "decode":
        res["bitwise_decode_vs_prefill"] = decode_bitwise(st, n_dec)
        res.update(decode_step_stats(st, steps, warmup))
    del st
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------ stage-table ablations
class NativeDecode:
    """"Native mixed" decode: the Decode workload's chunked (tensor-core) prefill, then
    token-recurrent steps on its fp32 final states, no resynchronisation."""

    def __init__(self, dev, n_steps):
        import infer_consistent_linear_gb300 as cpr
        from infer_consistent_linear_gb300.synth import make_inputs
        self.cpr = cpr
        self.lens = workload_lens("decode")
        H, d = WORKLOADS["decode"]["H"], WORKLOADS["decode"]["d"]
        self.c = cpr.default_contract(torch.bfloat16, d, dv_splits=2, operand_policy=cpr.CPR_POLICY_TC_BF16X3)
        full = [L + n_steps for L in self.lens]
        xd = make_inputs(full, H, d, d, io_dtype=torch.bfloat16, seed=0).to(dev)
        cu = xd.cu_seqlens.tolist()
        n_seq = len(self.lens)
        sel = torch.cat([torch.arange(cu[b], cu[b] + self.lens[b]) for b in range(n_seq)]).to(dev)
        cu_pre = torch.tensor([0] + torch.cumsum(torch.tensor(self.lens), 0).tolist(), dtype=torch.int32,
                              device=dev)
        _, self.state = cpr.cpr_gdn_fwd(xd.q[sel], xd.k[sel], xd.v[sel], xd.g[sel], xd.beta[sel], cu_pre,
                                        contract=self.c)
        idx = torch.tensor([[cu[b] + self.lens[b] + t for b in range(n_seq)] for t in range(n_steps)],
                           device=dev).reshape(-1)
        self.tok = [t.index_select(0, idx).view(n_steps, n_seq, *t.shape[1:]).contiguous()
                    for t in (xd.q, xd.k, xd.v, xd.g, xd.beta)]
        self.o_steps = torch.empty(n_steps, n_seq, H, d, device=dev)
        o_full, _ = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, contract=self.c,
                                    want_final=False)
        self.ref = o_full.index_select(0, idx).view_as(self.o_steps)   # what CPR's decode reproduces
        self.units = n_seq * H
        self.t = 0
        torch.cuda.synchronize()

    def run(self):
        q, k, v, g, b = (x[self.t] for x in self.tok)
        self.cpr.cpr_gdn_recurrent_step(q, k, v, g, b, self.state, contract=self.c, out=self.o_steps[self.t])
        self.t += 1


class ChunkwiseDecode:
    """"Chunkwise everywhere" decode on the Decode workload: every step re-runs the chunk
    forward (cpr_gdn_fwd) over the current chunk's tokens so far, for every sequence, from
    the committed chunk-start state, and the chunk's last step commits the next state.  One
    chunk of 64 steps after the 2048-token prefill; each step's packed batch of (p + 1) rows
    per sequence is laid out before timing."""

    def __init__(self, dev):
        import infer_consistent_linear_gb300 as cpr
        from infer_consistent_linear_gb300.synth import make_inputs
        self.cpr = cpr
        self.lens = workload_lens("decode")
        H, d = WORKLOADS["decode"]["H"], WORKLOADS["decode"]["d"]
        self.c = cpr.default_contract(torch.bfloat16, d, dv_splits=2, operand_policy=cpr.CPR_POLICY_TC_BF16X3)
        n_seq = len(self.lens)
        full = [L + C for L in self.lens]
        xd = make_inputs(full, H, d, d, io_dtype=torch.bfloat16, seed=0).to(dev)
        cu = xd.cu_seqlens.tolist()
        pre = torch.cat([torch.arange(cu[b], cu[b] + self.lens[b]) for b in range(n_seq)]).to(dev)
        cu_pre = torch.tensor([0] + torch.cumsum(torch.tensor(self.lens), 0).tolist(), dtype=torch.int32,
                              device=dev)
        _, self.h0 = cpr.cpr_gdn_fwd(xd.q[pre], xd.k[pre], xd.v[pre], xd.g[pre], xd.beta[pre], cu_pre,
                                     contract=self.c)
        o_full, _ = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, contract=self.c,
                                    want_final=False)
        self.batches, self.ref = [], []
        for p in range(C):
            idx = torch.cat([torch.arange(cu[b] + self.lens[b], cu[b] + self.lens[b] + p + 1)
                             for b in range(n_seq)]).to(dev)
            cub = torch.arange(0, n_seq + 1, dtype=torch.int32, device=dev) * (p + 1)
            n_tok = n_seq * (p + 1)
            last = torch.tensor([cu[b] + self.lens[b] + p for b in range(n_seq)], device=dev)
            self.batches.append(dict(q=xd.q[idx], k=xd.k[idx], v=xd.v[idx], g=xd.g[idx], beta=xd.beta[idx],
                                     cu=cub, o=torch.empty(n_tok, H, d, device=dev),
                                     last=cub[1:].long() - 1))
            self.ref.append(o_full.index_select(0, last))
        self.ws = torch.empty(cpr.workspace_bytes(self.c, cpr.CPR_OP_FWD, n_seq, n_seq * C, H),
                              dtype=torch.uint8, device=dev)
        self.fin = torch.empty_like(self.h0)
        del o_full
        self.t = 0
        torch.cuda.synchronize()

    def run(self):
        p = self.t % C
        bt = self.batches[p]
        self.cpr.cpr_gdn_fwd(bt["q"], bt["k"], bt["v"], bt["g"], bt["beta"], bt["cu"], h0=self.h0,
                             contract=self.c, out=bt["o"], final=self.fin if p == C - 1 else None,
                             want_final=p == C - 1, workspace=self.ws)
        self.t += 1

    def bitwise(self):
        """Each step's output row (the last row of every sequence's packed chunk) against the
        one-shot forward over the full sequences."""
        return bool(all(torch.equal(bt["o"].index_select(0, bt["last"]).view(torch.int32), r.view(torch.int32))
                        for bt, r in zip(self.batches, self.ref)))


class RecurrentDecode:
    """"Recurrent everywhere" decode on the Decode workload: a token-recurrent prefill of the
    2048 tokens, then token-recurrent steps on its state; compared bit for bit with the
    token recurrence over the full sequences."""

    def __init__(self, dev, n_steps):
        import infer_consistent_linear_gb300 as cpr
        from infer_consistent_linear_gb300.synth import make_inputs
        self.cpr = cpr
        self.lens = workload_lens("decode")
        H, d = WORKLOADS["decode"]["H"], WORKLOADS["decode"]["d"]
        self.c = cpr.default_contract(torch.bfloat16, d)
        full = [L + n_steps for L in self.lens]
        xd = make_inputs(full, H, d, d, io_dtype=torch.bfloat16, seed=0).to(dev)
        cu = xd.cu_seqlens.tolist()
        n_seq = len(self.lens)
        sel = torch.cat([torch.arange(cu[b], cu[b] + self.lens[b]) for b in range(n_seq)]).to(dev)
        cu_pre = torch.tensor([0] + torch.cumsum(torch.tensor(self.lens), 0).tolist(), dtype=torch.int32,
                              device=dev)
        _, self.state = cpr.cpr_gdn_recurrent_fwd(xd.q[sel], xd.k[sel], xd.v[sel], xd.g[sel], xd.beta[sel],
                                                  cu_pre, contract=self.c)
        idx = torch.tensor([[cu[b] + self.lens[b] + t for b in range(n_seq)] for t in range(n_steps)],
                           device=dev).reshape(-1)
        self.tok = [t.index_select(0, idx).view(n_steps, n_seq, *t.shape[1:]).contiguous()
                    for t in (xd.q, xd.k, xd.v, xd.g, xd.beta)]
        self.o_steps = torch.empty(n_steps, n_seq, H, d, device=dev)
        o_full, _ = cpr.cpr_gdn_recurrent_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, contract=self.c,
                                              want_final=False)
        self.ref = o_full.index_select(0, idx).view_as(self.o_steps)
        self.t = 0
        torch.cuda.synchronize()

    def run(self):
        q, k, v, g, b = (x[self.t] for x in self.tok)
        self.cpr.cpr_gdn_recurrent_step(q, k, v, g, b, self.state, contract=self.c, out=self.o_steps[self.t])
        self.t += 1


class RecurrentTrainer:
    """"Recurrent everywhere" training on the Trainer workload: the token recurrence
    forward (outputs) and its reverse recurrence (every gradient), per (sequence, head)."""

    def __init__(self, dev):
        import infer_consistent_linear_gb300 as cpr
        from infer_consistent_linear_gb300.synth import make_inputs
        self.cpr = cpr
        self.lens = workload_lens("trainer")
        H, d = WORKLOADS["trainer"]["H"], WORKLOADS["trainer"]["d"]
        self.c = cpr.default_contract(torch.bfloat16, d)
        self.xd = make_inputs(self.lens, H, d, d, io_dtype=torch.bfloat16, seed=0, with_grad=True).to(dev)
        n_tok, n_seq = sum(self.lens), len(self.lens)
        self.ws = torch.empty(cpr.recurrent_bwd_workspace_bytes(self.c, n_seq, n_tok, H), dtype=torch.uint8,
                              device=dev)
        self.o = torch.empty(n_tok, H, d, device=dev)
        self.outs = dict(dq=torch.empty(n_tok, H, d, device=dev), dk=torch.empty(n_tok, H, d, device=dev),
                         dv=torch.empty(n_tok, H, d, device=dev), dg=torch.empty(n_tok, H, device=dev),
                         dbeta=torch.empty(n_tok, H, device=dev), dh0=torch.empty(n_seq, H, d, d, device=dev))
        torch.cuda.synchronize()

    def run(self):
        x = self.xd
        self.cpr.cpr_gdn_recurrent_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, contract=self.c,
                                       want_final=False)
        self.cpr.cpr_gdn_recurrent_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, contract=self.c,
                                       workspace=self.ws, outs=self.outs)


class RecurrentPrefill:
    """"Recurrent everywhere" on the Prefill workload: the token recurrence over each
    whole sequence."""

    def __init__(self, dev):
        import infer_consistent_linear_gb300 as cpr
        from infer_consistent_linear_gb300.synth import make_inputs
        self.cpr = cpr
        self.lens = workload_lens("prefill")
        H, d = WORKLOADS["prefill"]["H"], WORKLOADS["prefill"]["d"]
        self.c = cpr.default_contract(torch.bfloat16, d)
        self.xd = make_inputs(self.lens, H, d, d, io_dtype=torch.bfloat16, seed=0).to(dev)
        torch.cuda.synchronize()

    def run(self):
        x = self.xd
        self.cpr.cpr_gdn_recurrent_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, contract=self.c)


class ContextParallelPrefill:
    """Context-parallel prefill emulated on one GPU: the Prefill workload's sequences cut
    into R chunk-aligned segments (one per emulated rank), run one after another with the
    fp32 state handed on as the next segment's h0."""

    def __init__(self, dev, R):
        import infer_consistent_linear_gb300 as cpr
        from infer_consistent_linear_gb300.synth import make_inputs
        self.cpr = cpr
        self.lens = workload_lens("prefill")
        H, d = WORKLOADS["prefill"]["H"], WORKLOADS["prefill"]["d"]
        self.c = cpr.default_contract(torch.bfloat16, d, dv_splits=2, operand_policy=cpr.CPR_POLICY_TC_BF16X3)
        x = make_inputs(self.lens, H, d, d, io_dtype=torch.bfloat16, seed=0).to(dev)
        self.o_ref, self.fin_ref = cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, contract=self.c)
        cu = x.cu_seqlens.tolist()
        n_seq = len(self.lens)
        self.segs = []
        for r in range(R):
            idx, seg_lens = [], []
            for b, L in enumerate(self.lens):
                nch = (L + C - 1) // C
                lo, hi = min(L, C * ((nch * r) // R)), min(L, C * ((nch * (r + 1)) // R))
                idx.append(torch.arange(cu[b] + lo, cu[b] + hi))
                seg_lens.append(hi - lo)
            idx = torch.cat(idx).to(dev)
            cus = torch.tensor([0] + torch.cumsum(torch.tensor(seg_lens), 0).tolist(), dtype=torch.int32,
                               device=dev)
            n_tok = int(idx.numel())
            self.segs.append(dict(idx=idx, q=x.q[idx], k=x.k[idx], v=x.v[idx], g=x.g[idx], beta=x.beta[idx],
                                  cu=cus, o=torch.empty(n_tok, H, d, device=dev),
                                  ws=torch.empty(cpr.workspace_bytes(self.c, cpr.CPR_OP_FWD, n_seq, n_tok, H),
                                                 dtype=torch.uint8, device=dev)))
        self.h = [torch.empty(n_seq, H, d, d, device=dev) for _ in range(R)]
        torch.cuda.synchronize()

    def run(self):
        h = None
        for s_, fin in zip(self.segs, self.h):
            self.cpr.cpr_gdn_fwd(s_["q"], s_["k"], s_["v"], s_["g"], s_["beta"], s_["cu"], h0=h,
                                 contract=self.c, out=s_["o"], final=fin, workspace=s_["ws"])
            h = fin

    def bitwise(self):
        ok = all(torch.equal(s_["o"].view(torch.int32), self.o_ref.index_select(0, s_["idx"]).view(torch.int32))
                 for s_ in self.segs)
        return bool(ok and torch.equal(self.h[-1].view(torch.int32), self.fin_ref.view(torch.int32)))


def context_parallel(dev, world, unsplit_ms, R=4):
    cp = ContextParallelPrefill(dev, R)
    ms, _ = time_device(cp, 10, 3, world, profile=False)
    res = {"workload": WORKLOADS["prefill"]["desc"] + f", {R} chunk-aligned segments per sequence "
                                                     "run in turn with the state handed on",
           "ms_per_step": round(ms, 4), "unsplit_ms_per_step": round(unsplit_ms, 4),
           "tokens_per_s": round(sum(cp.lens) / (ms * 1e-3) * world, 1),
           "bitwise_vs_unsplit": cp.bitwise()}
    del cp
    torch.cuda.empty_cache()
    return res


class ProjectionGemm:
    """The projection in front of the layer on the Prefill workload's tokens: X [16384,
    2048] bf16 times W [2048, 16 x 128] bf16, K in 4 fixed leaves of 512."""

    def __init__(self, dev, d_model=2048, leaf_k=512, M=None):
        import infer_consistent_linear_gb300 as cpr
        self.cpr = cpr
        w = WORKLOADS["prefill"]
        self.M = M if M is not None else sum(workload_lens("prefill"))
        self.K, self.N, self.leaf_k = d_model, w["H"] * w["d"], leaf_k
        g = torch.Generator().manual_seed(0)
        self.x = torch.randn(self.M, self.K, generator=g).to(torch.bfloat16).to(dev)
        self.w = (torch.randn(self.K, self.N, generator=g) / self.K ** 0.5).to(torch.bfloat16).to(dev)
        self.y = torch.empty(self.M, self.N, device=dev)
        torch.cuda.synchronize()

    def run(self):
        self.cpr.cpr_gemm(self.x, self.w, self.leaf_k, out=self.y)


def projection_gemm(dev, world, pk, M=None, steps=10, warmup=3):
    pg = ProjectionGemm(dev, M=M)
    ms, _ = time_device(pg, steps, warmup, world, profile=False)
    flops = 2.0 * pg.M * pg.N * pg.K
    tf = flops / (ms * 1e-3) / 1e12
    lo = min(1000, pg.M // 2)
    hi = min(pg.M, lo + 777)
    sub = pg.cpr.cpr_gemm(pg.x[lo:hi].contiguous(), pg.w, pg.leaf_k)
    inv = bool(torch.equal(sub.view(torch.int32), pg.y[lo:hi].view(torch.int32)))
    res = {"shape": f"X [{pg.M}, {pg.K}] x W [{pg.K}, {pg.N}], bf16 in, fp32 out, {pg.K // pg.leaf_k} "
                    f"leaves of {pg.leaf_k}",
           "ms": round(ms, 4), "roofline": {"bound": "tensor", "achieved": round(tf, 1),
                                            "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                                            "frac": round(tf / pk["bf16_tflops"], 4)},
           "rows_bitwise_in_a_sub_batch": inv}
    del pg, sub
    torch.cuda.empty_cache()
    return res


class ReadingB:
    """Reading B on the Prefill workload: the chunk-form training forward, then every
    chunk's outputs by the token recurrence from its boundary state."""

    def __init__(self, dev):
        import infer_consistent_linear_gb300 as cpr
        from infer_consistent_linear_gb300.synth import make_inputs
        self.cpr = cpr
        self.lens = workload_lens("prefill")
        H, d = WORKLOADS["prefill"]["H"], WORKLOADS["prefill"]["d"]
        self.H = H
        self.c = cpr.default_contract(torch.bfloat16, d, dv_splits=2, operand_policy=cpr.CPR_POLICY_TC_BF16X3,
                                      intra_order=cpr.CPR_ORDER_TOKENREC_V1)
        self.x_host = make_inputs(self.lens, H, d, d, io_dtype=torch.bfloat16, seed=0)
        self.xd = self.x_host.to(dev)
        n_tok, n_seq = sum(self.lens), len(self.lens)
        self.ws = torch.empty(cpr.workspace_bytes(self.c, cpr.CPR_OP_FWD, n_seq, n_tok, H), dtype=torch.uint8,
                              device=dev)
        torch.cuda.synchronize()

    def run(self):
        x = self.xd
        self.o, _ = self.cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, contract=self.c,
                                         workspace=self.ws)


class ReadingBDecode:
    """Reading B's decode on the Decode workload: a reading-B prefill of every sequence
    (the decode cache also keeps the running in-chunk state), then decode steps under the
    same contract (one token of the recurrence; the chunk form commits each completed
    chunk)."""

    def __init__(self, dev, n_steps, claim=True):
        import infer_consistent_linear_gb300 as cpr
        from infer_consistent_linear_gb300.synth import make_inputs
        self.cpr = cpr
        self.lens = workload_lens("decode")
        # the positions the caller knows from its lengths: a step that completes no chunk
        # runs as cpr_gdn_decode_step_nocommit (no commit launch) when `claim` is set
        self.claim = claim
        self.pos = [L % 64 for L in self.lens]
        self.claims = []
        H, d = WORKLOADS["decode"]["H"], WORKLOADS["decode"]["d"]
        self.c = cpr.default_contract(torch.bfloat16, d, dv_splits=2, operand_policy=cpr.CPR_POLICY_TC_BF16X3,
                                      intra_order=cpr.CPR_ORDER_TOKENREC_V1)
        n_seq = len(self.lens)
        xd = make_inputs(self.lens, H, d, d, io_dtype=torch.bfloat16, seed=0).to(dev)
        _, _, self.cache = cpr.cpr_gdn_prefill(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, contract=self.c,
                                               want_final=False)
        del xd
        tok = make_inputs([n_steps] * n_seq, H, d, d, io_dtype=torch.bfloat16, seed=1).to(dev)
        # token t of sequence b is row b * n_steps + t
        self.tok = [x.view(n_seq, n_steps, *x.shape[1:]).transpose(0, 1).contiguous()
                    for x in (tok.q, tok.k, tok.v, tok.g, tok.beta)]
        self.o = torch.empty(n_seq, H, d, device=dev)
        self.t = 0
        torch.cuda.synchronize()

    def run(self):
        q, k, v, g, b = (x[self.t] for x in self.tok)
        free = self.claim and all(p != 63 for p in self.pos)
        self.claims.append(free)
        self.cpr.cpr_gdn_decode_step(q, k, v, g, b, self.cache, contract=self.c, out=self.o, no_commit=free)
        self.pos = [(p + 1) % 64 for p in self.pos]
        self.t += 1


def reading_b(dev, world, reading_a_ms):
    """Speed of reading B (contract intra_order TOKENREC_V1) against reading A on the same
    workload, and how far apart the two readings' outputs are (both are checked against the
    oracle in the GPU tests)."""
    rb = ReadingB(dev)
    ms, _ = time_device(rb, 5, 2, world, profile=False)
    x = rb.xd
    ca = rb.cpr.Contract.from_buffer_copy(rb.c)      # the same contract under reading A
    ca.intra_order = rb.cpr.CPR_ORDER_ROWSEQ_V1
    oa, _ = rb.cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, contract=ca, want_final=False)
    ob = rb.o
    diff = float((ob - oa).abs().max()) / float(oa.pow(2).mean().sqrt())
    res = {"workload": WORKLOADS["prefill"]["desc"], "ms_per_step": round(ms, 4),
           "reading_a_ms_per_step": round(reading_a_ms, 4),
           "max_abs_diff_to_reading_a_over_rms": diff,
           "bitwise_equal_to_reading_a": bool(torch.equal(oa.view(torch.int32), ob.view(torch.int32)))}
    del rb, oa, ob
    torch.cuda.empty_cache()
    try:   # reading B's decode step on the Decode workload (its bits are checked in the GPU tests)
        # Step times without per-kernel events (one event pair per launch would add a few µs
        # to each of a step's launches); the kernel table from a separate profiled run
        K, W = 64, 3
        out = {"workload": WORKLOADS["decode"]["desc"], "steps": K}
        for claim, key in ((True, "us_per_step"), (False, "us_per_step_commit_every_step")):
            rd = ReadingBDecode(dev, K + W, claim=claim)
            ms_d, _ = time_device(rd, K, W, world, profile=False)
            out[key] = round(ms_d * 1e3, 3)
            if claim:
                out["timed_steps_without_commit_launch"] = int(sum(rd.claims[-K:]))
            out["error_word" if claim else "error_word_commit_every_step"] = rb_err(rd.cpr)
            del rd
            torch.cuda.empty_cache()
        rd = ReadingBDecode(dev, K + W)
        ms_p, prof_d = time_device(rd, K, W, world, profile=True)
        out["kernels"] = kernel_table(prof_d, ms_p)
        out["us_per_step_profiled"] = round(ms_p * 1e3, 3)
        del rd
        res["decode"] = out
    except Exception as e:   # reported, not fatal to the bench line
        res["decode"] = {"error": f"{type(e).__name__}: {e}"}
    torch.cuda.empty_cache()
    return res


def rb_err(cpr):
    return cpr.get_device_error(clear=True)


def stage_table(dev, world, pk, cpr_prefill_ms, sec):
    """The pages' stage comparison on this GPU: CPR (every stage bitwise consistent)
    against "native mixed" (chunked prefill and trainer, token-recurrent decode without
    resynchronisation) and "recurrent everywhere"."""
    K, W = 512, 3
    nd = NativeDecode(dev, K + W)
    ms_d, prof_d = time_device(nd, K, W, world, profile=True)
    n_steps = K + W
    bitwise = bool(torch.equal(nd.ref.view(torch.int32), nd.o_steps.contiguous().view(torch.int32)))
    us_launch = prof_d["cpr_rec_step"][1] / prof_d["cpr_rec_step"][0] * 1e3
    d = WORKLOADS["decode"]["d"]
    byt = nd.units * (2 * d * d * 4 + 3 * d * 2 + 8 + d * 4)   # state read + write, token in, o out
    native_decode = {"us_per_step": round(ms_d * 1e3, 3), "bitwise_decode_vs_prefill": bitwise,
                     "roofline": {"kernel": "cpr_rec_step", "bound": "hbm",
                                  "achieved": round(byt / (us_launch * 1e-6) / 1e9, 1),
                                  "peak": pk["hbm_gbs"], "unit": "GB/s",
                                  "frac": round(byt / (us_launch * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
                                  "algo_bytes_per_launch": byt}}
    del nd
    torch.cuda.empty_cache()
    cw = ChunkwiseDecode(dev)
    ms_cw, prof_cw = time_device(cw, C - 3, 3, world, profile=True)
    chunkwise_decode = {"us_per_step": round(ms_cw * 1e3, 3), "bitwise_decode_vs_prefill": cw.bitwise(),
                        "steps": C - 3, "kernels": kernel_table(prof_cw, ms_cw)}
    del cw
    torch.cuda.empty_cache()
    rd = RecurrentDecode(dev, K + W)
    ms_rd, _ = time_device(rd, K, W, world, profile=False)
    rec_decode = {"us_per_step": round(ms_rd * 1e3, 3),
                  "bitwise_decode_vs_prefill": bool(torch.equal(rd.ref.view(torch.int32),
                                                                rd.o_steps.contiguous().view(torch.int32)))}
    del rd
    torch.cuda.empty_cache()
    rp = RecurrentPrefill(dev)
    ms_p, _ = time_device(rp, 3, 2, world, profile=False)
    tok = sum(rp.lens)
    del rp
    torch.cuda.empty_cache()
    rt = RecurrentTrainer(dev)
    ms_t, prof_t = time_device(rt, 2, 1, world, profile=True)
    tok_t = sum(rt.lens)
    del rt
    torch.cuda.empty_cache()
    cpr_dec = sec.get("decode", {})
    cpr_tr = sec.get("trainer", {})
    return {
        "cpr": {"prefill_ms": round(cpr_prefill_ms, 4), "trainer_fwd_bwd_ms": cpr_tr.get("ms_per_step"),
                "decode_us_per_step": cpr_dec.get("value"),
                "bitwise_decode_vs_prefill": cpr_dec.get("bitwise_decode_vs_prefill")},
        "native_mixed": {"prefill_ms": round(cpr_prefill_ms, 4), "trainer_fwd_bwd_ms": cpr_tr.get("ms_per_step"),
                         "decode_us_per_step": native_decode["us_per_step"],
                         "bitwise_decode_vs_prefill": native_decode["bitwise_decode_vs_prefill"],
                         "decode_roofline": native_decode["roofline"]},
        "chunkwise_everywhere": {"prefill_ms": round(cpr_prefill_ms, 4),
                                 "trainer_fwd_bwd_ms": cpr_tr.get("ms_per_step"),
                                 "decode_us_per_step": chunkwise_decode["us_per_step"],
                                 "bitwise_decode_vs_prefill": chunkwise_decode["bitwise_decode_vs_prefill"],
                                 "decode_kernels": chunkwise_decode["kernels"]},
        "recurrent_everywhere": {"prefill_ms": round(ms_p, 4),
                                 "prefill_tokens_per_s": round(tok / (ms_p * 1e-3) * world, 1),
                                 "trainer_fwd_bwd_ms": round(ms_t, 4),
                                 "trainer_tokens_per_s": round(tok_t / (ms_t * 1e-3) * world, 1),
                                 "trainer_kernels": kernel_table(prof_t, ms_t),
                                 "decode_us_per_step": rec_decode["us_per_step"],
                                 "bitwise_decode_vs_prefill": rec_decode["bitwise_decode_vs_prefill"]},
        "note": "native mixed and chunkwise everywhere share this build's chunked prefill and "
                "trainer kernels; native mixed decodes with the token recurrence on the prefill's "
                "fp32 states (no resynchronisation), chunkwise everywhere re-runs the chunk forward "
                "over the current chunk every step, recurrent everywhere runs the token recurrence "
                "in every stage",
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="prefill")
    ap.add_argument("--no-secondary", action="store_true", help="only the headline workload")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--policy", choices=["tc", "simt"], default="tc",
                    help="operand policy of the contract (tc: tcgen05 tensor cores; simt: fp32 CUDA cores)")
    ap.add_argument("--n-seq", type=int, default=None,
                    help="run only the first n sequences of the workload (a smaller case for "
                         "profiler captures; the line then does not describe the named workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="leave out the oracle's timed CPU sample (for profiler runs)")
    ap.add_argument("--gemm-only", type=int, default=None, metavar="M",
                    help="time only the projection GEMM, on M rows of its workload, and print its "
                         "object (a case for profiler captures; no bench line)")
    args = ap.parse_args()
    global N_SEQ_OVERRIDE
    N_SEQ_OVERRIDE = args.n_seq
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import infer_consistent_linear_gb300 as cpr
    from infer_consistent_linear_gb300 import _build
    _build.build()
    cpr.load_library()
    pk = peaks()
    if args.gemm_only is not None:
        print(json.dumps(projection_gemm(dev, world, pk, M=args.gemm_only, steps=max(args.steps, 1),
                                         warmup=max(args.warmup, 1))), flush=True)
        return
    name = args.workload
    K, W = args.steps, max(args.warmup, 0)
    n_dec = K + W if WORKLOADS[name]["op"] == "decode" else 0
    step = OurStep(name, dev, n_decode_steps=n_dec, policy=args.policy)
    ms, prof, ck = measure(step, K, W, world, local)
    unit, hib = unit_of(name)
    value = value_of(name, ms, step.tokens_per_step(), world)
    e2e = None
    if not args.no_e2e:
        e_ms, h2d, d2h, ncpu = time_e2e(step, K, W, world)
        e2e = {"value": value_of(name, e_ms, step.tokens_per_step(), world), "unit": unit,
               "ms_per_step": round(e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "host_cpus_near_gpu": ncpu}
    extra = {}
    if WORKLOADS[name]["op"] == "decode":
        extra["bitwise_decode_vs_prefill"] = decode_bitwise(step, n_dec)
        extra.update(decode_step_stats(step, K, W))
    line ={"metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(ms, 4), "higher_is_better": hib, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16x3 MMA, f32 accumulate" if args.policy == "tc" else "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOADS[name]["desc"] + (f" [first {args.n_seq} sequences only]"
                                                               if args.n_seq else ""),
                       "l2": "working set > 129 MB L2, no flush",
                       "contract": {k: v for k, v in step.c.as_dict().items()},
                       "parallelism": f"replicas x{world} (independent sequences per GPU)"},
            "clocks": ck, "e2e": e2e, "gpu_launches": int(sum(n for n, _ in prof.values())),
            "roofline": roofline_for(step, prof, pk), "path_roofline": path_roofline(step, ms, pk),
            "kernels": kernel_table(prof, ms), **extra}
    del step
    torch.cuda.empty_cache()
    if not args.no_secondary:
        sec = {}
        plan = [("trainer", 5, 3), ("decode", 512, 3), ("varlen", 3, 3)]
        for nm, s, w in plan:
            if nm != name:
                sec[nm] = secondary(nm, dev, world, local, s, w, pk, args.policy)
        line["workloads"] = sec
        if name == "prefill" and args.policy == "tc" and args.n_seq is None:
            line["stage_table"] = stage_table(dev, world, pk, ms, sec)
            line["context_parallel"] = context_parallel(dev, world, ms)
            line["projection_gemm"] = projection_gemm(dev, world, pk)
            line["reading_b"] = reading_b(dev, world, ms)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        u, dt, desc, cores = cpu_sample(name)
        cv = round(dt * 1e6, 3) if WORKLOADS[name]["op"] == "decode" else round(u / dt, 1)
        line["cpu_baseline"] = {"value": cv, "unit": unit, "cores": cores, "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
