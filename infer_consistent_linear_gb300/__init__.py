"""Python binding of the CPR Gated DeltaNet library (libcpr_gdn.so).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/cpr_gdn.h.  PyTorch provides
device memory and the current stream.  There is no fallback: if the shared
library is missing or cannot be loaded, every entry point raises.

Functions carry the C names: cpr_gdn_fwd, cpr_gdn_prefill,
cpr_gdn_decode_step, cpr_gdn_bwd.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcpr_gdn.so")

CPR_OK = 0
ERRORS = {
    1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "ALIGNMENT", 4: "CONTRACT_MISMATCH",
    5: "UNALIGNED", 6: "CUDA", 7: "WORKSPACE", 8: "BAD_SEQLENS", 9: "DEVICE_TIMEOUT",
    10: "COMMIT_DUE",
}
CPR_ERR_INVALID_ARG = 1
CPR_ERR_UNSUPPORTED = 2
CPR_ERR_COMMIT_DUE = 10
CPR_DTYPE_F32 = 1
CPR_DTYPE_BF16 = 2
CPR_POLICY_SIMT_F32 = 1
CPR_POLICY_TC_BF16X3 = 2
CPR_ORDER_ROWSEQ_V1 = 1
CPR_ORDER_TOKENREC_V1 = 2   # reading B: token recurrence inside each chunk
CPR_SCHED_SEQ_CHUNKS = 1
CPR_OP_FWD = 1
CPR_OP_BWD = 2


class CprError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class Contract(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint32) for n in (
        "version", "chunk_size", "d_k", "d_v", "io_dtype", "out_dtype", "gate_dtype",
        "accum_dtype", "state_dtype", "operand_policy", "intra_order", "state_schedule",
        "dv_splits")] + [("scale", ctypes.c_float), ("kernel_build_id", ctypes.c_uint32)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class CacheLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "total_bytes", "header", "pos", "done", "state", "k_rows", "v_rows", "gam_rows",
        "beta_rows", "t_rows", "delta_rows", "state_tiles", "delta_tiles", "run", "rb_k", "rb_v",
        "rb_g", "rb_beta", "rb_cu", "rb_ws")]


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 40), ("launches", ctypes.c_uint32),
                ("total_ms", ctypes.c_double)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Loads the shared library (raises if it is absent)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"CPR GDN CUDA library not built: {path} is missing "
                          "(run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    P, I, U32, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_int64, ctypes.c_size_t
    CP = ctypes.POINTER(Contract)
    sig = {
        "cpr_kernel_build_id": (U32, []),
        "cpr_contract_init_default": (I, [CP, U32, U32, U32]),
        "cpr_contract_serialize": (I, [CP, P, ctypes.POINTER(SZ)]),
        "cpr_contract_digest": (I, [CP, P]),
        "cpr_contract_check": (I, [CP]),
        "cpr_sha256": (I, [P, SZ, P]),
        "cpr_deployment_digest": (I, [P, ctypes.c_char_p, SZ]),
        "cpr_gdn_workspace_size": (I, [CP, I, I, I64, I, ctypes.POINTER(SZ)]),
        "cpr_decode_cache_layout": (I, [CP, I, I, ctypes.POINTER(CacheLayout)]),
        "cpr_decode_cache_bytes": (I, [CP, I, I, ctypes.POINTER(SZ)]),
        "cpr_gdn_fwd": (I, [CP, P, P, P, P, P, P, P, I, I64, I, P, P, P, P, SZ, P]),
        "cpr_gdn_prefill": (I, [CP, P, P, P, P, P, P, P, I, I64, I, P, P, P, P, P, SZ, P]),
        "cpr_gdn_decode_step": (I, [CP, P, P, P, P, P, P, I, I, P, P, P]),
        "cpr_gdn_decode_step_nocommit": (I, [CP, P, P, P, P, P, P, I, I, P, P, P]),
        "cpr_gdn_bwd": (I, [CP, P, P, P, P, P, P, P, I, I64, I, P, P, P, P, P, P, P, P, P,
                            P, SZ, P]),
        "cpr_gdn_fwd_train": (I, [CP, P, P, P, P, P, P, P, I, I64, I, P, P, P, P, SZ, P]),
        "cpr_selftest_wait_timeout": (I, [U32, ctypes.POINTER(U32)]),
        "cpr_gdn_recurrent_fwd": (I, [CP, P, P, P, P, P, P, I, I64, I, P, P, P, P]),
        "cpr_gdn_recurrent_step": (I, [CP, P, P, P, P, P, I, I, P, P, P]),
        "cpr_gemm_bf16": (I, [P, P, P, I, I, I, I, P]),
        "cpr_gdn_recurrent_bwd_workspace_size": (I, [CP, I, I64, I, ctypes.POINTER(SZ)]),
        "cpr_gdn_recurrent_bwd": (I, [CP, P, P, P, P, P, P, I, I64, I, P, P, P, P, P, P, P, P, P,
                                      P, SZ, P]),
        "cpr_gdn_bwd_saved": (I, [CP, P, P, P, P, P, P, P, I, I64, I, P, P, P, P, P, P, P, P, P,
                                  P, SZ, P]),
        "cpr_gdn_fwd_noalloc": (I, [CP, P, P, P, P, P, P, P, I, I64, I, P, P, P, P]),
        "cpr_profile_begin": (I, []),
        "cpr_profile_end": (I, [P, I, ctypes.POINTER(I)]),
        "cpr_get_device_error": (I, [ctypes.POINTER(U32), I]),
        "cpr_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(rc: int):
    if rc != CPR_OK:
        raise CprError(rc, _lib.cpr_last_error().decode())


def kernel_build_id() -> int:
    return load_library().cpr_kernel_build_id()


def default_contract(io_dtype=torch.bfloat16, d_k: int = 128, d_v: Optional[int] = None,
                     **overrides) -> Contract:
    lib = load_library()
    c = Contract()
    dt = CPR_DTYPE_BF16 if io_dtype == torch.bfloat16 else CPR_DTYPE_F32
    rc = lib.cpr_contract_init_default(ctypes.byref(c), dt, d_k, d_v or d_k)
    for k_, v_ in overrides.items():
        setattr(c, k_, v_)
    if overrides:
        rc = lib.cpr_contract_check(ctypes.byref(c))
    _check(rc)
    return c


def simt_contract(io_dtype=torch.bfloat16, d_k: int = 128, d_v: Optional[int] = None,
                  **overrides) -> Contract:
    """The CUDA-core contract (operand policy SIMT_F32: fp32 fma chains) for shapes where
    the default is the tensor-core policy; d_v split count 4 at d_v >= 128, else 2."""
    kw = dict(operand_policy=CPR_POLICY_SIMT_F32, dv_splits=4 if (d_v or d_k) >= 128 else 2)
    kw.update(overrides)
    return default_contract(io_dtype, d_k, d_v, **kw)


def contract_bytes(c: Contract) -> bytes:
    lib = load_library()
    n = ctypes.c_size_t(76)
    buf = (ctypes.c_uint8 * 76)()
    _check(lib.cpr_contract_serialize(ctypes.byref(c), buf, ctypes.byref(n)))
    return bytes(buf[: n.value])


def contract_digest(c: Contract) -> bytes:
    lib = load_library()
    out = (ctypes.c_uint8 * 32)()
    _check(lib.cpr_contract_digest(ctypes.byref(c), out))
    return bytes(out)


def sha256(data: bytes) -> bytes:
    lib = load_library()
    out = (ctypes.c_uint8 * 32)()
    buf = ctypes.create_string_buffer(data, len(data))
    _check(lib.cpr_sha256(buf, len(data), out))
    return bytes(out)


def deployment_digest():
    """(digest, canonical text) of the current device's deployment identity: the compiled
    arch, the GPU, the CUDA runtime and driver and this library's kernel build."""
    lib = load_library()
    out = (ctypes.c_uint8 * 32)()
    text = ctypes.create_string_buffer(256)
    _check(lib.cpr_deployment_digest(out, text, 256))
    return bytes(out), text.value.decode()


def workspace_bytes(c: Contract, op: int, n_seq: int, n_tok: int, H: int) -> int:
    lib = load_library()
    n = ctypes.c_size_t(0)
    _check(lib.cpr_gdn_workspace_size(ctypes.byref(c), op, n_seq, n_tok, H, ctypes.byref(n)))
    return n.value


def cache_layout(c: Contract, n_seq: int, H: int) -> CacheLayout:
    lib = load_library()
    out = CacheLayout()
    _check(lib.cpr_decode_cache_layout(ctypes.byref(c), n_seq, H, ctypes.byref(out)))
    return out


def profile_begin():
    """Start recording CUDA-event timings around every library kernel launch."""
    _check(load_library().cpr_profile_begin())


def profile_end() -> dict:
    """Stop recording (synchronises); returns {kernel: (launches, total_ms)}."""
    lib = load_library()
    arr = (KernelTime * 32)()
    n = ctypes.c_int(0)
    _check(lib.cpr_profile_end(arr, 32, ctypes.byref(n)))
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms))
            for i in range(min(n.value, 32))}


def get_device_error(clear: bool = True) -> int:
    """Reads (and clears) the device error word.  Synchronises the device."""
    lib = load_library()
    code = ctypes.c_uint32(0)
    _check(lib.cpr_get_device_error(ctypes.byref(code), int(clear)))
    return code.value



def _ptr(t: Optional[torch.Tensor]):
    if t is None or t.numel() == 0:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dig(c: Contract, digest: Optional[bytes]):
    d = digest if digest is not None else contract_digest(c)
    return (ctypes.c_uint8 * 32).from_buffer_copy(d)


def _ws(c, op, n_seq, n_tok, H, device, workspace):
    need = workspace_bytes(c, op, n_seq, n_tok, H)
    if workspace is not None:
        _validate([_blob("workspace", workspace)])
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return workspace, workspace.numel()


@dataclass
class DecodeCache:
    """A caller-owned decode cache blob plus its section layout."""
    blob: torch.Tensor
    layout: CacheLayout
    n_seq: int
    H: int
    d_k: int
    d_v: int

    def state(self) -> torch.Tensor:
        """Chunk-start states H_n, [n_seq, H, d_k, d_v] fp32 (a view)."""
        n = self.n_seq * self.H * self.d_k * self.d_v
        o = self.layout.state
        return self.blob[o:o + 4 * n].view(torch.float32).view(self.n_seq, self.H, self.d_k, self.d_v)

    def pos(self) -> torch.Tensor:
        o = self.layout.pos
        return self.blob[o:o + 4 * self.n_seq].view(torch.int32)


def new_decode_cache(c: Contract, n_seq: int, H: int, device) -> DecodeCache:
    lay = cache_layout(c, n_seq, H)
    blob = torch.zeros(lay.total_bytes, dtype=torch.uint8, device=device)
    return DecodeCache(blob, lay, n_seq, H, c.d_k, c.d_v)


def _validate(specs):
    """Refuses, before anything is launched, tensors the kernels would not read as the C
    ABI describes them.  specs: (name, tensor or None, dtype, shape); None passes
    (optional arguments).  Every tensor is checked for its dtype, shape and contiguity
    first, then all must sit on one CUDA device (a host tensor would hand a kernel a host
    address)."""
    for name, t, dtype, shape in specs:
        if t is None:
            continue
        if not isinstance(t, torch.Tensor):
            raise CprError(CPR_ERR_INVALID_ARG, f"{name}: expected a torch.Tensor, got {type(t).__name__}")
        if t.dtype != dtype:
            raise CprError(CPR_ERR_INVALID_ARG, f"{name}: dtype {t.dtype}, expected {dtype}")
        if tuple(t.shape) != tuple(shape):
            raise CprError(CPR_ERR_INVALID_ARG, f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
        if not t.is_contiguous():
            raise CprError(CPR_ERR_INVALID_ARG, f"{name}: not contiguous")
    dev = None
    for name, t, _, _ in specs:
        if t is None:
            continue
        if t.device.type != "cuda":
            raise CprError(CPR_ERR_INVALID_ARG, f"{name}: on {t.device}, expected a CUDA device")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise CprError(CPR_ERR_INVALID_ARG, f"{name}: on {t.device}, the other tensors on {dev}")
    if dev is not None:
        _require_current(dev, torch.cuda.current_device())


def _require_current(dev: torch.device, current: int):
    """The kernels run on the current device's stream (and its workspace and cache are
    allocated there), so the tensors must live on the current device: addresses of another
    GPU's memory would be handed to this GPU's kernels."""
    idx = dev.index if dev.index is not None else current
    if idx != current:
        raise CprError(CPR_ERR_INVALID_ARG, f"tensors on cuda:{idx} but the current device is "
                                            f"cuda:{current} (use torch.cuda.device({idx}))")


def _check_cache(c: Contract, cache, n_seq: int, H: int):
    """A decode cache must have been made for this contract and batch shape: the kernels
    address it by the layout of (contract, n_seq, H), and the C ABI takes no size, so a
    cache made for fewer sequences or heads, another head size, or another reading (the
    reading-B layout appends a section) would be written past its end."""
    if not isinstance(cache, DecodeCache):
        raise CprError(CPR_ERR_INVALID_ARG, f"cache: expected a DecodeCache, got {type(cache).__name__}")
    if (cache.n_seq, cache.H, cache.d_k, cache.d_v) != (n_seq, H, c.d_k, c.d_v):
        raise CprError(CPR_ERR_INVALID_ARG,
                       f"cache: made for n_seq={cache.n_seq}, H={cache.H}, d_k={cache.d_k}, d_v={cache.d_v}; "
                       f"this call has n_seq={n_seq}, H={H}, d_k={c.d_k}, d_v={c.d_v}")
    need = cache_layout(c, n_seq, H)
    blob = cache.blob
    if not isinstance(blob, torch.Tensor) or blob.dtype != torch.uint8 or blob.dim() != 1:
        raise CprError(CPR_ERR_INVALID_ARG, "cache.blob: expected a 1-D uint8 tensor")
    if blob.numel() < need.total_bytes:
        raise CprError(CPR_ERR_INVALID_ARG, f"cache.blob: {blob.numel()} bytes, this contract's layout "
                                            f"needs {need.total_bytes}")
    diff = [f for f, _ in CacheLayout._fields_ if getattr(cache.layout, f) != getattr(need, f)]
    if diff:
        raise CprError(CPR_ERR_INVALID_ARG, f"cache: its layout differs from this contract's in {diff} "
                                            "(made under another contract)")


def _io_dtype(c: Contract):
    return torch.bfloat16 if c.io_dtype == CPR_DTYPE_BF16 else torch.float32


def _tok_specs(c: Contract, q, k, v, g, beta, cu_seqlens=None, h0=None, sfx=""):
    """Specs of one call's token tensors ([n, H, d]: n tokens, or n sequences for a decode
    step) under the contract; returns (specs, n, H)."""
    if not isinstance(q, torch.Tensor) or q.dim() != 3:
        raise CprError(CPR_ERR_INVALID_ARG, f"q{sfx}: expected a [n, H, d_k] tensor")
    n, H = int(q.shape[0]), int(q.shape[1])
    io = _io_dtype(c)
    specs = [("q" + sfx, q, io, (n, H, c.d_k)), ("k" + sfx, k, io, (n, H, c.d_k)),
             ("v" + sfx, v, io, (n, H, c.d_v)), ("g" + sfx, g, torch.float32, (n, H)),
             ("beta" + sfx, beta, torch.float32, (n, H))]
    if cu_seqlens is not None:
        if not isinstance(cu_seqlens, torch.Tensor) or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1:
            raise CprError(CPR_ERR_INVALID_ARG, "cu_seqlens: expected an int32 [n_seq + 1] tensor")
        specs += [("cu_seqlens", cu_seqlens, torch.int32, (cu_seqlens.numel(),)),
                  ("h0", h0, torch.float32, (cu_seqlens.numel() - 1, H, c.d_k, c.d_v))]
    return specs, n, H


def _blob(name, t):
    return (name, t, torch.uint8, (t.numel(),) if isinstance(t, torch.Tensor) else ())


def _shape_args(q, v, cu_seqlens):
    n_tok, H, _ = q.shape
    return int(n_tok), int(H), int(cu_seqlens.numel() - 1)


def cpr_gdn_fwd(q, k, v, g, beta, cu_seqlens, h0=None, contract: Optional[Contract] = None,
                digest: Optional[bytes] = None, want_final: bool = True, out=None,
                final=None, workspace=None, train: bool = False):
    """Trainer forward.  Returns (o [n_tok,H,d_v] fp32, final [n_seq,H,d_k,d_v] or None).
    With train=True (cpr_gdn_fwd_train) the workspace -- CPR_OP_BWD-sized, required -- also
    keeps the tiles cpr_gdn_bwd(..., saved=True) reads instead of recomputing the forward."""
    lib = load_library()
    c = contract or default_contract(q.dtype, q.shape[-1], v.shape[-1])
    specs, n_tok, H = _tok_specs(c, q, k, v, g, beta, cu_seqlens, h0)
    n_seq = int(cu_seqlens.numel() - 1)
    _validate(specs + [("out", out, torch.float32, (n_tok, H, c.d_v)),
                       ("final", final, torch.float32, (n_seq, H, c.d_k, c.d_v)),
                       _blob("workspace", workspace) if workspace is not None else ("workspace", None, None, None)])
    o = out if out is not None else torch.empty(n_tok, H, c.d_v, dtype=torch.float32, device=q.device)
    fin = final if final is not None else (
        torch.empty(n_seq, H, c.d_k, c.d_v, dtype=torch.float32, device=q.device) if want_final else None)
    if train and workspace is None:
        raise CprError(CPR_ERR_INVALID_ARG, "train=True needs a caller-owned CPR_OP_BWD workspace "
                                            "(passed on to the saved backward)")
    ws, wsb = _ws(c, CPR_OP_BWD if train else CPR_OP_FWD, n_seq, n_tok, H, q.device, workspace)
    fn = lib.cpr_gdn_fwd_train if train else lib.cpr_gdn_fwd
    _check(fn(ctypes.byref(c), _dig(c, digest), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
              _ptr(beta), _ptr(cu_seqlens), n_seq, n_tok, H, _ptr(h0), _ptr(o),
              _ptr(fin), _ptr(ws), wsb, _stream()))
    return o, fin


def cpr_gdn_prefill(q, k, v, g, beta, cu_seqlens, h0=None, contract: Optional[Contract] = None,
                    digest: Optional[bytes] = None, want_final: bool = True, cache=None,
                    out=None, workspace=None):
    """Rollout prefill.  Returns (o, final or None, DecodeCache)."""
    lib = load_library()
    c = contract or default_contract(q.dtype, q.shape[-1], v.shape[-1])
    specs, n_tok, H = _tok_specs(c, q, k, v, g, beta, cu_seqlens, h0)
    n_seq = int(cu_seqlens.numel() - 1)
    if cache is not None:
        _check_cache(c, cache, n_seq, H)
    _validate(specs + [("out", out, torch.float32, (n_tok, H, c.d_v)),
                       _blob("cache.blob", cache.blob) if cache is not None else ("cache", None, None, None),
                       _blob("workspace", workspace) if workspace is not None else ("workspace", None, None, None)])
    o = out if out is not None else torch.empty(n_tok, H, c.d_v, dtype=torch.float32, device=q.device)
    fin = torch.empty(n_seq, H, c.d_k, c.d_v, dtype=torch.float32, device=q.device) if want_final else None
    cache = cache or new_decode_cache(c, n_seq, H, q.device)
    ws, wsb = _ws(c, CPR_OP_FWD, n_seq, n_tok, H, q.device, workspace)
    _check(lib.cpr_gdn_prefill(ctypes.byref(c), _dig(c, digest), _ptr(q), _ptr(k), _ptr(v),
                               _ptr(g), _ptr(beta), _ptr(cu_seqlens), n_seq, n_tok, H, _ptr(h0),
                               _ptr(o), _ptr(fin), _ptr(cache.blob), _ptr(ws), wsb, _stream()))
    return o, fin, cache


def cpr_gdn_decode_step(q_t, k_t, v_t, g_t, beta_t, cache: DecodeCache,
                        contract: Optional[Contract] = None, digest: Optional[bytes] = None,
                        out=None, no_commit: bool = False):
    """One decode step; tokens [n_seq, H, d].  Returns o_t [n_seq, H, d_v] fp32.
    no_commit=True (cpr_gdn_decode_step_nocommit): the caller states that no sequence
    completes its chunk in this step; checked on the device (CPR_ERR_COMMIT_DUE)."""
    lib = load_library()
    c = contract or default_contract(q_t.dtype, q_t.shape[-1], v_t.shape[-1])
    specs, n_seq, H = _tok_specs(c, q_t, k_t, v_t, g_t, beta_t, sfx="_t")
    _check_cache(c, cache, n_seq, H)
    _validate(specs + [("out", out, torch.float32, (n_seq, H, c.d_v)), _blob("cache.blob", cache.blob)])
    o = out if out is not None else torch.empty(n_seq, H, c.d_v, dtype=torch.float32, device=q_t.device)
    fn = lib.cpr_gdn_decode_step_nocommit if no_commit else lib.cpr_gdn_decode_step
    _check(fn(ctypes.byref(c), _dig(c, digest), _ptr(q_t), _ptr(k_t), _ptr(v_t), _ptr(g_t),
              _ptr(beta_t), n_seq, H, _ptr(cache.blob), _ptr(o), _stream()))
    return o


def cpr_gdn_bwd(q, k, v, g, beta, cu_seqlens, dO, h0=None, dHT=None,
                contract: Optional[Contract] = None, digest: Optional[bytes] = None,
                workspace=None, outs=None, saved: bool = False):
    """Trainer backward.  Returns dict dq, dk, dv (fp32), dg, dbeta, dh0.  With saved=True
    (cpr_gdn_bwd_saved) `workspace` is the one a cpr_gdn_fwd(..., train=True) call filled
    for the same inputs; the forward is then not recomputed."""
    if saved and workspace is None:
        raise CprError(CPR_ERR_INVALID_ARG, "saved=True needs the training forward's workspace")
    lib = load_library()
    c = contract or default_contract(q.dtype, q.shape[-1], v.shape[-1])
    specs, n_tok, H = _tok_specs(c, q, k, v, g, beta, cu_seqlens, h0)
    n_seq = int(cu_seqlens.numel() - 1)
    dev = q.device
    if dO is None:
        raise CprError(CPR_ERR_INVALID_ARG, "dO is required")
    specs += [("dO", dO, torch.float32, (n_tok, H, c.d_v)), ("dHT", dHT, torch.float32, (n_seq, H, c.d_k, c.d_v))]
    if outs is not None:
        specs += [(name, outs.get(name), torch.float32, shape) for name, shape in (
            ("dq", (n_tok, H, c.d_k)), ("dk", (n_tok, H, c.d_k)), ("dv", (n_tok, H, c.d_v)),
            ("dg", (n_tok, H)), ("dbeta", (n_tok, H)), ("dh0", (n_seq, H, c.d_k, c.d_v)))]
    if workspace is not None:
        specs.append(_blob("workspace", workspace))
    _validate(specs)
    if outs is None:
        outs = dict(dq=torch.empty(n_tok, H, c.d_k, dtype=torch.float32, device=dev),
                    dk=torch.empty(n_tok, H, c.d_k, dtype=torch.float32, device=dev),
                    dv=torch.empty(n_tok, H, c.d_v, dtype=torch.float32, device=dev),
                    dg=torch.empty(n_tok, H, dtype=torch.float32, device=dev),
                    dbeta=torch.empty(n_tok, H, dtype=torch.float32, device=dev),
                    dh0=torch.empty(n_seq, H, c.d_k, c.d_v, dtype=torch.float32, device=dev))
    ws, wsb = _ws(c, CPR_OP_BWD, n_seq, n_tok, H, dev, workspace)
    fn = lib.cpr_gdn_bwd_saved if saved else lib.cpr_gdn_bwd
    _check(fn(ctypes.byref(c), _dig(c, digest), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                           _ptr(beta), _ptr(cu_seqlens), n_seq, n_tok, H, _ptr(h0), _ptr(dO),
                           _ptr(dHT), _ptr(outs["dq"]), _ptr(outs["dk"]), _ptr(outs["dv"]),
                           _ptr(outs["dg"]), _ptr(outs["dbeta"]), _ptr(outs["dh0"]), _ptr(ws),
                           wsb, _stream()))
    return outs


def cpr_gdn_recurrent_fwd(q, k, v, g, beta, cu_seqlens, h0=None, contract: Optional[Contract] = None,
                          want_final: bool = True):
    """Stage-table ablation "recurrent everywhere": the token recurrence over whole
    sequences (cpr_gdn_recurrent_fwd).  Returns (o fp32, final_state or None)."""
    lib = load_library()
    c = contract or default_contract(q.dtype, q.shape[-1], v.shape[-1])
    specs, n_tok, H = _tok_specs(c, q, k, v, g, beta, cu_seqlens, h0)
    _validate(specs)
    n_seq = int(cu_seqlens.numel() - 1)
    o = torch.empty(n_tok, H, c.d_v, dtype=torch.float32, device=q.device)
    fin = (torch.empty(n_seq, H, c.d_k, c.d_v, dtype=torch.float32, device=q.device)
           if want_final else None)
    _check(lib.cpr_gdn_recurrent_fwd(ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                     _ptr(cu_seqlens), n_seq, n_tok, H, _ptr(h0), _ptr(o), _ptr(fin),
                                     _stream()))
    return o, fin


def cpr_gdn_recurrent_step(q_t, k_t, v_t, g_t, beta_t, state, contract: Optional[Contract] = None,
                           out=None):
    """Stage-table ablation "native" decode: one token per sequence on the fp32 state
    [n_seq, H, d_k, d_v], updated in place (cpr_gdn_recurrent_step).  Returns o_t fp32."""
    lib = load_library()
    c = contract or default_contract(q_t.dtype, q_t.shape[-1], v_t.shape[-1])
    specs, n_seq, H = _tok_specs(c, q_t, k_t, v_t, g_t, beta_t, sfx="_t")
    if state is None:
        raise CprError(CPR_ERR_INVALID_ARG, "state is required")
    _validate(specs + [("state", state, torch.float32, (n_seq, H, c.d_k, c.d_v)),
                       ("out", out, torch.float32, (n_seq, H, c.d_v))])
    o = out if out is not None else torch.empty(n_seq, H, c.d_v, dtype=torch.float32, device=q_t.device)
    _check(lib.cpr_gdn_recurrent_step(ctypes.byref(c), _ptr(q_t), _ptr(k_t), _ptr(v_t), _ptr(g_t),
                                      _ptr(beta_t), n_seq, H, _ptr(state), _ptr(o), _stream()))
    return o


def recurrent_bwd_workspace_bytes(c: Contract, n_seq: int, n_tok: int, H: int) -> int:
    lib = load_library()
    n = ctypes.c_size_t(0)
    _check(lib.cpr_gdn_recurrent_bwd_workspace_size(ctypes.byref(c), n_seq, n_tok, H, ctypes.byref(n)))
    return n.value


def cpr_gdn_recurrent_bwd(q, k, v, g, beta, cu_seqlens, dO, h0=None, dHT=None,
                          contract: Optional[Contract] = None, workspace=None, outs=None):
    """Stage-table ablation "recurrent everywhere", training: the backward of
    cpr_gdn_recurrent_fwd by the reverse token recurrence (cpr_gdn_recurrent_bwd).  Returns
    dict dq, dk, dv, dg, dbeta, dh0 (fp32)."""
    lib = load_library()
    c = contract or default_contract(q.dtype, q.shape[-1], v.shape[-1])
    specs, n_tok, H = _tok_specs(c, q, k, v, g, beta, cu_seqlens, h0)
    n_seq = int(cu_seqlens.numel() - 1)
    if dO is None:
        raise CprError(CPR_ERR_INVALID_ARG, "dO is required")
    specs += [("dO", dO, torch.float32, (n_tok, H, c.d_v)), ("dHT", dHT, torch.float32, (n_seq, H, c.d_k, c.d_v))]
    if outs is not None:
        specs += [(name, outs.get(name), torch.float32, shape) for name, shape in (
            ("dq", (n_tok, H, c.d_k)), ("dk", (n_tok, H, c.d_k)), ("dv", (n_tok, H, c.d_v)),
            ("dg", (n_tok, H)), ("dbeta", (n_tok, H)), ("dh0", (n_seq, H, c.d_k, c.d_v)))]
    if workspace is not None:
        specs.append(_blob("workspace", workspace))
    _validate(specs)
    need = recurrent_bwd_workspace_bytes(c, n_seq, n_tok, H)
    dev = q.device
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    if outs is None:
        outs = dict(dq=torch.empty(n_tok, H, c.d_k, dtype=torch.float32, device=dev),
                    dk=torch.empty(n_tok, H, c.d_k, dtype=torch.float32, device=dev),
                    dv=torch.empty(n_tok, H, c.d_v, dtype=torch.float32, device=dev),
                    dg=torch.empty(n_tok, H, dtype=torch.float32, device=dev),
                    dbeta=torch.empty(n_tok, H, dtype=torch.float32, device=dev),
                    dh0=torch.empty(n_seq, H, c.d_k, c.d_v, dtype=torch.float32, device=dev))
    _check(lib.cpr_gdn_recurrent_bwd(ctypes.byref(c), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                     _ptr(cu_seqlens), n_seq, n_tok, H, _ptr(h0), _ptr(dO), _ptr(dHT),
                                     _ptr(outs["dq"]), _ptr(outs["dk"]), _ptr(outs["dv"]), _ptr(outs["dg"]),
                                     _ptr(outs["dbeta"]), _ptr(outs["dh0"]), _ptr(workspace),
                                     workspace.numel(), _stream()))
    return outs


def cpr_gemm(x, w, leaf_k: int, out=None):
    """Batch-invariant projection GEMM (cpr_gemm_bf16): x bf16 [M, K], w bf16 [K, N] ->
    fp32 [M, N], K in fixed leaves of leaf_k rows."""
    lib = load_library()
    if not isinstance(x, torch.Tensor) or x.dim() != 2 or not isinstance(w, torch.Tensor) or w.dim() != 2:
        raise CprError(CPR_ERR_INVALID_ARG, "cpr_gemm: x [M, K] and w [K, N] matrices expected")
    M, K = int(x.shape[0]), int(x.shape[1])
    N = int(w.shape[1])
    _validate([("x", x, torch.bfloat16, (M, K)), ("w", w, torch.bfloat16, (K, N)),
               ("out", out, torch.float32, (M, N))])
    y = out if out is not None else torch.empty(M, N, dtype=torch.float32, device=x.device)
    _check(lib.cpr_gemm_bf16(_ptr(x), _ptr(w), _ptr(y), M, N, K, leaf_k, _stream()))
    return y


def selftest_wait_timeout(poll_limit: int = 4096) -> bool:
    """Runs the device's bounded-wait expiry path once (see include/cpr_gdn.h);
    returns True when the wait ran out as it must."""
    lib = load_library()
    done = ctypes.c_uint32(1)
    _check(lib.cpr_selftest_wait_timeout(poll_limit, ctypes.byref(done)))
    return done.value == 0
