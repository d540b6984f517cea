"""CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it.

The arithmetic lives in ``gdn_oracle.cpp`` (fp64 token recurrence and its
hand-derived reverse recurrence); this module compiles it with g++ and wraps
it with ctypes.  See that file's header for the definition it follows
(page "IsoExec: 切换 SkyRL 中的训练器-推理不匹配", section
"Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet": Gated DeltaNet with a
recurrent decode form).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.cpp")
_LIB = os.path.join(_HERE, "_gdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library in place (g++, -O2, no fast-math)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
                   "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp]
            subprocess.check_call(cmd)
            os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    lib.oracle_gdn_fwd.argtypes = [I, P, I, I, I, D, P, P, P, P, P, P, P, P, I]
    lib.oracle_gdn_fwd.restype = I
    lib.oracle_gdn_bwd.argtypes = [I, P, I, I, I, D, P, P, P, P, P, P, P, P,
                                   P, P, P, P, P, P, I, I]
    lib.oracle_gdn_bwd.restype = I
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(_LIB)
    return _lib


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _shapes(q, v, cu):
    n_tok, H, dk = q.shape
    dv = v.shape[2]
    return n_tok, H, dk, dv, len(cu) - 1


def gdn_fwd(q, k, v, g, beta, cu_seqlens, h0=None, scale=1.0, n_threads=None, _lib_override=None):
    """fp64 forward.  Returns (o [n_tok,H,dv], hT [n_seq,H,dk,dv])."""
    lib = _lib_override or _load()
    q, k, v, g, beta, h0 = map(_f64, (q, k, v, g, beta, h0))
    cu = np.ascontiguousarray(np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens), dtype=np.int32)
    n_tok, H, dk, dv, n_seq = _shapes(q, v, cu)
    assert k.shape == q.shape and v.shape[:2] == (n_tok, H) and g.shape == (n_tok, H) == beta.shape
    assert int(cu[-1]) == n_tok
    o = np.zeros((n_tok, H, dv))
    hT = np.zeros((n_seq, H, dk, dv))
    rc = lib.oracle_gdn_fwd(n_seq, _ptr(cu), H, dk, dv, float(scale), _ptr(q), _ptr(k), _ptr(v),
                            _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(hT),
                            int(n_threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_gdn_fwd: bad arguments")
    return o, hT


def gdn_bwd(q, k, v, g, beta, cu_seqlens, dO, h0=None, dHT=None, scale=1.0, seg=64,
            n_threads=None, _lib_override=None):
    """fp64 backward.  Returns dict dq, dk, dv, dg, dbeta, dh0."""
    lib = _lib_override or _load()
    q, k, v, g, beta, h0, dO, dHT = map(_f64, (q, k, v, g, beta, h0, dO, dHT))
    cu = np.ascontiguousarray(np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens), dtype=np.int32)
    n_tok, H, dk, dv, n_seq = _shapes(q, v, cu)
    assert int(cu[-1]) == n_tok and dO.shape == (n_tok, H, dv)
    out = dict(dq=np.zeros((n_tok, H, dk)), dk=np.zeros((n_tok, H, dk)),
               dv=np.zeros((n_tok, H, dv)), dg=np.zeros((n_tok, H)),
               dbeta=np.zeros((n_tok, H)), dh0=np.zeros((n_seq, H, dk, dv)))
    rc = lib.oracle_gdn_bwd(n_seq, _ptr(cu), H, dk, dv, float(scale), _ptr(q), _ptr(k), _ptr(v),
                            _ptr(g), _ptr(beta), _ptr(h0), _ptr(dO), _ptr(dHT),
                            _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
                            _ptr(out["dbeta"]), _ptr(out["dh0"]), int(seg),
                            int(n_threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_gdn_bwd: bad arguments")
    return out


class OracleBuild:
    """The same wrapper bound to another build of the oracle source (used by
    the mutation test, which compiles deliberately broken copies)."""

    def __init__(self, so_path):
        self._lib = _bind(so_path)

    def gdn_fwd(self, *a, **kw):
        return gdn_fwd(*a, _lib_override=self._lib, **kw)

    def gdn_bwd(self, *a, **kw):
        return gdn_bwd(*a, _lib_override=self._lib, **kw)


def gemm(x, w):
    """Projection oracle: Y = X W in fp64 (numpy matmul of the exact inputs), the
    definition the batch-invariant split-K GEMM is checked against.  Pinned in
    tests/test_oracle_gemm.py against a brute-force triple loop on small shapes."""
    return _f64(x) @ _f64(w)
