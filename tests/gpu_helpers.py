"""Helpers shared by the GPU test modules."""
import numpy as np
import torch

import infer_consistent_linear_gb300 as cpr
import oracle

# Parity bar: max|gpu - oracle| <= TOL * RMS(oracle), per tensor;
# bf16 inputs: 4e-3, fp32 inputs: 1e-5.
TOL_BF16 = 4e-3
TOL_F32 = 1e-5


def rel_err(got, ref) -> float:
    if isinstance(got, torch.Tensor):
        got = got.detach().cpu().double().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return float(np.max(np.abs(got - ref))) / max(rms, 1e-300)


def assert_close(name, got, ref, tol):
    e = rel_err(got, ref)
    assert e <= tol, f"{name}: max|err|/RMS = {e:.3e} > {tol:.1e}"
    return e


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.int32)


def assert_bitwise(name, a, b):
    assert a.shape == b.shape, (name, a.shape, b.shape)
    if not torch.equal(bits(a), bits(b)):
        n = int((bits(a) != bits(b)).sum())
        raise AssertionError(f"{name}: {n} of {a.numel()} elements differ in bits")


def seq_head_slice(x, b, h):
    """Inputs of one (sequence, head) as a single-sequence, single-head batch."""
    cu = x.cu_seqlens.tolist()
    a, e = cu[b], cu[b + 1]
    sl = lambda t: t[a:e, h:h + 1]
    h0 = None if x.h0 is None else x.h0[b:b + 1, h:h + 1]
    dO = None if x.dO is None else sl(x.dO)
    return sl(x.q), sl(x.k), sl(x.v), sl(x.g), sl(x.beta), [0, e - a], h0, dO


def oracle_fwd_sh(x, b, h):
    q, k, v, g, beta, cu, h0, _ = seq_head_slice(x, b, h)
    return oracle.gdn_fwd(q, k, v, g, beta, cu, h0=h0)


def oracle_bwd_sh(x, b, h, dHT=None):
    q, k, v, g, beta, cu, h0, dO = seq_head_slice(x, b, h)
    return oracle.gdn_bwd(q, k, v, g, beta, cu, dO, h0=h0, dHT=dHT)


def require_gpu():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from infer_consistent_linear_gb300 import _build
    _build.build()
    cpr.load_library()
    oracle.build()
