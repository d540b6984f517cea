"""Host-side checks of the C ABI (no GPU needed): the library loads and
exports every function include/cpr_gdn.h declares; contract serialisation,
SHA-256 digest and claim checks; layouts; argument validation paths that
return before any CUDA call."""
import ctypes
import hashlib
import os
import re
import struct

import pytest
import torch

import infer_consistent_linear_gb300 as cpr
from infer_consistent_linear_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "cpr_gdn.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return cpr.load_library()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cpr_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 17
    for n in names:
        assert hasattr(lib, n), n


@pytest.mark.parametrize("n", [0, 1, 3, 55, 56, 63, 64, 65, 119, 120, 1000])
def test_sha256_matches_hashlib(lib, n):
    data = bytes((i * 37 + 11) & 0xFF for i in range(n))
    assert cpr.sha256(data) == hashlib.sha256(data).digest()


def test_contract_serialisation_and_digest(lib):
    c = cpr.default_contract(torch.bfloat16, 128)
    raw = cpr.contract_bytes(c)
    assert len(raw) == 76 and raw[:16] == b"CPR-GDN-CONTRACT"
    fields = struct.unpack("<13IfI", raw[16:])
    assert fields[0] == 1 and fields[1] == 64 and fields[2] == 128 and fields[3] == 128
    assert fields[13] == 1.0 and fields[14] == cpr.kernel_build_id()
    assert cpr.contract_digest(c) == hashlib.sha256(raw).digest()


def test_digest_changes_with_every_field(lib):
    base = cpr.default_contract(torch.bfloat16, 128)
    seen = {cpr.contract_digest(base)}
    for name, _ in cpr.Contract._fields_:
        c = cpr.Contract.from_buffer_copy(base)
        if name == "scale":
            c.scale = 0.5
        else:
            setattr(c, name, getattr(c, name) + 1)
        d = cpr.contract_digest(c)
        assert d not in seen, name
        seen.add(d)


def test_contract_checks(lib):
    c = cpr.default_contract(torch.bfloat16, 128)
    assert lib.cpr_contract_check(ctypes.byref(c)) == 0
    for field, val in [("chunk_size", 32), ("d_k", 96), ("operand_policy", 9), ("dv_splits", 3),
                       ("kernel_build_id", 999), ("version", 2), ("out_dtype", cpr.CPR_DTYPE_BF16)]:
        x = cpr.Contract.from_buffer_copy(c)
        setattr(x, field, val)
        assert lib.cpr_contract_check(ctypes.byref(x)) == 2, field
    x = cpr.Contract.from_buffer_copy(c)
    x.scale = float("nan")
    assert lib.cpr_contract_check(ctypes.byref(x)) == 1
    with pytest.raises(cpr.CprError):
        cpr.default_contract(torch.float32, 128)  # fp32 io: d = 64 only


def test_tensor_core_contract_rules(lib):
    c = cpr.default_contract(torch.bfloat16, 128, operand_policy=cpr.CPR_POLICY_TC_BF16X3,
                             dv_splits=2)
    assert lib.cpr_contract_check(ctypes.byref(c)) == 0
    assert cpr.contract_digest(c) != cpr.contract_digest(cpr.simt_contract(torch.bfloat16, 128, dv_splits=2))
    for field, val in [("dv_splits", 1), ("d_k", 64), ("io_dtype", cpr.CPR_DTYPE_F32)]:
        x = cpr.Contract.from_buffer_copy(c)
        setattr(x, field, val)
        if field == "d_k":
            x.d_v = 64
        assert lib.cpr_contract_check(ctypes.byref(x)) == 2, field
    # the TC forward workspace is one operand block per (chunk, head)
    n_chunks = 4 * 4096 // 64 + 4
    assert cpr.workspace_bytes(c, cpr.CPR_OP_FWD, 4, 4 * 4096, 16) >= n_chunks * 16 * 114944


def test_workspace_and_cache_layout(lib):
    c = cpr.default_contract(torch.bfloat16, 128)
    f = cpr.workspace_bytes(c, cpr.CPR_OP_FWD, 4, 4 * 4096, 16)
    b = cpr.workspace_bytes(c, cpr.CPR_OP_BWD, 4, 4 * 4096, 16)
    chunks = (4 * 4096) // 64 + 4
    assert f >= chunks * 16 * (64 * 128 * 4 * 2 + 64 * 64 * 4)
    assert b > f
    lay = cpr.cache_layout(c, 64, 32)
    offs = [lay.header, lay.pos, lay.done, lay.state, lay.k_rows, lay.v_rows, lay.gam_rows,
            lay.beta_rows, lay.t_rows, lay.delta_rows, lay.state_tiles, lay.delta_tiles]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lay.k_rows - lay.state >= 64 * 32 * 128 * 128 * 4
    assert lay.state_tiles - lay.delta_rows >= 64 * 32 * 64 * 128 * 4
    assert lay.delta_tiles - lay.state_tiles >= 64 * 32 * 128 * 128 * 4
    assert lay.total_bytes >= lay.delta_tiles + 64 * 32 * 64 * 128 * 4


def _call_fwd(lib, c, digest, ptrs, n_seq=1, n_tok=64, H=1, ws_bytes=1 << 30):
    q, k, v, g, beta, cu, o, ws = ptrs
    return lib.cpr_gdn_fwd(ctypes.byref(c), digest, q, k, v, g, beta, cu, n_seq, n_tok, H, None, o,
                           None, ws, ws_bytes, None)


def test_host_argument_errors(lib):
    c = cpr.default_contract(torch.bfloat16, 128)
    dig = (ctypes.c_uint8 * 32).from_buffer_copy(cpr.contract_digest(c))
    good = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(8)]
    bad = (ctypes.c_uint8 * 32).from_buffer_copy(bytes(32))
    assert _call_fwd(lib, c, bad, good) == 4          # digest mismatch
    p = list(good)
    p[0] = None
    assert _call_fwd(lib, c, dig, p) == 1             # null q
    p = list(good)
    p[2] = ctypes.c_void_p(0x10008)
    assert _call_fwd(lib, c, dig, p) == 3             # misaligned v
    assert _call_fwd(lib, c, dig, good, H=0) == 1
    assert _call_fwd(lib, c, dig, good, n_seq=-1) == 1
    assert _call_fwd(lib, c, dig, good, ws_bytes=16) == 7
    p = list(good)
    p[7] = ctypes.c_void_p(0x10010)
    assert _call_fwd(lib, c, dig, p) == 7             # workspace not 256-aligned
    x = cpr.Contract.from_buffer_copy(c)
    x.chunk_size = 128
    dx = (ctypes.c_uint8 * 32).from_buffer_copy(cpr.contract_digest(x))
    assert _call_fwd(lib, x, dx, good) == 2           # unsupported, even with its own digest
    assert "chunk_size" in lib.cpr_last_error().decode()
    assert lib.cpr_gdn_prefill(ctypes.byref(c), dig, *good[:6], 1, 64, 1, None, good[6], None,
                               None, good[7], 1 << 30, None) == 1   # cache required
    assert lib.cpr_gdn_decode_step(ctypes.byref(c), dig, *good[:5], 1, 1, None, good[6], None) == 1


def test_training_forward_and_saved_backward_need_tc_contract(lib):
    c = cpr.simt_contract(torch.bfloat16, 128)
    dig = (ctypes.c_uint8 * 32).from_buffer_copy(cpr.contract_digest(c))
    p = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(8)]
    rc = lib.cpr_gdn_fwd_train(ctypes.byref(c), dig, *p[:6], 1, 64, 1, None, p[6], None, p[7],
                               1 << 40, None)
    assert rc == 2 and "tensor-core" in lib.cpr_last_error().decode()
    rc = lib.cpr_gdn_bwd_saved(ctypes.byref(c), dig, *p[:6], 1, 64, 1, None, p[6], None,
                               *[ctypes.c_void_p(0x20000 * (i + 1)) for i in range(6)], p[7], 1 << 40, None)
    assert rc == 2
    t = cpr.default_contract(torch.bfloat16, 128, operand_policy=cpr.CPR_POLICY_TC_BF16X3, dv_splits=2)
    dt = (ctypes.c_uint8 * 32).from_buffer_copy(cpr.contract_digest(t))
    small = cpr.workspace_bytes(t, cpr.CPR_OP_FWD, 1, 64, 1)
    assert cpr.workspace_bytes(t, cpr.CPR_OP_BWD, 1, 64, 1) > small
    rc = lib.cpr_gdn_fwd_train(ctypes.byref(t), dt, *p[:6], 1, 64, 1, None, p[6], None, p[7],
                               small, None)
    assert rc == 7                                          # a forward-sized workspace is too small


def test_sector_store_outputs_need_32_byte_alignment(lib):
    """dq, dk under the tensor-core policy and the GEMM's Y are written in whole 32-byte
    sectors: a pointer that is 16- but not 32-byte aligned is refused on the host."""
    t = cpr.default_contract(torch.bfloat16, 128, operand_policy=cpr.CPR_POLICY_TC_BF16X3, dv_splits=2)
    dt = (ctypes.c_uint8 * 32).from_buffer_copy(cpr.contract_digest(t))
    p = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(8)]
    for which in (0, 1):                                    # dq, then dk
        grads = [ctypes.c_void_p(0x200000 * (i + 1)) for i in range(6)]
        grads[which] = ctypes.c_void_p(grads[which].value + 16)
        rc = lib.cpr_gdn_bwd_saved(ctypes.byref(t), dt, *p[:6], 1, 64, 1, None, p[6], None, *grads, p[7],
                                   1 << 40, None)
        assert rc == 3 and "32-byte" in lib.cpr_last_error().decode()
    x, w = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000)
    assert lib.cpr_gemm_bf16(x, w, ctypes.c_void_p(0x30010), 8, 128, 64, 64, None) == 3
    assert "32-byte" in lib.cpr_last_error().decode()


def test_reading_b_is_its_own_contract(lib):
    """intra_order TOKENREC_V1 (reading B): accepted on the tensor-core policy only, a digest
    of its own, a decode cache with the running in-chunk state appended, the training
    forward's workspace, and no training ops (refused on the host)."""
    a = cpr.default_contract(torch.bfloat16, 128, operand_policy=cpr.CPR_POLICY_TC_BF16X3, dv_splits=2)
    b = cpr.Contract.from_buffer_copy(a)
    b.intra_order = cpr.CPR_ORDER_TOKENREC_V1
    assert lib.cpr_contract_check(ctypes.byref(b)) == 0
    assert cpr.contract_digest(a) != cpr.contract_digest(b)
    s = cpr.simt_contract(torch.bfloat16, 128)
    s.intra_order = cpr.CPR_ORDER_TOKENREC_V1
    assert lib.cpr_contract_check(ctypes.byref(s)) == 2
    x = cpr.Contract.from_buffer_copy(a)
    x.intra_order = 3
    assert lib.cpr_contract_check(ctypes.byref(x)) == 2
    n_seq, H, d = 3, 4, 128
    la, lb = cpr.cache_layout(a, n_seq, H), cpr.cache_layout(b, n_seq, H)
    assert la.run == 0
    assert lb.run >= la.total_bytes and lb.run % 256 == 0
    assert lb.total_bytes >= lb.run + n_seq * H * d * d * 4
    for f in ("header", "pos", "state", "k_rows", "t_rows", "state_tiles", "delta_tiles"):
        assert getattr(la, f) == getattr(lb, f), f
    assert cpr.workspace_bytes(b, cpr.CPR_OP_FWD, n_seq, 4096, H) == cpr.workspace_bytes(a, cpr.CPR_OP_BWD, n_seq, 4096, H)
    db = (ctypes.c_uint8 * 32).from_buffer_copy(cpr.contract_digest(b))
    p = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(8)]
    grads = [ctypes.c_void_p(0x200000 * (i + 1)) for i in range(6)]
    rc = lib.cpr_gdn_fwd_train(ctypes.byref(b), db, *p[:6], 1, 64, 1, None, p[6], None, p[7], 1 << 40, None)
    assert rc == 2 and "TOKENREC" in lib.cpr_last_error().decode()
    rc = lib.cpr_gdn_bwd_saved(ctypes.byref(b), db, *p[:6], 1, 64, 1, None, p[6], None, *grads, p[7], 1 << 40, None)
    assert rc == 2 and "TOKENREC" in lib.cpr_last_error().decode()
    rc = lib.cpr_gdn_bwd(ctypes.byref(b), db, *p[:6], 1, 64, 1, None, p[6], None, *grads, p[7], 1 << 40, None)
    assert rc == 2


def test_deployment_digest_needs_a_device(lib):
    """Without a usable CUDA device the deployment identity cannot be formed: CPR_ERR_CUDA
    and a message, never a made-up digest.  (With a GPU it is checked in the GPU tests.)"""
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    out = (ctypes.c_uint8 * 32)()
    assert lib.cpr_deployment_digest(out, None, 0) == 6
    assert "device" in lib.cpr_last_error().decode()
    assert lib.cpr_deployment_digest(None, None, 0) == 1


def test_nocommit_step_checks_arguments_on_the_host(lib):
    """cpr_gdn_decode_step_nocommit refuses a missing cache or a wrong digest before any
    device work, under reading A (where it is the ordinary step) and reading B."""
    a = cpr.default_contract(torch.bfloat16, 128, operand_policy=cpr.CPR_POLICY_TC_BF16X3, dv_splits=2)
    b = cpr.Contract.from_buffer_copy(a)
    b.intra_order = cpr.CPR_ORDER_TOKENREC_V1
    p = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(8)]
    bad = (ctypes.c_uint8 * 32).from_buffer_copy(bytes(32))
    for c in (a, b):
        dig = (ctypes.c_uint8 * 32).from_buffer_copy(cpr.contract_digest(c))
        assert lib.cpr_gdn_decode_step_nocommit(ctypes.byref(c), dig, *p[:5], 1, 1, None, p[6], None) == 1
        assert lib.cpr_gdn_decode_step_nocommit(ctypes.byref(c), bad, *p[:5], 1, 1, p[5], p[6], None) == 4
