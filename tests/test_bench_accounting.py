"""bench.py's roofline bookkeeping (no GPU): the algorithmic bytes charged to each
tensor-core kernel add up to the path's algorithmic bytes, and the forward kernels' MMA
FLOPs to the forward's, so no kernel's roofline counts work twice or drops any."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


@pytest.mark.parametrize("lens", [[4096] * 4, [4096] * 8, [130, 64, 1, 8191]])
def test_kernel_byte_shares_add_up_to_the_path(lens):
    H, d = 16, 128
    ht = sum(lens) * H
    states = len(lens) * H * d * d * 4
    fwd = ht * bench.algo_fwd_bytes_per_head_token(d) + states
    bwd = ht * bench.algo_bwd_bytes_per_head_token(d) + states
    kb = lambda n: bench.tc_kernel_bytes(n, lens, H, d)
    assert kb("cpr_tc_prep") + kb("cpr_tc_state") == fwd
    assert kb("cpr_tc_state_bwd") + kb("cpr_tc_grad") == bwd


def test_forward_kernel_flops_add_up_to_the_forward():
    d = 128
    f = bench.tc_kernel_flops_per_chunk
    assert f("cpr_tc_prep", d) + f("cpr_tc_state", d) == bench.algo_fwd_flops_per_chunk(d)
    # the backward kernels' contraction list is the smaller count the roofline uses
    assert f("cpr_tc_state_bwd", d) + f("cpr_tc_grad", d) <= bench.algo_bwd_flops_per_chunk(d)


def test_prefill_kernels_are_hbm_bound_by_the_rule():
    """Prep's share: 4 C^2 d MACs per chunk against 776 bytes per head-token -> below the
    ridge of the measured peaks, so its roofline is the copy bandwidth."""
    pk = {"bf16_tflops": 1941.2, "hbm_gbs": 6777.6}
    lens, H, d = [4096] * 4, 16, 128
    units = bench.chunk_count(lens) * H
    t_f = bench.tc_kernel_flops_per_chunk("cpr_tc_prep", d) * units / (pk["bf16_tflops"] * 1e12)
    t_b = bench.tc_kernel_bytes("cpr_tc_prep", lens, H, d) / (pk["hbm_gbs"] * 1e9)
    assert t_b > 3 * t_f
