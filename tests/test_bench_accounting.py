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


def test_reference_arm_prints_its_line():
    """`bench.py --impl reference` times the oracle on the host (no GPU) and prints one
    JSON line with the keys the launch contract names."""
    import json
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([x for x in r.stdout.splitlines() if x.startswith("{")][-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0


def test_step_bytes_follow_the_methods_per_head_token_figures():
    """The roofline's byte rule: 1,032 B per head-token forward (bf16 o) plus the final
    states; the trainer adds 1,808 B per head-token backward plus dh0.  With fp32 outputs
    (what the kernels write) 1,288 and 2,832."""
    class S:
        d, H = 128, 16
    p = S()
    p.lens, p.op = [4096] * 4, "fwd"
    assert bench.step_bytes(p, 2) == 262144 * 1032 + 4 * 16 * 128 * 128 * 4 == 274_726_912
    assert bench.step_bytes(p, 4) == 262144 * 1288 + 4 * 16 * 128 * 128 * 4
    t = S()
    t.lens, t.op = [4096] * 8, "fwdbwd"
    assert bench.step_bytes(t, 2) == 524288 * (1032 + 1808) + 2 * 8 * 16 * 128 * 128 * 4
    assert bench.step_bytes(t, 4) == 524288 * (1288 + 2832) + 2 * 8 * 16 * 128 * 128 * 4


class _DecodeStep:
    """The parts of bench's decode step that roofline_for reads."""
    name, d, H, op = "decode", 128, 32, "decode"
    lens = [2048] * 64

    def kernel_units(self, name):
        return len(self.lens) * self.H


def test_stored_traffic_only_for_the_full_workload(monkeypatch):
    """profiles/traffic.json holds ncu DRAM bytes of a full-workload launch: the bench line
    carries them only while the kernel's sources still hash to the stored key and the run
    covers the whole workload (not --n-seq)."""
    pk = {"bf16_tflops": 1941.2, "hbm_gbs": 6777.6, "sm_max_mhz": 2070}
    prof = {"cpr_tc_decode": (512, 512 * 0.09)}
    key = bench.kernel_src_sha("cpr_tc_decode")
    monkeypatch.setattr(bench, "load_traffic", lambda: {
        "cpr_tc_decode/decode": {"bytes_per_launch": 123456789, "kernel_src_sha": key}})
    monkeypatch.setattr(bench, "N_SEQ_OVERRIDE", None)
    r = bench.roofline_for(_DecodeStep(), prof, pk)
    assert r["traffic"] == 123456789 and r["traffic_gbs"] == round(123456789 / 90e-6 / 1e9, 1)
    monkeypatch.setattr(bench, "N_SEQ_OVERRIDE", 16)
    assert bench.roofline_for(_DecodeStep(), prof, pk)["traffic"] is None
    monkeypatch.setattr(bench, "N_SEQ_OVERRIDE", None)
    monkeypatch.setattr(bench, "load_traffic", lambda: {
        "cpr_tc_decode/decode": {"bytes_per_launch": 123456789, "kernel_src_sha": "0" * 16}})
    assert bench.roofline_for(_DecodeStep(), prof, pk)["traffic"] is None
