"""CPU checks of bench.py's bookkeeping: the algorithmic bytes and FLOPs behind
the roofline object, the key of the committed ncu traffic table and its
source-hash guard, and the peak fallback.  No GPU."""
import hashlib
import os

import moe_inputs as mi

import bench


def test_mixtral_gemm1_bytes_and_flops():
    # 8 experts x W1 (2F x H bf16) + the permuted rows in + h out
    s = mi.MIXTRAL
    b = bench.gemm1_algorithmic_bytes(s, 8)
    assert b == 8 * 2 * 14336 * 4096 * 2 + 8192 * 4096 * 2 + 8192 * 14336 * 2
    assert b == 2181038080  # the figure the bench printed on the GPU for this workload
    assert s.flops() == 6.0 * 8192 * 4096 * 14336


def test_lowprec_gemm1_bytes_count_codes_and_scales():
    s = mi.LOWPREC
    per_expert = 2 * s.F * s.H / 2 + 2 * s.F * s.H / 16  # E2M1 codes + one E4M3 per 16
    rows = s.R * s.H * 2 + s.R * s.F * 2                   # f16 rows in, f16 h out
    assert bench.gemm1_algorithmic_bytes(s, 256) == 256 * per_expert + rows
    # MXFP4: one E8M0 per 32 values
    assert bench.gemm1_algorithmic_bytes(s, 256, 32) == \
        256 * (2 * s.F * s.H / 2 + 2 * s.F * s.H / 32) + rows


def test_decode_mlp_bytes_are_both_weights_rows_in_and_tokens_out():
    s = mi.DECODE.with_T(8)
    b = bench.decode_mlp_algorithmic_bytes(s, 54)
    assert b == 54 * 3 * 768 * 2048 * 2 + 64 * 2048 * 2 + 8 * 2048 * 2
    assert b == 509902848  # printed by the bench for T=8 (54 experts with tokens)


def test_traffic_key_names_the_workload_and_token_override():
    key = lambda argv: bench.traffic_key(bench.parse_args(argv))  # noqa: E731
    assert key([]) == "skewed"
    assert key(["--workload", "mixtral"]) == "mixtral"
    assert key(["--workload", "decode"]) == "decode"
    assert key(["--workload", "decode", "--T", "8"]) == "decode-T8"
    assert key(["--workload", "lowprec", "--E", "32"]) == "custom"
    assert key(["--workload", "skewed", "--k", "4"]) == "custom"


def test_traffic_table_is_used_only_for_the_captured_source():
    table = os.path.join(bench.ROOT, "profiles", "roofline_traffic.txt")
    rows = [l.split() for l in open(table) if l.strip() and not l.startswith("#")]
    csrc = os.path.join(bench.ROOT, "mixture_experts_ffn_permute_gb300", "csrc")
    files = {"grouped_mlp_decode_kernel": "grouped_mlp_decode.cu",
             "grouped_gemm_swap2_kernel": "grouped_gemm_swap2.cu",
             "grouped_gemm_swap_kernel": "grouped_gemm_swap.cu",
             "grouped_gemm_fp4_kernel": "grouped_gemm_fp4.cu",
             "grouped_gemm_bwd_kernel": "grouped_gemm_bwd.cu"}
    for sha, workload, kernel, rd, wr in rows:
        src = files[kernel]
        cur = hashlib.sha256(open(os.path.join(csrc, src), "rb").read()).hexdigest()[:16]
        got = bench.ncu_traffic(src, workload)
        if sha == cur:
            assert got == float(rd) + float(wr)
    # a workload without a row has no traffic figure
    assert bench.ncu_traffic("grouped_mlp_decode.cu", "decode-T3") is None
    assert bench.ncu_traffic("no_such_file.cu", "mixtral") is None


def test_peaks_fall_back_without_the_measured_file(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks == bench.FALLBACK_PEAKS


def test_default_workload_is_the_largest_single_gpu_config():
    a = bench.parse_args([])
    shape, _ = bench.WORKLOADS[a.workload]
    assert (shape.T, shape.H, shape.F, shape.E, shape.k) == (8192, 7168, 2048, 256, 8)


def test_layer_bytes_are_active_weights_x_logits_and_out():
    s = mi.SKEWED
    b = bench.layer_algorithmic_bytes(s, 196)
    assert b == 196 * 3 * 2048 * 7168 * 2 + 8192 * 7168 * 2 + 8192 * 256 * 4 + 8192 * 7168 * 2
    lp = mi.LOWPREC
    per = 3 * lp.F * lp.H / 2 + 3 * lp.F * lp.H / 16 + 8
    xin = lp.T * lp.H + lp.T * (lp.H // 128) * 4
    assert bench.layer_algorithmic_bytes(lp, 256) == 256 * per + xin + lp.T * 256 * 4 + \
        lp.T * lp.H * 2


def test_tensor_peak_is_burst_for_short_regions_and_sustained_for_long():
    peaks = {"hbm_gbs": 6775.6, "bf16_tflops": 1916.9, "bf16_tflops_sustained": 1719.2}
    assert bench.tensor_peak(peaks, 1.1)[:2] == (1916.9, "bf16_tflops")
    assert bench.tensor_peak(peaks, bench.SUSTAINED_AFTER_S)[:2] == \
        (1719.2, "bf16_tflops_sustained")


def test_fp8_layer_takes_the_fp8_tensor_peak():
    peaks = {"hbm_gbs": 6775.6, "bf16_tflops": 1916.9, "bf16_tflops_sustained": 1719.2}
    v, key, other = bench.tensor_peak(peaks, 1.0, fp8=True)
    assert v == 2 * 1916.9 and bench.peak_of(peaks, other) == 2 * 1719.2


def test_clock_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler(0)
    c.lines = ["1695, 2070, 702.3, Active, Not Active, Not Active, Not Active, 720.00",
               "1710, 2070, 698.1, Not Active, Not Active, Not Active, Not Active, 720.00",
               "1680, 2070, [N/A], Active, Not Active, Not Active, Not Active, 720.00",
               "garbage"]
    s = c.summary()
    assert s["sm_mhz"] == 1695.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w"] == 700.2 and s["power_limit_w"] == 720.0
    assert bench.ClockSampler(0).summary()["samples"] == 0
