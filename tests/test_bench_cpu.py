"""The bench's bookkeeping on CPU: the work and byte counts its roofline
divides by (the figures the method's definition fixes: 2 flops per
multiply-add, x read once), the traffic lookup that must not report counters
taken on other kernel source, and the reference arm's JSON line."""
import io
import json
import contextlib

import bench
import synth

W = synth.WORKLOADS


def test_flops_are_two_per_multiply_add():
    # 2 * N * Cout * Ho * Wo * Cin * 9
    assert bench.conv_flops(W["c2_min_tanh2"]) == 2 * 128 * 64 * 254 * 254 * 16 * 9
    assert abs(bench.conv_flops(W["c2_min_tanh2"]) / 1e9 - 152.2) < 0.1
    assert abs(bench.conv_flops(W["c3_mul_lrelu_gelu"]) / 1e9 - 304.4) < 0.1
    assert abs(bench.conv_flops(W["c4_scale_min"]) / 1e9 - 608.8) < 0.1
    assert abs(bench.conv_flops(W["c5_gn_pool_clamp"]) / 1e9 - 18.7) < 0.1


def test_algorithmic_bytes():
    c2 = W["c2_min_tanh2"]
    x = 128 * 16 * 256 * 256 * 4
    out = 128 * 254 * 254 * 4
    assert bench.algorithmic_bytes(c2) == x + (64 * 16 * 9 + 64) * 4 + out
    c5 = W["c5_gn_pool_clamp"]  # pooled output 31 x 31 per channel, three parameter vectors
    assert bench.algorithmic_bytes(c5) == 4 * (128 * 8 * 128 * 128 + 64 * 8 * 9 + 64 * 4 + 128 * 64 * 31 * 31)


def test_traffic_only_for_the_profiled_source():
    h = bench.kernel_hash()
    t = json.load(open(bench.os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for wl in ("c2_min_tanh2", "c3_mul_lrelu_gelu", "c4_scale_min", "c5_gn_pool_clamp"):
        want = t[wl]["dram_bytes_per_launch"] if t[wl]["src_sha1"] == h else None
        assert bench.traffic_for(h, wl) == want
        assert bench.traffic_for("0" * 40, wl) is None       # another kernel source
    assert bench.traffic_for(h, "no_such_workload") is None


def test_reference_arm_line():
    buf = io.StringIO()
    args = type("A", (), {"warmup": 0, "steps": 1, "ref_seconds": 0.0, "gpus": 1})()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(args, W["pr1_min_tanh2"], 1, 0) == 0
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_single_core_oracle_sample():
    """The cpu_baseline adds a one-image, one-thread oracle figure where an
    image's conv is short (the 32x32 case, C2, C5) and leaves it out where
    one image would take many seconds on one core (C3, C4)."""
    short = [n for n in W if bench.conv_flops(W[n].with_batch(1)) <= bench.SINGLE_CORE_MAX_FLOPS]
    assert sorted(short) == ["c2_min_tanh2", "c5_gn_pool_clamp", "pr1_min_tanh2"]
    v, el, done, cores = bench.oracle_sample(W["pr1_min_tanh2"], 0.0, 1, cores=1)
    assert cores == 1 and done == 1 and v > 0 and el > 0


def test_roofline_fractions_and_bound():
    """Both fractions of one forward, and the bound is the roofline with the
    longer ideal time at the given peaks."""
    c3, c4 = W["c3_mul_lrelu_gelu"], W["c4_scale_min"]
    r = bench.roofline_of(c4, 1.0, 1000.0, 8000.0)          # 1 ms
    assert abs(r["tflops"] - bench.conv_flops(c4) / 1e9) < 1e-9
    assert abs(r["tensor_frac"] - r["tflops"] / 1000.0) < 1e-12
    assert abs(r["hbm_gbs"] - bench.algorithmic_bytes(c4) / 1e6) < 1e-9
    assert r["bound"] == "tensor"                            # 558 flop/B, far above the ridge
    # C3 does 143 flop per algorithmic byte: above a ridge of 1000/8 = 125, below 2000/8 = 250
    assert bench.roofline_of(c3, 1.0, 1000.0, 8000.0)["bound"] == "tensor"
    assert bench.roofline_of(c3, 1.0, 2000.0, 8000.0)["bound"] == "hbm"


def test_headline_is_the_largest_workload():
    """With no flags the bench times the workload with the most work."""
    src = open(bench.__file__).read()
    assert '"--workload", default="c4_scale_min"' in src
    assert max(W, key=lambda n: bench.conv_flops(W[n])) == "c4_scale_min"


def test_fp32_mode_roofline_is_the_fma_rate():
    """--mode fp32 is measured against the CUDA cores' FMA rate (bound "alu"),
    from the sampled maximum clock or the GB300's 2070 MHz, with no DRAM
    traffic figure (the capture is of the tensor-core kernel)."""
    r = bench.fp32_roofline(40.25, 152, 2070.0)
    assert r["bound"] == "alu" and r["traffic"] is None
    assert abs(r["peak"] - 152 * 128 * 2 * 2.07e-3) < 1e-9
    assert abs(r["frac"] - 40.25 / r["peak"]) < 1e-12
    assert bench.fp32_roofline(40.25, 152, None)["peak"] == r["peak"]
