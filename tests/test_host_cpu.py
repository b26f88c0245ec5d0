"""Host logic of the product path checked against the oracle on CPU: the
library's sigma schedule (host code behind the C ABI, no GPU needed), and the
benchmark's FLOP accounting against the per-block formula 24 L D^2 + 4 L^2 D."""
import json
import numpy as np
import pytest

from diffusion_transformer_image_mmdit_gb300 import schedule
from oracle import mmdit_oracle as O


@pytest.fixture(scope="module")
def built():
    from diffusion_transformer_image_mmdit_gb300 import build
    build.build()


def test_schedule_matches_oracle(built):
    for n, tokens in ((50, 6889), (28, 4096), (4, 1024)):
        got = np.array(schedule.sigmas(n, schedule.mu_for_tokens(tokens)))
        ref = O.sigma_schedule(n, O.shift_mu(tokens))
        assert np.abs(got - ref).max() < 1e-15
    assert schedule.sigmas(4, 0.0) == [1.0, 0.75, 0.5, 0.25, 0.0]
    from diffusion_transformer_image_mmdit_gb300 import _lib
    with pytest.raises(_lib.MMDiTError):
        schedule.sigmas(0, 0.0)


def test_bench_flop_accounting():
    import bench
    c4 = bench.step_flops(bench.CONFIGS["c4"])
    L, D = 7401, 3072
    per_block = 24 * L * D * D + 4 * L * L * D
    assert c4["block_flops"] == per_block
    assert abs(c4["total"] - 57 * per_block) / c4["total"] < 2e-3  # + img_in, final, modulation, timestep
    assert abs(57 * per_block / 1e12 - 133.9) < 0.05
    c5 = bench.step_flops(bench.CONFIGS["c5"])
    assert abs(c5["total"] / 1e12 - 297.4) / 297.4 < 3e-3


def test_bench_e4m3_accounting():
    """The e4m3 configs count the same FLOPs as their bf16 twins; all block-linear FLOPs (not the embedder and
    final-layer GEMMs) are e4m3; the weights read per step shrink by the block linears' half."""
    import bench
    for f8, bf in (("c4_f8", "c4"), ("klein1024_f8", "klein1024")):
        a, b = bench.step_flops(bench.CONFIGS[f8]), bench.step_flops(bench.CONFIGS[bf])
        assert a["total"] == b["total"] and a["gemm"] == b["gemm"] and b["gemm_f8"] == 0
        c = bench.CONFIGS[f8]
        io = 2 * c["grid_h"] * c["grid_w"] * c["C_lat"] * c["D"] * 2 * c["B"]
        assert a["gemm"] - a["gemm_f8"] == io
        wa, wb = bench.step_weight_bytes(bench.CONFIGS[f8]), bench.step_weight_bytes(bench.CONFIGS[bf])
        assert 0.5 * wb < wa < 0.7 * wb


def test_clock_sampler_summary():
    """The bench's clock record from nvidia-smi CSV rows: median SM clock under load, the maximum clock,
    and every throttle reason seen active at any sample (the rules that reject or annotate a run)."""
    import bench
    cs = bench.ClockSampler(0)
    assert cs.summary()["reasons"] == ["unsampled"]
    line = "0, {sm}, 2070, {pw}, 0x{act}, {hw}, Not Active, Not Active, {cap}"
    cs.rows = [[x.strip() for x in line.format(sm=sm, pw=pw, act=a, hw=hw, cap=cap).split(",")]
               for sm, pw, a, hw, cap in ((1965, 1100.5, "4", "Not Active", "Active"),
                                          (1980, 1371.0, "4", "Not Active", "Active"),
                                          (1890, 900.25, "0", "Not Active", "Not Active"))]
    s = cs.summary()
    assert s["sm_mhz"] == 1965 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 1371.0
    cs.rows.append([x.strip() for x in line.format(sm=1200, pw=800, act="8", hw="Active", cap="Not Active").split(",")])
    assert bench.ClockSampler.summary(cs)["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_bench_configs_are_named_and_reference_arm_declines_gpu_only_ones(capsys):
    """Every bench workload has its name for the JSON line, and the reference arm (the oracle on the host)
    prints an 'unavailable' line for the workloads it does not time instead of running anything."""
    import sys
    import bench
    assert set(bench.WORKLOAD_NAME) == set(bench.CONFIGS)
    for name in ("sample1024", "ulysses_layout"):
        argv = sys.argv
        sys.argv = ["bench.py", "--impl", "reference", "--config", name]
        try:
            bench.main()
        finally:
            sys.argv = argv
        line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
        assert line["impl"] == "reference" and line["unavailable"]


def test_bench_gemm_hash_ignores_comments_only():
    """The hash that ties a committed ncu capture to the GEMM sources covers the code, not its comments:
    an edit of a comment keeps it, an edit of code (or of a string literal, which may be PTX) changes it."""
    import bench
    src = 'int a = 1; // note\n/* block\n comment */\nasm("x // y");\n\nint b = 2;\n'
    ref = bench._code_only(src)
    assert ref == 'int a = 1;\nasm("x // y");\nint b = 2;'
    assert bench._code_only(src.replace("// note", "// another note")) == ref
    assert bench._code_only(src.replace("block", "longer block")) == ref
    assert bench._code_only(src.replace("int b = 2", "int b = 3")) != ref
    assert bench._code_only(src.replace('"x // y"', '"x // z"')) != ref


def test_bench_gemm_bytes_and_traffic_source():
    """Algorithmic GEMM bytes count each problem's weights once (the two streams of a double block have
    their own), and the bench's per-launch DRAM traffic comes from the capture at the workload's own token
    count when one exists (no scaling), from the 512 + 64x64 capture scaled by token rows otherwise, and is
    absent for shapes or precisions no committed capture covers."""
    import bench
    c = dict(bench.CONFIGS["c4pair"])
    B, D, Dm, C = c["B"], c["D"], c["D_mlp"], c["C_lat"]
    L, Li = c["L_txt"] + c["grid_h"] * c["grid_w"], c["grid_h"] * c["grid_w"]
    M = B * L
    w_double = 2 * (3 * D * D + D * D + Dm * D + D * Dm) * 2  # both streams' weights, bf16
    w_single = ((3 * D + Dm) * D + D * (D + Dm)) * 2
    w_io = (D * C + C * D) * 2
    acts = ((M * D + M * 3 * D + M * D + M * D * 4 + M * D + M * Dm + M * Dm + M * D * 4)  # double: A, outputs, resid
            + (M * D + M * (3 * D + Dm) + M * (D + Dm) + M * D * 4)) * 2                    # single
    io_acts = (B * Li * C * 2 + B * Li * D * 4) + (B * Li * D * 2 + B * Li * C * 4)
    total = w_double + w_single + w_io + acts + io_acts
    assert abs(bench.gemm_algorithmic_bytes(c) * 8 - total) / total < 1e-12
    t, src = bench.gemm_traffic_scaled(bench.CONFIGS["c4"])
    if t is not None:  # the committed captures match the current GEMM sources
        assert "at this token count (7401 tokens)" in src
        rows = bench.gemm_launch_table("c4pair")
        dbl = sum((r[4] + r[5]) * 1e6 for r in rows if r[0] in ("qkv", "proj", "mlp_in", "mlp_out"))
        sng = sum((r[4] + r[5]) * 1e6 for r in rows if r[0] in ("lin1", "lin2"))
        io = sum((r[4] + r[5]) * 1e6 for r in rows if r[0] in ("img_in", "final"))
        assert abs(t - (19 * dbl + 38 * sng + io) / 154) < 1.0
        t5, src5 = bench.gemm_traffic_scaled(bench.CONFIGS["c5"])
        assert t5 is not None and "scaled by the token rows" in src5
    for name in ("klein1024", "klein_i2i", "c4_f8"):
        t, src = bench.gemm_traffic_scaled(bench.CONFIGS[name])
        assert t is None and src
