"""Kernel-level parity of the CUDA path against the float64 oracle, called
through the C ABI: RoPE tables (bit-exact), RoPE rotation, Euler, the int8
quantiser (bit-exact), LN+modulate, the GEMV, the tcgen05 GEMM with every
epilogue, and joint attention."""
import math

import numpy as np
import pytest
import torch

from diffusion_transformer_image_mmdit_gb300 import _lib, api, synthetic as S
from diffusion_transformer_image_mmdit_gb300.api import LinearDev
from oracle import mmdit_oracle as O
from tests.gpu_common import (CONFIGS, FULL, api_shape, assert_close, bf16, check_status, f32, gpu_tables, host,
                              need_gpu, rel_l2, tables)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    need_gpu()
    yield
    check_status()


# ------------------------------------------------------------------ RoPE
# image-to-image: 1200x800 target (75x50 latent grid) plus a reference latent of the same size
I2I_1200 = dict(B=1, L_txt=512, grid_h=75, grid_w=50, ref_h=75, ref_w=50, D=4096, H=32, d_head=128, D_mlp=12288,
                rope_axes=(16, 56, 56))


@pytest.mark.parametrize("cfg", [CONFIGS["c1"], CONFIGS["d128"], CONFIGS["tail"], FULL["c3"], FULL["c4"],
                                 dict(CONFIGS["d128"], ref_h=3, ref_w=7), I2I_1200])
def test_rope_tables_bit_exact(cfg):
    shape = api_shape(cfg)
    ids, cs, sn = gpu_tables(shape)
    torch.cuda.synchronize()
    ref_ids = O.rope_ids(cfg["L_txt"], cfg["grid_h"], cfg["grid_w"], cfg.get("ref_h", 0), cfg.get("ref_w", 0))
    c, s = tables(cfg)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    gc, gs = cs.cpu().numpy(), sn.cpu().numpy()
    mis_c = int((gc.view(np.uint32) != c.astype(np.float32).view(np.uint32)).sum())
    mis_s = int((gs.view(np.uint32) != s.astype(np.float32).view(np.uint32)).sum())
    assert mis_c == 0 and mis_s == 0, f"fp32 table entries differing: cos {mis_c}, sin {mis_s} of {gc.size}"


@pytest.mark.parametrize("cfg", [CONFIGS["c1"], CONFIGS["d128"]])
def test_rope_apply(cfg):
    shape = api_shape(cfg)
    _, cs, sn = gpu_tables(shape)
    B, L, H, d = cfg["B"], api.seq_len(shape), cfg["H"], cfg["d_head"]
    x = S.normal_bf16("ra.x", (B, L, H, d))
    row_stride = H * d + 64  # a padded row
    xp = np.zeros((B, L, row_stride))
    xp[..., :H * d] = x.reshape(B, L, H * d)
    xt = bf16(xp)
    api.rope2d_apply(shape, cs, sn, xt, row_stride)
    c, s = tables(cfg)
    ref = O.rope_apply(x, c, s).reshape(B, L, H * d)
    got = host(xt)
    assert_close(got[..., :H * d], ref, what="rope2d_apply")
    assert np.array_equal(got[..., H * d:], xp[..., H * d:]), "padding touched"


# ------------------------------------------------------------------ Euler
@pytest.mark.parametrize("n", [1, 7, 4096 + 3])
@pytest.mark.parametrize("vdt", [torch.float32, torch.bfloat16])
def test_euler(n, vdt):
    x = S.normal_f32("eu.x", (n,))
    v = S.normal_f32("eu.v", (n,)) if vdt == torch.float32 else S.normal_bf16("eu.v", (n,))
    xt, vt = f32(x), f32(v).to(vdt)
    sig = O.sigma_schedule(50, O.shift_mu(6889))
    api.euler_step(xt, vt, sig[0], sig[1])
    ref = O.euler_step(x, v, sig[0], sig[1])
    assert np.abs(host(xt) - ref).max() <= 1e-6 * (1 + np.abs(ref).max())


# ------------------------------------------------------------------ int8 quantiser
@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_quantize_bit_exact(dt):
    w = S.normal_bf16("qz.w", (70, 320), 0.02) if dt == torch.bfloat16 else S.normal_f32("qz.w", (70, 320), 0.02)
    w[3] = 0.0
    w[4, :6] = [127.0, 63.5, -0.5, 2.5, -2.5, 1.5]
    w[4, 6:] = 0.0
    wt = f32(w).to(dt)
    q = torch.empty((70, 320), dtype=torch.int8, device="cuda")
    s = torch.empty((70,), dtype=torch.float32, device="cuda")
    api.mmdit_quantize_w8(wt, q, s)
    rq, rs = O.quantize_w8(host(wt))
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


# ------------------------------------------------------------------ LN + modulate, GEMV
@pytest.mark.parametrize("D", [256, 3072])
def test_ln_modulate(D):
    B, rows = 2, 37
    x = S.normal_f32("ln.x", (B, rows, D)) * 2 + 0.5
    mod = S.normal_f32("ln.m", (B, 3 * D)) * 0.3
    xt, mt = f32(x), f32(mod)
    y = torch.empty((B, rows, D), dtype=torch.bfloat16, device="cuda")
    # shift at column 0, scale at column D of each sample's 3D-wide modulation row
    api.mmdit_ln_modulate(xt, mt[:, :D], mt[:, D:2 * D], 3 * D, 1e-6, y)
    ref = O.modulate(O.layer_norm(x, 1e-6), mod[:, None, :D], mod[:, None, D:2 * D])
    assert_close(host(y), ref, what="ln_modulate")


@pytest.mark.parametrize("D", [256, 3072])
def test_ln_modulate_f8_fused(D):
    """LN + modulate with its e4m3 rows written in the same pass (the activation
    path of the e4m3 blocks): the bf16 rows equal mmdit_ln_modulate's, and the
    codes and scales equal the oracle's row quantiser on those bf16 rows, bit
    for bit, with or without the bf16 rows stored."""
    B, rows = 2, 37
    x = S.normal_f32("lnq.x", (B, rows, D)) * 2 + 0.5
    mod = S.normal_f32("lnq.m", (B, 3 * D)) * 0.3
    x[1, 5] = 0.25  # a constant row: LN output 0, the row is the shift alone
    xt, mt = f32(x), f32(mod)
    sh, sc = mt[:, :D], mt[:, D:2 * D]
    y = torch.empty((B, rows, D), dtype=torch.bfloat16, device="cuda")
    api.mmdit_ln_modulate(xt, sh, sc, 3 * D, 1e-6, y)
    y1 = torch.empty_like(y)
    q1, s1 = api.mmdit_ln_modulate_f8(xt, sh, sc, 3 * D, 1e-6, y1)
    q0, s0 = api.mmdit_ln_modulate_f8(xt, sh, sc, 3 * D, 1e-6)
    check_status()
    assert torch.equal(y1, y)
    yb = host(y).reshape(B * rows, D)
    rq, rs = O.quantize_f8_rows(yb)
    for q, s in ((q1, s1), (q0, s0)):
        assert np.array_equal(host(s).reshape(-1).astype(np.float32), rs)
        assert np.array_equal(decode_e4m3(q.reshape(B * rows, D).cpu().numpy()), rq)


@pytest.mark.parametrize("i8", [False, True])
@pytest.mark.parametrize("act", [0, 1])
@pytest.mark.parametrize("B", [3, 12])
def test_gemv(i8, act, B):
    """B = 12 runs as two launches of 8 and 4 rows."""
    N, K = 1000, 3072
    w, b = S.linear_params("gv", N, K)
    x = S.normal_f32(f"gv.x{B}", (B, K))
    lin = LinearDev(bf16(w), f32(b))
    wref = w
    if i8:
        lin = api.quantize_linear(lin)
        wref = O.dequantize_w8(lin.w.cpu().numpy(), lin.scale.cpu().numpy())
    y = torch.empty((B, N), dtype=torch.float32, device="cuda")
    api.mmdit_gemv(lin, f32(x), act, y)
    ref = O.linear(O.silu(x) if act else x, wref, b)
    assert_close(host(y), ref, rel=1e-4, what="gemv")


# ------------------------------------------------------------------ GEMM
GEMM_SHAPES = [(1, 256, 64), (100, 512, 320), (300, 768, 256), (257, 128, 1024), (129, 1056, 192)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
@pytest.mark.parametrize("epi", ["bf16", "gelu", "f32", "resid"])
def test_linear_epilogues(M, N, K, epi):
    w, b = S.linear_params(f"gm{M}.{N}.{K}", N, K)
    w = w * 10  # unit-scale outputs
    w = S.round_bf16(w)
    x = S.normal_bf16("gm.x", (M, K))
    lin = LinearDev(bf16(w), f32(b))
    ref = O.linear(x, w, b)
    if epi in ("bf16", "gelu"):
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        api.mmdit_linear_fwd(lin, bf16(x), y, api.MMDIT_EPI_BF16 if epi == "bf16" else api.MMDIT_EPI_BF16_GELU)
        if epi == "gelu":
            ref = O.gelu_tanh(ref)
        # bf16 output: one rounding of at most 2^-9 relative on top of fp32 accumulation
        assert_close(host(y), ref, max_abs=2.0 ** -8 * max(1.0, np.abs(ref).max()), what=f"gemm {epi}")
    elif epi == "f32":
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        api.mmdit_linear_fwd(lin, bf16(x), y, api.MMDIT_EPI_F32)
        assert_close(host(y), ref, rel=1e-4, max_abs=1e-2, what="gemm f32")
    else:
        r0 = S.normal_f32("gm.r", (M, N))
        gate = S.normal_f32("gm.g", (N,))
        y = f32(r0)
        api.mmdit_linear_fwd(lin, bf16(x), y, api.MMDIT_EPI_RESID, gate=f32(gate))
        assert_close(host(y), r0 + gate * ref, rel=1e-4, max_abs=1e-2, what="gemm resid")


@pytest.mark.parametrize("M,N,K", [(300, 768, 256), (1, 256, 64)])
def test_linear_int8(M, N, K):
    w, b = S.linear_params("g8", N, K)
    x = S.normal_bf16("g8.x", (M, K))
    lin8 = api.quantize_linear(LinearDev(bf16(w), f32(b)))
    ws = api.alloc_workspace(N * K * 2)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    api.mmdit_linear_fwd(lin8, bf16(x), y, api.MMDIT_EPI_F32, ws=ws)
    wq = O.dequantize_w8(lin8.w.cpu().numpy(), lin8.scale.cpu().numpy())
    assert_close(host(y), O.linear(x, wq, b), rel=1e-4, max_abs=1e-3, what="int8 gemm vs dequantised")
    assert rel_l2(host(y), O.linear(x, w, b)) <= 3e-2


@pytest.mark.parametrize("M,F,K,i8", [(300, 256, 256, False), (1, 128, 64, False), (260, 384, 192, True)])
def test_linear_swiglu(M, F, K, i8):
    """W rows [gate; up] (2F of them); y = SiLU(x Wg^T + bg) * (x Wu^T + bu), F wide."""
    w, b = S.linear_params(f"sw{M}.{F}.{K}", 2 * F, K)
    w = S.round_bf16(w * 10)
    x = S.normal_bf16("sw.x", (M, K))
    lin = LinearDev(bf16(w), f32(b))
    ws = None
    if i8:
        lin = api.quantize_linear(lin)
        ws = api.alloc_workspace(2 * F * K * 2)
        w = O.dequantize_w8(lin.w.cpu().numpy(), lin.scale.cpu().numpy())
    y = torch.empty((M, F), dtype=torch.bfloat16, device="cuda")
    api.mmdit_linear_fwd(lin, bf16(x), y, api.MMDIT_EPI_SWIGLU, ws=ws)
    ref = O.swiglu(O.linear(x, w, b))
    assert_close(host(y), ref, max_abs=2.0 ** -8 * max(1.0, np.abs(ref).max()) + 1e-3, what="gemm swiglu")


# ------------------------------------------------------------------ FP8 (e4m3)
def decode_e4m3(codes) -> np.ndarray:
    """e4m3 byte codes to values, from the bit layout (no NaN codes expected)."""
    c = np.asarray(codes, np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e, m = (c >> 3) & 15, c & 7
    assert not ((e == 15) & (m == 7)).any()
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    return sign * mag


def test_quantize_f8_bit_exact():
    x = S.normal_bf16("q8.x", (37, 384), 3.0)
    x[5] = 0.0
    x[7] *= 1e-3  # small rows reach the subnormal range after scaling
    x = S.round_bf16(x)  # what the kernel reads
    q, s = api.quantize_f8(bf16(x))
    rq, rs = O.quantize_f8_rows(x)
    assert np.array_equal(host(s).astype(np.float32), rs)
    assert np.array_equal(decode_e4m3(q.cpu().numpy()), rq)
    w = S.normal_f32("q8.w", (40, 256), 0.02)
    qw, sw = api.quantize_f8(f32(w))
    rqw, rsw = O.quantize_f8_rows(w)
    assert np.array_equal(host(sw).astype(np.float32), rsw)
    assert np.array_equal(decode_e4m3(qw.cpu().numpy()), rqw)


def _e4m3_midpoints():
    """Every point where e4m3 rounding changes below 448: the midpoints between
    adjacent e4m3 values, normal binades 2^-6 .. 2^8 and the subnormal range."""
    mids = [(2 * k + 1) * 2.0 ** -10 for k in range(8)]
    for e in range(-6, 9):
        mids += [2.0 ** e * (1 + (2 * j + 1) / 16) for j in range(8)]
    return np.array([m for m in mids if m < 448.0])


@pytest.mark.parametrize("sv,inputs", [(1.75, ("bf16", "f32")), (1.875, ("f32",))])
def test_quantize_f8_ties(sv, inputs):
    """Rows whose scale is s = sv (max |x| = 448 sv) and whose entries are sv * m
    for every e4m3 midpoint m: each quotient x / s is exactly a tie, which
    e4m3 rounds to even.  For these two scales, a quotient formed as
    x * RN(1/s) lands an ulp off the tie for 78 and 109 of the 126 midpoints,
    and would round 30 and 46 of them to the wrong side, so the test tells a
    correctly rounded quotient from a reciprocal multiply.  The kernels must
    give the oracle's codes bit for bit (bf16 rows through the row kernel, fp32
    rows through the general kernel), alongside random entries."""
    mids = _e4m3_midpoints()
    K = 384
    rows = []
    for r in range(4):
        row = S.normal_f32(f"q8t.{sv}.{r}", (K,), 20.0)
        row[0] = 448.0 * sv
        row[1:1 + len(mids)] = sv * mids * (1 if r % 2 == 0 else -1)
        rows.append(np.clip(row, -448.0 * sv, 448.0 * sv))
    x = np.stack(rows).astype(np.float32)
    if "bf16" in inputs:
        x = S.round_bf16(x)
        assert np.all(x[0, 1:1 + len(mids)] == sv * mids), "tie inputs must be bf16-exact"
    rq, rs = O.quantize_f8_rows(x)
    assert np.all(rs == np.float32(sv))
    for kind in inputs:
        q, s_ = api.quantize_f8(bf16(x) if kind == "bf16" else f32(x))
        assert np.array_equal(host(s_).astype(np.float32), rs)
        assert np.array_equal(decode_e4m3(q.cpu().numpy()), rq), f"e4m3 ties differ ({kind} rows, s = {sv})"


@pytest.mark.parametrize("M,N,K", [(300, 512, 256), (1, 256, 128), (270, 384, 384)])
@pytest.mark.parametrize("epi", ["f32", "bf16", "gelu", "swiglu", "resid"])
def test_linear_f8(M, N, K, epi):
    w, b = S.linear_params(f"l8.{M}.{N}.{K}", N, K)
    x = S.normal_bf16("l8.x", (M, K))
    lin8 = api.quantize_linear_f8(LinearDev(bf16(w), f32(b)))
    x8, xs = api.quantize_f8(bf16(x))
    xd = decode_e4m3(x8.cpu().numpy()) * host(xs)[:, None]
    wd = decode_e4m3(lin8.w.cpu().numpy()) * host(lin8.scale)[:, None]
    ref = O.linear(xd, wd, b)
    if epi == "f32":
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        api.mmdit_linear_f8_fwd(lin8, x8, xs, y, api.MMDIT_EPI_F32)
        assert_close(host(y), ref, rel=1e-4, max_abs=1e-4, what="fp8 gemm f32")
        # the scheme against the exact product of the unquantised operands: the
        # e4m3 step (2^-3 relative) leaves at most 2^-4 per operand, ~5% rms per dot product
        assert rel_l2(host(y), O.linear(x, w, b)) <= 1e-1
    elif epi == "resid":
        r0 = S.normal_f32("l8.r", (M, N))
        gate = S.normal_f32("l8.g", (N,))
        y = f32(r0)
        api.mmdit_linear_f8_fwd(lin8, x8, xs, y, api.MMDIT_EPI_RESID, gate=f32(gate))
        assert_close(host(y), r0 + gate * ref, rel=1e-4, max_abs=1e-4, what="fp8 gemm resid")
    else:
        n_out = N // 2 if epi == "swiglu" else N
        y = torch.empty((M, n_out), dtype=torch.bfloat16, device="cuda")
        code = {"bf16": api.MMDIT_EPI_BF16, "gelu": api.MMDIT_EPI_BF16_GELU, "swiglu": api.MMDIT_EPI_SWIGLU}[epi]
        if epi == "swiglu" and N % 256:
            # gate and up must come in whole 128-row halves of a 256-row tile
            with pytest.raises(_lib.MMDiTError) as e:
                api.mmdit_linear_f8_fwd(lin8, x8, xs, y, code)
            assert e.value.status == -2
            return
        api.mmdit_linear_f8_fwd(lin8, x8, xs, y, code)
        r = {"bf16": ref, "gelu": O.gelu_tanh(ref), "swiglu": O.swiglu(ref)}[epi]
        assert_close(host(y), r, max_abs=2.0 ** -8 * max(1.0, np.abs(r).max()) + 1e-4, what=f"fp8 gemm {epi}")


@pytest.mark.parametrize("K", [192, 320])
def test_gemm_many_tiles_k_tail(K):
    """Several tiles per CTA pair with a K that ends in a one-slice stage (K = 192: one full stage and
    a half; K = 320: two and a half), so the ring stages and their barrier phases wrap across tiles,
    and the stage releases reach both CTAs except in each pair's last ring round; M tail of 77 rows."""
    M, N = 256 * 30 + 77, 2048  # 31 pair-rows x 8 N tiles = 248 tiles over at most 76 CTA pairs
    w, b = S.linear_params(f"gtail{K}", N, K)
    x = S.normal_bf16(f"gtail{K}.x", (M, K))
    lin = LinearDev(bf16(w), f32(b))
    ref = O.linear(x, w, b)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    api.mmdit_linear_fwd(lin, bf16(x), y, api.MMDIT_EPI_F32)
    assert_close(host(y), ref, rel=1e-4, max_abs=1e-2, what=f"gemm K={K} f32")
    r0 = S.normal_f32(f"gtail{K}.r", (M, N))
    gate = S.normal_f32(f"gtail{K}.g", (N,))
    y = f32(r0)
    api.mmdit_linear_fwd(lin, bf16(x), y, api.MMDIT_EPI_RESID, gate=f32(gate))
    assert_close(host(y), r0 + gate * ref, rel=1e-4, max_abs=1e-2, what=f"gemm K={K} resid")


def test_linear_f8_many_tiles_k_tail():
    """e4m3 GEMM with several tiles per CTA pair and K = 384: one stage of 256 K elements and one of
    128 per tile, gated-residual epilogue, M tail of 33 rows."""
    M, N, K = 4096 + 33, 2048, 384
    w, b = S.linear_params("l8tail", N, K)
    x = S.normal_bf16("l8tail.x", (M, K))
    lin8 = api.quantize_linear_f8(LinearDev(bf16(w), f32(b)))
    x8, xs = api.quantize_f8(bf16(x))
    xd = decode_e4m3(x8.cpu().numpy()) * host(xs)[:, None]
    wd = decode_e4m3(lin8.w.cpu().numpy()) * host(lin8.scale)[:, None]
    ref = O.linear(xd, wd, b)
    r0 = S.normal_f32("l8tail.r", (M, N))
    gate = S.normal_f32("l8tail.g", (N,))
    y = f32(r0)
    api.mmdit_linear_f8_fwd(lin8, x8, xs, y, api.MMDIT_EPI_RESID, gate=f32(gate))
    assert_close(host(y), r0 + gate * ref, rel=1e-4, max_abs=1e-4, what="fp8 gemm many tiles resid")


def test_gemm_large_tiles_and_ragged():
    """Several waves of persistent tiles, M tail of 9 rows, K = 3072."""
    M, N, K = 128 * 20 + 9, 1024, 3072
    w, b = S.linear_params("gbig", N, K)
    x = S.normal_bf16("gbig.x", (M, K))
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    api.mmdit_linear_fwd(LinearDev(bf16(w), f32(b)), bf16(x), y, api.MMDIT_EPI_F32)
    assert_close(host(y), O.linear(x, w, b), rel=1e-4, max_abs=1e-2, what="gemm large")


# ------------------------------------------------------------------ attention
# The persistent attention runs one CTA per SM over units (pairs of 128-row
# query tiles x heads x samples).  With more units than SMs it runs whole
# rounds, then splits the remaining units' KV tiles evenly over the CTAs:
# units cut at a CTA boundary are computed in two parts and merged.  These
# cases (152 SMs) exercise that tail, all rows compared with the oracle.
SPLIT_CASES = {
    # 168 units of 13 KV tiles: no whole round; every CTA takes 14-15 KV steps
    "split13": dict(B=2, L_txt=64, grid_h=40, grid_w=40, D=1536, H=12, d_head=128, D_mlp=1536,
                    rope_axes=(16, 56, 56)),
    # 192 units of 2 KV tiles: parts a single KV tile long
    "split2": dict(B=8, L_txt=56, grid_h=12, grid_w=12, D=3072, H=24, d_head=128, D_mlp=3072,
                   rope_axes=(16, 56, 56)),
    # 384 units of 8 KV tiles (ragged last tile): one whole round, then a tail of 232 units
    "round_tail": dict(B=4, L_txt=40, grid_h=30, grid_w=32, D=3072, H=24, d_head=128, D_mlp=3072,
                       rope_axes=(16, 56, 56)),
    # head width 64: 240 units of 5 KV tiles
    "split_d64": dict(B=2, L_txt=32, grid_h=24, grid_w=24, D=2560, H=40, d_head=64, D_mlp=2560,
                      rope_axes=(16, 24, 24)),
    # 192 units of a single (ragged) KV tile: more units than SMs, none of them splittable
    "one_kv_tile": dict(B=8, L_txt=19, grid_h=9, grid_w=9, D=3072, H=24, d_head=128, D_mlp=3072,
                        rope_axes=(16, 56, 56)),
}
ATTN_CASES = {**{k: CONFIGS[k] for k in ("c1", "d128", "ragged", "tail")}, **SPLIT_CASES}


@pytest.mark.parametrize("name", list(ATTN_CASES))
@pytest.mark.parametrize("norm", [True, False])
def test_joint_attention(name, norm):
    cfg = ATTN_CASES[name]
    shape = api_shape(cfg)
    B, L, H, d, D = cfg["B"], api.seq_len(shape), cfg["H"], cfg["d_head"], cfg["D"]
    Lt = cfg["L_txt"]
    qkv = S.normal_bf16(f"at.{name}", (B, L, 3, H, d))
    if not norm:
        qkv[:, :, :2] *= 0.3  # keep raw scores moderate
    g = [S.norm_gain(f"at.g{i}", d) for i in range(4)]
    _, cs, sn = gpu_tables(shape)
    row_stride = 3 * D
    out_stride = D + 64
    out = torch.zeros((B, L, out_stride), dtype=torch.bfloat16, device="cuda")
    ws = api.alloc_workspace(api.workspace_size(shape, api.MMDIT_OP_ATTENTION))
    qn = [f32(g[0]), f32(g[1])] if norm else None
    kn = [f32(g[2]), f32(g[3])] if norm else None
    api.joint_attention_fwd(shape, bf16(qkv.reshape(B, L, 3 * D)), row_stride, qn, kn, cs, sn, out, out_stride, ws)
    q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    if norm:
        q = np.concatenate([O.rms_norm(q[:, :Lt], g[0], 1e-6), O.rms_norm(q[:, Lt:], g[1], 1e-6)], axis=1)
        k = np.concatenate([O.rms_norm(k[:, :Lt], g[2], 1e-6), O.rms_norm(k[:, Lt:], g[3], 1e-6)], axis=1)
    c, s = tables(cfg)
    ref = O.attention(O.rope_apply(q, c, s), O.rope_apply(k, c, s), v).reshape(B, L, D)
    got = host(out)
    assert_close(got[..., :D], ref, what=f"attention {name}")
    assert np.all(got[..., D:] == 0)


def test_attention_single_key_returns_v():
    cfg = dict(B=1, L_txt=0, grid_h=1, grid_w=1, D=256, H=2, d_head=128, D_mlp=256, rope_axes=(16, 56, 56))
    shape = api_shape(cfg)
    qkv = S.normal_bf16("one", (1, 1, 3, 2, 128))
    out = torch.empty((1, 1, 256), dtype=torch.bfloat16, device="cuda")
    ws = api.alloc_workspace(api.workspace_size(shape, api.MMDIT_OP_ATTENTION))
    _, cs, sn = gpu_tables(shape)
    api.joint_attention_fwd(shape, bf16(qkv.reshape(1, 1, 768)), 768, None, None, cs, sn, out, 256, ws)
    assert np.array_equal(host(out).reshape(2, 128), qkv[0, 0, 2])
