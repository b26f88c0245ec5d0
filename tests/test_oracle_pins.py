"""Pins of the float64 oracle against things other than itself: brute force on
tiny inputs, closed forms, invariants, library routines that the oracle does
not call (torch CPU float64), the counts the Luminal blog prints for a
Flux.2 Klein step, and planted mistakes that a pin must catch."""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import mmdit_oracle as O
from diffusion_transformer_image_mmdit_gb300 import synthetic as S

GOLD = os.path.join(os.path.dirname(__file__), "golden")
torch.set_default_dtype(torch.float64)


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(np.asarray(b)), 1e-300))


def rnd(name, shape, std=1.0):
    return S.normal(name, shape, std)


# ------------------------------------------------------------------ attention
def _attention_brute(q, k, v):
    B, Lq, H, d = q.shape
    Lk = k.shape[1]
    out = np.zeros_like(q)
    for b in range(B):
        for h in range(H):
            for i in range(Lq):
                sc = [sum(q[b, i, h, c] * k[b, j, h, c] for c in range(d)) / math.sqrt(d) for j in range(Lk)]
                m = max(sc)
                e = [math.exp(s - m) for s in sc]
                z = sum(e)
                for c in range(d):
                    out[b, i, h, c] = sum(e[j] * v[b, j, h, c] for j in range(Lk)) / z
    return out


def test_attention_brute_force():
    q, k, v = (rnd(n, (1, 5, 2, 4)) for n in ("aq", "ak", "av"))
    assert rel(O.attention(q, k, v), _attention_brute(q, k, v)) < 1e-13


def test_attention_rectangular_brute_force():
    q = rnd("rq", (2, 3, 1, 8))
    k = rnd("rk", (2, 7, 1, 8)) * 2
    v = rnd("rv", (2, 7, 1, 8))
    assert rel(O.attention(q, k, v), _attention_brute(q, k, v)) < 1e-13


def test_attention_vs_torch_sdpa():
    q, k, v = (rnd(n, (2, 37, 3, 16)) * 3 for n in ("tq", "tk", "tv"))
    ref = F.scaled_dot_product_attention(*(torch.from_numpy(t).transpose(1, 2) for t in (q, k, v))).transpose(1, 2)
    assert rel(O.attention(q, k, v), ref.numpy()) < 1e-13


def test_attention_one_key_returns_v():
    q = rnd("oq", (1, 6, 2, 8))
    k = rnd("ok", (1, 1, 2, 8))
    v = rnd("ov", (1, 1, 2, 8))
    out = O.attention(q, k, v)
    assert np.array_equal(out, np.broadcast_to(v, out.shape))


def test_attention_zero_query_is_mean_of_v():
    q = np.zeros((1, 3, 2, 8))
    k, v = rnd("zk", (1, 9, 2, 8)), rnd("zv", (1, 9, 2, 8))
    out = O.attention(q, k, v)
    assert np.abs(out - v.mean(axis=1, keepdims=True)).max() < 1e-15


def test_attention_key_permutation_invariance():
    q, k, v = (rnd(n, (1, 11, 2, 8)) for n in ("pq", "pk", "pv"))
    perm = np.random.default_rng(0).permutation(11)
    assert np.abs(O.attention(q, k, v) - O.attention(q, k[:, perm], v[:, perm])).max() < 1e-14


# ------------------------------------------------------------------ RoPE
def test_rope_ids_layout():
    ids = O.rope_ids(2, 2, 3)
    expect = [[0, 0, 0], [0, 0, 0], [0, 0, 0], [0, 0, 1], [0, 0, 2], [0, 1, 0], [0, 1, 1], [0, 1, 2]]
    assert ids.dtype == np.int32 and ids.tolist() == expect


def test_rope_ids_with_reference_layout():
    """Reference grid 1 x 3 after a 2 x 2 target and 2 text tokens, written out
    by hand: the reference tokens sit at (1, h, w) on their own grid."""
    ids = O.rope_ids(2, 2, 2, 1, 3)
    expect = [[0, 0, 0], [0, 0, 0], [0, 0, 0], [0, 0, 1], [0, 1, 0], [0, 1, 1], [1, 0, 0], [1, 0, 1], [1, 0, 2]]
    assert ids.dtype == np.int32 and ids.tolist() == expect
    # a target token and the reference token at the same (h, w) differ only on the axis-0 pairs
    c, s = O.rope_tables(O.rope_ids(0, 2, 3, 2, 3), (16, 24, 24), 10000.0)
    assert np.array_equal(c[:6, 8:], c[6:, 8:]) and np.array_equal(s[:6, 8:], s[6:, 8:])
    assert not np.allclose(c[:6, :8], c[6:, :8])


def test_latent_token_counts_golden():
    g = json.load(open(os.path.join(GOLD, "latent_tokens.json")))
    for c in g["cases"]:
        gh, gw = c["height"] // 16, c["width"] // 16
        assert (gh, gw) == (c["grid_h"], c["grid_w"])
        ids = O.rope_ids(c["text_tokens"], gh, gw)
        assert ids.shape == (c["tokens"], 3)
        assert (ids[c["text_tokens"]:, 1:] != 0).any(axis=1).sum() == c["image_tokens"] - 1


def test_rope_angles_closed_form():
    ids = O.rope_ids(3, 5, 7)
    ang = O.rope_angles(ids, (16, 24, 24), 10000.0)
    assert ang.shape == (3 + 35, 32)
    assert np.all(ang[:, :8] == 0) and np.all(ang[:3] == 0)
    # pair 0 of each spatial axis turns at frequency 1: the angle is the coordinate itself
    assert np.array_equal(ang[:, 8], ids[:, 1].astype(float))
    assert np.array_equal(ang[:, 20], ids[:, 2].astype(float))
    assert ang[3 + 7 * 4 + 5, 9] == pytest.approx(4 * 10000.0 ** (-2 / 24), rel=1e-15)


def test_rope_preserves_pair_norms():
    x = rnd("rx", (1, 38, 2, 64))
    c, s = O.rope_tables(O.rope_ids(3, 5, 7), (16, 24, 24), 10000.0)
    y = O.rope_apply(x, c, s)
    nx = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    ny = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    assert np.abs(nx - ny).max() < 1e-13


def test_rope_text_tokens_untouched():
    x = rnd("rt", (1, 38, 2, 64))
    c, s = O.rope_tables(O.rope_ids(3, 5, 7), (16, 24, 24), 10000.0)
    y = O.rope_apply(x, c, s)
    assert np.array_equal(y[:, :3], x[:, :3])
    assert np.array_equal(y[..., :16], x[..., :16])


def test_rope_relative_position_identity():
    """<R_m q, R_n k> depends only on m - n (per axis)."""
    d = 128
    q = rnd("rrq", (d,))
    k = rnd("rrk", (d,))
    axes = (16, 56, 56)

    def rot(vec, pos):
        ids = np.array([pos], dtype=np.int32)
        c, s = O.rope_tables(ids, axes, 10000.0)
        return O.rope_apply(vec[None, None, :], c, s)[0, 0]

    rng = np.random.default_rng(1)
    for _ in range(20):
        delta = rng.integers(-40, 40, size=3)
        delta[0] = 0
        m = rng.integers(0, 60, size=3); m[0] = 0
        n = rng.integers(0, 60, size=3); n[0] = 0
        a = rot(q, m + delta) @ rot(k, m)
        b = rot(q, n + delta) @ rot(k, n)
        assert abs(a - b) < 1e-11 * (1 + abs(a))


def test_rope_matches_complex_multiplication():
    """Independent restatement: adjacent channel pairs as complex numbers times e^{i angle}."""
    x = rnd("rc", (2, 38, 3, 64))
    ids = O.rope_ids(3, 5, 7)
    c, s = O.rope_tables(ids, (16, 24, 24), 10000.0)
    ang = np.arctan2(s, c)
    z = torch.view_as_complex(torch.from_numpy(x).reshape(2, 38, 3, 32, 2).contiguous())
    ref = torch.view_as_real(z * torch.polar(torch.ones(38, 1, 32), torch.from_numpy(ang)[:, None, :])).reshape(x.shape)
    assert rel(O.rope_apply(x, c, s), ref.numpy()) < 1e-14


# ------------------------------------------------------------------ norms / activations
def test_layer_norm_moments_and_torch():
    x = rnd("ln", (4, 7, 96)) * 3 + 1.5
    y = O.layer_norm(x, 1e-6)
    assert np.abs(y.mean(-1)).max() < 1e-13
    assert np.abs((y ** 2).mean(-1) - 1).max() < 1e-5
    assert rel(y, F.layer_norm(torch.from_numpy(x), (96,), eps=1e-6).numpy()) < 1e-14


def test_rms_norm_unit_rms_and_torch():
    x = rnd("rms", (5, 3, 128)) * 2
    g = S.norm_gain("g", 128)
    y = O.rms_norm(x, np.ones(128), 0.0)
    assert np.abs(np.sqrt((y ** 2).mean(-1)) - 1).max() < 1e-14
    ref = F.rms_norm(torch.from_numpy(x), (128,), weight=torch.from_numpy(g), eps=1e-6)
    assert rel(O.rms_norm(x, g, 1e-6), ref.numpy()) < 1e-14


def test_gelu_tanh():
    x = np.linspace(-8, 8, 1001)
    y = O.gelu_tanh(x)
    assert O.gelu_tanh(np.array([0.0]))[0] == 0.0
    assert np.abs((y - O.gelu_tanh(-x)) - x).max() < 1e-14
    assert rel(y, F.gelu(torch.from_numpy(x), approximate="tanh").numpy()) < 1e-15


def test_silu_and_linear():
    x = rnd("sx", (3, 5))
    assert rel(O.silu(x), F.silu(torch.from_numpy(x)).numpy()) < 1e-15
    w, b = rnd("lw", (4, 5)), rnd("lb", (4,))
    brute = np.array([[sum(x[i, k] * w[n, k] for k in range(5)) + b[n] for n in range(4)] for i in range(3)])
    assert rel(O.linear(x, w, b), brute) < 1e-15


# ------------------------------------------------------------------ blocks
TINY = O.Shape(B=2, L_txt=5, grid_h=3, grid_w=4, D=64, H=2, d_head=32, D_mlp=96, rope_axes=(8, 12, 12))


def _tables(sh):
    return O.rope_tables(O.rope_ids(sh.L_txt, sh.grid_h, sh.grid_w), sh.rope_axes, sh.rope_theta)


def _torch_ids(sh):
    """Position ids written out in torch from the reading (independent of the
    oracle's rope_ids): text (0, 0, 0), target (0, h, w), reference (1, h, w)."""
    gh, gw, rh, rw = sh.grid_h, sh.grid_w, sh.ref_h, sh.ref_w
    tgt = torch.stack([torch.zeros(gh * gw), torch.arange(gh).repeat_interleave(gw), torch.arange(gw).repeat(gh)], 1)
    ref = torch.stack([torch.ones(rh * rw), torch.arange(rh).repeat_interleave(rw), torch.arange(rw).repeat(rh)], 1)
    return torch.cat([torch.zeros(sh.L_txt, 3), tgt, ref], 0).to(torch.int64).numpy()


def _torch_rope(x, sh):
    ids = _torch_ids(sh)
    ang = []
    for a, d_a in enumerate(sh.rope_axes):
        om = torch.tensor(sh.rope_theta) ** (-torch.arange(0, d_a, 2) / d_a)
        ang.append(torch.from_numpy(ids[:, a]).double()[:, None] * om[None, :])
    ang = torch.cat(ang, 1)
    B, L, H, d = x.shape
    z = torch.view_as_complex(x.reshape(B, L, H, d // 2, 2).contiguous())
    return torch.view_as_real(z * torch.polar(torch.ones_like(ang), ang)[:, None, :]).reshape(B, L, H, d)


def _torch_act(t, sh):
    if sh.mlp == "swiglu":
        gate, up = t.chunk(2, dim=-1)
        return F.silu(gate) * up
    return F.gelu(t, approximate="tanh")


def _torch_double(x_txt, x_img, vec, wt, sh):
    T = torch.from_numpy
    D, H, d = sh.D, sh.H, sh.d_head
    st = {}
    for s, x in (("txt", T(x_txt)), ("img", T(x_img))):
        w = {k: T(v) for k, v in wt[s].items()}
        m = F.linear(F.silu(T(vec)), w["mod_w"], w["mod_b"]).unsqueeze(1).chunk(6, dim=-1)
        y = F.layer_norm(x, (D,), eps=sh.eps_ln) * (1 + m[1]) + m[0]
        q, k, v = F.linear(y, w["qkv_w"], w["qkv_b"]).split(D, dim=-1)
        B, L, _ = q.shape
        q = F.rms_norm(q.reshape(B, L, H, d), (d,), weight=w["q_norm"], eps=sh.eps_rms)
        k = F.rms_norm(k.reshape(B, L, H, d), (d,), weight=w["k_norm"], eps=sh.eps_rms)
        st[s] = (x, w, m, q, k, v.reshape(B, L, H, d))
    q = _torch_rope(torch.cat([st["txt"][3], st["img"][3]], 1), sh)
    k = _torch_rope(torch.cat([st["txt"][4], st["img"][4]], 1), sh)
    v = torch.cat([st["txt"][5], st["img"][5]], 1)
    o = F.scaled_dot_product_attention(q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2)).transpose(1, 2)
    o = o.reshape(o.shape[0], o.shape[1], D)
    outs = []
    for s, sl in (("txt", slice(0, sh.L_txt)), ("img", slice(sh.L_txt, None))):
        x, w, m, *_ = st[s]
        x = x + m[2] * F.linear(o[:, sl], w["proj_w"], w["proj_b"])
        y = F.layer_norm(x, (D,), eps=sh.eps_ln) * (1 + m[4]) + m[3]
        x = x + m[5] * F.linear(_torch_act(F.linear(y, w["mlp_in_w"], w["mlp_in_b"]), sh), w["mlp_out_w"], w["mlp_out_b"])
        outs.append(x.numpy())
    return outs


def _torch_single(x, vec, wt, sh):
    T = torch.from_numpy
    D, H, d = sh.D, sh.H, sh.d_head
    w = {k: T(v) for k, v in wt.items()}
    x = T(x)
    m = F.linear(F.silu(T(vec)), w["mod_w"], w["mod_b"]).unsqueeze(1).chunk(3, dim=-1)
    y = F.layer_norm(x, (D,), eps=sh.eps_ln) * (1 + m[1]) + m[0]
    h = F.linear(y, w["lin1_w"], w["lin1_b"])
    q, k, v, mlp = h.split([D, D, D, h.shape[-1] - 3 * D], dim=-1)
    B, L, _ = q.shape
    q = _torch_rope(F.rms_norm(q.reshape(B, L, H, d), (d,), weight=w["q_norm"], eps=sh.eps_rms), sh)
    k = _torch_rope(F.rms_norm(k.reshape(B, L, H, d), (d,), weight=w["k_norm"], eps=sh.eps_rms), sh)
    o = F.scaled_dot_product_attention(q.transpose(1, 2), k.transpose(1, 2), v.reshape(B, L, H, d).transpose(1, 2))
    o = o.transpose(1, 2).reshape(B, L, D)
    return (x + m[2] * F.linear(torch.cat([o, _torch_act(mlp, sh)], -1), w["lin2_w"], w["lin2_b"])).numpy()


def _double_inputs(sh, scale_w=1.0):
    wt = S.double_block_params("pin.dbl", sh.D, sh.d_head, sh.D_mlp)
    if scale_w != 1.0:
        for s in wt.values():
            for k in s:
                if k.endswith("_w"):
                    s[k] = s[k] * scale_w
    a = S.activations(sh.B, sh.L_txt, sh.L_img, sh.D)
    return wt, a


def test_double_block_vs_torch_restatement():
    sh = TINY
    wt, a = _double_inputs(sh, scale_w=25.0)  # larger weights so every branch matters
    c, s = _tables(sh)
    got = O.double_block(a["x_txt"], a["x_img"], a["vec"], wt, sh, c, s)
    ref = _torch_double(a["x_txt"], a["x_img"], a["vec"], wt, sh)
    assert rel(got[0], ref[0]) < 1e-12 and rel(got[1], ref[1]) < 1e-12
    # the branches really move the residual stream
    assert rel(got[1], a["x_img"]) > 0.1


def test_double_block_row_subset_matches_full():
    sh = TINY
    wt, a = _double_inputs(sh, scale_w=25.0)
    c, s = _tables(sh)
    full = O.double_block(a["x_txt"], a["x_img"], a["vec"], wt, sh, c, s)
    part = O.double_block(a["x_txt"], a["x_img"], a["vec"], wt, sh, c, s, rows_txt=[0, 4], rows_img=[1, 11])
    assert rel(part[0], full[0][:, [0, 4]]) < 1e-14
    assert rel(part[1], full[1][:, [1, 11]]) < 1e-14


def test_single_block_vs_torch_restatement():
    sh = TINY
    w = S.single_block_params("pin.sgl", sh.D, sh.d_head, sh.D_mlp)
    for k in w:
        if k.endswith("_w"):
            w[k] = w[k] * 25.0
    x = S.normal_f32("pin.x", (sh.B, sh.L, sh.D))
    vec = S.normal_f32("pin.vec", (sh.B, sh.D))
    c, s = _tables(sh)
    got = O.single_block(x, vec, w, sh, c, s)
    assert rel(got, _torch_single(x, vec, w, sh)) < 1e-12
    part = O.single_block(x, vec, w, sh, c, s, rows=[0, 7, 16])
    assert rel(part, got[:, [0, 7, 16]]) < 1e-14


def test_swiglu_vs_torch():
    h = rnd("sw.h", (3, 5, 40), 3.0)
    got = O.swiglu(h)
    t = torch.from_numpy(h)
    assert got.shape == (3, 5, 20)
    assert rel(got, (F.silu(t[..., :20]) * t[..., 20:]).numpy()) < 1e-15
    assert rel(O.mlp_act(h, O.Shape(1, 1, 1, 1, 4, 1, 4, 4, mlp="swiglu")), got) == 0.0


@pytest.mark.parametrize("which", ["double", "single"])
def test_swiglu_blocks_vs_torch_restatement(which):
    import dataclasses
    sh = dataclasses.replace(TINY, mlp="swiglu")
    c, s = _tables(sh)
    if which == "double":
        wt = S.double_block_params("pin.swd", sh.D, sh.d_head, sh.D_mlp, mlp="swiglu")
        for st in wt.values():
            for k in st:
                if k.endswith("_w"):
                    st[k] = st[k] * 25.0
        a = S.activations(sh.B, sh.L_txt, sh.L_img, sh.D)
        got = O.double_block(a["x_txt"], a["x_img"], a["vec"], wt, sh, c, s)
        ref = _torch_double(a["x_txt"], a["x_img"], a["vec"], wt, sh)
        assert rel(got[0], ref[0]) < 1e-12 and rel(got[1], ref[1]) < 1e-12
        assert rel(got[1], a["x_img"]) > 0.1
    else:
        w = S.single_block_params("pin.sws", sh.D, sh.d_head, sh.D_mlp, mlp="swiglu")
        for k in w:
            if k.endswith("_w"):
                w[k] = w[k] * 25.0
        x = S.normal_f32("pin.swx", (sh.B, sh.L, sh.D))
        vec = S.normal_f32("pin.swv", (sh.B, sh.D))
        assert rel(O.single_block(x, vec, w, sh, c, s), _torch_single(x, vec, w, sh)) < 1e-12


def test_quantisation_hook_reaches_exactly_the_gemm_inputs():
    """qin sees the inputs of the four GEMM linears per stream (double) and of
    lin1 and lin2 (single), with their widths, and nothing else; identity
    leaves the block unchanged."""
    sh = TINY
    wt, a = _double_inputs(sh)
    c, s = _tables(sh)
    seen = []

    def spy(x):
        seen.append(x.shape[-1])
        return x
    plain = O.double_block(a["x_txt"], a["x_img"], a["vec"], wt, sh, c, s)
    got = O.double_block(a["x_txt"], a["x_img"], a["vec"], wt, sh, c, s, qin=spy)
    assert sorted(seen) == sorted([sh.D, sh.D, sh.D, sh.D_mlp] * 2)
    assert rel(got[1], plain[1]) == 0.0
    seen.clear()
    w = S.single_block_params("pin.q8s", sh.D, sh.d_head, sh.D_mlp)
    x = S.normal_f32("pin.q8x", (sh.B, sh.L, sh.D))
    vec = S.normal_f32("pin.q8v", (sh.B, sh.D))
    O.single_block(x, vec, w, sh, c, s, qin=spy)
    assert sorted(seen) == [sh.D, sh.D + sh.D_mlp]


def test_step_hooks_reach_every_block_linear():
    """denoise_step hands qin to every block: per double block the four GEMM inputs of each stream, per
    single block lin1's and lin2's; identity hooks leave the step bit-identical."""
    sh = O.Shape(B=1, L_txt=8, grid_h=4, grid_w=4, D=64, H=2, d_head=32, D_mlp=128, rope_axes=(8, 12, 12),
                 C_lat=16, t_dim=32)
    W = S.embed_params(sh.D, sh.C_lat, sh.t_dim, seed=9)
    W["double"] = [S.double_block_params(f"pin.sh.d{i}", sh.D, sh.d_head, sh.D_mlp) for i in range(2)]
    W["single"] = [S.single_block_params(f"pin.sh.s{i}", sh.D, sh.d_head, sh.D_mlp) for i in range(3)]
    x_lat = S.normal_f32("pin.sh.lat", (sh.B, sh.L_img, sh.C_lat))
    x_txt = S.normal_f32("pin.sh.txt", (sh.B, sh.L_txt, sh.D))
    seen = []

    def spy(x):
        seen.append(x.shape[-1])
        return x
    plain = O.denoise_step(x_lat, x_txt, 1.0, 0.9, W, sh)
    got = O.denoise_step(x_lat, x_txt, 1.0, 0.9, W, sh, qin=spy)
    assert sorted(seen) == sorted([sh.D, sh.D, sh.D, sh.D_mlp] * 2 * 2 + [sh.D, sh.D + sh.D_mlp] * 3)
    assert np.array_equal(got[0], plain[0]) and np.array_equal(got[1], plain[1])
    # an identity precision model only changes the fp64 evaluation order inside the attention
    ident = O.denoise_step(x_lat, x_txt, 1.0, 0.9, W, sh, rnd=lambda t: t)
    assert rel(ident[1], plain[1]) < 1e-12


def _zero_gates(mod_w, mod_b, n_chunks, gate_chunks):
    D = mod_w.shape[0] // n_chunks
    mod_w, mod_b = mod_w.copy(), mod_b.copy()
    for g in gate_chunks:
        mod_w[g * D:(g + 1) * D] = 0
        mod_b[g * D:(g + 1) * D] = 0
    return mod_w, mod_b


def test_precision_hook_is_inert_by_default_and_bf16_sized():
    """rnd=None is the plain definition; rnd=bf16 rounding moves the block
    output by the size of one bf16 rounding (2^-9) carried through."""
    sh = TINY
    wt, a = _double_inputs(sh)
    c, s = _tables(sh)
    plain = O.double_block(a["x_txt"], a["x_img"], a["vec"], wt, sh, c, s)
    ident = O.double_block(a["x_txt"], a["x_img"], a["vec"], wt, sh, c, s, rnd=lambda x: x)
    assert rel(ident[1], plain[1]) < 1e-14  # only the softmax normalisation order differs
    emu = O.double_block(a["x_txt"], a["x_img"], a["vec"], wt, sh, c, s, rnd=S.round_bf16)
    r = rel(emu[1] - a["x_img"], plain[1] - a["x_img"])
    assert 1e-4 < r < 2e-2


def test_zero_gates_make_blocks_identity():
    sh = TINY
    wt, a = _double_inputs(sh)
    c, s = _tables(sh)
    for st in wt.values():
        st["mod_w"], st["mod_b"] = _zero_gates(st["mod_w"], st["mod_b"], 6, (2, 5))
    t, i = O.double_block(a["x_txt"], a["x_img"], a["vec"], wt, sh, c, s)
    assert np.array_equal(t, a["x_txt"]) and np.array_equal(i, a["x_img"])
    w = S.single_block_params("pin.sgl", sh.D, sh.d_head, sh.D_mlp)
    w["mod_w"], w["mod_b"] = _zero_gates(w["mod_w"], w["mod_b"], 3, (2,))
    x = np.concatenate([a["x_txt"], a["x_img"]], 1)
    assert np.array_equal(O.single_block(x, a["vec"], w, sh, c, s), x)


def test_zero_branch_weights_leave_gated_biases():
    """With proj and MLP-out weights zero, each stream gets exactly
    x + gate1 * b_proj + gate2 * b_mlp_out."""
    sh = TINY
    wt, a = _double_inputs(sh)
    c, s = _tables(sh)
    for st in wt.values():
        st["proj_w"] = np.zeros_like(st["proj_w"])
        st["mlp_out_w"] = np.zeros_like(st["mlp_out_w"])
    t, i = O.double_block(a["x_txt"], a["x_img"], a["vec"], wt, sh, c, s)
    for name, x, out in (("txt", a["x_txt"], t), ("img", a["x_img"], i)):
        w = wt[name]
        m = O.silu(a["vec"]) @ w["mod_w"].T + w["mod_b"]
        D = sh.D
        g1, g2 = m[:, None, 2 * D:3 * D], m[:, None, 5 * D:6 * D]
        assert np.abs(out - (x + g1 * w["proj_b"] + g2 * w["mlp_out_b"])).max() < 1e-14


def test_klein_step_counts_golden():
    """One step of a Klein-shaped stack calls LN+modulate 57 times and
    RMSNorm (fused with RoPE on the pages) 80 times, with 32 attention sites."""
    g = json.load(open(os.path.join(GOLD, "klein_step_counts.json")))
    sh = O.Shape(B=1, L_txt=2, grid_h=2, grid_w=2, D=32, H=2, d_head=16, D_mlp=32, rope_axes=(4, 6, 6), C_lat=8, t_dim=16)
    W = S.embed_params(sh.D, sh.C_lat, sh.t_dim)
    W["double"] = [S.double_block_params(f"k.d{i}", sh.D, sh.d_head, sh.D_mlp) for i in range(g["n_double"])]
    W["single"] = [S.single_block_params(f"k.s{i}", sh.D, sh.d_head, sh.D_mlp) for i in range(g["n_single"])]
    counts = {"ln": 0, "rms": 0, "attn": 0}
    ln, rms, att = O.layer_norm, O.rms_norm, O.attention

    def c_ln(*a, **k):
        counts["ln"] += 1
        return ln(*a, **k)

    def c_rms(*a, **k):
        counts["rms"] += 1
        return rms(*a, **k)

    def c_att(*a, **k):
        counts["attn"] += 1
        return att(*a, **k)

    O.layer_norm, O.rms_norm, O.attention = c_ln, c_rms, c_att
    try:
        x_lat = S.normal_f32("k.lat", (1, 4, 8))
        x_txt = S.normal_f32("k.txt", (1, 2, 32))
        O.denoise_step(x_lat, x_txt, 1.0, 0.75, W, sh)
    finally:
        O.layer_norm, O.rms_norm, O.attention = ln, rms, att
    assert counts["ln"] == g["layernorm_modulate_per_step"]
    assert counts["rms"] == g["rmsnorm_rope_per_step"]
    assert counts["attn"] == 2 * g["n_double"] + g["n_single"]  # double blocks: one call per stream's query rows
    assert g["n_double"] + g["n_single"] == g["attention_sites_per_step"]


# ------------------------------------------------------------------ step pieces
def test_timestep_sinusoid_closed_forms():
    e = O.timestep_sinusoid([0.0, 3.0], 256)
    assert np.array_equal(e[0, :128], np.ones(128)) and np.array_equal(e[0, 128:], np.zeros(128))
    assert e[1, 0] == math.cos(3.0) and e[1, 128] == math.sin(3.0)
    assert e[1, 64] == pytest.approx(math.cos(3.0 * 10000.0 ** -0.5), rel=1e-14)


def test_sigma_schedule():
    s = O.sigma_schedule(4, 0.0)
    assert np.allclose(s, [1, 0.75, 0.5, 0.25, 0], rtol=0, atol=1e-16)
    s = O.sigma_schedule(2, math.log(3.0))
    assert np.allclose(s, [1.0, 0.75, 0.0], rtol=0, atol=1e-15)
    s = O.sigma_schedule(50, O.shift_mu(6889))
    assert s[0] == 1.0 and s[-1] == 0.0 and np.all(np.diff(s) < 0)
    assert O.shift_mu(4096) == pytest.approx(1.15) and O.shift_mu(256) == pytest.approx(0.5)


def test_euler_constant_velocity_telescopes():
    x0 = rnd("ex", (3, 10))
    v = rnd("ev", (3, 10))
    sig = O.sigma_schedule(28, O.shift_mu(4096))
    x = x0
    for i in range(28):
        x = O.euler_step(x, v, sig[i], sig[i + 1])
    assert np.abs(x - (x0 - v)).max() < 1e-13
    assert np.array_equal(O.euler_step(x0, v, 0.5, 0.5), x0)


def test_time_embed_and_final_layer_vs_torch():
    sh = O.Shape(B=2, L_txt=3, grid_h=2, grid_w=3, D=32, H=2, d_head=16, D_mlp=32, C_lat=8, t_dim=16)
    W = S.embed_params(sh.D, sh.C_lat, sh.t_dim)
    T = {k: torch.from_numpy(v) for k, v in W.items()}
    vec = O.time_embed(0.6, W, sh)
    half = 8
    f = torch.exp(-math.log(10000.0) * torch.arange(half) / half)
    a = torch.full((2, 1), 600.0) * f[None]
    ref = F.linear(F.silu(F.linear(torch.cat([a.cos(), a.sin()], 1), T["t_w1"], T["t_b1"])), T["t_w2"], T["t_b2"])
    assert rel(vec, ref.numpy()) < 1e-14
    x = S.normal_f32("fl.x", (2, 6, 32))
    m = F.linear(F.silu(torch.from_numpy(vec)), T["final_mod_w"], T["final_mod_b"]).unsqueeze(1).chunk(2, -1)
    y = F.layer_norm(torch.from_numpy(x), (32,), eps=1e-6) * (1 + m[1]) + m[0]
    assert rel(O.final_layer(x, vec, W, sh), F.linear(y, T["final_w"], T["final_b"]).numpy()) < 1e-14


# ------------------------------------------------------------------ FP8 (e4m3)
def _e4m3_table():
    """All finite e4m3 codes decoded from the bit layout: sign, 4 exponent bits
    (bias 7; 0 = subnormal), 3 mantissa bits; exponent 15 with mantissa 7 is
    NaN.  Returns (values, mantissa LSB) of the non-negative codes."""
    vals, lsb = [], []
    for code in range(128):
        e, m = (code >> 3) & 15, code & 7
        if e == 15 and m == 7:
            continue
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        vals.append(v)
        lsb.append(m & 1)
    return np.array(vals), np.array(lsb)


def test_round_e4m3_brute_force():
    vals, lsb = _e4m3_table()
    assert vals.max() == 448.0 and vals[vals > 0].min() == 2.0 ** -9 and len(vals) == 127
    xs = np.concatenate([rnd("f8.x", (4000,), 1.0), rnd("f8.y", (2000,), 60.0), rnd("f8.z", (1000,), 0.01),
                         (vals[1:] + vals[:-1]) / 2, -(vals[1:] + vals[:-1]) / 2, [500.0, -1e4, 0.0]])
    got = O.round_e4m3(xs)
    for x, g in zip(xs, got):
        a = min(abs(x), 448.0)
        d = np.abs(vals - a)
        cand = np.flatnonzero(d == d.min())
        pick = cand[0] if len(cand) == 1 else cand[lsb[cand] == 0][0]  # ties to the even mantissa
        assert g == math.copysign(vals[pick], x) or (x == 0 and g == 0), (x, g, vals[pick])


def test_quantize_f8_rows_invariants():
    x = rnd("f8.rows", (6, 100), 3.0)
    x[2] = 0.0
    q, s = O.quantize_f8_rows(x)
    assert np.abs(q).max() <= 448.0
    vals, _ = _e4m3_table()
    assert np.isin(np.abs(q), vals).all()
    for r in (0, 1, 3, 4, 5):
        assert np.abs(q[r]).max() == 448.0
    assert s[2] == 1.0 and not q[2].any()
    # every element within half a local e4m3 step (relative 2^-4 of the normal range) of x / s
    xs = x / s[:, None].astype(np.float64)
    step = np.exp2(np.maximum(np.floor(np.log2(np.maximum(np.abs(xs), 1e-30))), -6.0) - 3.0)
    assert (np.abs(q - xs) <= step / 2 * (1 + 1e-6) + 1e-12).all()


# ------------------------------------------------------------------ conditioning and the sampling loop
def _cond_params(sh, C_txt, C_pool):
    W = S.embed_params(sh.D, sh.C_lat, sh.t_dim, seed=5)
    W["txt_in_w"], W["txt_in_b"] = S.linear_params("cond.txt_in", sh.D, C_txt, 5)
    W["g_w1"], W["g_b1"] = S.linear_params("cond.guid1", sh.D, sh.t_dim, 5)
    W["g_w2"], W["g_b2"] = S.linear_params("cond.guid2", sh.D, sh.D, 5)
    W["y_w1"], W["y_b1"] = S.linear_params("cond.vec1", sh.D, C_pool, 5)
    W["y_w2"], W["y_b2"] = S.linear_params("cond.vec2", sh.D, sh.D, 5)
    return W


def _tiny_step_model(sh, seed=5):
    W = _cond_params(sh, 24, 12)
    W["double"] = [S.double_block_params(f"smp.d{i}", sh.D, sh.d_head, sh.D_mlp, seed) for i in range(sh.n_double)]
    W["single"] = [S.single_block_params(f"smp.s{i}", sh.D, sh.d_head, sh.D_mlp, seed) for i in range(sh.n_single)]
    return W


def _sample_inputs(sh):
    return (rnd("smp.x", (sh.B, sh.L_img, sh.C_lat)), rnd("smp.txt", (sh.B, sh.L_txt, 24)), rnd("smp.y", (sh.B, 12)))


SH_SAMPLE = O.Shape(B=2, L_txt=3, grid_h=2, grid_w=2, D=32, H=2, d_head=16, D_mlp=64, rope_axes=(4, 6, 6),
                    C_lat=8, t_dim=16, n_double=1, n_single=1)


def test_conditioning_embeddings_vs_torch():
    sh = O.Shape(B=2, L_txt=3, grid_h=2, grid_w=3, D=32, H=2, d_head=16, D_mlp=32, C_lat=8, t_dim=16)
    W = _cond_params(sh, 24, 12)
    T = {k: torch.from_numpy(v) for k, v in W.items()}
    half = 8
    f = torch.exp(-math.log(10000.0) * torch.arange(half) / half)
    a = torch.full((2, 1), 3500.0) * f[None]
    ref = F.linear(F.silu(F.linear(torch.cat([a.cos(), a.sin()], 1), T["g_w1"], T["g_b1"])), T["g_w2"], T["g_b2"])
    assert rel(O.guidance_embed(3.5, W, sh), ref.numpy()) < 1e-14
    y = rnd("cond.y", (2, 12))
    ref = F.linear(F.silu(F.linear(torch.from_numpy(y), T["y_w1"], T["y_b1"])), T["y_w2"], T["y_b2"])
    assert rel(O.pooled_embed(y, W), ref.numpy()) < 1e-14
    txt = rnd("cond.txt", (2, 3, 24))
    assert rel(O.txt_in(txt, W), F.linear(torch.from_numpy(txt), T["txt_in_w"], T["txt_in_b"]).numpy()) < 1e-14


def test_sample_constant_velocity_closed_form():
    """With a zero final projection the velocity is its bias b at every step,
    whatever the blocks and the conditioning do, so the loop telescopes to
    x_N = x_0 + (sigma_N - sigma_0) b = x_0 - b."""
    sh = SH_SAMPLE
    W = _tiny_step_model(sh)
    W["final_w"] = np.zeros_like(W["final_w"])
    x0, txt, y = _sample_inputs(sh)
    sig = O.sigma_schedule(3, O.shift_mu(sh.L_img))
    x = O.sample(x0, txt, y, 3.5, sig, W, sh)
    assert np.abs(x - (x0 - W["final_b"])).max() < 1e-12


def test_vec_add_is_a_shift_of_the_time_embedding_bias():
    """Adding a constant vector a to the timestep embedding is the same model
    as adding a to the output bias of the time MLP (B = 1)."""
    sh = O.Shape(B=1, L_txt=3, grid_h=2, grid_w=2, D=32, H=2, d_head=16, D_mlp=64, rope_axes=(4, 6, 6),
                 C_lat=8, t_dim=16, n_double=1, n_single=1)
    W = _tiny_step_model(sh)
    x0 = rnd("va.x", (1, sh.L_img, sh.C_lat))
    xt = rnd("va.t", (1, sh.L_txt, sh.D))
    a = rnd("va.a", (1, sh.D))
    got, _ = O.denoise_step(x0, xt, 0.8, 0.6, W, sh, vec_add=a)
    W2 = dict(W)
    W2["t_b2"] = W["t_b2"] + a[0]
    want, _ = O.denoise_step(x0, xt, 0.8, 0.6, W2, sh)
    assert rel(got, want) < 1e-13
    plain, _ = O.denoise_step(x0, xt, 0.8, 0.6, W, sh)
    assert rel(got, plain) > 1e-6  # the conditioning reaches the output


def test_sample_conditioning_acts_only_through_modulation_and_text():
    """With every modulation projection zero, the guidance scale and the
    pooled vector cannot reach the output; with a zero text projection, the
    text-encoder output cannot either (the text stream is its bias)."""
    sh = SH_SAMPLE
    W = _tiny_step_model(sh)
    x0, txt, y = _sample_inputs(sh)
    sig = O.sigma_schedule(2, 0.8)
    Z = dict(W)
    Z["final_mod_w"], Z["final_mod_b"] = np.zeros_like(W["final_mod_w"]), np.zeros_like(W["final_mod_b"])
    Z["double"] = [{st: {k: (np.zeros_like(v) if k.startswith("mod") else v) for k, v in blk[st].items()}
                    for st in ("txt", "img")} for blk in W["double"]]
    Z["single"] = [{k: (np.zeros_like(v) if k.startswith("mod") else v) for k, v in blk.items()} for blk in W["single"]]
    a = O.sample(x0, txt, y, 3.5, sig, Z, sh)
    b = O.sample(x0, txt, 2.0 * y + 1.0, 1.0, sig, Z, sh)
    assert np.array_equal(a, b)
    T = dict(W)
    T["txt_in_w"] = np.zeros_like(W["txt_in_w"])
    assert np.array_equal(O.sample(x0, txt, y, 3.5, sig, T, sh), O.sample(x0, -txt, y, 3.5, sig, T, sh))
    assert not np.array_equal(O.sample(x0, txt, y, 3.5, sig, W, sh), O.sample(x0, txt, y, 1.0, sig, W, sh))


# ------------------------------------------------------------------ whole step composition
# One denoising step in the order the Luminal blog's per-step operation list
# (section "What the compiler found on its own") and its model description
# (section "Flux.2 Klein 9B") give: timestep embedding, latent patch
# projection, the double-stream blocks on separate text and image streams,
# the concatenation [text; image], the single-stream blocks, the final
# LayerNorm + modulate + projection on the image tokens, and the Euler update
# of the sampler (section "The AMD MI300X pipeline").  Restated below with
# torch library routines (F.linear, F.layer_norm, scaled_dot_product_attention)
# and compared with the oracle's denoise_step.
SH_STEP = O.Shape(B=2, L_txt=5, grid_h=3, grid_w=4, D=64, H=2, d_head=32, D_mlp=96, rope_axes=(8, 12, 12),
                  C_lat=64, t_dim=32, n_double=2, n_single=2)


def _step_case(sh):
    """Weights scaled up (x10) so that every layer visibly moves the result;
    C_lat = D so that a step that skips the patch projection still runs."""
    W = S.embed_params(sh.D, sh.C_lat, sh.t_dim, seed=9)
    W["double"] = [S.double_block_params(f"stp.d{i}", sh.D, sh.d_head, sh.D_mlp, 9) for i in range(sh.n_double)]
    W["single"] = [S.single_block_params(f"stp.s{i}", sh.D, sh.d_head, sh.D_mlp, 9) for i in range(sh.n_single)]
    for d in [W] + W["single"] + [blk[st] for blk in W["double"] for st in ("txt", "img")]:
        for k in list(d):
            if k.endswith("_w"):
                d[k] = d[k] * 10.0
    x_lat = rnd("stp.lat", (sh.B, sh.L_gen, sh.C_lat))
    x_txt = rnd("stp.txt", (sh.B, sh.L_txt, sh.D))
    vec_add = rnd("stp.add", (sh.B, sh.D))
    return W, x_lat, x_txt, vec_add


def _torch_step(x_lat, x_txt, sigma, sigma_next, W, sh, vec_add, x_ref=None):
    T = torch.from_numpy
    w = {k: T(v) for k, v in W.items() if isinstance(v, np.ndarray)}
    half = sh.t_dim // 2
    f = torch.exp(-math.log(10000.0) * torch.arange(half) / half)
    a = torch.full((sh.B, 1), 1000.0 * sigma) * f[None]
    vec = F.linear(F.silu(F.linear(torch.cat([a.cos(), a.sin()], 1), w["t_w1"], w["t_b1"])), w["t_w2"], w["t_b2"])
    vec = vec + T(vec_add)
    h_txt = x_txt
    lat = T(x_lat) if x_ref is None else torch.cat([T(x_lat), T(x_ref)], 1)
    h_img = F.linear(lat, w["img_in_w"], w["img_in_b"]).numpy()
    for blk in W["double"]:
        h_txt, h_img = _torch_double(h_txt, h_img, vec.numpy(), blk, sh)
    x = torch.cat([T(h_txt), T(h_img)], 1)
    for blk in W["single"]:
        x = T(_torch_single(x.numpy(), vec.numpy(), blk, sh))
    m = F.linear(F.silu(vec), w["final_mod_w"], w["final_mod_b"]).unsqueeze(1).chunk(2, -1)
    y = F.layer_norm(x[:, sh.L_txt:sh.L_txt + sh.grid_h * sh.grid_w], (sh.D,), eps=sh.eps_ln) * (1 + m[1]) + m[0]
    v = F.linear(y, w["final_w"], w["final_b"])
    return (T(x_lat) + (sigma_next - sigma) * v).numpy(), v.numpy()


def test_denoise_step_vs_torch_restatement():
    sh = SH_STEP
    W, x_lat, x_txt, vec_add = _step_case(sh)
    sig = O.sigma_schedule(50, O.shift_mu(sh.L_img))
    got_x, got_v = O.denoise_step(x_lat, x_txt, sig[3], sig[4], W, sh, vec_add=vec_add)
    ref_x, ref_v = _torch_step(x_lat, x_txt, sig[3], sig[4], W, sh, vec_add)
    assert rel(got_v, ref_v) < 1e-12, rel(got_v, ref_v)
    assert rel(got_x - x_lat, ref_x - x_lat) < 1e-12
    assert rel(got_x, x_lat) > 1e-3  # the step moves the latent


def _step_variant(x_lat, x_txt, sigma, sigma_next, W, sh, vec_add=None, rnd=None, qin=None, x_ref=None, *,
                  final_head=False, skip_img_in=False, img_first=False, drop_vec_add=False, final_on_ref=False):
    """The step composed from the oracle's public pieces, with switches that
    each plant one composition mistake (all off: the oracle's own step)."""
    cos, sin = O.rope_tables(O.rope_ids(sh.L_txt, sh.grid_h, sh.grid_w, sh.ref_h, sh.ref_w), sh.rope_axes,
                             sh.rope_theta)
    vec = O.time_embed(sigma, W, sh)
    if vec_add is not None and not drop_vec_add:
        vec = vec + vec_add
    lat = x_lat if x_ref is None else np.concatenate([x_lat, x_ref], axis=1)
    h_img = np.asarray(lat, np.float64) if skip_img_in else O.img_in(lat, W)
    h_txt = x_txt
    for blk in W["double"]:
        h_txt, h_img = O.double_block(h_txt, h_img, vec, blk, sh, cos, sin)
    x = np.concatenate([h_img, h_txt] if img_first else [h_txt, h_img], axis=1)
    for blk in W["single"]:
        x = O.single_block(x, vec, blk, sh, cos, sin)
    if final_on_ref:
        img = x[:, sh.L_txt + sh.L_gen:]
    else:
        img = x[:, :sh.L_gen] if (img_first or final_head) else x[:, sh.L_txt:sh.L_txt + sh.L_gen]
    v = O.final_layer(img, vec, W, sh)
    return O.euler_step(x_lat, v, sigma, sigma_next), v


def test_step_variant_without_switches_is_the_oracle_step():
    sh = SH_STEP
    W, x_lat, x_txt, vec_add = _step_case(sh)
    a = O.denoise_step(x_lat, x_txt, 0.7, 0.65, W, sh, vec_add=vec_add)
    b = _step_variant(x_lat, x_txt, 0.7, 0.65, W, sh, vec_add)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("mistake", ["final_head", "skip_img_in", "img_first", "drop_vec_add"])
def test_planted_step_composition_mistakes_are_caught(monkeypatch, mistake):
    """Each plant: the final layer reading the first L_img rows (text
    included) instead of the image slice; the patch projection skipped; the
    sequence concatenated as [image; text]; the conditioning vector dropped."""
    def planted(*args, **kw):
        return _step_variant(*args, **kw, **{mistake: True})

    _planted(monkeypatch, "denoise_step", planted, test_denoise_step_vs_torch_restatement)


# Image-to-image: the reference latent is projected like the noise latent and
# appended to its tokens (Luminal blog, "The AMD MI300X pipeline"); positions
# (1, h, w) per the reading in rope_ids.  The reference grid has the target's
# size here so that a step reading the wrong image slice still runs.
SH_I2I = O.Shape(B=2, L_txt=5, grid_h=3, grid_w=4, D=64, H=2, d_head=32, D_mlp=96, rope_axes=(8, 12, 12),
                 C_lat=64, t_dim=32, n_double=2, n_single=2, ref_h=3, ref_w=4)


def test_i2i_step_vs_torch_restatement():
    sh = SH_I2I
    W, x_lat, x_txt, vec_add = _step_case(sh)
    x_ref = rnd("stp.ref", (sh.B, sh.L_ref, sh.C_lat))
    got_x, got_v = O.denoise_step(x_lat, x_txt, 0.8, 0.7, W, sh, vec_add=vec_add, x_ref=x_ref)
    ref_x, ref_v = _torch_step(x_lat, x_txt, 0.8, 0.7, W, sh, vec_add, x_ref=x_ref)
    assert got_v.shape == (sh.B, sh.L_gen, sh.C_lat)
    assert rel(got_v, ref_v) < 1e-12, rel(got_v, ref_v)
    assert rel(got_x - x_lat, ref_x - x_lat) < 1e-12
    # the reference reaches the velocity of the target tokens (through attention)
    other, _ = O.denoise_step(x_lat, x_txt, 0.8, 0.7, W, sh, vec_add=vec_add, x_ref=x_ref * 0.5)
    assert rel(other, got_x) > 1e-6


def test_planted_reference_mistakes_are_caught(monkeypatch):
    """Reference tokens at axis-0 index 0 (the target's positions); the final
    layer applied to the reference tokens instead of the target ones."""
    orig_ids, orig_step = O.rope_ids, O.denoise_step

    def ids_no_index(L_txt, gh, gw, rh=0, rw=0):
        ids = orig_ids(L_txt, gh, gw, rh, rw)
        ids[:, 0] = 0
        return ids

    _planted(monkeypatch, "rope_ids", ids_no_index, test_i2i_step_vs_torch_restatement)
    monkeypatch.setattr(O, "rope_ids", orig_ids)
    sh = SH_I2I
    W, x_lat, x_txt, vec_add = _step_case(sh)
    x_ref = rnd("stp.ref", (sh.B, sh.L_ref, sh.C_lat))
    a = O.denoise_step(x_lat, x_txt, 0.8, 0.7, W, sh, vec_add=vec_add, x_ref=x_ref)
    b = _step_variant(x_lat, x_txt, 0.8, 0.7, W, sh, vec_add, x_ref=x_ref)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])  # the variant without switches is the step

    def planted(*args, **kw):
        return _step_variant(*args, **kw, final_on_ref=True)

    _planted(monkeypatch, "denoise_step", planted, test_i2i_step_vs_torch_restatement)
    monkeypatch.setattr(O, "denoise_step", orig_step)


# ------------------------------------------------------------------ int8 quantiser
def test_quantize_w8_invariants():
    w = S.normal_bf16("q.w", (64, 96), 0.02)
    w[5] = 0.0
    q, s = O.quantize_w8(w)
    assert q.dtype == np.int8 and s.dtype == np.float32
    assert np.abs(q.astype(int)).max() <= 127
    nz = np.abs(w).max(1) > 0
    assert np.all(np.abs(q[nz].astype(int)).max(1) == 127)
    assert s[5] == 1.0 and np.all(q[5] == 0)
    # |w - q s| <= s/2, widened by the float32 rounding of the quotient w/s (|w/s| <= 127)
    assert np.all(np.abs(w - O.dequantize_w8(q, s)) <= s[:, None].astype(np.float64) * (0.5 + 128 * 2.0 ** -24))


def test_quantize_w8_ties_and_float32_decisions():
    w = np.array([[127.0, 63.5, -0.5, 2.5, -2.5, 1.4999999]], dtype=np.float64)
    q, s = O.quantize_w8(w)
    assert s[0] == np.float32(1.0)
    assert q[0].tolist() == [127, 64, 0, 2, -2, 1]


# ------------------------------------------------------------------ planted mistakes
def _planted(monkeypatch, name, fn, test):
    monkeypatch.setattr(O, name, fn)
    with pytest.raises(AssertionError):
        test()


def test_planted_mistakes_are_caught(monkeypatch):
    orig = {n: getattr(O, n) for n in ("attention", "rope_apply", "layer_norm", "gelu_tanh", "modulate", "rms_norm")}

    def att_noscale(q, k, v):
        return orig["attention"](q * math.sqrt(q.shape[-1]), k, v)

    def rope_half(x, c, s):  # rotate-half pairing instead of adjacent pairs
        h = x.shape[-1] // 2
        y = np.empty_like(x)
        y[..., :h] = x[..., :h] * c[:, None] - x[..., h:] * s[:, None]
        y[..., h:] = x[..., :h] * s[:, None] + x[..., h:] * c[:, None]
        return y

    def rope_sign(x, c, s):
        return orig["rope_apply"](x, c, -s)

    def ln_unbiased(x, eps):
        mu = x.mean(-1, keepdims=True)
        return (x - mu) / np.sqrt(x.var(-1, ddof=1, keepdims=True) + eps)

    def gelu_erf(x):
        return 0.5 * x * (1 + np.vectorize(math.erf)(x / math.sqrt(2)))

    def mod_noone(y, shift, scale):
        return y * scale + shift

    def rms_nog(x, g, eps):
        return orig["rms_norm"](x, np.ones_like(g), eps)

    cases = [
        ("attention", att_noscale, test_attention_brute_force),
        ("rope_apply", rope_half, test_rope_matches_complex_multiplication),
        ("rope_apply", rope_sign, test_rope_matches_complex_multiplication),
        ("layer_norm", ln_unbiased, test_layer_norm_moments_and_torch),
        ("gelu_tanh", gelu_erf, test_gelu_tanh),
        ("modulate", mod_noone, test_double_block_vs_torch_restatement),
        ("rms_norm", rms_nog, test_single_block_vs_torch_restatement),
        ("rope_apply", rope_half, test_double_block_vs_torch_restatement),
    ]
    for name, fn, t in cases:
        _planted(monkeypatch, name, fn, t)
        monkeypatch.setattr(O, name, orig[name])


def test_planted_mistakes_in_the_sampling_loop_are_caught(monkeypatch):
    orig_sinus, orig_denoise = O.timestep_sinusoid, O.denoise_step

    def guidance_no_1000(g, w, sh):  # guidance fed to the sinusoid without the x1000 of the timestep
        s = orig_sinus(np.full(sh.B, g), sh.t_dim)
        return O.linear(O.silu(O.linear(s, w["g_w1"], w["g_b1"])), w["g_w2"], w["g_b2"])

    def denoise_reversed(x, xt, s0, s1, W, sh, vec_add=None):  # Euler step with the wrong sign
        return orig_denoise(x, xt, s1, s0, W, sh, vec_add)

    def denoise_drop_vec_add(x, xt, s0, s1, W, sh, vec_add=None):
        return orig_denoise(x, xt, s0, s1, W, sh, None)

    orig_r8 = O.round_e4m3

    def round_e4m3_half_up(x):  # ties away from zero instead of to even
        x = np.asarray(x, np.float64)
        a = np.abs(x)
        e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6.0)
        qn = np.exp2(e - 3.0)
        return np.copysign(np.minimum(np.floor(a / qn + 0.5) * qn, 448.0), x)

    _planted(monkeypatch, "round_e4m3", round_e4m3_half_up, test_round_e4m3_brute_force)
    monkeypatch.setattr(O, "round_e4m3", orig_r8)
    orig_sw = O.swiglu

    def swiglu_swapped(h):
        n = h.shape[-1] // 2
        return O.silu(h[..., n:]) * h[..., :n]

    _planted(monkeypatch, "swiglu", swiglu_swapped, test_swiglu_vs_torch)
    monkeypatch.setattr(O, "swiglu", orig_sw)
    _planted(monkeypatch, "swiglu", swiglu_swapped, lambda: test_swiglu_blocks_vs_torch_restatement("double"))
    monkeypatch.setattr(O, "swiglu", orig_sw)
    orig_g = O.guidance_embed
    _planted(monkeypatch, "guidance_embed", guidance_no_1000, test_conditioning_embeddings_vs_torch)
    monkeypatch.setattr(O, "guidance_embed", orig_g)
    _planted(monkeypatch, "denoise_step", denoise_reversed, test_sample_constant_velocity_closed_form)
    monkeypatch.setattr(O, "denoise_step", orig_denoise)
    _planted(monkeypatch, "denoise_step", denoise_drop_vec_add,
             test_sample_conditioning_acts_only_through_modulation_and_text)
    monkeypatch.setattr(O, "denoise_step", orig_denoise)
