"""Plain float64 CPU oracle for one Flux-style MMDiT denoising step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests, the smoke check and the CPU-baseline leg of the benchmark do.
It shares no code with the CUDA library; it reads plain numpy arrays.

Sources.  The pages never print the block equations; the operations below are
the primitive definitions the Luminal blog post "Reducing image generation
cost with ..." gives in its section "What the compiler found on its own"
(matmul = broadcast-multiply then sum; attention = scores, scale, max, exp,
sum, divide; RMSNorm = square, sum, reciprocal square root, multiply;
LayerNorm adds a mean and a subtract; adaLN modulation = a scale and a shift;
RoPE = partner gather and multiply-add against cosine and sine tables; fused
elementwise = gate-and-residual add, concatenation of the text and image
streams, timestep embedding), the block counts and widths of its section
"Flux.2 Klein 9B" (double-stream and single-stream blocks, latent patches with
128 channels), and the Euler sampler of its section "The AMD MI300X pipeline".
Where the pages leave a step open, the reading taken is stated at the
function and collected in the design notes (RoPE pairing and frequencies,
chunk order, epsilons, shift schedule, quantiser).

Every function computes its plain definition in float64 with no tiling,
fusion or reordering: attention builds the full score matrix per head and
normalises it with a max-subtracted softmax.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np


# --------------------------------------------------------------------------
# shapes
@dataclass
class Shape:
    B: int
    L_txt: int
    grid_h: int
    grid_w: int
    D: int
    H: int
    d_head: int
    D_mlp: int
    rope_axes: tuple = (16, 56, 56)
    rope_theta: float = 10000.0
    eps_ln: float = 1e-6
    eps_rms: float = 1e-6
    C_lat: int = 128
    t_dim: int = 256
    n_double: int = 1
    n_single: int = 0
    mlp: str = "gelu"  # "gelu": GELU-tanh MLP; "swiglu": SiLU(gate) * up over [gate; up] projections
    ref_h: int = 0  # reference latent grid (image-to-image), 0 = none
    ref_w: int = 0

    @property
    def L_gen(self) -> int:
        """Target image tokens (the latent being denoised)."""
        return self.grid_h * self.grid_w

    @property
    def L_ref(self) -> int:
        return self.ref_h * self.ref_w

    @property
    def L_img(self) -> int:
        """All image-stream tokens: target, then reference."""
        return self.L_gen + self.L_ref

    @property
    def L(self) -> int:
        return self.L_txt + self.L_img


# --------------------------------------------------------------------------
# elementwise and row operations
def linear(x, w, b=None):
    """y = x W^T + b (matmul spelled as multiply-and-sum; a library matmul
    serves as the step)."""
    y = np.asarray(x, np.float64) @ np.asarray(w, np.float64).T
    if b is not None:
        y = y + b
    return y


def silu(x):
    return x / (1.0 + np.exp(-x))


def gelu_tanh(x):
    """GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))."""
    return 0.5 * x * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x ** 3)))


def layer_norm(x, eps):
    """LayerNorm without affine: subtract the row mean, divide by
    sqrt(biased variance + eps)."""
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps)


def swiglu(h):
    """SwiGLU over the last axis of h = [gate | up] (two halves): SiLU(gate) * up.
    The Luminal blog (section "What the compiler found on its own") lists the
    SwiGLU activation among the fused elementwise kernels of a Flux.2 Klein
    step; the [gate; up] order of the projection's output rows is the reading
    taken."""
    n = h.shape[-1] // 2
    return silu(h[..., :n]) * h[..., n:]


def mlp_act(h, sh):
    """The MLP activation of the model: GELU-tanh, or SwiGLU (which halves the
    width)."""
    return swiglu(h) if sh.mlp == "swiglu" else gelu_tanh(h)


def modulate(y, shift, scale):
    """adaLN modulation: a scale and a shift, y (1 + scale) + shift."""
    return y * (1.0 + scale) + shift


def rms_norm(x, g, eps):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * g."""
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * g


# --------------------------------------------------------------------------
# 2D axial RoPE
def rope_ids(L_txt: int, grid_h: int, grid_w: int, ref_h: int = 0, ref_w: int = 0) -> np.ndarray:
    """Position ids [L, 3] (int32).  Text tokens sit at (0, 0, 0); the image
    token at latent row h, column w (row-major after the text) sits at
    (0, h, w).

    Reference latent (image-to-image): the Luminal blog (section "The AMD
    MI300X pipeline") appends the once-computed reference latent to the noise
    tokens; no page gives its positions.  Reading taken: its ref_h x ref_w
    tokens follow the target tokens, row-major, at (1, h, w), so they keep
    their own 2D grid and differ from the target only on the first axis."""
    L_gen, L_ref = grid_h * grid_w, ref_h * ref_w
    ids = np.zeros((L_txt + L_gen + L_ref, 3), dtype=np.int32)
    hh, ww = np.meshgrid(np.arange(grid_h), np.arange(grid_w), indexing="ij")
    ids[L_txt:L_txt + L_gen, 1] = hh.reshape(-1)
    ids[L_txt:L_txt + L_gen, 2] = ww.reshape(-1)
    if L_ref:
        rh, rw = np.meshgrid(np.arange(ref_h), np.arange(ref_w), indexing="ij")
        ids[L_txt + L_gen:, 0] = 1
        ids[L_txt + L_gen:, 1] = rh.reshape(-1)
        ids[L_txt + L_gen:, 2] = rw.reshape(-1)
    return ids


def rope_angles(ids: np.ndarray, axes, theta: float) -> np.ndarray:
    """Angle per (token, channel pair) [L, sum(axes)/2], float64.
    Axis a owns axes[a]/2 consecutive pairs; pair i of axis a turns at
    frequency theta^(-2i/axes[a]) times the token's coordinate on that axis."""
    cols = []
    for a, d_a in enumerate(axes):
        i = np.arange(d_a // 2, dtype=np.float64)
        omega = theta ** (-2.0 * i / d_a)
        cols.append(ids[:, a:a + 1].astype(np.float64) * omega[None, :])
    return np.concatenate(cols, axis=1)


def rope_tables(ids, axes, theta):
    """cos and sin tables [L, d/2] in float64."""
    ang = rope_angles(ids, axes, theta)
    return np.cos(ang), np.sin(ang)


def rope_apply(x, cos, sin):
    """Rotate each channel pair (2i, 2i+1) of x [..., L, H, d] by the token's
    angle: (x0, x1) -> (x0 c - x1 s, x0 s + x1 c).  cos/sin are [L, d/2]."""
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    c = cos[:, None, :]
    s = sin[:, None, :]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


# --------------------------------------------------------------------------
# attention
def attention(q, k, v, rnd=None):
    """Softmax attention per sample and head with no mask.
    q [B, Lq, H, d], k, v [B, Lk, H, d] -> [B, Lq, H, d].
    Scores = q k^T / sqrt(d); subtract the row max; exponentiate; divide by
    the row sum; weight v.

    rnd (optional, precision model only): applied to the exponentials that
    weight v, while the row sum keeps them unrounded."""
    B, Lq, H, d = q.shape
    out = np.empty((B, Lq, H, d))
    for b in range(B):
        for h in range(H):
            s = q[b, :, h, :] @ k[b, :, h, :].T / math.sqrt(d)
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            if rnd is None:
                p = p / p.sum(axis=1, keepdims=True)
                out[b, :, h, :] = p @ v[b, :, h, :]
            else:
                out[b, :, h, :] = (rnd(p) @ v[b, :, h, :]) / p.sum(axis=1, keepdims=True)
    return out


# --------------------------------------------------------------------------
# blocks
def modulation(vec, w, b, n_chunks):
    """Linear(SiLU(vec)) split into n_chunks rows of width D, each [B, 1, D],
    in the order (shift, scale, gate[, shift2, scale2, gate2])."""
    m = linear(silu(vec), w, b)
    D = m.shape[-1] // n_chunks
    return [m[:, None, i * D:(i + 1) * D] for i in range(n_chunks)]


def _heads(x, H):
    B, L, D = x.shape
    return x.reshape(B, L, H, D // H)


def _ident(x):
    return x


def double_block(x_txt, x_img, vec, wt, sh: Shape, cos, sin, rows_txt=None, rows_img=None, rnd=None, qin=None):
    """Double-stream block.  x_txt [B, L_txt, D], x_img [B, L_img, D], vec
    [B, D]; wt['txt'] / wt['img'] hold each stream's weights.  Per stream:
    adaLN-Zero modulation from vec, LN+modulate, QKV linear, per-head RMSNorm
    of q and k; then RoPE on the concatenated [text; image] sequence and one
    joint softmax attention; per stream: output projection with gated
    residual, LN+modulate, MLP (GELU-tanh, or SwiGLU when sh.mlp is
    "swiglu") with gated residual.

    rows_txt / rows_img (optional index arrays) restrict the outputs to those
    query rows; keys and values always cover the whole sequence.

    rnd (optional) is a precision model, not part of the definition: when
    given, it is applied where a bf16 implementation stores a matmul operand
    (LN+modulate outputs, q/k after RoPE, v, softmax weights, attention
    output, MLP hidden).  Left as None the block is the plain definition.

    qin (optional) is a quantisation model of the inputs of the four GEMM
    linears (QKV, projection, both MLP projections), e.g. e4m3 rows; None
    leaves them exact."""
    R = _ident if rnd is None else rnd
    Q = _ident if qin is None else qin
    H = sh.H
    streams = (("txt", x_txt, rows_txt, 0), ("img", x_img, rows_img, sh.L_txt))
    qs, ks, vs, mods = [], [], [], {}
    for name, x, _, _ in streams:
        w = wt[name]
        sh1, sc1, g1, sh2, sc2, g2 = modulation(vec, w["mod_w"], w["mod_b"], 6)
        mods[name] = (sh1, sc1, g1, sh2, sc2, g2)
        y = R(modulate(layer_norm(x, sh.eps_ln), sh1, sc1))
        qkv = linear(Q(y), w["qkv_w"], w["qkv_b"])
        D = sh.D
        q = rms_norm(_heads(qkv[..., :D], H), w["q_norm"], sh.eps_rms)
        k = rms_norm(_heads(qkv[..., D:2 * D], H), w["k_norm"], sh.eps_rms)
        v = R(_heads(qkv[..., 2 * D:], H))
        qs.append(q), ks.append(k), vs.append(v)
    q = R(rope_apply(np.concatenate(qs, axis=1), cos, sin))
    k = R(rope_apply(np.concatenate(ks, axis=1), cos, sin))
    v = np.concatenate(vs, axis=1)
    outs = []
    for name, x, rows, off in streams:
        w = wt[name]
        sh1, sc1, g1, sh2, sc2, g2 = mods[name]
        idx = np.arange(x.shape[1]) if rows is None else np.asarray(rows)
        o = R(attention(q[:, off + idx], k, v, rnd).reshape(x.shape[0], len(idx), sh.D))
        xr = x[:, idx] + g1 * linear(Q(o), w["proj_w"], w["proj_b"])
        y2 = R(modulate(layer_norm(xr, sh.eps_ln), sh2, sc2))
        hid = R(mlp_act(linear(Q(y2), w["mlp_in_w"], w["mlp_in_b"]), sh))
        xr = xr + g2 * linear(Q(hid), w["mlp_out_w"], w["mlp_out_b"])
        outs.append(xr)
    return outs[0], outs[1]


def single_block(x, vec, w, sh: Shape, cos, sin, rows=None, rnd=None, qin=None):
    """Single-stream block on x = [text; image] [B, L, D]: LN+modulate, one
    linear D -> 3D + D_mlp (3D + 2 D_mlp with SwiGLU), RMSNorm of q and k,
    RoPE, joint attention in parallel with the MLP activation on the MLP
    columns, one linear over the concatenation [attention output | act(mlp)],
    gated residual.
    rnd: optional precision model, as in double_block."""
    Q = _ident if qin is None else qin  # quantisation model of the lin1 and lin2 inputs, as in double_block
    R = _ident if rnd is None else rnd
    D, H = sh.D, sh.H
    shift, scale, gate = modulation(vec, w["mod_w"], w["mod_b"], 3)
    y = R(modulate(layer_norm(x, sh.eps_ln), shift, scale))
    h = linear(Q(y), w["lin1_w"], w["lin1_b"])
    q = R(rope_apply(rms_norm(_heads(h[..., :D], H), w["q_norm"], sh.eps_rms), cos, sin))
    k = R(rope_apply(rms_norm(_heads(h[..., D:2 * D], H), w["k_norm"], sh.eps_rms), cos, sin))
    v = R(_heads(h[..., 2 * D:3 * D], H))
    idx = np.arange(x.shape[1]) if rows is None else np.asarray(rows)
    o = R(attention(q[:, idx], k, v, rnd).reshape(x.shape[0], len(idx), D))
    cat = np.concatenate([o, R(mlp_act(h[:, idx, 3 * D:], sh))], axis=-1)
    return x[:, idx] + gate * linear(Q(cat), w["lin2_w"], w["lin2_b"])


# --------------------------------------------------------------------------
# timestep embedding, input/output layers, sampler
def timestep_sinusoid(t, dim=256, max_period=10000.0):
    """[cos(t f_j) | sin(t f_j)], f_j = max_period^(-j/(dim/2)), j < dim/2.
    t is the model timestep 1000 * sigma, one value per sample."""
    t = np.atleast_1d(np.asarray(t, np.float64))
    half = dim // 2
    f = np.exp(-math.log(max_period) * np.arange(half) / half)
    a = t[:, None] * f[None, :]
    return np.concatenate([np.cos(a), np.sin(a)], axis=1)


def time_embed(sigma, w, sh: Shape):
    """vec = W_b SiLU(W_a sinusoid(1000 sigma) + b_a) + b_b, [B, D]."""
    s = timestep_sinusoid(np.full(sh.B, 1000.0 * sigma), sh.t_dim)
    return linear(silu(linear(s, w["t_w1"], w["t_b1"])), w["t_w2"], w["t_b2"])


def img_in(x_lat, w):
    """Patch-token projection C_lat -> D."""
    return linear(x_lat, w["img_in_w"], w["img_in_b"])


def final_layer(x_img, vec, w, sh: Shape):
    """LN + modulate (shift, scale) from vec, then linear D -> C_lat."""
    shift, scale = modulation(vec, w["final_mod_w"], w["final_mod_b"], 2)
    return linear(modulate(layer_norm(x_img, sh.eps_ln), shift, scale), w["final_w"], w["final_b"])


def shift_mu(L_img: int) -> float:
    """Shift parameter, linear in the image-token count through (256, 0.5)
    and (4096, 1.15)."""
    return 0.5 + (L_img - 256) * (1.15 - 0.5) / (4096 - 256)


def sigma_schedule(n_steps: int, mu: float) -> np.ndarray:
    """sigma_i = s t_i / (1 + (s - 1) t_i), t_i = 1 - i/n, s = e^mu, i = 0..n."""
    t = 1.0 - np.arange(n_steps + 1, dtype=np.float64) / n_steps
    s = math.exp(mu)
    return s * t / (1.0 + (s - 1.0) * t)


def euler_step(x, v, sigma, sigma_next):
    """Flow-matching Euler update x + (sigma_next - sigma) v."""
    return x + (sigma_next - sigma) * v


def denoise_step(x_lat, x_txt, sigma, sigma_next, W, sh: Shape, vec_add=None, rnd=None, qin=None, x_ref=None):
    """One full step: timestep embedding, img_in, the double blocks, the
    single blocks on [text; image], the final layer on the image tokens, the
    Euler update.  vec_add ([B, D] or None) is added to the timestep
    embedding (the step-independent conditioning of the sampling loop).
    rnd and qin are handed to every block unchanged (precision and
    activation-quantisation models, see double_block); None leaves the
    plain definition.
    x_ref ([B, ref_h ref_w, C_lat], with sh.ref_h, sh.ref_w set): the
    reference latent, projected by img_in like the noise latent and appended
    to its tokens (positions: see rope_ids); the final layer and the Euler
    update see the target tokens only.
    Returns (x_lat_next, v)."""
    ids = rope_ids(sh.L_txt, sh.grid_h, sh.grid_w, sh.ref_h, sh.ref_w)
    cos, sin = rope_tables(ids, sh.rope_axes, sh.rope_theta)
    vec = time_embed(sigma, W, sh)
    if vec_add is not None:
        vec = vec + vec_add
    assert (x_ref is None) == (sh.L_ref == 0), "x_ref is given exactly when the shape has a reference grid"
    h_img = img_in(x_lat if x_ref is None else np.concatenate([x_lat, x_ref], axis=1), W)
    h_txt = x_txt
    for blk in W["double"]:
        h_txt, h_img = double_block(h_txt, h_img, vec, blk, sh, cos, sin, rnd=rnd, qin=qin)
    x = np.concatenate([h_txt, h_img], axis=1)
    for blk in W["single"]:
        x = single_block(x, vec, blk, sh, cos, sin, rnd=rnd, qin=qin)
    v = final_layer(x[:, sh.L_txt:sh.L_txt + sh.L_gen], vec, W, sh)
    return euler_step(x_lat, v, sigma, sigma_next), v


# --------------------------------------------------------------------------
# conditioning and the sampling loop
#
# The pages name the pieces around the denoiser without defining them: a text
# encoder produces the conditioning embeddings that the DiT denoises against
# over 20-50 steps (SGLang blog, "Architecture"), and FLUX.1-dev is sampled
# with 28 steps at guidance 3.5 (flux-amd-rocm benchmark notes).  Readings
# taken, the plainest that fit: the text-encoder output enters through one
# linear projection to width D; the guidance scale goes through the same
# sinusoid (of 1000 g) and two-layer SiLU MLP shape as the timestep; the
# pooled text vector through a two-layer SiLU MLP; both are added to the
# timestep embedding, and neither depends on the step.
def txt_in(txt, w):
    """Text-token projection C_txt -> D: x_txt = txt W^T + b."""
    return linear(txt, w["txt_in_w"], w["txt_in_b"])


def guidance_embed(guidance, w, sh: Shape):
    """W_b SiLU(W_a sinusoid(1000 g) + b_a) + b_b, [B, D]."""
    s = timestep_sinusoid(np.full(sh.B, 1000.0 * guidance), sh.t_dim)
    return linear(silu(linear(s, w["g_w1"], w["g_b1"])), w["g_w2"], w["g_b2"])


def pooled_embed(pooled, w):
    """W_b SiLU(W_a y + b_a) + b_b on the pooled text vector y [B, C_pool]."""
    return linear(silu(linear(pooled, w["y_w1"], w["y_b1"])), w["y_w2"], w["y_b2"])


def sample(x_lat, txt, pooled, guidance, sigmas, W, sh: Shape):
    """The sampling loop over the schedule sigmas[0..n]: the text stream
    x_txt = txt_in(txt) and the conditioning vec_cond = guidance_embed(g) +
    pooled_embed(y) are formed once; step i runs denoise_step with sigma_i,
    sigma_{i+1} and vec_add = vec_cond.  Returns the final latent."""
    x_txt = txt_in(txt, W)
    vec_cond = guidance_embed(guidance, W, sh) + pooled_embed(pooled, W)
    x = np.asarray(x_lat, np.float64)
    for i in range(len(sigmas) - 1):
        x, _ = denoise_step(x, x_txt, sigmas[i], sigmas[i + 1], W, sh, vec_add=vec_cond)
    return x


# --------------------------------------------------------------------------
# int8 weight-only quantiser (decisions taken in float32 arithmetic)
def quantize_w8(w):
    """Per output channel n: s_n = max_k |w_nk| / 127 (float32; s_n = 1 for an
    all-zero row); q = clamp(rint(w / s_n), -127, 127), ties to even, with the
    division in float32.  Returns (q int8 [N, K], s float32 [N])."""
    w32 = np.asarray(w, dtype=np.float32)
    amax = np.abs(w32).max(axis=1)
    s = (amax / np.float32(127.0)).astype(np.float32)
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    r = np.rint((w32 / s[:, None]).astype(np.float32))
    q = np.clip(r, -127, 127).astype(np.int8)
    return q, s


def dequantize_w8(q, s):
    return q.astype(np.float64) * s.astype(np.float64)[:, None]


# --------------------------------------------------------------------------
# FP8 (e4m3) rows: the SGLang blog ("Architecture") names FP8 quantisation
# for serving; the scheme is not given.  Reading taken: each row (a weight's
# output channel, or an activation row) is scaled by s = max|row| / 448
# (float32; 1 for an all-zero row) and rounded to the nearest e4m3 value,
# ties to even, saturating at +-448; the product of two such rows is
# (q_x s_x) . (q_w s_w).
E4M3_MAX = 448.0


def round_e4m3(x):
    """Nearest e4m3 value (1 sign, 4 exponent bits with bias 7, 3 mantissa
    bits, no infinities; smallest normal 2^-6, subnormal step 2^-9), ties to
    even, magnitudes beyond 448 saturated to 448."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    quantum = np.exp2(e - 3.0)
    r = np.rint(a / quantum) * quantum
    r = np.minimum(r, E4M3_MAX)
    return np.where(a > 0, np.copysign(r, x), 0.0 * x)


def quantize_f8_rows(x):
    """Per row of x [..., K]: s = max|row| / 448 in float32 (1 for a zero
    row); q = round_e4m3(x / s) with the quotient in float32.  Returns
    (q float64 holding e4m3 values, s float32 [...])."""
    x32 = np.asarray(x, np.float32)
    amax = np.abs(x32).max(axis=-1)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    q = round_e4m3((x32 / s[..., None]).astype(np.float32))
    return q, s


def dequantize_f8_rows(q, s):
    return np.asarray(q, np.float64) * np.asarray(s, np.float64)[..., None]
