"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA-side tests.

This module holds no arithmetic of the method: it only draws numbers.  Each
tensor is identified by a name; its elements come from a counter-based
generator, so a tensor's values do not depend on which other tensors were
drawn before it, and any element can be regenerated on its own.

Generator (published definitions, restated):
  * SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014): z += 0x9E3779B97F4A7C15; z = (z ^ z>>30) *
    0xBF58476D1CE4E5B9; z = (z ^ z>>27) * 0x94D049BB133111EB; z ^= z>>31.
  * key(name, seed) = SplitMix64(FNV-1a-64(name) ^ SplitMix64(seed)).
  * u_j = ((SplitMix64(key + j) >> 11) + 1) * 2^-53, uniform in (0, 1].
  * Box-Muller (1958): for pair p, r = sqrt(-2 ln u_{2p}), a = 2 pi u_{2p+1};
    element 2p = r cos a, element 2p+1 = r sin a.

Values are drawn in float64 and then rounded to the storage type the kernels
read (bf16 via float32, round-to-nearest-even at each step); both sides of a
parity test consume the same rounded values.
"""
from __future__ import annotations

import numpy as np

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLD = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _splitmix64(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = z + _GOLD
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
        return z ^ (z >> np.uint64(31))


def _fnv1a64(name: str) -> int:
    h = 0xCBF29CE484222325
    for byte in name.encode():
        h ^= byte
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def tensor_key(name: str, seed: int = 0) -> np.uint64:
    s = _splitmix64(np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0]
    return _splitmix64(np.array([np.uint64(_fnv1a64(name)) ^ s], dtype=np.uint64))[0]


def uniform(name: str, n: int, seed: int = 0) -> np.ndarray:
    """n uniforms in (0, 1], float64."""
    key = tensor_key(name, seed)
    out = np.empty(n, dtype=np.float64)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        with np.errstate(over="ignore"):
            ctr = np.arange(lo, hi, dtype=np.uint64) + key
        z = _splitmix64(ctr)
        out[lo:hi] = ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    return out


def normal(name: str, shape, std: float = 1.0, mean: float = 0.0, seed: int = 0) -> np.ndarray:
    """float64 array of the given shape, N(mean, std^2), Box-Muller over uniform()."""
    shape = tuple(int(s) for s in np.atleast_1d(shape)) if not isinstance(shape, tuple) else shape
    n = int(np.prod(shape)) if len(shape) else 1
    npairs = (n + 1) // 2
    out = np.empty(2 * npairs, dtype=np.float64)
    key = tensor_key(name, seed)
    step = _CHUNK // 2
    for p0 in range(0, npairs, step):
        p1 = min(npairs, p0 + step)
        with np.errstate(over="ignore"):
            ctr = np.arange(2 * p0, 2 * p1, dtype=np.uint64) + key
        z = _splitmix64(ctr)
        u = ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        a = 2.0 * np.pi * u2
        out[2 * p0:2 * p1:2] = r * np.cos(a)
        out[2 * p0 + 1:2 * p1:2] = r * np.sin(a)
    return (out[:n] * std + mean).reshape(shape)


# ---------------------------------------------------------------- rounding
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern (uint16), round to nearest even; NaN kept quiet."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounding = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    r = ((u + rounding) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = np.uint16(0x7FC0)
    return r


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Values of x after rounding to float32 and then to bf16, as float64."""
    return bf16_bits_to_f64(f32_to_bf16_bits(np.asarray(x, dtype=np.float64).astype(np.float32)))


def round_f32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def normal_bf16(name: str, shape, std: float = 1.0, mean: float = 0.0, seed: int = 0) -> np.ndarray:
    return round_bf16(normal(name, shape, std, mean, seed))


def normal_f32(name: str, shape, std: float = 1.0, mean: float = 0.0, seed: int = 0) -> np.ndarray:
    return round_f32(normal(name, shape, std, mean, seed))


# ---------------------------------------------------------------- model parameters
# Initialisation recipe: every linear weight and bias N(0, 0.02) rounded to
# bf16 (the kernels' weight type); RMSNorm gains 1 + N(0, 0.02) rounded to
# float32; activations and the conditioning vector N(0, 1).
W_STD = 0.02


def linear_params(prefix: str, n_out: int, n_in: int, seed: int = 0, f32: bool = False):
    """f32: the same draws rounded to float32 instead of bf16 (a float32-weight
    model; the kernels then take bf16 operands of these weights)."""
    r = normal_f32 if f32 else normal_bf16
    return (r(prefix + ".w", (n_out, n_in), W_STD, seed=seed), r(prefix + ".b", (n_out,), W_STD, seed=seed))


def norm_gain(prefix: str, d: int, seed: int = 0):
    return normal_f32(prefix, (d,), W_STD, mean=1.0, seed=seed)


def double_block_params(prefix: str, D: int, d_head: int, D_mlp: int, seed: int = 0, mlp: str = "gelu",
                        f32: bool = False) -> dict:
    """mlp = "swiglu": the first MLP projection has 2 D_mlp output rows [gate; up].
    f32: float32 weights and biases (see linear_params)."""
    n_in = 2 * D_mlp if mlp == "swiglu" else D_mlp
    out = {}
    for s in ("txt", "img"):
        p = f"{prefix}.{s}"
        w = {}
        w["mod_w"], w["mod_b"] = linear_params(p + ".mod", 6 * D, D, seed, f32)
        w["qkv_w"], w["qkv_b"] = linear_params(p + ".qkv", 3 * D, D, seed, f32)
        w["proj_w"], w["proj_b"] = linear_params(p + ".proj", D, D, seed, f32)
        w["mlp_in_w"], w["mlp_in_b"] = linear_params(p + ".mlp_in", n_in, D, seed, f32)
        w["mlp_out_w"], w["mlp_out_b"] = linear_params(p + ".mlp_out", D, D_mlp, seed, f32)
        w["q_norm"] = norm_gain(p + ".q_norm", d_head, seed)
        w["k_norm"] = norm_gain(p + ".k_norm", d_head, seed)
        out[s] = w
    return out


def single_block_params(prefix: str, D: int, d_head: int, D_mlp: int, seed: int = 0, mlp: str = "gelu",
                        f32: bool = False) -> dict:
    """mlp = "swiglu": lin1 has 3 D + 2 D_mlp output rows [q; k; v; gate; up].
    f32: float32 weights and biases (see linear_params)."""
    w = {}
    w["mod_w"], w["mod_b"] = linear_params(prefix + ".mod", 3 * D, D, seed, f32)
    w["lin1_w"], w["lin1_b"] = linear_params(prefix + ".lin1", 3 * D + (2 if mlp == "swiglu" else 1) * D_mlp, D,
                                             seed, f32)
    w["lin2_w"], w["lin2_b"] = linear_params(prefix + ".lin2", D, D + D_mlp, seed, f32)
    w["q_norm"] = norm_gain(prefix + ".q_norm", d_head, seed)
    w["k_norm"] = norm_gain(prefix + ".k_norm", d_head, seed)
    return w


def embed_params(D: int, C_lat: int, t_dim: int = 256, seed: int = 0) -> dict:
    w = {}
    w["t_w1"], w["t_b1"] = linear_params("time_in.lin1", D, t_dim, seed)
    w["t_w2"], w["t_b2"] = linear_params("time_in.lin2", D, D, seed)
    w["img_in_w"], w["img_in_b"] = linear_params("img_in", D, C_lat, seed)
    w["final_mod_w"], w["final_mod_b"] = linear_params("final.mod", 2 * D, D, seed)
    w["final_w"], w["final_b"] = linear_params("final.lin", C_lat, D, seed)
    return w


def cond_params(D: int, t_dim: int, C_txt: int, C_pool: int, seed: int = 0) -> dict:
    """Conditioning layers of the sampling loop: text projection, guidance and
    pooled-text MLPs."""
    w = {}
    w["txt_in_w"], w["txt_in_b"] = linear_params("cond.txt_in", D, C_txt, seed)
    w["g_w1"], w["g_b1"] = linear_params("cond.guid1", D, t_dim, seed)
    w["g_w2"], w["g_b2"] = linear_params("cond.guid2", D, D, seed)
    w["y_w1"], w["y_b1"] = linear_params("cond.vec1", D, C_pool, seed)
    w["y_w2"], w["y_b2"] = linear_params("cond.vec2", D, D, seed)
    return w


def activations(B: int, L_txt: int, L_img: int, D: int, C_lat: int = 0, seed: int = 0) -> dict:
    a = {"vec": normal_f32("vec", (B, D), seed=seed),
         "x_txt": normal_f32("x_txt", (B, L_txt, D), seed=seed),
         "x_img": normal_f32("x_img", (B, L_img, D), seed=seed)}
    if C_lat:
        a["x_lat"] = normal_f32("x_lat", (B, L_img, C_lat), seed=seed)
    return a
