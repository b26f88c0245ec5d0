"""Shared helpers of the GPU parity tests: configs, device transfer, error
metrics.  The oracle sees exactly the values the kernels read (bf16-rounded
weights, fp32 activations)."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

from diffusion_transformer_image_mmdit_gb300 import api
from oracle import mmdit_oracle as O

# Parity bar for bf16 configs (per block output): relative L2 and max-abs error.
REL_L2 = 1e-2
MAX_ABS = 5e-2
# Int8 weight-only path against the oracle on the original (unquantised) weights.
REL_L2_INT8_SCHEME = 3e-2

CONFIGS = {
    # tiny double-stream block: hidden 256, 4 heads x 64, MLP 1024, 32 text + 16x16 image tokens, axes 16/24/24
    "c1": dict(B=1, L_txt=32, grid_h=16, grid_w=16, D=256, H=4, d_head=64, D_mlp=1024, rope_axes=(16, 24, 24)),
    # head width 128, batch 2, ragged sequence (160 = 1.25 tiles)
    "d128": dict(B=2, L_txt=40, grid_h=10, grid_w=12, D=256, H=2, d_head=128, D_mlp=512, rope_axes=(16, 56, 56)),
    # no text, 63 tokens (under one tile), D = 512
    "ragged": dict(B=1, L_txt=0, grid_h=7, grid_w=9, D=512, H=4, d_head=128, D_mlp=1024, rope_axes=(16, 56, 56)),
    # three tiles plus a tail of 5 queries/keys, D_mlp not a multiple of 256
    "tail": dict(B=1, L_txt=13, grid_h=14, grid_w=24, D=256, H=2, d_head=128, D_mlp=320, rope_axes=(16, 56, 56)),
}
FLUX = dict(D=3072, H=24, d_head=128, D_mlp=12288, rope_axes=(16, 56, 56))
FULL = {
    # Flux-shaped double block at 512^2: 512 text + 32x32 image tokens
    "c2": dict(B=1, L_txt=512, grid_h=32, grid_w=32, **FLUX),
    # Flux-shaped blocks at 1024^2: 512 text + 64x64 image tokens
    "c3": dict(B=1, L_txt=512, grid_h=64, grid_w=64, **FLUX),
    # 1328^2: 512 text + 83x83 image tokens
    "c4": dict(B=1, L_txt=512, grid_h=83, grid_w=83, **FLUX),
}


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def api_shape(cfg: dict, **kw) -> api.Shape:
    c = dict(cfg)
    c.update(kw)
    return api.make_shape(**c)


def oracle_shape(cfg: dict) -> O.Shape:
    return O.Shape(B=cfg["B"], L_txt=cfg["L_txt"], grid_h=cfg["grid_h"], grid_w=cfg["grid_w"], D=cfg["D"], H=cfg["H"],
                   d_head=cfg["d_head"], D_mlp=cfg["D_mlp"], rope_axes=tuple(cfg["rope_axes"]),
                   ref_h=cfg.get("ref_h", 0), ref_w=cfg.get("ref_w", 0))


def f32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def bf16(a) -> torch.Tensor:
    return f32(a).to(torch.bfloat16)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_l2(a, b) -> float:
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def report(line: str) -> None:
    """Prints a measured parity figure (shown by pytest for failures, or with
    -rP) and appends it to the file named by MMDIT_PARITY_LOG when set."""
    print(line)
    path = os.environ.get("MMDIT_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")


def assert_close(gpu, ref, rel=REL_L2, max_abs=MAX_ABS, what=""):
    r = rel_l2(gpu, ref)
    m = float(np.abs(np.asarray(gpu, np.float64) - np.asarray(ref, np.float64)).max()) if np.size(ref) else 0.0
    report(f"PARITY {what}: rel_l2={r:.3e} (bar {rel:.3g}) max_abs={m:.3e} (bar {max_abs:.3g})")
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    assert r <= rel and m <= max_abs, f"{what}: rel_l2={r:.3e} (<= {rel}) max_abs={m:.3e} (<= {max_abs})"
    return r, m


def tables(cfg):
    ids = O.rope_ids(cfg["L_txt"], cfg["grid_h"], cfg["grid_w"], cfg.get("ref_h", 0), cfg.get("ref_w", 0))
    return O.rope_tables(ids, tuple(cfg["rope_axes"]), 10000.0)


def gpu_tables(shape: api.Shape):
    L = api.seq_len(shape)
    half = shape.d_head // 2
    ids = torch.empty((L, 3), dtype=torch.int32, device="cuda")
    cs = torch.empty((L, half), dtype=torch.float32, device="cuda")
    sn = torch.empty((L, half), dtype=torch.float32, device="cuda")
    api.mmdit_rope2d_build(shape, ids, cs, sn)
    return ids, cs, sn


def check_status():
    assert api.sync_status() == 0, "a kernel reported a timeout"
