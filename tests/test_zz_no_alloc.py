"""joint_attention_fwd_noalloc, the attention entry point for callers that
cannot allocate device memory (for example a plugin whose host application
owns every device allocation): it must give what joint_attention_fwd gives
with a caller workspace, call after call, while using only the library's
fixed device scratch.  Collected last on purpose (file name), and written
to pass both alone in a fresh process and after the other GPU tests."""
import numpy as np
import pytest
import torch

from diffusion_transformer_image_mmdit_gb300 import _lib, api, synthetic as S
from oracle import mmdit_oracle as O
from tests.gpu_common import (CONFIGS, FULL, api_shape, assert_close, bf16, check_status, f32, gpu_tables, host, need_gpu,
                              tables)

pytestmark = pytest.mark.gpu


def _inputs(cfg, tag):
    shape = api_shape(cfg)
    B, L, H, d, D = cfg["B"], api.seq_len(shape), cfg["H"], cfg["d_head"], cfg["D"]
    qkv_h = S.normal_bf16(f"na.{tag}", (B, L, 3 * D))
    g_h = [S.norm_gain(f"na.{tag}.g{i}", d) for i in range(4)]
    return shape, bf16(qkv_h), [f32(g_h[0]), f32(g_h[1])], [f32(g_h[2]), f32(g_h[3])], qkv_h, g_h


def _oracle(cfg, qkv_h, g):
    """The float64 oracle of the same attention: per-stream RMSNorm of q and
    k (text gains for the first L_txt tokens), RoPE, softmax attention."""
    B, H, d, D, Lt = cfg["B"], cfg["H"], cfg["d_head"], cfg["D"], cfg["L_txt"]
    L = qkv_h.shape[1]
    x = qkv_h.reshape(B, L, 3, H, d)
    q, k, v = x[:, :, 0], x[:, :, 1], x[:, :, 2]
    q = np.concatenate([O.rms_norm(q[:, :Lt], g[0], 1e-6), O.rms_norm(q[:, Lt:], g[1], 1e-6)], axis=1)
    k = np.concatenate([O.rms_norm(k[:, :Lt], g[2], 1e-6), O.rms_norm(k[:, Lt:], g[3], 1e-6)], axis=1)
    c, s = tables(cfg)
    return O.attention(O.rope_apply(q, c, s), O.rope_apply(k, c, s), v).reshape(B, L, D)


def _with_workspace(shape, qkv, qn, kn, cs, sn):
    D = shape.D
    out = torch.empty((shape.B, api.seq_len(shape), D), dtype=torch.bfloat16, device="cuda")
    ws = api.alloc_workspace(api.workspace_size(shape, api.MMDIT_OP_ATTENTION))
    api.joint_attention_fwd(shape, qkv, 3 * D, qn, kn, cs, sn, out, D, ws)
    return out


def _no_alloc(shape, qkv, qn, kn, cs, sn):
    D = shape.D
    out = torch.empty((shape.B, api.seq_len(shape), D), dtype=torch.bfloat16, device="cuda")
    api.joint_attention_fwd_noalloc(shape, qkv, 3 * D, qn, kn, cs, sn, out, D)
    return out


NO_ALLOC_CASES = {"d128": CONFIGS["d128"], "c1": CONFIGS["c1"],
                  # image-to-image: reference latent tokens after the target tokens
                  "d128_ref": dict(CONFIGS["d128"], ref_h=3, ref_w=7)}


@pytest.mark.parametrize("name", list(NO_ALLOC_CASES))
def test_no_alloc_matches_workspace_variant_on_consecutive_calls(name):
    """Both variants run the same kernels on the same inputs (at these sizes,
    at most one attention unit per SM, neither splits a unit), so their
    outputs must be identical bit for bit; each is also checked against the
    oracle at the bf16 bar."""
    need_gpu()
    cfg = NO_ALLOC_CASES[name]
    for call in range(2):  # the second call runs on scratch the first one left behind
        shape, qkv, qn, kn, qkv_h, g_h = _inputs(cfg, f"{name}.{call}")
        _, cs, sn = gpu_tables(shape)
        ref = host(_with_workspace(shape, qkv, qn, kn, cs, sn))
        got = host(_no_alloc(shape, qkv, qn, kn, cs, sn))
        assert np.array_equal(got, ref), f"no-alloc attention differs from the workspace variant, call {call + 1}"
        assert_close(got, _oracle(cfg, qkv_h, g_h), what=f"no-alloc attention vs oracle, call {call + 1}")
    check_status()


def test_no_alloc_more_units_than_sms():
    """160 attention units (pairs of query tiles x heads), more than the
    152 SMs: the no-alloc variant runs them as whole units in two rounds,
    the workspace variant balances them by splitting units, so the two are
    each checked against the oracle rather than against one another."""
    need_gpu()
    cfg = dict(B=1, L_txt=64, grid_h=32, grid_w=32, D=4096, H=32, d_head=128, D_mlp=4096, rope_axes=(16, 56, 56))
    shape, qkv, qn, kn, qkv_h, g_h = _inputs(cfg, "units160")
    _, cs, sn = gpu_tables(shape)
    ref = _oracle(cfg, qkv_h, g_h)
    assert_close(host(_no_alloc(shape, qkv, qn, kn, cs, sn)), ref, what="no-alloc attention, 160 units")
    assert_close(host(_with_workspace(shape, qkv, qn, kn, cs, sn)), ref, what="workspace attention, 160 units")
    check_status()


def test_no_alloc_rejects_shapes_beyond_its_scratch():
    need_gpu()
    shape = api_shape(FULL["c3"])  # needs about 85 MB of scratch, more than the fixed 48 MiB
    D = shape.D
    qkv = torch.zeros((1, 8, 3 * D), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((1, 8, D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.MMDiTError) as e:
        api.joint_attention_fwd_noalloc(shape, qkv, 3 * D, None, None, None, None, out, D)
    assert e.value.status == -4
    assert torch.count_nonzero(out).item() == 0
    check_status()
