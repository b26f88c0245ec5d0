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
from tests.gpu_common import CONFIGS, FULL, api_shape, assert_close, bf16, check_status, f32, gpu_tables, host, need_gpu

pytestmark = pytest.mark.gpu


def _inputs(cfg, tag):
    shape = api_shape(cfg)
    B, L, H, d, D = cfg["B"], api.seq_len(shape), cfg["H"], cfg["d_head"], cfg["D"]
    qkv = bf16(S.normal_bf16(f"na.{tag}", (B, L, 3 * D)))
    g = [f32(S.norm_gain(f"na.{tag}.g{i}", d)) for i in range(4)]
    return shape, qkv, [g[0], g[1]], [g[2], g[3]]


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


@pytest.mark.parametrize("name", ["d128", "c1"])
def test_no_alloc_matches_workspace_variant_on_consecutive_calls(name):
    need_gpu()
    cfg = CONFIGS[name]
    for call in range(2):  # the second call runs on scratch the first one left behind
        shape, qkv, qn, kn = _inputs(cfg, f"{name}.{call}")
        _, cs, sn = gpu_tables(shape)
        ref = host(_with_workspace(shape, qkv, qn, kn, cs, sn))
        got = host(_no_alloc(shape, qkv, qn, kn, cs, sn))
        assert_close(got, ref, what=f"no-alloc attention, call {call + 1}")
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
