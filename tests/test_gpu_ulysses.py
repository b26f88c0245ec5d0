"""Ulysses sequence parallelism on one GPU: the exchange layout kernels
(mmdit_heads_pack / unpack) bit-exact against the layouts the CPU exchange
test uses, and whole sharded double and single blocks, P virtual ranks with
the exchanges done as copies, against the float64 oracle at the bf16 bar.
Multi-GPU runs of the same schedule are not measured here: every run of
this suite has one GPU."""
import numpy as np
import pytest
import torch

from diffusion_transformer_image_mmdit_gb300 import api, synthetic as S, ulysses as U, weights as Wt
from oracle import mmdit_oracle as O
from tests.gpu_common import api_shape, assert_close, bf16, check_status, f32, gpu_tables, host, need_gpu, oracle_shape, tables
from tests.test_ulysses_cpu import _pack, _unpack

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    need_gpu()
    yield
    check_status()


@pytest.mark.parametrize("rows,P,Dg", [(1, 2, 8), (37, 2, 256), (161, 4, 128), (5, 3, 64)])
def test_heads_pack_unpack_bit_exact(rows, P, Dg):
    x = S.normal_bf16("hp.x", (rows, 3 * P * Dg))
    send = torch.empty((P * rows, 3 * Dg), dtype=torch.bfloat16, device="cuda")
    api.mmdit_heads_pack(bf16(x), 3, P, Dg, send)
    assert np.array_equal(host(send), _pack(x, P, Dg))
    o = S.normal_bf16("hp.o", (P * rows, Dg))
    out = torch.empty((rows, P * Dg), dtype=torch.bfloat16, device="cuda")
    api.mmdit_heads_unpack(bf16(o), P, Dg, out)
    assert np.array_equal(host(out), _unpack(o, P, Dg))


# text and image rows shared unevenly among the ranks (one rank holds both kinds)
SP = {
    2: dict(B=1, L_txt=41, grid_h=10, grid_w=12, D=512, H=4, d_head=128, D_mlp=1024, rope_axes=(16, 56, 56)),
    4: dict(B=1, L_txt=50, grid_h=9, grid_w=13, D=1024, H=8, d_head=128, D_mlp=1024, rope_axes=(16, 56, 56)),
}


@pytest.mark.parametrize("P", [2, 4])
def test_ulysses_double_block_loopback(P):
    cfg = SP[P]
    shape = api_shape(cfg)
    sh = oracle_shape(cfg)
    p = S.double_block_params(f"sp.d{P}", cfg["D"], cfg["d_head"], cfg["D_mlp"])
    a = S.activations(1, cfg["L_txt"], sh.L_img, cfg["D"])
    _, cs, sn = gpu_tables(shape)
    block = U.UlyssesDoubleBlock(shape, Wt.double_from_host(p), P, cs, sn)
    xt, xi = f32(a["x_txt"][0]), f32(a["x_img"][0])
    U.double_block_loopback(block, xt, xi, f32(a["vec"]))
    c, s = tables(cfg)
    rt, ri = O.double_block(a["x_txt"], a["x_img"], a["vec"], p, sh, c, s)
    assert_close(host(xt)[None], rt, what=f"ulysses P={P} double x_txt")
    assert_close(host(xi)[None], ri, what=f"ulysses P={P} double x_img")


@pytest.mark.parametrize("P", [2, 4])
def test_ulysses_single_block_loopback(P):
    cfg = SP[P]
    shape = api_shape(cfg)
    sh = oracle_shape(cfg)
    p = S.single_block_params(f"sp.s{P}", cfg["D"], cfg["d_head"], cfg["D_mlp"])
    x = S.normal_f32("sp.x", (1, sh.L, cfg["D"]))
    vec = S.normal_f32("sp.vec", (1, cfg["D"]))
    _, cs, sn = gpu_tables(shape)
    block = U.UlyssesSingleBlock(shape, Wt.single_from_host(p), P, cs, sn)
    xg = f32(x[0])
    U.single_block_loopback(block, xg, f32(vec))
    c, s = tables(cfg)
    assert_close(host(xg)[None], O.single_block(x, vec, p, sh, c, s), what=f"ulysses P={P} single")
