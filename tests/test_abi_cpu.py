"""Host-side checks that need no GPU: the library builds and loads, exports
every function include/mmdit.h declares, sizes workspaces, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from diffusion_transformer_image_mmdit_gb300 import _lib, build
    build.build()
    return _lib.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "mmdit.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^(?:const\s+)?[A-Za-z_][\w ]*?[\s\*]+([A-Za-z_]\w*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "return")))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("mmdit_double_block_fwd", "mmdit_single_block_fwd", "joint_attention_fwd", "rope2d_apply",
                     "euler_step", "mmdit_rope2d_build", "mmdit_quantize_w8", "mmdit_linear_fwd"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from diffusion_transformer_image_mmdit_gb300 import _lib
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(_declared_functions()) <= set(_lib.SIGNATURES), "binding lacks a declared function"


def test_status_strings(lib):
    assert lib.mmdit_status_string(0) == b"ok"
    assert b"workspace" in lib.mmdit_status_string(-4)


def _shape(**kw):
    from diffusion_transformer_image_mmdit_gb300.api import make_shape
    base = dict(B=1, L_txt=32, grid_h=16, grid_w=16, D=256, H=4, d_head=64, D_mlp=1024, rope_axes=(16, 24, 24))
    base.update(kw)
    return make_shape(**base)


def test_workspace_sizes(lib):
    from diffusion_transformer_image_mmdit_gb300 import api
    s = _shape()
    d = api.workspace_size(s, api.MMDIT_OP_DOUBLE)
    g = api.workspace_size(s, api.MMDIT_OP_SINGLE)
    a = api.workspace_size(s, api.MMDIT_OP_ATTENTION)
    L, D = 288, 256
    assert a >= L * 2 * D * 2 + D * 288 * 2
    assert d > a and g > a
    s8 = _shape(w_dtype=api.MMDIT_I8W)
    assert api.workspace_size(s8, api.MMDIT_OP_SINGLE) >= g + (3 * D + 1024) * D * 2
    st = api.step_workspace_size(s, 2, 3)
    assert st > max(d, g)


@pytest.mark.parametrize("kw", [dict(D=200), dict(d_head=96, H=2, D=192), dict(H=3), dict(rope_axes=(16, 24, 26)),
                                dict(D_mlp=100), dict(B=0), dict(grid_h=0), dict(w_dtype=7)])
def test_bad_shapes_rejected(lib, kw):
    s = _shape(**kw)
    n = ctypes.c_size_t(0)
    assert lib.mmdit_workspace_size(ctypes.byref(s), 1, ctypes.byref(n)) in (-1, -2)


def test_null_and_misaligned_arguments_rejected_before_launch(lib):
    from diffusion_transformer_image_mmdit_gb300 import _lib
    s = _shape()
    assert lib.mmdit_double_block_fwd(ctypes.byref(s), None, None, None, None, None, None, None, None, 0, None) == -1
    assert lib.euler_step(None, None, 1, 1.0, 0.5, 10, None) == -1
    assert lib.euler_step(ctypes.c_void_p(16), ctypes.c_void_p(32), 9, 1.0, 0.5, 10, None) == -1
    assert lib.euler_step(ctypes.c_void_p(18), ctypes.c_void_p(32), 1, 1.0, 0.5, 10, None) == -3
    lin = _lib.Linear(ctypes.c_void_p(64), None, None)
    assert lib.mmdit_linear_fwd(ctypes.byref(lin), 8, 48, 64, ctypes.c_void_p(16), ctypes.c_void_p(32), 0, None, None,
                                0, None) == -2
    assert lib.mmdit_linear_fwd(ctypes.byref(lin), 8, 64, 60, ctypes.c_void_p(16), ctypes.c_void_p(32), 0, None, None,
                                0, None) == -2
    lin8 = _lib.Linear(ctypes.c_void_p(64), None, ctypes.c_void_p(128))
    assert lib.mmdit_linear_fwd(ctypes.byref(lin8), 8, 64, 64, ctypes.c_void_p(16), ctypes.c_void_p(32), 0, None,
                                None, 0, None) == -4
    a = (ctypes.c_void_p * 2)(None, None)
    assert lib.joint_attention_fwd(ctypes.byref(s), ctypes.c_void_p(16), 700, a, a, None, None, ctypes.c_void_p(16),
                                   256, ctypes.c_void_p(16), 1 << 30, None) == -2


def test_ln_modulate_f8_arguments_rejected_before_launch(lib):
    p16 = ctypes.c_void_p(256)
    # codes or scales missing
    assert lib.mmdit_ln_modulate_f8(p16, 1, 4, 256, p16, p16, 768, ctypes.c_float(1e-6), None, None, p16, None) == -1
    assert lib.mmdit_ln_modulate_f8(p16, 1, 4, 256, p16, p16, 768, ctypes.c_float(1e-6), None, p16, None, None) == -1
    # D not a multiple of 256, or above 4096
    assert lib.mmdit_ln_modulate_f8(p16, 1, 4, 384, p16, p16, 768, ctypes.c_float(1e-6), None, p16, p16, None) == -2
    assert lib.mmdit_ln_modulate_f8(p16, 1, 4, 4352, p16, p16, 768, ctypes.c_float(1e-6), None, p16, p16, None) == -2
    # misaligned codes, or a modulation stride that breaks the 16-byte rows
    assert lib.mmdit_ln_modulate_f8(p16, 1, 4, 256, p16, p16, 768, ctypes.c_float(1e-6), None, ctypes.c_void_p(264),
                                    p16, None) == -3
    assert lib.mmdit_ln_modulate_f8(p16, 1, 4, 256, p16, p16, 770, ctypes.c_float(1e-6), None, p16, p16, None) == -3


def test_sample_arguments_rejected_before_launch(lib):
    from diffusion_transformer_image_mmdit_gb300 import _lib
    s = _shape()
    s.C_lat, s.t_dim = 64, 256
    n_big = ctypes.c_size_t(0)
    n_small = ctypes.c_size_t(0)
    assert lib.mmdit_sample_workspace_size(ctypes.byref(s), 1, 1, 128, 28, ctypes.byref(n_big)) == 0
    assert lib.mmdit_sample_workspace_size(ctypes.byref(s), 1, 1, 128, 1, ctypes.byref(n_small)) == 0
    step = ctypes.c_size_t(0)
    assert lib.mmdit_step_workspace_size(ctypes.byref(s), 1, 1, ctypes.byref(step)) == 0
    assert n_big.value >= n_small.value > step.value
    assert lib.mmdit_sample_workspace_size(ctypes.byref(s), 1, 1, 128, 0, ctypes.byref(n_small)) == -1
    w = _lib.StepW()
    sig = (ctypes.c_double * 3)(1.0, 0.5, 0.0)
    p16 = ctypes.c_void_p(256)
    # no conditioning weights
    assert lib.mmdit_sample(ctypes.byref(s), ctypes.byref(w), None, p16, p16, p16, 3.5, sig, 2, 0, p16, 1 << 30,
                            None) == -1
    lin = _lib.Linear(ctypes.c_void_p(512), None, None)
    w.time1 = w.time2 = w.img_in = w.final_mod = w.final = lin
    c = _lib.CondW(lin, lin, lin, lin, lin, 96, 64)  # C_txt not a multiple of 64
    assert lib.mmdit_sample(ctypes.byref(s), ctypes.byref(w), ctypes.byref(c), p16, p16, p16, 3.5, sig, 2, 0, p16,
                            1 << 30, None) == -2
    c.C_txt = 128
    assert lib.mmdit_sample(ctypes.byref(s), ctypes.byref(w), ctypes.byref(c), p16, p16, p16, 3.5, sig, 2, 4, p16,
                            1 << 30, None) == -1  # unknown flag
    assert lib.mmdit_sample(ctypes.byref(s), ctypes.byref(w), ctypes.byref(c), ctypes.c_void_p(260), p16, p16, 3.5,
                            sig, 2, 0, p16, 1 << 30, None) == -3  # misaligned latent
    assert lib.mmdit_sample(ctypes.byref(s), ctypes.byref(w), ctypes.byref(c), p16, p16, p16, 3.5, sig, 2, 0, p16,
                            16, None) == -4  # workspace too small


def test_product_path_has_no_cpu_fallback():
    """The package never imports the oracle; the binding refuses to run without the library."""
    pkg = os.path.join(ROOT, "diffusion_transformer_image_mmdit_gb300")
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            src = open(os.path.join(pkg, f)).read()
            assert not re.search(r"^\s*(import|from)\s+oracle", src, flags=re.M), f
    from diffusion_transformer_image_mmdit_gb300 import _lib
    with pytest.raises(RuntimeError):
        _lib._lib = None
        try:
            _lib.load("/nonexistent/libmmdit.so")
        finally:
            _lib._lib = None
