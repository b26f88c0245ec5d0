"""Thin torch-facing binding of the C ABI: same entry-point names, tensors in.

Argument marshalling only: every step runs in the CUDA kernels of
libmmdit.so.  Tensors must already be on the GPU, contiguous, in the dtypes
the C header states; device memory and streams come from PyTorch.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

from . import _lib
from ._lib import (MMDIT_BF16, MMDIT_EPI_BF16, MMDIT_EPI_BF16_GELU, MMDIT_EPI_F32, MMDIT_EPI_RESID, MMDIT_F32,
                   MMDIT_I8W, MMDIT_F8W, MMDIT_OP_ATTENTION, MMDIT_OP_DOUBLE, MMDIT_OP_SINGLE, DoubleW, Linear, Shape, SingleW,
                   StepW, CondW, MMDIT_SAMPLE_GRAPH, MMDIT_EPI_SWIGLU, MMDIT_MLP_GELU, MMDIT_MLP_SWIGLU, call)


# ------------------------------------------------------------------ marshalling helpers
def ptr(t: Optional[torch.Tensor], strided_ok: bool = False):
    """Device address of a tensor (None -> NULL).  Views with gaps are only
    accepted where the C ABI takes an explicit stride."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on the GPU")
    if not strided_ok and not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def stream_handle(stream: Optional[torch.cuda.Stream] = None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_shape(B, L_txt, grid_h, grid_w, D, H, d_head, D_mlp, rope_axes=(16, 56, 56), rope_theta=10000.0,
               eps_ln=1e-6, eps_rms=1e-6, w_dtype=MMDIT_BF16, C_lat=128, t_dim=256, mlp_act=0, ref_h=0,
               ref_w=0) -> Shape:
    s = Shape()
    s.B, s.L_txt, s.grid_h, s.grid_w = B, L_txt, grid_h, grid_w
    s.D, s.H, s.d_head, s.D_mlp = D, H, d_head, D_mlp
    s.rope_axes[0], s.rope_axes[1], s.rope_axes[2] = rope_axes
    s.rope_theta, s.eps_ln, s.eps_rms = rope_theta, eps_ln, eps_rms
    s.w_dtype, s.C_lat, s.t_dim = w_dtype, C_lat, t_dim
    s.mlp_act = mlp_act
    s.ref_h, s.ref_w = ref_h, ref_w
    return s


def seq_len(s: Shape) -> int:
    """Tokens per sample: text, target image, reference image."""
    return s.L_txt + s.grid_h * s.grid_w + s.ref_h * s.ref_w


# ------------------------------------------------------------------ weights on the device
@dataclass
class LinearDev:
    w: torch.Tensor                    # bf16 [N, K] or int8 [N, K]
    b: Optional[torch.Tensor] = None   # fp32 [N]
    scale: Optional[torch.Tensor] = None  # fp32 [N] for int8

    def struct(self) -> Linear:
        return Linear(ptr(self.w), ptr(self.b), ptr(self.scale))

    @property
    def N(self) -> int:
        return self.w.shape[0]

    @property
    def K(self) -> int:
        return self.w.shape[1]


def quantize_linear(lin: LinearDev, stream=None) -> LinearDev:
    """int8 per-channel copy of a bf16 linear, quantised on the GPU."""
    N, K = lin.w.shape
    q = torch.empty((N, K), dtype=torch.int8, device=lin.w.device)
    s = torch.empty((N,), dtype=torch.float32, device=lin.w.device)
    mmdit_quantize_w8(lin.w, q, s, stream)
    return LinearDev(q, lin.b, s)


@dataclass
class DoubleWeights:
    mod: List[LinearDev]
    qkv: List[LinearDev]
    proj: List[LinearDev]
    mlp_in: List[LinearDev]
    mlp_out: List[LinearDev]
    q_norm: List[torch.Tensor]
    k_norm: List[torch.Tensor]

    def struct(self) -> DoubleW:
        s = DoubleW()
        for i in range(2):
            s.mod[i] = self.mod[i].struct()
            s.qkv[i] = self.qkv[i].struct()
            s.proj[i] = self.proj[i].struct()
            s.mlp_in[i] = self.mlp_in[i].struct()
            s.mlp_out[i] = self.mlp_out[i].struct()
            s.q_norm[i] = ptr(self.q_norm[i])
            s.k_norm[i] = ptr(self.k_norm[i])
        return s

    def quantized(self, stream=None) -> "DoubleWeights":
        q = lambda ls: [quantize_linear(l, stream) for l in ls]
        return DoubleWeights(q(self.mod), q(self.qkv), q(self.proj), q(self.mlp_in), q(self.mlp_out), self.q_norm,
                             self.k_norm)

    def quantized_f8(self, stream=None) -> "DoubleWeights":
        """MMDIT_F8W copy: the four GEMM linears in e4m3, modulation kept bf16."""
        q = lambda ls: [quantize_linear_f8(l, stream) for l in ls]
        return DoubleWeights(self.mod, q(self.qkv), q(self.proj), q(self.mlp_in), q(self.mlp_out), self.q_norm,
                             self.k_norm)


@dataclass
class SingleWeights:
    mod: LinearDev
    lin1: LinearDev
    lin2: LinearDev
    q_norm: torch.Tensor
    k_norm: torch.Tensor

    def struct(self) -> SingleW:
        s = SingleW()
        s.mod, s.lin1, s.lin2 = self.mod.struct(), self.lin1.struct(), self.lin2.struct()
        s.q_norm, s.k_norm = ptr(self.q_norm), ptr(self.k_norm)
        return s

    def quantized(self, stream=None) -> "SingleWeights":
        q = lambda l: quantize_linear(l, stream)
        return SingleWeights(q(self.mod), q(self.lin1), q(self.lin2), self.q_norm, self.k_norm)

    def quantized_f8(self, stream=None) -> "SingleWeights":
        """MMDIT_F8W copy: lin1 and lin2 in e4m3, modulation kept bf16."""
        q = lambda l: quantize_linear_f8(l, stream)
        return SingleWeights(self.mod, q(self.lin1), q(self.lin2), self.q_norm, self.k_norm)


@dataclass
class StepWeights:
    time1: LinearDev
    time2: LinearDev
    img_in: LinearDev
    final_mod: LinearDev
    final: LinearDev
    doubles: List[DoubleWeights]
    singles: List[SingleWeights]
    _keep: list = field(default_factory=list, repr=False)

    def struct(self) -> StepW:
        s = StepW()
        s.time1, s.time2, s.img_in = self.time1.struct(), self.time2.struct(), self.img_in.struct()
        s.final_mod, s.final = self.final_mod.struct(), self.final.struct()
        darr = (DoubleW * max(1, len(self.doubles)))(*[d.struct() for d in self.doubles])
        sarr = (SingleW * max(1, len(self.singles)))(*[b.struct() for b in self.singles])
        self._keep = [darr, sarr]
        s.doubles = ctypes.cast(darr, ctypes.POINTER(DoubleW))
        s.n_double = len(self.doubles)
        s.singles = ctypes.cast(sarr, ctypes.POINTER(SingleW))
        s.n_single = len(self.singles)
        return s

    def quantized(self, stream=None) -> "StepWeights":
        q = lambda l: quantize_linear(l, stream)
        return StepWeights(q(self.time1), q(self.time2), q(self.img_in), q(self.final_mod), q(self.final),
                           [d.quantized(stream) for d in self.doubles], [b.quantized(stream) for b in self.singles])

    def quantized_f8(self, stream=None) -> "StepWeights":
        """MMDIT_F8W copy: the block GEMM linears in e4m3; every other linear bf16."""
        return StepWeights(self.time1, self.time2, self.img_in, self.final_mod, self.final,
                           [d.quantized_f8(stream) for d in self.doubles], [b.quantized_f8(stream) for b in self.singles])


@dataclass
class CondWeights:
    """Conditioning layers of the sampling loop (mmdit_cond_w_t): the text
    projection C_txt -> D and the two-layer SiLU MLPs of the guidance scale
    (t_dim -> D -> D) and of the pooled text vector (C_pool -> D -> D)."""
    txt_in: LinearDev
    guid1: LinearDev
    guid2: LinearDev
    vec1: LinearDev
    vec2: LinearDev

    @property
    def C_txt(self) -> int:
        return self.txt_in.w.shape[1]

    @property
    def C_pool(self) -> int:
        return self.vec1.w.shape[1]

    def struct(self) -> CondW:
        c = CondW()
        c.txt_in, c.guid1, c.guid2 = self.txt_in.struct(), self.guid1.struct(), self.guid2.struct()
        c.vec1, c.vec2 = self.vec1.struct(), self.vec2.struct()
        c.C_txt, c.C_pool = self.C_txt, self.C_pool
        return c

    def quantized(self, stream=None) -> "CondWeights":
        q = lambda l: quantize_linear(l, stream)
        return CondWeights(q(self.txt_in), q(self.guid1), q(self.guid2), q(self.vec1), q(self.vec2))


# ------------------------------------------------------------------ entry points
def workspace_size(shape: Shape, op: int) -> int:
    n = ctypes.c_size_t(0)
    call("mmdit_workspace_size", ctypes.byref(shape), op, ctypes.byref(n))
    return n.value


def step_workspace_size(shape: Shape, n_double: int, n_single: int) -> int:
    n = ctypes.c_size_t(0)
    call("mmdit_step_workspace_size", ctypes.byref(shape), n_double, n_single, ctypes.byref(n))
    return n.value


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def sync_status(stream=None) -> int:
    return _lib.load().mmdit_sync_status(stream_handle(stream))


def selftest_wait_timeout(limit_us: int, stream=None) -> None:
    call("mmdit_selftest_wait_timeout", limit_us, stream_handle(stream))


def launch_count() -> int:
    return int(_lib.load().mmdit_launch_count())


def trace_begin(capacity: int) -> None:
    call("mmdit_trace_begin", capacity)


def trace_end() -> int:
    n = ctypes.c_int(0)
    call("mmdit_trace_end", ctypes.byref(n))
    return n.value


def trace_read(capacity: int):
    """[(kernel name, milliseconds)] of the launches recorded by the trace."""
    ids = (ctypes.c_int * capacity)()
    ms = (ctypes.c_float * capacity)()
    n = ctypes.c_int(0)
    call("mmdit_trace_read", ids, ms, capacity, ctypes.byref(n))
    lib = _lib.load()
    return [(lib.mmdit_kernel_name(ids[i]).decode(), float(ms[i])) for i in range(n.value)]


def mmdit_rope2d_build(shape: Shape, ids: Optional[torch.Tensor], cos: torch.Tensor, sin: torch.Tensor, stream=None):
    call("mmdit_rope2d_build", ctypes.byref(shape), ptr(ids), ptr(cos), ptr(sin), stream_handle(stream))


def rope2d_apply(shape: Shape, cos: torch.Tensor, sin: torch.Tensor, x: torch.Tensor, row_stride: int, stream=None):
    call("rope2d_apply", ctypes.byref(shape), ptr(cos), ptr(sin), ptr(x), row_stride, stream_handle(stream))


def _pair(ts: Optional[Sequence[Optional[torch.Tensor]]]):
    if ts is None:
        return None
    arr = (ctypes.c_void_p * 2)(ptr(ts[0]), ptr(ts[1]))
    return arr


def joint_attention_fwd(shape: Shape, qkv: torch.Tensor, qkv_row_stride: int, q_norm, k_norm, cos, sin,
                        out: torch.Tensor, out_row_stride: int, ws: torch.Tensor, stream=None):
    qn, kn = _pair(q_norm), _pair(k_norm)
    call("joint_attention_fwd", ctypes.byref(shape), ptr(qkv), qkv_row_stride,
         ctypes.cast(qn, ctypes.POINTER(ctypes.c_void_p)) if qn is not None else None,
         ctypes.cast(kn, ctypes.POINTER(ctypes.c_void_p)) if kn is not None else None, ptr(cos), ptr(sin), ptr(out),
         out_row_stride, ptr(ws), ws.numel(), stream_handle(stream))


def joint_attention_fwd_noalloc(shape: Shape, qkv: torch.Tensor, qkv_row_stride: int, q_norm, k_norm, cos, sin,
                                out: torch.Tensor, out_row_stride: int, stream=None):
    """joint_attention_fwd without a workspace: the library's fixed device
    scratch is used instead (for callers that cannot allocate)."""
    qn, kn = _pair(q_norm), _pair(k_norm)
    call("joint_attention_fwd_noalloc", ctypes.byref(shape), ptr(qkv), qkv_row_stride,
         ctypes.cast(qn, ctypes.POINTER(ctypes.c_void_p)) if qn is not None else None,
         ctypes.cast(kn, ctypes.POINTER(ctypes.c_void_p)) if kn is not None else None, ptr(cos), ptr(sin), ptr(out),
         out_row_stride, stream_handle(stream))


def mmdit_double_block_fwd(shape: Shape, w: DoubleWeights, vec, mod_precomputed, x_txt, x_img, cos, sin,
                           ws: torch.Tensor, stream=None):
    ws_struct = w.struct()
    call("mmdit_double_block_fwd", ctypes.byref(shape), ctypes.byref(ws_struct), ptr(vec), ptr(mod_precomputed),
         ptr(x_txt), ptr(x_img), ptr(cos), ptr(sin), ptr(ws), ws.numel(), stream_handle(stream))


def mmdit_single_block_fwd(shape: Shape, w: SingleWeights, vec, mod_precomputed, x, cos, sin, ws: torch.Tensor,
                           stream=None):
    st = w.struct()
    call("mmdit_single_block_fwd", ctypes.byref(shape), ctypes.byref(st), ptr(vec), ptr(mod_precomputed), ptr(x),
         ptr(cos), ptr(sin), ptr(ws), ws.numel(), stream_handle(stream))


def mmdit_step_fwd(shape: Shape, w: StepWeights, x_lat, x_txt_in, sigma: float, sigma_next: float, v_out,
                   ws: torch.Tensor, stream=None, step_struct: Optional[StepW] = None):
    st = step_struct if step_struct is not None else w.struct()
    call("mmdit_step_fwd", ctypes.byref(shape), ctypes.byref(st), ptr(x_lat), ptr(x_txt_in), float(sigma),
         float(sigma_next), ptr(v_out), ptr(ws), ws.numel(), stream_handle(stream))


def mmdit_step_i2i_fwd(shape: Shape, w: StepWeights, x_lat, x_ref, x_txt_in, sigma: float, sigma_next: float, v_out,
                       ws: torch.Tensor, stream=None, step_struct: Optional[StepW] = None):
    st = step_struct if step_struct is not None else w.struct()
    call("mmdit_step_i2i_fwd", ctypes.byref(shape), ctypes.byref(st), ptr(x_lat), ptr(x_ref), ptr(x_txt_in),
         float(sigma), float(sigma_next), ptr(v_out), ptr(ws), ws.numel(), stream_handle(stream))


def sample_workspace_size(shape: Shape, n_double: int, n_single: int, C_txt: int, n_steps: int) -> int:
    n = ctypes.c_size_t(0)
    call("mmdit_sample_workspace_size", ctypes.byref(shape), n_double, n_single, C_txt, n_steps, ctypes.byref(n))
    return n.value


def mmdit_sample(shape: Shape, w: StepWeights, cond: CondWeights, x_lat, txt, pooled, guidance: float, sigmas,
                 ws: torch.Tensor, graph: bool = True, stream=None, step_struct: Optional[StepW] = None):
    """The sampling loop over the host schedule sigmas (n_steps + 1 values),
    x_lat updated in place; graph=True replays steps 1.. from one captured
    CUDA graph (the call then waits for them)."""
    st = step_struct if step_struct is not None else w.struct()
    cs = cond.struct()
    sig = (ctypes.c_double * len(sigmas))(*[float(v) for v in sigmas])
    call("mmdit_sample", ctypes.byref(shape), ctypes.byref(st), ctypes.byref(cs), ptr(x_lat), ptr(txt), ptr(pooled),
         float(guidance), sig, len(sigmas) - 1, MMDIT_SAMPLE_GRAPH if graph else 0, ptr(ws), ws.numel(),
         stream_handle(stream))


def euler_step(x: torch.Tensor, v: torch.Tensor, sigma: float, sigma_next: float, stream=None):
    vd = {torch.float32: MMDIT_F32, torch.bfloat16: MMDIT_BF16}[v.dtype]
    call("euler_step", ptr(x), ptr(v), vd, float(sigma), float(sigma_next), x.numel(), stream_handle(stream))


def mmdit_quantize_w8(w: torch.Tensor, q: torch.Tensor, scale: torch.Tensor, stream=None):
    wd = {torch.float32: MMDIT_F32, torch.bfloat16: MMDIT_BF16}[w.dtype]
    call("mmdit_quantize_w8", ptr(w), wd, w.shape[0], w.shape[1], ptr(q), ptr(scale), stream_handle(stream))


def mmdit_linear_fwd(lin: LinearDev, x: torch.Tensor, y: torch.Tensor, epilogue: int, gate=None,
                     ws: Optional[torch.Tensor] = None, stream=None):
    M, K = x.shape
    N = lin.N
    st = lin.struct()
    call("mmdit_linear_fwd", ctypes.byref(st), M, N, K, ptr(x), ptr(y), epilogue, ptr(gate), ptr(ws),
         0 if ws is None else ws.numel(), stream_handle(stream))


def quantize_f8(x: torch.Tensor, stream=None):
    """Rows of a 2-D bf16 / fp32 tensor to e4m3 (uint8 codes) and fp32 row scales
    (s = max|row| / 448)."""
    rows, K = x.shape
    q = torch.empty((rows, K), dtype=torch.uint8, device=x.device)
    s = torch.empty((rows,), dtype=torch.float32, device=x.device)
    xd = {torch.float32: MMDIT_F32, torch.bfloat16: MMDIT_BF16}[x.dtype]
    call("mmdit_quantize_f8", ptr(x, strided_ok=True), xd, rows, K, x.stride(0), ptr(q), ptr(s), stream_handle(stream))
    return q, s


def quantize_linear_f8(lin: LinearDev, stream=None) -> LinearDev:
    """e4m3 per-channel copy of a bf16 linear (weights e4m3 codes, fp32 scales)."""
    q, s = quantize_f8(lin.w, stream)
    return LinearDev(q, lin.b, s)


def mmdit_linear_f8_fwd(lin: LinearDev, x8: torch.Tensor, x_scale: torch.Tensor, y: torch.Tensor, epilogue: int,
                        gate=None, stream=None):
    M, K = x8.shape
    st = lin.struct()
    call("mmdit_linear_f8_fwd", ctypes.byref(st), M, lin.N, K, ptr(x8), ptr(x_scale), ptr(y), epilogue, ptr(gate),
         stream_handle(stream))


def mmdit_ln_modulate(x: torch.Tensor, shift: torch.Tensor, scale: torch.Tensor, mod_stride: int, eps: float,
                      y: torch.Tensor, stream=None):
    B, rows, D = x.shape
    call("mmdit_ln_modulate", ptr(x), B, rows, D, ptr(shift, True), ptr(scale, True), mod_stride, eps, ptr(y),
         stream_handle(stream))


def mmdit_ln_modulate_f8(x: torch.Tensor, shift: torch.Tensor, scale: torch.Tensor, mod_stride: int, eps: float,
                         y: Optional[torch.Tensor] = None, stream=None):
    """LN + modulate with the e4m3 rows of its bf16 result: (codes uint8 [B, rows, D], scales fp32 [B, rows])."""
    B, rows, D = x.shape
    q = torch.empty((B, rows, D), dtype=torch.uint8, device=x.device)
    s = torch.empty((B, rows), dtype=torch.float32, device=x.device)
    call("mmdit_ln_modulate_f8", ptr(x), B, rows, D, ptr(shift, True), ptr(scale, True), mod_stride, eps, ptr(y),
         ptr(q), ptr(s), stream_handle(stream))
    return q, s


def mmdit_gemv(lin: LinearDev, x: torch.Tensor, act: int, y: torch.Tensor, stream=None):
    B, K = x.shape
    st = lin.struct()
    call("mmdit_gemv", ctypes.byref(st), B, lin.N, K, ptr(x), act, ptr(y), stream_handle(stream))


def mmdit_heads_pack(src: torch.Tensor, sections: int, groups: int, group_cols: int, dst: torch.Tensor,
                     stream=None):
    """src [rows, src_ld] bf16 -> dst [groups, rows, sections, group_cols] (see include/mmdit.h)."""
    rows, ld = src.shape
    call("mmdit_heads_pack", ptr(src), rows, ld, sections, groups, group_cols, ptr(dst), stream_handle(stream))


def mmdit_heads_unpack(src: torch.Tensor, groups: int, group_cols: int, dst: torch.Tensor, stream=None):
    """src [groups, rows, group_cols] bf16 -> dst [rows, dst_ld] (head group g at columns g * group_cols)."""
    rows, ld = dst.shape
    call("mmdit_heads_unpack", ptr(src), rows, groups, group_cols, ptr(dst), ld, stream_handle(stream))


def mmdit_time_embed(shape: Shape, time1: LinearDev, time2: LinearDev, sigma: float, vec: torch.Tensor,
                     ws: torch.Tensor, stream=None):
    a, b = time1.struct(), time2.struct()
    call("mmdit_time_embed", ctypes.byref(shape), ctypes.byref(a), ctypes.byref(b), float(sigma), ptr(vec), ptr(ws),
         stream_handle(stream))
