"""Ulysses sequence parallelism for the MMDiT blocks.

The SGLang blog ("Architecture Deep Dive", section "SGLang Diffusion
Serving") scales the diffusion transformer over several GPUs with USP, hybrid
Ulysses sequence parallelism and ring attention.  This module is the Ulysses
half.  Each of P ranks holds a contiguous shard of the token sequence
[text; image] and runs every token-wise step of a block on that shard alone:
modulation, LN + modulate, the linears, the gated residuals, the MLP.  Joint
attention needs every token, so around it two all-to-all exchanges trade the
rank's token shard of all heads for all tokens of its H / P heads, and back:

  pre      LN + modulate and the QKV linear on the shard; mmdit_heads_pack
           lays [q | k | v] out as one contiguous chunk per head group
  exchange sequence -> heads: rank r receives, from every rank s, s's tokens
           of head group r; concatenated in rank order they are all L tokens
  attend   joint_attention_fwd over all L tokens for the H / P heads (q/k
           RMSNorm and RoPE at the tokens' global positions)
  exchange heads -> sequence: rank r gets back its own tokens from every
           head group; mmdit_heads_unpack restores the [L_r, D] layout
  post     projection with gated residual and the MLP on the shard

The exchanges are passed in: over a process group they are
torch.distributed.all_to_all_single (NCCL on GPUs, gloo on CPU); on one
device a loopback of P virtual ranks stands in for them.  Every step of the
block runs in libmmdit's kernels through the C ABI; this module sequences the
calls and owns the buffers.  Batch 1 (the latency case that sequence
parallelism serves; independent samples shard across ranks as replicas).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Optional, Sequence

import torch

from . import api


# ------------------------------------------------------------------ the plan
@dataclass(frozen=True)
class ShardPlan:
    """Contiguous token shards of one sample's sequence [text; image] over P
    ranks: rank r holds global tokens [start(r), start(r) + size(r)), sizes
    differing by at most one (the first L % P ranks hold one more)."""
    L_txt: int
    L_img: int
    P: int

    @property
    def L(self) -> int:
        return self.L_txt + self.L_img

    def size(self, r: int) -> int:
        return self.L // self.P + (1 if r < self.L % self.P else 0)

    def start(self, r: int) -> int:
        return r * (self.L // self.P) + min(r, self.L % self.P)

    def sizes(self) -> List[int]:
        return [self.size(r) for r in range(self.P)]

    def text_rows(self, r: int):
        """Text tokens of rank r: (first text index, count)."""
        a, b = self.start(r), self.start(r) + self.size(r)
        lo, hi = min(a, self.L_txt), min(b, self.L_txt)
        return lo, hi - lo

    def image_rows(self, r: int):
        """Image tokens of rank r: (first image index, count); image index i is global token L_txt + i."""
        a, b = self.start(r), self.start(r) + self.size(r)
        lo, hi = max(a, self.L_txt), max(b, self.L_txt)
        return lo - self.L_txt, hi - lo


# ------------------------------------------------------------------ exchanges
def exchange_seq_to_heads(send: torch.Tensor, plan: ShardPlan, rank: int, group=None) -> torch.Tensor:
    """send: [P * size(rank), W], the chunk for head group g at rows
    g * size(rank) ..; returns [L, W], every rank's tokens of this rank's head
    group in global token order."""
    import torch.distributed as dist
    recv = torch.empty((plan.L, send.shape[1]), dtype=send.dtype, device=send.device)
    dist.all_to_all_single(recv, send, output_split_sizes=plan.sizes(), input_split_sizes=[plan.size(rank)] * plan.P,
                           group=group)
    return recv


def exchange_heads_to_seq(out: torch.Tensor, plan: ShardPlan, rank: int, group=None) -> torch.Tensor:
    """out: [L, W], this rank's head group for all tokens; returns
    [P * size(rank), W], this rank's tokens from head group g at rows
    g * size(rank) .."""
    import torch.distributed as dist
    back = torch.empty((plan.P * plan.size(rank), out.shape[1]), dtype=out.dtype, device=out.device)
    dist.all_to_all_single(back, out, output_split_sizes=[plan.size(rank)] * plan.P, input_split_sizes=plan.sizes(),
                           group=group)
    return back


def loopback_seq_to_heads(sends: Sequence[torch.Tensor], plan: ShardPlan) -> List[torch.Tensor]:
    """The sequence -> heads exchange of P virtual ranks on one device."""
    return [torch.cat([sends[s][r * plan.size(s):(r + 1) * plan.size(s)] for s in range(plan.P)], 0)
            for r in range(plan.P)]


def loopback_heads_to_seq(outs: Sequence[torch.Tensor], plan: ShardPlan) -> List[torch.Tensor]:
    """The heads -> sequence exchange of P virtual ranks on one device."""
    return [torch.cat([outs[g][plan.start(r):plan.start(r) + plan.size(r)] for g in range(plan.P)], 0)
            for r in range(plan.P)]


# ------------------------------------------------------------------ blocks
def _linear(lin: api.LinearDev, x: torch.Tensor, y: torch.Tensor, epi: int, gate=None, wdeq=None):
    if x.shape[0] > 0:
        api.mmdit_linear_fwd(lin, x, y, epi, gate, wdeq if lin.scale is not None else None)


def _ln_mod(x: torch.Tensor, shift: torch.Tensor, scale: torch.Tensor, eps: float, y: torch.Tensor):
    if x.shape[0] > 0:
        api.mmdit_ln_modulate(x.view(1, *x.shape), shift, scale, 0, eps, y.view(1, *y.shape))


class _UlyssesBase:
    def __init__(self, shape: api.Shape, P: int, cos: torch.Tensor, sin: torch.Tensor):
        if shape.B != 1:
            raise ValueError("sequence parallelism runs one sample (batch 1)")
        if shape.H % P:
            raise ValueError("the head count must divide by the number of ranks")
        self.shape, self.P = shape, P
        self.D, self.Dg = shape.D, shape.D // P
        self.plan = ShardPlan(shape.L_txt, shape.grid_h * shape.grid_w + shape.ref_h * shape.ref_w, P)
        self.cos, self.sin = cos, sin
        # the attention problem of one head group: H / P heads, all tokens and their global positions
        self.head_shape = api.make_shape(B=1, L_txt=shape.L_txt, grid_h=shape.grid_h, grid_w=shape.grid_w, D=self.Dg,
                                         H=shape.H // P, d_head=shape.d_head, D_mlp=shape.D_mlp,
                                         rope_axes=tuple(shape.rope_axes), rope_theta=shape.rope_theta,
                                         eps_ln=shape.eps_ln, eps_rms=shape.eps_rms, ref_h=shape.ref_h,
                                         ref_w=shape.ref_w)
        self.attn_ws = api.alloc_workspace(api.workspace_size(self.head_shape, api.MMDIT_OP_ATTENTION),
                                           device=cos.device)

    def _pack(self, qkv: torch.Tensor) -> torch.Tensor:
        n = qkv.shape[0]
        send = torch.empty((self.P * n, 3 * self.Dg), dtype=torch.bfloat16, device=qkv.device)
        if n:
            api.mmdit_heads_pack(qkv, 3, self.P, self.Dg, send)
        return send

    def _unpack(self, back: torch.Tensor, n: int) -> torch.Tensor:
        o = torch.empty((n, self.D), dtype=torch.bfloat16, device=back.device)
        if n:
            api.mmdit_heads_unpack(back, self.P, self.Dg, o)
        return o

    def _attend(self, recv: torch.Tensor, q_norm, k_norm) -> torch.Tensor:
        out = torch.empty((self.plan.L, self.Dg), dtype=torch.bfloat16, device=recv.device)
        api.joint_attention_fwd(self.head_shape, recv, 3 * self.Dg, q_norm, k_norm, self.cos, self.sin, out, self.Dg,
                                self.attn_ws)
        return out


class UlyssesDoubleBlock(_UlyssesBase):
    """A double-stream block under Ulysses sequence parallelism.  Rank r holds
    the text rows and the image rows of its token shard (fp32 residual
    stream, updated in place by post)."""

    def __init__(self, shape: api.Shape, w: api.DoubleWeights, P: int, cos: torch.Tensor, sin: torch.Tensor):
        super().__init__(shape, P, cos, sin)
        self.w = w
        self.swiglu = shape.mlp_act == api.MMDIT_MLP_SWIGLU
        big = max(l.N * l.K for ls in (w.qkv, w.proj, w.mlp_in, w.mlp_out) for l in ls)
        int8 = any(l.scale is not None for ls in (w.qkv, w.proj, w.mlp_in, w.mlp_out) for l in ls)
        self.wdeq = torch.empty(big, dtype=torch.bfloat16, device=cos.device) if int8 else None

    def modulation(self, vec: torch.Tensor) -> torch.Tensor:
        """[2, 6D] fp32: each stream's (shift1, scale1, gate1, shift2, scale2, gate2)."""
        mod = torch.empty((2, 6 * self.D), dtype=torch.float32, device=vec.device)
        for s in range(2):
            api.mmdit_gemv(self.w.mod[s], vec, 1, mod[s:s + 1])
        return mod

    def _parts(self, r: int, x_txt: torch.Tensor, x_img: torch.Tensor):
        return ((0, x_txt, 0), (1, x_img, x_txt.shape[0]))  # (stream, rows, first local row)

    def pre(self, r: int, x_txt: torch.Tensor, x_img: torch.Tensor, mod: torch.Tensor) -> torch.Tensor:
        D, n = self.D, x_txt.shape[0] + x_img.shape[0]
        y = torch.empty((n, D), dtype=torch.bfloat16, device=mod.device)
        qkv = torch.empty((n, 3 * D), dtype=torch.bfloat16, device=mod.device)
        for s, x, o in self._parts(r, x_txt, x_img):
            m = x.shape[0]
            _ln_mod(x, mod[s, 0:D], mod[s, D:2 * D], self.shape.eps_ln, y[o:o + m])
            _linear(self.w.qkv[s], y[o:o + m], qkv[o:o + m], api.MMDIT_EPI_BF16, wdeq=self.wdeq)
        return self._pack(qkv)

    def attend(self, recv: torch.Tensor) -> torch.Tensor:
        return self._attend(recv, self.w.q_norm, self.w.k_norm)

    def post(self, r: int, back: torch.Tensor, x_txt: torch.Tensor, x_img: torch.Tensor, mod: torch.Tensor):
        D, Dm = self.D, self.shape.D_mlp
        n = x_txt.shape[0] + x_img.shape[0]
        o_all = self._unpack(back, n)
        for s, x, o in self._parts(r, x_txt, x_img):
            m = x.shape[0]
            if m == 0:
                continue
            _linear(self.w.proj[s], o_all[o:o + m], x, api.MMDIT_EPI_RESID, mod[s, 2 * D:3 * D], self.wdeq)
            y2 = torch.empty((m, D), dtype=torch.bfloat16, device=x.device)
            _ln_mod(x, mod[s, 3 * D:4 * D], mod[s, 4 * D:5 * D], self.shape.eps_ln, y2)
            h = torch.empty((m, Dm), dtype=torch.bfloat16, device=x.device)
            _linear(self.w.mlp_in[s], y2, h, api.MMDIT_EPI_SWIGLU if self.swiglu else api.MMDIT_EPI_BF16_GELU,
                    wdeq=self.wdeq)
            _linear(self.w.mlp_out[s], h, x, api.MMDIT_EPI_RESID, mod[s, 5 * D:6 * D], self.wdeq)


class UlyssesSingleBlock(_UlyssesBase):
    """A single-stream block under Ulysses sequence parallelism.  The fused
    first linear is split by rows into its q/k/v part (exchanged) and its MLP
    part (kept on the shard); the output linear by columns into its
    attention part and its MLP part, whose two gated products both add to
    the residual (the bias once)."""

    def __init__(self, shape: api.Shape, w: api.SingleWeights, P: int, cos: torch.Tensor, sin: torch.Tensor):
        super().__init__(shape, P, cos, sin)
        if w.lin1.scale is not None or w.lin2.scale is not None:
            raise ValueError("sequence-parallel single blocks take bf16 weights")
        D = shape.D
        self.w = w
        self.swiglu = shape.mlp_act == api.MMDIT_MLP_SWIGLU
        b1 = w.lin1.b
        self.qkv = api.LinearDev(w.lin1.w[:3 * D].contiguous(), None if b1 is None else b1[:3 * D].contiguous())
        self.mlp = api.LinearDev(w.lin1.w[3 * D:].contiguous(), None if b1 is None else b1[3 * D:].contiguous())
        self.out_attn = api.LinearDev(w.lin2.w[:, :D].contiguous(), w.lin2.b)
        self.out_mlp = api.LinearDev(w.lin2.w[:, D:].contiguous(), None)

    def modulation(self, vec: torch.Tensor) -> torch.Tensor:
        """[3D] fp32: (shift, scale, gate)."""
        mod = torch.empty((1, 3 * self.D), dtype=torch.float32, device=vec.device)
        api.mmdit_gemv(self.w.mod, vec, 1, mod)
        return mod[0]

    def pre(self, r: int, x: torch.Tensor, mod: torch.Tensor):
        """Returns (the packed q/k/v chunks, the shard's activated MLP columns)."""
        D, Dm, n = self.D, self.shape.D_mlp, x.shape[0]
        y = torch.empty((n, D), dtype=torch.bfloat16, device=x.device)
        _ln_mod(x, mod[0:D], mod[D:2 * D], self.shape.eps_ln, y)
        qkv = torch.empty((n, 3 * D), dtype=torch.bfloat16, device=x.device)
        _linear(self.qkv, y, qkv, api.MMDIT_EPI_BF16)
        h = torch.empty((n, Dm), dtype=torch.bfloat16, device=x.device)
        _linear(self.mlp, y, h, api.MMDIT_EPI_SWIGLU if self.swiglu else api.MMDIT_EPI_BF16_GELU)
        return self._pack(qkv), h

    def attend(self, recv: torch.Tensor) -> torch.Tensor:
        return self._attend(recv, [self.w.q_norm, self.w.q_norm], [self.w.k_norm, self.w.k_norm])

    def post(self, r: int, back: torch.Tensor, x: torch.Tensor, mod: torch.Tensor, h: torch.Tensor):
        D, n = self.D, x.shape[0]
        o = self._unpack(back, n)
        _linear(self.out_attn, o, x, api.MMDIT_EPI_RESID, mod[2 * D:3 * D])
        _linear(self.out_mlp, h, x, api.MMDIT_EPI_RESID, mod[2 * D:3 * D])


# ------------------------------------------------------------------ drivers
def double_block_rank(block: UlyssesDoubleBlock, x_txt: torch.Tensor, x_img: torch.Tensor, vec: torch.Tensor,
                      rank: int, group=None) -> None:
    """One rank of a process group: its shard's text rows x_txt and image rows
    x_img (fp32, updated in place), the conditioning vector vec [1, D]."""
    mod = block.modulation(vec)
    recv = exchange_seq_to_heads(block.pre(rank, x_txt, x_img, mod), block.plan, rank, group)
    back = exchange_heads_to_seq(block.attend(recv), block.plan, rank, group)
    block.post(rank, back, x_txt, x_img, mod)


def single_block_rank(block: UlyssesSingleBlock, x: torch.Tensor, vec: torch.Tensor, rank: int, group=None) -> None:
    mod = block.modulation(vec)
    send, h = block.pre(rank, x, mod)
    recv = exchange_seq_to_heads(send, block.plan, rank, group)
    back = exchange_heads_to_seq(block.attend(recv), block.plan, rank, group)
    block.post(rank, back, x, mod, h)


def shard(x: torch.Tensor, plan: ShardPlan, r: int, L_off: int = 0) -> torch.Tensor:
    """Rank r's rows of a [L, D] (or, with L_off, a stream's) tensor: a copy."""
    a, n = plan.start(r) - L_off, plan.size(r)
    return x[max(a, 0):max(a + n, 0)].clone()


def double_block_loopback(block: UlyssesDoubleBlock, x_txt: torch.Tensor, x_img: torch.Tensor,
                          vec: torch.Tensor) -> None:
    """The sharded schedule of P virtual ranks on one device, the exchanges
    done as copies; x_txt [L_txt, D] and x_img [L_img, D] are updated in
    place."""
    plan = block.plan
    txt = [x_txt[a:a + n].clone() for a, n in (plan.text_rows(r) for r in range(plan.P))]
    img = [x_img[a:a + n].clone() for a, n in (plan.image_rows(r) for r in range(plan.P))]
    mod = block.modulation(vec)
    recvs = loopback_seq_to_heads([block.pre(r, txt[r], img[r], mod) for r in range(plan.P)], plan)
    backs = loopback_heads_to_seq([block.attend(recvs[r]) for r in range(plan.P)], plan)
    for r in range(plan.P):
        block.post(r, backs[r], txt[r], img[r], mod)
        (a, n), (b, m) = plan.text_rows(r), plan.image_rows(r)
        x_txt[a:a + n] = txt[r]
        x_img[b:b + m] = img[r]


def single_block_loopback(block: UlyssesSingleBlock, x: torch.Tensor, vec: torch.Tensor) -> None:
    plan = block.plan
    xs = [x[plan.start(r):plan.start(r) + plan.size(r)].clone() for r in range(plan.P)]
    mod = block.modulation(vec)
    pres = [block.pre(r, xs[r], mod) for r in range(plan.P)]
    recvs = loopback_seq_to_heads([p[0] for p in pres], plan)
    backs = loopback_heads_to_seq([block.attend(recvs[r]) for r in range(plan.P)], plan)
    for r in range(plan.P):
        block.post(r, backs[r], xs[r], mod, pres[r][1])
        x[plan.start(r):plan.start(r) + plan.size(r)] = xs[r]
