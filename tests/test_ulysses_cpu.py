"""Ulysses sequence parallelism, host side, on CPU: the token-shard plan, and
the two all-to-all exchanges run over a real gloo process group of two ranks.
The exchanged data is built from its own coordinates (token, section, head,
channel), so every element proves where it came from; the chunk layout of
the sends is the one mmdit_heads_pack writes (checked against these
layouts on the GPU in test_gpu_ulysses)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from diffusion_transformer_image_mmdit_gb300.ulysses import (ShardPlan, exchange_heads_to_seq, exchange_seq_to_heads,
                                                             loopback_heads_to_seq, loopback_seq_to_heads)


def test_shard_plan_covers_the_sequence():
    for L_txt, L_img, P in ((512, 6889, 2), (50, 111, 4), (3, 2, 4), (0, 7, 3)):
        plan = ShardPlan(L_txt, L_img, P)
        sizes = plan.sizes()
        assert sum(sizes) == L_txt + L_img and max(sizes) - min(sizes) <= 1
        assert [plan.start(r) for r in range(P)] == list(np.cumsum([0] + sizes[:-1]))
        txt = [plan.text_rows(r) for r in range(P)]
        img = [plan.image_rows(r) for r in range(P)]
        assert sum(n for _, n in txt) == L_txt and sum(n for _, n in img) == L_img
        for r in range(P):  # text rows precede image rows inside a shard, and together they are the shard
            assert txt[r][1] + img[r][1] == sizes[r]
            if txt[r][1]:
                assert txt[r][0] == plan.start(r)
            if img[r][1]:
                assert L_txt + img[r][0] == plan.start(r) + txt[r][1]


def _coords(tokens, P, Dg, sections=3):
    """Values of rows `tokens`: [n, sections * P * Dg], element (t, s, g, c) = t * 1e4 + s * 1e3 + g * 100 + c."""
    t = np.asarray(tokens, np.float64)[:, None, None, None]
    s = np.arange(sections)[None, :, None, None]
    g = np.arange(P)[None, None, :, None]
    c = np.arange(Dg)[None, None, None, :]
    return (t * 1e4 + s * 1e3 + g * 100 + c).reshape(len(tokens), sections * P * Dg)


def _pack(rows, P, Dg, sections=3):
    """The head-group chunk layout: [P * n, sections * Dg], chunk g holding sections x head group g."""
    n = rows.shape[0]
    return rows.reshape(n, sections, P, Dg).transpose(2, 0, 1, 3).reshape(P * n, sections * Dg)


def _unpack(back, P, Dg):
    n = back.shape[0] // P
    return back.reshape(P, n, Dg).transpose(1, 0, 2).reshape(n, P * Dg)


def _check_exchanges(plan, rank, exchange_fwd, exchange_back, Dg=8):
    P = plan.P
    mine = np.arange(plan.start(rank), plan.start(rank) + plan.size(rank))
    send = torch.from_numpy(_pack(_coords(mine, P, Dg), P, Dg))
    recv = exchange_fwd(send).numpy()
    # all L tokens, in global order, of this rank's head group, sections q | k | v
    want = _coords(np.arange(plan.L), P, Dg).reshape(plan.L, 3, P, Dg)[:, :, rank, :].reshape(plan.L, 3 * Dg)
    assert np.array_equal(recv, want)
    # a stand-in attention output for this head group: its q section
    out = torch.from_numpy(np.ascontiguousarray(recv[:, :Dg]))
    back = exchange_back(out).numpy()
    # this rank's tokens, every head group's q section, heads in group order
    want_back = _coords(mine, P, Dg).reshape(len(mine), 3, P * Dg)[:, 0, :]
    assert np.array_equal(_unpack(back, P, Dg), want_back)


def _worker(rank, world, port, cases, errors):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        for L_txt, L_img in cases:
            plan = ShardPlan(L_txt, L_img, world)
            _check_exchanges(plan, rank, lambda s: exchange_seq_to_heads(s, plan, rank),
                             lambda o: exchange_heads_to_seq(o, plan, rank))
        dist.barrier()
    except Exception as e:  # reported to the parent
        errors.put(f"rank {rank}: {e!r}")
        raise
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_exchanges_over_gloo_world_size_2():
    ctx = mp.get_context("spawn")
    errors = ctx.Queue()
    cases = [(5, 12), (4, 3), (0, 9), (512, 6889)]  # even and uneven shards; a rank straddling text and image
    mp.start_processes(_worker, args=(2, _free_port(), cases, errors), nprocs=2, join=True, start_method="spawn")
    assert errors.empty()


@pytest.mark.parametrize("P", [1, 2, 3, 4])
def test_loopback_exchanges_match_the_collective_layout(P):
    """The single-device loopback of P virtual ranks moves exactly what the
    collective moves."""
    plan = ShardPlan(7, 10, P)
    sends = [torch.from_numpy(_pack(_coords(np.arange(plan.start(r), plan.start(r) + plan.size(r)), P, 4), P, 4))
             for r in range(P)]
    recvs = loopback_seq_to_heads(sends, plan)
    outs = [torch.from_numpy(np.ascontiguousarray(recvs[r].numpy()[:, :4])) for r in range(P)]
    backs = loopback_heads_to_seq(outs, plan)
    for r in range(P):
        _check_exchanges(plan, r, lambda s, r=r: recvs[r], lambda o, r=r: backs[r], Dg=4)
