"""Ulysses sequence-parallel wrapper on CPU: two and four gloo ranks hold token shards; after
the all-to-all exchange, per-rank attention over their heads, and the exchange back, every
rank's output shard equals the fp64 oracle's rows for its tokens.  (The attention callable
here is the oracle; on GPUs it is the library call, and the exchange goes over NCCL.)"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle.fp64 as O
from video_diffusion_transformer_rope_gb300.ulysses import ulysses_rope3d_attn


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _oracle_attn(q, k, v, grid, sections, theta, scale):
    o, l = O.rope3d_attention(q, k, v, grid, sections if any(sections) else None, theta,
                              scale if scale > 0 else None)
    return torch.from_numpy(o), torch.from_numpy(l)


def _rank(rank, ws, port, grid, H, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    T, Hg, Wg = grid
    N = T * Hg * Wg
    g = torch.Generator().manual_seed(7)
    q, k, v = (torch.randn(2, N, H, 64, generator=g, dtype=torch.float64) for _ in range(3))
    Ns = N // ws
    sl = slice(rank * Ns, (rank + 1) * Ns)
    out, lse = ulysses_rope3d_attn(q[:, sl].contiguous(), k[:, sl].contiguous(), v[:, sl].contiguous(),
                                   grid, attn=_oracle_attn)
    ref_o, ref_l = O.rope3d_attention(q, k, v, grid)
    results[rank] = (float(np.abs(out.numpy() - ref_o[:, sl]).max()),
                     float(np.abs(lse.numpy() - ref_l[:, :, sl]).max()),
                     tuple(out.shape), tuple(lse.shape))
    dist.destroy_process_group()


@pytest.mark.parametrize("ws,grid,H", [(2, (2, 4, 6), 4), (4, (2, 4, 6), 8)])
def test_ulysses_matches_oracle(ws, grid, H):
    port = _free_port()
    results = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank, args=(ws, port, grid, H, results), nprocs=ws, join=True)
    N = grid[0] * grid[1] * grid[2]
    for r in range(ws):
        err_o, err_l, so, sl = results[r]
        assert so == (2, N // ws, H, 64) and sl == (2, H, N // ws)
        assert err_o < 1e-12 and err_l < 1e-12, (r, err_o, err_l)


def test_ulysses_rejects_bad_shards():
    port = _free_port()
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=0, world_size=1)
    try:
        x = torch.zeros(1, 10, 3, 64)
        with pytest.raises(ValueError):
            ulysses_rope3d_attn(x, x, x, (1, 3, 4), attn=_oracle_attn)
    finally:
        dist.destroy_process_group()
