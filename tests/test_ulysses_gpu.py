"""Ulysses sequence parallelism with the library's CUDA kernel doing the attention: P gloo
ranks (P = 2 and 4) hold contiguous token shards of q, k, v; the all-to-all exchanges run on
the host, and each rank runs vdx.rope3d_attn on cuda:0 for its H/P heads over all N tokens
(non-identity head shards: every rank's kernel sees a [B, N, H/P, d] tensor of other ranks'
tokens).  Every rank's output and lse shard is compared element by element with the fp64
oracle's rows for its tokens, at the bf16 tolerances.  The ranks share one GPU but never wait
on each other's kernels: all exchanges are host-side gloo collectives."""
import dataclasses
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle.fp64 as O
from video_diffusion_transformer_rope_gb300 import configs, synth

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, ws, port, H, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import video_diffusion_transformer_rope_gb300 as vdx
        from video_diffusion_transformer_rope_gb300.ulysses import ulysses_rope3d_attn
        torch.cuda.set_device(0)
        w = dataclasses.replace(configs.WAN13B_480P, B=2, H=H, T=2, Hg=8, Wg=20, seed=66)
        grid = (w.T, w.Hg, w.Wg)
        q, k, v = synth.make_qkv(w)                 # the same seeded draw on every rank
        Ns = w.N // ws
        sl = slice(rank * Ns, (rank + 1) * Ns)
        seen = []

        def attn_on_gpu(qh, kh, vh, grid_, sections_, theta_, scale_):
            seen.append(tuple(qh.shape))
            o, l = vdx.rope3d_attn(qh.cuda(), kh.cuda(), vh.cuda(), grid_, sections_, theta_, scale_)
            vdx.sync_check()
            return o.cpu(), l.cpu()

        out, lse = ulysses_rope3d_attn(q[:, sl].contiguous(), k[:, sl].contiguous(), v[:, sl].contiguous(),
                                       grid, w.sections, w.theta, attn=attn_on_gpu)
        ref_o, ref_l = O.rope3d_attention(q, k, v, grid, w.sections, w.theta)
        err = np.abs(out.double().numpy() - ref_o[:, sl])
        lerr = np.abs(lse.double().numpy() - ref_l[:, :, sl])
        results[rank] = (float(err.max()), float(err.mean()), float(lerr.max()), seen,
                         tuple(out.shape), tuple(lse.shape))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("ws,H", [(2, 4), (4, 8)])
def test_ulysses_with_cuda_kernel_matches_oracle(ws, H):
    from video_diffusion_transformer_rope_gb300 import _build
    _build.build()
    port = _free_port()
    results = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank, args=(ws, port, H, results), nprocs=ws, join=True)
    N = 2 * 8 * 20
    for r in range(ws):
        mx, mean, lerr, seen, so, sl = results[r]
        assert seen == [(2, N, H // ws, 128)], seen          # all tokens, this rank's heads
        assert so == (2, N // ws, H, 128) and sl == (2, H, N // ws)
        assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL, (r, mx, mean, lerr)
