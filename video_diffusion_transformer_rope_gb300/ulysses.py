"""Sequence-parallel 3D-RoPE attention across ranks, Ulysses style.

The vidax page ("vidax: A Unified JAX Framework for Video Generative Models on Accelerator
Meshes", §2 "Spatiotemporal tensor and sequence sharding") shards the token sequence over
devices and, around attention, uses all-to-all transposes to head-sharded views.  Here, with P
ranks: every rank holds a contiguous token shard [B, N/P, H, d] of q, k and v; one all_to_all
gives each rank all N tokens for H/P heads; attention runs locally (the library call, or any
callable with its signature); a second all_to_all returns the output to token shards.

torch.distributed provides the exchange (NCCL between GPUs; gloo works for host-side tests);
the attention itself is whatever `attn` is, by default the library's bf16 tensor-core call.
Requires H and N divisible by the group size.
"""
import torch
import torch.distributed as dist


def _seq_to_heads(x, P, group):
    """[B, N/P, H, d] token shard -> [B, N, H/P, d] head shard (all tokens)."""
    B, Ns, H, d = x.shape
    Hp = H // P
    send = x.reshape(B, Ns, P, Hp, d).permute(2, 0, 1, 3, 4).contiguous()    # [P, B, Ns, Hp, d]
    recv = torch.empty_like(send)                                            # [P(src), B, Ns, Hp, d]
    dist.all_to_all_single(recv, send, group=group)
    return recv.permute(1, 0, 2, 3, 4).reshape(B, P * Ns, Hp, d).contiguous()


def _heads_to_seq(y, P, group):
    """[B, N, H/P, d] head shard -> [B, N/P, H, d] token shard."""
    B, N, Hp, d = y.shape
    Ns = N // P
    send = y.reshape(B, P, Ns, Hp, d).permute(1, 0, 2, 3, 4).contiguous()    # [P(dst), B, Ns, Hp, d]
    recv = torch.empty_like(send)                                            # [P(src), B, Ns, Hp, d]
    dist.all_to_all_single(recv, send, group=group)
    return recv.permute(1, 2, 0, 3, 4).reshape(B, Ns, P * Hp, d).contiguous()


def _lse_heads_to_seq(l, P, group):
    """[B, H/P, N] -> [B, H, N/P]."""
    B, Hp, N = l.shape
    Ns = N // P
    send = l.reshape(B, Hp, P, Ns).permute(2, 0, 1, 3).contiguous()          # [P(dst), B, Hp, Ns]
    recv = torch.empty_like(send)                                            # [P(src), B, Hp, Ns]
    dist.all_to_all_single(recv, send, group=group)
    return recv.permute(1, 0, 2, 3).reshape(B, P * Hp, Ns).contiguous()


def ulysses_rope3d_attn(q, k, v, grid, sections=(0, 0, 0), theta=10000.0, scale=0.0,
                        group=None, attn=None):
    """Attention of this rank's token shard q, k, v ([B, N/P, H, d], tokens
    [r*N/P, (r+1)*N/P) on rank r) over the whole sequence of the grid.  Returns this rank's
    out [B, N/P, H, d] and lse [B, H, N/P].  `attn(q, k, v, grid, sections, theta, scale)` must
    return (out [B, N, h, d], lse [B, h, N]); default: the library's rope3d_attn."""
    P = dist.get_world_size(group)
    B, Ns, H, d = q.shape
    T, Hg, Wg = grid
    if H % P or Ns * P != T * Hg * Wg:
        raise ValueError(f"heads ({H}) must divide by the group size ({P}) and the shards must "
                         f"tile the grid ({Ns} x {P} tokens vs {T * Hg * Wg})")
    if attn is None:
        from ._binding import rope3d_attn

        def attn(qq, kk, vv, grid_, sections_, theta_, scale_):
            return rope3d_attn(qq, kk, vv, grid_, sections_, theta_, scale_)
    qh, kh, vh = (_seq_to_heads(x, P, group) for x in (q, k, v))
    out_h, lse_h = attn(qh, kh, vh, grid, sections, theta, scale)
    return _heads_to_seq(out_h, P, group), _lse_heads_to_seq(lse_h, P, group)
