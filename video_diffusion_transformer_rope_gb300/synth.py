"""Seeded synthetic inputs shared by the CUDA path's tests/bench and by the oracle.

This module only draws random numbers and rounds them to the workload's element type; it
holds none of the attention or rotary arithmetic.  The same tensor (after rounding) is what
both sides see: the GPU gets it on the device, the oracle gets it widened to fp64.

Recipe (Wan-shaped self-attention inputs, layout [B, N, H, d]):
  * Q, K, V ~ N(0, 1) iid, drawn in fp32 from a torch.Generator seeded with the workload
    seed, then rounded once to the workload dtype.
  * Stress workloads additionally scale, before rounding, round(0.01*d) channels per head
    (picked per head by a seeded CPU generator; the same channel in Q and K) by 8, and
    round(0.001*N) tokens (seeded; all heads, Q and K rows) by 4.  V is left as drawn.
"""
import torch

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def outlier_indices(w):
    """Seeded outlier channel per head (list of index tensors) and outlier token indices."""
    g = torch.Generator(device="cpu").manual_seed(w.seed + 1000)
    n_ch = max(1, round(0.01 * w.d))
    n_tok = max(1, round(0.001 * w.N))
    ch = torch.stack([torch.randperm(w.d, generator=g)[:n_ch] for _ in range(w.H)])  # [H, n_ch]
    tok = torch.randperm(w.N, generator=g)[:n_tok]
    return ch, tok


def make_qkv(w, device="cpu"):
    """Return (q, k, v) of shape [B, N, H, d] in the workload dtype on `device`.

    CPU draws use a CPU generator, CUDA draws a CUDA generator: values differ between the
    two, so a test takes one tensor set and hands the very same values to both sides.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(w.seed)
    shape = (w.B, w.N, w.H, w.d)
    out = []
    for which in ("q", "k", "v"):
        x = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
        if w.stress and which in ("q", "k"):
            ch, tok = outlier_indices(w)
            ch = ch.to(dev)
            tok = tok.to(dev)
            heads = torch.arange(w.H, device=dev)[:, None].expand_as(ch)
            x[:, :, heads, ch] *= 8.0
            x[:, tok, :, :] *= 4.0
        out.append(x.to(_DTYPES[w.dtype]).contiguous())
    return tuple(out)


def sample_rows(w, count=512, seed=None):
    """Seeded (b, h, n) query rows for sampled comparison at large N.

    Always includes the first and last token and rows from the final (ragged) 128-row
    block, spread over every (b, h) pair; `count` rows in all, drawn uniformly otherwise.
    For a stress workload every outlier token (outlier_indices) is added on top, each on one
    (b, h) pair, taking the pairs in turn: those rows hold the largest logits, and a uniform
    draw of a few hundred rows out of B*H*N would almost never pick one.
    """
    g = torch.Generator(device="cpu").manual_seed(w.seed + 2000 if seed is None else seed)
    rows = set()
    bh = [(b, h) for b in range(w.B) for h in range(w.H)]
    fixed_n = [0, w.N - 1, ((w.N - 1) // 128) * 128, max(0, w.N - 2)]   # start of the last 128-row block
    for i, n in enumerate(fixed_n):
        b, h = bh[i % len(bh)]
        rows.add((b, h, n))
    count = min(count, w.B * w.H * w.N)
    while len(rows) < count:
        i = int(torch.randint(len(bh), (1,), generator=g))
        n = int(torch.randint(w.N, (1,), generator=g))
        b, h = bh[i]
        rows.add((b, h, n))
    if w.stress:
        _, tok = outlier_indices(w)
        for i, n in enumerate(sorted(int(x) for x in tok)):
            b, h = bh[i % len(bh)]
            rows.add((b, h, n))
    return sorted(rows)
