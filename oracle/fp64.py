"""fp64 CPU oracle for 3D-RoPE full spatiotemporal self-attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module: it is used by
tests/, by __graft_entry__.smoke() to check one small GPU call, and by bench.py's CPU
baseline leg.  It shares no code, table or helper with the CUDA library.

What it computes (for every batch b, head h and query token n of a latent grid T x Hg x Wg):

    q'_n = R(n) q_n,  k'_m = R(m) k_m                       (3D rotary embedding)
    s_nm = scale * <q'_n, k'_m>                             (all m: full, non-causal)
    lse_n = log sum_m exp(s_nm)                             (natural log)
    o_n  = sum_m exp(s_nm - lse_n) v_m

Sources.  The vidax page ("vidax: A Unified JAX Framework for Video Generative Models on
Accelerator Meshes", §2 "3D RoPE, 3D VAEs, and flash attention") names 3D RoPE and a flash
attention that never materialises the quadratic query-key matrix; §1 "Motivation and gap"
gives the tens-of-thousands-token regime.  The pages print no formula for either step, so
the definition is the plain one for Wan-style rotary embeddings, with these readings:

  * head_dim is split into three rotary sections (t, h, w) in that order; default sizes
    t = d - 4*floor(d/6), h = w = 2*floor(d/6)  (24/20/20 at d=64, 44/42/42 at d=128);
  * pairs are adjacent channels (2i, 2i+1), rotated like a complex number times e^{i*angle};
  * each axis has its own frequency ladder w_{a,j} = theta^(-2j/S_a), j < S_a/2;
  * positions are the integer grid coordinates from 0: t = n // (Hg*Wg),
    h = (n // Wg) % Hg, w = n % Wg;
  * scale defaults to 1/sqrt(d); lse is in natural-log units of the scaled logits.

Layout: q, k, v, out are [B, N, H, d]; lse is [B, H, N].

Pins (tests/test_oracle.py): rotation orthogonality and per-pair norm, identity at the
origin, the relative-position property, hand-derived frequency values (tests/golden/),
the complex-number form, the d x d rotation-matrix form, torch's fp64 scaled-dot-product
attention and logsumexp on the rotated operands, N=1, zero keys, key permutation.
"""
import numpy as np


def default_sections(d):
    """Rotary dims per axis (t, h, w) when the caller gives none (Wan-style split)."""
    hw = 2 * (d // 6)
    return (d - 2 * hw, hw, hw)


def token_positions(T, Hg, Wg):
    """Integer (t, h, w) of every token n = t*Hg*Wg + h*Wg + w, as three int64 arrays."""
    n = np.arange(T * Hg * Wg, dtype=np.int64)
    return n // (Hg * Wg), (n // Wg) % Hg, n % Wg


def rope_frequencies(S, theta):
    """Angular frequencies of one axis with S rotary dims: theta^(-2j/S), j = 0..S/2-1."""
    j = np.arange(S // 2, dtype=np.float64)
    return np.power(np.float64(theta), -2.0 * j / S)


def rope3d_angles(pos_t, pos_h, pos_w, sections, theta):
    """Rotation angle of every (token, pair): shape [n_tokens, d/2], fp64.

    Pairs 0..S_t/2-1 turn with the frame index, the next S_h/2 with the row, the last
    S_w/2 with the column.
    """
    parts = []
    for pos, S in zip((pos_t, pos_h, pos_w), sections):
        if S == 0:
            continue
        parts.append(np.asarray(pos, dtype=np.float64)[:, None] * rope_frequencies(S, theta)[None, :])
    return np.concatenate(parts, axis=1)


def apply_rotary(x, angles):
    """Rotate adjacent pairs (x[2i], x[2i+1]) of the last axis by angles[..., i].

    x: [..., n_tokens, d] (tokens on the second-to-last axis), angles: [n_tokens, d/2].
    """
    x = np.asarray(x, dtype=np.float64)
    xe = x[..., 0::2]
    xo = x[..., 1::2]
    c = np.cos(angles)
    s = np.sin(angles)
    out = np.empty_like(x)
    out[..., 0::2] = xe * c - xo * s
    out[..., 1::2] = xe * s + xo * c
    return out


def rope3d(x_bnhd, grid, sections, theta):
    """3D RoPE of a [B, N, H, d] tensor: returns [B, H, N, d] fp64 (head-major for matmuls)."""
    T, Hg, Wg = grid
    ang = rope3d_angles(*token_positions(T, Hg, Wg), sections, theta)
    x = np.asarray(x_bnhd, dtype=np.float64).transpose(0, 2, 1, 3)   # [B, H, N, d]
    return apply_rotary(x, ang)


def attention_rows(qr, kr, v, scale):
    """Softmax attention of query rows qr [R, d] over keys kr [M, d] / values v [M, d].

    Returns (o [R, d], lse [R]) with lse = log sum_m exp(scale * qr.kr_m).
    """
    s = scale * (qr @ kr.T)                          # [R, M]
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    o = (p @ v) / l
    lse = (m + np.log(l))[:, 0]
    return o, lse


def _to64(x):
    if hasattr(x, "detach"):      # a torch tensor: widen to fp64 on the CPU
        import torch
        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def rope3d_attention(q, k, v, grid, sections=None, theta=10000.0, scale=None):
    """Full oracle: out [B, N, H, d] and lse [B, H, N], fp64."""
    q, k, v = _to64(q), _to64(k), _to64(v)
    B, N, H, d = q.shape
    sections = tuple(sections) if sections else default_sections(d)
    scale = d ** -0.5 if scale is None else scale
    qr = rope3d(q, grid, sections, theta)
    kr = rope3d(k, grid, sections, theta)
    vv = v.transpose(0, 2, 1, 3)
    out = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            out[b, h], lse[b, h] = attention_rows(qr[b, h], kr[b, h], vv[b, h], scale)
    return out.transpose(0, 2, 1, 3), lse


def rope3d_attention_rows(q, k, v, grid, rows, sections=None, theta=10000.0, scale=None):
    """Oracle on selected query rows only: rows is a list of (b, h, n).

    K/V of a head are rotated once for all rows of that head.  Returns (o [R, d], lse [R])
    in the order of `rows`.
    """
    B, N, H, d = q.shape
    sections = tuple(sections) if sections else default_sections(d)
    scale = d ** -0.5 if scale is None else scale
    T, Hg, Wg = grid
    pt, ph, pw = token_positions(T, Hg, Wg)
    by_head = {}
    for i, (b, h, n) in enumerate(rows):
        by_head.setdefault((b, h), []).append((i, n))
    o = np.empty((len(rows), d))
    lse = np.empty(len(rows))
    for (b, h), items in by_head.items():
        kh = _to64(k[b, :, h, :])
        vh = _to64(v[b, :, h, :])
        kr = apply_rotary(kh, rope3d_angles(pt, ph, pw, sections, theta))
        idx = np.array([n for _, n in items])
        if hasattr(q, "detach"):
            import torch
            qh = _to64(q[b, :, h, :][torch.from_numpy(idx).to(q.device)])
        else:
            qh = _to64(q[b, idx, h, :])
        qr = apply_rotary(qh, rope3d_angles(pt[idx], ph[idx], pw[idx], sections, theta))
        oo, ll = attention_rows(qr, kr, vh, scale)
        for j, (i, _) in enumerate(items):
            o[i] = oo[j]
            lse[i] = ll[j]
    return o, lse


# ---------------------------------------------------------------------------------------------
# Block-sparse variant (ScalingAttention's "bit-wise block-sparse kernel", named on the first
# page; the block masks themselves come from trained weights there, synthetic here).
#
# Definition: the keys are cut into blocks of `kblock` consecutive tokens and the queries into
# blocks of `qblock` consecutive tokens; query n attends only to the keys of the blocks that
# the mask marks for its query block.  A query whose mask row is empty has no keys: its
# output is 0 and its lse is -inf.  mask: bool array [B, H, n_qblocks, n_kblocks] (or
# [n_qblocks, n_kblocks], shared by every (b, h)).

def block_key_mask(mask_qk, N, qblock, kblock):
    """Expand a [n_qblocks, n_kblocks] block mask to a [N, N] bool matrix (query, key)."""
    qb = np.arange(N) // qblock
    kb = np.arange(N) // kblock
    return np.asarray(mask_qk, dtype=bool)[qb[:, None], kb[None, :]]


def attention_rows_masked(qr, kr, v, scale, allowed):
    """attention_rows restricted to allowed[r, m] keys; rows with no key give o = 0, lse = -inf."""
    s = scale * (qr @ kr.T)
    s = np.where(allowed, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    empty = ~np.isfinite(m[:, 0])
    m = np.where(np.isfinite(m), m, 0.0)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(empty[:, None], 0.0, (p @ v) / np.where(l > 0, l, 1.0))
        lse = np.where(empty, -np.inf, (m + np.log(np.where(l > 0, l, 1.0)))[:, 0])
    return o, lse


def rope3d_attention_blocksparse(q, k, v, grid, mask, qblock=256, kblock=128, sections=None,
                                 theta=10000.0, scale=None):
    """Block-sparse oracle: out [B, N, H, d], lse [B, H, N] (fp64)."""
    q, k, v = _to64(q), _to64(k), _to64(v)
    B, N, H, d = q.shape
    sections = tuple(sections) if sections else default_sections(d)
    scale = d ** -0.5 if scale is None else scale
    mask = np.asarray(mask, dtype=bool)
    qr = rope3d(q, grid, sections, theta)
    kr = rope3d(k, grid, sections, theta)
    vv = v.transpose(0, 2, 1, 3)
    out = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            mk = mask if mask.ndim == 2 else mask[b, h]
            allowed = block_key_mask(mk, N, qblock, kblock)
            out[b, h], lse[b, h] = attention_rows_masked(qr[b, h], kr[b, h], vv[b, h], scale, allowed)
    return out.transpose(0, 2, 1, 3), lse


# ---------------------------------------------------------------------------------------------
# Windowed 3D attention (the windowed-attention primitive of the vidax page, §2 "3D RoPE, 3D
# VAEs, and flash attention"), at block granularity: query block Qb attends to key block Kb
# when some query of Qb and some key of Kb lie within (wt, wh, ww) of each other on every
# grid axis (|dt| <= wt, |dh| <= wh, |dw| <= ww).  Expressed as a block mask for the
# block-sparse definition above.

def window_block_mask(grid, window, qblock=256, kblock=128):
    T, Hg, Wg = grid
    wt, wh, ww = window
    N = T * Hg * Wg
    t, h, w = token_positions(T, Hg, Wg)
    nq = (N + qblock - 1) // qblock
    nk = (N + kblock - 1) // kblock
    mask = np.zeros((nq, nk), dtype=bool)
    for qb in range(nq):
        qs = slice(qb * qblock, min(N, (qb + 1) * qblock))
        for kb in range(nk):
            ks = slice(kb * kblock, min(N, (kb + 1) * kblock))
            near = ((np.abs(t[qs][:, None] - t[ks][None, :]) <= wt) &
                    (np.abs(h[qs][:, None] - h[ks][None, :]) <= wh) &
                    (np.abs(w[qs][:, None] - w[ks][None, :]) <= ww))
            mask[qb, kb] = bool(near.any())
    return mask


def rope3d_attention_blocksparse_rows(q, k, v, grid, rows, mask, qblock=256, kblock=128,
                                      sections=None, theta=10000.0, scale=None):
    """Block-sparse oracle on selected query rows (b, h, n); returns (o [R, d], lse [R])."""
    B, N, H, d = q.shape
    sections = tuple(sections) if sections else default_sections(d)
    scale = d ** -0.5 if scale is None else scale
    mask = np.asarray(mask, dtype=bool)
    T, Hg, Wg = grid
    pt, ph, pw = token_positions(T, Hg, Wg)
    by_head = {}
    for i, (b, h, n) in enumerate(rows):
        by_head.setdefault((b, h), []).append((i, n))
    o = np.empty((len(rows), d))
    lse = np.empty(len(rows))
    kb_of = np.arange(N) // kblock
    for (b, h), items in by_head.items():
        kr = apply_rotary(_to64(k[b, :, h, :]), rope3d_angles(pt, ph, pw, sections, theta))
        vh = _to64(v[b, :, h, :])
        mk = mask if mask.ndim == 2 else mask[b, h]
        idx = np.array([n for _, n in items])
        if hasattr(q, "detach"):
            import torch
            qh = _to64(q[b, :, h, :][torch.from_numpy(idx).to(q.device)])
        else:
            qh = _to64(q[b, idx, h, :])
        qr = apply_rotary(qh, rope3d_angles(pt[idx], ph[idx], pw[idx], sections, theta))
        allowed = mk[(idx // qblock)[:, None], kb_of[None, :]]
        oo, ll = attention_rows_masked(qr, kr, vh, scale, allowed)
        for j, (i, _) in enumerate(items):
            o[i] = oo[j]
            lse[i] = ll[j]
    return o, lse
