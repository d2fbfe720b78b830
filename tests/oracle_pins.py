"""Checks that pin the fp64 oracle to facts outside itself.

Each pin takes the oracle module and raises AssertionError when the oracle disagrees with a
closed form, a hand-derived value (tests/golden/), a library routine (torch fp64 attention,
logsumexp), or an invariant of rotary embeddings / softmax attention.  test_oracle.py runs
them on the real oracle; test_oracle_mutants.py plants plausible mistakes into the oracle
and checks that at least one pin catches each.
"""
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rows(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out.append(line.split())
    return out


def _rng(seed=0):
    return np.random.default_rng(seed)


def pin_token_index(O):
    """Token n of a T x Hg x Wg grid sits at (t, h, w) with n = t*Hg*Wg + h*Wg + w."""
    T, Hg, Wg = 3, 8, 8
    t, h, w = O.token_positions(T, Hg, Wg)
    n = 0
    for tt in range(T):
        for hh in range(Hg):
            for ww in range(Wg):
                assert (t[n], h[n], w[n]) == (tt, hh, ww), n
                n += 1
    t, h, w = O.token_positions(2, 3, 5)
    assert (t[22], h[22], w[22]) == (1, 1, 2)


def pin_default_sections(O):
    """The measured workloads state 24/20/20 at d=64 and 44/42/42 at d=128."""
    assert tuple(O.default_sections(64)) == (24, 20, 20)
    assert tuple(O.default_sections(128)) == (44, 42, 42)


def pin_frequencies_golden(O):
    for theta, S, j, omega in _rows("rope_frequencies.txt"):
        got = O.rope_frequencies(int(S), float(theta))[int(j)]
        assert abs(got - float(omega)) <= 1e-15 * max(1.0, float(omega)), (theta, S, j, got)
        assert len(O.rope_frequencies(int(S), float(theta))) == int(S) // 2


def _rope_tokens(O, x_nd, grid, sections, theta):
    """Rotate a [N, d] array through the oracle's [B, N, H, d] entry point."""
    out = O.rope3d(x_nd[None, :, None, :], grid, sections, theta)    # [1, 1, N, d]
    return out[0, 0]


def pin_worked_example(O):
    grid, sections, theta, d = (3, 8, 8), (24, 20, 20), 10000.0, 64
    N = 3 * 8 * 8
    for tok, ch, e0, e1 in _rows("rope3d_worked_example.txt"):
        tok, ch = int(tok), int(ch)
        x = np.zeros((N, d))
        x[tok, ch] = 1.0
        y = _rope_tokens(O, x, grid, sections, theta)
        assert abs(y[tok, ch] - float(e0)) < 1e-14 and abs(y[tok, ch + 1] - float(e1)) < 1e-14, \
            (tok, ch, y[tok, ch], y[tok, ch + 1])
        rest = np.delete(y[tok], [ch, ch + 1])
        assert np.all(rest == 0.0)


def pin_identity_at_origin(O):
    """Token 0 is at (0,0,0): every angle is 0 and RoPE leaves it bit-for-bit unchanged."""
    x = _rng(1).standard_normal((1, 4, 3, 64))
    y = O.rope3d(x, (1, 2, 2), (24, 20, 20), 10000.0)      # [1, 3, 4, 64]
    assert np.array_equal(y[0, :, 0, :], x[0, 0, :, :])


def pin_pair_norm_and_orthogonality(O):
    """Each rotated pair keeps its length; the map is linear and orthogonal."""
    grid, sections, theta = (3, 5, 7), (44, 42, 42), 10000.0
    N, d = 105, 128
    x = _rng(2).standard_normal((N, d))
    y = _rope_tokens(O, x, grid, sections, theta)
    nx = np.hypot(x[:, 0::2], x[:, 1::2])
    ny = np.hypot(y[:, 0::2], y[:, 1::2])
    assert np.max(np.abs(nx - ny)) < 1e-13
    # d x d matrix of one token, built column by column from unit vectors: orthogonal, det 1.
    tok = 77
    cols = np.zeros((N, d, d))
    for c in range(d):
        e = np.zeros((N, d))
        e[tok, c] = 1.0
        cols[:, :, c] = _rope_tokens(O, e, grid, sections, theta)
    R = cols[tok]
    assert np.allclose(R @ R.T, np.eye(d), atol=1e-13)
    assert abs(np.linalg.det(R) - 1.0) < 1e-10
    # block-diagonal with 2x2 blocks only (adjacent-pair convention)
    mask = np.kron(np.eye(d // 2), np.ones((2, 2)))
    assert np.all(R[mask == 0] == 0.0)
    # linear: R x equals the oracle's rotation of x
    assert np.allclose(R @ x[tok], y[tok], atol=1e-13)


def pin_complex_form(O):
    """Pair i, viewed as x[2i] + i x[2i+1], is multiplied by exp(i * angle) (counter-clockwise)."""
    grid, sections, theta = (4, 3, 6), (24, 20, 20), 10000.0
    N, d = 72, 64
    x = _rng(3).standard_normal((N, d))
    y = _rope_tokens(O, x, grid, sections, theta)
    t, h, w = np.divmod(np.arange(N), 18)[0], (np.arange(N) // 6) % 3, np.arange(N) % 6
    # angles from the axis positions and this test's own frequency ladders: with
    # theta = 10^4, theta^(-2j/S) = 10^(-8j/S)
    lad_t = 10.0 ** (-8.0 * np.arange(12) / 24)
    lad_hw = 10.0 ** (-8.0 * np.arange(10) / 20)
    ang = np.concatenate([t[:, None] * lad_t, h[:, None] * lad_hw, w[:, None] * lad_hw], axis=1)
    z = (x[:, 0::2] + 1j * x[:, 1::2]) * np.exp(1j * ang)
    assert np.max(np.abs(z.real - y[:, 0::2])) < 1e-13
    assert np.max(np.abs(z.imag - y[:, 1::2])) < 1e-13


def pin_relative_position(O):
    """<R(p) q, R(p') k> depends only on p - p': shifting every position by the same
    (dt, dh, dw) leaves all dot products unchanged."""
    sections, theta, d = (44, 42, 42), 10000.0, 128
    rng = _rng(4)
    q = rng.standard_normal((16, d))
    k = rng.standard_normal((16, d))
    pos = [rng.integers(0, 20, 16) for _ in range(3)]
    shift = (7, 13, 29)
    a0 = O.rope3d_angles(*pos, sections, theta)
    a1 = O.rope3d_angles(*[p + s for p, s in zip(pos, shift)], sections, theta)
    dots0 = O.apply_rotary(q, a0) @ O.apply_rotary(k, a0).T
    dots1 = O.apply_rotary(q, a1) @ O.apply_rotary(k, a1).T
    assert np.max(np.abs(dots0 - dots1)) < 1e-11
    # and they do change when only one side moves (the embedding is not trivial)
    a2 = O.rope3d_angles(pos[0] + 1, pos[1], pos[2], sections, theta)
    dots2 = O.apply_rotary(q, a2) @ O.apply_rotary(k, a0).T
    assert np.max(np.abs(dots2 - dots0)) > 1e-3


def pin_one_axis_reduces_to_1d(O):
    """With the h and w sections empty, 3D RoPE is ordinary 1D RoPE along the frame index."""
    d, T = 16, 6
    x = _rng(5).standard_normal((T, d))
    y = _rope_tokens(O, x, (T, 1, 1), (d, 0, 0), 100.0)
    lad = 100.0 ** (-np.arange(d // 2) * 2.0 / d)
    z = (x[:, 0::2] + 1j * x[:, 1::2]) * np.exp(1j * np.arange(T)[:, None] * lad)
    assert np.allclose(y[:, 0::2], z.real, atol=1e-14) and np.allclose(y[:, 1::2], z.imag, atol=1e-14)


def _sdpa_reference(qr, kr, v, scale):
    """torch fp64 attention (math path) and logsumexp on already-rotated [B, H, N, d]."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(a)) for a in (qr, kr, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)
    lse = torch.logsumexp(torch.matmul(tq, tk.transpose(-1, -2)) * scale, dim=-1)
    return o.numpy(), lse.numpy()


def pin_attention_vs_torch(O):
    """Full oracle equals torch's fp64 scaled-dot-product attention on the rotated operands."""
    B, H, d, grid = 2, 3, 64, (3, 4, 5)
    N = 60
    rng = _rng(6)
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    sections, theta = (24, 20, 20), 10000.0
    out, lse = O.rope3d_attention(q, k, v, grid, sections, theta)
    qr = O.rope3d(q, grid, sections, theta)
    kr = O.rope3d(k, grid, sections, theta)
    ref_o, ref_lse = _sdpa_reference(qr, kr, v.transpose(0, 2, 1, 3), d ** -0.5)
    assert out.shape == (B, N, H, d) and lse.shape == (B, H, N)
    assert np.max(np.abs(out.transpose(0, 2, 1, 3) - ref_o)) < 1e-12
    assert np.max(np.abs(lse - ref_lse)) < 1e-12
    # explicit scale is honoured (torch's default is 1/sqrt(d); this one is not)
    out2, lse2 = O.rope3d_attention(q, k, v, grid, sections, theta, scale=0.3)
    ref_o2, ref_lse2 = _sdpa_reference(qr, kr, v.transpose(0, 2, 1, 3), 0.3)
    assert np.max(np.abs(out2.transpose(0, 2, 1, 3) - ref_o2)) < 1e-12
    assert np.max(np.abs(lse2 - ref_lse2)) < 1e-12


def pin_attention_large_logits(O):
    """Logits in the hundreds: still finite and equal to torch's fp64 result."""
    B, H, d, grid = 1, 2, 64, (2, 3, 4)
    rng = _rng(7)
    q, k, v = (rng.standard_normal((B, 24, H, d)) for _ in range(3))
    q *= 30.0
    k *= 30.0
    out, lse = O.rope3d_attention(q, k, v, grid)
    qr = O.rope3d(q, grid, (24, 20, 20), 10000.0)
    kr = O.rope3d(k, grid, (24, 20, 20), 10000.0)
    ref_o, ref_lse = _sdpa_reference(qr, kr, v.transpose(0, 2, 1, 3), d ** -0.5)
    assert np.all(np.isfinite(out)) and np.max(np.abs(lse)) > 100
    assert np.max(np.abs(out.transpose(0, 2, 1, 3) - ref_o)) < 1e-10
    assert np.max(np.abs(lse - ref_lse)) < 1e-10


def pin_single_token(O):
    """N = 1: the output is v itself and lse is the one scaled logit (token 0 is unrotated)."""
    rng = _rng(8)
    q, k, v = (rng.standard_normal((1, 1, 2, 64)) for _ in range(3))
    out, lse = O.rope3d_attention(q, k, v, (1, 1, 1))
    assert np.allclose(out, v, atol=1e-15, rtol=0)
    for h in range(2):
        assert abs(lse[0, h, 0] - np.dot(q[0, 0, h], k[0, 0, h]) / 8.0) < 1e-14


def pin_uniform_attention(O):
    """Zero keys (or zero queries) make every weight equal: o = mean of V, lse = ln N."""
    rng = _rng(9)
    grid = (2, 3, 4)
    N = 24
    q, v = rng.standard_normal((1, N, 2, 64)), rng.standard_normal((1, N, 2, 64))
    k = np.zeros_like(q)
    for qq, kk in ((q, k), (k, q)):
        out, lse = O.rope3d_attention(qq, kk, v, grid)
        assert np.allclose(out, v.mean(axis=1, keepdims=True), atol=1e-14)
        assert np.allclose(lse, np.log(N), atol=1e-14)


def pin_equal_rotated_keys(O):
    """All rotated keys equal to one vector k': o = mean of V, lse = scale*<q', k'> + ln N."""
    rng = _rng(10)
    qr = rng.standard_normal((5, 32))
    kr = np.tile(rng.standard_normal((1, 32)), (40, 1))
    v = rng.standard_normal((40, 32))
    o, lse = O.attention_rows(qr, kr, v, 0.25)
    assert np.allclose(o, v.mean(axis=0)[None, :], atol=1e-14)
    assert np.allclose(lse, 0.25 * qr @ kr[0] + np.log(40), atol=1e-13)


def pin_key_permutation(O):
    """Permuting (rotated) key/value tokens together leaves the attention output unchanged."""
    rng = _rng(11)
    qr, kr, v = rng.standard_normal((7, 32)), rng.standard_normal((50, 32)), rng.standard_normal((50, 32))
    perm = rng.permutation(50)
    o1, l1 = O.attention_rows(qr, kr, v, 0.2)
    o2, l2 = O.attention_rows(qr, kr[perm], v[perm], 0.2)
    assert np.allclose(o1, o2, atol=1e-14) and np.allclose(l1, l2, atol=1e-14)


def pin_rows_match_full(O):
    """The sampled-row entry point gives the same rows as the full oracle."""
    rng = _rng(12)
    B, N, H, d, grid = 2, 30, 3, 64, (2, 3, 5)
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    out, lse = O.rope3d_attention(q, k, v, grid)
    rows = [(0, 0, 0), (1, 2, 29), (0, 1, 17), (1, 0, 5), (1, 0, 6)]
    o, l = O.rope3d_attention_rows(q, k, v, grid, rows)
    for i, (b, h, n) in enumerate(rows):
        assert np.allclose(o[i], out[b, n, h], atol=1e-14)
        assert abs(l[i] - lse[b, h, n]) < 1e-14
    tq, tk, tv = (torch.from_numpy(a) for a in (q, k, v))
    o_t, l_t = O.rope3d_attention_rows(tq, tk, tv, grid, rows)
    assert np.allclose(o_t, o, atol=1e-15) and np.allclose(l_t, l, atol=1e-15)


def _rotated(O, B, N, H, d, grid, seed):
    rng = _rng(seed)
    q, k, v = (rng.standard_normal((B, N, H, d)) for _ in range(3))
    return q, k, v, O.rope3d(q, grid, (24, 20, 20), 10000.0), O.rope3d(k, grid, (24, 20, 20), 10000.0)


def pin_blocksparse_all_blocks_is_dense(O):
    """A mask with every block set is the dense oracle, bit for bit."""
    B, H, d, grid = 1, 2, 64, (2, 5, 60)
    N = 600
    q, k, v, _, _ = _rotated(O, B, N, H, d, grid, 13)
    dense_o, dense_l = O.rope3d_attention(q, k, v, grid)
    mask = np.ones((3, 5), dtype=bool)
    o, l = O.rope3d_attention_blocksparse(q, k, v, grid, mask)
    assert np.array_equal(o, dense_o) and np.array_equal(l, dense_l)


def pin_blocksparse_vs_torch_masked(O):
    """Random block masks (every query block keeps at least one key block) equal torch's fp64
    attention with a boolean attn_mask built from the block structure by this test."""
    B, H, d, grid = 2, 2, 64, (3, 4, 50)
    N = 600
    q, k, v, qr, kr = _rotated(O, B, N, H, d, grid, 14)
    rng = _rng(15)
    nq, nk = (N + 255) // 256, (N + 127) // 128
    mask = rng.random((B, H, nq, nk)) < 0.4
    mask[..., 0, 2] = True
    mask[..., 1, 0] = True
    mask[..., 2, 4] = True
    o, l = O.rope3d_attention_blocksparse(q, k, v, grid, mask)
    for b in range(B):
        for h in range(H):
            allowed = np.zeros((N, N), dtype=bool)
            for n in range(0, N, 8):                       # rows in steps (same block rows)
                for m in range(N):
                    allowed[n:n + 8, m] = mask[b, h, n // 256, m // 128]
            tq = torch.from_numpy(np.ascontiguousarray(qr[b, h]))[None]
            tk = torch.from_numpy(np.ascontiguousarray(kr[b, h]))[None]
            tv = torch.from_numpy(np.ascontiguousarray(v[b, :, h]))[None]
            ta = torch.from_numpy(allowed)[None]
            ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=ta)[0].numpy()
            sc = (tq[0] @ tk[0].T) * d ** -0.5
            ref_l = torch.logsumexp(sc.masked_fill(~ta[0], float("-inf")), dim=-1).numpy()
            assert np.max(np.abs(o[b, :, h] - ref)) < 1e-12
            assert np.max(np.abs(l[b, h] - ref_l)) < 1e-12


def pin_blocksparse_single_block_and_empty(O):
    """One key block: attention over exactly those (rotated) keys; no block: o = 0, lse = -inf."""
    B, H, d, grid = 1, 1, 64, (1, 6, 50)
    N = 300
    q, k, v, qr, kr = _rotated(O, B, N, H, d, grid, 16)
    mask = np.zeros((2, 3), dtype=bool)
    mask[0, 1] = True                                   # query rows 0-255 see keys 128-255
    o, l = O.rope3d_attention_blocksparse(q, k, v, grid, mask)
    s = (qr[0, 0, :256] @ kr[0, 0, 128:256].T) * d ** -0.5
    ref_l = np.log(np.exp(s - s.max(1, keepdims=True)).sum(1)) + s.max(1)
    ref_o = np.exp(s - ref_l[:, None]) @ v[0, 128:256, 0]
    assert np.max(np.abs(o[0, :256, 0] - ref_o)) < 1e-12 and np.max(np.abs(l[0, 0, :256] - ref_l)) < 1e-12
    assert np.all(o[0, 256:, 0] == 0.0) and np.all(np.isneginf(l[0, 0, 256:]))


def pin_window_block_mask_brute_force(O):
    """Window block mask against a pair-by-pair scan written out here."""
    grid, window = (3, 7, 20), (1, 2, 3)
    T, Hg, Wg = grid
    N = T * Hg * Wg
    mask = O.window_block_mask(grid, window)
    ref = np.zeros(((N + 255) // 256, (N + 127) // 128), dtype=bool)
    for a in range(N):
        ta, ha, wa = a // (Hg * Wg), (a // Wg) % Hg, a % Wg
        for c in range(N):
            tc, hc, wc = c // (Hg * Wg), (c // Wg) % Hg, c % Wg
            if abs(ta - tc) <= 1 and abs(ha - hc) <= 2 and abs(wa - wc) <= 3:
                ref[a // 256, c // 128] = True
    assert np.array_equal(mask, ref)
    assert O.window_block_mask(grid, (T, Hg, Wg)).all()


def pin_blocksparse_rows_match_full(O):
    """The sampled-row block-sparse entry gives the full block-sparse oracle's rows."""
    B, H, d, grid = 2, 2, 64, (2, 5, 60)
    N = 600
    q, k, v, _, _ = _rotated(O, B, N, H, d, grid, 17)
    mask = _rng(18).random((B, H, 3, 5)) < 0.5
    mask[0, 1, 2] = False                      # an empty query block
    out, lse = O.rope3d_attention_blocksparse(q, k, v, grid, mask)
    rows = [(0, 0, 0), (1, 1, 599), (0, 1, 550), (1, 0, 300), (0, 1, 511)]
    o, l = O.rope3d_attention_blocksparse_rows(q, k, v, grid, rows, mask)
    for i, (b, h, n) in enumerate(rows):
        assert np.allclose(o[i], out[b, n, h], atol=1e-14, rtol=0)
        assert (np.isneginf(l[i]) and np.isneginf(lse[b, h, n])) or abs(l[i] - lse[b, h, n]) < 1e-14


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
