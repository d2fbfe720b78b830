"""Seeded input recipe: shapes, determinism, element type, stress outliers (CPU only)."""
import dataclasses

import pytest

import torch

from video_diffusion_transformer_rope_gb300 import configs, synth


def test_shapes_dtypes_determinism():
    w = configs.TINY_F32
    q, k, v = synth.make_qkv(w)
    assert q.shape == (1, 192, 4, 64) and q.dtype == torch.float32
    q2, _, _ = synth.make_qkv(w)
    assert torch.equal(q, q2)
    wb = dataclasses.replace(w, dtype="bf16", seed=5)
    qb, kb, vb = synth.make_qkv(wb)
    assert qb.dtype == torch.bfloat16 and not torch.equal(qb.float(), kb.float())


def test_stress_outliers():
    w = dataclasses.replace(configs.LONG_STRESS, T=2, Hg=9, Wg=80, H=4)   # N = 1440
    q, k, v = synth.make_qkv(w)
    ch, tok = synth.outlier_indices(w)
    assert ch.shape == (4, 1) and tok.numel() == round(0.001 * w.N)
    base = dataclasses.replace(w, stress=False)
    q0, k0, v0 = synth.make_qkv(base)
    assert torch.equal(v, v0)
    ratio = (q.float() / q0.float()).nan_to_num(1.0)
    for h in range(4):
        c = int(ch[h, 0])
        others = [n for n in range(w.N) if n not in set(tok.tolist())]
        r = ratio[0, others, h, c]
        assert torch.allclose(r, torch.full_like(r, 8.0), rtol=1e-2)
    t0 = int(tok[0])
    assert torch.allclose(ratio[0, t0, 0, :3], torch.full((3,), 4.0), rtol=1e-2) or int(ch[0, 0]) < 3


def test_sample_rows_cover_tail():
    w = configs.WAN14B_720P
    rows = synth.sample_rows(w, 512)
    assert len(rows) == 512 and len(set(rows)) == 512
    ns = [n for _, _, n in rows]
    assert 0 in ns and w.N - 1 in ns and any(n >= (w.N // 128) * 128 for n in ns)
    assert all(0 <= b < w.B and 0 <= h < w.H and 0 <= n < w.N for b, h, n in rows)


@pytest.mark.parametrize("grid", [(1, 255, 128), (1, 1, 128), (1, 1, 1), (3, 5, 7)])
def test_sample_rows_stay_in_range(grid):
    # N a multiple of 128 included: the last block starts at N - 128, not at N.
    w = dataclasses.replace(configs.WAN13B_480P, B=1, H=2, T=grid[0], Hg=grid[1], Wg=grid[2])
    rows = synth.sample_rows(w, 64)
    assert all(0 <= b < w.B and 0 <= h < w.H and 0 <= n < w.N for b, h, n in rows)
    assert any(n == ((w.N - 1) // 128) * 128 for _, _, n in rows)


def test_sample_rows_include_every_outlier_token_of_a_stress_workload():
    # The long-clip stress workload's outlier tokens (x4 on Q and K) carry its largest logits;
    # the sampled comparison must see every one of them as a query row.
    w = configs.LONG_STRESS
    _, tok = synth.outlier_indices(w)
    assert tok.numel() == 112
    rows = synth.sample_rows(w, 512)
    assert len(rows) == len(set(rows)) and 512 <= len(rows) <= 512 + 112
    by_token = {}
    for b, h, n in rows:
        by_token.setdefault(n, set()).add((b, h))
    for n in tok.tolist():
        assert n in by_token, n
    # spread over the heads, not all on one (b, h) pair
    outlier_bh = {bh for n in tok.tolist() for bh in by_token[n]}
    assert len(outlier_bh) >= min(w.B * w.H, 40)
    # an ordinary workload gets exactly `count` rows and no extra ones
    assert len(synth.sample_rows(configs.WAN14B_720P, 512)) == 512
