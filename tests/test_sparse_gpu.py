"""Block-sparse and windowed 3D-RoPE attention on the GPU (through the C ABI) against the fp64
block-sparse oracle.  Same tolerances as the dense bf16 path (out max-abs <= 2e-2, out
mean-abs <= 2e-3, lse max-abs <= 1e-3); rows with no selected key must give out = 0 and
lse = -inf exactly."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle.fp64 as O
import video_diffusion_transformer_rope_gb300 as vdx
from video_diffusion_transformer_rope_gb300 import configs, synth

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from video_diffusion_transformer_rope_gb300 import _build
    _build.build()
    vdx.lib()


def _compare(w, mask_bool, qk="fp16", dev=None):
    q, k, v = dev if dev is not None else (t.cuda() for t in synth.make_qkv(w))
    words = torch.from_numpy(vdx.pack_block_mask(mask_bool).astype(np.int32)).cuda()
    out, lse = vdx.rope3d_attn_sparse(q, k, v, (w.T, w.Hg, w.Wg), words, w.sections, w.theta,
                                      qk_precision=vdx.QK_MODES[qk])
    vdx.sync_check()
    ref_o, ref_l = O.rope3d_attention_blocksparse(q, k, v, (w.T, w.Hg, w.Wg), mask_bool,
                                                  sections=w.sections, theta=w.theta)
    got_o = out.double().cpu().numpy()
    got_l = lse.double().cpu().numpy()
    empty = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(got_l), empty)
    assert np.all(got_o.transpose(0, 2, 1, 3)[empty] == 0.0)
    err = np.abs(got_o - ref_o)
    lerr = np.abs(got_l[~empty] - ref_l[~empty]).max() if (~empty).any() else 0.0
    return err.max(), err.mean(), lerr


GRIDS = [(4, 9, 13), (5, 12, 20), (3, 8, 8), (1, 1, 700)]


@pytest.mark.parametrize("grid", GRIDS, ids=lambda g: "x".join(map(str, g)))
@pytest.mark.parametrize("density", [0.15, 0.5, 1.0])
def test_random_per_head_masks(grid, density):
    w = dataclasses.replace(configs.WAN13B_480P, B=2, H=3, T=grid[0], Hg=grid[1], Wg=grid[2], seed=51)
    N = w.N
    nq, nk = (N + 255) // 256, (N + 127) // 128
    rng = np.random.default_rng(int(density * 100) + N)
    mask = rng.random((w.B, w.H, nq, nk)) < density
    mask[0, 0, 0] = False            # one query block with no keys at all
    mask[1, 2, -1] = False
    mask[1, 2, -1, -1] = True        # only the ragged last key tile
    mx, mean, lerr = _compare(w, mask)
    assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL, (mx, mean, lerr)


def test_shared_mask_and_all_ones_equals_dense():
    w = dataclasses.replace(configs.WAN13B_480P, B=1, H=2, T=3, Hg=10, Wg=30, seed=52)
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    nq, nk = (w.N + 255) // 256, (w.N + 127) // 128
    ones = torch.from_numpy(vdx.pack_block_mask(np.ones((nq, nk), bool)).astype(np.int32)).cuda()
    o1, l1 = vdx.rope3d_attn_sparse(q, k, v, (w.T, w.Hg, w.Wg), ones)
    o2, l2 = vdx.rope3d_attn(q, k, v, (w.T, w.Hg, w.Wg))
    vdx.sync_check()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    rng = np.random.default_rng(3)
    shared = rng.random((nq, nk)) < 0.4
    mx, mean, lerr = _compare(w, shared, dev=(q, k, v))
    assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL


def test_split_precision_sparse_on_stress_inputs():
    w = dataclasses.replace(configs.LONG_STRESS, B=1, H=3, T=2, Hg=9, Wg=40, seed=53)
    nq, nk = (w.N + 255) // 256, (w.N + 127) // 128
    mask = np.random.default_rng(4).random((w.B, w.H, nq, nk)) < 0.5
    mask[..., 0] = True
    mx, mean, lerr = _compare(w, mask, qk="split")
    assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL, (mx, mean, lerr)


@pytest.mark.parametrize("grid,window", [((4, 12, 20), (1, 2, 3)), ((6, 8, 16), (0, 1, 1))])
def test_windowed_attention(grid, window):
    w = dataclasses.replace(configs.WAN13B_480P, B=2, H=2, T=grid[0], Hg=grid[1], Wg=grid[2], seed=54)
    words = vdx.window_block_mask(grid, window)
    mask = O.window_block_mask(grid, window)
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    out, lse = vdx.rope3d_attn_sparse(q, k, v, grid, torch.from_numpy(words.astype(np.int32)).cuda())
    vdx.sync_check()
    ref_o, ref_l = O.rope3d_attention_blocksparse(q, k, v, grid, mask)
    err = np.abs(out.double().cpu().numpy() - ref_o)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN
    assert np.abs(lse.double().cpu().numpy() - ref_l).max() <= LSE_TOL


def test_windowed_720p_sampled_rows():
    w = configs.WAN14B_720P
    grid = (w.T, w.Hg, w.Wg)
    window = (2, 6, 10)
    words = vdx.window_block_mask(grid, window)
    q, k, v = synth.make_qkv(w, device="cuda")
    out, lse = vdx.rope3d_attn_sparse(q, k, v, grid, torch.from_numpy(words.astype(np.int32)).cuda())
    vdx.sync_check()
    nk = (w.N + 127) // 128
    bits = (words[:, :, None] >> np.arange(32, dtype=np.uint32)) & 1
    mask = bits.reshape(words.shape[0], -1)[:, :nk].astype(bool)
    rows = synth.sample_rows(w, 256)
    ref_o, ref_l = O.rope3d_attention_blocksparse_rows(q, k, v, grid, rows, mask, sections=w.sections)
    b = torch.tensor([r[0] for r in rows], device="cuda")
    h = torch.tensor([r[1] for r in rows], device="cuda")
    n = torch.tensor([r[2] for r in rows], device="cuda")
    err = np.abs(out[b, n, h].double().cpu().numpy() - ref_o)
    lerr = np.abs(lse[b, h, n].double().cpu().numpy() - ref_l)
    print(f"windowed 720p (density {mask.mean():.3f}): out max {err.max():.3e} lse max {lerr.max():.3e}")
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN and lerr.max() <= LSE_TOL


def test_sparse_rejects_bad_masks():
    w = dataclasses.replace(configs.WAN13B_480P, B=1, H=1, T=1, Hg=2, Wg=64)
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    with pytest.raises(vdx.VdxError):
        vdx.rope3d_attn_sparse(q, k, v, (1, 2, 64), torch.zeros(3, 3, dtype=torch.int32, device="cuda"))
    vdx.sync_check()
