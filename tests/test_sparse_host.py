"""Block-mask host helpers of the C ABI (no GPU): the window mask builder against the oracle's
brute-force definition, word counts, packing, argument checks."""
import ctypes

import numpy as np
import pytest

import oracle.fp64 as O
import video_diffusion_transformer_rope_gb300 as vdx
from video_diffusion_transformer_rope_gb300 import _binding, _build


@pytest.fixture(scope="module", autouse=True)
def _built():
    _build.build()
    vdx.lib()


def _unpack(words, nk):
    bits = (words[..., :, None] >> np.arange(32, dtype=np.uint32)) & 1
    return bits.reshape(words.shape[:-1] + (-1,))[..., :nk].astype(bool)


@pytest.mark.parametrize("grid,window", [((3, 7, 20), (1, 2, 3)), ((4, 9, 13), (0, 0, 0)),
                                         ((2, 30, 52), (1, 4, 6)), ((5, 8, 16), (2, 1, 20)),
                                         ((21, 45, 80), (2, 6, 10)), ((3, 5, 7), (5, 9, 9)),
                                         ((1, 1, 1), (0, 0, 0))])
def test_window_mask_matches_oracle(grid, window):
    N = grid[0] * grid[1] * grid[2]
    if N > 20000:
        pytest.importorskip("numpy")
        # the oracle's pair scan is quadratic: check the C builder on a sample of query blocks
        words = vdx.window_block_mask(grid, window)
        full = _unpack(words, (N + 127) // 128)
        T, Hg, Wg = grid
        t, h, w = O.token_positions(T, Hg, Wg)
        rng = np.random.default_rng(0)
        for qb in rng.choice(full.shape[0], 4, replace=False):
            qs = slice(qb * 256, min(N, qb * 256 + 256))
            for kb in range(full.shape[1]):
                ks = slice(kb * 128, min(N, kb * 128 + 128))
                near = ((np.abs(t[qs][:, None] - t[ks][None, :]) <= window[0]) &
                        (np.abs(h[qs][:, None] - h[ks][None, :]) <= window[1]) &
                        (np.abs(w[qs][:, None] - w[ks][None, :]) <= window[2])).any()
                assert full[qb, kb] == near, (qb, kb)
        return
    words = vdx.window_block_mask(grid, window)
    ref = O.window_block_mask(grid, window)
    assert words.shape == (ref.shape[0], (ref.shape[1] + 31) // 32)
    assert np.array_equal(_unpack(words, ref.shape[1]), ref)


def test_pack_and_words():
    rng = np.random.default_rng(1)
    m = rng.random((2, 3, 5, 70)) < 0.3
    p = vdx.pack_block_mask(m)
    assert p.shape == (2, 3, 5, 3) and p.dtype == np.uint32
    assert np.array_equal(_unpack(p, 70), m)
    assert vdx.block_mask_words((21, 45, 80)) == (591 + 31) // 32
    assert vdx.lib().vdx_rope3d_block_mask_words(0, 1, 1) == 0


def test_window_mask_rejects_bad_arguments():
    L = vdx.lib()
    buf = np.zeros(16, dtype=np.uint32)
    assert L.vdx_window_block_mask(buf.ctypes.data_as(ctypes.c_void_p), 1, 2, 2, -1, 0, 0) == _binding.VDX_ERR_ARG
    assert L.vdx_window_block_mask(None, 1, 2, 2, 0, 0, 0) == _binding.VDX_ERR_ARG
    assert L.vdx_window_block_mask(buf.ctypes.data_as(ctypes.c_void_p), 0, 2, 2, 0, 0, 0) == _binding.VDX_ERR_ARG
