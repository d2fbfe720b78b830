"""Plant plausible mistakes into the oracle (on the CPU) and check that the pins catch each.

A mutant replaces one oracle function for the duration of a test; the test passes when at
least one pin of tests/oracle_pins.py then fails.
"""
import numpy as np
import pytest

import oracle.fp64 as O
from oracle_pins import ALL_PINS

_orig = {name: getattr(O, name) for name in
         ("rope_frequencies", "token_positions", "rope3d_angles", "apply_rotary",
          "attention_rows", "rope3d", "default_sections", "block_key_mask",
          "attention_rows_masked", "window_block_mask")}


def _freq_no_two(S, theta):            # dropped factor 2 in the exponent
    return np.power(float(theta), -np.arange(S // 2) / S)


def _freq_global_ladder(S, theta):     # one ladder over a fixed head_dim instead of per axis
    return np.power(float(theta), -2.0 * np.arange(S // 2) / 128.0)


def _pos_hw_swapped(T, Hg, Wg):
    t, h, w = _orig["token_positions"](T, Hg, Wg)
    return t, w, h


def _pos_row_major_wrong(T, Hg, Wg):   # w taken from the wrong stride
    n = np.arange(T * Hg * Wg)
    return n // (Hg * Wg), (n // Hg) % Wg, n % Hg


def _angles_axes_reversed(pt, ph, pw, sections, theta):
    return _orig["rope3d_angles"](pw, ph, pt, sections[::-1], theta)


def _rot_clockwise(x, angles):
    return _orig["apply_rotary"](x, -np.asarray(angles))


def _rot_half_split(x, angles):        # NeoX-style pairing (i, i + d/2)
    x = np.asarray(x, dtype=np.float64)
    h = x.shape[-1] // 2
    a, b = x[..., :h], x[..., h:]
    c, s = np.cos(angles), np.sin(angles)
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def _rot_cos_only(x, angles):          # dropped sin term
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    out[..., 0::2] = x[..., 0::2] * np.cos(angles)
    out[..., 1::2] = x[..., 1::2] * np.cos(angles)
    return out


def _attn_no_scale(qr, kr, v, scale):
    return _orig["attention_rows"](qr, kr, v, 1.0)


def _attn_lse_without_max(qr, kr, v, scale):
    o, lse = _orig["attention_rows"](qr, kr, v, scale)
    s = scale * (qr @ kr.T)
    return o, lse - s.max(axis=1)


def _attn_no_max_subtraction(qr, kr, v, scale):
    s = scale * (qr @ kr.T)
    with np.errstate(over="ignore", invalid="ignore"):
        p = np.exp(s)
        l = p.sum(axis=1, keepdims=True)
        return (p @ v) / l, np.log(l)[:, 0]


def _attn_unnormalised(qr, kr, v, scale):
    s = scale * (qr @ kr.T)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    return p @ v, (m + np.log(p.sum(axis=1, keepdims=True)))[:, 0]


def _rope3d_no_transpose(x_bnhd, grid, sections, theta):
    T, Hg, Wg = grid
    ang = _orig["rope3d_angles"](*_orig["token_positions"](T, Hg, Wg), sections, theta)
    x = np.asarray(x_bnhd, dtype=np.float64)
    B, N, H, d = x.shape
    y = _orig["apply_rotary"](x.reshape(B, H, N, d), ang)   # heads and tokens mixed up
    return y


def _sections_thirds(d):
    return (d // 3 + d % 3, d // 3, d // 3)


def _mask_blocks_swapped(mask_qk, N, qblock, kblock):     # query/key block sizes swapped
    return _orig["block_key_mask"](mask_qk, N, kblock, qblock)


def _mask_ignored(mask_qk, N, qblock, kblock):             # mask not applied
    return np.ones((N, N), dtype=bool)


def _masked_empty_rows_uniform(qr, kr, v, scale, allowed):  # empty rows fall back to dense
    allowed = allowed | ~allowed.any(axis=1, keepdims=True)
    return _orig["attention_rows_masked"](qr, kr, v, scale, allowed)


def _window_strict(grid, window, qblock=256, kblock=128):  # < instead of <=
    return _orig["window_block_mask"](grid, tuple(max(0, x - 1) for x in window), qblock, kblock)


MUTANTS = {
    "mask_blocks_swapped": ("block_key_mask", _mask_blocks_swapped),
    "mask_ignored": ("block_key_mask", _mask_ignored),
    "masked_empty_rows_dense": ("attention_rows_masked", _masked_empty_rows_uniform),
    "window_strict": ("window_block_mask", _window_strict),
    "freq_no_two": ("rope_frequencies", _freq_no_two),
    "freq_global_ladder": ("rope_frequencies", _freq_global_ladder),
    "pos_hw_swapped": ("token_positions", _pos_hw_swapped),
    "pos_wrong_stride": ("token_positions", _pos_row_major_wrong),
    "axes_reversed": ("rope3d_angles", _angles_axes_reversed),
    "rotate_clockwise": ("apply_rotary", _rot_clockwise),
    "half_split_pairs": ("apply_rotary", _rot_half_split),
    "rotate_cos_only": ("apply_rotary", _rot_cos_only),
    "attn_no_scale": ("attention_rows", _attn_no_scale),
    "lse_without_max": ("attention_rows", _attn_lse_without_max),
    "softmax_no_max_subtraction": ("attention_rows", _attn_no_max_subtraction),
    "attn_unnormalised": ("attention_rows", _attn_unnormalised),
    "heads_tokens_mixed": ("rope3d", _rope3d_no_transpose),
    "sections_thirds": ("default_sections", _sections_thirds),
}


def _fails(pin):
    try:
        with np.errstate(all="ignore"):
            pin(O)
    except Exception:
        return True
    return False


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    caught = [p.__name__ for p in ALL_PINS if _fails(p)]
    assert caught, f"no pin catches the planted mistake {name}"
