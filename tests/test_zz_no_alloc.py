"""vdx_rope3d_attn_noalloc: the entry point for callers that cannot allocate device memory at
call time (a frozen memory pool, an allocator-free embedding, a host that sizes everything up
front).  It keeps its cos/sin table and rotated keys in a fixed static device array instead.

Checked here through the C ABI:
  * after one warm-up call, two calls in a row on two new shapes leave the device's free
    memory exactly as it was (nothing allocated);
  * both of those outputs match the fp64 oracle within the bf16 parity tolerances of the
    other GPU tests (this entry builds its cos/sin table on the device and rotates Q inside
    the attention kernel, so the oracle is what vouches for it), and match the ordinary entry
    point (vdx_rope3d_attn) within the same tolerances;
  * an over-size problem is refused without running anything.
Collected last on purpose.
"""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import oracle.fp64 as O
import video_diffusion_transformer_rope_gb300 as vdx
from video_diffusion_transformer_rope_gb300 import _binding, configs, synth

pytestmark = pytest.mark.gpu

OUT_MAX, OUT_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3     # the bf16 tolerances of test_parity_gpu.py


def _args(w, q, k, v, out, lse):
    return (ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
            w.B, w.H, w.T, w.Hg, w.Wg, w.d, *w.sections, w.theta, 0.0,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _check(status):
    if status != 0:
        raise vdx.VdxError(status, vdx.lib().vdx_last_error().decode())


def _within(got_o, got_l, ref_o, ref_l):
    err = np.abs(got_o - ref_o)
    lerr = np.abs(got_l - ref_l).max()
    return err.max() <= OUT_MAX and err.mean() <= OUT_MEAN and lerr <= LSE_MAX, (err.max(), err.mean(), lerr)


def test_noalloc_allocates_nothing_and_matches_oracle_twice():
    from video_diffusion_transformer_rope_gb300 import _build
    _build.build()
    L = vdx.lib()
    warm = dataclasses.replace(configs.WAN13B_480P, B=1, H=2, T=2, Hg=5, Wg=13, seed=40)
    shapes = [dataclasses.replace(configs.WAN13B_480P, B=2, H=3, T=3, Hg=9, Wg=21, seed=41),
              dataclasses.replace(configs.WAN13B_480P, B=1, H=4, T=5, Hg=12, Wg=16, seed=42)]
    # Every tensor this test touches exists before the measured calls.
    bufs = []
    for w in [warm] + shapes:
        q, k, v = (t.cuda() for t in synth.make_qkv(w))
        got_o = torch.full_like(q, float("nan"))
        got_l = torch.full((w.B, w.H, w.N), float("nan"), device="cuda")
        bufs.append((w, q, k, v, got_o, got_l))
    w, q, k, v, o, l = bufs[0]
    _check(L.vdx_rope3d_attn_noalloc(*_args(w, q, k, v, o, l)))     # first call on this device
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for w, q, k, v, o, l in bufs[1:]:
        _check(L.vdx_rope3d_attn_noalloc(*_args(w, q, k, v, o, l)))
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before, (free_before, free_after)
    vdx.sync_check()

    for w, q, k, v, got_o, got_l in bufs:
        ref_o, ref_l = O.rope3d_attention(q, k, v, (w.T, w.Hg, w.Wg), w.sections, w.theta)
        ok, errs = _within(got_o.double().cpu().numpy(), got_l.double().cpu().numpy(), ref_o, ref_l)
        assert ok, (w, errs)
        ord_o, ord_l = torch.empty_like(q), torch.empty(w.B, w.H, w.N, device="cuda")
        _check(L.vdx_rope3d_attn(*_args(w, q, k, v, ord_o, ord_l)))
        vdx.sync_check()
        ok, errs = _within(got_o.double().cpu().numpy(), got_l.double().cpu().numpy(),
                           ord_o.double().cpu().numpy(), ord_l.double().cpu().numpy())
        assert ok, (w, errs)


def test_noalloc_refuses_problems_beyond_its_scratch():
    L = vdx.lib()
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    ptr = ctypes.c_void_p(x.data_ptr())
    # B*N*H*d*2 = 2 * 75600 * 40 * 128 * 2 bytes > the static workspace: refused before launch
    st = L.vdx_rope3d_attn_noalloc(ptr, ptr, ptr, ctypes.c_void_p(x.data_ptr() + 4096), None,
                                   2, 40, 21, 45, 80, 128, 0, 0, 0, 10000.0, 0.0, None)
    assert st == _binding.VDX_ERR_UNSUPPORTED
    assert "no-allocation scratch" in L.vdx_last_error().decode()
