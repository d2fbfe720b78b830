"""vdx_rope3d_attn_noalloc: the entry point for callers that cannot allocate device memory at
call time (a frozen memory pool, an allocator-free embedding, a host that sizes everything up
front).  It keeps its cos/sin table and rotated keys in a fixed static device array instead.

Checked here through the C ABI: its output equals the ordinary entry point's (vdx_rope3d_attn)
within the bf16 parity tolerances used by the other GPU tests, on two calls in a row with
different shapes (so the second call rebuilds the table the first one left behind), and an
over-size problem is refused without running anything.  Collected last on purpose.
"""
import ctypes
import dataclasses

import pytest
import torch

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


def test_noalloc_matches_ordinary_entry_point_twice():
    from video_diffusion_transformer_rope_gb300 import _build
    _build.build()
    L = vdx.lib()
    shapes = [dataclasses.replace(configs.WAN13B_480P, B=2, H=3, T=3, Hg=9, Wg=21, seed=41),
              dataclasses.replace(configs.WAN13B_480P, B=1, H=4, T=5, Hg=12, Wg=16, seed=42)]
    for w in shapes:
        q, k, v = (t.cuda() for t in synth.make_qkv(w))
        ref_o, ref_l = torch.empty_like(q), torch.empty(w.B, w.H, w.N, device="cuda")
        got_o, got_l = torch.full_like(q, float("nan")), torch.full((w.B, w.H, w.N), float("nan"), device="cuda")
        _check(L.vdx_rope3d_attn(*_args(w, q, k, v, ref_o, ref_l)))
        _check(L.vdx_rope3d_attn_noalloc(*_args(w, q, k, v, got_o, got_l)))
        vdx.sync_check()
        err = (got_o.float() - ref_o.float()).abs()
        assert err.max().item() <= OUT_MAX and err.mean().item() <= OUT_MEAN, (err.max(), err.mean())
        assert (got_l - ref_l).abs().max().item() <= LSE_MAX


def test_noalloc_refuses_problems_beyond_its_scratch():
    L = vdx.lib()
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    ptr = ctypes.c_void_p(x.data_ptr())
    # B*N*H*d*2 = 2 * 75600 * 40 * 128 * 2 bytes > the static workspace: refused before launch
    st = L.vdx_rope3d_attn_noalloc(ptr, ptr, ptr, ctypes.c_void_p(x.data_ptr() + 4096), None,
                                   2, 40, 21, 45, 80, 128, 0, 0, 0, 10000.0, 0.0, None)
    assert st == _binding.VDX_ERR_UNSUPPORTED
    assert "no-allocation scratch" in L.vdx_last_error().decode()
