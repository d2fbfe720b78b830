"""The C-ABI library: loads without a GPU, exports every symbol include/vdx.h declares, and
rejects bad arguments before touching CUDA (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import video_diffusion_transformer_rope_gb300 as vdx
from video_diffusion_transformer_rope_gb300 import _binding, _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return vdx.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "vdx.h")) as f:
        hdr = f.read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return set(re.findall(r"^\s*(?:vdx_status|const char\s*\*|void|int|size_t)\s+(vdx_\w+)\s*\(", hdr, re.M))


def test_exports_every_declared_symbol(L):
    decl = _declared()
    assert {"vdx_rope3d_attn", "vdx_rope3d_attn_ex", "vdx_rope3d_attn_f32", "vdx_sync_check",
            "vdx_last_error", "vdx_shutdown", "vdx_version", "vdx_rope3d_workspace_bytes"} <= decl
    for name in decl:
        assert hasattr(L, name), name
    assert set(_binding.SIGNATURES) == decl
    assert L.vdx_version() == 100


FAKE = 0x7f0000000000          # 16-byte aligned, never dereferenced: every call below fails first


def _call(L, fn="vdx_rope3d_attn", q=FAKE, k=FAKE + (1 << 32), v=FAKE + (2 << 32),
          out=FAKE + (3 << 32), lse=0, B=1, H=2, T=2, Hg=3, Wg=4, d=128, st=0, sh=0, sw=0,
          theta=10000.0, scale=0.0):
    return getattr(L, fn)(ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v),
                          ctypes.c_void_p(out), ctypes.c_void_p(lse), B, H, T, Hg, Wg, d,
                          st, sh, sw, theta, scale, None)


@pytest.mark.parametrize("kw,status,msg", [
    (dict(d=64), _binding.VDX_ERR_UNSUPPORTED, "head_dim 128"),
    (dict(fn="vdx_rope3d_attn_f32", d=96), _binding.VDX_ERR_UNSUPPORTED, "64 or 128"),
    (dict(q=0), _binding.VDX_ERR_ARG, "non-NULL"),
    (dict(out=0), _binding.VDX_ERR_ARG, "non-NULL"),
    (dict(B=0), _binding.VDX_ERR_ARG, ">= 1"),
    (dict(H=0), _binding.VDX_ERR_ARG, ">= 1"),
    (dict(T=0), _binding.VDX_ERR_ARG, ">= 1"),
    (dict(Hg=0), _binding.VDX_ERR_ARG, ">= 1"),
    (dict(Wg=-3), _binding.VDX_ERR_ARG, ">= 1"),
    (dict(fn="vdx_rope3d_attn_f32", B=0), _binding.VDX_ERR_ARG, ">= 1"),
    (dict(st=44, sh=42, sw=41), _binding.VDX_ERR_ARG, "sections"),
    (dict(st=43, sh=43, sw=42), _binding.VDX_ERR_ARG, "sections"),
    (dict(st=40, sh=40, sw=40), _binding.VDX_ERR_ARG, "sum to d"),
    (dict(theta=0.0), _binding.VDX_ERR_ARG, "theta"),
    (dict(theta=-1.0), _binding.VDX_ERR_ARG, "theta"),
    (dict(scale=float("nan")), _binding.VDX_ERR_ARG, "scale"),
    (dict(k=FAKE + 8), _binding.VDX_ERR_ALIGN, "aligned"),
    (dict(lse=FAKE + (4 << 32) + 4), _binding.VDX_ERR_ALIGN, "aligned"),
    (dict(out=FAKE + 64), _binding.VDX_ERR_ARG, "overlaps"),
    (dict(lse=FAKE + (1 << 32) + 4096), _binding.VDX_ERR_ARG, "overlaps"),
    (dict(T=100000, Hg=1000, Wg=1000), _binding.VDX_ERR_ARG, "too large"),
])
def test_rejects_bad_arguments_without_cuda(L, kw, status, msg):
    assert _call(L, **kw) == status
    assert msg in L.vdx_last_error().decode()


@pytest.mark.parametrize("kw,status,msg", [
    (dict(out=FAKE + 64), _binding.VDX_ERR_ARG, "out overlaps"),
    (dict(lse=FAKE + (1 << 32) + 4096), _binding.VDX_ERR_ARG, "lse overlaps"),   # inside k
    (dict(lse=FAKE + (3 << 32) + 16), _binding.VDX_ERR_ARG, "lse overlaps"),     # inside out
    (dict(lse=FAKE - 16), _binding.VDX_ERR_ARG, "lse overlaps"),                 # its tail runs into q
    (dict(lse=FAKE + (4 << 32) + 4), _binding.VDX_ERR_ALIGN, "aligned"),
    (dict(d=64), _binding.VDX_ERR_UNSUPPORTED, "128"),
])
def test_noalloc_rejects_aliasing_without_cuda(L, kw, status, msg):
    # the no-allocation entry checks its arguments like the ordinary one, before any CUDA call
    assert _call(L, fn="vdx_rope3d_attn_noalloc", **kw) == status
    assert msg in L.vdx_last_error().decode()


def test_workspace_bytes(L):
    # rotated K and rotated Q (fp16 each), doubled again for the hi + lo split
    assert L.vdx_rope3d_workspace_bytes(2, 40, 21, 45, 80, 128, 0) == 2 * 75600 * 40 * 128 * 2 * 2
    assert L.vdx_rope3d_workspace_bytes(2, 40, 21, 45, 80, 128, 1) == 2 * 75600 * 40 * 128 * 4 * 2
    assert L.vdx_rope3d_workspace_bytes(0, 40, 21, 45, 80, 128, 0) == 0


def test_ex_rejects_bad_options(L):
    opt = _binding.AttnOptions(7, 0, None, 0, 0)
    r = L.vdx_rope3d_attn_ex(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + (1 << 32)),
                             ctypes.c_void_p(FAKE + (2 << 32)), ctypes.c_void_p(FAKE + (3 << 32)),
                             None, 1, 2, 2, 3, 4, 128, 0, 0, 0, 10000.0, 0.0, ctypes.byref(opt), None)
    assert r == _binding.VDX_ERR_ARG and "k_rope" in L.vdx_last_error().decode()
    for prec in (_binding.QK_SPLIT,):
        opt = _binding.AttnOptions(_binding.K_ROPE_FUSED, prec, None, 0, 0)
        r = L.vdx_rope3d_attn_ex(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + (1 << 32)),
                                 ctypes.c_void_p(FAKE + (2 << 32)), ctypes.c_void_p(FAKE + (3 << 32)),
                                 None, 1, 2, 2, 3, 4, 128, 0, 0, 0, 10000.0, 0.0, ctypes.byref(opt), None)
        assert r == _binding.VDX_ERR_UNSUPPORTED and "prepass" in L.vdx_last_error().decode()
    opt = _binding.AttnOptions(_binding.K_ROPE_PREPASS, 2, None, 0, 0)
    r = L.vdx_rope3d_attn_ex(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + (1 << 32)),
                             ctypes.c_void_p(FAKE + (2 << 32)), ctypes.c_void_p(FAKE + (3 << 32)),
                             None, 1, 2, 2, 3, 4, 128, 0, 0, 0, 10000.0, 0.0, ctypes.byref(opt), None)
    assert r == _binding.VDX_ERR_ARG and "qk_precision" in L.vdx_last_error().decode()


@pytest.mark.parametrize("k_rope,prec,kernel,status", [
    (_binding.K_ROPE_PREPASS, _binding.QK_FP16, 9, _binding.VDX_ERR_ARG),
    (_binding.K_ROPE_FUSED, _binding.QK_FP16, -1, _binding.VDX_ERR_ARG),
])
def test_ex_rejects_unknown_kernel_choices(L, k_rope, prec, kernel, status):
    opt = _binding.AttnOptions(k_rope, prec, None, 0, 0, kernel)
    r = L.vdx_rope3d_attn_ex(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + (1 << 32)),
                             ctypes.c_void_p(FAKE + (2 << 32)), ctypes.c_void_p(FAKE + (3 << 32)),
                             None, 1, 2, 2, 3, 4, 128, 0, 0, 0, 10000.0, 0.0, ctypes.byref(opt), None)
    assert r == status and "kernel" in L.vdx_last_error().decode().lower()


def test_sparse_and_subset_calls_reject_cta_pairs(L):
    # CTA pairs take dense calls only (with either K rotation); a block mask or a query subset
    # with VDX_KERNEL_PAIR is refused before any device work.
    opt = _binding.AttnOptions(_binding.K_ROPE_PREPASS, _binding.QK_FP16, None, 0, 0, _binding.KERNEL_PAIR)
    r = L.vdx_rope3d_attn_sparse(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + (1 << 32)),
                                 ctypes.c_void_p(FAKE + (2 << 32)), ctypes.c_void_p(FAKE + (3 << 32)),
                                 None, 1, 2, 2, 3, 4, 128, 0, 0, 0, 10000.0, 0.0,
                                 ctypes.c_void_p(FAKE + (4 << 32)), 0, ctypes.byref(opt), None)
    assert r == _binding.VDX_ERR_UNSUPPORTED and "dense" in L.vdx_last_error().decode()
    r = L.vdx_rope3d_attn_subset(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE + (1 << 32)),
                                 ctypes.c_void_p(FAKE + (2 << 32)), ctypes.c_void_p(FAKE + (3 << 32)),
                                 None, 1, 2, 2, 3, 4, 128, 0, 0, 0, 10000.0, 0.0,
                                 ctypes.c_void_p(FAKE + (4 << 32)), 8, 0, ctypes.byref(opt), None)
    assert r == _binding.VDX_ERR_UNSUPPORTED and "dense" in L.vdx_last_error().decode()


def test_python_binding_rejects_mismatched_grid(L):
    import torch
    q = torch.zeros(1, 10, 1, 128)
    with pytest.raises(vdx.VdxError):
        vdx.rope3d_attn(q, q, q, (2, 2, 2))
