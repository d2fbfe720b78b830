"""ctypes binding of libvdx.so (include/vdx.h).  Argument marshalling only: every step of the
computation runs in the library's CUDA kernels.  There is no fallback: if the library is not
built, or a call fails, this raises.
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libvdx.so")

(VDX_OK, VDX_ERR_ARG, VDX_ERR_ALIGN, VDX_ERR_UNSUPPORTED, VDX_ERR_CUDA, VDX_ERR_TIMEOUT,
 VDX_ERR_RANGE) = range(7)
STATUS_NAMES = {0: "VDX_OK", 1: "VDX_ERR_ARG", 2: "VDX_ERR_ALIGN", 3: "VDX_ERR_UNSUPPORTED",
                4: "VDX_ERR_CUDA", 5: "VDX_ERR_TIMEOUT", 6: "VDX_ERR_RANGE"}

_p, _i, _d, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_float

K_ROPE_DEFAULT, K_ROPE_PREPASS, K_ROPE_FUSED = 0, 1, 2
KERNEL_DEFAULT, KERNEL_SINGLE, KERNEL_PAIR = 0, 1, 2
QK_FP16, QK_SPLIT = 0, 1
QK_MODES = {"fp16": QK_FP16, "split": QK_SPLIT}


class AttnOptions(ctypes.Structure):
    """vdx_attn_options (include/vdx.h)."""
    _fields_ = [("k_rope", ctypes.c_int), ("qk_precision", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("test_withhold_kv", ctypes.c_int), ("kernel", ctypes.c_int)]
# name -> (restype, argtypes); mirrors include/vdx.h
SIGNATURES = {
    "vdx_rope3d_attn": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _d, _f, _p]),
    "vdx_rope3d_attn_ex": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _d, _f,
                                ctypes.POINTER(AttnOptions), _p]),
    "vdx_rope3d_workspace_bytes": (ctypes.c_size_t, [_i, _i, _i, _i, _i, _i, _i]),
    "vdx_rope3d_attn_f32": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _d, _f, _p]),
    "vdx_rope3d_attn_sparse": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _d, _f,
                                    _p, _i, ctypes.POINTER(AttnOptions), _p]),
    "vdx_rope3d_attn_subset": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _d, _f,
                                    _p, _i, _i, ctypes.POINTER(AttnOptions), _p]),
    "vdx_rope3d_block_mask_words": (_i, [_i, _i, _i]),
    "vdx_window_block_mask": (_i, [_p, _i, _i, _i, _i, _i, _i]),
    "vdx_rope3d_attn_noalloc": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _i, _d, _f, _p]),
    "vdx_sync_check": (_i, [_p]),
    "vdx_last_error": (ctypes.c_char_p, []),
    "vdx_shutdown": (None, []),
    "vdx_version": (_i, []),
}

_lib = None


class VdxError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


def lib():
    """Load libvdx.so once; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "video_diffusion_transformer_rope_gb300._build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status):
    if status != VDX_OK:
        raise VdxError(status, lib().vdx_last_error().decode())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def rope3d_attn(q, k, v, grid, sections=(0, 0, 0), theta=10000.0, scale=0.0, out=None,
                lse=None, return_lse=True, stream=None, k_rope=K_ROPE_DEFAULT, workspace=None,
                qk_precision=QK_FP16, kernel=KERNEL_DEFAULT):
    """3D-RoPE attention of CUDA tensors q, k, v laid out [B, N, H, d] (bf16 with d = 128, or
    float32 with d = 64/128).  grid = (T, Hgrid, Wgrid) with N = T*Hgrid*Wgrid.

    bf16 only: k_rope selects how K is rotated (K_ROPE_PREPASS, the default, or K_ROPE_FUSED);
    qk_precision QK_SPLIT keeps hi + lo fp16 parts of every rotated value (three products,
    for logits in the hundreds); workspace is an optional CUDA tensor of at least
    workspace_bytes(...) bytes for the prepass (None: the library's own per-device buffer);
    kernel selects KERNEL_SINGLE (one CTA per 256 query rows) or KERNEL_PAIR (CTA pairs sharing
    each K/V tile; dense calls only), KERNEL_DEFAULT the library's choice.

    Returns (out [B, N, H, d] in the input dtype, lse [B, H, N] float32 or None).  Enqueued on
    `stream` (default: torch's current stream); call sync_check() to surface device errors.
    """
    import torch
    T, Hg, Wg = (int(x) for x in grid)
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise VdxError(VDX_ERR_ARG, f"q, k, v must share one [B, N, H, d] shape, got "
                                    f"{tuple(q.shape)}, {tuple(k.shape)}, {tuple(v.shape)}")
    B, N, H, d = q.shape
    if N != T * Hg * Wg:
        raise VdxError(VDX_ERR_ARG, f"N={N} does not match grid {T}x{Hg}x{Wg}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype:
            raise VdxError(VDX_ERR_ARG, f"{name} must be a contiguous CUDA tensor of dtype {q.dtype}")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st, sh, sw = (int(x) for x in sections)
    args = (ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
            ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr() if lse is not None else 0),
            B, H, T, Hg, Wg, d, st, sh, sw, float(theta), float(scale), _stream_handle(stream))
    if q.dtype == torch.bfloat16:
        if k_rope == K_ROPE_DEFAULT and workspace is None and qk_precision == QK_FP16 and kernel == KERNEL_DEFAULT:
            _check(lib().vdx_rope3d_attn(*args))
        else:
            opt = AttnOptions(int(k_rope), int(qk_precision),
                              ctypes.c_void_p(workspace.data_ptr() if workspace is not None else 0),
                              workspace.numel() * workspace.element_size() if workspace is not None else 0,
                              0, int(kernel))
            _check(lib().vdx_rope3d_attn_ex(*args[:-1], ctypes.byref(opt), args[-1]))
    elif q.dtype == torch.float32:
        _check(lib().vdx_rope3d_attn_f32(*args))
    else:
        raise VdxError(VDX_ERR_UNSUPPORTED, f"dtype {q.dtype} (use bfloat16 or float32)")
    return out, lse


SPARSE_QBLOCK, SPARSE_KBLOCK = 256, 128


def block_mask_words(grid):
    """uint32 words per query block of a block mask for this grid."""
    T, Hg, Wg = (int(x) for x in grid)
    return lib().vdx_rope3d_block_mask_words(T, Hg, Wg)


def pack_block_mask(mask_bool):
    """Pack a boolean block mask [..., n_qblocks, n_kblocks] into uint32 words
    [..., n_qblocks, ceil(n_kblocks / 32)] (bit kb % 32 of word kb // 32)."""
    import numpy as np
    m = np.asarray(mask_bool, dtype=bool)
    nk = m.shape[-1]
    words = (nk + 31) // 32
    pad = np.zeros(m.shape[:-1] + (words * 32,), dtype=bool)
    pad[..., :nk] = m
    bits = pad.reshape(m.shape[:-1] + (words, 32)).astype(np.uint64)
    return (bits << np.arange(32, dtype=np.uint64)).sum(axis=-1).astype(np.uint32)


def window_block_mask(grid, window):
    """Block mask of 3D windowed attention (host numpy uint32 [n_qblocks, words]), built by
    the library's vdx_window_block_mask."""
    import numpy as np
    T, Hg, Wg = (int(x) for x in grid)
    N = T * Hg * Wg
    nqb = (N + SPARSE_QBLOCK - 1) // SPARSE_QBLOCK
    out = np.zeros((nqb, block_mask_words(grid)), dtype=np.uint32)
    wt, wh, ww = (int(x) for x in window)
    _check(lib().vdx_window_block_mask(out.ctypes.data_as(ctypes.c_void_p), T, Hg, Wg, wt, wh, ww))
    return out


def rope3d_attn_sparse(q, k, v, grid, block_mask, sections=(0, 0, 0), theta=10000.0, scale=0.0,
                       out=None, lse=None, return_lse=True, stream=None, workspace=None,
                       qk_precision=QK_FP16):
    """Block-sparse 3D-RoPE attention (bf16, d = 128).  block_mask: CUDA uint32/int32 tensor of
    packed words, shape [B, H, n_qblocks, W] (one mask per head) or [n_qblocks, W] (shared);
    see pack_block_mask / window_block_mask."""
    import torch
    T, Hg, Wg = (int(x) for x in grid)
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape or q.dtype != torch.bfloat16:
        raise VdxError(VDX_ERR_ARG, "q, k, v must be bf16 [B, N, H, d] tensors of one shape")
    B, N, H, d = q.shape
    if N != T * Hg * Wg:
        raise VdxError(VDX_ERR_ARG, f"N={N} does not match grid {T}x{Hg}x{Wg}")
    nqb = (N + SPARSE_QBLOCK - 1) // SPARSE_QBLOCK
    W = block_mask_words(grid)
    if block_mask.dtype not in (torch.int32, torch.uint32) or not block_mask.is_cuda or not block_mask.is_contiguous():
        raise VdxError(VDX_ERR_ARG, "block_mask must be a contiguous CUDA int32/uint32 tensor")
    if tuple(block_mask.shape) == (B, H, nqb, W):
        per_head = 1
    elif tuple(block_mask.shape) == (nqb, W):
        per_head = 0
    else:
        raise VdxError(VDX_ERR_ARG, f"block_mask shape {tuple(block_mask.shape)} is neither "
                                    f"{(B, H, nqb, W)} nor {(nqb, W)}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous():
            raise VdxError(VDX_ERR_ARG, f"{name} must be a contiguous CUDA tensor")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st, sh, sw = (int(x) for x in sections)
    opt = AttnOptions(K_ROPE_PREPASS, int(qk_precision),
                      ctypes.c_void_p(workspace.data_ptr() if workspace is not None else 0),
                      workspace.numel() * workspace.element_size() if workspace is not None else 0)
    _check(lib().vdx_rope3d_attn_sparse(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr() if lse is not None else 0),
        B, H, T, Hg, Wg, d, st, sh, sw, float(theta), float(scale),
        ctypes.c_void_p(block_mask.data_ptr()), per_head, ctypes.byref(opt), _stream_handle(stream)))
    return out, lse


def rope3d_attn_subset(q, k, v, grid, q_index, out, lse=None, sections=(0, 0, 0), theta=10000.0,
                       scale=0.0, stream=None, workspace=None, qk_precision=QK_FP16):
    """Active-query subset: the tokens in q_index (CUDA int32, [Nq] shared or [B, Nq]) attend to
    every key; their rows of `out` ([B, N, H, d], written in place) and `lse` ([B, H, N] or None)
    are updated, all other rows are left as they are."""
    import torch
    T, Hg, Wg = (int(x) for x in grid)
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape or q.dtype != torch.bfloat16:
        raise VdxError(VDX_ERR_ARG, "q, k, v must be bf16 [B, N, H, d] tensors of one shape")
    B, N, H, d = q.shape
    if N != T * Hg * Wg:
        raise VdxError(VDX_ERR_ARG, f"N={N} does not match grid {T}x{Hg}x{Wg}")
    if q_index.dtype != torch.int32 or not q_index.is_cuda or not q_index.is_contiguous():
        raise VdxError(VDX_ERR_ARG, "q_index must be a contiguous CUDA int32 tensor")
    if q_index.dim() == 1:
        per_batch, Nq = 0, q_index.shape[0]
    elif q_index.dim() == 2 and q_index.shape[0] == B:
        per_batch, Nq = 1, q_index.shape[1]
    else:
        raise VdxError(VDX_ERR_ARG, f"q_index shape {tuple(q_index.shape)} is neither [Nq] nor [B, Nq]")
    if out is None or out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise VdxError(VDX_ERR_ARG, "out must be a contiguous bf16 tensor shaped like q")
    st, sh, sw = (int(x) for x in sections)
    opt = AttnOptions(K_ROPE_PREPASS, int(qk_precision),
                      ctypes.c_void_p(workspace.data_ptr() if workspace is not None else 0),
                      workspace.numel() * workspace.element_size() if workspace is not None else 0)
    _check(lib().vdx_rope3d_attn_subset(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr() if lse is not None else 0),
        B, H, T, Hg, Wg, d, st, sh, sw, float(theta), float(scale),
        ctypes.c_void_p(q_index.data_ptr()), int(Nq), per_batch, ctypes.byref(opt),
        _stream_handle(stream)))
    return out, lse


def workspace_bytes(B, H, grid, d=128, qk_precision=QK_FP16):
    """Bytes of scratch the K prepass needs (vdx_rope3d_workspace_bytes)."""
    T, Hg, Wg = (int(x) for x in grid)
    return lib().vdx_rope3d_workspace_bytes(B, H, T, Hg, Wg, d, qk_precision)


def sync_check(stream=None):
    """Synchronise the stream and raise VdxError if a kernel reported a device-side problem."""
    _check(lib().vdx_sync_check(_stream_handle(stream)))


def shutdown():
    lib().vdx_shutdown()


def version():
    return lib().vdx_version()
