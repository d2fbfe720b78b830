"""vdx: 3D-RoPE full spatiotemporal self-attention for video diffusion transformers on one
GB300 (sm_103a).  The computation lives in libvdx.so (C ABI, include/vdx.h); this package
holds the ctypes binding, the build step, the measured workloads and the seeded input recipe.
"""
from ._binding import (VdxError, lib, rope3d_attn, sync_check, shutdown, version,  # noqa: F401
                       workspace_bytes, SIGNATURES, LIB_PATH, K_ROPE_DEFAULT, K_ROPE_PREPASS,
                       K_ROPE_FUSED, KERNEL_DEFAULT, KERNEL_SINGLE, KERNEL_PAIR, QK_FP16, QK_SPLIT, QK_MODES, rope3d_attn_sparse, pack_block_mask,
                       window_block_mask, block_mask_words, SPARSE_QBLOCK, SPARSE_KBLOCK,
                       rope3d_attn_subset)
