"""Device-side error reporting through vdx_sync_check (no fault, no hang is provoked)."""
import dataclasses

import pytest
import torch

import video_diffusion_transformer_rope_gb300 as vdx
from video_diffusion_transformer_rope_gb300 import configs, synth

pytestmark = pytest.mark.gpu


def test_fp16_range_flag_and_clear():
    w = dataclasses.replace(configs.WAN13B_480P, B=1, H=1, T=1, Hg=2, Wg=64, seed=31)
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    # Token 5 sits at t = 0, so channel pair (2, 3) (a t-axis pair) is not rotated.
    # K is stored as rotated: bf16 70144 is above the fp16 maximum 65504.
    k[0, 5, 0, 3] = 70000.0
    vdx.rope3d_attn(q, k, v, (1, 2, 64))
    with pytest.raises(vdx.VdxError) as ei:
        vdx.sync_check()
    assert ei.value.status == 6 and "fp16" in str(ei.value)
    k[0, 5, 0, 3] = 1.0
    # Q is stored multiplied by scale*log2(e) = 0.1275: 70000 fits, 600000 (bf16 599040) does not.
    q[0, 5, 0, 3] = 70000.0
    vdx.rope3d_attn(q, k, v, (1, 2, 64))
    vdx.sync_check()
    q[0, 5, 0, 3] = 600000.0
    vdx.rope3d_attn(q, k, v, (1, 2, 64))
    with pytest.raises(vdx.VdxError) as ei:
        vdx.sync_check()
    assert ei.value.status == 6
    # the word is cleared by the read; an in-range call afterwards is clean
    q[0, 5, 0, 3] = 1.0
    vdx.rope3d_attn(q, k, v, (1, 2, 64))
    vdx.sync_check()


def test_bad_arguments_raise_before_launch():
    q = torch.zeros(1, 8, 1, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vdx.VdxError) as ei:
        vdx.rope3d_attn(q, q.clone(), q.clone(), (1, 2, 4), sections=(44, 42, 40))
    assert ei.value.status == 1
    with pytest.raises(vdx.VdxError) as ei:
        vdx.rope3d_attn(q, q.clone(), q.clone(), (1, 2, 4), out=q)
    assert ei.value.status == 1
    vdx.sync_check()


@pytest.mark.parametrize("kernel", ["single", "pair", "pair_fused"])
def test_pipeline_wait_timeout_is_reported_and_context_stays_usable(kernel):
    # The producer withholds every K/V tile: the MMA and softmax waits run out after ~1 s, the
    # kernel stops cleanly (TMEM freed, its own copies drained), and the status says so.  With
    # CTA pairs both CTAs give up and meet at the final cluster barrier.
    import ctypes
    from video_diffusion_transformer_rope_gb300 import _binding
    w = dataclasses.replace(configs.WAN13B_480P, B=1, H=1, T=1, Hg=2, Wg=64, seed=32)
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    out = torch.empty_like(q)
    opt = _binding.AttnOptions(vdx.K_ROPE_FUSED if kernel == "pair_fused" else vdx.K_ROPE_PREPASS,
                               vdx.QK_FP16, None, 0, 1,
                               vdx.KERNEL_SINGLE if kernel == "single" else vdx.KERNEL_PAIR)
    L = vdx.lib()
    st = L.vdx_rope3d_attn_ex(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                              ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()), None,
                              1, 1, 1, 2, 64, 128, 0, 0, 0, 10000.0, 0.0, ctypes.byref(opt), None)
    assert st == 0
    with pytest.raises(vdx.VdxError) as ei:
        vdx.sync_check()
    assert ei.value.status == _binding.VDX_ERR_TIMEOUT
    # the next ordinary call on the same context is correct
    import oracle.fp64 as O
    import numpy as np
    o2, l2 = vdx.rope3d_attn(q, k, v, (1, 2, 64))
    vdx.sync_check()
    ref_o, _ = O.rope3d_attention(q, k, v, (1, 2, 64))
    assert np.abs(o2.double().cpu().numpy() - ref_o).max() <= 2e-2


def test_caller_workspace_next_to_an_input_is_accepted_and_an_overlap_rejected():
    # Split precision: the workspace is twice the size of q, so a check that sized q like the
    # workspace would flag a workspace that merely starts where q ends.
    w = dataclasses.replace(configs.LONG_STRESS, B=1, H=2, T=1, Hg=4, Wg=64, seed=33)
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    grid = (w.T, w.Hg, w.Wg)
    need = vdx.workspace_bytes(w.B, w.H, grid, w.d, vdx.QK_SPLIT)
    buf = torch.empty(q.numel() + need // 2, dtype=torch.bfloat16, device="cuda")
    qa = buf[:q.numel()].view(q.shape)
    qa.copy_(q)
    out, lse = vdx.rope3d_attn(qa, k, v, grid, w.sections, w.theta, workspace=buf[q.numel():],
                               qk_precision=vdx.QK_SPLIT)
    ref_o, ref_l = vdx.rope3d_attn(q, k, v, grid, w.sections, w.theta, qk_precision=vdx.QK_SPLIT)
    vdx.sync_check()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    with pytest.raises(vdx.VdxError) as ei:
        vdx.rope3d_attn(qa, k, v, grid, w.sections, w.theta, workspace=buf[q.numel() // 2:],
                        qk_precision=vdx.QK_SPLIT)
    assert ei.value.status == 1 and "overlaps" in str(ei.value)
    vdx.sync_check()
