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
    q[0, 5, 0, 3] = 70000.0          # bf16 70144: above the fp16 maximum 65504 at any angle
    vdx.rope3d_attn(q, k, v, (1, 2, 64))
    with pytest.raises(vdx.VdxError) as ei:
        vdx.sync_check()
    assert ei.value.status == 6 and "fp16" in str(ei.value)
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
