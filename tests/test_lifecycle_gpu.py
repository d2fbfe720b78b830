"""Library lifecycle on the GPU: cached tables and workspace for several grids, vdx_shutdown
releasing them, and calls afterwards (on a side stream) rebuilding them with identical results."""
import dataclasses

import pytest
import torch

import video_diffusion_transformer_rope_gb300 as vdx
from video_diffusion_transformer_rope_gb300 import configs, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from video_diffusion_transformer_rope_gb300 import _build
    _build.build()
    vdx.lib()


def test_shutdown_then_reuse_on_a_side_stream_is_bit_identical():
    shapes = [dataclasses.replace(configs.WAN13B_480P, B=1, H=2, T=2, Hg=7, Wg=19, seed=41),
              dataclasses.replace(configs.WAN13B_480P, B=2, H=1, T=3, Hg=5, Wg=33, seed=42,
                                  sections=(40, 44, 44), theta=5000.0)]
    inputs = [tuple(t.cuda() for t in synth.make_qkv(w)) for w in shapes]
    first = [vdx.rope3d_attn(q, k, v, (w.T, w.Hg, w.Wg), w.sections, w.theta)
             for w, (q, k, v) in zip(shapes, inputs)]
    vdx.sync_check()
    vdx.shutdown()                       # frees the cached tables and the library workspace
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        again = [vdx.rope3d_attn(q, k, v, (w.T, w.Hg, w.Wg), w.sections, w.theta, stream=side)
                 for w, (q, k, v) in zip(shapes, inputs)]
    vdx.sync_check(side)
    for (o1, l1), (o2, l2) in zip(first, again):
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
