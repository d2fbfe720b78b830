"""Library lifecycle on the GPU: cached tables and workspace for several grids, vdx_shutdown
releasing them, and calls afterwards (on a side stream) rebuilding them with identical results;
calls in flight at once on several streams (each with its own workspace) giving the results of
the same calls made alone."""
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


def test_concurrent_calls_on_three_streams_match_the_same_calls_alone():
    # Three problems in flight at once: two with their own prepass workspaces (one CTA per query
    # block; CTA pairs) and one with the fused K rotation, which needs none.  The library's
    # per-call state lives in the caller's buffers, so each result equals the same call made
    # alone, bit for bit (the kernels are deterministic).
    wa = dataclasses.replace(configs.WAN13B_480P, B=2, H=6, T=3, Hg=20, Wg=30, seed=71)
    wb = dataclasses.replace(configs.WAN13B_480P, B=1, H=8, T=2, Hg=30, Wg=40, seed=72)
    wc = dataclasses.replace(configs.WAN13B_480P, B=1, H=4, T=4, Hg=15, Wg=32, seed=73)
    jobs = []
    for w, kw in ((wa, {"kernel": vdx.KERNEL_SINGLE}), (wb, {"kernel": vdx.KERNEL_PAIR}),
                  (wc, {"k_rope": vdx.K_ROPE_FUSED})):
        q, k, v = synth.make_qkv(w, device="cuda")
        if "k_rope" not in kw:
            nbytes = vdx.workspace_bytes(w.B, w.H, (w.T, w.Hg, w.Wg))
            kw = dict(kw, workspace=torch.empty(nbytes // 2, dtype=torch.float16, device="cuda"))
        alone = vdx.rope3d_attn(q, k, v, (w.T, w.Hg, w.Wg), w.sections, w.theta, **kw)
        vdx.sync_check()
        jobs.append((w, q, k, v, kw, alone))
    streams = [torch.cuda.Stream() for _ in jobs]
    outs = [[(torch.empty_like(q), torch.empty(w.B, w.H, w.N, device="cuda")) for _ in range(3)]
            for (w, q, _, _, _, _) in jobs]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for r in range(3):
        for s, (w, q, k, v, kw, _), o in zip(streams, jobs, outs):
            vdx.rope3d_attn(q, k, v, (w.T, w.Hg, w.Wg), w.sections, w.theta, out=o[r][0], lse=o[r][1],
                            stream=s, **kw)
    for s in streams:
        vdx.sync_check(s)
    for (_, _, _, _, _, (o1, l1)), o in zip(jobs, outs):
        for o2, l2 in o:
            assert torch.equal(o1, o2) and torch.equal(l1, l2)
