"""Active-query subset on the GPU (through the C ABI): the listed tokens' rows equal the fp64
oracle's rows for those tokens (attention over all keys), every other row of out / lse is left
untouched, and indices outside [0, N) are skipped and reported."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle.fp64 as O
import video_diffusion_transformer_rope_gb300 as vdx
from video_diffusion_transformer_rope_gb300 import configs, synth

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from video_diffusion_transformer_rope_gb300 import _build
    _build.build()
    vdx.lib()


def _run_subset(w, idx_np, qk="fp16", seed_out=7.0):
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    out = torch.full_like(q, seed_out)
    lse = torch.full((w.B, w.H, w.N), -5.0, device="cuda")
    idx = torch.from_numpy(np.ascontiguousarray(idx_np, dtype=np.int32)).cuda()
    vdx.rope3d_attn_subset(q, k, v, (w.T, w.Hg, w.Wg), idx, out, lse, w.sections, w.theta,
                           qk_precision=vdx.QK_MODES[qk])
    vdx.sync_check()
    return q, k, v, out, lse


@pytest.mark.parametrize("grid,nq", [((4, 9, 13), 37), ((5, 12, 20), 300), ((3, 8, 8), 192),
                                     ((1, 1, 700), 1)])
def test_shared_index_list(grid, nq):
    w = dataclasses.replace(configs.WAN13B_480P, B=2, H=3, T=grid[0], Hg=grid[1], Wg=grid[2], seed=61)
    rng = np.random.default_rng(nq)
    idx = rng.choice(w.N, nq, replace=False)
    q, k, v, out, lse = _run_subset(w, idx)
    rows = [(b, h, int(n)) for b in range(w.B) for h in range(w.H) for n in idx]
    ref_o, ref_l = O.rope3d_attention_rows(q, k, v, (w.T, w.Hg, w.Wg), rows, w.sections, w.theta)
    b = torch.tensor([r[0] for r in rows]); h = torch.tensor([r[1] for r in rows]); n = torch.tensor([r[2] for r in rows])
    got_o = out.cpu()[b, n, h].double().numpy()
    got_l = lse.cpu()[b, h, n].double().numpy()
    err = np.abs(got_o - ref_o)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (err.max(), err.mean())
    assert np.abs(got_l - ref_l).max() <= LSE_TOL
    untouched = np.ones(w.N, dtype=bool)
    untouched[idx] = False
    assert torch.all(out[:, torch.from_numpy(untouched).cuda()] == 7.0)
    assert torch.all(lse[:, :, torch.from_numpy(untouched).cuda()] == -5.0)


def test_per_batch_lists_and_split_precision():
    w = dataclasses.replace(configs.LONG_STRESS, B=2, H=2, T=2, Hg=9, Wg=40, seed=62, qk="split")
    rng = np.random.default_rng(5)
    idx = np.stack([rng.choice(w.N, 200, replace=False) for _ in range(w.B)])
    q, k, v, out, lse = _run_subset(w, idx, qk="split")
    rows = [(b, h, int(n)) for b in range(w.B) for h in range(w.H) for n in idx[b]]
    ref_o, ref_l = O.rope3d_attention_rows(q, k, v, (w.T, w.Hg, w.Wg), rows, w.sections, w.theta)
    b = torch.tensor([r[0] for r in rows]); h = torch.tensor([r[1] for r in rows]); n = torch.tensor([r[2] for r in rows])
    err = np.abs(out.cpu()[b, n, h].double().numpy() - ref_o)
    assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN
    assert np.abs(lse.cpu()[b, h, n].double().numpy() - ref_l).max() <= LSE_TOL


def test_full_subset_equals_dense_call():
    w = dataclasses.replace(configs.WAN13B_480P, B=1, H=2, T=3, Hg=10, Wg=30, seed=63)
    q, k, v, out, lse = _run_subset(w, np.arange(w.N))
    o2, l2 = vdx.rope3d_attn(q, k, v, (w.T, w.Hg, w.Wg))
    vdx.sync_check()
    assert torch.equal(out, o2) and torch.equal(lse, l2)


def test_out_of_range_index_is_skipped_and_reported():
    w = dataclasses.replace(configs.WAN13B_480P, B=1, H=1, T=1, Hg=2, Wg=64, seed=64)
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    out = torch.full_like(q, 3.0)
    idx = torch.tensor([5, w.N + 10, -1, 7], dtype=torch.int32, device="cuda")
    vdx.rope3d_attn_subset(q, k, v, (1, 2, 64), idx, out, None)
    with pytest.raises(vdx.VdxError) as ei:
        vdx.sync_check()
    assert "q_index" in str(ei.value)
    assert not torch.all(out[0, 5] == 3.0) and not torch.all(out[0, 7] == 3.0)
    keep = [i for i in range(w.N) if i not in (5, 7)]
    assert torch.all(out[0, keep] == 3.0)


def test_ulysses_single_rank_nccl_on_gpu_matches_oracle():
    # One NCCL rank on this GPU: the exchanges are identities and the library does the work;
    # the result is checked against the oracle and equals the direct library call bit for bit.
    import os
    import socket
    import torch.distributed as dist
    from video_diffusion_transformer_rope_gb300.ulysses import ulysses_rope3d_attn
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        w = dataclasses.replace(configs.WAN13B_480P, B=2, H=4, T=2, Hg=8, Wg=20, seed=65)
        q, k, v = (t.cuda() for t in synth.make_qkv(w))
        o1, l1 = ulysses_rope3d_attn(q, k, v, (w.T, w.Hg, w.Wg), w.sections, w.theta)
        vdx.sync_check()
        ref_o, ref_l = O.rope3d_attention(q, k, v, (w.T, w.Hg, w.Wg), w.sections, w.theta)
        err = np.abs(o1.double().cpu().numpy() - ref_o)
        assert err.max() <= BF16_MAX and err.mean() <= BF16_MEAN, (err.max(), err.mean())
        assert np.abs(l1.double().cpu().numpy() - ref_l).max() <= LSE_TOL
        o2, l2 = vdx.rope3d_attn(q, k, v, (w.T, w.Hg, w.Wg), w.sections, w.theta)
        vdx.sync_check()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    finally:
        dist.destroy_process_group()
