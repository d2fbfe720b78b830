"""GPU path (through the C ABI) against the fp64 oracle, element by element on the same seeded
inputs.  Tolerances: fp32 path max-abs <= 1e-4; bf16 path out max-abs <= 2e-2, out mean-abs
<= 2e-3, lse max-abs <= 1e-3 (full comparison at small sizes, sampled rows at full size)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle.fp64 as O
import video_diffusion_transformer_rope_gb300 as vdx
from video_diffusion_transformer_rope_gb300 import configs, synth

pytestmark = pytest.mark.gpu

F32_TOL = 1e-4
BF16_MAX, BF16_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from video_diffusion_transformer_rope_gb300 import _build
    _build.build()
    vdx.lib()


def _run(w, q, k, v, **kw):
    kw.setdefault("qk_precision", vdx.QK_MODES[w.qk])
    out, lse = vdx.rope3d_attn(q, k, v, (w.T, w.Hg, w.Wg), w.sections, w.theta, **kw)
    vdx.sync_check()
    return out, lse


def _full_compare(w, dev_qkv=None, **kw):
    q, k, v = dev_qkv if dev_qkv is not None else (t.cuda() for t in synth.make_qkv(w))
    out, lse = _run(w, q, k, v, **kw)
    ref_o, ref_l = O.rope3d_attention(q, k, v, (w.T, w.Hg, w.Wg), w.sections, w.theta)
    got_o = out.double().cpu().numpy()
    got_l = lse.double().cpu().numpy()
    err = np.abs(got_o - ref_o)
    return err.max(), err.mean(), np.abs(got_l - ref_l).max()


def test_tiny_f32_config():
    mx, mean, lerr = _full_compare(configs.TINY_F32)
    assert mx <= F32_TOL and lerr <= F32_TOL, (mx, lerr)


@pytest.mark.parametrize("grid,d", [((3, 8, 8), 128), ((2, 9, 13), 64), ((1, 1, 1), 64),
                                    ((2, 1, 67), 128)])
def test_f32_shapes(grid, d):
    w = dataclasses.replace(configs.TINY_F32, T=grid[0], Hg=grid[1], Wg=grid[2], d=d,
                            sections=O.default_sections(d), B=2, H=3, seed=11)
    mx, mean, lerr = _full_compare(w)
    assert mx <= F32_TOL and lerr <= F32_TOL, (mx, lerr)


# Small bf16 shapes spanning several 128-key tiles, 256-row CTAs and ragged tails:
# N = 192 (tail 64), 105 (< one tile), 1, 129 (= 1 mod 128), 468, 640 (exact), T=1, Wg=1.
BF16_GRIDS = [(3, 8, 8), (3, 5, 7), (1, 1, 1), (1, 1, 129), (4, 9, 13), (5, 8, 16), (1, 16, 24),
              (7, 40, 1)]


K_MODES = {"prepass": vdx.K_ROPE_PREPASS, "fused": vdx.K_ROPE_FUSED}


@pytest.mark.parametrize("mode", sorted(K_MODES))
@pytest.mark.parametrize("grid", BF16_GRIDS, ids=lambda g: "x".join(map(str, g)))
def test_bf16_small_shapes(grid, mode):
    # the one-CTA kernel (fused calls default to CTA pairs, tested below)
    w = dataclasses.replace(configs.WAN13B_480P, B=2, H=3, T=grid[0], Hg=grid[1], Wg=grid[2], seed=21)
    mx, mean, lerr = _full_compare(w, k_rope=K_MODES[mode], kernel=vdx.KERNEL_SINGLE)
    assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL, (mx, mean, lerr)


# CTA pairs: N = 192 and 129 (one query block, so a padding CTA completes the pair), 468, 640
# (three blocks: padded to four), 1 (a single token), 280 (T = 7, Wg = 1).  With the fused K
# rotation each CTA rotates its own Q tiles and its 64 keys of every K tile.
@pytest.mark.parametrize("mode", sorted(K_MODES))
@pytest.mark.parametrize("grid", [(3, 8, 8), (1, 1, 129), (4, 9, 13), (5, 8, 16), (1, 1, 1), (7, 40, 1)],
                         ids=lambda g: "x".join(map(str, g)))
def test_bf16_cta_pair_small_shapes(grid, mode):
    w = dataclasses.replace(configs.WAN13B_480P, B=2, H=3, T=grid[0], Hg=grid[1], Wg=grid[2], seed=43)
    mx, mean, lerr = _full_compare(w, kernel=vdx.KERNEL_PAIR, k_rope=K_MODES[mode])
    assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL, (mx, mean, lerr)


@pytest.mark.parametrize("grid", [(2, 9, 40), (1, 1, 129), (4, 9, 13)], ids=lambda g: "x".join(map(str, g)))
def test_bf16_cta_pair_split_precision_stress_small(grid):
    # the stress recipe with split operands, run by CTA pairs
    w = dataclasses.replace(configs.LONG_STRESS, B=1, H=4, T=grid[0], Hg=grid[1], Wg=grid[2], seed=45)
    assert w.qk == "split"
    mx, mean, lerr = _full_compare(w, kernel=vdx.KERNEL_PAIR)
    assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL, (mx, mean, lerr)


@pytest.mark.parametrize("mode", sorted(K_MODES))
def test_bf16_cta_pair_agrees_with_single_cta_kernel(mode):
    # same fp16 operands (up to the rounding of the rotation angles in the fused mode) and
    # softmax, different MMA shapes: equal to rounding
    w = dataclasses.replace(configs.WAN13B_480P, B=2, H=5, T=3, Hg=10, Wg=30, seed=44)
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    o1, l1 = _run(w, q, k, v, kernel=vdx.KERNEL_SINGLE, k_rope=K_MODES[mode])
    o2, l2 = _run(w, q, k, v, kernel=vdx.KERNEL_PAIR, k_rope=K_MODES[mode])
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-3
    assert (l1 - l2).abs().max().item() <= 1e-4


@pytest.mark.parametrize("kernel", ["single", "pair"])
@pytest.mark.parametrize("grid", [(3, 8, 8), (1, 1, 129), (4, 9, 13), (7, 40, 1)],
                         ids=lambda g: "x".join(map(str, g)))
def test_bf16_split_precision_small_shapes(grid, kernel):
    w = dataclasses.replace(configs.WAN13B_480P, B=2, H=3, T=grid[0], Hg=grid[1], Wg=grid[2], seed=26,
                            qk="split")
    mx, mean, lerr = _full_compare(w, kernel=vdx.KERNEL_PAIR if kernel == "pair" else vdx.KERNEL_SINGLE)
    # hi + lo operands: the score error is far below fp16's, so lse is far inside its tolerance
    assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL / 10, (mx, mean, lerr)


def test_bf16_caller_workspace_matches_library_workspace():
    w = dataclasses.replace(configs.WAN13B_480P, B=2, H=2, T=2, Hg=7, Wg=19, seed=25)
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    nbytes = vdx.workspace_bytes(w.B, w.H, (w.T, w.Hg, w.Wg))
    assert nbytes == 2 * q.numel() * 2          # rotated K and rotated Q, fp16 each
    ws = torch.empty(nbytes // 2 + 64, dtype=torch.float16, device="cuda")
    o1, l1 = _run(w, q, k, v, workspace=ws)
    o2, l2 = _run(w, q, k, v)
    o3, l3 = _run(w, q, k, v, k_rope=vdx.K_ROPE_FUSED)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # the two K modes round the same rotated values to fp16 (same scores); the kernels may
    # order their sums differently, so the outputs agree to rounding, not bit for bit
    assert (o1.float() - o3.float()).abs().max().item() <= 2e-3
    assert (l1 - l3).abs().max().item() <= 1e-4
    with pytest.raises(vdx.VdxError) as ei:
        vdx.rope3d_attn(q, k, v, (w.T, w.Hg, w.Wg), workspace=ws[:100])
    assert ei.value.status == 1
    # A query subset rotates its gathered rows itself: the rotated-K half of the workspace is
    # enough, and every row then matches the dense call.
    idx = torch.arange(w.N, dtype=torch.int32, device="cuda")
    o4, l4 = torch.zeros_like(o1), torch.zeros_like(l1)
    vdx.rope3d_attn_subset(q, k, v, (w.T, w.Hg, w.Wg), idx, o4, l4, w.sections, w.theta,
                           workspace=ws[:q.numel()])
    vdx.sync_check()
    assert (o4.float() - o1.float()).abs().max().item() <= 2e-3
    assert (l4 - l1).abs().max().item() <= 1e-4


@pytest.mark.parametrize("grid", [(2, 8, 16), (3, 10, 10)], ids=["N256", "N300_ragged"])
def test_bf16_many_heads_several_waves(grid):
    # 300 (b, h) pairs with one CTA each: about two waves of one CTA per SM, every CTA on a
    # different head, each compared in full with the oracle.
    w = dataclasses.replace(configs.WAN13B_480P, B=2, H=150, T=grid[0], Hg=grid[1], Wg=grid[2], seed=36)
    mx, mean, lerr = _full_compare(w)
    assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL, (mx, mean, lerr)


# the fused mode run by CTA pairs takes its rotation angles from per-pair frequencies instead
# of the cos/sin table, so custom sections and theta go through both
@pytest.mark.parametrize("kw", [{}, {"k_rope": vdx.K_ROPE_FUSED, "kernel": vdx.KERNEL_PAIR}],
                         ids=["default", "fused_pair"])
def test_bf16_custom_sections_theta_scale(kw):
    w = dataclasses.replace(configs.WAN13B_480P, B=1, H=2, T=3, Hg=6, Wg=20, sections=(64, 32, 32),
                            theta=500.0, seed=22)
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    out, lse = vdx.rope3d_attn(q, k, v, (3, 6, 20), w.sections, w.theta, scale=0.05, **kw)
    vdx.sync_check()
    ref_o, ref_l = O.rope3d_attention(q, k, v, (3, 6, 20), w.sections, w.theta, scale=0.05)
    assert np.abs(out.double().cpu().numpy() - ref_o).max() <= BF16_MAX
    assert np.abs(lse.double().cpu().numpy() - ref_l).max() <= LSE_TOL


def test_bf16_large_logits_small():
    # the stress recipe on a small grid, run (like the long-clip workload) with split operands
    w = dataclasses.replace(configs.LONG_STRESS, B=1, H=4, T=2, Hg=9, Wg=40, seed=23)
    assert w.qk == "split"
    mx, mean, lerr = _full_compare(w)
    assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL, (mx, mean, lerr)
    # one fp16 value per operand cannot hold these logits to 1e-3 (about 0.05 here), which is
    # why this workload uses the split mode; the output itself stays within tolerance
    mx16, mean16, lerr16 = _full_compare(w, qk_precision=vdx.QK_FP16)
    assert mx16 <= BF16_MAX and lerr16 > LSE_TOL


def test_bf16_late_logit_jump():
    # keys of the last tile scaled x25: for most rows the running maximum jumps by far more
    # than the kernel's in-range margin on tile 3, which takes its exact reload route.  Logits
    # this large need the split operands (fp16 alone leaves ~3e-2 here, as on the stress set).
    w = dataclasses.replace(configs.WAN13B_480P, B=1, H=2, T=4, Hg=8, Wg=16, seed=27, qk="split")
    q, k, v = synth.make_qkv(w)
    k = k.float()
    k[:, 400:410] *= 25.0
    k = k.to(torch.bfloat16)
    dev = tuple(t.cuda() for t in (q, k, v))
    mx, mean, lerr = _full_compare(w, dev)
    assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL, (mx, mean, lerr)


@pytest.mark.parametrize("first", [458, 392], ids=["second_half", "first_half"])
def test_bf16_logit_jump_within_a_tile(first):
    # Ten keys of the last tile (tokens 384..511) scaled x25: at 458 they sit in its second
    # half (keys 64..127 of the tile), at 392 in its first half, so both repair routes of the
    # softmax run (the first half already stored, or nothing stored yet).  A jump that large
    # needs the split operands to hold the lse tolerance (see the late-jump test above).
    w = dataclasses.replace(configs.WAN13B_480P, B=1, H=2, T=4, Hg=8, Wg=16, seed=35, qk="split")
    q, k, v = synth.make_qkv(w)
    k = k.float()
    k[:, first:first + 10] *= 25.0
    k = k.to(torch.bfloat16)
    dev = tuple(t.cuda() for t in (q, k, v))
    mx, mean, lerr = _full_compare(w, dev)
    assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL, (mx, mean, lerr)


def test_bf16_deterministic_and_guard_bands():
    w = dataclasses.replace(configs.WAN13B_480P, B=1, H=2, T=2, Hg=10, Wg=13, seed=24)
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    numel = q.numel()
    guard = 4096
    buf = torch.full((numel + 2 * guard,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + numel].view_as(q)
    lbuf = torch.full((w.B * w.H * w.N + 2 * guard,), -3.0, dtype=torch.float32, device="cuda")
    lse = lbuf[guard:guard + w.B * w.H * w.N].view(w.B, w.H, w.N)
    vdx.rope3d_attn(q, k, v, (w.T, w.Hg, w.Wg), out=out, lse=lse)
    vdx.sync_check()
    first = out.clone(), lse.clone()
    vdx.rope3d_attn(q, k, v, (w.T, w.Hg, w.Wg), out=out, lse=lse)
    vdx.sync_check()
    assert torch.equal(first[0], out) and torch.equal(first[1], lse)
    assert torch.all(buf[:guard] == 7.0) and torch.all(buf[guard + numel:] == 7.0)
    assert torch.all(lbuf[:guard] == -3.0) and torch.all(lbuf[guard + w.B * w.H * w.N:] == -3.0)
    out2, none = vdx.rope3d_attn(q, k, v, (w.T, w.Hg, w.Wg), return_lse=False)
    vdx.sync_check()
    assert none is None and torch.equal(out2, out)


def _sampled_compare(w, rows=512, sel=None, **kw):
    """Sampled rows of one full-size call against the oracle: (out max-abs, out mean-abs,
    lse max-abs, stats) with stats holding the relative guards and, for a stress workload,
    the errors on its outlier-token rows alone.  `sel` overrides the sampled (b, h, n) rows."""
    q, k, v = synth.make_qkv(w, device="cuda")
    out, lse = _run(w, q, k, v, **kw)
    sel = synth.sample_rows(w, rows) if sel is None else sel
    ref_o, ref_l = O.rope3d_attention_rows(q, k, v, (w.T, w.Hg, w.Wg), sel, w.sections, w.theta)
    b = torch.tensor([r[0] for r in sel], device="cuda")
    h = torch.tensor([r[1] for r in sel], device="cuda")
    n = torch.tensor([r[2] for r in sel], device="cuda")
    got_o = out[b, n, h].double().cpu().numpy()
    got_l = lse[b, h, n].double().cpu().numpy()
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    err = np.abs(got_o - ref_o)
    lerr = np.abs(got_l - ref_l)
    cos = (got_o * ref_o).sum(1) / (np.linalg.norm(got_o, axis=1) * np.linalg.norm(ref_o, axis=1))
    stats = {"rel_mean": err.mean() / np.abs(ref_o).mean(), "min_row_cos": cos.min()}
    if w.stress:
        _, tok = synth.outlier_indices(w)
        hot = np.isin(np.array([r[2] for r in sel]), tok.numpy())
        stats.update(outlier_rows=int(hot.sum()), outlier_out_max=err[hot].max(),
                     outlier_out_mean=err[hot].mean(), outlier_lse_max=lerr[hot].max(),
                     outlier_rel_mean=err[hot].mean() / np.abs(ref_o[hot]).mean())
    return err.max(), err.mean(), lerr.max(), stats


# At full size the attention of an ordinary row is spread over tens of thousands of keys, so
# |out| is only ~0.005 and the absolute bounds alone would pass an all-zero output or an O
# that missed a rescale.  Relative guards on the same sampled rows (derived here, on top of
# the stated tolerances): mean |err| <= 1 % of mean |ref|, and every row's cosine with the
# oracle's row >= 0.999.
REL_MEAN, MIN_COS = 1e-2, 0.999


def _assert_sampled(w, mx, mean, lerr, stats):
    assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL, (mx, mean, lerr)
    assert stats["rel_mean"] <= REL_MEAN and stats["min_row_cos"] >= MIN_COS, stats
    if w.stress:
        assert stats["outlier_rows"] == round(0.001 * w.N), stats
        assert (stats["outlier_out_max"] <= BF16_MAX and stats["outlier_out_mean"] <= BF16_MEAN and
                stats["outlier_lse_max"] <= LSE_TOL and stats["outlier_rel_mean"] <= REL_MEAN), stats


# Tensors of more than 2^31 elements: B = 2, H = 40, grid 59 x 45 x 80 (N = 212400) is
# 2.17e9 elements (4.35 GB of bf16) per tensor, so the rows of batch entry 1 sit past element
# offset 2^31 in q, k, v, out and the prepass workspace.  Rows of three heads (both batch
# entries, first and last heads), including each head's first and last tokens.
@pytest.mark.parametrize("k_rope", ["prepass", "fused"])
def test_tensors_beyond_2_31_elements_sampled(k_rope):
    w = dataclasses.replace(configs.WAN14B_720P, B=2, H=40, T=59, Hg=45, Wg=80, seed=61)
    assert w.B * w.N * w.H * w.d > 2 ** 31
    rng = np.random.default_rng(61)
    sel = []
    for b, h in [(1, 39), (1, 0), (0, 20)]:
        ns = [0, 1, w.N // 2, w.N - 2, w.N - 1] + list(rng.integers(0, w.N, 35))
        sel += [(b, h, int(n)) for n in ns]
    kw = {} if k_rope == "prepass" else {"k_rope": vdx.K_ROPE_FUSED}
    try:
        mx, mean, lerr, stats = _sampled_compare(w, sel=sel, **kw)
    finally:
        torch.cuda.empty_cache()
    print(f"2^31+ elements ({k_rope}): out max {mx:.3e} mean {mean:.3e} lse max {lerr:.3e} {stats}")
    _assert_sampled(w, mx, mean, lerr, stats)


@pytest.mark.parametrize("w", [configs.WAN13B_480P, configs.WAN14B_480P, configs.WAN14B_720P,
                               configs.LONG_STRESS], ids=lambda w: w.name)
def test_full_size_configs_sampled(w):
    mx, mean, lerr, stats = _sampled_compare(w)
    print(f"{w.name}: out max {mx:.3e} mean {mean:.3e} lse max {lerr:.3e} "
          + " ".join(f"{k} {v:.3e}" if isinstance(v, float) else f"{k} {v}" for k, v in stats.items()))
    _assert_sampled(w, mx, mean, lerr, stats)


# The other kernel than the default at full size: CTA pairs where one CTA is the default
# (N < 65536), one CTA where pairs are.
@pytest.mark.parametrize("w,kernel", [(configs.WAN13B_480P, "pair"), (configs.WAN14B_720P, "single"),
                                      (configs.LONG_STRESS, "single")], ids=lambda x: getattr(x, "name", x))
def test_full_size_other_kernel_sampled(w, kernel):
    kern = vdx.KERNEL_PAIR if kernel == "pair" else vdx.KERNEL_SINGLE
    mx, mean, lerr, stats = _sampled_compare(w, kernel=kern)
    print(f"{w.name} ({kernel}): out max {mx:.3e} mean {mean:.3e} lse max {lerr:.3e} {stats}")
    _assert_sampled(w, mx, mean, lerr, stats)


@pytest.mark.parametrize("w,kernel", [(configs.WAN13B_480P, "single"), (configs.WAN14B_720P, "pair")],
                         ids=lambda x: getattr(x, "name", x))
def test_full_size_fused_k_mode_sampled(w, kernel):
    kern = vdx.KERNEL_PAIR if kernel == "pair" else vdx.KERNEL_SINGLE
    mx, mean, lerr, stats = _sampled_compare(w, k_rope=vdx.K_ROPE_FUSED, kernel=kern)
    print(f"{w.name} (fused, {kernel}): out max {mx:.3e} mean {mean:.3e} lse max {lerr:.3e} {stats}")
    _assert_sampled(w, mx, mean, lerr, stats)


@pytest.mark.parametrize("sections,theta", [((128, 0, 0), 10000.0), ((0, 64, 64), 10000.0),
                                            ((44, 42, 42), 1.0e6), ((2, 2, 124), 2.0)])
@pytest.mark.parametrize("kw", [{}, {"k_rope": vdx.K_ROPE_FUSED, "kernel": vdx.KERNEL_PAIR}],
                         ids=["default", "fused_pair"])
def test_bf16_degenerate_sections_and_theta(sections, theta, kw):
    w = dataclasses.replace(configs.WAN13B_480P, B=1, H=2, T=3, Hg=7, Wg=11, seed=28,
                            sections=sections, theta=theta)
    mx, mean, lerr = _full_compare(w, **kw)
    assert mx <= BF16_MAX and mean <= BF16_MEAN and lerr <= LSE_TOL, (mx, mean, lerr)


@pytest.mark.parametrize("which", ["k", "q"])
def test_bf16_uniform_attention_closed_form(which):
    # Zero keys (or zero queries) make every logit 0: out = mean of V, lse = ln N.
    w = dataclasses.replace(configs.WAN13B_480P, B=2, H=2, T=2, Hg=9, Wg=21, seed=29)
    q, k, v = (t.cuda() for t in synth.make_qkv(w))
    if which == "k":
        k = torch.zeros_like(k)
    else:
        q = torch.zeros_like(q)
    out, lse = _run(w, q, k, v)
    mean_v = v.double().mean(dim=1, keepdim=True)
    assert (out.double() - mean_v).abs().max().item() <= 4e-3      # bf16 P = 1 exactly; bf16 out
    assert (lse.double() - np.log(w.N)).abs().max().item() <= 1e-5


@pytest.mark.parametrize("grid", [(1, 255, 128), (1, 1, 32641)], ids=["N_multiple_of_128", "N_one_past"])
@pytest.mark.parametrize("k_rope", ["prepass", "fused", "fused_pair"])
def test_long_rows_with_and_without_a_ragged_tile(grid, k_rope):
    # N = 255*128 (no ragged key tile) and N = 256*128 + 1 (a last tile of one key); the prepass
    # mode rotates Q in the prepass, the fused mode in every CTA.
    w = dataclasses.replace(configs.WAN13B_480P, B=1, H=2, T=grid[0], Hg=grid[1], Wg=grid[2], seed=34)
    kw = {"prepass": {}, "fused": {"k_rope": vdx.K_ROPE_FUSED, "kernel": vdx.KERNEL_SINGLE},
          "fused_pair": {"k_rope": vdx.K_ROPE_FUSED, "kernel": vdx.KERNEL_PAIR}}[k_rope]
    mx, mean, lerr, stats = _sampled_compare(w, rows=256, **kw)
    _assert_sampled(w, mx, mean, lerr, stats)
