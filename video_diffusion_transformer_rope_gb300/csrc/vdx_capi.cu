// C-ABI front end: argument checks, the per-device cos/sin table cache, the device error
// word, and dispatch to the bf16 tensor-core kernel or the fp32 CUDA-core kernel.
//
// The cos/sin table realises the rotary angles of vidax: A Unified JAX Framework for Video
// Generative Models on Accelerator Meshes, §2 "3D RoPE, 3D VAEs, and flash attention": for
// axis a with S_a rotary dims and pair j < S_a/2, angle = pos * theta^(-2j/S_a), evaluated in
// double precision and stored as float (cos, sin).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include <algorithm>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "vdx.h"
#include "vdx_internal.h"

namespace {

thread_local std::string t_last_error;

vdx_status fail(vdx_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

using TableKey = std::tuple<int, int, int, int, int, int, int, double>;   // dev,T,Hg,Wg,st,sh,sw,theta
struct TableEntry {
  float2* ptr;
  int entries;
};
std::mutex g_mu;
std::map<TableKey, TableEntry> g_tables;
struct Workspace {
  void* ptr;
  size_t bytes;
};
std::map<int, Workspace> g_workspace;     // library-owned K-prepass scratch, per device
vdx::EncodeTiledFn g_encode = nullptr;

// Entries: [T][st/2] then [Hg][sh/2] then [Wg][sw/2], each (cos, sin) of pos * theta^(-2j/S).
std::vector<float2> build_table(int T, int Hg, int Wg, int st, int sh, int sw, double theta) {
  std::vector<float2> tab;
  const int extents[3] = {T, Hg, Wg};
  const int secs[3] = {st, sh, sw};
  for (int a = 0; a < 3; ++a) {
    const int half = secs[a] / 2;
    for (int pos = 0; pos < extents[a]; ++pos) {
      for (int j = 0; j < half; ++j) {
        const double omega = std::pow(theta, -2.0 * j / secs[a]);
        const double ang = static_cast<double>(pos) * omega;
        tab.push_back(make_float2(static_cast<float>(std::cos(ang)), static_cast<float>(std::sin(ang))));
      }
    }
  }
  return tab;
}

vdx_status get_table(int T, int Hg, int Wg, int st, int sh, int sw, double theta,
                     const float2** out, int* entries) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(VDX_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  const TableKey key{dev, T, Hg, Wg, st, sh, sw, theta};
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_tables.find(key);
  if (it == g_tables.end()) {
    std::vector<float2> host = build_table(T, Hg, Wg, st, sh, sw, theta);
    float2* d = nullptr;
    const size_t bytes = std::max<size_t>(host.size(), 1) * sizeof(float2);
    e = cudaMalloc(&d, bytes);
    if (e != cudaSuccess) return fail(VDX_ERR_CUDA, "cudaMalloc(table): %s", cudaGetErrorString(e));
    if (!host.empty()) {
      e = cudaMemcpy(d, host.data(), host.size() * sizeof(float2), cudaMemcpyHostToDevice);
      if (e != cudaSuccess) {
        cudaFree(d);
        return fail(VDX_ERR_CUDA, "cudaMemcpy(table): %s", cudaGetErrorString(e));
      }
    }
    it = g_tables.emplace(key, TableEntry{d, static_cast<int>(host.size())}).first;
  }
  *out = it->second.ptr;
  *entries = it->second.entries;
  return VDX_OK;
}

vdx_status get_encode(vdx::EncodeTiledFn* fn) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_encode == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || p == nullptr)
      return fail(VDX_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(e));
    g_encode = reinterpret_cast<vdx::EncodeTiledFn>(p);
  }
  *fn = g_encode;
  return VDX_OK;
}

// Library-owned scratch of at least `bytes` on the current device (grow-only; growing frees
// the old buffer, which cudaFree does only after work already queued on the device).
vdx_status get_workspace(size_t bytes, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(VDX_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& w = g_workspace[dev];
  if (w.bytes < bytes) {
    if (w.ptr) cudaFree(w.ptr);
    w.ptr = nullptr;
    w.bytes = 0;
    e = cudaMalloc(&w.ptr, bytes);
    if (e != cudaSuccess) {
      w.ptr = nullptr;
      return fail(VDX_ERR_CUDA, "cudaMalloc(workspace, %zu bytes): %s", bytes, cudaGetErrorString(e));
    }
    w.bytes = bytes;
  }
  *out = w.ptr;
  return VDX_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Shared argument checks; fills `p` (except the table) on success.
vdx_status prepare(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                   int H, int T, int Hg, int Wg, int d, int st, int sh, int sw, double theta,
                   float scale, size_t esize, vdx::Problem* p) {
  if (!q || !k || !v || !out) return fail(VDX_ERR_ARG, "q, k, v and out must be non-NULL");
  if (B < 1 || H < 1 || T < 1 || Hg < 1 || Wg < 1 || d < 2)
    return fail(VDX_ERR_ARG, "B, H, T, Hgrid, Wgrid must be >= 1 and d >= 2 (got %d %d %d %d %d, d=%d)",
                B, H, T, Hg, Wg, d);
  if (st == 0 && sh == 0 && sw == 0) {
    sh = sw = 2 * (d / 6);
    st = d - sh - sw;
  }
  if (st < 0 || sh < 0 || sw < 0 || (st | sh | sw) & 1 || st + sh + sw != d)
    return fail(VDX_ERR_ARG, "rotary sections %d/%d/%d must be even, non-negative and sum to d=%d",
                st, sh, sw, d);
  if (!(theta > 0.0) || !std::isfinite(theta)) return fail(VDX_ERR_ARG, "theta must be > 0");
  if (!std::isfinite(scale)) return fail(VDX_ERR_ARG, "scale must be finite");
  const long long N = static_cast<long long>(T) * Hg * Wg;
  if (N > 0x7fffffffLL / 2) return fail(VDX_ERR_ARG, "N = T*Hgrid*Wgrid = %lld is too large", N);
  const long long elems = static_cast<long long>(B) * N * H * d;
  if (elems > (1LL << 46)) return fail(VDX_ERR_ARG, "tensor too large");
  const void* ptrs[5] = {q, k, v, out, lse};
  for (int i = 0; i < 5; ++i)
    if (ptrs[i] && (reinterpret_cast<uintptr_t>(ptrs[i]) & 15))
      return fail(VDX_ERR_ALIGN, "pointer argument %d is not 16-byte aligned", i);
  const size_t bytes = static_cast<size_t>(elems) * esize;
  if (overlaps(out, bytes, q, bytes) || overlaps(out, bytes, k, bytes) || overlaps(out, bytes, v, bytes))
    return fail(VDX_ERR_ARG, "out overlaps q, k or v");
  if (lse) {
    const size_t lb = static_cast<size_t>(B) * H * N * sizeof(float);
    if (overlaps(lse, lb, out, bytes) || overlaps(lse, lb, q, bytes) || overlaps(lse, lb, k, bytes) ||
        overlaps(lse, lb, v, bytes))
      return fail(VDX_ERR_ARG, "lse overlaps q, k, v or out");
  }
  p->q = q; p->k = k; p->v = v; p->out = out; p->lse = lse;
  p->B = B; p->H = H; p->T = T; p->Hg = Hg; p->Wg = Wg; p->N = static_cast<int>(N); p->d = d;
  p->half_t = st / 2; p->half_h = sh / 2; p->half_w = sw / 2;
  p->scale = scale > 0.f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  const float2* tab = nullptr;
  int entries = 0;
  vdx_status s = get_table(T, Hg, Wg, st, sh, sw, theta, &tab, &entries);
  if (s != VDX_OK) return s;
  p->table = tab;
  p->table_entries = entries;
  p->theta = theta;
  return VDX_OK;
}

}  // namespace

namespace vdx {
void set_last_error(const char* message) { t_last_error = message; }
}  // namespace vdx

extern "C" {

// NVTX range over a host call (shows up in profilers that record NVTX; free otherwise).
struct NvtxScope {
  explicit NvtxScope(const char* name) { nvtxRangePushA(name); }
  ~NvtxScope() { nvtxRangePop(); }
};

static vdx_status attn_bf16(const void* q, const void* k, const void* v, void* out, float* lse,
                            int B, int H, int T, int Hgrid, int Wgrid, int d, int sec_t, int sec_h,
                            int sec_w, double theta, float scale, const vdx_attn_options* opt,
                            const uint32_t* block_mask, int mask_per_head, void* stream,
                            const int32_t* q_index = nullptr, int Nq = 0, int index_per_batch = 0) {
  NvtxScope nvtx(block_mask ? "vdx_rope3d_attn_sparse" : (q_index ? "vdx_rope3d_attn_subset" : "vdx_rope3d_attn"));
  t_last_error.clear();
  if (d != 128) return fail(VDX_ERR_UNSUPPORTED, "bf16 path supports head_dim 128 only (got %d)", d);
  const int mode = opt ? opt->k_rope : VDX_K_ROPE_DEFAULT;
  if (mode != VDX_K_ROPE_DEFAULT && mode != VDX_K_ROPE_PREPASS && mode != VDX_K_ROPE_FUSED)
    return fail(VDX_ERR_ARG, "unknown k_rope mode %d", mode);
  const int prec = opt ? opt->qk_precision : VDX_QK_FP16;
  if (prec != VDX_QK_FP16 && prec != VDX_QK_SPLIT)
    return fail(VDX_ERR_ARG, "unknown qk_precision %d", prec);
  const bool fused = mode == VDX_K_ROPE_FUSED;
  const bool split = prec == VDX_QK_SPLIT;
  const int kernel = opt ? opt->kernel : VDX_KERNEL_DEFAULT;
  if (kernel != VDX_KERNEL_DEFAULT && kernel != VDX_KERNEL_SINGLE && kernel != VDX_KERNEL_PAIR)
    return fail(VDX_ERR_ARG, "unknown kernel %d", kernel);
  if (kernel == VDX_KERNEL_PAIR && (block_mask || q_index))
    return fail(VDX_ERR_UNSUPPORTED, "VDX_KERNEL_PAIR takes dense calls only");
  // CTA pairs by default for dense calls with split operands (halving each CTA's K/V stages
  // lets its rings hold two stages instead of one: +16 % at N = 111600, +20 % at N = 32760)
  // and for long dense sequences with fp16 operands (N >= 65536, >= 512 key tiles per CTA): at
  // the same power pairs run ~7 % higher clocks (half the shared-memory operand reads and
  // L2->SM traffic per CTA), which outweighs their longer cross-SM signalling there (+0.8 % at
  // N = 75600); at N = 32760 they measured -1.8 % to +0.2 %, so shorter fp16 calls keep one CTA.
  // With the fused K rotation pairs halve each CTA's rotation work: 1.58x faster at N = 32760
  // and 75600 (H = 12 and 40).
  const long long n_tokens = static_cast<long long>(T) * Hgrid * Wgrid;
  const bool pair = kernel == VDX_KERNEL_PAIR ||
                    (kernel == VDX_KERNEL_DEFAULT && !block_mask && !q_index &&
                     (fused || split || n_tokens >= 65536));
  if (fused && split)
    return fail(VDX_ERR_UNSUPPORTED, "VDX_QK_SPLIT needs the K prepass (k_rope = VDX_K_ROPE_PREPASS)");
  vdx::Problem p{};
  vdx_status s = prepare(q, k, v, out, lse, B, H, T, Hgrid, Wgrid, d, sec_t, sec_h, sec_w, theta,
                         scale, 2, &p);
  if (s != VDX_OK) return s;
  p.withhold_kv = (opt && opt->test_withhold_kv) ? 1 : 0;
  if (q_index) {
    if (reinterpret_cast<uintptr_t>(q_index) & 3)
      return fail(VDX_ERR_ALIGN, "q_index is not 4-byte aligned");
    p.q_index = q_index;
    p.Nq = Nq;
    p.q_index_b_stride = index_per_batch ? Nq : 0;
  }
  if (block_mask) {
    if (reinterpret_cast<uintptr_t>(block_mask) & 3)
      return fail(VDX_ERR_ALIGN, "block_mask is not 4-byte aligned");
    const int nkv = (p.N + VDX_SPARSE_KBLOCK - 1) / VDX_SPARSE_KBLOCK;
    const int nqb = (p.N + VDX_SPARSE_QBLOCK - 1) / VDX_SPARSE_QBLOCK;
    p.kv_mask = block_mask;
    p.mask_words = (nkv + 31) / 32;
    p.mask_bh_stride = mask_per_head ? static_cast<long long>(nqb) * p.mask_words : 0;
  }
  // The prepass rotates Q as well (one bandwidth-bound pass at copy speed) instead of every CTA
  // rotating its two Q tiles in shared memory (about 8 us per CTA, latency-bound).  A query
  // subset gathers and rotates its rows in the kernel.
  const bool q_pre = !fused && p.q_index == nullptr;
  void* ws = nullptr;
  if (!fused) {
    const size_t need = vdx::prepass_workspace_bytes(p, split, q_pre);
    if (opt && opt->workspace) {
      if (opt->workspace_bytes < need)
        return fail(VDX_ERR_ARG, "workspace of %zu bytes is smaller than the %zu needed",
                    opt->workspace_bytes, need);
      if (reinterpret_cast<uintptr_t>(opt->workspace) & 15)
        return fail(VDX_ERR_ALIGN, "workspace is not 16-byte aligned");
      // q, k, v and out each span B*N*H*d bf16 values; the workspace spans `need` bytes
      // (twice a tensor in the split mode).
      const size_t tb = static_cast<size_t>(p.B) * p.N * p.H * p.d * 2;
      if (overlaps(opt->workspace, need, q, tb) || overlaps(opt->workspace, need, k, tb) ||
          overlaps(opt->workspace, need, v, tb) || overlaps(opt->workspace, need, out, tb) ||
          (lse && overlaps(opt->workspace, need, lse, static_cast<size_t>(p.B) * p.H * p.N * 4)))
        return fail(VDX_ERR_ARG, "workspace overlaps q, k, v, out or lse");
      ws = opt->workspace;
    } else if ((s = get_workspace(need, &ws)) != VDX_OK) {
      return s;
    }
  }
  vdx::EncodeTiledFn enc = nullptr;
  if ((s = get_encode(&enc)) != VDX_OK) return s;
  const char* what = nullptr;
  const vdx::KMode km = fused ? (pair ? vdx::KMode::kPairFused : vdx::KMode::kFused)
                              : (split ? (pair ? vdx::KMode::kPairSplit : vdx::KMode::kSplit)
                                       : (pair ? vdx::KMode::kPair : vdx::KMode::kPrepass));
  cudaError_t e = vdx::launch_attn_bf16_sm103(p, enc, km, ws, q_pre, static_cast<cudaStream_t>(stream),
                                              &what);
  if (e != cudaSuccess)
    return fail(VDX_ERR_CUDA, "%s: %s", what ? what : "launch", cudaGetErrorString(e));
  return VDX_OK;
}

vdx_status vdx_rope3d_attn_ex(const void* q, const void* k, const void* v, void* out, float* lse,
                              int B, int H, int T, int Hgrid, int Wgrid, int d, int sec_t,
                              int sec_h, int sec_w, double theta, float scale,
                              const vdx_attn_options* opt, void* stream) {
  return attn_bf16(q, k, v, out, lse, B, H, T, Hgrid, Wgrid, d, sec_t, sec_h, sec_w, theta, scale,
                   opt, nullptr, 0, stream);
}

vdx_status vdx_rope3d_attn(const void* q, const void* k, const void* v, void* out, float* lse,
                           int B, int H, int T, int Hgrid, int Wgrid, int d, int sec_t, int sec_h,
                           int sec_w, double theta, float scale, void* stream) {
  return vdx_rope3d_attn_ex(q, k, v, out, lse, B, H, T, Hgrid, Wgrid, d, sec_t, sec_h, sec_w,
                            theta, scale, nullptr, stream);
}

vdx_status vdx_rope3d_attn_sparse(const void* q, const void* k, const void* v, void* out,
                                  float* lse, int B, int H, int T, int Hgrid, int Wgrid, int d,
                                  int sec_t, int sec_h, int sec_w, double theta, float scale,
                                  const uint32_t* block_mask, int mask_per_head,
                                  const vdx_attn_options* opt, void* stream) {
  if (!block_mask) {
    t_last_error.clear();
    return fail(VDX_ERR_ARG, "block_mask must be non-NULL");
  }
  if (opt && opt->k_rope == VDX_K_ROPE_FUSED) {
    t_last_error.clear();
    // fused K rotation is kept for the dense call only
    return fail(VDX_ERR_UNSUPPORTED, "block-sparse calls use the K prepass");
  }
  return attn_bf16(q, k, v, out, lse, B, H, T, Hgrid, Wgrid, d, sec_t, sec_h, sec_w, theta, scale,
                   opt, block_mask, mask_per_head, stream);
}

vdx_status vdx_rope3d_attn_subset(const void* q, const void* k, const void* v, void* out,
                                  float* lse, int B, int H, int T, int Hgrid, int Wgrid, int d,
                                  int sec_t, int sec_h, int sec_w, double theta, float scale,
                                  const int32_t* q_index, int Nq, int index_per_batch,
                                  const vdx_attn_options* opt, void* stream) {
  if (!q_index || Nq < 0) {
    t_last_error.clear();
    return fail(VDX_ERR_ARG, "q_index must be non-NULL and Nq >= 0");
  }
  if (Nq == 0) {
    t_last_error.clear();
    return VDX_OK;
  }
  return attn_bf16(q, k, v, out, lse, B, H, T, Hgrid, Wgrid, d, sec_t, sec_h, sec_w, theta, scale,
                   opt, nullptr, 0, stream, q_index, Nq, index_per_batch);
}

int vdx_rope3d_block_mask_words(int T, int Hgrid, int Wgrid) {
  if (T < 1 || Hgrid < 1 || Wgrid < 1) return 0;
  const long long N = static_cast<long long>(T) * Hgrid * Wgrid;
  const long long nkv = (N + VDX_SPARSE_KBLOCK - 1) / VDX_SPARSE_KBLOCK;
  return static_cast<int>((nkv + 31) / 32);
}

vdx_status vdx_window_block_mask(uint32_t* mask, int T, int Hgrid, int Wgrid, int wt, int wh,
                                 int ww) {
  t_last_error.clear();
  if (!mask) return fail(VDX_ERR_ARG, "mask must be non-NULL");
  if (T < 1 || Hgrid < 1 || Wgrid < 1) return fail(VDX_ERR_ARG, "grid extents must be >= 1");
  if (wt < 0 || wh < 0 || ww < 0) return fail(VDX_ERR_ARG, "window half-widths must be >= 0");
  const long long N = static_cast<long long>(T) * Hgrid * Wgrid;
  if (N > 0x3fffffffLL) return fail(VDX_ERR_ARG, "grid too large");
  const int HW = Hgrid * Wgrid;
  // A block of consecutive tokens is a few runs along w: (t, h, w0..w1).
  struct Run { int t, h, w0, w1; };
  auto runs_of = [&](long long start, long long end, std::vector<Run>& out) {
    out.clear();
    for (long long n = start; n < end;) {
      const int t = static_cast<int>(n / HW), h = static_cast<int>((n / Wgrid) % Hgrid);
      const int w0 = static_cast<int>(n % Wgrid);
      const int w1 = static_cast<int>(std::min<long long>(Wgrid - 1, w0 + (end - 1 - n)));
      out.push_back({t, h, w0, w1});
      n += w1 - w0 + 1;
    }
  };
  const int nkv = static_cast<int>((N + VDX_SPARSE_KBLOCK - 1) / VDX_SPARSE_KBLOCK);
  const int nqb = static_cast<int>((N + VDX_SPARSE_QBLOCK - 1) / VDX_SPARSE_QBLOCK);
  const int words = (nkv + 31) / 32;
  std::vector<std::vector<Run>> kruns(nkv);
  for (int kb = 0; kb < nkv; ++kb)
    runs_of(static_cast<long long>(kb) * VDX_SPARSE_KBLOCK,
            std::min<long long>(N, static_cast<long long>(kb + 1) * VDX_SPARSE_KBLOCK), kruns[kb]);
  std::vector<Run> qruns;
  for (int qb = 0; qb < nqb; ++qb) {
    runs_of(static_cast<long long>(qb) * VDX_SPARSE_QBLOCK,
            std::min<long long>(N, static_cast<long long>(qb + 1) * VDX_SPARSE_QBLOCK), qruns);
    uint32_t* row = mask + static_cast<size_t>(qb) * words;
    for (int w = 0; w < words; ++w) row[w] = 0u;
    for (int kb = 0; kb < nkv; ++kb) {
      bool near = false;
      for (const Run& a : qruns) {
        for (const Run& c : kruns[kb]) {
          if (std::abs(a.t - c.t) <= wt && std::abs(a.h - c.h) <= wh && a.w0 <= c.w1 + ww &&
              c.w0 <= a.w1 + ww) {
            near = true;
            break;
          }
        }
        if (near) break;
      }
      if (near) row[kb / 32] |= 1u << (kb % 32);
    }
  }
  return VDX_OK;
}

size_t vdx_rope3d_workspace_bytes(int B, int H, int T, int Hgrid, int Wgrid, int d,
                                  int qk_precision) {
  if (B < 1 || H < 1 || T < 1 || Hgrid < 1 || Wgrid < 1 || d < 1) return 0;
  return static_cast<size_t>(B) * T * Hgrid * Wgrid * H * d * 2 * (qk_precision == VDX_QK_SPLIT ? 2 : 1) * 2;
}

vdx_status vdx_rope3d_attn_f32(const float* q, const float* k, const float* v, float* out,
                               float* lse, int B, int H, int T, int Hgrid, int Wgrid, int d,
                               int sec_t, int sec_h, int sec_w, double theta, float scale,
                               void* stream) {
  NvtxScope nvtx("vdx_rope3d_attn_f32");
  t_last_error.clear();
  if (d != 64 && d != 128)
    return fail(VDX_ERR_UNSUPPORTED, "fp32 path supports head_dim 64 or 128 (got %d)", d);
  vdx::Problem p{};
  vdx_status s = prepare(q, k, v, out, lse, B, H, T, Hgrid, Wgrid, d, sec_t, sec_h, sec_w, theta,
                         scale, 4, &p);
  if (s != VDX_OK) return s;
  cudaError_t e = vdx::launch_attn_f32(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(VDX_ERR_CUDA, "fp32 kernel launch: %s", cudaGetErrorString(e));
  return VDX_OK;
}

vdx_status vdx_sync_check(void* stream) {
  t_last_error.clear();
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(VDX_ERR_CUDA, "cudaStreamSynchronize: %s", cudaGetErrorString(e));
  unsigned int word = 0;
  e = vdx::read_and_clear_error_word_sm103(&word);
  if (e != cudaSuccess) return fail(VDX_ERR_CUDA, "reading the error word: %s", cudaGetErrorString(e));
  if (word & 1u)
    return fail(VDX_ERR_TIMEOUT, "a kernel pipeline wait gave up (site %u)", (word >> 8) & 0xff);
  if (word & 2u)
    return fail(VDX_ERR_RANGE, "a rotated q/k value exceeded the fp16 operand range (|x| > 65504); "
                               "it was clamped and the result is inexact");
  if (word & 4u)
    return fail(VDX_ERR_ARG, "a q_index entry was outside [0, N); those rows were skipped");
  return VDX_OK;
}

const char* vdx_last_error(void) { return t_last_error.c_str(); }

void vdx_shutdown(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto& kv : g_tables) {
    cudaSetDevice(std::get<0>(kv.first));
    cudaFree(kv.second.ptr);
  }
  for (auto& kv : g_workspace) {
    cudaSetDevice(kv.first);
    if (kv.second.ptr) cudaFree(kv.second.ptr);
  }
  cudaSetDevice(cur);
  g_tables.clear();
  g_workspace.clear();
}

int vdx_version(void) { return 100; }

}  // extern "C"
