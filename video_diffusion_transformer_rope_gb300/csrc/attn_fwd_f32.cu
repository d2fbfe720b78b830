// fp32 3D-RoPE attention on CUDA cores (d = 64 or 128), the library's full-precision path.
//
// Same operation as the tensor-core kernel (vidax: A Unified JAX Framework for Video
// Generative Models on Accelerator Meshes, §2 "3D RoPE, 3D VAEs, and flash attention"), with
// every product and sum in fp32, for callers that need fp32 accuracy (bf16 tensor-core
// operands cannot reach 1e-4).  One CTA = 16 query rows of one (batch, head); 4 warps, 4 rows
// each.  Key tiles of 32 tokens are rotated while being staged into shared memory; lane l of
// a warp scores key l, the row statistics come from warp shuffles, and lane l accumulates
// output channels l, l+32, ... with the online (running max / running sum) softmax.
#include <cuda_runtime.h>
#include <cstdint>
#include <cmath>

#include "vdx_internal.h"

namespace vdx {
namespace {

constexpr int kRows = 16;      // query rows per CTA
constexpr int kKeys = 32;      // keys per tile
constexpr int kWarps = 4;

struct F32Params {
  const float* q;
  const float* k;
  const float* v;
  float* out;
  float* lse;
  int B, H, N, Hg, Wg, HgWg;
  int half_t, half_h, half_w, off_h, off_w;
  float scale;
  const float2* table;
};

// Rotate the d channels of token n (src, stride 1) into dst.
template <int D>
__device__ __forceinline__ void rope_row(const F32Params& p, const float* __restrict__ src, int n,
                                         float* dst, int lane) {
  const int pt = n / p.HgWg;
  const int rem = n - pt * p.HgWg;
  const int ph = rem / p.Wg;
  const int pw = rem - ph * p.Wg;
  for (int pr = lane; pr < D / 2; pr += 32) {
    int idx;
    if (pr < p.half_t) idx = pt * p.half_t + pr;
    else if (pr < p.half_t + p.half_h) idx = p.off_h + ph * p.half_h + (pr - p.half_t);
    else idx = p.off_w + pw * p.half_w + (pr - p.half_t - p.half_h);
    const float2 cs = p.table[idx];
    const float x0 = src[2 * pr], x1 = src[2 * pr + 1];
    dst[2 * pr] = x0 * cs.x - x1 * cs.y;
    dst[2 * pr + 1] = x0 * cs.y + x1 * cs.x;
  }
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
attn_fwd_f32_kernel(const F32Params p) {
  __shared__ float sQ[kRows][D];
  __shared__ float sK[kKeys][D + 1];
  __shared__ float sV[kKeys][D];
  constexpr int kPer = D / 32;          // output channels per lane
  constexpr int kRowsPerWarp = kRows / kWarps;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qblk = (p.N + kRows - 1) / kRows;
  const int qblk = blockIdx.x % n_qblk;
  const int bh = blockIdx.x / n_qblk;
  const int b = bh / p.H, h = bh - b * p.H;
  const int q0 = qblk * kRows;
  const size_t tok_stride = static_cast<size_t>(p.H) * D;
  const size_t base = static_cast<size_t>(b) * p.N * tok_stride + static_cast<size_t>(h) * D;

  for (int r = warp; r < kRows; r += kWarps) {
    const int n = q0 + r;
    if (n < p.N) rope_row<D>(p, p.q + base + n * tok_stride, n, sQ[r], lane);
    else for (int c = lane; c < D; c += 32) sQ[r][c] = 0.f;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], o[kRowsPerWarp][kPer];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int u = 0; u < kPer; ++u) o[i][u] = 0.f;
  }

  for (int k0 = 0; k0 < p.N; k0 += kKeys) {
    __syncthreads();
    for (int r = warp; r < kKeys; r += kWarps) {
      const int n = k0 + r;
      if (n < p.N) {
        rope_row<D>(p, p.k + base + n * tok_stride, n, sK[r], lane);
        for (int c = lane; c < D; c += 32) sV[r][c] = p.v[base + n * tok_stride + c];
      } else {
        for (int c = lane; c < D; c += 32) { sK[r][c] = 0.f; sV[r][c] = 0.f; }
      }
    }
    __syncthreads();
    const bool key_live = (k0 + lane) < p.N;
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int r = warp * kRowsPerWarp + i;
      float s = 0.f;
#pragma unroll 8
      for (int c = 0; c < D; ++c) s = fmaf(sQ[r][c], sK[lane][c], s);
      s = key_live ? s * p.scale : -INFINITY;
      float mx = s;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_new = fmaxf(m[i], mx);
      const float alpha = expf(m[i] - m_new);   // 0 on the first tile (m = -inf)
      const float pk = key_live ? expf(s - m_new) : 0.f;
      float ps = pk;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l[i] = l[i] * alpha + ps;
      m[i] = m_new;
#pragma unroll
      for (int u = 0; u < kPer; ++u) o[i][u] *= alpha;
#pragma unroll 4
      for (int kk = 0; kk < kKeys; ++kk) {
        const float pw = __shfl_sync(0xffffffffu, pk, kk);
#pragma unroll
        for (int u = 0; u < kPer; ++u) o[i][u] = fmaf(pw, sV[kk][lane + 32 * u], o[i][u]);
      }
    }
  }

#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int n = q0 + warp * kRowsPerWarp + i;
    if (n >= p.N) continue;
    const float inv = 1.f / l[i];
    float* dst = p.out + base + n * tok_stride;
#pragma unroll
    for (int u = 0; u < kPer; ++u) dst[lane + 32 * u] = o[i][u] * inv;
    if (lane == 0 && p.lse != nullptr)
      p.lse[(static_cast<size_t>(b) * p.H + h) * p.N + n] = m[i] + logf(l[i]);
  }
}

}  // namespace

cudaError_t launch_attn_f32(const Problem& pr, cudaStream_t stream) {
  F32Params p{};
  p.q = static_cast<const float*>(pr.q);
  p.k = static_cast<const float*>(pr.k);
  p.v = static_cast<const float*>(pr.v);
  p.out = static_cast<float*>(pr.out);
  p.lse = pr.lse;
  p.B = pr.B; p.H = pr.H; p.N = pr.N; p.Hg = pr.Hg; p.Wg = pr.Wg; p.HgWg = pr.Hg * pr.Wg;
  p.half_t = pr.half_t; p.half_h = pr.half_h; p.half_w = pr.half_w;
  p.off_h = pr.T * pr.half_t;
  p.off_w = p.off_h + pr.Hg * pr.half_h;
  p.scale = pr.scale;
  p.table = pr.table;
  const long long grid = static_cast<long long>(pr.B) * pr.H * ((pr.N + kRows - 1) / kRows);
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (pr.d == 64) attn_fwd_f32_kernel<64><<<static_cast<unsigned>(grid), kWarps * 32, 0, stream>>>(p);
  else attn_fwd_f32_kernel<128><<<static_cast<unsigned>(grid), kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace vdx
