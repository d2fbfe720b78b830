// vdx_rope3d_attn_noalloc: the bf16 attention call for callers that cannot allocate device
// memory at call time -- for example code running while a memory pool is frozen, an
// allocator-free embedding that must not call cudaMalloc/cudaFree (both synchronise the
// device and are not allowed everywhere), or a host that pre-sizes every buffer up front.
//
// The ordinary entry point allocates twice on first use: a per-device cos/sin table and the
// workspace that holds the rotated keys.  Here both live in one file-scope static device
// array of fixed size, so nothing is allocated per call; the caller still passes q, k, v, out
// and lse.  Costs of that choice:
//   * the array (kScratchBytes, about 64 MiB) is held on every GPU that loads this library
//     until the process exits;
//   * problems whose rotated keys need more than kWorkspaceBytes, or whose table needs more
//     than kTableEntries entries, are rejected with VDX_ERR_UNSUPPORTED;
//   * every call shares the array and it keeps the last call's contents, so calls that may
//     overlap on the GPU (different streams without ordering between them) race on it;
//   * the first call on a device looks up the array's device address there (host code only
//     knows a host-side stand-in for its name); make that first call before any stream
//     capture.
// Nothing in the array needs to start at zero: each call rewrites the table entries and the
// rotated keys it reads.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "vdx.h"
#include "vdx_internal.h"

namespace {

constexpr size_t kTableEntries = VDX_NOALLOC_MAX_TABLE_ENTRIES;
constexpr size_t kTableBytes = kTableEntries * sizeof(float2);
constexpr size_t kWorkspaceBytes = VDX_NOALLOC_MAX_WORKSPACE_BYTES;
constexpr size_t kScratchBytes = kTableBytes + kWorkspaceBytes;
static_assert(kTableBytes % 256 == 0, "workspace must stay 256-byte aligned");

// The scratch: cos/sin table first, then the rotated-key workspace.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDevices] = {};
vdx::EncodeTiledFn g_encode_fn = nullptr;

vdx_status fail_na(vdx_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  vdx::set_last_error(buf);     // reported by vdx_last_error()
  return s;
}

// Entry (axis, pos, j) of the cos/sin table at pos * theta^(-2j/S), computed in double on the
// device.  Layout as the ordinary table: [T][st/2], then [Hg][sh/2], then [Wg][sw/2].
__global__ void build_table_kernel(float2* tab, int T, int Hg, int Wg, int st, int sh, int sw,
                                   double theta) {
  const int n_t = T * (st / 2), n_h = Hg * (sh / 2), n_w = Wg * (sw / 2);
  const int total = n_t + n_h + n_w;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    int S, half, k;
    if (i < n_t) { S = st; k = i; }
    else if (i < n_t + n_h) { S = sh; k = i - n_t; }
    else { S = sw; k = i - n_t - n_h; }
    half = S / 2;
    const int pos = k / half, j = k - pos * half;
    const double ang = static_cast<double>(pos) * pow(theta, -2.0 * j / S);
    double s, c;
    sincos(ang, &s, &c);
    tab[i] = make_float2(static_cast<float>(c), static_cast<float>(s));
  }
}

// Device address of the scratch on the current device, looked up once per device.
vdx_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_na(VDX_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail_na(VDX_ERR_UNSUPPORTED, "device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return fail_na(VDX_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  if (g_encode_fn == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
      return fail_na(VDX_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(e));
    g_encode_fn = reinterpret_cast<vdx::EncodeTiledFn>(fn);
  }
  *out = g_scratch_addr[dev];
  return VDX_OK;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

}  // namespace

extern "C" vdx_status vdx_rope3d_attn_noalloc(const void* q, const void* k, const void* v,
                                              void* out, float* lse, int B, int H, int T,
                                              int Hgrid, int Wgrid, int d, int sec_t, int sec_h,
                                              int sec_w, double theta, float scale, void* stream) {
  vdx::set_last_error("");
  if (!q || !k || !v || !out) return fail_na(VDX_ERR_ARG, "q, k, v and out must be non-NULL");
  if (d != 128) return fail_na(VDX_ERR_UNSUPPORTED, "head_dim must be 128 (got %d)", d);
  if (B < 1 || H < 1 || T < 1 || Hgrid < 1 || Wgrid < 1)
    return fail_na(VDX_ERR_ARG, "B, H, T, Hgrid, Wgrid must be >= 1");
  if (sec_t == 0 && sec_h == 0 && sec_w == 0) {
    sec_h = sec_w = 2 * (d / 6);
    sec_t = d - sec_h - sec_w;
  }
  if (sec_t < 0 || sec_h < 0 || sec_w < 0 || ((sec_t | sec_h | sec_w) & 1) || sec_t + sec_h + sec_w != d)
    return fail_na(VDX_ERR_ARG, "rotary sections %d/%d/%d must be even, non-negative and sum to d=%d",
                   sec_t, sec_h, sec_w, d);
  if (!(theta > 0.0) || !std::isfinite(theta)) return fail_na(VDX_ERR_ARG, "theta must be > 0");
  if (!std::isfinite(scale)) return fail_na(VDX_ERR_ARG, "scale must be finite");
  const long long N = static_cast<long long>(T) * Hgrid * Wgrid;
  if (N > 0x3fffffffLL) return fail_na(VDX_ERR_ARG, "N = T*Hgrid*Wgrid is too large");
  const size_t bytes = static_cast<size_t>(B) * N * H * d * 2;
  if (bytes > kWorkspaceBytes)
    return fail_na(VDX_ERR_UNSUPPORTED,
                   "rotated keys need %zu bytes; the no-allocation scratch holds %zu "
                   "(B*N*H*d must be <= %zu)", bytes, kWorkspaceBytes, kWorkspaceBytes / 2);
  const size_t entries = static_cast<size_t>(T) * (sec_t / 2) + static_cast<size_t>(Hgrid) * (sec_h / 2) +
                         static_cast<size_t>(Wgrid) * (sec_w / 2);
  if (entries > kTableEntries)
    return fail_na(VDX_ERR_UNSUPPORTED, "cos/sin table needs %zu entries; the no-allocation scratch "
                   "holds %zu", entries, kTableEntries);
  const void* ptrs[5] = {q, k, v, out, lse};
  for (int i = 0; i < 5; ++i)
    if (ptrs[i] && (reinterpret_cast<uintptr_t>(ptrs[i]) & 15))
      return fail_na(VDX_ERR_ALIGN, "pointer argument %d is not 16-byte aligned", i);
  if (overlap(out, bytes, q, bytes) || overlap(out, bytes, k, bytes) || overlap(out, bytes, v, bytes))
    return fail_na(VDX_ERR_ARG, "out overlaps q, k or v");
  if (lse) {
    const size_t lb = static_cast<size_t>(B) * H * N * sizeof(float);
    if (overlap(lse, lb, out, bytes) || overlap(lse, lb, q, bytes) || overlap(lse, lb, k, bytes) ||
        overlap(lse, lb, v, bytes))
      return fail_na(VDX_ERR_ARG, "lse overlaps q, k, v or out");
  }

  void* scratch = nullptr;
  vdx_status s = scratch_address(&scratch);
  if (s != VDX_OK) return s;
  float2* table = static_cast<float2*>(scratch);
  void* workspace = static_cast<unsigned char*>(scratch) + kTableBytes;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  const int blocks = static_cast<int>((entries + 255) / 256);
  build_table_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(table, T, Hgrid, Wgrid, sec_t, sec_h,
                                                              sec_w, theta);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_na(VDX_ERR_CUDA, "table kernel launch: %s", cudaGetErrorString(e));

  vdx::Problem p{};
  p.q = q; p.k = k; p.v = v; p.out = out; p.lse = lse;
  p.B = B; p.H = H; p.T = T; p.Hg = Hgrid; p.Wg = Wgrid; p.N = static_cast<int>(N); p.d = d;
  p.half_t = sec_t / 2; p.half_h = sec_h / 2; p.half_w = sec_w / 2;
  p.theta = theta;
  p.scale = scale > 0.f ? scale : static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  p.table = table;
  p.table_entries = static_cast<int>(entries);
  const char* what = nullptr;
  e = vdx::launch_attn_bf16_sm103(p, g_encode_fn, vdx::KMode::kPrepass, workspace,
                                  /*rotate_q_in_prepass=*/false, st, &what);
  if (e != cudaSuccess) return fail_na(VDX_ERR_CUDA, "%s: %s", what ? what : "launch", cudaGetErrorString(e));
  return VDX_OK;
}
