// Internal interface between the C-ABI front end (vdx_capi.cu) and the kernel translation
// units.  Not part of the public API.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <vector_types.h>
#include <cstdint>

namespace vdx {

// One attention problem, already validated, with its cos/sin table resident on the device.
// The table holds float2 (cos, sin) entries in three consecutive blocks:
//   [T][sec_t/2], then [Hgrid][sec_h/2], then [Wgrid][sec_w/2].
struct Problem {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;           // may be nullptr
  int B, H, T, Hg, Wg, N, d;
  int half_t, half_h, half_w;   // rotary pairs per axis
  double theta = 10000.0;       // rotary base
  float scale;
  const float2* table;
  int table_entries;
  // Optional block mask (device): row (b, h, query block of 256) at word offset
  // (b*H + h) * mask_bh_stride + qblock * mask_words; bit kb of word kb/32 selects key tile kb.
  // Optional active-query subset: rows are tokens q_index[b * q_index_b_stride + i], i < Nq.
  const int* q_index = nullptr;
  int Nq = 0;
  long long q_index_b_stride = 0;
  int withhold_kv = 0;        // testing only (vdx_attn_options.test_withhold_kv)
  const uint32_t* kv_mask = nullptr;
  int mask_words = 0;
  long long mask_bh_stride = 0;
};

// bf16, d = 128, tcgen05 kernel (attn_fwd_sm103.cu).  `encode` is cuTensorMapEncodeTiled.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// How K is rotated and how precise the QK^T operands are.
//   kPrepass: K is first rotated once into `workspace` (fp16 [B, N, H, d]) by a prepass kernel
//             on the same stream; fp16 QK operands.
//   kFused:   every CTA rotates its K tiles in shared memory; `workspace` is unused.
//   kSplit:   as kPrepass, with every rotated value split into fp16 hi + lo (workspace holds
//             both) and three QK products.
//   kPair:    as kPrepass, run by clusters of two CTAs that split every K/V tile between them
//             and multiply both CTAs' query rows with one cta_group::2 MMA (dense calls only).
//   kPairSplit: kSplit run by CTA pairs.
// With rotate_q_in_prepass (kPrepass / kSplit, no query subset) the prepass also rotates Q
// (multiplied by scale*log2(e)) into the workspace after K, and the attention kernel loads
// it rotated; otherwise every CTA rotates its Q tiles in shared memory.
enum class KMode { kPrepass, kFused, kSplit, kPair, kPairSplit, kPairFused };
cudaError_t launch_attn_bf16_sm103(const Problem& p, EncodeTiledFn encode, KMode mode,
                                   void* workspace, bool rotate_q_in_prepass, cudaStream_t stream,
                                   const char** what);
// Workspace bytes for kPrepass (split = false) or kSplit (split = true), with or without the
// rotated Q.
size_t prepass_workspace_bytes(const Problem& p, bool split, bool with_q);

// Read the tensor-core kernel's device error word (synchronous) and reset it to 0.
cudaError_t read_and_clear_error_word_sm103(unsigned int* word);

// Set the message vdx_last_error() returns on this host thread (vdx_capi.cu).
void set_last_error(const char* message);

// fp32, d in {64, 128}, CUDA-core kernel (attn_fwd_f32.cu).
cudaError_t launch_attn_f32(const Problem& p, cudaStream_t stream);

}  // namespace vdx
