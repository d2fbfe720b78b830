/* vdx — 3D-RoPE full spatiotemporal self-attention for video diffusion transformers, on one
 * GB300 (sm_103a).
 *
 * Operation (vidax: A Unified JAX Framework for Video Generative Models on Accelerator
 * Meshes, §2 "3D RoPE, 3D VAEs, and flash attention": rotary 3D position embedding on Q and
 * K, then attention that never materialises the N x N score matrix; §1 "Motivation and gap":
 * tens of thousands of latent-patch tokens).  For batch b, head h, query token n:
 *
 *     q'_n  = R(n) q_n,   k'_m = R(m) k_m
 *     lse_n = log sum_m exp(scale * <q'_n, k'_m>)           (natural log, all m: non-causal)
 *     out_n = sum_m exp(scale * <q'_n, k'_m> - lse_n) v_m
 *
 * R(n) rotates adjacent channel pairs (2i, 2i+1) like a complex number times exp(i*angle).
 * head_dim d is split into three rotary sections, in this order: sec_t dims turning with the
 * frame index t, sec_h with the grid row h, sec_w with the grid column w.  Within a section of
 * S dims, pair j turns at angle pos * theta^(-2j/S).  Token n = t*Hgrid*Wgrid + h*Wgrid + w.
 *
 * Layouts (row-major, contiguous):
 *   q, k, v, out : [B, N, H, d]   with N = T*Hgrid*Wgrid
 *   lse          : [B, H, N]      float32, may be NULL
 *
 * Ownership: every pointer is a device pointer owned by the caller.  The library owns only a
 * per-device cache of cos/sin tables (one per distinct grid/sections/theta; built on the
 * first call with that key, which allocates and uploads synchronously) and an error word;
 * vdx_shutdown() frees the tables.  Calls are asynchronous on `stream` (a cudaStream_t; NULL
 * means the legacy default stream).
 *
 * Errors: argument problems are reported before anything is launched and return a non-zero
 * vdx_status; vdx_last_error() gives a message (per host thread).  Device-side problems (a
 * pipeline wait that gave up after 1 s) are latched in a device error word read and cleared
 * by vdx_sync_check().
 */
#ifndef VDX_H_
#define VDX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  VDX_OK = 0,
  VDX_ERR_ARG = 1,          /* bad size, section split, NULL pointer, aliasing        */
  VDX_ERR_ALIGN = 2,        /* a pointer is not 16-byte aligned                       */
  VDX_ERR_UNSUPPORTED = 3,  /* valid, but outside what this build implements          */
  VDX_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed                      */
  VDX_ERR_TIMEOUT = 5,      /* a kernel pipeline wait gave up (see vdx_sync_check)    */
  VDX_ERR_RANGE = 6         /* a rotated q/k value left the fp16 operand range         */
} vdx_status;

/* How K gets rotated on the bf16 path. */
#define VDX_K_ROPE_DEFAULT 0  /* = VDX_K_ROPE_PREPASS                                          */
#define VDX_K_ROPE_PREPASS 1  /* a prepass kernel rotates every key token once into an fp16
                                 workspace [B, N, H, d]; the attention kernel streams it      */
#define VDX_K_ROPE_FUSED 2    /* each CTA rotates every K tile in shared memory as it lands
                                 (no workspace; the rotation is repeated per query block)     */

/* Precision of the rotated Q/K operands of QK^T on the bf16 path. */
#define VDX_QK_FP16 0         /* one fp16 value per rotated element (default; fastest)          */
#define VDX_QK_SPLIT 1        /* fp16 hi + lo per element and three products (~22 significant
                                 bits): for activations whose logits reach the hundreds; about
                                 half the speed; needs the K prepass and twice its workspace  */

/* Which attention kernel runs a dense bf16 call. */
#define VDX_KERNEL_DEFAULT 0  /* VDX_KERNEL_PAIR for dense calls with VDX_K_ROPE_FUSED, with
                                 VDX_QK_SPLIT, or with VDX_QK_FP16 and N >= 65536; else
                                 VDX_KERNEL_SINGLE                                                */
#define VDX_KERNEL_SINGLE 1   /* one CTA per 256 query rows, each streaming whole K/V tiles          */
#define VDX_KERNEL_PAIR 2     /* clusters of two CTAs: each holds half of every K/V tile and the pair
                                 multiplies both CTAs' 512 query rows with CTA-pair MMAs; dense
                                 calls only (block-sparse and query-subset calls get
                                 VDX_ERR_UNSUPPORTED).  With VDX_K_ROPE_FUSED each CTA rotates
                                 its own Q tiles and its 64 keys of every K tile                */

typedef struct vdx_attn_options {
  int k_rope;               /* one of VDX_K_ROPE_*                                              */
  int qk_precision;         /* one of VDX_QK_*                                                  */
  void* workspace;          /* device scratch for the prepass, >= vdx_rope3d_workspace_bytes()
                               bytes, 16-byte aligned, not overlapping q/k/v/out/lse; NULL = a
                               library-owned per-device buffer (allocated or grown with
                               cudaMalloc on first need; shared by every call on that device, so
                               calls that may overlap on different streams should pass their own) */
  size_t workspace_bytes;   /* size of `workspace` in bytes                                      */
  int test_withhold_kv;     /* testing only, keep 0: the kernel's copy engine issues no K/V tile,
                               so every pipeline wait runs out (after about 1 s); the kernel then
                               stops cleanly and vdx_sync_check reports VDX_ERR_TIMEOUT (this is
                               how the failure path is exercised without faulting the GPU)    */
  int kernel;               /* one of VDX_KERNEL_*                                              */
} vdx_attn_options;

/* bf16 path, tcgen05 tensor cores.  q, k, v, out: __nv_bfloat16 [B, N, H, d]; d must be 128.
 * Arithmetic: rotation in fp32; rotated k, and rotated q multiplied by scale*log2(e), rounded
 * to fp16 for QK^T (so |k| and |q|*scale*log2(e) must stay below ~46000, else values are
 * clamped and vdx_sync_check reports VDX_ERR_RANGE); scores (in log2 units), softmax
 * statistics and the output accumulator in fp32; P and v enter PV as bf16.
 * sec_t/sec_h/sec_w: even, sum to d; all three 0 selects d - 4*(d/6), 2*(d/6), 2*(d/6)
 * (44/42/42 at d = 128).  scale <= 0 selects 1/sqrt(d).  theta > 0 (10000 for Wan).
 * out must not overlap q, k or v.  B, H, T, Hgrid, Wgrid >= 1. */
vdx_status vdx_rope3d_attn(const void* q, const void* k, const void* v, void* out, float* lse,
                           int B, int H, int T, int Hgrid, int Wgrid, int d,
                           int sec_t, int sec_h, int sec_w, double theta, float scale,
                           void* stream);

/* Same as vdx_rope3d_attn with explicit options (NULL = defaults: K prepass, fp16 QK operands,
 * library-owned workspace). */
vdx_status vdx_rope3d_attn_ex(const void* q, const void* k, const void* v, void* out, float* lse,
                              int B, int H, int T, int Hgrid, int Wgrid, int d,
                              int sec_t, int sec_h, int sec_w, double theta, float scale,
                              const vdx_attn_options* opt, void* stream);

/* Bytes of workspace the prepass needs for this problem: the rotated K and the rotated,
 * scale*log2(e)-multiplied Q as fp16 [B, N, H, d] each (2*B*N*H*d*2), twice that with
 * VDX_QK_SPLIT (hi + lo parts); 0 for invalid sizes.  A query-subset call rotates its gathered
 * rows itself and uses only the first half (the rotated K). */
size_t vdx_rope3d_workspace_bytes(int B, int H, int T, int Hgrid, int Wgrid, int d,
                                  int qk_precision);

/* ---- Block-sparse attention (the bit-wise block-sparse kernel of the ScalingAttention abstract
 * on the papers page 2606.17566; masks here are caller-defined).  Keys are
 * cut into tiles of VDX_SPARSE_KBLOCK tokens and queries into blocks of VDX_SPARSE_QBLOCK
 * tokens; query n attends only to the key tiles its block's mask selects (a query whose mask
 * row selects nothing gets out = 0 and lse = -inf).  Skipped tiles cost no work.
 *   block_mask: device uint32 words, row-major [M][n_qblocks][W] with
 *     W = vdx_rope3d_block_mask_words(T, Hgrid, Wgrid), n_qblocks = ceil(N / 256),
 *     M = B*H (mask_per_head = 1, one mask per (b, h)) or 1 (mask_per_head = 0, shared);
 *     bit (kb % 32) of word kb / 32 selects key tile kb; bits at or beyond ceil(N/128) ignored.
 *   Other arguments, rules and options as vdx_rope3d_attn_ex (K prepass only). */
#define VDX_SPARSE_QBLOCK 256
#define VDX_SPARSE_KBLOCK 128
vdx_status vdx_rope3d_attn_sparse(const void* q, const void* k, const void* v, void* out,
                                  float* lse, int B, int H, int T, int Hgrid, int Wgrid, int d,
                                  int sec_t, int sec_h, int sec_w, double theta, float scale,
                                  const uint32_t* block_mask, int mask_per_head,
                                  const vdx_attn_options* opt, void* stream);

/* ---- Active-query subset (after the KV-cache synchronization of the Heterogeneous Step
 * Allocation abstract on the papers page 2606.17566: only active query tokens are recomputed,
 * against the full K/V).
 * Query rows are the tokens q_index[i], i < Nq (device int32; one list shared by every batch
 * entry when index_per_batch = 0, else [B][Nq]); each is rotated at its own grid position,
 * attends to all N keys, and its result is written to out[b, q_index[i], h, :] and
 * lse[b, h, q_index[i]].  Rows of out / lse not listed are left untouched.  An index outside
 * [0, N) is skipped and reported by vdx_sync_check (VDX_ERR_ARG).  Duplicate indices write
 * the same values twice.  Other arguments, rules and options as vdx_rope3d_attn_ex. */
vdx_status vdx_rope3d_attn_subset(const void* q, const void* k, const void* v, void* out,
                                  float* lse, int B, int H, int T, int Hgrid, int Wgrid, int d,
                                  int sec_t, int sec_h, int sec_w, double theta, float scale,
                                  const int32_t* q_index, int Nq, int index_per_batch,
                                  const vdx_attn_options* opt, void* stream);

/* Words per query block of a block mask for this grid (ceil(ceil(N/128)/32)); 0 if invalid. */
int vdx_rope3d_block_mask_words(int T, int Hgrid, int Wgrid);

/* Host helper: fill `mask` (host memory, [n_qblocks][W] words) with the block mask of 3D
 * windowed attention (the windowed-attention primitive of the vidax page, §2 "3D RoPE, 3D
 * VAEs, and flash attention"), at block granularity: query block Qb selects key tile Kb when
 * some token of Qb and some token of Kb are within (wt, wh, ww) of each other on every grid
 * axis (|dt| <= wt, |dh| <= wh, |dw| <= ww).  Pass it with mask_per_head = 0. */
vdx_status vdx_window_block_mask(uint32_t* mask, int T, int Hgrid, int Wgrid, int wt, int wh,
                                 int ww);

/* fp32 path (CUDA cores, fp32 arithmetic throughout).  Same operation and rules; q, k, v,
 * out are float [B, N, H, d]; d must be 64 or 128. */
vdx_status vdx_rope3d_attn_f32(const float* q, const float* k, const float* v, float* out,
                               float* lse, int B, int H, int T, int Hgrid, int Wgrid, int d,
                               int sec_t, int sec_h, int sec_w, double theta, float scale,
                               void* stream);

/* ---- No-allocation variant.  The vidax page has no counterpart: this is a deployment aid
 * for callers that cannot allocate device memory at call time (a frozen memory pool, an
 * allocator-free embedding, a host that sizes every buffer up front).  Same operation,
 * arguments, layouts and K-prepass arithmetic as vdx_rope3d_attn, but the cos/sin table and
 * the rotated keys live in one fixed static device array of the library instead of memory
 * allocated on first use, and the call makes no cudaMalloc/cudaFree.
 *   Limit: B*N*H*d*2 <= VDX_NOALLOC_MAX_WORKSPACE_BYTES and T*sec_t/2 + Hgrid*sec_h/2 +
 *   Wgrid*sec_w/2 <= VDX_NOALLOC_MAX_TABLE_ENTRIES; larger problems return
 *   VDX_ERR_UNSUPPORTED.
 *   The array (about 64 MiB) is held on every GPU that loads the library until exit.
 *   Every call shares it and it keeps the last call's contents, so calls that may overlap on
 *   the GPU (unordered streams) race; order them or use vdx_rope3d_attn_ex with a workspace.
 *   The first call on each device looks up the array's device address (make it before any
 *   stream capture). */
#define VDX_NOALLOC_MAX_WORKSPACE_BYTES (64ull << 20)
#define VDX_NOALLOC_MAX_TABLE_ENTRIES 8192
vdx_status vdx_rope3d_attn_noalloc(const void* q, const void* k, const void* v, void* out,
                                   float* lse, int B, int H, int T, int Hgrid, int Wgrid, int d,
                                   int sec_t, int sec_h, int sec_w, double theta, float scale,
                                   void* stream);

/* Synchronise `stream`, then read and clear the device error word.  Returns VDX_OK,
 * VDX_ERR_TIMEOUT (a kernel gave up on a pipeline wait; the output of that call is
 * undefined), VDX_ERR_RANGE (a rotated q/k value was clamped to the fp16 range; the output
 * is inexact), VDX_ERR_ARG (a q_index entry was out of range; its row was skipped) or
 * VDX_ERR_CUDA (an asynchronous CUDA error is pending). */
vdx_status vdx_sync_check(void* stream);

/* Message for the last non-OK status returned on this host thread ("" if none). */
const char* vdx_last_error(void);

/* Free every cached cos/sin table on every device.  Not to be called while work that uses
 * them is in flight. */
void vdx_shutdown(void);

/* Library version: major*10000 + minor*100 + patch. */
int vdx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VDX_H_ */
