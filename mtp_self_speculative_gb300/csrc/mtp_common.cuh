// Shared device helpers and the context layout of the MTP draft/verify
// library.  sm_103a only.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/mtp.h"

#ifndef __CUDA_ARCH__
#define MTP_HOST_ONLY 1
#endif

namespace mtp {

// ---------------------------------------------------------------- errors
// Device error word values match mtp_status.
__device__ __forceinline__ void set_error(int* err, int code) {
  atomicCAS(err, 0, code);
}

// Bounds-checked builds (-DMTP_CHECKED): MTP_IN_BOUNDS(err, i, n) is false,
// and records MTP_ERR_BOUNDS, when index i lies outside [0, n) of the
// buffer a store is about to write; callers skip the store then.  In other
// builds it is the constant true and costs nothing.
#ifdef MTP_CHECKED
__device__ __forceinline__ bool in_bounds_checked(int* err, long long i, long long n) {
  if (i >= 0 && i < n) return true;
  set_error(err, MTP_ERR_BOUNDS);
  return false;
}
#define MTP_IN_BOUNDS(err, i, n) ::mtp::in_bounds_checked((err), (long long)(i), (long long)(n))
#else
#define MTP_IN_BOUNDS(err, i, n) true
#endif
// ptr[i] = val, unless a bounds-checked build finds i outside [0, n).
#define MTP_STORE(err, ptr, i, n, val)                       \
  do {                                                       \
    const long long mtp_si_ = (long long)(i);                \
    if (MTP_IN_BOUNDS((err), mtp_si_, (n))) (ptr)[mtp_si_] = (val); \
  } while (0)

// ------------------------------------------------------- number formats

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int kPerVec = 4;  // elements per 16-byte vector
  __device__ static __forceinline__ float load1(const float* p) { return __ldg(p); }
  __device__ static __forceinline__ float loads(const float* p) { return *p; }  // any state space
  __device__ static __forceinline__ void store1(float* p, float v) { *p = v; }
};
template <> struct Elem<uint16_t> {
  static constexpr int kPerVec = 8;
  __device__ static __forceinline__ float load1(const uint16_t* p) {
    return __uint_as_float(((uint32_t)__ldg(p)) << 16);
  }
  __device__ static __forceinline__ float loads(const uint16_t* p) { return __uint_as_float(((uint32_t)*p) << 16); }
  __device__ static __forceinline__ void store1(uint16_t* p, float v) { *p = f32_to_bf16_rne(v); }
};

// 16-byte streaming load that bypasses L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Dot product of one 16-byte weight vector with the matching activations.
template <typename T>
__device__ __forceinline__ float dot_vec(const uint4& w, const float* x);

template <>
__device__ __forceinline__ float dot_vec<uint16_t>(const uint4& w, const float* x) {
  const float4 a = *reinterpret_cast<const float4*>(x);
  const float4 b = *reinterpret_cast<const float4*>(x + 4);
  float s = bf16_lo(w.x) * a.x;
  s = fmaf(bf16_hi(w.x), a.y, s);
  s = fmaf(bf16_lo(w.y), a.z, s);
  s = fmaf(bf16_hi(w.y), a.w, s);
  s = fmaf(bf16_lo(w.z), b.x, s);
  s = fmaf(bf16_hi(w.z), b.y, s);
  s = fmaf(bf16_lo(w.w), b.z, s);
  s = fmaf(bf16_hi(w.w), b.w, s);
  return s;
}

template <>
__device__ __forceinline__ float dot_vec<float>(const uint4& w, const float* x) {
  const float4 a = *reinterpret_cast<const float4*>(x);
  float s = __uint_as_float(w.x) * a.x;
  s = fmaf(__uint_as_float(w.y), a.y, s);
  s = fmaf(__uint_as_float(w.z), a.z, s);
  s = fmaf(__uint_as_float(w.w), a.w, s);
  return s;
}

// The GPU's global nanosecond timer.
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Orderable key for argmax with lowest-index tie break:
// (monotone float bits << 32) | (0xFFFFFFFF - index).  A larger key is a
// larger value, or an equal value at a smaller index.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
  if (v == 0.0f) v = 0.0f;  // -0 and +0 compare equal
  uint32_t b = __float_as_uint(v);
  uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t key_index(unsigned long long k) {
  return 0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull);
}
__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = umax64(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ------------------------------------------- programmatic dependent launch
// Each kernel lets its dependent start early (the dependent only prefetches
// weights before its own wait) and waits for its prerequisite grid before
// touching anything the previous kernel produced or still reads.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------ bulk copy + mbarrier
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false if the phase did not complete within `limit` polls.
// Non-blocking probe of a phase (producers that serve several queues).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// One-dimensional bulk (TMA) copy global -> shared, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// L2 policy for data read exactly once (streamed weights): evict first, so
// that the stream does not push out small data that is read again (norm
// weights, activations, the KV cache, block tables).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

}  // namespace mtp

// ------------------------------------------------------------ host context

struct mtp_ctx {
  mtp_config cfg;
  mtp_weights w;
  int has_weights;
  int device;
  int num_sms;
  int q_dim, kv_dim;
  int attn_target_ctas;
  int attn_max_splits;
  // workspace (one allocation)
  void* ws;
  size_t ws_bytes;
  float* hid;        // [maxB, H]   recursive hidden (decoder output)
  float* x;          // [maxB, H]   eh_proj output (residual stream)
  float* q;          // [maxB, q_dim] rotated queries
  float* attn;       // [maxB, q_dim] attention output
  float* h1;         // [maxB, H]   after attention residual
  float* act;        // [maxB, F]   silu(gate) * up
  float* attn_part;  // split-KV partials
  int* attn_cnt;     // [maxB, n_kv] arrival counters
  unsigned long long* lm_keys;  // [maxB] argmax keys
  int* lm_cnt;                  // [1]
  unsigned long long* ver_keys; // [maxB, max_k + 1]
  int* ver_cnt;                 // [1]
  int* err;                     // [1]
  int* req_bad;                 // [maxB] 1: pending was not 0 when the draft call began
  float2* rope;                 // [max_pos, head_dim / 2] (cos, sin)
  // tensor-core path (allocated when the shape allows it)
  void* tc_ws;
  int tc_min_batch;
  uint16_t* tc_xin_eh;          // [maxB, 2H] bf16 eh_proj input
  uint16_t* tc_xn;              // [maxB, H]  bf16 GEMM input y * w (RMS factor applied by the consumer)
  float* tc_ssq;                // [H / 128, maxB] per-tile sums of squares of y
  uint16_t* tc_attn;            // [maxB, q_dim] bf16 attention output
  uint16_t* tc_act;             // [maxB, F]  bf16 silu(g) * u
  // timing
  int prof_kernel;
  int prof_cap;
  int prof_n;
  cudaEvent_t* prof_ev;  // 2 * prof_cap
  long long launches;
  long long path_counts[MTP_PATH_COUNT];  // mtp_path_count
  // host-side caches (tensor maps need 64-byte aligned storage)
  void* tc_plan_cache;          // TcPlan[6][17], lazily allocated
  void* attn_map_cache;         // AttnMapCache, lazily allocated
  // small-batch projections: bit k set = kernel kind k streams its weights
  // through shared memory with bulk copies (else register streaming)
  int gemv_stream_mask;
  int gemv_budget_kb[6];         // shared memory per streamed-kernel CTA, per kind
  int lm_rows;                   // LM head of 2..4 requests on the tensor cores (0: streamed GEMV)
  int attn_force_bps;            // attention blocks per split (0: planned; tuning)
  int attn_cluster;              // tensor-core attention: splits combined in a thread-block cluster
  long long attn_cl_key;         // (capacity, G, clusters, split) of the cached cluster plan
  int attn_cl_fit, attn_cl_bps;  // ... its cluster size (0: none fits) and blocks per split
  int lm_balance;                // streamed LM head sizes each CTA's range by its SM's measured rate
  int lm_defer;                  // one request: the next eh_proj reduces the LM head's per-CTA keys
  int lm_defer_pending, lm_defer_grid;  // the last LM head launch deferred its argmax, over this many CTAs
  unsigned long long* lm_defer_tick;    // ... and left this claim counter to be zeroed
  unsigned long long* cta_keys;  // [num_sms] per-CTA argmax keys of a deferred LM head
  unsigned lm_seq;               // streamed LM head launches (picks the launch's claim counter)
  unsigned long long* lm_tick;   // [64] claim counters, one per launch in a ring
  float* lm_rate;                // [num_sms] per-SM streaming rates of the LM head
  int rows_proj;                 // short projections of 2..4 requests on the tensor cores (0: streamed GEMV)
  int rows_max_kc, rows_min_stages;  // their chunk plan: widest chunk (columns), fewest ring stages
  // persistent draft kernel (batches 1..p_max_batch; 0 = off)
  int p_max_batch;
  void* p_ws;
  float* p_rec;                  // [p_max_batch * n_kv, num_sms, G, 132] attention records
  int* p_seg_cnt;                // [p_max_batch * n_kv]
  unsigned long long* p_keys;    // [max_k, p_max_batch]
  unsigned long long* p_gbar;    // grid barrier: arrivals, completed barriers, abort flag (128 B apart)
  // quantized head (weight_format MTP_WEIGHTS_INT4_G64): owned copies
  int quantized;
  void* qw_buf;
  uint8_t* qw_tiles[6];          // per projection kind (and the LM head): fragment-ordered tiles
  int8_t* qw_q8;                 // INT8 embedding [V, H] (row gather for the next step's input)
  uint16_t* qw_s8;               // fp16 row scales [V]
  uint16_t* qw_s8_lm;            // LM-head row scales (== qw_s8 when tied)
  float qw_lm_sigma;             // power-of-two input scale of the LM head's fp16 operand
  int p_nslots[3];               // launch plan per batch width 1, 2, 4 (0 = not yet made)
  int p_warps[3];
  size_t p_smem[3];
};

namespace mtp {

// Launch helper: programmatic stream serialisation on every kernel.
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device);
// later calls with the same or a smaller size are free.
cudaError_t ensure_smem(const void* func, size_t bytes);

// Kernel timing hooks (host).
void prof_before(mtp_ctx* ctx, int kernel, cudaStream_t s);
void prof_after(mtp_ctx* ctx, int kernel, cudaStream_t s);

// Launchers implemented in the kernel translation units.
cudaError_t launch_draft_step(mtp_ctx* ctx, cudaStream_t s, int B, int k, int K, const void* hidden,
                              const void* embeds, const int32_t* positions, const mtp_kv* kv,
                              const int32_t* chain_ids, int32_t* draft_ids, float* logits, float* hidden_out);
cudaError_t launch_attention(mtp_ctx* ctx, cudaStream_t s, int B, int k, const mtp_kv* kv);
cudaError_t launch_draft_step_q(mtp_ctx* ctx, cudaStream_t s, int B, int k, int K, const void* hidden,
                                const void* embeds, const int32_t* positions, const mtp_kv* kv,
                                const int32_t* chain_ids, int32_t* draft_ids, float* logits, float* hidden_out);
cudaError_t launch_quant_int4(cudaStream_t s, const void* w, int rows, int cols, void* q, void* scales,
                              void* zeros);
cudaError_t launch_quant_int8(cudaStream_t s, const void* w, int rows, int cols, void* q, void* scales);
mtp_status quantize_head(mtp_ctx* ctx);
cudaError_t draft_one_step(mtp_ctx* ctx, cudaStream_t s, int B, int k, int K, const void* hidden, const void* embeds,
                           const int32_t* positions, const mtp_kv* kv, const int32_t* chain_ids, int32_t* draft_ids,
                           float* logits, float* hidden_out);
bool tc_supported(const mtp_ctx* ctx, int B);
bool persistent_supported(const mtp_ctx* ctx, int B);
cudaError_t launch_selftest_wait(mtp_ctx* ctx, cudaStream_t s, int which);
cudaError_t launch_draft_persistent(mtp_ctx* ctx, cudaStream_t s, int B, int K, const void* hidden,
                                    const void* embeds, const int32_t* positions, const mtp_kv* kv,
                                    const int32_t* chain_ids, int32_t* draft_ids, float* logits,
                                    float* hidden_out);
// Swizzled [16 x 64] tensor maps over the K and V pools (head_dim 128),
// cached in the context; false if they cannot be encoded.
bool attn_tensor_maps(mtp_ctx* ctx, const mtp_kv* kv, const CUtensorMap** km, const CUtensorMap** vm);
// 2-D bf16 tensor map over [rows, cols] (row-major) with a [box_rows, 64]
// box and 128-byte swizzle; false if the driver rejects it.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
cudaError_t launch_draft_step_tc(mtp_ctx* ctx, cudaStream_t s, int B, int k, int K, const void* hidden,
                                 const void* embeds, const int32_t* positions, const mtp_kv* kv,
                                 const int32_t* chain_ids, int32_t* draft_ids, float* logits, float* hidden_out);
cudaError_t launch_verify(mtp_ctx* ctx, cudaStream_t s, int B, const void* logits, int num_rows,
                          const int32_t* row_offsets,
                          const int32_t* drafts, int drafts_stride, const int32_t* num_drafts,
                          int32_t* accepted, int32_t* bonus);
cudaError_t launch_kv_edit(mtp_ctx* ctx, cudaStream_t s, int B, const mtp_kv* kv, int mode,
                           const int32_t* arg, int extra);
cudaError_t launch_stream_copy(cudaStream_t s, void* dst, const void* src, size_t bytes, int num_sms);
cudaError_t launch_stream_read(cudaStream_t s, const void* src, size_t bytes, int num_sms, int* err);

enum KvEditMode { KV_COMMIT = 0, KV_COMMIT_ACCEPTED = 1, KV_ROLLBACK = 2, KV_TRUNCATE = 3 };

}  // namespace mtp
