// Greedy verification, in-place KV commit / rollback / truncate, and the
// bandwidth yardstick copy.
//
// verify ("Speculative Decoding", "Overview"): for request b with K_b drafts,
// r_j = argmax of target row j (j = 0..K_b, lowest id on ties); the accepted
// count is the longest prefix with draft j == r_j; the bonus token is r_a.
// The rows of the logits tensor are scanned as one flat range split evenly
// over the grid (a few CTAs per SM), so every CTA streams the same number of
// bytes whatever the requests' draft counts; a CTA's share spans one or more
// row segments, each scanned with 16-byte loads (eight in flight per thread),
// reduced warp- then block-wide to a (value, id) key and folded into its
// row's 64-bit key with atomicMax.  The last CTA to finish (arrival counter)
// turns the keys into r_j for every request, runs the prefix scans, writes
// accepted/bonus and resets keys and counter.
//
// KV edits ("How OpenVINO MTP Speculative Decoding Works Internally",
// "Stateful execution"; "Speculative Decoding", "Tree Drafting" step 4 and
// "Prefix Caching with Speculative Decoding"): one CTA per request zeroes the
// slots that leave the cache with 16-byte stores through the block table and
// then updates seq_len and pending.
#include <mutex>

#include "mtp_common.cuh"

namespace mtp {

// One CTA per SM: warp 0 streams the CTA's chunks of the flat logit range
// into a ring of shared-memory stages with one-dimensional bulk copies;
// warps 1..8 each own every 8th chunk (and, the stage count being the warp
// count, always the same stage) and reduce it from shared memory.
constexpr int kVerifyConsumers = 8;
constexpr int kVerifyThreads = 32 * (1 + kVerifyConsumers);
constexpr int kVerifyStages = kVerifyConsumers;
constexpr uint32_t kVerifyStageBytes = 24576;
constexpr uint32_t kVerifyMinChunk = 2048;
constexpr uint32_t kVerifyWaitLimit = 1u << 24;

template <typename T>
struct VerifyArgs {
  const T* logits;
  const int32_t* row_offsets;
  const int32_t* drafts;
  int drafts_stride;
  const int32_t* num_drafts;
  int32_t* accepted;
  int32_t* bonus;
  unsigned long long* keys;  // [num_rows], zero on entry, zero again on exit
  int* cnt;                  // [1], zero on entry and on exit
  int* err;
  int V, max_k, B, num_rows;
  uint32_t chunk;            // bytes per chunk (multiple of 16, <= kVerifyStageBytes)
};

template <typename T> struct VecOps;
template <> struct VecOps<uint16_t> {
  __device__ static __forceinline__ uint32_t max2(uint32_t x, uint32_t y) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
    return r;
  }
  // maximum of the eight values (NaN entries are passed over by max.bf16x2;
  // NaN only if all eight are NaN)
  __device__ static __forceinline__ float vmax(const uint4& u) {
    const uint32_t m = max2(max2(u.x, u.y), max2(u.z, u.w));
    return fmaxf(bf16_lo(m), bf16_hi(m));
  }
  // lowest position in the vector holding a value equal to m (-0 == +0)
  __device__ static __forceinline__ int find(const uint4& u, float m) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    int at = -1;
#pragma unroll
    for (int i = 3; i >= 0; --i) {
      if (bf16_hi(w[i]) == m) at = 2 * i + 1;
      if (bf16_lo(w[i]) == m) at = 2 * i;
    }
    return at;
  }
};
template <> struct VecOps<float> {
  __device__ static __forceinline__ float vmax(const uint4& u) {
    return fmaxf(fmaxf(__uint_as_float(u.x), __uint_as_float(u.y)), fmaxf(__uint_as_float(u.z), __uint_as_float(u.w)));
  }
  __device__ static __forceinline__ int find(const uint4& u, float m) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    int at = -1;
#pragma unroll
    for (int i = 3; i >= 0; --i)
      if (__uint_as_float(w[i]) == m) at = i;
    return at;
  }
};

// (value, lowest id) key of the row segment seg[0, len) held in shared
// memory, whose first element is column col0 of its row.  Warp-collective;
// every lane returns the warp's key (0 when every entry is NaN).  Scalar head
// up to 16-byte alignment, 16-byte vector body, scalar tail.  Each lane keeps
// its running maximum and the first vector where it appeared (lanes visit
// their vectors in increasing order and move only on a strictly larger
// value); after the body, the lanes holding the warp's maximum look up its
// first position in that vector.
template <typename T>
__device__ __forceinline__ unsigned long long segment_key(const T* seg, int len, int col0, int lane) {
  using Ops = VecOps<T>;
  constexpr int VPE = Elem<T>::kPerVec;
  unsigned long long key = 0ull;
  const int mis = (int)((smem_addr(seg) & 15u) / sizeof(T));
  const int head = mis ? min(len, VPE - mis) : 0;
  if (lane < head) {
    const float x = Elem<T>::loads(seg + lane);
    if (x == x) key = argmax_key(x, (uint32_t)(col0 + lane));
  }
  const T* body = seg + head;
  const int nvec = (len - head) / VPE;
  float bv = -INFINITY;
  int bat = -1;
#pragma unroll 4
  for (int v = lane; v < nvec; v += 32) {
    const uint4 u = *reinterpret_cast<const uint4*>(body + (size_t)v * VPE);
    const float m = Ops::vmax(u);
    if (m > bv || (bat < 0 && m == m)) {
      bv = m;
      bat = v;
    }
  }
  const int tail0 = head + nvec * VPE;
  if (tail0 + lane < len) {
    const float x = Elem<T>::loads(seg + tail0 + lane);
    if (x == x) key = umax64(key, argmax_key(x, (uint32_t)(col0 + tail0 + lane)));
  }
  const float wm = warp_max(bv);
  if (bat >= 0 && bv == wm) {
    const int f = Ops::find(*reinterpret_cast<const uint4*>(body + (size_t)bat * VPE), bv);
    if (f >= 0) key = umax64(key, argmax_key(bv, (uint32_t)(col0 + head + bat * VPE + f)));
  }
  return warp_max_u64(key);
}

__device__ __forceinline__ void verify_cons_bar() {
  asm volatile("bar.sync 1, %0;" ::"r"(32 * kVerifyConsumers) : "memory");
}

constexpr int kWalkChunk = 9;  // K_b <= 8 in one round trip

template <typename T>
__global__ void __launch_bounds__(kVerifyThreads, 1) verify_kernel(const VerifyArgs<T> a) {
  extern __shared__ __align__(128) unsigned char vsm[];
  __shared__ __align__(8) uint64_t full_bar[kVerifyStages], empty_bar[kVerifyStages];
  __shared__ int am_last;
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The flat range [0, num_rows * V) of elements: its 16-byte aligned body
  // is cut into chunks of a.chunk bytes; the few elements before and after
  // the body are read directly by one warp.
  const long long n_elem = (long long)a.num_rows * a.V;
  const uintptr_t base = (uintptr_t)a.logits;
  const uintptr_t lo = (base + 15) & ~(uintptr_t)15;
  const uintptr_t hi = (base + (uintptr_t)n_elem * sizeof(T)) & ~(uintptr_t)15;
  const bool has_body = hi > lo;
  const long long body_bytes = has_body ? (long long)(hi - lo) : 0;
  const long long head_elems = has_body ? (long long)((lo - base) / sizeof(T)) : n_elem;
  const long long tail_elem0 = has_body ? (long long)((hi - base) / sizeof(T)) : n_elem;
  const long long nch = (body_bytes + a.chunk - 1) / a.chunk;
  const long long c0 = (long long)blockIdx.x * nch / gridDim.x;
  const int n = (int)((long long)(blockIdx.x + 1) * nch / gridDim.x - c0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kVerifyStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    // the logits may come from the kernel just before this one
    pdl_wait();
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();  // each logit is read once
      for (int it = 0; it < n; ++it) {
        const int s = it % kVerifyStages;
        if (!mbar_wait_bounded(&empty_bar[s], (uint32_t)(((it / kVerifyStages) & 1) ^ 1), kVerifyWaitLimit)) {
          set_error(a.err, MTP_ERR_TIMEOUT);
          break;
        }
        const long long off = (c0 + it) * (long long)a.chunk;
        const uint32_t bytes = (uint32_t)min((long long)a.chunk, body_bytes - off);
        mbar_expect_tx(&full_bar[s], bytes);
        bulk_g2s_hint(vsm + (size_t)s * kVerifyStageBytes, (const void*)(lo + off), bytes, &full_bar[s], pol);
      }
    }
    return;
  }

  pdl_wait();
  const int ct = threadIdx.x - 32;   // 0 .. 255
  // request metadata for the accept walk, in case this CTA is the last
  int pk = 0, pr0 = 0, pr1 = 0;
  if (ct < a.B) {
    pk = a.num_drafts[ct];
    pr0 = a.row_offsets[ct];
    pr1 = a.row_offsets[ct + 1];
  }
  // elements outside the aligned body (fewer than 16 bytes at each end)
  if (blockIdx.x == 0 && warp == 1) {
    const long long n_out = head_elems + (n_elem - tail_elem0);
    for (long long i = lane; i < n_out; i += 32) {
      const long long e = i < head_elems ? i : tail_elem0 + (i - head_elems);
      const float x = Elem<T>::load1(a.logits + e);
      const int r = (int)(e / a.V);
      if (x == x && MTP_IN_BOUNDS(a.err, r, a.num_rows))
        atomicMax(a.keys + r, argmax_key(x, (uint32_t)(e - (long long)r * a.V)));
    }
  }
  const int cw = warp - 1;
  bool timed_out = false;
  int it = cw;
  for (; it < n; it += kVerifyConsumers) {
    const int s = it % kVerifyStages;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full_bar[s], (uint32_t)((it / kVerifyStages) & 1),
                                                   kVerifyWaitLimit))) {
      timed_out = true;
      break;
    }
    const long long off = (c0 + it) * (long long)a.chunk;
    const long long cnt = min((long long)a.chunk, body_bytes - off) / (long long)sizeof(T);
    const long long e0 = head_elems + off / (long long)sizeof(T);
    const T* sp = reinterpret_cast<const T*>(vsm + (size_t)s * kVerifyStageBytes);
    for (long long e = e0; e < e0 + cnt;) {
      const int r = (int)(e / a.V);
      const long long r_end = min(e0 + cnt, (long long)(r + 1) * a.V);
      const unsigned long long key =
          segment_key<T>(sp + (e - e0), (int)(r_end - e), (int)(e - (long long)r * a.V), lane);
      if (lane == 0 && key && MTP_IN_BOUNDS(a.err, r, a.num_rows)) atomicMax(a.keys + r, key);
      e = r_end;
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty_bar[s])) : "memory");
  }
  if (timed_out) {
    if (lane == 0) set_error(a.err, MTP_ERR_TIMEOUT);
    // copies still in flight into this warp's stage get a bounded chance to land
    mbar_wait_bounded(&full_bar[it % kVerifyStages], (uint32_t)((it / kVerifyStages) & 1), kVerifyWaitLimit);
  }
  // Arrival: every lane fences its key updates, the consumer barrier
  // collects them, and a release-acquire add publishes the CTA's work; the
  // last CTA's reads come after its acquire (the barrier carries it to the
  // other consumer threads).
  __threadfence();
  verify_cons_bar();
  if (ct == 0) {
    int prev;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(a.cnt) : "memory");
    am_last = (prev == (int)gridDim.x - 1);
  }
  verify_cons_bar();
  if (!am_last) return;
  constexpr int kWalkThreads = 32 * kVerifyConsumers;
  for (int b = ct; b < a.B; b += kWalkThreads) {
    const int K_b = b < kWalkThreads ? pk : a.num_drafts[b];
    const int r0 = b < kWalkThreads ? pr0 : a.row_offsets[b];
    const int r1 = b < kWalkThreads ? pr1 : a.row_offsets[b + 1];
    const bool bad = K_b < 0 || K_b > a.max_k || K_b > a.drafts_stride || r1 - r0 != K_b + 1 || r0 < 0 ||
                     r0 + K_b + 1 > a.num_rows;
    if (bad) {
      MTP_STORE(a.err, a.accepted, b, a.B, -1);
      MTP_STORE(a.err, a.bonus, b, a.B, -1);
      set_error(a.err, MTP_ERR_DEVICE_ARGS);
      continue;
    }
    // Rows are read kWalkChunk at a time (independent loads): one round trip
    // to L2 per request for K_b < kWalkChunk.
    int acc = 0, bonus = -1;
    bool done = false;
    for (int j0 = 0; !done && j0 <= K_b; j0 += kWalkChunk) {
      int r[kWalkChunk], d[kWalkChunk];
#pragma unroll
      for (int q = 0; q < kWalkChunk; ++q) {
        const int jj = j0 + q;
        const unsigned long long k = jj <= K_b ? __ldcg(a.keys + r0 + jj) : 0ull;
        r[q] = k ? (int)key_index(k) : -1;
        d[q] = jj < K_b ? a.drafts[(size_t)b * a.drafts_stride + jj] : -1;
      }
#pragma unroll
      for (int q = 0; q < kWalkChunk; ++q) {
        const int jj = j0 + q;
        if (done || jj > K_b) continue;
        if (jj < K_b && d[q] == r[q]) {
          ++acc;
        } else {
          bonus = r[q];
          done = true;
        }
      }
    }
    MTP_STORE(a.err, a.accepted, b, a.B, acc);
    MTP_STORE(a.err, a.bonus, b, a.B, bonus);
  }
  verify_cons_bar();
  for (int r = ct; r < a.num_rows; r += kWalkThreads) a.keys[r] = 0ull;
  if (ct == 0) *a.cnt = 0;
}

// Chunk size and grid of the verify kernel for a flat range of `bytes`:
// about eight chunks per CTA (one per consumer warp) when the range is
// small, chunks of a whole stage when it is large; at most one CTA per SM.
static void verify_plan(int sms, long long bytes, uint32_t* chunk, int* grid) {
  long long c = (bytes + 8LL * sms - 1) / (8LL * sms);
  c = (c + 15) & ~15LL;
  if (c < (long long)kVerifyMinChunk) c = kVerifyMinChunk;
  if (c > (long long)kVerifyStageBytes) c = kVerifyStageBytes;
  const long long nch = (bytes + c - 1) / c;
  *chunk = (uint32_t)c;
  *grid = (int)(nch < 1 ? 1 : (nch < sms ? nch : sms));
}

constexpr size_t kVerifySmem = (size_t)kVerifyStages * kVerifyStageBytes;

// Launch of the verify kernel (shared by mtp_verify and the context-free
// variant): keys and cnt must be zero on entry, and the kernel's shared-
// memory limit raised to kVerifySmem on this device beforehand.
template <typename T>
static cudaError_t launch_verify_kernel(cudaStream_t s, int sms, VerifyArgs<T> a) {
  int grid = 1;
  verify_plan(sms, (long long)a.num_rows * a.V * (long long)sizeof(T), &a.chunk, &grid);
  return launch_pdl(verify_kernel<T>, dim3(grid), dim3(kVerifyThreads), kVerifySmem, s, a);
}

template <typename T>
struct KvEditArgs {
  T* k_pool;
  T* v_pool;
  const int32_t* block_table;
  int32_t* seq_len;
  int32_t* pending;
  const int32_t* arg;
  int* err;
  int mode, extra, n_kv, hd, bs, max_blocks, num_blocks;
};

template <typename T>
__global__ void __launch_bounds__(256) kv_edit_kernel(const KvEditArgs<T> a) {
  __shared__ int z0s, z1s, new_len, ok;
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    const int L = a.seq_len[b], P = a.pending[b];
    int z0 = 0, z1 = L + P, nl = L;
    bool good = L >= 0 && P >= 0;
    if (a.mode == KV_COMMIT || a.mode == KV_COMMIT_ACCEPTED || a.mode == KV_ROLLBACK) {
      int n = 0;
      if (a.mode == KV_COMMIT) {
        n = a.arg[b];
      } else if (a.mode == KV_COMMIT_ACCEPTED) {
        const int acc = a.arg[b];
        good = good && acc >= 0;
        n = min(acc + a.extra, P);
      }
      good = good && n >= 0 && n <= P;
      z0 = L + n;
      nl = L + n;
    } else {  // KV_TRUNCATE
      const int n = a.arg[b];
      good = good && n >= 0 && n <= L + P;
      z0 = n;
      nl = n;
    }
    if (!good) set_error(a.err, MTP_ERR_DEVICE_ARGS);
    ok = good;
    z0s = z0;
    z1s = z1;
    new_len = nl;
  }
  __syncthreads();
  if (!ok) return;
  const int z0 = z0s, z1 = z1s;
  const int vec_per_row = a.hd * (int)sizeof(T) / 16;
  const int per_slot = 2 * a.n_kv * vec_per_row;
  const long long total = (long long)(z1 - z0) * per_slot;
  for (long long idx = threadIdx.x; idx < total; idx += blockDim.x) {
    const int slot = z0 + (int)(idx / per_slot);
    int rem = (int)(idx % per_slot);
    const int which = rem / (a.n_kv * vec_per_row);  // 0: K, 1: V
    rem -= which * a.n_kv * vec_per_row;
    const int g = rem / vec_per_row, v = rem - g * vec_per_row;
    const int bi = slot / a.bs, off = slot - bi * a.bs;
    const int blk = (bi < a.max_blocks) ? a.block_table[(size_t)b * a.max_blocks + bi] : -1;
    if (blk < 0 || blk >= a.num_blocks) {
      set_error(a.err, MTP_ERR_CAPACITY);
      continue;
    }
    T* pool = which ? a.v_pool : a.k_pool;
    const long long e = (((long long)blk * a.n_kv + g) * a.bs + off) * a.hd + (long long)v * (16 / sizeof(T));
    if (!MTP_IN_BOUNDS(a.err, e + (16 / sizeof(T)) - 1, (long long)a.num_blocks * a.n_kv * a.bs * a.hd)) continue;
    *reinterpret_cast<uint4*>(pool + e) = make_uint4(0, 0, 0, 0);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    a.seq_len[b] = new_len;
    a.pending[b] = 0;
  }
}

cudaError_t launch_verify(mtp_ctx* ctx, cudaStream_t s, int B, const void* logits, int num_rows,
                          const int32_t* row_offsets,
                          const int32_t* drafts, int drafts_stride, const int32_t* num_drafts,
                          int32_t* accepted, int32_t* bonus) {
  const mtp_config& c = ctx->cfg;
  if (num_rows > c.max_batch * (c.max_k + 1)) return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem(c.dtype == MTP_DTYPE_BF16 ? (const void*)verify_kernel<uint16_t>
                                                         : (const void*)verify_kernel<float>, kVerifySmem);
  if (e != cudaSuccess) return e;
  prof_before(ctx, MTP_KERNEL_VERIFY, s);
  if (c.dtype == MTP_DTYPE_BF16) {
    VerifyArgs<uint16_t> a{(const uint16_t*)logits, row_offsets, drafts, drafts_stride, num_drafts, accepted, bonus,
                           ctx->ver_keys, ctx->ver_cnt, ctx->err, c.vocab, c.max_k, B, num_rows, 0u};
    e = launch_verify_kernel(s, ctx->num_sms, a);
  } else {
    VerifyArgs<float> a{(const float*)logits, row_offsets, drafts, drafts_stride, num_drafts, accepted, bonus,
                        ctx->ver_keys, ctx->ver_cnt, ctx->err, c.vocab, c.max_k, B, num_rows, 0u};
    e = launch_verify_kernel(s, ctx->num_sms, a);
  }
  prof_after(ctx, MTP_KERNEL_VERIFY, s);
  ctx->launches++;
  return e;
}

cudaError_t launch_kv_edit(mtp_ctx* ctx, cudaStream_t s, int B, const mtp_kv* kv, int mode, const int32_t* arg,
                           int extra) {
  const mtp_config& c = ctx->cfg;
  cudaError_t e;
  prof_before(ctx, MTP_KERNEL_KV_EDIT, s);
  if (c.dtype == MTP_DTYPE_BF16) {
    KvEditArgs<uint16_t> a{(uint16_t*)kv->k_pool, (uint16_t*)kv->v_pool, kv->block_table, kv->seq_len, kv->pending,
                           arg, ctx->err, mode, extra, c.n_kv_heads, c.head_dim, c.block_size, kv->max_blocks,
                           kv->num_blocks};
    e = launch_pdl(kv_edit_kernel<uint16_t>, dim3(B), dim3(256), 0, s, a);
  } else {
    KvEditArgs<float> a{(float*)kv->k_pool, (float*)kv->v_pool, kv->block_table, kv->seq_len, kv->pending,
                        arg, ctx->err, mode, extra, c.n_kv_heads, c.head_dim, c.block_size, kv->max_blocks,
                        kv->num_blocks};
    e = launch_pdl(kv_edit_kernel<float>, dim3(B), dim3(256), 0, s, a);
  }
  prof_after(ctx, MTP_KERNEL_KV_EDIT, s);
  ctx->launches++;
  return e;
}

// ------------------------------------------------------------ stream copy
__global__ void __launch_bounds__(256) stream_copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                          size_t n) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a0 = ld_stream(src + i), a1 = ld_stream(src + i + stride);
    const uint4 a2 = ld_stream(src + i + 2 * stride), a3 = ld_stream(src + i + 3 * stride);
    dst[i] = a0;
    dst[i + stride] = a1;
    dst[i + 2 * stride] = a2;
    dst[i + 3 * stride] = a3;
  }
  for (; i < n; i += stride) dst[i] = ld_stream(src + i);
}

cudaError_t launch_stream_copy(cudaStream_t s, void* dst, const void* src, size_t bytes, int num_sms) {
  const size_t n = bytes / 16;
  stream_copy_kernel<<<4 * num_sms, 256, 0, s>>>((uint4*)dst, (const uint4*)src, n);
  return cudaGetLastError();
}

// ------------------------------------------------------------ stream read
// Read-only yardstick: the bytes are streamed once into a ring of shared-
// memory stages with one-dimensional bulk copies (the same mechanism as the
// streamed projections and verify), one CTA per SM, a contiguous share per
// CTA, and nothing is computed; its duration is the floor of a kernel that
// only has to read those bytes.
constexpr int kReadStages = 8;
constexpr uint32_t kReadChunk = 16384;
constexpr uint32_t kReadWaitLimit = 1u << 24;

__global__ void __launch_bounds__(64, 1) stream_read_kernel(const unsigned char* __restrict__ src, size_t bytes,
                                                            int* err) {
  extern __shared__ __align__(128) unsigned char rsm[];
  __shared__ __align__(8) uint64_t full_bar[kReadStages], empty_bar[kReadStages];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long nch = (long long)((bytes + kReadChunk - 1) / kReadChunk);
  const long long c0 = (long long)blockIdx.x * nch / gridDim.x;
  const int n = (int)((long long)(blockIdx.x + 1) * nch / gridDim.x - c0);
  if (threadIdx.x == 0) {
    for (int st = 0; st < kReadStages; ++st) {
      mbar_init(&full_bar[st], 1);
      mbar_init(&empty_bar[st], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (lane != 0) return;
  if (warp == 0) {
    const uint64_t pol = l2_evict_first_policy();
    for (int it = 0; it < n; ++it) {
      const int st = it % kReadStages;
      if (!mbar_wait_bounded(&empty_bar[st], (uint32_t)(((it / kReadStages) & 1) ^ 1), kReadWaitLimit)) {
        if (err) set_error(err, MTP_ERR_TIMEOUT);
        return;
      }
      const size_t off = (size_t)(c0 + it) * kReadChunk;
      const uint32_t nb = (uint32_t)(bytes - off < kReadChunk ? bytes - off : kReadChunk);
      mbar_expect_tx(&full_bar[st], nb);
      bulk_g2s_hint(rsm + (size_t)st * kReadChunk, src + off, nb, &full_bar[st], pol);
    }
  } else {
    for (int it = 0; it < n; ++it) {
      const int st = it % kReadStages;
      if (!mbar_wait_bounded(&full_bar[st], (uint32_t)((it / kReadStages) & 1), kReadWaitLimit)) {
        if (err) set_error(err, MTP_ERR_TIMEOUT);
        // a copy still in flight gets a bounded chance to land
        mbar_wait_bounded(&full_bar[st], (uint32_t)((it / kReadStages) & 1), kReadWaitLimit);
        return;
      }
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty_bar[st])) : "memory");
    }
  }
}

cudaError_t launch_stream_read(cudaStream_t s, const void* src, size_t bytes, int num_sms, int* err) {
  const size_t smem = (size_t)kReadStages * kReadChunk;
  cudaError_t e = ensure_smem((const void*)stream_read_kernel, smem);
  if (e != cudaSuccess) return e;
  const long long nch = (long long)((bytes + kReadChunk - 1) / kReadChunk);
  const int grid = (int)(nch < num_sms ? nch : num_sms);
  stream_read_kernel<<<grid, 64, smem, s>>>((const unsigned char*)src, bytes, err);
  return cudaGetLastError();
}

}  // namespace mtp

// ------------------------------------------- allocation-free verification
//
// mtp_verify needs a context, and mtp_init allocates the context's workspace
// with cudaMalloc.  Some callers cannot allocate device memory at the point
// where they verify: a serving loop whose device memory is all owned by a
// fixed plan or by another framework's pool, or a loop on a latency budget
// where cudaMalloc's implicit device-wide synchronisation would stall every
// other stream.  mtp_verify_noalloc runs the same verify kernel with its
// scratch (argmax keys and the arrival counter) in the array below, which is part
// of the library's device image: it is created when the library's code is
// loaded on a GPU and stays resident there until the process exits.
namespace mtp {

constexpr int kNoAllocMaxKeys = 65536;   // B * (max_k + 1) rows
constexpr int kNoAllocMaxBatch = 4096;   // B
constexpr int kNoAllocMaxDevices = 64;

struct NoAllocScratch {
  unsigned long long keys[kNoAllocMaxKeys];
  int cnt[1];
  int err;
};

static __device__ __align__(256) NoAllocScratch g_noalloc_scratch;

static NoAllocScratch* g_noalloc_ptr[kNoAllocMaxDevices];
static int g_noalloc_sms[kNoAllocMaxDevices];
static std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device, looked up once
// per device (host code may not use the symbol itself as a device pointer).
static cudaError_t noalloc_setup(int dev, NoAllocScratch** out, int* sms) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // the verify kernel's shared-memory limit, once per device
    e = cudaFuncSetAttribute((const void*)verify_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kVerifySmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute((const void*)verify_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kVerifySmem);
    if (e != cudaSuccess) return e;
    g_noalloc_sms[dev] = n;
    g_noalloc_ptr[dev] = (NoAllocScratch*)p;
  }
  *out = g_noalloc_ptr[dev];
  *sms = g_noalloc_sms[dev];
  return cudaSuccess;
}

}  // namespace mtp

extern "C" mtp_status mtp_verify_noalloc(void* stream, int B, int vocab, int dtype, int max_k,
                                         const void* target_logits, int num_rows, const int32_t* row_offsets,
                                         const int32_t* drafts, int drafts_stride, const int32_t* num_drafts,
                                         int32_t* accepted, int32_t* bonus) {
  using namespace mtp;
  if (B < 1 || B > kNoAllocMaxBatch || max_k < 0 || max_k > 100 || (long long)B * (max_k + 1) > kNoAllocMaxKeys ||
      num_rows > kNoAllocMaxKeys)
    return MTP_ERR_INVALID;
  if (vocab < 1 || (dtype != MTP_DTYPE_F32 && dtype != MTP_DTYPE_BF16) || num_rows < 1 || drafts_stride < 1)
    return MTP_ERR_INVALID;
  if (!target_logits || !row_offsets || !drafts || !num_drafts || !accepted || !bonus) return MTP_ERR_INVALID;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return MTP_ERR_CUDA;
  NoAllocScratch* sc = nullptr;
  int sms = 0;
  if (noalloc_setup(dev, &sc, &sms) != cudaSuccess) {
    cudaGetLastError();
    return MTP_ERR_CUDA;
  }
  cudaStream_t s = (cudaStream_t)stream;
  // The array keeps whatever the previous call left: clear the part this
  // call counts on.
  const size_t key_bytes = (size_t)num_rows * sizeof(unsigned long long);
  if (cudaMemsetAsync(sc->keys, 0, key_bytes, s) != cudaSuccess ||
      cudaMemsetAsync(sc->cnt, 0, sizeof(int), s) != cudaSuccess ||
      cudaMemsetAsync(&sc->err, 0, sizeof(int), s) != cudaSuccess) {
    cudaGetLastError();
    return MTP_ERR_CUDA;
  }
  cudaError_t e;
  if (dtype == MTP_DTYPE_BF16) {
    VerifyArgs<uint16_t> a{(const uint16_t*)target_logits, row_offsets, drafts, drafts_stride, num_drafts, accepted,
                           bonus, sc->keys, sc->cnt, &sc->err, vocab, max_k, B, num_rows, 0u};
    e = launch_verify_kernel(s, sms, a);
  } else {
    VerifyArgs<float> a{(const float*)target_logits, row_offsets, drafts, drafts_stride, num_drafts, accepted, bonus,
                        sc->keys, sc->cnt, &sc->err, vocab, max_k, B, num_rows, 0u};
    e = launch_verify_kernel(s, sms, a);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}
