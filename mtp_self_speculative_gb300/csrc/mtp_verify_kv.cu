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

constexpr int kVerifyThreads = 256;

template <typename T>
struct VerifyArgs {
  const T* logits;
  const int32_t* row_offsets;
  const int32_t* drafts;
  int drafts_stride;
  const int32_t* num_drafts;
  int32_t* accepted;
  int32_t* bonus;
  unsigned long long* keys;  // [num_rows]
  int* cnt;                  // [1]
  int* err;
  int V, max_k, B, num_rows;
};

// Batch helpers of the vector scan.  A thread loads kVerifyBatch 16-byte
// vectors and takes their maximum with packed max instructions (about one
// instruction per two bf16 logits); it keeps only its running maximum and
// the vector where that maximum first appeared (the lowest vector of the
// batch holding it, looked up only when the running maximum moves).  The
// position inside the vector is found once per row segment: the lanes whose
// maximum equals their warp's take the first element equal to it in the
// vector they kept in registers.  Ids visited by a thread increase with
// q and within a vector, and the running maximum moves only on a strictly
// larger batch maximum, so that element is the thread's lowest id holding
// its maximum.  Vectors past the end are filled with -inf
// and never searched.  -0 equals +0 in every comparison; NaN logits are
// passed over (the packed max returns the other operand, a batch whose
// maximum is NaN is skipped, no search matches NaN), in the scalar head and
// tail as well.
template <typename T> struct VecOps;
template <> struct VecOps<uint16_t> {
  static constexpr uint32_t kFill = 0xFF80FF80u;  // -inf, -inf
  __device__ static __forceinline__ uint32_t max2(uint32_t x, uint32_t y) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
    return r;
  }
  __device__ static __forceinline__ uint32_t vmax(const uint4& u) { return max2(max2(u.x, u.y), max2(u.z, u.w)); }
  __device__ static __forceinline__ float finish(uint32_t m) { return fmaxf(bf16_lo(m), bf16_hi(m)); }
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
  static constexpr uint32_t kFill = 0xFF800000u;  // -inf
  __device__ static __forceinline__ uint32_t max2(uint32_t x, uint32_t y) {
    return __float_as_uint(fmaxf(__uint_as_float(x), __uint_as_float(y)));
  }
  __device__ static __forceinline__ uint32_t vmax(const uint4& u) { return max2(max2(u.x, u.y), max2(u.z, u.w)); }
  __device__ static __forceinline__ float finish(uint32_t m) { return __uint_as_float(m); }
  __device__ static __forceinline__ int find(const uint4& u, float m) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    int at = -1;
#pragma unroll
    for (int i = 3; i >= 0; --i)
      if (__uint_as_float(w[i]) == m) at = i;
    return at;
  }
};

constexpr int kVerifyBatch = 8;

// One thread's view of a row segment row[c0, c1): the (value, id) key of its
// scalar head and tail elements, and its running maximum over the vector
// body with the batch where that maximum first appeared.
template <typename T>
struct ScanState {
  const T* vbase;              // first 16-byte aligned element of the body
  int c;                       // its column
  int nvec;                    // vectors in the body
  float bv;
  int bat;                     // the vector where bv first appeared, -1 = none
  uint4 bu;                    // that vector's contents
  unsigned long long scalar;   // key of the head and tail elements
};

// Streams row[c0, c1): scalar head to 16-byte alignment, vector body with
// kVerifyBatch loads in flight per thread, scalar tail.
template <typename T>
__device__ __forceinline__ ScanState<T> scan_body(const T* row, int c0, int c1) {
  using Ops = VecOps<T>;
  constexpr int VPE = Elem<T>::kPerVec;
  constexpr int kStride = kVerifyThreads * kVerifyBatch;
  ScanState<T> st;
  st.scalar = 0ull;
  int c = c0;
  const int misalign = (int)(((uintptr_t)(row + c) & 15) / sizeof(T));
  const int head_end = misalign ? min(c1, c + (VPE - misalign)) : c;
  for (int i = c + threadIdx.x; i < head_end; i += kVerifyThreads) {
    const float x = Elem<T>::load1(row + i);
    if (x == x) st.scalar = umax64(st.scalar, argmax_key(x, (uint32_t)i));
  }
  c = head_end;
  st.c = c;
  st.nvec = max(0, (c1 - c) / VPE);
  st.vbase = row + c;
  st.bv = -INFINITY;
  st.bat = -1;
  st.bu = make_uint4(Ops::kFill, Ops::kFill, Ops::kFill, Ops::kFill);
  for (int v0 = threadIdx.x; v0 < st.nvec; v0 += kStride) {
    uint4 u[kVerifyBatch];
#pragma unroll
    for (int q = 0; q < kVerifyBatch; ++q) {
      const int v = v0 + q * kVerifyThreads;
      u[q] = v < st.nvec ? ld_stream(st.vbase + (size_t)v * VPE)
                         : make_uint4(Ops::kFill, Ops::kFill, Ops::kFill, Ops::kFill);
    }
    uint32_t vm[kVerifyBatch], m[kVerifyBatch];
#pragma unroll
    for (int q = 0; q < kVerifyBatch; ++q) m[q] = vm[q] = Ops::vmax(u[q]);
#pragma unroll
    for (int w = 1; w < kVerifyBatch; w *= 2)
#pragma unroll
      for (int q = 0; q + w < kVerifyBatch; q += 2 * w) m[q] = Ops::max2(m[q], m[q + w]);
    const float mf = Ops::finish(m[0]);
    if (mf > st.bv || (st.bat < 0 && mf == mf)) {
      // the lowest vector of the batch holding mf (filled vectors come last)
      int qi = 0;
      uint4 bu = u[0];
#pragma unroll
      for (int q = kVerifyBatch - 1; q >= 0; --q)
        if (Ops::finish(vm[q]) == mf) {
          qi = q;
          bu = u[q];
        }
      st.bv = mf;
      st.bat = v0 + qi * kVerifyThreads;
      st.bu = bu;
    }
  }
  for (int i = c + st.nvec * VPE + threadIdx.x; i < c1; i += kVerifyThreads) {
    const float x = Elem<T>::load1(row + i);
    if (x == x) st.scalar = umax64(st.scalar, argmax_key(x, (uint32_t)i));
  }
  return st;
}

// This thread's keys for up to two segments: the lanes holding their warp's
// maximum of a segment take the first element equal to it in the vector they
// kept.  Warp-collective; has_b is block-uniform.
template <typename T>
__device__ __forceinline__ void scan_locate2(const ScanState<T>& sa, const ScanState<T>& sb, bool has_b,
                                             unsigned long long& ka, unsigned long long& kb) {
  using Ops = VecOps<T>;
  constexpr int VPE = Elem<T>::kPerVec;
  float wa = sa.bv, wb = has_b ? sb.bv : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    wa = fmaxf(wa, __shfl_xor_sync(0xffffffffu, wa, o));
    wb = fmaxf(wb, __shfl_xor_sync(0xffffffffu, wb, o));
  }
  ka = sa.scalar;
  kb = has_b ? sb.scalar : 0ull;
  if (sa.bat >= 0 && sa.bat < sa.nvec && sa.bv == wa) {
    const int f = Ops::find(sa.bu, sa.bv);
    if (f >= 0) ka = umax64(ka, argmax_key(sa.bv, (uint32_t)(sa.c + sa.bat * VPE + f)));
  }
  if (has_b && sb.bat >= 0 && sb.bat < sb.nvec && sb.bv == wb) {
    const int f = Ops::find(sb.bu, sb.bv);
    if (f >= 0) kb = umax64(kb, argmax_key(sb.bv, (uint32_t)(sb.c + sb.bat * VPE + f)));
  }
}

// Block-wide maximum of two keys (all threads call; result valid in thread 0).
__device__ __forceinline__ void block_max2(unsigned long long& k0, unsigned long long& k1,
                                           unsigned long long (*red)[kVerifyThreads / 32]) {
  k0 = warp_max_u64(k0);
  k1 = warp_max_u64(k1);
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = k0;
    red[1][threadIdx.x >> 5] = k1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kVerifyThreads / 32; ++w) {
      k0 = umax64(k0, red[0][w]);
      k1 = umax64(k1, red[1][w]);
    }
  }
  __syncthreads();
}

constexpr int kWalkChunk = 9;  // K_b <= 8 in one round trip

template <typename T>
__global__ void __launch_bounds__(kVerifyThreads, 4) verify_kernel(const VerifyArgs<T> a) {
  __shared__ unsigned long long red[2][kVerifyThreads / 32];
  __shared__ int am_last;
  pdl_trigger();
  pdl_wait();
  // Request metadata for the accept walk, fetched while the scan runs in
  // case this CTA is the last (thread b holds request b, b < block size).
  int pk = 0, pr0 = 0, pr1 = 0;
  if (threadIdx.x < a.B) {
    pk = a.num_drafts[threadIdx.x];
    pr0 = a.row_offsets[threadIdx.x];
    pr1 = a.row_offsets[threadIdx.x + 1];
  }
  const long long total = (long long)a.num_rows * a.V;
  const long long per = (total + gridDim.x - 1) / gridDim.x;
  const long long e0 = (long long)blockIdx.x * per;
  const long long e1 = min(total, e0 + per);
  if (e0 < e1 && per <= a.V) {
    // The share lies in at most two rows: stream both parts back to back and
    // reduce once.
    const int rA = (int)(e0 / a.V);
    const int cA = (int)(e0 - (long long)rA * a.V);
    const int cA1 = (int)min((long long)a.V, (long long)cA + (e1 - e0));
    const int lenB = (int)((e1 - e0) - (cA1 - cA));
    const ScanState<T> sA = scan_body<T>(a.logits + (size_t)rA * a.V, cA, cA1);
    ScanState<T> sB = sA;
    if (lenB > 0) sB = scan_body<T>(a.logits + (size_t)(rA + 1) * a.V, 0, lenB);
    unsigned long long kA, kB;
    scan_locate2<T>(sA, sB, lenB > 0, kA, kB);
    block_max2(kA, kB, red);
    if (threadIdx.x == 0) {
      if (kA) atomicMax(a.keys + rA, kA);
      if (kB) atomicMax(a.keys + rA + 1, kB);
    }
  } else {
    for (long long e = e0; e < e1;) {
      const int r = (int)(e / a.V);
      const int c0 = (int)(e - (long long)r * a.V);
      const int c1 = (int)min((long long)a.V, (long long)c0 + (e1 - e));
      const ScanState<T> st = scan_body<T>(a.logits + (size_t)r * a.V, c0, c1);
      unsigned long long k, unused;
      scan_locate2<T>(st, st, false, k, unused);
      block_max2(k, unused, red);
      if (threadIdx.x == 0 && k) atomicMax(a.keys + r, k);
      e += c1 - c0;
    }
  }
  // Arrival: a release-acquire add orders this CTA's key updates (all made
  // by thread 0) before it, and the last CTA's reads after it (the barrier
  // carries the acquire to the other threads).
  if (threadIdx.x == 0) {
    int prev;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(a.cnt) : "memory");
    am_last = (prev == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!am_last) return;
  for (int b = threadIdx.x; b < a.B; b += kVerifyThreads) {
    const int K_b = b < kVerifyThreads ? pk : a.num_drafts[b];
    const int r0 = b < kVerifyThreads ? pr0 : a.row_offsets[b];
    const int r1 = b < kVerifyThreads ? pr1 : a.row_offsets[b + 1];
    const bool bad = K_b < 0 || K_b > a.max_k || K_b > a.drafts_stride || r1 - r0 != K_b + 1 || r0 < 0 ||
                     r0 + K_b + 1 > a.num_rows;
    if (bad) {
      a.accepted[b] = -1;
      a.bonus[b] = -1;
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
        r[q] = jj <= K_b ? (int)key_index(__ldcg(a.keys + r0 + jj)) : -1;
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
    a.accepted[b] = acc;
    a.bonus[b] = bonus;
  }
  __syncthreads();
  for (int r = threadIdx.x; r < a.num_rows; r += kVerifyThreads) a.keys[r] = 0ull;
  if (threadIdx.x == 0) *a.cnt = 0;
}

// Grid of the verify kernel: a few CTAs per SM, at least 16K elements each.
static int verify_grid(int sms, int num_rows, int V) {
  const long long total = (long long)num_rows * V;
  long long g = (total + 16383) / 16384;
  if (g > 4LL * sms) g = 4LL * sms;
  return g < 1 ? 1 : (int)g;
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
    uint4* dst = reinterpret_cast<uint4*>(pool + (((size_t)blk * a.n_kv + g) * a.bs + off) * a.hd) + v;
    *dst = make_uint4(0, 0, 0, 0);
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
  const dim3 grid(verify_grid(ctx->num_sms, num_rows, c.vocab));
  cudaError_t e;
  prof_before(ctx, MTP_KERNEL_VERIFY, s);
  if (c.dtype == MTP_DTYPE_BF16) {
    VerifyArgs<uint16_t> a{(const uint16_t*)logits, row_offsets, drafts, drafts_stride, num_drafts, accepted, bonus,
                           ctx->ver_keys, ctx->ver_cnt, ctx->err, c.vocab, c.max_k, B, num_rows};
    e = launch_pdl(verify_kernel<uint16_t>, grid, dim3(kVerifyThreads), 0, s, a);
  } else {
    VerifyArgs<float> a{(const float*)logits, row_offsets, drafts, drafts_stride, num_drafts, accepted, bonus,
                        ctx->ver_keys, ctx->ver_cnt, ctx->err, c.vocab, c.max_k, B, num_rows};
    e = launch_pdl(verify_kernel<float>, grid, dim3(kVerifyThreads), 0, s, a);
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
  const dim3 grid(verify_grid(sms, num_rows, vocab));
  cudaError_t e;
  if (dtype == MTP_DTYPE_BF16) {
    VerifyArgs<uint16_t> a{(const uint16_t*)target_logits, row_offsets, drafts, drafts_stride, num_drafts, accepted,
                           bonus, sc->keys, sc->cnt, &sc->err, vocab, max_k, B, num_rows};
    e = launch_pdl(verify_kernel<uint16_t>, grid, dim3(kVerifyThreads), 0, s, a);
  } else {
    VerifyArgs<float> a{(const float*)target_logits, row_offsets, drafts, drafts_stride, num_drafts, accepted, bonus,
                        sc->keys, sc->cnt, &sc->err, vocab, max_k, B, num_rows};
    e = launch_pdl(verify_kernel<float>, grid, dim3(kVerifyThreads), 0, s, a);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}
