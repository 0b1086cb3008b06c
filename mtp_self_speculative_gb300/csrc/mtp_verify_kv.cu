// Greedy verification, in-place KV commit / rollback / truncate, and the
// bandwidth yardstick copy.
//
// verify ("Speculative Decoding", "Overview"): for request b with K_b drafts,
// r_j = argmax of target row j (j = 0..K_b, lowest id on ties); the accepted
// count is the longest prefix with draft j == r_j; the bonus token is r_a.
// Grid (vocab splits, max_k + 1, B): each CTA scans one slice of one row with
// 16-byte loads, reduces (value, id) keys warp- then block-wide, and folds
// them into the row's 64-bit key with atomicMax.  The last CTA of a request
// (arrival counter) turns the keys into r_j, runs the prefix scan, writes
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
  unsigned long long* keys;  // [B, max_k + 1]
  int* cnt;                  // [B]
  int* err;
  int V, max_k, splits, num_rows;
};

// Running (value, index) maximum over one 16-byte vector of consecutive ids
// starting at base.  Each thread visits increasing ids, so a strict
// comparison keeps the lowest id among equal values (-0 equals +0).
template <typename T>
__device__ __forceinline__ void scan_vec(const uint4& u, int base, float& bv, int& bi);
template <>
__device__ __forceinline__ void scan_vec<uint16_t>(const uint4& u, int base, float& bv, int& bi) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = bf16_lo(w[i]), hi = bf16_hi(w[i]);
    if (lo > bv || bi < 0) { bv = lo; bi = base + 2 * i; }
    if (hi > bv) { bv = hi; bi = base + 2 * i + 1; }
  }
}
template <>
__device__ __forceinline__ void scan_vec<float>(const uint4& u, int base, float& bv, int& bi) {
  const float f[4] = {__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w)};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (f[i] > bv || bi < 0) { bv = f[i]; bi = base + i; }
}

template <typename T>
__global__ void __launch_bounds__(kVerifyThreads) verify_kernel(const VerifyArgs<T> a) {
  __shared__ unsigned long long red[kVerifyThreads / 32];
  __shared__ int am_last;
  pdl_trigger();
  pdl_wait();
  const int s = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int K_b = a.num_drafts[b];
  const int r0 = a.row_offsets[b];
  const bool bad = K_b < 0 || K_b > a.max_k || K_b > a.drafts_stride || a.row_offsets[b + 1] - r0 != K_b + 1 ||
                   r0 < 0 || r0 + K_b + 1 > a.num_rows;
  if (bad) {
    if (s == 0 && j == 0 && threadIdx.x == 0) {
      a.accepted[b] = -1;
      a.bonus[b] = -1;
      set_error(a.err, MTP_ERR_DEVICE_ARGS);
    }
    return;
  }
  if (j > K_b) return;

  // Slice [c0, c1) of row r0 + j.
  const int per = (a.V + a.splits - 1) / a.splits;
  const int c0 = s * per, c1 = min(a.V, c0 + per);
  const T* row = a.logits + (size_t)(r0 + j) * a.V;
  unsigned long long best = 0ull;
  if (c0 < c1) {
    constexpr int VPE = Elem<T>::kPerVec;
    constexpr int kBatch = 8;  // 16-byte loads in flight per thread
    // scalar head until 16-byte alignment, vector body, scalar tail; each
    // part keeps a running (value, index) maximum, folded into the key once
    int c = c0;
    const int misalign = (int)(((uintptr_t)(row + c) & 15) / sizeof(T));
    int head_end = misalign ? min(c1, c + (VPE - misalign)) : c;
    for (int i = c + threadIdx.x; i < head_end; i += kVerifyThreads)
      best = umax64(best, argmax_key(Elem<T>::load1(row + i), (uint32_t)i));
    c = head_end;
    const int nvec = (c1 - c) / VPE;
    const T* vbase = row + c;
    float bv = -INFINITY;
    int bi = -1;
    for (int v0 = threadIdx.x; v0 < nvec; v0 += kVerifyThreads * kBatch) {
      uint4 u[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int v = v0 + q * kVerifyThreads;
        u[q] = v < nvec ? ld_stream(vbase + (size_t)v * VPE) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int v = v0 + q * kVerifyThreads;
        if (v < nvec) scan_vec<T>(u[q], c + v * VPE, bv, bi);
      }
    }
    if (bi >= 0) best = umax64(best, argmax_key(bv, (uint32_t)bi));
    for (int i = c + nvec * VPE + threadIdx.x; i < c1; i += kVerifyThreads)
      best = umax64(best, argmax_key(Elem<T>::load1(row + i), (uint32_t)i));
  }
  best = warp_max_u64(best);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long m = 0ull;
    for (int w = 0; w < kVerifyThreads / 32; ++w) m = umax64(m, red[w]);
    if (m) atomicMax(a.keys + (size_t)b * (a.max_k + 1) + j, m);
    __threadfence();
    const int total = (K_b + 1) * a.splits;
    am_last = (atomicAdd(a.cnt + b, 1) == total - 1);
  }
  __syncthreads();
  if (!am_last || threadIdx.x != 0) return;
  __threadfence();
  unsigned long long* kb = a.keys + (size_t)b * (a.max_k + 1);
  int acc = 0;
  bool matching = true;
  int bonus = -1;
  for (int jj = 0; jj <= K_b; ++jj) {
    const int r = (int)key_index(atomicExch(kb + jj, 0ull));
    if (matching) {
      if (jj < K_b && a.drafts[(size_t)b * a.drafts_stride + jj] == r) {
        ++acc;
      } else {
        bonus = r;
        matching = false;
      }
    }
  }
  a.accepted[b] = acc;
  a.bonus[b] = bonus;
  atomicExch(a.cnt + b, 0);
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
  const int rows = B * (c.max_k + 1);
  int splits = (4 * ctx->num_sms + rows - 1) / rows;
  const int max_splits = (c.vocab + 2047) / 2048;
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  dim3 grid(splits, c.max_k + 1, B);
  cudaError_t e;
  prof_before(ctx, MTP_KERNEL_VERIFY, s);
  if (c.dtype == MTP_DTYPE_BF16) {
    VerifyArgs<uint16_t> a{(const uint16_t*)logits, row_offsets, drafts, drafts_stride, num_drafts, accepted, bonus,
                           ctx->ver_keys, ctx->ver_cnt, ctx->err, c.vocab, c.max_k, splits, num_rows};
    e = launch_pdl(verify_kernel<uint16_t>, grid, dim3(kVerifyThreads), 0, s, a);
  } else {
    VerifyArgs<float> a{(const float*)logits, row_offsets, drafts, drafts_stride, num_drafts, accepted, bonus,
                        ctx->ver_keys, ctx->ver_cnt, ctx->err, c.vocab, c.max_k, splits, num_rows};
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
// scratch (argmax keys and arrival counters) in the array below, which is part
// of the library's device image: it is created when the library's code is
// loaded on a GPU and stays resident there until the process exits.
namespace mtp {

constexpr int kNoAllocMaxKeys = 65536;   // B * (max_k + 1) rows
constexpr int kNoAllocMaxBatch = 4096;   // B
constexpr int kNoAllocMaxDevices = 64;

struct NoAllocScratch {
  unsigned long long keys[kNoAllocMaxKeys];
  int cnt[kNoAllocMaxBatch];
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
  if (B < 1 || B > kNoAllocMaxBatch || max_k < 0 || max_k > 100 || (long long)B * (max_k + 1) > kNoAllocMaxKeys)
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
  const size_t key_bytes = (size_t)B * (max_k + 1) * sizeof(unsigned long long);
  if (cudaMemsetAsync(sc->keys, 0, key_bytes, s) != cudaSuccess ||
      cudaMemsetAsync(sc->cnt, 0, (size_t)B * sizeof(int), s) != cudaSuccess ||
      cudaMemsetAsync(&sc->err, 0, sizeof(int), s) != cudaSuccess) {
    cudaGetLastError();
    return MTP_ERR_CUDA;
  }
  const int rows = B * (max_k + 1);
  int splits = (4 * sms + rows - 1) / rows;
  const int max_splits = (vocab + 2047) / 2048;
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  dim3 grid(splits, max_k + 1, B);
  cudaError_t e;
  if (dtype == MTP_DTYPE_BF16) {
    VerifyArgs<uint16_t> a{(const uint16_t*)target_logits, row_offsets, drafts, drafts_stride, num_drafts, accepted,
                           bonus, sc->keys, sc->cnt, &sc->err, vocab, max_k, splits, num_rows};
    e = launch_pdl(verify_kernel<uint16_t>, grid, dim3(kVerifyThreads), 0, s, a);
  } else {
    VerifyArgs<float> a{(const float*)target_logits, row_offsets, drafts, drafts_stride, num_drafts, accepted, bonus,
                        sc->keys, sc->cnt, &sc->err, vocab, max_k, splits, num_rows};
    e = launch_pdl(verify_kernel<float>, grid, dim3(kVerifyThreads), 0, s, a);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}
