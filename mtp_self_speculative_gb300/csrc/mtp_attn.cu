// Split-KV grouped-query decode attention over the paged single-layer MTP
// KV cache ("MTP (Multi-Token Prediction)", "Architecture": the decoder
// layer's attention; "How OpenVINO MTP Speculative Decoding Works
// Internally", "Why the MTP graph is a single decoder layer": its own
// one-layer cache).
//
// For request b at draft step k the query of every q head h attends to the
// T = seq_len[b] + k entries of its kv head g = h / G (G = n_q / n_kv):
//   o_h = softmax(q_h K_g^T / sqrt(d)) V_g.
//
// Grid (splits, n_kv, B); a CTA serves all G query heads of one kv head for
// a contiguous range of 16-token blocks.  Each of its 4 warps owns every 4th
// block of the range and stages it with one-dimensional bulk (TMA) copies --
// a K tile and a V tile, each 16 x d contiguous in the pool -- into its own
// ring of shared-memory stages, completed on per-stage mbarriers.  Scores:
// each lane holds d/32 dimensions of the G queries; per-token partial dot
// products are combined with a butterfly reduce-scatter so that lane l ends
// with the full score of token l & 15.  Softmax is online (running max and
// sum per head, base-2 exponentials with the scale folded into q).  Warps
// merge in shared memory; splits merge in the last CTA to finish (arrival
// counter), which writes o and resets the counter.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "mtp_common.cuh"
#include "mtp_attn_mma.cuh"

namespace mtp {

constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kStages = 3;
constexpr uint32_t kWaitLimit = 1u << 22;

template <typename T>
struct AttnArgs {
  const float* q;        // [B, n_q * d] rotated queries
  float* out;            // [B, n_q * d]
  uint16_t* out_bf16;    // [B, n_q * d] bf16 copy for the tensor-core O-proj, or null
  float* part;           // [B, n_q, max_splits, d + 4]: max, sum, -, -, o[d]
  int* cnt;              // [B, n_kv]
  int* err;
  const T* k_pool;
  const T* v_pool;
  const int32_t* block_table;
  const int32_t* seq_len;
  int k;                 // draft step (1-based): T = seq_len + k
  int n_q, n_kv, max_blocks, num_blocks, bps, max_splits;
  float qscale;          // log2(e) / sqrt(d)
};

template <typename T, int HD>
struct KVLane;
// Load the lane's d/32 contiguous elements of one row as floats.
template <int HD>
struct KVLane<uint16_t, HD> {
  static constexpr int DPL = HD / 32;
  __device__ static __forceinline__ void load(const uint16_t* row, int lane, float* o) {
    if constexpr (DPL == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(row + lane * 4);
      o[0] = bf16_lo(u.x); o[1] = bf16_hi(u.x); o[2] = bf16_lo(u.y); o[3] = bf16_hi(u.y);
    } else {
      const uint32_t u = *reinterpret_cast<const uint32_t*>(row + lane * 2);
      o[0] = bf16_lo(u); o[1] = bf16_hi(u);
    }
  }
};
template <int HD>
struct KVLane<float, HD> {
  static constexpr int DPL = HD / 32;
  __device__ static __forceinline__ void load(const float* row, int lane, float* o) {
    if constexpr (DPL == 4) {
      const float4 u = *reinterpret_cast<const float4*>(row + lane * 4);
      o[0] = u.x; o[1] = u.y; o[2] = u.z; o[3] = u.w;
    } else {
      const float2 u = *reinterpret_cast<const float2*>(row + lane * 2);
      o[0] = u.x; o[1] = u.y;
    }
  }
};

// Butterfly reduce-scatter of 16 per-lane partials: lane l returns the sum
// over all 32 lanes of partial[l & 15].
__device__ __forceinline__ float reduce_scatter16(float (&v)[16], int lane) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool hi = lane & 8;
    const float mine = hi ? v[i + 8] : v[i], other = hi ? v[i] : v[i + 8];
    v[i] = mine + __shfl_xor_sync(0xffffffffu, other, 8);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool hi = lane & 4;
    const float mine = hi ? v[i + 4] : v[i], other = hi ? v[i] : v[i + 4];
    v[i] = mine + __shfl_xor_sync(0xffffffffu, other, 4);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool hi = lane & 2;
    const float mine = hi ? v[i + 2] : v[i], other = hi ? v[i] : v[i + 2];
    v[i] = mine + __shfl_xor_sync(0xffffffffu, other, 2);
  }
  {
    const bool hi = lane & 1;
    const float mine = hi ? v[1] : v[0], other = hi ? v[0] : v[1];
    v[0] = mine + __shfl_xor_sync(0xffffffffu, other, 1);
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// Merge the per-warp online-softmax states of this CTA, then either write the
// output (one split) or a partial (M, L, O) and, in the last CTA of the
// (request, kv head), combine all splits: thread (head, 4 dims) merges the
// partials online, sixteen partials' loads in flight at a time.
template <typename T, int HD, int G>
__device__ __forceinline__ void attn_store_out(const AttnArgs<T>& a, int b, int g, int h, int d, float v) {
  const size_t oi = (size_t)b * a.n_q * HD + (size_t)(g * G + h) * HD + d;
  if (!MTP_IN_BOUNDS(a.err, oi, (long long)(b + 1) * a.n_q * HD)) return;
  a.out[oi] = v;
  if (a.out_bf16) a.out_bf16[oi] = f32_to_bf16_rne(v);
}

constexpr int kCombineBatch = 16;

// Online-softmax merge of (M, L, O) with another state (base-2 exponents).
__device__ __forceinline__ void merge_state(float& M, float& L, float4& O, float m2, float l2, float4 o2) {
  if (m2 == -INFINITY) return;
  const float Mn = fmaxf(M, m2);
  const float co = (M == -INFINITY) ? 0.0f : exp2f(M - Mn), cn = exp2f(m2 - Mn);
  L = L * co + l2 * cn;
  O.x = O.x * co + o2.x * cn;
  O.y = O.y * co + o2.y * cn;
  O.z = O.z * co + o2.z * cn;
  O.w = O.w * co + o2.w * cn;
  M = Mn;
}

// W warps per CTA.  Merge the per-warp online-softmax states of this CTA,
// then either write the output (one split) or a partial (M, L, O) and, in
// the last CTA of the (request, kv head), combine all splits: an item
// (head, 4 dims) is served by P = threads / items consecutive lanes (at
// least 1), lane p merging splits p, p + P, ... online (sixteen partials'
// loads in flight at a time); the P states then merge by shuffles.
template <typename T, int HD, int G, int W = kAttnWarps>
__device__ void attn_finish_merged(const AttnArgs<T>& a, const float* wacc, float (*wm)[G], float (*wl)[G], int s,
                                   int g, int b, int nsplit) {
  constexpr int RS = HD + 4;  // partial row stride (16-byte aligned rows)
  constexpr int NT = W * 32;
  constexpr int ITEMS = G * (HD / 4);
  constexpr int P = (NT / ITEMS) >= 8 ? 8 : (NT / ITEMS) >= 4 ? 4 : (NT / ITEMS) >= 2 ? 2 : 1;
  __shared__ int am_last;
  float* part_base = a.part + ((size_t)b * a.n_q + (size_t)g * G) * a.max_splits * RS;
  for (int idx = threadIdx.x; idx < G * HD; idx += NT) {
    const int h = idx / HD, d = idx - h * HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, wm[w][h]);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float f = (wm[w][h] == -INFINITY) ? 0.0f : exp2f(wm[w][h] - M);
      L += wl[w][h] * f;
      O += wacc[((size_t)w * G + h) * HD + d] * f;
    }
    if (nsplit == 1) {
      attn_store_out<T, HD, G>(a, b, g, h, d, O / L);
    } else {
      float* pp = part_base + ((size_t)h * a.max_splits + s) * RS;
      // this (request, head)'s row of partials: max_splits rows of RS floats
      if (MTP_IN_BOUNDS(a.err, (long long)s * RS + 4 + d, (long long)a.max_splits * RS)) {
        if (d == 0) { pp[0] = M; pp[1] = L; }
        pp[4 + d] = O;
      }
    }
  }
  if (nsplit == 1) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    // arrival with release (orders the CTA's partials, written before the
    // barrier) and acquire (the last CTA's reads below see every split's)
    int prev;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                 : "=r"(prev)
                 : "l"(a.cnt + (size_t)b * a.n_kv + g)
                 : "memory");
    am_last = (prev == nsplit - 1);
  }
  __syncthreads();
  if (!am_last) return;
  for (int it = threadIdx.x; it < ITEMS * P; it += NT) {
    const int item = it / P, p = it - item * P;
    const int h = item / (HD / 4), d4 = item - h * (HD / 4);
    const float* ph = part_base + (size_t)h * a.max_splits * RS;
    float Mr = -INFINITY, Lr = 0.0f;
    float4 Or = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int j0 = p; j0 < nsplit; j0 += P * kCombineBatch) {
      float mj[kCombineBatch], lj[kCombineBatch];
      float4 oj[kCombineBatch];
#pragma unroll
      for (int q = 0; q < kCombineBatch; ++q) {
        const int j = j0 + q * P;
        mj[q] = -INFINITY;
        lj[q] = 0.0f;
        oj[q] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (j < nsplit) {
          const float* r = ph + (size_t)j * RS;
          mj[q] = __ldcg(r);
          lj[q] = __ldcg(r + 1);
          oj[q] = __ldcg(reinterpret_cast<const float4*>(r + 4) + d4);
        }
      }
#pragma unroll
      for (int q = 0; q < kCombineBatch; ++q) merge_state(Mr, Lr, Or, mj[q], lj[q], oj[q]);
    }
    if constexpr (P > 1) {
      // all threads take part (ITEMS * P == NT): merge the P lanes of an item
#pragma unroll
      for (int o = 1; o < P; o <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, Mr, o), l2 = __shfl_xor_sync(0xffffffffu, Lr, o);
        float4 o2;
        o2.x = __shfl_xor_sync(0xffffffffu, Or.x, o);
        o2.y = __shfl_xor_sync(0xffffffffu, Or.y, o);
        o2.z = __shfl_xor_sync(0xffffffffu, Or.z, o);
        o2.w = __shfl_xor_sync(0xffffffffu, Or.w, o);
        merge_state(Mr, Lr, Or, m2, l2, o2);
      }
    }
    if (p == 0) {
      const float inv = 1.0f / Lr;
      attn_store_out<T, HD, G>(a, b, g, h, 4 * d4 + 0, Or.x * inv);
      attn_store_out<T, HD, G>(a, b, g, h, 4 * d4 + 1, Or.y * inv);
      attn_store_out<T, HD, G>(a, b, g, h, 4 * d4 + 2, Or.z * inv);
      attn_store_out<T, HD, G>(a, b, g, h, 4 * d4 + 3, Or.w * inv);
    }
  }
  if (threadIdx.x == 0) a.cnt[(size_t)b * a.n_kv + g] = 0;
}

template <typename T, int HD, int G, int DPL>
__device__ __forceinline__ void attn_finish(const AttnArgs<T>& a, unsigned char* smem_raw, float (*wm)[G],
                                            float (*wl)[G], const float (&m)[G], const float (&l)[G],
                                            const float (&acc)[G][DPL], int warp, int lane, int s, int g, int b,
                                            int nsplit) {
  float* wacc = reinterpret_cast<float*>(smem_raw);  // reuse stages: [warps][G][HD]
  __syncthreads();
  if (lane == 0)
#pragma unroll
    for (int h = 0; h < G; ++h) { wm[warp][h] = m[h]; wl[warp][h] = l[h]; }
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int j = 0; j < DPL; ++j) wacc[((size_t)warp * G + h) * HD + lane * DPL + j] = acc[h][j];
  __syncthreads();
  attn_finish_merged<T, HD, G>(a, wacc, wm, wl, s, g, b, nsplit);
}

// The CTA's slice of the request's block table, blocks s*bps .. s*bps +
// bps - 1 (those below max_blocks), into shared memory in one coalesced
// pass.  No kernel writes the block table, so this runs before the
// dependency wait; the tiles' copies then need no dependent L2 read each.
template <typename T>
__device__ __forceinline__ void load_block_slice(const AttnArgs<T>& a, int* s_bt, int s, int b,
                                                 int nthreads = kAttnThreads) {
  const int blk0 = s * a.bps;
  const int n = min(a.bps, a.max_blocks - blk0);
  for (int i = threadIdx.x; i < n; i += nthreads) s_bt[i] = a.block_table[(size_t)b * a.max_blocks + blk0 + i];
}

// Shared-memory bytes of the block-table slice (16-byte multiple).
__host__ __device__ __forceinline__ size_t block_slice_bytes(int bps) { return ((size_t)bps * 4 + 15) & ~(size_t)15; }

template <typename T, int HD, int G>
__global__ void __launch_bounds__(kAttnThreads, 2) attn_kernel(const AttnArgs<T> a) {
  constexpr int DPL = HD / 32;
  constexpr int TILE = 16 * HD;                      // elements per K (or V) tile
  constexpr uint32_t TILE_BYTES = TILE * sizeof(T);
  constexpr int HC = (G < 4) ? G : 4;                // heads per score pass
  extern __shared__ __align__(128) unsigned char smem_raw[];
  T* stage_base = reinterpret_cast<T*>(smem_raw);    // [warps][stages][2][TILE]
  __shared__ __align__(8) uint64_t bars[kAttnWarps][kStages];
  __shared__ float wm[kAttnWarps][G], wl[kAttnWarps][G];

  constexpr size_t kStageBytes = (size_t)kAttnWarps * kStages * 2 * TILE * sizeof(T);
  constexpr size_t kMergeBytes = (size_t)kAttnWarps * G * HD * sizeof(float);
  int* s_bt = reinterpret_cast<int*>(smem_raw + (kStageBytes > kMergeBytes ? kStageBytes : kMergeBytes));

  pdl_trigger();
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < kAttnWarps * kStages) mbar_init(&bars[threadIdx.x / kStages][threadIdx.x % kStages], 1);
  fence_mbar_init();
  load_block_slice(a, s_bt, s, b);
  __syncthreads();
  pdl_wait();

  const int T_len = a.seq_len[b] + a.k;
  const int nblk = (T_len + 15) >> 4;
  const int blk0 = s * a.bps;
  if (blk0 >= nblk || T_len <= 0) return;  // uniform across the CTA
  const int blk1 = min(nblk, blk0 + a.bps);
  const int nsplit = (nblk + a.bps - 1) / a.bps;

  // Queries of this group, scaled for base-2 softmax: lane holds dims [lane*DPL, +DPL).
  float qv[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int j = 0; j < DPL; ++j)
      qv[h][j] = a.q[(size_t)b * a.n_q * HD + (size_t)(g * G + h) * HD + lane * DPL + j] * a.qscale;

  float m[G], l[G], acc[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) acc[h][j] = 0.0f;
  }

  T* my_stage = stage_base + (size_t)warp * kStages * 2 * TILE;
  const size_t head_stride = (size_t)16 * HD;  // elements per (block, kv head) tile
  auto tile_src = [&](int bi, const T* pool) -> const T* {
    int blk = (bi < a.max_blocks) ? s_bt[bi - blk0] : -1;
    if (blk < 0 || blk >= a.num_blocks) {
      set_error(a.err, MTP_ERR_CAPACITY);
      blk = 0;
    }
    return pool + ((size_t)blk * a.n_kv + g) * head_stride;
  };
  auto issue = [&](int it, int bi) {
    const int st = it % kStages;
    T* dst = my_stage + (size_t)st * 2 * TILE;
    mbar_expect_tx(&bars[warp][st], 2 * TILE_BYTES);
    bulk_g2s(dst, tile_src(bi, a.k_pool), TILE_BYTES, &bars[warp][st]);
    bulk_g2s(dst + TILE, tile_src(bi, a.v_pool), TILE_BYTES, &bars[warp][st]);
  };

  // This warp's blocks: blk0 + warp, blk0 + warp + 4, ...
  const int first = blk0 + warp;
  const int count = (first < blk1) ? (blk1 - first + kAttnWarps - 1) / kAttnWarps : 0;
  if (lane == 0)
    for (int it = 0; it < count && it < kStages; ++it) issue(it, first + it * kAttnWarps);
  __syncwarp();

  int stop_at = -1;  // iteration whose wait ran out
  for (int it = 0; it < count; ++it) {
    const int st = it % kStages;
    const uint32_t parity = (uint32_t)((it / kStages) & 1);
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[warp][st], parity, kWaitLimit));
    if (!ok) {
      stop_at = it;
      break;
    }
    const T* kt = my_stage + (size_t)st * 2 * TILE;
    const T* vt = kt + TILE;
    const int bi = first + it * kAttnWarps;
    const int tok0 = bi * 16;
    const int my_tok = tok0 + (lane & 15);
    const bool valid = my_tok < T_len;

    // scores s[h] for token (lane & 15)
    float sc[G];
#pragma unroll
    for (int h0 = 0; h0 < G; h0 += HC) {
      float part[HC][16];
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        float kvv[DPL];
        KVLane<T, HD>::load(kt + t * HD, lane, kvv);
#pragma unroll
        for (int hh = 0; hh < HC; ++hh) {
          float p = 0.0f;
#pragma unroll
          for (int j = 0; j < DPL; ++j) p = fmaf(qv[h0 + hh][j], kvv[j], p);
          part[hh][t] = p;
        }
      }
#pragma unroll
      for (int hh = 0; hh < HC; ++hh) sc[h0 + hh] = reduce_scatter16(part[hh], lane);
    }

    float pr[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float sv = valid ? sc[h] : -INFINITY;
      float bmax = sv;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
      const float m_new = fmaxf(m[h], bmax);
      const float corr = (m[h] == -INFINITY) ? 0.0f : exp2f(m[h] - m_new);
      const float p = valid ? exp2f(sv - m_new) : 0.0f;
      float psum = p;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      l[h] = l[h] * corr + psum;
      m[h] = m_new;
#pragma unroll
      for (int j = 0; j < DPL; ++j) acc[h][j] *= corr;
      pr[h] = p;
    }
#pragma unroll
    for (int t = 0; t < 16; ++t) {
      float vv[DPL];
      KVLane<T, HD>::load(vt + t * HD, lane, vv);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float p = __shfl_sync(0xffffffffu, pr[h], t);
#pragma unroll
        for (int j = 0; j < DPL; ++j) acc[h][j] = fmaf(p, vv[j], acc[h][j]);
      }
    }
    __syncwarp();
    if (lane == 0 && it + kStages < count) issue(it + kStages, first + (it + kStages) * kAttnWarps);
    __syncwarp();
  }
  if (stop_at >= 0) {
    if (lane == 0) set_error(a.err, MTP_ERR_TIMEOUT);
    // give the copies still in flight (iterations stop_at .. stop_at + kStages - 1)
    // a bounded chance to land before the shared memory is reused
    for (int it = stop_at; it < count && it < stop_at + kStages; ++it)
      mbar_wait_bounded(&bars[warp][it % kStages], (uint32_t)((it / kStages) & 1), kWaitLimit);
  }

  attn_finish<T, HD, G, DPL>(a, smem_raw, wm, wl, m, l, acc, warp, lane, s, g, b, nsplit);
}

// ------------------------------------------------ split combine in a cluster
//
// All splits of one (request, kv head) form one thread-block cluster (at most
// 16 CTAs).  Each CTA merges its warps' online-softmax states into one
// partial (M, L, O) per query head in its own shared memory; after a cluster
// barrier, CTA r combines output columns r, r + S, ... (S = cluster size, one
// column = 4 values of one head), 16 lanes per column, lane j reading split
// j's partial through distributed shared memory; a second barrier keeps every
// CTA's partial alive until all reads are done.  Splits with no blocks hold
// an empty state (M = -inf), so the combine is the same as the global one:
// no partials in HBM, no arrival counter, no last-CTA pass.

__device__ __forceinline__ uint32_t attn_mapa(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void attn_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int HD, int G, int W>
__device__ void attn_finish_cluster(const AttnArgs<uint16_t>& a, const float* wacc, float (*wm)[G], float (*wl)[G],
                                    float* cpart, int g, int b) {
  constexpr int RS = HD + 4;  // partial row: M, L, -, -, O[HD] (16-byte aligned)
  constexpr int NT = W * 32;
  constexpr int ITEMS = G * (HD / 4);
  for (int idx = threadIdx.x; idx < G * HD; idx += NT) {
    const int h = idx / HD, d = idx - h * HD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, wm[w][h]);
    float L = 0.0f, O = 0.0f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float f = (wm[w][h] == -INFINITY) ? 0.0f : exp2f(wm[w][h] - M);
      L += wl[w][h] * f;
      O += wacc[((size_t)w * G + h) * HD + d] * f;
    }
    if (d == 0) {
      cpart[h * RS] = M;
      cpart[h * RS + 1] = L;
    }
    cpart[h * RS + 4 + d] = O;
  }
  attn_cluster_sync();
  const int S = (int)gridDim.x;  // the cluster spans the grid's x
  const int r = (int)blockIdx.x;
  const int per = (ITEMS + S - 1) / S;
  const uint32_t base = smem_addr(cpart);
  for (int t0 = 0; t0 < per * 16; t0 += NT) {
    const int t = t0 + (int)threadIdx.x;
    const int j = t & 15;
    const int item = r + (t >> 4) * S;
    const bool have = (t < per * 16) && item < ITEMS;
    const int h = have ? item / (HD / 4) : 0, d4 = have ? item - h * (HD / 4) : 0;
    float Mr = -INFINITY, Lr = 0.0f;
    float4 Or = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (have && j < S) {
      const uint32_t row = attn_mapa(base + (uint32_t)(h * RS) * 4u, (uint32_t)j);
      float2 ml;
      asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(ml.x), "=f"(ml.y) : "r"(row));
      asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(Or.x), "=f"(Or.y), "=f"(Or.z), "=f"(Or.w)
                   : "r"(row + 16u + 16u * (uint32_t)d4));
      Mr = ml.x;
      Lr = ml.y;
      if (Mr == -INFINITY) {
        Lr = 0.0f;
        Or = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
    }
    // merge the 16 lanes of the column (xor offsets below 16 stay in the group)
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, Mr, o), l2 = __shfl_xor_sync(0xffffffffu, Lr, o);
      float4 o2;
      o2.x = __shfl_xor_sync(0xffffffffu, Or.x, o);
      o2.y = __shfl_xor_sync(0xffffffffu, Or.y, o);
      o2.z = __shfl_xor_sync(0xffffffffu, Or.z, o);
      o2.w = __shfl_xor_sync(0xffffffffu, Or.w, o);
      merge_state(Mr, Lr, Or, m2, l2, o2);
    }
    if (have && j == 0) {
      const float inv = 1.0f / Lr;
      attn_store_out<uint16_t, HD, G>(a, b, g, h, 4 * d4 + 0, Or.x * inv);
      attn_store_out<uint16_t, HD, G>(a, b, g, h, 4 * d4 + 1, Or.y * inv);
      attn_store_out<uint16_t, HD, G>(a, b, g, h, 4 * d4 + 2, Or.z * inv);
      attn_store_out<uint16_t, HD, G>(a, b, g, h, 4 * d4 + 3, Or.w * inv);
    }
  }
  attn_cluster_sync();
}

// ------------------------------------------------ tensor-core attention
//
// bf16 cache, head_dim 128.  Same split-KV grid and per-warp block ownership
// as above; each block's arithmetic is attn_tile_mma (mma.sync m16n8k16 with
// the group's query heads on M, P kept in registers) on K/V tiles staged by
// swizzled 2-D tensor-map loads.

template <int G, int W, int NSTG, bool CL>
__global__ void __launch_bounds__(W * 32, (W <= 4) ? 2 : 1)
    attn_mma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    const AttnArgs<uint16_t> a) {
  constexpr int HD = 128;
  constexpr uint32_t TILE_BYTES = 16 * HD * 2;  // 4 KB per K or V tile
  extern __shared__ __align__(1024) unsigned char smem_raw_in[];
  unsigned char* smem_raw = (unsigned char*)(((uintptr_t)smem_raw_in + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t bars[W][NSTG];
  __shared__ float wm[W][G], wl[W][G];

  int* s_bt = reinterpret_cast<int*>(smem_raw + (size_t)W * NSTG * 2 * TILE_BYTES);

  pdl_trigger();
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = lane >> 2, ti = lane & 3;
  if (threadIdx.x < W * NSTG) mbar_init(&bars[threadIdx.x / NSTG][threadIdx.x % NSTG], 1);
  fence_mbar_init();
  load_block_slice(a, s_bt, s, b, W * 32);
  __syncthreads();
  pdl_wait();

  const int T_len = a.seq_len[b] + a.k;
  const int nblk = (T_len + 15) >> 4;
  const int blk0 = s * a.bps;
  // in a cluster every split stays to the combine (T_len is the cluster's
  // own, so that return is cluster-uniform)
  if (T_len <= 0 || (!CL && blk0 >= nblk)) return;
  const int blk1 = min(nblk, blk0 + a.bps);
  const int nsplit = (nblk + a.bps - 1) / a.bps;

  unsigned char* my_stage = smem_raw + (size_t)warp * NSTG * 2 * TILE_BYTES;
  auto tile_row = [&](int bi) -> int {
    int blk = (bi < a.max_blocks) ? s_bt[bi - blk0] : -1;
    if (blk < 0 || blk >= a.num_blocks) {
      set_error(a.err, MTP_ERR_CAPACITY);
      blk = 0;
    }
    return (blk * a.n_kv + g) * 16;
  };
  auto issue = [&](int it, int bi) {
    const int st = it % NSTG;
    tma_kv_tile(my_stage + (size_t)st * 2 * TILE_BYTES, &kmap, &vmap, tile_row(bi), &bars[warp][st]);
  };

  const int first = blk0 + warp;
  const int count = (first < blk1) ? (blk1 - first + W - 1) / W : 0;
  if (lane == 0)
    for (int it = 0; it < count && it < NSTG; ++it) issue(it, first + it * W);
  __syncwarp();

  // the query fragments load while the first tiles are in flight
  uint32_t qa[8][4];
  load_q_frags(qa, a.q + (size_t)b * a.n_q * HD + (size_t)(g * G) * HD, a.qscale, lane, G);
  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;

  int stop_at = -1;
  for (int it = 0; it < count; ++it) {
    const int st = it % NSTG;
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars[warp][st], (uint32_t)((it / NSTG) & 1),
                                                              kWaitLimit));
    if (!ok) {
      stop_at = it;
      break;
    }
    const uint32_t kt = smem_addr(my_stage + (size_t)st * 2 * TILE_BYTES);
    const uint32_t vt = kt + TILE_BYTES;
    const int tok0 = (first + it * W) * 16;

    attn_tile_mma(kt, vt, qa, o, m_run, l_run, tok0, T_len, lane);
    __syncwarp();
    if (lane == 0 && it + NSTG < count) issue(it + NSTG, first + (it + NSTG) * W);
    __syncwarp();
  }
  if (stop_at >= 0) {
    if (lane == 0) set_error(a.err, MTP_ERR_TIMEOUT);
    for (int it = stop_at; it < count && it < stop_at + NSTG; ++it)
      mbar_wait_bounded(&bars[warp][it % NSTG], (uint32_t)((it / NSTG) & 1), kWaitLimit);
  }

  // per-warp state -> shared memory, then the common merge/combine
  float* wacc = reinterpret_cast<float*>(smem_raw);  // [warps][G][HD]
  __syncthreads();
  if (gi < G && ti == 0) {
    wm[warp][gi] = m_run;
    wl[warp][gi] = l_run;
  }
  if (gi < G) {
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      wacc[((size_t)warp * G + gi) * HD + 8 * n + 2 * ti] = o[n][0];
      wacc[((size_t)warp * G + gi) * HD + 8 * n + 2 * ti + 1] = o[n][1];
    }
  }
  __syncthreads();
  if constexpr (CL)
    attn_finish_cluster<HD, G, W>(a, wacc, wm, wl, wacc + (size_t)W * G * HD, g, b);
  else
    attn_finish_merged<uint16_t, HD, G, W>(a, wacc, wm, wl, s, g, b, nsplit);
}

template <int G, int W, int NSTG>
static cudaError_t attn_mma_launch(dim3 grid, size_t smem, cudaStream_t s, const CUtensorMap& km,
                                   const CUtensorMap& vm, const AttnArgs<uint16_t>& ab) {
  auto kern = attn_mma_kernel<G, W, NSTG, false>;
  const cudaError_t e = ensure_smem((const void*)kern, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, dim3(W * 32), smem, s, km, vm, ab);
}

// The cluster form: grid.x splits (2..16) of one (request, kv head) per
// cluster.  `query` only asks how many such clusters fit on the GPU at once.
template <int G>
static cudaError_t attn_cluster_launch(dim3 grid, size_t smem, cudaStream_t s, const CUtensorMap* km,
                                       const CUtensorMap* vm, const AttnArgs<uint16_t>* ab, int* query) {
  auto kern = attn_mma_kernel<G, 8, 2, true>;
  cudaError_t e = ensure_smem((const void*)kern, smem);
  if (e != cudaSuccess) return e;
  static bool nonportable = false;
  if (!nonportable) {
    e = cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    nonportable = true;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = dim3(8 * 32);
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = grid.x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  if (query) {
    lc.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(query, (const void*)kern, &lc);
  }
  lc.numAttrs = 2;
  return cudaLaunchKernelEx(&lc, kern, *km, *vm, *ab);
}

template <typename T, int HD, int G>
static cudaError_t attn_launch(mtp_ctx* ctx, cudaStream_t s, const AttnArgs<T>& a, int B, int splits) {
  constexpr size_t stage_bytes = (size_t)kAttnWarps * kStages * 2 * 16 * HD * sizeof(T);
  constexpr size_t merge_bytes = (size_t)kAttnWarps * G * HD * sizeof(float);
  const size_t smem = (stage_bytes > merge_bytes ? stage_bytes : merge_bytes) + block_slice_bytes(a.bps);
  auto kern = attn_kernel<T, HD, G>;
  ensure_smem((const void*)kern, smem);
  return launch_pdl(kern, dim3(splits, ctx->cfg.n_kv_heads, B), dim3(kAttnThreads), smem, s, a);
}

// Blocks per split for a batch of B requests and max_blocks capacity: aim
// for about attn_target_ctas CTAs (several waves, so that the splits of the
// longest requests of a ragged batch do not set the kernel's length), never
// more than max_splits splits nor fewer than min_bps blocks per split.
static int attn_bps(const mtp_ctx* ctx, int B, int max_blocks, int min_bps) {
  const long long pairs = (long long)B * ctx->cfg.n_kv_heads;
  long long splits = (ctx->attn_target_ctas + pairs - 1) / pairs;
  if (splits < 1) splits = 1;
  if (splits > ctx->attn_max_splits) splits = ctx->attn_max_splits;
  int bps = (int)((max_blocks + splits - 1) / splits);
  if (bps < min_bps) bps = min_bps;
  while ((max_blocks + bps - 1) / bps > ctx->attn_max_splits) ++bps;
  return bps;
}

struct AttnMapCache {
  CUtensorMap km, vm;
  const void* k_pool;
  const void* v_pool;
  int num_blocks;
};

bool attn_tensor_maps(mtp_ctx* ctx, const mtp_kv* kv, const CUtensorMap** km, const CUtensorMap** vm) {
  // re-encoded only when the pools change
  if (!ctx->attn_map_cache) {
    ctx->attn_map_cache = aligned_alloc(64, sizeof(AttnMapCache));
    if (!ctx->attn_map_cache) return false;
    memset(ctx->attn_map_cache, 0, sizeof(AttnMapCache));
  }
  AttnMapCache* mc = (AttnMapCache*)ctx->attn_map_cache;
  if (mc->k_pool != kv->k_pool || mc->v_pool != kv->v_pool || mc->num_blocks != kv->num_blocks) {
    const uint64_t rows = (uint64_t)kv->num_blocks * ctx->cfg.n_kv_heads * 16;
    if (!make_map(&mc->km, kv->k_pool, rows, 128, 16) || !make_map(&mc->vm, kv->v_pool, rows, 128, 16)) {
      mc->k_pool = mc->v_pool = nullptr;
      return false;
    }
    mc->k_pool = kv->k_pool;
    mc->v_pool = kv->v_pool;
    mc->num_blocks = kv->num_blocks;
  }
  *km = &mc->km;
  *vm = &mc->vm;
  return true;
}

template <typename T>
static cudaError_t attention_t(mtp_ctx* ctx, cudaStream_t s, int B, int k, const mtp_kv* kv) {
  const mtp_config& c = ctx->cfg;
  AttnArgs<T> a;
  a.q = ctx->q; a.out = ctx->attn; a.out_bf16 = tc_supported(ctx, B) ? ctx->tc_attn : nullptr; a.part = ctx->attn_part; a.cnt = ctx->attn_cnt; a.err = ctx->err;
  a.k_pool = (const T*)kv->k_pool; a.v_pool = (const T*)kv->v_pool;
  a.block_table = kv->block_table; a.seq_len = kv->seq_len; a.k = k;
  a.n_q = c.n_q_heads; a.n_kv = c.n_kv_heads; a.max_blocks = kv->max_blocks; a.num_blocks = kv->num_blocks;
  const int G = c.n_q_heads / c.n_kv_heads;
  const int HD = c.head_dim;
  const bool use_mma = sizeof(T) == 2 && HD == 128;
  // the tensor-core kernel keeps at least 16 blocks per split to amortise
  // its set-up and the split combine (32 at 2-4 requests, where the planned
  // 16 gave up to 2 waves of narrow CTAs: per launch at B=2 16.3 against
  // 22.3 us, the bf=4 tree loop 1.4% faster); when its grid is short of two
  // CTAs per SM it runs eight warps per CTA (two blocks each at 16 blocks per
  // split)
  a.bps = attn_bps(ctx, B, kv->max_blocks, use_mma ? (B >= 2 && B <= 4 ? 32 : 16) : 2);
  if (ctx->attn_force_bps > 0) {
    // a forced split size (tuning) is taken only while the partials of all
    // splits fit the buffer sized for the planned ones
    int bps = ctx->attn_force_bps;
    while ((kv->max_blocks + bps - 1) / bps > ctx->attn_max_splits) ++bps;
    const long long rows = (long long)B * ((kv->max_blocks + bps - 1) / bps);
    if (rows <= (long long)ctx->attn_target_ctas / c.n_kv_heads + ctx->cfg.max_batch + 1) a.bps = bps;
  }
  const long long mma_ctas = (long long)((kv->max_blocks + a.bps - 1) / a.bps) * c.n_kv_heads * B;
  const bool wide = use_mma && mma_ctas <= 2LL * ctx->num_sms;
  const int splits = (kv->max_blocks + a.bps - 1) / a.bps;
  a.max_splits = splits;  // partial-buffer stride of this call
  a.qscale = 1.4426950408889634f / sqrtf((float)c.head_dim);
  if (use_mma) {
    const CUtensorMap *kmp, *vmp;
    if (!attn_tensor_maps(ctx, kv, &kmp, &vmp)) return cudaErrorInvalidValue;
    const CUtensorMap& km = *kmp;
    const CUtensorMap& vm = *vmp;
    const AttnArgs<uint16_t>& ab = reinterpret_cast<const AttnArgs<uint16_t>&>(a);
    dim3 grid(splits, c.n_kv_heads, B);
    if (ctx->attn_cluster && (G == 1 || G == 2 || G == 4 || G == 8)) {
      // every split of a (request, kv head) in one cluster of at most 16
      // CTAs: the largest cluster size (from the planned split) whose
      // B * n_kv clusters all fit on the GPU at once, planned once per
      // (capacity, G, clusters, forced split) and cached
      const long long key = ((long long)kv->max_blocks << 40) | ((long long)G << 32) |
                            ((long long)(c.n_kv_heads * B) << 12) | (long long)(a.bps & 0xfff);
      if (ctx->attn_cl_key != key) {
        ctx->attn_cl_key = key;
        ctx->attn_cl_fit = 0;
        ctx->attn_cl_bps = 0;
        int cs0 = (kv->max_blocks + a.bps - 1) / a.bps;
        if (cs0 > 16) cs0 = (ctx->attn_force_bps == 0) ? 16 : 0;
        // fewer splits lengthen every CTA's serial part: at most a quarter fewer
        const int want_min = (3 * cs0 + 3) / 4 > 2 ? (3 * cs0 + 3) / 4 : 2;
        for (int want = cs0; want >= want_min; --want) {
          const int bps = (kv->max_blocks + want - 1) / want;
          const int cs = (kv->max_blocks + bps - 1) / bps;
          if ((long long)cs * c.n_kv_heads * B > 2LL * ctx->num_sms) continue;
          const size_t smem = 1024 + (size_t)8 * 2 * 2 * 4096 + block_slice_bytes(bps);
          const dim3 gc(cs, c.n_kv_heads, B);
          int fit = 0;
          cudaError_t eq = (G == 1)   ? attn_cluster_launch<1>(gc, smem, s, nullptr, nullptr, nullptr, &fit)
                           : (G == 2) ? attn_cluster_launch<2>(gc, smem, s, nullptr, nullptr, nullptr, &fit)
                           : (G == 4) ? attn_cluster_launch<4>(gc, smem, s, nullptr, nullptr, nullptr, &fit)
                                      : attn_cluster_launch<8>(gc, smem, s, nullptr, nullptr, nullptr, &fit);
          if (eq != cudaSuccess) {
            cudaGetLastError();
            fit = 0;
          }
          if (getenv("MTP_ATTN_TRACE"))
            fprintf(stderr, "attention cluster: %d splits of %d blocks, G %d, %zu B smem: %d clusters fit, %d needed\n",
                    cs, bps, G, smem, fit, c.n_kv_heads * B);
          if (fit >= c.n_kv_heads * B) {
            ctx->attn_cl_fit = cs;
            ctx->attn_cl_bps = bps;
            break;
          }
          if (ctx->attn_force_bps) break;  // a forced split size is taken as it is or not at all
        }
      }
      if (ctx->attn_cl_fit >= 2) {
        const int cs = ctx->attn_cl_fit, bps = ctx->attn_cl_bps;
        const size_t smem = 1024 + (size_t)8 * 2 * 2 * 4096 + block_slice_bytes(bps);
        const dim3 gc(cs, c.n_kv_heads, B);
        AttnArgs<uint16_t> ac = ab;
        ac.bps = bps;
        ac.max_splits = cs;
        ctx->path_counts[MTP_PATH_ATTN_CLUSTER]++;
        switch (G) {
          case 1: return attn_cluster_launch<1>(gc, smem, s, &km, &vm, &ac, nullptr);
          case 2: return attn_cluster_launch<2>(gc, smem, s, &km, &vm, &ac, nullptr);
          case 4: return attn_cluster_launch<4>(gc, smem, s, &km, &vm, &ac, nullptr);
          case 8: return attn_cluster_launch<8>(gc, smem, s, &km, &vm, &ac, nullptr);
        }
      }
    }
    if (wide) {
      // few CTAs: 8 warps of 2 stages each, every tile of a 16-block split
      // requested at once
      const size_t smem = 1024 + (size_t)8 * 2 * 2 * 4096 + block_slice_bytes(a.bps);
      switch (G) {
        case 1: return attn_mma_launch<1, 8, 2>(grid, smem, s, km, vm, ab);
        case 2: return attn_mma_launch<2, 8, 2>(grid, smem, s, km, vm, ab);
        case 4: return attn_mma_launch<4, 8, 2>(grid, smem, s, km, vm, ab);
        case 8: return attn_mma_launch<8, 8, 2>(grid, smem, s, km, vm, ab);
      }
      return cudaErrorInvalidValue;
    }
    const size_t smem = 1024 + (size_t)kAttnWarps * kStages * 2 * 4096 + block_slice_bytes(a.bps);
    switch (G) {
      case 1: return attn_mma_launch<1, kAttnWarps, kStages>(grid, smem, s, km, vm, ab);
      case 2: return attn_mma_launch<2, kAttnWarps, kStages>(grid, smem, s, km, vm, ab);
      case 4: return attn_mma_launch<4, kAttnWarps, kStages>(grid, smem, s, km, vm, ab);
      case 8: return attn_mma_launch<8, kAttnWarps, kStages>(grid, smem, s, km, vm, ab);
    }
    return cudaErrorInvalidValue;
  }
  if (HD == 128) {
    switch (G) {
      case 1: return attn_launch<T, 128, 1>(ctx, s, a, B, splits);
      case 2: return attn_launch<T, 128, 2>(ctx, s, a, B, splits);
      case 4: return attn_launch<T, 128, 4>(ctx, s, a, B, splits);
      case 8: return attn_launch<T, 128, 8>(ctx, s, a, B, splits);
    }
  } else if (HD == 64) {
    switch (G) {
      case 1: return attn_launch<T, 64, 1>(ctx, s, a, B, splits);
      case 2: return attn_launch<T, 64, 2>(ctx, s, a, B, splits);
      case 4: return attn_launch<T, 64, 4>(ctx, s, a, B, splits);
      case 8: return attn_launch<T, 64, 8>(ctx, s, a, B, splits);
    }
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_attention(mtp_ctx* ctx, cudaStream_t s, int B, int k, const mtp_kv* kv) {
  prof_before(ctx, MTP_KERNEL_ATTENTION, s);
  cudaError_t e = (ctx->cfg.dtype == MTP_DTYPE_BF16) ? attention_t<uint16_t>(ctx, s, B, k, kv)
                                                     : attention_t<float>(ctx, s, B, k, kv);
  prof_after(ctx, MTP_KERNEL_ATTENTION, s);
  ctx->launches++;
  return e;
}

}  // namespace mtp
