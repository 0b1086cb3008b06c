// Weight-streaming kernels of one MTP draft step (small batch, CUDA cores).
//
// Every projection of the draft step is a matrix-vector product whose
// weights are read exactly once per step; the kernels are bound by HBM
// bandwidth.  One template covers all of them:
//
//   EH_PROJ   x   = W_eh [RMSNorm(h) w_h ; RMSNorm(e) w_e]           (2H -> H)
//   QKV_ROPE  q,k,v = W_{q,k,v} RMSNorm(x) w_in, rotary on q and k, k/v
//             appended to the paged KV cache (bf16 round-to-nearest-even)
//   O_PROJ    h1  = x + W_o o
//   GATE_UP   a   = silu(W_g n2) * (W_u n2),  n2 = RMSNorm(h1) w_post
//   DOWN      h2  = h1 + W_d a
//   LM_HEAD   z   = W_lm RMSNorm(h2) w_f, argmax (lowest id on ties)
//
// ("MTP (Multi-Token Prediction)", "Architecture": dual norm, concat,
// projection, one standard decoder layer, shared LM head.)
//
// Layout of the work: the grid is two CTAs per SM; CTA i owns a contiguous,
// balanced range of row pairs; its 8 warps take pairs round-robin.  A warp
// streams both rows of a pair with 16-byte non-allocating loads, U vectors
// per lane in flight per row, against the normalised input vector(s) staged
// once per CTA in shared memory as fp32.  Before waiting on the previous
// kernel (programmatic dependent launch) each warp prefetches the head of
// its first rows into L2, so the weight stream starts while the previous
// kernel drains.
#include "mtp_common.cuh"

namespace mtp {

enum GemvKind { EH_PROJ = 0, QKV_ROPE = 1, O_PROJ = 2, GATE_UP = 3, DOWN = 4, LM_HEAD = 5 };

template <typename T>
struct StepArgs {
  int B, H, q_dim, kv_dim, F, V, n_q, n_kv, hd, bs;
  float eps;
  int k, K;
  int max_pos, num_blocks, max_blocks;
  const T *w_norm_h, *w_norm_e, *w_eh, *w_norm_in, *w_q, *w_k, *w_v, *w_o;
  const T *w_norm_post, *w_gate, *w_up, *w_down, *w_norm_f, *embed, *lm_head;
  const T* hidden_in;
  const T* embeds_in;
  const int32_t* positions;
  const int32_t* chain_ids;
  int32_t* draft_ids;
  float* logits;
  float* hidden_out;
  T* k_pool;
  T* v_pool;
  const int32_t* block_table;
  const int32_t* seq_len;
  int32_t* pending;
  float *hid, *x, *q, *attn, *h1, *act;
  unsigned long long* lm_keys;
  int* lm_cnt;
  int* err;
  int* req_bad;
  const float2* rope;
};

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 8;

template <typename T>
__device__ __forceinline__ int gemv_cols(const StepArgs<T>& a, int kind) {
  switch (kind) {
    case EH_PROJ: return 2 * a.H;
    case O_PROJ: return a.q_dim;
    case DOWN: return a.F;
    default: return a.H;
  }
}

template <typename T>
__device__ __forceinline__ int gemv_pairs(const StepArgs<T>& a, int kind) {
  switch (kind) {
    case EH_PROJ: return a.H / 2;
    case QKV_ROPE: return (a.q_dim + 2 * a.kv_dim) / 2;
    case O_PROJ: return a.H / 2;
    case GATE_UP: return a.F;
    case DOWN: return a.H / 2;
    default: return (a.V + 1) / 2;
  }
}

// Rows (r0, r1) of pair p and their weight pointers.  r1 < 0: no second row.
template <typename T, int KIND>
__device__ __forceinline__ void pair_rows(const StepArgs<T>& a, int p, int C, int& r0, int& r1,
                                          const T*& w0, const T*& w1) {
  if constexpr (KIND == QKV_ROPE) {
    const int hp = a.hd / 2;
    const int grp = p / hp, i = p - grp * hp;
    r0 = grp * a.hd + i;
    r1 = r0 + hp;
    const T* base;
    int rr;
    if (r0 < a.q_dim) { base = a.w_q; rr = r0; }
    else if (r0 < a.q_dim + a.kv_dim) { base = a.w_k; rr = r0 - a.q_dim; }
    else { base = a.w_v; rr = r0 - a.q_dim - a.kv_dim; }
    w0 = base + (size_t)rr * C;
    w1 = w0 + (size_t)hp * C;
  } else if constexpr (KIND == GATE_UP) {
    r0 = p;
    r1 = p;
    w0 = a.w_gate + (size_t)p * C;
    w1 = a.w_up + (size_t)p * C;
  } else {
    const T* W = (KIND == EH_PROJ) ? a.w_eh : (KIND == O_PROJ) ? a.w_o : (KIND == DOWN) ? a.w_down : a.lm_head;
    const int R = (KIND == LM_HEAD) ? a.V : a.H;
    r0 = 2 * p;
    r1 = (2 * p + 1 < R) ? 2 * p + 1 : -1;
    w0 = W + (size_t)r0 * C;
    w1 = (r1 >= 0) ? w0 + C : nullptr;
  }
}

// Block-wide sum of one value per thread (result broadcast).
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float t = (l < kWarps) ? red[l] : 0.0f;
  return warp_sum(t);
}

template <typename T>
__device__ __forceinline__ float load_act(const T* p, int i) {
  return Elem<T>::load1(p + i);
}

// Copy n values (fp32 or T) into dst (fp32), then scale by rsqrt(mean sq + eps) * w
// when w != nullptr.
template <typename T, typename S>
__device__ __forceinline__ void stage_row(float* dst, const S* src, int n, const T* w, float eps, float* red) {
  float ss = 0.0f;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    float v;
    if constexpr (sizeof(S) == 4) v = src[i];
    else v = Elem<T>::load1(reinterpret_cast<const T*>(src) + i);
    dst[i] = v;
    ss = fmaf(v, v, ss);
  }
  if (w == nullptr) return;
  const float tot = block_sum(ss, red);
  const float scale = rsqrtf(tot / (float)n + eps);
  for (int i = threadIdx.x; i < n; i += kThreads) dst[i] = dst[i] * scale * Elem<T>::load1(w + i);
}

template <typename T, int KIND>
__device__ void stage_inputs(const StepArgs<T>& a, float* xs, int C, int b0, int nb, float* red) {
  for (int j = 0; j < nb; ++j) {
    const int b = b0 + j;
    float* dst = xs + (size_t)j * C;
    if constexpr (KIND == EH_PROJ) {
      if (a.k == 1) {
        stage_row<T, T>(dst, a.hidden_in + (size_t)b * a.H, a.H, a.w_norm_h, a.eps, red);
        stage_row<T, T>(dst + a.H, a.embeds_in + (size_t)b * a.H, a.H, a.w_norm_e, a.eps, red);
      } else {
        stage_row<T, float>(dst, a.hid + (size_t)b * a.H, a.H, a.w_norm_h, a.eps, red);
        int id = a.chain_ids ? a.chain_ids[(size_t)b * (a.K - 1) + (a.k - 2)]
                             : a.draft_ids[(size_t)b * a.K + (a.k - 2)];
        if (id < 0 || id >= a.V) {
          if (threadIdx.x == 0) set_error(a.err, MTP_ERR_DEVICE_ARGS);
          id = 0;
        }
        stage_row<T, T>(dst + a.H, a.embed + (size_t)id * a.H, a.H, a.w_norm_e, a.eps, red);
      }
    } else if constexpr (KIND == QKV_ROPE) {
      stage_row<T, float>(dst, a.x + (size_t)b * a.H, a.H, a.w_norm_in, a.eps, red);
    } else if constexpr (KIND == O_PROJ) {
      stage_row<T, float>(dst, a.attn + (size_t)b * a.q_dim, a.q_dim, (const T*)nullptr, a.eps, red);
    } else if constexpr (KIND == GATE_UP) {
      stage_row<T, float>(dst, a.h1 + (size_t)b * a.H, a.H, a.w_norm_post, a.eps, red);
    } else if constexpr (KIND == DOWN) {
      stage_row<T, float>(dst, a.act + (size_t)b * a.F, a.F, (const T*)nullptr, a.eps, red);
    } else {
      stage_row<T, float>(dst, a.hid + (size_t)b * a.H, a.H, a.w_norm_f, a.eps, red);
    }
  }
  __syncthreads();
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

// Epilogue for one pair and one batch row (runs on lane 0).
template <typename T, int KIND>
__device__ __forceinline__ void epilogue(const StepArgs<T>& a, int b, int r0, int r1, float v0, float v1,
                                         unsigned long long& best) {
  if constexpr (KIND == EH_PROJ) {
    a.x[(size_t)b * a.H + r0] = v0;
    if (r1 >= 0) a.x[(size_t)b * a.H + r1] = v1;
  } else if constexpr (KIND == O_PROJ) {
    a.h1[(size_t)b * a.H + r0] = a.x[(size_t)b * a.H + r0] + v0;
    if (r1 >= 0) a.h1[(size_t)b * a.H + r1] = a.x[(size_t)b * a.H + r1] + v1;
  } else if constexpr (KIND == DOWN) {
    const float o0 = a.h1[(size_t)b * a.H + r0] + v0;
    a.hid[(size_t)b * a.H + r0] = o0;
    if (a.hidden_out && a.k == a.K) a.hidden_out[(size_t)b * a.H + r0] = o0;
    if (r1 >= 0) {
      const float o1 = a.h1[(size_t)b * a.H + r1] + v1;
      a.hid[(size_t)b * a.H + r1] = o1;
      if (a.hidden_out && a.k == a.K) a.hidden_out[(size_t)b * a.H + r1] = o1;
    }
  } else if constexpr (KIND == GATE_UP) {
    a.act[(size_t)b * a.F + r0] = silu(v0) * v1;
  } else if constexpr (KIND == LM_HEAD) {
    float* lg = a.logits ? a.logits + ((size_t)b * a.K + (a.k - 1)) * a.V : nullptr;
    if (lg) lg[r0] = v0;
    best = umax64(best, argmax_key(v0, (uint32_t)r0));
    if (r1 >= 0) {
      if (lg) lg[r1] = v1;
      best = umax64(best, argmax_key(v1, (uint32_t)r1));
    }
  } else {  // QKV_ROPE
    const int hp = a.hd / 2;
    const int grp = r0 / a.hd, i = r0 - grp * a.hd;
    const int pos = a.positions[b] + a.k - 1;
    if (pos < 0 || pos >= a.max_pos) {
      set_error(a.err, MTP_ERR_CAPACITY);
      return;
    }
    if (grp < a.n_q) {
      const float2 cs = a.rope[(size_t)pos * hp + i];
      float* qb = a.q + (size_t)b * a.q_dim;
      qb[r0] = v0 * cs.x - v1 * cs.y;
      qb[r1] = v1 * cs.x + v0 * cs.y;
      return;
    }
    if (__ldcg(a.req_bad + b) || a.pending[b] != a.k - 1) {
      set_error(a.err, MTP_ERR_DEVICE_ARGS);
      return;
    }
    const int slot = a.seq_len[b] + a.k - 1;
    const int bi = slot / a.bs, off = slot - bi * a.bs;
    int blk = (bi < a.max_blocks && slot >= 0) ? a.block_table[(size_t)b * a.max_blocks + bi] : -1;
    if (blk < 0 || blk >= a.num_blocks) {
      set_error(a.err, MTP_ERR_CAPACITY);
      return;
    }
    float o0 = v0, o1 = v1;
    T* pool;
    int g;
    if (grp < a.n_q + a.n_kv) {
      const float2 cs = a.rope[(size_t)pos * hp + i];
      o0 = v0 * cs.x - v1 * cs.y;
      o1 = v1 * cs.x + v0 * cs.y;
      pool = a.k_pool;
      g = grp - a.n_q;
    } else {
      pool = a.v_pool;
      g = grp - a.n_q - a.n_kv;
    }
    T* dst = pool + (((size_t)blk * a.n_kv + g) * a.bs + off) * a.hd;
    Elem<T>::store1(dst + i, o0);
    Elem<T>::store1(dst + i + hp, o1);
  }
}

template <typename T, int KIND, int NB>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const StepArgs<T> a) {
  extern __shared__ __align__(16) float xs[];
  __shared__ float red[kWarps];
  __shared__ unsigned long long cta_best[kWarps][NB];
  __shared__ int am_last;

  pdl_trigger();
  const int C = gemv_cols(a, KIND);
  const int P = gemv_pairs(a, KIND);
  const int G = gridDim.x;
  const int p_begin = (int)(((long long)blockIdx.x * P) / G);
  const int p_end = (int)(((long long)(blockIdx.x + 1) * P) / G);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int VPE = Elem<T>::kPerVec;
  const int nvec = C / VPE;

  // Prefetch the head of this warp's first pair while the previous kernel drains.
  if (p_begin + warp < p_end) {
    int r0, r1;
    const T *w0, *w1;
    pair_rows<T, KIND>(a, p_begin + warp, C, r0, r1, w0, w1);
    const int bytes = C * (int)sizeof(T);
    for (int off = lane * 128; off < bytes && off < 8192; off += 32 * 128) {
      prefetch_l2(reinterpret_cast<const char*>(w0) + off);
      if (w1) prefetch_l2(reinterpret_cast<const char*>(w1) + off);
    }
  }
  pdl_wait();
  if (KIND == EH_PROJ && a.k == 1 && blockIdx.x == 0)
    for (int b = threadIdx.x; b < a.B; b += kThreads) a.req_bad[b] = (a.pending[b] != 0);

  for (int b0 = 0; b0 < a.B; b0 += NB) {
    const int nb = min(NB, a.B - b0);
    if (b0 > 0) __syncthreads();
    stage_inputs<T, KIND>(a, xs, C, b0, nb, red);

    unsigned long long best[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) best[j] = 0ull;

    for (int p = p_begin + warp; p < p_end; p += kWarps) {
      int r0, r1;
      const T *w0, *w1;
      pair_rows<T, KIND>(a, p, C, r0, r1, w0, w1);
      float acc0[NB], acc1[NB];
#pragma unroll
      for (int j = 0; j < NB; ++j) acc0[j] = acc1[j] = 0.0f;
      for (int v0 = lane; v0 < nvec; v0 += 32 * kUnroll) {
        uint4 wa[kUnroll], wb[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int idx = v0 + u * 32;
          if (idx < nvec) {
            wa[u] = ld_stream(w0 + (size_t)idx * VPE);
            wb[u] = w1 ? ld_stream(w1 + (size_t)idx * VPE) : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int idx = v0 + u * 32;
          if (idx < nvec) {
#pragma unroll
            for (int j = 0; j < NB; ++j) {
              if (j < nb) {
                const float* xp = xs + (size_t)j * C + (size_t)idx * VPE;
                acc0[j] += dot_vec<T>(wa[u], xp);
                acc1[j] += dot_vec<T>(wb[u], xp);
              }
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        acc0[j] = warp_sum(acc0[j]);
        acc1[j] = warp_sum(acc1[j]);
      }
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < NB; ++j)
          if (j < nb) epilogue<T, KIND>(a, b0 + j, r0, r1, acc0[j], acc1[j], best[j]);
      }
    }

    if constexpr (KIND == LM_HEAD) {
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < NB; ++j) cta_best[warp][j] = best[j];
      }
      __syncthreads();
      if (threadIdx.x < nb) {
        unsigned long long m = 0ull;
        for (int w = 0; w < kWarps; ++w) m = umax64(m, cta_best[w][threadIdx.x]);
        if (m) atomicMax(a.lm_keys + b0 + threadIdx.x, m);
      }
    }
  }

  if constexpr (KIND == LM_HEAD) {
    // The last CTA to finish turns the keys into draft ids and resets them.
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const int prev = atomicAdd(a.lm_cnt, 1);
      am_last = (prev == (int)gridDim.x - 1);
    }
    __syncthreads();
    if (am_last) {
      __threadfence();
      for (int b = threadIdx.x; b < a.B; b += kThreads) {
        const unsigned long long key = atomicExch(a.lm_keys + b, 0ull);
        a.draft_ids[(size_t)b * a.K + (a.k - 1)] = (int32_t)key_index(key);
        if (!__ldcg(a.req_bad + b)) a.pending[b] = a.k;
      }
      if (threadIdx.x == 0) atomicExch(a.lm_cnt, 0);
    }
  }
}

// ------------------------------------------------- TMA-streamed variant
//
// Same work split and epilogues as gemv_kernel, for batches of at most 4:
// one CTA per SM; warp 0 is a producer that streams this CTA's row pairs
// into a ring of shared-memory stages with one-dimensional bulk (TMA) copies
// (one copy per contiguous pair, two for rotary or gate/up pairs), completing
// on per-stage mbarriers; it starts before the dependency wait, so the ring
// (about 200 KB per SM) fills while the previous kernel drains.  Warps 1..8
// stage the normalised input, then consume pairs round-robin from shared
// memory and release each stage as soon as its values are in registers.
// The stage count is a multiple of the number of consuming warps, and pair
// it goes to stage it % stages and warp it % consumers (see below).

constexpr int kTmaConsumers = 8;
constexpr int kTmaThreads = 32 * (kTmaConsumers + 1);
constexpr int kMaxTmaStages = 16;
constexpr uint32_t kGemvWaitLimit = 1u << 24;

__device__ __forceinline__ void cons_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Eight consecutive values of an fp32 (activations, L2 only) or T row.
template <typename T, typename S>
__device__ __forceinline__ void load8_row(const S* p, float (&x)[8]) {
  if constexpr (sizeof(S) == 4) {
    const float4 t0 = __ldcg(reinterpret_cast<const float4*>(p));
    const float4 t1 = __ldcg(reinterpret_cast<const float4*>(p) + 1);
    x[0] = t0.x; x[1] = t0.y; x[2] = t0.z; x[3] = t0.w; x[4] = t1.x; x[5] = t1.y; x[6] = t1.z; x[7] = t1.w;
  } else {
    const uint4 t = __ldg(reinterpret_cast<const uint4*>(p));
    x[0] = bf16_lo(t.x); x[1] = bf16_hi(t.x); x[2] = bf16_lo(t.y); x[3] = bf16_hi(t.y);
    x[4] = bf16_lo(t.z); x[5] = bf16_hi(t.z); x[6] = bf16_lo(t.w); x[7] = bf16_hi(t.w);
  }
}

// Copy n values (fp32 or T; n % 8 == 0) into dst (fp32) times the norm
// weight w (if any); returns this thread's sum of squares of the raw
// values.  Source and weight loads are independent and vectorised, so a
// 4096-wide row costs each consumer thread two groups: about one L2 round
// trip.
template <typename T, typename S>
__device__ __forceinline__ float cons_stage_raw(float* dst, const S* src, int n, const T* w) {
  const int ct = threadIdx.x - 32;
  float ss = 0.0f;
#pragma unroll 2
  for (int i8 = ct; i8 < (n >> 3); i8 += 256) {
    float x[8], wv[8];
    load8_row<T, S>(src + (size_t)i8 * 8, x);
    if (w) load8_row<T, T>(w + (size_t)i8 * 8, wv);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      ss = fmaf(x[e], x[e], ss);
      if (w) x[e] *= wv[e];
    }
    float4* d = reinterpret_cast<float4*>(dst + (size_t)i8 * 8);
    d[0] = make_float4(x[0], x[1], x[2], x[3]);
    d[1] = make_float4(x[4], x[5], x[6], x[7]);
  }
  return ss;
}

// Stage the normalised input row(s) of all nb requests: one pass that stores
// x * w and sums x^2 for every vector, one block reduction for all of them,
// then the scalar RMS factors applied in shared memory.
template <typename T, int KIND>
__device__ void cons_stage_inputs(const StepArgs<T>& a, float* xs, int C, int nb, float* red) {
  constexpr bool kNorm = (KIND != O_PROJ && KIND != DOWN);
  float ss[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) ss[i] = 0.0f;
  for (int b = 0; b < nb; ++b) {
    float* dst = xs + (size_t)b * C;
    float s0 = 0.0f, s1 = 0.0f;
    if constexpr (KIND == EH_PROJ) {
      if (a.k == 1) {
        s0 = cons_stage_raw<T, T>(dst, a.hidden_in + (size_t)b * a.H, a.H, a.w_norm_h);
        s1 = cons_stage_raw<T, T>(dst + a.H, a.embeds_in + (size_t)b * a.H, a.H, a.w_norm_e);
      } else {
        int id = a.chain_ids ? a.chain_ids[(size_t)b * (a.K - 1) + (a.k - 2)]
                             : a.draft_ids[(size_t)b * a.K + (a.k - 2)];
        s0 = cons_stage_raw<T, float>(dst, a.hid + (size_t)b * a.H, a.H, a.w_norm_h);
        if (id < 0 || id >= a.V) {
          if (threadIdx.x == 32) set_error(a.err, MTP_ERR_DEVICE_ARGS);
          id = 0;
        }
        s1 = cons_stage_raw<T, T>(dst + a.H, a.embed + (size_t)id * a.H, a.H, a.w_norm_e);
      }
    } else if constexpr (KIND == QKV_ROPE) {
      s0 = cons_stage_raw<T, float>(dst, a.x + (size_t)b * a.H, a.H, a.w_norm_in);
    } else if constexpr (KIND == O_PROJ) {
      cons_stage_raw<T, float>(dst, a.attn + (size_t)b * a.q_dim, a.q_dim, (const T*)nullptr);
    } else if constexpr (KIND == GATE_UP) {
      s0 = cons_stage_raw<T, float>(dst, a.h1 + (size_t)b * a.H, a.H, a.w_norm_post);
    } else if constexpr (KIND == DOWN) {
      cons_stage_raw<T, float>(dst, a.act + (size_t)b * a.F, a.F, (const T*)nullptr);
    } else {
      s0 = cons_stage_raw<T, float>(dst, a.hid + (size_t)b * a.H, a.H, a.w_norm_f);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j == b) {
        ss[2 * j] = s0;
        ss[2 * j + 1] = s1;
      }
  }
  if constexpr (kNorm) {
    const int cw = (threadIdx.x >> 5) - 1, l = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float t = warp_sum(ss[i]);
      if (l == 0 && i < 2 * nb) red[cw * 8 + i] = t;
    }
    cons_bar();
    const int ct = threadIdx.x - 32;
    const int nvec = (KIND == EH_PROJ) ? 2 : 1;
    for (int b = 0; b < nb; ++b)
      for (int v = 0; v < nvec; ++v) {
        float t = 0.0f;
        for (int w = 0; w < kTmaConsumers; ++w) t += red[w * 8 + 2 * b + v];
        const float sc = rsqrtf(t / (float)a.H + a.eps);
        float* dst = xs + (size_t)b * C + (size_t)v * a.H;
        for (int i = ct; i < a.H; i += 256) dst[i] *= sc;
      }
  }
  cons_bar();
}

template <typename T, int KIND, int NB>
__global__ void __launch_bounds__(kTmaThreads, 1) gemv_tma_kernel(const StepArgs<T> a, int stages, int consumers) {
  extern __shared__ __align__(128) unsigned char gsm[];
  __shared__ __align__(8) uint64_t full_bar[kMaxTmaStages], empty_bar[kMaxTmaStages];
  __shared__ float red[kTmaConsumers * 8];
  __shared__ unsigned long long cta_best[kTmaConsumers][NB];
  __shared__ int am_last;

  pdl_trigger();
  const int C = gemv_cols(a, KIND);
  const int P = gemv_pairs(a, KIND);
  const int G = gridDim.x;
  const int p_begin = (int)(((long long)blockIdx.x * P) / G);
  const int p_end = (int)(((long long)(blockIdx.x + 1) * P) / G);
  const int n = p_end - p_begin;
  const uint32_t row_bytes = (uint32_t)C * sizeof(T);
  const uint32_t stage_stride = (2 * row_bytes + 127) & ~127u;
  float* xs = reinterpret_cast<float*>(gsm + (size_t)stages * stage_stride);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int VPE = Elem<T>::kPerVec;
  const int nvec = C / VPE;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();  // weights are read once per step
      for (int it = 0; it < n; ++it) {
        const int s = it % stages;
        if (!mbar_wait_bounded(&empty_bar[s], (uint32_t)(((it / stages) & 1) ^ 1), kGemvWaitLimit)) {
          set_error(a.err, MTP_ERR_TIMEOUT);
          break;
        }
        int r0, r1;
        const T *w0, *w1;
        pair_rows<T, KIND>(a, p_begin + it, C, r0, r1, w0, w1);
        unsigned char* st = gsm + (size_t)s * stage_stride;
        if (w1 == w0 + C) {
          mbar_expect_tx(&full_bar[s], 2 * row_bytes);
          bulk_g2s_hint(st, w0, 2 * row_bytes, &full_bar[s], pol);
        } else if (w1) {
          mbar_expect_tx(&full_bar[s], 2 * row_bytes);
          bulk_g2s_hint(st, w0, row_bytes, &full_bar[s], pol);
          bulk_g2s_hint(st + row_bytes, w1, row_bytes, &full_bar[s], pol);
        } else {
          mbar_expect_tx(&full_bar[s], row_bytes);
          bulk_g2s_hint(st, w0, row_bytes, &full_bar[s], pol);
        }
      }
    }
    return;
  }

  // consumers
  pdl_wait();
  if (KIND == EH_PROJ && a.k == 1 && blockIdx.x == 0)
    for (int b = threadIdx.x - 32; b < a.B; b += 32 * kTmaConsumers) a.req_bad[b] = (a.pending[b] != 0);
  const int nb = a.B;  // launched only for B <= NB
  cons_stage_inputs<T, KIND>(a, xs, C, nb, red);
  const int cw = warp - 1;
  // Full-barrier waits are by phase parity, so a warp may wait on a stage
  // only after the stage's previous fill has landed.  `stages` is a multiple
  // of the number of consuming warps A: pair it uses stage it % stages and
  // warp it % A, so consecutive uses of a stage belong to the same warp,
  // which consumed (hence saw land) the previous fill itself.
  const int active = consumers;
  unsigned long long best[NB];
#pragma unroll
  for (int j = 0; j < NB; ++j) best[j] = 0ull;
  for (int it = cw; cw < active && it < n; it += active) {
    const int s = it % stages;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full_bar[s], (uint32_t)((it / stages) & 1), kGemvWaitLimit))) {
      if (lane == 0) set_error(a.err, MTP_ERR_TIMEOUT);
      break;
    }
    int r0, r1;
    const T *w0, *w1;
    pair_rows<T, KIND>(a, p_begin + it, C, r0, r1, w0, w1);
    const T* s0 = reinterpret_cast<const T*>(gsm + (size_t)s * stage_stride);
    const T* s1 = s0 + C;
    const bool two = (w1 != nullptr);
    float acc0[NB], acc1[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) acc0[j] = acc1[j] = 0.0f;
#pragma unroll 4
    for (int v = lane; v < nvec; v += 32) {
      const uint4 wa = *reinterpret_cast<const uint4*>(s0 + (size_t)v * VPE);
      const uint4 wb = two ? *reinterpret_cast<const uint4*>(s1 + (size_t)v * VPE) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        if (j < nb) {
          const float* xp = xs + (size_t)j * C + (size_t)v * VPE;
          acc0[j] += dot_vec<T>(wa, xp);
          acc1[j] += dot_vec<T>(wb, xp);
        }
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty_bar[s])) : "memory");
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      acc0[j] = warp_sum(acc0[j]);
      acc1[j] = warp_sum(acc1[j]);
    }
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < NB; ++j)
        if (j < nb) epilogue<T, KIND>(a, j, r0, r1, acc0[j], acc1[j], best[j]);
    }
  }

  if constexpr (KIND == LM_HEAD) {
    if (lane == 0)
#pragma unroll
      for (int j = 0; j < NB; ++j) cta_best[cw][j] = best[j];
    cons_bar();
    const int ct = threadIdx.x - 32;
    if (ct < nb) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kTmaConsumers; ++w) m = umax64(m, cta_best[w][ct]);
      if (m) atomicMax(a.lm_keys + ct, m);
      __threadfence();
    }
    cons_bar();
    if (ct == 0) {
      __threadfence();
      am_last = (atomicAdd(a.lm_cnt, 1) == (int)gridDim.x - 1);
    }
    cons_bar();
    if (am_last) {
      __threadfence();
      for (int b = ct; b < a.B; b += 256) {
        const unsigned long long key = atomicExch(a.lm_keys + b, 0ull);
        a.draft_ids[(size_t)b * a.K + (a.k - 1)] = (int32_t)key_index(key);
        if (!__ldcg(a.req_bad + b)) a.pending[b] = a.k;
      }
      if (ct == 0) atomicExch(a.lm_cnt, 0);
    }
  }
}

template <typename T, int KIND>
static cudaError_t launch_kind(mtp_ctx* ctx, cudaStream_t s, const StepArgs<T>& a) {
  const int C = (KIND == EH_PROJ) ? 2 * a.H : (KIND == O_PROJ) ? a.q_dim : (KIND == DOWN) ? a.F : a.H;
  const int P = (KIND == EH_PROJ || KIND == O_PROJ || KIND == DOWN) ? a.H / 2
                : (KIND == QKV_ROPE) ? (a.q_dim + 2 * a.kv_dim) / 2
                : (KIND == GATE_UP) ? a.F
                                    : (a.V + 1) / 2;
  int grid = min((P + 1) / 2, 2 * ctx->num_sms);
  if (grid < 1) grid = 1;
  const size_t row_bytes = (size_t)C * sizeof(float);
  int nb = 4;
  while (nb > 1 && (nb * row_bytes > 100 * 1024 || nb > a.B)) nb >>= 1;
  const size_t smem = nb * row_bytes;
  const int kid = (KIND == EH_PROJ) ? MTP_KERNEL_EH_PROJ : (KIND == QKV_ROPE) ? MTP_KERNEL_QKV_ROPE
                  : (KIND == O_PROJ) ? MTP_KERNEL_O_PROJ : (KIND == GATE_UP) ? MTP_KERNEL_GATE_UP
                  : (KIND == DOWN) ? MTP_KERNEL_DOWN : MTP_KERNEL_LM_HEAD;
  cudaError_t e;
  prof_before(ctx, kid, s);
  // TMA-streamed variant for B <= 4
  {
    const int nbt = a.B <= 1 ? 1 : a.B <= 2 ? 2 : 4;
    const size_t stage_stride = ((size_t)2 * C * sizeof(T) + 127) & ~(size_t)127;
    const size_t xs_bytes = (size_t)nbt * C * sizeof(float);
    const size_t budget = (size_t)ctx->gemv_budget_kb[KIND] * 1024;
    int max_stages = xs_bytes < budget ? (int)((budget - xs_bytes) / stage_stride) : 0;
    if (max_stages > kMaxTmaStages) max_stages = kMaxTmaStages;
    // stages = consumers * k: pick the consumer count (4..8) that keeps the most stages
    int consumers = 0, stages = 0;
    for (int cw = kTmaConsumers; cw >= 1; --cw) {
      const int st = cw * (max_stages / cw);
      if (st > stages || (st == stages && st > 0 && cw > consumers && cw <= max_stages)) {
        stages = st;
        consumers = cw;
      }
      if (cw <= 4 && stages > 0) break;
    }
    if (((ctx->gemv_stream_mask >> KIND) & 1) && a.B <= 4 && stages >= 2 && consumers >= 2) {
      const size_t smem_t = stages * stage_stride + xs_bytes;
      const int gridt = min(ctx->num_sms, P);
      if (nbt == 1) {
        auto kern = gemv_tma_kernel<T, KIND, 1>;
        ensure_smem((const void*)kern, smem_t);
        e = launch_pdl(kern, dim3(gridt), dim3(kTmaThreads), smem_t, s, a, stages, consumers);
      } else if (nbt == 2) {
        auto kern = gemv_tma_kernel<T, KIND, 2>;
        ensure_smem((const void*)kern, smem_t);
        e = launch_pdl(kern, dim3(gridt), dim3(kTmaThreads), smem_t, s, a, stages, consumers);
      } else {
        auto kern = gemv_tma_kernel<T, KIND, 4>;
        ensure_smem((const void*)kern, smem_t);
        e = launch_pdl(kern, dim3(gridt), dim3(kTmaThreads), smem_t, s, a, stages, consumers);
      }
      prof_after(ctx, kid, s);
      ctx->launches++;
      return e;
    }
  }
  if (nb == 4) {
    auto kern = gemv_kernel<T, KIND, 4>;
    ensure_smem((const void*)kern, smem);
    e = launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a);
  } else if (nb == 2) {
    auto kern = gemv_kernel<T, KIND, 2>;
    ensure_smem((const void*)kern, smem);
    e = launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a);
  } else {
    auto kern = gemv_kernel<T, KIND, 1>;
    ensure_smem((const void*)kern, smem);
    e = launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a);
  }
  prof_after(ctx, kid, s);
  ctx->launches++;
  return e;
}

template <typename T>
static cudaError_t draft_step_t(mtp_ctx* ctx, cudaStream_t s, int B, int k, int K, const void* hidden,
                                const void* embeds, const int32_t* positions, const mtp_kv* kv,
                                const int32_t* chain_ids, int32_t* draft_ids, float* logits, float* hidden_out) {
  const mtp_config& c = ctx->cfg;
  StepArgs<T> a;
  a.B = B; a.H = c.hidden; a.q_dim = ctx->q_dim; a.kv_dim = ctx->kv_dim; a.F = c.ffn; a.V = c.vocab;
  a.n_q = c.n_q_heads; a.n_kv = c.n_kv_heads; a.hd = c.head_dim; a.bs = c.block_size; a.eps = c.eps;
  a.k = k; a.K = K; a.max_pos = c.max_pos; a.num_blocks = kv->num_blocks; a.max_blocks = kv->max_blocks;
  const mtp_weights& w = ctx->w;
  a.w_norm_h = (const T*)w.w_norm_h; a.w_norm_e = (const T*)w.w_norm_e; a.w_eh = (const T*)w.w_eh;
  a.w_norm_in = (const T*)w.w_norm_in; a.w_q = (const T*)w.w_q; a.w_k = (const T*)w.w_k; a.w_v = (const T*)w.w_v;
  a.w_o = (const T*)w.w_o; a.w_norm_post = (const T*)w.w_norm_post; a.w_gate = (const T*)w.w_gate;
  a.w_up = (const T*)w.w_up; a.w_down = (const T*)w.w_down; a.w_norm_f = (const T*)w.w_norm_f;
  a.embed = (const T*)w.embed; a.lm_head = (const T*)w.lm_head;
  a.hidden_in = (const T*)hidden; a.embeds_in = (const T*)embeds; a.positions = positions;
  a.chain_ids = chain_ids; a.draft_ids = draft_ids; a.logits = logits; a.hidden_out = hidden_out;
  a.k_pool = (T*)kv->k_pool; a.v_pool = (T*)kv->v_pool; a.block_table = kv->block_table;
  a.seq_len = kv->seq_len; a.pending = kv->pending;
  a.hid = ctx->hid; a.x = ctx->x; a.q = ctx->q; a.attn = ctx->attn; a.h1 = ctx->h1; a.act = ctx->act;
  a.lm_keys = ctx->lm_keys; a.lm_cnt = ctx->lm_cnt; a.err = ctx->err; a.rope = ctx->rope;
  a.req_bad = ctx->req_bad;

  cudaError_t e;
  if ((e = launch_kind<T, EH_PROJ>(ctx, s, a)) != cudaSuccess) return e;
  if ((e = launch_kind<T, QKV_ROPE>(ctx, s, a)) != cudaSuccess) return e;
  if ((e = launch_attention(ctx, s, B, k, kv)) != cudaSuccess) return e;
  if ((e = launch_kind<T, O_PROJ>(ctx, s, a)) != cudaSuccess) return e;
  if ((e = launch_kind<T, GATE_UP>(ctx, s, a)) != cudaSuccess) return e;
  if ((e = launch_kind<T, DOWN>(ctx, s, a)) != cudaSuccess) return e;
  return launch_kind<T, LM_HEAD>(ctx, s, a);
}

cudaError_t launch_draft_step(mtp_ctx* ctx, cudaStream_t s, int B, int k, int K, const void* hidden,
                              const void* embeds, const int32_t* positions, const mtp_kv* kv,
                              const int32_t* chain_ids, int32_t* draft_ids, float* logits, float* hidden_out) {
  if (ctx->cfg.dtype == MTP_DTYPE_BF16)
    return draft_step_t<uint16_t>(ctx, s, B, k, K, hidden, embeds, positions, kv, chain_ids, draft_ids, logits,
                                  hidden_out);
  return draft_step_t<float>(ctx, s, B, k, K, hidden, embeds, positions, kv, chain_ids, draft_ids, logits,
                             hidden_out);
}

}  // namespace mtp
