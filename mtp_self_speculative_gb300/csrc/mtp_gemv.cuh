// Shared pieces of the small-batch projection kernels (bf16/fp32 streamed
// GEMV in mtp_gemv.cu, quantized GEMV in mtp_quant.cu): the step arguments,
// the row-pair mapping of every projection kind, input staging and the
// epilogues ("MTP (Multi-Token Prediction)", "Architecture").
#pragma once

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
  // Streamed LM head, weighted ranges (null: equal ranges): packed (ticket,
  // first pair) claim counter of this launch, per-SM streaming rates
  // (pairs per ns, 0 = not yet measured) over lm_nsm SM ids.
  unsigned long long* lm_tick;
  float* lm_rate;
  int lm_nsm;
  // Deferred argmax (one request, every step but the last): the streamed LM
  // head stores each CTA's best (value, id) key in cta_keys[CTA] and stops
  // there (defer_out); the next step's eh_proj reduces the keys_n keys
  // itself (keys_in), writes the draft id, advances pending and zeroes the
  // LM launch's claim counter keys_tick.
  unsigned long long* cta_keys;
  unsigned long long* keys_tick;
  int defer_out, keys_in, keys_n;
  int* err;
  int* req_bad;
  const float2* rope;
  // Quantized head (null when dense): fragment-ordered tile streams per
  // GemvKind (INT4 projections, INT8 LM head), the INT8 embedding [V, H] with
  // its fp16 row scales [V] (row gather), the LM head's row scales and the
  // power-of-two scale of the LM head's fp16 input operand.
  const uint8_t* qt[6];
  const int8_t* q8;
  const uint16_t* s8;
  const uint16_t* s8_lm;
  float lm_sigma;
};

// Weighted ranges of the LM heads.  The SMs of a GPU stream at rates that
// differ by up to about 10% and stay the same from launch to launch (the
// rate follows the SM, not the data), so equal ranges leave the fastest SMs
// idle at the end.  Each CTA sizes its range of `total` units by its SM's
// measured rate (weight rows per ns, a running average shared by the LM-head
// kernels; SMs not yet measured count as the mean) and takes it with one atomic on a packed (ticket, next unit)
// counter: ranges are contiguous in ticket order and the last of the G
// tickets takes whatever remains, so the units are covered exactly once
// wherever the CTAs land.  Called by one whole warp; lane 0 writes
// range[0..1].
__device__ __forceinline__ void lm_weighted_range(const float* rate, int nsm, unsigned long long* tick, int total,
                                                  int G, int lane, int* range) {
  unsigned smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  float sum = 0.0f, known = 0.0f;
  for (int i = lane; i < nsm; i += 32) {
    const float r = __ldcg(rate + i);
    sum += r;
    known += (r > 0.0f) ? 1.0f : 0.0f;
  }
  sum = warp_sum(sum);
  known = warp_sum(known);
  if (lane == 0) {
    const float mean = known > 0.0f ? sum / known : 1.0f;
    const float all = known > 0.0f ? sum + ((float)nsm - known) * mean : (float)nsm;
    float mine = (smid < (unsigned)nsm) ? __ldcg(rate + smid) : 0.0f;
    if (!(mine > 0.0f)) mine = mean;
    int units = (int)((double)total * (double)mine / (double)all + 0.5);
    if (units < 1) units = 1;
    const unsigned long long old = atomicAdd(tick, (1ull << 32) | (unsigned long long)units);
    const int t = (int)(old >> 32);
    const long long st = (long long)(old & 0xffffffffull);
    const long long en = (t >= G - 1) ? (long long)total : st + units;
    range[0] = (int)(st < total ? st : total);
    range[1] = (int)(en < total ? en : total);
  }
}

// This SM's running rate estimate (0 if none), read early so that folding
// the CTA's own rate in at the end (lm_rate_store) is a plain store.
__device__ __forceinline__ float lm_rate_peek(const float* rate, int nsm) {
  unsigned smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  return smid < (unsigned)nsm ? __ldcg(rate + smid) : 0.0f;
}

// Fold this CTA's rate (`rows` weight rows since t0) into its SM's running
// estimate `old` (from lm_rate_peek).
__device__ __forceinline__ void lm_rate_store(float* rate, int nsm, int rows, unsigned long long t0, float old) {
  const unsigned long long dt = globaltimer_ns() - t0;
  unsigned smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  if (rows > 0 && dt > 0 && smid < (unsigned)nsm) {
    const float r = (float)rows / (float)dt;
    rate[smid] = old > 0.0f ? 0.75f * old + 0.25f * r : r;
  }
}

// CTA arrival with release (orders this CTA's earlier argmax updates) and
// acquire (the last CTA's later reads see every CTA's updates); returns the
// count before this arrival.
__device__ __forceinline__ int lm_arrive(int* cnt) {
  int prev;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(cnt) : "memory");
  return prev;
}

// LM head of 2..4 requests through mma.sync on whole staged rows
// (csrc/mtp_lm_rows.cu).
bool lm_rows_supported(const mtp_ctx* ctx, int B);
cudaError_t launch_lm_rows(mtp_ctx* ctx, cudaStream_t s, const StepArgs<uint16_t>& a);

// The short projections of 2..4 requests through mma.sync on staged row
// chunks (csrc/mtp_rows_proj.cu).
bool rows_proj_supported(const mtp_ctx* ctx, int kind, int B);
cudaError_t launch_rows_proj(mtp_ctx* ctx, cudaStream_t s, int kind, const StepArgs<uint16_t>& a);

// Source matrices of the quantized projections (canonical quantized copies).
enum QMat { QM_EH = 0, QM_Q = 1, QM_K = 2, QM_V = 3, QM_O = 4, QM_GATE = 5, QM_UP = 6, QM_DOWN = 7 };

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

// Rows per streamed unit: one for the wide-row kinds (eh_proj reads 2H
// columns, down F), so that a unit stays at 16-24 KB and the ring keeps
// enough stages; two (a "pair") otherwise.
__host__ __device__ constexpr int gemv_unit_rows(int kind) { return (kind == EH_PROJ || kind == DOWN) ? 1 : 2; }

// Number of units of a kind.
template <typename T>
__device__ __forceinline__ int gemv_pairs(const StepArgs<T>& a, int kind) {
  switch (kind) {
    case EH_PROJ: return a.H;
    case QKV_ROPE: return (a.q_dim + 2 * a.kv_dim) / 2;
    case O_PROJ: return a.H / 2;
    case GATE_UP: return a.F;
    case DOWN: return a.H;
    default: return (a.V + 1) / 2;
  }
}

// Rows (r0, r1) of unit p and their weight pointers.  r1 < 0: no second row.
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
  } else if constexpr (gemv_unit_rows(KIND) == 1) {
    r0 = p;
    r1 = -1;
    w0 = ((KIND == EH_PROJ) ? a.w_eh : a.w_down) + (size_t)p * C;
    w1 = nullptr;
  } else {
    const T* W = (KIND == O_PROJ) ? a.w_o : a.lm_head;
    const int R = (KIND == LM_HEAD) ? a.V : a.H;
    r0 = 2 * p;
    r1 = (2 * p + 1 < R) ? 2 * p + 1 : -1;
    w0 = W + (size_t)r0 * C;
    w1 = (r1 >= 0) ? w0 + C : nullptr;
  }
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + __expf(-g)); }

// Epilogue for one pair and one batch row (runs on lane 0).
template <typename T, int KIND>
__device__ __forceinline__ void epilogue(const StepArgs<T>& a, int b, int r0, int r1, float v0, float v1,
                                         unsigned long long& best) {
  const long long nBH = (long long)a.B * a.H;
  if constexpr (KIND == EH_PROJ) {
    MTP_STORE(a.err, a.x, (size_t)b * a.H + r0, nBH, v0);
    if (r1 >= 0) MTP_STORE(a.err, a.x, (size_t)b * a.H + r1, nBH, v1);
  } else if constexpr (KIND == O_PROJ) {
    MTP_STORE(a.err, a.h1, (size_t)b * a.H + r0, nBH, a.x[(size_t)b * a.H + r0] + v0);
    if (r1 >= 0) MTP_STORE(a.err, a.h1, (size_t)b * a.H + r1, nBH, a.x[(size_t)b * a.H + r1] + v1);
  } else if constexpr (KIND == DOWN) {
    const float o0 = a.h1[(size_t)b * a.H + r0] + v0;
    MTP_STORE(a.err, a.hid, (size_t)b * a.H + r0, nBH, o0);
    if (a.hidden_out && a.k == a.K) MTP_STORE(a.err, a.hidden_out, (size_t)b * a.H + r0, nBH, o0);
    if (r1 >= 0) {
      const float o1 = a.h1[(size_t)b * a.H + r1] + v1;
      MTP_STORE(a.err, a.hid, (size_t)b * a.H + r1, nBH, o1);
      if (a.hidden_out && a.k == a.K) MTP_STORE(a.err, a.hidden_out, (size_t)b * a.H + r1, nBH, o1);
    }
  } else if constexpr (KIND == GATE_UP) {
    MTP_STORE(a.err, a.act, (size_t)b * a.F + r0, (long long)a.B * a.F, silu(v0) * v1);
  } else if constexpr (KIND == LM_HEAD) {
    const long long row = ((long long)b * a.K + (a.k - 1)) * a.V;
    const long long nL = (long long)a.B * a.K * a.V;
    if (a.logits) MTP_STORE(a.err, a.logits, row + r0, nL, v0);
    best = umax64(best, argmax_key(v0, (uint32_t)r0));
    if (r1 >= 0) {
      if (a.logits) MTP_STORE(a.err, a.logits, row + r1, nL, v1);
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
      const long long nQ = (long long)a.B * a.q_dim;
      MTP_STORE(a.err, a.q, (size_t)b * a.q_dim + r0, nQ, v0 * cs.x - v1 * cs.y);
      MTP_STORE(a.err, a.q, (size_t)b * a.q_dim + r1, nQ, v1 * cs.x + v0 * cs.y);
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
    const long long e = (((long long)blk * a.n_kv + g) * a.bs + off) * a.hd + i;
    const long long nP = (long long)a.num_blocks * a.n_kv * a.bs * a.hd;
    if (MTP_IN_BOUNDS(a.err, e, nP)) Elem<T>::store1(pool + e, o0);
    if (MTP_IN_BOUNDS(a.err, e + hp, nP)) Elem<T>::store1(pool + e + hp, o1);
  }
}

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

// Layout of a staged input row (fp32, C values) in shared memory.  A
// consumer lane takes 16-byte weight vectors v = lane, lane + 32, ... and
// needs the vector's activations: 8 floats for bf16 weights.  Stored plainly
// they sit 32 bytes apart from lane to lane, so each 16-byte load of a warp
// touches every bank twice.  bf16 rows are therefore split in two planes:
// floats 0..3 of vector v at [4v], floats 4..7 at [C/2 + 4v], and each load
// of a warp reads 512 contiguous bytes.  fp32 weights (4 per vector) keep
// the plain layout.
template <typename T>
__device__ __forceinline__ int xs_index(int i, int C) {
  if constexpr (sizeof(T) == 2) return ((i & 7) >> 2) * (C >> 1) + ((i >> 3) << 2) + (i & 3);
  else return i;
}

// Dot product of one weight vector with its staged activations (same
// operation order as dot_vec).
template <typename T>
__device__ __forceinline__ float dot_vec_xs(const uint4& w, const float* row, int v, int C) {
  if constexpr (sizeof(T) == 2) {
    const float4 a = *reinterpret_cast<const float4*>(row + 4 * v);
    const float4 b = *reinterpret_cast<const float4*>(row + (C >> 1) + 4 * v);
    float s = bf16_lo(w.x) * a.x;
    s = fmaf(bf16_hi(w.x), a.y, s);
    s = fmaf(bf16_lo(w.y), a.z, s);
    s = fmaf(bf16_hi(w.y), a.w, s);
    s = fmaf(bf16_lo(w.z), b.x, s);
    s = fmaf(bf16_hi(w.z), b.y, s);
    s = fmaf(bf16_lo(w.w), b.z, s);
    s = fmaf(bf16_hi(w.w), b.w, s);
    return s;
  } else {
    return dot_vec<T>(w, row + 4 * v);
  }
}

// Copy n values (fp32 or T; n % 8 == 0) into elements [e0, e0 + n) of the
// staged row `row` (C values, layout above) times the norm weight w (if
// any); returns this thread's sum of squares of the raw values.  Source and
// weight loads are independent and vectorised, so a 4096-wide row costs each
// consumer thread two groups: about one L2 round trip.
template <typename T, typename S>
__device__ __forceinline__ float cons_stage_raw(float* row, int C, int e0, const S* src, int n, const T* w) {
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
    const int e = e0 + i8 * 8;
    float4* d0 = reinterpret_cast<float4*>(row + xs_index<T>(e, C));
    float4* d1 = reinterpret_cast<float4*>(row + xs_index<T>(e + 4, C));
    *d0 = make_float4(x[0], x[1], x[2], x[3]);
    *d1 = make_float4(x[4], x[5], x[6], x[7]);
  }
  return ss;
}

// The same without a norm weight (O and down inputs), for rows up to 8 * 256
// vectors per round trip to L2: every load of a batch is issued before any
// of its values is used (the down input of a 12288-wide FFN is staged in one
// round trip instead of three).
template <typename T>
__device__ __forceinline__ float cons_stage_plain(float* row, int C, const float* src, int n) {
  constexpr int kBatch = 8;
  const int ct = threadIdx.x - 32;
  const int nv = n >> 3;
  float ss = 0.0f;
  for (int base = ct; base < nv; base += 256 * kBatch) {
    float x[kBatch][8];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i8 = base + u * 256;
      if (i8 < nv) load8_row<T, float>(src + (size_t)i8 * 8, x[u]);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int i8 = base + u * 256;
      if (i8 < nv) {
        const int e = i8 * 8;
        *reinterpret_cast<float4*>(row + xs_index<T>(e, C)) = make_float4(x[u][0], x[u][1], x[u][2], x[u][3]);
        *reinterpret_cast<float4*>(row + xs_index<T>(e + 4, C)) = make_float4(x[u][4], x[u][5], x[u][6], x[u][7]);
      }
    }
  }
  return ss;
}

// Stage the input row(s) of all nb requests times their norm weights (layout
// above): one pass that stores x * w and sums x^2 for every vector, and the
// warps' sums in red for cons_rms_factors.
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
        s0 = cons_stage_raw<T, T>(dst, C, 0, a.hidden_in + (size_t)b * a.H, a.H, a.w_norm_h);
        s1 = cons_stage_raw<T, T>(dst, C, a.H, a.embeds_in + (size_t)b * a.H, a.H, a.w_norm_e);
      } else if (a.H <= 8 * 2 * 256) {
        // the previous step's draft id, the hidden row and the norm weights
        // load together, the embedding row as soon as the id is in: the two
        // halves' round trips overlap (at most two 8-value vectors per thread)
        const int ct = threadIdx.x - 32;
        float xh[2][8], wh[2][8], xe[2][8], we[2][8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int i8 = ct + 256 * u;
          if (8 * i8 < a.H) {
            load8_row<T, float>(a.hid + (size_t)b * a.H + 8 * i8, xh[u]);
            load8_row<T, T>(a.w_norm_h + 8 * i8, wh[u]);
            load8_row<T, T>(a.w_norm_e + 8 * i8, we[u]);
          }
        }
        const int prev = (a.keys_in || !a.chain_ids) ? eh_prev_draft(a, b) : 0;
        int id = a.chain_ids ? a.chain_ids[(size_t)b * (a.K - 1) + (a.k - 2)] : prev;
        if (id < 0 || id >= a.V) {
          if (threadIdx.x == 32) set_error(a.err, MTP_ERR_DEVICE_ARGS);
          id = 0;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int i8 = ct + 256 * u;
          if (8 * i8 < a.H) load8_row<T, T>(a.embed + (size_t)id * a.H + 8 * i8, xe[u]);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int i8 = ct + 256 * u;
          if (8 * i8 < a.H) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              s0 = fmaf(xh[u][e], xh[u][e], s0);
              s1 = fmaf(xe[u][e], xe[u][e], s1);
              xh[u][e] *= wh[u][e];
              xe[u][e] *= we[u][e];
            }
            const int eh = i8 * 8, ee = a.H + i8 * 8;
            *reinterpret_cast<float4*>(dst + xs_index<T>(eh, C)) = make_float4(xh[u][0], xh[u][1], xh[u][2], xh[u][3]);
            *reinterpret_cast<float4*>(dst + xs_index<T>(eh + 4, C)) = make_float4(xh[u][4], xh[u][5], xh[u][6], xh[u][7]);
            *reinterpret_cast<float4*>(dst + xs_index<T>(ee, C)) = make_float4(xe[u][0], xe[u][1], xe[u][2], xe[u][3]);
            *reinterpret_cast<float4*>(dst + xs_index<T>(ee + 4, C)) = make_float4(xe[u][4], xe[u][5], xe[u][6], xe[u][7]);
          }
        }
      } else {
        s0 = cons_stage_raw<T, float>(dst, C, 0, a.hid + (size_t)b * a.H, a.H, a.w_norm_h);
        const int prev = (a.keys_in || !a.chain_ids) ? eh_prev_draft(a, b) : 0;
        int id = a.chain_ids ? a.chain_ids[(size_t)b * (a.K - 1) + (a.k - 2)] : prev;
        if (id < 0 || id >= a.V) {
          if (threadIdx.x == 32) set_error(a.err, MTP_ERR_DEVICE_ARGS);
          id = 0;
        }
        s1 = cons_stage_raw<T, T>(dst, C, a.H, a.embed + (size_t)id * a.H, a.H, a.w_norm_e);
      }
    } else if constexpr (KIND == QKV_ROPE) {
      s0 = cons_stage_raw<T, float>(dst, C, 0, a.x + (size_t)b * a.H, a.H, a.w_norm_in);
    } else if constexpr (KIND == O_PROJ) {
      cons_stage_plain<T>(dst, C, a.attn + (size_t)b * a.q_dim, a.q_dim);
    } else if constexpr (KIND == GATE_UP) {
      s0 = cons_stage_raw<T, float>(dst, C, 0, a.h1 + (size_t)b * a.H, a.H, a.w_norm_post);
    } else if constexpr (KIND == DOWN) {
      cons_stage_plain<T>(dst, C, a.act + (size_t)b * a.F, a.F);
    } else {
      s0 = cons_stage_raw<T, float>(dst, C, 0, a.hid + (size_t)b * a.H, a.H, a.w_norm_f);
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
  }
  cons_bar();
}

// The previous step's draft id of request b, for eh_proj at k > 1 (called
// by whole warps): reduced from the deferred LM head's per-CTA keys -- every
// warp reduces them itself, so no barrier is needed -- or read from
// draft_ids.  With deferred keys, thread 32 of CTA 0 also writes the draft id,
// advances pending as the LM head's last CTA would have, and zeroes the LM
// launch's claim counter.
template <typename T>
__device__ __forceinline__ int eh_prev_draft(const StepArgs<T>& a, int b) {
  if (a.keys_in) {
    const int lane = threadIdx.x & 31;
    unsigned long long kk = 0ull;
    for (int i = lane; i < a.keys_n; i += 32) kk = umax64(kk, __ldcg(a.cta_keys + i));
    kk = warp_max_u64(kk);
    const int id = (int)key_index(kk);
    if (blockIdx.x == 0 && threadIdx.x == 32) {
      MTP_STORE(a.err, a.draft_ids, (size_t)b * a.K + (a.k - 2), (long long)a.B * a.K, id);
      if (!__ldcg(a.req_bad + b)) MTP_STORE(a.err, a.pending, b, a.B, a.k - 1);
      if (a.keys_tick) *a.keys_tick = 0ull;
    }
    return id;
  }
  return a.draft_ids[(size_t)b * a.K + (a.k - 2)];
}

// The RMS factors 1 / sqrt(mean(x^2) + eps) of the staged inputs (request
// b, input vector v: eh_proj's hidden and embedding halves), from the warps'
// sums of squares; 1 for the kinds without a norm.  The staged rows hold
// x * w unscaled: the factor multiplies the finished dot products, which
// takes a pass over the staged rows and a barrier off the critical path.
template <typename T, int KIND, int NB>
__device__ __forceinline__ void cons_rms_factors(const StepArgs<T>& a, const float* red, int nb, float (&rs)[NB][2]) {
  constexpr bool kNorm = (KIND != O_PROJ && KIND != DOWN);
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    rs[b][0] = rs[b][1] = 1.0f;
    if (kNorm && b < nb) {
#pragma unroll
      for (int v = 0; v < 2; ++v) {
        if (v == 0 || KIND == EH_PROJ) {
          float t = 0.0f;
          for (int w = 0; w < kTmaConsumers; ++w) t += red[w * 8 + 2 * b + v];
          rs[b][v] = rsqrtf(t / (float)a.H + a.eps);
        }
      }
    }
  }
}

}  // namespace mtp
