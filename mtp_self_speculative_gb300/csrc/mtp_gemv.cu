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
// Layout of the work (register-streaming variant below; the bulk-copy
// variant further down is the default for batches of at most 4): the grid
// is two CTAs per SM; CTA i owns a contiguous, balanced range of units (row
// pairs, single rows for eh_proj and down); its 8 warps take units
// round-robin.  A warp streams the rows of a unit with 16-byte
// non-allocating loads, U vectors
// per lane in flight per row, against the normalised input vector(s) staged
// once per CTA in shared memory as fp32.  Before waiting on the previous
// kernel (programmatic dependent launch) each warp prefetches the head of
// its first rows into L2, so the weight stream starts while the previous
// kernel drains.
#include <string.h>

#include "mtp_gemv.cuh"

namespace mtp {

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

template <typename T, int KIND, int NB>
__global__ void __launch_bounds__(kThreads, 2) mtp_regs_proj_kernel(const StepArgs<T> a) {
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
        MTP_STORE(a.err, a.draft_ids, (size_t)b * a.K + (a.k - 1), (long long)a.B * a.K, (int32_t)key_index(key));
        if (!__ldcg(a.req_bad + b)) MTP_STORE(a.err, a.pending, b, a.B, a.k);
      }
      if (threadIdx.x == 0) atomicExch(a.lm_cnt, 0);
    }
  }
}

// ------------------------------------------------- TMA-streamed variant
//
// Same work split and epilogues as mtp_regs_proj_kernel, for batches of at most 4:
// one CTA per SM; warp 0 is a producer that streams this CTA's units (row
// pairs, or single rows for eh_proj and down) into a ring of shared-memory
// stages with one-dimensional bulk (TMA) copies (one copy per contiguous
// unit, two for rotary or gate/up pairs), completing
// on per-stage mbarriers; it starts before the dependency wait, so the ring
// (about 200 KB per SM) fills while the previous kernel drains.  Warps 1..8
// stage the normalised input, then consume units round-robin from shared
// memory and release each stage as soon as its values are in registers.
// The stage count is a multiple of the number of consuming warps, and unit
// it goes to stage it % stages and warp it % consumers (see below).

template <typename T, int KIND, int NB>
__global__ void __launch_bounds__(kTmaThreads, 1) mtp_stream_proj_kernel(const StepArgs<T> a, int stages, int consumers) {
  extern __shared__ __align__(128) unsigned char gsm[];
  __shared__ __align__(8) uint64_t full_bar[kMaxTmaStages], empty_bar[kMaxTmaStages];
  __shared__ float red[kTmaConsumers * 8];
  __shared__ unsigned long long cta_best[kTmaConsumers][NB];
  __shared__ int am_last;
  __shared__ int s_range[2];
  __shared__ unsigned long long s_t0;

  pdl_trigger();
  const int C = gemv_cols(a, KIND);
  const int P = gemv_pairs(a, KIND);
  const int G = gridDim.x;
  int p_begin = (int)(((long long)blockIdx.x * P) / G);
  int p_end = (int)(((long long)(blockIdx.x + 1) * P) / G);
  const uint32_t row_bytes = (uint32_t)C * sizeof(T);
  const uint32_t stage_stride = (gemv_unit_rows(KIND) * row_bytes + 127) & ~127u;
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
  // LM head: ranges weighted by each SM's measured streaming rate (see
  // lm_weighted_range).  Every logit is computed the same way whichever CTA
  // owns its row, so the results do not depend on the split.
  if constexpr (KIND == LM_HEAD) {
    if (a.lm_tick && warp == 0) lm_weighted_range(a.lm_rate, a.lm_nsm, a.lm_tick, P, G, lane, s_range);
  }
  __syncthreads();
  if constexpr (KIND == LM_HEAD) {
    if (a.lm_tick) {
      p_begin = s_range[0];
      p_end = s_range[1];
    }
  }
  const int n = p_end - p_begin;

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
  float rate_old = 0.0f;
  if (threadIdx.x == 32) {
    s_t0 = globaltimer_ns();
    if (KIND == LM_HEAD && a.lm_tick) rate_old = lm_rate_peek(a.lm_rate, a.lm_nsm);
  }
  float rs[NB][2];
  cons_rms_factors<T, KIND, NB>(a, red, nb, rs);
  const int cw = warp - 1;
  // Full-barrier waits are by phase parity, so a warp may wait on a stage
  // only after the stage's previous fill has landed.  `stages` is a multiple
  // of the number of consuming warps A: unit it uses stage it % stages and
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
    if constexpr (KIND == EH_PROJ) {
      // the hidden half into acc0, the embedding half into acc1: each has
      // its own RMS factor
      const int nh = nvec >> 1;
#pragma unroll 4
      for (int v = lane; v < nh; v += 32) {
        const uint4 wa = *reinterpret_cast<const uint4*>(s0 + (size_t)v * VPE);
#pragma unroll
        for (int j = 0; j < NB; ++j)
          if (j < nb) acc0[j] += dot_vec_xs<T>(wa, xs + (size_t)j * C, v, C);
      }
#pragma unroll 4
      for (int v = nh + lane; v < nvec; v += 32) {
        const uint4 wa = *reinterpret_cast<const uint4*>(s0 + (size_t)v * VPE);
#pragma unroll
        for (int j = 0; j < NB; ++j)
          if (j < nb) acc1[j] += dot_vec_xs<T>(wa, xs + (size_t)j * C, v, C);
      }
    }
#pragma unroll 4
    for (int v = lane; KIND != EH_PROJ && v < nvec; v += 32) {
      const uint4 wa = *reinterpret_cast<const uint4*>(s0 + (size_t)v * VPE);
      if constexpr (gemv_unit_rows(KIND) == 1) {
#pragma unroll
        for (int j = 0; j < NB; ++j)
          if (j < nb) acc0[j] += dot_vec_xs<T>(wa, xs + (size_t)j * C, v, C);
      } else {
        const uint4 wb = two ? *reinterpret_cast<const uint4*>(s1 + (size_t)v * VPE) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          if (j < nb) {
            const float* xr = xs + (size_t)j * C;
            acc0[j] += dot_vec_xs<T>(wa, xr, v, C);
            acc1[j] += dot_vec_xs<T>(wb, xr, v, C);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty_bar[s])) : "memory");
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      acc0[j] = warp_sum(acc0[j]);
      if constexpr (gemv_unit_rows(KIND) == 2 || KIND == EH_PROJ) acc1[j] = warp_sum(acc1[j]);
    }
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        if (j < nb) {
          if constexpr (KIND == EH_PROJ)
            epilogue<T, KIND>(a, j, r0, r1, acc0[j] * rs[j][0] + acc1[j] * rs[j][1], 0.0f, best[j]);
          else
            epilogue<T, KIND>(a, j, r0, r1, acc0[j] * rs[j][0], acc1[j] * rs[j][0], best[j]);
        }
      }
    }
  }

  if constexpr (KIND == LM_HEAD) {
    if (lane == 0)
#pragma unroll
      for (int j = 0; j < NB; ++j) cta_best[cw][j] = best[j];
    cons_bar();
    const int ct = threadIdx.x - 32;
    if (a.defer_out) {
      // deferred argmax (one request): the CTA's best key goes to its own
      // slot; the next step's eh_proj reduces the slots, writes the draft id
      // and pending, and zeroes the claim counter
      if (ct == 0) {
        unsigned long long m = 0ull;
        for (int w = 0; w < kTmaConsumers; ++w) m = umax64(m, cta_best[w][0]);
        a.cta_keys[blockIdx.x] = m;
        if (a.lm_tick) lm_rate_store(a.lm_rate, a.lm_nsm, 2 * n, s_t0, rate_old);
      }
      return;
    }
    if (ct < nb) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kTmaConsumers; ++w) m = umax64(m, cta_best[w][ct]);
      if (m) atomicMax(a.lm_keys + ct, m);
      __threadfence();
    }
    cons_bar();
    if (ct == 0) {
      // this SM's streaming rate (rows from the staged input to the last pair)
      if (a.lm_tick) lm_rate_store(a.lm_rate, a.lm_nsm, 2 * n, s_t0, rate_old);
      am_last = (lm_arrive(a.lm_cnt) == (int)gridDim.x - 1);
    }
    cons_bar();
    if (am_last) {
      for (int b = ct; b < a.B; b += 256) {
        const unsigned long long key = atomicExch(a.lm_keys + b, 0ull);
        MTP_STORE(a.err, a.draft_ids, (size_t)b * a.K + (a.k - 1), (long long)a.B * a.K, (int32_t)key_index(key));
        if (!__ldcg(a.req_bad + b)) MTP_STORE(a.err, a.pending, b, a.B, a.k);
      }
      if (ct == 0) {
        atomicExch(a.lm_cnt, 0);
        if (a.lm_tick) atomicExch(a.lm_tick, 0ull);
      }
    }
  }
}

// The streamed variant's ring for this kind and batch: stages (a multiple
// of the consumer warps), consumer warps and dynamic shared memory.  False
// when the streamed variant is switched off for the kind or does not fit.
template <typename T, int KIND>
static bool stream_plan(const mtp_ctx* ctx, const StepArgs<T>& a, int* stages_out, int* consumers_out,
                        size_t* smem_out) {
  const int C = (KIND == EH_PROJ) ? 2 * a.H : (KIND == O_PROJ) ? a.q_dim : (KIND == DOWN) ? a.F : a.H;
  const int nbt = a.B <= 1 ? 1 : a.B <= 2 ? 2 : 4;
  const size_t stage_stride = ((size_t)gemv_unit_rows(KIND) * C * sizeof(T) + 127) & ~(size_t)127;
  const size_t xs_bytes = (size_t)nbt * C * sizeof(float);
  const size_t budget = (size_t)ctx->gemv_budget_kb[KIND] * 1024;
  int max_stages = xs_bytes < budget ? (int)((budget - xs_bytes) / stage_stride) : 0;
  if (max_stages > kMaxTmaStages) max_stages = kMaxTmaStages;
  // stages = consumers * k.  One row: pick the consumer count (4..8) that
  // keeps the most stages.  Two or four rows: the consumers' arithmetic
  // grows with the rows while the bytes do not, so keep all eight consumer
  // warps whenever eight stages fit.
  int consumers = 0, stages = 0;
  if (nbt >= 2 && max_stages >= kTmaConsumers) {
    consumers = kTmaConsumers;
    stages = kTmaConsumers * (max_stages / kTmaConsumers);
  }
  if (stages == 0) {
    for (int cw = kTmaConsumers; cw >= 1; --cw) {
      const int st = cw * (max_stages / cw);
      if (st > stages || (st == stages && st > 0 && cw > consumers && cw <= max_stages)) {
        stages = st;
        consumers = cw;
      }
      if (cw <= 4 && stages > 0) break;
    }
  }
  *stages_out = stages;
  *consumers_out = consumers;
  *smem_out = stages * stage_stride + xs_bytes;
  return ((ctx->gemv_stream_mask >> KIND) & 1) && a.B <= 4 && stages >= 2 && consumers >= 2;
}

// True when launch_kind runs the streamed variant for this kind and batch.
template <typename T, int KIND>
static bool runs_streamed(const mtp_ctx* ctx, const StepArgs<T>& a) {
  if (sizeof(T) == 2) {
    if (KIND == LM_HEAD && lm_rows_supported(ctx, a.B)) return false;
    if (KIND != LM_HEAD && rows_proj_supported(ctx, KIND, a.B)) return false;
  }
  int st, cw;
  size_t sm;
  return stream_plan<T, KIND>(ctx, a, &st, &cw, &sm);
}

template <typename T, int KIND>
static cudaError_t launch_kind(mtp_ctx* ctx, cudaStream_t s, const StepArgs<T>& a) {
  const int C = (KIND == EH_PROJ) ? 2 * a.H : (KIND == O_PROJ) ? a.q_dim : (KIND == DOWN) ? a.F : a.H;
  const int P = (KIND == EH_PROJ || KIND == DOWN) ? a.H
                : (KIND == O_PROJ) ? a.H / 2
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
  if constexpr (KIND == LM_HEAD && sizeof(T) == 2) {
    if (lm_rows_supported(ctx, a.B)) {
      e = launch_lm_rows(ctx, s, reinterpret_cast<const StepArgs<uint16_t>&>(a));
      prof_after(ctx, kid, s);
      ctx->launches++;
      return e;
    }
  }
  if constexpr (KIND != LM_HEAD && sizeof(T) == 2) {
    if (rows_proj_supported(ctx, KIND, a.B)) {
      e = launch_rows_proj(ctx, s, KIND, reinterpret_cast<const StepArgs<uint16_t>&>(a));
      prof_after(ctx, kid, s);
      ctx->launches++;
      return e;
    }
  }
  // TMA-streamed variant for B <= 4
  {
    const int nbt = a.B <= 1 ? 1 : a.B <= 2 ? 2 : 4;
    int stages = 0, consumers = 0;
    size_t smem_t = 0;
    if (stream_plan<T, KIND>(ctx, a, &stages, &consumers, &smem_t)) {
      const int gridt = min(ctx->num_sms, P);
      if (nbt == 1) {
        auto kern = mtp_stream_proj_kernel<T, KIND, 1>;
        ensure_smem((const void*)kern, smem_t);
        e = launch_pdl(kern, dim3(gridt), dim3(kTmaThreads), smem_t, s, a, stages, consumers);
      } else if (nbt == 2) {
        auto kern = mtp_stream_proj_kernel<T, KIND, 2>;
        ensure_smem((const void*)kern, smem_t);
        e = launch_pdl(kern, dim3(gridt), dim3(kTmaThreads), smem_t, s, a, stages, consumers);
      } else {
        auto kern = mtp_stream_proj_kernel<T, KIND, 4>;
        ensure_smem((const void*)kern, smem_t);
        e = launch_pdl(kern, dim3(gridt), dim3(kTmaThreads), smem_t, s, a, stages, consumers);
      }
      prof_after(ctx, kid, s);
      ctx->launches++;
      return e;
    }
  }
  if (nb == 4) {
    auto kern = mtp_regs_proj_kernel<T, KIND, 4>;
    ensure_smem((const void*)kern, smem);
    e = launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a);
  } else if (nb == 2) {
    auto kern = mtp_regs_proj_kernel<T, KIND, 2>;
    ensure_smem((const void*)kern, smem);
    e = launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a);
  } else {
    auto kern = mtp_regs_proj_kernel<T, KIND, 1>;
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
  StepArgs<T> a{};
  memset(&a, 0, sizeof(a));
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
  // each launch claims from its own counter of a ring of 64 (reset by the
  // launch's last CTA), so a launch that starts while an earlier LM head is
  // still finishing never sees that launch's counter
  a.lm_tick = ctx->lm_balance ? ctx->lm_tick + (ctx->lm_seq++ & 63) : nullptr;
  a.lm_rate = ctx->lm_rate;
  a.lm_nsm = ctx->num_sms;
  // Deferred argmax (one request, steps before the last, both kernels the
  // streamed variant): the LM head leaves one key per CTA and the next
  // step's eh_proj, which needs the id first thing, reduces them -- the LM
  // head's arrival counter and last-CTA tail drop out of every step but the
  // last.
  a.cta_keys = ctx->cta_keys;
  if (ctx->lm_defer_pending && k == 1 && ctx->lm_defer_tick) {
    // a deferred step whose successor never ran: zero its claim counter
    cudaError_t e0 = cudaMemsetAsync(ctx->lm_defer_tick, 0, sizeof(unsigned long long), s);
    if (e0 != cudaSuccess) return e0;
  }
  a.keys_in = ctx->lm_defer_pending && k > 1;
  a.keys_n = ctx->lm_defer_grid;
  a.keys_tick = ctx->lm_defer_tick;
  ctx->lm_defer_pending = 0;
  a.defer_out = ctx->lm_defer && B == 1 && k < K && runs_streamed<T, LM_HEAD>(ctx, a) &&
                runs_streamed<T, EH_PROJ>(ctx, a);

  cudaError_t e;
  if ((e = launch_kind<T, EH_PROJ>(ctx, s, a)) != cudaSuccess) return e;
  if ((e = launch_kind<T, QKV_ROPE>(ctx, s, a)) != cudaSuccess) return e;
  if ((e = launch_attention(ctx, s, B, k, kv)) != cudaSuccess) return e;
  if ((e = launch_kind<T, O_PROJ>(ctx, s, a)) != cudaSuccess) return e;
  if ((e = launch_kind<T, GATE_UP>(ctx, s, a)) != cudaSuccess) return e;
  if ((e = launch_kind<T, DOWN>(ctx, s, a)) != cudaSuccess) return e;
  if ((e = launch_kind<T, LM_HEAD>(ctx, s, a)) != cudaSuccess) return e;
  if (a.defer_out) {
    ctx->path_counts[MTP_PATH_LM_DEFERRED]++;
    ctx->lm_defer_pending = 1;
    ctx->lm_defer_grid = min(ctx->num_sms, (a.V + 1) / 2);
    ctx->lm_defer_tick = a.lm_tick;
  }
  return cudaSuccess;
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
