// LM head + argmax for 2 to 4 requests per call on the tensor cores
// ("MTP (Multi-Token Prediction)", "Architecture": the shared LM head gives
// each step's draft logits; the draft token is their argmax).
//
// The streamed GEMV reads each staged activation once per request for every
// 16-byte weight vector; at 4 requests that is 144 bytes of shared memory
// per 16 bytes of weights, more than an SM serves per clock.  Here the
// weights keep the streamed GEMV's data movement -- whole rows, one bulk
// copy each -- and the arithmetic runs on mma.sync m16n8k16 with the roles
// swapped: 8 vocabulary rows are the N dimension (the B operand, read
// straight from the staged rows) and the requests the M dimension (the A
// operand; rows NB..15 are zero).
//
// One CTA per SM owns a balanced contiguous range of 8-row units.  Warp 0
// streams each unit (8 rows of H bf16, one bulk copy per row, rows padded by
// 16 bytes so that the 8 rows' 4-byte B-fragment reads fall in distinct
// banks) into a ring of stages.  Every consumer warp takes part in every
// unit: warp w owns columns [w H/8, (w+1) H/8), holds its slice of the
// normalised activations in registers as A fragments for the whole kernel,
// runs its H/128 k-steps on the unit and releases the stage (the empty
// barrier counts the 8 warps).  The warps' partial sums (per request and
// row) meet in a double-buffered shared area; after a consumer barrier one
// thread per (request, row) adds them in warp order (deterministic), writes
// the logit and keeps its running (value, lowest id) key.  At the end one
// 64-bit atomicMax per request per CTA; the last CTA (arrival counter)
// writes the draft ids and advances pending.
//
// The activations are rounded to bf16 for the tensor cores, the same
// operand rounding the batched tensor-core path makes.
#include "mtp_common.cuh"
#include "mtp_attn_mma.cuh"
#include "mtp_gemv.cuh"

namespace mtp {

constexpr int kLrCons = 8;
constexpr int kLrThreads = 32 * (kLrCons + 1);
constexpr int kLrMaxStages = 4;
constexpr int kLrMaxKs = 32;  // k-steps per warp slice: H <= 32 * 16 * 8 = 4096
constexpr uint32_t kLrWaitLimit = 1u << 24;

__device__ __forceinline__ void lr_cons_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

template <int NB>
__global__ void __launch_bounds__(kLrThreads, 1) mtp_lm_rows_kernel(const StepArgs<uint16_t> a, int stages) {
  extern __shared__ __align__(128) unsigned char lrs[];
  __shared__ __align__(8) uint64_t full_bar[kLrMaxStages], empty_bar[kLrMaxStages];
  __shared__ float red[2][kLrCons][NB][8];
  __shared__ float rss[kLrCons][NB];
  __shared__ float srs[NB];
  __shared__ int am_last, s_abort[2];
  __shared__ int s_range[2];
  __shared__ unsigned long long s_t0;

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H;
  const uint32_t row_bytes = (uint32_t)H * 2;
  const uint32_t pitch = row_bytes + 16;
  const uint32_t stage_bytes = 8 * pitch;
  const int nunits = (a.V + 7) >> 3;
  int u0 = (int)(((long long)blockIdx.x * nunits) / gridDim.x);
  int u1 = (int)(((long long)(blockIdx.x + 1) * nunits) / gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kLrCons);
    }
    s_abort[0] = s_abort[1] = 0;
    fence_mbar_init();
  }
  // ranges of 8-row units weighted by each SM's measured streaming rate
  // (lm_weighted_range); the logits do not depend on the split
  if (a.lm_tick && warp == 0) lm_weighted_range(a.lm_rate, a.lm_nsm, a.lm_tick, nunits, gridDim.x, lane, s_range);
  __syncthreads();
  if (a.lm_tick) {
    u0 = s_range[0];
    u1 = s_range[1];
  }
  const int n = u1 - u0;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();  // the LM head is read once per step
      for (int it = 0; it < n; ++it) {
        const int s = it % stages;
        if (!mbar_wait_bounded(&empty_bar[s], (uint32_t)(((it / stages) & 1) ^ 1), kLrWaitLimit)) {
          set_error(a.err, MTP_ERR_TIMEOUT);
          break;
        }
        const int r0 = (u0 + it) * 8;
        const int nrows = min(8, a.V - r0);  // rows past the vocabulary are not read
        unsigned char* dst = lrs + (size_t)s * stage_bytes;
        mbar_expect_tx(&full_bar[s], (uint32_t)nrows * row_bytes);
        for (int r = 0; r < nrows; ++r)
          bulk_g2s_hint(dst + (size_t)r * pitch, a.lm_head + (size_t)(r0 + r) * H, row_bytes, &full_bar[s], pol);
      }
    }
    return;
  }

  // consumers: RMS factors of the requests' inputs (whole rows, all warps)
  pdl_wait();
  const int ct = threadIdx.x - 32, cw = warp - 1;
  const int gi = lane >> 2, ti = lane & 3;
  {
    float ss[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) ss[b] = 0.0f;
    for (int i = ct * 4; i < H; i += 4 * 32 * kLrCons) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b < a.B) {
          const float4 t = __ldcg(reinterpret_cast<const float4*>(a.hid + (size_t)b * H + i));
          ss[b] += t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float t = warp_sum(ss[b]);
      if (lane == 0) rss[cw][b] = t;
    }
    lr_cons_bar();
    if (ct < a.B) {
      float t = 0.0f;
      for (int w = 0; w < kLrCons; ++w) t += rss[w][ct];
      srs[ct] = rsqrtf(t / (float)H + a.eps);
    }
    lr_cons_bar();
  }
  // this warp's slice of the activations as A fragments: k-step j covers
  // columns c0 + 16 j .. + 15; a0 holds (2 ti, 2 ti + 1), a2 (2 ti + 8, 2 ti + 9)
  // of request gi (rows gi + 8 -- a1, a3 -- are zero)
  const int slice = H / kLrCons;
  const int nks = slice / 16;
  const int c0 = cw * slice;
  uint32_t xa[kLrMaxKs][2];
  {
    const bool real = gi < a.B;
    const float sc = real ? srs[gi] : 0.0f;
    const float* xr = a.hid + (size_t)(real ? gi : 0) * H;
#pragma unroll
    for (int j = 0; j < kLrMaxKs; ++j) {
      xa[j][0] = xa[j][1] = 0u;
      if (real && j < nks) {
        const int k = c0 + 16 * j + 2 * ti;
        const float2 p = __ldcg(reinterpret_cast<const float2*>(xr + k));
        const float2 q = __ldcg(reinterpret_cast<const float2*>(xr + k + 8));
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(a.w_norm_f + k);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(a.w_norm_f + k + 8);
        xa[j][0] = pack_bf16(p.x * sc * bf16_lo(w0), p.y * sc * bf16_hi(w0));
        xa[j][1] = pack_bf16(q.x * sc * bf16_lo(w1), q.y * sc * bf16_hi(w1));
      }
    }
  }

  float rate_old = 0.0f;
  if (ct == 0) {
    s_t0 = globaltimer_ns();
    if (a.lm_tick) rate_old = lm_rate_peek(a.lm_rate, a.lm_nsm);
  }
  const long long nL = (long long)a.B * a.K * a.V;
  // thread ct < NB * 8 sums request ct / 8, row ct % 8 of every unit
  const int my_b = ct >> 3, my_r = ct & 7;
  unsigned long long best = 0ull;
  // Every consumer warp meets the others at the barrier of every unit, so a
  // wait that runs out is turned into a decision all warps take together:
  // the warp records it in s_abort[it & 1] before the barrier, all read it
  // after.  The flag is double-buffered like the partial sums: a warp that
  // has passed this unit's barrier can write the next unit's flag before a
  // slower warp has read this one's.
  int it = 0;
  for (; it < n; ++it) {
    const int s = it % stages;
    const int buf = it & 1;
    const bool ok =
        __all_sync(0xffffffffu, mbar_wait_bounded(&full_bar[s], (uint32_t)((it / stages) & 1), kLrWaitLimit));
    if (ok) {
      // B operand: row gi of the unit (N = 8 rows), columns 2 ti, 2 ti + 1 (+8)
      const unsigned char* rowp =
          lrs + (size_t)s * stage_bytes + (size_t)gi * pitch + (size_t)(c0 + 2 * ti) * 2;
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int j = 0; j < kLrMaxKs; ++j) {
        if (j < nks) {
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(rowp + 32 * j);
          const uint32_t b1 = *reinterpret_cast<const uint32_t*>(rowp + 32 * j + 16);
          const uint32_t af[4] = {xa[j][0], 0u, xa[j][1], 0u};
          mma_bf16(acc, af, b0, b1);
        }
      }
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty_bar[s])) : "memory");
      // acc[0], acc[1]: request gi, rows 2 ti and 2 ti + 1 of the unit
      if (gi < NB) {
        red[buf][cw][gi][2 * ti] = acc[0];
        red[buf][cw][gi][2 * ti + 1] = acc[1];
      }
    } else if (lane == 0) {
      s_abort[buf] = 1;
    }
    lr_cons_bar();
    if (s_abort[buf]) break;
    if (ct < NB * 8 && my_b < a.B) {
      float z = 0.0f;
#pragma unroll
      for (int w = 0; w < kLrCons; ++w) z += red[buf][w][my_b][my_r];
      const int row = (u0 + it) * 8 + my_r;
      if (row < a.V) {
        if (a.logits) MTP_STORE(a.err, a.logits, ((long long)my_b * a.K + (a.k - 1)) * a.V + row, nL, z);
        best = umax64(best, argmax_key(z, (uint32_t)row));
      }
    }
  }
  if (it < n) {
    if (ct == 0) set_error(a.err, MTP_ERR_TIMEOUT);
    // copies still in flight into the ring (units it .. it + stages - 1) get
    // a bounded chance to land before the CTA's shared memory goes away
    if (lane == 0)
      for (int j = it; j < n && j < it + stages; ++j)
        mbar_wait_bounded(&full_bar[j % stages], (uint32_t)((j / stages) & 1), kLrWaitLimit);
    __syncwarp();
  }
  // per request: the 8 threads (ct = 8 b .. 8 b + 7, all in consumer warp 0)
  if (cw == 0) {
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, o));
    if (my_r == 0 && my_b < a.B && best) atomicMax(a.lm_keys + my_b, best);
    __threadfence();
  }
  lr_cons_bar();
  if (ct == 0) {
    // this SM's streaming rate (units from the staged input to the last unit)
    if (a.lm_tick) lm_rate_store(a.lm_rate, a.lm_nsm, 8 * n, s_t0, rate_old);
    am_last = (lm_arrive(a.lm_cnt) == (int)gridDim.x - 1);
  }
  lr_cons_bar();
  if (am_last) {
    for (int b = ct; b < a.B; b += 32 * kLrCons) {
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

bool lm_rows_supported(const mtp_ctx* ctx, int B) {
  const mtp_config& c = ctx->cfg;
  return B >= 2 && B <= 4 && c.dtype == MTP_DTYPE_BF16 && c.hidden % (16 * kLrCons) == 0 &&
         c.hidden <= 16 * kLrCons * kLrMaxKs && ctx->has_weights && ctx->lm_rows;
}

cudaError_t launch_lm_rows(mtp_ctx* ctx, cudaStream_t s, const StepArgs<uint16_t>& a) {
  const int nunits = (a.V + 7) / 8;
  const int grid = nunits < ctx->num_sms ? nunits : ctx->num_sms;
  const size_t stage_bytes = (size_t)8 * ((size_t)a.H * 2 + 16);
  int stages = (int)((size_t)(220 * 1024) / stage_bytes);
  if (stages > kLrMaxStages) stages = kLrMaxStages;
  if (stages < 2) return cudaErrorInvalidValue;
  const size_t smem = (size_t)stages * stage_bytes;
  cudaError_t e;
  if (a.B <= 2) {
    e = ensure_smem((const void*)mtp_lm_rows_kernel<2>, smem);
    if (e == cudaSuccess) e = launch_pdl(mtp_lm_rows_kernel<2>, dim3(grid), dim3(kLrThreads), smem, s, a, stages);
  } else {
    e = ensure_smem((const void*)mtp_lm_rows_kernel<4>, smem);
    if (e == cudaSuccess) e = launch_pdl(mtp_lm_rows_kernel<4>, dim3(grid), dim3(kLrThreads), smem, s, a, stages);
  }
  return e;
}

}  // namespace mtp
