// The short projections of the draft step (eh_proj, QKV + rotary, O-proj,
// gate/up, down) for 2 to 4 requests per call on the tensor cores
// ("MTP (Multi-Token Prediction)", "Architecture": the MTP module is one
// decoder layer -- RMSNorm, attention, SwiGLU MLP -- behind the projection of
// the concatenated, normalised hidden state and token embedding).
//
// At 2-4 requests the streamed GEMV reads every staged activation once per
// request for each weight vector and is bound by shared memory.  This kernel
// keeps the GEMV's data movement -- whole weight rows by bulk copies -- and
// runs the arithmetic on mma.sync m16n8k16 with the weights as the B operand:
// a unit is 8 weight rows (N = 8), the requests are rows of the A operand
// (M = 16, rows NB..15 zero).
//
// One CTA per SM owns a balanced range of the kind's row pairs (the pairs of
// the epilogues: rotary halves, gate and up rows, neighbouring rows; single
// rows for eh_proj and down) and takes them 8 rows at a time; the last unit
// of a range may hold fewer rows, so every CTA streams about the same bytes.
// Rows are wide (2H for eh_proj, F for down), so a unit streams in chunks of
// kc columns: a stage holds the chunk of all 8 rows, one bulk copy per row,
// rows padded by 16 bytes so that the 8 rows' B-fragment words fall in
// distinct banks.  Warp 0 fills a ring of such stages; every consumer warp
// takes its eighth of each chunk's columns, reads the A fragments of those
// columns from the staged input and the B fragments from the stage, and
// releases the stage (the empty barrier counts the 8 warps).  A unit's
// partial sums (per request and row) stay in registers over its chunks and
// are parked in a double-buffered shared area (sum_full counts the 8 warps);
// a tenth warp adds them in warp order (deterministic), runs the kind's
// epilogue -- whose loads of residuals, rotary table and cache metadata
// would otherwise hold up a consumer warp and with it every stage -- and
// hands the buffer back (sum_empty).
//
// The input is staged once per CTA as bf16 x * w (the RMSNorm weight; no
// weight for O-proj and down) with each request's sum of squares; the RMS
// factor 1 / sqrt(mean(x^2) + eps) multiplies the finished sums in the
// epilogue (eh_proj: one factor per half, the hidden and the embedding
// halves accumulated apart), so the main loop starts after a single pass
// over the input.  The rounding of the activations to bf16 is the operand
// rounding the batched tensor-core path makes.
#include "mtp_common.cuh"
#include "mtp_attn_mma.cuh"
#include "mtp_gemv.cuh"

namespace mtp {

constexpr int kRpCons = 8;
constexpr int kRpEpiWarp = kRpCons + 1;           // warp 0 copies, 1..8 multiply, 9 runs the epilogues
constexpr int kRpThreads = 32 * (kRpCons + 2);
constexpr int kRpMaxStages = 8;
constexpr uint32_t kRpWaitLimit = 1u << 24;

__device__ __forceinline__ void rp_cons_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Bounded wait that gives up early once another warp has given up.
__device__ __forceinline__ bool rp_wait(uint64_t* bar, uint32_t parity, const volatile int* abort) {
  for (uint32_t i = 0; i < kRpWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63 && *abort) return false;
  }
  return false;
}

// Pairs (epilogue units) per 8-row unit.
__host__ __device__ constexpr int rp_pairs_per_unit(int kind) { return gemv_unit_rows(kind) == 2 ? 4 : 8; }

template <int KIND, int NB>
__global__ void __launch_bounds__(kRpThreads, 1)
    mtp_rows_proj_kernel(const StepArgs<uint16_t> a, int stages, int kc) {
  constexpr int UPP = rp_pairs_per_unit(KIND);
  constexpr bool kNorm = (KIND != O_PROJ && KIND != DOWN);
  constexpr int NH = (KIND == EH_PROJ) ? 2 : 1;  // accumulated halves (RMS factors per request)
  extern __shared__ __align__(128) unsigned char rps[];
  __shared__ __align__(8) uint64_t full_bar[kRpMaxStages], empty_bar[kRpMaxStages];
  __shared__ float red[2][NH][kRpCons][NB][8];
  __shared__ float ssq[kRpCons][2 * NB];
  __shared__ __align__(8) uint64_t sum_full[2], sum_empty[2];
  __shared__ volatile int s_abort;

  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = gemv_cols(a, KIND);
  const int P = gemv_pairs(a, KIND);
  const int p0 = (int)(((long long)blockIdx.x * P) / gridDim.x);
  const int p1 = (int)(((long long)(blockIdx.x + 1) * P) / gridDim.x);
  const int nunits = (p1 - p0 + UPP - 1) / UPP;
  const int nch = C / kc;
  const uint32_t chunk_bytes = (uint32_t)kc * 2;
  const uint32_t rp = chunk_bytes + 16;        // row pitch in a stage
  const uint32_t stage_bytes = 8 * rp;
  const uint32_t ap = (uint32_t)C * 2 + 16;    // row pitch of the staged input
  unsigned char* xa = rps + (size_t)stages * stage_bytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kRpCons);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&sum_full[q], kRpCons);
      mbar_init(&sum_empty[q], 1);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();  // weights are read once per step
      int it = 0;
      for (int u = 0; u < nunits; ++u) {
        // rows of the unit: slot 2j / 2j + 1 = pair j's rows (pair kinds), slot j = pair j's row
        const uint16_t* src[8];
        int nrows = 0;
        for (int j = 0; j < UPP; ++j) {
          const int p = p0 + u * UPP + j;
          int r0, r1;
          const uint16_t *w0, *w1;
          if (p < p1) pair_rows<uint16_t, KIND>(a, p, C, r0, r1, w0, w1);
          else { w0 = w1 = nullptr; }
          if (UPP == 4) {
            src[2 * j] = w0;
            src[2 * j + 1] = w1;
          } else {
            src[j] = w0;
          }
        }
        for (int r = 0; r < 8; ++r) nrows += (src[r] != nullptr);
        for (int c = 0; c < nch; ++c, ++it) {
          const int s = it % stages;
          if (!rp_wait(&empty_bar[s], (uint32_t)(((it / stages) & 1) ^ 1), &s_abort)) {
            set_error(a.err, MTP_ERR_TIMEOUT);
            s_abort = 1;
            return;
          }
          unsigned char* dst = rps + (size_t)s * stage_bytes;
          mbar_expect_tx(&full_bar[s], (uint32_t)nrows * chunk_bytes);
          for (int r = 0; r < 8; ++r)
            if (src[r]) bulk_g2s_hint(dst + (size_t)r * rp, src[r] + (size_t)c * kc, chunk_bytes, &full_bar[s], pol);
        }
      }
    }
    return;
  }

  if (warp == kRpEpiWarp) {
    // Epilogue warp: for each unit, once the 8 consumer warps have parked
    // their sums (sum_full), add them in warp order, scale by the RMS
    // factors and run the kind's epilogue; then hand the buffer back
    // (sum_empty).  Its loads (residuals, rotary table, cache metadata) and
    // stores stay off the consumers' path.
    pdl_wait();
    const int my_b = lane >> 3, my_r = lane & 7;
    const bool mine = my_b < a.B;  // B <= NB, so red and ssq are indexed within bounds
    float sr[2] = {1.0f, 1.0f};
    unsigned long long best_unused = 0ull;
    for (int u = 0; u < nunits; ++u) {
      const int buf = u & 1;
      if (!__all_sync(0xffffffffu, rp_wait(&sum_full[buf], (uint32_t)((u >> 1) & 1), &s_abort))) {
        if (lane == 0) {
          set_error(a.err, MTP_ERR_TIMEOUT);
          s_abort = 1;
        }
        break;
      }
      if (u == 0 && kNorm && mine) {
        // the consumer warps wrote their sums of squares before their first arrival
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          float t = 0.0f;
          for (int w = 0; w < kRpCons; ++w) t += ssq[w][2 * my_b + h];
          sr[h] = rsqrtf(t / (float)a.H + a.eps);
        }
      }
      float v = 0.0f;
      if (mine) {
        float z[NH];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
          z[hh] = 0.0f;
#pragma unroll
          for (int w = 0; w < kRpCons; ++w) z[hh] += red[buf][hh][w][my_b][my_r];
        }
        v = z[0] * sr[0];
        if constexpr (NH == 2) v += z[NH - 1] * sr[1];
      }
      // pair kinds: the even slot's lane runs the pair's epilogue with its
      // odd neighbour's value; single-row kinds: every slot is one row
      const float vn = __shfl_down_sync(0xffffffffu, v, 1);
      const int j = (UPP == 4) ? (my_r >> 1) : my_r;
      const int p = p0 + u * UPP + j;
      if (mine && p < p1 && (UPP == 8 || (my_r & 1) == 0)) {
        int r0, r1;
        const uint16_t *w0, *w1;
        pair_rows<uint16_t, KIND>(a, p, C, r0, r1, w0, w1);
        epilogue<uint16_t, KIND>(a, my_b, r0, r1, v, (UPP == 4) ? vn : 0.0f, best_unused);
      }
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&sum_empty[buf])) : "memory");
    }
    return;
  }

  // consumers: stage x * w (bf16) of every request, sums of squares per
  // (request, half).  A thread takes 8-value vectors i = ct, ct + 256, ...
  // of each input half; the norm weights of its first two vectors are
  // constant and load before the dependency wait, and the inputs of all
  // requests for a vector load together (one round trip per vector pair).
  const int ct = threadIdx.x - 32, cw = warp - 1;
  const int nb = a.B;
  const int nvv = (KIND == EH_PROJ) ? (a.H >> 3) : (C >> 3);  // vectors per input half
  const uint16_t* wn[NH];
  if constexpr (KIND == EH_PROJ) {
    wn[0] = a.w_norm_h;
    wn[NH - 1] = a.w_norm_e;
  } else {
    wn[0] = (KIND == QKV_ROPE) ? a.w_norm_in : (KIND == GATE_UP) ? a.w_norm_post : nullptr;
  }
  float wpre[2][NH][8];
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int h = 0; h < NH; ++h)
      if (kNorm && ct + 256 * t < nvv) load8_row<uint16_t, uint16_t>(wn[h] + 8 * (ct + 256 * t), wpre[t][h]);
  pdl_wait();
  if (KIND == EH_PROJ && a.k == 1 && blockIdx.x == 0)
    for (int b = ct; b < a.B; b += 32 * kRpCons) a.req_bad[b] = (a.pending[b] != 0);
  {
    float ss[2 * NB];
#pragma unroll
    for (int q = 0; q < 2 * NB; ++q) ss[q] = 0.0f;
    int id[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) id[b] = 0;
    if constexpr (KIND == EH_PROJ) {
      if (a.k > 1) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (b < nb) {
            id[b] = a.chain_ids ? a.chain_ids[(size_t)b * (a.K - 1) + (a.k - 2)] : a.draft_ids[(size_t)b * a.K + (a.k - 2)];
            if (id[b] < 0 || id[b] >= a.V) {
              if (ct == 0) set_error(a.err, MTP_ERR_DEVICE_ARGS);
              id[b] = 0;
            }
          }
        }
      }
    }
    for (int i = ct, t = 0; i < nvv; i += 32 * kRpCons, ++t) {
      float w[NH][8];
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        if (!kNorm) break;
        if (t < 2) {
#pragma unroll
          for (int e = 0; e < 8; ++e) w[h][e] = (t == 0) ? wpre[0][h][e] : wpre[1][h][e];
        } else {
          load8_row<uint16_t, uint16_t>(wn[h] + 8 * i, w[h]);
        }
      }
      float x[NB][NH][8];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b < nb) {
          if constexpr (KIND == EH_PROJ) {
            if (a.k == 1) {
              load8_row<uint16_t, uint16_t>(a.hidden_in + (size_t)b * a.H + 8 * i, x[b][0]);
              load8_row<uint16_t, uint16_t>(a.embeds_in + (size_t)b * a.H + 8 * i, x[b][NH - 1]);
            } else {
              load8_row<uint16_t, float>(a.hid + (size_t)b * a.H + 8 * i, x[b][0]);
              load8_row<uint16_t, uint16_t>(a.embed + (size_t)id[b] * a.H + 8 * i, x[b][NH - 1]);
            }
          } else {
            const float* src = (KIND == QKV_ROPE) ? a.x : (KIND == O_PROJ) ? a.attn : (KIND == GATE_UP) ? a.h1 : a.act;
            load8_row<uint16_t, float>(src + (size_t)b * C + 8 * i, x[b][0]);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b < nb) {
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            float q = 0.0f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              q = fmaf(x[b][h][e], x[b][h][e], q);
              if (kNorm) x[b][h][e] *= w[h][e];
            }
            ss[2 * b + h] += q;
            unsigned char* dst = xa + (size_t)b * ap + (size_t)(h * a.H + 8 * i) * 2;
            *reinterpret_cast<uint4*>(dst) = make_uint4(pack_bf16(x[b][h][0], x[b][h][1]), pack_bf16(x[b][h][2], x[b][h][3]),
                                                        pack_bf16(x[b][h][4], x[b][h][5]), pack_bf16(x[b][h][6], x[b][h][7]));
          }
        }
      }
    }
    if constexpr (kNorm) {
#pragma unroll
      for (int i = 0; i < 2 * NB; ++i) {
        const float t = warp_sum(ss[i]);
        if (lane == 0) ssq[cw][i] = t;
      }
    }
    rp_cons_bar();
  }

  const int gi = lane >> 2, ti = lane & 3;
  const int kw = kc / kRpCons;                 // this warp's columns of a chunk
  const int nks = kw / 16;
  const bool real = gi < nb;
  const unsigned char* xrow = xa + (size_t)(real ? gi : 0) * ap;
  int it = 0;
  bool failed = false;
  for (int u = 0; u < nunits && !failed; ++u) {
    const int buf = u & 1;
    float acc[NH][4];
#pragma unroll
    for (int h = 0; h < NH; ++h) acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.0f;
    for (int c = 0; c < nch; ++c, ++it) {
      const int s = it % stages;
      if (!__all_sync(0xffffffffu, rp_wait(&full_bar[s], (uint32_t)((it / stages) & 1), &s_abort))) {
        failed = true;
        break;
      }
      const int col0 = c * kc + cw * kw;       // first column of this warp's slice
      const unsigned char* bp = rps + (size_t)s * stage_bytes + (size_t)gi * rp + (size_t)(cw * kw + 2 * ti) * 2;
      const unsigned char* apn = xrow + (size_t)(col0 + 2 * ti) * 2;
      const int h = (KIND == EH_PROJ && col0 >= a.H) ? 1 : 0;
      // two accumulator chains (even and odd k-steps), so that consecutive
      // MMAs of a warp do not wait on each other's results; nks is even
      float d[4] = {0.0f, 0.0f, 0.0f, 0.0f}, e[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 2
      for (int jj = 0; jj < nks; jj += 2) {
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(bp + 32 * jj);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(bp + 32 * jj + 16);
        const uint32_t b2 = *reinterpret_cast<const uint32_t*>(bp + 32 * jj + 32);
        const uint32_t b3 = *reinterpret_cast<const uint32_t*>(bp + 32 * jj + 48);
        uint32_t af[4] = {0u, 0u, 0u, 0u}, ag[4] = {0u, 0u, 0u, 0u};
        if (real) {
          af[0] = *reinterpret_cast<const uint32_t*>(apn + 32 * jj);
          af[2] = *reinterpret_cast<const uint32_t*>(apn + 32 * jj + 16);
          ag[0] = *reinterpret_cast<const uint32_t*>(apn + 32 * jj + 32);
          ag[2] = *reinterpret_cast<const uint32_t*>(apn + 32 * jj + 48);
        }
        mma_bf16(d, af, b0, b1);
        mma_bf16(e, ag, b2, b3);
      }
      d[0] += e[0];
      d[1] += e[1];
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty_bar[s])) : "memory");
      if (NH == 2 && h) {
        acc[NH - 1][0] += d[0];
        acc[NH - 1][1] += d[1];
      } else {
        acc[0][0] += d[0];
        acc[0][1] += d[1];
      }
    }
    if (failed) break;
    // the epilogue warp has finished with this buffer's previous unit (u - 2)
    if (u >= 2 &&
        !__all_sync(0xffffffffu, rp_wait(&sum_empty[buf], (uint32_t)(((u >> 1) - 1) & 1), &s_abort))) {
      failed = true;
      break;
    }
    // acc[h][0], acc[h][1]: request gi, row slots 2 ti and 2 ti + 1 of the unit
    if (real) {
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) {
        red[buf][hh][cw][gi][2 * ti] = acc[hh][0];
        red[buf][hh][cw][gi][2 * ti + 1] = acc[hh][1];
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&sum_full[buf])) : "memory");
  }
  if (failed) {
    if (lane == 0) {
      set_error(a.err, MTP_ERR_TIMEOUT);
      s_abort = 1;
      // copies still in flight into the ring get a bounded chance to land
      for (int q = 0; q < stages; ++q)
        mbar_wait_bounded(&full_bar[(it + q) % stages], (uint32_t)(((it + q) / stages) & 1), kRpWaitLimit >> 4);
    }
  }
}

// Dynamic shared memory a CTA of the kernel takes at most: 220 KB (filling
// the last few KB that the device's opt-in limit leaves -- three 64 KB
// stages beside a 4-request input -- measured about 1% slower on the tree
// loops than 5 stages of 32 KB), within that limit less the kernel's static
// shared memory and 64 bytes of slack.
static size_t rows_smem_budget(int kind, int nb) {
  static size_t budget[10] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
  if (kind < EH_PROJ || kind > DOWN) return 0;
  const int slot = kind * 2 + (nb > 2 ? 1 : 0);
  if (budget[slot]) return budget[slot];
  int dev = 0, optin = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaFuncAttributes fa{};
  const void* f = nullptr;
  switch (kind) {
    case EH_PROJ: f = nb > 2 ? (const void*)mtp_rows_proj_kernel<EH_PROJ, 4> : (const void*)mtp_rows_proj_kernel<EH_PROJ, 2>; break;
    case QKV_ROPE: f = nb > 2 ? (const void*)mtp_rows_proj_kernel<QKV_ROPE, 4> : (const void*)mtp_rows_proj_kernel<QKV_ROPE, 2>; break;
    case O_PROJ: f = nb > 2 ? (const void*)mtp_rows_proj_kernel<O_PROJ, 4> : (const void*)mtp_rows_proj_kernel<O_PROJ, 2>; break;
    case GATE_UP: f = nb > 2 ? (const void*)mtp_rows_proj_kernel<GATE_UP, 4> : (const void*)mtp_rows_proj_kernel<GATE_UP, 2>; break;
    case DOWN: f = nb > 2 ? (const void*)mtp_rows_proj_kernel<DOWN, 4> : (const void*)mtp_rows_proj_kernel<DOWN, 2>; break;
    default: return 0;
  }
  if (cudaFuncGetAttributes(&fa, f) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  size_t lim = (size_t)optin > fa.sharedSizeBytes + 64 ? (size_t)optin - fa.sharedSizeBytes - 64 : 0;
  if (lim > 220 * 1024) lim = 220 * 1024;
  budget[slot] = lim;
  return lim;
}

// Columns per chunk: the largest power of two from 256 to 4096 (MTP_ROWS_KC
// lowers the top) dividing C -- and H for eh_proj, so that a chunk lies in
// one half -- whose stages fit at least rows_min_stages times (3;
// MTP_ROWS_MIN_STAGES) into the shared memory the staged input leaves.
// Wider chunks (8 KB row copies) streamed better on the tree loops than
// more stages of narrower ones: 2 KB copies cost 9%, 1 KB copies 20%.
static bool rows_plan(const mtp_ctx* ctx, int kind, int C, int H, int nb, int* stages, int* kc) {
  const size_t budget = rows_smem_budget(kind, nb);
  const size_t xa = (size_t)nb * ((size_t)C * 2 + 16);
  if (budget == 0 || xa >= budget) return false;
  const size_t avail = budget - xa;
  for (int k = ctx->rows_max_kc; k >= 256; k >>= 1) {
    if (C % k || (kind == EH_PROJ && H % k)) continue;
    const size_t st = (size_t)8 * ((size_t)k * 2 + 16);
    int n = (int)(avail / st);
    if (n > kRpMaxStages) n = kRpMaxStages;
    if (n >= ctx->rows_min_stages) {
      *stages = n;
      *kc = k;
      return true;
    }
  }
  return false;
}

static int rows_cols(const mtp_ctx* ctx, int kind) {
  const mtp_config& c = ctx->cfg;
  return kind == EH_PROJ ? 2 * c.hidden : kind == O_PROJ ? ctx->q_dim : kind == DOWN ? c.ffn : c.hidden;
}

bool rows_proj_supported(const mtp_ctx* ctx, int kind, int B) {
  const mtp_config& c = ctx->cfg;
  if (!(B >= 2 && B <= 4 && c.dtype == MTP_DTYPE_BF16 && ctx->has_weights && ctx->rows_proj)) return false;
  if (kind == LM_HEAD) return false;
  const int C = rows_cols(ctx, kind);
  if (C % 128 || c.hidden % 8) return false;
  int st, kc;
  return rows_plan(ctx, kind, C, c.hidden, B <= 2 ? 2 : 4, &st, &kc);
}

template <int KIND, int NB>
static cudaError_t rows_launch(mtp_ctx* ctx, cudaStream_t s, const StepArgs<uint16_t>& a, int C) {
  int stages = 0, kc = 0;
  if (!rows_plan(ctx, KIND, C, a.H, NB, &stages, &kc)) return cudaErrorInvalidValue;
  const size_t smem = (size_t)stages * 8 * ((size_t)kc * 2 + 16) + (size_t)NB * ((size_t)C * 2 + 16);
  const int P = (KIND == EH_PROJ || KIND == DOWN) ? a.H
                : (KIND == O_PROJ) ? a.H / 2
                : (KIND == QKV_ROPE) ? (a.q_dim + 2 * a.kv_dim) / 2
                                     : a.F;
  const int grid = P < ctx->num_sms ? P : ctx->num_sms;
  auto kern = mtp_rows_proj_kernel<KIND, NB>;
  cudaError_t e = ensure_smem((const void*)kern, smem);
  if (e == cudaSuccess) e = launch_pdl(kern, dim3(grid), dim3(kRpThreads), smem, s, a, stages, kc);
  return e;
}

template <int KIND>
static cudaError_t rows_launch_kind(mtp_ctx* ctx, cudaStream_t s, const StepArgs<uint16_t>& a) {
  const int C = rows_cols(ctx, KIND);
  return a.B <= 2 ? rows_launch<KIND, 2>(ctx, s, a, C) : rows_launch<KIND, 4>(ctx, s, a, C);
}

cudaError_t launch_rows_proj(mtp_ctx* ctx, cudaStream_t s, int kind, const StepArgs<uint16_t>& a) {
  switch (kind) {
    case EH_PROJ: return rows_launch_kind<EH_PROJ>(ctx, s, a);
    case QKV_ROPE: return rows_launch_kind<QKV_ROPE>(ctx, s, a);
    case O_PROJ: return rows_launch_kind<O_PROJ>(ctx, s, a);
    case GATE_UP: return rows_launch_kind<GATE_UP>(ctx, s, a);
    case DOWN: return rows_launch_kind<DOWN>(ctx, s, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mtp
