// Quantized MTP head: the format the MTP component gets in the pages'
// OpenVINO export ("How OpenVINO MTP Speculative Decoding Works Internally",
// "Why MTP gets its own quantization configuration": 4-bit asymmetric,
// group size 64, with an INT8 symmetric backup).
//
// * Projections (eh_proj, q, k, v, o, gate, up, down): INT4 asymmetric in
//   groups of 64 consecutive input columns.  For a group w_0..w_63 (bf16):
//     lo = min(min w, 0), hi = max(max w, 0), s = (hi - lo) / 15 (1 if 0),
//     z = clamp(rint(-lo / s), 0, 15), q_i = clamp(rint(w_i / s) + z, 0, 15),
//   stored as packed codes (column 2k in the low nibble of byte k), the
//   scale as fp16 and the zero point as a byte; w' = (q - z) * fp16(s).
// * Shared embedding / LM head (the backup precision): INT8 symmetric per
//   row: s = max |w| / 127 (1 if 0), q_i = clamp(rint(w_i / s), -127, 127),
//   scale as fp16; w' = q * fp16(s).
// All of it in IEEE fp32 with round-half-to-even, so any implementation of
// the same formulas gets the same codes.
//
// The small-batch projections stream units of several row pairs (codes,
// scales, zero points) through the same bulk-copy ring as the dense kernels
// and dequantize in fp32: codes become floats through the exponent trick
// (code | 0x4B000000 reads as 2^23 + code), so a weight costs a shift, a
// logic op, an add and its multiply-add.
#include <string.h>

#include "mtp_gemv.cuh"

namespace mtp {

// ------------------------------------------------------------ quantizers

__device__ __forceinline__ float bf16_at(const uint16_t* p, int i) { return __uint_as_float((uint32_t)p[i] << 16); }

// One thread per group of 64.
__global__ void quant_int4_kernel(const uint16_t* w, int rows, int cols, uint8_t* q, uint16_t* scales,
                                  uint8_t* zeros) {
  const int gpr = cols / 64;
  const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= (long long)rows * gpr) return;
  const int r = (int)(g / gpr), gi = (int)(g - (long long)r * gpr);
  const uint16_t* src = w + (size_t)r * cols + (size_t)gi * 64;
  float lo = 0.0f, hi = 0.0f;
  for (int i = 0; i < 64; ++i) {
    const float v = bf16_at(src, i);
    lo = fminf(lo, v);
    hi = fmaxf(hi, v);
  }
  float s = (hi - lo) / 15.0f;
  if (s == 0.0f) s = 1.0f;
  const float z = fminf(fmaxf(rintf(-lo / s), 0.0f), 15.0f);
  uint8_t* dst = q + (size_t)r * (cols / 2) + (size_t)gi * 32;
  for (int k = 0; k < 32; ++k) {
    const int q0 = (int)fminf(fmaxf(rintf(bf16_at(src, 2 * k) / s) + z, 0.0f), 15.0f);
    const int q1 = (int)fminf(fmaxf(rintf(bf16_at(src, 2 * k + 1) / s) + z, 0.0f), 15.0f);
    dst[k] = (uint8_t)(q0 | (q1 << 4));
  }
  scales[(size_t)r * gpr + gi] = __half_as_ushort(__float2half_rn(s));
  zeros[(size_t)r * gpr + gi] = (uint8_t)z;
}

// One warp per row.
__global__ void quant_int8_kernel(const uint16_t* w, int rows, int cols, int8_t* q, uint16_t* scales) {
  const int lane = threadIdx.x & 31;
  const long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint16_t* src = w + (size_t)r * cols;
  float amax = 0.0f;
  for (int i = lane; i < cols; i += 32) amax = fmaxf(amax, fabsf(bf16_at(src, i)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  float s = amax / 127.0f;
  if (s == 0.0f) s = 1.0f;
  int8_t* dst = q + (size_t)r * cols;
  for (int i = lane; i < cols; i += 32) dst[i] = (int8_t)fminf(fmaxf(rintf(bf16_at(src, i) / s), -127.0f), 127.0f);
  if (lane == 0) scales[r] = __half_as_ushort(__float2half_rn(s));
}

cudaError_t launch_quant_int4(cudaStream_t s, const void* w, int rows, int cols, void* q, void* scales,
                              void* zeros) {
  const long long groups = (long long)rows * (cols / 64);
  const int threads = 128;
  quant_int4_kernel<<<(unsigned)((groups + threads - 1) / threads), threads, 0, s>>>(
      (const uint16_t*)w, rows, cols, (uint8_t*)q, (uint16_t*)scales, (uint8_t*)zeros);
  return cudaGetLastError();
}

cudaError_t launch_quant_int8(cudaStream_t s, const void* w, int rows, int cols, void* q, void* scales) {
  const int threads = 256;
  const int rows_per_block = threads / 32;
  quant_int8_kernel<<<(unsigned)((rows + rows_per_block - 1) / rows_per_block), threads, 0, s>>>(
      (const uint16_t*)w, rows, cols, (int8_t*)q, (uint16_t*)scales);
  return cudaGetLastError();
}

// ------------------------------------------------- quantized projections

// Code -> float: (code | 0x4B000000) reads as 2^23 + code.
__device__ __forceinline__ float nib(uint32_t u, int j) {
  return __uint_as_float(((u >> (4 * j)) & 0xFu) | 0x4B000000u) - 8388608.0f;
}

// Rows of pair p of a projection kind and where they live in the quantized
// matrices (slot, row within the slot).
template <int KIND>
__device__ __forceinline__ void qpair_rows(const StepArgs<uint16_t>& a, int p, int& r0, int& r1, int& m0, int& m1,
                                           int& rr0, int& rr1) {
  if constexpr (KIND == QKV_ROPE) {
    const int hp = a.hd / 2;
    const int grp = p / hp, i = p - grp * hp;
    r0 = grp * a.hd + i;
    r1 = r0 + hp;
    if (r0 < a.q_dim) { m0 = QM_Q; rr0 = r0; }
    else if (r0 < a.q_dim + a.kv_dim) { m0 = QM_K; rr0 = r0 - a.q_dim; }
    else { m0 = QM_V; rr0 = r0 - a.q_dim - a.kv_dim; }
    m1 = m0;
    rr1 = rr0 + hp;
  } else if constexpr (KIND == GATE_UP) {
    r0 = r1 = p;
    m0 = QM_GATE;
    m1 = QM_UP;
    rr0 = rr1 = p;
  } else {
    m0 = m1 = (KIND == EH_PROJ) ? QM_EH : (KIND == O_PROJ) ? QM_O : QM_DOWN;
    r0 = rr0 = 2 * p;
    r1 = rr1 = 2 * p + 1;
  }
}

// Bytes of one row pair in a ring slot: codes, fp16 scales, zero points of
// both rows, [q0 | q1 | s0 | s1 | z0 | z1].
__host__ __device__ __forceinline__ uint32_t q4_pair_bytes(int C) { return (uint32_t)(C + C / 16 + C / 32); }

// Projections (EH, QKV, O, GU, DOWN) with INT4 weights, B <= 4.  Same
// producer / consumer ring as gemv_tma_kernel; a unit is `ppu` consecutive
// row pairs, unit u sits in stage u % stages and is consumed by warp
// u % consumers (stages a multiple of consumers).  Per 32-column half group
// a lane forms sum q*x over its codes and adds s * (sum q*x - z * sum x),
// with the half-group sums of x staged once per CTA.
template <int KIND, int NB>
__global__ void __launch_bounds__(kTmaThreads, 1)
    gemv_q4_kernel(const StepArgs<uint16_t> a, int stages, int consumers, int ppu) {
  extern __shared__ __align__(128) unsigned char gsm[];
  __shared__ __align__(8) uint64_t full_bar[kMaxTmaStages], empty_bar[kMaxTmaStages];
  __shared__ float red[kTmaConsumers * 8];

  pdl_trigger();
  const int C = gemv_cols(a, KIND);
  const int P = gemv_pairs(a, KIND);
  const int G = gridDim.x;
  const int p_begin = (int)(((long long)blockIdx.x * P) / G);
  const int p_end = (int)(((long long)(blockIdx.x + 1) * P) / G);
  const int nunits = (p_end - p_begin + ppu - 1) / ppu;
  const uint32_t pair_bytes = q4_pair_bytes(C);
  const uint32_t stage_stride = ((uint32_t)ppu * pair_bytes + 127u) & ~127u;
  float* xs = reinterpret_cast<float*>(gsm + (size_t)stages * stage_stride);  // [NB][C]
  float* xh = xs + (size_t)NB * C;                                              // [NB][C / 32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

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
      const uint64_t pol = l2_evict_first_policy();
      for (int it = 0; it < nunits; ++it) {
        const int s = it % stages;
        if (!mbar_wait_bounded(&empty_bar[s], (uint32_t)(((it / stages) & 1) ^ 1), kGemvWaitLimit)) {
          set_error(a.err, MTP_ERR_TIMEOUT);
          break;
        }
        const int pa = p_begin + it * ppu, pe = min(p_end, pa + ppu);
        mbar_expect_tx(&full_bar[s], (uint32_t)(pe - pa) * pair_bytes);
        for (int p = pa; p < pe; ++p) {
          int r0, r1, m0, m1, rr0, rr1;
          qpair_rows<KIND>(a, p, r0, r1, m0, m1, rr0, rr1);
          unsigned char* dst = gsm + (size_t)s * stage_stride + (size_t)(p - pa) * pair_bytes;
          const uint32_t qb = (uint32_t)C / 2, sb = (uint32_t)C / 32, zb = (uint32_t)C / 64;
          if (m0 == m1 && rr1 == rr0 + 1) {
            bulk_g2s_hint(dst, a.q4[m0] + (size_t)rr0 * qb, 2 * qb, &full_bar[s], pol);
            bulk_g2s_hint(dst + 2 * qb, a.s4[m0] + (size_t)rr0 * (C / 64), 2 * sb, &full_bar[s], pol);
            bulk_g2s_hint(dst + 2 * qb + 2 * sb, a.z4[m0] + (size_t)rr0 * zb, 2 * zb, &full_bar[s], pol);
          } else {
            bulk_g2s_hint(dst, a.q4[m0] + (size_t)rr0 * qb, qb, &full_bar[s], pol);
            bulk_g2s_hint(dst + qb, a.q4[m1] + (size_t)rr1 * qb, qb, &full_bar[s], pol);
            bulk_g2s_hint(dst + 2 * qb, a.s4[m0] + (size_t)rr0 * (C / 64), sb, &full_bar[s], pol);
            bulk_g2s_hint(dst + 2 * qb + sb, a.s4[m1] + (size_t)rr1 * (C / 64), sb, &full_bar[s], pol);
            bulk_g2s_hint(dst + 2 * qb + 2 * sb, a.z4[m0] + (size_t)rr0 * zb, zb, &full_bar[s], pol);
            bulk_g2s_hint(dst + 2 * qb + 2 * sb + zb, a.z4[m1] + (size_t)rr1 * zb, zb, &full_bar[s], pol);
          }
        }
      }
    }
    return;
  }

  // consumers: stage the normalised input and its half-group sums
  pdl_wait();
  if (KIND == EH_PROJ && a.k == 1 && blockIdx.x == 0)
    for (int b = threadIdx.x - 32; b < a.B; b += 32 * kTmaConsumers) a.req_bad[b] = (a.pending[b] != 0);
  const int nb = a.B;
  cons_stage_inputs<uint16_t, KIND>(a, xs, C, nb, red);
  const int nh = C / 32;
  for (int i = threadIdx.x - 32; i < nb * nh; i += 256) {
    const int b = i / nh, v = i - b * nh;
    const float4* xp = reinterpret_cast<const float4*>(xs + (size_t)b * C + 32 * v);
    float t = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float4 f = xp[k];
      t += (f.x + f.y) + (f.z + f.w);
    }
    xh[(size_t)b * nh + v] = t;
  }
  cons_bar();

  const int cw = warp - 1;
  unsigned long long best_unused = 0ull;
  for (int it = cw; cw < consumers && it < nunits; it += consumers) {
    const int s = it % stages;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full_bar[s], (uint32_t)((it / stages) & 1), kGemvWaitLimit))) {
      if (lane == 0) set_error(a.err, MTP_ERR_TIMEOUT);
      break;
    }
    const int pa = p_begin + it * ppu, pe = min(p_end, pa + ppu);
    for (int p = pa; p < pe; ++p) {
      const unsigned char* base = gsm + (size_t)s * stage_stride + (size_t)(p - pa) * pair_bytes;
      const uint8_t* q0 = base;
      const uint8_t* q1 = base + C / 2;
      const uint16_t* s0 = reinterpret_cast<const uint16_t*>(base + C);
      const uint16_t* s1 = s0 + C / 64;
      const uint8_t* z0 = base + C + C / 16;
      const uint8_t* z1 = z0 + C / 64;
      float acc0[NB], acc1[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) acc0[b] = acc1[b] = 0.0f;
#pragma unroll 2
      for (int v = lane; v < nh; v += 32) {
        const uint4 wa = *reinterpret_cast<const uint4*>(q0 + 16 * v);
        const uint4 wb = *reinterpret_cast<const uint4*>(q1 + 16 * v);
        const int g = v >> 1;
        const float sa = __half2float(__ushort_as_half(s0[g])), sb = __half2float(__ushort_as_half(s1[g]));
        const float za = (float)z0[g], zb = (float)z1[g];
        const uint32_t ua[4] = {wa.x, wa.y, wa.z, wa.w}, ub[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (b < nb) {
            const float* xp = xs + (size_t)b * C + 32 * v;
            float da = 0.0f, db = 0.0f;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float4 x0 = *reinterpret_cast<const float4*>(xp + 8 * k);
              const float4 x1 = *reinterpret_cast<const float4*>(xp + 8 * k + 4);
              const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                da = fmaf(nib(ua[k], j), xv[j], da);
                db = fmaf(nib(ub[k], j), xv[j], db);
              }
            }
            const float hs = xh[(size_t)b * nh + v];
            acc0[b] = fmaf(sa, da - za * hs, acc0[b]);
            acc1[b] = fmaf(sb, db - zb * hs, acc1[b]);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        acc0[b] = warp_sum(acc0[b]);
        acc1[b] = warp_sum(acc1[b]);
      }
      if (lane == 0) {
        int r0, r1, m0, m1, rr0, rr1;
        qpair_rows<KIND>(a, p, r0, r1, m0, m1, rr0, rr1);
#pragma unroll
        for (int b = 0; b < NB; ++b)
          if (b < nb) epilogue<uint16_t, KIND>(a, b, r0, r1, acc0[b], acc1[b], best_unused);
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty_bar[s])) : "memory");
  }
}

// Signed byte j of u (after u ^= 0x80808080) as a float, exactly.
__device__ __forceinline__ float sbyte(uint32_t ux, int j) {
  return __uint_as_float(__byte_perm(ux, 0x4B000000u, 0x7540u | (uint32_t)j)) - 8388736.0f;
}

// LM head with INT8 rows, B <= 4: units of `ppu` row pairs (2 * ppu
// consecutive rows, one bulk copy); the CTA's row scales are staged in
// shared memory before the dependency wait (weights are constant).  The
// epilogue and the cross-CTA argmax are those of the dense kernel.
template <int NB>
__global__ void __launch_bounds__(kTmaThreads, 1)
    gemv_q8_lm_kernel(const StepArgs<uint16_t> a, int stages, int consumers, int ppu) {
  extern __shared__ __align__(128) unsigned char gsm[];
  __shared__ __align__(8) uint64_t full_bar[kMaxTmaStages], empty_bar[kMaxTmaStages];
  __shared__ float red[kTmaConsumers * 8];
  __shared__ unsigned long long cta_best[kTmaConsumers][NB];
  __shared__ int am_last;

  pdl_trigger();
  const int C = a.H;
  const int P = (a.V + 1) / 2;
  const int G = gridDim.x;
  const int p_begin = (int)(((long long)blockIdx.x * P) / G);
  const int p_end = (int)(((long long)(blockIdx.x + 1) * P) / G);
  const int nunits = (p_end - p_begin + ppu - 1) / ppu;
  const uint32_t stage_stride = ((uint32_t)ppu * 2u * (uint32_t)C + 127u) & ~127u;
  float* xs = reinterpret_cast<float*>(gsm + (size_t)stages * stage_stride);  // [NB][C]
  float* srow = xs + (size_t)NB * C;                                            // [2 * (p_end - p_begin)]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = 2 * p_begin, row1 = min(a.V, 2 * p_end);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    fence_mbar_init();
  }
  for (int r = row0 + (int)threadIdx.x; r < row1; r += kTmaThreads)
    srow[r - row0] = __half2float(__ushort_as_half(__ldg(a.s8_lm + r)));
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      for (int it = 0; it < nunits; ++it) {
        const int s = it % stages;
        if (!mbar_wait_bounded(&empty_bar[s], (uint32_t)(((it / stages) & 1) ^ 1), kGemvWaitLimit)) {
          set_error(a.err, MTP_ERR_TIMEOUT);
          break;
        }
        const int ra = 2 * (p_begin + it * ppu), re = min(row1, ra + 2 * ppu);
        const uint32_t bytes = (uint32_t)(re - ra) * (uint32_t)C;
        mbar_expect_tx(&full_bar[s], bytes);
        bulk_g2s_hint(gsm + (size_t)s * stage_stride, a.q8_lm + (size_t)ra * C, bytes, &full_bar[s], pol);
      }
    }
    return;
  }

  pdl_wait();
  const int nb = a.B;
  cons_stage_inputs<uint16_t, LM_HEAD>(a, xs, C, nb, red);
  const int cw = warp - 1;
  const int nv = C / 16;
  unsigned long long best[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) best[b] = 0ull;
  for (int it = cw; cw < consumers && it < nunits; it += consumers) {
    const int s = it % stages;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full_bar[s], (uint32_t)((it / stages) & 1), kGemvWaitLimit))) {
      if (lane == 0) set_error(a.err, MTP_ERR_TIMEOUT);
      break;
    }
    const int ra = 2 * (p_begin + it * ppu), re = min(row1, ra + 2 * ppu);
    for (int r0 = ra; r0 < re; r0 += 2) {
      const bool two = r0 + 1 < re;
      const int8_t* qa = reinterpret_cast<const int8_t*>(gsm + (size_t)s * stage_stride) + (size_t)(r0 - ra) * C;
      const int8_t* qb = qa + C;
      float acc0[NB], acc1[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) acc0[b] = acc1[b] = 0.0f;
#pragma unroll 2
      for (int v = lane; v < nv; v += 32) {
        const uint4 wa = *reinterpret_cast<const uint4*>(qa + 16 * v);
        const uint4 wb = two ? *reinterpret_cast<const uint4*>(qb + 16 * v) : make_uint4(0, 0, 0, 0);
        const uint32_t ua[4] = {wa.x ^ 0x80808080u, wa.y ^ 0x80808080u, wa.z ^ 0x80808080u, wa.w ^ 0x80808080u};
        const uint32_t ub[4] = {wb.x ^ 0x80808080u, wb.y ^ 0x80808080u, wb.z ^ 0x80808080u, wb.w ^ 0x80808080u};
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (b < nb) {
            const float* xp = xs + (size_t)b * C + 16 * v;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float4 x = *reinterpret_cast<const float4*>(xp + 4 * k);
              acc0[b] = fmaf(sbyte(ua[k], 0), x.x, acc0[b]);
              acc0[b] = fmaf(sbyte(ua[k], 1), x.y, acc0[b]);
              acc0[b] = fmaf(sbyte(ua[k], 2), x.z, acc0[b]);
              acc0[b] = fmaf(sbyte(ua[k], 3), x.w, acc0[b]);
              acc1[b] = fmaf(sbyte(ub[k], 0), x.x, acc1[b]);
              acc1[b] = fmaf(sbyte(ub[k], 1), x.y, acc1[b]);
              acc1[b] = fmaf(sbyte(ub[k], 2), x.z, acc1[b]);
              acc1[b] = fmaf(sbyte(ub[k], 3), x.w, acc1[b]);
            }
          }
        }
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        acc0[b] = warp_sum(acc0[b]);
        acc1[b] = warp_sum(acc1[b]);
      }
      if (lane == 0) {
        const float sa = srow[r0 - row0], sb = two ? srow[r0 + 1 - row0] : 0.0f;
#pragma unroll
        for (int b = 0; b < NB; ++b)
          if (b < nb) epilogue<uint16_t, LM_HEAD>(a, b, r0, two ? r0 + 1 : -1, acc0[b] * sa, acc1[b] * sb, best[b]);
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty_bar[s])) : "memory");
  }

  // cross-CTA argmax: as in the dense kernel
  if (lane == 0)
#pragma unroll
    for (int j = 0; j < NB; ++j) cta_best[cw][j] = best[j];
  cons_bar();
  const int ct = threadIdx.x - 32;
  if (ct < nb) {
    unsigned long long m = 0ull;
    for (int w = 0; w < consumers; ++w) m = umax64(m, cta_best[w][ct]);
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

// ------------------------------------------------------------------ host

// Stage count (multiple of the consumer count, at most kMaxTmaStages) and
// consumer warps for a ring of `stage` bytes next to `fixed` bytes, within
// the 227 KB a CTA may hold less 1 KB for the kernels' static shared memory.
static bool q_ring(size_t stage, size_t fixed, int* stages, int* consumers) {
  const size_t budget = 226 * 1024;
  int max_stages = fixed < budget ? (int)((budget - fixed) / stage) : 0;
  if (max_stages > kMaxTmaStages) max_stages = kMaxTmaStages;
  int best_s = 0, best_c = 0;
  for (int cw = kTmaConsumers; cw >= 1; --cw) {
    const int st = cw * (max_stages / cw);
    if (st > best_s || (st == best_s && st > 0 && cw > best_c)) {
      best_s = st;
      best_c = cw;
    }
    if (cw <= 4 && best_s > 0) break;
  }
  *stages = best_s;
  *consumers = best_c;
  return best_s >= 2 && best_c >= 2;
}

template <int KIND>
static cudaError_t launch_q4(mtp_ctx* ctx, cudaStream_t s, const StepArgs<uint16_t>& a) {
  const int C = (KIND == EH_PROJ) ? 2 * a.H : (KIND == O_PROJ) ? a.q_dim : (KIND == DOWN) ? a.F : a.H;
  const int P = (KIND == EH_PROJ || KIND == O_PROJ || KIND == DOWN) ? a.H / 2
                : (KIND == QKV_ROPE) ? (a.q_dim + 2 * a.kv_dim) / 2
                                     : a.F;
  const size_t pair = q4_pair_bytes(C);
  int ppu = (int)(20480 / pair);
  if (ppu < 1) ppu = 1;
  if (ppu > 8) ppu = 8;
  const size_t stage = ((size_t)ppu * pair + 127) & ~(size_t)127;
  const int nbt = a.B <= 1 ? 1 : a.B <= 2 ? 2 : 4;
  const size_t fixed = (size_t)nbt * C * 4 + (size_t)nbt * (C / 32) * 4;
  int stages, consumers;
  if (!q_ring(stage, fixed, &stages, &consumers)) return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)stages * stage + fixed;
  const int grid = min(ctx->num_sms, P);
  const int kid = (KIND == EH_PROJ) ? MTP_KERNEL_EH_PROJ : (KIND == QKV_ROPE) ? MTP_KERNEL_QKV_ROPE
                  : (KIND == O_PROJ) ? MTP_KERNEL_O_PROJ : (KIND == GATE_UP) ? MTP_KERNEL_GATE_UP
                                                         : MTP_KERNEL_DOWN;
  prof_before(ctx, kid, s);
  cudaError_t e;
  if (nbt == 1) {
    ensure_smem((const void*)gemv_q4_kernel<KIND, 1>, smem);
    e = launch_pdl(gemv_q4_kernel<KIND, 1>, dim3(grid), dim3(kTmaThreads), smem, s, a, stages, consumers, ppu);
  } else if (nbt == 2) {
    ensure_smem((const void*)gemv_q4_kernel<KIND, 2>, smem);
    e = launch_pdl(gemv_q4_kernel<KIND, 2>, dim3(grid), dim3(kTmaThreads), smem, s, a, stages, consumers, ppu);
  } else {
    ensure_smem((const void*)gemv_q4_kernel<KIND, 4>, smem);
    e = launch_pdl(gemv_q4_kernel<KIND, 4>, dim3(grid), dim3(kTmaThreads), smem, s, a, stages, consumers, ppu);
  }
  prof_after(ctx, kid, s);
  ctx->launches++;
  return e;
}

static cudaError_t launch_q8_lm(mtp_ctx* ctx, cudaStream_t s, const StepArgs<uint16_t>& a) {
  const int C = a.H;
  const int P = (a.V + 1) / 2;
  int ppu = (int)(20480 / (2 * (size_t)C));
  if (ppu < 1) ppu = 1;
  if (ppu > 8) ppu = 8;
  const size_t stage = ((size_t)ppu * 2 * C + 127) & ~(size_t)127;
  const int grid = min(ctx->num_sms, P);
  const int nbt = a.B <= 1 ? 1 : a.B <= 2 ? 2 : 4;
  const size_t rows_per_cta = 2 * (size_t)((P + grid - 1) / grid);
  const size_t fixed = (size_t)nbt * C * 4 + rows_per_cta * 4;
  int stages, consumers;
  if (!q_ring(stage, fixed, &stages, &consumers)) return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)stages * stage + fixed;
  prof_before(ctx, MTP_KERNEL_LM_HEAD, s);
  cudaError_t e;
  if (nbt == 1) {
    ensure_smem((const void*)gemv_q8_lm_kernel<1>, smem);
    e = launch_pdl(gemv_q8_lm_kernel<1>, dim3(grid), dim3(kTmaThreads), smem, s, a, stages, consumers, ppu);
  } else if (nbt == 2) {
    ensure_smem((const void*)gemv_q8_lm_kernel<2>, smem);
    e = launch_pdl(gemv_q8_lm_kernel<2>, dim3(grid), dim3(kTmaThreads), smem, s, a, stages, consumers, ppu);
  } else {
    ensure_smem((const void*)gemv_q8_lm_kernel<4>, smem);
    e = launch_pdl(gemv_q8_lm_kernel<4>, dim3(grid), dim3(kTmaThreads), smem, s, a, stages, consumers, ppu);
  }
  prof_after(ctx, MTP_KERNEL_LM_HEAD, s);
  ctx->launches++;
  return e;
}

cudaError_t launch_draft_step_q(mtp_ctx* ctx, cudaStream_t s, int B, int k, int K, const void* hidden,
                                const void* embeds, const int32_t* positions, const mtp_kv* kv,
                                const int32_t* chain_ids, int32_t* draft_ids, float* logits, float* hidden_out) {
  const mtp_config& c = ctx->cfg;
  StepArgs<uint16_t> a;
  memset(&a, 0, sizeof(a));
  a.B = B; a.H = c.hidden; a.q_dim = ctx->q_dim; a.kv_dim = ctx->kv_dim; a.F = c.ffn; a.V = c.vocab;
  a.n_q = c.n_q_heads; a.n_kv = c.n_kv_heads; a.hd = c.head_dim; a.bs = c.block_size; a.eps = c.eps;
  a.k = k; a.K = K; a.max_pos = c.max_pos; a.num_blocks = kv->num_blocks; a.max_blocks = kv->max_blocks;
  const mtp_weights& w = ctx->w;
  a.w_norm_h = (const uint16_t*)w.w_norm_h; a.w_norm_e = (const uint16_t*)w.w_norm_e;
  a.w_norm_in = (const uint16_t*)w.w_norm_in; a.w_norm_post = (const uint16_t*)w.w_norm_post;
  a.w_norm_f = (const uint16_t*)w.w_norm_f;
  a.hidden_in = (const uint16_t*)hidden; a.embeds_in = (const uint16_t*)embeds; a.positions = positions;
  a.chain_ids = chain_ids; a.draft_ids = draft_ids; a.logits = logits; a.hidden_out = hidden_out;
  a.k_pool = (uint16_t*)kv->k_pool; a.v_pool = (uint16_t*)kv->v_pool; a.block_table = kv->block_table;
  a.seq_len = kv->seq_len; a.pending = kv->pending;
  a.hid = ctx->hid; a.x = ctx->x; a.q = ctx->q; a.attn = ctx->attn; a.h1 = ctx->h1; a.act = ctx->act;
  a.lm_keys = ctx->lm_keys; a.lm_cnt = ctx->lm_cnt; a.err = ctx->err; a.rope = ctx->rope;
  a.req_bad = ctx->req_bad;
  for (int m = 0; m < 8; ++m) {
    a.q4[m] = ctx->qw_q4[m];
    a.s4[m] = ctx->qw_s4[m];
    a.z4[m] = ctx->qw_z4[m];
  }
  a.q8 = ctx->qw_q8; a.s8 = ctx->qw_s8; a.q8_lm = ctx->qw_q8_lm; a.s8_lm = ctx->qw_s8_lm;

  cudaError_t e;
  if ((e = launch_q4<EH_PROJ>(ctx, s, a)) != cudaSuccess) return e;
  if ((e = launch_q4<QKV_ROPE>(ctx, s, a)) != cudaSuccess) return e;
  if ((e = launch_attention(ctx, s, B, k, kv)) != cudaSuccess) return e;
  if ((e = launch_q4<O_PROJ>(ctx, s, a)) != cudaSuccess) return e;
  if ((e = launch_q4<GATE_UP>(ctx, s, a)) != cudaSuccess) return e;
  if ((e = launch_q4<DOWN>(ctx, s, a)) != cudaSuccess) return e;
  return launch_q8_lm(ctx, s, a);
}

}  // namespace mtp

// ------------------------------------------------------------ entry points

extern "C" mtp_status mtp_quantize_int4_g64(void* stream, const void* w, int rows, int cols, void* q, void* scales,
                                            void* zeros) {
  if (!w || !q || !scales || !zeros || rows < 1 || cols < 64 || cols % 64) return MTP_ERR_INVALID;
  if (mtp::launch_quant_int4((cudaStream_t)stream, w, rows, cols, q, scales, zeros) != cudaSuccess) {
    cudaGetLastError();
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

extern "C" mtp_status mtp_quantize_int8_rows(void* stream, const void* w, int rows, int cols, void* q,
                                             void* scales) {
  if (!w || !q || !scales || rows < 1 || cols < 1) return MTP_ERR_INVALID;
  if (mtp::launch_quant_int8((cudaStream_t)stream, w, rows, cols, q, scales) != cudaSuccess) {
    cudaGetLastError();
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}
