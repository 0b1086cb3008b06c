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
// Small-batch kernels (B <= 4).  The canonical codes are repacked once into
// tiles of 16 weight rows x 64 columns laid out in the register order of the
// mma.sync m16n8k16 A operand, so a lane turns its 16 bytes into operand
// registers with a shift and a logic op per pair of weights (INT4, as
// bf16 16 + q) or a byte permute and a subtract per pair (INT8, as fp16 q).
// Rows g and g + 8 of a tile are the two rows of one epilogue pair (RoPE
// pair, gate/up pair, or two consecutive rows).  The batch is the operand's
// N = 8 columns.  Tiles stream through the same bulk-copy ring as the dense
// kernels; each 64-column group folds its scale and zero point into fp32
// partial sums.
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

// ------------------------------------------------------------ tile layout

constexpr int kQ4Tile = 560;    // 512 B codes (16 B a lane), 8 scale pairs, 8 zero-point pairs
constexpr int kQ8Tile = 1024;   // two 512 B halves (16 B a lane each)
constexpr int kQ4UnitBytes = 36 * 1024;   // streamed unit (one bulk copy) at most: INT4 tiles
constexpr int kQ8UnitBytes = 16 * 1024;   // the same for the INT8 LM head
constexpr int kQStages = 32;    // ring stages at most

// Canonical quantized copies of the eight projection matrices.
struct QCanon {
  const uint8_t* q[8];
  const uint16_t* s[8];
  const uint8_t* z[8];
};

// Rows (r0, r1) of pair p of a projection kind and their source matrices
// and rows (slot, row within the slot).
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

__host__ __device__ __forceinline__ int q_cols(int kind, int H, int q_dim, int F) {
  return kind == EH_PROJ ? 2 * H : kind == O_PROJ ? q_dim : kind == DOWN ? F : H;
}
__host__ __device__ __forceinline__ int q_pairs(int kind, int H, int q_dim, int kv_dim, int F, int V) {
  return kind == QKV_ROPE ? (q_dim + 2 * kv_dim) / 2 : kind == GATE_UP ? F : kind == LM_HEAD ? (V + 1) / 2 : H / 2;
}

// Repack one INT4 projection into tiles [row block][group]: one thread per
// (tile, lane).  Lane (g, t) holds, for k-step j, one word whose nibbles
// 0..3 are the low and nibbles 4..7 the high elements of the operand
// registers {row g, row g+8} x {cols 2t, 2t+8} (+1 for the high element).
template <int KIND>
__global__ void repack_q4_kernel(const StepArgs<uint16_t> a, const QCanon cn, uint8_t* dst) {
  const int C = q_cols(KIND, a.H, a.q_dim, a.F);
  const int G = C / 64;
  const int nrb = q_pairs(KIND, a.H, a.q_dim, a.kv_dim, a.F, a.V) / 8;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (long long)nrb * G * 32) return;
  const int lane = (int)(gid & 31);
  const long long tile = gid >> 5;
  const int rb = (int)(tile / G), grp = (int)(tile - (long long)rb * G);
  const int g = lane >> 2, t = lane & 3;
  int r0, r1, m0, m1, rr0, rr1;
  qpair_rows<KIND>(a, 8 * rb + g, r0, r1, m0, m1, rr0, rr1);
  const uint8_t* c0 = cn.q[m0] + (size_t)rr0 * (C / 2);
  const uint8_t* c1 = cn.q[m1] + (size_t)rr1 * (C / 2);
  auto nib = [](const uint8_t* row, int c) -> uint32_t { return (row[c >> 1] >> (4 * (c & 1))) & 0xFu; };
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = 64 * grp + 16 * j + 2 * t;
    const uint32_t lo[4] = {nib(c0, c), nib(c1, c), nib(c0, c + 8), nib(c1, c + 8)};
    const uint32_t hi[4] = {nib(c0, c + 1), nib(c1, c + 1), nib(c0, c + 9), nib(c1, c + 9)};
    uint32_t x = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) x |= (lo[i] << (4 * i)) | (hi[i] << (16 + 4 * i));
    w[j] = x;
  }
  uint8_t* tp = dst + (size_t)tile * kQ4Tile;
  *reinterpret_cast<uint4*>(tp + 16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
  if (t == 0) {
    const size_t i0 = (size_t)rr0 * G + grp, i1 = (size_t)rr1 * G + grp;
    *reinterpret_cast<uint32_t*>(tp + 512 + 4 * g) = (uint32_t)cn.s[m0][i0] | ((uint32_t)cn.s[m1][i1] << 16);
    tp[544 + 2 * g] = cn.z[m0][i0];
    tp[545 + 2 * g] = cn.z[m1][i1];
  }
}

// Repack the INT8 LM head [V, H] into tiles [row block][group]: rows 2p and
// 2p + 1 of pair p = 8 rb + g are tile rows g and g + 8 (rows past V are
// zero).  Bytes are stored as q + 128.  Lane (g, t), k-step j: two words
// {row g, row g+8} x {cols c, c+1} and the same at c + 8, c = 16 j + 2 t,
// at byte (j / 2) * 512 + 16 * lane + (j % 2) * 8 of the tile.
__global__ void repack_q8_kernel(const int8_t* q8, int V, int H, uint8_t* dst) {
  const int G = H / 64;
  const int nrb = ((V + 1) / 2 + 7) / 8;
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (long long)nrb * G * 32) return;
  const int lane = (int)(gid & 31);
  const long long tile = gid >> 5;
  const int rb = (int)(tile / G), grp = (int)(tile - (long long)rb * G);
  const int g = lane >> 2, t = lane & 3;
  const int ra = 2 * (8 * rb + g), rbw = ra + 1;
  auto byte = [&](int row, int c) -> uint32_t {
    return row < V ? ((uint32_t)(uint8_t)q8[(size_t)row * H + c] ^ 0x80u) : 0x80u;
  };
  uint8_t* tp = dst + (size_t)tile * kQ8Tile;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = 64 * grp + 16 * j + 2 * t;
    const uint32_t w0 = byte(ra, c) | (byte(ra, c + 1) << 8) | (byte(rbw, c) << 16) | (byte(rbw, c + 1) << 24);
    const uint32_t w1 =
        byte(ra, c + 8) | (byte(ra, c + 9) << 8) | (byte(rbw, c + 8) << 16) | (byte(rbw, c + 9) << 24);
    *reinterpret_cast<uint2*>(tp + (j >> 1) * 512 + 16 * lane + (j & 1) * 8) = make_uint2(w0, w1);
  }
}

// max |w| of a bf16 vector into *out (one block).
__global__ void absmax_bf16_kernel(const uint16_t* w, int n, float* out) {
  float m = 0.0f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, fabsf(__uint_as_float((uint32_t)w[i] << 16)));
  __shared__ float sm[32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = 0.0f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) r = fmaxf(r, sm[i]);
    *out = r;
  }
}

// ------------------------------------------------------- operand helpers

__device__ __forceinline__ void mma_bf16_zc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// INT4 word -> four bf16x2 operand registers holding 16 + code: the code
// goes to mantissa bits 3..6 under the exponent of 16.0 (0x4180).
__device__ __forceinline__ void q4_operands(uint32_t w, uint32_t (&r)[4]) {
  r[0] = ((w << 3) & 0x00780078u) | 0x41804180u;
  r[1] = ((w >> 1) & 0x00780078u) | 0x41804180u;
  r[2] = ((w >> 5) & 0x00780078u) | 0x41804180u;
  r[3] = ((w >> 9) & 0x00780078u) | 0x41804180u;
}

// INT8 words (bytes q + 128) -> four fp16x2 operand registers holding q:
// byte u under the exponent of 1024.0 (0x64) reads 1024 + u; subtracting
// 1152 leaves u - 128 = q exactly.
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t x, uint32_t y) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(x), "r"(y));
  return d;
}
__device__ __forceinline__ void q8_operands(uint32_t w0, uint32_t w1, uint32_t (&r)[4]) {
  r[0] = hsub2_u32(__byte_perm(w0, 0x64646464u, 0x4140), 0x64806480u);
  r[1] = hsub2_u32(__byte_perm(w0, 0x64646464u, 0x4342), 0x64806480u);
  r[2] = hsub2_u32(__byte_perm(w1, 0x64646464u, 0x4140), 0x64806480u);
  r[3] = hsub2_u32(__byte_perm(w1, 0x64646464u, 0x4342), 0x64806480u);
}

// --------------------------------------------------------- input staging

// Eight consecutive raw input values (before the norm weight) of batch row b
// at column c of a projection kind's input.  EH: [hidden ; embedding], the
// embedding at step k >= 2 being the INT8 table row of the previous token
// (code times row scale, exact in fp32).
template <int KIND>
__device__ __forceinline__ void q_load8_raw(const StepArgs<uint16_t>& a, int b, int c, int id, float (&x)[8]) {
  if constexpr (KIND == EH_PROJ) {
    if (c < a.H) {
      if (a.k == 1) load8_row<uint16_t, uint16_t>(a.hidden_in + (size_t)b * a.H + c, x);
      else load8_row<uint16_t, float>(a.hid + (size_t)b * a.H + c, x);
    } else {
      const int cc = c - a.H;
      if (a.k == 1) {
        load8_row<uint16_t, uint16_t>(a.embeds_in + (size_t)b * a.H + cc, x);
      } else {
        const uint2 q = __ldg(reinterpret_cast<const uint2*>(a.q8 + (size_t)id * a.H + cc));
        const float s = __half2float(__ushort_as_half(__ldg(a.s8 + id)));
        const uint32_t u[2] = {q.x, q.y};
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = (float)(int8_t)((u[e >> 2] >> (8 * (e & 3))) & 0xFFu) * s;
      }
    }
  } else if constexpr (KIND == QKV_ROPE) {
    load8_row<uint16_t, float>(a.x + (size_t)b * a.H + c, x);
  } else if constexpr (KIND == O_PROJ) {
    load8_row<uint16_t, float>(a.attn + (size_t)b * a.q_dim + c, x);
  } else if constexpr (KIND == GATE_UP) {
    load8_row<uint16_t, float>(a.h1 + (size_t)b * a.H + c, x);
  } else if constexpr (KIND == DOWN) {
    load8_row<uint16_t, float>(a.act + (size_t)b * a.F + c, x);
  } else {
    load8_row<uint16_t, float>(a.hid + (size_t)b * a.H + c, x);
  }
}

template <int KIND>
__device__ __forceinline__ const uint16_t* q_norm_weight(const StepArgs<uint16_t>& a, int c) {
  if constexpr (KIND == EH_PROJ) return c < a.H ? a.w_norm_h + c : a.w_norm_e + (c - a.H);
  else if constexpr (KIND == QKV_ROPE) return a.w_norm_in + c;
  else if constexpr (KIND == GATE_UP) return a.w_norm_post + c;
  else if constexpr (KIND == LM_HEAD) return a.w_norm_f + c;
  else return nullptr;
}

// Sixteen raw input values (k-step j of a 64-column group) times the norm
// weight, if the kind has one.
template <int KIND>
__device__ __forceinline__ void q_load16(const StepArgs<uint16_t>& a, int b, int c, int id, float (&x)[16]) {
  float x0[8], x1[8];
  q_load8_raw<KIND>(a, b, c, id, x0);
  q_load8_raw<KIND>(a, b, c + 8, id, x1);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    x[e] = x0[e];
    x[8 + e] = x1[e];
  }
}

constexpr int kStageRegItems = 2;   // 16-value items a thread keeps in registers between the passes

// Item idx = (b, group, k-step j), j fastest: batch row, first column.
__device__ __forceinline__ void q_item(int idx, int G, int& b, int& c) {
  const int bg = idx >> 2;
  b = bg / G;
  c = 64 * (bg - b * G) + 16 * (idx & 3);
}

// The norm weights of a thread's register items (constant: loaded before
// the dependency wait, so that the staging after it needs one round trip).
template <int KIND>
__device__ __forceinline__ void stage_q_weights(const StepArgs<uint16_t>& a, int C, int nb,
                                                float (&wr)[kStageRegItems][16]) {
  if constexpr (KIND != O_PROJ && KIND != DOWN) {
    const int ct = threadIdx.x - 32;
    const int G = C / 64;
#pragma unroll
    for (int it = 0; it < kStageRegItems; ++it) {
      const int idx = ct + 256 * it;
      if (idx < nb * G * 4) {
        int b, c;
        q_item(idx, G, b, c);
        float w0[8], w1[8];
        const uint16_t* wp = q_norm_weight<KIND>(a, c);
        load8_row<uint16_t, uint16_t>(wp, w0);
        load8_row<uint16_t, uint16_t>(wp + 8, w1);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          wr[it][e] = w0[e];
          wr[it][8 + e] = w1[e];
        }
      }
    }
  }
}

// Stage the B operand of all nb batch rows: y = x * rms factor * norm weight
// (RMSNorm kinds; EH normalises its two halves separately), times `sigma`,
// rounded to bf16 (F16 false) or fp16 (F16 true), in the register order of
// the m16n8k16 B operand: per 64-column group, half h = k-steps 2h, 2h+1,
// lane (g = batch row, t) 16 bytes {b0(j), b1(j)} with
// b0(j) = (y[16j+2t], y[16j+2t+1]), b1(j) = (y[16j+2t+8], y[16j+2t+9]).
// Xs[group][b] = the fp32 sum of the rounded values of the group (0 for
// b >= nb), for the zero-point correction.
// Work items are (b, group, k-step j), j fastest, so the four items of a
// group sit in four neighbouring lanes and their sums combine by shuffles.
// The first kStageRegItems items of a thread stay in registers from the
// sums of squares to the rounding, so that at small batch the input is read
// once, all loads in flight together.
template <int KIND, bool F16>
__device__ void stage_q_inputs(const StepArgs<uint16_t>& a, unsigned char* xf, float* Xs, int C, int nb, float sigma,
                               float* red, int* sid, float* srs, const float (&wr)[kStageRegItems][16]) {
  constexpr bool kNorm = (KIND != O_PROJ && KIND != DOWN);
  const int ct = threadIdx.x - 32;
  const int cw = ct >> 5, l = ct & 31;
  const int G = C / 64;
  const int nitems = nb * G * 4;
  if (KIND == EH_PROJ && a.k > 1) {
    if (ct < nb) {
      int id = a.chain_ids ? a.chain_ids[(size_t)ct * (a.K - 1) + (a.k - 2)]
                           : a.draft_ids[(size_t)ct * a.K + (a.k - 2)];
      if (id < 0 || id >= a.V) {
        set_error(a.err, MTP_ERR_DEVICE_ARGS);
        id = 0;
      }
      sid[ct] = id;
    }
    cons_bar();
  }
  auto item = [&](int idx, int& b, int& grp, int& c, int& id) {
    q_item(idx, G, b, c);
    grp = c >> 6;
    id = (KIND == EH_PROJ && a.k > 1) ? sid[b] : 0;
  };
  float xr[kStageRegItems][16];
#pragma unroll
  for (int it = 0; it < kStageRegItems; ++it) {
    const int idx = ct + 256 * it;
    if (idx < nitems) {
      int b, grp, c, id;
      item(idx, b, grp, c, id);
      q_load16<KIND>(a, b, c, id, xr[it]);
    }
  }
  if constexpr (kNorm) {
    float ss[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) ss[i] = 0.0f;
    auto add = [&](int b, int c, const float (&x)[16]) {
      float t = 0.0f;
#pragma unroll
      for (int e = 0; e < 16; ++e) t = fmaf(x[e], x[e], t);
      const int slot = 2 * b + ((KIND == EH_PROJ && c >= a.H) ? 1 : 0);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i == slot) ss[i] += t;
    };
#pragma unroll
    for (int it = 0; it < kStageRegItems; ++it) {
      const int idx = ct + 256 * it;
      if (idx < nitems) {
        int b, grp, c, id;
        item(idx, b, grp, c, id);
        add(b, c, xr[it]);
      }
    }
    for (int idx = ct + 256 * kStageRegItems; idx < nitems; idx += 256) {
      int b, grp, c, id;
      item(idx, b, grp, c, id);
      float x[16];
      q_load16<KIND>(a, b, c, id, x);
      add(b, c, x);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float t = warp_sum(ss[i]);
      if (l == 0) red[cw * 8 + i] = t;
    }
    cons_bar();
    if (ct < 2 * nb) {
      float t = 0.0f;
      for (int w = 0; w < kTmaConsumers; ++w) t += red[w * 8 + ct];
      srs[ct] = rsqrtf(t / (float)a.H + a.eps);
    }
    cons_bar();
  }
  if constexpr (!F16)
    for (int i = ct; i < G * 8; i += 256)
      if ((i & 7) >= nb) Xs[i] = 0.0f;
  // rounding and layout; a warp runs while any of its lanes has an item, so
  // that the group sums can use full-warp shuffles
  auto emit = [&](int idx, bool valid, float (&x)[16], const float (&w)[16]) {
    int b = 0, grp = 0, c = 0, id = 0;
    if (valid) item(idx, b, grp, c, id);
    float X = 0.0f;
    if (valid) {
      const int half = (KIND == EH_PROJ && c >= a.H) ? 1 : 0;
      const float scale = (kNorm ? srs[2 * b + half] : 1.0f) * sigma;
      if constexpr (kNorm) {
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] *= w[e];
      }
      uint32_t h[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float y = x[e] * scale;
        if constexpr (F16) {
          h[e] = __half_as_ushort(__float2half_rn(y));
        } else {
          h[e] = __bfloat16_as_ushort(__float2bfloat16_rn(y));
          X += __uint_as_float(h[e] << 16);
        }
      }
      const int j = idx & 3;
      unsigned char* dst = xf + ((size_t)(grp * 2 + (j >> 1)) * (nb * 4) + b * 4) * 16 + (j & 1) * 8;
#pragma unroll
      for (int t = 0; t < 4; ++t)
        *reinterpret_cast<uint2*>(dst + 16 * t) =
            make_uint2(h[2 * t] | (h[2 * t + 1] << 16), h[2 * t + 8] | (h[2 * t + 9] << 16));
    }
    if constexpr (!F16) {
      X += __shfl_xor_sync(0xffffffffu, X, 1);
      X += __shfl_xor_sync(0xffffffffu, X, 2);
      if (valid && (idx & 3) == 0) Xs[grp * 8 + b] = X;
    }
  };
#pragma unroll
  for (int it = 0; it < kStageRegItems; ++it) {
    const int idx = ct + 256 * it;
    if (256 * it + 32 * cw < nitems) emit(idx, idx < nitems, xr[it], wr[it]);
  }
  for (int base = 256 * kStageRegItems; base < nitems; base += 256) {
    const int idx = base + ct;
    if (base + 32 * cw >= nitems) break;
    float x[16], w[16];
    const bool valid = idx < nitems;
    if (valid) {
      int b, grp, c, id;
      item(idx, b, grp, c, id);
      q_load16<KIND>(a, b, c, id, x);
      if constexpr (kNorm) {
        float w0[8], w1[8];
        const uint16_t* wp = q_norm_weight<KIND>(a, c);
        load8_row<uint16_t, uint16_t>(wp, w0);
        load8_row<uint16_t, uint16_t>(wp + 8, w1);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          w[e] = w0[e];
          w[8 + e] = w1[e];
        }
      }
    }
    emit(idx, valid, x, w);
  }
  cons_bar();
}

// ---------------------------------------------- INT4 projection kernel

// One CTA owns row blocks [rb0, rb1) (16 rows = 8 epilogue pairs each) and
// streams their tiles in chunks of gpc groups, one bulk copy per chunk
// (copies of 16 KB and more keep the memory system busy; smaller ones do
// not).  Every consumer warp takes part in every chunk: warp w handles
// groups w, w + A, ... of it and releases the stage (its empty barrier
// counts the A warps), so all warps walk the stages in the same order.  Per
// group a warp runs four m16n8k16 steps on fresh accumulators and folds
// them into its running sums of the row block:
//   tot += s * (acc - (16 + z) * Xs[group][batch]),
// since the operand holds 16 + code.  At the end of a row block the warps
// park their sums in one half of a double buffer, meet at a barrier, and
// warp rb % A adds them in warp order (deterministic) and runs the pair
// epilogue while the others go on.
template <int KIND, int NB>
__global__ void __launch_bounds__(kTmaThreads, 1)
    mtp_q4_proj_kernel(const StepArgs<uint16_t> a, int stages, int gpc) {
  extern __shared__ __align__(128) unsigned char gsm[];
  __shared__ __align__(8) uint64_t full_bar[kQStages], empty_bar[kQStages];
  __shared__ float red[kTmaConsumers * 8];
  __shared__ int sid[4];
  __shared__ float srs[8];

  pdl_trigger();
  constexpr int A = kTmaConsumers;
  const int C = q_cols(KIND, a.H, a.q_dim, a.F);
  const int G = C / 64;
  const int upr = G / gpc;
  const int NRB = q_pairs(KIND, a.H, a.q_dim, a.kv_dim, a.F, a.V) / 8;
  const int rb0 = (int)(((long long)blockIdx.x * NRB) / gridDim.x);
  const int rb1 = (int)(((long long)(blockIdx.x + 1) * NRB) / gridDim.x);
  const int nunits = (rb1 - rb0) * upr;
  const uint32_t kUnit = (uint32_t)gpc * kQ4Tile;
  const int nb = a.B;
  unsigned char* xf = gsm + (size_t)stages * kUnit;                     // [G][2][nb * 4][16 B]
  float* Xs = reinterpret_cast<float*>(xf + (size_t)G * 2 * NB * 64);   // [G][8]
  float* pbuf = Xs + (size_t)G * 8;                                    // [2][A][4][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], A);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      const unsigned char* src = a.qt[KIND] + (size_t)rb0 * G * kQ4Tile;
      int s = 0;
      uint32_t ph = 0;
      for (int u = 0; u < nunits; ++u) {
        if (!mbar_wait_bounded(&empty_bar[s], ph ^ 1u, kGemvWaitLimit)) {
          set_error(a.err, MTP_ERR_TIMEOUT);
          break;
        }
        mbar_expect_tx(&full_bar[s], kUnit);
        bulk_g2s_hint(gsm + (size_t)s * kUnit, src + (size_t)u * kUnit, kUnit, &full_bar[s], pol);
        if (++s == stages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    return;
  }

  float wr[kStageRegItems][16];
  stage_q_weights<KIND>(a, C, nb, wr);
  pdl_wait();
  const int ct = threadIdx.x - 32;
  if (KIND == EH_PROJ && a.k == 1 && blockIdx.x == 0)
    for (int b = ct; b < a.B; b += 256) a.req_bad[b] = (a.pending[b] != 0);
  stage_q_inputs<KIND, false>(a, xf, Xs, C, nb, 1.0f, red, sid, srs, wr);

  const int cw = warp - 1;
  const int g = lane >> 2, t = lane & 3;
  const bool has_b = g < nb;
  const size_t xrow = (size_t)nb * 64;          // bytes of one (group, half) slice of xf
  float tot[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  bool failed = false;                          // a wait ran out: skip the data, keep the barriers
  int s = 0, rbl = 0, ch = 0;
  uint32_t ph = 0;
  unsigned long long best_unused = 0ull;
  for (int u = 0; u < nunits; ++u) {
    if (!failed && !__all_sync(0xffffffffu, mbar_wait_bounded(&full_bar[s], ph, kGemvWaitLimit))) {
      if (lane == 0) set_error(a.err, MTP_ERR_TIMEOUT);
      failed = true;
    }
    if (!failed) {
      const unsigned char* st = gsm + (size_t)s * kUnit;
#pragma unroll 2
      for (int gi = cw; gi < gpc; gi += A) {
        const int grp = ch * gpc + gi;
        const unsigned char* tp = st + gi * kQ4Tile;
        const uint4 wq = *reinterpret_cast<const uint4*>(tp + 16 * lane);
        const uint32_t sp = *reinterpret_cast<const uint32_t*>(tp + 512 + 4 * g);
        const uint32_t zp = *reinterpret_cast<const uint16_t*>(tp + 544 + 2 * g);
        uint4 xa = make_uint4(0, 0, 0, 0), xb = make_uint4(0, 0, 0, 0);
        if (has_b) {
          xa = *reinterpret_cast<const uint4*>(xf + (size_t)(grp * 2) * xrow + 16 * lane);
          xb = *reinterpret_cast<const uint4*>(xf + (size_t)(grp * 2 + 1) * xrow + 16 * lane);
        }
        const float2 X = *reinterpret_cast<const float2*>(Xs + grp * 8 + 2 * t);
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        uint32_t r[4];
        q4_operands(wq.x, r);
        mma_bf16_zc(acc, r, xa.x, xa.y);
        q4_operands(wq.y, r);
        mma_bf16_zc(acc, r, xa.z, xa.w);
        q4_operands(wq.z, r);
        mma_bf16_zc(acc, r, xb.x, xb.y);
        q4_operands(wq.w, r);
        mma_bf16_zc(acc, r, xb.z, xb.w);
        const float s0 = __half2float(__ushort_as_half((unsigned short)(sp & 0xFFFFu)));
        const float s1 = __half2float(__ushort_as_half((unsigned short)(sp >> 16)));
        const float c0 = __uint_as_float(0x4B000000u | (zp & 0xFFu)) - 8388592.0f;   // 16 + z of row g
        const float c1 = __uint_as_float(0x4B000000u | (zp >> 8)) - 8388592.0f;      // 16 + z of row g + 8
        tot[0] = fmaf(s0, fmaf(-c0, X.x, acc[0]), tot[0]);
        tot[1] = fmaf(s0, fmaf(-c0, X.y, acc[1]), tot[1]);
        tot[2] = fmaf(s1, fmaf(-c1, X.x, acc[2]), tot[2]);
        tot[3] = fmaf(s1, fmaf(-c1, X.y, acc[3]), tot[3]);
      }
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty_bar[s])) : "memory");
    if (++s == stages) {
      s = 0;
      ph ^= 1u;
    }
    if (++ch == upr) {
      // row block complete: park the sums, meet, one warp combines
      float* pb = pbuf + ((size_t)(rbl & 1) * A + cw) * 128;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        pb[e * 32 + lane] = tot[e];
        tot[e] = 0.0f;
      }
      cons_bar();
      if (cw == rbl % A && !failed) {
        float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const float* pr = pbuf + (size_t)(rbl & 1) * A * 128;
        for (int w = 0; w < A; ++w)
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] += pr[w * 128 + e * 32 + lane];
        int r0, r1, m0, m1, rr0, rr1;
        qpair_rows<KIND>(a, 8 * (rb0 + rbl) + g, r0, r1, m0, m1, rr0, rr1);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int b = 2 * t + e;
          if (b < nb) epilogue<uint16_t, KIND>(a, b, r0, r1, v[e], v[2 + e], best_unused);
        }
      }
      ch = 0;
      ++rbl;
    }
  }
}

// ------------------------------------------------ INT8 LM-head kernel

// One CTA owns row blocks [rb0, rb1) of the LM head (16 rows = 8 pairs of
// consecutive vocabulary rows each); consumer warp w owns row blocks
// rb0 + w, rb0 + w + consumers, ...  Unit u = l * consumers + w is chunk
// l % upr of the warp's (l / upr)-th row block and goes to stage
// u % stages (a multiple of consumers), so every stage serves one warp in
// order; units past the warp's last row block are never issued.  The
// producer serves the warps' queues independently (one lane polls them).  The fp16
// B operand is the normalised input times a power-of-two sigma chosen at
// creation so that no value can overflow; the row scale and 1 / sigma are
// applied when a row block is complete, followed by the logits and the
// running argmax.  The cross-CTA argmax is that of the dense kernel.
template <int NB>
__global__ void __launch_bounds__(kTmaThreads, 1)
    mtp_q8_lm_kernel(const StepArgs<uint16_t> a, int stages, int consumers, int gpc) {
  extern __shared__ __align__(128) unsigned char gsm[];
  __shared__ __align__(8) uint64_t full_bar[kQStages], empty_bar[kQStages];
  __shared__ float red[kTmaConsumers * 8];
  __shared__ int sid[4];
  __shared__ float srs[8];
  __shared__ unsigned long long cta_best[kTmaConsumers][NB];
  __shared__ int am_last;

  pdl_trigger();
  const int C = a.H;
  const int G = C / 64;
  const int upr = G / gpc;
  const int P = (a.V + 1) / 2;
  const int NRB = (P + 7) / 8;
  const int rb0 = (int)(((long long)blockIdx.x * NRB) / gridDim.x);
  const int rb1 = (int)(((long long)(blockIdx.x + 1) * NRB) / gridDim.x);
  const int nrb = rb1 - rb0;
  const uint32_t kUnit = (uint32_t)gpc * kQ8Tile;
  const int nb = a.B;
  unsigned char* xf = gsm + (size_t)stages * kUnit;                          // [G][2][nb * 4][16 B]
  float* srow = reinterpret_cast<float*>(xf + (size_t)G * 2 * NB * 64);     // [16 * nrb] row scales
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    fence_mbar_init();
  }
  // the CTA's row scales (constant weights: before the dependency wait)
  for (int i = threadIdx.x; i < 16 * nrb; i += kTmaThreads) {
    const int r = 16 * rb0 + i;
    srow[i] = r < a.V ? __half2float(__ushort_as_half(__ldg(a.s8_lm + r))) : 0.0f;
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) {
      // one lane polls the warps' queues: a stage is refilled as soon as its
      // warp frees it (stage and phase of each queue kept incrementally)
      const uint64_t pol = l2_evict_first_policy();
      int q_rbl[kTmaConsumers], q_ch[kTmaConsumers], q_s[kTmaConsumers];
      uint32_t q_ph[kTmaConsumers];
      int remaining = 0;
#pragma unroll
      for (int w = 0; w < kTmaConsumers; ++w) {
        q_rbl[w] = w;
        q_ch[w] = 0;
        q_s[w] = w;
        q_ph[w] = 0;
        if (w < consumers && w < nrb) remaining += ((nrb - w + consumers - 1) / consumers) * upr;
      }
      uint32_t idle = 0;
      while (remaining > 0) {
        bool progress = false;
#pragma unroll
        for (int w = 0; w < kTmaConsumers; ++w) {
          if (w >= consumers || q_rbl[w] >= nrb) continue;
          const int s = q_s[w];
          if (!mbar_test_wait(&empty_bar[s], q_ph[w] ^ 1u)) continue;
          mbar_expect_tx(&full_bar[s], kUnit);
          const unsigned char* src =
              a.qt[LM_HEAD] + ((size_t)(rb0 + q_rbl[w]) * G + (size_t)q_ch[w] * gpc) * kQ8Tile;
          bulk_g2s_hint(gsm + (size_t)s * kUnit, src, kUnit, &full_bar[s], pol);
          if (++q_ch[w] == upr) {
            q_ch[w] = 0;
            q_rbl[w] += consumers;
          }
          q_s[w] = s + consumers;
          if (q_s[w] >= stages) {
            q_s[w] -= stages;
            q_ph[w] ^= 1u;
          }
          --remaining;
          progress = true;
        }
        if (progress) {
          idle = 0;
        } else if (++idle > kGemvWaitLimit) {
          set_error(a.err, MTP_ERR_TIMEOUT);
          break;
        }
      }
    }
    return;
  }

  float wr[kStageRegItems][16];
  stage_q_weights<LM_HEAD>(a, C, nb, wr);
  pdl_wait();
  stage_q_inputs<LM_HEAD, true>(a, xf, nullptr, C, nb, a.lm_sigma, red, sid, srs, wr);
  const float inv_sigma = 1.0f / a.lm_sigma;   // a power of two

  const int cw = warp - 1;
  const int g = lane >> 2, t = lane & 3;
  const bool has_b = g < nb;
  const size_t xrow = (size_t)nb * 64;
  unsigned long long best[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) best[b] = 0ull;
  float acc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = 0.0f;
  for (int l = 0; cw < consumers; ++l) {
    const int u = l * consumers + cw;
    const int rbl = (l / upr) * consumers + cw, ch = l - (l / upr) * upr;
    if (rbl >= nrb) break;
    const int s = u % stages;
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full_bar[s], (uint32_t)((u / stages) & 1), kGemvWaitLimit))) {
      if (lane == 0) set_error(a.err, MTP_ERR_TIMEOUT);
      break;
    }
    const unsigned char* st = gsm + (size_t)s * kUnit;
#pragma unroll 2
    for (int gi = 0; gi < gpc; ++gi) {
      const int grp = ch * gpc + gi;
      const unsigned char* tp = st + gi * kQ8Tile;
      const uint4 q0 = *reinterpret_cast<const uint4*>(tp + 16 * lane);
      const uint4 q1 = *reinterpret_cast<const uint4*>(tp + 512 + 16 * lane);
      uint4 xa = make_uint4(0, 0, 0, 0), xb = make_uint4(0, 0, 0, 0);
      if (has_b) {
        xa = *reinterpret_cast<const uint4*>(xf + (size_t)(grp * 2) * xrow + 16 * lane);
        xb = *reinterpret_cast<const uint4*>(xf + (size_t)(grp * 2 + 1) * xrow + 16 * lane);
      }
      uint32_t r[4];
      q8_operands(q0.x, q0.y, r);
      mma_f16(acc[0], r, xa.x, xa.y);
      q8_operands(q0.z, q0.w, r);
      mma_f16(acc[1], r, xa.z, xa.w);
      q8_operands(q1.x, q1.y, r);
      mma_f16(acc[2], r, xb.x, xb.y);
      q8_operands(q1.z, q1.w, r);
      mma_f16(acc[3], r, xb.z, xb.w);
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty_bar[s])) : "memory");
    if (ch == upr - 1) {
      // row block complete: rows 2p (tile row g) and 2p + 1 (tile row g + 8)
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[e] = (acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e]);
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j][e] = 0.0f;
      }
      const int p = 8 * (rb0 + rbl) + g;
      if (p < P) {
        const int r0 = 2 * p, r1 = (2 * p + 1 < a.V) ? 2 * p + 1 : -1;
        const float s0 = srow[r0 - 16 * rb0] * inv_sigma;
        const float s1 = srow[r0 + 1 - 16 * rb0] * inv_sigma;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          if (b < nb && (b >> 1) == t) {
            const int e = b & 1;
            epilogue<uint16_t, LM_HEAD>(a, b, r0, r1, v[e] * s0, v[2 + e] * s1, best[b]);
          }
        }
      }
    }
  }

  // CTA argmax, then across CTAs: as in the dense kernel
#pragma unroll
  for (int b = 0; b < NB; ++b) best[b] = warp_max_u64(best[b]);
  if (lane == 0 && cw < kTmaConsumers)
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
      MTP_STORE(a.err, a.draft_ids, (size_t)b * a.K + (a.k - 1), (long long)a.B * a.K, (int32_t)key_index(key));
      if (!__ldcg(a.req_bad + b)) MTP_STORE(a.err, a.pending, b, a.B, a.k);
    }
    if (ct == 0) atomicExch(a.lm_cnt, 0);
  }
}

// ------------------------------------------------------------------ host

// Dynamic shared memory of one CTA at most (the kernels' static shared
// memory is under 2 KB of the 227 KB a CTA may hold).
constexpr size_t kQSmemBudget = 225 * 1024;

// Groups per streamed unit: the largest divisor of G whose unit fits in
// `max_bytes` (bulk copies of 16 KB and more stream markedly better than
// 8 KB ones).
static int q_gpc(int G, int tile, int max_bytes) {
  int best = 1;
  for (int d = 1; d <= G; ++d)
    if (G % d == 0 && d * tile <= max_bytes) best = d;
  return best;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Ring plan: the most consumer warps (at least two stages each, stage count
// a multiple of the warp count) whose ring fits next to `fixed` bytes plus
// `per_warp` bytes a consumer warp, within 225 KB (the static shared memory
// of the kernels is under 2 KB).
static bool q_plan(size_t unit, size_t fixed, size_t per_warp, int* stages, int* consumers) {
  const size_t budget = kQSmemBudget;
  for (int cw = kTmaConsumers; cw >= 2; --cw) {
    const size_t f = fixed + per_warp * cw;
    if (f >= budget) continue;
    int st = (int)((budget - f) / unit);
    if (st > kQStages) st = kQStages;
    st -= st % cw;
    if (st >= 2 * cw) {
      *stages = st;
      *consumers = cw;
      return true;
    }
  }
  return false;
}

static int kind_kernel_id(int kind) {
  return kind == EH_PROJ ? MTP_KERNEL_EH_PROJ : kind == QKV_ROPE ? MTP_KERNEL_QKV_ROPE
         : kind == O_PROJ ? MTP_KERNEL_O_PROJ : kind == GATE_UP ? MTP_KERNEL_GATE_UP
         : kind == DOWN ? MTP_KERNEL_DOWN : MTP_KERNEL_LM_HEAD;
}

template <int KIND, int NB>
static cudaError_t launch_q4_nb(mtp_ctx* ctx, cudaStream_t s, const StepArgs<uint16_t>& a) {
  const int C = q_cols(KIND, a.H, a.q_dim, a.F);
  const int G = C / 64;
  const int nrb_all = q_pairs(KIND, a.H, a.q_dim, a.kv_dim, a.F, a.V) / 8;
  const int grid = min(ctx->num_sms, nrb_all);
  const size_t fixed = (size_t)G * 2 * NB * 64 + (size_t)G * 32 + (size_t)2 * kTmaConsumers * 512;
  // the largest chunk (a divisor of G, at most kQ4UnitBytes) that leaves
  // room for at least four stages
  int gpc = q_gpc(G, kQ4Tile, kQ4UnitBytes);
  while (gpc > 1 && (fixed + (size_t)4 * gpc * kQ4Tile > kQSmemBudget)) gpc = q_gpc(G, kQ4Tile, (gpc - 1) * kQ4Tile);
  if (fixed + (size_t)2 * gpc * kQ4Tile > kQSmemBudget) return cudaErrorInvalidConfiguration;
  int stages = (int)((kQSmemBudget - fixed) / ((size_t)gpc * kQ4Tile));
  if (stages > kQStages) stages = kQStages;
  const size_t smem = (size_t)stages * gpc * kQ4Tile + fixed;
  ensure_smem((const void*)mtp_q4_proj_kernel<KIND, NB>, smem);
  return launch_pdl(mtp_q4_proj_kernel<KIND, NB>, dim3(grid), dim3(kTmaThreads), smem, s, a, stages, gpc);
}

template <int KIND>
static cudaError_t launch_q4(mtp_ctx* ctx, cudaStream_t s, const StepArgs<uint16_t>& a) {
  const int kid = kind_kernel_id(KIND);
  prof_before(ctx, kid, s);
  const cudaError_t e = a.B <= 1 ? launch_q4_nb<KIND, 1>(ctx, s, a)
                        : a.B <= 2 ? launch_q4_nb<KIND, 2>(ctx, s, a)
                                   : launch_q4_nb<KIND, 4>(ctx, s, a);
  prof_after(ctx, kid, s);
  ctx->launches++;
  return e;
}

template <int NB>
static cudaError_t launch_q8_nb(mtp_ctx* ctx, cudaStream_t s, const StepArgs<uint16_t>& a) {
  const int G = a.H / 64;
  const int nrb_all = ((a.V + 1) / 2 + 7) / 8;
  const int grid = min(ctx->num_sms, nrb_all);
  const size_t fixed = (size_t)G * 2 * NB * 64 + (size_t)16 * ((nrb_all + grid - 1) / grid) * 4;
  const int gpc = q_gpc(G, kQ8Tile, kQ8UnitBytes);
  int stages, consumers;
  if (!q_plan((size_t)gpc * kQ8Tile, fixed, 0, &stages, &consumers)) return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)stages * gpc * kQ8Tile + fixed;
  ensure_smem((const void*)mtp_q8_lm_kernel<NB>, smem);
  return launch_pdl(mtp_q8_lm_kernel<NB>, dim3(grid), dim3(kTmaThreads), smem, s, a, stages, consumers, gpc);
}

static cudaError_t launch_q8_lm(mtp_ctx* ctx, cudaStream_t s, const StepArgs<uint16_t>& a) {
  prof_before(ctx, MTP_KERNEL_LM_HEAD, s);
  const cudaError_t e = a.B <= 1 ? launch_q8_nb<1>(ctx, s, a)
                        : a.B <= 2 ? launch_q8_nb<2>(ctx, s, a)
                                   : launch_q8_nb<4>(ctx, s, a);
  prof_after(ctx, MTP_KERNEL_LM_HEAD, s);
  ctx->launches++;
  return e;
}

static StepArgs<uint16_t> q_dims(const mtp_ctx* ctx) {
  const mtp_config& c = ctx->cfg;
  StepArgs<uint16_t> a{};
  memset(&a, 0, sizeof(a));
  a.H = c.hidden; a.q_dim = ctx->q_dim; a.kv_dim = ctx->kv_dim; a.F = c.ffn; a.V = c.vocab;
  a.n_q = c.n_q_heads; a.n_kv = c.n_kv_heads; a.hd = c.head_dim; a.bs = c.block_size; a.eps = c.eps;
  return a;
}

static size_t q4_tile_bytes(const StepArgs<uint16_t>& a, int kind) {
  const size_t C = q_cols(kind, a.H, a.q_dim, a.F);
  return (size_t)(q_pairs(kind, a.H, a.q_dim, a.kv_dim, a.F, a.V) / 8) * (C / 64) * kQ4Tile;
}

template <int KIND>
static cudaError_t repack_q4(const StepArgs<uint16_t>& a, const QCanon& cn, uint8_t* dst) {
  const long long threads = (long long)(q4_tile_bytes(a, KIND) / kQ4Tile) * 32;
  repack_q4_kernel<KIND><<<(unsigned)((threads + 255) / 256), 256>>>(a, cn, dst);
  return cudaGetLastError();
}

// Quantize the caller's bf16 weights into context-owned copies: canonical
// INT4 codes (temporary) repacked into the projection kernels' tiles, the
// INT8 embedding (kept for the row gather) and the LM head's tiles.
mtp_status quantize_head(mtp_ctx* ctx) {
  const mtp_config& c = ctx->cfg;
  const StepArgs<uint16_t> a = q_dims(ctx);
  const size_t H = c.hidden, F = c.ffn, V = c.vocab, qd = ctx->q_dim, kvd = ctx->kv_dim;
  const size_t rows[8] = {H, qd, kvd, kvd, H, F, F, H};
  const size_t cols[8] = {2 * H, H, H, H, qd, H, H, F};
  const void* src[8] = {ctx->w.w_eh, ctx->w.w_q, ctx->w.w_k, ctx->w.w_v, ctx->w.w_o, ctx->w.w_gate, ctx->w.w_up,
                        ctx->w.w_down};
  const bool tied = ctx->w.lm_head == ctx->w.embed;
  size_t toff = 0, oq[8], os[8], oz[8];
  auto ttake = [&](size_t bytes) {
    const size_t o = toff;
    toff = align_up(toff + bytes, 256);
    return o;
  };
  for (int m = 0; m < 8; ++m) {
    oq[m] = ttake(rows[m] * cols[m] / 2);
    os[m] = ttake(rows[m] * (cols[m] / 64) * 2);
    oz[m] = ttake(rows[m] * (cols[m] / 64));
  }
  const size_t o_lmq = tied ? 0 : ttake(V * H);
  const size_t o_max = ttake(sizeof(float));
  size_t off = 0, ot[6];
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  for (int k = 0; k < 5; ++k) ot[k] = take(q4_tile_bytes(a, k));
  ot[LM_HEAD] = take((size_t)(((V + 1) / 2 + 7) / 8) * (H / 64) * kQ8Tile);
  const size_t o8 = take(V * H), os8 = take(V * 2), os8l = tied ? os8 : take(V * 2);

  void* tmp = nullptr;
  if (cudaMalloc(&tmp, toff) != cudaSuccess) {
    cudaGetLastError();
    return MTP_ERR_OOM;
  }
  if (cudaMalloc(&ctx->qw_buf, off) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(tmp);
    ctx->qw_buf = nullptr;
    return MTP_ERR_OOM;
  }
  char* tb = (char*)tmp;
  char* base = (char*)ctx->qw_buf;
  QCanon cn;
  cudaError_t e = cudaSuccess;
  for (int m = 0; m < 8 && e == cudaSuccess; ++m) {
    cn.q[m] = (const uint8_t*)(tb + oq[m]);
    cn.s[m] = (const uint16_t*)(tb + os[m]);
    cn.z[m] = (const uint8_t*)(tb + oz[m]);
    e = launch_quant_int4(0, src[m], (int)rows[m], (int)cols[m], tb + oq[m], tb + os[m], tb + oz[m]);
  }
  for (int k = 0; k < 6; ++k) ctx->qw_tiles[k] = (uint8_t*)(base + ot[k]);
  ctx->qw_q8 = (int8_t*)(base + o8);
  ctx->qw_s8 = (uint16_t*)(base + os8);
  ctx->qw_s8_lm = (uint16_t*)(base + os8l);
  if (e == cudaSuccess) e = repack_q4<EH_PROJ>(a, cn, ctx->qw_tiles[EH_PROJ]);
  if (e == cudaSuccess) e = repack_q4<QKV_ROPE>(a, cn, ctx->qw_tiles[QKV_ROPE]);
  if (e == cudaSuccess) e = repack_q4<O_PROJ>(a, cn, ctx->qw_tiles[O_PROJ]);
  if (e == cudaSuccess) e = repack_q4<GATE_UP>(a, cn, ctx->qw_tiles[GATE_UP]);
  if (e == cudaSuccess) e = repack_q4<DOWN>(a, cn, ctx->qw_tiles[DOWN]);
  if (e == cudaSuccess) e = launch_quant_int8(0, ctx->w.embed, (int)V, (int)H, ctx->qw_q8, ctx->qw_s8);
  const int8_t* lmq = ctx->qw_q8;
  if (e == cudaSuccess && !tied) {
    e = launch_quant_int8(0, ctx->w.lm_head, (int)V, (int)H, tb + o_lmq, ctx->qw_s8_lm);
    lmq = (const int8_t*)(tb + o_lmq);
  }
  if (e == cudaSuccess) {
    const int G = (int)(H / 64);
    const long long threads = (long long)(((V + 1) / 2 + 7) / 8) * G * 32;
    repack_q8_kernel<<<(unsigned)((threads + 255) / 256), 256>>>(lmq, (int)V, (int)H, ctx->qw_tiles[LM_HEAD]);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    absmax_bf16_kernel<<<1, 1024>>>((const uint16_t*)ctx->w.w_norm_f, (int)H, (float*)(tb + o_max));
    e = cudaGetLastError();
  }
  float wmax = 0.0f;
  if (e == cudaSuccess) e = cudaMemcpy(&wmax, tb + o_max, sizeof(float), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  cudaFree(tmp);
  if (e != cudaSuccess) {
    cudaGetLastError();
    cudaFree(ctx->qw_buf);
    ctx->qw_buf = nullptr;
    return MTP_ERR_CUDA;
  }
  // |normalised input| <= sqrt(H) * max |w_norm_f| < 2^E: scale by 2^(15 - E)
  // so that every fp16 operand stays below 2^15.
  float sigma = 1.0f;
  const float bound = sqrtf((float)H) * wmax;
  if (bound > 0.0f && isfinite(bound)) {
    int E = 0;
    frexpf(bound, &E);
    sigma = ldexpf(1.0f, max(-60, min(60, 15 - E)));
  }
  ctx->qw_lm_sigma = sigma;
  ctx->quantized = 1;
  return MTP_OK;
}

cudaError_t launch_draft_step_q(mtp_ctx* ctx, cudaStream_t s, int B, int k, int K, const void* hidden,
                                const void* embeds, const int32_t* positions, const mtp_kv* kv,
                                const int32_t* chain_ids, int32_t* draft_ids, float* logits, float* hidden_out) {
  const mtp_config& c = ctx->cfg;
  StepArgs<uint16_t> a = q_dims(ctx);
  a.B = B; a.k = k; a.K = K; a.max_pos = c.max_pos; a.num_blocks = kv->num_blocks; a.max_blocks = kv->max_blocks;
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
  for (int i = 0; i < 6; ++i) a.qt[i] = ctx->qw_tiles[i];
  a.q8 = ctx->qw_q8; a.s8 = ctx->qw_s8; a.s8_lm = ctx->qw_s8_lm; a.lm_sigma = ctx->qw_lm_sigma;

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
