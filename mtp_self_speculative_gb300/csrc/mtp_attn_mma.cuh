// Tensor-core (mma.sync m16n8k16, bf16 in / fp32 accumulate) arithmetic of
// one 16-token block of grouped-query decode attention, head_dim 128.
//
// The G query heads of one kv head sit on the M dimension (rows G..15 are
// zero padding):
//   S^T[16 x 16 tokens] = Q[16 x 128] . K^T   -- 2 n-tiles x 8 k-steps
//   O[16 x 128]        += P[16 x 16] . V      -- 16 n-tiles, k = 16 tokens
// K and V tiles are staged by 2-D tensor-map loads with 128-byte swizzle (two
// 64-dim halves of 2 KB per tile), so the ldmatrix reads of 8 token rows hit
// distinct banks.  The S accumulators of the two token n-tiles are exactly
// the A fragment of P, so P never leaves registers.  Softmax is online with
// base-2 exponentials; log2(e)/sqrt(d) is folded into q.
//
// ("MTP (Multi-Token Prediction)", "Architecture": the attention of the MTP
// decoder layer.)
#pragma once

#include "mtp_common.cuh"

namespace mtp {

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return (uint32_t)f32_to_bf16_rne(lo) | ((uint32_t)f32_to_bf16_rne(hi) << 16);
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Shared-memory address of 16-byte chunk c (0..15 over 128 dims) of token row
// `row` (0..15) in a tile stored as two 2 KB swizzled halves.
__device__ __forceinline__ uint32_t sw_chunk(uint32_t tile, int row, int c) {
  return tile + (uint32_t)((c >> 3) * 2048 + row * 128 + (((c & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// K then V tile of pool row `row` (= (block * n_kv + g) * 16) into 8 KB at
// dst (1024-byte aligned): K halves at +0 / +2 KB, V halves at +4 / +6 KB.
__device__ __forceinline__ void tma_kv_tile(unsigned char* dst, const CUtensorMap* kmap, const CUtensorMap* vmap,
                                            int row, uint64_t* bar) {
  mbar_expect_tx(bar, 8192);
  tma_2d(dst, kmap, 0, row, bar);
  tma_2d(dst + 2048, kmap, 64, row, bar);
  tma_2d(dst + 4096, vmap, 0, row, bar);
  tma_2d(dst + 6144, vmap, 64, row, bar);
}

// A-operand fragments of the G queries of one kv head (row gi = lane / 4 is
// head gi; rows >= G and 8..15 are zero), scaled for base-2 softmax.  qh
// points at head 0 of the group; the loads bypass L1 (q may have been
// written by another CTA of the same grid).
__device__ __forceinline__ void load_q_frags(uint32_t (&qa)[8][4], const float* qh, float qscale, int lane, int G) {
  const int gi = lane >> 2, ti = lane & 3;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    if (gi < G) {
      const float* r = qh + (size_t)gi * 128 + 16 * kk + 2 * ti;
      qa[kk][0] = pack_bf16(__ldcg(r) * qscale, __ldcg(r + 1) * qscale);
      qa[kk][2] = pack_bf16(__ldcg(r + 8) * qscale, __ldcg(r + 9) * qscale);
    } else {
      qa[kk][0] = qa[kk][2] = 0u;
    }
    qa[kk][1] = qa[kk][3] = 0u;
  }
}

// One 16-token block: tokens tok0 .. tok0 + 15, those >= T_len masked.
// kt / vt: shared addresses of the swizzled K and V tiles.  Updates the
// warp's running max m_run, sum l_run (both per head row gi) and O rows.
__device__ __forceinline__ void attn_tile_mma(uint32_t kt, uint32_t vt, const uint32_t (&qa)[8][4],
                                              float (&o)[16][4], float& m_run, float& l_run, int tok0, int T_len,
                                              int lane) {
  const int ti = lane & 3;
  // S^T = Q K^T: n-tile j covers tokens 8j..8j+7
  float sc[2][4];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < 8; kk += 2) {
      const int mi = lane >> 3, ri = lane & 7;
      const int c = 2 * (kk + (mi >> 1)) + (mi & 1);
      uint32_t r0, r1, r2, r3;
      ldsm_x4(sw_chunk(kt, 8 * j + ri, c), r0, r1, r2, r3);
      mma_bf16(sc[j], qa[kk], r0, r1);
      mma_bf16(sc[j], qa[kk + 1], r2, r3);
    }
  }
  // online softmax on row gi (tokens 2ti, 2ti+1 of each n-tile); rows 8..15 are padding
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int tok = tok0 + 8 * j + 2 * ti + e;
      if (tok >= T_len) sc[j][e] = -INFINITY;
      mx = fmaxf(mx, sc[j][e]);
    }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const float m_new = fmaxf(m_run, mx);
  const float corr = (m_run == -INFINITY) ? 0.0f : exp2f(m_run - m_new);
  float p[2][2], rs = 0.0f;
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      p[j][e] = (sc[j][e] == -INFINITY) ? 0.0f : exp2f(sc[j][e] - m_new);
      rs += p[j][e];
    }
  rs += __shfl_xor_sync(0xffffffffu, rs, 1);
  rs += __shfl_xor_sync(0xffffffffu, rs, 2);
  l_run = l_run * corr + rs;
  m_run = m_new;
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    o[n][0] *= corr;
    o[n][1] *= corr;
  }
  uint32_t pa[4];
  pa[0] = pack_bf16(p[0][0], p[0][1]);
  pa[1] = 0u;
  pa[2] = pack_bf16(p[1][0], p[1][1]);
  pa[3] = 0u;
  // O += P V: n-tile n covers dims 8n..8n+7
#pragma unroll
  for (int c = 0; c < 16; c += 2) {
    const int mi = lane >> 3, ri = lane & 7;
    const int tok = 8 * (mi & 1) + ri;
    uint32_t r0, r1, r2, r3;
    ldsm_x4_t(sw_chunk(vt, tok, c + (mi >> 1)), r0, r1, r2, r3);
    mma_bf16(o[c], pa, r0, r1);
    mma_bf16(o[c + 1], pa, r2, r3);
  }
}

}  // namespace mtp
