// Tensor-core (tcgen05) path of the draft step for batches of 16..256
// requests, bf16 weights, head_dim 128.
//
// Every projection of "MTP (Multi-Token Prediction)", "Architecture" becomes
// a skinny GEMM  D[128-row weight tile, N] = W_tile . X^T  with the weights
// as the 128-row A operand and the (padded) batch as N: the weight stream is
// read once per draft step, the activations (<= 2.6 MB) stay in L2.
//
// Kernel organisation (one CTA per SM, 6 warps):
//   warp 0   TMA producer: 2-D tensor-map loads of the weight tile (128 x 64
//            bf16, 128-byte swizzle) and the activation tile (N x 64) into a
//            ring of shared-memory stages (full/empty mbarriers).  The weight
//            loads of the first stages are issued before the programmatic
//            dependency wait, so the stream starts while the previous kernel
//            drains.
//   warp 1   owns the TMEM allocation (2 accumulators of N fp32 columns) and
//            issues tcgen05.mma (M=128, N, K=16) from one thread; commits
//            free the stages and publish finished accumulators.
//   warps 2-5 epilogue: tcgen05.ld of the accumulator rows (warp w reads TMEM
//            lanes 32*(w%4)..+31), fused epilogue per kind, stores.
// Work split (no global fix-up, deterministic):
//   * kinds with at least as many 128-row tiles as CTAs (LM head, large
//     FFNs) take whole tiles, a balanced contiguous range per CTA, with two
//     TMEM accumulators so the epilogue of one tile overlaps the next tile's
//     MMAs (the LM head's ranges are counted in 16-row units, its last tile
//     per CTA loaded as 16-row boxes);
//   * kinds with fewer tiles than CTAs are split along K over a thread-block
//     cluster of S <= 8 CTAs per tile: each CTA accumulates its K-slice in
//     TMEM, parks the partial tile in its (drained) stage memory, and after a
//     cluster barrier CTA rank r sums column slice r over the S partials in
//     rank order through distributed shared memory and applies the epilogue.
// Two CTAs per SM whenever the ring and TMEM allow it.
//
// Epilogue kinds: EH_PROJ (x = D), QKV_ROPE (rotary pairs (i, i+64) of one
// head exchanged through shared memory; q stored fp32, k/v rounded to bf16
// into the paged cache), O_PROJ (h1 = x + D), GATE_UP (tile = 64 gate rows +
// the matching 64 up rows; act = silu(g) * u stored bf16), DOWN (h2 = h1 + D),
// LM_HEAD (logits; per-column argmax with warp max-reduce + ballot, CTA best
// in shared memory, one 64-bit atomicMax per request per CTA, last CTA writes
// the draft ids).
//
// The eh_proj input (two RMSNorms with their own scales) comes from a small
// prep kernel; every other RMSNorm is folded into the neighbouring GEMMs: the
// producing GEMM's epilogue writes bf16(y * w) and per-tile sums of y^2, the
// consuming GEMM scales its accumulators by each request's RMS factor.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "mtp_common.cuh"

namespace mtp {

enum TcKind { TC_EH = 0, TC_QKV = 1, TC_O = 2, TC_GU = 3, TC_DOWN = 4, TC_LM = 5 };

constexpr int kTcThreads = 192;
constexpr int kTcEpiThreads = 128;
constexpr uint32_t kTcWaitLimit = 1u << 26;
constexpr int kTcTileBytesA = 128 * 64 * 2;   // 16 KB

struct TcMaps {
  CUtensorMap a0, a1, a2;  // weight maps (QKV: q, k, v; GATE_UP: gate, up)
  CUtensorMap b;           // activation map [B rows, C] bf16
};

struct TcArgs {
  int kind;
  int B, NT, H, q_dim, kv_dim, F, V, n_q, n_kv, bs, k, K;
  int C, nkb, n_tiles, stages, max_pos, num_blocks, max_blocks;
  int ksplit;              // 1: whole tiles per CTA; S > 1: cluster of S CTAs per tile
  const int32_t* positions;
  int32_t* draft_ids;
  float* logits;
  float* hidden_out;
  uint16_t* k_pool;
  uint16_t* v_pool;
  const int32_t* block_table;
  const int32_t* seq_len;
  int32_t* pending;
  float *hid, *x, *q, *h1;
  uint16_t* act_bf16;
  unsigned long long* lm_keys;
  int* lm_cnt;
  int* err;
  int* req_bad;
  const float2* rope;
  // RMSNorm of the next projection's input, folded into this one:
  // EH, O and DOWN (producers) also write xn_out = bf16(y * w_next) and, per
  // 128-row tile and request, the sum of y^2 into ssq[tile * B + b]; QKV, GU
  // and the LM head (consumers, scale_in) multiply their accumulators by
  // rsqrt(sum over tiles / H + eps) of each request.
  const uint16_t* w_next;
  uint16_t* xn_out;
  float* ssq;
  int scale_in;
  float eps;
};

// ------------------------------------------------------------ primitives

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// The same with an L2 cache policy (weights: evict first).
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;               // leading offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;     // 1024 B between 8-row groups
  d |= (uint64_t)1 << 46;               // descriptor version
  d |= (uint64_t)2 << 61;               // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ uint32_t ordered_bits(float v) {
  if (v == 0.0f) v = 0.0f;
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Bounded wait that also gives up once another role has given up.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t i = 0; i < kTcWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 1023) == 1023 && *abort_flag) return false;
  }
  return false;
}


// ----------------------------------------------------------- epilogues


// Per-request metadata of the QKV epilogue, cached in shared memory once per
// CTA: rotary position (-1: out of range) and the element offset of the new
// KV slot in the pools at kv head 0 (-1: invalid slot or pending mismatch).
struct QkvMeta {
  int pos[256];
  long long kv[256];
};

__device__ void qkv_meta_fill(const TcArgs& a, QkvMeta* meta, int tid, int nthreads) {
  for (int b = tid; b < a.B; b += nthreads) {
    int pos = a.positions[b] + a.k - 1;
    if (pos < 0 || pos >= a.max_pos) {
      set_error(a.err, MTP_ERR_CAPACITY);
      pos = -1;
    }
    meta->pos[b] = pos;
    long long kvoff = -1;
    if (__ldcg(a.req_bad + b) || a.pending[b] != a.k - 1) {
      set_error(a.err, MTP_ERR_DEVICE_ARGS);
    } else {
      const int slot = a.seq_len[b] + a.k - 1;
      const int bi = slot / a.bs, off = slot - bi * a.bs;
      const int blk = (slot >= 0 && bi < a.max_blocks) ? a.block_table[(size_t)b * a.max_blocks + bi] : -1;
      if (blk < 0 || blk >= a.num_blocks) set_error(a.err, MTP_ERR_CAPACITY);
      else kvoff = ((long long)blk * a.n_kv * a.bs + off) * 128;
    }
    meta->kv[b] = kvoff;
  }
}

struct EpiCtx {
  int tile, m, lane, quarter;  // m = row of the tile held by this thread
  int row0, row_end;           // LM head: first row of the tile, end of the CTA's rows
  float* xbuf;                 // [64][16] exchange buffer
  const float* rms;            // [B] RMS factor per request (1 unless folded)
  unsigned long long* cta_best;
  const QkvMeta* meta;
};

// Rotary factors of QKV pair (i, i + 64) of head `tile` for batch row b
// (identity for value heads, gate/up pairs and positions out of range).
__device__ __forceinline__ float2 tc_pair_rope(const TcArgs& a, const QkvMeta* meta, int tile, int i, int b) {
  if (a.kind != TC_QKV || tile >= a.n_q + a.n_kv) return make_float2(1.0f, 0.0f);
  const int pos = meta->pos[b];
  if (pos < 0) return make_float2(1.0f, 0.0f);
  return __ldg(a.rope + (size_t)pos * 64 + i);
}

// Pair kinds, one output pair: rows i and i + 64 of the tile for batch row b;
// cs = tc_pair_rope(...).
__device__ __forceinline__ void tc_pair_store_cs(const TcArgs& a, const QkvMeta* meta, int tile, int i, int b,
                                                 float v0, float v1, float2 cs) {
  if (a.kind == TC_GU) {
    const int f = tile * 64 + i;
    if (f < a.F)
      MTP_STORE(a.err, a.act_bf16, (size_t)b * a.F + f, (long long)a.B * a.F, f32_to_bf16_rne(v0 / (1.0f + __expf(-v0)) * v1));
    return;
  }
  // TC_QKV: tile = head
  const int grp = tile;
  const int pos = meta->pos[b];
  if (pos < 0) return;
  if (grp < a.n_q) {
    const size_t qo = (size_t)b * a.q_dim + grp * 128;
    const long long nQ = (long long)a.B * a.q_dim;
    MTP_STORE(a.err, a.q, qo + i, nQ, v0 * cs.x - v1 * cs.y);
    MTP_STORE(a.err, a.q, qo + i + 64, nQ, v1 * cs.x + v0 * cs.y);
    return;
  }
  const long long kvoff = meta->kv[b];
  if (kvoff < 0) return;
  float o0 = v0, o1 = v1;
  uint16_t* pool;
  int g;
  if (grp < a.n_q + a.n_kv) {
    o0 = v0 * cs.x - v1 * cs.y;
    o1 = v1 * cs.x + v0 * cs.y;
    pool = a.k_pool;
    g = grp - a.n_q;
  } else {
    pool = a.v_pool;
    g = grp - a.n_q - a.n_kv;
  }
  const long long e = kvoff + (long long)g * a.bs * 128 + i;
  const long long nP = (long long)a.num_blocks * a.n_kv * a.bs * 128;
  MTP_STORE(a.err, pool, e, nP, f32_to_bf16_rne(o0));
  MTP_STORE(a.err, pool, e + 64, nP, f32_to_bf16_rne(o1));
}

// Residual input of plain output row r for batch row b (x for O, h1 for
// DOWN, none for EH).
__device__ __forceinline__ float tc_plain_residual(const TcArgs& a, int r, int b) {
  if (r >= a.H || a.kind == TC_EH) return 0.0f;
  const size_t o = (size_t)b * a.H + r;
  return __ldcg(a.kind == TC_O ? a.x + o : a.h1 + o);
}

// Plain kinds, one output: row r of the layer output for batch row b;
// res = tc_plain_residual(...).
__device__ __forceinline__ void tc_plain_store_res(const TcArgs& a, int r, int b, float v, float res) {
  if (r >= a.H) return;
  const size_t o = (size_t)b * a.H + r;
  const long long nBH = (long long)a.B * a.H;
  if (a.kind == TC_EH) {
    MTP_STORE(a.err, a.x, o, nBH, v);
  } else if (a.kind == TC_O) {
    MTP_STORE(a.err, a.h1, o, nBH, res + v);
  } else {
    const float hv = res + v;
    MTP_STORE(a.err, a.hid, o, nBH, hv);
    if (a.hidden_out && a.k == a.K) MTP_STORE(a.err, a.hidden_out, o, nBH, hv);
  }
}


// Apply the epilogue to 16 columns [c0, c0 + 16) of this thread's row.
__device__ void tc_epilogue(const TcArgs& a, const EpiCtx& e, int c0, const float (&v)[16]) {
  const int kind = a.kind;
  if (kind == TC_EH || kind == TC_O || kind == TC_DOWN) {
    // all sixteen residuals are loaded before the first store; the outputs'
    // squares are summed over the tile's 128 rows (warp, then the four
    // warps through xbuf) for the next RMSNorm
    const int r = e.tile * 128 + e.m;
    const float wn = bf16_lo((uint32_t)__ldg(a.w_next + r));
    float res[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) res[j] = (c0 + j < a.B) ? tc_plain_residual(a, r, c0 + j) : 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float y = (kind == TC_EH) ? v[j] : res[j] + v[j];
      if (c0 + j < a.B) {
        tc_plain_store_res(a, r, c0 + j, v[j], res[j]);
        MTP_STORE(a.err, a.xn_out, (size_t)(c0 + j) * a.H + r, (long long)a.B * a.H, f32_to_bf16_rne(y * wn));
      }
      const float q = warp_sum((c0 + j < a.B) ? y * y : 0.0f);
      if (e.lane == 0) e.xbuf[e.quarter * 16 + j] = q;
    }
    epi_bar();
    const int t = threadIdx.x - 64;
    if (t < 16 && c0 + t < a.B)
      MTP_STORE(a.err, a.ssq, (size_t)e.tile * a.B + c0 + t, (long long)(a.H / 128) * a.B,
                e.xbuf[t] + e.xbuf[16 + t] + e.xbuf[32 + t] + e.xbuf[48 + t]);
    epi_bar();
    return;
  }
  if (kind == TC_LM) {
    // rows at or past row_end are another CTA's (or past the vocabulary):
    // their accumulators hold whatever the stage's unused rows held
    const int r = e.row0 + e.m;
    const bool row_ok = r < e.row_end;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int b = c0 + j;
      if (b >= a.B) continue;  // uniform across the warp
      const float z = v[j] * e.rms[b];
      if (a.logits && row_ok)
        MTP_STORE(a.err, a.logits, ((size_t)b * a.K + (a.k - 1)) * a.V + r, (long long)a.B * a.K * a.V, z);
      const uint32_t ord = row_ok ? ordered_bits(z) : 0u;
      const uint32_t mx = __reduce_max_sync(0xffffffffu, ord);
      const uint32_t bal = __ballot_sync(0xffffffffu, ord == mx);
      if (e.lane == (b & 31)) {
        const uint32_t row = (uint32_t)(e.row0 + e.quarter * 32 + (__ffs(bal) - 1));
        const unsigned long long key = ((unsigned long long)mx << 32) | (unsigned long long)(0xFFFFFFFFu - row);
        atomicMax(e.cta_best + b, key);
      }
    }
    return;
  }
  // Pair kinds: rows m and m + 64 of the tile belong together.
  const bool upper = e.m >= 64;
  if (upper) {
#pragma unroll
    for (int j = 0; j < 16; ++j) e.xbuf[(e.m - 64) * 16 + j] = v[j];
  }
  epi_bar();
  if (!upper) {
    float2 cs[16];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      cs[j] = (c0 + j < a.B) ? tc_pair_rope(a, e.meta, e.tile, e.m, c0 + j) : make_float2(1.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (c0 + j < a.B) {
        const float sc = e.rms[c0 + j];
        tc_pair_store_cs(a, e.meta, e.tile, e.m, c0 + j, v[j] * sc, e.xbuf[e.m * 16 + j] * sc, cs[j]);
      }
  }
  epi_bar();
}

__device__ __forceinline__ uint32_t mapa(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// Read four floats of a peer's shared memory.  Volatile keeps it after the
// cluster barrier; no memory clobber, so independent loads and stores around
// it can overlap.
__device__ __forceinline__ float4 ld_dsmem4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}

// Four consecutive output rows r..r+3 (r % 4 == 0, all below H) of a plain
// kind for batch row b.
__device__ __forceinline__ float4 tc_plain_residual4(const TcArgs& a, int r, int b) {
  if (a.kind == TC_EH) return make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  const size_t o = (size_t)b * a.H + r;
  return __ldcg(reinterpret_cast<const float4*>((a.kind == TC_O ? a.x : a.h1) + o));
}
// Stores the four outputs, their bf16(y * w_next) copy for the next GEMM, and
// returns the sum of their squares.
__device__ __forceinline__ float tc_plain_store4(const TcArgs& a, int r, int b, float4 v, float4 res) {
  const size_t o = (size_t)b * a.H + r;
  const float4 t = (a.kind == TC_EH) ? v : make_float4(res.x + v.x, res.y + v.y, res.z + v.z, res.w + v.w);
  if (!MTP_IN_BOUNDS(a.err, (long long)o + 3, (long long)a.B * a.H)) return 0.0f;
  if (a.kind == TC_EH) {
    *reinterpret_cast<float4*>(a.x + o) = t;
  } else if (a.kind == TC_O) {
    *reinterpret_cast<float4*>(a.h1 + o) = t;
  } else {
    *reinterpret_cast<float4*>(a.hid + o) = t;
    if (a.hidden_out && a.k == a.K) *reinterpret_cast<float4*>(a.hidden_out + o) = t;
  }
  const uint2 wn = __ldg(reinterpret_cast<const uint2*>(a.w_next + r));
  uint2 xo;
  xo.x = (uint32_t)f32_to_bf16_rne(t.x * bf16_lo(wn.x)) | ((uint32_t)f32_to_bf16_rne(t.y * bf16_hi(wn.x)) << 16);
  xo.y = (uint32_t)f32_to_bf16_rne(t.z * bf16_lo(wn.y)) | ((uint32_t)f32_to_bf16_rne(t.w * bf16_hi(wn.y)) << 16);
  *reinterpret_cast<uint2*>(a.xn_out + o) = xo;
  return t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- kernel

// Work of one CTA: a list of segments (tile, k-blocks [k0, k1)).
//   ksplit == 1: whole tiles, a balanced contiguous range per CTA.
//   ksplit == S: CTA blockIdx.x is rank r of the cluster for tile
//                blockIdx.x / S and owns k-blocks [r*nkb/S, (r+1)*nkb/S).
//   LM head: a balanced contiguous range of rows [r0, r1) in 16-row units,
//                as tiles of 128 rows from r0 (the last one may be shorter):
//                every CTA streams within 16 rows of the same bytes.
struct SegList {
  int t0, count, k0, k1;  // ksplit == 1: tiles t0..t0+count-1 with [0, nkb)
  int r0, r1;             // LM head: the CTA's rows
};
__device__ __forceinline__ SegList seg_list(const TcArgs& a) {
  SegList L;
  L.r0 = L.r1 = 0;
  if (a.kind == TC_LM) {
    const long long G = gridDim.x, U = (a.V + 15) / 16;
    const int u0 = (int)(((long long)blockIdx.x * U) / G), u1 = (int)(((long long)(blockIdx.x + 1) * U) / G);
    L.r0 = min(16 * u0, a.V);
    L.r1 = min(16 * u1, a.V);
    L.t0 = 0;
    L.count = (L.r1 - L.r0 + 127) / 128;
    L.k0 = 0;
    L.k1 = a.nkb;
    return L;
  }
  if (a.ksplit == 1) {
    const long long G = gridDim.x;
    L.t0 = (int)(((long long)blockIdx.x * a.n_tiles) / G);
    L.count = (int)(((long long)(blockIdx.x + 1) * a.n_tiles) / G) - L.t0;
    L.k0 = 0;
    L.k1 = a.nkb;
  } else {
    const int r = blockIdx.x % a.ksplit;
    L.t0 = blockIdx.x / a.ksplit;
    L.count = 1;
    L.k0 = (int)(((long long)r * a.nkb) / a.ksplit);
    L.k1 = (int)(((long long)(r + 1) * a.nkb) / a.ksplit);
  }
  return L;
}

__global__ void __launch_bounds__(kTcThreads, 1) mtp_tc_proj_kernel(const __grid_constant__ TcMaps maps, const TcArgs a) {
  extern __shared__ __align__(1024) unsigned char tc_smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[8], empty_bar[8], accf_bar[2], acce_bar[2];
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;
  __shared__ int last_flag, stop_snap;
  __shared__ float xbuf[64 * 16];
  __shared__ float s_rms[256];
  __shared__ unsigned long long cta_best[256];
  __shared__ QkvMeta qkv_meta;

  unsigned char* smem = (unsigned char*)(((uintptr_t)tc_smem_raw + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = a.NT, NS = a.stages;
  const uint32_t bytes_b = (uint32_t)NT * 128;
  const uint32_t stage_bytes = kTcTileBytesA + bytes_b;
  const int nacc = (a.ksplit == 1) ? 2 : 1;
  const uint32_t need = (uint32_t)(nacc * NT);
  const uint32_t tmem_cols = need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : need <= 256 ? 256 : 512;

  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int st = 0; st < NS; ++st) {
      mbar_init(&full_bar[st], 1);
      mbar_init(&empty_bar[st], 1);
    }
    mbar_init(&accf_bar[0], 1);
    mbar_init(&accf_bar[1], 1);
    mbar_init(&acce_bar[0], 4);
    mbar_init(&acce_bar[1], 4);
    abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < 256; i += kTcThreads) cta_best[i] = 0ull;
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_base)),
                 "r"(tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const SegList L = seg_list(a);
  const int per_seg = L.k1 - L.k0;

  if (warp == 0) {
    if (lane == 0) {
      // producer: segments in order, their k-blocks in order.  Weight tiles
      // are read once per step: evict first, so that the activation operand
      // every tile re-reads stays in L2.
      const uint64_t pol = l2_evict_first_policy();
      auto issue_a = [&](int st, int tile, int kb) {
        unsigned char* dst = smem + (size_t)st * stage_bytes;
        if (a.kind == TC_GU) {
          tma_load_2d_hint(dst, &maps.a0, kb * 64, tile * 64, &full_bar[st], pol);
          tma_load_2d_hint(dst + 8192, &maps.a1, kb * 64, tile * 64, &full_bar[st], pol);
        } else if (a.kind == TC_QKV) {
          if (tile < a.n_q) tma_load_2d_hint(dst, &maps.a0, kb * 64, tile * 128, &full_bar[st], pol);
          else if (tile < a.n_q + a.n_kv)
            tma_load_2d_hint(dst, &maps.a1, kb * 64, (tile - a.n_q) * 128, &full_bar[st], pol);
          else tma_load_2d_hint(dst, &maps.a2, kb * 64, (tile - a.n_q - a.n_kv) * 128, &full_bar[st], pol);
        } else if (a.kind == TC_LM) {
          // tile = segment: 128 rows from r0 + 128 * seg; a shorter last
          // segment loads only its own 16-row boxes (map a1) -- each lands at
          // a 2 KB offset, so the 128-byte swizzle pattern is the same
          const int rb = L.r0 + 128 * tile;
          const int nr = min(128, L.r1 - rb);
          if (nr == 128) {
            tma_load_2d_hint(dst, &maps.a0, kb * 64, rb, &full_bar[st], pol);
          } else {
            for (int i = 0; 16 * i < nr; ++i)
              tma_load_2d_hint(dst + 2048 * i, &maps.a1, kb * 64, rb + 16 * i, &full_bar[st], pol);
          }
        } else {
          tma_load_2d_hint(dst, &maps.a0, kb * 64, tile * 128, &full_bar[st], pol);
        }
      };
      // bytes of the A operand of a segment (tile index for the other kinds)
      auto a_bytes = [&](int seg) -> uint32_t {
        if (a.kind != TC_LM) return (uint32_t)kTcTileBytesA;
        const int nr = min(128, L.r1 - (L.r0 + 128 * seg));
        return nr == 128 ? (uint32_t)kTcTileBytesA : (uint32_t)(((nr + 15) / 16) * 2048);
      };
      auto issue_b = [&](int st, int kb) {
        tma_load_2d(smem + (size_t)st * stage_bytes + kTcTileBytesA, &maps.b, kb * 64, 0, &full_bar[st]);
      };
      const int n_it = L.count * per_seg;
      const int pre = n_it < NS ? n_it : NS;
      for (int it = 0; it < pre; ++it) {
        mbar_expect_tx(&full_bar[it], a_bytes(it / per_seg) + bytes_b);
        issue_a(it, L.t0 + it / per_seg, L.k0 + it % per_seg);
      }
      pdl_wait();
      for (int it = 0; it < pre; ++it) issue_b(it, L.k0 + it % per_seg);
      for (int it = pre; it < n_it; ++it) {
        const int st = it % NS;
        if (!tc_wait(&empty_bar[st], ((it / NS) & 1) ^ 1, &abort_flag)) {
          abort_flag = 1;
          set_error(a.err, MTP_ERR_TIMEOUT);
          break;
        }
        mbar_expect_tx(&full_bar[st], a_bytes(it / per_seg) + bytes_b);
        issue_a(st, L.t0 + it / per_seg, L.k0 + it % per_seg);
        issue_b(st, L.k0 + it % per_seg);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issuer
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NT >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
      int it = 0;
      bool ok = true;
      for (int seg = 0; seg < L.count && ok; ++seg) {
        const int buf = seg & 1;
        if (!tc_wait(&acce_bar[buf], ((seg >> 1) & 1) ^ 1, &abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * NT);
        for (int kk_ = 0; kk_ < per_seg; ++kk_, ++it) {
          const int st = it % NS;
          if (!tc_wait(&full_bar[st], (it / NS) & 1, &abort_flag)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa_ = smem_addr(smem + (size_t)st * stage_bytes);
          const uint32_t sb_ = sa_ + kTcTileBytesA;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma(d, sw128_desc(sa_ + kk * 32), sw128_desc(sb_ + kk * 32), idesc, (kk_ > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty_bar[st]);
        }
        if (!ok) break;
        tc_commit(&accf_bar[buf]);
      }
      if (!ok) {
        abort_flag = 1;
        set_error(a.err, MTP_ERR_TIMEOUT);
      }
    }
  } else {
    // epilogue warps 2..5
    pdl_wait();
    const int quarter = warp & 3;
    const int m = quarter * 32 + lane;
    const int epi_tid = threadIdx.x - 64;
    // RMS factor of each request's input (consumers of a folded RMSNorm):
    // the tiles' sums of squares in tile order
    const int ntile_h = a.H / 128;
    for (int b = epi_tid; b < a.B; b += kTcEpiThreads) {
      float r = 1.0f;
      if (a.scale_in) {
        float t = 0.0f;
#pragma unroll 8
        for (int ti = 0; ti < ntile_h; ++ti) t += __ldcg(a.ssq + (size_t)ti * a.B + b);
        r = rsqrtf(t / (float)a.H + a.eps);
      }
      s_rms[b] = r;
    }
    epi_bar();
    EpiCtx e;
    e.m = m;
    e.lane = lane;
    e.quarter = quarter;
    e.xbuf = xbuf;
    e.rms = s_rms;
    e.cta_best = cta_best;
    e.meta = &qkv_meta;
    if (a.kind == TC_QKV) {
      qkv_meta_fill(a, &qkv_meta, epi_tid, kTcEpiThreads);
      epi_bar();
    }
    for (int seg = 0; seg < L.count; ++seg) {
      const int buf = seg & 1;
      e.tile = L.t0 + seg;
      e.row0 = L.r0 + 128 * seg;
      e.row_end = L.r1;
      bool ok = tc_wait(&accf_bar[buf], (seg >> 1) & 1, &abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && lane == 0) {
        abort_flag = 1;
        set_error(a.err, MTP_ERR_TIMEOUT);
      }
      // the four epilogue warps take the same decision (named barriers follow)
      epi_bar();
      if (epi_tid == 0) stop_snap = abort_flag;
      epi_bar();
      if (stop_snap) break;
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * NT);
      if (a.ksplit == 1) {
        for (int c0 = 0; c0 < NT; c0 += 16) {
          float v[16];
          tmem_ld16(tbase + c0, v);
          tc_epilogue(a, e, c0, v);
        }
      } else {
        // partial tile -> shared memory (the stages are drained): part[c][row]
        float* part = reinterpret_cast<float*>(smem);
        for (int c0 = 0; c0 < NT; c0 += 16) {
          float v[16];
          tmem_ld16(tbase + c0, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) part[(c0 + j) * 128 + m] = v[j];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&acce_bar[buf])) : "memory");
    }
    if (a.kind == TC_LM) {
      epi_bar();
      for (int b = epi_tid; b < a.B; b += kTcEpiThreads)
        if (cta_best[b]) atomicMax(a.lm_keys + b, cta_best[b]);
      __threadfence();
      epi_bar();
      if (epi_tid == 0) last_flag = (atomicAdd(a.lm_cnt, 1) == (int)gridDim.x - 1);
      epi_bar();
      if (last_flag) {
        __threadfence();
        for (int b = epi_tid; b < a.B; b += kTcEpiThreads) {
          const unsigned long long key = atomicExch(a.lm_keys + b, 0ull);
          MTP_STORE(a.err, a.draft_ids, (size_t)b * a.K + (a.k - 1), (long long)a.B * a.K, (int32_t)key_index(key));
          if (!__ldcg(a.req_bad + b)) MTP_STORE(a.err, a.pending, b, a.B, a.k);
        }
        if (epi_tid == 0) atomicExch(a.lm_cnt, 0);
      }
    }
  }

  if (a.ksplit > 1) {
    // Cluster reduction: every CTA of the cluster holds one k-slice partial of
    // the same tile in shared memory; rank r sums the column slice
    // [r*NT/S, (r+1)*NT/S) over ranks 0..S-1 in order (deterministic) through
    // distributed shared memory and applies the epilogue to it.
    __syncwarp();
    cluster_sync_all();
    if (warp >= 2 && !abort_flag) {
      const int S = a.ksplit;
      const int r = blockIdx.x % S;
      const int tile = blockIdx.x / S;
      const int c_lo = (r * NT) / S, c_hi = ((r + 1) * NT) / S;
      const int rows = (a.kind == TC_QKV || a.kind == TC_GU) ? 64 : 128;
      const uint32_t part_local = smem_addr(smem);
      uint32_t base[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) base[j] = (j < S) ? mapa(part_local, (uint32_t)j) : 0u;
      // item = (column, four consecutive rows): one float4 load per rank, all
      // issued before the sum; then the item's side inputs and its stores
      const int nq = rows / 4;
      const int items = (c_hi - c_lo) * nq;
      for (int idx = threadIdx.x - 64; idx < items; idx += kTcEpiThreads) {
        const int c = c_lo + idx / nq, mq = (idx % nq) * 4;
        if (c >= a.B) continue;
        const uint32_t off0 = (uint32_t)((c * 128 + mq) * 4), off1 = off0 + 64 * 4;
        float4 r0[8], r1[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < S) {
            r0[j] = ld_dsmem4(base[j] + off0);
            if (rows == 64) r1[j] = ld_dsmem4(base[j] + off1);
          }
        float4 v0 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), v1 = v0;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < S) {
            v0.x += r0[j].x; v0.y += r0[j].y; v0.z += r0[j].z; v0.w += r0[j].w;
            if (rows == 64) { v1.x += r1[j].x; v1.y += r1[j].y; v1.z += r1[j].z; v1.w += r1[j].w; }
          }
        if (rows == 64) {
          float2 cs[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) cs[e] = tc_pair_rope(a, &qkv_meta, tile, mq + e, c);
          const float sc = a.scale_in ? s_rms[c] : 1.0f;
          tc_pair_store_cs(a, &qkv_meta, tile, mq + 0, c, v0.x * sc, v1.x * sc, cs[0]);
          tc_pair_store_cs(a, &qkv_meta, tile, mq + 1, c, v0.y * sc, v1.y * sc, cs[1]);
          tc_pair_store_cs(a, &qkv_meta, tile, mq + 2, c, v0.z * sc, v1.z * sc, cs[2]);
          tc_pair_store_cs(a, &qkv_meta, tile, mq + 3, c, v0.w * sc, v1.w * sc, cs[3]);
        } else {
          // the warp holds all 128 rows of column c: its sum of squares is the
          // tile's partial for the next RMSNorm
          const int r = tile * 128 + mq;
          const float q = warp_sum(tc_plain_store4(a, r, c, v0, tc_plain_residual4(a, r, c)));
          if (lane == 0) MTP_STORE(a.err, a.ssq, (size_t)tile * a.B + c, (long long)(a.H / 128) * a.B, q);
        }
      }
    }
    __syncwarp();
    cluster_sync_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols));
  }
}

// ------------------------------------------------------------ prep kernels

// xin[b] = [bf16(RMSNorm(h_b) w_h), bf16(RMSNorm(e_b) w_e)], e_b = embeds_in (k == 1)
// or the embedding row of the previous draft / chain token.
struct PrepEhArgs {
  int B, H, V, k, K;
  const uint16_t* hidden_in;
  const uint16_t* embeds_in;
  const float* hid;
  const int32_t* chain_ids;
  const int32_t* draft_ids;
  const uint16_t* embed;
  const uint16_t* w_h;
  const uint16_t* w_e;
  float eps;
  uint16_t* out;  // [B, 2H]
  int* err;
  const int32_t* pending;
  int* req_bad;   // written at step 1: pending was not 0 on entry
};



// Single pass: each thread keeps its (up to kPrepPer) elements in registers
// between the sum of squares and the scaled bf16 store.  512 threads, 4
// contiguous elements per thread per slot (16-byte fp32 / 8-byte bf16 I/O).
constexpr int kPrepThreads = 512;
constexpr int kPrepPer = 8;  // slots of 4 elements: rows up to 512 * 4 * 8 = 16384 wide

__device__ __forceinline__ float prep_sum(float v, float* red) {
  v = warp_sum(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = ((threadIdx.x & 31) < (kPrepThreads / 32)) ? red[threadIdx.x & 31] : 0.0f;
  return warp_sum(t);
}

__device__ __forceinline__ void store_bf16x4(uint16_t* dst, float a0, float a1, float a2, float a3) {
  uint2 u;
  u.x = (uint32_t)f32_to_bf16_rne(a0) | ((uint32_t)f32_to_bf16_rne(a1) << 16);
  u.y = (uint32_t)f32_to_bf16_rne(a2) | ((uint32_t)f32_to_bf16_rne(a3) << 16);
  *reinterpret_cast<uint2*>(dst) = u;
}

// Normalise one row of n (multiple of 4) elements given as fp32 (src32) or
// bf16 (src16) and write bf16(x * rsqrt(mean x^2 + eps) * w) to dst.
__device__ __forceinline__ void prep_row(const float* src32, const uint16_t* src16, const uint16_t* w, uint16_t* dst,
                                         int n, float eps, float* red) {
  float4 v[kPrepPer];
  float ss = 0.0f;
#pragma unroll
  for (int j = 0; j < kPrepPer; ++j) {
    const int i = (threadIdx.x + j * kPrepThreads) * 4;
    if (i < n) {
      if (src32) {
        v[j] = *reinterpret_cast<const float4*>(src32 + i);
      } else {
        const uint2 u = *reinterpret_cast<const uint2*>(src16 + i);
        v[j] = make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
      }
      ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
    }
  }
  const float sc = rsqrtf(prep_sum(ss, red) / (float)n + eps);
#pragma unroll
  for (int j = 0; j < kPrepPer; ++j) {
    const int i = (threadIdx.x + j * kPrepThreads) * 4;
    if (i < n) {
      const uint2 wu = *reinterpret_cast<const uint2*>(w + i);
      store_bf16x4(dst + i, v[j].x * sc * bf16_lo(wu.x), v[j].y * sc * bf16_hi(wu.x), v[j].z * sc * bf16_lo(wu.y),
                   v[j].w * sc * bf16_hi(wu.y));
    }
  }
}

__global__ void __launch_bounds__(kPrepThreads) prep_eh_kernel(const PrepEhArgs a) {
  __shared__ float red[kPrepThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x;
  if (a.k == 1 && threadIdx.x == 0) a.req_bad[b] = (a.pending[b] != 0);
  uint16_t* out = a.out + (size_t)b * 2 * a.H;
  // hidden half: step 1 reads the caller's bf16 state, later steps the fp32 recursion
  if (a.k == 1) prep_row(nullptr, a.hidden_in + (size_t)b * a.H, a.w_h, out, a.H, a.eps, red);
  else prep_row(a.hid + (size_t)b * a.H, nullptr, a.w_h, out, a.H, a.eps, red);
  // embedding half
  const uint16_t* e;
  if (a.k == 1) {
    e = a.embeds_in + (size_t)b * a.H;
  } else {
    int id = a.chain_ids ? a.chain_ids[(size_t)b * (a.K - 1) + (a.k - 2)] : a.draft_ids[(size_t)b * a.K + (a.k - 2)];
    if (id < 0 || id >= a.V) {
      if (threadIdx.x == 0) set_error(a.err, MTP_ERR_DEVICE_ARGS);
      id = 0;
    }
    e = a.embed + (size_t)id * a.H;
  }
  prep_row(nullptr, e, a.w_e, out + a.H, a.H, a.eps, red);
}


// -------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static bool get_encode() {
  if (g_encode) return true;
  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      !fn)
    return false;
  g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  return true;
}

// 2-D bf16 map over [rows, cols] with box [box_rows, 64] and 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  if (!get_encode()) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_supported(const mtp_ctx* ctx, int B) {
  const mtp_config& c = ctx->cfg;
  return ctx->tc_ws != nullptr && c.dtype == MTP_DTYPE_BF16 && c.head_dim == 128 && B >= ctx->tc_min_batch &&
         B <= 256 && c.hidden % 128 == 0 && c.hidden <= 16384 && c.ffn % 64 == 0 && ctx->q_dim % 64 == 0;
}

// Launch plan of one GEMM kind at one padded batch width NT: tensor maps,
// ring depth, cluster size, grid.  Computed once per context and cached (the
// maps depend only on the weights and the context's activation buffers).
struct TcPlan {
  TcMaps maps;
  int valid, stages, S, grid, n_tiles, C;
  size_t smem;
};
constexpr int kTcPlanSlots = 17;  // NT / 16 for NT <= 256

static TcPlan* tc_plan(mtp_ctx* ctx, cudaStream_t s, int kind, int NT) {
  if (!ctx->tc_plan_cache) {
    const size_t bytes = sizeof(TcPlan) * 6 * kTcPlanSlots;
    ctx->tc_plan_cache = aligned_alloc(64, (bytes + 63) / 64 * 64);
    if (!ctx->tc_plan_cache) return nullptr;
    memset(ctx->tc_plan_cache, 0, bytes);
  }
  TcPlan* p = &((TcPlan*)ctx->tc_plan_cache)[kind * kTcPlanSlots + NT / 16];
  if (p->valid) return p;
  const mtp_config& c = ctx->cfg;
  const mtp_weights& w = ctx->w;
  TcMaps& maps = p->maps;
  int C = 0, n_tiles = 0;
  bool ok = true;
  switch (kind) {
    case TC_EH:
      C = 2 * c.hidden; n_tiles = c.hidden / 128;
      ok = make_map(&maps.a0, w.w_eh, c.hidden, C, 128) && make_map(&maps.b, ctx->tc_xin_eh, c.max_batch, C, NT);
      break;
    case TC_QKV:
      C = c.hidden; n_tiles = c.n_q_heads + 2 * c.n_kv_heads;
      ok = make_map(&maps.a0, w.w_q, ctx->q_dim, C, 128) && make_map(&maps.a1, w.w_k, ctx->kv_dim, C, 128) &&
           make_map(&maps.a2, w.w_v, ctx->kv_dim, C, 128) && make_map(&maps.b, ctx->tc_xn, c.max_batch, C, NT);
      break;
    case TC_O:
      C = ctx->q_dim; n_tiles = c.hidden / 128;
      ok = make_map(&maps.a0, w.w_o, c.hidden, C, 128) && make_map(&maps.b, ctx->tc_attn, c.max_batch, C, NT);
      break;
    case TC_GU:
      C = c.hidden; n_tiles = c.ffn / 64;
      ok = make_map(&maps.a0, w.w_gate, c.ffn, C, 64) && make_map(&maps.a1, w.w_up, c.ffn, C, 64) &&
           make_map(&maps.b, ctx->tc_xn, c.max_batch, C, NT);
      break;
    case TC_DOWN:
      C = c.ffn; n_tiles = c.hidden / 128;
      ok = make_map(&maps.a0, w.w_down, c.hidden, C, 128) && make_map(&maps.b, ctx->tc_act, c.max_batch, C, NT);
      break;
    default:
      C = c.hidden; n_tiles = (c.vocab + 127) / 128;
      ok = make_map(&maps.a0, w.lm_head, c.vocab, C, 128) && make_map(&maps.a1, w.lm_head, c.vocab, C, 16) &&
           make_map(&maps.b, ctx->tc_xn, c.max_batch, C, NT);
      break;
  }
  if (!ok) return nullptr;
  const int nkb = C / 64;
  const int stage_bytes = kTcTileBytesA + NT * 128;
  // two CTAs per SM when a ring of >= 3 stages fits in ~100 KB and both CTAs'
  // accumulators fit in TMEM (512 columns)
  const bool two_per_sm = 3 * stage_bytes <= 100 * 1024 && 2 * (2 * NT) <= 512;
  const int budget = two_per_sm ? 100 * 1024 : 200 * 1024;
  int stages = budget / stage_bytes;
  if (stages > 8) stages = 8;
  if (stages < 2) stages = 2;
  const int slots = (two_per_sm ? 2 : 1) * ctx->num_sms;
  // Clusters are placed one CTA per SM, so a split-K launch gets the whole
  // SM's shared memory for its ring.
  int cl_stages = (200 * 1024) / stage_bytes;
  if (cl_stages > 8) cl_stages = 8;
  const size_t cl_smem = 1024 + (size_t)cl_stages * stage_bytes;
  size_t smem = 1024 + (size_t)stages * stage_bytes;
  if (ensure_smem((const void*)mtp_tc_proj_kernel, cl_smem > smem ? cl_smem : smem) != cudaSuccess) return nullptr;
  int S = 1;
  if (kind != TC_LM && n_tiles < slots && (size_t)cl_stages * stage_bytes >= (size_t)NT * 128 * 4) {
    // the LM head keeps whole tiles (argmax epilogue).  Largest cluster size
    // S <= 8 whose clusters all fit on the GPU at once (one wave).
    int s_max = ctx->num_sms / n_tiles;
    if (s_max > 8) s_max = 8;
    if (s_max > nkb / 2) s_max = nkb / 2;
    for (int cand = s_max; cand >= 2; --cand) {
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(n_tiles * cand);
      q.blockDim = dim3(kTcThreads);
      q.dynamicSmemBytes = cl_smem;
      q.stream = s;
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = (unsigned)cand;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      q.attrs = qa;
      q.numAttrs = 1;
      int clusters = 0;
      if (cudaOccupancyMaxActiveClusters(&clusters, (const void*)mtp_tc_proj_kernel, &q) != cudaSuccess) {
        cudaGetLastError();
        continue;
      }
      if (clusters >= n_tiles) {
        S = cand;
        break;
      }
    }
  }
  // split-K clusters, and whole-tile launches with at most one CTA per SM,
  // get the whole SM's shared memory for a deeper ring
  if (S > 1 || n_tiles <= ctx->num_sms) {
    stages = cl_stages;
    smem = cl_smem;
  }
  p->stages = stages;
  p->S = S;
  p->grid = (S > 1) ? n_tiles * S : (n_tiles < slots ? n_tiles : slots);
  p->n_tiles = n_tiles;
  p->C = C;
  p->smem = smem;
  p->valid = 1;
  if (getenv("MTP_TC_TRACE"))
    fprintf(stderr, "tc kind %d: NT %d tiles %d nkb %d stages %d two_per_sm %d cluster %d grid %d\n", kind, NT,
            n_tiles, nkb, stages, (int)two_per_sm, S, p->grid);
  return p;
}

static cudaError_t tc_launch(mtp_ctx* ctx, cudaStream_t s, int kind, int B, int k, int K, const int32_t* positions,
                             const mtp_kv* kv, int32_t* draft_ids, float* logits, float* hidden_out) {
  const mtp_config& c = ctx->cfg;
  const int NT = ((B + 15) / 16) * 16;
  const TcPlan* pl = tc_plan(ctx, s, kind, NT);
  if (!pl) return cudaErrorInvalidValue;
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.kind = kind; a.B = B; a.NT = NT; a.H = c.hidden; a.q_dim = ctx->q_dim; a.kv_dim = ctx->kv_dim; a.F = c.ffn;
  a.V = c.vocab; a.n_q = c.n_q_heads; a.n_kv = c.n_kv_heads; a.bs = c.block_size; a.k = k; a.K = K;
  a.C = pl->C; a.nkb = pl->C / 64; a.n_tiles = pl->n_tiles; a.max_pos = c.max_pos;
  a.num_blocks = kv->num_blocks; a.max_blocks = kv->max_blocks;
  a.positions = positions; a.draft_ids = draft_ids; a.logits = logits; a.hidden_out = hidden_out;
  a.k_pool = (uint16_t*)kv->k_pool; a.v_pool = (uint16_t*)kv->v_pool; a.block_table = kv->block_table;
  a.seq_len = kv->seq_len; a.pending = kv->pending;
  a.hid = ctx->hid; a.x = ctx->x; a.q = ctx->q; a.h1 = ctx->h1; a.act_bf16 = ctx->tc_act;
  a.lm_keys = ctx->lm_keys; a.lm_cnt = ctx->lm_cnt;
  a.err = ctx->err; a.rope = ctx->rope; a.req_bad = ctx->req_bad;
  a.stages = pl->stages;
  a.ksplit = pl->S;
  a.eps = c.eps;
  a.ssq = ctx->tc_ssq;
  a.xn_out = ctx->tc_xn;
  a.scale_in = (kind == TC_QKV || kind == TC_GU || kind == TC_LM) ? 1 : 0;
  a.w_next = (const uint16_t*)(kind == TC_EH ? ctx->w.w_norm_in : kind == TC_O ? ctx->w.w_norm_post
                               : kind == TC_DOWN ? ctx->w.w_norm_f : nullptr);
  const int kid = (kind == TC_EH) ? MTP_KERNEL_EH_PROJ : (kind == TC_QKV) ? MTP_KERNEL_QKV_ROPE
                  : (kind == TC_O) ? MTP_KERNEL_O_PROJ : (kind == TC_GU) ? MTP_KERNEL_GATE_UP
                  : (kind == TC_DOWN) ? MTP_KERNEL_DOWN : MTP_KERNEL_LM_HEAD;
  prof_before(ctx, kid, s);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(pl->grid);
  lc.blockDim = dim3(kTcThreads);
  lc.dynamicSmemBytes = pl->smem;
  lc.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)pl->S;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = (pl->S > 1) ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&lc, mtp_tc_proj_kernel, pl->maps, a);
  prof_after(ctx, kid, s);
  ctx->launches++;
  return e;
}

cudaError_t launch_draft_step_tc(mtp_ctx* ctx, cudaStream_t s, int B, int k, int K, const void* hidden,
                                 const void* embeds, const int32_t* positions, const mtp_kv* kv,
                                 const int32_t* chain_ids, int32_t* draft_ids, float* logits, float* hidden_out) {
  const mtp_config& c = ctx->cfg;
  cudaError_t e;
  PrepEhArgs pa;
  pa.B = B; pa.H = c.hidden; pa.V = c.vocab; pa.k = k; pa.K = K;
  pa.hidden_in = (const uint16_t*)hidden; pa.embeds_in = (const uint16_t*)embeds; pa.hid = ctx->hid;
  pa.chain_ids = chain_ids; pa.draft_ids = draft_ids; pa.embed = (const uint16_t*)ctx->w.embed;
  pa.w_h = (const uint16_t*)ctx->w.w_norm_h; pa.w_e = (const uint16_t*)ctx->w.w_norm_e; pa.eps = c.eps;
  pa.out = ctx->tc_xin_eh; pa.err = ctx->err; pa.pending = kv->pending; pa.req_bad = ctx->req_bad;
  ctx->launches++;
  if ((e = launch_pdl(prep_eh_kernel, dim3(B), dim3(kPrepThreads), 0, s, pa)) != cudaSuccess) return e;
  // EH, O and DOWN also write the next projection's bf16 input and its
  // per-tile sums of squares (RMSNorm folded into the GEMMs)
  if ((e = tc_launch(ctx, s, TC_EH, B, k, K, positions, kv, draft_ids, logits, hidden_out)) != cudaSuccess) return e;
  if ((e = tc_launch(ctx, s, TC_QKV, B, k, K, positions, kv, draft_ids, logits, hidden_out)) != cudaSuccess) return e;
  if ((e = launch_attention(ctx, s, B, k, kv)) != cudaSuccess) return e;
  if ((e = tc_launch(ctx, s, TC_O, B, k, K, positions, kv, draft_ids, logits, hidden_out)) != cudaSuccess) return e;
  if ((e = tc_launch(ctx, s, TC_GU, B, k, K, positions, kv, draft_ids, logits, hidden_out)) != cudaSuccess) return e;
  if ((e = tc_launch(ctx, s, TC_DOWN, B, k, K, positions, kv, draft_ids, logits, hidden_out)) != cudaSuccess) return e;
  return tc_launch(ctx, s, TC_LM, B, k, K, positions, kv, draft_ids, logits, hidden_out);
}

}  // namespace mtp
