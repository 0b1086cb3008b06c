// Persistent draft kernel for small batches: all K recursive draft steps of
// one mtp_draft call in a single cooperative launch with one CTA per SM.
//
// Draft step k runs seven phases, each closed by a grid-wide barrier
// ("MTP (Multi-Token Prediction)", "Architecture": dual norm, concat,
// projection, one standard decoder layer, shared LM head, recursion):
//   EH    x  = W_eh [RMSNorm(h) w_h ; RMSNorm(e) w_e]
//   QKV   q, k, v = W_{q,k,v} RMSNorm(x) w_in, rotary on q and k, k/v
//         rounded to bf16 and appended to the paged cache at slot seq_len+k-1
//   ATTN  o = softmax(q K^T / sqrt(d)) V over the seq_len + k cached entries
//   O     h1 = x + W_o o
//   GU    a  = silu(W_g n2) * (W_u n2),  n2 = RMSNorm(h1) w_post
//   DOWN  h2 = h1 + W_d a
//   LM    z  = W_lm RMSNorm(h2) w_f,  d_k = argmax z (lowest id on ties)
// and step k+1 embeds d_k (or the teacher-forced chain id) and continues from
// h2, the decoder output before the final norm.
//
// Warp 0 of every CTA is the producer: one thread walks the CTA's share of
// every phase of every step in order and streams it into a ring of 16 KB
// shared-memory slots with bulk (TMA) copies -- weight row pairs for the
// projections, swizzled K/V tiles for attention.  Weights do not depend on
// the activations, so the ring keeps filling across phase barriers and the
// HBM stream does not drain at phase boundaries.  The one producer-side
// dependency is a cache block holding entries appended during this call: it
// is loaded only after the QKV barrier of its step.
//
// Warps 1..8 consume, every warp waiting on every slot in order:
//  * projections: a unit is one row pair times one column chunk (at most
//    4096 columns, so a unit is at most 16 KB).  Each consumer warp owns a
//    fixed slice of the chunk's columns and keeps the matching slice of the
//    normalised input in registers; per-warp partial dot products go through
//    a small shared buffer and are summed in warp order, chunk after chunk,
//    so the results do not depend on timing.
//  * attention: a unit is one 16-token block of one kv head.  The CTA owns a
//    contiguous range of the flattened (request, kv head, block) list; warps
//    take its blocks round-robin (attn_tile_mma), merge per kv head in shared
//    memory, and write one (max, sum, output) record per kv head; the last
//    CTA to finish a kv head combines its records.
//
// Every wait (slot, grid barrier, copies in flight) gives up after 2 s; a CTA
// that gives up sets MTP_ERR_TIMEOUT and a sticky abort word that makes the
// other CTAs, and later calls until the error is read, stop early.
#include <stdlib.h>
#include <string.h>

#include "mtp_common.cuh"
#include "mtp_attn_mma.cuh"

namespace mtp {

constexpr int kPW = 8;                  // consumer warps
constexpr int kPCT = kPW * 32;          // consumer threads
constexpr int kPThreads = kPCT + 32;    // + the producer warp
constexpr int kPMaxSlots = 16;
constexpr uint32_t kPSlot = 16384;      // bytes per ring slot
constexpr int kPMaxCW = 4096;           // columns per chunk
constexpr int kPMaxG = 8;               // query heads per kv head
constexpr unsigned long long kPSpinNs = 2000000000ull;  // any single wait gives up after 2 s

enum PPhase { P_EH = 0, P_QKV = 1, P_ATTN = 2, P_O = 3, P_GU = 4, P_DOWN = 5, P_LM = 6, P_NUM = 7 };

struct PArgs {
  int B, H, q_dim, kv_dim, F, V, n_q, n_kv, G, K, max_pos, num_blocks, max_blocks;
  int cw_h, cw_q, cw_f;  // column chunk widths of H-, q_dim- and F-wide rows
  int nslots;            // ring slots
  int max_recs;          // attention records per kv head (= grid size)
  float eps, qscale;
  const uint16_t *w_norm_h, *w_norm_e, *w_eh, *w_norm_in, *w_q, *w_k, *w_v, *w_o;
  const uint16_t *w_norm_post, *w_gate, *w_up, *w_down, *w_norm_f, *embed, *lm_head;
  const uint16_t* hidden_in;
  const uint16_t* embeds_in;
  const int32_t* positions;
  const int32_t* chain_ids;
  int32_t* draft_ids;
  float* logits;
  float* hidden_out;
  uint16_t* k_pool;
  uint16_t* v_pool;
  const int32_t* block_table;
  const int32_t* seq_len;
  int32_t* pending;
  float *hid, *x, *q, *attn, *h1, *act;
  float* rec;                 // [B * n_kv][max_recs][G][132] attention records: max, sum, -, -, o[128]
  int* seg_cnt;               // [B * n_kv] tiles merged so far
  unsigned long long* keys;   // [K][B] argmax keys
  unsigned long long* gbar;   // [0] barrier arrivals (only grows), [32] sticky abort flag (another line)
  int* err;
  const float2* rope;
};

// ------------------------------------------------------------ primitives

__device__ __forceinline__ unsigned long long p_clock_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned long long p_ld_acquire(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long p_ld_volatile(const unsigned long long* p) {
  return *(const volatile unsigned long long*)p;
}
__device__ __forceinline__ void p_fence_proxy_async() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void p_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Record that this CTA gives up: device error, CTA flag, grid-wide flag.
__device__ __forceinline__ void p_give_up(const PArgs& a, volatile int* s_abort) {
  set_error(a.err, MTP_ERR_TIMEOUT);
  *s_abort = 1;
  atomicExch(&a.gbar[32], 1ull);
}

// mbarrier phase wait; false after kPSpinNs (sets the abort state) or as soon
// as the CTA is aborting.
__device__ __forceinline__ bool p_wait(const PArgs& a, uint64_t* bar, uint32_t parity, volatile int* s_abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = p_clock_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255) == 0) {
      if (*s_abort) return false;
      if (p_clock_ns() - t0 > kPSpinNs) {
        p_give_up(a, s_abort);
        return false;
      }
    }
  }
}

// Bounded wait with no abort state, for draining copies in flight.
__device__ __forceinline__ void p_wait_landed(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = p_clock_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return;
    if ((i & 255) == 255 && p_clock_ns() - t0 > kPSpinNs) return;
  }
}

// Grid barrier: every CTA adds one to a 64-bit arrival counter that only
// grows (a launch adds a whole number of grid sizes); barrier j of a launch
// whose counter started at `base` is passed once the counter reaches
// base + (j + 1) * grid.  The arrival is a fire-and-forget release reduction,
// so a barrier costs about two L2 round trips (the arrival landing, the poll
// that sees the last one).  Wait until the counter reaches `target`.
__device__ bool p_wait_count(const PArgs& a, unsigned long long target, volatile int* s_abort) {
  const unsigned long long t0 = p_clock_ns();
  for (uint32_t n = 0;; ++n) {
    if (p_ld_acquire(&a.gbar[0]) >= target) return true;
    if ((n & 63) == 63) {
      if (*s_abort || p_ld_volatile(&a.gbar[32])) {
        *s_abort = 1;
        return false;
      }
      if (p_clock_ns() - t0 > kPSpinNs) {
        p_give_up(a, s_abort);
        return false;
      }
    }
  }
}

__device__ __forceinline__ int p_atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void p_arrive_grid(unsigned long long* counter) {
  asm volatile("fence.acq_rel.gpu;\n\tred.release.gpu.global.add.u64 [%0], 1;" ::"l"(counter) : "memory");
}

// Reduce N (a power of two <= 32) per-lane values over the warp: lane l ends
// with the total of value l >> (5 - log2 N).
template <int N>
__device__ __forceinline__ float p_reduce_scatter(float (&v)[N], int lane) {
#pragma unroll
  for (int h = N / 2, o = 16; h >= 1; h >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? v[i] : v[i + h];
      const float keep = up ? v[i + h] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float r = v[0];
#pragma unroll
  for (int o = 16 / N; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}

__device__ __forceinline__ float p_silu(float g) { return g / (1.0f + __expf(-g)); }

// ------------------------------------------------------ phase geometry

__device__ __forceinline__ int p_cols(const PArgs& a, int ph) {
  return ph == P_EH ? 2 * a.H : ph == P_O ? a.q_dim : ph == P_DOWN ? a.F : a.H;
}
__device__ __forceinline__ int p_cw(const PArgs& a, int ph) {
  return ph == P_O ? a.cw_q : ph == P_DOWN ? a.cw_f : a.cw_h;
}
__device__ __forceinline__ int p_pairs(const PArgs& a, int ph) {
  switch (ph) {
    case P_EH: case P_O: case P_DOWN: return a.H / 2;
    case P_QKV: return (a.q_dim + 2 * a.kv_dim) / 2;
    case P_GU: return a.F;
    default: return (a.V + 1) / 2;
  }
}
__device__ __forceinline__ void p_split(int n, int i, int G, int& beg, int& end) {
  beg = (int)(((long long)i * n) / G);
  end = (int)(((long long)(i + 1) * n) / G);
}

// Rows (r0, r1) of pair p and their weight rows (w1 null: no second row).
// QKV pairs are the rotary pairs (i, i + 64) of one head; GU pairs are the
// gate and up rows of one inner unit; the rest are rows 2p, 2p + 1.
__device__ __forceinline__ void p_pair(const PArgs& a, int ph, int p, int C, int& r0, int& r1, const uint16_t*& w0,
                                       const uint16_t*& w1) {
  if (ph == P_QKV) {
    const int grp = p >> 6, i = p & 63;
    r0 = grp * 128 + i;
    r1 = r0 + 64;
    const uint16_t* base;
    int rr;
    if (r0 < a.q_dim) { base = a.w_q; rr = r0; }
    else if (r0 < a.q_dim + a.kv_dim) { base = a.w_k; rr = r0 - a.q_dim; }
    else { base = a.w_v; rr = r0 - a.q_dim - a.kv_dim; }
    w0 = base + (size_t)rr * C;
    w1 = w0 + (size_t)64 * C;
  } else if (ph == P_GU) {
    r0 = r1 = p;
    w0 = a.w_gate + (size_t)p * C;
    w1 = a.w_up + (size_t)p * C;
  } else {
    const uint16_t* W = ph == P_EH ? a.w_eh : ph == P_O ? a.w_o : ph == P_DOWN ? a.w_down : a.lm_head;
    const int R = ph == P_LM ? a.V : a.H;
    r0 = 2 * p;
    r1 = (2 * p + 1 < R) ? 2 * p + 1 : -1;
    w0 = W + (size_t)r0 * C;
    w1 = r1 >= 0 ? w0 + C : nullptr;
  }
}

// Flattened attention tiles of step k: request b owns n_kv * nblk[b] tiles
// starting at base[b] (kv head major, then block).
struct PAttnGeo {
  int nblk[4];
  long long base[5];
};
__device__ __forceinline__ void p_attn_geo(const PArgs& a, const int* s_seq, int k, PAttnGeo& g) {
  long long t = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    const int T = b < a.B ? s_seq[b] + k : 0;
    g.nblk[b] = T > 0 ? (T + 15) >> 4 : 0;
    g.base[b] = t;
    t += (long long)a.n_kv * g.nblk[b];
  }
  g.base[4] = t;
}

// The one input vector of a projection phase (two for EH), for request b.
struct PVec {
  const float* f;     // fp32 source, or
  const uint16_t* h;  // bf16 source
  const uint16_t* w;  // RMSNorm weight, null: no norm
};
__device__ __forceinline__ PVec p_vec(const PArgs& a, int ph, int vec, int k, int b, int id) {
  PVec v = {nullptr, nullptr, nullptr};
  switch (ph) {
    case P_EH:
      if (vec == 0) {
        if (k == 1) v.h = a.hidden_in + (size_t)b * a.H;
        else v.f = a.hid + (size_t)b * a.H;
        v.w = a.w_norm_h;
      } else {
        v.h = (k == 1) ? a.embeds_in + (size_t)b * a.H : a.embed + (size_t)id * a.H;
        v.w = a.w_norm_e;
      }
      break;
    case P_QKV: v.f = a.x + (size_t)b * a.H; v.w = a.w_norm_in; break;
    case P_O: v.f = a.attn + (size_t)b * a.q_dim; break;
    case P_GU: v.f = a.h1 + (size_t)b * a.H; v.w = a.w_norm_post; break;
    case P_DOWN: v.f = a.act + (size_t)b * a.F; break;
    default: v.f = a.hid + (size_t)b * a.H; v.w = a.w_norm_f; break;
  }
  return v;
}

// Epilogue of pair p of request b with the full dot products (v0, v1).
// Returns the LM argmax key (0 for other phases).
// bad_mask bit b: request b had pending != 0 when the call began (no KV
// writes for it at any step).
__device__ __forceinline__ unsigned long long p_epilogue(const PArgs& a, int ph, int k, int b, int p, float v0,
                                                         float v1, unsigned bad_mask) {
  const size_t bh = (size_t)b * a.H;
  const long long nBH = (long long)a.B * a.H;
  switch (ph) {
    case P_EH:
      MTP_STORE(a.err, a.x, bh + 2 * p, nBH, v0);
      MTP_STORE(a.err, a.x, bh + 2 * p + 1, nBH, v1);
      return 0ull;
    case P_O:
      MTP_STORE(a.err, a.h1, bh + 2 * p, nBH, __ldcg(a.x + bh + 2 * p) + v0);
      MTP_STORE(a.err, a.h1, bh + 2 * p + 1, nBH, __ldcg(a.x + bh + 2 * p + 1) + v1);
      return 0ull;
    case P_GU:
      MTP_STORE(a.err, a.act, (size_t)b * a.F + p, (long long)a.B * a.F, p_silu(v0) * v1);
      return 0ull;
    case P_DOWN: {
      const float o0 = __ldcg(a.h1 + bh + 2 * p) + v0, o1 = __ldcg(a.h1 + bh + 2 * p + 1) + v1;
      MTP_STORE(a.err, a.hid, bh + 2 * p, nBH, o0);
      MTP_STORE(a.err, a.hid, bh + 2 * p + 1, nBH, o1);
      if (a.hidden_out && k == a.K) {
        MTP_STORE(a.err, a.hidden_out, bh + 2 * p, nBH, o0);
        MTP_STORE(a.err, a.hidden_out, bh + 2 * p + 1, nBH, o1);
      }
      return 0ull;
    }
    case P_LM: {
      const int r0 = 2 * p, r1 = 2 * p + 1;
      const long long row = ((long long)b * a.K + (k - 1)) * a.V, nL = (long long)a.B * a.K * a.V;
      if (a.logits) MTP_STORE(a.err, a.logits, row + r0, nL, v0);
      unsigned long long key = argmax_key(v0, (uint32_t)r0);
      if (r1 < a.V) {
        if (a.logits) MTP_STORE(a.err, a.logits, row + r1, nL, v1);
        key = umax64(key, argmax_key(v1, (uint32_t)r1));
      }
      return key;
    }
    default: {  // P_QKV: rotary pair (i, i + 64) of head grp
      const int grp = p >> 6, i = p & 63;
      const int r0 = grp * 128 + i;
      const int pos = a.positions[b] + k - 1;
      if (pos < 0 || pos >= a.max_pos) {
        set_error(a.err, MTP_ERR_CAPACITY);
        return 0ull;
      }
      const float2 cs = a.rope[(size_t)pos * 64 + i];
      if (grp < a.n_q) {
        const long long nQ = (long long)a.B * a.q_dim;
        MTP_STORE(a.err, a.q, (size_t)b * a.q_dim + r0, nQ, v0 * cs.x - v1 * cs.y);
        MTP_STORE(a.err, a.q, (size_t)b * a.q_dim + r0 + 64, nQ, v1 * cs.x + v0 * cs.y);
        return 0ull;
      }
      if ((bad_mask >> b) & 1u) {
        set_error(a.err, MTP_ERR_DEVICE_ARGS);
        return 0ull;
      }
      const int slot = a.seq_len[b] + k - 1;
      const int bi = slot >> 4, off = slot & 15;
      const int blk = (bi < a.max_blocks && slot >= 0) ? a.block_table[(size_t)b * a.max_blocks + bi] : -1;
      if (blk < 0 || blk >= a.num_blocks) {
        set_error(a.err, MTP_ERR_CAPACITY);
        return 0ull;
      }
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
      const long long e = (((long long)blk * a.n_kv + g) * 16 + off) * 128 + i;
      const long long nP = (long long)a.num_blocks * a.n_kv * 16 * 128;
      MTP_STORE(a.err, pool, e, nP, f32_to_bf16_rne(o0));
      MTP_STORE(a.err, pool, e + 64, nP, f32_to_bf16_rne(o1));
      return 0ull;
    }
  }
}

// ------------------------------------------------------------ producer

// Run by the whole producer warp: every lane walks the same unit sequence,
// lane 0 waits for slots and issues the copies, and in attention phases the
// 32 lanes look up the cache blocks of 32 tiles at once (block-table reads
// would otherwise serialise one L2 round trip per tile).
__device__ void p_produce(const PArgs& a, const CUtensorMap* kmap, const CUtensorMap* vmap, unsigned char* ring,
                          uint64_t* full, uint64_t* empty, const int* s_seq, unsigned long long base,
                          volatile int* s_abort) {
  const int lane = threadIdx.x & 31;
  const int Gd = gridDim.x, cta = blockIdx.x;
  const uint32_t NS = (uint32_t)a.nslots;
  uint32_t u = 0;
  bool ok = true;  // uniform across the warp
  // slot of unit uu is free once its consumer released the previous use
  auto acquire = [&](uint32_t uu) -> bool {
    int r = 1;
    if (lane == 0) r = p_wait(a, &empty[uu % NS], ((uu / NS) & 1u) ^ 1u, s_abort) ? 1 : 0;
    return __shfl_sync(0xffffffffu, r, 0) != 0;
  };
  for (int k = 1; k <= a.K && ok; ++k) {
    for (int ph = 0; ph < P_NUM && ok; ++ph) {
      if (ph == P_ATTN) {
        PAttnGeo geo;
        p_attn_geo(a, s_seq, k, geo);
        const long long T = geo.base[4];
        const long long tb = (long long)cta * T / Gd, te = (long long)(cta + 1) * T / Gd;
        bool released = false;
        for (long long t0 = tb; t0 < te && ok; t0 += 32) {
          const long long t = t0 + lane;
          int b = 0, g = 0, bi = 0, blk = 0;
          if (t < te) {
            while (t >= geo.base[b + 1]) ++b;
            const int rel = (int)(t - geo.base[b]);
            g = rel / geo.nblk[b];
            bi = rel - g * geo.nblk[b];
            blk = (bi < a.max_blocks) ? a.block_table[(size_t)b * a.max_blocks + bi] : -1;
            if (blk < 0 || blk >= a.num_blocks) {
              set_error(a.err, MTP_ERR_CAPACITY);
              blk = 0;
            }
          }
          const int n = (int)((te - t0) < 32 ? (te - t0) : 32);
          for (int j = 0; j < n && ok; ++j) {
            const int bj = __shfl_sync(0xffffffffu, b, j), gj = __shfl_sync(0xffffffffu, g, j);
            const int bij = __shfl_sync(0xffffffffu, bi, j), blkj = __shfl_sync(0xffffffffu, blk, j);
            if (!released && (bij + 1) * 16 > s_seq[bj]) {
              // block holds entries appended during this call: after the QKV barrier of step k
              int r = 1;
              if (lane == 0) {
                r = p_wait_count(a, base + (unsigned long long)(P_NUM * (k - 1) + 2) * Gd, s_abort) ? 1 : 0;
                p_fence_proxy_async();
              }
              ok = __shfl_sync(0xffffffffu, r, 0) != 0;
              released = true;
              if (!ok) break;
            }
            if (!(ok = acquire(u))) break;
            if (lane == 0) {
              const uint32_t s = u % NS;
              tma_kv_tile(ring + (size_t)s * kPSlot, kmap, vmap, (blkj * a.n_kv + gj) * 16, &full[s]);
            }
            ++u;
          }
        }
      } else {
        const int C = p_cols(a, ph), CW = p_cw(a, ph), nch = C / CW, P = p_pairs(a, ph);
        int pb, pe;
        p_split(P, cta, Gd, pb, pe);
        const uint32_t rb = (uint32_t)CW * 2u;
        // lane 0 alone; the other lanes wait at the broadcast of its status
        if (lane == 0) {
          const uint64_t pol = l2_evict_first_policy();  // weights are read once per step
          for (int c = 0; c < nch && ok; ++c)
            for (int p = pb; p < pe && ok; ++p) {
              if (!(ok = p_wait(a, &empty[u % NS], ((u / NS) & 1u) ^ 1u, s_abort))) break;
              int r0, r1;
              const uint16_t *w0, *w1;
              p_pair(a, ph, p, C, r0, r1, w0, w1);
              const uint32_t s = u % NS;
              unsigned char* dst = ring + (size_t)s * kPSlot;
              if (nch == 1 && w1 == w0 + C) {
                mbar_expect_tx(&full[s], 2u * rb);
                bulk_g2s_hint(dst, w0, 2u * rb, &full[s], pol);
              } else {
                mbar_expect_tx(&full[s], w1 ? 2u * rb : rb);
                bulk_g2s_hint(dst, w0 + (size_t)c * CW, rb, &full[s], pol);
                if (w1) bulk_g2s_hint(dst + rb, w1 + (size_t)c * CW, rb, &full[s], pol);
              }
              ++u;
            }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        u = __shfl_sync(0xffffffffu, u, 0);
      }
    }
  }
  // the copies still in flight land before the CTA may exit
  if (lane == 0)
    for (uint32_t v = (u > NS ? u - NS : 0u); v < u; ++v) p_wait_landed(&full[v % NS], (v / NS) & 1u);
}

// ------------------------------------------------------------- the kernel
//
// Block: warp 0 = producer, warps 1..A = consumers (A = blockDim / 32 - 1,
// at most kPW).  Unit u of the CTA's sequence sits in slot u % S and is
// consumed by warp u % A alone; S is a multiple of A, so consecutive uses of
// a slot belong to the same warp, which saw the previous fill land before it
// waits on the slot's next phase (the parity wait cannot match a stale
// phase).

template <int NB>
__global__ void __launch_bounds__(kPThreads, 1)
    p_draft_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const PArgs a) {
  extern __shared__ __align__(1024) unsigned char p_smem_in[];
  unsigned char* ring = (unsigned char*)(((uintptr_t)p_smem_in + 1023) & ~(uintptr_t)1023);
  float* uni = reinterpret_cast<float*>(ring + (size_t)a.nslots * kPSlot);
  __shared__ __align__(8) uint64_t full[kPMaxSlots], empty[kPMaxSlots];
  __shared__ float red[kPW][2 * NB];
  __shared__ float s_scale[2][4];
  __shared__ float wm[kPW][kPMaxG], wl[kPW][kPMaxG];
  __shared__ unsigned long long sbest[kPW][NB];
  __shared__ int s_seq[4];
  __shared__ unsigned s_bad;  // bit b: pending[b] != 0 on entry
  __shared__ unsigned long long s_base;
  __shared__ volatile int s_abort;
  __shared__ int s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int A = (int)(blockDim.x >> 5) - 1;  // consumer warps
  const int nct = 32 * A;                    // consumer threads
  if (threadIdx.x == 0) {
    for (int s = 0; s < a.nslots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
    // CTAs that already arrived at barrier 0 add less than one grid size
    const unsigned long long c0 = p_ld_acquire(&a.gbar[0]);
    s_base = c0 - c0 % gridDim.x;
    s_abort = p_ld_volatile(&a.gbar[32]) ? 1 : 0;
  }
  if (threadIdx.x < 4) s_seq[threadIdx.x] = (int)threadIdx.x < a.B ? a.seq_len[threadIdx.x] : 0;
  if (threadIdx.x == 32) {
    unsigned m = 0;
    for (int b = 0; b < a.B; ++b)
      if (a.pending[b] != 0) m |= 1u << b;
    s_bad = m;
  }
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < a.K * a.B; i += blockDim.x) a.keys[i] = 0ull;
  __syncthreads();
  if (s_abort) {
    if (threadIdx.x == 0) set_error(a.err, MTP_ERR_TIMEOUT);
    return;
  }

  if (warp == 0) {
    p_produce(a, &kmap, &vmap, ring, full, empty, s_seq, s_base, &s_abort);
    return;
  }

  // ----------------------------------------------------------- consumers
  const int wc = warp - 1, ct = threadIdx.x - 32;
  const int Gd = gridDim.x, cta = blockIdx.x;
  const uint32_t NS = (uint32_t)a.nslots;
  uint32_t u = 0;       // first unit of the current phase in the producer's sequence
  unsigned bar_j = 0;   // grid barriers passed
  auto cons_sync = [&]() { asm volatile("bar.sync 1, %0;" ::"r"(nct) : "memory"); };

  // proxy: the barrier after QKV also orders the cache rows written there
  // before the bulk copies that read them back
  auto grid_sync = [&](bool proxy) -> bool {
    cons_sync();
    if (ct == 0 && !s_abort) {
      if (proxy) p_fence_proxy_async();
      p_arrive_grid(&a.gbar[0]);
      p_wait_count(a, s_base + (unsigned long long)(bar_j + 1) * Gd, &s_abort);
    }
    ++bar_j;
    cons_sync();
    return !s_abort;
  };

  // projection phases: input chunk (fp32) at uni[0 .. NB*CW), then the
  // per-unit results of multi-chunk phases [nch][np][2][NB]
  float* xs = uni;

  auto weights_phase = [&](int ph, int k) {
    const int C = p_cols(a, ph), CW = p_cw(a, ph), nch = C / CW, P = p_pairs(a, ph);
    int pb, pe;
    p_split(P, cta, Gd, pb, pe);
    const int np = pe - pb, nv = CW >> 3;
    const int nvec = (ph == P_EH) ? 2 : 1;
    const int cpv = nch / nvec;  // chunks per input vector
    float* res = uni + (size_t)NB * CW;

    // Input normalisation.  When every input vector is a single chunk
    // (H <= 4096) the sum of squares is taken in the same pass that stages
    // the raw values times the norm weight, and the per-request RMS factor
    // multiplies the dot products in the epilogue: one L2 round trip and one
    // CTA sync before the first unit.  Wider vectors take a statistics pass
    // first and stage already-normalised values.
    const bool normed = (ph != P_O && ph != P_DOWN);
    const bool fused = normed && cpv == 1;
    // token ids of EH at k >= 2 (validated where used, so the loads stay in
    // flight while chunk 0 is staged and consumed)
    int ids[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      ids[b] = 0;
      if (ph == P_EH && k > 1 && b < a.B)
        ids[b] = a.chain_ids ? a.chain_ids[(size_t)b * (a.K - 1) + (k - 2)]
                             : (int)key_index(__ldcg(a.keys + (size_t)(k - 2) * a.B + b));
    }
    auto id_of = [&](int b) {
      int r = 0;
#pragma unroll
      for (int bb = 0; bb < NB; ++bb)
        if (bb == b) r = ids[bb];
      if (r < 0 || r >= a.V) {
        set_error(a.err, MTP_ERR_DEVICE_ARGS);
        r = 0;
      }
      return r;
    };
    float scale[2][NB];
#pragma unroll
    for (int v = 0; v < 2; ++v)
#pragma unroll
      for (int b = 0; b < NB; ++b) scale[v][b] = 1.0f;
    // RMS factors of input vector `vec` from per-thread sums of squares
    auto reduce_scale = [&](int vec, float (&ss)[NB]) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float t = warp_sum(ss[b]);
        if (lane == 0) red[wc][b] = t;
      }
      cons_sync();
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float t = 0.0f;
        for (int w = 0; w < A; ++w) t += red[w][b];
        const float r = rsqrtf(t / (float)a.H + a.eps);
        if (vec == 0) scale[0][b] = r;
        else scale[1][b] = r;
        if (ct == b) s_scale[vec][b] = r;
      }
    };
    auto load8 = [&](const PVec& src, int col, float (&x)[8]) {
      if (src.f) {
        const float4 t0 = __ldcg(reinterpret_cast<const float4*>(src.f + col));
        const float4 t1 = __ldcg(reinterpret_cast<const float4*>(src.f + col + 4));
        x[0] = t0.x; x[1] = t0.y; x[2] = t0.z; x[3] = t0.w;
        x[4] = t1.x; x[5] = t1.y; x[6] = t1.z; x[7] = t1.w;
      } else {
        const uint4 t = __ldg(reinterpret_cast<const uint4*>(src.h + col));
        x[0] = bf16_lo(t.x); x[1] = bf16_hi(t.x); x[2] = bf16_lo(t.y); x[3] = bf16_hi(t.y);
        x[4] = bf16_lo(t.z); x[5] = bf16_hi(t.z); x[6] = bf16_lo(t.w); x[7] = bf16_hi(t.w);
      }
    };

    if (normed && !fused) {
      for (int v = 0; v < nvec; ++v) {
        float ss[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          ss[b] = 0.0f;
          if (b < a.B) {
            const PVec src = p_vec(a, ph, v, k, b, id_of(b));
            for (int i8 = ct; i8 < (a.H >> 3); i8 += nct) {
              float x[8];
              load8(src, i8 * 8, x);
#pragma unroll
              for (int e = 0; e < 8; ++e) ss[b] = fmaf(x[e], x[e], ss[b]);
            }
          }
        }
        reduce_scale(v, ss);
        cons_sync();  // red is reused by the next vector
      }
    }

    unsigned long long best[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) best[b] = 0ull;

    for (int c = 0; c < nch; ++c) {
      // stage this chunk of the input once all warps are done with the
      // previous one
      if (c > 0) cons_sync();
      const int vec = c / cpv, col0 = (c - vec * cpv) * CW;
      const bool stats = fused;  // fused: each chunk is the whole of its vector
      float ss[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) ss[b] = 0.0f;
#pragma unroll 2
      for (int it = ct; it < a.B * nv; it += nct) {
        const int b = it / nv, vi = it - b * nv;
        const PVec src = p_vec(a, ph, vec, k, b, vec ? id_of(b) : 0);
        const int col = col0 + vi * 8;
        // every load of the iteration is in flight before any arithmetic
        float x[8];
        load8(src, col, x);
        uint4 wn = make_uint4(0u, 0u, 0u, 0u);
        if (src.w) wn = __ldg(reinterpret_cast<const uint4*>(src.w + col));
        if (stats) {
          float q = 0.0f;
#pragma unroll
          for (int e = 0; e < 8; ++e) q = fmaf(x[e], x[e], q);
#pragma unroll
          for (int bb = 0; bb < NB; ++bb)
            if (bb == b) ss[bb] += q;
        }
        if (src.w) {
          const float sc = fused ? 1.0f : s_scale[vec][b];
          x[0] *= sc * bf16_lo(wn.x); x[1] *= sc * bf16_hi(wn.x);
          x[2] *= sc * bf16_lo(wn.y); x[3] *= sc * bf16_hi(wn.y);
          x[4] *= sc * bf16_lo(wn.z); x[5] *= sc * bf16_hi(wn.z);
          x[6] *= sc * bf16_lo(wn.w); x[7] *= sc * bf16_hi(wn.w);
        }
        float4* d = reinterpret_cast<float4*>(xs + (size_t)b * CW + vi * 8);
        d[0] = make_float4(x[0], x[1], x[2], x[3]);
        d[1] = make_float4(x[4], x[5], x[6], x[7]);
      }
      if (stats) reduce_scale(vec, ss);  // includes the sync that publishes the chunk
      else cons_sync();

      // this warp's units of the chunk
      const uint32_t u0 = u + (uint32_t)(c * np);
      for (int i = (int)((uint32_t)(wc + A) - u0 % (uint32_t)A) % A; i < np; i += A) {
        const uint32_t uu = u0 + (uint32_t)i;
        const uint32_t s = uu % NS;
        const bool ok = p_wait(a, &full[s], (uu / NS) & 1u, &s_abort);
        const int p = pb + i;
        const bool two = !(ph == P_LM && 2 * p + 1 >= a.V);
        float v[2 * NB];
#pragma unroll
        for (int t = 0; t < 2 * NB; ++t) v[t] = 0.0f;
        if (ok) {
          const uint16_t* s0 = reinterpret_cast<const uint16_t*>(ring + (size_t)s * kPSlot);
          const uint16_t* s1 = s0 + CW;
#pragma unroll 4
          for (int vi = lane; vi < nv; vi += 32) {
            const uint4 w0 = *reinterpret_cast<const uint4*>(s0 + vi * 8);
            const uint4 w1 = two ? *reinterpret_cast<const uint4*>(s1 + vi * 8) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              if (b < a.B) {
                const float* xp = xs + (size_t)b * CW + vi * 8;
                v[b] += dot_vec<uint16_t>(w0, xp);
                v[NB + b] += dot_vec<uint16_t>(w1, xp);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) p_arrive(&empty[s]);
        // totals to lane 0: value t of the reduce-scatter sits in lane t << kShift
        const float r = p_reduce_scatter<2 * NB>(v, lane);
        constexpr int kShift = (2 * NB == 2) ? 4 : (2 * NB == 4) ? 3 : 2;
        float tot[2 * NB];
#pragma unroll
        for (int t = 0; t < 2 * NB; ++t) tot[t] = __shfl_sync(0xffffffffu, r, t << kShift);
        if (lane == 0 && ok) {
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            if (b < a.B) {
              if (nch == 1) {
                const float m = fused ? scale[0][b] : 1.0f;
                best[b] = umax64(best[b], p_epilogue(a, ph, k, b, p, tot[b] * m, tot[NB + b] * m, s_bad));
              } else {
                float* rr = res + ((size_t)c * np + i) * 2 * NB;
                rr[b] = tot[b];
                rr[NB + b] = tot[NB + b];
              }
            }
          }
        }
      }
    }
    u += (uint32_t)(nch * np);

    if (nch > 1) {
      // sum the chunks of every pair in chunk order, then the epilogue
      cons_sync();
      if (!s_abort)
        for (int it = ct; it < np * a.B; it += nct) {
          const int i = it / a.B, b = it - i * a.B;
          float s0 = 0.0f, s1 = 0.0f;
          for (int c = 0; c < nch; ++c) {
            const float* rr = res + ((size_t)c * np + i) * 2 * NB;
            const float m = fused ? s_scale[c / cpv][b] : 1.0f;
            s0 = fmaf(rr[b], m, s0);
            s1 = fmaf(rr[NB + b], m, s1);
          }
          const unsigned long long key = p_epilogue(a, ph, k, b, pb + i, s0, s1, s_bad);
#pragma unroll
          for (int bb = 0; bb < NB; ++bb)
            if (bb == b) best[bb] = umax64(best[bb], key);
        }
    }
    if (ph == P_QKV) p_fence_proxy_async();  // cache rows are read back by bulk copies

    if (ph == P_LM) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const unsigned long long m = warp_max_u64(best[b]);
        if (lane == 0) sbest[wc][b] = m;
      }
      cons_sync();
      if (ct < a.B && !s_abort) {
        unsigned long long m = 0ull;
        for (int w = 0; w < A; ++w)
#pragma unroll
          for (int b = 0; b < NB; ++b)
            if (b == ct) m = umax64(m, sbest[w][b]);
        if (m) atomicMax(a.keys + (size_t)(k - 1) * a.B + ct, m);
      }
    }
  };

  auto attn_phase = [&](int k) {
    PAttnGeo geo;
    p_attn_geo(a, s_seq, k, geo);
    const long long T = geo.base[4];
    const long long tb = (long long)cta * T / Gd, te = (long long)(cta + 1) * T / Gd;
    const int G = a.G;
    const int gi = lane >> 2, ti = lane & 3;
    long long t = tb;
    while (t < te) {
      int b = 0;
      while (t >= geo.base[b + 1]) ++b;
      const int nbk = geo.nblk[b];
      const int rel = (int)(t - geo.base[b]);
      const int g = rel / nbk, bi0 = rel - g * nbk;
      const long long S = geo.base[b] + (long long)g * nbk, E = S + nbk;
      const int n_local = (int)((te < E ? te : E) - t);
      const int T_len = s_seq[b] + k;

      float o[16][4];
#pragma unroll
      for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
      float m_run = -INFINITY, l_run = 0.0f;
      const int j0 = (int)((uint32_t)(wc + A) - u % (uint32_t)A) % A;  // this warp's first tile
      if (j0 < n_local) {
        uint32_t qa[8][4];
        load_q_frags(qa, a.q + (size_t)b * a.q_dim + (size_t)g * G * 128, a.qscale, lane, G);
        for (int j = j0; j < n_local; j += A) {
          const uint32_t uu = u + (uint32_t)j;
          const uint32_t s = uu % NS;
          const bool ok = p_wait(a, &full[s], (uu / NS) & 1u, &s_abort);
          if (ok) {
            const uint32_t kt = smem_addr(ring + (size_t)s * kPSlot);
            attn_tile_mma(kt, kt + 4096, qa, o, m_run, l_run, (bi0 + j) * 16, T_len, lane);
          }
          __syncwarp();
          if (lane == 0) p_arrive(&empty[s]);
        }
      }
      u += (uint32_t)n_local;

      // merge the warps of this CTA for kv head (b, g).  CTAs i0..i1 span the
      // kv head's tiles (records indexed by CTA - i0); when there are fewer
      // tiles than CTAs some of them own none and write no record.
      const int seg = b * a.n_kv + g;
      const int i0 = (int)(((S + 1) * Gd - 1) / T), i1 = (int)((E * Gd - 1) / T);
      const int nrec = i1 - i0 + 1, ridx = cta - i0;
      const bool whole = (n_local == nbk);  // this CTA holds every tile of the kv head
      float* wacc = uni;                    // [A][G][128]
      cons_sync();
      if (gi < G) {
        if (ti == 0) {
          wm[wc][gi] = m_run;
          wl[wc][gi] = l_run;
        }
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          wacc[((size_t)wc * G + gi) * 128 + 8 * n + 2 * ti] = o[n][0];
          wacc[((size_t)wc * G + gi) * 128 + 8 * n + 2 * ti + 1] = o[n][1];
        }
      }
      cons_sync();
      float* recs = a.rec + (size_t)seg * a.max_recs * G * 132;
      float* out = a.attn + (size_t)b * a.q_dim + (size_t)g * G * 128;
      if (!s_abort)
        for (int idx = ct; idx < G * 128; idx += nct) {
          const int h = idx >> 7, d = idx & 127;
          float M = -INFINITY;
          for (int w = 0; w < A; ++w) M = fmaxf(M, wm[w][h]);
          float L = 0.0f, O = 0.0f;
          for (int w = 0; w < A; ++w) {
            const float f = (wm[w][h] == -INFINITY) ? 0.0f : exp2f(wm[w][h] - M);
            L += wl[w][h] * f;
            O += wacc[((size_t)w * G + h) * 128 + d] * f;
          }
          if (whole) {
            out[(size_t)h * 128 + d] = O / L;
          } else {
            float* r = recs + ((size_t)ridx * G + h) * 132;
            if (d == 0) {
              r[0] = M;
              r[1] = L;
            }
            r[4 + d] = O;
          }
        }
      if (!whole) {
        // arrivals are counted in tiles: the CTA that completes the kv head's
        // tile count combines
        cons_sync();
        if (ct == 0) s_last = (p_atom_add_acq_rel(a.seg_cnt + seg, n_local) + n_local == nbk);
        cons_sync();
        if (s_last) {
          // thread (h, 4 dims) merges the records online, eight records' loads
          // in flight at a time; CTAs that hold no tile of this kv head wrote
          // no record
          for (int it = ct; it < G * 32; it += nct) {
            const int h = it >> 5, d4 = it & 31;
            float Mr = -INFINITY, Lr = 0.0f;
            float4 Or = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            for (int j0 = 0; j0 < nrec; j0 += 8) {
              float mj[8], lj[8];
              float4 oj[8];
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const int jr = j0 + q;
                const long long jb = (long long)(i0 + jr) * T / Gd, je = (long long)(i0 + jr + 1) * T / Gd;
                const bool valid = jr < nrec && (jb > S ? jb : S) < (je < E ? je : E);
                mj[q] = -INFINITY;
                lj[q] = 0.0f;
                oj[q] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (valid) {
                  const float* r = recs + ((size_t)jr * G + h) * 132;
                  mj[q] = __ldcg(r);
                  lj[q] = __ldcg(r + 1);
                  oj[q] = __ldcg(reinterpret_cast<const float4*>(r + 4) + d4);
                }
              }
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                if (mj[q] == -INFINITY) continue;
                const float Mn = fmaxf(Mr, mj[q]);
                const float co = (Mr == -INFINITY) ? 0.0f : exp2f(Mr - Mn), cn = exp2f(mj[q] - Mn);
                Lr = Lr * co + lj[q] * cn;
                Or.x = Or.x * co + oj[q].x * cn;
                Or.y = Or.y * co + oj[q].y * cn;
                Or.z = Or.z * co + oj[q].z * cn;
                Or.w = Or.w * co + oj[q].w * cn;
                Mr = Mn;
              }
            }
            const float inv = 1.0f / Lr;
            *reinterpret_cast<float4*>(out + (size_t)h * 128 + d4 * 4) =
                make_float4(Or.x * inv, Or.y * inv, Or.z * inv, Or.w * inv);
          }
          if (ct == 0) a.seg_cnt[seg] = 0;
        }
      }
      cons_sync();  // shared merge space is reused
      t += n_local;
    }
  };

  for (int k = 1; k <= a.K; ++k) {
    weights_phase(P_EH, k);
    if (!grid_sync(false)) return;
    weights_phase(P_QKV, k);
    if (!grid_sync(true)) return;
    attn_phase(k);
    if (!grid_sync(false)) return;
    weights_phase(P_O, k);
    if (!grid_sync(false)) return;
    weights_phase(P_GU, k);
    if (!grid_sync(false)) return;
    weights_phase(P_DOWN, k);
    if (!grid_sync(false)) return;
    if (k == a.K) pdl_trigger();
    weights_phase(P_LM, k);
    if (!grid_sync(false)) return;
    if (cta == 0 && ct < a.B) {
      const unsigned long long key = __ldcg(a.keys + (size_t)(k - 1) * a.B + ct);
      MTP_STORE(a.err, a.draft_ids, (size_t)ct * a.K + (k - 1), (long long)a.B * a.K, (int32_t)key_index(key));
      if (!((s_bad >> ct) & 1u)) MTP_STORE(a.err, a.pending, ct, a.B, k);
    }
  }
}

// ------------------------------------------------------------------ host

// Chunk width for rows of C columns: the fewest chunks of at most kPMaxCW
// columns that split C evenly into multiples of 8.
static int p_chunk(int C) {
  int n = (C + kPMaxCW - 1) / kPMaxCW;
  while (n <= C && (C % n || (C / n) % 8)) ++n;
  return C / n;
}

struct PPlan {
  int nslots, warps;
  size_t smem;
};

template <int NB>
static bool p_plan(const mtp_ctx* ctx, int grid, PPlan* plan) {
  const mtp_config& c = ctx->cfg;
  const int G = c.n_q_heads / c.n_kv_heads;
  // projection phases: the fp32 input chunk, plus per-unit results when a
  // row spans several chunks
  const int P[6] = {c.hidden / 2, (ctx->q_dim + 2 * ctx->kv_dim) / 2, c.hidden / 2, c.ffn, c.hidden / 2,
                    (c.vocab + 1) / 2};
  const int C[6] = {2 * c.hidden, c.hidden, ctx->q_dim, c.hidden, c.ffn, c.hidden};
  const int CW[6] = {p_chunk(c.hidden), p_chunk(c.hidden), p_chunk(ctx->q_dim), p_chunk(c.hidden),
                     p_chunk(c.ffn), p_chunk(c.hidden)};
  size_t weights_bytes = 0;
  for (int i = 0; i < 6; ++i) {
    const int nch = C[i] / CW[i];
    size_t bytes = (size_t)NB * CW[i] * 4;
    if (nch > 1) bytes += (size_t)nch * (((size_t)P[i] + grid - 1) / grid) * 2 * NB * 4;
    if (bytes > weights_bytes) weights_bytes = bytes;
  }
  const size_t attn_bytes = (size_t)kPW * G * 128 * 4;
  const size_t uni = weights_bytes > attn_bytes ? weights_bytes : attn_bytes;
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, p_draft_kernel<NB>) != cudaSuccess) return false;
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, ctx->device) != cudaSuccess)
    return false;
  const long long room = (long long)optin - (long long)fa.sharedSizeBytes - 1024 - (long long)uni;
  int max_slots = room > 0 ? (int)(room / kPSlot) : 0;
  if (max_slots > kPMaxSlots) max_slots = kPMaxSlots;
  // slots must be a multiple of the consumer warps: the most slots, then the
  // most warps
  int best_ns = 0, best_w = 0;
  for (int w = kPW; w >= 2; --w) {
    const int ns = w * (max_slots / w);
    if (ns > best_ns) {
      best_ns = ns;
      best_w = w;
    }
  }
  if (best_ns < 4) return false;
  plan->nslots = best_ns;
  plan->warps = best_w;
  plan->smem = 1024 + (size_t)best_ns * kPSlot + uni;
  return true;
}

bool persistent_supported(const mtp_ctx* ctx, int B) {
  const mtp_config& c = ctx->cfg;
  return ctx->p_ws != nullptr && B >= 1 && B <= ctx->p_max_batch && c.dtype == MTP_DTYPE_BF16 &&
         c.head_dim == 128 && c.hidden % 8 == 0 && c.ffn % 8 == 0;
}

template <int NB>
static cudaError_t p_launch(mtp_ctx* ctx, cudaStream_t s, const PArgs& a, const CUtensorMap& km,
                            const CUtensorMap& vm) {
  const int pi = NB == 1 ? 0 : NB == 2 ? 1 : 2;
  auto kern = p_draft_kernel<NB>;
  if (ctx->p_nslots[pi] == 0) {
    PPlan plan;
    if (!p_plan<NB>(ctx, a.max_recs, &plan)) return cudaErrorInvalidConfiguration;
    cudaError_t e = ensure_smem((const void*)kern, plan.smem);
    if (e != cudaSuccess) return e;
    ctx->p_nslots[pi] = plan.nslots;
    ctx->p_warps[pi] = plan.warps;
    ctx->p_smem[pi] = plan.smem;
  }
  PArgs args = a;
  args.nslots = ctx->p_nslots[pi];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.max_recs);
  cfg.blockDim = dim3(32 * (ctx->p_warps[pi] + 1));
  cfg.dynamicSmemBytes = ctx->p_smem[pi];
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, km, vm, args);
}

cudaError_t launch_draft_persistent(mtp_ctx* ctx, cudaStream_t s, int B, int K, const void* hidden,
                                    const void* embeds, const int32_t* positions, const mtp_kv* kv,
                                    const int32_t* chain_ids, int32_t* draft_ids, float* logits,
                                    float* hidden_out) {
  const mtp_config& c = ctx->cfg;
  const CUtensorMap *kmp, *vmp;
  if (!attn_tensor_maps(ctx, kv, &kmp, &vmp)) return cudaErrorInvalidValue;
  PArgs a;
  memset(&a, 0, sizeof(a));
  a.B = B; a.H = c.hidden; a.q_dim = ctx->q_dim; a.kv_dim = ctx->kv_dim; a.F = c.ffn; a.V = c.vocab;
  a.n_q = c.n_q_heads; a.n_kv = c.n_kv_heads; a.G = c.n_q_heads / c.n_kv_heads; a.K = K;
  a.max_pos = c.max_pos; a.num_blocks = kv->num_blocks; a.max_blocks = kv->max_blocks;
  a.cw_h = p_chunk(c.hidden); a.cw_q = p_chunk(ctx->q_dim); a.cw_f = p_chunk(c.ffn);
  a.max_recs = ctx->num_sms;
  a.eps = c.eps;
  a.qscale = 1.4426950408889634f / sqrtf((float)c.head_dim);
  const mtp_weights& w = ctx->w;
  a.w_norm_h = (const uint16_t*)w.w_norm_h; a.w_norm_e = (const uint16_t*)w.w_norm_e;
  a.w_eh = (const uint16_t*)w.w_eh; a.w_norm_in = (const uint16_t*)w.w_norm_in;
  a.w_q = (const uint16_t*)w.w_q; a.w_k = (const uint16_t*)w.w_k; a.w_v = (const uint16_t*)w.w_v;
  a.w_o = (const uint16_t*)w.w_o; a.w_norm_post = (const uint16_t*)w.w_norm_post;
  a.w_gate = (const uint16_t*)w.w_gate; a.w_up = (const uint16_t*)w.w_up; a.w_down = (const uint16_t*)w.w_down;
  a.w_norm_f = (const uint16_t*)w.w_norm_f; a.embed = (const uint16_t*)w.embed;
  a.lm_head = (const uint16_t*)w.lm_head;
  a.hidden_in = (const uint16_t*)hidden; a.embeds_in = (const uint16_t*)embeds; a.positions = positions;
  a.chain_ids = chain_ids; a.draft_ids = draft_ids; a.logits = logits; a.hidden_out = hidden_out;
  a.k_pool = (uint16_t*)kv->k_pool; a.v_pool = (uint16_t*)kv->v_pool; a.block_table = kv->block_table;
  a.seq_len = kv->seq_len; a.pending = kv->pending;
  a.hid = ctx->hid; a.x = ctx->x; a.q = ctx->q; a.attn = ctx->attn; a.h1 = ctx->h1; a.act = ctx->act;
  a.rec = ctx->p_rec; a.seg_cnt = ctx->p_seg_cnt; a.keys = ctx->p_keys; a.gbar = ctx->p_gbar;
  a.err = ctx->err; a.rope = ctx->rope;

  prof_before(ctx, MTP_KERNEL_DRAFT_PERSISTENT, s);
  cudaError_t e;
  if (B <= 1) e = p_launch<1>(ctx, s, a, *kmp, *vmp);
  else if (B <= 2) e = p_launch<2>(ctx, s, a, *kmp, *vmp);
  else e = p_launch<4>(ctx, s, a, *kmp, *vmp);
  prof_after(ctx, MTP_KERNEL_DRAFT_PERSISTENT, s);
  ctx->launches++;
  return e;
}

// ------------------------------------------------------------ diagnostics
//
// Runs one of the library's bounded waits on a condition that never becomes
// true, so that it runs out the way a lost arrival or a missing CTA would make
// it run out in a real launch: which = 0, the mbarrier phase wait of the
// streamed kernels (an mbarrier nobody arrives at, kSelftestPolls polls);
// which = 1, the persistent kernel's grid-barrier counter wait (a private
// counter nobody increments; 2 s of %globaltimer).  No copy is ever in flight,
// so the CTA may exit as soon as the wait gives up.
constexpr uint32_t kSelftestPolls = 1u << 12;
static __device__ unsigned long long g_selftest_counter[64];

__global__ void selftest_wait_kernel(int which, int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_abort;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    s_abort = 0;
  }
  fence_mbar_init();
  __syncthreads();
  if (which == 0) {
    const bool ok = mbar_wait_bounded(&bar, 0u, kSelftestPolls);
    if (!ok && threadIdx.x == 0) set_error(err, MTP_ERR_TIMEOUT);
  } else if (threadIdx.x == 0) {
    PArgs a;
    memset(&a, 0, sizeof(a));
    a.gbar = g_selftest_counter;
    a.err = err;
    p_wait_count(a, 1ull, &s_abort);
  }
}

cudaError_t launch_selftest_wait(mtp_ctx* ctx, cudaStream_t s, int which) {
  void* counter = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&counter, g_selftest_counter);
  if (e != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(counter, 0, sizeof(g_selftest_counter), s)) != cudaSuccess) return e;
  selftest_wait_kernel<<<1, 64, 0, s>>>(which, ctx->err);
  ctx->launches++;
  return cudaGetLastError();
}

}  // namespace mtp
