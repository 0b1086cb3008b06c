// Tree drafting with the MTP head ("Speculative Decoding" (OpenVINO GenAI),
// "Tree Drafting", "How Tree Drafting Works" steps 1-4, with its validation
// rules), tree verification and the cache commit of the accepted path.
//
// Layer 1 is the MTP step from the verifier's hidden state and the last
// token; it proposes the bf most probable tokens.  At layer l >= 2 the bf
// candidates of layer l-1 with the highest cumulative log-probability (all of
// them at l = 2) are expanded, each by one MTP step whose input is the node's
// token and the output hidden state of the step that proposed it, at position
// p + l - 1, attending over the committed cache plus the MTP entries of its
// ancestors.  Expansions run on the per-step kernels as "virtual requests":
// a block table that shares the request's committed blocks and holds private
// copies of the blocks from the one containing the last committed slot on
// (the root entry and the ancestors' entries live there), with the step
// counted as the second of a call (its hidden state read from the fp32
// recursion buffer, its token given as the chain input).  The n_assist
// candidates with the best cumulative score form the packed tree (parents
// first).  Verification walks from the root along children whose token is
// the verifier's prediction; the commit keeps the root's entry and the
// accepted nodes' entries that were expanded.
#include <string.h>

#include "mtp_common.cuh"

namespace mtp {

constexpr int kTreeMaxBf = 8;
constexpr int kTreeMaxDepth = 16;
constexpr int kTreeMaxAssist = 64;
constexpr int kTreeMaxCand = 1024;

// Workspace layout of one tree call (byte offsets, 256-byte aligned).
struct TreeLayout {
  int nV, NL, NC, rows;
  size_t root_hid, hid_out, step_logits, step_ids, chain, vbt, vseq, vpend, vpos, topk_tok, topk_lp;
  size_t cand_tok, cand_par, cand_depth, cand_src, cand_exp, cand_score, cand_n, surv, sel, keys, path_nodes;
  size_t copy_src, copy_dst, part_ms, part_keys, total;
};

constexpr int kTopkSlices = 64;

static size_t tl_align(size_t x) { return (x + 255) & ~(size_t)255; }

static TreeLayout tree_layout(const mtp_ctx* ctx, int B, int bf, int td, int n_assist, int max_blocks) {
  TreeLayout t;
  const size_t H = ctx->cfg.hidden, V = ctx->cfg.vocab;
  t.nV = B * bf;
  t.NL = td - 1;
  t.NC = bf + bf * bf * t.NL;
  t.rows = B > t.nV ? B : t.nV;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t r = o;
    o = tl_align(o + bytes);
    return r;
  };
  // sizes independent of the cache's block-table width first, so that the
  // verify step (which has no cache) finds its buffers at the same offsets
  t.root_hid = take((size_t)B * H * 4);
  t.hid_out = take((size_t)(t.NL > 0 ? t.NL : 1) * t.nV * H * 4);
  t.step_logits = take((size_t)t.rows * 2 * V * 4);
  t.step_ids = take((size_t)t.rows * 2 * 4);
  t.chain = take((size_t)t.nV * 4);
  t.topk_tok = take((size_t)t.rows * bf * 4);
  t.topk_lp = take((size_t)t.rows * bf * 4);
  const size_t nc = (size_t)B * t.NC;
  t.cand_tok = take(nc * 4);
  t.cand_par = take(nc * 4);
  t.cand_depth = take(nc * 4);
  t.cand_src = take(nc * 4);
  t.cand_exp = take(nc * 4);
  t.cand_score = take(nc * 4);
  t.cand_n = take((size_t)B * 4);
  t.surv = take((size_t)B * bf * 4);
  t.sel = take((size_t)B * n_assist * 4);
  t.keys = take((size_t)B * (1 + n_assist) * 8);
  t.path_nodes = take((size_t)B * td * 4);
  t.copy_src = take((size_t)t.nV * 2 * 4);
  t.copy_dst = take((size_t)t.nV * 2 * 4);
  t.part_ms = take((size_t)t.rows * kTopkSlices * 2 * 4);
  t.part_keys = take((size_t)t.rows * kTopkSlices * bf * 8);
  const size_t nl = (size_t)(t.NL > 0 ? t.NL : 1) * t.nV;
  t.vseq = take(nl * 4);
  t.vpend = take(nl * 4);
  t.vpos = take(nl * 4);
  t.vbt = take(nl * max_blocks * 4);
  t.total = o;
  return t;
}

// Top-bf tokens of a logits row (larger first, lower id on ties) and their
// log-softmax values, in two kernels.  Partial: grid (slices, rows); each
// block takes one vocabulary slice and writes its max, its sum of
// exp(z - max) and its top-bf keys (orderable value, lowest id on ties).
__global__ void tree_topk_partial_kernel(const float* logits, size_t row_stride, size_t row_off, int V, int bf,
                                         float* part_ms, unsigned long long* part_keys) {
  __shared__ unsigned long long cand[256 * kTreeMaxBf];
  __shared__ float red[8];
  const int row = blockIdx.y, sl = blockIdx.x;
  const float* z = logits + (size_t)row * row_stride + row_off;
  const int per = (V + kTopkSlices - 1) / kTopkSlices;
  const int v0 = sl * per, v1 = min(V, v0 + per);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  float m = -INFINITY;
  unsigned long long top[kTreeMaxBf];
#pragma unroll
  for (int i = 0; i < kTreeMaxBf; ++i) top[i] = 0ull;
  for (int v = v0 + threadIdx.x; v < v1; v += 256) {
    const float x = z[v];
    m = fmaxf(m, x);
    unsigned long long key = argmax_key(x, (uint32_t)v);
#pragma unroll
    for (int i = 0; i < kTreeMaxBf; ++i) {   // insertion into the descending list
      if (i < bf && key > top[i]) {
        const unsigned long long t = top[i];
        top[i] = key;
        key = t;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[w] = m;
#pragma unroll
  for (int i = 0; i < kTreeMaxBf; ++i) cand[threadIdx.x * kTreeMaxBf + i] = (i < bf) ? top[i] : 0ull;
  __syncthreads();
  m = red[0];
  for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  float sum = 0.0f;
  if (m > -INFINITY)
    for (int v = v0 + threadIdx.x; v < v1; v += 256) sum += expf(z[v] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) red[w] = sum;
  __syncthreads();
  if (w == 0) {
    const size_t pk = ((size_t)row * kTopkSlices + sl) * bf;
    for (int r = 0; r < bf; ++r) {
      unsigned long long best = 0ull;
      for (int i = lane; i < 256 * kTreeMaxBf; i += 32) best = umax64(best, cand[i]);
      best = warp_max_u64(best);
      for (int i = lane; i < 256 * kTreeMaxBf; i += 32)
        if (cand[i] == best) cand[i] = 0ull;
      __syncwarp();
      if (lane == 0) part_keys[pk + r] = best;
    }
    if (lane == 0) {
      float tot = 0.0f;
      for (int i = 0; i < 8; ++i) tot += red[i];
      part_ms[((size_t)row * kTopkSlices + sl) * 2] = m;
      part_ms[((size_t)row * kTopkSlices + sl) * 2 + 1] = tot;
    }
  }
}

// Merge: one warp per row; slices combined in order (deterministic).
__global__ void tree_topk_merge_kernel(const float* logits, size_t row_stride, size_t row_off, int bf,
                                       const float* part_ms, unsigned long long* part_keys, int32_t* out_tok,
                                       float* out_lp) {
  const int row = blockIdx.x, lane = threadIdx.x;
  const float* z = logits + (size_t)row * row_stride + row_off;
  const float* pm = part_ms + (size_t)row * kTopkSlices * 2;
  float m = -INFINITY;
  for (int i = 0; i < kTopkSlices; ++i) m = fmaxf(m, pm[2 * i]);
  float sum = 0.0f;
  for (int i = 0; i < kTopkSlices; ++i)
    if (pm[2 * i] > -INFINITY) sum += pm[2 * i + 1] * expf(pm[2 * i] - m);
  const float lse = m + logf(sum);
  unsigned long long* pk = part_keys + (size_t)row * kTopkSlices * bf;
  for (int r = 0; r < bf; ++r) {
    unsigned long long best = 0ull;
    for (int i = lane; i < kTopkSlices * bf; i += 32) best = umax64(best, pk[i]);
    best = warp_max_u64(best);
    for (int i = lane; i < kTopkSlices * bf; i += 32)
      if (pk[i] == best) pk[i] = 0ull;
    __syncwarp();
    if (lane == 0) {
      const int idx = best ? (int)key_index(best) : 0;
      out_tok[(size_t)row * bf + r] = idx;
      out_lp[(size_t)row * bf + r] = z[idx] - lse;
    }
  }
}

struct TreeCand {
  int32_t *tok, *par, *depth, *src, *exp, *n;
  float* score;
};

// Layer 1: the root's bf children.
__global__ void tree_root_kernel(int B, int bf, int NC, const int32_t* topk_tok, const float* topk_lp, TreeCand c) {
  const int b = blockIdx.x;
  for (int i = threadIdx.x; i < bf; i += blockDim.x) {
    const size_t k = (size_t)b * NC + i;
    c.tok[k] = topk_tok[(size_t)b * bf + i];
    c.score[k] = topk_lp[(size_t)b * bf + i];
    c.par[k] = -1;
    c.depth[k] = 1;
    c.src[k] = -1;
    c.exp[k] = -1;
  }
  if (threadIdx.x == 0) c.n[b] = bf;
}

// Children of layer l's expansions: survivor i of request b expanded as
// virtual request v = b * bf + i proposes its bf most probable tokens.
__global__ void tree_children_kernel(int bf, int NC, int l, const int32_t* surv, const int32_t* topk_tok,
                                     const float* topk_lp, TreeCand c) {
  const int b = blockIdx.x;
  const int n0 = c.n[b];
  for (int t = threadIdx.x; t < bf * bf; t += blockDim.x) {
    const int i = t / bf, j = t - i * bf;
    const int v = b * bf + i;
    const int s = surv[(size_t)b * bf + i];
    const size_t k = (size_t)b * NC + n0 + t;
    c.tok[k] = topk_tok[(size_t)v * bf + j];
    c.score[k] = c.score[(size_t)b * NC + s] + topk_lp[(size_t)v * bf + j];
    c.par[k] = s;
    c.depth[k] = l;
    c.src[k] = v;
    c.exp[k] = -1;
  }
  __syncthreads();
  if (threadIdx.x == 0) c.n[b] = n0 + bf * bf;
}

// a is better than b: higher score, then smaller depth, then created earlier.
__device__ __forceinline__ bool cand_better(float sa, int da, int ia, float sb, int db, int ib) {
  if (sa != sb) return sa > sb;
  if (da != db) return da < db;
  return ia < ib;
}

// Set up layer l (>= 2): pick the survivors, give each a virtual request
// (block table, length, pending, position, token), gather its hidden state
// (the output of the step that proposed it) into the recursion buffer, and
// list the private blocks to copy.  One block per request.
struct TreeSetupArgs {
  int B, bf, NC, l, H, max_blocks, num_blocks, nV;
  const int32_t* real_bt;        // [B, max_blocks]
  const int32_t* real_seq;       // [B]
  const int32_t* positions;      // [B]
  const int32_t* scratch;        // [(td - 1) * nV * 2] free block ids
  const float* root_hid;         // [B, H]
  const float* hid_out;          // [NL, nV, H]
  float* hid;                    // the context's recursion buffer [maxB, H]
  int32_t *vbt, *vseq, *vpend, *vpos;   // this layer's slices
  const int32_t* vbt_prev;       // the previous layer's block tables (l >= 3)
  int32_t *chain, *surv, *copy_src, *copy_dst;
  int* err;
};

__global__ void tree_setup_kernel(TreeSetupArgs a, TreeCand c) {
  __shared__ int s_surv[kTreeMaxBf];
  __shared__ float s_score[kTreeMaxBf * kTreeMaxBf];
  __shared__ int s_depth[kTreeMaxBf * kTreeMaxBf];
  const int b = blockIdx.x;
  const int bf = a.bf, l = a.l, e = l - 2;
  const int n = c.n[b];
  const size_t cb = (size_t)b * a.NC;
  if (l == 2) {
    if (threadIdx.x < bf) s_surv[threadIdx.x] = threadIdx.x;
  } else {
    // the bf * bf candidates of layer l - 1 are the last ones created; rank
    // them (higher score, then earlier creation) and keep the first bf
    const int c0 = n - bf * bf;
    for (int t = threadIdx.x; t < bf * bf; t += blockDim.x) {
      s_score[t] = c.score[cb + c0 + t];
      s_depth[t] = c.depth[cb + c0 + t];
    }
    __syncthreads();
    for (int t = threadIdx.x; t < bf * bf; t += blockDim.x) {
      int rank = 0;
      for (int u = 0; u < bf * bf; ++u)
        if (u != t && cand_better(s_score[u], s_depth[u], c0 + u, s_score[t], s_depth[t], c0 + t)) ++rank;
      if (rank < bf) s_surv[rank] = c0 + t;
    }
  }
  __syncthreads();
  const int L = a.real_seq[b];
  const int bL = L / 16;
  const bool fits = bL + 1 < a.max_blocks;
  __shared__ int s_p0[kTreeMaxBf], s_p1[kTreeMaxBf], s_ok[kTreeMaxBf];
  if (!fits && threadIdx.x == 0) set_error(a.err, MTP_ERR_CAPACITY);
  const int32_t* real = a.real_bt + (size_t)b * a.max_blocks;
  for (int i = threadIdx.x; i < bf; i += blockDim.x) {
    const int s = s_surv[i];
    const int v = b * bf + i;
    a.surv[(size_t)b * bf + i] = s;
    c.exp[cb + s] = v;
    a.chain[v] = c.tok[cb + s];
    a.vseq[v] = L + l - 2;
    a.vpend[v] = 1;
    a.vpos[v] = a.positions[b] + l - 2;
    const int32_t p0 = a.scratch[((size_t)e * a.nV + v) * 2], p1 = a.scratch[((size_t)e * a.nV + v) * 2 + 1];
    const bool ok = fits && p0 >= 0 && p0 < a.num_blocks && p1 >= 0 && p1 < a.num_blocks;
    if (!ok) set_error(a.err, MTP_ERR_DEVICE_ARGS);
    s_p0[i] = p0;
    s_p1[i] = p1;
    s_ok[i] = ok;
    // private blocks start as copies of the proposer's: the request's own
    // blocks for a layer-1 node, the proposing expansion's private blocks
    // otherwise; the second holds entries only once the path reaches it
    const int src = c.src[cb + s];
    const int32_t* from = (src < 0) ? real : a.vbt_prev + (size_t)src * a.max_blocks;
    a.copy_src[v * 2] = (ok) ? from[bL] : -1;
    a.copy_dst[v * 2] = (ok) ? p0 : -1;
    const int last_slot = L + l - 2;   // the proposer's own entry
    a.copy_src[v * 2 + 1] = (ok && last_slot >= (bL + 1) * 16) ? from[bL + 1] : -1;
    a.copy_dst[v * 2 + 1] = (ok && last_slot >= (bL + 1) * 16) ? p1 : -1;
  }
  __syncthreads();
  // block tables: the request's own, with the two private blocks in place
  for (int t = threadIdx.x; t < bf * a.max_blocks; t += blockDim.x) {
    const int i = t / a.max_blocks, j = t - i * a.max_blocks;
    int32_t val = real[j];
    if (s_ok[i] && j == bL) val = s_p0[i];
    if (s_ok[i] && j == bL + 1) val = s_p1[i];
    a.vbt[(size_t)(b * bf + i) * a.max_blocks + j] = val;
  }
  // hidden states of the survivors' proposers: 16-byte copies, four loads
  // issued before their stores (the rows are 16-byte aligned when H % 4 == 0)
  for (int i = 0; i < bf; ++i) {
    const int src = c.src[cb + s_surv[i]];
    const float* from = (src < 0) ? a.root_hid + (size_t)b * a.H
                                  : a.hid_out + ((size_t)(e - 1) * a.nV + src) * a.H;
    float* to = a.hid + (size_t)(b * bf + i) * a.H;
    const bool vec = (a.H & 3) == 0 && ((uintptr_t)from & 15) == 0 && ((uintptr_t)to & 15) == 0;
    if (vec) {
      const int n4 = a.H >> 2;
      const float4* f4 = reinterpret_cast<const float4*>(from);
      float4* t4 = reinterpret_cast<float4*>(to);
      for (int h0 = threadIdx.x; h0 < n4; h0 += 4 * blockDim.x) {
        float4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int h = h0 + q * blockDim.x;
          if (h < n4) v[q] = __ldcg(f4 + h);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int h = h0 + q * blockDim.x;
          if (h < n4) t4[h] = v[q];
        }
      }
    } else {
      for (int h = threadIdx.x; h < a.H; h += blockDim.x) to[h] = __ldcg(from + h);
    }
  }
}

// Copy whole cache blocks (K and V pools) for the pairs listed (-1: none).
template <typename T>
__global__ void tree_block_copy_kernel(const int32_t* src, const int32_t* dst, T* k_pool, T* v_pool,
                                       size_t block_elems, int num_blocks) {
  const int pair = blockIdx.y;
  const int s = src[pair], d = dst[pair];
  if (s < 0 || d < 0 || s >= num_blocks || d >= num_blocks) return;
  const size_t n16 = block_elems * sizeof(T) / 16;
  const uint4* ks = reinterpret_cast<const uint4*>(k_pool + (size_t)s * block_elems);
  const uint4* vs = reinterpret_cast<const uint4*>(v_pool + (size_t)s * block_elems);
  uint4* kd = reinterpret_cast<uint4*>(k_pool + (size_t)d * block_elems);
  uint4* vd = reinterpret_cast<uint4*>(v_pool + (size_t)d * block_elems);
  for (size_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
}

// The packed tree: the n_assist best candidates (score, then depth, then
// creation), ordered by (depth, creation) so that parents come first.
__global__ void tree_select_kernel(int n_assist, int NC, TreeCand c, int32_t* sel, int32_t* tokens, int32_t* parents,
                                   int32_t* depths) {
  __shared__ int s_pos[kTreeMaxCand];   // packed position of a selected candidate, -1 otherwise
  const int b = blockIdx.x;
  const size_t cb = (size_t)b * NC;
  const int n = c.n[b];
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    int rank = 0;
    for (int j = 0; j < n; ++j)
      if (j != i && cand_better(c.score[cb + j], c.depth[cb + j], j, c.score[cb + i], c.depth[cb + i], i)) ++rank;
    s_pos[i] = rank < n_assist ? 0 : -1;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    if (s_pos[i] < 0) continue;
    int pos = 0;
    for (int j = 0; j < n; ++j)
      if (s_pos[j] >= 0 && (c.depth[cb + j] < c.depth[cb + i] || (c.depth[cb + j] == c.depth[cb + i] && j < i))) ++pos;
    sel[(size_t)b * n_assist + pos] = i;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < n_assist; p += blockDim.x) {
    const int i = sel[(size_t)b * n_assist + p];
    s_pos[i] = p;
  }
  __syncthreads();
  for (int p = threadIdx.x; p < n_assist; p += blockDim.x) {
    const int i = sel[(size_t)b * n_assist + p];
    const int par = c.par[cb + i];
    tokens[(size_t)b * n_assist + p] = c.tok[cb + i];
    depths[(size_t)b * n_assist + p] = c.depth[cb + i];
    parents[(size_t)b * n_assist + p] = par < 0 ? -1 : s_pos[par];
  }
}

// ------------------------------------------------------------ verification

__device__ __forceinline__ uint64_t t_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Synthetic verifier rows of the packed trees (the loop harness's verifier,
// include/mtp.h): request b's rows start at b * (1 + n_assist); row 0 follows
// the committed prefix, row 1 + i the prefix extended by node i's path.
template <typename T>
__global__ void tree_synth_kernel(int n_assist, int depth_max, const int32_t* tokens, const int32_t* parents,
                                  const uint64_t* seq_hash, const int32_t* last_tok, uint64_t thr, int V, int slice,
                                  T* logits) {
  const int r = blockIdx.y;
  const int b = r / (1 + n_assist), i = r - b * (1 + n_assist) - 1;
  uint64_t h = seq_hash[b];
  int32_t last = last_tok[b];
  if (i >= 0) {
    int32_t path[kTreeMaxDepth];
    int len = 0, node = i;
    while (node >= 0 && len < depth_max) {
      path[len++] = tokens[(size_t)b * n_assist + node];
      node = parents[(size_t)b * n_assist + node];
    }
    for (int j = len - 1; j >= 0; --j) {
      h = t_mix64(h + 0x9E3779B97F4A7C15ull * (uint64_t)((int64_t)path[j] + 1));
      last = path[j];
    }
  }
  int32_t tgt;
  if ((t_mix64(h ^ 0xD1B54A32D192ED03ull) >> 11) < thr) tgt = last;
  else tgt = (int32_t)(t_mix64(h ^ 0x8CB92BA72F3D8DD7ull) % (uint64_t)V);
  const int v0 = blockIdx.x * slice, v1 = min(V, v0 + slice);
  T* row = logits + (size_t)r * V;
  for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
    const float x = (v == tgt) ? 8.0f
                               : (float)(uint32_t)(t_mix64(h ^ (0x9E3779B97F4A7C15ull * ((uint64_t)v + 1))) >> 40) *
                                         5.9604644775390625e-08f - 0.5f;
    if constexpr (sizeof(T) == 2) row[v] = f32_to_bf16_rne(x);
    else row[v] = x;
  }
}

// Row argmax keys (orderable value, lowest id on ties) by slices.
template <typename T>
__global__ void tree_row_argmax_kernel(const T* logits, int V, int slice, unsigned long long* keys) {
  const int r = blockIdx.y;
  const T* row = logits + (size_t)r * V;
  const int v0 = blockIdx.x * slice, v1 = min(V, v0 + slice);
  unsigned long long best = 0ull;
  for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
    float x;
    if constexpr (sizeof(T) == 2) x = __uint_as_float((uint32_t)row[v] << 16);
    else x = row[v];
    best = umax64(best, argmax_key(x, (uint32_t)v));
  }
  best = warp_max_u64(best);
  if ((threadIdx.x & 31) == 0 && best) atomicMax(keys + r, best);
}

// Walk from the root along the child whose token is the current prediction.
__global__ void tree_accept_kernel(int B, int n_assist, int td, const int32_t* tokens, const int32_t* parents,
                                   unsigned long long* keys, int32_t* accepted, int32_t* bonus, int32_t* path_tokens,
                                   int32_t* path_nodes) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  unsigned long long* kb = keys + (size_t)b * (1 + n_assist);
  int node = -1, a = 0;
  int32_t pred = (int32_t)key_index(kb[0]);
  while (a < td) {
    int next = -1;
    for (int i = 0; i < n_assist; ++i)
      if (parents[(size_t)b * n_assist + i] == node && tokens[(size_t)b * n_assist + i] == pred) {
        next = i;
        break;
      }
    if (next < 0) break;
    path_tokens[(size_t)b * td + a] = pred;
    path_nodes[(size_t)b * td + a] = next;
    ++a;
    node = next;
    pred = (int32_t)key_index(kb[1 + node]);
  }
  accepted[b] = a;
  bonus[b] = pred;
  for (int i = 0; i <= n_assist; ++i) kb[i] = 0ull;   // ready for the next call
}

// Keep the root's entry (slot L, written by the root step) and the entries
// of the accepted nodes that were expanded (node at depth d: slot L + d of
// its expansion's private block), then advance the cache.
template <typename T>
__global__ void tree_commit_kernel(int n_assist, int NC, int td, int n_kv, int hd, int max_blocks, int num_blocks,
                                   const int32_t* accepted, const int32_t* path_nodes, const int32_t* sel,
                                   const int32_t* cand_exp, const int32_t* vbt, int nV, T* k_pool, T* v_pool,
                                   const int32_t* real_bt, int32_t* seq_len, int32_t* pending, int* err) {
  __shared__ int s_m;
  const int b = blockIdx.x;
  const int L = seq_len[b];
  if (threadIdx.x == 0) {
    int m = 0;
    const int a = accepted[b];
    while (m < a) {
      const int node = path_nodes[(size_t)b * td + m];
      const int cand = sel[(size_t)b * n_assist + node];
      if (cand_exp[(size_t)b * NC + cand] < 0) break;
      ++m;
    }
    s_m = m;
  }
  __syncthreads();
  const int m = s_m;
  const size_t ent = (size_t)n_kv * hd;   // elements of one slot over the kv heads
  for (int j = 0; j < m; ++j) {
    const int d = j + 1;
    const int node = path_nodes[(size_t)b * td + j];
    const int v = cand_exp[(size_t)b * NC + sel[(size_t)b * n_assist + node]];
    const int slot = L + d;
    const int sb = vbt[((size_t)j * nV + v) * max_blocks + slot / 16];
    const int db = (slot / 16 < max_blocks) ? real_bt[(size_t)b * max_blocks + slot / 16] : -1;
    if (sb < 0 || sb >= num_blocks || db < 0 || db >= num_blocks) {
      if (threadIdx.x == 0) set_error(err, MTP_ERR_CAPACITY);
      break;
    }
    for (size_t t = threadIdx.x; t < ent; t += blockDim.x) {
      const int h = (int)(t / hd), x = (int)(t - (size_t)h * hd);
      const size_t so = (((size_t)sb * n_kv + h) * 16 + slot % 16) * hd + x;
      const size_t dof = (((size_t)db * n_kv + h) * 16 + slot % 16) * hd + x;
      k_pool[dof] = k_pool[so];
      v_pool[dof] = v_pool[so];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    seq_len[b] = L + 1 + m;
    pending[b] = 0;
  }
}

}  // namespace mtp

// ------------------------------------------------------------------ host

using namespace mtp;

static mtp_status tree_status(cudaError_t e) {
  if (e == cudaSuccess) return MTP_OK;
  cudaGetLastError();
  return MTP_ERR_CUDA;
}

static bool tree_shape_ok(const mtp_ctx* ctx, const mtp_tree* t) {
  if (!ctx || !t || t->B < 1 || t->branching < 1 || t->branching > kTreeMaxBf) return false;
  if (t->depth < 1 || t->depth > kTreeMaxDepth || t->n_assist > kTreeMaxAssist) return false;
  const int bf = t->branching, td = t->depth;
  if (bf * bf * (td - 1) + bf < t->n_assist || t->n_assist < td) return false;   // the page's two rules
  if (bf + bf * bf * (td - 1) > kTreeMaxCand) return false;
  if (t->B * bf > ctx->cfg.max_batch || t->B > ctx->cfg.max_batch) return false;
  if (td >= 2 && ctx->cfg.max_k < 2) return false;
  return t->ws && t->tokens && t->parents && t->depths;
}

extern "C" size_t mtp_tree_workspace_bytes(const mtp_ctx* ctx, int B, int branching, int depth, int n_assist,
                                           int max_blocks) {
  if (!ctx || B < 1 || branching < 1 || depth < 1 || n_assist < 1 || max_blocks < 1) return 0;
  return tree_layout(ctx, B, branching, depth, n_assist, max_blocks).total;
}

static TreeCand tree_cands(const TreeLayout& L, char* ws) {
  TreeCand c;
  c.tok = (int32_t*)(ws + L.cand_tok);
  c.par = (int32_t*)(ws + L.cand_par);
  c.depth = (int32_t*)(ws + L.cand_depth);
  c.src = (int32_t*)(ws + L.cand_src);
  c.exp = (int32_t*)(ws + L.cand_exp);
  c.n = (int32_t*)(ws + L.cand_n);
  c.score = (float*)(ws + L.cand_score);
  return c;
}

extern "C" mtp_status mtp_draft_tree(mtp_ctx* ctx, void* stream, const void* hidden, const void* embeds,
                                     const int32_t* positions, const mtp_kv* kv, const mtp_tree* t) {
  if (!tree_shape_ok(ctx, t) || !ctx->has_weights || !hidden || !embeds || !positions || !kv) return MTP_ERR_INVALID;
  if (!kv->k_pool || !kv->v_pool || !kv->block_table || !kv->seq_len || !kv->pending || kv->max_blocks < 2)
    return MTP_ERR_INVALID;
  if (t->depth >= 2 && !t->scratch_blocks) return MTP_ERR_INVALID;
  const int B = t->B, bf = t->branching, td = t->depth;
  const TreeLayout Lo = tree_layout(ctx, B, bf, td, t->n_assist, kv->max_blocks);
  if (t->ws_bytes < Lo.total) return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = (char*)t->ws;
  const size_t V = ctx->cfg.vocab, H = ctx->cfg.hidden;
  float* step_logits = (float*)(ws + Lo.step_logits);
  int32_t* step_ids = (int32_t*)(ws + Lo.step_ids);
  int32_t* topk_tok = (int32_t*)(ws + Lo.topk_tok);
  float* topk_lp = (float*)(ws + Lo.topk_lp);
  TreeCand c = tree_cands(Lo, ws);
  cudaError_t e;
  // layer 1: the root step on the requests' own caches (slot L)
  if ((e = draft_one_step(ctx, s, B, 1, 1, hidden, embeds, positions, kv, nullptr, step_ids, step_logits,
                          (float*)(ws + Lo.root_hid))) != cudaSuccess)
    return tree_status(e);
  float* part_ms = (float*)(ws + Lo.part_ms);
  unsigned long long* part_keys = (unsigned long long*)(ws + Lo.part_keys);
  tree_topk_partial_kernel<<<dim3(kTopkSlices, B), 256, 0, s>>>(step_logits, V, 0, (int)V, bf, part_ms, part_keys);
  tree_topk_merge_kernel<<<B, 32, 0, s>>>(step_logits, V, 0, bf, part_ms, part_keys, topk_tok, topk_lp);
  tree_root_kernel<<<B, 32, 0, s>>>(B, bf, Lo.NC, topk_tok, topk_lp, c);
  ctx->launches += 3;
  const size_t block_elems = (size_t)ctx->cfg.n_kv_heads * 16 * ctx->cfg.head_dim;
  for (int l = 2; l <= td; ++l) {
    const int ei = l - 2;
    TreeSetupArgs a;
    a.B = B; a.bf = bf; a.NC = Lo.NC; a.l = l; a.H = (int)H; a.max_blocks = kv->max_blocks;
    a.num_blocks = kv->num_blocks; a.nV = Lo.nV;
    a.real_bt = kv->block_table; a.real_seq = kv->seq_len; a.positions = positions; a.scratch = t->scratch_blocks;
    a.root_hid = (const float*)(ws + Lo.root_hid); a.hid_out = (const float*)(ws + Lo.hid_out); a.hid = ctx->hid;
    int32_t* vbt = (int32_t*)(ws + Lo.vbt) + (size_t)ei * Lo.nV * kv->max_blocks;
    a.vbt = vbt;
    a.vseq = (int32_t*)(ws + Lo.vseq) + (size_t)ei * Lo.nV;
    a.vpend = (int32_t*)(ws + Lo.vpend) + (size_t)ei * Lo.nV;
    a.vpos = (int32_t*)(ws + Lo.vpos) + (size_t)ei * Lo.nV;
    a.vbt_prev = ei > 0 ? vbt - (size_t)Lo.nV * kv->max_blocks : nullptr;
    a.chain = (int32_t*)(ws + Lo.chain); a.surv = (int32_t*)(ws + Lo.surv);
    a.copy_src = (int32_t*)(ws + Lo.copy_src); a.copy_dst = (int32_t*)(ws + Lo.copy_dst); a.err = ctx->err;
    tree_setup_kernel<<<B, 256, 0, s>>>(a, c);
    const dim3 cg(8, Lo.nV * 2);
    if (ctx->cfg.dtype == MTP_DTYPE_BF16)
      tree_block_copy_kernel<uint16_t><<<cg, 256, 0, s>>>(a.copy_src, a.copy_dst, (uint16_t*)kv->k_pool,
                                                          (uint16_t*)kv->v_pool, block_elems, kv->num_blocks);
    else
      tree_block_copy_kernel<float><<<cg, 256, 0, s>>>(a.copy_src, a.copy_dst, (float*)kv->k_pool,
                                                       (float*)kv->v_pool, block_elems, kv->num_blocks);
    ctx->launches += 2;
    if ((e = cudaMemsetAsync(ctx->req_bad, 0, (size_t)Lo.nV * sizeof(int), s)) != cudaSuccess) return tree_status(e);
    mtp_kv vk = *kv;
    vk.block_table = a.vbt;
    vk.seq_len = a.vseq;
    vk.pending = a.vpend;
    // the expansion, counted as the second step of a two-step call
    if ((e = draft_one_step(ctx, s, Lo.nV, 2, 2, hidden, embeds, a.vpos, &vk, a.chain, step_ids, step_logits,
                            (float*)(ws + Lo.hid_out) + (size_t)ei * Lo.nV * H)) != cudaSuccess)
      return tree_status(e);
    tree_topk_partial_kernel<<<dim3(kTopkSlices, Lo.nV), 256, 0, s>>>(step_logits, 2 * V, V, (int)V, bf, part_ms,
                                                                         part_keys);
    tree_topk_merge_kernel<<<Lo.nV, 32, 0, s>>>(step_logits, 2 * V, V, bf, part_ms, part_keys, topk_tok, topk_lp);
    tree_children_kernel<<<B, 64, 0, s>>>(bf, Lo.NC, l, a.surv, topk_tok, topk_lp, c);
    ctx->launches += 3;
  }
  tree_select_kernel<<<B, 256, 0, s>>>(t->n_assist, Lo.NC, c, (int32_t*)(ws + Lo.sel), t->tokens, t->parents,
                                       t->depths);
  ctx->launches++;
  return tree_status(cudaGetLastError());
}

__global__ void tree_offsets_kernel(int B, int per, int32_t* row_offsets) {
  for (int b = threadIdx.x; b <= B; b += blockDim.x) row_offsets[b] = b * per;
}

extern "C" mtp_status mtp_synth_target_tree(mtp_ctx* ctx, void* stream, const mtp_tree* t, const uint64_t* seq_hash,
                                            const int32_t* last_tok, uint64_t sticky_thr, void* logits,
                                            int32_t* row_offsets) {
  if (!tree_shape_ok(ctx, t) || !seq_hash || !last_tok || !logits) return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  const int V = ctx->cfg.vocab;
  const dim3 grid((V + 4095) / 4096, t->B * (1 + t->n_assist));
  if (ctx->cfg.dtype == MTP_DTYPE_BF16)
    tree_synth_kernel<uint16_t><<<grid, 256, 0, s>>>(t->n_assist, t->depth, t->tokens, t->parents, seq_hash, last_tok,
                                                      sticky_thr, V, 4096, (uint16_t*)logits);
  else
    tree_synth_kernel<float><<<grid, 256, 0, s>>>(t->n_assist, t->depth, t->tokens, t->parents, seq_hash, last_tok,
                                                   sticky_thr, V, 4096, (float*)logits);
  ctx->launches++;
  if (row_offsets) {
    tree_offsets_kernel<<<1, 128, 0, s>>>(t->B, 1 + t->n_assist, row_offsets);
    ctx->launches++;
  }
  return tree_status(cudaGetLastError());
}

extern "C" mtp_status mtp_verify_tree(mtp_ctx* ctx, void* stream, const mtp_tree* t, const void* target_logits,
                                      int32_t* accepted, int32_t* bonus, int32_t* path_tokens) {
  if (!tree_shape_ok(ctx, t) || !target_logits || !accepted || !bonus || !path_tokens) return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = (char*)t->ws;
  const TreeLayout Lo = tree_layout(ctx, t->B, t->branching, t->depth, t->n_assist, 1);
  unsigned long long* keys = (unsigned long long*)(ws + Lo.keys);
  const int rows = t->B * (1 + t->n_assist);
  cudaError_t e = cudaMemsetAsync(keys, 0, (size_t)rows * 8, s);
  if (e != cudaSuccess) return tree_status(e);
  const int V = ctx->cfg.vocab;
  const dim3 grid((V + 4095) / 4096, rows);
  if (ctx->cfg.dtype == MTP_DTYPE_BF16)
    tree_row_argmax_kernel<uint16_t><<<grid, 256, 0, s>>>((const uint16_t*)target_logits, V, 4096, keys);
  else
    tree_row_argmax_kernel<float><<<grid, 256, 0, s>>>((const float*)target_logits, V, 4096, keys);
  tree_accept_kernel<<<(t->B + 127) / 128, 128, 0, s>>>(t->B, t->n_assist, t->depth, t->tokens, t->parents, keys,
                                                         accepted, bonus, path_tokens,
                                                         (int32_t*)(ws + Lo.path_nodes));
  ctx->launches += 2;
  return tree_status(cudaGetLastError());
}

extern "C" mtp_status mtp_tree_commit(mtp_ctx* ctx, void* stream, const mtp_kv* kv, const mtp_tree* t,
                                      const int32_t* accepted) {
  if (!tree_shape_ok(ctx, t) || !kv || !accepted || !kv->block_table || !kv->seq_len || !kv->pending)
    return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  char* ws = (char*)t->ws;
  const TreeLayout Lo = tree_layout(ctx, t->B, t->branching, t->depth, t->n_assist, kv->max_blocks);
  const int n_kv = ctx->cfg.n_kv_heads, hd = ctx->cfg.head_dim;
  if (ctx->cfg.dtype == MTP_DTYPE_BF16)
    tree_commit_kernel<uint16_t><<<t->B, 256, 0, s>>>(
        t->n_assist, Lo.NC, t->depth, n_kv, hd, kv->max_blocks, kv->num_blocks, accepted,
        (const int32_t*)(ws + Lo.path_nodes), (const int32_t*)(ws + Lo.sel), (const int32_t*)(ws + Lo.cand_exp),
        (const int32_t*)(ws + Lo.vbt), Lo.nV, (uint16_t*)kv->k_pool, (uint16_t*)kv->v_pool, kv->block_table,
        kv->seq_len, kv->pending, ctx->err);
  else
    tree_commit_kernel<float><<<t->B, 256, 0, s>>>(
        t->n_assist, Lo.NC, t->depth, n_kv, hd, kv->max_blocks, kv->num_blocks, accepted,
        (const int32_t*)(ws + Lo.path_nodes), (const int32_t*)(ws + Lo.sel), (const int32_t*)(ws + Lo.cand_exp),
        (const int32_t*)(ws + Lo.vbt), Lo.nV, (float*)kv->k_pool, (float*)kv->v_pool, kv->block_table,
        kv->seq_len, kv->pending, ctx->err);
  ctx->launches++;
  return tree_status(cudaGetLastError());
}

extern "C" mtp_status mtp_tree_loop(mtp_ctx* ctx, void* stream, const mtp_kv* kv, const mtp_loop* lp,
                                    const mtp_tree* t, int iters) {
  if (!tree_shape_ok(ctx, t) || !lp || !kv || iters < 0 || lp->B != t->B) return MTP_ERR_INVALID;
  if (!lp->drafts || !lp->accepted || !lp->bonus || !lp->target_logits) return MTP_ERR_INVALID;
  mtp_status st = MTP_OK;
  for (int it = 0; it < iters && st == MTP_OK; ++it) {
    st = mtp_draft_tree(ctx, stream, lp->hidden, lp->embeds, lp->positions, kv, t);
    if (st == MTP_OK)
      st = mtp_synth_target_tree(ctx, stream, t, lp->seq_hash, lp->last_tok, lp->sticky_thr, lp->target_logits,
                                 nullptr);
    if (st == MTP_OK) st = mtp_verify_tree(ctx, stream, t, lp->target_logits, lp->accepted, lp->bonus, lp->drafts);
    if (st == MTP_OK) st = mtp_tree_commit(ctx, stream, kv, t, lp->accepted);
    if (st == MTP_OK)
      st = mtp_loop_advance(ctx, stream, t->B, t->depth, lp->drafts, lp->accepted, lp->bonus, lp->seq_hash,
                            lp->last_tok, lp->positions, lp->hidden, lp->embeds, lp->out_tokens, lp->out_len,
                            lp->out_cap);
  }
  return st;
}
