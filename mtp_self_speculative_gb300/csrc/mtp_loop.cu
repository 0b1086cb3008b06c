// The speculative loop around the draft-and-verify step, with a
// deterministic synthetic verifier standing in for the target model
// ("How OpenVINO MTP Speculative Decoding Works Internally": the speculative
// result equals the main model's greedy result; "Speculative Decoding",
// "Overview").  The verifier is a pure function of the token prefix built on
// the SplitMix64 finaliser (Steele, Lea & Flood, OOPSLA 2014); its
// definition is in include/mtp.h.
#include "mtp_common.cuh"

namespace mtp {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kSticky = 0xD1B54A32D192ED03ull;
constexpr uint64_t kToken = 0x8CB92BA72F3D8DD7ull;
constexpr uint64_t kHidden = 0x2545F4914F6CDD1Dull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
__device__ __forceinline__ uint64_t fold_tok(uint64_t h, int32_t t) {
  return mix64(h + kGolden * (uint64_t)((int64_t)t + 1));
}
__device__ __forceinline__ int32_t predict_tok(uint64_t h, int32_t last, uint64_t thr, int V) {
  if ((mix64(h ^ kSticky) >> 11) < thr) return last;
  return (int32_t)(mix64(h ^ kToken) % (uint64_t)V);
}
// (mix(h ^ (golden * i1)) >> 40) * 2^-24 - 0.5: a 24-bit fraction, exact in fp32
__device__ __forceinline__ float uhalf(uint64_t h, uint64_t i1) {
  return (float)(uint32_t)(mix64(h ^ (kGolden * i1)) >> 40) * 5.9604644775390625e-08f - 0.5f;
}

template <typename T>
__device__ __forceinline__ void store_val(T* p, float v);
template <>
__device__ __forceinline__ void store_val<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_val<uint16_t>(uint16_t* p, float v) { *p = f32_to_bf16_rne(v); }

// grid (V slices, B * (K + 1)); request b has nd_b = num_drafts[b] (K when
// num_drafts is NULL) drafts and nd_b + 1 rows starting at sum_{c<b}(nd_c + 1);
// blocks past the last row return.  Each thread recomputes its row's prefix
// hash (at most K folds) and writes a strided share of the slice.
template <typename T>
__global__ void synth_target_kernel(int B, int K, const int32_t* num_drafts, const uint64_t* seq_hash,
                                    const int32_t* last_tok, const int32_t* drafts, uint64_t thr, int V, int slice,
                                    T* logits, int32_t* row_offsets) {
  const int r = blockIdx.y;
  int b = 0, row0 = 0;
  for (; b < B; ++b) {
    const int nd = num_drafts ? min(max(num_drafts[b], 0), K) : K;
    if (r < row0 + nd + 1) break;
    row0 += nd + 1;
  }
  if (row_offsets && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    int o = 0;
    for (int c = 0; c < B; ++c) {
      row_offsets[c] = o;
      o += (num_drafts ? min(max(num_drafts[c], 0), K) : K) + 1;
    }
    row_offsets[B] = o;
  }
  if (b >= B) return;
  const int j = r - row0;
  uint64_t h = seq_hash[b];
  int32_t last = last_tok[b];
  for (int i = 0; i < j; ++i) {
    const int32_t t = drafts[(size_t)b * K + i];
    h = fold_tok(h, t);
    last = t;
  }
  const int32_t tgt = predict_tok(h, last, thr, V);
  const int v0 = blockIdx.x * slice, v1 = min(V, v0 + slice);
  T* row = logits + (size_t)r * V;
  for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x)
    store_val<T>(row + v, v == tgt ? 8.0f : uhalf(h, (uint64_t)v + 1));
}

// Probability of the argmax under each draft step's logits: one block per
// (request, step), max then sum of exp(z - max) over the vocabulary with a
// fixed-order block reduction; conf = 1 / sum.
__global__ void draft_conf_kernel(const float* logits, int V, float* conf) {
  __shared__ float red[32];
  const float* z = logits + (size_t)blockIdx.x * V;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float m = -INFINITY;
  for (int v = threadIdx.x; v < V; v += blockDim.x) m = fmaxf(m, z[v]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[w] = m;
  __syncthreads();
  m = red[0];
  for (int i = 1; i < nw; ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  float sum = 0.0f;
  for (int v = threadIdx.x; v < V; v += blockDim.x) sum += expf(z[v] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) red[w] = sum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.0f;
    for (int i = 0; i < nw; ++i) t += red[i];
    conf[blockIdx.x] = 1.0f / t;
  }
}

// Leading run of draft steps whose confidence exceeds tau, per request.
__global__ void leading_run_kernel(int B, int K, const float* conf, float tau, int32_t* num_drafts) {
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
    int n = 0;
    while (n < K && conf[(size_t)b * K + n] > tau) ++n;
    num_drafts[b] = n;
  }
}

template <typename T>
__global__ void loop_advance_kernel(int K, const int32_t* drafts, const int32_t* accepted, const int32_t* bonus,
                                    uint64_t* seq_hash, int32_t* last_tok, int32_t* positions, T* hidden, T* embeds,
                                    const T* table, int H, int V, int32_t* out_tokens, int32_t* out_len, int out_cap,
                                    int* err) {
  __shared__ uint64_t s_h;
  __shared__ int s_ok, s_bonus;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    const int a = accepted[b], beta = bonus[b];
    s_ok = (a >= 0 && a <= K && beta >= 0 && beta < V);
    if (!s_ok) {
      set_error(err, MTP_ERR_DEVICE_ARGS);
    } else {
      uint64_t h = seq_hash[b];
      int n = out_len[b];
      for (int i = 0; i <= a; ++i) {
        const int32_t t = (i < a) ? drafts[(size_t)b * K + i] : beta;
        h = fold_tok(h, t);
        if (n < out_cap) out_tokens[(size_t)b * out_cap + n] = t;
        else set_error(err, MTP_ERR_CAPACITY);
        ++n;
      }
      out_len[b] = n;
      seq_hash[b] = h;
      last_tok[b] = beta;
      positions[b] += a + 1;
      s_h = h;
      s_bonus = beta;
    }
  }
  __syncthreads();
  if (!s_ok) return;
  const uint64_t hh = s_h ^ kHidden;
  const T* src = table + (size_t)s_bonus * H;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    store_val<T>(hidden + (size_t)b * H + i, 2.0f * uhalf(hh, (uint64_t)i + 1));
    embeds[(size_t)b * H + i] = src[i];
  }
}

__global__ void fill_i32_kernel(int32_t* p, int n, int32_t v) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = v;
}

}  // namespace mtp

using namespace mtp;

static mtp_status loop_status(cudaError_t e) {
  if (e == cudaSuccess) return MTP_OK;
  cudaGetLastError();
  return MTP_ERR_CUDA;
}

extern "C" mtp_status mtp_synth_target(mtp_ctx* ctx, void* stream, int B, int K, const int32_t* num_drafts,
                                       const uint64_t* seq_hash, const int32_t* last_tok, const int32_t* drafts,
                                       uint64_t sticky_thr, void* logits, int32_t* row_offsets) {
  if (!ctx || B < 1 || B > ctx->cfg.max_batch || K < 0 || K > ctx->cfg.max_k) return MTP_ERR_INVALID;
  if (!seq_hash || !last_tok || !logits || (K > 0 && !drafts)) return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  const int V = ctx->cfg.vocab;
  const int slices = (V + 4095) / 4096;
  const dim3 grid(slices, B * (K + 1));
  cudaStream_t s = (cudaStream_t)stream;
  if (ctx->cfg.dtype == MTP_DTYPE_BF16)
    synth_target_kernel<uint16_t><<<grid, 256, 0, s>>>(B, K, num_drafts, seq_hash, last_tok, drafts, sticky_thr, V,
                                                        4096, (uint16_t*)logits, row_offsets);
  else
    synth_target_kernel<float><<<grid, 256, 0, s>>>(B, K, num_drafts, seq_hash, last_tok, drafts, sticky_thr, V,
                                                     4096, (float*)logits, row_offsets);
  ctx->launches++;
  return loop_status(cudaGetLastError());
}

extern "C" mtp_status mtp_loop_advance(mtp_ctx* ctx, void* stream, int B, int K, const int32_t* drafts,
                                       const int32_t* accepted, const int32_t* bonus, uint64_t* seq_hash,
                                       int32_t* last_tok, int32_t* positions, void* hidden, void* embeds,
                                       int32_t* out_tokens, int32_t* out_len, int out_cap) {
  if (!ctx || !ctx->has_weights || B < 1 || B > ctx->cfg.max_batch || K < 0 || K > ctx->cfg.max_k)
    return MTP_ERR_INVALID;
  if ((K > 0 && !drafts) || !accepted || !bonus || !seq_hash || !last_tok || !positions || !hidden || !embeds ||
      !out_len || out_cap < 0 || (out_cap > 0 && !out_tokens))
    return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  const int H = ctx->cfg.hidden, V = ctx->cfg.vocab;
  if (ctx->cfg.dtype == MTP_DTYPE_BF16)
    loop_advance_kernel<uint16_t><<<B, 256, 0, s>>>(K, drafts, accepted, bonus, seq_hash, last_tok, positions,
                                                     (uint16_t*)hidden, (uint16_t*)embeds,
                                                     (const uint16_t*)ctx->w.embed, H, V, out_tokens, out_len,
                                                     out_cap, ctx->err);
  else
    loop_advance_kernel<float><<<B, 256, 0, s>>>(K, drafts, accepted, bonus, seq_hash, last_tok, positions,
                                                  (float*)hidden, (float*)embeds, (const float*)ctx->w.embed, H, V,
                                                  out_tokens, out_len, out_cap, ctx->err);
  ctx->launches++;
  return loop_status(cudaGetLastError());
}

extern "C" mtp_status mtp_draft_confidence(mtp_ctx* ctx, void* stream, int B, int K, const float* logits,
                                           float tau, float* conf, int32_t* num_drafts) {
  if (!ctx || B < 1 || B > ctx->cfg.max_batch || K < 1 || K > ctx->cfg.max_k || !logits || !conf)
    return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  draft_conf_kernel<<<B * K, 512, 0, s>>>(logits, ctx->cfg.vocab, conf);
  ctx->launches++;
  if (num_drafts) {
    leading_run_kernel<<<(B + 127) / 128, 128, 0, s>>>(B, K, conf, tau, num_drafts);
    ctx->launches++;
  }
  return loop_status(cudaGetLastError());
}

extern "C" int mtp_adapt_k(int K, int accepted, int drafted, int k_min, int k_max) {
  if (drafted > 0 && accepted == drafted) return K + 2 < k_max ? K + 2 : k_max;
  return K - 1 > k_min ? K - 1 : k_min;
}

extern "C" mtp_status mtp_spec_loop(mtp_ctx* ctx, void* stream, const mtp_kv* kv, const mtp_loop* lp, int iters) {
  if (!ctx || !ctx->has_weights || !lp || iters < 0) return MTP_ERR_INVALID;
  const int B = lp->B, K = lp->K;
  if (B < 1 || B > ctx->cfg.max_batch || K < 0 || K > ctx->cfg.max_k) return MTP_ERR_INVALID;
  if (!lp->drafts || !lp->accepted || !lp->bonus || !lp->num_drafts || !lp->row_offsets || !lp->target_logits)
    return MTP_ERR_INVALID;
  if (K > 0 && !kv) return MTP_ERR_INVALID;
  const bool conf_stop = lp->conf_threshold > 0.0f && K > 0;
  if (conf_stop && (!lp->draft_logits || !lp->conf)) return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  fill_i32_kernel<<<1, 128, 0, s>>>(lp->num_drafts, B, K);
  ctx->launches++;
  mtp_status st = loop_status(cudaGetLastError());
  const int stride = K > 0 ? K : 1;
  for (int it = 0; it < iters && st == MTP_OK; ++it) {
    if (K > 0)
      st = mtp_draft(ctx, stream, B, lp->hidden, lp->embeds, lp->positions, kv, K, nullptr, lp->drafts,
                     conf_stop ? lp->draft_logits : nullptr, nullptr);
    if (st == MTP_OK && conf_stop)
      st = mtp_draft_confidence(ctx, stream, B, K, lp->draft_logits, lp->conf_threshold, lp->conf, lp->num_drafts);
    if (st == MTP_OK)
      st = mtp_synth_target(ctx, stream, B, K, lp->num_drafts, lp->seq_hash, lp->last_tok, lp->drafts,
                            lp->sticky_thr, lp->target_logits, lp->row_offsets);
    if (st == MTP_OK)
      st = mtp_verify(ctx, stream, B, lp->target_logits, B * (K + 1), lp->row_offsets, lp->drafts, stride,
                      lp->num_drafts, lp->accepted, lp->bonus);
    if (st == MTP_OK && K > 0) st = mtp_kv_commit_accepted(ctx, stream, B, kv, lp->accepted, 1);
    if (st == MTP_OK)
      st = mtp_loop_advance(ctx, stream, B, K, lp->drafts, lp->accepted, lp->bonus, lp->seq_hash, lp->last_tok,
                            lp->positions, lp->hidden, lp->embeds, lp->out_tokens, lp->out_len, lp->out_cap);
  }
  return st;
}
