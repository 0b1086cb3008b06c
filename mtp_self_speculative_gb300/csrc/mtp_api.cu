// Host side of the C ABI: argument validation, workspace, rotary table,
// launch sequencing and kernel timing.  Every step of the method runs in the
// kernels of the other translation units; this file only checks, allocates
// and launches.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "mtp_common.cuh"

namespace mtp {

void prof_before(mtp_ctx* ctx, int kernel, cudaStream_t s) {
  if (ctx->prof_kernel == kernel && ctx->prof_n < ctx->prof_cap) cudaEventRecord(ctx->prof_ev[2 * ctx->prof_n], s);
}
void prof_after(mtp_ctx* ctx, int kernel, cudaStream_t s) {
  if (ctx->prof_kernel == kernel && ctx->prof_n < ctx->prof_cap) {
    cudaEventRecord(ctx->prof_ev[2 * ctx->prof_n + 1], s);
    ctx->prof_n++;
  }
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

cudaError_t ensure_smem(const void* func, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> done;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = done[std::make_pair(func, dev)];
  if (bytes <= have) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

}  // namespace mtp

using namespace mtp;

// One draft step k of K for B requests on the per-step kernels (quantized,
// tensor-core or streamed, as mtp_draft chooses).
cudaError_t mtp::draft_one_step(mtp_ctx* ctx, cudaStream_t s, int B, int k, int K, const void* hidden,
                                const void* embeds, const int32_t* positions, const mtp_kv* kv,
                                const int32_t* chain_ids, int32_t* draft_ids, float* logits, float* hidden_out) {
  if (ctx->quantized)
    return launch_draft_step_q(ctx, s, B, k, K, hidden, embeds, positions, kv, chain_ids, draft_ids, logits,
                               hidden_out);
  if (tc_supported(ctx, B))
    return launch_draft_step_tc(ctx, s, B, k, K, hidden, embeds, positions, kv, chain_ids, draft_ids, logits,
                                hidden_out);
  return launch_draft_step(ctx, s, B, k, K, hidden, embeds, positions, kv, chain_ids, draft_ids, logits,
                           hidden_out);
}


extern "C" {

const char* mtp_status_str(mtp_status s) {
  switch (s) {
    case MTP_OK: return "ok";
    case MTP_ERR_INVALID: return "invalid argument";
    case MTP_ERR_CUDA: return "CUDA error";
    case MTP_ERR_OOM: return "out of device memory";
    case MTP_ERR_CAPACITY: return "KV capacity or position range exceeded";
    case MTP_ERR_TIMEOUT: return "bounded device wait ran out";
    case MTP_ERR_DEVICE_ARGS: return "inconsistent device-side arguments";
    case MTP_ERR_BOUNDS: return "store outside its output (bounds-checked build)";
  }
  return "unknown status";
}

static bool config_ok(const mtp_config* c, bool with_weights) {
  if (!c) return false;
  if (c->dtype != MTP_DTYPE_F32 && c->dtype != MTP_DTYPE_BF16) return false;
  if (c->n_kv_heads <= 0 || c->n_q_heads <= 0 || c->n_q_heads % c->n_kv_heads) return false;
  const int G = c->n_q_heads / c->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->vocab <= 0 || c->max_batch <= 0 || c->max_k < 1 || c->max_k > 100) return false;
  if (c->block_size != 16) return false;
  if (with_weights) {
    if (c->hidden <= 0 || c->hidden % 8 || c->ffn <= 0 || c->ffn % 8) return false;
    if (!(c->eps > 0.0f) || !(c->rope_theta > 0.0f) || c->max_pos <= 0) return false;
  }
  if (c->weight_format != MTP_WEIGHTS_DENSE && c->weight_format != MTP_WEIGHTS_INT4_G64) return false;
  if (c->weight_format == MTP_WEIGHTS_INT4_G64) {
    // quantized head: bf16 source weights, the small-batch kernels only, rows
    // whose per-group metadata is a whole number of 16-byte bulk copies
    if (!with_weights || c->dtype != MTP_DTYPE_BF16 || c->max_batch > 4) return false;
    if (c->hidden % 1024 || c->ffn % 1024 || (c->n_q_heads * c->head_dim) % 1024) return false;
  }
  return true;
}


mtp_status mtp_init(const mtp_config* cfg, const mtp_weights* weights, int device, mtp_ctx** out) {
  if (!out) return MTP_ERR_INVALID;
  *out = nullptr;
  const bool with_w = weights != nullptr;
  if (!config_ok(cfg, with_w)) return MTP_ERR_INVALID;
  if (with_w) {
    const void* req[] = {weights->w_norm_h, weights->w_norm_e, weights->w_eh, weights->w_norm_in, weights->w_q,
                         weights->w_k, weights->w_v, weights->w_o, weights->w_norm_post, weights->w_gate,
                         weights->w_up, weights->w_down, weights->w_norm_f, weights->embed};
    for (const void* p : req)
      if (!p) return MTP_ERR_INVALID;
  }
  if (cudaSetDevice(device) != cudaSuccess) return MTP_ERR_CUDA;
  mtp_ctx* ctx = (mtp_ctx*)calloc(1, sizeof(mtp_ctx));
  if (!ctx) return MTP_ERR_OOM;
  ctx->cfg = *cfg;
  ctx->device = device;
  ctx->has_weights = with_w;
  if (with_w) {
    ctx->w = *weights;
    if (!ctx->w.lm_head) ctx->w.lm_head = ctx->w.embed;
  }
  ctx->prof_kernel = -1;
  // Which small-batch projection kinds use the bulk-copy streamed kernel
  // (bit = kind: eh, qkv, o, gate_up, down, lm_head); MTP_GEMV_STREAM
  // overrides the default for tuning.
  ctx->gemv_stream_mask = 0x3F;
  if (const char* env = getenv("MTP_GEMV_STREAM")) ctx->gemv_stream_mask = (int)strtol(env, nullptr, 0);
  // LM head of 2..4 requests on the tensor cores; MTP_LM_ROWS=0 keeps the
  // streamed GEMV for it (comparison).
  ctx->lm_rows = 1;
  if (const char* env = getenv("MTP_LM_ROWS")) ctx->lm_rows = (int)strtol(env, nullptr, 0) != 0;
  // streamed LM head: ranges weighted by each SM's measured streaming rate;
  // MTP_LM_BALANCE=0 keeps equal ranges (comparison)
  ctx->lm_balance = 1;
  ctx->lm_seq = 0;
  if (const char* env = getenv("MTP_LM_BALANCE")) ctx->lm_balance = (int)strtol(env, nullptr, 0) != 0;
  // one request: every draft step but the last leaves its argmax to the next
  // eh_proj; MTP_LM_DEFER=0 keeps the LM head's last-CTA argmax (comparison)
  ctx->lm_defer = 1;
  ctx->lm_defer_pending = 0;
  ctx->lm_defer_grid = 0;
  ctx->lm_defer_tick = nullptr;
  if (const char* env = getenv("MTP_LM_DEFER")) ctx->lm_defer = (int)strtol(env, nullptr, 0) != 0;
  // the short projections of 2..4 requests likewise; MTP_ROWS_PROJ=0 keeps
  // the streamed GEMV for them (comparison)
  ctx->rows_proj = 1;
  if (const char* env = getenv("MTP_ROWS_PROJ")) ctx->rows_proj = (int)strtol(env, nullptr, 0) != 0;
  ctx->rows_max_kc = 4096;
  ctx->rows_min_stages = 3;
  if (const char* env = getenv("MTP_ROWS_KC")) ctx->rows_max_kc = (int)strtol(env, nullptr, 0);
  if (const char* env = getenv("MTP_ROWS_MIN_STAGES")) ctx->rows_min_stages = (int)strtol(env, nullptr, 0);
  if (ctx->rows_max_kc < 256 || ctx->rows_max_kc > 4096 || (ctx->rows_max_kc & (ctx->rows_max_kc - 1)))
    ctx->rows_max_kc = 4096;
  if (ctx->rows_min_stages < 2 || ctx->rows_min_stages > 8) ctx->rows_min_stages = 3;
  // Shared-memory budget of the streamed kernel per kind, in KB;
  // MTP_GEMV_BUDGET ("eh,qkv,o,gu,down,lm") overrides it for tuning.
  for (int i = 0; i < 6; ++i) ctx->gemv_budget_kb[i] = 220;
  if (const char* env = getenv("MTP_GEMV_BUDGET")) {
    const char* q = env;
    for (int i = 0; i < 6 && *q; ++i) {
      char* end = nullptr;
      const long v = strtol(q, &end, 10);
      if (end == q) break;
      if (v >= 32 && v <= 220) ctx->gemv_budget_kb[i] = (int)v;
      q = (*end == ',') ? end + 1 : end;
    }
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
    free(ctx);
    return MTP_ERR_CUDA;
  }
  ctx->num_sms = sms;
  const mtp_config& c = ctx->cfg;
  const size_t maxB = c.max_batch;
  ctx->q_dim = c.n_q_heads * c.head_dim;
  ctx->kv_dim = c.n_kv_heads * c.head_dim;
  ctx->attn_target_ctas = 16 * sms;  // about eight waves of two CTAs per SM: ragged batches stay balanced
  if (const char* env = getenv("MTP_ATTN_WAVES")) {
    const long v = strtol(env, nullptr, 0);
    if (v >= 1 && v <= 256) ctx->attn_target_ctas = (int)v * sms;
  }
  ctx->attn_max_splits = 64;
  ctx->attn_force_bps = 0;
  // MTP_ATTN_CLUSTER=0 keeps the split combine through HBM partials (comparison)
  ctx->attn_cluster = 1;
  ctx->attn_cl_key = -1;
  ctx->attn_cl_fit = 0;
  ctx->attn_cl_bps = 0;
  if (const char* env = getenv("MTP_ATTN_CLUSTER")) ctx->attn_cluster = (int)strtol(env, nullptr, 0) != 0;
  if (const char* env = getenv("MTP_ATTN_BPS")) {
    const long v = strtol(env, nullptr, 0);
    if (v >= 1 && v <= 4096) ctx->attn_force_bps = (int)v;
  }
  const size_t H = with_w ? c.hidden : 0, F = with_w ? c.ffn : 0;
  const size_t qd = with_w ? ctx->q_dim : 0;
  const size_t part_rows = with_w ? (size_t)(ctx->attn_target_ctas / c.n_kv_heads + maxB + 1) * c.n_q_heads : 0;
  const size_t rope_n = with_w ? (size_t)c.max_pos * (c.head_dim / 2) : 0;

  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t o_hid = take(maxB * H * 4), o_x = take(maxB * H * 4), o_q = take(maxB * qd * 4);
  const size_t o_attn = take(maxB * qd * 4), o_h1 = take(maxB * H * 4), o_act = take(maxB * F * 4);
  const size_t o_part = take(part_rows * (c.head_dim + 4) * 4);
  const size_t o_acnt = take(maxB * c.n_kv_heads * 4);
  const size_t o_lmk = take(maxB * 8), o_lmc = take(4);
  const size_t o_lmt = take(64 * 8), o_lmr = take((size_t)ctx->num_sms * 4);
  const size_t o_ctk = take((size_t)ctx->num_sms * 8);
  const size_t o_vk = take(maxB * (c.max_k + 1) * 8), o_vc = take(256);
  const size_t o_err = take(4);
  const size_t o_bad = take(maxB * 4);
  const size_t o_rope = take(rope_n * sizeof(float2));
  ctx->ws_bytes = off;
  if (cudaMalloc(&ctx->ws, off) != cudaSuccess) {
    cudaGetLastError();
    free(ctx);
    return MTP_ERR_OOM;
  }
  char* base = (char*)ctx->ws;
  ctx->hid = (float*)(base + o_hid);
  ctx->x = (float*)(base + o_x);
  ctx->q = (float*)(base + o_q);
  ctx->attn = (float*)(base + o_attn);
  ctx->h1 = (float*)(base + o_h1);
  ctx->act = (float*)(base + o_act);
  ctx->attn_part = (float*)(base + o_part);
  ctx->attn_cnt = (int*)(base + o_acnt);
  ctx->lm_keys = (unsigned long long*)(base + o_lmk);
  ctx->lm_cnt = (int*)(base + o_lmc);
  ctx->lm_tick = (unsigned long long*)(base + o_lmt);
  ctx->lm_rate = (float*)(base + o_lmr);
  ctx->cta_keys = (unsigned long long*)(base + o_ctk);
  ctx->ver_keys = (unsigned long long*)(base + o_vk);
  ctx->ver_cnt = (int*)(base + o_vc);
  ctx->err = (int*)(base + o_err);
  ctx->req_bad = (int*)(base + o_bad);
  ctx->rope = (float2*)(base + o_rope);
  cudaError_t e = cudaMemset(ctx->ws, 0, off);
  if (e == cudaSuccess && rope_n) {
    // Rotary table: angle = pos * theta^(-2i/d), evaluated in double.
    std::vector<float2> tab(rope_n);
    const int half = c.head_dim / 2;
    for (int p = 0; p < c.max_pos; ++p)
      for (int i = 0; i < half; ++i) {
        const double ang = (double)p * pow((double)c.rope_theta, -2.0 * i / c.head_dim);
        tab[(size_t)p * half + i] = make_float2((float)cos(ang), (float)sin(ang));
      }
    e = cudaMemcpy(ctx->rope, tab.data(), rope_n * sizeof(float2), cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) {
    cudaFree(ctx->ws);
    free(ctx);
    return MTP_ERR_CUDA;
  }
  // tensor-core path workspace
  ctx->tc_min_batch = c.tc_min_batch > 0 ? c.tc_min_batch : 5;
  if (with_w && c.dtype == MTP_DTYPE_BF16 && c.head_dim == 128 && c.hidden % 128 == 0 && c.ffn % 64 == 0 &&
      ctx->q_dim % 64 == 0 && c.max_batch >= ctx->tc_min_batch && c.weight_format == MTP_WEIGHTS_DENSE) {
    const size_t mb = (size_t)c.max_batch;
    size_t o2 = 0;
    auto take2 = [&](size_t bytes) {
      const size_t o = o2;
      o2 = align_up(o2 + bytes, 1024);
      return o;
    };
    const size_t t_eh = take2(mb * 2 * c.hidden * 2), t_xn = take2(mb * c.hidden * 2);
    const size_t t_at = take2(mb * ctx->q_dim * 2), t_act = take2(mb * c.ffn * 2);
    const size_t t_ssq = take2((size_t)(c.hidden / 128) * mb * 4);
    if (cudaMalloc(&ctx->tc_ws, o2) != cudaSuccess || cudaMemset(ctx->tc_ws, 0, o2) != cudaSuccess) {
      cudaGetLastError();
      if (ctx->tc_ws) cudaFree(ctx->tc_ws);
      cudaFree(ctx->ws);
      free(ctx);
      return MTP_ERR_OOM;
    }
    char* tb = (char*)ctx->tc_ws;
    ctx->tc_xin_eh = (uint16_t*)(tb + t_eh);
    ctx->tc_xn = (uint16_t*)(tb + t_xn);
    ctx->tc_attn = (uint16_t*)(tb + t_at);
    ctx->tc_act = (uint16_t*)(tb + t_act);
    ctx->tc_ssq = (float*)(tb + t_ssq);
  }
  // persistent draft kernel workspace: attention records, counters, argmax
  // keys and the grid-barrier words
  ctx->p_max_batch = c.persistent_max_batch > 0 ? c.persistent_max_batch : 0;
  if (ctx->p_max_batch > 4) ctx->p_max_batch = 4;
  if (ctx->p_max_batch > c.max_batch) ctx->p_max_batch = c.max_batch;
  if (!(with_w && c.dtype == MTP_DTYPE_BF16 && c.head_dim == 128) || c.weight_format != MTP_WEIGHTS_DENSE)
    ctx->p_max_batch = 0;
  if (ctx->p_max_batch > 0) {
    const size_t pb = (size_t)ctx->p_max_batch;
    size_t o3 = 0;
    auto take3 = [&](size_t bytes) {
      const size_t o = o3;
      o3 = align_up(o3 + bytes, 256);
      return o;
    };
    const size_t p_rec = take3(pb * c.n_q_heads * (size_t)sms * 132 * 4);
    const size_t p_cnt = take3(pb * c.n_kv_heads * 4);
    const size_t p_keys = take3((size_t)c.max_k * pb * 8);
    const size_t p_bar = take3(384);
    if (cudaMalloc(&ctx->p_ws, o3) != cudaSuccess || cudaMemset(ctx->p_ws, 0, o3) != cudaSuccess) {
      cudaGetLastError();
      if (ctx->p_ws) cudaFree(ctx->p_ws);
  if (ctx->qw_buf) cudaFree(ctx->qw_buf);
      if (ctx->tc_ws) cudaFree(ctx->tc_ws);
      cudaFree(ctx->ws);
      free(ctx);
      return MTP_ERR_OOM;
    }
    char* pbase = (char*)ctx->p_ws;
    ctx->p_rec = (float*)(pbase + p_rec);
    ctx->p_seg_cnt = (int*)(pbase + p_cnt);
    ctx->p_keys = (unsigned long long*)(pbase + p_keys);
    ctx->p_gbar = (unsigned long long*)(pbase + p_bar);
  }
  if (c.weight_format == MTP_WEIGHTS_INT4_G64) {
    const mtp_status st = quantize_head(ctx);
    if (st != MTP_OK) {
      mtp_destroy(ctx);
      return st;
    }
  }
  *out = ctx;
  return MTP_OK;
}

void mtp_destroy(mtp_ctx* ctx) {
  if (!ctx) return;
  cudaSetDevice(ctx->device);
  if (ctx->prof_ev) {
    for (int i = 0; i < 2 * ctx->prof_cap; ++i) cudaEventDestroy(ctx->prof_ev[i]);
    free(ctx->prof_ev);
  }
  cudaFree(ctx->ws);
  if (ctx->tc_ws) cudaFree(ctx->tc_ws);
  if (ctx->p_ws) cudaFree(ctx->p_ws);
  if (ctx->qw_buf) cudaFree(ctx->qw_buf);
  free(ctx->tc_plan_cache);
  free(ctx->attn_map_cache);
  free(ctx);
}

static bool kv_ok(const mtp_kv* kv) {
  return kv && kv->k_pool && kv->v_pool && kv->block_table && kv->seq_len && kv->pending && kv->num_blocks > 0 &&
         kv->max_blocks > 0;
}

static mtp_status after_launch(cudaError_t e) {
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MTP_ERR_CUDA;
  }
  return MTP_OK;
}

mtp_status mtp_draft(mtp_ctx* ctx, void* stream, int B, const void* hidden, const void* embeds,
                     const int32_t* positions, const mtp_kv* kv, int K, const int32_t* chain_ids,
                     int32_t* draft_ids, float* logits, float* hidden_out) {
  if (!ctx || !ctx->has_weights) return MTP_ERR_INVALID;
  if (B < 1 || B > ctx->cfg.max_batch || K < 1 || K > ctx->cfg.max_k) return MTP_ERR_INVALID;
  if (!hidden || !embeds || !positions || !draft_ids || !kv_ok(kv)) return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  if (ctx->quantized) {
    for (int k = 1; k <= K; ++k) {
      cudaError_t e = launch_draft_step_q(ctx, s, B, k, K, hidden, embeds, positions, kv, chain_ids, draft_ids,
                                          logits, hidden_out);
      if (e != cudaSuccess) return after_launch(e);
    }
    return after_launch(cudaGetLastError());
  }
  if (persistent_supported(ctx, B))
    return after_launch(launch_draft_persistent(ctx, s, B, K, hidden, embeds, positions, kv, chain_ids, draft_ids,
                                                logits, hidden_out));
  for (int k = 1; k <= K; ++k) {
    cudaError_t e = draft_one_step(ctx, s, B, k, K, hidden, embeds, positions, kv, chain_ids, draft_ids, logits,
                                   hidden_out);
    if (e != cudaSuccess) return after_launch(e);
  }
  return after_launch(cudaGetLastError());
}

mtp_status mtp_verify(mtp_ctx* ctx, void* stream, int B, const void* target_logits, int num_rows,
                      const int32_t* row_offsets, const int32_t* drafts, int drafts_stride,
                      const int32_t* num_drafts, int32_t* accepted, int32_t* bonus) {
  if (!ctx || B < 1 || B > ctx->cfg.max_batch || num_rows < 1 ||
      num_rows > ctx->cfg.max_batch * (ctx->cfg.max_k + 1))
    return MTP_ERR_INVALID;
  if (!target_logits || !row_offsets || !drafts || !num_drafts || !accepted || !bonus || drafts_stride < 1)
    return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  return after_launch(launch_verify(ctx, (cudaStream_t)stream, B, target_logits, num_rows, row_offsets, drafts,
                                    drafts_stride, num_drafts, accepted, bonus));
}

static mtp_status kv_edit(mtp_ctx* ctx, void* stream, int B, const mtp_kv* kv, int mode, const int32_t* arg,
                          int extra) {
  if (!ctx || B < 1 || B > ctx->cfg.max_batch || !kv_ok(kv)) return MTP_ERR_INVALID;
  if (mode != KV_ROLLBACK && !arg) return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  return after_launch(launch_kv_edit(ctx, (cudaStream_t)stream, B, kv, mode, arg, extra));
}

mtp_status mtp_kv_commit(mtp_ctx* ctx, void* stream, int B, const mtp_kv* kv, const int32_t* n_keep) {
  return kv_edit(ctx, stream, B, kv, KV_COMMIT, n_keep, 0);
}

mtp_status mtp_kv_commit_accepted(mtp_ctx* ctx, void* stream, int B, const mtp_kv* kv, const int32_t* accepted,
                                  int extra) {
  if (extra < 0 || extra > 1) return MTP_ERR_INVALID;
  return kv_edit(ctx, stream, B, kv, KV_COMMIT_ACCEPTED, accepted, extra);
}

mtp_status mtp_kv_rollback(mtp_ctx* ctx, void* stream, int B, const mtp_kv* kv) {
  return kv_edit(ctx, stream, B, kv, KV_ROLLBACK, nullptr, 0);
}

mtp_status mtp_kv_truncate(mtp_ctx* ctx, void* stream, int B, const mtp_kv* kv, const int32_t* new_len) {
  return kv_edit(ctx, stream, B, kv, KV_TRUNCATE, new_len, 0);
}

mtp_status mtp_selftest_wait_timeout(mtp_ctx* ctx, void* stream, int which) {
  if (!ctx || (which != 0 && which != 1)) return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  return after_launch(launch_selftest_wait(ctx, (cudaStream_t)stream, which));
}

mtp_status mtp_get_device_error(mtp_ctx* ctx) {
  if (!ctx) return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return MTP_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, ctx->err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MTP_ERR_CUDA;
  if (word && cudaMemset(ctx->err, 0, 4) != cudaSuccess) return MTP_ERR_CUDA;
  // a persistent draft call that gave up leaves its grid-barrier words
  // (arrivals, abort flag) inconsistent: start them afresh
  if (word == MTP_ERR_TIMEOUT && ctx->p_gbar && cudaMemset(ctx->p_gbar, 0, 384) != cudaSuccess) return MTP_ERR_CUDA;
  // an LM head that gave up may leave its arrival and claim counters and
  // argmax keys part-way: start them afresh as well
  if (word == MTP_ERR_TIMEOUT && ctx->lm_cnt &&
      (cudaMemset(ctx->lm_cnt, 0, 4) != cudaSuccess || cudaMemset(ctx->lm_tick, 0, 64 * 8) != cudaSuccess ||
       cudaMemset(ctx->lm_keys, 0, (size_t)ctx->cfg.max_batch * 8) != cudaSuccess))
    return MTP_ERR_CUDA;
  return (mtp_status)word;
}

mtp_status mtp_stream_copy(void* stream, void* dst, const void* src, size_t bytes) {
  if (!dst || !src || bytes == 0 || bytes % 16 || ((uintptr_t)dst & 15) || ((uintptr_t)src & 15))
    return MTP_ERR_INVALID;
  const char* d = (const char*)dst;
  const char* s = (const char*)src;
  if (d < s + bytes && s < d + bytes) return MTP_ERR_INVALID;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MTP_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MTP_ERR_CUDA;
  return after_launch(launch_stream_copy((cudaStream_t)stream, dst, src, bytes, sms));
}

namespace mtp {
// One store one element past a 4-element extent, through the bounds check.
// The destination has room beyond those 4 elements (workspace scratch), so
// even a build whose check failed to skip would write inside an allocation.
__global__ void selftest_bounds_kernel(int* err, float* scratch) { MTP_STORE(err, scratch, 4, 4, 1.0f); }
}  // namespace mtp

mtp_status mtp_selftest_bounds(mtp_ctx* ctx, void* stream) {
  if (!ctx) return MTP_ERR_INVALID;
#ifdef MTP_CHECKED
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  selftest_bounds_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(ctx->err, ctx->hid);
  return after_launch(cudaGetLastError());
#else
  (void)stream;
  return MTP_ERR_INVALID;
#endif
}

mtp_status mtp_stream_read(void* stream, const void* src, size_t bytes, int* err_word) {
  if (!src || bytes == 0 || bytes % 16 || ((uintptr_t)src & 15)) return MTP_ERR_INVALID;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MTP_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MTP_ERR_CUDA;
  return after_launch(launch_stream_read((cudaStream_t)stream, src, bytes, sms, err_word));
}

mtp_status mtp_profile_begin(mtp_ctx* ctx, int kernel, int capacity) {
  if (!ctx || kernel < 0 || kernel >= MTP_KERNEL_COUNT || capacity < 1 || capacity > (1 << 20))
    return MTP_ERR_INVALID;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  if (ctx->prof_ev) {
    for (int i = 0; i < 2 * ctx->prof_cap; ++i) cudaEventDestroy(ctx->prof_ev[i]);
    free(ctx->prof_ev);
    ctx->prof_ev = nullptr;
  }
  ctx->prof_ev = (cudaEvent_t*)calloc(2 * (size_t)capacity, sizeof(cudaEvent_t));
  if (!ctx->prof_ev) return MTP_ERR_OOM;
  for (int i = 0; i < 2 * capacity; ++i)
    if (cudaEventCreate(&ctx->prof_ev[i]) != cudaSuccess) return MTP_ERR_CUDA;
  ctx->prof_cap = capacity;
  ctx->prof_n = 0;
  ctx->prof_kernel = kernel;
  return MTP_OK;
}

mtp_status mtp_profile_end(mtp_ctx* ctx, float* ms_out, int max_out, int* n_out) {
  if (!ctx || !n_out || (max_out > 0 && !ms_out)) return MTP_ERR_INVALID;
  ctx->prof_kernel = -1;
  const int n = ctx->prof_n;
  *n_out = 0;
  if (cudaSetDevice(ctx->device) != cudaSuccess) return MTP_ERR_CUDA;
  for (int i = 0; i < n && i < max_out; ++i) {
    if (cudaEventSynchronize(ctx->prof_ev[2 * i + 1]) != cudaSuccess) return MTP_ERR_CUDA;
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, ctx->prof_ev[2 * i], ctx->prof_ev[2 * i + 1]) != cudaSuccess) return MTP_ERR_CUDA;
    ms_out[i] = ms;
    *n_out = i + 1;
  }
  return MTP_OK;
}

int64_t mtp_launch_count(const mtp_ctx* ctx) { return ctx ? ctx->launches : 0; }

int64_t mtp_path_count(const mtp_ctx* ctx, int path) {
  if (!ctx || path < 0 || path >= MTP_PATH_COUNT) return 0;
  return ctx->path_counts[path];
}

}  // extern "C"
