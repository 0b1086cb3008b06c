/*
 * mtp.h -- C ABI of the MTP self-speculative draft-and-verify step (one GPU,
 * sm_103a).
 *
 * The operations come from these pages (title, section):
 *   "MTP (Multi-Token Prediction)" (speculators user guide), "Architecture":
 *     the MTP head normalises the verifier's hidden state and the token
 *     embedding separately, concatenates them, projects 2H -> H, runs one
 *     standard decoder layer (attention + MLP) and applies the shared LM head;
 *     its output hidden state feeds the next step recursively.
 *   "How OpenVINO MTP Speculative Decoding Works Internally", "The MTP
 *     inputs" (hidden_states, inputs_embeds, attention metadata, position_ids,
 *     the MTP KV cache), "Shared embeddings reduce duplication" (the head
 *     reads the target's embedding table), "Stateful execution" (the
 *     one-layer cache is updated in place on every invocation).
 *   "Speculative Decoding" (OpenVINO GenAI), "Overview": greedy
 *     verification keeps the drafts the target would have produced and
 *     replaces the first divergent one by the target's token;
 *     "Tree Drafting" step 4 and "Prefix Caching with Speculative Decoding":
 *     caches advance to the accepted prefix or return to a common prefix.
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers unless stated, row-major,
 *     owned by the caller.  The library borrows them for the duration of the
 *     asynchronous work it enqueues; it never frees them.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; outputs are valid once the
 *     stream has been synchronised.
 *   - A host-detectable argument error returns MTP_ERR_INVALID and enqueues
 *     nothing.  Errors found on the device (inconsistent device-side lengths,
 *     KV capacity, a bounded wait that ran out) set a device error word, leave
 *     the affected outputs undefined, and are reported by
 *     mtp_get_device_error().
 *   - dtype MTP_DTYPE_BF16: weights, KV pools, hidden/embeds and verify
 *     logits are bf16 (uint16 bit patterns); MTP_DTYPE_F32: all float32.
 *     Draft logits and hidden_out are always float32.
 */
#ifndef MTP_H_
#define MTP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MTP_OK = 0,
  MTP_ERR_INVALID = 1,      /* bad host argument; nothing enqueued            */
  MTP_ERR_CUDA = 2,         /* a CUDA runtime call or launch failed           */
  MTP_ERR_OOM = 3,          /* workspace allocation failed                    */
  MTP_ERR_CAPACITY = 4,     /* device: KV slot outside block table / pool     */
  MTP_ERR_TIMEOUT = 5,      /* device: a bounded wait ran out                 */
  MTP_ERR_DEVICE_ARGS = 6,  /* device: inconsistent lengths/offsets/pending   */
  MTP_ERR_BOUNDS = 7        /* device, bounds-checked build only: a store fell
                               outside its output's extent and was skipped    */
} mtp_status;

typedef enum { MTP_DTYPE_F32 = 0, MTP_DTYPE_BF16 = 1 } mtp_dtype;

/* Storage of the head's weights inside the context.  DENSE: the caller's
 * tensors are read in place (dtype).  INT4_G64: the format of the pages'
 * quantized MTP component ("Why MTP gets its own quantization
 * configuration": 4-bit asymmetric, group size 64, INT8 symmetric backup):
 * mtp_init quantizes the caller's bf16 weights once into context-owned
 * buffers -- projections to INT4 with groups of 64 input columns
 * (mtp_quantize_int4_g64), the shared embedding / LM head to INT8 per row
 * (mtp_quantize_int8_rows) -- and every draft reads only those.  Requires
 * bf16, max_batch <= 4 and hidden, ffn, n_q_heads*head_dim multiples of 1024. */
typedef enum { MTP_WEIGHTS_DENSE = 0, MTP_WEIGHTS_INT4_G64 = 1 } mtp_weight_format;

/* Shape of the MTP head and the limits of one context. */
typedef struct {
  int hidden;            /* H; multiple of 8                                  */
  int n_q_heads;         /* query heads; multiple of n_kv_heads               */
  int n_kv_heads;        /* key/value heads (grouped-query attention)         */
  int head_dim;          /* 64 or 128                                         */
  int ffn;               /* SwiGLU inner size F; multiple of 8                */
  int vocab;             /* V (rows of the embedding table / LM head)         */
  float eps;             /* RMSNorm epsilon                                   */
  float rope_theta;      /* rotary base                                       */
  int dtype;             /* mtp_dtype                                         */
  int max_batch;         /* largest B of any call                             */
  int max_k;             /* largest draft count K of any call (1..100)        */
  int block_size;        /* KV tokens per paged block; must be 16             */
  int max_pos;           /* positions + K - 1 must stay below this            */
  int tc_min_batch;      /* batches of at least this many requests use the
                            tensor-core (tcgen05) path when the shape allows
                            it (bf16, head_dim 128, H % 128 == 0, F and
                            n_q*head_dim % 64 == 0, B <= 256); 0 = 5       */
  int persistent_max_batch; /* batches of 1 .. this many requests run all K
                            draft steps in one persistent cooperative kernel
                            (bf16, head_dim 128) instead of the per-step
                            streamed kernels; 0 or negative = never (the
                            default); capped at 4 and at max_batch          */
  int weight_format;     /* mtp_weight_format; 0 = dense                     */
} mtp_config;

/* Borrowed head weights (device pointers, layouts [out, in] row-major).
 * Norm weights are [H].  w_eh is [H, 2H]: columns [0, H) act on the
 * normalised hidden state, [H, 2H) on the normalised embedding.  w_q is
 * [n_q*d, H], w_k and w_v [n_kv*d, H], w_o [H, n_q*d], w_gate and w_up [F, H],
 * w_down [H, F].  embed is the shared [V, H] token-embedding table; lm_head is
 * [V, H] and may equal embed (tied). */
typedef struct {
  const void *w_norm_h, *w_norm_e, *w_eh;
  const void *w_norm_in, *w_q, *w_k, *w_v, *w_o;
  const void *w_norm_post, *w_gate, *w_up, *w_down;
  const void *w_norm_f, *embed, *lm_head;
} mtp_weights;

/* The single-layer MTP KV cache, paged (device pointers, borrowed).
 *   k_pool, v_pool: [num_blocks, n_kv, block_size, head_dim] in the dtype.
 *   block_table:    [B, max_blocks] int32; slot s of request b lives in block
 *                   block_table[b*max_blocks + s/block_size] at row s%block_size.
 *   seq_len:        [B] int32 committed entries per request.
 *   pending:        [B] int32 drafted, not yet committed entries.
 * Invariant kept by every entry point: each pool slot that no request holds
 * (at or beyond seq_len + pending) is all-zero bits, provided the pools start
 * zeroed or filled only below seq_len. */
typedef struct {
  void* k_pool;
  void* v_pool;
  int32_t* block_table;
  int32_t* seq_len;
  int32_t* pending;
  int num_blocks;
  int max_blocks;
} mtp_kv;

typedef struct mtp_ctx mtp_ctx;

/* Create a context on `device`.  `weights` may be NULL for a context that
 * only verifies and edits the KV cache.  Allocates the context's workspace
 * (activations, split-KV partials, argmax keys, counters, error word) and the
 * rotary table (angles computed in double on the host).  Returns
 * MTP_ERR_INVALID on a bad shape, MTP_ERR_OOM / MTP_ERR_CUDA on failure; on
 * success *out owns the workspace until mtp_destroy. */
mtp_status mtp_init(const mtp_config* cfg, const mtp_weights* weights, int device, mtp_ctx** out);

/* K recursive MTP draft steps for B requests ("Architecture" of the MTP
 * page; inputs as in "The MTP inputs").
 *   hidden    [B, H]  verifier hidden state per request (dtype).
 *   embeds    [B, H]  embedding of the token at positions[b] (dtype).
 *   positions [B]     int32; step k (1-based) runs at positions[b] + k - 1
 *                     and writes KV slot seq_len[b] + k - 1.
 *   kv        the MTP cache; requires pending[b] == 0 on entry, leaves
 *             pending[b] == K (commit or roll back before the next draft).
 *   K         1..max_k.
 *   chain_ids [B, K-1] int32 or NULL: when given, step k >= 2 embeds
 *             chain_ids[b, k-2] (a given token chain, as in training)
 *             instead of the previous draft.
 *   draft_ids [B, K] int32 out: argmax of each step's logits, lowest id on
 *             ties.
 *   logits    [B, K, V] float32 out, or NULL.
 *   hidden_out[B, H] float32 out (decoder output of step K), or NULL.
 * Host errors: ctx without weights, B outside 1..max_batch, K outside
 * 1..max_k, NULL required pointers.  Device errors (MTP_ERR_DEVICE_ARGS,
 * MTP_ERR_CAPACITY; read with mtp_get_device_error): pending != 0 on entry
 * -- that request's cache and pending are then left untouched at every step
 * --, a slot beyond the block table or pool, a position beyond max_pos (that
 * write is skipped).  Batches of 1..persistent_max_batch run in one
 * cooperative launch that holds every SM of the device; its waits give up
 * after 2 s with MTP_ERR_TIMEOUT, and the context then refuses further
 * persistent drafts (they return at once with the same error) until
 * mtp_get_device_error has read it. */
mtp_status mtp_draft(mtp_ctx* ctx, void* stream, int B, const void* hidden, const void* embeds,
                     const int32_t* positions, const mtp_kv* kv, int K, const int32_t* chain_ids,
                     int32_t* draft_ids, float* logits, float* hidden_out);

/* Greedy verification ("Overview" of the speculative-decoding page).
 * For request b with K_b = num_drafts[b] (0..max_k) drafts, target rows
 * row_offsets[b] .. row_offsets[b] + K_b of target_logits [num_rows, V]
 * (dtype) give r_j = argmax of row j (lowest id on ties, -0 equal to +0, NaN
 * entries passed over; a row of NaN only gives r_j = -1); accepted[b] = the
 * largest a <= K_b with drafts[b*drafts_stride + j] == r_j for all j < a;
 * bonus[b] = r_a.  Device-checked per request: K_b <= min(max_k,
 * drafts_stride), row_offsets[b+1] - row_offsets[b] == K_b + 1, and the rows
 * lie inside [0, num_rows); on violation accepted[b] = bonus[b] = -1 and the
 * error word is set.  Every one of the num_rows rows is read (the rows are
 * scanned as one flat range split evenly over the grid), so num_rows must not
 * exceed the rows target_logits holds; host-checked: 1 <= num_rows <=
 * max_batch * (max_k + 1), else MTP_ERR_INVALID. */
mtp_status mtp_verify(mtp_ctx* ctx, void* stream, int B, const void* target_logits, int num_rows,
                      const int32_t* row_offsets, const int32_t* drafts, int drafts_stride,
                      const int32_t* num_drafts, int32_t* accepted, int32_t* bonus);

/* Greedy verification without a context and without allocating.  The
 * pages have no counterpart: this is a deployment variant of mtp_verify for
 * callers that cannot allocate device memory where they verify -- a serving
 * loop whose device memory is wholly owned by a fixed plan or another
 * framework's pool, or a latency-bound loop that cannot afford the implicit
 * device-wide synchronisation of cudaMalloc (mtp_init allocates, so such a
 * caller cannot create a context there).  Same arguments and results as
 * mtp_verify, with the shape passed directly: vocab, dtype (mtp_dtype) and
 * max_k (0..100) in place of the context.
 *   Scratch: a fixed array of 65536 argmax keys and one arrival counter
 *   (about 512 KB) that is part of the library's device image; every GPU that
 *   loads the library holds it until the process exits.  Requires B <= 4096,
 *   B * (max_k + 1) <= 65536 and num_rows <= 65536, else MTP_ERR_INVALID.
 *   Set-up: the first call on a device looks up that array's device address
 *   (once per device, under a lock); make that first call before any stream
 *   capture on the device.
 *   Sharing: every call uses the same array and clears the part it needs on
 *   `stream` before its kernel; calls whose work overlaps on the GPU (other
 *   streams, other host threads) race on it and must be serialised by the
 *   caller.  Device-detected argument errors give accepted[b] = bonus[b] = -1
 *   (there is no context error word).  Nothing is allocated: no cudaMalloc,
 *   cudaFree or allocating library routine is called. */
mtp_status mtp_verify_noalloc(void* stream, int B, int vocab, int dtype, int max_k, const void* target_logits,
                              int num_rows, const int32_t* row_offsets, const int32_t* drafts,
                              int drafts_stride, const int32_t* num_drafts, int32_t* accepted,
                              int32_t* bonus);

/* Commit ("Stateful execution"; "Tree Drafting" step 4): request b keeps
 * its first n_keep[b] drafted slots, the other drafted slots are zeroed in
 * place, seq_len[b] += n_keep[b], pending[b] = 0.  n_keep [B] int32 device
 * array, 0 <= n_keep[b] <= pending[b] (device-checked; a request that fails
 * the check is left unchanged and the error word is set). */
mtp_status mtp_kv_commit(mtp_ctx* ctx, void* stream, int B, const mtp_kv* kv, const int32_t* n_keep);

/* Commit with n_keep[b] = min(accepted[b] + extra, pending[b]) computed on
 * the device from mtp_verify's output.  extra = 1 keeps the slot of the last
 * confirmed input token; extra = 0 keeps only accepted drafts. */
mtp_status mtp_kv_commit_accepted(mtp_ctx* ctx, void* stream, int B, const mtp_kv* kv,
                                  const int32_t* accepted, int extra);

/* Roll back every drafted slot: commit with n_keep = 0. */
mtp_status mtp_kv_rollback(mtp_ctx* ctx, void* stream, int B, const mtp_kv* kv);

/* Return request b to a prefix of new_len[b] entries ("Prefix Caching with
 * Speculative Decoding"): slots new_len[b] .. seq_len[b]+pending[b]-1 are
 * zeroed, seq_len[b] = new_len[b], pending[b] = 0.  Requires
 * 0 <= new_len[b] <= seq_len[b] + pending[b] (device-checked). */
mtp_status mtp_kv_truncate(mtp_ctx* ctx, void* stream, int B, const mtp_kv* kv, const int32_t* new_len);

/* INT4 asymmetric quantization of a bf16 matrix [rows, cols] (row-major,
 * cols a multiple of 64) in groups of 64 consecutive columns: for a group,
 * lo = min(min w, 0), hi = max(max w, 0), s = (hi - lo) / 15 (1 if 0),
 * z = clamp(rint(-lo / s), 0, 15), q = clamp(rint(w / s) + z, 0, 15), all in
 * IEEE fp32 with round-half-to-even.  Outputs (device, caller-owned): q
 * [rows, cols/2] bytes, column 2k in the low nibble of byte k; scales [rows,
 * cols/64] fp16 (s rounded to nearest even); zeros [rows, cols/64] bytes.
 * Dequantized weight: (q - z) * scale.  Asynchronous on `stream`;
 * MTP_ERR_INVALID for NULL pointers or a bad shape. */
mtp_status mtp_quantize_int4_g64(void* stream, const void* w, int rows, int cols, void* q, void* scales,
                                 void* zeros);

/* INT8 symmetric quantization of a bf16 matrix [rows, cols] per row:
 * s = max |w| / 127 (1 if 0), q = clamp(rint(w / s), -127, 127) in IEEE fp32
 * with round-half-to-even.  Outputs: q [rows, cols] int8, scales [rows] fp16.
 * Dequantized weight: q * scale. */
mtp_status mtp_quantize_int8_rows(void* stream, const void* w, int rows, int cols, void* q, void* scales);

/* ------------------------------------------------------------------------
 * The speculative loop around the step (an end-to-end harness).
 *
 * No trained target model exists in this library's tests, so a
 * deterministic synthetic verifier stands in for it; it is a pure function
 * of the token prefix, so plain greedy decoding with it is well defined and
 * the speculative loop must reproduce it token for token ("How OpenVINO MTP
 * Speculative Decoding Works Internally": the speculative result is the
 * main model's greedy result; "Speculative Decoding", "Overview").  Hashing
 * is the SplitMix64 finaliser mix() on 64-bit words:
 *   fold(h, t) = mix(h + 0x9E3779B97F4A7C15 * (t + 1))   (prefix + token t)
 *   prediction after a prefix (hash h, last token l): l if
 *     (mix(h ^ 0xD1B54A32D192ED03) >> 11) < sticky_thr, else
 *     mix(h ^ 0x8CB92BA72F3D8DD7) mod V
 *   logits: ((mix(h ^ (0x9E3779B97F4A7C15 * (v + 1))) >> 40) * 2^-24 - 0.5
 *     in the context's dtype, 8.0 at the prediction
 *   hidden state: 2 * ((mix(h ^ 0x2545F4914F6CDD1D ^ (0x9E3779B97F4A7C15 *
 *     (i + 1))) >> 40) * 2^-24 - 0.5) in the context's dtype.
 * ---------------------------------------------------------------------- */

/* Verifier rows for B requests with nd_b = num_drafts[b] drafts each (K for
 * every request when num_drafts is NULL; 0 <= nd_b <= K <= max_k): request
 * b's rows start at o_b = sum_{c<b} (nd_c + 1), and row o_b + j is the
 * verifier's output for the prefix (seq_hash[b], last_tok[b]) extended by
 * drafts[b*K .. b*K+j-1], j = 0..nd_b.  logits [B*(K+1), V] in the context's
 * dtype (rows past the last are untouched); row_offsets [B+1] (optional)
 * receives o_b.  drafts may be NULL when K = 0.  All device, caller-owned;
 * asynchronous. */
mtp_status mtp_synth_target(mtp_ctx* ctx, void* stream, int B, int K, const int32_t* num_drafts,
                            const uint64_t* seq_hash, const int32_t* last_tok, const int32_t* drafts,
                            uint64_t sticky_thr, void* logits, int32_t* row_offsets);

/* Dynamic draft length ("Speculative Decoding", "Fast Draft": the drafter
 * keeps proposing while the candidate token's probability exceeds a
 * threshold).  conf [B, K] receives the probability of each draft step's
 * argmax token under its logits (logits [B, K, V] fp32 as mtp_draft writes
 * them): 1 / sum_v exp(z_v - max z).  num_drafts [B] (optional) receives the
 * length of the leading run of steps with conf > tau. */
mtp_status mtp_draft_confidence(mtp_ctx* ctx, void* stream, int B, int K, const float* logits, float tau,
                                float* conf, int32_t* num_drafts);

/* The next step's draft count from recent acceptance (host-side; the pages
 * adapt the number of assistant tokens per step without giving a rule): K + 2
 * after a step whose `drafted` drafts were all accepted, K - 1 otherwise,
 * clamped to [k_min, k_max]. */
int mtp_adapt_k(int K, int accepted, int drafted, int k_min, int k_max);

/* Advance the loop state after verification: request b emits drafts
 * drafts[b*K .. b*K+accepted[b]-1] and bonus[b] (appended to
 * out_tokens[b*out_cap + out_len[b] ...] while they fit; out_len[b] counts
 * every emitted token, and a token past out_cap sets the device error
 * MTP_ERR_CAPACITY), folds them into seq_hash[b], sets last_tok[b] =
 * bonus[b], advances positions[b] by accepted[b] + 1, and writes the next
 * step's inputs: hidden[b] = the verifier hidden state of the new prefix,
 * embeds[b] = row bonus[b] of the context's embedding table ([B, H] each, the
 * context's dtype).  accepted[b] outside 0..K or bonus[b] outside the
 * vocabulary set MTP_ERR_DEVICE_ARGS and leave request b unchanged. */
mtp_status mtp_loop_advance(mtp_ctx* ctx, void* stream, int B, int K, const int32_t* drafts,
                            const int32_t* accepted, const int32_t* bonus, uint64_t* seq_hash, int32_t* last_tok,
                            int32_t* positions, void* hidden, void* embeds, int32_t* out_tokens,
                            int32_t* out_len, int out_cap);

/* State and scratch of mtp_spec_loop (all device pointers, caller-owned). */
typedef struct {
  int B;                  /* requests (1..max_batch) */
  int K;                  /* drafts per step (1..max_k); 0 = plain greedy decoding with the verifier */
  uint64_t sticky_thr;    /* verifier parameter (see above) */
  uint64_t* seq_hash;     /* [B] */
  int32_t* last_tok;      /* [B] */
  int32_t* positions;     /* [B] position of last_tok (the next draft input) */
  void* hidden;           /* [B, H] verifier hidden state for the next draft */
  void* embeds;           /* [B, H] embedding of last_tok */
  int32_t* drafts;        /* [B, max(K, 1)] scratch */
  int32_t* accepted;      /* [B] scratch (the last step's accepted counts on return) */
  int32_t* bonus;         /* [B] scratch */
  int32_t* num_drafts;    /* [B] scratch */
  int32_t* row_offsets;   /* [B + 1] scratch */
  void* target_logits;    /* [B * (K + 1), V] scratch, the context's dtype */
  int32_t* out_tokens;    /* [B, out_cap] emitted tokens */
  int32_t* out_len;       /* [B] emitted counts */
  int out_cap;
  float conf_threshold;   /* > 0: propose only the leading drafts whose probability exceeds it */
  float* draft_logits;    /* [B, K, V] fp32 scratch (with conf_threshold) */
  float* conf;            /* [B, K] scratch (with conf_threshold) */
} mtp_loop;

/* `iters` steps of the speculative loop on `stream`, no host synchronisation:
 * mtp_draft (K drafts) [-> mtp_draft_confidence: num_drafts from the
 * threshold] -> mtp_synth_target -> mtp_verify -> mtp_kv_commit_accepted
 * (extra = 1) -> mtp_loop_advance.  With K = 0 each
 * step is one token of plain greedy decoding (no drafting, no cache edit).
 * The cache must have room for the committed entries of all steps. */
mtp_status mtp_spec_loop(mtp_ctx* ctx, void* stream, const mtp_kv* kv, const mtp_loop* loop, int iters);

/* ------------------------------------------------------------------------
 * Tree drafting ("Speculative Decoding", "Tree Drafting", "How Tree Drafting
 * Works"), with the MTP head as the drafter.  Layer 1 is the MTP step from
 * the verifier's hidden state and the last token; it proposes the
 * `branching` most probable tokens.  At layer l >= 2 the `branching`
 * candidates of layer l-1 with the highest cumulative log-probability (all
 * of them at l = 2) are each expanded by one MTP step (input: the node's
 * token and the output hidden state of the step that proposed it; position
 * p + l - 1; attention over the committed cache plus the MTP entries of the
 * node's ancestors) into their `branching` most probable children.  The
 * `n_assist` candidates with the best cumulative score (ties: smaller depth,
 * then earlier creation) form the packed tree, ordered by (depth, creation)
 * so that parents come first.  The page's rules are enforced:
 * branching^2 (depth-1) + branching >= n_assist >= depth.  Limits:
 * branching <= 8, depth <= 16, n_assist <= 64, B * branching <= max_batch,
 * max_k >= 2 when depth >= 2.
 * ---------------------------------------------------------------------- */
typedef struct {
  int B, branching, depth, n_assist;
  int32_t* scratch_blocks;   /* [(depth-1) * B * branching * 2] ids of free blocks of the cache pool,
                                used for the expansions' private copies (device) */
  void* ws;                  /* workspace of at least mtp_tree_workspace_bytes(...) bytes (device) */
  size_t ws_bytes;
  int32_t* tokens;           /* [B, n_assist] packed nodes' tokens (device, written by mtp_draft_tree) */
  int32_t* parents;          /* [B, n_assist] parent node index, -1 for a child of the root */
  int32_t* depths;           /* [B, n_assist] 1..depth */
} mtp_tree;

/* Workspace bytes of one tree call for a cache whose block tables have
 * `max_blocks` entries; 0 for a bad shape. */
size_t mtp_tree_workspace_bytes(const mtp_ctx* ctx, int B, int branching, int depth, int n_assist, int max_blocks);

/* Draft the trees of B requests (inputs as mtp_draft's).  The root step
 * writes slot seq_len[b] of each request's cache (pending[b] = 1; pending
 * must be 0 on entry); expansions write only the private scratch blocks.
 * Every slot seq_len[b] .. seq_len[b] + depth must lie in the block table
 * (device-checked: MTP_ERR_CAPACITY). */
mtp_status mtp_draft_tree(mtp_ctx* ctx, void* stream, const void* hidden, const void* embeds,
                          const int32_t* positions, const mtp_kv* kv, const mtp_tree* tree);

/* The synthetic verifier's rows for the packed trees: request b's rows start
 * at b * (1 + n_assist); row 0 follows the committed prefix, row 1 + i the
 * prefix extended by node i's path.  row_offsets [B+1] optional. */
mtp_status mtp_synth_target_tree(mtp_ctx* ctx, void* stream, const mtp_tree* tree, const uint64_t* seq_hash,
                                 const int32_t* last_tok, uint64_t sticky_thr, void* logits, int32_t* row_offsets);

/* Tree verification: starting at the root, follow the child whose token is
 * the verifier's argmax (lowest id on ties) after the current prefix, while
 * one exists.  accepted [B] nodes on that path, their tokens in
 * path_tokens [B, depth], bonus [B] the last argmax.  target_logits
 * [B * (1 + n_assist), V] in the context's dtype, rows as above. */
mtp_status mtp_verify_tree(mtp_ctx* ctx, void* stream, const mtp_tree* tree, const void* target_logits,
                           int32_t* accepted, int32_t* bonus, int32_t* path_tokens);

/* Keep the root's entry and the entries of the accepted nodes that were
 * expanded (in path order, slots seq_len[b] + 1, ...), then advance
 * seq_len[b] by their count and clear pending[b]. */
mtp_status mtp_tree_commit(mtp_ctx* ctx, void* stream, const mtp_kv* kv, const mtp_tree* tree,
                           const int32_t* accepted);

/* `iters` steps of the speculative loop with tree drafting: mtp_draft_tree
 * -> mtp_synth_target_tree -> mtp_verify_tree (path into loop->drafts
 * [B, depth]) -> mtp_tree_commit -> mtp_loop_advance.  loop->target_logits
 * holds B * (1 + n_assist) rows. */
mtp_status mtp_tree_loop(mtp_ctx* ctx, void* stream, const mtp_kv* kv, const mtp_loop* loop, const mtp_tree* tree,
                         int iters);

/* Failure-detection diagnostic.  Runs one of the library's bounded waits on
 * a condition that never becomes true, so that the wait runs out as it would
 * for a lost arrival in a real launch: which = 0, the shared-memory barrier
 * phase wait of the streamed kernels (a barrier nobody arrives at, 4096
 * polls); which = 1, the persistent kernel's grid-barrier counter wait (a
 * private counter nobody increments, 2 s of the GPU's global timer).  The
 * kernel records MTP_ERR_TIMEOUT in the context's error word and returns; it
 * touches nothing else, so the context stays usable.  Returns MTP_ERR_INVALID
 * for a null context or another `which`; asynchronous on `stream` otherwise.
 * mtp_get_device_error then reads (and clears) MTP_ERR_TIMEOUT. */
mtp_status mtp_selftest_wait_timeout(mtp_ctx* ctx, void* stream, int which);

/* Synchronise the context's device, return the device error word as an
 * mtp_status (MTP_OK if none) and clear it. */
mtp_status mtp_get_device_error(mtp_ctx* ctx);

/* Free the workspace and the context.  NULL is a no-op. */
void mtp_destroy(mtp_ctx* ctx);

/* Static string naming a status. */
const char* mtp_status_str(mtp_status s);

/* Device-to-device copy of `bytes` bytes with 16-byte vector loads/stores
 * over a grid sized to the SM count (the bandwidth yardstick measured next
 * to the kernels).  dst and src must be 16-byte aligned and not overlap;
 * bytes a multiple of 16. */
mtp_status mtp_stream_copy(void* stream, void* dst, const void* src, size_t bytes);

/* Bounds-checked builds.  A library compiled with -DMTP_CHECKED (the
 * package builds it as libmtp_checked.so; the binding loads it when the
 * environment variable MTP_LIBRARY names it) checks every output store of
 * the draft, verify and KV kernels against the extent of its buffer for the
 * call (logits B*K*V, draft ids B*K, hidden_out B*H, accepted/bonus B,
 * activations B*width, the KV pools num_blocks*n_kv*block_size*head_dim,
 * the verify keys num_rows, the attention partials); a store outside is
 * skipped and the error word records MTP_ERR_BOUNDS -- no trap.  It is the
 * stand-in for a memory checker, which is not available here.
 * mtp_selftest_bounds: checked builds run one store one element past a
 * 4-element extent through the check (nothing is written) and return
 * MTP_OK, leaving MTP_ERR_BOUNDS in the context's error word; other builds
 * return MTP_ERR_INVALID and launch nothing.  Errors: MTP_ERR_INVALID for
 * a NULL context. */
mtp_status mtp_selftest_bounds(mtp_ctx* ctx, void* stream);

/* Read-only yardstick: `bytes` bytes at src (device memory, 16-byte aligned,
 * bytes a multiple of 16) are streamed once into shared memory with bulk
 * copies -- one CTA per SM, a contiguous share each, the mechanism of the
 * streamed kernels -- and nothing is computed or written.  Its duration is
 * the floor of a kernel that only has to read that many bytes (launch,
 * first-byte latency and tail included).  err_word: optional caller-owned
 * device int that receives MTP_ERR_TIMEOUT if a bounded wait ran out (NULL:
 * not reported).  Asynchronous on `stream`; MTP_ERR_INVALID for bad
 * arguments. */
mtp_status mtp_stream_read(void* stream, const void* src, size_t bytes, int* err_word);

/* Kernel timing.  Kernel ids for mtp_profile_begin. */
typedef enum {
  MTP_KERNEL_EH_PROJ = 0,
  MTP_KERNEL_QKV_ROPE = 1,
  MTP_KERNEL_ATTENTION = 2,
  MTP_KERNEL_O_PROJ = 3,
  MTP_KERNEL_GATE_UP = 4,
  MTP_KERNEL_DOWN = 5,
  MTP_KERNEL_LM_HEAD = 6,
  MTP_KERNEL_VERIFY = 7,
  MTP_KERNEL_KV_EDIT = 8,
  MTP_KERNEL_DRAFT_PERSISTENT = 9, /* all K steps of one small-batch draft call */
  MTP_KERNEL_COUNT = 10
} mtp_kernel_id;

/* Start recording CUDA events around every launch of kernel `kernel` (up to
 * `capacity` launches) on the stream it is launched on.  Recording adds one
 * event pair per launch.  Returns MTP_ERR_INVALID for a bad id or capacity. */
mtp_status mtp_profile_begin(mtp_ctx* ctx, int kernel, int capacity);

/* Stop recording; synchronise; write up to `max_out` per-launch durations in
 * milliseconds to ms_out (host array) and their count to *n_out. */
mtp_status mtp_profile_end(mtp_ctx* ctx, float* ms_out, int max_out, int* n_out);

/* Number of kernel launches the context has issued since creation (all
 * entry points), for launch accounting. */
int64_t mtp_launch_count(const mtp_ctx* ctx);

/* Launch-time path choices the context has taken since creation, for tests
 * and diagnostics (which of two equivalent forms ran).  Ids for
 * mtp_path_count: */
typedef enum {
  MTP_PATH_LM_DEFERRED = 0,  /* one-request draft steps before the last whose LM head left its argmax
                                to the next step's eh_proj ("MTP (Multi-Token Prediction)",
                                "Architecture": each step's token feeds the next step) */
  MTP_PATH_ATTN_CLUSTER = 1, /* attention launches whose splits were combined in a thread-block
                                cluster instead of through HBM partials */
  MTP_PATH_COUNT = 2
} mtp_path_id;

/* Count of path `path` (an mtp_path_id); 0 for a NULL context or an unknown
 * id.  Host-side counter, no synchronisation. */
int64_t mtp_path_count(const mtp_ctx* ctx, int path);

#ifdef __cplusplus
}
#endif

#endif /* MTP_H_ */
