"""Plain float64 oracle of the MTP draft-and-verify step.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Nothing here is tuned:
every step is written the way the pages describe it, request by request, with
numpy matrix products as the only library primitive.

Sources (page title, section):
  [P1] "How OpenVINO MTP Speculative Decoding Works Internally":
       "The MTP inputs", "Why the MTP graph is a single decoder layer",
       "Shared embeddings reduce duplication", "Stateful execution".
  [P2] "MTP 深度解析：把投机能力训进模型里": section 4.2 (self-speculation
       example), section 4.4 (chained conditioning on the previous token).
  [P3] "Speculative Decoding" (OpenVINO GenAI): "Overview" (greedy accept
       rule, near-tie caveat), "Tree Drafting" step 4 (caches advanced to the
       accepted prefix), "Prefix Caching with Speculative Decoding" (restore
       to a common prefix).
  [P4] "MTP (Multi-Token Prediction)" (speculators user guide):
       "Architecture" (dual norm, concat, project, decoder layer, shared LM
       head, recursion), "Training Process" (step k conditions on the token
       at t+k).

Readings where the pages leave a step open (each is also listed in the
design notes):
  R1  concat order [norm(hidden) ; norm(embedding)], hidden first, as listed.
  R2  a final RMSNorm with its own weight precedes the shared LM head; the
      hidden passed to the next step is the decoder layer output before it.
  R3  "standard decoder layer": pre-norm attention block then pre-norm SwiGLU
      block, each with a residual add; no per-head q/k norm.
  R4  rotary embedding: rotate-half pairs (i, i + d/2) over the full head
      dim, inv_freq_i = theta^(-2i/d); keys are cached after rotation.
  R5  attention scale 1/sqrt(d); q head h reads kv head h // (n_q / n_kv);
      the query of draft step k sees the committed entries and drafted
      entries 1..k (its own included).
  R6  RMSNorm y = x / sqrt(mean(x^2) + eps) * w.
  R8  argmax ties resolve to the lowest id.
  R9  kv_commit(n_keep) keeps the first n_keep drafted slots and zeroes the
      rest; rollback = commit(0).
  R10 verify rows are ragged, located by row offsets.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, Optional, Tuple

import numpy as np

# ------------------------------------------------------------ number formats


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact conversion of stored values to float64.  ``dtype`` "bf16" means
    ``x`` holds bf16 bit patterns (uint16): the value is those 16 bits placed
    in the upper half of an IEEE float32."""
    if dtype == "bf16":
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 precision, nearest-even.

    bf16 keeps 8 significant bits (1 implicit + 7 stored).  With
    x = m * 2^e and 0.5 <= |m| < 1 (frexp), the bf16 value is
    rint(m * 2^8) * 2^(e - 8); numpy's rint rounds halves to even.  Valid for
    the normal range, which is all the KV values here ever reach."""
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def bf16_bits_of(x_bf16_valued: np.ndarray) -> np.ndarray:
    """Bit patterns of values that are already exactly representable in bf16."""
    f = np.asarray(x_bf16_valued, dtype=np.float32)   # exact for such values
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def store_kv_values(x: np.ndarray, dtype: str) -> np.ndarray:
    """Values as the KV cache holds them: bf16 bits, or float32."""
    if dtype == "bf16":
        return bf16_bits_of(round_to_bf16(x))
    return np.asarray(x, dtype=np.float32)


# --------------------------------------------------------------- primitives


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """R6: y = x / sqrt(mean(x^2) + eps) * w along the last axis.
    [P4] "Architecture": hidden state and embedding are normalised separately;
    the decoder layer and LM head inputs are normalised the same way."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rope(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """R4: rotate-half rotary embedding of ``x`` [n_heads, d] at position
    ``pos``.  Pair i couples element i with element i + d/2 and turns it by
    pos * theta^(-2i/d) radians (angles in float64)."""
    d = x.shape[-1]
    half = d // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / d)
    ang = float(pos) * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """R5: per q head h, o_h = softmax(q_h . K_g^T / sqrt(d)) V_g with
    g = h // (n_q / n_kv).  q [n_q, d]; k, v [T, n_kv, d].  Softmax in two
    passes: subtract the max, exponentiate, divide by the sum.
    [P4] "Architecture" (attention of the standard decoder layer);
    [P1] "Why the MTP graph is a single decoder layer" (its own one-layer
    cache)."""
    n_q, d = q.shape
    n_kv = k.shape[1]
    group = n_q // n_kv
    out = np.empty_like(q)
    for h in range(n_q):
        g = h // group
        scores = (k[:, g, :] @ q[h]) / np.sqrt(d)
        m = np.max(scores)
        p = np.exp(scores - m)
        p = p / np.sum(p)
        out[h] = p @ v[:, g, :]
    return out


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def swiglu_mlp(n2: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """W_down (silu(W_gate n) * (W_up n)); rows of n2 are independent."""
    return (silu(n2 @ w_gate.T) * (n2 @ w_up.T)) @ w_down.T


def eh_proj(h: np.ndarray, e: np.ndarray, W: "MTPWeights64") -> np.ndarray:
    """[P4] "Architecture": normalise hidden and embedding separately,
    concatenate (R1: hidden first), project 2H -> H."""
    cat = np.concatenate([rmsnorm(h, W.w_norm_h, W.eps), rmsnorm(e, W.w_norm_e, W.eps)], axis=-1)
    return cat @ W.w_eh.T


def lm_head(h2: np.ndarray, W: "MTPWeights64") -> np.ndarray:
    """R2 + [P4] "Architecture" ("a shared LM head produces draft logits"):
    z = W_lm . RMSNorm_f(h2).  Rows of the LM head are processed in chunks of
    rows only to bound memory; every logit is one whole dot product."""
    n = rmsnorm(h2, W.w_norm_f, W.eps)
    V = W.lm_rows
    z = np.empty(n.shape[:-1] + (V,), dtype=np.float64)
    step = 16384
    for r0 in range(0, V, step):
        r1 = min(V, r0 + step)
        z[..., r0:r1] = n @ W.lm_chunk(r0, r1).T
    return z


def argmax_lowest(z: np.ndarray) -> np.ndarray:
    """R8: index of the maximum along the last axis; ties -> lowest index
    (numpy's argmax returns the first occurrence)."""
    return np.argmax(z, axis=-1).astype(np.int32)


def top2_gap(z: np.ndarray) -> np.ndarray:
    """Difference between the largest and second-largest logit per row."""
    part = np.partition(z, -2, axis=-1)
    return part[..., -1] - part[..., -2]


# ------------------------------------------------------------------ weights


@dataclass
class MTPWeights64:
    """Head weights widened to float64, plus the bf16/f32 embedding table kept
    as stored (widened on use)."""
    w_norm_h: np.ndarray
    w_norm_e: np.ndarray
    w_eh: np.ndarray
    w_norm_in: np.ndarray
    w_q: np.ndarray
    w_k: np.ndarray
    w_v: np.ndarray
    w_o: np.ndarray
    w_norm_post: np.ndarray
    w_gate: np.ndarray
    w_up: np.ndarray
    w_down: np.ndarray
    w_norm_f: np.ndarray
    embed_stored: np.ndarray      # [V, H] as stored (bf16 bits or float32)
    lm_stored: np.ndarray         # [V, H]; the same array when tied
    dtype: str
    n_q: int
    n_kv: int
    head_dim: int
    eps: float
    rope_theta: float

    @property
    def lm_rows(self) -> int:
        return self.lm_stored.shape[0]

    def lm_chunk(self, r0: int, r1: int) -> np.ndarray:
        return widen(self.lm_stored[r0:r1], self.dtype)

    def embed_rows(self, ids: np.ndarray) -> np.ndarray:
        """[P1] "Shared embeddings reduce duplication": the MTP head reads the
        target's own embedding table."""
        return widen(self.embed_stored[np.asarray(ids)], self.dtype)

    @staticmethod
    def from_stored(w: Dict[str, np.ndarray], dtype: str, n_q: int, n_kv: int, head_dim: int,
                    eps: float, rope_theta: float, lm_head: Optional[np.ndarray] = None) -> "MTPWeights64":
        wd = {k: widen(v, dtype) for k, v in w.items() if k != "embed"}
        return MTPWeights64(embed_stored=w["embed"],
                            lm_stored=w["embed"] if lm_head is None else lm_head,
                            dtype=dtype, n_q=n_q, n_kv=n_kv, head_dim=head_dim, eps=eps,
                            rope_theta=rope_theta, **wd)


# ----------------------------------------------------------------- KV cache


def _slot_index(kv, b: int, slot: int) -> Tuple[int, int]:
    bs = kv.block_size
    return int(kv.block_table[b, slot // bs]), slot % bs


def kv_read_slots(kv, b: int, n_slots: int, dtype: str) -> Tuple[np.ndarray, np.ndarray]:
    """Logical view of request b's first n_slots entries: k, v [T, n_kv, d]
    in float64, read through the block table one slot at a time."""
    n_kv, d = kv.k_pool.shape[1], kv.k_pool.shape[3]
    k = np.empty((n_slots, n_kv, d), dtype=np.float64)
    v = np.empty((n_slots, n_kv, d), dtype=np.float64)
    bs = kv.block_size
    for t0 in range(0, n_slots, bs):
        blk = int(kv.block_table[b, t0 // bs])
        t1 = min(n_slots, t0 + bs)
        k[t0:t1] = widen(kv.k_pool[blk, :, :t1 - t0, :], dtype).transpose(1, 0, 2)
        v[t0:t1] = widen(kv.v_pool[blk, :, :t1 - t0, :], dtype).transpose(1, 0, 2)
    return k, v


def _kv_write_slot(kv, b: int, slot: int, k_row: np.ndarray, v_row: np.ndarray, dtype: str) -> None:
    blk, off = _slot_index(kv, b, slot)
    kv.k_pool[blk, :, off, :] = store_kv_values(k_row, dtype)
    kv.v_pool[blk, :, off, :] = store_kv_values(v_row, dtype)


def kv_commit(kv, n_keep: np.ndarray, dtype: str) -> None:
    """R9, in place: keep the first n_keep[b] drafted slots of request b, zero
    the other drafted slots, advance seq_len by n_keep[b], clear pending.
    [P1] "Stateful execution" (the one-layer cache is updated, not rebuilt);
    [P3] "Tree Drafting" step 4 (caches advanced to the accepted tokens)."""
    for b in range(len(kv.seq_len)):
        L, P, n = int(kv.seq_len[b]), int(kv.pending[b]), int(n_keep[b])
        assert 0 <= n <= P
        for slot in range(L + n, L + P):
            blk, off = _slot_index(kv, b, slot)
            kv.k_pool[blk, :, off, :] = 0
            kv.v_pool[blk, :, off, :] = 0
        kv.seq_len[b] = L + n
        kv.pending[b] = 0


def kv_rollback(kv, dtype: str) -> None:
    """R9: discard every drafted slot (commit nothing)."""
    kv_commit(kv, np.zeros(len(kv.seq_len), dtype=np.int32), dtype)


def kv_truncate(kv, new_len: np.ndarray, dtype: str) -> None:
    """[P3] "Prefix Caching with Speculative Decoding": restore a request to a
    shorter common prefix.  Slots from new_len[b] up to seq_len[b] + pending[b]
    are zeroed; seq_len = new_len, pending = 0."""
    for b in range(len(kv.seq_len)):
        L, P, n = int(kv.seq_len[b]), int(kv.pending[b]), int(new_len[b])
        assert 0 <= n <= L + P
        for slot in range(n, L + P):
            blk, off = _slot_index(kv, b, slot)
            kv.k_pool[blk, :, off, :] = 0
            kv.v_pool[blk, :, off, :] = 0
        kv.seq_len[b] = n
        kv.pending[b] = 0


# -------------------------------------------------------------------- draft


@dataclass
class DraftResult:
    logits: np.ndarray        # [B, K, V] float64
    ids: np.ndarray           # [B, K] int32, argmax of each step's logits
    hidden_out: np.ndarray    # [B, H] float64, decoder output of the last step
    q_last: Optional[np.ndarray] = None


def draft(W: MTPWeights64, hidden: np.ndarray, embeds: np.ndarray, positions: np.ndarray,
          kv, K: int, chain_ids: Optional[np.ndarray] = None) -> DraftResult:
    """K recursive MTP draft steps for every request, appending to ``kv`` in
    place (pending becomes K).

    [P4] "Architecture": at each step the head normalises the verifier hidden
    state and the token embedding separately, concatenates them, projects 2H
    to H, runs one standard decoder layer (attention + MLP), and the shared LM
    head gives the step's draft logits; the step's output hidden state feeds
    the next step.
    [P2] section 4.4 / [P4] "Training Process": step k >= 2 is conditioned on
    the embedding of the token at t+k-1 -- at inference the previous draft
    (its argmax).  ``chain_ids`` [B, K-1], when given, supplies those tokens
    instead (the ground-truth chain used in training).

    hidden, embeds: [B, H] float64 (already widened); positions[b] is the
    position of the token whose embedding is embeds[b]; step k uses
    positions[b] + k - 1 and writes KV slot seq_len[b] + k - 1.
    """
    B, H = hidden.shape
    V = W.lm_rows
    d = W.head_dim
    logits = np.empty((B, K, V), dtype=np.float64)
    ids = np.empty((B, K), dtype=np.int32)
    h = hidden.copy()
    e = embeds.copy()
    for b in range(B):
        assert int(kv.pending[b]) == 0
    for k in range(1, K + 1):
        # a2: dual RMSNorm + concat + eh_proj
        x = eh_proj(h, e, W)
        # a3: input RMSNorm, q/k/v projections, rotary embedding, KV append
        n = rmsnorm(x, W.w_norm_in, W.eps)
        q_all = n @ W.w_q.T
        k_all = n @ W.w_k.T
        v_all = n @ W.w_v.T
        o = np.empty((B, W.n_q * d), dtype=np.float64)
        for b in range(B):
            pos = int(positions[b]) + k - 1
            q = rope(q_all[b].reshape(W.n_q, d), pos, W.rope_theta)
            kr = rope(k_all[b].reshape(W.n_kv, d), pos, W.rope_theta)
            vr = v_all[b].reshape(W.n_kv, d)
            slot = int(kv.seq_len[b]) + k - 1
            _kv_write_slot(kv, b, slot, kr, vr, W.dtype)
            kv.pending[b] = k
            # a4: attention over the committed entries and drafted entries 1..k
            kk, vv = kv_read_slots(kv, b, slot + 1, W.dtype)
            o[b] = attention(q, kk, vv).reshape(-1)
        # a5: output projection + residual
        h1 = x + o @ W.w_o.T
        # a6: post-attention RMSNorm + SwiGLU MLP + residual
        h2 = h1 + swiglu_mlp(rmsnorm(h1, W.w_norm_post, W.eps), W.w_gate, W.w_up, W.w_down)
        # a7: final RMSNorm + shared LM head + argmax
        z = lm_head(h2, W)
        logits[:, k - 1, :] = z
        ids[:, k - 1] = argmax_lowest(z)
        # a1 for the next step: recursion on the hidden state; the next
        # embedding is the previous draft's (or the supplied chain token's)
        h = h2
        if k < K:
            nxt = ids[:, k - 1] if chain_ids is None else np.asarray(chain_ids)[:, k - 1]
            e = W.embed_rows(nxt)
    return DraftResult(logits, ids, h)


# ------------------------------------------------------------------- verify


def verify(target_logits: np.ndarray, row_offsets: np.ndarray, drafts: np.ndarray,
           num_drafts: np.ndarray, dtype: str) -> Tuple[np.ndarray, np.ndarray]:
    """Greedy verification, per request b with K_b = num_drafts[b] drafts:
    r_j = argmax of target row j (j = 0..K_b), a = the length of the longest
    prefix with drafts[b, j] == r_j, bonus = r_a.

    [P3] "Overview": tokens the target would have produced anyway are
    accepted; the first divergent token is replaced by the target's own
    token.  [P2] section 4.2 is the K = 1 case."""
    B = len(num_drafts)
    accepted = np.empty(B, dtype=np.int32)
    bonus = np.empty(B, dtype=np.int32)
    for b in range(B):
        K_b = int(num_drafts[b])
        r0 = int(row_offsets[b])
        assert int(row_offsets[b + 1]) - r0 == K_b + 1
        r = argmax_lowest(widen(target_logits[r0:r0 + K_b + 1], dtype))
        a = 0
        while a < K_b and int(drafts[b, a]) == int(r[a]):
            a += 1
        accepted[b] = a
        bonus[b] = r[a]
    return accepted, bonus


def verify_sequential(target_tokens: np.ndarray, drafts: np.ndarray) -> Tuple[int, list]:
    """[P2] section 4.2, stated step by step for a chain of drafts: at each
    step the target's own next token t' is compared with the pending draft t;
    if equal, t is confirmed and the next draft is examined; otherwise t' is
    taken and drafting restarts from there.  If every draft is confirmed the
    target's next token is emitted as well.  Returns (number of confirmed
    drafts, emitted tokens).  ``target_tokens[j]`` is the target's token after
    the first j drafts."""
    emitted = []
    for j in range(len(drafts)):
        t_target = int(target_tokens[j])
        if t_target == int(drafts[j]):
            emitted.append(int(drafts[j]))
            continue
        emitted.append(t_target)
        return j, emitted
    emitted.append(int(target_tokens[len(drafts)]))
    return len(drafts), emitted
