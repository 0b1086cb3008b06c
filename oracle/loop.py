"""The full speculative loop around the draft-and-verify step, with a
deterministic synthetic verifier standing in for the target model.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources (page title, section):
  [P1] "How OpenVINO MTP Speculative Decoding Works Internally": the
       speculative result must be the result plain greedy decoding of the main
       model gives (the equivalence the loop is checked against).
  [P3] "Speculative Decoding" (OpenVINO GenAI), "Overview": drafts are kept
       up to the first token the main model would not have produced; the
       main model's own token follows.

The synthetic verifier (a stand-in: no trained target model exists here) is a
pure function of the token prefix.  Hashing uses the SplitMix64 finaliser
(Steele, Lea & Flood, OOPSLA 2014) on unsigned 64-bit words:
  mix(z):  z = (z ^ z>>30) * 0xBF58476D1CE4E5B9; z = (z ^ z>>27) * 0x94D049BB133111EB; z ^ z>>31
  fold(h, token) = mix(h + 0x9E3779B97F4A7C15 * (token + 1))
For a prefix with hash h and last token l:
  u = mix(h ^ 0xD1B54A32D192ED03); if (u >> 11) < thr: the prediction is l
  (a "sticky" target, so a drafter that repeats its input is accepted with
  probability thr / 2^53), else mix(h ^ 0x8CB92BA72F3D8DD7) mod V;
  logits: x_v = (mix(h ^ (0x9E3779B97F4A7C15 * (v + 1))) >> 40) * 2^-24 - 0.5,
  stored in the logits dtype, and 8.0 at the prediction (a unique argmax);
  hidden state: y_i = 2 * ((mix(h ^ 0x2545F4914F6CDD1D ^ (0x9E3779B97F4A7C15 *
  (i + 1))) >> 40) * 2^-24 - 0.5), stored in the activation dtype.
Each step of the loop:
  draft K tokens d_1..d_K from (hidden, embedding of l, position),
  verifier rows j = 0..K for the prefixes seq + d_1..d_j,
  a, bonus = verify (longest prefix of drafts equal to the row argmaxes),
  the MTP cache keeps min(a + 1, K) drafted entries,
  emit d_1..d_a, bonus; fold them into h; l = bonus; position += a + 1;
  hidden = the verifier hidden of the new prefix; embedding = E[bonus].
"""
from dataclasses import dataclass
from typing import List

import numpy as np

from .dynamic import draft_confidence, num_drafts_from_confidence
from .mtp_oracle import draft, kv_commit, round_to_bf16, verify

M64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
C_STICKY = 0xD1B54A32D192ED03
C_TOKEN = 0x8CB92BA72F3D8DD7
C_HIDDEN = 0x2545F4914F6CDD1D


def mix64(z):
    """SplitMix64 finaliser on uint64 numpy arrays (arithmetic modulo 2^64)."""
    z = np.asarray(z, dtype=np.uint64)
    shape = z.shape
    z = z.reshape(-1)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return (z ^ (z >> np.uint64(31))).reshape(shape)


def fold(h: int, token: int) -> int:
    """Hash of a prefix extended by one token."""
    return int(mix64(np.uint64((h + GOLDEN * (token + 1)) & M64)))


def predict(h: int, last: int, thr: int, V: int) -> int:
    """The verifier's greedy next token after a prefix (hash h, last token)."""
    u = int(mix64(np.uint64(h ^ C_STICKY)))
    if (u >> 11) < thr:
        return last
    return int(mix64(np.uint64(h ^ C_TOKEN))) % V


def uniform_half(h: int, n: int) -> np.ndarray:
    """x_i = (mix(h ^ (GOLDEN * (i + 1))) >> 40) * 2^-24 - 0.5, i < n."""
    i = np.arange(1, n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = mix64(np.uint64(h) ^ (np.uint64(GOLDEN) * i))
    return (z >> np.uint64(40)).astype(np.float64) * 2.0 ** -24 - 0.5


def store(x: np.ndarray, dtype: str) -> np.ndarray:
    """Values as the GPU stores them (bf16 round-to-nearest-even, or fp32)."""
    return round_to_bf16(x) if dtype == "bf16" else x.astype(np.float32).astype(np.float64)


def target_row(h: int, last: int, thr: int, V: int, dtype: str) -> np.ndarray:
    z = store(uniform_half(h, V), dtype)
    z[predict(h, last, thr, V)] = 8.0
    return z


def target_hidden(h: int, H: int, dtype: str) -> np.ndarray:
    return store(2.0 * uniform_half(h ^ C_HIDDEN, H), dtype)


@dataclass
class LoopState:
    seq_hash: List[int]       # per request: hash of the sequence so far
    last: List[int]           # last token
    position: List[int]       # position of the last token (the next draft input)
    out: List[List[int]]      # emitted tokens


def greedy(h: int, last: int, thr: int, V: int, n: int) -> List[int]:
    """Plain greedy decoding with the verifier alone: n tokens."""
    toks = []
    for _ in range(n):
        t = predict(h, last, thr, V)
        toks.append(t)
        h = fold(h, t)
        last = t
    return toks


def spec_loop(W, kv, st: LoopState, K: int, thr: int, iters: int, dtype: str, embed_rows=None, conf_tau=None):
    """`iters` speculative steps for every request, updating `st` and `kv`
    (the oracle's draft, verify and commit).  ``embed_rows`` gives the
    embedding the verifier hands to the first draft step (default: the
    head's own table; a quantized head's caller passes the dense table).
    ``conf_tau``: propose only each request's leading drafts whose
    probability exceeds it (the confidence stop of the dynamic module).
    Returns the accepted counts per step [iters, B]."""
    B = len(st.last)
    V = W.lm_rows
    H = W.w_eh.shape[0]
    acc_hist = np.zeros((iters, B), dtype=np.int32)
    for it in range(iters):
        hidden = np.stack([target_hidden(st.seq_hash[b], H, dtype) for b in range(B)])
        embeds = (embed_rows or W.embed_rows)(np.array(st.last))
        res = draft(W, hidden, embeds, np.array(st.position, dtype=np.int32), kv, K)
        nd = np.full(B, K, dtype=np.int32)
        if conf_tau is not None:
            nd = num_drafts_from_confidence(draft_confidence(res.logits), conf_tau)
        rows = []
        for b in range(B):
            h, l = st.seq_hash[b], st.last[b]
            rows.append(target_row(h, l, thr, V, dtype))
            for j in range(int(nd[b])):
                h = fold(h, int(res.ids[b, j]))
                l = int(res.ids[b, j])
                rows.append(target_row(h, l, thr, V, dtype))
        logits = np.stack(rows)
        offs = np.concatenate([[0], np.cumsum(nd.astype(np.int64) + 1)])
        # the rows already hold the stored values (exact in float64)
        a, bonus = verify(logits, offs, res.ids, nd, "f32")
        kv_commit(kv, np.minimum(a + 1, K).astype(np.int32), dtype)
        for b in range(B):
            emitted = [int(t) for t in res.ids[b, :a[b]]] + [int(bonus[b])]
            for t in emitted:
                st.seq_hash[b] = fold(st.seq_hash[b], t)
            st.out[b].extend(emitted)
            st.last[b] = int(bonus[b])
            st.position[b] += int(a[b]) + 1
        acc_hist[it] = a
    return acc_hist
