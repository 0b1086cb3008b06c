"""Tree drafting and tree verification for the oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: [P3] "Speculative Decoding" (OpenVINO GenAI), "Tree Drafting" and
"How Tree Drafting Works" steps 1-4, with its two validation rules.  The page
describes the procedure for an EAGLE3 head; here the drafter is the MTP head.

Readings (listed in the design notes):
  T1  layer 1 is the MTP step from the verifier's hidden state and the last
      token; it proposes the branching_factor (bf) most probable tokens.  At
      layer l >= 2 the surviving nodes are the bf candidates of layer l-1
      with the highest cumulative score (all bf candidates at l = 2), and
      each is expanded into its bf most probable children: bf + bf^2 (td-1)
      candidates over td layers.
  T2  expanding a node is one MTP step whose input is the node's token, whose
      hidden state is the output of the step that proposed the node (the
      recursion of chain drafting), at position p + depth, attending over the
      committed cache plus the MTP entries of the node's ancestors (the tree
      attention mask applied to the MTP's own cache).
  T3  score = sum of log-softmax probabilities along the path; order: higher
      score first, then smaller depth, then earlier creation.  Scores do not
      increase along a path, so the top n_assist candidates form a tree (every
      selected node's parent is selected); they are packed in (depth,
      creation) order, parents first.
  T4  verification: verifier row 0 is the prediction after the committed
      sequence, row 1 + i the prediction after node i's path; starting at the
      root, the child whose token equals the current prediction is accepted
      (children of a node have distinct tokens, so at most one matches) until
      none does; the bonus token is the last prediction.
  T5  the MTP cache keeps the root's entry and the entries of the accepted
      nodes that were expanded, in path order (chain drafting's min(a+1, K)).
"""
from dataclasses import dataclass
from typing import List, Optional, Tuple

import numpy as np

from .mtp_oracle import draft


def tree_is_valid(bf: int, td: int, n_assist: int) -> bool:
    """The two validation rules of "How Tree Drafting Works"."""
    return bf * bf * (td - 1) + bf >= n_assist and n_assist >= td


def log_softmax(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    m = z.max()
    return z - (m + np.log(np.exp(z - m).sum()))


def top_k(z: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest values, larger first, lower index first on
    ties."""
    order = np.lexsort((np.arange(len(z)), -np.asarray(z, dtype=np.float64)))
    return order[:k]


@dataclass
class Cand:
    token: int
    parent: int               # index in the candidate list, -1 = the root
    depth: int                # 1..td
    score: float
    hidden_from: np.ndarray   # output hidden of the step that proposed it
    kv_from: object           # cache state (one request) of that step, its entry included
    expanded: bool = False
    entry_k: Optional[np.ndarray] = None   # its own MTP entry when expanded
    entry_v: Optional[np.ndarray] = None


@dataclass
class TreeResult:
    tokens: np.ndarray        # [n_assist]
    parents: np.ndarray       # [n_assist], index into tokens or -1
    depths: np.ndarray        # [n_assist]
    scores: np.ndarray        # [n_assist]
    cands: List[Cand]         # every candidate, creation order
    selected: List[int]       # candidate index of each packed node
    root_k: np.ndarray        # the root step's MTP entry
    root_v: np.ndarray
    min_margin: float         # smallest top-k / survivor gap met (near-tie indicator)


def _one_request_kv(kv, b):
    import synth
    return synth.KVState(kv.k_pool.copy(), kv.v_pool.copy(), kv.block_table[b:b + 1].copy(),
                         kv.seq_len[b:b + 1].copy(), kv.pending[b:b + 1].copy(), kv.block_size)


def _entry(kv, slot):
    bs = kv.block_size
    blk = int(kv.block_table[0, slot // bs])
    return kv.k_pool[blk, :, slot % bs].copy(), kv.v_pool[blk, :, slot % bs].copy()


def tree_draft_one(W, hidden: np.ndarray, embed: np.ndarray, position: int, kv1, bf: int, td: int,
                   n_assist: int) -> TreeResult:
    """Tree drafting for one request (hidden, embed: [H] float64; kv1 a
    one-request cache with pending = 0; it is not modified)."""
    assert tree_is_valid(bf, td, n_assist)
    L = int(kv1.seq_len[0])
    root_kv = kv1.copy()
    res = draft(W, hidden[None], embed[None], np.array([position], dtype=np.int32), root_kv, 1)
    root_k, root_v = _entry(root_kv, L)
    lp = log_softmax(res.logits[0, 0])
    kids = top_k(res.logits[0, 0], bf + 1)
    margin = float(res.logits[0, 0, kids[bf - 1]] - res.logits[0, 0, kids[bf]]) if len(kids) > bf else np.inf
    cands: List[Cand] = []
    for t in kids[:bf]:
        cands.append(Cand(int(t), -1, 1, float(lp[t]), res.hidden_out[0].copy(), root_kv))
    layer = list(range(len(cands)))
    for l in range(2, td + 1):
        if l == 2:
            surv = layer
        else:
            order = sorted(layer, key=lambda i: (-cands[i].score, i))
            surv = order[:bf]
            if len(order) > bf:
                margin = min(margin, cands[order[bf - 1]].score - cands[order[bf]].score)
        nxt = []
        for i in surv:
            c = cands[i]
            kv = c.kv_from.copy()
            # the node's step: its own entry goes to slot L + depth, after the
            # committed entries, the root's and the ancestors'
            kv.seq_len[0] = L + c.depth
            kv.pending[0] = 0
            r = draft(W, c.hidden_from[None], W.embed_rows(np.array([c.token])), np.array([position + c.depth]),
                      kv, 1)
            c.expanded = True
            c.entry_k, c.entry_v = _entry(kv, L + c.depth)
            z = r.logits[0, 0]
            lpc = log_softmax(z)
            kk = top_k(z, bf + 1)
            if len(kk) > bf:
                margin = min(margin, float(z[kk[bf - 1]] - z[kk[bf]]))
            for t in kk[:bf]:
                cands.append(Cand(int(t), i, l, c.score + float(lpc[t]), r.hidden_out[0].copy(), kv))
                nxt.append(len(cands) - 1)
        layer = nxt
    order = sorted(range(len(cands)), key=lambda i: (-cands[i].score, cands[i].depth, i))
    if len(order) > n_assist:
        margin = min(margin, cands[order[n_assist - 1]].score - cands[order[n_assist]].score)
    sel = sorted(order[:n_assist], key=lambda i: (cands[i].depth, i))
    pos_of = {c: j for j, c in enumerate(sel)}
    parents = np.array([pos_of[cands[c].parent] if cands[c].parent >= 0 else -1 for c in sel], dtype=np.int32)
    assert all(cands[c].parent < 0 or cands[c].parent in pos_of for c in sel)
    return TreeResult(np.array([cands[c].token for c in sel], dtype=np.int32), parents,
                      np.array([cands[c].depth for c in sel], dtype=np.int32),
                      np.array([cands[c].score for c in sel]), cands, sel, root_k, root_v, margin)


def verify_tree(preds: np.ndarray, tokens: np.ndarray, parents: np.ndarray) -> Tuple[int, List[int], int]:
    """T4.  preds[0] is the prediction after the committed sequence,
    preds[1 + i] after node i's path.  Returns (accepted count, accepted node
    indices in path order, bonus token)."""
    node, path = -1, []
    while True:
        want = int(preds[0 if node < 0 else 1 + node])
        kids = [i for i in range(len(tokens)) if parents[i] == node and int(tokens[i]) == want]
        if not kids:
            return len(path), path, want
        assert len(kids) == 1
        node = kids[0]
        path.append(node)


def verify_tree_bruteforce(preds: np.ndarray, tokens: np.ndarray, parents: np.ndarray) -> Tuple[int, int]:
    """The longest root-to-node path whose every token equals the prediction
    after its prefix, by enumerating all paths; returns (length, bonus)."""
    best, best_bonus = 0, int(preds[0])
    for i in range(len(tokens)):
        chain = []
        j = i
        while j >= 0:
            chain.append(j)
            j = int(parents[j])
        chain.reverse()
        ok = all(int(tokens[n]) == int(preds[0 if k == 0 else 1 + chain[k - 1]]) for k, n in enumerate(chain))
        if ok and len(chain) > best:
            best, best_bonus = len(chain), int(preds[1 + chain[-1]])
    return best, best_bonus


def commit_tree(kv, b: int, tr: TreeResult, path: List[int]) -> int:
    """T5 in place on request b of `kv` (pending = 0 on entry): write the
    root's entry and the accepted expanded nodes' entries at slots L, L+1, ...
    and advance seq_len.  Returns the number of entries kept."""
    L = int(kv.seq_len[b])
    bs = kv.block_size
    entries = [(tr.root_k, tr.root_v)]
    for node in path:
        c = tr.cands[tr.selected[node]]
        if not c.expanded:
            break
        entries.append((c.entry_k, c.entry_v))
    for j, (k, v) in enumerate(entries):
        slot = L + j
        blk = int(kv.block_table[b, slot // bs])
        kv.k_pool[blk, :, slot % bs] = k
        kv.v_pool[blk, :, slot % bs] = v
    kv.seq_len[b] = L + len(entries)
    return len(entries)


def node_prefix_tokens(i: int, tokens: np.ndarray, parents: np.ndarray) -> List[int]:
    """Tokens on the path from the root to node i (inclusive), root first."""
    chain = []
    while i >= 0:
        chain.append(int(tokens[i]))
        i = int(parents[i])
    return chain[::-1]


def tree_spec_loop(W, kv, st, bf: int, td: int, n_assist: int, thr: int, iters: int, dtype: str,
                   embed_rows=None) -> np.ndarray:
    """The speculative loop with tree drafting and the synthetic verifier of
    the loop module; updates `st` (LoopState) and `kv`.  Returns the accepted
    counts [iters, B]."""
    from . import loop as L
    B = len(st.last)
    V = W.lm_rows
    H = W.w_eh.shape[0]
    acc = np.zeros((iters, B), dtype=np.int32)
    rows_of = embed_rows or W.embed_rows
    for it in range(iters):
        for b in range(B):
            hidden = L.target_hidden(st.seq_hash[b], H, dtype)
            embed = rows_of(np.array([st.last[b]]))[0]
            kv1 = _one_request_kv(kv, b)
            kv1.pending[0] = 0
            tr = tree_draft_one(W, hidden, embed, st.position[b], kv1, bf, td, n_assist)
            preds = [L.predict(st.seq_hash[b], st.last[b], thr, V)]
            for i in range(len(tr.tokens)):
                h = st.seq_hash[b]
                for t in node_prefix_tokens(i, tr.tokens, tr.parents):
                    h = L.fold(h, t)
                preds.append(L.predict(h, int(tr.tokens[i]), thr, V))
            a, path, bonus = verify_tree(np.array(preds), tr.tokens, tr.parents)
            commit_tree(kv, b, tr, path)
            emitted = [int(tr.tokens[n]) for n in path] + [bonus]
            for t in emitted:
                st.seq_hash[b] = L.fold(st.seq_hash[b], t)
            st.out[b].extend(emitted)
            st.last[b] = bonus
            st.position[b] += a + 1
            acc[it, b] = a
    return acc
