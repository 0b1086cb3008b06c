"""Helpers for the GPU parity tests: move generator output to the device and
back, create contexts, and compare with the oracle under the stated
tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import synth

# Tolerances (draft-step numerics, bf16 weights vs float64 oracle):
LOGIT_TOL = 2e-2       # max_v |z_gpu - z_oracle| / max_v |z_oracle| per (request, step)
NEAR_TIE = 2e-2        # ids may differ only where the oracle's top-2 gap < NEAR_TIE * max|z|
F32_LOGIT_TOL = 1e-3   # the all-float32 head: only summation order differs


def dev(arr: np.ndarray) -> torch.Tensor:
    arr = np.ascontiguousarray(arr)
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(arr).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def upload_weights(w):
    return {k: dev(v) for k, v in w.items()}


# Guard bands (compute-sanitizer is not available, so out-of-bounds writes
# next to an output are looked for directly): every output buffer a test
# hands to the library sits between two bands of a sentinel byte, and the
# bands are checked after the call.
GUARD = 256            # bytes before and after a guarded buffer (keeps 256-byte alignment)
SENTINEL = 0xA5


class Guarded:
    """A device tensor ``t`` of ``shape``/``dtype`` placed inside a larger
    byte buffer whose first and last GUARD bytes hold SENTINEL."""

    def __init__(self, shape, dtype, fill=None):
        esize = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape)) * esize
        self.raw = torch.full((2 * GUARD + n,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(tuple(shape))
        if fill is not None:
            self.t.fill_(fill)

    def check(self, name="buffer"):
        assert bool((self.raw[:GUARD] == SENTINEL).all()), "bytes before %s overwritten" % name
        assert bool((self.raw[-GUARD:] == SENTINEL).all()), "bytes after %s overwritten" % name


def guarded_like(arr: np.ndarray) -> Guarded:
    """A guarded device copy of a host array."""
    arr = np.ascontiguousarray(arr)
    t = dev(arr)
    g = Guarded(tuple(t.shape), t.dtype)
    g.t.copy_(t)
    return g


def upload_kv(kv: synth.KVState):
    """Device copy of the cache; each pool sits between two guard blocks of
    SENTINEL bytes that no block id can reach (checked by download_kv)."""
    import mtp_self_speculative_gb300 as M
    pools = []
    for pool in (kv.k_pool, kv.v_pool):
        raw = np.full((pool.shape[0] + 2,) + pool.shape[1:], 0, dtype=pool.dtype)
        raw.view(np.uint8)[...] = SENTINEL
        raw[1:-1] = pool
        t = dev(raw)
        pools.append((t, t[1:-1]))
    out = M.KVCache(pools[0][1], pools[1][1], dev(kv.block_table), dev(kv.seq_len), dev(kv.pending))
    out.guarded_pools = (pools[0][0], pools[1][0])
    return out


def check_kv_guards(kvd) -> None:
    for raw, name in zip(getattr(kvd, "guarded_pools", ()), ("k_pool", "v_pool")):
        first, last = raw[0].contiguous().view(torch.uint8), raw[-1].contiguous().view(torch.uint8)
        assert bool((first == SENTINEL).all()), "block before %s overwritten" % name
        assert bool((last == SENTINEL).all()), "block after %s overwritten" % name


def download_kv(kvd) -> synth.KVState:
    check_kv_guards(kvd)
    return synth.KVState(host(kvd.k_pool), host(kvd.v_pool), host(kvd.block_table), host(kvd.seq_len),
                         host(kvd.pending))


def make_context(cfg: synth.MTPShape, wdev=None, max_batch=None, max_k=None, max_pos=None, tc_min_batch=0,
                 persistent_max_batch=0, weight_format="dense"):
    import mtp_self_speculative_gb300 as M
    c = M.make_config(cfg.H, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.ffn, cfg.vocab, cfg.eps, cfg.rope_theta,
                      cfg.dtype, max_batch or cfg.batch, max_k or cfg.K, cfg.block_size,
                      max_pos or (cfg.ctx_hi + 64), tc_min_batch, persistent_max_batch, weight_format)
    return M.mtp_init(c, wdev)


def oracle_weights(cfg: synth.MTPShape, w, weight_format="dense") -> O.MTPWeights64:
    if weight_format == "int4_g64":
        from oracle import quant
        return quant.quantized_weights(w, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    return O.MTPWeights64.from_stored(w, cfg.dtype, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)


def check_logits(z_gpu: np.ndarray, z_ora: np.ndarray, tol: float) -> float:
    """Normwise relative error per row; returns the worst."""
    err = np.max(np.abs(z_gpu.astype(np.float64) - z_ora), axis=-1) / np.max(np.abs(z_ora), axis=-1)
    worst = float(np.max(err))
    assert worst <= tol, "logit error %.3e > %.1e" % (worst, tol)
    return worst


def check_ids(ids_gpu: np.ndarray, z_ora: np.ndarray) -> int:
    """ids equal the oracle argmax except at near-ties, where they must be one
    of the near-tied ids.  Returns the number of exact matches."""
    ids_o = O.argmax_lowest(z_ora)
    zmax = np.max(z_ora, axis=-1)
    scale = np.max(np.abs(z_ora), axis=-1)
    exact = 0
    for idx in np.ndindex(ids_gpu.shape):
        g, o = int(ids_gpu[idx]), int(ids_o[idx])
        if g == o:
            exact += 1
            continue
        thr = zmax[idx] - NEAR_TIE * scale[idx]
        assert z_ora[idx][g] >= thr, "id %d at %s is not near-tied with the oracle's %d" % (g, idx, o)
    return exact


def check_ids_are_argmax_of_own_logits(ids_gpu: np.ndarray, logits_gpu: np.ndarray) -> None:
    """The fused cross-CTA argmax is exact: every draft id is the lowest-index
    maximum of the float32 logits the same kernel wrote, bit for bit."""
    np.testing.assert_array_equal(ids_gpu, O.argmax_lowest(logits_gpu))


def exact_floor(n_steps: int) -> int:
    """Least number of steps whose GPU id must equal the oracle's argmax
    exactly.  A bf16 head's logits differ from the oracle's by about 2^-9 of
    their scale, so an id can differ only where the oracle's top-2 gap is
    that small: a few percent of steps at most on random heads.  One step in
    ten (at least one) may differ."""
    return n_steps - max(1, n_steps // 10)


def kv_slots(kv: synth.KVState, b: int, lo: int, hi: int) -> tuple:
    """Raw stored entries of request b's slots [lo, hi): (k, v) [n, n_kv, d]."""
    bs = kv.block_size
    if hi <= lo:
        shape = (0,) + kv.k_pool.shape[1:2] + kv.k_pool.shape[3:]
        return np.zeros(shape, kv.k_pool.dtype), np.zeros(shape, kv.v_pool.dtype)
    ks, vs = [], []
    for s in range(lo, hi):
        blk = int(kv.block_table[b, s // bs])
        ks.append(kv.k_pool[blk, :, s % bs])
        vs.append(kv.v_pool[blk, :, s % bs])
    return np.stack(ks), np.stack(vs)
