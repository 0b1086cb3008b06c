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


def upload_kv(kv: synth.KVState):
    import mtp_self_speculative_gb300 as M
    return M.KVCache(dev(kv.k_pool), dev(kv.v_pool), dev(kv.block_table), dev(kv.seq_len), dev(kv.pending))


def download_kv(kvd) -> synth.KVState:
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
