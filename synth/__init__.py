"""Seeded synthetic inputs for the MTP draft-and-verify step.

This module is shared by the tests, the bench and the oracle-side checks.  It
turns (seed, tensor id, index) into numbers and lays them out the way the
draft/verify path expects; it holds none of the method's arithmetic (no norm,
projection, attention, argmax or accept rule).

Recipes (all seeded, all synthetic):
  * linear weights N(0, 0.02); norm weights 1.0 (``norm="ones"``) or
    N(1, 0.1) (``norm="random"``, for unit tests where a dropped weight must
    show);
  * shared token-embedding table E [V, H] N(0, 0.02), tied with the LM head;
  * verifier hidden states N(0, 1); token ids uniform over the vocabulary;
    ``inputs_embeds`` are rows of E gathered at those ids;
  * the MTP KV cache is prefilled with N(0, 1) values (treated as keys that
    already carry their rotary embedding) in paged 16-token blocks;
  * verify logits are N(0, 1) rows with a +8 spike planted at a chosen id per
    row; drafts copy the planted ids up to a seeded accepted length, then
    differ.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field, replace
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_gen.c")
_SO = os.path.join(_HERE, "libsynth.so")
_lib_handle = None

BASE_SEED = 0x4D5450


def build(force: bool = False) -> str:
    """Compile the generator (gcc, OpenMP when available)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", _SO + ".tmp", "-lm"]
    try:
        subprocess.run(base[:4] + ["-fopenmp"] + base[4:], check=True,
                       stdout=subprocess.PIPE, stderr=subprocess.PIPE)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(_SO + ".tmp", _SO)
    return _SO


def _lib():
    global _lib_handle
    if _lib_handle is None:
        build()
        lib = ctypes.CDLL(_SO)
        u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.synth_normal_f32.argtypes = [u64, u64, u64, i64, dbl, dbl, vp]
        lib.synth_normal_bf16.argtypes = [u64, u64, u64, i64, dbl, dbl, vp]
        lib.synth_uniform_i32.argtypes = [u64, u64, u64, i64, i64, i64, vp]
        lib.synth_uniform_f64.argtypes = [u64, u64, u64, i64, vp]
        lib.synth_raw_u64.argtypes = [u64, u64, u64, i64, vp]
        lib.synth_splitmix64_seq.argtypes = [u64, i64, vp]
        for f in (lib.synth_normal_f32, lib.synth_normal_bf16, lib.synth_uniform_i32,
                  lib.synth_uniform_f64, lib.synth_raw_u64, lib.synth_splitmix64_seq):
            f.restype = None
        _lib_handle = lib
    return _lib_handle


# ---------------------------------------------------------------- primitives

def normal(seed, stream, shape, mean=0.0, std=1.0, dtype="bf16", offset=0):
    """N(mean, std) samples; dtype "bf16" returns uint16 bit patterns."""
    n = int(np.prod(shape))
    if dtype == "bf16":
        out = np.empty(n, dtype=np.uint16)
        _lib().synth_normal_bf16(seed, stream, offset, n, mean, std, out.ctypes.data)
    else:
        out = np.empty(n, dtype=np.float32)
        _lib().synth_normal_f32(seed, stream, offset, n, mean, std, out.ctypes.data)
    return out.reshape(shape)


def uniform_int(seed, stream, shape, lo, hi, offset=0):
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.int32)
    _lib().synth_uniform_i32(seed, stream, offset, n, int(lo), int(hi), out.ctypes.data)
    return out.reshape(shape)


def uniform01(seed, stream, shape, offset=0):
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float64)
    _lib().synth_uniform_f64(seed, stream, offset, n, out.ctypes.data)
    return out.reshape(shape)


def raw_u64(seed, stream, n, offset=0):
    out = np.empty(n, dtype=np.uint64)
    _lib().synth_raw_u64(seed, stream, offset, n, out.ctypes.data)
    return out


def splitmix64_seq(state, n):
    out = np.empty(n, dtype=np.uint64)
    _lib().synth_splitmix64_seq(state, n, out.ctypes.data)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


# ------------------------------------------------------------------- configs

@dataclass(frozen=True)
class MTPShape:
    """Shape of an MTP head and of one draft/verify workload."""
    name: str
    H: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int
    batch: int
    K: int
    dtype: str                 # "f32" or "bf16": weights, KV, hidden, target logits
    ctx_lo: int                # committed MTP context per request: uniform in
    ctx_hi: int                # [ctx_lo, ctx_hi] (equal for fixed length)
    eps: float = 1e-6
    rope_theta: float = 1e6
    block_size: int = 16
    paged_shuffle: bool = False  # blocks of the pool in seeded random order
    k_lo: int = 0              # per-request draft counts for verify-only
    k_hi: int = 0              # workloads (0: use K for every request)
    seed_index: int = 0

    @property
    def q_dim(self):
        return self.n_q * self.head_dim

    @property
    def kv_dim(self):
        return self.n_kv * self.head_dim

    @property
    def seed(self):
        return BASE_SEED + self.seed_index

    @property
    def elem_bytes(self):
        return 4 if self.dtype == "f32" else 2

    def weight_shapes(self) -> Dict[str, tuple]:
        H, F, V = self.H, self.ffn, self.vocab
        return {
            "w_norm_h": (H,), "w_norm_e": (H,), "w_eh": (H, 2 * H),
            "w_norm_in": (H,), "w_q": (self.q_dim, H), "w_k": (self.kv_dim, H),
            "w_v": (self.kv_dim, H), "w_o": (H, self.q_dim),
            "w_norm_post": (H,), "w_gate": (F, H), "w_up": (F, H), "w_down": (H, F),
            "w_norm_f": (H,), "embed": (V, H),
        }

    def weight_bytes(self) -> int:
        """Bytes of all weights read once per draft step (tied LM head = embed)."""
        return sum(int(np.prod(s)) for s in self.weight_shapes().values()) * self.elem_bytes


# The five workloads.  Sizes follow the recipe text; names say what they are.
TINY_F32 = MTPShape("tiny_f32_h256", H=256, n_q=4, n_kv=2, head_dim=64, ffn=1024, vocab=4096,
                    batch=1, K=3, dtype="f32", ctx_lo=128, ctx_hi=128, seed_index=1)
QWEN3_8B_B1 = MTPShape("qwen3_8b_mtp_b1", H=4096, n_q=32, n_kv=8, head_dim=128, ffn=12288,
                       vocab=151936, batch=1, K=5, dtype="bf16", ctx_lo=4096, ctx_hi=4096,
                       seed_index=2)
QWEN3_8B_CB32 = MTPShape("qwen3_8b_mtp_cb32", H=4096, n_q=32, n_kv=8, head_dim=128, ffn=12288,
                         vocab=151936, batch=32, K=5, dtype="bf16", ctx_lo=512, ctx_hi=8192,
                         paged_shuffle=True, seed_index=3)
VERIFY_B64 = MTPShape("verify_rollback_b64", H=0, n_q=8, n_kv=8, head_dim=128, ffn=0,
                      vocab=151936, batch=64, K=8, dtype="bf16", ctx_lo=2048, ctx_hi=2048,
                      k_lo=1, k_hi=8, seed_index=4)
QWEN3_32B_B128 = MTPShape("qwen3_32b_mtp_b128", H=5120, n_q=64, n_kv=8, head_dim=128, ffn=25600,
                          vocab=151936, batch=128, K=3, dtype="bf16", ctx_lo=16384,
                          ctx_hi=16384, seed_index=5)

CONFIGS = [TINY_F32, QWEN3_8B_B1, QWEN3_8B_CB32, VERIFY_B64, QWEN3_32B_B128]

# Tensor ids (the "stream" argument of the generator), fixed once.
_STREAM = {
    "w_norm_h": 1, "w_norm_e": 2, "w_eh": 3, "w_norm_in": 4, "w_q": 5, "w_k": 6, "w_v": 7,
    "w_o": 8, "w_norm_post": 9, "w_gate": 10, "w_up": 11, "w_down": 12, "w_norm_f": 13,
    "embed": 14, "hidden": 20, "token_ids": 21, "ctx_len": 22, "block_perm": 23,
    "k_pool": 24, "v_pool": 25, "verify_logits": 30, "spike_ids": 31, "accept_len": 32,
    "mismatch_ids": 33, "tail_ids": 34, "num_drafts": 35, "spike_noise": 36,
    "loop_hash": 40,
}


def stream_id(name: str) -> int:
    return _STREAM[name]


def _gen(cfg: MTPShape, name: str, shape, mean=0.0, std=1.0, seed=None):
    return normal(cfg.seed if seed is None else seed, _STREAM[name], shape, mean, std,
                  dtype=cfg.dtype)


def make_weights(cfg: MTPShape, norm: str = "ones", seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """All head weights.  bf16 configs return uint16 bit patterns, f32 float32."""
    out = {}
    for name, shape in cfg.weight_shapes().items():
        if name.startswith("w_norm"):
            if norm == "ones":
                arr = np.ones(shape, dtype=np.float32)
                out[name] = f32_to_bf16_bits(arr) if cfg.dtype == "bf16" else arr
            else:
                out[name] = _gen(cfg, name, shape, 1.0, 0.1, seed)
        else:
            out[name] = _gen(cfg, name, shape, 0.0, 0.02, seed)
    return out


@dataclass
class KVState:
    """Paged single-layer MTP KV cache (host copy).

    k_pool, v_pool: [num_blocks, n_kv, block_size, head_dim] (uint16 bf16 bits
    or float32); block_table: [B, max_blocks] int32; seq_len, pending: [B] int32.
    """
    k_pool: np.ndarray
    v_pool: np.ndarray
    block_table: np.ndarray
    seq_len: np.ndarray
    pending: np.ndarray
    block_size: int = 16

    def copy(self) -> "KVState":
        return KVState(self.k_pool.copy(), self.v_pool.copy(), self.block_table.copy(),
                       self.seq_len.copy(), self.pending.copy(), self.block_size)


def context_lengths(cfg: MTPShape, batch: Optional[int] = None) -> np.ndarray:
    B = cfg.batch if batch is None else batch
    if cfg.ctx_lo == cfg.ctx_hi:
        return np.full(B, cfg.ctx_lo, dtype=np.int32)
    return uniform_int(cfg.seed, _STREAM["ctx_len"], (B,), cfg.ctx_lo, cfg.ctx_hi + 1)


def make_kv(cfg: MTPShape, lens: np.ndarray, extra_slots: int, prefill_slots: Optional[np.ndarray] = None,
            seed: Optional[int] = None) -> KVState:
    """Paged pools holding ``prefill_slots[b]`` (default ``lens[b]``) N(0,1)
    entries per request and room for ``extra_slots`` more; every other slot is
    zero.  With ``paged_shuffle`` the pool blocks are assigned in a seeded
    random order."""
    bs = cfg.block_size
    B = len(lens)
    if prefill_slots is None:
        prefill_slots = lens
    need = [(int(l) + extra_slots + bs - 1) // bs for l in lens]
    max_blocks = max(need)
    nblk = int(sum(need))
    order = np.arange(nblk, dtype=np.int64)
    if cfg.paged_shuffle:
        keys = uniform01(cfg.seed if seed is None else seed, _STREAM["block_perm"], (nblk,))
        order = np.argsort(keys, kind="stable")
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        table[b, :need[b]] = order[pos:pos + need[b]]
        pos += need[b]
    shape = (nblk, cfg.n_kv, bs, cfg.head_dim)
    dt = np.uint16 if cfg.dtype == "bf16" else np.float32
    k_pool = np.zeros(shape, dtype=dt)
    v_pool = np.zeros(shape, dtype=dt)
    s = cfg.seed if seed is None else seed
    row = cfg.n_kv * cfg.head_dim
    # Entries are drawn per (request, slot) so that any request can be
    # regenerated alone: element index = (b * 2^24 + slot) * row + j.
    for b in range(B):
        L = int(prefill_slots[b])
        if L == 0:
            continue
        base = (b << 24) * row
        kv_k = normal(s, _STREAM["k_pool"], (L, cfg.n_kv, cfg.head_dim), dtype=cfg.dtype, offset=base)
        kv_v = normal(s, _STREAM["v_pool"], (L, cfg.n_kv, cfg.head_dim), dtype=cfg.dtype, offset=base)
        nfull = L // bs
        blocks = table[b, :nfull]
        if nfull:
            k_pool[blocks] = kv_k[:nfull * bs].reshape(nfull, bs, cfg.n_kv, cfg.head_dim).transpose(0, 2, 1, 3)
            v_pool[blocks] = kv_v[:nfull * bs].reshape(nfull, bs, cfg.n_kv, cfg.head_dim).transpose(0, 2, 1, 3)
        rem = L - nfull * bs
        if rem:
            blk = table[b, nfull]
            k_pool[blk, :, :rem] = kv_k[nfull * bs:].transpose(1, 0, 2)
            v_pool[blk, :, :rem] = kv_v[nfull * bs:].transpose(1, 0, 2)
    return KVState(k_pool, v_pool, table, np.asarray(lens, dtype=np.int32).copy(),
                   np.zeros(B, dtype=np.int32), bs)


@dataclass
class DraftInputs:
    hidden: np.ndarray      # [B, H] (bf16 bits or f32)
    token_ids: np.ndarray   # [B] int32, the tokens whose embeddings are given
    embeds: np.ndarray      # [B, H] rows of the embedding table at token_ids
    positions: np.ndarray   # [B] int32


def make_draft_inputs(cfg: MTPShape, weights: Dict[str, np.ndarray], lens: np.ndarray,
                      seed: Optional[int] = None) -> DraftInputs:
    B = len(lens)
    s = cfg.seed if seed is None else seed
    hidden = normal(s, _STREAM["hidden"], (B, cfg.H), 0.0, 1.0, dtype=cfg.dtype)
    ids = uniform_int(s, _STREAM["token_ids"], (B,), 0, cfg.vocab)
    embeds = weights["embed"][ids].copy()
    positions = np.asarray(lens, dtype=np.int32).copy()
    return DraftInputs(hidden, ids, embeds, positions)


@dataclass
class VerifyInputs:
    logits: np.ndarray       # [R, V] rows (bf16 bits or f32), R = sum(num_drafts + 1)
    row_offsets: np.ndarray  # [B + 1] int32
    drafts: np.ndarray       # [B, max_k] int32 (entries past num_drafts[b] are -1)
    num_drafts: np.ndarray   # [B] int32
    planted: np.ndarray      # [R] int32, id carrying the +8 spike in each row
    accept_len: np.ndarray   # [B] int32, length of the copied prefix
    max_k: int


def geometric_len(u: np.ndarray, alpha: float) -> np.ndarray:
    """n with P(n) = (1 - alpha) alpha^n, by inversion: floor(ln u / ln alpha), u in (0, 1]."""
    return np.floor(np.log(u) / math.log(alpha)).astype(np.int64)


def make_verify_inputs(cfg: MTPShape, num_drafts: Optional[np.ndarray] = None, alpha: float = 0.8,
                       spike: float = 8.0, planted_ids: Optional[np.ndarray] = None,
                       seed: Optional[int] = None, len_mode: str = "geometric") -> VerifyInputs:
    """Target logits for verification with a known accepted prefix.

    Row j of request b holds N(0,1) values plus ``spike`` at id planted[b,j].
    Drafts copy planted[b, j] for j < n_b, then a different id at j = n_b,
    then uniform ids.  n_b is geometric(alpha) truncated at K_b
    (``len_mode="geometric"``) or uniform over 0..K_b (``"uniform"``).
    ``planted_ids`` ([B, max_k+1]) fixes the spike ids (e.g. to a run's own
    drafts); otherwise they are uniform."""
    s = cfg.seed if seed is None else seed
    B, V = cfg.batch, cfg.vocab
    if num_drafts is None:
        if cfg.k_hi > 0:
            num_drafts = uniform_int(s, _STREAM["num_drafts"], (B,), cfg.k_lo, cfg.k_hi + 1)
        else:
            num_drafts = np.full(B, cfg.K, dtype=np.int32)
    num_drafts = np.asarray(num_drafts, dtype=np.int32)
    max_k = int(max(cfg.K, num_drafts.max()))
    rows = num_drafts + 1
    row_offsets = np.zeros(B + 1, dtype=np.int32)
    row_offsets[1:] = np.cumsum(rows)
    R = int(row_offsets[-1])
    if planted_ids is None:
        planted_full = uniform_int(s, _STREAM["spike_ids"], (B, max_k + 1), 0, V)
    else:
        planted_full = np.asarray(planted_ids, dtype=np.int32)
    if len_mode == "geometric":
        u = 1.0 - uniform01(s, _STREAM["accept_len"], (B,))       # (0, 1]
        n = np.minimum(geometric_len(u, alpha), num_drafts).astype(np.int32)
    else:
        n = (uniform01(s, _STREAM["accept_len"], (B,)) * (num_drafts + 1)).astype(np.int32)
    mism = uniform_int(s, _STREAM["mismatch_ids"], (B,), 0, V - 1)
    tail = uniform_int(s, _STREAM["tail_ids"], (B, max_k), 0, V)
    drafts = np.full((B, max_k), -1, dtype=np.int32)
    planted = np.empty(R, dtype=np.int32)
    for b in range(B):
        K_b = int(num_drafts[b])
        planted[row_offsets[b]:row_offsets[b + 1]] = planted_full[b, :K_b + 1]
        for j in range(K_b):
            if j < n[b]:
                drafts[b, j] = planted_full[b, j]
            elif j == n[b]:
                m = int(mism[b])
                drafts[b, j] = m + 1 if m >= planted_full[b, j] else m
            else:
                drafts[b, j] = tail[b, j]
    # N(0,1) rows generated in float32, spike added, then rounded to the dtype.
    noise = normal(s, _STREAM["verify_logits"], (R, V), dtype="f32")
    noise[np.arange(R), planted] += np.float32(spike)
    logits = f32_to_bf16_bits(noise) if cfg.dtype == "bf16" else noise
    return VerifyInputs(logits, row_offsets, drafts, num_drafts, planted, n, max_k)


def expected_accept_len(K: int, alpha: float) -> float:
    """E[min(G, K)] for G geometric with P(G >= n) = alpha^n."""
    return sum(alpha ** n for n in range(1, K + 1))


def shrink(cfg: MTPShape, **kw) -> MTPShape:
    return replace(cfg, **kw)


# ------------------------------------------------------- speculative loop

def copy_head(cfg: MTPShape, w: Dict[str, np.ndarray], residual_scale: float = 0.01) -> Dict[str, np.ndarray]:
    """A head whose drafts repeat their input token: eh_proj = [0 | I] (the
    projection passes the normalised embedding through), o_proj and down_proj
    scaled by ``residual_scale`` (the layer still runs, but adds little), so
    the tied LM head's self-dot of the input row wins.  Used to give the
    speculative-loop tests drafts that a sticky synthetic verifier accepts."""
    H = cfg.H
    out = dict(w)
    eh = np.concatenate([np.zeros((H, H), dtype=np.float32), np.eye(H, dtype=np.float32)], axis=1)

    def conv(x):
        return f32_to_bf16_bits(x) if cfg.dtype == "bf16" else x.astype(np.float32)

    def scaled(name):
        x = bf16_to_f32(w[name]) if cfg.dtype == "bf16" else w[name].astype(np.float32)
        return conv(x * np.float32(residual_scale))

    out["w_eh"] = conv(eh)
    out["w_o"] = scaled("w_o")
    out["w_down"] = scaled("w_down")
    return out


def loop_start_hashes(cfg: MTPShape, B: int) -> np.ndarray:
    """Seeded 64-bit hashes standing for each request's prompt (the
    synthetic verifier's state at the start of the loop)."""
    return raw_u64(cfg.seed, _STREAM["loop_hash"], B)
