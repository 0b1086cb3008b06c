"""MTP self-speculative draft-and-verify step on one GB300 (sm_103a).

A thin binding over the C ABI of ``libmtp.so`` (declared in include/mtp.h):
the functions below carry the C names and only marshal arguments -- torch
tensors become device pointers, torch streams become cudaStream_t handles.
Every step of the method runs in the library's CUDA kernels; PyTorch is used
for device memory and streams only.  There is no CPU path: if the library is
missing, importing the binding raises.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Dict, Optional

import torch

from . import _lib as L
from ._lib import (  # noqa: F401
    KERNEL_NAMES, MTP_DTYPE_BF16, MTP_DTYPE_F32, MTP_ERR_BOUNDS, MTP_ERR_CAPACITY, MTP_ERR_CUDA, MTP_ERR_DEVICE_ARGS,
    MTP_ERR_INVALID, MTP_ERR_OOM, MTP_ERR_TIMEOUT, MTP_KERNEL_ATTENTION, MTP_KERNEL_DOWN, MTP_KERNEL_EH_PROJ,
    MTP_KERNEL_GATE_UP, MTP_KERNEL_KV_EDIT, MTP_KERNEL_LM_HEAD, MTP_KERNEL_O_PROJ, MTP_KERNEL_QKV_ROPE,
    MTP_KERNEL_VERIFY, MTP_KERNEL_DRAFT_PERSISTENT, MTP_OK, MTP_WEIGHTS_DENSE, MTP_WEIGHTS_INT4_G64, MTPConfig, MTPKV,
    MTPLoop, MTPTree, MTPWeights, WEIGHT_FIELDS,
)

_clib = L.load()


class MTPError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (%d)" % (where, _clib.mtp_status_str(status).decode(), status))


def _check(status: int, where: str) -> None:
    if status != MTP_OK:
        raise MTPError(status, where)


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def torch_dtype(dtype_code: int) -> torch.dtype:
    return torch.bfloat16 if dtype_code == MTP_DTYPE_BF16 else torch.float32


@dataclass
class KVCache:
    """Caller-owned paged MTP KV cache (device tensors)."""
    k_pool: torch.Tensor        # [num_blocks, n_kv, block_size, head_dim]
    v_pool: torch.Tensor
    block_table: torch.Tensor   # [B, max_blocks] int32
    seq_len: torch.Tensor       # [B] int32
    pending: torch.Tensor       # [B] int32

    def struct(self) -> MTPKV:
        return MTPKV(_ptr(self.k_pool, name="k_pool"), _ptr(self.v_pool, name="v_pool"),
                     _ptr(self.block_table, torch.int32, "block_table"), _ptr(self.seq_len, torch.int32, "seq_len"),
                     _ptr(self.pending, torch.int32, "pending"), int(self.k_pool.shape[0]),
                     int(self.block_table.shape[1]))


class Context:
    """Owns an mtp_ctx handle and keeps the borrowed weight tensors alive."""

    def __init__(self, handle: int, cfg: MTPConfig, weights: Optional[Dict[str, torch.Tensor]]):
        self.handle = handle
        self.cfg = cfg
        self.weights = weights

    def close(self):
        if self.handle:
            _clib.mtp_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def make_config(hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab, eps=1e-6, rope_theta=1e6, dtype="bf16",
                max_batch=1, max_k=5, block_size=16, max_pos=32768, tc_min_batch=0,
                persistent_max_batch=0, weight_format="dense") -> MTPConfig:
    code = MTP_DTYPE_BF16 if dtype in ("bf16", MTP_DTYPE_BF16, torch.bfloat16) else MTP_DTYPE_F32
    wf = MTP_WEIGHTS_INT4_G64 if weight_format in ("int4_g64", MTP_WEIGHTS_INT4_G64) else MTP_WEIGHTS_DENSE
    return MTPConfig(hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab, eps, rope_theta, code, max_batch, max_k,
                     block_size, max_pos, tc_min_batch, persistent_max_batch, wf)


def mtp_init(cfg: MTPConfig, weights: Optional[Dict[str, torch.Tensor]] = None, device: Optional[int] = None
             ) -> Context:
    """Create a context.  ``weights`` maps the mtp_weights field names to
    device tensors (``lm_head`` optional: tied to ``embed``); None for a
    verify/KV-only context."""
    if device is None:
        device = torch.cuda.current_device()
    wst = None
    if weights is not None:
        dt = torch_dtype(cfg.dtype)
        wst = MTPWeights(*[_ptr(weights.get(n), dt, n) if weights.get(n) is not None else None
                           for n in WEIGHT_FIELDS])
    out = ctypes.c_void_p()
    _check(_clib.mtp_init(ctypes.byref(cfg), ctypes.byref(wst) if wst is not None else None, int(device),
                         ctypes.byref(out)), "mtp_init")
    return Context(out.value, cfg, weights)


def mtp_draft(ctx: Context, hidden: torch.Tensor, embeds: torch.Tensor, positions: torch.Tensor, kv: KVCache, K: int,
              draft_ids: torch.Tensor, logits: Optional[torch.Tensor] = None, hidden_out: Optional[torch.Tensor] = None,
              chain_ids: Optional[torch.Tensor] = None, stream=None) -> None:
    dt = torch_dtype(ctx.cfg.dtype)
    B = int(hidden.shape[0])
    kvs = kv.struct()
    _check(_clib.mtp_draft(ctx.handle, _stream(stream), B, _ptr(hidden, dt, "hidden"), _ptr(embeds, dt, "embeds"),
                          _ptr(positions, torch.int32, "positions"), ctypes.byref(kvs), int(K),
                          _ptr(chain_ids, torch.int32, "chain_ids"), _ptr(draft_ids, torch.int32, "draft_ids"),
                          _ptr(logits, torch.float32, "logits"), _ptr(hidden_out, torch.float32, "hidden_out")),
           "mtp_draft")


def _check_verify_shapes(target_logits: torch.Tensor, row_offsets: torch.Tensor, drafts: torch.Tensor,
                         num_drafts: torch.Tensor, accepted: torch.Tensor, bonus: torch.Tensor, vocab: int,
                         where: str) -> int:
    """Shape checks the C entry points cannot make (they receive plain
    pointers): the kernel reads num_rows x vocab logits and B + 1 offsets and
    writes B results, so a mismatch here would read or write past a buffer.
    Returns B."""
    if target_logits.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("%s: target_logits must be float32 or bfloat16, got %s" % (where, target_logits.dtype))
    if target_logits.dim() != 2 or int(target_logits.shape[1]) != int(vocab) or int(target_logits.shape[0]) < 1:
        raise ValueError("%s: target_logits must be [num_rows >= 1, vocab=%d], got %s"
                         % (where, vocab, tuple(target_logits.shape)))
    if num_drafts.dim() != 1:
        raise ValueError("%s: num_drafts must be 1-D [B]" % where)
    B = int(num_drafts.shape[0])
    if row_offsets.dim() != 1 or int(row_offsets.shape[0]) != B + 1:
        raise ValueError("%s: row_offsets must be [B + 1] = [%d], got %s" % (where, B + 1, tuple(row_offsets.shape)))
    if drafts.dim() != 2 or int(drafts.shape[0]) != B:
        raise ValueError("%s: drafts must be [B=%d, stride], got %s" % (where, B, tuple(drafts.shape)))
    for t, name in ((accepted, "accepted"), (bonus, "bonus")):
        if t.numel() != B:
            raise ValueError("%s: %s must hold B=%d entries, got %d" % (where, name, B, t.numel()))
    return B


def mtp_verify(ctx: Context, target_logits: torch.Tensor, row_offsets: torch.Tensor, drafts: torch.Tensor,
               num_drafts: torch.Tensor, accepted: torch.Tensor, bonus: torch.Tensor, stream=None) -> None:
    dt = torch_dtype(ctx.cfg.dtype)
    B = _check_verify_shapes(target_logits, row_offsets, drafts, num_drafts, accepted, bonus, ctx.cfg.vocab,
                             "mtp_verify")
    _check(_clib.mtp_verify(ctx.handle, _stream(stream), B, _ptr(target_logits, dt, "target_logits"),
                           int(target_logits.shape[0]), _ptr(row_offsets, torch.int32, "row_offsets"), _ptr(drafts, torch.int32, "drafts"),
                           int(drafts.shape[1]), _ptr(num_drafts, torch.int32, "num_drafts"),
                           _ptr(accepted, torch.int32, "accepted"), _ptr(bonus, torch.int32, "bonus")), "mtp_verify")


def mtp_verify_noalloc(target_logits: torch.Tensor, row_offsets: torch.Tensor, drafts: torch.Tensor,
                       num_drafts: torch.Tensor, accepted: torch.Tensor, bonus: torch.Tensor, vocab: int,
                       max_k: int, stream=None) -> None:
    """mtp_verify without a context and without any device allocation (for
    callers whose device memory is owned by a fixed plan or another pool, or
    who cannot take cudaMalloc's device-wide synchronisation); the shape is
    passed directly and the scratch is the library's fixed device array.
    target_logits must be float32 or bfloat16 [num_rows, vocab]; the shape
    checks run before anything reaches the library."""
    B = _check_verify_shapes(target_logits, row_offsets, drafts, num_drafts, accepted, bonus, vocab,
                             "mtp_verify_noalloc")
    code = MTP_DTYPE_BF16 if target_logits.dtype == torch.bfloat16 else MTP_DTYPE_F32
    _check(_clib.mtp_verify_noalloc(_stream(stream), B, int(vocab), code, int(max_k),
                                    _ptr(target_logits, name="target_logits"), int(target_logits.shape[0]),
                                    _ptr(row_offsets, torch.int32, "row_offsets"), _ptr(drafts, torch.int32, "drafts"),
                                    int(drafts.shape[1]), _ptr(num_drafts, torch.int32, "num_drafts"),
                                    _ptr(accepted, torch.int32, "accepted"), _ptr(bonus, torch.int32, "bonus")),
           "mtp_verify_noalloc")


# ------------------------------------------------ speculative loop harness

def mtp_synth_target(ctx: Context, seq_hash: torch.Tensor, last_tok: torch.Tensor, drafts: Optional[torch.Tensor],
                     K: int, sticky_thr: int, logits: torch.Tensor, row_offsets: Optional[torch.Tensor] = None,
                     num_drafts: Optional[torch.Tensor] = None, stream=None) -> None:
    """Synthetic verifier rows (include/mtp.h): seq_hash is an int64 tensor
    holding the 64-bit prefix hashes."""
    B = int(last_tok.shape[0])
    dt = torch_dtype(ctx.cfg.dtype)
    _check(_clib.mtp_synth_target(ctx.handle, _stream(stream), B, int(K), _ptr(num_drafts, torch.int32, "num_drafts"),
                                  _ptr(seq_hash, torch.int64, "seq_hash"),
                                  _ptr(last_tok, torch.int32, "last_tok"), _ptr(drafts, torch.int32, "drafts"),
                                  ctypes.c_uint64(int(sticky_thr)), _ptr(logits, dt, "logits"),
                                  _ptr(row_offsets, torch.int32, "row_offsets")), "mtp_synth_target")


def mtp_loop_advance(ctx: Context, K: int, drafts: Optional[torch.Tensor], accepted: torch.Tensor,
                     bonus: torch.Tensor, seq_hash: torch.Tensor, last_tok: torch.Tensor, positions: torch.Tensor,
                     hidden: torch.Tensor, embeds: torch.Tensor, out_tokens: torch.Tensor, out_len: torch.Tensor,
                     stream=None) -> None:
    B = int(accepted.shape[0])
    dt = torch_dtype(ctx.cfg.dtype)
    _check(_clib.mtp_loop_advance(ctx.handle, _stream(stream), B, int(K), _ptr(drafts, torch.int32, "drafts"),
                                  _ptr(accepted, torch.int32, "accepted"), _ptr(bonus, torch.int32, "bonus"),
                                  _ptr(seq_hash, torch.int64, "seq_hash"), _ptr(last_tok, torch.int32, "last_tok"),
                                  _ptr(positions, torch.int32, "positions"), _ptr(hidden, dt, "hidden"),
                                  _ptr(embeds, dt, "embeds"), _ptr(out_tokens, torch.int32, "out_tokens"),
                                  _ptr(out_len, torch.int32, "out_len"), int(out_tokens.shape[1])),
           "mtp_loop_advance")


def mtp_draft_confidence(ctx: Context, logits: torch.Tensor, tau: float, conf: torch.Tensor,
                         num_drafts: Optional[torch.Tensor] = None, stream=None) -> None:
    """conf [B, K] = probability of each draft step's argmax under logits
    [B, K, V] (fp32); num_drafts [B] = leading run with conf > tau."""
    B, K = int(logits.shape[0]), int(logits.shape[1])
    _check(_clib.mtp_draft_confidence(ctx.handle, _stream(stream), B, K, _ptr(logits, torch.float32, "logits"),
                                      float(tau), _ptr(conf, torch.float32, "conf"),
                                      _ptr(num_drafts, torch.int32, "num_drafts")), "mtp_draft_confidence")


def mtp_adapt_k(K: int, accepted: int, drafted: int, k_min: int, k_max: int) -> int:
    return int(_clib.mtp_adapt_k(int(K), int(accepted), int(drafted), int(k_min), int(k_max)))


class SpecLoop:
    """Device state and scratch of mtp_spec_loop for B requests, K drafts per
    step (K = 0: plain greedy decoding with the verifier), out_cap tokens;
    conf_threshold > 0 proposes only the leading confident drafts."""

    def __init__(self, ctx: Context, B: int, K: int, sticky_thr: int, out_cap: int, device="cuda",
                 conf_threshold: float = 0.0):
        dt = torch_dtype(ctx.cfg.dtype)
        H, V = ctx.cfg.hidden, ctx.cfg.vocab
        i32 = dict(dtype=torch.int32, device=device)
        self.B, self.K, self.sticky_thr = B, K, int(sticky_thr)
        self.seq_hash = torch.zeros(B, dtype=torch.int64, device=device)
        self.last_tok = torch.zeros(B, **i32)
        self.positions = torch.zeros(B, **i32)
        self.hidden = torch.zeros((B, H), dtype=dt, device=device)
        self.embeds = torch.zeros((B, H), dtype=dt, device=device)
        self.drafts = torch.zeros((B, max(K, 1)), **i32)
        self.accepted = torch.zeros(B, **i32)
        self.bonus = torch.zeros(B, **i32)
        self.num_drafts = torch.zeros(B, **i32)
        self.row_offsets = torch.zeros(B + 1, **i32)
        self.target_logits = torch.zeros((B * (K + 1), V), dtype=dt, device=device)
        self.out_tokens = torch.zeros((B, out_cap), **i32)
        self.out_len = torch.zeros(B, **i32)
        self.conf_threshold = float(conf_threshold)
        on = conf_threshold > 0 and K > 0
        self.draft_logits = torch.zeros((B, K, V) if on else (1,), dtype=torch.float32, device=device)
        self.conf = torch.zeros((B, K) if on else (1,), dtype=torch.float32, device=device)

    def struct(self) -> MTPLoop:
        return MTPLoop(self.B, self.K, self.sticky_thr, self.seq_hash.data_ptr(), self.last_tok.data_ptr(),
                       self.positions.data_ptr(), self.hidden.data_ptr(), self.embeds.data_ptr(),
                       self.drafts.data_ptr(), self.accepted.data_ptr(), self.bonus.data_ptr(),
                       self.num_drafts.data_ptr(), self.row_offsets.data_ptr(), self.target_logits.data_ptr(),
                       self.out_tokens.data_ptr(), self.out_len.data_ptr(), int(self.out_tokens.shape[1]),
                       self.conf_threshold, self.draft_logits.data_ptr(), self.conf.data_ptr())


def mtp_spec_loop(ctx: Context, kv: Optional[KVCache], loop: SpecLoop, iters: int, stream=None) -> None:
    st = loop.struct()
    kvs = kv.struct() if kv is not None else None
    _check(_clib.mtp_spec_loop(ctx.handle, _stream(stream), ctypes.byref(kvs) if kvs is not None else None,
                               ctypes.byref(st), int(iters)), "mtp_spec_loop")


class TreeDraft:
    """Buffers of tree drafting for B requests (branching, depth, n_assist);
    ``scratch_blocks`` is an int32 device tensor of free block ids of the cache
    pool ((depth-1) * B * branching * 2 of them)."""

    def __init__(self, ctx: Context, B: int, branching: int, depth: int, n_assist: int, max_blocks: int,
                 scratch_blocks: Optional[torch.Tensor], device="cuda"):
        n = int(_clib.mtp_tree_workspace_bytes(ctx.handle, B, branching, depth, n_assist, max_blocks))
        if n == 0:
            raise MTPError(MTP_ERR_INVALID, "mtp_tree_workspace_bytes")
        self.B, self.branching, self.depth, self.n_assist = B, branching, depth, n_assist
        self.ws = torch.empty(n, dtype=torch.uint8, device=device)
        self.scratch_blocks = scratch_blocks
        i32 = dict(dtype=torch.int32, device=device)
        self.tokens = torch.zeros((B, n_assist), **i32)
        self.parents = torch.zeros((B, n_assist), **i32)
        self.depths = torch.zeros((B, n_assist), **i32)

    def struct(self) -> MTPTree:
        sb = self.scratch_blocks.data_ptr() if self.scratch_blocks is not None else None
        return MTPTree(self.B, self.branching, self.depth, self.n_assist, sb, self.ws.data_ptr(),
                       int(self.ws.numel()), self.tokens.data_ptr(), self.parents.data_ptr(), self.depths.data_ptr())


def mtp_draft_tree(ctx: Context, hidden: torch.Tensor, embeds: torch.Tensor, positions: torch.Tensor, kv: KVCache,
                   tree: TreeDraft, stream=None) -> None:
    dt = torch_dtype(ctx.cfg.dtype)
    kvs, ts = kv.struct(), tree.struct()
    _check(_clib.mtp_draft_tree(ctx.handle, _stream(stream), _ptr(hidden, dt, "hidden"), _ptr(embeds, dt, "embeds"),
                                _ptr(positions, torch.int32, "positions"), ctypes.byref(kvs), ctypes.byref(ts)),
           "mtp_draft_tree")


def mtp_synth_target_tree(ctx: Context, tree: TreeDraft, seq_hash: torch.Tensor, last_tok: torch.Tensor,
                          sticky_thr: int, logits: torch.Tensor, row_offsets: Optional[torch.Tensor] = None,
                          stream=None) -> None:
    ts = tree.struct()
    _check(_clib.mtp_synth_target_tree(ctx.handle, _stream(stream), ctypes.byref(ts),
                                       _ptr(seq_hash, torch.int64, "seq_hash"), _ptr(last_tok, torch.int32, "last_tok"),
                                       ctypes.c_uint64(int(sticky_thr)), _ptr(logits, torch_dtype(ctx.cfg.dtype), "logits"),
                                       _ptr(row_offsets, torch.int32, "row_offsets")), "mtp_synth_target_tree")


def mtp_verify_tree(ctx: Context, tree: TreeDraft, target_logits: torch.Tensor, accepted: torch.Tensor,
                    bonus: torch.Tensor, path_tokens: torch.Tensor, stream=None) -> None:
    ts = tree.struct()
    _check(_clib.mtp_verify_tree(ctx.handle, _stream(stream), ctypes.byref(ts),
                                 _ptr(target_logits, torch_dtype(ctx.cfg.dtype), "target_logits"),
                                 _ptr(accepted, torch.int32, "accepted"), _ptr(bonus, torch.int32, "bonus"),
                                 _ptr(path_tokens, torch.int32, "path_tokens")), "mtp_verify_tree")


def mtp_tree_commit(ctx: Context, kv: KVCache, tree: TreeDraft, accepted: torch.Tensor, stream=None) -> None:
    kvs, ts = kv.struct(), tree.struct()
    _check(_clib.mtp_tree_commit(ctx.handle, _stream(stream), ctypes.byref(kvs), ctypes.byref(ts),
                                 _ptr(accepted, torch.int32, "accepted")), "mtp_tree_commit")


def mtp_tree_loop(ctx: Context, kv: KVCache, loop: SpecLoop, tree: TreeDraft, iters: int, stream=None) -> None:
    kvs, ls, ts = kv.struct(), loop.struct(), tree.struct()
    _check(_clib.mtp_tree_loop(ctx.handle, _stream(stream), ctypes.byref(kvs), ctypes.byref(ls), ctypes.byref(ts),
                               int(iters)), "mtp_tree_loop")


def mtp_quantize_int4_g64(w: torch.Tensor, q: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor,
                          stream=None) -> None:
    """INT4 asymmetric group-64 quantization of a bf16 matrix [rows, cols]:
    q [rows, cols/2] uint8, scales [rows, cols/64] fp16 (or int16 bits),
    zeros [rows, cols/64] uint8."""
    rows, cols = int(w.shape[0]), int(w.shape[1])
    _check(_clib.mtp_quantize_int4_g64(_stream(stream), _ptr(w, name="w"), rows, cols, _ptr(q, name="q"),
                                       _ptr(scales, name="scales"), _ptr(zeros, name="zeros")),
           "mtp_quantize_int4_g64")


def mtp_quantize_int8_rows(w: torch.Tensor, q: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    """INT8 symmetric per-row quantization of a bf16 matrix [rows, cols]:
    q [rows, cols] int8, scales [rows] fp16 (or int16 bits)."""
    rows, cols = int(w.shape[0]), int(w.shape[1])
    _check(_clib.mtp_quantize_int8_rows(_stream(stream), _ptr(w, name="w"), rows, cols, _ptr(q, name="q"),
                                        _ptr(scales, name="scales")), "mtp_quantize_int8_rows")


def mtp_kv_commit(ctx: Context, kv: KVCache, n_keep: torch.Tensor, stream=None) -> None:
    kvs = kv.struct()
    _check(_clib.mtp_kv_commit(ctx.handle, _stream(stream), int(kv.seq_len.shape[0]), ctypes.byref(kvs),
                              _ptr(n_keep, torch.int32, "n_keep")), "mtp_kv_commit")


def mtp_kv_commit_accepted(ctx: Context, kv: KVCache, accepted: torch.Tensor, extra: int = 1, stream=None) -> None:
    kvs = kv.struct()
    _check(_clib.mtp_kv_commit_accepted(ctx.handle, _stream(stream), int(kv.seq_len.shape[0]), ctypes.byref(kvs),
                                       _ptr(accepted, torch.int32, "accepted"), int(extra)), "mtp_kv_commit_accepted")


def mtp_kv_rollback(ctx: Context, kv: KVCache, stream=None) -> None:
    kvs = kv.struct()
    _check(_clib.mtp_kv_rollback(ctx.handle, _stream(stream), int(kv.seq_len.shape[0]), ctypes.byref(kvs)),
           "mtp_kv_rollback")


def mtp_kv_truncate(ctx: Context, kv: KVCache, new_len: torch.Tensor, stream=None) -> None:
    kvs = kv.struct()
    _check(_clib.mtp_kv_truncate(ctx.handle, _stream(stream), int(kv.seq_len.shape[0]), ctypes.byref(kvs),
                                _ptr(new_len, torch.int32, "new_len")), "mtp_kv_truncate")


def mtp_selftest_wait_timeout(ctx: Context, which: int, stream=None) -> None:
    _check(_clib.mtp_selftest_wait_timeout(ctx.handle, _stream(stream), int(which)), "mtp_selftest_wait_timeout")


def mtp_selftest_bounds(ctx: Context, stream=None) -> None:
    _check(_clib.mtp_selftest_bounds(ctx.handle, _stream(stream)), "mtp_selftest_bounds")


def mtp_get_device_error(ctx: Context) -> int:
    return int(_clib.mtp_get_device_error(ctx.handle))


def mtp_destroy(ctx: Context) -> None:
    ctx.close()


def mtp_status_str(status: int) -> str:
    return _clib.mtp_status_str(int(status)).decode()


def mtp_stream_copy(dst: torch.Tensor, src: torch.Tensor, nbytes: Optional[int] = None, stream=None) -> None:
    n = src.numel() * src.element_size() if nbytes is None else nbytes
    _check(_clib.mtp_stream_copy(_stream(stream), _ptr(dst, name="dst"), _ptr(src, name="src"), n),
           "mtp_stream_copy")


def mtp_stream_read(src: torch.Tensor, nbytes: Optional[int] = None, err_word: Optional[torch.Tensor] = None,
                    stream=None) -> None:
    n = src.numel() * src.element_size() if nbytes is None else nbytes
    _check(_clib.mtp_stream_read(_stream(stream), _ptr(src, name="src"), n, _ptr(err_word, torch.int32, "err_word")),
           "mtp_stream_read")


def mtp_profile_begin(ctx: Context, kernel: int, capacity: int) -> None:
    _check(_clib.mtp_profile_begin(ctx.handle, int(kernel), int(capacity)), "mtp_profile_begin")


def mtp_profile_end(ctx: Context, max_out: int = 1 << 16):
    buf = (ctypes.c_float * max_out)()
    n = ctypes.c_int(0)
    _check(_clib.mtp_profile_end(ctx.handle, buf, max_out, ctypes.byref(n)), "mtp_profile_end")
    return [float(buf[i]) for i in range(n.value)]


def mtp_launch_count(ctx: Context) -> int:
    return int(_clib.mtp_launch_count(ctx.handle))


MTP_PATH_LM_DEFERRED = 0
MTP_PATH_ATTN_CLUSTER = 1


def mtp_path_count(ctx: Context, path: int) -> int:
    """How often the context took launch-time path `path` (include/mtp.h)."""
    return int(_clib.mtp_path_count(ctx.handle, int(path)))
