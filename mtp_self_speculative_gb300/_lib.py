"""ctypes declarations of the C ABI in include/mtp.h.

Loading fails loudly when libmtp.so is missing: there is no other
implementation to fall back to."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# MTP_LIBRARY may name another build of the same library (the bounds-checked
# libmtp_checked.so); the default is the in-tree libmtp.so.
LIB_PATH = os.environ.get("MTP_LIBRARY") or os.path.join(HERE, "libmtp.so")

c_int, c_float, c_void_p, c_size_t = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
c_int64 = ctypes.c_int64
P_i32 = ctypes.c_void_p  # device int32 pointers are passed as plain addresses

(MTP_OK, MTP_ERR_INVALID, MTP_ERR_CUDA, MTP_ERR_OOM, MTP_ERR_CAPACITY, MTP_ERR_TIMEOUT, MTP_ERR_DEVICE_ARGS,
 MTP_ERR_BOUNDS) = range(8)
MTP_DTYPE_F32, MTP_DTYPE_BF16 = 0, 1
MTP_WEIGHTS_DENSE, MTP_WEIGHTS_INT4_G64 = 0, 1
(MTP_KERNEL_EH_PROJ, MTP_KERNEL_QKV_ROPE, MTP_KERNEL_ATTENTION, MTP_KERNEL_O_PROJ, MTP_KERNEL_GATE_UP,
 MTP_KERNEL_DOWN, MTP_KERNEL_LM_HEAD, MTP_KERNEL_VERIFY, MTP_KERNEL_KV_EDIT, MTP_KERNEL_DRAFT_PERSISTENT,
 MTP_KERNEL_COUNT) = range(11)
KERNEL_NAMES = ["eh_proj", "qkv_rope", "attention", "o_proj", "gate_up", "down", "lm_head", "verify", "kv_edit",
                "draft_persistent"]


class MTPConfig(ctypes.Structure):
    _fields_ = [("hidden", c_int), ("n_q_heads", c_int), ("n_kv_heads", c_int), ("head_dim", c_int),
                ("ffn", c_int), ("vocab", c_int), ("eps", c_float), ("rope_theta", c_float), ("dtype", c_int),
                ("max_batch", c_int), ("max_k", c_int), ("block_size", c_int), ("max_pos", c_int),
                ("tc_min_batch", c_int), ("persistent_max_batch", c_int), ("weight_format", c_int)]


WEIGHT_FIELDS = ["w_norm_h", "w_norm_e", "w_eh", "w_norm_in", "w_q", "w_k", "w_v", "w_o", "w_norm_post",
                 "w_gate", "w_up", "w_down", "w_norm_f", "embed", "lm_head"]


class MTPWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in WEIGHT_FIELDS]


class MTPKV(ctypes.Structure):
    _fields_ = [("k_pool", c_void_p), ("v_pool", c_void_p), ("block_table", c_void_p), ("seq_len", c_void_p),
                ("pending", c_void_p), ("num_blocks", c_int), ("max_blocks", c_int)]


class MTPLoop(ctypes.Structure):
    _fields_ = [("B", c_int), ("K", c_int), ("sticky_thr", ctypes.c_uint64), ("seq_hash", c_void_p),
                ("last_tok", c_void_p), ("positions", c_void_p), ("hidden", c_void_p), ("embeds", c_void_p),
                ("drafts", c_void_p), ("accepted", c_void_p), ("bonus", c_void_p), ("num_drafts", c_void_p),
                ("row_offsets", c_void_p), ("target_logits", c_void_p), ("out_tokens", c_void_p),
                ("out_len", c_void_p), ("out_cap", c_int), ("conf_threshold", c_float), ("draft_logits", c_void_p),
                ("conf", c_void_p)]


class MTPTree(ctypes.Structure):
    _fields_ = [("B", c_int), ("branching", c_int), ("depth", c_int), ("n_assist", c_int),
                ("scratch_blocks", c_void_p), ("ws", c_void_p), ("ws_bytes", c_size_t), ("tokens", c_void_p),
                ("parents", c_void_p), ("depths", c_void_p)]


# name -> (restype, argtypes); every symbol declared in include/mtp.h
SIGNATURES = {
    "mtp_init": (c_int, [ctypes.POINTER(MTPConfig), ctypes.POINTER(MTPWeights), c_int, ctypes.POINTER(c_void_p)]),
    "mtp_draft": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_void_p, P_i32, ctypes.POINTER(MTPKV), c_int,
                          P_i32, P_i32, c_void_p, c_void_p]),
    "mtp_verify": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int, P_i32, P_i32, c_int, P_i32, P_i32, P_i32]),
    "mtp_verify_noalloc": (c_int, [c_void_p, c_int, c_int, c_int, c_int, c_void_p, c_int, P_i32, P_i32, c_int,
                                   P_i32, P_i32, P_i32]),
    "mtp_quantize_int4_g64": (c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "mtp_quantize_int8_rows": (c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p, c_void_p]),
    "mtp_kv_commit": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MTPKV), P_i32]),
    "mtp_kv_commit_accepted": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MTPKV), P_i32, c_int]),
    "mtp_kv_rollback": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MTPKV)]),
    "mtp_kv_truncate": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MTPKV), P_i32]),
    "mtp_synth_target": (c_int, [c_void_p, c_void_p, c_int, c_int, P_i32, c_void_p, P_i32, P_i32,
                                 ctypes.c_uint64, c_void_p, P_i32]),
    "mtp_draft_confidence": (c_int, [c_void_p, c_void_p, c_int, c_int, c_void_p, c_float, c_void_p, P_i32]),
    "mtp_adapt_k": (c_int, [c_int, c_int, c_int, c_int, c_int]),
    "mtp_loop_advance": (c_int, [c_void_p, c_void_p, c_int, c_int, P_i32, P_i32, P_i32, c_void_p, P_i32, P_i32,
                                 c_void_p, c_void_p, P_i32, P_i32, c_int]),
    "mtp_spec_loop": (c_int, [c_void_p, c_void_p, ctypes.POINTER(MTPKV), ctypes.POINTER(MTPLoop), c_int]),
    "mtp_tree_workspace_bytes": (c_size_t, [c_void_p, c_int, c_int, c_int, c_int, c_int]),
    "mtp_draft_tree": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, P_i32, ctypes.POINTER(MTPKV),
                               ctypes.POINTER(MTPTree)]),
    "mtp_synth_target_tree": (c_int, [c_void_p, c_void_p, ctypes.POINTER(MTPTree), c_void_p, P_i32, ctypes.c_uint64,
                                      c_void_p, P_i32]),
    "mtp_verify_tree": (c_int, [c_void_p, c_void_p, ctypes.POINTER(MTPTree), c_void_p, P_i32, P_i32, P_i32]),
    "mtp_tree_commit": (c_int, [c_void_p, c_void_p, ctypes.POINTER(MTPKV), ctypes.POINTER(MTPTree), P_i32]),
    "mtp_tree_loop": (c_int, [c_void_p, c_void_p, ctypes.POINTER(MTPKV), ctypes.POINTER(MTPLoop),
                              ctypes.POINTER(MTPTree), c_int]),
    "mtp_selftest_wait_timeout": (c_int, [c_void_p, c_void_p, c_int]),
    "mtp_get_device_error": (c_int, [c_void_p]),
    "mtp_destroy": (None, [c_void_p]),
    "mtp_status_str": (ctypes.c_char_p, [c_int]),
    "mtp_stream_copy": (c_int, [c_void_p, c_void_p, c_void_p, c_size_t]),
    "mtp_stream_read": (c_int, [c_void_p, c_void_p, c_size_t, c_void_p]),
    "mtp_selftest_bounds": (c_int, [c_void_p, c_void_p]),
    "mtp_profile_begin": (c_int, [c_void_p, c_int, c_int]),
    "mtp_profile_end": (c_int, [c_void_p, ctypes.POINTER(c_float), c_int, ctypes.POINTER(c_int)]),
    "mtp_launch_count": (c_int64, [c_void_p]),
    "mtp_path_count": (c_int64, [c_void_p, c_int]),
}

_lib = None


def load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError("the MTP library is not built (%s); run __graft_entry__.build() or "
                          "python -m mtp_self_speculative_gb300._build" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
