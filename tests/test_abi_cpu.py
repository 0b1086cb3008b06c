"""The C ABI library loads and exports every entry point that include/mtp.h
declares; host-side argument checks reject bad calls before touching a
device.  CPU only: no call here launches work."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mtp.h")


@pytest.fixture(scope="module")
def lib():
    from mtp_self_speculative_gb300 import _lib
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:mtp_status|void|const char\*|int64_t)\s+(mtp_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("mtp_init", "mtp_draft", "mtp_verify", "mtp_kv_commit", "mtp_kv_rollback",
                     "mtp_destroy", "mtp_get_device_error", "mtp_status_str"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    from mtp_self_speculative_gb300 import _lib
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, "binding lacks " + name


def test_status_strings(lib):
    assert lib.mtp_status_str(0) == b"ok"
    assert b"invalid" in lib.mtp_status_str(1)
    assert lib.mtp_status_str(99) == b"unknown status"


def _cfg(**kw):
    from mtp_self_speculative_gb300 import _lib
    base = dict(hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=1024, vocab=4096, eps=1e-6,
                rope_theta=1e6, dtype=0, max_batch=1, max_k=3, block_size=16, max_pos=1024)
    base.update(kw)
    return _lib.MTPConfig(**base)


@pytest.mark.parametrize("bad", [dict(head_dim=96), dict(n_q_heads=6), dict(n_q_heads=48, n_kv_heads=3),
                                 dict(block_size=32), dict(max_k=0), dict(max_k=101), dict(dtype=7),
                                 dict(hidden=100), dict(ffn=1001), dict(vocab=0), dict(max_batch=0),
                                 dict(eps=0.0)])
def test_init_rejects_bad_config_without_a_device(lib, bad):
    from mtp_self_speculative_gb300 import _lib
    out = ctypes.c_void_p()
    w = _lib.MTPWeights(*([1] * 15))
    st = lib.mtp_init(ctypes.byref(_cfg(**bad)), ctypes.byref(w), 0, ctypes.byref(out))
    assert st == _lib.MTP_ERR_INVALID
    assert out.value is None


def test_init_rejects_missing_weight_pointer(lib):
    from mtp_self_speculative_gb300 import _lib
    out = ctypes.c_void_p()
    w = _lib.MTPWeights(*([1] * 15))
    w.w_o = None
    assert lib.mtp_init(ctypes.byref(_cfg()), ctypes.byref(w), 0, ctypes.byref(out)) == _lib.MTP_ERR_INVALID


def test_calls_without_context_are_rejected(lib):
    from mtp_self_speculative_gb300 import _lib
    kv = _lib.MTPKV(1, 1, 1, 1, 1, 1, 1)
    assert lib.mtp_draft(None, None, 1, 1, 1, 1, ctypes.byref(kv), 1, None, 1, None, None) == _lib.MTP_ERR_INVALID
    assert lib.mtp_verify(None, None, 1, 1, 1, 1, 1, 1, 1, 1, 1) == _lib.MTP_ERR_INVALID
    assert lib.mtp_kv_commit(None, None, 1, ctypes.byref(kv), 1) == _lib.MTP_ERR_INVALID
    assert lib.mtp_kv_rollback(None, None, 1, ctypes.byref(kv)) == _lib.MTP_ERR_INVALID
    assert lib.mtp_kv_truncate(None, None, 1, ctypes.byref(kv), 1) == _lib.MTP_ERR_INVALID
    assert lib.mtp_get_device_error(None) == _lib.MTP_ERR_INVALID
    assert lib.mtp_selftest_wait_timeout(None, None, 0) == _lib.MTP_ERR_INVALID
    assert lib.mtp_profile_begin(None, 0, 1) == _lib.MTP_ERR_INVALID
    assert lib.mtp_launch_count(None) == 0
    assert lib.mtp_path_count(None, 0) == 0
    lib.mtp_destroy(None)


def test_stream_copy_rejects_unaligned_or_overlapping(lib):
    from mtp_self_speculative_gb300 import _lib
    assert lib.mtp_stream_copy(None, 16, 4096, 15) == _lib.MTP_ERR_INVALID
    assert lib.mtp_stream_copy(None, 17, 4096, 16) == _lib.MTP_ERR_INVALID
    assert lib.mtp_stream_copy(None, 4096, 4096 + 16, 64) == _lib.MTP_ERR_INVALID


def test_verify_wrappers_check_shapes_before_any_call():
    """The C entry points receive plain pointers, so the binding checks what
    they cannot: logits dtype (float32 or bfloat16), a 2-D [rows, vocab]
    logits tensor, B + 1 row offsets, B draft rows, B outputs.  Every bad
    case raises before anything reaches the library; the well-formed case
    (CPU tensors here) stops at the device-pointer check."""
    import torch
    import mtp_self_speculative_gb300 as M
    V, B = 100, 3
    i32 = dict(dtype=torch.int32)
    good = dict(target_logits=torch.zeros((8, V), dtype=torch.bfloat16), row_offsets=torch.zeros(B + 1, **i32),
                drafts=torch.zeros((B, 4), **i32), num_drafts=torch.zeros(B, **i32),
                accepted=torch.zeros(B, **i32), bonus=torch.zeros(B, **i32))
    bad = [("target_logits", torch.zeros((8, V), dtype=torch.float16), "float32 or bfloat16"),
           ("target_logits", torch.zeros((2, 4, V), dtype=torch.bfloat16), "vocab"),
           ("target_logits", torch.zeros((8, V + 1), dtype=torch.bfloat16), "vocab"),
           ("row_offsets", torch.zeros(B, **i32), "row_offsets"),
           ("drafts", torch.zeros((B + 1, 4), **i32), "drafts"),
           ("drafts", torch.zeros(B * 4, **i32), "drafts"),
           ("accepted", torch.zeros(B - 1, **i32), "accepted"),
           ("bonus", torch.zeros(B + 1, **i32), "bonus")]
    ctx = M.Context(0, M.make_config(256, 4, 2, 64, 1024, V, dtype="bf16", max_batch=B, max_k=4), None)
    calls = [lambda kw: M.mtp_verify_noalloc(vocab=V, max_k=4, **kw), lambda kw: M.mtp_verify(ctx, **kw)]
    for call in calls:
        for name, t, msg in bad:
            with pytest.raises(ValueError, match=msg):
                call(dict(good, **{name: t}))
        with pytest.raises(ValueError, match="CUDA tensor"):
            call(dict(good, stream=_NullStream()))


class _NullStream:
    """Stands in for a torch stream on a machine without a GPU (handle 0)."""
    cuda_stream = 0


def test_stream_read_rejects_bad_arguments(lib):
    from mtp_self_speculative_gb300 import _lib
    assert lib.mtp_stream_read(None, None, 4096, None) == _lib.MTP_ERR_INVALID
    assert lib.mtp_stream_read(None, 16, 0, None) == _lib.MTP_ERR_INVALID
    assert lib.mtp_stream_read(None, 16, 4008, None) == _lib.MTP_ERR_INVALID
    assert lib.mtp_stream_read(None, 24, 4096, None) == _lib.MTP_ERR_INVALID


def test_bounds_selftest_needs_a_context(lib):
    from mtp_self_speculative_gb300 import _lib
    assert lib.mtp_selftest_bounds(None, None) == _lib.MTP_ERR_INVALID


def test_binding_constants_equal_the_header_enums():
    """Every enumerator of include/mtp.h (status codes, dtypes, weight formats,
    kernel ids, path ids; the *_COUNT bounds aside) exists in the Python
    binding with the header's value."""
    import mtp_self_speculative_gb300 as M
    text = open(HEADER).read()
    enums = re.findall(r"\b(MTP_[A-Z0-9_]+)\s*=\s*(\d+)", text)
    assert len(enums) >= 20
    for name, value in enums:
        if name.endswith("_COUNT"):
            continue
        assert hasattr(M, name), "binding lacks " + name
        assert getattr(M, name) == int(value), name
