#!/usr/bin/env python
"""Benchmark of the MTP draft+verify step on one GB300 per process.

A step is one pass of the whole hot path for one batch:
    mtp_draft (K recursive draft steps: eh_proj, QKV+rotary+KV append,
    split-KV attention, O-proj, SwiGLU MLP, LM head + argmax)
    -> mtp_verify (greedy accept against target logits)
    -> mtp_kv_commit_accepted (keep min(a+1, K) drafted slots)
    -> mtp_kv_truncate (return the cache to its starting length so that
       every step sees the same state).
The target logits are built once before timing: one untimed draft gives the
draft ids, and the target rows carry a +8 spike on those ids for a seeded
geometric(0.8) prefix, then a mismatch -- so the verify step accepts a known
prefix.  Inputs (1.7 GB of weights for the Qwen3-8B shape) are far larger than
L2, so no cache flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank drives its own GPU as an independent replica (the
path has no data-path exchange); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import glob
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MTP draft+verify steps/s and accepted tok/s (Qwen3-8B shape); % HBM roofline"
# dram__bytes_read.sum + dram__bytes_write.sum of one LM-head launch from an ncu capture of the
# current kernel (profiles/lm_head_argmax_qwen3_8b_mtp_b1.md); other workloads report null.
LM_TRAFFIC = {
    "qwen3_8b_mtp_b1": 1244766976 + 3336448,
    "qwen3_8b_mtp_b1:int4_g64": 622737408 + 3309056,
}
# The same for one verify launch (profiles/verify_rollback_b64.md).
VERIFY_TRAFFIC = {
    "verify_rollback_b64": 111259136 + 3191296,
}
# The same for one launch of the persistent draft kernel (all K steps); null until captured.
PERSISTENT_TRAFFIC = {}
WORKLOADS = {c.name: c for c in synth.CONFIGS}
DEFAULT_WORKLOAD = synth.QWEN3_8B_B1.name


# ------------------------------------------------------------------ helpers

def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(value: float, world: int) -> float:
    """Max over ranks (harness timing only)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def blas_threads() -> int:
    try:
        import ctypes
        libdir = os.path.join(os.path.dirname(np.__file__) + ".libs")
        for so in glob.glob(os.path.join(libdir, "*openblas*.so*")):
            lib = ctypes.CDLL(so)
            for name in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_",
                         "openblas_get_num_threads"):
                if hasattr(lib, name):
                    return int(getattr(lib, name)())
    except Exception:
        pass
    return os.cpu_count() or 1


def mat_bytes(cfg: synth.MTPShape, rows: int, cols: int, fmt: str, table: bool = False) -> int:
    """Stored bytes of one weight matrix: dense elements, or the quantized
    format (projections: 4-bit codes plus an fp16 scale and a byte zero point
    per 64 columns; the embedding / LM head table: int8 codes plus an fp16
    scale per row)."""
    if fmt == "dense":
        return rows * cols * cfg.elem_bytes
    if table:
        return rows * cols + rows * 2
    return rows * cols // 2 + rows * (cols // 64) * 3


def weight_bytes(cfg: synth.MTPShape, fmt: str = "dense") -> int:
    """Bytes of all weights read once per draft step (tied LM head = embed)."""
    if fmt == "dense":
        return cfg.weight_bytes()
    H, F, V, qd, kvd = cfg.H, cfg.ffn, cfg.vocab, cfg.q_dim, cfg.kv_dim
    mats = (mat_bytes(cfg, H, 2 * H, fmt) + mat_bytes(cfg, qd + 2 * kvd, H, fmt) + mat_bytes(cfg, H, qd, fmt)
            + mat_bytes(cfg, 2 * F, H, fmt) + mat_bytes(cfg, H, F, fmt) + mat_bytes(cfg, V, H, fmt, table=True))
    return mats + 5 * H * cfg.elem_bytes


def step_bytes(cfg: synth.MTPShape, lens: np.ndarray, K: int, with_logits: bool = True, fmt: str = "dense") -> dict:
    """Algorithmic bytes of one step: every weight and KV entry read once per
    draft step, plus the writes of logits, ids and new KV entries."""
    e = cfg.elem_bytes
    B = len(lens)
    w = weight_bytes(cfg, fmt)
    kv_row = 2 * cfg.n_kv * cfg.head_dim * e           # K and V of one slot
    lm = mat_bytes(cfg, cfg.vocab, cfg.H, fmt, table=True) + cfg.H * e   # LM head rows + final norm weight
    draft = 0
    for k in range(1, K + 1):
        kv_read = int(np.sum(lens + k)) * kv_row
        draft += w + kv_read + B * kv_row + (B * cfg.vocab * 4 if with_logits else 0) + B * 4
    verify = B * (K + 1) * cfg.vocab * e
    commit = B * K * kv_row                               # at most K slots rewritten
    return {"draft": draft, "verify": verify, "commit": commit, "total": draft + verify + commit,
            "lm_head_launch": lm + B * cfg.H * 4 + (B * cfg.vocab * 4 if with_logits else 0),
            "weights": w}


def kernel_bytes(cfg: synth.MTPShape, lens: np.ndarray, K: int, with_logits: bool = True,
                 fmt: str = "dense") -> dict:
    """Algorithmic bytes of one launch of each kernel (draft kernels: one
    draft step, attention averaged over k = 1..K)."""
    e = cfg.elem_bytes
    B = len(lens)
    H, F, V, qd, kvd = cfg.H, cfg.ffn, cfg.vocab, cfg.q_dim, cfg.kv_dim
    kv_row = 2 * kvd * e
    mean_ctx = float(np.sum(lens)) + B * (K + 1) / 2.0
    m = lambda r, c, table=False: mat_bytes(cfg, r, c, fmt, table)
    return {
        "eh_proj": m(H, 2 * H) + 2 * H * e + B * 2 * H * e + B * H * 4,
        "qkv_rope": m(qd + 2 * kvd, H) + H * e + B * H * 4 + B * (qd * 4 + kv_row),
        "attention": mean_ctx * kv_row + B * qd * 8,
        "o_proj": m(H, qd) + B * (qd + 2 * H) * 4,
        "gate_up": m(2 * F, H) + H * e + B * (H * 4 + F * 4),
        "down": m(H, F) + B * (F * 4 + 2 * H * 4),
        "lm_head": m(V, H, True) + H * e + B * H * 4 + (B * V * 4 if with_logits else 0),
        "verify": B * (K + 1) * V * e,
        "draft_persistent": step_bytes(cfg, lens, K, with_logits, fmt)["draft"],
    }


def kernel_breakdown(wl, steps: int) -> dict:
    """Mean live duration of each kernel (CUDA events around its launches,
    one kernel id at a time) and its bandwidth against its algorithmic
    bytes.  Events break the programmatic overlap at the timed kernel's
    boundaries, so these are per-kernel, not additive, figures."""
    import torch
    import mtp_self_speculative_gb300 as M
    kb = kernel_bytes(wl.cfg, wl.lens, wl.K, fmt=wl.weight_format)
    peak = float(measured_peaks()[0]["hbm_gbs"])
    out = {}
    for kid, name in enumerate(M.KERNEL_NAMES):
        per_step = wl.K if kid <= M.MTP_KERNEL_LM_HEAD else (2 if kid == M.MTP_KERNEL_KV_EDIT else 1)
        if kid == M.MTP_KERNEL_DRAFT_PERSISTENT:
            per_step = 1
        M.mtp_profile_begin(wl.ctx, kid, steps * per_step)
        for _ in range(steps):
            wl.step()
        torch.cuda.synchronize()
        ms = M.mtp_profile_end(wl.ctx, steps * per_step)
        if not ms:
            continue
        us = 1e3 * statistics.mean(ms)
        entry = {"us": round(us, 2), "launches": len(ms)}
        if name in kb:
            gbs = kb[name] / (us * 1e-6) / 1e9
            entry.update({"bytes": int(kb[name]), "gbs": round(gbs, 1), "frac": round(gbs / peak, 3)})
        out[name] = entry
    return out


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, "--query-gpu=" + self.FIELDS, "--format=csv,noheader",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def mhz(s):
            try:
                return float(s.split()[0])
            except Exception:
                return float("nan")
        sm = [mhz(r[1]) for r in rows]
        smax = [mhz(r[2]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        load = [s for s in sm if not math.isnan(s)]
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(s for s in smax if not math.isnan(s)) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((mhz(r[3]) for r in rows), default=None)}


def gpu_id_for_smi(local_rank: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(local_rank).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[local_rank] if vis else str(local_rank)


# ------------------------------------------------------------- workload

class Workload:
    """Device-resident inputs and outputs of one draft+verify step."""

    def __init__(self, cfg: synth.MTPShape, K: int, persistent_max_batch: int = 0, weight_format: str = "dense"):
        import torch
        import mtp_self_speculative_gb300 as M
        self.cfg, self.K = cfg, K
        self.weight_format = weight_format
        self.w = synth.make_weights(cfg, norm="ones")
        self.lens = synth.context_lengths(cfg)
        self.B = B = len(self.lens)
        self.kv0 = synth.make_kv(cfg, self.lens, extra_slots=K + 1)
        self.di = synth.make_draft_inputs(cfg, self.w, self.lens)
        tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32

        def dev(a):
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
            return torch.from_numpy(a).cuda()
        self.dev = dev
        self.wdev = {k: dev(v) for k, v in self.w.items()}
        self.ctx = M.mtp_init(M.make_config(cfg.H, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.ffn, cfg.vocab, cfg.eps,
                                            cfg.rope_theta, cfg.dtype, B, K, cfg.block_size,
                                            int(self.lens.max()) + K + 8,
                                            persistent_max_batch=persistent_max_batch,
                                            weight_format=weight_format), self.wdev)
        self.kv = M.KVCache(dev(self.kv0.k_pool), dev(self.kv0.v_pool), dev(self.kv0.block_table),
                            dev(self.kv0.seq_len), dev(self.kv0.pending))
        self.L0 = dev(self.lens.astype(np.int32))
        self.hidden, self.embeds, self.positions = dev(self.di.hidden), dev(self.di.embeds), dev(self.di.positions)
        self.ids = torch.empty((B, K), dtype=torch.int32, device="cuda")
        self.logits = torch.empty((B, K, cfg.vocab), dtype=torch.float32, device="cuda")
        self.acc = torch.empty(B, dtype=torch.int32, device="cuda")
        self.bonus = torch.empty(B, dtype=torch.int32, device="cuda")
        self.tdt = tdt
        # one untimed draft: its ids carry the target spikes
        self.draft()
        M.mtp_kv_rollback(self.ctx, self.kv)
        torch.cuda.synchronize()
        ids0 = self.ids.cpu().numpy()
        self.ids0 = ids0
        u = 1.0 - synth.uniform01(cfg.seed, 60, (B,))
        n = np.minimum(synth.geometric_len(u, 0.8), K).astype(np.int32)
        other = synth.uniform_int(cfg.seed, 61, (B, K + 1), 0, cfg.vocab - 1)
        planted = np.empty((B, K + 1), dtype=np.int32)
        for b in range(B):
            for j in range(K + 1):
                if j < n[b]:
                    planted[b, j] = ids0[b, j]
                else:
                    x = int(other[b, j])
                    planted[b, j] = x + 1 if (j < K and x >= ids0[b, j]) else x
        vcfg = synth.shrink(cfg, batch=B, k_lo=0, k_hi=0)
        vi = synth.make_verify_inputs(vcfg, num_drafts=np.full(B, K, dtype=np.int32), planted_ids=planted)
        self.planted_len = n
        self.target = dev(vi.logits)
        self.row_offsets = dev(vi.row_offsets)
        self.num_drafts = dev(vi.num_drafts)
        self.vi = vi

    def draft(self, logits=True):
        import mtp_self_speculative_gb300 as M
        M.mtp_draft(self.ctx, self.hidden, self.embeds, self.positions, self.kv, self.K, self.ids,
                    self.logits if logits else None)

    def step(self):
        import mtp_self_speculative_gb300 as M
        self.draft()
        M.mtp_verify(self.ctx, self.target, self.row_offsets, self.ids, self.num_drafts, self.acc, self.bonus)
        M.mtp_kv_commit_accepted(self.ctx, self.kv, self.acc, extra=1)
        M.mtp_kv_truncate(self.ctx, self.kv, self.L0)


def run_ours(args, rank, world, local_rank):
    import torch
    torch.cuda.set_device(local_rank)
    import mtp_self_speculative_gb300 as M
    cfg = WORKLOADS[args.workload]
    if cfg.H == 0:
        return run_verify_workload(args, cfg, rank, world, local_rank)
    if args.loop:
        return run_loop_workload(args, cfg, rank, world, local_rank)
    K = cfg.K
    wl = Workload(cfg, K, args.persistent_max_batch, args.weights)
    stream = torch.cuda.current_stream()

    # bandwidth yardstick in the same run: 1 GiB device-to-device copy
    nbytes = 1 << 30
    src = torch.empty(nbytes // 2, dtype=torch.int16, device="cuda").fill_(1)
    dst = torch.empty_like(src)
    for _ in range(3):
        M.mtp_stream_copy(dst, src)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    copies = []
    for _ in range(10):
        e0.record(stream)
        M.mtp_stream_copy(dst, src)
        e1.record(stream)
        e1.synchronize()
        copies.append(e0.elapsed_time(e1))
    copy_gbs = 2 * nbytes / (min(copies) * 1e-3) / 1e9
    del src, dst
    kb0 = kernel_bytes(cfg, wl.lens, K, fmt=args.weights)
    read_floor = read_floor_us({n: kb0[n] for n in ("eh_proj", "qkv_rope", "attention", "o_proj", "gate_up", "down",
                                                    "lm_head", "verify")}, stream)

    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    assert M.mtp_get_device_error(wl.ctx) == 0

    launches0 = M.mtp_launch_count(wl.ctx)
    sampler = ClockSampler(gpu_id_for_smi(local_rank)) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        wl.step()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    launches = M.mtp_launch_count(wl.ctx) - launches0
    elapsed_ms = t0.elapsed_time(t1)
    # Roofline kernel: CUDA events around every launch of the dominant kernel
    # (the persistent draft kernel when the batch runs on it, else the LM
    # head), recorded by the library on its stream, over a second pass of the
    # same steps (event records between kernels cancel the programmatic
    # overlap, so they stay out of the timed region above).
    lm_steps = min(args.steps, 400)
    roof_kid, per = M.MTP_KERNEL_DRAFT_PERSISTENT, 1
    M.mtp_profile_begin(wl.ctx, roof_kid, lm_steps * per)
    for _ in range(lm_steps):
        wl.step()
    torch.cuda.synchronize()
    lm_ms = M.mtp_profile_end(wl.ctx, lm_steps * per)
    if not lm_ms:
        roof_kid, per = M.MTP_KERNEL_LM_HEAD, K
        M.mtp_profile_begin(wl.ctx, roof_kid, lm_steps * per)
        for _ in range(lm_steps):
            wl.step()
        torch.cuda.synchronize()
        lm_ms = M.mtp_profile_end(wl.ctx, lm_steps * per)
    assert M.mtp_get_device_error(wl.ctx) == 0
    ids_now = wl.ids.cpu().numpy()
    deterministic = bool(np.array_equal(ids_now, wl.ids0))
    acc = wl.acc.cpu().numpy()
    elapsed_max = reduce_max(elapsed_ms, world)

    # draft-only timing (the roofline target is the draft step)
    M.mtp_kv_rollback(wl.ctx, wl.kv)
    nd = max(10, args.steps // 4)
    t0.record(stream)
    for _ in range(nd):
        wl.draft()
        M.mtp_kv_rollback(wl.ctx, wl.kv)
    t1.record(stream)
    torch.cuda.synchronize()
    draft_ms = t0.elapsed_time(t1) / nd

    kernels = kernel_breakdown(wl, 20)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(wl, max(5, min(args.steps // 4, 200)))

    # the first draft's ids and logits (the workload is deterministic: every
    # draft from the starting state gives them), for the exact-id report
    wl.draft()
    M.mtp_kv_rollback(wl.ctx, wl.kv)
    torch.cuda.synchronize()
    first_ids, first_logits = wl.ids.cpu().numpy(), wl.logits.cpu().numpy()

    # the other configurations, measured in the same process (N = 1 only)
    others = None
    if world == 1 and not args.no_workloads and args.workload == DEFAULT_WORKLOAD and args.weights == "dense" \
            and args.persistent_max_batch == 0 and args.ctx is None:
        others = measure_other_workloads(args, local_rank)

    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    sb = step_bytes(cfg, wl.lens, K, fmt=args.weights)
    ms_per_step = elapsed_max / args.steps
    steps_s = world * args.steps / (elapsed_max * 1e-3)
    emitted = int(np.sum(acc + 1))
    lm_avg_ms = statistics.mean(lm_ms) if lm_ms else float("nan")
    persistent = roof_kid == M.MTP_KERNEL_DRAFT_PERSISTENT
    roof_bytes = sb["draft"] if persistent else sb["lm_head_launch"]
    lm_gbs = roof_bytes / (lm_avg_ms * 1e-3) / 1e9
    tkey = cfg.name if args.weights == "dense" else cfg.name + ":" + args.weights
    if persistent:
        traffic = args.lm_traffic if args.lm_traffic is not None else PERSISTENT_TRAFFIC.get(tkey)
    else:
        traffic = args.lm_traffic if args.lm_traffic is not None else LM_TRAFFIC.get(tkey)
    peak = float(peaks["hbm_gbs"])
    line = {
        "metric": METRIC,
        "value": steps_s,
        "unit": "steps/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype if args.weights == "dense" else "int4/int8 weights, f32 arithmetic, bf16 KV",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) hidden/KV, uniform token ids)",
        "config": {"workload": cfg.name, "hidden": cfg.H, "q_heads": cfg.n_q, "kv_heads": cfg.n_kv,
                   "head_dim": cfg.head_dim, "ffn": cfg.ffn, "vocab": cfg.vocab, "batch": wl.B,
                   "draft_steps_K": K, "mtp_context": [int(wl.lens.min()), int(wl.lens.max())],
                   "tied_lm_head": True, "parallelism": "replicas" if world > 1 else "single",
                   "weights": args.weights if args.weights == "dense" else
                              "int4_g64 asymmetric projections, int8 symmetric per-row embedding/LM head",
                   "l2": "inputs larger than L2 (%.2f GB of weights streamed per draft step)" %
                         (sb["weights"] / 1e9)},
        "accepted_tok_s": {"emitted": emitted * steps_s, "accepted_drafts": int(np.sum(acc)) * steps_s,
                           "mean_emitted_per_step": emitted / wl.B},
        "draft": {"ms_per_draft_call": draft_ms, "ms_per_draft_step": draft_ms / K,
                  "bytes_per_draft_step": sb["draft"] / K,
                  "hbm_frac_of_measured": sb["draft"] / (draft_ms * 1e-3) / 1e9 / peak},
        "step_hbm": {"bytes_per_step": sb["total"],
                     "achieved_gbs": sb["total"] / (ms_per_step * 1e-3) / 1e9,
                     "frac_of_measured": sb["total"] / (ms_per_step * 1e-3) / 1e9 / peak},
        "roofline": {"kernel": "draft_persistent" if persistent else
                               ("lm_head_argmax" if args.weights == "dense" else "lm_head_argmax_int8"), "bound": "hbm",
                     "achieved": lm_gbs, "peak": peak, "unit": "GB/s", "frac": lm_gbs / peak,
                     "peak_source": peak_kind + " hbm_gbs", "traffic": traffic,
                     "launches_timed": len(lm_ms), "bytes_per_launch": roof_bytes},
        "kernels": kernels,
        "stream_copy_gbs": copy_gbs,
        "read_floor": read_floor,
        "gpu_launches": int(launches),
        "deterministic_ids": deterministic,
        "clocks": clocks,
    }
    if e2e:
        line["e2e"] = e2e
    if others:
        line["workloads"] = others
    if world == 1 and not args.no_cpu_baseline:
        cb, parity = cpu_baseline(cfg, fmt=args.weights, gpu_ids=first_ids, gpu_logits=first_logits)
        line["cpu_baseline"] = cb
        line["draft_parity"] = parity
    print(json.dumps(line), flush=True)


def l2_flush(buf) -> None:
    """Evicts L2 by reading a buffer larger than it.  A read leaves clean
    lines behind: a write would leave the next kernel to write back up to
    the whole L2 of dirty lines as it misses, which is not that kernel's
    traffic.  The bytes are summed as int64 words, so that no widened copy
    of the buffer is written first."""
    import torch
    buf.view(torch.int64).sum()


def read_floor_us(sizes: dict, stream, reps: int = 10) -> dict:
    """Best time of the read-only yardstick (mtp_stream_read: the bytes
    streamed once into shared memory, nothing computed) for each named byte
    count, L2 flushed by a read before every timed call: the least a kernel
    that only reads that many bytes takes, launch and tail included."""
    import torch
    import mtp_self_speculative_gb300 as M
    biggest = max(int(v) for v in sizes.values())
    buf = torch.empty((biggest + 4095) // 4096 * 4096, dtype=torch.uint8, device="cuda")
    buf.fill_(1)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda").fill_(1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out = {}
    for name, n in sizes.items():
        n = int(n) // 16 * 16
        best = float("inf")
        for r in range(reps + 2):
            l2_flush(flush)
            e0.record(stream)
            M.mtp_stream_read(buf, n, err)
            e1.record(stream)
            e1.synchronize()
            if r >= 2:
                best = min(best, e0.elapsed_time(e1))
        out[name] = {"bytes": n, "us": round(best * 1e3, 2), "gbs": round(n / (best * 1e-3) / 1e9, 1)}
    assert int(err.item()) == 0
    del buf, flush
    return out


def timed_steps(fn, n: int, stream) -> float:
    """Mean milliseconds of n calls of fn, CUDA events on the launching
    stream, synchronised on both sides."""
    import torch
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(n):
        fn()
    t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / n


def measure_draft_workload(cfg: synth.MTPShape, local_rank: int, steps: int, warmup: int, peak: float) -> dict:
    """Full steps (draft K + verify + commit + truncate) and draft-only calls
    of one draft configuration, with its per-kernel breakdown and the clocks
    seen while its steps ran."""
    import torch
    import mtp_self_speculative_gb300 as M
    wl = Workload(cfg, cfg.K)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        wl.step()
    torch.cuda.synchronize()
    assert M.mtp_get_device_error(wl.ctx) == 0
    sampler = ClockSampler(gpu_id_for_smi(local_rank))
    sampler.start()
    ms_step = timed_steps(wl.step, steps, stream)

    def draft_only():
        wl.draft()
        M.mtp_kv_rollback(wl.ctx, wl.kv)
    ms_draft = timed_steps(draft_only, steps, stream)
    clocks = sampler.stop()
    kernels = kernel_breakdown(wl, max(3, steps // 2))
    assert M.mtp_get_device_error(wl.ctx) == 0
    sb = step_bytes(cfg, wl.lens, cfg.K)
    acc = wl.acc.cpu().numpy()
    out = {
        "batch": wl.B, "draft_steps_K": cfg.K, "hidden": cfg.H, "ffn": cfg.ffn, "q_heads": cfg.n_q,
        "mtp_context": [int(wl.lens.min()), int(wl.lens.max())], "dtype": cfg.dtype,
        "steps_s": 1e3 / ms_step, "ms_per_step": ms_step,
        "accepted_tok_s": {"emitted": float(np.sum(acc + 1)) * 1e3 / ms_step,
                           "accepted_drafts": float(np.sum(acc)) * 1e3 / ms_step},
        "draft": {"ms_per_draft_step": ms_draft / cfg.K, "bytes_per_draft_step": sb["draft"] / cfg.K,
                  "hbm_frac_of_measured": sb["draft"] / (ms_draft * 1e-3) / 1e9 / peak},
        "step_hbm_frac_of_measured": sb["total"] / (ms_step * 1e-3) / 1e9 / peak,
        "kernels": kernels, "clocks": clocks, "timed_steps": steps,
    }
    M.mtp_destroy(wl.ctx)
    del wl
    torch.cuda.empty_cache()
    return out


def measure_verify_workload(cfg: synth.MTPShape, local_rank: int, calls: int, peak: float) -> dict:
    """mtp_verify + mtp_kv_commit_accepted on the 64-request verify inputs,
    each call timed with CUDA events, L2 flushed between calls."""
    import torch
    import mtp_self_speculative_gb300 as M
    vi = synth.make_verify_inputs(cfg)
    lens = synth.context_lengths(cfg)
    kv0 = synth.make_kv(cfg, lens, extra_slots=int(vi.num_drafts.max()) + 1, prefill_slots=lens + vi.num_drafts)
    kv0.pending = vi.num_drafts.astype(np.int32).copy()
    B = len(lens)

    def dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(a).cuda()
    ctx = M.mtp_init(M.make_config(1, cfg.n_q, cfg.n_kv, cfg.head_dim, 8, cfg.vocab, dtype=cfg.dtype, max_batch=B,
                                   max_k=vi.max_k, block_size=cfg.block_size))
    kv = M.KVCache(dev(kv0.k_pool), dev(kv0.v_pool), dev(kv0.block_table), dev(kv0.seq_len), dev(kv0.pending))
    seq0, pend0 = dev(kv0.seq_len), dev(kv0.pending)
    logits, ro, drafts, nd = dev(vi.logits), dev(vi.row_offsets), dev(vi.drafts), dev(vi.num_drafts)
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    bon = torch.empty(B, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(calls)]
    for i in range(3 + calls):
        e = ev[i - 3] if i >= 3 else None
        if e:
            e[0].record(stream)
        M.mtp_verify(ctx, logits, ro, drafts, nd, acc, bon)
        if e:
            e[1].record(stream)
        M.mtp_kv_commit_accepted(ctx, kv, acc, extra=1)
        if e:
            e[2].record(stream)
        kv.seq_len.copy_(seq0)
        kv.pending.copy_(pend0)
        l2_flush(flush)
        if i == 2:
            torch.cuda.synchronize()
            sampler = ClockSampler(gpu_id_for_smi(local_rank))
            sampler.start()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    assert M.mtp_get_device_error(ctx) == 0
    t_ver = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    t_com = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    ver_bytes = int(vi.row_offsets[-1]) * cfg.vocab * cfg.elem_bytes
    gbs = ver_bytes / (t_ver * 1e-3) / 1e9
    M.mtp_destroy(ctx)
    del logits, flush
    floor = read_floor_us({"verify": ver_bytes}, stream)["verify"]
    return {"batch": B, "k_range": [int(vi.num_drafts.min()), int(vi.num_drafts.max())], "read_floor": floor,
            "verify_rows": int(vi.row_offsets[-1]), "calls_s": 1e3 / (t_ver + t_com), "verify_ms": t_ver,
            "commit_ms": t_com, "verify_bytes": ver_bytes, "verify_gbs": gbs, "verify_hbm_frac_of_measured": gbs / peak,
            "l2": "flushed between calls (256 MB read outside the events)", "timed_calls": calls, "clocks": clocks}


def measure_small_batch(local_rank: int, steps: int = 6) -> dict:
    """The Qwen3-8B-shaped head at 1, 2 and 4 requests (tree expansions and
    small batches): draft-step time and HBM fraction, and every kernel's mean
    live duration per launch from the per-kernel events, with its time
    relative to the 1-request launch."""
    import dataclasses
    import torch
    import mtp_self_speculative_gb300 as M
    peak = float(measured_peaks()[0]["hbm_gbs"])
    out = {}
    for B in (1, 2, 4):
        cfg = dataclasses.replace(synth.QWEN3_8B_B1, name="qwen3_8b_mtp_b%d" % B, batch=B)
        wl = Workload(cfg, cfg.K)
        for _ in range(3):
            wl.step()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()

        def draft_only():
            wl.draft()
            M.mtp_kv_rollback(wl.ctx, wl.kv)
        ms_draft = timed_steps(draft_only, steps * 4, stream)
        kernels = kernel_breakdown(wl, steps)
        assert M.mtp_get_device_error(wl.ctx) == 0
        sb = step_bytes(cfg, wl.lens, cfg.K)
        out["b%d" % B] = {
            "ms_per_draft_step": round(ms_draft / cfg.K, 4),
            "draft_hbm_frac_of_measured": round(sb["draft"] / (ms_draft * 1e-3) / 1e9 / peak, 4),
            "kernels_us": {k: v["us"] for k, v in kernels.items() if k not in ("verify", "kv_edit")},
            "lm_head_frac": kernels["lm_head"]["frac"]}
        M.mtp_destroy(wl.ctx)
        del wl
        torch.cuda.empty_cache()
    for k in ("b2", "b4"):
        out[k]["vs_b1"] = {n: round(us / out["b1"]["kernels_us"][n], 3)
                           for n, us in out[k]["kernels_us"].items() if out["b1"]["kernels_us"].get(n)}
    out["note"] = "per-kernel CUDA events inside full steps (L2 holds no weights: 1.7 GB per draft step)"
    return out


def measure_other_workloads(args, local_rank: int) -> dict:
    """The continuous-batching, large-batch and verify configurations, each
    set up, measured at a few steps and freed in turn, and the Qwen3-8B
    shape at 1, 2 and 4 requests."""
    peak = float(measured_peaks()[0]["hbm_gbs"])
    out = {"small_batch": measure_small_batch(local_rank)}
    for cfg, steps in ((synth.QWEN3_8B_CB32, 20), (synth.QWEN3_32B_B128, 6)):
        out[cfg.name] = measure_draft_workload(cfg, local_rank, steps, 3, peak)
    out[synth.VERIFY_B64.name] = measure_verify_workload(synth.VERIFY_B64, local_rank, 50, peak)
    return out


def run_e2e(wl: Workload, n: int) -> dict:
    """steps/s through the public API with pinned host inputs copied in and
    the step's results (draft ids, accepted counts, bonus ids) read back every
    step."""
    import torch
    import mtp_self_speculative_gb300 as M
    h_hidden = wl.hidden.cpu().pin_memory()
    h_embeds = wl.embeds.cpu().pin_memory()
    h_pos = wl.positions.cpu().pin_memory()
    h_target = wl.target.cpu().pin_memory()
    h_ids = torch.empty_like(wl.ids, device="cpu").pin_memory()
    h_acc = torch.empty_like(wl.acc, device="cpu").pin_memory()
    h_bonus = torch.empty_like(wl.bonus, device="cpu").pin_memory()
    bi = sum(t.numel() * t.element_size() for t in (h_hidden, h_embeds, h_pos, h_target))
    bo = sum(t.numel() * t.element_size() for t in (h_ids, h_acc, h_bonus))

    def one():
        wl.hidden.copy_(h_hidden, non_blocking=True)
        wl.embeds.copy_(h_embeds, non_blocking=True)
        wl.positions.copy_(h_pos, non_blocking=True)
        wl.target.copy_(h_target, non_blocking=True)
        M.mtp_draft(wl.ctx, wl.hidden, wl.embeds, wl.positions, wl.kv, wl.K, wl.ids, wl.logits)
        M.mtp_verify(wl.ctx, wl.target, wl.row_offsets, wl.ids, wl.num_drafts, wl.acc, wl.bonus)
        M.mtp_kv_commit_accepted(wl.ctx, wl.kv, wl.acc, extra=1)
        M.mtp_kv_truncate(wl.ctx, wl.kv, wl.L0)
        h_ids.copy_(wl.ids, non_blocking=True)
        h_acc.copy_(wl.acc, non_blocking=True)
        h_bonus.copy_(wl.bonus, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(3):
        one()
    torch.cuda.synchronize()
    t = time.perf_counter()
    for _ in range(n):
        one()
    dt = time.perf_counter() - t
    return {"value": n / dt, "unit": "steps/s", "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo),
            "steps": n}


# ------------------------------------------------------- CPU / oracle legs

LOOP_METRIC = "speculative loop emitted tokens/s (draft + synthetic verifier + verify + commit)"


def run_loop_workload(args, cfg, rank, world, local_rank):
    """The full speculative loop (mtp_spec_loop) on the draft workload's
    shape: the copy-head weight recipe (drafts repeat their input token) and
    the synthetic verifier with a sticky probability of --loop-alpha, so that
    drafts are accepted at a controlled rate.  One step = one loop iteration
    (K drafts, K + 1 verifier rows, verify, commit, state advance); value =
    emitted tokens per second over all requests."""
    import torch
    import mtp_self_speculative_gb300 as M
    K = cfg.K
    B = cfg.batch
    lens = synth.context_lengths(cfg)
    w = synth.copy_head(cfg, synth.make_weights(cfg, norm="ones"))
    thr = int(args.loop_alpha * 2 ** 53)
    total = args.warmup + args.steps + 2 * max(5, args.steps // 4) + 8
    tree_shape = tuple(int(x) for x in args.tree.split(",")) if args.tree else None
    if tree_shape:
        K = tree_shape[1]                      # an accepted path is at most tree_depth long
    kv0 = synth.make_kv(cfg, lens, extra_slots=(K + 1) * total + K + 1)
    scratch = None
    if tree_shape:
        bf_, td_, _ = tree_shape
        n_extra = max(td_ - 1, 1) * B * bf_ * 2
        zeros = np.zeros((n_extra,) + kv0.k_pool.shape[1:], dtype=kv0.k_pool.dtype)
        scratch = np.arange(kv0.k_pool.shape[0], kv0.k_pool.shape[0] + n_extra, dtype=np.int32)
        kv0 = synth.KVState(np.concatenate([kv0.k_pool, zeros]), np.concatenate([kv0.v_pool, zeros]),
                            kv0.block_table, kv0.seq_len, kv0.pending, kv0.block_size)

    def dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(a).cuda()
    wdev = {k: dev(v) for k, v in w.items()}
    max_batch = B * tree_shape[0] if tree_shape else B
    ctx = M.mtp_init(M.make_config(cfg.H, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.ffn, cfg.vocab, cfg.eps,
                                   cfg.rope_theta, cfg.dtype, max_batch, max(K, 2), cfg.block_size,
                                   int(lens.max()) + (K + 1) * total + 8,
                                   weight_format=args.weights), wdev)
    kv = M.KVCache(dev(kv0.k_pool), dev(kv0.v_pool), dev(kv0.block_table), dev(kv0.seq_len), dev(kv0.pending))
    lp = M.SpecLoop(ctx, B, K, thr, out_cap=(K + 1) * total, conf_threshold=args.conf_threshold)
    tree = None
    if tree_shape:
        tree = M.TreeDraft(ctx, B, tree_shape[0], tree_shape[1], tree_shape[2], kv0.block_table.shape[1],
                           dev(scratch))
        lp.target_logits = torch.zeros((B * (1 + tree_shape[2]), cfg.vocab), dtype=lp.target_logits.dtype,
                                       device="cuda")

    def run_loop(n):
        if tree is not None:
            M.mtp_tree_loop(ctx, kv, lp, tree, n)
        else:
            M.mtp_spec_loop(ctx, kv, lp, n)
    h0 = synth.loop_start_hashes(cfg, B)
    last0 = synth.uniform_int(cfg.seed, 95, (B,), 0, cfg.vocab)
    lp.seq_hash.copy_(torch.from_numpy(h0.view(np.int64)).cuda())
    lp.last_tok.copy_(dev(last0))
    lp.positions.copy_(dev(lens.astype(np.int32)))
    lp.embeds.copy_(dev(w["embed"][last0]))
    # the first step's hidden state: any value (the loop writes the verifier's from then on)
    lp.hidden.copy_(dev(synth.make_draft_inputs(cfg, w, lens).hidden))
    stream = torch.cuda.current_stream()

    run_loop(args.warmup)
    torch.cuda.synchronize()
    assert M.mtp_get_device_error(ctx) == 0
    n0 = int(lp.out_len.sum().item())
    launches0 = M.mtp_launch_count(ctx)
    sampler = ClockSampler(gpu_id_for_smi(local_rank)) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    run_loop(args.steps)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    launches = M.mtp_launch_count(ctx) - launches0
    ms = reduce_max(t0.elapsed_time(t1), world)
    emitted = int(lp.out_len.sum().item()) - n0
    assert M.mtp_get_device_error(ctx) == 0

    # LM-head launches timed on the library's stream (separate pass)
    nprof = max(5, args.steps // 4)
    M.mtp_profile_begin(ctx, M.MTP_KERNEL_LM_HEAD, nprof * K)
    run_loop(nprof)
    torch.cuda.synchronize()
    lm_ms = M.mtp_profile_end(ctx, nprof * K)

    # end to end: one host read of the emitted counts per step (synchronising)
    ne = max(5, args.steps // 4)
    h_len = torch.empty(B, dtype=torch.int32).pin_memory()
    e0 = int(lp.out_len.sum().item())
    te = time.perf_counter()
    for _ in range(ne):
        run_loop(1)
        h_len.copy_(lp.out_len, non_blocking=True)
        torch.cuda.synchronize()
    te = time.perf_counter() - te
    e_emitted = int(h_len.sum().item()) - e0
    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    fmt = args.weights
    lm_bytes = kernel_bytes(cfg, lens, K, with_logits=bool(tree_shape or args.conf_threshold > 0),
                            fmt=fmt)["lm_head"]
    lm_gbs = lm_bytes / (statistics.mean(lm_ms) * 1e-3) / 1e9
    value = world * emitted / (ms * 1e-3)
    line = {
        "metric": LOOP_METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": cfg.dtype if fmt == "dense" else "int4/int8 weights, f32 arithmetic, bf16 KV",
        "data": "synthetic (copy-head weights, deterministic synthetic verifier)",
        "config": {"workload": "spec_loop_" + cfg.name, "batch": B, "draft_steps_K": K,
                   "sticky_alpha": args.loop_alpha, "weights": fmt, "conf_threshold": args.conf_threshold,
                   "tree": ({"branching_factor": tree_shape[0], "tree_depth": tree_shape[1],
                             "num_assistant_tokens": tree_shape[2]} if tree_shape else None),
                   "mean_emitted_per_step": emitted / (B * args.steps),
                   "l2": "inputs larger than L2 (weights streamed every draft step)"},
        "roofline": {"kernel": "lm_head_argmax" if fmt == "dense" else "lm_head_argmax_int8", "bound": "hbm",
                     "achieved": lm_gbs, "peak": peak, "unit": "GB/s", "frac": lm_gbs / peak,
                     "peak_source": peak_kind + " hbm_gbs", "traffic": None, "launches_timed": len(lm_ms),
                     "bytes_per_launch": lm_bytes},
        "e2e": {"value": world * e_emitted / te, "unit": "tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 4 * B},
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline and tree_shape is None:
        line["cpu_baseline"] = loop_cpu_baseline(cfg, w, lens, h0, last0, thr, fmt)
    print(json.dumps(line), flush=True)


def loop_cpu_baseline(cfg, w, lens, h0, last0, thr, fmt) -> dict:
    """One step of the oracle's speculative loop on the same state."""
    import oracle as O
    import oracle.loop as OL
    W = oracle_head(cfg, w, fmt)
    kv = synth.make_kv(cfg, lens, extra_slots=cfg.K + 1)
    st = OL.LoopState([int(x) for x in h0], [int(x) for x in last0], [int(x) for x in lens],
                      [[] for _ in range(len(lens))])
    dense = None if fmt == "dense" else (lambda ids: O.widen(w["embed"][np.asarray(ids)], cfg.dtype))
    t = time.perf_counter()
    OL.spec_loop(W, kv, st, cfg.K, thr, 1, cfg.dtype, embed_rows=dense)
    dt = time.perf_counter() - t
    n = sum(len(o) for o in st.out)
    return {"value": n / dt, "unit": "tok/s", "cores": blas_threads(), "nproc": os.cpu_count(), "kind": "oracle",
            "sample": "1 loop step (K=%d draft steps, verifier rows, verify, commit), B=%d, float64 numpy" %
                      (cfg.K, len(lens))}


VERIFY_METRIC = "MTP verify + KV commit calls/s (64 requests, K_b uniform 1..8); % HBM roofline"


def run_verify_workload(args, cfg, rank, world, local_rank):
    """The verify + rollback workload (no draft head): one call is mtp_verify
    over the ragged target-logit rows followed by mtp_kv_commit_accepted
    (extra=1).  Verify and commit are timed separately and together with
    CUDA events around each call; seq_len and pending are restored after
    every call, outside the events."""
    import torch
    torch.cuda.set_device(local_rank)
    import mtp_self_speculative_gb300 as M
    import oracle as O
    vi = synth.make_verify_inputs(cfg)
    lens = synth.context_lengths(cfg)
    kv0 = synth.make_kv(cfg, lens, extra_slots=int(vi.num_drafts.max()) + 1, prefill_slots=lens + vi.num_drafts)
    kv0.pending = vi.num_drafts.astype(np.int32).copy()
    B = len(lens)

    def dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(a).cuda()
    ctx = M.mtp_init(M.make_config(1, cfg.n_q, cfg.n_kv, cfg.head_dim, 8, cfg.vocab, dtype=cfg.dtype, max_batch=B,
                                   max_k=vi.max_k, block_size=cfg.block_size))
    kv = M.KVCache(dev(kv0.k_pool), dev(kv0.v_pool), dev(kv0.block_table), dev(kv0.seq_len), dev(kv0.pending))
    seq0, pend0 = dev(kv0.seq_len), dev(kv0.pending)
    logits, ro, drafts, nd = dev(vi.logits), dev(vi.row_offsets), dev(vi.drafts), dev(vi.num_drafts)
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    bon = torch.empty(B, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")  # larger than L2

    def reset():
        kv.seq_len.copy_(seq0)
        kv.pending.copy_(pend0)
        l2_flush(flush)  # the 111 MB of logits would otherwise stay in the 126 MB L2

    for _ in range(args.warmup):
        M.mtp_verify(ctx, logits, ro, drafts, nd, acc, bon)
        M.mtp_kv_commit_accepted(ctx, kv, acc, extra=1)
        reset()
    torch.cuda.synchronize()
    assert M.mtp_get_device_error(ctx) == 0
    acc_o, bon_o = O.verify(vi.logits, vi.row_offsets, vi.drafts, vi.num_drafts, cfg.dtype)
    assert np.array_equal(acc.cpu().numpy(), acc_o) and np.array_equal(bon.cpu().numpy(), bon_o)

    n = min(args.steps, 1000)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    launches0 = M.mtp_launch_count(ctx)
    sampler = ClockSampler(gpu_id_for_smi(local_rank)) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    for i in range(n):
        ev[i][0].record(stream)
        M.mtp_verify(ctx, logits, ro, drafts, nd, acc, bon)
        ev[i][1].record(stream)
        M.mtp_kv_commit_accepted(ctx, kv, acc, extra=1)
        ev[i][2].record(stream)
        reset()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    launches = (M.mtp_launch_count(ctx) - launches0) / n
    t_ver = [e[0].elapsed_time(e[1]) for e in ev]
    t_com = [e[1].elapsed_time(e[2]) for e in ev]
    t_all = statistics.median([a + b for a, b in zip(t_ver, t_com)])
    t_all = reduce_max(t_all, world)
    # end to end: host logits copied in, accepted counts and bonus ids read back
    h_logits = logits.cpu().pin_memory()
    h_acc = torch.empty_like(acc, device="cpu").pin_memory()
    h_bon = torch.empty_like(bon, device="cpu").pin_memory()
    ne = max(5, min(n // 10, 50))
    t0 = time.perf_counter()
    for _ in range(ne):
        logits.copy_(h_logits, non_blocking=True)
        M.mtp_verify(ctx, logits, ro, drafts, nd, acc, bon)
        M.mtp_kv_commit_accepted(ctx, kv, acc, extra=1)
        h_acc.copy_(acc, non_blocking=True)
        h_bon.copy_(bon, non_blocking=True)
        stream.synchronize()
        reset()
    e2e_s = (time.perf_counter() - t0) / ne
    assert M.mtp_get_device_error(ctx) == 0
    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["hbm_gbs"])
    ver_bytes = int(vi.row_offsets[-1]) * cfg.vocab * cfg.elem_bytes
    kv_row = 2 * cfg.n_kv * cfg.head_dim * cfg.elem_bytes
    com_bytes = int(np.sum(vi.num_drafts - np.minimum(acc_o + 1, vi.num_drafts))) * kv_row
    tv = statistics.median(t_ver)
    ver_gbs = ver_bytes / (tv * 1e-3) / 1e9
    world_calls = world / (t_all * 1e-3)
    # the oracle as it stands on the host: the same verify + commit
    kv_c = kv0.copy()
    t = time.perf_counter()
    reps = 0
    while reps < 3 or time.perf_counter() - t < 2.0:
        O.verify(vi.logits, vi.row_offsets, vi.drafts, vi.num_drafts, cfg.dtype)
        kv_c = kv0.copy()
        O.kv_commit(kv_c, np.minimum(acc_o + 1, vi.num_drafts), cfg.dtype)
        reps += 1
    cpu = reps / (time.perf_counter() - t)
    line = {
        "metric": VERIFY_METRIC, "value": world_calls, "unit": "calls/s", "n_gpus": world, "steps": n,
        "warmup": args.warmup, "ms_per_step": t_all, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic (seeded N(0,1) logits with planted spikes)",
        "config": {"workload": cfg.name, "batch": B, "k_range": [int(vi.num_drafts.min()), int(vi.num_drafts.max())],
                   "vocab": cfg.vocab, "verify_rows": int(vi.row_offsets[-1]), "context": int(lens[0]),
                   "l2": "L2 flushed between calls (256 MB read, outside the timed events); "
                         "%.1f MB of logits per call" % (ver_bytes / 1e6)},
        "verify_ms": tv, "commit_ms": statistics.median(t_com),
        "roofline": {"kernel": "verify", "bound": "hbm", "achieved": ver_gbs, "peak": peak, "unit": "GB/s",
                     "frac": ver_gbs / peak, "peak_source": peak_kind + " hbm_gbs",
                     "traffic": VERIFY_TRAFFIC.get(cfg.name), "bytes_per_launch": ver_bytes},
        "commit_bytes": com_bytes,
        "read_floor": read_floor_us({"verify": ver_bytes}, stream)["verify"],
        "e2e": {"value": 1.0 / e2e_s, "unit": "calls/s", "h2d_bytes_per_step": ver_bytes,
                "d2h_bytes_per_step": 2 * B * 4},
        "gpu_launches": launches,
        "cpu_baseline": {"value": cpu, "unit": "calls/s", "cores": blas_threads(), "nproc": os.cpu_count(), "kind": "oracle",
                         "sample": "%d full call(s): float64 numpy verify + commit of the same inputs" % reps},
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def oracle_head(cfg: synth.MTPShape, w, fmt: str):
    """The oracle's weights for the bench's weight format."""
    import oracle as O
    if fmt == "int4_g64":
        from oracle import quant
        return quant.quantized_weights(w, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)
    return O.MTPWeights64.from_stored(w, cfg.dtype, cfg.n_q, cfg.n_kv, cfg.head_dim, cfg.eps, cfg.rope_theta)


def cpu_baseline(cfg: synth.MTPShape, sample_steps: int = 1, fmt: str = "dense", gpu_ids=None, gpu_logits=None):
    """The float64 oracle as it stands, one full step (K draft steps, verify,
    commit) for the same workload on the host cores.  With the GPU's first
    draft (ids [B, K], logits [B, K, V]) of the same inputs, also returns the
    draft parity of that call: exact-id matches step by step while the two
    free-running chains agree, the near-ties among them, and the worst
    normwise logit error."""
    import oracle as O
    w = synth.make_weights(cfg, norm="ones")
    lens = synth.context_lengths(cfg)
    kv = synth.make_kv(cfg, lens, extra_slots=cfg.K + 1)
    di = synth.make_draft_inputs(cfg, w, lens)
    W = oracle_head(cfg, w, fmt)
    vi = synth.make_verify_inputs(synth.shrink(cfg, k_lo=0, k_hi=0), num_drafts=np.full(len(lens), cfg.K, np.int32))
    t = time.perf_counter()
    for _ in range(sample_steps):
        res = O.draft(W, O.widen(di.hidden, cfg.dtype), O.widen(di.embeds, cfg.dtype), di.positions, kv, cfg.K)
        acc, _ = O.verify(vi.logits, vi.row_offsets, res.ids, vi.num_drafts, cfg.dtype)
        O.kv_commit(kv, np.minimum(acc + 1, cfg.K), cfg.dtype)
        O.kv_truncate(kv, lens, cfg.dtype)
    dt = (time.perf_counter() - t) / sample_steps
    cb = {"value": 1.0 / dt, "unit": "steps/s", "cores": blas_threads(), "nproc": os.cpu_count(), "kind": "oracle",
          "sample": "%d full step(s): %d draft steps + verify + commit, B=%d, float64 numpy" %
                    (sample_steps, cfg.K, len(lens))}
    if gpu_ids is None:
        return cb
    z = res.logits
    compared = exact = near = 0
    worst = 0.0
    for b in range(len(lens)):
        for k in range(cfg.K):
            zo = z[b, k]
            scale = float(np.max(np.abs(zo)))
            worst = max(worst, float(np.max(np.abs(gpu_logits[b, k].astype(np.float64) - zo))) / scale)
            compared += 1
            exact += int(gpu_ids[b, k] == res.ids[b, k])
            near += int(O.top2_gap(zo[None])[0] < 2e-2 * scale)
            if gpu_ids[b, k] != res.ids[b, k]:
                break            # the chains now follow different tokens
    parity = {"compared_steps": compared, "exact_ids": exact, "oracle_near_ties": near,
              "max_logit_rel_err": worst, "tolerance": 2e-2,
              "note": "GPU free-running draft vs the float64 oracle on the same inputs; steps compared "
                      "until the first id difference"}
    return cb, parity


def reference_budget_s() -> float:
    return float(os.environ.get("MTP_REFERENCE_BUDGET_S", "150"))


def run_reference_verify(args, cfg, world):
    """Reference arm of the verify workload: the oracle's verify + commit of
    the same inputs, one call per step, on this arm's metric and config."""
    import oracle as O
    vi = synth.make_verify_inputs(cfg)
    lens = synth.context_lengths(cfg)
    kv0 = synth.make_kv(cfg, lens, extra_slots=int(vi.num_drafts.max()) + 1, prefill_slots=lens + vi.num_drafts)
    kv0.pending = vi.num_drafts.astype(np.int32).copy()
    B = len(lens)
    ver_bytes = int(vi.row_offsets[-1]) * cfg.vocab * cfg.elem_bytes

    def call():
        kv_c = kv0.copy()
        t = time.perf_counter()
        acc, _ = O.verify(vi.logits, vi.row_offsets, vi.drafts, vi.num_drafts, cfg.dtype)
        O.kv_commit(kv_c, np.minimum(acc + 1, vi.num_drafts), cfg.dtype)
        return time.perf_counter() - t

    t_start = time.perf_counter()
    for _ in range(min(args.warmup, 1)):
        call()
    times = []
    for _ in range(args.steps):
        times.append(call())
        if time.perf_counter() - t_start > reference_budget_s():
            break
    per_call = statistics.mean(times)
    value = 1.0 / per_call
    line = {"impl": "reference", "metric": VERIFY_METRIC, "value": value, "unit": "calls/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_call * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) logits with planted spikes)",
            "config": {"workload": cfg.name, "batch": B, "k_range": [int(vi.num_drafts.min()), int(vi.num_drafts.max())],
                       "vocab": cfg.vocab, "verify_rows": int(vi.row_offsets[-1]), "context": int(lens[0]),
                       "l2": "L2 flushed between calls (256 MB read, outside the timed events); "
                             "%.1f MB of logits per call" % (ver_bytes / 1e6)},
            "cpu_baseline": {"value": value, "unit": "calls/s", "cores": blas_threads(), "nproc": os.cpu_count(), "kind": "oracle",
                             "sample": "%d full call(s): float64 numpy verify + commit of the same inputs%s" %
                                       (len(times), "; capped by the time budget" if len(times) < args.steps else "")},
            "e2e": {"value": value, "unit": "calls/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "samples_run": len(times)}
    print(json.dumps(line), flush=True)


def run_reference_loop(args, cfg, world):
    """Reference arm of the speculative loop: the oracle's loop (chain,
    confidence stop or tree drafting, as selected) on the same copy-head
    weights and synthetic verifier, one loop iteration per step."""
    import oracle as O
    import oracle.loop as OL
    import oracle.tree as OT
    B, K = cfg.batch, cfg.K
    lens = synth.context_lengths(cfg)
    w = synth.copy_head(cfg, synth.make_weights(cfg, norm="ones"))
    thr = int(args.loop_alpha * 2 ** 53)
    tree_shape = tuple(int(x) for x in args.tree.split(",")) if args.tree else None
    if tree_shape:
        K = tree_shape[1]
    W = oracle_head(cfg, w, args.weights)
    total = args.steps + 2
    kv = synth.make_kv(cfg, lens, extra_slots=(K + 1) * total + K + 1)
    st = OL.LoopState([int(x) for x in synth.loop_start_hashes(cfg, B)],
                      [int(x) for x in synth.uniform_int(cfg.seed, 95, (B,), 0, cfg.vocab)], [int(x) for x in lens],
                      [[] for _ in range(B)])
    dense = None if args.weights == "dense" else (lambda ids: O.widen(w["embed"][np.asarray(ids)], cfg.dtype))
    conf = args.conf_threshold if args.conf_threshold > 0 else None

    def one():
        n0 = sum(len(o) for o in st.out)
        t = time.perf_counter()
        if tree_shape:
            OT.tree_spec_loop(W, kv, st, tree_shape[0], tree_shape[1], tree_shape[2], thr, 1, cfg.dtype,
                              embed_rows=dense)
        else:
            OL.spec_loop(W, kv, st, K, thr, 1, cfg.dtype, embed_rows=dense, conf_tau=conf)
        return time.perf_counter() - t, sum(len(o) for o in st.out) - n0

    t_start = time.perf_counter()
    for _ in range(min(args.warmup, 1)):
        one()
    dts, toks = [], 0
    for _ in range(args.steps):
        dt, n = one()
        dts.append(dt)
        toks += n
        if time.perf_counter() - t_start > reference_budget_s():
            break
    value = toks / sum(dts)
    line = {"impl": "reference", "metric": LOOP_METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(dts) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (copy-head weights, deterministic synthetic verifier)",
            "config": {"workload": "spec_loop_" + cfg.name, "batch": B, "draft_steps_K": K,
                       "sticky_alpha": args.loop_alpha, "weights": args.weights,
                       "conf_threshold": args.conf_threshold,
                       "tree": ({"branching_factor": tree_shape[0], "tree_depth": tree_shape[1],
                                 "num_assistant_tokens": tree_shape[2]} if tree_shape else None),
                       "mean_emitted_per_step": toks / (B * len(dts)),
                       "l2": "inputs larger than L2 (weights streamed every draft step)"},
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": blas_threads(), "nproc": os.cpu_count(), "kind": "oracle",
                             "sample": "%d loop iteration(s) of the float64 numpy oracle%s" %
                                       (len(dts), "; capped by the time budget" if len(dts) < args.steps else "")},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "samples_run": len(dts)}
    print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The oracle timed as the reference arm.  A step is sampled as one of
    the K draft steps (the decoder layer, LM head and argmax for the whole
    batch) plus one K-th of the verify rows; the full step is K such samples.
    The number of samples is capped so the run stays within a few minutes.
    The verify workload and the speculative loop have arms of their own."""
    if rank != 0:
        return
    import oracle as O
    cfg = WORKLOADS[args.workload]
    if cfg.H == 0:
        return run_reference_verify(args, cfg, world)
    if args.loop:
        return run_reference_loop(args, cfg, world)
    w = synth.make_weights(cfg, norm="ones")
    lens = synth.context_lengths(cfg)
    kv = synth.make_kv(cfg, lens, extra_slots=cfg.K + 1)
    di = synth.make_draft_inputs(cfg, w, lens)
    W = oracle_head(cfg, w, args.weights)
    vi = synth.make_verify_inputs(synth.shrink(cfg, k_lo=0, k_hi=0), num_drafts=np.full(len(lens), cfg.K, np.int32))
    hid, emb = O.widen(di.hidden, cfg.dtype), O.widen(di.embeds, cfg.dtype)

    def sample():
        res = O.draft(W, hid, emb, di.positions, kv, 1)
        O.kv_rollback(kv, cfg.dtype)
        O.verify(vi.logits, vi.row_offsets, np.repeat(res.ids, cfg.K, axis=1), vi.num_drafts, cfg.dtype)

    budget = reference_budget_s()
    t_start = time.perf_counter()
    for _ in range(min(args.warmup, 1)):
        sample()
    times = []
    for i in range(args.steps):
        t = time.perf_counter()
        sample()
        times.append(time.perf_counter() - t)
        if time.perf_counter() - t_start > budget:
            break
    # one sample is one draft step plus verify (verify is counted K times; it is
    # under 1% of the sample), so a full step costs K samples
    per_step = cfg.K * statistics.mean(times)
    value = 1.0 / per_step
    cores = blas_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "batch": len(lens), "draft_steps_K": cfg.K},
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": cores, "nproc": os.cpu_count(), "kind": "oracle",
                             "sample": "%d sampled draft step(s) of the float64 numpy oracle (decoder layer, "
                                       "LM head, argmax, verify), scaled by K=%d to a full step%s" %
                                       (len(times), cfg.K, "; capped by the time budget" if len(times) < args.steps
                                        else "")},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "samples_run": len(times)}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--persistent-max-batch", type=int, default=0,
                    help="largest batch for the persistent draft kernel (0: never, the library default)")
    ap.add_argument("--weights", choices=["dense", "int4_g64"], default="dense",
                    help="weight format of the head: dense (the workload's dtype) or the quantized format "
                         "(int4 group-64 projections, int8 per-row embedding / LM head)")
    ap.add_argument("--loop", action="store_true",
                    help="time the full speculative loop (mtp_spec_loop with the synthetic verifier) instead")
    ap.add_argument("--loop-alpha", type=float, default=0.8,
                    help="probability that the synthetic verifier repeats the last token (--loop)")
    ap.add_argument("--conf-threshold", type=float, default=0.0,
                    help="with --loop: propose only the leading drafts whose probability exceeds it (0: off)")
    ap.add_argument("--tree", default=None,
                    help="with --loop: tree drafting 'branching_factor,tree_depth,num_assistant_tokens'")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other configurations measured after the headline workload")
    ap.add_argument("--ctx", type=int, default=None,
                    help="override the committed MTP context length (smaller cases for profiling)")
    ap.add_argument("--lm-traffic", type=float, default=None,
                    help="ncu dram bytes per LM-head launch of the current kernel, if captured")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    if args.ctx is not None:
        import dataclasses
        WORKLOADS[args.workload] = dataclasses.replace(WORKLOADS[args.workload], ctx_lo=args.ctx, ctx_hi=args.ctx)
    rank, world, local_rank = rank_info()
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "ours":
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
