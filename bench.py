"""Benchmark of the sparse MLA attention forward on GB300.

One step = one smla_fwd_ws call over the whole workload (every step of the hot
path: work setup, gather, dequant, QK^T, softmax, PV, epilogue, and the
combine when the plan splits the top-k range) with inputs resident in HBM.

Headline workload: the bf16 prefill shape — one 8192-token sequence, h=128
heads, d_qk=576, d_v=512, topk=2048, token i selecting min(i+1, 2048)
distinct slots of [0, i] — the h=128 / topk=2048 case whose compute roofline
is the tensor cores.  The decode shape (T=64, h=128, topk=2048, 2 M-slot bf16
pool) is reported beside it under "secondary".

Metric: TFLOP/s with FLOPs = sum_t 2 * h * v_t * (d_qk + d_v) over the actual
valid counts v_t, plus query-tokens/s; `value` is the whole-job TFLOP/s over
all ranks.  N > 1 (torchrun): every rank runs its own copy of the workload
(independent problems, no data-path collective), so scaling is weak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_mla_attention_02_gb300 import workloads as W  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                  "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024
FLUSH_BYTES = 256 * 1024 * 1024     # written between cold-L2 steps (> L2)
METRIC = ("sparse MLA fwd TFLOP/s & query-tokens/s at h=128 topk=2048; "
          "% of roofline")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def flops_of(w) -> float:
    v = w.valid_len.to(torch.float64).clamp(0, w.topk)
    return float(2.0 * w.h * (w.d_qk + w.d_v) * v.sum().item())


def row_bytes(w) -> int:
    if w.kv_dtype == W.KV_FP8_DS_MLA:
        return 656                      # 512 E4M3 + 4 fp32 scales + 64 bf16
    return 2 * w.d_qk if w.kv_dtype == W.KV_BF16 else w.d_qk


def bytes_model(w):
    """Algorithmic bytes: per-token terms (q, O, LSE, indices, valid) plus the
    selected rows once per token (G) or once overall (U)."""
    G = (w.d_qk + 127) // 128
    scale_b = 4 * G if w.kv_dtype == W.KV_FP8_E4M3_GROUP128 else \
        16 if w.kv_dtype == W.KV_FP8_E4M3_GROUP4_KPE else 0
    per_tok = w.T * (2 * w.h * w.d_qk + 2 * w.h * w.d_v + 4 * w.h
                     + 4 * w.topk + 4)
    v = w.valid_len.clamp(0, w.topk)
    gathered = int(v.sum().item()) * (row_bytes(w) + scale_b)
    mask = torch.arange(w.topk, device=w.indices.device)[None, :] < v[:, None]
    uniq = int(torch.unique(w.indices[mask & (w.indices >= 0)]).numel())
    return per_tok + uniq * (row_bytes(w) + scale_b), per_tok + gathered


# The sources each kernel is built from: a traffic figure measured on a
# kernel stays valid while these files are unchanged.
KERNEL_SOURCES = {
    "tc_heads": ("smla_tc.cu", "tc_common.cuh", "tc_ptx.cuh", "smla_internal.h"),
    "tc_keys": ("smla_tc_keys.cu", "tc_common.cuh", "tc_ptx.cuh", "smla_internal.h"),
    "tc_keys_fp8": ("smla_tc_fp8.cu", "tc_common.cuh", "tc_ptx.cuh", "smla_internal.h"),
    "cache_write": ("smla_cache.cu", "smla_internal.h"),
}


def sources_digest(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "sparse_mla_attention_02_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary
    (profiles/traffic.json), if it was taken on the current sources of that
    kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            e = json.load(f)[workload]
        if e.get("kernel") == kernel and e.get("sources_sha") == sources_digest(kernel):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except Exception:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        loaded = [s for s in sm if mx and s >= 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def workload_seed(name: str, rank: int) -> int:
    """Each rank draws its own replica of the workload (independent problems,
    weak scaling): same recipe, a different seed per rank."""
    return 1000 + list(W.CONFIGS).index(name) + 7919 * rank


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's time (the job is done when every rank is done)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, steps: int, t_max: float) -> float:
    """Whole-job rate: every rank's units over the slowest rank's time."""
    return world * units_per_rank * steps / t_max


def time_steps(fn, steps, stream):
    """K steps back to back on `stream`, timed with CUDA events there (a
    step may find its inputs in L2 from the step before: warm L2)."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3


def time_steps_cold(fn, steps, stream, flush):
    """K steps, each after `flush` (a buffer larger than L2) was written on
    `stream`, so that every step starts with a cold L2; each step alone is
    timed with CUDA events on `stream` (the flush is outside), and the times
    are summed."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
    evs[-1][1].synchronize()
    return sum(a.elapsed_time(b) for a, b in evs) / 1e3


def run_ours(args, rank, world, local_rank):
    import sparse_mla_attention_02_gb300 as smla
    import torch.distributed as dist
    from sparse_mla_attention_02_gb300 import build
    build.build()
    smla.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    pk, pk_src = peaks()

    def setup(name, rank_, tokens=0):
        w = W.CONFIGS[name](device=dev, seed=workload_seed(name, rank_))
        if tokens and tokens < w.T:
            # the last `tokens` tokens (same kernel, a smaller launch)
            w = W.token_subset(w, np.arange(w.T - tokens, w.T), device=dev)
        n = smla.smla_workspace_size(w.T, w.h, w.d_qk, w.topk, w.kv_dtype)
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
        out = torch.empty((w.T, w.h, w.d_v), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((w.T, w.h), dtype=torch.float32, device=dev)
        return w, ws, out, lse, n

    def step_fn(w, ws, out, lse):
        def f():
            smla.smla_fwd_ws(w.q, w.kv, w.kv_dtype, w.k_scale, w.indices,
                             w.valid_len, w.sm_scale, ws, out=out, lse=lse,
                             num_slots=w.num_slots, stream=stream)
        return f

    def barrier():
        if world > 1:
            dist.barrier()

    def ranks_max(x):
        return max_over_ranks(x, world, dev)

    def cache_write_bench():
        """The group-quantizing E4M3 cache write: 131072 token rows
        [kv_c | k_pe] (bf16, 151 MB) to random slots of a 262144-slot cache;
        per row 1152 B read + 576 B codes + 20 B scales written + 4 B slot
        id (1752 B), more than L2 per launch."""
        Ncw, Scw = 131072, 262144
        gcw = torch.Generator(device=dev).manual_seed(4242 + 7919 * rank)
        kv_c = torch.randn((Ncw, 512), generator=gcw, device=dev).to(torch.bfloat16)
        k_pe = torch.randn((Ncw, 64), generator=gcw, device=dev).to(torch.bfloat16)
        slots = torch.randperm(Scw, generator=gcw, device=dev)[:Ncw].int().contiguous()
        cache = torch.empty((Scw, 576), dtype=torch.uint8, device=dev)
        scales = torch.empty((Scw, 5), dtype=torch.float32, device=dev)

        def f4():
            smla.smla_cache_write_e4m3_group(kv_c, k_pe, slots, cache, scales, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                f4()
        stream.synchronize()
        barrier()
        k4 = max(args.steps, 20)
        t4 = ranks_max(time_steps(f4, k4, stream)) / k4
        b4 = Ncw * (2 * 576 + 576 + 4 * 5 + 4)
        res = {
            "rows_per_s": round(world * Ncw / t4, 1),
            "ms_per_step": round(1e3 * t4, 4),
            "hbm_gbs": round(b4 / t4 / 1e9, 1),
            "frac_hbm": round(b4 / t4 / 1e9 / pk["hbm_gbs"], 4),
            "bytes_per_row": 1752,
            "bytes_per_launch": b4,
            "traffic": ncu_traffic("fp8_group_cache_write", "cache_write"),
            "kernel": "smla_cache_write_kernel",
        }
        del kv_c, k_pe, slots, cache, scales
        torch.cuda.empty_cache()
        return res

    if args.cache_write_only:
        res = cache_write_bench()
        if rank == 0:
            print(json.dumps({"config": "fp8_group_cache_write", **res}))
        return

    # ---- headline: bf16 prefill --------------------------------------------
    w, ws, out, lse, ws_n = setup(args.config, rank, args.tokens)
    fl = flops_of(w)
    U, G = bytes_model(w)
    f = step_fn(w, ws, out, lse)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            f()
    stream.synchronize()
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as cs:
        elapsed = time_steps(f, args.steps, stream)
        torch.cuda.synchronize(dev)
    barrier()
    clocks = cs.summary()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    cold_el = ranks_max(time_steps_cold(f, args.steps, stream, flush))
    t_max = ranks_max(elapsed)
    ms = 1e3 * t_max / args.steps
    launches_per_step = 1 + (1 if ws_n > 0 else 0)
    value = job_throughput(fl, world, args.steps, t_max) / 1e12
    tok_s = job_throughput(w.T, world, args.steps, t_max)
    kernel_s = elapsed / args.steps
    achieved = fl / kernel_s / 1e12
    bound_tensor = fl / (pk["bf16_tflops"] * 1e12) >= U / (pk["hbm_gbs"] * 1e9)
    roof = {
        "kernel": "smla_fwd main kernel" + (" + combine" if ws_n else ""),
        "bound": "tensor" if bound_tensor else "hbm",
        "achieved": round(achieved if bound_tensor else U / kernel_s / 1e9, 3),
        "peak": pk["bf16_tflops"] if bound_tensor else pk["hbm_gbs"],
        "unit": "TFLOP/s" if bound_tensor else "GB/s",
        "peak_source": f"{pk_src} ({'bf16 burst' if bound_tensor else 'copy'})",
        "traffic": ncu_traffic(args.config, smla.smla_plan_info(
            w.T, w.h, w.d_qk, w.topk, w.kv_dtype)["kernel"]),
        "algorithmic_flops_per_launch": fl,
        "algorithmic_bytes_per_launch": {"U": U, "G": G},
    }
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["ms_per_step_cold_l2"] = round(1e3 * cold_el / args.steps, 4)
    roof["frac_of_sustained"] = round(achieved / pk["bf16_tflops_sustained"], 4) \
        if bound_tensor else None

    if args.main_only:
        if rank == 0:
            print(json.dumps({"config": args.config, "T": w.T,
                              "ms_per_step": round(ms, 4),
                              "ms_per_step_cold_l2": round(1e3 * cold_el / args.steps, 4),
                              "tflops": round(value, 3),
                              "gbs_G": round(G / (elapsed / args.steps) / 1e9, 1),
                              "kernel": smla.smla_plan_info(w.T, w.h, w.d_qk, w.topk,
                                                            w.kv_dtype)["kernel"],
                              "flops_per_launch": fl, "U": U, "G": G}), flush=True)
        return

    # ---- e2e: host buffers, copies inside the timed region -----------------
    h_q = torch.empty(w.q.shape, dtype=w.q.dtype, pin_memory=True)
    h_q.copy_(w.q)
    h_idx = torch.empty(w.indices.shape, dtype=torch.int32, pin_memory=True)
    h_idx.copy_(w.indices)
    h_vl = torch.empty(w.valid_len.shape, dtype=torch.int32, pin_memory=True)
    h_vl.copy_(w.valid_len)
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h_lse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    # smla_fwd_host: the public entry point for host-resident tensors; it
    # copies each chunk of tokens in, runs the forward and copies the results
    # out, with the three overlapped (its device staging is the workspace).
    host_ws = torch.empty(
        max(1, smla.smla_fwd_host_workspace_size(w.T, w.h, w.d_qk, w.topk,
                                                 w.kv_dtype, w.d_v)),
        dtype=torch.uint8, device=w.kv.device)

    def e2e_step():
        smla.smla_fwd_host(h_q, w.kv, w.kv_dtype, w.k_scale, h_idx, h_vl,
                           w.sm_scale, out=h_out, lse=h_lse,
                           num_slots=w.num_slots, workspace=host_ws,
                           stream=stream)
    e2e_step()
    stream.synchronize()
    e2e_steps = max(3, args.steps // 2)
    barrier()
    e2e_el = ranks_max(time_steps(e2e_step, e2e_steps, stream))
    h2d = h_q.numel() * 2 + h_idx.numel() * 4 + h_vl.numel() * 4
    d2h = h_out.numel() * 2 + h_lse.numel() * 4
    e2e = {"value": round(world * fl * e2e_steps / e2e_el / 1e12, 3),
           "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h,
           "tokens_per_s": round(world * w.T * e2e_steps / e2e_el, 1),
           "ms_per_step": round(1e3 * e2e_el / e2e_steps, 3),
           "resident": "kv cache (model state); q, indices, valid_len copied in, "
                       "O and LSE copied out each step",
           "api": "smla_fwd_host (pinned host buffers; copies of chunk i+1 in "
                  "and chunk i-1 out overlap the forward of chunk i)"}
    del h_q, h_idx, h_vl, h_out, h_lse, host_ws

    # ---- cpu baseline: the oracle on a bounded sample (rank 0, N=1) ---------
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w, args.cpu_seconds)

    del w, ws, out, lse
    torch.cuda.empty_cache()

    # ---- secondary: bf16 decode ----------------------------------------------
    secondary = {}
    if not args.no_secondary:
        for name in ["bf16_decode", "fp8_nope_decode", "mixed_fp8_group", "ds_mla_decode"]:
            w2, ws2, out2, lse2, n2 = setup(name, rank)
            f2 = step_fn(w2, ws2, out2, lse2)
            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    f2()
            stream.synchronize()
            barrier()
            k2 = max(args.steps, 20) if name != "mixed_fp8_group" else max(3, args.steps)
            el2 = ranks_max(time_steps(f2, k2, stream))
            cold2 = ranks_max(time_steps_cold(f2, k2, stream, flush))
            fl2 = flops_of(w2)
            U2, G2 = bytes_model(w2)
            t2, tc2 = el2 / k2, cold2 / k2
            roof2 = max(fl2 / (pk["bf16_tflops"] * 1e12), U2 / (pk["hbm_gbs"] * 1e9))
            secondary[name] = {
                "tflops": round(world * fl2 / t2 / 1e12, 3),
                "tokens_per_s": round(world * w2.T / t2, 1),
                "ms_per_step": round(1e3 * t2, 4),
                "ms_per_step_cold_l2": round(1e3 * tc2, 4),
                "hbm_gbs_U": round(U2 / t2 / 1e9, 1),
                "frac_hbm_U": round(U2 / t2 / 1e9 / pk["hbm_gbs"], 4),
                "roofline_frac": round(roof2 / t2, 4),
                "roofline_frac_cold_l2": round(roof2 / tc2, 4),
                # gathered bytes (every selected row once per token) per second
                "hbm_gbs_G": round(G2 / t2 / 1e9, 1),
                "frac_hbm_G": round(G2 / t2 / 1e9 / pk["hbm_gbs"], 4),
                "frac_hbm_G_cold_l2": round(G2 / tc2 / 1e9 / pk["hbm_gbs"], 4),
                "bytes_per_launch": {"U": U2, "G": G2},
                "traffic": ncu_traffic(name, smla.smla_plan_info(
                    w2.T, w2.h, w2.d_qk, w2.topk, w2.kv_dtype)["kernel"]),
                "splits_workspace_bytes": n2,
                "kernel": smla.smla_plan_info(w2.T, w2.h, w2.d_qk, w2.topk,
                                              w2.kv_dtype)["kernel"],
            }
            if rank == 0 and world == 1 and not args.no_cpu:
                secondary[name]["cpu_baseline"] = cpu_baseline(w2, args.cpu_seconds / 3)
            if name == "bf16_decode":
                # The same decode step on request-local positions through
                # smla_fwd_paged: request r's 32768-slot context as 512
                # blocks of 64 (block_table[r, page] = 512 r + page); the
                # translation runs inside the kernel's slot-id load.
                per_req, bs = w2.num_slots // w2.T, 64
                req = torch.arange(w2.T, dtype=torch.int32, device=dev)
                table = (torch.arange(w2.T, device=dev)[:, None] * (per_req // bs) +
                         torch.arange(per_req // bs, device=dev)[None, :]).int().contiguous()
                local = torch.where(w2.indices >= 0,
                                    w2.indices - req[:, None] * per_req,
                                    w2.indices).int().contiguous()

                def f3():
                    smla.smla_fwd_paged(w2.q, w2.kv, w2.kv_dtype, w2.k_scale, local,
                                        req, table, bs, w2.sm_scale,
                                        valid_len=w2.valid_len, out=out2, lse=lse2,
                                        num_slots=w2.num_slots,
                                        workspace=ws2 if n2 > 0 else None,
                                        stream=stream)
                with torch.cuda.stream(stream):
                    for _ in range(args.warmup):
                        f3()
                stream.synchronize()
                barrier()
                el3 = ranks_max(time_steps(f3, k2, stream))
                t3 = el3 / k2
                secondary["bf16_decode_paged"] = {
                    "tflops": round(world * fl2 / t3 / 1e12, 3),
                    "tokens_per_s": round(world * w2.T / t3, 1),
                    "ms_per_step": round(1e3 * t3, 4),
                    "vs_global_indices": round(t2 / t3, 4),
                    "kernel": "as bf16_decode, request-local indices + block table",
                }
            del w2, ws2, out2, lse2
            torch.cuda.empty_cache()

        secondary["fp8_group_cache_write"] = cache_write_bench()
    del flush

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; shapes and selection structure of the "
                    "pages' workloads)",
            "config": {"workload": f"{args.config}: T=8192 h=128 d_qk=576 "
                                   "d_v=512 topk=2048, valid=min(i+1,2048), "
                                   "8192-slot bf16 pool",
                       "T": 8192, "h": 128, "topk": 2048, "kv": "bf16",
                       "l2": "inputs larger than L2 (q 1.21 GB, O 1.07 GB); "
                             "the 9.4 MB pool is L2-resident by nature",
                       "parallelism": f"replicas x{world} (independent problems)"},
            "tokens_per_s": round(tok_s, 1),
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "secondary": secondary,
        }
        print(json.dumps(line), flush=True)


def _oracle_inputs(sub):
    q = sub.q.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    if sub.kv.dtype == torch.bfloat16:
        kv = sub.kv.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    else:
        kv = sub.kv.contiguous().cpu().numpy()
    ks = None if sub.k_scale is None else sub.k_scale.cpu().numpy()
    return q, kv, ks, sub.indices.cpu().numpy(), sub.valid_len.cpu().numpy()


def oracle_sample_rate(w, seconds, rng_seed=0):
    """Run the oracle on growing token samples until one takes >= seconds/4,
    then on a sample sized for ~seconds.  Returns (TFLOP/s, tokens/s, n, s)."""
    import oracle
    T = w.T
    cores = oracle.default_threads()
    n = max(cores, 8)
    while True:
        sel = np.unique(np.linspace(0, T - 1, min(n, T)).astype(np.int64))
        sub = W.token_subset(w, sel)
        q, kv, ks, idx, vl = _oracle_inputs(sub)
        t0 = time.perf_counter()
        oracle.sparse_mla_fwd(q, kv, sub.kv_dtype, ks, idx, vl, sub.sm_scale,
                              num_slots=sub.num_slots, n_threads=cores)
        dt = time.perf_counter() - t0
        fl = flops_of(sub)
        if dt >= seconds / 4 or len(sel) >= T:
            if dt < seconds / 2 and len(sel) < T:
                n = int(n * min(8.0, seconds / max(dt, 1e-3)))
                continue
            return fl / dt / 1e12, len(sel) / dt, len(sel), dt, cores
        n = int(n * min(8.0, max(2.0, seconds / 4 / max(dt, 1e-3))))


def cpu_baseline(w, seconds):
    """The oracle as it stands (never tuned for this), on the host cores,
    over an evenly spaced token sample of the same workload sized for about
    `seconds` of CPU work."""
    tf, tok, n, dt, cores = oracle_sample_rate(w, seconds)
    return {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle", "tokens_per_s": round(tok, 3),
            "sample": f"{n} of {w.T} tokens evenly spaced over the sequence "
                      f"(all heads, their own valid counts), {dt:.1f} s, fp64 "
                      f"C oracle on {cores} threads"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step is the fp64 CPU oracle on a
    bounded token sample of the same workload (rank 0 only)."""
    if rank != 0:
        return
    w = W.CONFIGS[args.config](device="cpu", seed=1003)
    import oracle
    cores = oracle.default_threads()
    T = w.T
    n = args.ref_tokens
    sel = np.unique(np.linspace(T // 4, T - 1, n).astype(np.int64))
    sub = W.token_subset(w, sel)
    q, kv, ks, idx, vl = _oracle_inputs(sub)
    fl = flops_of(sub)

    def step():
        oracle.sparse_mla_fwd(q, kv, sub.kv_dtype, ks, idx, vl, sub.sm_scale,
                              num_slots=sub.num_slots, n_threads=cores)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = fl * args.steps / dt / 1e12
    sample = (f"{len(sel)} of {T} tokens evenly spaced over the last 3/4 of "
              f"the sequence per step, fp64 C oracle on {cores} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6),
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": f"{args.config}: T={T} h={w.h} d_qk={w.d_qk} "
                               f"d_v={w.d_v} topk={w.topk} (token sample, see "
                               "cpu_baseline)"},
        "tokens_per_s": round(len(sel) * args.steps / dt, 3),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s",
                         "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def spawn_ranks(args) -> int:
    """--gpus N > 1 without a launcher: start N ranks (one per GPU) with
    torch.distributed.run on this node and return its exit code; refuse when
    fewer than N GPUs are visible (never report fewer GPUs than asked)."""
    if args.impl == "ours":
        n = torch.cuda.device_count()
        if n < args.gpus:
            print(f"bench.py: --gpus {args.gpus} requested, {n} GPU(s) visible",
                  file=sys.stderr)
            return 2
    import socket
    sk = socket.socket()
    sk.bind(("127.0.0.1", 0))
    port = sk.getsockname()[1]
    sk.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="bf16_prefill")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-tokens", type=int, default=32)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--tokens", type=int, default=0,
                    help="use only the last N tokens of the config (profiling)")
    ap.add_argument("--main-only", action="store_true",
                    help="time only the main step loop (profiling)")
    ap.add_argument("--cache-write-only", action="store_true",
                    help="time only the E4M3 group cache write (profiling)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(spawn_ranks(args))
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
        sys.exit(2)
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) \
            else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend)
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
