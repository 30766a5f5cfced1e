"""Benchmark of the hot path: one streaming step = quantize-append of a new
chunk into the INT2 window cache, rotation of the current chunk, and the
Jensen-bias-corrected chunk attention with P_S / P_R (all through libkvq).

Default workload: one layer, 24 heads, head_dim 128, a 4680-token chunk
(3 latent frames x 30 x 52) over a 4-chunk (18720-token) INT2 g32 window --
the configuration the headline metric is quoted on.  Synthetic inputs.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on a
bounded sample of the same workload instead.

Multi-GPU: heads are independent, so each rank runs its own full workload
(weak scaling, no collective on the data path); the step time is the max over
ranks and the value the sum of all ranks' FLOPs over that time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "corrected INT2-KV chunk-attention TFLOP/s and % of roofline; quantize GB/s"
UNIT = "TFLOP/s"
CORR_NAMES = {0: "none", 1: "taylor", 2: "exact"}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p.get("hbm_gbs", 6800.0), p.get("bf16_tflops", 1900.0), \
            p.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def _workload(name):
    from quantized_kv_cache_quantize_gb300 import synth
    return synth.WORKLOADS[name]


def _config(w, extra=None):
    cfg = {"workload": f"{w.name}: {w.heads} heads, head_dim {w.head_dim}, chunk {w.chunk_tokens} "
                       f"tokens (queries = current keys), window {w.n_chunks} chunks = {w.n_s} "
                       f"tokens INT{w.bits} g{w.group}, batch {w.batch}",
           "step": "quantize-append 1 chunk + rotate current chunk + corrected attention with "
                   "P_S/P_R"}
    if extra:
        cfg.update(extra)
    return cfg


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def kernel_source_hash() -> str:
    """First 16 hex digits of the SHA-256 of the attention kernel's source
    (the kernel templates, the headers they include and the unit that
    instantiates the default mode)."""
    h = hashlib.sha256()
    for name in ("kvq_attn_kernel.cuh", "kvq_attn.cu", "kvq_sm100.cuh", "kvq_checks.cuh",
                 "kvq_fwht.cuh", "kvq_tmap.cuh"):
        with open(os.path.join(ROOT, "quantized_kv_cache_quantize_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _traffic_for_current_kernel():
    """DRAM bytes per attention launch from the committed ncu summary, or
    None when the kernel source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "attn_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    h = kernel_source_hash()
    if rec.get("source_sha256_16") != h:
        return None
    return rec.get("dram_bytes_per_launch_full")


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (a step time): the whole job is as
    slow as its slowest rank.  One all-reduce; a no-op on one rank."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def check_world(gpus: int, env=None):
    """--gpus N must match the number of ranks the launcher started (one
    process per GPU: ``torchrun --nproc-per-node N bench.py --gpus N``); a
    plain ``python bench.py`` is one rank.  A mismatch would time a different
    number of replicas than the line reports, so it stops the run."""
    env = os.environ if env is None else env
    world = int(env.get("WORLD_SIZE", "1"))
    if gpus != world:
        sys.stderr.write(f"bench.py: --gpus {gpus} but {world} rank(s) were launched; run "
                         f"`python -m torch.distributed.run --nproc-per-node {gpus} bench.py "
                         f"--gpus {gpus}` (one process per GPU)\n")
        raise SystemExit(2)
    return world


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from quantized_kv_cache_quantize_gb300 import kvq, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = _workload(args.workload)
    x = synth.inputs(w, seed=args.seed)
    signs = synth.hadamard_signs(w.head_dim, seed=args.seed)
    B, H, d = w.batch, w.heads, w.head_dim

    cache = kvq.KVCache(B, H, d, w.bits, w.group, w.chunk_tokens, w.n_chunks, signs, device=dev,
                        key_mode=args.key_mode)
    kwin, vwin = x["k_win"].to(dev), x["v_win"].to(dev)
    for c in range(w.n_chunks):
        sl = slice(c * w.chunk_tokens, (c + 1) * w.chunk_tokens)
        kvq.quantize_append(cache, kwin[:, :, sl].contiguous(), vwin[:, :, sl].contiguous())
    del kwin, vwin
    q, kc, vc = x["q"].to(dev), x["k_cur"].to(dev), x["v_cur"].to(dev)
    kn, vn = x["k_new"].to(dev), x["v_new"].to(dev)
    out = torch.empty_like(q)
    ps = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
    pr = torch.empty_like(ps)
    ws = torch.empty(cache.workspace_bytes(w.n_q, w.n_r), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kvq.quantize_append(cache, kn, vn, stream=stream)
        kvq.lib().kvq_attention_corrected(
            kvq.ctypes.byref(cache.struct), kvq._ptr(q), kvq._ptr(kc), kvq._ptr(vc), w.n_q, w.n_r,
            kvq.ctypes.c_float(w.scale), args.corr, args.flags, kvq._ptr(ws), ws.numel(),
            kvq._ptr(out), kvq._ptr(ps), kvq._ptr(pr), kvq._stream(stream))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert kvq.last_device_status() == 0

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    kvq.profile_begin()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = kvq.profile_kernel_launches()
    prof = kvq.profile_end()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ms_step = e0.elapsed_time(e1) / args.steps
    status = kvq.last_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    ms_max = max_over_ranks(ms_step, world, dev)
    flops = w.attention_flops()
    value = flops * world / (ms_max * 1e-3) / 1e12

    # per-kernel device times inside the timed region (CUDA events on the launch stream)
    k3_ms = prof["attention"]["ms_total"] / max(1, prof["attention"]["launches"])
    # per step: the per-channel key mode appends with two launches (values per
    # token, keys per channel)
    k1_ms = prof["quantize_append"]["ms_total"] / args.steps
    k2_ms = prof["rotate"]["ms_total"] / max(1, prof["rotate"]["launches"])
    hbm, bf16_burst, bf16_sust, peak_kind = _peaks()
    k3_tflops = flops / (k3_ms * 1e-3) / 1e12
    # the timed loop runs back to back for ~seconds: the sustained (power-capped) peak applies
    # when the region is long, the burst peak otherwise
    region_s = ms_step * args.steps / 1e3
    peak = bf16_sust if region_s >= 1.0 else bf16_burst
    q_bytes = w.append_bytes()
    k1_gbs = q_bytes / (k1_ms * 1e-3) / 1e9
    # the rotation kernel reads the BF16 query and current values and writes
    # them as FP16, and the query's FP16 remainder whenever the precise split
    # may run: with the flag, or in the per-head automatic choice (head_dim
    # 128, per-token keys, Taylor or no correction, no one-CTA flag)
    auto = (d == 128 and args.key_mode == 0 and args.corr != 2 and not args.flags & 4)
    rot_bytes = (w.n_q + w.n_r) * d * B * H * 4.0 + \
        (w.n_q * d * B * H * 2.0 if (args.flags & 1 or auto) else 0.0)
    # in the automatic choice the same timed scope holds the per-head selection
    # pass: it reads the window's (step, zero) words and the BF16 query
    if auto:
        rot_bytes += w.n_s * (d // w.group) * 4.0 * B * H + w.n_q * d * 2.0 * B * H

    # end to end through the public API with host buffers (pinned), copies inside the timed
    # region.  Serving-style pipeline: step i's inputs are copied in on one stream while
    # step i-1 computes, and its results are copied out on a third stream; device buffers
    # are double-buffered and every hand-off is an event.
    host = {k: x[k].pin_memory() for k in ("q", "k_cur", "v_cur", "k_new", "v_new")}
    dev_in = [{k: torch.empty_like(host[k], device=dev) for k in host} for _ in range(2)]
    dev_out = [(torch.empty_like(out), torch.empty_like(ps), torch.empty_like(pr)) for _ in range(2)]
    host_out = [(torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                 torch.empty(ps.shape, dtype=ps.dtype).pin_memory(),
                 torch.empty(pr.shape, dtype=pr.dtype).pin_memory()) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for b_ in range(2):   # every event recorded once so the first waits are satisfied
        ev_done[b_].record(stream)
        ev_out[b_].record(stream)

    def e2e_step(i):
        b_ = i & 1
        di, (o_d, ps_d, pr_d), (o_h, ps_h, pr_h) = dev_in[b_], dev_out[b_], host_out[b_]
        s_in.wait_event(ev_done[b_])          # step i-2 has finished reading these inputs
        with torch.cuda.stream(s_in):
            for k in host:
                di[k].copy_(host[k], non_blocking=True)
        ev_in[b_].record(s_in)
        stream.wait_event(ev_in[b_])
        stream.wait_event(ev_out[b_])         # step i-2's results have left these buffers
        kvq.quantize_append(cache, di["k_new"], di["v_new"], stream=stream)
        kvq.lib().kvq_attention_corrected(
            kvq.ctypes.byref(cache.struct), kvq._ptr(di["q"]), kvq._ptr(di["k_cur"]),
            kvq._ptr(di["v_cur"]), w.n_q, w.n_r, kvq.ctypes.c_float(w.scale),
            args.corr, args.flags, kvq._ptr(ws), ws.numel(), kvq._ptr(o_d), kvq._ptr(ps_d),
            kvq._ptr(pr_d), kvq._stream(stream))
        ev_done[b_].record(stream)
        s_out.wait_event(ev_done[b_])
        with torch.cuda.stream(s_out):
            o_h.copy_(o_d, non_blocking=True)
            ps_h.copy_(ps_d, non_blocking=True)
            pr_h.copy_(pr_d, non_blocking=True)
        ev_out[b_].record(s_out)

    e2e_steps = max(3, min(args.steps, 50))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)

    result = None
    if rank == 0:
        cpu = cpu_baseline(w, args) if (world == 1 and not args.no_cpu_baseline) else None
        others = None
        if world == 1 and not args.no_other_configs:
            others = other_configs(dev, bf16_burst, hbm)
        acc = None
        if not args.no_accuracy:
            same = w.name in ACCURACY_WORKLOADS and args.seed == 0
            acc = accuracy_report(x if same else synth.inputs(_workload("w4_int2")), dev)
        ws_bytes = (w.append_bytes() + 2 * w.n_s * d * w.bits / 8 * B * H
                    + 3 * w.n_q * d * 2 * B * H)
        result = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp16 MMA operands / fp32 accumulate over an INT2 cache (BF16 I/O)",
            "data": "synthetic (seeded; video-shaped token counts; random K/V/Q with outlier "
                    "channels)",
            "config": _config(w, {
                "l2": f"inputs larger than L2: {ws_bytes / 1e6:.0f} MB read per step vs 129 MB L2",
                "parallelism": f"replicas x{world} (heads independent, no collective)",
                "correction": CORR_NAMES[args.corr], "flags": args.flags,
                "keys": "per channel over 128-token blocks" if args.key_mode else
                        "per token and group"}),
            "clocks": clk,
            "e2e": {"value": round(flops * world / (e2e_ms * 1e-3) / 1e12, 3), "unit": UNIT,
                    "ms_per_step": round(e2e_ms, 4),
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "schedule": "copy-in, compute and copy-out on three streams, device "
                                "buffers double-buffered (step i's copies overlap step i-1)"},
            "gpu_launches": launches,
            "kernels_ms": {"quantize_append": round(k1_ms, 5), "rotate": round(k2_ms, 5),
                           "attention": round(k3_ms, 5)},
            "quantize_gbs": round(k1_gbs, 1),
            "quantize_frac_of_hbm": round(k1_gbs / hbm, 4),
            "rotate_gbs": round(rot_bytes / (k2_ms * 1e-3) / 1e9, 1),
            "rotate_frac_of_hbm": round(rot_bytes / (k2_ms * 1e-3) / 1e9 / hbm, 4),
            "rotate_scope": "rotation of Q and V_R" + (" + per-head selection pass" if auto else ""),
            "roofline": {"bound": "tensor", "achieved": round(k3_tflops, 2),
                         "peak": peak, "unit": "TFLOP/s", "frac": round(k3_tflops / peak, 4),
                         "peak_source": f"{peak_kind} bf16 "
                                        f"{'sustained' if peak == bf16_sust else 'burst'} "
                                        "(FP16 dense rate = BF16 rate)",
                         "traffic": _traffic_for_current_kernel(),
                         "kernel": "attention (fused corrected chunk attention)"},
            "cpu_baseline": cpu,
            "accuracy": acc,
            "other_configs": others,
        }
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return result


ACCURACY_REFS = os.path.join(ROOT, "tests", "golden", "accuracy_w4.npz")
ACCURACY_WORKLOADS = ("w4_int2", "w4_int4")


def _input_fingerprint(x: dict, h: int) -> str:
    """SHA-256 over the BF16 bit patterns of head h's q, k_cur, v_cur, k_win,
    v_win (as fp32, an exact widening): the key the stored answers carry."""
    fp = hashlib.sha256()
    for k in ("q", "k_cur", "v_cur", "k_win", "v_win"):
        fp.update(x[k][0, h].float().numpy().tobytes())
    return fp.hexdigest()


def accuracy_report(x, dev, reps: int = 10):
    """INT2 g32 against INT4 g64 on the same seeded inputs (24 heads, head_dim
    128, 4680-token chunk, 18720-token window): for each cache and each
    correction mode, the CUDA path's O and P_S / P_R on the sampled heads and
    rows against the oracle's stored answers (tests/golden/accuracy_w4.npz,
    written from the oracle alone by tests/golden/make_accuracy_refs.py), the
    mean attention mass on the cache and its shift from the unquantized
    window ("Quantized Keys Steal Attention": abstract, section 1, Figure 2),
    and the attention's throughput with the default (Taylor) correction.
    ``x``: the workload's seeded BF16 inputs (both caches use the same ones)."""
    import numpy as np
    import torch

    from quantized_kv_cache_quantize_gb300 import kvq, synth

    if not os.path.exists(ACCURACY_REFS):
        return {"unavailable": "tests/golden/accuracy_w4.npz not found"}
    z = np.load(ACCURACY_REFS)
    signs = synth.hadamard_signs(128)
    q, kc, vc = x["q"].to(dev), x["k_cur"].to(dev), x["v_cur"].to(dev)
    rep = {"refs": "tests/golden/accuracy_w4.npz (oracle answers on sampled heads and rows)",
           "metrics": "err_o = max|O - O_oracle| / max|O_oracle|; err_ps, err_pr = max abs "
                      "error of the masses; ps_mean = mean P_S on the sampled rows; shift = "
                      "ps_mean - the oracle's mean P_S over the unquantized BF16 window"}
    for name in ACCURACY_WORKLOADS:
        w = synth.WORKLOADS[name]
        heads, rows = z[f"{name}/heads"], z[f"{name}/rows"]
        entry = {"cache": f"INT{w.bits} g{w.group}",
                 "heads": [int(h) for h in heads], "rows_per_head": int(len(rows))}
        match = all(_input_fingerprint(x, int(h)) == str(z[f"{name}/fp"][i])
                    for i, h in enumerate(heads))
        entry["inputs_match_refs"] = bool(match)
        cache = kvq.KVCache(w.batch, w.heads, w.head_dim, w.bits, w.group, w.chunk_tokens,
                            w.n_chunks, signs, device=dev)
        kw, vw = x["k_win"].to(dev), x["v_win"].to(dev)
        for c in range(w.n_chunks):
            sl = slice(c * w.chunk_tokens, (c + 1) * w.chunk_tokens)
            kvq.quantize_append(cache, kw[:, :, sl].contiguous(), vw[:, :, sl].contiguous())
        del kw, vw
        ps_u = z[f"{name}/ps_unquantized"]
        entry["ps_unquantized_mean"] = round(float(ps_u.mean()), 6)
        for cname, corr in (("none", kvq.CORR_NONE), ("taylor", kvq.CORR_TAYLOR),
                            ("exact", kvq.CORR_EXACT)):
            out, ps, pr = kvq.attention_corrected(cache, q, kc, vc, corr=corr, with_mass=True)
            torch.cuda.synchronize()
            if kvq.last_device_status() != 0:
                raise RuntimeError(f"device status after the {name} {cname} accuracy call")
            idx = torch.as_tensor(rows, device=dev)
            o_g = out[0][:, idx][torch.as_tensor(heads, device=dev)].float().cpu().numpy()
            ps_g = ps[0][:, idx][torch.as_tensor(heads, device=dev)].cpu().numpy().astype(np.float64)
            pr_g = pr[0][:, idx][torch.as_tensor(heads, device=dev)].cpu().numpy().astype(np.float64)
            o_r = z[f"{name}/o_{cname}"].astype(np.float64)
            entry[cname] = {
                "err_o": float(f"{np.abs(o_g - o_r).max() / np.abs(o_r).max():.3e}"),
                "err_ps": float(f"{np.abs(ps_g - z[f'{name}/ps_{cname}']).max():.3e}"),
                "err_pr": float(f"{np.abs(pr_g - z[f'{name}/pr_{cname}']).max():.3e}"),
                "ps_mean": round(float(ps_g.mean()), 6),
                "shift": round(float(ps_g.mean() - ps_u.mean()), 6),
            }
        # throughput of the default call (Taylor correction) on this cache
        out = torch.empty_like(q)
        ps = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
        pr = torch.empty_like(ps)
        ws = torch.empty(cache.workspace_bytes(w.n_q, w.n_r), dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream(dev)

        def call():
            kvq.lib().kvq_attention_corrected(
                kvq.ctypes.byref(cache.struct), kvq._ptr(q), kvq._ptr(kc), kvq._ptr(vc), w.n_q,
                w.n_r, kvq.ctypes.c_float(w.scale), kvq.CORR_TAYLOR, 0, kvq._ptr(ws), ws.numel(),
                kvq._ptr(out), kvq._ptr(ps), kvq._ptr(pr), kvq._stream(stream))

        for _ in range(3):
            call()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        entry["attention_ms"] = round(ms, 4)
        entry["attention_tflops"] = round(w.attention_flops() / (ms * 1e-3) / 1e12, 2)
        entry["cache_mb"] = round(w.batch * w.heads * w.n_s * 2 *
                                  (w.head_dim * w.bits / 8 + 4 * w.head_dim / w.group) / 1e6, 2)
        rep[name] = entry
        del cache
    return rep


OTHER_WORKLOADS = ("w8_int2", "hires_t3")


def other_configs(dev, peak: float, hbm: float, reps: int = 5):
    """The larger configurations in one line each (default call: Taylor
    term, per-head choice of the precise split): the attention call's
    device time (CUDA events, `reps` calls after 2 untimed ones) and the
    quantize-append of one chunk, on the workloads' seeded inputs."""
    import torch

    from quantized_kv_cache_quantize_gb300 import kvq, synth

    out_rep = {}
    for name in OTHER_WORKLOADS:
        w = synth.WORKLOADS[name]
        x = synth.inputs(w)
        signs = synth.hadamard_signs(w.head_dim)
        cache = kvq.KVCache(w.batch, w.heads, w.head_dim, w.bits, w.group, w.chunk_tokens,
                            w.n_chunks, signs, device=dev)
        kw, vw = x["k_win"].to(dev), x["v_win"].to(dev)
        for c in range(w.n_chunks):
            sl = slice(c * w.chunk_tokens, (c + 1) * w.chunk_tokens)
            kvq.quantize_append(cache, kw[:, :, sl].contiguous(), vw[:, :, sl].contiguous())
        del kw, vw
        q, kc, vc = x["q"].to(dev), x["k_cur"].to(dev), x["v_cur"].to(dev)
        kn, vn = x["k_new"].to(dev), x["v_new"].to(dev)
        out = torch.empty_like(q)
        ps = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
        pr = torch.empty_like(ps)
        ws = torch.empty(cache.workspace_bytes(w.n_q, w.n_r), dtype=torch.uint8, device=dev)
        stream = torch.cuda.current_stream(dev)

        def attn():
            kvq.lib().kvq_attention_corrected(
                kvq.ctypes.byref(cache.struct), kvq._ptr(q), kvq._ptr(kc), kvq._ptr(vc), w.n_q,
                w.n_r, kvq.ctypes.c_float(w.scale), kvq.CORR_TAYLOR, 0, kvq._ptr(ws), ws.numel(),
                kvq._ptr(out), kvq._ptr(ps), kvq._ptr(pr), kvq._stream(stream))

        def timed(fn, n):
            for _ in range(2):
                fn()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / n

        a_ms = timed(attn, reps)
        q_ms = timed(lambda: kvq.quantize_append(cache, kn, vn, stream=stream), max(reps, 10))
        if kvq.last_device_status() != 0:
            raise RuntimeError(f"device status after the {name} runs")
        flops = w.attention_flops()
        out_rep[name] = {
            "workload": _config(w)["workload"],
            "attention_ms": round(a_ms, 4),
            "attention_tflops": round(flops / (a_ms * 1e-3) / 1e12, 2),
            "attention_frac": round(flops / (a_ms * 1e-3) / 1e12 / peak, 4),
            "quantize_append_us": round(q_ms * 1e3, 2),
            "quantize_gbs": round(w.append_bytes() / (q_ms * 1e-3) / 1e9, 1),
            "quantize_frac_of_hbm": round(w.append_bytes() / (q_ms * 1e-3) / 1e9 / hbm, 4),
        }
        del cache, x, q, kc, vc, kn, vn, out, ps, pr, ws
        torch.cuda.empty_cache()
    out_rep["timing"] = (f"attention: CUDA events around {reps} calls after 2 untimed ones "
                         "(bias term counted, burst peak); quantize-append: one chunk, 10 calls")
    return out_rep


def _oracle_sample(w, head: int, rows: int, seed: int, corr: int = 1, key_mode: int = 0):
    """One bounded sample of the step on the CPU oracle, for one head.

    As on the GPU, the window is already cached when the step starts: its
    quantization (earlier appends) is done before the clock starts.  Timed:
    the quantize-append of the head's new chunk (K and V), the dequantization
    of the cached window, and the corrected attention of ``rows`` query rows
    over the window and the current chunk.  The attention's cost is linear in
    the query rows, so the head's step time is estimated as the fixed part
    plus the sampled rows' time times n_q / rows (exact when rows = n_q).

    Returns (attention FLOPs of the head's n_q rows, estimated step time of
    the head, wall time spent in the timed parts)."""
    import numpy as np

    from oracle import kvq_oracle as O
    from quantized_kv_cache_quantize_gb300 import synth
    x = synth.head_inputs(w, head, seed=seed)
    s = synth.hadamard_signs(w.head_dim, seed=seed)
    rows = max(1, min(rows, w.n_q))
    # the cached window (not timed)
    _, vd, vz, _, vcod = O.quantize_rows(x["v_win"].float().numpy(), s, w.bits, w.group)
    if key_mode:
        kf = x["k_win"].float().numpy()
        kparts = [O.quantize_key_chunk(kf[c0:c0 + w.chunk_tokens], s, w.bits)
                  for c0 in range(0, kf.shape[0], w.chunk_tokens)]
    else:
        _, kd, kz, _, kc = O.quantize_rows(x["k_win"].float().numpy(), s, w.bits, w.group)
    q = x["q"].float().numpy()[:rows]
    k_cur, v_cur = x["k_cur"].float().numpy(), x["v_cur"].float().numpy()
    # the step: append the new chunk, dequantize the window, attend
    t0 = time.perf_counter()
    O.quantize_rows(x["v_new"].float().numpy(), s, w.bits, w.group)
    if key_mode:
        # per-channel keys: the chunk per channel over 128-token blocks
        O.quantize_key_chunk(x["k_new"].float().numpy(), s, w.bits)
        k_hat = np.concatenate([O.dequantize_key_channels(c[4], c[1], c[2]) for c in kparts])
        k_steps = np.concatenate([O.key_channel_token_steps(c[1], c[4].shape[0]) for c in kparts])
        group = 1
    else:
        O.quantize_rows(x["k_new"].float().numpy(), s, w.bits, w.group)
        k_hat, k_steps, group = O.dequantize(kc, kd, kz, w.group), kd, w.group
    v_hat = O.dequantize(vcod, vd, vz, w.group)
    t1 = time.perf_counter()
    O.chunk_attention(q, k_hat, v_hat, k_steps, k_cur, v_cur, s, w.scale, group, corr)
    t2 = time.perf_counter()
    t_step = (t1 - t0) + (t2 - t1) * (w.n_q / rows)
    return w.attention_flops(heads=1), t_step, t2 - t0


def _cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count()


def cpu_baseline(w, args):
    """Oracle throughput on a bounded sample: heads are run one after
    another until ``--cpu-seconds`` of wall time have been spent (at least
    one head, at most all of them), each with ``--cpu-rows`` query rows (the
    whole chunk by default) and its step time estimated as in
    ``_oracle_sample``."""
    # the oracle's exact correction evaluates log(sinh a / a) per channel and
    # score: its default sample is 128 query rows per head instead of the chunk
    rows = min(args.cpu_rows, w.n_q) if args.cpu_rows > 0 else (128 if args.corr == 2 else w.n_q)
    # one untimed warm-up sample (first-touch page faults, BLAS thread start)
    _oracle_sample(w, 0, min(rows, 128), args.seed, args.corr, args.key_mode)
    tot_f, tot_t, wall, heads = 0.0, 0.0, 0.0, 0
    while heads < w.heads and (heads == 0 or wall < args.cpu_seconds):
        f, t_step, t_wall = _oracle_sample(w, heads, rows, args.seed, args.corr, args.key_mode)
        tot_f += f
        tot_t += t_step
        wall += t_wall
        heads += 1
    return {"value": round(tot_f / tot_t / 1e12, 6), "unit": UNIT, "cores": _cores(),
            "kind": "oracle",
            "sample": f"{heads} head(s) of {w.name} with the window already cached (its "
                      f"quantization not timed), each: oracle quantize-append of the new chunk "
                      f"(K,V), dequantization of the {w.n_s}-token window and corrected "
                      f"attention of {rows} of {w.n_q} query rows over {w.n_s} cached + "
                      f"{w.n_r} current keys; value = the heads' attention FLOPs / their step "
                      f"time (sampled rows scaled to {w.n_q}; {wall:.1f} s of CPU work)"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    w = _workload(args.workload)
    rows = args.ref_rows
    for _ in range(args.warmup):
        _oracle_sample(w, 0, rows, args.seed, args.corr, args.key_mode)
    tot_f, tot_t, wall = 0.0, 0.0, 0.0
    for k in range(args.steps):
        f, t_step, t_wall = _oracle_sample(w, k % w.heads, rows, args.seed, args.corr,
                                           args.key_mode)
        tot_f += f
        tot_t += t_step
        wall += t_wall
    value = tot_f / tot_t / 1e12
    sample = (f"per step one head of {w.name} with the window already cached (its quantization "
              f"not timed): oracle quantize-append of the new chunk (K and V), dequantization of "
              f"the {w.n_s}-token window and corrected attention of {rows} of {w.n_q} query rows "
              f"over {w.n_s} cached + {w.n_r} current keys; value = the head's attention FLOPs "
              f"/ its step time with the rows' time scaled to {w.n_q} rows "
              f"({tot_t / args.steps * 1e3:.0f} ms per head); ms_per_step = wall time of one "
              f"sampled step")
    result = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(wall / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (fp32 quantizer)",
        "data": "synthetic (seeded)", "config": _config(w),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": _cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)
    return result


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="w4_int2")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="wall-time budget of the oracle CPU baseline sample")
    ap.add_argument("--cpu-rows", type=int, default=0,
                    help="query rows per head of the cpu_baseline sample (0: the whole chunk)")
    ap.add_argument("--ref-rows", type=int, default=128,
                    help="query rows per step of the --impl reference sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the one-line timings of the 32-head long-window and the 40-head "
                         "high-resolution workloads")
    ap.add_argument("--no-accuracy", action="store_true",
                    help="skip the INT2 g32 / INT4 g64 accuracy report (CUDA path against the "
                         "oracle's stored answers, attention-mass shift, throughput)")
    ap.add_argument("--precise-query", action="store_true",
                    help="split the rotated query into FP16 high + low parts")
    ap.add_argument("--staged-words", action="store_true",
                    help="stage the cached tiles' packed words into shared memory with TMA bulk "
                         "copies (head_dim 128, INT2 g32; for comparisons)")
    ap.add_argument("--one-cta", action="store_true",
                    help="run the one-CTA attention kernel where the SM-pair kernel applies "
                         "(for comparisons)")
    ap.add_argument("--keys", choices=["token", "channel"], default="token",
                    help="key quantization: per token and group (default) or per channel over "
                         "128-token blocks of each chunk (KIVI-style)")
    ap.add_argument("--corr", choices=["taylor", "exact", "none"], default="taylor",
                    help="correction of the cached scores (default: the second-order Taylor "
                         "term; exact: log(sinh a / a) per channel)")
    args = ap.parse_args(argv)
    check_world(args.gpus)
    args.warmup = max(3, args.warmup)   # at least 3 untimed warm-up steps
    args.corr = {v: k for k, v in CORR_NAMES.items()}[args.corr]
    args.flags = (1 if args.precise_query else 0) | (4 if args.one_cta else 0) | \
        (8 if args.staged_words else 0)
    args.key_mode = 1 if args.keys == "channel" else 0
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    main()
