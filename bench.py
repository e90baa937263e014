"""Forward-pass throughput of the nanochat-style GPT on B300 through the nc C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload d12] [--impl ours|reference]

One step = one nc_forward over a [B, T] batch of synthetic tokens (every kernel of the hot
path).  `value` = tokens/s over all ranks with inputs already in HBM; `e2e` = the same metric
through nc_forward_host (pinned host tokens in, host logits out, copies inside the timed
region).  The dominant kernel's roofline numbers come from CUDA events recorded around every
launch on the launching stream during the timed region.  `--impl reference` times the fp64
CPU oracle (the only reference this path has) on a bounded sample of the same workload.
Under torchrun each rank runs an independent replica (the forward needs no collective).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "forward tokens/sec at d12 T=2048 on 1 B300; % of BF16 tensor-core peak"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The largest of the ranks' times: the job ends with its slowest rank (an all-reduce MAX
    over the default process group when world > 1)."""
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, units_per_rank: float, ms: float) -> float:
    """Units per second over the whole job: every rank processes units_per_rank (a replica of the
    full workload, weak scaling) within the slowest rank's ms."""
    return world * units_per_rank / (ms / 1000.0)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def window_pairs(T: int, W: int) -> int:
    """Visible (query, key) pairs of one head over one row: sum_i min(i+1, W+1) (W < 0: full)."""
    if W < 0 or W >= T:
        return T * (T + 1) // 2
    return (W + 1) * (W + 2) // 2 + (T - W - 1) * (W + 1)


def decode_step_bytes(cfg, B: int, pos: int):
    """Algorithmic bytes of one decode step at position pos: every weight once (the packed q|k|v
    with its gate rows, the out-projection, fc, down projection, the lm_head; bf16) and the cached
    keys and values each layer attends to (positions max(0, pos - W) .. pos - 1; the new position's
    come from the step itself).  Returns (weight bytes, cache bytes)."""
    H, Hkv, D, C, F, L, V = (cfg.n_head, cfg.n_kv_head, cfg.head_dim, cfg.n_embd, cfg.mlp_hidden, cfg.n_layer,
                             cfg.vocab_size)
    w = 2 * (sum(((H + 2 * Hkv) * D + (Hkv * 16 if cfg.has_ve[i] else 0)) * C + C * H * D + 2 * F * C
                 for i in range(L)) + V * C)
    kv = sum(B * (pos - (0 if cfg.window_left[i] < 0 else max(0, pos - cfg.window_left[i]))) * Hkv * D * 2 * 2
             for i in range(L))
    return w, kv


def kernel_work(cfg, B: int, T: int):
    """Algorithmic work per launch of each kernel class (FLOPs for contractions, bytes otherwise)."""
    M = B * T
    C, H, Hkv, D, F, V, L = (cfg.n_embd, cfg.n_head, cfg.n_kv_head, cfg.head_dim, cfg.mlp_hidden,
                             cfg.vocab_size, cfg.n_layer)
    attn_flops = sum(4 * D * H * B * window_pairs(T, cfg.window_left[i]) for i in range(L)) / L
    return {
        "qkv_rope_qknorm_ve": ("tensor", 2.0 * M * C * (H + 2 * Hkv) * D),
        "attention": ("tensor", attn_flops),
        "oproj_residual": ("tensor", 2.0 * M * H * D * C),
        "fc_relu2": ("tensor", 2.0 * M * C * F),
        "proj_residual": ("tensor", 2.0 * M * F * C),
        "lmhead_softcap": ("tensor", 2.0 * M * C * V),
        # wte row gather (bf16), x0 and x written (fp32), bf16 copy, token ids
        "embed_smear": ("hbm", M * C * (2 + 4 + 4 + 2) + M * 4),
    }


def model_flops(cfg, B, T):
    w = kernel_work(cfg, B, T)
    L = cfg.n_layer
    per_layer = sum(w[k][1] for k in ("qkv_rope_qknorm_ve", "attention", "oproj_residual", "fc_relu2",
                                      "proj_residual"))
    return L * per_layer + w["lmhead_softcap"][1]


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
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
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "power_w_max": max(pw),
                "samples": len(sm), "reasons": sorted(reasons)}


def oracle_sample(wl, wts, tok, n_tokens: int, rows: int = 1):
    """Run the fp64 oracle on the first n_tokens positions of batch rows 0..rows-1; returns seconds."""
    import numpy as np
    import oracle as O
    W = O.OracleWeights.from_synth(wl.model, wts)
    t0 = time.perf_counter()
    for r in range(rows):
        O.forward_row(wl.model, W, tok[r, :n_tokens].numpy())
    return time.perf_counter() - t0


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        n = [i.get("num_threads") for i in info if i.get("internal_api") in ("openblas", "mkl", "blis")]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def run_reference(args, rank, world):
    """The CPU oracle timed on the host cores, rank 0 only."""
    if rank != 0:
        return
    from synth import get_workload, make_tokens, make_weights
    wl = get_workload(args.workload)
    wts = make_weights(wl.model, seed=wl.seed, init=wl.init)
    tok = make_tokens(wl)
    n = min(args.ref_tokens, wl.T)
    for _ in range(args.warmup):
        oracle_sample(wl, wts, tok, n)
    secs = [oracle_sample(wl, wts, tok, n) for _ in range(args.steps)]
    total = sum(secs)
    value = n * args.steps / total
    sample = f"positions 0..{n - 1} of batch row 0 of the {wl.name} workload (causal prefix, exact logits)"
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "sample_tokens_per_step": n},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def roofline(ktimes, work, peaks, peak_src):
    """Per-kernel achieved rates and the roofline entry of the dominant kernel class (largest summed
    event time).  A contraction is compared with the burst bf16 figure, since each launch runs for
    tens of microseconds to a millisecond inside a sub-second timed region (the sustained figure,
    from seconds of back-to-back GEMMs at a power-capped clock, is reported beside the model
    rate); a memory-bound kernel with the measured copy bandwidth."""
    kern = {}
    total = max(1e-9, sum(t for t, _ in ktimes.values()))
    for name, (tot, n) in ktimes.items():
        if n and name in work:
            b, wk = work[name]
            s = tot / n / 1000.0
            kern[name] = {"ms_total": tot, "launches": n, "ms_per_launch": tot / n, "share": tot / total,
                          "achieved": wk / s / (1e12 if b == "tensor" else 1e9),
                          "unit": "TFLOP/s" if b == "tensor" else "GB/s"}
    dom = max(kern, key=lambda k: kern[k]["ms_total"])
    bound = work[dom][0]
    key = "bf16_tflops" if bound == "tensor" else "hbm_gbs"
    peak = float(peaks.get(key, FALLBACK_PEAKS[key]))
    for name in kern:
        pk = float(peaks.get("bf16_tflops" if work[name][0] == "tensor" else "hbm_gbs", FALLBACK_PEAKS[key]))
        kern[name]["frac"] = kern[name]["achieved"] / pk
    achieved = kern[dom]["achieved"]
    return kern, dom, {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak,
                       "unit": kern[dom]["unit"], "frac": achieved / peak, "traffic": None,
                       "peak_source": f"{peak_src} ({key}, of measured)" if peak_src == "measured"
                       else f"{peak_src} ({key}, of fallback)"}


def measure_workload(name, steps, dev, world, peaks, peak_src, cpu_tokens, do_cpu):
    """One of the other full-size workloads: forward tokens/s (CUDA events over `steps` forwards
    after 3 warm-up ones), the model FLOP rate against the burst peak, the per-kernel breakdown
    with the dominant kernel's roofline entry, and an oracle sample on the host cores."""
    import torch
    import torch.distributed as dist
    from synth import get_workload, make_tokens, make_weights
    from decoder_only_forward_02_b300 import binding as NB
    wl = get_workload(name)
    cfg = wl.model
    wts_cpu = make_weights(cfg, seed=wl.seed, init=wl.init)
    wts = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in wts_cpu.items()}
    tok_cpu = make_tokens(wl)
    tok = tok_cpu.to(dev)
    model = NB.Model(cfg, wts, device=dev)
    B, T, V = wl.B, wl.T, cfg.vocab_size
    logits = torch.empty((B, T, V), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        model.forward(tok, out=logits)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        model.forward(tok, out=logits)
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    if model.status() != 0:
        raise RuntimeError(f"device status set on the {name} workload")
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    model.timing(True)
    for _ in range(steps):
        model.forward(tok, out=logits)
    torch.cuda.synchronize()
    model.timing(False)
    ktimes = model.timing_read()
    ms_step = ms / steps
    tflops = model_flops(cfg, B, T) / (ms_step / 1000.0) / 1e12
    kern, dom, roof = roofline(ktimes, kernel_work(cfg, B, T), peaks, peak_src)
    out = {"workload": name, "B": B, "T": T, "value": job_rate(world, B * T * steps, ms), "unit": UNIT,
           "ms_per_step": ms_step, "steps": steps, "model_tflops": tflops,
           "pct_bf16_peak": 100.0 * tflops / float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
           "gpu_launches_per_step": model.launch_count(), "roofline": roof, "kernels": kern}
    del model, logits, wts
    torch.cuda.empty_cache()
    if do_cpu:
        n = min(cpu_tokens, T)
        secs = oracle_sample(wl, wts_cpu, tok_cpu, n, 1)
        out["cpu_baseline"] = {"value": n / secs, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                               "sample": f"fp64 oracle on positions 0..{n - 1} of batch row 0 ({secs:.1f} s)"}
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from synth import get_workload, make_tokens, make_weights
    from decoder_only_forward_02_b300 import build
    build.build()
    from decoder_only_forward_02_b300 import binding as NB

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = get_workload(args.workload)
    cfg = wl.model
    wts_cpu = make_weights(cfg, seed=wl.seed, init=wl.init)
    wts = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in wts_cpu.items()}
    tok_cpu = make_tokens(wl)
    tok = tok_cpu.to(dev)
    model = NB.Model(cfg, wts, device=dev)
    B, T, V = wl.B, wl.T, cfg.vocab_size
    logits = torch.empty((B, T, V), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        model.forward(tok, out=logits)
    torch.cuda.synchronize()
    st = model.status()
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)   # let the sampler start before the timed region
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        model.forward(tok, out=logits)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = e0.elapsed_time(e1)
    clk = clocks.stop()
    if model.status() != 0:
        raise RuntimeError("device status set during the timed region")
    # Per-kernel times: the same steps again, with a CUDA-event pair recorded around every
    # launch on the launching stream (kept out of the region that gives `value`).
    model.timing(True)
    for _ in range(args.steps):
        model.forward(tok, out=logits)
    torch.cuda.synchronize()
    model.timing(False)
    ktimes = model.timing_read()

    # The same forward captured once in a CUDA graph and replayed (reported beside the eager value,
    # which is the call a user makes; the difference is the host's launch work)
    fwd_graph = None
    try:
        gf = torch.cuda.CUDAGraph()
        gfs = torch.cuda.Stream()
        gfs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(gfs):
            with torch.cuda.graph(gf, stream=gfs):
                model.forward(tok, out=logits)
        torch.cuda.current_stream().wait_stream(gfs)
        for _ in range(3):
            gf.replay()
        n_g = max(1, min(args.steps, 50))
        barrier()
        torch.cuda.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(n_g):
            gf.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        barrier()
        g_ms = max_over_ranks(g0.elapsed_time(g1), world, dev) / n_g
        fwd_graph = {"value": job_rate(world, B * T, g_ms), "unit": UNIT, "ms_per_step": g_ms, "steps": n_g,
                     "note": "nc_forward captured once in a CUDA graph and replayed"}
        del gf
    except RuntimeError as exc:   # a capture the runtime refuses leaves the eager numbers standing
        fwd_graph = {"unavailable": str(exc).splitlines()[0][:200]}

    # The loss path (nc_forward_loss: the lm_head fused with the soft-cap and the next-token
    # cross-entropy, no logits written), timed the same way on the same batch; targets are the
    # next tokens, the last position of each row ignored.
    loss_path = None
    if not args.no_loss_path:
        tgt = torch.full_like(tok, -1)
        tgt[:, :-1] = tok[:, 1:]
        lbuf = torch.empty((B, T), dtype=torch.float32, device=dev)
        sbuf = torch.empty((2,), dtype=torch.float32, device=dev)
        for _ in range(3):
            model.forward_loss(tok, tgt, loss=lbuf, stats=sbuf)
        n_loss = max(1, min(args.steps, 50))
        barrier()
        torch.cuda.synchronize()
        e2 = torch.cuda.Event(enable_timing=True)
        e3 = torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        for _ in range(n_loss):
            model.forward_loss(tok, tgt, loss=lbuf, stats=sbuf)
        e3.record(stream)
        torch.cuda.synchronize()
        barrier()
        if model.status() != 0:
            raise RuntimeError("device status set on the loss path")
        loss_ms = max_over_ranks(e2.elapsed_time(e3), world, dev) / n_loss
        loss_path = {"metric": "forward + cross-entropy tokens/s", "value": job_rate(world, B * T, loss_ms),
                     "unit": UNIT, "ms_per_step": loss_ms, "steps": n_loss,
                     "gpu_launches_per_step": model.launch_count(loss=True),
                     "mean_loss_nats": float(sbuf[0].item()),
                     "note": "nc_forward_loss: lm_head fused with soft-cap and cross-entropy, no logits written"}

    # The backward's first part (nc_forward_loss_grad_tail): the loss path, then the gradient of the
    # mean loss with respect to the lm_head and the last block's MLP and attention output projection,
    # timed the same way; a second pass with per-kernel events gives each backward class its rate.
    grad_tail = None
    if not args.no_grad_tail:
        tgt = torch.full_like(tok, -1)
        tgt[:, :-1] = tok[:, 1:]
        for _ in range(3):
            model.loss_grad_tail(tok, tgt)
        n_bw = max(1, min(args.steps, 20))
        barrier()
        torch.cuda.synchronize()
        e4 = torch.cuda.Event(enable_timing=True)
        e5 = torch.cuda.Event(enable_timing=True)
        e4.record(stream)
        for _ in range(n_bw):
            st_bw, _ = model.loss_grad_tail(tok, tgt)
        e5.record(stream)
        torch.cuda.synchronize()
        barrier()
        if model.status() != 0:
            raise RuntimeError("device status set on the backward path")
        bw_ms = max_over_ranks(e4.elapsed_time(e5), world, dev) / n_bw
        model.timing(True)
        model.loss_grad_tail(tok, tgt)
        torch.cuda.synchronize()
        bt = model.timing_read()
        model.timing(False)
        M = B * T
        C, F, V, HD = cfg.n_embd, cfg.mlp_hidden, cfg.vocab_size, cfg.n_head * cfg.head_dim
        bw_work = {"lmhead_grad": ("tensor", 2.0 * M * C * V), "mlp_grad": ("tensor", 2.0 * M * C * F),
                   "oproj_grad": ("tensor", 2.0 * M * C * HD),
                   # G and x read (fp32), the residual gradient or the fp32 copy, the bf16 copy
                   "rmsnorm_grad": ("hbm", 14.0 * M * C)}
        bw_peaks, bw_src = load_peaks()
        bw_k, _, _ = roofline({k: v for k, v in bt.items() if k in bw_work}, bw_work, bw_peaks, bw_src)
        grad_tail = {"metric": "forward + loss + tail gradients tokens/s", "value": job_rate(world, M, bw_ms),
                     "unit": UNIT, "ms_per_step": bw_ms, "steps": n_bw,
                     "gpu_launches_per_step": model.grad_tail_launch_count(),
                     "mean_loss_nats": float(st_bw[0].item()), "kernels": bw_k,
                     "note": "nc_forward_loss_grad_tail: loss path, then d(mean loss)/d(lm_head, last block's "
                             "c_proj, c_fc, attention c_proj); the lm_head runs three times (loss, gradient "
                             "at its output, recomputed; input and weight gradients)"}

    # The decode path (nc_prefill of T-1 tokens, then nc_decode_step: one new token per batch row
    # at position T-1, the longest context, read from the KV cache), repeated at that position.
    decode_path = None
    if not args.no_decode_path:
        T0 = T - 1
        cache = model.kv_cache(B, T)
        model.prefill(tok[:, :T0].contiguous(), cache, T)
        prev, cur = tok[:, T0 - 1].contiguous(), tok[:, T0].contiguous()
        lg = torch.empty((B, V), dtype=torch.float32, device=dev)
        for _ in range(3):
            model.decode_step(prev, cur, T0, cache, T, out=lg)
        n_dec = max(1, min(args.steps, 50))
        barrier()
        torch.cuda.synchronize()
        e4 = torch.cuda.Event(enable_timing=True)
        e5 = torch.cuda.Event(enable_timing=True)
        e4.record(stream)
        for _ in range(n_dec):
            model.decode_step(prev, cur, T0, cache, T, out=lg)
        e5.record(stream)
        torch.cuda.synchronize()
        barrier()
        if model.status() != 0:
            raise RuntimeError("device status set on the decode path")
        dec_ms = max_over_ranks(e4.elapsed_time(e5), world, dev) / n_dec
        # the same step captured once in a CUDA graph and replayed (no per-launch host work)
        gph = torch.cuda.CUDAGraph()
        gs = torch.cuda.Stream()
        gs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(gs):
            with torch.cuda.graph(gph, stream=gs):
                model.decode_step(prev, cur, T0, cache, T, out=lg)
        torch.cuda.current_stream().wait_stream(gs)
        for _ in range(3):
            gph.replay()
        barrier()
        torch.cuda.synchronize()
        e4.record(stream)
        for _ in range(n_dec):
            gph.replay()
        e5.record(stream)
        torch.cuda.synchronize()
        barrier()
        if model.status() != 0:
            raise RuntimeError("device status set on the decode path (graph)")
        dec_graph_ms = max_over_ranks(e4.elapsed_time(e5), world, dev) / n_dec
        del gph
        model.timing(True)   # per-kernel-class times of the step (events around every launch)
        for _ in range(10):
            model.decode_step(prev, cur, T0, cache, T, out=lg)
        torch.cuda.synchronize()
        dk = model.timing_read()
        model.timing(False)
        dec_kernels = {k: {"launches_per_step": n // 10, "us_per_step": 1000.0 * ms / 10} for k, (ms, n) in dk.items() if n}
        w_bytes, kv_bytes = decode_step_bytes(cfg, B, T0)
        dec_peak = load_peaks()[0].get("hbm_gbs")
        decode_path = {"metric": "decode tokens/s (one new token per batch row)", "value": job_rate(world, B, dec_ms),
                       "unit": UNIT, "ms_per_step": dec_ms, "steps": n_dec, "batch": B, "context": T,
                       "gpu_launches_per_step": model.launch_count(kv=True),
                       "kernels": dec_kernels,
                       "graph": {"value": job_rate(world, B, dec_graph_ms), "unit": UNIT,
                                 "ms_per_step": dec_graph_ms,
                                 "note": "the same nc_decode_step captured once in a CUDA graph and replayed"},
                       "roofline": {"bound": "hbm", "bytes_per_step": w_bytes + kv_bytes, "weight_bytes": w_bytes,
                                    "kv_bytes": kv_bytes,
                                    "achieved": (w_bytes + kv_bytes) / (dec_graph_ms * 1e-3) / 1e9, "unit": "GB/s",
                                    "peak": dec_peak,
                                    "frac": ((w_bytes + kv_bytes) / (dec_graph_ms * 1e-3) / 1e9 / dec_peak)
                                    if dec_peak else None,
                                    "note": "algorithmic bytes of a step over the graph-replay time, against the "
                                            "measured HBM copy rate: the step is a chain of 62 dependent launches, "
                                            "so it is latency-bound, not bandwidth-bound"},
                       "note": "nc_decode_step at position T-1 after nc_prefill of T-1 tokens, repeated at that "
                               "position; small-row weight-streaming products and a one-launch attention per "
                               "layer, bound by the chain of dependent launches"}
        del cache

    # The same forward writing bf16 logits (nc_config.logits_bf16: the soft-capped values rounded to
    # nearest even, half the 2.15 GB write), on device and end to end through host buffers.
    logits_bf16 = None
    if not args.no_bf16_logits:
        m16 = NB.Model(cfg, wts, device=dev, logits_bf16=True)
        z16 = torch.empty((B, T, V), dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            m16.forward(tok, out=z16)
        n16 = max(1, min(args.steps, 50))
        barrier()
        torch.cuda.synchronize()
        e6 = torch.cuda.Event(enable_timing=True)
        e7 = torch.cuda.Event(enable_timing=True)
        e6.record(stream)
        for _ in range(n16):
            m16.forward(tok, out=z16)
        e7.record(stream)
        torch.cuda.synchronize()
        barrier()
        if m16.status() != 0:
            raise RuntimeError("device status set on the bf16-logits forward")
        ms16 = max_over_ranks(e6.elapsed_time(e7), world, dev) / n16
        logits_bf16 = {"metric": "forward tokens/s, bf16 logits", "value": job_rate(world, B * T, ms16), "unit": UNIT,
                       "ms_per_step": ms16, "steps": n16, "gpu_launches_per_step": m16.launch_count(),
                       "note": "nc_forward with logits_bf16: the same logits rounded to nearest even "
                               "(bitwise the rounding of the fp32 output)"}
        if not args.no_e2e:
            tok_h = tok_cpu.pin_memory()
            out_h = torch.empty((B, T, V), dtype=torch.bfloat16).pin_memory()
            for _ in range(2):
                m16.forward_host(tok_h, out_h)
            k = max(1, min(args.steps, args.e2e_steps))
            barrier()
            torch.cuda.synchronize()
            h0 = time.perf_counter()
            for _ in range(k):
                m16.forward_host(tok_h, out_h)
            torch.cuda.synchronize()
            h_ms = 1000 * (time.perf_counter() - h0)
            logits_bf16["e2e"] = {"value": job_rate(world, B * T * k, max_over_ranks(h_ms, world, dev)), "unit": UNIT,
                                  "h2d_bytes_per_step": int(tok_h.numel() * 4),
                                  "d2h_bytes_per_step": int(out_h.numel() * 2), "steps": k}
            del out_h
        del m16, z16
        torch.cuda.empty_cache()

    # The 8-bit path (every linear layer in e4m3 at tensorwise scales, activations quantised on the
    # fly): the same forward timed the same way, with per-kernel rates; contractions against the
    # e4m3 peak (the measured bf16 figure times 2, the nominal dense ratio), quantisation against HBM.
    fp8_path = None
    ms_step_bf16 = ms / max(args.steps, 1)   # this rank's bf16 forward, for the ratio below
    if not args.no_fp8:
        m8 = NB.Model(cfg, wts, device=dev, fp8=True)
        z8 = torch.empty((B, T, V), dtype=torch.float32, device=dev)
        for _ in range(3):
            m8.forward(tok, out=z8)
        n8 = max(1, min(args.steps, 50))
        barrier()
        torch.cuda.synchronize()
        e8 = torch.cuda.Event(enable_timing=True)
        e9 = torch.cuda.Event(enable_timing=True)
        e8.record(stream)
        for _ in range(n8):
            m8.forward(tok, out=z8)
        e9.record(stream)
        torch.cuda.synchronize()
        barrier()
        if m8.status() != 0:
            raise RuntimeError("device status set on the 8-bit forward")
        ms8 = max_over_ranks(e8.elapsed_time(e9), world, dev) / n8
        m8.timing(True)
        for _ in range(3):
            m8.forward(tok, out=z8)
        torch.cuda.synchronize()
        t8 = m8.timing_read()
        m8.timing(False)
        pk8, src8 = load_peaks()
        pk8 = dict(pk8)
        pk8["bf16_tflops"] = 2.0 * float(pk8.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        w8 = dict(kernel_work(cfg, B, T))
        M_ = B * T
        # per quantisation launch (amax or codes): the mean tensor read, plus the 1-byte codes on half
        # the launches: (the normed stream fp32 twice, y and h bf16) / 4 layer inputs
        C_, HD_, F_ = cfg.n_embd, cfg.n_head * cfg.head_dim, cfg.mlp_hidden
        w8["fp8_quantize"] = ("hbm", M_ * (2 * C_ * 4 + HD_ * 2 + F_ * 2) / 4.0 + M_ * (2 * C_ + HD_ + F_) / 8.0)
        k8, _, _ = roofline({k: v for k, v in t8.items() if k in w8}, w8, pk8, src8)
        fp8_path = {"metric": "forward tokens/s, e4m3 linear layers", "value": job_rate(world, B * T, ms8),
                    "unit": UNIT, "ms_per_step": ms8, "steps": n8, "gpu_launches_per_step": m8.launch_count(),
                    "tflops_model": model_flops(cfg, B, T) / (ms8 / 1000.0) / 1e12,
                    "peak_e4m3_tflops": pk8["bf16_tflops"], "kernels": k8,
                    "vs_bf16_forward": ms_step_bf16 / ms8 if ms_step_bf16 else None,
                    "note": "nc_forward with fp8: q, k, v, output projection, MLP and lm_head on e4m3 copies "
                            "(weights quantised at model creation, each layer input per call over the whole "
                            "batch; the stream's and the MLP hidden layer's maxima come from the epilogues "
                            "that write them), fp32 accumulation; attention, norms and gates in bf16/fp32; "
                            "vs_bf16_forward = bf16 ms per forward / 8-bit ms per forward, same run"}
        del m8, z8
        torch.cuda.empty_cache()

    ms_max = max_over_ranks(ms, world, dev)
    ms_step = ms_max / args.steps
    value = job_rate(world, B * T * args.steps, ms_max)

    # end to end through host buffers
    e2e = None
    if not args.no_e2e:
        tok_h = tok_cpu.pin_memory()
        out_h = torch.empty((B, T, V), dtype=torch.float32).pin_memory()
        for _ in range(2):
            model.forward_host(tok_h, out_h)
        e2e_steps = max(1, min(args.steps, args.e2e_steps))
        barrier()
        torch.cuda.synchronize()
        h0 = time.perf_counter()
        for _ in range(e2e_steps):
            model.forward_host(tok_h, out_h)
        torch.cuda.synchronize()
        h_ms = 1000 * (time.perf_counter() - h0)
        e2e = {"value": job_rate(world, B * T * e2e_steps, max_over_ranks(h_ms, world, dev)), "unit": UNIT,
               "h2d_bytes_per_step": int(tok_h.numel() * 4), "d2h_bytes_per_step": int(out_h.numel() * 4),
               "steps": e2e_steps}
        del out_h

    # the other full-size workloads (d20 with grouped-query attention, the long-context d12 whose
    # short windows skip most key tiles, d24), each measured the same way on a shorter loop (every
    # rank runs them: the timing takes the max over ranks)
    peaks, peak_src = load_peaks()
    launches = model.launch_count() * args.steps
    workloads = []
    extra = [w for w in args.extra_workloads.split(",") if w and w != wl.name]
    if extra:
        del logits, model, wts
        torch.cuda.empty_cache()
        workloads = [measure_workload(w, args.extra_steps, dev, world, peaks, peak_src, args.extra_cpu_tokens,
                                      rank == 0 and not args.no_cpu_baseline) for w in extra]
    if rank != 0:
        return
    work = kernel_work(cfg, B, T)
    kern, dom, roof = roofline(ktimes, work, peaks, peak_src)
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        t = json.load(open(tpath))
        if t.get("kernel") == dom and t.get("workload") == wl.name and \
                t.get("source_hash") == _src_hash(t.get("sources")):
            traffic = t.get("bytes_per_launch")
    flops = model_flops(cfg, B, T)
    tflops = flops / (ms_step / 1000.0) / 1e12
    roof["traffic"] = traffic
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) bf16 weights, uniform tokens)",
        "config": {"workload": wl.name, "B": B, "T": T, "n_layer": cfg.n_layer, "n_embd": cfg.n_embd,
                   "n_head": cfg.n_head, "n_kv_head": cfg.n_kv_head, "vocab": V,
                   "windows": "SSSL short=%d" % max(cfg.window_left), "logits": "fp32",
                   "l2": "no flush: each step writes %.2f GB of logits and reads %.2f GB of weights, "
                         "far above the 126 MB L2" % (B * T * V * 4 / 1e9, _weight_bytes(wts_cpu) / 1e9),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "model_tflops": tflops,
        "pct_bf16_peak": 100.0 * tflops / float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
        "pct_bf16_peak_sustained": 100.0 * tflops / float(
            peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])),
        "roofline": roof,
        "kernels": kern,
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": e2e,
        "loss_path": loss_path,
        "graph": fwd_graph,
        "decode_path": decode_path,
        "grad_tail": grad_tail,
        "logits_bf16": logits_bf16,
        "fp8_path": fp8_path,
    }
    if workloads:
        line["workloads"] = workloads
    if not args.no_cpu_baseline and world >= 1:
        n = min(args.cpu_tokens, T)
        rows = max(1, min(args.cpu_rows, B))
        secs = oracle_sample(wl, wts_cpu, tok_cpu, n, rows)
        line["cpu_baseline"] = {"value": rows * n / secs, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                                "sample": f"fp64 oracle on positions 0..{n - 1} of batch rows 0..{rows - 1} "
                                          f"({secs:.1f} s; rows are independent and a causal prefix gives "
                                          f"exact logits for its positions)"}
    print(json.dumps(line), flush=True)


def run_single_kernel(args):
    """Launch one kernel class `--launches` times at the workload's shapes through the per-kernel
    entry points (small device footprint; used for profiler captures of one kernel)."""
    import torch
    from synth import get_workload
    from decoder_only_forward_02_b300 import build
    build.build()
    from decoder_only_forward_02_b300 import binding as NB
    ops = NB.ops
    wl = get_workload(args.workload)
    c = wl.model
    M, C, H, Hkv, D, F, V = wl.M, c.n_embd, c.n_head, c.n_kv_head, c.head_dim, c.mlp_hidden, c.vocab_size
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(0)

    def rnd(shape, scale=1.0, dtype=torch.bfloat16):
        return (torch.randn(shape, generator=g, device=dev) * scale).to(dtype)

    def unit(t):
        return (t.float() / t.float().pow(2).mean(-1, keepdim=True).sqrt()).to(torch.bfloat16)

    k = args.only_kernel
    window = max(c.window_left) if args.window is None else args.window
    if k == "qkv":   # a value-embedding layer's q|k|v projection (gate rows packed after each kv head's v)
        xb = rnd((M, C))
        w = ops.pack_qkv(rnd((H * D, C), 0.02), rnd((Hkv * D, C), 0.02), rnd((Hkv * D, C), 0.02),
                         rnd((Hkv, C), 0.02), D)
        ssp = torch.rand((M, C // 128), generator=g, device=dev) * 100
        rope = ops.rope_table(wl.T, D, c.rope_base, dev)
        ve, tok = rnd((V, Hkv * D), 0.02), torch.randint(0, V, (M,), generator=g, device=dev, dtype=torch.int32)
        fn = lambda: ops.qkv(xb, w, wl.T, H, Hkv, D, rope, c.rms_eps, ssp, True, 1.0, ve, tok, V)
    elif k == "attention":
        q, kk, v = unit(rnd((M, H, D))).reshape(M, -1), unit(rnd((M, Hkv, D))).reshape(M, -1), rnd((M, Hkv * D))
        fn = lambda: ops.attention(q, kk, v, wl.B, wl.T, H, Hkv, D, window)
    elif k in ("oproj", "proj"):
        K = H * D if k == "oproj" else F
        a, w, x, x0 = rnd((M, K)), rnd((C, K), 0.02), rnd((M, C), 1.0, torch.float32), rnd((M, C), 1.0, torch.float32)
        if k == "oproj":
            fn = lambda: ops.gemm_residual(a, w, x, x_out=x)
        else:   # the MLP down projection with the next block's mix
            fn = lambda: ops.gemm_residual(a, w, x, 0.9, 0.1, x0, x, None)
    elif k == "fc":
        a, w = rnd((M, C)), rnd((F, C), 0.02)
        ssp = torch.rand((M, C // 128), generator=g, device=dev) * 100
        fn = lambda: ops.gemm(a, w, "relu2_bf16", ssp=ssp, C=C)
    elif k == "lmhead":
        a, w = rnd((M, C)), rnd((V, C), 0.02)
        ssp = torch.rand((M, C // 128), generator=g, device=dev) * 100
        out = torch.empty((M, V), dtype=torch.float32, device=dev)
        fn = lambda: ops.gemm(a, w, "softcap_f32", out=out, ssp=ssp, C=C, cap=c.softcap)
    elif k == "lmhead_ce":   # the loss path's lm_head: soft-cap + cross-entropy partials, no logits
        a, w = rnd((M, C)), rnd((V, C), 0.02)
        ssp = torch.rand((M, C // 128), generator=g, device=dev) * 100
        tgt = torch.randint(0, V, (M,), generator=g, device=dev, dtype=torch.int32)
        fn = lambda: ops.lmhead_ce(a, w, tgt, ssp=ssp, C=C, cap=c.softcap)
    elif k == "ce_grad":   # the gradient at the lm_head's output (the logits recomputed; lse from the loss pass)
        a, w = rnd((M, C)), rnd((V, C), 0.02)
        ssp = torch.rand((M, C // 128), generator=g, device=dev) * 100
        tgt = torch.randint(0, V, (M,), generator=g, device=dev, dtype=torch.int32)
        part, zt = ops.lmhead_ce(a, w, tgt, ssp=ssp, C=C, cap=c.softcap)
        _, _, lse, invc = ops.ce_finalize(part, zt, tgt, V, with_lse=True)
        fn = lambda: ops.lmhead_ce_grad(a, w, tgt, lse, invc, ssp=ssp, C=C, cap=c.softcap)
    elif k == "lmhead_dgrad":   # G = dlt . W_lm: the lm_head's input gradient (W_lm read N-contiguous)
        dlt, w = rnd((M, V), 1e-6), rnd((V, C), 0.02)
        out = torch.empty((M, C), dtype=torch.float32, device=dev)
        fn = lambda: ops.gemm_t(dlt, w, a_mn=False, b_mn=True, epi="f32", out=out)
    elif k == "lmhead_wgrad":   # dW_lm = dlt^T . xb: both operands token-major
        dlt, xb = rnd((M, V), 1e-6), rnd((M, C))
        out = torch.empty((V, C), dtype=torch.float32, device=dev)
        fn = lambda: ops.gemm_t(dlt, xb, a_mn=True, b_mn=True, epi="f32", out=out, split=True)
    elif k == "mlp_wgrad":      # dW_proj = dxl^T . h, split over the tokens
        dxl, h = rnd((M, C)), rnd((M, F))
        out = torch.empty((C, F), dtype=torch.float32, device=dev)
        fn = lambda: ops.gemm_t(dxl, h, a_mn=True, b_mn=True, epi="f32", out=out, split=True)
    elif k == "mlp_hidden_grad":   # rs * (dxl . W_proj) * 2 sqrt(h)
        dxl, w, h = rnd((M, C)), rnd((C, F), 0.02), rnd((M, F)).abs()
        ssp = torch.rand((M, C // 128), generator=g, device=dev) * 100
        fn = lambda: ops.mlp_hidden_grad(dxl, w, h, ssp=ssp)
    elif k == "fc_fp8":   # the MLP up projection on e4m3 copies (squared ReLU epilogue)
        a8 = rnd((M, C), 30.0, torch.float32).to(torch.float8_e4m3fn)
        w8 = rnd((F, C), 30.0, torch.float32).to(torch.float8_e4m3fn)
        sa, sw = torch.full((1,), 1e-3, device=dev), torch.full((1,), 1e-3, device=dev)
        fn = lambda: ops.gemm_fp8(a8, w8, sa, sw, epi="relu2_bf16")
    elif k == "fp8_quantize":   # the MLP hidden layer's tensorwise quantisation (amax, then codes)
        h = rnd((M, F)).abs()
        fn = lambda: ops.fp8_quantize(h)
    elif k == "rms_backward":
        G, x = rnd((M, C), 1.0, torch.float32), rnd((M, C), 1.0, torch.float32)
        ssp = torch.rand((M, C // 128), generator=g, device=dev) * 100
        fn = lambda: ops.rms_backward(G, x, ssp, add=G)
    elif k == "embed":
        tok = torch.randint(0, V, (wl.B, wl.T), generator=g, device=dev, dtype=torch.int32)
        wte, sg = rnd((V, C), 0.02), rnd((C,), 0.02)
        fn = lambda: ops.embed_smear(tok, wte, sg, C)
    elif k == "decode":   # decode steps at the last position after a prefill of T-1 tokens (cache append, split attention)
        from synth import make_tokens, make_weights
        wts = {n: (v.to(dev) if torch.is_tensor(v) else v) for n, v in make_weights(c, seed=wl.seed, init=wl.init).items()}
        model = NB.Model(c, wts, device=dev)
        tokd = make_tokens(wl).to(dev)
        T0 = wl.T - 1
        cache = model.kv_cache(wl.B, wl.T)
        model.prefill(tokd[:, :T0].contiguous(), cache, wl.T)
        prev, cur = tokd[:, T0 - 1].contiguous(), tokd[:, T0].contiguous()
        fn = lambda: model.decode_step(prev, cur, T0, cache, wl.T)
    else:
        raise SystemExit(f"unknown kernel {k}")
    for _ in range(args.launches):
        fn()
    torch.cuda.synchronize()
    print(json.dumps({"kernel": k, "workload": wl.name, "launches": args.launches, "ok": True}))


def _src_hash(files=None):
    """sha1 (12 hex digits) of the named csrc files (all of csrc when None), in sorted order: the
    sources the recorded DRAM traffic of a kernel depends on."""
    import hashlib
    h = hashlib.sha1()
    d = os.path.join(ROOT, "decoder_only_forward_02_b300", "csrc")
    for f in sorted(files if files else os.listdir(d)):
        p = os.path.join(d, f)
        if not os.path.isfile(p):
            return None
        h.update(open(p, "rb").read())
    return h.hexdigest()[:12]


def _weight_bytes(w):
    import torch
    return sum(v.numel() * v.element_size() for v in w.values() if torch.is_tensor(v))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="d12")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-loss-path", action="store_true", help="skip timing the fused cross-entropy path")
    ap.add_argument("--no-grad-tail", action="store_true", help="skip timing the tail backward")
    ap.add_argument("--no-fp8", action="store_true", help="skip timing the e4m3 forward")
    ap.add_argument("--no-decode-path", action="store_true", help="skip timing the KV-cache decode step")
    ap.add_argument("--no-bf16-logits", action="store_true", help="skip timing the forward with bf16 logits")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-tokens", type=int, default=2048)
    ap.add_argument("--cpu-rows", type=int, default=4, help="batch rows the CPU baseline times")
    ap.add_argument("--ref-tokens", type=int, default=256,
                    help="positions of batch row 0 the reference arm runs per step (a bounded sample)")
    ap.add_argument("--extra-workloads", default="d20,d12_long,d24",
                    help="other full-size workloads measured after the headline one (comma list; empty: none)")
    ap.add_argument("--extra-steps", type=int, default=20)
    ap.add_argument("--extra-cpu-tokens", type=int, default=128,
                    help="positions of batch row 0 the oracle runs for each extra workload's CPU baseline")
    ap.add_argument("--only-kernel", default=None,
                    help="launch one kernel class (qkv, attention, oproj, fc, proj, lmhead, lmhead_ce, embed, decode, "
                         "ce_grad, lmhead_dgrad, lmhead_wgrad, mlp_wgrad, mlp_hidden_grad, rms_backward, fc_fp8, "
                         "fp8_quantize) "
                         "at the workload's shapes, for profiler captures")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--window", type=int, default=None)
    args = ap.parse_args()
    if args.only_kernel:
        run_single_kernel(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
