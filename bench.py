"""Benchmark: 4-bit-KV decode attention step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config b32_ctx32k] [--no-cpu-baseline] [--no-fp8]

One step = quantise-on-append of the step's new tokens (T per sequence) into
the paged 4-bit cache, then paged decode attention over the whole cache
(q rotation, split partials, log-sum-exp combine, output rotation).  The
workload is batch 32, context 32768 (counting the new token), 8 KV heads,
64 query heads, head_dim 128, page size 16, seeded synthetic bf16 K/V with 2 %
outlier channels x16; pages are randomly permuted in one shared pool.

value      = algorithmic KV bytes read per step / device time per step (GB/s),
             inputs resident in HBM; the KV cache (1.14 GB) is larger than L2.
e2e        = the same metric through the public API with host buffers: the
             step's q and new K/V are copied from pinned host memory and the
             output is copied back inside the timed region.
roofline   = the decode split kernel alone (CUDA events around each launch in
             the timed region) against the measured HBM copy bandwidth.
cpu_baseline = the CPU oracle on a bounded sample of the same workload.
Multi-GPU: every rank runs an independent replica (the path has no exchange
step); value sums the units of all ranks over the max elapsed time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_kv_cache_rotate_b300 import workloads as W  # noqa: E402

FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0
DECODE_SOURCES = ("bit_kv_cache_rotate_b300/csrc/kv4_decode_mma.cu",
                  "bit_kv_cache_rotate_b300/csrc/kv4_extend_tc.cu",
                  "bit_kv_cache_rotate_b300/csrc/kv4_decode_mla.cu",
                  "bit_kv_cache_rotate_b300/csrc/kv4_decode_mla_tc.cu",
                  "bit_kv_cache_rotate_b300/csrc/kv4_mma_common.cuh",
                  "bit_kv_cache_rotate_b300/csrc/kv4_decode.h")
KERNEL_NAMES = {1: "warp-MMA kernel, split form", 2: "tcgen05 extend kernel", 3: "warp-MMA latent kernel",
                4: "general CUDA-core kernel", 5: "warp-specialised tcgen05 decode kernel",
                6: "tcgen05 latent kernel", 7: "warp-MMA kernel, flat mode"}
METRIC = "4-bit-KV decode attention: HBM GB/s (% of peak) and ms/step at 32K ctx, batch 32"
EXTEND_METRIC = "4-bit-KV extend attention: TFLOP/s (% of peak) and ms/step"


def kv_bytes_4bit(cfg, lens) -> int:
    per_tok = 2 * (cfg.head_dim // 2 + cfg.head_dim // 32) * cfg.num_kv_heads
    if cfg.latent:
        per_tok //= 2
    return int(np.asarray(lens, dtype=np.int64).sum()) * per_tok


def attn_flops(cfg, lens) -> int:
    """Q.K^T and P.V multiply-adds of one step: position j of a sequence with
    context L attends to L - T + 1 + j tokens, 4 * D flops per (token, query head)."""
    T = cfg.q_per_seq
    lens = np.asarray(lens, dtype=np.int64)
    visible = T * (lens - T + 1) + T * (T - 1) // 2
    return int(visible.sum()) * 4 * cfg.head_dim * cfg.num_q_heads


def is_extend(cfg) -> bool:
    return cfg.q_per_seq > 8


def kv_bytes_fp8(cfg, lens) -> int:
    return int(np.asarray(lens, dtype=np.int64).sum()) * 2 * cfg.head_dim * cfg.num_kv_heads


def source_hash() -> str:
    h = hashlib.sha256()
    for rel in DECODE_SOURCES + ("bit_kv_cache_rotate_b300/csrc/kv4_common.cuh",):
        p = os.path.join(ROOT, rel)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def max_over_ranks(x: float, world: int) -> float:
    """Maximum of x over the ranks of the default process group (x when world == 1)."""
    if world <= 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_gbs(bytes_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s of `world` independent replicas timed by the slowest rank."""
    return bytes_per_rank * world / (ms_per_step * 1e-3) / 1e9


def measured_peak(key: str = "hbm_gbs", fallback: float = FALLBACK_HBM_GBS):
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return float(json.load(open(p))[key]), "measured"
        except Exception:
            pass
    return fallback, "fallback"


def stored_traffic(config_name: str):
    """DRAM bytes per decode launch from a committed ncu summary, if taken on
    the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        if d.get("source_hash") != source_hash():
            return None
        return d.get("per_launch_bytes", {}).get(config_name)
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9], parts[4]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
class Workload:
    """The cache state before the timed step, built on the device."""

    def __init__(self, cfg, kv4, with_fp8: bool):
        self.cfg = cfg
        self.lay = W.make_layout(cfg)
        lay = self.lay
        B, T, P = cfg.batch, cfg.q_per_seq, cfg.page_size
        dev = torch.device("cuda")
        self.kc = kv4.empty_cache(lay.num_pages, cfg.num_kv_heads, cfg.head_dim)
        self.vc = None if cfg.latent else kv4.empty_cache(lay.num_pages, cfg.num_kv_heads, cfg.head_dim)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        # Generate every token once (shared prefix appended once), keep bf16 on the
        # device for the FP8 calibration, append all but the step's new tokens.
        chain = None
        n_chain = int(lay.prefix_pages.max()) * P if B else 0
        if n_chain:
            chain = W.chain_tokens(cfg, lay, 0, int(lay.chain.size) * P)
        ks, vs, slots = [], [], []
        new_k, new_v, new_slots = [], [], []
        if n_chain:
            ks.append(chain[0][:n_chain].to(dev))
            vs.append(None if cfg.latent else chain[1][:n_chain].to(dev))
            slots.append(torch.from_numpy(W.chain_slots(cfg, lay, 0, n_chain)).to(dev))
        for b in range(B):
            L = int(lay.context_lens[b])
            start = int(lay.prefix_pages[b]) * P
            kp, vp = W.private_tokens(cfg, lay, b)
            kp = kp.to(dev)
            vp = None if vp is None else vp.to(dev)
            s = torch.from_numpy(W.slots_for(lay, b, start, L, P)).to(dev)
            n_old = L - T - start
            ks.append(kp[:n_old])
            vs.append(None if vp is None else vp[:n_old])
            slots.append(s[:n_old])
            new_k.append(kp[n_old:])
            new_v.append(None if vp is None else vp[n_old:])
            new_slots.append(s[n_old:])
        self.new_k = torch.cat(new_k).contiguous()
        self.new_v = None if cfg.latent else torch.cat(new_v).contiguous()
        self.new_slots = torch.cat(new_slots).contiguous()
        for k, v, s in zip(ks, vs, slots):
            kv4.kv4_append_quantize(k.contiguous(), None if v is None else v.contiguous(), s.contiguous(),
                                    self.kc, self.vc, lay.num_pages, dev_error=self.err)
        self.q = W.queries(cfg).to(dev)
        self.tab = torch.from_numpy(lay.block_tables.clip(min=0)).to(dev)
        self.lens = torch.from_numpy(lay.context_lens).to(dev)
        self.S = kv4.kv4_decode_auto_splits(B, T, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim, P,
                                            lay.max_pages)
        self.ws = kv4.workspace(B, T, cfg.num_q_heads, cfg.head_dim, self.S)
        self.out = torch.empty((B, T, cfg.num_q_heads, cfg.head_dim), dtype=torch.float32, device=dev)
        self.fp8 = None
        if with_fp8 and not cfg.latent:
            allk = torch.cat(ks + [self.new_k])
            allv = torch.cat(vs + [self.new_v])
            amk = allk.float().abs().amax(dim=(0, 2)).double().clamp_min(1e-30)
            amv = allv.float().abs().amax(dim=(0, 2)).double().clamp_min(1e-30)
            k_scale, v_scale = (amk / 448).float(), (amv / 448).float()
            k_inv, v_inv = (1.0 / k_scale.double()).float(), (1.0 / v_scale.double()).float()
            fkc = kv4.empty_cache(lay.num_pages, cfg.num_kv_heads, cfg.head_dim, fp8=True)
            fvc = kv4.empty_cache(lay.num_pages, cfg.num_kv_heads, cfg.head_dim, fp8=True)
            for k, v, s in zip(ks, vs, slots):
                kv4.fp8_append_quantize(k.contiguous(), v.contiguous(), s.contiguous(), k_inv, v_inv, fkc, fvc,
                                        lay.num_pages, dev_error=self.err)
            self.fp8 = dict(kc=fkc, vc=fvc, k_scale=k_scale, v_scale=v_scale, k_inv=k_inv, v_inv=v_inv,
                            ws=kv4.workspace(B, T, cfg.num_q_heads, cfg.head_dim, self.S))
            del allk, allv
        del ks, vs, slots
        torch.cuda.synchronize()
        assert int(self.err.item()) == 0, "append reported a bounds error"
        torch.cuda.empty_cache()


def run_ours(args, rank, world, local_rank):
    import bit_kv_cache_rotate_b300 as kv4
    torch.cuda.set_device(local_rank)
    cfg = W.CONFIGS[args.config]
    wl = Workload(cfg, kv4, with_fp8=not args.no_fp8)
    lay = wl.lay
    nbytes = kv_bytes_4bit(cfg, lay.context_lens)
    stream = torch.cuda.current_stream()

    po, pl = kv4.split_views(wl.ws, cfg.batch, cfg.q_per_seq, cfg.num_q_heads, cfg.head_dim, wl.S)

    def step(ev_a=None, ev_b=None):
        cur = torch.cuda.current_stream()
        kv4.kv4_append_quantize(wl.new_k, wl.new_v, wl.new_slots, wl.kc, wl.vc, lay.num_pages)
        if ev_a is not None:
            ev_a.record(cur)
        if args.kernel:
            # an explicit split kernel: split + combine in one call (the events
            # then bracket both; the combine is a few microseconds)
            kv4.kv4_decode_attention_select(wl.q, wl.kc, wl.vc, wl.tab, wl.lens, cfg.num_kv_heads, lay.num_pages,
                                            cfg.softmax_scale, args.kernel, num_splits=wl.S, workspace_buf=wl.ws,
                                            out=wl.out)
            if ev_b is not None:
                ev_b.record(cur)
            return
        kv4.kv4_decode_partials(wl.q, wl.kc, wl.vc, wl.tab, wl.lens, cfg.num_kv_heads, lay.num_pages,
                                cfg.softmax_scale, wl.S, wl.ws)
        if ev_b is not None:
            ev_b.record(cur)
        kv4.kv4_split_combine(po, pl, out=wl.out)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # The K timed steps are captured once as a CUDA graph (the way a serving
    # loop issues decode) so the measurement is of the GPU, not of Python's
    # launch overhead.  External event nodes bracket every decode launch.
    evs = [(torch.cuda.Event(enable_timing=True, external=True),
            torch.cuda.Event(enable_timing=True, external=True)) for _ in range(args.steps)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(args.steps):
            step(*evs[i])
    graph.replay()  # untimed: first replay uploads the graph
    torch.cuda.synchronize()
    barrier()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        torch.cuda.synchronize()
        t0.record(stream)
        graph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
    barrier()
    elapsed_ms = t0.elapsed_time(t1)
    kern_ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    del graph
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    ms_per_step = elapsed_ms / args.steps
    value = replica_gbs(nbytes, world, ms_per_step)

    # ---- e2e through the public API with host buffers.  Every step copies its
    # inputs (q, the new K/V and their slots) from pinned host memory and reads
    # its output back, as a serving loop does.  The inputs travel as one packed
    # buffer (one copy per step instead of four); the copies run on a second
    # stream into double-buffered device buffers, so step i + 1's inputs and
    # step i's output move while step i computes.
    parts = [wl.q, wl.new_k] + ([] if wl.new_v is None else [wl.new_v]) + [wl.new_slots]
    offs, n_in = [], 0
    for x in parts:
        offs.append(n_in)
        n_in += (x.numel() * x.element_size() + 255) // 256 * 256
    h_in = torch.empty(n_in, dtype=torch.uint8).pin_memory()
    for x, o in zip(parts, offs):
        h_in[o:o + x.numel() * x.element_size()].copy_(x.contiguous().view(-1).view(torch.uint8).cpu())
    d_in = [torch.empty(n_in, dtype=torch.uint8, device=wl.q.device) for _ in range(2)]

    def unpack(buf):
        views = [buf[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape) for x, o in zip(parts, offs)]
        if wl.new_v is None:
            views.insert(2, None)
        return views  # q, k, v, slots

    d_views = [unpack(b) for b in d_in]
    h_out = [torch.empty(wl.out.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    d_out = [torch.empty_like(wl.out) for _ in range(2)]
    copy_stream = torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]

    def h2d(j):
        with torch.cuda.stream(copy_stream):
            d_in[j].copy_(h_in, non_blocking=True)
            ev_in[j].record(copy_stream)

    def compute(j):
        stream.wait_event(ev_in[j])
        q, k, v, s = d_views[j]
        kv4.kv4_append_quantize(k, v, s, wl.kc, wl.vc, lay.num_pages, stream=stream)
        kv4.kv4_decode_attention(q, wl.kc, wl.vc, wl.tab, wl.lens, cfg.num_kv_heads, lay.num_pages,
                                 cfg.softmax_scale, num_splits=wl.S, workspace_buf=wl.ws, out=d_out[j],
                                 stream=stream)
        ev_done[j].record(stream)

    def d2h(j):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(ev_done[j])
            h_out[j].copy_(d_out[j], non_blocking=True)

    def e2e_run(n):
        # copy-stream order: in(0), in(1), out(0), in(2), out(1), ...; in(i + 2)
        # reuses the buffers of step i after out(i), which waits for step i
        h2d(0)
        for i in range(n):
            if i + 1 < n:
                h2d((i + 1) % 2)
            compute(i % 2)
            d2h(i % 2)

    e2e_steps = max(1, min(args.steps, 200))
    e2e_run(3)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    e2e_run(e2e_steps)
    stream.wait_stream(copy_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world)
    assert torch.equal(h_out[(e2e_steps - 1) % 2], d_out[(e2e_steps - 1) % 2].cpu())
    h2d_bytes = h_in.numel()
    d2h_bytes = h_out[0].numel() * h_out[0].element_size()

    # ---- the step's append and combine alone: each launch repeated in a graph of
    # its own (idempotent: the same tokens land in the same slots), so the
    # step's own timing carries no extra event nodes
    def timed_graph(fn, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(n):
                fn()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        del g
        return a.elapsed_time(b) / n

    n_parts = max(1, min(args.steps, 200))
    append_ms = timed_graph(lambda: kv4.kv4_append_quantize(wl.new_k, wl.new_v, wl.new_slots, wl.kc, wl.vc,
                                                            lay.num_pages), n_parts)
    combine_ms = timed_graph(lambda: kv4.kv4_split_combine(po, pl, out=wl.out), n_parts)

    # ---- FP8 comparator on identical inputs
    fp8_info = None
    if wl.fp8 is not None:
        f = wl.fp8

        def fp8_step():
            kv4.fp8_append_quantize(wl.new_k, wl.new_v, wl.new_slots, f["k_inv"], f["v_inv"], f["kc"], f["vc"],
                                    lay.num_pages)
            kv4.fp8_decode_attention(wl.q, f["kc"], f["vc"], f["k_scale"], f["v_scale"], wl.tab, wl.lens,
                                     cfg.num_kv_heads, lay.num_pages, cfg.softmax_scale, num_splits=wl.S,
                                     workspace_buf=f["ws"], out=wl.out)
        for _ in range(max(3, args.warmup)):
            fp8_step()
        torch.cuda.synchronize()
        n8 = max(1, min(args.steps, 200))
        g8 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g8):
            for _ in range(n8):
                fp8_step()
        g8.replay()
        torch.cuda.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        g8.replay()
        f1.record(stream)
        torch.cuda.synchronize()
        del g8
        fms = f0.elapsed_time(f1) / n8
        fbytes = kv_bytes_fp8(cfg, lay.context_lens)
        fp8_info = {"ms_per_step": round(fms, 5), "GB/s": round(fbytes / (fms * 1e-3) / 1e9, 1),
                    "kv_bytes_per_step": fbytes, "speedup_4bit_vs_fp8": round(fms / ms_per_step, 3)}

    flops = attn_flops(cfg, lay.context_lens)
    extend = is_extend(cfg)
    if extend:
        # many positions per sequence: a dense contraction, bound by the tensor pipes
        peak, peak_kind = measured_peak("bf16_tflops", FALLBACK_BF16_TFLOPS)
        achieved = flops / (kern_ms * 1e-3) / 1e12
        metric, unit = EXTEND_METRIC, "TFLOP/s"
        value = flops * world / (ms_per_step * 1e-3) / 1e12
        e2e_value = flops * world / (e2e_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": "kv4 extend kernel (tcgen05: mxf4 Q.K^T, f16 P.V)",
                    "achieved": round(achieved, 1), "peak": peak,
                    "peak_kind": f"{peak_kind} (dense bf16 GEMM, burst; f16 MMAs run at the bf16 rate)",
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": stored_traffic(cfg.name),
                    "kernel_ms": round(kern_ms, 5)}
    else:
        peak, peak_kind = measured_peak()
        achieved = nbytes / (kern_ms * 1e-3) / 1e9
        metric, unit = METRIC, "GB/s"
        e2e_value = replica_gbs(nbytes, world, e2e_ms)
        kid = args.kernel or kv4.kv4_decode_kernel_choice(cfg.batch, cfg.q_per_seq, cfg.num_q_heads,
                                                          cfg.num_kv_heads, cfg.head_dim, wl.S, cfg.latent)
        roofline = {"bound": "hbm", "kernel": f"kv4 decode split kernel: {KERNEL_NAMES.get(kid, kid)}"
                                              + (" (explicit choice, timed with the combine)" if args.kernel else ""),
                    "achieved": round(achieved, 1),
                    "peak": peak, "peak_kind": f"{peak_kind} (hbm copy)", "unit": "GB/s",
                    "frac": round(achieved / peak, 4), "traffic": (stored_traffic(cfg.name) if not args.kernel else None),
                    "kernel_ms": round(kern_ms, 5)}
    res = {
        "metric": metric,
        "value": round(value, 1),
        "unit": unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp4-e2m1+ue8m0 cache, bf16 q, f32 accumulate",
        "data": "synthetic (seeded bf16 K/V/Q, 2% outlier channels x16, randomly permuted page pool)",
        "config": {"workload": f"{cfg.name}: batch {cfg.batch}, ctx {int(lay.context_lens.max())}, "
                               f"{cfg.num_kv_heads} kv heads, {cfg.num_q_heads} q heads, head_dim {cfg.head_dim}, "
                               f"page {cfg.page_size}, T={cfg.q_per_seq}",
                   "kv_bytes_per_step": nbytes, "flops_per_step": flops, "num_splits": wl.S,
                   "l2": "inputs larger than L2 (KV cache per step >> 126 MB)",
                   "launch": "timed steps captured as one CUDA graph (append, decode split, combine per step)",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline,
        "e2e": {"value": round(e2e_value, 1), "unit": unit,
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
                "how": "kv4_append_quantize + kv4_decode_attention through the Python binding, issued eagerly "
                       "each step; inputs copied from pinned host memory and the output read back every step "
                       "on a second stream, double-buffered (step i+1's copies overlap step i's compute); "
                       "the step's inputs packed in one pinned buffer, one host-to-device copy per step"},
        "gpu_launches": 3 * args.steps,
        "step_parts_ms": {"append": round(append_ms, 5), "decode_split": round(kern_ms, 5),
                          "combine": round(combine_ms, 5),
                          "note": f"append quantises the step's {cfg.batch * cfg.q_per_seq} new tokens x "
                                  f"{cfg.num_kv_heads} kv heads; append and combine timed alone, "
                                  f"{n_parts} launches in a CUDA graph"},
        "clocks": clk.summary(),
    }
    if fp8_info:
        res["fp8_comparator"] = fp8_info
    return res, wl


def oracle_sample(cfg, lay, n_seqs: int, head=None):
    """Build the oracle's cache for the first n_seqs sequences (all but the step's
    new tokens), optionally restricted to one kv head (and its query heads).
    Returns a callable doing one oracle step (append of the new tokens + decode
    attention) and the KV bytes that step reads."""
    import dataclasses
    import oracle
    P, T = cfg.page_size, cfg.q_per_seq
    seqs = list(range(n_seqs))
    Hkv = cfg.num_kv_heads if head is None else 1
    bb = oracle.block_bytes(P, cfg.head_dim)
    kc = np.zeros(lay.num_pages * Hkv * bb, np.uint8)
    vc = None if cfg.latent else np.zeros_like(kc)
    hs = slice(None) if head is None else slice(head, head + 1)
    news = []
    for b in seqs:
        k, v = W.sequence_tokens(cfg, lay, b)
        k = k[:, hs].contiguous()
        v = None if v is None else v[:, hs].contiguous()
        L = int(lay.context_lens[b])
        slots = W.slots_for(lay, b, 0, L, P)
        oracle.append_quantize(k[:L - T], None if v is None else v[:L - T], slots[:L - T], kc, vc, lay.num_pages, P)
        news.append((k[L - T:].contiguous(), None if v is None else v[L - T:].contiguous(), slots[L - T:].copy()))
    q = W.queries(cfg)
    if head is not None:
        G = cfg.group
        q = q[:, :, head * G:(head + 1) * G].contiguous()
    tab = lay.block_tables.clip(min=0)

    def step():
        for k, v, s in news:
            oracle.append_quantize(k, v, s, kc, vc, lay.num_pages, P)
        return oracle.decode_attention(q, kc, vc, tab, lay.context_lens, Hkv, P, lay.num_pages,
                                       cfg.softmax_scale, latent=cfg.latent, seqs=seqs)
    nbytes = kv_bytes_4bit(dataclasses.replace(cfg, num_kv_heads=Hkv), lay.context_lens[:n_seqs])
    return step, nbytes


def cpu_baseline(cfg, lay, budget_s: float = 12.0, single_budget_s: float = 4.0):
    """The oracle on the first sequences of the workload (all kv heads): its
    OpenMP loop runs over the sample's (sequence, kv head) pairs, so the sample
    holds enough sequences to give every host thread one pair; a single-thread
    figure is timed beside it."""
    import oracle
    host = oracle.max_threads()
    n_seqs = max(1, min(cfg.batch, -(-host // cfg.num_kv_heads)))
    step, nbytes = oracle_sample(cfg, lay, n_seqs)
    threads = max(1, min(host, n_seqs * cfg.num_kv_heads))

    def timed(budget):
        n, t0 = 0, time.perf_counter()
        while True:
            step()
            n += 1
            if time.perf_counter() - t0 >= budget:
                break
        return (time.perf_counter() - t0) / n, n

    default_threads = oracle.max_threads()
    oracle.set_threads(threads)
    dt, n = timed(budget_s)
    oracle.set_threads(1)
    dt1, n1 = timed(single_budget_s)
    oracle.set_threads(default_threads)
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_seqs} of {cfg.batch} sequences (all {cfg.num_kv_heads} kv heads, "
                      f"{int(lay.context_lens[:n_seqs].sum())} tokens): append of the step's new tokens + fp64 "
                      f"decode attention; {n} repetitions in {n * dt:.1f} s on {threads} threads",
            "single_thread": {"value": round(nbytes / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"the same sample on one thread, {n1} repetitions in {n1 * dt1:.1f} s"},
            "host_cpus": os.cpu_count()}


def run_reference(args):
    """The CPU oracle as it stands, timed on the host cores.  Each step is one
    bounded sample of the workload: sequence 0, kv head (step mod Hkv) with its
    query heads, the full context (append of the new token + fp64 decode)."""
    cfg = W.CONFIGS[args.config]
    lay = W.make_layout(cfg)
    steps = [oracle_sample(cfg, lay, 1, head=h) for h in range(min(cfg.num_kv_heads, 2))]
    nbytes = steps[0][1]
    for i in range(args.warmup):
        steps[i % len(steps)][0]()
    t0 = time.perf_counter()
    for i in range(args.steps):
        steps[i % len(steps)][0]()
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / dt / 1e9
    threads = int(os.environ.get("OMP_NUM_THREADS", "0")) or (os.cpu_count() or 1)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{cfg.name} (per step: one sequence x one kv head sample)",
                   "kv_bytes_per_step": nbytes},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1 if cfg.group else threads,
                         "kind": "oracle",
                         "sample": f"each step: sequence 0 of {cfg.batch}, one of {cfg.num_kv_heads} kv heads with "
                                   f"its {cfg.group} query heads, {int(lay.context_lens[0])} tokens "
                                   f"(append of the new token + fp64 decode attention)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="b32_ctx32k", choices=sorted(W.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--kernel", type=int, default=0,
                    help="explicit split kernel (KV4_KERNEL_*); 0 = the automatic choice")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res, wl = run_ours(args, rank, world, local_rank)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not is_extend(wl.cfg):
        res["cpu_baseline"] = cpu_baseline(wl.cfg, wl.lay)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
