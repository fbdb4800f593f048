#!/usr/bin/env python3
"""Throughput of the beam-search hot path on GB300: beam-steps/s and logits GB/s.

Workload (the Llama-3-8B-shaped beam step): batch 64 sentences x W 4 beams over
V = 128256, bf16 logits N(0, 2.5) plus a Zipf bias -ln(rank) (synthetic,
seeded), EOS 2, GNMT alpha 0.6, early_stopping False, 200-step decodes after a
1000-token prompt, KV cache 32 layers x 8 KV heads x 128 dims bf16 (128 KiB per
token) in 16-token paged blocks with copy-on-write.

One step = one fused bs_step launch (row LSE, score add, top-2W, EOS /
finished set / stopping test, outputs, sequence gather) + kv_paged_reorder
(table remap, reference counts, free stacks, copy-on-write of shared tail
blocks).  Decodes restart every 200 steps (bs_reset + kv_paged_restore, both
device-side).  The logits rotate through 10 device buffers (657 MB > 4 x L2).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun with N > 1 every rank runs its own batch (weak scaling, no
collective on the data path); the time is the max over ranks.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "beam-steps/s and logits-scanned GB/s (fraction of GB300 HBM peak), 1 GPU"
UNIT = "beam-steps/s"
WORKLOAD = dict(B=64, W=4, V=128256, eos=2, alpha=0.6, T=200, P=1000, L=32, H=8, D=128, block=16, seed=1236)
WORKLOAD_NAME = ("Llama-3-8B-shaped beam step: batch 64, W 4, V 128256 bf16 Zipf-skewed logits, prompt 1000, "
                 "200-step decodes, paged KV 32 layers x 8 KV heads x 128 dims bf16 (16-token blocks, "
                 "copy-on-write)")
RING = 10
LAUNCHES_PER_STEP = 3          # bs_cluster_kernel, kv_paged_remap_kernel, kv_cow_vec_kernel
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------------------------
# helpers (also used by the CPU tests of the multi-rank logic)
# ------------------------------------------------------------------------------------

def dist_env():
    """(rank, local_rank, world) from the torchrun environment (1 process when absent)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def rank_seed(base: int, rank: int) -> int:
    """Each rank decodes its own batch: distinct seeded inputs per rank."""
    return base + 7919 * rank


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_sha(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "verify_bs_step_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the kernel changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
        if rec["source_sha"] != source_sha(*rec["sources"]):
            return None
        return rec
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, filtered to a time window."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = []
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts + frac, float(parts[1]), float(parts[2]), parts[5:9]))
            except Exception:
                continue
        os.unlink(self.file.name)
        inside = [r for r in rows if t0 - 0.06 <= r[0] <= t1 + 0.06] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


class NvmlClocks:
    """SM clock and clock-event reasons read through NVML (ctypes, read-only) every ~0.2 ms
    from a host thread while the timed region runs; None if NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int):
        self.samples, self.stop_flag, self.thread, self.lib, self.dev = [], False, None, None, None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            dev = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(dev)) != 0:
                return
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(dev, 1, ctypes.byref(mx)) == 0 else None
            self.lib, self.dev = lib, dev
        except Exception:
            self.lib = None

    def _run(self):
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_flag:
            if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(mhz)) == 0:
                r = rs.value if self.reasons_fn(self.dev, ctypes.byref(rs)) == 0 else 0
                self.samples.append((float(mhz.value), int(r)))
            time.sleep(0.0002)

    def start(self):
        if self.lib is None:
            return
        import threading
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self):
        if self.lib is None or self.thread is None:
            return None
        self.stop_flag = True
        self.thread.join()
        if not self.samples:
            return None
        reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples), "source": "NVML during the timed region"}


# ------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------

def make_logits_ring(torch, synth, n, seed, device, B, W, V):
    bias = synth.zipf_bias(V, seed, device)
    ring = []
    for i in range(n):
        ring.append(synth.batch_logits("llama", B, W, V, seed=seed, step=1000 + i, dtype=torch.bfloat16,
                                       bias=bias, device=device))
    return ring


def run_ours(args, rank, local_rank, world):
    import torch

    import synth
    import verify_bs_step_gb300 as vbs
    from verify_bs_step_gb300 import _build

    torch.cuda.set_device(local_rank)
    if rank == 0:
        _build.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    dev = torch.device("cuda", local_rank)
    wl = dict(WORKLOAD)
    B, W, V, T, P = wl["B"], wl["W"], wl["V"], wl["T"], wl["P"]
    L, H, D, blk = wl["L"], wl["H"], wl["D"], wl["block"]
    R = B * W
    seed = rank_seed(wl["seed"], rank)
    stream = torch.cuda.Stream(dev)
    L_ = vbs.lib()
    with torch.cuda.stream(stream):
        ring = make_logits_ring(torch, synth, RING, seed, dev, B, W, V)
        bs = vbs.BeamSearch(B, W, V, eos=wl["eos"], alpha=wl["alpha"], early_stopping=vbs.ES_FALSE,
                            lp_kind=vbs.LP_GNMT, max_len=T, dtype=torch.bfloat16, device=dev)
        S = -(-P // blk) + W * (-(-T // blk) + 2)
        MB = -(-(P + T + 1) // blk) + 1
        pk = vbs.PagedKV(B, W, L, H, D, blocks_per_sentence=S, max_blocks=MB, block=blk, dtype=torch.bfloat16,
                         device=dev)
        pk.prefill(P)
        # the prompt's K/V content does not change the work; the pool starts zeroed
        pk.prepare(P)
        pk.save()
        torch.cuda.synchronize(dev)

        vp = ctypes.c_void_p
        ctx_bs, ctx_pk = bs.ctx, pk.ctx
        p_scores, p_seqs = vp(bs.scores.data_ptr()), vp(bs.seqs.data_ptr())
        p_bi, p_tok, p_done = vp(bs.beam_idx.data_ptr()), vp(bs.tokens.data_ptr()), vp(bs.all_done.data_ptr())
        p_ring = [vp(x.data_ptr()) for x in ring]
        bs_step, paged_reorder = L_.bs_step, L_.kv_paged_reorder
        bs_reset, paged_restore = L_.bs_reset, L_.kv_paged_restore

        state = {"t": 0, "launches": 0, "resets": 0}

        def restart():
            assert bs_reset(ctx_bs, p_scores, p_seqs) == 0
            assert paged_restore(ctx_pk) == 0
            state["t"] = 0
            state["launches"] += 1
            state["resets"] += 1

        def one_step(i, ev=None):
            if state["t"] == T:
                restart()
            if ev is not None:
                ev[0].record(stream)
            st = bs_step(ctx_bs, p_ring[i % RING], V, p_scores, p_seqs, p_bi, p_tok, p_done)
            if ev is not None:
                ev[1].record(stream)
            st |= paged_reorder(ctx_pk, p_bi, P + state["t"])
            if ev is not None:
                ev[2].record(stream)
            state["t"] += 1
            state["launches"] += LAUNCHES_PER_STEP
            if st:
                raise RuntimeError(f"step failed: {st}")

        restart()
        for i in range(args.warmup):
            one_step(i)
        torch.cuda.synchronize(dev)

        # The timed loop replays CUDA graphs of decode segments, so host launch cost stays
        # out of it.  It starts mid-decode: a restart and the first S0 steps run untimed right
        # before it; inside it the decode runs on to step T, then restarts every T steps as in
        # the workload.
        K = args.steps
        S0 = min(20, T - 1)

        def capture(n, start_t):
            g = torch.cuda.CUDAGraph()
            state["launches"] = 0
            with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
                if start_t == 0:
                    restart()
                else:
                    state["t"] = start_t
                for i in range(n):
                    one_step(i)
            return g, n, state["launches"]

        lead = capture(S0, 0)                            # untimed: a restart and S0 steps
        n1 = min(K, T - S0)
        graphs = [capture(n1, S0)]                       # (graph, steps, launches)
        rest = K - n1
        if rest // T:
            graphs += [capture(T, 0)] * (rest // T)
        if rest % T:
            graphs.append(capture(rest % T, 0))
        for g, _, _ in [lead] + list({id(x[0]): x for x in graphs}.values()):
            g.replay()                                   # each graph once, untimed
        lead[0].replay()
        torch.cuda.synchronize(dev)
        cow0 = pk.cow_slots()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks = ClockSampler(local_rank)
        clocks.start()
        poll = NvmlClocks(local_rank)
        time.sleep(0.3)
        torch.cuda.synchronize(dev)
        poll.start()
        w0 = time.time()
        e0.record(stream)
        h0 = time.perf_counter()
        for g, _, _ in graphs:
            g.replay()
        h1 = time.perf_counter()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        w1 = time.time()
        polled = poll.stop()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        clk = polled if polled is not None else clocks.stop(w0, w1)
        if polled is not None:
            clocks.stop(w0, w1)
        ms = e0.elapsed_time(e1)
        assert bs.status() == 0 and pk.status() == 0
        cow_slots_timed = pk.cow_slots() - cow0
        launches = sum(n for _, _, n in graphs)

        # Per-kernel times (outside the timed loop): each call bracketed by events, the
        # host queueing ahead of the GPU behind a spin, so no host gap lands between events.
        t_bs, t_kv = [], []
        restart()
        for rep in range(3):
            n = min(T - 1, 150)
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
            torch.cuda.synchronize(dev)
            torch.cuda._sleep(60_000_000)
            restart()
            for i in range(n):
                one_step(i, evs[i])
            torch.cuda.synchronize(dev)
            t_bs += [evs[i][0].elapsed_time(evs[i][1]) for i in range(5, n)]
            t_kv += [evs[i][1].elapsed_time(evs[i][2]) for i in range(5, n)]
        assert bs.status() == 0 and pk.status() == 0

    ms_max = max_over_ranks(ms, world, dev)
    steps_all = K * world
    value = steps_all / (ms_max / 1e3)
    peak, peak_kind = measured_peaks()
    es = 2
    bytes_bs = R * V * es + R * 16                      # logits once + scores/tokens/beam_idx/append
    avg_bs_ms = statistics.fmean(t_bs)
    ach_bs = bytes_bs / (avg_bs_ms / 1e3) / 1e9
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_max / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "global_batch": B * world, "beams": W, "vocab": V,
                   "prompt": P, "decode_steps": T, "kv": "paged 16-token blocks, copy-on-write",
                   "parallelism": f"replicas x{world} (sentences sharded, no collective)",
                   "l2": f"logits rotate through {RING} device buffers of {R * V * es / 1e6:.1f} MB "
                         f"({RING * R * V * es / 1e6:.0f} MB > 4 x L2)"},
        "logits_gbs": round(R * V * es * steps_all / (ms_max / 1e3) / 1e9, 1),
        "rows_steps_per_s": round(value * R, 1),
        "kernel_ms": {"bs_step_avg": round(avg_bs_ms, 5), "bs_step_median": round(statistics.median(t_bs), 5),
                      "kv_paged_reorder_avg": round(statistics.fmean(t_kv), 5),
                      "host_ms_per_step_timed_loop": round((h1 - h0) * 1e3 / K, 5),
                      "note": "per-kernel times from a separate pass of event-bracketed calls queued "
                              "ahead of the GPU; the timed loop replays CUDA graphs of whole decodes"},
        "gpu_launches": launches,
        "clocks": clk,
    }
    rec = recorded_traffic("bs_step_kernel")
    out["roofline"] = {"kernel": "bs_cluster_kernel (one launch per step)", "bound": "hbm", "achieved": round(ach_bs, 1),
                       "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                       "frac": round(ach_bs / peak, 4),
                       "traffic": rec["dram_bytes_per_launch"] if rec else None,
                       "algorithmic_bytes": bytes_bs}
    # copy-on-write bytes actually moved in the timed region (read + write), per reorder call
    cow_bytes = 2 * cow_slots_timed * D * es / K
    avg_kv_ms = statistics.fmean(t_kv)
    out["roofline_kv_paged"] = {"kernels": "kv_paged_remap_kernel + kv_cow_vec_kernel", "bound": "hbm",
                                "achieved": round(cow_bytes / (avg_kv_ms / 1e3) / 1e9, 1), "peak": peak,
                                "unit": "GB/s", "frac": round(cow_bytes / (avg_kv_ms / 1e3) / 1e9 / peak, 4),
                                "algorithmic_bytes": int(cow_bytes), "traffic": None}
    share_bs = sum(t_bs) / max(1e-9, sum(t_bs) + sum(t_kv))
    out["time_share"] = {"bs_step": round(share_bs, 3), "kv_paged_reorder": round(1 - share_bs, 3)}

    # the chip's bandwidth measured in this run by the library's own kernels
    out["peak_inrun"] = run_peaks(torch, vbs, dev, stream, ring)
    # end to end through the public API with host buffers
    out["e2e"] = run_e2e(args, torch, vbs, synth, dev, stream, ring, seed, world)
    if rank == 0 and world == 1 and not args.no_extras:
        out["extra"] = run_extras(args, torch, vbs, synth, dev, stream, peak)
    bs.close()
    pk.close()
    return out


def run_peaks(torch, vbs, dev, stream, ring):
    """In-run memory peaks from the library's own kernels: a vector copy over 1 GiB (read +
    write bytes, best of 10), and read-only streaming over one step's logits (65.67 MB,
    rotating over the logits ring so every launch reads HBM) at 128, #SM and 2 x #SM CTAs,
    both as the mean of 50 back-to-back launches and as the median of event-bracketed
    single launches."""
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {"sms": nsm}
    with torch.cuda.stream(stream):
        n = 1 << 30
        a = torch.empty(n // 2, dtype=torch.bfloat16, device=dev).fill_(1.0)
        b = torch.empty_like(a)
        best = None
        for rep in range(12):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            vbs.peak_copy(a, b, 4 * nsm)
            e1.record(stream)
            e1.synchronize()
            if rep >= 2:
                ms = e0.elapsed_time(e1)
                best = ms if best is None else min(best, ms)
        out["copy_gbs"] = round(2 * n / (best / 1e3) / 1e9, 1)
        del a, b
        sink = torch.zeros(4 * nsm, dtype=torch.int32, device=dev)
        nbytes = ring[0].nbytes
        reads = {}
        for mode, tag in ((1, "ring"), (0, "ld")):
            for grid in (128, nsm, 2 * nsm):
                for i in range(5):
                    vbs.peak_read(ring[i % len(ring)], grid, mode, sink)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for i in range(50):
                    vbs.peak_read(ring[i % len(ring)], grid, mode, sink)
                e1.record(stream)
                e1.synchronize()
                b2b = e0.elapsed_time(e1) / 50
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(30)]
                torch.cuda._sleep(20_000_000)
                for i, (x, y) in enumerate(evs):
                    x.record(stream)
                    vbs.peak_read(ring[i % len(ring)], grid, mode, sink)
                    y.record(stream)
                torch.cuda.synchronize(dev)
                single = statistics.median(x.elapsed_time(y) for x, y in evs)
                reads[f"{tag}_{grid}"] = {"us_back_to_back": round(b2b * 1e3, 2), "gbs_back_to_back":
                                          round(nbytes / (b2b / 1e3) / 1e9, 1), "us_single": round(single * 1e3, 2),
                                          "gbs_single": round(nbytes / (single / 1e3) / 1e9, 1)}
        out["read_bytes"] = nbytes
        out["read"] = reads
    assert vbs.lib().vbs_stateless_status(vbs._stream(dev)) == 0
    return out


def run_e2e(args, torch, vbs, synth, dev, stream, ring, seed, world):
    """Same metric through BeamSearch.step / PagedKV.reorder, inputs copied from pinned host memory."""
    wl = WORKLOAD
    B, W, V, T, P = wl["B"], wl["W"], wl["V"], wl["T"], wl["P"]
    L, H, D, blk = wl["L"], wl["H"], wl["D"], wl["block"]
    R = B * W
    K = max(50, min(args.steps // 10, 2000))
    with torch.cuda.stream(stream):
        host = [x.cpu().pin_memory() for x in ring]
        dbuf = torch.empty_like(ring[0])
        bs = vbs.BeamSearch(B, W, V, eos=wl["eos"], alpha=wl["alpha"], max_len=T, dtype=torch.bfloat16, device=dev)
        S = -(-P // blk) + W * (-(-T // blk) + 2)
        MB = -(-(P + T + 1) // blk) + 1
        pk = vbs.PagedKV(B, W, L, H, D, blocks_per_sentence=S, max_blocks=MB, block=blk, dtype=torch.bfloat16,
                         device=dev)
        pk.prefill(P)
        pk.prepare(P)
        pk.save()
        outs = [torch.empty(3, R, dtype=torch.int32).pin_memory() for _ in range(4)]
        for i in range(3):                       # warm-up, untimed
            dbuf.copy_(host[i], non_blocking=True)
            bi, tok, sc = bs.step(dbuf)
            pk.reorder(bi, P + i)
        bs.reset()
        pk.restore()
        t = 0
        # the next step's logits copy on a second stream while this step computes (two device
        # buffers; each copy waits until the step two back has released its buffer)
        copy_s = torch.cuda.Stream(dev)
        dbufs = [dbuf, torch.empty_like(dbuf)]
        ready = [torch.cuda.Event() for _ in range(2)]
        free = [torch.cuda.Event() for _ in range(2)]
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0 = time.perf_counter()
        e0.record(stream)
        copy_s.wait_stream(stream)
        with torch.cuda.stream(copy_s):
            dbufs[0].copy_(host[0], non_blocking=True)
            ready[0].record(copy_s)
        for i in range(K):
            j = i % 2
            if i + 1 < K:
                with torch.cuda.stream(copy_s):
                    if i >= 1:
                        copy_s.wait_event(free[1 - j])
                    dbufs[1 - j].copy_(host[(i + 1) % RING], non_blocking=True)
                    ready[1 - j].record(copy_s)
            if t == T:
                bs.reset()
                pk.restore()
                t = 0
            stream.wait_event(ready[j])
            bi, tok, sc = bs.step(dbufs[j])
            pk.reorder(bi, P + t)
            free[j].record(stream)
            o = outs[i % 4]
            o[0].copy_(bi, non_blocking=True)
            o[1].copy_(tok, non_blocking=True)
            o[2].copy_(sc.view(torch.int32), non_blocking=True)
            t += 1
        e1.record(stream)
        torch.cuda.synchronize(dev)
        w1 = time.perf_counter()
        ms = e0.elapsed_time(e1)
        wall_ms = (w1 - w0) * 1e3
        bs.close()
        pk.close()
    ms_max = max_over_ranks(max(ms, wall_ms), world, dev)
    return {"value": round(K * world / (ms_max / 1e3), 2), "unit": UNIT, "steps": K,
            "h2d_bytes_per_step": R * V * 2, "d2h_bytes_per_step": R * 12,
            "note": "BeamSearch.step + PagedKV.reorder; logits copied from pinned host memory each step "
                    "(the next step's copy overlaps this step's compute, two device buffers), "
                    "beam_idx/tokens/scores copied back each step"}


def _timed(torch, stream, fn, reps, ahead=True):
    """Event-bracketed calls; with `ahead`, the host queues them behind a GPU spin so that no
    host launch gap lands between a call's events."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    torch.cuda.synchronize()
    if ahead:
        torch.cuda._sleep(int(2e5) * reps)
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def _looped(torch, stream, fn, reps):
    """Mean time of `reps` back-to-back calls between two events, queued behind a GPU spin
    (calls in a row, as in a decode loop: a call's launch may overlap the previous call)."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    torch.cuda._sleep(int(2e5) * reps)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def run_extras(args, torch, vbs, synth, dev, stream, peak):
    """Secondary lines: bs_step alone (Llama, T-base), naive KV gather, blockwise verify."""
    import ctypes
    extra = {}
    with torch.cuda.stream(stream):
        # -- bs_step alone, Llama and T-base shapes --------------------------------------
        # bs_step_two_pass_llama: the two-pass coarse-selection ablation on the same workload
        for name, kind, B, W, V, T in (("bs_step_llama", "llama", 64, 4, 128256, 200),
                                       ("bs_step_tbase", "tbase", 128, 4, 32000, 64),
                                       ("bs_step_two_pass_llama", "llama", 64, 4, 128256, 200)):
            R = B * W
            n = max(RING, -(-4 * 129_000_000 // (R * V * 2)) + 1)
            if kind == "llama":
                ring = make_logits_ring(torch, synth, n, 99, dev, B, W, V)
            else:
                ring = [synth.batch_logits("tbase", B, W, V, seed=98, step=i, dtype=torch.bfloat16, device=dev)
                        for i in range(n)]
            bs = vbs.BeamSearch(B, W, V, eos=2, alpha=0.6, max_len=T, dtype=torch.bfloat16, device=dev)
            L_ = vbs.lib()
            vp = ctypes.c_void_p
            a_ = [vp(bs.scores.data_ptr()), vp(bs.seqs.data_ptr()), vp(bs.beam_idx.data_ptr()),
                  vp(bs.tokens.data_ptr()), vp(bs.all_done.data_ptr())]
            prs = [vp(x.data_ptr()) for x in ring]
            step_fn = L_.bs_step_two_pass if name.startswith("bs_step_two_pass") else L_.bs_step
            ts, i = [], 0
            while len(ts) < 400:
                # one decode: the first step (only beam 0 of each sentence is live) is not timed
                L_.bs_reset(bs.ctx, a_[0], a_[1])
                step_fn(bs.ctx, prs[i % n], V, *a_)
                i += 1
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(T - 1)]
                torch.cuda._sleep(int(2e5) * (T - 1))      # the host queues the decode ahead of the GPU
                for e_a, e_b in evs:
                    e_a.record(stream)
                    step_fn(bs.ctx, prs[i % n], V, *a_)
                    e_b.record(stream)
                    i += 1
                torch.cuda.synchronize()
                ts.extend(e_a.elapsed_time(e_b) for e_a, e_b in evs)
            ts = ts[20:]                                            # the first ones warm up
            byts = R * V * 2 + R * 16
            avg = statistics.fmean(ts)
            extra[name] = {"B": B, "W": W, "V": V, "avg_us": round(avg * 1e3, 3),
                           "steps_per_s": round(1e3 / avg, 1), "achieved_gbs": round(byts / (avg / 1e3) / 1e9, 1),
                           "frac_of_peak": round(byts / (avg / 1e3) / 1e9 / peak, 4), "bytes": byts}
            if step_fn is not L_.bs_step:
                extra[name]["logit_bytes_read"] = 2 * R * V * 2       # two passes over the logits
            bs.close()
            del ring
        # -- naive KV gather at the Llama shape (t_valid = 1000) ---------------------------
        try:
            L, Rk, H, Tm, D = 32, 256, 8, 1008, 128
            src = torch.zeros(L, 2, Rk, H, Tm, D, dtype=torch.bfloat16, device=dev)
            dst = torch.zeros_like(src)
            bi = torch.arange(Rk, dtype=torch.int32, device=dev).flip(0)
            ts = _timed(torch, stream, lambda: vbs.kv_reorder(src, dst, bi, 1000), 3)
            byts = 2 * L * 2 * Rk * H * 1000 * D * 2
            avg = statistics.fmean(ts[1:])
            extra["kv_naive_llama_t1000"] = {"avg_ms": round(avg, 3), "bytes": byts,
                                             "achieved_gbs": round(byts / (avg / 1e3) / 1e9, 1),
                                             "frac_of_peak": round(byts / (avg / 1e3) / 1e9 / peak, 4)}
            del src, dst
        except torch.cuda.OutOfMemoryError:
            extra["kv_naive_llama_t1000"] = "out of memory"
        torch.cuda.empty_cache()
        # -- blockwise verify: [256, 8, 8, 32000] bf16 ---------------------------------------
        B, k, V = 256, 8, 32000
        bufs = []
        for i in range(4):
            base, props, heads = synth.geometric_prefix_proposals(B, k, V, seed=500 + i, step=i)
            logits = synth.planted_rows(heads.to(dev), V, seed=500 + i, salt=i, device=dev)
            agree = torch.ones(B, dtype=torch.int64)
            run = torch.ones(B, dtype=torch.bool)
            for q in range(1, k):
                run &= props[:, q] == base[:, q - 1]
                agree += run.long()
            bufs.append((logits, props.to(torch.int32).to(dev), agree))
        khat = torch.empty(B, dtype=torch.int32, device=dev)
        nxt = torch.empty(B, k, dtype=torch.int32, device=dev)
        cnt = {"i": 0}

        def verify():
            lg, pr, _ = bufs[cnt["i"] % 4]
            vbs.bpd_verify(lg, pr, -1, khat, nxt)
            cnt["i"] += 1

        for _ in range(8):
            verify()
        reps = 100
        ts = _timed(torch, stream, verify, reps)
        byts = [int(((b[2] + k - 1) * V * 2).sum().item()) + B * k * 12 for b in bufs]
        alg = statistics.fmean(byts[(8 + i) % 4] for i in range(reps))
        avg = statistics.fmean(ts)
        loop = _looped(torch, stream, verify, reps)
        extra["bpd_verify"] = {"B": B, "k": k, "V": V, "avg_us": round(loop * 1e3, 3),
                               "iters_per_s": round(1e3 / loop, 1), "mean_khat": round(float(bufs[0][2].float().mean()), 3),
                               "algorithmic_bytes": int(alg), "achieved_gbs": round(alg / (loop / 1e3) / 1e9, 1),
                               "frac_of_peak": round(alg / (loop / 1e3) / 1e9 / peak, 4),
                               "per_call_us": round(avg * 1e3, 3),
                               "per_call_frac_of_peak": round(alg / (avg / 1e3) / 1e9 / peak, 4),
                               "timing": f"avg_us: {reps} calls back to back between two events (a call's launch "
                                         f"overlaps the previous call); per_call_us: each call between its own events"}
        # the relaxed verify tests of §5 on the same inputs: the rows read are still
        # khat + k - 1 per element, khat now from the relaxed test (taken from the call)
        for name, crit, param in (("bpd_verify_topk2", vbs.BPD_TOPK, 2), ("bpd_verify_distance1", vbs.BPD_DISTANCE, 1)):
            kh_r = []
            for j in range(4):
                lg, pr, _ = bufs[j]
                kh_j, _ = vbs.bpd_verify(lg, pr, -1, criterion=crit, param=param)
                kh_r.append(kh_j.to(torch.int64).cpu())

            def verify_r():
                lg, pr, _ = bufs[cnt["i"] % 4]
                vbs.bpd_verify(lg, pr, -1, khat, nxt, criterion=crit, param=param)
                cnt["i"] += 1

            cnt["i"] = 0
            for _ in range(8):
                verify_r()
            ts = _timed(torch, stream, verify_r, reps)
            byts_r = [int(((kh_r[j] + k - 1) * V * 2).sum().item()) + B * k * 12 for j in range(4)]
            alg_r = statistics.fmean(byts_r[(8 + i) % 4] for i in range(reps))
            avg_r = statistics.fmean(ts)
            loop_r = _looped(torch, stream, verify_r, reps)
            extra[name] = {"criterion": name.split("_")[-1], "avg_us": round(loop_r * 1e3, 3),
                           "mean_khat": round(float(torch.cat(kh_r).float().mean()), 3),
                           "algorithmic_bytes": int(alg_r), "achieved_gbs": round(alg_r / (loop_r / 1e3) / 1e9, 1),
                           "frac_of_peak": round(alg_r / (loop_r / 1e3) / 1e9 / peak, 4),
                           "per_call_us": round(avg_r * 1e3, 3)}
    return extra


def run_sweep(only=None):
    """bs_step alone over the sweep grid: batch {1, 32, 256} x W {1, 4, 16} x V {32000, 128256,
    256000} x {fp32, bf16}, N(0, 2) logits with the EOS logit lifted above the row maximum on ~2 % of
    rows, GNMT alpha 0.6, early_stopping False.  One JSON line per shape.

    Each shape runs 50-step decodes (the first step of each, where only beam 0 is live, untimed)
    until 200 steps are timed; every step reads a different logits buffer of a ring that spans
    more than 4 x L2 (distinct batches up to 32 of them, then copies at other addresses)."""
    import torch

    import synth
    import verify_bs_step_gb300 as vbs
    from verify_bs_step_gb300 import _build

    _build.build()
    dev = torch.device("cuda", 0)
    peak, peak_src = measured_peaks()
    stream = torch.cuda.Stream(dev)
    vp = ctypes.c_void_p
    T, EOS = 50, 7
    for V in (32000, 128256, 256000):
        for B in (1, 32, 256):
            for W in (1, 4, 16):
                for dt, dname, esz in ((torch.float32, "f32", 4), (torch.bfloat16, "bf16", 2)):
                    if only and (B, W, V, dname) not in only:
                        continue
                    R = B * W
                    per = R * V * esz
                    n = max(2, -(-4 * 129_000_000 // per) + 1)
                    base = [synth.batch_logits("sweep", B, W, V, seed=2024 + i, step=i, eos=EOS, dtype=dt,
                                               device=dev) for i in range(min(n, 32))]
                    ring = [base[i] if i < len(base) else base[i % len(base)].clone() for i in range(n)]
                    with torch.cuda.stream(stream):
                        bs = vbs.BeamSearch(B, W, V, eos=EOS, alpha=0.6, early_stopping=vbs.ES_FALSE, max_len=T,
                                            dtype=dt, device=dev)
                        L_ = vbs.lib()
                        a_ = [vp(bs.scores.data_ptr()), vp(bs.seqs.data_ptr()), vp(bs.beam_idx.data_ptr()),
                              vp(bs.tokens.data_ptr()), vp(bs.all_done.data_ptr())]
                        prs = [vp(x.data_ptr()) for x in ring]
                        ts, i = [], 0
                        while len(ts) < 210:
                            L_.bs_reset(bs.ctx, a_[0], a_[1])
                            L_.bs_step(bs.ctx, prs[i % n], V, *a_)
                            i += 1
                            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                                   for _ in range(T - 1)]
                            torch.cuda.synchronize()
                            torch.cuda._sleep(int(2e5) * (T - 1))
                            for e_a, e_b in evs:
                                e_a.record(stream)
                                L_.bs_step(bs.ctx, prs[i % n], V, *a_)
                                e_b.record(stream)
                                i += 1
                            torch.cuda.synchronize()
                            ts.extend(e_a.elapsed_time(e_b) for e_a, e_b in evs)
                        assert bs.status() == 0
                        bs.close()
                    ts = ts[10:]
                    avg = statistics.fmean(ts)
                    byts = per + R * 16
                    gbs = byts / (avg / 1e3) / 1e9
                    print(json.dumps({"sweep": {"B": B, "W": W, "V": V, "dtype": dname}, "avg_us": round(avg * 1e3, 3),
                                      "median_us": round(statistics.median(ts) * 1e3, 3),
                                      "steps_per_s": round(1e3 / avg, 1), "bytes": byts,
                                      "achieved_gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
                                      "peak": f"{peak} GB/s ({peak_src})", "ring": n}), flush=True)
                    del ring, base
                    torch.cuda.empty_cache()


# ------------------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and the reference arm)
# ------------------------------------------------------------------------------------

def oracle_sample(seconds: float, seed: int = 1236, max_units: int | None = None):
    """Time the oracle's beam step + paged reorder on sampled sentences of the workload.

    Returns (sentence_steps, elapsed_s, description).  One unit = one sentence's
    step: log-softmax of its W rows, the walk, and its KV table remap with
    copy-on-write (the pool at full Llama size for that one sentence).
    """
    import numpy as np
    import torch

    import synth
    from oracle import beam as obeam
    from oracle import kv as okv

    wl = WORKLOAD
    W, V, P, T = wl["W"], wl["V"], wl["P"], wl["T"]
    bias = synth.zipf_bias(V, seed)
    ora = obeam.BeamSearch(1, W, V, eos=wl["eos"], alpha=wl["alpha"], max_len=T)
    kv = okv.PagedKV(1, W, -(-P // 16) + W * 16, wl["L"], wl["H"], wl["D"], block=16, dtype=np.float32)
    kv.prefill(P)
    kv.prepare(P)
    units, t = 0, 0
    t0 = time.perf_counter()
    while True:
        t += 1
        rows = synth.beam_logits("llama", W, V, seed=seed, step=t, sentence=0, dtype=torch.bfloat16, bias=bias)
        res = ora.step(rows.float().numpy())
        kv.reorder(res.beam_idx, P + t - 1)
        units += 1
        el = time.perf_counter() - t0
        if el >= seconds or (max_units and units >= max_units) or t >= T:
            if el >= seconds or (max_units and units >= max_units):
                break
            ora.reset()
            kv = okv.PagedKV(1, W, -(-P // 16) + W * 16, wl["L"], wl["H"], wl["D"], block=16, dtype=np.float32)
            kv.prefill(P)
            kv.prepare(P)
            t = 0
    return units, time.perf_counter() - t0


def _oracle_worker(seconds, seed, start, out):
    """One process of the all-core sample: its own sentence, timed after every worker is ready."""
    os.environ["OMP_NUM_THREADS"] = "1"
    import torch
    torch.set_num_threads(1)
    oracle_sample(0.0, seed=seed, max_units=1)          # imports and first-touch outside the timing
    start.wait()
    out.put(oracle_sample(seconds, seed=seed))


def oracle_all_cores(seconds: float, n: int | None = None):
    """The oracle over independent sentences, one spawned process per host core (sentences do not
    interact, so the batch splits across processes).  Returns (sentence_steps, elapsed_s, cores)."""
    import multiprocessing as mp
    if n is None:
        n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    ctx = mp.get_context("spawn")
    start, out = ctx.Barrier(n), ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(seconds, 1236 + 7919 * i, start, out)) for i in range(n)]
    for p in procs:
        p.start()
    res = [out.get(timeout=600) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    return sum(u for u, _ in res), max(e for _, e in res), n


def cpu_baseline(seconds: float):
    units, el = oracle_sample(seconds)
    B = WORKLOAD["B"]
    out = {"value": round(units / B / el, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": f"{units} sentence-steps of the workload (one sentence's W rows: fp64 log-softmax, "
                     f"top-2W walk, paged KV remap + copy-on-write on a full-size pool), scaled by 1/{B} "
                     f"to full-batch beam-steps; {el:.1f} s on 1 host core"}
    try:
        ua, ea, n = oracle_all_cores(seconds)
        out["all_cores"] = {"value": round(ua / B / ea, 4), "unit": UNIT, "cores": n,
                            "sample": f"{ua} sentence-steps in {ea:.1f} s, {n} processes (one per core, "
                                      f"one sentence each, 1 thread each)"}
    except Exception as e:                               # the single-core figure stands on its own
        out["all_cores"] = f"not measured: {type(e).__name__}: {e}"
    return out


def run_reference(args, rank, world):
    """The oracle as its own arm, on whole steps of the workload: each step is the fp64 beam
    step of all B sentences (log-softmax of every row, the top-2W walk, finished sets) and the
    paged KV reorder of the whole batch (table remap, reference counts, copy-on-write), decodes
    restarting every T steps.  The pool holds 2-byte elements, as the workload's bf16 cache
    does (numpy has no bf16; float16 moves the same bytes).  The logits come from a ring of
    whole-batch tensors generated before the timed region."""
    if rank != 0:
        return None
    import numpy as np
    import torch

    import synth
    from oracle import beam as obeam
    from oracle import kv as okv

    torch.set_num_threads(1)
    wl = WORKLOAD
    B, W, V, P, T, blk = wl["B"], wl["W"], wl["V"], wl["P"], wl["T"], wl["block"]
    S = -(-P // blk) + W * (-(-T // blk) + 2)
    bias = synth.zipf_bias(V, wl["seed"])
    ring = [synth.batch_logits("llama", B, W, V, seed=wl["seed"], step=1000 + i, dtype=torch.bfloat16, bias=bias)
            for i in range(4)]
    state = {}

    def restart():
        state["ora"] = obeam.BeamSearch(B, W, V, eos=wl["eos"], alpha=wl["alpha"], max_len=T)
        kv = okv.PagedKV(B, W, S, wl["L"], wl["H"], wl["D"], block=blk, dtype=np.float16)
        kv.prefill(P)
        kv.prepare(P)
        state["kv"], state["t"] = kv, 0

    def one_step(i):
        if state["t"] == T:
            restart()
        res = state["ora"].step(ring[i % len(ring)].float().numpy())
        state["t"] += 1
        state["kv"].reorder(res.beam_idx, P + state["t"] - 1)

    restart()
    for i in range(args.warmup):
        one_step(i)
    restart()
    t0 = time.perf_counter()
    for i in range(args.steps):
        one_step(i)
    el = time.perf_counter() - t0
    value = args.steps / el
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD_NAME, "global_batch": B, "beams": W, "vocab": V, "prompt": P,
                       "decode_steps": T, "kv": "paged 16-token blocks, copy-on-write",
                       "sample": "whole-batch steps"},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} whole-batch steps ({B} sentences each) in {el:.1f} s on one "
                                       f"host core, after {args.warmup} untimed"},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_profile(kernel: str):
    """A few launches of one kernel on its workload, for ncu (inputs > L2, a few GB at most)."""
    import torch

    import synth
    import verify_bs_step_gb300 as vbs
    from verify_bs_step_gb300 import _build

    _build.build()
    dev = torch.device("cuda", 0)
    wl = WORKLOAD
    if kernel in ("bs_step", "bs_step_two_pass"):
        B, W, V, T = wl["B"], wl["W"], wl["V"], wl["T"]
        ring = make_logits_ring(torch, synth, 3, wl["seed"], dev, B, W, V)
        bs = vbs.BeamSearch(B, W, V, eos=wl["eos"], alpha=wl["alpha"], max_len=T, dtype=torch.bfloat16, device=dev)
        for i in range(8):
            if kernel == "bs_step":
                bs.step(ring[i % 3])
            else:
                bs.step_two_pass(ring[i % 3])
        bs.close()
    elif kernel == "bs_step_w16":
        # the wide-beam sweep shape 256 x 16 x 32000 bf16 (two-kernel path, K = 32)
        B, W, V = 256, 16, 32000
        ring = [synth.batch_logits("sweep", B, W, V, seed=2024 + i, step=i, eos=7, dtype=torch.bfloat16, device=dev)
                for i in range(3)]
        bs = vbs.BeamSearch(B, W, V, eos=7, alpha=0.6, max_len=50, dtype=torch.bfloat16, device=dev)
        for i in range(6):
            bs.step(ring[i % 3])
        bs.close()
    elif kernel == "bpd_verify":
        B, k, V = 256, 8, 32000
        base, props, heads = synth.geometric_prefix_proposals(B, k, V, seed=500, step=0)
        logits = synth.planted_rows(heads.to(dev), V, seed=500, salt=0, device=dev)
        pr = props.to(torch.int32).to(dev)
        for _ in range(6):
            vbs.bpd_verify(logits, pr)
    elif kernel == "kv_paged":
        # 8 of the workload's 64 sentences: the same per-sentence remap and copy work,
        # a 2 GB pool instead of 16.5 GB (a profiler saves and restores device memory)
        B, W, V, T, P = 8, wl["W"], wl["V"], wl["T"], wl["P"]
        L, H, D, blk = wl["L"], wl["H"], wl["D"], wl["block"]
        ring = make_logits_ring(torch, synth, 3, wl["seed"], dev, B, W, V)
        bs = vbs.BeamSearch(B, W, V, eos=wl["eos"], alpha=wl["alpha"], max_len=T, dtype=torch.bfloat16, device=dev)
        S = -(-P // blk) + W * (-(-T // blk) + 2)
        MB = -(-(P + T + 1) // blk) + 1
        pk = vbs.PagedKV(B, W, L, H, D, blocks_per_sentence=S, max_blocks=MB, block=blk, device=dev)
        pk.prefill(P)
        pk.prepare(P)
        for i in range(8):
            bi, _, _ = bs.step(ring[i % 3])
            pk.reorder(bi, P + i)
        bs.close()
        pk.close()
    else:
        raise SystemExit(f"unknown kernel {kernel}")
    torch.cuda.synchronize()
    print(f"profile run of {kernel}: ok")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="skip the secondary lines")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle time budget for cpu_baseline")
    ap.add_argument("--profile", default=None, help="run a few launches of one kernel (for ncu) and exit")
    ap.add_argument("--sweep", action="store_true", help="time bs_step alone over the sweep grid and exit")
    args = ap.parse_args(argv)
    if args.profile:
        run_profile(args.profile)
        return
    if args.sweep:
        run_sweep()
        return
    rank, local_rank, world = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, local_rank, world)
        if rank == 0 and world == 1:
            out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
