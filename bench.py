"""Benchmark: masked attention forward on GB300, in TFLOPS of unmasked work.

One step = one pass of the hot path over the workload: the fused forward (O
and LSE) with the block mask of the batch. The block mask depends only on the
mask and the shapes, so it is built once per mask and reused by every step
(FlexAttention page, the item on exploiting mask sparsity); its build time is
measured and reported beside the step, not inside it. The default workload
is the largest single-GPU one: bf16 GQA PrefixLM + soft-cap 50 (B=2, Hq=32,
Hkv=8, S=8192, D=128) with seeded synthetic inputs. FLOPs counted = 4 * D *
(kept (q, kv) pairs summed over batch and heads): neither the pairs the mask
removes nor the masked pairs inside partial tiles are counted.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 2|3|4|5]

Multi-GPU (torchrun): every rank runs its own replica of the workload (the
path has no exchange step), so scaling is weak; rank 0 prints one JSON line.
``--impl reference`` times the fp64 CPU oracle on the host's cores instead,
on a bounded sample of the same workload.
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

WORKLOAD = 4
METRIC = "attention fwd TFLOPS (unmasked FLOPs) and % of GB300 bf16 dense peak"
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}


def kept_pairs(w) -> int:
    """Kept (q, kv) pairs of one head, summed over the batch (mask evaluated
    row-slab by row-slab; the count defines the FLOPs of the metric)."""
    return sum(kept_pairs_per_batch(w))


def kept_pairs_per_batch(w) -> list:
    """Kept (q, kv) pairs of one head of each batch element."""
    import numpy as np
    out = []
    j = np.arange(w.Skv)[None, :]
    for b in range(w.B):
        total = 0
        for s in range(0, w.Sq, 1024):
            i = np.arange(s, min(s + 1024, w.Sq))[:, None]
            keep = np.ones((i.shape[0], w.Skv), bool)
            if w.causal:
                keep &= j <= i
            if w.window is not None:
                keep &= (i - j) < w.window
            if w.document:
                keep &= w.doc_id[b][i] == w.doc_id[b][j]
            if w.prefix:
                keep |= j < int(w.prefix_len[b])
            total += int(keep.sum())
        out.append(total)
    return out


def visited_pairs(w, tile: int = 128) -> int:
    """(q, kv) pairs inside the 128 x 128 tiles that hold at least one kept
    pair (the tiles the forward visits; their in-bounds area), one head,
    summed over the batch: the executed work beside the algorithmic one."""
    import numpy as np
    total = 0
    j = np.arange(w.Skv)[None, :]
    nkv = (w.Skv + tile - 1) // tile
    for b in range(w.B):
        for s in range(0, w.Sq, tile):
            i = np.arange(s, min(s + tile, w.Sq))[:, None]
            keep = np.ones((i.shape[0], w.Skv), bool)
            if w.causal:
                keep &= j <= i
            if w.window is not None:
                keep &= (i - j) < w.window
            if w.document:
                keep &= w.doc_id[b][i] == w.doc_id[b][j]
            if w.prefix:
                keep |= j < int(w.prefix_len[b])
            pad = np.zeros((keep.shape[0], nkv * tile), bool)
            pad[:, :w.Skv] = keep
            hit = pad.reshape(keep.shape[0], nkv, tile).any(axis=(0, 2))
            widths = np.minimum(tile, w.Skv - np.arange(nkv) * tile)
            total += int((widths * hit).sum()) * keep.shape[0]
    return total


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def source_digest() -> str:
    h = hashlib.sha256()
    for name in ("fwd_tc_kernel.cuh", "fwd_tc.cu", "common.cuh"):
        with open(os.path.join(ROOT, "masked_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# committed ncu summaries of the forward, by workload number
PROFILES = {3: "fwd_tc_doc_window_causal_b1h16s16384d128.md",
            4: "fwd_tc_gqa_prefix_softcap_b2h32s8192d128.md",
            5: "fwd_tc_causal_b8h16s4096d128.md"}


def profiled_traffic(kernel_digest: str, number: int):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if it was taken on the current kernel source."""
    if number not in PROFILES:
        return None
    path = os.path.join(ROOT, "profiles", PROFILES[number])
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    digest = traffic = None
    for line in text.splitlines():
        if line.startswith("source_digest:"):
            digest = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    return traffic if digest == kernel_digest else None


NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled during the timed
    region: NVML read through ctypes every 1 ms on a background thread (the
    timed region can be a few milliseconds), else nvidia-smi every 200 ms.
    Only reads; changes no setting."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.samples = []  # (sm_mhz, reasons bitmask)
        self.max_mhz = None
        self.source = None
        self.out = ""

    def _nvml_handle(self):
        import ctypes
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        handle = ctypes.c_void_p()
        uuid = getattr(torch.cuda.get_device_properties(self.idx), "uuid", None)
        ok = False
        if uuid is not None:
            ok = lib.nvmlDeviceGetHandleByUUID(("GPU-" + str(uuid)).encode(),
                                               ctypes.byref(handle)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.idx, ctypes.byref(handle)) != 0:
            return None
        return lib, handle

    def _poll(self, lib, handle):
        import ctypes
        clk, reasons = ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if (lib.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(clk)) == 0 and
                    get_reasons(handle, ctypes.byref(reasons)) == 0):
                self.samples.append((float(clk.value), int(reasons.value)))
            self._stop.wait(0.001)

    def __enter__(self):
        import threading
        self._stop = threading.Event()
        self._thread = None
        try:
            got = self._nvml_handle()
        except (OSError, AttributeError):
            got = None
        if got is not None:
            import ctypes
            lib, handle = got
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.source = "nvml"
            self._thread = threading.Thread(target=self._poll, args=got, daemon=True)
            self._thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if self.source == "nvml" and self.samples:
            sm = [c for c, _ in self.samples]
            bits = 0
            for _, r in self.samples:
                bits |= r
            reasons = sorted(n for k, n in NVML_REASONS.items() if bits & k)
            return {"sm_mhz": statistics.median(sm), "sm_max_mhz": self.max_mhz,
                    "reasons": reasons, "samples": len(sm), "source": "nvml, 1 ms"}
        rows = [r.split(",") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4)
                          if r[5 + k].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "source": "nvidia-smi, 200 ms"}


class OracleTimer:
    """Times the CPU oracle on whole (b, h) heads of the workload, one head per
    worker process of a pool started once (spawn, before any GPU work)."""

    def __init__(self, w, cores: int, number: int = WORKLOAD):
        import multiprocessing as mp
        self.w = w
        self.cores = cores
        per_b = kept_pairs_per_batch(w)
        self.heads = [(b, h) for b in range(w.B) for h in range(w.Hq)]
        self.head_flops = {bh: 4.0 * w.D * per_b[bh[0]] for bh in self.heads}
        self.pool = mp.get_context("spawn").Pool(processes=cores,
                                                 initializer=_oracle_worker_init,
                                                 initargs=(number,))
        self.pool.map(_oracle_head, self.heads[:cores])  # loads the inputs in every worker
        self.next = 0

    def step(self, seconds: float):
        """At least one round of `cores` heads and about `seconds` of work;
        returns (TFLOPS, heads timed)."""
        done = 0
        flops = 0.0
        t0 = time.perf_counter()
        while done == 0 or time.perf_counter() - t0 < seconds:
            batch = [self.heads[(self.next + k) % len(self.heads)] for k in range(self.cores)]
            self.next = (self.next + self.cores) % len(self.heads)
            self.pool.map(_oracle_head, batch)
            done += len(batch)
            flops += sum(self.head_flops[bh] for bh in batch)
        dt = time.perf_counter() - t0
        return flops / dt / 1e12, done

    def close(self):
        self.pool.close()
        self.pool.join()


def oracle_leg(w, seconds_target: float, cores: int, number: int = WORKLOAD):
    """One bounded timing of the oracle; returns (TFLOPS, sample description, cores)."""
    timer = OracleTimer(w, cores, number)
    try:
        tf, done = timer.step(seconds_target)
    finally:
        timer.close()
    return tf, f"{done} (b, h) heads of {len(timer.heads)}, whole rows, fp64", cores


_W = None


def _oracle_worker_init(number):
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    global _W
    from synth import make_workload
    _W = make_workload(number)


def _oracle_head(bh):
    from oracle import attention_forward
    from tests.helpers import oracle_spec
    attention_forward(_W.q, _W.k, _W.v, oracle_spec(_W), heads=[bh])
    return bh


REFERENCE_BUDGET_S = 150.0  # whole --impl reference run, warm-up included


def run_reference(args, rank: int, world: int) -> None:
    """The CPU oracle as it stands, on the host's cores: each step times a
    bounded sample of whole heads, sized so the whole run stays within a few
    minutes whatever --steps and --warmup are."""
    if rank != 0:
        return
    from synth import make_workload
    w = make_workload(WORKLOAD, with_tensors=False)
    cores = os.cpu_count() or 1
    per_step = min(8.0, max(0.5, REFERENCE_BUDGET_S / max(1, args.steps + args.warmup)))
    timer = OracleTimer(w, cores)
    try:
        for _ in range(args.warmup):
            timer.step(per_step)
        steps = [timer.step(per_step) for _ in range(args.steps)]
    finally:
        timer.close()
    value = statistics.median(tf for tf, _ in steps)
    sample = (f"about {per_step:.1f} s of whole (b, h) heads per step "
              f"({steps[0][1]} to {max(d for _, d in steps)} of {len(timer.heads)} heads), fp64")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(w),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def variant_of(w, M):
    """The library's variant bits for a workload (its mask and score terms)."""
    v = 0
    v |= M.MASK_CAUSAL if w.causal else 0
    v |= M.MASK_WINDOW if w.window is not None else 0
    v |= M.MASK_DOCUMENT if w.document else 0
    v |= M.MASK_PREFIX if w.prefix else 0
    v |= M.SCORE_ALIBI if w.alibi else 0
    v |= M.SCORE_SOFTCAP if w.softcap is not None else 0
    v |= M.SCORE_RELBIAS if w.relbias else 0
    return v


def config_dict(w):
    terms = [t for t, on in (("causal", w.causal), (f"window {w.window}", w.window is not None),
                             ("document", w.document), ("prefix", w.prefix),
                             ("ALiBi slope_h = 2^(-8(h+1)/H)", w.alibi),
                             (f"soft-cap {w.softcap}", w.softcap is not None),
                             ("relative-position bias table", w.relbias)) if on]
    return {"workload": f"{w.name} attention forward, B={w.B} Hq={w.Hq} Hkv={w.Hkv} "
                        f"S={w.Sq} D={w.D}",
            "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.Sq, "D": w.D,
            "variant": " + ".join(terms), "seed": w.seed,
            "l2": "flushed between timed steps (512 MiB write)",
            "step": "attn_fwd with the block mask of the batch (built once per mask, "
                    "timed separately)"}


def reduce_max(vals, world: int, device) -> tuple:
    """Element-wise maximum of ``vals`` over the ranks (each rank's timed
    seconds, so the slowest rank sets the job's time); ``vals`` itself when
    there is one rank. ``device``: where the collective runs (the GPU under
    NCCL, the CPU under gloo)."""
    if world == 1:
        return tuple(vals)
    import torch
    import torch.distributed as dist
    t = torch.tensor(vals, device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return tuple(float(x) for x in t)


def run_ours(args, rank: int, world: int) -> None:
    import torch
    import torch.distributed as dist

    import masked_attention_gb300 as M
    from synth import make_workload

    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    over = {"B": args.batch} if args.batch else {}
    if args.relbias:
        over["relbias"] = True
    w = make_workload(args.workload, **over)
    variant = variant_of(w, M)
    pairs = kept_pairs(w)
    flops = 4.0 * w.D * pairs * w.Hq  # per step, whole batch
    stream = torch.cuda.current_stream()

    q, k, v = (t.to(dev) for t in (w.q, w.k, w.v))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device=dev)
    bm_buf = torch.empty(M.attn_block_mask_bytes(w.B, w.Sq, w.Skv), dtype=torch.uint8,
                         device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    doc = torch.from_numpy(w.doc_id).to(dev) if w.document else None
    pre = torch.from_numpy(w.prefix_len).to(dev) if w.prefix else None
    mkw = dict(window=w.window or 0, doc_id=doc, prefix_len=pre)
    fkw = dict(mkw, softcap=w.softcap or 0.0)
    if w.relbias:
        fkw["rel_bias"] = w.rel_bias.to(dev)
    if args.paged:
        # the same K/V in a paged pool [B * pages, Hkv, page, D] under a shuffled page table
        ps = args.paged
        pps = (w.Skv + ps - 1) // ps
        pad = pps * ps - w.Skv
        gen = torch.Generator().manual_seed(w.seed)
        perm = torch.randperm(w.B * pps, generator=gen)

        def pool(t):
            t = torch.nn.functional.pad(t, (0, 0, 0, pad)) if pad else t
            pages = t.reshape(w.B, w.Hkv, pps, ps, w.D).permute(0, 2, 1, 3, 4)
            out = torch.empty(w.B * pps, w.Hkv, ps, w.D, dtype=t.dtype, device=dev)
            out[perm.to(dev)] = pages.reshape(w.B * pps, w.Hkv, ps, w.D)
            return out

        k, v = pool(k), pool(v)
        fkw.update(page_table=perm.reshape(w.B, pps).to(torch.int32).to(dev), page_size=ps,
                   Skv=w.Skv)

    # the block mask: built once per mask and reused by every step; its build
    # is timed on its own (median of several builds, L2 flushed before each)
    mask_ms = []
    for _ in range(8):
        flush.fill_(3)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        bm = M.build_block_mask(variant & 0xF, w.B, w.Sq, w.Skv, buf=bm_buf, stream=stream, **mkw)
        e1.record(stream)
        torch.cuda.synchronize()
        mask_ms.append(e0.elapsed_time(e1))
    mask_ms = sorted(mask_ms)[len(mask_ms) // 2]

    def step():
        M.attn_fwd(q, k, v, o, lse, variant, block_mask=bm, stream=stream, **fkw)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(*vals):
        return reduce_max(vals, world, dev)

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        step()
    if M.attn_check_status() != M.ATTN_OK:
        raise RuntimeError("device status error during warm-up")

    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2))
          for _ in range(args.steps)]
    barrier()
    with ClockSampler(local) as clocks:
        for s in range(args.steps):
            flush.fill_(s & 0xFF)  # L2 flush, outside the events
            ev[s][0].record(stream)
            step()
            ev[s][1].record(stream)
        barrier()
    if M.attn_check_status() != M.ATTN_OK:
        raise RuntimeError("device status error during the timed steps")
    fwd_each = sorted(a.elapsed_time(b) for a, b in ev)  # ms per forward launch
    fwd_s = sum(fwd_each) / 1e3
    (total_s,) = max_over_ranks(fwd_s)

    e2e = None
    if not args.no_e2e and not args.paged:
        # End to end through the public API: every step copies its Q, K, V in
        # from pinned host memory and its O and LSE back out. Timed two ways:
        # serially (copy in, forward, copy out on one stream, L2 flushed
        # between steps outside the events) and as a pipeline of steps, the
        # way a server runs them: step s's inputs are copied in on one stream
        # and step s-1's outputs out on another while step s-1's forward runs
        # (device buffers double-buffered), timed from the first copy in to
        # the last copy out. Each step's inputs (201 MB) exceed the L2 and
        # are written through it by the copy. `value` is the pipelined one.
        hq, hk, hv = (t.pin_memory() for t in (w.q, w.k, w.v))
        ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
        d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            step()  # the block mask stays the one built above
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)

        for _ in range(3):
            flush.fill_(2)
            e2e_step()
        eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        barrier()
        for s in range(args.steps):
            flush.fill_(s & 0xFF)
            eev[s][0].record(stream)
            e2e_step()
            eev[s][1].record(stream)
        barrier()
        (e2e_serial_s,) = max_over_ranks(sum(a.elapsed_time(b) for a, b in eev) / 1e3)

        # pipelined: two sets of device buffers, a copy-in and a copy-out stream
        bufs = [(q, k, v, o, lse), tuple(torch.empty_like(t) for t in (q, k, v, o, lse))]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def pipeline(nsteps):
            e_in = [torch.cuda.Event() for _ in range(nsteps)]
            e_fwd = [torch.cuda.Event() for _ in range(nsteps)]
            e_out = [torch.cuda.Event() for _ in range(nsteps)]
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(s_in)
            for s in range(nsteps):
                bq, bk, bv, bo, bl = bufs[s & 1]
                with torch.cuda.stream(s_in):
                    if s >= 2:
                        s_in.wait_event(e_fwd[s - 2])  # the forward of s-2 has read this set
                    bq.copy_(hq, non_blocking=True)
                    bk.copy_(hk, non_blocking=True)
                    bv.copy_(hv, non_blocking=True)
                    e_in[s].record(s_in)
                stream.wait_event(e_in[s])
                if s >= 2:
                    stream.wait_event(e_out[s - 2])  # O and LSE of s-2 are out
                M.attn_fwd(bq, bk, bv, bo, bl, variant, block_mask=bm, stream=stream, **fkw)
                e_fwd[s].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(e_fwd[s])
                    ho.copy_(bo, non_blocking=True)
                    hl.copy_(bl, non_blocking=True)
                    e_out[s].record(s_out)
            t1.record(s_out)
            return t0, t1

        pipeline(3)
        barrier()
        t0, t1 = pipeline(args.steps)
        barrier()
        (e2e_s,) = max_over_ranks(t0.elapsed_time(t1) / 1e3)
        if M.attn_check_status() != M.ATTN_OK:
            raise RuntimeError("device status error during the end-to-end steps")
        e2e = {"value": world * flops * args.steps / e2e_s / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "mode": "pipelined: step s+1's copy in and step s-1's copy out overlap "
                       "step s's forward; timed from the first copy in to the last copy out",
               "serial_value": world * flops * args.steps / e2e_serial_s / 1e12}

    if rank != 0:
        return
    peaks, peak_kind = read_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    value = world * flops * args.steps / total_s / 1e12
    fwd_tflops = flops * args.steps / fwd_s / 1e12
    digest = source_digest()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_s / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_dict(w),
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "achieved": fwd_tflops, "peak": peak,
                     "unit": "TFLOP/s", "frac": fwd_tflops / peak,
                     "traffic": (profiled_traffic(digest, args.workload)
                                 if not args.batch and not args.relbias and not args.paged
                                 else None),
                     "kernel": f"fwd_tc_kernel<D={w.D}>",
                     "peak_source": ("measured bf16 dense burst (MEASURED_PEAKS.json)"
                                     if peak_kind == "measured" else "fallback 1.9 PFLOP/s")},
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
        "flops_per_step": flops,
        # context: 4 D per pair of every visited tile, and of the dense S x S square
        "flops_executed_per_step": 4.0 * w.D * visited_pairs(w) * w.Hq,
        "flops_dense_per_step": 4.0 * w.D * w.B * w.Sq * w.Skv * w.Hq,
        "fwd_ms_per_launch": fwd_s / args.steps * 1e3,
        "fwd_ms_median": fwd_each[len(fwd_each) // 2],
        "fwd_ms_min": fwd_each[0],
        "mask_build_ms": mask_ms,
        "source_digest": digest,
    }
    if not args.no_cpu_baseline:
        tf, sample, cores = oracle_leg(w, args.cpu_seconds, os.cpu_count() or 1, args.workload)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOPS", "cores": cores,
                                "kind": "oracle", "sample": sample}
    print(json.dumps(line), flush=True)


def run_backward(args) -> None:
    """Diagnostic: the backward of the bf16 causal training workload (B=8,
    Hq=Hkv=16, S=4096, D=128) after one forward, timed with CUDA events per
    launch, in TFLOPS of 2.5 x the forward's unmasked FLOPs; one line per
    path: bf16 operands with their rounding remainders (the minimal
    workspace), and fp16 operands (a workspace with room for the fp16 copies
    of Q, K, V, dO; their conversion is inside the timed call)."""
    import torch

    import masked_attention_gb300 as M
    from synth import make_workload

    w = make_workload(5, **({"B": args.batch} if args.batch else {}))
    dev = torch.device("cuda", 0)
    variant = variant_of(w, M)
    flops = 2.5 * 4.0 * w.D * kept_pairs(w) * w.Hq
    q, k, v, do = (t.to(dev) for t in (w.q, w.k, w.v, w.do))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bm = M.build_block_mask(variant & 0xF, w.B, w.Sq, w.Skv, transposed=True)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    M.attn_fwd(q, k, v, o, lse, variant, block_mask=bm)
    for path, nbytes in (("bf16", M.attn_bwd_workspace_bytes(w.B, w.Hq, w.Sq)),
                         ("f16", M.attn_bwd_workspace_bytes_f16(w.B, w.Hq, w.Hkv, w.Sq, w.Skv,
                                                                w.D))):
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        for _ in range(max(args.warmup, 3)):
            M.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, variant, block_mask=bm)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        torch.cuda.synchronize()
        for s_ in range(args.steps):
            flush.fill_(s_ & 0xFF)
            ev[s_][0].record()
            M.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, variant, block_mask=bm)
            ev[s_][1].record()
        torch.cuda.synchronize()
        if M.attn_check_status() != M.ATTN_OK:
            raise RuntimeError("device status error during the backward")
        ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
        print(json.dumps({"diagnostic": "backward", "path": path,
                          "workload": config_dict(w)["workload"],
                          "workspace_bytes": nbytes, "ms_per_launch": ms,
                          "flops_per_launch": flops, "tflops": flops / ms / 1e9,
                          "source_digest": source_digest()}), flush=True)
        del ws


def run_combine(args) -> None:
    """Diagnostic: attn_combine merging the partial results of n key/value
    shards for the document + window workload's queries (B=1, H=16, S=16384,
    D=128, bf16), one launch timed with CUDA events, against the measured
    HBM copy bandwidth. Algorithmic bytes per launch: every part's O row and
    LSE read once, the merged row and LSE written once."""
    import torch

    import masked_attention_gb300 as M

    n, B, H, S, D = args.combine, 1, 16, 16384, 128
    rows = B * H * S
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(11)
    o_parts = torch.randn(n, rows, D, generator=g, device=dev).to(torch.bfloat16)
    l_parts = torch.randn(n, rows, generator=g, device=dev) * 4.0
    o = torch.empty(rows, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(rows, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 3)):
        M.attn_combine(o_parts, l_parts, o, lse)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    torch.cuda.synchronize()
    for s_ in range(args.steps):
        flush.fill_(s_ & 0xFF)
        ev[s_][0].record()
        M.attn_combine(o_parts, l_parts, o, lse)
        ev[s_][1].record()
    torch.cuda.synchronize()
    ms = sorted(a.elapsed_time(b) for a, b in ev)[args.steps // 2]
    nbytes = (n + 1) * rows * (2 * D + 4)
    peaks, src = read_peaks()
    gbs = nbytes / ms / 1e6
    print(json.dumps({"diagnostic": "combine", "parts": n, "rows": rows, "D": D,
                      "ms_per_launch": ms, "bytes_per_launch": nbytes, "gbs": gbs,
                      "frac_of_hbm": gbs / peaks["hbm_gbs"], "peak_source": src}), flush=True)


# Decode workload: the grouped-query model shape of the prefix-LM workload
# (Hq=32, Hkv=8, D=128, bf16), one new token per sequence at the end of a
# 32768-token cache, 16 sequences: K and V total 2.1 GB, far above L2.
DECODE_SHAPE = dict(B=16, Hq=32, Hkv=8, Sq=1, Skv=32768, D=128)
# (label, page size or 0 for contiguous, sliding window or 0)
DECODE_CASES = [("contiguous causal", 0, 0), ("paged 16 causal", 16, 0),
                ("paged 64 causal", 64, 0), ("paged 64 causal + window 4096", 64, 4096)]


def run_decode(args) -> None:
    """Diagnostic: attn_decode (PagedAttention, alone and with a sliding
    window) on the decode workload, contiguous and paged caches, one launch
    sequence (decode kernel, then the merge of the key splits) timed with
    CUDA events, L2 flushed between launches, against the measured HBM copy
    bandwidth. Algorithmic bytes per launch: the K and V rows of the kept
    keys read once per key/value head, Q read, O and LSE written, the page
    table entries of the kept pages read."""
    import torch

    import masked_attention_gb300 as M

    sh = dict(DECODE_SHAPE)
    if args.batch:
        sh["B"] = args.batch
    B, Hq, Hkv, Sq, Skv, D = (sh[x] for x in ("B", "Hq", "Hkv", "Sq", "Skv", "D"))
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(21)
    q = torch.randn(B, Hq, Sq, D, generator=g, device=dev).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(B, Hq, Sq, device=dev)
    ws = torch.empty(max(M.attn_decode_workspace_bytes(B, Hq, Hkv, Sq, Skv, D), 256),
                     dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peaks, src = read_peaks()
    variant_base = M.MASK_CAUSAL
    for label, ps, window in DECODE_CASES:
        if ps:
            pps = Skv // ps
            num_pages = B * pps
            kc = torch.randn(num_pages, Hkv, ps, D, generator=g, device=dev).to(torch.bfloat16)
            vc = torch.randn(num_pages, Hkv, ps, D, generator=g, device=dev).to(torch.bfloat16)
            perm = torch.randperm(num_pages, generator=g, device=dev).to(torch.int32)
            kw = dict(page_table=perm.view(B, pps), page_size=ps, Skv=Skv)
        else:
            kc = torch.randn(B, Hkv, Skv, D, generator=g, device=dev).to(torch.bfloat16)
            vc = torch.randn(B, Hkv, Skv, D, generator=g, device=dev).to(torch.bfloat16)
            kw = {}
        variant = variant_base | (M.MASK_WINDOW if window else 0)
        call = lambda: M.attn_decode(q, kc, vc, o, lse, variant, workspace=ws, window=window,
                                     q_offset=Skv - Sq, **kw)
        for _ in range(max(args.warmup, 3)):
            call()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        torch.cuda.synchronize()
        for s_ in range(args.steps):
            flush.fill_(s_ & 0xFF)
            ev[s_][0].record()
            call()
            ev[s_][1].record()
        torch.cuda.synchronize()
        if M.attn_check_status() != M.ATTN_OK:
            raise RuntimeError("device status error during decode")
        times = sorted(a.elapsed_time(b) for a, b in ev)
        ms = times[args.steps // 2]
        kept = min(window, Skv) if window else Skv
        nbytes = (2 * B * Hkv * kept * D * 2 + 2 * B * Hq * Sq * D * 2 + 4 * B * Hq * Sq
                  + (4 * B * ((kept + ps - 1) // ps + 1) if ps else 0))
        gbs = nbytes / ms / 1e6
        print(json.dumps({"diagnostic": "decode", "case": label, "B": B, "Hq": Hq, "Hkv": Hkv,
                          "Sq": Sq, "Skv": Skv, "D": D, "page_size": ps, "window": window,
                          "splits_workspace_bytes": ws.numel(), "ms_per_launch": ms,
                          "ms_min": times[0], "bytes_per_launch": nbytes, "gbs": gbs,
                          "frac_of_hbm": gbs / peaks["hbm_gbs"], "peak_source": src}),
              flush=True)
        del kc, vc


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch", type=int, default=0, help="override B (profiling cases only)")
    ap.add_argument("--workload", type=int, default=WORKLOAD, choices=[2, 3, 4, 5],
                    help="diagnostic runs on the other bf16 workloads (forward only)")
    ap.add_argument("--paged", type=int, default=0, choices=[0, 16, 32, 64, 128],
                    help="diagnostic: read K/V from a paged cache with this page size")
    ap.add_argument("--relbias", action="store_true",
                    help="diagnostic: add a relative-position bias table to the workload")
    ap.add_argument("--backward", action="store_true",
                    help="diagnostic: time the backward of the training workload instead")
    ap.add_argument("--combine", type=int, default=0,
                    help="diagnostic: time attn_combine over this many key/value shards")
    ap.add_argument("--decode", action="store_true",
                    help="diagnostic: time attn_decode on the decode workload")
    args = ap.parse_args()
    if args.decode:
        run_decode(args)
        return
    if args.combine:
        run_combine(args)
        return
    if args.backward:
        run_backward(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
