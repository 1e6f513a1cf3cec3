"""Benchmark of the product-VQ KV-cache hot path on GB300.

Default workload (N=1): batched GQA decode -- B=32 sequences, H_q=32 query
heads over H_kv=8 KV heads, D=128, one query token each attending over
S_kv=32768 coded keys (uint8 K and V codes, 256x4 codebooks).  One step =
vq_decode_attend (the split-KV kernel + its combine pass).

Other workloads (--workload): decode-1seq (encode 8192 new keys + attend),
gqa-decode-ragged, gqa-decode-packed, decode-append, bulk-encode, bulk-encode-packed,
chunked-prefill.

Prints ONE JSON line (rank 0).  `value` is device-timed throughput with
inputs resident in HBM; `e2e` repeats the step through the same C-ABI calls
from pinned host buffers with the host<->device copies inside the timed
region.  L2 is flushed (a 256 MiB write) before every timed step.

--impl reference times the float64 CPU oracle on a bounded sample of the
same workload (the CPU baseline) on all host cores; under torchrun only
rank 0 runs it.  The GPU line's cpu_baseline reports the same oracle on one
thread and on all host cores, and `parity` compares the oracle's results on
that sample with the GPU step's (code mismatches / near ties, or the
attention rows' max error).
"""
from __future__ import annotations

import argparse
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
sys.path.insert(0, ROOT)

from product_vq_compressed_gb300.workloads import WORKLOADS, make_inputs  # noqa: E402

L2_FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------- metrics

METRICS = {
    "decode-1seq": ("decode tokens/s (encode 8192 keys + attend, B=1 H=8 D=128)",
                    "tokens/s"),
    "gqa-decode": ("decode tokens/s (B=32 Hq=32 Hkv=8 S_kv=32768)", "tokens/s"),
    "bulk-encode": ("key-encode vectors/s ([4,32,8192,128] K+V encode)", "vectors/s"),
    "bulk-encode-packed": ("key-encode vectors/s ([4,32,8192,128] K+V encode, 10-bit packed "
                           "key codes, 20 B/token-head)", "vectors/s"),
    "chunked-prefill": ("prefill tokens/s (S_q=2048, window 4096)", "tokens/s"),
    "decode-append": ("decode tokens/s (one launch: append 1 token's K/V codes into a 8256-row "
                      "cache + attend over 8192, B=1 H=8 D=128)", "tokens/s"),
    "gqa-decode-ragged": ("decode tokens/s (B=32 Hq=32 Hkv=8, cache lengths U[16384, 32768])",
                          "tokens/s"),
    "gqa-decode-packed": ("decode tokens/s (B=32 Hq=32 Hkv=8 S_kv=32768, 10-bit packed key "
                          "codes of a 1024x8 codebook, 20 B + 32 B per token-head)", "tokens/s"),
}


def units_per_step(name, spec):
    if name.startswith("bulk-encode"):
        return spec.B * spec.H_kv * spec.enc_len       # key vectors
    return spec.B * spec.S_q                           # query tokens


def _bits(n_centroids):
    """Bits per bit-packed code: 2^bits >= n_centroids."""
    b = 1
    while (1 << b) < n_centroids:
        b += 1
    return b


def pack_rows(codes, bits, torch):
    """Codes [..., n] (a device tensor) as int32 rows of bit-packed codes:
    code m at bits [m bits, (m + 1) bits) of the row's little-endian 32-bit
    words (the cache layout of code_bytes 0)."""
    n = codes.shape[-1]
    words = (n * bits + 31) // 32
    c = codes.to(torch.int64)
    out = torch.zeros(codes.shape[:-1] + (words + 1,), dtype=torch.int64, device=codes.device)
    for m in range(n):
        w, sh = divmod(m * bits, 32)
        v = c[..., m] << sh
        out[..., w] |= v & 0xFFFFFFFF
        out[..., w + 1] |= v >> 32
    out = out[..., :words]
    return (out - ((out >> 31) << 32)).to(torch.int32).contiguous()


def unpack_rows(rows, n, bits):
    """Inverse of pack_rows on the host: int32 rows [..., words] -> codes
    [..., n] (int64)."""
    w = rows.reshape(-1, rows.shape[-1]).view(np.uint32).astype(np.uint64)
    w = np.concatenate([w, np.zeros((w.shape[0], 1), np.uint64)], axis=1)
    out = np.zeros((w.shape[0], n), np.int64)
    for m in range(n):
        i, sh = divmod(m * bits, 32)
        v = (w[:, i] | (w[:, i + 1] << np.uint64(32))) >> np.uint64(sh)
        out[:, m] = (v & np.uint64((1 << bits) - 1)).astype(np.int64)
    return out.reshape(rows.shape[:-1] + (n,))


def algorithmic(name, spec, lens=None):
    """(dominant kernel, bound, work per launch, unit) -- the per-unit
    figures are stated with the design notes."""
    if name in ("decode-1seq", "bulk-encode", "bulk-encode-packed"):
        n_sub = spec.B * spec.H_kv * spec.enc_len * spec.n_k
        flops = 2.0 * spec.k_d * spec.k_N * n_sub     # one multiply-add per dim and candidate
        return "encode", "alu", flops, "TFLOP/s"
    if name in ("gqa-decode", "decode-append", "gqa-decode-ragged", "gqa-decode-packed"):
        k_row = 4 * ((spec.n_k * _bits(spec.k_N) + 31) // 32) if spec.packed_keys else \
            spec.n_k * np.dtype(spec.k_code_dtype).itemsize
        per_tok = k_row + spec.n_v * np.dtype(spec.v_code_dtype).itemsize
        keys = spec.B * spec.S_kv if lens is None else int(np.sum(lens))
        byts = spec.H_kv * keys * per_tok + 2 * spec.B * spec.H_q * spec.S_q * spec.D * 2
        return "decode", "hbm", float(byts), "GB/s"
    # chunked prefill: QK^T and PV over each query's visible keys
    vis = min(spec.window, spec.S_kv) if spec.window else spec.S_kv
    flops = 4.0 * spec.D * spec.S_q * vis * spec.H_q * spec.B
    return "prefill", "tensor", flops, "TFLOP/s"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
            "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}, "fallback"


def peak_for(bound, peaks):
    if bound == "hbm":
        return peaks["hbm_gbs"], "GB/s"
    if bound == "tensor":
        # fp16 inputs with fp32 accumulation run at the bf16 dense rate
        return peaks["bf16_tflops"], "TFLOP/s"
    # fp32 FMA: 152 SMs x 128 lanes x 2 FLOP x max SM clock
    return 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12, "TFLOP/s"


def measured_traffic(name):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None when the kernel source changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        entry = json.load(open(path))[name]
        src = open(os.path.join(ROOT, entry["source"]), "rb").read()
    except (OSError, KeyError, ValueError):
        return None
    if hashlib.sha256(src).hexdigest() != entry["sha256"]:
        return None
    return entry["bytes_per_launch"]


# ------------------------------------------------------------- ranks

def max_over_ranks(seconds: float, world: int, device: str) -> float:
    """Slowest rank's timed seconds (all ranks join; identity at world 1)."""
    if world <= 1:
        return seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Weak scaling: every rank runs its own replica of the workload, so the
    job processes units_per_rank * world units in the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None
        self.first = 0   # samples before this line index are not counted

    def _lines(self):
        try:
            with open(self.path) as f:
                return sum(1 for _ in f)
        except OSError:
            return 0

    def mark(self):
        """Count only the samples taken from now on."""
        self.first = self._lines()

    def wait_for_sample(self, timeout_s=0.5):
        """A timed region shorter than the 100 ms sampling period may end
        before any sample: then take the first sample that follows it."""
        t0 = time.perf_counter()
        while self.proc is not None and self._lines() <= self.first and \
                time.perf_counter() - t0 < timeout_s:
            time.sleep(0.01)

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index),
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in list(open(self.path))[self.first:]:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for _, _, r in rows for k in range(4)
                          if r[k].lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------- GPU arm

class Runner:
    """Holds device inputs of one workload and runs one step."""

    def __init__(self, name, spec, inp, torch, vq, stream):
        self.name, self.spec, self.torch, self.vq = name, spec, torch, vq
        self.stream = stream
        t = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        self.d = {k: t(v) for k, v in inp.items() if isinstance(v, np.ndarray)}
        s = spec
        dev = self.d
        self.launches = 0
        if name == "decode-1seq":
            # values pre-encoded once, outside the timed region
            dev["v_codes"], _ = vq.encode_values(dev["values"], dev["v_codebook"], s.v_d,
                                                 stream=stream)
            dev["k_codes"] = torch.empty((s.B, s.H_kv, s.enc_len, s.n_k),
                                         dtype=vq.code_dtype(s.k_N), device="cuda")
        if name.startswith("bulk-encode"):
            kw = vq.packed_row_words(s.n_k, s.k_N) if s.packed_keys else s.n_k
            dev["k_codes"] = torch.empty((s.B, s.H_kv, s.enc_len, kw),
                                         dtype=torch.int32 if s.packed_keys else
                                         vq.code_dtype(s.k_N), device="cuda")
            dev["v_codes"] = torch.empty((s.B, s.H_kv, s.enc_len, s.n_v),
                                         dtype=vq.code_dtype(s.v_N), device="cuda")
            dev["k_hat"] = torch.empty_like(dev["keys"])
        if s.packed_keys and not name.startswith("bulk-encode"):
            # the drawn key codes as the cache stores them: 10-bit packed rows
            dev["k_codes"] = pack_rows(dev["k_codes"], _bits(s.k_N), torch)
        if name == "decode-append":
            # the cache: buffers of `capacity` rows holding S_kv - 1 cached
            # tokens; each step writes the new token into row S_kv - 1
            for k in ("k_codes", "v_codes"):
                buf = torch.zeros((s.B, s.H_kv, s.capacity, dev[k].shape[-1]),
                                  dtype=dev[k].dtype, device="cuda")
                buf[:, :, :s.S_kv] = dev[k]
                dev[k] = buf
        dev["out"] = torch.empty_like(dev["q"])
        if not name.startswith("bulk-encode"):
            args = vq.make_attend_args(dev["q"], dev["k_codes"], dev["k_codebook"],
                                       dev["v_codes"], dev["v_codebook"],
                                       dev.get("smooth"), s.sm_scale, s.causal,
                                       s.window, dev["out"], s_kv=s.S_kv,
                                       kv_lens=dev.get("kv_lens"))
            need = vq.attend_workspace_bytes(args)
            dev["ws"] = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")

    def step(self, ev=None):
        """One pass of the hot path; ev = (start, mid) events around the
        dominant kernel (recorded on the launch stream)."""
        s, d, vq, st = self.spec, self.d, self.vq, self.stream
        if self.name == "decode-1seq":
            if ev: ev[0].record(st)
            vq.encode_keys(d["keys"], d["k_codebook"], s.k_d, d["smooth"],
                           codes=d["k_codes"], stream=st)
            if ev: ev[1].record(st)
            vq.decode_attend(d["q"], d["k_codes"], d["k_codebook"], d["v_codes"],
                             d["v_codebook"], d["smooth"], s.sm_scale, s.causal,
                             s.window, out=d["out"], workspace=d["ws"], stream=st)
            return 3
        if self.name == "decode-append":
            # one launch: the new token's K and V into row S_kv - 1, attention
            # over the S_kv cached tokens, merge of the key splits
            if ev: ev[0].record(st)
            vq.decode_step(d["q"], d["keys"], d["values"], d["k_codes"], d["k_codebook"],
                           d["v_codes"], d["v_codebook"], d["smooth"], s.sm_scale, s.causal,
                           s.window, out=d["out"], workspace=d["ws"], stream=st, s_kv=s.S_kv)
            if ev: ev[1].record(st)
            return 1
        if self.name.startswith("bulk-encode"):
            if ev: ev[0].record(st)
            vq.encode_keys(d["keys"], d["k_codebook"], s.k_d, d["smooth"],
                           codes=d["k_codes"], k_hat=d["k_hat"], stream=st)
            if ev: ev[1].record(st)
            vq.encode_values(d["values"], d["v_codebook"], s.v_d, codes=d["v_codes"],
                             stream=st)
            return 2
        fn = vq.prefill_attend if self.name == "chunked-prefill" else vq.decode_attend
        if ev: ev[0].record(st)
        fn(d["q"], d["k_codes"], d["k_codebook"], d["v_codes"], d["v_codebook"],
           d["smooth"], s.sm_scale, s.causal, s.window, out=d["out"],
           workspace=d["ws"], stream=st, kv_lens=d.get("kv_lens"))
        if ev: ev[1].record(st)
        return 2


def run_gpu(args, name, rank, world):
    import torch
    import torch.distributed as dist

    from product_vq_compressed_gb300 import binding as vq

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    # the clock sampler runs from here so that it is sampling when the timed
    # region starts; only samples from that point on are reported
    clk = ClockSampler(local).__enter__()
    spec = WORKLOADS[name]
    inp = make_inputs(spec)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        r = Runner(name, spec, inp, torch, vq, stream)
    torch.cuda.synchronize()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    for _ in range(args.warmup):
        r.step()
    torch.cuda.synchronize()
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    launches = 0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clk.mark()
    wall0 = time.perf_counter()
    for k in range(K):
        # evict L2 between timed steps: the flush starts after the
        # previous step and the next step after the flush
        torch.cuda.current_stream().wait_stream(stream)
        flush.fill_(float(k))
        stream.wait_stream(torch.cuda.current_stream())
        e_start, e_mid, e_end = evs[k]
        launches += r.step(ev=(e_start, e_mid))
        e_end.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clk.wait_for_sample()
    clk.__exit__(None, None, None)
    if world > 1:
        dist.barrier()
    out_t = r.d["k_codes"] if name.startswith("bulk-encode") else r.d["out"]
    finite = bool(torch.isfinite(out_t.float()).all()) if out_t.is_floating_point() else True
    if not finite:
        print("warning: non-finite values in the step's output", file=sys.stderr)
    step_ms = [evs[k][0].elapsed_time(evs[k][2]) for k in range(K)]
    dom_ms = [evs[k][0].elapsed_time(evs[k][1]) for k in range(K)]
    total_s = max_over_ranks(sum(step_ms) / 1e3, world, "cuda")
    value = whole_job_value(units_per_step(name, spec) * K, world, total_s)

    # ---- the same step with nothing flushed between repetitions (small
    #      workloads then run from L2): reported beside the flushed numbers
    with torch.cuda.stream(stream):
        for _ in range(2):
            r.step()
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        Kr = max(3, min(K, 20))
        r0.record(stream)
        for _ in range(Kr):
            r.step()
        r1.record(stream)
    torch.cuda.synchronize()
    resident_ms = r0.elapsed_time(r1) / Kr

    # ---- end to end from pinned host buffers (same C-ABI calls)
    e2e = None
    if name in METRICS:
        in_keys = {"decode-1seq": ["keys", "q"], "bulk-encode": ["keys", "values"],
                   "bulk-encode-packed": ["keys", "values"],
                   "decode-append": ["keys", "values", "q"]}.get(name, ["q"])
        host = {k: torch.from_numpy(np.ascontiguousarray(inp[k])).pin_memory()
                for k in in_keys}
        out_name = "k_codes" if name.startswith("bulk-encode") else "out"
        host_out = torch.empty(r.d[out_name].shape, dtype=r.d[out_name].dtype).pin_memory()
        h2d = sum(h.numel() * h.element_size() for h in host.values())
        d2h = host_out.numel() * host_out.element_size()
        with torch.cuda.stream(stream):
            for _ in range(2):
                for k in in_keys:
                    r.d[k].copy_(host[k], non_blocking=True)
                r.step()
                host_out.copy_(r.d[out_name], non_blocking=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        Ke = max(3, min(K, 20))
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(Ke):
                for k in in_keys:
                    r.d[k].copy_(host[k], non_blocking=True)
                r.step()
                host_out.copy_(r.d[out_name], non_blocking=True)
            e1.record(stream)
        torch.cuda.synchronize()
        e2e_s = e0.elapsed_time(e1) / 1e3
        e2e = {"value": units_per_step(name, spec) * Ke / e2e_s,
               "unit": METRICS[name][1], "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h)}

    kernel, bound, work, wunit = algorithmic(name, spec, inp.get("kv_lens"))
    peaks, peak_src = load_peaks()
    peak, punit = peak_for(bound, peaks)
    dom_s = statistics.mean(dom_ms) / 1e3
    achieved = (work / dom_s) / (1e9 if wunit == "GB/s" else 1e12)
    roof = {"bound": bound, "kernel": kernel, "achieved": round(achieved, 3),
            "peak": round(peak, 1), "unit": punit, "frac": round(achieved / peak, 4),
            "peak_source": peak_src, "traffic": measured_traffic(name),
            "kernel_ms": round(dom_s * 1e3, 4)}
    clocks = clk.summary()
    metric, unit = METRICS[name]
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": total_s * 1e3 / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": name, "B": spec.B, "H_q": spec.H_q, "H_kv": spec.H_kv,
                   "D": spec.D, "S_kv": spec.S_kv, "S_q": spec.S_q,
                   "k_codebook": [spec.k_N, spec.k_d], "v_codebook": [spec.v_N, spec.v_d],
                   "sliding_window": spec.window, "l2": "flushed before every timed step",
                   "parallelism": f"replicas x{world}"},
        "e2e": e2e, "gpu_launches": launches, "roofline": roof, "clocks": clocks,
        "wall_s_timed_region": round(wall, 4), "output_finite": finite,
        "l2_resident": {"ms_per_step": round(resident_ms, 5),
                        "value": units_per_step(name, spec) / (resident_ms / 1e3),
                        "note": "the same step back to back, L2 not flushed"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gpu_out = {}
        if name in ("decode-1seq", "bulk-encode"):
            gpu_out["k_codes"] = r.d["k_codes"].cpu().numpy()
        elif name == "bulk-encode-packed":
            gpu_out["k_codes"] = unpack_rows(r.d["k_codes"].cpu().numpy(), spec.n_k,
                                             _bits(spec.k_N))
        elif not name.startswith("bulk-encode"):
            gpu_out["out"] = r.d["out"].float().cpu().numpy()
        cb = cpu_baseline(name, spec, inp, budget_s=args.cpu_budget, gpu=gpu_out)
        line["parity"] = cb.pop("parity", None)
        line["cpu_baseline"] = cb
    return line


# ------------------------------------------------------------- CPU arm (oracle)

def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _concurrent_wall(fn, args_list):
    """Wall seconds to run fn over args_list on one thread each (the oracle
    is C behind ctypes, which releases the GIL: the threads run in parallel)."""
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=len(args_list)) as ex:
        t0 = time.perf_counter()
        list(ex.map(fn, args_list))
        return time.perf_counter() - t0


def cpu_baseline(name, spec, inp, budget_s=10.0, gpu=None):
    """Time the float64 oracle, as it stands, on a bounded sample of the
    workload and scale it to the metric's unit: once on one thread and once
    on every host core (threads over disjoint parts of the sample).  With
    ``gpu`` (the GPU step's outputs as numpy arrays) the oracle's results on
    the sample are also compared with the GPU's (the parity counts)."""
    import oracle
    from oracle import parity as par
    oracle.build()
    D = spec.D
    cores = host_cores()
    n_bg = spec.B * spec.H_kv
    n_rows = spec.B * spec.H_q * spec.S_q
    report = {}

    def encode_sample(seed, n_vec):
        keys = inp["keys"].reshape(-1, D)
        heads = np.broadcast_to(np.arange(spec.H_kv)[None, :, None],
                                inp["keys"].shape[:3]).reshape(-1)
        idx = np.random.default_rng(seed).integers(0, keys.shape[0], n_vec)
        t0 = time.perf_counter()
        out = oracle.encode(keys[idx], inp["k_codebook"], heads=heads[idx], smooth=inp["smooth"])
        return time.perf_counter() - t0, idx, out

    def attend_sample(pair, n_rows_s):
        """Oracle attention of n_rows_s rows of one (batch, kv head): the
        K_hat reconstruction of that head plus the rows."""
        b, g = divmod(pair % n_bg, spec.H_kv)
        if "k_codes" in inp:
            kc, vc = inp["k_codes"][b:b + 1, g:g + 1], inp["v_codes"][b:b + 1, g:g + 1]
        else:
            r = np.random.default_rng(pair)
            kc = r.integers(0, spec.k_N, (1, 1, spec.S_kv, spec.n_k))
            vc = r.integers(0, spec.v_N, (1, 1, spec.S_kv, spec.n_v))
        if "kv_lens" in inp:
            L = int(inp["kv_lens"][b])
            kc, vc = kc[:, :, :L], vc[:, :, :L]
        rows = np.array([[0, r % spec.G, spec.S_q - 1 - (r // spec.G) % spec.S_q]
                         for r in range(n_rows_s)])
        q = inp["q"][b:b + 1, g * spec.G:(g + 1) * spec.G]
        sm = None if inp["smooth"] is None else inp["smooth"][g:g + 1]
        t0 = time.perf_counter()
        out = oracle.attend_rows(q, kc, inp["k_codebook"], vc, inp["v_codebook"], sm,
                                 spec.sm_scale, spec.causal, spec.window, rows)
        return time.perf_counter() - t0, (b, g, rows), out

    def attend_model(pair):
        """(per-head cost, per-row cost, seconds spent, rows, their outputs):
        one row and 1 + kExtra rows of the same head, the difference over
        kExtra rows giving the per-row cost (enough rows that it stands
        above the run-to-run noise of the per-head part)."""
        kExtra = 16
        t1 = attend_sample(pair, 1)[0]
        tn, where, out = attend_sample(pair, 1 + kExtra)
        per_row = max((tn - t1) / kExtra, 0.0)
        return max(t1 - per_row, 0.0), per_row, t1 + tn, where, out

    def attend_parity(where, out):
        if gpu is None or "out" not in gpu:
            return
        b, g, rows = where
        got = np.stack([gpu["out"][b, g * spec.G + h, i] for _, h, i in rows]).astype(np.float64)
        ok, err, _ = par.allclose_report(got, oracle.to_f16(out).astype(np.float64))
        report["parity"] = {"attention_rows": int(len(rows)), "max_abs_err": err,
                            "tolerance": "2e-3 + 1e-2 |ref|", "ok": ok}

    if name in ("decode-1seq", "bulk-encode", "bulk-encode-packed"):
        n_total = spec.B * spec.H_kv * spec.enc_len
        per = encode_sample(0, 64)[0] / 64
        n_s = int(max(64, min(n_total, 0.5 * budget_s / max(per, 1e-9))))
        t1, idx, out = encode_sample(1, n_s)
        wall = _concurrent_wall(lambda k: encode_sample(2 + k, n_s), list(range(cores)))
        full1 = t1 * n_total / n_s
        fullN = wall * n_total / (n_s * cores)
        sample = f"oracle key encode of {n_s} of {n_total} vectors (per thread), scaled"
        if gpu is not None and "k_codes" in gpu:
            res = par.check_codes(gpu["k_codes"].reshape(n_total, -1)[idx].astype(np.int64), out)
            report["parity"] = {"codes": res}
        if name == "decode-1seq":
            ph, pr, tt, _, _ = attend_model(0)
            wall = _concurrent_wall(attend_model, list(range(cores)))
            full1 += n_bg * ph + n_rows * pr
            fullN += (n_bg * ph + n_rows * pr) * wall / (cores * tt)
            sample += (f"; oracle attention of 1 and 17 rows of one kv head over "
                       f"{spec.S_kv} keys, scaled to {n_bg} heads and {n_rows} rows")
            value1, valueN = spec.B * spec.S_q / full1, spec.B * spec.S_q / fullN
        else:
            value1, valueN = n_total / full1, n_total / fullN
    else:
        ph, pr, tt, where, out = attend_model(0)
        attend_parity(where, out)
        wall = _concurrent_wall(attend_model, list(range(cores)))
        # per-batch cache lengths: both costs scale with the keys attended
        frac = float(np.mean(inp["kv_lens"])) / spec.S_kv if "kv_lens" in inp else 1.0
        full1 = (n_bg * ph + n_rows * pr) * frac
        fullN = full1 * wall / (cores * tt)
        sample = (f"oracle attention of 1 and 17 rows of one (batch, kv head) over "
                  f"{spec.S_kv} keys (per thread), scaled to {n_bg} pairs and {n_rows} rows")
        if frac != 1.0:
            sample += f" and by the mean cache length ({frac:.3f} of S_kv)"
        if name == "decode-append":
            n_new = spec.B * spec.H_kv * spec.enc_len
            t_enc = encode_sample(0, n_new)[0]
            t0 = time.perf_counter()
            oracle.encode(inp["values"].reshape(-1, D), inp["v_codebook"], rotate=False)
            t_enc += time.perf_counter() - t0
            full1 += t_enc
            fullN += t_enc   # a handful of vectors: not split across threads
            sample = f"oracle key and value encode of the {n_new} new vectors; " + sample
        value1, valueN = spec.B * spec.S_q / full1, spec.B * spec.S_q / fullN
    report.update({"value": valueN, "unit": METRICS[name][1], "cores": cores,
                   "kind": "oracle", "sample": sample, "est_step_s": fullN,
                   "single_core": {"value": value1, "cores": 1, "est_step_s": full1}})
    return report


def run_reference(args, name):
    spec = WORKLOADS[name]
    inp = make_inputs(spec)
    vals = []
    for _ in range(min(args.warmup, 1)):
        cpu_baseline(name, spec, inp, budget_s=1.0)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(name, spec, inp, budget_s=args.cpu_budget / max(1, args.steps)))
    wall = time.perf_counter() - t0
    v = statistics.median(x["value"] for x in vals)
    metric, unit = METRICS[name]
    cb = dict(vals[-1])
    cb["value"] = v
    return {"impl": "reference", "metric": metric, "value": v, "unit": unit,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": wall * 1e3 / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "B": spec.B, "H_q": spec.H_q, "H_kv": spec.H_kv,
                       "D": spec.D, "S_kv": spec.S_kv, "S_q": spec.S_q},
            "cpu_baseline": cb,
            "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gqa-decode", choices=sorted(METRICS))
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, args.workload)), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    line = run_gpu(args, args.workload, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
