#!/usr/bin/env python3
"""Benchmark of the TurboQuant KV-cache hot path on GB300 (one JSON line on stdout).

Workload (N=1): the Llama-3.1-8B-shaped decode.
* Shape: 32 layers, 32 query heads, 8 KV heads (GQA 4:1), head_dim 128, batch 1, context 32768.
* Codes: 3-bit keys (2-bit Lloyd-Max + 1-bit QJL), 2-bit values in groups of 32, 128-token bf16 ring.
* Inputs: bf16 N(0,1) with 4 random K channels per head scaled x10, generated per layer with seed 1000+layer.

One step = for every layer: append one token (ring write; ring overflow quantises a 128-token block)
and run hybrid decode attention. The step is captured once as a CUDA graph and replayed. The
sequence state lives on the device, so every replay advances the context by one token.

Each step reads about 785 MB of packed records, more than the 129 MB L2. Consecutive steps
therefore cannot hit L2 for the previous step's layers, and no flush is needed.

Also reported:
* roofline: the split-K decode kernel alone, from a graph of its 32 per-layer launches, against
  the measured copy bandwidth.
* e2e: the same step through the public API, with pinned-host H2D copies of q/k/v and D2H of the
  output inside the timed region.
* quantize: bulk prefill of 65536 bf16 tokens x 8 KV heads x 32 layers (seed 4, K outliers), in tok/s.
* cpu_baseline: the fp64 oracle timed on a bounded sample, on this host's cores.

`--impl reference` times the oracle as the reference arm, on the same metric and workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attn context-tok/s & packed-KV HBM GB/s (% of 8 TB/s); quantize tok/s"
UNIT = "context-tok/s"
# Decode workloads (--workload). `ctx` is the context of every row at the first timed step; `lens`
# draws ragged per-row contexts uniform in [lo, hi] instead; inputs are seeded per layer with
# seed * 1000 + layer.
WORKLOADS = {
    "llama8b": dict(name="llama3.1-8b-shaped decode, batch 1, context 32768, K3/V2", layers=32, hq=32, hkv=8,
                    d=128, batch=1, ctx=32768, lens=None, vb=2, kb=3, outliers=("random", 4, 10.0), dist="normal",
                    seed=1),
    "batched": dict(name="llama3.1-8b-shaped batched decode, batch 16, ragged context U[4096, 8192], K3/V4",
                    layers=32, hq=32, hkv=8, d=128, batch=16, ctx=8192, lens=(4096, 8192), vb=4, kb=3,
                    outliers=None, dist="normal", seed=2),
    "d256": dict(name="head_dim 256 decode, 16 layers, batch 4, context 16384, Student-t nu=5, K3/V2", layers=16,
                 hq=32, hkv=8, d=256, batch=4, ctx=16384, lens=None, vb=2, kb=3, outliers=None, dist="student_t5",
                 seed=3),
    "long": dict(name="long-context decode, batch 32, context 131072, K3/V2 (about 99 GB of packed cache)", layers=32,
                 hq=32, hkv=8, d=128, batch=32, ctx=131072, lens=None, vb=2, kb=3, outliers=("random", 4, 10.0),
                 dist="normal", seed=4),
}
WL = dict(WORKLOADS["llama8b"])
PREFILL = dict(tokens=65536, hkv=8, layers=32, d=128, vb=2, kb=3, seed=4)
NOMINAL_HBM_GBS = 8000.0


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# --------------------------------------------------------------------------------------------
# clocks during the timed region: NVML read-only queries polled every millisecond (nvidia-smi's
# sampling period is longer than a short timed region); nvidia-smi as a fallback
# --------------------------------------------------------------------------------------------
class NvmlClocks:
    """Polls SM clock, power and the clock-event reasons of one GPU through NVML (read-only queries)."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid, period_s=0.001):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError(f"no NVML device {uuid}")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM
        self.max_mhz = float(mx.value)
        self.period = period_s
        self.samples = []
        self._stop = threading.Event()
        self.thread = None

    def _one(self):
        ct = self.ct
        mhz, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz))
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw))
        self.reasons_fn(self.h, ct.byref(rs))
        return time.time(), float(mhz.value), mw.value / 1000.0, int(rs.value)

    def _run(self):
        while not self._stop.is_set():
            self.samples.append(self._one())
            time.sleep(self.period)

    def start(self):
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def stop(self):
        self._stop.set()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        window = "timed"
        if not inside:
            inside, window = self.samples[-3:], "after the timed region (no sample inside it)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0, "source": "nvml"}
        reasons = sorted({name for x in inside for bit, name in self.REASONS.items() if x[3] & bit})
        return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(x[1] for x in inside), "power_w_max": max(x[2] for x in inside),
                "reasons": reasons, "samples": len(inside), "window": window, "source": "nvml, 1 ms polling"}


class SmiClocks:
    """nvidia-smi sampler (fallback when NVML cannot be loaded)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-i", str(self.gpu_id),
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for t, s in self.samples if t0 <= t <= t1 and len(s) >= 9]
        window = "timed"
        if not inside:
            inside = [s for _, s in self.samples if len(s) >= 9]
            window = "warm-up and timed (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "note": "nvidia-smi unavailable"}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[1]) for s in inside if num(s[1]) is not None]
        mx = [num(s[2]) for s in inside if num(s[2]) is not None]
        pw = [num(s[3]) for s in inside if num(s[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4) if s[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "reasons": reasons, "samples": len(inside), "window": window,
                "source": "nvidia-smi"}


def clock_sampler(dev):
    import torch
    uuid = str(torch.cuda.get_device_properties(dev).uuid)
    uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    try:
        return NvmlClocks(uuid)
    except Exception:
        return SmiClocks(uuid)


# --------------------------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------------------------
def aggregate_over_ranks(ms, units, world, device):
    """Whole-job throughput of `world` replicas: every rank processed `units`; time = max over ranks."""
    t_max = float(ms)
    if world > 1:
        import torch
        import torch.distributed as dist
        tt = torch.tensor([t_max], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t_max = float(tt.item())
    return t_max, units * world / (t_max * 1e-3)


def record_bytes(wl):
    """Canonical key + value record bytes of one token and KV head."""
    d = wl["d"]
    return (d * (wl["kb"] - 1) // 8 + d // 8 + 4) + (d * wl["vb"] // 8 + d // 16)


def nominal_step_bytes(wl, mode="hybrid"):
    """Algorithmic bytes of one decode step at the workload's nominal contexts (packed records + ring +
    q + out, all layers); a description of the workload, identical in both arms."""
    lens = (synth_lengths(wl) if wl["lens"] is not None else [wl["ctx"]] * wl["batch"])
    total = 0
    for L in lens:
        packed = L if mode == "full_tq" else 128 * ((L - 1) // 128)
        total += wl["layers"] * (wl["hkv"] * (packed * record_bytes(wl) + (L - packed) * wl["d"] * 4)
                                 + wl["hq"] * wl["d"] * 6)
    return total


def synth_lengths(wl):
    from kv_cache_quantization_quantize_gb300 import synth
    return synth.ragged_lengths(wl["batch"], wl["lens"][0], wl["lens"][1], seed=wl["seed"])


def workload_config(wl, mode="hybrid"):
    cfg = {"workload": wl["name"], "layers": wl["layers"], "q_heads": wl["hq"], "kv_heads": wl["hkv"],
           "head_dim": wl["d"], "batch_per_gpu": wl["batch"], "context": wl["ctx"], "key_bits": wl["kb"],
           "value_bits": wl["vb"], "ring": 128,
           "l2": f"inputs larger than L2 ({nominal_step_bytes(wl, mode) / 1e6:.0f} MB of packed records per step vs "
                 f"129 MB L2)",
           "step": f"append 1 token + hybrid decode attention, all {wl['layers']} layers"}
    if wl["lens"] is not None:
        cfg.update(context=f"ragged, uniform in [{wl['lens'][0]}, {wl['lens'][1]}] (seed {wl['seed']})")
    if mode == "full_tq":
        cfg.update(workload=wl["name"] + ", full_tq mode", ring=0, mode="full_tq",
                   step=f"append 1 token (quantised at once) + decode over packed tokens only, all {wl['layers']} "
                        "layers")
    return cfg


def bench_config(world, mode="hybrid", layout="contiguous"):
    """The `config` of the JSON line. It depends on the workload and flags only, so both arms print the
    same one."""
    cfg = dict(workload_config(WL, mode), parallelism="replicas" if world > 1 else "single GPU")
    if layout == "paged":
        cfg["layout"] = "paged (scrambled block table)"
    elif layout == "paged-ordered":
        cfg["layout"] = "paged (block table in allocation order)"
    return cfg


DECODE_SOURCES = ("tq_decode.cu", "tq_decode_common.cuh", "tq_quantize_common.cuh", "tq_device.cuh", "tq_internal.h")
DECODE_PROFILE = os.path.join(ROOT, "profiles", "k_decode_llama8b_b1_ctx32k.md")


def decode_source_digest():
    """sha256 over the code of the sources that make up the decode kernel, with comments and whitespace
    removed (ties ncu counters to a kernel version; an edit of a comment keeps them)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "kv_cache_quantization_quantize_gb300", "csrc", name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)  # block comments
        text = re.sub(r"//[^\n]*", " ", text)                 # line comments
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


def profiled_traffic(path=DECODE_PROFILE):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current sources."""
    try:
        with open(path) as f:
            text = f.read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        line = line.strip().strip("`- ")
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("source_digest") != decode_source_digest():
        return None
    try:
        return int(fields["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def fidelity_report(cache, k, v, L, n_max=4096):
    """Mean per-vector cosine similarity of dequantised packed tokens against the inputs they were coded
    from (the guide's §六 fidelity figure): layer 0, row 0, every KV head, the first min(n_max, packed)
    tokens. Keys with and without the QJL term, values at the workload's value bits.
    Dequantised on the device by tq_dequantize_tokens."""
    import torch
    import torch.nn.functional as F
    Hkv, d = k.shape[1], k.shape[2]
    n = min(n_max, 128 * ((L - 1) // 128))  # packed tokens of the row (the ring holds the rest)
    nq = 16  # N(0, 1) queries per head for the score vectors
    gen = torch.Generator(device=k.device)
    gen.manual_seed(17)
    acc = {"key_cos_mse": 0.0, "key_cos_qjl": 0.0, "value_cos": 0.0, "score_cos_mse": 0.0, "score_cos_qjl": 0.0}
    for h in range(Hkv):
        ko, vo = k[:n, h].float(), v[:n, h].float()
        k_mse, v_hat = cache.dequantize(0, 0, h, 0, n, with_qjl=False)
        k_qjl, _ = cache.dequantize(0, 0, h, 0, n, with_qjl=True)
        acc["key_cos_mse"] += F.cosine_similarity(k_mse, ko, dim=1).mean().item() / Hkv
        acc["key_cos_qjl"] += F.cosine_similarity(k_qjl, ko, dim=1).mean().item() / Hkv
        acc["value_cos"] += F.cosine_similarity(v_hat, vo, dim=1).mean().item() / Hkv
        # the score vector of a query over the tokens: <q, k_hat_t> is the decode's estimate of <q, k_t>
        q = torch.randn((nq, d), generator=gen, device=k.device)
        s_ref = q @ ko.T
        acc["score_cos_mse"] += F.cosine_similarity(q @ k_mse.T, s_ref, dim=1).mean().item() / Hkv
        acc["score_cos_qjl"] += F.cosine_similarity(q @ k_qjl.T, s_ref, dim=1).mean().item() / Hkv
    acc["tokens"] = n * Hkv
    acc["sample"] = (f"layer 0, row 0, {Hkv} KV heads x the first {n} packed tokens, against the bf16 inputs; "
                     f"score vectors of {nq} N(0,1) queries per head over those tokens")
    return acc


def measure_decode(tqm, synth, dev, wl, args, K, W, world, headline):
    """One decode workload: prefill the cache, capture the step (append 1 token + decode, every layer) as
    a CUDA graph, time K replays after W warm-up replays, and time the split-K kernel alone. With
    `headline`, also the two end-to-end figures (graph replay and eager per-layer API calls, both with
    pinned-host copies inside the timed region)."""
    import torch
    import torch.distributed as dist
    L_layers, Hq, Hkv, d, B, ctx, vb = wl["layers"], wl["hq"], wl["hkv"], wl["d"], wl["batch"], wl["ctx"], wl["vb"]
    n_e2e_warm = 2
    # tokens appended after prefill by all passes (eager step, warm-up, timed, both e2e passes)
    extra = 1 + W + K + (2 * (n_e2e_warm + K) if headline else 0) + 8
    lens = synth_lengths(wl) if wl["lens"] is not None else [ctx] * B  # context of each row at the first timed step
    max_ctx = max(lens) + extra
    full = args.mode == "full_tq"
    paged = args.layout.startswith("paged") and headline
    max_pages = (max_ctx + 127) // 128
    cfg = tqm.config(head_dim=d, value_bits=vb, key_bits=wl["kb"], n_layers=L_layers, n_kv_heads=Hkv, n_q_heads=Hq,
                     max_seqs=B, max_ctx=max_ctx, seed=1, mode=args.mode if headline else "hybrid",
                     n_blocks=B * max_pages if paged else 0)
    cache = tqm.TurboQuantCache(cfg, device=dev)
    ids = torch.arange(B, dtype=torch.int32, device=dev)
    if paged:  # every page of every row mapped to a block of a seeded permutation of the pool (or in order)
        if args.layout == "paged":
            perm = torch.randperm(B * max_pages, generator=torch.Generator().manual_seed(11)).to(torch.int32)
        else:
            perm = torch.arange(B * max_pages, dtype=torch.int32)
        cache.block_table.copy_(perm.view(B, max_pages).to(dev))
    # after the eager step and the W warm-up replays, the first timed step of row b attends lens[b] tokens
    L0 = [n - W - 2 for n in lens]
    for l in range(L_layers):
        k, v = synth.kv_tokens(max(L0), Hkv, d, seed=wl["seed"] * 1000 + l, dist=wl["dist"], outliers=wl["outliers"],
                               device=dev)
        for b in range(B):  # one row per call: rows share the layer's tokens, each with its own length
            cache.append(l, k[None], v[None], ids[b:b + 1], torch.full((1,), L0[b], dtype=torch.int32, device=dev))
        if l == 0:
            fidelity = fidelity_report(cache, k, v, L0[0])
        del k, v
    torch.cuda.synchronize()
    if cache.check_status():
        raise RuntimeError("device status after prefill")
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    knew = torch.randn((L_layers, B, 1, Hkv, d), generator=gen, device=dev).to(torch.bfloat16)
    vnew = torch.randn((L_layers, B, 1, Hkv, d), generator=gen, device=dev).to(torch.bfloat16)
    qs = torch.randn((L_layers, B, Hq, d), generator=gen, device=dev).to(torch.bfloat16)
    outs = torch.empty((L_layers, B, Hq, d), dtype=torch.float32, device=dev)
    ones = torch.ones(B, dtype=torch.int32, device=dev)
    ws = cache.workspace(B, max_ctx)
    s = torch.cuda.Stream(device=dev)

    fused = getattr(args, "step_call", "fused") == "fused"

    def step():
        for l in range(L_layers):
            if fused:  # the one-token append and the decode in one launch
                cache.decode_step(l, knew[l, :, 0], vnew[l, :, 0], qs[l], ids, out=outs[l], max_ctx_hint=max_ctx,
                                  workspace=ws, stream=s)
            else:
                cache.append(l, knew[l], vnew[l], ids, ones, stream=s)
                cache.decode(l, qs[l], ids, out=outs[l], max_ctx_hint=max_ctx, workspace=ws, stream=s)

    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # eager: sets kernel attributes before capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    # per layer: the fused step kernel, or the small append and the split-K decode (query prep and combine
    # inside the decode either way)
    launches_per_step = L_layers * (1 if fused and not full else 2)  # full_tq: tq_decode_step runs both

    sampler = clock_sampler(dev)
    sampler.start()
    time.sleep(0.05)
    with torch.cuda.stream(s):
        for _ in range(W):
            g.replay()
    torch.cuda.synchronize()
    L_first = [cache.state(0, b)[0] + 1 for b in range(B)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    ev0.record(s)
    with torch.cuda.stream(s):
        for _ in range(K):
            g.replay()
    ev1.record(s)
    ev1.synchronize()
    t_host1 = time.time()
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        dist.barrier()
    sampler.stop()
    clocks = sampler.summary(t_host0, t_host1)
    status = cache.check_status()
    ctx_tokens = sum(Lb + i for Lb in L_first for i in range(K))  # each step attends every row's full context
    t_max, value = aggregate_over_ranks(ms, ctx_tokens, world, dev)  # max over ranks; whole-job throughput
    ms_per_step = t_max / K

    # algorithmic bytes per step: packed records + ring (K,V bf16) + q + out, all layers
    rec = record_bytes(wl)
    step_bytes = 0.0
    for Lb in L_first:
        Lmid = Lb + (K - 1) / 2.0
        packed = Lmid if full else 128 * ((Lmid - 1) // 128)
        ring = Lmid - packed
        step_bytes += L_layers * (Hkv * (packed * rec + ring * d * 2 * 2) + Hq * d * (2 + 4))
    hbm_gbs = step_bytes / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()

    # ---- the split-K kernel alone: a graph of its per-layer launches ----
    for l in range(L_layers):
        cache.decode_phase(0, l, qs[l], ids, outs[l], max_ctx_hint=max_ctx, workspace=ws, stream=s)
    torch.cuda.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s):
        for l in range(L_layers):
            cache.decode_phase(1, l, qs[l], ids, outs[l], max_ctx_hint=max_ctx, workspace=ws, stream=s)
    with torch.cuda.stream(s):
        for _ in range(3):
            g2.replay()
    torch.cuda.synchronize()
    kern_bytes = 0
    for b in range(B):
        Lk, Fk = cache.state(0, b)
        packed_k = 128 * ((Lk - 1) // 128) + Fk
        ring_k = Lk - packed_k
        kern_bytes += Hkv * (packed_k * rec + ring_k * d * 2 * 2) + Hq * d * (2 + 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(K, 10)
    e0.record(s)
    with torch.cuda.stream(s):
        for _ in range(reps):
            g2.replay()
    e1.record(s)
    torch.cuda.synchronize()
    kern_us = e0.elapsed_time(e1) * 1e3 / (reps * L_layers)
    kern_gbs = kern_bytes / (kern_us * 1e-6) / 1e9
    roof = {"kernel": "k_decode (split-K decode over packed pages + ring split)", "bound": "hbm",
            "achieved": kern_gbs, "peak": peak, "unit": "GB/s", "frac": kern_gbs / peak, "peak_kind": peak_kind,
            "bytes_per_launch": kern_bytes, "us_per_launch": kern_us, "frac_of_8TBps": kern_gbs / NOMINAL_HBM_GBS}
    res = {"workload": wl["name"], "value": value, "unit": UNIT, "ms_per_step": ms_per_step, "steps": K,
           "hbm_gbs": hbm_gbs, "pct_of_8TBps": 100.0 * hbm_gbs / NOMINAL_HBM_GBS,
           "pct_of_measured_hbm": 100.0 * hbm_gbs / peak, "step_bytes": step_bytes, "roofline": roof,
           "clocks": clocks, "gpu_launches": launches_per_step * K, "device_status": status,
           "step_call": "tq_decode_step (append + decode in one launch per layer)" if fused
           else "tq_quantize_append + tq_decode_attention (two launches per layer)",
           "cos_sim": fidelity}
    del g2
    if headline:
        res.update(measure_e2e(cache, s, qs, knew, vnew, outs, ids, ones, ws, max_ctx, g, K, n_e2e_warm, world, B,
                               L_layers, fused))
    del g
    del cache, knew, vnew, qs, outs, ws
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def measure_e2e(cache, s, qs, knew, vnew, outs, ids, ones, ws, max_ctx, g, K, n_warm, world, B, L_layers, fused):
    """The step end to end with host buffers: every step copies q, k and v from pinned host memory to the
    device and the outputs back, inside the timed region. `e2e` replays the captured graph between the
    copies; `e2e_api` calls the step's entry points per layer through the Python binding (ctypes -> C
    ABI), with no graph: tq_decode_step, or tq_quantize_append and tq_decode_attention."""
    import torch
    hq = torch.empty(qs.shape, dtype=qs.dtype, pin_memory=True)
    hk = torch.empty(knew.shape, dtype=knew.dtype, pin_memory=True)
    hv = torch.empty(vnew.shape, dtype=vnew.dtype, pin_memory=True)
    ho = torch.empty(outs.shape, dtype=outs.dtype, pin_memory=True)
    hq.copy_(qs)
    hk.copy_(knew)
    hv.copy_(vnew)
    h2d = hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2
    d2h = ho.numel() * 4

    def graph_step():
        with torch.cuda.stream(s):
            qs.copy_(hq, non_blocking=True)
            knew.copy_(hk, non_blocking=True)
            vnew.copy_(hv, non_blocking=True)
            g.replay()
            ho.copy_(outs, non_blocking=True)

    def api_step():
        with torch.cuda.stream(s):
            qs.copy_(hq, non_blocking=True)
            knew.copy_(hk, non_blocking=True)
            vnew.copy_(hv, non_blocking=True)
            for l in range(L_layers):
                if fused:
                    cache.decode_step(l, knew[l, :, 0], vnew[l, :, 0], qs[l], ids, out=outs[l], max_ctx_hint=max_ctx,
                                      workspace=ws, stream=s)
                else:
                    cache.append(l, knew[l], vnew[l], ids, ones, stream=s)
                    cache.decode(l, qs[l], ids, out=outs[l], max_ctx_hint=max_ctx, workspace=ws, stream=s)
            ho.copy_(outs, non_blocking=True)

    out = {}
    for key, fn, launches in (("e2e", graph_step, "one CUDA graph replay"),
                              ("e2e_api", api_step, "per-layer tq_decode_step calls" if fused
                               else "per-layer tq_quantize_append + tq_decode_attention calls")):
        for _ in range(n_warm):
            fn()
        torch.cuda.synchronize()
        L0 = [cache.state(0, b)[0] + 1 for b in range(B)]
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(s)
        for _ in range(K):
            fn()
        f1.record(s)
        torch.cuda.synchronize()
        e_ms = f0.elapsed_time(f1)
        out[key] = {"value": sum(Lb + i for Lb in L0 for i in range(K)) * world / (e_ms * 1e-3), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / K,
                    "launch": launches}
        if cache.check_status():
            out[key]["device_status"] = "non-zero"
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from kv_cache_quantization_quantize_gb300 import build as _build
    _build.build()
    import kv_cache_quantization_quantize_gb300 as tqm
    from kv_cache_quantization_quantize_gb300 import synth

    K, W = args.steps, args.warmup
    head = measure_decode(tqm, synth, dev, WL, args, K, W, world, headline=True)
    full, paged = args.mode == "full_tq", args.layout.startswith("paged")
    traffic = None if full or paged or WL["name"] != WORKLOADS["llama8b"]["name"] else profiled_traffic()
    head["roofline"]["traffic"] = traffic
    peak, _ = measured_peaks()

    quant = None
    if not args.skip_quantize:
        quant = bench_quantize(tqm, synth, dev, args, peak)
    # the other decode workloads, each with its own cache (freed after it), as nested records
    nested = {}
    if args.nested and WL["name"] == WORKLOADS["llama8b"]["name"] and not full and not paged:
        for name, over in (("batched", {}), ("d256", {}), ("d256_v4", {"vb": 4}), ("long", {})):
            wl = dict(WORKLOADS[name.split("_")[0]], **over)
            if over:
                wl["name"] = wl["name"].replace("K3/V2", f"K3/V{over['vb']}")
            r = measure_decode(tqm, synth, dev, wl, args, max(10, min(K, 50)), W, world, headline=False)
            r["config"] = workload_config(wl)
            nested[name] = r

    # prefill attention of a 512-query chunk at the end of the 32K sequence, on the default path and on the
    # CUDA-core path it replaces, as a nested record
    prefill = None
    if args.nested and WL["name"] == WORKLOADS["llama8b"]["name"] and not full and not paged and rank == 0:
        prefill = measure_prefill(tqm, synth, dev, 512, False, 5)
        cc = measure_prefill(tqm, synth, dev, 512, True, 2, warm=1)
        prefill["cuda_core_path_ms_per_layer"] = cc["ms_per_layer"]

    line = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 tensor-core products, f32 accumulate and softmax", "data": "synthetic",
        "config": bench_config(world, args.mode, args.layout),
        "hbm_gbs": head["hbm_gbs"], "pct_of_8TBps": head["pct_of_8TBps"],
        "pct_of_measured_hbm": head["pct_of_measured_hbm"],
        "roofline": head["roofline"], "e2e": head["e2e"], "e2e_api": head["e2e_api"],
        "gpu_launches": head["gpu_launches"], "clocks": head["clocks"], "device_status": head["device_status"],
        "step_call": head["step_call"], "cos_sim": head["cos_sim"],
    }
    if quant is not None:
        line["quantize_tok_s"] = quant["tok_s"]
        line["quantize"] = quant
    if nested:
        line["workloads"] = nested
    if prefill is not None:
        line["prefill"] = prefill
    if (rank == 0 and world == 1 and not args.no_cpu_baseline and not full and not paged
            and WL["kb"] == 3 and args.head_dim == 128):  # the oracle on this workload
        line["cpu_baseline"] = cpu_baseline(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def bench_quantize(tqm, synth, dev, args, peak):
    import torch
    T, Hkv, L_layers, d, vb = PREFILL["tokens"], PREFILL["hkv"], PREFILL["layers"], PREFILL["d"], PREFILL["vb"]
    layout = getattr(args, "layout", "contiguous")
    paged = layout.startswith("paged")
    max_pages = (T + 127) // 128
    cfg = tqm.config(head_dim=d, value_bits=vb, key_bits=PREFILL["kb"], n_layers=L_layers, n_kv_heads=Hkv,
                     n_q_heads=4 * Hkv, max_seqs=1,
                     max_ctx=T, seed=PREFILL["seed"], n_blocks=max_pages if paged else 0)
    qc = tqm.TurboQuantCache(cfg, device=dev)
    if paged:
        perm = (torch.randperm(max_pages, generator=torch.Generator().manual_seed(12)).to(torch.int32)
                if layout == "paged" else torch.arange(max_pages, dtype=torch.int32))
        qc.block_table.copy_(perm.view(1, max_pages).to(dev))
    k, v = synth.kv_tokens(T, Hkv, d, seed=PREFILL["seed"], outliers=WL["outliers"], device=dev)
    k, v = k[None].contiguous(), v[None].contiguous()
    ids = torch.zeros(1, dtype=torch.int32, device=dev)
    nn = torch.full((1,), T, dtype=torch.int32, device=dev)

    def one_pass():
        qc.reset(ids)
        for l in range(L_layers):
            qc.append(l, k, v, ids, nn)

    for _ in range(3):
        one_pass()
    torch.cuda.synchronize()
    reps = 20
    sampler = clock_sampler(dev)
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record()
    for _ in range(reps):
        one_pass()
    e1.record()
    e1.synchronize()
    t1 = time.time()
    sampler.stop()
    ms = e0.elapsed_time(e1) / reps
    if qc.check_status():
        raise RuntimeError("device status after quantise")
    rec = (d * (WL["kb"] - 1) // 8 + d // 8 + 4) + (d * vb // 8 + d // 16)
    packed = 128 * ((T - 1) // 128)
    ring = T - packed
    bytes_pass = L_layers * Hkv * (T * d * 2 * 2 + packed * rec + ring * d * 2 * 2)
    gbs = bytes_pass / (ms * 1e-3) / 1e9
    return {"tok_s": T / (ms * 1e-3), "token_head_layers_per_s": T * Hkv * L_layers / (ms * 1e-3),
            "ms_per_pass": ms, "passes": reps, "clocks": sampler.summary(t0, t1), "workload": f"bulk prefill {T} bf16 tokens x {Hkv} KV heads x {L_layers} layers, d={d}, K{PREFILL['kb']}/V{vb}",
            "path": ("tcgen05 rotation (H diag(D)) and QJL projection (bf16 hi/lo) into TMEM, thread-per-token "
                     "coding, TMA page loads" if d in (64, 128) else
                     "tcgen05 rotation (two 128-point H diag(D_i) products, butterfly on CUDA cores) and QJL "
                     "projection (bf16 hi/lo, S streamed in 32-row chunks) into TMEM, thread-per-token coding, "
                     "TMA page loads" if d == 256 else
                     "CUDA-core quantise kernel (QJL projection as an f16 mma.sync GEMM per 32-token block)"),
            "hbm_gbs": gbs, "frac_of_measured_hbm": gbs / peak, "bytes_per_pass": bytes_pass}


def measure_prefill(tqm, synth, dev, Tq, force_cc, reps, warm=3):
    """Prefill attention of one chunk over the cache: the Llama-3.1-8B shape (8 KV heads, 32 q heads,
    d=128, K3/V2), one sequence of 32768 tokens whose last `Tq` tokens are the chunk, all 32 layers (32
    layers of packed history, 785 MB, more than L2). `warm` untimed passes, then `reps` timed passes of
    all layers (CUDA events on the stream). Returns a dict."""
    import torch
    from kv_cache_quantization_quantize_gb300 import _abi
    L_layers, Hq, Hkv, d, ctx, vb = WL["layers"], WL["hq"], WL["hkv"], WL["d"], WL["ctx"], WL["vb"]
    lib = _abi.load()
    lib.tq_debug_prefill_path(1 if force_cc else 0)
    tc = not force_cc and d == 128 and WL["kb"] == 3 and Hq == 4 * Hkv and Tq >= 32
    cfg = tqm.config(head_dim=d, value_bits=vb, key_bits=WL["kb"], n_layers=L_layers, n_kv_heads=Hkv, n_q_heads=Hq,
                     max_seqs=1, max_ctx=ctx, seed=1)
    cache = tqm.TurboQuantCache(cfg, device=dev)
    ids = torch.zeros(1, dtype=torch.int32, device=dev)
    for l in range(L_layers):
        k, v = synth.kv_tokens(ctx, Hkv, d, seed=1000 + l, outliers=WL["outliers"], device=dev)
        cache.append(l, k[None].contiguous(), v[None].contiguous(), ids, torch.full((1,), ctx, dtype=torch.int32,
                                                                                     device=dev))
        del k, v
    gen = torch.Generator(device=dev)
    gen.manual_seed(9)
    q = torch.randn((L_layers, 1, Tq, Hq, d), generator=gen, device=dev).to(torch.bfloat16)
    out = torch.empty((L_layers, 1, Tq, Hq, d), dtype=torch.float32, device=dev)
    nq = torch.full((1,), Tq, dtype=torch.int32, device=dev)
    ws = cache.prefill_workspace(1, Tq, ctx)
    try:
        for _ in range(warm):
            for l in range(L_layers):
                cache.prefill(l, q[l], ids, nq, out=out[l], max_ctx_hint=ctx, workspace=ws)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            for l in range(L_layers):
                cache.prefill(l, q[l], ids, nq, out=out[l], max_ctx_hint=ctx, workspace=ws)
        e1.record()
        torch.cuda.synchronize()
    finally:
        lib.tq_debug_prefill_path(0)
    ms = e0.elapsed_time(e1) / reps
    status = cache.check_status()
    del cache, q, out, ws
    torch.cuda.empty_cache()
    return {"value": Tq / (ms * 1e-3), "unit": "query-tok/s", "ms_per_chunk": ms, "ms_per_layer": ms / L_layers,
            "passes": reps, "warmup": warm,
            "config": {"workload": f"{WL['name']}: prefill chunk of {Tq} queries at the end of a "
                                   f"{ctx}-token sequence", "layers": L_layers},
            "path": ("tcgen05: tiles of 32 queries x 4 heads; query operands in TMEM, key planes and values "
                     "expanded once per page and tile into rotating shared-memory tiles while the previous "
                     "MMAs run, scores and P.V into TMEM; then the exact ring split and the combine, one CTA per (query, KV head)") if tc
            else "one split-K decode launch over chunk-query rows (causal length per row)",
            "device_status": status}


def bench_prefill(args):
    """`--prefill-chunk TQ`: one JSON line (query tokens/s) for the prefill of a TQ-query chunk; it is not
    the bench line of the decode step."""
    import torch
    import kv_cache_quantization_quantize_gb300 as tqm
    from kv_cache_quantization_quantize_gb300 import synth, build as _build
    _build.build()
    dev = torch.device("cuda", 0)
    force_cc = getattr(args, "prefill_path", "auto") == "cuda-core"
    r = measure_prefill(tqm, synth, dev, args.prefill_chunk, force_cc, max(1, min(args.steps, 5)),
                        warm=max(1, min(args.warmup, 3)))
    print(json.dumps(dict({"metric": "prefill attention query tokens/s (all layers)"}, **r)), flush=True)


def bench_codec(args):
    """Comparison codec (KIVI 2-bit or Bonsai 1-bit) over the whole 32K-token KV cache of the
    Llama-3.1-8B shape: 32 layers x 8 KV heads x 128, one quantise launch per layer (K and V together),
    then one dequantise launch per layer. Every layer has its own input (134 MB, above L2). Prints one
    JSON line (tokens/s of quantisation; HBM fraction per launch); it is not the bench line of the decode
    step."""
    import torch
    from kv_cache_quantization_quantize_gb300 import codecs, synth
    dev = torch.device("cuda", 0)
    L_layers, Hkv, d, T = args.codec_layers or WL["layers"], WL["hkv"], WL["d"], WL["ctx"]
    peak, peak_kind = measured_peaks()
    kv = [synth.kv_tokens(T, Hkv, d, seed=2000 + l, outliers=WL["outliers"], device=dev) for l in range(L_layers)]
    deq_out = tuple(torch.empty(T, Hkv, d, dtype=torch.bfloat16, device=dev) for _ in range(2))
    if args.codec == "kivi2":
        outs = [codecs.kivi2_alloc(T, Hkv, d, dev) for _ in range(L_layers)]
        quant = lambda l: codecs.kivi2_quantize(kv[l][0], kv[l][1], out=outs[l])
        dequant = lambda l: codecs.kivi2_dequantize(outs[l], T, Hkv, d, out=deq_out)
    else:
        outs = [codecs.bonsai1_alloc(T * Hkv, d, dev) for _ in range(L_layers)]
        quant = lambda l: codecs.bonsai1_quantize(kv[l][0], kv[l][1], out=outs[l])
        dequant = lambda l: codecs.bonsai1_dequantize(outs[l], T, Hkv, d, out=deq_out)
    code_bytes = sum(t.numel() * t.element_size() for t in outs[0].values())
    in_bytes = 2 * T * Hkv * d * 2

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            for l in range(L_layers):
                fn(l)
        torch.cuda.synchronize()
        reps = max(1, min(args.steps, 10))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            for l in range(L_layers):
                fn(l)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    mq, md = timed(quant), timed(dequant)
    per = lambda ms: (in_bytes + code_bytes) / (ms * 1e-3 / L_layers) / 1e9
    print(json.dumps({
        "metric": f"{args.codec} KV quantisation tokens/s (all layers)", "value": T / (mq * 1e-3), "unit": "tok/s",
        "ms_per_pass": mq, "us_per_launch": 1e3 * mq / L_layers,
        "roofline": {"bound": "hbm", "achieved": per(mq), "peak": peak, "unit": "GB/s", "frac": per(mq) / peak,
                     "peak_kind": peak_kind, "bytes_per_launch": in_bytes + code_bytes},
        "dequantize": {"ms_per_pass": md, "us_per_launch": 1e3 * md / L_layers, "achieved_gbs": per(md),
                       "frac": per(md) / peak},
        "stored_bytes_all_layers": code_bytes * L_layers,
        "config": {"workload": f"{args.codec} over the KV cache of {WL['name'].split(',')[0]}: {T} tokens x {Hkv} KV "
                               f"heads x {L_layers} layers, d={d}, bf16 in", "l2": "each layer's input exceeds L2"},
    }), flush=True)


def profile_quantize(passes):
    """A small quantise-only run for profilers: one layer of the prefill workload, `passes` times.

    Prints one line with the measured time per layer; it is not a bench line.
    """
    import torch
    import kv_cache_quantization_quantize_gb300 as tqm
    from kv_cache_quantization_quantize_gb300 import synth
    dev = torch.device("cuda", 0)
    T, Hkv, d, vb = PREFILL["tokens"], PREFILL["hkv"], PREFILL["d"], PREFILL["vb"]
    cfg = tqm.config(head_dim=d, value_bits=vb, key_bits=PREFILL["kb"], n_layers=1, n_kv_heads=Hkv,
                     n_q_heads=4 * Hkv, max_seqs=1, max_ctx=T, seed=PREFILL["seed"])
    qc = tqm.TurboQuantCache(cfg, device=dev)
    k, v = synth.kv_tokens(T, Hkv, d, seed=PREFILL["seed"], outliers=WL["outliers"], device=dev)
    k, v = k[None].contiguous(), v[None].contiguous()
    ids = torch.zeros(1, dtype=torch.int32, device=dev)
    nn = torch.full((1,), T, dtype=torch.int32, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(passes):
        qc.reset(ids)
        e0.record()
        qc.append(0, k, v, ids, nn)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    if qc.check_status():
        raise RuntimeError("device status after quantise")
    print(json.dumps({"profile": "quantize", "tokens": T, "kv_heads": Hkv, "head_dim": d, "value_bits": vb,
                      "ms_per_layer": times}), flush=True)


# --------------------------------------------------------------------------------------------
# oracle timing (cpu_baseline leg and --impl reference)
# --------------------------------------------------------------------------------------------
def oracle_unit_setup(k, v):
    """Packed records + ring of one (layer, KV head) unit, built by the oracle from that unit's fp64 K and V
    [ctx, d] (the unit's context), with the new decode token taken as the last one."""
    import numpy as np
    import oracle
    d, ctx, Hkv = WL["d"], k.shape[0], WL["hkv"]
    D = oracle.rademacher_signs(1, d)
    S = oracle.gaussian_matrix_bf16(1, d)
    c, t = oracle.lloyd_max_codebook(d, WL["kb"] - 1)
    Np, R = oracle.history_split(ctx)
    keys = oracle.quantize_keys(k[:Np], D, S, c, t)
    vals = oracle.quantize_values(v[:Np], D, WL["vb"])
    q = np.random.default_rng(0).standard_normal((WL["hq"] // Hkv, d))
    return dict(keys=keys, vals=vals, rk=k[Np:], rv=v[Np:], q=q, D=D, S=S, c=c, t=t, k_new=k[-1:], v_new=v[-1:])


def oracle_sample_setup():
    """Records + ring of one (layer 0, KV head 0) unit of the workload."""
    from kv_cache_quantization_quantize_gb300 import synth
    k, v = synth.kv_tokens(WL["ctx"], WL["hkv"], WL["d"], seed=WL["seed"] * 1000, dist=WL["dist"],
                           outliers=WL["outliers"])
    return oracle_unit_setup(k[:, 0].double().numpy(), v[:, 0].double().numpy())


def oracle_unit_step(st):
    """One decode step of one (layer, KV head): quantise the new token's records, then attend."""
    import oracle
    oracle.quantize_keys(st["k_new"], st["D"], st["S"], st["c"], st["t"])
    oracle.quantize_values(st["v_new"], st["D"], WL["vb"])
    return oracle.decode_attention(st["q"], st["keys"], st["vals"], st["rk"], st["rv"], st["D"], st["S"], st["c"])


def oracle_units():
    """(layer, KV head, row) units of one decode step; the oracle times one and extrapolates."""
    return WL["layers"] * WL["hkv"] * WL["batch"]


def oracle_sample_reps():
    """Timed oracle steps: 150 at 32K context, fewer at longer contexts (a bounded sample)."""
    return max(10, 150 * 32768 // WL["ctx"])


def _oracle_child(threads, args, mode="--oracle-sample", arg=None):
    """Runs an oracle timing in a child process limited to `threads` BLAS/OpenMP threads."""
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), mode, str(arg if arg is not None else oracle_sample_reps()),
           "--workload", args.workload]
    if args.value_bits:
        cmd += ["--value-bits", str(args.value_bits)]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=900)
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(args):
    """Times the oracle in child processes so that their thread counts are known. On the batch-1 32K
    workload the all-core figure is one full decode step (every layer and KV head, each with its own
    records); elsewhere, and on one thread, a sample of one (layer, KV head, row) unit extrapolated over
    the step's units."""
    cores = os.cpu_count() or 1
    full = WL["name"] == WORKLOADS["llama8b"]["name"]
    try:
        res = _oracle_child(cores, args, "--oracle-full-step", 1) if full else _oracle_child(cores, args)
    except Exception as e:  # report, do not fail the GPU line
        return {"value": None, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": f"failed: {e}"}
    line = {"value": res["value"], "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": res["sample"], "seconds": res["seconds"]}
    try:
        one = _oracle_child(1, args)
        line["single_thread"] = {"value": one["value"], "unit": UNIT, "cores": 1, "seconds": one["seconds"],
                                 "sample": one["sample"]}
    except Exception as e:
        line["single_thread"] = {"value": None, "note": f"failed: {e}"}
    return line


def oracle_sample_main(reps):
    st = oracle_sample_setup()
    oracle_unit_step(st)  # warm
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_unit_step(st)
    dt = (time.perf_counter() - t0) / reps
    units = oracle_units()
    step_s = dt * units  # extrapolated linearly to all layers, KV heads and rows
    value = WL["batch"] * WL["ctx"] / step_s
    print(json.dumps({"value": value, "seconds": dt * reps,
                      "sample": f"{reps} decode steps of 1 layer x 1 KV head x 1 row ({WL['hq'] // WL['hkv']} query "
                                f"heads, {WL['ctx']} context, head_dim {WL['d']}) timed; extrapolated linearly x{units} "
                                f"({WL['layers']} layers x {WL['hkv']} KV heads x {WL['batch']} rows)"}))


def oracle_full_step_main(steps):
    """Whole decode steps of the batch-1 workload by the oracle: the records of one layer's KV heads are
    built first (untimed, inputs seeded like the GPU arm's layer 0), then `steps` steps are timed, each
    quantising the new token and attending over the records and ring of every (layer, KV head) unit. The
    layers reuse layer 0's records: the oracle's cost does not depend on the values, and building 32
    layers' records would only lengthen the untimed setup."""
    from kv_cache_quantization_quantize_gb300 import synth
    k, v = synth.kv_tokens(WL["ctx"], WL["hkv"], WL["d"], seed=WL["seed"] * 1000, dist=WL["dist"],
                           outliers=WL["outliers"])
    k, v = k.double().numpy(), v.double().numpy()
    heads = [oracle_unit_setup(k[:, h].copy(), v[:, h].copy()) for h in range(WL["hkv"])]
    del k, v
    oracle_unit_step(heads[0])  # warm
    t0 = time.perf_counter()
    for _ in range(steps):
        for _layer in range(WL["layers"]):
            for st in heads:
                oracle_unit_step(st)
    dt = (time.perf_counter() - t0) / steps
    print(json.dumps({"value": WL["batch"] * WL["ctx"] / dt, "seconds": dt * steps,
                      "sample": f"{steps} full decode step(s): {WL['layers']} layers x {WL['hkv']} KV heads "
                                f"({WL['ctx']} context, {WL['hq'] // WL['hkv']} query heads, head_dim {WL['d']}), the "
                                f"layers on layer 0's records; not extrapolated"}))


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    st = oracle_sample_setup()
    for _ in range(args.warmup):
        oracle_unit_step(st)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_unit_step(st)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    units = oracle_units()
    value = WL["batch"] * WL["ctx"] / (dt * units)
    cores = os.cpu_count() or 1
    sample = (f"each step = 1 layer x 1 KV head (4 query heads) of the {WL['ctx']}-token decode step, "
              f"extrapolated linearly x{units}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * units * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(world, args.mode, args.layout),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1400, help="timed decode steps (1400: about 1 s at batch 1)")
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--skip-quantize", action="store_true")
    p.add_argument("--step-call", default="fused", choices=["fused", "separate"],
                   help="fused: tq_decode_step (one launch per layer); separate: tq_quantize_append + "
                        "tq_decode_attention")
    p.add_argument("--mode", default="hybrid", choices=["hybrid", "full_tq"],
                   help="full_tq: no exact recent buffer, every token quantised on append")
    p.add_argument("--prefill-path", default="auto", choices=["auto", "cuda-core"],
                   help="with --prefill-chunk: cuda-core forces the decode-kernel path where tcgen05 applies")
    p.add_argument("--prefill-chunk", type=int, default=0, metavar="TQ",
                   help="time prefill attention of a TQ-token chunk instead (one JSON line of its own)")
    p.add_argument("--workload", default="llama8b", choices=sorted(WORKLOADS),
                   help="decode workload of the step: llama8b (batch 1, 32K), batched (batch 16, ragged 4K-8K, V4), "
                        "d256 (head_dim 256, batch 4, 16K), long (batch 32, 128K)")
    p.add_argument("--value-bits", type=int, default=0, choices=[0, 2, 4], help="override the workload's value bits")
    p.add_argument("--head-dim", type=int, default=128, choices=[64, 128, 256],
                   help="the same decode and prefill shapes with another head_dim (synthetic variants)")
    p.add_argument("--key-bits", type=int, default=3, choices=[3, 4],
                   help="4: 3-bit Lloyd-Max index + QJL sign with 4-bit values (the 4-bit configuration)")
    p.add_argument("--layout", default="contiguous", choices=["contiguous", "paged", "paged-ordered"],
                   help="paged: the packed pages live in a block pool addressed through a scrambled block table; "
                        "paged-ordered: the same pool with every row's blocks in allocation order")
    p.add_argument("--codec", default="", choices=["", "kivi2", "bonsai1"],
                   help="time a comparison codec over the 32K-token KV cache instead (one JSON line of its own)")
    p.add_argument("--codec-layers", type=int, default=0, help=argparse.SUPPRESS)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-nested", dest="nested", action="store_false",
                   help="skip the nested records of the other decode workloads (batched, d256, d256_v4, long) "
                        "and of the 512-query prefill")
    p.add_argument("--oracle-sample", type=int, default=0, help=argparse.SUPPRESS)
    p.add_argument("--oracle-full-step", type=int, default=0, help=argparse.SUPPRESS)
    p.add_argument("--profile-quantize", type=int, default=0, metavar="PASSES",
                   help="only run one layer of the prefill quantisation PASSES times (for profilers)")
    args = p.parse_args()
    if args.workload != "llama8b":
        WL.update(WORKLOADS[args.workload])
        args.skip_quantize = True  # the prefill quantise line belongs to the default run
    if args.value_bits:
        WL.update(vb=args.value_bits, name=WL["name"].replace(f"/V{WL['vb']}", f"/V{args.value_bits}"))
    if args.head_dim != 128:
        WL.update(d=args.head_dim, name=f"llama3.1-8b-shaped decode with head_dim {args.head_dim}, batch 1, "
                                        f"context 32768, K3/V2")
        PREFILL.update(d=args.head_dim)
    if args.key_bits == 4:
        WL.update(kb=4, vb=4, name=WL["name"].replace("K3/V2", "K4/V4"))
        PREFILL.update(kb=4, vb=4)
    if args.warmup < 3:
        args.warmup = 3
    if args.profile_quantize:
        profile_quantize(args.profile_quantize)
    elif args.prefill_chunk:
        bench_prefill(args)
    elif args.codec:
        bench_codec(args)
    elif args.oracle_sample:
        oracle_sample_main(args.oracle_sample)
    elif args.oracle_full_step:
        oracle_full_step_main(args.oracle_full_step)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
