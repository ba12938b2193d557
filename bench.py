"""Benchmark of the low-bit MLA decode hot path (qmla_append + qmla_decode).

One step = append one new token to every sequence (quantize + pack) and run
one decode over the whole cache (split-KV attention + log-sum-exp merge).
Default workload (the headline): C4R4 cache, 4 sequences of 131072 tokens,
128 heads (c4r4_b4_h128_l131072).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..4]
                  [--format C4R4|C2R4|BF16] [--impl ours|reference]
                  [--cpu-procs P] [--no-also] [--no-footprint]

Prints ONE JSON line on rank 0.  `value` is cached tokens attended per second
(sum over the sequences of the tokens each decode attends, divided by the
device time of the steps), aggregated over all ranks.  Inputs are synthetic
and seeded (bit_mla_kv_qmla_gb300/workloads.py).  `--impl reference` times the
CPU oracle on the host cores instead (all of them by default, one process
per core), on a bounded sample of the same workload.  Besides the contract's
keys the line carries `roofline` (the decode call against the measured
peaks, with the tensor-pipe activity ncu recorded for the same kernel
sources), `cpu_baseline`, `e2e` (one qmla_decode_step call per step through
the C ABI, host buffers in and out, copies inside the timed region),
`footprint_150GB` (the largest
number of 131072-token sequences a 150 GB pool holds per format, and the
decode rate measured at that concurrency), `capacity_sim` (the
cache-pressure scheduler simulation) and, unless --no-also, `also`: the
other workloads, the multi-token query decode, the folded-transform error
and the RoPE-at-INT2 comparison.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "low-bit MLA decode: cached tokens attended/s and % of roofline at 1 GPU"
UNIT = "tokens/s"
L2_BYTES = 129 * 2**20
TOKEN_BYTES = {"C4R4": 324, "C2R4": 196, "BF16": 1152, "C4R2": 308, "C2R2": 180}
FLOP_PER_TOKEN_HEAD = 2 * (576 + 512)
IO_BYTES_PER_HEAD = 576 * 2 + 512 * 2 + 4  # q in, O out, LSE out
DECODE_SOURCES = ["decode_tc.cu", "decode_tc16.cu", "decode_simt.cu", "plan.cuh",
                  "qmla_internal.cuh", "tc_common.cuh", "tc_ptx.cuh", "combine.cu"]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def decode_kernel_hash():
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        p = os.path.join(ROOT, "bit_mla_kv_qmla_gb300", "csrc", f)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def recorded_profile(workload_name):
    """The committed ncu figures of one decode launch of the workload's
    dominant kernel (DRAM bytes, tensor-pipe activity), if they were taken on
    the current decode kernel sources; else {}."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return {}
    d = json.load(open(p))
    ent = d.get(workload_name)
    if not ent or ent.get("kernel_hash") != decode_kernel_hash():
        return {}
    return ent


def recorded_traffic(workload_name):
    """DRAM bytes per decode launch from the committed ncu summary, or None."""
    return recorded_profile(workload_name).get("traffic_bytes_per_launch")


def host_cpu():
    """Model name and logical core count of the host CPU."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    import platform
    return {"model": model, "arch": platform.machine(), "logical_cores": os.cpu_count()}


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.device_index = device_index

    def start(self):
        try:
            import torch
            ident = str(self.device_index)
            try:
                u = str(torch.cuda.get_device_properties(self.device_index).uuid)
                ident = u if u.startswith("GPU-") else "GPU-" + u
            except Exception:
                pass
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", ident], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 7]
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].strip().replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[4 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def roofline_for(fmt, heads, lens, t_s, pk, traffic):
    tokens = sum(lens)
    B = len(lens)
    nbytes = tokens * TOKEN_BYTES[fmt] + B * heads * IO_BYTES_PER_HEAD
    flops = tokens * heads * FLOP_PER_TOKEN_HEAD
    t_mem = nbytes / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_tflops"] * 1e12)
    if t_mem >= t_tc:
        ach = nbytes / t_s / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / pk["hbm_gbs"], 4), "traffic": traffic,
                "algorithmic_bytes": nbytes, "peak_source": pk["source"]}
    ach = flops / t_s / 1e12
    return {"bound": "tensor", "achieved": round(ach, 1), "peak": pk["bf16_tflops"],
            "unit": "TFLOP/s", "frac": round(ach / pk["bf16_tflops"], 4), "traffic": traffic,
            "algorithmic_flops": flops, "peak_source": pk["source"],
            "peak_note": "f16 operands: same nominal dense rate as bf16"}


def step_launches(w, n_app, tc):
    """Library kernels one step launches: decode and merge; the planner
    kernel too for the 128-head kernel and for the 16-head one above 64
    sequences (it plans for itself up to there; the CUDA-core kernel always
    does); the append (advancing the lengths itself for one token, with a
    second kernel for several)."""
    k = 2
    if tc and (w.heads != 16 or w.batch > 64):
        k += 1
    if n_app == 1:
        k += 1
    elif n_app > 1:
        k += 2
    return k


# The error tables are measured with the library's quantizer: every group's
# scale and zero on its binary16-exact grid (z = Z*2^E, s = M*2^E, integers
# Z and Z + levels*M within +-2047), codes rounded half to even.
QUANTIZER_NOTE = ("binary16-exact grid per 64-channel group: z = Z*2^E, s = M*2^E "
                  "(|Z|, |Z + levels*M| <= 2047), codes round-half-even")


def append_per_step(cfg, w):
    """Tokens appended per sequence per step: one for the serving steps
    (configurations 1 and 4), the workload's own count otherwise."""
    return max(1, w.n_append) if cfg in (1, 4) else w.n_append


def run_ours(args, rank, world, device):
    import torch
    import bit_mla_kv_qmla_gb300 as q
    from bit_mla_kv_qmla_gb300 import workloads as W
    from bit_mla_kv_qmla_gb300.cache import Decoder, build_cache

    w = W.with_format(W.WORKLOADS[args.config], args.format or W.WORKLOADS[args.config].fmt)
    lens0 = W.seq_lens(w)
    n_app = append_per_step(args.config, w)
    total_steps = args.steps + args.warmup
    extra = n_app * (total_steps + 2 * args.e2e_steps + 4)
    cache_bytes = sum(W.blocks_needed(lens0, extra)) * q.qmla_block_bytes(w.fmt)
    copies = 1 if cache_bytes >= 2 * L2_BYTES else max(2, math.ceil(2 * L2_BYTES / cache_bytes))
    caches = [build_cache(w, device, extra_tokens=extra) for _ in range(copies)]
    max_len = max(lens0) + extra
    decs = [Decoder(c, w.heads, max_len) for c in caches]
    qc, qr = W.queries(w, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(1234 + rank)
    new_lat = torch.randn(copies, w.batch, max(n_app, 1), 512, generator=g, device=device)
    new_rope = torch.randn(copies, w.batch, max(n_app, 1), 64, generator=g, device=device)
    new_lat, new_rope = new_lat.to(torch.bfloat16), new_rope.to(torch.bfloat16)
    stream = torch.cuda.current_stream(device)
    torch.cuda.synchronize(device)
    for c in caches:
        assert c.status.item() == 0

    def step(k):
        i = k % copies
        if n_app:
            caches[i].append(new_lat[i, :, :n_app], new_rope[i, :, :n_app])
        decs[i](qc, qr, w.scale)

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize(device)

    # The step (append + decode, all in the library's kernels) is captured once
    # per cache copy into a CUDA graph and replayed, so the timed region
    # measures the device work, not Python/ctypes launch overhead (the e2e
    # figure below keeps that overhead).  Decode-only graphs time the decode
    # call for the roofline.
    use_graph = not args.no_graph
    if use_graph:
        g_step, g_dec = [], []
        for i in range(copies):
            gs = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gs):
                if n_app:
                    caches[i].append(new_lat[i, :, :n_app], new_rope[i, :, :n_app])
                decs[i](qc, qr, w.scale)
            g_step.append(gs)
            gd = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gd):
                decs[i](qc, qr, w.scale)
            g_dec.append(gd)
        torch.cuda.synchronize(device)
        # capturing records the work without running it; replay each step
        # graph once so every copy has run a graph step before timing
        for i in range(copies):
            g_step[i].replay()
        torch.cuda.synchronize(device)
    lens_at = [list(c.seq_lens.cpu().tolist()) for c in caches]

    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.15)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    tokens = 0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t0.record(stream)
    for k in range(args.steps):
        i = k % copies
        if n_app:
            lens_at[i] = [L + n_app for L in lens_at[i]]
        if use_graph:
            g_step[i].replay()
        else:
            if n_app:
                caches[i].append(new_lat[i, :, :n_app], new_rope[i, :, :n_app])
            e = ev[k]
            e[0].record(stream)
            decs[i](qc, qr, w.scale)
            e[1].record(stream)
        tokens += sum(lens_at[i])
    t1.record(stream)
    torch.cuda.synchronize(device)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    elapsed = t0.elapsed_time(t1) / 1e3
    if use_graph:  # decode-only replays, one event pair each, L2 rotated by the copies
        for k in range(args.steps):
            e = ev[k]
            e[0].record(stream)
            g_dec[k % copies].replay()
            e[1].record(stream)
        torch.cuda.synchronize(device)
    t_dec = statistics.mean(a.elapsed_time(b) for a, b in ev) / 1e3
    for c in caches:
        assert c.status.item() == 0, "device status flag set during the benchmark"

    # End to end through the public API with host buffers: per step one call
    # of qmla_decode_step (C ABI) from a page-locked host buffer holding that
    # step's inputs (new tokens and queries, different for every step) to a
    # page-locked host buffer receiving O and LSE: inside the call one host ->
    # device copy, the append and length update, the decode (planner, decode,
    # merge), one device -> host copy, and the wait for it.
    e2e = None
    if args.e2e_steps > 0:
        n_sets = args.e2e_steps + 3
        lay = q.qmla_decode_step_layout(w.batch, w.heads, n_app)
        h_ins = []
        for k in range(n_sets):
            qck, qrk = W.queries(w, step=k + 1)
            srcs = [(lay[2], qck), (lay[3], qrk)]
            if n_app:
                lat = torch.stack([W.tokens(w, b, n_app, offset_seed=10_000 + k)[0]
                                   for b in range(w.batch)])
                rope = torch.stack([W.tokens(w, b, n_app, offset_seed=10_000 + k)[1]
                                    for b in range(w.batch)])
                srcs = [(lay[0], lat), (lay[1], rope)] + srcs
            h = torch.zeros(lay[4], dtype=torch.uint8).pin_memory()
            for o, t in srcs:
                raw = t.contiguous().reshape(-1).view(torch.uint8)
                h[o:o + raw.numel()].copy_(raw)
            h_ins.append(h)
        h_out = torch.empty(lay[7], dtype=torch.uint8).pin_memory()
        ws_step = [torch.empty(q.qmla_decode_step_workspace_bytes(w.fmt, w.batch, w.heads, n_app,
                                                                  d.max_seq_len),
                               dtype=torch.uint8, device=device) for d in decs]
        h2d = lay[4]
        d2h = lay[7]

        def e2e_step(k):
            i = k % copies
            c = caches[i]
            q.qmla_decode_step(w.fmt, c.blocks, c.block_table, c.seq_lens, decs[i].max_seq_len,
                               w.heads, n_app, h_ins[k], w.scale, h_out, ws_step[i], c.status,
                               stream)

        for k in range(3):
            e2e_step(k)
            lens_at[k % copies] = [L + n_app for L in lens_at[k % copies]]
        tok_e2e = 0
        s0 = time.perf_counter()
        for k in range(3, n_sets):
            e2e_step(k)
            i = k % copies
            lens_at[i] = [L + n_app for L in lens_at[i]]
            tok_e2e += sum(lens_at[i])
        e2e_t = time.perf_counter() - s0
        e2e = {"value": tok_e2e / e2e_t, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
               "ms_per_step": 1e3 * e2e_t / args.e2e_steps,
               "issue": "one qmla_decode_step call per step: page-locked host buffers in and "
                        "out, fresh inputs every step"}

    lens_mid = [L for L in lens_at[0]]
    pk = peaks()
    prof = recorded_profile(w.name)
    roof = roofline_for(w.fmt, w.heads, lens_mid, t_dec, pk, prof.get("traffic_bytes_per_launch"))
    roof["decode_ms"] = round(t_dec * 1e3, 5)
    if prof.get("tensor_pipe_active_pct") is not None:
        # ncu's sm__pipe_tensor_cycles_active of the same kernel sources (one
        # launch, profiles/), next to the achieved fraction of the peak
        roof["tensor_pipe_active_pct"] = prof["tensor_pipe_active_pct"]
        roof["dram_throughput_pct"] = prof.get("dram_throughput_pct")
    tc = w.heads in (16, 128) and w.fmt in ("C4R4", "C2R4", "BF16")
    roof["kernel"] = ((f"decode_tc{w.heads} (tcgen05"
                       + (", plans its own pieces)" if w.heads == 16 and w.batch <= 64
                          else ") + plan") + " + combine") if tc else
                      "decode_simt (CUDA cores) + combine") + ", CUDA events per qmla_decode call"
    res = {"tokens": tokens, "elapsed": elapsed, "t_dec": t_dec, "roofline": roof,
           "dtype": "f16" if tc else "f32",
           "clocks": clocks, "e2e": e2e, "workload": w, "copies": copies,
           "cache_bytes": cache_bytes,
           "launches": args.steps * step_launches(w, n_app, tc),
           "graph": use_graph}
    return res


def measure_also(args, device):
    """Device-timed decode of the other workloads and formats (decode only,
    median of 10 calls with L2 flushed between them), for context."""
    import torch
    from bit_mla_kv_qmla_gb300 import workloads as W
    from bit_mla_kv_qmla_gb300.cache import Decoder, build_cache
    out = {}
    pk = peaks()
    head = (args.config, args.format or W.WORKLOADS[args.config].fmt)
    runs = [(1, "C4R4"), (1, "BF16"), (4, "C4R4"), (4, "C2R4"), (4, "BF16"), (2, "C4R4"),
            (3, "C2R4")]
    for cfg, fmt in [r for r in runs if r != head]:
        w = W.with_format(W.WORKLOADS[cfg], fmt)
        lens = W.seq_lens(w)
        cache = build_cache(w, device)
        dec = Decoder(cache, w.heads, max(lens))
        qc, qr = W.queries(w, device=device)
        for _ in range(3):
            dec(qc, qr, w.scale)
        torch.cuda.synchronize(device)
        n = 10
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n)]
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
        for a, b in evs:
            flush.fill_(1.0)  # evict the cache from L2 between calls (untimed)
            a.record()
            dec(qc, qr, w.scale)
            b.record()
        torch.cuda.synchronize(device)
        assert cache.status.item() == 0
        t = statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3
        roof = roofline_for(fmt, w.heads, lens, t, pk, recorded_traffic(w.name))
        out[w.name] = {"tokens_per_s": sum(lens) / t, "decode_us": round(t * 1e6, 2),
                       "roofline": {k: roof[k] for k in ("bound", "achieved", "unit", "frac")},
                       "cache_bytes": cache.blocks.numel()}
        del cache, dec, flush
        torch.cuda.empty_cache()
    out.update(measure_multi(device, pk))
    out.update(measure_fold(device))
    out.update(measure_rope_bits(device))
    return out


def measure_fold(device):
    """Error of the low-bit decode with and without an orthogonal transform
    folded into the content latent and query (c R, q_c R; the output rotated
    back), on 8 x 2048-token sequences whose latents have 1% of the channels
    at 10x gain.  Reference: the BF16-cache decode of the unrotated tokens.
    Reported: mean |dLSE| and RMS output error relative to the reference's
    RMS, for C4R4 and C2R4."""
    import torch
    from bit_mla_kv_qmla_gb300 import workloads as W
    from bit_mla_kv_qmla_gb300.cache import Decoder, PagedCache
    R = W.orthogonal(512, 3).to(device)
    res = {}
    ref = None
    for fmt in ("BF16", "C4R4", "C2R4"):
        w = W.Workload(f"fold_{fmt}", fmt, 8, 16, 2048, 0, "x10pct1", 0, 5)
        lens = W.seq_lens(w)
        table, nblocks = W.block_table(w, lens)
        qc, qr = W.queries(w, device=device)
        row = {}
        for rot in ((False,) if fmt == "BF16" else (False, True)):
            cache = PagedCache(fmt, table, nblocks, device)
            for b, L in enumerate(lens):
                lat, rope = W.tokens(w, b, L, device=device)
                cache.append_seq(b, W.rotate(lat, R) if rot else lat, rope)
            out, lse = Decoder(cache, 16, max(lens))(W.rotate(qc, R) if rot else qc, qr, w.scale)
            o = out.double() @ R.T if rot else out.double()
            if fmt == "BF16":
                ref = (o, lse.double())
                continue
            rms = torch.sqrt(((o - ref[0]) ** 2).mean() / (ref[0] ** 2).mean()).item()
            dl = (lse.double() - ref[1]).abs().mean().item()
            row["rotated" if rot else "plain"] = {"mean_abs_dlse": round(dl, 5),
                                                  "rel_rms_dO": round(rms, 5)}
            del cache
        if row:
            res[fmt] = row
    torch.cuda.empty_cache()
    res["quantizer"] = QUANTIZER_NOTE
    return {"folded_rotation_error_b8_h16_l2048_x10pct1": res}


def measure_rope_bits(device):
    """The equal-bits comparison: the RoPE key at INT4 (C4R4, C2R4) against
    INT2 (C4R2, C2R2), as a generic quantizer that gives both halves of the
    cache one bit width would store it.  Synthetic latents with 1% of the
    channels at 10x gain, N(0, 1) RoPE keys and queries, 16 heads.
    * score error: 4096 one-token sequences, so that each LSE is exactly that
      token's score (natural-log units, scale included); the content path
      alone (q_r = 0), the RoPE path alone (q_c = 0) and both, as RMS of the
      difference to the BF16-cache scores;
    * decode error: 8 x 2048-token sequences, mean |dLSE| and the RMS output
      error relative to the BF16-cache decode's RMS.
    The INT2-RoPE formats run on the CUDA-core decode kernel."""
    import torch
    from bit_mla_kv_qmla_gb300 import qmla_block_bytes
    from bit_mla_kv_qmla_gb300 import workloads as W
    from bit_mla_kv_qmla_gb300.cache import Decoder, PagedCache
    fmts = ("BF16", "C4R4", "C4R2", "C2R4", "C2R2")
    # scores: B one-token sequences
    w1 = W.Workload("ropebits_l1", "BF16", 4096, 16, 1, 0, "x10pct1", 0, 6)
    lat, rope = W.tokens(w1, 0, w1.batch, device=device)
    qc, qr = W.queries(w1, device=device)
    variants = {"both": (qc, qr), "content_path": (qc, torch.zeros_like(qr)),
                "rope_path": (torch.zeros_like(qc), qr)}
    table, nblocks = W.block_table(w1, [1] * w1.batch)
    scores = {}
    for fmt in fmts:
        cache = PagedCache(fmt, table, nblocks, device)
        cache.append(lat[:, None].contiguous(), rope[:, None].contiguous())
        dec = Decoder(cache, 16, 1)
        scores[fmt] = {k: dec(a, b, w1.scale)[1].double().clone() for k, (a, b) in variants.items()}
        assert int(cache.status.item()) == 0
        del cache, dec
    score_err = {}
    for fmt in fmts[1:]:
        score_err[fmt] = {k: round(torch.sqrt(((scores[fmt][k] - scores["BF16"][k]) ** 2)
                                              .mean()).item(), 5) for k in variants}
    score_rms = {k: round(torch.sqrt((scores["BF16"][k] ** 2).mean()).item(), 4)
                 for k in variants}
    # attention outputs
    dec_err, ref = {}, None
    for fmt in fmts:
        w = W.Workload(f"ropebits_{fmt}", fmt, 8, 16, 2048, 0, "x10pct1", 0, 5)
        lens = W.seq_lens(w)
        t2, nb2 = W.block_table(w, lens)
        q2c, q2r = W.queries(w, device=device)
        cache = PagedCache(fmt, t2, nb2, device)
        for b, L in enumerate(lens):
            cache.append_seq(b, *W.tokens(w, b, L, device=device))
        out, lse = Decoder(cache, 16, max(lens))(q2c, q2r, w.scale)
        o, l = out.double(), lse.double()
        if fmt == "BF16":
            ref = (o, l)
        else:
            dec_err[fmt] = {
                "mean_abs_dlse": round((l - ref[1]).abs().mean().item(), 5),
                "rel_rms_dO": round(torch.sqrt(((o - ref[0]) ** 2).mean()
                                               / (ref[0] ** 2).mean()).item(), 5)}
        del cache
    torch.cuda.empty_cache()
    return {"rope_bits_ablation_h16_x10pct1": {
        "quantizer": QUANTIZER_NOTE,
        "bytes_per_token": {f: qmla_block_bytes(f) // 64 for f in fmts},
        "score_rms_bf16_l1_b4096": score_rms,
        "score_rms_error_l1_b4096": score_err,
        "decode_error_b8_l2048": dec_err}}


def measure_multi(device, pk):
    """Multi-token query decode (qmla_decode_multi) on the 32 x 8K C4R4 cache
    with 16 heads and 8 query tokens per sequence: 128 query rows per
    sequence on the 128-head tensor-core kernel.  tokens_per_s counts every
    query's visible tokens; the roofline counts the cache once and the
    tensor work of every (query row, visible token)."""
    import torch
    from bit_mla_kv_qmla_gb300 import workloads as W
    from bit_mla_kv_qmla_gb300.cache import Decoder, build_cache
    w = W.WORKLOADS[1]
    q_len = 8
    lens = W.seq_lens(w)
    cache = build_cache(w, device)
    dec = Decoder(cache, w.heads, max(lens), q_len=q_len)
    g = torch.Generator(device=device)
    g.manual_seed(77)
    qc = torch.randn(w.batch, q_len, w.heads, 512, generator=g, device=device).to(torch.bfloat16)
    qr = torch.randn(w.batch, q_len, w.heads, 64, generator=g, device=device).to(torch.bfloat16)
    for _ in range(3):
        dec(qc, qr, w.scale)
    torch.cuda.synchronize(device)
    n = 10
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
    for a, b in evs:
        flush.fill_(1.0)
        a.record()
        dec(qc, qr, w.scale)
        b.record()
    torch.cuda.synchronize(device)
    assert cache.status.item() == 0
    t = statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3
    seen = sum(max(0, L - (q_len - 1 - i)) for L in lens for i in range(q_len))
    flops = seen * w.heads * FLOP_PER_TOKEN_HEAD
    bytes_alg = sum(lens) * TOKEN_BYTES["C4R4"] + w.batch * q_len * w.heads * IO_BYTES_PER_HEAD
    t_mem = bytes_alg / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_tflops"] * 1e12)
    roof = ({"bound": "tensor", "achieved": round(flops / t / 1e12, 1), "unit": "TFLOP/s"}
            if t_tc > t_mem else
            {"bound": "hbm", "achieved": round(bytes_alg / t / 1e9, 1), "unit": "GB/s"})
    roof["frac"] = round(max(t_mem, t_tc) / t, 4)
    res = {"tokens_per_s": seen / t, "decode_us": round(t * 1e6, 2), "q_len": q_len,
           "query_rows": w.heads * q_len, "roofline": roof}
    del cache, dec, flush
    torch.cuda.empty_cache()
    return {f"c4r4_b32_h16x{q_len}_l8192_multiquery": res}


def footprint_decode(device, budget=150e9, seq_len=131072, heads=128):
    """The 150 GB footprint sweep, measured.  Per format: the largest number N
    of seq_len-token sequences whose blocks fit the budget; a pool of exactly
    those N x seq_len/64 blocks is filled from library-written blocks (one
    sequence appended through qmla_append, its blocks then replicated with
    device-to-device copies, one cudaMemcpyAsync per chunk of at most 4 GB),
    and a 128-head decode over all N sequences is timed (median of 3, CUDA
    events).  Reported: N, decode tokens/s (N sequences / step time) and
    cached tokens attended/s.  If the device cannot hold the budget plus the
    decode's buffers, the budget is lowered to what it can hold and stated."""
    import torch
    import bit_mla_kv_qmla_gb300 as q
    from bit_mla_kv_qmla_gb300 import workloads as W
    from bit_mla_kv_qmla_gb300.cache import Decoder, PagedCache
    w4 = W.WORKLOADS[4]
    nblk = seq_len // 64
    free, total = torch.cuda.mem_get_info(device)
    # decode buffers: queries, O and the split partials are a few GB at most
    obtained = min(budget, free - 12e9)
    per_seq = {f: nblk * q.qmla_block_bytes(f) for f in ("BF16", "C4R4", "C2R4")}
    n_max = {f: int(budget // per_seq[f]) for f in per_seq}
    res = {"budget_bytes": int(budget), "budget_obtained_bytes": int(obtained),
           "seq_len": seq_len, "heads": heads, "bytes_per_seq": per_seq,
           "max_sequences": n_max,
           "gain_vs_bf16": {f: round(n_max[f] / n_max["BF16"], 3) for f in n_max},
           "measured": {}}
    for f in ("C4R4", "C2R4", "BF16"):
        n = int(obtained // per_seq[f])
        if n < 1:
            continue
        table = torch.arange(n * nblk, dtype=torch.int32).view(n, nblk)
        cache = PagedCache(f, table, n * nblk, device)
        lat, rope = W.tokens(w4, 0, seq_len, device=device)
        cache.append_seq(0, lat, rope)
        del lat, rope
        seg = nblk * cache.block_bytes
        chunk = max(1, int(4e9 // seg))
        filled = 1
        while filled < n:
            k = min(filled, n - filled, chunk)
            cache.blocks[filled * seg:(filled + k) * seg].copy_(cache.blocks[:k * seg])
            filled += k
        cache.seq_lens.fill_(seq_len)
        g = torch.Generator(device=device)
        g.manual_seed(4242)
        qc = torch.randn(n, heads, W.D_C, generator=g, device=device).to(torch.bfloat16)
        qr = torch.randn(n, heads, W.D_R, generator=g, device=device).to(torch.bfloat16)
        dec = Decoder(cache, heads, seq_len)
        for _ in range(2):
            dec(qc, qr, w4.scale)
        torch.cuda.synchronize(device)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(3)]
        for a, b in evs:
            a.record()
            dec(qc, qr, w4.scale)
            b.record()
        torch.cuda.synchronize(device)
        assert int(cache.status.item()) == 0, "device status flag set in the footprint decode"
        t = statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3
        res["measured"][f] = {"sequences": n, "pool_bytes": n * seg, "decode_ms": round(t * 1e3, 3),
                              "decode_tokens_per_s": round(n / t, 1),
                              "tokens_attended_per_s": n * seq_len / t}
        del cache, dec, qc, qr, table
        torch.cuda.empty_cache()
    m = res["measured"]
    if "BF16" in m:
        res["decode_tokens_per_s_vs_bf16"] = {
            f: round(m[f]["decode_tokens_per_s"] / m["BF16"]["decode_tokens_per_s"], 3) for f in m}
    return res


def capacity_sweep(rates):
    """The cache-pressure mechanism behind the pages' whole-job result,
    replayed by bit_mla_kv_qmla_gb300.capacity: 512 requests with prompts
    uniform in [8K, 128K] tokens and 1024 generated tokens each, at most 256
    running, cache budgets of 8, 16 and 32 GB.  Per format and budget:
    preemptions, tokens recomputed on readmission, decode steps and mean
    running sequences; and, where this run measured the format's decode rate
    on the matching shape (128 heads, 131072-token sequences, the footprint
    decode), the job's decode time at that rate (tokens attended / rate)."""
    import bit_mla_kv_qmla_gb300 as q
    from bit_mla_kv_qmla_gb300 import capacity as C
    reqs = C.synthetic_requests(512, 8192, 131072, 1024, seed=1)
    out = {}
    for gb in (8, 16, 32):
        row = {}
        for f in ("BF16", "C4R4", "C2R4"):
            r = C.simulate(q.qmla_block_bytes(f), gb * 10 ** 9, reqs, 256)
            ent = {k: r[k] for k in ("preemptions", "recomputed_tokens", "steps")}
            ent["mean_running"] = round(r["mean_running"], 1)
            if rates.get(f):
                ent["decode_s_at_measured_rate"] = round(r["attended_tokens"] / rates[f], 3)
            row[f] = ent
        out[f"{gb}GB"] = row
    return {"requests": "512, prompts U[8192, 131072], 1024 generated, <= 256 running",
            "rates_tokens_attended_per_s": {f: round(v) for f, v in rates.items() if v},
            "rate_shape": "128 heads, 131072-token sequences, decode at the 150 GB footprint",
            "by_budget": out}


# ---------------------------------------------------------------------------
# CPU oracle arm (reference and cpu_baseline)
# ---------------------------------------------------------------------------

class OracleRunner:
    """The oracle's step (append one token to each sampled sequence, then
    decode them) on the host, single-threaded, for sequences first ..
    first+n_seq-1 and heads h0 .. h0+n_heads-1 of the workload.  A step's
    tokens attended are counted in whole-decode units: the sampled
    sequences' lengths times n_heads / heads (every head attends every
    token, so a head subset is that fraction of the decode's work)."""

    def __init__(self, cfg, fmt, n_seq, max_steps, first=0, h0=0, n_heads=None):
        import numpy as np
        import oracle
        from bit_mla_kv_qmla_gb300 import workloads as W
        self.np, self.oracle, self.W = np, oracle, W
        self.w = w = W.with_format(W.WORKLOADS[cfg], fmt)
        self.n_seq = n_seq
        self.first = first
        self.n_heads = w.heads if n_heads is None else n_heads
        lens = W.seq_lens(w)[first:first + n_seq]
        self.f = W.FORMATS[w.fmt]
        need = [(L + max_steps + 1 + 63) // 64 for L in lens]
        self.table = np.full((n_seq, max(need)), -1, np.int32)
        k = 0
        for b, n in enumerate(need):
            self.table[b, :n] = np.arange(k, k + n)
            k += n
        self.pool = np.zeros(k * oracle.block_bytes(self.f), np.uint8)
        for b, L in enumerate(lens):
            lat, rope = W.tokens(w, first + b, L)
            oracle.append(self.f, self.pool, self.table[b:b + 1], np.array([0], np.int32),
                          lat[None], rope[None])
        qc, qr = W.queries(w)
        hs = slice(h0, h0 + self.n_heads)
        self.qc = qc[first:first + n_seq, hs].contiguous()
        self.qr = qr[first:first + n_seq, hs].contiguous()
        self.cur = np.array(lens, np.int32)
        self.s = 0
        self.sample = (f"{n_seq} of {w.batch} sequences x {self.n_heads} of {w.heads} heads "
                       "per step")

    def step(self):
        self.s += 1
        # each sequence's appended token from its own stream, so that any
        # split of the sequences over processes appends the same data
        import torch
        toks = [self.W.tokens(self.w, self.first + b, 1, offset_seed=self.s)
                for b in range(self.n_seq)]
        lat = torch.stack([t[0] for t in toks])
        rope = torch.stack([t[1] for t in toks])
        self.oracle.append(self.f, self.pool, self.table, self.cur, lat, rope)
        self.cur = self.cur + 1
        self.oracle.decode(self.f, self.pool, self.table, self.cur, self.qc, self.qr, self.w.scale)
        return float(self.cur.sum()) * self.n_heads / self.w.heads


def _oracle_worker(args):
    """One process of the multi-core oracle timing: its own runner over its
    own (sequences, heads) unit, timed between two barriers."""
    import torch
    torch.set_num_threads(1)  # one core per process (input generation included)
    cfg, fmt, n_seq, first, h0, n_heads, steps, warmup, barrier = args
    r = OracleRunner(cfg, fmt, n_seq, steps + warmup, first=first, h0=h0, n_heads=n_heads)
    for _ in range(warmup):
        r.step()
    barrier.wait()
    tokens, t0 = 0.0, time.perf_counter()
    for _ in range(steps):
        tokens += r.step()
    return tokens, time.perf_counter() - t0


def oracle_sample_shape(cfg):
    """Per-process sample of the oracle timing: (sequences, heads).  Sized so
    one step is about a second of single-core work."""
    return {1: (2, 16), 2: (1, 32), 3: (1, 32), 4: (1, 8)}.get(cfg, (1, 16))


def oracle_multicore(cfg, fmt, procs, steps, warmup):
    """The oracle's step over procs disjoint (sequences, heads) units of the
    workload, one process each (started with spawn), all timed together.
    Returns (tokens attended / the slowest process's time, that time, the
    units' description)."""
    import multiprocessing as mp
    from bit_mla_kv_qmla_gb300 import workloads as W
    w = W.WORKLOADS[cfg]
    n_seq, n_heads = oracle_sample_shape(cfg)
    units = [(b, h) for h in range(0, w.heads, n_heads) for b in range(0, w.batch, n_seq)]
    procs = max(1, min(procs, len(units)))
    jobs = [(cfg, fmt, n_seq, units[p][0], units[p][1], n_heads, steps, warmup)
            for p in range(procs)]
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        barrier = mgr.Barrier(procs)
        with ctx.Pool(procs) as pool:
            res = pool.map(_oracle_worker, [j + (barrier,) for j in jobs])
    tokens = sum(r[0] for r in res)
    t = max(r[1] for r in res)
    desc = (f"{procs} processes, each {n_seq} of {w.batch} sequences x {n_heads} of {w.heads} "
            "heads (disjoint units), tokens attended counted as that fraction of a decode")
    return tokens / t, t, desc, procs


def cpu_baseline(cfg, fmt):
    """The oracle timed on one core on a bounded sample (about 10 s of host
    work after building the sample's cache)."""
    n_seq, n_heads = {1: (8, 16), 4: (1, 16)}.get(cfg, (1, 16))
    r = OracleRunner(cfg, fmt, n_seq=n_seq, max_steps=64, n_heads=n_heads)
    tokens, t0 = 0.0, time.perf_counter()
    steps = 0
    while steps < 64 and (time.perf_counter() - t0 < 10.0 or steps < 1):
        tokens += r.step()
        steps += 1
    dt = time.perf_counter() - t0
    return {"value": tokens / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"{r.sample}, {steps} step(s), {dt:.1f} s; tokens attended counted "
                       f"as {n_heads}/{r.w.heads} of a decode per sequence"),
            "cpu": host_cpu()}


# ---------------------------------------------------------------------------

def aggregate_ranks(elapsed, tokens, world, device):
    """Whole-job figures of a weak-scaling run: each rank decodes its own
    batch (no data-path collective), so the job takes the slowest rank's time
    and processes the sum of the ranks' tokens."""
    if world <= 1:
        return elapsed, tokens
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor([tokens], dtype=torch.float64, device=device)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=4, choices=[1, 2, 3, 4])
    ap.add_argument("--format", default=None, choices=["C4R4", "C2R4", "BF16"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-procs", type=int, default=0,
                    help="--impl reference: time the oracle in this many processes "
                         "(0: one per host core)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-also", action="store_true")
    ap.add_argument("--no-footprint", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch each timed step's calls eagerly instead of replaying a CUDA graph")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        from bit_mla_kv_qmla_gb300 import workloads as W
        w = W.with_format(W.WORKLOADS[args.config], args.format or W.WORKLOADS[args.config].fmt)
        procs = args.cpu_procs if args.cpu_procs > 0 else (os.cpu_count() or 1)
        v, t_all, sample, procs = oracle_multicore(args.config, w.fmt, procs, args.steps,
                                                   args.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 0,
                "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * t_all / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": w.name, "format": w.fmt, "batch": w.batch,
                           "heads": w.heads, "seq_len": w.seq_len,
                           "append_per_step": append_per_step(args.config, w)},
                "cpu_baseline": {"value": v, "unit": UNIT, "cores": procs, "kind": "oracle",
                                 "sample": sample, "cpu": host_cpu()},
                "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import __graft_entry__
    __graft_entry__.build()

    res = run_ours(args, rank, world, device)
    el, tok = aggregate_ranks(float(res["elapsed"]), float(res["tokens"]), world, device)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    w = res["workload"]
    torch.cuda.empty_cache()
    also = None if args.no_also or world > 1 else measure_also(args, device)
    foot = None if args.no_footprint or world > 1 else footprint_decode(device)
    rates = {f: m["tokens_attended_per_s"] for f, m in (foot or {}).get("measured", {}).items()}
    line = {
        "metric": METRIC, "value": tok / el, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": res["dtype"], "data": "synthetic (seeded, bit_mla_kv_qmla_gb300/workloads.py)",
        "config": {"workload": w.name, "format": w.fmt, "batch": w.batch, "heads": w.heads,
                   "seq_len": w.seq_len, "append_per_step": append_per_step(args.config, w),
                   "launch": ("CUDA graph replay of each step's library calls" if res["graph"]
                              else "eager library calls"),
                   "l2": (f"rotating {res['copies']} cache copies of "
                          f"{res['cache_bytes'] / 1e6:.0f} MB (> L2 129 MB in total)"
                          if res["copies"] > 1 else "cache larger than L2")},
        "roofline": res["roofline"],
        "cpu_baseline": None if args.no_cpu_baseline else cpu_baseline(args.config, w.fmt),
        "e2e": res["e2e"],
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "footprint_150GB": foot,
        "capacity_sim": capacity_sweep(rates),
        "also": also,
    }
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
