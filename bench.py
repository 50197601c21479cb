"""Benchmark: MLA decode tokens/s and latent-KV HBM GB/s on one GB300.

Default workload: DeepSeek-V3-shaped decode, B=32 sequences x context 4096,
H=128 heads, page 64, one query token per sequence (seeded synthetic data,
random weights). One step = mla_decode_plan -> mla_absorb_q ->
mla_decode_paged_planned -> mla_combine -> mla_out_proj for the whole batch
(the split plan is computed beside the previous kernel); tokens/s = query
tokens per step / step time. Steps run back to back (CUDA graphs of consecutive steps) over three
complete input sets at distinct addresses used in rotation, so every step reads
inputs that are no longer in L2 (the sets together are ~4.5x the L2); the timed
region is bracketed by CUDA events on the launching stream. The JSON line also
carries per-call phase times (each call back to back over the same rotation),
the decode call's roofline, one step replayed alone after an L2 flush, and the
end-to-end rate through the Python API with host copies.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs the same per-GPU batch on its own GPU (replicas,
weak scaling, no data-path collective); rank 0 prints one JSON line with the
max-over-ranks time. ``--impl reference`` times the CPU oracle (fp32 absorbed
loops) on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import mla_inputs as mi  # noqa: E402

METRIC = "MLA decode tokens/s & latent-KV HBM GB/s (% of GB300 roofline), 1 GPU"
UNIT = "tokens/s"
WORKLOAD_INDEX = 2
NSETS = 3        # rotating input sets in the timed region
D_MODEL = 7168   # hidden width of the cache-append phase (DeepSeek-V3)
D_Q = 1536       # compressed query width of the query-side absorption line (DeepSeek-V3's; the pages leave it open)
ROTATIONS = 10   # passes over the sets per graph replay


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def roofline_bound(flops: float, nbytes: float, us: float, hbm_gbs: float, tflops: float) -> dict:
    """The roofline a kernel sits under: HBM below the ridge point of the peaks (flops per
    byte at which both take the same time), the tensor pipe above it."""
    intensity = flops / nbytes
    gbs = nbytes / (us * 1e-6) / 1e9
    if intensity <= tflops * 1e12 / (hbm_gbs * 1e9):
        out = {"bound": "hbm", "achieved": gbs, "peak": hbm_gbs, "unit": "GB/s", "frac": gbs / hbm_gbs}
    else:
        tf = flops / (us * 1e-6) / 1e12
        out = {"bound": "tensor", "achieved": tf, "peak": tflops, "unit": "TFLOP/s", "frac": tf / tflops,
               "hbm_gbs_achieved": gbs}
    out["flop_per_byte"] = intensity
    return out


def max_over_ranks(x: float, dist, device) -> float:
    """The largest x over the ranks of the process group (x itself without one)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world: int, tokens_per_rank_step: int, steps: int, total_s: float) -> float:
    """Whole-job tokens/s of replicas: every rank runs its own batch (weak scaling),
    so all ranks' tokens over the slowest rank's time."""
    return world * tokens_per_rank_step * steps / total_s


def cpu_baseline(inp, budget_s: float = 12.0, max_seqs: int | None = None):
    """Time the oracle's fp32 absorbed path on whole sequences (all heads) of ``inp``."""
    import oracle
    oracle.build()
    H, n_q = inp.H, inp.n_q
    seqs_done, t_total, reps = 0, 0.0, 0
    order = list(range(inp.B))
    while t_total < budget_s and (max_seqs is None or seqs_done < max_seqs):
        b = order[reps % inp.B]
        rows = np.arange(b * n_q * H, (b + 1) * n_q * H, dtype=np.int64)
        t0 = time.perf_counter()
        oracle.absorbed_f32(inp, rows)
        t_total += time.perf_counter() - t0
        seqs_done += 1
        reps += 1
    tokens = seqs_done * n_q
    return {"value": tokens / t_total, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{seqs_done} whole sequences x {H} heads (fp32 absorbed loops, same workload)",
            "seconds": round(t_total, 3)}


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    inp = mi.workload_inputs(args.workload)
    T = inp.B * inp.n_q
    per_step = max(1, min(inp.B, 4))
    times = []
    steps = args.warmup + args.steps
    import oracle
    oracle.build()
    for s in range(steps):
        seqs = [(s * per_step + i) % inp.B for i in range(per_step)]
        rows = np.concatenate([np.arange(b * inp.n_q * inp.H, (b + 1) * inp.n_q * inp.H) for b in seqs])
        t0 = time.perf_counter()
        oracle.absorbed_f32(inp, rows.astype(np.int64))
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
    tok = per_step * inp.n_q
    value = tok * len(times) / sum(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(inp, None),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{per_step} whole sequences (all {inp.H} heads) per step of the "
                                   f"B={inp.B} batch"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(inp, num_splits):
    lens = inp.seq_lens
    ctx = (f"context {int(lens[0])}" if (lens == lens[0]).all()
           else f"contexts {int(lens.min())}..{int(lens.max())} (mean {float(lens.mean()):.0f})")
    return {"workload": f"DeepSeek-V3-shaped MLA decode: B={inp.B} x {ctx}, H={inp.H}, d_c=512, d_r=64, "
                        f"page 64, n_q={inp.n_q}",
            "batch": inp.B, "context": int(lens[0]) if (lens == lens[0]).all() else float(lens.mean()),
            "heads": inp.H, "n_q": inp.n_q,
            "page_size": 64, "num_splits": num_splits, "cache_bytes": int(inp.seq_lens.sum()) * 1152,
            "l2": f"inputs larger than L2: {NSETS} rotating input sets of ~190 MB (latent cache, weights, "
                  "queries, tables), steps back to back, no flush"}


def run_ours(args):
    import torch
    import mla_latent_kv_paged_gb300 as mla

    ws_, rank, local = dist_env()
    dist = None
    if ws_ > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    mla.build()

    inp = mi.workload_inputs(args.workload)
    pg = mi.make_paged(inp, spare_pages=mi.WORKLOADS[args.workload].spare_pages)
    T, H, B, n_q = inp.B * inp.n_q, inp.H, inp.B, inp.n_q

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    G = mla.default_splits(n_q)
    # NSETS complete input sets (queries, weights, latent cache, block table,
    # lengths, work buffers) at distinct addresses, used in rotation: a step
    # touches ~190 MB, so the set a step reads was last touched NSETS - 1 steps
    # (~380 MB of other traffic) earlier and is no longer in the 126 MB L2.
    # Consecutive steps run back to back, as consecutive layers of a serving
    # loop would; no L2 flush is needed between them.
    rng = np.random.default_rng(7168)
    h_bits = mi.f32_to_bf16(rng.standard_normal((T, D_MODEL)).astype(np.float32))
    w_dkr_bits = mi.f32_to_bf16((rng.standard_normal((576, D_MODEL)) / np.sqrt(D_MODEL)).astype(np.float32))
    c_q_bits, w_uq_bits = mi.latent_query_inputs(T, H, D_Q, seed=1536)
    w_uq_dev = to_dev(w_uq_bits)
    w_o_dev = to_dev(mi.output_projection(D_MODEL, H, seed=7169))
    sets = []
    for _ in range(NSETS):
        sets.append(dict(
            h=to_dev(h_bits), w_dkr=to_dev(w_dkr_bits),
            ws_app=torch.zeros(mla.append_workspace_bytes(T, D_MODEL), dtype=torch.uint8, device=dev),
            q_nope=to_dev(inp.q_nope.reshape(T, H, -1)), q_rope=to_dev(inp.q_rope.reshape(T, H, -1)),
            w_uk=to_dev(inp.w_uk), w_uv=to_dev(inp.w_uv), cache=to_dev(pg.cache),
            bt=torch.from_numpy(pg.block_table).to(dev), sl=torch.from_numpy(inp.seq_lens).to(dev),
            q_abs=torch.empty((T, H, 576), dtype=torch.bfloat16, device=dev),
            workspace=torch.empty(mla.workspace_bytes(B, n_q, H, G), dtype=torch.uint8, device=dev),
            u=torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev),
            lse=torch.empty((T, H), dtype=torch.float32, device=dev),
            out=torch.empty((T, H, 128), dtype=torch.bfloat16, device=dev),
            c_q=to_dev(c_q_bits)))
        sets[-1]["w_kq"] = mla.merge_w_kq(w_uq_dev, sets[-1]["w_uk"])
        sets[-1]["w_comb"] = mla.merge_w_comb(sets[-1]["w_uv"], w_o_dev)
        sets[-1]["ws_comb"] = torch.empty(mla.out_comb_workspace_bytes(T, H, D_MODEL), dtype=torch.uint8, device=dev)
        sets[-1]["out_model"] = torch.empty((T, D_MODEL), dtype=torch.bfloat16, device=dev)
    del w_uq_dev, w_o_dev
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def absorb(S):
        mla.absorb_q(S["q_nope"], S["q_rope"], S["w_uk"], S["q_abs"])

    def decode(S):  # the plan and the split-KV decode kernel in one call
        mla.decode_paged(S["q_abs"], S["cache"], S["bt"], S["sl"], n_q=n_q, num_splits=G,
                         workspace=S["workspace"], err_word=err)

    def plan(S):  # the split plan alone (in the step: enqueued before absorb_q)
        mla.decode_plan(S["sl"], n_q=n_q, H=H, max_pages=pg.max_pages, num_pages=pg.num_pages, num_splits=G,
                        workspace=S["workspace"], err_word=err)

    def decode_planned(S):  # the split-KV decode kernel alone, on the workspace's plan
        mla.decode_paged(S["q_abs"], S["cache"], S["bt"], S["sl"], n_q=n_q, num_splits=G,
                         workspace=S["workspace"], err_word=err, planned=True)

    def combine(S):
        mla.combine(S["workspace"], B=B, n_q=n_q, H=H, num_splits=G, u=S["u"], lse=S["lse"])

    def out_proj(S):
        mla.out_proj(S["u"], S["w_uv"], S["out"])

    def append(S):  # the cache-append step (not part of the timed decode step)
        mla.append_kv(S["h"], S["w_dkr"], S["cache"], S["bt"], S["sl"], n_q=n_q, workspace=S["ws_app"],
                      err_word=err)

    def absorb_latent(S):  # the query-side absorption through the merged W_KQ (not part of the timed step)
        mla.absorb_q_latent(S["c_q"], S["q_rope"], S["w_kq"], S["q_abs"])

    def out_comb(S):  # the layer output through the merged W_comb (not part of the timed step)
        mla.out_comb(S["u"], S["w_comb"], S["out_model"], workspace=S["ws_comb"])

    def step(S):
        plan(S)
        absorb(S)
        decode_planned(S)
        combine(S)
        out_proj(S)

    # FP8 latent cache (e4m3 codes, per-column scales): the same pages quantised on
    # the device, then the planned decode call on them (not part of the timed step)
    fp8_scales = torch.from_numpy(mi.fp8_channel_scales(inp)).to(dev)

    def fp8_setup():
        for S in sets:
            S["cache8"] = mla.quantize_fp8(S["cache"], fp8_scales)

    def quantize8(S):
        mla.quantize_fp8(S["cache"], fp8_scales, S["cache8"])

    def decode8_planned(S):
        mla.decode_paged_fp8(S["q_abs"], S["cache8"], fp8_scales, S["bt"], S["sl"], n_q=n_q, num_splits=G,
                             workspace=S["workspace"], err_word=err, planned=True)

    def step8(S):  # the whole step on the FP8 cache
        plan(S)
        absorb(S)
        decode8_planned(S)
        combine(S)
        out_proj(S)

    # eager warm-up (checks the error word), then CUDA graphs of back-to-back
    # steps so the timed region measures device time, not host launches
    for k in range(args.warmup):
        step(sets[k % NSETS])
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise SystemExit(f"device error word {int(err.item())}")
    if args.profile_phase:  # one side call alone, eagerly (short profiling runs)
        fn = {"absorb_q_latent": absorb_latent, "out_comb": out_comb, "append_kv": append,
              "fp8_decode": decode8_planned}[args.profile_phase]
        if args.profile_phase == "fp8_decode":
            fp8_setup()
            for k in range(NSETS):
                plan(sets[k])
        for k in range(6):
            fn(sets[k % NSETS])
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise SystemExit(f"device error word {int(err.item())}")
        if rank == 0:
            print(json.dumps({"profile_phase": args.profile_phase, "calls": 6}), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    R = min(args.steps, ROTATIONS * NSETS)  # steps per graph replay
    graph = capture(lambda: [step(sets[k % NSETS]) for k in range(R)])
    rest = args.steps % R
    graph_rest = capture(lambda: [step(sets[k % NSETS]) for k in range(rest)]) if rest else None
    for _ in range(max(1, args.warmup // R)):
        graph.replay()
    torch.cuda.synchronize()

    t0_ev, t1_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    t0_ev.record(stream)
    for _ in range(args.steps // R):
        graph.replay()
    if graph_rest is not None:
        graph_rest.replay()
    t1_ev.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    total_ms = max_over_ranks(t0_ev.elapsed_time(t1_ev), dist, dev)
    ms_per_step = total_ms / args.steps
    value = job_rate(ws_, T, args.steps, total_ms * 1e-3)

    # per-call phase times: each call alone, R times back to back over the
    # rotating sets in one graph (the decode call is the plan and decode kernels)
    def per_call_us(fn, reps=20):
        g = capture(lambda: [fn(sets[k % NSETS]) for k in range(R)])
        g.replay()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for e0, e1 in ev:
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return 1e3 * float(np.median([e0.elapsed_time(e1) for e0, e1 in ev])) / R

    if args.quick:  # timed region only (short profiling runs)
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_, "steps": args.steps,
                              "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
                              "quick": True, "config": workload_config(inp, G)}), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    for k in range(NSETS):  # every set's workspace holds its plan for the planned decode calls
        plan(sets[k])
    phases = {"decode_plan": per_call_us(plan), "absorb_q": per_call_us(absorb),
              "decode_paged_planned": per_call_us(decode_planned), "combine": per_call_us(combine),
              "out_proj": per_call_us(out_proj),
              # for reference: the plan and the decode kernel in one call
              "decode_paged": per_call_us(decode)}
    append_us = per_call_us(append)
    latent_us = per_call_us(absorb_latent)
    comb_us = per_call_us(out_comb)

    # the FP8 cache's planned decode call, timed like the bf16 one
    fp8_setup()
    for k in range(NSETS):
        plan(sets[k])
    fp8_dec_us = per_call_us(decode8_planned)
    fp8_step_us = per_call_us(step8)
    fp8_quant_us = per_call_us(quantize8)
    for k in range(NSETS):
        plan(sets[k])
        decode_planned(sets[k])  # the bf16 partials back in the workspaces
    # for reference: one step replayed alone after an L2 flush (cold caches,
    # including the graph launch, about 6.6 us on this system)
    g1 = capture(lambda: step(sets[0]))
    single = []
    for _ in range(50):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g1.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        single.append(1e3 * e0.elapsed_time(e1))
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise SystemExit(f"device error word {int(err.item())}")

    # ---------------------------------------------------------------- end to end
    # Per step: the new queries, block table and context lengths go host->device
    # from pinned memory; out and lse come back device->host. The latent cache
    # and weights stay resident in HBM (the KV cache is device state). The step
    # is the library's CapturedStep with host I/O (one CUDA graph per
    # fixed-shape batch holding the copies and the step, as a serving loop would
    # keep it), called through its public Python API, then the host waits for it.
    S0 = sets[0]
    captured = mla.CapturedStep(S0["w_uk"], S0["w_uv"], S0["cache"], S0["bt"], S0["sl"], n_q=n_q, num_splits=G,
                                err_word=err, host_io=True)
    hio = captured.host
    hio["q_nope"].copy_(torch.from_numpy(inp.q_nope.reshape(T, H, -1).view(np.int16)).view(torch.bfloat16))
    hio["q_rope"].copy_(torch.from_numpy(inp.q_rope.reshape(T, H, -1).view(np.int16)).view(torch.bfloat16))
    hio["block_table"].copy_(torch.from_numpy(pg.block_table))
    hio["seq_lens"].copy_(torch.from_numpy(inp.seq_lens))
    h2d = sum(hio[k].numel() * hio[k].element_size() for k in ("q_nope", "q_rope", "block_table", "seq_lens"))
    d2h = sum(hio[k].numel() * hio[k].element_size() for k in ("out", "lse"))

    def e2e_step():
        captured.replay_host()
        stream.synchronize()

    for _ in range(args.warmup):
        e2e_step()
    e2e_times = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step()
        e2e_times.append(time.perf_counter() - t0)
    e2e_total = max_over_ranks(sum(e2e_times), dist, dev)
    e2e_value = job_rate(ws_, T, args.steps, e2e_total)
    e2e_parts = e2e_breakdown(captured, S0["w_uv"], stream, flush, e2e_times)

    if rank == 0:
        hbm, tflops, src = peaks()
        wb = mi.workload_bytes(inp)
        dec_us = phases["decode_paged_planned"]
        dec_bytes, _ = decode_alg(inp)
        bound = roofline_bound(wb["decode_flops"], dec_bytes, dec_us, hbm, tflops)
        traffic = stored_traffic(args.workload)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(inp, G),
            "phases_us": phases,
            "single_step_flushed_us": float(np.median(single)),
            "roofline": {"kernel": "mla_decode_paged_planned (the split-KV decode kernel)", **bound,
                         "traffic": traffic, "peak_source": src,
                         "alg_bytes_per_launch": dec_bytes, "alg_flops_per_launch": wb["decode_flops"],
                         "tflops_achieved": wb["decode_flops"] / (dec_us * 1e-6) / 1e12,
                         "tensor_peak_tflops": tflops,
                         "duration": f"per call, {R} calls back to back over {NSETS} rotating input sets"},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "breakdown_us": e2e_parts},
            "decode_plus_combine": decode_combine_line(dec_us, phases["combine"], dec_bytes, inp, hbm),
            "append_kv": append_line(append_us, T, hbm),
            "absorb_q_latent": latent_line(latent_us, phases["absorb_q"], T, H, hbm),
            "out_comb": comb_line(comb_us, phases["out_proj"], T, H, hbm),
            "fp8_decode": fp8_line(fp8_dec_us, fp8_quant_us, inp, hbm, tflops, src, dec_us, fp8_step_us),
            "gpu_launches": 5 * args.steps,
            "timing": (f"CUDA events around the timed region: graphs of {R} back-to-back steps over "
                       f"{NSETS} rotating input sets, replayed until {args.steps} steps ran"),
            "clocks": clk,
            "wall_s_timed_region": wall,
        }
        if ws_ == 1 and not args.no_workloads:
            line["workloads"] = side_workloads(mla, dev, err, hbm, tflops, src, exclude=args.workload)
        if ws_ == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(inp, budget_s=args.cpu_budget)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def e2e_breakdown(captured, w_uv, stream, flush, e2e_times, reps=30):
    """Where an end-to-end step's time goes (medians, microseconds): the host's wall time
    for one replay of the host-I/O graph plus its synchronisation; the device time of that
    graph (CUDA events on the stream around the replay: the input copy and the step, whose
    out_proj and combine write out and lse into pinned host memory); the packed input copy
    alone (events around one mla_copy16 of the same pinned buffers); out_proj alone writing
    its output into the pinned host buffer and into device memory (the difference is what
    the output's trip over the host link adds); and the rest of the wall time (graph launch
    and the host's wake-up after the stream completes)."""
    import torch
    import mla_latent_kv_paged_gb300 as mla

    def timed(fn):
        acc = []
        for _ in range(reps):
            flush.zero_()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            stream.synchronize()
            acc.append(1e3 * e0.elapsed_time(e1))
        return float(np.median(acc))

    device = timed(captured.replay_host)
    h2d = timed(lambda: mla.copy16(captured._host_in, captured._dev_in, stream))
    u = captured.bufs["u"]
    out_host = timed(lambda: mla.out_proj(u, w_uv, captured.host["out"], stream))
    out_dev = timed(lambda: mla.out_proj(u, w_uv, captured.bufs["out"], stream))
    wall = 1e6 * float(np.median(e2e_times))
    return {"wall": wall, "device_graph": device, "h2d_copy": h2d, "out_proj_to_host": out_host,
            "out_proj_to_device": out_dev, "host_launch_and_wait": wall - device}


def decode_combine_line(dec_us, comb_us, dec_bytes, inp, hbm):
    """The decode unit of the measurement plan: the split-KV decode kernel and the merge of
    its partials, with the merge's output (u in bf16, lse in fp32) added to the bytes."""
    T, H = inp.B * inp.n_q, inp.H
    nbytes = dec_bytes + T * H * (mi.D_C * 2 + 4)
    us = dec_us + comb_us
    achieved = nbytes / (us * 1e-6) / 1e9
    return {"us": us, "alg_bytes": nbytes, "achieved_gbs": achieved, "peak_gbs": hbm, "frac": achieved / hbm,
            "bound": "hbm"}


def decode_alg(inp):
    """Algorithmic bytes and flops of one decode-kernel launch: the cache read once, the absorbed
    queries, lengths and block-table entries in use (the split partials are not counted)."""
    wb = mi.workload_bytes(inp)
    T, H = inp.B * inp.n_q, inp.H
    nbytes = wb["cache_bytes"] + T * H * 576 * 2 + inp.B * 4 + int(mi.pages_for(inp.seq_lens).sum()) * 4
    return nbytes, wb["decode_flops"]


def side_workloads(mla, dev, err, hbm, tflops, src, exclude=None, calls=20, reps=10):
    """The pages' other decode workloads (ragged batch, long contexts, two query tokens), one
    input set each (every latent cache is 0.6-1.25 GB, far beyond L2): the decode kernel's time
    per call and its roofline, and the whole step's, each as ``calls`` back-to-back calls in a
    CUDA graph replayed ``reps`` times (median)."""
    import torch
    res = {}
    stream = torch.cuda.current_stream()
    names = {3: "ragged", 4: "long_context", 5: "two_query_tokens"}
    for idx in (3, 4, 5):
        if idx == exclude:
            continue
        inp = mi.workload_inputs(idx)
        pg = mi.make_paged(inp, spare_pages=mi.WORKLOADS[idx].spare_pages)
        T, H, B, n_q = inp.B * inp.n_q, inp.H, inp.B, inp.n_q

        def to_dev(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

        S = dict(q_nope=to_dev(inp.q_nope.reshape(T, H, -1)), q_rope=to_dev(inp.q_rope.reshape(T, H, -1)),
                 w_uk=to_dev(inp.w_uk), w_uv=to_dev(inp.w_uv), cache=to_dev(pg.cache),
                 bt=torch.from_numpy(pg.block_table).to(dev), sl=torch.from_numpy(inp.seq_lens).to(dev))
        G = mla.default_splits(n_q)
        bufs = dict(q_abs=torch.empty((T, H, 576), dtype=torch.bfloat16, device=dev),
                    workspace=torch.empty(mla.workspace_bytes(B, n_q, H, G), dtype=torch.uint8, device=dev),
                    u=torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev),
                    lse=torch.empty((T, H), dtype=torch.float32, device=dev),
                    out=torch.empty((T, H, 128), dtype=torch.bfloat16, device=dev))

        def step():
            mla.decode_step(S["q_nope"], S["q_rope"], S["w_uk"], S["w_uv"], S["cache"], S["bt"], S["sl"], n_q=n_q,
                            num_splits=G, bufs=bufs, err_word=err)

        def decode_planned():
            mla.decode_paged(bufs["q_abs"], S["cache"], S["bt"], S["sl"], n_q=n_q, num_splits=G,
                             workspace=bufs["workspace"], err_word=err, planned=True)

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        if int(err.item()) != 0:
            raise SystemExit(f"device error word {int(err.item())} on workload {idx}")

        def timed(fn):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(calls):
                    fn()
            g.replay()
            torch.cuda.synchronize()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for e0, e1 in ev:
                e0.record(stream)
                g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            return 1e3 * float(np.median([e0.elapsed_time(e1) for e0, e1 in ev])) / calls

        step_us = timed(step)
        dec_us = timed(decode_planned)  # the plan of the last step is in the workspace
        nbytes, flops = decode_alg(inp)
        bound = roofline_bound(flops, nbytes, dec_us, hbm, tflops)
        res[names[idx]] = {
            "workload": workload_config(inp, G)["workload"], "decode_us": dec_us, "step_us": step_us,
            "tokens_per_s": T / (step_us * 1e-6), "alg_bytes_per_launch": nbytes, "alg_flops_per_launch": flops,
            **bound, "tflops_achieved": flops / (dec_us * 1e-6) / 1e12, "peak_source": src,
            "traffic": stored_traffic(idx),
            "duration": f"per call, {calls} calls back to back in a CUDA graph, median of {reps} replays"}
        del S, bufs
        torch.cuda.empty_cache()
    return res


def fp8_line(us, quant_us, inp, hbm, tflops, src, bf16_us, step_us=None):
    """The decode kernel on the FP8 cache (e4m3 codes, one float scale per column): its time
    per call and roofline. The cache bytes halve, so the flops per byte double (past the
    ridge point of the measured peaks: tensor bound). quantize_us: the whole cache quantised
    once (151 MB read, 75 MB written), for context. step_us: the whole step on the FP8 cache
    (steps back to back), with its tokens/s."""
    T, H = inp.B * inp.n_q, inp.H
    wb = mi.workload_bytes(inp)
    cache8 = int(inp.seq_lens.sum()) * 576
    nbytes = cache8 + T * H * 576 * 2 + inp.B * 4 + int(mi.pages_for(inp.seq_lens).sum()) * 4 + 576 * 4
    return {"kernel": "mla_decode_paged_planned_fp8", "decode_us": us, "cache_bytes": cache8,
            "cache_bytes_bf16": wb["cache_bytes"], "alg_bytes_per_launch": nbytes,
            "alg_flops_per_launch": wb["decode_flops"],
            **roofline_bound(wb["decode_flops"], nbytes, us, hbm, tflops), "peak_source": src,
            "traffic": stored_traffic("fp8"),
            "speedup_vs_bf16_decode": bf16_us / us, "quantize_us": quant_us,
            **({"step_us": step_us, "step_tokens_per_s": T / (step_us * 1e-6)} if step_us else {}),
            "duration": "per call, back to back over the rotating input sets"}


def append_line(us, T, hbm):
    """The cache-append call (c = h W^DKV, k^R = RoPE(h W^KR) into the pages): its time per call
    and its HBM roofline (weights + hidden states read, the new rows written)."""
    alg = 576 * D_MODEL * 2 + T * D_MODEL * 2 + T * 576 * 2
    gbs = alg / (us * 1e-6) / 1e9
    return {"us": us, "d_model": D_MODEL, "rows": T, "alg_bytes": alg, "achieved_gbs": gbs, "peak_gbs": hbm,
            "frac": gbs / hbm, "bound": "hbm"}


def latent_line(us, absorb_us, T, H, hbm):
    """The query-side absorption through the merged weight (q_abs = c_q W_KQ, W_KQ = W_UQ W_UK per
    head): its time per call and HBM roofline, beside the weight bytes of the unmerged route."""
    alg = D_Q * H * 512 * 2 + T * D_Q * 2 + T * H * 64 * 2 + T * H * 576 * 2
    gbs = alg / (us * 1e-6) / 1e9
    return {"us": us, "d_q": D_Q, "rows": T, "heads": H, "alg_bytes": alg, "achieved_gbs": gbs, "peak_gbs": hbm,
            "frac": gbs / hbm, "bound": "hbm", "merged_weight_bytes": D_Q * H * 512 * 2,
            "unmerged_weight_bytes": D_Q * H * 128 * 2 + H * 128 * 512 * 2, "absorb_q_us": absorb_us}


def comb_line(us, out_proj_us, T, H, hbm):
    """The layer output through the merged value/output weight (out = sum_h u_h W_comb,h, W_comb =
    W_UV W_O per head): its time per call and HBM roofline, beside the weight bytes of the unmerged
    route (out_proj, then the output projection)."""
    alg = D_MODEL * H * 512 * 2 + T * H * 512 * 2 + T * D_MODEL * 2
    gbs = alg / (us * 1e-6) / 1e9
    return {"us": us, "d_model": D_MODEL, "rows": T, "heads": H, "alg_bytes": alg, "achieved_gbs": gbs,
            "peak_gbs": hbm, "frac": gbs / hbm, "bound": "hbm", "merged_weight_bytes": D_MODEL * H * 512 * 2,
            "unmerged_weight_bytes": H * 128 * 512 * 2 + D_MODEL * H * 128 * 2, "out_proj_us": out_proj_us}


TRAFFIC_PROFILES = {2: "decode_tc_b32_l4096.md", 3: "decode_tc_ragged_b128.md", 4: "decode_tc_long_b4_l131072.md",
                    5: "decode_tc_two_token_b64_l8192.md", "fp8": "decode_tc_fp8_b32_l4096.md"}


def stored_traffic(workload=WORKLOAD_INDEX):
    """dram bytes per decode launch from the committed ncu summary of this workload, if the
    kernel is unchanged since (None otherwise)."""
    if workload not in TRAFFIC_PROFILES:
        return None
    path = os.path.join(ROOT, "profiles", TRAFFIC_PROFILES[workload])
    try:
        kv = dict(ln.split(":", 1) for ln in open(path) if ln.startswith(("traffic_bytes_per_launch:", "kernel_rev:")))
        if kv.get("kernel_rev", "").strip() == mla_kernel_rev():
            return int(kv["traffic_bytes_per_launch"])
    except Exception:
        pass
    return None


def mla_kernel_rev():
    """A digest of the decode kernel sources, to tell whether stored counters are stale."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_latent_kv_paged_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.startswith("decode") or name.endswith(".cuh"):
            h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the 'workloads' block (the ragged, long-context and two-token decode workloads)")
    ap.add_argument("--workload", type=int, default=WORKLOAD_INDEX, choices=[2, 3, 4, 5],
                    help="the decode workload (2: 32 x 4096, the default; 3: 128 ragged; 4: 4 x 131072; "
                         "5: 64 x 8192 with two query tokens)")
    ap.add_argument("--quick", action="store_true",
                    help="time the steps only (no phase times, end-to-end leg or CPU baseline): for profiling runs")
    ap.add_argument("--profile-phase", choices=["absorb_q_latent", "out_comb", "append_kv", "fp8_decode"],
                    default=None,
                    help="after the warm-up, run this call 6 times over the rotating sets and stop: for profiling runs")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
