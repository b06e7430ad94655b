"""Benchmark of the PIC link step on GB300.

One step = the whole link hot path for one request batch: row selection, splice,
RoPE tables, re-rotation of cached K, fresh K/V, link attention (+ LSE merge).
Default workload: 100 chunks x 1000 tokens linked in a random order + a 256-token
query, k = 8, Hq = 32, Hkv = 8, d = 128, bf16, 16-token pages (100,256 tokens).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line (rank 0).  value = context tokens (T + q, summed over requests
and ranks) per second of device time, the pool and inputs resident in HBM; L2 is
flushed (512 MB read, untimed) before every timed step.  e2e = the same metric
through the Python binding with per-step host->device copies of the step's inputs
from pinned memory and a device->host copy of the attention output.
`per_config` times the other workloads (the RAG prompt, the 20-chunk sink prompt,
the 16-request batch) with the same step.  On rank 0 at N = 1 the float64 oracle
then runs on the host cores, in full, on every workload: its time is
`cpu_baseline` (headline) and `per_config[].oracle`, and its output gives the GPU
outputs' parity errors (`parity`, `per_config[].parity`).
`--impl reference` times the oracle on slices of the headline workload (see
OracleSlices).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "PIC link: context tokens/s per layer; % of HBM / bf16 tensor-core roofline"
UNIT = "tokens/s"

# ncu DRAM bytes (read + write) per launch of each timed kernel (per call for the
# two-launch composition), with the kernel source they were taken from; reported
# as roofline traffic only while the source is unchanged.
NCU_TRAFFIC = {
    # link_attn_tc_kernel<0>, long_context_100x1000: 665.66 MB read + 138.84 MB written
    ("attention", "1941c91a9f32e19f"): 804495360,
    # link_attn_tc_kernel<1> (rotate-on-read), long_context_100x1000: 643.53 MB read + 145.00 MB written
    ("rotate_on_read", "1941c91a9f32e19f"): 788534784,
    # rerotate_kernel<bf16>, long_context_100x1000: 201.36 MB read + 140.36 MB written
    ("rerotate", "f862c45770d2a0fa"): 341722880,
    # rope_cached_kernel<bf16> (scheme B), long_context_100x1000: 304.83 MB read + 144.01 MB written
    ("scheme_b", "f862c45770d2a0fa"): 448839168,
    # decode_kernel<4>, one row per request over the long-context link: 420.65 MB read + 4.84 MB written
    ("decode", "3e15b5e3dc89f7e3"): 425493760,
    # compose_kernel, 32 heads x 100-chunk chain, both levels: 417.43 + 14.76 MB read + 3.60 MB written
    ("compose", "51b0a7600676d22a"): 435783936,
}


def _src_hash(name):
    p = os.path.join(ROOT, "position_independent_kv_pic_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _workload(name):
    from position_independent_kv_pic_gb300 import inputs
    if name not in inputs.PRESETS:
        raise SystemExit(f"unknown workload {name}; choose from {sorted(inputs.PRESETS)}")
    return inputs.PRESETS[name]()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- aggregation

def reduce_max(x: float, device: str) -> float:
    """Max of a per-rank float over the process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(world: int, steps: int, tokens_per_rank_step: int, max_total_ms: float) -> float:
    """Tokens all ranks processed divided by the slowest rank's timed region."""
    return world * steps * tokens_per_rank_step / (max_total_ms / 1e3)


# ----------------------------------------------------------------------------- GPU arm

# the pages' other prompt shapes, timed after the headline workload with the same step
PER_CONFIG = ("rag_prompt_6chunks", "many_chunk_sink_20", "batched_shared_16req")


def step_work(batch):
    """Algorithmic work of one link step, from the step's own outputs: re-rotated
    bytes (K read + written) and attention flops 4 d Hq sum(p_r + 1)."""
    wl = batch.wl
    rows = batch.rows.cpu().numpy().astype(np.int64)
    rot = batch.rot.cpu().numpy()
    lohi = np.ascontiguousarray(rot[:, 3]).view(np.int16).reshape(-1, 2) if len(rot) else np.zeros((0, 2), np.int16)
    rot_tokens = int((lohi[:, 1].astype(np.int64) - lohi[:, 0]).sum())
    el = 2 if wl.dtype == "bf16" else 4
    return 2 * rot_tokens * wl.Hkv * wl.d * el, 4.0 * wl.d * wl.Hq * float((rows + 1).sum())


def time_link(batch, steps, l2_flush, stream):
    """Per-step CUDA-event times (ms) of `steps` link steps, L2 flushed before each:
    (whole step, re-rotation pass, attention run)."""
    import torch
    ev = lambda: torch.cuda.Event(enable_timing=True)
    step_ev = [(ev(), ev()) for _ in range(steps)]
    rot_ev = [(ev(), ev()) for _ in range(steps)]
    att_ev = [(ev(), ev()) for _ in range(steps)]
    for i in range(steps):
        l2_flush()
        step_ev[i][0].record(stream)
        batch.run(marks={"rerotate": rot_ev[i], "attention": att_ev[i]})
        step_ev[i][1].record(stream)
    torch.cuda.synchronize()
    return ([a.elapsed_time(b) for a, b in step_ev], [a.elapsed_time(b) for a, b in rot_ev],
            [a.elapsed_time(b) for a, b in att_ev])


def time_graph(batch, steps, warmup, l2_flush, stream):
    """The same step captured as one CUDA graph (LinkGraph), `steps` replays timed with
    CUDA events, L2 flushed before each.  Returns (per-replay ms, None) or (None, the
    reason the capture failed)."""
    import torch
    from position_independent_kv_pic_gb300.link import LinkGraph
    try:
        g = LinkGraph(batch)
    except RuntimeError as e:  # reported in the result line; the eager step stands
        torch.cuda.synchronize()
        return None, str(e).splitlines()[0][:200]
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    evs = [(ev(), ev()) for _ in range(steps)]
    for i in range(steps):
        l2_flush()
        evs[i][0].record(stream)
        g.replay()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    del g
    return [a.elapsed_time(b) for a, b in evs], None


def link_output(batch):
    """The step's attention output from the pool as cached (the in-place re-rotation
    of a repeated step would rotate K again), copied to the host."""
    import torch
    batch.reset_pool()
    batch.err.zero_()
    batch.run()
    torch.cuda.synchronize()
    if batch.error() != 0:
        raise SystemExit(f"device error ({batch.wl.name}): {batch.error()}")
    return batch.out.double().cpu().numpy()


def per_config_gpu(name, steps, warmup, l2_flush, stream, hbm, tf_burst):
    """One of the other workloads: mean step time, tokens/s, attention and
    re-rotation roofline fractions, and the step's output (for the parity check)."""
    import torch
    from position_independent_kv_pic_gb300.link import LinkBatch
    wl = _workload(name)
    b = LinkBatch(wl)
    for _ in range(warmup):
        b.run()
    torch.cuda.synchronize()
    if b.error() != 0:
        raise SystemExit(f"device error ({name}): {b.error()}")
    rot_bytes, flops = step_work(b)
    st, ro, at = time_link(b, steps, l2_flush, stream)
    if b.error() != 0:
        raise SystemExit(f"device error ({name}): {b.error()}")
    ms, rms, ams = statistics.mean(st), statistics.mean(ro), statistics.mean(at)
    gms, gerr = time_graph(b, steps, warmup, l2_flush, stream)
    if b.error() != 0:
        raise SystemExit(f"device error ({name}, graph): {b.error()}")
    entry = {"workload": name, "requests": b.n_req, "chunks": b.n_chunks, "tokens": b.tokens, "rows": b.n_rows,
             "steps": steps, "ms_per_step": ms, "tokens_per_s": b.tokens / (ms / 1e3),
             "graph": ({"ms_per_step": statistics.mean(gms), "tokens_per_s": b.tokens / (statistics.mean(gms) / 1e3)}
                       if gms else {"error": gerr}),
             "attention": {"ms": ams, "tflops": flops / (ams / 1e3) / 1e12,
                           "frac": flops / (ams / 1e3) / 1e12 / tf_burst, "flop": flops},
             "rerotate": {"ms": rms, "gbs": rot_bytes / (rms / 1e3) / 1e9,
                          "frac": rot_bytes / (rms / 1e3) / 1e9 / hbm, "bytes": rot_bytes}}
    out = link_output(b)
    del b
    torch.cuda.empty_cache()
    return entry, out


def run_gpu(args, rank, world):
    import torch
    import torch.distributed as dist

    import position_independent_kv_pic_gb300 as pic
    from position_independent_kv_pic_gb300 import build as pic_build
    from position_independent_kv_pic_gb300.link import LinkBatch, LinkPipeline

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if rank == 0 or world == 1:
        pic_build.build()
    if world > 1:
        dist.barrier()
    pic.load()

    wl = _workload(args.workload)
    batch = LinkBatch(wl)
    stream = torch.cuda.current_stream()
    # L2 flush before every timed step: a 512 MB read (four times L2) evicts every
    # line and writes back any dirty one while untimed; a memset would instead leave
    # L2 full of dirty lines whose write-back lands inside the next timed kernel
    flush = torch.zeros(512 * 1024 * 1024 // 4, dtype=torch.int32, device="cuda")

    def l2_flush():
        flush.sum()

    for _ in range(args.warmup):
        batch.run()
    torch.cuda.synchronize()
    if batch.error() != 0:
        raise SystemExit(f"device error: {pic.pic_strerror(batch.error())}")

    rot_bytes, attn_flops = step_work(batch)
    el = 2 if wl.dtype == "bf16" else 4
    K = args.steps
    ev = lambda: torch.cuda.Event(enable_timing=True)

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t_wall0 = time.perf_counter()
        # eager steps (eleven launches from the host on three streams), with the re-rotation
        # and attention runs timed inside, then the same step as one CUDA graph launch
        step_ms, rot_ms, att_ms = time_link(batch, K, l2_flush, stream)
        graph_ms, graph_err = time_graph(batch, K, args.warmup, l2_flush, stream)
        t_wall = time.perf_counter() - t_wall0
    if world > 1:
        dist.barrier()
    if batch.error() != 0:
        raise SystemExit(f"device error: {pic.pic_strerror(batch.error())}")

    eager_total_ms = reduce_max(sum(step_ms), "cuda")
    total_ms = reduce_max(sum(graph_ms), "cuda") if graph_ms else eager_total_ms
    tokens = batch.tokens
    value = whole_job_throughput(world, K, tokens, total_ms)

    # end to end through the binding: every step uploads its inputs from pinned host
    # memory and reads its result back to pinned host memory; LinkPipeline runs the
    # copies on their own streams, overlapped with the neighbouring steps' kernels (the
    # steps as CUDA graphs when the capture above worked)
    batch.pin_host_inputs()
    pipe = LinkPipeline(batch, graphs=graph_ms is not None)
    Ke = max(3, min(K, 50))
    for _ in range(2):
        pipe.submit(batch.host_pinned, stream)
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    e0.record(stream)
    pipe.begin(stream)
    last = None
    for _ in range(Ke):
        _, last = pipe.submit(batch.host_pinned, stream)
    stream.wait_event(last)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / Ke

    # decode after the link (one new row per request over the linked cache): its own
    # timed loop after the link step's, L2 flushed before every step
    dec = None
    if wl.dtype == "bf16" and pic.pic_decode_workspace(batch.n_req, wl.Hq, wl.Hkv, wl.d, batch.pic_dtype) > 0:
        batch.setup_decode()
        for _ in range(args.warmup):
            batch.run_decode()
        torch.cuda.synchronize()
        Kd = max(3, min(K, 50))
        dstep = [(ev(), ev()) for _ in range(Kd)]
        datt = [(ev(), ev()) for _ in range(Kd)]
        for i in range(Kd):
            l2_flush()
            dstep[i][0].record(stream)
            batch.run_decode(marks={"decode": datt[i]})
            dstep[i][1].record(stream)
        torch.cuda.synchronize()
        if batch.error() != 0:
            raise SystemExit(f"device error: {pic.pic_strerror(batch.error())}")
        dec = (statistics.mean(a.elapsed_time(b) for a, b in dstep),
               statistics.mean(a.elapsed_time(b) for a, b in datt), batch.dec_bytes, Kd)

    # scheme B (chunks cached without position encoding, encoded at the global
    # position by the step): the same step with pic_rope_cached_k in place of the
    # re-rotation (out of place into private pages when chunks are shared)
    schb = None
    bb = LinkBatch(wl, scheme="nope")
    for _ in range(args.warmup):
        bb.run()
    torch.cuda.synchronize()
    Kb = max(3, min(K, 50))
    bstep = [(ev(), ev()) for _ in range(Kb)]
    brope = [(ev(), ev()) for _ in range(Kb)]
    for i in range(Kb):
        l2_flush()
        bstep[i][0].record(stream)
        bb.run(marks={"rerotate": brope[i]})
        bstep[i][1].record(stream)
    torch.cuda.synchronize()
    if bb.error() != 0:
        raise SystemExit(f"device error (scheme B): {pic.pic_strerror(bb.error())}")
    kept = int(bb.chunk_lens.sum()) - (bb.n_rows - int(bb.q_len.sum()))  # cached slots encoded
    rope_bytes = 2 * kept * wl.Hkv * wl.d * el  # K read + written; the position table's rows are not counted
    schb = (statistics.mean(a.elapsed_time(b) for a, b in bstep),
            statistics.mean(a.elapsed_time(b) for a, b in brope), rope_bytes, Kb, bb.tokens)
    del bb
    torch.cuda.empty_cache()

    # rotate-on-read: the same step with the correction applied inside link attention
    # (no re-rotation pass; the cached pages are read as cached)
    ror = None
    if pic.pic_link_attention_workspace(batch.n_rows, batch.n_req, wl.Hq, wl.Hkv, wl.d, batch.pic_dtype) > 0:
        rb = LinkBatch(wl, scheme="ror")
        for _ in range(args.warmup):
            rb.run()
        torch.cuda.synchronize()
        Kr = max(3, min(K, 50))
        rstep = [(ev(), ev()) for _ in range(Kr)]
        ratt = [(ev(), ev()) for _ in range(Kr)]
        for i in range(Kr):
            l2_flush()
            rstep[i][0].record(stream)
            rb.run(marks={"attention": ratt[i]})
            rstep[i][1].record(stream)
        torch.cuda.synchronize()
        if rb.error() != 0:
            raise SystemExit(f"device error (rotate-on-read): {pic.pic_strerror(rb.error())}")
        ror = (statistics.mean(a.elapsed_time(b) for a, b in rstep),
               statistics.mean(a.elapsed_time(b) for a, b in ratt), Kr, rb.tokens, rb.launches_per_step)
        # decode after the rotate-on-read link: the pages keep each chunk's frame
        if wl.dtype == "bf16" and pic.pic_decode_workspace(rb.n_req, wl.Hq, wl.Hkv, wl.d, rb.pic_dtype) > 0:
            rb.setup_decode()
            for _ in range(args.warmup):
                rb.run_decode()
            torch.cuda.synchronize()
            rdec = [(ev(), ev()) for _ in range(Kr)]
            for i in range(Kr):
                l2_flush()
                rb.run_decode(marks={"decode": rdec[i]})
            torch.cuda.synchronize()
            if rb.error() != 0:
                raise SystemExit(f"device error (decode after rotate-on-read): {pic.pic_strerror(rb.error())}")
            ror = ror + (statistics.mean(a.elapsed_time(b) for a, b in rdec), rb.dec_bytes)
        del rb
        torch.cuda.empty_cache()

    # linear-layer state composition (a hybrid model's linear-attention layer over the
    # same chunk chains: 32 heads of 128 x 128 states per chunk)
    comp = None
    if wl.d == 128:
        from position_independent_kv_pic_gb300 import inputs
        from position_independent_kv_pic_gb300.states import ComposeBatch
        T, S, chains = inputs.linear_states(wl, H=32, d=128)
        cbatch = ComposeBatch(T, S, chains)
        del T, S
        for _ in range(args.warmup):
            cbatch.run()
        torch.cuda.synchronize()
        Kc = max(3, min(K, 50))
        cev = [(ev(), ev()) for _ in range(Kc)]
        for i in range(Kc):
            l2_flush()
            cev[i][0].record(stream)
            cbatch.run()
            cev[i][1].record(stream)
        torch.cuda.synchronize()
        if cbatch.error() != 0:
            raise SystemExit(f"device error (composition): {pic.pic_strerror(cbatch.error())}")
        comp = (statistics.mean(a.elapsed_time(b) for a, b in cev), cbatch.algorithmic_bytes, Kc, cbatch.seg,
                cbatch.n_req * cbatch.H, cbatch.n_elems, cbatch.launches)
        del cbatch
        torch.cuda.empty_cache()

    hbm, tf_burst, tf_sus, peak_kind = _peaks()
    # the other workloads (rank 0 reports them; every rank runs the same work)
    per_config, outputs = [], {}
    if not args.no_per_config:
        for name in PER_CONFIG:
            entry, out = per_config_gpu(name, max(3, min(K, 20)), args.warmup, l2_flush, stream, hbm, tf_burst)
            per_config.append(entry)
            outputs[name] = out
    outputs[wl.name] = link_output(batch)
    att_avg = statistics.mean(att_ms)
    rot_avg = statistics.mean(rot_ms)
    att_tflops = attn_flops / (att_avg / 1e3) / 1e12
    rot_gbs = rot_bytes / (rot_avg / 1e3) / 1e9
    traffic = NCU_TRAFFIC.get(("attention", _src_hash("attention.cu")))
    ortraffic = NCU_TRAFFIC.get(("rotate_on_read", _src_hash("attention.cu")))
    rtraffic = NCU_TRAFFIC.get(("rerotate", _src_hash("rotate.cu")))
    btraffic = NCU_TRAFFIC.get(("scheme_b", _src_hash("rotate.cu")))
    dtraffic = NCU_TRAFFIC.get(("decode", _src_hash("decode.cu")))
    ctraffic = NCU_TRAFFIC.get(("compose", _src_hash("compose.cu")))

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": total_ms / K, "ms_per_step_eager": eager_total_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic: seeded N(0,1) K/V/Q, cached K drawn as stored (position-encoded) keys",
        "config": {"workload": wl.name, "requests": batch.n_req, "chunks": batch.n_chunks,
                   "tokens": tokens, "rows": batch.n_rows, "Hq": wl.Hq, "Hkv": wl.Hkv, "d": wl.d,
                   "page": 16, "pages": batch.n_pages, "rot_pages": batch.n_rot,
                   "l2": "flushed (512 MB read, untimed) before every timed step",
                   "launch": ("one CUDA graph per step (the step's eleven kernels on three streams)" if graph_ms
                              else f"eager (graph capture failed: {graph_err})"),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": att_tflops, "peak": tf_burst, "unit": "TFLOP/s",
                     "frac": att_tflops / tf_burst, "traffic": traffic,
                     "traffic_kernel": "link_attn_tc_kernel (ncu dram__bytes_read+write, one launch)",
                     "kernel": "pic_link_attention_run (tcgen05 attention + LSE merge; the unit plan and the Q "
                               "pre-pass run beside the re-rotation pass on another stream)",
                     "algorithmic": f"4*d*Hq*sum(p_r+1) = {attn_flops:.4e} flop per launch",
                     "peak_source": f"{peak_kind} bf16 dense burst"},
        "rooflines": {
            "attention": {"bound": "tensor", "achieved": att_tflops, "peak": tf_burst, "unit": "TFLOP/s",
                          "frac": att_tflops / tf_burst, "ms": att_avg, "traffic": traffic,
                          "frac_of_sustained": att_tflops / tf_sus if tf_sus else None},
            **({"decode": {"bound": "hbm", "achieved": dec[2] / (dec[1] / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                           "frac": dec[2] / (dec[1] / 1e3) / 1e9 / hbm, "ms": dec[1], "ms_per_decode_step": dec[0],
                           "algorithmic_bytes": dec[2], "steps": dec[3], "traffic": dtraffic,
                           "kernel": "pic_decode_attention (split-KV decode + merge), one new row per request; "
                                     "the step adds its RoPE table and K/V write"}} if dec else {}),
            **({"scheme_b": {"bound": "hbm", "achieved": schb[2] / (schb[1] / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                             "frac": schb[2] / (schb[1] / 1e3) / 1e9 / hbm, "ms": schb[1],
                             "algorithmic_bytes": schb[2], "ms_per_step": schb[0], "traffic": btraffic,
                             "tokens_per_s": world * schb[4] / (schb[0] / 1e3), "steps": schb[3],
                             "kernel": "pic_rope_cached_k (scheme B: cached K encoded at its global position "
                                       "from a per-position table; bytes = K read + written only, the table "
                                       "rows it also reads are not counted); the step runs it in place of "
                                       "the offset table and the re-rotation"}}
               if schb else {}),
            **({"rotate_on_read": {"bound": "tensor", "achieved": attn_flops / (ror[1] / 1e3) / 1e12,
                                   "peak": tf_burst, "unit": "TFLOP/s",
                                   "frac": attn_flops / (ror[1] / 1e3) / 1e12 / tf_burst, "ms": ror[1],
                                   "ms_per_step": ror[0], "tokens_per_s": world * ror[3] / (ror[0] / 1e3),
                                   "traffic": ortraffic,
                                   "steps": ror[2], "launches_per_step": ror[4],
                                   "kernel": "pic_link_attention_ror (framed page layout: each chunk's keys stay "
                                             "in its frame, Q is rotated back by the chunk's offset at frame "
                                             "changes); the step has no re-rotation pass"}} if ror else {}),
            **({"decode_after_ror": {"bound": "hbm", "achieved": ror[6] / (ror[5] / 1e3) / 1e9, "peak": hbm,
                                     "unit": "GB/s", "frac": ror[6] / (ror[5] / 1e3) / 1e9 / hbm, "ms": ror[5],
                                     "algorithmic_bytes": ror[6],
                                     "kernel": "pic_decode_attention over the rotate-on-read link's framed pages "
                                               "(Q fragments rotated per frame)"}} if ror and len(ror) > 5 else {}),
            **({"compose": {"bound": "hbm", "achieved": comp[1] / (comp[0] / 1e3) / 1e9, "peak": hbm,
                            "unit": "GB/s", "frac": comp[1] / (comp[0] / 1e3) / 1e9 / hbm, "ms": comp[0],
                            "algorithmic_bytes": comp[1], "steps": comp[2], "seg": comp[3], "chains": comp[4], "traffic": ctraffic,
                            "chain_elements": comp[5], "launches": comp[6],
                            "kernel": "pic_compose_states (linear-layer state S = T_n(..(T_2 S_1 + S_2)..) + S_n "
                                      "per request and head, 32 heads of 128 x 128 fp32 states; bytes = S of "
                                      "every element + T of every non-first element + the output)"}}
               if comp else {}),
            "rerotate": {"bound": "hbm", "achieved": rot_gbs, "peak": hbm, "unit": "GB/s", "frac": rot_gbs / hbm,
                         "ms": rot_avg, "traffic": rtraffic, "algorithmic_bytes": rot_bytes,
                         "frac_of_8tbs": rot_gbs / 8000.0},
        },
        "e2e": {"value": world * tokens / (e2e_ms / 1e3), "unit": UNIT, "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": batch.h2d_bytes(), "d2h_bytes_per_step": batch.d2h_bytes()},
        "clocks": clocks.summary(),
        "gpu_launches": K * batch.launches_per_step,
        "wall_s_timed_region": t_wall,
    }
    if per_config:
        result["per_config"] = per_config
    return result, batch, outputs


# ----------------------------------------------------------------------------- CPU oracle

def _oracle_inputs(wl):
    """The workload's inputs as the oracle takes them, float64, one tuple per request
    (chunks' stored K and V in link order, q, k, un-roped Q / K_new and V_new of the
    request's recomputed rows).  Drawn from the same seeded generators as the GPU arm."""
    import oracle.pic_oracle as O
    from position_independent_kv_pic_gb300 import inputs
    kst, vst, off = inputs.chunk_store(wl)
    counts = [O.count_rows(wl.chunk_lens[r.chunk_ids], r.q, r.k) for r in wl.requests]
    qr, kn, vn = (t.double().numpy() for t in inputs.row_inputs(wl, int(sum(counts))))
    reqs, a = [], 0
    for req, n in zip(wl.requests, counts):
        ck = [kst[off[c]:off[c + 1]].double().numpy() for c in req.chunk_ids]
        cv = [vst[off[c]:off[c + 1]].double().numpy() for c in req.chunk_ids]
        reqs.append((ck, cv, req.q, req.k, qr[a:a + n], kn[a:a + n], vn[a:a + n]))
        a += n
    return reqs


def oracle_step(wl, reqs, threads=None):
    """The float64 oracle, as it stands, on the whole link step of every request (row
    selection, splice with the re-rotation of every chunk, fresh K/V, attention of
    every recomputed row).  Returns (seconds, output rows [n_rows][Hq][d])."""
    import torch

    import oracle.pic_oracle as O
    prev = torch.get_num_threads()
    if threads:
        torch.set_num_threads(threads)
    try:
        t0 = time.perf_counter()
        outs = [O.link_request(*r, wl.theta, wl.dtype)["out"] for r in reqs]
        dt = time.perf_counter() - t0
    finally:
        torch.set_num_threads(prev)
    return dt, np.concatenate(outs) if outs else np.zeros((0, wl.Hq, wl.d))


def timed_oracle(wl, reqs, threads=None, reps=3):
    """One untimed warm-up, then the median of `reps` whole-step runs (the KV-cache
    blog's timing method: warm-ups, then the median).  Returns (seconds, output)."""
    _, out = oracle_step(wl, reqs, threads)
    ts = [oracle_step(wl, reqs, threads)[0] for _ in range(reps)]
    return statistics.median(ts), out


def parity_errors(gpu_out, ref):
    e = np.abs(gpu_out - ref)
    return {"max_abs": float(e.max()) if e.size else 0.0, "mean_abs": float(e.mean()) if e.size else 0.0,
            "tol_max_abs": 2e-2, "tol_mean_abs": 2e-3, "rows": int(ref.shape[0])}


def cpu_legs(result, wl, outputs):
    """rank 0, N = 1: the oracle timed on the host cores, in full (no sampling), and
    the GPU outputs' errors against it.  Headline workload: one whole-step run on
    all cores.  Other workloads: all cores and one core, 1 warm-up + median of 3
    (the 16-request batch, about 2e12 float64 flop: one all-core run)."""
    import torch
    threads = torch.get_num_threads()
    host = {"threads": threads, "cpu_count": os.cpu_count()}
    t, ref = oracle_step(wl, _oracle_inputs(wl))
    result["cpu_baseline"] = {
        "value": wl.total_tokens() / t, "unit": UNIT, "cores": threads, "kind": "oracle", "seconds": t,
        "sample": f"the whole step of {wl.name} (all {ref.shape[0]} recomputed rows, every chunk re-rotated; no "
                  f"sampling, no extrapolation), one run on {threads} threads"}
    result["parity"] = {wl.name: parity_errors(outputs[wl.name], ref)}
    for entry in result.get("per_config", []):
        name = entry["workload"]
        cwl = _workload(name)
        reqs = _oracle_inputs(cwl)
        if name == "batched_shared_16req":
            t_all, ref = oracle_step(cwl, reqs)
            orc = {"all_cores_s": t_all, "runs": "one", **host}
        else:
            t_all, ref = timed_oracle(cwl, reqs)
            t_one, _ = timed_oracle(cwl, reqs, threads=1)
            orc = {"all_cores_s": t_all, "one_core_s": t_one, "runs": "1 warm-up + median of 3", **host,
                   "one_core_tokens_per_s": entry["tokens"] / t_one}
        orc["all_cores_tokens_per_s"] = entry["tokens"] / t_all
        orc["gpu_speedup_all_cores"] = t_all / (entry["ms_per_step"] / 1e3)
        entry["oracle"] = orc
        entry["parity"] = parity_errors(outputs[name], ref)
        del reqs, ref


class OracleSlices:
    """`--impl reference`: the float64 oracle, as it stands, on slices of the link step.

    Set-up (untimed): the workload's inputs and the oracle's spliced context of every
    request.  Slice i of m: the oracle's re-rotation of the chunks c >= 1 with
    c = i (mod m) and its attention on the recomputed rows j = i (mod m) of every
    request.  A slice is timed whole and credited with 1/m of the step's context
    tokens, so ms_per_step is the time the slice really took."""

    def __init__(self, wl, m=8):
        import torch

        import oracle.pic_oracle as O
        self.O, self.wl, self.m = O, wl, m
        self.threads = torch.get_num_threads()
        self.reqs = []
        for ck, cv, q, k, qr, kn, vn in _oracle_inputs(wl):
            K, V, rows, starts, _ = O.splice_context(ck, cv, q, k, kn, vn, wl.theta, wl.dtype)
            q_rot = O.round_to(O.rope(qr, rows, wl.theta), wl.dtype) if len(rows) else None
            self.reqs.append((ck, starts, rows, q_rot, K, V))

    def run(self, i):
        O, wl, m = self.O, self.wl, self.m
        t0 = time.perf_counter()
        for ck, starts, rows, q_rot, K, V in self.reqs:
            for c in range(1, len(ck)):
                if c % m == i % m:
                    O.rerotate_k(ck[c], int(starts[c]), wl.theta, wl.dtype)
            which = list(range(i % m, len(rows), m))
            if which:
                O.attention_rows(q_rot, rows, K, V, 1.0 / np.sqrt(wl.d), which=which)
        return time.perf_counter() - t0

    def describe(self):
        return (f"float64 oracle as it stands on 1/{self.m} slices of the step: re-rotation of every "
                f"{self.m}-th chunk and attention of every {self.m}-th recomputed row of each request (offset "
                f"cycling over steps); each slice timed whole and credited with 1/{self.m} of the context "
                f"tokens; spliced context built once, untimed; {self.threads} threads")


def run_reference(args):
    wl = _workload(args.workload)
    tokens = wl.total_tokens()
    sl = OracleSlices(wl)
    for i in range(args.warmup):
        sl.run(i)
    times = [sl.run(args.warmup + i) for i in range(args.steps)]
    step_s = statistics.mean(times)
    value = tokens / sl.m / step_s
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded inputs as the GPU arm)",
        "config": {"workload": wl.name, "tokens": tokens, "tokens_per_step": tokens / sl.m},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": sl.threads, "kind": "oracle",
                         "sample": sl.describe() + f"; mean over {args.steps} slices"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long_context_100x1000")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="time the headline workload only")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    result, batch, outputs = run_gpu(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            cpu_legs(result, batch.wl, outputs)
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
