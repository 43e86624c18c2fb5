"""Benchmark of the paged decode step on the mixed-length serving batch.

Workload (seeded, synthetic; no dataset): an OPT-13B-shaped attention layer,
40 heads x head_dim 128, fp16, block size 16, 256 sequences whose prompt
lengths are lognormal (median 200, cap 1536) and whose outputs are lognormal
(median 250), total context capped at 2048, block tables fragmented across a
shuffled pool, contexts over 512 tokens on the split-context path.  The
batch runs as a steady-state continuous batch: every step appends one token
to every sequence; a sequence that reaches its drawn total length is freed
and replaced by a newly drawn one, so the length mix stays stationary over
thousands of steps.  (A newcomer's prompt K/V is not written -- prefill is
another kernel -- its blocks keep the finite values of earlier occupants.)

One step = the whole hot path: host block manager (pa_decode_step_prepare:
append and table export), one packed metadata upload, copy-on-write copies
(none in this workload), the slot write of the new K/V, and decode attention
(split + merge).  ``value`` is K/V token positions attended per second
(sum of context lengths / step time), inputs resident in HBM (the K/V
working set, ~3.5 GB, is far larger than L2, so no L2 flush is needed).
``e2e`` repeats the step with q / k / v uploaded from pinned host memory and
the output read back to host every step, wall-clock timed.  After the timed
region, ``kernels`` adds the 64-sequence batch (context uniform in
[128, 2048]) against the HBM roof, parallel sampling with copy-on-write
(L2-resident, GB/s only) and causal prefill of the mixed batch's prompts
against its binding roof.
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

METRIC = "paged decode-attn seq-tokens/s (1 GB300) + achieved HBM GB/s vs ~8 TB/s peak"
UNIT = "seq-tokens/s"


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _code_sha256(path: str) -> str:
    """sha256 of a C/CUDA source with its comments and whitespace removed, so
    that a profile taken on a kernel stays attached to it across comment
    edits (any change to the code itself changes the hash)."""
    import hashlib
    import re
    src = open(path).read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return hashlib.sha256(" ".join(src.split()).encode()).hexdigest()


def _kernel_traffic(kernel_src: str, name: str = "decode_attention_traffic.json"):
    """The committed ncu traffic summary of a kernel (DRAM bytes of one
    captured launch of a small case over that launch's algorithmic bytes), if
    it was taken on the current code of the kernel (else None)."""
    p = os.path.join(ROOT, "profiles", name)
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("code_sha256") == _code_sha256(kernel_src):
            return d
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.out.seek(0)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_across_ranks(to_sum, to_max, device):
    """Whole-job numbers: work summed over ranks, times maxed over ranks
    (no-op without an initialised process group)."""
    import torch
    import torch.distributed as dist

    tot = torch.tensor([float(x) for x in to_sum], dtype=torch.float64, device=device)
    mx = torch.tensor([float(x) for x in to_max], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(tot, op=dist.ReduceOp.SUM)
        dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    return tot.tolist(), mx.tolist()


def _pool_setup(pk, w):
    desc = pk.PoolDesc(w.num_blocks, w.block_size, num_layers=1, num_heads=w.num_heads,
                       head_dim=w.head_dim, partition_tokens=w.split_tokens,
                       free_order=w.free_order)
    pool = pk.pa_pool_create(desc)
    for i, n in enumerate(w.prompt_lens):
        pk.pa_seq_add(pool, i, n, want_slots=False)
    return desc, pool


class SteadyBatch:
    """Host side of the continuous batch: replaces finished sequences.
    Newcomers' (prompt, target) lengths are seeded inputs, drawn in blocks.
    A sequence is replaced at the first step whose admission sees it hold at
    least its target length; that step is known when it is admitted, so
    each step looks up only its own list (in ascending batch index)."""

    DRAW_BLOCK = 4096

    def __init__(self, pk, pool, w, rng):
        self.pk, self.pool, self.rng = pk, pool, rng
        self.prompt = np.array(w.prompt_lens, np.int64)   # tokens held when admitted
        self.target = np.array(w.targets, np.int64)
        self.since = np.zeros(len(self.prompt), np.int64)  # step of admission
        self.step = 0
        self.due = {}
        for i in range(len(self.prompt)):
            self._schedule(i, 0)
        self.next_id = len(w.prompt_lens)
        self.replaced = 0
        self._draws, self._next_draw = None, self.DRAW_BLOCK

    @property
    def held(self):
        """Tokens each sequence of the batch holds now."""
        return self.prompt + (self.step - self.since)

    def _schedule(self, i, first):
        # held at step self.step + j is prompt + j; replaced at the first
        # j >= first with prompt + j >= target
        j = max(first, int(self.target[i] - self.prompt[i]))
        self.due.setdefault(self.step + j, []).append(i)

    def _draw(self):
        if self._next_draw == self.DRAW_BLOCK:
            from workloads import draw_mixed_sequences
            p, t = draw_mixed_sequences(self.rng, self.DRAW_BLOCK)
            self._draws, self._next_draw = (p.tolist(), t.tolist()), 0
        i = self._next_draw
        self._next_draw += 1
        return self._draws[0][i], self._draws[1][i]

    def admit(self, ids):
        due = self.due.pop(self.step, None)
        if not due:
            return
        for i in sorted(due):
            self.pk.pa_seq_free(self.pool, int(ids[i]))
            prompt, target = self._draw()
            self.pk.pa_seq_add(self.pool, self.next_id, prompt, want_slots=False)
            ids[i] = self.next_id
            self.next_id += 1
            self.prompt[i], self.target[i], self.since[i] = prompt, target, self.step
            self._schedule(i, 1)
            self.replaced += 1

    def appended(self):
        self.step += 1


def other_rows(args) -> dict:
    """Short runs of the other measured rows for the default bench line:
    the 40-layer pool-filling step (plain and with beam groups sharing
    blocks), beam-search churn and prefix caching, each summarised from its
    own mode's line."""
    import copy

    import torch

    out = {}
    a = copy.copy(args)
    a.warmup, a.steps, a.beam, a.prompts = 3, 10, False, 0
    f = run_full40(a, quiet=True)
    out["full_40l_step"] = {
        "workload": f["config"]["workload"], "sequences": f["config"]["sequences"],
        "pool_bytes": f["config"]["pool_bytes"], "steps": a.steps,
        "seq_tokens_per_s": f["value"], "ms_per_step": f["ms_per_step"],
        "attention_GB/s": f["roofline"]["achieved"], "frac": f["roofline"]["frac"],
        "peak": f["roofline"]["peak"], "bound": "hbm",
        "algorithmic_bytes_per_step": f["roofline"]["algorithmic_bytes_per_step"]}
    torch.cuda.empty_cache()
    a.beam = True
    f = run_full40(a, quiet=True)
    out["full_40l_beam_step"] = {
        "workload": f["config"]["workload"], "sequences": f["config"]["sequences"],
        "pool_bytes": f["config"]["pool_bytes"], "steps": a.steps,
        "logical_over_unique_blocks": f["config"]["logical_over_unique_blocks"],
        "copies_per_step": f["config"]["copies_per_step"],
        "seq_tokens_per_s": f["value"], "ms_per_step": f["ms_per_step"],
        "logical_attention_GB/s": f["roofline"]["achieved"],
        "note": "logical bytes count blocks shared by a group's beams once per beam; the "
                "beams of a group re-read them from L2, so this is not an HBM roofline"}
    a.beam = False
    torch.cuda.empty_cache()
    a.warmup, a.steps = 3, 20
    b = run_beam_churn(a, quiet=True)
    out["beam_churn"] = {"workload": b["config"]["workload"], "steps": a.steps,
                         "ms_per_step": b["ms_per_step"], "seq_tokens_per_s": b["value"],
                         "per_step": b["per_step"], "host_us_per_step": b["host_us_per_step"],
                         "logical_attention_GB/s": b["logical_attention_GB/s"]}
    torch.cuda.empty_cache()
    a.warmup, a.steps = 2, 5
    c = run_prefix_cache(a, quiet=True)
    out["prefix_cache"] = {"workload": c["config"]["workload"], "steps": a.steps,
                           "speedup": c["speedup"], "cached": c["cached"],
                           "uncached": c["uncached"]}
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    import paged_kv_cache_106_gb300 as pk
    import workloads as wl
    from paged_kv_cache_106_gb300.step import DecodeStepRunner

    ws, rank, local = _dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)

    w = wl.mixed_b256(batch=args.batch, steady_state=True)
    if args.partition:
        w.split_tokens = args.partition
    H, D, B = w.num_heads, w.head_dim, w.block_size
    desc, pool = _pool_setup(pk, w)
    ids = np.arange(len(w.prompt_lens), dtype=np.int32)
    S = len(ids)
    max_blocks = -(-wl.CTX_CAP // B)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed + 1000 * rank)
    kc = torch.empty((w.num_blocks, H, B, D), dtype=torch.float16, device=dev)
    vc = torch.empty_like(kc)
    kc.normal_(generator=gen)
    vc.normal_(generator=gen)
    q = torch.randn((S, H, D), dtype=torch.float16, device=dev, generator=gen)
    k_new = torch.randn((S, H, D), dtype=torch.float16, device=dev, generator=gen)
    v_new = torch.randn((S, H, D), dtype=torch.float16, device=dev, generator=gen)
    out = torch.empty((S, H, D), dtype=torch.float16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    runner = DecodeStepRunner(pool, desc, ids, max_blocks, device=dev, stream=stream)
    runner.ids = ids                       # the batch edits ids in place on replacement
    batch = SteadyBatch(pk, pool, w, np.random.default_rng(w.seed + 7 + rank))
    merge = pk.pa_decode_workspace_bytes(S, max_blocks, desc) > 0
    bytes_fixed = S * H * D * 2 * 2       # q read + o written
    bytes_new = S * H * D * 2 * 4         # the new tokens' K and V read and stored in the cache

    dump = [] if args.dump_steps else None

    host_s = []

    def step(ev_pair=None, stats=None):
        h0 = time.perf_counter()
        batch.admit(ids)
        h_admit = time.perf_counter() - h0
        n_cp = runner.prepare()
        if stats is not None:
            host_s.append((h_admit, runner.host_seconds))
        batch.appended()
        ctx = runner.ctx_host.astype(np.int64)
        if dump is not None:
            nblk_d = (ctx + B - 1) // B
            dump.append({"tokens": int(ctx.sum()),
                         "attn_bytes": int(ctx.sum()) * H * D * 4 + int(nblk_d.sum()) * 4
                         + S * 4 + bytes_fixed + bytes_new})
        runner.copy_blocks([kc], [vc])
        if ev_pair is not None:
            ev_pair[0].record(stream)
        # the new tokens' slot write inside the attention launch
        runner.step_attention(out, q, k_new, v_new, kc, vc, w.scale)
        if ev_pair is not None:
            ev_pair[1].record(stream)
        if stats is not None:
            stats["tokens"] += int(ctx.sum())
            nblk = (ctx + B - 1) // B
            stats["attn_bytes"] += int(ctx.sum()) * H * D * 2 * 2 + int(nblk.sum()) * 4 + S * 4 \
                + bytes_fixed + bytes_new
            stats["launches"] += 1 + (1 if merge else 0) + (1 if n_cp else 0)
            stats["copies"] += n_cp

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()

    sampler = ClockSampler(local)
    sampler.start()
    stats = {"tokens": 0, "attn_bytes": 0, "launches": 0, "copies": 0}
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2))
           for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i], stats)
        t1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    clocks = sampler.stop()
    if dump is not None and rank == 0:
        with open(args.dump_steps, "w") as f:
            json.dump({"warmup": args.warmup, "steps": dump}, f)
    elapsed = t0.elapsed_time(t1) / 1e3
    attn_ms = [e[0].elapsed_time(e[1]) for e in evs]
    copy_stats = time_copy_blocks(pk, pool, desc, w, kc, vc, stream) if rank == 0 else None
    # the step's slot write alone, 50 launches back to back between two events
    # (inside the step loop each launch also carries its own events)
    with torch.cuda.stream(stream):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(50):
            runner.write_kv(k_new, v_new, kc, vc)
        b.record(stream)
    torch.cuda.synchronize()
    write_b2b_us = a.elapsed_time(b) * 1e3 / 50
    swap_stats = time_swap_blocks(pk, desc, w, kc, vc, stream) if rank == 0 else None
    assert runner.status.item() == 0, f"device status {runner.status.item()}"

    # ---- e2e: host buffers, H2D of q/k/v and D2H of o inside every step
    h_q = torch.empty((S, H, D), dtype=torch.float16, pin_memory=True)
    h_k = torch.empty_like(h_q).pin_memory()
    h_v = torch.empty_like(h_q).pin_memory()
    h_o = torch.empty_like(h_q).pin_memory()
    h_q.copy_(q.cpu()), h_k.copy_(k_new.cpu()), h_v.copy_(v_new.cpu())
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    e2e_tokens = 0
    meta_bytes = runner.nbytes
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    # Serving-loop order, two steps deep: while the GPU runs step i, the host
    # prepares step i+1 (sequence replacement, block manager) and enqueues it
    # (q/k/v upload from pinned memory, metadata, kernels, output read-back
    # into the other pinned buffer); then it waits for step i's output to be
    # on the host.  Stream order keeps each step's inputs and output intact.
    h_out = [h_o, torch.empty_like(h_o).pin_memory()]
    # untimed passes through the copy path: the first transfers through freshly
    # pinned pages run several times slower than the steady state (measured on
    # the Grace host: 6-37 GB/s for the first two, then 190-210 GB/s)
    with torch.cuda.stream(stream):
        for _ in range(3):
            q.copy_(h_q, non_blocking=True)
            k_new.copy_(h_k, non_blocking=True)
            v_new.copy_(h_v, non_blocking=True)
            for h in h_out:
                h.copy_(out, non_blocking=True)
    torch.cuda.synchronize()

    def host_prep():
        batch.admit(ids)
        runner.prepare_host()
        batch.appended()

    # the step's q/k/v go up on a copy stream into device set i & 1 and its
    # output comes back on another, ordered by events with the compute stream,
    # so these copies overlap the previous step's kernels; the block-table
    # upload (small, one device buffer) stays on the compute stream, after the
    # previous step's kernels that read it
    bufs = [(q, k_new, v_new, out), tuple(torch.empty_like(q) for _ in range(4))]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "comp", "out")}
    used = [False, False]

    def enqueue(i):
        sidx = i & 1
        qq, kk, vv, oo = bufs[sidx]
        if used[sidx]:
            s_in.wait_event(ev["comp"][sidx])      # step i - 2 has read this set's inputs
        with torch.cuda.stream(s_in):
            qq.copy_(h_q, non_blocking=True)
            kk.copy_(h_k, non_blocking=True)
            vv.copy_(h_v, non_blocking=True)
        ev["in"][sidx].record(s_in)
        stream.wait_event(ev["in"][sidx])
        if used[sidx]:
            stream.wait_event(ev["out"][sidx])     # step i - 2's output has left this set
        runner.upload()
        n_tok = int(runner.ctx_host.sum())
        runner.copy_blocks([kc], [vc])
        runner.step_attention(oo, qq, kk, vv, kc, vc, w.scale)
        ev["comp"][sidx].record(stream)
        s_out.wait_event(ev["comp"][sidx])
        with torch.cuda.stream(s_out):
            h_out[sidx].copy_(oo, non_blocking=True)
        ev["out"][sidx].record(s_out)
        used[sidx] = True
        return ev["out"][sidx], n_tok

    w0 = time.perf_counter()
    with torch.cuda.stream(stream):
        host_prep()
        pending = enqueue(0)
        for i in range(e2e_steps):
            nxt = None
            if i + 1 < e2e_steps:
                host_prep()
                nxt = enqueue(i + 1)
            pending[0].synchronize()       # step i's output is on the host
            e2e_tokens += pending[1]
            pending = nxt
    e2e_time = time.perf_counter() - w0

    # ---- reduce over ranks: max time, summed work
    (tokens_all, e2e_tokens_all), (elapsed_max, e2e_max) = reduce_across_ranks(
        [stats["tokens"], e2e_tokens], [elapsed, e2e_time], dev)

    # ---- the other measured rows, on rank 0, after the timed region: the
    # 64-sequence batch, parallel sampling with copy-on-write, and causal
    # prefill of the mixed batch's prompts against its binding roof
    extra = {}
    if rank == 0 and not args.no_extra:
        extra["decode_opt13b_b64"] = decode_b64_stats(dev)
        extra["parallel_sampling"] = parallel_sampling_stats(dev)
        pb = PrefillBatch(dev)
        pf_work = (f"causal prefill of {len(pb.lens)} whole prompts (lognormal, median 200, "
                   f"cap 1536; {pb.T} tokens), OPT-13B layer 40x128, block 16")
        _, fs_ms = pb.time_fused(20, 3)
        fs = pb.roofline(fs_ms, fused=True)
        fs.update({"workload": pf_work + "; the prompts' slot write and attention in one launch",
                   "launches": 20, "prompt_tokens_per_s": pb.T / (fs_ms / 1e3)})
        extra["pa_prefill_step_attention"] = fs
        _, pf_ms, pf_wkv_ms = pb.time_steps(20, 3)
        pf = pb.roofline(pf_ms)
        pf.update({"workload": pf_work + "; attention alone (after pa_write_kv)", "launches": 20,
                   "prompt_tokens_per_s": pb.T / (pf_ms / 1e3),
                   "slot_write_us_for_the_prompts": pf_wkv_ms * 1e3})
        extra["pa_prefill_attention"] = pf
        pb.close()
        del pb
        torch.cuda.empty_cache()
        extra.update(other_rows(args))

    if rank == 0:
        peak, peak_kind = _peaks()
        attn_avg_s = sum(attn_ms) / len(attn_ms) / 1e3
        achieved = stats["attn_bytes"] / args.steps / attn_avg_s / 1e9
        src = os.path.join(ROOT, "paged_kv_cache_106_gb300", "csrc", "decode_attention.cu")
        traffic = _kernel_traffic(src)
        line = {
            "metric": METRIC,
            "value": tokens_all / elapsed_max,
            "unit": UNIT,
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": elapsed_max * 1e3 / args.steps,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f16 (fp32 accumulate)",
            "data": "synthetic (seeded N(0,1) fp16 K/V/q; lognormal length mix)",
            "config": {
                **_decode_config(w, ws),
                "mean_ctx": stats["tokens"] / args.steps / S,
                "sequences_replaced": batch.replaced,
                "l2": "working set ~%.1f GB per step >> 129 MB L2, no flush"
                      % (stats["attn_bytes"] / args.steps / 1e9),
            },
            "gpu_launches": stats["launches"],
            "roofline": {
                "bound": "hbm",
                "kernel": "paged_decode_persistent + paged_merge_kernel (pa_decode_step_attention: the new tokens' slot write and attention)",
                "achieved": achieved,
                "peak": peak,
                "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "unit": "GB/s",
                "frac": achieved / peak,
                "frac_of_nominal_7900": achieved / 7900.0,
                # DRAM bytes of the small-case capture per algorithmic byte, times
                # this launch's algorithmic bytes
                "traffic": None if traffic is None else
                traffic["traffic_over_algorithmic"] * stats["attn_bytes"] / args.steps,
                "traffic_from": None if traffic is None else traffic["capture"],
                "traffic_over_algorithmic": None if traffic is None
                else traffic["traffic_over_algorithmic"],
                "algorithmic_bytes_per_launch": stats["attn_bytes"] / args.steps,
                "attn_ms_per_launch": attn_avg_s * 1e3,
                "attn_share_of_step": attn_avg_s / (elapsed_max / args.steps),
            },
            "decode_tokens_per_s": ws * S * args.steps / elapsed_max,
            "kernels": {
                "pa_write_kv": {
                    "us_per_launch": write_b2b_us,
                    "algorithmic_bytes": 2 * 2 * S * H * D * 2 + 8 * S,
                    "GB/s": (2 * 2 * S * H * D * 2 + 8 * S) / (write_b2b_us / 1e6) / 1e9,
                    "in_step": "none: the timed decode step stores its new tokens inside the "
                               "attention launch (pa_decode_step_attention)",
                    "note": "the separate slot write of the batch's new K/V (what a caller of "
                            "pa_write_kv runs): 50 launches back to back between two CUDA events, "
                            "launch gaps included",
                },
                **extra,
                "pa_copy_blocks": copy_stats,
                "pa_swap_blocks": swap_stats,
                "host_block_manager": {
                    "us_per_step": 1e6 * sum(a + b for a, b in host_s) / len(host_s),
                    "admission_us_per_step": 1e6 * sum(a for a, _ in host_s) / len(host_s),
                    "step_prepare_us_per_step": 1e6 * sum(b for _, b in host_s) / len(host_s),
                    "note": "host wall clock per step: free/admit finished sequences, then "
                            "pa_decode_step_prepare_rows (one token per sequence, lengths and "
                            "the changed table rows into the pinned staging buffer); waits on the "
                            "GPU excluded",
                },
            },
            "e2e": {
                "value": e2e_tokens_all / e2e_max,
                "unit": UNIT,
                "h2d_bytes_per_step": 3 * S * H * D * 2 + meta_bytes,
                "d2h_bytes_per_step": S * H * D * 2,
                "steps": e2e_steps,
                "timing": "wall clock; every step uploads q/k/v and reads o back; two "
                          "steps in flight (step i+1 prepared and enqueued while step i runs; "
                          "q/k/v uploads and the read-back on copy streams, overlapping the "
                          "previous step's kernels)",
            },
            "clocks": clocks,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args.cpu_seconds, args.cpu_seqs)
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    pk.pa_pool_destroy(pool)


def time_copy_blocks(pk, pool, desc, w, kc, vc, stream, n_pairs=256, reps=50):
    """Copy-on-write-sized batch of block copies (one layer, K and V): live
    blocks into free ones, timed with CUDA events on the launching stream."""
    import torch

    free = pk.pa_pool_free_queue(pool, w.num_blocks)
    refs = pk.pa_pool_refcounts(pool, w.num_blocks)
    used = np.nonzero(refs > 0)[0]
    n = int(min(n_pairs, len(free), len(used)))
    if n == 0:
        return None
    rng = np.random.default_rng(5)
    pairs = np.stack([rng.choice(used, n, replace=False), free[:n]], axis=1).astype(np.int32)
    d_pairs = torch.from_numpy(pairs).to(kc.device)
    status = torch.zeros(1, dtype=torch.int32, device=kc.device)
    with torch.cuda.stream(stream):
        for _ in range(3):
            pk.pa_copy_blocks([kc], [vc], d_pairs, desc, status=status, stream=stream)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            pk.pa_copy_blocks([kc], [vc], d_pairs, desc, status=status, stream=stream)
        b.record(stream)
    torch.cuda.synchronize()
    assert status.item() == 0
    us = a.elapsed_time(b) * 1e3 / reps
    nbytes = n * 2 * w.num_heads * w.block_size * w.head_dim * 2 * 2 + n * 8
    return {"pairs": n, "layers": 1, "us_per_launch": us, "algorithmic_bytes": nbytes,
            "GB/s": nbytes / (us / 1e6) / 1e9,
            "note": "blocks of live sequences copied into free blocks, K and V (read + write)"}


def run_full40(args, quiet: bool = False):
    """The 40-layer decode step over a pool-filling cache (one GPU).

    The K/V pool takes min(120 GB, half the free device memory); sequences
    with context uniform in [512, 2048] fill it; with --beam, groups of 4 beams
    share the first 55 % of their blocks.  One step = host block manager,
    metadata upload, block copies (every layer) and, per layer, slot write and
    decode attention.  Contexts grow by one token per step (warm-up + timed
    steps must stay within the one spare block per sequence: <= 16).
    """
    import torch

    import paged_kv_cache_106_gb300 as pk
    import workloads as wl
    from paged_kv_cache_106_gb300.step import DecodeStepRunner, admit_workload

    ws, rank, local = _dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    free, _ = torch.cuda.mem_get_info(dev)
    pool_bytes = int(min(120e9, 0.5 * free))
    w = wl.full_40l(pool_bytes, beam=args.beam)
    L, H, D, B = w.num_layers, w.num_heads, w.head_dim, w.block_size
    if args.warmup + args.steps > 16:
        raise SystemExit("full_40l: warm-up + steps must be <= 16 (one spare block per sequence)")
    desc = pk.PoolDesc(w.num_blocks, B, num_layers=L, num_heads=H, head_dim=D,
                       partition_tokens=w.split_tokens, free_order=w.free_order)
    pool = pk.pa_pool_create(desc)
    ids = np.array(admit_workload(pool, w), dtype=np.int32)
    S = len(ids)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    kc_all = torch.empty((L, w.num_blocks, H, B, D), dtype=torch.float16, device=dev)
    vc_all = torch.empty_like(kc_all)
    kc_all.normal_(generator=gen)
    vc_all.normal_(generator=gen)
    kcs, vcs = list(kc_all.unbind(0)), list(vc_all.unbind(0))
    q = torch.randn((S, H, D), dtype=torch.float16, device=dev, generator=gen)
    k_new, v_new = torch.randn_like(q), torch.randn_like(q)
    out = torch.empty_like(q)
    stream = torch.cuda.Stream(device=dev)
    max_blocks = -(-(wl.CTX_CAP + 16) // B)
    runner = DecodeStepRunner(pool, desc, ids, max_blocks, device=dev, stream=stream)
    refs = pk.pa_pool_refcounts(pool, w.num_blocks)

    def step(evs=None, stats=None):
        runner.prepare()
        ctx = runner.ctx_host.astype(np.int64)
        runner.copy_blocks(kcs, vcs)
        for l in range(L):
            if evs is not None:
                evs[l][0].record(stream)
            runner.step_attention(out, q, k_new, v_new, kcs[l], vcs[l], w.scale)
            if evs is not None:
                evs[l][1].record(stream)
        if stats is not None:
            nblk = (ctx + B - 1) // B
            stats["tokens"] += int(ctx.sum()) * L
            stats["attn_bytes"] += L * (int(ctx.sum()) * H * D * 4 + int(nblk.sum()) * 4 + S * 4
                                        + S * H * D * 4 + S * H * D * 8)
            stats["copies"] += runner.n_copies

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    stats = {"tokens": 0, "attn_bytes": 0, "copies": 0}
    evs = [[tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(L)]
           for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(args.steps):
            step(evs[i], stats)
        t1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    assert runner.status.item() == 0, f"device status {runner.status.item()}"
    elapsed = t0.elapsed_time(t1) / 1e3
    attn_s = sum(a.elapsed_time(b) for layer in evs for a, b in layer) / 1e3
    peak, peak_kind = _peaks()
    achieved = stats["attn_bytes"] / attn_s / 1e9
    line = {
        "metric": METRIC, "value": stats["tokens"] / elapsed, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": "full 40-layer OPT-13B-shaped decode step, pool-filling cache"
                               + (", beam groups of 4 sharing 55 % of blocks" if args.beam else ""),
                   "pool_bytes": pool_bytes, "pool_blocks": w.num_blocks, "sequences": S,
                   "layers": L, "mean_ctx": stats["tokens"] / L / args.steps / S,
                   "shared_blocks": int((refs > 1).sum()),
                   "logical_over_unique_blocks": float((refs.sum()) / max(1, (refs > 0).sum())),
                   "copies_per_step": stats["copies"] / args.steps},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": achieved / peak,
                     "algorithmic_bytes_per_step": stats["attn_bytes"] / args.steps,
                     "attn_share_of_step": attn_s / elapsed,
                     "note": "K/V counted once per referencing sequence (shared blocks once "
                             "per beam): logical bytes"},
        "clocks": clocks,
    }
    if not quiet:
        print(json.dumps(line), flush=True)
    pk.pa_pool_destroy(pool)
    return line


def time_swap_blocks(pk, desc, w, kc, vc, stream, n_pairs=256, reps=20):
    """Swap-sized batches of block copies between the GPU cache and swap space
    in pinned host memory (over NVLink-C2C), each direction, one launch each."""
    import torch

    hk = torch.empty((n_pairs, w.num_heads, w.block_size, w.head_dim), dtype=torch.float16,
                     pin_memory=True)
    hv = torch.empty_like(hk).pin_memory()
    rng = np.random.default_rng(6)
    src = rng.choice(w.num_blocks, n_pairs, replace=False)
    out_pairs = torch.from_numpy(np.stack([src, np.arange(n_pairs)], 1).astype(np.int32)).to(kc.device)
    in_pairs = torch.from_numpy(np.stack([np.arange(n_pairs), src], 1).astype(np.int32)).to(kc.device)
    status = torch.zeros(1, dtype=torch.int32, device=kc.device)
    res = {}
    for name, args in (("gpu_to_host", ([kc], [vc], w.num_blocks, [hk], [hv], n_pairs, out_pairs)),
                       ("host_to_gpu", ([hk], [hv], n_pairs, [kc], [vc], w.num_blocks, in_pairs))):
        with torch.cuda.stream(stream):
            for _ in range(3):
                pk.pa_swap_blocks(*args, desc, status=status, stream=stream)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                pk.pa_swap_blocks(*args, desc, status=status, stream=stream)
            b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / reps
        moved = n_pairs * 2 * w.num_heads * w.block_size * w.head_dim * 2
        res[name] = {"us_per_launch": us, "bytes_moved": moved, "GB/s": moved / (us / 1e6) / 1e9}
    assert status.item() == 0
    res["pairs"] = n_pairs
    res["note"] = "pa_swap_blocks: K and V of 256 blocks, one layer, one launch per direction"
    return res


def decode_b64_stats(dev, steps: int = 200, warmup: int = 5) -> dict:
    """The 64-sequence OPT-13B batch (context uniform in [128, 2048], pool
    1.25x the blocks needed, shuffled free queue): decode steps through the
    runner, attention per launch timed with CUDA events on its stream, its
    algorithmic bytes from the step's contexts (K/V of every attended token,
    tables, lengths, q read, o written)."""
    import torch

    import paged_kv_cache_106_gb300 as pk
    import workloads as wl
    from paged_kv_cache_106_gb300.step import DecodeStepRunner

    w = wl.opt13b_b64()
    H, D, B = w.num_heads, w.head_dim, w.block_size
    desc, pool = _pool_setup(pk, w)
    S = len(w.prompt_lens)
    ids = np.arange(S, dtype=np.int32)
    max_blocks = -(-(max(w.prompt_lens) + warmup + steps + 1) // B)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    kc = torch.empty((w.num_blocks, H, B, D), dtype=torch.float16, device=dev).normal_(generator=gen)
    vc = torch.empty_like(kc).normal_(generator=gen)
    q, k_new, v_new = (torch.randn((S, H, D), dtype=torch.float16, device=dev, generator=gen)
                       for _ in range(3))
    out = torch.empty_like(q)
    stream = torch.cuda.Stream(device=dev)
    runner = DecodeStepRunner(pool, desc, ids, max_blocks, device=dev, stream=stream)
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(steps)]
    nbytes, tokens = 0, 0
    with torch.cuda.stream(stream):
        for i in range(warmup + steps):
            runner.prepare()
            ctx = runner.ctx_host.astype(np.int64)
            runner.copy_blocks([kc], [vc])
            j = i - warmup
            if j >= 0:
                evs[j][0].record(stream)
            runner.step_attention(out, q, k_new, v_new, kc, vc, w.scale)
            if j >= 0:
                evs[j][1].record(stream)
                tokens += int(ctx.sum())
                nbytes += int(ctx.sum()) * H * D * 4 + int(((ctx + B - 1) // B).sum()) * 4 \
                    + S * 4 + S * H * D * 4 + S * H * D * 8
    torch.cuda.synchronize()
    assert runner.status.item() == 0, runner.status.item()
    ms = sum(a.elapsed_time(b) for a, b in evs) / steps
    peak, kind = _peaks()
    achieved = nbytes / steps / (ms / 1e3) / 1e9
    pk.pa_pool_destroy(pool)
    return {"workload": "64 sequences, OPT-13B layer 40x128, block 16, context uniform in "
                        "[128, 2048], pool 1.25x the blocks needed, shuffled free queue",
            "bound": "hbm", "launches": steps, "mean_ctx": tokens / steps / S,
            "us_per_launch": ms * 1e3, "algorithmic_bytes_per_launch": nbytes / steps,
            "achieved": achieved, "peak": peak, "peak_kind": f"{kind} hbm_gbs", "unit": "GB/s",
            "frac": achieved / peak, "seq_tokens_per_s": tokens / steps / (ms / 1e3),
            "l2": "K/V working set %.2f GB per launch >> 129 MB L2, no flush" % (nbytes / steps / 1e9)}


def parallel_sampling_stats(dev) -> dict:
    """16 prompts (lognormal, median 160, cap 1024) x 4 samples forked from
    them, 64 decode steps: copy-on-write of each shared partial last block,
    slot write, attention.  Per step the GPU time of its kernels (copies,
    slot write, attention) from CUDA events.  Logical bytes count a shared
    block once per sequence that reads it; unique bytes once.  The unique
    working set is a few hundred MB at most and the samples re-read the
    shared prompt blocks from L2, so the GB/s are not an HBM roofline."""
    import torch

    import paged_kv_cache_106_gb300 as pk
    import workloads as wl
    from paged_kv_cache_106_gb300.step import DecodeStepRunner

    res = None
    for episode in range(2):              # the first one warms up; the second is timed
        w = wl.parallel_sampling()
        H, D, B = w.num_heads, w.head_dim, w.block_size
        desc, pool = _pool_setup(pk, w)
        ids = list(range(len(w.prompt_lens)))
        nxt = len(ids)
        for root, extra in w.forks:
            for _ in range(extra):
                pk.pa_seq_fork(pool, root, nxt)
                ids.append(nxt)
                nxt += 1
        S = len(ids)
        max_blocks = -(-(max(w.prompt_lens) + w.decode_steps + 1) // B)
        gen = torch.Generator(device=dev)
        gen.manual_seed(w.seed)
        kc = torch.empty((w.num_blocks, H, B, D), dtype=torch.float16, device=dev).normal_(generator=gen)
        vc = torch.empty_like(kc).normal_(generator=gen)
        q, k_new, v_new = (torch.randn((S, H, D), dtype=torch.float16, device=dev, generator=gen)
                           for _ in range(3))
        out = torch.empty_like(q)
        stream = torch.cuda.Stream(device=dev)
        runner = DecodeStepRunner(pool, desc, ids, max_blocks, device=dev, stream=stream)
        evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3))
               for _ in range(w.decode_steps)]
        logical, unique, copies, tokens = 0, 0, 0, 0
        with torch.cuda.stream(stream):
            for i in range(w.decode_steps):
                runner.prepare()
                ctx = runner.ctx_host.astype(np.int64)
                tables = runner._views(runner.host[(runner.i - 1) & 1])[2]
                evs[i][0].record(stream)
                runner.copy_blocks([kc], [vc])
                evs[i][1].record(stream)
                runner.step_attention(out, q, k_new, v_new, kc, vc, w.scale)
                evs[i][2].record(stream)
                copies += runner.n_copies
                tokens += int(ctx.sum())
                logical += int(ctx.sum()) * H * D * 4
                blocks = np.unique(tables[tables >= 0])
                unique += len(blocks) * B * H * D * 4      # whole blocks, an upper bound
        torch.cuda.synchronize()
        assert runner.status.item() == 0, runner.status.item()
        n = w.decode_steps
        step_ms = sum(a.elapsed_time(c) for a, _, c in evs) / n
        attn_ms = sum(b.elapsed_time(c) for _, b, c in evs) / n
        res = {"workload": "16 prompts lognormal (median 160, cap 1024) x 4 samples sharing the "
                           "prompt blocks, 64 decode steps, OPT-13B layer 40x128, block 16",
               "sequences": S, "steps": n, "cow_copies": copies,
               "us_per_step": step_ms * 1e3, "attention_us_per_step": attn_ms * 1e3,
               "seq_tokens_per_s": tokens / n / (attn_ms / 1e3),
               "logical_GB/s": logical / n / (attn_ms / 1e3) / 1e9,
               "unique_GB/s": unique / n / (attn_ms / 1e3) / 1e9,
               "unique_bytes_per_step": unique / n,
               "l2_resident": True,
               "note": "GPU time of the step's kernels (copy-on-write copies, then the slot "
                       "write and attention in one call); logical bytes count shared blocks once per reading "
                       "sequence, unique bytes once (whole blocks); the samples' re-reads of "
                       "shared blocks hit L2, so this is not an HBM roofline"}
        pk.pa_pool_destroy(pool)
    return res


def run_beam_churn(args, quiet: bool = False):
    """Beam-search churn: 64 requests x 4 beams (OPT-13B layer shapes), every
    step = prune (fork repeated survivors, free the rest), host block
    manager, copy-on-write copies, slot write, decode attention."""
    import torch

    import paged_kv_cache_106_gb300 as pk
    import workloads as wl
    from paged_kv_cache_106_gb300.step import BeamGroups, DecodeStepRunner

    _, _, local = _dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    churn = wl.beam_churn(groups=64, width=4)
    H, D, B = wl.OPT13B_HEADS, wl.OPT13B_HEAD_DIM, wl.DEFAULT_BLOCK
    total = args.warmup + args.steps
    nb = sum(-(-n // B) for n in churn.prompt_lens) * churn.width \
        + churn.groups * churn.width * (total // B + 4)
    order = np.random.default_rng(churn.seed).permutation(nb)
    desc = pk.PoolDesc(nb, B, num_heads=H, head_dim=D, free_order=order)
    pool = pk.pa_pool_create(desc)
    bg = BeamGroups(pool, churn)
    S = len(bg.ids())
    gen = torch.Generator(device=dev)
    gen.manual_seed(churn.seed)
    kc = torch.empty((nb, H, B, D), dtype=torch.float16, device=dev).normal_(generator=gen)
    vc = torch.empty_like(kc).normal_(generator=gen)
    q = torch.randn((S, H, D), dtype=torch.float16, device=dev, generator=gen)
    k_new, v_new, out = torch.randn_like(q), torch.randn_like(q), torch.empty_like(q)
    stream = torch.cuda.Stream(device=dev)
    mb = -(-(max(churn.prompt_lens) + total) // B) + 1
    runner = DecodeStepRunner(pool, desc, bg.ids(), mb, device=dev, stream=stream)
    rng = np.random.default_rng(churn.seed + 1)
    # the seeded survivor draws are inputs: drawn before any timing, as counts
    # of each beam among its group's survivors
    def counts_of(surv):
        c = np.zeros((churn.groups, churn.width), np.int32)
        for g, keep in enumerate(surv):
            c[g] = np.bincount(keep, minlength=churn.width)
        return c
    draws = iter([counts_of(churn.survivors(rng)) for _ in range(total)])
    host, stats = [], {"copies": 0, "forks": 0, "frees": 0, "tokens": 0, "bytes": 0}

    split = {"prepare_wait": 0.0, "block_manager": 0.0, "launches": 0.0, "prune": 0.0}

    def step(record):
        h0 = time.perf_counter()
        runner.ids = bg.id_array()
        runner.prepare()
        h1 = time.perf_counter()
        ctx = runner.ctx_host.astype(np.int64)
        runner.copy_blocks([kc], [vc])
        runner.step_attention(out, q, k_new, v_new, kc, vc, 1 / math.sqrt(D))
        h2 = time.perf_counter()
        f, fr = bg.prune(next(draws))
        h3 = time.perf_counter()
        if record:
            host.append(h3 - h0 - (h1 - h0 - runner.host_seconds))
            split["prepare_wait"] += h1 - h0 - runner.host_seconds
            split["block_manager"] += runner.host_seconds
            split["launches"] += h2 - h1
            split["prune"] += h3 - h2
            stats["copies"] += runner.n_copies
            stats["forks"] += f
            stats["frees"] += fr
            stats["tokens"] += int(ctx.sum())
            stats["bytes"] += int(ctx.sum()) * H * D * 4 + S * H * D * 4

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(False)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(args.steps):
            step(True)
        t1.record(stream)
    torch.cuda.synchronize()
    assert runner.status.item() == 0
    el = t0.elapsed_time(t1) / 1e3
    line = {
        "metric": METRIC, "value": stats["tokens"] / el, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "data": "synthetic",
        "config": {"workload": "beam-search churn, 64 requests x 4 beams, OPT-13B layer 40x128, "
                               "block 16, prune + fork every step", "pool_blocks": nb},
        "per_step": {k: stats[k] / args.steps for k in ("copies", "forks", "frees")},
        "host_us_per_step": 1e6 * sum(host) / len(host),
        "host_split_us_per_step": {k: 1e6 * v / args.steps for k, v in split.items()},
        "logical_attention_GB/s": stats["bytes"] / el / 1e9,
        "note": "logical bytes count shared blocks once per beam; host time = pruning + "
                "block manager + Python launch path (the wait on the GPU excluded)",
    }
    if not quiet:
        print(json.dumps(line), flush=True)
    pk.pa_pool_destroy(pool)
    return line


PREFILL_METRIC = "paged prefill-attn prompt-tokens/s (1 GB300) + achieved TFLOP/s"
PREFILL_UNIT = "prompt-tokens/s"


def prefill_flops(lens_ctx, lens_q, num_heads, head_dim):
    """Algorithmic flops of causal prefill: the query at position p takes
    p + 1 dot products of length D for the scores and as many scaled value
    rows: 4 * D * (p + 1) flops per head."""
    tot = 0
    for c, n in zip(lens_ctx, lens_q):
        first = c - n                       # positions first .. c-1 are queries
        tot += (c * (c + 1) - first * (first + 1)) // 2
    return 4 * head_dim * num_heads * tot


def _prefill_cpu_baseline(seconds: float):
    """The oracle on a bounded sample of the prefill batch: its first 8 prompts."""
    from oracle import attention as oa
    import workloads as wl
    from oracle.alloc import BlockManager

    w = wl.prefill_b256()
    H, D, B = w.num_heads, w.head_dim, w.block_size
    lens = w.prompt_lens[:8]
    m = BlockManager(w.num_blocks, B, w.free_order)
    for i, n in enumerate(lens):
        m.add(i, n)
    used = sorted({b for i in range(len(lens)) for b in m.block_table(i)})
    rng = wl.value_rng(w, 3)
    kc = np.zeros((w.num_blocks, H, B, D), np.float16)
    vc = np.zeros_like(kc)
    for b in used:
        kc[b] = wl.normal_f16(rng, (H, B, D))
        vc[b] = wl.normal_f16(rng, (H, B, D))
    mb = -(-max(lens) // B)
    tables = np.array(m.padded_tables(list(range(len(lens))), mb), np.int32)
    ctx = np.array(lens, np.int32)
    qs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = wl.normal_f16(rng, (int(qs[-1]), H, D))
    passes, t0 = 0, time.perf_counter()
    while True:
        oa.paged_prefill(q, kc, vc, tables, ctx, qs, w.scale)
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": passes * int(qs[-1]) / dt, "unit": PREFILL_UNIT, "cores": oa.max_threads(),
            "kind": "oracle",
            "sample": f"first 8 of the 256 prompts ({int(qs[-1])} tokens), {passes} passes in "
                      f"{dt:.1f} s, fp64 C + OpenMP"}


def _tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return (float(json.load(f)["bf16_tflops"]),
                    "measured bf16 burst (MEASURED_PEAKS.json; fp16 has the same nominal rate)")
    except Exception:
        return 1900.0, "fallback 1.9 PFLOP/s"


class PrefillBatch:
    """The prompt phase of the mixed batch on one GPU: 256 whole prompts
    admitted through the block manager, their new K/V, queries and output."""

    def __init__(self, dev, seed: int = 112, prompts: int = 0):
        import torch

        import paged_kv_cache_106_gb300 as pk
        import workloads as wl

        self.pk = pk
        w = wl.prefill_b256(seed=seed)
        if prompts:
            w.prompt_lens = w.prompt_lens[:prompts]
        self.w = w
        H, D, B = w.num_heads, w.head_dim, w.block_size
        lens = np.array(w.prompt_lens, np.int64)
        self.lens = lens
        self.desc = pk.PoolDesc(w.num_blocks, B, num_heads=H, head_dim=D, free_order=w.free_order)
        self.pool = pk.pa_pool_create(self.desc)
        slots = np.concatenate([pk.pa_seq_add(self.pool, i, int(n)) for i, n in enumerate(lens)])
        mb = -(-int(lens.max()) // B)
        tables, ctx = pk.pa_get_block_tables(self.pool, list(range(len(lens))), mb)
        self.T = T = int(lens.sum())
        qs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        gen = torch.Generator(device=dev)
        gen.manual_seed(w.seed)
        self.kc = torch.empty((w.num_blocks, H, B, D), dtype=torch.float16, device=dev).normal_(generator=gen)
        self.vc = torch.empty_like(self.kc).normal_(generator=gen)
        self.q = torch.randn((T, H, D), dtype=torch.float16, device=dev, generator=gen)
        self.k_new, self.v_new = torch.randn_like(self.q), torch.randn_like(self.q)
        self.out = torch.empty_like(self.q)
        self.d_slots = torch.from_numpy(slots).to(dev)
        self.d_tables, self.d_ctx, self.d_qs = (torch.from_numpy(x).to(dev) for x in (tables, ctx, qs))
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.Stream(device=dev)
        self.mql = int(lens.max())
        self.flops = prefill_flops(ctx.tolist(), lens.tolist(), H, D)
        # bytes the attention must move at least: K and V of every prompt
        # token read, q read, o written, tables and lengths read
        self.unique_bytes = 4 * T * H * D * 2 + int(((lens + B - 1) // B).sum()) * 4 + 12 * len(lens)
        # the one-call step (pa_prefill_step_attention) also stores every
        # prompt token's K and V into the cache
        self.write_bytes = 2 * T * H * D * 2

    def write(self, k=None, v=None):
        self.pk.pa_write_kv(self.k_new if k is None else k, self.v_new if v is None else v,
                            self.d_slots, self.kc, self.vc, self.desc, status=self.status,
                            stream=self.stream)

    def attend(self, q=None, out=None):
        self.pk.pa_prefill_attention(self.out if out is None else out, self.q if q is None else q,
                                     self.kc, self.vc, self.d_tables, self.d_ctx, self.d_qs,
                                     self.w.scale, self.desc, max_q_len=self.mql,
                                     status=self.status, stream=self.stream)

    def fused(self, q=None, out=None, k=None, v=None):
        self.pk.pa_prefill_step_attention(
            self.out if out is None else out, self.q if q is None else q,
            self.k_new if k is None else k, self.v_new if v is None else v, self.kc, self.vc,
            self.d_tables, self.d_ctx, self.d_qs, self.w.scale, self.desc, max_q_len=self.mql,
            status=self.status, stream=self.stream)

    def time_fused(self, steps: int, warmup: int):
        """The one-call step (slot write and attention in one launch); returns
        (elapsed s, ms per launch) from CUDA events on the stream."""
        import torch

        with torch.cuda.stream(self.stream):
            for _ in range(warmup):
                self.fused()
        torch.cuda.synchronize()
        evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2)) for _ in range(steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(self.stream)
        for i in range(steps):
            evs[i][0].record(self.stream)
            self.fused()
            evs[i][1].record(self.stream)
        t1.record(self.stream)
        torch.cuda.synchronize()
        assert self.status.item() == 0, self.status.item()
        return t0.elapsed_time(t1) / 1e3, sum(a.elapsed_time(b) for a, b in evs) / steps

    def time_steps(self, steps: int, warmup: int):
        """Slot write + attention per step; returns (elapsed s, attention ms per
        launch, slot-write ms per launch) from CUDA events on the stream."""
        import torch

        with torch.cuda.stream(self.stream):
            for _ in range(warmup):
                self.write()
                self.attend()
        torch.cuda.synchronize()
        evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(self.stream)
        for i in range(steps):
            evs[i][2].record(self.stream)
            self.write()
            evs[i][0].record(self.stream)
            self.attend()
            evs[i][1].record(self.stream)
        t1.record(self.stream)
        torch.cuda.synchronize()
        assert self.status.item() == 0, self.status.item()
        attn_ms = sum(a.elapsed_time(b) for a, b, _ in evs) / steps
        wkv_ms = sum(c.elapsed_time(a) for a, _, c in evs) / steps
        return t0.elapsed_time(t1) / 1e3, attn_ms, wkv_ms

    def roofline(self, attn_ms: float, fused: bool = False) -> dict:
        """The binding roof of the attention call (with ``fused``, of the
        one-call step, whose bytes include the cache writes): the larger of
        the HBM time of its unique bytes and the tensor time of its causal
        flops."""
        hbm, hbm_kind = _peaks()
        tf, tf_kind = _tensor_peak()
        ub = self.unique_bytes + (self.write_bytes if fused else 0)
        t_hbm = ub / (hbm * 1e9) * 1e3
        t_tc = self.flops / (tf * 1e12) * 1e3
        bound = "hbm" if t_hbm >= t_tc else "tensor"
        if bound == "hbm":
            achieved, peak, unit = ub / (attn_ms / 1e3) / 1e9, hbm, "GB/s"
            kind = f"{hbm_kind} hbm_gbs"
        else:
            achieved, peak, unit = self.flops / (attn_ms / 1e3) / 1e12, tf, "TFLOP/s"
            kind = tf_kind
        return {"bound": bound, "achieved": achieved, "peak": peak, "peak_kind": kind, "unit": unit,
                "frac": achieved / peak, "ms_per_launch": attn_ms,
                "unique_bytes_per_launch": ub, "hbm_floor_ms": t_hbm,
                "algorithmic_flops_per_launch": self.flops, "tensor_floor_ms": t_tc,
                "tflops": self.flops / (attn_ms / 1e3) / 1e12,
                "GB/s": ub / (attn_ms / 1e3) / 1e9,
                **self.traffic(fused)}

    def traffic(self, fused: bool = False) -> dict:
        """DRAM bytes per launch from the committed ncu capture of the full
        256-prompt batch (its DRAM bytes over unique bytes, times this batch's
        unique bytes), if it was taken on the current kernel code and this is
        that batch (the ratio does not carry over to a subset of prompts)."""
        t = _kernel_traffic(os.path.join(ROOT, "paged_kv_cache_106_gb300", "csrc", "prefill_attention.cu"),
                            "prefill_attention_traffic.json")
        full = t is not None and t.get("prompt_tokens") == self.T
        if fused:   # the one-call step's kernel, captured on its own
            t = t.get("fused") if full else None
            full = t is not None
            ub = self.unique_bytes + self.write_bytes
            name = "paged_prefill_tc<128, true> (pa_prefill_step_attention)"
        else:
            ub = self.unique_bytes
            name = "paged_prefill_tc<128, false> (pa_prefill_attention)"
        return {"kernel": name,
                "traffic": t["traffic_over_algorithmic"] * ub if full else None,
                "traffic_over_algorithmic": t["traffic_over_algorithmic"] if full else None,
                "traffic_from": t["capture"] if full else None}

    def close(self):
        self.pk.pa_pool_destroy(self.pool)


def run_prefill(args):
    """Prompt phase of the mixed batch: every step stores the K/V of all 256
    prompts into the pool and runs causal paged prefill attention over them
    (one OPT-13B layer), in one call (pa_prefill_step_attention); the same
    step as two calls (pa_write_kv, pa_prefill_attention) is timed beside it."""
    import torch

    ws, rank, local = _dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pb = PrefillBatch(dev, seed=112 + rank, prompts=args.prompts)
    w, lens, T = pb.w, pb.lens, pb.T
    H, D = w.num_heads, w.head_dim
    q, k_new, v_new, out = pb.q, pb.k_new, pb.v_new, pb.out
    stream, status = pb.stream, pb.status
    clocks = ClockSampler(local)
    clocks.start()
    el, fused_ms = pb.time_fused(args.steps, args.warmup)   # the step: one call
    clk = clocks.stop()
    el_sep, attn_ms, wkv_ms = pb.time_steps(args.steps, args.warmup)   # the same, as two calls
    # end to end through the same calls: the step's new K/V and queries come
    # from pinned host memory, the output goes back to it
    h_k, h_v, h_q = (torch.empty(q.shape, dtype=q.dtype, pin_memory=True) for _ in range(3))
    h_o = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    for h in (h_k, h_v, h_q):
        h.normal_()
    e2e_steps = max(1, min(args.e2e_steps, 20))
    # Serving-loop order, two steps in flight: step i uses device buffer set
    # i & 1; its uploads (a copy stream), its kernels (the compute stream) and
    # its read-back (another copy stream) are ordered by events, so the
    # uploads of step i + 1 and the read-back of step i - 1 overlap step i;
    # the host waits for step i - 1's output after enqueueing step i.
    bufs = [(k_new, v_new, q, out), tuple(torch.empty_like(q) for _ in range(4))]
    h_out = [h_o, torch.empty(q.shape, dtype=q.dtype, pin_memory=True)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {k: [torch.cuda.Event(), torch.cuda.Event()] for k in ("in", "comp", "out")}
    used = [False, False]

    def e2e_enqueue(i):
        s = i & 1
        kn, vn, qq, oo = bufs[s]
        if used[s]:
            s_in.wait_event(ev["comp"][s])     # step i - 2 has read this set's inputs
        with torch.cuda.stream(s_in):
            kn.copy_(h_k, non_blocking=True)
            vn.copy_(h_v, non_blocking=True)
            qq.copy_(h_q, non_blocking=True)
        ev["in"][s].record(s_in)
        stream.wait_event(ev["in"][s])
        if used[s]:
            stream.wait_event(ev["out"][s])    # step i - 2's output has left this set
        pb.fused(qq, oo, kn, vn)
        ev["comp"][s].record(stream)
        s_out.wait_event(ev["comp"][s])
        with torch.cuda.stream(s_out):
            h_out[s].copy_(oo, non_blocking=True)
        ev["out"][s].record(s_out)
        used[s] = True

    def run_e2e(n):
        for i in range(n):
            e2e_enqueue(i)
            if i >= 1:
                ev["out"][(i - 1) & 1].synchronize()   # step i - 1's output is on the host
        ev["out"][(n - 1) & 1].synchronize()

    # untimed steps first: the first transfers through freshly pinned pages run
    # several times slower than the steady state
    run_e2e(3)
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    run_e2e(e2e_steps)
    e2e_s = (time.perf_counter() - w0) / e2e_steps
    assert status.item() == 0, status.item()
    (tok_all, e2e_tok), (el_max, e2e_max) = reduce_across_ranks(
        [T * args.steps, T * e2e_steps], [el, e2e_s * e2e_steps], dev)
    if rank == 0:
        roof = pb.roofline(fused_ms, fused=True)
        line = {
            "metric": PREFILL_METRIC, "value": tok_all / el_max, "unit": PREFILL_UNIT,
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16 (fp32 accumulate)", "data": "synthetic",
            "config": {"workload": f"prompt phase of the mixed batch: {len(lens)} whole prompts, "
                                   "lognormal (median 200, cap 1536), OPT-13B layer 40x128, block 16",
                       "prompt_tokens": T, "pool_blocks": w.num_blocks,
                       "l2": "K/V written and read back per step ~1.7 GB >> 129 MB L2, no flush"},
            "gpu_launches": args.steps,
            "roofline": roof,
            "kernels": {"separate_calls": {
                            "ms_per_step": el_sep * 1e3 / args.steps,
                            "prompt_tokens_per_s": T * args.steps / el_sep,
                            "pa_write_kv_us_per_launch": wkv_ms * 1e3,
                            "pa_prefill_attention": pb.roofline(attn_ms),
                            "note": "the same step as pa_write_kv then pa_prefill_attention"}},
            "e2e": {"value": e2e_tok / e2e_max, "unit": PREFILL_UNIT,
                    "h2d_bytes_per_step": 3 * T * H * D * 2, "d2h_bytes_per_step": T * H * D * 2,
                    "steps": e2e_steps, "timing": "wall clock over the loop, after 3 untimed steps; two steps in flight "
                              "(uploads of step i+1 and read-back of step i-1 overlap step i)"},
            "clocks": clk,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = _prefill_cpu_baseline(args.cpu_seconds)
        print(json.dumps(line), flush=True)
    pb.close()


def _decode_config(w, ws):
    """The fixed part of the decode bench's config (both arms)."""
    return {"workload": f"mixed-length serving batch, OPT-13B-shaped layer 40x128, block 16, "
                        f"batch {len(w.prompt_lens)}/GPU, ctx<=2048, split>512, steady-state continuous batch",
            "batch_per_gpu": len(w.prompt_lens), "num_heads": w.num_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "partition_tokens": w.split_tokens,
            "pool_blocks": w.num_blocks,
            "parallelism": f"replicas x{ws} (sequences independent, no collective)"}


def _oracle_sample(n_seqs):
    """Host data for the first n_seqs sequences of the same workload, laid
    out by the oracle's own block manager."""
    import workloads as wl
    from oracle.alloc import BlockManager

    w = wl.mixed_b256(steady_state=True)
    H, D, B = w.num_heads, w.head_dim, w.block_size
    m = BlockManager(w.num_blocks, B, w.free_order)
    for i, n in enumerate(w.prompt_lens):
        m.add(i, n)
    ids = list(range(n_seqs))
    m.alloc_slots(list(range(len(w.prompt_lens))))
    used = sorted({b for s in ids for b in m.block_table(s)})
    kc = np.empty((w.num_blocks, H, B, D), np.float16)   # untouched pages stay unbacked
    vc = np.empty_like(kc)
    rng = wl.value_rng(w, 2)
    for b in used:
        kc[b] = wl.normal_f16(rng, (H, B, D))
        vc[b] = wl.normal_f16(rng, (H, B, D))
    mb = -(-wl.CTX_CAP // B)
    tables = np.array(m.padded_tables(ids, mb), np.int32)
    ctx = np.array([m.num_tokens(s) for s in ids], np.int32)
    q = wl.normal_f16(rng, (n_seqs, H, D))
    return q, kc, vc, tables, ctx, w.scale


def cpu_baseline(seconds: float, n_seqs: int):
    from oracle import attention as oa

    q, kc, vc, tables, ctx, scale = _oracle_sample(n_seqs)
    oa.paged_attention(q[:1], kc, vc, tables[:1], ctx[:1], scale)       # build + warm
    passes, t0 = 0, time.perf_counter()
    while True:
        oa.paged_attention(q, kc, vc, tables, ctx, scale)
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": passes * int(ctx.sum()) / dt, "unit": UNIT, "cores": oa.max_threads(),
            "kind": "oracle",
            "sample": f"first {n_seqs} of the 256 sequences (sum ctx {int(ctx.sum())}), "
                      f"{passes} passes in {dt:.1f} s, fp64 C + OpenMP"}


def run_reference(args):
    """The oracle as it stands, timed on the host cores, as the reference arm."""
    ws, rank, _ = _dist_env()
    if rank != 0:
        return
    import workloads as wl
    from oracle import attention as oa

    q, kc, vc, tables, ctx, scale = _oracle_sample(args.ref_seqs)
    for _ in range(args.warmup):
        oa.paged_attention(q, kc, vc, tables, ctx, scale)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oa.paged_attention(q, kc, vc, tables, ctx, scale)
    dt = time.perf_counter() - t0
    value = args.steps * int(ctx.sum()) / dt
    sample = (f"first {args.ref_seqs} of the 256 sequences of the mixed batch (sum ctx "
              f"{int(ctx.sum())}) per step; fp64 C oracle, OpenMP")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _decode_config(wl.mixed_b256(steady_state=True), ws),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oa.max_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_prefix_cache(args, quiet: bool = False):
    """Prefix caching: 256 prompts = one shared 512-token system prompt + a
    suffix of their own (lognormal, median 200, cap 1024), OPT-13B layer
    shapes.  One step admits every prompt through the hash-chained block
    cache (the system prompt's 32 full blocks are found cached; each step
    draws new suffix tokens, so nothing else hits), writes K/V for the
    uncached tokens only and prefills only those queries over the whole
    context, then frees the prompts (their blocks stay cached, evictable).
    The same step without caching (every token written and prefilled) is
    timed beside it.  value = prompt tokens (cached ones included) per
    second of GPU time."""
    import torch

    import paged_kv_cache_106_gb300 as pk
    import workloads as wl

    _, _, local = _dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    H, D, B = wl.OPT13B_HEADS, wl.OPT13B_HEAD_DIM, wl.DEFAULT_BLOCK
    n_p, sys_len, seed = (args.prompts or 256), 512, 113
    rng = np.random.default_rng(seed)
    suf = np.clip(np.round(rng.lognormal(np.log(200.0), 1.0, n_p)), 1, 1024).astype(np.int64)
    lens = sys_len + suf
    T = int(lens.sum())
    system = rng.integers(0, 50000, sys_len).astype(np.int32)
    total = args.warmup + args.steps
    # the token ids are inputs, drawn before any timing: new suffixes every step
    suffixes = [[rng.integers(0, 50000, int(n)).astype(np.int32) for n in suf] for _ in range(total)]
    need = int(sum(-(-int(n) // B) for n in lens))
    shared = sys_len // B
    pools = {}
    for name, flags, nb in (("cached", pk.PA_POOL_PREFIX_CACHING, int(1.25 * (need - (n_p - 1) * shared)) + 64),
                            ("uncached", 0, int(1.1 * need) + 64)):
        desc = pk.PoolDesc(nb, B, num_heads=H, head_dim=D, flags=flags,
                           free_order=np.random.default_rng(seed + 1).permutation(nb).astype(np.int32))
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
        kc = torch.empty((nb, H, B, D), dtype=torch.float16, device=dev).normal_(generator=gen)
        pools[name] = (desc, pk.pa_pool_create(desc), kc, torch.empty_like(kc).normal_(generator=gen))
    q = torch.randn((T, H, D), dtype=torch.float16, device=dev)
    k_new, v_new, out = torch.randn_like(q), torch.randn_like(q), torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    mb = -(-int(lens.max()) // B)
    res = {}
    for name in ("cached", "uncached"):
        desc, pool, kc, vc = pools[name]
        admit_s, gpu_ms, new_tok = 0.0, 0.0, 0
        for it in range(total):
            h0 = time.perf_counter()
            slot_parts, n_new = [], []
            for i in range(n_p):
                toks = np.concatenate([system, suffixes[it][i]])
                if name == "cached":
                    slots, nc = pk.pa_seq_add_tokens(pool, i, toks)
                else:
                    slots, nc = pk.pa_seq_add(pool, i, int(toks.shape[0])), 0
                slot_parts.append(slots[nc:])
                n_new.append(int(toks.shape[0]) - nc)
            tables, ctx = pk.pa_get_block_tables(pool, list(range(n_p)), mb)
            h1 = time.perf_counter()
            slots = np.concatenate(slot_parts)
            qs = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
            tn = int(qs[-1])
            d_slots = torch.from_numpy(slots).to(dev)
            d_tab, d_ctx, d_qs = (torch.from_numpy(x).to(dev) for x in (tables, ctx, qs))
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                pk.pa_write_kv(k_new[:tn], v_new[:tn], d_slots, kc, vc, desc, status=status, stream=stream)
                pk.pa_prefill_attention(out, q, kc, vc, d_tab, d_ctx, d_qs, 1 / math.sqrt(D), desc,
                                        max_q_len=int(max(n_new)), status=status, stream=stream,
                                        q_rows=tn)
                e1.record(stream)
            torch.cuda.synchronize()
            for i in range(n_p):
                pk.pa_seq_free(pool, i)
            if it >= args.warmup:
                admit_s += h1 - h0
                gpu_ms += e0.elapsed_time(e1)
                new_tok += tn
        assert status.item() == 0, pk.pa_last_error_string()
        res[name] = {"gpu_ms_per_step": gpu_ms / args.steps,
                     "prompt_tokens_per_s": T * args.steps / (gpu_ms / 1e3),
                     "computed_tokens_per_step": new_tok // args.steps,
                     "host_us_per_admission": admit_s / args.steps / n_p * 1e6}
        pk.pa_pool_destroy(pool)
    c, u = res["cached"], res["uncached"]
    line = {
        "metric": "prefix-cached prefill prompt-tokens/s (1 GB300)", "value": c["prompt_tokens_per_s"],
        "unit": "prompt-tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": c["gpu_ms_per_step"], "higher_is_better": True, "data": "synthetic",
        "dtype": "f16 (fp32 accumulate)",
        "config": {"workload": f"{n_p} prompts = shared {sys_len}-token system prompt + own suffix "
                               "(lognormal median 200, cap 1024), OPT-13B layer 40x128, block 16",
                   "prompt_tokens": T},
        "gpu_launches": 2 * args.steps,
        "cached": c, "uncached": u, "speedup": c["prompt_tokens_per_s"] / u["prompt_tokens_per_s"],
        "timing": "GPU: CUDA events around the slot write + prefill of a step; host: wall clock of "
                  "the admissions (Python calls into the C block manager) and the table read",
    }
    if not quiet:
        print(json.dumps(line), flush=True)
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batch", type=int, default=256)
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="default workload: skip the other rows measured after the timed "
                         "region (64 sequences, parallel sampling, prefill, 40 layers, beam "
                         "churn, prefix cache)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-seqs", type=int, default=32)
    ap.add_argument("--ref-seqs", type=int, default=16)
    ap.add_argument("--workload",
                    choices=["mixed_b256", "full_40l", "beam_churn", "prefill", "prefix_cache"],
                    default="mixed_b256",
                    help="mixed_b256: the headline workload; full_40l: 40-layer pool-filling "
                         "step; beam_churn: beam search with pruning; prefill: causal "
                         "prefill of the mixed batch's prompts; prefix_cache: prompts sharing "
                         "a system prompt, admitted through the block cache")
    ap.add_argument("--beam", action="store_true", help="full_40l: beam groups sharing blocks")
    ap.add_argument("--prompts", type=int, default=0,
                    help="prefill: use only the first N prompts of the batch (small profiling case)")
    ap.add_argument("--dump-steps", default="",
                    help="write each warm-up and timed step's algorithmic attention bytes here")
    ap.add_argument("--partition", type=int, default=0,
                    help="split-context partition in tokens (default: the workload's 512)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "full_40l":
        run_full40(args)
    elif args.workload == "beam_churn":
        run_beam_churn(args)
    elif args.workload == "prefill":
        run_prefill(args)
    elif args.workload == "prefix_cache":
        run_prefix_cache(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
