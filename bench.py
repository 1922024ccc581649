#!/usr/bin/env python
"""Benchmark of the paged-KV attention hot path on GB300.

Default workload: the Llama-3-8B-shaped mixed step -- 32 query / 8 KV heads,
head_dim 128, block_size 16, bf16 -- the largest workload that fits one GPU.
One step is one pass of the whole hot path: 120 decode sequences with
context lengths uniform in [1024, 32768] (append of each sequence's new token
with RoPE at position ctx-1, the rotation of q, and split-KV GQA decode with
its planner, block-table gather and in-launch merge: one launch,
pkv_decode_step), then 8 ragged causal prefill chunks of 512 tokens over
cached prefixes uniform in [0, 8192] whose pairs share prefix blocks (one
launch).  The step's 8.3 GB of K/V far exceed the 129 MB L2.  The timed
steps replay a CUDA graph; K steps form one timed window, and windows repeat
for at least a second (median, p10, p90).  The Qwen2.5-3B-shaped decode
step is timed after it and carried in the same line.

``--config 2|3|5`` times another workload's step instead; ``--part`` times
one part or next-step row on its own.  Prints one JSON line (rank 0).
``--impl reference`` times the CPU oracle on a bounded sample of the same
workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("paged decode attention KV GB/s and % of HBM peak; attention tokens/s on 1 GB300")
FALLBACK_HBM_GBS = 6800.0


# -------------------------------------------------------------- plumbing --

def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    p.add_argument("--config", type=int, default=4, choices=[2, 3, 4, 5],
                   help="workload: 4 Llama-3-8B mixed step (default: the largest single-GPU "
                        "workload), 2 Qwen2.5-3B decode, 3 Qwen3-4B decode+append, 5 FP8 "
                        "two-layer decode")
    p.add_argument("--no-carry", action="store_true",
                   help="skip the Qwen2.5-3B decode figures carried beside the mixed step")
    p.add_argument("--part", choices=["step", "prefill", "cascade", "verify", "cow", "ring",
                                      "ring-prefill", "fp8-prefill"], default="step",
                   help="step: the workload's whole step (default); prefill: the ragged causal "
                        "prefill part of workload 4 alone, timed against the tensor-core peak; "
                        "cascade / verify / cow / ring / ring-prefill / fp8-prefill: the next-step "
                        "rows, each "
                        "on its own seeded workload")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--decode-first", action="store_true",
                   help="mixed step: decode, then prefill waiting for it (the order before "
                        "PKV_DESC_INDEPENDENT)")
    p.add_argument("--no-prefetch-kv", action="store_true",
                   help="decode steps read nothing before the previous kernel ends "
                        "(PKV_DESC_PREFETCH_KV off)")
    p.add_argument("--chunk-blocks", type=int, default=0,
                   help="decode chunk length in blocks passed to the library (0: the planner's "
                        "choice)")
    p.add_argument("--two-launch", action="store_true",
                   help="run append and decode as two launches per layer instead of the "
                        "fused decode step")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="CPU seconds the oracle baseline sample aims at")
    return p.parse_args()


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group(backend, device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0


FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def measured_tensor_peak(sustained=False):
    """Dense bf16 TFLOP/s: the burst figure (a kernel timed alone), or the
    sustained one (a kernel timed inside a long step)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if key in d:
            return float(d[key]), "measured"
    return (FALLBACK_BF16_TFLOPS_SUSTAINED if sustained else FALLBACK_BF16_TFLOPS), "fallback"


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        ident = str(device_index)
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-i", ident, "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = {"decode_kernel": "decode.cu", "prefill_tc_kernel": "prefill_tc.cu"}


def kernel_traffic_per_launch(kernel, config):
    """DRAM bytes (read + write) per launch of `kernel` on workload `config`
    from profiles/traffic.json (machine-readable; the ncu summaries beside it
    explain the figures), if they were taken on the current kernel source
    (else None)."""
    if not os.path.exists(TRAFFIC_JSON):
        return None
    with open(TRAFFIC_JSON) as f:
        d = json.load(f)
    ent = d.get(kernel)
    if not ent:
        return None
    src = os.path.join(ROOT, "paged_kv_attention_21_gb300", "csrc", KERNEL_SOURCES[kernel])
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if ent.get("source_sha256_16") != sha:
        return None
    v = ent.get("dram_bytes_per_launch", {}).get(str(config))
    return None if v is None else float(v)


# ------------------------------------------------------------- workloads --

class DecodeWorkload:
    """A decode workload: instances over disjoint regions of one pool (per
    layer), each with its own device workspace-free inputs."""

    def __init__(self, config, dev, rank, fused=True, chunk=0, prefetch=True, prefill_first=True):
        import paged_kv_attention_21_gb300 as pkv
        self.fused = fused
        # The fused step's predecessor on the stream never writes the K/V
        # rows, tables or lengths it reads: the previous step used another
        # batch's pool region (or another layer's pools, or it was the
        # prefill, which writes no pool), so the decode may start its first
        # K/V loads while that kernel drains.  The two-launch step's
        # predecessor is the append kernel, which writes the rows it reads.
        self.prefetch = bool(prefetch and fused)
        # The mixed step's two halves -- the decode tokens' attention and the
        # prefill chunks' -- both read one layer's QKV output and touch
        # different sequences' blocks and different outputs: the prefill runs
        # first and the decode after it without waiting for it (its CTAs take
        # the SMs the prefill's last CTAs leave idle), then waits at its end.
        self.independent = bool(config == 4 and fused and prefill_first)
        self.chunk = chunk
        from paged_kv_attention_21_gb300 import workloads as wl
        self.pkv = pkv
        spec = wl.CONFIGS[config]
        if rank:
            spec = wl.dataclasses.replace(spec, seed=spec.seed + 7919 * rank)
        self.spec = spec
        self.config = config
        one_bytes = None
        n_inst = 4
        if config in (4, 5):
            n_inst = 1  # 8.3 GB / 1.1 GB of K/V per step: far beyond L2 already
        self.insts = wl.make_decode_instances(spec, n_inst, dev)
        self.layers = [self.insts]
        if config == 5:
            # second layer: sliding window 128, its own pools and scales
            first = self.insts[0]
            g = torch.Generator(device=dev).manual_seed(spec.seed + 1)
            shape = tuple(first.k_cache.shape)
            k2, ks2 = wl.fill_e4m3(shape, g, dev)
            v2, vs2 = wl.fill_e4m3(shape, g, dev)
            import copy
            layer2 = []
            for b in self.insts:
                c = copy.copy(b)
                c.k_cache, c.v_cache, c.k_scale, c.v_scale = k2, v2, ks2, vs2
                layer2.append(c)
            self.layers.append(layer2)
        self.windows = [-1] if config != 5 else [-1, wl.FP8_WINDOW]
        b0 = self.insts[0]
        self.desc = pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                                  head_dim=spec.head_dim, num_blocks=b0.k_cache.shape[0],
                                  max_blocks_per_seq=b0.tables_host.shape[1],
                                  kv_dtype=spec.kv_dtype,
                                  flags=(pkv.DESC_PREFETCH_KV if self.prefetch else 0) |
                                        (pkv.DESC_INDEPENDENT if self.independent else 0))
        self.max_ctx = spec.ctx_hi
        ws = max(pkv.pkv_decode_workspace_size(self.desc, spec.batch, self.max_ctx, w, chunk)
                 for w in self.windows)
        self.ws = torch.zeros(max(ws, 256), dtype=torch.uint8, device=dev)
        self.table = torch.from_numpy(pkv.pkv_rope_cos_sin_table(spec.rope_theta, spec.head_dim,
                                                                 spec.ctx_hi)).to(dev)
        self.seq_ids = torch.arange(spec.batch, dtype=torch.int32, device=dev)
        self.pos = [(b.context_lens - 1).to(torch.int32) for b in self.insts]
        self.out = torch.empty_like(b0.q)
        self.lse = torch.empty(b0.q.shape[:2], dtype=torch.float32, device=dev)
        self.prefill = None
        if config == 4:
            self.prefill = PrefillPart(dev, rank)
        del one_bytes

    @property
    def n_inst(self):
        return len(self.insts)

    def kv_bytes(self, i):
        total = 0
        for layer, w in zip(self.layers, self.windows):
            total += layer[i].kv_bytes(w)
        if self.prefill is not None:
            total += self.prefill.kv_bytes
        return total

    def tokens(self, i):
        return self.spec.batch + (self.prefill.tokens if self.prefill is not None else 0)

    def step(self, i, ev_pairs=None, pev=None):
        """Launch one step for instance i; ev_pairs (list of (start, end)) are
        recorded around each decode launch, pev around the prefill launch.
        Returns the launch count."""
        pkv = self.pkv
        n = 0
        if self.prefill is not None and self.independent:
            n += self._prefill(pev)
        for li, (layer, w) in enumerate(zip(self.layers, self.windows)):
            b = layer[i]
            if self.fused:
                # one launch: append + RoPE of the new token, q rotation, decode
                if ev_pairs is not None:
                    ev_pairs[li][0].record()
                pkv.pkv_decode_step(self.desc, b.q, b.k_new, b.v_new, b.k_cache, b.v_cache,
                                    b.block_tables, b.context_lens, self.max_ctx,
                                    self.spec.sm_scale, self.out, self.lse, self.ws,
                                    cos_sin=self.table, window=w, chunk_blocks=self.chunk,
                                    k_scale=b.k_scale, v_scale=b.v_scale)
                if ev_pairs is not None:
                    ev_pairs[li][1].record()
                n += 1
                continue
            pkv.pkv_append_rope(self.desc, b.k_cache, b.v_cache, b.block_tables, self.seq_ids,
                                self.pos[i], b.k_new, b.v_new, q=b.q, cos_sin=self.table,
                                k_scale=b.k_scale, v_scale=b.v_scale)
            if ev_pairs is not None:
                ev_pairs[li][0].record()
            pkv.pkv_decode_attention(self.desc, b.q, b.k_cache, b.v_cache, b.block_tables,
                                     b.context_lens, self.max_ctx, self.spec.sm_scale, self.out,
                                     self.lse, self.ws, window=w, chunk_blocks=self.chunk,
                                     k_scale=b.k_scale, v_scale=b.v_scale)
            if ev_pairs is not None:
                ev_pairs[li][1].record()
            n += 2
        if self.prefill is not None and not self.independent:
            n += self._prefill(pev)
        return n

    def _prefill(self, pev):
        if pev is not None:
            pev[0].record()
        self.prefill.run()
        if pev is not None:
            pev[1].record()
        return 1


class PrefillPart:
    """The prefill half of the Llama-3-8B-shaped mixed step."""

    def __init__(self, dev, rank):
        import paged_kv_attention_21_gb300 as pkv
        from paged_kv_attention_21_gb300 import workloads as wl
        self.pkv = pkv
        spec = wl.LLAMA3_8B_PREFILL
        self.spec = spec
        self.pb = wl.make_prefill_batch(spec, dev)
        pb = self.pb
        self.desc = pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                                  head_dim=spec.head_dim, num_blocks=pb.k_cache.shape[0],
                                  max_blocks_per_seq=pb.tables_host.shape[1])
        self.out = torch.empty_like(pb.q)
        self.tokens = pb.total_q
        vis = pb.kv_lens_host.astype(np.int64)
        self.kv_bytes = int(vis.sum()) * spec.num_kv_heads * spec.head_dim * 2 * 2
        self.flops = pb.flops()

    def run(self):
        pb = self.pb
        self.pkv.pkv_prefill_attention_ragged(self.desc, pb.q, pb.qo_indptr, pb.k_cache,
                                              pb.v_cache, pb.block_tables, pb.kv_lens,
                                              self.spec.sm_scale, self.out,
                                              qo_indptr_host=pb.qo_indptr_host,
                                              kv_lens_host=pb.kv_lens_host)


# ---------------------------------------------------------------- timing --

def graph_len(K, n_inst):
    """Steps per captured graph: a divisor of K (so the timed steps are
    exactly K), at most 64, and at least the instance count when K allows."""
    best = 1
    for r in range(1, min(K, 64) + 1):
        if K % r == 0:
            best = r
    return best


def time_pkv(args, rank, world, local, config=None, steps=None, min_seconds=2.0,
             with_e2e=True):
    """Time one workload's step as replays of a captured CUDA graph.

    A window is exactly K steps, bracketed by CUDA events on the launching
    stream (after a barrier and a synchronize); windows repeat back to back
    until at least `min_seconds` have passed (and at least 3 windows).  The
    step time is the median window (max over ranks), with p10 / p90 beside it.
    CUDA events inside the graph bracket the decode launch (and the prefill
    launch of the mixed step) of every `stride`-th step; they give the
    per-kernel launch times the rooflines use."""
    import paged_kv_attention_21_gb300 as pkv
    config = args.config if config is None else config
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    W = DecodeWorkload(config, dev, rank, fused=not args.two_launch, chunk=args.chunk_blocks,
                       prefetch=not args.no_prefetch_kv, prefill_first=not args.decode_first)
    K = max(1, args.steps if steps is None else steps)
    Wm = max(3, args.warmup)
    R = graph_len(K, W.n_inst)
    nlayers = len(W.layers)

    # eager warm-up of every instance (first calls set up device state)
    for i in range(W.n_inst):
        W.step(i)
    torch.cuda.synchronize()
    pkv.pkv_device_errors(reset=True)

    # Timing events sit around the decode launches (and the prefill launch) of
    # every `stride`-th step only (a stride coprime with the instance count,
    # so every instance is sampled): an event between two launches breaks
    # their programmatic dependent launch, so the other steps keep
    # back-to-back launches.
    stride = 11   # coprime with the 1- and 4-batch rotations
    sampled = list(range(0, R, stride))
    mk = lambda: (torch.cuda.Event(enable_timing=True, external=True),
                  torch.cuda.Event(enable_timing=True, external=True))
    evs = {j: [mk() for _ in range(nlayers)] for j in sampled}
    pevs = {j: mk() for j in sampled} if W.prefill is not None else {}
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    launches_per_replay = 0
    with torch.cuda.graph(graph, stream=cap):
        for j in range(R):
            launches_per_replay += W.step(j % W.n_inst, evs.get(j), pevs.get(j))
    torch.cuda.synchronize()
    replays = K // R
    for _ in range(max(1, -(-Wm // R))):   # warm-up replays: >= W steps
        graph.replay()
    torch.cuda.synchronize()

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    win_ms, dec_ms, pre_ms = [], [[] for _ in range(nlayers)], []
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    while True:
        start.record()
        for _ in range(replays):
            graph.replay()
        end.record()
        end.synchronize()
        win_ms.append(start.elapsed_time(end))
        # the events of the window's last replay
        for j in sampled:
            for li in range(nlayers):
                dec_ms[li].append(evs[j][li][0].elapsed_time(evs[j][li][1]))
            if pevs:
                pre_ms.append(pevs[j][0].elapsed_time(pevs[j][1]))
        wall = time.perf_counter() - t0
        if len(win_ms) >= 3 and (wall >= min_seconds or len(win_ms) >= 2000):
            break
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    err = pkv.pkv_device_errors(reset=True)
    if err:
        raise RuntimeError("device error word 0x%x after the timed region" % err)

    n_samp = len(sampled)
    dec_bytes = [[W.layers[li][j % W.n_inst].kv_bytes(W.windows[li]) for j in sampled]
                 for li in range(nlayers)]
    li_dom = int(np.argmax([sum(x) for x in dec_bytes]))   # the layer with the most bytes
    dom_ms = float(np.mean(dec_ms[li_dom]))
    dom_bytes = float(np.mean(dec_bytes[li_dom]))
    # per-launch byte-weighted rate over every sampled launch of every window
    reps = len(win_ms)
    samp_bytes = np.tile(np.array(dec_bytes[li_dom], dtype=np.float64), reps)
    per_launch_gbs = samp_bytes / (np.array(dec_ms[li_dom]) / 1e3) / 1e9

    med_ms = float(np.median(win_ms))
    bytes_per_window = sum(W.kv_bytes(j % W.n_inst) for j in range(K))
    tokens_per_window = sum(W.tokens(j % W.n_inst) for j in range(K))
    t_max = reduce_max(med_ms / 1e3, world)
    total_bytes = reduce_sum(bytes_per_window, world)
    total_tokens = reduce_sum(tokens_per_window, world)
    res = dict(W=W, K=K, R=R, elapsed_s=t_max, wall_s=wall, total_bytes=total_bytes,
               ev_stride=stride, total_tokens=total_tokens, dom_ms=dom_ms, dom_bytes=dom_bytes,
               dom_layer=li_dom, dec_ms=dec_ms, clocks=clocks, windows=len(win_ms),
               win_p10=float(np.percentile(win_ms, 10)), win_p90=float(np.percentile(win_ms, 90)),
               dec_p10=float(np.percentile(dec_ms[li_dom], 10)),
               dec_p90=float(np.percentile(dec_ms[li_dom], 90)),
               per_launch_gbs=float(np.median(per_launch_gbs)),
               launches=launches_per_replay * replays * len(win_ms),
               launches_per_step=launches_per_replay / R,
               step_ms=med_ms / K, step_bytes=bytes_per_window / K)
    if pre_ms:
        res.update(pre_ms=float(np.mean(pre_ms)), pre_p10=float(np.percentile(pre_ms, 10)),
                   pre_p90=float(np.percentile(pre_ms, 90)))
    if with_e2e:
        e2e = time_e2e(W, dev, max(20, min(K, 256)))
        res["e2e"] = e2e
        res["e2e_val"] = reduce_sum(e2e["bytes"], world) / reduce_max(e2e["seconds"], world) / 1e9
        if e2e["direct"] is not None:
            e2e["direct_val"] = (reduce_sum(e2e["direct"]["bytes"], world) /
                                 reduce_max(e2e["direct"]["seconds"], world) / 1e9)
        if e2e.get("pipelined") is not None:
            e2e["pipelined_val"] = (reduce_sum(e2e["pipelined"]["bytes"], world) /
                                    reduce_max(e2e["pipelined"]["seconds"], world) / 1e9)
    return res


class PrefillHostIO:
    """The prefill part's per-step inputs (q, qo_indptr, kv_lens, block
    tables) in one pinned host buffer with 256-byte aligned fields, copied
    to a device buffer of the same layout; its output read back into pinned
    host memory."""

    def __init__(self, P, dev):
        pb = P.pb
        self.P = P
        src = {"q": pb.q, "qo_indptr": pb.qo_indptr, "kv_lens": pb.kv_lens,
               "block_tables": pb.block_tables}
        offs, total = {}, 0
        for k, t in src.items():
            offs[k] = total
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        self.host = torch.empty(total, dtype=torch.uint8).pin_memory()
        for k, t in src.items():
            n = t.numel() * t.element_size()
            self.host[offs[k]:offs[k] + n].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
        self.dev_all = torch.empty(total, dtype=torch.uint8, device=dev)
        self.buf = {k: self.dev_all[offs[k]:offs[k] + t.numel() * t.element_size()]
                    .view(t.dtype).view(t.shape) for k, t in src.items()}
        self.out_h = torch.empty(P.out.shape, dtype=P.out.dtype).pin_memory()
        self.h2d = sum(t.numel() * t.element_size() for t in src.values())
        self.d2h = self.out_h.numel() * self.out_h.element_size()

    def step(self):
        P, b = self.P, self.buf
        self.dev_all.copy_(self.host, non_blocking=True)
        P.pkv.pkv_prefill_attention_ragged(P.desc, b["q"], b["qo_indptr"], P.pb.k_cache,
                                           P.pb.v_cache, b["block_tables"], b["kv_lens"],
                                           P.spec.sm_scale, P.out,
                                           qo_indptr_host=P.pb.qo_indptr_host,
                                           kv_lens_host=P.pb.kv_lens_host)
        self.out_h.copy_(P.out, non_blocking=True)


def time_e2e(W, dev, steps):
    """The same step through the public API with host buffers: each step
    copies its inputs from pinned host memory (one copy of one packed buffer
    per part), runs the decode step (append + decode) and, in the mixed step,
    the prefill, and reads the outputs back to the host."""
    pkv = W.pkv
    # A step's inputs sit in one pinned host buffer (256-byte aligned fields)
    # and go over in one copy into one device buffer with the same layout.
    names = ["q", "k_new", "v_new", "block_tables", "context_lens"] + ([] if W.fused else ["pos"])
    src0 = {k: (W.pos[0] if k == "pos" else getattr(W.insts[0], k)) for k in names}
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += (src0[k].numel() * src0[k].element_size() + 255) // 256 * 256
    host = []
    for b, pos in zip(W.insts, W.pos):
        hb = torch.empty(total, dtype=torch.uint8).pin_memory()
        for k in names:
            t = (pos if k == "pos" else getattr(b, k)).cpu().contiguous()
            nbytes = t.numel() * t.element_size()
            hb[offs[k]:offs[k] + nbytes].copy_(t.view(-1).view(torch.uint8))
        host.append(hb)
    dev_all = torch.empty(total, dtype=torch.uint8, device=dev)
    devbuf = {}
    for k in names:
        t = src0[k]
        nbytes = t.numel() * t.element_size()
        devbuf[k] = dev_all[offs[k]:offs[k] + nbytes].view(t.dtype).view(t.shape)
    out_h = torch.empty(W.out.shape, dtype=W.out.dtype).pin_memory()
    pio = PrefillHostIO(W.prefill, dev) if W.prefill is not None else None
    h2d = sum(src0[k].numel() * src0[k].element_size() for k in names) + (pio.h2d if pio else 0)
    d2h = out_h.numel() * out_h.element_size() + (pio.d2h if pio else 0)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream  # the raw handle, passed to the API calls

    # the decode-step calls of each (batch, layer), marshalled once (bound buffers)
    bound = {}
    if W.fused:
        for j in range(W.n_inst):
            for li, (layer, w) in enumerate(zip(W.layers, W.windows)):
                b = layer[j]
                bound[(j, li)] = pkv.bind_decode_step(
                    W.desc, devbuf["q"], devbuf["k_new"], devbuf["v_new"], b.k_cache, b.v_cache,
                    devbuf["block_tables"], devbuf["context_lens"], W.max_ctx, W.spec.sm_scale,
                    W.out, None, W.ws, cos_sin=W.table, window=w, chunk_blocks=W.chunk,
                    k_scale=b.k_scale, v_scale=b.v_scale, stream=sh)

    def one(i):
        dev_all.copy_(host[i % W.n_inst], non_blocking=True)
        for li, (layer, w) in enumerate(zip(W.layers, W.windows)):
            b = layer[i % W.n_inst]
            if W.fused:
                bound[(i % W.n_inst, li)]()
                continue
            pkv.pkv_append_rope(W.desc, b.k_cache, b.v_cache, devbuf["block_tables"], W.seq_ids,
                                devbuf["pos"], devbuf["k_new"], devbuf["v_new"], q=devbuf["q"],
                                cos_sin=W.table, k_scale=b.k_scale, v_scale=b.v_scale)
            pkv.pkv_decode_attention(W.desc, devbuf["q"], b.k_cache, b.v_cache,
                                     devbuf["block_tables"], devbuf["context_lens"], W.max_ctx,
                                     W.spec.sm_scale, W.out, None, W.ws, window=w,
                                     chunk_blocks=W.chunk, k_scale=b.k_scale, v_scale=b.v_scale)
        out_h.copy_(W.out, non_blocking=True)
        if pio is not None:
            pio.step()
        stream.synchronize()   # the host reads the step's result

    for i in range(8):
        one(i)
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    sec = time.perf_counter() - t0
    nbytes = sum(W.kv_bytes(i % W.n_inst) for i in range(steps))
    res = {"seconds": sec, "bytes": nbytes, "steps": steps, "h2d": h2d, "d2h": d2h, "direct": None}
    if not W.fused:
        return res

    # The same step with the decode's per-step arrays left in pinned host
    # memory: the decode step reads q, k_new, v_new, the tables and lengths
    # over the host link and writes the output into pinned host memory (no
    # copy-engine transfers); the prefill part of a mixed step still copies
    # its inputs in and its output out.  Then the host syncs and reads.
    views = []
    for hb in host:
        views.append({k: hb[offs[k]:offs[k] + src0[k].numel() * src0[k].element_size()]
                      .view(src0[k].dtype).view(src0[k].shape) for k in names})
    direct = {}
    for j in range(W.n_inst):
        v = views[j]
        for li, (layer, w) in enumerate(zip(W.layers, W.windows)):
            b = layer[j]
            direct[(j, li)] = pkv.bind_decode_step(
                W.desc, v["q"], v["k_new"], v["v_new"], b.k_cache, b.v_cache, v["block_tables"],
                v["context_lens"], W.max_ctx, W.spec.sm_scale, out_h, None, W.ws, cos_sin=W.table,
                window=w, chunk_blocks=W.chunk, k_scale=b.k_scale, v_scale=b.v_scale, stream=sh)

    def step_direct(i):
        for li in range(len(W.layers)):
            direct[(i % W.n_inst, li)]()
        if pio is not None:
            pio.step()
        stream.synchronize()   # the host reads the step's result (already in out_h)

    for i in range(8):
        step_direct(i)
    t0 = time.perf_counter()
    for i in range(steps):
        step_direct(i)
    res["direct"] = {"seconds": time.perf_counter() - t0, "bytes": nbytes}

    # Pipelined, as a serving loop runs it: the same copies and calls, with
    # two slots of device inputs and outputs.  Step i+1's inputs go H2D on a
    # copy stream while step i computes, and step i's outputs come back D2H
    # on another while step i+1 computes; events order each slot's reuse.
    # The host reads every step's result (one step behind the issue).
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    dev_in = [dev_all, torch.empty_like(dev_all)]
    bufs = [devbuf, {k: dev_in[1][offs[k]:offs[k] + src0[k].numel() * src0[k].element_size()]
                     .view(src0[k].dtype).view(src0[k].shape) for k in names}]
    outs = [W.out, torch.empty_like(W.out)]
    outs_h = [out_h, torch.empty(W.out.shape, dtype=W.out.dtype).pin_memory()]
    slot_calls = {}
    for sl in range(2):
        for j in range(W.n_inst):
            for li, (layer, w) in enumerate(zip(W.layers, W.windows)):
                b = layer[j]
                slot_calls[(sl, j, li)] = pkv.bind_decode_step(
                    W.desc, bufs[sl]["q"], bufs[sl]["k_new"], bufs[sl]["v_new"], b.k_cache, b.v_cache,
                    bufs[sl]["block_tables"], bufs[sl]["context_lens"], W.max_ctx, W.spec.sm_scale,
                    outs[sl], None, W.ws, cos_sin=W.table, window=w, chunk_blocks=W.chunk,
                    k_scale=b.k_scale, v_scale=b.v_scale, stream=sh)
    if pio is not None:
        P = W.prefill
        p_dev = [pio.dev_all, torch.empty_like(pio.dev_all)]
        p_buf = [pio.buf, {k: p_dev[1][v.data_ptr() - pio.dev_all.data_ptr():
                                       v.data_ptr() - pio.dev_all.data_ptr() + v.numel() * v.element_size()]
                           .view(v.dtype).view(v.shape) for k, v in pio.buf.items()}]
        p_out = [P.out, torch.empty_like(P.out)]
        p_out_h = [pio.out_h, torch.empty(P.out.shape, dtype=P.out.dtype).pin_memory()]
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_comp = [torch.cuda.Event(), torch.cuda.Event()]
    ev_out = [torch.cuda.Event(), torch.cuda.Event()]

    def issue_in(i):
        sl = i % 2
        if i >= 2:
            s_in.wait_event(ev_comp[sl])      # step i-2 is done with this slot's inputs
        with torch.cuda.stream(s_in):
            dev_in[sl].copy_(host[i % W.n_inst], non_blocking=True)
            if pio is not None:
                p_dev[sl].copy_(pio.host, non_blocking=True)
        ev_in[sl].record(s_in)

    def issue_compute(i):
        sl = i % 2
        stream.wait_event(ev_in[sl])
        if i >= 2:
            stream.wait_event(ev_out[sl])     # step i-2's outputs have left this slot
        def prefill():
            b = p_buf[sl]
            pkv.pkv_prefill_attention_ragged(P.desc, b["q"], b["qo_indptr"], P.pb.k_cache, P.pb.v_cache,
                                             b["block_tables"], b["kv_lens"], P.spec.sm_scale, p_out[sl],
                                             qo_indptr_host=P.pb.qo_indptr_host,
                                             kv_lens_host=P.pb.kv_lens_host, stream=sh)
        if pio is not None and W.independent:
            prefill()   # the step's order, as in the timed graph
        for li in range(len(W.layers)):
            slot_calls[(sl, i % W.n_inst, li)]()
        if pio is not None and not W.independent:
            prefill()
        ev_comp[sl].record(stream)

    def issue_out(i):
        sl = i % 2
        s_out.wait_event(ev_comp[sl])
        with torch.cuda.stream(s_out):
            outs_h[sl].copy_(outs[sl], non_blocking=True)
            if pio is not None:
                p_out_h[sl].copy_(p_out[sl], non_blocking=True)
        ev_out[sl].record(s_out)

    def run_pipelined(n):
        issue_in(0)
        for i in range(n):
            if i + 1 < n:
                issue_in(i + 1)
            issue_compute(i)
            issue_out(i)
            if i >= 1:
                ev_out[(i - 1) % 2].synchronize()   # the host reads step i-1's result
        ev_out[(n - 1) % 2].synchronize()

    run_pipelined(8)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run_pipelined(steps)
    res["pipelined"] = {"seconds": time.perf_counter() - t0, "bytes": nbytes}
    torch.cuda.synchronize()
    return res


def e2e_line(e, copy_val, mixed=False):
    """The e2e object of the bench line.  Every variant moves each step's
    inputs host -> device and its output device -> host inside the timed
    region; the line's value is the fastest public-API variant, and all of
    them are listed."""
    copies = {"value": round(copy_val, 2), "unit": "GB/s",
              "note": "per step: one pinned H2D of the step's packed inputs (copy engine), the "
                      "decode-step call (append+RoPE+decode; arguments bound once with "
                      "bind_decode_step), D2H of the output (copy engine), host sync"}
    base = {"unit": "GB/s", "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
            "steps": e["steps"]}
    if mixed:
        base["prefill_part"] = ("each step also copies the prefill part's q, qo_indptr, kv_lens "
                                "and block tables H2D (one packed pinned buffer, copy engine), "
                                "runs the ragged prefill, and copies its output D2H")
    if e.get("direct_val") is None:
        return dict(base, value=copies["value"], note=copies["note"])
    direct = {"value": round(e["direct_val"], 2), "unit": "GB/s",
              "note": "per step: the decode-step call with the step's inputs in pinned host "
                      "memory (q, k_new, v_new, block tables, lengths; the kernel reads them over "
                      "NVLink-C2C) and its output written into pinned host memory, then a host "
                      "sync; table entries past a sequence's blocks are not read"}
    variants = {"with_copies": copies, "direct": direct}
    if e.get("pipelined_val") is not None:
        variants["pipelined"] = {
            "value": round(e["pipelined_val"], 2), "unit": "GB/s",
            "note": "per step, as a serving loop runs it: the step's packed inputs go H2D (copy "
                    "engine, pinned host memory) on one stream while the previous step computes, "
                    "the decode-step call (and the prefill) run on the compute stream, the outputs "
                    "come back D2H on a third stream while the next step computes; two slots of "
                    "device inputs and outputs, ordered by events; the host waits for every "
                    "step's output, one step behind the issue"}
    # the line's value is the fastest of the public-API variants; all are listed
    best = max(variants, key=lambda k: variants[k]["value"])
    return dict(base, value=variants[best]["value"], note=variants[best]["note"], variant=best,
                variants=variants)


# ---------------------------------------------------------- CPU baseline --

def oracle_sample(W, seconds, nthreads):
    """Time the CPU oracle on whole sequences of instance 0 (all heads) until
    about `seconds` of wall time; returns (GB/s, description, threads)."""
    import oracle
    b = W.insts[0]
    spec = W.spec

    def host_pool(seqs):
        tabs = b.tables_host[seqs]
        ids = np.unique(tabs[tabs >= 0])
        remap = np.full(int(b.k_cache.shape[0]), -1, dtype=np.int64)
        remap[ids] = np.arange(len(ids))
        idx = torch.from_numpy(ids.astype(np.int64)).to(b.k_cache.device)
        to_np = (lambda t: t.cpu().numpy()) if b.k_cache.dtype == torch.uint8 else \
            (lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16))
        k = to_np(b.k_cache.index_select(0, idx))
        v = to_np(b.v_cache.index_select(0, idx))
        return k, v, np.where(tabs >= 0, remap[np.maximum(tabs, 0)], -1).astype(np.int32)

    q_all = b.q.view(torch.int16).cpu().numpy().view(np.uint16)
    ks = None if b.k_scale is None else b.k_scale.cpu().numpy()
    vs = None if b.v_scale is None else b.v_scale.cpu().numpy()
    kvd = 1 if spec.kv_dtype == "fp8_e4m3" else 0
    elem = 1 if kvd else 2
    order = np.argsort(b.lens_host)  # start short, grow; wrap around until the time is spent
    done_bytes, done_s, seqs_done = 0, 0.0, 0
    batch = 1
    pos = 0
    while done_s < seconds:
        seqs = [int(order[(pos + j) % len(order)]) for j in range(batch)]
        k, v, tabs = host_pool(seqs)
        lens = b.lens_host[seqs]
        t0 = time.perf_counter()
        oracle.paged_attention(q=q_all[seqs], k_cache=k, v_cache=v, block_tables=tabs,
                               qo_indptr=np.arange(len(seqs) + 1), kv_lens=lens,
                               num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                               sm_scale=spec.sm_scale, kv_dtype=kvd, k_scale=ks, v_scale=vs,
                               nthreads=nthreads, with_lse=False)
        done_s += time.perf_counter() - t0
        done_bytes += int(lens.sum()) * spec.num_kv_heads * spec.head_dim * elem * 2
        seqs_done += len(seqs)
        pos += batch
        batch = min(batch * 2, len(order))
    desc = ("%d sequence passes over one %d-sequence batch (all %d query heads, "
            "host copies of their blocks), %.1f s of oracle time" % (
                seqs_done, spec.batch, spec.num_q_heads, done_s))
    return done_bytes / done_s / 1e9, desc, nthreads


# ------------------------------------------------------------------ main --

def workload_config(W, extra=None):
    s = W.spec
    cfg = {"workload": s.name, "batch": s.batch, "num_q_heads": s.num_q_heads,
           "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim, "block_size": s.block_size,
           "kv_dtype": s.kv_dtype, "ctx": [s.ctx_lo, s.ctx_hi], "pool_blocks":
               int(W.insts[0].k_cache.shape[0]),
           "l2": "%d batches over disjoint pool regions rotate step by step (%.0f MB of K/V "
                 "per rotation > 129 MB L2)" % (W.n_inst, sum(W.kv_bytes(i) for i in
                                                               range(W.n_inst)) / 1e6)
           if W.n_inst > 1 else "K/V per step (%.1f GB) far exceeds the 129 MB L2" %
                                 (W.kv_bytes(0) / 1e9),
           "parallelism": "replicas: independent batches per GPU, no collective",
           "step": ("one launch per layer: append+RoPE of the new token fused into split-KV "
                    "decode (pkv_decode_step), replayed as a CUDA graph" if W.fused else
                    "append+RoPE of the new token, then split-KV decode: two launches per "
                    "layer, replayed as a CUDA graph")}
    if W.prefill is not None:
        cfg["step"] = (("ragged causal prefill of 8x512 tokens over shared prefixes, then " + cfg["step"] +
                        "; the decode does not wait for the prefill (PKV_DESC_INDEPENDENT: the two "
                        "halves of one layer's mixed step) and waits at its end")
                       if W.independent else
                       cfg["step"] + " + ragged causal prefill of 8x512 tokens over shared prefixes")
    cfg["prefetch_kv"] = W.prefetch
    if extra:
        cfg.update(extra)
    return cfg


def main_prefill(args, rank, world, local):
    """The prefill part of the Llama-3-8B-shaped mixed step on its own: 8 chunks
    of 512 query tokens over cached prefixes U[0, 8192], 32/8 heads, D 128,
    causal.  Each timed launch follows an L2 flush (L2Flush)."""
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    P = PrefillPart(dev, rank)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        P.run()
    torch.cuda.synchronize(dev)
    K = max(1, args.steps)
    times = []
    sampler = ClockSampler(dev.index)
    barrier(world)
    for _ in range(K):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        P.run()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    barrier(world)
    ms = reduce_max(float(np.mean(times)), world)
    flags = P.pkv.pkv_device_errors(reset=True)
    if flags:
        raise RuntimeError("device error word 0x%x after the prefill runs" % flags)
    if rank != 0:
        return
    peak, kind = measured_tensor_peak()
    tflops = P.flops / (ms / 1e3) / 1e12
    line = {
        "metric": "ragged causal chunked-prefill attention TFLOP/s on 1 GB300",
        "value": round(tflops * world, 1),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": max(3, args.warmup),
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) q/K/V, shared-prefix block tables",
        "config": {"workload": P.spec.name, "num_q_heads": P.spec.num_q_heads,
                   "num_kv_heads": P.spec.num_kv_heads, "head_dim": P.spec.head_dim,
                   "q_tokens": P.tokens, "causal": True,
                   "l2": L2_NOTE},
        "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                     "traffic": kernel_traffic_per_launch("prefill_tc_kernel", 4),
                     "kernel": "prefill_tc_kernel (tcgen05, two query tiles per CTA)",
                     "peak_source": "%s bf16_tflops (burst)" % kind,
                     "algorithmic_flops_per_launch": int(P.flops),
                     "avg_launch_ms": round(ms, 5),
                     "p10_ms": round(float(np.percentile(times, 10)), 5),
                     "p90_ms": round(float(np.percentile(times, 90)), 5)},
        "gpu_launches": K,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------ next-step parts --

class L2Flush:
    """Between timed launches: write a 256 MiB buffer (twice L2), then read
    another 256 MiB buffer.  The read evicts the written lines, so their
    write-back to DRAM happens here and not inside the next timed launch,
    which then starts against an L2 of clean lines that hold none of its
    inputs."""

    def __init__(self, dev):
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(64 << 20, dtype=torch.int32, device=dev)

    def zero_(self):
        self.w.zero_()
        self.r.sum()


L2_NOTE = "before every timed launch a 256 MiB write, then a 256 MiB read (L2 left clean)"


def _timed_launches(run, K, W, dev, flush):
    """W untimed launches, then K launches each after an L2 flush (L2Flush,
    outside the events), timed with CUDA events on the launching stream.
    Returns (per-launch ms list, clocks)."""
    stream = torch.cuda.current_stream(dev)
    for _ in range(W):
        run()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index)
    times = []
    for _ in range(K):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    torch.cuda.synchronize(dev)
    return times, sampler.stop()


def _part_line(args, world, metric, value, unit, ms_list, dtype, config, roofline, launches,
               clocks, extra=None):
    ms = float(np.mean(ms_list))
    roofline = dict(roofline, avg_launch_ms=round(ms, 5),
                    p10_ms=round(float(np.percentile(ms_list, 10)), 5),
                    p90_ms=round(float(np.percentile(ms_list, 90)), 5))
    line = {"metric": metric, "value": round(value, 2), "unit": unit, "n_gpus": world,
            "steps": len(ms_list), "warmup": max(3, args.warmup), "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
            "data": "synthetic: seeded N(0,1) values, seeded lengths and scattered block tables",
            "config": dict(config, l2=L2_NOTE),
            "roofline": roofline, "gpu_launches": launches * len(ms_list), "clocks": clocks}
    if extra:
        line.update(extra)
    print(json.dumps(line), flush=True)


def main_next(args, rank, world, local):
    """One next-step row on its own seeded workload (rank 0 reports):
      cascade     shared-prefix decode (16 groups x 8 sequences, 32/8 heads, D128), KV GB/s
                  with each prefix read once, beside plain decode over the same contexts;
      verify      speculative-verify queries of 2-8 tokens per sequence through the ragged
                  kernel on the Qwen2.5-3B-shaped cache, KV GB/s and query tokens/s;
      cow         copy-on-write of 4096 whole blocks of that pool, GB/s moved;
      ring        the FP8 workload's window-128 layer over a 9-block ring cache with sink
                  logits, one decode step (append + decode), KV GB/s;
      ring-prefill the FP8 workload's window layer taking a 512-token prefill chunk per
                  sequence over its 9-block ring: staging of the window, the cache commit
                  and the ragged prefill, GB/s of the bytes the path must move;
      fp8-prefill the Llama-3-8B-shaped prefill part over e4m3 pools (tcgen05 prefill,
                  tiles converted to f16 in shared memory), TFLOP/s."""
    import paged_kv_attention_21_gb300 as pkv
    from paged_kv_attention_21_gb300 import workloads as wl
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    flush = L2Flush(dev)
    K, W = max(1, args.steps), max(3, args.warmup)
    hbm, hbm_kind = measured_peaks()
    part = args.part

    if part == "cascade":
        spec = wl.CASCADE_DECODE
        if rank:
            spec = wl.dataclasses.replace(spec, seed=spec.seed + 7919 * rank)
        cb = wl.make_cascade_batch(spec, dev)
        B = spec.groups * spec.group_size
        desc = pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                             head_dim=spec.head_dim, num_blocks=cb.k_cache.shape[0],
                             max_blocks_per_seq=cb.prefix_tables.shape[1])
        max_suffix = int(cb.suffix_host.max())
        ws = torch.zeros(max(pkv.pkv_cascade_workspace_size(desc, spec.groups, B,
                                                            int(cb.prefix_host.max()), max_suffix), 256),
                         dtype=torch.uint8, device=dev)
        out = torch.empty_like(cb.q)
        run = lambda: pkv.pkv_cascade_decode(desc, cb.q, cb.k_cache, cb.v_cache, cb.group_indptr,
                                             cb.group_indptr_host, cb.prefix_tables, cb.prefix_lens,
                                             cb.prefix_host, cb.suffix_tables, cb.suffix_lens,
                                             max_suffix, spec.sm_scale, out, None, ws)
        times, clocks = _timed_launches(run, K, W, dev, flush)
        max_ctx = int(cb.prefix_host.max() + cb.suffix_host.max())
        wsd = torch.zeros(max(pkv.pkv_decode_workspace_size(desc, B, max_ctx, -1, 0), 256),
                          dtype=torch.uint8, device=dev)
        plain = lambda: pkv.pkv_decode_attention(desc, cb.q, cb.k_cache, cb.v_cache,
                                                 cb.concat_tables, cb.concat_lens, max_ctx,
                                                 spec.sm_scale, out, None, wsd)
        ptimes, _ = _timed_launches(plain, K, W, dev, flush)
        ms = reduce_max(float(np.mean(times)), world)
        pms = reduce_max(float(np.mean(ptimes)), world)
        if rank:
            return
        nbytes = cb.cascade_kv_bytes()
        gbs = nbytes / (ms / 1e3) / 1e9
        _part_line(args, world, "shared-prefix (cascade) decode KV GB/s, each prefix read once",
                   gbs * world, "GB/s", times, "bf16",
                   {"workload": spec.name, "sequences": B, "groups": spec.groups},
                   {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(gbs / hbm, 4), "traffic": None,
                    "kernel": "prefix pass (prefill_tc_kernel) + suffix decode + merge_kernel",
                    "peak_source": "%s hbm_gbs" % hbm_kind, "algorithmic_bytes_per_launch": nbytes},
                   3, clocks,
                   {"plain_decode": {"ms": round(pms, 5), "kv_bytes": cb.uncached_kv_bytes(),
                                     "speedup_of_cascade": round(pms / ms, 3),
                                     "note": "pkv_decode_attention over each sequence's "
                                             "concatenated prefix + suffix table"}})
        return

    if part in ("verify", "cow"):
        spec = wl.QWEN25_3B
        if rank:
            spec = wl.dataclasses.replace(spec, seed=spec.seed + 7919 * rank)
        b = wl.make_decode_batch(spec, dev)
        desc = pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                             head_dim=spec.head_dim, num_blocks=b.k_cache.shape[0],
                             max_blocks_per_seq=b.tables_host.shape[1])
        if part == "verify":
            rng = np.random.default_rng(spec.seed + 3)
            lo, hi = wl.VERIFY_Q_LENS
            ql = rng.integers(lo, hi + 1, size=spec.batch).astype(np.int32)
            qo = np.zeros(spec.batch + 1, np.int32)
            qo[1:] = np.cumsum(ql)
            g = torch.Generator(device=dev).manual_seed(spec.seed + 3)
            q = wl.fill_bf16((int(qo[-1]), spec.num_q_heads, spec.head_dim), g, dev)
            qo_d = torch.from_numpy(qo).to(dev)
            out = torch.empty_like(q)
            run = lambda: pkv.pkv_prefill_attention_ragged(
                desc, q, qo_d, b.k_cache, b.v_cache, b.block_tables, b.context_lens,
                spec.sm_scale, out, qo_indptr_host=qo, kv_lens_host=b.lens_host)
            times, clocks = _timed_launches(run, K, W, dev, flush)
            ms = reduce_max(float(np.mean(times)), world)
            if rank:
                return
            nbytes = b.kv_bytes()
            gbs = nbytes / (ms / 1e3) / 1e9
            _part_line(args, world, "speculative-verify attention (2-8 query tokens per sequence) "
                       "KV GB/s", gbs * world, "GB/s", times, "bf16",
                       {"workload": spec.name + ", q_len U[2,8] per sequence", "query_tokens":
                        int(qo[-1])},
                       {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                        "frac": round(gbs / hbm, 4), "traffic": None,
                        "kernel": "prefill_tc_kernel (one query tile holds every verify token)",
                        "peak_source": "%s hbm_gbs" % hbm_kind,
                        "algorithmic_bytes_per_launch": nbytes},
                       1, clocks, {"query_tokens_per_s": round(int(qo[-1]) / (ms / 1e3), 1)})
            return
        # cow: 4096 (src, dst) pairs, dst blocks outside every table
        used = set(b.tables_host[b.tables_host >= 0].tolist())
        free = np.array([i for i in range(b.k_cache.shape[0]) if i not in used], np.int32)
        rng = np.random.default_rng(spec.seed + 5)
        npairs = 4096
        src = rng.choice(np.array(sorted(used), np.int32), npairs, replace=False)
        dst = rng.choice(free, npairs, replace=False)
        src_d = torch.from_numpy(src.astype(np.int32)).to(dev)
        dst_d = torch.from_numpy(dst.astype(np.int32)).to(dev)
        run = lambda: pkv.pkv_copy_blocks(desc, b.k_cache, b.v_cache, src_d, dst_d)
        times, clocks = _timed_launches(run, K, W, dev, flush)
        ms = reduce_max(float(np.mean(times)), world)
        if rank:
            return
        block_bytes = spec.num_kv_heads * spec.block_size * spec.head_dim * 2
        nbytes = npairs * 2 * 2 * block_bytes  # K and V, read and written
        gbs = nbytes / (ms / 1e3) / 1e9
        _part_line(args, world, "copy-on-write block copy GB/s (read + write)", gbs * world, "GB/s",
                   times, "bytes", {"workload": "4096 whole-block copies in the Qwen2.5-3B-shaped "
                                                "pool (16 x 2 x 128 bf16 per block and pool)"},
                   {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(gbs / hbm, 4), "traffic": None, "kernel": "copy_blocks_kernel",
                    "peak_source": "%s hbm_gbs" % hbm_kind, "algorithmic_bytes_per_launch": nbytes},
                   1, clocks)
        return

    if part == "ring":
        spec = wl.FP8_DECODE
        if rank:
            spec = wl.dataclasses.replace(spec, seed=spec.seed + 7919 * rank)
        R, window = wl.FP8_RING, wl.FP8_WINDOW
        rng = np.random.default_rng(spec.seed + 11)
        lens = wl.draw_lengths(spec, rng)
        B = spec.batch
        g = torch.Generator(device=dev).manual_seed(spec.seed + 11)
        shape = (B * R, spec.num_kv_heads, spec.block_size, spec.head_dim)
        kc, ks = wl.fill_e4m3(shape, g, dev)
        vc, vs = wl.fill_e4m3(shape, g, dev)
        perm = rng.permutation(B * R).astype(np.int32).reshape(B, R)
        tabs = torch.from_numpy(perm).to(dev)
        lens_d = torch.from_numpy(lens.astype(np.int32)).to(dev)
        q = wl.fill_bf16((B, spec.num_q_heads, spec.head_dim), g, dev)
        kn = wl.fill_bf16((B, spec.num_kv_heads, spec.head_dim), g, dev)
        vn = wl.fill_bf16((B, spec.num_kv_heads, spec.head_dim), g, dev)
        sinks = torch.from_numpy(rng.uniform(-1.0, 3.0, spec.num_q_heads).astype(np.float32)).to(dev)
        table = torch.from_numpy(pkv.pkv_rope_cos_sin_table(spec.rope_theta, spec.head_dim,
                                                            spec.ctx_hi)).to(dev)
        desc = pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                             head_dim=spec.head_dim, num_blocks=B * R, max_blocks_per_seq=R,
                             kv_dtype=pkv.KV_FP8_E4M3, ring_blocks=R)
        max_ctx = int(lens.max())
        ws = torch.zeros(max(pkv.pkv_decode_workspace_size(desc, B, max_ctx, window, 0), 256),
                         dtype=torch.uint8, device=dev)
        out = torch.empty_like(q)
        run = lambda: pkv.pkv_decode_step(desc, q, kn, vn, kc, vc, tabs, lens_d, max_ctx,
                                          spec.sm_scale, out, None, ws, cos_sin=table,
                                          window=window, k_scale=ks, v_scale=vs, sinks=sinks)
        times, clocks = _timed_launches(run, K, W, dev, flush)
        ms = reduce_max(float(np.mean(times)), world)
        if rank:
            return
        nbytes = int(np.minimum(lens, window).astype(np.int64).sum()) * spec.num_kv_heads * \
            spec.head_dim * 1 * 2
        gbs = nbytes / (ms / 1e3) / 1e9
        _part_line(args, world, "sliding-window (128) decode step over a 9-block ring cache with "
                   "sink logits, KV GB/s", gbs * world, "GB/s", times, "e4m3 KV, bf16 q/o, fp32 "
                   "accumulate", {"workload": "FP8 workload's window layer: B128, 64/8 heads, D64, "
                                              "ctx U[1024,16384], ring of 9 blocks per sequence"},
                   {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(gbs / hbm, 4), "traffic": None,
                    "kernel": "decode_kernel (fused append, ring tables, sinks)",
                    "peak_source": "%s hbm_gbs" % hbm_kind, "algorithmic_bytes_per_launch": nbytes},
                   1, clocks)
        return

    if part == "ring-prefill":
        # 8 sequences of the FP8 workload's window layer each take a chunk of
        # 512 prompt tokens over a cached prefix U[1024, 16384], through the
        # ring cache: stage the window, commit the chunk, run the prefill
        spec = wl.FP8_DECODE
        R, window = wl.FP8_RING, wl.FP8_WINDOW
        rng = np.random.default_rng(spec.seed + 13 + 7919 * rank)
        B, ql = 8, 512
        prefix = rng.integers(spec.ctx_lo, spec.ctx_hi + 1, size=B).astype(np.int32)
        kv = (prefix + ql).astype(np.int32)
        g = torch.Generator(device=dev).manual_seed(spec.seed + 13 + 7919 * rank)
        shape = (B * R, spec.num_kv_heads, spec.block_size, spec.head_dim)
        kc, ks = wl.fill_e4m3(shape, g, dev)
        vc, vs = wl.fill_e4m3(shape, g, dev)
        perm = rng.permutation(B * R).astype(np.int32).reshape(B, R)
        tabs = torch.from_numpy(perm).to(dev)
        T = B * ql
        qo = np.arange(0, T + 1, ql, dtype=np.int32)
        q = wl.fill_bf16((T, spec.num_q_heads, spec.head_dim), g, dev)
        kch = wl.fill_bf16((T, spec.num_kv_heads, spec.head_dim), g, dev)
        vch = wl.fill_bf16((T, spec.num_kv_heads, spec.head_dim), g, dev)
        desc = pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                             head_dim=spec.head_dim, num_blocks=B * R, max_blocks_per_seq=R,
                             kv_dtype=pkv.KV_FP8_E4M3, ring_blocks=R)
        ws = torch.empty(pkv.pkv_prefill_ring_workspace_size(desc, B, window, ql), dtype=torch.uint8,
                         device=dev)
        out = torch.empty_like(q)
        qo_d = torch.from_numpy(qo).to(dev)
        kv_d = torch.from_numpy(kv).to(dev)
        run = lambda: pkv.pkv_prefill_ring_commit(desc, q, qo_d, kch, vch, kc, vc, tabs, kv_d,
                                                  spec.sm_scale, window, out, qo, kv, ws,
                                                  k_scale=ks, v_scale=vs)
        times, clocks = _timed_launches(run, K, W, dev, flush)
        ms = reduce_max(float(np.mean(times)), world)
        if rank:
            return
        # bytes the path must move: the ring keys of each window below the
        # chunk (e4m3 K and V), the chunk's K and V (bf16), the committed ring
        # slots (e4m3 K and V), q in and o out (bf16)
        H, D, Hq = spec.num_kv_heads, spec.head_dim, spec.num_q_heads
        below = int(np.minimum(prefix, window - 1).sum())
        committed = B * min(ql, R * spec.block_size)
        nbytes = (below * H * D * 2 + T * H * D * 2 * 2 + committed * H * D * 2 +
                  2 * T * Hq * D * 2)
        gbs = nbytes / (ms / 1e3) / 1e9
        _part_line(args, world, "sliding-window (128) ring-cache prefill with the cache commit, "
                   "GB/s of the bytes the path must move", gbs * world, "GB/s", times,
                   "e4m3 ring, bf16 chunk K/V, q and o, fp32 accumulate",
                   {"workload": "FP8 workload's window layer (64/8 heads, D64, 9-block ring per "
                                "sequence): 8 sequences x 512-token chunks over prefixes "
                                "U[1024,16384]", "q_tokens": T,
                    "query_tokens_per_s": round(T / (ms / 1e3), 1)},
                   {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(gbs / hbm, 4), "traffic": None,
                    "kernel": "stage_ring_kernel + commit_ring_kernel + prefill_tc_kernel",
                    "peak_source": "%s hbm_gbs" % hbm_kind, "algorithmic_bytes_per_launch": nbytes},
                   3, clocks)
        return

    # fp8-prefill: workload 4's prefill part with its pools quantised to e4m3
    P = PrefillPart(dev, rank)
    pb = P.pb
    amax_k = pb.k_cache.float().abs().amax(dim=(0, 2, 3))
    amax_v = pb.v_cache.float().abs().amax(dim=(0, 2, 3))
    ks = (amax_k / 448.0).contiguous()
    vs = (amax_v / 448.0).contiguous()
    k8 = (pb.k_cache.float() / ks.view(1, -1, 1, 1)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = (pb.v_cache.float() / vs.view(1, -1, 1, 1)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    spec = P.spec
    desc8 = pkv.make_desc(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                          head_dim=spec.head_dim, num_blocks=k8.shape[0],
                          max_blocks_per_seq=pb.tables_host.shape[1], kv_dtype=pkv.KV_FP8_E4M3)
    # no workspace: the tcgen05 kernel converts e4m3 tiles in shared memory
    run = lambda: pkv.pkv_prefill_attention_ragged(
        desc8, pb.q, pb.qo_indptr, k8, v8, pb.block_tables, pb.kv_lens, spec.sm_scale, P.out,
        qo_indptr_host=pb.qo_indptr_host, kv_lens_host=pb.kv_lens_host, k_scale=ks, v_scale=vs)
    times, clocks = _timed_launches(run, K, W, dev, flush)
    ms = reduce_max(float(np.mean(times)), world)
    if rank:
        return
    peak, kind = measured_tensor_peak()
    tflops = P.flops / (ms / 1e3) / 1e12
    _part_line(args, world, "ragged causal chunked-prefill attention over an e4m3 cache TFLOP/s",
               tflops * world, "TFLOP/s", times, "e4m3 KV converted to f16 in shared memory, f16 MMA, "
               "fp32 accumulate",
               {"workload": spec.name + ", e4m3 pools with per-head scales", "q_tokens": P.tokens},
               {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(tflops / peak, 4), "traffic": None,
                "kernel": "prefill_tc_kernel<e4m3> (K / V tiles converted to f16 in shared memory)",
                "peak_source": "%s bf16_tflops (burst; f16 runs at the bf16 rate)" % kind,
                "algorithmic_flops_per_launch": int(P.flops)},
               1, clocks)


NOMINAL_HBM_GBS = 8000.0   # GB300 HBM3e, nominal (~8 TB/s)

MIXED_STEP_NAME = ("Llama-3-8B-shaped mixed step: 120 decodes (ctx 1024-32768) + 8x512-token "
                   "causal prefill chunks over cached prefixes 0-8192, 32/8 heads, D128, bf16")


def workload_name(config):
    from paged_kv_attention_21_gb300 import workloads as wl
    return MIXED_STEP_NAME if config == 4 else wl.CONFIGS[config].name


def decode_roofline(r, peak, peak_kind, fused, config):
    """The decode kernel's roofline.  When every launch of the step is a
    decode_kernel launch (no prefill, no separate append), the timed windows
    themselves give its average launch duration as launches run back to back:
    window time / launches.  Events around single launches (kept below as
    isolated_*) cut the programmatic dependent launch between neighbours, so
    they time a launch without the overlap the stream gives it.  The mixed
    step also runs the prefill, so there the bracketed launches are the
    measurement."""
    iso = r["dom_bytes"] / (r["dom_ms"] / 1e3) / 1e9
    whole = fused and r["W"].prefill is None
    if whole:
        n = r["launches_per_step"]
        bytes_launch = r["step_bytes"] / n
        ms_launch = r["step_ms"] / n
    else:
        bytes_launch, ms_launch = r["dom_bytes"], r["dom_ms"]
    achieved = bytes_launch / (ms_launch / 1e3) / 1e9
    out = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
           "frac": round(achieved / peak, 4),
           "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
           "traffic": kernel_traffic_per_launch("decode_kernel", config),
           "kernel": ("decode_kernel (append+RoPE, split-KV GQA decode and merge, one launch)"
                      if fused else "decode_kernel (split-KV GQA decode, merge fused)"),
           "peak_source": "%s hbm_gbs" % peak_kind,
           "algorithmic_bytes_per_launch": int(bytes_launch),
           "avg_launch_ms": round(ms_launch, 5)}
    if whole:
        out.update({
            "timed_by": "CUDA events around each timed window of graph replays; every launch "
                        "of the step is decode_kernel: window time / launches",
            "isolated_launch_ms": round(r["dom_ms"], 5),
            "isolated_bytes_per_launch": int(r["dom_bytes"]),
            "frac_isolated": round(iso / peak, 4),
            "isolated_timed_by": "CUDA events around the decode launch of every %d-th step of the "
                                 "last graph replay of every window (an event between two launches "
                                 "cuts their overlap)" % r["ev_stride"]})
    else:
        out["timed_by"] = ("CUDA events around the decode launch of every %d-th step of every "
                           "timed window's last graph replay" % r["ev_stride"])
    out.update({"p10_launch_ms": round(r["dec_p10"], 5), "p90_launch_ms": round(r["dec_p90"], 5),
                "median_launch_gbs": round(r["per_launch_gbs"], 1)})
    return out


def main():
    args = parse_args()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        return main_reference(args, rank, world, local)
    if args.part == "prefill":
        return main_prefill(args, rank, world, local)
    if args.part != "step":
        return main_next(args, rank, world, local)
    r = time_pkv(args, rank, world, local)
    carry = None
    if args.config == 4 and not args.no_carry:
        # the Qwen2.5-3B-shaped decode step, carried beside the headline: its
        # short (~30 us) launches show the start-up and tail costs
        carry = time_pkv(args, rank, world, local, config=2, steps=640, min_seconds=0.5,
                         with_e2e=False)
    if rank != 0:
        return
    W = r["W"]
    peak, peak_kind = measured_peaks()
    value = r["total_bytes"] / r["elapsed_s"] / 1e9
    roof = decode_roofline(r, peak, peak_kind, W.fused, args.config)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": r["K"],
        "warmup": max(3, args.warmup),
        "ms_per_step": round(r["elapsed_s"] * 1e3 / r["K"], 5),
        "ms_per_step_p10": round(r["win_p10"] / r["K"], 5),
        "ms_per_step_p90": round(r["win_p90"] / r["K"], 5),
        "windows": r["windows"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if W.spec.kv_dtype == "bf16" else "e4m3 KV, bf16 q/o, fp32 accumulate",
        "data": "synthetic: seeded N(0,1) K/V/q, uniform context lengths, scattered block tables",
        "config": workload_config(W, {"workload": workload_name(args.config),
                                      "timing": "%d back-to-back windows of %d steps (CUDA "
                                                "events, graph replays); ms_per_step is the "
                                                "median window" % (r["windows"], r["K"])}),
        "pct_hbm_peak": round(100.0 * value / world / peak, 2),
        "pct_nominal_hbm": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
        "attention_tokens_per_s": round(r["total_tokens"] / r["elapsed_s"], 1),
        "roofline": roof,
        "e2e": e2e_line(r["e2e"], r["e2e_val"], W.prefill is not None),
        "gpu_launches": r["launches"],
        "gpu_launches_per_step": r["launches_per_step"],
        "clocks": r["clocks"],
    }
    roof["decode"] = {k: v for k, v in roof.items() if k != "decode"}
    if W.prefill is not None:
        tpeak, tkind = measured_tensor_peak()
        tsus, _ = measured_tensor_peak(sustained=True)
        P = W.prefill
        tflops = P.flops / (r["pre_ms"] / 1e3) / 1e12
        roof["prefill"] = {
            "bound": "tensor", "achieved": round(tflops, 1), "peak": tpeak, "unit": "TFLOP/s",
            "frac": round(tflops / tpeak, 4), "frac_of_sustained": round(tflops / tsus, 4),
            "traffic": kernel_traffic_per_launch("prefill_tc_kernel", 4),
            "kernel": "prefill_tc_kernel (tcgen05, two query tiles per CTA)",
            "peak_source": "%s bf16_tflops (burst); frac_of_sustained against "
                           "bf16_tflops_sustained" % tkind,
            "algorithmic_flops_per_launch": int(P.flops),
            "avg_launch_ms": round(r["pre_ms"], 5),
            "p10_launch_ms": round(r["pre_p10"], 5), "p90_launch_ms": round(r["pre_p90"], 5),
            "timed_by": "CUDA events around the prefill launch of every %d-th step of every "
                        "timed window's last graph replay" % r["ev_stride"]}
        line["prefill"] = {"tokens": P.tokens, "flops": P.flops, "kv_bytes": P.kv_bytes}
    if carry is not None:
        cW = carry["W"]
        cv = carry["total_bytes"] / carry["elapsed_s"] / 1e9
        croof = decode_roofline(carry, peak, peak_kind, cW.fused, 2)
        line["qwen25_3b_decode"] = {
            "workload": workload_name(2), "value": round(cv, 2), "unit": "GB/s",
            "steps": carry["K"], "windows": carry["windows"],
            "ms_per_step": round(carry["elapsed_s"] * 1e3 / carry["K"], 5),
            "frac_per_step": round(cv / world / peak, 4),
            "frac_per_launch": croof["frac"], "avg_launch_ms": croof["avg_launch_ms"],
            "frac_isolated_launch": croof.get("frac_isolated"),
            "isolated_launch_ms": croof.get("isolated_launch_ms"),
            "prefetch_kv": cW.prefetch,
            "median_launch_gbs": croof["median_launch_gbs"],
            "algorithmic_bytes_per_launch": croof["algorithmic_bytes_per_launch"],
            "traffic": croof["traffic"],
            "l2": "4 batches over disjoint pool regions rotate step by step"}
    if not args.no_cpu_baseline:
        ncores = os.cpu_count() or 1
        v, desc, thr = oracle_sample(W, args.cpu_seconds, ncores)
        v1, desc1, _ = oracle_sample(W, max(2.0, args.cpu_seconds / 3), 1)
        line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": thr,
                                "kind": "oracle", "sample": desc,
                                "single_core": {"value": round(v1, 4), "unit": "GB/s",
                                                "cores": 1, "sample": desc1}}
    print(json.dumps(line), flush=True)


def main_reference(args, rank, world, local):
    """The reference arm: the CPU oracle, as it stands, on the host cores,
    each step a bounded sample of the same workload."""
    if rank != 0:
        return
    import oracle
    from paged_kv_attention_21_gb300 import workloads as wl
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    spec = wl.CONFIGS[args.config]
    b = wl.make_decode_batch(spec, "cpu" if dev.type == "cpu" else dev)
    nthreads = os.cpu_count() or 1
    q_all = b.q.view(torch.int16).cpu().numpy().view(np.uint16)
    to_np = (lambda t: t.cpu().numpy()) if b.k_cache.dtype == torch.uint8 else \
        (lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16))
    # host copy of the first few sequences' blocks
    nseq = min(spec.batch, 8)
    tabs = b.tables_host[:nseq]
    ids = np.unique(tabs[tabs >= 0])
    remap = np.full(int(b.k_cache.shape[0]), -1, dtype=np.int64)
    remap[ids] = np.arange(len(ids))
    idx = torch.from_numpy(ids.astype(np.int64)).to(b.k_cache.device)
    k, v = to_np(b.k_cache.index_select(0, idx)), to_np(b.v_cache.index_select(0, idx))
    tabs = np.where(tabs >= 0, remap[np.maximum(tabs, 0)], -1).astype(np.int32)
    ks = None if b.k_scale is None else b.k_scale.cpu().numpy()
    vs = None if b.v_scale is None else b.v_scale.cpu().numpy()
    kvd = 1 if spec.kv_dtype == "fp8_e4m3" else 0
    elem = 1 if kvd else 2
    budget = 150.0  # seconds for the whole warm-up + timed run
    # time one sequence to size the per-step sample
    t0 = time.perf_counter()
    oracle.paged_attention(q=q_all[:1], k_cache=k, v_cache=v, block_tables=tabs[:1],
                           qo_indptr=[0, 1], kv_lens=b.lens_host[:1],
                           num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                           sm_scale=spec.sm_scale, kv_dtype=kvd, k_scale=ks, v_scale=vs,
                           nthreads=nthreads, with_lse=False)
    t_one = max(time.perf_counter() - t0, 1e-5)
    steps_total = args.steps + max(3, args.warmup)
    per_step = budget / steps_total
    nseq_step = int(max(1, min(nseq, per_step / t_one)))

    def step(i):
        s0 = (i * nseq_step) % nseq
        sel = [(s0 + j) % nseq for j in range(nseq_step)]
        oracle.paged_attention(q=q_all[sel], k_cache=k, v_cache=v, block_tables=tabs[sel],
                               qo_indptr=np.arange(len(sel) + 1), kv_lens=b.lens_host[sel],
                               num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                               sm_scale=spec.sm_scale, kv_dtype=kvd, k_scale=ks, v_scale=vs,
                               nthreads=nthreads, with_lse=False)
        return int(b.lens_host[sel].sum()) * spec.num_kv_heads * spec.head_dim * elem * 2, len(sel)

    for i in range(max(3, args.warmup)):
        step(i)
    t0 = time.perf_counter()
    nbytes = ntok = 0
    for i in range(args.steps):
        bb, nt = step(i)
        nbytes += bb
        ntok += nt
    sec = time.perf_counter() - t0
    value = nbytes / sec / 1e9
    sample = ("per step %d of the first %d decode sequences of one %s batch (all query heads)"
              % (nseq_step, nseq, spec.name))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": round(sec * 1e3 / max(1, args.steps), 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic: the same seeded workload", "config": {
                "workload": workload_name(args.config), "sample": sample},
            "attention_tokens_per_s": round(ntok / sec, 2),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nthreads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
