"""Benchmark of the write-time KV-cache hot path on GB300 (one JSON line on stdout).

Workload (default): the steady denoise step of a 60-block streaming video DiT --
every block has its own 5,788-slot ring of 16 heads x 128; each step writes one
757-token chunk per block and runs 4 attention calls per block (240 per step),
with the position reset (one delta rotation of every cached K) every 42 steps.
A "step" is one pass of the whole hot path: [rebase when due] + 60 x write +
240 x attend, enqueued through the C ABI on one stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvring|reference]

* value: steps/s over all ranks (replicas: each rank runs the full workload on
  its own GPU; no data-path collective), inputs resident in HBM.
* e2e: the same steps with each step's K, V, Q copied host->device from pinned
  memory and all 240 attention outputs (one buffer per layer and pass) copied
  back to pinned host memory, inside the timed region; one copy per kind and
  step (the chunks laid out contiguously), on a second stream.
* The timed steps start at a reset step (positions reset before that step's
  writes), so K timed steps hold ceil(K / 42) rebases: at least the reset's
  share of the path, never less.
* roofline: the attention call (Q-prep + attention + split combine launches),
  algorithmic FLOP 4*T*R*d*H per call at a full ring, against the measured
  bf16 peak x 2 (FP8); plus the write kernel against measured HBM bandwidth.
* cpu_baseline / --impl reference: the CPU oracle (naive per-call upkeep, then
  float64 attention) timed on this host.  A full step is hours of CPU work, so
  one timed "step" of the reference arm is one block's step (1 write + 4
  attention calls) and the step time is that x 60 blocks, marked extrapolated;
  the line's `steps` counts the full steps actually timed (block steps / 60).
  The tiny configuration (100 steps) and one production write + attention are
  timed whole, beside the GPU's time for the same work.  `upkeep` times the
  oracle's naive per-call upkeep against the write-time ring's on one block (the
  CPU analogue of the pages' upkeep comparison).
* --session: the unsharded-width session (60 blocks x 64 heads, 1,000 steps,
  resets every 42): per-step times (median, p99) and the drift against the
  oracle at steps 1, 41, 42, 43, 500 and 999.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 129 * 2 ** 20              # GB300 L2 cache
METRIC = "cache upkeep ms/step & GB/s; FP8 attn TFLOP/s (757q×5788kv); % of GB300 roofline"
WORKLOAD = dict(name="steady denoise step: 60 blocks x (1 write + 4 attention calls), reset every 42 steps",
                L=60, H=16, d=128, R=5788, T=757, passes=4, reset_every=42)
TINY = dict(name="tiny: 1 block, 2 heads x 64, 96 slots, 32-token writes, 4 attention calls per step, 100 steps, "
                 "resets every 42", L=1, H=2, d=64, R=96, T=32, passes=4, reset_every=42, steps=100)
SMALL = dict(name="small check: 4 blocks x (1 write + 4 attention calls)", L=4, H=16, d=128, R=5788, T=757,
             passes=4, reset_every=42)
# 3-D (time, height, width) video RoPE: frames of 11 x 17 latent tokens, writes of 4
# frames (748 tokens), a ring of 31 frames (5,797 slots, the nearest whole-frame
# size to 5,788); band split 22 / 21 / 21 pairs of d = 128 (time / height / width).
ROPE_3D = dict(T=748, R=5797, rope_3d=(187, 17, 22, 21))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"kvring_bench_clocks_gpu{index}_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        load = [x for x in sm if smax and x > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(load) if load else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def make_pool(cfg, torch, device):
    from kv_cache_gb300 import synthetic
    T, H, d = cfg["T"], cfg["H"], cfg["d"]
    host = {r: [synthetic.chunk(r, i, T, H, d, outliers=True) for i in range(synthetic.POOL)] for r in ("k", "v", "q")}
    dev = {r: [torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(device) for b in host[r]] for r in host}
    return host, dev


def run_gpu(args, cfg, rank, world):
    import torch
    from kv_cache_gb300 import kvring as kv
    from kv_cache_gb300 import synthetic

    device = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(device)
    kv.load()
    L, H, d, R, T, P, RE = (cfg[k] for k in ("L", "H", "d", "R", "T", "passes", "reset_every"))
    WP = cfg["writes_per_step"]           # 1, or P when every pass rewrites the newest chunk
    NV = cfg.get("naive_upkeep", False)   # the comparison scheme: refresh the whole window per call
    ring = kv.KVRing(L, H, d, R, T, max_position=R + RE * T, naive_upkeep=NV, rope_3d=cfg.get("rope_3d"))
    host, pool = make_pool(cfg, torch, device)
    stream = torch.cuda.current_stream(device)
    # one output buffer per (layer, pass), as a model keeps each block's attention output
    outs = [torch.empty((T, H, d), dtype=torch.float32, device=device) for _ in range(L * P)]

    step_counter = [0]

    def one_step(timers=None, inputs=None, out_bufs=None):
        s = step_counter[0]
        step_counter[0] += 1
        if s > 0 and s % RE == 0:
            if timers is not None:
                timers["rebase"][0].record(stream)
            ring.rebase(stream)
            if timers is not None:
                timers["rebase"][1].record(stream)
                timers["n_rebase"] += 1
        ob = out_bufs or outs
        for p in range(P):
            for l in range(L):
                if p < WP:
                    i = synthetic.pool_index(s, l, 4 if p == 0 else p, L)
                    k = inputs["k"][p * L + l] if inputs else pool["k"][i]
                    v = inputs["v"][p * L + l] if inputs else pool["v"][i]
                    if timers is not None:
                        ev = timers["write"][timers["nw"]]
                        ev[0].record(stream)
                    if p == 0:
                        ring.write(l, k, v, stream=stream)
                    else:
                        ring.rewrite(l, k, v, stream=stream)
                    if timers is not None:
                        ev[1].record(stream)
                        timers["nw"] += 1
                if NV:
                    if timers is not None:
                        ev = timers["refresh"][timers["nr"]]
                        ev[0].record(stream)
                    ring.naive_refresh(l, stream=stream)
                    if timers is not None:
                        ev[1].record(stream)
                        timers["nr"] += 1
                q = inputs["q"][p * L + l] if inputs else pool["q"][synthetic.pool_index(s, l, p, L)]
                if timers is not None:
                    ev = timers["attend"][timers["na"]]
                    ev[0].record(stream)
                ring.attend(l, q, ob[p * L + l], stream=stream)
                if timers is not None:
                    ev[1].record(stream)
                    timers["na"] += 1

    def to_reset_step():
        """Untimed steps until the next step is a reset step (so a timed run of K
        steps holds ceil(K / RE) rebases, the first in its first step)."""
        while step_counter[0] % RE != 0:
            one_step()

    # fill the rings (untimed): 8 writes reach the steady state (count = R)
    fill = -(-R // T)
    for _ in range(fill):
        one_step()
    for _ in range(args.warmup):
        one_step()
    to_reset_step()
    torch.cuda.synchronize(device)
    ring.check_device(stream)

    K = args.steps
    mk = lambda: torch.cuda.Event(enable_timing=True)
    timers = {"write": [(mk(), mk()) for _ in range(K * L * WP)], "attend": [(mk(), mk()) for _ in range(K * L * P)],
              "rebase": (mk(), mk()), "nw": 0, "na": 0, "n_rebase": 0,
              "refresh": [(mk(), mk()) for _ in range(K * L * P if NV else 0)], "nr": 0}
    launches0 = ring.launch_count()
    first_timed = step_counter[0]
    sampler = ClockSampler(device.index)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(device)
    sampler.start()
    t0, t1 = mk(), mk()
    t0.record(stream)
    for _ in range(K):
        one_step()                 # nothing but the path's own calls between t0 and t1
    t1.record(stream)
    torch.cuda.synchronize(device)
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    launches = ring.launch_count() - launches0
    resets_timed = sum(1 for st in range(first_timed, first_timed + K) if st > 0 and st % RE == 0)
    if ring.check_device(stream) != kv.KVRING_OK:
        raise RuntimeError("device wait timed out during the timed region: " + kv.kvring_last_error(ring.handle))
    ms = t0.elapsed_time(t1)
    # per-call breakdown: the same number of steps again, from a reset step, with an
    # event pair around each call (events between calls keep consecutive kernels
    # from overlapping, so these are taken apart from the step time above)
    to_reset_step()
    for _ in range(K):
        one_step(timers)
    torch.cuda.synchronize(device)
    if ring.check_device(stream) != kv.KVRING_OK:
        raise RuntimeError("device wait timed out during the breakdown pass: " + kv.kvring_last_error(ring.handle))
    w_ms = [a.elapsed_time(b) for a, b in timers["write"][:timers["nw"]]]
    a_ms = [a.elapsed_time(b) for a, b in timers["attend"][:timers["na"]]]
    r_ms = [a.elapsed_time(b) for a, b in timers["refresh"][:timers["nr"]]]
    rb_ms = timers["rebase"][0].elapsed_time(timers["rebase"][1]) if timers["n_rebase"] else None
    del timers
    # the write kernel back to back, GPU side: 3 x L rewrites of the newest chunk
    # (the same kernel and bytes as a write) captured in one CUDA graph, so no host
    # launch cost sits between them; the inputs rotate through copies of the pool
    # larger than L2, so every call reads HBM.  Beside it, the same bytes through a
    # plain elementwise kernel (K xor V into a buffer of the codes' size: 2 x T x H
    # x d x 2 bytes in, T x H x d x 2 out), captured the same way: the floor a
    # launch of this size reaches on this GPU.
    nb = -(-2 * L2_BYTES // (2 * T * H * d * 2)) + 1
    wk = [pool["k"][i % len(pool["k"])].clone() for i in range(nb)]
    wv = [pool["v"][i % len(pool["v"])].clone() for i in range(nb)]
    floor_out = torch.empty((T, H, d), dtype=torch.int16, device=device)
    wb_n = 3 * L
    side = torch.cuda.Stream(device)
    side.wait_stream(stream)
    g_write, g_floor = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_write, stream=side):
            for n in range(wb_n):
                ring.rewrite(n % L, wk[n % nb], wv[n % nb])
        with torch.cuda.graph(g_floor, stream=side):
            for n in range(wb_n):
                torch.bitwise_xor(wk[n % nb].view(torch.int16), wv[n % nb].view(torch.int16), out=floor_out)
    stream.wait_stream(side)
    graph_ms = {}
    for name, g in (("write", g_write), ("floor", g_floor)):
        g.replay()
        torch.cuda.synchronize(device)
        g0, g1 = mk(), mk()
        g0.record(stream)
        g.replay()
        g1.record(stream)
        torch.cuda.synchronize(device)
        graph_ms[name] = g0.elapsed_time(g1) / wb_n
    w_b2b_ms, w_floor_ms = graph_ms["write"], graph_ms["floor"]
    del g_write, g_floor, wk, wv, floor_out

    # ---- end to end: host inputs (pinned) -> device, all attention outputs -> host, every step.
    # Two device buffer sets: one copy stream brings step s + 1's K, V and Q in
    # while step s computes, another reads step s's 240 outputs back once it has
    # finished (the way a serving loop overlaps its transfers; the two directions
    # use separate copy engines); every step's copies are inside the timed region.  Each kind moves as one copy per step (a step's K,
    # V and Q chunks laid out contiguously in pinned memory, its outputs in one
    # device buffer), so the host issues 4 copies per step instead of one per
    # tensor and the loop does not wait on the host.
    e2e_steps = max(1, min(K, args.e2e_steps))
    nk, nq = L * WP, L * P
    chunk = (T, H, d)
    host_in = {"k": torch.empty((nk,) + chunk, dtype=torch.bfloat16, pin_memory=True),
               "v": torch.empty((nk,) + chunk, dtype=torch.bfloat16, pin_memory=True),
               "q": torch.empty((nq,) + chunk, dtype=torch.bfloat16, pin_memory=True)}
    for l in range(L):            # one step's inputs, from the pool (the same bytes every step)
        for p in range(WP):
            i = synthetic.pool_index(0, l, 4 if p == 0 else p, L)
            host_in["k"][p * L + l].copy_(torch.from_numpy(host["k"][i].view(np.int16)).view(torch.bfloat16))
            host_in["v"][p * L + l].copy_(torch.from_numpy(host["v"][i].view(np.int16)).view(torch.bfloat16))
        for p in range(P):
            i = synthetic.pool_index(0, l, p, L)
            host_in["q"][p * L + l].copy_(torch.from_numpy(host["q"][i].view(np.int16)).view(torch.bfloat16))
    host_out = torch.empty((nq,) + chunk, dtype=torch.float32, pin_memory=True)
    NB = 2
    dev_in = [{kind: torch.empty_like(host_in[kind], device=device) for kind in host_in} for _ in range(NB)]
    dev_out = [torch.empty((nq,) + chunk, dtype=torch.float32, device=device) for _ in range(NB)]
    dev_in_views = [{kind: list(dev_in[b][kind].unbind(0)) for kind in dev_in[b]} for b in range(NB)]
    dev_out_views = [list(dev_out[b].unbind(0)) for b in range(NB)]
    cs = torch.cuda.Stream(device)          # host -> device
    cs_out = torch.cuda.Stream(device)      # device -> host: the two directions run at once
    ev = lambda: torch.cuda.Event()
    in_ready, comp_done, out_read = [ev() for _ in range(NB)], [ev() for _ in range(NB)], [ev() for _ in range(NB)]
    h2d = d2h = 0
    to_reset_step()

    def issue_inputs(n):
        nonlocal h2d
        b = n % NB
        with torch.cuda.stream(cs):
            if n >= NB:
                cs.wait_event(comp_done[b])      # the step that last read slot b has finished
            for kind in ("k", "v", "q"):
                dev_in[b][kind].copy_(host_in[kind], non_blocking=True)
            in_ready[b].record(cs)
        h2d += sum(t.numel() * t.element_size() for t in host_in.values())

    torch.cuda.synchronize(device)
    e0, e1 = mk(), mk()
    e0.record(stream)
    cs.wait_event(e0)
    issue_inputs(0)
    for n in range(e2e_steps):
        b = n % NB
        if n + 1 < e2e_steps:
            issue_inputs(n + 1)
        stream.wait_event(in_ready[b])
        if n >= NB:
            stream.wait_event(out_read[b])       # step n - 2's outputs are read back
        one_step(inputs=dev_in_views[b], out_bufs=dev_out_views[b])
        comp_done[b].record(stream)
        with torch.cuda.stream(cs_out):
            cs_out.wait_event(comp_done[b])
            host_out.copy_(dev_out[b], non_blocking=True)
            out_read[b].record(cs_out)
        d2h += host_out.numel() * host_out.element_size()
    fin, fin_out = ev(), ev()
    fin.record(cs)
    fin_out.record(cs_out)
    stream.wait_event(fin)
    stream.wait_event(fin_out)
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = e0.elapsed_time(e1)
    del dev_in, dev_out, dev_in_views, dev_out_views, host_out, host_in
    # five more resets, each after one more chunk per block (untimed) so that every
    # layer has a delta to turn by, with an event pair around each: the median
    # beside the one reset inside the breakdown pass
    rb_more = []
    for i in range(5):
        s = step_counter[0] + i
        for l in range(L):
            j = synthetic.pool_index(s, l, 4, L)
            ring.write(l, pool["k"][j], pool["v"][j], stream=stream)
        b0, b1 = mk(), mk()
        b0.record(stream)
        ring.rebase(stream)
        b1.record(stream)
        torch.cuda.synchronize(device)
        rb_more.append(b0.elapsed_time(b1))
    if ring.check_device(stream) != kv.KVRING_OK:
        raise RuntimeError("device wait timed out after the extra resets: " + kv.kvring_last_error(ring.handle))
    ring.close()
    return dict(ms=ms, w_ms=w_ms, a_ms=a_ms, r_ms=r_ms, rb_ms=rb_ms, rb_more=rb_more, launches=launches,
                clocks=clocks, w_b2b_ms=w_b2b_ms, w_floor_ms=w_floor_ms, e2e_ms=e2e_ms, e2e_steps=e2e_steps,
                h2d=h2d // e2e_steps, d2h=d2h // e2e_steps, resets_timed=resets_timed)


def run_whole_configs_gpu(torch_device_index=0, reps=20):
    """GPU time of the two configurations the CPU oracle is also timed on whole:
    the tiny case (1 block, 2 heads x 64, 96 slots, 32-token writes, 4 attention
    calls per step, 100 steps with resets every 42) and one production write +
    one 757-query attention call on a full 5,788-slot ring of 16 heads x 128."""
    import torch
    from kv_cache_gb300 import kvring as kv
    from kv_cache_gb300 import synthetic
    device = torch.device("cuda", torch_device_index)
    stream = torch.cuda.current_stream(device)
    mk = lambda: torch.cuda.Event(enable_timing=True)
    dev = lambda bits: torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(device)
    out = {}
    # tiny: 100 steps, whole
    tc = TINY
    ring = kv.KVRing(1, tc["H"], tc["d"], tc["R"], tc["T"], max_position=tc["R"] + 42 * tc["T"])
    kin = [dev(synthetic.chunk("k", i, tc["T"], tc["H"], tc["d"])) for i in range(synthetic.POOL)]
    vin = [dev(synthetic.chunk("v", i, tc["T"], tc["H"], tc["d"])) for i in range(synthetic.POOL)]
    qin = [dev(synthetic.chunk("q", i, tc["T"], tc["H"], tc["d"])) for i in range(synthetic.POOL)]
    o = torch.empty((tc["T"], tc["H"], tc["d"]), dtype=torch.float32, device=device)

    def tiny_run():
        for s in range(tc["steps"]):
            if s > 0 and s % 42 == 0:
                ring.rebase(stream)
            ring.write(0, kin[s % 16], vin[s % 16], stream=stream)
            for p in range(tc["passes"]):
                ring.attend(0, qin[(s + p) % 16], o, stream=stream)

    tiny_run()        # warm-up (a fresh ring each time would re-create it; the schedule repeats)
    ring.close()
    ring = kv.KVRing(1, tc["H"], tc["d"], tc["R"], tc["T"], max_position=tc["R"] + 42 * tc["T"])
    torch.cuda.synchronize(device)
    e0, e1 = mk(), mk()
    e0.record(stream)
    tiny_run()
    e1.record(stream)
    torch.cuda.synchronize(device)
    out["tiny_100_steps_ms"] = e0.elapsed_time(e1)
    ring.close()
    # one production write + one attention call on a full ring
    c = WORKLOAD
    ring = kv.KVRing(1, c["H"], c["d"], c["R"], c["T"], max_position=c["R"] + 42 * c["T"])
    kin = [dev(synthetic.chunk("k", i, c["T"], c["H"], c["d"], True)) for i in range(4)]
    vin = [dev(synthetic.chunk("v", i, c["T"], c["H"], c["d"], True)) for i in range(4)]
    qin = dev(synthetic.chunk("q", 0, c["T"], c["H"], c["d"], True))
    o = torch.empty((c["T"], c["H"], c["d"]), dtype=torch.float32, device=device)
    for w in range(-(-c["R"] // c["T"])):
        ring.write(0, kin[w % 4], vin[w % 4], stream=stream)
    ts = []
    for r in range(reps + 3):
        e0, e1 = mk(), mk()
        e0.record(stream)
        ring.write(0, kin[r % 4], vin[r % 4], stream=stream)
        ring.attend(0, qin, o, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        if r >= 3:
            ts.append(e0.elapsed_time(e1))
    out["single_layer_write_attend_ms"] = statistics.median(ts)
    if ring.check_device(stream) != kv.KVRING_OK:
        raise RuntimeError(kv.kvring_last_error(ring.handle))
    ring.close()
    return out


SESSION = dict(name="unsharded-width session: 60 blocks of 64 heads x (1 write + 4 attention calls), 1,000 steps, "
                    "resets every 42", L=60, H=64, d=128, R=5788, T=757, passes=4, reset_every=42, steps=1000,
               checks=(1, 41, 42, 43, 500, 999), replay=10)


def run_session(args, cfg):
    """The unsharded-width session: every step is [rebase when due] + L writes + 4L
    attention calls, each step timed with its own event pair.  At the check steps
    the cache of the first and last block is compared with an oracle ring whose
    bookkeeping comes from a bookkeeping-only oracle ring (1 head, d = 2, every
    step) and which replays the last `replay` steps with data (the ring holds the
    chunks of the last 8 steps, and a reset inside the replayed steps turns only
    chunks written inside them), and the step's last attention call of those
    blocks is compared on 4 heads x 64 query rows."""
    import copy
    from collections import deque

    import torch
    from kv_cache_gb300 import kvring as kv
    from kv_cache_gb300 import synthetic
    from oracle import e4m3
    from oracle.schemes import WriteTimeRing

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    L, H, d, R, T, P, RE = (cfg[k] for k in ("L", "H", "d", "R", "T", "passes", "reset_every"))
    steps, checks, replay = cfg["steps"], [c for c in cfg["checks"] if c < cfg["steps"]], cfg["replay"]
    ring = kv.KVRing(L, H, d, R, T, max_position=R + RE * T)
    host, pool = make_pool(cfg, torch, device)
    f32 = synthetic.bf16_to_f32
    stream = torch.cuda.current_stream(device)
    outs = [torch.empty((T, H, d), dtype=torch.float32, device=device) for _ in range(L * P)]
    mk = lambda: torch.cuda.Event(enable_timing=True)

    def one_step(s, timers=None):
        if s > 0 and s % RE == 0:
            if timers:
                timers["rebase"][0].record(stream)
            ring.rebase(stream)
            if timers:
                timers["rebase"][1].record(stream)
        for p in range(P):
            for l in range(L):
                if p == 0:
                    i = synthetic.pool_index(s, l, 4, L)
                    if timers:
                        timers["write"].append((mk(), mk()))
                        timers["write"][-1][0].record(stream)
                    ring.write(l, pool["k"][i], pool["v"][i], stream=stream)
                    if timers:
                        timers["write"][-1][1].record(stream)
                if timers:
                    timers["attend"].append((mk(), mk()))
                    timers["attend"][-1][0].record(stream)
                ring.attend(l, pool["q"][synthetic.pool_index(s, l, p, L)], outs[p * L + l], stream=stream)
                if timers:
                    timers["attend"][-1][1].record(stream)

    tiny = WriteTimeRing(R, 1, 2)
    z = np.zeros((T, 1, 2), np.float32)
    before = deque(maxlen=replay)
    rng = np.random.default_rng(21)
    heads = np.array([0, 21, 42, 63])
    rows = np.unique(np.concatenate([rng.choice(T, 60, replace=False), [0, 255, 256, 756]]))
    ev = [(mk(), mk()) for _ in range(steps)]
    drift = []
    sampler = ClockSampler(0)
    sampler.start()
    for s in range(steps):
        before.append(copy.deepcopy(tiny))
        if s > 0 and s % RE == 0:
            tiny.rebase()
        tiny.write(z, z)
        ev[s][0].record(stream)
        one_step(s)
        ev[s][1].record(stream)
        if s not in checks:
            continue
        torch.cuda.synchronize(device)
        if ring.check_device(stream) != kv.KVRING_OK:
            raise RuntimeError("device wait timed out in the session: " + kv.kvring_last_error(ring.handle))
        first = s - len(before) + 1
        for l in (0, L - 1):
            o = WriteTimeRing(R, H, d)
            for f in ("head", "count", "next_pos", "writes", "resets", "last_pos", "last_n"):
                setattr(o, f, getattr(before[0], f))
            o.pos, o.chunk = before[0].pos.copy(), before[0].chunk.copy()
            for t in range(first, s + 1):
                if t > 0 and t % RE == 0:
                    o.rebase()
                i = synthetic.pool_index(t, l, 4, L)
                o.write(f32(host["k"][i]), f32(host["v"][i]))
            snap = ring.snapshot(l, stream)
            valid = o.pos >= 0
            st = ring.state(l)
            book = (st["head"], st["count"], st["next_pos"], st["writes"]) == (o.head, o.count, o.next_pos, o.writes)
            book = book and bool(np.array_equal(snap["pos"].astype(np.int64), o.pos))
            gk, gv = snap["k"][:, valid], snap["v"][:, valid]
            rk, rv = o.k8[:, valid], o.v8[:, valid]
            kstep = float(np.max(np.abs(e4m3.decode(gk) - e4m3.decode(rk)) /
                                 e4m3.ulp_at(np.maximum(np.abs(e4m3.decode(gk)), np.abs(e4m3.decode(rk))))))
            qi = synthetic.pool_index(s, l, P - 1, L)
            got = outs[(P - 1) * L + l].cpu().numpy()[np.ix_(rows, heads)].astype(np.float64)
            ref = o.attend(f32(host["q"][qi]), heads=heads, rows=rows)
            drift.append({"step": s, "block": l, "bookkeeping_exact": book,
                          "k_identical": float(np.mean(gk == rk)), "v_identical": float(np.mean(gv == rv)),
                          "k_max_steps": kstep, "attn_max_abs": float(np.max(np.abs(got - ref))),
                          "attn_mean_rel": float(np.sum(np.abs(got - ref)) / np.sum(np.abs(ref)))})
    torch.cuda.synchronize(device)
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    # per-call breakdown from a reset step, RE steps with an event pair around each call
    s = steps
    while s % RE:
        one_step(s)
        s += 1
    timers = {"write": [], "attend": [], "rebase": (mk(), mk())}
    for k in range(RE):
        one_step(s + k, timers)
    torch.cuda.synchronize(device)
    if ring.check_device(stream) != kv.KVRING_OK:
        raise RuntimeError(kv.kvring_last_error(ring.handle))
    w = [a.elapsed_time(b) for a, b in timers["write"]]
    a = [a_.elapsed_time(b) for a_, b in timers["attend"]]
    rb = timers["rebase"][0].elapsed_time(timers["rebase"][1])
    ring.close()
    return dict(step_ms=step_ms, drift=drift, clocks=clocks, w_ms=w, a_ms=a, rb_ms=rb)


def session_line(r, cfg, peaks, peak_src):
    L, H, d, R, T, P = (cfg[k] for k in ("L", "H", "d", "R", "T", "passes"))
    write_bytes, attend_flop, rebase_bytes = algorithmic(cfg)
    st = sorted(r["step_ms"])
    med = statistics.median(st)
    p99 = st[min(len(st) - 1, int(round(0.99 * (len(st) - 1))))]
    total = sum(r["step_ms"])
    w_avg, a_avg = statistics.mean(r["w_ms"]), statistics.mean(r["a_ms"])
    fp8 = 2.0 * peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    first = [x for x in r["drift"] if x["step"] == min(x["step"] for x in r["drift"])]
    last = [x for x in r["drift"] if x["step"] == max(x["step"] for x in r["drift"])]
    band = max(x["attn_max_abs"] for x in first)
    band_rel = max(x["attn_mean_rel"] for x in first)
    codes_exact = all(x["k_identical"] == 1.0 and x["v_identical"] == 1.0 and x["bookkeeping_exact"]
                      for x in r["drift"])
    return {
        "metric": "sustained ms/step over the session, and drift against the oracle", "value": total / len(st),
        "unit": "ms/step", "higher_is_better": False, "n_gpus": 1, "steps": len(st), "dtype": "fp8_e4m3",
        "data": "synthetic",
        "config": {"workload": cfg["name"], "blocks": L, "heads": H, "head_dim": d, "ring_slots": R,
                   "tokens_per_write": T, "attention_calls_per_step": L * P,
                   "l2": f"inputs larger than L2: {2 * L * H * R * d / 1e9:.2f} GB of e4m3 rings read per step"},
        "step_ms": {"mean": total / len(st), "median": med, "p99": p99, "max": st[-1], "min": st[0]},
        "breakdown": {"upkeep_ms_per_step": w_avg * L, "write_us_per_call": w_avg * 1e3,
                      "write_gbs": write_bytes / (w_avg * 1e-3) / 1e9,
                      "attend_us_per_call": a_avg * 1e3, "attend_ms_per_step": a_avg * L * P,
                      "attend_tflops_per_call": attend_flop / (a_avg * 1e-3) / 1e12,
                      "attend_frac_fp8": attend_flop / (a_avg * 1e-3) / 1e12 / fp8,
                      "rebase_ms": r["rb_ms"], "rebase_gbs": rebase_bytes / (r["rb_ms"] * 1e-3) / 1e9,
                      "rebase_frac_hbm": rebase_bytes / (r["rb_ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
                      "peaks": f"{peak_src}: HBM {peaks['hbm_gbs']} GB/s, FP8 2 x bf16 sustained"},
        "drift": r["drift"],
        "no_drift": bool(codes_exact and all(x["attn_max_abs"] <= max(2 * band, 1e-3) and
                                             x["attn_mean_rel"] <= max(2 * band_rel, 1e-4) for x in last)),
        "drift_rule": "cache bytes and bookkeeping identical to the oracle at every check; attention errors at the "
                      "last check within twice those at the first",
        "clocks": r["clocks"],
    }


def run_rebase_stress(args, cfg, rounds=10):
    """Position-reset stress: the rings filled, then `rounds` resets, each after one
    more chunk per block (so every layer has a delta); only the rebases are timed."""
    import torch
    from kv_cache_gb300 import kvring as kv
    from kv_cache_gb300 import synthetic
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    L, H, d, R, T = (cfg[k] for k in ("L", "H", "d", "R", "T"))
    ring = kv.KVRing(L, H, d, R, T, max_position=R + 42 * T, rope_3d=cfg.get("rope_3d"))
    _, pool = make_pool(cfg, torch, device)
    stream = torch.cuda.current_stream(device)
    for w in range(41):                      # 41 steps of writes: full rings, positions far from 0
        for l in range(L):
            i = synthetic.pool_index(w, l, 4, L)
            ring.write(l, pool["k"][i], pool["v"][i], stream=stream)
    ts = []
    for r in range(rounds + 1):
        if r > 0:
            for l in range(L):
                i = synthetic.pool_index(41 + r, l, 4, L)
                ring.write(l, pool["k"][i], pool["v"][i], stream=stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ring.rebase(stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        if r > 0:                            # the first reset (delta 41 chunks) is a warm-up
            ts.append(e0.elapsed_time(e1))
    if ring.check_device(stream) != kv.KVRING_OK:
        raise RuntimeError(kv.kvring_last_error(ring.handle))
    ring.close()
    return ts


def cpu_model():
    """The host CPU's model name (lscpu), for the CPU baseline's record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_sample(cfg, n=1, warm=0):
    """Time the CPU oracle on one block: a full window of writes (untimed), then
    `warm` untimed and `n` timed block steps, each one write + 4 attention calls
    (naive per-call upkeep, float64 attention).  Returns the per-block-step
    times and the full-step figure extrapolated to all blocks."""
    from kv_cache_gb300 import synthetic
    from oracle.schemes import NaiveWindow

    L, H, d, R, T, P = (cfg[k] for k in ("L", "H", "d", "R", "T", "passes"))
    naive = NaiveWindow(R, H, d, layout=cfg.get("rope_3d"))
    f32 = synthetic.bf16_to_f32
    fill = -(-R // T)
    for w in range(fill):
        naive.write(f32(synthetic.chunk("k", w, T, H, d, True)), f32(synthetic.chunk("v", w, T, H, d, True)))
    qs = [f32(synthetic.chunk("q", p, T, H, d, True)) for p in range(P)]
    WP = cfg.get("writes_per_step", 1)
    times = []
    for i in range(warm + n):
        k = f32(synthetic.chunk("k", fill + i, T, H, d, True))
        v = f32(synthetic.chunk("v", fill + i, T, H, d, True))
        t0 = time.perf_counter()
        naive.write(k, v)
        for p in range(P):
            if 0 < p < WP:
                naive.rewrite(k, v)
            naive.attend(qs[p])
        if i >= warm:
            times.append(time.perf_counter() - t0)
    block_s = statistics.median(times)
    threads = os.cpu_count()
    return dict(block_s=block_s, block_times_s=times, step_s=block_s * L, cores=threads, cpu_model=cpu_model(),
                sample=f"{n} block step(s) (1 write + {WP - 1} rewrites + {P} attention calls each, naive per-call "
                       f"upkeep, float64 attention{', 3-D RoPE' if cfg.get('rope_3d') else ''}) at {H} heads x {d}, "
                       f"R={R}, T={T}; full step = median block step x {L} blocks (extrapolated)")


def oracle_whole_configs():
    """The CPU oracle timed whole on the two small configurations: the tiny case
    (100 steps: write, 4 naive attention calls, resets every 42) and one
    production write + one attention call on a full 16-head ring."""
    from kv_cache_gb300 import synthetic
    from oracle.schemes import NaiveWindow

    f32 = synthetic.bf16_to_f32
    tc = TINY
    naive = NaiveWindow(tc["R"], tc["H"], tc["d"])
    kin = [f32(synthetic.chunk("k", i, tc["T"], tc["H"], tc["d"])) for i in range(synthetic.POOL)]
    vin = [f32(synthetic.chunk("v", i, tc["T"], tc["H"], tc["d"])) for i in range(synthetic.POOL)]
    qin = [f32(synthetic.chunk("q", i, tc["T"], tc["H"], tc["d"])) for i in range(synthetic.POOL)]
    t0 = time.perf_counter()
    for s in range(tc["steps"]):
        if s > 0 and s % tc["reset_every"] == 0:
            naive.rebase()
        naive.write(kin[s % 16], vin[s % 16])
        for p in range(tc["passes"]):
            naive.attend(qin[(s + p) % 16])
    tiny_s = time.perf_counter() - t0
    c = WORKLOAD
    naive = NaiveWindow(c["R"], c["H"], c["d"])
    for w in range(-(-c["R"] // c["T"])):
        naive.write(f32(synthetic.chunk("k", w % 4, c["T"], c["H"], c["d"], True)),
                    f32(synthetic.chunk("v", w % 4, c["T"], c["H"], c["d"], True)))
    k = f32(synthetic.chunk("k", 1, c["T"], c["H"], c["d"], True))
    v = f32(synthetic.chunk("v", 1, c["T"], c["H"], c["d"], True))
    q = f32(synthetic.chunk("q", 0, c["T"], c["H"], c["d"], True))
    t0 = time.perf_counter()
    naive.write(k, v)
    naive.attend(q)
    single_s = time.perf_counter() - t0
    return {"tiny_100_steps_ms": tiny_s * 1e3, "single_layer_write_attend_ms": single_s * 1e3,
            "tiny_workload": tc["name"],
            "single_layer_workload": "one write of 757 tokens + one 757-query attention call, full 5,788-slot "
                                     "ring of 16 heads x 128 (naive per-call upkeep, float64 attention)"}


def oracle_upkeep_sample(cfg):
    """The CPU analogue of the pages' upkeep comparison, timed with the oracle on
    one block: the naive scheme's per-step upkeep (a write that shifts the window,
    then the whole window re-rotated and re-quantised before each of the P calls)
    against the write-time ring's (RoPE and FP8 of the new chunk once, plus one
    delta rotation of the ring every reset_every steps), both x L blocks."""
    from kv_cache_gb300 import synthetic
    from oracle.schemes import NaiveWindow, WriteTimeRing

    L, H, d, R, T, P, RE = (cfg[k] for k in ("L", "H", "d", "R", "T", "passes", "reset_every"))
    lay = cfg.get("rope_3d")
    naive = NaiveWindow(R, H, d, layout=lay)
    ring = WriteTimeRing(R, H, d, layout=lay)
    f32 = synthetic.bf16_to_f32
    fill = -(-R // T)
    for w in range(fill):
        k, v = f32(synthetic.chunk("k", w, T, H, d, True)), f32(synthetic.chunk("v", w, T, H, d, True))
        naive.write(k, v)
        ring.write(k, v)
    k, v = f32(synthetic.chunk("k", fill, T, H, d, True)), f32(synthetic.chunk("v", fill, T, H, d, True))
    t0 = time.perf_counter()
    naive.write(k, v)
    for _ in range(P):
        naive.cache_codes()
    t_naive = time.perf_counter() - t0
    t0 = time.perf_counter()
    ring.write(k, v)
    t_write = time.perf_counter() - t0
    t0 = time.perf_counter()
    ring.rebase()
    t_rebase = time.perf_counter() - t0
    naive_ms = t_naive * L * 1e3
    ring_ms = (t_write + t_rebase / RE) * L * 1e3
    return {"naive_ms_per_step": naive_ms, "write_time_ms_per_step": ring_ms, "ratio": naive_ms / ring_ms,
            "sample": f"one block: naive = 1 shifting write + {P} whole-window refreshes; write-time = 1 write "
                      f"+ 1/{RE} of a full-ring rebase; x{L} blocks (extrapolated)"}


# DRAM bytes (read + write) per attend_kernel launch, from the ncu capture summarised
# in profiles/attend_kernel_production_ring_8_blocks.md; valid only for the attention
# source it was taken on (sha256 prefix), else reported as null.
ATTEND_TRAFFIC = {"bytes": 26.77e6, "source_sha256": "7f6d94254698a4c2",
                  "shape": {"H": 16, "d": 128, "R": 5788, "T": 757}}


def attend_traffic(cfg):
    import hashlib
    if any(cfg[k] != v for k, v in ATTEND_TRAFFIC["shape"].items()):
        return None
    path = os.path.join(ROOT, "kv_cache_gb300", "csrc", "k_attend.cu")
    try:
        digest = hashlib.sha256(open(path, "rb").read()).hexdigest()
    except OSError:
        return None
    return ATTEND_TRAFFIC["bytes"] if digest.startswith(ATTEND_TRAFFIC["source_sha256"]) else None


def max_over_ranks(values, world):
    """Each value's maximum over the ranks (the slowest replica sets the job's time).
    NCCL reduces on the GPU, gloo on the host; one rank returns its own values."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    device = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def probe_peaks(n=8192, iters=20):
    """Library GEMM throughput on this GPU, FP8 e4m3 (per-tensor scales) and bf16 (a yardstick only)."""
    import torch
    dev = torch.device("cuda", 0)
    a16 = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    b16 = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    a8 = a16.to(torch.float8_e4m3fn)
    b8 = b16.to(torch.float8_e4m3fn).t().contiguous().t()     # column-major second operand
    one = torch.ones((), device=dev, dtype=torch.float32)
    runs = {"fp8": lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one, out_dtype=torch.bfloat16),
            "bf16": lambda: a16 @ b16}
    out = {"probe": "gemm", "n": n}
    for name, fn in runs.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        out[f"{name}_tflops"] = 2.0 * n ** 3 * iters / (e0.elapsed_time(e1) * 1e-3) / 1e12
    out["fp8_over_bf16"] = out["fp8_tflops"] / out["bf16_tflops"]
    return out


def rebase_row_bytes(cfg):
    """Bytes of one cached K row that a reset reads (and writes back): the whole row
    in 1-D; with 3-D RoPE only the 16-byte pieces that hold time-band pairs."""
    if not cfg.get("rope_3d"):
        return cfg["d"]
    pt = cfg["rope_3d"][2]
    return -(-pt // 8) * 16


def algorithmic(cfg):
    L, H, d, R, T, P = (cfg[k] for k in ("L", "H", "d", "R", "T", "passes"))
    write_bytes = T * H * d * 2 * 2 + T * H * d * 2           # bf16 K,V in + e4m3 K,V out
    attend_flop = 4.0 * T * R * d * H
    rebase_bytes = 2.0 * L * H * R * rebase_row_bytes(cfg)   # e4m3 K read + write, full rings
    return write_bytes, attend_flop, rebase_bytes


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=42)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvring", choices=["kvring", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=12)
    ap.add_argument("--small", action="store_true", help="4 blocks instead of 60 (quick checks)")
    ap.add_argument("--heads", type=int, default=0,
                    help="number of heads (64 = the unsharded model width; default 16, one tensor-parallel shard)")
    ap.add_argument("--rebase-stress", action="store_true",
                    help="the reset stress workload: full rings, then 10 timed resets (one JSON line)")
    ap.add_argument("--probe-peaks", action="store_true",
                    help="time an 8192^3 FP8 (torch._scaled_mm) and bf16 GEMM on this GPU and print their ratio, "
                         "the check of the FP8 = 2 x bf16 roofline denominator")
    ap.add_argument("--blocks", type=int, default=0,
                    help="number of blocks (profiling cases; 8 blocks already keep one layer's ring out of L2 "
                         "between its visits)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--session", action="store_true",
                    help="the unsharded-width session: 60 blocks x 64 heads, 1,000 steps, resets every 42; "
                         "per-step times and drift against the oracle (one JSON line)")
    ap.add_argument("--session-steps", type=int, default=0, help="steps of --session (default 1,000)")
    ap.add_argument("--naive-upkeep", action="store_true",
                    help="the comparison scheme: shift the bf16 window on write, re-rotate and re-quantise "
                         "all of it before every attention call (kvring_naive_refresh)")
    ap.add_argument("--rewrite-per-pass", action="store_true",
                    help="passes 1..3 rewrite the newest chunk with new K/V (kvring_write_ex, no advance)")
    ap.add_argument("--rope-3d", action="store_true",
                    help="3-D (time, height, width) video RoPE: frames of 11 x 17 tokens, 4-frame writes "
                         "(748 tokens), a 31-frame ring (5,797 slots)")
    args = ap.parse_args()
    cfg = dict(SMALL if args.small else WORKLOAD)
    if args.rope_3d:
        cfg.update(ROPE_3D)
        cfg["name"] = cfg["name"] + ", 3-D video RoPE (frames of 11 x 17 tokens, 4-frame writes of 748, 31-frame ring of 5,797)"
    if args.heads > 0:
        cfg["name"] = cfg["name"].replace("60 blocks", f"60 blocks of {args.heads} heads")
        cfg["H"] = args.heads
    if args.blocks > 0:
        cfg["name"] = cfg["name"].replace(f"{cfg['L']} blocks", f"{args.blocks} blocks")
        cfg["L"] = args.blocks
    if args.probe_peaks:
        print(json.dumps(probe_peaks()))
        return
    if args.session:
        scfg = dict(SESSION)
        if args.session_steps > 0:
            scfg["steps"] = args.session_steps
            scfg["name"] = scfg["name"].replace("1,000 steps", f"{args.session_steps} steps")
        if args.blocks > 0:
            scfg["name"] = scfg["name"].replace("60 blocks", f"{args.blocks} blocks")
            scfg["L"] = args.blocks
        peaks, peak_src = load_peaks()
        print(json.dumps(session_line(run_session(args, scfg), scfg, peaks, peak_src)))
        return
    if args.rebase_stress:
        ts = run_rebase_stress(args, cfg)
        peaks, peak_src = load_peaks()
        med = statistics.median(ts)
        nbytes = 2.0 * cfg["L"] * cfg["H"] * cfg["R"] * rebase_row_bytes(cfg)
        print(json.dumps({
            "metric": "rebase ms (position reset of every cached K)", "value": med, "unit": "ms",
            "higher_is_better": False, "n_gpus": 1, "steps": len(ts), "dtype": "fp8_e4m3", "data": "synthetic",
            "config": {"workload": f"reset stress: {cfg['L']} blocks x {cfg['H']} heads x {cfg['d']}, "
                                   f"R={cfg['R']}, filled over 41 steps, then {len(ts)} resets"
                                   + (f", 3-D RoPE (frames of {cfg['rope_3d'][0]}; only the time band turns)"
                                      if cfg.get("rope_3d") else ""),
                       "l2": f"{nbytes / 1e9:.2f} GB of K codes read and written per reset (larger than L2)"},
            "samples_ms": ts, "min_ms": min(ts),
            "roofline": {"bound": "hbm", "achieved": nbytes / (med * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": nbytes / (med * 1e-3) / 1e9 / peaks["hbm_gbs"],
                         "peak_source": peak_src}}))
        return
    cfg["writes_per_step"] = cfg["passes"] if args.rewrite_per_pass else 1
    cfg["naive_upkeep"] = bool(args.naive_upkeep)
    if args.rewrite_per_pass:
        cfg["name"] = cfg["name"].replace("(1 write + 4 attention calls)", "(1 write + 3 rewrites + 4 attention calls)")
    if args.naive_upkeep:
        cfg["name"] = cfg["name"].replace("attention calls)", "attention calls, each after a naive whole-window "
                                          "re-rotation + re-quantisation; window shifted by copy on write)")
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    L, H, d, R, T, P = (cfg[k] for k in ("L", "H", "d", "R", "T", "passes"))
    write_bytes, attend_flop, rebase_bytes = algorithmic(cfg)
    config = {"workload": cfg["name"], "blocks": L, "heads": H, "head_dim": d, "ring_slots": R,
              "tokens_per_write": T, "attention_calls_per_step": L * P, "reset_every_steps": cfg["reset_every"],
              "l2": (f"inputs larger than L2: {2 * L * H * R * d / 1e9:.2f} GB of e4m3 rings read per step"
                     if 2 * L * H * R * d > 129e6 else
                     f"check run, not a bench number: {2 * L * H * R * d / 1e9:.2f} GB of rings fit in L2"),
              "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
              "timed_steps": "start at a reset step, so K timed steps hold ceil(K / 42) rebases"}

    if args.impl == "reference":
        if rank != 0:
            return
        # each timed "step" is one block's step; the full step is extrapolated x L
        n = max(1, args.steps)
        cb = oracle_sample(cfg, n=n, warm=min(args.warmup, 1))
        step_s = cb["step_s"]
        line = {"impl": "reference", "metric": METRIC, "value": 1.0 / step_s, "unit": "steps/s", "n_gpus": 0,
                "steps": n / L, "block_steps_timed": n, "warmup": min(args.warmup, 1),
                "ms_per_step": step_s * 1e3, "extrapolated": True, "extrapolation_factor": L,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": 1.0 / step_s, "unit": "steps/s", "cores": cb["cores"],
                                 "cpu_model": cb["cpu_model"], "kind": "oracle", "sample": cb["sample"],
                                 "block_step_ms": [t * 1e3 for t in cb["block_times_s"]],
                                 "upkeep": oracle_upkeep_sample(cfg), "whole": oracle_whole_configs()},
                "e2e": {"value": 1.0 / step_s, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    r = run_gpu(args, cfg, rank, world)
    ms = r["ms"]
    e2e_ms = r["e2e_ms"]
    ms, e2e_per = max_over_ranks([ms, e2e_ms / r["e2e_steps"]], world)
    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    fp8_sustained = 2.0 * peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    K = args.steps
    ms_step = ms / K
    w_avg = statistics.mean(r["w_ms"]) if r["w_ms"] else float("nan")
    a_avg = statistics.mean(r["a_ms"]) if r["a_ms"] else float("nan")
    rb_samples = ([r["rb_ms"]] if r["rb_ms"] else []) + list(r.get("rb_more") or [])
    rb_med = statistics.median(rb_samples) if rb_samples else None
    attn_tflops = attend_flop / (a_avg * 1e-3) / 1e12
    write_gbs = write_bytes / (w_avg * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": world * K / (ms * 1e-3), "unit": "steps/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3", "data": "synthetic", "config": config,
        "e2e": {"value": world * 1e3 / e2e_per, "unit": "steps/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"], "steps": r["e2e_steps"]},
        "gpu_launches": r["launches"],
        "resets_in_timed_steps": r["resets_timed"],
        "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": fp8_sustained, "unit": "TFLOP/s",
                     "frac": attn_tflops / fp8_sustained, "traffic": attend_traffic(cfg),
                     "traffic_unit": "bytes per attend_kernel launch (ncu, 8-block run)",
                     "kernel": "attention call (q-prep + attention + split combine)",
                     "peak_source": f"{peak_src}: 2 x bf16_tflops_sustained (FP8 = 2 x bf16 nominal ratio)"},
        "breakdown": {
            "upkeep_ms_per_step": w_avg * L * cfg["writes_per_step"] + (sum(r["r_ms"]) / K if r["r_ms"] else 0.0),
            "upkeep_gbs": write_gbs,
            "naive_refresh_us_per_call": (statistics.mean(r["r_ms"]) * 1e3) if r["r_ms"] else None,
            "writes_per_block_per_step": cfg["writes_per_step"],
            "upkeep_frac_hbm": write_gbs / peaks["hbm_gbs"],
            "write_us_per_call": w_avg * 1e3,
            "write_us_per_call_graph": r["w_b2b_ms"] * 1e3,
            "write_frac_hbm_graph": write_bytes / (r["w_b2b_ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "write_floor_us_per_call_graph": r["w_floor_ms"] * 1e3,
            "write_floor_frac_hbm_graph": write_bytes / (r["w_floor_ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "write_graph_note": "3 x blocks back-to-back calls in one CUDA graph; floor = the same bytes through "
                                "torch.bitwise_xor (one elementwise kernel per call)",
            "attend_us_per_call": a_avg * 1e3, "attend_tflops_per_call": attn_tflops,
            "attend_ms_per_step": a_avg * L * P,
            "attention_tflops_step": attend_flop * L * P / (a_avg * L * P * 1e-3) / 1e12,
            "rebase_ms": rb_med,
            "rebase_gbs": (rebase_bytes / (rb_med * 1e-3) / 1e9) if rb_med else None,
            "rebase_frac_hbm": (rebase_bytes / (rb_med * 1e-3) / 1e9 / peaks["hbm_gbs"]) if rb_med else None,
            "rebase_ms_note": "median of the breakdown pass's reset and five more, each after one more chunk "
                              "per block; samples in rebase_ms_samples",
            "rebase_ms_samples": rb_samples,
            "hbm_peak_gbs": peaks["hbm_gbs"], "peaks": peak_src,
        },
        "clocks": r["clocks"],
    }
    if not args.no_cpu_baseline:
        cb = oracle_sample(cfg)
        whole_cpu = oracle_whole_configs()
        whole_gpu = run_whole_configs_gpu()
        line["cpu_baseline"] = {"value": 1.0 / cb["step_s"], "unit": "steps/s", "cores": cb["cores"],
                                "cpu_model": cb["cpu_model"], "kind": "oracle", "sample": cb["sample"],
                                "upkeep": oracle_upkeep_sample(cfg),
                                "whole": {k: {"cpu_ms": whole_cpu[k], "gpu_ms": whole_gpu[k],
                                              "workload": whole_cpu["tiny_workload" if k.startswith("tiny")
                                                                    else "single_layer_workload"]}
                                          for k in ("tiny_100_steps_ms", "single_layer_write_attend_ms")}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
