"""Benchmark of the ring-order attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  prefill (B=1, Hq=32, Hkv=8, S=131072, d=128, bf16, causal, N=16 virtual ranks):
    zigzag partition -> gather Q/K/V into the ranks' head-tail layout ->
    ring-order attention -> restore O and LSE to token order;
  decode (64 requests, context U[4096, 131072], Hq=32, Hkv=8, d=128, bf16,
    block 128, interleave 16, pcp=2, dcp=4): slot mapping + cache write of the
    new token of every request -> split-KV partials -> LSE merge.

Prints one JSON line.  ``value`` is causal-adjusted attention TFLOP/s over the
whole timed step (prefill + decode); the decode+merge GB/s and the per-kernel
rooflines are reported beside it.  ``--impl reference`` times the float64
oracle instead (a bounded sample per step on the host cores).

On one GPU the step runs the single-device kernels.  Under torchrun with N > 1
ranks (or with --cp-dist) the same step is split across the ranks: the prefill
as a ring of N ranks, each holding its head-tail chunk pair and passing K/V
blocks to the next over NCCL, and the decode with the cache's devices spread
over the ranks and merged by cp_lse_ag_out_rs (strong scaling: the work is the
same at every N).
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from context_long_sequence_ring_gb300 import inputs as I  # noqa: E402

METRIC = "ring-attn fwd TFLOP/s (causal-adj) & % bf16 peak; decode+merge GB/s % HBM"
PREFILL = dict(B=1, Hq=32, Hkv=8, S=131072, d=128, N=16, seed=5)
DECODE = dict(R=64, lo=4096, hi=131072, Hq=32, Hkv=8, d=128, bs=128, I=16, pcp=2, dcp=4, seed=4, split=16)
# sources whose contents the recorded DRAM traffic of each kernel was measured on
KERNEL_SOURCES = {"ring_attn_bf16": ["ra_attn_bf16.cu", "ra_attn_pair.cuh", "ra_ring_sched.cuh", "ra_attn_tc.cuh",
                                     "ra_sm100.cuh"],
                  "cp_decode": ["ra_decode.cu"]}


def causal_flops(B, Hq, S, d):
    """Algorithmic FLOPs of causal attention forward: QK^T and PV, 2 per MAC."""
    return 4.0 * B * Hq * d * S * (S + 1) / 2


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        sus_mhz = (m.get("clocks_under_load") or {}).get("sm_mhz_median")
        return dict(hbm=m["hbm_gbs"], bf16=m["bf16_tflops"], bf16_sus=m["bf16_tflops_sustained"], src="measured",
                    sus_mhz=sus_mhz)
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback", sus_mhz=None)


def _source_hash(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "context_long_sequence_ring_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


TRAFFIC_JSON = os.path.join(ROOT, "profiles", "traffic.json")


def _traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it is for this source."""
    try:
        with open(TRAFFIC_JSON) as f:
            t = json.load(f)[kernel]
        if t.get("source_sha256_16") != _source_hash(KERNEL_SOURCES[kernel]):
            return None
        return t["dram_bytes_per_launch"]
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = [r.split(",") for r in (self.out or "").strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip().lower() == "active"})
        pw = [float(r[3]) for r in rows if r[3].strip().replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------- our arm

class Workload:
    def __init__(self, ra, dev, parts=("prefill", "decode")):
        self.ra, self.dev = ra, dev
        self.parts = parts
        P, D = PREFILL, DECODE
        tab = I.normal_table(torch.bfloat16)
        self.launches_per_step = 0
        if "prefill" in parts:
            self._init_prefill(tab)
            self.launches_per_step += 7
        if "decode" in parts:
            self._init_decode(tab)
            self.launches_per_step += 4
        torch.cuda.synchronize()

    def _init_prefill(self, tab):
        ra, dev, P = self.ra, self.dev, PREFILL
        n = P["B"] * P["S"]
        self.q = ra.synth_fill(I.tensor_key(P["seed"], I.TID_Q), tab, (n, P["Hq"], P["d"]), dev)
        self.k = ra.synth_fill(I.tensor_key(P["seed"], I.TID_K), tab, (n, P["Hkv"], P["d"]), dev)
        self.v = ra.synth_fill(I.tensor_key(P["seed"], I.TID_V), tab, (n, P["Hkv"], P["d"]), dev)
        self.seq_lens = [P["S"]] * P["B"]
        self.perm = torch.empty(n, dtype=torch.int32, device=dev)
        self.restore = torch.empty(n, dtype=torch.int32, device=dev)
        self.qz, self.kz, self.vz = (torch.empty_like(x) for x in (self.q, self.k, self.v))
        self.oz = torch.empty_like(self.q)
        self.lz = torch.empty((n, P["Hq"]), dtype=torch.float32, device=dev)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty_like(self.lz)

    def _init_decode(self, tab):
        # cache filled once (slot mapping + scatter of every context token)
        ra, dev, D = self.ra, self.dev, DECODE
        wl = I.decode_workload(D["seed"], D["R"], D["lo"], D["hi"], D["bs"], D["pcp"], D["dcp"])
        self.wl = wl
        W = D["pcp"] * D["dcp"]
        T = wl["total_tokens"]
        kt = ra.synth_fill(I.tensor_key(D["seed"], I.TID_K), tab, (T, D["Hkv"], D["d"]), dev)
        vt = ra.synth_fill(I.tensor_key(D["seed"], I.TID_V), tab, (T, D["Hkv"], D["d"]), dev)
        ctx = wl["ctx_lens"]
        qsl = torch.zeros(D["R"] + 1, dtype=torch.int32)
        qsl[1:] = torch.cumsum(ctx, 0)
        pos = torch.cat([torch.arange(int(L), dtype=torch.int32) for L in ctx])
        self.bt = wl["block_table"].to(dev)
        self.ctx = ctx.to(dev)
        slot = ra.cp_slot_mapping(qsl.to(dev), pos.to(dev), self.bt, D["bs"], D["I"], D["pcp"], D["dcp"])
        self.kc = torch.empty((W, wl["num_blocks"], D["Hkv"], D["bs"], D["d"]), dtype=torch.bfloat16, device=dev)
        self.vc = torch.empty_like(self.kc)
        ra.cp_kv_scatter(kt, vt, slot, self.kc, self.vc)
        # the step's new tokens: the last token of every request (position L-1)
        last = (qsl[1:] - 1).long()
        self.new_k = kt[last.to(dev)].contiguous()
        self.new_v = vt[last.to(dev)].contiguous()
        del kt, vt, slot
        self.new_pos = (ctx - 1).to(torch.int32).to(dev)
        self.new_qsl = torch.arange(D["R"] + 1, dtype=torch.int32, device=dev)
        self.new_slot = torch.empty((W, D["R"]), dtype=torch.int32, device=dev)
        self.qd = I.synth_normal(D["seed"], I.TID_Q, (D["R"], D["Hq"], D["d"]), torch.bfloat16).to(dev)
        self.od = torch.empty((D["R"], D["Hq"], D["d"]), dtype=torch.bfloat16, device=dev)
        self.ld = torch.empty((D["R"], D["Hq"]), dtype=torch.float32, device=dev)
        ws = ra.cp_decode_workspace_size(D["R"], D["Hq"], D["d"], wl["max_vblocks"], D["pcp"], D["dcp"], D["split"])
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)

    def decode_bytes(self):
        D = self.ctx.cpu().numpy().astype(np.int64)
        P = DECODE
        W = P["pcp"] * P["dcp"]
        vbs = P["bs"] * W
        kv = int(D.sum()) * P["Hkv"] * P["d"] * 2 * 2
        nvb = -(-D // vbs)
        live = int(np.sum(W * (-(-nvb // P["split"]))))            # partials written and read once
        part = live * P["Hq"] * (P["d"] + 1) * 4 * 2
        q_o = 2 * P["R"] * P["Hq"] * P["d"] * 2
        return kv + part + q_o, kv

    def step(self, events=None):
        ra, P, D = self.ra, PREFILL, DECODE
        e = events
        if e: e[0].record()
        if "prefill" not in self.parts:
            for i in (1, 2, 3):
                if e: e[i].record()
        else:
            self._prefill(e)
        if "decode" not in self.parts:
            for i in (4, 5):
                if e: e[i].record()
        else:
            self._decode(e)

    def _prefill(self, e):
        ra, P = self.ra, PREFILL
        # a1: head-tail partition of the batch (device kernel), a2: gather to rank-major layout
        ra.lib().ra_zigzag_partition((ra._c.c_int64 * P["B"])(*([P["S"]] * P["B"])), P["B"], P["N"], self.perm.data_ptr(),
                                     self.restore.data_ptr(), None, None, ra._stream())
        ra.gather_rows(self.q, self.perm, self.qz)
        ra.gather_rows(self.k, self.perm, self.kz)
        ra.gather_rows(self.v, self.perm, self.vz)
        if e: e[1].record()
        # a3-a5: ring-order attention over the N virtual ranks
        ra.ring_attn_fwd(self.qz, self.kz, self.vz, True, P["N"], B=P["B"], layout="zigzag", o=self.oz, lse=self.lz,
                         variant=RING_VARIANT[0])
        if e: e[2].record()
        # a2: restore token order
        ra.gather_rows(self.oz, self.restore, self.o)
        ra.gather_rows(self.lz, self.restore, self.lse)
        if e: e[3].record()

    def _decode(self, e):
        ra, D = self.ra, DECODE
        # a6: slot mapping + cache write of the new tokens; a7: split-KV decode; a8: LSE merge
        ra.cp_slot_mapping(self.new_qsl, self.new_pos, self.bt, D["bs"], D["I"], D["pcp"], D["dcp"], out=self.new_slot)
        ra.cp_kv_scatter(self.new_k, self.new_v, self.new_slot, self.kc, self.vc)
        if e: e[4].record()
        ra.cp_decode(self.qd, self.kc, self.vc, self.bt, self.ctx, D["I"], D["pcp"], D["dcp"], split_blocks=D["split"],
                     workspace=self.ws, o=self.od, lse=self.ld)
        if e: e[5].record()


def e2e_pipelined(wl, host_in, host_out, steps):
    """Milliseconds for `steps` end-to-end steps with the host copies overlapped: H2D on one
    stream, D2H on another, the step on the current stream, two sets of per-step input and
    output buffers.  Every step's inputs are copied in and its results copied out inside
    the timed region."""
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    sets = [{n: getattr(wl, n) for n in list(host_in) + list(host_out)}]
    sets.append({n: torch.empty_like(t) for n, t in sets[0].items()})
    in_ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    s_in.wait_stream(comp)
    s_out.wait_stream(comp)
    for i in range(steps):
        b = i % 2
        bufs = sets[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(in_free[b])          # step i-2 has read this set's inputs
            for n, h in host_in.items():
                bufs[n].copy_(h, non_blocking=True)
            in_ready[b].record(s_in)
        comp.wait_event(in_ready[b])
        if i >= 2:
            comp.wait_event(out_free[b])             # step i-2's results have left this set
        for n, t in bufs.items():
            setattr(wl, n, t)
        wl.step()
        in_free[b].record(comp)
        out_ready[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(out_ready[b])
            for n, h in host_out.items():
                h.copy_(bufs[n], non_blocking=True)
            out_free[b].record(s_out)
    comp.wait_stream(s_in)
    comp.wait_stream(s_out)
    e1.record(comp)
    torch.cuda.synchronize()
    last = sets[(steps - 1) % 2]
    for n, h in host_out.items():   # the results that left the GPU are the last step's
        if not torch.equal(h[:64], last[n][:64].cpu()):
            raise RuntimeError("pipelined end-to-end step: host copy of %s differs from the device" % n)
    for n, t in sets[0].items():
        setattr(wl, n, t)
    return e0.elapsed_time(e1)


# ---------------------------------------------------------------------------- the step split across ranks

class DistWorkload:
    """The same step split across the ranks of the job (context parallelism across devices).

    Prefill: the S-token sequence is cut into 2*world chunks by the head-tail partition and rank r
    holds chunks r and 2*world-1-r of Q, K and V.  The ranks form a ring: at each of the world steps
    a rank runs one ring-step kernel on the K/V block it holds while NCCL point-to-point copies pass
    that block to the next rank (double buffering).  Decode: the cache's W = pcp*dcp devices are
    spread over the ranks (W/world each, device w on rank w // (W/world)); a rank computes the
    split-KV partials of its devices, merges them, and the ranks combine their results with
    cp_lse_ag_out_rs (all-gather of the LSEs, rescale kernel, reduce-scatter of the output over
    heads), so rank r ends with heads [r*Hq/world, (r+1)*Hq/world) of the decode output."""

    def __init__(self, ra, dev, rank, world):
        from context_long_sequence_ring_gb300 import cp_dist
        self.ra, self.dev, self.rank, self.world, self.cp = ra, dev, rank, world, cp_dist
        P, D = PREFILL, DECODE
        W = D["pcp"] * D["dcp"]
        if P["B"] != 1 or P["S"] % (2 * world) != 0:
            raise ValueError("the split prefill needs B=1 and S a multiple of 2*world")
        if W % world != 0 or D["Hq"] % world != 0:
            raise ValueError("pcp*dcp (%d) and Hq (%d) must be multiples of the number of ranks (%d)"
                             % (W, D["Hq"], world))
        tab = I.normal_table(torch.bfloat16)
        S, c = P["S"], P["S"] // (2 * world)
        perm, _ = ra.zigzag_partition([S], world)
        loc = perm[rank * 2 * c:(rank + 1) * 2 * c].contiguous()
        for name, tid, H in (("q", I.TID_Q, P["Hq"]), ("k", I.TID_K, P["Hkv"]), ("v", I.TID_V, P["Hkv"])):
            full = ra.synth_fill(I.tensor_key(P["seed"], tid), tab, (S, H, P["d"]), dev)
            setattr(self, name, ra.gather_rows(full, loc))
            del full
        self.exchange = cp_dist.P2PExchange() if world > 1 else None
        self.ring_step = ra.ring_step_fn(world, rank, True)
        # decode: the shards of this rank's devices
        wl = I.decode_workload(D["seed"], D["R"], D["lo"], D["hi"], D["bs"], D["pcp"], D["dcp"])
        T = wl["total_tokens"]
        kt = ra.synth_fill(I.tensor_key(D["seed"], I.TID_K), tab, (T, D["Hkv"], D["d"]), dev)
        vt = ra.synth_fill(I.tensor_key(D["seed"], I.TID_V), tab, (T, D["Hkv"], D["d"]), dev)
        ctx = wl["ctx_lens"]
        qsl = torch.zeros(D["R"] + 1, dtype=torch.int32)
        qsl[1:] = torch.cumsum(ctx, 0)
        pos = torch.cat([torch.arange(int(L), dtype=torch.int32) for L in ctx])
        self.bt = wl["block_table"].to(dev)
        self.ctx = ctx.to(dev)
        self.n_dev = W // world
        self.dev0 = rank * self.n_dev
        slot = ra.cp_slot_mapping(qsl.to(dev), pos.to(dev), self.bt, D["bs"], D["I"], D["pcp"], D["dcp"])
        self.kc = torch.empty((self.n_dev, wl["num_blocks"], D["Hkv"], D["bs"], D["d"]), dtype=torch.bfloat16,
                              device=dev)
        self.vc = torch.empty_like(self.kc)
        ra.cp_kv_scatter(kt, vt, slot[self.dev0:self.dev0 + self.n_dev], self.kc, self.vc)
        last = (qsl[1:] - 1).long()
        self.new_k = kt[last.to(dev)].contiguous()
        self.new_v = vt[last.to(dev)].contiguous()
        del kt, vt, slot
        self.new_pos = (ctx - 1).to(torch.int32).to(dev)
        self.new_qsl = torch.arange(D["R"] + 1, dtype=torch.int32, device=dev)
        self.new_slot = torch.empty((W, D["R"]), dtype=torch.int32, device=dev)
        self.qd = I.synth_normal(D["seed"], I.TID_Q, (D["R"], D["Hq"], D["d"]), torch.bfloat16).to(dev)
        self.op, self.lp = ra.cp_decode_partials(self.qd, self.kc, self.vc, self.bt, self.ctx, D["I"], D["pcp"],
                                                 D["dcp"], dev0=self.dev0, split_blocks=D["split"])
        self.o_loc = torch.empty((D["R"], D["Hq"], D["d"]), dtype=torch.float32, device=dev)
        self.l_loc = torch.empty((D["R"], D["Hq"]), dtype=torch.float32, device=dev)
        self.rescale = ra.cp_lse_rescale_fn()
        self.ctx_host = ctx
        self.parts = ("prefill", "decode")
        torch.cuda.synchronize()

    def step(self, e=None):
        ra, D = self.ra, DECODE
        if e: e[0].record()
        self.o, self.lse = self.cp.ring_attention(self.q, self.k, self.v, step=self.ring_step, exchange=self.exchange,
                                                  out_dtype=torch.bfloat16)
        if e: e[1].record()
        ra.cp_slot_mapping(self.new_qsl, self.new_pos, self.bt, D["bs"], D["I"], D["pcp"], D["dcp"], out=self.new_slot)
        ra.cp_kv_scatter(self.new_k, self.new_v, self.new_slot[self.dev0:self.dev0 + self.n_dev], self.kc, self.vc)
        if e: e[2].record()
        ra.cp_decode_partials(self.qd, self.kc, self.vc, self.bt, self.ctx, D["I"], D["pcp"], D["dcp"],
                              dev0=self.dev0, split_blocks=D["split"], o_parts=self.op, lse_parts=self.lp)
        ra.lse_merge(self.op, self.lp, o=self.o_loc, lse=self.l_loc)
        self.od, self.ld = self.cp.cp_lse_ag_out_rs(self.o_loc, self.l_loc, rescale=self.rescale)
        if e: e[3].record()

    def decode_bytes(self):
        return Workload.decode_bytes(self)


def run_dist(args, rank, world, dev):
    """The benchmark line of the step split across `world` ranks (strong scaling: the same prefill
    and decode, whatever the number of ranks)."""
    from context_long_sequence_ring_gb300 import ringattn as ra
    ra.lib()
    wl = DistWorkload(ra, dev, rank, world)
    P = PREFILL
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    if ra.device_status() != 0:
        raise RuntimeError("device status after warm-up: %s" % ra.last_error())
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        t0.record()
        for i in range(args.steps):
            wl.step(evs[i])
        t1.record()
        torch.cuda.synchronize()
    _barrier(world)
    ms_step = _max_over_ranks(t0.elapsed_time(t1), world, dev) / args.steps
    if ra.device_status() != 0:
        raise RuntimeError("device status after timing: %s" % ra.last_error())
    ring_ms = _max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in evs), world, dev)
    dec_ms = _max_over_ranks(statistics.mean(e[2].elapsed_time(e[3]) for e in evs), world, dev)
    flops = causal_flops(P["B"], P["Hq"], P["S"], P["d"])
    dec_bytes, kv_bytes = wl.decode_bytes()
    pk = _peaks()
    # end to end, copies serial with the step: this rank's inputs in from pinned host buffers, its
    # outputs (its rows of O and LSE, its heads of the decode output) back
    host_in = {n: getattr(wl, n).cpu().pin_memory() for n in ("q", "k", "v", "qd", "new_k", "new_v")}
    wl.step()
    torch.cuda.synchronize()
    host_out = {n: torch.empty(getattr(wl, n).shape, dtype=getattr(wl, n).dtype).pin_memory()
                for n in ("o", "lse", "od", "ld")}
    n_e2e = max(1, min(args.steps, 5))
    _barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n_e2e):
        for n, h in host_in.items():
            getattr(wl, n).copy_(h, non_blocking=True)
        wl.step()
        for n, h in host_out.items():
            h.copy_(getattr(wl, n), non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1), world, dev) / n_e2e
    h2d = sum(x.numel() * x.element_size() for x in host_in.values())
    d2h = sum(x.numel() * x.element_size() for x in host_out.values())
    per_gpu = flops / world / (ring_ms * 1e-3) / 1e12
    return {
        "metric": METRIC, "value": round(flops / (ms_step * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded counter-based N(0,1), bf16)",
        "config": {"workload": workload_name(), "prefill": PREFILL, "decode": dict(DECODE),
                   "l2": "inputs larger than L2",
                   "parallelism": "context parallel over %d ranks: prefill ring of %d zigzag ranks (K/V blocks passed "
                                  "by NCCL send/recv), decode KV cache sharded %d devices per rank with "
                                  "cp_lse_ag_out_rs" % (world, world, wl.n_dev)},
        "parts": {"ring_ms": round(ring_ms, 3), "ring_tflops_per_gpu": round(per_gpu, 1),
                  "decode_merge_ms": round(dec_ms, 4), "decode_merge_gbs": round(dec_bytes / (dec_ms * 1e-3) / 1e9, 1),
                  "decode_kv_bytes": kv_bytes, "decode_alg_bytes": dec_bytes},
        "roofline": {"bound": "tensor", "achieved": round(per_gpu, 1), "peak": pk["bf16"], "unit": "TFLOP/s",
                     "frac": round(per_gpu / pk["bf16"], 4), "traffic": None,
                     "kernel": "attn_pair_kernel<StepPolicy> (one ring step per launch, %d per rank)" % world,
                     "peak_kind": "bf16 dense burst (%s)" % pk["src"],
                     "algorithmic": "%.4g FLOP per rank over its %d steps, time including exposed communication"
                                    % (flops / world, world)},
        "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                "copies": "serial with the step, this rank's shard in and its outputs out"},
        "gpu_launches": (world + 5) * args.steps,
        "clocks": clk.summary(),
    }


def run_ours(args, rank, world, dev):
    """The benchmark line on one GPU: the single-device kernels (the ring of N virtual ranks in one
    launch, the decode over all W cache devices with one merge).  More ranks run run_dist."""
    from context_long_sequence_ring_gb300 import ringattn as ra
    ra.lib()
    wl = Workload(ra, dev)
    P = PREFILL
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    st = ra.device_status()
    if st != 0:
        raise RuntimeError("device status %d after warm-up: %s" % (st, ra.last_error()))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        t_start.record()
        for i in range(args.steps):
            wl.step(evs[i])
        t_end.record()
        torch.cuda.synchronize()
    _barrier(world)
    ms_total = t_start.elapsed_time(t_end)
    ms_total = _max_over_ranks(ms_total, world, dev)
    st = ra.device_status()
    if st != 0:
        raise RuntimeError("device status %d after timing: %s" % (st, ra.last_error()))
    attn_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    prefill_ms = statistics.mean(e[0].elapsed_time(e[3]) for e in evs)
    decode_kernel_ms = statistics.mean(e[4].elapsed_time(e[5]) for e in evs)
    decode_ms = statistics.mean(e[3].elapsed_time(e[5]) for e in evs)
    partition_gather_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    restore_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    slot_scatter_ms = statistics.mean(e[3].elapsed_time(e[4]) for e in evs)
    flops = causal_flops(P["B"], P["Hq"], P["S"], P["d"])
    dec_bytes, kv_bytes = wl.decode_bytes()
    pk = _peaks()
    ms_step = ms_total / args.steps
    value = flops / (ms_step * 1e-3) / 1e12

    # e2e through the public API from pinned host buffers: H2D Q/K/V and the decode step's
    # inputs, the full step, D2H of O/LSE and the decode output.
    hq, hk, hv = (x.cpu().pin_memory() for x in (wl.q, wl.k, wl.v))
    hqd, hnk, hnv = (x.cpu().pin_memory() for x in (wl.qd, wl.new_k, wl.new_v))
    ho, hl = torch.empty_like(hq).pin_memory(), torch.empty_like(wl.lse, device="cpu").pin_memory()
    hod, hld = torch.empty_like(hqd).pin_memory(), torch.empty_like(wl.ld, device="cpu").pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hqd, hnk, hnv))
    d2h = sum(x.numel() * x.element_size() for x in (ho, hl, hod, hld))
    # the same K steps as the device-timed value, so that the pipeline's fill (the first step's inputs)
    # and drain (the last step's results) weigh as little as in a serving loop of that length
    e2e_steps = max(1, args.steps)
    host_in = {"q": hq, "k": hk, "v": hv, "qd": hqd, "new_k": hnk, "new_v": hnv}
    host_out = {"o": ho, "lse": hl, "od": hod, "ld": hld}
    # serial: copy in, step, copy out, one after the other on one stream
    _barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(e2e_steps):
        for n, h in host_in.items():
            getattr(wl, n).copy_(h, non_blocking=True)
        wl.step()
        for n, h in host_out.items():
            h.copy_(getattr(wl, n), non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    serial_ms = _max_over_ranks(e0.elapsed_time(e1), world, dev) / e2e_steps
    _barrier(world)
    # pipelined: the same copies on two copy streams with double-buffered step inputs and
    # outputs, so that step i+1's inputs arrive and step i-1's results leave while step i runs
    e2e_ms = _max_over_ranks(e2e_pipelined(wl, host_in, host_out, e2e_steps), world, dev) / e2e_steps
    _barrier(world)

    attn_tflops = flops / (attn_ms * 1e-3) / 1e12
    dec_gbs = dec_bytes / (decode_kernel_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 3), "higher_is_better": True, "scaling": "strong",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded counter-based N(0,1), bf16)",
        "config": {"workload": workload_name(),
                   "prefill": PREFILL, "decode": {k: v for k, v in DECODE.items()},
                   "l2": "inputs larger than L2 (Q 1 GiB, K/V 256 MiB each, KV cache %.1f GB)" % (
                       2 * wl.kc.numel() * 2 / 1e9),
                   "parallelism": "1 GPU (N virtual context-parallel ranks in one kernel)"},
        "parts": {
            "prefill_ms": round(prefill_ms, 3), "ring_attn_kernel_ms": round(attn_ms, 3),
            "ring_attn_tflops": round(attn_tflops, 1),
            "decode_merge_ms": round(decode_kernel_ms, 4), "decode_step_ms": round(decode_ms, 4),
            "decode_merge_gbs": round(dec_gbs, 1), "decode_kv_bytes": kv_bytes, "decode_alg_bytes": dec_bytes,
            "partition_gather_ms": round(partition_gather_ms, 4), "restore_ms": round(restore_ms, 4),
            "slot_mapping_scatter_ms": round(slot_scatter_ms, 4),
        },
        "roofline": ring_roofline(attn_tflops, flops, pk, clk.summary()),
        "roofline_decode": {"bound": "hbm", "achieved": round(dec_gbs, 1), "peak": pk["hbm"], "unit": "GB/s",
                            "frac": round(dec_gbs / pk["hbm"], 4), "traffic": _traffic("cp_decode"),
                            "kernel": "cp_decode_kernel + lse_merge_kernel", "peak_kind": "HBM copy (%s)" % pk["src"],
                            "algorithmic": "%d bytes per step" % dec_bytes},
        "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                "copies": "pipelined on two copy streams, double-buffered step inputs and outputs",
                "serial": {"value": round(flops / (serial_ms * 1e-3) / 1e12, 2),
                           "ms_per_step": round(serial_ms, 3)}},
        "gpu_launches": wl.launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    line["next_segmented_prefill"] = measure_segmented(ra, dev)
    line["next_kv_reorg"] = measure_kv_reorg(ra, wl)
    line["next_rope_prologue"] = measure_rope(ra, wl)
    line["merge_stress"] = measure_merge(ra, dev)
    line["varlen_prefill"] = measure_varlen(ra, dev)
    line["cp_ring_emulated"] = measure_ring_dist(ra, wl)
    line["cp_allgather_emulated"] = measure_allgather(ra, wl)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_rows)
    return line


def ring_roofline(attn_tflops, flops, pk, clocks):
    """Roofline of the ring-attention kernel.  The headline fraction is taken against the burst bf16
    GEMM peak: the sustained GEMM figure was measured at a lower median SM clock than the ring kernel
    runs at inside the step, so it would flatter the kernel.  The sustained fraction and both clocks
    are given beside it."""
    return {"bound": "tensor", "achieved": round(attn_tflops, 1), "peak": pk["bf16"], "unit": "TFLOP/s",
            "frac": round(attn_tflops / pk["bf16"], 4), "traffic": _traffic("ring_attn_bf16"),
            "kernel": "attn_pair_kernel<RingPolicy> (ring order, two GQA heads per CTA)",
            "peak_kind": "bf16 dense burst (%s)" % pk["src"],
            "peak_sustained": pk["bf16_sus"], "frac_sustained": round(attn_tflops / pk["bf16_sus"], 4),
            "sm_mhz_kernel_median": clocks.get("sm_mhz"), "sm_mhz_sustained_gemm_median": pk.get("sus_mhz"),
            "algorithmic": "%.4g FLOP per launch" % flops}


def run_parts(args, dev):
    """Run only some parts of the step (for profiler captures); prints part times, no headline."""
    from context_long_sequence_ring_gb300 import ringattn as ra
    parts = tuple(args.parts.split(","))
    wl = Workload(ra, dev, parts)
    for _ in range(args.warmup):
        wl.step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for i in range(args.steps):
        wl.step(evs[i])
    torch.cuda.synchronize()
    st = ra.device_status()
    if st != 0:
        raise RuntimeError("device status %d: %s" % (st, ra.last_error()))
    out = {"parts": list(parts), "prefill": PREFILL if "prefill" in parts else None,
           "ring_attn_kernel_ms": statistics.mean(e[1].elapsed_time(e[2]) for e in evs),
           "decode_merge_ms": statistics.mean(e[4].elapsed_time(e[5]) for e in evs)}
    if "prefill" in parts:
        P = PREFILL
        out["ring_attn_tflops"] = causal_flops(P["B"], P["Hq"], P["S"], P["d"]) / (out["ring_attn_kernel_ms"] * 1e-3) / 1e12
    if "decode" in parts:
        out["decode_merge_gbs"] = wl.decode_bytes()[0] / (out["decode_merge_ms"] * 1e-3) / 1e9
    if "rope" in parts:
        out["rope"] = measure_rope(ra, wl)
    if "reorg" in parts:
        out["reorg"] = measure_kv_reorg(ra, wl, n_req=min(8, DECODE["R"]))
    if "merge" in parts:
        out["merge"] = measure_merge(ra, dev)
    if "segmented" in parts:
        out["segmented"] = measure_segmented(ra, dev)
    if "varlen" in parts:
        out["varlen"] = measure_varlen(ra, dev)
    if "ringdist" in parts:
        out["ringdist"] = measure_ring_dist(ra, wl)
    if "allgather" in parts:
        out["allgather"] = measure_allgather(ra, wl)
    print(json.dumps(out), flush=True)


SEGMENTED = dict(ctx=122880, Tq=8192, Hq=32, Hkv=8, d=128, seg=32768, seed=6)


def measure_segmented(ra, dev, reps=5):
    """Chunked prefill with bounded KV per round (the next scope row): Tq new tokens after ctx cached
    ones, key segments of `seg` tokens, partials merged by LSE.  Timed alone with CUDA events."""
    S = SEGMENTED
    T = S["ctx"] + S["Tq"]
    tab = I.normal_table(torch.bfloat16)
    q = ra.synth_fill(I.tensor_key(S["seed"], I.TID_Q), tab, (S["Tq"], S["Hq"], S["d"]), dev)
    k = ra.synth_fill(I.tensor_key(S["seed"], I.TID_K), tab, (T, S["Hkv"], S["d"]), dev)
    v = ra.synth_fill(I.tensor_key(S["seed"], I.TID_V), tab, (T, S["Hkv"], S["d"]), dev)
    for _ in range(2):
        ra.segmented_prefill_fwd(q, k, v, S["ctx"], S["seg"])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        ra.segmented_prefill_fwd(q, k, v, S["ctx"], S["seg"])
    e1.record()
    torch.cuda.synchronize()
    if ra.device_status() != 0:
        raise RuntimeError("device status after the segmented prefill: %s" % ra.last_error())
    ms = e0.elapsed_time(e1) / reps
    pairs = sum(range(S["ctx"] + 1, T + 1))          # query at position i sees i+1 keys
    flops = 4.0 * S["Hq"] * S["d"] * pairs
    return {"config": S, "ms": round(ms, 3), "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
            "frac_of_bf16_sustained": round(flops / (ms * 1e-3) / 1e12 / _peaks()["bf16_sus"], 4)}


def measure_kv_reorg(ra, wl, n_req=8, reps=5):
    """Reorg of the sharded cache back to contiguous per-request K/V (the next scope row after the
    segmented prefill): every context token of the first n_req decode requests, timed alone."""
    D = DECODE
    ctx = wl.ctx[:n_req].cpu()
    qsl = torch.zeros(n_req + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(ctx, 0)
    pos = torch.cat([torch.arange(int(L), dtype=torch.int32) for L in ctx]).to(wl.dev)
    qsl = qsl.to(wl.dev)
    bt = wl.bt[:n_req].contiguous()
    T = int(pos.numel())
    k_out = torch.empty((T, D["Hkv"], D["d"]), dtype=torch.bfloat16, device=wl.dev)
    v_out = torch.empty_like(k_out)
    for _ in range(2):
        ra.cp_kv_gather(wl.kc, wl.vc, bt, qsl, pos, D["I"], D["pcp"], D["dcp"], k_out, v_out)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        ra.cp_kv_gather(wl.kc, wl.vc, bt, qsl, pos, D["I"], D["pcp"], D["dcp"], k_out, v_out)
    e1.record()
    torch.cuda.synchronize()
    if ra.device_status() != 0:
        raise RuntimeError("device status after the KV reorg: %s" % ra.last_error())
    ms = e0.elapsed_time(e1) / reps
    nbytes = 2 * 2 * T * D["Hkv"] * D["d"] * 2          # K and V, read once and written once
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"requests": n_req, "tokens": T, "ms": round(ms, 3), "gbs": round(gbs, 1),
            "frac_of_hbm": round(gbs / _peaks()["hbm"], 4)}


VARLEN = dict(lens=[65536, 32768, 16384, 12288, 4096, 100], N=16, Hq=32, Hkv=8, d=128, seed=10)


def measure_varlen(ra, dev, reps=5):
    """Several requests of different lengths in one ring call, on the head-tail gathered layout
    (the pages' multi-request PCP prefill); causal attention FLOPs of the real tokens only."""
    V = VARLEN
    tab = I.normal_table(torch.bfloat16)
    G = sum(-(-L // (2 * V["N"])) * 2 * V["N"] for L in V["lens"])
    q = ra.synth_fill(I.tensor_key(V["seed"], I.TID_Q), tab, (G, V["Hq"], V["d"]), dev)
    k = ra.synth_fill(I.tensor_key(V["seed"], I.TID_K), tab, (G, V["Hkv"], V["d"]), dev)
    v = ra.synth_fill(I.tensor_key(V["seed"], I.TID_V), tab, (G, V["Hkv"], V["d"]), dev)
    o, lse = torch.empty_like(q), torch.empty((G, V["Hq"]), dtype=torch.float32, device=dev)
    for _ in range(2):
        ra.ring_attn_fwd_varlen(q, k, v, V["lens"], True, V["N"], o=o, lse=lse)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        ra.ring_attn_fwd_varlen(q, k, v, V["lens"], True, V["N"], o=o, lse=lse)
    e1.record()
    torch.cuda.synchronize()
    if ra.device_status() != 0:
        raise RuntimeError("device status after the varlen prefill: %s" % ra.last_error())
    ms = e0.elapsed_time(e1) / reps
    flops = sum(causal_flops(1, V["Hq"], L, V["d"]) for L in V["lens"])
    tf = flops / (ms * 1e-3) / 1e12
    return {"config": V, "ms": round(ms, 3), "tflops": round(tf, 1),
            "frac_of_bf16_sustained": round(tf / _peaks()["bf16_sus"], 4)}


RING_DIST = dict(ranks=8)
RING_VARIANT = [0]   # kernel variant of ra_ring_attn_fwd_ex (0: the library's choice)


def measure_ring_dist(ra, wl, reps=3):
    """The prefill as the ranks of a ring across devices, all emulated on this GPU: each rank holds
    its head-tail chunk pair, every step is one ra_ring_step_fwd launch on the block the rank holds,
    and the blocks move between the ranks' buffers by device copies on a side stream (double
    buffering).  All ranks' steps run one after the other here, so the time is the work of the whole
    ring on one device; on N devices each would run 1/N of it."""
    from context_long_sequence_ring_gb300 import cp_dist
    P = PREFILL
    if "prefill" not in wl.parts or P["B"] != 1:
        return None
    N = RING_DIST["ranks"]
    perm, _ = ra.zigzag_partition([P["S"]], N)
    c = P["S"] // (2 * N)
    locs = [perm[r * 2 * c:(r + 1) * 2 * c] for r in range(N)]
    qs = [ra.gather_rows(wl.q, i) for i in locs]
    ks = [ra.gather_rows(wl.k, i) for i in locs]
    vs = [ra.gather_rows(wl.v, i) for i in locs]
    steps = [ra.ring_step_fn(N, r, True) for r in range(N)]

    def run():
        return cp_dist.ring_attention_local(qs, ks, vs, step=lambda r, *a: steps[r](*a))
    run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        run()
    e1.record()
    torch.cuda.synchronize()
    if ra.device_status() != 0:
        raise RuntimeError("device status after the emulated ring: %s" % ra.last_error())
    ms = e0.elapsed_time(e1) / reps
    tf = causal_flops(1, P["Hq"], P["S"], P["d"]) / (ms * 1e-3) / 1e12
    del qs, ks, vs
    return {"ranks": N, "step_launches": N * N, "ms_all_ranks": round(ms, 3), "tflops": round(tf, 1),
            "frac_of_bf16_burst": round(tf / _peaks()["bf16"], 4),
            "note": "every rank's ring steps on one GPU, blocks rotated by device copies; not in value"}


def measure_allgather(ra, wl, reps=2):
    """The prefill in the form with the K/V all-gathered (the ranks' chunk pairs concatenated are the
    gathered order), ranks emulated on this GPU: per rank, the restore of the gathered K/V to token
    order (row-gather kernel) and its two chunks' attention over the keys in token order, in
    32768-key segments (segmented prefill kernels).  All ranks run one after the other here."""
    P = PREFILL
    if "prefill" not in wl.parts or P["B"] != 1:
        return None
    N, S = RING_DIST["ranks"], P["S"]
    c = S // (2 * N)
    perm, restore = ra.zigzag_partition([S], N)
    kz, vz = ra.gather_rows(wl.k, perm), ra.gather_rows(wl.v, perm)
    qs = [ra.gather_rows(wl.q, perm[r * 2 * c:(r + 1) * 2 * c]) for r in range(N)]
    k_nat, v_nat = torch.empty_like(kz), torch.empty_like(vz)
    o = torch.empty_like(qs[0])
    lse = torch.empty(qs[0].shape[:2], dtype=torch.float32, device=wl.dev)
    attends = [ra.allgather_attend_fn(S, N, r, True) for r in range(N)]

    def run():
        for r in range(N):
            ra.gather_rows(kz, restore, k_nat)
            ra.gather_rows(vz, restore, v_nat)
            attends[r](qs[r], k_nat, v_nat, o, lse)
    run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        run()
    e1.record()
    torch.cuda.synchronize()
    if ra.device_status() != 0:
        raise RuntimeError("device status after the all-gather prefill: %s" % ra.last_error())
    ms = e0.elapsed_time(e1) / reps
    tf = causal_flops(1, P["Hq"], S, P["d"]) / (ms * 1e-3) / 1e12
    del qs, kz, vz, k_nat, v_nat
    return {"ranks": N, "ms_all_ranks": round(ms, 3), "tflops": round(tf, 1),
            "frac_of_bf16_burst": round(tf / _peaks()["bf16"], 4),
            "note": "every rank's restore and attention on one GPU (the all-gather itself is communication); "
                    "not in value"}


MERGE = dict(P=8, T=32768, H=32, d=128, seed=7)


def measure_merge(ra, dev, reps=10):
    """The LSE merge on its own at a size where it is HBM-bound: P fp32 partials of [T, H, d]
    (4.3 GB read) merged into a bf16 O and an fp32 LSE.  Timed with CUDA events."""
    M = MERGE
    P, T, H, d = M["P"], M["T"], M["H"], M["d"]
    tab = I.normal_table(torch.float32)
    o_parts = ra.synth_fill(I.tensor_key(M["seed"], 0), tab, (P, T, H, d), dev)
    lse_parts = ra.synth_fill(I.tensor_key(M["seed"], 1), tab, (P, T, H), dev)
    o = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, H), dtype=torch.float32, device=dev)
    for _ in range(2):
        ra.lse_merge(o_parts, lse_parts, o=o, lse=lse)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        ra.lse_merge(o_parts, lse_parts, o=o, lse=lse)
    e1.record()
    torch.cuda.synchronize()
    if ra.device_status() != 0:
        raise RuntimeError("device status after the merge stress: %s" % ra.last_error())
    ms = e0.elapsed_time(e1) / reps
    nbytes = P * T * H * (d + 1) * 4 + T * H * (d * 2 + 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    del o_parts, lse_parts
    return {"config": M, "ms": round(ms, 4), "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / _peaks()["hbm"], 4)}


def measure_rope(ra, wl, reps=5):
    """RoPE prologue (the next scope row after the KV reorg): the prefill's Q and K rotated by
    their positions while they are gathered to the zigzag layout, against the plain gather of the
    same rows.  Timed alone with CUDA events; the partition comes from the last bench step."""
    P = PREFILL
    if "prefill" not in wl.parts:
        return None
    pos = torch.arange(P["S"], dtype=torch.int32, device=wl.dev).repeat(P["B"])

    def rope():
        ra.rope_gather(wl.q, pos, wl.perm, out=wl.qz)
        ra.rope_gather(wl.k, pos, wl.perm, out=wl.kz)

    def plain():
        ra.gather_rows(wl.q, wl.perm, wl.qz)
        ra.gather_rows(wl.k, wl.perm, wl.kz)

    res = {}
    for name, fn in (("rope", rope), ("plain", plain)):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) / reps
    if ra.device_status() != 0:
        raise RuntimeError("device status after the RoPE prologue: %s" % ra.last_error())
    rows = P["B"] * P["S"]
    G = int(wl.perm.numel())
    # Q and K rows read once and written once, plus the gather index and one position per row
    nbytes = (rows + G) * (P["Hq"] + P["Hkv"]) * P["d"] * 2 + 2 * (G * 4 + rows * 4)
    gbs = nbytes / (res["rope"] * 1e-3) / 1e9
    return {"tensors": "Q [%d, %d, %d] and K [%d, %d, %d] bf16, base 10000" % (rows, P["Hq"], P["d"], rows, P["Hkv"],
                                                                               P["d"]),
            "ms": round(res["rope"], 4), "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / _peaks()["hbm"], 4),
            "plain_gather_ms": round(res["plain"], 4), "vs_plain_gather": round(res["rope"] / res["plain"], 3)}


# ---------------------------------------------------------------------------- oracle arm

def _threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


class OracleSample:
    """The float64 oracle on a sample of query rows of the prefill workload."""

    def __init__(self, rows_per_step):
        P = PREFILL
        S, Hkv, d = P["S"], P["Hkv"], P["d"]
        self.k = I.synth_rows(P["seed"], I.TID_K, np.arange(S), Hkv * d, torch.bfloat16).reshape(S, Hkv, d)
        self.v = I.synth_rows(P["seed"], I.TID_V, np.arange(S), Hkv * d, torch.bfloat16).reshape(S, Hkv, d)
        self.k64 = self.k.double().numpy()
        self.v64 = self.v.double().numpy()
        self.rng = np.random.default_rng(77)
        self.n = rows_per_step

    def step(self):
        import oracle
        P = PREFILL
        rows = np.sort(self.rng.integers(0, P["S"], size=self.n))
        qr = I.synth_rows(P["seed"], I.TID_Q, rows, P["Hq"] * P["d"], torch.bfloat16).reshape(-1, P["Hq"], P["d"])
        t0 = time.perf_counter()
        oracle.attention_rows(qr, rows, self.k64, self.v64, True)
        dt = time.perf_counter() - t0
        flops = 4.0 * P["Hq"] * P["d"] * float(np.sum(rows + 1))     # causal pairs of the sampled rows
        return flops, dt


def cpu_baseline(rows):
    s = OracleSample(rows)
    s.step()  # warm
    fl, dt = 0.0, 0.0
    while dt < 10.0:
        f, t = s.step()
        fl += f
        dt += t
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": _threads(), "kind": "oracle",
            "sample": "%d random query rows x 32 heads of the S=131072 causal prefill per call, float64 numpy, "
                      "%.1f s of CPU time; the rate is extrapolated to the full prefill (about %.0f s)"
                      % (rows, dt, causal_flops(PREFILL["B"], PREFILL["Hq"], PREFILL["S"], PREFILL["d"]) / (fl / dt))}


def workload_name():
    """Name of the measured workload, built from the sizes the run actually uses."""
    P, D = PREFILL, DECODE
    return ("causal GQA ring prefill B=%d Hq=%d Hkv=%d S=%d d=%d N=%d zigzag ranks "
            "+ CP decode %d req ctx U[%d,%d] Hq=%d Hkv=%d d=%d bs=%d I=%d pcp=%d dcp=%d"
            % (P["B"], P["Hq"], P["Hkv"], P["S"], P["d"], P["N"], D["R"], D["lo"], D["hi"], D["Hq"], D["Hkv"],
               D["d"], D["bs"], D["I"], D["pcp"], D["dcp"]))


def run_reference(args):
    s = OracleSample(args.cpu_rows)
    for _ in range(args.warmup):
        s.step()
    fl, dt = 0.0, 0.0
    for _ in range(args.steps):
        f, t = s.step()
        fl += f
        dt += t
    value = fl / dt / 1e12
    cb = {"value": round(value, 6), "unit": "TFLOP/s", "cores": _threads(), "kind": "oracle",
          "sample": "%d random query rows x 32 heads per step of the S=131072 causal prefill, float64 numpy; "
                    "the step's decode (about 71 GFLOP over 4.3 M cached tokens, against the prefill's 140.7 TFLOP) "
                    "is not timed" % args.cpu_rows}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_name(), "prefill": PREFILL, "decode": {k: v for k, v in DECODE.items()},
                       "sample": "prefill query rows sampled at random, rate extrapolated to the whole step"},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------- driver

def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


def _max_over_ranks(x, world, dev):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--parts", default="all",
                    help="'all' for the benchmark line, else a comma list of 'prefill', 'decode', 'rope' (the "
                         "RoPE prologue, needs 'prefill'), 'reorg' (the KV reorg, needs 'decode'), 'merge', "
                         "'segmented', 'varlen', 'ringdist' (the ring across emulated devices, needs 'prefill') and "
                         "'allgather' (the all-gather-KV prefill across emulated devices, needs 'prefill') to run "
                         "only those parts (profiler captures)")
    ap.add_argument("--prefill-seq", type=int, default=None, help="override S of the prefill (multiple of 2N)")
    ap.add_argument("--decode-requests", type=int, default=None, help="override the number of decode requests")
    ap.add_argument("--merge-tokens", type=int, default=None, help="override T of the stand-alone merge")
    ap.add_argument("--decode-split", type=int, default=None, help="override the decode's virtual blocks per split")
    ap.add_argument("--ring-variant", type=int, default=None,
                    help="bf16 kernel variant of the ring attention (ra_ring_attn_fwd_ex), for --parts runs")
    ap.add_argument("--cp-dist", action="store_true",
                    help="run the step split across the job's ranks (the path used for more than one GPU) even "
                         "on one rank")
    ap.add_argument("--prefill-shape", default=None,
                    help="B,Hq,Hkv,S,N of the prefill, for the parts runs (e.g. 1,8,8,8192,8 or 2,32,8,32768,8)")
    args = ap.parse_args()
    if args.parts == "all":
        for flag, val in (("--prefill-shape", args.prefill_shape), ("--prefill-seq", args.prefill_seq),
                          ("--ring-variant", args.ring_variant),
                          ("--decode-requests", args.decode_requests), ("--merge-tokens", args.merge_tokens),
                          ("--decode-split", args.decode_split)):
            if val is not None:
                ap.error("%s is for --parts runs; the benchmark line keeps its workload" % flag)
    if args.prefill_shape:
        B, Hq, Hkv, S, N = (int(x) for x in args.prefill_shape.split(","))
        PREFILL.update(B=B, Hq=Hq, Hkv=Hkv, S=S, N=N)
    if args.prefill_seq:
        PREFILL["S"] = args.prefill_seq
    if args.ring_variant is not None:
        RING_VARIANT[0] = args.ring_variant
    if args.decode_requests:
        DECODE["R"] = args.decode_requests
    if args.merge_tokens:
        MERGE["T"] = args.merge_tokens
    if args.decode_split:
        DECODE["split"] = args.decode_split
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.parts != "all":
        run_parts(args, dev)
        return
    if world > 1 or args.cp_dist:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29533")
        os.environ.setdefault("RANK", str(rank))
        os.environ.setdefault("WORLD_SIZE", str(world))
        torch.distributed.init_process_group("nccl", device_id=dev)
    line = run_dist(args, rank, world, dev) if (world > 1 or args.cp_dist) else run_ours(args, rank, world, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
