"""Benchmark: paged absorbed-MLA decode, microseconds per layer-call, on one GB300.

Workload (default): 64 slots x 24 MLA layers, every slot at 4096 tokens (64
pages), 96 heads, kv_lora 512 + rope 64, seed 2 -- synthetic, device-resident
(7.25 GB slab, 302 MB of latent per layer, so every layer's inputs exceed the
129 MB L2; no flush is needed between steps).

A step is one pass of the whole hot path over the batch, for every layer: the
new token's latent row appended into its mapped page, q absorbed, and the paged
decode (split decode + merge / W_UV expansion).  The host page claim (pool
ensure + table) runs once per step in the end-to-end leg.

JSON line fields beyond the usual ones:
  value            us per layer-call (24-layer step replayed as a CUDA graph / 24)
  latent_gbs       latent bytes read per layer-call / time
  roofline         the paged-decode call (split decode + merge/expand kernels):
                   algorithmic bytes / its device time (24 decode calls in one
                   CUDA graph, timed with events, / 24) vs measured HBM
  layer_roofline   the same for the whole layer-call (append + absorb + decode)
  e2e              the same metric through the C ABI with host buffers: pinned
                   H2D of the step's q / new rows / tables and D2H of the outputs
                   inside the timed region (host page claims, then the step's
                   copies and kernels replayed as one CUDA graph)
  cpu_baseline     the CPU oracle on a bounded sample of the workload (all host
                   threads, and one thread)
  workloads        long8, ragged16 and padding128 under the default per-slot
                   split (and ragged16 under the opt-in batch-planned split)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_latent_attention_k3mla_gb300 import synth  # noqa: E402

METRIC = "absorbed-MLA decode µs/layer and latent GB/s vs HBM/tensor roofline"
H, NOPE, ROPE, V, LORA, ROW, PAGE = 96, 128, 64, 128, 512, 576, 64
XR = NOPE + ROPE + V   # one head's row of the expanded cache: K nope, K rope, V
WORKLOAD_DESC = {
    "steady64": "64 slots x 24 MLA layers x 4096 tokens (seed 2)",
    "ragged16": "16 slots x 24 MLA layers, ctx U[1,4096] (seed 1)",
    "long8": "8 slots x 24 MLA layers x 32768 tokens, heavy-tailed rows (seed 3)",
    "padding128": "128 rows, 40% padding, ctx U[1,256] (seed 4)",
    "tiny": "1 slot x 1 layer x 130 tokens (seed 0)",
}
MAX_CTX = {"steady64": 4096, "ragged16": 4096, "long8": 32768, "padding128": 256, "tiny": 256}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev=0):
        self.dev = dev
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[0]))
                mx = max(mx, float(f[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def alg_bytes(wl):
    lat = wl.latent_bytes()
    q = wl.B * H * (NOPE + ROPE) * 2
    out = wl.B * H * V * 2
    w = H * (NOPE + V) * LORA * 2
    return dict(latent=lat, layer=lat + q + out + w + wl.B * ROW * 2,
                decode=lat + wl.B * H * ROW * 2 + H * V * LORA * 2 + out)


def alg_flops(wl):
    n = int(wl.ctx_len.astype(np.int64).clip(min=0).sum())
    return n * H * 2 * (ROW + LORA) + 2 * 2 * wl.B * H * 128 * LORA


def _oracle_sample(wl, layers, slots, nthreads):
    """Seconds the oracle (absorption + decode chain, as it stands) takes for the listed slots of the
    listed layers, on `nthreads` host threads."""
    import oracle
    tbl = wl.block_table[slots]
    used = sorted(set(int(x) for x in tbl.ravel() if x >= 0))
    remap = {p: i for i, p in enumerate(used)}
    idx = torch.tensor(used if used else [0], dtype=torch.long, device=wl.slab.device)
    t2 = np.vectorize(lambda x: remap.get(int(x), -1))(tbl).astype(np.int32)
    dt = 0.0
    for layer in layers:
        slab = synth.bf16_bits(wl.slab.index_select(0, idx)[:, layer:layer + 1])
        q = synth.bf16_bits(wl.q[layer][slots])
        w = synth.bf16_bits(wl.w_kv_b[layer])
        t0 = time.perf_counter()
        qa = oracle.absorb(q, w)
        oracle.decode(qa, slab, 0, t2, wl.ctx_len[slots].astype(np.int32), w, wl.scale_bits, nthreads=nthreads)
        dt += time.perf_counter() - t0
    return dt


def cpu_baseline(wl):
    """The oracle (as it stands) on a bounded sample of the workload: all slots of up to 8 layers on
    every host core (about 10 s), and 2 slots of one layer on one thread; both scaled to one
    layer-call of the whole batch."""
    B = wl.B
    ncores = os.cpu_count() or 1
    n_slots = B if int(wl.ctx_len.max()) <= 4096 else 2
    layers = list(range(min(wl.n_layers, 8)))
    dt = _oracle_sample(wl, layers, list(range(n_slots)), ncores)
    us = dt * 1e6 / len(layers) * (B / n_slots)
    n1 = min(B, 2)
    dt1 = _oracle_sample(wl, [0], list(range(n1)), 1)
    us1 = dt1 * 1e6 * (B / n1)
    return {"value": us, "unit": "us/layer-call", "cores": ncores, "kind": "oracle",
            "sample": f"{n_slots} of {B} slots x {len(layers)} layer-call(s) (absorb + decode chain), "
                      f"{dt:.2f} s wall on {ncores} threads, scaled to one {B}-slot layer-call",
            "single_thread": {"value": us1, "unit": "us/layer-call", "cores": 1,
                              "sample": f"{n1} of {B} slots x 1 layer-call, {dt1:.2f} s wall on 1 thread, "
                                        f"scaled to one {B}-slot layer-call"}}


def config_for(name, wl, split, layers=None):
    """The bench line's config (both arms print the same dict for the same workload)."""
    L = wl.n_layers
    return {"workload": WORKLOAD_DESC[name] if layers is None else f"{WORKLOAD_DESC[name]}, first {L} layer(s) only",
            "slots": wl.B, "layers": L, "context_tokens": int(wl.ctx_len.max()),
            "split_tokens": "auto (per slot: ceil(ctx/4096) equal splits)" if split == 0 else split,
            "l2": "inputs larger than L2 (302 MB latent + 25 MB weights per layer, 7.8 GB per step)"
                  if name in ("steady64", "long8") else "per-layer inputs may be L2-resident",
            "timing": "24-layer step as one CUDA graph of k3mla_decode_layer calls (append carried by the "
                      "absorption's launch, then split decode and merge/expansion), CUDA events on the launch stream"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl = synth.make_workload(args.workload, device="cuda" if torch.cuda.is_available() else "cpu")
    ncores = os.cpu_count() or 1
    n_slots = min(wl.B, 16 if int(wl.ctx_len.max()) <= 4096 else 1)
    slots = list(range(n_slots))
    for _ in range(args.warmup):
        pass  # the oracle keeps no state between calls; nothing to warm
    step_s = []
    for _ in range(args.steps):
        step_s.append(_oracle_sample(wl, [0], slots, ncores))   # one step: the sample below, timed
    ms_step = statistics.mean(step_s) * 1e3
    v = ms_step * 1e3 * (wl.B / n_slots)   # us per layer-call of the whole batch
    sample = (f"{n_slots} of {wl.B} slots x 1 layer-call (absorb + decode chain) per step, on {ncores} threads; "
              f"value scales the measured step by {wl.B}/{n_slots} slots to one {wl.B}-slot layer-call")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "us/layer-call",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": config_for(args.workload, wl, 0, args.layers),
            "step_is_sample": {"slots": n_slots, "layers": 1,
                               "scale_to_layer_call": wl.B / n_slots,
                               "scaled_ms_per_full_step": v * wl.n_layers / 1e3},
            "cpu_baseline": {"kind": "oracle", "cores": ncores, "sample": sample, "value": v,
                             "unit": "us/layer-call"},
            "e2e": {"value": v, "unit": "us/layer-call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


class Runner:
    """One workload resident on the device, the hot path captured as CUDA graphs: the 24-layer step
    (absorption carrying the append, then the paged decode, per layer) and the paged-decode calls
    alone (24 calls), each replayed and timed with CUDA events on the launch stream."""

    def __init__(self, name, split, layers=None, fused=True, wl=None):
        from paged_latent_attention_k3mla_gb300 import k3mla
        self.k3mla = k3mla
        dev = "cuda"
        self.name = name
        self.wl = wl = synth.make_workload(name, device=dev, n_layers=layers) if wl is None else wl
        self.B, self.L = wl.B, wl.n_layers
        self.max_ctx = MAX_CTX[name]
        # a1: page claims from the host free-list pool (shuffled), table to the device.  The workload's
        # unmapped entries stay unmapped: its padding rows (every entry -1) claim nothing, and its holes
        # are -1 in the table the device sees (their appends are then flagged DEV_UNMAPPED and skipped)
        self.pool = k3mla.Pool(n_slots=self.B, max_ctx=self.max_ctx, n_pages=wl.n_pages, shuffle_seed=wl.seed + 1)
        self.unmapped = wl.block_table == -1
        self.claim_len = np.where(self.unmapped.all(axis=1), 0, wl.ctx_len).astype(np.int32)
        for b in range(self.B):
            rc = self.pool.ensure(b, int(self.claim_len[b]))
            assert rc == 0, rc
        self.host_table = self.mapped_table()
        # the one device-error bit the workload itself explains: appends into its unmapped pages
        last = np.maximum(wl.ctx_len - 1, 0) // PAGE
        hits = (wl.ctx_len > 0) & self.unmapped[np.arange(self.B), np.minimum(last, self.unmapped.shape[1] - 1)]
        self.err_ok = k3mla.DEV_UNMAPPED if hits.any() else 0
        self.table = torch.from_numpy(self.host_table).to(dev)
        self.ctx = torch.from_numpy(wl.ctx_len).to(dev)
        self.pos = torch.from_numpy(wl.pos).to(dev)
        self.split = split
        self.q_abs = torch.empty(self.B, H, ROW, dtype=torch.bfloat16, device=dev)
        self.out = torch.empty(self.L, self.B, H, V, dtype=torch.bfloat16, device=dev)
        self.ws = torch.empty(k3mla.decode_workspace_bytes(self.B, self.max_ctx, split), dtype=torch.uint8,
                              device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.Stream()
        # one public call per layer-call (k3mla_decode_layer: append at ctx - 1, absorption, paged decode
        # under the default split); a fixed split length goes through the separate calls instead
        self.fused = fused and split == 0
        self.lws = (torch.empty(k3mla.decode_layer_workspace_bytes(self.B, self.max_ctx), dtype=torch.uint8,
                                device=dev) if self.fused else None)

    def mapped_table(self):
        return np.where(self.unmapped, -1, self.pool.table()).astype(np.int32)

    def absorb_append(self, layer, q, c, r):
        # a2 + a3 in one launch: the append rides on the absorption's grid (neither reads the other)
        wl = self.wl
        self.k3mla.absorb_q_append(q, wl.w_kv_b[layer], self.q_abs, wl.slab, layer, self.table, self.pos, c, r,
                                   dev_err=self.err, stream=self.stream)

    def decode(self, layer):
        wl = self.wl
        self.k3mla.paged_decode(self.q_abs, wl.slab, layer, self.table, self.ctx, wl.w_kv_b[layer], wl.scale_bits,
                                self.out[layer], self.ws, self.max_ctx, self.split, dev_err=self.err,
                                stream=self.stream)

    def layer_call(self, layer, q, c, r):
        if self.fused:
            wl = self.wl
            self.k3mla.decode_layer(q, wl.w_kv_b[layer], wl.slab, layer, self.table, self.ctx, c, r, wl.scale_bits,
                                    self.out[layer], self.lws, self.max_ctx, dev_err=self.err, stream=self.stream)
        else:
            self.absorb_append(layer, q, c, r)
            self.decode(layer)

    def step(self):
        wl = self.wl
        for layer in range(self.L):
            self.layer_call(layer, wl.q[layer], wl.new_c[layer], wl.new_rope[layer])

    def decode_calls(self):
        for layer in range(self.L):
            self.decode(layer)

    def _graph(self, fn):
        with torch.cuda.stream(self.stream):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            fn()
        return g

    def _load(self, g, seconds):
        """Untimed replays for about `seconds` (keeps the GPU under this load while clocks are sampled)."""
        t0 = time.perf_counter()
        with torch.cuda.stream(self.stream):
            while time.perf_counter() - t0 < seconds:
                for _ in range(8):
                    g.replay()
                torch.cuda.synchronize()

    def _time_graph(self, g, steps, warmup, clocks=None):
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ctx = clocks if clocks is not None else _Null()
        with ctx:
            if clocks is not None:
                self._load(g, 0.5)      # the clock samples before the timed region see the same load
            torch.cuda.synchronize()
            ev0.record(self.stream)
            with torch.cuda.stream(self.stream):
                for _ in range(steps):
                    g.replay()
            ev1.record(self.stream)
            torch.cuda.synchronize()
            if clocks is not None:
                self._load(g, 0.5)
        return ev0.elapsed_time(ev1) / steps

    def measure(self, steps, warmup, clocks=None):
        """ms per 24-layer step, and ms per paged-decode call (24 paged-decode calls in one graph)."""
        g_step = self._graph(self.step)
        ms_step = self._time_graph(g_step, steps, warmup, clocks)
        assert self.err.item() & ~self.err_ok == 0, f"device error bits {self.err.item()}"
        del g_step
        if self.fused:  # the decode calls below read the absorbed q the layer calls left in their workspace
            self.q_abs = self.lws[:self.B * H * ROW * 2].view(torch.bfloat16).view(self.B, H, ROW)
        g_dec = self._graph(self.decode_calls)
        ms_dec = self._time_graph(g_dec, steps, warmup) / self.L
        assert self.err.item() & ~self.err_ok == 0, f"device error bits {self.err.item()}"
        del g_dec
        return ms_step, ms_dec

    def figures(self, ms_step, ms_dec, hbm):
        ab = alg_bytes(self.wl)
        us_layer = ms_step * 1e3 / self.L
        return {"us_per_layer_call": round(us_layer, 3), "decode_call_us": round(ms_dec * 1e3, 3),
                "decode_hbm_frac": round(ab["decode"] / (ms_dec * 1e-3) / 1e9 / hbm, 4),
                "layer_hbm_frac": round(ab["layer"] / (us_layer * 1e-6) / 1e9 / hbm, 4),
                "latent_gbs": round(ab["latent"] / (us_layer * 1e-6) / 1e9, 1)}


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def e2e_leg(run, steps, warmup):
    """The same step through the C ABI with host buffers: every step's inputs copied in from pinned
    host memory and every layer's output read back inside the timed region (host page claims and
    table refresh first, then one CUDA graph holding the copies -- on a copy stream, layer by layer,
    overlapping the compute -- and the 24 layer-calls)."""
    wl, L, stream = run.wl, run.L, run.stream
    q_all, c_all, r_all = wl.q, wl.new_c, wl.new_rope
    q_h = q_all.cpu().pin_memory()
    c_h = c_all.cpu().pin_memory()
    r_h = r_all.cpu().pin_memory()
    pos_h = torch.from_numpy(wl.pos).pin_memory()
    ctx_h = torch.from_numpy(wl.ctx_len).pin_memory()
    out_h = torch.empty(run.out.shape, dtype=run.out.dtype).pin_memory()
    q_d, c_d, r_d = torch.empty_like(q_all), torch.empty_like(c_all), torch.empty_like(r_all)
    h2d = (q_h.numel() + c_h.numel() + r_h.numel()) * 2 + (pos_h.numel() + ctx_h.numel()) * 4 + run.host_table.nbytes
    d2h = out_h.numel() * 2
    tbl_pin = torch.from_numpy(run.host_table.copy()).pin_memory()
    copy_s = torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(L)]
    # the compute stream waits for its inputs once per group of layers, the groups doubling (1, 1,
    # 2, 4, 8, ...) so that each group's copies finish while the layers before it compute; a wait on
    # another stream costs the overlap of the kernels around it, so fewer waits are cheaper
    first_of_group, start, size = {}, 0, 1
    while start < L:
        end = min(L, start + size)
        first_of_group[start] = end - 1             # wait for the last copy of the group
        start, size = end, (size if start == 0 else 2 * size)
    ev_dec = [torch.cuda.Event() for _ in range(L)]
    ev_out, ev_start = torch.cuda.Event(), torch.cuda.Event()

    def e2e_device_step():
        with torch.cuda.stream(stream):
            run.table.copy_(tbl_pin, non_blocking=True)
            run.pos.copy_(pos_h, non_blocking=True)
            run.ctx.copy_(ctx_h, non_blocking=True)
        ev_start.record(stream)                 # everything before (the previous step) is done
        copy_s.wait_event(ev_start)
        with torch.cuda.stream(copy_s):
            for layer in range(L):
                q_d[layer].copy_(q_h[layer], non_blocking=True)
                c_d[layer].copy_(c_h[layer], non_blocking=True)
                r_d[layer].copy_(r_h[layer], non_blocking=True)
                ev_in[layer].record(copy_s)
        for layer in range(L):
            if layer in first_of_group:             # the inputs of this group of layers have landed
                stream.wait_event(ev_in[first_of_group[layer]])
            with torch.cuda.stream(stream):
                run.layer_call(layer, q_d[layer], c_d[layer], r_d[layer])
                ev_dec[layer].record(stream)
            copy_s.wait_event(ev_dec[layer])
            with torch.cuda.stream(copy_s):
                out_h[layer].copy_(run.out[layer], non_blocking=True)
        ev_out.record(copy_s)
        stream.wait_event(ev_out)

    with torch.cuda.stream(stream):
        e2e_device_step()
    torch.cuda.synchronize()
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph, stream=stream):
        e2e_device_step()

    def e2e_step():
        rc = run.pool.ensure_all(run.claim_len)  # a1: claims on 64-token boundaries (none in steady state)
        assert rc == 0, rc
        t_now = run.mapped_table()
        if not np.array_equal(t_now, tbl_pin.numpy()):
            stream.synchronize()
            tbl_pin.numpy()[:] = t_now
        with torch.cuda.stream(stream):
            e2e_graph.replay()

    for _ in range(warmup):
        e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max(e0.elapsed_time(e1), (time.perf_counter() - t0) * 1e3) / steps
    digest = hashlib.sha256(out_h.view(torch.int16).numpy().tobytes()).hexdigest()[:16]
    return e2e_ms, int(h2d), int(d2h), digest


def extra_workloads(hbm, steps, warmup):
    """The other configurations' figures (parity cases, not the bench's value): each as its own
    24-layer CUDA-graph step under the default per-slot split; the ragged batch also under a fixed
    512-token split (as batch-invariant as the default: the latency setting for small batches) and
    under the opt-in batch-planned split (whose numerics depend on the batch)."""
    from paged_latent_attention_k3mla_gb300 import k3mla
    res = {}
    for name, split_kind in (("long8", "auto"), ("ragged16", "auto"), ("ragged16", "split512"),
                             ("ragged16", "planned"), ("padding128", "auto")):
        split = 512 if split_kind == "split512" else 0
        if split_kind == "planned":
            wl0 = synth.make_workload(name, device="cpu", n_layers=1)
            split = k3mla.batch_planned_split_tokens(wl0.ctx_len, MAX_CTX[name])
        run = Runner(name, split)
        ms_step, ms_dec = run.measure(steps, warmup)
        fig = run.figures(ms_step, ms_dec, hbm)
        fig["split_tokens"] = "auto" if split == 0 else split
        fig["layers"] = run.L
        fig["path"] = ("k3mla_decode_layer per layer-call" if run.fused else
                       "k3mla_absorb_q_append + k3mla_paged_decode per layer-call")
        if split_kind == "planned":
            fig["numerics"] = "batch-dependent (opt-in k3mla_batch_planned_split_tokens)"
        elif split_kind == "split512":
            fig["numerics"] = "batch-invariant (a fixed split length the caller chooses once)"
        res[name if split_kind == "auto" else f"{name}_{split_kind}"] = fig
        del run
        torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="steady64", choices=list(WORKLOAD_DESC))
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--no-next", action="store_true", help="skip the page-copy / chunked-prefill figures")
    ap.add_argument("--no-extra", action="store_true", help="skip the other workloads' figures")
    ap.add_argument("--split", type=int, default=0, help="split_tokens (0: the default per-slot rule)")
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling aid: fewer layers of the same per-layer workload")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        run_reference(args)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != 1 or world != 1:
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps({"metric": METRIC, "unavailable": "single-GPU build: the decode needs no "
                              "collective and runs as independent replicas only; no multi-GPU path is built"}))
        return

    from paged_latent_attention_k3mla_gb300 import k3mla
    torch.cuda.set_device(0)
    k3mla.load()
    hbm, tflops, src = peaks()
    run = Runner(args.workload, args.split, args.layers)
    wl, L, B = run.wl, run.L, run.B
    clk = Clocks()
    ms_step, ms_dec = run.measure(args.steps, args.warmup, clocks=clk)
    us_per_layer = ms_step * 1e3 / L
    e2e_ms, h2d, d2h, digest = e2e_leg(run, args.steps, args.warmup)
    nxt = None if args.no_next else next_rows(wl, run.table, run.max_ctx, run.stream, hbm, tflops, ms_dec * 1e3)
    ab = alg_bytes(wl)
    layer_gbs = ab["layer"] / (us_per_layer * 1e-6) / 1e9
    flops = alg_flops(wl)
    traffic = None
    prof = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if os.path.exists(prof):
        try:
            d = json.load(open(prof))
            if d.get("workload") == args.workload and d.get("kernel_rev") == kernel_rev():
                traffic = d.get("bytes_per_call")
        except (ValueError, OSError):
            traffic = None
    dec_gbs = ab["decode"] / (ms_dec * 1e-3) / 1e9
    roofline = {"kernel": "k3mla_paged_decode (split decode + merge/W_UV expansion)", "bound": "hbm",
                "achieved": round(dec_gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(dec_gbs / hbm, 4),
                "traffic": traffic, "alg_bytes_per_call": ab["decode"], "avg_call_us": round(ms_dec * 1e3, 3),
                "timing": f"{L} paged-decode calls in one CUDA graph, replayed; CUDA events on the launch "
                          f"stream; per call = graph time / {L}",
                "peak_source": f"{src} hbm_gbs"}
    cpu = None if args.no_cpu else cpu_baseline(wl)
    cfg = config_for(args.workload, wl, args.split, args.layers)
    del run, wl
    torch.cuda.empty_cache()
    extra = None if args.no_extra or args.layers is not None else extra_workloads(hbm, min(args.steps, 20), 3)
    line = {
        "metric": METRIC, "value": round(us_per_layer, 3), "unit": "us/layer-call", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": cfg,
        "latent_gbs": round(ab["latent"] / (us_per_layer * 1e-6) / 1e9, 1),
        "roofline": roofline,
        "layer_roofline": {"bound": "hbm", "achieved": round(layer_gbs, 1), "peak": hbm, "unit": "GB/s",
                           "frac": round(layer_gbs / hbm, 4), "alg_bytes_per_layer_call": ab["layer"],
                           "tensor_frac": round(flops / (us_per_layer * 1e-6) / 1e12 / tflops, 4),
                           "tensor_peak_tflops": tflops},
        "e2e": {"value": round(e2e_ms * 1e3 / L, 3), "unit": "us/layer-call", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * L * 3,   # per layer-call: absorption + append, split decode, merge/expansion
        "clocks": clk.summary(),
        "out_sha256_16": digest,
        "cpu_baseline": cpu,
        "workloads": extra,
        "next_rows": nxt,
    }
    print(json.dumps(line))


def _time_ms(fn, stream, warmup=2, reps=5):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def next_rows(wl, table, max_ctx, stream, hbm, tflops, absorbed_call_us):
    """Figures for the calls beyond the decode step, run after the timed step (they write the
    cache): a whole-page copy between two slabs (prefill adoption) against the HBM copy bandwidth,
    the causal attention of 64-token chunks of 16 slots at their 4096-token contexts, the
    exact-chain decode of one layer of the full batch, and the expanded-cache design (per-head K and
    V rows built from the latent, ordinary attention over them) on one layer of the full batch."""
    from paged_latent_attention_k3mla_gb300 import k3mla
    dev = "cuda"
    L = wl.n_layers
    n = 256
    dst = torch.empty(n, L, PAGE, ROW, dtype=torch.bfloat16, device=dev)
    src_ids = torch.arange(n, dtype=torch.int32, device=dev)
    dst_ids = torch.arange(n - 1, -1, -1, dtype=torch.int32, device=dev)
    ms = _time_ms(lambda: k3mla.copy_pages(dst, wl.slab, src_ids, dst_ids, stream=stream), stream, reps=20)
    moved = 2 * n * L * PAGE * ROW * 2                 # every page read once and written once
    gbs = moved / (ms * 1e-3) / 1e9
    res = {"copy_pages": {"pages": n, "layers": L, "ms": round(ms, 4), "achieved": round(gbs, 1), "peak": hbm,
                          "unit": "GB/s (read + write)", "frac": round(gbs / hbm, 4)}}
    del dst

    nb, T = 16, 64
    B = wl.B
    tbl = table[:nb].contiguous()
    pos0 = torch.from_numpy((wl.ctx_len[:nb] - T).astype(np.int32)).to(dev)
    row_start = torch.arange(0, nb * T + 1, T, dtype=torch.int32, device=dev)
    R = nb * T
    M = tbl.shape[1]
    vt = torch.empty(R, M, dtype=torch.int32, device=dev)
    vc = torch.empty(R, dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev).manual_seed(7)
    q = torch.randn(R, H, 192, generator=g, device=dev).to(torch.bfloat16)
    c = torch.randn(R, 512, generator=g, device=dev).to(torch.bfloat16)
    r = torch.randn(R, 64, generator=g, device=dev).to(torch.bfloat16)
    q_abs = torch.empty(R, H, ROW, dtype=torch.bfloat16, device=dev)
    split = k3mla.SPLIT_AUTO
    ws_v = torch.empty(k3mla.decode_workspace_bytes(R, max_ctx, split), dtype=torch.uint8, device=dev)
    ws = torch.empty(k3mla.chunk_decode_workspace_bytes(nb, R, max_ctx), dtype=torch.uint8, device=dev)
    out = torch.empty(R, H, V, dtype=torch.bfloat16, device=dev)
    out_v = torch.empty(R, H, V, dtype=torch.bfloat16, device=dev)

    def chunk_layer():  # multi-query: up to four token rows of a slot share each page load
        k3mla.append_latent_rows(wl.slab, 0, tbl, pos0, row_start, c, r, max_rows=T, stream=stream)
        k3mla.absorb_q(q, wl.w_kv_b[0], q_abs, stream=stream)
        k3mla.chunk_decode(q_abs, wl.slab, 0, tbl, pos0, row_start, wl.w_kv_b[0], wl.scale_bits, out, ws, max_ctx,
                           stream=stream)

    def chunk_layer_views():  # one view per token row, each streaming its slot's pages
        k3mla.append_latent_rows(wl.slab, 0, tbl, pos0, row_start, c, r, max_rows=T, stream=stream)
        k3mla.chunk_views(tbl, pos0, row_start, vt, vc, stream=stream)
        k3mla.absorb_q(q, wl.w_kv_b[0], q_abs, stream=stream)
        k3mla.paged_decode(q_abs, wl.slab, 0, vt, vc, wl.w_kv_b[0], wl.scale_bits, out_v, ws_v, max_ctx, split,
                           stream=stream)

    ms = _time_ms(chunk_layer, stream)
    ms_v = _time_ms(chunk_layer_views, stream)
    torch.cuda.synchronize()
    # every context here fits one split, so the two forms agree bit for bit
    same = bool(torch.equal(out.view(torch.int16), out_v.view(torch.int16)))
    # causal attention: token j of a chunk attends over pos0 + j + 1 tokens (scores 576 wide, latent
    # accumulation 512 wide, 96 heads), plus the absorption and the W_UV expansion of every token
    seen = int(sum(int(p0) * T + T * (T + 1) // 2 for p0 in (wl.ctx_len[:nb] - T)))
    flops = seen * H * 2 * (ROW + LORA) + 2 * 2 * R * H * NOPE * LORA
    tf = flops / (ms * 1e-3) / 1e12
    res["chunked_prefill"] = {"slots": nb, "chunk_tokens": T, "context_tokens": int(wl.ctx_len[:nb].max()),
                              "token_rows": R, "us_per_layer": round(ms * 1e3, 1),
                              "tokens_per_s_per_layer": round(R / (ms * 1e-3), 1),
                              "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": tflops,
                                           "unit": "TFLOP/s", "frac": round(tf / tflops, 4)},
                              "how": "row append + absorption + k3mla_chunk_decode (multi-query: up to four "
                                     "token rows of a slot share each page load, 32 heads of each)",
                              "views_us_per_layer": round(ms_v * 1e3, 1),
                              "views_tokens_per_s_per_layer": round(R / (ms_v * 1e-3), 1),
                              "views_how": "row append + per-token causal views + absorption + paged decode over "
                                           "the views (each view streams its slot's pages)",
                              "views_equal_bitwise": same}
    del ws_v, out_v
    del ws, out

    # exact-chain mode (absorption + decode, CUDA-core sequential sums) on the full batch of one layer
    ws = torch.empty(k3mla.decode_exact_workspace_bytes(B, max_ctx), dtype=torch.uint8, device=dev)
    out = torch.empty(B, H, V, dtype=torch.bfloat16, device=dev)
    ctx = torch.from_numpy(wl.ctx_len).to(dev)
    ms = _time_ms(lambda: k3mla.decode_exact(wl.q[0], wl.slab, 0, table, ctx, wl.w_kv_b[0], wl.scale_bits, out, ws,
                                             max_ctx, stream=stream), stream, warmup=1, reps=3)
    res["exact_chain"] = {"slots": B, "context_tokens": int(wl.ctx_len.max()), "us_per_layer": round(ms * 1e3, 1),
                          "how": "k3mla_decode_exact: the rounding chain's sums in order on CUDA cores, "
                                 "bitwise equal to the CPU oracle"}
    del ws, out
    torch.cuda.empty_cache()

    # the expanded-cache design, A/B: layer 0's per-head K (192) and V (128) rows for every page, then
    # ordinary attention over them; the cache (61,440 B a token) is far larger than L2
    n_pages = wl.slab.shape[0]
    x = torch.empty(n_pages, PAGE, H, XR, dtype=torch.bfloat16, device=dev)
    out = torch.empty(B, H, V, dtype=torch.bfloat16, device=dev)
    ms_build = _time_ms(lambda: k3mla.expand_latent_cache(wl.slab, 0, wl.w_kv_b[0], x, stream=stream), stream,
                        warmup=1, reps=3)
    ms_xd = _time_ms(lambda: k3mla.expanded_decode(wl.q[0], x, table, ctx, wl.scale_bits, out, max_ctx,
                                                   stream=stream), stream, warmup=2, reps=10)
    tokens = int(wl.ctx_len.sum())
    xd_bytes = tokens * H * XR * 2 + B * H * (192 + V) * 2      # K and V rows read, q read, out written
    xd_gbs = xd_bytes / (ms_xd * 1e-3) / 1e9
    build_bytes = n_pages * PAGE * (H * XR * 2 + ROW * 2)        # the cache written, each latent row read
    res["expanded_ab"] = {
        "layer": 0, "slots": B, "tokens": tokens, "cache_bytes": x.numel() * 2,
        "bytes_per_token_per_layer": H * XR * 2, "latent_bytes_per_token_per_layer": ROW * 2,
        "build_ms": round(ms_build, 3),
        "build_gbs": round(build_bytes / (ms_build * 1e-3) / 1e9, 1),
        "decode_us": round(ms_xd * 1e3, 1),
        "roofline": {"bound": "hbm", "achieved": round(xd_gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(xd_gbs / hbm, 4)},
        "absorbed_decode_call_us": round(absorbed_call_us, 3),
        "expanded_over_absorbed": round(ms_xd * 1e3 / absorbed_call_us, 2),
        "how": "k3mla_expand_latent_cache (tcgen05, W_UK / W_UV of a head x a page's latent) then "
               "k3mla_expanded_decode (a warp per slot and head, CUDA cores); absorbed figure: the "
               "paged-decode call timed above"}
    del x, out
    torch.cuda.empty_cache()
    return res


def kernel_rev() -> str:
    """Hash of the code (comments and blank space left out) of the paged-decode call: the split
    and merge kernels and what they include, so stored ncu traffic is only used for the kernels it
    measured."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "paged_latent_attention_k3mla_gb300", "csrc")
    for f in ("common.cuh", "decode.cu", "host_common.cu", "merge_expand.cu", "ptx.cuh"):
        src = open(os.path.join(d, f)).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:12]


if __name__ == "__main__":
    main()
