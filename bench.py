#!/usr/bin/env python3
"""Benchmark of the hybrid local/global GQA attention path on B300.

Workload ("full context"): 52 layers (39 local with a 2048-slot ring and
RoPE, 13 global), batch 1.  A 131072-token prompt is prefilled in
8192-token chunks through every layer (prefill + append), the 16-token
speculative verify runs against the 131072-token cache, then decode steps
run at positions 131072, 131073, ...  One timed step = one decode token
through all 52 layers (fused append + split-KV decode, then combine), replayed from a
CUDA graph of the C-ABI calls.  The headline value is decode attention HBM
throughput (algorithmic K/V + q/o bytes / time); prefill TFLOP/s and the
verify numbers are measured in the same run and reported beside it.

`--impl reference` times the fp64 CPU oracle (the reference arm) on a
bounded sample of the same decode workload.
"""
import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attn HBM GB/s (% of 8 TB/s) @128K; prefill attn TFLOP/s (% bf16 peak)"
PROMPT = 131072
CHUNK = 8192
N_LAYERS = 52
NOMINAL_HBM_GBS = 8000.0
KV_BYTES_PER_KEY = 1024          # K+V of one position, both KV heads, one layer
QO_BYTES_PER_TOKEN = 2 * 32 * 128 * 2  # q read + o written, one layer
PREFILL_FLOP_PER_PAIR = 4 * 128  # QK^T and PV, 2 flop per MAC, per (query head, key)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def max_over_ranks(x, device, world):
    """Largest value of x over all ranks: the job takes as long as its
    slowest rank.  world == 1 returns x unchanged."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, seconds, world):
    """Whole-job throughput: every rank processes units_per_rank (weak
    scaling, independent replicas) within the slowest rank's time."""
    return units_per_rank * world / seconds


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


def decode_layer_bytes(kind, p):
    keys = min(p + 1, 2048) if kind == 0 else p + 1
    return keys * KV_BYTES_PER_KEY + QO_BYTES_PER_TOKEN


def prefill_layer_flops(kind, c0, n):
    # sum over queries q in [c0, c0+n) of |key set of q|, times 32 heads
    if kind == 1:
        pairs = (c0 + n) * (c0 + n + 1) // 2 - c0 * (c0 + 1) // 2
    else:
        pairs = sum(min(q + 1, 2048) for q in range(c0, c0 + n))
    return pairs * 32 * PREFILL_FLOP_PER_PAIR


def verify_layer_bytes(kind, p0, n):
    keys = min(p0, 2047) + n if kind == 0 else p0 + n
    return keys * KV_BYTES_PER_KEY + n * QO_BYTES_PER_TOKEN


def verify_layer_flops(kind, p0, n):
    pairs = 0
    for i in range(n):
        q = p0 + i
        pairs += min(q + 1, 2048) if kind == 0 else q + 1
    return pairs * 32 * PREFILL_FLOP_PER_PAIR


class Clocks:
    """nvidia-smi sampling during a timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


def profile_traffic(kernel_file, profile_name, keys):
    """DRAM traffic of one launch over `keys` keys, from the per-key traffic
    a committed ncu summary measured (K/V traffic grows in proportion to the
    keys), if that summary was taken on the current kernel source (sha256
    recorded in the summary)."""
    src = os.path.join(ROOT, "hybrid_local_global_attn_b300", "csrc", kernel_file)
    prof = os.path.join(ROOT, "profiles", profile_name)
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        text = open(prof).read()
        m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
        m_tr = re.search(r"traffic_bytes_per_key:\s*([0-9.eE+]+)", text)
        if m_sha and m_tr and m_sha.group(1) == sha:
            return float(m_tr.group(1)) * keys
    except OSError:
        pass
    return None


# ------------------------------------------------------------- oracle arm ----
def oracle_decode_sample(budget_s, max_steps):
    """Time the fp64 oracle on decode steps of one global layer at context
    131072 (the dominant layer of the workload).  Returns (GB/s, info)."""
    import torch
    from hybrid_local_global_attn_b300 import synth
    from oracle import oracle as orc
    p = PROMPT
    k, v = synth.history(1, p + 1, 0, 3)
    q = synth.queries(1, max_steps, 0, 3)
    lay = orc.layer(orc.GLOBAL)
    kk, vv = orc.bits(k[0]), orc.bits(v[0])
    times = []
    t_start = time.perf_counter()
    for i in range(max_steps):
        t0 = time.perf_counter()
        orc.attention(lay, kk, vv, [p], q[:, i])
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > budget_s:
            break
    per = statistics.mean(times)
    nbytes = decode_layer_bytes(1, p)
    return nbytes / per / 1e9, {"steps_run": len(times), "s_per_step": per,
                                "threads": orc.threads(), "bytes_per_step": nbytes}


def run_reference(args, rank):
    if rank != 0:
        return 0
    from oracle import build as ob
    ob.build()
    budget = float(os.environ.get("MG_REF_BUDGET_S", "150"))
    gbs_w, info_w = oracle_decode_sample(min(20.0, budget / 4), max(args.warmup, 1))
    gbs, info = oracle_decode_sample(budget, max(args.steps, 1))
    sample = (f"fp64 oracle, decode of one token through one global layer at context 131072 "
              f"(all 32 heads, {info['bytes_per_step']} algorithmic bytes per step); "
              f"{info['steps_run']} of {args.steps} steps run within a {budget:.0f} s budget")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": info["s_per_step"] * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "full context decode at 131072 (oracle sample of the dominant "
                               "global layer)", "global_batch": 1, "seq_len": PROMPT},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": info["threads"],
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm ----
class Workload:
    """Device state of the 52-layer stack: caches, decode / verify inputs."""

    def __init__(self, args, dev, n_dec):
        import torch
        from hybrid_local_global_attn_b300 import mg
        self.mg, self.dev, self.n_dec = mg, dev, n_dec
        self.cap = PROMPT + max(n_dec, 16)
        self.kinds = [mg.mg_layer_kind(l) for l in range(N_LAYERS)]
        self.layers = [mg.make_layer(k) for k in self.kinds]
        self.caches = [mg.KVCache(k, 1, self.cap, device=dev) for k in self.kinds]
        self.err = mg.error_word(device=dev)
        self.gen = torch.Generator(device=dev)
        bf = torch.bfloat16
        self.dec_q = torch.empty((n_dec, N_LAYERS, 1, 32, 128), dtype=bf, device=dev)
        self.dec_k = torch.empty((n_dec, N_LAYERS, 1, 1, 2, 128), dtype=bf, device=dev)
        self.dec_v = torch.empty_like(self.dec_k)
        self.ver_q = torch.empty((N_LAYERS, 1, 16, 32, 128), dtype=bf, device=dev)
        self.ver_k = torch.empty((N_LAYERS, 1, 16, 2, 128), dtype=bf, device=dev)
        self.ver_v = torch.empty_like(self.ver_k)

    def randn(self, shape, seed):
        import torch
        self.gen.manual_seed(seed)
        return torch.randn(shape, generator=self.gen, device=self.dev,
                           dtype=torch.float32).to(torch.bfloat16)

    def layer_inputs(self, l, seed=0):
        """Prompt q/k/v of layer l (k/v extend past the prompt for decode)."""
        q = self.randn((1, PROMPT, 32, 128), 1000 * seed + 10 * l + 0)
        k = self.randn((1, PROMPT + self.n_dec, 2, 128), 1000 * seed + 10 * l + 1)
        v = self.randn((1, PROMPT + self.n_dec, 2, 128), 1000 * seed + 10 * l + 2)
        return q, k, v

    def keep_step_inputs(self, l, k, v, seed=0):
        self.dec_k[:, l, 0, 0] = k[0, PROMPT:PROMPT + self.n_dec]
        self.dec_v[:, l, 0, 0] = v[0, PROMPT:PROMPT + self.n_dec]
        self.dec_q[:, l, 0] = self.randn((self.n_dec, 32, 128), 1000 * seed + 10 * l + 5)
        self.ver_k[l, 0] = k[0, PROMPT:PROMPT + 16]
        self.ver_v[l, 0] = v[0, PROMPT:PROMPT + 16]
        self.ver_q[l, 0] = self.randn((16, 32, 128), 1000 * seed + 10 * l + 6)


def leg_prefill(wl, fill_only=False):
    """Prefill the prompt through every layer in 8192-token chunks (then
    append each chunk).  fill_only: write the cache directly (random
    contents, no attention) -- used only by profiling runs."""
    import torch
    mg, dev, err = wl.mg, wl.dev, wl.err
    ws = torch.empty(max(mg.mg_workspace_bytes(mg.OP_PREFILL, wl.layers[0], 1, CHUNK, PROMPT), 256),
                     dtype=torch.uint8, device=dev)
    o = torch.empty((1, CHUNK, 32, 128), dtype=torch.bfloat16, device=dev)
    pos_chunks = torch.arange(0, PROMPT, CHUNK, dtype=torch.int32, device=dev)
    if not fill_only:
        for k in (mg.LOCAL, mg.GLOBAL):  # warm-up into scratch caches
            scratch = mg.KVCache(k, 1, CHUNK, device=dev)
            qw, kw, vw = (wl.randn((1, CHUNK, 32, 128), 1), wl.randn((1, CHUNK, 2, 128), 2),
                          wl.randn((1, CHUNK, 2, 128), 3))
            for _ in range(3):
                mg.mg_attn_prefill(mg.make_layer(k), scratch, pos_chunks[:1], CHUNK, qw, kw, vw, o,
                                   ws, err)
            del scratch
    torch.cuda.synchronize()
    res = {"ms": 0.0, "flop": 0, "ms_k": {0: 0.0, 1: 0.0}, "flop_k": {0: 0, 1: 0}}
    clk = Clocks(dev.index)
    if not fill_only:
        clk.start()
    for l in range(N_LAYERS):
        kind = wl.kinds[l]
        q, k, v = wl.layer_inputs(l)
        if fill_only:
            for c0 in range(0, PROMPT, CHUNK):
                mg.mg_kv_append(wl.layers[l], wl.caches[l], pos_chunks[c0 // CHUNK:c0 // CHUNK + 1],
                                k[:, c0:c0 + CHUNK], v[:, c0:c0 + CHUNK], err)
        else:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for ci, c0 in enumerate(range(0, PROMPT, CHUNK)):
                kc, vc = k[:, c0:c0 + CHUNK], v[:, c0:c0 + CHUNK]
                mg.mg_attn_prefill(wl.layers[l], wl.caches[l], pos_chunks[ci:ci + 1], c0 + CHUNK,
                                   q[:, c0:c0 + CHUNK], kc, vc, o, ws, err)
                mg.mg_kv_append(wl.layers[l], wl.caches[l], pos_chunks[ci:ci + 1], kc, vc, err)
            e1.record()
            e1.synchronize()
            ms = e0.elapsed_time(e1)
            f = sum(prefill_layer_flops(kind, c0, CHUNK) for c0 in range(0, PROMPT, CHUNK))
            res["ms"] += ms
            res["flop"] += f
            res["ms_k"][kind] += ms
            res["flop_k"][kind] += f
        wl.keep_step_inputs(l, k, v)
        del q, k, v
    torch.cuda.synchronize()
    if not fill_only:
        res["clocks"] = clk.stop()
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x} after prefill"
    return res


def leg_verify_batches(wl, batches=(2, 8), reps=5):
    """The verify pass (16 draft tokens per sequence at p0 = 131072, all 52
    layers, one graph) at larger batches: caches of batch B filled with
    N(0, 1) values for positions 0 .. 131071 (the prompt's contents do not
    change the work), every sequence at the same position."""
    import torch
    mg, dev, err = wl.mg, wl.dev, wl.err
    res = {}
    for B in batches:
        caches = []
        for l in range(N_LAYERS):
            c = mg.KVCache(wl.kinds[l], B, PROMPT + 16, device=dev)
            c.k.normal_()
            c.v.normal_()
            caches.append(c)
        ws = [mg.workspace(mg.OP_VERIFY, wl.layers[l], B, 16, PROMPT + 16, device=dev)
              for l in range(N_LAYERS)]
        q = torch.randn((N_LAYERS, B, 16, 32, 128), device=dev).to(torch.bfloat16)
        kn = torch.randn((N_LAYERS, B, 16, 2, 128), device=dev).to(torch.bfloat16)
        vn = torch.randn_like(kn)
        o = torch.empty_like(q)
        p0 = torch.full((B,), PROMPT, dtype=torch.int32, device=dev)

        def run():
            for l in range(N_LAYERS):
                mg.mg_attn_verify(wl.layers[l], caches[l], p0, PROMPT + 16, q[l], kn[l], vn[l], o[l],
                                  ws[l], err)

        us = _graph_us(run, reps=reps)
        nbytes = B * sum(verify_layer_bytes(k, PROMPT, 16) for k in wl.kinds)
        flops = B * sum(verify_layer_flops(k, PROMPT, 16) for k in wl.kinds)
        res[f"b{B}"] = {"us_per_pass_52_layers": us, "gbs": nbytes / us / 1e3,
                        "tflops": flops / us / 1e6}
        del caches, ws, q, kn, vn, o
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x} after verify batches"
    return res


def leg_pr1(wl, P0=2000, steps=256):
    """The two-layer workload: one local (window 2048, RoPE) and one global
    layer, batch 1, caches filled for positions 0 .. P0-1, then `steps`
    single-token steps at P0, P0+1, ... (crossing the ring wrap at 2048),
    each an append of the token's K/V and a decode, in both layers.  The
    whole sequence of steps is one CUDA graph (so the host launch cost is
    not timed); reported per step, as two calls per layer (mg_kv_append +
    mg_attn_decode) and with the append fused (mg_append_decode)."""
    import torch
    mg, dev, err = wl.mg, wl.dev, wl.err
    T = P0 + steps
    kinds = (mg.LOCAL, mg.GLOBAL)
    layers = [mg.make_layer(k) for k in kinds]
    caches = [mg.KVCache(k, 1, T, device=dev) for k in kinds]
    pos0 = torch.zeros(1, dtype=torch.int32, device=dev)
    for c, lay in zip(caches, layers):
        mg.mg_kv_append(lay, c, pos0, wl.randn((1, P0, 2, 128), 7), wl.randn((1, P0, 2, 128), 8), err)
    ws = [mg.workspace(mg.OP_DECODE, lay, 1, 1, T, device=dev) for lay in layers]
    q = wl.randn((steps, 2, 1, 32, 128), 9)
    kn = wl.randn((steps, 2, 1, 1, 2, 128), 10)
    vn = wl.randn((steps, 2, 1, 1, 2, 128), 11)
    o = torch.empty((steps, 2, 1, 32, 128), dtype=torch.bfloat16, device=dev)
    pos = torch.arange(P0, T, dtype=torch.int32, device=dev)

    def separate():
        for i in range(steps):
            for j in range(2):
                mg.mg_kv_append(layers[j], caches[j], pos[i:i + 1], kn[i, j], vn[i, j], err)
                mg.mg_attn_decode(layers[j], caches[j], pos[i:i + 1], T, q[i, j], o[i, j], ws[j], err)

    def fused(early=False):
        for i in range(steps):
            for j in range(2):
                # MG_EARLY_START only: the steps follow each other in one
                # graph, and a layer's next step reads the row this one appends
                append_decode(mg.EARLY_START if early else 0, layers[j], caches[j], pos[i:i + 1], T,
                              q[i, j], kn[i, j], vn[i, j], o[i, j], ws[j], err)

    us_sep = _graph_us(separate, reps=5, calls=steps)
    us_fused = _graph_us(fused, reps=5, calls=steps)
    us_early = _graph_us(lambda: fused(True), reps=5, calls=steps)
    nbytes = sum(decode_layer_bytes(k, p) for p in range(P0, T) for k in kinds) / steps
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x} after PR1"
    del caches, ws, q, kn, vn, o
    torch.cuda.empty_cache()
    return {"positions": [P0, T - 1], "us_per_step_append_then_decode": us_sep,
            "us_per_step_fused": us_fused, "us_per_step_fused_early": us_early, "bytes_per_step": nbytes,
            "gbs_fused": nbytes / us_fused / 1e3}


def leg_prefill_32k(wl, T=32768, chunk=4096, reps=3):
    """Causal chunked prefill of a 32768-token prompt in 4096-token chunks
    (prefill each chunk, then append it), one global and one local layer,
    batch 1; TFLOP/s of the unmasked (query head, key) pairs."""
    import torch
    mg, dev, err = wl.mg, wl.dev, wl.err
    res = {"prompt": T, "chunk": chunk}
    for kind in (mg.GLOBAL, mg.LOCAL):
        lay = mg.make_layer(kind)
        cache = mg.KVCache(kind, 1, T, device=dev)
        q = wl.randn((1, T, 32, 128), 20 + kind)
        k = wl.randn((1, T, 2, 128), 22 + kind)
        v = wl.randn((1, T, 2, 128), 24 + kind)
        ws = mg.workspace(mg.OP_PREFILL, lay, 1, chunk, T, device=dev)
        o = torch.empty((1, chunk, 32, 128), dtype=torch.bfloat16, device=dev)
        pos = torch.arange(0, T, chunk, dtype=torch.int32, device=dev)

        def run():
            for ci, c0 in enumerate(range(0, T, chunk)):
                kc, vc = k[:, c0:c0 + chunk], v[:, c0:c0 + chunk]
                mg.mg_attn_prefill(lay, cache, pos[ci:ci + 1], c0 + chunk, q[:, c0:c0 + chunk], kc,
                                   vc, o, ws, err)
                mg.mg_kv_append(lay, cache, pos[ci:ci + 1], kc, vc, err)

        ms = _graph_us(run, reps=reps) / 1e3
        f = sum(prefill_layer_flops(kind, c0, chunk) for c0 in range(0, T, chunk))
        name = "global" if kind == mg.GLOBAL else "local"
        res[name] = {"ms": ms, "tflops": f / ms / 1e9, "flop": f}
        del cache, q, k, v, ws, o
        torch.cuda.empty_cache()
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x} after 32K prefill"
    return res


def leg_qkv(wl, reps=5):
    """The QKV projection with the KV append fused into its epilogue
    (mg_qkv_append): hidden 6656 -> 4608 features (32 q + 2 k + 2 v heads),
    weights N(0, 1/64^2) in bf16.  A prefill chunk of 8192 tokens (TFLOP/s of
    2 * M * 6656 * 4608) and decode of 1 and 16 tokens (GB/s of the 61 MB of
    weights every call streams, plus x and the outputs)."""
    import torch
    mg, dev, err = wl.mg, wl.dev, wl.err
    w = (wl.randn((4608, 6656), 31).float() / 64).to(torch.bfloat16)
    lay = mg.make_layer(mg.GLOBAL)
    res = {}
    for name, B, n in (("prefill_8192", 1, 8192), ("decode_b1", 1, 1), ("decode_b16", 16, 1)):
        cache = mg.KVCache(mg.GLOBAL, B, 8192 + 8, device=dev)
        x = wl.randn((B, n, 6656), 32)
        q = torch.empty((B, n, 32, 128), dtype=torch.bfloat16, device=dev)
        ws = mg.qkv_workspace(B, n, device=dev)
        pos = torch.full((B,), 0 if n > 1 else 8192, dtype=torch.int32, device=dev)
        us = _graph_us(lambda: mg.mg_qkv_append(lay, cache, pos, x, w, q, ws, err), reps=reps)
        flop = 2 * B * n * 6656 * 4608
        nbytes = 4608 * 6656 * 2 + B * n * (6656 + 4608) * 2
        res[name] = {"us": us, "tflops": flop / us / 1e6, "gbs": nbytes / us / 1e3}
        del cache, x, q, ws
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x} after qkv"
    return res


def leg_verify(wl):
    import torch
    mg, dev, err = wl.mg, wl.dev, wl.err
    ws = [mg.workspace(mg.OP_VERIFY, wl.layers[l], 1, 16, PROMPT + 16, device=dev)
          for l in range(N_LAYERS)]
    o = torch.empty((N_LAYERS, 1, 16, 32, 128), dtype=torch.bfloat16, device=dev)
    p0 = torch.tensor([PROMPT], dtype=torch.int32, device=dev)

    def one(l):
        mg.mg_attn_verify(wl.layers[l], wl.caches[l], p0, PROMPT + 16, wl.ver_q[l], wl.ver_k[l],
                          wl.ver_v[l], o[l], ws[l], err)

    for l in range(N_LAYERS):
        one(l)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for l in range(N_LAYERS):
            one(l)
    for _ in range(3):
        g.replay()
    reps = 10
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    e1.synchronize()
    ms = e0.elapsed_time(e1) / reps
    # the 13 global-layer verify calls back to back from one graph
    glob = [l for l in range(N_LAYERS) if wl.kinds[l] == mg.GLOBAL]
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2):
        for l in glob:
            one(l)
    g2.replay()
    e0.record()
    for _ in range(reps):
        g2.replay()
    e1.record()
    e1.synchronize()
    g_ms = e0.elapsed_time(e1) / (reps * len(glob))
    # speculative commit of the whole block (the anchor and 15 accepted
    # drafts) into all 52 caches, one call per layer, from one graph
    count = torch.full((1,), 16, dtype=torch.int32, device=dev)
    pos_next = torch.empty_like(p0)
    g3 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g3):
        for l in range(N_LAYERS):
            mg.mg_kv_commit(wl.layers[l], wl.caches[l], p0, count, wl.ver_k[l], wl.ver_v[l], err,
                            pos_next=pos_next)
    g3.replay()
    e0.record()
    for _ in range(reps):
        g3.replay()
    e1.record()
    e1.synchronize()
    c_ms = e0.elapsed_time(e1) / reps
    # the same commit into all 52 caches in one launch
    g4 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g4):
        mg.mg_kv_commit_layers(wl.layers, wl.caches, p0, count, wl.ver_k, wl.ver_v, err,
                               pos_next=pos_next)
    g4.replay()
    e0.record()
    for _ in range(reps):
        g4.replay()
    e1.record()
    e1.synchronize()
    c1_ms = e0.elapsed_time(e1) / reps
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x} after verify"
    assert int(pos_next.item()) == PROMPT + 16
    nbytes = sum(verify_layer_bytes(k, PROMPT, 16) for k in wl.kinds)
    flops = sum(verify_layer_flops(k, PROMPT, 16) for k in wl.kinds)
    return {"gbs": nbytes / ms / 1e6, "tflops": flops / ms / 1e9, "us_per_pass_52_layers": ms * 1e3,
            "global_layer_us": g_ms * 1e3,
            "global_layer_gbs": verify_layer_bytes(1, PROMPT, 16) / g_ms / 1e6,
            "global_layer_tflops": verify_layer_flops(1, PROMPT, 16) / g_ms / 1e9,
            "commit_us_52_layers": c1_ms * 1e3, "commit_us_52_layers_per_layer_calls": c_ms * 1e3}


def append_decode(flags, *args):
    """mg_append_decode (flags 0), or mg_append_decode_ex with the given flags."""
    from hybrid_local_global_attn_b300 import mg
    if flags:
        mg.mg_append_decode_ex(*args, flags)
    else:
        mg.mg_append_decode(*args)


def step_flags():
    """The flags of the calls of one decode step: every call's cache and
    position are written by no other call of the step (the positions are
    set before it), and consecutive steps are separate graph launches or
    have a position update between them, so each call may start loading
    under all the calls before it in the step."""
    from hybrid_local_global_attn_b300 import mg
    return mg.EARLY_START | mg.OVERLAP_NEXT


def _graph_us(fn, reps=8, calls=1):
    """Mean device time (us) of one of `calls` calls captured by fn into a graph."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    e1.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (reps * calls)


def leg_paged(wl, page_size=256):
    """Global layers through a paged cache.  (a, b) The full-context cache of
    one global layer copied into a pool of page_size-token pages in shuffled
    order; 13 decode and 13 verify calls from one graph, beside the same calls
    on that layer's linear cache.  (c) Four sequences of different lengths in
    one pool (pages handed out in shuffled order), decoded together, beside
    the same batch in a linear cache sized for the longest."""
    import torch
    mg, dev, err = wl.mg, wl.dev, wl.err
    ps = page_size
    rng = torch.Generator().manual_seed(5)
    l0 = next(l for l in range(N_LAYERS) if wl.kinds[l] == mg.GLOBAL)
    lin, lay = wl.caches[l0], wl.layers[l0]
    slots = (wl.cap + ps - 1) // ps * ps
    npg = slots // ps
    paged = mg.PagedKVCache(1, slots, npg, ps, device=dev)
    perm = torch.randperm(npg, generator=rng)
    paged.table[0] = perm.to(device=dev, dtype=torch.int32)
    for src, dst in ((lin.k, paged.k), (lin.v, paged.v)):
        full = torch.zeros((2, slots, 128), dtype=torch.bfloat16, device=dev)
        full[:, :wl.cap] = src[0]
        dst[perm.to(dev)] = full.view(2, npg, ps, 128).permute(1, 0, 2, 3)
        del full
    n_glob = sum(1 for k in wl.kinds if k == mg.GLOBAL)
    p = PROMPT - 1
    pos = torch.tensor([p], dtype=torch.int32, device=dev)
    q = wl.ver_q[l0][:, 0].contiguous()
    o = torch.empty((1, 32, 128), dtype=torch.bfloat16, device=dev)
    ws = mg.workspace(mg.OP_DECODE, lay, 1, 1, PROMPT, device=dev)
    res = {"page_size": ps}
    for name, cache in (("linear", lin), ("paged", paged)):
        us = _graph_us(lambda: [mg.mg_attn_decode(lay, cache, pos, PROMPT, q, o, ws, err)
                                for _ in range(n_glob)], calls=n_glob)
        res[f"decode_us_{name}"] = us
        res[f"decode_gbs_{name}"] = decode_layer_bytes(1, p) / us / 1e3
    p0 = torch.tensor([PROMPT], dtype=torch.int32, device=dev)
    wsv = mg.workspace(mg.OP_VERIFY, lay, 1, 16, PROMPT + 16, device=dev)
    ov = torch.empty((1, 16, 32, 128), dtype=torch.bfloat16, device=dev)
    for name, cache in (("linear", lin), ("paged", paged)):
        us = _graph_us(lambda: [mg.mg_attn_verify(lay, cache, p0, PROMPT + 16, wl.ver_q[l0],
                                                  wl.ver_k[l0], wl.ver_v[l0], ov, wsv, err)
                                for _ in range(n_glob)], calls=n_glob)
        res[f"verify_us_{name}"] = us
        res[f"verify_gbs_{name}"] = verify_layer_bytes(1, PROMPT, 16) / us / 1e3
    del paged
    # (c) a batch of different lengths sharing one pool
    lens = [PROMPT, PROMPT // 2, PROMPT // 4, PROMPT // 16]
    B = len(lens)
    need = [(n + ps - 1) // ps for n in lens]
    pool = mg.PagedKVCache(B, slots, sum(need), ps, device=dev)
    order = torch.randperm(sum(need), generator=rng).tolist()
    for b, m in enumerate(need):
        pool.table[b, :m] = torch.tensor(order[:m], dtype=torch.int32)
        del order[:m]
    pool.k.normal_()
    pool.v.normal_()
    linb = mg.KVCache(mg.GLOBAL, B, slots, device=dev)
    for b, n in enumerate(lens):
        kb, vb = pool.linear(b, n)
        linb.k[b, :, :n] = kb
        linb.v[b, :, :n] = vb
    posb = torch.tensor([n - 1 for n in lens], dtype=torch.int32, device=dev)
    qb = torch.randn((B, 32, 128), device=dev).to(torch.bfloat16)
    ob = torch.empty_like(qb)
    wsb = mg.workspace(mg.OP_DECODE, lay, B, 1, PROMPT, device=dev)
    nbytes = sum(decode_layer_bytes(1, n - 1) for n in lens)
    batch = {"lengths": lens, "pool_mib": pool.nbytes() / 2 ** 20,
             "linear_mib": linb.nbytes() / 2 ** 20}
    for name, cache in (("linear", linb), ("paged", pool)):
        us = _graph_us(lambda: [mg.mg_attn_decode(lay, cache, posb, PROMPT, qb, ob, wsb, err)
                                for _ in range(n_glob)], calls=n_glob)
        batch[f"decode_us_{name}"] = us
        batch[f"decode_gbs_{name}"] = nbytes / us / 1e3
    res["batch4_variable_length"] = batch
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x} after the paged leg"
    return res


def leg_e4m3(wl, steps=16):
    """Global layers from FP8 (e4m3) caches: each of the 13 global caches is
    quantised into its own FP8 cache (per-head scales 1.0: N(0,1) data sits
    well inside the e4m3 range), then (a) the 13 global decodes from one
    graph, (b) the whole 52-layer decode step with the global layers on
    FP8, beside the same graphs on the bf16 caches, and (c) that step with
    the decode leg's calls (fused append, the step flags)."""
    import torch
    mg, dev, err = wl.mg, wl.dev, wl.err
    glob = [l for l in range(N_LAYERS) if wl.kinds[l] == mg.GLOBAL]
    p_q = PROMPT - 1
    e4 = {}
    for l in glob:
        c = mg.E4M3KVCache(1, wl.cap, device=dev)
        src = wl.caches[l]
        for a in range(0, PROMPT, 16384):  # quantise through the library's append
            z = min(PROMPT, a + 16384)
            kn = src.k[0, :, a:z].permute(1, 0, 2).unsqueeze(0).contiguous()
            vn = src.v[0, :, a:z].permute(1, 0, 2).unsqueeze(0).contiguous()
            mg.mg_kv_append(wl.layers[l], c, torch.tensor([a], dtype=torch.int32, device=dev), kn, vn,
                            err)
        e4[l] = c
    torch.cuda.synchronize()
    pos = torch.tensor([p_q], dtype=torch.int32, device=dev)
    q = torch.randn((N_LAYERS, 1, 32, 128), device=dev).to(torch.bfloat16)
    o = torch.empty_like(q)
    ws = [mg.workspace(mg.OP_DECODE, wl.layers[l], 1, 1, PROMPT, device=dev) for l in range(N_LAYERS)]
    res = {"scales": "1.0 per KV head", "caches_mib": sum(c.nbytes() for c in e4.values()) / 2 ** 20}
    for name, caches in (("bf16", {l: wl.caches[l] for l in glob}), ("e4m3", e4)):
        us = _graph_us(lambda: [mg.mg_attn_decode(wl.layers[l], caches[l], pos, PROMPT, q[l], o[l],
                                                  ws[l], err) for l in glob], calls=len(glob))
        nbytes = (p_q + 1) * (KV_BYTES_PER_KEY if name == "bf16" else KV_BYTES_PER_KEY // 2) \
            + QO_BYTES_PER_TOKEN
        res[f"global_decode_us_{name}"] = us
        res[f"global_decode_gbs_{name}"] = nbytes / us / 1e3
    # the whole step: 39 local layers (bf16 ring) + 13 global layers
    for name in ("bf16", "e4m3"):
        caches = [e4[l] if (name == "e4m3" and l in e4) else wl.caches[l] for l in range(N_LAYERS)]
        us = _graph_us(lambda: [mg.mg_attn_decode(wl.layers[l], caches[l], pos, PROMPT, q[l], o[l],
                                                  ws[l], err) for l in range(N_LAYERS)])
        res[f"step_us_{name}"] = us
        res[f"tokens_per_s_{name}"] = 1e6 / us
    # (c) the step as the decode leg makes its calls: each layer appends the
    # token's own K/V (position PROMPT) and passes MG_EARLY_START |
    # MG_OVERLAP_NEXT (FP8 global layers honour the second flag only)
    kn = torch.randn((N_LAYERS, 1, 1, 2, 128), device=dev).to(torch.bfloat16)
    vn = torch.randn_like(kn)
    pos_n = torch.tensor([PROMPT], dtype=torch.int32, device=dev)
    ws_n = [mg.workspace(mg.OP_DECODE, wl.layers[l], 1, 1, PROMPT + 1, device=dev) for l in range(N_LAYERS)]
    for name in ("bf16", "e4m3"):
        caches = [e4[l] if (name == "e4m3" and l in e4) else wl.caches[l] for l in range(N_LAYERS)]
        us = _graph_us(lambda: [append_decode(step_flags(), wl.layers[l], caches[l], pos_n, PROMPT + 1, q[l],
                                              kn[l], vn[l], o[l], ws_n[l], err) for l in range(N_LAYERS)])
        res[f"step_us_fused_overlap_{name}"] = us
        res[f"tokens_per_s_fused_overlap_{name}"] = 1e6 / us
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x} after the e4m3 leg"
    del e4
    return res


def leg_sweep(wl, hbm_peak, ctx=32768, batches=(1, 4, 16), steps=128):
    """The decode sweep: one fused append + decode step through all 52 layers
    at context `ctx` for each batch size, from a CUDA graph (caches filled
    with N(0,1) values; every sequence at the same position).  GB/s of
    algorithmic bytes (K/V of each key set + q/o)."""
    import torch
    mg, dev, err = wl.mg, wl.dev, wl.err
    bf = torch.bfloat16
    res = {"context": ctx}
    for B in batches:
        cap = ctx + steps + 8
        layers = [mg.make_layer(mg.mg_layer_kind(l)) for l in range(N_LAYERS)]
        caches = []
        for l in range(N_LAYERS):
            c = mg.KVCache(mg.mg_layer_kind(l), B, cap, device=dev)
            c.k.normal_()
            c.v.normal_()
            caches.append(c)
        ws = [mg.workspace(mg.OP_DECODE, layers[l], B, 1, cap, device=dev) for l in range(N_LAYERS)]
        q = torch.randn((N_LAYERS, B, 32, 128), device=dev).to(bf)
        kn = torch.randn((N_LAYERS, B, 1, 2, 128), device=dev).to(bf)
        vn = torch.randn_like(kn)
        o = torch.empty_like(q)
        pos = torch.full((B,), ctx, dtype=torch.int32, device=dev)

        def step():
            for l in range(N_LAYERS):
                append_decode(step_flags(), layers[l], caches[l], pos, cap, q[l], kn[l], vn[l], o[l],
                              ws[l], err)

        step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(3):
            g.replay()
        e0.record()
        for i in range(steps):
            pos.fill_(ctx + i)  # positions ctx .. ctx + steps - 1
            g.replay()
        e1.record()
        e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / steps
        nbytes = B * sum(decode_layer_bytes(mg.mg_layer_kind(l), ctx + i) for l in range(N_LAYERS)
                         for i in range(steps)) / steps
        res[f"b{B}"] = {"us_per_step": us, "gbs": nbytes / us / 1e3,
                        "frac_of_measured_hbm": nbytes / us / 1e3 / hbm_peak,
                        "tokens_per_s": B * 1e6 / us}
        del caches, ws, q, kn, vn, o
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x} after the sweep"
    return res


def run_gpu(args, rank, world):
    import torch
    from hybrid_local_global_attn_b300 import mg

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    hbm_peak, tf_peak, tf_sus, peak_src = measured_peaks()
    W, K = args.warmup, args.steps
    legs = set(args.legs.split(","))
    wl = Workload(args, dev, n_dec=max(W + 2 * K, 16))  # warm-up, timed, then the e2e pass
    kinds, layers, caches, err, cap = wl.kinds, wl.layers, wl.caches, wl.err, wl.cap
    line_extra = {}

    pre = leg_prefill(wl, fill_only=(args.fill == "random" or "prefill" not in legs))
    if "prefill" in legs and args.fill != "random":
        line_extra["prefill"] = {
            "tflops": pre["flop"] / pre["ms"] / 1e9, "ms": pre["ms"], "flop": pre["flop"],
            "frac_of_bf16_peak": pre["flop"] / pre["ms"] / 1e9 / tf_peak,
            "frac_of_bf16_sustained": pre["flop"] / pre["ms"] / 1e9 / tf_sus if tf_sus else None,
            "global_tflops": pre["flop_k"][1] / pre["ms_k"][1] / 1e9,
            "local_tflops": pre["flop_k"][0] / pre["ms_k"][0] / 1e9,
            "global_ms": pre["ms_k"][1], "local_ms": pre["ms_k"][0], "clocks": pre["clocks"]}
        log("prefill: " + json.dumps(line_extra["prefill"]))
    if "verify" in legs:
        line_extra["verify"] = leg_verify(wl)
        log("verify: " + json.dumps(line_extra["verify"]))
    if "paged" in legs:
        line_extra["paged"] = leg_paged(wl)
        log("paged: " + json.dumps(line_extra["paged"]))
    if "e4m3" in legs:
        line_extra["e4m3"] = leg_e4m3(wl)
        log("e4m3: " + json.dumps(line_extra["e4m3"]))
    if "sweep" in legs:
        line_extra["decode_sweep"] = leg_sweep(wl, hbm_peak)
        log("sweep: " + json.dumps(line_extra["decode_sweep"]))
    if "verify_batches" in legs:
        line_extra["verify_batches"] = leg_verify_batches(wl)
        log("verify batches: " + json.dumps(line_extra["verify_batches"]))
    if "pr1" in legs:
        line_extra["pr1"] = leg_pr1(wl)
        log("pr1: " + json.dumps(line_extra["pr1"]))
    if "qkv" in legs:
        line_extra["qkv_projection"] = leg_qkv(wl)
        d = line_extra["qkv_projection"]
        d["prefill_8192"]["frac_of_bf16_peak"] = d["prefill_8192"]["tflops"] / tf_peak
        for nm in ("decode_b1", "decode_b16"):
            d[nm]["frac_of_measured_hbm"] = d[nm]["gbs"] / hbm_peak
        log("qkv: " + json.dumps(d))
    if "prefill32k" in legs:
        line_extra["prefill_32k"] = leg_prefill_32k(wl)
        for nm in ("global", "local"):
            d = line_extra["prefill_32k"][nm]
            d["frac_of_bf16_peak"] = d["tflops"] / tf_peak
            d["frac_of_bf16_sustained"] = d["tflops"] / tf_sus if tf_sus else None
        log("prefill 32k: " + json.dumps(line_extra["prefill_32k"]))

    # ------------------------------------------------------------- decode ----
    ws_dec = [mg.workspace(mg.OP_DECODE, layers[l], 1, 1, cap, device=dev) for l in range(N_LAYERS)]
    # One step's inputs (q, k, v of every layer and the position) are views
    # of one device buffer, so the end-to-end pass brings them in with a
    # single host-to-device copy.
    qb, kvb = N_LAYERS * 32 * 128 * 2, N_LAYERS * 2 * 128 * 2
    stage_bytes = qb + 2 * kvb + 16
    stage_dev = torch.zeros(stage_bytes, dtype=torch.uint8, device=dev)

    def stage_view(off, nbytes, dtype, shape):
        return stage_dev[off:off + nbytes].view(dtype).view(shape)

    q_cur = stage_view(0, qb, torch.bfloat16, (N_LAYERS, 1, 32, 128))
    k_cur = stage_view(qb, kvb, torch.bfloat16, (N_LAYERS, 1, 1, 2, 128))
    v_cur = stage_view(qb + kvb, kvb, torch.bfloat16, (N_LAYERS, 1, 1, 2, 128))
    pos_cur = stage_view(qb + 2 * kvb, 4, torch.int32, (1,))
    o_cur = torch.empty((N_LAYERS, 1, 32, 128), dtype=torch.bfloat16, device=dev)

    # No decode call of a step writes another call's cache or the position
    # (set before the step): the calls pass MG_EARLY_START | MG_OVERLAP_NEXT,
    # so each layer's cache loads start under the layers before it (the
    # plain-call step is timed too, below).
    def decode_step(early=True):
        for l in range(N_LAYERS):
            append_decode(step_flags() if early else 0, layers[l], caches[l], pos_cur, cap, q_cur[l],
                          k_cur[l], v_cur[l], o_cur[l], ws_dec[l], err)

    def stage(i):
        pos_cur.fill_(PROMPT + i)
        q_cur.copy_(wl.dec_q[i])
        k_cur.copy_(wl.dec_k[i])
        v_cur.copy_(wl.dec_v[i])

    stage(0)
    decode_step()  # eager once: TMA descriptors and kernel attributes get set up
    torch.cuda.synchronize()
    g_dec = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_dec):
        decode_step()
    # local layer: one ring kernel (append fused, splits merged in the
    # cluster); global layer: the split pass with the fused append, then the
    # combine kernel
    launches_per_step = sum(mg.mg_decode_kernel_count(layers[l], 1, cap) for l in range(N_LAYERS))
    # The device-timed steps replay one graph per step, captured over that
    # step's inputs where they already lie in HBM (q / k / v of every layer,
    # the position), so nothing but the 52 layers' kernels runs per step.
    pos_steps = torch.arange(PROMPT, PROMPT + W + K, dtype=torch.int32, device=dev)

    def decode_step_at(i, early=True):
        for l in range(N_LAYERS):
            append_decode(step_flags() if early else 0, layers[l], caches[l], pos_steps[i:i + 1], cap,
                          wl.dec_q[i, l],
                          wl.dec_k[i, l], wl.dec_v[i, l], o_cur[l], ws_dec[l], err)

    step_graphs = []
    for i in range(W + K):
        gi = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gi):
            decode_step_at(i)
        step_graphs.append(gi)
    for i in range(W):
        step_graphs[i].replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clk = Clocks(dev.index)
    clk.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(W, W + K):
        step_graphs[i].replay()
    e1.record()
    e1.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.stop()
    del step_graphs
    dec_ms = max_over_ranks(e0.elapsed_time(e1), dev, world)
    # the same steps through plain mg_append_decode calls (no early start)
    plain_graphs = []
    for i in range(W, W + K):
        gi = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gi):
            decode_step_at(i, early=False)
        plain_graphs.append(gi)
    plain_graphs[0].replay()
    torch.cuda.synchronize()
    e0.record()
    for gi in plain_graphs:
        gi.replay()
    e1.record()
    e1.synchronize()
    plain_us = e0.elapsed_time(e1) / K * 1e3
    del plain_graphs
    dec_bytes = sum(decode_layer_bytes(kinds[l], PROMPT + i) for i in range(W, W + K)
                    for l in range(N_LAYERS))
    gbs = job_throughput(dec_bytes, dec_ms / 1e3, world) / 1e9
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x} after decode"
    log(f"decode: {dec_ms / K * 1e3:.1f} us/step, {gbs:.1f} GB/s, clocks {clocks}")

    # ------------------------------------------ roofline: global decode pass ----
    # The 13 global-layer decode calls of the last timed step, as that step
    # makes them (fused append of the step's own token -- the same rows
    # again -- and the early start), back to back from one CUDA graph (so
    # host launch overhead is not timed), averaged over the launches; the
    # same pass through plain mg_attn_decode calls is timed beside it.
    glob = [l for l in range(N_LAYERS) if kinds[l] == mg.GLOBAL]
    i_last = W + K - 1
    p_last = PROMPT + i_last
    pos_r = pos_steps[i_last:i_last + 1]

    def roof_pass(early):
        for l in glob:
            if early:
                append_decode(step_flags(), layers[l], caches[l], pos_r, cap, wl.dec_q[i_last, l],
                              wl.dec_k[i_last, l], wl.dec_v[i_last, l], o_cur[l], ws_dec[l], err)
            else:
                mg.mg_attn_decode(layers[l], caches[l], pos_r, cap, wl.dec_q[i_last, l], o_cur[l],
                                  ws_dec[l], err)

    roof_ms = {}
    for early in (True, False):
        roof_pass(early)
        torch.cuda.synchronize()
        g_r = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_r):
            roof_pass(early)
        g_r.replay()
        reps = 8
        e0.record()
        for _ in range(reps):
            g_r.replay()
        e1.record()
        e1.synchronize()
        roof_ms[early] = e0.elapsed_time(e1) / (reps * len(glob))
        del g_r
    kern_ms = roof_ms[True]
    kern_bytes = decode_layer_bytes(1, p_last)
    achieved = kern_bytes / (kern_ms / 1e3) / 1e9
    achieved_plain = kern_bytes / (roof_ms[False] / 1e3) / 1e9
    traffic = profile_traffic("attn_decode.cu", "attn_decode_global_262k.md", p_last + 1)

    # ---------------------------------------------------------------- e2e ----
    # Inputs in pinned host memory; every step copies its inputs in, replays
    # the captured C-ABI calls and copies its outputs back to the host.  Each
    # step's inputs are packed as a device staging buffer lays them out, so
    # one copy per step brings them in.  Two staging / output buffers (and
    # one graph over each) let a copy stream bring step j+1's inputs in and
    # take step j's outputs out while step j+1 computes, as a serving loop
    # would; every step's copies are inside the timed region, which ends when
    # the last step's outputs are on the host.
    ee = K
    h_stage = torch.zeros((ee, stage_bytes), dtype=torch.uint8).pin_memory()
    for j, i in enumerate(range(W + K, W + K + ee)):
        h_stage[j, :qb] = wl.dec_q[i].cpu().contiguous().view(torch.uint8).reshape(-1)
        h_stage[j, qb:qb + kvb] = wl.dec_k[i].cpu().contiguous().view(torch.uint8).reshape(-1)
        h_stage[j, qb + kvb:qb + 2 * kvb] = wl.dec_v[i].cpu().contiguous().view(torch.uint8).reshape(-1)
        h_stage[j, qb + 2 * kvb:qb + 2 * kvb + 4] = torch.tensor([PROMPT + i], dtype=torch.int32).view(torch.uint8)
    h_o = torch.empty((ee, N_LAYERS, 1, 32, 128), dtype=torch.bfloat16).pin_memory()
    stage2 = [stage_dev, torch.zeros(stage_bytes, dtype=torch.uint8, device=dev)]
    out2 = [o_cur, torch.empty_like(o_cur)]
    graphs2 = [g_dec]
    with torch.cuda.graph(g2 := torch.cuda.CUDAGraph()):
        sd = stage2[1]
        q2 = sd[0:qb].view(torch.bfloat16).view(N_LAYERS, 1, 32, 128)
        k2 = sd[qb:qb + kvb].view(torch.bfloat16).view(N_LAYERS, 1, 1, 2, 128)
        v2 = sd[qb + kvb:qb + 2 * kvb].view(torch.bfloat16).view(N_LAYERS, 1, 1, 2, 128)
        p2 = sd[qb + 2 * kvb:qb + 2 * kvb + 4].view(torch.int32)
        for l in range(N_LAYERS):
            append_decode(step_flags(), layers[l], caches[l], p2, cap, q2[l], k2[l], v2[l], out2[1][l],
                          ws_dec[l], err)
    graphs2.append(g2)
    main = torch.cuda.current_stream()
    copy_s = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]
    ev_out = [torch.cuda.Event(), torch.cuda.Event()]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(copy_s):
        stage2[0].copy_(h_stage[0], non_blocking=True)
        ev_in[0].record(copy_s)
    for j in range(ee):
        s_ = j % 2
        if j + 1 < ee:  # the next step's inputs, once step j-1 has released that buffer
            with torch.cuda.stream(copy_s):
                if j >= 1:
                    copy_s.wait_event(ev_done[1 - s_])
                stage2[1 - s_].copy_(h_stage[j + 1], non_blocking=True)
                ev_in[1 - s_].record(copy_s)
        main.wait_event(ev_in[s_])
        if j >= 2:
            main.wait_event(ev_out[s_])  # step j-2's outputs have left this buffer
        graphs2[s_].replay()
        ev_done[s_].record(main)
        with torch.cuda.stream(copy_s):
            copy_s.wait_event(ev_done[s_])
            h_o[j].copy_(out2[s_], non_blocking=True)
            ev_out[s_].record(copy_s)
    copy_s.synchronize()
    main.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dev, world)
    e2e_bytes = sum(decode_layer_bytes(kinds[l], PROMPT + i) for i in range(W + K, W + K + ee)
                    for l in range(N_LAYERS))
    e2e_gbs = job_throughput(e2e_bytes, e2e_s, world) / 1e9
    h2d = stage_bytes
    d2h = N_LAYERS * 32 * 128 * 2
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x} after e2e"

    model_global = sum(mg.mg_cache_bytes(k, 1, PROMPT) for k in kinds if k == mg.GLOBAL)
    model_local = sum(mg.mg_cache_bytes(k, 1, PROMPT) for k in kinds if k == mg.LOCAL)
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": dec_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": "full context: 131072-token prompt prefilled in 8192-token chunks "
                        "through 52 layers (39 local ring w=2048 RoPE, 13 global), then one "
                        "decode token per step through all 52 layers, batch 1 per GPU",
            "global_batch": world, "seq_len": PROMPT, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2: 1.74 GB of K/V read per step",
            "decode_positions": [PROMPT + W, PROMPT + W + K - 1],
            "cache_fill": "prefill" if args.fill != "random" else "random (profiling run)"},
        "pct_of_8tbs": gbs / world / NOMINAL_HBM_GBS,
        "pct_of_measured_hbm": gbs / world / hbm_peak,
        "decode_calls": "mg_append_decode_ex with MG_EARLY_START | MG_OVERLAP_NEXT (a layer's cache loads start under the layers before it in the step)",
        "plain_calls_us_per_step": plain_us,
        "roofline": {"bound": "hbm", "kernel": "attn_decode (split-KV pass + combine), global "
                                              "layer at context 131072+",
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": peak_src,
                     "frac_nominal": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": kern_bytes, "ms_per_launch": kern_ms,
                     "calls": "as in the timed step (fused append, MG_EARLY_START | MG_OVERLAP_NEXT)",
                     "achieved_plain_calls": achieved_plain,
                     "ms_per_launch_plain_calls": roof_ms[False],
                     "traffic": traffic},
        **line_extra,
        "allocator": {"model_global_gib_at_131072": model_global / 2 ** 30,
                      "model_local_mib": model_local / 2 ** 20,
                      "allocated_global_gib": sum(c.nbytes() for c, k in zip(caches, kinds)
                                                  if k == mg.GLOBAL) / 2 ** 30,
                      "allocated_local_mib": sum(c.nbytes() for c, k in zip(caches, kinds)
                                                 if k == mg.LOCAL) / 2 ** 20,
                      "global_capacity_tokens": cap},
        "e2e": {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s / ee * 1e3},
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        gbs_cpu, info = oracle_decode_sample(float(os.environ.get("MG_CPU_BUDGET_S", "20")), 64)
        line["cpu_baseline"] = {
            "value": gbs_cpu, "unit": "GB/s", "cores": info["threads"], "kind": "oracle",
            "sample": f"fp64 oracle decode of one token through one global layer at context "
                      f"131072 ({info['steps_run']} tokens timed)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_micro():
    """Per-call cost of each entry point inside a CUDA graph of back-to-back
    calls (warm, launch gaps included): 39 local-layer decodes, 13
    global-layer decodes at 131072 keys, one-token appends.  Prints one JSON
    line; used to see where a decode step's time goes."""
    import torch
    from hybrid_local_global_attn_b300 import mg
    dev = torch.device("cuda", 0)
    err = mg.error_word()
    bf = torch.bfloat16
    T = PROMPT + 64
    out = {}

    def timed(fn, reps=20):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        e1.synchronize()
        return e0.elapsed_time(e1) / reps * 1e3  # us per graph

    for kind, n_layers, name in ((mg.LOCAL, 39, "local"), (mg.GLOBAL, 13, "global")):
        lay = mg.make_layer(kind)
        caches = [mg.KVCache(kind, 1, T) for _ in range(n_layers)]
        for c in caches:
            c.k.normal_()
            c.v.normal_()
        q = torch.randn((n_layers, 1, 32, 128), device=dev).to(bf)
        kn = torch.randn((n_layers, 1, 1, 2, 128), device=dev).to(bf)
        vn = torch.randn_like(kn)
        o = torch.empty_like(q)
        ws = [mg.workspace(mg.OP_DECODE, lay, 1, 1, T) for _ in range(n_layers)]
        pos = torch.tensor([PROMPT], dtype=torch.int32, device=dev)

        def dec():
            for l in range(n_layers):
                mg.mg_attn_decode(lay, caches[l], pos, T, q[l], o[l], ws[l], err)

        def appdec():
            for l in range(n_layers):
                mg.mg_append_decode(lay, caches[l], pos, T, q[l], kn[l], vn[l], o[l], ws[l], err)

        def app():
            for l in range(n_layers):
                mg.mg_kv_append(lay, caches[l], pos, kn[l], vn[l], err)

        out[f"{name}_decode_us"] = timed(dec) / n_layers
        out[f"{name}_append_decode_us"] = timed(appdec) / n_layers
        out[f"{name}_append_us"] = timed(app) / n_layers
        del caches
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x}"
    print(json.dumps(out), flush=True)
    return 0


def run_ncu_case(name):
    """Small, self-contained launches of one kernel for ncu captures: inputs
    larger than L2 where the kernel streams memory, a few GB at most."""
    import torch
    from hybrid_local_global_attn_b300 import mg
    dev = torch.device("cuda", 0)
    err = mg.error_word()
    bf = torch.bfloat16
    if name == "decode_global_e4m3":
        T = 262144  # 128 MB of FP8 K/V codes: larger than L2
        cache = mg.E4M3KVCache(1, T)
        cache.k.random_(0, 0x7E)  # finite codes
        cache.v.random_(0, 0x7E)
        lay = mg.make_layer(mg.GLOBAL)
        ws = mg.workspace(mg.OP_DECODE, lay, 1, 1, T)
        q = torch.randn((1, 32, 128), device=dev).to(bf)
        o = torch.empty_like(q)
        pos = torch.tensor([T - 1], dtype=torch.int32, device=dev)
        for _ in range(4):
            mg.mg_attn_decode(lay, cache, pos, T, q, o, ws, err)
    elif name in ("decode_global", "verify_global"):
        T = 262144  # 256 MB of K/V per layer
        cache = mg.KVCache(mg.GLOBAL, 1, T)
        cache.k.normal_()
        cache.v.normal_()
        lay = mg.make_layer(mg.GLOBAL)
        if name == "decode_global":
            ws = mg.workspace(mg.OP_DECODE, lay, 1, 1, T)
            q = torch.randn((1, 32, 128), device=dev).to(bf)
            o = torch.empty_like(q)
            pos = torch.tensor([T - 1], dtype=torch.int32, device=dev)
            for _ in range(4):
                mg.mg_attn_decode(lay, cache, pos, T, q, o, ws, err)
        else:
            n = 16
            ws = mg.workspace(mg.OP_VERIFY, lay, 1, n, T)
            q = torch.randn((1, n, 32, 128), device=dev).to(bf)
            kn = torch.randn((1, n, 2, 128), device=dev).to(bf)
            vn = torch.randn((1, n, 2, 128), device=dev).to(bf)
            o = torch.empty_like(q)
            pos = torch.tensor([T - n], dtype=torch.int32, device=dev)
            for _ in range(4):
                mg.mg_attn_verify(lay, cache, pos, T, q, kn, vn, o, ws, err)
    elif name in ("decode_local", "verify_local", "decode_local_b16", "verify_local_b8"):
        # one local layer at context 131072 (a full 2048-slot ring), batch 1;
        # batch 16 (decode) and 8 (verify) run the kernels whose CTAs walk
        # their ring piece in rounds
        T = 131072
        B = 16 if name == "decode_local_b16" else 8 if name == "verify_local_b8" else 1
        cache = mg.KVCache(mg.LOCAL, B, T + 16)
        cache.k.normal_()
        cache.v.normal_()
        lay = mg.make_layer(mg.LOCAL)
        n = 1 if name.startswith("decode") else 16
        op = mg.OP_DECODE if n == 1 else mg.OP_VERIFY
        ws = mg.workspace(op, lay, B, n, T + 16)
        q = torch.randn((B, n, 32, 128), device=dev).to(bf)
        kn = torch.randn((B, n, 2, 128), device=dev).to(bf)
        vn = torch.randn((B, n, 2, 128), device=dev).to(bf)
        o = torch.empty_like(q)
        pos = torch.full((B,), T, dtype=torch.int32, device=dev)
        for _ in range(4):
            if n == 1:
                mg.mg_append_decode(lay, cache, pos, T + 16, q[:, 0], kn, vn, o[:, 0], ws, err)
            else:
                mg.mg_attn_verify(lay, cache, pos, T + 16, q, kn, vn, o, ws, err)
    elif name in ("prefill_global", "prefill_local"):
        kind = mg.GLOBAL if name == "prefill_global" else mg.LOCAL
        c0, n = 28672, 4096  # last 4096-token chunk of a 32768-token prompt
        cache = mg.KVCache(kind, 1, c0 + n)
        cache.k.normal_()
        cache.v.normal_()
        lay = mg.make_layer(kind)
        ws = mg.workspace(mg.OP_PREFILL, lay, 1, n, c0 + n)
        q = torch.randn((1, n, 32, 128), device=dev).to(bf)
        kn = torch.randn((1, n, 2, 128), device=dev).to(bf)
        vn = torch.randn((1, n, 2, 128), device=dev).to(bf)
        o = torch.empty_like(q)
        pos = torch.tensor([c0], dtype=torch.int32, device=dev)
        for _ in range(4):
            mg.mg_attn_prefill(lay, cache, pos, c0 + n, q, kn, vn, o, ws, err)
    elif name in ("qkv_prefill", "qkv_decode"):
        # the fused projection: an 8192-token chunk (x 109 MB + W 61 MB, more
        # than L2), or one decode token (W streamed from HBM)
        n = 8192 if name == "qkv_prefill" else 1
        lay = mg.make_layer(mg.GLOBAL)
        cache = mg.KVCache(mg.GLOBAL, 1, 8192 + 8)
        w = (torch.randn((4608, 6656), device=dev) / 64).to(bf)
        x = torch.randn((1, n, 6656), device=dev).to(bf)
        q = torch.empty((1, n, 32, 128), dtype=bf, device=dev)
        ws = mg.qkv_workspace(1, n)
        pos = torch.tensor([0 if n > 1 else 8192], dtype=torch.int32, device=dev)
        for _ in range(4):
            mg.mg_qkv_append(lay, cache, pos, x, w, q, ws, err)
    elif name in ("append_chunk", "commit_layers"):
        if name == "append_chunk":  # an 8192-token chunk into a global cache (16 MB moved)
            lay = mg.make_layer(mg.GLOBAL)
            cache = mg.KVCache(mg.GLOBAL, 1, 131072)
            kn = torch.randn((1, 8192, 2, 128), device=dev).to(bf)
            vn = torch.randn_like(kn)
            pos = torch.tensor([65536], dtype=torch.int32, device=dev)
            for _ in range(4):
                mg.mg_kv_append(lay, cache, pos, kn, vn, err)
        else:  # a verified 16-token block into all 52 caches in one launch
            layers = [mg.make_layer(mg.mg_layer_kind(l)) for l in range(52)]
            caches = [mg.KVCache(mg.mg_layer_kind(l), 1, 4096) for l in range(52)]
            kn = torch.randn((52, 1, 16, 2, 128), device=dev).to(bf)
            vn = torch.randn_like(kn)
            pos = torch.tensor([3000], dtype=torch.int32, device=dev)
            cnt = torch.tensor([11], dtype=torch.int32, device=dev)
            for _ in range(4):
                mg.mg_kv_commit_layers(layers, caches, pos, cnt, kn, vn, err)
    else:
        raise SystemExit(f"unknown ncu case {name}")
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error word {int(err.item()):#x}"
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="mg", choices=["mg", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--legs",
                    default="prefill,verify,paged,e4m3,sweep,verify_batches,pr1,prefill32k,qkv,decode",
                    help="comma list of legs to run besides decode")
    ap.add_argument("--fill", default="prefill", choices=["prefill", "random"],
                    help="random: fill caches without attention (profiling runs only)")
    ap.add_argument("--ncu-case", default=None,
                    help="decode_global | decode_global_e4m3 | verify_global | decode_local | verify_local | "
                         "decode_local_b16 | verify_local_b8 | "
                         "prefill_global | prefill_local | qkv_prefill | qkv_decode | append_chunk | "
                         "commit_layers")
    ap.add_argument("--micro", action="store_true",
                    help="per-call cost of each entry point in graphs of back-to-back calls")
    args = ap.parse_args()
    if args.micro:
        return run_micro()
    if args.ncu_case:
        return run_ncu_case(args.ncu_case)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    try:
        return run_gpu(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
