"""Benchmark: decode attention on the packed TurboQuant KV cache (+ quantize-append).

Workload (one step): Llama-3-8B-shaped GQA decode -- batch 16, 32 query / 8 KV
heads, head_dim 128, 32 layers, context 8192 (+1 token per step), bf16 K/V with
per-(head, channel) lognormal(0, 1) scales, 4-bit keys and values with fp32
norms, Hadamard rotation per layer, paged 16-token blocks under a shuffled block
table.  A step appends one new token per sequence to every layer (quantize-
append) and runs decode attention over every layer: one tq_decode_step call per
layer, whose decode kernel quantizes the new token itself.  All inputs are synthetic
and already resident in HBM; one step reads ~4.6 GB of packed cache, more
than L2, so no flush is needed between steps.

Reported: value = packed K/V bytes read by decode per step / step time (GB/s);
roofline for the decode call; quantize-append vectors/s from the prefill and
from the dense-rotation burst (36 layers x 11,000 tokens); decode GB/s of a
k8v4 layer (FP8 keys, 4-bit values) and the PolarQuant variant's append and
decode (4-bit angles, fp16 radius) at the same shape; decode GB/s at the
long-context shape (4 x 131,072 tokens, groups of 8, 3/4 bits); e2e through the public
API with host buffers; the oracle's CPU throughput.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tq|reference]
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

B, HQ, HKV, D, T0, LAYERS = 16, 32, 8, 128, 8192, 32
BLOCK = 16
SPLITS = 0  # decode context splits; 0 lets the library choose
BYTES_PER_TOKEN_HEAD = 2 * (D * 4 // 8 + 4)  # 4-bit K and V records + two fp32 norms = 136 B
APPEND_BYTES_PER_VECTOR = 2 * D + (D * 4 // 8 + 4)  # bf16 read + record written
METRIC = "decode-attn packed-KV GB/s"
WORKLOAD = "llama3-8b-shaped GQA decode, B16 Hq32 Hkv8 d128 ctx8192, 32 layers, 4-bit K/V, Hadamard"


def job_ms(ms_local, device=None):
    """The job's timed-region length in ms: the maximum over ranks (the job ends with
    its slowest rank); a single process returns its own."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(ms_local)
    t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank, world, ms_total):
    """Whole-job throughput (units per second): the units all ranks processed (each
    rank runs an independent replica of the same work) over the job's time."""
    return units_per_rank * world / (ms_total * 1e-3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "tq_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
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
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- GPU setup

def setup(torch, tq, steps_total, dev):
    """Per-layer caches filled with 8192 prefilled tokens; returns state dict."""
    mb = (T0 + steps_total + BLOCK - 1) // BLOCK + 1
    nb = B * mb
    import numpy as np
    import workloads
    bt_np, _ = workloads.shuffled_block_table(1234, B, mb, num_blocks=nb)
    bt = torch.from_numpy(bt_np).to(dev)
    gen = torch.Generator(device=dev).manual_seed(2024)
    sk = torch.exp(torch.randn(HKV, D, generator=gen, device=dev))
    sv = torch.exp(torch.randn(HKV, D, generator=gen, device=dev))
    kpre = (torch.randn(B * T0, HKV, D, generator=gen, device=dev) * sk).to(torch.bfloat16)
    vpre = (torch.randn(B * T0, HKV, D, generator=gen, device=dev) * sv).to(torch.bfloat16)
    slots_pre = torch.from_numpy(workloads.prefill_slots(bt_np, T0)).to(dev)
    layers = [tq.Layer(nb, HKV, bits_k=4, bits_v=4, seed=0, layer=l, device=dev) for l in range(LAYERS)]
    # prefill (timed: quantize-append throughput on 2 x 1,048,576 vectors per layer)
    for l in range(min(2, LAYERS)):  # untimed first appends
        layers[l].append(kpre, vpre, slots_pre)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(LAYERS)]
    for l in range(LAYERS):
        ev[l][0].record()
        layers[l].append(kpre, vpre, slots_pre)
        ev[l][1].record()
    torch.cuda.synchronize()
    append_ms = [a.elapsed_time(b) for a, b in ev]
    n_vec = 2 * B * T0 * HKV
    # a sample of the prefill keys and their slots (layer 0), for the tie-band report
    tie_tok = 2048
    tie_x = kpre[:tie_tok].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    tie_slots = slots_pre[:tie_tok].cpu().numpy()
    del kpre, vpre
    q = [torch.randn(B, HQ, D, generator=gen, device=dev).to(torch.bfloat16) for _ in range(LAYERS)]
    knew = [torch.randn(B, HKV, D, generator=gen, device=dev).to(torch.bfloat16) for _ in range(LAYERS)]
    vnew = [torch.randn(B, HKV, D, generator=gen, device=dev).to(torch.bfloat16) for _ in range(LAYERS)]
    out = [torch.empty(B, HQ, D, dtype=torch.bfloat16, device=dev) for _ in range(LAYERS)]
    ctx = torch.full((B,), T0, dtype=torch.int32, device=dev)
    slot_new = torch.empty(B, dtype=torch.int64, device=dev)
    ws_bytes = layers[0].workspace_bytes(B, HQ, mb, SPLITS)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)  # zero before first use
    return dict(tie_x=tie_x, tie_slots=tie_slots,
                layers=layers, bt=bt, bt_np=bt_np, mb=mb, nb=nb, q=q, knew=knew, vnew=vnew, out=out, ctx=ctx,
                slot_new=slot_new, ws=ws, append_ms=append_ms, append_vectors=n_vec)


def dense_workload(torch, tq, dev, peak, decode_steps=256):
    """The dense-rotation workload: 36 layers x 8 KV heads x 11,000 prefilled bf16
    tokens, K and V scaled by a per-layer lambda ~ U(0.5, 4), a dense Haar rotation
    per layer, 4-bit codes.

    Burst append: 6,336,000 vectors in one batched call (tq_quantize_append_layers);
    one untimed burst, then one timed with CUDA events around the call (1.6 GB of
    inputs: larger than L2).
    Decode phase: `decode_steps` incremental steps at batch 1 with 32 query heads;
    a step appends one new token to every layer and decodes every layer
    (tq_append_decode per layer, the step captured as one CUDA graph), reading
    36 x 8 x ctx x 136 B of packed cache (~431 MB per step, above L2); timed with
    CUDA events around all steps."""
    import workloads
    n_layers, n_tok = 36, 11000
    lam = workloads.layer_scales(36, n_layers)
    gen = torch.Generator(device=dev).manual_seed(36)
    nb = (n_tok + decode_steps + 8 + BLOCK - 1) // BLOCK + 1
    layers = [tq.Layer(nb, HKV, bits_k=4, bits_v=4, rot_kind=tq.TQ_ROT_DENSE, seed=36, layer=l, device=dev)
              for l in range(n_layers)]
    ks = [(torch.randn(n_tok, HKV, D, generator=gen, device=dev) * float(lam[l])).to(torch.bfloat16)
          for l in range(n_layers)]
    vs = [(torch.randn(n_tok, HKV, D, generator=gen, device=dev) * float(lam[l])).to(torch.bfloat16)
          for l in range(n_layers)]
    slots = torch.arange(n_tok, dtype=torch.int64, device=dev)
    tq.append_layers(layers, ks, vs, slots)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = tq.launch_count()
    e0.record()
    tq.append_layers(layers, ks, vs, slots)  # one batched append of all 36 layers
    e1.record()
    torch.cuda.synchronize()
    launches = tq.launch_count() - n0
    ms = e0.elapsed_time(e1)
    n_vec = 2 * n_layers * n_tok * HKV
    gbs = n_vec * APPEND_BYTES_PER_VECTOR / (ms * 1e-3) / 1e9
    status = tq.get_device_status()
    del ks, vs
    burst = {"workload": "36 layers x 8 KV heads x 11000 tokens, bf16 K and V, dense Haar rotation per layer, 4-bit",
             "vectors": n_vec, "ms": round(ms, 4), "vectors_per_s": round(n_vec / (ms * 1e-3), 1),
             "gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "bytes_per_vector": APPEND_BYTES_PER_VECTOR,
             "gpu_launches": launches, "device_status": status}

    # decode phase: batch 1, one block table (the identity: the burst filled slots 0..n_tok-1)
    hq = 32
    bt = torch.arange(nb, dtype=torch.int32, device=dev).reshape(1, nb)
    ctx = torch.full((1,), n_tok, dtype=torch.int32, device=dev)
    slot = torch.empty(1, dtype=torch.int64, device=dev)
    q = [torch.randn(1, hq, D, generator=gen, device=dev).to(torch.bfloat16) for _ in range(n_layers)]
    kn = [(torch.randn(1, HKV, D, generator=gen, device=dev) * float(lam[l])).to(torch.bfloat16)
          for l in range(n_layers)]
    vn = [(torch.randn(1, HKV, D, generator=gen, device=dev) * float(lam[l])).to(torch.bfloat16)
          for l in range(n_layers)]
    out = [torch.empty(1, hq, D, dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
    ws = torch.zeros(layers[0].workspace_bytes(1, hq, nb), dtype=torch.uint8, device=dev)

    def step():
        slot.copy_(ctx.to(torch.int64))  # identity table: the new token's slot is its position
        ctx.add_(1)
        for l in range(n_layers):
            layers[l].append_decode(kn[l], vn[l], slot, q[l], bt, ctx, out=out[l], workspace=ws)

    for l in range(n_layers):  # eager warm-up before capture
        layers[l].decode(q[l], bt, ctx, out=out[l], workspace=ws)
    torch.cuda.synchronize()
    ctx0 = ctx.clone()
    g = torch.cuda.CUDAGraph()
    n0 = tq.launch_count()
    with torch.cuda.graph(g):
        step()
    per_step_launches = tq.launch_count() - n0
    ctx.copy_(ctx0)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    c_start = int(ctx[0].item())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(decode_steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    dms = e0.elapsed_time(e1)
    nbytes = sum(n_layers * HKV * (c_start + i + 1) * BYTES_PER_TOKEN_HEAD for i in range(decode_steps))
    dgbs = nbytes / (dms * 1e-3) / 1e9
    dec = {"workload": "36 dense-rotation layers x 8 KV heads x ~11000 tokens, batch 1, 32 query heads, %d "
                       "incremental steps (append + decode of every layer per step, CUDA graph)" % decode_steps,
           "steps": decode_steps, "bytes_per_step": nbytes // decode_steps, "ms_per_step": round(dms / decode_steps, 4),
           "gbs": round(dgbs, 1), "frac": round(dgbs / peak, 4), "gpu_launches": per_step_launches * decode_steps,
           "device_status": tq.get_device_status()}
    del layers, ws, q, kn, vn, out
    torch.cuda.empty_cache()
    return burst, dec


def mixed62(torch, tq, dev, peak, steps=6):
    """The mixed-precision cache: 62 layers where layers 0, 1, 60 and 61 keep bf16 K/V
    and the other 58 hold 4-bit TurboQuant codes, 8 KV heads, batch 8, 32 query
    heads, 100,000-token contexts (bf16 N(0, 1) inputs, identity block tables).  A
    step appends one token per sequence to every layer and decodes every layer
    (tq_append_decode per layer, one CUDA graph): 58 x 870.4 MB + 4 x 3.277 GB =
    63.6 GB of cache read per step.  Also one layer of the QJL variant (2-bit keys
    + 1-bit QJL residual, 4-bit values: 124 B per token and KV head, ~793.6 MB)
    timed alone.  CUDA events around all steps / calls."""
    n_layers, b8, hq, t = 62, 8, 32, 100000
    bf16_ids = (0, 1, 60, 61)
    gen = torch.Generator(device=dev).manual_seed(62)
    mb = (t + steps + 8 + BLOCK - 1) // BLOCK + 1
    nb = b8 * mb
    bt = torch.arange(nb, dtype=torch.int32, device=dev).reshape(b8, mb)
    slots_pre = (torch.arange(b8, device=dev, dtype=torch.int64)[:, None] * (mb * BLOCK)
                 + torch.arange(t, device=dev, dtype=torch.int64)[None, :]).reshape(-1)
    layers = []
    for l in range(n_layers):
        if l in bf16_ids:
            layers.append(tq.Layer(nb, HKV, kv_format="bf16", device=dev))
        else:
            layers.append(tq.Layer(nb, HKV, bits_k=4, bits_v=4, seed=62, layer=l, device=dev))
    chunk = 1 << 18  # tokens per append call (bf16 inputs of 512 MB for K and V)
    for i0 in range(0, b8 * t, chunk):
        sl = slots_pre[i0:i0 + chunk]
        k = torch.randn(sl.numel(), HKV, D, generator=gen, device=dev).to(torch.bfloat16)
        v = torch.randn(sl.numel(), HKV, D, generator=gen, device=dev).to(torch.bfloat16)
        for layer in layers:  # the same tokens in every layer (different rotations per layer)
            layer.append(k, v, sl)
        del k, v
    torch.cuda.synchronize()
    ctx = torch.full((b8,), t, dtype=torch.int32, device=dev)
    slot = torch.empty(b8, dtype=torch.int64, device=dev)
    q = [torch.randn(b8, hq, D, generator=gen, device=dev).to(torch.bfloat16) for _ in range(n_layers)]
    kn = torch.randn(b8, HKV, D, generator=gen, device=dev).to(torch.bfloat16)
    vn = torch.randn(b8, HKV, D, generator=gen, device=dev).to(torch.bfloat16)
    out = [torch.empty(b8, hq, D, dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
    ws = torch.zeros(max(layer.workspace_bytes(b8, hq, mb) for layer in layers), dtype=torch.uint8, device=dev)
    row0 = torch.arange(b8, device=dev, dtype=torch.int64) * (mb * BLOCK)

    def step():
        slot.copy_(row0 + ctx.to(torch.int64))
        ctx.add_(1)
        for l in range(n_layers):
            layers[l].append_decode(kn, vn, slot, q[l], bt, ctx, out=out[l], workspace=ws)

    for l in range(n_layers):
        layers[l].decode(q[l], bt, ctx, out=out[l], workspace=ws)
    torch.cuda.synchronize()
    ctx0 = ctx.clone()
    g = torch.cuda.CUDAGraph()
    n0 = tq.launch_count()
    with torch.cuda.graph(g):
        step()
    per_step_launches = tq.launch_count() - n0
    ctx.copy_(ctx0)
    g.replay()
    torch.cuda.synchronize()
    c_start = int(ctx[0].item())
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    per_tok = 58 * BYTES_PER_TOKEN_HEAD + 4 * 2 * D * 2  # bytes per token and KV head over all layers
    nbytes = sum(b8 * HKV * (c_start + i + 1) * per_tok for i in range(steps))
    gbs = nbytes / (ms * 1e-3) / 1e9
    res = {"workload": "62 layers (0, 1, 60, 61 bf16; 58 x 4-bit), B8 Hq32 Hkv8 d128 ctx100000, append + decode "
                       "of every layer per step (CUDA graph)", "steps": steps, "bytes_per_step": nbytes // steps,
           "ms_per_step": round(ms / steps, 4), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
           "gpu_launches": per_step_launches * steps, "device_status": tq.get_device_status()}
    del layers, out, q
    torch.cuda.empty_cache()

    # one layer of the QJL variant: 2-bit keys + QJL residual, 4-bit values
    layer = tq.Layer(nb, HKV, bits_k=2, bits_v=4, qjl=True, seed=62, layer=2, device=dev)
    for i0 in range(0, b8 * t, chunk):
        sl = slots_pre[i0:i0 + chunk]
        k = torch.randn(sl.numel(), HKV, D, generator=gen, device=dev).to(torch.bfloat16)
        v = torch.randn(sl.numel(), HKV, D, generator=gen, device=dev).to(torch.bfloat16)
        layer.append(k, v, sl)
        del k, v
    ctx.fill_(t)
    qq = torch.randn(b8, hq, D, generator=gen, device=dev).to(torch.bfloat16)
    oo = torch.empty(b8, hq, D, dtype=torch.bfloat16, device=dev)
    wq = torch.zeros(layer.workspace_bytes(b8, hq, mb), dtype=torch.uint8, device=dev)
    for _ in range(3):
        layer.decode(qq, bt, ctx, out=oo, workspace=wq)
    torch.cuda.synchronize()
    ms_q = []
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        layer.decode(qq, bt, ctx, out=oo, workspace=wq)
        e1.record()
        torch.cuda.synchronize()
        ms_q.append(e0.elapsed_time(e1))
    mq = statistics.median(ms_q)
    qbytes = b8 * HKV * t * (D * 2 // 8 + 4 + D // 8 + 4 + D * 4 // 8 + 4)
    res["qjl_layer"] = {"workload": "one layer, 2-bit keys + 1-bit QJL residual (m = 128), 4-bit values, B8 Hq32 "
                                    "Hkv8 ctx100000", "bytes": qbytes, "ms": round(mq, 4),
                        "gbs": round(qbytes / (mq * 1e-3) / 1e9, 1),
                        "frac": round(qbytes / (mq * 1e-3) / 1e9 / peak, 4), "device_status": tq.get_device_status()}
    del layer, wq
    torch.cuda.empty_cache()
    return res


def decode_k8v4(torch, tq, dev, peak, reps=20):
    """Decode on a k8v4 layer (FP8 E4M3 keys, 4-bit TurboQuant values) at the headline
    shape (batch 16, 32/8 heads, context 8192, lognormal channels, shuffled table):
    196 B per token and KV head (128 B of keys + 68 B value record), ~205.5 MB per
    call, more than L2.  Median of `reps` calls timed with CUDA events."""
    import workloads
    mb = T0 // BLOCK + 1
    bt_np, nb = workloads.shuffled_block_table(777, B, mb)
    bt = torch.from_numpy(bt_np).to(dev)
    layer = tq.Layer(nb, HKV, kv_format="k8v4", bits_v=4, seed=0, layer=0, device=dev)
    gen = torch.Generator(device=dev).manual_seed(778)
    sk = torch.exp(torch.randn(HKV, D, generator=gen, device=dev))
    sv = torch.exp(torch.randn(HKV, D, generator=gen, device=dev))
    k = (torch.randn(B * T0, HKV, D, generator=gen, device=dev) * sk).to(torch.bfloat16)
    v = (torch.randn(B * T0, HKV, D, generator=gen, device=dev) * sv).to(torch.bfloat16)
    layer.append(k, v, torch.from_numpy(workloads.prefill_slots(bt_np, T0)).to(dev))
    del k, v
    q = torch.randn(B, HQ, D, generator=gen, device=dev).to(torch.bfloat16)
    ctx = torch.full((B,), T0, dtype=torch.int32, device=dev)
    out = torch.empty(B, HQ, D, dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(layer.workspace_bytes(B, HQ, mb), dtype=torch.uint8, device=dev)
    for _ in range(3):
        layer.decode(q, bt, ctx, out=out, workspace=ws)
    torch.cuda.synchronize()
    ms = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        layer.decode(q, bt, ctx, out=out, workspace=ws)
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    med = statistics.median(ms)
    nbytes = B * HKV * T0 * (D + D * 4 // 8 + 4)
    gbs = nbytes / (med * 1e-3) / 1e9
    status = tq.get_device_status()
    del layer
    torch.cuda.empty_cache()
    return {"workload": "k8v4 layer: B16 Hq32 Hkv8 d128 ctx8192, FP8 E4M3 keys + 4-bit values", "bytes": nbytes,
            "ms": round(med, 4), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "calls": reps,
            "device_status": status}


def decode_long_context(torch, tq, dev, peak, reps=10):
    """Decode at the long-context shape (batch 4, 64 query / 8 KV heads: groups of 8,
    context 131,072, 3-bit keys / 4-bit values, Hadamard, bf16 with 1 % Student-t(3)
    elements, shuffled table): 120 B per token and KV head, ~503.3 MB per call.
    Median of `reps` calls timed with CUDA events."""
    import workloads
    b4, hq, hkv, t = 4, 64, 8, 131072
    mb = t // BLOCK
    bt_np, nb = workloads.shuffled_block_table(781, b4, mb)
    bt = torch.from_numpy(bt_np).to(dev)
    layer = tq.Layer(nb, hkv, bits_k=3, bits_v=4, seed=1, layer=0, device=dev)
    gen = torch.Generator(device=dev).manual_seed(782)
    slots = torch.from_numpy(workloads.prefill_slots(bt_np, t)).to(dev)
    for half in range(2):  # append in two halves (bf16 inputs of 1 GB each)
        sl = slots[half * (b4 * t // 2):(half + 1) * (b4 * t // 2)]
        n = sl.numel()
        def heavy():  # N(0, 1) with 1 % of the elements replaced by Student-t(3) draws
            x = torch.randn(n, hkv, D, generator=gen, device=dev)
            m = torch.rand(n, hkv, D, generator=gen, device=dev) < 0.01
            z = torch.randn(4, int(m.sum()), generator=gen, device=dev)
            x[m] = z[0] / torch.sqrt((z[1] ** 2 + z[2] ** 2 + z[3] ** 2) / 3.0)
            return x.to(torch.bfloat16)
        layer.append(heavy(), heavy(), sl)
    q = torch.randn(b4, hq, D, generator=gen, device=dev).to(torch.bfloat16)
    ctx = torch.full((b4,), t, dtype=torch.int32, device=dev)
    out = torch.empty(b4, hq, D, dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(layer.workspace_bytes(b4, hq, mb), dtype=torch.uint8, device=dev)
    for _ in range(3):
        layer.decode(q, bt, ctx, out=out, workspace=ws)
    torch.cuda.synchronize()
    ms = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        layer.decode(q, bt, ctx, out=out, workspace=ws)
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    med = statistics.median(ms)
    nbytes = b4 * hkv * t * (D * 3 // 8 + 4 + D * 4 // 8 + 4)
    gbs = nbytes / (med * 1e-3) / 1e9
    status = tq.get_device_status()
    del layer, ws
    torch.cuda.empty_cache()
    return {"workload": "long context: B4 Hq64 Hkv8 d128 ctx131072, 3-bit K / 4-bit V, 1% Student-t(3) elements",
            "bytes": nbytes, "ms": round(med, 4), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
            "calls": reps, "device_status": status}


def polar_layer(torch, tq, dev, peak, reps=20):
    """The PolarQuant variant at the headline shape (batch 16, 32/8 heads, context
    8192, lognormal channels, shuffled table, 4-bit angles): the prefill append of
    2,097,152 vectors (256 B read + 66 B written each) and decode over 132 B per token
    and KV head (~138.4 MB per call, more than L2).  Medians of CUDA-event timings."""
    import workloads
    mb = T0 // BLOCK + 1
    bt_np, nb = workloads.shuffled_block_table(779, B, mb)
    bt = torch.from_numpy(bt_np).to(dev)
    layer = tq.Layer(nb, HKV, kv_format="polar", bits_k=4, bits_v=4, seed=0, layer=0, device=dev)
    gen = torch.Generator(device=dev).manual_seed(780)
    sk = torch.exp(torch.randn(HKV, D, generator=gen, device=dev))
    sv = torch.exp(torch.randn(HKV, D, generator=gen, device=dev))
    k = (torch.randn(B * T0, HKV, D, generator=gen, device=dev) * sk).to(torch.bfloat16)
    v = (torch.randn(B * T0, HKV, D, generator=gen, device=dev) * sv).to(torch.bfloat16)
    slots = torch.from_numpy(workloads.prefill_slots(bt_np, T0)).to(dev)
    for _ in range(3):
        layer.append(k, v, slots)
    torch.cuda.synchronize()
    app = []
    for _ in range(max(3, reps // 4)):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        layer.append(k, v, slots)
        e1.record()
        torch.cuda.synchronize()
        app.append(e0.elapsed_time(e1))
    del k, v
    q = torch.randn(B, HQ, D, generator=gen, device=dev).to(torch.bfloat16)
    ctx = torch.full((B,), T0, dtype=torch.int32, device=dev)
    out = torch.empty(B, HQ, D, dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(layer.workspace_bytes(B, HQ, mb), dtype=torch.uint8, device=dev)
    for _ in range(3):
        layer.decode(q, bt, ctx, out=out, workspace=ws)
    torch.cuda.synchronize()
    ms = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        layer.decode(q, bt, ctx, out=out, workspace=ws)
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    med = statistics.median(ms)
    nbytes = B * HKV * T0 * 2 * (D * 4 // 8 + 2)
    gbs = nbytes / (med * 1e-3) / 1e9
    app_ms = statistics.median(app)
    n_vec = 2 * B * T0 * HKV
    app_gbs = n_vec * (2 * D + D * 4 // 8 + 2) / (app_ms * 1e-3) / 1e9
    status = tq.get_device_status()
    del layer
    torch.cuda.empty_cache()
    return {"workload": "polar layer: B16 Hq32 Hkv8 d128 ctx8192, 4-bit angles + fp16 radius (K and V)",
            "decode_bytes": nbytes, "decode_ms": round(med, 4), "decode_gbs": round(gbs, 1),
            "decode_frac": round(gbs / peak, 4), "append_vectors": n_vec, "append_ms": round(app_ms, 4),
            "append_vectors_per_s": round(n_vec / (app_ms * 1e-3), 1), "append_gbs": round(app_gbs, 1),
            "append_frac": round(app_gbs / peak, 4), "device_status": status}


def offload_restore(torch, st, reps=5):
    """Offload every block of one benchmark layer (the pages of its K and V pools,
    block ids in block-table order, i.e. shuffled) to a pinned host image and
    restore them; median GB/s of each direction over `reps` rounds, timed with
    CUDA events."""
    layer = st["layers"][0]
    blocks = st["bt_np"].reshape(-1)
    image = layer.offload(blocks)
    torch.cuda.synchronize()
    nbytes = image.numel()
    d2h, h2d = [], []
    for _ in range(reps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        layer.offload(blocks, image=image)
        e[1].record()
        layer.restore(blocks, image)
        e[2].record()
        torch.cuda.synchronize()
        d2h.append(nbytes / (e[0].elapsed_time(e[1]) * 1e-3) / 1e9)
        h2d.append(nbytes / (e[1].elapsed_time(e[2]) * 1e-3) / 1e9)
    return {"workload": "all %d blocks of one layer (K and V pages, shuffled ids) to a pinned host image and back"
                        % blocks.size, "bytes": nbytes, "offload_gbs": round(statistics.median(d2h), 1),
            "restore_gbs": round(statistics.median(h2d), 1)}


def incremental_dequant_baseline(torch, tq, st, dev, peak, reps=20):
    """The incremental-dequant baseline the pages compare against: a bf16 running
    cache (a bf16 layer) holding the dequantized keys and values of one benchmark
    layer; per step the new token of every sequence is appended to the packed
    layer, dequantized from it (tq_dequantize) and appended to the bf16 cache, and
    decode runs over the bf16 cache (512 B per token and KV head).  Compared with
    the fused step on the packed layer (tq_append_decode, 136 B per token and KV
    head).  Medians of `reps` steps timed with CUDA events."""
    import workloads
    layer = st["layers"][0]
    nb = st["nb"]
    shadow = tq.Layer(nb, HKV, kv_format="bf16", device=dev)
    # dequantize the whole context so far (prefill + the tokens of the timed steps) once
    ctx_now = int(st["ctx"][0].item())
    slots_all = torch.from_numpy(workloads.prefill_slots(st["bt_np"], ctx_now)).to(dev)
    for i0 in range(0, slots_all.numel(), 1 << 16):
        sl = slots_all[i0: i0 + (1 << 16)]
        shadow.append(layer.dequantize(0, sl, out_dtype=torch.bfloat16), layer.dequantize(1, sl, out_dtype=torch.bfloat16),
                      sl)
    out = torch.empty(B, HQ, D, dtype=torch.bfloat16, device=dev)
    ws = torch.zeros(shadow.workspace_bytes(B, HQ, st["mb"]), dtype=torch.uint8, device=dev)
    last_slots(torch, st)
    q, knew, vnew, slot = st["q"][0], st["knew"][0], st["vnew"][0], st["slot_new"]
    ctx = st["ctx"]

    def baseline_step():
        layer.append(knew, vnew, slot)
        shadow.append(layer.dequantize(0, slot, out_dtype=torch.bfloat16), layer.dequantize(1, slot, out_dtype=torch.bfloat16),
                      slot)
        shadow.decode(q, st["bt"], ctx, out=out, workspace=ws)

    def fused_step():
        layer.append_decode(knew, vnew, slot, q, st["bt"], ctx, out=out, workspace=st["ws"], num_splits=SPLITS)

    def bf16_decode():
        shadow.decode(q, st["bt"], ctx, out=out, workspace=ws)

    res = {}
    for name, fn in (("baseline_step_ms", baseline_step), ("fused_step_ms", fused_step),
                     ("bf16_decode_ms", bf16_decode)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ms = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        res[name] = round(statistics.median(ms), 4)
    bf16_bytes = B * HKV * (int(ctx[0].item())) * 2 * D * 2
    res["bf16_decode_gbs"] = round(bf16_bytes / (res["bf16_decode_ms"] * 1e-3) / 1e9, 1)
    res["bf16_decode_frac"] = round(res["bf16_decode_gbs"] / peak, 4)
    res["speedup_fused_vs_baseline"] = round(res["baseline_step_ms"] / res["fused_step_ms"], 3)
    res["workload"] = ("one layer, B16 Hq32 Hkv8 d128 ctx8192: packed 4/4 cache + bf16 running cache of its "
                       "dequantized contents; eager calls (launch gaps included)")
    del shadow
    torch.cuda.empty_cache()
    return res


def step_prepare(torch, st):
    """ctx += 1: the step's new token goes to position ctx (tq_decode_step finds its slot
    from the block table itself)."""
    st["ctx"].add_(1)


def last_slots(torch, st):
    """slot_new = the slots of position ctx - 1 of every sequence (the newest token)."""
    ctx64 = st["ctx"].to(torch.int64) - 1
    blk = torch.gather(st["bt"], 1, (ctx64 // BLOCK).unsqueeze(1)).squeeze(1).to(torch.int64)
    st["slot_new"].copy_(blk * BLOCK + ctx64 % BLOCK)


def layer_decode(st, l):
    st["layers"][l].decode(st["q"][l], st["bt"], st["ctx"], out=st["out"][l], workspace=st["ws"], num_splits=SPLITS)


def layer_step(st, l):
    """Append the new token of every sequence and decode, in one kernel (tq_decode_step)."""
    st["layers"][l].decode_step(st["knew"][l], st["vnew"][l], st["q"][l], st["bt"], st["ctx"],
                                out=st["out"][l], workspace=st["ws"], num_splits=SPLITS)


def run_tq(args):
    import numpy as np
    import torch

    import turboquant_quantized_kv_gb300 as tq
    from turboquant_quantized_kv_gb300 import build as tqbuild

    tqbuild.build()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    st = setup(torch, tq, args.warmup + 2 * args.steps + 4, dev)
    stream = torch.cuda.current_stream()

    # The step (slot bookkeeping, then append + decode of every layer) is one CUDA graph.
    torch.cuda.synchronize()
    for l in range(LAYERS):  # eager warm-up (module load, attributes) before capture
        layer_decode(st, l)
    torch.cuda.synchronize()
    ctx_save = st["ctx"].clone()
    g = torch.cuda.CUDAGraph()
    n_before = tq.launch_count()
    with torch.cuda.graph(g):
        step_prepare(torch, st)
        for l in range(LAYERS):
            layer_step(st, l)
    launches_per_step = tq.launch_count() - n_before  # libtq kernels in one step's graph
    st["ctx"].copy_(ctx_save)
    torch.cuda.synchronize()

    for w in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ctx_start = int(st["ctx"][0].item())
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.synchronize()
    t0.record(stream)
    for s_ in range(args.steps):
        g.replay()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms_total = job_ms(t0.elapsed_time(t1), dev)
    ms_step = ms_total / args.steps
    status = tq.get_device_status()
    # algorithmic bytes: every decode call of the timed steps reads ctx tokens x H_kv
    # records of 136 B (4-bit K + V + fp32 norms) per sequence, plus block table, q, out
    def call_bytes(ctx_s):
        return B * HKV * ctx_s * BYTES_PER_TOKEN_HEAD + B * st["mb"] * 4 + 2 * B * HQ * D * 2
    bytes_steps = sum(LAYERS * call_bytes(ctx_start + s_ + 1) for s_ in range(args.steps))
    value = job_value(bytes_steps, world, ms_total) / 1e9
    peak, peak_kind = peaks()
    # the decode kernel alone: a graph of the decode calls of all layers (no appends, the
    # context as the timed steps left it), replayed; CUDA events around each replay
    gd = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gd):
        for l in range(LAYERS):
            layer_decode(st, l)
    for _ in range(3):
        gd.replay()
    torch.cuda.synchronize()
    rep_ms = []
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gd.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        rep_ms.append(e0.elapsed_time(e1))
    dec_avg_ms = statistics.median(rep_ms) / LAYERS
    achieved = call_bytes(int(st["ctx"][0].item())) / (dec_avg_ms * 1e-3) / 1e9
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if os.path.exists(tpath):  # counters from one ncu capture, valid only for the kernel source they came from
        try:
            import hashlib
            with open(tpath) as f:
                tj = json.load(f)
            with open(os.path.join(ROOT, "turboquant_quantized_kv_gb300", "csrc", "tq_decode.cu"), "rb") as f:
                sha = hashlib.sha256(f.read()).hexdigest()
            traffic = tj.get("bytes_per_launch") if tj.get("source_sha256") == sha else None
        except Exception:
            traffic = None
    app_ms = statistics.median(st["append_ms"][2:] if len(st["append_ms"]) > 2 else st["append_ms"])
    app_vps = st["append_vectors"] / (app_ms * 1e-3)
    app_gbs = app_vps * APPEND_BYTES_PER_VECTOR / 1e9

    # end to end through the public API with host buffers (pinned), eager calls
    e2e = run_e2e(torch, st, args, stream) if args.e2e else None
    dense, dense_dec = dense_workload(torch, tq, dev, peak, args.vlm_steps) if args.dense_burst else (None, None)
    mixed = mixed62(torch, tq, dev, peak) if args.mixed else None
    k8 = decode_k8v4(torch, tq, dev, peak) if args.k8v4 else None
    lc = decode_long_context(torch, tq, dev, peak) if args.long_context else None
    pol = polar_layer(torch, tq, dev, peak) if args.polar else None
    off = offload_restore(torch, st) if args.offload else None
    incr = incremental_dequant_baseline(torch, tq, st, dev, peak) if args.incremental else None

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u4 codes + fp32 norms (bf16 q/out, fp16 MMA with fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": B, "num_q_heads": HQ, "num_kv_heads": HKV, "head_dim": D,
                   "context": T0, "layers": LAYERS, "bits_k": 4, "bits_v": 4, "block_size": BLOCK,
                   "splits": st["layers"][0].auto_splits(B, HQ, st["mb"]) if SPLITS == 0 else SPLITS,
                   "l2": "inputs larger than L2 (~4.6 GB of packed cache per step)", "parallelism": "replicas"},
        "roofline": {"kernel": "k_decode (tq_decode_attention: split-K decode with the merge and inverse rotation "
                               "fused)", "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind, "traffic": traffic,
                     "timing": "graph of the %d layers' decode calls, median of 10 replays / %d (%.2f us per call)"
                               % (LAYERS, LAYERS, dec_avg_ms * 1e3)},
        "append": {"vectors_per_s": round(app_vps, 1), "gbs": round(app_gbs, 1), "frac": round(app_gbs / peak, 4),
                   "vectors": st["append_vectors"], "bytes_per_vector": APPEND_BYTES_PER_VECTOR},
        "append_dense_burst": dense,
        "decode_vlm_b1": dense_dec,
        "decode_mixed62": mixed,
        "decode_k8v4": k8,
        "decode_long_context": lc,
        "polar": pol,
        "offload_restore": off,
        "incremental_dequant_baseline": incr,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clk,
        "device_status": status,
    }
    if rank == 0 and args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(st, args)
        line["append_tie_band"] = tie_band(st)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_e2e(torch, st, args, stream):
    """Public API, host buffers: per step the H2D copy of the new K/V tokens and queries
    of every layer from one pinned staging buffer, append + decode per layer through
    Layer.decode_step, and the D2H copy of all layers' outputs; the copies go in
    chunks of 8 layers on a second stream, each layer waiting only for its own chunk."""
    parts = [t for l in range(LAYERS) for t in (st["knew"][l], st["vnew"][l], st["q"][l])]
    sizes = [t.numel() for t in parts]
    h_in = torch.empty(sum(sizes), dtype=torch.bfloat16).pin_memory()
    off = 0
    for t, n in zip(parts, sizes):
        h_in[off:off + n].copy_(t.reshape(-1).cpu())
        off += n
    d_in = torch.empty_like(h_in, device=st["q"][0].device)
    views, off = [], 0
    for t, n in zip(parts, sizes):
        views.append(d_in[off:off + n].view(t.shape))
        off += n
    d_out = torch.empty(LAYERS, B, HQ, D, dtype=torch.bfloat16, device=d_in.device)
    h_out = torch.empty(d_out.shape, dtype=torch.bfloat16).pin_memory()
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size()
    # the copies run on a second stream in chunks of `per` layers, ordered by events, so
    # that they overlap the layers that do not need them
    per = 8 if LAYERS % 8 == 0 else LAYERS
    n_chunks = LAYERS // per
    in_bounds = [0]
    for c in range(n_chunks):
        in_bounds.append(in_bounds[-1] + sum(sizes[3 * per * c:3 * per * (c + 1)]))
    cs = torch.cuda.Stream(device=d_in.device)
    ev_in = [torch.cuda.Event() for _ in range(n_chunks)]
    ev_out = [torch.cuda.Event() for _ in range(n_chunks)]

    def step():
        step_prepare(torch, st)
        cs.wait_stream(stream)  # the previous step is done with the staging buffers
        with torch.cuda.stream(cs):
            for c in range(n_chunks):
                d_in[in_bounds[c]:in_bounds[c + 1]].copy_(h_in[in_bounds[c]:in_bounds[c + 1]], non_blocking=True)
                ev_in[c].record(cs)
        for l in range(LAYERS):
            c = l // per
            if l % per == 0:
                stream.wait_event(ev_in[c])
            k, v, q = views[3 * l], views[3 * l + 1], views[3 * l + 2]
            st["layers"][l].decode_step(k, v, q, st["bt"], st["ctx"], out=d_out[l], workspace=st["ws"],
                                        num_splits=SPLITS)
            if l % per == per - 1:
                ev_out[c].record(stream)
                cs.wait_event(ev_out[c])
                with torch.cuda.stream(cs):
                    h_out[c * per:(c + 1) * per].copy_(d_out[c * per:(c + 1) * per], non_blocking=True)
        stream.wait_stream(cs)  # the step ends with its outputs on the host

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    ctx_start = int(st["ctx"][0].item())
    n = max(2, args.steps // 2)
    t = time.perf_counter()
    for _ in range(n):
        step()
    torch.cuda.synchronize()
    dt = time.perf_counter() - t
    nbytes = sum(LAYERS * B * HKV * (ctx_start + s + 1) * BYTES_PER_TOKEN_HEAD for s in range(n))
    return {"value": round(nbytes / dt / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n, "ms_per_step": round(dt / n * 1e3, 4)}


# ------------------------------------------------------------- oracle (CPU)

def _oracle_unit(payload):
    """One (sequence, KV head) unit of the oracle decode: unpack + exact attention."""
    import numpy as np
    from oracle import attention as oa, codebook as ocb, pack as opack, rotation as orot
    kpages, vpages, q, layer_idx = payload
    c4 = ocb.codebook_fp32(D, 4)[0].astype(np.float64)
    pi = orot.hadamard_rotation_seeded(0, layer_idx, D)
    kc, kg = opack.split_pages(kpages, D, 4)
    vc, vg = opack.split_pages(vpages, D, 4)
    khat = (c4[kc.reshape(-1, D)] * kg.reshape(-1)[:, None]) @ pi
    vhat = (c4[vc.reshape(-1, D)] * vg.reshape(-1)[:, None]) @ pi
    for h in range(q.shape[0]):
        s = (khat @ q[h]) / math.sqrt(D)
        oa.softmax_weights(s) @ vhat
    return kpages.nbytes + vpages.nbytes


def _oracle_payload(u):
    """Packed pages of one (sequence, KV head) unit of 8192 tokens, made by the oracle."""
    import numpy as np
    import workloads
    from oracle import codebook as ocb, pack as opack, quantize as oq, rotation as orot
    c4, b4 = ocb.codebook_fp32(D, 4)
    kb, vb = workloads.lognormal_channel_kv(u, T0, 1, D)
    pi = orot.hadamard_rotation_seeded(0, u % 32, D)
    pages = []
    for xb in (kb, vb):
        idx, gamma, _ = oq.quantize(oq.bf16_bits_to_f64(xb[:, 0]), pi, c4, b4)
        rec = opack.pack_records(idx, 4).reshape(T0 // BLOCK, BLOCK * 64)
        g = gamma.astype("<f4").view(np.uint8).reshape(T0 // BLOCK, BLOCK * 4)
        pages.append(np.concatenate([rec, g], axis=1))
    q = oq.bf16_bits_to_f64(workloads.queries(u, 1, HQ // HKV, D))[0]
    return pages[0], pages[1], q, u % 32


def _oracle_payloads(n_units, pool=None):
    return pool.map(_oracle_payload, range(n_units)) if pool else [_oracle_payload(u) for u in range(n_units)]


def cpu_baseline(st, args):
    """The oracle as it stands on the host cores, on a bounded sample (spawned pool)."""
    import multiprocessing as mp
    cores = min(os.cpu_count() or 1, 16)
    n_units = cores * 12
    ctxm = mp.get_context("spawn")
    env_keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in env_keep:
        os.environ[k] = "1"
    try:
        with ctxm.Pool(cores) as pool:
            payloads = _oracle_payloads(n_units, pool)  # untimed: the oracle packs the sample
            pool.map(_oracle_unit, payloads[:cores])  # warm the workers
            t = time.perf_counter()
            nbytes = sum(pool.map(_oracle_unit, payloads))
            dt = time.perf_counter() - t
    finally:
        for k, v in env_keep.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d (sequence, KV head) units x 8192 tokens x 4 query heads of one layer each "
                      "(packed by the oracle), unpack + exact fp64 attention; %d worker processes, 1 BLAS thread each"
                      % (n_units, cores), "seconds": round(dt, 2)}


def tie_band(st):
    """Codes of the benchmark's own prefill keys against the oracle's: 2,048 tokens x 8
    KV heads of layer 0 (bf16 inputs, Hadamard rotation of seed 0, 4-bit codes), the
    oracle quantizing the same bf16 vectors in fp64 and the GPU's codes read from its
    pages.  Reports the fraction of coordinates whose codes differ and the largest
    distance |y - beta| between the oracle's rotated coordinate and the boundary
    separating the two codes among them (the parity rule allows 1e-5).  Part of the
    CPU leg, the one place the benchmark runs the oracle."""
    import numpy as np
    from oracle import codebook as ocb, pack as opack, quantize as oq, rotation as orot
    c4, b4 = ocb.codebook_fp32(D, 4)
    x = oq.bf16_bits_to_f64(st["tie_x"])  # [tok][H][d]
    pi = orot.hadamard_rotation_seeded(0, 0, D)
    idx, _, y = oq.quantize(x, pi, c4, b4)
    layer = st["layers"][0]
    pool = layer.k_cache.cpu().numpy()
    pages = opack.pool_pages(pool, layer.num_blocks, HKV, opack.page_bytes(D, 4))
    slots = st["tie_slots"]
    codes, _ = opack.split_pages(pages[slots // BLOCK], D, 4)  # [tok][H][16][d]
    gpu = codes[np.arange(slots.size), :, slots % BLOCK]       # [tok][H][d]
    mism = gpu != idx
    worst = 0.0
    if mism.any():
        lo = np.minimum(gpu, idx)[mism]
        beta = np.asarray(b4, np.float64)[np.clip(lo, 0, len(b4) - 1)]
        worst = float(np.max(np.abs(y[mism] - beta)))
    return {"sample": "%d prefill tokens x %d KV heads of layer 0 (%d coordinates)" % (slots.size, HKV, mism.size),
            "mismatch_rate": float(mism.mean()), "mismatches": int(mism.sum()), "max_abs_y_minus_beta": worst,
            "tau": 1e-5}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import multiprocessing as mp
    cores = min(os.cpu_count() or 1, 16)
    per_step = cores
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    ctxm = mp.get_context("spawn")
    with ctxm.Pool(cores) as pool:
        payloads = _oracle_payloads(per_step, pool)
        for _ in range(args.warmup):
            pool.map(_oracle_unit, payloads)
        t = time.perf_counter()
        nbytes = 0
        for _ in range(args.steps):
            nbytes += sum(pool.map(_oracle_unit, payloads))
        dt = time.perf_counter() - t
    value = nbytes / dt / 1e9
    sample = ("per step %d (sequence, KV head) units x 8192 tokens x 4 query heads (1/%d of one layer-step "
              "of the workload), unpack + exact fp64 attention, %d processes" % (per_step, B * HKV // per_step
                                                                               if per_step <= B * HKV else 1, cores))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": B, "num_q_heads": HQ, "num_kv_heads": HKV, "head_dim": D,
                   "context": T0, "layers": LAYERS, "bits_k": 4, "bits_v": 4, "block_size": BLOCK},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle", "cores": cores,
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="tq", choices=["tq", "reference"])
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-k8v4", dest="k8v4", action="store_false", help="skip the k8v4 decode measurement")
    ap.add_argument("--no-offload", dest="offload", action="store_false", help="skip the offload/restore measurement")
    ap.add_argument("--no-polar", dest="polar", action="store_false", help="skip the PolarQuant-variant measurement")
    ap.add_argument("--no-long-context", dest="long_context", action="store_false",
                    help="skip the long-context (131,072-token, groups of 8) decode measurement")
    ap.add_argument("--no-incremental", dest="incremental", action="store_false",
                    help="skip the incremental-dequant baseline measurement")
    ap.add_argument("--no-dense-burst", dest="dense_burst", action="store_false",
                    help="skip the dense-rotation workload (burst append of 36 layers x 11000 tokens, then "
                         "batch-1 decode steps)")
    ap.add_argument("--vlm-steps", type=int, default=256,
                    help="batch-1 decode steps of the dense-rotation workload (profiling runs use fewer)")
    ap.add_argument("--no-mixed", dest="mixed", action="store_false",
                    help="skip the 62-layer mixed bf16 / 4-bit step (B8, 100,000 tokens, 64 GB of cache)")
    ap.add_argument("--layers", type=int, default=LAYERS, help="layers per step (profiling runs use fewer)")
    ap.add_argument("--splits", type=int, default=0, help="decode context splits (0 = library default)")
    args = ap.parse_args()
    globals()["LAYERS"] = args.layers
    globals()["SPLITS"] = args.splits
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_tq(args)


if __name__ == "__main__":
    main()
