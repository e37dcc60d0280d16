#!/usr/bin/env python
"""Benchmark of the KVarN K4V2 g128 hot path on GB300.

Workload (default): one decode step of paged attention over a K4V2 g128 packed cache --
batch 64, seq_len = 128 * U{8..128} (mean ~8.7K tokens), 32 query heads over 8 KV heads,
head_dim 128, randomly permuted block table; the cache is built from the synthetic outlier
generator by kvarn_quantize_tiles.  One step = kvarn_append_token (one new fp16 K/V token per
sequence, sealing full tiles) + kvarn_decode_attention over the sealed pages and the partial
tile.  The metric counts attended KV tokens (all heads of a token) per second.

Also measured in the same run: kvarn_quantize_tiles throughput on one layer of 8 KV heads x
16384 tokens x head_dim 128 (L2 flushed between launches).

--impl reference times the float64 CPU oracle on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs an independent replica (weak scaling, no collective on
the data path); value = tokens of all ranks / slowest rank's time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "K4V2 g128 decode-attn KV tokens/s & HBM GB/s; quantize tokens/s (1 GB300)"
QUANT_OPS_PER_ELEMENT = 38  # fp32 ops per quantised element (derivation at the quantize timing)
SM_MAX_MHZ = 2070.0
ADAPTIVE_TOL = 0.05  # early-stop tolerance of the normalisation (log-factor change per iteration)
DEC_EVENT_SAMPLES = 40  # live samples of the decode call's duration, spread over the timed steps
DEC_EVENT_EVERY_MIN = 5  # ... on at most one step in five, so most steps keep their launch overlap
WORKLOAD = ("paged decode attention + append: batch 64, seq_len 128*U{8..128}, 32 q heads / 8 kv "
            "heads, head_dim 128, K4V2 g128 packed cache, permuted block table")
BATCH, HQ, HKV, D0, MIN_PAGES, MAX_PAGES, SEED = 64, 32, 8, 128, 8, 128, 3
Q_TOKENS, Q_HEADS = 16384, 8   # quantise-throughput layer


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# DRAM traffic / algorithmic bytes of one decode_kernel launch, from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum at batch 24), valid only for the sources it was
# taken on (decode.cu and decode_util.cuh, which holds the page partition): the traffic is
# reported as null once either changes.
DECODE_TRAFFIC = {"sources_sha256": "254ea2120da7c12ce795533a3645deee08d4b37d5c670276bcc800834b4d1815",
                  "dram_over_algorithmic": 1.0235}
DECODE_SOURCES = ("decode.cu", "decode_util.cuh")


def _decode_sources_digest():
    """sha256 over the decode sources named in DECODE_SOURCES, in that order."""
    import hashlib
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "calibration_free_kv_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _decode_traffic_ratio():
    """DRAM bytes / algorithmic bytes of the decode kernel, or None when its sources changed
    since the capture DECODE_TRAFFIC records."""
    try:
        digest = _decode_sources_digest()
    except OSError:
        return None
    if DECODE_TRAFFIC["dram_over_algorithmic"] is None or digest != DECODE_TRAFFIC["sources_sha256"]:
        return None
    return float(DECODE_TRAFFIC["dram_over_algorithmic"])


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _aggregate_over_ranks(torch, world, per_rank_ms, tokens_per_rank, device):
    """Whole-job throughput of `world` independent replicas: every timing is the maximum over
    ranks (the slowest replica ends the job) and the tokens are those of all ranks.
    Returns (max timings in ms, throughputs per second)."""
    t = torch.tensor([float(x) for x in per_rank_ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms = [float(x) for x in t]
    return ms, [world * tok / (m * 1e-3) for tok, m in zip(tokens_per_rank, ms)]


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,power.draw")

    def __init__(self, device_id: str):
        self.device_id = device_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.device_id, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        """Host time, to bracket the timed region."""
        return time.time()

    def stop(self, window=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        lines = self.lines
        inside = [ln for t, ln in lines if window is None or window[0] <= t <= window[1]]
        where = "during the timed region"
        if not inside and window is not None and lines:  # a region shorter than the sampling interval
            mid = 0.5 * (window[0] + window[1])
            inside = [ln for t, ln in sorted(lines, key=lambda x: abs(x[0] - mid))[:3]]
            where = "nearest the timed region (shorter than the 50 ms sampling interval)"
        for line in inside:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[2:6]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "sampled": where}


def _device_id(torch):
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(0).uuid).replace("GPU-", "")
    except Exception:
        return os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0]


# ------------------------------------------------------------------------------------------------
# KVarN (CUDA) arm
# ------------------------------------------------------------------------------------------------

def _setup_decode(torch, kv, synth, steps_total):
    dev = torch.device("cuda")
    shape = synth.decode_batch(BATCH, HQ, HKV, D0, seed=SEED, min_pages=MIN_PAGES, max_pages=MAX_PAGES)
    lens0 = _initial_lens()  # sealed pages + raw tokens of the open tile
    phase = lens0 % 128
    base_table = shape["block_table"]
    n_seal_pages = int((lens0 // 128).sum())
    grow = steps_total // 128 + 2                    # pages each sequence may seal while timed
    width = base_table.shape[1] + grow
    n_pool = n_seal_pages + BATCH * grow
    table = torch.zeros((BATCH, width), dtype=torch.int32)
    extra = torch.arange(n_seal_pages, n_pool, dtype=torch.int32).view(BATCH, grow)
    for b in range(BATCH):
        n = int(lens0[b]) // 128
        table[b, :n] = base_table[b, :n]
        table[b, n:n + grow] = extra[b]
    desc = kv.desc_from_preset(D0, HKV)
    assert desc.page_record_bytes == REC_BYTES
    pool = kv.alloc_pool(desc, n_pool, device=dev)
    total = 128 * n_seal_pages  # the sealed tokens (the open tiles come from another draw)
    k_all, v_all = synth.outlier_kv(total, HKV, D0, seed=SEED, device=dev)
    page_ids = torch.cat([base_table[b, :int(lens0[b]) // 128] for b in range(BATCH)]).to(dev)
    kv.quantize_tiles(desc, k_all, v_all, page_ids, pool)
    # the open tile of sequence b holds phase[b] raw fp16 tokens of the same generator
    kp, vp = synth.outlier_kv(BATCH * 128, HKV, D0, seed=SEED + 9, device=dev)
    rows = (torch.arange(128, device=dev)[None, :] < phase.to(dev)[:, None]).to(torch.float16)
    pk = (kp.view(BATCH, 128, HKV, D0).transpose(1, 2) * rows[:, None, :, None]).contiguous()
    pv = (vp.view(BATCH, 128, HKV, D0).transpose(1, 2) * rows[:, None, :, None]).contiguous()
    torch.cuda.synchronize()
    del k_all, v_all, kp, vp
    torch.cuda.empty_cache()
    g = torch.Generator(device=dev)
    g.manual_seed(SEED + 1)
    n_sets = 4
    qs = [torch.randn((BATCH, HQ, D0), generator=g, device=dev).half() for _ in range(n_sets)]
    kn = [torch.randn((BATCH, HKV, D0), generator=g, device=dev).half() for _ in range(n_sets)]
    vn = [torch.randn((BATCH, HKV, D0), generator=g, device=dev).half() for _ in range(n_sets)]
    return {
        "desc": desc, "pool": pool, "table": table.to(dev), "lens0": lens0, "qs": qs, "kn": kn, "vn": vn,
        "pk": pk, "pv": pv,
        "lens": [lens0.to(torch.int32).to(dev), torch.zeros(BATCH, dtype=torch.int32, device=dev)],
        "out": torch.empty((BATCH, HQ, D0), dtype=torch.float16, device=dev),
        "ws": kv.alloc_workspace(desc, BATCH, HQ, width, device=dev),
        "status": torch.zeros(1, dtype=torch.int32, device=dev),
        "rec_bytes": desc.page_record_bytes,
    }


REC_BYTES = 13824  # one kvarn_k4v2_g128 page record at head_dim 128 (checked against the library)


def _initial_lens():
    """Lengths of the decode workload before its first step: 128 * U{8..128} sealed tokens plus
    U{0..127} raw tokens in each sequence's open tile (CPU int64 [BATCH])."""
    import torch
    from calibration_free_kv_gb300 import synth
    shape = synth.decode_batch(BATCH, HQ, HKV, D0, seed=SEED, min_pages=MIN_PAGES, max_pages=MAX_PAGES)
    return shape["seq_lens"].to(torch.int64) + synth.partial_phases(BATCH, SEED + 7)


def _workload_config(lens_before, steps):
    """The `config` object of the bench line, the same for both arms: lens_before are the
    lengths when the timed steps start (CPU int64 [BATCH])."""
    mean0 = float(lens_before.double().mean())
    return {
        "workload": WORKLOAD.replace("batch 64", "batch %d" % BATCH),
        "batch": BATCH, "num_q_heads": HQ, "num_kv_heads": HKV, "head_dim": D0,
        "seq_len": "128*U{8..128} sealed + U{0..127} raw tokens in the open tile",
        "mean_seq_len": mean0,
        "growth": "each step appends one token per sequence (a tile seals every 128 steps per "
                  "sequence, at random phases); mean length over the timed steps %.0f"
                  % (mean0 + (steps + 1) / 2),
        "preset": "kvarn_k4v2_g128",
        "l2": "inputs larger than L2: each decode reads %.0f MB of packed cache"
              % (_decode_bytes((lens_before + 1).tolist(), REC_BYTES) / 1e6),
    }


def _decode_bytes(lens, rec_bytes):
    """Algorithmic bytes of one decode call: packed pages + raw fp16 tokens of the open tiles + q +
    out."""
    sealed = sum(int(L) // 128 for L in lens)
    part = sum(int(L) % 128 for L in lens)
    return (sealed * HKV * rec_bytes + part * HKV * D0 * 2 * 2 + 2 * BATCH * HQ * D0 * 2)


def _decode_kernel_bytes(lens, rec_bytes):
    """Algorithmic bytes of decode_kernel alone (kvarn_decode_partials): the packed pages and q.
    The raw tokens of the open tiles and the output belong to the merge kernel, which attends to
    the open tiles itself."""
    sealed = sum(int(L) // 128 for L in lens)
    return sealed * HKV * rec_bytes + BATCH * HQ * D0 * 2


def _time_quantize(torch, kv, synth, dev, stream, preset="kvarn_k4v2_g128", reps=20, tol=None, d0=D0):
    """Median ms of kvarn_quantize_tiles on one layer (8 kv heads x 16384 tokens x head_dim d0,
    K and V), L2 flushed with a 512 MB write before every launch; and its algorithmic bytes.
    With tol: kvarn_quantize_tiles_adaptive, and also the mean iterations used."""
    qdesc = kv.desc_from_preset(d0, Q_HEADS, preset=preset)
    kq, vq = synth.outlier_kv(Q_TOKENS, Q_HEADS, d0, seed=2, device=dev)
    qpool = kv.alloc_pool(qdesc, Q_TOKENS // 128, device=dev)
    qids = torch.arange(Q_TOKENS // 128, dtype=torch.int32, device=dev)
    used = torch.zeros((Q_TOKENS // 128, Q_HEADS, 2), dtype=torch.int32, device=dev) if tol is not None else None
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    q_ms = []
    for rep in range(3 + reps):
        flush.fill_(float(rep))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        kv.quantize_tiles(qdesc, kq, vq, qids, qpool, stream=stream, sinkhorn_tol=tol, iters_used=used)
        b.record(stream)
        torch.cuda.synchronize()
        if rep >= 3:
            q_ms.append(a.elapsed_time(b))
    nbytes = 2 * Q_TOKENS * Q_HEADS * d0 * 2 + (Q_TOKENS // 128) * Q_HEADS * qdesc.page_record_bytes
    mean_iters = float(used.double().mean()) if used is not None else None
    del kq, vq, qpool, flush
    torch.cuda.empty_cache()
    if tol is not None:
        return statistics.median(q_ms), nbytes, mean_iters
    return statistics.median(q_ms), nbytes


def _time_error_telemetry(torch, kv, synth, dev, stream, reps=10):
    """kvarn_quantization_error over the quantise layer (8 kv heads x 16384 tokens x d 128): every
    record checked against its fp16 tiles, L2 flushed before each launch.  Returns us and the
    bytes it reads (fp16 tiles + records)."""
    qdesc = kv.desc_from_preset(D0, Q_HEADS)
    kq, vq = synth.outlier_kv(Q_TOKENS, Q_HEADS, D0, seed=2, device=dev)
    qpool = kv.alloc_pool(qdesc, Q_TOKENS // 128, device=dev)
    qids = torch.arange(Q_TOKENS // 128, dtype=torch.int32, device=dev)
    kv.quantize_tiles(qdesc, kq, vq, qids, qpool, stream=stream)
    err = torch.zeros((Q_TOKENS // 128, Q_HEADS, 2, 4), dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    ms = []
    for rep in range(3 + reps):
        flush.fill_(float(rep))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        kv.quantization_error(qdesc, kq, vq, qids, qpool, err, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        if rep >= 3:
            ms.append(a.elapsed_time(b))
    e = err.double()
    rel_k = torch.sqrt(e[:, :, 0, 0] / e[:, :, 0, 1])
    rel_v = torch.sqrt(e[:, :, 1, 0] / e[:, :, 1, 1])
    nbytes = 2 * Q_TOKENS * Q_HEADS * D0 * 2 + (Q_TOKENS // 128) * Q_HEADS * qdesc.page_record_bytes
    t = statistics.median(ms)
    del kq, vq, qpool, flush
    torch.cuda.empty_cache()
    return {"us": t * 1e3, "algorithmic_bytes": nbytes, "hbm_gbs": nbytes / (t * 1e-3) / 1e9,
            "rel_frobenius_error_k_mean": float(rel_k.mean()), "rel_frobenius_error_k_max": float(rel_k.max()),
            "rel_frobenius_error_v_mean": float(rel_v.mean()), "rel_frobenius_error_v_max": float(rel_v.max())}


def _time_decode_layers(torch, kv, synth, batch, seq_len, hq, hkv, d0, layers, seed, reps=5,
                        preset="kvarn_k4v2_g128", kernel=None):
    """Decode over `layers` independent packed caches (one pool per layer, one shared permuted
    block table, every sequence at seq_len), launched back to back on one stream: median ms
    per pass over all layers, and the algorithmic bytes of one pass."""
    dev = torch.device("cuda")
    pages = seq_len // 128
    desc = kv.desc_from_preset(d0, hkv, preset=preset)
    g = torch.Generator().manual_seed(seed)
    table = torch.randperm(batch * pages, generator=g).view(batch, pages).to(torch.int32).to(dev)
    page_ids = table.reshape(-1).contiguous()
    lens = torch.full((batch,), seq_len, dtype=torch.int32, device=dev)
    # the packed caches first, as a serving process allocates its cache pool before per-step
    # buffers: a pool placed behind the fp16 K/V temporaries, in memory another configuration
    # had just released, decoded ~20 % slower at head_dim 96 in every repetition
    pools = [kv.alloc_pool(desc, batch * pages, device=dev) for _ in range(layers)]
    qs = []
    for layer in range(layers):
        k, v = synth.outlier_kv(batch * seq_len, hkv, d0, seed=seed * 1000 + layer, device=dev)
        pool = pools[layer]
        kv.quantize_tiles(desc, k, v, page_ids, pool)
        del k, v
        qs.append(torch.randn((batch, hq, d0), generator=g).half().to(dev))
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    outs = [torch.empty((batch, hq, d0), dtype=torch.float16, device=dev) for _ in range(layers)]
    ws = kv.alloc_workspace(desc, batch, hq, pages, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    scale = 1.0 / math.sqrt(d0)

    def one_pass():
        for layer in range(layers):
            kv.decode_attention(desc, qs[layer], pools[layer], table, lens, outs[layer], ws,
                                softmax_scale=scale, status=status, stream=stream)

    # kernel "tc": the library's tcgen05 decode of GQA 8 (selected by KVARN_DECODE_KERNEL)
    saved = os.environ.get("KVARN_DECODE_KERNEL")
    if kernel is not None:
        os.environ["KVARN_DECODE_KERNEL"] = kernel
    try:
        for _ in range(3):
            one_pass()
        ms = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            # keep the GPU busy (~100 us) while the host enqueues the pass, so that the events
            # time the kernels and not the host's launch latency of the first one
            torch.cuda._sleep(200000)
            a.record(stream)
            one_pass()
            b.record(stream)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
    finally:
        if saved is None:
            os.environ.pop("KVARN_DECODE_KERNEL", None)
        else:
            os.environ["KVARN_DECODE_KERNEL"] = saved
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in the layered decode" % int(status.item()))
    nbytes = layers * (batch * pages * hkv * desc.page_record_bytes + 2 * batch * hq * d0 * 2)
    del pools, outs, ws
    torch.cuda.empty_cache()
    return statistics.median(ms), nbytes


def _quality(torch, kv, synth):
    """Attention-output cosine against full-precision attention over the raw fp16 K/V (float64,
    torch), for the KVarN K4V2 cache decoded by the library, and, as an ablation, for plain
    asymmetric round-to-nearest at the same bits on the raw 128-token tiles (K 4-bit per
    channel, V 2-bit per token; no rotation, no variance normalisation)."""
    dev = torch.device("cuda")
    B, L, hkv, G, d = 4, 4096, HKV, HQ // HKV, D0
    pages = L // 128
    desc = kv.desc_from_preset(d, hkv)
    k, v = synth.outlier_kv(B * L, hkv, d, seed=SEED + 100, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(SEED + 101)
    q = torch.randn((B, hkv * G, d), generator=gen, device=dev).half()
    table = torch.arange(B * pages, dtype=torch.int32, device=dev).view(B, pages)
    pool = kv.alloc_pool(desc, B * pages, device=dev)
    kv.quantize_tiles(desc, k, v, table.reshape(-1).contiguous(), pool)
    out = torch.empty_like(q)
    ws = kv.alloc_workspace(desc, B, hkv * G, pages, device=dev)
    lens = torch.full((B,), L, dtype=torch.int32, device=dev)
    kv.decode_attention(desc, q, pool, table, lens, out, ws, softmax_scale=1 / math.sqrt(d))
    torch.cuda.synchronize()
    qq = q.double().view(B, hkv, G, d)

    def attend(kk, vv):  # [B, L, hkv, d] -> [B, hkv * G, d]
        p = torch.softmax(torch.einsum("bhgd,blhd->bhgl", qq, kk) / math.sqrt(d), dim=-1)
        return torch.einsum("bhgl,blhd->bhgd", p, vv).reshape(B, hkv * G, d)

    def rtn(x, bits, dim):
        lo, hi = x.amin(dim=dim, keepdim=True), x.amax(dim=dim, keepdim=True)
        s = ((hi - lo) / (2 ** bits - 1)).clamp_min(1e-8)
        return torch.round((x - lo) / s).clamp(0, 2 ** bits - 1) * s + lo

    kk, vv = k.double().view(B, L, hkv, d), v.double().view(B, L, hkv, d)
    ref = attend(kk, vv)
    k_rtn = rtn(kk.view(B, pages, 128, hkv, d), 4, 2).view(B, L, hkv, d)
    v_rtn = rtn(vv.view(B, pages, 128, hkv, d), 2, 4).view(B, L, hkv, d)
    naive = attend(k_rtn, v_rtn)

    def cos(a):
        return torch.nn.functional.cosine_similarity(a.reshape(-1, d), ref.reshape(-1, d), dim=-1)

    def dist(c):  # per (sequence, query head) cosines
        qs = torch.quantile(c, torch.tensor([0.01, 0.05, 0.25, 0.5], dtype=c.dtype, device=c.device))
        return {"mean": float(c.mean()), "min": float(c.min()), "p1": float(qs[0]), "p5": float(qs[1]),
                "p25": float(qs[2]), "median": float(qs[3])}

    c_kv, c_rtn = cos(out.double()), cos(naive)
    res = {
        "cosine_vs_full_precision": float(c_kv.mean()), "cosine_min": float(c_kv.min()),
        "naive_rtn_cosine": float(c_rtn.mean()), "naive_rtn_cosine_min": float(c_rtn.min()),
        "q_unit_normal": {"kvarn": dist(c_kv), "naive_rtn": dist(c_rtn)},
    }
    # the same caches with q / sqrt(d) (the tiny configuration's query scale): softer
    # attention, so fewer heads sit on a near-tie between two keys
    qs = (q.float() / math.sqrt(d)).half()
    out2 = torch.empty_like(q)
    kv.decode_attention(desc, qs, pool, table, lens, out2, ws, softmax_scale=1 / math.sqrt(d))
    torch.cuda.synchronize()
    qq = qs.double().view(B, hkv, G, d)
    ref = attend(kk, vv)
    c_kv2, c_rtn2 = cos(out2.double()), cos(attend(k_rtn, v_rtn))
    res["q_over_sqrt_d"] = {"kvarn": dist(c_kv2), "naive_rtn": dist(c_rtn2)}
    res["sample"] = ("%d sequences x %d tokens, %d q heads / %d kv heads, head_dim %d, outlier "
                     "generator; q ~ N(0,1) and q ~ N(0,1)/sqrt(d); per (sequence, query head) "
                     "cosines; reference: float64 softmax attention over the raw fp16 K/V"
                     % (B, L, hkv * G, hkv, d))
    res["note"] = "a quality figure, not a target"
    return res


def _time_prefill(torch, kv, synth, batch=8, cache_len=8192, chunk=64, hq=32, hkv=8, d0=128, seed=7, reps=10):
    """kvarn_prefill_attention: `chunk` new tokens per sequence over `cache_len` cached tokens
    (sealed pages only) plus themselves, causal.  Returns median ms and the reported figures."""
    dev = torch.device("cuda")
    pages = cache_len // 128
    desc = kv.desc_from_preset(d0, hkv)
    g = torch.Generator().manual_seed(seed)
    table = torch.randperm(batch * pages, generator=g).view(batch, pages).to(torch.int32).to(dev)
    k, v = synth.outlier_kv(batch * cache_len, hkv, d0, seed=seed, device=dev)
    pool = kv.alloc_pool(desc, batch * pages, device=dev)
    kv.quantize_tiles(desc, k, v, table.reshape(-1).contiguous(), pool)
    del k, v
    q = torch.randn((batch, chunk, hq, d0), generator=g).half().to(dev)
    ck = torch.randn((batch, chunk, hkv, d0), generator=g).half().to(dev)
    cv = torch.randn((batch, chunk, hkv, d0), generator=g).half().to(dev)
    out = torch.empty_like(q)
    lens = torch.full((batch,), cache_len, dtype=torch.int32, device=dev)
    ws = kv.alloc_prefill_workspace(desc, batch, hq, chunk, pages, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        kv.prefill_attention(desc, q, ck, cv, pool, table, lens, out, ws, status=status, stream=stream)
    ms = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        kv.prefill_attention(desc, q, ck, cv, pool, table, lens, out, ws, status=status, stream=stream)
        b.record(stream)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in prefill" % int(status.item()))
    t = statistics.median(ms)
    flops = 4.0 * batch * chunk * hq * (cache_len + (chunk + 1) / 2.0) * d0
    cache_bytes = batch * pages * hkv * desc.page_record_bytes
    del pool, ws
    torch.cuda.empty_cache()
    return {
        "workload": "batch %d, %d new tokens each over %d cached tokens, %d q heads / %d kv heads, "
                    "head_dim %d, K4V2" % (batch, chunk, cache_len, hq, hkv, d0),
        "ms": t, "prefill_tokens_per_s": batch * chunk / (t * 1e-3),
        "attention_tflops": flops / (t * 1e-3) / 1e12, "cache_bytes": cache_bytes,
        "cache_gbs_once": cache_bytes / (t * 1e-3) / 1e9,
    }


def _time_fp16_baseline(torch, kv, S, stream, peak, reps=20, tail=64):
    """Packed-cache decode against the uncompressed fp16 paged decode on the same lengths.

    Both kernels run alone, back to back, on the decode workload's sequences with `tail` extra
    tokens each (a partial tile for the packed cache, a partly filled last page for fp16); both
    caches are larger than L2 (0.5 GB packed, 2.3 GB fp16)."""
    dev = torch.device("cuda")
    lens = (S["lens0"] + tail).to(torch.int32)
    pages = ((lens + 127) // 128).tolist()
    n_pool = sum(pages)
    g = torch.Generator(device=dev)
    g.manual_seed(SEED + 5)
    pool = torch.randn((n_pool, HKV, 2, 128, D0), generator=g, device=dev).half()
    table = torch.zeros((BATCH, max(pages)), dtype=torch.int32)
    perm = torch.randperm(n_pool, generator=torch.Generator().manual_seed(SEED + 6)).to(torch.int32)
    off = 0
    for b in range(BATCH):
        table[b, :pages[b]] = perm[off:off + pages[b]]
        off += pages[b]
    table = table.to(dev)
    lens_d = lens.to(dev)
    q = S["qs"][0]
    out = torch.empty_like(S["out"])
    ws = kv.alloc_fp16_workspace(D0, BATCH, HQ, table.shape[1], device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def fp16_call():
        kv.fp16_decode_attention(HKV, q, pool, table, lens_d, out, ws, softmax_scale=1 / math.sqrt(D0),
                                 status=status, stream=stream)

    def kvarn_call():
        kv.decode_attention(S["desc"], q, S["pool"], S["table"], lens_d, out, S["ws"],
                            partial_k=S["pk"], partial_v=S["pv"], softmax_scale=1 / math.sqrt(D0),
                            status=status, stream=stream)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    f_ms = timed(fp16_call)
    k_ms = timed(kvarn_call)
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in the fp16 comparison" % int(status.item()))
    tokens = int(lens.sum())
    f_bytes = tokens * HKV * D0 * 2 * 2 + 2 * BATCH * HQ * D0 * 2
    k_bytes = _decode_bytes(lens.tolist(), S["rec_bytes"])
    del pool
    torch.cuda.empty_cache()
    return {
        "workload": "the decode workload's %d sequences at their lengths + %d tokens, alone, back to "
                    "back (%d launches each)" % (BATCH, tail, reps),
        "fp16_us": f_ms * 1e3, "fp16_tokens_per_s": tokens / (f_ms * 1e-3),
        "fp16_hbm_gbs": f_bytes / (f_ms * 1e-3) / 1e9, "fp16_frac": f_bytes / (f_ms * 1e-3) / 1e9 / peak,
        "fp16_bytes": f_bytes,
        "kvarn_us": k_ms * 1e3, "kvarn_tokens_per_s": tokens / (k_ms * 1e-3),
        "kvarn_hbm_gbs": k_bytes / (k_ms * 1e-3) / 1e9, "kvarn_bytes": k_bytes,
        "speedup_vs_fp16": f_ms / k_ms, "cache_bytes_ratio": f_bytes / k_bytes,
    }


def _time_long_stream(torch, kv, synth, d0, peak, steps=512, batch=4, hq=32, hkv=8, seed=5):
    """Streaming decode at long context: `steps` steps of append + decode for `batch` sequences
    starting at 130560 + {0, 1, 64, 127} tokens (1020 sealed pages each plus an open tile),
    head_dim d0 (96 is zero-padded to 128); every tile that fills seals into a packed page inside
    the timed steps.  The steps run twice from the same state: the first pass warms up, the
    second (which rewrites the same sealed pages with the same bytes) is timed."""
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    desc = kv.desc_from_preset(d0, hkv)
    rec = desc.page_record_bytes
    starts = torch.tensor([130560, 130561, 130624, 130687][:batch], dtype=torch.int64)
    sealed0 = starts // 128
    width = int((starts.max() + steps) // 128) + 1
    n_pool = batch * width
    g = torch.Generator().manual_seed(seed)
    table = torch.randperm(n_pool, generator=g).view(batch, width).to(torch.int32)
    pool = kv.alloc_pool(desc, n_pool, device=dev)  # before the temporaries, as in the layered runs
    k, v = synth.outlier_kv(int(sealed0.sum()) * 128, hkv, d0, seed=seed, device=dev)
    ids = torch.cat([table[b, :int(sealed0[b])] for b in range(batch)]).to(dev)
    kv.quantize_tiles(desc, k, v, ids, pool)
    del k, v
    kp, vp = synth.outlier_kv(batch * 128, hkv, d0, seed=seed + 1, device=dev)
    rows = (torch.arange(128, device=dev)[None, :] < (starts % 128).to(dev)[:, None]).to(torch.float16)
    pk0 = (kp.view(batch, 128, hkv, d0).transpose(1, 2) * rows[:, None, :, None]).contiguous()
    pv0 = (vp.view(batch, 128, hkv, d0).transpose(1, 2) * rows[:, None, :, None]).contiguous()
    pk, pv = pk0.clone(), pv0.clone()
    gd = torch.Generator(device=dev)
    gd.manual_seed(seed + 2)
    qs = [torch.randn((batch, hq, d0), generator=gd, device=dev).half() for _ in range(4)]
    kn = [torch.randn((batch, hkv, d0), generator=gd, device=dev).half() for _ in range(4)]
    vn = [torch.randn((batch, hkv, d0), generator=gd, device=dev).half() for _ in range(4)]
    lens = [torch.empty(batch, dtype=torch.int32, device=dev) for _ in range(2)]
    out = torch.empty((batch, hq, d0), dtype=torch.float16, device=dev)
    table = table.to(dev)
    ws = kv.alloc_workspace(desc, batch, hq, width, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(d0)
    every = 5
    for rep in range(2):
        lens[0].copy_(starts.to(torch.int32))
        pk.copy_(pk0)
        pv.copy_(pv0)
        ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(0, steps, every)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        torch.cuda._sleep(200000)  # the host enqueues the first steps while the GPU waits
        t0.record(stream)
        for i in range(steps):
            c = i % 2
            kv.append_token(desc, kn[i % 4], vn[i % 4], pk, pv, lens[c], table, pool,
                            seq_lens_out=lens[1 - c], status=status, stream=stream)
            dargs = (desc, qs[i % 4], pool, table, lens[1 - c], out, ws)
            dkw = dict(partial_k=pk, partial_v=pv, softmax_scale=scale, status=status, stream=stream)
            if i % every == 0:  # decode_kernel and combine_kernel as two calls, events around
                e = ev[i // every]
                e[0].record(stream)
                kv.decode_attention(*dargs, phase="partials", **dkw)
                e[1].record(stream)
                kv.decode_attention(*dargs, phase="combine", **dkw)
                e[2].record(stream)
            else:
                kv.decode_attention(*dargs, **dkw)
        t1.record(stream)
        torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status %d in the long-context stream" % int(status.item()))
    total_ms = t0.elapsed_time(t1)
    dec_ms = [a.elapsed_time(b) for a, b, _ in ev]
    call_ms = [a.elapsed_time(c) for a, _, c in ev]
    d_pad = desc.head_dim_padded
    new_tok = 2 * batch * hkv * d0 * 2            # k_new + v_new
    dec_bytes, step_bytes, seals = [], 0, 0
    for i in range(steps):
        L = starts + i + 1                          # lengths the step's decode attends to
        sealed = int((L // 128).sum())
        part = int((L % 128).sum())
        db = sealed * hkv * rec + part * hkv * d0 * 2 * 2 + 2 * batch * hq * d0 * 2  # the call
        n_seal = int(((starts + i) % 128 == 127).sum())   # tiles that fill in this step's append
        seals += n_seal
        ab = 2 * new_tok + n_seal * hkv * (2 * 128 * d0 * 2 + rec)  # read + write the token; seal
        step_bytes += db + ab
        if i % every == 0:
            dec_bytes.append(sealed * hkv * rec + batch * hq * d0 * 2)  # decode_kernel: pages + q
    dec_gbs = statistics.mean(dec_bytes) / (statistics.mean(dec_ms) * 1e-3) / 1e9
    step_gbs = step_bytes / (total_ms * 1e-3) / 1e9
    del pool, ws
    torch.cuda.empty_cache()
    return {
        "workload": "%d steps of append + decode, batch %d from %s tokens, %d q heads / %d kv heads, "
                    "head_dim %d (padded %d), K4V2; %d tiles sealed inside the timed steps"
                    % (steps, batch, "/".join(str(int(x)) for x in starts), hq, hkv, d0, d_pad,
                       seals * hkv),
        "us_per_step": total_ms * 1e3 / steps,
        "algorithmic_bytes_per_step": step_bytes / steps,
        "hbm_gbs": step_gbs, "frac": step_gbs / peak,
        "decode_us": statistics.mean(dec_ms) * 1e3, "decode_hbm_gbs": dec_gbs, "decode_frac": dec_gbs / peak,
        "decode_call_us": statistics.mean(call_ms) * 1e3,
        "decode_duration_source": "CUDA events around decode_kernel (decode_us) and around the whole "
                                  "decode call with the merge (decode_call_us) on every %dth step" % every,
        "kv_tokens_per_s": sum(int((starts + i + 1).sum()) for i in range(steps)) / (total_ms * 1e-3),
    }


def _decode_configs(torch, kv, synth, peak, args):
    """The 32B-class 64-layer decode step and the long-context shapes, each against bytes/peak."""
    res = {}
    for key, group, cfg in (
            ("decode_32b_step", "32b", dict(batch=32, seq_len=16384, hq=64, hkv=8, d0=128, layers=64, seed=4)),
            ("decode_32b_8_layers_tcgen05", "32b", dict(batch=32, seq_len=16384, hq=64, hkv=8, d0=128, layers=8,
                                                        seed=4, kernel="tc")),
            ("decode_long_d256", "long", dict(batch=4, seq_len=131072, hq=32, hkv=8, d0=256, layers=1, seed=5)),
            ("decode_long_d96", "long", dict(batch=4, seq_len=131072, hq=32, hkv=8, d0=96, layers=1, seed=5)),
            ("preset_kvarn_k4v2_g128", "presets", dict(batch=64, seq_len=8704, hq=32, hkv=8, d0=128, layers=1,
                                                       seed=6, preset="kvarn_k4v2_g128")),
            ("preset_kvarn_k4v4_g128", "presets", dict(batch=64, seq_len=8704, hq=32, hkv=8, d0=128, layers=1,
                                                       seed=6, preset="kvarn_k4v4_g128")),
            ("preset_kvarn_k2v2_g128", "presets", dict(batch=64, seq_len=8704, hq=32, hkv=8, d0=128, layers=1,
                                                       seed=6, preset="kvarn_k2v2_g128")),
            ("preset_kvarn_k8v4_g128", "presets", dict(batch=64, seq_len=8704, hq=32, hkv=8, d0=128, layers=1,
                                                       seed=6, preset="kvarn_k8v4_g128"))):
        if args.extras not in ("all", group):
            continue
        if args.extra_batch:
            cfg["batch"] = args.extra_batch
        if args.extra_layers and cfg["layers"] > 1:
            cfg["layers"] = args.extra_layers
        ms, nbytes = _time_decode_layers(torch, kv, synth, **cfg)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[key] = {
            "workload": "%d layer(s) x batch %d at %d tokens, %d q heads / %d kv heads, head_dim %d, %s%s"
                        % (cfg["layers"], cfg["batch"], cfg["seq_len"], cfg["hq"], cfg["hkv"], cfg["d0"],
                           cfg.get("preset", "kvarn_k4v2_g128"),
                           ", tcgen05 kernel" if cfg.get("kernel") == "tc" else ""),
            "ms_per_step": ms, "algorithmic_bytes": nbytes, "hbm_gbs": gbs, "frac": gbs / peak,
            "ideal_ms_at_peak": nbytes / (peak * 1e9) * 1e3,
            "kv_tokens_per_s": cfg["batch"] * cfg["seq_len"] / (ms * 1e-3),
        }
    if args.extras in ("all", "long"):
        for d0 in (256, 96):
            res["decode_long_stream_d%d" % d0] = _time_long_stream(torch, kv, synth, d0, peak)
    return res


def _run_kvarn(args, torch, world, rank):
    from calibration_free_kv_gb300 import build as kbuild
    kbuild.build()
    from calibration_free_kv_gb300 import kvarn as kv
    from calibration_free_kv_gb300 import synth

    dev = torch.device("cuda")
    S = _setup_decode(torch, kv, synth, 2 * args.warmup + 2 * args.steps + 4)
    stream = torch.cuda.current_stream()
    state = {"cur": 0, "step": 0}

    def step(q=None, kn=None, vn=None, ev=None, out=None):
        i = state["step"] % len(S["qs"])
        q = S["qs"][i] if q is None else q
        kn = S["kn"][i] if kn is None else kn
        vn = S["vn"][i] if vn is None else vn
        c = state["cur"]
        kv.append_token(S["desc"], kn, vn, S["pk"], S["pv"], S["lens"][c], S["table"], S["pool"],
                        seq_lens_out=S["lens"][1 - c], status=S["status"], stream=stream)
        args = (S["desc"], q, S["pool"], S["table"], S["lens"][1 - c], S["out"] if out is None else out,
                S["ws"])
        kw = dict(partial_k=S["pk"], partial_v=S["pv"], softmax_scale=1 / math.sqrt(D0),
                  status=S["status"], stream=stream)
        if ev is None:
            kv.decode_attention(*args, **kw)
        else:  # the same two kernels as two calls, an event between them
            ev[0].record(stream)
            kv.decode_attention(*args, phase="partials", **kw)
            ev[1].record(stream)
            kv.decode_attention(*args, phase="combine", **kw)
            ev[2].record(stream)
        state["cur"] = 1 - c
        state["step"] += 1

    # The decode call's own duration is sampled live on at most DEC_EVENT_SAMPLES evenly spaced
    # timed steps, at most one in DEC_EVENT_EVERY_MIN: an event recorded between append and
    # decode ends their programmatic-launch overlap, so the other steps run without it.
    every = max(DEC_EVENT_EVERY_MIN, args.steps // DEC_EVENT_SAMPLES)
    sampled = [i for i in range(args.steps) if i % every == 0]
    dec_ev = {i: tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for i in sampled}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # the clock sampler starts before the warm-up: its start-up wait (0.3 s for nvidia-smi's
    # first samples) left the GPU idle between the warm-up and the timed steps, and a short
    # timed window then began cold (20 steps: decode_kernel 101 us against 93 us at the same
    # lengths in a 200-step window)
    clocks = ClockSampler(_device_id(torch))
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    lens_before = S["lens"][state["cur"]].to(torch.int64).cpu()
    w0 = clocks.mark()
    t0.record(stream)
    for i in range(args.steps):
        step(ev=dec_ev.get(i))
    t1.record(stream)
    torch.cuda.synchronize()
    w1 = clocks.mark()
    clk = clocks.stop(window=(w0, w1))
    elapsed_ms = t0.elapsed_time(t1)
    dec_ms = [a.elapsed_time(b) for a, b, _ in dec_ev.values()]      # decode_kernel
    call_ms = [a.elapsed_time(c) for a, _, c in dec_ev.values()]     # decode_kernel + combine_kernel
    status = int(S["status"].item())
    if status != 0:
        raise RuntimeError("device status %d during the timed steps" % status)

    # attended tokens per step: lengths after each step's append
    tokens = sum(int(lens_before.sum()) + BATCH * (i + 1) for i in range(args.steps))
    dec_bytes = [_decode_kernel_bytes((lens_before + i + 1).tolist(), S["rec_bytes"]) for i in sampled]
    call_bytes = [_decode_bytes((lens_before + i + 1).tolist(), S["rec_bytes"]) for i in sampled]
    peak, peak_kind = _peaks()
    avg_dec = statistics.mean(dec_ms)
    avg_call = statistics.mean(call_ms)
    achieved = statistics.mean(dec_bytes) / (avg_dec * 1e-3) / 1e9

    # ---- end to end through the public API: pinned host q/k/v in, fp16 out back each step.
    # As a serving loop would, the copies run on their own stream: step i+1's inputs (one
    # pinned buffer holding q, k_new, v_new) go up and step i-1's output comes down while step
    # i computes; inputs and outputs are double-buffered and ordered by events.
    h_in = [torch.cat([S["qs"][j].flatten(), S["kn"][j].flatten(), S["vn"][j].flatten()]).cpu().pin_memory()
            for j in range(len(S["qs"]))]
    h_out = [torch.empty((BATCH, HQ, D0), dtype=torch.float16).pin_memory() for _ in range(2)]
    d_in = [torch.empty_like(h_in[0], device=dev) for _ in range(2)]
    d_out = [torch.empty((BATCH, HQ, D0), dtype=torch.float16, device=dev) for _ in range(2)]
    nq, nk = S["qs"][0].numel(), S["kn"][0].numel()
    views = [(b[:nq].view(S["qs"][0].shape), b[nq:nq + nk].view(S["kn"][0].shape),
              b[nq + nk:].view(S["vn"][0].shape)) for b in d_in]
    copy = torch.cuda.Stream()
    e_steps = args.steps
    up = [torch.cuda.Event() for _ in range(e_steps)]        # inputs of step i on the device
    done = [torch.cuda.Event() for _ in range(e_steps)]      # step i computed
    down = [torch.cuda.Event() for _ in range(e_steps)]      # output of step i on the host
    # the same W warm-up steps as before the timed steps, after the host-side set-up above, so
    # that the end-to-end steps do not begin on an idle GPU
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    lens_e = S["lens"][state["cur"]].to(torch.int64).cpu()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy.wait_stream(stream)
    with torch.cuda.stream(copy):
        d_in[0].copy_(h_in[0], non_blocking=True)
        up[0].record(copy)
    for i in range(e_steps):
        if i + 1 < e_steps:  # next inputs, once step i-1 no longer reads that buffer
            with torch.cuda.stream(copy):
                if i >= 1:
                    copy.wait_event(done[i - 1])
                d_in[(i + 1) % 2].copy_(h_in[(i + 1) % len(h_in)], non_blocking=True)
                up[i + 1].record(copy)
        stream.wait_event(up[i])
        if i >= 2:  # step i-2's output has left d_out[i % 2]
            stream.wait_event(down[i - 2])
        q_i, k_i, v_i = views[i % 2]
        step(q=q_i, kn=k_i, vn=v_i, out=d_out[i % 2])
        done[i].record(stream)
        with torch.cuda.stream(copy):
            copy.wait_event(done[i])
            h_out[i % 2].copy_(d_out[i % 2], non_blocking=True)
            down[i].record(copy)
    stream.wait_event(down[e_steps - 1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_tokens = sum(int(lens_e.sum()) + BATCH * (i + 1) for i in range(e_steps))

    # ---- quantise throughput: one layer, 8 KV heads x 16384 tokens x head_dim 128
    q_med, q_bytes = _time_quantize(torch, kv, synth, dev, stream)
    q_gbs = q_bytes / (q_med * 1e-3) / 1e9
    a_ms, _, a_iters = _time_quantize(torch, kv, synth, dev, stream, reps=10, tol=ADAPTIVE_TOL)
    q_adaptive = {"sinkhorn_tol": ADAPTIVE_TOL, "us": a_ms * 1e3, "tokens_per_s": Q_TOKENS / (a_ms * 1e-3),
                  "mean_iterations": a_iters, "max_iterations": 4}
    q_telemetry = _time_error_telemetry(torch, kv, synth, dev, stream)
    q_dims = {}
    for d0 in (64, 256):  # the CUDA-core rotation path (head_dim 64 and 256)
        ms, nb = _time_quantize(torch, kv, synth, dev, stream, reps=10, d0=d0)
        q_dims["head_dim_%d" % d0] = {"us": ms * 1e3, "tokens_per_s": Q_TOKENS / (ms * 1e-3),
                                      "algorithmic_bytes": nb, "hbm_gbs": nb / (ms * 1e-3) / 1e9,
                                      "frac": nb / (ms * 1e-3) / 1e9 / peak}
    q_presets = {}
    if args.extras in ("all", "presets"):
        for name in ("kvarn_k4v4_g128", "kvarn_k2v2_g128", "kvarn_k8v4_g128"):
            ms, nb = _time_quantize(torch, kv, synth, dev, stream, preset=name, reps=10)
            q_presets[name] = {"us": ms * 1e3, "tokens_per_s": Q_TOKENS / (ms * 1e-3),
                               "hbm_gbs": nb / (ms * 1e-3) / 1e9}
    # Quantisation is bound by fp32 arithmetic, not by HBM.  Per element it needs 38 fp32 ops:
    # 4 in each of the 8 std steps (product with the other axis' factor, its share of the
    # pairwise sum, minus the half-line mean, square-accumulate), 3 for the group extremes
    # (product, min, max) and 3 to quantise (product with the row factor, fused product with the
    # column factor minus the zero point, fused product with 1/s plus the rounding constant).
    # Peak: one fp32 op per lane per clock, 128 lanes per SM.
    q_elems = 2 * Q_TOKENS * Q_HEADS * D0
    q_ops = QUANT_OPS_PER_ELEMENT * q_elems / (q_med * 1e-3) / 1e9
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    # ---- the 32B-class step (64 layers, GQA 8) and the long-context shapes (not timed steps)
    extra = _decode_configs(torch, kv, synth, peak, args)
    if args.extras in ("all", "prefill"):
        extra["prefill"] = _time_prefill(torch, kv, synth)
    if args.extras in ("all", "fp16"):
        extra["fp16_baseline"] = _time_fp16_baseline(torch, kv, S, stream, peak)
    quality = _quality(torch, kv, synth)

    # ---- aggregate over ranks (replicas)
    (elapsed_ms, e2e_ms), (value, e2e_value) = _aggregate_over_ranks(
        torch, world, [elapsed_ms, e2e_ms], [tokens, e2e_tokens], dev)
    if rank != 0:
        return None
    return {
        "metric": METRIC,
        "value": value,
        "unit": "KV tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "dtype_detail": "fp16 MMA operands (exact integer codes, hi+lo split scales) with f32 "
                        "accumulation; f32 quantisation; u4/u2 packed cache",
        "data": "synthetic (outlier generator: N(0,1), 4 channels x20-50 per head, lognormal token "
                "scales; seeds 3 and 2)",
        "config": _workload_config(lens_before, args.steps),
        "decode_hbm_gbs": achieved,
        "decode_us": avg_dec * 1e3,
        "decode_call": {"us": avg_call * 1e3,
                        "algorithmic_bytes": statistics.mean(call_bytes),
                        "hbm_gbs": statistics.mean(call_bytes) / (avg_call * 1e-3) / 1e9,
                        "frac": statistics.mean(call_bytes) / (avg_call * 1e-3) / 1e9 / peak,
                        "note": "kvarn_decode_attention as a whole: decode_kernel + combine_kernel "
                                "(the raw open tiles, the merge of the splits and the inverse "
                                "rotation)"},
        "roofline": {
            "kernel": "decode_kernel (kvarn_decode_partials)",
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback 6.8 TB/s",
            "traffic": (None if _decode_traffic_ratio() is None
                        else _decode_traffic_ratio() * statistics.mean(dec_bytes)),
            "traffic_source": "ncu dram__bytes_read+write of one decode_kernel launch at batch 24 "
                              "(DECODE_TRAFFIC), scaled by algorithmic bytes; null when decode.cu "
                              "or decode_util.cuh changed since that capture",
            "algorithmic_bytes_per_launch": statistics.mean(dec_bytes),
            "duration_source": "CUDA events on the launching stream around decode_kernel (the "
                               "decode call as kvarn_decode_partials + kvarn_decode_combine, an "
                               "event between them) on every %dth timed step (%d of %d)"
                               % (every, len(dec_ms), args.steps),
        },
        "quantize": {
            "workload": "one layer, 8 KV heads x 16384 tokens x head_dim 128 (K and V), L2 flushed",
            "tokens_per_s": Q_TOKENS / (q_med * 1e-3),
            "us": q_med * 1e3, "hbm_gbs": q_gbs, "frac": q_gbs / peak,
            "algorithmic_bytes": q_bytes,
            "other_presets": q_presets,
            "other_head_dims": q_dims,
            "error_telemetry": q_telemetry,
            "adaptive_stop": q_adaptive,
            "roofline": {
                "kernel": "quantize_tc_kernel", "bound": "alu", "achieved": q_ops,
                "peak": sms * 128 * (clk.get("sm_mhz") or SM_MAX_MHZ) * 1e-3, "unit": "Gop/s",
                "frac": q_ops / (sms * 128 * (clk.get("sm_mhz") or SM_MAX_MHZ) * 1e-3),
                "peak_source": "%d SMs x 128 fp32 lanes x median SM clock under load" % sms,
                "ops_per_element": QUANT_OPS_PER_ELEMENT,
            },
        },
        **extra,
        "quality": quality,
        "e2e": {"value": e2e_value, "unit": "KV tokens/s",
                "h2d_bytes_per_step": (BATCH * HQ * D0 + 2 * BATCH * HKV * D0) * 2,
                "d2h_bytes_per_step": BATCH * HQ * D0 * 2},
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
    }


# ------------------------------------------------------------------------------------------------
# CPU oracle (baseline) arm
# ------------------------------------------------------------------------------------------------

_ORACLE_UNITS = None


def _oracle_units(seed: int, n_units: int = 4, max_pages=None):
    """(q rows, oracle page records, L) of n_units (sequence, kv head) decode units of the
    workload, quantised by the oracle (not timed); with max_pages, each unit keeps its first
    max_pages pages (a shorter sequence of the same data)."""
    import numpy as np
    from calibration_free_kv_gb300 import synth
    from oracle import kvarn_oracle as ko

    shape = synth.decode_batch(BATCH, HQ, HKV, D0, seed=seed, min_pages=MIN_PAGES, max_pages=MAX_PAGES)
    lens = shape["seq_lens"].tolist()
    q = shape["q"].double().numpy()
    group = HQ // HKV
    units = []
    for b in range(n_units):
        L = lens[b]
        k, v = synth.outlier_kv(L, 1, D0, seed=seed * 7 + b)
        n = L // 128
        kq = ko.quantize_tile(k[:, 0].double().numpy().reshape(n, 128, D0), "K")
        vq = ko.quantize_tile(v[:, 0].double().numpy().reshape(n, 128, D0), "V")
        fields = ("codes", "scale", "zero", "factor")
        recs = [ko.pack_record({f: kq[f][i] for f in fields}, {f: vq[f][i] for f in fields})
                for i in range(n)]
        if max_pages is not None and len(recs) > max_pages:
            recs, L = recs[:max_pages], 128 * max_pages
        units.append((np.ascontiguousarray(q[b, :group]), recs, L))
    return units


def _oracle_init(units):
    global _ORACLE_UNITS
    _ORACLE_UNITS = units


def _oracle_work(seconds: float):
    """Decode the prepared units through the float64 oracle for `seconds`: (KV token-heads, s)."""
    from oracle import kvarn_oracle as ko
    tokens, i = 0, 0
    t0 = time.perf_counter()
    while True:
        q, recs, L = _ORACLE_UNITS[i % len(_ORACLE_UNITS)]
        ko.decode_sequence(q, recs, None, None, 1 / math.sqrt(D0), D0)
        tokens += L
        i += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return tokens, el


class OracleTimer:
    """The float64 oracle's decode attention timed on the host cores: one spawned process per
    core (single-threaded BLAS each), or one process alone."""

    def __init__(self, seed: int = SEED, max_pages=None):
        import multiprocessing as mp
        self.max_pages = max_pages
        self.units = _oracle_units(seed, max_pages=max_pages)
        self.cores = os.cpu_count() or 1
        keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
        saved = {k: os.environ.get(k) for k in keys}
        for k in keys:
            os.environ[k] = "1"
        try:
            ctx = mp.get_context("spawn")
            self.pool = ctx.Pool(self.cores, initializer=_oracle_init, initargs=(self.units,))
            self.pool.map(_oracle_work, [0.0] * self.cores)  # workers up and warm
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def run(self, seconds: float, cores: int):
        """KV tokens/s (all heads of a token) over `cores` processes working `seconds` each."""
        res = self.pool.map(_oracle_work, [seconds] * cores, chunksize=1)
        tokens = sum(t for t, _ in res)
        wall = max(e for _, e in res)
        return tokens / HKV / wall, wall

    def describe(self):
        pages = sum(len(r) for _, r, _ in self.units)
        which = ("whole" if self.max_pages is None else
                 "first-%d-page (short steps)" % self.max_pages)
        return ("%d %s (sequence, kv head) decode units of the workload (%d pages, 4 query heads "
                "each), decoded repeatedly through the float64 oracle (dequantise + textbook "
                "attention), one single-threaded process per core" % (len(self.units), which, pages))

    def close(self):
        self.pool.close()
        self.pool.join()


def _cpu_baseline(seconds: float):
    ot = OracleTimer()
    try:
        v_all, _ = ot.run(seconds / 2, ot.cores)
        v_one, _ = ot.run(seconds / 2, 1)
    finally:
        ot.close()
    return {"value": v_all, "unit": "KV tokens/s", "cores": ot.cores, "kind": "oracle",
            "value_1core": v_one, "sample": ot.describe() + "; %.1f s on all cores, %.1f s on one"
            % (seconds / 2, seconds / 2)}


def _run_reference(args, world, rank):
    if rank != 0:
        return None
    # about a minute of oracle work in all: 1 s a step for short runs, down to one decode unit
    # a step (a few tens of ms) when many steps are asked for
    per_step = min(1.0, max(0.02, 60.0 / max(1, args.steps + args.warmup)))
    # a whole unit (tens of pages) takes a few tenths of a second: short steps take 4-page units
    ot = OracleTimer(max_pages=None if per_step >= 0.5 else 4)
    try:
        for _ in range(args.warmup):
            ot.run(per_step * 0.25, ot.cores)
        vals, total_t = [], 0.0
        for i in range(args.steps):
            v, t = ot.run(per_step, ot.cores)
            vals.append(v)
            total_t += t
    finally:
        ot.close()
    descs = [ot.describe()]
    value = statistics.mean(vals)
    cores = ot.cores
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "KV tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (outlier generator)",
        "config": _workload_config(_initial_lens() + args.warmup, args.steps),
        "cpu_baseline": {"value": value, "unit": "KV tokens/s", "cores": cores, "kind": "oracle",
                         "sample": descs[0] if descs else ""},
        "e2e": {"value": value, "unit": "KV tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("kvarn", "reference"), default="kvarn")
    ap.add_argument("--batch", type=int, default=64,
                    help="decode batch (64 = the benchmark workload; smaller only for profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="CPU work of the oracle baseline sample (kvarn arm)")
    ap.add_argument("--extras", choices=("all", "none", "32b", "long", "presets", "prefill", "fp16"), default="all",
                    help="which extra measurements to take: the 64-layer and long-context decode "
                         "shapes, other presets, prefill, the fp16 paged decode baseline")
    ap.add_argument("--extra-batch", type=int, default=0,
                    help="batch of those shapes (0 = the workload's; smaller only for profiling)")
    ap.add_argument("--extra-layers", type=int, default=0,
                    help="layers of the 32B-class step (0 = 64; fewer only for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    global BATCH
    BATCH = args.batch
    world, rank, local = _dist_env()

    if args.impl == "reference":
        if world > 1 and rank != 0:
            return
        res = _run_reference(args, world, rank)
        if res is not None:
            print(json.dumps(res))
        return

    import torch
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    res = _run_kvarn(args, torch, world, rank)
    if rank == 0 and res is not None:
        res["cpu_baseline"] = _cpu_baseline(args.cpu_seconds)
        print(json.dumps(res))
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
