"""Shared comparison helpers for the GPU parity tests (oracle on the CPU side).

Tolerances (stated once, used by every GPU test):
  * codes: bit-exact, except codes whose oracle float64 pre-round value lies within 1e-5 of
    a k+0.5 boundary; those may differ by one level, and at most 1e-4 of all codes may.
    Both figures grow with (2^b - 1) / 15 above 4 bits: the kernel's fp32 pre-round value
    (N - m) / s with s = (M - m) / (2^b - 1) moves by (2^b - 1) eps for an fp32 error of
    eps (M - m) in N or m, so its band around a boundary widens with the level count.
  * stored fp16 scale / zero / factor: within one fp16 ulp of the oracle's.
  * dequantised fp16 values: |gpu - oracle| <= 1e-3 |oracle| + 1e-5 max|tile| (same bytes).
  * decode output (fp16): |gpu - oracle| <= 2e-3 max(1, max_j |oracle_j|) per query head.
"""

from __future__ import annotations

import math

import numpy as np
import torch

from oracle import kvarn_oracle as ko

CODE_BOUNDARY = 1e-5
CODE_MISMATCH_FRACTION = 1e-4
DEQUANT_RTOL = 1e-3
DECODE_TOL = 2e-3


def oracle_quantize(k_tiles: np.ndarray, v_tiles: np.ndarray, iters: int = ko.SINKHORN_ITERS,
                    k_bits: int = ko.K_BITS, v_bits: int = ko.V_BITS):
    """k_tiles, v_tiles: [n, 128, d0] float arrays -> (records list, kq dict, vq dict) batched."""
    d = ko.padded_head_dim(k_tiles.shape[-1])
    kq = ko.quantize_tile(k_tiles, "K", d, iters, bits=k_bits)
    vq = ko.quantize_tile(v_tiles, "V", d, iters, bits=v_bits)
    fields = ("codes", "scale", "zero", "factor")
    recs = []
    for i in range(k_tiles.shape[0]):
        recs.append(ko.pack_record(dict({key: kq[key][i] for key in fields}, bits=k_bits),
                                   dict({key: vq[key][i] for key in fields}, bits=v_bits)))
    return recs, kq, vq


def tile_of(q: dict, i: int) -> dict:
    """Tile i of a batched quantize_tile result (arrays sliced, the scalar code width kept)."""
    return {key: (val if key == "bits" else val[i]) for key, val in q.items()}


def record_bytes_of(pool: torch.Tensor, page: int, head: int) -> bytes:
    return bytes(pool[page, head].cpu().numpy().tobytes())


def _width_factor(bits: int) -> float:
    return max(1.0, ((1 << bits) - 1) / 15.0)


def compare_codes(gpu_codes, ora_codes, ora_pre, bits: int = 4):
    """Returns (mismatches, total, allowed mismatches); asserts every mismatch is an exempt
    boundary case."""
    g = np.asarray(gpu_codes).astype(np.int64)
    o = np.asarray(ora_codes).astype(np.int64)
    bad = g != o
    n_bad = int(bad.sum())
    band = CODE_BOUNDARY * _width_factor(bits)
    if n_bad:
        pre = np.asarray(ora_pre)[bad]
        dist = np.abs(pre - (np.floor(pre) + 0.5))
        assert np.all(dist < band), (
            "code mismatch away from a rounding boundary: %s" % list(zip(pre[dist >= band][:5],
                                                                   g[bad][dist >= band][:5],
                                                                   o[bad][dist >= band][:5])))
        assert np.all(np.abs(g[bad] - o[bad]) == 1)
    return n_bad, g.size, CODE_MISMATCH_FRACTION * _width_factor(bits) * g.size


def assert_f16_within_ulp(gpu, ora, what):
    g = np.asarray(gpu, dtype=np.float16).astype(np.float64)
    o = np.asarray(ora, dtype=np.float16).astype(np.float64)
    ulp = np.maximum(np.spacing(np.abs(o).astype(np.float16)).astype(np.float64),
                     np.spacing(np.abs(g).astype(np.float16)).astype(np.float64))
    bad = np.abs(g - o) > ulp * 1.0001
    assert not bad.any(), "%s: %d values differ by more than 1 fp16 ulp, e.g. gpu %s oracle %s" % (
        what, int(bad.sum()), g[bad][:4], o[bad][:4])


def compare_record(gpu_rec: bytes, kq_i: dict, vq_i: dict, d: int, stats: list,
                   k_bits: int = ko.K_BITS, v_bits: int = ko.V_BITS):
    """Compare one GPU page record with the oracle's quantised K/V (dicts of one tile)."""
    gk, gv = ko.unpack_record(gpu_rec, d, k_bits, v_bits)
    stats.append(compare_codes(gk["codes"], kq_i["codes"], kq_i["pre"], k_bits))
    stats.append(compare_codes(gv["codes"], vq_i["codes"], vq_i["pre"], v_bits))
    for key in ("scale", "zero", "factor"):
        assert_f16_within_ulp(gk[key], kq_i[key], "K " + key)
        assert_f16_within_ulp(gv[key], vq_i[key], "V " + key)


def assert_mismatch_budget(stats):
    bad = sum(s[0] for s in stats)
    total = sum(s[1] for s in stats)
    allowed = sum(s[2] for s in stats)
    assert bad <= allowed, "%d of %d codes differ" % (bad, total)
    return bad, total


def assert_decode_close(gpu_out, ref, what=""):
    g = np.asarray(gpu_out, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    scale = np.maximum(1.0, np.abs(r).max(axis=-1, keepdims=True))
    err = np.abs(g - r) / scale
    assert np.all(np.isfinite(g)), what + ": non-finite output"
    assert err.max() <= DECODE_TOL, "%s: max scaled error %.3e" % (what, err.max())
    return float(err.max())


def upload_records(pool: torch.Tensor, page_head_recs):
    """Write oracle records into a device pool: iterable of (page, head, bytes)."""
    for page, head, rec in page_head_recs:
        pool[page, head] = torch.frombuffer(bytearray(rec), dtype=torch.uint8).to(pool.device)


def softmax_scale(d0: int) -> float:
    return 1.0 / math.sqrt(d0)
