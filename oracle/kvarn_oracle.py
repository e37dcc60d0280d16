"""Plain float64 CPU oracle for KVarN's K4V2 g128 KV-cache path (and the other k/v bit presets).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module.  The
product path (``calibration_free_kv_gb300``) never imports it, and this module
imports nothing from the product path: the two share no code.

Everything is numpy float64, written for a reader to check against the pages
by eye.  Sources, cited by page title and section:

[hotdry]  blog.hotdry.top, "KVarN Hadamard 旋转与方差归一化：KV-cache 量化的校准算法实现"
[aifeeds] ai-feeds.com, "KVarN: 方差归一化的KV-Cache量化缓解推理任务中的误差累积"
[vatt]    vatt-ghern.pages.dev, "KV cache 為什麼能壓到 4-bit／2-bit 還不掉準確度——從 variance
          normalization 講起"
[jdon]    jdon.com, "华为开源KV Cache量化技术让大模型上下文提升5倍！"

Per 128-token tile of one KV head, K and V separately:
  1. zero-pad head_dim to a power of two          [aifeeds §局限, "维度限制与填充开销"]
  2. rotate along head_dim: X = Z_pad . H / sqrt(d) [hotdry §Hadamard 旋转; vatt §四個步驟, Hadamard rotation]
  3. log-space Sinkhorn-style normalisation, channel std step then token std
     step, a fixed number of iterations           [hotdry §迭代方差归一化; vatt §四個步驟, iterative variance normalization]
  4. asymmetric round-to-nearest: K 4-bit per channel, V 2-bit per token (other presets:
     other widths, same steps)
                                                  [hotdry §非对称量化与尺度折叠; vatt §為什麼樸素的 2-bit…, worked example]
  5. normalisation factors folded into the stored scales ("scale folding")
                                                  [hotdry §非对称量化与尺度折叠; vatt §四個步驟, asymmetric quantization]
Decode attention is the textbook softmax attention over the dequantised cache
(plus the raw fp16 tokens of the unsealed partial tile), in the original basis.

Readings where the pages are silent:
  * Sylvester Hadamard in natural order, no random signs; scaled by 1/sqrt(d).
  * std is the population std (ddof 0, mean subtracted).  A row or column whose std is
    below EPS=1e-6 has nothing to normalise and keeps its factor (its log factor gains 0);
    dividing it by EPS instead would grow its factor by 1/EPS every iteration and overflow
    the fp16 metadata of constant or all-zero tiles.
  * one iteration = channel-std step then token-std step.
  * zero-point is the float group minimum; scale floor 1e-8; round half to even.
  * stored scales, zero-points and factors are IEEE binary16.
  * codes are computed from the unrounded float64 values.

Parity status of each function is stated in its docstring ("pinned by" names
the tests in tests/test_oracle.py that tie it to the pages or to mathematics).
"""

from __future__ import annotations

import numpy as np

TILE_TOKENS = 128          # one tile == one paged-attention block  [vatt §怎麼用, knob table: tile=128]
K_BITS = 4                 # preset kvarn_k4v2_g128                  [hotdry §核心配置参数]
V_BITS = 2
# Other presets run the same pipeline with other code widths [vatt §四個步驟, bit-width
# assignment: other k/v bit presets take the same path; vatt §怎麼用, key/value bits knobs].
# Reading: widths of 2, 4 and 8 bits on either side; tiles stay 128 tokens.
PRESETS = {"kvarn_k4v2_g128": (4, 2), "kvarn_k4v4_g128": (4, 4), "kvarn_k2v2_g128": (2, 2),
           "kvarn_k8v4_g128": (8, 4)}
CODE_BITS = (2, 4, 8)
SINKHORN_ITERS = 4         # typical count three to five             [hotdry §迭代方差归一化, step 3]
SINKHORN_EPS = 1e-6        # reading: stds below this are not normalised (pages give no value)
SCALE_FLOOR = 1e-8         # reading: quantiser step floor for constant groups


# ----------------------------------------------------------------------------
# 1-2. padding and rotation
# ----------------------------------------------------------------------------

def padded_head_dim(d0: int) -> int:
    """Next power of two >= d0.  [aifeeds §局限: a head_dim that is not a power of two is
    padded up to the nearest one]

    Pinned by: test_padded_head_dim.
    """
    if d0 < 1:
        raise ValueError("head_dim must be positive")
    d = 1
    while d < d0:
        d *= 2
    return d


def sylvester_hadamard(n: int) -> np.ndarray:
    """Sylvester construction H_1=[1], H_2m=[[H,H],[H,-H]]; entries +-1, H H^T = nI.

    [hotdry §Hadamard 旋转: elements only +-1, H H^T = nI]
    Pinned by: test_hadamard_matches_scipy, test_hadamard_orthogonality.
    """
    if n < 1 or n & (n - 1):
        raise ValueError("Hadamard order must be a power of two")
    h = np.ones((1, 1), dtype=np.float64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def zero_pad(z: np.ndarray, d: int) -> np.ndarray:
    """Zero-pad the last axis of z to length d.  [aifeeds §局限]"""
    z = np.asarray(z, dtype=np.float64)
    out = np.zeros(z.shape[:-1] + (d,), dtype=np.float64)
    out[..., : z.shape[-1]] = z
    return out


def rotate(z: np.ndarray, d: int) -> np.ndarray:
    """X = pad(Z) . H_d / sqrt(d) along the last (head_dim) axis, as a dense product.

    Orthonormal: inner products and norms are preserved and applying it twice
    gives back the input.  [hotdry §Hadamard 旋转; vatt §四個步驟, Hadamard rotation:
    orthonormal, attention inner products unchanged]
    Pinned by: test_rotation_* (norm, inner product, involution, fast transform,
    single-outlier spread).
    """
    return zero_pad(z, d) @ sylvester_hadamard(d) / np.sqrt(d)


# ----------------------------------------------------------------------------
# 3. log-space Sinkhorn-style variance normalisation
# ----------------------------------------------------------------------------

def sinkhorn_normalise(x: np.ndarray, iters: int = SINKHORN_ITERS,
                       eps: float = SINKHORN_EPS, tol: float = 0.0, return_iters: bool = False):
    """Alternate channel-std and token-std normalisation with log-space factors.

    x: [..., T, d] rotated tile (tokens x channels).  Keeps log row factors lr[T]
    and log column factors lc[d].  Each iteration:
      column step: sigma_j = std_i(x_ij e^{-lr_i - lc_j}); lc_j += ln sigma_j if sigma_j >= eps
      row step:    sigma_i = std_j(x_ij e^{-lr_i - lc_j}); lr_i += ln sigma_i if sigma_i >= eps
    Returns N = x / (r_i c_j), r = e^{lr}, c = e^{lc} (and the iterations each tile used
    when return_iters).
    With tol > 0 a tile stops after the first iteration in which no log factor moved by
    more than tol (reading of the typical count of three to five and of the alternation approaching a
    fixed point; at most `iters` iterations either way).
    [hotdry §迭代方差归一化 steps 1-3 and the log-space paragraph;
     vatt §四個步驟, the Sinkhorn paragraph: column then row, log domain, alternate until
     both directions balance]
    Pinned by: test_sinkhorn_closed_form, test_sinkhorn_final_rows_unit_std,
    test_sinkhorn_converges, test_sinkhorn_invariances, test_adaptive_stop_*.
    """
    x = np.asarray(x, dtype=np.float64)
    lr = np.zeros(x.shape[:-1], dtype=np.float64)
    lc = np.zeros(x.shape[:-2] + x.shape[-1:], dtype=np.float64)
    active = np.ones(x.shape[:-2], dtype=bool)
    used = np.zeros(x.shape[:-2], dtype=np.int64)
    for _ in range(iters):
        if not active.any():
            break
        cur = x * np.exp(-lr[..., :, None] - lc[..., None, :])
        sigma_c = cur.std(axis=-2)
        dc = np.where(active[..., None], np.log(np.where(sigma_c >= eps, sigma_c, 1.0)), 0.0)
        lc = lc + dc
        cur = x * np.exp(-lr[..., :, None] - lc[..., None, :])
        sigma_r = cur.std(axis=-1)
        dr = np.where(active[..., None], np.log(np.where(sigma_r >= eps, sigma_r, 1.0)), 0.0)
        lr = lr + dr
        used = used + active
        if tol > 0:
            change = np.maximum(np.abs(dc).max(axis=-1), np.abs(dr).max(axis=-1))
            active = active & (change > tol)
    r = np.exp(lr)
    c = np.exp(lc)
    n = x / (r[..., :, None] * c[..., None, :])
    if return_iters:
        return n, r, c, used
    return n, r, c


# ----------------------------------------------------------------------------
# 4. asymmetric round-to-nearest
# ----------------------------------------------------------------------------

def rtn_asymmetric(x: np.ndarray, bits: int, axis: int):
    """Asymmetric RTN over groups along `axis`.

    m = min, M = max, s = max((M-m)/(2^b-1), floor), q = clip(rint((x-m)/s), 0, 2^b-1).
    Returns (codes uint8, s, m, pre) with s and m squeezed along `axis` and
    pre = (x-m)/s, the float64 value before rounding.
    [vatt §為什麼樸素的 2-bit…: range [min,max] split into 2^bits cells, round to
     nearest index, scale = cell width, zero-point = offset of min; worked example
     scale = (max-min)/3; hotdry §非对称量化与尺度折叠]
    Pinned by: test_worked_2bit_example (golden), test_rtn_matches_brute_force,
    test_rtn_error_bound.
    """
    x = np.asarray(x, dtype=np.float64)
    qmax = (1 << bits) - 1
    m = x.min(axis=axis, keepdims=True)
    mx = x.max(axis=axis, keepdims=True)
    s = np.maximum((mx - m) / qmax, SCALE_FLOOR)
    pre = (x - m) / s
    q = np.clip(np.rint(pre), 0, qmax).astype(np.uint8)
    return q, np.squeeze(s, axis=axis), np.squeeze(m, axis=axis), pre


def rtn_dequantize(q: np.ndarray, s: np.ndarray, m: np.ndarray, axis: int) -> np.ndarray:
    """x_hat = q * s + m, scale/zero broadcast along `axis`.  [vatt worked example: code 0 -> min]"""
    return q.astype(np.float64) * np.expand_dims(s, axis) + np.expand_dims(m, axis)


# ----------------------------------------------------------------------------
# 5. one tile end to end (quantise, fold, store as fp16 metadata)
# ----------------------------------------------------------------------------

def _f16(a):
    return np.asarray(a, dtype=np.float64).astype(np.float16)


def quantize_tile(tile: np.ndarray, kind: str, d: int | None = None,
                  iters: int = SINKHORN_ITERS, eps: float = SINKHORN_EPS, bits: int | None = None,
                  tol: float = 0.0):
    """Quantise a [..., 128, d0] tile of keys (kind 'K') or values (kind 'V').

    K: 4-bit (default), scale/zero per channel over the 128 tokens; stored s'_j = s_j c_j,
       z'_j = m_j c_j (fp16) and the token factor r_i (fp16).
    V: 2-bit (default), scale/zero per token over the channels; stored s'_i = s_i r_i,
       z'_i = m_i r_i (fp16) and the channel factor c_j (fp16).
    `bits` overrides the width (2, 4 or 8) for the other presets; `tol` > 0 stops the
    normalisation early (see sinkhorn_normalise).
    Returns dict(codes [...,T,d] uint8, scale fp16, zero fp16, factor fp16, pre f64, bits,
    iters = iterations used per tile).
    [hotdry §非对称量化与尺度折叠: keys 4-bit, values 2-bit; key scales per channel,
     value scales per token, scales multiplied back on read; vatt §四個步驟 table:
     KEY per-channel 4-bit, VALUE per-token 2-bit]
    Pinned by: test_quantize_tile_closed_form, test_quantize_tile_dequant_error.
    """
    tile = np.asarray(tile, dtype=np.float64)
    if d is None:
        d = padded_head_dim(tile.shape[-1])
    x = rotate(tile, d)
    n, r, c, used = sinkhorn_normalise(x, iters, eps, tol, return_iters=True)
    if kind == "K":
        bits = K_BITS if bits is None else bits
        q, s, m, pre = rtn_asymmetric(n, bits, axis=-2)
        scale, zero, factor = _f16(s * c), _f16(m * c), _f16(r)
    elif kind == "V":
        bits = V_BITS if bits is None else bits
        q, s, m, pre = rtn_asymmetric(n, bits, axis=-1)
        scale, zero, factor = _f16(s * r), _f16(m * r), _f16(c)
    else:
        raise ValueError("kind must be 'K' or 'V'")
    return {"codes": q, "scale": scale, "zero": zero, "factor": factor, "pre": pre, "bits": bits,
            "iters": used}


def dequantize_tile(codes, scale, zero, factor, kind: str, d0: int) -> np.ndarray:
    """Rebuild the tile in the original basis from codes and the stored fp16 metadata.

    K: K~_ij = r_i (q_ij s'_j + z'_j);  V: V~_ij = c_j (q_ij s'_i + z'_i);
    then undo the rotation (the orthonormal Hadamard is its own inverse) and drop
    the padded channels.  [hotdry §非对称量化与尺度折叠: scale multiplied back at read;
    aifeeds §方法 3: dequantisation restores the original scale]
    Pinned by: test_quantize_tile_closed_form, test_quantize_tile_dequant_error.
    """
    q = np.asarray(codes, dtype=np.float64)
    s = np.asarray(scale, dtype=np.float64)
    z = np.asarray(zero, dtype=np.float64)
    f = np.asarray(factor, dtype=np.float64)
    d = q.shape[-1]
    if kind == "K":
        xt = f[..., :, None] * (q * s[..., None, :] + z[..., None, :])
    elif kind == "V":
        xt = f[..., None, :] * (q * s[..., :, None] + z[..., :, None])
    else:
        raise ValueError("kind must be 'K' or 'V'")
    return rotate(xt, d)[..., :d0]


def quantization_error(tile: np.ndarray, codes, scale, zero, factor, kind: str) -> np.ndarray:
    """Error statistics of one quantised tile against the tile it came from.

    tile: [128, d0] source values; codes / scale / zero / factor: one K or V half of a page
    record (as quantize_tile returns or unpack_record gives back).  With x the source and
    x^ = dequantize_tile(...) the dequantised tile in the original basis, returns
    [sum (x - x^)^2, sum x^2, max |x - x^|, max |x|] over the 128 x d0 values.
    [hotdry §监控要点: sample the dequantised values periodically and watch the quantisation
     error]
    Pinned by: test_quantization_error_* (rotated-domain equality, power-of-two scaling,
    bit-width order, zero tile).
    """
    x = np.asarray(tile, dtype=np.float64)
    d0 = x.shape[-1]
    e = x - dequantize_tile(codes, scale, zero, factor, kind, d0)
    return np.array([np.sum(e * e), np.sum(x * x), np.max(np.abs(e)), np.max(np.abs(x))])


# ----------------------------------------------------------------------------
# page record: byte layout of one (page, kv head) in the packed cache
# ----------------------------------------------------------------------------
#
# The layout is this build's own contract (the pages fix only that the scales
# live with the 128-token block: vatt §怎麼用, "scales hang on each block's
# metadata").  Sections, all 16-byte aligned, T = 128, d = padded head_dim,
# kb / vb = K / V code bits (4 / 2 for kvarn_k4v2_g128):
#   K codes  T*d*kb/8 bytes of uint32 words
#   K scale[d], K zero[d], K token factor[T]  (fp16, little endian)
#   V codes  T*d*vb/8 bytes of uint32 words
#   V scale[T], V zero[T], V channel factor[d] (fp16, little endian)
#
# Every word carries m16n8k16 A-operand fragments (16 x 16 blocks, lane = 4g + tq,
# g = lane//4, tq = lane%4; element (rho, h, p) of a fragment sits at row g + 8rho,
# column 8h + 2tq + p of its block).  K's A operand is codes[token, channel]; V's is
# codes^T[channel, token].  Blocks are indexed (o, i): K o = token block, i = channel
# block; V o = token block, i = channel block; ni4 = d // 64.
#   4-bit: word ((o*ni4 + i//4)*32 + lane)*4 + i%4 holds fragment (o, i), element
#          (rho, h, p) at nibble h + 2rho + 4p.
#   2-bit: word ((o//2*ni4 + i//4)*32 + lane)*4 + i%4 holds fragments (o, i) for both
#          o of the pair, element (rho, h, p) of block o at slot 2(o%2) + h + 4rho + 8p.
#   8-bit: words ((o*ni2 + i//2)*32 + lane)*4 + 2(i%2) + h, h = 0, 1, hold fragment (o, i),
#          element (rho, h, p) at byte rho + 2p of word h; ni2 = d // 32.
# For kvarn_k4v2_g128: K word (mi, kk, lane) holds token t = 16mi + g + 8rho and channel
# j = 16kk + 8h + 2tq + p at nibble h + 2rho + 4p; V word (ks2, mc, lane) holds channel
# j = 16mc + g + 8rho and token t = 16(2ks2+f) + 8h + 2tq + p at 2-bit slot
# 2f + h + 4rho + 8p.

def record_bytes(d: int, tokens: int = TILE_TOKENS, k_bits: int = K_BITS, v_bits: int = V_BITS) -> int:
    """Bytes of one page record: kb + vb bits of codes per token-channel plus fp16 metadata.

    The record layout is defined for padded head_dim 64, 128 and 256 (its code words tile
    64-channel groups); smaller padded widths have no record (ValueError).
    Pinned by: test_record_bytes (13824 B at d=128 for K4V2, ratio vs fp16 below 1/4, as
    the vatt capacity widget's "<0.25x, about 4x" for kvarn_k4v2_g128), test_record_bytes_presets.
    """
    _check_record_dim(d)
    return tokens * d * k_bits // 8 + tokens * d * v_bits // 8 + 2 * (3 * d + 3 * tokens)


def _check_record_dim(d: int) -> None:
    if d not in (64, 128, 256):
        raise ValueError("page records exist for padded head_dim 64, 128 and 256 only")


def _section_offsets(d: int, k_bits: int = K_BITS, v_bits: int = V_BITS):
    """Byte offsets (K codes, V codes, K scale, K zero, K factor, V scale, V zero, V factor)."""
    t = TILE_TOKENS
    o_kc = 0
    o_ks = t * d * k_bits // 8
    o_kz = o_ks + 2 * d
    o_kr = o_kz + 2 * d
    o_vc = o_kr + 2 * t
    o_vs = o_vc + t * d * v_bits // 8
    o_vz = o_vs + 2 * t
    o_vcf = o_vz + 2 * t
    return o_kc, o_vc, o_ks, o_kz, o_kr, o_vs, o_vz, o_vcf


def _code_positions(kind: str, bits: int, d: int):
    """(word index, bit shift) for every (token, channel) of a K or V code section."""
    t = np.arange(TILE_TOKENS)[:, None]
    j = np.arange(d)[None, :]
    if kind == "K":      # rows are tokens, columns channels
        o, row, i, col = t // 16, t % 16, j // 16, j % 16
    elif kind == "V":    # rows are channels, columns tokens
        o, col, i, row = t // 16, t % 16, j // 16, j % 16
    else:
        raise ValueError("kind must be 'K' or 'V'")
    _check_record_dim(d)
    g, rho = row % 8, row // 8
    h, tq, p = col // 8, (col % 8) // 2, col % 2
    lane = 4 * g + tq
    ni4 = d // 64
    if bits == 4:
        word = ((o * ni4 + i // 4) * 32 + lane) * 4 + i % 4
        shift = 4 * (h + 2 * rho + 4 * p)
    elif bits == 2:
        word = (((o // 2) * ni4 + i // 4) * 32 + lane) * 4 + i % 4
        shift = 2 * (2 * (o % 2) + h + 4 * rho + 8 * p)
    elif bits == 8:
        word = ((o * (d // 32) + i // 2) * 32 + lane) * 4 + 2 * (i % 2) + h
        shift = 8 * (rho + 2 * p)
    else:
        raise ValueError("code bits must be 2, 4 or 8")
    return word, shift


def _k_positions(d: int, bits: int = K_BITS):
    """(word index, bit shift) for every (token, channel) of the K code section."""
    return _code_positions("K", bits, d)


def _v_positions(d: int, bits: int = V_BITS):
    """(word index, bit shift) for every (token, channel) of the V code section."""
    return _code_positions("V", bits, d)


def pack_record(k: dict, v: dict) -> bytes:
    """Pack the quantised K and V tiles of one (page, kv head) into a page record; the code
    widths come from the dicts' "bits" (4 and 2 when absent).

    Pinned by: test_pack_roundtrip, test_pack_is_bijective, test_record_bytes,
    test_code_words_are_mma_fragments.
    """
    kb, vb = k.get("bits", K_BITS), v.get("bits", V_BITS)
    qk = np.asarray(k["codes"], dtype=np.uint32)
    qv = np.asarray(v["codes"], dtype=np.uint32)
    if qk.max(initial=0) >= (1 << kb) or qv.max(initial=0) >= (1 << vb):
        raise ValueError("code outside its bit width")
    d = qk.shape[-1]
    kw = np.zeros(TILE_TOKENS * d * kb // 32, dtype=np.uint32)
    word, shift = _k_positions(d, kb)
    np.bitwise_or.at(kw, word.ravel(), (qk << shift.astype(np.uint32)).ravel())
    vw = np.zeros(TILE_TOKENS * d * vb // 32, dtype=np.uint32)
    word, shift = _v_positions(d, vb)
    np.bitwise_or.at(vw, word.ravel(), (qv << shift.astype(np.uint32)).ravel())

    def f16(a):
        return np.asarray(a, dtype=np.float16).astype("<f2").tobytes()

    parts = [kw.astype("<u4").tobytes(), f16(k["scale"]), f16(k["zero"]), f16(k["factor"]),
             vw.astype("<u4").tobytes(), f16(v["scale"]), f16(v["zero"]), f16(v["factor"])]
    out = b"".join(parts)
    assert len(out) == record_bytes(d, k_bits=kb, v_bits=vb)
    return out


def unpack_record(rec, d: int, k_bits: int = K_BITS, v_bits: int = V_BITS):
    """Inverse of pack_record: returns (k dict, v dict) with codes and fp16 metadata."""
    buf = np.frombuffer(bytes(rec), dtype=np.uint8)
    if buf.size != record_bytes(d, k_bits=k_bits, v_bits=v_bits):
        raise ValueError("record size does not match head_dim and code bits")
    o_kc, o_vc, o_ks, o_kz, o_kr, o_vs, o_vz, o_vcf = _section_offsets(d, k_bits, v_bits)
    t = TILE_TOKENS
    kw = buf[o_kc:o_ks].view("<u4").astype(np.uint32)
    vw = buf[o_vc:o_vs].view("<u4").astype(np.uint32)
    word, shift = _k_positions(d, k_bits)
    qk = ((kw[word] >> shift.astype(np.uint32)) & ((1 << k_bits) - 1)).astype(np.uint8)
    word, shift = _v_positions(d, v_bits)
    qv = ((vw[word] >> shift.astype(np.uint32)) & ((1 << v_bits) - 1)).astype(np.uint8)

    def f16(lo, n):
        return buf[lo:lo + 2 * n].view("<f2").astype(np.float16)

    k = {"codes": qk, "scale": f16(o_ks, d), "zero": f16(o_kz, d), "factor": f16(o_kr, t), "bits": k_bits}
    v = {"codes": qv, "scale": f16(o_vs, t), "zero": f16(o_vz, t), "factor": f16(o_vcf, d), "bits": v_bits}
    return k, v


def quantize_page(k_tile, v_tile, iters: int = SINKHORN_ITERS, eps: float = SINKHORN_EPS,
                  k_bits: int = K_BITS, v_bits: int = V_BITS):
    """Quantise one (page, kv head): fp16 K/V tiles [128, d0] -> (record bytes, k, v)."""
    d = padded_head_dim(np.asarray(k_tile).shape[-1])
    k = quantize_tile(k_tile, "K", d, iters, eps, bits=k_bits)
    v = quantize_tile(v_tile, "V", d, iters, eps, bits=v_bits)
    return pack_record(k, v), k, v


def dequantize_record(rec, d0: int, k_bits: int = K_BITS, v_bits: int = V_BITS):
    """Page record -> (K_hat [128, d0], V_hat [128, d0]) float64 in the original basis."""
    d = padded_head_dim(d0)
    k, v = unpack_record(rec, d, k_bits, v_bits)
    kh = dequantize_tile(k["codes"], k["scale"], k["zero"], k["factor"], "K", d0)
    vh = dequantize_tile(v["codes"], v["scale"], v["zero"], v["factor"], "V", d0)
    return kh, vh


# ----------------------------------------------------------------------------
# decode attention over the packed cache
# ----------------------------------------------------------------------------

def softmax_attention(q: np.ndarray, keys: np.ndarray, values: np.ndarray,
                      softmax_scale: float) -> np.ndarray:
    """Textbook attention for one query: o = sum_t softmax(tau q.k_t) v_t (float64).

    Empty key set gives zeros (reading: a sequence of length 0 attends to nothing).
    Pinned by: test_attention_* (single token, identical keys, scipy softmax,
    split invariance).
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    if keys.shape[0] == 0:
        return np.zeros(values.shape[-1], dtype=np.float64)
    logits = softmax_scale * (keys @ q)
    w = np.exp(logits - logits.max())
    return (w / w.sum()) @ values


def decode_sequence(q_heads: np.ndarray, records, partial_k, partial_v,
                    softmax_scale: float, d0: int, k_bits: int = K_BITS,
                    v_bits: int = V_BITS) -> np.ndarray:
    """Attention output of one sequence for all its query heads of ONE kv head.

    q_heads: [G, d0] queries sharing this kv head (grouped-query attention).
    records: the page records of the sequence's sealed 128-token pages, in order.
    partial_k/partial_v: [n, d0] raw fp16 tokens of the unsealed tile (n < 128).
    [vatt §一次 16K context…: every decode step reads all cached K/V of the
     sequence; hotdry §核心配置参数: compute in float16 over the quantised cache]
    """
    ks, vs = [], []
    for rec in records:
        kh, vh = dequantize_record(rec, d0, k_bits, v_bits)
        ks.append(kh)
        vs.append(vh)
    if partial_k is not None and len(partial_k):
        ks.append(np.asarray(partial_k, dtype=np.float64)[:, :d0])
        vs.append(np.asarray(partial_v, dtype=np.float64)[:, :d0])
    keys = np.concatenate(ks, axis=0) if ks else np.zeros((0, d0))
    vals = np.concatenate(vs, axis=0) if vs else np.zeros((0, d0))
    return np.stack([softmax_attention(qh, keys, vals, softmax_scale)
                     for qh in np.asarray(q_heads, dtype=np.float64)])


def fp16_decode_sequence(q_heads: np.ndarray, keys: np.ndarray, values: np.ndarray,
                         softmax_scale: float) -> np.ndarray:
    """Decode attention of the query heads of ONE kv head over an uncompressed fp16 cache.

    keys, values: [L, d] the sequence's cached tokens as stored (fp16), no rotation and no
    quantisation: the baseline the packed cache is compared with.  Returns [G, d].
    [hotdry §监控要点: throughput is judged against an fp16 KV cache; vatt §一次 16K
     context…: decode reads the whole cache every step]
    Pinned by: test_fp16_decode_* (two-token closed form, paging invariance) and the
    softmax_attention pins.
    """
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    return np.stack([softmax_attention(qh, keys, values, softmax_scale)
                     for qh in np.asarray(q_heads, dtype=np.float64)])


def prefill_sequence(q: np.ndarray, records, partial_k, partial_v, chunk_k: np.ndarray,
                     chunk_v: np.ndarray, softmax_scale: float, d0: int,
                     k_bits: int = K_BITS, v_bits: int = V_BITS) -> np.ndarray:
    """Chunked-prefill attention of one sequence for the query heads of ONE kv head.

    q: [C, G, d0] queries of the chunk's C tokens; chunk_k / chunk_v: [C, d0] the chunk's own
    raw keys and values.  Query token c attends to every cached token (the dequantised sealed
    pages, then the raw partial-tile tokens) and to chunk tokens 0..c: textbook causal
    attention over the concatenation, in the original basis.  Returns [C, G, d0].
    [vatt §怎麼用: the paged blocks hold the quantised cache; the step before decode reads
     the same cache]
    Pinned by: test_prefill_* (single token == decode with it appended, causal invariance,
    full-precision cache limit).
    """
    ks, vs = [], []
    for rec in records:
        kh, vh = dequantize_record(rec, d0, k_bits, v_bits)
        ks.append(kh)
        vs.append(vh)
    if partial_k is not None and len(partial_k):
        ks.append(np.asarray(partial_k, dtype=np.float64)[:, :d0])
        vs.append(np.asarray(partial_v, dtype=np.float64)[:, :d0])
    cache_k = np.concatenate(ks, axis=0) if ks else np.zeros((0, d0))
    cache_v = np.concatenate(vs, axis=0) if vs else np.zeros((0, d0))
    ck = np.asarray(chunk_k, dtype=np.float64)[:, :d0]
    cv = np.asarray(chunk_v, dtype=np.float64)[:, :d0]
    q = np.asarray(q, dtype=np.float64)
    out = np.zeros(q.shape, dtype=np.float64)
    for c in range(q.shape[0]):
        keys = np.concatenate([cache_k, ck[:c + 1]], axis=0)
        vals = np.concatenate([cache_v, cv[:c + 1]], axis=0)
        for g in range(q.shape[1]):
            out[c, g] = softmax_attention(q[c, g], keys, vals, softmax_scale)
    return out


# ----------------------------------------------------------------------------
# byte accounting
# ----------------------------------------------------------------------------

def fp16_kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int) -> int:
    """2 (K and V) x layers x kv_heads x head_dim x 2 bytes.

    [vatt §一次 16K context 的推論…: 2 x 64 x 8 x 128 x 2 = 262144 bytes per token]
    Pinned by: test_bytes_per_token (golden).
    """
    return 2 * layers * kv_heads * head_dim * 2


def packed_kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int,
                              k_bits: int = K_BITS, v_bits: int = V_BITS) -> float:
    """Packed bytes per token (K4V2 by default) including the fp16 metadata of its page."""
    d = padded_head_dim(head_dim)
    return layers * kv_heads * record_bytes(d, k_bits=k_bits, v_bits=v_bits) / TILE_TOKENS
