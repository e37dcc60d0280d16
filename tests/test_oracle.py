"""Pins of the float64 CPU oracle against the pages, closed forms and library routines.

CPU only.  Each test names the page passage or the mathematical fact it checks.
"""

import math
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.special
import torch

from oracle import kvarn_oracle as ko
from calibration_free_kv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _fwht_rows(a):
    """Iterative in-place fast Walsh-Hadamard butterflies (unnormalised), rows of a."""
    a = np.array(a, dtype=np.float64, copy=True)
    n = a.shape[-1]
    h = 1
    while h < n:
        for i in range(0, n, 2 * h):
            x = a[..., i:i + h].copy()
            y = a[..., i + h:i + 2 * h].copy()
            a[..., i:i + h] = x + y
            a[..., i + h:i + 2 * h] = x - y
        h *= 2
    return a


def _checker(t, d):
    return (-1.0) ** (np.arange(t)[:, None] + np.arange(d)[None, :])


# --- padding and rotation ----------------------------------------------------

def test_padded_head_dim():
    # aifeeds §局限: a head_dim that is not a power of two is padded up to the next power of
    # two; a power of two is kept as it is, however small
    for d0, want in ((1, 1), (3, 4), (8, 8), (16, 16), (32, 32), (33, 64), (64, 64), (96, 128),
                     (128, 128), (129, 256), (256, 256)):
        assert ko.padded_head_dim(d0) == want, d0


@pytest.mark.parametrize("d0", [8, 16, 32])
def test_small_head_dims_rotate_by_their_own_order(d0):
    # aifeeds §局限: d0 = 8/16/32 are powers of two, so the rotation is H_d0 / sqrt(d0) itself
    # (no padding): a unit vector e_0 becomes the constant row 1/sqrt(d0)
    x = np.zeros((1, d0))
    x[0, 0] = 1.0
    np.testing.assert_allclose(ko.rotate(x, ko.padded_head_dim(d0)), np.full((1, d0), d0 ** -0.5),
                               rtol=0, atol=1e-15)
    # and such widths have no page record (the record's code words tile 64-channel groups)
    with pytest.raises(ValueError):
        ko.record_bytes(d0)


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_hadamard_matches_scipy(n):
    # Sylvester ordering as produced by the library routine
    np.testing.assert_array_equal(ko.sylvester_hadamard(n), scipy.linalg.hadamard(n))


@pytest.mark.parametrize("n", [2, 64, 128, 256])
def test_hadamard_orthogonality(n):
    # hotdry §Hadamard 旋转: entries +-1 and H H^T = n I
    h = ko.sylvester_hadamard(n)
    assert set(np.unique(h)) == {-1.0, 1.0}
    np.testing.assert_array_equal(h @ h.T, n * np.eye(n))


def test_rotation_preserves_norms_and_inner_products():
    # vatt §四個步驟, Hadamard rotation: orthonormal, attention inner products unchanged
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 96))
    y = rng.standard_normal((5, 96))
    rx, ry = ko.rotate(x, 128), ko.rotate(y, 128)
    np.testing.assert_allclose(np.linalg.norm(rx, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    np.testing.assert_allclose(np.sum(rx * ry, axis=1), np.sum(x * y, axis=1), rtol=1e-12,
                               atol=1e-12)


def test_rotation_is_an_involution():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 256))
    np.testing.assert_allclose(ko.rotate(ko.rotate(x, 256), 256), x, atol=1e-12)


@pytest.mark.parametrize("n", [2, 8, 64, 128, 256])
def test_rotation_matches_fast_transform(n):
    # hotdry §Hadamard 旋转: the FWHT computes the same product in O(n log n)
    rng = np.random.default_rng(n)
    z = rng.integers(-1000, 1000, size=(3, n)).astype(np.float64)
    np.testing.assert_allclose(ko.rotate(z, n) * np.sqrt(n), _fwht_rows(z), rtol=1e-13, atol=1e-9)


def test_rotation_spreads_single_outlier():
    # vatt §為什麼樸素的 2-bit…: after rotation the outlier's max drops from 28 to single digits
    x = np.zeros(128)
    x[77] = 28.0
    r = ko.rotate(x, 128)
    assert np.allclose(np.abs(r), 28.0 / math.sqrt(128.0))
    assert np.abs(r).max() < 10.0


# --- quantiser ---------------------------------------------------------------

def test_worked_2bit_example():
    rows = _read_golden("worked_2bit_example.txt")
    kv = {r[0]: r[1:] for r in rows if r[0] not in ("quant", "dequant")}
    bits = int(kv["bits"][0])
    vals = np.array([float(v) for v in kv["values"]])
    q, s, m, pre = ko.rtn_asymmetric(vals, bits, axis=0)
    assert float(m) == pytest.approx(float(kv["min"][0]), abs=1e-15)
    assert float(m) + 3 * float(s) == pytest.approx(float(kv["max"][0]), abs=1e-12)
    assert float(s) == pytest.approx(float(kv["scale"][0]), rel=1e-12)
    lookup = dict(zip(vals.tolist(), q.tolist()))
    for r in rows:
        if r[0] == "quant":
            assert lookup[float(r[1])] == int(r[2])
        if r[0] == "dequant":
            xh = ko.rtn_dequantize(np.array([int(r[1])]), s, m, axis=0)
            assert xh[0] == pytest.approx(float(r[2]), abs=1e-12)
    # code 3 restores the outlier exactly
    assert ko.rtn_dequantize(np.array([3]), s, m, axis=0)[0] == pytest.approx(28.0, abs=1e-12)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_rtn_matches_brute_force(bits):
    # round-to-nearest == the nearest of the 2^b grid points (ties aside)
    rng = np.random.default_rng(10 + bits)
    for trial in range(200):
        n = int(rng.integers(2, 40))
        x = rng.standard_normal(n) * rng.uniform(0.01, 100.0) + rng.uniform(-5, 5)
        q, s, m, _ = ko.rtn_asymmetric(x, bits, axis=0)
        grid = np.arange(1 << bits) * float(s) + float(m)
        dist = np.abs(x[:, None] - grid[None, :])
        best = dist.argmin(axis=1)
        srt = np.sort(dist, axis=1)
        clear = (srt[:, 1] - srt[:, 0]) > 1e-9 * float(s)
        np.testing.assert_array_equal(q[clear], best[clear])


def test_rtn_error_bound():
    # round to nearest on a grid of step s: |z - z_hat| <= s / 2 inside [min, max]
    # (vatt §為什麼樸素的 2-bit…: the range split into 2^bits - 1 steps, nearest level)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((128, 64)) * 3.0
    for bits, axis in ((4, 0), (2, 1)):
        q, s, m, _ = ko.rtn_asymmetric(x, bits, axis=axis)
        xh = ko.rtn_dequantize(q, s, m, axis=axis)
        assert np.all(np.abs(x - xh) <= np.expand_dims(s, axis) * 0.5 * (1 + 1e-12))


def test_rtn_constant_group():
    q, s, m, _ = ko.rtn_asymmetric(np.full(8, 2.5), 4, axis=0)
    assert np.all(q == 0) and float(s) == ko.SCALE_FLOOR and float(m) == 2.5


# --- Sinkhorn-style normalisation --------------------------------------------

def _rank_one_scaled(t, d, seed):
    rng = np.random.default_rng(seed)
    r = 2.0 ** rng.integers(-3, 4, size=t)
    c = 2.0 ** rng.integers(-3, 4, size=d)
    return r, c, r[:, None] * _checker(t, d) * c[None, :]


@pytest.mark.parametrize("iters", [1, 4, 7])
def test_sinkhorn_closed_form(iters):
    # X = diag(r) Y diag(c) with Y = (-1)^(i+j) (every row/column mean 0, std 1):
    # one column+row step normalises exactly, later steps add ln(1) = 0.
    r, c, x = _rank_one_scaled(128, 128, iters)
    n, ro, co = ko.sinkhorn_normalise(x, iters)
    np.testing.assert_allclose(n, _checker(128, 128), atol=1e-12)
    np.testing.assert_allclose(ro[:, None] * co[None, :], r[:, None] * c[None, :], rtol=1e-12)
    # by hand: the first column step divides column j by c_j S, S = population std over i
    # of r_i (-1)^i; the row step then leaves r_i / S.  Later steps add ln 1 = 0.
    alt = r * (-1.0) ** np.arange(128)
    big_s = math.sqrt(float(np.mean(alt ** 2) - np.mean(alt) ** 2))
    np.testing.assert_allclose(co, c * big_s, rtol=1e-12)
    np.testing.assert_allclose(ro, r / big_s, rtol=1e-12)


def test_sinkhorn_subtracts_the_mean():
    # std (not RMS): X_ij = c_j (Y_ij + 3) normalises to Y + 3
    c = 2.0 ** np.arange(-4, 4).repeat(16)
    x = (_checker(128, 128) + 3.0) * c[None, :]
    n, _, _ = ko.sinkhorn_normalise(x, 4)
    np.testing.assert_allclose(n, _checker(128, 128) + 3.0, atol=1e-12)


def test_sinkhorn_final_rows_unit_std():
    # the last half-step is the token (row) step, so every row std is 1 afterwards
    k, _ = synth.outlier_kv(128, 1, 128, seed=5)
    x = ko.rotate(k[:, 0].double().numpy(), 128)
    for iters in (1, 2, 4):
        n, _, _ = ko.sinkhorn_normalise(x, iters)
        np.testing.assert_allclose(n.std(axis=1), 1.0, atol=1e-12)


def test_sinkhorn_leaves_constant_and_zero_tiles_finite():
    # rows/columns without variance keep their factors: a zero tile keeps r = c = 1 and a
    # constant column is not blown up by 1/eps (reading of the epsilon floor)
    n, r, c = ko.sinkhorn_normalise(np.zeros((128, 128)), 4)
    assert np.all(r == 1.0) and np.all(c == 1.0) and np.all(n == 0.0)
    x = np.random.default_rng(8).standard_normal((128, 128))
    x[:, 5] = 2.5
    n, r, c = ko.sinkhorn_normalise(x, 4)
    assert np.all(np.isfinite(n)) and np.abs(np.log(r)).max() < 20 and np.abs(np.log(c)).max() < 20
    # the zero tile dequantises to zeros through the fp16 metadata
    q = ko.quantize_tile(np.zeros((128, 64)), "K")
    assert np.all(np.isfinite(q["factor"].astype(np.float64)))
    back = ko.dequantize_tile(q["codes"], q["scale"], q["zero"], q["factor"], "K", 64)
    np.testing.assert_array_equal(back, 0.0)


def test_sinkhorn_converges():
    # hotdry §迭代方差归一化 step 3 / vatt §四個步驟: the alternation converges and leaves
    # every row and every column with a similar variance (3-5 iterations usually enough)
    k, _ = synth.outlier_kv(128, 1, 128, seed=6)
    x = ko.rotate(k[:, 0].double().numpy(), 128)
    steps, spread, prev = [], [], None
    for iters in range(1, 11):
        n, _, _ = ko.sinkhorn_normalise(x, iters)
        sc = n.std(axis=0)
        spread.append((sc.max() - sc.min()) / sc.mean())
        if prev is not None:
            steps.append(np.abs(n - prev).max() / np.abs(n).max())
        prev = n
    print("N change per iteration:", ["%.1e" % v for v in steps])
    print("column-std spread after 1..10 iterations:", ["%.1e" % v for v in spread])
    assert all(steps[i + 1] < 0.5 * steps[i] for i in range(len(steps) - 1))
    assert spread[3] < 1e-2 * spread[0]
    assert steps[-1] < 1e-6


def test_sinkhorn_invariances():
    # channel scaling is absorbed by the first (column) step; a global power of two too
    rng = np.random.default_rng(7)
    x = rng.standard_normal((128, 128)) * np.exp(rng.standard_normal((128, 1)))
    n0, r0, c0 = ko.sinkhorn_normalise(x, 4)
    xs = x.copy()
    xs[:, 11] *= 8.0
    n1, r1, c1 = ko.sinkhorn_normalise(xs, 4)
    np.testing.assert_allclose(n1, n0, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(c1[11], 8.0 * c0[11], rtol=1e-12)
    n2, _, _ = ko.sinkhorn_normalise(x * 0.25, 4)
    np.testing.assert_allclose(n2, n0, rtol=1e-12, atol=1e-12)


# --- whole tile ----------------------------------------------------------------

def test_quantize_tile_closed_form():
    # tile whose rotation is diag(r) Y diag(c): codes are the two extreme levels and the
    # fold reproduces the tile up to the fp16 metadata rounding
    r, c, x = _rank_one_scaled(128, 128, 11)
    tile = ko.rotate(x, 128)                   # rotate(tile) == x
    y = _checker(128, 128)
    k = ko.quantize_tile(tile, "K")
    v = ko.quantize_tile(tile, "V")
    np.testing.assert_array_equal(k["codes"], (15 * (y + 1) / 2).astype(np.uint8))
    np.testing.assert_array_equal(v["codes"], (3 * (y + 1) / 2).astype(np.uint8))
    for kind, qd in (("K", k), ("V", v)):
        back = ko.dequantize_tile(qd["codes"], qd["scale"], qd["zero"], qd["factor"], kind, 128)
        assert np.abs(back - tile).max() <= 4e-3 * np.abs(tile).max()


def test_quantize_axes_without_normalisation():
    # iters = 0 reduces to plain asymmetric RTN: K groups a channel over tokens,
    # V groups a token over channels (vatt §四個步驟 table)
    y = _checker(128, 128)
    c = 2.0 ** np.arange(-4, 4).repeat(16)
    xk = y * c[None, :]                        # channel-dependent range
    k = ko.quantize_tile(ko.rotate(xk, 128), "K", iters=0)
    np.testing.assert_array_equal(k["codes"], (15 * (y + 1) / 2).astype(np.uint8))
    xv = c[:, None] * y                        # token-dependent range
    v = ko.quantize_tile(ko.rotate(xv, 128), "V", iters=0)
    np.testing.assert_array_equal(v["codes"], (3 * (y + 1) / 2).astype(np.uint8))


def test_quantize_tile_dequant_error():
    # reconstruction error bounded by half a quantisation step (times the folded factors)
    k, v = synth.outlier_kv(128, 1, 96, seed=12)
    for kind, t in (("K", k), ("V", v)):
        tile = t[:, 0].double().numpy()
        qd = ko.quantize_tile(tile, kind)
        x = ko.rotate(tile, 128)
        back = ko.rotate(ko.dequantize_tile(qd["codes"], qd["scale"], qd["zero"], qd["factor"],
                                            kind, 128), 128)
        s = qd["scale"].astype(np.float64)
        f = qd["factor"].astype(np.float64)
        step = f[:, None] * s[None, :] if kind == "K" else s[:, None] * f[None, :]
        assert np.all(np.abs(back - x) <= 0.5 * step * 1.01 + 1e-3 * np.abs(x) + 1e-6)


def test_kvarn_beats_naive_rtn():
    # vatt §為什麼樸素的 2-bit…: rotation + normalisation cuts the error of bare RTN
    k, v = synth.outlier_kv(128, 1, 128, seed=13)
    for kind, t, bits, axis in (("K", k, 4, 0), ("V", v, 2, 1)):
        tile = t[:, 0].double().numpy()
        qd = ko.quantize_tile(tile, kind)
        ours = ko.dequantize_tile(qd["codes"], qd["scale"], qd["zero"], qd["factor"], kind, 128)
        q, s, m, _ = ko.rtn_asymmetric(tile, bits, axis=axis)
        naive = ko.rtn_dequantize(q, s, m, axis=axis)
        e_ours = np.linalg.norm(ours - tile) / np.linalg.norm(tile)
        e_naive = np.linalg.norm(naive - tile) / np.linalg.norm(tile)
        print(kind, "relative error kvarn %.4f naive %.4f" % (e_ours, e_naive))
        assert e_ours < e_naive


# --- page record --------------------------------------------------------------

def test_record_bytes():
    assert ko.record_bytes(128) == 13824
    assert ko.record_bytes(256) == 26880
    fp16_page = 2 * 128 * 128 * 2
    ratio = ko.record_bytes(128) / fp16_page
    # vatt capacity widget for kvarn_k4v2_g128: "below 0.25x, about 4x"
    assert ratio < 0.25 and 4.0 < 1.0 / ratio < 5.0


def test_bytes_per_token():
    g = {r[0]: int(r[1]) for r in _read_golden("bytes_per_token.txt")}
    b = ko.fp16_kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"])
    assert b == g["bytes_per_token"]
    assert b * g["context"] == g["bytes_per_sequence"]
    assert ko.packed_kv_bytes_per_token(64, 8, 128) == 64 * 8 * 108


@pytest.mark.parametrize("d", [64, 128, 256])
def test_pack_is_bijective(d):
    for pos, bits, per_word in ((ko._k_positions(d), 4, 8), (ko._v_positions(d), 2, 16)):
        word, shift = pos
        keys = word.astype(np.int64) * 64 + shift
        assert np.unique(keys).size == 128 * d
        assert word.max() + 1 == 128 * d // per_word
        assert set(np.unique(shift)) == set(range(0, 32, bits))


def _mma_a_fragment(mat, g, tq):
    """m16n8k16 A-operand registers a0..a3 of lane (g, tq) for a 16x16 block, as listed in
    the PTX ISA fragment table: a0 (g, 2tq..2tq+1), a1 (g+8, ..), a2 (g, 2tq+8..), a3 (g+8, ..+8)."""
    return [(mat[g, 2 * tq], mat[g, 2 * tq + 1]), (mat[g + 8, 2 * tq], mat[g + 8, 2 * tq + 1]),
            (mat[g, 2 * tq + 8], mat[g, 2 * tq + 9]), (mat[g + 8, 2 * tq + 8], mat[g + 8, 2 * tq + 9])]


@pytest.mark.parametrize("d", [64, 128, 256])
def test_code_words_are_mma_fragments(d):
    # each K word carries one m16n8k16 A fragment of codes[token, channel] and each V word two
    # A fragments of codes^T[channel, token]; register r takes its (lo, hi) pair from the
    # 4-bit slots (n, n+4) / 2-bit slots (n, n+8) listed below
    rng = np.random.default_rng(d + 1)
    qk = rng.integers(0, 16, (128, d)).astype(np.uint8)
    qv = rng.integers(0, 4, (128, d)).astype(np.uint8)
    zero = np.zeros(d, np.float16)
    rec = ko.pack_record({"codes": qk, "scale": zero, "zero": zero, "factor": np.zeros(128, np.float16)},
                         {"codes": qv, "scale": np.zeros(128, np.float16), "zero": np.zeros(128, np.float16),
                          "factor": zero})
    buf = np.frombuffer(rec, np.uint8)
    o_kc, o_vc, o_ks, _, _, o_vs, _, _ = ko._section_offsets(d)
    kw = buf[o_kc:o_ks].view("<u4")
    vw = buf[o_vc:o_vs].view("<u4")
    # the K half (codes + metadata) precedes the V half; sections are 16-byte aligned
    assert o_ks == 128 * d // 2 and o_vc == 128 * d // 2 + 4 * d + 2 * 128
    assert all(o % 16 == 0 for o in ko._section_offsets(d))
    k_slots = (0, 2, 1, 3)
    v_slots = ((0, 4, 1, 5), (2, 6, 3, 7))
    for lane in range(32):
        g, tq = lane // 4, lane % 4
        for mi in range(8):
            for kk in range(d // 16):
                w = int(kw[((mi * (d // 64) + kk // 4) * 32 + lane) * 4 + kk % 4])
                want = _mma_a_fragment(qk[16 * mi:16 * mi + 16, 16 * kk:16 * kk + 16], g, tq)
                got = [((w >> 4 * n) & 15, (w >> 4 * (n + 4)) & 15) for n in k_slots]
                assert got == [tuple(int(x) for x in p) for p in want]
        for ks2 in range(4):
            for mc in range(d // 16):
                w = int(vw[((ks2 * (d // 64) + mc // 4) * 32 + lane) * 4 + mc % 4])
                for f in range(2):
                    ks = 2 * ks2 + f
                    vt = qv[16 * ks:16 * ks + 16, 16 * mc:16 * mc + 16].T
                    want = _mma_a_fragment(vt, g, tq)
                    got = [((w >> 2 * n) & 3, (w >> 2 * (n + 8)) & 3) for n in v_slots[f]]
                    assert got == [tuple(int(x) for x in p) for p in want]


@pytest.mark.parametrize("d", [64, 128, 256])
def test_pack_roundtrip(d):
    rng = np.random.default_rng(d)
    k = {"codes": rng.integers(0, 16, (128, d)).astype(np.uint8),
         "scale": rng.standard_normal(d).astype(np.float16),
         "zero": rng.standard_normal(d).astype(np.float16),
         "factor": rng.standard_normal(128).astype(np.float16)}
    v = {"codes": rng.integers(0, 4, (128, d)).astype(np.uint8),
         "scale": rng.standard_normal(128).astype(np.float16),
         "zero": rng.standard_normal(128).astype(np.float16),
         "factor": rng.standard_normal(d).astype(np.float16)}
    rec = ko.pack_record(k, v)
    k2, v2 = ko.unpack_record(rec, d)
    for a, b in ((k, k2), (v, v2)):
        for key in a:
            np.testing.assert_array_equal(a[key], b[key])


# --- other k/v bit presets (vatt §四個步驟, bit-width assignment: same pipeline) ----------

_WIDTHS = [(4, 2), (4, 4), (2, 2), (2, 4), (8, 4), (4, 8)]


def test_record_bytes_presets():
    # T*d*(kb+vb)/8 code bytes + 2*(3d + 3T) fp16 metadata, by hand
    assert ko.record_bytes(128, k_bits=4, v_bits=4) == 8192 + 8192 + 1536 == 17920
    assert ko.record_bytes(128, k_bits=2, v_bits=2) == 4096 + 4096 + 1536 == 9728
    assert ko.record_bytes(256, k_bits=4, v_bits=4) == 16384 + 16384 + 2304
    assert ko.record_bytes(64, k_bits=2, v_bits=4) == 2048 + 4096 + 1152
    assert ko.record_bytes(128, k_bits=8, v_bits=4) == 16384 + 8192 + 1536 == 26112
    assert ko.record_bytes(256, k_bits=8, v_bits=4) == 32768 + 16384 + 2304
    assert set(ko.PRESETS.values()) <= set(_WIDTHS)
    assert ko.PRESETS["kvarn_k4v2_g128"] == (ko.K_BITS, ko.V_BITS)
    for kb, vb in _WIDTHS:
        assert all(o % 16 == 0 for o in ko._section_offsets(128, kb, vb))


@pytest.mark.parametrize("kind", ["K", "V"])
@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("d", [64, 256])
def test_code_positions_bijective(kind, bits, d):
    word, shift = ko._code_positions(kind, bits, d)
    keys = word.astype(np.int64) * 64 + shift
    assert np.unique(keys).size == 128 * d
    assert word.max() + 1 == 128 * d * bits // 32
    assert set(np.unique(shift)) == set(range(0, 32, bits))


@pytest.mark.parametrize("kb,vb", _WIDTHS)
def test_code_words_are_mma_fragments_all_widths(kb, vb):
    # the words of every width carry m16n8k16 A fragments (PTX fragment table): K's of
    # codes[token, channel], V's of codes^T[channel, token]; 4-bit words one fragment with
    # register r's (lo, hi) pair at nibbles (n, n+4), 2-bit words the fragments of two
    # consecutive token blocks (K: rows, V: columns) with pairs at slots (n, n+8), 8-bit
    # fragments two consecutive words (registers 0, 1 in the first, 2, 3 in the second) with
    # pairs at bytes (n, n+2)
    d = 64
    rng = np.random.default_rng(kb * 10 + vb)
    qk = rng.integers(0, 1 << kb, (128, d)).astype(np.uint8)
    qv = rng.integers(0, 1 << vb, (128, d)).astype(np.uint8)
    zd, zt = np.zeros(d, np.float16), np.zeros(128, np.float16)
    rec = ko.pack_record({"codes": qk, "scale": zd, "zero": zd, "factor": zt, "bits": kb},
                         {"codes": qv, "scale": zt, "zero": zt, "factor": zd, "bits": vb})
    buf = np.frombuffer(rec, np.uint8)
    o_kc, o_vc, o_ks, _, _, o_vs, _, _ = ko._section_offsets(d, kb, vb)
    for kind, words, bits, codes in (("K", buf[o_kc:o_ks].view("<u4"), kb, qk),
                                     ("V", buf[o_vc:o_vs].view("<u4"), vb, qv)):
        mask = (1 << bits) - 1
        for lane in range(32):
            g, tq = lane // 4, lane % 4
            for o in range(8):
                for i in range(d // 16):
                    blk = codes[16 * o:16 * o + 16, 16 * i:16 * i + 16]
                    mat = blk if kind == "K" else blk.T
                    want = _mma_a_fragment(mat, g, tq)
                    if bits == 4:
                        w = int(words[((o * (d // 64) + i // 4) * 32 + lane) * 4 + i % 4])
                        got = [((w >> 4 * n) & mask, (w >> 4 * (n + 4)) & mask) for n in (0, 2, 1, 3)]
                    elif bits == 8:
                        base = ((o * (d // 32) + i // 2) * 32 + lane) * 4 + 2 * (i % 2)
                        got = []
                        for w in (int(words[base]), int(words[base + 1])):
                            got += [((w >> 8 * n) & mask, (w >> 8 * (n + 2)) & mask) for n in (0, 1)]
                    else:
                        w = int(words[(((o // 2) * (d // 64) + i // 4) * 32 + lane) * 4 + i % 4])
                        f = o % 2
                        got = [((w >> 2 * n) & mask, (w >> 2 * (n + 8)) & mask)
                               for n in (2 * f, 2 * f + 4, 2 * f + 1, 2 * f + 5)]
                    assert got == [tuple(int(x) for x in pr) for pr in want], (kind, bits, lane, o, i)


@pytest.mark.parametrize("kb,vb", _WIDTHS)
def test_pack_roundtrip_all_widths(kb, vb):
    rng = np.random.default_rng(kb + 7 * vb)
    d = 128
    k = {"codes": rng.integers(0, 1 << kb, (128, d)).astype(np.uint8),
         "scale": rng.standard_normal(d).astype(np.float16),
         "zero": rng.standard_normal(d).astype(np.float16),
         "factor": rng.standard_normal(128).astype(np.float16), "bits": kb}
    v = {"codes": rng.integers(0, 1 << vb, (128, d)).astype(np.uint8),
         "scale": rng.standard_normal(128).astype(np.float16),
         "zero": rng.standard_normal(128).astype(np.float16),
         "factor": rng.standard_normal(d).astype(np.float16), "bits": vb}
    rec = ko.pack_record(k, v)
    assert len(rec) == ko.record_bytes(d, k_bits=kb, v_bits=vb)
    k2, v2 = ko.unpack_record(rec, d, kb, vb)
    for a, b in ((k, k2), (v, v2)):
        for key in a:
            np.testing.assert_array_equal(a[key], b[key])
    with pytest.raises(ValueError):   # a code wider than its section
        ko.pack_record(dict(k, codes=np.full((128, d), 1 << kb, np.uint16)), v)


def test_quantize_widths_closed_form_and_error_order():
    # the closed-form tile quantises to the extreme levels 0 and 2^b - 1 at every width
    r, c, x = _rank_one_scaled(128, 128, 11)
    tile = ko.rotate(x, 128)
    y = _checker(128, 128)
    for bits in (2, 4, 8):
        for kind in ("K", "V"):
            qd = ko.quantize_tile(tile, kind, bits=bits)
            assert qd["bits"] == bits
            np.testing.assert_array_equal(qd["codes"], ((2 ** bits - 1) * (y + 1) / 2).astype(np.uint8))
    # on outlier data more bits give a smaller reconstruction error, within half a step
    k, v = synth.outlier_kv(128, 1, 128, seed=14)
    for kind, t in (("K", k), ("V", v)):
        tile = t[:, 0].double().numpy()
        errs = []
        for bits in (2, 4, 8):
            qd = ko.quantize_tile(tile, kind, bits=bits)
            assert qd["codes"].max() <= 2 ** bits - 1
            back = ko.dequantize_tile(qd["codes"], qd["scale"], qd["zero"], qd["factor"], kind, 128)
            errs.append(np.linalg.norm(back - tile) / np.linalg.norm(tile))
            xr = ko.rotate(tile, 128)
            br = ko.rotate(back, 128)
            s = qd["scale"].astype(np.float64)
            f = qd["factor"].astype(np.float64)
            step = f[:, None] * s[None, :] if kind == "K" else s[:, None] * f[None, :]
            # half a step of rounding, plus the fp16 storage of factor, scale and zero (each
            # within 2^-11 relative): |f16(f)(q f16(s) + f16(z)) - f(q s + z)| <= 2^-10 f (q s + |z|)
            q = qd["codes"].astype(np.float64)
            z = np.abs(qd["zero"].astype(np.float64))
            meta = f[:, None] * (q * s[None, :] + z[None, :]) if kind == "K" else \
                f[None, :] * (q * s[:, None] + z[:, None])
            assert np.all(np.abs(br - xr) <= (0.5 * step + 2.0 ** -10 * meta) * 1.01 + 1e-6)
        assert errs[2] < errs[1] < errs[0]


def test_decode_sequence_presets_roundtrip():
    # decode over records of each preset equals attention over that preset's dequantised
    # tiles (pack/unpack/dequantise consistent at every width)
    k, v = synth.outlier_kv(256, 1, 128, seed=15)
    q = np.random.default_rng(15).standard_normal((2, 128))
    for name, (kb, vb) in ko.PRESETS.items():
        recs, ks, vs = [], [], []
        for p in range(2):
            kt = k[128 * p:128 * p + 128, 0].double().numpy()
            vt = v[128 * p:128 * p + 128, 0].double().numpy()
            rec, kq, vq = ko.quantize_page(kt, vt, k_bits=kb, v_bits=vb)
            recs.append(rec)
            ks.append(ko.dequantize_tile(kq["codes"], kq["scale"], kq["zero"], kq["factor"], "K", 128))
            vs.append(ko.dequantize_tile(vq["codes"], vq["scale"], vq["zero"], vq["factor"], "V", 128))
        got = ko.decode_sequence(q, recs, None, None, 0.1, 128, kb, vb)
        keys, vals = np.concatenate(ks), np.concatenate(vs)
        want = np.stack([ko.softmax_attention(qh, keys, vals, 0.1) for qh in q])
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12, err_msg=name)


# --- adaptive stop of the normalisation (hotdry §迭代方差归一化: three to five iterations typical) ---

def _iteration_changes(x, iters):
    """Largest |log factor change| of each iteration, recomputed from runs with fixed counts."""
    out = []
    prev_r, prev_c = np.ones(x.shape[-2]), np.ones(x.shape[-1])
    for t in range(1, iters + 1):
        _, r, c = ko.sinkhorn_normalise(x, t)
        out.append(max(np.abs(np.log(r / prev_r)).max(), np.abs(np.log(c / prev_c)).max()))
        prev_r, prev_c = r, c
    return out


def test_adaptive_stop_zero_tol_is_fixed():
    x = ko.rotate(synth.outlier_kv(128, 1, 128, seed=16)[0][:, 0].double().numpy(), 128)
    a = ko.sinkhorn_normalise(x, 4)
    n, r, c, used = ko.sinkhorn_normalise(x, 4, tol=0.0, return_iters=True)
    assert int(used) == 4
    for u, w in zip(a, (n, r, c)):
        np.testing.assert_array_equal(u, w)


def test_adaptive_stop_closed_form():
    # diag(r) Y diag(c) is normalised exactly by the first iteration, so the second moves
    # nothing and the iteration stops there
    _, _, x = _rank_one_scaled(128, 128, 21)
    n, r, c, used = ko.sinkhorn_normalise(x, 8, tol=1e-9, return_iters=True)
    assert int(used) == 2
    np.testing.assert_allclose(np.abs(n), 1.0, rtol=1e-12)


def test_adaptive_stop_rule_and_batching():
    # each tile stops at the first iteration whose largest log-factor change is <= tol
    # (changes recomputed independently from fixed-count runs); batched == one by one;
    # a looser tol never uses more iterations
    tiles = [ko.rotate(synth.outlier_kv(128, 1, 128, seed=30 + i)[j][:, 0].double().numpy(), 128)
             for i in range(3) for j in (0, 1)]
    for tol in (0.3, 0.05, 0.01):
        _, _, _, used = ko.sinkhorn_normalise(np.stack(tiles), 8, tol=tol, return_iters=True)
        for x, u in zip(tiles, used):
            ch = _iteration_changes(x, 8)
            want = next((t + 1 for t, v in enumerate(ch) if v <= tol), 8)
            assert int(u) == want, (tol, ch)
            _, _, _, u1 = ko.sinkhorn_normalise(x, 8, tol=tol, return_iters=True)
            assert int(u1) == int(u)
    u_loose = ko.sinkhorn_normalise(np.stack(tiles), 8, tol=0.3, return_iters=True)[3]
    u_tight = ko.sinkhorn_normalise(np.stack(tiles), 8, tol=0.01, return_iters=True)[3]
    assert np.all(u_loose <= u_tight)
    q = ko.quantize_tile(np.stack([t[:, :128] for t in tiles]), "K", tol=0.05)
    assert q["iters"].shape == (6,) and q["iters"].max() <= ko.SINKHORN_ITERS


# --- attention ----------------------------------------------------------------

def test_attention_single_token():
    rng = np.random.default_rng(20)
    vals = rng.standard_normal((1, 32))
    o = ko.softmax_attention(rng.standard_normal(32), rng.standard_normal((1, 32)), vals, 0.3)
    np.testing.assert_allclose(o, vals[0], rtol=1e-15)


def test_attention_identical_keys_give_mean():
    rng = np.random.default_rng(21)
    keys = np.tile(rng.standard_normal(16), (9, 1))
    vals = rng.standard_normal((9, 16))
    o = ko.softmax_attention(rng.standard_normal(16), keys, vals, 1.0)
    np.testing.assert_allclose(o, vals.mean(axis=0), rtol=1e-12)


def test_attention_matches_scipy_softmax_and_splits():
    rng = np.random.default_rng(22)
    q = rng.standard_normal(64)
    keys = rng.standard_normal((300, 64)) * 3
    vals = rng.standard_normal((300, 64))
    tau = 1 / 8
    ref = scipy.special.softmax(tau * keys @ q) @ vals
    o = ko.softmax_attention(q, keys, vals, tau)
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-14)
    # log-sum-exp merge of two halves gives the same result (split invariance)
    parts = []
    for sl in (slice(0, 137), slice(137, 300)):
        lg = tau * keys[sl] @ q
        mx = lg.max()
        w = np.exp(lg - mx)
        parts.append((mx, w.sum(), w @ vals[sl]))
    m = max(p[0] for p in parts)
    num = sum(np.exp(p[0] - m) * p[2] for p in parts)
    den = sum(np.exp(p[0] - m) * p[1] for p in parts)
    np.testing.assert_allclose(num / den, ref, rtol=1e-12, atol=1e-14)


def test_attention_large_logits_stay_finite():
    # logits in the hundreds: the max-shifted exponentials neither overflow nor lose the winner
    keys = np.zeros((4, 8))
    keys[:, 0] = [900.0, 100.0, -900.0, 899.0]
    vals = np.eye(4, 8)
    o = ko.softmax_attention(np.eye(8)[0], keys, vals, 1.0)
    assert np.all(np.isfinite(o))
    w = np.exp(-1.0)
    np.testing.assert_allclose(o[:4], [1 / (1 + w), 0, 0, w / (1 + w)], rtol=1e-12, atol=1e-300)


def test_fp16_decode_two_tokens_closed_form():
    # two keys whose scaled logits differ by ln 3: weights 3/4 and 1/4 for every query head
    tau = 0.5
    q = np.array([[1.0, 0.0, 0.0, 0.0], [2.0, 0.0, 0.0, 0.0]])
    keys = np.array([[2 * np.log(3.0), 0.0, 0.0, 0.0], [0.0, 5.0, 0.0, 0.0]])
    vals = np.array([[4.0, 0.0, -8.0, 1.0], [0.0, 4.0, 8.0, 1.0]])
    o = ko.fp16_decode_sequence(q, keys, vals, tau)
    np.testing.assert_allclose(o[0], [3.0, 1.0, -4.0, 1.0], rtol=1e-14)
    # the second head doubles the logit gap: weights 9/10 and 1/10
    np.testing.assert_allclose(o[1], [3.6, 0.4, -6.4, 1.0], rtol=1e-14)


def test_fp16_decode_paging_invariance():
    # the answer depends on the cached tokens only, not on how pages would split them: the
    # log-sum-exp merge of per-128-token parts equals the whole (what split-K computes)
    rng = np.random.default_rng(24)
    q = rng.standard_normal((4, 64))
    keys = rng.standard_normal((300, 64)) * 2
    vals = rng.standard_normal((300, 64))
    whole = ko.fp16_decode_sequence(q, keys, vals, 0.125)
    for gi in range(4):
        parts = []
        for a in range(0, 300, 128):
            lg = 0.125 * keys[a:a + 128] @ q[gi]
            w = np.exp(lg - lg.max())
            parts.append((lg.max(), w.sum(), w @ vals[a:a + 128]))
        m = max(p[0] for p in parts)
        num = sum(np.exp(p[0] - m) * p[2] for p in parts)
        den = sum(np.exp(p[0] - m) * p[1] for p in parts)
        np.testing.assert_allclose(whole[gi], num / den, rtol=1e-12, atol=1e-14)


def test_attention_empty_is_zero():
    o = ko.softmax_attention(np.ones(8), np.zeros((0, 8)), np.zeros((0, 8)), 1.0)
    np.testing.assert_array_equal(o, np.zeros(8))


def test_rotated_basis_logits_equal_original():
    # the decode kernel works in the rotated basis; orthonormality makes it the same
    # as attention over the dequantised cache in the original basis
    k, v = synth.outlier_kv(128, 1, 96, seed=23)
    qd = ko.quantize_tile(k[:, 0].double().numpy(), "K")
    kt_rot = qd["factor"].astype(np.float64)[:, None] * (
        qd["codes"] * qd["scale"].astype(np.float64)[None, :]
        + qd["zero"].astype(np.float64)[None, :])
    kh = ko.dequantize_tile(qd["codes"], qd["scale"], qd["zero"], qd["factor"], "K", 96)
    q = np.random.default_rng(24).standard_normal(96)
    np.testing.assert_allclose(kt_rot @ ko.rotate(q, 128), kh @ q, rtol=1e-10, atol=1e-9)


def test_tiny_quality_figure():
    # quality figure (reported, loosely gated): attention over the K4V2 cache vs fp16 cache
    k, v, q = synth.tiny_case()
    rec, _, _ = ko.quantize_page(k[:, 0].double().numpy(), v[:, 0].double().numpy())
    o = ko.decode_sequence(q[0].double().numpy(), [rec], None, None, 1 / math.sqrt(128), 128)
    ref = ko.softmax_attention(q[0, 0].double().numpy(), k[:, 0].double().numpy(),
                               v[:, 0].double().numpy(), 1 / math.sqrt(128))
    cos = float(o[0] @ ref / np.linalg.norm(o[0]) / np.linalg.norm(ref))
    print("tiny attention-output cosine vs fp16 cache: %.5f" % cos)
    assert cos > 0.9


# --- chunked prefill (the step before decode over the same packed cache) -------------------

def _small_cache(seed, pages, part):
    k, v = synth.outlier_kv(128 * pages + part, 1, 128, seed=seed)
    recs = [ko.quantize_page(k[128 * i:128 * i + 128, 0].double().numpy(),
                             v[128 * i:128 * i + 128, 0].double().numpy())[0] for i in range(pages)]
    pk = k[128 * pages:, 0].double().numpy()
    pv = v[128 * pages:, 0].double().numpy()
    return recs, pk, pv


def test_prefill_single_token_is_decode_with_it_appended():
    recs, pk, pv = _small_cache(70, 2, 5)
    rng = np.random.default_rng(70)
    q = rng.standard_normal((1, 3, 128))
    ck, cv = rng.standard_normal((1, 128)), rng.standard_normal((1, 128))
    got = ko.prefill_sequence(q, recs, pk, pv, ck, cv, 0.09, 128)
    want = ko.decode_sequence(q[0], recs, np.concatenate([pk, ck]), np.concatenate([pv, cv]), 0.09, 128)
    np.testing.assert_allclose(got[0], want, rtol=0, atol=1e-12)


def test_prefill_is_causal():
    # changing chunk token t changes no output before t, and changes the output at t
    recs, pk, pv = _small_cache(71, 1, 0)
    rng = np.random.default_rng(71)
    q = rng.standard_normal((6, 2, 128))
    ck, cv = rng.standard_normal((6, 128)), rng.standard_normal((6, 128))
    a = ko.prefill_sequence(q, recs, pk, pv, ck, cv, 0.1, 128)
    ck2, cv2 = ck.copy(), cv.copy()
    ck2[3] = 400.0 * q[3, 0] / np.linalg.norm(q[3, 0])   # dominates query 3's first head
    cv2[3] -= 3.0
    b = ko.prefill_sequence(q, recs, pk, pv, ck2, cv2, 0.1, 128)
    np.testing.assert_array_equal(a[:3], b[:3])
    assert np.abs(a[3:] - b[3:]).max() > 1e-3


def test_prefill_empty_cache_is_causal_self_attention():
    # with nothing cached, token c attends to chunk tokens 0..c only: token 0 returns v_0
    rng = np.random.default_rng(72)
    q = rng.standard_normal((4, 1, 64))
    ck, cv = rng.standard_normal((4, 64)), rng.standard_normal((4, 64))
    out = ko.prefill_sequence(q, [], None, None, ck, cv, 0.125, 64)
    np.testing.assert_allclose(out[0, 0], cv[0], rtol=0, atol=1e-12)
    w = np.exp(0.125 * ck[:3] @ q[2, 0] - (0.125 * ck[:3] @ q[2, 0]).max())
    np.testing.assert_allclose(out[2, 0], (w / w.sum()) @ cv[:3], rtol=1e-12, atol=1e-12)


# --- quantisation-error telemetry (hotdry §监控要点) ----------------------------------------

def _stats(tile, kind, bits=None):
    q = ko.quantize_tile(tile, kind, bits=bits)
    return ko.quantization_error(tile, q["codes"], q["scale"], q["zero"], q["factor"], kind), q


@pytest.mark.parametrize("kind", ["K", "V"])
def test_quantization_error_equals_rotated_domain_error(kind):
    # the rotation is orthonormal, so at d0 = d the original-basis error equals the error of
    # the stored values against X = rotate(tile) in the rotated domain, computed here without
    # any inverse rotation
    k, v = synth.outlier_kv(128, 1, 128, seed=31)
    tile = (k if kind == "K" else v)[:, 0].double().numpy()
    st, q = _stats(tile, kind)
    x = ko.rotate(tile, 128)
    s, z, f = (q[n].astype(np.float64) for n in ("scale", "zero", "factor"))
    if kind == "K":
        xt = f[:, None] * (q["codes"] * s[None, :] + z[None, :])
    else:
        xt = f[None, :] * (q["codes"] * s[:, None] + z[:, None])
    np.testing.assert_allclose(st[0], np.sum((x - xt) ** 2), rtol=1e-10)
    np.testing.assert_allclose(st[1], np.sum(tile ** 2), rtol=1e-12)
    assert st[3] == np.max(np.abs(tile))
    assert 0 < st[0] < st[1] and 0 < st[2] <= st[3]


def test_quantization_error_scales_with_powers_of_two():
    # every step is equivariant under x -> 2^k x (fp16 metadata rounding included), so the two
    # sums scale by 4^k and the two maxima by 2^k
    k, _ = synth.outlier_kv(128, 1, 96, seed=32)
    tile = k[:, 0].double().numpy()
    a, _ = _stats(tile, "K")
    b, _ = _stats(tile * 8.0, "K")
    np.testing.assert_allclose(b, a * np.array([64.0, 64.0, 8.0, 8.0]), rtol=1e-9)


def test_quantization_error_falls_with_code_width():
    # more code bits on the same tile give a smaller reconstruction error
    _, v = synth.outlier_kv(128, 1, 128, seed=33)
    tile = v[:, 0].double().numpy()
    e2, e4, e8 = (_stats(tile, "V", bits=b)[0][0] for b in (2, 4, 8))
    assert e8 < e4 < e2


def test_quantization_error_of_a_zero_tile():
    st, _ = _stats(np.zeros((128, 128)), "K")
    np.testing.assert_array_equal(st, np.zeros(4))
