"""GPU quantise / dequantise kernels against the float64 oracle (through the C ABI)."""

import numpy as np
import pytest
import torch

from calibration_free_kv_gb300 import synth
from oracle import kvarn_oracle as ko
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kv():
    from calibration_free_kv_gb300 import build
    build.build()
    from calibration_free_kv_gb300 import kvarn
    return kvarn


def _quantize_and_compare(kv, k, v, d0, page_ids=None, iters=None, check_units=None):
    """k, v: fp16 CUDA [tokens, Hkv, d0].  Quantises on the GPU and compares the records of
    `check_units` ((tile, head) pairs; all when None) with the oracle."""
    tokens, hkv, _ = k.shape
    n_tiles = tokens // 128
    desc = kv.desc_from_preset(d0, hkv, sinkhorn_iters=iters)
    if page_ids is None:
        page_ids = torch.arange(n_tiles, dtype=torch.int32, device="cuda")
    n_pool = int(page_ids.max().item()) + 1
    pool = kv.alloc_pool(desc, n_pool)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.quantize_tiles(desc, k, v, page_ids, pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    if check_units is None:
        check_units = [(t, h) for t in range(n_tiles) for h in range(hkv)]
    kc = k.cpu().double().numpy()
    vc = v.cpu().double().numpy()
    kt = np.stack([kc[128 * t:128 * t + 128, h] for t, h in check_units])
    vt = np.stack([vc[128 * t:128 * t + 128, h] for t, h in check_units])
    _, kq, vq = H.oracle_quantize(kt, vt, iters=desc.sinkhorn_iters)
    d = desc.head_dim_padded
    stats = []
    pids = page_ids.cpu().numpy()
    for i, (t, h) in enumerate(check_units):
        rec = H.record_bytes_of(pool, int(pids[t]), h)
        H.compare_record(rec, H.tile_of(kq, i), H.tile_of(vq, i), d, stats)
    bad, total = H.assert_mismatch_budget(stats)
    return desc, pool, bad, total


@pytest.mark.parametrize("d0", [128])
def test_tiny_quantize_parity(kv, d0):
    k, v, _ = synth.tiny_case("cuda")
    _, _, bad, total = _quantize_and_compare(kv, k, v, d0)
    print("tiny: %d of %d codes on a boundary differ" % (bad, total))


@pytest.mark.parametrize("d0,hkv,tiles", [(128, 2, 3), (96, 3, 2), (256, 2, 2), (64, 2, 2), (200, 1, 2)])
def test_quantize_parity_shapes(kv, d0, hkv, tiles):
    k, v = synth.outlier_kv(128 * tiles, hkv, d0, seed=100 + d0, device="cuda")
    perm = torch.randperm(tiles + 3, generator=torch.Generator().manual_seed(d0))[:tiles]
    _quantize_and_compare(kv, k, v, d0, page_ids=perm.to(torch.int32).cuda())


def test_quantize_strided_input(kv):
    # heads interleaved in a wider buffer: token stride 3*Hkv*d0, head stride d0
    base_k, base_v = synth.outlier_kv(256, 6, 128, seed=7, device="cuda")
    k = base_k[:, ::2]
    v = base_v[:, ::2]
    assert k.stride() == (6 * 128, 256, 1)
    _quantize_and_compare(kv, k, v, 128)


@pytest.mark.parametrize("iters", [0, 1, 8])
def test_quantize_iteration_counts(kv, iters):
    k, v = synth.outlier_kv(256, 2, 128, seed=11, device="cuda")
    _quantize_and_compare(kv, k, v, 128, iters=iters)


def test_quantize_degenerate_tiles(kv):
    # zero tile, constant tile, one huge outlier, a row of zeros
    k = torch.zeros((512, 1, 128), dtype=torch.float16, device="cuda")
    k[128:256] = 3.0
    k[256:384, 0, 17] = 60000.0
    k[384:512] = torch.randn((128, 1, 128), generator=torch.Generator().manual_seed(5)).half().cuda()
    k[384 + 5] = 0.0
    v = k.flip(0).contiguous()
    _quantize_and_compare(kv, k, v, 128)


def test_quantize_full_size_sampled(kv):
    # one layer, 8 KV heads x 16384 tokens x head_dim 128 (the quantise-throughput workload)
    k, v = synth.outlier_kv(16384, 8, 128, seed=2, device="cuda")
    rng = np.random.default_rng(2)
    units = sorted({(int(rng.integers(128)), int(rng.integers(8))) for _ in range(48)})
    units += [(0, 0), (127, 7)]
    desc, pool, bad, total = _quantize_and_compare(kv, k, v, 128, check_units=units)
    print("full size: %d of %d sampled codes on a boundary differ" % (bad, total))
    # bit-identical on a second run (no nondeterminism in the kernel)
    pool2 = kv.alloc_pool(desc, 128)
    kv.quantize_tiles(desc, k, v, torch.arange(128, dtype=torch.int32, device="cuda"), pool2)
    torch.cuda.synchronize()
    assert torch.equal(pool, pool2)
    # the fp16 metadata of every record is finite
    o_kc, o_vc, o_ks, _, _, o_vs, _, _ = ko._section_offsets(128)
    for lo, hi in ((o_ks, o_vc), (o_vs, pool.shape[-1])):
        meta = pool[:, :, lo:hi].contiguous().view(torch.float16)
        assert torch.isfinite(meta.float()).all()


@pytest.mark.parametrize("d0", [128, 96, 256])
def test_dequantize_parity(kv, d0):
    hkv, tiles = 2, 3
    k, v = synth.outlier_kv(128 * tiles, hkv, d0, seed=30 + d0, device="cuda")
    desc = kv.desc_from_preset(d0, hkv)
    ids = torch.tensor([2, 0, 1], dtype=torch.int32, device="cuda")
    pool = kv.alloc_pool(desc, tiles)
    kv.quantize_tiles(desc, k, v, ids, pool)
    ko_ = torch.empty((tiles, hkv, 128, d0), dtype=torch.float16, device="cuda")
    vo_ = torch.empty_like(ko_)
    kv.dequantize_tiles(desc, pool, ids, ko_, vo_)
    torch.cuda.synchronize()
    kc, vc = ko_.cpu().double().numpy(), vo_.cpu().double().numpy()
    for i, p in enumerate(ids.cpu().tolist()):
        for h in range(hkv):
            kh, vh = ko.dequantize_record(H.record_bytes_of(pool, p, h), d0)
            for g, o in ((kc[i, h], kh), (vc[i, h], vh)):
                tol = H.DEQUANT_RTOL * np.abs(o) + 1e-5 * np.abs(o).max()
                assert np.all(np.abs(g - o) <= tol), np.abs(g - o).max()
            # quality figure: the round trip stays close to the input
            src = k[128 * i:128 * i + 128, h].double().cpu().numpy()
            rel = np.linalg.norm(kc[i, h] - src) / np.linalg.norm(src)
            assert rel < 0.2


@pytest.mark.parametrize("d0", [128, 256])
def test_quantize_page_id_outside_pool(kv, d0):
    # a tile whose page id lies outside the pool is flagged and writes nothing; the other tiles
    # are quantised as usual and the pool keeps no stray bytes
    k, v = synth.outlier_kv(128 * 3, 2, d0, seed=61, device="cuda")
    desc = kv.desc_from_preset(d0, 2)
    pool = kv.alloc_pool(desc, 3)
    pool.fill_(0xA5)
    ids = torch.tensor([2, 7, 0], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.quantize_tiles(desc, k, v, ids, pool, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & kv.DEV_BAD_PAGE_ID
    assert bool((pool[1] == 0xA5).all()), "page 1 (no tile) was written"
    ref = kv.alloc_pool(desc, 3)
    kv.quantize_tiles(desc, k, v, torch.tensor([2, 1, 0], dtype=torch.int32, device="cuda"), ref)
    torch.cuda.synchronize()
    assert torch.equal(pool[0], ref[0]) and torch.equal(pool[2], ref[2])
