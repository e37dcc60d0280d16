"""Quantisation-error telemetry (kvarn_quantization_error) against the float64 oracle (GPU).

The statistics are computed from the same packed bytes on both sides: the GPU-written records
are unpacked by the oracle, which dequantises them in float64 and compares them with the same
fp16 source tiles [hotdry §监控要点: sample the dequantised values, watch the error].
Tolerances: the two sums within 1e-4 relative (float32 accumulation of 128 x d0 terms), the
maxima within 1e-4 of max |x| (float32 dequantisation of the same bytes).
"""

import numpy as np
import pytest
import torch

from calibration_free_kv_gb300 import synth
from oracle import kvarn_oracle as ko
from tests import helpers as H

pytestmark = pytest.mark.gpu

SUM_RTOL = 1e-4
MAX_TOL = 1e-4


@pytest.fixture(scope="module")
def kv():
    from calibration_free_kv_gb300 import build
    build.build()
    from calibration_free_kv_gb300 import kvarn
    return kvarn


@pytest.mark.parametrize("d0,hkv,tiles,preset", [(128, 2, 3, "kvarn_k4v2_g128"), (96, 2, 2, "kvarn_k4v2_g128"),
                                                 (256, 1, 2, "kvarn_k4v2_g128"), (64, 2, 2, "kvarn_k2v2_g128"),
                                                 (128, 1, 2, "kvarn_k8v4_g128")])
def test_error_stats_match_oracle(kv, d0, hkv, tiles, preset):
    k, v = synth.outlier_kv(128 * tiles, hkv, d0, seed=40 + d0 + tiles, device="cuda")
    desc = kv.desc_from_preset(d0, hkv, preset=preset)
    ids = torch.randperm(tiles + 3, generator=torch.Generator().manual_seed(d0))[:tiles]
    ids = ids.to(torch.int32).cuda()
    pool = kv.alloc_pool(desc, tiles + 3)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.quantize_tiles(desc, k, v, ids, pool, status=status)
    err = torch.full((tiles, hkv, 2, 4), float("nan"), dtype=torch.float32, device="cuda")
    kv.quantization_error(desc, k, v, ids, pool, err, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = err.cpu().double().numpy()
    kc, vc = k.cpu().double().numpy(), v.cpu().double().numpy()
    d = desc.head_dim_padded
    for t in range(tiles):
        for h in range(hkv):
            rk, rv = ko.unpack_record(H.record_bytes_of(pool, int(ids[t]), h), d, desc.k_bits, desc.v_bits)
            for half, (src, r, kind) in enumerate(((kc, rk, "K"), (vc, rv, "V"))):
                tile = src[128 * t:128 * t + 128, h]
                want = ko.quantization_error(tile, r["codes"], r["scale"], r["zero"], r["factor"], kind)
                g = got[t, h, half]
                np.testing.assert_allclose(g[:2], want[:2], rtol=SUM_RTOL, err_msg="%s sums" % kind)
                assert abs(g[2] - want[2]) <= MAX_TOL * want[3], (kind, g, want)
                assert abs(g[3] - want[3]) <= MAX_TOL * want[3], (kind, g, want)
                # the relative error is the quality figure this feeds: finite and below 1
                assert 0.0 < g[0] < g[1]


def test_error_stats_on_a_sample_of_tiles(kv):
    # a monitor samples: tile 5 alone (pointer offset into the layer, its own page id) gives
    # the same statistics as in the full pass
    hkv, d0, tiles = 2, 128, 8
    k, v = synth.outlier_kv(128 * tiles, hkv, d0, seed=51, device="cuda")
    desc = kv.desc_from_preset(d0, hkv)
    ids = torch.arange(tiles, dtype=torch.int32, device="cuda")
    pool = kv.alloc_pool(desc, tiles)
    kv.quantize_tiles(desc, k, v, ids, pool)
    full = torch.zeros((tiles, hkv, 2, 4), dtype=torch.float32, device="cuda")
    kv.quantization_error(desc, k, v, ids, pool, full)
    one = torch.zeros((1, hkv, 2, 4), dtype=torch.float32, device="cuda")
    kv.quantization_error(desc, k[640:768], v[640:768], ids[5:6].contiguous(), pool, one)
    torch.cuda.synchronize()
    assert torch.equal(one[0], full[5])
