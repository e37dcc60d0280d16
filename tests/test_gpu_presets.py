"""The other k/v bit presets (kvarn_k4v4_g128, kvarn_k2v2_g128, kvarn_k8v4_g128) through the
same GPU pipeline, against the float64 oracle at the same widths: quantisation,
dequantisation, decode over an oracle-built cache (with raw partial tiles, GQA 4 and 8), and
append sealing."""

import math

import numpy as np
import pytest
import torch

from calibration_free_kv_gb300 import synth
from oracle import kvarn_oracle as ko
from tests import helpers as H

pytestmark = pytest.mark.gpu

OTHER = ["kvarn_k4v4_g128", "kvarn_k2v2_g128", "kvarn_k8v4_g128"]


@pytest.fixture(scope="module")
def kv():
    from calibration_free_kv_gb300 import build
    build.build()
    from calibration_free_kv_gb300 import kvarn
    return kvarn


def test_preset_descriptors(kv):
    for name, (kb, vb) in ko.PRESETS.items():
        for d0 in (64, 96, 128, 256):
            desc = kv.desc_from_preset(d0, 2, preset=name)
            assert (desc.k_bits, desc.v_bits) == (kb, vb)
            assert desc.page_record_bytes == ko.record_bytes(ko.padded_head_dim(d0), k_bits=kb, v_bits=vb)
    with pytest.raises(kv.KvarnError):
        kv.desc_from_preset(128, 2, preset="kvarn_k3v2_g128")


@pytest.mark.parametrize("preset", OTHER)
@pytest.mark.parametrize("d0,hkv,tiles", [(128, 2, 3), (96, 1, 2), (64, 2, 2), (256, 1, 2)])
def test_preset_quantize_and_dequantize(kv, preset, d0, hkv, tiles):
    kb, vb = ko.PRESETS[preset]
    k, v = synth.outlier_kv(128 * tiles, hkv, d0, seed=40 + d0 + kb, device="cuda")
    desc = kv.desc_from_preset(d0, hkv, preset=preset)
    ids = torch.arange(tiles - 1, -1, -1, dtype=torch.int32, device="cuda")
    pool = kv.alloc_pool(desc, tiles)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.quantize_tiles(desc, k, v, ids, pool, status=status)
    ko_ = torch.empty((tiles, hkv, 128, d0), dtype=torch.float16, device="cuda")
    vo_ = torch.empty_like(ko_)
    kv.dequantize_tiles(desc, pool, ids, ko_, vo_, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kc, vc = k.cpu().double().numpy(), v.cpu().double().numpy()
    d = desc.head_dim_padded
    stats = []
    pids = ids.cpu().numpy()
    for t in range(tiles):
        kt = np.stack([kc[128 * t:128 * t + 128, h] for h in range(hkv)])
        vt = np.stack([vc[128 * t:128 * t + 128, h] for h in range(hkv)])
        _, kq, vq = H.oracle_quantize(kt, vt, k_bits=kb, v_bits=vb)
        for h in range(hkv):
            rec = H.record_bytes_of(pool, int(pids[t]), h)
            H.compare_record(rec, H.tile_of(kq, h), H.tile_of(vq, h), d, stats, kb, vb)
            # dequantisation of the GPU's own bytes against the oracle's reading of them
            kh, vh = ko.dequantize_record(rec, d0, kb, vb)
            for got, want in ((ko_[t, h], kh), (vo_[t, h], vh)):
                g = got.cpu().double().numpy()
                tol = H.DEQUANT_RTOL * np.abs(want) + 1e-5 * np.abs(want).max()
                assert np.all(np.abs(g - want) <= tol), np.abs(g - want).max()
    bad, total = H.assert_mismatch_budget(stats)
    print("%s d0=%d: %d of %d codes on a boundary differ" % (preset, d0, bad, total))


def _oracle_cache_decode(kv, preset, d0, group, seq_lens, seed, **synth_kw):
    kb, vb = ko.PRESETS[preset]
    hkv = 2
    batch = len(seq_lens)
    g = torch.Generator().manual_seed(seed)
    pages = [L // 128 for L in seq_lens]
    n_pool = sum(pages) + 1
    perm = torch.randperm(n_pool, generator=g).tolist()
    width = max(max(pages), 1)
    table = np.zeros((batch, width), dtype=np.int32)
    desc = kv.desc_from_preset(d0, hkv, preset=preset)
    pool = kv.alloc_pool(desc, n_pool)
    pk = torch.zeros((batch, hkv, 128, d0), dtype=torch.float16)
    pv = torch.zeros_like(pk)
    recs, tails = {}, {}
    off = 0
    for b, L in enumerate(seq_lens):
        k, v = synth.outlier_kv(max(L, 1), hkv, d0, seed=seed * 100 + b, **synth_kw)
        k, v = k[:L], v[:L]
        n = pages[b]
        table[b, :n] = perm[off:off + n]
        off += n
        if n:
            kk = k[:128 * n].double().numpy().reshape(n, 128, hkv, d0)
            vv = v[:128 * n].double().numpy().reshape(n, 128, hkv, d0)
            for h in range(hkv):
                r, _, _ = H.oracle_quantize(kk[:, :, h], vv[:, :, h], k_bits=kb, v_bits=vb)
                for i in range(n):
                    recs[(b, i, h)] = r[i]
        rem = L - 128 * n
        if rem:
            pk[b, :, :rem] = k[128 * n:].transpose(0, 1)
            pv[b, :, :rem] = v[128 * n:].transpose(0, 1)
        tails[b] = (k[128 * n:], v[128 * n:])
    H.upload_records(pool, [(int(table[b, i]), h, r) for (b, i, h), r in recs.items()])
    q = torch.randn((batch, hkv * group, d0), generator=g).half()
    out = torch.empty((batch, hkv * group, d0), dtype=torch.float16, device="cuda")
    ws = kv.alloc_workspace(desc, batch, hkv * group, width)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d0)
    kv.decode_attention(desc, q.cuda(), pool, torch.from_numpy(table).cuda(),
                        torch.tensor(seq_lens, dtype=torch.int32, device="cuda"), out, ws,
                        partial_k=pk.cuda(), partial_v=pv.cuda(), softmax_scale=scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().double().numpy()
    worst = 0.0
    for b, L in enumerate(seq_lens):
        tk, tv = tails[b]
        for h in range(hkv):
            rl = [recs[(b, i, h)] for i in range(pages[b])]
            ref = ko.decode_sequence(q[b, h * group:(h + 1) * group].double().numpy(), rl,
                                     tk[:, h].double().numpy() if len(tk) else None,
                                     tv[:, h].double().numpy() if len(tv) else None, scale, d0, kb, vb)
            worst = max(worst, H.assert_decode_close(got[b, h * group:(h + 1) * group], ref,
                                                     "%s d0=%d G=%d b=%d h=%d" % (preset, d0, group, b, h)))
    return worst


@pytest.mark.parametrize("preset", OTHER)
@pytest.mark.parametrize("d0,group", [(128, 4), (128, 8), (96, 4), (64, 8), (256, 4)])
def test_preset_decode_parity(kv, preset, d0, group):
    err = _oracle_cache_decode(kv, preset, d0, group, [0, 77, 128, 1000, 4096 + 5, 300], seed=7 + d0)
    print("%s d0=%d G=%d: max scaled error %.2e" % (preset, d0, group, err))


@pytest.mark.parametrize("preset", ["kvarn_k4v2_g128"] + OTHER)
@pytest.mark.parametrize("d0,group", [(128, 4), (128, 8)])
def test_preset_decode_extreme_outliers(kv, preset, d0, group):
    # outlier channels x1000..x4000 (values up to the fp16 clamp of 60000): the lifted QK
    # operand and the PV weights stay finite and the output matches the oracle
    err = _oracle_cache_decode(kv, preset, d0, group, [77, 1000, 4096 + 5], seed=21 + d0,
                               scale_lo=1000.0, scale_hi=4000.0)
    print("%s d0=%d G=%d, outliers x1000..x4000: max scaled error %.2e" % (preset, d0, group, err))


@pytest.mark.parametrize("preset", OTHER)
def test_preset_append_seals_like_batch(kv, preset):
    # tokens appended one at a time seal into the same bytes as batch quantisation of the tile
    desc = kv.desc_from_preset(128, 2, preset=preset)
    batch, hkv, d0 = 2, 2, 128
    l0 = [120, 3]
    table = torch.tensor([[1, 0], [2, 3]], dtype=torch.int32, device="cuda")
    pool = kv.alloc_pool(desc, 4)
    pk = torch.zeros((batch, hkv, 128, d0), dtype=torch.float16, device="cuda")
    pv = torch.zeros_like(pk)
    g = torch.Generator().manual_seed(3)
    toks = (torch.randn((batch, 140, hkv, d0), generator=g) * 2).half()
    for b, L in enumerate(l0):
        pk[b, :, :L] = toks[b, :L].transpose(0, 1).cuda()
        pv[b, :, :L] = (toks[b, :L] * 0.5).transpose(0, 1).cuda()
    lens = [torch.tensor(l0, dtype=torch.int32, device="cuda"), torch.zeros(batch, dtype=torch.int32, device="cuda")]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cur = 0
    for step in range(10):
        idx = torch.tensor(l0) + step
        kn = torch.stack([toks[b, int(idx[b])] for b in range(batch)]).cuda()
        vn = torch.stack([toks[b, int(idx[b])] * 0.5 for b in range(batch)]).cuda()
        kv.append_token(desc, kn, vn, pk, pv, lens[cur], table, pool, seq_lens_out=lens[1 - cur], status=status)
        cur = 1 - cur
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # sequence 0 sealed its first page (tokens 0..127) into page table[0, 0] = 1
    ref = kv.alloc_pool(desc, 1)
    kv.quantize_tiles(desc, toks[0, :128].cuda().contiguous(), (toks[0, :128] * 0.5).cuda().contiguous(),
                      torch.zeros(1, dtype=torch.int32, device="cuda"), ref)
    torch.cuda.synchronize()
    assert torch.equal(pool[1], ref[0])
