"""Chunked-prefill attention on the GPU against the float64 oracle (through the C ABI).

The packed cache is built by the oracle (its records uploaded), so every expected value
comes from the CPU side; the chunk's own keys and values are raw fp16."""

import math

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


def _prefill_case(kv, cache_lens, chunk, hkv, group, d0, seed, preset="kvarn_k4v2_g128"):
    kb, vb = ko.PRESETS[preset]
    batch = len(cache_lens)
    g = torch.Generator().manual_seed(seed)
    pages = [L // 128 for L in cache_lens]
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
    for b, L in enumerate(cache_lens):
        k, v = synth.outlier_kv(max(L, 1), hkv, d0, seed=seed * 100 + b)
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
    q = torch.randn((batch, chunk, hkv * group, d0), generator=g).half()
    ck = (torch.randn((batch, chunk, hkv, d0), generator=g) * 2).half()
    cv = torch.randn((batch, chunk, hkv, d0), generator=g).half()
    out = torch.full((batch, chunk, hkv * group, d0), float("nan"), dtype=torch.float16, device="cuda")
    ws = kv.alloc_prefill_workspace(desc, batch, hkv * group, chunk, width)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d0)
    kv.prefill_attention(desc, q.cuda(), ck.cuda(), cv.cuda(), pool, torch.from_numpy(table).cuda(),
                         torch.tensor(cache_lens, dtype=torch.int32, device="cuda"), out, ws,
                         partial_k=pk.cuda(), partial_v=pv.cuda(), softmax_scale=scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().double().numpy()
    worst = 0.0
    for b in range(batch):
        tk, tv = tails[b]
        for h in range(hkv):
            rl = [recs[(b, i, h)] for i in range(pages[b])]
            ref = ko.prefill_sequence(q[b, :, h * group:(h + 1) * group].double().numpy(), rl,
                                      tk[:, h].double().numpy() if len(tk) else None,
                                      tv[:, h].double().numpy() if len(tv) else None,
                                      ck[b, :, h].double().numpy(), cv[b, :, h].double().numpy(),
                                      scale, d0, kb, vb)
            for c in range(chunk):
                worst = max(worst, H.assert_decode_close(got[b, c, h * group:(h + 1) * group], ref[c],
                                                         "prefill b=%d c=%d h=%d" % (b, c, h)))
    return worst


@pytest.mark.parametrize("chunk,group,d0", [(1, 4, 128), (5, 4, 128), (16, 8, 128), (7, 1, 96),
                                            (9, 8, 64), (6, 4, 256), (3, 8, 256)])
def test_prefill_parity(kv, chunk, group, d0):
    err = _prefill_case(kv, [0, 77, 128, 1000, 2 * 4096 + 5], chunk, 2, group, d0, seed=chunk + group + d0)
    print("prefill chunk=%d G=%d d0=%d: max scaled error %.2e" % (chunk, group, d0, err))


@pytest.mark.parametrize("preset", ["kvarn_k4v4_g128", "kvarn_k2v2_g128", "kvarn_k8v4_g128"])
def test_prefill_other_presets(kv, preset):
    err = _prefill_case(kv, [300, 4096], 8, 2, 4, 128, seed=11, preset=preset)
    print("prefill %s: max scaled error %.2e" % (preset, err))


def test_prefill_long_chunk(kv):
    # a 33-token chunk over one long cached sequence, GQA 4
    err = _prefill_case(kv, [16384 + 40], 33, 1, 4, 128, seed=12)
    print("prefill chunk 33 over 16424 cached tokens: max scaled error %.2e" % err)


@pytest.mark.parametrize("chunk,group,d0,cache_lens", [(150, 4, 128, [0, 300]), (130, 8, 96, [200]),
                                                       (70, 1, 64, [129])])
def test_prefill_multi_block_chunk(kv, chunk, group, d0, cache_lens):
    # chunks longer than one 64-token stage of the causal part and query rows over several CTAs
    # of 128 rows (600, 1040 and 70 rows), so the online softmax runs over 2-3 stages and rows
    # past the chunk's end pad the last CTA
    err = _prefill_case(kv, cache_lens, chunk, 1, group, d0, seed=chunk + group)
    print("prefill chunk=%d G=%d d0=%d: max scaled error %.2e" % (chunk, group, d0, err))


def test_prefill_chunk64(kv):
    # the bench's prefill shape at a smaller batch: 64-token chunks, GQA 4 (256 query vectors
    # per kv head, four CTAs of 64), 8195 and 2000 cached tokens
    err = _prefill_case(kv, [8192 + 3, 2000], 64, 2, 4, 128, seed=13)
    print("prefill chunk 64: max scaled error %.2e" % err)
