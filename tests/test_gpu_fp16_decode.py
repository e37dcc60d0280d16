"""GPU uncompressed fp16 paged decode (the baseline kernel) against the float64 oracle.

The fp16 cache is written by torch indexing from seeded synthetic K/V; rows of a partly
filled last page and every unused page are filled with NaN, so reading a row past a
sequence's length shows up as a non-finite output.
"""

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


def _build(hkv, group, d, seq_lens, seed, max_pages=None):
    g = torch.Generator().manual_seed(seed)
    pages = [(L + 127) // 128 for L in seq_lens]
    n_pool = sum(pages) + 2
    perm = torch.randperm(n_pool, generator=g).tolist()
    width = max_pages or max(max(pages), 1)
    table = np.zeros((len(seq_lens), width), dtype=np.int32)
    pool = torch.full((n_pool, hkv, 2, 128, d), float("nan"), dtype=torch.float16)
    seqs = []
    off = 0
    for b, L in enumerate(seq_lens):
        k, v = synth.outlier_kv(max(L, 1), hkv, d, seed=seed * 1000 + b)
        k, v = k[:L], v[:L]
        seqs.append((k, v))
        for i in range(pages[b]):
            pid = perm[off + i]
            table[b, i] = pid
            rows = min(128, L - 128 * i)
            pool[pid, :, 0, :rows] = k[128 * i:128 * i + rows].transpose(0, 1)
            pool[pid, :, 1, :rows] = v[128 * i:128 * i + rows].transpose(0, 1)
        off += pages[b]
    q = torch.randn((len(seq_lens), hkv * group, d), generator=g).half()
    return seqs, table, pool, q


def _run(kv, hkv, q, pool, table, seq_lens, scale):
    batch, hq, d = q.shape
    out = torch.empty((batch, hq, d), dtype=torch.float16, device="cuda")
    ws = kv.alloc_fp16_workspace(d, batch, hq, table.shape[1])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.fp16_decode_attention(hkv, q.cuda(), pool.cuda(), torch.from_numpy(table).cuda(),
                             torch.tensor(seq_lens, dtype=torch.int32, device="cuda"), out, ws,
                             softmax_scale=scale, status=status)
    torch.cuda.synchronize()
    return out.cpu().double().numpy(), int(status.item())


def _check(got, seqs, q, hkv, group, scale, only=None):
    err = 0.0
    for b, (k, v) in enumerate(seqs):
        for h in range(hkv):
            if only is not None and (b, h) not in only:
                continue
            ref = ko.fp16_decode_sequence(q[b, h * group:(h + 1) * group].double().numpy(),
                                          k[:, h].double().numpy(), v[:, h].double().numpy(), scale)
            err = max(err, H.assert_decode_close(got[b, h * group:(h + 1) * group], ref,
                                                 "fp16 decode b=%d h=%d" % (b, h)))
    return err


@pytest.mark.parametrize("d,group", [(128, 4), (128, 1), (128, 2), (128, 8), (64, 4), (64, 8)])
def test_fp16_decode_parity_ragged(kv, d, group):
    # lengths: empty, one token, a partly filled page, exactly one page, a page and a token,
    # several pages with a tail, more pages than one split (32) holds
    seq_lens = [0, 1, 77, 128, 129, 300, 17 * 128 + 5, 33 * 128 + 77]
    hkv = 2
    seqs, table, pool, q = _build(hkv, group, d, seq_lens, seed=d + group)
    scale = 1.0 / math.sqrt(d)
    got, st = _run(kv, hkv, q, pool, table, seq_lens, scale)
    assert st == 0
    assert np.all(np.isfinite(got))
    assert np.all(got[0] == 0.0)  # length 0 attends to nothing
    err = _check(got, seqs, q, hkv, group, scale)
    print("fp16 decode d=%d G=%d: max scaled err %.2e" % (d, group, err))


def test_fp16_decode_full_size_sampled(kv):
    # the decode workload at full size (batch 64, 128 * U{8..128} tokens + 77, 32 q heads over
    # 8 kv heads, head_dim 128, permuted block table); three sampled (sequence, kv head)
    # outputs against the oracle, every output finite
    hkv, group, d, batch = 8, 4, 128, 64
    shape = synth.decode_batch(batch, hkv * group, hkv, d, seed=3, min_pages=8, max_pages=128)
    seq_lens = [int(L) + 77 for L in shape["seq_lens"].tolist()]
    pages = [(L + 127) // 128 for L in seq_lens]
    g = torch.Generator().manual_seed(9)
    n_pool = sum(pages)
    perm = torch.randperm(n_pool, generator=g)
    table = np.zeros((batch, max(pages)), dtype=np.int32)
    off = 0
    for b in range(batch):
        table[b, :pages[b]] = perm[off:off + pages[b]].numpy()
        off += pages[b]
    pool = torch.empty((n_pool, hkv, 2, 128, d), dtype=torch.float16, device="cuda")
    picks = [(int(np.argmax(seq_lens)), 7), (int(np.argmin(seq_lens)), 0), (17, 3)]
    seqs = {}
    for b in range(batch):
        L = seq_lens[b]
        k, v = synth.outlier_kv(pages[b] * 128, hkv, d, seed=1000 + b, device="cuda")
        kk = k.view(pages[b], 128, hkv, d).permute(0, 2, 1, 3)
        vv = v.view(pages[b], 128, hkv, d).permute(0, 2, 1, 3)
        idx = torch.from_numpy(table[b, :pages[b]].astype(np.int64)).cuda()
        pool[idx, :, 0] = kk
        pool[idx, :, 1] = vv
        if any(pb == b for pb, _ in picks):
            seqs[b] = (k[:L].cpu(), v[:L].cpu())
    q = shape["q"]
    scale = 1.0 / math.sqrt(d)
    out = torch.empty((batch, hkv * group, d), dtype=torch.float16, device="cuda")
    ws = kv.alloc_fp16_workspace(d, batch, hkv * group, table.shape[1])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.fp16_decode_attention(hkv, q.cuda(), pool, torch.from_numpy(table).cuda(),
                             torch.tensor(seq_lens, dtype=torch.int32, device="cuda"), out, ws,
                             softmax_scale=scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().double().numpy()
    assert np.all(np.isfinite(got))
    for b, h in picks:
        k, v = seqs[b]
        ref = ko.fp16_decode_sequence(q[b, h * group:(h + 1) * group].double().numpy(),
                                      k[:, h].double().numpy(), v[:, h].double().numpy(), scale)
        err = H.assert_decode_close(got[b, h * group:(h + 1) * group], ref, "fp16 full b=%d h=%d" % (b, h))
        print("fp16 full size b=%d (L=%d) h=%d: max scaled err %.2e" % (b, seq_lens[b], h, err))


def test_fp16_decode_status_flags(kv):
    hkv, group, d = 1, 4, 128
    seqs, table, pool, q = _build(hkv, group, d, [200], seed=5)
    bad = table.copy()
    bad[0, 1] = pool.shape[0] + 7  # page id outside the pool
    _, st = _run(kv, hkv, q, pool, bad, [200], 0.1)
    assert st & kv.DEV_BAD_PAGE_ID
    _, st = _run(kv, hkv, q, pool, table, [3 * 128], 0.1)  # more pages than the table holds
    assert st & kv.DEV_SEQ_TOO_LONG
