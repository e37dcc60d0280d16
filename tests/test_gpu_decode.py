"""GPU paged decode attention against the float64 oracle (through the C ABI).

The packed cache fed to the GPU decode is built by the ORACLE (its own quantisation of
the same fp16 inputs, uploaded into the page pool), so every expected value comes from
the CPU side; a second set of tests decodes GPU-quantised records and compares with the
oracle's attention over those same bytes.
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


def _build_case(batch, hkv, group, d0, seq_lens, seed, pool_extra=3):
    """Synthetic cache: per sequence fp16 K/V [L, Hkv, d0], random block table, q."""
    g = torch.Generator().manual_seed(seed)
    seq_lens = [int(x) for x in seq_lens]
    pages = [L // 128 for L in seq_lens]
    n_pool = sum(pages) + pool_extra
    perm = torch.randperm(n_pool, generator=g).tolist()
    width = max(max(pages), 1)
    table = np.zeros((batch, width), dtype=np.int32)
    seqs = []
    off = 0
    for b, L in enumerate(seq_lens):
        k, v = synth.outlier_kv(max(L, 1), hkv, d0, seed=seed * 1000 + b)
        seqs.append((k[:L], v[:L]))
        table[b, :pages[b]] = perm[off:off + pages[b]]
        off += pages[b]
    q = torch.randn((batch, hkv * group, d0), generator=g).half()
    return seqs, table, n_pool, q


def _oracle_records(seqs, hkv, d0):
    """(b, page index, head) -> record bytes, quantised by the oracle."""
    recs = {}
    for b, (k, v) in enumerate(seqs):
        n = k.shape[0] // 128
        if n == 0:
            continue
        kk = k[:128 * n].double().numpy().reshape(n, 128, hkv, d0)
        vv = v[:128 * n].double().numpy().reshape(n, 128, hkv, d0)
        for h in range(hkv):
            r, _, _ = H.oracle_quantize(kk[:, :, h], vv[:, :, h])
            for i in range(n):
                recs[(b, i, h)] = r[i]
    return recs


def _partials(seqs, hkv, d0):
    batch = len(seqs)
    pk = torch.zeros((batch, hkv, 128, d0), dtype=torch.float16)
    pv = torch.zeros_like(pk)
    for b, (k, v) in enumerate(seqs):
        n = k.shape[0] % 128
        if n:
            pk[b, :, :n] = k[k.shape[0] - n:].transpose(0, 1)
            pv[b, :, :n] = v[v.shape[0] - n:].transpose(0, 1)
    return pk, pv


def _oracle_decode(recs, seqs, q, hkv, group, d0, scale, only=None):
    out = np.zeros(q.shape, dtype=np.float64)
    for b, (k, v) in enumerate(seqs):
        n = k.shape[0] // 128
        rem = k.shape[0] % 128
        for h in range(hkv):
            if only is not None and (b, h) not in only:
                continue
            rl = [recs[(b, i, h)] for i in range(n)]
            pk = k[128 * n:, h].double().numpy() if rem else None
            pv = v[128 * n:, h].double().numpy() if rem else None
            out[b, h * group:(h + 1) * group] = ko.decode_sequence(
                q[b, h * group:(h + 1) * group].double().numpy(), rl, pk, pv, scale, d0)
    return out


def _gpu_decode(kv, desc, pool, table, seq_lens, q, pk, pv, scale):
    batch, hq, d0 = q.shape
    out = torch.empty((batch, hq, d0), dtype=torch.float16, device="cuda")
    ws = kv.alloc_workspace(desc, batch, hq, table.shape[1])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.decode_attention(desc, q.cuda(), pool, torch.from_numpy(table).cuda(),
                        torch.tensor(seq_lens, dtype=torch.int32, device="cuda"), out, ws,
                        partial_k=pk.cuda() if pk is not None else None,
                        partial_v=pv.cuda() if pv is not None else None,
                        softmax_scale=scale, status=status)
    torch.cuda.synchronize()
    return out.cpu().double().numpy(), int(status.item())


def _run_oracle_cache_case(kv, batch, hkv, group, d0, seq_lens, seed):
    seqs, table, n_pool, q = _build_case(batch, hkv, group, d0, seq_lens, seed)
    desc = kv.desc_from_preset(d0, hkv)
    recs = _oracle_records(seqs, hkv, d0)
    pool = kv.alloc_pool(desc, n_pool)
    H.upload_records(pool, [(int(table[b, i]), h, r) for (b, i, h), r in recs.items()])
    pk, pv = _partials(seqs, hkv, d0)
    scale = H.softmax_scale(d0)
    got, st = _gpu_decode(kv, desc, pool, table, seq_lens, q, pk, pv, scale)
    assert st == 0
    ref = _oracle_decode(recs, seqs, q, hkv, group, d0, scale)
    return H.assert_decode_close(got, ref, "decode d0=%d G=%d" % (d0, group))


def test_tiny_decode(kv):
    # 1 KV head, d 128, one sealed tile, a single query N(0,1)/sqrt(128)
    k, v, q = synth.tiny_case()
    desc = kv.desc_from_preset(128, 1)
    rec, _, _ = ko.quantize_page(k[:, 0].double().numpy(), v[:, 0].double().numpy())
    pool = kv.alloc_pool(desc, 1)
    H.upload_records(pool, [(0, 0, rec)])
    table = np.zeros((1, 1), dtype=np.int32)
    got, st = _gpu_decode(kv, desc, pool, table, [128], q, None, None, 1 / math.sqrt(128))
    assert st == 0
    ref = ko.decode_sequence(q[0].double().numpy(), [rec], None, None, 1 / math.sqrt(128), 128)
    err = H.assert_decode_close(got[0], ref, "tiny")
    full = ko.softmax_attention(q[0, 0].double().numpy(), k[:, 0].double().numpy(),
                                v[:, 0].double().numpy(), 1 / math.sqrt(128))
    cos = float(got[0, 0] @ full / np.linalg.norm(got[0, 0]) / np.linalg.norm(full))
    print("tiny decode: scaled err %.2e, cosine vs fp16 attention %.4f" % (err, cos))


@pytest.mark.parametrize("d0,group", [(128, 4), (128, 1), (128, 2), (128, 8), (96, 4), (256, 4),
                                      (64, 8), (256, 1), (96, 8)])
def test_decode_parity_ragged(kv, d0, group):
    # lengths: empty, sub-tile, exactly one tile, tile + tail, several tiles with tails,
    # more pages than one split (16 pages) holds
    seq_lens = [0, 1, 127, 128, 129, 300, 17 * 128 + 5, 2048]
    err = _run_oracle_cache_case(kv, len(seq_lens), 2, group, d0, seq_lens, seed=d0 + group)
    print("d0=%d G=%d max scaled err %.2e" % (d0, group, err))


@pytest.mark.parametrize("group,kernel,tiles", [(8, "tc", "merge"), (8, "persistent", "merge"),
                                                (8, "split", "merge"), (4, "persistent", "merge"),
                                                (4, "split", "merge"), (2, "persistent", "merge"),
                                                (4, "persistent", "split"), (4, "split", "split"),
                                                (8, "tc", "split"), (1, "persistent", "merge")])
def test_decode_partition(kv, group, kernel, tiles, monkeypatch):
    # The persistent kernels (mma.sync "persistent", tcgen05 "tc") cut a line of virtual pages
    # (each row with sealed pages: 8 units for a segment's fixed work, then one per page) into
    # equal ranges of at least 32 units: here 316 pages of 16 rows, 444 units over 13 ranges, so
    # rows split across CTAs (up to three segments), some rows have no sealed page, and raw
    # partial tiles follow; "split" runs one CTA per split.  The raw partial tiles are attended
    # by the merge kernel ("merge") or by the decode kernels as splits of their own ("split").
    monkeypatch.setenv("KVARN_DECODE_KERNEL", kernel)
    monkeypatch.setenv("KVARN_DECODE_OPEN_TILES", tiles)
    seq_lens = [0, 5 * 128, 129, 40 * 128 + 17, 128, 64 * 128, 3, 33 * 128, 1000, 7 * 128 + 127]
    err = _run_oracle_cache_case(kv, len(seq_lens), 2, group, 128, seq_lens, seed=808)
    print("G=%d partition (%s, open tiles: %s) max scaled err %.2e" % (group, kernel, tiles, err))


@pytest.mark.parametrize("group,kernel", [(4, "persistent"), (8, "persistent"), (8, "tc"), (1, "persistent")])
def test_decode_partition_short_rows(kv, group, kernel, monkeypatch):
    # 48 sequences of 0-3 sealed pages plus raw tails, 2 kv heads: 72 rows with pages, 720
    # virtual units over 22 ranges, so most ranges hold several rows, 14 of the 21 range ends
    # fall inside a row's fixed units (the next CTA starts at that row's first page) and rows of
    # two or three pages split across two CTAs
    monkeypatch.setenv("KVARN_DECODE_KERNEL", kernel)
    seq_lens = [128 * ((i * 7) % 4) + (i * 37) % 128 for i in range(48)]
    err = _run_oracle_cache_case(kv, len(seq_lens), 2, group, 128, seq_lens, seed=909)
    print("G=%d short rows (%s) max scaled err %.2e" % (group, kernel, err))


def test_decode_gpu_quantised_cache(kv):
    # the composed path: GPU-quantised records, decoded on the GPU, against the oracle's
    # attention over the very same bytes
    hkv, group, d0 = 2, 4, 128
    seq_lens = [256, 640, 1000]
    seqs, table, n_pool, q = _build_case(3, hkv, group, d0, seq_lens, seed=77)
    desc = kv.desc_from_preset(d0, hkv)
    pool = kv.alloc_pool(desc, n_pool)
    for b, (k, v) in enumerate(seqs):
        n = k.shape[0] // 128
        ids = torch.from_numpy(table[b, :n].copy()).cuda()
        kv.quantize_tiles(desc, k[:128 * n].cuda(), v[:128 * n].cuda(), ids, pool)
    torch.cuda.synchronize()
    recs = {}
    for b, (k, _) in enumerate(seqs):
        for i in range(k.shape[0] // 128):
            for h in range(hkv):
                recs[(b, i, h)] = H.record_bytes_of(pool, int(table[b, i]), h)
    pk, pv = _partials(seqs, hkv, d0)
    scale = H.softmax_scale(d0)
    got, st = _gpu_decode(kv, desc, pool, table, seq_lens, q, pk, pv, scale)
    assert st == 0
    ref = _oracle_decode(recs, seqs, q, hkv, group, d0, scale)
    H.assert_decode_close(got, ref, "gpu-quantised cache")


def test_decode_page_placement_invariance(kv):
    # the same sequence stored at different pool pages decodes to identical bits
    hkv, group, d0 = 1, 4, 128
    k, v = synth.outlier_kv(640, hkv, d0, seed=5, device="cuda")
    desc = kv.desc_from_preset(d0, hkv)
    pool = kv.alloc_pool(desc, 12)
    kv.quantize_tiles(desc, k, v, torch.tensor([0, 1, 2, 3, 4], dtype=torch.int32, device="cuda"), pool)
    kv.quantize_tiles(desc, k, v, torch.tensor([11, 7, 9, 5, 6], dtype=torch.int32, device="cuda"), pool)
    table = np.array([[0, 1, 2, 3, 4], [11, 7, 9, 5, 6]], dtype=np.int32)
    q = torch.randn((1, 4, d0), generator=torch.Generator().manual_seed(3)).half().repeat(2, 1, 1)
    got, st = _gpu_decode(kv, desc, pool, table, [640, 640], q, None, None, 0.088)
    assert st == 0
    assert np.array_equal(got[0], got[1])


def test_decode_status_flags(kv):
    hkv, d0 = 1, 128
    desc = kv.desc_from_preset(d0, hkv)
    pool = kv.alloc_pool(desc, 2)
    table = np.array([[0, 5]], dtype=np.int32)        # page 5 is outside the 2-page pool
    q = torch.ones((1, 4, d0), dtype=torch.float16)
    out, st = _gpu_decode(kv, desc, pool, table, [256], q, None, None, 0.1)
    assert st & kv.DEV_BAD_PAGE_ID
    assert np.all(np.isfinite(out))
    out, st = _gpu_decode(kv, desc, pool, np.array([[0, 1]], dtype=np.int32), [2 * 128 + 128], q,
                          None, None, 0.1)
    assert st & kv.DEV_SEQ_TOO_LONG
    out, st = _gpu_decode(kv, desc, pool, np.array([[0, 1]], dtype=np.int32), [130], q, None, None, 0.1)
    assert st & kv.DEV_NO_PARTIAL


def test_decode_empty_sequences_are_zero(kv):
    desc = kv.desc_from_preset(128, 2)
    pool = kv.alloc_pool(desc, 1)
    q = torch.randn((3, 8, 128), generator=torch.Generator().manual_seed(1)).half()
    out, st = _gpu_decode(kv, desc, pool, np.zeros((3, 1), dtype=np.int32), [0, 0, 0], q, None, None, 0.1)
    assert st == 0 and np.all(out == 0.0)


def test_decode_full_size_sampled(kv):
    # batch 64, seq_len = 128 * U{8..128}, 32 query heads over 8 KV heads, head_dim 128,
    # permuted block table: the decode workload at full size.  The GPU quantises the whole
    # cache; three sampled (sequence, kv head) caches are replaced by oracle records and
    # their outputs compared.
    hkv, group, d0, batch = 8, 4, 128, 64
    shape = synth.decode_batch(batch, hkv * group, hkv, d0, seed=3, min_pages=8, max_pages=128)
    seq_lens = shape["seq_lens"].tolist()
    table = shape["block_table"].numpy()
    n_pool = shape["pool_pages"]
    desc = kv.desc_from_preset(d0, hkv)
    pool = kv.alloc_pool(desc, n_pool)
    total = sum(seq_lens)
    k_all, v_all = synth.outlier_kv(total, hkv, d0, seed=3, device="cuda")
    page_ids = torch.from_numpy(np.concatenate([table[b, :L // 128] for b, L in enumerate(seq_lens)])).cuda()
    kv.quantize_tiles(desc, k_all, v_all, page_ids, pool)
    torch.cuda.synchronize()
    longest = int(np.argmax(seq_lens))
    shortest = int(np.argmin(seq_lens))
    picks = [(longest, 7), (shortest, 0), (17, 3)]
    offs = np.concatenate([[0], np.cumsum(seq_lens)])
    recs = {}
    for b, h in picks:
        L = seq_lens[b]
        kk = k_all[offs[b]:offs[b] + L, h].cpu().double().numpy().reshape(L // 128, 128, d0)
        vv = v_all[offs[b]:offs[b] + L, h].cpu().double().numpy().reshape(L // 128, 128, d0)
        r, _, _ = H.oracle_quantize(kk, vv)
        for i in range(L // 128):
            recs[(b, i, h)] = r[i]
    H.upload_records(pool, [(int(table[b, i]), h, r) for (b, i, h), r in recs.items()])
    q = shape["q"]
    scale = 1.0 / math.sqrt(128.0)
    got, st = _gpu_decode(kv, desc, pool, table, seq_lens, q, None, None, scale)
    assert st == 0
    assert np.all(np.isfinite(got))
    for b, h in picks:
        L = seq_lens[b]
        rl = [recs[(b, i, h)] for i in range(L // 128)]
        ref = ko.decode_sequence(q[b, h * group:(h + 1) * group].double().numpy(), rl, None, None, scale, d0)
        err = H.assert_decode_close(got[b, h * group:(h + 1) * group], ref, "full size b=%d h=%d" % (b, h))
        print("full size b=%d (L=%d) h=%d: max scaled err %.2e" % (b, L, h, err))


@pytest.mark.parametrize("kernel", ["default", "tc", "split"])
def test_decode_32b_layer_sampled(kv, kernel, monkeypatch):
    # one layer of the 32B-class decode step: batch 32 at 16384 tokens, 64 query heads over
    # 8 KV heads (GQA 8), head_dim 128, permuted block table, GPU-quantised cache; three
    # sampled (sequence, kv head) caches are replaced by oracle records and compared; on the
    # default kernel (persistent mma.sync), the tcgen05 kernel and the one-CTA-per-split form
    if kernel == "default":
        monkeypatch.delenv("KVARN_DECODE_KERNEL", raising=False)
    else:
        monkeypatch.setenv("KVARN_DECODE_KERNEL", kernel)
    hkv, group, d0, batch, L = 8, 8, 128, 32, 16384
    pages = L // 128
    g = torch.Generator().manual_seed(4)
    table = torch.randperm(batch * pages, generator=g).view(batch, pages).to(torch.int32)
    desc = kv.desc_from_preset(d0, hkv)
    pool = kv.alloc_pool(desc, batch * pages)
    k_all, v_all = synth.outlier_kv(batch * L, hkv, d0, seed=4, device="cuda")
    kv.quantize_tiles(desc, k_all, v_all, table.reshape(-1).cuda(), pool)
    torch.cuda.synchronize()
    picks = [(0, 0), (31, 7), (13, 4)]
    recs = {}
    for b, h in picks:
        kk = k_all[b * L:(b + 1) * L, h].cpu().double().numpy().reshape(pages, 128, d0)
        vv = v_all[b * L:(b + 1) * L, h].cpu().double().numpy().reshape(pages, 128, d0)
        r, _, _ = H.oracle_quantize(kk, vv)
        for i in range(pages):
            recs[(b, i, h)] = r[i]
    del k_all, v_all
    H.upload_records(pool, [(int(table[b, i]), h, r) for (b, i, h), r in recs.items()])
    q = torch.randn((batch, hkv * group, d0), generator=g).half()
    scale = 1.0 / math.sqrt(128.0)
    got, st = _gpu_decode(kv, desc, pool, table.numpy(), [L] * batch, q, None, None, scale)
    assert st == 0
    assert np.all(np.isfinite(got))
    for b, h in picks:
        rl = [recs[(b, i, h)] for i in range(pages)]
        ref = ko.decode_sequence(q[b, h * group:(h + 1) * group].double().numpy(), rl, None, None, scale, d0)
        err = H.assert_decode_close(got[b, h * group:(h + 1) * group], ref, "32B layer b=%d h=%d" % (b, h))
        print("32B layer b=%d h=%d: max scaled err %.2e" % (b, h, err))


def test_decode_longest_block_table(kv):
    # 1024-page block tables (131072 tokens): one sequence with a 77-token partial tile, one
    # exactly full; 32 splits plus the partial tile reach the combine step
    err = _run_oracle_cache_case(kv, 2, 1, 4, 128, [1024 * 128 + 77, 1024 * 128], seed=11)
    print("1024 pages: max scaled err %.2e" % err)


def test_bounded_wait_times_out_and_the_context_stays_usable(kv):
    # a wait on an mbarrier that nothing completes gives up (~2 s) with a status bit; a decode
    # launched afterwards on the same context still runs and matches the oracle
    import time
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    kv.selftest_wait_timeout(status)
    torch.cuda.synchronize()
    waited = time.time() - t0
    assert int(status.item()) == kv.DEV_WAIT_TIMEOUT
    assert 0.5 < waited < 30.0
    err = _run_oracle_cache_case(kv, 2, 1, 4, 128, [300, 129], seed=21)
    print("wait gave up after %.2f s; decode afterwards: max scaled err %.2e" % (waited, err))


@pytest.mark.parametrize("group,kernel", [(4, "split"), (4, "persistent"), (8, "persistent"), (8, "split"),
                                          (8, "tc")])
def test_two_phase_decode_matches_one_call(kv, group, kernel, monkeypatch):
    # kvarn_decode_partials then kvarn_decode_combine give the bytes of kvarn_decode_attention
    monkeypatch.setenv("KVARN_DECODE_KERNEL", kernel)
    hkv, d0 = 2, 128
    lens = [0, 5, 128, 700, 4096 + 77]
    seqs, table, n_pool, q = _build_case(len(lens), hkv, group, d0, lens, seed=77)
    desc = kv.desc_from_preset(d0, hkv)
    pool = kv.alloc_pool(desc, n_pool)
    for b, (k, v) in enumerate(seqs):
        n = k.shape[0] // 128
        if n:
            kv.quantize_tiles(desc, k[:128 * n].cuda(), v[:128 * n].cuda(),
                              torch.from_numpy(table[b, :n].copy()).cuda(), pool)
    pk, pv = (t.cuda() for t in _partials(seqs, hkv, d0))
    qd, tb = q.cuda(), torch.from_numpy(table).cuda()
    ln = torch.tensor(lens, dtype=torch.int32, device="cuda")
    ws = kv.alloc_workspace(desc, len(lens), q.shape[1], table.shape[1])
    one = torch.empty_like(qd)
    kv.decode_attention(desc, qd, pool, tb, ln, one, ws, partial_k=pk, partial_v=pv)
    two = torch.full_like(qd, float("nan"))
    for phase in ("partials", "combine"):
        kv.decode_attention(desc, qd, pool, tb, ln, two, ws, partial_k=pk, partial_v=pv, phase=phase)
    torch.cuda.synchronize()
    assert torch.equal(one, two)
