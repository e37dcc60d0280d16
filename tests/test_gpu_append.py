"""Streaming append / seal on the GPU: sealed pages against batch quantisation and the oracle,
and decode over sealed pages plus the raw fp16 partial tile."""

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


class Stream:
    """A batch of sequences grown one token per step through kvarn_append_token."""

    def __init__(self, kv, batch, hkv, d0, l0, max_pages, seed, group=4):
        self.kv, self.batch, self.hkv, self.d0, self.group = kv, batch, hkv, d0, group
        self.desc = kv.desc_from_preset(d0, hkv)
        g = torch.Generator().manual_seed(seed)
        self.gen = g
        n_pool = batch * max_pages + 2
        perm = torch.randperm(n_pool, generator=g)[:batch * max_pages]
        self.table = perm.view(batch, max_pages).to(torch.int32)
        self.table_d = self.table.cuda()
        self.pool = kv.alloc_pool(self.desc, n_pool)
        self.pk = torch.zeros((batch, hkv, 128, d0), dtype=torch.float16, device="cuda")
        self.pv = torch.zeros_like(self.pk)
        self.init = []            # per sequence: initial (k, v) [L0, Hkv, d0] fp16 on the GPU
        self.appended = [[] for _ in range(batch)]   # per sequence: appended (k, v) [Hkv, d0] CPU
        for b, L in enumerate(l0):
            k, v = synth.outlier_kv(max(L, 1), hkv, d0, seed=seed * 100 + b, device="cuda")
            k, v = k[:L], v[:L]
            n = L // 128
            if n:
                kv.quantize_tiles(self.desc, k[:128 * n].contiguous(), v[:128 * n].contiguous(),
                                  self.table_d[b, :n].contiguous(), self.pool)
            rem = L - 128 * n
            if rem:
                self.pk[b, :, :rem] = k[128 * n:].transpose(0, 1)
                self.pv[b, :, :rem] = v[128 * n:].transpose(0, 1)
            self.init.append((k, v))
        self.lens = [torch.tensor(l0, dtype=torch.int32, device="cuda"),
                     torch.zeros(batch, dtype=torch.int32, device="cuda")]
        self.cur = 0
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step(self):
        kn = (torch.randn((self.batch, self.hkv, self.d0), generator=self.gen) * 2).half()
        vn = torch.randn((self.batch, self.hkv, self.d0), generator=self.gen).half()
        self.kv.append_token(self.desc, kn.cuda(), vn.cuda(), self.pk, self.pv, self.lens[self.cur],
                             self.table_d, self.pool, seq_lens_out=self.lens[1 - self.cur],
                             status=self.status)
        self.cur = 1 - self.cur
        for b in range(self.batch):
            self.appended[b].append((kn[b], vn[b]))

    def tokens(self, b, lo, hi):
        """fp16 CPU (k, v) [hi - lo, Hkv, d0] of sequence b's tokens lo..hi-1."""
        k0, v0 = self.init[b]
        l0 = k0.shape[0]
        ks, vs = [], []
        if lo < l0:
            ks.append(k0[lo:min(hi, l0)].cpu())
            vs.append(v0[lo:min(hi, l0)].cpu())
        for t in range(max(lo, l0), hi):
            ks.append(self.appended[b][t - l0][0][None])
            vs.append(self.appended[b][t - l0][1][None])
        if not ks:
            return (torch.zeros((0, self.hkv, self.d0), dtype=torch.float16),) * 2
        return torch.cat(ks), torch.cat(vs)

    def seq_lens(self):
        return [int(x) for x in self.lens[self.cur].cpu()]

    def decode(self, q):
        out = torch.empty((self.batch, self.hkv * self.group, self.d0), dtype=torch.float16, device="cuda")
        ws = self.kv.alloc_workspace(self.desc, self.batch, self.hkv * self.group, self.table.shape[1])
        self.kv.decode_attention(self.desc, q.cuda(), self.pool, self.table_d, self.lens[self.cur], out, ws,
                                 partial_k=self.pk, partial_v=self.pv,
                                 softmax_scale=1 / math.sqrt(self.d0), status=self.status)
        torch.cuda.synchronize()
        return out.cpu().double().numpy()


def _check_sealed_pages(st, pages_per_seq=None):
    """Every sealed page == GPU batch quantisation of its 128 tokens (bit-exact) and == the
    oracle (codes with the boundary exemption, metadata within one fp16 ulp)."""
    kv, desc = st.kv, st.desc
    stats = []
    for b, L in enumerate(st.seq_lens()):
        n = L // 128
        pages = range(n) if pages_per_seq is None else [i for i in pages_per_seq if i < n]
        for i in pages:
            k, v = st.tokens(b, 128 * i, 128 * i + 128)
            pool2 = kv.alloc_pool(desc, 1)
            kv.quantize_tiles(desc, k.cuda().contiguous(), v.cuda().contiguous(),
                              torch.zeros(1, dtype=torch.int32, device="cuda"), pool2)
            torch.cuda.synchronize()
            page = int(st.table[b, i])
            assert torch.equal(st.pool[page], pool2[0]), "sealed page differs from batch quantisation"
            kt = k.double().numpy().transpose(1, 0, 2)
            vt = v.double().numpy().transpose(1, 0, 2)
            _, kq, vq = H.oracle_quantize(kt, vt)
            for h in range(st.hkv):
                H.compare_record(H.record_bytes_of(st.pool, page, h), H.tile_of(kq, h),
                                 H.tile_of(vq, h), desc.head_dim_padded, stats)
    if stats:
        H.assert_mismatch_budget(stats)


def _check_decode(st, q, only=None):
    got = st.decode(q)
    lens = st.seq_lens()
    group, d0 = st.group, st.d0
    for b, L in enumerate(lens):
        n = L // 128
        k, v = st.tokens(b, 128 * n, L)
        for h in range(st.hkv):
            if only is not None and (b, h) not in only:
                continue
            recs = [H.record_bytes_of(st.pool, int(st.table[b, i]), h) for i in range(n)]
            ref = ko.decode_sequence(q[b, h * group:(h + 1) * group].double().numpy(), recs,
                                     k[:, h].double().numpy(), v[:, h].double().numpy(),
                                     1 / math.sqrt(d0), d0)
            H.assert_decode_close(got[b, h * group:(h + 1) * group], ref, "append b=%d h=%d" % (b, h))


@pytest.mark.parametrize("d0", [128, 96, 256])
def test_append_seal_and_decode(kv, d0):
    st = Stream(kv, batch=3, hkv=2, d0=d0, l0=[0, 5, 127], max_pages=4, seed=d0)
    q = torch.randn((3, 8, d0), generator=torch.Generator().manual_seed(9)).half()
    for i in range(300):
        st.step()
        if i in (0, 122, 123):  # just before / after sealing a tile of the second sequence
            _check_decode(st, q)
    assert int(st.status.item()) == 0
    assert st.seq_lens() == [300, 305, 427]
    # partial tile rows hold the raw tail tokens
    for b, L in enumerate(st.seq_lens()):
        rem = L % 128
        k, _ = st.tokens(b, L - rem, L)
        assert torch.equal(st.pk[b, :, :rem].cpu(), k.transpose(0, 1))
    _check_sealed_pages(st)
    _check_decode(st, q)


def test_append_rejects_full_block_table(kv):
    st = Stream(kv, batch=1, hkv=1, d0=128, l0=[256], max_pages=2, seed=3)
    st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) & kv.DEV_SEQ_TOO_LONG


@pytest.mark.parametrize("d0", [256, 96])
def test_long_context_streaming_sampled(kv, d0):
    # batch 4 at 130560 + {0, 1, 64, 127} tokens, head_dim 256 (and 96, zero-padded to 128),
    # 8 KV heads, 32 query heads; 512 appends (every seal of every sequence is checked);
    # sampled heads decoded at the end
    st = Stream(kv, batch=4, hkv=8, d0=d0, l0=[130560, 130561, 130624, 130687], max_pages=1030,
                seed=5)
    q = torch.randn((4, 32, d0), generator=torch.Generator().manual_seed(10)).half()
    for _ in range(512):
        st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    lens = st.seq_lens()
    assert lens == [131072, 131073, 131136, 131199]
    _check_sealed_pages(st, pages_per_seq=[1020, 1021, 1022, 1023, 1024])
    _check_decode(st, q, only={(0, 3), (3, 6)})
