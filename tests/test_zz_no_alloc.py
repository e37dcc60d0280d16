"""The allocation-free decode entry point against the regular one (GPU).

kvarn_decode_attention_noalloc serves callers that cannot allocate a device workspace (for
example engine plugins whose device memory is planned and owned by the engine): it keeps the
decode's split partials in a fixed buffer inside the library.  Its output must match
kvarn_decode_attention's on the same inputs, call after call, although every call reuses the
buffer the previous call left behind.  This file is collected last on purpose.
"""

import math

import numpy as np
import pytest
import torch

from calibration_free_kv_gb300 import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kv():
    from calibration_free_kv_gb300 import build
    build.build()
    from calibration_free_kv_gb300 import kvarn
    return kvarn


def _case(kv, seed, seq_lens, hkv=2, group=4, d0=128):
    """A GPU-quantised paged cache with raw partial tiles, a permuted block table and q."""
    g = torch.Generator().manual_seed(seed)
    batch = len(seq_lens)
    pages = [L // 128 for L in seq_lens]
    width = max(max(pages), 1)
    n_pool = sum(pages) + 2
    perm = torch.randperm(n_pool, generator=g)
    table = torch.zeros((batch, width), dtype=torch.int32)
    desc = kv.desc_from_preset(d0, hkv)
    pool = kv.alloc_pool(desc, n_pool)
    pk = torch.zeros((batch, hkv, 128, d0), dtype=torch.float16, device="cuda")
    pv = torch.zeros_like(pk)
    off = 0
    for b, L in enumerate(seq_lens):
        table[b, :pages[b]] = perm[off:off + pages[b]].to(torch.int32)
        off += pages[b]
        k, v = synth.outlier_kv(max(L, 1), hkv, d0, seed=seed * 100 + b, device="cuda")
        n = pages[b]
        if n:
            kv.quantize_tiles(desc, k[:128 * n].contiguous(), v[:128 * n].contiguous(),
                              table[b, :n].cuda(), pool)
        rem = L - 128 * n
        if rem:
            pk[b, :, :rem] = k[128 * n:L].transpose(0, 1)
            pv[b, :, :rem] = v[128 * n:L].transpose(0, 1)
    q = torch.randn((batch, hkv * group, d0), generator=g).half().cuda()
    lens = torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    return desc, pool, table.cuda(), lens, q, pk, pv


def _both(kv, case):
    desc, pool, table, lens, q, pk, pv = case
    scale = 1.0 / math.sqrt(q.shape[-1])
    ref = torch.empty_like(q)
    ws = kv.alloc_workspace(desc, q.shape[0], q.shape[1], table.shape[1])
    kv.decode_attention(desc, q, pool, table, lens, ref, ws, partial_k=pk, partial_v=pv,
                        softmax_scale=scale)
    got = torch.full_like(q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.decode_attention_noalloc(desc, q, pool, table, lens, got, partial_k=pk, partial_v=pv,
                                softmax_scale=scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return got.double().cpu().numpy(), ref.double().cpu().numpy()


def test_noalloc_matches_workspace_entry_point(kv):
    # two different shapes back to back, then the first again: each call must not depend on
    # what the previous call left in the shared buffer
    cases = [_case(kv, 1, [0, 130, 1000, 2048 + 77, 300]),
             _case(kv, 2, [4096, 5, 128], group=8)]
    for call, idx in enumerate((0, 1, 0)):
        got, ref = _both(kv, cases[idx])
        # the same kernels on the same inputs in the same order: bit-identical outputs (a stale
        # partial left by the previous call would show here even inside the decode tolerance)
        assert np.array_equal(got, ref), "no-alloc call %d differs from the workspace call" % call
        H.assert_decode_close(got, ref, "no-alloc call %d" % call)
        assert np.all(np.isfinite(got))


def test_noalloc_rejects_shapes_beyond_its_buffer(kv):
    # 512 sequences x 64 query heads x 1024 pages need far more partials than the buffer
    # holds; the call must refuse before launching anything
    desc = kv.desc_from_preset(128, 8)
    need = kv.decode_workspace_bytes(desc, 512, 64, 1024)
    assert need > kv.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((512, 64, 128), dtype=torch.float16, device="cuda")
    out = torch.zeros_like(q)
    pool = kv.alloc_pool(desc, 1)
    table = torch.zeros((512, 1024), dtype=torch.int32, device="cuda")
    lens = torch.zeros(512, dtype=torch.int32, device="cuda")
    with pytest.raises(kv.KvarnError) as err:
        kv.decode_attention_noalloc(desc, q, pool, table, lens, out)
    assert err.value.status == kv.KVARN_ERR_WORKSPACE_TOO_SMALL
