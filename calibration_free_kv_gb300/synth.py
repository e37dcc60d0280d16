"""Seeded synthetic inputs shaped like the KVarN workloads.

This module holds only random-number recipes: none of the method's arithmetic.
It serves the CUDA path, the tests and the CPU oracle alike, so both sides of
every parity check see the same fp16 tensors.

Recipe (a stand-in for real K/V activations, which are not available here):
values N(0,1); a few outlier channels per KV head multiplied by x20..x50;
every (token, head) row multiplied by exp(N(0,1)) (token-scale outliers);
clamped to +-60000 and cast to fp16.  K and V are drawn independently.
"""

from __future__ import annotations

import math

import torch

FP16_CLAMP = 60000.0


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def outlier_tensor(num_tokens: int, num_kv_heads: int, head_dim: int, *, gen: torch.Generator,
                   device, outlier_channels=None, outlier_scale=None, n_outliers: int = 4,
                   scale_lo: float = 20.0, scale_hi: float = 50.0) -> torch.Tensor:
    """One fp16 tensor [num_tokens, num_kv_heads, head_dim] from the outlier recipe.

    outlier_channels: fixed channel list used for every head (with outlier_scale),
    or None for n_outliers random channels per head with scales U[scale_lo, scale_hi].
    """
    x = torch.randn((num_tokens, num_kv_heads, head_dim), generator=gen, device=device,
                    dtype=torch.float32)
    chan = torch.ones((num_kv_heads, head_dim), device=device, dtype=torch.float32)
    if outlier_channels is not None:
        for c in outlier_channels:
            chan[:, c] = float(outlier_scale)
    else:
        for h in range(num_kv_heads):
            idx = torch.randperm(head_dim, generator=gen, device=device)[:n_outliers]
            sc = scale_lo + (scale_hi - scale_lo) * torch.rand(
                (n_outliers,), generator=gen, device=device)
            chan[h, idx] = sc
    tok = torch.exp(torch.randn((num_tokens, num_kv_heads, 1), generator=gen, device=device))
    x = x * chan.unsqueeze(0) * tok
    return x.clamp_(-FP16_CLAMP, FP16_CLAMP).to(torch.float16)


def outlier_kv(num_tokens: int, num_kv_heads: int, head_dim: int, seed: int, device="cpu",
               **kw):
    """(K, V) fp16 tensors [num_tokens, num_kv_heads, head_dim], drawn independently."""
    g = _gen(seed, device)
    k = outlier_tensor(num_tokens, num_kv_heads, head_dim, gen=g, device=device, **kw)
    v = outlier_tensor(num_tokens, num_kv_heads, head_dim, gen=g, device=device, **kw)
    return k, v


def tiny_case(device="cpu"):
    """1 KV head, head_dim 128, one 128-token K and V tile, seed 0; channels 3 and 77 x50;
    a single query N(0,1)/sqrt(128).  Returns (k [128,1,128], v, q [1,1,128])."""
    g = _gen(0, device)
    k = outlier_tensor(128, 1, 128, gen=g, device=device, outlier_channels=(3, 77),
                       outlier_scale=50.0)
    v = outlier_tensor(128, 1, 128, gen=g, device=device, outlier_channels=(3, 77),
                       outlier_scale=50.0)
    q = (torch.randn((1, 1, 128), generator=g, device=device) / math.sqrt(128.0)).to(torch.float16)
    return k, v, q


def decode_batch(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, seed: int,
                 min_pages: int, max_pages: int, device="cpu", pool_pages: int | None = None,
                 seq_lens=None):
    """Shapes of one paged decode step.

    seq_len_b = 128 * U{min_pages..max_pages} unless seq_lens is given; the block
    table maps each sequence's logical pages to a random permutation of the pool.
    Returns dict(seq_lens int32 [B], block_table int32 [B, max_pages_per_seq],
    q fp16 [B, Hq, d0] ~ N(0,1), pool_pages).
    """
    g = _gen(seed, "cpu")
    if seq_lens is None:
        pages = torch.randint(min_pages, max_pages + 1, (batch,), generator=g)
        seq_lens = pages * 128
    seq_lens = torch.as_tensor(seq_lens, dtype=torch.int64)
    pages_per_seq = (seq_lens + 127) // 128
    total = int(pages_per_seq.sum())
    n_pool = total if pool_pages is None else int(pool_pages)
    perm = torch.randperm(n_pool, generator=g)[:total]
    width = max(int(pages_per_seq.max()), 1)
    table = torch.zeros((batch, width), dtype=torch.int32)
    off = 0
    for b in range(batch):
        n = int(pages_per_seq[b])
        table[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    q = torch.randn((batch, num_q_heads, head_dim), generator=g).to(torch.float16)
    return {"seq_lens": seq_lens.to(torch.int32).to(device), "block_table": table.to(device),
            "q": q.to(device), "pool_pages": n_pool}


def partial_phases(batch: int, seed: int) -> torch.Tensor:
    """Raw tokens already in each sequence's unsealed tile, U{0..127} (int64 [batch], CPU):
    a decode loop meets its sequences at random points of their current 128-token tile."""
    g = _gen(seed, "cpu")
    return torch.randint(0, 128, (batch,), generator=g)
