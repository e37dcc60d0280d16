"""ctypes binding of libkvarn.so: argument marshalling only.

Every function forwards torch tensors (device memory) to the C ABI declared in
include/kvarn.h and raises KvarnError on a non-zero status.  All arithmetic runs in
the library's CUDA kernels; there is no CPU or PyTorch fallback.  Importing this module
loads the library and raises if it has not been built (see ``build.build``).
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvarn.so")

KVARN_OK = 0
KVARN_ERR_INVALID_ARG = -1
KVARN_ERR_UNSUPPORTED = -2
KVARN_ERR_WORKSPACE_TOO_SMALL = -3
KVARN_ERR_CUDA = -4
DEV_BAD_PAGE_ID = 1
DEV_SEQ_TOO_LONG = 2
DEV_WAIT_TIMEOUT = 4
DEV_NO_PARTIAL = 8

EXPORTED_SYMBOLS = (
    "kvarn_desc_from_preset",
    "kvarn_page_record_bytes",
    "kvarn_quantize_tiles",
    "kvarn_quantize_tiles_adaptive",
    "kvarn_append_token",
    "kvarn_decode_workspace_bytes",
    "kvarn_decode_attention",
    "kvarn_prefill_workspace_bytes",
    "kvarn_prefill_attention",
    "kvarn_dequantize_tiles",
    "kvarn_status_string",
    "kvarn_decode_attention_noalloc",
    "kvarn_fp16_page_bytes",
    "kvarn_fp16_decode_workspace_bytes",
    "kvarn_fp16_decode_attention",
    "kvarn_selftest_wait_timeout",
    "kvarn_quantization_error",
    "kvarn_decode_partials",
    "kvarn_decode_combine",
)

# Size of the library's fixed decode scratch (KVARN_DECODE_NOALLOC_SCRATCH_BYTES in kvarn.h).
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


class KvarnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (where, status_string(status), status))


class KvarnDesc(ctypes.Structure):
    _fields_ = [
        ("head_dim", ctypes.c_int32),
        ("head_dim_padded", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("tile_tokens", ctypes.c_int32),
        ("k_bits", ctypes.c_int32),
        ("v_bits", ctypes.c_int32),
        ("sinkhorn_iters", ctypes.c_int32),
        ("sinkhorn_eps", ctypes.c_float),
        ("page_record_bytes", ctypes.c_int64),
    ]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError("libkvarn.so is not built (run calibration_free_kv_gb300.build.build() "
                          "or __graft_entry__.build()); there is no fallback path")
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    i32, i64 = ctypes.c_int, ctypes.c_int64
    D = ctypes.POINTER(KvarnDesc)
    sig = {
        "kvarn_desc_from_preset": (i32, [ctypes.c_char_p, i32, i32, D]),
        "kvarn_page_record_bytes": (i64, [D]),
        "kvarn_quantize_tiles": (i32, [D, P, P, i64, i64, i32, P, P, i64, P, P]),
        "kvarn_quantize_tiles_adaptive": (i32, [D, P, P, i64, i64, i32, P, P, i64, ctypes.c_float, P, P, P]),
        "kvarn_append_token": (i32, [D, i32, P, P, P, P, P, P, P, i32, P, i64, P, P]),
        "kvarn_decode_workspace_bytes": (ctypes.c_size_t, [D, i32, i32, i32]),
        "kvarn_decode_attention": (i32, [D, i32, i32, P, P, i64, P, i32, P, P, P, ctypes.c_float,
                                         P, P, ctypes.c_size_t, P, P]),
        "kvarn_dequantize_tiles": (i32, [D, P, i64, P, i32, P, P, P, P]),
        "kvarn_prefill_workspace_bytes": (ctypes.c_size_t, [D, i32, i32, i32, i32]),
        "kvarn_prefill_attention": (i32, [D, i32, i32, i32, P, P, P, P, i64, P, i32, P, P, P,
                                          ctypes.c_float, P, P, ctypes.c_size_t, P, P]),
        "kvarn_status_string": (ctypes.c_char_p, [i32]),
        "kvarn_decode_attention_noalloc": (i32, [D, i32, i32, P, P, i64, P, i32, P, P, P,
                                                 ctypes.c_float, P, P, P]),
        "kvarn_fp16_page_bytes": (ctypes.c_size_t, [i32]),
        "kvarn_fp16_decode_workspace_bytes": (ctypes.c_size_t, [i32, i32, i32, i32]),
        "kvarn_fp16_decode_attention": (i32, [i32, i32, i32, i32, P, P, i64, P, i32, P, ctypes.c_float,
                                              P, P, ctypes.c_size_t, P, P]),
        "kvarn_selftest_wait_timeout": (i32, [P, P]),
        "kvarn_quantization_error": (i32, [D, P, P, i64, i64, i32, P, P, i64, P, P, P]),
        "kvarn_decode_partials": (i32, [D, i32, i32, P, P, i64, P, i32, P, P, P, ctypes.c_float,
                                        P, P, ctypes.c_size_t, P, P]),
        "kvarn_decode_combine": (i32, [D, i32, i32, P, P, i64, P, i32, P, P, P, ctypes.c_float,
                                       P, P, ctypes.c_size_t, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def library_path() -> str:
    return _LIB_PATH


def status_string(status: int) -> str:
    return _lib.kvarn_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != KVARN_OK:
        raise KvarnError(status, where)


def _ptr(t):
    """Device pointer of a tensor argument (None -> NULL).  Every buffer the library takes is
    device memory, so a host tensor is refused here rather than handed to a kernel."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("every tensor argument must be a CUDA tensor (got one on %s)" % t.device)
    return ctypes.c_void_p(t.data_ptr())


def _dev(t, dtype, name):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s" % (name, dtype))
    return t


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def desc_from_preset(head_dim: int, num_kv_heads: int, preset: str = "kvarn_k4v2_g128",
                     sinkhorn_iters: int | None = None) -> KvarnDesc:
    d = KvarnDesc()
    _check(_lib.kvarn_desc_from_preset(preset.encode(), int(head_dim), int(num_kv_heads),
                                       ctypes.byref(d)), "kvarn_desc_from_preset")
    if sinkhorn_iters is not None:
        d.sinkhorn_iters = int(sinkhorn_iters)
    return d


def page_record_bytes(desc: KvarnDesc) -> int:
    return int(_lib.kvarn_page_record_bytes(ctypes.byref(desc)))


def alloc_pool(desc: KvarnDesc, num_pages: int, device="cuda") -> torch.Tensor:
    """A page pool tensor [num_pages, Hkv, record_bytes] of uint8 (caller-owned memory)."""
    return torch.zeros((num_pages, desc.num_kv_heads, desc.page_record_bytes), dtype=torch.uint8,
                       device=device)


def quantize_tiles(desc: KvarnDesc, k: torch.Tensor, v: torch.Tensor, page_ids: torch.Tensor,
                   pool: torch.Tensor, status: torch.Tensor | None = None, stream=None,
                   sinkhorn_tol: float | None = None, iters_used: torch.Tensor | None = None):
    """k, v: fp16 [tokens, Hkv, d0] (token and head strides taken from the tensors).
    With sinkhorn_tol or iters_used (int32 [tiles, Hkv, 2]) this calls
    kvarn_quantize_tiles_adaptive."""
    _dev(k, torch.float16, "k")
    _dev(v, torch.float16, "v")
    _dev(page_ids, torch.int32, "page_ids")
    if k.shape != v.shape or k.stride() != v.stride() or k.dim() != 3 or k.stride(2) != 1:
        raise ValueError("k and v must be [tokens, Hkv, d0] with matching strides, channels contiguous")
    num_tiles = k.shape[0] // 128
    if page_ids.numel() < num_tiles:
        raise ValueError("page_ids shorter than the number of tiles")
    if sinkhorn_tol is not None or iters_used is not None:
        if iters_used is not None:
            _dev(iters_used, torch.int32, "iters_used")
            if iters_used.numel() < num_tiles * desc.num_kv_heads * 2:
                raise ValueError("iters_used holds fewer than tiles x Hkv x 2 entries")
        _check(_lib.kvarn_quantize_tiles_adaptive(
            ctypes.byref(desc), _ptr(k), _ptr(v), k.stride(0), k.stride(1), num_tiles, _ptr(page_ids),
            _ptr(pool), pool.shape[0], float(sinkhorn_tol or 0.0), _ptr(iters_used), _ptr(status),
            _stream(stream)), "kvarn_quantize_tiles_adaptive")
        return
    _check(_lib.kvarn_quantize_tiles(ctypes.byref(desc), _ptr(k), _ptr(v), k.stride(0), k.stride(1),
                                     num_tiles, _ptr(page_ids), _ptr(pool), pool.shape[0],
                                     _ptr(status), _stream(stream)), "kvarn_quantize_tiles")


def append_token(desc: KvarnDesc, k_new, v_new, partial_k, partial_v, seq_lens, block_table, pool,
                 seq_lens_out=None, status=None, stream=None):
    batch = seq_lens.shape[0]
    _check(_lib.kvarn_append_token(ctypes.byref(desc), batch, _ptr(k_new), _ptr(v_new),
                                   _ptr(partial_k), _ptr(partial_v), _ptr(seq_lens),
                                   _ptr(seq_lens_out), _ptr(block_table), block_table.shape[1],
                                   _ptr(pool), pool.shape[0], _ptr(status), _stream(stream)),
           "kvarn_append_token")


def decode_workspace_bytes(desc: KvarnDesc, batch: int, num_q_heads: int, max_pages: int) -> int:
    return int(_lib.kvarn_decode_workspace_bytes(ctypes.byref(desc), batch, num_q_heads, max_pages))


def alloc_workspace(desc: KvarnDesc, batch: int, num_q_heads: int, max_pages: int, device="cuda"):
    n = decode_workspace_bytes(desc, batch, num_q_heads, max_pages)
    return torch.empty((max(n, 16) + 15) // 16 * 4, dtype=torch.float32, device=device)


def decode_attention(desc: KvarnDesc, q, pool, block_table, seq_lens, out, workspace,
                     partial_k=None, partial_v=None, softmax_scale=None, status=None, stream=None,
                     phase: str = "all"):
    """q, out: fp16 [batch, Hq, d0]; seq_lens: int32 [batch] total lengths.  phase "all"
    (kvarn_decode_attention), or "partials" then "combine" with the same arguments
    (kvarn_decode_partials / kvarn_decode_combine)."""
    fn = {"all": "kvarn_decode_attention", "partials": "kvarn_decode_partials",
          "combine": "kvarn_decode_combine"}[phase]
    batch, hq, d0 = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d0)
    _check(getattr(_lib, fn)(ctypes.byref(desc), batch, hq, _ptr(q), _ptr(pool),
                             pool.shape[0], _ptr(block_table), block_table.shape[1],
                             _ptr(seq_lens), _ptr(partial_k), _ptr(partial_v),
                             float(softmax_scale), _ptr(out), _ptr(workspace),
                             workspace.numel() * workspace.element_size(),
                             _ptr(status), _stream(stream)), fn)


def prefill_workspace_bytes(desc: KvarnDesc, batch: int, num_q_heads: int, chunk_len: int,
                            max_pages: int) -> int:
    return int(_lib.kvarn_prefill_workspace_bytes(ctypes.byref(desc), batch, num_q_heads, chunk_len,
                                                  max_pages))


def alloc_prefill_workspace(desc: KvarnDesc, batch: int, num_q_heads: int, chunk_len: int,
                            max_pages: int, device="cuda"):
    n = prefill_workspace_bytes(desc, batch, num_q_heads, chunk_len, max_pages)
    return torch.empty((max(n, 16) + 15) // 16 * 4, dtype=torch.float32, device=device)


def prefill_attention(desc: KvarnDesc, q, chunk_k, chunk_v, pool, block_table, cache_lens, out,
                      workspace, partial_k=None, partial_v=None, softmax_scale=None, status=None,
                      stream=None):
    """q, out: fp16 [batch, chunk, Hq, d0]; chunk_k/v: fp16 [batch, chunk, Hkv, d0];
    cache_lens: int32 [batch] tokens already cached (sealed pages + partial tile)."""
    batch, chunk, hq, d0 = q.shape
    if chunk_k.shape != (batch, chunk, desc.num_kv_heads, d0) or chunk_v.shape != chunk_k.shape:
        raise ValueError("chunk_k / chunk_v must be [batch, chunk, Hkv, d0]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d0)
    _check(_lib.kvarn_prefill_attention(ctypes.byref(desc), batch, hq, chunk, _ptr(q), _ptr(chunk_k),
                                        _ptr(chunk_v), _ptr(pool), pool.shape[0], _ptr(block_table),
                                        block_table.shape[1], _ptr(cache_lens), _ptr(partial_k),
                                        _ptr(partial_v), float(softmax_scale), _ptr(out),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _ptr(status), _stream(stream)), "kvarn_prefill_attention")


def decode_attention_noalloc(desc: KvarnDesc, q, pool, block_table, seq_lens, out, partial_k=None,
                             partial_v=None, softmax_scale=None, status=None, stream=None):
    """decode_attention without a workspace: the split partials go to the library's fixed
    device buffer (for callers that cannot allocate).  Calls on one device share that buffer,
    so calls overlapping on the GPU must be serialised by the caller."""
    batch, hq, d0 = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d0)
    _check(_lib.kvarn_decode_attention_noalloc(ctypes.byref(desc), batch, hq, _ptr(q), _ptr(pool),
                                               pool.shape[0], _ptr(block_table), block_table.shape[1],
                                               _ptr(seq_lens), _ptr(partial_k), _ptr(partial_v),
                                               float(softmax_scale), _ptr(out), _ptr(status),
                                               _stream(stream)), "kvarn_decode_attention_noalloc")


def fp16_page_bytes(head_dim: int) -> int:
    """Bytes of one uncompressed fp16 (page, kv head) record: K rows then V rows [2][128][d]."""
    return int(_lib.kvarn_fp16_page_bytes(head_dim))


def alloc_fp16_workspace(head_dim: int, batch: int, num_q_heads: int, max_pages: int, device="cuda"):
    n = int(_lib.kvarn_fp16_decode_workspace_bytes(head_dim, batch, num_q_heads, max_pages))
    return torch.empty((max(n, 16) + 15) // 16 * 4, dtype=torch.float32, device=device)


def fp16_decode_attention(num_kv_heads: int, q, pool, block_table, seq_lens, out, workspace,
                          softmax_scale=None, status=None, stream=None):
    """Uncompressed fp16 paged decode (the baseline): q, out fp16 [batch, Hq, d];
    pool fp16 [pages, Hkv, 2, 128, d] (K rows then V rows per page and kv head)."""
    batch, hq, d = q.shape
    if pool.dim() != 5 or pool.shape[1:] != (num_kv_heads, 2, 128, d):
        raise ValueError("pool must be fp16 [pages, Hkv, 2, 128, head_dim]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    _check(_lib.kvarn_fp16_decode_attention(d, num_kv_heads, batch, hq, _ptr(q), _ptr(pool), pool.shape[0],
                                            _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                            float(softmax_scale), _ptr(out), _ptr(workspace),
                                            workspace.numel() * workspace.element_size(), _ptr(status),
                                            _stream(stream)), "kvarn_fp16_decode_attention")


def selftest_wait_timeout(status, stream=None):
    """Launch the bounded-wait self-test: ~2 s later DEV_WAIT_TIMEOUT is set in `status`."""
    _check(_lib.kvarn_selftest_wait_timeout(_ptr(status), _stream(stream)), "kvarn_selftest_wait_timeout")


def dequantize_tiles(desc: KvarnDesc, pool, page_ids, k_out, v_out, status=None, stream=None):
    _check(_lib.kvarn_dequantize_tiles(ctypes.byref(desc), _ptr(pool), pool.shape[0],
                                       _ptr(page_ids), page_ids.numel(), _ptr(k_out), _ptr(v_out),
                                       _ptr(status), _stream(stream)), "kvarn_dequantize_tiles")


def quantization_error(desc: KvarnDesc, k, v, page_ids, pool, err_stats, status=None, stream=None):
    """Error telemetry of the records page_ids[i] against the fp16 tiles of k, v ([tokens, Hkv,
    d0], as given to quantize_tiles): err_stats float32 [tiles, Hkv, 2, 4] receives, per unit,
    sum (x - x^)^2, sum x^2, max |x - x^|, max |x|."""
    _dev(k, torch.float16, "k")
    _dev(v, torch.float16, "v")
    _dev(page_ids, torch.int32, "page_ids")
    _dev(err_stats, torch.float32, "err_stats")
    if k.shape != v.shape or k.stride() != v.stride() or k.dim() != 3 or k.stride(2) != 1:
        raise ValueError("k and v must be [tokens, Hkv, d0] with matching strides, channels contiguous")
    num_tiles = k.shape[0] // 128
    if page_ids.numel() < num_tiles or err_stats.numel() < num_tiles * desc.num_kv_heads * 8:
        raise ValueError("page_ids or err_stats too short for the tiles")
    _check(_lib.kvarn_quantization_error(ctypes.byref(desc), _ptr(k), _ptr(v), k.stride(0), k.stride(1),
                                         num_tiles, _ptr(page_ids), _ptr(pool), pool.shape[0],
                                         _ptr(err_stats), _ptr(status), _stream(stream)),
           "kvarn_quantization_error")
