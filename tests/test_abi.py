"""The C-ABI library builds, loads and exports every symbol kvarn.h declares (CPU only).

Only host-side entry points are called here (descriptor, sizes, status strings and the
argument validation that returns before any CUDA call).
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kv():
    from calibration_free_kv_gb300 import build
    build.build()
    from calibration_free_kv_gb300 import kvarn
    return kvarn


def _declared_functions():
    with open(os.path.join(ROOT, "include", "kvarn.h")) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvarn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("kvarn_quantize_tiles", "kvarn_append_token", "kvarn_decode_attention",
                     "kvarn_dequantize_tiles"):
        assert required in names


def test_library_exports_every_declared_symbol(kv):
    lib = ctypes.CDLL(kv.library_path())
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) <= set(kv.EXPORTED_SYMBOLS) | set()


def test_preset_descriptor(kv):
    d = kv.desc_from_preset(128, 8)
    assert (d.head_dim, d.head_dim_padded, d.num_kv_heads) == (128, 128, 8)
    assert (d.tile_tokens, d.k_bits, d.v_bits, d.sinkhorn_iters) == (128, 4, 2, 4)
    assert d.page_record_bytes == 13824 == kv.page_record_bytes(d)
    assert kv.desc_from_preset(96, 8).head_dim_padded == 128
    assert kv.desc_from_preset(256, 4).page_record_bytes == 26880


def test_record_bytes_match_oracle(kv):
    from oracle import kvarn_oracle as ko
    for d0 in (64, 96, 128, 200, 256):
        desc = kv.desc_from_preset(d0, 2)
        assert desc.page_record_bytes == ko.record_bytes(ko.padded_head_dim(d0))


def test_every_oracle_preset_has_a_descriptor(kv):
    # the library's preset table and the oracle's agree on names, widths and record sizes
    from oracle import kvarn_oracle as ko
    for name, (kb, vb) in ko.PRESETS.items():
        for d0 in (64, 96, 128, 256):
            desc = kv.desc_from_preset(d0, 3, preset=name)
            assert (desc.k_bits, desc.v_bits) == (kb, vb)
            assert desc.page_record_bytes == kv.page_record_bytes(desc) == \
                ko.record_bytes(ko.padded_head_dim(d0), k_bits=kb, v_bits=vb)


def test_preset_rejections(kv):
    with pytest.raises(kv.KvarnError) as e:
        kv.desc_from_preset(128, 8, preset="kvarn_k2v2_g64")
    assert e.value.status == kv.KVARN_ERR_UNSUPPORTED
    for bad in (0, 7, 100, 264):
        with pytest.raises(kv.KvarnError):
            kv.desc_from_preset(bad, 8)
    # head_dim <= 32 pads to itself (8, 16, 32 or 32 for 24), which has no page record
    for small in (8, 16, 24, 32):
        with pytest.raises(kv.KvarnError) as e:
            kv.desc_from_preset(small, 8)
        assert e.value.status == kv.KVARN_ERR_UNSUPPORTED
    assert kv.desc_from_preset(40, 8).head_dim_padded == 64


def test_workspace_size(kv):
    d = kv.desc_from_preset(128, 8)
    n = kv.decode_workspace_bytes(d, 64, 32, 128)
    splits = (128 + 31) // 32 + 2  # 32-page splits, the partial tile's, and one more
    assert n == 64 * 32 * splits * (128 + 4) * 4


def test_validation_returns_before_launch(kv):
    lib = kv._lib
    d = kv.desc_from_preset(128, 8)
    null = ctypes.c_void_p(0)
    st = lib.kvarn_quantize_tiles(ctypes.byref(d), null, null, 1024, 128, 4, null, null, 8, null, null)
    assert st == kv.KVARN_ERR_INVALID_ARG
    assert lib.kvarn_quantize_tiles(ctypes.byref(d), null, null, 1024, 128, 0, null, null, 8, null,
                                    null) == kv.KVARN_OK
    # G = 3 is not a supported group size
    st = lib.kvarn_decode_attention(ctypes.byref(d), 2, 24, null, null, 8, null, 4, null, null, null,
                                    ctypes.c_float(0.1), null, null, 0, null, null)
    assert st == kv.KVARN_ERR_UNSUPPORTED
    st = lib.kvarn_decode_attention(ctypes.byref(d), 2, 32, ctypes.c_void_p(16), ctypes.c_void_p(16), 8,
                                    ctypes.c_void_p(16), 4, ctypes.c_void_p(16), null, null,
                                    ctypes.c_float(0.1), ctypes.c_void_p(16), ctypes.c_void_p(16), 8,
                                    null, null)
    assert st == kv.KVARN_ERR_WORKSPACE_TOO_SMALL
    # partial tiles are staged with bulk copies: a misaligned one is refused before any launch
    st = lib.kvarn_decode_attention(ctypes.byref(d), 2, 32, ctypes.c_void_p(16), ctypes.c_void_p(16), 8,
                                    ctypes.c_void_p(16), 4, ctypes.c_void_p(16), ctypes.c_void_p(24),
                                    ctypes.c_void_p(16), ctypes.c_float(0.1), ctypes.c_void_p(16),
                                    ctypes.c_void_p(16), 1 << 30, null, null)
    assert st == kv.KVARN_ERR_INVALID_ARG
    bad = kv.KvarnDesc.from_buffer_copy(d)
    bad.k_bits = 3
    assert lib.kvarn_dequantize_tiles(ctypes.byref(bad), null, 1, null, 1, null, null, null,
                                      null) == kv.KVARN_ERR_UNSUPPORTED
    assert "workspace" in kv.status_string(kv.KVARN_ERR_WORKSPACE_TOO_SMALL)


def test_noalloc_argument_errors_match_the_workspace_entry_point(kv):
    # the allocation-free decode checks its arguments before it looks up its buffer (no CUDA
    # call): the same bad arguments give the same codes as kvarn_decode_attention, and an empty
    # batch is a no-op; host only
    lib = kv._lib
    d = kv.desc_from_preset(128, 8)
    null = ctypes.c_void_p(0)
    p16 = ctypes.c_void_p(16)
    bad_bits = kv.KvarnDesc.from_buffer_copy(d)
    bad_bits.k_bits = 3
    cases = [
        (None, 2, 32, p16, p16, 8, p16, 4, p16, null, null, 0.1, p16),          # no descriptor
        (bad_bits, 2, 32, p16, p16, 8, p16, 4, p16, null, null, 0.1, p16),      # unsupported bits
        (d, 2, 24, p16, p16, 8, p16, 4, p16, null, null, 0.1, p16),             # G = 3
        (d, -1, 32, p16, p16, 8, p16, 4, p16, null, null, 0.1, p16),            # negative batch
        (d, 2, 32, null, p16, 8, p16, 4, p16, null, null, 0.1, p16),            # no q
        (d, 2, 32, p16, p16, 8, p16, 4, p16, ctypes.c_void_p(24), p16, 0.1, p16),  # misaligned partial
        (d, 2, 32, p16, p16, 8, p16, 4, p16, p16, null, 0.1, p16),              # one partial only
        (d, 2, 32, p16, p16, 8, p16, 4, p16, null, null, 0.0, p16),             # softmax scale 0
        (d, 0, 32, null, null, 8, null, 4, null, null, null, 0.1, null),        # empty batch: ok
    ]
    for c in cases:
        desc = ctypes.POINTER(kv.KvarnDesc)() if c[0] is None else ctypes.byref(c[0])
        args = (desc,) + c[1:11] + (ctypes.c_float(c[11]), c[12])
        want = lib.kvarn_decode_attention(*args, ctypes.c_void_p(16), 1 << 30, null, null)
        got = lib.kvarn_decode_attention_noalloc(*args, null, null)
        assert got == want, (c, got, want)
    assert want == kv.KVARN_OK


def test_fp16_baseline_validation(kv):
    # the fp16 baseline decode refuses unsupported shapes and bad arguments before any launch
    lib = kv._lib
    null = ctypes.c_void_p(0)
    p16 = ctypes.c_void_p(16)
    assert kv.fp16_page_bytes(128) == 2 * 128 * 128 * 2
    assert kv.fp16_page_bytes(96) == 0
    assert lib.kvarn_fp16_decode_workspace_bytes(128, 2, 32, 4) == 2 * 32 * 1 * (128 + 4) * 4
    args = lambda hd, hkv, hq, ws_bytes, pool=p16: (hd, hkv, 2, hq, p16, pool, 8, p16, 4, p16,
                                                     ctypes.c_float(0.1), p16, p16, ws_bytes, null, null)
    assert lib.kvarn_fp16_decode_attention(*args(96, 8, 32, 1 << 20)) == kv.KVARN_ERR_UNSUPPORTED
    assert lib.kvarn_fp16_decode_attention(*args(128, 8, 24, 1 << 20)) == kv.KVARN_ERR_UNSUPPORTED
    assert lib.kvarn_fp16_decode_attention(*args(128, 8, 32, 16)) == kv.KVARN_ERR_WORKSPACE_TOO_SMALL
    assert lib.kvarn_fp16_decode_attention(*args(128, 8, 32, 1 << 20, ctypes.c_void_p(24))) == \
        kv.KVARN_ERR_INVALID_ARG
    assert lib.kvarn_selftest_wait_timeout(null, null) == kv.KVARN_ERR_INVALID_ARG


_C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "kvarn.h"

int main(void) {
  kvarn_desc d;
  if (kvarn_desc_from_preset("kvarn_k4v2_g128", 128, 8, &d) != KVARN_OK) return 1;
  if (d.page_record_bytes != 13824 || kvarn_page_record_bytes(&d) != 13824) return 2;
  if (kvarn_desc_from_preset("no_such_preset", 128, 8, &d) != KVARN_ERR_UNSUPPORTED) return 3;
  if (kvarn_desc_from_preset("kvarn_k4v2_g128", 128, 8, &d) != KVARN_OK) return 4;
  if (kvarn_decode_workspace_bytes(&d, 64, 32, 128) == 0) return 5;
  /* argument errors return before any CUDA call */
  if (kvarn_decode_attention(NULL, 1, 4, NULL, NULL, 1, NULL, 1, NULL, NULL, NULL, 0.1f, NULL,
                             NULL, 0, NULL, NULL) != KVARN_ERR_INVALID_ARG) return 6;
  if (strlen(kvarn_status_string(KVARN_ERR_WORKSPACE_TOO_SMALL)) == 0) return 7;
  printf("ok %lld\n", (long long)d.page_record_bytes);
  return 0;
}
"""


def test_header_is_plain_c_and_links(kv, tmp_path):
    # a C11 client compiles against kvarn.h alone (no C++ in the declarations) and links the
    # shared library by its exported C names
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(_C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(kv.library_path())
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", libdir, "-lkvarn", "-Wl,-rpath," + libdir, "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.strip() == "ok 13824"


def test_binding_fails_loudly_without_the_library(tmp_path):
    # the binding has no fallback: without libkvarn.so importing it raises
    import shutil
    import subprocess
    import sys
    pkg = tmp_path / "calibration_free_kv_gb300"
    pkg.mkdir()
    for name in ("__init__.py", "kvarn.py", "synth.py", "build.py"):
        shutil.copy(os.path.join(ROOT, "calibration_free_kv_gb300", name), pkg / name)
    r = subprocess.run([sys.executable, "-c", "from calibration_free_kv_gb300 import kvarn"],
                       cwd=str(tmp_path), capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, PYTHONPATH=str(tmp_path)))
    assert r.returncode != 0
    assert "libkvarn.so is not built" in r.stderr and "no fallback" in r.stderr


def test_binding_rejects_host_tensors(kv):
    # every tensor argument must be device memory: a CPU tensor is refused before any call
    import torch
    d = kv.desc_from_preset(128, 2)
    q = torch.zeros((1, 8, 128), dtype=torch.float16)
    pool = torch.zeros((2, 2, d.page_record_bytes), dtype=torch.uint8)
    table = torch.zeros((1, 1), dtype=torch.int32)
    lens = torch.zeros(1, dtype=torch.int32)
    out = torch.zeros_like(q)
    ws = torch.zeros(kv.decode_workspace_bytes(d, 1, 8, 1), dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        kv.decode_attention(d, q, pool, table, lens, out, ws)
