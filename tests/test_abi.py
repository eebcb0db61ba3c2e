"""The C ABI on the host (CPU only): the library loads, exports every function
include/lcc.h declares, and rejects invalid arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

import long_context_compressed_15_b300 as lcc
from long_context_compressed_15_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    build.build()
    return lcc.load()


def declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(lcc_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ("lcc_csa_compress", "lcc_hca_compress", "lcc_lightning_index_topk", "lcc_csa_sparse_attn",
              "lcc_hca_dense_attn", "lcc_swa_attn", "lcc_attn_merge", "lcc_last_error", "lcc_sync_status"):
        assert f in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.lcc_version().decode().startswith("lcc")


def test_binding_covers_every_function(lib):
    for name in declared_functions():
        assert name in lcc._SIGS, name


def status(call):
    return int(call)


def test_null_and_shape_errors_are_reported_on_host(lib):
    P = ctypes.c_void_p
    # null K
    st = lib.lcc_csa_compress(None, P(16), P(16), 1, 1, 128, 0, 0, P(16), P(16), 0, None)
    assert st == 1 and "null" in lcc.last_error()
    # unsupported D
    st = lib.lcc_hca_compress(P(16), P(16), P(16), 1, 1, 96, 0, 0, P(16), P(16), 0, None)
    assert st == 2 and "D=96" in lcc.last_error()
    # misaligned K
    st = lib.lcc_csa_compress(P(18), P(16), P(16), 1, 1, 128, 0, 0, P(16), P(16), 0, None)
    assert st == 3
    # empty work is a no-op success
    assert lib.lcc_csa_compress(None, None, None, 0, 5, 128, 0, 0, None, None, 0, None) == 0
    # indexer: bad head count, bad k, missing workspace
    args = [P(16), P(16), 1, 1, 6, 64, P(16), 0, P(16), None, P(16), 1024, 4, 128, P(16), None, None, 0, None]
    assert lib.lcc_lightning_index_topk(*args) == 2
    args[4] = 8
    args[13] = 5000
    assert lib.lcc_lightning_index_topk(*args) == 2
    args[13] = 128
    assert lib.lcc_lightning_index_topk(*args) == 8 and "workspace" in lcc.last_error()
    # NVFP4 keys need their scales
    args[7] = 1
    assert lib.lcc_lightning_index_topk(*args) == 1
    # attention: head count not a multiple of 8
    st = lib.lcc_csa_sparse_attn(P(16), 1, 1, 12, 128, 1.0, P(16), P(16), 128, 10, P(16), 4, P(16), P(16), None)
    assert st == 2
    st = lib.lcc_swa_attn(P(16), 1, 1, 64, 128, 1.0, P(16), P(16), P(16), 128, 10, P(16), 0, P(16), P(16), None)
    assert st == 2 and "W=0" in lcc.last_error()
    # merge: too many parts
    assert lib.lcc_attn_merge(5, None, None, 10, 128, None, None, None, None) == 1


def test_workspace_sizes(lib):
    # per query row: scores, one group maximum per 16 entries, two counters and, for rows longer than
    # one 16384-entry top-k segment, a 1024-entry candidate list and a count per segment
    def row_bytes(n):
        nseg = (n + 16383) // 16384
        return n * 4 + (n + 15) // 16 * 4 + 8 + (nseg * (1024 * 8 + 4) if nseg > 1 else 0)
    assert lcc.index_topk_workspace(32, 1, 16384, 128) >= 32 * row_bytes(16384)
    assert lcc.index_topk_workspace(4, 1, 262160, 128) >= 4 * row_bytes(262160)
    # prefill scores are processed in bounded query chunks (2^28 scores)
    rows = (1 << 28) // 32768
    assert lcc.index_topk_workspace(1, 131072, 32768, 128) <= rows * row_bytes(32768) + 6 * 256
    assert lcc.layer_attn_workspace(32, 1, 64, 128, 256) > 0      # decode layers split the key list
    assert lcc.layer_attn_workspace(1, 4096, 64, 128, 256) == 0   # prefill layers write bf16 directly
    assert lcc.dense_attn_workspace(8, 1, 64, 128, 8192) > 0      # decode splits the key range
    assert lcc.dense_attn_workspace(1, 32768, 64, 128, 8448) == 0  # prefill needs none


def test_nvfp4_and_fp4_indexer_host_checks(lib):
    P = ctypes.c_void_p
    # quantiser: D not a multiple of 16, row stride below D, misaligned input; empty work is a no-op
    assert lib.lcc_nvfp4_quantize(P(16), 4, 24, 24, P(16), P(16), P(16), None) == 2 and "D=24" in lcc.last_error()
    assert lib.lcc_nvfp4_quantize(P(16), 4, 64, 32, P(16), P(16), P(16), None) == 2
    assert lib.lcc_nvfp4_quantize(P(18), 4, 64, 64, P(16), P(16), P(16), None) == 3
    assert lib.lcc_nvfp4_quantize(None, 0, 64, 64, None, None, None, None) == 0
    assert lib.lcc_nvfp4_dequantize(None, P(16), 4, 64, P(16), None) == 1
    assert lib.lcc_nvfp4_dequantize(P(12), P(16), 4, 64, P(16), None) == 3
    # the FP4 indexer takes the NVFP4 shapes (8 heads of 64) and needs its workspace
    args = [P(16), P(16), 1, 300, 8, 64, P(16), P(16), P(16), P(16), 32768, 4, 128, P(16), None, None, 0, None]
    assert lib.lcc_fp4_index_topk(*args) == 8 and "workspace" in lcc.last_error()
    args[4] = 4
    assert lib.lcc_fp4_index_topk(*args) == 2
    # workspace: the dequantised query, plus the keys expanded to bf16 (prefill shapes) or the
    # indexer's scratch (decode shapes)
    assert lcc.fp4_index_topk_workspace(1, 300, 8, 64, 32768, 128) >= 300 * 8 * 64 * 2 + 32768 * 64 * 2
    assert (lcc.fp4_index_topk_workspace(4, 1, 8, 64, 262160, 128)
            >= 4 * 8 * 64 * 2 + lcc.index_topk_workspace(4, 1, 262160, 128))
