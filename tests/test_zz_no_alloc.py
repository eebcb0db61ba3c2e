"""The allocation-free indexer entry point, called through the C ABI.

lcc_lightning_index_topk_noalloc serves callers that cannot allocate device
memory (code running under CUDA-graph capture, hosts that pass a routine
only its input and output buffers, decode loops that must stay off the
allocator): its scratch is a fixed 8 MiB array inside the library instead of
a caller workspace.  Its results must equal those of
lcc_lightning_index_topk (index lists bit-exact, the bar every top-k test
here uses; scores to 1e-6 relative), on consecutive calls that reuse the
shared scratch with different sizes.  This file is collected last so that a
run stopping at its first failure has run every other test already.
"""
import ctypes

import pytest
import torch

import datagen
import long_context_compressed_15_b300 as lcc

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(seed, B, Tq, Ncap, k, q_pos0, n_valid, HI=8, DI=64):
    return dict(
        qI=datagen.normal_bf16(seed, 5, (B, Tq, HI, DI)).to(DEV),
        w=datagen.uniform_f32(seed, 6, (B, Tq, HI)).to(DEV),
        kI=datagen.normal_bf16(seed, 7, (B, Ncap, DI)).to(DEV),
        q_pos0=torch.tensor(q_pos0, dtype=torch.int64, device=DEV),
        n_valid=torch.tensor(n_valid, dtype=torch.int32, device=DEV),
        B=B, Tq=Tq, Ncap=Ncap, k=k, HI=HI, DI=DI)


def _noalloc(lib, c):
    idx = torch.full((c["B"], c["Tq"], c["k"]), -7, dtype=torch.int32, device=DEV)
    sc = torch.full((c["B"], c["Tq"], c["k"]), 7.0, dtype=torch.float32, device=DEV)
    P = ctypes.c_void_p
    st = lib.lcc_lightning_index_topk_noalloc(
        P(c["qI"].data_ptr()), P(c["w"].data_ptr()), c["B"], c["Tq"], c["HI"], c["DI"], P(c["q_pos0"].data_ptr()),
        0, P(c["kI"].data_ptr()), None, P(c["n_valid"].data_ptr()), c["Ncap"], 4, c["k"], P(idx.data_ptr()),
        P(sc.data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lcc.last_error()
    return idx, sc


def _reference(c):
    sc = torch.empty((c["B"], c["Tq"], c["k"]), dtype=torch.float32, device=DEV)
    idx = lcc.lightning_index_topk(c["qI"], c["w"], c["q_pos0"], c["kI"], c["n_valid"], 4, c["k"], score=sc)
    return idx, sc


def _same(a, b):
    ia, sa = a
    ib, sb = b
    assert torch.equal(ia, ib)
    fin = torch.isfinite(sb)
    assert torch.equal(torch.isfinite(sa), fin)
    assert torch.allclose(sa[fin], sb[fin], rtol=1e-6, atol=0)


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    lib = lcc.load()
    # decode-sized: two-stage top-k (Ncap > 8192), ragged n_valid, one query chunk
    dec = _case(41, 4, 1, 20000, 128, [4 * 20000 - 1] * 4, [20000, 9000, 100, 1])
    # prefill-sized: 300 causal queries need 10.8 MB of scores, so the fixed
    # scratch is used in several query chunks
    pre = _case(42, 1, 300, 9000, 64, [4 * 9000 - 300], [9000])
    first = _noalloc(lib, dec)
    second = _noalloc(lib, pre)        # reuses the scratch the first call left behind
    third = _noalloc(lib, dec)         # and back, after a larger call
    torch.cuda.synchronize()
    lcc.sync_status()
    ref_dec, ref_pre = _reference(dec), _reference(pre)
    torch.cuda.synchronize()
    _same(first, ref_dec)
    _same(second, ref_pre)
    _same(third, ref_dec)
    assert torch.all(first[0][2, 0, 100:] == -1) and torch.all(first[0][3, 0, 1:] == -1)


def test_noalloc_rejects_requests_beyond_its_scratch():
    lib = lcc.load()
    P = ctypes.c_void_p
    # 64 sequences x 100000 entries need 25.6 MB of scores for a single query row
    st = lib.lcc_lightning_index_topk_noalloc(P(16), P(16), 64, 1, 8, 64, P(16), 0, P(16), None, P(16), 100000, 4,
                                              128, P(16), None, None)
    assert st == 8 and "scratch" in lcc.last_error()
