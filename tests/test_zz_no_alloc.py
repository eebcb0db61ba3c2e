"""The allocation-free indexer entry point, called through the C ABI.

lcc_lightning_index_topk_noalloc serves callers that cannot allocate device
memory (code running under CUDA-graph capture, hosts that pass a routine
only its input and output buffers, decode loops that must stay off the
allocator): its scratch is a fixed 8 MiB array inside the library instead of
a caller workspace.  Its results must equal those of
lcc_lightning_index_topk (index lists bit-exact, the bar every top-k test
here uses; scores to 1e-6 relative) and match the fp64 oracle under the
near-tie rule, on consecutive calls that reuse the shared scratch with
different layouts:

* decode batches (one query chunk, segmented top-k over 20000 entries);
* k = 512 with bf16 keys: 300 causal queries in chunks of 128;
* NVFP4 keys: 40 queries over 60000 entries in chunks of 16, 16 and 8;
* 64 sequences x 20000 entries: one query row per chunk (two chunks);
* a prefill-shaped request (fused top-k) far larger than the array, which
  uses no scratch and is accepted.

This file is collected last so that a run stopping at its first failure has
run every other test already.
"""
import ctypes

import numpy as np
import pytest
import torch

import datagen
import long_context_compressed_15_b300 as lcc
import oracle
from parity import check_topk_rows, host

pytestmark = pytest.mark.gpu
DEV = "cuda"
M = 4


def _case(seed, B, Tq, Ncap, k, q_pos0, n_valid, HI=8, DI=64, fp4=False):
    c = dict(
        qI=datagen.normal_bf16(seed, 5, (B, Tq, HI, DI)).to(DEV),
        w=datagen.uniform_f32(seed, 6, (B, Tq, HI)).to(DEV),
        q_pos0=torch.tensor(q_pos0, dtype=torch.int64, device=DEV),
        n_valid=torch.tensor(n_valid, dtype=torch.int32, device=DEV),
        B=B, Tq=Tq, Ncap=Ncap, k=k, HI=HI, DI=DI, fp4=fp4)
    if fp4:
        kp, ks = datagen.nvfp4_normal(seed, 7, B * Ncap, DI)
        c["kI"] = kp.reshape(B, Ncap, DI // 2).to(DEV)
        c["kI_scale"] = ks.reshape(B, Ncap, DI // 16).to(DEV)
    else:
        c["kI"] = datagen.normal_bf16(seed, 7, (B, Ncap, DI)).to(DEV)
        c["kI_scale"] = None
    return c


def _noalloc(lib, c):
    idx = torch.full((c["B"], c["Tq"], c["k"]), -7, dtype=torch.int32, device=DEV)
    sc = torch.full((c["B"], c["Tq"], c["k"]), 7.0, dtype=torch.float32, device=DEV)
    P = ctypes.c_void_p
    scale = P(c["kI_scale"].data_ptr()) if c["fp4"] else None
    st = lib.lcc_lightning_index_topk_noalloc(
        P(c["qI"].data_ptr()), P(c["w"].data_ptr()), c["B"], c["Tq"], c["HI"], c["DI"], P(c["q_pos0"].data_ptr()),
        1 if c["fp4"] else 0, P(c["kI"].data_ptr()), scale, P(c["n_valid"].data_ptr()), c["Ncap"], M, c["k"],
        P(idx.data_ptr()), P(sc.data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lcc.last_error()
    return idx, sc


def _reference(c):
    sc = torch.empty((c["B"], c["Tq"], c["k"]), dtype=torch.float32, device=DEV)
    idx = lcc.lightning_index_topk(c["qI"], c["w"], c["q_pos0"], c["kI"], c["n_valid"], M, c["k"],
                                   kI_scale=c["kI_scale"], score=sc)
    return idx, sc


def _same(a, b):
    ia, sa = a
    ib, sb = b
    assert torch.equal(ia, ib)
    fin = torch.isfinite(sb)
    assert torch.equal(torch.isfinite(sa), fin)
    assert torch.allclose(sa[fin], sb[fin], rtol=1e-6, atol=0)


def _oracle_rows(c, idx, max_near):
    """Every row's index set against the fp64 oracle (near-tie rule)."""
    qI = host(c["qI"]).astype(np.uint16)
    w = host(c["w"]).astype(np.float64)
    if c["fp4"]:
        kp, ks = host(c["kI"]), host(c["kI_scale"])
    else:
        kI = oracle.bf16_to_f64(host(c["kI"]))
    pos0, nval = host(c["q_pos0"]), host(c["n_valid"])
    gi = host(idx)
    near = 0
    for b in range(c["B"]):
        keys = oracle.nvfp4_decode(kp[b], ks[b]) if c["fp4"] else kI[b]
        refs = []
        for i in range(c["Tq"]):
            nv = oracle.visible_count(int(pos0[b]) + i, M, int(nval[b]))
            s = oracle.index_scores(oracle.bf16_to_f64(qI[b, i]), w[b, i], keys[:nv])
            oi, kth = oracle.topk_select(s, c["k"])
            refs.append(dict(idx=oi, scores=s, kth=kth))
        near += check_topk_rows(gi[b], refs, c["k"], f"batch {b}")
    assert near <= max_near


def test_noalloc_matches_workspace_entry_and_oracle_on_consecutive_calls():
    lib = lcc.load()
    # decode-sized: segmented top-k (Ncap > 16384), ragged n_valid, one query chunk
    dec = _case(41, 4, 1, 20000, 128, [M * 20000 - 1] * 4, [20000, 9000, 100, 1])
    # k > 256 keeps bf16 prefill requests off the fused top-k: 300 queries need
    # 11.5 MB of scratch, so they run in chunks of 128, 128 and 44 queries
    big_k = _case(42, 1, 300, 9000, 512, [M * 9000 - 300], [9000])
    # NVFP4 keys always take the score + top-k kernels: 40 queries over 60000
    # entries run in chunks of 16, 16 and 8 queries
    fp4 = _case(43, 1, 40, 60000, 128, [M * 60000 - 40], [60000], fp4=True)
    # one query row of 64 sequences x 20000 entries fills most of the array:
    # two queries run as two chunks of one
    wide = _case(44, 64, 2, 20000, 128, [M * 20000 - 2] * 64, [20000 - 37 * (b % 3) for b in range(64)])
    calls = [("dec", dec), ("big_k", big_k), ("dec", dec), ("fp4", fp4), ("dec", dec), ("wide", wide),
             ("big_k", big_k), ("dec", dec)]
    got = [(name, _noalloc(lib, c)) for name, c in calls]
    torch.cuda.synchronize()
    lcc.sync_status()
    cases = dict(dec=dec, big_k=big_k, fp4=fp4, wide=wide)
    refs = {name: _reference(c) for name, c in cases.items()}
    torch.cuda.synchronize()
    lcc.sync_status()
    for name, res in got:
        _same(res, refs[name])
    for name, c in cases.items():
        _oracle_rows(c, refs[name][0], max_near=max(2, c["B"] * c["Tq"] // 100))
    d = got[0][1][0]
    assert torch.all(d[2, 0, 100:] == -1) and torch.all(d[3, 0, 1:] == -1)


def test_noalloc_fused_prefill_request_needs_no_scratch():
    lib = lcc.load()
    # 64 sequences x 40000 entries: one query row alone needs 12 MB of scores on
    # the unfused path, but 3 queries x 8 heads take the fused top-k
    big = _case(45, 64, 3, 40000, 128, [M * 40000 - 3] * 64, [40000] * 64)
    a = _noalloc(lib, big)
    torch.cuda.synchronize()
    lcc.sync_status()
    _same(a, _reference(big))


def test_noalloc_rejects_requests_beyond_its_scratch():
    lib = lcc.load()
    P = ctypes.c_void_p
    # 64 sequences x 100000 entries need 25.6 MB of scores for a single query row
    st = lib.lcc_lightning_index_topk_noalloc(P(16), P(16), 64, 1, 8, 64, P(16), 0, P(16), None, P(16), 100000, 4,
                                              128, P(16), None, None)
    assert st == 8 and "scratch" in lcc.last_error()
