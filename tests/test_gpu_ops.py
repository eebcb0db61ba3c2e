"""Per-call parity of the CUDA path (through the C ABI) against the fp64
oracle, at sizes the oracle finishes in seconds that still span several
tiles, ragged tails and the method's degenerate cases."""
import numpy as np
import pytest
import torch

import datagen
import long_context_compressed_15_b300 as lcc
import oracle
from oracle import runs
from parity import assert_close, assert_lse_close, bits, check_topk_rows, host, topk_set_ok

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lcc.load()


def f64(t):
    return runs.f64(host(t))


# ---------------------------------------------------------------------------
# compression
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("m,D,R", [(4, 128, 4 * 37 + 3), (4, 64, 4 * 300 + 1), (128, 128, 128 * 3 + 50),
                                   (128, 64, 128 * 2)])
def test_compress_parity(m, D, R):
    B = 3
    K = datagen.normal_bf16(11, 1, (B, R, D))
    V = datagen.normal_bf16(11, 2, (B, R, D))
    g = datagen.normal_f32(11, 3, (B, R))
    n = R // m
    Kc = torch.full((B, n + 2, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    Vc = torch.full_like(Kc, float("nan"))
    fn = lcc.csa_compress if m == 4 else lcc.hca_compress
    fn(K.to(DEV), V.to(DEV), g.to(DEV), Kc, Vc)
    torch.cuda.synchronize()
    for b in range(B):
        ex_k, ex_v = oracle.pool_exact(f64(K[b]), f64(V[b]), f64(g[b]), m)
        st_k, st_v = oracle.pool(f64(K[b]), f64(V[b]), f64(g[b]), m)
        for gpu, ex, st in ((Kc[b, :n], ex_k, st_k), (Vc[b, :n], ex_v, st_v)):
            gv = f64(gpu)
            ulp = np.ldexp(1.0, np.frexp(np.abs(ex))[1] - 8)
            assert np.all(np.abs(gv - ex) <= ulp), "pooled entry off by more than one bf16 ulp"
            assert np.mean(gv == st) > 0.99
        # entries past the last complete block are untouched
        assert torch.isnan(Kc[b, n:].float()).all()


@pytest.mark.parametrize("m,D,R", [(4, 128, 4 * 37 + 3), (128, 64, 128 * 3 + 50)])
def test_compress_at_device_positions(m, D, R):
    # positions and n_valid on the device: sequence 0 from token 0, sequence 1 from a later block,
    # sequence 2 running past Ncap (blocks beyond it dropped), sequence 3 misaligned (skipped, reported)
    B, n = 4, R // m
    Ncap = n + 12
    K = datagen.normal_bf16(15, 1, (B, R, D))
    V = datagen.normal_bf16(15, 2, (B, R, D))
    g = datagen.normal_f32(15, 3, (B, R))
    e0 = [0, 9, Ncap - 5, 0]
    tok0 = torch.tensor([e * m for e in e0[:3]] + [m + 1], dtype=torch.int64, device=DEV)
    nv0 = [3, n + 20, 0, 2]
    n_valid = torch.tensor(nv0, dtype=torch.int32, device=DEV)
    Kc = torch.full((B, Ncap, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    Vc = torch.full_like(Kc, float("nan"))
    lcc.compress_at(m, K.to(DEV), V.to(DEV), g.to(DEV), tok0, Kc, Vc, n_valid=n_valid)
    torch.cuda.synchronize()
    with pytest.raises(lcc.LccError, match="not a multiple of m"):
        lcc.sync_status()
    want_nv = [max(nv0[b], min(Ncap, e0[b] + n)) for b in range(3)] + [nv0[3]]
    assert n_valid.cpu().tolist() == want_nv
    for b in range(3):
        ex_k, ex_v = oracle.pool_exact(f64(K[b]), f64(V[b]), f64(g[b]), m)
        # fp32 arithmetic before the bf16 rounding: weights (exp, division) and the m products
        # each within a few fp32 ulps of sum_i a_i |x_i|, which matters where the entry cancels
        mag_k, mag_v = oracle.pool_exact(np.abs(f64(K[b])), np.abs(f64(V[b])), f64(g[b]), m)
        lo, hi = e0[b], min(Ncap, e0[b] + n)
        for what, gpu, ex, mag in (("K", Kc[b, lo:hi], ex_k[:hi - lo], mag_k[:hi - lo]),
                                   ("V", Vc[b, lo:hi], ex_v[:hi - lo], mag_v[:hi - lo])):
            gv = f64(gpu)
            ulp = np.ldexp(1.0, np.frexp(np.abs(ex))[1] - 8) + np.ldexp(mag, -20)
            r = np.abs(gv - ex) / ulp
            assert np.isfinite(gv).all(), f"sequence {b} {what}: {np.sum(~np.isfinite(gv))} entries not written"
            assert r.max() <= 1.0, f"sequence {b} {what}: {r.max():.3f} of the bound at {np.unravel_index(r.argmax(), r.shape)}"
        assert torch.isnan(Kc[b, :lo].float()).all() and torch.isnan(Kc[b, hi:].float()).all()
    assert torch.isnan(Kc[3].float()).all() and torch.isnan(Vc[3].float()).all()


def test_compress_m1_is_a_copy():
    # m = 1 (the DSA comparator's cache): every token is its own entry
    B, R, D = 2, 77, 128
    K = datagen.normal_bf16(14, 1, (B, R, D)).to(DEV)
    V = datagen.normal_bf16(14, 2, (B, R, D)).to(DEV)
    g = datagen.normal_f32(14, 3, (B, R)).to(DEV)
    Kc = torch.full((B, R, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    Vc = torch.full_like(Kc, float("nan"))
    lcc.compress(1, K, V, g, Kc, Vc)
    torch.cuda.synchronize()
    assert torch.equal(Kc, K) and torch.equal(Vc, V)


def test_compress_one_block_at_offset():
    # a decode step pools one freshly completed block from the middle of a raw buffer
    B, R, D = 2, 40, 128
    K = datagen.normal_bf16(12, 1, (B, R, D))
    V = datagen.normal_bf16(12, 2, (B, R, D))
    g = datagen.normal_f32(12, 3, (B, R))
    Kc = torch.zeros((B, 10, D), dtype=torch.bfloat16, device=DEV)
    Vc = torch.zeros_like(Kc)
    Kd, Vd, gd = K.to(DEV), V.to(DEV), g.to(DEV)
    lcc.csa_compress(Kd[:, 20:], Vd[:, 20:], gd[:, 20:], Kc[:, 7:], Vc[:, 7:], n_blocks=1)
    torch.cuda.synchronize()
    for b in range(B):
        st_k, st_v = oracle.pool(f64(K[b, 20:24]), f64(V[b, 20:24]), f64(g[b, 20:24]), 4)
        assert np.max(np.abs(f64(Kc[b, 7]) - st_k[0])) <= np.max(np.abs(st_k)) * 2 ** -7
        assert torch.count_nonzero(Kc[b, :7].float()) == 0 and torch.count_nonzero(Kc[b, 8:].float()) == 0


# ---------------------------------------------------------------------------
# lightning indexer + top-k
# ---------------------------------------------------------------------------
def _index_case(seed, B, Tq, HI, DI, Ncap, m, k, q_pos0, n_valid, nvfp4=False):
    qI = datagen.normal_bf16(seed, 5, (B, Tq, HI, DI))
    w = datagen.uniform_f32(seed, 6, (B, Tq, HI))
    if nvfp4:
        kp, ks = datagen.nvfp4_normal(seed, 7, B * Ncap, DI)
        kp, ks = kp.reshape(B, Ncap, DI // 2), ks.reshape(B, Ncap, DI // 16)
        kI_host = oracle.nvfp4_decode(kp.numpy(), ks.numpy())
        idx = lcc.lightning_index_topk(qI.to(DEV), w.to(DEV), torch.tensor(q_pos0, device=DEV),
                                       kp.to(DEV), torch.tensor(n_valid, dtype=torch.int32, device=DEV),
                                       m, k, kI_scale=ks.to(DEV))
    else:
        kI = datagen.normal_bf16(seed, 7, (B, Ncap, DI))
        kI_host = f64(kI)
        idx = lcc.lightning_index_topk(qI.to(DEV), w.to(DEV), torch.tensor(q_pos0, device=DEV), kI.to(DEV),
                                       torch.tensor(n_valid, dtype=torch.int32, device=DEV), m, k)
    torch.cuda.synchronize()
    lcc.sync_status()
    g = idx.cpu().numpy()
    near = 0
    for b in range(B):
        rows = []
        for i in range(Tq):
            nv = oracle.visible_count(q_pos0[b] + i, m, min(n_valid[b], Ncap))
            s = oracle.index_scores(f64(qI[b, i]), f64(w[b, i]), kI_host[b, :nv])
            oi, kth = oracle.topk_select(s, k)
            rows.append(dict(idx=oi, scores=s, kth=kth))
        near += check_topk_rows(g[b], rows, k, what=f"batch {b}")
    return near, g


@pytest.mark.parametrize("HI,DI", [(8, 64), (4, 32), (8, 32), (4, 64)])
def test_index_topk_decode_two_stage(HI, DI):
    # rows longer than 16384 entries (625 score groups of 32); ragged n_valid
    B, Ncap = 3, 20000
    near, g = _index_case(21, B, 1, HI, DI, Ncap, 4, 128, q_pos0=[4 * Ncap - 1] * B, n_valid=[Ncap, 8193, 100])
    assert np.all(g[2, 0, 100:] == -1) and np.all(g[2, 0, :100] == np.arange(100))
    assert near <= 1


@pytest.mark.parametrize("HI,DI", [(8, 64), (4, 32)])
def test_index_topk_decode_cluster(HI, DI):
    # the visible counts cover a full 16384-entry row, rows whose group maxima give no threshold
    # (fewer than k groups of 32: 4000 and 2049 entries, the latter one entry into a new group),
    # a row just above k and one below it
    B, Ncap = 5, 16384
    near, g = _index_case(26, B, 1, HI, DI, Ncap, 4, 128, q_pos0=[4 * Ncap - 1] * B,
                          n_valid=[Ncap, 4000, 2049, 129, 50])
    assert np.all(g[4, 0, 50:] == -1) and np.all(g[4, 0, :50] == np.arange(50))
    assert near <= 1


def test_index_topk_prefill_causal_with_ties():
    # 4 heads: about 1 in 16 entries scores exactly 0 (all four ReLUs vanish); early
    # queries see fewer than k entries and must be padded
    near, g = _index_case(22, 1, 700, 4, 32, 175, 4, 16, q_pos0=[0], n_valid=[175])
    assert np.all(g[0, :3] == -1)
    assert list(g[0, 3, :2]) == [0, -1]
    assert near <= 2


@pytest.mark.parametrize("Ncap", [3000, 40000])
def test_index_topk_zero_score_ties_bit_exact(Ncap):
    # weights of zero make every score 0: the top-k must be the lowest indices (3000 entries: one
    # top-k CTA whose candidate list overflows; 40000: three segments whose lists overflow)
    B, k = 2, 64
    qI = datagen.normal_bf16(23, 5, (B, 1, 8, 64)).to(DEV)
    w = torch.zeros((B, 1, 8), dtype=torch.float32, device=DEV)
    kI = datagen.normal_bf16(23, 7, (B, Ncap, 64)).to(DEV)
    idx = lcc.lightning_index_topk(qI, w, 4 * Ncap, kI, Ncap, 4, k)
    torch.cuda.synchronize()
    assert torch.equal(idx.cpu(), torch.arange(k, dtype=torch.int32).expand(B, 1, k))


def test_index_topk_nvfp4_keys():
    B, Ncap = 2, 9000
    near, _ = _index_case(24, B, 2, 8, 64, Ncap, 4, 128, q_pos0=[4 * Ncap - 2] * B, n_valid=[Ncap, 5000],
                          nvfp4=True)
    assert near <= 1


def test_index_nvfp4_scores_exact_for_any_query_scale():
    # each (query, head) row of qI scaled by its own power of two in 2^-30 .. 2^30:
    # rounding bf16 queries to fp16 would lose or overflow them; the per-row
    # power-of-two scaling keeps the scores at fp32 accuracy
    B, Tq, N, HI, DI = 2, 3, 3000, 8, 64
    kp, ks = datagen.nvfp4_normal(19, 1, B * N, DI)
    kI, kIs = kp.reshape(B, N, DI // 2).to(DEV), ks.reshape(B, N, DI // 16).to(DEV)
    exps = (torch.arange(B * Tq * HI, dtype=torch.float32).reshape(B, Tq, HI, 1) * 17) % 61 - 30
    qI = (datagen.normal_bf16(19, 2, (B, Tq, HI, DI)).float() * torch.exp2(exps)).to(torch.bfloat16).to(DEV)
    w = (datagen.uniform_f32(19, 3, (B, Tq, HI)) * torch.exp2(-exps[..., 0])).to(DEV)
    pos = torch.full((B,), 4 * N - Tq, dtype=torch.int64, device=DEV)
    sc = lcc.lightning_index_scores(qI, w, pos, kI, N, 4, kI_scale=kIs)
    torch.cuda.synchronize()
    for b in range(B):
        keys = oracle.nvfp4_decode(host(kI[b]), host(kIs[b]))
        for i in range(Tq):
            nv = oracle.visible_count(4 * N - Tq + i, 4, N)
            want = oracle.index_scores(f64(qI[b, i]), host(w[b, i]).astype(np.float64), keys[:nv])
            got = sc[b, i, :nv].cpu().numpy().astype(np.float64)
            np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-5 * np.max(np.abs(want)))


def test_index_topk_scores_output():
    B, Ncap, k = 1, 500, 32
    qI = datagen.normal_bf16(25, 5, (B, 1, 8, 64))
    w = datagen.uniform_f32(25, 6, (B, 1, 8))
    kI = datagen.normal_bf16(25, 7, (B, Ncap, 64))
    sc = torch.empty((B, 1, k), dtype=torch.float32, device=DEV)
    idx = lcc.lightning_index_topk(qI.to(DEV), w.to(DEV), 4 * Ncap, kI.to(DEV), Ncap, 4, k, score=sc)
    torch.cuda.synchronize()
    s = oracle.index_scores(f64(qI[0, 0]), f64(w[0, 0]), f64(kI[0]))
    ids = idx[0, 0].cpu().numpy()
    np.testing.assert_allclose(sc[0, 0].cpu().numpy(), s[ids], rtol=1e-5, atol=1e-5)


# ---------------------------------------------------------------------------
# NVFP4 quantiser and the FP4 indexer
# ---------------------------------------------------------------------------
def _nvfp4_quant_rows():
    """Groups of 16 that cover every finite bf16 value, every e4m3 scale with
    elements on and beside each e2m1 rounding midpoint, and random rows."""
    every = np.arange(65536, dtype=np.uint16)
    every = every[((every >> 7) & 0xFF) != 0xFF]                 # finite values only
    v = oracle.bf16_to_f64(every)
    groups = list(v[np.argsort(np.abs(v), kind="stable")].reshape(-1, 16))
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for c in range(1, 127):
        s = float(oracle.e4m3_value(c))
        vals = []
        for mu in mids:
            b = int(oracle.f64_to_bf16_bits(np.array([mu * s]))[0])
            vals += [mu * s, float(oracle.bf16_to_f64(np.array([b + 1]))[0]),
                     float(oracle.bf16_to_f64(np.array([b - 1]))[0])]
        vals += [-mu * s for mu in mids]
        groups.append(np.array([6.0 * s] + vals[:15]))
        groups.append(np.array([-6.0 * s] + vals[15:] + [0.0] * (30 - len(vals))))
    x = np.stack(groups).reshape(-1, 64)
    r = np.random.default_rng(31)
    rnd = r.standard_normal((256, 64)) * np.exp(r.uniform(-8, 8, size=(256, 1)))
    x = np.concatenate([x, oracle.round_bf16(rnd)])
    assert np.array_equal(oracle.round_bf16(x), x)
    return x


def test_nvfp4_quantize_bit_exact():
    x = _nvfp4_quant_rows()
    xt = torch.from_numpy(x).to(torch.bfloat16)
    packed, scale, xq = lcc.nvfp4_quantize(xt.to(DEV))
    torch.cuda.synchronize()
    want_p, want_s = oracle.nvfp4_quantize(x)
    assert np.array_equal(scale.cpu().numpy(), want_s)
    assert np.array_equal(packed.cpu().numpy(), want_p)
    want_xq = torch.from_numpy(oracle.nvfp4_decode(want_p, want_s)).to(torch.bfloat16)
    assert np.array_equal(bits(xq), bits(want_xq))
    # strided rows (ld = 96 elements), and the dequantiser on the codes
    big = torch.zeros((x.shape[0], 96), dtype=torch.bfloat16)
    big[:, :64] = xt
    p2, s2, _ = lcc.nvfp4_quantize(big.to(DEV)[:, :64])
    back = lcc.nvfp4_dequantize(p2, s2)
    torch.cuda.synchronize()
    assert torch.equal(p2.cpu(), packed.cpu()) and torch.equal(s2.cpu(), scale.cpu())
    assert np.array_equal(bits(back), bits(want_xq))


def test_nvfp4_dequantize_every_code_and_scale():
    codes = np.arange(256, dtype=np.uint8)
    scales = np.array([c for c in range(255) if c != 0x7F], dtype=np.uint8)    # not NaN
    packed = np.tile(codes, (scales.size, 1)).reshape(-1, 8)                   # 32 groups per scale
    sc = np.repeat(scales, 32)[:, None]
    out = lcc.nvfp4_dequantize(torch.from_numpy(packed).to(DEV), torch.from_numpy(sc).to(DEV))
    torch.cuda.synchronize()
    want = torch.from_numpy(oracle.nvfp4_decode(packed, sc)).to(torch.bfloat16)
    assert np.array_equal(bits(out), bits(want))


@pytest.mark.parametrize("B,Tq,Ncap,k,nv", [(2, 150, 3000, 64, [3000, 1700]),     # prefill: fused top-k
                                            (3, 1, 20000, 128, [20000, 9000, 77])])  # decode: NVFP4-key indexer
def test_fp4_index_topk_parity(B, Tq, Ncap, k, nv):
    seed, HI, DI, m = 41 + Tq, 8, 64, 4
    qI = datagen.normal_bf16(seed, 5, (B, Tq, HI, DI))
    w = datagen.uniform_f32(seed, 6, (B, Tq, HI))
    kp, ks = datagen.nvfp4_normal(seed, 7, B * Ncap, DI)
    kp, ks = kp.reshape(B, Ncap, DI // 2), ks.reshape(B, Ncap, DI // 16)
    pos0 = [m * Ncap - Tq] * B
    sc = torch.empty((B, Tq, k), dtype=torch.float32, device=DEV)
    idx = lcc.fp4_index_topk(qI.to(DEV), w.to(DEV), torch.tensor(pos0, device=DEV), kp.to(DEV), ks.to(DEV),
                             torch.tensor(nv, dtype=torch.int32, device=DEV), m, k, score=sc)
    torch.cuda.synchronize()
    lcc.sync_status()
    g, gs = idx.cpu().numpy(), sc.cpu().numpy()
    near, moved = 0, 0
    for b in range(B):
        rows = []
        for i in range(Tq):
            n = oracle.visible_count(pos0[b] + i, m, nv[b])
            s = oracle.index_scores_fp4(f64(qI[b, i]), f64(w[b, i]), kp[b, :n].numpy(), ks[b, :n].numpy())
            oi, kth = oracle.topk_select(s, k)
            rows.append(dict(idx=oi, scores=s, kth=kth))
            sel = g[b, i][g[b, i] >= 0]
            np.testing.assert_allclose(gs[b, i, :sel.size], s[sel], rtol=1e-5, atol=1e-5 * np.abs(s).max())
            # the query really was quantised: bf16-query scores differ
            plain = oracle.index_scores(f64(qI[b, i]), f64(w[b, i]), oracle.nvfp4_decode(kp[b, :n].numpy(),
                                                                                           ks[b, :n].numpy()))
            moved += int(np.abs(plain[sel] - s[sel]).max() > 1e-3 * np.abs(s).max())
        near += check_topk_rows(g[b], rows, k, what=f"batch {b}")
    assert near <= max(1, B * Tq // 100)
    assert moved == B * Tq


# ---------------------------------------------------------------------------
# attention branches
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("H,D,k", [(64, 128, 128), (8, 64, 16), (16, 128, 40), (128, 64, 70)])
def test_sparse_attn_parity(H, D, k):
    B, Tq, Ncap = 2, 5, 300
    q = datagen.normal_bf16(31, 4, (B, Tq, H, D), scale=D ** -0.5)
    Kc = datagen.normal_bf16(31, 8, (B, Ncap, D))
    Vc = datagen.normal_bf16(31, 9, (B, Ncap, D))
    vis = torch.tensor([Ncap, 3, 0, k, 200] * B)[: B * Tq]
    idx = datagen.random_index_lists(31, 17, vis, k).reshape(B, Tq, k)
    O, lse = lcc.csa_sparse_attn(q.to(DEV), Kc.to(DEV), Vc.to(DEV), idx.to(DEV))
    torch.cuda.synchronize()
    lcc.sync_status()
    for b in range(B):
        for i in range(Tq):
            sel = idx[b, i].numpy()
            sel = sel[sel >= 0]
            Oo, Lo = oracle.attend(f64(q[b, i]), f64(Kc[b])[sel], f64(Vc[b])[sel])
            assert_close(O[b, i].cpu().numpy(), Oo, f"O[{b},{i}]")
            assert_lse_close(lse[b, i].cpu().numpy(), Lo, f"lse[{b},{i}]")


def test_sparse_attn_gather_many_queries_parity():
    # 300 queries of 128 heads, 130 selected entries each (a ragged last key tile), lists with -1
    # padding and one-entry lists
    B, Tq, H, D, Ncap, k = 2, 150, 128, 128, 500, 130
    q = datagen.normal_bf16(38, 4, (B, Tq, H, D), scale=D ** -0.5)
    Kc = datagen.normal_bf16(38, 8, (B, Ncap, D))
    Vc = datagen.normal_bf16(38, 9, (B, Ncap, D))
    vis = torch.tensor(([Ncap, 3, k, 200, 129, 1] * (B * Tq))[: B * Tq])
    idx = datagen.random_index_lists(38, 17, vis, k).reshape(B, Tq, k)
    O, lse = lcc.csa_sparse_attn(q.to(DEV), Kc.to(DEV), Vc.to(DEV), idx.to(DEV))
    torch.cuda.synchronize()
    lcc.sync_status()
    for b in range(B):
        for i in range(Tq):
            sel = idx[b, i].numpy()
            sel = sel[sel >= 0]
            Oo, Lo = oracle.attend(f64(q[b, i]), f64(Kc[b])[sel], f64(Vc[b])[sel])
            assert_close(O[b, i].cpu().numpy(), Oo, f"O[{b},{i}]")
            assert_lse_close(lse[b, i].cpu().numpy(), Lo, f"lse[{b},{i}]")


def test_sparse_attn_rejects_out_of_range_index():
    B, Tq, H, D, Ncap, k = 1, 1, 64, 128, 50, 8
    q = torch.zeros((B, Tq, H, D), dtype=torch.bfloat16, device=DEV)
    Kc = torch.zeros((B, Ncap, D), dtype=torch.bfloat16, device=DEV)
    idx = torch.tensor([[[0, 1, 2, 77, -1, -1, -1, -1]]], dtype=torch.int32, device=DEV)
    lcc.csa_sparse_attn(q, Kc, Kc, idx)
    with pytest.raises(lcc.LccError) as e:
        lcc.sync_status()
    assert e.value.status == 7
    lcc.sync_status()  # the error word is cleared once reported


@pytest.mark.parametrize("m,H,D", [(4, 8, 64), (128, 64, 128)])
def test_dense_attn_prefill_parity(m, H, D):
    T = 4 * m + 9
    q = datagen.normal_bf16(32, 4, (1, T, H, D), scale=D ** -0.5)
    K = datagen.normal_bf16(32, 1, (1, T, D))
    V = datagen.normal_bf16(32, 2, (1, T, D))
    g = datagen.normal_f32(32, 3, (1, T))
    n = T // m
    Kc = torch.zeros((1, n, D), dtype=torch.bfloat16, device=DEV)
    Vc = torch.zeros_like(Kc)
    (lcc.csa_compress if m == 4 else lcc.hca_compress)(K.to(DEV), V.to(DEV), g.to(DEV), Kc, Vc)
    O, lse = lcc.hca_dense_attn(q.to(DEV), Kc, Vc, 0, n, m)
    torch.cuda.synchronize()
    Kh, Vh = f64(Kc[0]), f64(Vc[0])   # attention parity on the kernel's own pooled entries is
    Ko, Vo = oracle.pool(f64(K[0]), f64(V[0]), f64(g[0]), m)   # ... checked against the oracle's pooling too
    assert np.max(np.abs(Kh - Ko)) <= 2 ** -6 * max(1.0, np.max(np.abs(Ko)))
    for t in range(T):
        r = runs.hca_branch(f64(q[0, t]), t, Ko, Vo, m)
        assert_close(O[0, t].cpu().numpy(), r["O"], f"O[{t}]")
        assert_lse_close(lse[0, t].cpu().numpy(), r["lse"], f"lse[{t}]")


def test_dense_attn_decode_split_ragged():
    B, H, D, Ncap, m = 3, 64, 128, 1000, 128
    q = datagen.normal_bf16(33, 4, (B, 1, H, D), scale=D ** -0.5)
    Kc = datagen.normal_bf16(33, 8, (B, Ncap, D))
    Vc = datagen.normal_bf16(33, 9, (B, Ncap, D))
    n_valid = [Ncap, 37, 0]
    pos = m * Ncap + 5
    O, lse = lcc.hca_dense_attn(q.to(DEV), Kc.to(DEV), Vc.to(DEV), pos,
                                torch.tensor(n_valid, dtype=torch.int32, device=DEV), m)
    torch.cuda.synchronize()
    for b in range(B):
        r = runs.hca_branch(f64(q[b, 0]), pos, f64(Kc[b]), f64(Vc[b]), m, n_valid=n_valid[b])
        assert_close(O[b, 0].cpu().numpy(), r["O"], f"O[{b}]")
        assert_lse_close(lse[b, 0].cpu().numpy(), r["lse"], f"lse[{b}]")


@pytest.mark.parametrize("W,H,D", [(32, 8, 64), (128, 64, 128), (100, 16, 128)])
def test_swa_prefill_parity(W, H, D):
    T = 300
    q = datagen.normal_bf16(34, 4, (1, T, H, D), scale=D ** -0.5)
    K = datagen.normal_bf16(34, 1, (1, T, D))
    V = datagen.normal_bf16(34, 2, (1, T, D))
    O, lse = lcc.swa_attn(q.to(DEV), K.to(DEV), V.to(DEV), 0, 0, W)
    torch.cuda.synchronize()
    for t in range(T):
        r = runs.swa_branch(f64(q[0, t]), t, f64(K[0]), f64(V[0]), 0, W)
        assert_close(O[0, t].cpu().numpy(), r["O"], f"O[{t}]")
        assert_lse_close(lse[0, t].cpu().numpy(), r["lse"], f"lse[{t}]")


def test_swa_decode_buffer_offsets():
    # raw buffers that start after position 0 and hold only part of some windows
    B, H, D, W, R = 3, 64, 128, 128, 150
    q = datagen.normal_bf16(35, 4, (B, 2, H, D), scale=D ** -0.5)
    Kr = datagen.normal_bf16(35, 1, (B, R, D))
    Vr = datagen.normal_bf16(35, 2, (B, R, D))
    raw0 = [1000, 1060, 900]
    qpos = [1000 + 127, 1100, 900 + 149 - 1]
    O, lse = lcc.swa_attn(q.to(DEV), Kr.to(DEV), Vr.to(DEV), torch.tensor(qpos, device=DEV),
                          torch.tensor(raw0, device=DEV), W)
    torch.cuda.synchronize()
    for b in range(B):
        for i in range(2):
            r = runs.swa_branch(f64(q[b, i]), qpos[b] + i, f64(Kr[b]), f64(Vr[b]), raw0[b], W)
            assert_close(O[b, i].cpu().numpy(), r["O"], f"O[{b},{i}]")
            assert_lse_close(lse[b, i].cpu().numpy(), r["lse"], f"lse[{b},{i}]")


@pytest.mark.parametrize("nb,D", [(2, 128), (3, 64), (4, 128)])
def test_merge_parity(nb, D):
    rows = 777
    parts = []
    for p in range(nb):
        O = torch.randn((rows, D), generator=torch.Generator().manual_seed(p), dtype=torch.float32)
        L = torch.randn((rows,), generator=torch.Generator().manual_seed(100 + p), dtype=torch.float32) * 3
        L[p::nb] = -float("inf")     # empty branches
        parts.append((O, L))
    L_all_empty = list(range(0, rows, 97))
    for p in range(nb):
        parts[p][1][L_all_empty] = -float("inf")
    out_f32 = torch.empty((rows, D), dtype=torch.float32, device=DEV)
    lse_out = torch.empty((rows,), dtype=torch.float32, device=DEV)
    out = lcc.attn_merge([(o.to(DEV), l.to(DEV)) for o, l in parts], out_f32=out_f32, lse_out=lse_out)
    torch.cuda.synchronize()
    Oo, Lo = oracle.merge([o.double().numpy() for o, _ in parts],
                          [l.double().numpy() for _, l in parts])
    assert_close(out_f32.cpu().numpy(), Oo, "merge f32", max_abs=1e-5, mean_abs=1e-6)
    assert_close(out.float().cpu().numpy(), Oo, "merge bf16")
    assert_lse_close(lse_out.cpu().numpy(), Lo, "merge lse", tol=1e-5)
    assert np.all(out_f32.cpu().numpy()[L_all_empty] == 0)


# ---------------------------------------------------------------------------
# whole layers in one pass: compressed keys ++ window keys, one softmax
# ---------------------------------------------------------------------------
# the first three run the warp-split kernels (short key lists; with D = 128 the selected entries
# arrive by TMA gather4, including empty lists and a ragged k = 70); the last is long enough for
# the split-across-CTAs path with its combine kernel
@pytest.mark.parametrize("B,Tq,H,D,k,W,Ncap", [(3, 1, 64, 128, 128, 128, 400), (2, 40, 8, 64, 16, 32, 400),
                                               (1, 7, 16, 128, 70, 100, 400), (2, 1, 64, 128, 1000, 128, 1500)])
def test_csa_layer_attn_parity(B, Tq, H, D, k, W, Ncap):
    R = 160
    q = datagen.normal_bf16(36, 4, (B, Tq, H, D), scale=D ** -0.5)
    Kc = datagen.normal_bf16(36, 8, (B, Ncap, D))
    Vc = datagen.normal_bf16(36, 9, (B, Ncap, D))
    Kr = datagen.normal_bf16(36, 1, (B, R, D))
    Vr = datagen.normal_bf16(36, 2, (B, R, D))
    vis = torch.tensor(([Ncap, 3, 0, k, 200] * (B * Tq))[: B * Tq])
    idx = datagen.random_index_lists(36, 17, vis, k).reshape(B, Tq, k)
    raw0 = [500 + 30 * b for b in range(B)]
    qpos = [raw0[b] + R - Tq - 5 * b for b in range(B)]
    lse = torch.empty((B, Tq, H), dtype=torch.float32, device=DEV)
    out = lcc.csa_layer_attn(q.to(DEV), Kc.to(DEV), Vc.to(DEV), idx.to(DEV), Kr.to(DEV), Vr.to(DEV),
                             torch.tensor(qpos, device=DEV), torch.tensor(raw0, device=DEV), W, lse_out=lse)
    lcc.sync_status()
    for b in range(B):
        for i in range(Tq):
            sel = idx[b, i].numpy()
            sel = sel[sel >= 0]
            cO, cL = oracle.attend(f64(q[b, i]), f64(Kc[b])[sel], f64(Vc[b])[sel])
            sw = runs.swa_branch(f64(q[b, i]), qpos[b] + i, f64(Kr[b]), f64(Vr[b]), raw0[b], W)
            O, L = oracle.merge([cO, sw["O"]], [cL, sw["lse"]])
            assert_close(out[b, i].float().cpu().numpy(), O, f"CSA layer [{b},{i}]")
            assert_lse_close(lse[b, i].cpu().numpy(), L, f"CSA layer lse [{b},{i}]")


def test_csa_layer_attn_prefill_parity():
    # a prefill-shaped CSA layer: 301 consecutive queries of 64 heads, 200 selected entries each
    # (empty, short and full lists) plus the 128-token window of every query
    B, Tq, H, D, k, W, Ncap = 1, 301, 64, 128, 200, 128, 2000
    R = Tq + W - 1
    q = datagen.normal_bf16(39, 4, (B, Tq, H, D), scale=D ** -0.5)
    Kc = datagen.normal_bf16(39, 8, (B, Ncap, D))
    Vc = datagen.normal_bf16(39, 9, (B, Ncap, D))
    Kr = datagen.normal_bf16(39, 1, (B, R, D))
    Vr = datagen.normal_bf16(39, 2, (B, R, D))
    vis = torch.tensor(([Ncap, 3, 0, k, 1500, 129] * (B * Tq))[: B * Tq])
    idx = datagen.random_index_lists(39, 17, vis, k).reshape(B, Tq, k)
    raw0, qpos = 10000, 10000 + W - 1
    lse = torch.empty((B, Tq, H), dtype=torch.float32, device=DEV)
    out = lcc.csa_layer_attn(q.to(DEV), Kc.to(DEV), Vc.to(DEV), idx.to(DEV), Kr.to(DEV), Vr.to(DEV),
                             torch.tensor([qpos], device=DEV), torch.tensor([raw0], device=DEV), W, lse_out=lse)
    lcc.sync_status()
    for i in range(Tq):
        sel = idx[0, i].numpy()
        sel = sel[sel >= 0]
        cO, cL = oracle.attend(f64(q[0, i]), f64(Kc[0])[sel], f64(Vc[0])[sel])
        sw = runs.swa_branch(f64(q[0, i]), qpos + i, f64(Kr[0]), f64(Vr[0]), raw0, W)
        O, L = oracle.merge([cO, sw["O"]], [cL, sw["lse"]])
        assert_close(out[0, i].float().cpu().numpy(), O, f"CSA layer [{i}]")
        assert_lse_close(lse[0, i].cpu().numpy(), L, f"CSA layer lse [{i}]")


# warp-split kernel for the short lists; 3000 entries take the split-across-CTAs path; 2000 prefill
# queries fill enough CTAs for the single-pass kernel that writes bf16 directly
# 8 decode sequences of 2000 entries + window (ragged visible counts): the tensor-core split-KV path
@pytest.mark.parametrize("B,Tq,H,D,m,W,Ncap", [(3, 1, 64, 128, 128, 128, 700), (1, 300, 8, 64, 4, 32, 700),
                                               (2, 9, 64, 128, 4, 128, 700), (3, 1, 64, 128, 128, 128, 3000),
                                               (1, 2000, 64, 128, 4, 128, 600), (8, 1, 64, 128, 128, 128, 2000)])
def test_hca_layer_attn_parity(B, Tq, H, D, m, W, Ncap):
    R = 300 if Tq < 300 else Tq
    q = datagen.normal_bf16(37, 4, (B, Tq, H, D), scale=D ** -0.5)
    Kc = datagen.normal_bf16(37, 8, (B, Ncap, D))
    Vc = datagen.normal_bf16(37, 9, (B, Ncap, D))
    Kr = datagen.normal_bf16(37, 1, (B, R, D))
    Vr = datagen.normal_bf16(37, 2, (B, R, D))
    n_valid = ([Ncap, 37, 0] * B)[:B] if Tq == 1 else [Ncap] * B
    # decode: queries far into the context; prefill: the raw buffer starts at 0 and queries at 0
    qpos = [m * Ncap + 5] * B if Tq == 1 else [0] * B
    raw0 = [qpos[b] + Tq - R + 3 for b in range(B)] if Tq == 1 else [0] * B
    lse = torch.empty((B, Tq, H), dtype=torch.float32, device=DEV)
    out = lcc.hca_layer_attn(q.to(DEV), Kc.to(DEV), Vc.to(DEV),
                             torch.tensor(n_valid, dtype=torch.int32, device=DEV), m, Kr.to(DEV), Vr.to(DEV),
                             torch.tensor(qpos, device=DEV), torch.tensor(raw0, device=DEV), W, lse_out=lse)
    lcc.sync_status()
    rows = range(Tq) if Tq <= 300 else sorted(set(range(0, Tq, 7)) | {Tq - 1})
    for b in range(B):
        for i in rows:
            t = qpos[b] + i
            h = runs.hca_branch(f64(q[b, i]), t, f64(Kc[b]), f64(Vc[b]), m, n_valid=n_valid[b])
            sw = runs.swa_branch(f64(q[b, i]), t, f64(Kr[b]), f64(Vr[b]), raw0[b], W)
            O, L = oracle.merge([h["O"], sw["O"]], [h["lse"], sw["lse"]])
            assert_close(out[b, i].float().cpu().numpy(), O, f"HCA layer [{b},{i}]")
            assert_lse_close(lse[b, i].cpu().numpy(), L, f"HCA layer lse [{b},{i}]")


@pytest.mark.parametrize("DI,k", [(64, 200), (32, 128), (64, 240)])
def test_index_topk_prefill_fused_parity(DI, k):
    # prefill-shaped calls with 8 indexer heads: k up to 224 uses warp-private candidate buffers per
    # (query, lane quadrant), larger k the shared per-query buffers; 301 queries leave a ragged
    # last group, and the visible counts grow along the chunk
    near, g = _index_case(27, 1, 301, 8, DI, 3000, 4, k, q_pos0=[8000], n_valid=[3000])
    assert near <= 2


@pytest.mark.parametrize("Ncap,Tq,q0,k", [(20000, 200, 4 * 20000 - 200, 128), (2000, 800, 0, 128),
                                           (30000, 48, 4 * 30000 - 48, 1), (6000, 100, 4 * 6000 - 100, 16)])
def test_index_topk_prefill_passes_parity(Ncap, Tq, q0, k):
    # the prefill top-k fused into the indexer (8 heads): long rows; a causal block from
    # position 0 (empty rows, rows below k, short rows); k = 1; a short k
    near, g = _index_case(28, 1, Tq, 8, 64, Ncap, 4, k, q_pos0=[q0], n_valid=[Ncap])
    assert near <= 2


@pytest.mark.parametrize("k", [128, 224])
def test_index_topk_prefill_fused_signed_weights(k):
    # head weights of both signs (scores below zero, keys on both sides of +0) and the largest k the
    # fused kernel's warp-private buffers take; rows long enough for every buffer cut and the
    # shared bound of the quadrant warps
    B, Tq, HI, DI, Ncap, m = 1, 200, 8, 64, 6000, 4
    qI = datagen.normal_bf16(33, 5, (B, Tq, HI, DI))
    w = datagen.uniform_f32(33, 6, (B, Tq, HI)) * 2.0 - 1.0
    kI = datagen.normal_bf16(33, 7, (B, Ncap, DI))
    q0 = m * Ncap - Tq
    sc = torch.empty((B, Tq, k), dtype=torch.float32, device=DEV)
    idx = lcc.lightning_index_topk(qI.to(DEV), w.to(DEV), q0, kI.to(DEV), Ncap, m, k, score=sc)
    torch.cuda.synchronize()
    lcc.sync_status()
    g, gs = idx.cpu().numpy()[0], sc.cpu().numpy()[0]
    rows = []
    for i in range(Tq):
        vis = min(Ncap, (q0 + i + 1) // m)
        s = oracle.index_scores(f64(qI[0, i]), f64(w[0, i]), f64(kI[0, :vis]))
        oi, kth = oracle.topk_select(s, k)
        rows.append(dict(idx=oi, scores=s, kth=kth))
        sel = g[i][g[i] >= 0]
        np.testing.assert_allclose(gs[i, :sel.size], s[sel], rtol=1e-5, atol=1e-5 * np.abs(s).max())
    assert min(float(r["scores"].min()) for r in rows) < 0, "the case must hold negative scores"
    assert check_topk_rows(g, rows, k) <= 2


def test_index_topk_prefill_passes_integer_score_ties():
    # scores that are small integers (binary keys, one head): thousands of exact ties around the
    # k-th score (candidate buffers fill with equal keys); the result must be bit-exact
    B, Tq, HI, DI, Ncap, k = 1, 64, 8, 64, 12000, 100
    qI = torch.ones((B, Tq, HI, DI), dtype=torch.bfloat16)
    w = torch.zeros((B, Tq, HI), dtype=torch.float32)
    w[..., 0] = 1.0
    bits01 = (datagen.uniform_f32(29, 1, (B, Ncap, DI)) < 0.3).to(torch.bfloat16)
    q0 = 4 * Ncap - Tq
    idx = lcc.lightning_index_topk(qI.to(DEV), w.to(DEV), q0, bits01.to(DEV), Ncap, 4, k)
    torch.cuda.synchronize()
    g = idx.cpu().numpy()[0]
    kI = f64(bits01[0])
    for i in range(Tq):
        vis = min(Ncap, (q0 + i + 1) // 4)
        sc = oracle.index_scores(f64(qI[0, i]), host(w[0, i]).astype(np.float64), kI[:vis])
        want, _ = oracle.topk_select(sc, k)
        assert np.array_equal(g[i], want), f"row {i}"


@pytest.mark.parametrize("Ncap", [16384, 20000, 300000])
def test_index_topk_decode_integer_score_ties(Ncap):
    # decode rows (one query per sequence) whose scores are small integers (binary keys, one
    # head): hundreds of exact ties at the k-th score.  16384 entries take the cluster top-k,
    # 20000 and 300000 the group-selected one (partition maxima for its threshold); the
    # candidate lists exceed one per thread, so the histogram selections run too
    B, HI, DI, k = 2, 8, 64, 128
    qI = torch.ones((B, 1, HI, DI), dtype=torch.bfloat16)
    w = torch.zeros((B, 1, HI), dtype=torch.float32)
    w[..., 0] = 1.0
    dens = torch.tensor([0.3, 0.5]).view(B, 1, 1)
    bits01 = (datagen.uniform_f32(30, 1, (B, Ncap, DI)) < dens).to(torch.bfloat16)
    pos = [4 * Ncap - 1, 4 * Ncap - 1]
    nval = [Ncap, Ncap - 77]
    idx = lcc.lightning_index_topk(qI.to(DEV), w.to(DEV), torch.tensor(pos, device=DEV), bits01.to(DEV),
                                   torch.tensor(nval, dtype=torch.int32, device=DEV), 4, k)
    torch.cuda.synchronize()
    lcc.sync_status()
    g = idx.cpu().numpy()
    for b in range(B):
        vis = oracle.visible_count(pos[b], 4, nval[b])
        sc = oracle.index_scores(f64(qI[b, 0]), host(w[b, 0]).astype(np.float64), f64(bits01[b, :vis]))
        want, kth = oracle.topk_select(sc, k)
        assert np.sum(sc == kth) > 1, "the case must tie at the k-th score"
        assert np.array_equal(g[b, 0], want), f"batch {b}"


def test_index_topk_prefill_fused_zero_score_ties():
    # prefill-shaped calls keep a running top-k inside the indexer; with zero weights every score
    # ties, so each query must keep its lowest visible indices (candidate buffers compact often)
    B, Tq, HI, DI, Ncap, k, m = 1, 300, 8, 64, 1000, 64, 4
    qI = datagen.normal_bf16(26, 5, (B, Tq, HI, DI)).to(DEV)
    w = torch.zeros((B, Tq, HI), dtype=torch.float32, device=DEV)
    kI = datagen.normal_bf16(26, 7, (B, Ncap, DI)).to(DEV)
    q0 = 3000
    idx = lcc.lightning_index_topk(qI, w, q0, kI, Ncap, m, k)
    torch.cuda.synchronize()
    g = idx.cpu().numpy()[0]
    for i in range(Tq):
        vis = min(Ncap, (q0 + i + 1) // m)
        want = np.arange(min(vis, k))
        assert np.array_equal(g[i, :len(want)], want) and np.all(g[i, len(want):] == -1), f"row {i}"


# ---------------------------------------------------------------------------
# CSA2 re-index mode (lcc_lightning_reindex_topk)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("HI,DI,fp4,n_notes,k", [(8, 64, False, 512, 128), (4, 32, False, 300, 64),
                                                 (8, 64, True, 1024, 128), (8, 64, False, 200, 200)])
def test_reindex_topk_parity(HI, DI, fp4, n_notes, k):
    B, Tq, N = 3, 4, 5000
    qI0 = datagen.normal_bf16(17, 1, (B, Tq, HI, DI)).to(DEV)
    w0 = datagen.uniform_f32(17, 2, (B, Tq, HI)).to(DEV)
    qI1 = datagen.normal_bf16(17, 3, (B, Tq, HI, DI)).to(DEV)
    w1 = datagen.uniform_f32(17, 4, (B, Tq, HI)).to(DEV)
    if fp4:
        kp, ks = datagen.nvfp4_normal(17, 5, B * N, DI)
        kI, kIs = kp.reshape(B, N, DI // 2).to(DEV), ks.reshape(B, N, DI // 16).to(DEV)
        keys = [oracle.nvfp4_decode(host(kI[b]), host(kIs[b])) for b in range(B)]
    else:
        kI, kIs = datagen.normal_bf16(17, 5, (B, N, DI)).to(DEV), None
        keys = [f64(kI[b]) for b in range(B)]
    # the full layer's notes: its n_notes best entries (the last query sees only 1200 entries)
    pos = torch.tensor([4 * N - Tq, 4 * N - Tq, 4 * 1200 - Tq], dtype=torch.int64, device=DEV)
    notes = lcc.lightning_index_topk(qI0, w0, pos, kI, N, 4, n_notes, kI_scale=kIs)
    sc = torch.empty((B, Tq, k), dtype=torch.float32, device=DEV)
    idx = lcc.lightning_reindex_topk(qI1, w1, kI, notes, k, kI_scale=kIs, score=sc)
    lcc.sync_status()
    gi, gn, gs = host(idx), host(notes), host(sc)
    near = 0
    for b in range(B):
        for i in range(Tq):
            cand = gn[b, i][gn[b, i] >= 0]
            s_c = oracle.index_scores(f64(qI1[b, i]), host(w1[b, i]).astype(np.float64), keys[b][cand])
            pick, kth = oracle.topk_select(s_c, k)
            want = np.full(k, -1, dtype=np.int64)
            want[:np.sum(pick >= 0)] = np.sort(cand[pick[pick >= 0]])
            full = np.full(int(cand.max()) + 1 if cand.size else 1, -np.inf)
            full[cand] = s_c                                  # scores by entry number for the tie rule
            ok, exact = topk_set_ok(gi[b, i], want, full, kth, k)
            assert ok, f"b={b} i={i}: re-index set differs"
            near += not exact
            got = gi[b, i][gi[b, i] >= 0]
            np.testing.assert_allclose(gs[b, i][:got.size], full[got], rtol=2e-5, atol=2e-5)
            assert np.all(gs[b, i][got.size:] == -np.inf)
    assert near <= 1


def test_reindex_topk_ties_and_short_lists():
    # all-zero scores: every candidate ties, the lowest entry numbers win; a list
    # shorter than k is kept whole and padded
    B, Tq, N, HI, DI, k = 1, 2, 900, 8, 64, 16
    qI = torch.zeros((B, Tq, HI, DI), dtype=torch.bfloat16, device=DEV)
    w = torch.ones((B, Tq, HI), dtype=torch.float32, device=DEV)
    kI = datagen.normal_bf16(18, 1, (B, N, DI)).to(DEV)
    cand = torch.full((B, Tq, 40), -1, dtype=torch.int32, device=DEV)
    cand[0, 0, :40] = torch.arange(100, 900, 20, dtype=torch.int32)
    cand[0, 1, :7] = torch.tensor([3, 9, 10, 500, 501, 502, 899], dtype=torch.int32)
    idx = lcc.lightning_reindex_topk(qI, w, kI, cand, k)
    lcc.sync_status()
    assert idx[0, 0].tolist() == list(range(100, 100 + 20 * k, 20))
    assert idx[0, 1].tolist() == [3, 9, 10, 500, 501, 502, 899] + [-1] * (k - 7)


# ---------------------------------------------------------------------------
# query / KV prologue (RMSNorm + partial RoPE)
# ---------------------------------------------------------------------------
def _within_one_ulp(gpu_bf16, exact, what):
    """One bf16 ulp of the fp64 value, plus the fp32 arithmetic's own error on the
    row's scale (a rotated channel can cancel to near zero)."""
    g = f64(gpu_bf16)
    ulp = np.ldexp(1.0, np.frexp(np.abs(exact))[1] - 8)
    fp32 = 2.0 ** -20 * np.max(np.abs(exact), axis=-1, keepdims=True)
    bad = np.abs(g - exact) > ulp + fp32
    assert not bad.any(), f"{what}: {bad.sum()} elements more than one bf16 ulp from the fp64 value"


@pytest.mark.parametrize("H,D,d_rope,with_v", [(64, 128, 64, True), (8, 64, 32, True), (5, 128, 128, False),
                                                (16, 128, 0, True)])
def test_qkv_prologue_parity(H, D, d_rope, with_v):
    B, T = 2, 37
    q = datagen.normal_bf16(15, 1, (B, T, H, D), 3.0)
    k = datagen.normal_bf16(15, 2, (B, T, D))
    v = datagen.normal_bf16(15, 3, (B, T, D), 0.5)
    gq, gk, gv = (1.0 + 0.1 * datagen.normal_f32(15, 4 + i, (D,)) for i in range(3))
    pos0 = torch.tensor([0, 1048576 - 5], dtype=torch.int64)
    qo, ko, vo = lcc.qkv_prologue(q.to(DEV), k.to(DEV), v.to(DEV) if with_v else None, gq.to(DEV), gk.to(DEV),
                                  gv.to(DEV) if with_v else None, pos0.to(DEV), d_rope=d_rope)
    torch.cuda.synchronize()
    qh, kh, vh = f64(q), f64(k), f64(v)
    for b in range(B):
        for t in range(T):
            p = int(pos0[b]) + t
            eq, ek, ev = oracle.qkv_prologue(qh[b, t], kh[b, t], vh[b, t], p, f64(gq), f64(gk), f64(gv), 1e-6,
                                             d_rope)
            _within_one_ulp(qo[b, t], eq, f"q b={b} t={t}")
            _within_one_ulp(ko[b, t], ek, f"k b={b} t={t}")
            if with_v:
                _within_one_ulp(vo[b, t], ev, f"v b={b} t={t}")
    assert vo is None or with_v


def test_qkv_prologue_in_place():
    B, T, H, D = 1, 300, 64, 128
    q = datagen.normal_bf16(16, 1, (B, T, H, D)).to(DEV)
    k = datagen.normal_bf16(16, 2, (B, T, D)).to(DEV)
    g = torch.ones(D, dtype=torch.float32, device=DEV)
    want = lcc.qkv_prologue(q, k, None, g, g, None, 1000)
    lcc.qkv_prologue(q, k, None, g, g, None, 1000, q_out=q, k_out=k)
    torch.cuda.synchronize()
    assert torch.equal(q, want[0]) and torch.equal(k, want[1])


# ---------------------------------------------------------------------------
# decode-step update of a layer's caches (lcc_decode_append)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("m,D", [(4, 128), (4, 64), (128, 128), (1, 128)])
def test_decode_append_parity(m, D):
    # three sequences at different positions, raw buffers that begin with the
    # context rows only; enough steps that every sequence completes blocks
    B, W, steps, DI = 3, 8 if m < 128 else 130, 2 * m + 5, 64
    R = W + steps
    ctx = [m * 50, m * 50 + 1, m * 50 + m - 1]                 # block boundary, just past it, just before it
    Kfull = datagen.normal_bf16(13, 1, (B, R, D))
    Vfull = datagen.normal_bf16(13, 2, (B, R, D))
    gfull = datagen.normal_f32(13, 3, (B, R))
    kI_tok = datagen.normal_bf16(13, 4, (steps, B, DI))        # indexer key offered with each new token
    Kr = torch.zeros((B, R, D), dtype=torch.bfloat16, device=DEV)
    Vr = torch.zeros_like(Kr)
    gr = torch.zeros((B, R), dtype=torch.float32, device=DEV)
    Kr[:, :W], Vr[:, :W], gr[:, :W] = Kfull[:, :W].to(DEV), Vfull[:, :W].to(DEV), gfull[:, :W].to(DEV)
    Ncap = max(ctx) // m + steps // m + 2
    Kc = torch.full((B, Ncap, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    Vc = torch.full_like(Kc, float("nan"))
    kI = torch.zeros((B, Ncap, DI), dtype=torch.bfloat16, device=DEV)
    n_valid = torch.tensor([c // m for c in ctx], dtype=torch.int32, device=DEV)
    raw0 = torch.tensor([c - W for c in ctx], dtype=torch.int64, device=DEV)
    pos = raw0 + W
    for s in range(steps):
        lcc.decode_append(m, Kfull[:, W + s].contiguous().to(DEV), Vfull[:, W + s].contiguous().to(DEV),
                          gfull[:, W + s].contiguous().to(DEV), pos, Kr, Vr, gr, raw0, Kc, Vc, n_valid,
                          kI_new=kI_tok[s].to(DEV), kI=kI)
        pos += 1
    lcc.sync_status()
    # raw buffers now hold every token, bit for bit
    assert torch.equal(Kr.cpu(), Kfull) and torch.equal(Vr.cpu(), Vfull) and torch.equal(gr.cpu(), gfull)
    for b in range(B):
        first = ctx[b] // m                                      # the block under way at ctx completes first
        last = (ctx[b] + steps) // m                             # one past the last completed block
        assert int(n_valid[b]) == last
        # each completed block: the oracle's pooled entry over its raw rows
        for j in range(first, last):
            r0 = j * m - int(raw0[b])
            ex_k, ex_v = oracle.pool_exact(f64(Kfull[b, r0:r0 + m]), f64(Vfull[b, r0:r0 + m]),
                                           f64(gfull[b, r0:r0 + m]), m)
            for gpu, ex in ((Kc[b, j], ex_k[0]), (Vc[b, j], ex_v[0])):
                ulp = np.ldexp(1.0, np.frexp(np.abs(ex))[1] - 8)
                assert np.all(np.abs(f64(gpu) - ex) <= ulp)
            s_done = (j + 1) * m - 1 - ctx[b]                    # the step whose token completed block j
            assert torch.equal(kI[b, j].cpu(), kI_tok[s_done, b])
        assert torch.isnan(Kc[b, last:].float()).all() and torch.isnan(Kc[b, :first].float()).all()
    # the pooled entries equal what the compression call writes for the same rows
    for b in range(B):
        r0 = (ctx[b] // m) * m - int(raw0[b])
        n = (ctx[b] + steps) // m - ctx[b] // m
        Kc2 = torch.empty((1, n, D), dtype=torch.bfloat16, device=DEV)
        Vc2 = torch.empty_like(Kc2)
        if m in (4, 128):
            fn = lcc.csa_compress if m == 4 else lcc.hca_compress
            fn(Kr[b:b + 1, r0:r0 + n * m], Vr[b:b + 1, r0:r0 + n * m], gr[b:b + 1, r0:r0 + n * m], Kc2, Vc2)
            torch.cuda.synchronize()
            assert torch.equal(Kc2[0], Kc[b, ctx[b] // m:ctx[b] // m + n])
            assert torch.equal(Vc2[0], Vc[b, ctx[b] // m:ctx[b] // m + n])
        else:  # m = 1: an entry is its token
            assert torch.equal(Kc[b, ctx[b]:ctx[b] + n].cpu(), Kfull[b, r0:r0 + n])


def test_decode_append_out_of_range_is_reported():
    B, R, D, m = 2, 16, 128, 4
    Kr = torch.zeros((B, R, D), dtype=torch.bfloat16, device=DEV)
    Vr = torch.zeros_like(Kr)
    gr = torch.zeros((B, R), dtype=torch.float32, device=DEV)
    Kc = torch.zeros((B, 8, D), dtype=torch.bfloat16, device=DEV)
    Vc = torch.zeros_like(Kc)
    n_valid = torch.zeros(B, dtype=torch.int32, device=DEV)
    kn = torch.ones((B, D), dtype=torch.bfloat16, device=DEV)
    gn = torch.zeros(B, dtype=torch.float32, device=DEV)
    raw0 = torch.zeros(B, dtype=torch.int64, device=DEV)
    pos = torch.tensor([3, R], dtype=torch.int64, device=DEV)   # sequence 1 is past its raw buffer
    lcc.decode_append(m, kn, kn, gn, pos, Kr, Vr, gr, raw0, Kc, Vc, n_valid)
    with pytest.raises(lcc.LccError) as e:
        lcc.sync_status()
    assert e.value.status == 7 and "decode append" in str(e.value)
    assert int(n_valid[0]) == 1 and int(n_valid[1]) == 0       # sequence 0 still completed its block
    assert torch.equal(Kr[0, 3].cpu(), kn[0].cpu()) and float(Kr[1].float().abs().sum()) == 0.0


# ---------------------------------------------------------------------------
# bounded device waits: a wait that nothing completes runs out, the kernel
# winds down (drains its own copies and MMAs, frees TMEM) and the host reads
# LCC_ERR_TIMEOUT; the context stays usable and the next call is correct
# ---------------------------------------------------------------------------
def test_bounded_wait_runs_out_and_context_survives():
    B, N, HI, DI = 32, 16384, 8, 64          # 14 key-range splits of 10 tiles per sequence
    qI = datagen.normal_bf16(61, 5, (B, 1, HI, DI)).to(DEV)
    w = datagen.uniform_f32(61, 6, (B, 1, HI)).to(DEV)
    kI = datagen.normal_bf16(61, 7, (B, N, DI)).to(DEV)
    pos = torch.full((B,), 4 * N - 1, dtype=torch.int64, device=DEV)
    nval = torch.full((B,), N, dtype=torch.int32, device=DEV)
    ref = lcc.lightning_index_scores(qI, w, pos, kI, nval, 4)
    lcc.sync_status()
    try:
        # 20 ms waits; every CTA skips its second key tile
        lcc.test_set_wait_fault(20_000_000, 1)
        lcc.lightning_index_scores(qI, w, pos, kI, nval, 4)
        with pytest.raises(lcc.LccError) as e:
            lcc.sync_status()
        assert e.value.status == 6 and "gave up" in str(e.value)
    finally:
        lcc.test_set_wait_fault(0, -1)
    again = lcc.lightning_index_scores(qI, w, pos, kI, nval, 4)
    lcc.sync_status()
    assert torch.equal(again, ref)
    sc = oracle.index_scores(runs.f64(host(qI[0, 0])), host(w[0, 0]).astype(np.float64), runs.f64(host(kI[0])))
    np.testing.assert_allclose(again[0, 0].cpu().numpy(), sc, rtol=1e-4, atol=1e-4)


# ---------------------------------------------------------------------------
# CSA layer, decode-shaped: top-k and attention in one cluster per query
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("H,B,Tq,Ncap,k,nval,nvfp4", [
    (64, 3, 2, 16384, 128, [16384, 300, 50], False),   # 4 CTAs per query; rows above, near and below k
    (16, 2, 1, 4000, 64, [4000, 1000], False),         # one CTA per query
    (128, 2, 1, 10000, 128, [10000, 129], True),       # 8 CTAs per query, NVFP4 indexer keys
])
def test_csa_layer_decode_one_cluster_per_query(H, B, Tq, Ncap, k, nval, nvfp4):
    # the whole layer call against the two-call composition (index + top-k, then the layer
    # attention over that list): the same index lists and outputs equal up to rounding; and
    # the layer call against the oracle on every row
    D, W, HI, DI, m = 128, 128, 8, 64, 4
    seed = 40 + H
    q = datagen.normal_bf16(seed, 1, (B, Tq, H, D), 1.0 / np.sqrt(D))
    qI = datagen.normal_bf16(seed, 2, (B, Tq, HI, DI))
    w = datagen.uniform_f32(seed, 3, (B, Tq, HI))
    Kc = datagen.normal_bf16(seed, 4, (B, Ncap, D))
    Vc = datagen.normal_bf16(seed, 5, (B, Ncap, D))
    Rcap = W + Tq
    Kr = datagen.normal_bf16(seed, 6, (B, Rcap, D))
    Vr = datagen.normal_bf16(seed, 7, (B, Rcap, D))
    if nvfp4:
        kp, ks = datagen.nvfp4_normal(seed, 8, B * Ncap, DI)
        kI, kIs = kp.reshape(B, Ncap, DI // 2), ks.reshape(B, Ncap, DI // 16)
        kI_host = oracle.nvfp4_decode(kI.numpy(), kIs.numpy())
        kIs_d = kIs.to(DEV)
    else:
        kI = datagen.normal_bf16(seed, 8, (B, Ncap, DI))
        kI_host, kIs_d = f64(kI), None
    pos = [4 * n + 3 - Tq + 1 for n in nval]        # the last query sees every valid entry
    raw0 = [p - W + 1 for p in pos]                 # window rows of the first query present
    dv = {n: t.to(DEV) for n, t in dict(q=q, qI=qI, w=w, Kc=Kc, Vc=Vc, Kr=Kr, Vr=Vr, kI=kI).items()}
    pos_d = torch.tensor(pos, device=DEV)
    raw_d = torch.tensor(raw0, device=DEV)
    nval_d = torch.tensor(nval, dtype=torch.int32, device=DEV)
    idx1 = torch.full((B, Tq, k), -7, dtype=torch.int32, device=DEV)
    out1 = lcc.csa_layer(dv["q"], dv["qI"], dv["w"], pos_d, dv["kI"], nval_d, m, k, dv["Kc"], dv["Vc"], dv["Kr"],
                         dv["Vr"], raw_d, W, kI_scale=kIs_d, idx=idx1)
    idx2 = lcc.lightning_index_topk(dv["qI"], dv["w"], pos_d, dv["kI"], nval_d, m, k, kI_scale=kIs_d)
    out2 = lcc.csa_layer_attn(dv["q"], dv["Kc"], dv["Vc"], idx2, dv["Kr"], dv["Vr"], pos_d, raw_d, W)
    torch.cuda.synchronize()
    lcc.sync_status()
    assert torch.equal(idx1, idx2)
    # the one-cluster path attends in 16-key tiles, the two-call path in 32-key ones: equal up to rounding
    assert_close(out1.float().cpu().numpy(), out2.float().cpu().numpy(), "one cluster vs two calls")
    g, go = idx1.cpu().numpy(), out1.float().cpu().numpy()
    qh, Kch, Vch, Krh, Vrh = f64(q), f64(Kc), f64(Vc), f64(Kr), f64(Vr)
    near = 0
    for b in range(B):
        for i in range(Tq):
            t = pos[b] + i
            nv = oracle.visible_count(t, m, nval[b])
            sc = oracle.index_scores(f64(qI[b, i]), f64(w[b, i]), kI_host[b, :nv])
            oi, kth = oracle.topk_select(sc, k)
            ok, exact = topk_set_ok(g[b, i], oi, sc, kth, k)
            assert ok, f"batch {b} query {i}: top-k set differs"
            near += not exact
            sel = g[b, i][g[b, i] >= 0]
            cO, cL = oracle.attend(qh[b, i], Kch[b, sel], Vch[b, sel])
            sw = runs.swa_branch(qh[b, i], t, Krh[b], Vrh[b], raw0[b], W)
            O, _ = oracle.merge([cO, sw["O"]], [cL, sw["lse"]])
            assert_close(go[b, i], O, f"batch {b} query {i}")
    assert near <= 1
