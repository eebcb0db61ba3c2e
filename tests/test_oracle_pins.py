"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test fixes one function by a closed form, a hand-worked value, brute
force on a tiny input, or a special case that reduces to a library routine,
so that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails here.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import runs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


def _bf16_grid(shape, scale=1.0):
    """Random float64 values that are exactly bf16 (via torch's own rounding)."""
    x = torch.from_numpy(rng.standard_normal(shape) * scale).to(torch.bfloat16)
    return x.to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------
def test_bf16_rne_hand_cases():
    one = 1.0
    cases = {
        one: one,
        one + 2 ** -8: one,                        # tie -> even mantissa (0)
        one + 3 * 2 ** -8: one + 2 ** -6,          # tie between odd 1+2^-7 and even 1+2^-6
        one + 2 ** -8 + 2 ** -30: one + 2 ** -7,   # just above the tie
        -(one + 2 ** -8): -one,
        3.0 * 2 ** -20: 3.0 * 2 ** -20,
        257.0: 256.0,                              # 257 needs 9 bits; tie -> 256
        259.0: 260.0,
    }
    for x, want in cases.items():
        assert oracle.round_bf16(np.array([x]))[0] == want, x


def test_bf16_matches_library_rounding():
    x32 = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    lib = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = oracle.f64_to_bf16_bits(x32.astype(np.float64))
    assert np.array_equal(lib, ours)
    back = oracle.bf16_to_f64(ours)
    assert np.array_equal(back, torch.from_numpy(x32).to(torch.bfloat16).double().numpy())


def test_e4m3_all_codes_vs_library():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_value(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(lib)
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], lib[~nan])
    # closed forms: largest normal, smallest normal, smallest subnormal
    assert oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x08) == 2.0 ** -6
    assert oracle.e4m3_value(0x01) == 2.0 ** -9
    assert oracle.e4m3_value(0x38) == 1.0


def test_e2m1_table():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    vals = oracle.e2m1_value(np.arange(16))
    assert list(vals[:8]) == mags
    assert list(vals[8:]) == [-m for m in mags]


def test_nvfp4_decode_layout():
    # byte 0x21: low nibble code 1 (0.5) is element 0, high nibble code 2 (1.0) element 1
    packed = np.zeros((1, 8), np.uint8)
    packed[0, 0] = 0x21
    packed[0, 7] = 0xF9            # element 14 = code 9 (-0.5), element 15 = code 15 (-6)
    scale = np.array([[0x38]], np.uint8)   # 1.0
    v = oracle.nvfp4_decode(packed, scale)
    assert v.shape == (1, 16)
    assert v[0, 0] == 0.5 and v[0, 1] == 1.0 and v[0, 14] == -0.5 and v[0, 15] == -6.0
    assert np.all(v[0, 2:14] == 0)
    # second group uses its own scale: 0x40 = 2.0
    packed2 = np.full((1, 16), 0x77, np.uint8)
    v2 = oracle.nvfp4_decode(packed2, np.array([[0x38, 0x40]], np.uint8))
    assert np.all(v2[0, :16] == 6.0) and np.all(v2[0, 16:] == 12.0)


def test_nvfp4_values_fit_bf16_exactly():
    # every e2m1 x e4m3 product is a bf16 value (<= 6 significant bits, in range)
    prod = np.outer(oracle.e2m1_value(np.arange(16)),
                    oracle.e4m3_value(np.array([c for c in range(256) if c not in (0x7F, 0xFF)])))
    assert np.array_equal(oracle.round_bf16(prod.ravel()), prod.ravel())


# NVFP4 quantisation of the indexer query (reading R16)
def test_nvfp4_quantize_hand_case():
    # amax 3 -> scale 3/6 = 0.5 = e4m3 0x30; x/0.5: 0.2 -> 0, -0.4 -> -0.5 (code 9),
    # 6 -> 6 (code 7), 1.4 -> 1.5 (code 3); element 2i in the low nibble of byte i
    x = np.array([[0.1, -0.2, 3.0, 0.7] * 4])
    packed, scale = oracle.nvfp4_quantize(x)
    assert scale.tolist() == [[0x30]]
    assert packed.tolist() == [[0x90, 0x37] * 4]
    assert oracle.nvfp4_decode(packed, scale).tolist() == [[0.0, -0.25, 3.0, 0.75] * 4]


def test_nvfp4_quantize_ties_go_to_even_codes():
    # x/scale exactly between two e2m1 values: the neighbour with the even code
    # (even mantissa bit) is kept; hand table of the seven midpoints
    want = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for s in (2.0 ** -9, 2.0 ** -6, 0.375, 1.0, 13.0, 448.0):
        for mid, v in want.items():
            row = np.zeros(16)
            row[0] = 6.0 * s            # amax = 6 s -> scale exactly s
            row[1], row[2] = mid * s, -mid * s
            p, sc = oracle.nvfp4_quantize(row[None])
            d = oracle.nvfp4_decode(p, sc)[0]
            assert oracle.e4m3_value(sc[0, 0]) == s
            assert d[1] == v * s and d[2] == -v * s, (s, mid)


def test_nvfp4_quantize_grid_values_round_trip():
    # values already on the grid of a group whose amax is 6*scale come back unchanged
    r = np.random.default_rng(7)
    codes = r.integers(0, 16, size=(300, 64))
    codes[:, ::16] = 7                       # each group holds +6
    codes = np.where(codes == 8, 0, codes)   # -0 is stored as +0
    scales = r.integers(1, 127, size=(300, 4)).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    x = oracle.nvfp4_decode(packed, scales)
    p2, s2 = oracle.nvfp4_quantize(x)
    assert np.array_equal(s2, scales) and np.array_equal(p2, packed)


def test_nvfp4_quantize_is_nearest_by_brute_force():
    # every element lands on a grid value of its group no farther than any other one
    r = np.random.default_rng(8)
    x = _bf16_grid((64, 64)) * np.exp(r.uniform(-6, 6, size=(64, 1)))
    p, sc = oracle.nvfp4_quantize(x)
    d = oracle.nvfp4_decode(p, sc)
    s = np.repeat(oracle.e4m3_value(sc), 16, axis=-1)
    grid = oracle.e2m1_value(np.arange(16))                 # all 16 codes
    err = np.abs(x - d)
    best = np.abs(x[..., None] - grid * s[..., None]).min(axis=-1)
    assert np.all(err <= best)


def test_nvfp4_scale_every_bf16_amax_vs_library_rounding():
    # every positive finite bf16 value as a group maximum: the scale is the e4m3
    # value nearest to amax/6 -- torch's float8_e4m3fn rounding below 448, and
    # saturation at 448 above it
    bits = np.arange(1, 0x7F80, dtype=np.uint16)
    amax = oracle.bf16_to_f64(bits)
    g = np.zeros((amax.size, 16))
    g[:, 5] = amax
    _, sc = oracle.nvfp4_quantize(g)
    got = oracle.e4m3_value(sc[:, 0])
    small = amax / 6.0 < 448.0
    lib = torch.from_numpy(amax[small] / 6.0).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(got[small], lib)
    assert np.all(got[~small] == 448.0)


def test_nvfp4_quantize_agrees_with_the_key_encoder():
    # the input generator encodes NVFP4 keys by formulas (frexp/round), the
    # oracle by distance to every table value: two independent codings of R7
    import datagen
    r = np.random.default_rng(9)
    x = _bf16_grid((512, 64)) * np.exp(r.uniform(-12, 8, size=(512, 1)))
    p1, s1 = oracle.nvfp4_quantize(x)
    p2, s2 = datagen.nvfp4_encode(torch.from_numpy(x))
    assert np.array_equal(s1, s2.numpy()) and np.array_equal(p1, p2.numpy())


def test_index_scores_fp4_hand_case():
    # query head 0: amax 6 -> scale 1: [6, 3, 0.7, -0.2] -> [6, 3, 0.5, 0];
    # head 1 is its negative.  Key: codes 1, 2, 4 (0.5, 1, 2) at scale 2 -> [1, 2, 4].
    # head 0: 6 + 6 + 2 = 14, weight 0.5 -> 7; head 1: ReLU(-14) = 0
    qI = np.zeros((2, 16))
    qI[0, :4] = [6.0, 3.0, 0.7, -0.2]
    qI[1] = -qI[0]
    w = np.array([0.5, 3.0])
    kp = np.zeros((1, 8), np.uint8)
    kp[0, 0] = 0x21
    kp[0, 1] = 0x04
    ks = np.array([[0x40]], np.uint8)
    assert oracle.index_scores_fp4(qI, w, kp, ks).tolist() == [7.0]


# ---------------------------------------------------------------------------
# pooling
# ---------------------------------------------------------------------------
def test_pool_weights_golden():
    g = json.load(open(os.path.join(GOLDEN, "pool_hand.json")))
    for c in g["cases"]:
        a = oracle.pool_weights(np.array(c["gates"]))
        np.testing.assert_allclose(a, c["weights"], rtol=0, atol=1e-15)
    blk = g["block"]
    Kc, Vc = oracle.pool_exact(np.array(blk["K_rows"]), np.array(blk["V_rows"]),
                               np.array(blk["gates"]), 4)
    np.testing.assert_allclose(Kc[0], blk["Kc"], atol=1e-14)
    np.testing.assert_allclose(Vc[0], blk["Vc"], atol=1e-14)


def test_pool_weights_invariants():
    g = rng.standard_normal((1000, 128))
    a = oracle.pool_weights(g)
    np.testing.assert_allclose(a.sum(1), 1.0, atol=1e-15)
    np.testing.assert_allclose(oracle.pool_weights(g + 7.25), a, atol=1e-15)
    hot = oracle.pool_weights(np.array([100.0, 0.0, 0.0, 0.0]))
    assert abs(hot[0] - 1.0) < 1e-40 + 1e-15 and hot[1] < 1e-43


def test_pool_block_structure_and_tail():
    T, D, m = 10, 3, 4
    K = np.repeat(np.arange(T, dtype=np.float64)[:, None], D, axis=1)
    V = -2.0 * K
    Kc, Vc = oracle.pool_exact(K, V, np.zeros(T), m)
    assert Kc.shape == (2, D)                          # tokens 8, 9 form no entry
    np.testing.assert_allclose(Kc[:, 0], [1.5, 5.5])   # means of 0..3 and 4..7
    np.testing.assert_allclose(Vc[:, 0], [-3.0, -11.0])
    # weights follow the block's own gates, and K and V share them
    gate = np.zeros(T)
    gate[7] = math.log(5.0)
    Kc, Vc = oracle.pool_exact(K, V, gate, m)
    np.testing.assert_allclose(Kc[1, 0], (4 + 5 + 6) / 8 + 7 * 5 / 8)
    np.testing.assert_allclose(Kc[0, 0], 1.5)
    np.testing.assert_allclose(Vc[1, 0], -2 * Kc[1, 0])


def test_pool_m1_is_identity_and_rounding():
    K = _bf16_grid((50, 8))
    V = _bf16_grid((50, 8))
    Kc, Vc = oracle.pool(K, V, rng.standard_normal(50), 1)
    assert np.array_equal(Kc, K) and np.array_equal(Vc, V)
    K = _bf16_grid((64, 8))
    g = rng.standard_normal(64)
    ex, _ = oracle.pool_exact(K, K, g, 4)
    st, _ = oracle.pool(K, K, g, 4)
    assert np.array_equal(st, oracle.round_bf16(ex))
    assert np.max(np.abs(st - ex)) <= np.max(np.abs(ex)) * 2 ** -8


# ---------------------------------------------------------------------------
# visibility
# ---------------------------------------------------------------------------
def test_visible_count_hand():
    assert [oracle.visible_count(t, 4) for t in range(9)] == [0, 0, 0, 1, 1, 1, 1, 2, 2]
    assert oracle.visible_count(126, 128) == 0 and oracle.visible_count(127, 128) == 1
    assert oracle.visible_count(1048575, 128) == 8192
    assert oracle.visible_count(10 ** 6, 4, n_valid=7) == 7


@pytest.mark.parametrize("m", [1, 4, 128])
def test_visible_means_block_complete(m):
    # an entry is visible exactly when its last token is at or before the query
    for t in range(0, 4 * m + 3):
        v = oracle.visible_count(t, m)
        for j in range(0, t // m + 3):
            assert (j < v) == (j * m + m - 1 <= t)


# ---------------------------------------------------------------------------
# indexer and top-k
# ---------------------------------------------------------------------------
def test_index_scores_brute_force():
    HI, DI, n = 3, 5, 17
    qI, w, kI = rng.standard_normal((HI, DI)), rng.uniform(0, 1, HI), rng.standard_normal((n, DI))
    s = oracle.index_scores(qI, w, kI)
    for j in range(n):
        want = 0.0
        for h in range(HI):
            dot = 0.0
            for c in range(DI):
                dot += qI[h][c] * kI[j][c]
            want += w[h] * (dot if dot > 0 else 0.0)
        assert abs(s[j] - want) < 1e-12


def test_index_scores_one_hot_weight_and_relu():
    qI, kI = rng.standard_normal((4, 8)), rng.standard_normal((30, 8))
    for h in range(4):
        w = np.zeros(4)
        w[h] = 1.0
        np.testing.assert_allclose(oracle.index_scores(qI, w, kI), np.maximum(kI @ qI[h], 0), atol=1e-13)
    assert np.all(oracle.index_scores(qI, np.ones(4), -np.abs(kI) * 0) == 0)


def test_topk_matches_full_sort_with_ties():
    for n, k in [(50, 16), (7, 16), (200, 128), (0, 4), (16, 16)]:
        s = rng.integers(0, 6, n).astype(np.float64)   # many exact ties
        idx, kth = oracle.topk_select(s, k)
        full = sorted(range(n), key=lambda j: (-s[j], j))[:k]
        assert list(idx[idx >= 0]) == sorted(full)
        assert np.all(idx[len(full):] == -1)
        if n >= k:
            assert kth == s[full[-1]]
        else:
            assert kth == -np.inf


def test_topk_ties_go_to_lower_index():
    s = np.zeros(40)
    s[[5, 30]] = 1.0
    idx, _ = oracle.topk_select(s, 4)
    assert list(idx) == [0, 1, 5, 30]


# ---------------------------------------------------------------------------
# attention and merge
# ---------------------------------------------------------------------------
def test_attend_vs_library_sdpa():
    H, D, n = 6, 16, 23
    q, K, V = rng.standard_normal((H, D)), rng.standard_normal((n, D)), rng.standard_normal((n, D))
    O, lse = oracle.attend(q, K, V, scale=0.3)
    tq, tk, tv = (torch.from_numpy(x)[None] for x in (q, K, V))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.3)[0].numpy()
    np.testing.assert_allclose(O, ref, atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.from_numpy(0.3 * q @ K.T), 1).numpy(), atol=1e-12)


def test_attend_empty():
    O, lse = oracle.attend(rng.standard_normal((4, 8)), np.zeros((0, 8)), np.zeros((0, 8)))
    assert np.all(O == 0) and np.all(lse == -np.inf)


def _causal_dense(q, K, V):
    """Textbook causal attention through the library: softmax(QK^T + mask) V."""
    T = K.shape[0]
    mask = torch.full((T, T), -float("inf"), dtype=torch.float64).triu(1)
    outs = []
    for h in range(q.shape[1]):
        z = torch.from_numpy(q[:, h] @ K.T) + mask
        outs.append((torch.softmax(z, 1) @ torch.from_numpy(V)).numpy())
    return np.stack(outs, 1)


def test_hca_m1_no_window_equals_dense_causal():
    T, H, D = 40, 3, 8
    K, V, q = _bf16_grid((T, D)), _bf16_grid((T, D)), rng.standard_normal((T, H, D)) * 0.4
    Kc, Vc = oracle.pool(K, V, rng.standard_normal(T), 1)
    ref = _causal_dense(q, K, V)
    for t in range(T):
        r = runs.hca_branch(q[t], t, Kc, Vc, 1)
        np.testing.assert_allclose(r["O"], ref[t], atol=1e-12)


def test_swa_wide_window_equals_dense_causal():
    T, H, D = 33, 2, 8
    K, V, q = _bf16_grid((T, D)), _bf16_grid((T, D)), rng.standard_normal((T, H, D)) * 0.4
    ref = _causal_dense(q, K, V)
    for t in range(T):
        r = runs.swa_branch(q[t], t, K, V, 0, W=T + 5)
        np.testing.assert_allclose(r["O"], ref[t], atol=1e-12)
    # a narrow window holds exactly positions t-W+1 .. t
    assert list(oracle.window_positions(10, 4)) == [7, 8, 9, 10]
    assert list(oracle.window_positions(2, 4)) == [0, 1, 2]
    assert list(oracle.window_positions(10, 4, raw_pos0=9)) == [9, 10]


def test_csa_with_large_k_equals_hca_m4():
    T, H, D, HI, DI = 64, 2, 8, 2, 4
    K, V = _bf16_grid((T, D)), _bf16_grid((T, D))
    g = rng.standard_normal(T)
    Kc, Vc = oracle.pool(K, V, g, 4)
    kI = rng.standard_normal((T // 4, DI))
    for t in range(T):
        q = rng.standard_normal((H, D))
        c = runs.csa_branch(q, t, rng.standard_normal((HI, DI)), rng.uniform(0, 1, HI), kI, Kc, Vc, 4, k=T)
        h = runs.hca_branch(q, t, Kc, Vc, 4)
        np.testing.assert_allclose(c["O"], h["O"], atol=1e-12)
        np.testing.assert_allclose(c["lse"], h["lse"], atol=1e-12)
        assert c["n_visible"] == h["n_visible"] == (t + 1) // 4


def test_dsa_m1_with_large_k_equals_dense_causal():
    # the DSA comparator ([THREAD] "주요 댓글": the indexer runs over the full KV,
    # attention over the tokens it selects) is CSA with m = 1; when k covers
    # every visible token it is textbook causal attention, and with a small k
    # it attends exactly to the brute-force best-scoring tokens
    T, H, D, HI, DI, k = 30, 2, 8, 2, 4, 5
    K, V = _bf16_grid((T, D)), _bf16_grid((T, D))
    Kc, Vc = oracle.pool(K, V, rng.standard_normal(T), 1)
    kI = rng.standard_normal((T, DI))
    q = rng.standard_normal((T, H, D)) * 0.4
    ref = _causal_dense(q, K, V)
    for t in range(T):
        qI, w = rng.standard_normal((HI, DI)), rng.uniform(0, 1, HI)
        c = runs.csa_branch(q[t], t, qI, w, kI, Kc, Vc, 1, k=T)
        np.testing.assert_allclose(c["O"], ref[t], atol=1e-12)
        assert c["n_visible"] == t + 1
        small = runs.csa_branch(q[t], t, qI, w, kI, Kc, Vc, 1, k=k)
        sc = [sum(w[h] * max(0.0, float(qI[h] @ kI[j])) for h in range(HI)) for j in range(t + 1)]
        best = sorted(range(t + 1), key=lambda j: (-sc[j], j))[:k]
        assert sorted(best) == [j for j in small["idx"] if j >= 0]
        O, _ = oracle.attend(q[t], K[sorted(best)], V[sorted(best)])
        np.testing.assert_allclose(small["O"], O, atol=1e-12)


def test_merge_equals_softmax_over_concatenation():
    H, D = 4, 8
    q = rng.standard_normal((H, D))
    parts = [(rng.standard_normal((n, D)), rng.standard_normal((n, D))) for n in (5, 9, 3)]
    res = [oracle.attend(q, Kp, Vp) for Kp, Vp in parts]
    O, L = oracle.merge([r[0] for r in res], [r[1] for r in res])
    Ocat, Lcat = oracle.attend(q, np.concatenate([p[0] for p in parts]), np.concatenate([p[1] for p in parts]))
    np.testing.assert_allclose(O, Ocat, atol=1e-12)
    np.testing.assert_allclose(L, Lcat, atol=1e-12)


def test_merge_with_empty_branches():
    H, D = 3, 4
    O1, L1 = rng.standard_normal((H, D)), rng.standard_normal(H)
    O, L = oracle.merge([np.zeros((H, D)), O1], [np.full(H, -np.inf), L1])
    np.testing.assert_allclose(O, O1, atol=1e-15)
    np.testing.assert_allclose(L, L1, atol=1e-15)
    O, L = oracle.merge([np.zeros((H, D)), np.zeros((H, D))], [np.full(H, -np.inf)] * 2)
    assert np.all(O == 0) and np.all(L == -np.inf)


def test_tiny_prefill_early_rows_have_empty_compressed_branches():
    from datagen.workloads import TinyPrefill
    cfg = TinyPrefill()
    inp = {k: (v.view(torch.int16).numpy().view(np.uint16) if v.dtype == torch.bfloat16 else v.numpy())
           for k, v in cfg.make().items()}
    out = runs.tiny_prefill(inp, cfg, rows=[0, 2, 3, 127, 2047])
    r = {x["t"]: x for x in out["rows"]}
    for t in (0, 2):
        assert np.all(r[t]["csa"]["lse"] == -np.inf) and np.all(r[t]["csa"]["idx"] == -1)
        np.testing.assert_allclose(r[t]["csa_layer"][0], r[t]["swa"]["O"], atol=1e-15)
    assert list(r[3]["csa"]["idx"][:2]) == [0, -1]
    assert r[127]["hca"]["n_visible"] == 1 and r[127]["swa"]["n_keys"] == 32
    assert r[2047]["csa"]["n_visible"] == 512 and np.all(r[2047]["csa"]["idx"] >= 0)


def test_page_facts_match_workloads():
    from datagen.workloads import CsaDecode, CsaPrefill, HcaDecode, PairDecode
    f = json.load(open(os.path.join(GOLDEN, "pages_facts.json")))["facts"]
    assert CsaPrefill().m == PairDecode().m_csa == f["csa_tokens_per_entry"]["value"]
    assert HcaDecode().m == PairDecode().m_hca == f["hca_tokens_per_entry"]["value"]
    assert abs(HcaDecode().N - f["hca_entries_at_1m_tokens_approx"]["value"]) / 8000 < 0.03
    assert HcaDecode().ctx // HcaDecode().m == HcaDecode().N
    assert PairDecode().m_hca // PairDecode().m_csa == f["hca_lighter_than_csa"]["value"]
    for c in (CsaDecode(), CsaPrefill(), PairDecode()):
        assert c.k == f["csa_topk_typical"]["value"] and c.W == f["window_tokens"]["value"]


# ---------------------------------------------------------------------------
# layer compositions over time: every expected value below comes from one
# contiguous token sequence pooled in full (oracle.pool over the whole
# sequence) and the branch functions pinned above, applied at each absolute
# position; the compositions under test instead pool blocks out of raw
# buffers at offsets of their own.  [HYBRID] "두 가지 압축 전략: CSA 및 HCA":
# entries pool m consecutive tokens and the window branch runs beside them;
# [VIDEO] "쉽게 이해하기": the window is the most recent tokens (128 in the
# model).  These fix reading R9 (where each new token sits in the raw buffer,
# which raw rows a completed block pools, and from which step on the new
# entry is visible).
# ---------------------------------------------------------------------------
def _bits(x):
    return oracle.f64_to_bf16_bits(x)


def test_pair_decode_matches_full_sequence_pooling():
    from datagen.workloads import PairDecode
    cfg = PairDecode(B=1, ctx=16, steps=9, D=8, H=2, HI=2, DI=16, k=3, W=4, m_csa=4, m_hca=8)
    L = cfg.ctx + cfg.steps                                   # 25 tokens in all
    K, V, g = _bf16_grid((L, cfg.D)), _bf16_grid((L, cfg.D)), rng.standard_normal(L)
    Kh, Vh, gh = _bf16_grid((L, cfg.D)), _bf16_grid((L, cfg.D)), rng.standard_normal(L)
    kI = _bf16_grid((cfg.Ncap_csa, cfg.DI))
    q = _bf16_grid((cfg.steps, 1, cfg.H, cfg.D), 0.5)
    qI = _bf16_grid((cfg.steps, 1, cfg.HI, cfg.DI))
    w = rng.uniform(0, 1, (cfg.steps, 1, cfg.HI))
    # whole-sequence pooling: every entry that exists at the end of the run
    Kc_all, Vc_all = oracle.pool(K, V, g, cfg.m_csa)          # 6 entries
    Kh_all, Vh_all = oracle.pool(Kh, Vh, gh, cfg.m_hca)       # 3 entries (the last completes at step 7)
    assert len(Kc_all) == cfg.Ncap_csa and len(Kh_all) == 3
    r0 = cfg.ctx - cfg.W                                      # raw buffers start W tokens before ctx
    inp = dict(Kr=_bits(K[None, r0:]), Vr=_bits(V[None, r0:]), gate=g[None, r0:],
               Kr_h=_bits(Kh[None, r0:]), Vr_h=_bits(Vh[None, r0:]), gate_h=gh[None, r0:],
               Kc=_bits(Kc_all[None, :cfg.N_csa]), Vc=_bits(Vc_all[None, :cfg.N_csa]),
               Kc_h=_bits(Kh_all[None, :cfg.N_hca]), Vc_h=_bits(Vh_all[None, :cfg.N_hca]),
               q=_bits(q), qI=_bits(qI), w=w)
    got = runs.pair_decode(inp, cfg, kI=kI[None])
    seen_csa, seen_hca = [], []
    for s in range(cfg.steps):
        t = cfg.ctx + s
        c = runs.csa_branch(q[s, 0], t, qI[s, 0], w[s, 0], kI, Kc_all, Vc_all, cfg.m_csa, cfg.k)
        sw = runs.swa_branch(q[s, 0], t, K, V, 0, cfg.W)
        h = runs.hca_branch(q[s, 0], t, Kh_all, Vh_all, cfg.m_hca)
        swh = runs.swa_branch(q[s, 0], t, Kh, Vh, 0, cfg.W)
        want_c = oracle.merge([c["O"], sw["O"]], [c["lse"], sw["lse"]])
        want_h = oracle.merge([h["O"], swh["O"]], [h["lse"], swh["lse"]])
        r = got[(s, 0)]
        assert np.array_equal(r["idx"], c["idx"]), s
        np.testing.assert_allclose(r["scores"], c["scores"], atol=1e-12)
        for a, b in ((r["csa"], want_c), (r["hca"], want_h)):
            np.testing.assert_allclose(a[0], b[0], atol=1e-12)
            np.testing.assert_allclose(a[1], b[1], atol=1e-12)
        seen_csa.append(c["n_visible"])
        seen_hca.append(h["n_visible"])
        assert sw["n_keys"] == cfg.W
    # the schedule: CSA entry 4 becomes visible at position 19 (step 3), entry 5 at
    # position 23 (step 7); HCA entry 2 at position 23 (step 7)
    assert seen_csa == [4, 4, 4, 5, 5, 5, 5, 6, 6]
    assert seen_hca == [2, 2, 2, 2, 2, 2, 2, 3, 3]
    new = got[(cfg.steps - 1, 0)]
    assert sorted(new["new_entries"]) == [4, 5] and sorted(new["new_entries_h"]) == [2]
    np.testing.assert_array_equal(new["new_entries"][5][0], Kc_all[5])
    np.testing.assert_array_equal(new["new_entries_h"][2][1], Vh_all[2])


def test_hca_prefill_matches_full_sequence_pooling():
    from datagen.workloads import HcaPrefill
    cfg = HcaPrefill(ctx=32, Tc=24, N0=4, D=8, H=2, W=4, m=8)
    L = cfg.ctx + cfg.Tc                                       # 56 tokens in all
    K, V, g = _bf16_grid((L, cfg.D)), _bf16_grid((L, cfg.D)), rng.standard_normal(L)
    q = _bf16_grid((cfg.Tc, cfg.H, cfg.D), 0.5)
    Kc_all, Vc_all = oracle.pool(K, V, g, cfg.m)               # 7 entries
    assert len(Kc_all) == cfg.Ncap
    r0 = cfg.raw_pos0                                          # W-1 tokens before the chunk
    Kc0 = np.zeros((1, cfg.Ncap, cfg.D))
    Kc0[0, :cfg.N0] = Kc_all[:cfg.N0]
    Vc0 = np.zeros((1, cfg.Ncap, cfg.D))
    Vc0[0, :cfg.N0] = Vc_all[:cfg.N0]
    inp = dict(Kr=_bits(K[None, r0:]), Vr=_bits(V[None, r0:]), gate=g[None, r0:],
               Kc=_bits(Kc0), Vc=_bits(Vc0))
    rows = list(range(cfg.Tc))
    got = runs.hca_prefill(inp, cfg, rows, _bits(q))
    np.testing.assert_array_equal(got["Kc_new"], Kc_all[cfg.N0:])
    np.testing.assert_array_equal(got["Vc_new"], Vc_all[cfg.N0:])
    for i in rows:
        t = cfg.ctx + i
        h = runs.hca_branch(q[i], t, Kc_all, Vc_all, cfg.m)
        sw = runs.swa_branch(q[i], t, K, V, 0, cfg.W)
        want = oracle.merge([h["O"], sw["O"]], [h["lse"], sw["lse"]])
        r = got["rows"][i]
        assert r["hca"]["n_visible"] == (t + 1) // cfg.m
        np.testing.assert_allclose(r["layer"][0], want[0], atol=1e-12)
        np.testing.assert_allclose(r["layer"][1], want[1], atol=1e-12)


def test_swa_replay_bounds_the_window_and_restores_the_last_state():
    # [V41], SWA Bounded Replay: only the last R tokens are replayed against the
    # kept compressed caches.  Every expected value comes from whole-sequence
    # pooling and the pinned branch functions with a raw buffer that holds the
    # entire history.
    from datagen.workloads import PairDecode
    cfg = PairDecode(B=1, ctx=32, steps=1, D=8, H=2, HI=2, DI=16, k=3, W=8, m_csa=4, m_hca=8)
    R = cfg.W
    L = cfg.ctx
    K, V, g = _bf16_grid((L, cfg.D)), _bf16_grid((L, cfg.D)), rng.standard_normal(L)
    Kh, Vh, gh = _bf16_grid((L, cfg.D)), _bf16_grid((L, cfg.D)), rng.standard_normal(L)
    Kc, Vc = oracle.pool(K, V, g, cfg.m_csa)
    Khc, Vhc = oracle.pool(Kh, Vh, gh, cfg.m_hca)
    # NVFP4 keys: codes and scales chosen at random, decoded by the pinned decoder
    kp = rng.integers(0, 256, (1, cfg.N_csa, cfg.DI // 2), dtype=np.uint8)
    ks = rng.integers(0x20, 0x48, (1, cfg.N_csa, cfg.DI // 16), dtype=np.uint8)
    kI = oracle.nvfp4_decode(kp[0], ks[0])
    rq = _bf16_grid((R, 1, cfg.H, cfg.D), 0.5)
    rqI = _bf16_grid((R, 1, cfg.HI, cfg.DI))
    rw = rng.uniform(0, 1, (R, 1, cfg.HI))
    r0 = cfg.ctx - cfg.W
    inp = dict(Kr=_bits(K[None, r0:]), Vr=_bits(V[None, r0:]), Kr_h=_bits(Kh[None, r0:]), Vr_h=_bits(Vh[None, r0:]),
               Kc=_bits(Kc[None]), Vc=_bits(Vc[None]), Kc_h=_bits(Khc[None]), Vc_h=_bits(Vhc[None]),
               kI_packed=kp, kI_scale=ks, rq=_bits(rq), rqI=_bits(rqI), rw=rw)
    got = runs.swa_replay(inp, cfg, R)
    for i in range(R):
        t = cfg.ctx - R + i
        r = got[(i, 0)]
        assert r["window"] == i + 1                      # the rebuilt window only holds replayed tokens
        c = runs.csa_branch(rq[i, 0], t, rqI[i, 0], rw[i, 0], kI, Kc, Vc, cfg.m_csa, cfg.k)
        assert np.array_equal(r["idx"], c["idx"])
        sw_full = runs.swa_branch(rq[i, 0], t, K, V, 0, cfg.W)
        sw_rep = runs.swa_branch(rq[i, 0], t, K[cfg.ctx - R:], V[cfg.ctx - R:], cfg.ctx - R, cfg.W)
        want = oracle.merge([c["O"], sw_rep["O"]], [c["lse"], sw_rep["lse"]])
        np.testing.assert_allclose(r["csa"][0], want[0], atol=1e-12)
        if i == R - 1:
            # the last replayed position has its full window: its output equals
            # the unbounded recomputation of the whole prompt's state
            full_c = oracle.merge([c["O"], sw_full["O"]], [c["lse"], sw_full["lse"]])
            h = runs.hca_branch(rq[i, 0], t, Khc, Vhc, cfg.m_hca)
            swh = runs.swa_branch(rq[i, 0], t, Kh, Vh, 0, cfg.W)
            full_h = oracle.merge([h["O"], swh["O"]], [h["lse"], swh["lse"]])
            np.testing.assert_allclose(r["csa"][0], full_c[0], atol=1e-12)
            np.testing.assert_allclose(r["hca"][0], full_h[0], atol=1e-12)
        else:
            assert sw_full["n_keys"] == cfg.W > r["window"]


# ---------------------------------------------------------------------------
# query / KV prologue ([HYBRID]: query and KV normalisation, partial RoPE)
# ---------------------------------------------------------------------------
def test_rms_norm_hand_values():
    # row (3, 4): mean square 12.5; eps 0 -> (3, 4) / sqrt(12.5)
    y = oracle.rms_norm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.0)
    np.testing.assert_allclose(y, [[3 / math.sqrt(12.5), 8 / math.sqrt(12.5)]], rtol=1e-15)
    # unit gains: mean square of the output is ms / (ms + eps)
    x = rng.standard_normal((5, 128))
    y = oracle.rms_norm(x, np.ones(128), 1e-6)
    ms = np.mean(x * x, 1)
    np.testing.assert_allclose(np.mean(y * y, 1), ms / (ms + 1e-6), rtol=1e-12)
    # scale invariance (up to eps)
    np.testing.assert_allclose(oracle.rms_norm(7.0 * x, np.ones(128), 0.0), oracle.rms_norm(x, np.ones(128), 0.0),
                               rtol=1e-13)


def test_rope_matches_complex_rotation_and_leaves_the_rest():
    D, d, pos = 128, 64, 12345
    x = rng.standard_normal((3, D))
    y = oracle.rope_partial(x, pos, d)
    np.testing.assert_array_equal(y[:, :D - d], x[:, :D - d])
    z = (x[:, D - d:D - d // 2] + 1j * x[:, D - d // 2:]) * np.exp(
        1j * pos * 10000.0 ** (-np.arange(d // 2) * 2.0 / d))
    np.testing.assert_allclose(y[:, D - d:D - d // 2], z.real, atol=1e-12)
    np.testing.assert_allclose(y[:, D - d // 2:], z.imag, atol=1e-12)
    np.testing.assert_array_equal(oracle.rope_partial(x, 0, d), x)          # position 0: identity


def test_rope_scores_depend_on_relative_position_only():
    D, d = 128, 64
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    for p, s, c in ((10, 3, 1000), (70000, 1, 5), (1048575, 1048000, -1040000)):
        a = oracle.rope_partial(q, p, d) @ oracle.rope_partial(k, s, d)
        b = oracle.rope_partial(q, p + c, d) @ oracle.rope_partial(k, s + c, d)
        assert abs(a - b) <= 1e-9 * (abs(a) + 1)
    # rotating by p then by -p restores the row (the map is orthogonal)
    np.testing.assert_allclose(oracle.rope_partial(oracle.rope_partial(q, 777, d), -777, d), q, atol=1e-12)


def test_prologue_order_norm_then_rope_and_v_unrotated():
    H, D, d = 3, 128, 64
    q, k, v = rng.standard_normal((H, D)), rng.standard_normal(D), rng.standard_normal(D)
    gq, gk, gv = 1 + 0.1 * rng.standard_normal((3, D))
    qn, kn, vn = oracle.qkv_prologue(q, k, v, 99, gq, gk, gv, 1e-6, d)
    np.testing.assert_allclose(qn, oracle.rope_partial(oracle.rms_norm(q, gq, 1e-6), 99, d), atol=0)
    np.testing.assert_allclose(kn, oracle.rope_partial(oracle.rms_norm(k, gk, 1e-6), 99, d), atol=0)
    np.testing.assert_allclose(vn, oracle.rms_norm(v, gv, 1e-6), atol=0)
    # the rotation keeps each pair's length: |q| after norm equals |q| after norm and rope
    np.testing.assert_allclose(np.linalg.norm(qn, axis=1),
                               np.linalg.norm(oracle.rms_norm(q, gq, 1e-6), axis=1), rtol=1e-13)


# ---------------------------------------------------------------------------
# CSA2 index sharing ([V41], the CSA2 passage: full / re-index / reuse modes)
# ---------------------------------------------------------------------------
def test_csa2_modes_brute_force_and_special_cases():
    N, D, H, HI, DI, k, n_notes, m = 40, 8, 2, 2, 4, 4, 10, 4
    t = N * m - 1
    kI = rng.standard_normal((N, DI))
    caches = [(_bf16_grid((N, D)), _bf16_grid((N, D))) for _ in range(4)]
    qIs = [rng.standard_normal((HI, DI)) for _ in range(3)]
    ws = [rng.uniform(0, 1, HI) for _ in range(3)]
    qs = [rng.standard_normal((H, D)) * 0.4 for _ in range(4)]
    layers = [dict(mode="full", q=qs[0], qI=qIs[0], w=ws[0], Kc=caches[0][0], Vc=caches[0][1]),
              dict(mode="reindex", q=qs[1], qI=qIs[1], w=ws[1], Kc=caches[1][0], Vc=caches[1][1]),
              dict(mode="reuse", q=qs[2], Kc=caches[2][0], Vc=caches[2][1]),
              dict(mode="reindex", q=qs[3], qI=qIs[0], w=ws[0], Kc=caches[3][0], Vc=caches[3][1])]
    out = runs.csa2_group(None, t, layers, kI, m, k, n_notes)

    def score(qI, w, j):
        return sum(w[h] * max(0.0, sum(qI[h, c] * kI[j, c] for c in range(DI))) for h in range(HI))
    s0 = [score(qIs[0], ws[0], j) for j in range(N)]
    notes = sorted(sorted(range(N), key=lambda j: (-s0[j], j))[:n_notes])
    assert [j for j in out[0]["notes"] if j >= 0] == notes
    assert [j for j in out[0]["idx"] if j >= 0] == sorted(sorted(range(N), key=lambda j: (-s0[j], j))[:k])
    s1 = {j: score(qIs[1], ws[1], j) for j in notes}
    assert [j for j in out[1]["idx"] if j >= 0] == sorted(sorted(notes, key=lambda j: (-s1[j], j))[:k])
    # reuse copies the previous layer's selection and attends to its own cache
    assert np.array_equal(out[2]["idx"], out[1]["idx"])
    sel = out[1]["idx"][out[1]["idx"] >= 0]
    O, _ = oracle.attend(qs[2], caches[2][0][sel], caches[2][1][sel])
    np.testing.assert_allclose(out[2]["O"], O, atol=1e-12)
    # re-indexing the notes with the full layer's own query gives the full layer's top-k
    assert np.array_equal(out[3]["idx"], out[0]["idx"])
    # notes covering every visible entry: re-index = full mode with the layer's own query
    wide = runs.csa2_group(None, t, layers[:2], kI, m, k, n_notes=N)
    full1 = runs.csa_branch(qs[1], t, qIs[1], ws[1], kI, caches[1][0], caches[1][1], m, k)
    assert np.array_equal(wide[1]["idx"], full1["idx"])
    np.testing.assert_allclose(wide[1]["O"], full1["O"], atol=1e-12)
