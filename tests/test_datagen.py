"""Host checks of the seeded input generator (CPU only)."""
import numpy as np
import torch

import datagen
import oracle


def test_deterministic_and_seed_dependent():
    a = datagen.normal_bf16(5, 1, (64, 32))
    b = datagen.normal_bf16(5, 1, (64, 32))
    c = datagen.normal_bf16(6, 1, (64, 32))
    d = datagen.normal_bf16(5, 2, (64, 32))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), c.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), d.view(torch.int16))


def test_rows_regenerate_exactly():
    full = datagen.normal_bf16(3, 4, (100, 48), scale=0.125)
    rows = torch.tensor([0, 17, 99])
    idx = (rows[:, None] * 48 + torch.arange(48)[None, :]).reshape(-1)
    part = datagen.normal_bf16_at(3, 4, idx, 0.125).reshape(3, 48)
    assert torch.equal(full[rows].view(torch.int16), part.view(torch.int16))


def test_moments():
    x = datagen.normal_bf16(0, 1, (1 << 20,)).double()
    assert abs(x.mean().item()) < 5e-3 and abs(x.std().item() - 1) < 5e-3
    u = datagen.uniform_f32(0, 2, (1 << 20,)).double()
    assert 0 < u.min().item() and u.max().item() < 1
    assert abs(u.mean().item() - 0.5) < 2e-3 and abs(u.var().item() - 1 / 12) < 1e-3
    g = datagen.normal_f32(0, 3, (1 << 20,)).double()
    assert abs(g.std().item() - 1) < 5e-3


def test_nvfp4_encoder_round_trip():
    z = datagen.normal_f64(9, 7, (4096, 64))
    packed, scale = datagen.nvfp4_encode(z)
    dec = oracle.nvfp4_decode(packed.numpy(), scale.numpy())
    zz = z.numpy().reshape(4096, 4, 16)
    s = oracle.e4m3_value(scale.numpy())
    err = np.abs(dec.reshape(4096, 4, 16) - zz)
    # RNE on the e2m1 grid: error at most half the widest gap (2) times the scale,
    # plus saturation when the scale rounded down
    amax = np.abs(zz).max(-1)
    bound = np.maximum(s, amax - 6 * s)[..., None] + 1e-12
    assert np.all(err <= bound)
    # the scale is the e4m3 rounding of amax / 6
    assert np.all(np.abs(s - amax / 6) <= amax / 6 * 2 ** -4 + 1e-12)
    # every code is used and the largest element lands near +-6 * scale
    codes = np.concatenate([packed.numpy() & 15, packed.numpy() >> 4]).ravel()
    assert set(np.unique(codes)) == set(range(16)) - {8} or set(np.unique(codes)) == set(range(16))


def test_random_index_lists():
    vis = torch.tensor([0, 1, 5, 16, 1000])
    idx = datagen.random_index_lists(1, 17, vis, 16)
    for r, v in enumerate(vis.tolist()):
        row = idx[r]
        sel = row[row >= 0]
        assert len(sel) == min(16, v)
        assert torch.all(sel < max(v, 1)) and torch.all(sel[1:] > sel[:-1])
        assert torch.all(row[len(sel):] == -1)
