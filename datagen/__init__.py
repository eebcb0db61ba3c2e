"""Seeded synthetic inputs for the hybrid compressed-attention path.

Shared by the CPU oracle's tests, the CUDA parity tests, the benchmark and
the smoke run.  It holds no step of the attention method: only a
counter-based bit generator, the quantile tables those bits index, an NVFP4
encoder that turns normal samples into quantised indexer keys, random index
lists for testing the sparse-attention call on its own, and the tensor
recipes of the workloads (``workloads.py``).

Every tensor is a pure function of (seed, tensor id, flat element index):

* bits  = mix32(mix32(index XOR key) XOR key2), where mix32 is the
  "lowbias32" integer hash published by C. Wellons (hash-prospector) and
  (key, key2) are derived from (seed, tensor id) with the same hash;
* N(0,1) samples = a 65536-entry table of normal quantiles,
  ndtri((u + 1/2) / 65536), indexed by the top 16 bits and rounded once to
  the target format on the host in fp64;
* U(0,1) samples = (top 24 bits + 1/2) / 2^24, exact in fp32.

Only int64 arithmetic (with no signed overflow) and table gathers run on the
device, so the bytes are identical on the CPU and on the GPU, and any row of
any tensor can be regenerated alone on the host for a sampled oracle check.
"""
from __future__ import annotations

import functools

import numpy as np
import torch
from scipy.special import ndtri

M32 = 0xFFFFFFFF
_CHUNK = 1 << 25  # elements generated per pass (bounds int64 temporaries)


# ---------------------------------------------------------------------------
# counter-based bits
# ---------------------------------------------------------------------------
def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for 0 <= x < 2^32 without int64 overflow."""
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & M32


def _mix32(x: torch.Tensor) -> torch.Tensor:
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _mix32_int(x: int) -> int:
    x &= M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & M32
    x ^= x >> 16
    return x


def _keys(seed: int, tid: int) -> tuple[int, int]:
    k1 = _mix32_int((seed * 0x9E3779B9 + tid * 0x632BE5AB + 0x1234567) & M32)
    k2 = _mix32_int(k1 ^ 0xA5A5A5A5 ^ (tid << 8))
    return k1, k2


def bits32(seed: int, tid: int, index: torch.Tensor) -> torch.Tensor:
    """32 random bits (as int64 in [0, 2^32)) for each flat element index."""
    index = index.to(torch.int64)
    if index.numel() and int(index.max()) > M32:
        raise ValueError("element index exceeds 2^32")
    k1, k2 = _keys(seed, tid)
    return _mix32(_mix32(index ^ k1) ^ k2)


# ---------------------------------------------------------------------------
# quantile tables (host fp64, then cached per device)
# ---------------------------------------------------------------------------
def _bf16_bits_rne(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bit patterns, round to nearest even (finite, normal range)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    r = np.rint(m * 256.0)  # 8 significant bits, ties to even
    v = np.ldexp(r, e - 8).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


@functools.lru_cache(maxsize=None)
def _quantiles_f64() -> np.ndarray:
    u = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
    return ndtri(u)


@functools.lru_cache(maxsize=None)
def _table(kind: str, scale: float, device: str) -> torch.Tensor:
    z = _quantiles_f64() * scale
    if kind == "bf16":
        t = torch.from_numpy(_bf16_bits_rne(z).view(np.int16).copy())
    elif kind == "f32":
        t = torch.from_numpy(z.astype(np.float32))
    elif kind == "f64":
        t = torch.from_numpy(z.copy())
    else:
        raise ValueError(kind)
    return t.to(device)


def _gen(seed, tid, numel, device, fn, out_dtype, offset=0):
    out = torch.empty(numel, dtype=out_dtype, device=device)
    for s in range(0, numel, _CHUNK):
        n = min(_CHUNK, numel - s)
        idx = torch.arange(offset + s, offset + s + n, dtype=torch.int64, device=device)
        out[s:s + n] = fn(bits32(seed, tid, idx))
    return out


def normal_bf16(seed, tid, shape, scale=1.0, device="cpu"):
    """bf16 tensor whose elements are RNE(scale * z), z a N(0,1) quantile."""
    shape = tuple(int(s) for s in shape)
    numel = int(np.prod(shape)) if shape else 1
    tab = _table("bf16", float(scale), str(device))
    out = _gen(seed, tid, numel, device, lambda b: tab[b >> 16], torch.int16)
    return out.view(torch.bfloat16).reshape(shape)


def normal_bf16_at(seed, tid, index, scale=1.0):
    """Same values as normal_bf16 at the given flat element indices."""
    tab = _table("bf16", float(scale), str(index.device))
    return tab[bits32(seed, tid, index) >> 16].view(torch.bfloat16)


def normal_f32(seed, tid, shape, device="cpu"):
    shape = tuple(int(s) for s in shape)
    numel = int(np.prod(shape)) if shape else 1
    tab = _table("f32", 1.0, str(device))
    return _gen(seed, tid, numel, device, lambda b: tab[b >> 16], torch.float32).reshape(shape)


def normal_f32_at(seed, tid, index):
    tab = _table("f32", 1.0, str(index.device))
    return tab[bits32(seed, tid, index) >> 16]


def normal_f64(seed, tid, shape, device="cpu"):
    shape = tuple(int(s) for s in shape)
    numel = int(np.prod(shape)) if shape else 1
    tab = _table("f64", 1.0, str(device))
    return _gen(seed, tid, numel, device, lambda b: tab[b >> 16], torch.float64).reshape(shape)


def uniform_f32(seed, tid, shape, device="cpu"):
    """U(0,1) fp32: (top 24 bits + 1/2) / 2^24, exact."""
    shape = tuple(int(s) for s in shape)
    numel = int(np.prod(shape)) if shape else 1
    fn = lambda b: ((b >> 8).to(torch.float64) + 0.5).mul(1.0 / 16777216.0).to(torch.float32)
    return _gen(seed, tid, numel, device, fn, torch.float32).reshape(shape)


def uniform_f32_at(seed, tid, index):
    b = bits32(seed, tid, index)
    return ((b >> 8).to(torch.float64) + 0.5).mul(1.0 / 16777216.0).to(torch.float32)


# ---------------------------------------------------------------------------
# NVFP4 encoder: e2m1 codes with one e4m3 scale per 16 consecutive elements
# ---------------------------------------------------------------------------
def _e4m3_round_pos(v: torch.Tensor) -> torch.Tensor:
    """Round positive fp64 values to the e4m3 grid (RNE, saturate at 448)."""
    sub = torch.round(v * 512.0) / 512.0  # subnormal grid, spacing 2^-9
    m, e = torch.frexp(v)  # v = m * 2^e, m in [0.5, 1)
    E = (e - 1).to(torch.float64)
    p = torch.pow(2.0, E)
    nrm = torch.round((v / p) * 8.0) / 8.0 * p
    q = torch.where(v < 2.0 ** -6, sub, nrm)
    return torch.clamp(q, max=448.0)


def _e4m3_bits_pos(q: torch.Tensor) -> torch.Tensor:
    """Bit patterns of positive values already on the e4m3 grid."""
    sub_bits = torch.round(q * 512.0)
    m, e = torch.frexp(torch.where(q > 0, q, torch.ones_like(q)))
    E = (e - 1).to(torch.float64)
    mant = torch.round((q / torch.pow(2.0, E) - 1.0) * 8.0)
    nrm_bits = (E + 7.0) * 8.0 + mant
    bits = torch.where(q < 2.0 ** -6, sub_bits, nrm_bits)
    return bits.to(torch.uint8)


def _e2m1_codes(y: torch.Tensor) -> torch.Tensor:
    """RNE of fp64 values onto {0,.5,1,1.5,2,3,4,6} (saturating); 4-bit codes."""
    a = y.abs()
    mag = ((a > 0.25).to(torch.int64) + (a >= 0.75) + (a > 1.25) + (a >= 1.75)
           + (a > 2.5) + (a >= 3.5) + (a > 5.0))
    sign = (y < 0).to(torch.int64) * 8
    return (mag + torch.where(mag > 0, sign, torch.zeros_like(sign))).to(torch.uint8)


def nvfp4_encode(x: torch.Tensor):
    """Quantise fp64 [..., D] (D % 16 == 0) to NVFP4.

    Returns (packed uint8 [..., D/2], scale uint8 [..., D/16]).  Element 2i
    of a row sits in the low nibble of byte i; the scale of each group of 16
    is e4m3(RNE(amax/6)), and the values are RNE onto the e2m1 grid after
    division by that scale.
    """
    D = x.shape[-1]
    assert D % 16 == 0
    g = x.reshape(*x.shape[:-1], D // 16, 16)
    amax = g.abs().amax(-1)
    s = _e4m3_round_pos(amax / 6.0)
    safe = torch.where(s > 0, s, torch.ones_like(s))
    y = torch.where(s[..., None] > 0, g / safe[..., None], torch.zeros_like(g))
    codes = _e2m1_codes(y).reshape(*x.shape[:-1], D).to(torch.int64)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).to(torch.uint8)
    return packed, _e4m3_bits_pos(s)


def nvfp4_normal(seed, tid, rows, dim, device="cpu", row0=0):
    """NVFP4 indexer keys for rows [row0, row0+rows) of a [*, dim] N(0,1) tensor."""
    packed = torch.empty((rows, dim // 2), dtype=torch.uint8, device=device)
    scale = torch.empty((rows, dim // 16), dtype=torch.uint8, device=device)
    tab = _table("f64", 1.0, str(device))
    step = max(1, _CHUNK // dim)
    for r in range(0, rows, step):
        n = min(step, rows - r)
        idx = torch.arange((row0 + r) * dim, (row0 + r + n) * dim, dtype=torch.int64, device=device)
        z = tab[bits32(seed, tid, idx) >> 16].reshape(n, dim)
        p, s = nvfp4_encode(z)
        packed[r:r + n] = p
        scale[r:r + n] = s
    return packed, scale


# ---------------------------------------------------------------------------
# random index lists (inputs for testing the sparse-attention call alone)
# ---------------------------------------------------------------------------
def random_index_lists(seed, tid, visible: torch.Tensor, k: int):
    """For each row r pick min(k, visible[r]) distinct indices in [0, visible[r]).

    Returns int32 [R, k], ascending, padded with -1.  Drawn by ranking the
    hash of (r, j) over j, so the result is identical on every device.
    """
    visible = visible.to(torch.int64)
    R = visible.numel()
    nmax = int(visible.max()) if R else 0
    out = torch.full((R, k), -1, dtype=torch.int32, device=visible.device)
    if nmax == 0:
        return out
    j = torch.arange(nmax, device=visible.device, dtype=torch.int64)
    for r0 in range(0, R, max(1, _CHUNK // max(nmax, 1))):
        r1 = min(R, r0 + max(1, _CHUNK // max(nmax, 1)))
        rows = torch.arange(r0, r1, device=visible.device, dtype=torch.int64)
        h = bits32(seed, tid, (rows[:, None] * nmax + j[None, :]) & M32)
        h = torch.where(j[None, :] < visible[r0:r1, None], h, torch.full_like(h, -1))
        top = torch.topk(h, min(k, nmax), dim=1).indices  # distinct keys: no ties
        cnt = torch.clamp(visible[r0:r1], max=k)
        sel = torch.where(torch.arange(top.shape[1], device=top.device)[None, :] < cnt[:, None],
                          top, torch.full_like(top, 1 << 40))
        sel = torch.sort(sel, dim=1).values
        sel = torch.where(sel == (1 << 40), torch.full_like(sel, -1), sel)
        out[r0:r1, :sel.shape[1]] = sel.to(torch.int32)
    return out


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a (CPU or GPU) bf16 tensor as numpy uint16."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
