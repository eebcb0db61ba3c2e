"""Tensor recipes of the five synthetic workloads.

Each workload is a frozen dataclass: its fields are the sizes, its ``make``
method generates every input tensor on a device, and ``rows`` regenerates a
subset of rows of one tensor on the host (for sampled oracle checks).  The
recipes hold no step of the method; layouts are row-major:

* raw K/V ``[B, R, D]`` bf16 (row r of batch b is absolute position
  ``raw_pos0 + r``), gate logits ``[B, R]`` fp32;
* compressed K/V ``[B, Ncap, D]`` bf16 (entry j covers positions
  ``[j*m, j*m + m - 1]``);
* queries ``[B, Tq, H, D]`` bf16, indexer queries ``[B, Tq, HI, DI]`` bf16,
  indexer head weights ``[B, Tq, HI]`` fp32;
* indexer keys ``[B, Ncap, DI]`` bf16, or NVFP4 packed ``[B, Ncap, DI/2]``
  uint8 plus e4m3 scales ``[B, Ncap, DI/16]`` uint8.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

from . import (normal_bf16, normal_bf16_at, normal_f32, normal_f32_at, normal_f64,
               nvfp4_normal, uniform_f32, uniform_f32_at)

# tensor ids (stable: changing one changes every input derived from it)
T_K, T_V, T_GATE, T_Q, T_QI, T_W, T_KI = 1, 2, 3, 4, 5, 6, 7
T_KC, T_VC, T_KR, T_VR = 8, 9, 10, 11
T_KC_H, T_VC_H, T_KR_H, T_VR_H, T_GATE_H = 12, 13, 14, 15, 16
T_IDX = 17
T_RQ, T_RQI, T_RW = 18, 19, 20

QSCALE_128 = 1.0 / math.sqrt(128.0)


def _rows_bf16(seed, tid, row_ids, row_len, scale=1.0):
    idx = (row_ids.to(torch.int64)[:, None] * row_len
           + torch.arange(row_len, dtype=torch.int64)[None, :])
    return normal_bf16_at(seed, tid, idx.reshape(-1), scale).reshape(-1, row_len)


@dataclass(frozen=True)
class TinyPrefill:
    """2048-token CSA+HCA prefill: 8 query heads of dim 64 share one KV head."""
    seed: int = 0
    B: int = 1
    T: int = 2048
    H: int = 8
    D: int = 64
    m_csa: int = 4
    m_hca: int = 128
    HI: int = 4
    DI: int = 32
    k: int = 16
    W: int = 32
    q_scale: float = 1.0 / 8.0

    @property
    def n_csa(self):
        return self.T // self.m_csa

    @property
    def n_hca(self):
        return self.T // self.m_hca

    def make(self, device="cpu"):
        s, B, T = self.seed, self.B, self.T
        return dict(
            K=normal_bf16(s, T_K, (B, T, self.D), device=device),
            V=normal_bf16(s, T_V, (B, T, self.D), device=device),
            gate=normal_f32(s, T_GATE, (B, T), device=device),
            q=normal_bf16(s, T_Q, (B, T, self.H, self.D), self.q_scale, device=device),
            qI=normal_bf16(s, T_QI, (B, T, self.HI, self.DI), device=device),
            w=uniform_f32(s, T_W, (B, T, self.HI), device=device),
            kI=normal_bf16(s, T_KI, (B, self.n_csa, self.DI), device=device),
        )


@dataclass(frozen=True)
class CsaDecode:
    """CSA decode: 32 sequences, 65536-token context, 16384 precompressed entries."""
    seed: int = 1
    B: int = 32
    ctx: int = 65536
    N: int = 16384
    D: int = 128
    H: int = 64
    HI: int = 8
    DI: int = 64
    k: int = 128
    W: int = 128
    m: int = 4
    q_scale: float = QSCALE_128

    @property
    def q_pos(self):
        return self.ctx - 1

    @property
    def raw_pos0(self):
        return self.ctx - self.W

    def make(self, device="cpu", rot=0):
        s = self.seed + 7919 * rot
        B, N = self.B, self.N
        return dict(
            Kc=normal_bf16(s, T_KC, (B, N, self.D), device=device),
            Vc=normal_bf16(s, T_VC, (B, N, self.D), device=device),
            kI=normal_bf16(s, T_KI, (B, N, self.DI), device=device),
            Kr=normal_bf16(s, T_KR, (B, self.W, self.D), device=device),
            Vr=normal_bf16(s, T_VR, (B, self.W, self.D), device=device),
            q=normal_bf16(s, T_Q, (B, 1, self.H, self.D), self.q_scale, device=device),
            qI=normal_bf16(s, T_QI, (B, 1, self.HI, self.DI), device=device),
            w=uniform_f32(s, T_W, (B, 1, self.HI), device=device),
        )


@dataclass(frozen=True)
class DsaDecode:
    """The DSA comparator of the CSA decode: the same 32 sequences and 65536-token
    context, but every raw token is its own entry (m = 1), so the indexer scores
    all 65536 tokens; the window rows are the cache's last W rows."""
    seed: int = 5
    B: int = 32
    ctx: int = 65536
    D: int = 128
    H: int = 64
    HI: int = 8
    DI: int = 64
    k: int = 128
    W: int = 128
    m: int = 1
    q_scale: float = QSCALE_128

    @property
    def N(self):
        return self.ctx // self.m

    @property
    def q_pos(self):
        return self.ctx - 1

    @property
    def raw_pos0(self):
        return self.ctx - self.W

    def make(self, device="cpu", rot=0):
        s = self.seed + 7919 * rot
        B, N = self.B, self.N
        Kc = normal_bf16(s, T_KC, (B, N, self.D), device=device)
        Vc = normal_bf16(s, T_VC, (B, N, self.D), device=device)
        return dict(
            Kc=Kc, Vc=Vc,
            kI=normal_bf16(s, T_KI, (B, N, self.DI), device=device),
            Kr=Kc[:, N - self.W:].contiguous(),
            Vr=Vc[:, N - self.W:].contiguous(),
            q=normal_bf16(s, T_Q, (B, 1, self.H, self.D), self.q_scale, device=device),
            qI=normal_bf16(s, T_QI, (B, 1, self.HI, self.DI), device=device),
            w=uniform_f32(s, T_W, (B, 1, self.HI), device=device),
        )


@dataclass(frozen=True)
class CsaPrefill:
    """CSA prefill of one 131072-token sequence, processed in 4096-query chunks."""
    seed: int = 2
    B: int = 1
    T: int = 131072
    chunk: int = 4096
    D: int = 128
    H: int = 64
    HI: int = 8
    DI: int = 64
    k: int = 128
    W: int = 128
    m: int = 4
    q_scale: float = QSCALE_128

    @property
    def N(self):
        return self.T // self.m

    def make(self, device="cpu", with_q=True):
        s, B, T = self.seed, self.B, self.T
        d = dict(
            K=normal_bf16(s, T_K, (B, T, self.D), device=device),
            V=normal_bf16(s, T_V, (B, T, self.D), device=device),
            gate=normal_f32(s, T_GATE, (B, T), device=device),
            qI=normal_bf16(s, T_QI, (B, T, self.HI, self.DI), device=device),
            w=uniform_f32(s, T_W, (B, T, self.HI), device=device),
            kI=normal_bf16(s, T_KI, (B, self.N, self.DI), device=device),
        )
        if with_q:
            d["q"] = normal_bf16(s, T_Q, (B, T, self.H, self.D), self.q_scale, device=device)
        return d

    def q_rows(self, t_ids):
        """Queries of absolute positions t_ids (batch 0) on the host: [n, H, D]."""
        r = _rows_bf16(self.seed, T_Q, torch.as_tensor(t_ids), self.H * self.D, self.q_scale)
        return r.reshape(-1, self.H, self.D)


@dataclass(frozen=True)
class HcaDecode:
    """HCA decode at 1M context: 8 sequences, 8192 entries of m=128 each."""
    seed: int = 3
    B: int = 8
    ctx: int = 1048576
    N: int = 8192
    D: int = 128
    H: int = 64
    W: int = 128
    m: int = 128
    q_scale: float = QSCALE_128

    @property
    def q_pos(self):
        return self.ctx - 1

    @property
    def raw_pos0(self):
        return self.ctx - self.W

    def make(self, device="cpu", rot=0):
        s = self.seed + 7919 * rot
        B = self.B
        return dict(
            Kc=normal_bf16(s, T_KC_H, (B, self.N, self.D), device=device),
            Vc=normal_bf16(s, T_VC_H, (B, self.N, self.D), device=device),
            Kr=normal_bf16(s, T_KR_H, (B, self.W, self.D), device=device),
            Vr=normal_bf16(s, T_VR_H, (B, self.W, self.D), device=device),
            q=normal_bf16(s, T_Q, (B, 1, self.H, self.D), self.q_scale, device=device),
        )


@dataclass(frozen=True)
class HcaPrefill:
    """A 32768-token chunk appended to a 1M-token context (8192 m=128 entries).

    The raw buffer holds the W-1 tokens before the chunk, then the chunk;
    hca_compress pools the chunk's 256 blocks into entries 8192..8447.
    """
    seed: int = 3
    B: int = 1
    ctx: int = 1048576
    Tc: int = 32768
    N0: int = 8192
    D: int = 128
    H: int = 64
    W: int = 128
    m: int = 128
    q_scale: float = QSCALE_128

    @property
    def Ncap(self):
        return self.N0 + self.Tc // self.m

    @property
    def R(self):
        return self.W - 1 + self.Tc

    @property
    def raw_pos0(self):
        return self.ctx - (self.W - 1)

    @property
    def q_pos0(self):
        return self.ctx

    def make(self, device="cpu", with_q=True):
        s, B = self.seed + 101, self.B
        Kc = torch.zeros((B, self.Ncap, self.D), dtype=torch.bfloat16, device=device)
        Vc = torch.zeros_like(Kc)
        Kc[:, :self.N0] = normal_bf16(s, T_KC_H, (B, self.N0, self.D), device=device)
        Vc[:, :self.N0] = normal_bf16(s, T_VC_H, (B, self.N0, self.D), device=device)
        d = dict(
            Kc=Kc, Vc=Vc,
            Kr=normal_bf16(s, T_KR_H, (B, self.R, self.D), device=device),
            Vr=normal_bf16(s, T_VR_H, (B, self.R, self.D), device=device),
            gate=normal_f32(s, T_GATE_H, (B, self.R), device=device),
        )
        if with_q:
            d["q"] = normal_bf16(s, T_Q, (B, self.Tc, self.H, self.D), self.q_scale, device=device)
        return d

    def q_rows(self, i_ids):
        """Queries of chunk rows i_ids (batch 0) on the host: [n, H, D]."""
        r = _rows_bf16(self.seed + 101, T_Q, torch.as_tensor(i_ids), self.H * self.D, self.q_scale)
        return r.reshape(-1, self.H, self.D)


@dataclass(frozen=True)
class PairDecode:
    """Interleaved CSA/HCA layer pair, decode from a 1M-token context.

    Each layer has its own raw buffer (``[B, W + steps, D]``, rows from
    position ctx - W), compressed K/V and, for CSA, NVFP4 indexer keys for
    every entry that exists or will be pooled during the run.  Step s feeds
    one new token at position ctx + s to both layers; both layers attend with
    the same query heads.
    """
    seed: int = 4
    B: int = 4
    ctx: int = 1048576
    steps: int = 64
    D: int = 128
    H: int = 64
    HI: int = 8
    DI: int = 64
    k: int = 128
    W: int = 128
    m_csa: int = 4
    m_hca: int = 128
    q_scale: float = QSCALE_128

    @property
    def N_csa(self):
        return self.ctx // self.m_csa

    @property
    def Ncap_csa(self):
        return (self.ctx + self.steps) // self.m_csa

    @property
    def N_hca(self):
        return self.ctx // self.m_hca

    @property
    def R(self):
        return self.W + self.steps

    @property
    def raw_pos0(self):
        return self.ctx - self.W

    def make(self, device="cpu"):
        s, B, D = self.seed, self.B, self.D
        Kc = torch.zeros((B, self.Ncap_csa, D), dtype=torch.bfloat16, device=device)
        Vc = torch.zeros_like(Kc)
        Kc[:, :self.N_csa] = normal_bf16(s, T_KC, (B, self.N_csa, D), device=device)
        Vc[:, :self.N_csa] = normal_bf16(s, T_VC, (B, self.N_csa, D), device=device)
        kp, ks = nvfp4_normal(s, T_KI, B * self.Ncap_csa, self.DI, device=device)
        return dict(
            Kc=Kc, Vc=Vc,
            kI_packed=kp.reshape(B, self.Ncap_csa, self.DI // 2),
            kI_scale=ks.reshape(B, self.Ncap_csa, self.DI // 16),
            Kr=normal_bf16(s, T_KR, (B, self.R, D), device=device),
            Vr=normal_bf16(s, T_VR, (B, self.R, D), device=device),
            gate=normal_f32(s, T_GATE, (B, self.R), device=device),
            gate_h=normal_f32(s, T_GATE_H, (B, self.R), device=device),
            Kc_h=normal_bf16(s, T_KC_H, (B, self.N_hca, D), device=device),
            Vc_h=normal_bf16(s, T_VC_H, (B, self.N_hca, D), device=device),
            Kr_h=normal_bf16(s, T_KR_H, (B, self.R, D), device=device),
            Vr_h=normal_bf16(s, T_VR_H, (B, self.R, D), device=device),
            q=normal_bf16(s, T_Q, (self.steps, B, self.H, D), self.q_scale, device=device),
            qI=normal_bf16(s, T_QI, (self.steps, B, self.HI, self.DI), device=device),
            w=uniform_f32(s, T_W, (self.steps, B, self.HI), device=device),
        )

    def make_replay(self, R, device="cpu"):
        """Queries of the last R context tokens (positions ctx-R .. ctx-1), [R, B, ...]:
        the inputs of a bounded replay of the window state."""
        s, B = self.seed, self.B
        return dict(
            rq=normal_bf16(s, T_RQ, (R, B, self.H, self.D), self.q_scale, device=device),
            rqI=normal_bf16(s, T_RQI, (R, B, self.HI, self.DI), device=device),
            rw=uniform_f32(s, T_RW, (R, B, self.HI), device=device),
        )


WORKLOADS = {
    "tiny_prefill": TinyPrefill,
    "csa_decode": CsaDecode,
    "dsa_decode": DsaDecode,
    "csa_prefill": CsaPrefill,
    "hca_decode": HcaDecode,
    "hca_prefill": HcaPrefill,
    "pair_decode": PairDecode,
}
