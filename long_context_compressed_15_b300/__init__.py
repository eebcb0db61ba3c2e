"""Python binding of liblcc.so, the B300 hybrid compressed-attention library.

Argument marshalling only: every function checks shapes, dtypes and
devices of torch tensors, passes their device pointers and the current CUDA
stream to the C function of the same name (``lcc_<name>`` in include/lcc.h)
and raises :class:`LccError` on a non-OK status.  All computation happens
in the library's CUDA kernels; there is no fallback path -- importing works
without a GPU, but every call needs the built ``liblcc.so`` and a CUDA
device.  PyTorch supplies device memory (outputs and workspace are
allocated here when the caller does not pass them) and streams.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "LccError", "load", "qkv_prologue", "csa_compress", "hca_compress", "compress", "decode_append", "lightning_index_topk", "lightning_index_scores",
    "lightning_index_topk_noalloc", "lightning_reindex_topk",
    "index_topk_workspace", "csa_sparse_attn", "hca_dense_attn", "dense_attn_workspace",
    "swa_attn", "attn_merge", "csa_layer_attn", "hca_layer_attn", "layer_attn_workspace", "csa_layer",
    "csa_layer_workspace",
    "sync_status", "last_error", "KEY_BF16", "KEY_NVFP4",
]

KEY_BF16, KEY_NVFP4 = 0, 1
_STATUS = {0: "OK", 1: "ERR_ARG", 2: "ERR_SHAPE", 3: "ERR_ALIGN", 4: "ERR_UNSUPPORTED",
           5: "ERR_CUDA", 6: "ERR_TIMEOUT", 7: "ERR_DEVICE", 8: "ERR_WORKSPACE"}
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liblcc.so")

_lib = None
_P, _I, _L, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t

# name -> argument types (return type is int status unless listed in _RET)
_SIGS = {
    "lcc_csa_compress": [_P, _P, _P, _I, _I, _I, _L, _L, _P, _P, _L, _P],
    "lcc_hca_compress": [_P, _P, _P, _I, _I, _I, _L, _L, _P, _P, _L, _P],
    "lcc_compress": [_I, _P, _P, _P, _I, _I, _I, _L, _L, _P, _P, _L, _P],
    "lcc_compress_at": [_I, _P, _P, _P, _I, _I, _I, _L, _L, _P, _P, _P, _I, _L, _P, _P],
    "lcc_decode_append": [_I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _L, _L, _I, _P, _P, _P, _L, _I, _P, _I, _I,
                          _P, _P, _P, _P, _P],
    "lcc_qkv_prologue": [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _F, _I, _F, _P, _P, _P, _P, _P],
    "lcc_lightning_reindex_topk": [_P, _P, _I, _I, _I, _I, _I, _P, _P, _I, _P, _I, _I, _P, _P, _P],
    "lcc_index_topk_workspace": [_I, _I, _I, _I],
    "lcc_lightning_index_topk": [_P, _P, _I, _I, _I, _I, _P, _I, _P, _P, _P, _I, _I, _I, _P, _P, _P, _Z, _P],
    "lcc_lightning_index_topk_noalloc": [_P, _P, _I, _I, _I, _I, _P, _I, _P, _P, _P, _I, _I, _I, _P, _P, _P],
    "lcc_nvfp4_quantize": [_P, _L, _I, _L, _P, _P, _P, _P],
    "lcc_nvfp4_dequantize": [_P, _P, _L, _I, _P, _P],
    "lcc_fp4_index_topk_workspace": [_I, _I, _I, _I, _I, _I],
    "lcc_fp4_index_topk": [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _Z, _P],
    "lcc_lightning_index_scores": [_P, _P, _I, _I, _I, _I, _P, _I, _P, _P, _P, _I, _I, _P, _P],
    "lcc_csa_sparse_attn": [_P, _I, _I, _I, _I, _F, _P, _P, _L, _I, _P, _I, _P, _P, _P],
    "lcc_dense_attn_workspace": [_I, _I, _I, _I, _I],
    "lcc_hca_dense_attn": [_P, _I, _I, _I, _I, _F, _P, _P, _P, _L, _I, _P, _I, _P, _P, _P, _Z, _P],
    "lcc_swa_attn": [_P, _I, _I, _I, _I, _F, _P, _P, _P, _L, _I, _P, _I, _P, _P, _P],
    "lcc_attn_merge": [_I, _P, _P, _L, _I, _P, _P, _P, _P],
    "lcc_layer_attn_workspace": [_I, _I, _I, _I, _I],
    "lcc_csa_layer_workspace": [_I, _I, _I, _I, _I, _I, _I],
    "lcc_csa_layer": [_P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _I, _P, _P, _P, _P, _P, _L, _I, _I, _I,
                      _P, _P, _L, _I, _P, _I, _P, _P, _P, _P, _Z, _P],
    "lcc_csa_layer_attn": [_P, _I, _I, _I, _I, _F, _P, _P, _P, _L, _I, _P, _I, _P, _P, _L, _I, _P, _I,
                           _P, _P, _P, _Z, _P],
    "lcc_hca_layer_attn": [_P, _I, _I, _I, _I, _F, _P, _P, _P, _L, _I, _P, _I, _P, _P, _L, _I, _P, _I,
                           _P, _P, _P, _Z, _P],
    "lcc_last_error": [],
    "lcc_version": [],
    "lcc_sync_status": [_P],
    "lcc_launch_count": [],
    "lcc_test_set_wait_fault": [ctypes.c_uint64, _I],
}
_RET = {"lcc_index_topk_workspace": _Z, "lcc_fp4_index_topk_workspace": _Z, "lcc_dense_attn_workspace": _Z, "lcc_layer_attn_workspace": _Z, "lcc_csa_layer_workspace": _Z,
        "lcc_last_error": ctypes.c_char_p, "lcc_version": ctypes.c_char_p, "lcc_launch_count": ctypes.c_uint64}


class LccError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: {_STATUS.get(status, status)}: {msg}")
        self.status = status


def load(path: str | None = None):
    """Load liblcc.so (once).  Raises if the library has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"liblcc.so not found at {p}: build it with "
                           "`python -m long_context_compressed_15_b300.build`")
    lib = ctypes.CDLL(p)
    for name, args in _SIGS.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = _RET.get(name, ctypes.c_int)
    _lib = lib
    return lib


def launch_count() -> int:
    """Kernels enqueued by the library so far (graph captures count once)."""
    return int(load().lcc_launch_count())


def last_error() -> str:
    return load().lcc_last_error().decode()


def _call(name, *args):
    lib = load()
    st = getattr(lib, name)(*args)
    if st != 0:
        raise LccError(name, st, lib.lcc_last_error().decode())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(t, dtype, name, dim=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims, got shape {tuple(t.shape)}")


def _rows(t, name):
    """[B, R, D] with unit element stride and contiguous rows; returns (batch stride, row stride)."""
    if t.stride(2) != 1:
        raise ValueError(f"{name}: last dim must be contiguous")
    return t.stride(0), t.stride(1)


def _positions(x, B, device, dtype=torch.int64):
    if isinstance(x, torch.Tensor):
        _need(x, dtype, "positions")
        return x
    return torch.full((B,), int(x), dtype=dtype, device=device)


# ---------------------------------------------------------------------------
# query / KV prologue
# ---------------------------------------------------------------------------
def qkv_prologue(q, k, v, gamma_q, gamma_k, gamma_v, pos0, d_rope=64, eps=1e-6, rope_base=10000.0,
                 q_out=None, k_out=None, v_out=None, stream=None):
    """RMSNorm of q [B, T, H, D], k and v [B, T, D] (bf16) with gains [D] fp32, then
    rotary embedding of the last d_rope channels of q and k at positions pos0 + t.
    v (with gamma_v) may be None.  Outputs default to new tensors; pass the inputs
    to work in place.  Returns (q_out, k_out, v_out)."""
    _need(q, torch.bfloat16, "q", 4)
    _need(k, torch.bfloat16, "k", 3)
    B, T, H, D = q.shape
    for t, n in ((gamma_q, "gamma_q"), (gamma_k, "gamma_k")):
        _need(t, torch.float32, n, 1)
    if v is not None:
        _need(v, torch.bfloat16, "v", 3)
        _need(gamma_v, torch.float32, "gamma_v", 1)
    if not (q.is_contiguous() and k.is_contiguous() and (v is None or v.is_contiguous())):
        raise ValueError("q, k and v must be contiguous")
    q_out = torch.empty_like(q) if q_out is None else q_out
    k_out = torch.empty_like(k) if k_out is None else k_out
    if v is not None and v_out is None:
        v_out = torch.empty_like(v)
    pos0 = _positions(pos0, B, q.device)
    _call("lcc_qkv_prologue", _ptr(q), _ptr(k), _ptr(v), B, T, H, D, _ptr(gamma_q), _ptr(gamma_k), _ptr(gamma_v),
          float(eps), int(d_rope), float(rope_base), _ptr(pos0), _ptr(q_out), _ptr(k_out), _ptr(v_out),
          _stream(stream))
    return q_out, k_out, v_out


# ---------------------------------------------------------------------------
# compression
# ---------------------------------------------------------------------------
def _compress(fname, m, K, V, gate, Kc, Vc, n_blocks, stream, pass_m=False):
    for t, n in ((K, "K"), (V, "V"), (Kc, "Kc"), (Vc, "Vc")):
        _need(t, torch.bfloat16, n, 3)
    _need(gate, torch.float32, "gate", 2)
    B, R, D = K.shape
    kv_bs, kv_rs = _rows(K, "K")
    if kv_rs != D or V.stride() != K.stride() or gate.stride(1) != 1:
        raise ValueError("K/V rows must be contiguous with identical strides; gate contiguous per batch")
    c_bs, c_rs = _rows(Kc, "Kc")
    if c_rs != D or Vc.stride() != Kc.stride():
        raise ValueError("Kc/Vc rows must be contiguous with identical strides")
    n_blocks = R // m if n_blocks is None else int(n_blocks)
    if n_blocks > Kc.shape[1] or n_blocks * m > R:
        raise ValueError("n_blocks exceeds the input rows or the output entries")
    args = (_ptr(K), _ptr(V), _ptr(gate), B, n_blocks, D, kv_bs, gate.stride(0), _ptr(Kc), _ptr(Vc), c_bs,
            _stream(stream))
    _call(fname, *(((int(m),) + args) if pass_m else args))
    return Kc, Vc


def csa_compress(K, V, gate, Kc, Vc, n_blocks=None, stream=None):
    """Pool every 4 tokens of K/V [B, R, D] into entries of Kc/Vc [B, N, D]."""
    return _compress("lcc_csa_compress", 4, K, V, gate, Kc, Vc, n_blocks, stream)


def hca_compress(K, V, gate, Kc, Vc, n_blocks=None, stream=None):
    """Pool every 128 tokens of K/V [B, R, D] into entries of Kc/Vc [B, N, D]."""
    return _compress("lcc_hca_compress", 128, K, V, gate, Kc, Vc, n_blocks, stream)


def compress(m, K, V, gate, Kc, Vc, n_blocks=None, stream=None):
    """Pool every m in {1, 4, 128} tokens of K/V [B, R, D] into Kc/Vc [B, N, D] (m = 1: a copy)."""
    return _compress("lcc_compress", m, K, V, gate, Kc, Vc, n_blocks, stream, pass_m=True)


def compress_at(m, K, V, gate, tok0, Kc, Vc, n_valid=None, n_tokens=None, stream=None):
    """Pool the complete blocks of K/V [B, R, D] (rows = tokens tok0[b] ..) into entries tok0[b]/m .. of
    Kc/Vc [B, Ncap, D], raising n_valid [B] (int32, optional) on the device (lcc_compress_at)."""
    for t, n in ((K, "K"), (V, "V"), (Kc, "Kc"), (Vc, "Vc")):
        _need(t, torch.bfloat16, n, 3)
    _need(gate, torch.float32, "gate", 2)
    B, R, D = K.shape
    kv_bs, kv_rs = _rows(K, "K")
    if kv_rs != D or V.stride() != K.stride() or gate.stride(1) != 1:
        raise ValueError("K/V rows must be contiguous with identical strides; gate contiguous per batch")
    c_bs, c_rs = _rows(Kc, "Kc")
    if c_rs != D or Vc.stride() != Kc.stride():
        raise ValueError("Kc/Vc rows must be contiguous with identical strides")
    n_tokens = R if n_tokens is None else int(n_tokens)
    if n_tokens > R:
        raise ValueError("n_tokens exceeds the input rows")
    tok0 = _positions(tok0, B, K.device)
    if n_valid is not None:
        _need(n_valid, torch.int32, "n_valid", 1)
    _call("lcc_compress_at", int(m), _ptr(K), _ptr(V), _ptr(gate), B, n_tokens, D, kv_bs, gate.stride(0),
          _ptr(tok0), _ptr(Kc), _ptr(Vc), Kc.shape[1], c_bs, _ptr(n_valid), _stream(stream))
    return Kc, Vc


def decode_append(m, k_new, v_new, g_new, pos, Kr, Vr, gate_r, raw_pos0, Kc, Vc, n_valid,
                  kI_new=None, kI=None, kI_scale_new=None, kI_scale=None, stream=None):
    """One decode step of one layer's caches (lcc_decode_append).

    The new tokens (k_new, v_new [B, D] bf16, g_new [B] fp32, at positions pos
    [B] int64) go to raw row pos - raw_pos0 of Kr/Vr [B, Rcap, D] and gate_r
    [B, Rcap]; a token that completes a block of m pools it into Kc/Vc
    [B, Ncap, D], copies kI_new [B, DI] (bf16, or NVFP4 uint8 [B, DI/2] with
    kI_scale_new [B, DI/16]) into kI/kI_scale and sets n_valid [B] (int32).
    pos, raw_pos0 and n_valid must be device tensors for graph capture.
    """
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, torch.bfloat16, n, 2)
    _need(g_new, torch.float32, "g_new", 1)
    for t, n in ((Kr, "Kr"), (Vr, "Vr"), (Kc, "Kc"), (Vc, "Vc")):
        _need(t, torch.bfloat16, n, 3)
    _need(gate_r, torch.float32, "gate_r", 2)
    B, D = k_new.shape
    if not (k_new.is_contiguous() and v_new.is_contiguous() and g_new.is_contiguous()):
        raise ValueError("k_new, v_new and g_new must be contiguous")
    r_bs, r_rs = _rows(Kr, "Kr")
    c_bs, c_rs = _rows(Kc, "Kc")
    if r_rs != D or Vr.stride() != Kr.stride() or c_rs != D or Vc.stride() != Kc.stride() or gate_r.stride(1) != 1:
        raise ValueError("raw and compressed rows must be contiguous with identical K/V strides")
    dev = k_new.device
    pos = _positions(pos, B, dev)
    raw_pos0 = _positions(raw_pos0, B, dev)
    _need(n_valid, torch.int32, "n_valid", 1)
    fmt, DI = KEY_BF16, 0
    if kI_new is not None:
        if kI is None:
            raise ValueError("kI_new needs kI")
        if kI_new.dtype == torch.uint8:
            fmt, DI = KEY_NVFP4, kI_new.shape[1] * 2
            if kI_scale_new is None or kI_scale is None:
                raise ValueError("NVFP4 keys need kI_scale_new and kI_scale")
        else:
            _need(kI_new, torch.bfloat16, "kI_new", 2)
            DI = kI_new.shape[1]
        if not (kI_new.is_contiguous() and kI.is_contiguous()):
            raise ValueError("kI_new and kI must be contiguous")
    _call("lcc_decode_append", int(m), B, D, _ptr(k_new), _ptr(v_new), _ptr(g_new), _ptr(pos), _ptr(Kr), _ptr(Vr),
          _ptr(gate_r), r_bs, gate_r.stride(0), Kr.shape[1], _ptr(raw_pos0), _ptr(Kc), _ptr(Vc), c_bs, Kc.shape[1],
          _ptr(n_valid), fmt, DI, _ptr(kI_new), _ptr(kI_scale_new), _ptr(kI), _ptr(kI_scale), _stream(stream))


# ---------------------------------------------------------------------------
# lightning indexer + top-k
# ---------------------------------------------------------------------------
def index_topk_workspace(B, Tq, Ncap, k) -> int:
    return int(load().lcc_index_topk_workspace(B, Tq, Ncap, k))


def lightning_index_topk(qI, w, q_pos0, kI, n_valid, m, k, kI_scale=None, idx=None, score=None,
                         workspace=None, stream=None):
    """Top-k compressed entries per query by the ReLU-weighted indexer score.

    qI [B, Tq, HI, DI] bf16; w [B, Tq, HI] fp32; kI [B, Ncap, DI] bf16, or
    NVFP4 packed uint8 [B, Ncap, DI/2] with kI_scale uint8 [B, Ncap, DI/16];
    q_pos0 / n_valid: int or [B] device tensors.  Returns idx [B, Tq, k] int32
    (and writes score [B, Tq, k] fp32 if given).
    """
    _need(qI, torch.bfloat16, "qI", 4)
    _need(w, torch.float32, "w", 3)
    B, Tq, HI, DI = qI.shape
    if not (qI.is_contiguous() and w.is_contiguous() and kI.is_contiguous()):
        raise ValueError("qI, w and kI must be contiguous")
    if kI.dtype == torch.uint8:
        fmt = KEY_NVFP4
        _need(kI_scale, torch.uint8, "kI_scale", 3)
        if not kI_scale.is_contiguous():
            raise ValueError("kI_scale must be contiguous")
    else:
        fmt = KEY_BF16
        _need(kI, torch.bfloat16, "kI", 3)
    Ncap = kI.shape[1]
    dev = qI.device
    q_pos0 = _positions(q_pos0, B, dev)
    n_valid = _positions(n_valid, B, dev, torch.int32)
    if idx is None:
        idx = torch.empty((B, Tq, k), dtype=torch.int32, device=dev)
    _need(idx, torch.int32, "idx", 3)
    if score is not None:
        _need(score, torch.float32, "score", 3)
    need = index_topk_workspace(B, Tq, Ncap, k)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _call("lcc_lightning_index_topk", _ptr(qI), _ptr(w), B, Tq, HI, DI, _ptr(q_pos0), fmt, _ptr(kI),
          _ptr(kI_scale), _ptr(n_valid), Ncap, int(m), int(k), _ptr(idx), _ptr(score),
          _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    return idx


def nvfp4_quantize(x, packed=None, scale=None, xq=None, stream=None):
    """NVFP4 quantisation of the rows of x [..., D] bf16 (D % 16 == 0, rows may
    be strided): per group of 16, scale = e4m3 nearest to amax/6 and codes =
    e2m1 nearest to x/scale (ties to even, saturating).  Returns (packed uint8
    [..., D/2], scale uint8 [..., D/16], xq bf16 [..., D] dequantised)."""
    _need(x, torch.bfloat16, "x")
    D = x.shape[-1]
    rows = x.numel() // D if D else 0
    x2 = x.reshape(rows, D) if x.dim() != 2 else x
    if x2.stride(1) != 1:
        raise ValueError("x rows must be contiguous in their last dimension")
    lead = tuple(x.shape[:-1])
    dev = x.device
    if packed is None:
        packed = torch.empty(lead + (D // 2,), dtype=torch.uint8, device=dev)
    if scale is None:
        scale = torch.empty(lead + (D // 16,), dtype=torch.uint8, device=dev)
    if xq is None:
        xq = torch.empty(lead + (D,), dtype=torch.bfloat16, device=dev)
    for t, n in ((packed, "packed"), (scale, "scale"), (xq, "xq")):
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    _call("lcc_nvfp4_quantize", _ptr(x2), rows, D, x2.stride(0) if rows else D, _ptr(packed), _ptr(scale),
          _ptr(xq), _stream(stream))
    return packed, scale, xq


def nvfp4_dequantize(packed, scale, out=None, stream=None):
    """NVFP4 rows (packed uint8 [..., D/2], scale uint8 [..., D/16]) -> bf16 [..., D] (exact)."""
    _need(packed, torch.uint8, "packed")
    _need(scale, torch.uint8, "scale")
    if not (packed.is_contiguous() and scale.is_contiguous()):
        raise ValueError("packed and scale must be contiguous")
    D = packed.shape[-1] * 2
    rows = packed.numel() // packed.shape[-1] if packed.shape[-1] else 0
    if out is None:
        out = torch.empty(tuple(packed.shape[:-1]) + (D,), dtype=torch.bfloat16, device=packed.device)
    _call("lcc_nvfp4_dequantize", _ptr(packed), _ptr(scale), rows, D, _ptr(out), _stream(stream))
    return out


def fp4_index_topk_workspace(B, Tq, HI, DI, Ncap, k) -> int:
    return int(load().lcc_fp4_index_topk_workspace(B, Tq, HI, DI, Ncap, k))


def fp4_index_topk(qI, w, q_pos0, kI, kI_scale, n_valid, m, k, idx=None, score=None, workspace=None, stream=None):
    """The lightning indexer in FP4: qI [B, Tq, 8, 64] bf16 is quantised to NVFP4
    (nvfp4_quantize's rule) and scored against the NVFP4 keys kI [B, Ncap, 32]
    uint8 / kI_scale [B, Ncap, 4]; otherwise as lightning_index_topk.  Returns
    idx [B, Tq, k] int32 (and writes score [B, Tq, k] fp32 if given)."""
    _need(qI, torch.bfloat16, "qI", 4)
    _need(w, torch.float32, "w", 3)
    _need(kI, torch.uint8, "kI", 3)
    _need(kI_scale, torch.uint8, "kI_scale", 3)
    if not (qI.is_contiguous() and w.is_contiguous() and kI.is_contiguous() and kI_scale.is_contiguous()):
        raise ValueError("qI, w, kI and kI_scale must be contiguous")
    B, Tq, HI, DI = qI.shape
    Ncap = kI.shape[1]
    dev = qI.device
    q_pos0 = _positions(q_pos0, B, dev)
    n_valid = _positions(n_valid, B, dev, torch.int32)
    if idx is None:
        idx = torch.empty((B, Tq, k), dtype=torch.int32, device=dev)
    _need(idx, torch.int32, "idx", 3)
    if score is not None:
        _need(score, torch.float32, "score", 3)
    need = fp4_index_topk_workspace(B, Tq, HI, DI, Ncap, k)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _call("lcc_fp4_index_topk", _ptr(qI), _ptr(w), B, Tq, HI, DI, _ptr(q_pos0), _ptr(kI), _ptr(kI_scale),
          _ptr(n_valid), Ncap, int(m), int(k), _ptr(idx), _ptr(score), _ptr(workspace),
          workspace.numel() * workspace.element_size(), _stream(stream))
    return idx


def lightning_index_topk_noalloc(qI, w, q_pos0, kI, n_valid, m, k, kI_scale=None, idx=None, score=None,
                                 stream=None):
    """lightning_index_topk without a workspace, for callers that cannot allocate device memory.

    The library keeps its scratch in a fixed 8 MiB device array shared by all
    calls (overlapping calls race; make the first call on a device before any
    graph capture); prefill-shaped requests (bf16 keys, Tq*HI > 16, k <= 256)
    take the fused top-k and use no scratch.  idx must be passed in so that
    nothing is allocated here.
    """
    _need(qI, torch.bfloat16, "qI", 4)
    _need(w, torch.float32, "w", 3)
    _need(idx, torch.int32, "idx", 3)
    B, Tq, HI, DI = qI.shape
    fmt = KEY_NVFP4 if kI.dtype == torch.uint8 else KEY_BF16
    if not isinstance(q_pos0, torch.Tensor) or not isinstance(n_valid, torch.Tensor):
        raise ValueError("q_pos0 and n_valid must be device tensors (nothing is allocated here)")
    _call("lcc_lightning_index_topk_noalloc", _ptr(qI), _ptr(w), B, Tq, HI, DI, _ptr(q_pos0), fmt, _ptr(kI),
          _ptr(kI_scale), _ptr(n_valid), kI.shape[1], int(m), int(k), _ptr(idx), _ptr(score), _stream(stream))
    return idx


def lightning_reindex_topk(qI, w, kI, cand, k, kI_scale=None, idx=None, score=None, stream=None):
    """CSA2 re-index mode: top-k of each query's candidate entries cand [B, Tq, n]
    (another layer's selection) by this layer's indexer query qI / weights w and
    the keys kI (bf16 [B, Ncap, DI], or NVFP4 uint8 with kI_scale).  Returns idx
    [B, Tq, k] int32 in ascending index order (score [B, Tq, k] if given)."""
    _need(qI, torch.bfloat16, "qI", 4)
    _need(w, torch.float32, "w", 3)
    _need(cand, torch.int32, "cand", 3)
    B, Tq, HI, DI = qI.shape
    fmt = KEY_NVFP4 if kI.dtype == torch.uint8 else KEY_BF16
    if not (qI.is_contiguous() and w.is_contiguous() and kI.is_contiguous() and cand.is_contiguous()):
        raise ValueError("qI, w, kI and cand must be contiguous")
    if idx is None:
        idx = torch.empty((B, Tq, k), dtype=torch.int32, device=qI.device)
    _need(idx, torch.int32, "idx", 3)
    _call("lcc_lightning_reindex_topk", _ptr(qI), _ptr(w), B, Tq, HI, DI, fmt, _ptr(kI), _ptr(kI_scale),
          kI.shape[1], _ptr(cand), cand.shape[2], int(k), _ptr(idx), _ptr(score), _stream(stream))
    return idx


def lightning_index_scores(qI, w, q_pos0, kI, n_valid, m, kI_scale=None, scores=None, stream=None):
    """Indexer scores of every visible entry: scores [B, Tq, Ncap] fp32 (others untouched)."""
    _need(qI, torch.bfloat16, "qI", 4)
    _need(w, torch.float32, "w", 3)
    B, Tq, HI, DI = qI.shape
    fmt = KEY_NVFP4 if kI.dtype == torch.uint8 else KEY_BF16
    Ncap = kI.shape[1]
    q_pos0 = _positions(q_pos0, B, qI.device)
    n_valid = _positions(n_valid, B, qI.device, torch.int32)
    if scores is None:
        scores = torch.full((B, Tq, Ncap), float("nan"), dtype=torch.float32, device=qI.device)
    _need(scores, torch.float32, "scores", 3)
    _call("lcc_lightning_index_scores", _ptr(qI), _ptr(w), B, Tq, HI, DI, _ptr(q_pos0), fmt, _ptr(kI),
          _ptr(kI_scale), _ptr(n_valid), Ncap, int(m), _ptr(scores), _stream(stream))
    return scores


# ---------------------------------------------------------------------------
# attention branches
# ---------------------------------------------------------------------------
def _attn_out(q, O, lse):
    B, Tq, H, D = q.shape
    if O is None:
        O = torch.empty((B, Tq, H, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Tq, H), dtype=torch.float32, device=q.device)
    _need(O, torch.float32, "O", 4)
    _need(lse, torch.float32, "lse", 3)
    if not (O.is_contiguous() and lse.is_contiguous() and q.is_contiguous()):
        raise ValueError("q, O and lse must be contiguous")
    return O, lse


def _kv(Kc, Vc):
    _need(Kc, torch.bfloat16, "K", 3)
    _need(Vc, torch.bfloat16, "V", 3)
    bs, rs = _rows(Kc, "K")
    if (bs, rs) != _rows(Vc, "V") or bs != Kc.shape[1] * rs:
        raise ValueError("K and V must share strides, with batch stride = rows * row stride")
    return rs


def csa_sparse_attn(q, Kc, Vc, idx, scale=1.0, O=None, lse=None, stream=None):
    """MQA over the idx-selected compressed entries; returns (O, lse)."""
    _need(q, torch.bfloat16, "q", 4)
    _need(idx, torch.int32, "idx", 3)
    B, Tq, H, D = q.shape
    rs = _kv(Kc, Vc)
    O, lse = _attn_out(q, O, lse)
    _call("lcc_csa_sparse_attn", _ptr(q), B, Tq, H, D, float(scale), _ptr(Kc), _ptr(Vc), rs, Kc.shape[1],
          _ptr(idx.contiguous()), idx.shape[2], _ptr(O), _ptr(lse), _stream(stream))
    return O, lse


def dense_attn_workspace(B, Tq, H, D, Ncap) -> int:
    return int(load().lcc_dense_attn_workspace(B, Tq, H, D, Ncap))


def hca_dense_attn(q, Kc, Vc, q_pos0, n_valid, m, scale=1.0, O=None, lse=None, workspace=None, stream=None):
    """MQA over every compressed entry visible at each query; returns (O, lse)."""
    _need(q, torch.bfloat16, "q", 4)
    B, Tq, H, D = q.shape
    rs = _kv(Kc, Vc)
    O, lse = _attn_out(q, O, lse)
    q_pos0 = _positions(q_pos0, B, q.device)
    n_valid = _positions(n_valid, B, q.device, torch.int32)
    need = dense_attn_workspace(B, Tq, H, D, Kc.shape[1])
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _call("lcc_hca_dense_attn", _ptr(q), B, Tq, H, D, float(scale), _ptr(q_pos0), _ptr(Kc), _ptr(Vc), rs,
          Kc.shape[1], _ptr(n_valid), int(m), _ptr(O), _ptr(lse), _ptr(workspace), nbytes, _stream(stream))
    return O, lse


def swa_attn(q, Kr, Vr, q_pos0, raw_pos0, W, scale=1.0, O=None, lse=None, stream=None):
    """MQA over the raw tokens of each query's window; returns (O, lse)."""
    _need(q, torch.bfloat16, "q", 4)
    B, Tq, H, D = q.shape
    rs = _kv(Kr, Vr)
    O, lse = _attn_out(q, O, lse)
    q_pos0 = _positions(q_pos0, B, q.device)
    raw_pos0 = _positions(raw_pos0, B, q.device)
    _call("lcc_swa_attn", _ptr(q), B, Tq, H, D, float(scale), _ptr(q_pos0), _ptr(Kr), _ptr(Vr), rs,
          Kr.shape[1], _ptr(raw_pos0), int(W), _ptr(O), _ptr(lse), _stream(stream))
    return O, lse


def attn_merge(parts, out=None, out_f32=None, lse_out=None, stream=None):
    """Log-sum-exp merge of [(O, lse), ...] (O [..., D] fp32, lse [...] fp32) -> bf16 out."""
    Os = [p[0] for p in parts]
    Ls = [p[1] for p in parts]
    for o, l in zip(Os, Ls):
        _need(o, torch.float32, "O part")
        _need(l, torch.float32, "lse part")
        if not (o.is_contiguous() and l.is_contiguous()):
            raise ValueError("parts must be contiguous")
    D = Os[0].shape[-1]
    rows = Os[0].numel() // D
    if out is None:
        out = torch.empty(Os[0].shape, dtype=torch.bfloat16, device=Os[0].device)
    nb = len(parts)
    Oarr = (ctypes.c_void_p * nb)(*[o.data_ptr() for o in Os])
    Larr = (ctypes.c_void_p * nb)(*[l.data_ptr() for l in Ls])
    _call("lcc_attn_merge", nb, ctypes.cast(Oarr, ctypes.c_void_p), ctypes.cast(Larr, ctypes.c_void_p), rows, D,
          _ptr(out), _ptr(out_f32), _ptr(lse_out), _stream(stream))
    return out


# ---------------------------------------------------------------------------
# whole layers in one pass (compressed branch ++ window)
# ---------------------------------------------------------------------------
def layer_attn_workspace(B, Tq, H, D, n_keys) -> int:
    return int(load().lcc_layer_attn_workspace(B, Tq, H, D, n_keys))


def _layer_out(q, out, lse_out):
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    _need(out, torch.bfloat16, "out", 4)
    if not (out.is_contiguous() and q.is_contiguous()):
        raise ValueError("q and out must be contiguous")
    if lse_out is not None:
        _need(lse_out, torch.float32, "lse_out", 3)
    return out


def _ws(workspace, need, dev):
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    return workspace, (workspace.numel() * workspace.element_size() if workspace is not None else 0)


def csa_layer_attn(q, Kc, Vc, idx, Kr, Vr, q_pos0, raw_pos0, W, scale=1.0, out=None, lse_out=None,
                   workspace=None, stream=None):
    """CSA layer: softmax over the idx-selected entries and the window rows -> bf16 [B, Tq, H, D]."""
    _need(q, torch.bfloat16, "q", 4)
    _need(idx, torch.int32, "idx", 3)
    B, Tq, H, D = q.shape
    rs, rr = _kv(Kc, Vc), _kv(Kr, Vr)
    out = _layer_out(q, out, lse_out)
    q_pos0 = _positions(q_pos0, B, q.device)
    raw_pos0 = _positions(raw_pos0, B, q.device)
    k = idx.shape[2]
    workspace, nbytes = _ws(workspace, layer_attn_workspace(B, Tq, H, D, k + int(W)), q.device)
    _call("lcc_csa_layer_attn", _ptr(q), B, Tq, H, D, float(scale), _ptr(q_pos0), _ptr(Kc), _ptr(Vc), rs,
          Kc.shape[1], _ptr(idx.contiguous()), k, _ptr(Kr), _ptr(Vr), rr, Kr.shape[1], _ptr(raw_pos0), int(W),
          _ptr(out), _ptr(lse_out), _ptr(workspace), nbytes, _stream(stream))
    return out


def csa_layer_workspace(B, Tq, H, D, Ncap, k, W) -> int:
    return int(load().lcc_csa_layer_workspace(B, Tq, H, D, Ncap, k, W))


def csa_layer(q, qI, w, q_pos0, kI, n_valid, m, k, Kc, Vc, Kr, Vr, raw_pos0, W, kI_scale=None, scale=1.0,
              idx=None, out=None, lse_out=None, workspace=None, stream=None):
    """A whole CSA layer (indexer + top-k + attention over the selected entries and the window) -> bf16."""
    _need(q, torch.bfloat16, "q", 4)
    _need(qI, torch.bfloat16, "qI", 4)
    _need(w, torch.float32, "w", 3)
    B, Tq, H, D = q.shape
    _, _, HI, DI = qI.shape
    if not (qI.is_contiguous() and w.is_contiguous() and kI.is_contiguous()):
        raise ValueError("qI, w and kI must be contiguous")
    if kI.dtype == torch.uint8:
        fmt = KEY_NVFP4
        _need(kI_scale, torch.uint8, "kI_scale", 3)
    else:
        fmt = KEY_BF16
        _need(kI, torch.bfloat16, "kI", 3)
    rs, rr = _kv(Kc, Vc), _kv(Kr, Vr)
    out = _layer_out(q, out, lse_out)
    dev = q.device
    q_pos0 = _positions(q_pos0, B, dev)
    raw_pos0 = _positions(raw_pos0, B, dev)
    n_valid = _positions(n_valid, B, dev, torch.int32)
    Ncap = kI.shape[1]
    if Kc.shape[1] != Ncap:
        raise ValueError("kI and Kc must hold the same number of entries")
    if idx is None:
        idx = torch.empty((B, Tq, k), dtype=torch.int32, device=dev)
    _need(idx, torch.int32, "idx", 3)
    workspace, nbytes = _ws(workspace, csa_layer_workspace(B, Tq, H, D, Ncap, k, int(W)), dev)
    _call("lcc_csa_layer", _ptr(q), _ptr(qI), _ptr(w), B, Tq, H, D, HI, DI, float(scale), _ptr(q_pos0), fmt,
          _ptr(kI), _ptr(kI_scale), _ptr(n_valid), _ptr(Kc), _ptr(Vc), rs, Ncap, int(m), int(k), _ptr(Kr), _ptr(Vr),
          rr, Kr.shape[1], _ptr(raw_pos0), int(W), _ptr(idx), _ptr(out), _ptr(lse_out), _ptr(workspace), nbytes,
          _stream(stream))
    return out


def hca_layer_attn(q, Kc, Vc, n_valid, m, Kr, Vr, q_pos0, raw_pos0, W, scale=1.0, out=None, lse_out=None,
                   workspace=None, stream=None):
    """HCA layer: softmax over every visible entry and the window rows -> bf16 [B, Tq, H, D]."""
    _need(q, torch.bfloat16, "q", 4)
    B, Tq, H, D = q.shape
    rs, rr = _kv(Kc, Vc), _kv(Kr, Vr)
    out = _layer_out(q, out, lse_out)
    q_pos0 = _positions(q_pos0, B, q.device)
    raw_pos0 = _positions(raw_pos0, B, q.device)
    n_valid = _positions(n_valid, B, q.device, torch.int32)
    workspace, nbytes = _ws(workspace, layer_attn_workspace(B, Tq, H, D, Kc.shape[1] + int(W)), q.device)
    _call("lcc_hca_layer_attn", _ptr(q), B, Tq, H, D, float(scale), _ptr(q_pos0), _ptr(Kc), _ptr(Vc), rs,
          Kc.shape[1], _ptr(n_valid), int(m), _ptr(Kr), _ptr(Vr), rr, Kr.shape[1], _ptr(raw_pos0), int(W),
          _ptr(out), _ptr(lse_out), _ptr(workspace), nbytes, _stream(stream))
    return out


def test_set_wait_fault(wait_limit_ns=0, drop_tile=-1):
    """Test hook: shorten every bounded device wait (0 = the default 2 s) and
    make the decode indexer skip one key tile per CTA (-1 = none), so that a
    test can make a wait run out.  See lcc_test_set_wait_fault in lcc.h."""
    _call("lcc_test_set_wait_fault", int(wait_limit_ns), int(drop_tile))


def sync_status(stream=None):
    """Synchronise the stream and raise if a kernel recorded a device-side error."""
    _call("lcc_sync_status", _stream(stream))
