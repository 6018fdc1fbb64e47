"""Online-softmax attention for GB300 (sm_103a): Python binding of liboattn.so.

Thin ctypes marshalling over the C ABI in ``include/oattn.h``: every function
takes torch CUDA tensors, checks shapes, dtypes and contiguity, and passes raw
device pointers plus the current CUDA stream.  All arithmetic runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and importing the
package fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

__all__ = ["attn_fwd", "attn_fwd_bn", "attn_fwd_splitk", "attn_fwd_splitk_noalloc", "splitk_combine", "splitk_chunk",
           "attn_mask_words", "attn_mask_pack", "attn_fwd_masked", "attn_fwd_splitk_masked",
           "attn_mask_blocks_words", "attn_mask_blocks", "attn_fwd_masked_blocks",
           "attn_splitk_counters", "attn_fwd_splitk_fused", "attn_fwd_host",
           "device_error", "OattnError", "library_path", "lib"]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "_build", "liboattn.so")

OK, INVALID_ARG, UNSUPPORTED, CUDA_ERR, TIMEOUT = 0, 1, 2, 3, 4
F16, BF16, F32 = 0, 1, 2


class OattnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lib.oattn_status_string(status).decode()} (status {status})")


def _load():
    if not os.path.exists(library_path):
        raise ImportError(
            f"{library_path} is missing: build it with `python -m online_softmax_gb300.build` "
            "(the package has no fallback path)")
    L = ctypes.CDLL(library_path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    L.attn_fwd_bn.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    L.attn_fwd_splitk.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, vp, i, vp]
    L.attn_fwd_splitk_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp]
    L.splitk_combine.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, vp]
    L.splitk_chunk.argtypes = [i, i]
    ll = ctypes.c_longlong
    L.attn_mask_words.argtypes = [i]
    L.attn_mask_pack.argtypes = [vp, vp, ll, i, ll, vp]
    L.attn_fwd_masked.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, ll, ll, ll, vp]
    L.attn_mask_blocks_words.argtypes = [i, i, i, i, ll, ll]
    L.attn_mask_blocks_words.restype = ll
    L.attn_mask_blocks.argtypes = [vp, ll, ll, ll, i, i, i, i, vp, vp]
    L.attn_fwd_masked_blocks.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, ll, ll, ll, vp, vp]
    L.attn_fwd_splitk_masked.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, vp, i,
                                         vp, ll, ll, ll, vp]
    L.attn_splitk_counters.argtypes = [i, i, i]
    L.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    L.attn_fwd_splitk_fused.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, vp, i, vp,
                                        vp, ll, ll, ll, vp]
    L.oattn_status_string.argtypes = [i]
    L.oattn_status_string.restype = ctypes.c_char_p
    L.oattn_device_error.argtypes = [ctypes.POINTER(ctypes.c_int)]
    L.oattn_selftest_wait.argtypes = [vp, vp]
    for name in ("attn_fwd", "attn_fwd_bn", "attn_fwd_splitk", "attn_fwd_splitk_noalloc", "splitk_combine",
                 "splitk_chunk", "oattn_device_error", "attn_mask_words", "attn_mask_pack", "attn_fwd_masked",
                 "attn_fwd_splitk_masked", "attn_splitk_counters", "attn_fwd_splitk_fused", "attn_fwd_host",
                 "oattn_selftest_wait", "attn_mask_blocks", "attn_fwd_masked_blocks"):
        getattr(L, name).restype = ctypes.c_int
    return L


class _Lazy:
    """Loads the library on first use, so that building it (``python -m
    online_softmax_gb300.build``) does not need it to exist yet."""
    _L = None

    def __getattr__(self, name):
        if _Lazy._L is None:
            _Lazy._L = _load()
        return getattr(_Lazy._L, name)


lib = _Lazy()


def _dtype_code(t) -> int:
    import torch
    if t == torch.float16:
        return F16
    if t == torch.bfloat16:
        return BF16
    if t == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t}")


def _ptr(x):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(x, name, dtype=None, shape=None):
    if x is None:
        return
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and x.dtype != dtype:
        raise TypeError(f"{name} has dtype {x.dtype}, expected {dtype}")
    if shape is not None and tuple(x.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(x.shape)}, expected {tuple(shape)}")


def _raise(st, what):
    if st != OK:
        raise OattnError(st, what)


def attn_fwd_bn(q, k, v, o, lse=None, causal=False, scale=None, block_n=0, stream=None):
    """Attention forward.  q, k, v, o: [B, H, N, D] f16/bf16; lse: [B, H, N] f32 or None."""
    import torch
    B, H, N, D = q.shape
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, q.shape)
    _check(o, "o", q.dtype, q.shape); _check(lse, "lse", torch.float32, (B, H, N))
    scale = D ** -0.5 if scale is None else float(scale)
    st = lib.attn_fwd_bn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D, int(bool(causal)),
                         scale, _dtype_code(q.dtype), int(block_n), _stream(stream))
    _raise(st, "attn_fwd_bn")
    return o, lse


def attn_fwd_host(q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d, o_d, lse_d=None, causal=False, scale=None,
                  chunk_heads=0, stream=None):
    """Attention forward on HOST tensors (pinned CPU tensors [B, H, N, D]; lse_h [B, H, N]
    float32 or None), through caller-owned device staging tensors of the same shapes: the
    copies in and out overlap the attention of neighbouring chunks of heads."""
    import torch
    B, H, N, D = q_h.shape
    for x, name in ((q_h, "q_h"), (k_h, "k_h"), (v_h, "v_h"), (o_h, "o_h")):
        if x.is_cuda or not x.is_contiguous() or tuple(x.shape) != (B, H, N, D) or x.dtype != q_h.dtype:
            raise ValueError(f"{name} must be a contiguous CPU tensor like q_h")
    if (lse_h is None) != (lse_d is None):
        raise ValueError("lse_h and lse_d go together")
    if lse_h is not None and (lse_h.is_cuda or not lse_h.is_contiguous() or lse_h.dtype != torch.float32
                              or tuple(lse_h.shape) != (B, H, N)):
        raise ValueError("lse_h must be a contiguous float32 CPU tensor [B, H, N]")
    _check(q_d, "q_d", q_h.dtype, q_h.shape); _check(k_d, "k_d", q_h.dtype, q_h.shape)
    _check(v_d, "v_d", q_h.dtype, q_h.shape); _check(o_d, "o_d", q_h.dtype, q_h.shape)
    _check(lse_d, "lse_d", torch.float32, (B, H, N))
    scale = D ** -0.5 if scale is None else float(scale)
    st = lib.attn_fwd_host(_ptr(q_h), _ptr(k_h), _ptr(v_h), _ptr(o_h), _ptr(lse_h), _ptr(q_d), _ptr(k_d),
                           _ptr(v_d), _ptr(o_d), _ptr(lse_d), B, H, N, D, int(bool(causal)), scale,
                           _dtype_code(q_h.dtype), int(chunk_heads), _stream(stream))
    _raise(st, "attn_fwd_host")
    return o_h, lse_h


def attn_fwd(q, k, v, o, lse=None, causal=False, scale=None, stream=None):
    """Attention forward with the default key tile (see attn_fwd_bn)."""
    import torch
    B, H, N, D = q.shape
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, q.shape)
    _check(o, "o", q.dtype, q.shape); _check(lse, "lse", torch.float32, (B, H, N))
    scale = D ** -0.5 if scale is None else float(scale)
    st = lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D, int(bool(causal)),
                      scale, _dtype_code(q.dtype), _stream(stream))
    _raise(st, "attn_fwd")
    return o, lse


def splitk_chunk(nkv: int, P: int) -> int:
    """Keys per split-K partition used by attn_fwd_splitk."""
    return lib.splitk_chunk(int(nkv), int(P))


def attn_fwd_splitk(q, k, v, P, o_partial, lse_partial, o=None, lse=None, causal=False,
                    scale=None, stream=None):
    """Split-K attention.  q: [B, H, Nq, D]; k, v: [B, H, Nkv, D];
    o_partial: [P, B*H*Nq, D] f32 or q.dtype; lse_partial: [P, B*H*Nq] f32 (base 2);
    o: [B, H, Nq, D] q.dtype or None; lse: [B, H, Nq] f32 (natural log) or None."""
    import torch
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    _check(q, "q"); _check(k, "k", q.dtype, (B, H, Nkv, D)); _check(v, "v", q.dtype, (B, H, Nkv, D))
    _check(o_partial, "o_partial", None, (P, B * H * Nq, D))
    _check(lse_partial, "lse_partial", torch.float32, (P, B * H * Nq))
    _check(o, "o", q.dtype, q.shape); _check(lse, "lse", torch.float32, (B, H, Nq))
    scale = D ** -0.5 if scale is None else float(scale)
    st = lib.attn_fwd_splitk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nkv, D,
                             int(bool(causal)), scale, _dtype_code(q.dtype), int(P), _ptr(o_partial),
                             _ptr(lse_partial), _dtype_code(o_partial.dtype), _stream(stream))
    _raise(st, "attn_fwd_splitk")
    return o_partial, lse_partial, o, lse


def attn_fwd_splitk_noalloc(q, k, v, P, o, lse=None, causal=False, scale=None, stream=None):
    """Split-K attention without caller-provided workspace: the float32 partials live in
    a fixed device array inside the library (for callers that cannot allocate device
    memory).  Calls that overlap on the GPU share that array and race."""
    import torch
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    _check(q, "q"); _check(k, "k", q.dtype, (B, H, Nkv, D)); _check(v, "v", q.dtype, (B, H, Nkv, D))
    _check(o, "o", q.dtype, q.shape); _check(lse, "lse", torch.float32, (B, H, Nq))
    scale = D ** -0.5 if scale is None else float(scale)
    st = lib.attn_fwd_splitk_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nkv, D,
                                     int(bool(causal)), scale, _dtype_code(q.dtype), int(P), _stream(stream))
    _raise(st, "attn_fwd_splitk_noalloc")
    return o, lse


def splitk_combine(o_partial, lse_partial, o, lse_out=None, rows=None, heads=1, stream=None):
    """LSE-weighted combine.  o_partial: [P, RH, depth]; lse_partial: [P, RH] f32 (base 2);
    o: [RH, depth] (any shape with RH*depth elements); lse_out: [RH] f32 or None.
    RH = rows * heads (rows defaults to RH / heads)."""
    import torch
    P, RH, depth = o_partial.shape
    if rows is None:
        rows = RH // heads
    if rows * heads != RH:
        raise ValueError("rows * heads must equal the row-head count")
    _check(o_partial, "o_partial"); _check(lse_partial, "lse_partial", torch.float32, (P, RH))
    _check(o, "o")
    if o.numel() != RH * depth:
        raise ValueError("o must hold rows*heads*depth elements")
    _check(lse_out, "lse_out", torch.float32)
    if lse_out is not None and lse_out.numel() != RH:
        raise ValueError("lse_out must hold rows*heads elements")
    st = lib.splitk_combine(_ptr(o_partial), _ptr(lse_partial), _ptr(o), _ptr(lse_out), int(P),
                            int(rows), int(heads), int(depth), _dtype_code(o_partial.dtype),
                            _dtype_code(o.dtype), _stream(stream))
    _raise(st, "splitk_combine")
    return o, lse_out


def attn_mask_words(nkv: int) -> int:
    """32-bit words per packed mask row: 4 * ceil(nkv / 128)."""
    return lib.attn_mask_words(int(nkv))


def attn_mask_pack(mask, bits=None, stream=None):
    """Pack a Boolean mask [..., Nq, Nkv] (bool or uint8 CUDA tensor; nonzero = the key is
    visible) into the bit layout the masked kernels read: int32 [..., Nq, W] with
    W = attn_mask_words(Nkv), bit j of word w = key 32*w + j.  The rows must be evenly
    strided: a contiguous tensor, or a 2-D slice [:, :Nkv] of a wider buffer."""
    import torch
    if not mask.is_cuda:
        raise ValueError("mask must be a CUDA tensor")
    if mask.dtype not in (torch.bool, torch.uint8):
        raise TypeError("mask must be bool or uint8")
    if mask.dim() < 2:
        raise ValueError("mask needs at least two dimensions [..., Nq, Nkv]")
    nkv = mask.shape[-1]
    rows = mask.numel() // nkv if nkv else 0
    if mask.is_contiguous():
        row_stride = nkv
    elif mask.dim() == 2 and mask.stride(-1) == 1 and mask.stride(0) >= nkv:
        row_stride = mask.stride(0)  # rows of a wider buffer
    else:
        raise ValueError("mask must be contiguous, or a 2-D slice of rows with a contiguous key axis")
    W = attn_mask_words(nkv)
    if bits is None:
        bits = torch.empty(*mask.shape[:-1], W, dtype=torch.int32, device=mask.device)
    _check(bits, "bits", torch.int32, tuple(mask.shape[:-1]) + (W,))
    st = lib.attn_mask_pack(_ptr(mask), _ptr(bits), int(rows), int(nkv), int(row_stride), _stream(stream))
    _raise(st, "attn_mask_pack")
    return bits


def _mask_strides(bits, B, H, Nq, Nkv, stream):
    """Packed mask (int32 [..., W]) or Boolean mask (packed here) broadcast against
    [B, H, Nq, *] -> (tensor kept alive, pointer, stride_b, stride_h, stride_q)."""
    import torch
    if bits.dtype in (torch.bool, torch.uint8):
        bits = attn_mask_pack(bits if bits.is_contiguous() or bits.dim() == 2 else bits.contiguous(), stream=stream)
    if bits.dtype != torch.int32 or not bits.is_cuda:
        raise TypeError("mask must be a CUDA bool/uint8 mask or its int32 packed bits")
    W = attn_mask_words(Nkv)
    if bits.shape[-1] != W or bits.stride(-1) != 1:
        raise ValueError(f"packed mask rows must hold {W} contiguous words")
    while bits.dim() < 4:
        bits = bits.unsqueeze(0)
    if stream is not None:
        bits.record_stream(stream)  # a mask packed here must outlive the launch on `stream`
    bits = bits.expand(B, H, Nq, W)
    sb, sh, sq = (bits.stride(0) if B > 1 else 0, bits.stride(1) if H > 1 else 0, bits.stride(2) if Nq > 1 else 0)
    return bits, _ptr(bits), sb, sh, sq


def attn_fwd_masked(q, k, v, o, mask, lse=None, causal=False, scale=None, stream=None):
    """Attention forward with the optional Boolean mask.  q, k, v, o: [B, H, N, D];
    mask: Boolean [.., N, N] broadcastable to [B, H, N, N] (True = visible), or its
    packed bits from attn_mask_pack (int32 [.., N, W])."""
    import torch
    B, H, N, D = q.shape
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, q.shape)
    _check(o, "o", q.dtype, q.shape); _check(lse, "lse", torch.float32, (B, H, N))
    scale = D ** -0.5 if scale is None else float(scale)
    keep, mp, sb, sh, sq = _mask_strides(mask, B, H, N, N, stream)
    st = lib.attn_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D, int(bool(causal)),
                             scale, _dtype_code(q.dtype), mp, sb, sh, sq, _stream(stream))
    _raise(st, "attn_fwd_masked")
    return o, lse


def attn_mask_blocks_words(B: int, H: int, Nq: int, Nkv: int, stride_b: int, stride_h: int) -> int:
    """32-bit words of the block summary of a mask with these strides (0 = shared)."""
    return lib.attn_mask_blocks_words(int(B), int(H), int(Nq), int(Nkv), int(stride_b), int(stride_h))


def attn_mask_blocks(mask, B, H, Nq, Nkv=None, blocks=None, stream=None):
    """Block summary of a mask broadcast against [B, H, Nq, Nkv] (Boolean, or its packed
    bits): one bit per (mask head, 256 query rows, 128-key tile), set when some row of
    the block sees some key of the tile.  Returns int32 [attn_mask_blocks_words(...)]."""
    import torch
    Nkv = Nq if Nkv is None else Nkv
    keep, mp, sb, sh, sq = _mask_strides(mask, B, H, Nq, Nkv, stream)
    n = attn_mask_blocks_words(B, H, Nq, Nkv, sb, sh)
    if blocks is None:
        blocks = torch.empty(max(n, 1), dtype=torch.int32, device=keep.device)
    if blocks.dtype != torch.int32 or not blocks.is_cuda or not blocks.is_contiguous() or blocks.numel() < n:
        raise ValueError(f"blocks must be a contiguous CUDA int32 tensor of at least {n} words")
    st = lib.attn_mask_blocks(mp, sb, sh, sq, int(B), int(H), int(Nq), int(Nkv), _ptr(blocks), _stream(stream))
    _raise(st, "attn_mask_blocks")
    return blocks


def attn_fwd_masked_blocks(q, k, v, o, mask, blocks, lse=None, causal=False, scale=None, stream=None):
    """attn_fwd_masked with the block summary of the same mask (attn_mask_blocks with
    the same mask and B, H, Nq = Nkv = N): the persistent kernel visits only the key
    tiles the summary marks."""
    import torch
    B, H, N, D = q.shape
    _check(q, "q"); _check(k, "k", q.dtype, q.shape); _check(v, "v", q.dtype, q.shape)
    _check(o, "o", q.dtype, q.shape); _check(lse, "lse", torch.float32, (B, H, N))
    scale = D ** -0.5 if scale is None else float(scale)
    keep, mp, sb, sh, sq = _mask_strides(mask, B, H, N, N, stream)
    n = attn_mask_blocks_words(B, H, N, N, sb, sh)
    if blocks.dtype != torch.int32 or not blocks.is_cuda or not blocks.is_contiguous() or blocks.numel() < n:
        raise ValueError(f"blocks must be the summary of this mask: a contiguous CUDA int32 tensor of {n} words")
    st = lib.attn_fwd_masked_blocks(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, D, int(bool(causal)),
                                    scale, _dtype_code(q.dtype), mp, sb, sh, sq, _ptr(blocks), _stream(stream))
    _raise(st, "attn_fwd_masked_blocks")
    return o, lse


def attn_fwd_splitk_masked(q, k, v, P, o_partial, lse_partial, mask, o=None, lse=None, causal=False,
                           scale=None, stream=None):
    """Split-K attention with the optional Boolean mask [.., Nq, Nkv] (or its packed
    bits), otherwise as attn_fwd_splitk."""
    import torch
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    _check(q, "q"); _check(k, "k", q.dtype, (B, H, Nkv, D)); _check(v, "v", q.dtype, (B, H, Nkv, D))
    _check(o_partial, "o_partial", None, (P, B * H * Nq, D))
    _check(lse_partial, "lse_partial", torch.float32, (P, B * H * Nq))
    _check(o, "o", q.dtype, q.shape); _check(lse, "lse", torch.float32, (B, H, Nq))
    scale = D ** -0.5 if scale is None else float(scale)
    keep, mp, sb, sh, sq = _mask_strides(mask, B, H, Nq, Nkv, stream)
    st = lib.attn_fwd_splitk_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nkv, D,
                                    int(bool(causal)), scale, _dtype_code(q.dtype), int(P), _ptr(o_partial),
                                    _ptr(lse_partial), _dtype_code(o_partial.dtype), mp, sb, sh, sq,
                                    _stream(stream))
    _raise(st, "attn_fwd_splitk_masked")
    return o_partial, lse_partial, o, lse


def attn_splitk_counters(B: int, H: int, Nq: int) -> int:
    """Counter words attn_fwd_splitk_fused needs (at most B*H*Nq)."""
    return lib.attn_splitk_counters(int(B), int(H), int(Nq))


def attn_fwd_splitk_fused(q, k, v, P, o_partial, lse_partial, counters, o, lse=None, mask=None,
                          causal=False, scale=None, stream=None):
    """Split-K attention whose partitions are merged inside the attention kernel by the
    last CTA of each group.  counters: int32 CUDA tensor with at least
    attn_splitk_counters(B, H, Nq) elements, zero before the first call (each completed
    call leaves it zero).  mask: None, or as in attn_fwd_splitk_masked.  Other arguments
    as attn_fwd_splitk (o required)."""
    import torch
    B, H, Nq, D = q.shape
    Nkv = k.shape[2]
    _check(q, "q"); _check(k, "k", q.dtype, (B, H, Nkv, D)); _check(v, "v", q.dtype, (B, H, Nkv, D))
    _check(o_partial, "o_partial", None, (P, B * H * Nq, D))
    _check(lse_partial, "lse_partial", torch.float32, (P, B * H * Nq))
    _check(o, "o", q.dtype, q.shape); _check(lse, "lse", torch.float32, (B, H, Nq))
    _check(counters, "counters", torch.int32)
    if counters.numel() < attn_splitk_counters(B, H, Nq):
        raise ValueError(f"counters needs {attn_splitk_counters(B, H, Nq)} elements")
    scale = D ** -0.5 if scale is None else float(scale)
    keep, mp, sb, sh, sq = (None, None, 0, 0, 0) if mask is None else _mask_strides(mask, B, H, Nq, Nkv, stream)
    st = lib.attn_fwd_splitk_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nkv, D,
                                   int(bool(causal)), scale, _dtype_code(q.dtype), int(P), _ptr(o_partial),
                                   _ptr(lse_partial), _dtype_code(o_partial.dtype), _ptr(counters), mp, sb, sh, sq,
                                   _stream(stream))
    _raise(st, "attn_fwd_splitk_fused")
    return o, lse


SELFTEST_SITE = 0x1F0  # site code recorded by selftest_wait's wait


def selftest_wait(flags=None, stream=None):
    """Run the device self-test of the bounded-wait failure path (about 2 s): a wait on a
    phase that never completes gives up, records SELFTEST_SITE in the device status word
    and the kernel returns; read the word afterwards with device_error().  `flags`: an
    optional int32 CUDA tensor of 2 elements, set to 0 where a wait gave up."""
    import torch
    if flags is not None and (not flags.is_cuda or flags.dtype != torch.int32 or flags.numel() < 2):
        raise ValueError("flags must be an int32 CUDA tensor of at least 2 elements")
    st = lib.oattn_selftest_wait(_ptr(flags), _stream(stream))
    _raise(st, "oattn_selftest_wait")


def device_error() -> int:
    """Read and clear the device status word (synchronises the device); 0 = no wait gave up."""
    code = ctypes.c_int(0)
    st = lib.oattn_device_error(ctypes.byref(code))
    if st not in (OK, TIMEOUT):
        raise OattnError(st, "oattn_device_error")
    return code.value
