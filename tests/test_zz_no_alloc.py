"""The allocation-free split-K entry point, checked against the FP64 oracle and against
attn_fwd_splitk.

attn_fwd_splitk_noalloc serves callers that cannot allocate device memory: it keeps the
partition workspace in a fixed array inside the library instead of caller buffers.
These tests call it through the C ABI, on two calls in a row (the second call runs on a
workspace that still holds the first call's partials), and compare each call with the
FP64 oracle's attention (an independent check: a fault shared by both CUDA entry points
would not hide) and with the entry point that takes caller-owned workspace.  The file
sorts last so that a run that stops at the first failure has run every other test
first."""
import ctypes
import math

import numpy as np
import pytest

import oracle
import synth
from tests import helpers as H

A = ctypes.c_void_p(0x1000)


def test_rejects_sizes_beyond_the_workspace():
    """Oversized problems fail with OATTN_ERR_UNSUPPORTED before touching the device."""
    import online_softmax_gb300 as ops
    from online_softmax_gb300 import build as b
    import os
    if not os.path.exists(ops.library_path):
        b.build()
    L = ops.lib
    # 64 x 32 heads x 1 query x D=128 x P=64 partials = 16.8 M floats > 10 Mi
    assert L.attn_fwd_splitk_noalloc(A, A, A, A, None, 64, 32, 1, 32768, 128, 0, 0.1, 1, 64, None) == 2
    # LSE slots: P * rows = 256 * 2048 > 256 Ki
    assert L.attn_fwd_splitk_noalloc(A, A, A, A, None, 64, 32, 1, 1024, 16, 0, 0.1, 1, 256, None) == 2
    assert L.attn_fwd_splitk_noalloc(A, A, A, None, None, 1, 1, 1, 8, 64, 0, 0.1, 1, 2, None) == 1


def _reference(ops, torch, q, k, v, P, causal):
    B, Hh, Nq, D = q.shape
    op = torch.empty((P, B * Hh * Nq, D), dtype=torch.float32, device="cuda")
    lp = torch.empty((P, B * Hh * Nq), dtype=torch.float32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, Hh, Nq), dtype=torch.float32, device="cuda")
    ops.attn_fwd_splitk(q, k, v, P, op, lp, o, lse, causal=causal)
    return o, lse


def _noalloc(ops, torch, q, k, v, P, causal):
    B, Hh, Nq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hh, Nq), dtype=torch.float32, device="cuda")
    st = ops.lib.attn_fwd_splitk_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
        ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), B, Hh, Nq, k.shape[2], D,
        int(causal), 1.0 / math.sqrt(D), ops.BF16, P, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, ops.lib.oattn_status_string(st)
    return o, lse


@pytest.mark.gpu
@pytest.mark.parametrize("B,Hh,Nq,Nkv,D,P,causal", [
    (8, 4, 1, 5000, 128, 8, False),     # one-query decode (CUDA-core partitions)
    (1, 2, 1000, 1000, 64, 3, True),    # several queries (tensor-core partitions), causal
])
def test_noalloc_matches_caller_workspace(B, Hh, Nq, Nkv, D, P, causal):
    torch = pytest.importorskip("torch")
    import online_softmax_gb300 as ops
    assert torch.cuda.is_available()
    qb, kb, vb = H.qkv_host(61, B, Hh, Nq, D, "bf16", nkv=Nkv)
    q, k, v = (H.to_device(x, "bf16") for x in (qb, kb, vb))
    O_or, L_or = oracle.attention(synth.to_f64(qb, "bf16"), synth.to_f64(kb, "bf16"), synth.to_f64(vb, "bf16"),
                                  1.0 / math.sqrt(D), causal)
    o_ref, lse_ref = _reference(ops, torch, q, k, v, P, causal)
    for call in range(2):
        o, lse = _noalloc(ops, torch, q, k, v, P, causal)
        torch.cuda.synchronize()
        H.check16(H.to_f64(o), O_or, f"call {call} O vs oracle")
        H.check32(H.to_f64(lse), L_or, f"call {call} LSE vs oracle")
        H.check16(H.to_f64(o), H.to_f64(o_ref), f"call {call} O vs attn_fwd_splitk")
        H.check32(H.to_f64(lse), H.to_f64(lse_ref), f"call {call} LSE vs attn_fwd_splitk")
    assert ops.device_error() == 0
