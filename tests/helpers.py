"""Shared helpers for the GPU parity tests: seeded inputs on the device, exact
widening of device results, and the tolerance checks the parity bar states."""
from __future__ import annotations

import numpy as np

import synth

# 16-bit outputs: max-abs and relative Frobenius error against the FP64 oracle.
TOL16_MAX_ABS = 2e-2
TOL16_REL_FROB = 1e-2
# FP32 LSE and FP32 combine: |d| <= 1e-5 * max(1, |ref|), infinities exact.
TOL32_REL = 1e-5

TORCH_DT = {}


def torch_dtype(name):
    import torch
    return {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[name]


def to_device(bits: np.ndarray, dtype: str):
    """Upload stored bits (uint16 for 16-bit types, float32 otherwise) to cuda:0."""
    import torch
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.float32)).cuda()
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch_dtype(dtype)).cuda()


def to_f64(t) -> np.ndarray:
    """Exact float64 copy of a device tensor (16-bit and f32 widen exactly)."""
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def check16(out: np.ndarray, ref: np.ndarray, what: str = ""):
    d = np.abs(out - ref)
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    max_abs = float(d.max()) if d.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(out - ref)) / nref if nref > 0 else float(np.linalg.norm(out - ref))
    assert max_abs <= TOL16_MAX_ABS, f"{what}: max-abs {max_abs:.3e} > {TOL16_MAX_ABS}"
    assert rel <= TOL16_REL_FROB, f"{what}: rel-Frobenius {rel:.3e} > {TOL16_REL_FROB}"
    return max_abs, rel


def check32(out: np.ndarray, ref: np.ndarray, what: str = "", tol: float = TOL32_REL):
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    inf_ref = ~np.isfinite(ref)
    assert np.array_equal(out[inf_ref], ref[inf_ref]), f"{what}: infinities differ"
    assert np.all(np.isfinite(out[~inf_ref])), f"{what}: non-finite where the oracle is finite"
    d = np.abs(out[~inf_ref] - ref[~inf_ref])
    bound = tol * np.maximum(1.0, np.abs(ref[~inf_ref]))
    worst = float((d / bound).max()) if d.size else 0.0
    assert worst <= 1.0, f"{what}: error {worst:.2f}x the bound {tol}*max(1,|ref|)"
    return worst


def qkv_host(seed: int, B: int, H: int, N: int, D: int, dtype: str, nkv: int | None = None):
    """Q [B,H,N,D], K/V [B,H,nkv,D] stored bits from the seeded generator."""
    nkv = N if nkv is None else nkv
    q = synth.tensor(seed, synth.STREAM_Q, (B, H, N, D), dtype)
    k = synth.tensor(seed, synth.STREAM_K, (B, H, nkv, D), dtype)
    v = synth.tensor(seed, synth.STREAM_V, (B, H, nkv, D), dtype)
    return q, k, v


def head_slice(seed: int, stream: int, bh: int, n: int, D: int, dtype: str, rows=None) -> np.ndarray:
    """Float64 values of rows of head `bh` (flat [BH, n, D] layout) of one tensor."""
    if rows is None:
        rows = np.arange(n)
    rows = np.asarray(rows, dtype=np.int64)
    idx = (bh * n + rows)[:, None] * D + np.arange(D)[None, :]
    z = synth.normal_at(seed, stream, idx.ravel()).reshape(len(rows), D)
    return synth.to_f64(synth.round_to(z, dtype), dtype)
