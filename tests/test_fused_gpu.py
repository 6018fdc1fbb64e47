"""Parity of attn_fwd_splitk_fused (split-K with the merge inside the attention kernel,
through the C ABI) against the FP64 oracle, and the counter protocol: a completed call
leaves every counter at zero, so calls can follow one another."""
import math

import numpy as np
import pytest

import oracle
import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
ops = pytest.importorskip("online_softmax_gb300")


@pytest.fixture(autouse=True)
def _no_device_errors():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    assert ops.device_error() == 0, "a bounded device wait gave up"


def run_fused(q, k, v, P, causal, partial="f32", mask=None, counters=None):
    B, Hh, Nq, D = q.shape
    RH = B * Hh * Nq
    pdt = torch.float32 if partial == "f32" else q.dtype
    op = torch.empty((P, RH, D), dtype=pdt, device="cuda")
    lp = torch.empty((P, RH), dtype=torch.float32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, Hh, Nq), dtype=torch.float32, device="cuda")
    if counters is None:
        counters = torch.zeros(ops.attn_splitk_counters(B, Hh, Nq), dtype=torch.int32, device="cuda")
    ops.attn_fwd_splitk_fused(q, k, v, P, op, lp, counters, o, lse, mask=mask, causal=causal)
    torch.cuda.synchronize()
    assert int(counters.abs().sum()) == 0, "a completed call must leave the counters at zero"
    return op, lp, o, lse


def check_fused(qb, kb, vb, dtype, P, causal, partial, what, mask=None):
    B, Hh, Nq, D = qb.shape
    scale = 1.0 / math.sqrt(D)
    q, k, v = (H.to_device(x, dtype) for x in (qb, kb, vb))
    mt = None if mask is None else torch.from_numpy(np.array(mask, dtype=bool, copy=True)).cuda()
    op, lp, o, lse = run_fused(q, k, v, P, causal, partial, mt)
    qd, kd, vd = (synth.to_f64(x, dtype) for x in (qb, kb, vb))
    Op, Lp = oracle.splitk_partials(qd, kd, vd, scale, causal, P, 128, mask=mask)
    O, L = oracle.attention(qd, kd, vd, scale, causal, mask=mask)
    H.check16(H.to_f64(op), Op.reshape(P, -1, D), what + " O_p")
    H.check32(H.to_f64(lp), Lp.reshape(P, -1), what + " lse_p")
    H.check16(H.to_f64(o), O, what + " O")
    H.check32(H.to_f64(lse), L, what + " LSE")
    dead = np.isneginf(L)
    if dead.any():
        got = H.to_f64(o)[dead]
        assert np.all(got == 0) and not np.any(np.signbit(got)), "rows with no visible key must be +0"
    return q, k, v, o, lse


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("Nkv,P", [(1, 1), (100, 3), (1000, 8), (1000, 1), (300, 16)])
@pytest.mark.parametrize("dtype,partial", [("bf16", "f32"), ("f16", "f16")])
def test_fused_decode(D, Nkv, P, dtype, partial):
    qb, kb, vb = H.qkv_host(120 + D, 2, 3, 1, D, dtype, nkv=Nkv)
    check_fused(qb, kb, vb, dtype, P, False, partial, f"fused decode D{D} Nkv{Nkv} P{P}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("P", [1, 3, 8])
@pytest.mark.parametrize("D,partial", [(64, "f32"), (128, "bf16"), (16, "f32")])
def test_fused_splitk_prefill(causal, P, D, partial):
    qb, kb, vb = H.qkv_host(130 + P, 1, 2, 700, D, "bf16")
    check_fused(qb, kb, vb, "bf16", P, causal, partial, f"fused splitk D{D} P{P} c{causal}")


def test_fused_masked():
    B, Hh = 3, 2
    qb, kb, vb = H.qkv_host(140, B, Hh, 1, 64, "bf16", nkv=900)
    check_fused(qb, kb, vb, "bf16", 4, False, "f32", "fused decode key padding",
                mask=synth.key_padding(141, B, 900, min_len=1))
    qb, kb, vb = H.qkv_host(142, 1, 2, 400, 64, "bf16")
    m = synth.hide_rows(143, synth.mask_random(143, (400, 400), 0.3), 0.05)
    check_fused(qb, kb, vb, "bf16", 3, True, "f32", "fused splitk random mask", mask=m)


def test_fused_matches_unfused_and_repeats():
    """Two fused calls in a row on one counter array give identical results, close to the
    unfused path (which merges in a separate kernel)."""
    qb, kb, vb = H.qkv_host(150, 2, 4, 1, 128, "bf16", nkv=5000)
    q, k, v = (H.to_device(x, "bf16") for x in (qb, kb, vb))
    counters = torch.zeros(ops.attn_splitk_counters(2, 4, 1), dtype=torch.int32, device="cuda")
    _, _, o1, l1 = run_fused(q, k, v, 8, False, counters=counters)
    _, _, o2, l2 = run_fused(q, k, v, 8, False, counters=counters)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    op = torch.empty((8, 8, 128), dtype=torch.float32, device="cuda")
    lp = torch.empty((8, 8), dtype=torch.float32, device="cuda")
    o3, l3 = torch.empty_like(q), torch.empty_like(l1)
    ops.attn_fwd_splitk(q, k, v, 8, op, lp, o3, l3)
    torch.cuda.synchronize()
    H.check16(H.to_f64(o1), H.to_f64(o3), "fused vs unfused O")
    H.check32(H.to_f64(l1), H.to_f64(l3), "fused vs unfused LSE")


@pytest.mark.parametrize("P", [16, 37])
def test_fused_decode_full_size_sampled(P):
    """64 sequences x 1 query, 32 heads, 32768 keys, D = 128, bf16, FP32 partials."""
    import synth.cuda as sc
    B, Hh, Nkv, D, seed = 64, 32, 32768, 128, 5
    q = sc.fill_normal(torch.empty((B, Hh, 1, D), dtype=torch.bfloat16, device="cuda"), seed,
                       synth.STREAM_Q, "bf16")
    k = sc.fill_normal(torch.empty((B, Hh, Nkv, D), dtype=torch.bfloat16, device="cuda"), seed,
                       synth.STREAM_K, "bf16")
    v = sc.fill_normal(torch.empty((B, Hh, Nkv, D), dtype=torch.bfloat16, device="cuda"), seed,
                       synth.STREAM_V, "bf16")
    _, _, o, lse = run_fused(q, k, v, P, False)
    del k, v
    scale = 1.0 / math.sqrt(D)
    for bh in (0, 777, B * Hh - 1):
        qr = H.head_slice(seed, synth.STREAM_Q, bh, 1, D, "bf16")
        kh = H.head_slice(seed, synth.STREAM_K, bh, Nkv, D, "bf16")
        vh = H.head_slice(seed, synth.STREAM_V, bh, Nkv, D, "bf16")
        O, L = oracle.attention_rows(qr, np.array([0]), kh, vh, scale, False)
        b, h = divmod(bh, Hh)
        H.check16(H.to_f64(o[b, h]), O, f"fused decode P{P} bh{bh} O")
        H.check32(H.to_f64(lse[b, h]), L, f"fused decode P{P} bh{bh} LSE")
