"""attn_fwd_host (host buffers in and out, copies overlapped with the attention of
neighbouring chunks of heads) against attn_fwd on device buffers: bit for bit, for every
chunking, and against the oracle."""
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


def host_tensors(qb, kb, vb, dtype, pinned):
    qh, kh, vh = (H.to_device(x, dtype).cpu() for x in (qb, kb, vb))
    if pinned:
        qh, kh, vh = (x.pin_memory() for x in (qh, kh, vh))
    oh = torch.empty_like(qh)
    lh = torch.empty(qh.shape[:3], dtype=torch.float32)
    if pinned:
        oh, lh = oh.pin_memory(), lh.pin_memory()
    return qh, kh, vh, oh, lh


@pytest.mark.parametrize("chunk", [0, 1, 4, 7, 64])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_matches_device_bitwise(chunk, causal, pinned):
    B, Hh, N, D = 2, 3, 333, 64
    qb, kb, vb = H.qkv_host(160, B, Hh, N, D, "bf16")
    qh, kh, vh, oh, lh = host_tensors(qb, kb, vb, "bf16", pinned)
    qd, kd, vd = (torch.empty(qh.shape, dtype=qh.dtype, device="cuda") for _ in range(3))
    od = torch.empty_like(qd)
    ld = torch.empty(qh.shape[:3], dtype=torch.float32, device="cuda")
    ops.attn_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, causal=causal, chunk_heads=chunk)
    torch.cuda.synchronize()
    q, k, v = (H.to_device(x, "bf16") for x in (qb, kb, vb))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    ops.attn_fwd(q, k, v, o, lse, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(oh, o.cpu()) and torch.equal(lh, lse.cpu())


def test_host_against_oracle_without_lse():
    B, Hh, N, D = 1, 4, 200, 128
    qb, kb, vb = H.qkv_host(161, B, Hh, N, D, "f16")
    qh, kh, vh, oh, _ = host_tensors(qb, kb, vb, "f16", True)
    qd, kd, vd, od = (torch.empty(qh.shape, dtype=qh.dtype, device="cuda") for _ in range(4))
    ops.attn_fwd_host(qh, kh, vh, oh, None, qd, kd, vd, od, None, causal=True, chunk_heads=3)
    torch.cuda.synchronize()
    O, _ = oracle.attention(synth.to_f64(qb, "f16"), synth.to_f64(kb, "f16"), synth.to_f64(vb, "f16"),
                            1.0 / math.sqrt(D), True)
    H.check16(H.to_f64(oh), O, "host path O")


def test_host_calls_from_four_threads():
    """Four host threads call attn_fwd_host at once, each with its own stream and staging
    buffers; the calls share the library's internal streams and events, and each result
    still equals attn_fwd on device buffers bit for bit."""
    import threading
    B, Hh, N, D = 1, 6, 300, 64
    cases = []
    for i in range(4):
        qb, kb, vb = H.qkv_host(170 + i, B, Hh, N, D, "bf16")
        qh, kh, vh, oh, lh = host_tensors(qb, kb, vb, "bf16", True)
        staging = [torch.empty(qh.shape, dtype=qh.dtype, device="cuda") for _ in range(4)]
        staging.append(torch.empty(qh.shape[:3], dtype=torch.float32, device="cuda"))
        cases.append(((qb, kb, vb), (qh, kh, vh, oh, lh), staging, torch.cuda.Stream()))
    torch.cuda.synchronize()
    errors = []

    def run(case):
        _, (qh, kh, vh, oh, lh), (qd, kd, vd, od, ld), st = case
        try:
            for _ in range(5):
                ops.attn_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, causal=True, chunk_heads=2, stream=st)
            st.synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(c,)) for c in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for (qb, kb, vb), (_, _, _, oh, lh), _, _ in cases:
        q, k, v = (H.to_device(x, "bf16") for x in (qb, kb, vb))
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
        ops.attn_fwd(q, k, v, o, lse, causal=True)
        torch.cuda.synchronize()
        assert torch.equal(oh, o.cpu()) and torch.equal(lh, lse.cpu())
