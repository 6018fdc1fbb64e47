"""The bounded-wait failure path on the GPU, without a fault: a wait on an mbarrier phase
that never completes gives up after the library's limit (2 s), records its site code in
the device status word and raises its CTA's abort flag; the CTA's other waiting warp
leaves through that flag before its own limit; the kernel returns and the context stays
usable for the next call."""
import math

import pytest

import oracle
import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
ops = pytest.importorskip("online_softmax_gb300")


def test_wait_gives_up_and_the_context_survives():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    assert ops.device_error() == 0
    flags = torch.full((2,), 7, dtype=torch.int32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    ops.selftest_wait(flags)
    e1.record()
    torch.cuda.synchronize()
    seconds = e0.elapsed_time(e1) / 1e3
    assert flags.tolist() == [0, 0], "both waits must have given up"
    assert ops.device_error() == ops.SELFTEST_SITE
    assert ops.device_error() == 0, "reading the status word clears it"
    # thread 0 gives up at the 2 s limit; the second warp, whose own limit ends 0.5 s
    # later, must have left through the abort flag before that
    assert 1.9 < seconds < 2.45, seconds
    # the context still works: a small causal attention call against the oracle
    qb, kb, vb = H.qkv_host(195, 1, 2, 200, 64, "bf16")
    q, k, v = (H.to_device(x, "bf16") for x in (qb, kb, vb))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    ops.attn_fwd(q, k, v, o, lse, causal=True)
    torch.cuda.synchronize()
    O, L = oracle.attention(synth.to_f64(qb, "bf16"), synth.to_f64(kb, "bf16"), synth.to_f64(vb, "bf16"),
                            1.0 / math.sqrt(64), True)
    H.check16(H.to_f64(o), O, "O after the self-test")
    H.check32(H.to_f64(lse), L, "LSE after the self-test")
    assert ops.device_error() == 0


def test_selftest_rejects_a_misaligned_flags_pointer():
    flags = torch.zeros(4, dtype=torch.int32, device="cuda")
    import ctypes
    st = ops.lib.oattn_selftest_wait(ctypes.c_void_p(flags.data_ptr() + 2), None)
    assert st == 1  # OATTN_ERR_INVALID_ARG, nothing launched
    assert ops.device_error() == 0
