"""Parity of attn_fwd (tcgen05/TMA kernel, through the C ABI) against the FP64 oracle."""
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


def run_attn(q, k, v, causal, block_n=0, scale=None, with_lse=True):
    B, Hh, N, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hh, N), dtype=torch.float32, device=q.device) if with_lse else None
    ops.attn_fwd_bn(q, k, v, o, lse, causal=causal, scale=scale, block_n=block_n)
    torch.cuda.synchronize()
    return o, lse


def check_full(qb, kb, vb, dtype, causal, block_n=0, scale=None, what=""):
    D = qb.shape[-1]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    q, k, v = (H.to_device(x, dtype) for x in (qb, kb, vb))
    o, lse = run_attn(q, k, v, causal, block_n, scale)
    O_ref, L_ref = oracle.attention(synth.to_f64(qb, dtype), synth.to_f64(kb, dtype),
                                    synth.to_f64(vb, dtype), scale, causal)
    H.check16(H.to_f64(o), O_ref, what + " O")
    H.check32(H.to_f64(lse), L_ref, what + " LSE")


def test_single_head_n128_d64():
    """B=1, H=1, N=128, D=64, bf16, non-causal, scale 1/sqrt(D)."""
    qb, kb, vb = H.qkv_host(1, 1, 1, 128, 64, "bf16")
    check_full(qb, kb, vb, "bf16", False, what="n128")


# The workshop's case matrix: D x N x dtype x causal x BN, three value regimes.
@pytest.mark.parametrize("regime", ["normal", "uniform", "large"])
@pytest.mark.parametrize("block_n", [32, 64])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("N", [1, 1000, 2048])
@pytest.mark.parametrize("D", [16, 32, 64])
def test_workshop_sweep(D, N, dtype, causal, block_n, regime):
    seed = 100 + D + N % 7
    qb, kb, vb = H.qkv_host(seed, 1, 1, N, D, dtype)
    if regime == "uniform":
        qb = synth.round_to(np.zeros(qb.shape, np.float32), dtype)
    elif regime == "large":  # Q scaled by 8 (a power of two: exact in both dtypes)
        qb = synth.round_to((synth.to_f64(qb, dtype) * 8.0).astype(np.float32), dtype)
    check_full(qb, kb, vb, dtype, causal, block_n, what=f"D{D} N{N} {dtype} c{causal} bn{block_n} {regime}")


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_default_tile_multihead_ragged(D, causal):
    qb, kb, vb = H.qkv_host(7, 2, 3, 333, D, "bf16")
    check_full(qb, kb, vb, "bf16", causal, what=f"D{D} multihead")


# attn_fwd runs one CTA per SM walking work units (a query-tile pair, or for causal the
# pairs p and npairs-1-p of one head) in groups of 8 heads.  These shapes give an odd
# number of pairs (a unit holding the middle pair alone), a last pair whose second query
# tile is past the end (N % 256 <= 128), head counts that are not a multiple of 8 and
# more units than SMs; every row is compared with the oracle.
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hh,N,D", [(1, 37, 1100, 64), (2, 19, 2000, 128), (3, 5, 130, 32)])
def test_persistent_work_units(B, Hh, N, D, causal):
    qb, kb, vb = H.qkv_host(41 + N % 13, B, Hh, N, D, "bf16")
    check_full(qb, kb, vb, "bf16", causal, what=f"B{B} H{Hh} N{N} D{D} c{causal}")


@pytest.mark.parametrize("block_n", [32, 64, 128])
def test_d128_tiles_and_scale(block_n):
    qb, kb, vb = H.qkv_host(8, 1, 2, 700, 128, "f16")
    check_full(qb, kb, vb, "f16", True, block_n, scale=0.3, what=f"d128 bn{block_n}")


def test_lse_optional_and_n_zero():
    qb, kb, vb = H.qkv_host(9, 1, 1, 200, 64, "bf16")
    q, k, v = (H.to_device(x, "bf16") for x in (qb, kb, vb))
    o1, l1 = run_attn(q, k, v, True)
    o2, _ = run_attn(q, k, v, True, with_lse=False)
    assert torch.equal(o1, o2)
    z = torch.empty((1, 1, 0, 64), dtype=torch.bfloat16, device="cuda")
    ops.attn_fwd(z, z, z, torch.empty_like(z), None)


def test_causal_future_perturbation_bitwise():
    """Changing K and V rows at and after j leaves every earlier causal row bit-identical."""
    N, D = 1000, 64
    qb, kb, vb = H.qkv_host(11, 1, 2, N, D, "bf16")
    q, k, v = (H.to_device(x, "bf16") for x in (qb, kb, vb))
    o, lse = run_attn(q, k, v, True)
    for j in (1, 300, 512, 999):
        k2, v2 = k.clone(), v.clone()
        k2[:, :, j:] = torch.randn_like(k2[:, :, j:])
        v2[:, :, j:] = torch.randn_like(v2[:, :, j:])
        o2, lse2 = run_attn(q, k2, v2, True)
        assert torch.equal(o2[:, :, :j], o[:, :, :j]), f"row < {j} changed"
        assert torch.equal(lse2[:, :, :j], lse[:, :, :j])
        assert not torch.equal(o2[:, :, j:], o[:, :, j:])


# ---- full prefill size: B=4, H=32, N=4096, D=128, bf16 (inputs drawn on the device)
PREFILL = dict(B=4, H=32, N=4096, D=128, seed=3)


def prefill_inputs(dtype="bf16"):
    import synth.cuda as sc
    B, Hh, N, D, seed = (PREFILL[x] for x in ("B", "H", "N", "D", "seed"))
    t = lambda: torch.empty((B, Hh, N, D), dtype=H.torch_dtype(dtype), device="cuda")
    q = sc.fill_normal(t(), seed, synth.STREAM_Q, dtype)
    k = sc.fill_normal(t(), seed, synth.STREAM_K, dtype)
    v = sc.fill_normal(t(), seed, synth.STREAM_V, dtype)
    return q, k, v


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_full_size_every_row(causal):
    """The whole prefill problem (B=4, H=32, N=4096, D=128, bf16) against the FP64 oracle:
    every row of every head, in the launch configuration the bench times.  The inputs
    are drawn on the device (bit-identical to the host generator, see
    test_device_generator_bit_identical) and each head is copied back to the host for
    the oracle, so a fault in how CTAs map to heads, query tiles or rows cannot hide
    behind a sample."""
    B, Hh, N, D = (PREFILL[x] for x in ("B", "H", "N", "D"))
    q, k, v = prefill_inputs()
    o, lse = run_attn(q, k, v, causal)
    scale = 1.0 / math.sqrt(D)
    worst16, worst32 = 0.0, 0.0
    for bh in range(B * Hh):
        b, h = divmod(bh, Hh)
        O_ref, L_ref = oracle.attention(H.to_f64(q[b, h]), H.to_f64(k[b, h]), H.to_f64(v[b, h]), scale, causal)
        max_abs, _ = H.check16(H.to_f64(o[b, h]), O_ref, f"prefill b{b} h{h} O")
        worst16 = max(worst16, max_abs)
        worst32 = max(worst32, H.check32(H.to_f64(lse[b, h]), L_ref, f"prefill b{b} h{h} LSE"))
    print(f"prefill causal={causal}: {B * Hh} heads x {N} rows, worst O max-abs {worst16:.2e}, "
          f"worst LSE error {worst32:.2f} of the bound")


def test_prefill_deterministic():
    q, k, v = prefill_inputs()
    o1, l1 = run_attn(q, k, v, True)
    o2, l2 = run_attn(q, k, v, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_growing_scores_move_the_stabiliser(causal, dtype):
    """Scores that grow from key tile to key tile (K rows scaled up along the sequence)
    make the kernel move its stabiliser again and again (redo a tile against the exact
    maximum, rescale O and l); the result must still match the oracle."""
    N, D = 1000, 64
    qb, kb, vb = H.qkv_host(12, 1, 2, N, D, dtype)
    ramp = 1.0 + np.arange(N, dtype=np.float64) / 40.0  # row maximum grows ~25x along the keys
    kb = synth.round_to((synth.to_f64(kb, dtype) * ramp[None, None, :, None]).astype(np.float32), dtype)
    check_full(qb, kb, vb, dtype, causal, what=f"growing scores {dtype} c{causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_sampled(causal):
    """N = 16384 (four times the prefill length), D = 128, bf16: sampled rows, tile
    boundaries and the last row included, against the oracle."""
    import synth.cuda as sc
    B, Hh, N, D, seed = 1, 2, 16384, 128, 13
    t = lambda: torch.empty((B, Hh, N, D), dtype=torch.bfloat16, device="cuda")
    q = sc.fill_normal(t(), seed, synth.STREAM_Q, "bf16")
    k = sc.fill_normal(t(), seed, synth.STREAM_K, "bf16")
    v = sc.fill_normal(t(), seed, synth.STREAM_V, "bf16")
    o, lse = run_attn(q, k, v, causal)
    rows = np.unique(np.r_[0, 127, 128, 255, 256, 8191, 8192, 16383, np.random.default_rng(7).integers(0, N, 24)])
    for bh in range(B * Hh):
        qr = H.head_slice(seed, synth.STREAM_Q, bh, N, D, "bf16", rows)
        kh = H.head_slice(seed, synth.STREAM_K, bh, N, D, "bf16")
        vh = H.head_slice(seed, synth.STREAM_V, bh, N, D, "bf16")
        O_ref, L_ref = oracle.attention_rows(qr, rows, kh, vh, 1.0 / math.sqrt(D), causal)
        H.check16(H.to_f64(o[0, bh, rows]), O_ref, f"long bh{bh} O")
        H.check32(H.to_f64(lse[0, bh, rows]), L_ref, f"long bh{bh} LSE")


def test_second_copy_of_the_library_in_one_process(tmp_path):
    """A second copy of the library loaded next to the first keeps its own per-device
    set-up (kernel attributes, status word): both copies launch and agree bit for bit."""
    import ctypes
    import shutil
    copy = tmp_path / "liboattn_copy.so"
    shutil.copy(ops.library_path, copy)
    L2 = ctypes.CDLL(str(copy))
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    L2.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    qb, kb, vb = H.qkv_host(190, 1, 2, 300, 128, "bf16")
    q, k, v = (H.to_device(x, "bf16") for x in (qb, kb, vb))
    o1, l1 = run_attn(q, k, v, True)
    o2, l2 = torch.empty_like(q), torch.empty_like(l1)
    st = torch.cuda.current_stream().cuda_stream
    rc = L2.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), l2.data_ptr(), 1, 2, 300, 128, 1,
                     1.0 / math.sqrt(128), ops.BF16, st)
    torch.cuda.synchronize()
    assert rc == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
