"""Parity of attn_fwd_splitk and splitk_combine (through the C ABI) against the FP64 oracle,
and bit-identity of the device-side input generator with the host definition."""
import math

import numpy as np
import pytest

import oracle
import synth
from tests import helpers as H

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
ops = pytest.importorskip("online_softmax_gb300")
sc = pytest.importorskip("synth.cuda")


@pytest.fixture(autouse=True)
def _no_device_errors():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    assert ops.device_error() == 0, "a bounded device wait gave up"


# ------------------------------------------------------------------ generator
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_device_generator_bit_identical(dtype):
    n, start = 1 << 20, 12345
    t = torch.empty(n, dtype=H.torch_dtype(dtype), device="cuda")
    sc.fill_normal(t, 9, synth.STREAM_K, dtype, start=start)
    ref = synth.round_to(synth.normal(9, synth.STREAM_K, start, n), dtype)
    got = t.cpu().numpy() if dtype == "f32" else t.cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got.view(np.uint32) if dtype == "f32" else got,
                          ref.view(np.uint32) if dtype == "f32" else ref)
    u = torch.empty(n, dtype=torch.float32, device="cuda")
    sc.fill_normal(u, 9, synth.STREAM_LSE, "f32", mu=10.0, sigma=2.0)
    assert np.array_equal(u.cpu().numpy(), synth.normal(9, synth.STREAM_LSE, 0, n, 10.0, 2.0))


def test_device_lse_generator_bit_identical():
    P, RH = 5, 20000
    t = sc.fill_lse(torch.empty((P, RH), dtype=torch.float32, device="cuda"), 4)
    assert np.array_equal(t.cpu().numpy(), synth.lse_partials(4, P, RH))


# ------------------------------------------------------------------ combine
def opart_device(seed, P, RH, depth, dtype):
    t = torch.empty((P, RH, depth), dtype=H.torch_dtype(dtype), device="cuda")
    return sc.fill_normal(t, seed, synth.STREAM_OPART, dtype)


def opart_host_rows(seed, P, RH, depth, dtype, rh_idx):
    idx = ((np.arange(P)[:, None] * RH + rh_idx[None, :])[:, :, None] * depth
           + np.arange(depth)[None, None, :])
    z = synth.normal_at(seed, synth.STREAM_OPART, idx.ravel()).reshape(P, len(rh_idx), depth)
    return synth.to_f64(synth.round_to(z, dtype), dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("P", [2, 8, 16, 32, 37])
def test_combine_full_size(P, dtype):
    """4096 tokens x 32 heads, depth 128; lse ~ N(10, 2) with 5% -inf entries and
    0.1% of row-heads all -inf."""
    seed, rows, heads, depth = 21, 4096, 32, 128
    RH = rows * heads
    op = opart_device(seed, P, RH, depth, dtype)
    lp = sc.fill_lse(torch.empty((P, RH), dtype=torch.float32, device="cuda"), seed)
    o = torch.empty((RH, depth), dtype=H.torch_dtype(dtype), device="cuda")
    g = torch.empty(RH, dtype=torch.float32, device="cuda")
    ops.splitk_combine(op, lp, o, g, rows=rows, heads=heads)
    torch.cuda.synchronize()
    rng = np.random.default_rng(P)
    dead = np.flatnonzero(synth.bernoulli(seed, synth.STREAM_ROW_DROP, 0, RH, 0.001))
    rh_idx = np.unique(np.r_[rng.integers(0, RH, 3000), dead, 0, RH - 1])
    O_ref, G_ref = oracle.combine(opart_host_rows(seed, P, RH, depth, dtype, rh_idx),
                                  synth.lse_partials_at(seed, P, RH, rh_idx))
    idx = torch.from_numpy(rh_idx).cuda()
    got = H.to_f64(o[idx])
    if dtype == "f32":
        H.check32(got, O_ref, f"combine P{P} O")
    else:
        H.check16(got, O_ref, f"combine P{P} O")
    H.check32(H.to_f64(g[idx]), G_ref, f"combine P{P} G")
    # row-heads with every partition -inf: exact +0 output and -inf LSE
    assert len(dead) > 0
    od = o[torch.from_numpy(dead).cuda()]
    assert torch.all(od.float() == 0) and not torch.any(torch.signbit(od.float()))
    assert torch.all(torch.isneginf(g[torch.from_numpy(dead).cuda()]))


@pytest.mark.parametrize("P", [1, 2, 3, 4, 5, 8, 16, 32, 64, 100, 256])
@pytest.mark.parametrize("depth,in_dt,out_dt", [(128, "f32", "f32"), (64, "bf16", "bf16"),
                                                (256, "f16", "f32"), (32, "f32", "bf16"),
                                                (16, "bf16", "f16"), (128, "bf16", "f32"),
                                                (128, "f16", "f16"), (64, "f32", "f32")])
def test_combine_small_full_oracle(P, depth, in_dt, out_dt):
    seed, RH = 30 + P, 300
    o_b = synth.tensor(seed, synth.STREAM_OPART, (P, RH, depth), in_dt)
    lse = synth.lse_partials(seed, P, RH, drop=0.2, row_drop=0.02)
    op = H.to_device(o_b, in_dt)
    lp = torch.from_numpy(lse).cuda()
    o = torch.empty((RH, depth), dtype=H.torch_dtype(out_dt), device="cuda")
    g = torch.empty(RH, dtype=torch.float32, device="cuda")
    ops.splitk_combine(op, lp, o, g)
    torch.cuda.synchronize()
    O_ref, G_ref = oracle.combine(synth.to_f64(o_b, in_dt), lse)
    if in_dt == "f32" and out_dt == "f32":
        H.check32(H.to_f64(o), O_ref, "O")
    else:
        H.check16(H.to_f64(o), O_ref, "O")
    H.check32(H.to_f64(g), G_ref, "G")


# ------------------------------------------------------------------ split-K attention
def run_splitk(q, k, v, P, causal, partial="f32"):
    B, Hh, Nq, D = q.shape
    RH = B * Hh * Nq
    pdt = H.torch_dtype(partial) if partial == "f32" else q.dtype
    op = torch.empty((P, RH, D), dtype=pdt, device="cuda")
    lp = torch.empty((P, RH), dtype=torch.float32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, Hh, Nq), dtype=torch.float32, device="cuda")
    ops.attn_fwd_splitk(q, k, v, P, op, lp, o, lse, causal=causal)
    torch.cuda.synchronize()
    return op, lp, o, lse


def check_splitk_full(qb, kb, vb, dtype, P, causal, partial, what):
    B, Hh, Nq, D = qb.shape
    Nkv = kb.shape[2]
    scale = 1.0 / math.sqrt(D)
    q, k, v = (H.to_device(x, dtype) for x in (qb, kb, vb))
    op, lp, o, lse = run_splitk(q, k, v, P, causal, partial)
    qd, kd, vd = (synth.to_f64(x, dtype) for x in (qb, kb, vb))
    chunk = ops.splitk_chunk(Nkv, P)
    assert oracle.splitk_bounds(Nkv, P, 128)[0] == (0, min(chunk, Nkv))
    Op, Lp = oracle.splitk_partials(qd, kd, vd, scale, causal, P, 128)
    O, L = oracle.attention(qd, kd, vd, scale, causal)
    H.check16(H.to_f64(op), Op.reshape(P, -1, D), what + " O_p")
    H.check32(H.to_f64(lp), Lp.reshape(P, -1), what + " lse_p")
    empty = np.isneginf(Lp.reshape(P, -1))
    got = H.to_f64(op).reshape(P, -1, D)[empty]
    assert np.all(got == 0) and not np.any(np.signbit(got)), "empty partitions must store +0"
    H.check16(H.to_f64(o), O, what + " O")
    H.check32(H.to_f64(lse), L, what + " LSE")


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("Nkv,P", [(1, 1), (100, 3), (1000, 8), (1000, 1), (200, 8)])
@pytest.mark.parametrize("dtype,partial", [("bf16", "f32"), ("f16", "f16")])
def test_decode_small(D, Nkv, P, dtype, partial):
    qb, kb, vb = H.qkv_host(40 + D, 2, 3, 1, D, dtype, nkv=Nkv)
    check_splitk_full(qb, kb, vb, dtype, P, False, partial, f"decode D{D} Nkv{Nkv} P{P}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("P", [1, 3, 8])
@pytest.mark.parametrize("D,partial", [(64, "f32"), (128, "bf16"), (32, "f32")])
def test_splitk_prefill_tcgen05(causal, P, D, partial):
    qb, kb, vb = H.qkv_host(50 + P, 1, 2, 1000, D, "bf16")
    check_splitk_full(qb, kb, vb, "bf16", P, causal, partial, f"splitk D{D} P{P} c{causal}")


# ---- full decode size: 64 sequences x 1 query, 32 heads, 32768 keys, D = 128, bf16
def test_decode_full_size_256_row_heads():
    """The decode workload at full size for every P of the workload (4, 8, 16, 37): the
    partials O_p and lse_p, the merged O and the LSE of 256 row-heads (8 sequences
    spread over the batch x all 32 heads) against the FP64 oracle.  K and V (34 GB) are
    drawn once on the device (bit-identical to the host generator) and each checked
    head is copied back for the oracle."""
    B, Hh, Nkv, D, seed = 64, 32, 32768, 128, 5
    Ps = (4, 8, 16, 37)
    q = sc.fill_normal(torch.empty((B, Hh, 1, D), dtype=torch.bfloat16, device="cuda"), seed,
                       synth.STREAM_Q, "bf16")
    k = sc.fill_normal(torch.empty((B, Hh, Nkv, D), dtype=torch.bfloat16, device="cuda"), seed,
                       synth.STREAM_K, "bf16")
    v = sc.fill_normal(torch.empty((B, Hh, Nkv, D), dtype=torch.bfloat16, device="cuda"), seed,
                       synth.STREAM_V, "bf16")
    results = {P: tuple(t.cpu() for t in run_splitk(q, k, v, P, False, "f32")) for P in Ps}
    scale = 1.0 / math.sqrt(D)
    bounds = {P: oracle.splitk_bounds(Nkv, P, 128) for P in Ps}
    seqs = np.linspace(0, B - 1, 8).round().astype(int)
    checked = 0
    for b in seqs:
        for h in range(Hh):
            bh = int(b) * Hh + h
            qr, kh, vh = (H.to_f64(x[b, h]) for x in (q, k, v))
            O, L = oracle.attention_rows(qr, np.array([0]), kh, vh, scale, False)
            for P in Ps:
                op, lp, o, lse = results[P]
                Op, Lp = oracle.splitk_partials_rows(qr, np.array([0]), kh, vh, scale, False, bounds[P])
                H.check16(H.to_f64(op[:, bh]), Op[:, 0], f"decode P{P} b{b} h{h} O_p")
                H.check32(H.to_f64(lp[:, bh]), Lp[:, 0], f"decode P{P} b{b} h{h} lse_p")
                H.check16(H.to_f64(o[b, h]), O, f"decode P{P} b{b} h{h} O")
                H.check32(H.to_f64(lse[b, h]), L, f"decode P{P} b{b} h{h} LSE")
            checked += 1
    assert checked == 256


@pytest.mark.parametrize("Nq", [1, 300])
def test_splitk_max_partitions(Nq):
    """P = 256 (the largest the ABI takes) over 40000 keys: most partitions are empty
    or short; the merged result must still be the attention."""
    qb, kb, vb = H.qkv_host(170 + Nq, 1, 2, Nq, 64, "bf16", nkv=40000)
    B, Hh, _, D = qb.shape
    q, k, v = (H.to_device(x, "bf16") for x in (qb, kb, vb))
    op, lp, o, lse = run_splitk(q, k, v, 256, False, "f32")
    rows = np.unique(np.r_[0, Nq - 1, np.arange(0, Nq, 37)])
    for bh in range(B * Hh):
        qr = synth.to_f64(qb, "bf16")[0, bh, rows]
        kh, vh = synth.to_f64(kb, "bf16")[0, bh], synth.to_f64(vb, "bf16")[0, bh]
        O, L = oracle.attention_rows(qr, rows, kh, vh, 1.0 / math.sqrt(D), False)
        H.check16(H.to_f64(o[0, bh, rows]), O, f"P256 Nq{Nq} bh{bh} O")
        H.check32(H.to_f64(lse[0, bh, rows]), L, f"P256 Nq{Nq} bh{bh} LSE")


@pytest.mark.parametrize("RH", [1, 3, 301, 1027])
@pytest.mark.parametrize("P", [2, 3, 8, 16, 37])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_combine_16bit_rows_ragged_row_heads(RH, P, dtype):
    """16-bit partials at depth 128 (the half-warp-per-row-head kernels, several row-heads
    per half-warp at P = 8) with row-head counts that leave a warp partly empty."""
    seed, depth = 400 + RH + P, 128
    o_b = synth.tensor(seed, synth.STREAM_OPART, (P, RH, depth), dtype)
    lse = synth.lse_partials(seed, P, RH, drop=0.2, row_drop=0.05)
    op = H.to_device(o_b, dtype)
    lp = torch.from_numpy(lse).cuda()
    o = torch.full((RH + 1, depth), 7.0, dtype=H.torch_dtype(dtype), device="cuda")  # one guard row
    g = torch.full((RH + 1,), 7.0, dtype=torch.float32, device="cuda")
    ops.splitk_combine(op, lp, o[:RH], g[:RH])
    torch.cuda.synchronize()
    O_ref, G_ref = oracle.combine(synth.to_f64(o_b, dtype), lse)
    H.check16(H.to_f64(o[:RH]), O_ref, f"RH{RH} P{P} O")
    H.check32(H.to_f64(g[:RH]), G_ref, f"RH{RH} P{P} G")
    assert torch.all(o[RH] == 7.0) and g[RH].item() == 7.0, "a row-head past the end was written"
