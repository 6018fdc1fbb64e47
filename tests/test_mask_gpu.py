"""Parity of the optional Boolean mask path (attn_mask_pack, attn_fwd_masked,
attn_fwd_splitk_masked, through the C ABI) against the FP64 oracle, and of the packed
layout against its plain definition."""
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


def pack_definition(mask: np.ndarray) -> np.ndarray:
    """The packed layout written out: W = 4*ceil(nk/128) words per row, bit j of word w
    is key 32*w + j, bits past nk zero."""
    m = np.asarray(mask, dtype=bool)
    nk = m.shape[-1]
    W = 4 * (-(-nk // 128))
    padded = np.zeros(m.shape[:-1] + (32 * W,), dtype=np.uint64)
    padded[..., :nk] = m
    lanes = padded.reshape(m.shape[:-1] + (W, 32)) << np.arange(32, dtype=np.uint64)
    return lanes.sum(axis=-1).astype(np.uint32)


def mask_kind(kind, seed, shape):
    """Seeded masks of the recipes in synth, shaped [..., nq, nk]."""
    nq, nk = shape[-2:]
    if kind == "random":
        m = synth.mask_random(seed, shape, 0.5)
    elif kind == "sparse":  # mostly hidden, some rows fully hidden
        m = synth.hide_rows(seed, synth.mask_random(seed, shape, 0.05), 0.1)
    elif kind == "band":
        m = np.broadcast_to(synth.mask_band(nq, nk, 37), shape)
    elif kind == "blocks":
        m = np.broadcast_to(synth.mask_blocks(seed, nq, nk, 64, 0.5), shape)
    else:
        raise ValueError(kind)
    return np.ascontiguousarray(m)


def to_bool(mask):
    return torch.from_numpy(np.array(mask, dtype=bool, copy=True)).cuda()


def check_rows_hidden(o, lse, mask_full, causal):
    """Rows whose every key is hidden: output exactly +0, LSE -inf."""
    nq, nk = mask_full.shape[-2:]
    vis = mask_full & oracle.visible(nq, nk, causal)
    dead = ~vis.any(axis=-1)
    if dead.any():
        got = H.to_f64(o)[dead]
        assert np.all(got == 0) and not np.any(np.signbit(got)), "hidden rows must store +0"
        assert np.all(np.isneginf(H.to_f64(lse)[dead])), "hidden rows must have LSE -inf"
    return int(dead.sum())


# ------------------------------------------------------------------ packing
@pytest.mark.parametrize("nk", [1, 31, 32, 33, 127, 128, 129, 1000, 4100])
@pytest.mark.parametrize("layout", ["bool", "bytes", "strided_odd", "strided16"])
def test_mask_pack_matches_definition(nk, layout):
    rows = 37
    m = synth.mask_random(11 + nk, (rows, nk), 0.5)
    if layout == "bool":
        t = to_bool(m)
    elif layout == "bytes":  # nonzero bytes of any value count as visible
        vals = (synth.words(12, synth.STREAM_MASK, 0, rows * nk) % np.uint64(255) + np.uint64(1)).astype(np.uint8)
        t = torch.from_numpy(np.where(m.ravel(), vals, 0).astype(np.uint8).reshape(rows, nk)).cuda()
    else:  # rows inside a wider buffer (odd stride: byte path; multiple of 16: vector path)
        stride = nk + 3 if layout == "strided_odd" else 16 * (-(-nk // 16)) + 16
        buf = torch.ones((rows, stride), dtype=torch.bool, device="cuda")
        buf[:, :nk] = to_bool(m)
        t = buf[:, :nk]
    bits = ops.attn_mask_pack(t)
    torch.cuda.synchronize()
    got = bits.cpu().numpy().view(np.uint32)
    assert got.shape == (rows, ops.attn_mask_words(nk))
    assert np.array_equal(got, pack_definition(m))


def test_mask_pack_leading_dims():
    m = synth.mask_random(13, (2, 3, 5, 200), 0.3)
    got = ops.attn_mask_pack(to_bool(m)).cpu().numpy().view(np.uint32)
    assert np.array_equal(got, pack_definition(m))


# ------------------------------------------------------------------ attention
def run_masked(q, k, v, mask, causal, scale=None):
    B, Hh, N, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, Hh, N), dtype=torch.float32, device="cuda")
    ops.attn_fwd_masked(q, k, v, o, mask, lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o, lse


def check_masked(qb, kb, vb, dtype, mask, causal, what, packed=False):
    B, Hh, N, D = qb.shape
    scale = 1.0 / math.sqrt(D)
    q, k, v = (H.to_device(x, dtype) for x in (qb, kb, vb))
    m = to_bool(mask)
    if packed:
        m = ops.attn_mask_pack(m)
    o, lse = run_masked(q, k, v, m, causal)
    O_ref, L_ref = oracle.attention(synth.to_f64(qb, dtype), synth.to_f64(kb, dtype),
                                    synth.to_f64(vb, dtype), scale, causal, mask=mask)
    H.check16(H.to_f64(o), O_ref, what + " O")
    H.check32(H.to_f64(lse), L_ref, what + " LSE")
    return check_rows_hidden(o, lse, np.broadcast_to(mask, (B, Hh, N, N)), causal)


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("N", [1, 77, 300])
@pytest.mark.parametrize("kind", ["random", "sparse", "band", "blocks"])
@pytest.mark.parametrize("causal", [False, True])
def test_masked_attention_shared_mask(D, N, kind, causal):
    qb, kb, vb = H.qkv_host(60 + D + N, 2, 3, N, D, "bf16")
    mask = mask_kind(kind, 7 + N, (N, N))
    check_masked(qb, kb, vb, "bf16", mask, causal, f"D{D} N{N} {kind} c{causal}")


@pytest.mark.parametrize("D,dtype", [(64, "f16"), (128, "bf16"), (32, "bf16")])
@pytest.mark.parametrize("causal", [False, True])
def test_masked_attention_per_head_mask(D, dtype, causal):
    N = 261
    qb, kb, vb = H.qkv_host(70 + D, 2, 3, N, D, dtype)
    mask = mask_kind("sparse", 71, (2, 3, N, N))
    dead = check_masked(qb, kb, vb, dtype, mask, causal, f"per-head D{D} {dtype} c{causal}", packed=True)
    assert dead > 0  # the recipe hides whole rows; make sure the case is exercised


def test_all_visible_mask_is_bitwise_unmasked():
    """An all-True mask takes the whole-tile path: the result must be the unmasked
    kernel's, bit for bit."""
    for causal in (False, True):
        qb, kb, vb = H.qkv_host(81, 2, 2, 300, 128, "bf16")
        q, k, v = (H.to_device(x, "bf16") for x in (qb, kb, vb))
        o1, l1 = run_masked(q, k, v, torch.ones((300, 300), dtype=torch.bool, device="cuda"), causal)
        o2 = torch.empty_like(q)
        l2 = torch.empty_like(l1)
        ops.attn_fwd(q, k, v, o2, l2, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_key_padding_mask(causal):
    """A [B, 1, 1, N] key-padding mask reaches the kernel with zero head and query
    strides (the rows are shared)."""
    B, Hh, N, D = 3, 2, 200, 64
    qb, kb, vb = H.qkv_host(91, B, Hh, N, D, "bf16")
    mask = synth.key_padding(92, B, N, min_len=1)
    check_masked(qb, kb, vb, "bf16", mask, causal, f"key padding c{causal}")


def test_fully_hidden_problem():
    qb, kb, vb = H.qkv_host(93, 1, 2, 130, 64, "bf16")
    dead = check_masked(qb, kb, vb, "bf16", np.zeros((130, 130), bool), False, "all hidden")
    assert dead == 2 * 130


# ------------------------------------------------------------------ skipped key tiles
def skip_masks(N):
    """Masks whose key tiles are invisible to whole CTAs (256 query rows) or whole query
    tiles (128 rows), so the masked kernel walks only part of the key range."""
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    out = {}
    out["window 100"] = synth.mask_band(N, N, 100)
    # rows 0-127 see nothing; rows 128-255 only keys 128-255; the rest a 300-key window
    m = synth.mask_band(N, N, 300)
    m[:128] = False
    m[128:256] = (j >= 128) & (j < 256)
    out["first tile hidden"] = m
    # one whole CTA (rows 256-511) sees nothing; key tiles 0 and 5 only for the others
    m = ((j // 128) == 0) | ((j // 128) == 5)
    m = np.broadcast_to(m, (N, N)).copy()
    m[256:512] = False
    out["CTA hidden, tiles 0 and 5"] = m
    # short key padding: keys 0-99 only
    out["keys 0-99"] = np.broadcast_to(j < 100, (N, N)).copy()
    return out


@pytest.mark.parametrize("name", ["window 100", "first tile hidden", "CTA hidden, tiles 0 and 5", "keys 0-99"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_masked_tiles_skipped(name, causal, D):
    N = 1100
    qb, kb, vb = H.qkv_host(200 + D, 1, 2, N, D, "bf16")
    mask = skip_masks(N)[name]
    dead = check_masked(qb, kb, vb, "bf16", mask, causal, f"{name} D{D} c{causal}")
    if name in ("first tile hidden", "CTA hidden, tiles 0 and 5"):
        assert dead > 0  # the recipe hides whole query tiles; make sure they are exercised


def test_masked_tiles_skipped_split_k():
    N = 1100
    qb, kb, vb = H.qkv_host(210, 1, 2, N, 128, "bf16")
    for name, mask in skip_masks(N).items():
        for causal in (False, True):
            check_splitk_masked(qb, kb, vb, "bf16", 3, mask, causal, "f32", f"split {name} c{causal}")


# ------------------------------------------------------------------ split-K
def run_splitk_masked(q, k, v, P, mask, causal, partial="f32"):
    B, Hh, Nq, D = q.shape
    RH = B * Hh * Nq
    pdt = torch.float32 if partial == "f32" else q.dtype
    op = torch.empty((P, RH, D), dtype=pdt, device="cuda")
    lp = torch.empty((P, RH), dtype=torch.float32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, Hh, Nq), dtype=torch.float32, device="cuda")
    ops.attn_fwd_splitk_masked(q, k, v, P, op, lp, mask, o, lse, causal=causal)
    torch.cuda.synchronize()
    return op, lp, o, lse


def check_splitk_masked(qb, kb, vb, dtype, P, mask, causal, partial, what):
    B, Hh, Nq, D = qb.shape
    scale = 1.0 / math.sqrt(D)
    q, k, v = (H.to_device(x, dtype) for x in (qb, kb, vb))
    op, lp, o, lse = run_splitk_masked(q, k, v, P, to_bool(mask), causal, partial)
    qd, kd, vd = (synth.to_f64(x, dtype) for x in (qb, kb, vb))
    Op, Lp = oracle.splitk_partials(qd, kd, vd, scale, causal, P, 128, mask=mask)
    O, L = oracle.attention(qd, kd, vd, scale, causal, mask=mask)
    H.check16(H.to_f64(op), Op.reshape(P, -1, D), what + " O_p")
    H.check32(H.to_f64(lp), Lp.reshape(P, -1), what + " lse_p")
    empty = np.isneginf(Lp.reshape(P, -1))
    got = H.to_f64(op).reshape(P, -1, D)[empty]
    assert np.all(got == 0) and not np.any(np.signbit(got)), "hidden partitions must store +0"
    H.check16(H.to_f64(o), O, what + " O")
    H.check32(H.to_f64(lse), L, what + " LSE")


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("Nkv,P", [(1, 1), (300, 3), (1000, 8), (2000, 1)])
@pytest.mark.parametrize("kind", ["padding", "random", "sparse"])
def test_decode_masked(D, Nkv, P, kind):
    B, Hh = 3, 2
    qb, kb, vb = H.qkv_host(100 + D, B, Hh, 1, D, "bf16", nkv=Nkv)
    if kind == "padding":
        mask = synth.key_padding(101 + Nkv, B, Nkv, min_len=1)
    else:
        mask = mask_kind(kind, 102 + Nkv, (B, Hh, 1, Nkv))
    check_splitk_masked(qb, kb, vb, "bf16", P, mask, False, "f32", f"decode D{D} Nkv{Nkv} P{P} {kind}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("P", [1, 3, 8])
@pytest.mark.parametrize("kind", ["random", "band", "sparse"])
def test_splitk_prefill_masked(causal, P, kind):
    qb, kb, vb = H.qkv_host(110 + P, 1, 2, 700, 64, "bf16")
    mask = mask_kind(kind, 111, (700, 700))
    check_splitk_masked(qb, kb, vb, "bf16", P, mask, causal, "f32", f"splitk P{P} {kind} c{causal}")


# ------------------------------------------------------------------ full prefill size
def test_masked_prefill_full_size_sampled():
    """B=4, H=32, N=4096, D=128, bf16, causal, one shared sliding-window mask (width
    1024) with some rows hidden; sampled rows against the oracle."""
    import synth.cuda as sc
    B, Hh, N, D, seed = 4, 32, 4096, 128, 3
    t = lambda: torch.empty((B, Hh, N, D), dtype=torch.bfloat16, device="cuda")
    q = sc.fill_normal(t(), seed, synth.STREAM_Q, "bf16")
    k = sc.fill_normal(t(), seed, synth.STREAM_K, "bf16")
    v = sc.fill_normal(t(), seed, synth.STREAM_V, "bf16")
    mask = synth.hide_rows(17, synth.mask_band(N, N, 1024), 0.01)
    o, lse = run_masked(q, k, v, to_bool(mask), True)
    hidden = np.flatnonzero(~mask.any(axis=1))
    assert hidden.size > 0
    rng = np.random.default_rng(6)
    rows = np.unique(np.r_[0, 1, 127, 128, 1023, 1024, 2047, 4095, hidden[:8], rng.integers(0, N, 48)])
    for bh in (0, 37, B * Hh - 1):
        qr = H.head_slice(seed, synth.STREAM_Q, bh, N, D, "bf16", rows)
        kh = H.head_slice(seed, synth.STREAM_K, bh, N, D, "bf16")
        vh = H.head_slice(seed, synth.STREAM_V, bh, N, D, "bf16")
        O_ref, L_ref = oracle.attention_rows(qr, rows, kh, vh, 1.0 / math.sqrt(D), True, mask_rows=mask[rows])
        b, h = divmod(bh, Hh)
        H.check16(H.to_f64(o[b, h, rows]), O_ref, f"masked prefill bh{bh} O")
        H.check32(H.to_f64(lse[b, h, rows]), L_ref, f"masked prefill bh{bh} LSE")
    dead = H.to_f64(o[:, :, hidden])
    assert np.all(dead == 0) and not np.any(np.signbit(dead))
    assert torch.isneginf(lse[:, :, hidden]).all()
