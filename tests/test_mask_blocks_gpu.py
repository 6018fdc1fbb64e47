"""The block summary of a mask (attn_mask_blocks) against its plain definition, and the
persistent masked forward that walks it (attn_fwd_masked_blocks, through the C ABI)
against the FP64 oracle and, bit for bit, against attn_fwd_masked: both visit the key
tiles in ascending order and a tile that a row cannot see adds exact zeros, so the
summary changes which hidden tiles are visited, never a result."""
import math

import numpy as np
import pytest

import oracle
import synth
from tests import helpers as H
from tests.test_mask_gpu import check_rows_hidden, mask_kind, skip_masks, to_bool

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
ops = pytest.importorskip("online_softmax_gb300")


@pytest.fixture(autouse=True)
def _no_device_errors():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    yield
    assert ops.device_error() == 0, "a bounded device wait gave up"


def summary_definition(mask: np.ndarray) -> np.ndarray:
    """The summary written out: for each leading index, block of 256 rows p and key tile
    j of 128 keys, bit j % 32 of word j // 32 of the block is any(mask[rows, keys])."""
    m = np.asarray(mask, dtype=bool)
    nq, nk = m.shape[-2:]
    nblk, ntiles = -(-nq // 256), -(-nk // 128)
    wpb = -(-ntiles // 32)
    pad = np.zeros(m.shape[:-2] + (nblk * 256, ntiles * 128), dtype=bool)
    pad[..., :nq, :nk] = m
    blk = pad.reshape(m.shape[:-2] + (nblk, 256, ntiles, 128)).any(axis=(-3, -1))
    bits = np.zeros(m.shape[:-2] + (nblk, wpb * 32), dtype=np.uint64)
    bits[..., :ntiles] = blk
    words = (bits.reshape(m.shape[:-2] + (nblk, wpb, 32)) << np.arange(32, dtype=np.uint64)).sum(axis=-1)
    return words.astype(np.uint32).ravel()


@pytest.mark.parametrize("layout,B,Hh,nq,nk", [
    ("shared", 2, 3, 300, 300), ("shared", 1, 1, 4096, 4096), ("per-head", 2, 3, 261, 261),
    ("per-batch", 3, 2, 520, 1000), ("key-padding", 3, 2, 200, 5000), ("shared", 1, 2, 1, 1),
    ("per-head", 1, 2, 700, 4200),
])
def test_summary_matches_definition(layout, B, Hh, nq, nk):
    seed = 300 + nq + nk
    if layout == "shared":
        m = synth.hide_rows(seed, synth.mask_random(seed, (nq, nk), 0.002), 0.2)
        full = m
    elif layout == "per-head":
        m = mask_kind("sparse", seed, (B, Hh, nq, nk))
        full = m
    elif layout == "per-batch":
        m = synth.mask_random(seed, (B, 1, nq, nk), 0.001)
        full = m[:, 0]
    else:  # [B, 1, 1, nk]: zero head and query strides
        m = synth.key_padding(seed, B, nk, min_len=1)
        full = np.broadcast_to(m[:, :, 0, :], (B, nq, nk))
    got = ops.attn_mask_blocks(to_bool(m), B, Hh, nq, nk).cpu().numpy().view(np.uint32)
    want = summary_definition(full)
    assert got.size >= want.size
    assert np.array_equal(got[:want.size], want)


def run_pair(q, k, v, mask, causal):
    """attn_fwd_masked_blocks (with a fresh summary) and attn_fwd_masked on the same mask."""
    B, Hh, N, D = q.shape
    bits = ops.attn_mask_pack(mask) if mask.dtype == torch.bool else mask
    blocks = ops.attn_mask_blocks(bits, B, Hh, N)
    out = []
    for use_blocks in (True, False):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hh, N), float("nan"), dtype=torch.float32, device="cuda")
        if use_blocks:
            ops.attn_fwd_masked_blocks(q, k, v, o, bits, blocks, lse, causal=causal)
        else:
            ops.attn_fwd_masked(q, k, v, o, bits, lse, causal=causal)
        torch.cuda.synchronize()
        out.append((o, lse))
    return out


def check_blocks(qb, kb, vb, dtype, mask, causal, what, heads=None):
    B, Hh, N, D = qb.shape
    q, k, v = (H.to_device(x, dtype) for x in (qb, kb, vb))
    (o, lse), (o2, l2) = run_pair(q, k, v, to_bool(mask), causal)
    assert torch.equal(o, o2) and torch.equal(lse, l2), what + ": differs from attn_fwd_masked"
    scale = 1.0 / math.sqrt(D)
    full = np.broadcast_to(mask, (B, Hh, N, N))
    if heads is None:
        O_ref, L_ref = oracle.attention(synth.to_f64(qb, dtype), synth.to_f64(kb, dtype),
                                        synth.to_f64(vb, dtype), scale, causal, mask=mask)
        H.check16(H.to_f64(o), O_ref, what + " O")
        H.check32(H.to_f64(lse), L_ref, what + " LSE")
    else:
        for b, h in heads:
            sl = lambda x: x[b:b + 1, h:h + 1]
            O_ref, L_ref = oracle.attention(synth.to_f64(sl(qb), dtype), synth.to_f64(sl(kb), dtype),
                                            synth.to_f64(sl(vb), dtype), scale, causal, mask=full[b, h])
            H.check16(H.to_f64(o[b:b + 1, h:h + 1]), O_ref, f"{what} head ({b},{h}) O")
            H.check32(H.to_f64(lse[b:b + 1, h:h + 1]), L_ref, f"{what} head ({b},{h}) LSE")
    return check_rows_hidden(o, lse, full, causal)


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("N", [1, 77, 300, 1100])
@pytest.mark.parametrize("kind", ["random", "sparse", "band", "blocks"])
@pytest.mark.parametrize("causal", [False, True])
def test_blocks_shared_mask(D, N, kind, causal):
    qb, kb, vb = H.qkv_host(400 + D + N, 2, 3, N, D, "bf16")
    mask = mask_kind(kind, 9 + N, (N, N))
    check_blocks(qb, kb, vb, "bf16", mask, causal, f"blocks D{D} N{N} {kind} c{causal}")


@pytest.mark.parametrize("name", ["window 100", "first tile hidden", "CTA hidden, tiles 0 and 5", "keys 0-99"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(64, "f16"), (128, "bf16")])
def test_blocks_skipped_tiles(name, causal, D, dtype):
    """Masks that leave whole query tiles, whole 256-row blocks and runs of key tiles
    unmarked: a query tile with nothing marked writes +0 and -inf."""
    N = 1100
    qb, kb, vb = H.qkv_host(410 + D, 1, 2, N, D, dtype)
    dead = check_blocks(qb, kb, vb, dtype, skip_masks(N)[name], causal, f"blocks {name} D{D} c{causal}")
    if name in ("first tile hidden", "CTA hidden, tiles 0 and 5"):
        assert dead > 0


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,dtype", [(32, "bf16"), (128, "f16")])
def test_blocks_per_head_mask(causal, D, dtype):
    """Per-head masks (nonzero batch and head strides) with hidden rows and a head whose
    block 1 is hidden altogether."""
    B, Hh, N = 2, 3, 600
    qb, kb, vb = H.qkv_host(420 + D, B, Hh, N, D, dtype)
    mask = mask_kind("sparse", 421, (B, Hh, N, N))
    mask[1, 2, 256:512] = False
    dead = check_blocks(qb, kb, vb, dtype, mask, causal, f"blocks per-head D{D} c{causal}")
    assert dead >= 256


@pytest.mark.parametrize("causal", [False, True])
def test_blocks_key_padding(causal):
    B, Hh, N, D = 3, 2, 700, 64
    qb, kb, vb = H.qkv_host(430, B, Hh, N, D, "bf16")
    check_blocks(qb, kb, vb, "bf16", synth.key_padding(431, B, N, min_len=1), causal, f"blocks padding c{causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_blocks_many_units_per_cta(causal):
    """More work units than SMs (B*H = 320 heads of 1100 rows): each CTA walks several
    units and finds each item's summary words by its position in the CTA's list.  The
    per-head masks differ, so a wrong position shows."""
    B, Hh, N, D = 4, 80, 1100, 32
    qb, kb, vb = H.qkv_host(440, B, Hh, N, D, "bf16")
    mask = np.empty((B, Hh, N, N), dtype=bool)
    j = np.arange(N)
    for b in range(B):
        for h in range(Hh):
            w = 64 + 37 * ((b * Hh + h) % 23)  # a band of its own per head
            mask[b, h] = np.abs(j[:, None] - j[None, :]) < w
            if (b * Hh + h) % 7 == 3:
                mask[b, h, 512:768] = False  # a hidden block
    check_blocks(qb, kb, vb, "bf16", mask, causal, f"blocks many units c{causal}",
                 heads=[(0, 0), (1, 3), (2, 45), (3, 79)])


@pytest.mark.parametrize("causal", [False, True])
def test_blocks_two_summary_words(causal):
    """N = 5000: 40 key tiles, two summary words per block, per-head masks (the head
    stride of the summary counts whole blocks of two words).  Head 0's band leaves key
    tile 31 hidden, so its walk jumps from word 0 to word 1."""
    B, Hh, N, D = 1, 2, 5000, 64
    qb, kb, vb = H.qkv_host(470, B, Hh, N, D, "bf16")
    m0 = synth.mask_band(N, N, 600)
    m0[:, (np.arange(N) // 128) == 31] = False
    mask = np.stack([m0, synth.mask_band(N, N, 1500)])[None]
    check_blocks(qb, kb, vb, "bf16", mask, causal, f"blocks two words c{causal}")


def test_blocks_all_visible_is_bitwise_unmasked():
    for causal in (False, True):
        qb, kb, vb = H.qkv_host(450, 2, 2, 700, 128, "bf16")
        q, k, v = (H.to_device(x, "bf16") for x in (qb, kb, vb))
        (o1, l1), _ = run_pair(q, k, v, torch.ones((700, 700), dtype=torch.bool, device="cuda"), causal)
        o2 = torch.empty_like(q)
        l2 = torch.empty_like(l1)
        ops.attn_fwd(q, k, v, o2, l2, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_blocks_list_overflow_runs_the_scan():
    """A CTA whose share of the summary exceeds its list (B*H = 40 heads of 33 000 rows,
    non-causal: 2 * ceil(2600 units / SMs) * 9 words > 256) runs as attn_fwd_masked."""
    B, Hh, N, D = 1, 40, 33000, 64
    g = torch.Generator(device="cuda").manual_seed(460)
    q, k, v = (torch.randn((B, Hh, N, D), generator=g, device="cuda").to(torch.bfloat16) for _ in range(3))
    i = torch.arange(N, device="cuda")
    mask = (i[:, None] - i[None, :]).abs() < 3000
    (o, lse), (o2, l2) = run_pair(q, k, v, mask, False)
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    assert torch.isfinite(lse).all()
