"""Seeded, counter-based synthetic inputs shared by the tests, the bench and the
oracle's callers.

This module holds no attention arithmetic.  It only defines how the input
tensors of every workload are drawn, so that the CPU side (numpy, here) and the
GPU side (``synth/gen.cu``, the same definition written in CUDA) can produce
bit-identical values for any slice of any tensor without materialising the rest.

Definition
----------
* Word generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014; the finaliser constants are the
  ones Vigna published with ``splitmix64.c``).  Element ``i`` of stream
  ``stream`` under ``seed`` is ``mix64(GAMMA * (i + 1 + stream * 2**40 + seed * 2**48))``
  (all arithmetic mod 2**64).  With ``seed = stream = 0`` this is exactly the
  SplitMix64 sequence started from state 0, whose first output is the published
  test vector 0xE220A8397B1DCDAF.  Distinct (seed, stream) pairs are disjoint
  blocks of that sequence while ``i < 2**40``, ``stream < 256``, ``seed < 2**16``.
* Standard normal (approximate): Irwin-Hall sum of the word's four 16-bit
  fields, centred and scaled to unit variance in float32:
  ``z = float32(a + b + c + d - 131070) * C`` with ``C`` = float32 of
  ``1/sqrt((65536**2 - 1) / 3)`` (bits 0x37DDB3D7).  Mean 0, variance 1,
  support bounded at about +-3.46.  ``mu + sigma * z`` is formed as one float32
  multiply then one float32 add (no fused multiply-add) on both sides.
* Bernoulli(prob): the word's upper 32 bits compared with ``floor(prob * 2**32)``.
* Boolean attention masks (True = the key is visible), four recipes: independent
  Bernoulli entries; a sliding-window band |i - j| < w; block-sparse (one
  Bernoulli draw per b x b block); key padding (per batch entry a visible
  prefix of random length).  ``hide_rows`` hides every key of a Bernoulli subset
  of rows, to exercise the fully masked case.
* 16-bit storage: float32 rounded to bfloat16 or float16 with round-to-nearest-even.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
NORM_SCALE = np.array([0x37DDB3D7], dtype=np.uint32).view(np.float32)[0]

# Stream identifiers: one per tensor role, so every tensor is an independent block.
STREAM_Q, STREAM_K, STREAM_V = 1, 2, 3
STREAM_LSE, STREAM_LSE_DROP, STREAM_ROW_DROP = 4, 5, 6
STREAM_OPART = 7
STREAM_MASK, STREAM_MASK_ROWS = 8, 9

DTYPES = ("f16", "bf16", "f32")


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def words_at(seed: int, stream: int, idx) -> np.ndarray:
    """Raw 64-bit words for arbitrary element indices of (seed, stream)."""
    if not (0 <= stream < 256 and 0 <= seed < 2**16):
        raise ValueError("stream must be < 256 and seed < 2**16")
    idx = np.asarray(idx, dtype=np.int64)
    if idx.size and (idx.min() < 0 or idx.max() >= 2**40):
        raise ValueError("element index out of the stream's 2**40 block")
    base = np.uint64((1 + stream * 2**40 + seed * 2**48) % 2**64)
    with np.errstate(over="ignore"):
        ctr = (idx.astype(np.uint64) + base) * GAMMA
    return mix64(ctr)


def words(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Raw 64-bit words for elements [start, start+count) of (seed, stream)."""
    return words_at(seed, stream, np.arange(start, start + count, dtype=np.int64))


def normal_at(seed: int, stream: int, idx, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    """float32 approximately-normal values at arbitrary element indices."""
    return _irwin_hall(words_at(seed, stream, idx), mu, sigma)


def normal(seed: int, stream: int, start: int, count: int,
           mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    """float32 approximately-normal values (Irwin-Hall of four 16-bit fields)."""
    return _irwin_hall(words(seed, stream, start, count), mu, sigma)


def _irwin_hall(w: np.ndarray, mu: float, sigma: float) -> np.ndarray:
    m16 = np.uint64(0xFFFF)
    s = ((w & m16) + ((w >> np.uint64(16)) & m16)
         + ((w >> np.uint64(32)) & m16) + (w >> np.uint64(48)))
    z = (s.astype(np.int64) - 131070).astype(np.float32) * NORM_SCALE
    if sigma != 1.0:
        z = z * np.float32(sigma)
    if mu != 0.0:
        z = z + np.float32(mu)
    return z.astype(np.float32)


def bernoulli(seed: int, stream: int, start: int, count: int, prob: float) -> np.ndarray:
    """Boolean draws with P(True) = floor(prob * 2**32) / 2**32."""
    thresh = np.uint64(int(np.floor(prob * 2**32)))
    return (words(seed, stream, start, count) >> np.uint64(32)) < thresh


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits.
    Inputs here are finite, so no NaN handling is needed."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rnd = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + rnd) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << np.uint32(16)).view(np.float32)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Storage bits for dtype: uint16 for f16/bf16, float32 for f32."""
    x = np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "f32":
        return x
    raise ValueError(dtype)


def to_f64(stored: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of stored bits (widening is exact)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(stored).astype(np.float64)
    if dtype == "f16":
        return np.asarray(stored, dtype=np.uint16).view(np.float16).astype(np.float64)
    return np.asarray(stored, dtype=np.float32).astype(np.float64)


def tensor(seed: int, stream: int, shape, dtype: str, start: int = 0,
           mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    """Storage bits of a whole (small) tensor, row-major, element index = flat index."""
    n = int(np.prod(shape)) if len(shape) else 1
    return round_to(normal(seed, stream, start, n, mu, sigma), dtype).reshape(shape)


def lse_partials(seed: int, P: int, RH: int, start_rh: int = 0, count_rh: int | None = None,
                 mu: float = 10.0, sigma: float = 2.0, drop: float = 0.05,
                 row_drop: float = 0.001) -> np.ndarray:
    """float32 [P, count_rh] log2-domain partition LSEs for the standalone combine
    workload: N(mu, sigma) values, each (row-head, partition) entry -inf with
    probability `drop`, and every partition of a row-head -inf with probability
    `row_drop`.  Element (p, rh) uses counter p*RH + rh; the row draw uses rh."""
    if count_rh is None:
        count_rh = RH - start_rh
    out = np.empty((P, count_rh), dtype=np.float32)
    dead = bernoulli(seed, STREAM_ROW_DROP, start_rh, count_rh, row_drop)
    for p in range(P):
        s = p * RH + start_rh
        v = normal(seed, STREAM_LSE, s, count_rh, mu, sigma)
        d = bernoulli(seed, STREAM_LSE_DROP, s, count_rh, drop)
        v[d | dead] = -np.inf
        out[p] = v
    return out


def bernoulli_at(seed: int, stream: int, idx, prob: float) -> np.ndarray:
    thresh = np.uint64(int(np.floor(prob * 2**32)))
    return (words_at(seed, stream, idx) >> np.uint64(32)) < thresh


def lse_partials_at(seed: int, P: int, RH: int, rh_idx, mu: float = 10.0, sigma: float = 2.0,
                    drop: float = 0.05, row_drop: float = 0.001) -> np.ndarray:
    """lse_partials restricted to the row-heads `rh_idx`: float32 [P, len(rh_idx)]."""
    rh_idx = np.asarray(rh_idx, dtype=np.int64)
    dead = bernoulli_at(seed, STREAM_ROW_DROP, rh_idx, row_drop)
    out = np.empty((P, len(rh_idx)), dtype=np.float32)
    for p in range(P):
        j = p * RH + rh_idx
        v = normal_at(seed, STREAM_LSE, j, mu, sigma)
        v[bernoulli_at(seed, STREAM_LSE_DROP, j, drop) | dead] = -np.inf
        out[p] = v
    return out


# ---------------------------------------------------------------------------
# Boolean masks (True = visible); host-side only, uploaded as bool tensors.
# ---------------------------------------------------------------------------
def mask_random(seed: int, shape, prob: float) -> np.ndarray:
    """Independent Bernoulli(prob) entries; element index = flat index."""
    n = int(np.prod(shape))
    return bernoulli(seed, STREAM_MASK, 0, n, prob).reshape(shape)


def mask_band(nq: int, nk: int, window: int) -> np.ndarray:
    """Sliding window: query i sees keys j with |i - j| < window."""
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    return np.abs(i - j) < window


def mask_blocks(seed: int, nq: int, nk: int, block: int, prob: float) -> np.ndarray:
    """Block-sparse: each block x block tile is visible with probability prob."""
    bq, bk = -(-nq // block), -(-nk // block)
    tiles = bernoulli(seed, STREAM_MASK, 0, bq * bk, prob).reshape(bq, bk)
    return np.repeat(np.repeat(tiles, block, axis=0), block, axis=1)[:nq, :nk]


def key_padding(seed: int, batch: int, nk: int, min_len: int = 1) -> np.ndarray:
    """[batch, 1, 1, nk]: batch entry b sees keys j < len_b, len_b uniform-ish in
    [min_len, nk] (from the word's upper 32 bits)."""
    w = words(seed, STREAM_MASK, 0, batch) >> np.uint64(32)
    span = nk - min_len + 1
    lens = min_len + (w % np.uint64(span)).astype(np.int64)
    return (np.arange(nk)[None, :] < lens[:, None]).reshape(batch, 1, 1, nk)


def hide_rows(seed: int, mask: np.ndarray, prob: float) -> np.ndarray:
    """Copy of mask [..., nq, nk] with a Bernoulli(prob) subset of its rows fully hidden."""
    out = np.array(mask, dtype=bool, copy=True)
    rows = out.reshape(-1, out.shape[-1])
    rows[bernoulli(seed, STREAM_MASK_ROWS, 0, rows.shape[0], prob)] = False
    return out
