"""FP64 CPU oracle for online-softmax attention, its split-K partitions and the
LSE-weighted combine.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports, links or runs this
package; only the tests, ``__graft_entry__.smoke()`` and the bench's CPU
baseline do.  It shares no code with the CUDA path: inputs come in as float64
arrays holding the exact values the GPU reads (16-bit bits widened exactly),
and everything here is plain numpy in float64.

Pages it restates (by title and section):
  * "Streaming attention and online state", section "Online statistics": the
    state (m, l) with empty state (-inf, 0), m' = max(m, rowmax x),
    alpha = exp(m - m'), p = exp(x - m'), l' = alpha*l + rowsum p, numerator
    o' = alpha*o + p V, normalise after the last tile, fully masked rows give
    output 0 and log-sum-exp -inf.  Section "Attention as a consumer": the
    worked kernel takes an optional Boolean M x N mask (here True = visible,
    combined with the causal and bounds rules).
  * "A3. Tiled attention with online normalization", sections "Keep three
    quantities for each query row" (the recurrence, softmax(QK^T/sqrt(D)) V) and
    "Masks that preserve the recurrence" (causal keeps key <= query).
  * "fa4_splitk_combine" (Mojo module doc): partition p stores its locally
    normalised O_p and lse_p = log2(l_p) + m_p (log2 domain); the combine takes
    m* = max_p lse_p, G = log2(sum_p 2^(lse_p - m*)) + m*,
    O = sum_p 2^(lse_p - G) O_p.

Readings where the pages leave a step open (each one also listed in the design
notes):
  * attention LSE is the natural-log log-sum-exp; split-K partition LSEs and the
    combine's G are base 2, as the combine page states;
  * split-K partition bounds: chunk C = ceil(ceil(Nkv/P)/BN)*BN keys, partition
    p holds keys [p*C, min((p+1)*C, Nkv)); an empty partition stores O_p = 0 and
    lse_p = -inf;
  * in the combine a partition whose lse_p is -inf contributes nothing; a row
    whose every lse_p is -inf gives O = +0 and G = -inf.
  * the optional mask may hide every key of a row (the workshop page leaves that
    policy to the caller); such a row takes the fully-masked convention of the
    online statistics: O = +0, LSE = -inf.

Every function below is pinned by tests under ``tests/test_oracle.py`` against
values the pages print (the worked trace, the two-zeros update), closed forms
(one key; uniform logits), brute force on tiny inputs and the combine identity.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

LOG2E = 1.0 / math.log(2.0)


# ---------------------------------------------------------------------------
# The online statistics, step by step ("Streaming attention and online state",
# Online statistics; "A3. Tiled attention ...", Keep three quantities).
# ---------------------------------------------------------------------------
@dataclass
class SoftmaxState:
    """Running maximum m and unnormalised sum l of one row; empty is (-inf, 0)."""
    maximum: float = -math.inf
    sum: float = 0.0


@dataclass
class Update:
    state: SoftmaxState
    weights: np.ndarray   # p = exp(x - m'), zero for masked (-inf) scores
    rescale: float        # alpha = exp(m - m'), the factor for the old numerator


def softmax_update(state: SoftmaxState, x) -> Update:
    """One tile of scores x (finite, or -inf where masked) folded into the state.

    m' = max(m, max x); alpha = exp(m - m'); p = exp(x - m'); l' = alpha l + sum p.
    Explicit selects give an empty update zero weights instead of evaluating
    -inf - -inf: when m' is -inf every weight is 0 and alpha is taken as 1
    (nothing to rescale); when only m is -inf, alpha = exp(-inf) = 0."""
    x = np.asarray(x, dtype=np.float64)
    m_new = max(state.maximum, float(np.max(x))) if x.size else state.maximum
    if m_new == -math.inf:
        return Update(SoftmaxState(-math.inf, state.sum), np.zeros_like(x), 1.0)
    alpha = math.exp(state.maximum - m_new) if state.maximum != -math.inf else 0.0
    p = np.where(x == -math.inf, 0.0, np.exp(np.where(x == -math.inf, 0.0, x) - m_new))
    return Update(SoftmaxState(m_new, alpha * state.sum + float(np.sum(p))), p, alpha)


def softmax_normalize(weights, state: SoftmaxState) -> np.ndarray:
    """Divide by the running sum; a zero sum (fully masked) normalises to zeros."""
    w = np.asarray(weights, dtype=np.float64)
    if state.sum == 0.0:
        return np.zeros_like(w)
    return w / state.sum


def numerator_update(a: np.ndarray, alpha: float, p: np.ndarray, v_tile: np.ndarray) -> np.ndarray:
    """o' = alpha * o + p V for one tile (p: [n], v_tile: [n, Dv])."""
    return alpha * a + p @ v_tile


def streaming_row(logit_tiles, v_tiles):
    """Run the recurrence for ONE query row over its tiles of already-scaled
    logits (each a 1-D array, -inf where masked) and matching V tiles
    ([n, Dv] arrays).  Returns (output, state, numerator); output is a/l, or
    zeros when every logit was masked."""
    st = SoftmaxState()
    dv = np.asarray(v_tiles[0], dtype=np.float64).reshape(len(logit_tiles[0]), -1).shape[1]
    a = np.zeros(dv)
    for x, vt in zip(logit_tiles, v_tiles):
        vt = np.asarray(vt, dtype=np.float64).reshape(len(x), -1)
        u = softmax_update(st, x)
        a = numerator_update(a, u.rescale, u.weights, vt)
        st = u.state
    out = softmax_normalize(a, st)
    return out, st, a


# ---------------------------------------------------------------------------
# Dense definition: softmax(scale * Q K^T) V with the masks of the pages.
# ---------------------------------------------------------------------------
def visible(nq: int, nk: int, causal: bool, q_rows=None, k_lo: int = 0, k_hi: int | None = None) -> np.ndarray:
    """Boolean [rows, nk] mask of the keys each query may see: keys in
    [k_lo, k_hi) and, when causal, key index <= query index (diagonal included)."""
    if k_hi is None:
        k_hi = nk
    rows = np.arange(nq) if q_rows is None else np.asarray(q_rows)
    j = np.arange(nk)
    vis = (j[None, :] >= k_lo) & (j[None, :] < k_hi)
    if causal:
        vis = vis & (j[None, :] <= rows[:, None])
    return np.broadcast_to(vis, (len(rows), nk))


def masked_softmax_attention(s: np.ndarray, vis: np.ndarray, v: np.ndarray):
    """Rows of scaled scores s [r, nk] with visibility vis, values v [nk, Dv].
    Returns (O [r, Dv], M [r], L [r]) with M the row max over visible keys and
    L = sum exp(s - M).  A row with no visible key gives O = +0, M = -inf, L = 0."""
    s = np.where(vis, s, -np.inf)
    M = np.max(s, axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    empty = ~np.isfinite(M)
    Msafe = np.where(empty, 0.0, M)
    e = np.where(vis, np.exp(np.where(vis, s, 0.0) - Msafe[:, None]), 0.0)
    L = e.sum(axis=1)
    O = e @ v
    O = np.where(empty[:, None], 0.0, O / np.where(empty, 1.0, L)[:, None])
    return O + 0.0, M, L


def attention(q, k, v, scale: float, causal: bool, mask=None):
    """Scaled dot-product attention for one head or a batch of heads.

    q [..., Nq, D], k [..., Nk, D], v [..., Nk, Dv], all float64 holding the
    exact input values.  Returns O [..., Nq, Dv] and natural-log
    LSE [..., Nq] (= M + ln L; -inf for a row with no visible key).
    Causal requires Nq == Nk ("Masks that preserve the recurrence": rectangular
    causal lengths are rejected).

    mask: optional Boolean [Nq, Nk] (shared by every head) or [..., Nq, Nk] (one per
    head), True = the key is visible ("Streaming attention and online state",
    Attention as a consumer: an optional Boolean M x N mask).  It is combined with the
    causal rule; a row left with no visible key gives O = +0 and LSE = -inf (Online
    statistics: entirely masked rows normalise to zero with log-sum-exp -inf)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq, nk = q.shape[-2], k.shape[-2]
    if causal and nq != nk:
        raise ValueError("causal attention needs equal query and key lengths")
    lead = q.shape[:-2]
    qf = q.reshape(-1, nq, q.shape[-1])
    kf = k.reshape(-1, nk, k.shape[-1])
    vf = v.reshape(-1, nk, v.shape[-1])
    O = np.empty((qf.shape[0], nq, vf.shape[-1]))
    LSE = np.empty((qf.shape[0], nq))
    vis = visible(nq, nk, causal)
    if mask is not None:
        mask = np.asarray(mask, dtype=bool)
        mask = np.broadcast_to(mask, lead + (nq, nk)).reshape(-1, nq, nk)
    for h in range(qf.shape[0]):
        s = scale * (qf[h] @ kf[h].T)
        vis_h = vis if mask is None else (vis & mask[h])
        o, M, L = masked_softmax_attention(s, vis_h, vf[h])
        O[h] = o
        LSE[h] = np.where(np.isfinite(M), M + np.log(np.where(L > 0, L, 1.0)), -np.inf)
    return O.reshape(*lead, nq, vf.shape[-1]), LSE.reshape(*lead, nq)


def attention_rows(q_rows, rows, k, v, scale: float, causal: bool, mask_rows=None):
    """Attention for selected query rows of one head: q_rows [r, D] are the
    queries at global indices `rows`; k [Nk, D], v [Nk, Dv]; mask_rows [r, Nk]
    Boolean or None (the selected rows of the optional mask).  Same definition
    as `attention`, so sampled outputs of a large problem can be checked."""
    q_rows = np.asarray(q_rows, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = scale * (q_rows @ k.T)
    vis = visible(len(rows), k.shape[0], causal, q_rows=rows)
    if mask_rows is not None:
        vis = vis & np.asarray(mask_rows, dtype=bool)
    O, M, L = masked_softmax_attention(s, vis, v)
    lse = np.where(np.isfinite(M), M + np.log(np.where(L > 0, L, 1.0)), -np.inf)
    return O, lse


# ---------------------------------------------------------------------------
# Split-K partitions and the LSE-weighted combine ("fa4_splitk_combine").
# ---------------------------------------------------------------------------
def splitk_bounds(nkv: int, P: int, block_n: int):
    """Key range [lo, hi) of each partition: chunk C = ceil(ceil(nkv/P)/block_n)*block_n,
    partition p = [p*C, min((p+1)*C, nkv)); trailing partitions may be empty."""
    per = -(-nkv // P)
    C = -(-per // block_n) * block_n
    return [(min(p * C, nkv), min((p + 1) * C, nkv)) for p in range(P)]


def splitk_partials_rows(q_rows, rows, k, v, scale: float, causal: bool, bounds, mask_rows=None):
    """Per-partition locally normalised outputs and base-2 LSEs for selected
    query rows of one head (mask_rows: [r, Nk] Boolean or None, as in
    `attention_rows`).  Returns O_p [P, r, Dv] and lse_p [P, r] where
    lse_p = log2(l_p) + m_p with m_p the row max in log2 units, i.e.
    (M_p + ln L_p) * log2(e); an empty (row, partition) gives O_p = 0, lse_p = -inf."""
    q_rows = np.asarray(q_rows, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = scale * (q_rows @ k.T)
    Op = np.zeros((len(bounds), len(rows), v.shape[1]))
    lsep = np.full((len(bounds), len(rows)), -np.inf)
    for p, (lo, hi) in enumerate(bounds):
        vis = visible(len(rows), k.shape[0], causal, q_rows=rows, k_lo=lo, k_hi=hi)
        if mask_rows is not None:
            vis = vis & np.asarray(mask_rows, dtype=bool)
        o, M, L = masked_softmax_attention(s, vis, v)
        Op[p] = o
        ok = np.isfinite(M)
        lsep[p] = np.where(ok, (M + np.log(np.where(L > 0, L, 1.0))) * LOG2E, -np.inf)
    return Op, lsep


def splitk_partials(q, k, v, scale: float, causal: bool, P: int, block_n: int, mask=None):
    """Split-K partials for every row of every head: q [..., Nq, D]; mask as in
    `attention` (Boolean, broadcast against [..., Nq, Nk]) or None.
    Returns O_p [P, ..., Nq, Dv] and lse_p [P, ..., Nq] (base 2)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq, nk = q.shape[-2], k.shape[-2]
    if causal and nq != nk:
        raise ValueError("causal attention needs equal query and key lengths")
    bounds = splitk_bounds(nk, P, block_n)
    lead = q.shape[:-2]
    qf = q.reshape(-1, nq, q.shape[-1])
    kf = k.reshape(-1, nk, k.shape[-1])
    vf = v.reshape(-1, nk, v.shape[-1])
    Op = np.zeros((P, qf.shape[0], nq, vf.shape[-1]))
    lsep = np.full((P, qf.shape[0], nq), -np.inf)
    if mask is not None:
        mask = np.broadcast_to(np.asarray(mask, dtype=bool), lead + (nq, nk)).reshape(-1, nq, nk)
    for h in range(qf.shape[0]):
        o, l = splitk_partials_rows(qf[h], np.arange(nq), kf[h], vf[h], scale, causal, bounds,
                                    None if mask is None else mask[h])
        Op[:, h] = o
        lsep[:, h] = l
    return Op.reshape(P, *lead, nq, vf.shape[-1]), lsep.reshape(P, *lead, nq)


def combine(o_partial, lse_partial):
    """LSE-weighted merge of P partitions.

    o_partial [P, RH, Dv] (locally normalised), lse_partial [P, RH] base 2.
    m* = max_p lse_p; G = log2(sum_p 2^(lse_p - m*)) + m*;
    O[d] = sum_p 2^(lse_p - G) O_p[d], skipping partitions with lse_p = -inf.
    A row-head whose every lse_p is -inf gives O = +0 and G = -inf.
    Returns (O [RH, Dv], G [RH])."""
    o = np.asarray(o_partial, dtype=np.float64)
    lse = np.asarray(lse_partial, dtype=np.float64)
    live = np.isfinite(lse)
    mstar = np.max(lse, axis=0)
    dead = ~np.isfinite(mstar)
    msafe = np.where(dead, 0.0, mstar)
    w = np.where(live, np.exp2(np.where(live, lse, 0.0) - msafe[None, :]), 0.0)
    G = np.where(dead, -np.inf, np.log2(np.where(dead, 1.0, w.sum(axis=0))) + msafe)
    Gsafe = np.where(dead, 0.0, G)
    scale = np.where(live, np.exp2(np.where(live, lse, 0.0) - Gsafe[None, :]), 0.0)
    O = np.einsum("pr,prd->rd", scale, np.where(live[:, :, None], o, 0.0))
    O = np.where(dead[:, None], 0.0, O) + 0.0
    return O, G
