"""Pins for the FP64 oracle: values the pages print, closed forms, invariants
and brute force, chosen so that a dropped term, a wrong sign or index or a
transposed operand in the oracle fails at least one of them.  CPU only."""
import json
import math
import os

import numpy as np
import pytest

import oracle
from tests.conftest import GOLDEN


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _num(x):
    return math.log(2.0) if x == "ln2" else float(x)


# --- values printed on the pages -------------------------------------------------
def test_worked_trace_recurrence():
    g = _golden("worked_trace.json")
    tiles = [np.array([_num(x) for x in t]) for t in g["logit_tiles"]]
    vt = [np.array(t).reshape(-1, 1) for t in g["v_tiles"]]
    # after the first tile
    out1, st1, a1 = oracle.streaming_row(tiles[:1], vt[:1])
    assert st1.maximum == g["after_tile_1"]["m"]
    assert st1.sum == g["after_tile_1"]["l"]
    assert a1[0] == g["after_tile_1"]["a"]
    # second tile: alpha = exp(0 - ln 2) = 1/2
    u = oracle.softmax_update(st1, tiles[1])
    assert u.rescale == pytest.approx(g["alpha_tile_2"], abs=1e-15)
    out, st, a = oracle.streaming_row(tiles, vt)
    assert st.sum == pytest.approx(g["after_tile_2"]["l"], abs=1e-15)
    assert a[0] == pytest.approx(g["after_tile_2"]["a"], abs=1e-14)
    assert out[0] == pytest.approx(g["output"], abs=1e-14)


def test_worked_trace_planted_bug_gives_seven(monkeypatch):
    """Rescaling l but not the numerator must give 7, so the pin above is able
    to tell the correct recurrence from that bug."""
    g = _golden("worked_trace.json")
    tiles = [np.array([_num(x) for x in t]) for t in g["logit_tiles"]]
    vt = [np.array(t).reshape(-1, 1) for t in g["v_tiles"]]
    monkeypatch.setattr(oracle, "numerator_update", lambda a, alpha, p, v: a + p @ v)
    out, _, _ = oracle.streaming_row(tiles, vt)
    assert out[0] == pytest.approx(g["output_if_only_l_is_rescaled"], abs=1e-14)


def test_worked_trace_dense_definition():
    g = _golden("worked_trace.json")
    logits = [_num(x) for t in g["logit_tiles"] for x in t]
    vals = [x for t in g["v_tiles"] for x in t]
    # D = 1: q = [1], k_j = logit_j, scale 1 gives exactly the printed logits
    q = np.array([[1.0]])
    k = np.array(logits).reshape(-1, 1)
    v = np.array(vals).reshape(-1, 1)
    O, lse = oracle.attention(q, k, v, scale=1.0, causal=False)
    assert O[0, 0] == pytest.approx(g["output"], abs=1e-14)
    w = np.exp(np.array(logits) - lse[0])
    np.testing.assert_allclose(w, g["full_softmax_weights"], atol=1e-15)
    assert lse[0] == pytest.approx(math.log(4.0), abs=1e-15)


def test_softmax_update_two_zeros():
    g = _golden("softmax_update_two_zeros.json")
    u = oracle.softmax_update(oracle.SoftmaxState(), g["scores"])
    assert (u.state.maximum, u.state.sum, u.rescale) == (
        g["state_maximum"], g["state_sum"], g["rescale"])
    np.testing.assert_array_equal(oracle.softmax_normalize(u.weights, u.state),
                                  g["normalized_weights"])


def test_fully_masked_row_convention():
    g = _golden("fully_masked_row.json")
    # recurrence: every score masked
    out, st, _ = oracle.streaming_row([np.array([-np.inf, -np.inf])], [np.array([[1.0], [2.0]])])
    assert st.maximum == -math.inf and st.sum == 0.0
    assert out[0] == 0.0 and not math.copysign(1.0, out[0]) < 0
    # dense helper with no visible key
    O, M, L = oracle.masked_softmax_attention(np.zeros((1, 3)), np.zeros((1, 3), bool),
                                              np.ones((3, 2)))
    assert np.all(O == 0.0) and not np.any(np.signbit(O))
    assert M[0] == -math.inf and L[0] == 0.0
    assert np.float32(O[0, 0]).view(np.uint32) == int(g["output_bits_f32_hex"], 16)
    assert np.float32(-np.inf).view(np.uint32) == int(g["lse_bits_f32_hex"], 16)


# --- brute force on tiny inputs (pure-Python loops) ----------------------------
def _brute_attention(q, k, v, scale, causal):
    nq, nk, dv = len(q), len(k), len(v[0])
    O, LSE = [], []
    for i in range(nq):
        s = []
        for j in range(nk):
            if causal and j > i:
                continue
            s.append((j, scale * sum(q[i][d] * k[j][d] for d in range(len(q[i])))))
        m = max(x for _, x in s)
        e = [(j, math.exp(x - m)) for j, x in s]
        L = math.fsum(w for _, w in e)
        O.append([math.fsum(w * v[j][d] for j, w in e) / L for d in range(dv)])
        LSE.append(m + math.log(L))
    return np.array(O), np.array(LSE)


@pytest.mark.parametrize("nq,nk,d,dv,causal", [
    (1, 1, 3, 2, False), (4, 7, 5, 3, False), (6, 6, 4, 4, True), (9, 9, 2, 5, True),
    (3, 11, 8, 1, False),
])
def test_attention_brute_force(nq, nk, d, dv, causal):
    rng = np.random.default_rng(nq * 100 + nk * 10 + d)
    q = rng.normal(size=(nq, d)) * 2
    k = rng.normal(size=(nk, d))
    v = rng.normal(size=(nk, dv))
    scale = 1.0 / math.sqrt(d)
    O, lse = oracle.attention(q, k, v, scale, causal)
    Ob, lb = _brute_attention(q.tolist(), k.tolist(), v.tolist(), scale, causal)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lb, rtol=0, atol=1e-12)


def test_attention_not_transposed():
    """A non-square V and distinct per-key values catch a transposed operand."""
    q = np.array([[1.0, 0.0]])
    k = np.array([[3.0, 0.0], [0.0, 3.0], [0.0, 0.0]])
    v = np.array([[1.0, 0.0, 0.0, 0.0], [0.0, 1.0, 0.0, 0.0], [0.0, 0.0, 1.0, 0.0]])
    O, lse = oracle.attention(q, k, v, scale=1.0, causal=False)
    e = np.array([math.exp(3.0), 1.0, 1.0])
    np.testing.assert_allclose(O[0], np.r_[e / e.sum(), 0.0], atol=1e-15)
    assert lse[0] == pytest.approx(math.log(e.sum()), abs=1e-14)


def test_streaming_matches_dense_for_every_tiling():
    rng = np.random.default_rng(7)
    nk, d, dv = 13, 4, 3
    q = rng.normal(size=(1, d))
    k = rng.normal(size=(nk, d))
    v = rng.normal(size=(nk, dv))
    O, lse = oracle.attention(q, k, v, 0.5, False)
    s = 0.5 * (q @ k.T)[0]
    for bn in range(1, nk + 1):
        tiles = [s[i:i + bn] for i in range(0, nk, bn)]
        vts = [v[i:i + bn] for i in range(0, nk, bn)]
        out, st, _ = oracle.streaming_row(tiles, vts)
        np.testing.assert_allclose(out, O[0], atol=1e-13)
        assert st.maximum + math.log(st.sum) == pytest.approx(lse[0], abs=1e-13)


# --- closed forms -------------------------------------------------------------
def test_single_key_closed_form():
    q = np.array([[0.3, -1.2]])
    k = np.array([[2.0, 0.5]])
    v = np.array([[4.0, -5.0, 6.0]])
    for causal in (False, True):
        O, lse = oracle.attention(q, k, v, 0.7, causal)
        np.testing.assert_array_equal(O[0], v[0])
        assert lse[0] == pytest.approx(0.7 * (0.3 * 2.0 - 1.2 * 0.5), abs=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_logits_closed_form(causal):
    rng = np.random.default_rng(3)
    n, d = 9, 4
    q = np.zeros((n, d))
    k = rng.normal(size=(n, d))
    v = rng.normal(size=(n, 2))
    O, lse = oracle.attention(q, k, v, 0.5, causal)
    for i in range(n):
        cnt = i + 1 if causal else n
        np.testing.assert_allclose(O[i], v[:cnt].mean(axis=0), atol=1e-14)
        assert lse[i] == pytest.approx(math.log(cnt), abs=1e-14)


def test_large_logits_finite_and_brute():
    rng = np.random.default_rng(11)
    q = 8.0 * rng.normal(size=(5, 16))
    k = rng.normal(size=(5, 16))
    v = rng.normal(size=(5, 3))
    O, lse = oracle.attention(q, k, v, 0.25, True)
    assert np.all(np.isfinite(O)) and np.all(np.isfinite(lse))
    Ob, lb = _brute_attention(q.tolist(), k.tolist(), v.tolist(), 0.25, True)
    np.testing.assert_allclose(O, Ob, atol=1e-12)
    np.testing.assert_allclose(lse, lb, atol=1e-12)


def test_causal_future_perturbation_leaves_earlier_rows():
    rng = np.random.default_rng(5)
    n, d = 12, 4
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    O, lse = oracle.attention(q, k, v, 0.5, True)
    for j in (1, 5, 11):
        v2 = v.copy()
        v2[j:] = rng.normal(size=(n - j, d))
        k2 = k.copy()
        k2[j:] = rng.normal(size=(n - j, d))
        O2, lse2 = oracle.attention(q, k2, v2, 0.5, True)
        np.testing.assert_array_equal(O2[:j], O[:j])
        np.testing.assert_array_equal(lse2[:j], lse[:j])
        assert not np.array_equal(O2[j:], O[j:])


def test_causal_rectangular_rejected():
    with pytest.raises(ValueError):
        oracle.attention(np.zeros((2, 2)), np.zeros((3, 2)), np.zeros((3, 2)), 1.0, True)


# --- split-K and the combine --------------------------------------------------
def test_splitk_bounds_reading():
    # chunk = ceil(ceil(Nkv/P)/BN)*BN; trailing partitions may be short or empty
    b = oracle.splitk_bounds(32768, 37, 128)
    assert b[0] == (0, 896) and b[35] == (35 * 896, 36 * 896) and b[36] == (36 * 896, 32768)
    assert oracle.splitk_bounds(32768, 4, 128)[1] == (8192, 16384)
    assert oracle.splitk_bounds(10, 8, 4) == [(0, 4), (4, 8), (8, 10)] + [(10, 10)] * 5


def _brute_combine(o, lse):
    P, RH, dv = o.shape
    O = np.zeros((RH, dv))
    G = np.zeros(RH)
    for r in range(RH):
        live = [p for p in range(P) if lse[p, r] != -math.inf]
        if not live:
            G[r] = -math.inf
            continue
        m = max(lse[p, r] for p in live)
        G[r] = math.log2(math.fsum(2.0 ** (lse[p, r] - m) for p in live)) + m
        for d in range(dv):
            O[r, d] = math.fsum(2.0 ** (lse[p, r] - G[r]) * o[p, r, d] for p in live)
    return O, G


def test_combine_brute_force():
    rng = np.random.default_rng(13)
    P, RH, dv = 5, 7, 3
    o = rng.normal(size=(P, RH, dv))
    lse = rng.normal(10, 2, size=(P, RH))
    lse[rng.random((P, RH)) < 0.3] = -np.inf
    lse[:, 2] = -np.inf
    O, G = oracle.combine(o, lse)
    Ob, Gb = _brute_combine(o, lse)
    np.testing.assert_allclose(O, Ob, atol=1e-13)
    np.testing.assert_array_equal(np.isinf(G), np.isinf(Gb))
    np.testing.assert_allclose(G[np.isfinite(G)], Gb[np.isfinite(Gb)], atol=1e-13)
    assert np.all(O[2] == 0.0) and not np.any(np.signbit(O[2])) and G[2] == -np.inf


def test_combine_single_partition_is_identity():
    rng = np.random.default_rng(17)
    o = rng.normal(size=(1, 6, 4))
    lse = rng.normal(size=(1, 6))
    O, G = oracle.combine(o, lse)
    np.testing.assert_allclose(O, o[0], atol=1e-15)
    np.testing.assert_allclose(G, lse[0], atol=1e-15)


def test_combine_shift_invariance():
    rng = np.random.default_rng(19)
    o = rng.normal(size=(4, 5, 3))
    lse = rng.normal(size=(4, 5))
    O, G = oracle.combine(o, lse)
    O2, G2 = oracle.combine(o, lse + 37.5)
    np.testing.assert_allclose(O2, O, atol=1e-14)
    np.testing.assert_allclose(G2, G + 37.5, atol=1e-12)


def test_combine_skips_dead_partitions():
    o = np.array([[[1.0, 2.0]], [[np.nan, np.inf]]])
    lse = np.array([[3.0], [-np.inf]])
    O, G = oracle.combine(o, lse)
    np.testing.assert_array_equal(O, [[1.0, 2.0]])
    assert G[0] == 3.0


@pytest.mark.parametrize("P,bn,causal", [(1, 4, False), (2, 4, False), (3, 2, True),
                                         (8, 4, True), (5, 1, False), (4, 16, True)])
def test_combine_of_partials_equals_unsplit(P, bn, causal):
    """The closed-form identity of the combine: merging the partitions' locally
    normalised outputs by their LSEs reproduces unsplit attention."""
    rng = np.random.default_rng(P * 10 + bn)
    n, d = 10, 4
    q, k, v = (rng.normal(size=(2, n, d)) for _ in range(3))
    O, lse = oracle.attention(q, k, v, 0.5, causal)
    Op, lsep = oracle.splitk_partials(q, k, v, 0.5, causal, P, bn)
    Oc, G = oracle.combine(Op.reshape(P, -1, d), lsep.reshape(P, -1))
    np.testing.assert_allclose(Oc.reshape(O.shape), O, atol=1e-13)
    np.testing.assert_allclose(G.reshape(lse.shape) * math.log(2.0), lse, atol=1e-12)


def test_partition_with_no_visible_key():
    g = _golden("fully_masked_row.json")
    rng = np.random.default_rng(23)
    n, d = 8, 2
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    # causal, partitions of 4 keys: rows 0..3 see nothing in partition 1
    Op, lsep = oracle.splitk_partials(q, k, v, 1.0, True, 2, 4)
    assert np.all(lsep[1, :4] == -np.inf)
    assert np.all(Op[1, :4] == float(g["output"])) and not np.any(np.signbit(Op[1, :4]))
    assert np.all(np.isfinite(lsep[1, 4:]))


@pytest.mark.parametrize("causal", [False, True])
def test_attention_rows_brute_force(causal):
    """Sampled rows (used for the full-size checks) against pure-Python loops."""
    rng = np.random.default_rng(29)
    n, d = 11, 3
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    rows = np.array([0, 4, 10])
    O, lse = oracle.attention_rows(q[rows], rows, k, v, 0.7, causal)
    Ob, lb = _brute_attention(q.tolist(), k.tolist(), v.tolist(), 0.7, causal)
    np.testing.assert_allclose(O, Ob[rows], atol=1e-12)
    np.testing.assert_allclose(lse, lb[rows], atol=1e-12)


def test_splitk_partials_rows_brute_force():
    """Per-partition outputs and base-2 LSEs against pure-Python loops over each range."""
    rng = np.random.default_rng(31)
    n, d = 9, 2
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    rows = np.array([1, 5, 8])
    bounds = [(0, 4), (4, 8), (8, 9), (9, 9)]
    Op, lp = oracle.splitk_partials_rows(q[rows], rows, k, v, 1.0, True, bounds)
    for p, (lo, hi) in enumerate(bounds):
        for ri, i in enumerate(rows):
            s = [(j, float(q[i] @ k[j])) for j in range(lo, hi) if j <= i]
            if not s:
                assert lp[p, ri] == -math.inf and np.all(Op[p, ri] == 0.0)
                continue
            m = max(x for _, x in s)
            w = [(j, math.exp(x - m)) for j, x in s]
            L = math.fsum(x for _, x in w)
            assert lp[p, ri] == pytest.approx((m + math.log(L)) / math.log(2.0), abs=1e-12)
            for dd in range(d):
                assert Op[p, ri, dd] == pytest.approx(math.fsum(x * v[j][dd] for j, x in w) / L, abs=1e-12)


# --- the optional Boolean mask ---------------------------------------------------
def _brute_masked(q, k, v, scale, causal, mask):
    nq, nk, dv = len(q), len(k), len(v[0])
    O, LSE = [], []
    for i in range(nq):
        s = [(j, scale * sum(q[i][d] * k[j][d] for d in range(len(q[i]))))
             for j in range(nk) if mask[i][j] and (not causal or j <= i)]
        if not s:
            O.append([0.0] * dv)
            LSE.append(-math.inf)
            continue
        m = max(x for _, x in s)
        e = [(j, math.exp(x - m)) for j, x in s]
        L = math.fsum(w for _, w in e)
        O.append([math.fsum(w * v[j][d] for j, w in e) / L for d in range(dv)])
        LSE.append(m + math.log(L))
    return np.array(O), np.array(LSE)


@pytest.mark.parametrize("causal", [False, True])
def test_masked_attention_brute_force(causal):
    rng = np.random.default_rng(41)
    n, d = 10, 3
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    mask = rng.random((n, n)) < 0.4
    mask[2, :] = False                      # a fully masked row
    O, lse = oracle.attention(q, k, v, 0.6, causal, mask=mask)
    Ob, lb = _brute_masked(q.tolist(), k.tolist(), v.tolist(), 0.6, causal, mask.tolist())
    np.testing.assert_allclose(O, Ob, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(lb))
    np.testing.assert_allclose(lse[np.isfinite(lb)], lb[np.isfinite(lb)], atol=1e-12)
    assert np.all(O[2] == 0.0) and not np.any(np.signbit(O[2])) and lse[2] == -np.inf


def test_mask_special_cases_reduce_to_known_rules():
    rng = np.random.default_rng(43)
    n, d = 9, 4
    q, k, v = (rng.normal(size=(2, n, d)) for _ in range(3))
    O, lse = oracle.attention(q, k, v, 0.5, False)
    O1, l1 = oracle.attention(q, k, v, 0.5, False, mask=np.ones((n, n), bool))
    np.testing.assert_array_equal(O1, O)
    np.testing.assert_array_equal(l1, lse)
    Oc, lc = oracle.attention(q, k, v, 0.5, True)
    O2, l2 = oracle.attention(q, k, v, 0.5, False, mask=np.tril(np.ones((n, n), bool)))
    np.testing.assert_allclose(O2, Oc, atol=1e-14)
    np.testing.assert_allclose(l2, lc, atol=1e-14)
    # one mask per head
    per_head = np.stack([np.tril(np.ones((n, n), bool)), np.ones((n, n), bool)])
    O3, l3 = oracle.attention(q, k, v, 0.5, False, mask=per_head)
    np.testing.assert_allclose(O3[0], Oc[0], atol=1e-14)
    np.testing.assert_allclose(O3[1], O[1], atol=1e-14)


def test_masked_splitk_partials_merge_to_masked_attention():
    """Cutting the key axis commutes with an arbitrary mask: the partitions of a masked
    problem, merged by the combine, give the masked attention (with rows that a whole
    partition, or the whole mask, hides)."""
    rng = np.random.default_rng(47)
    n, d, P = 12, 4, 3
    q, k, v = (rng.normal(size=(2, n, d)) for _ in range(3))
    mask = rng.random((2, n, n)) < 0.5
    mask[0, 5, :] = False
    mask[1, 7, :4] = False
    Op, lsep = oracle.splitk_partials(q, k, v, 0.7, False, P, 4, mask=mask)
    O, G = oracle.combine(Op.reshape(P, -1, d), lsep.reshape(P, -1))
    Oa, la = oracle.attention(q, k, v, 0.7, False, mask=mask)
    np.testing.assert_allclose(O.reshape(2, n, d), Oa, atol=1e-12)
    la2 = la.reshape(-1) * oracle.LOG2E
    np.testing.assert_array_equal(np.isneginf(G), np.isneginf(la2))
    np.testing.assert_allclose(G[np.isfinite(G)], la2[np.isfinite(la2)], atol=1e-12)
    assert np.isneginf(lsep[:, 0, 5]).all() and np.isneginf(lsep[0, 1, 7])


def test_masked_attention_rows_match_full():
    rng = np.random.default_rng(53)
    n, d = 11, 3
    q, k, v = (rng.normal(size=(n, d)) for _ in range(3))
    mask = rng.random((n, n)) < 0.3
    O, lse = oracle.attention(q, k, v, 0.9, True, mask=mask)
    rows = np.array([0, 4, 10])
    Or, lr = oracle.attention_rows(q[rows], rows, k, v, 0.9, True, mask_rows=mask[rows])
    np.testing.assert_array_equal(Or, O[rows])
    np.testing.assert_array_equal(lr, lse[rows])
