"""Pins for the fp64 oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or the mathematics
fix -- hand-derived closed forms (tests/golden), invariants and special cases
of masked softmax attention -- chosen so that a dropped term, a wrong sign or
index, a transposed operand, a wrong log base or an off-by-one in a mask fails
at least one of them (see test_pins_catch_planted_mistakes).
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "two_key_closed_form.json")
MODES = ["rows", "literal"]


def run(mode, q, k, v, scale, causal, key_lens=None, window=0):
    if mode == "rows":
        return oracle.attention_rows(q, k, v, scale, causal, key_lens, threads=2, window=window)
    O, lse, _ = oracle.attention_literal(q, k, v, scale, causal, key_lens, window=window)
    return O, lse


def rnd(seed, B, H, N, d, scale=1.0):
    r = np.random.default_rng(seed)
    return [scale * r.standard_normal((B, H, N, d)) for _ in range(3)]


# --- hand-derived closed forms -------------------------------------------------

@pytest.mark.parametrize("mode", MODES)
def test_golden_closed_forms(mode):
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        q = np.array(c["q"])[None, None]
        k = np.array(c["k"])[None, None]
        v = np.array(c["v"])[None, None]
        kl = None if c["key_len"] is None else np.array([c["key_len"]], dtype=np.int32)
        O, lse = run(mode, q, k, v, c["scale"], c["causal"], kl)
        np.testing.assert_allclose(O[0, 0], np.array(c["O"]), rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(lse[0, 0], np.array(c["lse"]), rtol=0, atol=1e-12, err_msg=c["name"])


@pytest.mark.parametrize("mode", MODES)
def test_textbook_two_term_softmax(mode):
    # d = 1, N = 2: softmax of two logits is the logistic function of their
    # difference, O = v0 + (v1 - v0) * sigma(s1 - s0).
    r = np.random.default_rng(5)
    for _ in range(20):
        q, k, v = r.standard_normal((3, 1, 1, 2, 1))
        scale = r.uniform(0.1, 2.0)
        O, lse = run(mode, q, k, v, scale, False)
        for i in range(2):
            s0, s1 = scale * q[0, 0, i, 0] * k[0, 0, 0, 0], scale * q[0, 0, i, 0] * k[0, 0, 1, 0]
            sig = 1.0 / (1.0 + math.exp(-(s1 - s0)))
            want = v[0, 0, 0, 0] + (v[0, 0, 1, 0] - v[0, 0, 0, 0]) * sig
            assert abs(O[0, 0, i, 0] - want) < 1e-12
            assert abs(lse[0, 0, i] - (max(s0, s1) + math.log1p(math.exp(-abs(s1 - s0))))) < 1e-12


# --- invariants and special cases ---------------------------------------------

def test_literal_rows_sum_to_one():
    q, k, v = rnd(1, 2, 2, 19, 4)
    for causal in (False, True):
        for kl in (None, np.array([3, 19], dtype=np.int32)):
            _, _, P = oracle.attention_literal(q, k, v, 0.5, causal, kl)
            np.testing.assert_allclose(P.sum(-1), 1.0, atol=1e-12)
            assert (P >= 0).all()


@pytest.mark.parametrize("mode", MODES)
def test_constant_v_gives_that_row(mode):
    q, k, _ = rnd(2, 2, 3, 23, 6, scale=2.0)
    c = np.random.default_rng(3).standard_normal(6)
    v = np.broadcast_to(c, q.shape).copy()
    for causal in (False, True):
        O, _ = run(mode, q, k, v, 0.7, causal, np.array([1, 23], dtype=np.int32))
        np.testing.assert_allclose(O, np.broadcast_to(c, O.shape), atol=1e-12)


@pytest.mark.parametrize("mode", MODES)
def test_zero_q_gives_mean_of_visible_v(mode):
    _, k, v = rnd(4, 2, 2, 21, 5)
    q = np.zeros_like(k)
    kl = np.array([7, 21], dtype=np.int32)
    O, lse = run(mode, q, k, v, 0.9, False, kl)
    for b in range(2):
        n = kl[b]
        np.testing.assert_allclose(O[b], np.broadcast_to(v[b, :, :n].mean(axis=1, keepdims=True), O[b].shape),
                                   atol=1e-12)
        np.testing.assert_allclose(lse[b], math.log(n), atol=1e-12)
    # causal: row i sees keys 0..i
    O, lse = run(mode, q, k, v, 0.9, True, None)
    for i in range(21):
        np.testing.assert_allclose(O[:, :, i], v[:, :, : i + 1].mean(axis=2), atol=1e-12)
        np.testing.assert_allclose(lse[:, :, i], math.log(i + 1), atol=1e-12)


@pytest.mark.parametrize("mode", MODES)
def test_causal_row0_is_v0(mode):
    q, k, v = rnd(6, 2, 3, 17, 8)
    O, lse = run(mode, q, k, v, 0.25, True)
    np.testing.assert_allclose(O[:, :, 0], v[:, :, 0], atol=1e-12)
    s00 = 0.25 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], s00, atol=1e-12)


@pytest.mark.parametrize("mode", MODES)
def test_single_visible_key(mode):
    q, k, v = rnd(7, 3, 2, 13, 4, scale=3.0)
    kl = np.ones(3, dtype=np.int32)
    for causal in (False, True):
        O, lse = run(mode, q, k, v, 1.0, causal, kl)
        np.testing.assert_allclose(O, np.broadcast_to(v[:, :, :1], O.shape), atol=1e-12)
        s = np.einsum("bhid,bhd->bhi", q, k[:, :, 0])
        np.testing.assert_allclose(lse, s, atol=1e-12)


@pytest.mark.parametrize("mode", MODES)
def test_no_visible_key_gives_zero_and_minus_inf(mode):
    q, k, v = rnd(8, 2, 1, 9, 4)
    O, lse = run(mode, q, k, v, 1.0, False, np.array([0, 9], dtype=np.int32))
    assert np.all(O[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(O[1])) and np.all(np.isfinite(lse[1]))


@pytest.mark.parametrize("mode", MODES)
def test_key_permutation_invariance(mode):
    q, k, v = rnd(9, 1, 2, 31, 8)
    perm = np.random.default_rng(10).permutation(31)
    O1, l1 = run(mode, q, k, v, 0.4, False)
    O2, l2 = run(mode, q, k[:, :, perm], v[:, :, perm], 0.4, False)
    np.testing.assert_allclose(O1, O2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


@pytest.mark.parametrize("mode", MODES)
def test_shift_invariance(mode):
    # K -> K + 1 u^T shifts row i's logits by scale*(q_i . u): O is unchanged and
    # lse moves by exactly that amount.
    q, k, v = rnd(11, 2, 2, 25, 6)
    u = np.random.default_rng(12).standard_normal(6) * 3.0
    for causal in (False, True):
        O1, l1 = run(mode, q, k, v, 0.6, causal)
        O2, l2 = run(mode, q, k + u, v, 0.6, causal)
        np.testing.assert_allclose(O1, O2, atol=1e-10)
        np.testing.assert_allclose(l2 - l1, 0.6 * (q @ u), atol=1e-10)


@pytest.mark.parametrize("mode", MODES)
def test_linearity_in_v(mode):
    q, k, v1 = rnd(13, 2, 2, 18, 4)
    v2 = np.random.default_rng(14).standard_normal(v1.shape)
    for causal in (False, True):
        a, _ = run(mode, q, k, v1, 0.5, causal)
        b, _ = run(mode, q, k, v2, 0.5, causal)
        c, _ = run(mode, q, k, v1 + v2, 0.5, causal)
        np.testing.assert_allclose(a + b, c, atol=1e-12)


@pytest.mark.parametrize("mode", MODES)
def test_huge_logits_stay_finite(mode):
    # Without the max shift exp(1000) overflows; with it the softmax becomes a
    # hard argmax and O is the V row of the largest logit.
    q = np.zeros((1, 1, 3, 2)); q[..., 0] = 1.0
    k = np.zeros((1, 1, 3, 2)); k[0, 0, :, 0] = [1000.0, 1200.0, 900.0]
    v = np.arange(6, dtype=np.float64).reshape(1, 1, 3, 2)
    O, lse = run(mode, q, k, v, 1.0, False)
    np.testing.assert_allclose(O[0, 0], np.broadcast_to(v[0, 0, 1], (3, 2)), atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], 1200.0, atol=1e-9)


def test_chunked_lse_and_merge_identity():
    # aicoding.csdn.net "Why attention stalls large-model training", sec. 2.2:
    # lse(x) = M + ln sum_chunks exp(lse_chunk - M) for any chunking.  The same
    # identity merges partial outputs: O = sum_c exp(lse_c - lse) O_c.
    q, k, v = rnd(15, 1, 2, 40, 8, scale=1.5)
    O, lse = oracle.attention_rows(q, k, v, 0.35, False)
    bounds = [0, 7, 8, 23, 40]
    Os, ls = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        Oc, lc = oracle.attention_rows(q, np.ascontiguousarray(k[:, :, a:b]), v[:, :, a:b].copy(), 0.35, False,
                                       rows=np.arange(40))
        Os.append(Oc); ls.append(lc)
    # the chunks are [a, b) key ranges computed on sub-sequences of length b - a;
    # rows index the query positions of the full sequence
    ls = np.stack(ls)
    M = ls.max(axis=0)
    lse_merged = M + np.log(np.exp(ls - M).sum(axis=0))
    np.testing.assert_allclose(lse_merged, lse, atol=1e-12)
    O_merged = sum(np.exp(lc - lse)[..., None] * Oc for lc, Oc in zip(ls, Os))
    np.testing.assert_allclose(O_merged, O, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_rows_equal_literal_brute_force(causal):
    for (B, H, N, d) in [(1, 1, 1, 1), (2, 3, 16, 8), (1, 2, 13, 3), (3, 1, 7, 5)]:
        q, k, v = rnd(100 + N, B, H, N, d, scale=2.0)
        kl = np.random.default_rng(N).integers(0, N + 1, size=B).astype(np.int32)
        for key_lens in (None, kl):
            O1, l1 = oracle.attention_rows(q, k, v, 0.45, causal, key_lens)
            O2, l2, _ = oracle.attention_literal(q, k, v, 0.45, causal, key_lens)
            np.testing.assert_allclose(O1, O2, atol=1e-12)
            np.testing.assert_array_equal(np.isneginf(l1), np.isneginf(l2))
            fin = np.isfinite(l2)
            np.testing.assert_allclose(l1[fin], l2[fin], atol=1e-12)


def test_row_subset_matches_full():
    q, k, v = rnd(16, 2, 2, 33, 4)
    O, l = oracle.attention_rows(q, k, v, 0.5, True, np.array([20, 33], dtype=np.int32))
    rows = [0, 5, 19, 20, 32]
    Os, ls = oracle.attention_rows(q, k, v, 0.5, True, np.array([20, 33], dtype=np.int32), rows=rows)
    np.testing.assert_array_equal(Os, O[:, :, rows])
    np.testing.assert_array_equal(ls, l[:, :, rows])


def test_bf16_decode_is_exact():
    bits = np.array([0x0000, 0x8000, 0x3F80, 0xBF80, 0x4049, 0x7F7F, 0x0001], dtype=np.uint16)
    want = [0.0, -0.0, 1.0, -1.0, 3.140625, 3.3895313892515355e38, 2.0 ** -133]
    np.testing.assert_array_equal(oracle.bf16_to_f64(bits), np.array(want))


# --- sliding window (query i sees keys j > i - w) --------------------------------

@pytest.mark.parametrize("mode", MODES)
def test_window_one_causal_is_self_attention_to_own_row(mode):
    # w = 1 with the causal rule leaves exactly key i for query i.
    q, k, v = rnd(31, 2, 2, 19, 5)
    O, lse = run(mode, q, k, v, 0.8, True, window=1)
    np.testing.assert_allclose(O, v, atol=1e-12)
    np.testing.assert_allclose(lse, 0.8 * np.einsum("bhid,bhid->bhi", q, k), atol=1e-12)


@pytest.mark.parametrize("mode", MODES)
def test_window_zero_q_gives_mean_over_window(mode):
    _, k, v = rnd(32, 2, 1, 23, 4)
    q = np.zeros_like(k)
    w = 5
    kl = np.array([23, 17], dtype=np.int32)
    for causal in (True, False):
        O, lse = run(mode, q, k, v, 1.3, causal, kl, window=w)
        for b in range(2):
            for i in range(23):
                lo = max(0, i - w + 1)
                hi = min(i + 1, int(kl[b])) if causal else int(kl[b])
                if hi <= lo:
                    assert np.all(O[b, :, i] == 0.0) and np.all(np.isneginf(lse[b, :, i]))
                    continue
                np.testing.assert_allclose(O[b, :, i], v[b, :, lo:hi].mean(axis=1), atol=1e-12)
                np.testing.assert_allclose(lse[b, :, i], math.log(hi - lo), atol=1e-12)


@pytest.mark.parametrize("mode", MODES)
def test_window_wider_than_sequence_is_no_window(mode):
    q, k, v = rnd(33, 1, 2, 15, 6)
    for causal in (False, True):
        O0, l0 = run(mode, q, k, v, 0.5, causal)
        for w in (15, 16, 1000):
            O1, l1 = run(mode, q, k, v, 0.5, causal, window=w)
            np.testing.assert_array_equal(O0, O1)
            np.testing.assert_array_equal(l0, l1)


@pytest.mark.parametrize("causal", [False, True])
def test_window_rows_equal_literal_brute_force(causal):
    q, k, v = rnd(34, 2, 2, 14, 3, scale=2.0)
    kl = np.array([9, 14], dtype=np.int32)
    for w in (1, 2, 3, 7, 13):
        O1, l1 = run("rows", q, k, v, 0.7, causal, kl, window=w)
        O2, l2 = run("literal", q, k, v, 0.7, causal, kl, window=w)
        np.testing.assert_allclose(O1, O2, atol=1e-12)
        np.testing.assert_array_equal(np.isneginf(l1), np.isneginf(l2))
        fin = np.isfinite(l2)
        np.testing.assert_allclose(l1[fin], l2[fin], atol=1e-12)


def test_bad_arguments_rejected():
    q, k, v = rnd(17, 1, 1, 4, 2)
    with pytest.raises(ValueError):
        oracle.attention_rows(q, k, v, 1.0, False, rows=[0, 4])


# --- the pins must catch plausible mistakes -------------------------------------

def _mutant(kind):
    """A copy of the literal definition with one planted mistake."""
    def f(q, k, v, scale, causal, key_lens=None, window=0):
        q, k, v = [np.asarray(x, dtype=np.float64) for x in (q, k, v)]
        B, H, N, d = q.shape
        sc = 1.0 if kind == "no_scale" else scale
        S = sc * (np.matmul(k, np.swapaxes(q, -1, -2)) if kind == "transposed" else
                  np.matmul(q, np.swapaxes(k, -1, -2)))
        i = np.arange(N)[:, None]; j = np.arange(N)[None, :]
        keep = np.ones((B, 1, N, N), dtype=bool)
        for b in range(B):
            if key_lens is not None:
                kl = int(key_lens[b])
                keep[b, 0] &= (i < kl) if kind == "mask_queries" else (j < kl)
            if causal:
                keep[b, 0] &= (j < i) if kind == "causal_strict" else (j <= i)
            if window > 0:
                keep[b, 0] &= (j >= i - window) if kind == "window_off_by_one" else (j > i - window)
        S = np.where(keep, S, -np.inf)
        m = S.max(-1, keepdims=True)
        m = np.where(np.isfinite(m), m, 0.0)
        E = np.where(keep, np.exp(S - m), 0.0)
        l = E.sum(-1, keepdims=True)
        l = np.where(l > 0, l, 1.0)
        P = E / (1.0 if kind == "no_normalise" else l)
        O = np.matmul(P, v)
        lse = (m + (np.log2(l) if kind == "log2_lse" else np.log(l)))[..., 0]
        if kind == "lse_no_max":
            lse = np.log(l)[..., 0]
        return O, lse
    return f


def _all_pins_pass(fn):
    """Re-run the value pins above against ``fn``; False as soon as one fails."""
    checks = []
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        q = np.array(c["q"])[None, None]; k = np.array(c["k"])[None, None]; v = np.array(c["v"])[None, None]
        kl = None if c["key_len"] is None else np.array([c["key_len"]], dtype=np.int32)
        O, lse = fn(q, k, v, c["scale"], c["causal"], kl)
        checks.append(np.allclose(O[0, 0], c["O"], atol=1e-9) and np.allclose(lse[0, 0], c["lse"], atol=1e-9))
    q, k, v = rnd(6, 1, 2, 9, 4)
    O, lse = fn(q, k, v, 0.25, True)
    checks.append(np.allclose(O[:, :, 0], v[:, :, 0], atol=1e-9))
    qz = np.zeros_like(q)
    O, lse = fn(qz, k, v, 0.9, False, np.array([4], dtype=np.int32))
    checks.append(np.allclose(O[0], v[0, :, :4].mean(axis=1, keepdims=True), atol=1e-9)
                  and np.allclose(lse, math.log(4), atol=1e-9))
    O, lse = fn(q, k, v, 0.8, True, None, window=1)
    checks.append(np.allclose(O, v, atol=1e-9))
    return all(checks)


@pytest.mark.parametrize("kind", ["no_scale", "transposed", "mask_queries", "causal_strict",
                                  "no_normalise", "log2_lse", "lse_no_max", "window_off_by_one"])
def test_pins_catch_planted_mistakes(kind):
    assert _all_pins_pass(_mutant("none"))
    assert not _all_pins_pass(_mutant(kind)), kind


# --- one query against a key/value cache (decode) -------------------------------

def test_decode_rows_match_literal_square_problem():
    # A decode query (Nq = 1) seeing keys 0..cache_len-1 is row i of a square
    # non-causal problem whose key lengths are cache_len: the literal
    # materialised-matrix oracle computes that row independently.
    r = np.random.default_rng(41)
    B, H, L, d = 2, 3, 17, 5
    k = r.standard_normal((B, H, L, d))
    v = r.standard_normal((B, H, L, d))
    q1 = r.standard_normal((B, H, 1, d))
    cl = np.array([11, 17], dtype=np.int32)
    O1, l1 = oracle.attention_rows(q1, k, v, 0.45, False, cl, threads=2)
    for i in (0, 7, 16):
        Q = r.standard_normal((B, H, L, d))
        Q[:, :, i] = q1[:, :, 0]
        O2, l2, _ = oracle.attention_literal(Q, k, v, 0.45, False, cl)
        np.testing.assert_allclose(O1[:, :, 0], O2[:, :, i], atol=1e-12)
        np.testing.assert_allclose(l1[:, :, 0], l2[:, :, i], atol=1e-12)


def test_decode_zero_query_and_empty_cache():
    r = np.random.default_rng(42)
    B, H, L, d = 3, 2, 12, 4
    k = r.standard_normal((B, H, L, d))
    v = r.standard_normal((B, H, L, d))
    q1 = np.zeros((B, H, 1, d))
    cl = np.array([5, 0, 12], dtype=np.int32)
    O, lse = oracle.attention_rows(q1, k, v, 0.7, False, cl, threads=2)
    for b in range(B):
        n = int(cl[b])
        if n == 0:
            assert np.all(O[b] == 0.0) and np.all(np.isneginf(lse[b]))
        else:
            np.testing.assert_allclose(O[b, :, 0], v[b, :, :n].mean(axis=1), atol=1e-12)
            np.testing.assert_allclose(lse[b, :, 0], math.log(n), atol=1e-12)


# --- multi-head block (projections + attention + output projection) -------------

def _bf16_grid(r, shape, scale=1.0):
    # values that are exact in bfloat16, so rounding does not blur the pins
    return oracle.round_bf16(scale * r.standard_normal(shape))


def test_round_bf16_matches_known_values():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e-3, 1.0 + 2 ** -9])
    want = np.array([1.0, 1.0, 1.0 + 2 ** -6, -2.5, 0.0030059814453125, 1.0])
    np.testing.assert_array_equal(oracle.round_bf16(vals), want)
    x = np.random.default_rng(3).standard_normal(1000)
    r = oracle.round_bf16(x)
    assert np.all(np.abs(r - x) <= np.abs(x) * 2.0 ** -8)
    assert np.array_equal(oracle.round_bf16(r), r)


def test_mha_block_brute_force():
    # Element by element from the definition, with plain loops.
    r = np.random.default_rng(51)
    B, N, E, H = 2, 5, 4, 2
    d = E // H
    x = _bf16_grid(r, (B, N, E))
    wqkv = _bf16_grid(r, (E, 3 * E), 0.5)
    wo = _bf16_grid(r, (E, E), 0.5)
    kl = np.array([3, 5], dtype=np.int32)
    for causal in (False, True):
        out, lse = oracle.mha_block(x, wqkv, wo, H, causal, kl, threads=1)
        for b in range(B):
            proj = np.zeros((N, 3 * E))
            for n in range(N):
                for c in range(3 * E):
                    proj[n, c] = sum(x[b, n, e] * wqkv[e, c] for e in range(E))
            proj = oracle.round_bf16(proj)
            merged = np.zeros((N, E))
            for h in range(H):
                for i in range(N):
                    vis = [j for j in range(N) if j < kl[b] and (not causal or j <= i)]
                    s = [sum(proj[i, h * d + t] * proj[j, E + h * d + t] for t in range(d)) / math.sqrt(d) for j in vis]
                    m = max(s)
                    w = [math.exp(z - m) for z in s]
                    tot = sum(w)
                    for t in range(d):
                        merged[i, h * d + t] = sum(wj * proj[j, 2 * E + h * d + t] for wj, j in zip(w, vis)) / tot
                    assert abs(lse[b, h, i] - (m + math.log(tot))) < 1e-12
            merged = oracle.round_bf16(merged)
            want = np.array([[sum(merged[n, e] * wo[e, c] for e in range(E)) for c in range(E)] for n in range(N)])
            np.testing.assert_allclose(out[b], want, atol=1e-12)


def test_mha_block_head_permutation_invariance():
    # Relabelling heads consistently (Q/K/V column blocks and the rows of the
    # output projection) leaves the block's output unchanged.
    r = np.random.default_rng(52)
    B, N, E, H = 1, 7, 8, 4
    d = E // H
    x = _bf16_grid(r, (B, N, E))
    wqkv = _bf16_grid(r, (E, 3 * E), 0.4)
    wo = _bf16_grid(r, (E, E), 0.4)
    perm = np.array([2, 0, 3, 1])
    cols = np.concatenate([np.arange(h * d, (h + 1) * d) for h in perm])
    wqkv2 = np.concatenate([wqkv[:, part * E:(part + 1) * E][:, cols] for part in range(3)], axis=1)
    wo2 = wo[cols]
    o1, l1 = oracle.mha_block(x, wqkv, wo, H, True)
    o2, l2 = oracle.mha_block(x, wqkv2, wo2, H, True)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1[:, perm], l2, atol=1e-12)


# --- backward: gradients of the forward ------------------------------------------

def _loss(q, k, v, g, scale, causal, kl, window=0):
    O, _, _ = oracle.attention_literal(q, k, v, scale, causal, kl, window)
    return float((O * g).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    # d(sum(O * G))/dX by central differences, element by element.
    r = np.random.default_rng(61)
    B, H, N, d = 1, 2, 5, 3
    q, k, v, g = (r.standard_normal((B, H, N, d)) for _ in range(4))
    kl = np.array([4], dtype=np.int32)
    dQ, dK, dV = oracle.attention_backward_literal(q, k, v, g, 0.7, causal, kl)
    eps = 1e-6
    for X, dX in ((q, dQ), (k, dK), (v, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            old = X[idx]
            X[idx] = old + eps
            up = _loss(q, k, v, g, 0.7, causal, kl)
            X[idx] = old - eps
            dn = _loss(q, k, v, g, 0.7, causal, kl)
            X[idx] = old
            num[idx] = (up - dn) / (2 * eps)
        np.testing.assert_allclose(dX, num, atol=1e-7)
    assert np.all(dK[:, :, 4:] == 0.0) and np.all(dV[:, :, 4:] == 0.0)  # hidden keys get no gradient


@pytest.mark.parametrize("causal", [False, True])
def test_backward_window_matches_finite_differences(causal):
    # The sliding window (query i sees keys j > i - w) changes which scores
    # exist; the gradients must be those of that function.
    r = np.random.default_rng(65)
    B, H, N, d, w = 1, 1, 7, 3, 3
    q, k, v, g = (r.standard_normal((B, H, N, d)) for _ in range(4))
    kl = np.array([6], dtype=np.int32)
    dQ, dK, dV = oracle.attention_backward_literal(q, k, v, g, 0.6, causal, kl, window=w)
    eps = 1e-6
    for X, dX in ((q, dQ), (k, dK), (v, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            old = X[idx]
            X[idx] = old + eps
            up = _loss(q, k, v, g, 0.6, causal, kl, w)
            X[idx] = old - eps
            dn = _loss(q, k, v, g, 0.6, causal, kl, w)
            X[idx] = old
            num[idx] = (up - dn) / (2 * eps)
        np.testing.assert_allclose(dX, num, atol=1e-7)
    # with causal and w = 1 every row sees only itself: P = I, so dV = dO and
    # dS = P (dP - D) = 0 gives dQ = dK = 0 (on the rows whose key is visible)
    dQ1, dK1, dV1 = oracle.attention_backward_literal(q, k, v, g, 0.6, True, None, window=1)
    np.testing.assert_allclose(dV1, g, atol=1e-12)
    np.testing.assert_allclose(dQ1, 0.0, atol=1e-12)
    np.testing.assert_allclose(dK1, 0.0, atol=1e-12)
    # a window covering everything is no window
    for a, b_ in zip(oracle.attention_backward_literal(q, k, v, g, 0.6, causal, kl, window=N),
                     oracle.attention_backward_literal(q, k, v, g, 0.6, causal, kl)):
        np.testing.assert_array_equal(a, b_)


def test_backward_sampled_matches_literal():
    r = np.random.default_rng(62)
    B, H, N, d = 2, 2, 37, 8
    q, k, v, g = (r.standard_normal((B, H, N, d)) for _ in range(4))
    kl = np.array([30, 37], dtype=np.int32)
    for causal in (False, True):
        dQ, dK, dV = oracle.attention_backward_literal(q, k, v, g, 0.4, causal, kl)
        rows = [0, 5, 29, 36]
        got = oracle.attention_backward_sampled(q, k, v, g, 0.4, causal, kl, heads=[(0, 1), (1, 0)], q_rows=rows,
                                                k_rows=rows)
        for (b, h), (sq, sk, sv) in got.items():
            np.testing.assert_allclose(sq, dQ[b, h, rows], atol=1e-11)
            np.testing.assert_allclose(sk, dK[b, h, rows], atol=1e-11)
            np.testing.assert_allclose(sv, dV[b, h, rows], atol=1e-11)
        # and with a sliding window
        dQ, dK, dV = oracle.attention_backward_literal(q, k, v, g, 0.4, causal, kl, window=9)
        got = oracle.attention_backward_sampled(q, k, v, g, 0.4, causal, kl, heads=[(0, 1), (1, 0)], q_rows=rows,
                                                k_rows=rows, window=9)
        for (b, h), (sq, sk, sv) in got.items():
            np.testing.assert_allclose(sq, dQ[b, h, rows], atol=1e-11)
            np.testing.assert_allclose(sk, dK[b, h, rows], atol=1e-11)
            np.testing.assert_allclose(sv, dV[b, h, rows], atol=1e-11)


def test_backward_with_stored_output_identity():
    # D from dO . O (O the exact forward output) equals D from P and dP, so
    # passing the exact output changes nothing; a perturbed output moves dQ
    # and dK (through dS) but never dV.
    r = np.random.default_rng(64)
    B, H, N, d = 2, 2, 9, 4
    q, k, v, g = (r.standard_normal((B, H, N, d)) for _ in range(4))
    kl = np.array([7, 9], dtype=np.int32)
    for causal in (False, True):
        ref = oracle.attention_backward_literal(q, k, v, g, 0.6, causal, kl)
        O, _, _ = oracle.attention_literal(q, k, v, 0.6, causal, kl)
        same = oracle.attention_backward_literal(q, k, v, g, 0.6, causal, kl, out=O)
        for a, b in zip(ref, same):
            np.testing.assert_allclose(a, b, atol=1e-12)
        moved = oracle.attention_backward_literal(q, k, v, g, 0.6, causal, kl, out=O + 0.01)
        np.testing.assert_array_equal(moved[2], ref[2])
        assert np.abs(moved[0] - ref[0]).max() > 1e-4 and np.abs(moved[1] - ref[1]).max() > 1e-4
        rows = [0, 3, 8]
        sm = oracle.attention_backward_sampled(q, k, v, g, 0.6, causal, kl, heads=[(1, 0)], q_rows=rows,
                                               k_rows=rows, out=O + 0.01)
        for got, want in zip(sm[(1, 0)], moved):
            np.testing.assert_allclose(got, want[1, 0, rows], atol=1e-11)


def test_backward_uniform_attention_closed_form():
    # Q = 0: P is uniform over the visible keys, so dV_j = (1/n) sum over the
    # rows that see key j of dO_i, computed here with explicit counts.
    r = np.random.default_rng(63)
    B, H, N, d = 1, 1, 6, 2
    k, v, g = (r.standard_normal((B, H, N, d)) for _ in range(3))
    q = np.zeros_like(k)
    _, _, dV = oracle.attention_backward_literal(q, k, v, g, 1.0, True)
    for j in range(N):
        want = sum(g[0, 0, i] / (i + 1) for i in range(j, N))
        np.testing.assert_allclose(dV[0, 0, j], want, atol=1e-12)
