"""GPU parity of the attention backward (attn_bwd: dQ, dK, dV) against the
fp64 oracle on the same seeded inputs.

Tolerances (per gradient tensor G, oracle R): rel-L2 ||G - R|| / ||R|| <=
5e-3 and max |G - R| <= 1e-2 * max|R| + 1e-4.  The kernel's errors are the
bf16 rounding of its result (<= 2^-9 relative), of P^T (the A operand of
dV += P^T dO) and of dS (the operand of dK and dQ), each <= 2^-9 relative
per element and averaging out over the summed keys/queries, plus D taken
from the bf16 forward output (|dO| |O| 2^-9); together a few 2^-9 of the
largest gradient entry at most, and ~1.2 * 2^-9 in L2.  The 1e-4 floor
covers tensors whose exact gradient is zero (a single visible key:
dS = P (dP - D) cancels to rounding noise).

Peaked softmax rows (large logits, or causal rows that see only a few keys)
are the exception for dQ and dK: there dP - D cancels, dS is small, and the
bf16 rounding of the stored output O (through D = dO . O) no longer sits far
below it.  So every case is checked twice: at the bounds above against the
oracle given that stored output for D (the identity the kernel uses, applied
to the same O), and against the exact D at the same bounds for dV (which does
not involve D) and at PEAKED_REL_L2 / 2 * MAX_REL_TO_PEAK for dQ and dK."""
import numpy as np
import pytest

import oracle
import scaled_dot_product_18_b300 as sdp
from scaled_dot_product_18_b300 import inputs as I

from gpu_util import to_dev, torch

pytestmark = pytest.mark.gpu

REL_L2 = 5e-3
PEAKED_REL_L2 = 2e-2
MAX_REL_TO_PEAK = 1e-2
ABS_FLOOR = 1e-4
GUARD = 4096


def run_bwd(q, k, v, dout, scale, causal, key_lens=None, want_out=False, window=0):
    """Forward then backward through the C ABI; gradients as float64 arrays
    (and the forward's bf16 output, as float64, with want_out).  dq/dk/dv
    live inside NaN-filled buffers whose tails must stay NaN."""
    t = torch()
    B, H, N, d = q.shape
    tq, tk, tv, tdo = (to_dev(x) for x in (q, k, v, dout))
    kl = t.from_numpy(np.asarray(key_lens, dtype=np.int32)).cuda() if key_lens is not None else None
    out, lse = sdp.attention(tq, tk, tv, causal=causal, key_lens=kl, scale=scale, window=window)
    n = B * H * N * d
    bufs = [t.full((n + GUARD,), float("nan"), dtype=t.bfloat16, device="cuda") for _ in range(3)]
    ws = t.full((sdp.attn_bwd_workspace_size(B, H, N, d),), 0xFF, dtype=t.uint8, device="cuda")
    stream = t.cuda.current_stream()
    if window:
        st = sdp.attn_bwd_window(tq, tk, tv, out, tdo, lse, bufs[0], bufs[1], bufs[2], B, H, N, d, scale, causal, kl,
                                 window, ws, ws.numel(), stream)
    else:
        st = sdp.attn_bwd(tq, tk, tv, out, tdo, lse, bufs[0], bufs[1], bufs[2], B, H, N, d, scale, causal, kl, ws,
                          ws.numel(), stream)
    assert st == sdp.ATTN_OK, sdp.attn_status_str(st)
    assert sdp.attn_check_device(stream) == sdp.ATTN_OK
    res = []
    for b in bufs:
        assert t.isnan(b[n:].float()).all(), "stray write past the end of a gradient"
        res.append(b[:n].float().cpu().numpy().astype(np.float64).reshape(B, H, N, d))
    if want_out:
        return res, out.float().cpu().numpy().astype(np.float64)
    return res


def assert_grad_close(G, R, what, rel_l2=REL_L2, max_rel=MAX_REL_TO_PEAK):
    assert not np.isnan(G).any(), "%s: unwritten (NaN canary) rows" % what
    err = float(np.abs(G - R).max()) if G.size else 0.0
    peak = float(np.abs(R).max()) if R.size else 0.0
    assert err <= max_rel * peak + ABS_FLOOR, "%s: max-abs %.3e (peak %.3e)" % (what, err, peak)
    nr = float(np.linalg.norm(R))
    if nr > 0:
        rel = float(np.linalg.norm(G - R)) / nr
        assert rel <= rel_l2, "%s: rel-L2 %.3e" % (what, rel)


def check_grads(got, O, ref_exact, ref_stored, what, peaked=True):
    """peaked=False: no row is peaked (no causal mask, no key length below 64,
    at least 64 keys), so dQ and dK meet the tight bounds against the exact D
    as well."""
    for name, G, R, Rs in zip(("dQ", "dK", "dV"), got, ref_exact, ref_stored):
        assert_grad_close(G, Rs, "%s %s (D from the stored output)" % (name, what))
        loose = name != "dV" and peaked
        assert_grad_close(G, R, "%s %s" % (name, what), rel_l2=PEAKED_REL_L2 if loose else REL_L2,
                          max_rel=2 * MAX_REL_TO_PEAK if loose else MAX_REL_TO_PEAK)


CASES = [
    (1, 2, 1, None),
    (1, 2, 64, None),
    (1, 2, 128, None),
    (2, 2, 129, [1, 129]),
    (2, 2, 300, [200, 300]),
    (2, 1, 257, [0, 130]),     # a batch element with no visible key
    (1, 2, 700, None),
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_grid(d, causal):
    for B, H, N, kl in CASES:
        seed = 31 * N + d + (5 if causal else 0)
        q, k, v, do = (I.make_tensor_bits(seed, s, (B, H, N, d)) for s in (0, 1, 2, 4))
        scale = 1.0 / np.sqrt(d)
        kla = None if kl is None else np.array(kl, dtype=np.int32)
        got, O = run_bwd(q, k, v, do, scale, causal, kla, want_out=True)
        ref = oracle.attention_backward_literal(q, k, v, do, scale, causal, kla)
        ref_stored = oracle.attention_backward_literal(q, k, v, do, scale, causal, kla, out=O)
        peaked = causal or N < 64 or (kl is not None and min(kl) < 64)
        check_grads(got, O, ref, ref_stored, "B%d H%d N%d d%d causal=%s kl=%s" % (B, H, N, d, causal, kl), peaked)
        if kla is not None:
            for b in range(B):
                # keys past the key length get exactly zero dK and dV
                assert (got[1][b, :, kla[b]:] == 0).all() and (got[2][b, :, kla[b]:] == 0).all()
                if kla[b] == 0:
                    assert (got[0][b] == 0).all()


def test_backward_custom_scale_and_large_logits():
    # amplitude 3 with scale 0.2: peaked softmax rows (logits of several tens)
    B, H, N, d = 1, 2, 300, 128
    q, k, v = (I.make_tensor_bits(77, s, (B, H, N, d), amplitude=3.0) for s in (0, 1, 2))
    do = I.make_tensor_bits(77, 4, (B, H, N, d))
    for causal in (False, True):
        got, O = run_bwd(q, k, v, do, 0.2, causal, want_out=True)
        ref = oracle.attention_backward_literal(q, k, v, do, 0.2, causal)
        ref_stored = oracle.attention_backward_literal(q, k, v, do, 0.2, causal, out=O)
        check_grads(got, O, ref, ref_stored, "large logits causal=%s" % causal)


def test_backward_dk_dv_deterministic():
    # dK and dV are accumulated in one CTA in a fixed order: bit-identical
    # across calls (dQ adds partials with atomics in no fixed order).
    B, H, N, d = 2, 4, 1000, 128
    q, k, v, do = (I.make_tensor_bits(5, s, (B, H, N, d)) for s in (0, 1, 2, 4))
    a = run_bwd(q, k, v, do, 0.09, True)
    b = run_bwd(q, k, v, do, 0.09, True)
    np.testing.assert_array_equal(a[1], b[1])
    np.testing.assert_array_equal(a[2], b[2])
    assert np.abs(a[0] - b[0]).max() <= MAX_REL_TO_PEAK * np.abs(a[0]).max()


def _sample(N, rng, n_random=8):
    fixed = [0, 1, 127, 128, 129, N // 2, N - 129, N - 1]
    rows = set(r for r in fixed if 0 <= r < N) | set(rng.integers(0, N, size=n_random).tolist())
    return sorted(rows)


@pytest.mark.parametrize("name", ["c4_b4h32n4096d128_causal", "c5_b1h32n16384d128_causal"])
def test_backward_sampled_full_size(name):
    # The full-size problem the backward benchmark times; the oracle rebuilds
    # sampled rows of dQ and dK/dV of sampled heads.
    w = I.WORKLOADS[name]
    x = I.make_inputs(w)
    do = I.make_dout(w)
    got, O = run_bwd(x.q, x.k, x.v, do, w.scale, w.causal, x.key_lens, want_out=True)
    rng = np.random.default_rng(99)
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    rows = _sample(w.N, rng)
    kw = dict(heads=heads, q_rows=rows, k_rows=rows)
    ref = oracle.attention_backward_sampled(x.q, x.k, x.v, do, w.scale, w.causal, x.key_lens, **kw)
    ref_stored = oracle.attention_backward_sampled(x.q, x.k, x.v, do, w.scale, w.causal, x.key_lens, out=O, **kw)
    for (b, h) in heads:
        mine = [g[b, h, rows] for g in got]
        check_grads(mine, None, ref[(b, h)], ref_stored[(b, h)], "%s b%d h%d" % (name, b, h))
    for G in got:
        assert np.isfinite(G).all()


@pytest.mark.parametrize("causal", [True, False])
def test_backward_d64_long_sequence_sampled(causal):
    # d = 64 (dQ staged in half a ring stage) over N = 4096 with key lengths.
    B, H, N, d = 2, 2, 4096, 64
    q, k, v, do = (I.make_tensor_bits(52, s, (B, H, N, d)) for s in (0, 1, 2, 4))
    kl = np.array([N, 2500], dtype=np.int32)
    got, O = run_bwd(q, k, v, do, 0.125, causal, kl, want_out=True)
    rows = _sample(N, np.random.default_rng(8))
    heads = [(0, 1), (1, 0)]
    kw = dict(heads=heads, q_rows=rows, k_rows=rows)
    ref = oracle.attention_backward_sampled(q, k, v, do, 0.125, causal, kl, **kw)
    ref_stored = oracle.attention_backward_sampled(q, k, v, do, 0.125, causal, kl, out=O, **kw)
    for (b, h) in heads:
        check_grads([g[b, h, rows] for g in got], None, ref[(b, h)], ref_stored[(b, h)],
                    "d64 N4096 causal=%s b%d h%d" % (causal, b, h))
    assert (got[1][1, :, 2500:] == 0).all() and (got[2][1, :, 2500:] == 0).all()


WINDOW_CASES = [(1, 129, 1), (2, 300, 64), (2, 300, 127), (2, 300, 129), (1, 700, 200), (2, 257, 300)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_window_grid(d, causal):
    # attn_bwd_window against the oracle's windowed backward (query i sees
    # keys j > i - w), with key lengths on two-batch cases; w >= N is no window.
    for B, N, w in WINDOW_CASES:
        H = 2
        seed = 17 * N + w + d + (7 if causal else 0)
        q, k, v, do = (I.make_tensor_bits(seed, s, (B, H, N, d)) for s in (0, 1, 2, 4))
        kla = np.array([max(1, (2 * N) // 3), N][:B], dtype=np.int32) if B == 2 else None
        scale = 1.0 / np.sqrt(d)
        got, O = run_bwd(q, k, v, do, scale, causal, kla, want_out=True, window=w)
        ref = oracle.attention_backward_literal(q, k, v, do, scale, causal, kla, window=w)
        ref_stored = oracle.attention_backward_literal(q, k, v, do, scale, causal, kla, out=O, window=w)
        check_grads(got, O, ref, ref_stored, "window N%d w%d d%d causal=%s kl=%s" % (N, w, d, causal, kla))


def test_backward_window_covering_everything_matches_attn_bwd():
    B, H, N, d = 2, 2, 333, 128
    q, k, v, do = (I.make_tensor_bits(91, s, (B, H, N, d)) for s in (0, 1, 2, 4))
    kl = np.array([200, 333], dtype=np.int32)
    for causal in (False, True):
        a = run_bwd(q, k, v, do, 0.09, causal, kl)
        b = run_bwd(q, k, v, do, 0.09, causal, kl, window=N + 5)
        np.testing.assert_array_equal(a[1], b[1])
        np.testing.assert_array_equal(a[2], b[2])


def test_backward_window_sampled_full_size():
    # The long-context workload with the pages' window of 512 (the launch
    # `bench.py --backward --window 512` times); sampled rows of two heads.
    w = I.WORKLOADS["c5_b1h32n16384d128_causal"]
    window = 512
    x = I.make_inputs(w)
    do = I.make_dout(w)
    got, O = run_bwd(x.q, x.k, x.v, do, w.scale, w.causal, x.key_lens, want_out=True, window=window)
    rng = np.random.default_rng(7)
    heads = [(0, 0), (0, w.H - 1)]
    rows = _sample(w.N, rng)
    kw = dict(heads=heads, q_rows=rows, k_rows=rows, window=window)
    ref = oracle.attention_backward_sampled(x.q, x.k, x.v, do, w.scale, w.causal, x.key_lens, **kw)
    ref_stored = oracle.attention_backward_sampled(x.q, x.k, x.v, do, w.scale, w.causal, x.key_lens, out=O, **kw)
    for (b, h) in heads:
        mine = [g[b, h, rows] for g in got]
        check_grads(mine, None, ref[(b, h)], ref_stored[(b, h)], "window512 b%d h%d" % (b, h))
    for G in got:
        assert np.isfinite(G).all()
