"""GPU parity of the sliding-window entry point (attn_fwd_window) against the
fp64 oracle: query i sees keys j > i - window, together with the causal and
key-length rules."""
import numpy as np
import pytest

import oracle
import scaled_dot_product_18_b300 as sdp
from scaled_dot_product_18_b300 import inputs as I

from gpu_util import assert_close, run_cuda

pytestmark = pytest.mark.gpu


def windowed(window):
    def fn(q, k, v, out, lse, B, H, N, d, scale, causal, kl, stream):
        return sdp.attn_fwd_window(q, k, v, out, lse, B, H, N, d, scale, causal, kl, window, stream)
    return fn


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
def test_window_edge_grid(d, causal):
    for N in (1, 65, 129, 300, 700):
        for w in (1, 2, 64, 127, 128, 129, 300):
            if w >= N and N > 1:
                continue
            B, H = 2, 2
            seed = 7 * N + w + d + (3 if causal else 0)
            q, k, v = (I.make_tensor_bits(seed, s, (B, H, N, d)) for s in (0, 1, 2))
            kl = np.array([max(1, (2 * N) // 3), N], dtype=np.int32)
            scale = 1.0 / np.sqrt(d)
            O, lse = run_cuda(q, k, v, scale, causal, kl, entry=windowed(w))
            O_ref, lse_ref = oracle.attention_rows(q, k, v, scale, causal, kl, window=w)
            assert_close(O, lse, O_ref, lse_ref, "N=%d w=%d d=%d causal=%s" % (N, w, d, causal))


def test_window_covering_everything_matches_attn_fwd():
    B, H, N, d = 2, 3, 333, 128
    q, k, v = (I.make_tensor_bits(44, s, (B, H, N, d)) for s in (0, 1, 2))
    kl = np.array([200, 333], dtype=np.int32)
    for causal in (False, True):
        O0, l0 = run_cuda(q, k, v, 0.09, causal, kl)
        for w in (0, N, N + 5):
            O1, l1 = run_cuda(q, k, v, 0.09, causal, kl, entry=windowed(w))
            np.testing.assert_array_equal(O0, O1)
            np.testing.assert_array_equal(l0, l1)


@pytest.mark.parametrize("causal", [True, False])
def test_window_mask_probe_exact(causal):
    # V[j] = e_j: output row i is row i of P itself; keys outside the window
    # must get exactly zero weight, keys inside a positive weight.
    N, d, B, H, w = 100, 128, 2, 2, 37
    q, k = (I.make_tensor_bits(9, s, (B, H, N, d)) for s in (0, 1))
    eye = np.zeros((N, d))
    eye[np.arange(N), np.arange(N)] = 1.0
    v = np.broadcast_to(I.f64_to_bf16_bits(eye), (B, H, N, d)).copy()
    kl = np.array([61, N], dtype=np.int32)
    O, lse = run_cuda(q, k, v, 1.0 / np.sqrt(d), causal, kl, entry=windowed(w))
    for b in range(B):
        keep = oracle.visible_mask(N, causal, int(kl[b]), w)
        Pg = O[b, :, :, :N]
        assert np.all(Pg[:, ~keep] == 0.0), "weight on a hidden key"
        rows = keep.any(axis=1)
        assert np.all(Pg[:, keep] > 0.0), "zero weight on a visible key"
        assert np.all(O[b, :, ~rows] == 0.0) and np.all(np.isneginf(lse[b, :, ~rows]))


def test_window_rows_without_visible_keys():
    # key_len 10 and a causal window of 4: rows i >= 13 see nothing.
    B, H, N, d = 1, 2, 300, 64
    q, k, v = (I.make_tensor_bits(12, s, (B, H, N, d)) for s in (0, 1, 2))
    kl = np.array([10], dtype=np.int32)
    O, lse = run_cuda(q, k, v, 0.125, True, kl, entry=windowed(4))
    assert np.all(O[:, :, 13:] == 0.0) and np.all(np.isneginf(lse[:, :, 13:]))
    O_ref, lse_ref = oracle.attention_rows(q, k, v, 0.125, True, kl, window=4)
    assert_close(O, lse, O_ref, lse_ref, "rows without visible keys")


def test_window_long_context_sampled():
    # The long-context shape with the pages' window w = 512, the launch a
    # sliding-window bench would time; the oracle computes sampled rows.
    w = I.WORKLOADS["c5_b1h32n16384d128_causal"]
    x = I.make_inputs(w)
    O, lse = run_cuda(x.q, x.k, x.v, w.scale, True, None, entry=windowed(512))
    rng = np.random.default_rng(77)
    rows = np.array(sorted(set([0, 1, 511, 512, 513, 1000, 16383] + rng.integers(0, w.N, 30).tolist())), dtype=np.int64)
    for h in (0, 13, 31):
        sl = slice(h, h + 1)
        O_ref, lse_ref = oracle.attention_rows(x.q[:, sl], x.k[:, sl], x.v[:, sl], w.scale, True, None, rows=rows,
                                               window=512)
        assert_close(O[:, sl, rows], lse[:, sl, rows], O_ref, lse_ref, "w=512 head %d" % h)
    assert np.isfinite(O).all() and np.isfinite(lse).all()
