"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs, plus exact mask agreement and full-size properties."""
import numpy as np
import pytest

import oracle
from scaled_dot_product_18_b300 import inputs as I

from gpu_util import assert_close, run_cuda

pytestmark = pytest.mark.gpu

SMALL = ["c1_b1h2n128d64", "c2_b2h8n100d64_keylens", "c3_b16h12n512d64_keylens_x1.5"]
LARGE = ["c4_b4h32n4096d128_causal", "c5_b1h32n16384d128_causal"]


@pytest.mark.parametrize("name", SMALL)
def test_workload_full_parity(name):
    w = I.WORKLOADS[name]
    x = I.make_inputs(w)
    O, lse = run_cuda(x.q, x.k, x.v, w.scale, w.causal, x.key_lens)
    O_ref, lse_ref = oracle.attention_rows(x.q, x.k, x.v, w.scale, w.causal, x.key_lens)
    assert_close(O, lse, O_ref, lse_ref, name)


def _sample_rows(N, rng, n_random=40):
    fixed = [0, 1, 2, 63, 64, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1]
    rows = set(r for r in fixed if 0 <= r < N)
    rows |= set(rng.integers(0, N, size=n_random).tolist())
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("name", LARGE + list(I.EXTRA_WORKLOADS))
def test_workload_sampled_parity(name):
    # Full size, the launch the benchmark times; the oracle computes sampled
    # rows of sampled heads, and whole-tensor properties cover every row.
    w = I.WORKLOADS[name] if name in I.WORKLOADS else I.EXTRA_WORKLOADS[name]
    x = I.make_inputs(w)
    O, lse = run_cuda(x.q, x.k, x.v, w.scale, w.causal, x.key_lens)
    rng = np.random.default_rng(1234)
    rows = _sample_rows(w.N, rng)
    heads = [(0, 0), (w.B - 1, w.H - 1)] + [(int(rng.integers(w.B)), int(rng.integers(w.H))) for _ in range(4)]
    for b, h in heads:
        q = x.q[b:b + 1, h:h + 1]
        k = x.k[b:b + 1, h:h + 1]
        v = x.v[b:b + 1, h:h + 1]
        kl = None if x.key_lens is None else x.key_lens[b:b + 1]
        O_ref, lse_ref = oracle.attention_rows(q, k, v, w.scale, w.causal, kl, rows=rows)
        assert_close(O[b:b + 1, h:h + 1, rows], lse[b:b + 1, h:h + 1, rows], O_ref, lse_ref, "%s b%d h%d" % (name, b, h))
    # every row written and finite
    assert np.isfinite(O).all() and np.isfinite(lse).all()
    if w.causal:
        # causal row 0 sees only key 0: O = V[0] exactly (weight 1), lse = s_00
        v0 = oracle.bf16_to_f64(x.v[:, :, 0])
        np.testing.assert_array_equal(O[:, :, 0], v0)
        s00 = w.scale * np.einsum("bhd,bhd->bh", oracle.bf16_to_f64(x.q[:, :, 0]), oracle.bf16_to_f64(x.k[:, :, 0]))
        assert np.abs(lse[:, :, 0] - s00).max() <= 1e-3
    # convex combination of V rows: every output lies inside the V range
    assert O.max() <= oracle.bf16_to_f64(x.v).max() + 1e-2 and O.min() >= oracle.bf16_to_f64(x.v).min() - 1e-2


@pytest.mark.parametrize("causal", [True, False])
def test_d64_long_sequence_sampled(causal):
    # The d = 64 instance (8-slot K/V ring) over many ring wraps: N = 8192,
    # with key lengths on the second batch element; sampled rows.
    B, H, N, d = 2, 3, 8192, 64
    q, k, v = (I.make_tensor_bits(51, s, (B, H, N, d)) for s in (0, 1, 2))
    kl = np.array([N, 5000], dtype=np.int32)
    O, lse = run_cuda(q, k, v, 0.125, causal, kl)
    rows = _sample_rows(N, np.random.default_rng(5))
    for b, h in ((0, 0), (1, 2)):
        O_ref, lse_ref = oracle.attention_rows(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], 0.125,
                                               causal, kl[b:b + 1], rows=rows)
        assert_close(O[b:b + 1, h:h + 1, rows], lse[b:b + 1, h:h + 1, rows], O_ref, lse_ref,
                     "d64 N8192 causal=%s b%d h%d" % (causal, b, h))
    assert np.isfinite(O).all() and np.isfinite(lse).all()


EDGE_N = [1, 2, 63, 64, 65, 127, 128, 129, 255, 257]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_edge_grid(d, causal):
    for N in EDGE_N:
        for kl0 in sorted({1, max(N - 1, 1), N}):
            B, H = 2, 2
            seed = 1000 * N + kl0 + (7 if causal else 0) + d
            q = I.make_tensor_bits(seed, I.STREAM_Q, (B, H, N, d))
            k = I.make_tensor_bits(seed, I.STREAM_K, (B, H, N, d))
            v = I.make_tensor_bits(seed, I.STREAM_V, (B, H, N, d))
            kl = np.array([kl0, N], dtype=np.int32)
            scale = 1.0 / np.sqrt(d)
            O, lse = run_cuda(q, k, v, scale, causal, kl)
            O_ref, lse_ref = oracle.attention_rows(q, k, v, scale, causal, kl)
            assert_close(O, lse, O_ref, lse_ref, "N=%d key_len=%d d=%d causal=%s" % (N, kl0, d, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_key_len_zero_gives_zero_and_minus_inf(causal):
    B, H, N, d = 3, 2, 130, 64
    q, k, v = (I.make_tensor_bits(5, s, (B, H, N, d)) for s in (0, 1, 2))
    kl = np.array([0, 77, 130], dtype=np.int32)
    O, lse = run_cuda(q, k, v, 0.125, causal, kl)
    assert np.all(O[0] == 0.0) and np.all(np.isneginf(lse[0]))
    O_ref, lse_ref = oracle.attention_rows(q, k, v, 0.125, causal, kl)
    assert_close(O, lse, O_ref, lse_ref, "key_len 0")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_mask_probe_exact(d, causal):
    # With V[j] = e_j (one-hot, N <= d) the output row i is row i of the
    # softmax matrix P itself: hidden keys must get exactly 0, visible keys a
    # positive weight.  Exact agreement on which positions are masked.
    N = min(d, 100)
    B, H = 2, 2
    q, k = (I.make_tensor_bits(9, s, (B, H, N, d)) for s in (0, 1))
    eye = np.zeros((N, d))
    eye[np.arange(N), np.arange(N)] = 1.0
    from scaled_dot_product_18_b300.inputs import f64_to_bf16_bits
    v = np.broadcast_to(f64_to_bf16_bits(eye), (B, H, N, d)).copy()
    kl = np.array([37, N], dtype=np.int32)
    O, lse = run_cuda(q, k, v, 1.0 / np.sqrt(d), causal, kl)
    for b in range(B):
        keep = oracle.visible_mask(N, causal, int(kl[b]))
        Pg = O[b, :, :, :N]
        assert np.all(Pg[:, ~keep] == 0.0), "weight on a hidden key"
        assert np.all(Pg[:, keep] > 0.0), "zero weight on a visible key"
        assert np.all(O[b, :, :, N:] == 0.0)
    O_ref, lse_ref = oracle.attention_rows(q, k, v, 1.0 / np.sqrt(d), causal, kl)
    assert_close(O, lse, O_ref, lse_ref, "one-hot probe")


@pytest.mark.parametrize("d", [64, 128])
def test_large_logits_and_lazy_rescale(d):
    # Key norms grow along the sequence so each row's running max keeps rising
    # across key tiles (the rescale path), with logits far beyond exp's range.
    # d = 64 keeps P in its own TMEM columns, d = 128 over the scores.
    B, H, N = 1, 4, 640
    base_q = oracle.bf16_to_f64(I.make_tensor_bits(21, 0, (B, H, N, d)))
    base_k = oracle.bf16_to_f64(I.make_tensor_bits(21, 1, (B, H, N, d)))
    ramp = (1.0 + 6.0 * np.arange(N) / N)[None, None, :, None]
    from scaled_dot_product_18_b300.inputs import f64_to_bf16_bits
    q = f64_to_bf16_bits(base_q * 3.0)
    k = f64_to_bf16_bits(base_k * ramp)
    v = I.make_tensor_bits(21, 2, (B, H, N, d))
    for causal in (False, True):
        O, lse = run_cuda(q, k, v, 1.0 / np.sqrt(d), causal)
        O_ref, lse_ref = oracle.attention_rows(q, k, v, 1.0 / np.sqrt(d), causal)
        assert np.abs(lse_ref).max() > 50  # far outside exp's fp32 range without the max shift
        assert_close(O, lse, O_ref, lse_ref, "large logits causal=%s d=%d" % (causal, d))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("jump", [12.0, 30.0])
def test_max_jump_inside_a_key_tile(jump, d):
    # Within one 128-key tile the row max is settled from the first 64 keys;
    # here keys 64..127 of the first tile (and of the third) score `jump`
    # higher than keys 0..63 (log2 units: x 1.44).  jump 12: the second half
    # stays below the in-tile margin, its weights reach ~2^17 and the next
    # tile moves the max; jump 30: past the margin, the first half's stored
    # weights are rescaled in place.  Rows differ (a per-row jump), so warps
    # hold rows that do and rows that do not move.
    from scaled_dot_product_18_b300.inputs import f64_to_bf16_bits
    B, H, N = 1, 2, 384
    rng_q = oracle.bf16_to_f64(I.make_tensor_bits(23, 0, (B, H, N, d)))
    rng_k = oracle.bf16_to_f64(I.make_tensor_bits(23, 1, (B, H, N, d)))
    q = rng_q * 0.2
    k = rng_k * 0.2
    # unit direction e_0 carries the jump: q_i[0] = a_i, k_j[0] = 1 on the
    # boosted keys, so s_ij gains a_i / sqrt(d) * sqrt(d) = a_i with scale 1/sqrt(d)
    a = jump * (0.5 + 0.5 * (np.arange(N) % 2))  # half the rows jump fully, half by half
    q[..., 0] = a[None, None, :] * np.sqrt(d)
    boost = np.zeros(N)
    boost[64:128] = 1.0
    boost[320:384] = 1.0
    k[..., 0] = boost[None, None, :]
    qb, kb = f64_to_bf16_bits(q), f64_to_bf16_bits(k)
    v = I.make_tensor_bits(23, 2, (B, H, N, d))
    scale = 1.0 / np.sqrt(d)
    O, lse = run_cuda(qb, kb, v, scale, False)
    O_ref, lse_ref = oracle.attention_rows(qb, kb, v, scale, False)
    assert_close(O, lse, O_ref, lse_ref, "in-tile max jump %.0f d=%d" % (jump, d))


def test_custom_scale_no_lse_and_side_stream():
    import torch
    B, H, N, d = 2, 3, 300, 128
    q, k, v = (I.make_tensor_bits(31, s, (B, H, N, d)) for s in (0, 1, 2))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        O, lse = run_cuda(q, k, v, 0.3, True, None, with_lse=False, stream=s)
    assert lse is None
    O_ref, _ = oracle.attention_rows(q, k, v, 0.3, True)
    assert_close(O, None, O_ref, None, "scale 0.3, no lse, side stream")


@pytest.mark.parametrize("d", [64, 128])
def test_output_only_16_byte_aligned(d):
    # O 16 bytes past a 512-byte boundary: the d = 128 epilogue falls back
    # from 32-byte to 16-byte row stores, the d = 64 O tensor map starts
    # off the usual alignment.
    B, H, N = 2, 3, 333
    q, k, v = (I.make_tensor_bits(57, s, (B, H, N, d)) for s in (0, 1, 2))
    scale = 1.0 / np.sqrt(d)
    O, lse = run_cuda(q, k, v, scale, True, out_offset=8)
    O_ref, lse_ref = oracle.attention_rows(q, k, v, scale, True)
    assert_close(O, lse, O_ref, lse_ref, "O at +16 bytes, d=%d" % d)


def test_deterministic():
    B, H, N, d = 1, 4, 1000, 128
    q, k, v = (I.make_tensor_bits(41, s, (B, H, N, d)) for s in (0, 1, 2))
    O1, l1 = run_cuda(q, k, v, 0.1, True)
    O2, l2 = run_cuda(q, k, v, 0.1, True)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_many_items_per_cta_with_empty_items(d, causal):
    # 192 heads x 2 query pairs = 384 work items for at most one CTA per SM:
    # without the causal mask each CTA walks two or three items, carrying its
    # barrier phases, ring position and Q buffers from one to the next, and
    # some items have no visible key at all (key length 0) or one.
    B, H, N = 48, 4, 300
    q, k, v = (I.make_tensor_bits(57 + d, s, (B, H, N, d)) for s in (0, 1, 2))
    rng = np.random.default_rng(5 + d)
    kl = rng.integers(0, N + 1, size=B).astype(np.int32)
    kl[::7] = 0
    kl[3::11] = 1
    kl[5::13] = N
    O, lse = run_cuda(q, k, v, 1.0 / np.sqrt(d), causal, kl)
    O_ref, lse_ref = oracle.attention_rows(q, k, v, 1.0 / np.sqrt(d), causal, kl)
    assert_close(O, lse, O_ref, lse_ref, "many items d=%d causal=%s" % (d, causal))
