"""GPU parity of attn_decode (one query per (b, h) against a key/value cache)
with the fp64 oracle, which takes the query as a one-row query block."""
import numpy as np
import pytest

import oracle
import scaled_dot_product_18_b300 as sdp
from scaled_dot_product_18_b300 import inputs as I

from gpu_util import LSE_ABS, MAX_ABS, REL_L2, to_dev

pytestmark = pytest.mark.gpu


def run_decode(q, k, v, scale, cache_lens=None, ws_fill=float("nan"), calls=1):
    import torch
    B, H, L, d = k.shape
    tq = to_dev(q)
    tk = to_dev(k) if L > 0 else torch.empty((B, H, 0, d), dtype=torch.bfloat16, device="cuda")
    tv = to_dev(v) if L > 0 else torch.empty((B, H, 0, d), dtype=torch.bfloat16, device="cuda")
    out = torch.full((B, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    nbytes = sdp.attn_decode_workspace_size(B, H, max(L, 1), d)
    ws = torch.full((nbytes // 4,), ws_fill, dtype=torch.float32, device="cuda")
    cl = torch.from_numpy(np.asarray(cache_lens, dtype=np.int32)).cuda() if cache_lens is not None else None
    res = []
    for _ in range(calls):
        st = sdp.attn_decode(tq, tk if L > 0 else None, tv if L > 0 else None, out, lse, B, H, L, d, scale, cl, ws,
                             nbytes, torch.cuda.current_stream())
        assert st == sdp.ATTN_OK, sdp.attn_status_str(st)
        assert sdp.attn_check_device(torch.cuda.current_stream()) == sdp.ATTN_OK
        res.append((out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)))
    return res if calls > 1 else res[0]


def check(O, lse, O_ref, lse_ref, what):
    assert not np.isnan(O).any() and not np.isnan(lse).any(), what
    err = float(np.abs(O - O_ref).max())
    denom = float(np.linalg.norm(O_ref))
    rel = float(np.linalg.norm(O - O_ref)) / denom if denom > 0 else float(np.linalg.norm(O))
    assert err <= MAX_ABS, "%s: max-abs %.3e" % (what, err)
    assert rel <= REL_L2, "%s: rel-L2 %.3e" % (what, rel)
    fin = np.isfinite(lse_ref)
    np.testing.assert_array_equal(np.isneginf(lse), ~fin, err_msg=what)
    if fin.any():
        assert float(np.abs(lse[fin] - lse_ref[fin]).max()) <= LSE_ABS, what


def oracle_decode(q, k, v, scale, cache_lens=None):
    O, lse = oracle.attention_rows(q[:, :, None], k, v, scale, False, cache_lens)
    return O[:, :, 0], lse[:, :, 0]


@pytest.mark.parametrize("d", [64, 128])
def test_decode_grid(d):
    for (B, H, L) in [(1, 1, 1), (2, 3, 63), (3, 2, 257), (2, 4, 1000), (1, 8, 4100)]:
        seed = B * 1000 + H * 100 + L + d
        q = I.make_tensor_bits(seed, 0, (B, H, d))
        k = I.make_tensor_bits(seed, 1, (B, H, L, d))
        v = I.make_tensor_bits(seed, 2, (B, H, L, d))
        scale = 1.0 / np.sqrt(d)
        for cl in (None, np.array(([L, 1, max(1, L // 3)] * B)[:B], dtype=np.int32)):
            O, lse = run_decode(q, k, v, scale, cl)
            O_ref, lse_ref = oracle_decode(q, k, v, scale, cl)
            check(O, lse, O_ref, lse_ref, "B=%d H=%d L=%d d=%d lens=%s" % (B, H, L, d, cl))


def test_decode_empty_caches():
    B, H, L, d = 3, 2, 500, 128
    q = I.make_tensor_bits(3, 0, (B, H, d))
    k = I.make_tensor_bits(3, 1, (B, H, L, d))
    v = I.make_tensor_bits(3, 2, (B, H, L, d))
    cl = np.array([0, 7, 0], dtype=np.int32)
    O, lse = run_decode(q, k, v, 0.1, cl)
    assert np.all(O[[0, 2]] == 0.0) and np.all(np.isneginf(lse[[0, 2]]))
    check(O, lse, *oracle_decode(q, k, v, 0.1, cl), "empty caches")
    O, lse = run_decode(q, k[:, :, :0], v[:, :, :0], 0.1, None)  # L = 0
    assert np.all(O == 0.0) and np.all(np.isneginf(lse))


def test_decode_workspace_reuse_and_garbage():
    # The workspace needs no clearing: garbage in it and back-to-back calls on
    # the same workspace give the same bits.
    B, H, L, d = 2, 5, 3000, 128
    q = I.make_tensor_bits(8, 0, (B, H, d))
    k = I.make_tensor_bits(8, 1, (B, H, L, d))
    v = I.make_tensor_bits(8, 2, (B, H, L, d))
    (O1, l1), (O2, l2) = run_decode(q, k, v, 0.09, np.array([3000, 1234], dtype=np.int32), ws_fill=1e30, calls=2)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(l1, l2)
    check(O1, l1, *oracle_decode(q, k, v, 0.09, np.array([3000, 1234], dtype=np.int32)), "reuse")


def test_decode_zero_query_is_mean_of_cache():
    B, H, L, d = 2, 3, 777, 64
    q = I.f64_to_bf16_bits(np.zeros((B, H, d)))
    k = I.make_tensor_bits(5, 1, (B, H, L, d))
    v = I.make_tensor_bits(5, 2, (B, H, L, d))
    O, lse = run_decode(q, k, v, 0.125, np.array([777, 100], dtype=np.int32))
    vv = oracle.bf16_to_f64(v)
    np.testing.assert_allclose(O[0], vv[0].mean(axis=1), atol=2e-2)
    np.testing.assert_allclose(O[1], vv[1, :, :100].mean(axis=1), atol=2e-2)
    np.testing.assert_allclose(lse, np.log(np.array([[777.0] * H, [100.0] * H])), atol=1e-3)


@pytest.mark.parametrize("name", list(I.DECODE_WORKLOADS))
def test_decode_workloads_sampled(name):
    # Full-size caches, the launch the decode bench times; the oracle checks
    # sampled heads.
    w = I.DECODE_WORKLOADS[name]
    x = I.make_decode_inputs(w)
    O, lse = run_decode(x.q, x.k, x.v, w.scale, x.key_lens)
    assert np.isfinite(O).all() and np.isfinite(lse).all()
    rng = np.random.default_rng(5)
    for b, h in [(0, 0), (w.B - 1, w.H - 1)] + [(int(rng.integers(w.B)), int(rng.integers(w.H))) for _ in range(3)]:
        q = x.q[b:b + 1, h:h + 1]
        k = x.k[b:b + 1, h:h + 1]
        v = x.v[b:b + 1, h:h + 1]
        O_ref, lse_ref = oracle_decode(q, k, v, w.scale, None)
        check(O[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], O_ref, lse_ref, "%s b%d h%d" % (name, b, h))
