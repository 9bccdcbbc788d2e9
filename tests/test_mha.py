"""GPU parity of attn_mha_fwd (fused QKV projection, heads, attention, output
projection) with the fp64 block oracle, which rounds Q/K/V and the merged
heads to bf16 at the same two points."""
import numpy as np
import pytest

import oracle
import scaled_dot_product_18_b300 as sdp
from scaled_dot_product_18_b300 import inputs as I

from gpu_util import MAX_ABS, REL_L2, to_dev

pytestmark = pytest.mark.gpu

# Q/K/V are bf16 roundings of fp32 GEMM sums on the GPU and of exact sums in
# the oracle; where an exact sum lies within the fp32 error of a bf16
# rounding midpoint the two round one ulp (2^-8 relative) apart.  One such q
# or k element moves a logit by at most 2^-8 |q_t k_t| / sqrt(d); with
# |q_t|, |k_t| <= 5 and d >= 64 that is 0.012, which bounds the shift of a
# row's log-sum-exp.  The block's output is held to the attention tolerances.
BLOCK_LSE_ABS = 1.2e-2


def run_mha(w: I.MhaWorkload, x: I.MhaInputs):
    import torch
    tx, tw, to = to_dev(x.x), to_dev(x.w_qkv), to_dev(x.w_o)
    out = torch.full((w.B, w.N, w.E), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.H, w.N), float("nan"), dtype=torch.float32, device="cuda")
    nbytes = sdp.attn_mha_workspace_size(w.B, w.N, w.E)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    kl = torch.from_numpy(x.key_lens).cuda() if x.key_lens is not None else None
    st = sdp.attn_mha_fwd(tx, tw, to, out, lse, w.B, w.N, w.E, w.H, w.causal, kl, ws, nbytes,
                          torch.cuda.current_stream())
    assert st == sdp.ATTN_OK, sdp.attn_status_str(st)
    assert sdp.attn_check_device(torch.cuda.current_stream()) == sdp.ATTN_OK
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def check(out, lse, out_ref, lse_ref, what):
    assert not np.isnan(out).any() and not np.isnan(lse).any(), what
    err = float(np.abs(out - out_ref).max())
    rel = float(np.linalg.norm(out - out_ref) / np.linalg.norm(out_ref))
    assert err <= MAX_ABS, "%s: max-abs %.3e" % (what, err)
    assert rel <= REL_L2, "%s: rel-L2 %.3e" % (what, rel)
    assert float(np.abs(lse - lse_ref).max()) <= BLOCK_LSE_ABS, what
    assert float(np.median(np.abs(lse - lse_ref))) <= 1e-4, what  # flips are rare: most rows agree closely


@pytest.mark.parametrize("name", ["mha_b2n100e512h8", "mha_b16n512e768h12_keylens"])
def test_mha_workloads(name):
    w = I.MHA_WORKLOADS[name]
    x = I.make_mha_inputs(w)
    out, lse = run_mha(w, x)
    out_ref, lse_ref = oracle.mha_block(x.x, x.w_qkv, x.w_o, w.H, w.causal, x.key_lens)
    check(out, lse, out_ref, lse_ref, name)


@pytest.mark.parametrize("B,N,E,H,causal,lens", [
    (1, 300, 1024, 8, True, None),
    (3, 257, 256, 2, False, (1, 257)),
    (2, 129, 384, 6, True, (100, 129)),
])
def test_mha_shapes(B, N, E, H, causal, lens):
    w = I.MhaWorkload("t", B, N, E, H, causal, lens, seed=B * 7 + N)
    x = I.make_mha_inputs(w)
    out, lse = run_mha(w, x)
    out_ref, lse_ref = oracle.mha_block(x.x, x.w_qkv, x.w_o, w.H, w.causal, x.key_lens)
    check(out, lse, out_ref, lse_ref, "B=%d N=%d E=%d H=%d" % (B, N, E, H))


def test_mha_long_context_sampled():
    # The long-context block at full size (B=1 N=16384 E=4096 H=32 causal), the
    # launch the benchmark times.  The oracle follows the block's steps for
    # sampled rows only: K and V for every key (one fp64 projection, rounded
    # to bf16 as in the block), Q for the sampled rows, attention of those
    # rows in every head, the merged row rounded to bf16, the output
    # projection.  Rows are independent up to the attention, so this is the
    # block oracle restricted to those rows.
    w = I.MHA_WORKLOADS["mha_b1n16384e4096h32_causal"]
    x = I.make_mha_inputs(w)
    out, lse = run_mha(w, x)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    E, H, d, N = w.E, w.H, w.E // w.H, w.N
    rows = np.array([0, 1, 127, 128, 4095, 8191, 12289, N - 1], dtype=np.int64)
    xf = oracle.bf16_to_f64(x.x)[0]
    wqkv = oracle.bf16_to_f64(x.w_qkv)
    kv = oracle.round_bf16(xf @ wqkv[:, E:])                                  # [N, 2E]
    q = oracle.round_bf16(xf[rows] @ wqkv[:, :E])                             # [R, E]
    heads = lambda t, n: np.ascontiguousarray(t.reshape(1, n, H, d).transpose(0, 2, 1, 3))  # noqa: E731
    k, v = heads(kv[:, :E], N), heads(kv[:, E:], N)
    # attention_rows wants the query tensor at full length: place the sampled
    # rows at their positions (other rows are not computed).
    qf = np.zeros((1, H, N, d))
    qf[:, :, rows] = heads(q, len(rows))
    O_ref, lse_ref = oracle.attention_rows(qf, k, v, 1.0 / np.sqrt(d), True, None, rows=rows)
    attn = oracle.round_bf16(O_ref.transpose(0, 2, 1, 3).reshape(1, len(rows), E))
    out_ref = attn @ oracle.bf16_to_f64(x.w_o)
    check(out[:, rows], lse[:, :, rows], out_ref, lse_ref, "long-context block, sampled rows")


def test_mha_long_context_projections_elementwise():
    # Both projection GEMMs of the long-context block at full size, every
    # element: the workspace holds the bf16 [B*N, 3E] Q/K/V rows (x W_qkv)
    # and, 256-byte aligned after them, the merged heads M; `out` is M W_o.
    # Each is compared with the fp64 product of the same bf16 operands.  The
    # GPU accumulates in fp32 in another order, so where the exact sum lies
    # within the fp32 error of a bf16 rounding midpoint (about 0.2 % of the
    # elements at K = 4096), or cancels to far below the terms' size, it may
    # round differently.
    import torch
    w = I.MHA_WORKLOADS["mha_b1n16384e4096h32_causal"]
    x = I.make_mha_inputs(w)
    tx, tw, to = to_dev(x.x), to_dev(x.w_qkv), to_dev(x.w_o)
    out = torch.empty((w.B, w.N, w.E), dtype=torch.bfloat16, device="cuda")
    nbytes = sdp.attn_mha_workspace_size(w.B, w.N, w.E)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    st = sdp.attn_mha_fwd(tx, tw, to, out, None, w.B, w.N, w.E, w.H, w.causal, None, ws, nbytes,
                          torch.cuda.current_stream())
    assert st == sdp.ATTN_OK, sdp.attn_status_str(st)
    assert sdp.attn_check_device(torch.cuda.current_stream()) == sdp.ATTN_OK
    rows, E = w.B * w.N, w.E
    qkv_bytes = (rows * 3 * E * 2 + 255) // 256 * 256
    qkv = ws[: rows * 3 * E * 2].view(torch.int16).cpu().numpy().view(np.uint16).reshape(rows, 3 * E)
    merged = ws[qkv_bytes: qkv_bytes + rows * E * 2].view(torch.int16).cpu().numpy().view(np.uint16).reshape(rows, E)
    got_out = out.view(torch.int16).cpu().numpy().view(np.uint16).reshape(rows, E)

    def check_gemm(a_bits, b_bits, got_bits, what):
        a, b = oracle.bf16_to_f64(a_bits), oracle.bf16_to_f64(b_bits)
        exact = a @ b
        got = oracle.bf16_to_f64(got_bits)
        # Bound per element: the bf16 rounding of the result (half a step,
        # 2^-9 relative, doubled for the GPU rounding its own fp32 value) plus
        # the fp32 accumulation error, which is a few 2^-24 sqrt(K) times the
        # size of the terms; 2^-18 |a_i| |b_j| (row and column norms, which
        # bound |sum_k a_ik b_kj| by Cauchy-Schwarz) covers it at K = 4096
        # while a dropped K step or a misplaced tile is orders larger.
        tau = 2.0 ** -18 * np.linalg.norm(a, axis=1)[:, None] * np.linalg.norm(b, axis=0)[None, :]
        err = np.abs(got - exact)
        bad = err > 2.0 ** -8 * np.abs(exact) + tau
        assert not bad.any(), "%s: %d elements off, worst %.3e (bound %.3e)" % (
            what, int(bad.sum()), float(err[bad].max()), float((2.0 ** -8 * np.abs(exact) + tau)[bad].max()))
        # Most elements are the correctly rounded value itself.
        frac = float((got != oracle.round_bf16(exact)).mean())
        assert frac < 1e-2, "%s: %.2e of the elements differ from the rounded exact product" % (what, frac)

    check_gemm(x.x.reshape(rows, E), x.w_qkv, qkv, "x W_qkv")
    check_gemm(merged, x.w_o, got_out, "M W_o")
