"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs and compare it with the fp64 oracle."""
from __future__ import annotations

import numpy as np

import oracle
import scaled_dot_product_18_b300 as sdp

# Tolerances for bf16 inputs with fp32 accumulation and a bf16 output.
MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_ABS = 1e-3
GUARD = 4096  # elements past the end of each output that must stay untouched


def torch():
    import torch as t
    return t


def to_dev(bits: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(t.bfloat16)


def run_cuda(q_bits, k_bits, v_bits, scale, causal, key_lens=None, with_lse=True, stream=None, entry=None,
             out_offset=0):
    """Run attn_fwd via the C ABI.  Returns (O float64 [B,H,N,d], lse float64
    [B,H,N] or None).  Outputs live inside larger buffers pre-filled with a
    NaN canary; the guard zones around them are checked for stray writes.
    out_offset (elements) moves O off the allocator's alignment."""
    t = torch()
    B, H, N, d = q_bits.shape
    q, k, v = to_dev(q_bits), to_dev(k_bits), to_dev(v_bits)
    n_out = B * H * N * d
    out_alloc = t.full((out_offset + n_out + GUARD,), float("nan"), dtype=t.bfloat16, device="cuda")
    out_buf = out_alloc[out_offset:]
    lse_buf = t.full((B * H * N + GUARD,), float("nan"), dtype=t.float32, device="cuda")
    kl = t.from_numpy(np.asarray(key_lens, dtype=np.int32)).cuda() if key_lens is not None else None
    fn = entry or sdp.attn_fwd
    st = fn(q, k, v, out_buf, lse_buf if with_lse else None, B, H, N, d, scale, causal, kl,
            stream if stream is not None else t.cuda.current_stream())
    assert st == sdp.ATTN_OK, sdp.attn_status_str(st)
    assert sdp.attn_check_device(stream if stream is not None else t.cuda.current_stream()) == sdp.ATTN_OK
    tail = out_buf[n_out:].float()
    assert t.isnan(tail).all(), "stray write past the end of out"
    assert t.isnan(out_alloc[:out_offset].float()).all(), "stray write before out"
    O = out_buf[:n_out].float().cpu().numpy().astype(np.float64).reshape(B, H, N, d)
    lse = None
    if with_lse:
        assert t.isnan(lse_buf[B * H * N:]).all(), "stray write past the end of lse"
        lse = lse_buf[: B * H * N].cpu().numpy().astype(np.float64).reshape(B, H, N)
    else:
        assert t.isnan(lse_buf).all()
    return O, lse


def assert_close(O, lse, O_ref, lse_ref, what=""):
    assert not np.isnan(O).any(), "%s: unwritten (NaN canary) output rows" % what
    err = np.abs(O - O_ref)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(O_ref))
    rel = float(np.linalg.norm(O - O_ref)) / denom if denom > 0 else float(np.linalg.norm(O - O_ref))
    assert max_abs <= MAX_ABS, "%s: max-abs %.3e" % (what, max_abs)
    assert rel <= REL_L2, "%s: rel-L2 %.3e" % (what, rel)
    if lse is not None:
        assert not np.isnan(lse).any(), "%s: unwritten lse" % what
        fin = np.isfinite(lse_ref)
        np.testing.assert_array_equal(np.isneginf(lse), ~fin, err_msg=what + ": -inf lse rows differ")
        if fin.any():
            dl = float(np.abs(lse[fin] - lse_ref[fin]).max())
            assert dl <= LSE_ABS, "%s: |dlse| %.3e" % (what, dl)
    return max_abs, rel


def oracle_full(inp_q, inp_k, inp_v, scale, causal, key_lens=None):
    return oracle.attention_rows(inp_q, inp_k, inp_v, scale, causal, key_lens)
