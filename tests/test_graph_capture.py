"""The forward, backward and decode calls can be recorded into a CUDA graph
and replayed: each call only encodes tensor maps on the host, launches
kernels on the given stream and allocates nothing, so a graph holding it
reproduces the direct call bit for bit on the same buffers.  (One direct
call per device comes first: it sets each kernel's shared-memory limit.)
Replaying many small calls from one graph is how latency-bound shapes are
meant to be driven."""
import numpy as np
import pytest

import scaled_dot_product_18_b300 as sdp
from scaled_dot_product_18_b300 import inputs as I

from gpu_util import to_dev, torch

pytestmark = pytest.mark.gpu


def _replay_matches(run, outputs):
    """run(stream) enqueues the call; outputs are the tensors it writes."""
    t = torch()
    s = t.cuda.Stream()
    with t.cuda.stream(s):
        assert run(s) == sdp.ATTN_OK
    s.synchronize()
    want = [o.clone() for o in outputs]
    for o in outputs:
        o.fill_(float("nan"))
    g = t.cuda.CUDAGraph()
    with t.cuda.graph(g, stream=s):
        assert run(s) == sdp.ATTN_OK
    for o in outputs:  # nothing ran during capture
        assert t.isnan(o.float()).all()
    for _ in range(3):
        g.replay()
    t.cuda.synchronize()
    assert sdp.attn_check_device(None) == sdp.ATTN_OK
    for o, w in zip(outputs, want):
        assert t.equal(o, w)


def test_forward_in_a_graph():
    t = torch()
    B, H, N, d = 2, 3, 300, 128
    q, k, v = (to_dev(I.make_tensor_bits(31, s, (B, H, N, d))) for s in (0, 1, 2))
    kl = t.from_numpy(np.array([200, 300], dtype=np.int32)).cuda()
    out = t.empty_like(q)
    lse = t.empty((B, H, N), dtype=t.float32, device="cuda")
    _replay_matches(lambda s: sdp.attn_fwd(q, k, v, out, lse, B, H, N, d, 0.1, 1, kl, s), [out, lse])
    _replay_matches(lambda s: sdp.attn_fwd_window(q, k, v, out, lse, B, H, N, d, 0.1, 1, kl, 64, s), [out, lse])


def test_backward_in_a_graph():
    t = torch()
    B, H, N, d = 1, 2, 257, 64
    q, k, v, g = (to_dev(I.make_tensor_bits(32, s, (B, H, N, d))) for s in (0, 1, 2, 4))
    out, lse = sdp.attention(q, k, v, causal=True)
    dq, dk, dv = t.empty_like(q), t.empty_like(q), t.empty_like(q)
    nb = sdp.attn_bwd_workspace_size(B, H, N, d)
    ws = t.empty(nb, dtype=t.uint8, device="cuda")
    # dq is summed with atomics in no fixed order, so only dk and dv are
    # compared bit for bit; dq is compared with a tolerance below.
    def run(s):
        return sdp.attn_bwd(q, k, v, out, g, lse, dq, dk, dv, B, H, N, d, d ** -0.5, 1, None, ws, nb, s)
    _replay_matches(run, [dk, dv])
    ref = dq.clone()
    t.cuda.synchronize()
    s = t.cuda.Stream()
    with t.cuda.stream(s):
        assert run(s) == sdp.ATTN_OK
    s.synchronize()
    assert float((dq.float() - ref.float()).abs().max()) <= 1e-2 * float(ref.float().abs().max())


def test_decode_in_a_graph():
    t = torch()
    B, H, L, d = 3, 4, 1000, 128
    q = to_dev(I.make_tensor_bits(33, 0, (B, H, d)))
    kc = to_dev(I.make_tensor_bits(33, 1, (B, H, L, d)))
    vc = to_dev(I.make_tensor_bits(33, 2, (B, H, L, d)))
    cl = t.from_numpy(np.array([1000, 17, 640], dtype=np.int32)).cuda()
    out = t.empty((B, H, d), dtype=t.bfloat16, device="cuda")
    lse = t.empty((B, H), dtype=t.float32, device="cuda")
    nb = sdp.attn_decode_workspace_size(B, H, L, d)
    ws = t.empty(nb, dtype=t.uint8, device="cuda")
    _replay_matches(lambda s: sdp.attn_decode(q, kc, vc, out, lse, B, H, L, d, 0.09, cl, ws, nb, s), [out, lse])
