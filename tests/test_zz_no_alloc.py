"""attn_decode_noalloc: the decode entry point for callers that cannot
allocate device memory while running (it uses a fixed scratch array inside
the library instead of a caller workspace).  Its results must match
attn_decode's on the same inputs, on two calls in a row, and problems larger
than its fixed scratch area must be refused before anything runs.

This file is collected last, so a run that stops at its first failure has
already run every other test."""
import numpy as np
import pytest

import scaled_dot_product_18_b300 as sdp
from scaled_dot_product_18_b300 import inputs as I


def test_no_alloc_rejects_problems_beyond_its_scratch():
    # 40,000 (batch, head) pairs need ~20 MB of partials, more than the 8 MiB
    # area; refused on the host, before any CUDA call (fake pointers).
    P = 1 << 20
    sdp.load_library()
    st = sdp.attn_decode_noalloc(P, P, P, P, None, 40000, 1, 4096, 128, 0.1, None, None)
    assert st == sdp.ATTN_ETOOLARGE
    assert "scratch" in sdp.attn_status_str(st)


@pytest.mark.parametrize("args,want", [
    (dict(scale=float("nan")), sdp.ATTN_EINVAL),
    (dict(scale=0.0), sdp.ATTN_EINVAL),
    (dict(q=None), sdp.ATTN_EINVAL),
    (dict(out=None), sdp.ATTN_EINVAL),
    (dict(k=None), sdp.ATTN_EINVAL),
    (dict(d=96), sdp.ATTN_EUNSUPPORTED),
    (dict(B=-1), sdp.ATTN_EINVAL),
])
def test_no_alloc_checks_arguments_before_the_size(args, want):
    # A problem far too large for the fixed area (40,000 heads) with one bad
    # argument gets the same status as attn_decode gives for that argument,
    # not ATTN_ETOOLARGE; both are decided on the host (fake pointers).
    P = 1 << 20
    sdp.load_library()
    a = dict(q=P, k=P, v=P, out=P, lse=None, B=40000, H=1, L=4096, d=128, scale=0.1, cl=None)
    a.update(args)
    order = ("q", "k", "v", "out", "lse", "B", "H", "L", "d", "scale", "cl")
    st = sdp.attn_decode_noalloc(*(a[n] for n in order), None)
    assert st == want, sdp.attn_status_str(st)
    ws = sdp.attn_decode(*(a[n] for n in order), P, 1 << 30, None)
    assert ws == want, sdp.attn_status_str(ws)


@pytest.mark.gpu
def test_no_alloc_matches_attn_decode_twice():
    import torch
    from gpu_util import LSE_ABS, MAX_ABS, to_dev

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    for call, (B, H, L, d, seed) in enumerate([(4, 32, 3000, 128, 61), (3, 7, 777, 64, 62)]):
        q = to_dev(I.make_tensor_bits(seed, 0, (B, H, d)))
        k = to_dev(I.make_tensor_bits(seed, 1, (B, H, L, d)))
        v = to_dev(I.make_tensor_bits(seed, 2, (B, H, L, d)))
        cl = torch.from_numpy(np.array(([L, L // 2, 1, 0] * B)[:B], dtype=np.int32)).cuda()
        scale = 1.0 / np.sqrt(d)
        outs = []
        for noalloc in (False, True):
            out = torch.full((B, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
            lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
            if noalloc:
                st = sdp.attn_decode_noalloc(q, k, v, out, lse, B, H, L, d, scale, cl, stream)
            else:
                nbytes = sdp.attn_decode_workspace_size(B, H, L, d)
                ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
                st = sdp.attn_decode(q, k, v, out, lse, B, H, L, d, scale, cl, ws, nbytes, stream)
            assert st == sdp.ATTN_OK, sdp.attn_status_str(st)
            assert sdp.attn_check_device(stream) == sdp.ATTN_OK
            outs.append((out.float().cpu().numpy(), lse.cpu().numpy()))
        (O_ref, l_ref), (O, l) = outs
        assert not np.isnan(O).any() and not np.isnan(l).any(), "call %d: unwritten output" % call
        assert float(np.abs(O - O_ref).max()) <= MAX_ABS, "call %d" % call
        np.testing.assert_array_equal(np.isneginf(l), np.isneginf(l_ref))
        fin = np.isfinite(l_ref)
        assert float(np.abs(l[fin] - l_ref[fin]).max()) <= LSE_ABS, "call %d" % call
