"""The library's tensor-map cache: a call whose buffers, sizes and strides
were seen before reuses the encoded maps; a changed input address is a miss,
and the results do not depend on whether a map came from the cache."""
import numpy as np
import pytest

import scaled_dot_product_18_b300 as sdp
from scaled_dot_product_18_b300 import inputs as I


def test_stats_are_readable_without_a_gpu():
    hits, misses = sdp.attn_tensor_map_cache_stats()
    assert hits >= 0 and misses >= 0


@pytest.mark.gpu
def test_reused_buffers_hit_and_a_new_pointer_misses():
    import torch
    from gpu_util import to_dev

    torch.cuda.set_device(0)
    B, H, N, d = 1, 3, 300, 64
    q, k, v = (to_dev(I.make_tensor_bits(71, s, (B, H, N, d))) for s in (0, 1, 2))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    scale = 1.0 / np.sqrt(d)

    def call(qq, o):
        st = sdp.attn_fwd(qq, k, v, o, lse, B, H, N, d, scale, True)
        assert st == sdp.ATTN_OK, sdp.attn_status_str(st)

    call(q, out)  # the maps of these buffers are now in the table
    h0, m0 = sdp.attn_tensor_map_cache_stats()
    call(q, out)
    h1, m1 = sdp.attn_tensor_map_cache_stats()
    per_call = h1 - h0  # one map per tensor the call reads or writes through TMA
    assert per_call >= 3 and m1 == m0
    first = out.clone()
    q2 = q.clone()  # a different address: one new map, the others reused
    call(q2, out)
    h2, m2 = sdp.attn_tensor_map_cache_stats()
    assert (h2 - h1, m2 - m1) == (per_call - 1, 1)
    assert sdp.attn_check_device() == sdp.ATTN_OK
    assert torch.equal(first, out)  # same inputs through a freshly encoded map
