"""A bounded device wait that runs out: the forward's wind-down path.

Every mbarrier wait in the kernels gives up after a time limit: it raises the
CTA's abort flag, records the error (and the site of the first wait that ran
out) in the library's device error word, and the CTA waits -- again with a
limit -- for its own copies and MMAs, frees its tensor memory and returns
without storing output.

The product library never stalls on purpose.  The test library
(libattn_waittest.so: the same sources built with SDP18_WAIT_TEST, which
shortens the limit to 5 ms and adds a hook that makes the forward's TMA
producer stop issuing K/V copies from a given ring item on) lets this test
make the MMA warp's wait for the next K/V tile run out.  Nothing faults, traps
or hangs: the wait ends by its own limit and the context stays usable, which
the test checks by running a normal call on the same device and library
afterwards and comparing it with the oracle.
"""
import ctypes
import time

import numpy as np
import pytest

import scaled_dot_product_18_b300 as sdp
from scaled_dot_product_18_b300 import _build
from scaled_dot_product_18_b300 import inputs as I

# Wait sites of the forward kernel (the number stored in bits 8.. of the
# error word): 4 / 7 = the MMA warp waiting for a V / K tile (at d = 64 it
# waits for K_{j+1} before V_j, so with the producer stopped before V1 its
# wait for K2 is the one that runs out), 10/11 = the softmax warps of tile
# 0/1 waiting for their next score tile.  The waits start within about a
# microsecond of each other; which limit expires first depends on the
# global timer's granularity.
SITES_ACCEPTED = {4, 7, 10, 11}


def test_test_library_is_a_separate_build():
    # The stall hook exists only in the test library: the product library
    # exports no test symbol.
    import os
    lib = sdp.load_library()
    assert not hasattr(lib, "attn_test_set_stall")
    assert os.path.basename(_build.WAIT_TEST_LIB) != os.path.basename(sdp.LIB_PATH)


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_a_stalled_producer_makes_the_wait_run_out_and_the_next_call_is_clean(d):
    import torch
    from gpu_util import assert_close, oracle_full, to_dev

    lib = sdp.bind(ctypes.CDLL(_build.build_wait_test()))
    lib.attn_test_set_stall.argtypes = [ctypes.c_int]
    lib.attn_test_set_stall.restype = ctypes.c_int
    lib.attn_test_error_word.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.attn_test_error_word.restype = ctypes.c_int

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    sh = stream.cuda_stream
    # 2 heads x 2 query pairs = 4 work items, each streaming 4 key tiles = 8
    # ring items (K0, V0, K1, V1, ...); the producer stops before item 3 (V1).
    # d = 64 and d = 128 run different MMA orders (P in its own TMEM columns
    # or over the scores).
    B, H, N = 1, 2, 512
    qb, kb, vb = (I.make_tensor_bits(83, s, (B, H, N, d)) for s in (0, 1, 2))
    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    scale = 1.0 / np.sqrt(d)

    def call():
        out = torch.full((B, H, N, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        st = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, d,
                          scale, 0, None, sh)
        assert st == sdp.ATTN_OK
        return out, lse

    word = ctypes.c_int(0)
    assert lib.attn_check_device(sh) == sdp.ATTN_OK  # clear anything left over
    assert lib.attn_test_set_stall(3) == 0
    try:
        t0 = time.perf_counter()
        out, lse = call()
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        assert lib.attn_test_set_stall(-1) == 0
    assert lib.attn_test_error_word(ctypes.byref(word)) == 0
    w = word.value
    assert w & 0xFF == 1, "timeout flag not set: %#x" % w
    assert (w >> 8) in SITES_ACCEPTED, "first site %d" % (w >> 8)
    # The CTAs gave up after the test library's 5 ms limit, far below the
    # product's 1 s, and stored nothing.
    assert 0.004 < elapsed < 0.9, elapsed
    assert torch.isnan(out.float()).all() and torch.isnan(lse).all()
    # attn_check_device reports the error once and clears the word.
    assert lib.attn_check_device(sh) == sdp.ATTN_EDEVICE
    assert lib.attn_test_error_word(ctypes.byref(word)) == 0 and word.value == 0
    assert lib.attn_check_device(sh) == sdp.ATTN_OK

    # The next call on the same device and library runs normally.
    out, lse = call()
    assert lib.attn_check_device(sh) == sdp.ATTN_OK
    O = out.float().cpu().numpy().astype(np.float64)
    L = lse.cpu().numpy().astype(np.float64)
    O_ref, L_ref = oracle_full(qb, kb, vb, scale, False)
    assert_close(O, L, O_ref, L_ref, "after the timeout, d=%d" % d)
