"""The C-ABI library: it loads without a GPU, exports what include/attn.h
declares, and rejects bad arguments on the host before touching CUDA."""
import os
import re

import pytest

import scaled_dot_product_18_b300 as sdp
from scaled_dot_product_18_b300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sdp.load_library()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", txt, flags=re.M))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"attn_fwd", "attn_fwd_window", "attn_decode", "attn_decode_workspace_size", "attn_mha_fwd",
            "attn_mha_workspace_size", "attn_bwd", "attn_bwd_window", "attn_bwd_workspace_size", "attn_check_device",
            "attn_status_str",
            "attn_abi_version", "attn_tensor_map_cache_stats"} <= names
    assert names == set(sdp.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_status_strings(lib):
    assert sdp.attn_abi_version() == 6
    for code in (0, -1, -2, -3, -4, -5):
        assert sdp.attn_status_str(code).startswith("ATTN_")
    assert sdp.attn_status_str(7) == "unknown attn_status"


# Arguments the host can reject without any CUDA call (pointers are fake
# integers; nothing is dereferenced on these paths).
P = 1 << 20  # a 16-byte aligned fake address


@pytest.mark.parametrize("args,want", [
    (dict(d=96), sdp.ATTN_EUNSUPPORTED),
    (dict(d=32), sdp.ATTN_EUNSUPPORTED),
    (dict(B=-1), sdp.ATTN_EINVAL),
    (dict(H=-2), sdp.ATTN_EINVAL),
    (dict(N=-3), sdp.ATTN_EINVAL),
    (dict(scale=0.0), sdp.ATTN_EINVAL),
    (dict(scale=-0.125), sdp.ATTN_EINVAL),
    (dict(scale=float("nan")), sdp.ATTN_EINVAL),
    (dict(scale=float("inf")), sdp.ATTN_EINVAL),
    (dict(q=None), sdp.ATTN_EINVAL),
    (dict(k=None), sdp.ATTN_EINVAL),
    (dict(v=None), sdp.ATTN_EINVAL),
    (dict(out=None), sdp.ATTN_EINVAL),
    (dict(q=P + 8), sdp.ATTN_EALIGN),
    (dict(k=P + 2), sdp.ATTN_EALIGN),
    (dict(v=P + 1), sdp.ATTN_EALIGN),
    (dict(out=P + 4), sdp.ATTN_EALIGN),
    (dict(lse=P + 2), sdp.ATTN_EALIGN),
    (dict(key_lens=P + 1), sdp.ATTN_EALIGN),
    (dict(B=1 << 16, H=1 << 15), sdp.ATTN_EINVAL),          # B*H >= 2^31
    (dict(B=1 << 12, H=1 << 12, N=1 << 20), sdp.ATTN_EINVAL),  # tile grid >= 2^31
    (dict(B=0, q=None, k=None, v=None, out=None), sdp.ATTN_OK),  # empty: no-op
    (dict(N=0), sdp.ATTN_OK),
    (dict(H=0, d=128), sdp.ATTN_OK),
])
def test_host_side_rejections(lib, args, want):
    a = dict(q=P, k=P, v=P, out=P, lse=None, B=2, H=3, N=5, d=64, scale=0.125, causal=0,
             key_lens=None, stream=None)
    a.update(args)
    st = lib.attn_fwd(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"], a["H"], a["N"], a["d"],
                      a["scale"], a["causal"], a["key_lens"], a["stream"])
    assert st == want, (args, st)


@pytest.mark.parametrize("window,want", [(-1, sdp.ATTN_EINVAL), (-100, sdp.ATTN_EINVAL)])
def test_window_rejections(lib, window, want):
    st = lib.attn_fwd_window(P, P, P, P, None, 2, 3, 5, 64, 0.125, 1, None, window, None)
    assert st == want


def test_window_empty_problem_is_ok(lib):
    assert lib.attn_fwd_window(None, None, None, None, None, 0, 3, 5, 64, 0.125, 1, None, 7, None) == sdp.ATTN_OK


def test_decode_workspace_size(lib):
    n = sdp.attn_decode_workspace_size(4, 32, 16384, 128)
    assert n > 0 and n % 4 == 0
    assert sdp.attn_decode_workspace_size(4, 32, 16384, 96) == 0
    assert sdp.attn_decode_workspace_size(0, 32, 16384, 128) == 0
    # more splits per head when there are few heads, never more than one per 256 keys
    assert sdp.attn_decode_workspace_size(1, 1, 256, 64) == (256 + 4)  # one split: 64 floats (256 B) + 1 lse
    assert sdp.attn_decode_workspace_size(1, 1, 100000, 128) > sdp.attn_decode_workspace_size(64, 1, 100000, 128) / 64


@pytest.mark.parametrize("args,want", [
    (dict(d=96), sdp.ATTN_EUNSUPPORTED),
    (dict(B=-1), sdp.ATTN_EINVAL),
    (dict(L=-1), sdp.ATTN_EINVAL),
    (dict(scale=0.0), sdp.ATTN_EINVAL),
    (dict(q=None), sdp.ATTN_EINVAL),
    (dict(out=None), sdp.ATTN_EINVAL),
    (dict(k=None), sdp.ATTN_EINVAL),
    (dict(ws=None), sdp.ATTN_EINVAL),
    (dict(ws_bytes=16), sdp.ATTN_EINVAL),
    (dict(q=P + 8), sdp.ATTN_EALIGN),
    (dict(v=P + 4), sdp.ATTN_EALIGN),
    (dict(ws=P + 8), sdp.ATTN_EALIGN),
    (dict(B=0, q=None, out=None, ws=None), sdp.ATTN_OK),
])
def test_decode_host_side_rejections(lib, args, want):
    a = dict(q=P, k=P, v=P, out=P, lse=None, B=2, H=3, L=1000, d=128, scale=0.1, cl=None, ws=P,
             ws_bytes=1 << 30, stream=None)
    a.update(args)
    st = lib.attn_decode(a["q"], a["k"], a["v"], a["out"], a["lse"], a["B"], a["H"], a["L"], a["d"], a["scale"],
                         a["cl"], a["ws"], a["ws_bytes"], a["stream"])
    assert st == want, (args, st)


@pytest.mark.parametrize("args,want", [
    (dict(E=96, H=1), sdp.ATTN_EUNSUPPORTED),   # d = 96
    (dict(E=512, H=3), sdp.ATTN_EINVAL),        # E % H != 0
    (dict(H=0), sdp.ATTN_EINVAL),
    (dict(B=-1), sdp.ATTN_EINVAL),
    (dict(x=None), sdp.ATTN_EINVAL),
    (dict(wo=None), sdp.ATTN_EINVAL),
    (dict(ws=None), sdp.ATTN_EINVAL),
    (dict(ws_bytes=1024), sdp.ATTN_EINVAL),
    (dict(x=P + 2), sdp.ATTN_EALIGN),
    (dict(out=P + 8), sdp.ATTN_EALIGN),
    (dict(B=0, x=None, ws=None), sdp.ATTN_OK),
])
def test_mha_host_side_rejections(lib, args, want):
    a = dict(x=P, wqkv=P, wo=P, out=P, lse=None, B=2, N=100, E=512, H=8, causal=0, kl=None, ws=P,
             ws_bytes=1 << 40, stream=None)
    a.update(args)
    st = lib.attn_mha_fwd(a["x"], a["wqkv"], a["wo"], a["out"], a["lse"], a["B"], a["N"], a["E"], a["H"],
                          a["causal"], a["kl"], a["ws"], a["ws_bytes"], a["stream"])
    assert st == want, (args, st)


def test_mha_workspace_size(lib):
    n = sdp.attn_mha_workspace_size(2, 100, 512)
    assert n >= 2 * 100 * 512 * 2 * 4 and sdp.attn_mha_workspace_size(0, 100, 512) == 0


def test_binding_raises_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(sdp, "_lib", None)
    monkeypatch.setattr(sdp, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        sdp.load_library()


def test_oracle_not_imported_by_product():
    # the product package never reaches into the oracle (test infrastructure)
    pkg = os.path.join(ROOT, "scaled_dot_product_18_b300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, fn
                assert "attn_oracle" not in txt, fn


def test_bwd_workspace_size(lib):
    # fp32 dQ accumulator, then two fp32 values (lse*log2e, D) per query row
    # padded to a multiple of 128; each part rounded up to 256 bytes
    assert sdp.attn_bwd_workspace_size(2, 3, 5, 64) == 2 * 3 * 5 * 64 * 4 + 2 * 6 * 128 * 4
    assert sdp.attn_bwd_workspace_size(1, 32, 16384, 128) == 32 * 16384 * (128 + 2) * 4
    assert sdp.attn_bwd_workspace_size(1, 1, 8, 96) == 0
    assert sdp.attn_bwd_workspace_size(0, 1, 8, 64) == 0


@pytest.mark.parametrize("args,want", [
    (dict(d=96), sdp.ATTN_EUNSUPPORTED),
    (dict(B=-1), sdp.ATTN_EINVAL),
    (dict(N=-1), sdp.ATTN_EINVAL),
    (dict(scale=0.0), sdp.ATTN_EINVAL),
    (dict(scale=float("nan")), sdp.ATTN_EINVAL),
    (dict(q=None), sdp.ATTN_EINVAL),
    (dict(out=None), sdp.ATTN_EINVAL),
    (dict(dout=None), sdp.ATTN_EINVAL),
    (dict(lse=None), sdp.ATTN_EINVAL),
    (dict(dq=None), sdp.ATTN_EINVAL),
    (dict(dv=None), sdp.ATTN_EINVAL),
    (dict(ws=None), sdp.ATTN_EINVAL),
    (dict(ws_bytes=64), sdp.ATTN_EINVAL),
    (dict(k=P + 8), sdp.ATTN_EALIGN),
    (dict(dout=P + 2), sdp.ATTN_EALIGN),
    (dict(dk=P + 4), sdp.ATTN_EALIGN),
    (dict(lse=P + 2), sdp.ATTN_EALIGN),
    (dict(ws=P + 8), sdp.ATTN_EALIGN),
    (dict(key_lens=P + 1), sdp.ATTN_EALIGN),
    (dict(B=1 << 16, H=1 << 15), sdp.ATTN_EINVAL),
    (dict(B=0, q=None, ws=None), sdp.ATTN_OK),
    (dict(N=0), sdp.ATTN_OK),
])
def test_bwd_host_side_rejections(lib, args, want):
    a = dict(q=P, k=P, v=P, out=P, dout=P, lse=P, dq=P, dk=P, dv=P, B=2, H=3, N=5, d=64, scale=0.125, causal=1,
             key_lens=None, ws=P, ws_bytes=1 << 30, stream=None)
    a.update(args)
    st = lib.attn_bwd(a["q"], a["k"], a["v"], a["out"], a["dout"], a["lse"], a["dq"], a["dk"], a["dv"], a["B"],
                      a["H"], a["N"], a["d"], a["scale"], a["causal"], a["key_lens"], a["ws"], a["ws_bytes"],
                      a["stream"])
    assert st == want, (args, st)


@pytest.mark.parametrize("window,want", [(-1, sdp.ATTN_EINVAL), (-7, sdp.ATTN_EINVAL)])
def test_bwd_window_rejections(lib, window, want):
    st = lib.attn_bwd_window(P, P, P, P, P, P, P, P, P, 2, 3, 5, 64, 0.125, 1, None, window, P, 1 << 30, None)
    assert st == want


def test_bwd_window_host_checks_match_attn_bwd(lib):
    # same argument checks as attn_bwd (window 0 = none)
    assert lib.attn_bwd_window(P, P, P, P, P, P, P, P, P, 2, 3, 5, 96, 0.125, 1, None, 4, P, 1 << 30,
                               None) == sdp.ATTN_EUNSUPPORTED
    assert lib.attn_bwd_window(P, P, P, P, P, None, P, P, P, 2, 3, 5, 64, 0.125, 1, None, 4, P, 1 << 30,
                               None) == sdp.ATTN_EINVAL
    assert lib.attn_bwd_window(None, None, None, None, None, None, None, None, None, 0, 3, 5, 64, 0.125, 1, None, 4,
                               None, 0, None) == sdp.ATTN_OK
