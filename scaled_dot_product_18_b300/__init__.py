"""B300-native multi-head scaled dot-product attention forward.

Python binding of the C ABI in ``include/attn.h`` (library ``libattn.so``,
built in-tree by ``_build.build()``).  The functions with the C names only
marshal arguments -- tensors or integer device pointers, a torch stream or a
raw handle -- and return the C status; all of the computation runs in the
sm_103a kernel.  There is no fallback: if the library is missing or cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

from . import inputs  # noqa: F401  (seeded input generator)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn.so")

ATTN_OK = 0
ATTN_EINVAL = -1
ATTN_EUNSUPPORTED = -2
ATTN_EALIGN = -3
ATTN_ECUDA = -4
ATTN_EDEVICE = -5
ATTN_ETOOLARGE = -6

# Symbols declared in include/attn.h.
EXPORTS = ("attn_fwd", "attn_fwd_window", "attn_decode", "attn_decode_workspace_size", "attn_decode_noalloc",
           "attn_mha_fwd", "attn_mha_workspace_size", "attn_bwd", "attn_bwd_window", "attn_bwd_workspace_size", "attn_check_device",
           "attn_status_str", "attn_abi_version", "attn_tensor_map_cache_stats")

_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str = "attn_fwd"):
        super().__init__("%s failed: %s (%d)" % (what, attn_status_str(status), status))
        self.status = status


def load_library():
    """Load libattn.so (raises if it is missing: there is no other path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libattn.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
    _lib = bind(ctypes.CDLL(LIB_PATH))
    return _lib


def bind(lib):
    """Declare the argument and result types of every symbol of include/attn.h
    on a loaded copy of the library; returns it."""
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, i, vp, vp]
    lib.attn_fwd.restype = i
    lib.attn_fwd_window.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, i, vp, i, vp]
    lib.attn_fwd_window.restype = i
    lib.attn_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, vp, vp, ctypes.c_size_t, vp]
    lib.attn_decode.restype = i
    lib.attn_decode_workspace_size.argtypes = [i, i, i, i]
    lib.attn_decode_workspace_size.restype = ctypes.c_size_t
    lib.attn_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, vp, vp]
    lib.attn_decode_noalloc.restype = i
    lib.attn_mha_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, vp, vp, ctypes.c_size_t, vp]
    lib.attn_mha_fwd.restype = i
    lib.attn_mha_workspace_size.argtypes = [i, i, i]
    lib.attn_mha_workspace_size.restype = ctypes.c_size_t
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, i, vp, vp,
                             ctypes.c_size_t, vp]
    lib.attn_bwd.restype = i
    lib.attn_bwd_window.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, i, vp, i, vp,
                                    ctypes.c_size_t, vp]
    lib.attn_bwd_window.restype = i
    lib.attn_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.attn_bwd_workspace_size.restype = ctypes.c_size_t
    lib.attn_check_device.argtypes = [vp]
    lib.attn_check_device.restype = i
    lib.attn_status_str.argtypes = [i]
    lib.attn_status_str.restype = ctypes.c_char_p
    lib.attn_abi_version.argtypes = []
    lib.attn_abi_version.restype = i
    lib.attn_tensor_map_cache_stats.argtypes = [ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]
    lib.attn_tensor_map_cache_stats.restype = None
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream) if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def attn_fwd(q, k, v, out, lse, B: int, H: int, N: int, d: int, scale: float, causal,
             key_lens=None, stream=None) -> int:
    """The C ``attn_fwd``: pointers (tensors or ints), sizes, flags; returns the status."""
    lib = load_library()
    return lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(B), int(H), int(N), int(d),
                        float(scale), 1 if causal else 0, _ptr(key_lens), _stream(stream))


def attn_fwd_window(q, k, v, out, lse, B: int, H: int, N: int, d: int, scale: float, causal,
                    key_lens=None, window: int = 0, stream=None) -> int:
    """The C ``attn_fwd_window``: ``attn_fwd`` with a sliding window (keys j > i - window)."""
    lib = load_library()
    return lib.attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), int(B), int(H), int(N), int(d),
                               float(scale), 1 if causal else 0, _ptr(key_lens), int(window), _stream(stream))


def attn_decode(q, k_cache, v_cache, out, lse, B: int, H: int, L: int, d: int, scale: float, cache_lens=None,
                workspace=None, workspace_bytes: int = 0, stream=None) -> int:
    """The C ``attn_decode``: one query per (b, h) against a [B, H, L, d] cache."""
    lib = load_library()
    return lib.attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), int(B), int(H), int(L),
                           int(d), float(scale), _ptr(cache_lens), _ptr(workspace), int(workspace_bytes),
                           _stream(stream))


def attn_decode_noalloc(q, k_cache, v_cache, out, lse, B: int, H: int, L: int, d: int, scale: float,
                        cache_lens=None, stream=None) -> int:
    """The C ``attn_decode_noalloc``: ``attn_decode`` on the library's fixed
    per-device scratch array, for callers that cannot allocate."""
    lib = load_library()
    return lib.attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), int(B), int(H),
                                   int(L), int(d), float(scale), _ptr(cache_lens), _stream(stream))


def attn_decode_workspace_size(B: int, H: int, L: int, d: int) -> int:
    return int(load_library().attn_decode_workspace_size(int(B), int(H), int(L), int(d)))


def decode(q, k_cache, v_cache, cache_lens=None, scale: float | None = None, stream=None, out=None, lse=None,
           workspace=None):
    """Convenience wrapper over ``attn_decode`` for torch tensors: q [B, H, d],
    caches [B, H, L, d] (bf16, CUDA, contiguous).  Allocates out, lse and the
    workspace with torch when not given; raises ``AttnError`` on failure."""
    import torch
    B, H, L, d = k_cache.shape
    if out is None:
        out = torch.empty((B, H, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    nbytes = attn_decode_workspace_size(B, H, max(L, 1), d)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = attn_decode(q, k_cache, v_cache, out, lse, B, H, L, d, scale, cache_lens, workspace,
                     workspace.numel() * workspace.element_size(), stream)
    if st != ATTN_OK:
        raise AttnError(st, "attn_decode")
    return out, lse


def attn_mha_fwd(x, w_qkv, w_o, out, lse, B: int, N: int, E: int, H: int, causal, key_lens=None,
                 workspace=None, workspace_bytes: int = 0, stream=None) -> int:
    """The C ``attn_mha_fwd``: projections, heads, attention, output projection."""
    lib = load_library()
    return lib.attn_mha_fwd(_ptr(x), _ptr(w_qkv), _ptr(w_o), _ptr(out), _ptr(lse), int(B), int(N), int(E), int(H),
                            1 if causal else 0, _ptr(key_lens), _ptr(workspace), int(workspace_bytes),
                            _stream(stream))


def attn_mha_workspace_size(B: int, N: int, E: int) -> int:
    return int(load_library().attn_mha_workspace_size(int(B), int(N), int(E)))


def attn_bwd(q, k, v, out, dout, lse, dq, dk, dv, B: int, H: int, N: int, d: int, scale: float, causal,
             key_lens=None, workspace=None, workspace_bytes: int = 0, stream=None) -> int:
    """The C ``attn_bwd``: dQ, dK, dV of the attention forward."""
    lib = load_library()
    return lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                        int(B), int(H), int(N), int(d), float(scale), 1 if causal else 0, _ptr(key_lens),
                        _ptr(workspace), int(workspace_bytes), _stream(stream))


def attn_bwd_window(q, k, v, out, dout, lse, dq, dk, dv, B: int, H: int, N: int, d: int, scale: float, causal,
                    key_lens=None, window: int = 0, workspace=None, workspace_bytes: int = 0, stream=None) -> int:
    """The C ``attn_bwd_window``: the backward of the sliding-window forward."""
    lib = load_library()
    return lib.attn_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                               _ptr(dv), int(B), int(H), int(N), int(d), float(scale), 1 if causal else 0,
                               _ptr(key_lens), int(window), _ptr(workspace), int(workspace_bytes), _stream(stream))


def attn_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().attn_bwd_workspace_size(int(B), int(H), int(N), int(d)))


def attention_backward(q, k, v, out, lse, dout, causal: bool = False, key_lens=None, scale: float | None = None,
                       stream=None, workspace=None, window: int = 0):
    """Convenience wrapper over ``attn_bwd`` (``attn_bwd_window`` when window >
    0) for torch tensors of the forward's layout; allocates dq, dk, dv (and the
    workspace when not given) with torch and raises ``AttnError`` on a non-OK
    status.  Returns (dq, dk, dv)."""
    import torch
    B, H, N, d = q.shape
    for t in (q, k, v, out, dout):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (B, H, N, d):
            raise ValueError("q, k, v, out, dout must be contiguous bf16 CUDA tensors of one shape [B, H, N, d]")
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [B, H, N]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = attn_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nbytes = workspace.numel() * workspace.element_size()
    if window:
        st = attn_bwd_window(q, k, v, out, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, key_lens, window,
                             workspace, nbytes, stream)
    else:
        st = attn_bwd(q, k, v, out, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, key_lens, workspace, nbytes,
                      stream)
    if st != ATTN_OK:
        raise AttnError(st, "attn_bwd")
    return dq, dk, dv


def attn_check_device(stream=None) -> int:
    return load_library().attn_check_device(_stream(stream))


def attn_status_str(status: int) -> str:
    return load_library().attn_status_str(int(status)).decode()


def attn_abi_version() -> int:
    return load_library().attn_abi_version()


def attn_tensor_map_cache_stats() -> tuple[int, int]:
    """(hits, misses) of the library's tensor-map cache since it was loaded."""
    h, m = ctypes.c_uint64(0), ctypes.c_uint64(0)
    load_library().attn_tensor_map_cache_stats(ctypes.byref(h), ctypes.byref(m))
    return int(h.value), int(m.value)


def attention(q, k, v, causal: bool = False, key_lens=None, scale: float | None = None, stream=None,
              out=None, lse=None, window: int = 0):
    """Convenience wrapper over ``attn_fwd`` for torch tensors.

    q, k, v: bf16 CUDA tensors [B, H, N, d], contiguous.  key_lens: int32 CUDA
    tensor [B] or None.  window > 0: sliding window (keys j > i - window).  Allocates ``out`` (bf16) and ``lse`` (fp32) with
    torch when not given, raises ``AttnError`` on a non-OK status.
    """
    import torch
    B, H, N, d = q.shape
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != (B, H, N, d):
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors of one shape [B, H, N, d]")
    if key_lens is not None and (key_lens.dtype != torch.int32 or not key_lens.is_cuda or key_lens.numel() != B):
        raise ValueError("key_lens must be an int32 CUDA tensor of B elements")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if window:
        st = attn_fwd_window(q, k, v, out, lse, B, H, N, d, scale, causal, key_lens, window, stream)
    else:
        st = attn_fwd(q, k, v, out, lse, B, H, N, d, scale, causal, key_lens, stream)
    if st != ATTN_OK:
        raise AttnError(st)
    return out, lse
