"""fp64 CPU oracle for the attention forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  It shares no code with the CUDA path
(``scaled_dot_product_18_b300``) and never imports it; the two meet only in the
tests' comparisons, on inputs drawn by the seeded generator.

Two independent implementations of the same definition:

* ``attention_rows`` -- plain C (``attn_oracle.c``), float64, one query row at a
  time with a two-pass max-shifted softmax, threaded over rows.  Used for
  parity at every size (on sampled rows at the large ones) and as the timed
  CPU baseline.
* ``attention_literal`` -- numpy float64, materialises the full score matrix,
  applies the mask by filling with -inf, takes the softmax along the key axis
  and multiplies by V, in the order the pages' reference snippets write it
  (hotelren.com "AI attention: essence and evolution", ch.1 code and sec. 2.1;
  qqiyuan.cn "Multi-head attention in the Transformer: implementation and
  performance", baseline implementation).  Tiny inputs only.

Every function is pinned by ``tests/test_oracle.py`` against closed forms,
invariants and hand-derived fixtures (``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no fast-math: sums stay in key order)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        f = lib.oracle_attn_fwd
        dp = ctypes.POINTER(ctypes.c_double)
        f.argtypes = [dp, dp, dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                      ctypes.c_double, ctypes.c_int, ctypes.c_int64, ctypes.POINTER(ctypes.c_int32),
                      ctypes.POINTER(ctypes.c_int64), ctypes.c_int64, dp, dp, ctypes.c_int]
        f.restype = ctypes.c_int
        _lib = lib
    return _lib


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact decode of bfloat16 bit patterns (uint16) to float64."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def _as_f64(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        x = bf16_to_f64(x)
    return np.ascontiguousarray(x, dtype=np.float64)


def default_threads() -> int:
    return os.cpu_count() or 1


def attention_rows(q, k, v, scale: float, causal: bool, key_lens=None, rows=None,
                   threads: int | None = None, window: int = 0):
    """Row-mode oracle.  q: [B, H, Nq, d]; k, v: [B, H, Nk, d] (float64, or
    uint16 bf16 bits).  Query and key positions share one axis from 0, so the
    causal rule is j <= i; self-attention has Nq == Nk.

    key_lens: int [B] or None (all keys visible).  rows: query indices to
    compute (the same for every (b, h)) or None for all.  window: if > 0,
    query i sees only keys j > i - window (a sliding window of the last
    ``window`` positions; aicoding.csdn.net sec. 4.3).  Returns
    ``(O, lse)`` as float64 arrays [B, H, R, d] and [B, H, R].
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    assert k.shape == (B, H, Nk, d) and v.shape == k.shape
    if rows is None:
        rows_arr, n_rows = None, Nq
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n_rows = rows_arr.size
    out = np.zeros((B, H, n_rows, d), dtype=np.float64)
    lse = np.zeros((B, H, n_rows), dtype=np.float64)
    kl = None
    if key_lens is not None:
        kl = np.ascontiguousarray(np.asarray(key_lens, dtype=np.int32))
        assert kl.shape == (B,)
    dp = ctypes.POINTER(ctypes.c_double)
    lib = _load()
    rc = lib.oracle_attn_fwd(
        q.ctypes.data_as(dp), k.ctypes.data_as(dp), v.ctypes.data_as(dp), B, H, Nq, Nk, d,
        float(scale), int(bool(causal)), int(window),
        kl.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if kl is not None else None,
        rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if rows_arr is not None else None,
        n_rows, out.ctypes.data_as(dp), lse.ctypes.data_as(dp),
        int(threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_attn_fwd rejected its arguments (rc=%d)" % rc)
    return out, lse


def visible_mask(N: int, causal: bool, key_len: int | None, window: int = 0) -> np.ndarray:
    """[N, N] boolean: key j visible to query i (j < key_len, j <= i if causal,
    j > i - window if window > 0)."""
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    keep = np.ones((N, N), dtype=bool)
    if key_len is not None:
        keep &= j < key_len
    if causal:
        keep &= j <= i
    if window > 0:
        keep &= j > i - window
    return keep


def attention_literal(q, k, v, scale: float, causal: bool, key_lens=None, window: int = 0):
    """Materialised-matrix oracle: returns ``(O, lse, P)``, all float64.

    S = scale * Q K^T; S[~visible] = -inf; P = softmax(S) along keys; O = P V;
    lse = max + ln(sum exp(S - max)).  A row with no visible key gets P = 0,
    O = 0 and lse = -inf (instead of the NaN a literal -inf fill would give).
    """
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, N, d = q.shape
    S = scale * np.matmul(q, np.swapaxes(k, -1, -2))  # [B, H, N, N]
    keep = np.stack([visible_mask(N, causal, None if key_lens is None else int(key_lens[b]), window)
                     for b in range(B)])[:, None]  # [B, 1, N, N]
    S = np.where(keep, S, -np.inf)
    m = S.max(axis=-1, keepdims=True)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    E = np.where(keep, np.exp(S - m_safe), 0.0)
    l = E.sum(axis=-1, keepdims=True)
    P = np.where(empty, 0.0, E / np.where(empty, 1.0, l))
    O = np.matmul(P, v)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, l)))[..., 0]
    return O, lse, P


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), returned
    as float64.  Done on the float64 bit pattern (one rounding): keep the
    sign, the 11 exponent bits and the top 7 fraction bits.  Finite values
    in the normal float32 range only (true for every tensor it sees here)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    bits = x.view(np.uint64)
    keep = np.uint64(45)  # 52 - 7 fraction bits dropped
    half = np.uint64(1) << (keep - np.uint64(1))
    lsb = (bits >> keep) & np.uint64(1)
    r = (bits + (half - np.uint64(1)) + lsb) & ~((np.uint64(1) << keep) - np.uint64(1))
    return r.view(np.float64)


def mha_block(x, w_qkv, w_o, H: int, causal: bool, key_lens=None, threads: int | None = None):
    """Multi-head self-attention block without biases (cnnetsun.cn
    "Transformer QKV bottlenecks on long sequences", sec. 2, MinimalSelfAttention:
    Q/K/V projections, split into heads, scaled dot-product attention, merge
    heads, output projection; qqiyuan.cn's variant fuses the three projections
    into one [E, 3E] matrix, as here).

    x: [B, N, E]; w_qkv: [E, 3E] with Q, K, V columns in that order; w_o:
    [E, E].  Q/K/V and the merged attention output are bf16 tensors in the
    method (rounded to nearest even here, at the same two points); everything
    else is float64.  Returns (out [B, N, E], lse [B, H, N]).
    """
    x, w_qkv, w_o = _as_f64(x), _as_f64(w_qkv), _as_f64(w_o)
    B, N, E = x.shape
    d = E // H
    qkv = round_bf16(np.matmul(x, w_qkv))                        # [B, N, 3E]
    heads = lambda t: t.reshape(B, N, H, d).transpose(0, 2, 1, 3)  # noqa: E731  [B, H, N, d]
    q = np.ascontiguousarray(heads(qkv[..., :E]))
    k = np.ascontiguousarray(heads(qkv[..., E:2 * E]))
    v = np.ascontiguousarray(heads(qkv[..., 2 * E:]))
    O, lse = attention_rows(q, k, v, 1.0 / np.sqrt(d), causal, key_lens, threads=threads)
    attn = round_bf16(O.transpose(0, 2, 1, 3).reshape(B, N, E))  # merge heads
    return np.matmul(attn, w_o), lse


def attention_backward_literal(q, k, v, dout, scale: float, causal: bool, key_lens=None, out=None,
                               window: int = 0):
    """Gradients of the attention forward with respect to Q, K and V, float64,
    from the materialised score matrix (tiny and moderate sizes):

        P = softmax(S), S = scale Q K^T (hidden keys excluded)
        dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,
        dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q

    (the chain rule through O = P V and the softmax; the pages reuse the
    softmax output in the backward pass, hotelren.com sec. 4.2).  Rows with
    no visible key contribute nothing.  Returns (dQ, dK, dV).

    out: optional stored forward output [B, H, N, d] (for instance bf16 bit
    patterns).  When given, D_i is taken as dO_i . out_i -- the identity
    sum_j P_ij dP_ij = dO_i . (P V)_i applied to that stored output -- instead
    of from P and dP; everything else is unchanged.

    window: the sliding window of attention_literal (query i sees keys
    j > i - window when > 0); P, and so every gradient, follows it.
    """
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    _, _, P = attention_literal(q, k, v, scale, causal, key_lens, window)
    dV = np.matmul(np.swapaxes(P, -1, -2), dout)
    dP = np.matmul(dout, np.swapaxes(v, -1, -2))
    if out is None:
        D = (P * dP).sum(-1, keepdims=True)
    else:
        D = (dout * _as_f64(out)).sum(-1, keepdims=True)
    dS = P * (dP - D)
    dQ = scale * np.matmul(dS, k)
    dK = scale * np.matmul(np.swapaxes(dS, -1, -2), q)
    return dQ, dK, dV


def attention_backward_sampled(q, k, v, dout, scale: float, causal: bool, key_lens=None, heads=None,
                               q_rows=None, k_rows=None, out=None, window: int = 0):
    """The same gradients for selected (b, h) heads, dQ rows and dK/dV rows,
    without the full N x N matrix: each row of P is rebuilt from the row
    oracle's log-sum-exp, P_ij = exp(s_ij - lse_i) over the visible keys.
    out: optional stored forward output [B, H, N, d]; D_i is then dO_i . out_i
    (as in attention_backward_literal).  window: the forward's sliding window
    (query i sees keys j > i - window when > 0).  Returns dicts keyed by
    (b, h): dQ [len(q_rows), d], dK and dV [len(k_rows), d]."""
    q, k, v, dout = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dout)
    stored = out
    B, H, N, d = q.shape
    res = {}
    for b, h in heads:
        kl = N if key_lens is None else int(key_lens[b])
        O, lse = attention_rows(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], scale, causal,
                                None if key_lens is None else np.array([kl], dtype=np.int32), window=window)
        O, lse = O[0, 0], lse[0, 0]
        if stored is not None:
            O = _as_f64(stored[b, h])
        Dvec = (dout[b, h] * O).sum(-1)  # D_i = sum_j P_ij dP_ij = dO_i . O_i
        qb, kb, vb, db = q[b, h], k[b, h], v[b, h], dout[b, h]

        def p_row(i):  # P[i, :] over all keys (zeros where hidden)
            keep = np.arange(N) < kl
            if causal:
                keep &= np.arange(N) <= i
            if window > 0:
                keep &= np.arange(N) > i - window
            if not np.isfinite(lse[i]):
                return np.zeros(N)
            s = scale * (kb @ qb[i])
            return np.where(keep, np.exp(np.where(keep, s, 0.0) - lse[i]), 0.0)

        dQ = np.zeros((len(q_rows), d))
        for r, i in enumerate(q_rows):
            p = p_row(i)
            dp = vb @ db[i]
            dQ[r] = scale * ((p * (dp - Dvec[i])) @ kb)
        dK = np.zeros((len(k_rows), d))
        dV = np.zeros((len(k_rows), d))
        for r, j in enumerate(k_rows):
            col = np.zeros(N)  # P[:, j]
            for i in range(N):
                if j < kl and (not causal or j <= i) and (window <= 0 or j > i - window) and np.isfinite(lse[i]):
                    col[i] = np.exp(scale * (qb[i] @ kb[j]) - lse[i])
            dpj = db @ vb[j]  # dP[:, j]
            ds = col * (dpj - Dvec)
            dV[r] = col @ db
            dK[r] = scale * (ds @ qb)
        res[(b, h)] = (dQ, dK, dV)
    return res
