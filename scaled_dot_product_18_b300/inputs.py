"""Seeded synthetic inputs for the attention forward (Q, K, V, key_lens).

This module is shared by the tests, the benchmark and the smoke check, and it
holds none of the attention arithmetic: it only draws numbers.

Generator (counter-based, so any element can be drawn on its own):

* ``x = splitmix64_mix(key(seed, stream) + (i + 1) * GOLDEN)`` for counter ``i``,
  where ``splitmix64_mix`` is the output function of Steele, Lea and Flood's
  SplitMix64 ("Fast splittable pseudorandom number generators", OOPSLA 2014)
  and ``GOLDEN = 0x9E3779B97F4A7C15``.
* Uniforms ``u = (x >> 11) * 2**-53`` in [0, 1).
* Normals by the Box-Muller transform on counter pairs (2p, 2p+1):
  ``r = sqrt(-2 ln(1 - u0))``, element 2p gets ``r cos(2 pi u1)``, element 2p+1
  gets ``r sin(2 pi u1)``; all of it in float64.
* The float64 value (times an optional amplitude, e.g. 1.5) is rounded ONCE to
  bfloat16, round-to-nearest-even, and returned as raw uint16 bit patterns.

Streams: 0 = Q, 1 = K, 2 = V, 3 = key_lens.  ``key_lens[b] = lo + floor(u_b *
(hi - lo + 1))`` with ``u_b`` the b-th uniform of stream 3.

Workload shapes follow the attention pages' examples: the long-context
B=1, H=32, N=16384, d=128 case ("Why does attention stall large-model
training?", aicoding.csdn.net, ch.1 "typical stall scenario"), the
embed-512/8-head, length-100 test of ``MinimalSelfAttention`` (cnnetsun.cn,
"Transformer QKV bottlenecks on long sequences", sec. 2 "quick start"), and a
BERT-base-like B=16, H=12, N=512 shape.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM_Q, STREAM_K, STREAM_V, STREAM_KEYLEN, STREAM_DOUT = 0, 1, 2, 3, 4

_CHUNK = 1 << 19  # Box-Muller pairs per vectorised block (keeps temporaries small)
_THREADS = max(1, min(16, os.cpu_count() or 1))


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.array([(seed * 0x100000001B3 + stream * 0x2545F4914F6CDD1D + 0x243F6A8885A308D3)
                         & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix(base)[0]


def raw_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Counters start .. start+count-1 of one stream, as uint64 words."""
    key = _stream_key(seed, stream)
    ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + ctr * GOLDEN)


def uniforms(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Float64 uniforms in [0, 1) with 53 random bits."""
    return (raw_u64(seed, stream, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def _normal_pairs(seed: int, stream: int, a: int, b: int, out: np.ndarray) -> None:
    """Box-Muller pairs a .. b-1 written to ``out`` (length 2*(b-a))."""
    u = uniforms(seed, stream, 2 * a, 2 * (b - a))
    u0, u1 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log1p(-u0))
    th = (2.0 * np.pi) * u1
    out[0::2] = r * np.cos(th)
    out[1::2] = r * np.sin(th)


def normals_f64(seed: int, stream: int, count: int, start: int = 0) -> np.ndarray:
    """Standard normals (float64) for elements start .. start+count-1 of a stream."""
    if count == 0:
        return np.zeros(0, dtype=np.float64)
    p0 = start // 2
    p1 = (start + count + 1) // 2
    out = np.empty(2 * (p1 - p0), dtype=np.float64)

    def job(a: int) -> None:
        b = min(p1, a + _CHUNK)
        _normal_pairs(seed, stream, a, b, out[2 * (a - p0): 2 * (b - p0)])

    blocks = range(p0, p1, _CHUNK)
    if len(blocks) > 1 and _THREADS > 1:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(job, blocks))
    else:
        for a in blocks:
            job(a)
    off = start - 2 * p0
    return out[off: off + count]


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values once to bfloat16 (nearest, ties to even).

    Works on the float64 bit pattern so there is a single rounding step.  Values
    must be finite and inside the float32 normal range or exactly zero (true for
    every generated input); tiny magnitudes below 2**-126 are rounded through
    float32, which is exact enough for them.
    """
    x = np.asarray(x, dtype=np.float64)
    bits = x.view(np.uint64)
    # keep 1 sign + 11 exponent + 7 mantissa bits of the float64 -> drop 45 bits
    lsb = (bits >> np.uint64(45)) & np.uint64(1)
    rounded = (bits + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    as_f32 = rounded.view(np.float64).astype(np.float32)  # exact: 8 significant bits
    out = (as_f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    tiny = np.abs(x) < 2.0 ** -126
    if np.any(tiny):
        f = x[tiny].astype(np.float32).view(np.uint32)
        r = (f + np.uint32(0x7FFF) + ((f >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        out[tiny] = r.astype(np.uint16)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32 (for display/tests)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention-forward problem: shapes, mask and input recipe."""
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    key_len_range: tuple[int, int] | None = None  # inclusive [lo, hi], drawn per batch element
    amplitude: float = 1.0  # N(0,1) * amplitude, rounded once to bf16
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    def flops(self) -> float:
        """Nominal forward flops 4*B*H*N^2*d, halved for causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def algorithmic_bytes(self) -> int:
        """Q, K, V read once plus O written once (bf16) and the fp32 LSE."""
        return 4 * self.B * self.H * self.N * self.d * 2 + self.B * self.H * self.N * 4


# The five workloads (the pages' shapes; see the module docstring).
WORKLOADS = {
    "c1_b1h2n128d64": Workload("c1_b1h2n128d64", 1, 2, 128, 64, False),
    "c2_b2h8n100d64_keylens": Workload("c2_b2h8n100d64_keylens", 2, 8, 100, 64, False, (1, 100)),
    "c3_b16h12n512d64_keylens_x1.5": Workload("c3_b16h12n512d64_keylens_x1.5", 16, 12, 512, 64, False,
                                               (256, 512), amplitude=1.5),
    "c4_b4h32n4096d128_causal": Workload("c4_b4h32n4096d128_causal", 4, 32, 4096, 128, True),
    "c5_b1h32n16384d128_causal": Workload("c5_b1h32n16384d128_causal", 1, 32, 16384, 128, True),
}
WORKLOAD_ORDER = list(WORKLOADS)

# Further measured shapes: the B=4 H=32 N=4096 d=128 shape without the causal
# mask (the non-causal, tensor-bound counterpart of the causal workloads).
EXTRA_WORKLOADS = {
    "c4nc_b4h32n4096d128": Workload("c4nc_b4h32n4096d128", 4, 32, 4096, 128, False),
}


def make_tensor_bits(seed: int, stream: int, shape: tuple[int, ...], amplitude: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of N(0,1)*amplitude, C-contiguous, in ``shape``."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    pairs = (n + 1) // 2

    def job(a: int) -> None:
        b = min(pairs, a + _CHUNK)
        x = np.empty(2 * (b - a), dtype=np.float64)
        _normal_pairs(seed, stream, a, b, x)
        if amplitude != 1.0:
            x *= amplitude
        lo, hi = 2 * a, min(n, 2 * b)
        out[lo:hi] = f64_to_bf16_bits(x[: hi - lo])

    blocks = range(0, pairs, _CHUNK)
    if len(blocks) > 1 and _THREADS > 1:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(job, blocks))
    else:
        for a in blocks:
            job(a)
    return out.reshape(shape)


def make_key_lens(seed: int, B: int, lo: int, hi: int) -> np.ndarray:
    u = uniforms(seed, STREAM_KEYLEN, 0, B)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int32)


@dataclasses.dataclass
class HostInputs:
    """Host copies of one problem's inputs: bf16 bits for Q/K/V, int32 key_lens."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    key_lens: np.ndarray | None


def make_inputs(w: Workload, seed: int | None = None) -> HostInputs:
    s = w.seed if seed is None else seed
    shape = (w.B, w.H, w.N, w.d)
    q = make_tensor_bits(s, STREAM_Q, shape, w.amplitude)
    k = make_tensor_bits(s, STREAM_K, shape, w.amplitude)
    v = make_tensor_bits(s, STREAM_V, shape, w.amplitude)
    kl = make_key_lens(s, w.B, *w.key_len_range) if w.key_len_range else None
    return HostInputs(q, k, v, kl)


def make_dout(w: Workload, seed: int | None = None) -> np.ndarray:
    """bf16 bits of the loss gradient dO [B, H, N, d] for the backward: N(0,1),
    its own stream of the workload's seed."""
    s = w.seed if seed is None else seed
    return make_tensor_bits(s, STREAM_DOUT, (w.B, w.H, w.N, w.d))


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """One query per (batch, head) against a [B, H, L, d] key/value cache, the
    cache layout of the pages' KV-cache section (hotelren.com "AI attention:
    essence and evolution", sec. 3.1).  cache_len_range: inclusive [lo, hi]
    drawn per batch element, or None for full caches."""
    name: str
    B: int
    H: int
    L: int
    d: int
    cache_len_range: tuple[int, int] | None = None
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    def bytes_moved(self, cache_lens=None) -> int:
        """K and V rows read for the visible keys, plus q, O (bf16) and lse."""
        rows = self.B * self.L if cache_lens is None else int(np.sum(np.clip(cache_lens, 0, self.L)))
        return rows * self.H * self.d * 2 * 2 + 2 * self.B * self.H * self.d * 2 + self.B * self.H * 4


# Llama-3-8B-like heads (32 x 128) at the pages' 2048-token input length, and
# the long-context length of the 16K example.
DECODE_WORKLOADS = {
    "decode_b16h32l2048d128": DecodeWorkload("decode_b16h32l2048d128", 16, 32, 2048, 128),
    "decode_b4h32l16384d128": DecodeWorkload("decode_b4h32l16384d128", 4, 32, 16384, 128),
}


def make_decode_inputs(w: DecodeWorkload, seed: int | None = None) -> HostInputs:
    """q [B, H, d], caches [B, H, L, d] (bf16 bits), cache_lens [B] or None."""
    s = w.seed if seed is None else seed
    q = make_tensor_bits(s, STREAM_Q, (w.B, w.H, w.d))
    k = make_tensor_bits(s, STREAM_K, (w.B, w.H, w.L, w.d))
    v = make_tensor_bits(s, STREAM_V, (w.B, w.H, w.L, w.d))
    cl = make_key_lens(s, w.B, *w.cache_len_range) if w.cache_len_range else None
    return HostInputs(q, k, v, cl)


@dataclasses.dataclass(frozen=True)
class MhaWorkload:
    """A multi-head self-attention block: x [B, N, E] ~ N(0, 1), projection
    weights ~ N(0, 1/E) (so Q, K, V and the output stay O(1)), H heads of
    d = E/H, causal flag and optional per-batch key lengths."""
    name: str
    B: int
    N: int
    E: int
    H: int
    causal: bool
    key_len_range: tuple[int, int] | None = None
    seed: int = 0

    @property
    def d(self) -> int:
        return self.E // self.H

    def flops(self) -> float:
        """Projections 2*B*N*E*4E plus nominal attention 4*B*H*N^2*d (halved for causal)."""
        att = 4.0 * self.B * self.H * self.N * self.N * self.d
        return 2.0 * self.B * self.N * self.E * 4 * self.E + (att / 2 if self.causal else att)


MHA_WORKLOADS = {
    # cnnetsun.cn's MinimalSelfAttention check: input (2, 100, 512), 8 heads
    "mha_b2n100e512h8": MhaWorkload("mha_b2n100e512h8", 2, 100, 512, 8, False),
    # BERT-base-like block (embed 768, 12 heads) with padded sequences
    "mha_b16n512e768h12_keylens": MhaWorkload("mha_b16n512e768h12_keylens", 16, 512, 768, 12, False, (256, 512)),
    # long-context block with 32 heads of 128 (embed 4096), causal
    "mha_b1n16384e4096h32_causal": MhaWorkload("mha_b1n16384e4096h32_causal", 1, 16384, 4096, 32, True),
}


@dataclasses.dataclass
class MhaInputs:
    x: np.ndarray       # bf16 bits [B, N, E]
    w_qkv: np.ndarray   # bf16 bits [E, 3E]
    w_o: np.ndarray     # bf16 bits [E, E]
    key_lens: np.ndarray | None


def make_mha_inputs(w: MhaWorkload, seed: int | None = None) -> MhaInputs:
    s = w.seed if seed is None else seed
    x = make_tensor_bits(s, STREAM_Q, (w.B, w.N, w.E))
    wqkv = make_tensor_bits(s, STREAM_K, (w.E, 3 * w.E), amplitude=1.0 / float(np.sqrt(w.E)))
    wo = make_tensor_bits(s, STREAM_V, (w.E, w.E), amplitude=1.0 / float(np.sqrt(w.E)))
    kl = make_key_lens(s, w.B, *w.key_len_range) if w.key_len_range else None
    return MhaInputs(x, wqkv, wo, kl)
