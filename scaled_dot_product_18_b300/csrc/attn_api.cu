// C ABI of the attention forward: argument checks on the host, tensor-map
// encoding, launch, and the device error word.  The operation and every
// argument are specified in include/attn.h.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn.h"
#include "attn_internal.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up through the runtime so the
// library does not link against libcuda (it loads on machines without a GPU).
EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Element strides of the rows, heads and batches of a bf16 [.., d] tensor.
struct Strides {
    int64_t row, head, batch;
};

// ------------------------------------------------------------- tensor-map cache
//
// Encoding a tensor map costs about 1.5 us of host time, and a call encodes up
// to five; at the small shapes that is more than the kernel takes.  A map is
// a pure function of its encode arguments (address, type, sizes, strides,
// box, swizzle), so maps are kept in a fixed table keyed on all of them and
// copied out on a hit: a reused buffer layout costs a lookup, a new address
// or shape one encode.  The table never allocates; when full, the oldest
// entry is replaced.
struct MapKey {
    uint64_t base;
    uint64_t dims[4];
    uint64_t strides[3];
    uint32_t box[4];
    uint32_t rank, dtype, swizzle;
    bool operator==(const MapKey &o) const
    {
        if (base != o.base || rank != o.rank || dtype != o.dtype || swizzle != o.swizzle) return false;
        for (int i = 0; i < 4; ++i)
            if (dims[i] != o.dims[i] || box[i] != o.box[i]) return false;
        for (int i = 0; i < 3; ++i)
            if (strides[i] != o.strides[i]) return false;
        return true;
    }
};

constexpr int kMapCacheSize = 256;
struct MapCache {
    std::mutex mu;
    MapKey key[kMapCacheSize];
    CUtensorMap map[kMapCacheSize];
    int used = 0, next = 0;
    uint64_t hits = 0, misses = 0;
};
MapCache &map_cache()
{
    static MapCache c;
    return c;
}

// Encodes (or fetches from the cache) a tiled map of `rank` dimensions.
bool cached_encode(CUtensorMap *m, CUtensorMapDataType dtype, uint32_t rank, const void *base, const cuuint64_t *dims,
                   const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle swizzle)
{
    MapKey k{};
    k.base = reinterpret_cast<uint64_t>(base);
    k.rank = rank;
    k.dtype = static_cast<uint32_t>(dtype);
    k.swizzle = static_cast<uint32_t>(swizzle);
    for (uint32_t i = 0; i < rank; ++i) {
        k.dims[i] = dims[i];
        k.box[i] = box[i];
        if (i + 1 < rank) k.strides[i] = strides[i];
    }
    MapCache &c = map_cache();
    {
        std::lock_guard<std::mutex> lock(c.mu);
        for (int i = 0; i < c.used; ++i)
            if (c.key[i] == k) {
                *m = c.map[i];
                ++c.hits;
                return true;
            }
    }
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (enc(m, dtype, rank, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    std::lock_guard<std::mutex> lock(c.mu);
    ++c.misses;
    const int slot = c.used < kMapCacheSize ? c.used++ : c.next;
    c.next = (slot + 1) % kMapCacheSize;
    c.key[slot] = k;
    c.map[slot] = *m;
    return true;
}

// 4-D view {d, N, H, B} of a bf16 tensor with the given element strides,
// box = 64 head-dim columns x box_rows rows x 1 head x 1 batch, 128-byte
// swizzle (one box row = 128 bytes).  Rows past N read as zeros and are
// clipped on store, so ragged N needs no padding.
bool make_map(CUtensorMap *m, const void *base, int B, int H, int N, int d, Strides st, int box_rows = 128)
{
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.row) * 2, static_cast<cuuint64_t>(st.head) * 2,
                                   static_cast<cuuint64_t>(st.batch) * 2};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
    return cached_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Contiguous [B, H, N, d].
Strides bhnd(int H, int N, int d)
{
    return {d, static_cast<int64_t>(N) * d, static_cast<int64_t>(H) * N * d};
}

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

// Launch on Q/K/V/O with the given layouts (validated by the callers).
attn_status launch_forward(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int N,
                           int d, float scale, int causal, const int32_t *key_lens, int window, Strides in_st,
                           Strides out_st, attn_stream_t stream)
{
    CUtensorMap tq, tk, tv, to;
    if (!make_map(&tq, q, B, H, N, d, in_st) || !make_map(&tk, k, B, H, N, d, in_st) ||
        !make_map(&tv, v, B, H, N, d, in_st) || !make_map(&to, out, B, H, N, d, out_st, 32))
        return ATTN_ECUDA;
    sdp18::AttnLaunch a{};
    a.tm_q = &tq;
    a.tm_k = &tk;
    a.tm_v = &tv;
    a.tm_o = &to;
    a.out = out;
    a.ost = {out_st.row, out_st.head, out_st.batch};
    a.lse = lse;
    a.key_lens = key_lens;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    a.causal = causal ? 1 : 0;
    a.window = window >= N ? 0 : window;  // a window covering every key is no window
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    const int rc = sdp18::attn_fwd_launch(a);
    if (rc == -2) return ATTN_EUNSUPPORTED;
    return rc == 0 ? ATTN_OK : ATTN_ECUDA;
}

attn_status forward(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int N, int d,
                    float scale, int causal, const int32_t *key_lens, int window, attn_stream_t stream)
{
    if (B < 0 || H < 0 || N < 0 || window < 0) return ATTN_EINVAL;
    if (d != 64 && d != 128) return ATTN_EUNSUPPORTED;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_EINVAL;
    if (B == 0 || H == 0 || N == 0) return ATTN_OK;
    if (!q || !k || !v || !out) return ATTN_EINVAL;
    const int64_t bh = static_cast<int64_t>(B) * H;
    const int64_t q_tiles = (static_cast<int64_t>(N) + 127) / 128;
    if (bh > INT32_MAX || q_tiles * bh > INT32_MAX) return ATTN_EINVAL;
    if (misaligned(q) || misaligned(k) || misaligned(v) || misaligned(out)) return ATTN_EALIGN;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_EALIGN;
    if (key_lens && (reinterpret_cast<uintptr_t>(key_lens) & 3u)) return ATTN_EALIGN;

    return launch_forward(q, k, v, out, lse, B, H, N, d, scale, causal, key_lens, window, bhnd(H, N, d),
                          bhnd(H, N, d), stream);
}

// ------------------------------------------------------------- multi-head block

// 2-D view {inner, outer} of a row-major bf16 matrix with rows of `ld`
// elements, 128-byte swizzled boxes of 64 x box_rows.
bool make_map_2d(CUtensorMap *m, const void *base, int inner, int outer, int64_t ld, int box_rows)
{
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    return cached_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// C[M, N] = A[M, K] B[K, N], all row-major bf16 (leading dimensions K, N, N),
// on this library's tcgen05 GEMM kernel.
attn_status gemm_bf16(int M, int N, int K, const void *A, const void *Bm, void *C, cudaStream_t stream)
{
    CUtensorMap ta, tb;
    if (!make_map_2d(&ta, A, K, M, K, 128) || !make_map_2d(&tb, Bm, N, K, N, 64)) return ATTN_ECUDA;
    sdp18::GemmLaunch g{};
    g.tm_a = &ta;
    g.tm_b = &tb;
    g.c = C;
    g.ldc = N;
    g.M = M;
    g.N = N;
    g.K = K;
    g.stream = stream;
    const int rc = sdp18::gemm_bf16_launch(g);
    if (rc == -2) return ATTN_EUNSUPPORTED;
    return rc == 0 ? ATTN_OK : ATTN_ECUDA;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" {

size_t attn_mha_workspace_size(int B, int N, int E)
{
    if (B <= 0 || N <= 0 || E <= 0) return 0;
    const size_t rows = static_cast<size_t>(B) * N;
    return round256(rows * 3 * E * 2) + round256(rows * E * 2);
}

attn_status attn_mha_fwd(const void *x, const void *w_qkv, const void *w_o, void *out, float *lse, int B, int N,
                         int E, int H, int causal, const int32_t *key_lens, void *workspace, size_t workspace_bytes,
                         attn_stream_t stream)
{
    if (B < 0 || N < 0 || E <= 0 || H <= 0 || E % H != 0) return ATTN_EINVAL;
    const int d = E / H;
    if (d != 64 && d != 128) return ATTN_EUNSUPPORTED;
    if (B == 0 || N == 0) return ATTN_OK;
    if (!x || !w_qkv || !w_o || !out || !workspace) return ATTN_EINVAL;
    const int64_t rows = static_cast<int64_t>(B) * N;
    if (rows * 3 * E > INT32_MAX || static_cast<int64_t>(B) * H * ((N + 127) / 128) > INT32_MAX) return ATTN_EINVAL;
    if (workspace_bytes < attn_mha_workspace_size(B, N, E)) return ATTN_EINVAL;
    if (misaligned(x) || misaligned(w_qkv) || misaligned(w_o) || misaligned(out) || misaligned(workspace))
        return ATTN_EALIGN;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_EALIGN;
    if (key_lens && (reinterpret_cast<uintptr_t>(key_lens) & 3u)) return ATTN_EALIGN;

    char *ws = static_cast<char *>(workspace);
    const size_t qkv_bytes = round256(static_cast<size_t>(rows) * 3 * E * 2);
    auto *qkv = reinterpret_cast<__nv_bfloat16 *>(ws);
    auto *attn = reinterpret_cast<__nv_bfloat16 *>(ws + qkv_bytes);
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    // 1. [Q | K | V] = x W_qkv: rows of [B*N, 3E], head h at columns h*d of each part.
    attn_status st = gemm_bf16(static_cast<int>(rows), 3 * E, E, x, w_qkv, qkv, s);
    if (st != ATTN_OK) return st;
    // 2. Attention straight from the interleaved rows ([B, N, H, d] views), the
    //    merged heads written as rows of [B*N, E].
    const Strides in_st{3 * static_cast<int64_t>(E), d, static_cast<int64_t>(N) * 3 * E};
    const Strides out_st{E, d, static_cast<int64_t>(N) * E};
    st = launch_forward(qkv, qkv + E, qkv + 2 * E, attn, lse, B, H, N, d,
                        static_cast<float>(1.0 / std::sqrt(static_cast<double>(d))), causal, key_lens, 0, in_st,
                        out_st, stream);
    if (st != ATTN_OK) return st;
    // 3. out = merged W_o.
    return gemm_bf16(static_cast<int>(rows), E, E, attn, w_o, out, s);
}


attn_status attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int N, int d,
                     float scale, int causal, const int32_t *key_lens, attn_stream_t stream)
{
    return forward(q, k, v, out, lse, B, H, N, d, scale, causal, key_lens, 0, stream);
}

attn_status attn_fwd_window(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int N,
                            int d, float scale, int causal, const int32_t *key_lens, int window,
                            attn_stream_t stream)
{
    return forward(q, k, v, out, lse, B, H, N, d, scale, causal, key_lens, window, stream);
}

size_t attn_decode_workspace_size(int B, int H, int L, int d)
{
    if (B <= 0 || H <= 0 || L <= 0 || (d != 64 && d != 128)) return 0;
    const sdp18::DecodeSplit sp = sdp18::decode_split(B, H, L);
    const size_t slots = static_cast<size_t>(B) * H * sp.splits;
    const size_t o_bytes = (slots * d * sizeof(float) + 255) / 256 * 256;
    return o_bytes + slots * sizeof(float);
}

attn_status attn_decode(const void *q, const void *k_cache, const void *v_cache, void *out, float *lse, int B, int H,
                        int L, int d, float scale, const int32_t *cache_lens, void *workspace,
                        size_t workspace_bytes, attn_stream_t stream)
{
    if (B < 0 || H < 0 || L < 0) return ATTN_EINVAL;
    if (d != 64 && d != 128) return ATTN_EUNSUPPORTED;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_EINVAL;
    if (B == 0 || H == 0) return ATTN_OK;
    if (!q || !out) return ATTN_EINVAL;
    if (static_cast<int64_t>(B) * H > INT32_MAX / 64) return ATTN_EINVAL;
    if (L > 0 && (!k_cache || !v_cache)) return ATTN_EINVAL;
    const size_t need = attn_decode_workspace_size(B, H, L > 0 ? L : 1, d);
    if (!workspace || workspace_bytes < need) return ATTN_EINVAL;
    if (misaligned(q) || misaligned(out) || misaligned(workspace) || (L > 0 && (misaligned(k_cache) || misaligned(v_cache))))
        return ATTN_EALIGN;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return ATTN_EALIGN;
    if (cache_lens && (reinterpret_cast<uintptr_t>(cache_lens) & 3u)) return ATTN_EALIGN;

    const int Lx = L > 0 ? L : 1;  // an empty cache runs one empty split per head
    const sdp18::DecodeSplit sp = sdp18::decode_split(B, H, Lx);
    const size_t slots = static_cast<size_t>(B) * H * sp.splits;
    sdp18::DecodeLaunch a{};
    a.q = q;
    a.k = L > 0 ? k_cache : q;  // never read when L == 0 (L_keys = 0: every split is empty)
    a.v = L > 0 ? v_cache : q;
    a.out = out;
    a.lse = lse;
    a.cache_lens = L > 0 ? cache_lens : nullptr;
    a.part_o = static_cast<float *>(workspace);
    a.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + (slots * d * sizeof(float) + 255) / 256 * 256);
    a.B = B;
    a.H = H;
    a.L = Lx;
    a.L_keys = L;
    a.d = d;
    a.splits = sp.splits;
    a.chunk = sp.chunk;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    const int rc = sdp18::attn_decode_launch(a);
    if (rc == -2) return ATTN_EUNSUPPORTED;
    return rc == 0 ? ATTN_OK : ATTN_ECUDA;
}

size_t attn_bwd_workspace_size(int B, int H, int N, int d)
{
    if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
    const size_t bh = static_cast<size_t>(B) * H;
    const size_t n_pad = (static_cast<size_t>(N) + 127) / 128 * 128;
    // fp32 dQ accumulator [B*H*N, d], then lse*log2e and D per padded query row
    return round256(bh * N * d * sizeof(float)) + round256(2 * bh * n_pad * sizeof(float));
}

namespace {

// 3-D view {d, N, B*H} of the fp32 dQ accumulator with 32 x 32 boxes (128-byte
// rows, 128-byte swizzle): the target of the backward's TMA reductions.
bool make_dq_map(CUtensorMap *m, float *base, int64_t BH, int N, int d)
{
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(N) * d * 4};
    const cuuint32_t box[3] = {32, 32, 1};
    return cached_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

namespace {

attn_status backward(const void *q, const void *k, const void *v, const void *out, const void *dout, const float *lse,
                     void *dq, void *dk, void *dv, int B, int H, int N, int d, float scale, int causal,
                     const int32_t *key_lens, int window, void *workspace, size_t workspace_bytes,
                     attn_stream_t stream)
{
    if (B < 0 || H < 0 || N < 0 || window < 0) return ATTN_EINVAL;
    if (d != 64 && d != 128) return ATTN_EUNSUPPORTED;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_EINVAL;
    if (B == 0 || H == 0 || N == 0) return ATTN_OK;
    if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv || !workspace) return ATTN_EINVAL;
    const int64_t bh = static_cast<int64_t>(B) * H;
    const int64_t tiles = (static_cast<int64_t>(N) + 127) / 128;
    if (bh > INT32_MAX || tiles * bh > INT32_MAX || bh * N * d > (int64_t(1) << 40)) return ATTN_EINVAL;
    if (workspace_bytes < attn_bwd_workspace_size(B, H, N, d)) return ATTN_EINVAL;
    for (const void *p : {q, k, v, out, dout, static_cast<const void *>(dq), static_cast<const void *>(dk),
                          static_cast<const void *>(dv), static_cast<const void *>(workspace)})
        if (misaligned(p)) return ATTN_EALIGN;
    if (reinterpret_cast<uintptr_t>(lse) & 3u) return ATTN_EALIGN;
    if (key_lens && (reinterpret_cast<uintptr_t>(key_lens) & 3u)) return ATTN_EALIGN;

    const Strides st = bhnd(H, N, d);
    CUtensorMap tq, tk, tv, tdo;
    if (!make_map(&tq, q, B, H, N, d, st) || !make_map(&tk, k, B, H, N, d, st) || !make_map(&tv, v, B, H, N, d, st) ||
        !make_map(&tdo, dout, B, H, N, d, st))
        return ATTN_ECUDA;
    const size_t rows = static_cast<size_t>(bh) * N;
    float *dqacc = static_cast<float *>(workspace);
    CUtensorMap tdq;
    if (!make_dq_map(&tdq, dqacc, bh, N, d)) return ATTN_ECUDA;
    sdp18::BwdLaunch a{};
    a.tm_q = &tq;
    a.tm_k = &tk;
    a.tm_v = &tv;
    a.tm_do = &tdo;
    a.tm_dq = &tdq;
    a.out = out;
    a.dout = dout;
    a.lse = lse;
    a.dqacc = dqacc;
    a.stats = reinterpret_cast<float *>(static_cast<char *>(workspace) + round256(rows * d * sizeof(float)));
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.key_lens = key_lens;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.window = window >= N ? 0 : window;
    a.stream = reinterpret_cast<cudaStream_t>(stream);
    const int rc = sdp18::attn_bwd_launch(a);
    if (rc == -2) return ATTN_EUNSUPPORTED;
    return rc == 0 ? ATTN_OK : ATTN_ECUDA;
}

}  // namespace

attn_status attn_bwd(const void *q, const void *k, const void *v, const void *out, const void *dout, const float *lse,
                     void *dq, void *dk, void *dv, int B, int H, int N, int d, float scale, int causal,
                     const int32_t *key_lens, void *workspace, size_t workspace_bytes, attn_stream_t stream)
{
    return backward(q, k, v, out, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, key_lens, 0, workspace,
                    workspace_bytes, stream);
}

attn_status attn_bwd_window(const void *q, const void *k, const void *v, const void *out, const void *dout,
                            const float *lse, void *dq, void *dk, void *dv, int B, int H, int N, int d, float scale,
                            int causal, const int32_t *key_lens, int window, void *workspace, size_t workspace_bytes,
                            attn_stream_t stream)
{
    return backward(q, k, v, out, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, key_lens, window, workspace,
                    workspace_bytes, stream);
}

attn_status attn_check_device(attn_stream_t stream)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ECUDA;
    int v = 0, vb = 0, vg = 0;
    if (sdp18::read_and_clear_device_error(&v) != 0) return ATTN_ECUDA;
    if (sdp18::read_and_clear_bwd_error(&vb) != 0) return ATTN_ECUDA;
    if (sdp18::read_and_clear_gemm_error(&vg) != 0) return ATTN_ECUDA;
    return (v != 0 || vb != 0 || vg != 0) ? ATTN_EDEVICE : ATTN_OK;
}

const char *attn_status_str(attn_status s)
{
    switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_EINVAL: return "ATTN_EINVAL: invalid argument";
    case ATTN_EUNSUPPORTED: return "ATTN_EUNSUPPORTED: head dimension must be 64 or 128";
    case ATTN_EALIGN: return "ATTN_EALIGN: tensor pointer not 16-byte aligned";
    case ATTN_ECUDA: return "ATTN_ECUDA: CUDA error";
    case ATTN_EDEVICE: return "ATTN_EDEVICE: kernel gave up on a bounded wait";
    case ATTN_ETOOLARGE: return "ATTN_ETOOLARGE: problem exceeds the fixed scratch area of attn_decode_noalloc";
    }
    return "unknown attn_status";
}

int attn_abi_version(void) { return ATTN_ABI_VERSION; }

void attn_tensor_map_cache_stats(uint64_t *hits, uint64_t *misses)
{
    MapCache &c = map_cache();
    std::lock_guard<std::mutex> lock(c.mu);
    if (hits) *hits = c.hits;
    if (misses) *misses = c.misses;
}

}  // extern "C"
