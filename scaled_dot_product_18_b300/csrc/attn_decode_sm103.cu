// Attention for one new query per (batch, head) against a key/value cache
// (decode): O = softmax(q K^T * scale) V over the cached keys j < cache_len.
//
// The cache layout is the pages' [batch, heads, seq_len, head_dim]
// (hotelren.com "AI attention: essence and evolution", sec. 3.1, KV cache:
// each step appends one key/value row and reuses the rest).  One query row
// makes S a vector, so the work is a streaming read of K and V: 2 flops per
// byte, bound by HBM bandwidth, not by the tensor cores.  It runs on CUDA
// cores, split along the cache so every SM streams:
//
//   decode_partial  CTA (b,h,split): keys [split*chunk, ...) of the cache.
//                   16 threads share a key row (16 bytes each, d = 128; 8
//                   threads at d = 64), so a step reads 8 (16) whole rows of
//                   K and V with coalesced 16-byte loads.  Each row group keeps
//                   its own running max / sum / partial O (online softmax in
//                   the log2 domain); the groups merge through shared memory
//                   and the split writes O_split (normalised, fp32) and its
//                   natural-log lse_split to the workspace.
//   decode_combine  CTA (b,h): lse = ln sum_s exp(lse_s), O = sum_s
//                   exp(lse_s - lse) O_s (the log-sum-exp merge of
//                   aicoding.csdn.net "Why does attention stall large-model
//                   training", sec. 2.2, chunked logsumexp), bf16 out.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn.h"
#include "attn_internal.h"

namespace sdp18 {
namespace {

constexpr int kDecThreads = 128;

__device__ __forceinline__ float ex2f_fast(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Eight bf16 (one 16-byte load) -> eight floats, exactly.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Streaming 16-byte load (each cache byte is read once).
__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}

template <int D>
__global__ void __launch_bounds__(kDecThreads)
    decode_partial(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
                   const __nv_bfloat16 *__restrict__ v, const int32_t *__restrict__ cache_lens, int H, int L,
                   int L_keys, int splits, int chunk, float scale_log2, float *__restrict__ part_o,
                   float *__restrict__ part_lse)
{
    constexpr int kSeg = D / 8;                 // threads per key row
    constexpr int kRows = kDecThreads / kSeg;   // key rows per step
    constexpr int kUnroll = 8;                  // steps with loads in flight
    __shared__ float s_o[kRows][D];
    __shared__ float s_m[kRows], s_l[kRows];

    const int bh = blockIdx.x / splits;
    const int sp = blockIdx.x % splits;
    const int b = bh / H;
    int len = L_keys;  // L is the row stride of the cache, L_keys <= L the rows that hold keys
    if (cache_lens != nullptr) len = min(max(cache_lens[b], 0), L_keys);
    const int j0 = sp * chunk;
    const int j1 = min(j0 + chunk, len);

    const int t = threadIdx.x;
    const int r = t / kSeg;    // row group
    const int seg = t % kSeg;  // 8-element segment of the row

    float qf[8];
    bf16x8_to_f32(*reinterpret_cast<const uint4 *>(q + static_cast<size_t>(bh) * D + seg * 8), qf);
    const __nv_bfloat16 *kp = k + static_cast<size_t>(bh) * L * D + seg * 8;
    const __nv_bfloat16 *vp = v + static_cast<size_t>(bh) * L * D + seg * 8;

    float m = -INFINITY, l = 0.f;
    float o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = 0.f;

    for (int jb = j0; jb < j1; jb += kRows * kUnroll) {
        uint4 kr[kUnroll], vr[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) kr[u] = vr[u] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = jb + u * kRows + r;
            if (j < j1) {
                kr[u] = ld_stream(kp + static_cast<size_t>(j) * D);
                vr[u] = ld_stream(vp + static_cast<size_t>(j) * D);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = jb + u * kRows + r;
            float kf[8];
            bf16x8_to_f32(kr[u], kf);
            float dot = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) dot = fmaf(qf[i], kf[i], dot);
#pragma unroll
            for (int off = kSeg / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
            if (j < j1) {
                const float s = dot * scale_log2;
                if (s > m) {
                    const float alpha = ex2f_fast(m - s);  // 0 while m = -inf
                    m = s;
                    l *= alpha;
#pragma unroll
                    for (int i = 0; i < 8; ++i) o[i] *= alpha;
                }
                const float p = ex2f_fast(s - m);
                l += p;
                float vf[8];
                bf16x8_to_f32(vr[u], vf);
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = fmaf(p, vf[i], o[i]);
            }
        }
    }

    // Merge the row groups (same log2-domain statistics in every thread of a group).
#pragma unroll
    for (int i = 0; i < 8; ++i) s_o[r][seg * 8 + i] = o[i];
    if (seg == 0) {
        s_m[r] = m;
        s_l[r] = l;
    }
    __syncthreads();
    if (t < D) {
        float mm = -INFINITY;
#pragma unroll
        for (int g = 0; g < kRows; ++g) mm = fmaxf(mm, s_m[g]);
        float lt = 0.f, ot = 0.f;
        if (mm != -INFINITY) {
#pragma unroll
            for (int g = 0; g < kRows; ++g) {
                const float w = s_m[g] == -INFINITY ? 0.f : ex2f_fast(s_m[g] - mm);
                lt = fmaf(w, s_l[g], lt);
                ot = fmaf(w, s_o[g][t], ot);
            }
        }
        const size_t slot = static_cast<size_t>(bh) * splits + sp;
        part_o[slot * D + t] = lt > 0.f ? ot / lt : 0.f;
        if (t == 0) part_lse[slot] = lt > 0.f ? (mm + log2f(lt)) * 0.69314718055994531f : -INFINITY;
    }
}

template <int D>
__global__ void __launch_bounds__(D)
    decode_combine(const float *__restrict__ part_o, const float *__restrict__ part_lse, int splits,
                   __nv_bfloat16 *__restrict__ out, float *__restrict__ lse)
{
    const int bh = blockIdx.x;
    const int c = threadIdx.x;
    const float *pl = part_lse + static_cast<size_t>(bh) * splits;
    float mm = -INFINITY;
    for (int s = 0; s < splits; ++s) mm = fmaxf(mm, pl[s]);
    float den = 0.f, acc = 0.f;
    if (mm != -INFINITY) {
        for (int s = 0; s < splits; ++s) {
            const float w = pl[s] == -INFINITY ? 0.f : __expf(pl[s] - mm);
            den += w;
            acc = fmaf(w, part_o[(static_cast<size_t>(bh) * splits + s) * D + c], acc);
        }
    }
    out[static_cast<size_t>(bh) * D + c] = __float2bfloat16_rn(den > 0.f ? acc / den : 0.f);
    if (c == 0 && lse != nullptr) lse[bh] = den > 0.f ? mm + logf(den) : -INFINITY;
}

template <int D>
int launch_decode(const DecodeLaunch &a)
{
    const int bh = a.B * a.H;
    decode_partial<D><<<static_cast<unsigned>(bh) * a.splits, kDecThreads, 0, a.stream>>>(
        static_cast<const __nv_bfloat16 *>(a.q), static_cast<const __nv_bfloat16 *>(a.k),
        static_cast<const __nv_bfloat16 *>(a.v), a.cache_lens, a.H, a.L, a.L_keys, a.splits, a.chunk, a.scale_log2,
        a.part_o,
        a.part_lse);
    if (cudaGetLastError() != cudaSuccess) return -1;
    decode_combine<D><<<bh, D, 0, a.stream>>>(a.part_o, a.part_lse, a.splits, static_cast<__nv_bfloat16 *>(a.out),
                                               a.lse);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

// Streaming multiprocessors of the current device (148 on a B300 when no
// device can be queried, e.g. for a size query on a host without a GPU).
int sm_count()
{
    constexpr int kMaxDevices = 64;
    static int cached[kMaxDevices] = {};  // 0 = not queried yet (benign race: every writer stores the same value)
    int dev = -1, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();  // the failed query must not surface at the next launch
        return 148;
    }
    if (dev >= 0 && dev < kMaxDevices && cached[dev] > 0) return cached[dev];
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return 148;
    }
    if (dev >= 0 && dev < kMaxDevices) cached[dev] = n;
    return n;
}

DecodeSplit decode_split(int B, int H, int L)
{
    // Enough CTAs for every SM to keep many 16-byte loads in flight: about
    // sixteen per SM, each split at least 256 keys, chunks a multiple of 64.
    const int64_t heads = static_cast<int64_t>(B) * H;
    const int64_t target = static_cast<int64_t>(sm_count()) * 16;
    int64_t splits = (target + heads - 1) / heads;
    const int64_t max_splits = (static_cast<int64_t>(L) + 255) / 256;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    int64_t chunk = (static_cast<int64_t>(L) + splits - 1) / splits;
    chunk = (chunk + 63) / 64 * 64;
    splits = (static_cast<int64_t>(L) + chunk - 1) / chunk;
    if (splits < 1) splits = 1;
    return {static_cast<int>(splits), static_cast<int>(chunk)};
}

int attn_decode_launch(const DecodeLaunch &a)
{
    if (a.d == 64) return launch_decode<64>(a);
    if (a.d == 128) return launch_decode<128>(a);
    return -2;
}

}  // namespace sdp18

// ---------------------------------------------------------------------------
// attn_decode_noalloc: attn_decode on a workspace the library owns.
//
// Some callers cannot allocate device memory once they are running: a serving
// or real-time loop that fixed its memory budget at start-up, a host
// application that hands this library a stream but no allocator, or code that
// must not pay cudaMalloc's implicit device synchronisation on every step.
// For them the split partials live in one fixed array of device memory that
// is part of the loaded library.  Its device address is looked up once per
// device (the first call on that device does it), and each call then passes
// that address as the workspace of attn_decode.
namespace sdp18 {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr int kMaxDevices = 64;

// Lives on every device that loads the library, for as long as the process
// runs.  Host code may not use this name as a pointer: on the host it only
// identifies the symbol, so its device address is fetched below.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Process-unique id of the current CUDA context (0 if it cannot be read).
// cudaDeviceReset destroys a device's primary context and reloads the
// library's module in the next one, which moves g_decode_scratch; context ids
// are never reused, so a cached address is valid only for the id it was
// taken under.
unsigned long long current_context_id()
{
    static std::once_flag once;
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of g_decode_scratch on the current device, or nullptr.  The
// address is looked up once per device and context (the first call after the
// device's context was created does it) and cached.
void *static_scratch()
{
    static std::mutex mu;
    static void *addr[kMaxDevices] = {};
    static unsigned long long ctx_id[kMaxDevices] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    const unsigned long long id = current_context_id();  // 0 before the thread's first CUDA call
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr || id == 0 || ctx_id[dev] != id) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
        addr[dev] = p;
        ctx_id[dev] = current_context_id();  // the lookup has made the device's context current
    }
    return addr[dev];
}

}  // namespace
}  // namespace sdp18

extern "C" attn_status attn_decode_noalloc(const void *q, const void *k_cache, const void *v_cache, void *out,
                                           float *lse, int B, int H, int L, int d, float scale,
                                           const int32_t *cache_lens, attn_stream_t stream)
{
    // attn_decode's own argument checks come first, so that both entry points
    // return the same status for the same bad argument; only a valid problem
    // that does not fit the fixed area gets ATTN_ETOOLARGE.
    if (B < 0 || H < 0 || L < 0) return ATTN_EINVAL;
    if (d != 64 && d != 128) return ATTN_EUNSUPPORTED;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_EINVAL;
    if (B == 0 || H == 0) return ATTN_OK;
    if (!q || !out) return ATTN_EINVAL;
    if (static_cast<int64_t>(B) * H > INT32_MAX / 64) return ATTN_EINVAL;
    if (L > 0 && (!k_cache || !v_cache)) return ATTN_EINVAL;
    const size_t need = attn_decode_workspace_size(B, H, L > 0 ? L : 1, d);
    if (need == 0) return ATTN_EINVAL;
    if (need > sdp18::kStaticScratchBytes) return ATTN_ETOOLARGE;
    void *ws = sdp18::static_scratch();
    if (ws == nullptr) return ATTN_ECUDA;
    // Nothing in the workspace needs to start at zero: every split writes all
    // of its partial slots before the combine kernel reads them.
    return attn_decode(q, k_cache, v_cache, out, lse, B, H, L, d, scale, cache_lens, ws, sdp18::kStaticScratchBytes,
                       stream);
}
