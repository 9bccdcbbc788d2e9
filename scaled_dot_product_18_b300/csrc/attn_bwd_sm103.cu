// Attention backward for B300 (sm_103a): dQ, dK, dV of the forward in
// attn_fwd_sm103.cu, recomputing P from the saved log-sum-exp instead of
// storing it (the pages reuse the forward's softmax statistics in the
// backward pass, hotelren.com "AI attention: essence and evolution",
// sec. 4.2).
//
// With S = scale Q K^T, P = softmax(S), O = P V and the loss gradient dO:
//   dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij = dO_i . O_i,
//   dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q.
//
// One CTA owns a 128-key tile of one (batch, head) and walks the query tiles
// that can see it (all of them, or those at or after the diagonal when
// causal, and with a sliding window of w positions -- query i sees keys
// j > i - w -- only those before query k0 + 127 + w).  Per query tile, in tensor memory (512 columns):
//   S^T = K Q_i^T          columns   0..127  (keys in TMEM lanes, queries in columns)
//   dP^T = V dO_i^T        columns 128..255, later dQ_i = dS K (queries in lanes)
//   P^T -> bf16 packed over columns 0..31 and 64..95 of S^T, dS^T over
//          columns 32..63 and 96..127 (each half of the compute warps
//          overwrites only columns it has read): the TMEM A operands of
//          dV += P^T dO_i and dK += dS^T Q_i
//   dS^T -> also bf16 in shared memory, the A operand of the dQ MMA
//   dV, dK accumulate in columns 256.. across the query tiles.
// The MMA order per tile is S, dP, dV, dK, dQ: S^T is issued as soon as the
// previous tile's dQ MMAs are queued, the compute warps turn S^T into P while
// dP^T is being computed, and dS while dV is.  Four dQ warps take dQ_i out of
// tensor memory, stage it (times scale, fp32) in the (Q_i, dO_i) ring stage
// that the tile's MMAs have finished with, and add it to an fp32 accumulator
// in global memory with TMA reductions; they then hand the stage back to the
// producer.  This keeps the accumulation off the compute warps' path.  A
// pre-pass computes D and the scaled LSE and clears the accumulator; a
// post-pass converts it to bf16.
//
//   warps 0-7   compute: warp w serves key rows 32 (w % 4) .. +31 (its TMEM
//               lanes) and query columns 64 (w / 4) .. +63: P^T, dS^T; at
//               the end dK and dV for head-dim half w / 4.
//   warps 8-11  dQ: query rows 32 (w % 4) .. +31 of dQ_i.
//   warp 12     TMA producer: K, V once; (Q_i, dO_i, LSE, D) through a 2-stage ring.
//   warp 13     allocates TMEM and issues the five MMAs of each query tile.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "attn_internal.h"
#include "ptx_sm103.cuh"

namespace sdp18 {

// Device error word of the backward kernel (each translation unit keeps its own
// word: the library is built without relocatable device code).
__device__ int g_sdp18_bwd_error = 0;

namespace {

constexpr int kKeys = 128;    // keys per CTA
constexpr int kQTile = 128;   // queries per step
constexpr int kCompute = 8;   // compute warps
constexpr int kDqWarp0 = kCompute;  // 4 dQ warps
constexpr int kTmaWarp = kCompute + 4;
constexpr int kMmaWarp = kCompute + 5;
constexpr int kThreads = (kCompute + 6) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTS = 0, kTDP = 128, kTDV = 256;  // dK at kTDV + D
constexpr float kLog2e = 1.4426950408889634f;
enum : int { kErrSmemAlign = 4 };

template <int D>
struct BwdSmem {
    static constexpr int kTileBytes = 128 * D * 2;  // one [128 x D] bf16 tile
    static constexpr int kStages = 2;               // (Q_i, dO_i, stats) stages
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kTileBytes;
    static constexpr int kOffRing = kOffV + kTileBytes;  // stage s: Q at +0, dO at +kTileBytes
    static constexpr int kOffDS = kOffRing + kStages * 2 * kTileBytes;  // [128 keys x 128 q] bf16
    static constexpr int kOffStat = kOffDS + kKeys * kQTile * 2;      // stage s: lse*log2e [128], D [128]
    static constexpr int kStatBytes = 2 * kQTile * 4;
    static constexpr int kOffBar = kOffStat + kStages * kStatBytes;
    static constexpr int kBarKV = 0;
    static constexpr int kBarFull = 1;                    // [kStages]
    static constexpr int kBarEmpty = kBarFull + kStages;  // [kStages]
    static constexpr int kBarS = kBarEmpty + kStages;
    static constexpr int kBarDP = kBarS + 1;
    static constexpr int kBarP = kBarDP + 1;
    static constexpr int kBarDS = kBarP + 1;
    static constexpr int kBarDQ = kBarDS + 1;
    static constexpr int kBarDQUsed = kBarDQ + 1;
    static constexpr int kBarDKV = kBarDQUsed + 1;
    static constexpr int kBarDrain = kBarDKV + 1;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kBytes = kOffMisc + 16;
    static_assert(kBytes <= 227 * 1024, "shared memory budget");
    static_assert(kTDV + 2 * D <= kTmemCols, "TMEM budget");
    // dQ_i (128 x D fp32) is staged in one ring stage: 32 x 32 boxes of 4 KB.
    static_assert(128 * D * 4 <= 2 * kTileBytes, "dQ staging fits a ring stage");
};

__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk)
{
    return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ld_shared_v4f(uint32_t addr, float &a, float &b, float &c, float &d)
{
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(a), "=f"(b), "=f"(c), "=f"(d) : "r"(addr));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const float *__restrict__ stats,
                    __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv,
                    const int32_t *__restrict__ key_lens, int H, int N, int n_tiles, int num_bh, int head_group,
                    float scale, float scale_log2, int causal, int window)
{
    using L = BwdSmem<D>;
    // The tiles are 128-byte swizzled and need a 1024-byte aligned base.  The
    // check is uniform over the CTA, before any barrier or TMEM is touched.
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t s_base = smem_addr(smem);
    if (s_base & 1023u) {
        if (threadIdx.x == 0) atomicOr(&g_sdp18_bwd_error, kErrSmemAlign);
        return;
    }
    const uint32_t sK = s_base + L::kOffK, sV = s_base + L::kOffV, sDS = s_base + L::kOffDS;
    auto sQ = [&](int st) -> uint32_t { return s_base + L::kOffRing + st * 2 * L::kTileBytes; };
    auto sDO = [&](int st) -> uint32_t { return sQ(st) + L::kTileBytes; };
    auto sStat = [&](int st) -> uint32_t { return s_base + L::kOffStat + st * L::kStatBytes; };
    auto bar = [&](int i) -> uint32_t { return s_base + L::kOffBar + 8 * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Key tiles in ascending order (the first ones see the most query tiles
    // when causal), all heads of one key tile together -- within groups of
    // head_group heads (all heads in one group unless the host chose smaller
    // groups so that a group's q, k, v and dO stay in L2).
    const int per_group = head_group * n_tiles;
    const int grp = static_cast<int>(blockIdx.x / per_group);
    const int g_heads = min(head_group, num_bh - grp * head_group);
    const int in_grp = static_cast<int>(blockIdx.x) - grp * per_group;
    const int bh = grp * head_group + in_grp % g_heads;
    const int kt = in_grp / g_heads;
    const int b = bh / H, h = bh % H;
    int kv_len = N;
    if (key_lens != nullptr) kv_len = min(max(key_lens[b], 0), N);
    const int k0 = kt * kKeys;
    // Query tiles this key tile meets: from the diagonal when causal, up to
    // the last query whose window reaches the tile's last visible key.
    const int i_first = (causal && k0 < kv_len) ? kt : 0;
    int i_last = n_tiles - 1;
    if (window > 0 && k0 < kv_len) {
        const int64_t i_max = static_cast<int64_t>(min(k0 + kKeys, kv_len) - 1) + window - 1;
        i_last = static_cast<int>(i_max / kQTile < i_last ? i_max / kQTile : i_last);
    }
    const int n_q = k0 < kv_len ? max(0, i_last - i_first + 1) : 0;
    const int n_pad = n_tiles * kQTile;

    if (threadIdx.x == 0) {
        mbar_init(bar(L::kBarKV), 1);
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(bar(L::kBarFull + s), 1);
            mbar_init(bar(L::kBarEmpty + s), 4 * 32);  // the dQ warps release a stage
        }
        mbar_init(bar(L::kBarS), 1);
        mbar_init(bar(L::kBarDP), 1);
        mbar_init(bar(L::kBarP), kCompute * 32);
        mbar_init(bar(L::kBarDS), kCompute * 32);
        mbar_init(bar(L::kBarDQ), 1);
        mbar_init(bar(L::kBarDQUsed), 4 * 32);
        mbar_init(bar(L::kBarDKV), 1);
        mbar_init(bar(L::kBarDrain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto wait_warp = [&](uint32_t b_addr, uint32_t parity, int site) -> bool {
        return __all_sync(0xffffffffu, wait_bounded(b_addr, parity, abort_flag, site, &g_sdp18_bwd_error));
    };

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ producer
        if (n_q > 0) {
            mbar_arrive_expect_tx_one(bar(L::kBarKV), 2 * L::kTileBytes);
            for (int cb = 0; cb < D / 64; ++cb) {
                tma_load_4d_one(sK + cb * 128 * 128, &tm_k, bar(L::kBarKV), cb * 64, k0, h, b);
                tma_load_4d_one(sV + cb * 128 * 128, &tm_v, bar(L::kBarKV), cb * 64, k0, h, b);
            }
            const float *lse2 = stats + static_cast<int64_t>(bh) * n_pad;
            const float *dvec = stats + static_cast<int64_t>(num_bh) * n_pad + static_cast<int64_t>(bh) * n_pad;
            int issued = 0;
            for (int ii = 0; ii < n_q; ++ii) {
                const int st = ii % L::kStages;
                if (!wait_warp(bar(L::kBarEmpty + st), ((ii / L::kStages) & 1) ^ 1, 20)) break;
                const int q0 = (i_first + ii) * kQTile;
                mbar_arrive_expect_tx_one(bar(L::kBarFull + st), 2 * L::kTileBytes + L::kStatBytes);
                for (int cb = 0; cb < D / 64; ++cb) {
                    tma_load_4d_one(sQ(st) + cb * 128 * 128, &tm_q, bar(L::kBarFull + st), cb * 64, q0, h, b);
                    tma_load_4d_one(sDO(st) + cb * 128 * 128, &tm_do, bar(L::kBarFull + st), cb * 64, q0, h, b);
                }
                bulk_load_one(sStat(st), lse2 + q0, kQTile * 4, bar(L::kBarFull + st));
                bulk_load_one(sStat(st) + kQTile * 4, dvec + q0, kQTile * 4, bar(L::kBarFull + st));
                ++issued;
            }
            wait_drain(bar(L::kBarKV), 0);
            for (int i = max(0, issued - L::kStages); i < issued; ++i)
                wait_drain(bar(L::kBarFull + i % L::kStages), (i / L::kStages) & 1);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (n_q > 0) {
            const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
            constexpr uint32_t kIdS = idesc_bf16_f32_mn(kKeys, kQTile, false, false);  // S^T, dP^T
            constexpr uint32_t kIdKV = idesc_bf16_f32_mn(kKeys, D, false, true);       // dV, dK
            constexpr uint32_t kIdQ = idesc_bf16_f32_mn(kQTile, D, true, true);        // dQ
            bool ok = wait_warp(bar(L::kBarKV), 0, 21);
            for (int ii = 0; ii < n_q && ok; ++ii) {
                const int st = ii % L::kStages;
                ok = wait_warp(bar(L::kBarFull + st), (ii / L::kStages) & 1, 22);
                if (!ok) break;
                tc_fence_after();
                // S^T = K Q_i^T (keys x queries, K = D).  The previous tile's P^T
                // and dS^T in these columns were consumed by its dV and dK MMAs,
                // queued earlier.
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
                    mma_bf16_ss_one(tm + kTS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ(st) + off, 16, 1024),
                                    kIdS, kk > 0 ? 1u : 0u);
                }
                mma_commit_one(bar(L::kBarS));
                // dP^T = V dO_i^T overwrites dQ_{i-1}: wait until it has been read.
                if (ii > 0 && !(ok = wait_warp(bar(L::kBarDQUsed), (ii - 1) & 1, 23))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
                    mma_bf16_ss_one(tm + kTDP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO(st) + off, 16, 1024),
                                    kIdS, kk > 0 ? 1u : 0u);
                }
                mma_commit_one(bar(L::kBarDP));
                if (!(ok = wait_warp(bar(L::kBarP), ii & 1, 24))) break;
                tc_fence_after();
                // dV += P^T dO_i: A = P^T from TMEM (16 queries = 8 packed
                // columns per step; queries 64.. start at column 64), B = dO_i
                // query-major (N = D).
#pragma unroll
                for (int kk = 0; kk < kQTile / 16; ++kk)
                    mma_bf16_ts_one(tm + kTDV, tm + kTS + (kk >> 2) * 64 + (kk & 3) * 8,
                                    sdesc_sw128(sDO(st) + kk * 16 * 128, 128 * 128, 1024), kIdKV,
                                    (ii > 0 || kk > 0) ? 1u : 0u);
                if (!(ok = wait_warp(bar(L::kBarDS), ii & 1, 25))) break;
                tc_fence_after();
                // dK += dS^T Q_i: A = dS^T from TMEM (packed next to P^T), B = Q_i query-major.
#pragma unroll
                for (int kk = 0; kk < kQTile / 16; ++kk)
                    mma_bf16_ts_one(tm + kTDV + D, tm + kTS + 32 + (kk >> 2) * 64 + (kk & 3) * 8,
                                    sdesc_sw128(sQ(st) + kk * 16 * 128, 128 * 128, 1024), kIdKV,
                                    (ii > 0 || kk > 0) ? 1u : 0u);
                // dQ_i = dS K: A = dS^T read query-major (M = queries), B = K key-major (N = D).
#pragma unroll
                for (int kk = 0; kk < kKeys / 16; ++kk)
                    mma_bf16_ss_one(tm + kTDP, sdesc_sw128(sDS + kk * 16 * 128, 128 * 128, 1024),
                                    sdesc_sw128(sK + kk * 16 * 128, 128 * 128, 1024), kIdQ, kk > 0 ? 1u : 0u);
                mma_commit_one(bar(L::kBarDQ));
            }
            if (ok) mma_commit_one(bar(L::kBarDKV));
            mma_commit_one(bar(L::kBarDrain));
            wait_drain(bar(L::kBarDrain), 0);
        }
    } else if (warp >= kDqWarp0) {
        // ------------------------------------------------------------ dQ warps
        const int g = warp & 3;  // TMEM lane quarter = query rows 32g..32g+31 of the tile
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * g) << 16);
        bool ok = true;
        for (int ii = 0; ii < n_q && ok; ++ii) {
            const int st = ii % L::kStages;
            const int qrow = (i_first + ii) * kQTile + 32 * g;
            if (!wait_warp(bar(L::kBarDQ), ii & 1, 26)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // The tile's dV and dK MMAs, which read this stage, finished before
            // dQ_i did: stage this warp's 32 x D block there as D/32 boxes.
            const uint32_t s_box = sQ(st) + g * (D / 32) * 4096;
#pragma unroll 1
            for (int j = 0; j < D / 32; ++j) {
                uint32_t o[32];
                tmem_ld32(t_lane + kTDP + 32 * j, o);
                tmem_ld_wait(o);
                if (j == D / 32 - 1) {
                    tc_fence_before();
                    mbar_arrive(bar(L::kBarDQUsed));
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    st_shared_v4(s_box + j * 4096 + sw128_offset(lane, u),
                                 __float_as_uint(scale * __uint_as_float(o[4 * u])),
                                 __float_as_uint(scale * __uint_as_float(o[4 * u + 1])),
                                 __float_as_uint(scale * __uint_as_float(o[4 * u + 2])),
                                 __float_as_uint(scale * __uint_as_float(o[4 * u + 3])));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && qrow < N) {
                for (int j = 0; j < D / 32; ++j) tma_reduce_add_3d(&tm_dq, s_box + j * 4096, 32 * j, qrow, bh);
                tma_store_commit();
            }
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            mbar_arrive(bar(L::kBarEmpty + st));
        }
        // Every reduction issued by this warp has completed (not only read).
        if (lane == 0) tma_store_wait_all();
        __syncwarp();
        tc_fence_before();
    } else {
        // ------------------------------------------------------------ compute warps
        const int g = warp & 3;   // TMEM lane quarter: key rows 32g..32g+31
        const int hf = warp >> 2;  // query-column half (P, dS) and head-dim half (dK, dV)
        const int r = 32 * g + lane;  // key row == TMEM lane
        const int kj = k0 + r;
        const bool key_ok = kj < kv_len;
        const bool tail_keys = k0 + kKeys > kv_len;  // some key of this tile is hidden
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * g) << 16);
        // This warp's 4 KB of the dS^T buffer (its key rows, its query half).
        const uint32_t s_mine = sDS + hf * (128 * 128) + g * 4096;
        bool ok = true;
        for (int ii = 0; ii < n_q && ok; ++ii) {
            const int st = ii % L::kStages;
            const int q0 = (i_first + ii) * kQTile;
            // per-element visibility needed: hidden keys, the diagonal, or
            // queries past some key's window (i >= j + w) in this tile
            const bool masked = tail_keys || (causal && q0 == k0) || (window > 0 && q0 + kQTile - 1 - k0 >= window);
            // S_i done implies the previous tile's MMAs (dK, dQ reading dS^T) are done.
            if (!wait_warp(bar(L::kBarFull + st), (ii / L::kStages) & 1, 27) || !wait_warp(bar(L::kBarS), ii & 1, 28)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // P^T = exp2(S^T * scale*log2e - lse*log2e) over this warp's 64
            // query columns, 16 at a time; fp32 kept for dS, bf16 into TMEM.
            float p[64];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int c0 = 64 * hf + 16 * c;  // first query column of the step
                uint32_t sv[16];
                tmem_ld16(t_lane + kTS + c0, sv);
                float l2[16];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    ld_shared_v4f(sStat(st) + (c0 + 4 * e) * 4, l2[4 * e], l2[4 * e + 1], l2[4 * e + 2], l2[4 * e + 3]);
                tmem_ld_wait_only();
                reg_fence16(sv);
                if (!masked) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) p[16 * c + e] = ex2(fmaf(__uint_as_float(sv[e]), scale_log2, -l2[e]));
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int qi = q0 + c0 + e;
                        const bool vis = key_ok && (!causal || qi >= kj) && (window <= 0 || qi - kj < window);
                        p[16 * c + e] = vis ? ex2(fmaf(__uint_as_float(sv[e]), scale_log2, -l2[e])) : 0.f;
                    }
                }
                uint32_t pk[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) pk[e] = pack_bf16x2(p[16 * c + 2 * e], p[16 * c + 2 * e + 1]);
                tmem_st8(t_lane + kTS + 64 * hf + 8 * c, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(L::kBarP));
            if (!wait_warp(bar(L::kBarDP), ii & 1, 29)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // dS^T = P^T (dP^T - D) -> bf16: into TMEM next to P^T and, swizzled
            // keys x queries, into shared memory.
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int c0 = 64 * hf + 16 * c;
                uint32_t dpv[16];
                tmem_ld16(t_lane + kTDP + c0, dpv);
                float dd[16];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    ld_shared_v4f(sStat(st) + kQTile * 4 + (c0 + 4 * e) * 4, dd[4 * e], dd[4 * e + 1], dd[4 * e + 2],
                                  dd[4 * e + 3]);
                tmem_ld_wait_only();
                reg_fence16(dpv);
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    w[e] = pack_bf16x2(p[16 * c + 2 * e] * (__uint_as_float(dpv[2 * e]) - dd[2 * e]),
                                       p[16 * c + 2 * e + 1] * (__uint_as_float(dpv[2 * e + 1]) - dd[2 * e + 1]));
                tmem_st8(t_lane + kTS + 32 + 64 * hf + 8 * c, w);
                const int c16 = 2 * c;  // 16-byte chunk within the half's 128-byte row
                st_shared_v4(s_mine + sw128_offset(lane, c16), w[0], w[1], w[2], w[3]);
                st_shared_v4(s_mine + sw128_offset(lane, c16 + 1), w[4], w[5], w[6], w[7]);
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(L::kBarDS));
        }
        // ------------------------------------------------------------ dK, dV
        // Warp-uniform: TMEM loads are collective; only the stores depend on
        // the row.  Rows of hidden keys hold exact zeros.
        const bool have = ok && n_q > 0 && wait_warp(bar(L::kBarDKV), 0, 30);
        if (have) tc_fence_after();
        if (ok) {
            __nv_bfloat16 *pdv = dv + (static_cast<int64_t>(bh) * N + kj) * D + hf * (D / 2);
            __nv_bfloat16 *pdk = dk + (static_cast<int64_t>(bh) * N + kj) * D + hf * (D / 2);
#pragma unroll 1
            for (int c = 0; c < D / 64; ++c) {
                uint32_t a[32], gk[32];
                if (have) {
                    tmem_ld32(t_lane + kTDV + hf * (D / 2) + 32 * c, a);
                    tmem_ld32(t_lane + kTDV + D + hf * (D / 2) + 32 * c, gk);
                    tmem_ld_wait_only();
                    reg_fence(a);
                    reg_fence(gk);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) a[e] = gk[e] = 0u;
                }
                if (kj < N) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        uint4 wv, wk;
                        wv.x = pack_bf16x2(__uint_as_float(a[8 * u + 0]), __uint_as_float(a[8 * u + 1]));
                        wv.y = pack_bf16x2(__uint_as_float(a[8 * u + 2]), __uint_as_float(a[8 * u + 3]));
                        wv.z = pack_bf16x2(__uint_as_float(a[8 * u + 4]), __uint_as_float(a[8 * u + 5]));
                        wv.w = pack_bf16x2(__uint_as_float(a[8 * u + 6]), __uint_as_float(a[8 * u + 7]));
                        wk.x = pack_bf16x2(scale * __uint_as_float(gk[8 * u + 0]), scale * __uint_as_float(gk[8 * u + 1]));
                        wk.y = pack_bf16x2(scale * __uint_as_float(gk[8 * u + 2]), scale * __uint_as_float(gk[8 * u + 3]));
                        wk.z = pack_bf16x2(scale * __uint_as_float(gk[8 * u + 4]), scale * __uint_as_float(gk[8 * u + 5]));
                        wk.w = pack_bf16x2(scale * __uint_as_float(gk[8 * u + 6]), scale * __uint_as_float(gk[8 * u + 7]));
                        *reinterpret_cast<uint4 *>(pdv + 32 * c + 8 * u) = wv;
                        *reinterpret_cast<uint4 *>(pdk + 32 * c + 8 * u) = wk;
                    }
                }
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Per (head, padded query row): lse*log2e (+inf for a row with no visible key
// or past N, so that exp2 gives P = 0), D_i = dO_i . O_i (0 past N), and the
// row of the dQ accumulator cleared.  D/8 threads per row.
template <int D>
__global__ void __launch_bounds__(256) bwd_prepare(const __nv_bfloat16 *__restrict__ out,
                                                   const __nv_bfloat16 *__restrict__ dout,
                                                   const float *__restrict__ lse, float *__restrict__ stats,
                                                   float *__restrict__ dqacc, int N, int n_pad, int64_t rows_pad)
{
    constexpr int kSeg = D / 8;
    const int64_t prow = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) / kSeg;
    const int seg = threadIdx.x % kSeg;
    const int64_t bh = prow / n_pad;
    const int q = static_cast<int>(prow - bh * n_pad);
    const bool live = prow < rows_pad && q < N;
    const int64_t row = bh * N + q;
    float acc = 0.f;
    if (live) {
        const uint4 o = *reinterpret_cast<const uint4 *>(out + row * D + seg * 8);
        const uint4 gv = *reinterpret_cast<const uint4 *>(dout + row * D + seg * 8);
        const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc = fmaf(__uint_as_float(ow[i] << 16), __uint_as_float(gw[i] << 16), acc);
            acc = fmaf(__uint_as_float(ow[i] & 0xFFFF0000u), __uint_as_float(gw[i] & 0xFFFF0000u), acc);
        }
        float4 *z = reinterpret_cast<float4 *>(dqacc + row * D + seg * 8);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int off = kSeg / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (prow < rows_pad && seg == 0) {
        float l2 = INFINITY;
        if (live) {
            const float v = lse[row];
            if (v > -INFINITY) l2 = v * kLog2e;
        }
        stats[prow] = l2;
        stats[rows_pad + prow] = acc;
    }
}

__global__ void __launch_bounds__(256) bwd_finish(const float *__restrict__ dqacc, __nv_bfloat16 *__restrict__ dq,
                                                  int64_t n4)
{
    const int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
    if (i >= n4) return;
    const float4 v = reinterpret_cast<const float4 *>(dqacc)[i];
    uint2 w;
    w.x = pack_bf16x2(v.x, v.y);
    w.y = pack_bf16x2(v.z, v.w);
    reinterpret_cast<uint2 *>(dq)[i] = w;
}

template <int D>
int launch_bwd(const BwdLaunch &a)
{
    using L = BwdSmem<D>;
    static int configured_device = -1;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (configured_device != dev) {
        if (cudaFuncSetAttribute(attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes) !=
            cudaSuccess)
            return -1;
        configured_device = dev;
    }
    const int n_tiles = (a.N + 127) / 128;
    const int num_bh = a.B * a.H;
    const int n_pad = n_tiles * 128;
    const int64_t rows_pad = static_cast<int64_t>(num_bh) * n_pad;
    const int64_t seg_threads = rows_pad * (D / 8);
    bwd_prepare<D><<<static_cast<unsigned>((seg_threads + 255) / 256), 256, 0, a.stream>>>(
        static_cast<const __nv_bfloat16 *>(a.out), static_cast<const __nv_bfloat16 *>(a.dout), a.lse, a.stats,
        a.dqacc, a.N, n_pad, rows_pad);
    if (cudaGetLastError() != cudaSuccess) return -1;
    // With key tile 0 of every head first, the running CTAs spread over all
    // heads: each streams its own head's Q and dO and adds into its own rows
    // of the fp32 dQ accumulator, a working set far above L2 (B=4 H=32
    // N=4096: ~148 heads; B=1 H=32 N=16384: 32 heads of 16 MiB plus 268 MB of
    // accumulator).  Groups of heads whose q, k, v and dO fit 64 MiB keep
    // most of it in L2: 2.17 -> 1.58 ms and 5.18 -> 4.79 ms on those shapes
    // (2032 MHz).
    const int64_t per_head = static_cast<int64_t>(a.N) * D * 2 * 4;
    const int head_group =
        static_cast<int>(std::min<int64_t>(num_bh, std::max<int64_t>(1, (int64_t(64) << 20) / per_head)));
    attn_bwd_kernel<D><<<static_cast<unsigned>(n_tiles) * num_bh, kThreads, L::kBytes, a.stream>>>(
        *a.tm_q, *a.tm_k, *a.tm_v, *a.tm_do, *a.tm_dq, a.stats, static_cast<__nv_bfloat16 *>(a.dk),
        static_cast<__nv_bfloat16 *>(a.dv), a.key_lens, a.H, a.N, n_tiles, num_bh, head_group, a.scale,
        a.scale * kLog2e, a.causal, a.window);
    if (cudaGetLastError() != cudaSuccess) return -1;
    const int64_t n4 = static_cast<int64_t>(num_bh) * a.N * D / 4;
    bwd_finish<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, a.stream>>>(a.dqacc,
                                                                            static_cast<__nv_bfloat16 *>(a.dq), n4);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int attn_bwd_launch(const BwdLaunch &a)
{
    if (a.d == 64) return launch_bwd<64>(a);
    if (a.d == 128) return launch_bwd<128>(a);
    return -2;
}

int read_and_clear_bwd_error(int *value)
{
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_sdp18_bwd_error, sizeof(int)) != cudaSuccess) return -1;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_sdp18_bwd_error, &zero, sizeof(int)) != cudaSuccess) return -1;
    }
    *value = v;
    return 0;
}

}  // namespace sdp18
