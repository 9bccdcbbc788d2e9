// Attention forward for B300 (sm_103a): one CTA per 128-row query tile.
//
// The method is the tiled forward with an online softmax (hotelren.com "AI
// attention: essence and evolution", sec. 4.1, FlashAttention-1): for a query
// tile, stream the key/value tiles, form S = Q K^T for the pair, fold it
// into running row statistics (max, sum), accumulate P V, and never write S
// out.  Tiles that the causal mask hides completely are not visited
// (hotelren.com sec. 5, "only load active K/V blocks").
//
// How it maps onto sm_103a:
//   warp 4       TMA producer: Q once, then K_j, V_j through a ring of
//                shared-memory slots guarded by full/empty mbarriers.
//   warp 5       allocates tensor memory (TMEM) and, from one thread, issues
//                every tcgen05.mma: S_j = Q K_j^T into one of two fp32 TMEM
//                buffers (so S_{j+1} is computed while S_j is in softmax),
//                then O += P_j V_j into an fp32 TMEM accumulator.
//   warps 0-3    softmax: thread t owns query row t of the tile (TMEM lane
//                t), so every row reduction stays inside one thread.  They
//                read S_j from TMEM, mask, take the running max in the log2
//                domain, exponentiate with ex2, write P_j as bf16 into shared
//                memory for the second MMA, rescale O in TMEM when the max
//                moved far enough, and finally write O / l (bf16, via a TMA
//                store) and the natural-log LSE.
//
// Memory layout (all 128-byte swizzled, 1024-byte aligned tiles):
//   Q tile   : d/64 column blocks of [128 rows x 64 bf16]; reused to stage O
//   P tile   : 2 column blocks of [128 query rows x 64 keys] bf16
//   K/V ring : NSLOT slots of d/64 blocks of [128 keys x 64 bf16]
// TMEM (512 columns): S buffers at columns 0 and 128, O at column 256.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "attn_internal.h"
#include "ptx_sm103.cuh"

namespace sdp18 {

// Device error word of this library (read and cleared by the host).
__device__ int g_sdp18_error = 0;

namespace {

constexpr int kBM = 128;           // query rows per tile
constexpr int kBN = 128;           // keys per tile
constexpr int kThreads = 192;      // 4 softmax warps + TMA warp + MMA warp
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS0 = 0, kTmemO = 256;
// Lazy rescaling: the running max used for P only moves when a row's true max
// exceeds it by more than 2^8, so P stays <= 256 and O/l need a rescale only
// rarely.  Exact: O and l always share the same stale max.
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct Smem {
    static constexpr int kNumSlots = 4;
    static constexpr int kQBytes = kBM * D * 2;
    static constexpr int kPBytes = kBM * kBN * 2;
    static constexpr int kKVBytes = kBN * D * 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffP = kOffQ + kQBytes;
    static constexpr int kOffRing = kOffP + kPBytes;
    static constexpr int kOffBar = kOffRing + kNumSlots * kKVBytes;
    // barriers: q_full, full[S], empty[S], s_full[2], s_free[2], p_full, pv_done, mma_drain
    static constexpr int kBarQFull = 0;
    static constexpr int kBarFull = 1;
    static constexpr int kBarEmpty = kBarFull + kNumSlots;
    static constexpr int kBarSFull = kBarEmpty + kNumSlots;
    static constexpr int kBarSFree = kBarSFull + 2;
    static constexpr int kBarPFull = kBarSFree + 2;
    static constexpr int kBarPVDone = kBarPFull + 1;
    static constexpr int kBarDrain = kBarPVDone + 1;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem address, abort flag
    static constexpr int kBytes = kOffMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024
};

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside one
// [rows x 64 bf16] block with the 128-byte swizzle: chunk index XOR (row % 8).
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk)
{
    return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    float *__restrict__ lse, const int32_t *__restrict__ key_lens, int H, int N, int num_q_tiles,
                    int num_bh, float scale_log2, int causal)
{
    using L = Smem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_addr(smem);
    const uint32_t sQ = s_base + L::kOffQ;
    const uint32_t sP = s_base + L::kOffP;
    const uint32_t sRing = s_base + L::kOffRing;
    auto bar = [&](int i) -> uint32_t { return s_base + L::kOffBar + 8 * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Heaviest causal tiles (largest query index) first: the tile grid is
    // ordered by descending query tile, all heads of one query tile together.
    const int bh = blockIdx.x % num_bh;
    const int qt = num_q_tiles - 1 - static_cast<int>(blockIdx.x / num_bh);
    const int q0 = qt * kBM;
    const int b = bh / H;
    int kv_len = N;
    if (key_lens != nullptr) kv_len = min(max(key_lens[b], 0), N);
    const int kv_end = causal ? min(kv_len, q0 + kBM) : kv_len;
    const int n_kv = (kv_end + kBN - 1) / kBN;

    if (threadIdx.x == 0) {
        mbar_init(bar(L::kBarQFull), 1);
        for (int s = 0; s < L::kNumSlots; ++s) {
            mbar_init(bar(L::kBarFull + s), 1);
            mbar_init(bar(L::kBarEmpty + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(L::kBarSFull + s), 1);
            mbar_init(bar(L::kBarSFree + s), 4 * 32);
        }
        mbar_init(bar(L::kBarPFull), 4 * 32);
        mbar_init(bar(L::kBarPVDone), 1);
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

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && n_kv > 0) {
            tma_prefetch_map(&tm_q);
            tma_prefetch_map(&tm_k);
            tma_prefetch_map(&tm_v);
            mbar_arrive_expect_tx(bar(L::kBarQFull), L::kQBytes);
            for (int cb = 0; cb < D / 64; ++cb) tma_load_3d(sQ + cb * kBM * 128, &tm_q, bar(L::kBarQFull), cb * 64, q0, bh);
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < n_kv && ok; ++j) {
                for (int which = 0; which < 2; ++which) {
                    const int item = 2 * j + which;
                    const int s = item % L::kNumSlots;
                    const uint32_t round = static_cast<uint32_t>(item / L::kNumSlots);
                    if (!wait_bounded(bar(L::kBarEmpty + s), (round & 1) ^ 1, abort_flag, 1, &g_sdp18_error)) {
                        ok = false;
                        break;
                    }
                    const CUtensorMap *map = which ? &tm_v : &tm_k;
                    const uint32_t dst = sRing + s * L::kKVBytes;
                    mbar_arrive_expect_tx(bar(L::kBarFull + s), L::kKVBytes);
                    for (int cb = 0; cb < D / 64; ++cb)
                        tma_load_3d(dst + cb * kBN * 128, map, bar(L::kBarFull + s), cb * 64, j * kBN, bh);
                    ++issued;
                }
            }
            // Copies must have landed before the CTA's shared memory goes away.
            wait_drain(bar(L::kBarQFull), 0);
            for (int item = max(0, issued - L::kNumSlots); item < issued; ++item)
                wait_drain(bar(L::kBarFull + item % L::kNumSlots), (item / L::kNumSlots) & 1);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && n_kv > 0) {
            constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, true);
            bool ok = wait_bounded(bar(L::kBarQFull), 0, abort_flag, 2, &g_sdp18_error);
            tc_fence_after();

            auto issue_s = [&](int j) -> bool {
                const int sb = j & 1;
                const uint32_t use = static_cast<uint32_t>(j >> 1);
                if (!wait_bounded(bar(L::kBarSFree + sb), (use & 1) ^ 1, abort_flag, 3, &g_sdp18_error)) return false;
                const int item = 2 * j;
                const int s = item % L::kNumSlots;
                if (!wait_bounded(bar(L::kBarFull + s), (item / L::kNumSlots) & 1, abort_flag, 4, &g_sdp18_error)) return false;
                tc_fence_after();
                const uint32_t kbase = sRing + s * L::kKVBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
                    const uint64_t a = sdesc_sw128(sQ + off, 16, 1024);
                    const uint64_t bd = sdesc_sw128(kbase + (kk >> 2) * (kBN * 128) + (kk & 3) * 32, 16, 1024);
                    mma_bf16_ss(tmem + kTmemS0 + sb * kBN, a, bd, kIdescS, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar(L::kBarSFull + sb));
                mma_commit(bar(L::kBarEmpty + s));
                return true;
            };
            auto issue_pv = [&](int j) -> bool {
                if (!wait_bounded(bar(L::kBarPFull), j & 1, abort_flag, 5, &g_sdp18_error)) return false;
                const int item = 2 * j + 1;
                const int s = item % L::kNumSlots;
                if (!wait_bounded(bar(L::kBarFull + s), (item / L::kNumSlots) & 1, abort_flag, 6, &g_sdp18_error)) return false;
                tc_fence_after();
                const uint32_t vbase = sRing + s * L::kKVBytes;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t a = sdesc_sw128(sP + (kk >> 2) * (kBM * 128) + (kk & 3) * 32, 16, 1024);
                    // V is the B operand in MN-major form: 16 keys = 16 rows of
                    // 128 bytes per K step; the next 64 head-dim columns sit one
                    // [128 x 64] block further on (leading byte offset).
                    const uint64_t bd = sdesc_sw128(vbase + kk * 16 * 128, kBN * 128, 1024);
                    mma_bf16_ss(tmem + kTmemO, a, bd, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(bar(L::kBarPVDone));
                mma_commit(bar(L::kBarEmpty + s));
                return true;
            };

            if (ok) ok = issue_s(0);
            for (int j = 0; j < n_kv && ok; ++j) {
                if (j + 1 < n_kv) ok = issue_s(j + 1);
                if (ok) ok = issue_pv(j);
            }
            // Every MMA must be finished before TMEM is released.
            mma_commit(bar(L::kBarDrain));
            wait_drain(bar(L::kBarDrain), 0);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int row = threadIdx.x;  // 0..127 == TMEM lane
        const int q_abs = q0 + row;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        float m = -INFINITY;  // running max of scale*log2(e)*s used for P
        float l = 0.f;        // running sum of P in fp32 (exact weights: gives the LSE)
        float l_mma = 0.f;    // running sum of P as rounded to bf16 for the PV MMA
        bool ok = true;
        // The TMEM loads/stores below are warp-collective, so a wait's outcome
        // is made warp-uniform by a vote.
        auto wait_warp = [&](uint32_t b_addr, uint32_t parity, int site) -> bool {
            return __all_sync(0xffffffffu, wait_bounded(b_addr, parity, abort_flag, site, &g_sdp18_error));
        };

        for (int j = 0; j < n_kv; ++j) {
            const int sb = j & 1;
            if (!wait_warp(bar(L::kBarSFull + sb), (j >> 1) & 1, 7)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t r0[32], r1[32], r2[32], r3[32];
            const uint32_t ts = t_lane + kTmemS0 + sb * kBN;
            tmem_ld32(ts + 0, r0);
            tmem_ld32(ts + 32, r1);
            tmem_ld32(ts + 64, r2);
            tmem_ld32(ts + 96, r3);
            tmem_ld_wait_only();
            reg_fence(r0);
            reg_fence(r1);
            reg_fence(r2);
            reg_fence(r3);
            tc_fence_before();
            mbar_arrive(bar(L::kBarSFree + sb));

            float s[kBN];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                s[c] = __uint_as_float(r0[c]);
                s[32 + c] = __uint_as_float(r1[c]);
                s[64 + c] = __uint_as_float(r2[c]);
                s[96 + c] = __uint_as_float(r3[c]);
            }
            if (j == n_kv - 1) {
                // Only the last tile can hold hidden keys (ragged key tail or
                // the causal diagonal); earlier tiles are fully visible.
                int lim = kv_len - j * kBN;
                if (causal) lim = min(lim, q_abs - j * kBN + 1);
#pragma unroll
                for (int c = 0; c < kBN; ++c)
                    if (c >= lim) s[c] = -INFINITY;
            }
            float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
            for (int c = 4; c < kBN; c += 4) {
                mx0 = fmaxf(mx0, s[c]);
                mx1 = fmaxf(mx1, s[c + 1]);
                mx2 = fmaxf(mx2, s[c + 2]);
                mx3 = fmaxf(mx3, s[c + 3]);
            }
            const float t_max = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * scale_log2;
            float alpha = 1.f;
            if (t_max > m + kRescaleThreshold) {
                alpha = ex2(m - t_max);  // 0 on the first tile (m = -inf)
                m = t_max;
            }
            const float neg_m = -m;
            uint32_t pk[kBN / 2];
            float sum0 = 0.f, sum1 = 0.f, rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int c = 0; c < kBN / 2; ++c) {
                const float p0 = ex2(fmaf(s[2 * c], scale_log2, neg_m));
                const float p1 = ex2(fmaf(s[2 * c + 1], scale_log2, neg_m));
                sum0 += p0;
                sum1 += p1;
                pk[c] = pack_bf16x2(p0, p1);
                // the bf16 values the MMA multiplies V by, widened exactly
                rs0 += __uint_as_float(pk[c] << 16);
                rs1 += __uint_as_float(pk[c] & 0xFFFF0000u);
            }
            l = l * alpha + (sum0 + sum1);
            // O is normalised by the sum of the weights it was built from, so
            // O / l_mma is an exact convex combination of V rows up to the
            // bf16 rounding of their relative sizes.
            l_mma = l_mma * alpha + (rs0 + rs1);

            if (j > 0) {
                // P_{j-1} V_{j-1} must be done: it frees the P tile and O is
                // only rescaled when no MMA is writing it.
                if (!wait_warp(bar(L::kBarPVDone), (j - 1) & 1, 8)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(t_lane + kTmemO + c * 32, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(t_lane + kTmemO + c * 32, o);
                    }
                    tmem_st_wait();
                }
            }
            // P row -> shared memory, K-major 128B-swizzled A operand.
#pragma unroll
            for (int c16 = 0; c16 < kBN / 8; ++c16) {
                const uint32_t addr = sP + (c16 >> 3) * (kBM * 128) + sw128_offset(row, c16 & 7);
                st_shared_v4(addr, pk[4 * c16], pk[4 * c16 + 1], pk[4 * c16 + 2], pk[4 * c16 + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(L::kBarPFull));
        }

        // ------------------------------------------------------------ epilogue
        if (ok) {
            bool have = n_kv > 0;
            if (have) {
                have = wait_warp(bar(L::kBarPVDone), (n_kv - 1) & 1, 9);
                ok = have;
                tc_fence_after();
            }
            if (ok) {
                const float inv_l = have ? 1.f / l_mma : 0.f;
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    if (have) {
                        tmem_ld32(t_lane + kTmemO + c * 32, o);
                        tmem_ld_wait(o);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = 0u;
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int c16 = c * 4 + t;  // 16-byte chunk of the output row
                        const uint32_t addr = sQ + (c16 >> 3) * (kBM * 128) + sw128_offset(row, c16 & 7);
                        st_shared_v4(addr, w[4 * t], w[4 * t + 1], w[4 * t + 2], w[4 * t + 3]);
                    }
                }
                if (lse != nullptr && q_abs < N) {
                    const float v = have ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
                    lse[static_cast<int64_t>(bh) * N + q_abs] = v;
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_sync(1, 4 * 32);
        if (threadIdx.x == 0 && !*abort_flag) {
            for (int cb = 0; cb < D / 64; ++cb) tma_store_3d(&tm_o, sQ + cb * kBM * 128, cb * 64, q0, bh);
            tma_store_commit();
            tma_store_wait_all();
        }
    }

    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D>
int launch(const AttnLaunch &a)
{
    using L = Smem<D>;
    static int configured_device = -1;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (configured_device != dev) {
        if (cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc) !=
            cudaSuccess)
            return -1;
        configured_device = dev;
    }
    const int num_q_tiles = (a.N + kBM - 1) / kBM;
    const int num_bh = a.B * a.H;
    const unsigned grid = static_cast<unsigned>(num_q_tiles) * static_cast<unsigned>(num_bh);
    attn_fwd_kernel<D><<<grid, kThreads, L::kAlloc, a.stream>>>(*a.tm_q, *a.tm_k, *a.tm_v, *a.tm_o, a.lse,
                                                                 a.key_lens, a.H, a.N, num_q_tiles, num_bh,
                                                                 a.scale_log2, a.causal);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int attn_fwd_launch(const AttnLaunch &a)
{
    if (a.d == 64) return launch<64>(a);
    if (a.d == 128) return launch<128>(a);
    return -2;
}

int read_and_clear_device_error(int *value)
{
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_sdp18_error, sizeof(int)) != cudaSuccess) return -1;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_sdp18_error, &zero, sizeof(int)) != cudaSuccess) return -1;
    }
    *value = v;
    return 0;
}

}  // namespace sdp18
