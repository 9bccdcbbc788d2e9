// Dense bf16 GEMM for the multi-head block's projections on B300 (sm_103a):
// C[M, N] = A[M, K] B[K, N], A and B row-major bf16, fp32 accumulation, C
// rounded to bf16 (nearest even).
//
// The block's two projections (cnnetsun.cn "Transformer QKV bottlenecks on
// long sequences", sec. 2, MinimalSelfAttention: Q/K/V projections and the
// output projection; qqiyuan.cn "Multi-head attention in the Transformer:
// implementation and performance optimisation": one fused [E, 3E] projection)
// are x W_qkv and M W_o, plain dense products.
//
// Persistent CTAs, one per SM, each computing 128 x 256 output tiles:
//   warp 0       TMA producer: per 64-wide K step, the A tile [128 x 64]
//                (K-major) and the B tile [64 x 256] as four MN-major
//                [64 x 64] blocks, into a 4-stage ring (48 KB per stage).
//   warp 1       allocates TMEM and issues tcgen05.mma M=128 N=256 K=16 from
//                one elected lane, four per stage, into one of two 256-column
//                fp32 accumulators; commits the tile to the epilogue.
//   warps 2-5    epilogue: each thread reads its row of the accumulator from
//                TMEM (its warp's lane quarter), rounds to bf16 and writes it
//                with 16-byte stores, then frees the accumulator -- while the
//                MMA warp already accumulates the next tile in the other one.
// Tiles are visited in bands of M-blocks (N blocks outer, M blocks inner
// within a band), the band sized so that its A rows (about 48 MB) stay in L2
// while every column block of B streams past them once: B is read from DRAM
// once per band, A once.  Rows past M and columns past N read as zero (TMA)
// and are not stored.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "attn_internal.h"
#include "ptx_sm103.cuh"

namespace sdp18 {

// Device error word of the GEMM kernel (read and cleared by the host).
__device__ int g_sdp18_gemm_error = 0;

namespace {

constexpr int kGM = 128;         // output rows per tile
constexpr int kGN = 256;         // output columns per tile
constexpr int kGK = 64;          // K per stage (one 128-byte swizzle row of bf16)
constexpr int kStages = 4;
constexpr int kGThreads = 192;   // producer, MMA, 4 epilogue warps
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr uint32_t kAccCols = 256;

struct GSmem {
    static constexpr int kABytes = kGM * kGK * 2;        // 16 KB
    static constexpr int kBBlock = kGK * 64 * 2;         // one [64 K x 64 N] block, 8 KB
    static constexpr int kBBytes = kBBlock * (kGN / 64);  // 32 KB
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kOffBar = kStages * kStageBytes;
    static constexpr int kBarFull = 0;
    static constexpr int kBarEmpty = kBarFull + kStages;
    static constexpr int kBarAccFull = kBarEmpty + kStages;    // [2]
    static constexpr int kBarAccEmpty = kBarAccFull + 2;       // [2]
    static constexpr int kBarDrain = kBarAccEmpty + 2;
    static constexpr int kNumBars = kBarDrain + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;    // tmem address, abort flag
    static constexpr int kBytes = kOffMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;
    static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

// Output block (mb, nb) of tile t in the banded order.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int band_m, int &mb, int &nb)
{
    const int band = t / (band_m * tiles_n);
    const int r = t - band * band_m * tiles_n;
    const int rows = min(band_m, tiles_m - band * band_m);
    nb = r / rows;
    mb = band * band_m + r % rows;
}

__global__ void __launch_bounds__(kGThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     __nv_bfloat16 *__restrict__ c, int64_t ldc, int M, int N, int K, int tiles_m, int tiles_n,
                     int band_m)
{
    using L = GSmem;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_addr(smem);
    auto sA = [&](int s) -> uint32_t { return s_base + s * L::kStageBytes; };
    auto sB = [&](int s) -> uint32_t { return s_base + s * L::kStageBytes + L::kABytes; };
    auto bar = [&](int i) -> uint32_t { return s_base + L::kOffBar + 8 * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);
    const int warp = threadIdx.x >> 5;
    const int num_tiles = tiles_m * tiles_n;
    const int k_steps = K / kGK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(L::kBarFull + s), 1);
            mbar_init(bar(L::kBarEmpty + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(L::kBarAccFull + a), 1);
            mbar_init(bar(L::kBarAccEmpty + a), 4 * 32);
        }
        mbar_init(bar(L::kBarDrain), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), 2 * kAccCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto wait_warp = [&](uint32_t b_addr, uint32_t parity, int site) -> bool {
        return __all_sync(0xffffffffu, wait_bounded(b_addr, parity, abort_flag, site, &g_sdp18_gemm_error));
    };

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        tma_prefetch_map(&tm_a);
        tma_prefetch_map(&tm_b);
        int stage = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            int mb, nb;
            tile_coords(t, tiles_m, tiles_n, band_m, mb, nb);
            for (int kb = 0; kb < k_steps; ++kb, ++stage) {
                const int s = stage % kStages;
                if (!(ok = wait_warp(bar(L::kBarEmpty + s), ((stage / kStages) & 1) ^ 1, 40))) break;
                mbar_arrive_expect_tx_one(bar(L::kBarFull + s), L::kStageBytes);
                tma_load_2d_one(sA(s), &tm_a, bar(L::kBarFull + s), kb * kGK, mb * kGM);
#pragma unroll
                for (int i = 0; i < kGN / 64; ++i)
                    tma_load_2d_one(sB(s) + i * L::kBBlock, &tm_b, bar(L::kBarFull + s), nb * kGN + i * 64, kb * kGK);
            }
        }
        // Copies must have landed before the CTA's shared memory goes away.
        for (int i = max(0, stage - kStages); i < stage; ++i)
            wait_drain(bar(L::kBarFull + i % kStages), (i / kStages) & 1);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t kIdesc = idesc_bf16_f32(kGM, kGN, true);
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
        int stage = 0, tcount = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++tcount) {
            const int acc = tcount & 1;
            // The epilogue has read this accumulator's previous tile out.
            if (!(ok = wait_warp(bar(L::kBarAccEmpty + acc), ((tcount >> 1) & 1) ^ 1, 41))) break;
            tc_fence_after();
            const uint32_t d = tm + acc * kAccCols;
            for (int kb = 0; kb < k_steps; ++kb, ++stage) {
                const int s = stage % kStages;
                if (!(ok = wait_warp(bar(L::kBarFull + s), (stage / kStages) & 1, 42))) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kGK / 16; ++kk) {
                    // A: K-major, 16 K values = 32 bytes along the swizzled row.
                    const uint64_t a = sdesc_sw128(sA(s) + kk * 32, 16, 1024);
                    // B: MN-major, 16 K rows of 128 bytes per step; the next
                    // 64 output columns sit one [64 x 64] block further on.
                    const uint64_t b = sdesc_sw128(sB(s) + kk * 16 * 128, L::kBBlock, 1024);
                    mma_bf16_ss_one(d, a, b, kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit_one(bar(L::kBarEmpty + s));
            }
            if (!ok) break;
            mma_commit_one(bar(L::kBarAccFull + acc));
        }
        mma_commit_one(bar(L::kBarDrain));
        wait_drain(bar(L::kBarDrain), 0);
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // lane quarter this warp can read
        const int row_local = q * 32 + (threadIdx.x & 31);
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
        int tcount = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++tcount) {
            int mb, nb;
            tile_coords(t, tiles_m, tiles_n, band_m, mb, nb);
            const int acc = tcount & 1;
            if (!(ok = wait_warp(bar(L::kBarAccFull + acc), (tcount >> 1) & 1, 43))) break;
            tc_fence_after();
            const int row = mb * kGM + row_local;
            __nv_bfloat16 *crow = c + static_cast<int64_t>(row) * ldc + nb * kGN;
#pragma unroll 1
            for (int ch = 0; ch < kGN / 32; ++ch) {
                uint32_t r[32];
                tmem_ld32(t_lane + acc * kAccCols + ch * 32, r);
                tmem_ld_wait(r);
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
                if (row < M) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int col = nb * kGN + ch * 32 + u * 8;
                        if (col < N) st_global_v4(crow + ch * 32 + u * 8, w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(L::kBarAccEmpty + acc));
        }
    }

    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * kAccCols);
    }
}

}  // namespace

int gemm_bf16_launch(const GemmLaunch &g)
{
    static int configured_device = -1;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (configured_device != dev) {
        if (cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GSmem::kAlloc) !=
            cudaSuccess)
            return -1;
        configured_device = dev;
    }
    if (g.M <= 0 || g.N <= 0 || g.K <= 0 || g.K % kGK != 0) return -2;
    const int tiles_m = (g.M + kGM - 1) / kGM, tiles_n = (g.N + kGN - 1) / kGN;
    const int64_t tiles = static_cast<int64_t>(tiles_m) * tiles_n;
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>(tiles, sm_count()));
    // M-blocks per band: their A rows (kGM x K bf16 each) within ~48 MB.
    const int64_t a_block = static_cast<int64_t>(kGM) * g.K * 2;
    const int band_m = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(tiles_m, (int64_t(48) << 20) / a_block)));
    gemm_bf16_kernel<<<grid, kGThreads, GSmem::kAlloc, g.stream>>>(*g.tm_a, *g.tm_b,
                                                                    static_cast<__nv_bfloat16 *>(g.c), g.ldc, g.M,
                                                                    g.N, g.K, tiles_m, tiles_n, band_m);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int read_and_clear_gemm_error(int *value)
{
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_sdp18_gemm_error, sizeof(int)) != cudaSuccess) return -1;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_sdp18_gemm_error, &zero, sizeof(int)) != cudaSuccess) return -1;
    }
    *value = v;
    return 0;
}

}  // namespace sdp18
