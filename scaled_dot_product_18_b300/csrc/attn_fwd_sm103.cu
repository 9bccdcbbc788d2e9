// Attention forward for B300 (sm_103a): persistent CTAs, one per SM, each
// working through pairs of 128-row query tiles of one (batch, head).
//
// The method is the tiled forward with an online softmax (hotelren.com "AI
// attention: essence and evolution", sec. 4.1, FlashAttention-1): for a query
// tile, stream the key/value tiles, form S = Q K^T for the pair, fold it into
// running row statistics (max, sum), accumulate P V, and never write S out.
// Key tiles that the mask hides completely are not visited (hotelren.com
// sec. 5, "only load active K/V blocks").  An optional sliding window limits
// query i to keys j > i - w (aicoding.csdn.net "Why does attention stall
// large-model training", sec. 4.3): each query tile then visits only the key
// tiles that intersect its rows' windows.
//
// How it maps onto sm_103a.  The CTA owns two query tiles, Q0 (rows q0 ..
// q0+127) and Q1 (rows q0+128 .. q0+255), which share every K/V tile:
//   warps 0-3    softmax of tile 0: thread t owns query row t (TMEM lane t),
//                so every row reduction stays inside one thread.
//   warps 4-7    softmax of tile 1, same layout.
//   warp 8       allocates tensor memory (TMEM) and, from one thread, issues
//                every tcgen05.mma in the order
//                  S0 = Q0 K_j^T, S1 = Q1 K_j^T,
//                  O0 += P0 V_j, S0 = Q0 K_{j+1}^T, O1 += P1 V_j, S1 = ...
//                so the tensor core works on one tile while the other tile's
//                warps run the softmax.
//   warp 9       TMA producer: works out each work item of the CTA once and
//                publishes it to the other warps in a small ring of
//                shared-memory descriptors, then loads Q0, Q1 of the item
//                and K_j, V_j through a ring of shared-memory slots guarded
//                by full/empty mbarriers.
// A softmax warp reads S_t from TMEM, masks the last key tile, takes the
// running max in the log2 domain, exponentiates with ex2, and writes P_t as
// packed bf16 back into the first 64 columns of S_t's TMEM region, where the
// P V MMA reads it as its A operand.  The tensor core runs a thread's MMAs in
// issue order, so S_t for key tile j+1 (issued after O_t += P_t V_j) only
// overwrites P_t after that MMA has read it, and the commit that signals
// "S_t(j+1) ready" also covers O_t += P_t V_j: a softmax warp that holds
// S_t(j+1) may rescale O_t in place, no MMA is writing it.  At d = 64 the
// two O tiles leave room for P_t in its own TMEM columns, so S_t(j+1) is
// issued as soon as the softmax warps have read S_t(j).
//
// Work items.  An item is a pair of query tiles of one (batch, head).  Work
// units (an item, or two causal items of equal total cost) run in one fixed
// order: heaviest causal pair first, within groups of heads whose keys and
// values stay in L2.  With enough units per SM the grid is min(units, SMs)
// persistent CTAs and CTA c takes units c, c + grid, ... (a static version
// of the hardware's greedy block scheduling, without the per-CTA set-up);
// otherwise each causal item gets its own CTA.  TMEM is allocated,
// barriers initialised and tensor maps prefetched once per CTA; every
// barrier keeps counting phases across items.  The softmax warps write O_t
// from registers (d = 128) or through a small per-warp staging buffer and a
// TMA store (d = 64), never through the Q buffers, so a Q buffer is free as
// soon as its last S MMA has run: the next item's Q is loaded while the
// current item's last key tiles and its epilogue are still in flight, and
// the tensor core starts the next item while the previous one's O is
// written.
//
// Q, K and V are addressed through 4-D tensor maps {d, N, H, B} and O through
// element strides, all with arbitrary row, head and batch strides, so the
// heads may sit in [B, H, N, d] tensors or interleaved in [B, N, H, d] rows
// (the output of a fused QKV projection) without a transpose.
//
// Memory layout (all 128-byte swizzled, 1024-byte aligned tiles):
//   Q tile t : d/64 column blocks of [128 rows x 64 bf16]
//   K/V ring : NSLOT slots of d/64 blocks of [128 keys x 64 bf16]
// TMEM (512 columns): S0 at 0, S1 at 128, O0 at 256, O1 at 256 + d; at
// d = 64, P0 at 384 and P1 at 448.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "attn_internal.h"
#include "ptx_sm103.cuh"

namespace sdp18 {

// Device error word of this library (read and cleared by the host).
__device__ int g_sdp18_error = 0;

#ifdef SDP18_WAIT_TEST
// Test library only: when >= 0, the producer issues no K/V copy from this
// ring item on, so the MMA warp's bounded wait for it runs out and the CTA
// winds down (abort flag, error word, drain, TMEM freed).
__device__ int g_test_stall_items = -1;
#endif

namespace {

constexpr int kBM = 128;           // query rows per tile
constexpr int kBN = 128;           // keys per tile
constexpr int kTilesPerCta = 2;    // query tiles per CTA
constexpr int kRowsPerCta = kBM * kTilesPerCta;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kThreads = 320;      // 8 softmax warps + MMA warp + TMA warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;     // S_t at kTmemS + t * kBN
constexpr uint32_t kTmemO = 256;   // O_t at kTmemO + t * D
constexpr uint32_t kTmemP = 384;   // d = 64 only: P_t (packed bf16) at kTmemP + t * kBN / 2
// Lazy rescaling: the running max used for P only moves when a row's true max
// exceeds it by more than 2^8, so P stays <= 256 and O needs a rescale only
// rarely.  Exact: O and l always share the same stale max.
constexpr float kRescaleThreshold = 8.0f;
// Within a key tile the max is settled from the first 64 score columns; the
// second half moves it only past this margin (P <= 2^32 otherwise, exact in
// the fp32 sums and the bf16 P), since moving it there means rescaling the
// first half's P, already stored as bf16, a second rounding.
constexpr float kInTileLimit = 32.0f;

// 32-byte store of eight 32-bit words (sm_100+; the address must be 32-byte
// aligned).
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t *w)
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// The producer warp works out each item of the CTA's schedule once and
// publishes it in a small ring of shared-memory descriptors; the MMA and
// softmax warps read it there instead of repeating the schedule arithmetic
// (integer divisions, key ranges) at every item boundary.
constexpr int kDescSlots = 4;
// Three int4: {q0, b, h, bh}, {kv_len, kr0.first, kr0.end, kr1.first},
// {kr1.end, j_begin, n_max, valid}.
constexpr int kDescBytes = 48;
constexpr int kDescConsumers = 1 + 8;  // the MMA warp and the 8 softmax warps (one arrival per warp)

template <int D>
struct Smem {
    static constexpr int kNumSlots = D == 128 ? 5 : 8;
    static constexpr int kQBytes = kBM * D * 2;   // one query tile
    static constexpr int kKVBytes = kBN * D * 2;  // one K or V tile
    static constexpr int kOffQ = 0;               // Q tile t at kOffQ + t * kQBytes
    static constexpr int kOffRing = kOffQ + kTilesPerCta * kQBytes;
    // d = 64 epilogue staging: each softmax warp's 32 rows x 64 columns (4 KB).
    // (d = 128 has no room next to a 5-slot ring and stores O from registers.)
    static constexpr int kOffStage = kOffRing + kNumSlots * kKVBytes;
    static constexpr int kStageBytes = D == 64 ? 32 * 128 : 0;
    static constexpr int kOffBar = kOffStage + 8 * kStageBytes;
    static constexpr int kBarQFull = 0;                      // [2] Q_t landed
    static constexpr int kBarQFree = 2;                      // [2] last S_t MMA of an item done
    static constexpr int kBarFull = 4;
    static constexpr int kBarEmpty = kBarFull + kNumSlots;
    static constexpr int kBarSFull = kBarEmpty + kNumSlots;  // [2]
    static constexpr int kBarPFull = kBarSFull + 2;          // [2]
    static constexpr int kBarODone = kBarPFull + 2;          // [2]
    static constexpr int kBarSFree = kBarODone + 2;          // [2] d = 64: S_t read into registers
    static constexpr int kBarPVDone = kBarSFree + 2;         // [2] d = 64: O_t += P_t V done
    static constexpr int kBarDrain = kBarPVDone + 2;
    static constexpr int kBarDescFull = kBarDrain + 1;               // [kDescSlots] item published
    static constexpr int kBarDescEmpty = kBarDescFull + kDescSlots;  // [kDescSlots] read by all consumers
    static constexpr int kNumBars = kBarDescEmpty + kDescSlots;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem address, abort flag
    static constexpr int kOffDesc = (kOffMisc + 16 + 15) & ~15;  // kDescSlots item descriptors (int4 aligned)
    static constexpr int kBytes = kOffDesc + kDescSlots * kDescBytes;
    static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024
    static_assert(kAlloc <= 227 * 1024, "shared memory budget");
    static_assert(kOffBar % 8 == 0 && kOffDesc % 16 == 0 && kDescBytes % 16 == 0, "barrier / descriptor alignment");
    static_assert(kTmemO + 2 * D <= kTmemCols, "TMEM budget");
    static_assert(D != 64 || kTmemP == kTmemO + 2 * D, "d = 64 keeps P next to O");
};

// Key tiles [first, end) that query tile q0t visits; empty when first >= end.
// The upper end follows the key length and the causal diagonal of the
// tile's last row, the lower end the window of its first row.
struct KeyRange {
    int first, end;
    __device__ __forceinline__ int count() const { return end > first ? end - first : 0; }
};
__device__ __forceinline__ KeyRange key_range(int q0t, int N, int kv_len, int causal, int window)
{
    if (q0t >= N) return {0, 0};
    const int kv_end = causal ? min(kv_len, q0t + kBM) : kv_len;
    const int lo = window > 0 ? max(0, q0t - window + 1) : 0;
    return {lo / kBN, (kv_end + kBN - 1) / kBN};
}

// One work item: a pair of query tiles of one (batch, head), the key tiles
// each tile visits and the tiles the CTA streams.
struct Item {
    int bh, b, h, q0, kv_len;
    KeyRange kr[2];
    int n[2];              // key tiles visited by query tile t
    int j_begin, n_max;    // key tiles streamed: [j_begin, j_begin + n_max)
};

// The schedule: work units in a fixed order, unit u going to CTA u % grid.
// A unit is one query pair, or -- for causal attention without a window,
// where pair p costs 2p + 2 key tiles -- the two pairs nqp-1-p and p of one
// head, so that every unit costs the same and a static assignment is as
// balanced as the hardware's greedy one.  Units run head group by head group
// (all heads in one group unless the host chose smaller groups so that a
// group's keys and values stay in L2), heads innermost, heaviest pairs first.
struct Sched {
    int H, N, nqp, num_bh, head_group, paired;
    int o_v8;  // O's base and strides are 32-byte aligned: rows are written 32 bytes per store
};

// The query pairs of unit u (1 or 2, heaviest first) and its (batch, head).
__device__ __forceinline__ int unit_pairs(const Sched &sc, int u, int (&qp)[2], int &bh)
{
    const int per_head = sc.paired ? (sc.nqp + 1) / 2 : sc.nqp;
    const int per_group = sc.head_group * per_head;
    const int grp = u / per_group;
    const int g_heads = min(sc.head_group, sc.num_bh - grp * sc.head_group);
    const int in_grp = u - grp * per_group;
    bh = grp * sc.head_group + in_grp % g_heads;
    const int p = in_grp / g_heads;
    qp[0] = sc.nqp - 1 - p;
    qp[1] = p;
    return sc.paired && qp[1] != qp[0] ? 2 : 1;
}

__device__ __forceinline__ Item make_item(const Sched &sc, int qp, int bh, const int32_t *key_lens, int causal,
                                          int window)
{
    Item it;
    const int N = sc.N;
    it.bh = bh;
    it.q0 = qp * kRowsPerCta;
    it.b = bh / sc.H;
    it.h = bh % sc.H;
    it.kv_len = N;
    if (key_lens != nullptr) it.kv_len = min(max(key_lens[it.b], 0), N);
    it.kr[0] = key_range(it.q0, N, it.kv_len, causal, window);
    it.kr[1] = key_range(it.q0 + kBM, N, it.kv_len, causal, window);
    it.n[0] = it.kr[0].count();
    it.n[1] = it.kr[1].count();
    // The CTA streams key tiles [j_begin, j_end), the union of both ranges;
    // a key tile in the union that neither range holds is still streamed and
    // consumed, so the ring stays in step.
    const int n0 = it.n[0], n1 = it.n[1];
    it.j_begin = n0 == 0 ? it.kr[1].first : n1 == 0 ? it.kr[0].first : min(it.kr[0].first, it.kr[1].first);
    const int j_end = n0 == 0 ? it.kr[1].end : n1 == 0 ? it.kr[0].end : max(it.kr[0].end, it.kr[1].end);
    it.n_max = n0 + n1 > 0 ? j_end - it.j_begin : 0;
    return it;
}

// kWindow = false compiles the plain causal / key-length kernel; true adds
// the sliding-window ranges, the lower-edge mask and the guards for rows that
// have not seen a visible key yet.
template <int D, bool kWindow>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    __nv_bfloat16 *__restrict__ out, OStrides ost,
                    float *__restrict__ lse, const int32_t *__restrict__ key_lens, Sched sc, int num_units,
                    float scale_log2, int causal, int window)
{
    using L = Smem<D>;
    // At d = 64 the two O tiles leave 128 TMEM columns free: P_t gets its own
    // columns, so S_t(j+1) need not wait for P_t(j) V_j (which reads P_t(j)
    // out of S_t's columns at d = 128) and the softmax warps run from one key
    // tile to the next without waiting for the tensor core.
    constexpr bool kSplitP = D == 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_addr(smem);
    const uint32_t sRing = s_base + L::kOffRing;
    auto sQ = [&](int t) -> uint32_t { return s_base + L::kOffQ + t * L::kQBytes; };
    auto bar = [&](int i) -> uint32_t { return s_base + L::kOffBar + 8 * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    if constexpr (!kWindow) window = 0;
    const int N = sc.N;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(bar(L::kBarQFull + t), 1);
            mbar_init(bar(L::kBarQFree + t), 1);
            mbar_init(bar(L::kBarSFull + t), 1);
            mbar_init(bar(L::kBarPFull + t), 4 * 32);
            mbar_init(bar(L::kBarODone + t), 1);
            mbar_init(bar(L::kBarSFree + t), 4 * 32);
            mbar_init(bar(L::kBarPVDone + t), 1);
        }
        for (int s = 0; s < L::kNumSlots; ++s) {
            mbar_init(bar(L::kBarFull + s), 1);
            mbar_init(bar(L::kBarEmpty + s), 1);
        }
        mbar_init(bar(L::kBarDrain), 1);
        for (int i = 0; i < kDescSlots; ++i) {
            mbar_init(bar(L::kBarDescFull + i), 1);
            mbar_init(bar(L::kBarDescEmpty + i), kDescConsumers);
        }
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

    // The producer and MMA warps run their loops with all 32 lanes (waits
    // agreed by a vote); one elected lane issues each copy, MMA and commit.
    auto wait_warp = [&](uint32_t b_addr, uint32_t parity, int site) -> bool {
        return __all_sync(0xffffffffu, wait_bounded(b_addr, parity, abort_flag, site, &g_sdp18_error));
    };
    // Item descriptor k of this CTA: slot k % kDescSlots, phase k / kDescSlots.
    auto desc_ptr = [&](int k) -> int4 * {
        return reinterpret_cast<int4 *>(smem + L::kOffDesc + (k % kDescSlots) * kDescBytes);
    };
    // Consumer side (whole warp): wait for descriptor k, copy it, release the
    // slot.  valid = false marks the end of the CTA's items.
    auto read_desc = [&](int k, Item &it, bool &valid) -> bool {
        if (!wait_warp(bar(L::kBarDescFull + k % kDescSlots), (k / kDescSlots) & 1, 9)) return false;
        const int4 *dp = desc_ptr(k);
        const int4 a = dp[0], c = dp[1], e = dp[2];
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(bar(L::kBarDescEmpty + k % kDescSlots));
        it.q0 = a.x;
        it.b = a.y;
        it.h = a.z;
        it.bh = a.w;
        it.kv_len = c.x;
        it.kr[0] = {c.y, c.z};
        it.kr[1] = {c.w, e.x};
        it.n[0] = it.kr[0].count();
        it.n[1] = it.kr[1].count();
        it.j_begin = e.y;
        it.n_max = e.z;
        valid = e.w != 0;
        return true;
    };

    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ producer
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
        int ring = 0;              // K/V copies issued so far (ring position)
        int q_loads[2] = {0, 0};   // Q_t copies issued so far
        bool ok = true;
        int published = 0;  // item descriptors written
        // Lane 0 writes descriptor `published` once its slot has been read by
        // every consumer (kDescSlots items back).
        auto publish = [&](const Item &it, int valid) -> bool {
            const int k = published;
            if (k >= kDescSlots &&
                !wait_warp(bar(L::kBarDescEmpty + k % kDescSlots), ((k / kDescSlots) - 1) & 1, 14))
                return false;
            if ((threadIdx.x & 31) == 0) {
                int4 *dp = desc_ptr(k);
                dp[0] = make_int4(it.q0, it.b, it.h, it.bh);
                dp[1] = make_int4(it.kv_len, it.kr[0].first, it.kr[0].end, it.kr[1].first);
                dp[2] = make_int4(it.kr[1].end, it.j_begin, it.n_max, valid);
                mbar_arrive(bar(L::kBarDescFull + k % kDescSlots));  // release: the stores are visible
            }
            __syncwarp();
            ++published;
            return true;
        };
        for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x)
        for (int qps[2], bh_u, n_u = unit_pairs(sc, u, qps, bh_u), s_u = 0; s_u < n_u && ok; ++s_u) {
            const Item it = make_item(sc, qps[s_u], bh_u, key_lens, causal, window);
            // Every item is published, also those with no key tile: their
            // softmax warps still write O = 0 and lse = -inf.
            if (!(ok = publish(it, 1))) break;
            if (it.n_max == 0) continue;
            // Q_t of this item goes where the previous item's Q_t was, once
            // that item's last S_t MMA has read it.
            for (int t = 0; t < 2 && ok; ++t) {
                if (it.n[t] == 0) continue;
                if (q_loads[t] > 0 && !(ok = wait_warp(bar(L::kBarQFree + t), (q_loads[t] - 1) & 1, 8))) break;
                mbar_arrive_expect_tx_one(bar(L::kBarQFull + t), L::kQBytes);
                for (int cb = 0; cb < D / 64; ++cb)
                    tma_load_4d_one(sQ(t) + cb * kBM * 128, &tm_q, bar(L::kBarQFull + t), cb * 64, it.q0 + t * kBM,
                                    it.h, it.b);
                ++q_loads[t];
            }
            for (int i = 0; i < 2 * it.n_max && ok; ++i) {
#ifdef SDP18_WAIT_TEST
                if (g_test_stall_items >= 0 && ring >= g_test_stall_items) {
                    ok = false;
                    break;
                }
#endif
                const int s = ring % L::kNumSlots;
                const uint32_t round = static_cast<uint32_t>(ring / L::kNumSlots);
                if (!(ok = wait_warp(bar(L::kBarEmpty + s), (round & 1) ^ 1, 1))) break;
                const CUtensorMap *map = (i & 1) ? &tm_v : &tm_k;
                const uint32_t dst = sRing + s * L::kKVBytes;
                mbar_arrive_expect_tx_one(bar(L::kBarFull + s), L::kKVBytes);
                for (int cb = 0; cb < D / 64; ++cb)
                    tma_load_4d_one(dst + cb * kBN * 128, map, bar(L::kBarFull + s), cb * 64,
                                    (it.j_begin + (i >> 1)) * kBN, it.h, it.b);
                ++ring;
            }
        }
        if (ok) {
            Item end_it{};
            publish(end_it, 0);
        }
        // Copies must have landed before the CTA's shared memory goes away.
        for (int t = 0; t < 2; ++t)
            if (q_loads[t] > 0) wait_drain(bar(L::kBarQFull + t), (q_loads[t] - 1) & 1);
        for (int i = max(0, ring - L::kNumSlots); i < ring; ++i)
            wait_drain(bar(L::kBarFull + i % L::kNumSlots), (i / L::kNumSlots) & 1);
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false);
        constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, true);
        const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);  // warp-uniform
        int ring = 0;              // ring position of the item's first K tile
        int q_used[2] = {0, 0};    // Q_t phases consumed
        int steps[2] = {0, 0};     // S_t / P_t phases used
        bool ok = true;
        auto wait_full = [&](int item, int site) -> bool {
            const bool r = wait_warp(bar(L::kBarFull + item % L::kNumSlots), (item / L::kNumSlots) & 1, site);
            tc_fence_after();
            return r;
        };
        // S_t = Q_t K^T from the K tile in ring slot `ks`.
        auto issue_s = [&](int t, int ks) {
            const uint32_t kbase = sRing + ks * L::kKVBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * (kBM * 128) + (kk & 3) * 32;
                const uint64_t a = sdesc_sw128(sQ(t) + off, 16, 1024);
                const uint64_t bd = sdesc_sw128(kbase + (kk >> 2) * (kBN * 128) + (kk & 3) * 32, 16, 1024);
                mma_bf16_ss_one(tm + kTmemS + t * kBN, a, bd, kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit_one(bar(L::kBarSFull + t));
        };
        // O_t (+)= P_t V from the V tile in ring slot `vs`; P_t is read
        // from TMEM, 16 keys (8 packed columns) per MMA.
        auto issue_pv = [&](int t, int vs, bool acc) {
            const uint32_t vbase = sRing + vs * L::kKVBytes;
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk) {
                // V is the B operand in MN-major form: 16 keys = 16 rows of
                // 128 bytes per K step; the next 64 head-dim columns sit one
                // [128 x 64] block further on (leading byte offset).
                const uint64_t bd = sdesc_sw128(vbase + kk * 16 * 128, kBN * 128, 1024);
                const uint32_t a_tmem = kSplitP ? tm + kTmemP + t * (kBN / 2) + kk * 8 : tm + kTmemS + t * kBN + kk * 8;
                mma_bf16_ts_one(tm + kTmemO + t * D, a_tmem, bd, kIdescPV, (acc || kk > 0) ? 1u : 0u);
            }
        };
        for (int k = 0; ok; ++k) {
            Item it;
            bool valid;
            if (!(ok = read_desc(k, it, valid)) || !valid) break;
            if (it.n_max == 0) continue;
            const int n_t[2] = {it.n[0], it.n[1]};
            // Tile t is active at key tile j (0-based in the stream) when its
            // range holds it; its local iteration index is j - first.
            const int f_t[2] = {it.kr[0].first - it.j_begin, it.kr[1].first - it.j_begin};
            auto active = [&](int t, int j) { return n_t[t] > 0 && j >= f_t[t] && j < f_t[t] + n_t[t]; };
            // S_t of the tile's last visited key tile: the Q_t buffer may
            // be refilled once it is done.
            auto issue_s_q = [&](int t, int ks, bool last) {
                issue_s(t, ks);
                if (last) mma_commit_one(bar(L::kBarQFree + t));
            };
            // The previous item's O_t is read out by its softmax warps before
            // they hand over P_t of this item, so O_t is free when the first
            // P V MMA (which overwrites it) is issued.
            for (int t = 0; t < 2 && ok; ++t)
                if (n_t[t] > 0) ok = wait_warp(bar(L::kBarQFull + t), q_used[t] & 1, 2);
            if (ok) ok = wait_full(ring, 3);
            if (ok) {
#pragma unroll
                for (int t = 0; t < 2; ++t)
                    if (active(t, 0)) issue_s_q(t, ring % L::kNumSlots, n_t[t] == 1);
                mma_commit_one(bar(L::kBarEmpty + ring % L::kNumSlots));
            }
            if constexpr (kSplitP) {
                // Per key tile: S_t(j+1) for each tile as soon as its softmax
                // warps have read S_t(j), then P_t(j) V_j once they have stored
                // P_t(j).  Covers the plain and the sliding-window kernel.
                for (int j = 0; j < it.n_max && ok; ++j) {
                    const int v_item = ring + 2 * j + 1, k_item = ring + 2 * j + 2;
                    const int vs = v_item % L::kNumSlots, ks = k_item % L::kNumSlots;
                    if (j + 1 < it.n_max) {  // K_{j+1} is streamed
                        ok = wait_full(k_item, 7);
                        for (int t = 0; t < 2 && ok; ++t) {
                            if (!active(t, j + 1)) continue;
                            // (A tile's first S of the item overwrites scores the
                            // previous item's last P hand-off has released.)
                            if (active(t, j)) {
                                ok = wait_warp(bar(L::kBarSFree + t), (steps[t] + j - f_t[t]) & 1, 16 + t);
                                if (!ok) break;
                                tc_fence_after();
                            }
                            issue_s_q(t, ks, j + 2 - f_t[t] == n_t[t]);
                        }
                        if (!ok) break;
                        mma_commit_one(bar(L::kBarEmpty + ks));
                    }
                    ok = wait_full(v_item, 4);
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (!active(t, j)) continue;
                        const int jj = j - f_t[t];
                        ok = wait_warp(bar(L::kBarPFull + t), (steps[t] + jj) & 1, 5 + t);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(t, vs, jj > 0);
                        mma_commit_one(bar(L::kBarPVDone + t));
                    }
                    if (!ok) break;
                    mma_commit_one(bar(L::kBarEmpty + vs));
                }
            } else if constexpr (!kWindow) {
                // Both tiles start at key tile 0; tile 1 may run one tile longer.
                for (int j = 0; j < it.n_max && ok; ++j) {
                    const int v_item = ring + 2 * j + 1, k_item = ring + 2 * j + 2;
                    const int vs = v_item % L::kNumSlots, ks = k_item % L::kNumSlots;
                    ok = wait_full(v_item, 4);
                    bool k_ready = false;
                    for (int t = 0; t < 2 && ok; ++t) {
                        if (j >= n_t[t]) continue;
                        ok = wait_warp(bar(L::kBarPFull + t), (steps[t] + j) & 1, 5 + t);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(t, vs, j > 0);
                        if (j + 1 < n_t[t]) {
                            if (!k_ready) {
                                ok = wait_full(k_item, 7);
                                if (!ok) break;
                                k_ready = true;
                            }
                            issue_s_q(t, ks, j + 2 == n_t[t]);
                        } else {
                            mma_commit_one(bar(L::kBarODone + t));
                        }
                    }
                    if (!ok) break;
                    mma_commit_one(bar(L::kBarEmpty + vs));
                    if (k_ready) mma_commit_one(bar(L::kBarEmpty + ks));
                }
            } else {
                for (int j = 0; j < it.n_max && ok; ++j) {
                    const int v_item = ring + 2 * j + 1, k_item = ring + 2 * j + 2;
                    const int vs = v_item % L::kNumSlots, ks = k_item % L::kNumSlots;
                    ok = wait_full(v_item, 4);
                    const bool k_next = j + 1 < it.n_max;  // K_{j+1} is streamed: consume it below
                    bool k_ready = false;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (!ok) break;
                        if (active(t, j)) {
                            const int jj = j - f_t[t];
                            ok = wait_warp(bar(L::kBarPFull + t), (steps[t] + jj) & 1, 5 + t);
                            if (!ok) break;
                            tc_fence_after();
                            issue_pv(t, vs, jj > 0);
                            if (jj + 1 == n_t[t]) mma_commit_one(bar(L::kBarODone + t));
                        }
                        if (k_next && active(t, j + 1)) {
                            if (!k_ready) {
                                ok = wait_full(k_item, 7);
                                if (!ok) break;
                                k_ready = true;
                            }
                            issue_s_q(t, ks, j + 1 - f_t[t] + 1 == n_t[t]);
                        }
                    }
                    if (ok && k_next && !k_ready) {
                        ok = wait_full(k_item, 7);  // streamed but used by neither tile
                        k_ready = ok;
                    }
                    if (!ok) break;
                    mma_commit_one(bar(L::kBarEmpty + vs));
                    if (k_ready) mma_commit_one(bar(L::kBarEmpty + ks));
                }
            }
            ring += 2 * it.n_max;
            for (int t = 0; t < 2; ++t) {
                steps[t] += n_t[t];
                q_used[t] += n_t[t] > 0;
            }
        }
        // Every MMA must be finished before TMEM is released.
        mma_commit_one(bar(L::kBarDrain));
        wait_drain(bar(L::kBarDrain), 0);
    } else {
        // ------------------------------------------------------------ softmax
        const int t = warp >> 2;            // query tile of this warpgroup
        const int row = threadIdx.x & 127;  // == TMEM lane
        const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t tS = t_lane + kTmemS + t * kBN;
        const uint32_t tO = t_lane + kTmemO + t * D;
        // P_t goes over the first 64 score columns (d = 128) or to its own
        // columns (d = 64).
        const uint32_t tP = kSplitP ? t_lane + kTmemP + t * (kBN / 2) : tS;
        const float2 sl2 = make_float2(scale_log2, scale_log2);
        int step = 0;      // S_t / P_t phases used
        int o_done = 0;    // O_t phases used
        bool ok = true;
        for (int k = 0; ok; ++k) {
            Item it;
            bool valid;
            if (!(ok = read_desc(k, it, valid)) || !valid) break;
            const int q0t = it.q0 + t * kBM;
            const int q_abs = q0t + row;
            const int n_kv = it.n[t];
            const int j_first = it.kr[t].first;  // first key tile of this query tile
            const int kv_len = it.kv_len;
            float m = -INFINITY;  // running max of scale*log2(e)*s used for P
            float l = 0.f;        // running sum of P in fp32 (exact weights: gives the LSE)
            float l_o = 0.f;      // running sum of P as rounded to bf16 for the P V MMA

            for (int jj = 0; jj < n_kv; ++jj) {
                const int j = j_first + jj;  // key tile index
                if (!wait_warp(bar(L::kBarSFull + t), (step + jj) & 1, 10 + t)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // Hidden keys sit in the last key tile (ragged key tail or the
                // causal diagonal) and, with a window, in the first tiles (keys
                // j <= i - w).  Columns c of this tile are visible iff
                // lim_lo <= c < lim.
                const bool last = jj == n_kv - 1;
                int lim = kBN;
                if (last) {
                    lim = kv_len - j * kBN;
                    if (causal) lim = min(lim, q_abs - j * kBN + 1);
                }
                const bool lower = kWindow && j * kBN < q0t + kBM - window;  // some row's window starts here
                const int lim_lo = q_abs - window + 1 - j * kBN;
                // 64 score columns from TMEM (two 32-column loads), masked.
                auto load64 = [&](int c0, uint32_t (&ra)[32], uint32_t (&rb)[32]) {
                    tmem_ld32(tS + c0, ra);
                    tmem_ld32(tS + c0 + 32, rb);
                    tmem_ld_wait_only();
                    reg_fence(ra);
                    reg_fence(rb);
                    if (last) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            if (c0 + c >= lim) ra[c] = 0xff800000u;  // -inf
                            if (c0 + 32 + c >= lim) rb[c] = 0xff800000u;
                        }
                    }
                    if (lower) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            if (c0 + c < lim_lo) ra[c] = 0xff800000u;
                            if (c0 + 32 + c < lim_lo) rb[c] = 0xff800000u;
                        }
                    }
                };

                // One pass over S: each 64-column half is loaded from TMEM once,
                // its max taken and its P formed against the running max m, which
                // the first half moves when a score passes it by more than the
                // lazy threshold.  The second half moves it only past
                // kInTileLimit; then the first half's stored P and its sums are
                // scaled by 2^(m_before - m) in place.
                struct Sums {
                    float2 a0, a1;  // fp32 sums of P (two chains)
                    float r[4];     // sums of P as rounded to bf16
                };
                auto exp_pack = [&](const uint32_t (&r)[32], uint32_t p_col, float2 nm2, Sums &sm) {
                    uint32_t pk[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float2 x = __ffma2_rn(make_float2(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1])),
                                                    sl2, nm2);
                        const float2 p = make_float2(ex2(x.x), ex2(x.y));
                        if (c & 1)
                            sm.a1 = __fadd2_rn(sm.a1, p);
                        else
                            sm.a0 = __fadd2_rn(sm.a0, p);
                        pk[c] = pack_bf16x2(p.x, p.y);
                        add_bf16x2_f32(sm.r[2 * (c & 1)], sm.r[2 * (c & 1) + 1], pk[c]);
                    }
                    tmem_st16(tP + p_col, pk);
                };
                auto half_max = [&](const uint32_t (&ra)[32], const uint32_t (&rb)[32]) -> float {
                    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        mx[c & 3] = fmax3(mx[c & 3], __uint_as_float(ra[2 * c]), __uint_as_float(ra[2 * c + 1]));
                        mx[c & 3] = fmax3(mx[c & 3], __uint_as_float(rb[2 * c]), __uint_as_float(rb[2 * c + 1]));
                    }
                    return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * scale_log2;
                };
                const float m_old = m;
                Sums sA = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), {0.f, 0.f, 0.f, 0.f}};
                Sums sB = sA;
                uint32_t ra[32], rb[32];
                load64(0, ra, rb);
                {
                    const float t0 = half_max(ra, rb);
                    if (t0 > m + kRescaleThreshold) m = t0;
                }
                if constexpr (kSplitP) {
                    // P_t(j-1) V_{j-1} must have read P_t and updated O_t before
                    // P_t(j) is stored and O_t rescaled.
                    if (jj > 0) {
                        if (!wait_warp(bar(L::kBarPVDone + t), (step + jj - 1) & 1, 18 + t)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                }
                // A row that has seen no visible key yet keeps m = -inf; its
                // scores are all -inf too, so any finite shift gives P = 0.
                float m_use = m == -INFINITY ? 0.f : m;
                exp_pack(ra, 0, make_float2(-m_use, -m_use), sA);
                exp_pack(rb, 16, make_float2(-m_use, -m_use), sA);
                // Second half: score columns 64..127, untouched by the P columns
                // 0..31 written so far.
                load64(64, ra, rb);
                if constexpr (kSplitP) {
                    // All of S_t(j) is in registers: S_t(j+1) may overwrite it.
                    tc_fence_before();
                    mbar_arrive(bar(L::kBarSFree + t));
                }
                {
                    const float t1 = half_max(ra, rb);
                    const bool move = t1 > m + kInTileLimit;
                    // The TMEM loads and stores below are warp-collective: the
                    // whole warp takes the branch; rows whose max did not move
                    // rewrite their P unchanged (beta = 1 is exact).
                    if (__any_sync(0xffffffffu, move)) {
                        const float beta = move ? ex2(m_use - t1) : 1.f;
                        tmem_st_wait();
                        uint32_t pr[32];
                        tmem_ld32(tP, pr);
                        tmem_ld_wait(pr);
                        float r4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            pr[c] = pack_bf16x2(__uint_as_float(pr[c] << 16) * beta,
                                                __uint_as_float(pr[c] & 0xFFFF0000u) * beta);
                            add_bf16x2_f32(r4[2 * (c & 1)], r4[2 * (c & 1) + 1], pr[c]);
                        }
                        tmem_st32(tP, pr);
                        if (move) {
                            m = t1;
                            m_use = t1;
                            sA.r[0] = r4[0];
                            sA.r[1] = r4[1];
                            sA.r[2] = r4[2];
                            sA.r[3] = r4[3];
                            sA.a0 = make_float2(sA.a0.x * beta, sA.a0.y * beta);
                            sA.a1 = make_float2(sA.a1.x * beta, sA.a1.y * beta);
                        }
                    }
                }
                exp_pack(ra, 32, make_float2(-m_use, -m_use), sB);
                exp_pack(rb, 48, make_float2(-m_use, -m_use), sB);
                const float alpha = m != m_old ? ex2(m_old - m) : 1.f;  // 0 on the first visible tile

                // O_t += P_t V_{j-1} is complete (at d = 128 the S_t commit covers
                // it, at d = 64 the wait above), so O_t can be rescaled here; rows
                // whose max did not move keep alpha = 1.
                if (jj > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tO + c * 32, o);
                        tmem_ld_wait(o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st32(tO + c * 32, o);
                    }
                }
                const float2 acc = __fadd2_rn(__fadd2_rn(sA.a0, sA.a1), __fadd2_rn(sB.a0, sB.a1));
                l = fmaf(l, alpha, acc.x + acc.y);
                // O is normalised by the sum of the weights it was built from, so
                // O / l_o is a convex combination of V rows up to the bf16
                // rounding of their relative sizes.
                l_o = fmaf(l_o, alpha,
                           ((sA.r[0] + sA.r[1]) + (sA.r[2] + sA.r[3])) + ((sB.r[0] + sB.r[1]) + (sB.r[2] + sB.r[3])));
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(bar(L::kBarPFull + t));
            }
            if (!ok) break;
            step += n_kv;

            // -------------------------------------------------------- epilogue
            // O_t / l_o -> bf16.  d = 64: 64 columns per warp go through the
            // warp's own 4 KB of shared memory (128-byte swizzle) to one TMA
            // store, which clips rows past N (coalesced: the item's tail is
            // short at this size).  d = 128: 16-byte stores straight from
            // registers (rows past N skipped).  The TMEM reads complete before
            // this warp hands over the next item's P_t, so the next item's
            // first P V MMA cannot overwrite O_t early.
            if (q0t < N) {
                const bool have = n_kv > 0;
                if (have) {
                    // The item's last P V MMA: ODone (d = 128) or the last PVDone
                    // phase (d = 64, step already counts this item's tiles).
                    ok = kSplitP ? wait_warp(bar(L::kBarPVDone + t), (step - 1) & 1, 12 + t)
                                 : wait_warp(bar(L::kBarODone + t), o_done & 1, 12 + t);
                    ++o_done;
                    tc_fence_after();
                    if (!ok) break;
                }
                // Rows with no visible key (l_o = 0) get O = 0 and lse = -inf.
                const float inv_l = have && (!kWindow || l_o > 0.f) ? 1.f / l_o : 0.f;
                auto load_pack = [&](int c, uint32_t (&w)[16]) {
                    uint32_t o[32];
                    if (have) {
                        tmem_ld32(tO + c * 32, o);
                        tmem_ld_wait(o);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = 0u;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
                };
                if constexpr (D == 64) {
                    const int lane = threadIdx.x & 31;
                    const uint32_t stage = s_base + L::kOffStage + warp * L::kStageBytes;
                    // The staging buffer is free once this warp's previous
                    // store has read it.
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int hc = 0; hc < 2; ++hc) {
                        uint32_t w[16];
                        load_pack(hc, w);
                        // Row `lane`, 16-byte chunk u of 8: chunk index XOR (row % 8).
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            st_shared_v4(stage + lane * 128 + (((4 * hc + u) ^ (lane & 7)) << 4), w[4 * u],
                                         w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_4d(&tm_o, stage, 0, q0t + (warp & 3) * 32, it.h, it.b);
                        tma_store_commit();
                    }
                } else {
                    __nv_bfloat16 *orow = out + static_cast<int64_t>(it.b) * ost.batch +
                                          static_cast<int64_t>(it.h) * ost.head + static_cast<int64_t>(q_abs) * ost.row;
#pragma unroll 1
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t w[16];
                        load_pack(c, w);
                        if (q_abs < N) {
                            // Each thread writes its own row: 32-byte stores
                            // fill whole L2 sectors, half as many requests as
                            // 16-byte ones.
                            if (sc.o_v8) {
                                st_global_v8(orow + c * 32, w);
                                st_global_v8(orow + c * 32 + 16, w + 8);
                            } else {
#pragma unroll
                                for (int u = 0; u < 4; ++u)
                                    st_global_v4(orow + c * 32 + u * 8, w[4 * u], w[4 * u + 1], w[4 * u + 2],
                                                 w[4 * u + 3]);
                            }
                        }
                    }
                }
                if (lse != nullptr && q_abs < N) {
                    const float v =
                        have && (!kWindow || l > 0.f) ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
                    lse[static_cast<int64_t>(it.bh) * N + q_abs] = v;
                }
            }
        }
        // Shared memory must outlive the warp's last O store (d = 64).
        if (D == 64 && (threadIdx.x & 31) == 0) tma_store_wait_all();
        __syncwarp();
        tc_fence_before();
    }

    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool kWindow>
int launch(const AttnLaunch &a)
{
    using L = Smem<D>;
    static int configured_device = -1;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (configured_device != dev) {
        if (cudaFuncSetAttribute(attn_fwd_kernel<D, kWindow>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 L::kAlloc) != cudaSuccess)
            return -1;
        configured_device = dev;
    }
    Sched sc{};
    sc.o_v8 = reinterpret_cast<uintptr_t>(a.out) % 32 == 0 && a.ost.batch % 16 == 0 && a.ost.head % 16 == 0 &&
              a.ost.row % 16 == 0;
    sc.H = a.H;
    sc.N = a.N;
    sc.nqp = (a.N + kRowsPerCta - 1) / kRowsPerCta;
    sc.num_bh = a.B * a.H;
    // With the heaviest-first order over all heads, the running CTAs spread
    // over every head and the pairs of one head run at different times, each
    // re-reading the head's keys and values from DRAM (3.8x the K/V bytes at
    // B=4 H=32 N=4096 d=128).  Ordering within groups of heads whose K/V fit
    // 32 MiB keeps them in L2: 0.506 -> ~0.46 ms there and 1.51 -> 1.46 ms at
    // B=1 H=32 N=16384 (2032 MHz, measured with cool-downs; budgets of 64 and
    // 128 MiB gave 1.47 and 1.48 ms).
    const int64_t kv_head = static_cast<int64_t>(a.N) * D * 2 * 2;
    sc.head_group =
        static_cast<int>(std::min<int64_t>(sc.num_bh, std::max<int64_t>(1, (int64_t(32) << 20) / kv_head)));
    // Schedule.  Causal pairs cost 2p + 2 key tiles: pairing p with nqp-1-p
    // makes equal units, which a static stride balances once there are a few
    // per SM (long-context shape: 6.9 per SM, makespan 1.2 % over ideal in a
    // simulation).  With fewer (e.g. 8 heads at N = 16384: 1.7 per SM, a
    // whole unit of tail) or with key lengths, each CTA takes one item and
    // the hardware hands CTAs to SMs as they free up (greedy, heaviest
    // first).  Without the causal mask (or with a window) items cost about
    // the same, and persistent CTAs striding over them keep set-up and drain
    // off the tensor core.
    const int sms = sm_count();
    const int64_t items = static_cast<int64_t>(sc.nqp) * sc.num_bh;
    const int64_t pair_units = static_cast<int64_t>((sc.nqp + 1) / 2) * sc.num_bh;
    const bool causal_full = a.causal && a.window == 0;
    sc.paired = causal_full && a.key_lens == nullptr && pair_units >= 4 * static_cast<int64_t>(sms) ? 1 : 0;
    const int64_t units = sc.paired ? pair_units : items;
    // One CTA per SM (the kernel's shared memory and TMEM allow no more).
    const unsigned grid = static_cast<unsigned>(causal_full && !sc.paired ? units : std::min<int64_t>(units, sms));
    attn_fwd_kernel<D, kWindow><<<grid, kThreads, L::kAlloc, a.stream>>>(
        *a.tm_q, *a.tm_k, *a.tm_v, *a.tm_o, static_cast<__nv_bfloat16 *>(a.out), a.ost, a.lse, a.key_lens, sc,
        static_cast<int>(units), a.scale_log2, a.causal, a.window);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int attn_fwd_launch(const AttnLaunch &a)
{
    const bool w = a.window > 0;
    if (a.d == 64) return w ? launch<64, true>(a) : launch<64, false>(a);
    if (a.d == 128) return w ? launch<128, true>(a) : launch<128, false>(a);
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

#ifdef SDP18_WAIT_TEST
// Test library only (not part of include/attn.h): set the stall item of the
// forward's producer (-1 = none) and read the device error word without
// clearing it.  Both return 0 on success.
extern "C" int attn_test_set_stall(int items)
{
    return cudaMemcpyToSymbol(sdp18::g_test_stall_items, &items, sizeof(int)) == cudaSuccess ? 0 : -1;
}

extern "C" int attn_test_error_word(int *word)
{
    return cudaMemcpyFromSymbol(word, sdp18::g_sdp18_error, sizeof(int)) == cudaSuccess ? 0 : -1;
}
#endif
