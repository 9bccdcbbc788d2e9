// Internal interface between the C ABI (attn_api.cu) and the kernel launcher
// (attn_fwd_sm103.cu).  Not installed, not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace sdp18 {

// Element strides of the output's rows, heads and batches (row stride a
// multiple of 8 elements: rows are written with 16-byte stores).
struct OStrides {
    int64_t row, head, batch;
};

struct AttnLaunch {
    const CUtensorMap *tm_q, *tm_k, *tm_v;  // 4-D maps {d, N, H, B} bf16, 64 x 128 boxes
    const CUtensorMap *tm_o;                // 4-D map {d, N, H, B} bf16, 64 x 32 boxes (d = 64 stores)
    void *out;                              // the same output, addressed through ost (d = 128 stores)
    OStrides ost;
    float *lse;                             // [B*H*N] fp32 or nullptr
    const int32_t *key_lens;                       // [B] or nullptr
    int B, H, N, d;
    float scale_log2;  // scale * log2(e)
    int causal;
    int window;  // > 0: query i sees keys j > i - window; 0: no window
    cudaStream_t stream;
};

// 0 on success, -1 on a CUDA error, -2 for an unsupported head dimension.
int attn_fwd_launch(const AttnLaunch &a);

// Streaming multiprocessors of the current device (148 when it cannot be
// queried, e.g. a size query on a host without a GPU).
int sm_count();

// Decode (one query per (b, h) against a K/V cache of L rows).
struct DecodeSplit {
    int splits;  // cache chunks per (b, h)
    int chunk;   // keys per chunk (a multiple of 64)
};
DecodeSplit decode_split(int B, int H, int L);

struct DecodeLaunch {
    const void *q, *k, *v;      // bf16 [B*H, d], [B*H, L, d], [B*H, L, d]
    void *out;                  // bf16 [B*H, d]
    float *lse;                 // fp32 [B*H] or nullptr
    const int32_t *cache_lens;  // [B] or nullptr
    float *part_o;              // fp32 [B*H, splits, d] workspace
    float *part_lse;            // fp32 [B*H, splits] workspace
    int B, H, L, d, splits, chunk;
    int L_keys;  // cached rows that hold keys (L_keys <= L; L is the row stride)
    float scale_log2;
    cudaStream_t stream;
};
// 0 on success, -1 on a CUDA error, -2 for an unsupported head dimension.
int attn_decode_launch(const DecodeLaunch &a);

// Backward (dQ, dK, dV).
struct BwdLaunch {
    const CUtensorMap *tm_q, *tm_k, *tm_v, *tm_do;  // 4-D maps {d, N, H, B} bf16, 64 x 128 boxes
    const CUtensorMap *tm_dq;                       // 3-D map {d, N, B*H} fp32 over dqacc, 32 x 32 boxes
    const void *out, *dout;                         // bf16 [B*H*N, d] (contiguous)
    const float *lse;                               // [B*H*N] natural log, from the forward
    float *stats;                                   // workspace [2][B*H][n_pad]: lse*log2e, D = dO . O
    float *dqacc;                                   // workspace [B*H*N, d]: fp32 dQ accumulator
    void *dq, *dk, *dv;                             // bf16 [B*H*N, d]
    const int32_t *key_lens;
    int B, H, N, d;
    float scale;
    int causal;
    int window;  // > 0: query i sees keys j > i - window
    cudaStream_t stream;
};
// 0 on success, -1 on a CUDA error, -2 for an unsupported head dimension.
int attn_bwd_launch(const BwdLaunch &a);

// Dense bf16 GEMM C[M, N] = A[M, K] B[K, N] (row-major, fp32 accumulation,
// bf16 out) for the multi-head block's projections.
struct GemmLaunch {
    const CUtensorMap *tm_a;  // 2-D {K, M} bf16, box 64 x 128, 128-byte swizzle
    const CUtensorMap *tm_b;  // 2-D {N, K} bf16, box 64 x 64, 128-byte swizzle
    void *c;                  // bf16 rows of ldc elements (16-byte aligned rows)
    int64_t ldc;
    int M, N, K;              // K a multiple of 64, N a multiple of 8
    cudaStream_t stream;
};
// 0 on success, -1 on a CUDA error, -2 for unsupported sizes.
int gemm_bf16_launch(const GemmLaunch &g);
int read_and_clear_gemm_error(int *value);

// Reads the device error word of the current device and clears it.
int read_and_clear_device_error(int *value);
// Same for the word the backward kernel writes.
int read_and_clear_bwd_error(int *value);

}  // namespace sdp18
