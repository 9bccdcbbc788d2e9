// Internal interface between the C ABI (attn_api.cu) and the kernel launcher
// (attn_fwd_sm103.cu).  Not installed, not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace sdp18 {

struct AttnLaunch {
    const CUtensorMap *tm_q, *tm_k, *tm_v, *tm_o;  // 3-D maps over [B*H, N, d] bf16
    float *lse;                                    // [B*H*N] fp32 or nullptr
    const int32_t *key_lens;                       // [B] or nullptr
    int B, H, N, d;
    float scale_log2;  // scale * log2(e)
    int causal;
    int window;  // > 0: query i sees keys j > i - window; 0: no window
    cudaStream_t stream;
};

// 0 on success, -1 on a CUDA error, -2 for an unsupported head dimension.
int attn_fwd_launch(const AttnLaunch &a);

// Reads the device error word of the current device and clears it.
int read_and_clear_device_error(int *value);

}  // namespace sdp18
