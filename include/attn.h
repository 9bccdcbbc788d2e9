/*
 * attn.h -- C ABI of the B300 (sm_103a) multi-head scaled dot-product
 * attention forward.
 *
 * The operation (one call computes every batch b and head h):
 *
 *   O[b,h] = softmax(Q[b,h] K[b,h]^T * scale + mask) V[b,h]
 *   lse[b,h,i] = ln sum_j exp(scale * q_i . k_j)     over the visible keys j
 *
 *   -- hotelren.com "AI attention: essence and evolution", sec. 2.1 (the
 *      softmax-attention formula, scaled by 1/sqrt(d_k)) and ch.1 code (the
 *      mask fills hidden scores with -inf before the softmax);
 *   -- aicoding.csdn.net "Why attention stalls large-model training",
 *      sec. 2.2 (max-shifted softmax and the log-sum-exp, natural log);
 *   -- hotelren.com sec. 4.1 (FlashAttention-1: tiles of Q and K/V, online
 *      softmax, the n x n score matrix is never written out).
 *
 * attn_fwd_window adds a sliding window (keys j > i - w only); attn_decode
 * computes one query per (batch, head) against a key/value cache;
 * attn_mha_fwd runs a whole multi-head self-attention block.
 *
 * Mask (attn_fwd): key j is visible to query i iff j < key_lens[b] (a key-padding mask,
 * lshu.cn "Self-attention meets the compute wall", sec. 4.1 and 5.2) and,
 * when causal != 0, j <= i (only earlier positions and the query itself;
 * hotelren.com sec. 2.1 note 2).  A hidden key gets exactly zero weight.
 * A query row with no visible key (only possible with key_lens[b] == 0)
 * gets O = 0 and lse = -inf.
 *
 * Every call is asynchronous on `stream`; the library never allocates device
 * memory and never synchronises inside attn_fwd.
 */
#ifndef SDP18_ATTN_H
#define SDP18_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_EINVAL = -1,      /* bad argument: null pointer, negative size, index overflow, scale */
    ATTN_EUNSUPPORTED = -2,/* head dimension d other than 64 or 128 */
    ATTN_EALIGN = -3,      /* a tensor pointer not 16-byte aligned (TMA requirement) */
    ATTN_ECUDA = -4,       /* CUDA runtime/driver error (launch, tensor-map encode, no sm_103a device) */
    ATTN_EDEVICE = -5,     /* the kernel reported an error (a bounded wait ran out) */
    ATTN_ETOOLARGE = -6    /* the problem needs more scratch than attn_decode_noalloc's fixed area */
} attn_status;

/*
 * attn_fwd -- attention forward for all B*H heads in one launch.
 *
 * q, k, v : device, bf16, [B, H, N, d], contiguous, d fastest (the
 *           multi-head split layout (batch, heads, seq_len, head_dim) of
 *           hotelren.com sec. 2.2).  Read only.
 * out     : device, bf16, [B, H, N, d], contiguous.  Written: every row
 *           0..N-1 of every head, fp32-accumulated and rounded to nearest
 *           even.  Must not overlap q, k, v or lse.
 * lse     : device, fp32, [B, H, N], or NULL (not written).  Natural-log
 *           log-sum-exp of the scaled, masked logits of each query row.
 * B, H, N : batch, heads, sequence length (queries = keys = N).  Negative
 *           -> ATTN_EINVAL.  B*H*N == 0 -> ATTN_OK, nothing launched, no
 *           pointer checked.  B*H and N must each be < 2^31 and the tile
 *           grid ceil(N/128)*B*H must fit a 1-D grid, else ATTN_EINVAL.
 * d       : head dimension, 64 or 128 (else ATTN_EUNSUPPORTED).
 * scale   : multiplier of q.k, finite and > 0 (else ATTN_EINVAL); usually
 *           1/sqrt(d).
 * causal  : non-zero = query i sees keys j <= i only.
 * key_lens: device, int32 [B], or NULL (all N keys visible).  The kernel
 *           clamps each value to [0, N]; keys j >= key_lens[b] are hidden
 *           for every head and every query of batch b.  Query rows are never
 *           masked: all N rows are computed and written.
 * stream  : CUDA stream the kernel is launched on.
 *
 * Ownership: every buffer belongs to the caller and must stay valid until
 * the stream has finished the call.  Returns ATTN_OK once launched; errors
 * found on the host are returned before anything is enqueued.  Device-side
 * errors are reported by attn_check_device.
 */
attn_status attn_fwd(const void *q, const void *k, const void *v,
                     void *out, float *lse,
                     int B, int H, int N, int d, float scale, int causal,
                     const int32_t *key_lens, attn_stream_t stream);

/*
 * attn_fwd_window -- attn_fwd with a sliding window of `window` positions.
 *
 * Same arguments, layout, ownership and errors as attn_fwd, plus:
 * window  : >= 0.  When 0 < window < N, query i additionally sees only keys
 *           j > i - window: with causal != 0 that is the last `window`
 *           positions up to and including i (sliding-window attention,
 *           aicoding.csdn.net "Why does attention stall large-model
 *           training", sec. 4.3, window w = 512; local window attention at
 *           O(n w), hotelren.com "AI attention: essence and evolution",
 *           ch.1 table).  0 or >= N: no window (identical to attn_fwd).
 *           Negative -> ATTN_EINVAL.  Key tiles outside every row's window
 *           are not visited.  A row whose window holds no visible key (only
 *           possible together with key_lens) gets O = 0 and lse = -inf.
 */
attn_status attn_fwd_window(const void *q, const void *k, const void *v,
                            void *out, float *lse,
                            int B, int H, int N, int d, float scale, int causal,
                            const int32_t *key_lens, int window, attn_stream_t stream);

/*
 * attn_decode -- one new query per (batch, head) against a key/value cache.
 *
 *   O[b,h] = softmax(q[b,h] K[b,h,:len]^T * scale) V[b,h,:len],
 *   lse[b,h] = ln sum_{j < len} exp(scale * q . k_j),   len = cache_lens[b]
 *
 * The cache is the pages' [batch, heads, seq_len, head_dim] key/value store
 * that each generation step appends one row to (hotelren.com "AI attention:
 * essence and evolution", sec. 3.1); the new token's own key and value are
 * expected to be appended already, so every cached key is visible.
 *
 * q        : device, bf16, [B, H, d] contiguous.
 * k_cache,
 * v_cache  : device, bf16, [B, H, L, d] contiguous (L = allocated rows).
 * out      : device, bf16, [B, H, d].  lse: device fp32 [B, H] or NULL.
 * d        : 64 or 128 (else ATTN_EUNSUPPORTED); scale finite and > 0.
 * cache_lens: device int32 [B] or NULL (all L rows hold keys); clamped to
 *           [0, L] on the device.  len == 0 gives O = 0, lse = -inf.
 * workspace: device scratch of at least attn_decode_workspace_size(B, H, L,
 *           d) bytes, 16-byte aligned, owned by the caller; the call
 *           overwrites it (no zeroing needed) and it must not be shared with
 *           another call in flight.  Missing or too small -> ATTN_EINVAL.
 * All tensor pointers 16-byte aligned (else ATTN_EALIGN).  B*H == 0 -> OK,
 * nothing launched.  Asynchronous on `stream`; allocates nothing.
 */
attn_status attn_decode(const void *q, const void *k_cache, const void *v_cache,
                        void *out, float *lse,
                        int B, int H, int L, int d, float scale,
                        const int32_t *cache_lens, void *workspace, size_t workspace_bytes,
                        attn_stream_t stream);

/* Bytes of workspace attn_decode needs for these sizes (0 for invalid sizes). */
size_t attn_decode_workspace_size(int B, int H, int L, int d);

/*
 * attn_decode_noalloc -- attn_decode for callers that cannot allocate.
 *
 * The pages have no counterpart; this entry point exists for callers that
 * may not call cudaMalloc once they are running (a serving or real-time loop
 * whose memory was fixed at start-up, a host program that lends this library
 * a stream but no allocator, or a step loop that cannot afford cudaMalloc's
 * implicit device synchronisation).  Same arguments, results and errors as
 * attn_decode, without the workspace: the split partials go to one fixed
 * 8 MiB array of device memory that the library holds on every device that
 * loads it, for the life of the process.  The call allocates nothing.
 *
 * - Arguments are checked exactly as attn_decode checks them, and in the
 *   same order; only then do problems whose attn_decode_workspace_size
 *   exceeds 8 MiB return ATTN_ETOOLARGE, before anything is launched (about
 *   16,000 (batch, head) pairs at d = 128; use attn_decode with a caller
 *   workspace beyond that).
 * - The first call on each device looks up that device's array address
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   The address is cached per device together with the id of the context it
 *   was taken in; after cudaDeviceReset (a new context) the next call looks
 *   it up again.
 * - Every call on a device shares the one array and leaves its partials in
 *   it.  Nothing in it needs clearing (each call writes every slot it reads),
 *   but calls that overlap on the GPU -- on different streams, or from
 *   different host threads without ordering -- race on it: serialise them.
 */
attn_status attn_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                void *out, float *lse,
                                int B, int H, int L, int d, float scale,
                                const int32_t *cache_lens, attn_stream_t stream);

/*
 * attn_mha_fwd -- a multi-head self-attention block without biases:
 *
 *   [Q | K | V] = x W_qkv,  heads split from the columns (head h = columns
 *   h*d .. h*d+d-1 of each part),  O_h = attention(Q_h, K_h, V_h) with scale
 *   1/sqrt(d) (the causal and key-length rules of attn_fwd),  merged heads
 *   M = [O_0 | ... | O_{H-1}],  out = M W_o
 *
 * -- cnnetsun.cn "Transformer QKV bottlenecks on long sequences", sec. 2
 *    (MinimalSelfAttention: Q/K/V projections, split heads, scaled dot-product
 *    attention, merge, output projection); qqiyuan.cn "Multi-head attention in
 *    the Transformer: implementation and performance optimisation" (one fused
 *    [E, 3E] projection in place of three).
 *
 * x      : device bf16 [B, N, E] (E = H * d, d = 64 or 128, else
 *          ATTN_EUNSUPPORTED; E % H != 0 -> ATTN_EINVAL).
 * w_qkv  : device bf16 [E, 3E] row-major, Q, K, V column blocks in order.
 * w_o    : device bf16 [E, E] row-major.
 * out    : device bf16 [B, N, E].  lse: device fp32 [B, H, N] or NULL.
 * key_lens: as in attn_fwd.  causal: as in attn_fwd.
 * workspace: caller-owned device memory of attn_mha_workspace_size(B, N, E)
 *          bytes (16-byte aligned) that the call overwrites: the bf16 Q/K/V
 *          rows and the merged heads.
 * Q/K/V and M are bf16 tensors (fp32 accumulation, rounded to nearest even).
 * The two projections run on this library's tcgen05 GEMM kernel (128 x 256
 * output tiles, persistent CTAs), the attention on its attention kernel,
 * which reads the heads straight out of the [B, N, 3E] rows through strided
 * tensor maps (no transpose kernels).  Three launches, asynchronous on
 * `stream`; nothing is allocated.
 */
attn_status attn_mha_fwd(const void *x, const void *w_qkv, const void *w_o, void *out, float *lse,
                         int B, int N, int E, int H, int causal, const int32_t *key_lens,
                         void *workspace, size_t workspace_bytes, attn_stream_t stream);

/* Bytes of workspace attn_mha_fwd needs (0 for invalid sizes). */
size_t attn_mha_workspace_size(int B, int N, int E);

/*
 * attn_bwd -- gradients of attn_fwd with respect to q, k and v:
 *
 *   P = softmax(scale q k^T + mask) (rebuilt from lse, never stored),
 *   dV = P^T dO,  dP = dO V^T,  D_i = dO_i . O_i,  dS = P * (dP - D),
 *   dQ = scale dS K,  dK = scale dS^T Q
 *
 * -- the chain rule through O = P V and the row softmax; the backward pass
 *    reuses the softmax probabilities kept from the forward (hotelren.com
 *    "AI attention: essence and evolution", sec. 4.2), here recomputed from
 *    the forward's log-sum-exp so that no N x N matrix exists.
 *
 * q, k, v : device bf16 [B, H, N, d] contiguous, the forward's inputs.
 * out     : device bf16 [B, H, N, d], the forward's output for q, k, v.
 * dout    : device bf16 [B, H, N, d], the gradient of the loss w.r.t. out.
 * lse     : device fp32 [B, H, N], the forward's log-sum-exp (not NULL).
 * dq, dk, dv: device bf16 [B, H, N, d], written (fp32 accumulation, rounded
 *           to nearest even).  Rows of dk/dv for hidden keys are 0; rows of
 *           dq for queries with no visible key are 0.
 * B, H, N, d, scale, causal, key_lens: as in attn_fwd (same checks, same
 *           errors).
 * workspace: caller-owned device memory of attn_bwd_workspace_size(B, H, N, d)
 *           bytes, 16-byte aligned, overwritten by the call (an fp32 dQ
 *           accumulator and the D vector).
 * Three launches on `stream` (D and accumulator reset; one CTA per 128 keys
 * of one head accumulating dK, dV in tensor memory and adding its dQ partials
 * into the fp32 accumulator with bulk tensor reduce-add copies; dQ
 * conversion).  The order of the fp32 dQ additions is not fixed, so dq may
 * differ between runs in the last bf16 place.
 */
attn_status attn_bwd(const void *q, const void *k, const void *v, const void *out, const void *dout,
                     const float *lse, void *dq, void *dk, void *dv,
                     int B, int H, int N, int d, float scale, int causal,
                     const int32_t *key_lens, void *workspace, size_t workspace_bytes,
                     attn_stream_t stream);

/*
 * attn_bwd_window -- attn_bwd for the forward of attn_fwd_window: the same
 * arguments, layout, ownership and errors, plus
 * window  : >= 0, the forward's window (query i sees keys j > i - window when
 *           0 < window < N; 0 or >= N: none).  Negative -> ATTN_EINVAL.  lse
 *           and out must come from attn_fwd_window with the same window.  Key
 *           tiles meet only the query tiles inside their windows.
 */
attn_status attn_bwd_window(const void *q, const void *k, const void *v, const void *out, const void *dout,
                            const float *lse, void *dq, void *dk, void *dv,
                            int B, int H, int N, int d, float scale, int causal,
                            const int32_t *key_lens, int window, void *workspace, size_t workspace_bytes,
                            attn_stream_t stream);

/* Bytes of workspace attn_bwd and attn_bwd_window need (0 for invalid sizes). */
size_t attn_bwd_workspace_size(int B, int H, int N, int d);

/*
 * attn_check_device -- synchronise `stream`, then read and clear the
 * library's device error word on the current device.  Returns ATTN_EDEVICE
 * if a kernel since the last check gave up on a bounded wait (its outputs are
 * then incomplete), ATTN_ECUDA on a CUDA error, else ATTN_OK.
 */
attn_status attn_check_device(attn_stream_t stream);

/* Static, human-readable name of a status code. */
const char *attn_status_str(attn_status s);

/* ABI version of this header (bumped on any signature change). */
int attn_abi_version(void);

/*
 * attn_tensor_map_cache_stats -- counters of the library's tensor-map cache.
 *
 * Every call describes its tensors to the TMA engine with tensor maps; an
 * encoded map depends only on the buffer address, the sizes, strides and the
 * tile shape, so the library keeps the last 256 distinct maps (a fixed table
 * guarded by a mutex; nothing is allocated) and re-encodes only on a miss
 * (see the latency-bound shapes of lshu.cn "Self-attention meets the compute
 * wall", sec. 4.1: many small padded batches).  A caller that reuses its
 * buffers pays a table lookup instead of up to five encodes per call.
 * hits, misses: host pointers (either may be NULL) that receive the number of
 * maps found in, and added to, the table since the library was loaded.
 */
void attn_tensor_map_cache_stats(uint64_t *hits, uint64_t *misses);

#define ATTN_ABI_VERSION 6

#ifdef __cplusplus
}
#endif

#endif /* SDP18_ATTN_H */
