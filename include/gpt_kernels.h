/*
 * gpt_kernels.h - per-step entry points of the GB300 GPT library.
 *
 * Each call runs ONE step of the forward pass (the same kernels gpt_forward
 * launches) on caller-owned device buffers, so that every step can be checked
 * on its own against the definitions it implements. All pointers are device
 * pointers, 16-byte aligned; all calls are stream-ordered and asynchronous.
 * Device-side errors (out-of-range ids, expired waits) are recorded in a
 * library-wide device error word that gptk_status() reads and clears.
 *
 * dtype selects the arithmetic: 0 = fp32 SIMT kernels (fp32 operands),
 * 1 = bf16 operands on the tcgen05 tensor-core kernels with fp32 accumulation.
 */
#ifndef GPT_GB300_KERNELS_H
#define GPT_GB300_KERNELS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* GEMM epilogues */
enum {
  GPTK_EPI_BIAS = 0,        /* out = A W^T + bias, stored in dtype (bf16 or fp32) */
  GPTK_EPI_BIAS_GELU = 1,   /* out = gelu_tanh(A W^T + bias) ("第 25 章" §25.3) */
  GPTK_EPI_BIAS_RESID = 2,  /* out (fp32) += A W^T + bias: the residual add (§25.1) */
  GPTK_EPI_F32 = 3          /* out (fp32) = A W^T (+ bias if non-NULL) */
};

/*
 * out[M,N] = epilogue(A[M,K] . W[N,K]^T + bias[N]).
 * A and W are row-major in dtype (nn.Linear orientation, §25.5); bias fp32
 * [N] or NULL; out row-major with row stride N. K and N must be multiples of
 * 8 on the bf16 path (16-byte TMA row strides). Where the bf16 tiles would not
 * fill whole waves of the GPU and K >= 1536, epilogues 0-2 split tiles along K
 * between two CTAs (stream-K, fixed summation order: results do not depend on
 * timing); their fp32 partial tiles and flags are allocated on the stream
 * (stream-ordered allocator) and freed there after the launch.
 */
int gptk_gemm(const void* A, const void* W, const float* bias, void* out, int32_t M, int32_t N,
              int32_t K, int32_t epilogue, int32_t dtype, void* stream);

/*
 * The bf16 products on pairs of CTAs: clusters of two whose tcgen05.mma.cta_group::2 computes
 * 256 x 256 tiles, each CTA staging 128 rows of A and 128 of the tile's W rows per K step.
 * The epilogues of gptk_gemm: GPTK_EPI_BIAS and GPTK_EPI_BIAS_GELU (out bf16), GPTK_EPI_BIAS_RESID
 * (out fp32 += A W^T + bias, the residual add), GPTK_EPI_F32 (out fp32 = A W^T + bias). A and W
 * bf16 row-major [M,K] and [N,K], K and N multiples of 8, 16-byte aligned pointers; bias fp32 [N]
 * or NULL; out row-major [M, N]. ksplit <= 1: whole tiles,
 * or stream-K (as gptk_gemm, workspace on the stream) where whole tiles would leave a part-idle
 * last wave and K >= 1536; ksplit > 1 (GPTK_EPI_BIAS_RESID only): each tile's K range is cut
 * into ksplit slices whose partial products are added into out separately (bias must be NULL;
 * the order of those fp32 additions varies between runs). GPT_ECONFIG if clusters of two with
 * this kernel's shared memory cannot be resident on the device.
 */
int gptk_gemm_pair(const void* A, const void* W, const float* bias, void* out, int32_t M, int32_t N,
                   int32_t K, int32_t epilogue, int32_t ksplit, void* stream);

/*
 * Causal self-attention of one layer ("第 25 章" §25.2).
 * qkv: [B, T, 3C] in dtype (Q, K, U thirds; head h = columns [hD, (h+1)D) of each);
 * y:   [B, T, C] in dtype, heads merged. C = H*D; bf16 path: D in {32, 64}.
 */
int gptk_attention(const void* qkv, void* y, int32_t B, int32_t T, int32_t H, int32_t D,
                   int32_t dtype, void* stream);

/*
 * gptk_attention on the bf16 path that also writes, for every query row, the base-2
 * log-sum-exp of its scaled scores: lse2[(b H + h) T + t] = log2 sum_{s <= t} 2^(q_t . k_s log2(e) / sqrt(D))
 * (fp32, [B*H*T]); the softmax normaliser of "第 25 章" §25.2 that the derivative below reuses.
 */
int gptk_attention_lse(const void* qkv, void* y, float* lse2, int32_t B, int32_t T, int32_t H, int32_t D,
                       void* stream);

/*
 * Derivative of the causal self-attention of one layer (bf16 path; the chain rule through the
 * definitions of §25.2, as the training loop of "预训练一个 Mini GPT" needs it): from qkv [B, T, 3C],
 * the output y [B, T, C] and lse2 of gptk_attention_lse, and dy [B, T, C] (the loss gradient with
 * respect to y), writes dqkv [B, T, 3C] bf16: dQ, dK and dU in the thirds of qkv's layout. D in {32, 64};
 * all four bf16 arrays 16-byte aligned. Its fp32 dQ accumulator (B*T*C*4 bytes) and Dsum scratch are
 * allocated on the stream and freed there after the launches.
 */
int gptk_attention_bwd(const void* qkv, const void* y, const void* dy, const float* lse2, void* dqkv, int32_t B,
                       int32_t T, int32_t H, int32_t D, void* stream);

/*
 * LayerNorm over rows of x [M, C] fp32 ("预训练一个 Mini GPT" 第4步; "GPT-1 学习笔记" §3.2):
 * out (dtype) = (x - mean)/sqrt(var + eps) * g + b; out_f32 (fp32, may alias x, may be NULL)
 * receives the same values in fp32. C must be a multiple of 8 and at most 2048.
 */
int gptk_layernorm(const float* x, const float* g, const float* b, void* out, float* out_f32,
                   int32_t M, int32_t C, float eps, int32_t dtype, void* stream);

/*
 * x[b,t,:] = E[ids[b,t],:] + P[t,:] as fp32 [B*T, C] ("第 25 章" §25.1).
 * wte [V, C] and wpe [>=T, C] in dtype.
 */
int gptk_embed(const int32_t* ids, const void* wte, const void* wpe, float* x, int32_t B,
               int32_t T, int32_t C, int32_t V, int32_t dtype, void* stream);

/*
 * Tied head + per-row cross-entropy: nll[m] = logsumexp_j(h_m . E_j) - h_m . E_{targets[m]}
 * ("第 25 章" §25.4, "预训练一个 Mini GPT" 第6步). h [M, C] and wte [V, C] in dtype;
 * nll fp32 [M]; logits fp32 [M, V] or NULL (written only when non-NULL).
 * The bf16 path allocates its partial-logsumexp scratch on the stream.
 */
int gptk_lmhead_ce(const void* h, const void* wte, const int32_t* targets, float* nll,
                   float* logits, int32_t M, int32_t V, int32_t C, int32_t dtype, void* stream);

/*
 * gptk_lmhead_ce without any device allocation (bf16 path only; the source
 * pages have no counterpart: this is an operational variant of the step
 * above). For callers that cannot allocate device memory while they run: a
 * server whose memory budget is fixed at start-up, a framework whose caching
 * allocator already holds the free memory, or a loop that cannot take the
 * synchronisation an allocation may cause. The scratch lives in a fixed
 * library array of 2,097,152 floats (8 MiB) that every GPU loading the library
 * keeps until the process exits; the call returns GPT_EINVAL when
 * M * (2 * ceil(V / 256) + 1) exceeds it (e.g. at most 5,309 rows for V = 50257).
 * The first call on each device looks up that array's device address (with the
 * device current); make that first call before any stream capture. All calls
 * share the array, so calls whose GPU work overlaps race; order them on one
 * stream. The looked-up address is kept for the life of the process: do not
 * use this entry after a reset of the device (cudaDeviceReset or a destroyed
 * and recreated primary context), which invalidates it. d_err: caller-owned
 * device int that receives a nonzero code (and keeps the first one) if a target
 * is outside [0, V) or a bounded wait expired; the nll of a row whose target is
 * out of range is then unspecified, the other rows are still correct. With
 * d_err NULL such errors are not reported anywhere. nll as in gptk_lmhead_ce.
 * No logits.
 */
int gptk_lmhead_ce_noalloc(const void* h, const void* wte, const int32_t* targets, float* nll,
                           int32_t M, int32_t V, int32_t C, int32_t* d_err, void* stream);

/* Deterministic mean of nll[0..M) into *loss (device fp32). */
int gptk_mean(const float* nll, int32_t M, float* loss, void* stream);

/* Synchronise the stream, then read and clear the per-step device error word. */
int gptk_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GPT_GB300_KERNELS_H */
