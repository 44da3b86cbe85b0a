// Host-side launchers of the library's kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gptgb {

// device error codes written to the error word (the host maps them to GPT_E* values)
enum : int {
  GPT_DEV_OK = 0,
  GPT_DEV_ETOKEN = 1,     // a token id outside [0, V)
  GPT_DEV_ETARGET = 2,    // a target outside [0, V)
  GPT_DEV_ETIMEOUT = 3,   // a bounded wait expired
  GPT_DEV_EALIGN = 4,     // dynamic shared memory not 1024-byte aligned
};

enum Epilogue : int {
  EPI_BIAS_OUT = 0,       // out (bf16 or fp32) = acc + bias
  EPI_BIAS_GELU_OUT = 1,  // out = gelu(acc + bias)
  EPI_BIAS_RESID = 2,     // out fp32 += acc + bias
  EPI_F32 = 3,            // out fp32 = acc (+ bias)
  EPI_CE = 4,             // per-row partial logsumexp of the tile, target capture
  EPI_CE_GRAD = 5,        // out bf16 = (exp(z - lse) - [col == target]) * scale, lse = nll + ztgt per row
  EPI_F32_OUT = 6,        // out fp32 = acc (+ bias) through the TMA store (fp32 [M,N] box 32x32)
  EPI_GELU_GRAD = 7,      // out bf16 = acc * gelu'(u), u = aux bf16 [M, N] (the GELU's input)
  EPI_BIAS_GELU_UOUT = 8, // out bf16 = gelu(acc + bias) through tmC and u = acc + bias (bf16) through tmC2
};

struct GemmArgs {
  int M, N, K;
  const float* bias;        // [N] or nullptr
  void* out;                // row-major, row stride ldo
  int ldo;
  int gelu_erf;             // 0 tanh form, 1 erf form
  const int32_t* targets;   // EPI_CE: [M]
  float* pmax;              // EPI_CE: [NB, M] per tile a reference logit m: one of the row's logits
                            //         in the tile, at most 64 ln 2 below their maximum
  float* psum;              // EPI_CE: [NB, M] sum over the tile of exp(z - m)
  float* ztgt;              // EPI_CE: [M] the target's logit
  float* logits;            // EPI_CE: [M, ldo] fp32 or nullptr
  int* err;                 // device error word
  int m_fastest;            // tile order: 1 = consecutive tiles walk M
  // Stream-K (EPI_BIAS_OUT, EPI_BIAS_GELU_OUT, EPI_BIAS_RESID): each CTA takes an equal
  // range of (tile, K block) units; a tile split between two CTAs is finished by the
  // CTA holding its first K blocks after adding the other's fp32 partial.
  float* sk_part;           // [grid + 2][BM x 256] fp32 partial tiles, or nullptr: whole tiles per CTA
  int* sk_flag;             // [grid + 2][4] per-warp "partial written" flags, zero between launches
  const int* sk_wait_flag;  // nullptr, or flags the finishing CTAs wait on instead of sk_flag (set by nobody:
                            //   the failure-detection check makes those bounded waits expire)
  long long wait_limit;     // SM cycles a finishing CTA waits for its partner's flag (0: kWaitLimitCycles)
  // Split-K (EPI_BIAS_RESID without bias, whole-tile launches): ksplit > 1 deals (tile, K slice)
  // units, slice s covering K blocks [s KB / ksplit, (s + 1) KB / ksplit); each adds its partial
  // into the fp32 output with the reduce-add store.
  int ksplit;
  int mn_major;             // EPI_BIAS_RESID: both operands MN-major, A stored [K, M] and W [K, N] row-major
                            //   (tensor maps with 64 x 64 boxes): out[M, N] += A^T W summed over K
  int b_const;              // 1: W was not written by the previous kernel on the stream (weights), so its
                            //    first stages may be requested before waiting for that kernel
  const void* aux;          // EPI_GELU_GRAD: u, bf16 [M, N] row-major
  const float* row_nll;     // EPI_CE_GRAD: [M] per-row loss; with ztgt gives the row's logsumexp
  float scale;              // EPI_CE_GRAD: factor of the gradient (1 / rows of the mean)
};
// Floats of stream-K partial workspace for a grid of `grid` CTAs, and ints of flags.
size_t gemm_sk_part_floats(int grid);
size_t gemm_sk_flag_ints(int grid);
// Whether launch_gemm_tc splits tiles across CTAs (given a workspace) for this shape.
bool gemm_tc_stream_k(int M, int N, int K, int epi, int grid_limit);

// ---- tensor-core (bf16) path
constexpr int kGemmBM = 128;
constexpr int kGemmBK = 64;
int gemm_tc_bn();                      // N extent of a GEMM tile (TMA box rows of W)
int gemm_tc_num_ntiles(int N);
// tmC: the output for the TMA-store epilogues (bf16 [M,N] box 64x32 for EPI_BIAS_OUT /
// EPI_BIAS_GELU_OUT, fp32 [M,N] box 32x32 for EPI_BIAS_RESID / EPI_F32; unused by EPI_CE).
constexpr int kEpiRows = 32;
cudaError_t launch_gemm_tc(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                           const GemmArgs& a, int epi, int grid_limit, cudaStream_t s);
// EPI_BIAS_RESID (out fp32 += A W^T + bias), EPI_F32_OUT (out fp32 = A W^T + bias), EPI_BIAS_OUT or
// EPI_BIAS_GELU_OUT (bf16 out) on CTA pairs (clusters of two, tcgen05.mma.cta_group::2): 256 x 256
// tiles, each CTA staging its 128 A rows and 128 of the tile's W rows per K block, so tmB must have a
// box of 128 rows (kGemmBM) instead of gemm_tc_bn(); tmC as for launch_gemm_tc. Whole tiles, stream-K (given the
// workspace, for K >= 1536 where whole tiles leave a part-idle last wave) or split-K (EPI_BIAS_RESID,
// ksplit > 1, no bias). At most max_pairs pairs (and no more than can be resident).
// cudaErrorNotSupported: clusters of two with this kernel's shared memory cannot run on this device
// (use launch_gemm_tc).
cudaError_t launch_gemm_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, const GemmArgs& a,
                             int epi, int max_pairs, cudaStream_t s);
int gemm_pair_capacity();               // CTA pairs of that kernel resident at once (0: none)
bool gemm_pair_stream_k(int M, int N, int K, int max_pairs);   // whether it splits tiles (needs the workspace)
// The same with a second output map (EPI_BIAS_GELU_UOUT: tmC2 receives the GELU's input).
cudaError_t launch_gemm_tc2(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                            const CUtensorMap& tmC2, const GemmArgs& a, int epi, int grid_limit, cudaStream_t s);

constexpr int kAttnBQ = 128;
// sched: 2 device ints, zero before the launch; the kernel's CTAs take work items from it and the
// last CTA to finish sets it back to zero. Launches sharing one sched must be ordered.
// lse2 (nullable): fp32 [B*H][T] receives each query row's base-2 log-sum-exp of its scaled scores
// (log2 of the softmax denominator in units where the probabilities are 2^(s log2(e)/sqrt(D) - lse2)).
cudaError_t launch_attention_tc(const CUtensorMap& tm_qkv, void* y, int B, int T, int H, int D,
                                int* err, int* sched, cudaStream_t s, float* lse2 = nullptr);

// ---- row-wise kernels (both paths)
// Row m is token m of its sequence at position pos0 + m % T (pos0 read from pos_dev when non-null).
cudaError_t launch_embed(const int32_t* ids, const void* wte, const void* wpe, int wdt, float* x,
                         void* out, int out_mode, int odt, const float* g, const float* b,
                         int M, int T, int C, int V, float eps, int* err, cudaStream_t s, int pos0 = 0,
                         const int* pos_dev = nullptr);
cudaError_t launch_layernorm(const float* x, const float* g, const float* b, void* out, int odt,
                             float* out_f32, int M, int C, float eps, cudaStream_t s);
// nll per row from the head's partials; block_sums (nullable) receives one sum of
// nll per ce_combine_blocks(M) block, in a fixed order, for launch_mean.
cudaError_t launch_ce_combine(const float* pmax, const float* psum, const float* ztgt,
                              const int32_t* targets, float* nll, float* block_sums, int M, int NB, int V,
                              int* err, cudaStream_t s);
int ce_combine_blocks(int M);
// loss = sum(part[0..n)) / M in a fixed order
cudaError_t launch_mean(const float* part, int n, int M, float* loss, cudaStream_t s);

// ---- fp32 SIMT parity path
cudaError_t launch_gemm_simt(const float* A, const float* W, const float* bias, float* out,
                             int M, int N, int K, int ldo, int epi, int gelu_erf, cudaStream_t s);
cudaError_t launch_attention_simt(const float* qkv, float* y, int B, int T, int H, int D,
                                  cudaStream_t s);
cudaError_t launch_ce_rows(const float* logits, const int32_t* targets, float* nll, int M, int V,
                           int* err, cudaStream_t s);

// ---- backward pass (bf16 path)
// dst[c * ldd + r] = src[r * lds + c] for a bf16 [rows, cols] matrix; colsum (nullable) += its column sums.
cudaError_t launch_transpose_bf16(const void* src, int rows, int cols, int lds, void* dst, int ldd, cudaStream_t s,
                                  float* colsum = nullptr);
// fp32 [rows, cols] (dense) -> bf16 copy dst (nullable) and bf16 transpose dstT [cols, ldt] (nullable);
// colsum (nullable, needs dstT) += the column sums of the fp32 values.
cudaError_t launch_cast_transpose(const float* src, int rows, int cols, void* dst, void* dstT, int ldt, cudaStream_t s,
                                  float* colsum = nullptr);
// out[c] += sum over rows of src[r * lds + c] (src bf16 or fp32).
cudaError_t launch_colsum(const void* src, int bf16, int rows, int cols, int lds, float* out, int num_sms,
                          cudaStream_t s);
// LayerNorm derivative per row: dx_io = (add ? dx_io : 0) + dLN/dx . dy; dg += sum dy xh, db += sum dy.
// dy may be dx_io itself when add == 0.
cudaError_t launch_layernorm_bwd(const float* x, const float* g, const float* dy, float* dx_io, int add, float* dg,
                                 float* db, int M, int C, float eps, int num_sms, cudaStream_t s);
// dE[id[m]] += dx0[m], dP[m % T] += dx0[m].
cudaError_t launch_embed_bwd(const float* dx0, const int32_t* ids, float* dE, float* dP, int M, int T, int C, int V,
                             cudaStream_t s);
// Causal attention derivative on tcgen05, from the forward's row log-sum-exp (lse2 [B*H][T], base 2 of the
// scaled scores): dqkv [B*T, 3C] bf16 from qkv [B*T, 3C], the output y and its gradient dy ([B*T, C] bf16).
// tm_qkv is the qkv map of make_tmap_qkv (128-row boxes), tm_dy the same over dy [B][T][C], tm_dkv
// make_tmap_attn_out over dqkv [B][T][3C] (dK and dU are stored there), tm_dq make_tmap_bt_f32 over dqacc
// [B][T][C] fp32 scratch (cleared by the call; dQ goes to dqkv's first third). dsum: fp32 [B*H][T]
// scratch. sched: 2 ints as for launch_attention_tc. D = 32 or 64. A memset and three kernels: Dsum, the
// derivative, dQ to bf16.
cudaError_t launch_attention_bwd_tc(const CUtensorMap& tm_qkv, const CUtensorMap& tm_dy, const CUtensorMap& tm_dkv,
                                    const CUtensorMap& tm_dq, const void* y, const void* dy, const float* lse2,
                                    float* dsum, float* dqacc, void* dqkv, int B, int T, int H, int D, int* err,
                                    int* sched, cudaStream_t s);

// One parameter tensor for the optimiser: values [off, off + n) of the flat gradient, master and
// moment arrays, stored at dst (bf16 when bf16 != 0, else fp32); decay: decoupled weight decay applies.
struct OptSeg {
  long long off, n;
  void* dst;
  int bf16, decay;
};
// AdamW over nseg segments (see adamw_kernel); bc1 = 1 - b1^t, bc2 = 1 - b2^t.
cudaError_t launch_adamw(const OptSeg* segs, int nseg, const float* grad, float* master, float* m1, float* m2, float lr,
                         float b1, float b2, float eps, float wd, float bc1, float bc2, cudaStream_t s);
// master = the parameters' current values.
cudaError_t launch_master_init(const OptSeg* segs, int nseg, float* master, cudaStream_t s);

// ---- TMA descriptors (host)
// 2-D row-major bf16 matrix [rows, cols] (row stride ld elements, 0 = cols) with a box of
// box_rows x 64 columns, 128-byte swizzle.
bool make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_rows, uint64_t ld = 0);
// General 2-D row-major matrix (bf16 or fp32) with a box of box_rows x box_cols, box_cols * elem_bytes == 128,
// 128-byte swizzle (the GEMM epilogue's staging layout); row stride ld elements (0 = cols).
bool make_tmap_2d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t rows, uint64_t cols,
                  uint32_t box_cols, uint32_t box_rows, uint64_t ld = 0);
// qkv viewed as [B][T][3C] bf16 with a box of 128 rows x D columns (one batch).
bool make_tmap_qkv(CUtensorMap* map, const void* base, int B, int T, int C3, int D);
// y viewed as [B][T][C] bf16 with a box of 32 rows x D columns (the attention kernel's output stores).
bool make_tmap_attn_out(CUtensorMap* map, const void* base, int B, int T, int C, int D);
// fp32 [B][T][C] with a box of 32 rows x 32 columns (the attention derivative's dQ reduce-adds).
bool make_tmap_bt_f32(CUtensorMap* map, const void* base, int B, int T, int C);

// ---- incremental decoding (bf16)
constexpr int kGemvMaxRows = 16;       // rows per matrix-vector launch
// out[r, :] = epilogue(a[r, :] W^T (+ bias)) for r < M (any M; a: bf16 rows of stride lda,
// W: bf16 [N, K] with K % 8 == 0; epi as for the GEMMs: bf16 out, bf16 GELU out, fp32 +=, fp32 out).
cudaError_t launch_gemv(const void* a, int lda, const void* W, const float* bias, void* out, int ldo, int M, int N,
                        int K, int epi, int gelu_erf, cudaStream_t s);
// The new tokens' attention at position pos = *pos_dev (0 <= pos < ctx, checked by the caller):
// stores each one's key and value (from qkv [B, 3C]) in the layer's cache [batch][ctx][2C] at pos,
// then y[b] = softmax over keys 0..pos.
cudaError_t launch_attention_decode(const void* qkv, void* cache_layer, void* y, int B, int H, int D, int ctx,
                                    const int* pos_dev, cudaStream_t s);
// *p = v (the decode position, written on the stream before a captured decode step runs).
cudaError_t launch_set_int(int* p, int v, cudaStream_t s);
// Next-token draw per row of logits [B, V] fp32 (temperature <= 0: greedy; top_k / top_p
// filters; uniform[b] in [0, 1)); V <= kSampleMaxV (the row's probabilities sit in shared memory).
constexpr int kSampleMaxV = 55296;
cudaError_t launch_sample(const float* logits, int B, int V, float temperature, int top_k, float top_p,
                          const float* uniform, int32_t* out, cudaStream_t s);
// cache[b][t][0:2C] = qkv[b, t][C:3C] for a prompt of T tokens.
cudaError_t launch_kv_store(const void* qkv, void* cache_layer, int B, int T, int C, int ctx, cudaStream_t s);

}  // namespace gptgb
