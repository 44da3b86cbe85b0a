// Incremental decoding with a key/value cache ("预训练一个 Mini GPT", the
// sections on the KV cache and on the prefill and decode phases; "第 25 章"
// §25.2 for the attention it computes):
// one new token per sequence, whose query attends to every cached key of its
// sequence plus its own.
//
// Decode is bound by memory traffic, not by tensor-core throughput: each step
// reads every weight once and each sequence's cached keys and values once,
// while the rows (B new tokens) are few. So the projections here are
// matrix-vector products on the SIMT units (one warp per output column,
// 16-byte coalesced weight loads, fp32 accumulation) rather than 128-row
// tensor-core tiles that would be almost empty, and the attention is a
// per-(sequence, head) reduction over the cache.
//
// Cache layout (bf16): per layer [batch][ctx][2C]: row (b, t) holds the key
// (columns [0, C)) and the value (columns [C, 2C)) of token t of sequence b,
// heads as column offsets h*D, exactly the K and U thirds of that token's qkv row.
#include "common.cuh"
#include "kernels.h"
#include "launch.h"

#include <math.h>

namespace gptgb {

namespace {

constexpr int kGemvWarps = 8;                 // output columns per block
constexpr int kAttnDecThreads = 128;

__device__ __forceinline__ void unpack8(const uint4 u, float (&f)[8]) {
  float2 t;
  t = unpack_bf16x2(u.x); f[0] = t.x; f[1] = t.y;
  t = unpack_bf16x2(u.y); f[2] = t.x; f[3] = t.y;
  t = unpack_bf16x2(u.z); f[4] = t.x; f[5] = t.y;
  t = unpack_bf16x2(u.w); f[6] = t.x; f[7] = t.y;
}

// Weights are read once per step: a streaming load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ float gelu_dec(float x, int erf_form) {
  if (erf_form) return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
  constexpr float c0 = 0.7978845608028654f;             // sqrt(2/pi)
  constexpr float c1 = 0.7978845608028654f * 0.044715f;
  const float u = x * fmaf(x * x, c1, c0);
  const float h = 0.5f * x;
  return fmaf(h, tanh_approx(u), h);
}

// out[r, n] = epilogue(sum_k a[r, k] W[n, k] (+ bias[n])) for rows r < M <= MR.
// SPLIT warps share a column n: the 16-byte chunks c of W's row n (K / 8 of
// them) are dealt c = part * 32 + lane + i * 32 * SPLIT, so every warp load
// covers 512 contiguous bytes, and up to four loads per lane are in flight
// before the arithmetic. The rows of a are L1-resident (all warps of the grid
// read the same few rows). The SPLIT partial sums meet in shared memory in a
// fixed order. K % 8 == 0.
template <int EPI, int MR, int SPLIT>
__global__ void __launch_bounds__(kGemvWarps * 32)
gemv_kernel(const __nv_bfloat16* __restrict__ a, int lda, const __nv_bfloat16* __restrict__ W,
            const float* __restrict__ bias, void* out, int ldo, int M, int N, int K, int gelu_erf) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[kGemvWarps][MR];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int part = warp % SPLIT;
  const int n = blockIdx.x * (kGemvWarps / SPLIT) + warp / SPLIT;
  const bool live = n < N;                                   // the block's barrier below needs every warp
  const __nv_bfloat16* wr = W + (size_t)(live ? n : 0) * K;
  const int chunks = K / 8;
  float acc[MR];
#pragma unroll
  for (int r = 0; r < MR; ++r) acc[r] = 0.0f;
  constexpr int U = 4;                                       // loads in flight per lane
  for (int c0 = part * 32 + lane; live && c0 < chunks; c0 += U * 32 * SPLIT) {
    uint4 wv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 32 * SPLIT;
      wv[u] = c < chunks ? ld_stream_u4(wr + 8 * c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 32 * SPLIT;
      if (c >= chunks) break;
      float wf[8];
      unpack8(wv[u], wf);
#pragma unroll
      for (int r = 0; r < MR; ++r) {
        if (r < M) {
          float af[8];
          unpack8(*reinterpret_cast<const uint4*>(a + (size_t)r * lda + 8 * c), af);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[r] = fmaf(af[i], wf[i], acc[r]);
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < MR; ++r) {
    float v = acc[r];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    acc[r] = v;
  }
  if (SPLIT > 1) {
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < MR; ++r) red[warp][r] = acc[r];
    }
    __syncthreads();
    if (part != 0) return;
#pragma unroll
    for (int r = 0; r < MR; ++r) {
      float v = 0.0f;
#pragma unroll
      for (int q = 0; q < SPLIT; ++q) v += red[warp + q][r];
      acc[r] = v;
    }
  }
  if (!live) return;
  float mine = 0.0f;                                         // lane r keeps row r's total
#pragma unroll
  for (int r = 0; r < MR; ++r)
    if (lane == r) mine = acc[r];
  if (lane >= M) return;
  const int r = lane;
  if (bias != nullptr) mine += __ldg(bias + n);
  if (EPI == EPI_BIAS_OUT) {
    reinterpret_cast<__nv_bfloat16*>(out)[(size_t)r * ldo + n] = __float2bfloat16_rn(mine);
  } else if (EPI == EPI_BIAS_GELU_OUT) {
    reinterpret_cast<__nv_bfloat16*>(out)[(size_t)r * ldo + n] = __float2bfloat16_rn(gelu_dec(mine, gelu_erf));
  } else if (EPI == EPI_BIAS_RESID) {
    reinterpret_cast<float*>(out)[(size_t)r * ldo + n] += mine;     // one writer per element
  } else {
    reinterpret_cast<float*>(out)[(size_t)r * ldo + n] = mine;
  }
}

// One (sequence b, head h) per block. The new token's key and value (from its
// qkv row) are first stored in the cache at position pos; then every thread
// takes keys j = tid, tid + 128, ... <= pos with its own running (max, sum,
// output) in base 2, and the block merges the 128 partial results.
template <int D>
__global__ void __launch_bounds__(kAttnDecThreads)
attn_decode_kernel(const __nv_bfloat16* __restrict__ qkv, __nv_bfloat16* cache, __nv_bfloat16* __restrict__ y,
                   int H, int C, int ctx, const int* __restrict__ pos_dev, float scale_log2) {
  pdl_wait();
  pdl_trigger();
  const int pos = *pos_dev;
  __shared__ float s_m[kAttnDecThreads];
  __shared__ float s_l[kAttnDecThreads];
  __shared__ float s_o[D][kAttnDecThreads + 1];
  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int tid = threadIdx.x;
  const __nv_bfloat16* qrow = qkv + (size_t)b * 3 * C;
  __nv_bfloat16* cb = cache + (size_t)b * ctx * 2 * C;             // this sequence's rows
  constexpr int V8 = D / 8;                                        // 16-byte chunks per head slice
  if (tid < 2 * V8) {                                              // key chunks, then value chunks
    const int part = tid / V8, c8 = tid % V8;
    const uint4 v = *reinterpret_cast<const uint4*>(qrow + (1 + part) * C + h * D + 8 * c8);
    *reinterpret_cast<uint4*>(cb + (size_t)pos * 2 * C + part * C + h * D + 8 * c8) = v;
  }
  __syncthreads();                                                 // the new row is visible to the block
  float q[D];
#pragma unroll
  for (int c8 = 0; c8 < V8; ++c8) {
    float f[8];
    unpack8(*reinterpret_cast<const uint4*>(qrow + h * D + 8 * c8), f);
#pragma unroll
    for (int i = 0; i < 8; ++i) q[8 * c8 + i] = f[i] * scale_log2;
  }
  float m = -INFINITY, l = 0.0f, o[D];
#pragma unroll
  for (int d = 0; d < D; ++d) o[d] = 0.0f;
  for (int j = tid; j <= pos; j += kAttnDecThreads) {
    const __nv_bfloat16* kr = cb + (size_t)j * 2 * C + h * D;
    float sc = 0.0f;
#pragma unroll
    for (int c8 = 0; c8 < V8; ++c8) {
      float f[8];
      unpack8(*reinterpret_cast<const uint4*>(kr + 8 * c8), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) sc = fmaf(q[8 * c8 + i], f[i], sc);
    }
    if (sc > m) {                                                  // raise the running max
      const float alpha = ex2_approx(m - sc);                      // 0 for the first key
      l *= alpha;
#pragma unroll
      for (int d = 0; d < D; ++d) o[d] *= alpha;
      m = sc;
    }
    const float p = ex2_approx(sc - m);
    l += p;
    const __nv_bfloat16* vr = kr + C;
#pragma unroll
    for (int c8 = 0; c8 < V8; ++c8) {
      float f[8];
      unpack8(*reinterpret_cast<const uint4*>(vr + 8 * c8), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[8 * c8 + i] = fmaf(p, f[i], o[8 * c8 + i]);
    }
  }
  s_m[tid] = m;
  __syncthreads();
  float gm = -INFINITY;                                            // key 0 is always present: finite
  for (int t = 0; t < kAttnDecThreads; ++t) gm = fmaxf(gm, s_m[t]);
  const float w = (m == -INFINITY) ? 0.0f : ex2_approx(m - gm);  // threads without keys add nothing
  s_l[tid] = l * w;
#pragma unroll
  for (int d = 0; d < D; ++d) s_o[d][tid] = o[d] * w;
  __syncthreads();
  if (tid < D) {
    float num = 0.0f, den = 0.0f;
    for (int t = 0; t < kAttnDecThreads; ++t) {                    // fixed order: deterministic
      num += s_o[tid][t];
      den += s_l[t];
    }
    y[(size_t)b * C + h * D + tid] = __float2bfloat16_rn(num / den);
  }
}

// cache[b][t][0:2C] = qkv[b, t][C:3C] for the T prompt tokens (16-byte chunks).
__global__ void __launch_bounds__(256)
kv_store_kernel(const __nv_bfloat16* __restrict__ qkv, __nv_bfloat16* __restrict__ cache, int B, int T, int C,
                int ctx) {
  pdl_wait();
  pdl_trigger();
  const int c8n = 2 * C / 8;                                       // chunks per token
  const long long total = (long long)B * T * c8n;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c8 = static_cast<int>(i % c8n);
    const long long row = i / c8n;                                 // b * T + t
    const int b = static_cast<int>(row / T), t = static_cast<int>(row % T);
    const uint4 v = *reinterpret_cast<const uint4*>(qkv + row * 3 * C + C + 8 * c8);
    *reinterpret_cast<uint4*>(cache + ((size_t)b * ctx + t) * 2 * C + 8 * c8) = v;
  }
}

__global__ void set_int_kernel(int* p, int v) { *p = v; }

template <int EPI, int SPLIT>
cudaError_t gemv_rows(const __nv_bfloat16* a, int lda, const __nv_bfloat16* W, const float* bias, void* out,
                      int ldo, int M, int N, int K, int gelu_erf, cudaStream_t s) {
  const dim3 grid((N + kGemvWarps / SPLIT - 1) / (kGemvWarps / SPLIT)), block(kGemvWarps * 32);
#define GPT_GEMV(MRV) \
  return launch_k(gemv_kernel<EPI, MRV, SPLIT>, grid, block, 0, s, a, lda, W, bias, out, ldo, M, N, K, gelu_erf)
  if (M <= 1) GPT_GEMV(1);
  if (M <= 2) GPT_GEMV(2);
  if (M <= 4) GPT_GEMV(4);
  if (M <= 8) GPT_GEMV(8);
  GPT_GEMV(16);
#undef GPT_GEMV
}

// Warps per column: enough warps in the grid (about 2048) to keep loads in flight on
// every SM when N is small, but not more than the 512-byte rows of a weight row.
template <int EPI>
cudaError_t gemv_dispatch(const __nv_bfloat16* a, int lda, const __nv_bfloat16* W, const float* bias, void* out,
                          int ldo, int M, int N, int K, int gelu_erf, cudaStream_t s) {
  const int rows512 = (K / 8 + 31) / 32;
  int split = 1;
  while (split < 8 && N * split < 2048 && split * 2 <= rows512) split *= 2;
  switch (split) {
    case 1: return gemv_rows<EPI, 1>(a, lda, W, bias, out, ldo, M, N, K, gelu_erf, s);
    case 2: return gemv_rows<EPI, 2>(a, lda, W, bias, out, ldo, M, N, K, gelu_erf, s);
    case 4: return gemv_rows<EPI, 4>(a, lda, W, bias, out, ldo, M, N, K, gelu_erf, s);
    default: return gemv_rows<EPI, 8>(a, lda, W, bias, out, ldo, M, N, K, gelu_erf, s);
  }
}

}  // namespace

cudaError_t launch_gemv(const void* a, int lda, const void* W, const float* bias, void* out, int ldo, int M, int N,
                        int K, int epi, int gelu_erf, cudaStream_t s) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (K <= 0 || (K % 8) || (lda % 8)) return cudaErrorInvalidValue;
  const auto* A = reinterpret_cast<const __nv_bfloat16*>(a);
  const auto* Wb = reinterpret_cast<const __nv_bfloat16*>(W);
  for (int r0 = 0; r0 < M; r0 += kGemvMaxRows) {               // 16 rows per launch
    const int mr = (M - r0 < kGemvMaxRows) ? M - r0 : kGemvMaxRows;
    const __nv_bfloat16* ar = A + (size_t)r0 * lda;
    void* orow = (epi == EPI_BIAS_OUT || epi == EPI_BIAS_GELU_OUT)
                     ? static_cast<void*>(reinterpret_cast<__nv_bfloat16*>(out) + (size_t)r0 * ldo)
                     : static_cast<void*>(reinterpret_cast<float*>(out) + (size_t)r0 * ldo);
    cudaError_t e;
    switch (epi) {
      case EPI_BIAS_OUT: e = gemv_dispatch<EPI_BIAS_OUT>(ar, lda, Wb, bias, orow, ldo, mr, N, K, gelu_erf, s); break;
      case EPI_BIAS_GELU_OUT:
        e = gemv_dispatch<EPI_BIAS_GELU_OUT>(ar, lda, Wb, bias, orow, ldo, mr, N, K, gelu_erf, s);
        break;
      case EPI_BIAS_RESID: e = gemv_dispatch<EPI_BIAS_RESID>(ar, lda, Wb, bias, orow, ldo, mr, N, K, gelu_erf, s); break;
      case EPI_F32: e = gemv_dispatch<EPI_F32>(ar, lda, Wb, bias, orow, ldo, mr, N, K, gelu_erf, s); break;
      default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_attention_decode(const void* qkv, void* cache_layer, void* y, int B, int H, int D, int ctx,
                                    const int* pos_dev, cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  if (pos_dev == nullptr) return cudaErrorInvalidValue;
  const int C = H * D;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(D));
  const auto* q = reinterpret_cast<const __nv_bfloat16*>(qkv);
  auto* c = reinterpret_cast<__nv_bfloat16*>(cache_layer);
  auto* yo = reinterpret_cast<__nv_bfloat16*>(y);
  if (D == 64)
    return launch_k(attn_decode_kernel<64>, dim3(B * H), dim3(kAttnDecThreads), 0, s, q, c, yo, H, C, ctx, pos_dev,
                    scale_log2);
  if (D == 32)
    return launch_k(attn_decode_kernel<32>, dim3(B * H), dim3(kAttnDecThreads), 0, s, q, c, yo, H, C, ctx, pos_dev,
                    scale_log2);
  return cudaErrorInvalidValue;
}

cudaError_t launch_set_int(int* p, int v, cudaStream_t s) {
  set_int_kernel<<<1, 1, 0, s>>>(p, v);
  return cudaGetLastError();
}

cudaError_t launch_kv_store(const void* qkv, void* cache_layer, int B, int T, int C, int ctx, cudaStream_t s) {
  if (B <= 0 || T <= 0) return cudaSuccess;
  const long long chunks = (long long)B * T * (2 * C / 8);
  long long blocks = (chunks + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  return launch_k(kv_store_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                  reinterpret_cast<const __nv_bfloat16*>(qkv), reinterpret_cast<__nv_bfloat16*>(cache_layer), B, T,
                  C, ctx);
}

}  // namespace gptgb
