// fp32 SIMT kernels: the exact-precision mode of the library (dtype 0).
//
// The same steps as the bf16 tensor-core path, in fp32 FMA arithmetic with no
// operand rounding: used where the fp32 tolerance (logits within 1e-3, loss
// within 1e-4 of the fp64 definition) is asked for, and for models whose
// shapes the tensor-core path does not take. Not tuned for speed.
#include "common.cuh"
#include "kernels.h"

#include <math.h>

namespace gptgb {

namespace {

constexpr int TM = 64, TN = 64, TK = 16;

__device__ __forceinline__ float gelu_exact_f(float x, int erf_form) {
  if (erf_form) return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
  return 0.5f * x * (1.0f + tanhf(0.7978845608028654f * (x + 0.044715f * x * x * x)));
}

// out[M,N] = epi(A[M,K] . W[N,K]^T + bias): 64x64 tiles, 256 threads, 4x4 per thread.
__global__ void __launch_bounds__(256)
gemm_simt_kernel(const float* __restrict__ A, const float* __restrict__ W, const float* __restrict__ bias,
                 float* __restrict__ out, int M, int N, int K, int ldo, int epi, int gelu_erf) {
  __shared__ float sa[TK][TM + 4];
  __shared__ float sw[TK][TN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += TK) {
    for (int i = threadIdx.x; i < TM * TK; i += 256) {
      const int r = i / TK, c = i % TK;
      const int gm = m0 + r, gk = k0 + c;
      sa[c][r] = (gm < M && gk < K) ? A[(size_t)gm * K + gk] : 0.0f;
      const int gn = n0 + r;
      sw[c][r] = (gn < N && gk < K) ? W[(size_t)gn * K + gk] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = sa[kk][ty * 4 + i]; w[i] = sw[kk][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= N) continue;
      float v = acc[i][j] + (bias ? bias[gn] : 0.0f);
      float* o = out + (size_t)gm * ldo + gn;
      if (epi == EPI_BIAS_GELU_OUT) v = gelu_exact_f(v, gelu_erf);
      if (epi == EPI_BIAS_RESID) *o += v;
      else *o = v;
    }
  }
}

// One warp per (b, h, t): scores of the allowed keys s <= t in shared memory,
// max-subtracted softmax, then the weighted sum of U with lanes over D.
constexpr int kAttnWarps = 4;

__global__ void __launch_bounds__(kAttnWarps * 32)
attention_simt_kernel(const float* __restrict__ qkv, float* __restrict__ y, int B, int T, int H, int D,
                      float scale) {
  extern __shared__ float sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * kAttnWarps + warp;     // (b, h, t)
  if (item >= (long long)B * H * T) return;
  const int t = static_cast<int>(item % T);
  const int h = static_cast<int>((item / T) % H);
  const int b = static_cast<int>(item / ((long long)T * H));
  const int C = H * D;
  float* q = sm + warp * (D + T);
  float* p = q + D;
  const float* base = qkv + (size_t)b * T * 3 * C;
  for (int d = lane; d < D; d += 32) q[d] = base[(size_t)t * 3 * C + h * D + d];
  __syncwarp();
  float mx = -INFINITY;
  for (int s = lane; s <= t; s += 32) {
    const float* k = base + (size_t)s * 3 * C + C + h * D;
    float acc = 0.0f;
    for (int d = 0; d < D; ++d) acc = fmaf(q[d], k[d], acc);
    acc *= scale;
    p[s] = acc;
    mx = fmaxf(mx, acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float sum = 0.0f;
  for (int s = lane; s <= t; s += 32) {
    const float e = expf(p[s] - mx);
    p[s] = e;
    sum += e;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  __syncwarp();
  const float inv = 1.0f / sum;
  for (int d = lane; d < D; d += 32) {
    float acc = 0.0f;
    for (int s = 0; s <= t; ++s) acc = fmaf(p[s], base[(size_t)s * 3 * C + 2 * C + h * D + d], acc);
    y[((size_t)b * T + t) * C + h * D + d] = acc * inv;
  }
}

// Per-row cross-entropy from materialised logits, one warp per row.
__global__ void __launch_bounds__(256)
ce_rows_kernel(const float* __restrict__ logits, const int32_t* __restrict__ targets, float* __restrict__ nll,
               int M, int V, int* err) {
  const int row = (blockIdx.x * 256 + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  const int tg = targets[row];
  if (tg < 0 || tg >= V) {
    if (lane == 0) { record_error(err, GPT_DEV_ETARGET); nll[row] = 0.0f; }
    return;
  }
  const float* z = logits + (size_t)row * V;
  float mx = -INFINITY;
  for (int j = lane; j < V; j += 32) mx = fmaxf(mx, z[j]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  float s = 0.0f;
  for (int j = lane; j < V; j += 32) s += expf(z[j] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) nll[row] = mx + logf(s) - z[tg];
}

}  // namespace

cudaError_t launch_gemm_simt(const float* A, const float* W, const float* bias, float* out, int M, int N, int K,
                             int ldo, int epi, int gelu_erf, cudaStream_t s) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((N + TN - 1) / TN, (M + TM - 1) / TM);
  if (grid.y > 65535) return cudaErrorInvalidValue;
  gemm_simt_kernel<<<grid, 256, 0, s>>>(A, W, bias, out, M, N, K, ldo, epi, gelu_erf);
  return cudaGetLastError();
}

cudaError_t launch_attention_simt(const float* qkv, float* y, int B, int T, int H, int D, cudaStream_t s) {
  const long long items = (long long)B * H * T;
  if (items <= 0) return cudaSuccess;
  const long long blocks = (items + kAttnWarps - 1) / kAttnWarps;
  const size_t smem = (size_t)kAttnWarps * (D + T) * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(attention_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  attention_simt_kernel<<<static_cast<unsigned>(blocks), kAttnWarps * 32, smem, s>>>(
      qkv, y, B, T, H, D, 1.0f / sqrtf(static_cast<float>(D)));
  return cudaGetLastError();
}

cudaError_t launch_ce_rows(const float* logits, const int32_t* targets, float* nll, int M, int V, int* err,
                           cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  ce_rows_kernel<<<(M + 7) / 8, 256, 0, s>>>(logits, targets, nll, M, V, err);
  return cudaGetLastError();
}

}  // namespace gptgb
