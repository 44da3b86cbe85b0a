// Kernels of the backward pass (bf16 path): layout changes, column sums, and the
// derivatives of LayerNorm, GELU, the embedding lookup and causal attention.
//
// The training step of "预训练一个 Mini GPT" (训练循环) back-propagates the mean
// next-token cross-entropy to every parameter; the projections' derivatives are
// GEMMs on the tcgen05 kernel (k_gemm_tc.cu), these kernels are the rest. The
// tied table collects both uses ("第 25 章 从小 GPT 到 GPT-2" §25.4).
#include "common.cuh"
#include "kernels.h"
#include "launch.h"

#include <cuda_bf16.h>
#include <math.h>

namespace gptgb {

namespace {

constexpr int kTr = 32;                      // transpose tile edge

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// dst[c][r] = src[r][c]: a 32 x 32 tile per block through shared memory (the padded
// row of 34 halves puts a column's 32 entries in 32 different banks).
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint16_t* __restrict__ src, int rows, int cols,
                                                             int lds, uint16_t* __restrict__ dst, int ldd) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint16_t t[kTr][kTr + 2];
  const int c0 = blockIdx.x * kTr, r0 = blockIdx.y * kTr;
  for (int i = threadIdx.y; i < kTr; i += 8) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    t[i][threadIdx.x] = (r < rows && c < cols) ? src[static_cast<size_t>(r) * lds + c] : uint16_t(0);
  }
  __syncthreads();
  for (int i = threadIdx.y; i < kTr; i += 8) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (c < cols && r < rows) dst[static_cast<size_t>(c) * ldd + r] = t[threadIdx.x][i];
  }
}

// fp32 [rows, cols] -> bf16 copy (dst, nullable) and bf16 transpose (dstT [cols, rows], nullable).
__global__ void __launch_bounds__(256) cast_transpose_kernel(const float* __restrict__ src, int rows, int cols,
                                                             uint16_t* __restrict__ dst, uint16_t* __restrict__ dstT,
                                                             int ldt) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint16_t t[kTr][kTr + 2];
  const int c0 = blockIdx.x * kTr, r0 = blockIdx.y * kTr;
  for (int i = threadIdx.y; i < kTr; i += 8) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    uint16_t h = 0;
    if (r < rows && c < cols) {
      h = f2bf(src[static_cast<size_t>(r) * cols + c]);
      if (dst) dst[static_cast<size_t>(r) * cols + c] = h;
    }
    t[i][threadIdx.x] = h;
  }
  __syncthreads();
  if (dstT == nullptr) return;                // a plain cast (block-uniform)
  for (int i = threadIdx.y; i < kTr; i += 8) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (c < cols && r < rows) dstT[static_cast<size_t>(c) * ldt + r] = t[threadIdx.x][i];
  }
}

// out[c] += sum over rows of src[r][c]: a block sums 32 columns over a range of rows
// (8 row lanes), then adds its partial with one atomic per column.
template <bool BF16>
__global__ void __launch_bounds__(256) colsum_kernel(const void* __restrict__ src, int rows, int cols, int lds,
                                                     float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  __shared__ float part[8][33];
  const int c = blockIdx.x * 32 + threadIdx.x;
  const int per = (rows + gridDim.y - 1) / gridDim.y;
  const int rb = blockIdx.y * per, re = min(rows, rb + per);
  float s = 0.0f;
  if (c < cols) {
    for (int r = rb + threadIdx.y; r < re; r += 8) {
      const size_t i = static_cast<size_t>(r) * lds + c;
      s += BF16 ? bf2f(static_cast<const uint16_t*>(src)[i]) : static_cast<const float*>(src)[i];
    }
  }
  part[threadIdx.y][threadIdx.x] = s;
  __syncthreads();
  if (threadIdx.y == 0 && c < cols) {
    float t = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += part[i][threadIdx.x];
    atomicAdd(out + c, t);
  }
}

// LayerNorm derivative, one warp per row ("预训练一个 Mini GPT" 第4步 defines the forward:
// xh = (x - mean) r, r = 1 / sqrt(var + eps), y = g xh + b). With dxh = dy g:
// dx = r (dxh - mean(dxh) - xh mean(dxh xh)); dg = sum over rows of dy xh; db = sum of dy.
// dx_io = dx (add = 0) or dx_io + dx (add = 1: the residual path's gradient joins here).
// dg and db: per-block partials in shared memory, then one atomic per column and block.
__global__ void __launch_bounds__(256) layernorm_bwd_kernel(const float* __restrict__ x, const float* __restrict__ g,
                                                            const float* dy, float* dx_io,
                                                            int add, float* __restrict__ dg, float* __restrict__ db,
                                                            int M, int C, float eps) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float sh[];                       // [2][C]: dg and db partials
  float* sg = sh;
  float* sb = sh + C;
  for (int i = threadIdx.x; i < 2 * C; i += blockDim.x) sh[i] = 0.0f;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, wpb = blockDim.x >> 5;
  const float invC = 1.0f / static_cast<float>(C);
  for (int row = blockIdx.x * wpb + warp; row < M; row += gridDim.x * wpb) {
    const float* xr = x + static_cast<size_t>(row) * C;
    const float* dr = dy + static_cast<size_t>(row) * C;
    float s = 0.0f;
    for (int c = lane; c < C; c += 32) s += xr[c];
    const float mean = warp_sum(s) * invC;
    float v = 0.0f;
    for (int c = lane; c < C; c += 32) {
      const float d = xr[c] - mean;
      v += d * d;
    }
    const float r = rsqrtf(warp_sum(v) * invC + eps);
    float s1 = 0.0f, s2 = 0.0f;
    for (int c = lane; c < C; c += 32) {
      const float xh = (xr[c] - mean) * r;
      const float d = dr[c];
      const float dxh = d * g[c];
      s1 += dxh;
      s2 += dxh * xh;
      atomicAdd(sg + c, d * xh);
      atomicAdd(sb + c, d);
    }
    const float m1 = warp_sum(s1) * invC, m2 = warp_sum(s2) * invC;
    float* o = dx_io + static_cast<size_t>(row) * C;
    for (int c = lane; c < C; c += 32) {
      const float xh = (xr[c] - mean) * r;
      const float val = r * (dr[c] * g[c] - m1 - xh * m2);
      o[c] = add ? o[c] + val : val;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < C; i += blockDim.x) {
    atomicAdd(dg + i, sg[i]);
    atomicAdd(db + i, sb[i]);
  }
}

// du = dg * gelu'(u), elementwise over bf16 (du may alias dg). tanh form ("GPT-1 学习笔记" §3.6):
// gelu = 0.5 u (1 + tanh s), s = c (u + 0.044715 u^3), c = sqrt(2/pi), so
// gelu' = 0.5 (1 + tanh s) + 0.5 u (1 - tanh^2 s) c (1 + 3 * 0.044715 u^2);
// erf form gelu = u Phi(u): gelu' = Phi(u) + u phi(u).
__global__ void __launch_bounds__(256) gelu_bwd_kernel(const uint4* __restrict__ u, const uint4* dg, uint4* du,
                                                       size_t n8, int erf_form) {
  pdl_wait();
  pdl_trigger();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint4 uu = u[i], gg = dg[i];
    const uint32_t uw[4] = {uu.x, uu.y, uu.z, uu.w};
    const uint32_t gw[4] = {gg.x, gg.y, gg.z, gg.w};
    uint32_t ow[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 uv = unpack_bf16x2(uw[q]);
      const float2 gv = unpack_bf16x2(gw[q]);
      float d[2];
      const float xs[2] = {uv.x, uv.y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float xv = xs[e];
        if (erf_form) {
          d[e] = 0.5f * (1.0f + erff(xv * 0.70710678118654752f)) + xv * 0.39894228040143268f * expf(-0.5f * xv * xv);
        } else {
          constexpr float c0 = 0.7978845608028654f;
          const float t = tanhf(c0 * (xv + 0.044715f * xv * xv * xv));
          d[e] = 0.5f * (1.0f + t) + 0.5f * xv * (1.0f - t * t) * c0 * (1.0f + 3.0f * 0.044715f * xv * xv);
        }
      }
      ow[q] = pack_bf16x2(gv.x * d[0], gv.y * d[1]);
    }
    du[i] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
  }
}

// x0[m] = E[id[m]] + P[m % T]: dE[id[m]] += dx0[m], dP[m % T] += dx0[m] (atomics; one warp per row).
__global__ void __launch_bounds__(256) embed_bwd_kernel(const float* __restrict__ dx0, const int32_t* __restrict__ ids,
                                                        float* __restrict__ dE, float* __restrict__ dP, int M, int T,
                                                        int C, int V) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= M) return;
  const int id = ids[row];
  const float* d = dx0 + static_cast<size_t>(row) * C;
  float* e = (id >= 0 && id < V) ? dE + static_cast<size_t>(id) * C : nullptr;
  float* p = dP + static_cast<size_t>(row % T) * C;
  for (int c = lane; c < C; c += 32) {
    const float v = d[c];
    if (e) atomicAdd(e + c, v);
    atomicAdd(p + c, v);
  }
}

}  // namespace

cudaError_t launch_transpose_bf16(const void* src, int rows, int cols, int lds, void* dst, int ldd, cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const dim3 grid((cols + kTr - 1) / kTr, (rows + kTr - 1) / kTr), block(kTr, 8);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  return launch_k(transpose_bf16_kernel, grid, block, 0, s, static_cast<const uint16_t*>(src), rows, cols, lds,
                  static_cast<uint16_t*>(dst), ldd);
}

cudaError_t launch_cast_transpose(const float* src, int rows, int cols, void* dst, void* dstT, int ldt, cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const dim3 grid((cols + kTr - 1) / kTr, (rows + kTr - 1) / kTr), block(kTr, 8);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  return launch_k(cast_transpose_kernel, grid, block, 0, s, src, rows, cols, static_cast<uint16_t*>(dst),
                  static_cast<uint16_t*>(dstT), ldt);
}

cudaError_t launch_colsum(const void* src, int bf16, int rows, int cols, int lds, float* out, int num_sms,
                          cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const int gx = (cols + 31) / 32;
  int gy = (4 * num_sms + gx - 1) / gx;
  gy = gy < 1 ? 1 : gy;
  const int max_gy = (rows + 63) / 64;
  gy = gy > max_gy ? max_gy : gy;
  const dim3 grid(gx, gy), block(32, 8);
  return bf16 ? launch_k(colsum_kernel<true>, grid, block, 0, s, src, rows, cols, lds, out)
              : launch_k(colsum_kernel<false>, grid, block, 0, s, src, rows, cols, lds, out);
}

cudaError_t launch_layernorm_bwd(const float* x, const float* g, const float* dy, float* dx_io, int add, float* dg,
                                 float* db, int M, int C, float eps, int num_sms, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  const int wpb = 8;
  int grid = (M + wpb - 1) / wpb;
  if (grid > 2 * num_sms) grid = 2 * num_sms;
  const size_t smem = 2 * static_cast<size_t>(C) * sizeof(float);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  return launch_k(layernorm_bwd_kernel, dim3(grid), dim3(wpb * 32), smem, s, x, g, dy, dx_io, add, dg, db, M, C, eps);
}

cudaError_t launch_gelu_bwd(const void* u, const void* dg, void* du, size_t n, int erf_form, int num_sms,
                            cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (n % 8) return cudaErrorInvalidValue;
  const size_t n8 = n / 8;
  size_t grid = (n8 + 255) / 256;
  if (grid > static_cast<size_t>(8 * num_sms)) grid = 8 * num_sms;
  return launch_k(gelu_bwd_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0, s, static_cast<const uint4*>(u),
                  static_cast<const uint4*>(dg), static_cast<uint4*>(du), n8, erf_form);
}

cudaError_t launch_embed_bwd(const float* dx0, const int32_t* ids, float* dE, float* dP, int M, int T, int C, int V,
                             cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  return launch_k(embed_bwd_kernel, dim3((M + 7) / 8), dim3(256), 0, s, dx0, ids, dE, dP, M, T, C, V);
}

}  // namespace gptgb
