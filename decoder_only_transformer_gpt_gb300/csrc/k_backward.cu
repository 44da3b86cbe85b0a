// Kernels of the backward pass (bf16 path): layout changes, column sums, and the
// derivatives of LayerNorm and the embedding lookup, and the optimiser step (the GELU and
// causal-attention derivatives live in k_gemm_tc.cu and k_attn_bwd.cu).
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


__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
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

// The same for bf16 rows with 16-byte loads: a thread sums 8 consecutive columns (one uint4 per row, four
// rows' loads in flight at a time, added in row order), a block covers 256 columns over its range of rows
// with 8 row lanes, then one atomic per column.
__global__ void __launch_bounds__(256) colsum8_bf16_kernel(const uint16_t* __restrict__ src, int rows, int cols,
                                                           int lds, float* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  __shared__ float part[8][256 + 4];
  const int c0 = blockIdx.x * 256 + threadIdx.x * 8;
  const int per = (rows + gridDim.y - 1) / gridDim.y;
  const int rb = blockIdx.y * per, re = min(rows, rb + per);
  float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
  auto add8 = [&](const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = unpack_bf16x2(w[k]);
      acc[2 * k] += f.x;
      acc[2 * k + 1] += f.y;
    }
  };
  if (c0 < cols) {
    int r = rb + threadIdx.y;
    for (; r + 24 < re; r += 32) {                  // four rows' loads in flight per thread
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = *reinterpret_cast<const uint4*>(src + static_cast<size_t>(r + 8 * i) * lds + c0);
#pragma unroll
      for (int i = 0; i < 4; ++i) add8(v[i]);
    }
    for (; r < re; r += 8) add8(*reinterpret_cast<const uint4*>(src + static_cast<size_t>(r) * lds + c0));
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) part[threadIdx.y][threadIdx.x * 8 + k] = acc[k];
  __syncthreads();
  const int t = threadIdx.y * 32 + threadIdx.x;           // 256 threads, one column each
  const int c = blockIdx.x * 256 + t;
  if (c < cols) {
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += part[i][t];
    atomicAdd(out + c, sum);
  }
}

// dst (bf16) = src (fp32), rows of `cols` values, and colsum[c] += the column sums (the bias gradient of the
// product that produced src): the shape of colsum8_bf16_kernel, a thread taking 8 consecutive columns of
// every 8th row of its block's range with four rows' loads in flight, so each warp access covers 1 KB of
// fp32 and 512 contiguous bytes of bf16. cols % 8 == 0, 16-byte aligned rows.
__global__ void __launch_bounds__(256) cast_colsum_kernel(const float* __restrict__ src, int rows, int cols,
                                                          uint16_t* __restrict__ dst, float* __restrict__ colsum) {
  pdl_wait();
  pdl_trigger();
  __shared__ float part[8][256 + 4];
  const int c0 = blockIdx.x * 256 + threadIdx.x * 8;
  const int per = (rows + gridDim.y - 1) / gridDim.y;
  const int rb = blockIdx.y * per, re = min(rows, rb + per);
  float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
  auto row8 = [&](int r, const float4 a, const float4 b) {
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    *reinterpret_cast<uint4*>(dst + static_cast<size_t>(r) * cols + c0) =
        make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
  };
  if (c0 < cols) {
    int r = rb + threadIdx.y;
    for (; r + 24 < re; r += 32) {
      float4 va[4], vb[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4* p = reinterpret_cast<const float4*>(src + static_cast<size_t>(r + 8 * i) * cols + c0);
        va[i] = p[0];
        vb[i] = p[1];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) row8(r + 8 * i, va[i], vb[i]);
    }
    for (; r < re; r += 8) {
      const float4* p = reinterpret_cast<const float4*>(src + static_cast<size_t>(r) * cols + c0);
      row8(r, p[0], p[1]);
    }
  }
  if (colsum == nullptr) return;                           // block-uniform
#pragma unroll
  for (int k = 0; k < 8; ++k) part[threadIdx.y][threadIdx.x * 8 + k] = acc[k];
  __syncthreads();
  const int t = threadIdx.y * 32 + threadIdx.x;
  const int c = blockIdx.x * 256 + t;
  if (c < cols) {
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += part[i][t];
    atomicAdd(colsum + c, sum);
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

// 64 x 64 tiles with 16-byte global accesses. Load: 8 threads per 128-byte row segment into a
// shared tile (row stride 72 halves keeps 16-byte alignment); store: consecutive threads take
// consecutive output rows (tile columns), so the column gathers from shared memory hit 16
// different banks per warp, and each thread writes 8 consecutive outputs (16 bytes).
// SRC_F32: the source is fp32 [rows, cols] (dense), converted to bf16, also copied to dst_copy.
constexpr int kT64 = 64, kT64S = 72;

// colsum (nullable): out[c] += the tile's column sums (of the fp32 values for an fp32 source).
template <bool SRC_F32>
__global__ void __launch_bounds__(256) transpose64_kernel(const void* __restrict__ src, int rows, int cols, int lds,
                                                          uint16_t* __restrict__ dst_copy, uint16_t* __restrict__ dstT,
                                                          int ldt, int vec, float* __restrict__ colsum) {
  pdl_wait();
  pdl_trigger();
  __shared__ __align__(16) uint16_t t[kT64][kT64S];
  __shared__ float csum[kT64];
  const int c0 = blockIdx.x * kT64, r0 = blockIdx.y * kT64;
  if (colsum) {
    if (threadIdx.x < kT64) csum[threadIdx.x] = 0.0f;
    __syncthreads();
  }
  float part[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
  for (int i = threadIdx.x; i < kT64 * 8; i += 256) {
    const int r = i >> 3, ch = i & 7;
    const int gr = r0 + r, gc = c0 + ch * 8;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (gr < rows) {
      if (SRC_F32) {
        const float* sp = static_cast<const float*>(src) + static_cast<size_t>(gr) * lds + gc;
        float f[8];
        if (vec && gc + 8 <= cols) {
          const float4 a = *reinterpret_cast<const float4*>(sp), b = *reinterpret_cast<const float4*>(sp + 4);
          f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) f[k] = gc + k < cols ? sp[k] : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) part[k] += f[k];
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = pack_bf16x2(f[2 * k], f[2 * k + 1]);
        if (dst_copy) {
          uint16_t* dp = dst_copy + static_cast<size_t>(gr) * lds + gc;
          if (vec && gc + 8 <= cols) {
            *reinterpret_cast<uint4*>(dp) = make_uint4(w[0], w[1], w[2], w[3]);
          } else {
            for (int k = 0; k < 8 && gc + k < cols; ++k) dp[k] = static_cast<uint16_t>(w[k >> 1] >> (16 * (k & 1)));
          }
        }
      } else {
        const uint16_t* sp = static_cast<const uint16_t*>(src) + static_cast<size_t>(gr) * lds + gc;
        if (vec && gc + 8 <= cols) {
          const uint4 v = *reinterpret_cast<const uint4*>(sp);
          w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (gc + k < cols) w[k >> 1] |= static_cast<uint32_t>(sp[k]) << (16 * (k & 1));
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f2 = unpack_bf16x2(w[k]);
          part[2 * k] += f2.x;
          part[2 * k + 1] += f2.y;
        }
      }
    }
    *reinterpret_cast<uint4*>(&t[r][ch * 8]) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (colsum) {                  // a thread's columns are ch * 8 .. + 7, ch = lane & 7: fold lanes ch, +8, +16, +24
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float v = part[k];
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      if (lane < 8) atomicAdd(csum + lane * 8 + k, v);
    }
  }
  __syncthreads();
  if (colsum && threadIdx.x < kT64 && c0 + threadIdx.x < cols) atomicAdd(colsum + c0 + threadIdx.x, csum[threadIdx.x]);
  if (dstT == nullptr) return;                             // a cast (block-uniform)
  for (int i = threadIdx.x; i < kT64 * 8; i += 256) {
    const int cc = i & 63, ch = i >> 6;
    const int oc = c0 + cc, orow = r0 + ch * 8;          // output row oc, columns orow .. orow + 7
    if (oc >= cols || orow >= rows) continue;
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      w[k] = static_cast<uint32_t>(t[ch * 8 + 2 * k][cc]) | (static_cast<uint32_t>(t[ch * 8 + 2 * k + 1][cc]) << 16);
    uint16_t* dp = dstT + static_cast<size_t>(oc) * ldt + orow;
    if (vec && orow + 8 <= rows) {
      *reinterpret_cast<uint4*>(dp) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      for (int k = 0; k < 8 && orow + k < rows; ++k) dp[k] = static_cast<uint16_t>(w[k >> 1] >> (16 * (k & 1)));
    }
  }
}

// LayerNorm derivative with the row held in registers: C = 32 NPL, lane j-th column lane + 32 j
// (128-byte coalesced). The gain and its per-warp gain and shift gradient partials live in shared memory
// (each lane owns its columns, so no atomics within a warp), summed over the block's four warps and
// added once per block (global). Holding them in registers took 168 registers (12 resident warps per
// SM, latency-bound); this form takes 72 (28 warps). x and dy are read once.
template <int NPL>
__global__ void __launch_bounds__(128) layernorm_bwd_reg_kernel(const float* __restrict__ x, const float* __restrict__ g,
                                                                const float* dy, float* dx_io, int add,
                                                                float* __restrict__ dg, float* __restrict__ db, int M,
                                                                float eps) {
  pdl_wait();
  pdl_trigger();
  constexpr int C = 32 * NPL;
  constexpr int W = 4;
  __shared__ float sgam[C];
  __shared__ float wacc[W][2][C];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, wpb = blockDim.x >> 5;
  for (int i = threadIdx.x; i < C; i += blockDim.x) sgam[i] = g[i];
  for (int i = lane; i < C; i += 32) { wacc[warp][0][i] = 0.0f; wacc[warp][1][i] = 0.0f; }
  __syncthreads();
  constexpr float invC = 1.0f / static_cast<float>(C);
  for (int row = blockIdx.x * wpb + warp; row < M; row += gridDim.x * wpb) {
    const float* xr = x + static_cast<size_t>(row) * C;
    const float* dr = dy + static_cast<size_t>(row) * C;
    float xv[NPL], dv[NPL];
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      xv[j] = xr[lane + 32 * j];
      dv[j] = dr[lane + 32 * j];
      s += xv[j];
    }
    const float mean = warp_sum(s) * invC;
    float v = 0.0f;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      xv[j] -= mean;
      v += xv[j] * xv[j];
    }
    const float r = rsqrtf(warp_sum(v) * invC + eps);
    float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      xv[j] *= r;
      const float dxh = dv[j] * sgam[lane + 32 * j];
      s1 += dxh;
      s2 += dxh * xv[j];
      wacc[warp][0][lane + 32 * j] += dv[j] * xv[j];
      wacc[warp][1][lane + 32 * j] += dv[j];
    }
    const float m1 = warp_sum(s1) * invC, m2 = warp_sum(s2) * invC;
    float* o = dx_io + static_cast<size_t>(row) * C;
#pragma unroll
    for (int j = 0; j < NPL; ++j) {
      const float val = r * (dv[j] * sgam[lane + 32 * j] - m1 - xv[j] * m2);
      o[lane + 32 * j] = add ? o[lane + 32 * j] + val : val;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < C; i += blockDim.x) {
    float ag = 0.0f, ab = 0.0f;
#pragma unroll
    for (int w = 0; w < W; ++w) { ag += wacc[w][0][i]; ab += wacc[w][1][i]; }
    atomicAdd(dg + i, ag);
    atomicAdd(db + i, ab);
  }
}

// AdamW over every parameter: block row blockIdx.y is one parameter tensor (segment), whose values
// sit at [off, off + n) of the flat gradient / master / moment arrays and are written back to dst
// (bf16 or fp32). Decoupled decay for decay segments; bias corrections bc1 = 1 - b1^t, bc2 = 1 - b2^t.
__global__ void __launch_bounds__(256) adamw_kernel(const OptSeg* __restrict__ segs, const float* __restrict__ grad,
                                                    float* __restrict__ master, float* __restrict__ m1,
                                                    float* __restrict__ m2, float lr, float b1, float b2, float eps,
                                                    float wd, float bc1, float bc2) {
  pdl_wait();
  pdl_trigger();
  const OptSeg sg = segs[blockIdx.y];
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < sg.n; i += static_cast<long long>(gridDim.x) * 256) {
    const long long k = sg.off + i;
    const float g = grad[k];
    float p = master[k];
    if (sg.decay) p -= lr * wd * p;
    const float mm = b1 * m1[k] + (1.0f - b1) * g;
    const float vv = b2 * m2[k] + (1.0f - b2) * g * g;
    p -= lr * (mm / bc1) / (sqrtf(vv / bc2) + eps);
    master[k] = p;
    m1[k] = mm;
    m2[k] = vv;
    if (sg.bf16) static_cast<uint16_t*>(sg.dst)[i] = f2bf(p);
    else static_cast<float*>(sg.dst)[i] = p;
  }
}

// master[off + i] = the parameter's current value (bf16 or fp32 storage).
__global__ void __launch_bounds__(256) master_init_kernel(const OptSeg* __restrict__ segs, float* __restrict__ master) {
  pdl_wait();
  pdl_trigger();
  const OptSeg sg = segs[blockIdx.y];
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < sg.n; i += static_cast<long long>(gridDim.x) * 256)
    master[sg.off + i] = sg.bf16 ? bf2f(static_cast<const uint16_t*>(sg.dst)[i]) : static_cast<const float*>(sg.dst)[i];
}

}  // namespace

cudaError_t launch_adamw(const OptSeg* segs, int nseg, const float* grad, float* master, float* m1, float* m2, float lr,
                         float b1, float b2, float eps, float wd, float bc1, float bc2, cudaStream_t s) {
  if (nseg <= 0) return cudaSuccess;
  if (nseg > 65535) return cudaErrorInvalidValue;
  // 512 blocks per segment: the largest tensors (the token table) keep every SM streaming to the end
  return launch_k(adamw_kernel, dim3(512, nseg), dim3(256), 0, s, segs, grad, master, m1, m2, lr, b1, b2, eps, wd, bc1,
                  bc2);
}

cudaError_t launch_master_init(const OptSeg* segs, int nseg, float* master, cudaStream_t s) {
  if (nseg <= 0) return cudaSuccess;
  if (nseg > 65535) return cudaErrorInvalidValue;
  return launch_k(master_init_kernel, dim3(512, nseg), dim3(256), 0, s, segs, master);
}

cudaError_t launch_transpose_bf16(const void* src, int rows, int cols, int lds, void* dst, int ldd, cudaStream_t s,
                                  float* colsum) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const dim3 grid((cols + kT64 - 1) / kT64, (rows + kT64 - 1) / kT64);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  const int vec = (lds % 8 == 0) && (ldd % 8 == 0) && (reinterpret_cast<uintptr_t>(src) % 16 == 0) &&
                  (reinterpret_cast<uintptr_t>(dst) % 16 == 0);
  return launch_k(transpose64_kernel<false>, grid, dim3(256), 0, s, src, rows, cols, lds, static_cast<uint16_t*>(nullptr),
                  static_cast<uint16_t*>(dst), ldd, vec, colsum);
}

cudaError_t launch_cast_transpose(const float* src, int rows, int cols, void* dst, void* dstT, int ldt, cudaStream_t s,
                                  float* colsum) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  if (dstT == nullptr && dst != nullptr && cols % 8 == 0 && reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
      reinterpret_cast<uintptr_t>(dst) % 16 == 0) {          // a cast (+ column sums): the streaming kernel
    static int num_sms = 0;
    if (num_sms == 0) {
      int dev = 0;
      cudaError_t e = cudaGetDevice(&dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
    }
    const int gx = (cols + 255) / 256;
    int gy = (4 * num_sms + gx - 1) / gx;
    const int max_gy = (rows + 63) / 64;
    gy = gy > max_gy ? max_gy : (gy < 1 ? 1 : gy);
    return launch_k(cast_colsum_kernel, dim3(gx, gy), dim3(32, 8), 0, s, src, rows, cols, static_cast<uint16_t*>(dst),
                    colsum);
  }
  const dim3 grid((cols + kT64 - 1) / kT64, (rows + kT64 - 1) / kT64);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  const int vec = (cols % 8 == 0) && (dstT == nullptr || ldt % 8 == 0) && (reinterpret_cast<uintptr_t>(src) % 16 == 0) &&
                  (reinterpret_cast<uintptr_t>(dst) % 16 == 0) && (reinterpret_cast<uintptr_t>(dstT) % 16 == 0);
  return launch_k(transpose64_kernel<true>, grid, dim3(256), 0, s, static_cast<const void*>(src), rows, cols, cols,
                  static_cast<uint16_t*>(dst), static_cast<uint16_t*>(dstT), ldt, vec, colsum);
}

cudaError_t launch_colsum(const void* src, int bf16, int rows, int cols, int lds, float* out, int num_sms,
                          cudaStream_t s) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  if (bf16 && cols % 8 == 0 && lds % 8 == 0 && reinterpret_cast<uintptr_t>(src) % 16 == 0) {
    const int gx8 = (cols + 255) / 256;
    int gy8 = (8 * num_sms + gx8 - 1) / gx8;
    const int max_gy8 = (rows + 63) / 64;
    gy8 = gy8 > max_gy8 ? max_gy8 : (gy8 < 1 ? 1 : gy8);
    return launch_k(colsum8_bf16_kernel, dim3(gx8, gy8), dim3(32, 8), 0, s, static_cast<const uint16_t*>(src), rows,
                    cols, lds, out);
  }
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
  int wpb = 4;                                  // 128-thread blocks (the kernel assumes four warps)
  int grid = (M + wpb - 1) / wpb;
  if (grid > 8 * num_sms) grid = 8 * num_sms;
#define GPT_LNB(NPL)                                                                                          \
  if (C == 32 * NPL)                                                                                          \
    return launch_k(layernorm_bwd_reg_kernel<NPL>, dim3(grid), dim3(wpb * 32), 0, s, x, g, dy, dx_io, add, dg, \
                    db, M, eps);
  GPT_LNB(2) GPT_LNB(4) GPT_LNB(8) GPT_LNB(12) GPT_LNB(16) GPT_LNB(24) GPT_LNB(32)
#undef GPT_LNB
  wpb = 8;
  grid = (M + wpb - 1) / wpb;
  if (grid > 2 * num_sms) grid = 2 * num_sms;
  const size_t smem = 2 * static_cast<size_t>(C) * sizeof(float);
  if (smem > 48 * 1024) return cudaErrorInvalidValue;
  return launch_k(layernorm_bwd_kernel, dim3(grid), dim3(wpb * 32), smem, s, x, g, dy, dx_io, add, dg, db, M, C, eps);
}

cudaError_t launch_embed_bwd(const float* dx0, const int32_t* ids, float* dE, float* dP, int M, int T, int C, int V,
                             cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  return launch_k(embed_bwd_kernel, dim3((M + 7) / 8), dim3(256), 0, s, dx0, ids, dE, dP, M, T, C, V);
}

}  // namespace gptgb
