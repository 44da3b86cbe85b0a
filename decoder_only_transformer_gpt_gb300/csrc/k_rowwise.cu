// Row-wise, HBM-bound kernels: embedding gather-add (optionally fused with the
// first LayerNorm), LayerNorm, cross-entropy combine and the mean of the loss.
//
// One warp owns one row of C values; each lane holds C/256 chunks of 8
// consecutive values, loaded with 128-bit accesses (8 bf16 or two float4), so a
// warp instruction moves 512 contiguous bytes. Statistics use warp shuffles
// only: no shared memory, no block barrier.
#include "common.cuh"
#include "kernels.h"
#include "launch.h"

#include <math.h>

namespace gptgb {

namespace {

constexpr int kRowThreads = 256;       // 8 warps = 8 rows per block

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}


// 8 consecutive values of a row as fp32
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  float2 f;
  f = unpack_bf16x2(u.x); v[0] = f.x; v[1] = f.y;
  f = unpack_bf16x2(u.y); v[2] = f.x; v[3] = f.y;
  f = unpack_bf16x2(u.z); v[4] = f.x; v[5] = f.y;
  f = unpack_bf16x2(u.w); v[6] = f.x; v[7] = f.y;
}

__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 u;
  u.x = pack_bf16x2(v[0], v[1]);
  u.y = pack_bf16x2(v[2], v[3]);
  u.z = pack_bf16x2(v[4], v[5]);
  u.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = u;
}

// Normalise the warp's row held in v[NV][8] (elements e = (k*32 + lane)*8 + i);
// with g == nullptr the row is only cast to the output type.
template <int NV, typename OT>
__device__ __forceinline__ void ln_row(float (&v)[NV][8], int lane, int C, float eps, const float* __restrict__ g,
                                       const float* __restrict__ bta, OT* out_row, float* f32_row) {
  if (g == nullptr) {                 // no normalisation: a plain cast of the row
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int e = (k * 32 + lane) * 8;
      if (e < C) {
        store8(out_row + e, v[k]);
        if (f32_row) store8(f32_row + e, v[k]);
      }
    }
    return;
  }
  float s = 0.0f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if ((k * 32 + lane) * 8 < C) {
#pragma unroll
      for (int i = 0; i < 8; ++i) s += v[k][i];
    }
  }
  const float mean = warp_sum(s) / static_cast<float>(C);
  float q = 0.0f;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    if ((k * 32 + lane) * 8 < C) {
#pragma unroll
      for (int i = 0; i < 8; ++i) { const float d = v[k][i] - mean; q += d * d; }
    }
  }
  const float var = warp_sum(q) / static_cast<float>(C);      // biased variance
  const float rstd = rsqrtf(var + eps);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int e = (k * 32 + lane) * 8;
    if (e < C) {
      float gg[8], bb[8], yv[8];
      load8(g + e, gg);
      load8(bta + e, bb);
#pragma unroll
      for (int i = 0; i < 8; ++i) yv[i] = (v[k][i] - mean) * rstd * gg[i] + bb[i];
      store8(out_row + e, yv);
      if (f32_row) store8(f32_row + e, yv);
    }
  }
}

// x[m] = E[ids[m]] + P[m % T]; then out_mode 0: nothing more, 1: out = x (cast),
// 2: out = LN(x) with (g, b).
template <int NV, typename WT, typename OT>
__global__ void __launch_bounds__(kRowThreads)
embed_kernel(const int32_t* __restrict__ ids, const WT* __restrict__ wte, const WT* __restrict__ wpe,
             float* __restrict__ x, OT* __restrict__ out, int out_mode, const float* __restrict__ g,
             const float* __restrict__ b, int M, int T, int C, int V, float eps, int* err, int pos0,
             const int* __restrict__ pos_dev) {
  pdl_wait();
  pdl_trigger();
  const int warp = (blockIdx.x * kRowThreads + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= M) return;
  int id = __ldg(ids + warp);
  if (id < 0 || id >= V) {
    if (lane == 0) record_error(err, GPT_DEV_ETOKEN);
    id = 0;                                   // keep the row defined; the call reports the error
  }
  const int t = (pos_dev != nullptr ? *pos_dev : pos0) + warp % T;
  const WT* erow = wte + (size_t)id * C;
  const WT* prow = wpe + (size_t)t * C;
  float* xrow = x + (size_t)warp * C;
  float v[NV][8];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int e = (k * 32 + lane) * 8;
    if (e < C) {
      float pe[8];
      load8(erow + e, v[k]);
      load8(prow + e, pe);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[k][i] += pe[i];
      store8(xrow + e, v[k]);
      if (out_mode == 1) store8(out + (size_t)warp * C + e, v[k]);
    }
  }
  if (out_mode == 2) ln_row<NV, OT>(v, lane, C, eps, g, b, out + (size_t)warp * C, nullptr);
}

// One warp per row; the row's loads are all issued before any arithmetic.
template <int NV, typename OT>
__global__ void __launch_bounds__(kRowThreads)
layernorm_kernel(const float* x, const float* __restrict__ g, const float* __restrict__ b, OT* __restrict__ out,
                 float* out_f32, int M, int C, float eps) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (kRowThreads / 32) + (threadIdx.x >> 5);
  if (row >= M) return;
  float v[NV][8];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int e = (k * 32 + lane) * 8;
    if (e < C) load8(x + (size_t)row * C + e, v[k]);
  }
  ln_row<NV, OT>(v, lane, C, eps, g, b, out + (size_t)row * C, out_f32 ? out_f32 + (size_t)row * C : nullptr);
}

template <typename WT, typename OT>
cudaError_t embed_dispatch(const int32_t* ids, const WT* wte, const WT* wpe, float* x, OT* out, int out_mode,
                           const float* g, const float* b, int M, int T, int C, int V, float eps, int* err,
                           cudaStream_t s, int pos0, const int* pos_dev) {
  const int blocks = (M + 7) / 8;
  const int nv = (C + 255) / 256;
  cudaError_t e = cudaSuccess;
#define GPT_EMB(NVV) e = launch_k(embed_kernel<NVV, WT, OT>, dim3(blocks), dim3(kRowThreads), 0, s, ids, wte, wpe, x, out, out_mode, g, b, M, T, C, V, eps, err, pos0, pos_dev)
  switch (nv) {
    case 1: GPT_EMB(1); break;
    case 2: GPT_EMB(2); break;
    case 3: GPT_EMB(3); break;
    case 4: GPT_EMB(4); break;
    case 5: case 6: GPT_EMB(6); break;
    case 7: case 8: GPT_EMB(8); break;
    default: return cudaErrorInvalidValue;
  }
#undef GPT_EMB
  return e;
}

template <typename OT>
cudaError_t ln_dispatch(const float* x, const float* g, const float* b, OT* out, float* out_f32, int M, int C,
                        float eps, cudaStream_t s) {
  const int blocks = (M + 7) / 8;
  const int nv = (C + 255) / 256;
  cudaError_t e = cudaSuccess;
#define GPT_LN(NVV) e = launch_k(layernorm_kernel<NVV, OT>, dim3(blocks), dim3(kRowThreads), 0, s, x, g, b, out, out_f32, M, C, eps)
  switch (nv) {
    case 1: GPT_LN(1); break;
    case 2: GPT_LN(2); break;
    case 3: GPT_LN(3); break;
    case 4: GPT_LN(4); break;
    case 5: case 6: GPT_LN(6); break;
    case 7: case 8: GPT_LN(8); break;
    default: return cudaErrorInvalidValue;
  }
#undef GPT_LN
  return e;
}

// nll[m] = logsumexp over the row's tile partials - target logit, in one pass.
// A block owns 32 rows (lane = row); its 8 warps split the NB column tiles and
// fold them online into (max, sum), then merge through shared memory. The
// block also writes the sum of its rows' nll for the mean (fixed order).
constexpr int kCeRows = 32;
constexpr int kCeWarps = 8;
constexpr int kCeGroup = 16;          // tiles per warp whose partials are loaded together

__global__ void __launch_bounds__(kCeRows * kCeWarps)
ce_combine_kernel(const float* __restrict__ pmax, const float* __restrict__ psum,
                  const float* __restrict__ ztgt, const int32_t* __restrict__ targets,
                  float* __restrict__ nll, float* __restrict__ block_sums, int M, int NB, int V, int* err) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sm_m[kCeWarps][kCeRows];
  __shared__ float sm_s[kCeWarps][kCeRows];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int m = blockIdx.x * kCeRows + lane;
  float mx = -INFINITY, s = 0.0f;
  if (m < M) {
    // this warp's tiles t = warp, warp + 8, ...: kCeGroup of them loaded at once,
    // then folded into the running (max, sum) with one rescale per group
    for (int t0 = warp; t0 < NB; t0 += kCeGroup * kCeWarps) {
      float pm[kCeGroup], ps[kCeGroup];
#pragma unroll
      for (int k = 0; k < kCeGroup; ++k) {
        const int t = t0 + k * kCeWarps;
        pm[k] = t < NB ? __ldg(pmax + (size_t)t * M + m) : -INFINITY;
        ps[k] = t < NB ? __ldg(psum + (size_t)t * M + m) : 0.0f;
      }
      float gm = mx;
#pragma unroll
      for (int k = 0; k < kCeGroup; ++k) gm = fmaxf(gm, pm[k]);
      if (gm != -INFINITY) {
        float acc = (mx == -INFINITY) ? 0.0f : s * expf(mx - gm);
#pragma unroll
        for (int k = 0; k < kCeGroup; ++k)
          if (pm[k] != -INFINITY) acc += ps[k] * expf(pm[k] - gm);
        s = acc;
        mx = gm;
      }
    }
  }
  sm_m[warp][lane] = mx;
  sm_s[warp][lane] = s;
  __syncthreads();
  if (warp == 0) {
    float v = 0.0f;
    if (m < M) {
      float gm = -INFINITY;
#pragma unroll
      for (int w = 0; w < kCeWarps; ++w) gm = fmaxf(gm, sm_m[w][lane]);
      float gs = 0.0f;
#pragma unroll
      for (int w = 0; w < kCeWarps; ++w)
        if (sm_m[w][lane] != -INFINITY) gs += sm_s[w][lane] * expf(sm_m[w][lane] - gm);
      const int tg = __ldg(targets + m);
      if (tg < 0 || tg >= V) {
        record_error(err, GPT_DEV_ETARGET);
      } else {
        v = gm + logf(gs) - __ldg(ztgt + m);
      }
      nll[m] = v;
    }
    // fixed-order sum of this block's 32 values
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0 && block_sums) block_sums[blockIdx.x] = v;
  }
}

// loss = (sum of the partial sums) / M in a fixed order: each lane of one warp
// sums a strided slice in fp64 (four loads in flight), then a shuffle tree in fp64.
__global__ void __launch_bounds__(32) mean_kernel(const float* __restrict__ part, int n, int M, float* loss) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x;
  double s = 0.0;
  int i = lane;
  for (; i + 96 < n; i += 128) {
    const float a = part[i], b = part[i + 32], c = part[i + 64], d = part[i + 96];
    s += static_cast<double>(a);
    s += static_cast<double>(b);
    s += static_cast<double>(c);
    s += static_cast<double>(d);
  }
  for (; i < n; i += 32) s += static_cast<double>(part[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) *loss = static_cast<float>(s / static_cast<double>(M));
}

}  // namespace

cudaError_t launch_embed(const int32_t* ids, const void* wte, const void* wpe, int wdt, float* x, void* out,
                         int out_mode, int odt, const float* g, const float* b, int M, int T, int C, int V,
                         float eps, int* err, cudaStream_t s, int pos0, const int* pos_dev) {
  if (M <= 0) return cudaSuccess;
  if (wdt == 1) {
    const __nv_bfloat16* E = reinterpret_cast<const __nv_bfloat16*>(wte);
    const __nv_bfloat16* P = reinterpret_cast<const __nv_bfloat16*>(wpe);
    if (odt == 1)
      return embed_dispatch(ids, E, P, x, reinterpret_cast<__nv_bfloat16*>(out), out_mode, g, b, M, T, C, V, eps, err, s, pos0, pos_dev);
    return embed_dispatch(ids, E, P, x, reinterpret_cast<float*>(out), out_mode, g, b, M, T, C, V, eps, err, s, pos0, pos_dev);
  }
  const float* E = reinterpret_cast<const float*>(wte);
  const float* P = reinterpret_cast<const float*>(wpe);
  if (odt == 1)
    return embed_dispatch(ids, E, P, x, reinterpret_cast<__nv_bfloat16*>(out), out_mode, g, b, M, T, C, V, eps, err, s, pos0, pos_dev);
  return embed_dispatch(ids, E, P, x, reinterpret_cast<float*>(out), out_mode, g, b, M, T, C, V, eps, err, s, pos0, pos_dev);
}

cudaError_t launch_layernorm(const float* x, const float* g, const float* b, void* out, int odt, float* out_f32,
                             int M, int C, float eps, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (odt == 1) return ln_dispatch(x, g, b, reinterpret_cast<__nv_bfloat16*>(out), out_f32, M, C, eps, s);
  return ln_dispatch(x, g, b, reinterpret_cast<float*>(out), out_f32, M, C, eps, s);
}

cudaError_t launch_ce_combine(const float* pmax, const float* psum, const float* ztgt, const int32_t* targets,
                              float* nll, float* block_sums, int M, int NB, int V, int* err, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  return launch_k(ce_combine_kernel, dim3((M + kCeRows - 1) / kCeRows), dim3(kCeRows * kCeWarps), 0, s, pmax, psum,
                  ztgt, targets, nll, block_sums, M, NB, V, err);
}

int ce_combine_blocks(int M) { return (M + kCeRows - 1) / kCeRows; }

cudaError_t launch_mean(const float* part, int n, int M, float* loss, cudaStream_t s) {
  if (M <= 0 || n <= 0) return cudaSuccess;
  return launch_k(mean_kernel, dim3(1), dim3(32), 0, s, part, n, M, loss);
}

}  // namespace gptgb
