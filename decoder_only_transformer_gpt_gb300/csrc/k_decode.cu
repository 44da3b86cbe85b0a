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
constexpr int kAttnDecWarps = 8;

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
  constexpr int STEP = U * 32 * SPLIT;
  // The weights do not depend on the previous kernel: the first loads are issued before
  // waiting for it, so their latency overlaps its tail.
  int c0 = part * 32 + lane;
  uint4 wv[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int c = c0 + u * 32 * SPLIT;
    wv[u] = (live && c < chunks) ? ld_stream_u4(wr + 8 * c) : make_uint4(0, 0, 0, 0);
  }
  pdl_wait();
  pdl_trigger();
  for (; live && c0 < chunks; c0 += STEP) {
    uint4 cur[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      cur[u] = wv[u];
      const int c = c0 + STEP + u * 32 * SPLIT;              // the next batch, in flight during this one
      wv[u] = c < chunks ? ld_stream_u4(wr + 8 * c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * 32 * SPLIT;
      if (c >= chunks) break;
      float wf[8];
      unpack8(cur[u], wf);
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

// One (sequence b, head h) per block of kAttnDecWarps warps. The new token's key
// and value (from its qkv row) are first stored in the cache at position pos;
// then warp w takes the 32-key chunks w, w + kAttnDecWarps, ... of keys 0..pos:
// lane i scores key 32c + i against q (shared memory), the warp turns the
// chunk's scores into probabilities against its running max (base 2), and each
// lane accumulates its D/32 output columns over the chunk's 32 value rows (each
// row read by the whole warp: 128 contiguous bytes at D = 64). The warps' partial
// results are merged in a fixed order.
template <int D>
__global__ void __launch_bounds__(kAttnDecWarps * 32)
attn_decode_kernel(const __nv_bfloat16* __restrict__ qkv, __nv_bfloat16* cache, __nv_bfloat16* __restrict__ y,
                   int H, int C, int ctx, const int* __restrict__ pos_dev, float scale_log2) {
  constexpr int DL = D / 32;                                       // output columns per lane
  constexpr int V8 = D / 8;                                        // 16-byte chunks per head slice
  __shared__ float s_q[D];
  __shared__ float s_m[kAttnDecWarps], s_l[kAttnDecWarps];
  __shared__ float s_o[kAttnDecWarps][D];
  pdl_wait();
  pdl_trigger();
  const int pos = *pos_dev;
  const int b = blockIdx.x / H, h = blockIdx.x % H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const __nv_bfloat16* qrow = qkv + (size_t)b * 3 * C;
  __nv_bfloat16* cb = cache + (size_t)b * ctx * 2 * C;             // this sequence's rows
  if (threadIdx.x < 2 * V8) {                                      // key chunks, then value chunks
    const int part = threadIdx.x / V8, c8 = threadIdx.x % V8;
    const uint4 v = *reinterpret_cast<const uint4*>(qrow + (1 + part) * C + h * D + 8 * c8);
    *reinterpret_cast<uint4*>(cb + (size_t)pos * 2 * C + part * C + h * D + 8 * c8) = v;
  }
  if (threadIdx.x < D) s_q[threadIdx.x] = __bfloat162float(qrow[h * D + threadIdx.x]) * scale_log2;
  __syncthreads();                                                 // the new row and q are visible
  float m = -INFINITY, l = 0.0f, o[DL];
#pragma unroll
  for (int d = 0; d < DL; ++d) o[d] = 0.0f;
  for (int c = warp; c * 32 <= pos; c += kAttnDecWarps) {
    const int j = c * 32 + lane;
    float sc = -INFINITY;
    if (j <= pos) {
      const __nv_bfloat16* kr = cb + (size_t)j * 2 * C + h * D;
      uint4 kv[V8];
#pragma unroll
      for (int c8 = 0; c8 < V8; ++c8) kv[c8] = *reinterpret_cast<const uint4*>(kr + 8 * c8);
      sc = 0.0f;
#pragma unroll
      for (int c8 = 0; c8 < V8; ++c8) {
        float f[8];
        unpack8(kv[c8], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) sc = fmaf(s_q[8 * c8 + i], f[i], sc);
      }
    }
    float cm = sc;                                                 // the chunk's maximum
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
    const float mn = fmaxf(m, cm);                                 // finite: key 32c <= pos exists
    const float alpha = ex2_approx(m - mn);                        // 0 on the first chunk
    const float p = ex2_approx(sc - mn);                           // 0 past pos
    float ps = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
#pragma unroll
    for (int d = 0; d < DL; ++d) o[d] *= alpha;
    m = mn;
    const int nk = min(32, pos + 1 - c * 32);                      // valid keys of this chunk
    const __nv_bfloat16* vb = cb + (size_t)(c * 32) * 2 * C + C + h * D + lane * DL;
    // all of the chunk's value loads first (32 in flight per lane), then the sums
    uint32_t vv[32];
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const __nv_bfloat16* vr = vb + (size_t)jj * 2 * C;
      if (DL == 2) vv[jj] = jj < nk ? *reinterpret_cast<const uint32_t*>(vr) : 0u;
      else vv[jj] = jj < nk ? static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(vr)) : 0u;
    }
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);             // 0 for keys past pos
      if (DL == 2) {
        const float2 v2 = unpack_bf16x2(vv[jj]);
        o[0] = fmaf(pj, v2.x, o[0]);
        o[DL - 1] = fmaf(pj, v2.y, o[DL - 1]);
      } else {
        o[0] = fmaf(pj, unpack_bf16x2(vv[jj]).x, o[0]);               // the low half holds the value
      }
    }
  }
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = l;
  }
#pragma unroll
  for (int d = 0; d < DL; ++d) s_o[warp][lane * DL + d] = o[d];
  __syncthreads();
  if (threadIdx.x < D) {
    float gm = -INFINITY;
    for (int w = 0; w < kAttnDecWarps; ++w) gm = fmaxf(gm, s_m[w]);
    float num = 0.0f, den = 0.0f;
    for (int w = 0; w < kAttnDecWarps; ++w) {                      // fixed order: deterministic
      const float sw = (s_m[w] == -INFINITY) ? 0.0f : ex2_approx(s_m[w] - gm);   // warps without keys add 0
      num = fmaf(sw, s_o[w][threadIdx.x], num);
      den = fmaf(sw, s_l[w], den);
    }
    y[(size_t)b * C + h * D + threadIdx.x] = __float2bfloat16_rn(num / den);
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

// ---------------------------------------------------------------- sampling

constexpr int kSampThreads = 1024;

// Block-wide sum (fixed order: lanes, then warps), result in every thread.
__device__ __forceinline__ float block_sum(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();                                   // scratch free from the previous use
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float t = 0.0f;
  for (int w = 0; w < kSampThreads / 32; ++w) t += scratch[w];
  return t;
}

__device__ __forceinline__ float block_max(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float t = -INFINITY;
  for (int w = 0; w < kSampThreads / 32; ++w) t = fmaxf(t, scratch[w]);
  return t;
}

// Exclusive prefix sum over threads (thread order = index order: each thread owns a
// contiguous chunk of the row), and the total.
__device__ __forceinline__ int block_scan_int(int v, int* scan, int& total) {
  __syncthreads();
  scan[threadIdx.x] = v;
  __syncthreads();
  for (int off = 1; off < kSampThreads; off <<= 1) {   // Hillis-Steele
    const int add = threadIdx.x >= off ? scan[threadIdx.x - off] : 0;
    __syncthreads();
    scan[threadIdx.x] += add;
    __syncthreads();
  }
  total = scan[kSampThreads - 1];
  return scan[threadIdx.x] - v;
}

__device__ __forceinline__ float block_scan_float(float v, float* scan, float& total) {
  __syncthreads();
  scan[threadIdx.x] = v;
  __syncthreads();
  for (int off = 1; off < kSampThreads; off <<= 1) {
    const float add = threadIdx.x >= off ? scan[threadIdx.x - off] : 0.0f;
    __syncthreads();
    scan[threadIdx.x] += add;
    __syncthreads();
  }
  total = scan[kSampThreads - 1];
  return scan[threadIdx.x] - v;
}

// One row per block: temperature, top-k, top-p and the inverse-CDF draw in index
// order ("预训练一个 Mini GPT" 第7步; "02 GPT 架构" 8.1-8.3). The probabilities of
// the row live in shared memory; thread t owns indices [t * chunk, (t + 1) * chunk),
// so per-thread counts and sums scanned over threads follow index order. Ranking
// among equal probabilities is by index, lower first.
__global__ void __launch_bounds__(kSampThreads)
sample_kernel(const float* __restrict__ logits, int V, float temperature, int top_k, float top_p,
              const float* __restrict__ uniform, int32_t* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float sp[];                      // [V] probabilities, then scratch
  float* red = sp + V;                               // [32]
  float* fscan = red + 32;                           // [kSampThreads]
  int* iscan = reinterpret_cast<int*>(fscan + kSampThreads);
  const float* z = logits + (size_t)blockIdx.x * V;
  const int chunk = (V + kSampThreads - 1) / kSampThreads;
  const int i0 = threadIdx.x * chunk;
  const int i1 = min(V, i0 + chunk);
  if (temperature <= 0.0f) {                         // greedy: the first maximum
    float best = -INFINITY;
    int bi = V;
    for (int i = i0; i < i1; ++i)
      if (z[i] > best) { best = z[i]; bi = i; }
    const float gm = block_max(best, red);
    int cand = (best == gm) ? bi : V;                // the lowest index holding the maximum
    for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) iscan[threadIdx.x >> 5] = cand;
    __syncthreads();
    if (threadIdx.x == 0) {
      int r = V;
      for (int w = 0; w < kSampThreads / 32; ++w) r = min(r, iscan[w]);
      out[blockIdx.x] = r;
    }
    return;
  }
  const float inv_t = 1.0f / temperature;
  float lm = -INFINITY;
  for (int i = i0; i < i1; ++i) {
    const float v = z[i] * inv_t;
    sp[i] = v;
    lm = fmaxf(lm, v);
  }
  const float zmax = block_max(lm, red);
  float ls = 0.0f;
  for (int i = i0; i < i1; ++i) {
    const float e = expf(sp[i] - zmax);
    sp[i] = e;                                       // unnormalised: every filter is scale-free
    ls += e;
  }
  float mass = block_sum(ls, red);
  // ---- top-k: the k-th largest value by a radix select on the bits (p >= 0: bit order = value order)
  if (top_k > 0 && top_k < V) {
    unsigned prefix = 0u, mask = 0u;
    int remaining = top_k;
    for (int shift = 24; shift >= 0; shift -= 8) {
      __syncthreads();
      for (int d = threadIdx.x; d < 256; d += kSampThreads) iscan[d] = 0;
      __syncthreads();
      for (int i = i0; i < i1; ++i) {
        const unsigned b = __float_as_uint(sp[i]);
        if ((b & mask) == prefix) atomicAdd(&iscan[(b >> shift) & 0xffu], 1);
      }
      __syncthreads();
      int d = 255, above = 0;
      while (d > 0 && above + iscan[d] < remaining) { above += iscan[d]; --d; }
      remaining -= above;                            // elements still needed among digit d
      prefix |= static_cast<unsigned>(d) << shift;
      mask |= 0xffu << shift;
    }
    // keep bits > prefix, and the first `remaining` elements equal to it in index order
    int ties = 0;
    for (int i = i0; i < i1; ++i) ties += __float_as_uint(sp[i]) == prefix;
    int total_ties;
    int rank = block_scan_int(ties, iscan, total_ties);
    float kept = 0.0f;
    for (int i = i0; i < i1; ++i) {
      const unsigned b = __float_as_uint(sp[i]);
      bool keep = b > prefix;
      if (b == prefix) keep = rank++ < remaining;
      if (!keep) sp[i] = 0.0f;
      kept += sp[i];
    }
    mass = block_sum(kept, red);
  }
  // ---- top-p: the smallest leading set (by value, then index) whose mass reaches top_p of the total
  if (top_p > 0.0f && top_p < 1.0f) {
    const float target = top_p * mass;
    unsigned v = 0u;                                 // largest v with mass(p >= v) >= target
    for (int bit = 30; bit >= 0; --bit) {
      const unsigned cand = v | (1u << bit);
      float part = 0.0f;
      for (int i = i0; i < i1; ++i)
        if (__float_as_uint(sp[i]) >= cand) part += sp[i];
      if (block_sum(part, red) >= target) v = cand;
    }
    float gt = 0.0f;
    int ties = 0;
    for (int i = i0; i < i1; ++i) {
      const unsigned b = __float_as_uint(sp[i]);
      if (b > v) gt += sp[i];
      ties += b == v;
    }
    const float mass_gt = block_sum(gt, red);
    const float pv = __uint_as_float(v);
    int total_ties;
    int rank = block_scan_int(ties, iscan, total_ties);
    // equal values added in index order until the target is reached (at least one, at most all)
    int need = total_ties;
    if (pv > 0.0f) {
      const float n = ceilf((target - mass_gt) / pv);
      need = n < 1.0f ? 1 : (n > static_cast<float>(total_ties) ? total_ties : static_cast<int>(n));
    }
    float kept = 0.0f;
    for (int i = i0; i < i1; ++i) {
      const unsigned b = __float_as_uint(sp[i]);
      bool keep = b > v;
      if (b == v && pv > 0.0f) keep = rank++ < need;
      if (!keep) sp[i] = 0.0f;
      kept += sp[i];
    }
    mass = block_sum(kept, red);
  }
  // ---- the draw: first index whose cumulative kept mass exceeds u * mass
  float mine = 0.0f;
  for (int i = i0; i < i1; ++i) mine += sp[i];
  float tot;
  const float before = block_scan_float(mine, fscan, tot);
  const float thr = uniform[blockIdx.x] * tot;
  int last = -1;                                     // the last kept index of this chunk
  for (int i = i0; i < i1; ++i)
    if (sp[i] > 0.0f) last = i;
  int found = V;
  if (before <= thr && before + mine > thr) {        // the crossing lies in this chunk
    float acc = before;
    for (int i = i0; i < i1; ++i) {
      acc += sp[i];
      if (acc > thr && sp[i] > 0.0f) { found = i; break; }
    }
    if (found == V) found = last;                    // rounding between the two summation orders
  }
  __syncthreads();
  int cand = found;
  for (int o = 16; o > 0; o >>= 1) cand = min(cand, __shfl_xor_sync(0xffffffffu, cand, o));
  int lmax = last;
  for (int o = 16; o > 0; o >>= 1) lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
  if ((threadIdx.x & 31) == 0) {
    iscan[threadIdx.x >> 5] = cand;
    iscan[32 + (threadIdx.x >> 5)] = lmax;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int r = V, lk = -1;
    for (int w = 0; w < kSampThreads / 32; ++w) {
      r = min(r, iscan[w]);
      lk = max(lk, iscan[32 + w]);
    }
    out[blockIdx.x] = r < V ? r : lk;
  }
}

// 5..16 rows: the rows are the 16-row A operand of mma.sync m16n8k16 (bf16 in,
// fp32 accumulate). Block = one 8-column tile of out; its 8 warps split K into
// contiguous ranges of whole 16-wide steps, and their 16 x 8 partial tiles are
// summed in shared memory in warp order. Fragment layout of m16n8k16: lane =
// 4 g + t holds A (g, 2t..2t+1), (g+8, ..), (g, 2t+8..), (g+8, 2t+8..);
// B (k = 2t..2t+1 and 2t+8.., n = g); C (g, 2t..2t+1) and (g+8, 2t..2t+1).
__device__ __forceinline__ uint32_t ld_u32_or0(const __nv_bfloat16* p, bool ok) {
  return ok ? *reinterpret_cast<const uint32_t*>(p) : 0u;
}

template <int EPI>
__global__ void __launch_bounds__(kGemvWarps * 32)
gemv_mma_kernel(const __nv_bfloat16* __restrict__ a, int lda, const __nv_bfloat16* __restrict__ W,
                const float* __restrict__ bias, void* out, int ldo, int M, int N, int K, int gelu_erf) {
  __shared__ float red[kGemvWarps][16][8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int n0 = blockIdx.x * 8;
  const int n = n0 + g;                                       // this lane's B column
  const bool ncol = n < N;
  const int steps = K / 16;                                   // whole 16-wide K steps (K % 16 == 0)
  const int per = (steps + kGemvWarps - 1) / kGemvWarps;
  const int s0 = warp * per, s1 = min(steps, s0 + per);
  const __nv_bfloat16* wr = W + (size_t)(ncol ? n : 0) * K;
  // the weights do not depend on the previous kernel: the first step's B is loaded before the wait
  uint32_t b0 = 0u, b1 = 0u;
  if (s0 < s1) {
    b0 = ld_u32_or0(wr + s0 * 16 + 2 * t, ncol);
    b1 = ld_u32_or0(wr + s0 * 16 + 2 * t + 8, ncol);
  }
  pdl_wait();
  pdl_trigger();
  float c0 = 0.0f, c1 = 0.0f, c2 = 0.0f, c3 = 0.0f;
  const bool r0 = g < M, r1 = g + 8 < M;
  for (int st = s0; st < s1; ++st) {
    const int k = st * 16 + 2 * t;
    uint32_t nb0 = 0u, nb1 = 0u;
    if (st + 1 < s1) {                                        // next step's weights in flight
      nb0 = ld_u32_or0(wr + k + 16, ncol);
      nb1 = ld_u32_or0(wr + k + 24, ncol);
    }
    const uint32_t a0 = ld_u32_or0(a + (size_t)g * lda + k, r0);
    const uint32_t a1 = ld_u32_or0(a + (size_t)(g + 8) * lda + k, r1);
    const uint32_t a2 = ld_u32_or0(a + (size_t)g * lda + k + 8, r0);
    const uint32_t a3 = ld_u32_or0(a + (size_t)(g + 8) * lda + k + 8, r1);
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c0), "+f"(c1), "+f"(c2), "+f"(c3)
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    b0 = nb0;
    b1 = nb1;
  }
  red[warp][g][2 * t] = c0;
  red[warp][g][2 * t + 1] = c1;
  red[warp][g + 8][2 * t] = c2;
  red[warp][g + 8][2 * t + 1] = c3;
  __syncthreads();
  for (int e = threadIdx.x; e < 16 * 8; e += kGemvWarps * 32) {
    const int r = e >> 3, cn = e & 7;
    const int col = n0 + cn;
    if (r >= M || col >= N) continue;
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kGemvWarps; ++w) v += red[w][r][cn];   // fixed order
    if (bias != nullptr) v += __ldg(bias + col);
    if (EPI == EPI_BIAS_OUT) {
      reinterpret_cast<__nv_bfloat16*>(out)[(size_t)r * ldo + col] = __float2bfloat16_rn(v);
    } else if (EPI == EPI_BIAS_GELU_OUT) {
      reinterpret_cast<__nv_bfloat16*>(out)[(size_t)r * ldo + col] = __float2bfloat16_rn(gelu_dec(v, gelu_erf));
    } else if (EPI == EPI_BIAS_RESID) {
      reinterpret_cast<float*>(out)[(size_t)r * ldo + col] += v;
    } else {
      reinterpret_cast<float*>(out)[(size_t)r * ldo + col] = v;
    }
  }
}

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
  if (M > 4 && K % 16 == 0)                                    // 5..16 rows: tensor-core tiles
    return launch_k(gemv_mma_kernel<EPI>, dim3((N + 7) / 8), dim3(kGemvWarps * 32), 0, s, a, lda, W, bias, out, ldo,
                    M, N, K, gelu_erf);
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
    return launch_k(attn_decode_kernel<64>, dim3(B * H), dim3(kAttnDecWarps * 32), 0, s, q, c, yo, H, C, ctx, pos_dev,
                    scale_log2);
  if (D == 32)
    return launch_k(attn_decode_kernel<32>, dim3(B * H), dim3(kAttnDecWarps * 32), 0, s, q, c, yo, H, C, ctx, pos_dev,
                    scale_log2);
  return cudaErrorInvalidValue;
}

cudaError_t launch_set_int(int* p, int v, cudaStream_t s) {
  set_int_kernel<<<1, 1, 0, s>>>(p, v);
  return cudaGetLastError();
}

cudaError_t launch_sample(const float* logits, int B, int V, float temperature, int top_k, float top_p,
                          const float* uniform, int32_t* out, cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  if (V <= 0 || V > kSampleMaxV) return cudaErrorInvalidValue;
  const size_t smem = (static_cast<size_t>(V) + 32 + 2 * kSampThreads) * 4;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>((kSampleMaxV + 32 + 2 * kSampThreads) * 4));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_k(sample_kernel, dim3(B), dim3(kSampThreads), smem, s, logits, V, temperature, top_k, top_p, uniform,
                  out);
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
