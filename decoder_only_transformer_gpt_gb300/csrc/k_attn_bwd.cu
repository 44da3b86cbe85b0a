// Derivative of causal self-attention on the tensor cores with mma.sync m16n8k16
// (bf16 operands, fp32 accumulation).
//
// Forward ("第 25 章 从小 GPT 到 GPT-2" §25.2): S = Q K^T / sqrt(D) with s > t
// masked, A = softmax(S) per row, Y = A U. With A recomputed from the row's
// log-sum-exp and Dsum[t] = sum_d dY[t,d] Y[t,d] (= sum_s A[t,s] dA[t,s]):
//   dA = dY U^T, dS = A * (dA - Dsum), dQ = dS K / sqrt(D), dK = dS^T Q / sqrt(D), dU = A^T dY.
// Two kernels, neither with atomics: the first owns 16 query rows per warp (the
// row statistics, then dQ), the second 16 key rows per warp (dK and dU over the
// queries that can see them). Fragment layout of m16n8k16 (lane = 4 g + c):
// A (g, 2c..2c+1), (g+8, ..), (g, 2c+8..), (g+8, 2c+8..); B (k = 2c..2c+1 and
// 2c+8.., n = g); C (g, 2c..2c+1) and (g+8, 2c..2c+1). Operands whose k index
// runs along rows in memory (K for dQ, Q and dY for dK and dU) go through a
// transposed 16-row staging tile in shared memory.
#include "common.cuh"
#include "kernels.h"
#include "launch.h"

#include <cuda_bf16.h>
#include <math.h>

namespace gptgb {

namespace {

constexpr int kAbWarps = 4;     // warps per block, 16 rows each
constexpr int kTs = 24;         // row stride (halves) of a transposed staging tile: 12 words, conflict-free reads

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t ld32(const __nv_bfloat16* p, bool ok) {
  return ok ? *reinterpret_cast<const uint32_t*>(p) : 0u;
}

__device__ __forceinline__ float dot2(uint32_t u, uint32_t v) {
  const float2 a = unpack_bf16x2(u), b = unpack_bf16x2(v);
  return a.x * b.x + a.y * b.y;
}

// A operand (16 rows r0.. of X, row stride ldx, all D columns) as KK fragments; rows >= T read as 0.
template <int D>
__device__ __forceinline__ void load_a(uint32_t (&a)[D / 16][4], const __nv_bfloat16* X, int ldx, int r0, int T,
                                       int g, int c) {
  const int ra = r0 + g, rb = r0 + g + 8;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int col = kk * 16 + 2 * c;
    a[kk][0] = ld32(X + static_cast<size_t>(ra) * ldx + col, ra < T);
    a[kk][1] = ld32(X + static_cast<size_t>(rb) * ldx + col, rb < T);
    a[kk][2] = ld32(X + static_cast<size_t>(ra) * ldx + col + 8, ra < T);
    a[kk][3] = ld32(X + static_cast<size_t>(rb) * ldx + col + 8, rb < T);
  }
}

// st[j] (16 x 8, j = 0, 1) = A . X[r0 + 8j .. r0 + 8j + 7]^T over the D columns: B comes straight
// from X's rows (k = the column, contiguous in memory).
template <int D>
__device__ __forceinline__ void tile16(float (&st)[2][4], const uint32_t (&a)[D / 16][4], const __nv_bfloat16* X,
                                       int ldx, int r0, int T, int g, int c) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    st[j][0] = st[j][1] = st[j][2] = st[j][3] = 0.0f;
    const int r = r0 + 8 * j + g;
    const bool ok = r < T;
    const __nv_bfloat16* xr = X + static_cast<size_t>(ok ? r : 0) * ldx + 2 * c;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) mma16816(st[j], a[kk], ld32(xr + kk * 16, ok), ld32(xr + kk * 16 + 8, ok));
  }
}

// xt[d][r] = X[r0 + r][d] for r < 16 (0 past T): the B operand of a product whose k index is the row.
template <int D>
__device__ __forceinline__ void stage_t(uint16_t* xt, const __nv_bfloat16* X, int ldx, int r0, int T, int lane) {
  for (int e = lane; e < 16 * (D / 2); e += 32) {
    const int r = e / (D / 2), p = e - r * (D / 2);
    const uint32_t v = ld32(X + static_cast<size_t>(r0 + r) * ldx + 2 * p, r0 + r < T);
    xt[(2 * p) * kTs + r] = static_cast<uint16_t>(v & 0xffffu);
    xt[(2 * p + 1) * kTs + r] = static_cast<uint16_t>(v >> 16);
  }
}

// acc[jd] += a . B, B[k][n] = xt[8 jd + n][k] (k < 16), for the D / 8 column tiles.
template <int D>
__device__ __forceinline__ void acc_from_stage(float (&acc)[D / 8][4], const uint32_t (&a)[4], const uint16_t* xt,
                                               int g, int c) {
#pragma unroll
  for (int jd = 0; jd < D / 8; ++jd) {
    const uint16_t* row = xt + (8 * jd + g) * kTs + 2 * c;
    mma16816(acc[jd], a, *reinterpret_cast<const uint32_t*>(row), *reinterpret_cast<const uint32_t*>(row + 8));
  }
}

// C fragments of a 16 x 16 tile (two n8 tiles) as the A operand of the next product.
__device__ __forceinline__ void c_to_a(uint32_t (&a)[4], const float (&v)[2][4]) {
  a[0] = pack_bf16x2(v[0][0], v[0][1]);
  a[1] = pack_bf16x2(v[0][2], v[0][3]);
  a[2] = pack_bf16x2(v[1][0], v[1][1]);
  a[3] = pack_bf16x2(v[1][2], v[1][3]);
}

// ---- dQ: a warp owns query rows t0 .. t0 + 15 of one (sequence, head)
template <int D>
__global__ void __launch_bounds__(kAbWarps * 32)
attn_bwd_dq_kernel(const __nv_bfloat16* __restrict__ qkv, const __nv_bfloat16* __restrict__ y,
                   const __nv_bfloat16* __restrict__ dy, __nv_bfloat16* __restrict__ dqkv, float* __restrict__ lse2_out,
                   float* __restrict__ dsum_out, int T, int H, float sl2, float rsd) {
  pdl_wait();
  pdl_trigger();
  constexpr int KK = D / 16, ND = D / 8;
  __shared__ __align__(16) uint16_t stage[kAbWarps][D * kTs];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int bh = blockIdx.y, b = bh / H, h = bh - b * H;
  const int C = H * D, C3 = 3 * C;
  const int t0 = blockIdx.x * (kAbWarps * 16) + warp * 16;
  if (t0 >= T) return;
  const size_t base = static_cast<size_t>(b) * T;
  const __nv_bfloat16* Q = qkv + base * C3 + h * D;
  const __nv_bfloat16* K = Q + C;
  const __nv_bfloat16* U = Q + 2 * C;
  const __nv_bfloat16* O = y + base * C + h * D;
  const __nv_bfloat16* dO = dy + base * C + h * D;
  const int ra = t0 + g, rb = t0 + g + 8;

  uint32_t qa[KK][4], da[KK][4];
  load_a<D>(qa, Q, C3, t0, T, g, c);
  load_a<D>(da, dO, C, t0, T, g, c);
  float dsa = 0.0f, dsb = 0.0f;              // Dsum of rows ra and rb (this lane's columns, then the quad's)
#pragma unroll
  for (int kk = 0; kk < KK; ++kk) {
    const int col = kk * 16 + 2 * c;
    dsa += dot2(da[kk][0], ld32(O + static_cast<size_t>(ra) * C + col, ra < T)) +
           dot2(da[kk][2], ld32(O + static_cast<size_t>(ra) * C + col + 8, ra < T));
    dsb += dot2(da[kk][1], ld32(O + static_cast<size_t>(rb) * C + col, rb < T)) +
           dot2(da[kk][3], ld32(O + static_cast<size_t>(rb) * C + col + 8, rb < T));
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    dsa += __shfl_xor_sync(0xffffffffu, dsa, o);
    dsb += __shfl_xor_sync(0xffffffffu, dsb, o);
  }

  // pass 1: the rows' log-sum-exp (base 2) over keys 0 .. min(T, t0 + 16) - 1
  const int kend = min(T, t0 + 16);
  float ma = -INFINITY, la = 0.0f, mb = -INFINITY, lb = 0.0f;
  for (int s0 = 0; s0 < kend; s0 += 16) {
    float st[2][4];
    tile16<D>(st, qa, K, C3, s0, T, g, c);
    float v[2][4];
    float xa = -INFINITY, xb = -INFINITY;
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = s0 + 8 * j + 2 * c + (e & 1);
        const int row = e < 2 ? ra : rb;
        v[j][e] = (key <= row && key < T) ? st[j][e] * sl2 : -INFINITY;
        if (e < 2) xa = fmaxf(xa, v[j][e]); else xb = fmaxf(xb, v[j][e]);
      }
    if (xa > -INFINITY) {
      const float nm = fmaxf(ma, xa);
      float acc = la * ex2_approx(ma - nm);
#pragma unroll
      for (int j = 0; j < 2; ++j) acc += ex2_approx(v[j][0] - nm) + ex2_approx(v[j][1] - nm);
      la = acc;
      ma = nm;
    }
    if (xb > -INFINITY) {
      const float nm = fmaxf(mb, xb);
      float acc = lb * ex2_approx(mb - nm);
#pragma unroll
      for (int j = 0; j < 2; ++j) acc += ex2_approx(v[j][2] - nm) + ex2_approx(v[j][3] - nm);
      lb = acc;
      mb = nm;
    }
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    const float moa = __shfl_xor_sync(0xffffffffu, ma, o), loa = __shfl_xor_sync(0xffffffffu, la, o);
    const float mob = __shfl_xor_sync(0xffffffffu, mb, o), lob = __shfl_xor_sync(0xffffffffu, lb, o);
    const float na = fmaxf(ma, moa), nb = fmaxf(mb, mob);
    if (na > -INFINITY) {
      la = (ma > -INFINITY ? la * ex2_approx(ma - na) : 0.0f) + (moa > -INFINITY ? loa * ex2_approx(moa - na) : 0.0f);
      ma = na;
    }
    if (nb > -INFINITY) {
      lb = (mb > -INFINITY ? lb * ex2_approx(mb - nb) : 0.0f) + (mob > -INFINITY ? lob * ex2_approx(mob - nb) : 0.0f);
      mb = nb;
    }
  }
  const float lsa = ma + log2f(la), lsb = mb + log2f(lb);

  // pass 2: dS = A * (dA - Dsum) tile by tile, dQ += dS K
  float dq[ND][4];
#pragma unroll
  for (int jd = 0; jd < ND; ++jd) dq[jd][0] = dq[jd][1] = dq[jd][2] = dq[jd][3] = 0.0f;
  uint16_t* xt = stage[warp];
  for (int s0 = 0; s0 < kend; s0 += 16) {
    float st[2][4], dp[2][4];
    tile16<D>(st, qa, K, C3, s0, T, g, c);
    tile16<D>(dp, da, U, C3, s0, T, g, c);
    float ds[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = s0 + 8 * j + 2 * c + (e & 1);
        const int row = e < 2 ? ra : rb;
        const float p = (key <= row && key < T) ? ex2_approx(st[j][e] * sl2 - (e < 2 ? lsa : lsb)) : 0.0f;
        ds[j][e] = p * (dp[j][e] - (e < 2 ? dsa : dsb));
      }
    uint32_t a[4];
    c_to_a(a, ds);
    __syncwarp();
    stage_t<D>(xt, K, C3, s0, T, lane);
    __syncwarp();
    acc_from_stage<D>(dq, a, xt, g, c);
  }
  __nv_bfloat16* dQ = dqkv + base * C3 + h * D;
#pragma unroll
  for (int jd = 0; jd < ND; ++jd) {
    const int col = 8 * jd + 2 * c;
    if (ra < T)
      *reinterpret_cast<uint32_t*>(dQ + static_cast<size_t>(ra) * C3 + col) = pack_bf16x2(dq[jd][0] * rsd, dq[jd][1] * rsd);
    if (rb < T)
      *reinterpret_cast<uint32_t*>(dQ + static_cast<size_t>(rb) * C3 + col) = pack_bf16x2(dq[jd][2] * rsd, dq[jd][3] * rsd);
  }
  if (c == 0) {
    const size_t r0 = static_cast<size_t>(bh) * T;
    if (ra < T) { lse2_out[r0 + ra] = lsa; dsum_out[r0 + ra] = dsa; }
    if (rb < T) { lse2_out[r0 + rb] = lsb; dsum_out[r0 + rb] = dsb; }
  }
}

// ---- dK and dU: a warp owns key rows s0 .. s0 + 15 and walks the queries t >= s0
template <int D>
__global__ void __launch_bounds__(kAbWarps * 32)
attn_bwd_dkv_kernel(const __nv_bfloat16* __restrict__ qkv, const __nv_bfloat16* __restrict__ dy,
                    const float* __restrict__ lse2, const float* __restrict__ dsum, __nv_bfloat16* __restrict__ dqkv,
                    int T, int H, float sl2, float rsd) {
  pdl_wait();
  pdl_trigger();
  constexpr int KK = D / 16, ND = D / 8;
  __shared__ __align__(16) uint16_t stage[kAbWarps][2][D * kTs];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int bh = blockIdx.y, b = bh / H, h = bh - b * H;
  const int C = H * D, C3 = 3 * C;
  const int s0 = blockIdx.x * (kAbWarps * 16) + warp * 16;
  if (s0 >= T) return;
  const size_t base = static_cast<size_t>(b) * T;
  const __nv_bfloat16* Q = qkv + base * C3 + h * D;
  const __nv_bfloat16* K = Q + C;
  const __nv_bfloat16* U = Q + 2 * C;
  const __nv_bfloat16* dO = dy + base * C + h * D;
  const float* ls = lse2 + static_cast<size_t>(bh) * T;
  const float* dsm = dsum + static_cast<size_t>(bh) * T;
  const int ka = s0 + g, kb = s0 + g + 8;

  uint32_t kfr[KK][4], ufr[KK][4];
  load_a<D>(kfr, K, C3, s0, T, g, c);
  load_a<D>(ufr, U, C3, s0, T, g, c);
  float dk[ND][4], du[ND][4];
#pragma unroll
  for (int jd = 0; jd < ND; ++jd)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[jd][e] = du[jd][e] = 0.0f;
  uint16_t* qt = stage[warp][0];
  uint16_t* ot = stage[warp][1];
  for (int t0 = s0; t0 < T; t0 += 16) {
    float st[2][4], dp[2][4];
    tile16<D>(st, kfr, Q, C3, t0, T, g, c);       // S^T: keys x queries
    tile16<D>(dp, ufr, dO, C, t0, T, g, c);       // dA^T = U dY^T
    float p[2][4], ds[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int q = t0 + 8 * j + 2 * c + h2;
        const bool qok = q < T;
        const float l = qok ? ls[q] : 0.0f;
        const float dq = qok ? dsm[q] : 0.0f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int e = 2 * half + h2;
          const int key = half == 0 ? ka : kb;
          const float pv = (qok && key <= q) ? ex2_approx(st[j][e] * sl2 - l) : 0.0f;
          p[j][e] = pv;
          ds[j][e] = pv * (dp[j][e] - dq);
        }
      }
    }
    uint32_t ap[4], as[4];
    c_to_a(ap, p);
    c_to_a(as, ds);
    __syncwarp();
    stage_t<D>(qt, Q, C3, t0, T, lane);
    stage_t<D>(ot, dO, C, t0, T, lane);
    __syncwarp();
    acc_from_stage<D>(du, ap, ot, g, c);          // dU += A^T dY
    acc_from_stage<D>(dk, as, qt, g, c);          // dK += dS^T Q
  }
  __nv_bfloat16* dK = dqkv + base * C3 + C + h * D;
  __nv_bfloat16* dU = dK + C;
#pragma unroll
  for (int jd = 0; jd < ND; ++jd) {
    const int col = 8 * jd + 2 * c;
    if (ka < T) {
      *reinterpret_cast<uint32_t*>(dK + static_cast<size_t>(ka) * C3 + col) = pack_bf16x2(dk[jd][0] * rsd, dk[jd][1] * rsd);
      *reinterpret_cast<uint32_t*>(dU + static_cast<size_t>(ka) * C3 + col) = pack_bf16x2(du[jd][0], du[jd][1]);
    }
    if (kb < T) {
      *reinterpret_cast<uint32_t*>(dK + static_cast<size_t>(kb) * C3 + col) = pack_bf16x2(dk[jd][2] * rsd, dk[jd][3] * rsd);
      *reinterpret_cast<uint32_t*>(dU + static_cast<size_t>(kb) * C3 + col) = pack_bf16x2(du[jd][2], du[jd][3]);
    }
  }
}

}  // namespace

cudaError_t launch_attention_bwd(const void* qkv, const void* y, const void* dy, void* dqkv, float* lse2, float* dsum,
                                 int B, int T, int H, int D, cudaStream_t s) {
  if (B <= 0 || T <= 0) return cudaSuccess;
  const dim3 grid((T + kAbWarps * 16 - 1) / (kAbWarps * 16), B * H), block(kAbWarps * 32);
  const float rsd = 1.0f / sqrtf(static_cast<float>(D));
  const float sl2 = rsd * 1.4426950408889634f;
  const auto* q = static_cast<const __nv_bfloat16*>(qkv);
  const auto* yy = static_cast<const __nv_bfloat16*>(y);
  const auto* d = static_cast<const __nv_bfloat16*>(dy);
  auto* o = static_cast<__nv_bfloat16*>(dqkv);
  cudaError_t e;
  if (D == 64) {
    e = launch_k(attn_bwd_dq_kernel<64>, grid, block, 0, s, q, yy, d, o, lse2, dsum, T, H, sl2, rsd);
    if (e != cudaSuccess) return e;
    return launch_k(attn_bwd_dkv_kernel<64>, grid, block, 0, s, q, d, static_cast<const float*>(lse2),
                    static_cast<const float*>(dsum), o, T, H, sl2, rsd);
  }
  if (D == 32) {
    e = launch_k(attn_bwd_dq_kernel<32>, grid, block, 0, s, q, yy, d, o, lse2, dsum, T, H, sl2, rsd);
    if (e != cudaSuccess) return e;
    return launch_k(attn_bwd_dkv_kernel<32>, grid, block, 0, s, q, d, static_cast<const float*>(lse2),
                    static_cast<const float*>(dsum), o, T, H, sl2, rsd);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gptgb
