// Derivative of causal self-attention on the tensor cores with mma.sync m16n8k16
// (bf16 operands, fp32 accumulation).
//
// Forward ("第 25 章 从小 GPT 到 GPT-2" §25.2): S = Q K^T / sqrt(D) with s > t
// masked, A = softmax(S) per row, Y = A U. With A recomputed from the row's
// log-sum-exp and Dsum[t] = sum_d dY[t,d] Y[t,d] (= sum_s A[t,s] dA[t,s]):
//   dA = dY U^T, dS = A * (dA - Dsum), dQ = dS K / sqrt(D), dK = dS^T Q / sqrt(D), dU = A^T dY.
// Two kernels, neither with atomics. A block owns 64 rows (4 warps x 16): the
// first 64 queries (their row statistics, then dQ over the keys they see), the
// second 64 keys (dK and dU over the queries that see them). The other side's
// rows stream through shared memory in 64-row tiles with cp.async, double
// buffered; fragments come from shared memory with ldmatrix, transposed
// (.trans) where the product's k index runs along the tile's rows.
//
// m16n8k16 fragments (lane = 4 g + c): A (g, 2c..2c+1), (g+8, ..), (g, 2c+8..),
// (g+8, 2c+8..); B (k = 2c..2c+1 and 2c+8.., n = g); C (g, 2c..2c+1), (g+8, ..).
#include "common.cuh"
#include "kernels.h"
#include "launch.h"

#include <cuda_bf16.h>
#include <math.h>

namespace gptgb {

namespace {

constexpr int kAbRows = 64;      // rows per block and per streamed tile
constexpr int kAbThreads = 128;  // 4 warps x 16 rows

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const uint16_t* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const uint16_t* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// 16 bytes global -> shared, zero-filled when !ok (no bytes are read then).
__device__ __forceinline__ void cp_async16(uint16_t* dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(ok ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Rows r0 .. r0 + 63 of a head's [T, D] slice (row stride ld elements) into a [64][D + 8] tile;
// rows past T are zeros.
template <int D>
__device__ __forceinline__ void load_tile(uint16_t* dst, const __nv_bfloat16* src, int ld, int r0, int T, int tid) {
  constexpr int RS = D + 8, CPR = D / 8;
  for (int i = tid; i < kAbRows * CPR; i += kAbThreads) {
    const int r = i / CPR, ch = i - r * CPR;
    const bool ok = r0 + r < T;
    cp_async16(dst + r * RS + ch * 8, src + static_cast<size_t>(ok ? r0 + r : 0) * ld + ch * 8, ok);
  }
}

// A operand (16 rows rb.. of a tile, all D columns) as D/16 fragments.
template <int D>
__device__ __forceinline__ void frag_a(uint32_t (&a)[D / 16][4], const uint16_t* tile, int rb, int lane) {
  constexpr int RS = D + 8;
  const int i = lane >> 3, j = lane & 7;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) ldsm_x4(a[kk], tile + (rb + (i & 1) * 8 + j) * RS + kk * 16 + (i >> 1) * 8);
}

// acc[n] (n = 0..3: tile rows nb + 8n .. as the product's n index) += a . B over the D columns,
// B[k = column][n = tile row]: rows of the tile are contiguous in k (no transpose).
template <int D>
__device__ __forceinline__ void mma_rows(float (&acc)[4][4], const uint32_t (&a)[D / 16][4], const uint16_t* tile,
                                         int nb, int lane) {
  constexpr int RS = D + 8;
  const int i = lane >> 3, j = lane & 7;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t b[4];
      ldsm_x4(b, tile + (nb + 16 * np + (i >> 1) * 8 + j) * RS + kk * 16 + (i & 1) * 8);
      mma16816(acc[2 * np], a[kk], b[0], b[1]);
      mma16816(acc[2 * np + 1], a[kk], b[2], b[3]);
    }
}

// acc[jd] (D/8 column tiles) += a . B, B[k = tile row kb + 0..15][n = column]: the tile's rows
// run along k, so the fragments are loaded transposed.
template <int D>
__device__ __forceinline__ void mma_cols(float (&acc)[D / 8][4], const uint32_t (&a)[4], const uint16_t* tile, int kb,
                                         int lane) {
  constexpr int RS = D + 8;
  const int i = lane >> 3, j = lane & 7;
#pragma unroll
  for (int dp = 0; dp < D / 16; ++dp) {
    uint32_t b[4];
    ldsm_x4_t(b, tile + (kb + (i & 1) * 8 + j) * RS + dp * 16 + (i >> 1) * 8);
    mma16816(acc[2 * dp], a, b[0], b[1]);
    mma16816(acc[2 * dp + 1], a, b[2], b[3]);
  }
}

// Two adjacent n8 C tiles (16 x 16) as the A operand of the next product.
__device__ __forceinline__ void c_to_a(uint32_t (&a)[4], const float (&v0)[4], const float (&v1)[4]) {
  a[0] = pack_bf16x2(v0[0], v0[1]);
  a[1] = pack_bf16x2(v0[2], v0[3]);
  a[2] = pack_bf16x2(v1[0], v1[1]);
  a[3] = pack_bf16x2(v1[2], v1[3]);
}

template <int D>
__host__ __device__ constexpr int tile_halves() { return kAbRows * (D + 8); }

// ---- dK and dU: a block owns keys s0 .. s0 + 63 of one (sequence, head); query tiles q0 = s0,
// s0 + 64, .. stream through shared memory (Q, dY, and the rows' log-sum-exp and Dsum).
// Dynamic shared memory: K, U, then two buffers of (Q, dY) tiles, then two of (lse, Dsum).
template <int D>
__global__ void __launch_bounds__(kAbThreads)
attn_bwd_dkv_kernel(const __nv_bfloat16* __restrict__ qkv, const __nv_bfloat16* __restrict__ dy,
                    const float* __restrict__ lse2, const float* __restrict__ dsum, __nv_bfloat16* __restrict__ dqkv,
                    int T, int H, float sl2, float rsd) {
  constexpr int TH = tile_halves<D>(), ND = D / 8;
  extern __shared__ __align__(16) uint16_t smem_ab[];
  uint16_t* sK = smem_ab;
  uint16_t* sU = sK + TH;
  uint16_t* sQ = sU + TH;                                   // [2][TH]
  uint16_t* sO = sQ + 2 * TH;                               // [2][TH]
  float* sL = reinterpret_cast<float*>(sO + 2 * TH);        // [2][64]
  float* sS = sL + 2 * kAbRows;                             // [2][64]
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int bh = blockIdx.y, b = bh / H, h = bh - b * H;
  const int C = H * D, C3 = 3 * C;
  const int s0 = blockIdx.x * kAbRows;
  const size_t base = static_cast<size_t>(b) * T;
  const __nv_bfloat16* Q = qkv + base * C3 + h * D;
  const __nv_bfloat16* dO = dy + base * C + h * D;
  const float* ls = lse2 + static_cast<size_t>(bh) * T;
  const float* dsm = dsum + static_cast<size_t>(bh) * T;

  load_tile<D>(sK, Q + C, C3, s0, T, tid);
  load_tile<D>(sU, Q + 2 * C, C3, s0, T, tid);
  load_tile<D>(sQ, Q, C3, s0, T, tid);
  load_tile<D>(sO, dO, C, s0, T, tid);
  if (tid < kAbRows) {
    const int q = s0 + tid;
    sL[tid] = q < T ? ls[q] : 0.0f;
    sS[tid] = q < T ? dsm[q] : 0.0f;
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  uint32_t kfr[D / 16][4], ufr[D / 16][4];
  frag_a<D>(kfr, sK, warp * 16, lane);
  frag_a<D>(ufr, sU, warp * 16, lane);
  float dk[ND][4], du[ND][4];
#pragma unroll
  for (int jd = 0; jd < ND; ++jd)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[jd][e] = du[jd][e] = 0.0f;
  const int ka = s0 + warp * 16 + g, kb = ka + 8;          // this lane's key rows

  int buf = 0;
  for (int q0 = s0; q0 < T; q0 += kAbRows, buf ^= 1) {
    const int nq = q0 + kAbRows;
    if (nq < T) {                                           // the next tile, into the other buffer
      load_tile<D>(sQ + (buf ^ 1) * TH, Q, C3, nq, T, tid);
      load_tile<D>(sO + (buf ^ 1) * TH, dO, C, nq, T, tid);
      if (tid < kAbRows) {
        const int q = nq + tid;
        sL[(buf ^ 1) * kAbRows + tid] = q < T ? ls[q] : 0.0f;
        sS[(buf ^ 1) * kAbRows + tid] = q < T ? dsm[q] : 0.0f;
      }
    }
    cp_async_commit();
    cp_async_wait<1>();                                     // this tile has landed
    __syncthreads();
    const uint16_t* tq = sQ + buf * TH;
    const uint16_t* to = sO + buf * TH;
    const float* tl = sL + buf * kAbRows;
    const float* ts = sS + buf * kAbRows;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {                 // 32 queries at a time
      const int qb = half * 32;
      float st[4][4], dp[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) st[n][e] = dp[n][e] = 0.0f;
      mma_rows<D>(st, kfr, tq, qb, lane);                   // S^T: keys x queries
      mma_rows<D>(dp, ufr, to, qb, lane);                   // dA^T = U dY^T
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int ql = qb + 8 * n + 2 * c + (e & 1);      // query within the tile
          const int q = q0 + ql;
          const int key = (e < 2) ? ka : kb;
          const float p = (q < T && key <= q) ? ex2_approx(st[n][e] * sl2 - tl[ql]) : 0.0f;
          st[n][e] = p;
          dp[n][e] = p * (dp[n][e] - ts[ql]);
        }
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {                      // 16 queries per k step
        uint32_t ap[4], as[4];
        c_to_a(ap, st[2 * ks], st[2 * ks + 1]);
        c_to_a(as, dp[2 * ks], dp[2 * ks + 1]);
        mma_cols<D>(du, ap, to, qb + 16 * ks, lane);        // dU += A^T dY
        mma_cols<D>(dk, as, tq, qb + 16 * ks, lane);        // dK += dS^T Q
      }
    }
    __syncthreads();                                        // the buffer is free for the tile after next
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

// ---- dQ: a block owns queries q0 .. q0 + 63 of one (sequence, head). Pass 1 streams the key
// tiles 0 .. q0 for the rows' log-sum-exp (base 2); pass 2 streams key and value tiles again for
// dS and dQ += dS K. Dynamic shared memory: Q, dY, two buffers of (K, U) tiles, Dsum.
template <int D>
__global__ void __launch_bounds__(kAbThreads)
attn_bwd_dq_kernel(const __nv_bfloat16* __restrict__ qkv, const __nv_bfloat16* __restrict__ y,
                   const __nv_bfloat16* __restrict__ dy, __nv_bfloat16* __restrict__ dqkv, float* __restrict__ lse2_out,
                   float* __restrict__ dsum_out, int T, int H, float sl2, float rsd) {
  constexpr int TH = tile_halves<D>(), ND = D / 8;
  extern __shared__ __align__(16) uint16_t smem_ab[];
  uint16_t* sQ = smem_ab;
  uint16_t* sO = sQ + TH;
  uint16_t* sK = sO + TH;                                   // [2][TH]
  uint16_t* sU = sK + 2 * TH;                               // [2][TH]
  float* sD = reinterpret_cast<float*>(sU + 2 * TH);        // [64] Dsum
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int bh = blockIdx.y, b = bh / H, h = bh - b * H;
  const int C = H * D, C3 = 3 * C;
  const int q0 = blockIdx.x * kAbRows;
  const size_t base = static_cast<size_t>(b) * T;
  const __nv_bfloat16* Q = qkv + base * C3 + h * D;
  const __nv_bfloat16* K = Q + C;
  const __nv_bfloat16* U = Q + 2 * C;
  const __nv_bfloat16* dO = dy + base * C + h * D;
  const __nv_bfloat16* O = y + base * C + h * D;

  load_tile<D>(sQ, Q, C3, q0, T, tid);
  load_tile<D>(sO, dO, C, q0, T, tid);
  load_tile<D>(sK, K, C3, 0, T, tid);                       // pass 1's first key tile
  cp_async_commit();
  {                                                         // Dsum of row tid / 2, two threads per row
    const int r = tid >> 1, hf = tid & 1;
    const int q = q0 + r;
    float acc = 0.0f;
    if (q < T) {
#pragma unroll
      for (int v = 0; v < D / 16; ++v) {
        const int col = hf * (D / 2) + v * 8;
        const uint4 a4 = *reinterpret_cast<const uint4*>(dO + static_cast<size_t>(q) * C + col);
        const uint4 o4 = *reinterpret_cast<const uint4*>(O + static_cast<size_t>(q) * C + col);
        const uint32_t aw[4] = {a4.x, a4.y, a4.z, a4.w}, ow[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 x = unpack_bf16x2(aw[k]), z = unpack_bf16x2(ow[k]);
          acc += x.x * z.x + x.y * z.y;
        }
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    if (hf == 0) sD[r] = acc;
  }
  cp_async_wait<0>();
  __syncthreads();
  uint32_t qa[D / 16][4], da[D / 16][4];
  frag_a<D>(qa, sQ, warp * 16, lane);
  frag_a<D>(da, sO, warp * 16, lane);
  const int ra = q0 + warp * 16 + g, rb = ra + 8;          // this lane's query rows
  const float dsa = sD[warp * 16 + g], dsb = sD[warp * 16 + g + 8];
  const int nkt = q0 / kAbRows + 1;                         // key tiles 0 .. q0 (the last on the diagonal)

  // pass 1: running (max, sum) of the scaled scores per row, this lane's columns
  float ma = -INFINITY, la = 0.0f, mb = -INFINITY, lb = 0.0f;
  for (int it = 0; it < nkt; ++it) {
    const int buf = it & 1, kt = it * kAbRows;
    if (it + 1 < nkt) load_tile<D>(sK + (buf ^ 1) * TH, K, C3, kt + kAbRows, T, tid);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint16_t* tk = sK + buf * TH;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      const int kb0 = half * 32;
      float st[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n) st[n][0] = st[n][1] = st[n][2] = st[n][3] = 0.0f;
      mma_rows<D>(st, qa, tk, kb0, lane);
      float xa = -INFINITY, xb = -INFINITY;
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kt + kb0 + 8 * n + 2 * c + (e & 1);
          const int row = e < 2 ? ra : rb;
          st[n][e] = (key <= row && key < T) ? st[n][e] * sl2 : -INFINITY;
          if (e < 2) xa = fmaxf(xa, st[n][e]); else xb = fmaxf(xb, st[n][e]);
        }
      if (xa > -INFINITY) {
        const float nm = fmaxf(ma, xa);
        float acc = la * ex2_approx(ma - nm);
#pragma unroll
        for (int n = 0; n < 4; ++n) acc += ex2_approx(st[n][0] - nm) + ex2_approx(st[n][1] - nm);
        la = acc;
        ma = nm;
      }
      if (xb > -INFINITY) {
        const float nm = fmaxf(mb, xb);
        float acc = lb * ex2_approx(mb - nm);
#pragma unroll
        for (int n = 0; n < 4; ++n) acc += ex2_approx(st[n][2] - nm) + ex2_approx(st[n][3] - nm);
        lb = acc;
        mb = nm;
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {                        // the quad's columns together
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

  // pass 2: dS = A * (dA - Dsum) and dQ += dS K, key tile by key tile
  float dq[ND][4];
#pragma unroll
  for (int jd = 0; jd < ND; ++jd) dq[jd][0] = dq[jd][1] = dq[jd][2] = dq[jd][3] = 0.0f;
  load_tile<D>(sK, K, C3, 0, T, tid);
  load_tile<D>(sU, U, C3, 0, T, tid);
  cp_async_commit();
  for (int it = 0; it < nkt; ++it) {
    const int buf = it & 1, kt = it * kAbRows;
    if (it + 1 < nkt) {
      load_tile<D>(sK + (buf ^ 1) * TH, K, C3, kt + kAbRows, T, tid);
      load_tile<D>(sU + (buf ^ 1) * TH, U, C3, kt + kAbRows, T, tid);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint16_t* tk = sK + buf * TH;
    const uint16_t* tu = sU + buf * TH;
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      const int kb0 = half * 32;
      float st[4][4], dp[4][4];
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) st[n][e] = dp[n][e] = 0.0f;
      mma_rows<D>(st, qa, tk, kb0, lane);
      mma_rows<D>(dp, da, tu, kb0, lane);
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kt + kb0 + 8 * n + 2 * c + (e & 1);
          const int row = e < 2 ? ra : rb;
          const float p = (key <= row && key < T) ? ex2_approx(st[n][e] * sl2 - (e < 2 ? lsa : lsb)) : 0.0f;
          dp[n][e] = p * (dp[n][e] - (e < 2 ? dsa : dsb));
        }
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint32_t as[4];
        c_to_a(as, dp[2 * ks], dp[2 * ks + 1]);
        mma_cols<D>(dq, as, tk, kb0 + 16 * ks, lane);       // dQ += dS K
      }
    }
    __syncthreads();
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

template <int D>
constexpr size_t dkv_smem() { return (6u * tile_halves<D>()) * 2u + 4u * kAbRows * 4u; }
template <int D>
constexpr size_t dq_smem() { return (6u * tile_halves<D>()) * 2u + kAbRows * 4u; }

template <int D>
cudaError_t attention_bwd_d(const __nv_bfloat16* q, const __nv_bfloat16* yy, const __nv_bfloat16* d,
                            __nv_bfloat16* o, float* lse2, float* dsum, int B, int T, int H, float sl2, float rsd,
                            cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(dq_smem<D>()));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_bwd_dkv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(dkv_smem<D>()));
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const dim3 grid((T + kAbRows - 1) / kAbRows, B * H), block(kAbThreads);
  cudaError_t e = launch_k(attn_bwd_dq_kernel<D>, grid, block, dq_smem<D>(), s, q, yy, d, o, lse2, dsum, T, H, sl2, rsd);
  if (e != cudaSuccess) return e;
  return launch_k(attn_bwd_dkv_kernel<D>, grid, block, dkv_smem<D>(), s, q, d, static_cast<const float*>(lse2),
                  static_cast<const float*>(dsum), o, T, H, sl2, rsd);
}

}  // namespace

cudaError_t launch_attention_bwd(const void* qkv, const void* y, const void* dy, void* dqkv, float* lse2, float* dsum,
                                 int B, int T, int H, int D, cudaStream_t s) {
  if (B <= 0 || T <= 0) return cudaSuccess;
  if (B * H > 65535) return cudaErrorInvalidValue;
  const float rsd = 1.0f / sqrtf(static_cast<float>(D));
  const float sl2 = rsd * 1.4426950408889634f;
  const auto* q = static_cast<const __nv_bfloat16*>(qkv);
  const auto* yy = static_cast<const __nv_bfloat16*>(y);
  const auto* d = static_cast<const __nv_bfloat16*>(dy);
  auto* o = static_cast<__nv_bfloat16*>(dqkv);
  if (D == 64) return attention_bwd_d<64>(q, yy, d, o, lse2, dsum, B, T, H, sl2, rsd, s);
  if (D == 32) return attention_bwd_d<32>(q, yy, d, o, lse2, dsum, B, T, H, sl2, rsd, s);
  return cudaErrorInvalidValue;
}

}  // namespace gptgb
