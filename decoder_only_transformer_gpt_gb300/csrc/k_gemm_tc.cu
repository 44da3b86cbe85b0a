// Persistent tcgen05 GEMM for sm_103a: out = epilogue(A[M,K] . W[N,K]^T).
//
// Used for c_attn, attention c_proj, c_fc and mlp c_proj ("第 25 章 从小 GPT 到
// GPT-2" §25.2-25.3: every projection is an nn.Linear, W stored [out, in]) and
// for the tied LM head with its cross-entropy epilogue (§25.4; "预训练一个 Mini
// GPT" 第6步).
//
// Layout: A and W are K-major bf16; TMA copies 128 x 64 (A) and BN x 64 (W)
// boxes with the 128-byte swizzle into a STAGES-deep shared-memory ring. One
// thread issues tcgen05.mma (M=128, N=BN, K=16) into one of two TMEM
// accumulators of BN fp32 columns, so the epilogue of tile i overlaps the main
// loop of tile i+1. Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer (one elected lane)
//   warp 1      TMEM allocator and MMA issuer (the whole warp runs the loop, one elected lane issues)
//   warps 2-5   epilogue: warp w reads TMEM lanes 32*(w%4).., one output row per thread
#include "common.cuh"
#include "kernels.h"
#include "launch.h"

#include <math.h>

namespace gptgb {

namespace {

constexpr int BM = kGemmBM;
constexpr int BK = kGemmBK;
constexpr int BN = 256;
constexpr int MAX_STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;              // 16 KB
constexpr int B_BYTES = BN * BK * 2;              // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;                 // 512: two accumulators
constexpr int THREADS = 192;
constexpr int EPI_WARPS = 4;
constexpr int EPI_BUF = kEpiRows * 128;            // one warp's 32-row x 128-byte staging box
constexpr int EPI_NBUF = 1;                        // staging boxes per warp

// Shared-memory layout per epilogue kind: the TMA-store epilogues add a staging
// box per epilogue warp and a copy of the tile's bias.
template <int EPI>
struct Layout {
  static constexpr bool kTmaOut =
      (EPI == EPI_BIAS_OUT || EPI == EPI_BIAS_GELU_OUT || EPI == EPI_BIAS_RESID || EPI == EPI_CE_GRAD ||
       EPI == EPI_F32_OUT || EPI == EPI_GELU_GRAD || EPI == EPI_BIAS_GELU_UOUT);
  static constexpr int STAGES = 4;
  static constexpr int STAGING = STAGES * STAGE_BYTES;
  static constexpr int BIAS = STAGING + (kTmaOut ? EPI_WARPS * EPI_NBUF * EPI_BUF : 0);   // each warp's copy of the tile's bias
  static constexpr int BAR = BIAS + (kTmaOut ? EPI_WARPS * BN * 4 : 0);
  static constexpr int SMEM = BAR + 256 + 1024;      // + barriers + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(STAGES <= MAX_STAGES, "barrier arrays");
};
constexpr float kLog2e = 1.4426950408889634f;
__device__ constexpr float kLog2eDev = 1.4426950408889634f;

struct __align__(8) Bars {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// Fetch the 128-byte line holding p into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

__device__ __forceinline__ void tile_coords(int tile, int MB, int NB, int m_fastest, int& mb, int& nb) {
  if (m_fastest) { mb = tile % MB; nb = tile / MB; }
  else           { nb = tile % NB; mb = tile / NB; }
}


// GELU, tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), evaluated as
// u = x (c0 + c1 x^2), h = x / 2, h + h tanh(u): five ALU instructions and one
// tanh (the ALU count matters: it runs beside the tensor core's main loop).
__device__ __forceinline__ float gelu_f(float x, int erf_form) {
  if (erf_form) return 0.5f * x * (1.0f + erff(x * 0.70710678118654752f));
  constexpr float c0 = 0.7978845608028654f;             // sqrt(2/pi)
  constexpr float c1 = 0.7978845608028654f * 0.044715f;
  const float u = x * fmaf(x * x, c1, c0);
  const float h = 0.5f * x;
  return fmaf(h, tanh_approx(u), h);
}

// ---------------------------------------------------------------- epilogues

template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const GemmArgs& a, const uint32_t* r, int grow, int n0) {
  const bool full = (n0 + 32 <= a.N);
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
  if (a.bias != nullptr) {
    if (full) {
      const float4* b4 = reinterpret_cast<const float4*>(a.bias + n0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 bb = __ldg(b4 + q);
        v[4 * q + 0] += bb.x; v[4 * q + 1] += bb.y; v[4 * q + 2] += bb.z; v[4 * q + 3] += bb.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] += (n0 + i < a.N) ? __ldg(a.bias + n0 + i) : 0.0f;
    }
  }
  if (EPI == EPI_BIAS_GELU_OUT) {
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = gelu_f(v[i], a.gelu_erf);
  }
  if (EPI == EPI_BIAS_OUT || EPI == EPI_BIAS_GELU_OUT) {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.out) + (size_t)grow * a.ldo + n0;
    if (full) {
      uint4* o4 = reinterpret_cast<uint4*>(o);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
        w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
        w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
        w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
        o4[q] = w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n0 + i < a.N) o[i] = __float2bfloat16_rn(v[i]);
    }
  } else if (EPI == EPI_BIAS_RESID) {
    float* o = reinterpret_cast<float*>(a.out) + (size_t)grow * a.ldo + n0;
    if (full) {
      float4* o4 = reinterpret_cast<float4*>(o);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 x = o4[q];
        x.x += v[4 * q + 0]; x.y += v[4 * q + 1]; x.z += v[4 * q + 2]; x.w += v[4 * q + 3];
        o4[q] = x;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n0 + i < a.N) o[i] += v[i];
    }
  } else if (EPI == EPI_F32) {
    float* o = reinterpret_cast<float*>(a.out) + (size_t)grow * a.ldo + n0;
    if (full) {
      float4* o4 = reinterpret_cast<float4*>(o);
#pragma unroll
      for (int q = 0; q < 8; ++q) o4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n0 + i < a.N) o[i] = v[i];
    }
  }
}

// Fold 32 logits (-inf for none) into a row's (reference m, sum s of exp(z - m)) against
// the exact maximum of the chunk and m; m = -inf with s = 0 before the first.
constexpr float kCeChunkSumLimit = 18446744073709551616.0f;    // 2^64
__device__ __forceinline__ float ce_fold_exact(const float (&z)[32], float& m, float s) {
  float c4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
  for (int i = 0; i < 32; i += 8)
#pragma unroll
    for (int k = 0; k < 4; ++k) c4[k] = fmax3(c4[k], z[i + 2 * k], z[i + 2 * k + 1]);
  const float cm = fmaxf(fmaxf(c4[0], c4[1]), fmaxf(c4[2], c4[3]));
  if (cm == -INFINITY) return s;
  const float nm = fmaxf(m, cm);
  const float nml = nm * kLog2e;
  const float2 l2e = make_float2(kLog2e, kLog2e), nm2 = make_float2(-nml, -nml);
  float2 acc2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 x = fma2_rn(make_float2(z[i], z[i + 1]), l2e, nm2);
    acc2[(i >> 1) & 1] = add2_rn(acc2[(i >> 1) & 1], make_float2(ex2_approx(x.x), ex2_approx(x.y)));
  }
  const float2 a2 = add2_rn(acc2[0], acc2[1]);
  const float out = s * ex2_approx((m - nm) * kLog2e) + (a2.x + a2.y);   // m = -inf: scale 0
  m = nm;
  return out;
}

// Cross-entropy epilogue for one 32-column chunk: fold the chunk into the
// row's running (reference m, sum s of exp(z - m)) for this tile, capture the
// target's logit, and store logits if asked.
__device__ __forceinline__ void ce_chunk(const GemmArgs& a, const uint32_t* r, int grow, int n0, int tgt,
                                         float& m, float& s) {
  float z[32];
  const bool whole = n0 + 32 <= a.N;                 // warp-uniform: only the last tile is ragged
  if (whole) {
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = __uint_as_float(r[i]);
    // s = sum exp(z - m) needs m only as a reference, not the maximum: a row's first logit
    // of the tile starts it, and a chunk is summed against the current reference in one
    // pass; only a chunk whose sum passes 2^64 (or overflows) is redone below against its max.
    if (m == -INFINITY) m = z[0];
    const float nml = m * kLog2e;
    const float2 l2e = make_float2(kLog2e, kLog2e), nm2 = make_float2(-nml, -nml);
    float2 acc2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      const float2 x = fma2_rn(make_float2(z[i], z[i + 1]), l2e, nm2);
      acc2[(i >> 1) & 1] = add2_rn(acc2[(i >> 1) & 1], make_float2(ex2_approx(x.x), ex2_approx(x.y)));
    }
    const float2 a2 = add2_rn(acc2[0], acc2[1]);
    const float cs = a2.x + a2.y;
    if (cs <= kCeChunkSumLimit) {
      s += cs;
    } else {
      s = ce_fold_exact(z, m, s);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = (n0 + i < a.N) ? __uint_as_float(r[i]) : -INFINITY;
    s = ce_fold_exact(z, m, s);
  }
  if (static_cast<unsigned>(tgt - n0) < 32u) {
    float zt = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i == tgt - n0) zt = z[i];
    a.ztgt[grow] = zt;
  }
  if (a.logits != nullptr) {
    float* o = a.logits + (size_t)grow * a.ldo + n0;
    if (n0 + 32 <= a.N && (a.ldo & 3) == 0) {
      float4* o4 = reinterpret_cast<float4*>(o);
#pragma unroll
      for (int q = 0; q < 8; ++q) o4[q] = make_float4(z[4 * q], z[4 * q + 1], z[4 * q + 2], z[4 * q + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (n0 + i < a.N) o[i] = z[i];
    }
  }
}

// One warp's 32 x 128-byte chunk into its staging box: row = lane, 16-byte unit u
// of the row at position u ^ (row & 7) (the 128-byte swizzle the TMA store reads).
__device__ __forceinline__ void stage_row(uint8_t* buf, int lane, const uint32_t (&w)[32]) {
  uint8_t* row = buf + lane * 128;
#pragma unroll
  for (int u = 0; u < 8; ++u)
    *reinterpret_cast<uint4*>(row + ((u ^ (lane & 7)) << 4)) = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
}

// Bias (+ GELU) of CW consecutive columns, packed for the store: bf16 pairs when
// CW == 64, fp32 bits when CW == 32. sbias: the chunk's bias in shared memory
// (zeros past N), or nullptr.
template <int EPI, int CW>
__device__ __forceinline__ void finish_chunk(const GemmArgs& a, const uint32_t* r, const float* sbias,
                                             uint32_t (&w)[32]) {
  // element pairs go through the packed f32x2 instructions
  float2 v2[CW / 2];
#pragma unroll
  for (int i = 0; i < CW / 2; ++i) v2[i] = make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
  if (sbias != nullptr) {
    const float4* b4 = reinterpret_cast<const float4*>(sbias);     // same address in every lane: broadcast
#pragma unroll
    for (int q = 0; q < CW / 4; ++q) {
      const float4 bb = b4[q];
      v2[2 * q] = add2_rn(v2[2 * q], make_float2(bb.x, bb.y));
      v2[2 * q + 1] = add2_rn(v2[2 * q + 1], make_float2(bb.z, bb.w));
    }
  }
  if (EPI == EPI_BIAS_GELU_OUT) {
    if (a.gelu_erf) {
#pragma unroll
      for (int i = 0; i < CW / 2; ++i) v2[i] = make_float2(gelu_f(v2[i].x, 1), gelu_f(v2[i].y, 1));
    } else {
      // 0.5 x (1 + tanh(u)), u = sqrt(2/pi) (x + 0.044715 x^3), as h + h tanh(u) with h = x / 2
      constexpr float c0 = 0.7978845608028654f;
      constexpr float c1 = 0.7978845608028654f * 0.044715f;
      const float2 c0v = make_float2(c0, c0), c1v = make_float2(c1, c1), half = make_float2(0.5f, 0.5f);
#pragma unroll
      for (int i = 0; i < CW / 2; ++i) {
        const float2 x = v2[i];
        const float2 u = mul2_rn(x, fma2_rn(mul2_rn(x, x), c1v, c0v));
        const float2 h = mul2_rn(x, half);
        v2[i] = fma2_rn(h, make_float2(tanh_approx(u.x), tanh_approx(u.y)), h);
      }
    }
  }
  float v[CW];
#pragma unroll
  for (int i = 0; i < CW / 2; ++i) {
    v[2 * i] = v2[i].x;
    v[2 * i + 1] = v2[i].y;
  }
  if (CW == 64) {
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(v[2 * i], v[(2 * i + 1) % CW]);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i % CW]);
  }
}

// Cross-entropy gradient of 64 consecutive logits of one row, packed as bf16 pairs:
// (exp(z - lse) - [column == tcol]) * scale, tcol the target's column within the chunk
// (outside [0, 64) when the target is elsewhere). z <= lse, so every exponential is <= 1.
__device__ __forceinline__ void ce_grad_chunk(const uint32_t* r, float lse, int tcol, float scale, uint32_t (&w)[32]) {
  const float l2 = lse * kLog2eDev;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float p0 = ex2_approx(fmaf(__uint_as_float(r[2 * i]), kLog2eDev, -l2));
    float p1 = ex2_approx(fmaf(__uint_as_float(r[2 * i + 1]), kLog2eDev, -l2));
    if (2 * i == tcol) p0 -= 1.0f;
    if (2 * i + 1 == tcol) p1 -= 1.0f;
    w[i] = pack_bf16x2(p0 * scale, p1 * scale);
  }
}

// 64 consecutive columns of one row times GELU's derivative at u (the row's 64 bf16 inputs at
// urow, or fewer when the chunk passes N), packed as bf16 pairs. tanh form:
// gelu' = 0.5 (1 + t) + 0.5 x (1 - t^2) c (1 + 3 * 0.044715 x^2), t = tanh(c (x + 0.044715 x^3));
// erf form: Phi(x) + x phi(x).
__device__ __forceinline__ void gelu_grad_chunk(const uint32_t* r, const __nv_bfloat16* urow, int nvalid, int erf_form,
                                                uint32_t (&w)[32]) {
  uint32_t uw[32];
  if (nvalid >= 64) {
    const uint4* u4 = reinterpret_cast<const uint4*>(urow);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint4 v = __ldg(u4 + q);
      uw[4 * q] = v.x; uw[4 * q + 1] = v.y; uw[4 * q + 2] = v.z; uw[4 * q + 3] = v.w;
    }
  } else {
    const uint16_t* u16 = reinterpret_cast<const uint16_t*>(urow);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t lo = (2 * i < nvalid) ? u16[2 * i] : 0u, hi = (2 * i + 1 < nvalid) ? u16[2 * i + 1] : 0u;
      uw[i] = lo | (hi << 16);
    }
  }
  constexpr float c0 = 0.7978845608028654f;
  if (erf_form) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float2 x = unpack_bf16x2(uw[i]);
      float d[2];
      const float xs[2] = {x.x, x.y};
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float xv = xs[e];
        d[e] = 0.5f * (1.0f + erff(xv * 0.70710678118654752f)) + xv * 0.39894228040143268f * __expf(-0.5f * xv * xv);
      }
      w[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * d[0], __uint_as_float(r[2 * i + 1]) * d[1]);
    }
    return;
  }
  // tanh form, on element pairs with the packed f32x2 instructions:
  // gelu'(x) = (1 + t) / 2 + (x / 2) (1 - t^2) c0 (1 + 3 * 0.044715 x^2), t = tanh(c0 x (1 + 0.044715 x^2))
  const float2 one = make_float2(1.0f, 1.0f), half = make_float2(0.5f, 0.5f), mone = make_float2(-1.0f, -1.0f);
  const float2 k1 = make_float2(0.044715f, 0.044715f), k3 = make_float2(3.0f * 0.044715f, 3.0f * 0.044715f);
  const float2 c0v = make_float2(c0, c0), hc0 = make_float2(0.5f * c0, 0.5f * c0);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float2 x = unpack_bf16x2(uw[i]);
    const float2 x2 = mul2_rn(x, x);
    const float2 arg = mul2_rn(mul2_rn(x, c0v), fma2_rn(x2, k1, one));
    const float2 t = make_float2(tanh_approx(arg.x), tanh_approx(arg.y));
    const float2 omt2 = fma2_rn(mul2_rn(t, mone), t, one);                       // 1 - t^2
    const float2 b = mul2_rn(mul2_rn(x, hc0), mul2_rn(omt2, fma2_rn(x2, k3, one)));
    const float2 d = add2_rn(fma2_rn(t, half, half), b);
    const float2 o = mul2_rn(make_float2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), d);
    w[i] = pack_bf16x2(o.x, o.y);
  }
}

// ---------------------------------------------------------------- work list

// A CTA's work as a sequence of segments (tile, K blocks [kb0, kb1)).
//
// Whole tiles: tiles blockIdx.x, blockIdx.x + gridDim.x, ...
//
// Stream-K (tiles not a whole number of waves): the first S tiles, S = one wave
// plus the remainder, form a region whose tiles x KB (tile, K block) units are
// dealt in equal contiguous shares, one per CTA; each share is at least KB units,
// so a tile is split between at most two CTAs: the one holding its first K blocks
// (a prefix: the CTA's last segment of the region) and the next CTA (a suffix:
// its first segment). The remaining tiles are whole waves, dealt as above. The
// region comes first so that a split tile's fixup overlaps later whole tiles, and
// it is a small contiguous range of tiles so that co-running CTAs share operands
// in L2.
struct SegIter {
  int KB;
  long long k, kend;          // stream-K units still to deal
  int t, stride, count;       // whole tiles (or split-K units) still to deal
  int ksplit;
  template <bool KS>
  __device__ __forceinline__ bool next(int& tile, int& kb0, int& kb1) {
    if (k < kend) {
      tile = static_cast<int>(k / KB);
      kb0 = static_cast<int>(k - static_cast<long long>(tile) * KB);
      const long long left = kend - k;
      kb1 = (KB - kb0 < left) ? KB : kb0 + static_cast<int>(left);
      k += kb1 - kb0;
      return true;
    }
    if (t >= count) return false;
    if (KS) {
      tile = t / ksplit;
      const int sl = t - tile * ksplit;
      kb0 = static_cast<int>(static_cast<long long>(sl) * KB / ksplit);
      kb1 = static_cast<int>(static_cast<long long>(sl + 1) * KB / ksplit);
    } else {
      tile = t;
      kb0 = 0;
      kb1 = KB;
    }
    t += stride;
    return true;
  }
};

// The work of worker `idx` of G (a CTA, or a CTA pair).
__device__ __forceinline__ SegIter make_seg_iter_of(bool sk, bool ks, int num_tiles, int KB, int ksplit, int G, int idx) {
  const int S = !sk ? 0 : (num_tiles >= 2 * G ? G + num_tiles % G : num_tiles);
  SegIter it;
  it.KB = KB;
  const long long units = static_cast<long long>(S) * KB;
  it.k = units * idx / G;
  it.kend = units * (idx + 1) / G;
  it.t = S + idx;
  it.stride = G;
  it.ksplit = (ks && ksplit > 1) ? ksplit : 1;
  it.count = num_tiles * it.ksplit;
  return it;
}

__device__ __forceinline__ SegIter make_seg_iter(bool sk, bool ks, int num_tiles, int KB, int ksplit) {
  return make_seg_iter_of(sk, ks, num_tiles, KB, ksplit, gridDim.x, blockIdx.x);
}

// ---------------------------------------------------------------- kernel

// MODE 0: whole tiles; 1: stream-K (tiles split between CTAs, partials fixed up);
// 2: split-K (units of (tile, K slice) added with reduce-add stores). Each mode is
// its own instantiation, so whole-tile launches carry no segment bookkeeping.
// (The stream-K notes below say SK for MODE == 1.) Whole-tile launches use their
// own instantiation, whose loops have no segment bookkeeping.
// MN: both operands MN-major (A stored [K][M], W stored [K][N], M and N contiguous): a stage
// holds BM/64 (A) and BN/64 (W) boxes of 64 (M or N) x 64 (K) at 8 KB strides, the MMA reads
// them with the MN-major 128-byte-swizzle layout (64-element atoms 8 KB apart, 8-row K groups
// 1 KB apart), and a K step of 16 advances 16 rows (2 KB).
template <int EPI, int MODE, bool MN = false>
__global__ void __launch_bounds__(THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2,
               const GemmArgs args) {
  using LY = Layout<EPI>;
  constexpr int STAGES = LY::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* sE = smem + LY::STAGING;
  float* sBias = reinterpret_cast<float*>(smem + LY::BIAS);
  Bars* bars = reinterpret_cast<Bars*>(smem + LY::BAR);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int MB = (args.M + BM - 1) / BM;
  const int NB = (args.N + BN - 1) / BN;
  const int KB = (args.K + BK - 1) / BK;
  const int num_tiles = MB * NB;
  constexpr bool SK = MODE == 1, KS = MODE == 2;
  constexpr bool sk = SK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) { mbar_init(&bars->full[s], 1); mbar_init(&bars->empty[s], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&bars->tfull[i], 1); mbar_init(&bars->tempty[i], 4); }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  constexpr bool kTmaOut = LY::kTmaOut;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (kTmaOut) tma_prefetch_desc(&tmC);
    if (EPI == EPI_BIAS_GELU_UOUT) tma_prefetch_desc(&tmC2);
  }
  if (warp == 1) tmem_alloc(&bars->tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  pdl_trigger();                    // the next kernel may begin its prologue

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_par = 0;
      bool ok = true;
      auto load_a = [&](int st, int kb, int mb) {
        if (MN) {
#pragma unroll
          for (int i = 0; i < BM / 64; ++i)
            tma_load_2d(sA + st * A_BYTES + i * 8192, &tmA, &bars->full[st], mb * BM + 64 * i, kb * BK);
        } else {
          tma_load_2d(sA + st * A_BYTES, &tmA, &bars->full[st], kb * BK, mb * BM);
        }
      };
      auto load_b = [&](int st, int kb, int nb) {
        if (MN) {
#pragma unroll
          for (int i = 0; i < BN / 64; ++i)
            tma_load_2d(sB + st * B_BYTES + i * 8192, &tmB, &bars->full[st], nb * BN + 64 * i, kb * BK);
        } else {
          tma_load_2d(sB + st * B_BYTES, &tmB, &bars->full[st], kb * BK, nb * BN);
        }
      };
      // Weights (B, when b_const) do not depend on the previous kernel: the first tile's
      // first stages of B are requested before waiting for that kernel to finish.
      int pre = 0;
      SegIter it = make_seg_iter(sk, KS, num_tiles, KB, args.ksplit);
      if (args.b_const) {
        SegIter it0 = it;
        int tile0, kb00, kb10;
        if (it0.template next<KS>(tile0, kb00, kb10)) {
          int mb0, nb0;
          tile_coords(tile0, MB, NB, args.m_fastest, mb0, nb0);
          pre = (kb10 - kb00) < STAGES ? (kb10 - kb00) : STAGES;
          for (int i = 0; i < pre; ++i) {
            mbar_arrive_expect_tx(&bars->full[i], STAGE_BYTES);
            load_b(i, kb00 + i, nb0);
          }
        }
      }
      pdl_wait();                     // A, written by the previous kernel, is now visible
      int tile, kb0, kb1;
      while (ok && it.template next<KS>(tile, kb0, kb1)) {
        int mb, nb;
        tile_coords(tile, MB, NB, args.m_fastest, mb, nb);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (pre > 0) {                // stage armed and its B requested above
            --pre;
            load_a(stage, kb, mb);
          } else {
            if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, args.err)) { ok = false; break; }
            mbar_arrive_expect_tx(&bars->full[stage], STAGE_BYTES);
            load_a(stage, kb, mb);
            load_b(stage, kb, nb);
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // never leave with copies in flight into this CTA's shared memory
      for (int s = 0; s < STAGES; ++s)
        if (issued & (1u << s)) mbar_wait_drain(&bars->full[s], (last_par >> s) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (whole warp; one elected lane issues)
    {
      const uint32_t idesc = idesc_bf16_f32(BM, BN, MN) | (MN ? (1u << 15) : 0u);   // bit 15: A MN-major
      // base descriptors of stage 0 (K-major: 8-row groups 1024 bytes apart; MN-major: 64-element
      // atoms 8 KB apart, 8-row K groups 1024 bytes apart; 128-byte swizzle); the start address
      // is the low field, so other stages and K steps are plain adds
      const uint64_t da0 = smem_desc(smem_u32(sA), MN ? 8192 : 16, 1024, SWZ_128B);
      const uint64_t db0 = smem_desc(smem_u32(sB), MN ? 8192 : 16, 1024, SWZ_128B);
      constexpr uint64_t kstep = MN ? (16 * 128) >> 4 : 2;    // one K step of 16, in 16-byte units
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      SegIter it = make_seg_iter(sk, KS, num_tiles, KB, args.ksplit);
      int tile, kb0, kb1;
      while (ok && it.template next<KS>(tile, kb0, kb1)) {
        if (!mbar_wait_warp(&bars->tempty[acc], acc_phase ^ 1u, abort_flag, args.err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_warp(&bars->full[stage], phase, abort_flag, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint64_t da = da0 + static_cast<uint64_t>((stage * A_BYTES) >> 4);
          const uint64_t db = db0 + static_cast<uint64_t>((stage * B_BYTES) >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma_bf16_warp(d_tmem, da + kstep * k, db + kstep * k, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
          tc_commit_warp(&bars->empty[stage]);           // frees the stage once these MMAs finish
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit_warp(&bars->tfull[acc]);               // accumulator ready for the epilogue
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      tc_commit_warp(&bars->drain);                      // all issued MMAs have completed after this
      mbar_wait_drain(&bars->drain, 0);
    }
  } else {
    // ------------------------------------------------ epilogue warps
    const int sub = warp & 3;
    const int row = sub * 32 + lane;
    uint8_t* my_stage = sE + sub * EPI_NBUF * EPI_BUF;
    float* my_bias = sBias + sub * BN;
    uint32_t n_staged = 0;                           // chunks this warp has staged (buffer ring position)
    pdl_wait();                                      // outputs may be read-modified-written below
    int acc = 0;
    uint32_t acc_phase = 0;
    SegIter it = make_seg_iter(sk, KS, num_tiles, KB, args.ksplit);
    int tile, kb0, kb1;
    while (it.template next<KS>(tile, kb0, kb1)) {
      int mb, nb;
      tile_coords(tile, MB, NB, args.m_fastest, mb, nb);
      // stream-K: a suffix (kb0 > 0) hands its fp32 partial to the CTA before, in
      // slot blockIdx.x; a prefix (kb1 < KB) takes the next CTA's from slot blockIdx.x + 1
      const bool writer = kb0 > 0;
      const bool owner = kb0 == 0 && kb1 < KB;
      if (kTmaOut && args.bias != nullptr && !writer) {
        // this tile's BN bias values into the warp's shared copy, while the main loop runs
        const int nbase = nb * BN + lane * (BN / 32);
#pragma unroll
        for (int i = 0; i < BN / 32; ++i)
          my_bias[lane * (BN / 32) + i] = (nbase + i < args.N) ? __ldg(args.bias + nbase + i) : 0.0f;
        __syncwarp();
      }
      if (EPI == EPI_GELU_GRAD && mb * BM + row < args.M) {
        // this row's GELU inputs for the tile into L2 while the tile's main loop runs: the chunks
        // below then wait on L2, not on DRAM, for them
        const __nv_bfloat16* urow = static_cast<const __nv_bfloat16*>(args.aux) + static_cast<size_t>(mb * BM + row) * args.N;
#pragma unroll
        for (int q = 0; q < BN / 64; ++q)
          if (nb * BN + q * 64 < args.N) prefetch_l2(urow + nb * BN + q * 64);
      }
      if (!mbar_wait(&bars->tfull[acc], acc_phase, abort_flag, args.err)) break;
      tc_fence_after();
      const int grow = mb * BM + row;
      const bool row_ok = grow < args.M;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if (SK && kTmaOut && writer) {
        // this warp's 32 rows of the partial tile, then its flag. Layout of a slot:
        // [warp][64-column chunk][float4 q][lane], so that each store (and the
        // owner's matching load) covers 512 contiguous bytes
        float4* pw = reinterpret_cast<float4*>(args.sk_part) + ((size_t)blockIdx.x * 4 + sub) * (BN / 64) * 16 * 32 + lane;
#pragma unroll 1
        for (int c2 = 0; c2 < BN / 64; ++c2) {
          uint32_t r[64];
          tmem_ld_32x32b_x64(tbase + c2 * 64, r);
          tmem_ld_wait();
          if (c2 == BN / 64 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->tempty[acc]);
          }
#pragma unroll
          for (int q = 0; q < 16; ++q)
            pw[(c2 * 16 + q) * 32] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]), __uint_as_float(r[4 * q + 2]),
                                 __uint_as_float(r[4 * q + 3]));
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(args.sk_flag + blockIdx.x * 4 + sub, 1);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
        continue;
      }
      const float4* ppart = nullptr;                  // owner: the other CTA's partial rows
      if (SK && kTmaOut && owner) {
        // wait (bounded) for the writer's flag, then clear it for the next launch
        const int fi = (blockIdx.x + 1) * 4 + sub;
        int* flag = args.sk_wait_flag != nullptr ? const_cast<int*>(args.sk_wait_flag) + fi : args.sk_flag + fi;
        const long long limit = args.wait_limit > 0 ? args.wait_limit : kWaitLimitCycles;
        bool seen = ld_acquire_gpu(flag) != 0;
        if (!seen) {
          const long long t0 = clock64();
          while (!(seen = (ld_acquire_gpu(flag) != 0))) {
            if (*abort_flag || clock64() - t0 > limit) break;
          }
        }
        if (!__all_sync(0xffffffffu, seen)) {
          if (lane == 0) { record_error(args.err, GPT_DEV_ETIMEOUT); *abort_flag = 1; }
        } else if (lane == 0) {
          *flag = 0;
        }
        ppart = reinterpret_cast<const float4*>(args.sk_part) + ((size_t)(blockIdx.x + 1) * 4 + sub) * (BN / 64) * 16 * 32 + lane;
      }
      // the accumulator is read 64 columns per tcgen05.ld (see tmem_ld_32x32b_x64)
      if (EPI == EPI_CE) {
        const int tgt = row_ok ? __ldg(args.targets + grow) : -1;
        float m = -INFINITY, s = 0.0f;
#pragma unroll 1
        for (int c2 = 0; c2 < BN / 64; ++c2) {
          uint32_t r[64];
          tmem_ld_32x32b_x64(tbase + c2 * 64, r);
          tmem_ld_wait();
          if (c2 == BN / 64 - 1) {                    // accumulator fully read: hand it back early
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->tempty[acc]);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int n0 = nb * BN + c2 * 64 + h * 32;
            if (row_ok && n0 < args.N) ce_chunk(args, r + h * 32, grow, n0, tgt, m, s);
          }
        }
        if (row_ok) {
          args.pmax[(size_t)nb * args.M + grow] = m;
          args.psum[(size_t)nb * args.M + grow] = s;
        }
      } else if (kTmaOut) {
        constexpr int CW = (EPI == EPI_BIAS_RESID || EPI == EPI_F32_OUT) ? 32 : 64;   // columns per 128-byte row
        const int m0 = mb * BM + sub * 32;
        float row_lse = 0.0f;
        int row_tgt = -1;
        if (EPI == EPI_CE_GRAD && row_ok) {
          row_lse = __ldg(args.row_nll + grow) + __ldg(args.ztgt + grow);
          row_tgt = __ldg(args.targets + grow);
        }
#pragma unroll 1
        for (int c2 = 0; c2 < BN / 64; ++c2) {
          uint32_t r[64];
          tmem_ld_32x32b_x64(tbase + c2 * 64, r);
          tmem_ld_wait();
          if (c2 == BN / 64 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->tempty[acc]);
          }
          if (SK && ppart != nullptr) {               // finish a split tile: + the suffix's K blocks
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float4 p4 = ppart[(c2 * 16 + q) * 32];
              r[4 * q + 0] = __float_as_uint(__uint_as_float(r[4 * q + 0]) + p4.x);
              r[4 * q + 1] = __float_as_uint(__uint_as_float(r[4 * q + 1]) + p4.y);
              r[4 * q + 2] = __float_as_uint(__uint_as_float(r[4 * q + 2]) + p4.z);
              r[4 * q + 3] = __float_as_uint(__uint_as_float(r[4 * q + 3]) + p4.w);
            }
          }
#pragma unroll
          for (int h = 0; h < 64 / CW; ++h) {
            const int c = c2 * (64 / CW) + h;            // chunk of CW columns within the tile
            const int n0 = nb * BN + c * CW;
            if (n0 >= args.N) continue;                  // the whole chunk is past N (warp-uniform)
            uint32_t w[32];
            // the chunk through the warp's staging box to the map (a TMA store, or the reduce-add into x)
            auto stage_store = [&](const CUtensorMap* map) {
              uint8_t* buf = my_stage + (n_staged % EPI_NBUF) * EPI_BUF;
              ++n_staged;
              if (lane == 0) bulk_wait_read<EPI_NBUF - 1>();   // the store that last used this box has read it
              __syncwarp();
              stage_row(buf, lane, w);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                if (EPI == EPI_BIAS_RESID) tma_reduce_add_2d(map, buf, n0, m0);   // x += tile, in L2
                else tma_store_2d(map, buf, n0, m0);
                bulk_commit();
              }
            };
            if (EPI == EPI_CE_GRAD) {
              ce_grad_chunk(r + h * CW, row_lse, row_tgt - n0, args.scale, w);
            } else if (EPI == EPI_GELU_GRAD) {
              gelu_grad_chunk(r + h * CW,
                              static_cast<const __nv_bfloat16*>(args.aux) + static_cast<size_t>(row_ok ? grow : 0) * args.N + n0,
                              row_ok ? args.N - n0 : 0, args.gelu_erf, w);
            } else if (EPI == EPI_BIAS_GELU_UOUT) {          // u = acc + bias first, then gelu(u)
              finish_chunk<EPI_BIAS_OUT, CW>(args, r + h * CW, args.bias != nullptr ? my_bias + c * CW : nullptr, w);
              stage_store(&tmC2);
              finish_chunk<EPI_BIAS_GELU_OUT, CW>(args, r + h * CW, args.bias != nullptr ? my_bias + c * CW : nullptr, w);
            } else {
              finish_chunk<EPI, CW>(args, r + h * CW, args.bias != nullptr ? my_bias + c * CW : nullptr, w);
            }
            stage_store(&tmC);
          }
        }
      } else {
#pragma unroll 1
        for (int c2 = 0; c2 < BN / 64; ++c2) {
          uint32_t r[64];
          tmem_ld_32x32b_x64(tbase + c2 * 64, r);
          tmem_ld_wait();
          if (c2 == BN / 64 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->tempty[acc]);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int n0 = nb * BN + c2 * 64 + h * 32;
            if (row_ok && n0 < args.N) epilogue_chunk<EPI>(args, r + h * 32, grow, n0);
          }
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (kTmaOut && lane == 0) bulk_wait_all();        // stores complete before the CTA exits
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- CTA-pair kernel (cta_group::2)

// The products with a tensor-store epilogue (EPI_BIAS_RESID: x += A W^T + bias; EPI_F32_OUT: out = A W^T
// + bias; EPI_BIAS_OUT, EPI_BIAS_GELU_OUT: bf16 out) on a pair of CTAs in a cluster of two:
// one tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16), issued by the even CTA, reads the pair's
// 256 A rows from both CTAs' shared memory (128 each) and the 256 W rows likewise (128 each), and
// leaves rows 0-127 of the 256 x 256 accumulator in the even CTA's TMEM and rows 128-255 in the odd
// one's. Each CTA therefore stages 32 KB per K block instead of 48 KB (A 16 KB and half of W), and
// the same shared memory holds a six-stage ring (2 us of MMA work at the measured peak) instead of
// four. Each CTA's TMA copies land in its own shared memory and count towards the even CTA's "full"
// barrier; the even CTA's commits arrive on both CTAs' barriers at once (multicast). Warp roles as
// in gemm_tc_kernel; the odd CTA's warp 1 only allocates and frees TMEM.
constexpr int P_MAX_STAGES = 6;
constexpr int P_A_BYTES = BM * BK * 2;            // this CTA's 128 of the pair's 256 A rows
constexpr int P_B_BYTES = (BN / 2) * BK * 2;      // this CTA's 128 of the tile's 256 W rows
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
// EW epilogue warps per CTA: 4 (one per TMEM lane quarter, all 256 columns each; six stages) or 8 (two
// per lane quarter, 128 columns each, for the GELU epilogue whose arithmetic bounds a tile; their staging
// boxes leave room for five stages).
template <int EW>
struct PairCfg {
  static constexpr int THREADS = 64 + 32 * EW;
  static constexpr int STAGES = EW == 4 ? 6 : 5;
  static constexpr int CHUNKS = (BN / 64) * 4 / EW;   // 64-column chunks per epilogue warp
  static constexpr int STAGING = STAGES * P_STAGE_BYTES;
  static constexpr int BIAS = STAGING + EW * EPI_BUF;
  static constexpr int BAR = BIAS + EW * BN * 4;
  static constexpr int SMEM = BAR + 256 + 1024;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(STAGES <= P_MAX_STAGES, "barrier arrays");
};

struct __align__(8) PairBars {
  uint64_t full[P_MAX_STAGES];    // even CTA: both CTAs' copies of the stage have landed (2 x 32 KB)
  uint64_t empty[P_MAX_STAGES];   // each CTA: the pair's MMAs have read its copy of the stage
  uint64_t tfull[2];          // each CTA: its half of the accumulator is complete
  uint64_t tempty[2];         // even CTA: both CTAs' epilogue warps (2 EW) have read the accumulator
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(PairBars) <= 256, "barrier block");

__device__ __forceinline__ uint32_t cluster_cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of the variable at shared::cta address `saddr` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t saddr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
  return d;
}

// Every thread of both CTAs: release this CTA's earlier writes, wait for the other CTA's.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(cluster_bar) : "memory");
}

// A tiled copy into this CTA's shared memory whose bytes count towards a barrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t cluster_bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];"
      :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(c0), "r"(c1)
      : "memory");
}

// TMEM allocation for the pair: one warp of each CTA executes it (the whole warp).
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

// The pair's MMA, issued by one elected lane of the even CTA's converged warp.
__device__ __forceinline__ void tc_mma_pair_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

// One arrival on the barrier at this shared-memory offset in both CTAs once the pair's earlier MMAs
// have completed.
__device__ __forceinline__ void tc_commit_pair_both_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}\n"
      :: "r"(smem_u32(bar)), "h"(static_cast<uint16_t>(3)) : "memory");
}

// The same on this CTA's barrier only.
__device__ __forceinline__ void tc_commit_pair_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}\n"
      :: "r"(smem_u32(bar)) : "memory");
}

// MODE as gemm_tc_kernel (0 whole tiles, 1 stream-K, 2 split-K), over pair tiles of 256 x 256 and
// pairs of CTAs: pair p = blockIdx.x / 2 takes the work gemm_tc_kernel gives CTA p of gridDim.x / 2.
// A stream-K partial is handed between the CTAs of equal rank in neighbouring pairs (slot blockIdx.x,
// taken from slot blockIdx.x + 2).
template <int EPI, int MODE, int EW, bool MN = false>
__global__ void __launch_bounds__(PairCfg<EW>::THREADS, 1)
gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
  using CF = PairCfg<EW>;
  constexpr int P_STAGES = CF::STAGES;
  static_assert(EW == 4 || MODE != 1, "stream-K partials are laid out for four epilogue warps");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;   // the same in both CTAs
  uint8_t* smem = smem_raw + pad;
  uint8_t* sA = smem;
  uint8_t* sB = smem + P_STAGES * P_A_BYTES;
  uint8_t* sE = smem + CF::STAGING;
  float* sBias = reinterpret_cast<float*>(smem + CF::BIAS);
  PairBars* bars = reinterpret_cast<PairBars*>(smem + CF::BAR);
  volatile int* abort_flag = &bars->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_cta_rank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int npairs = static_cast<int>(gridDim.x >> 1);
  const int MB = (args.M + 2 * BM - 1) / (2 * BM);
  const int NB = (args.N + BN - 1) / BN;
  const int KB = (args.K + BK - 1) / BK;
  const int num_tiles = MB * NB;
  constexpr bool SK = MODE == 1, KS = MODE == 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P_STAGES; ++s) { mbar_init(&bars->full[s], 1); mbar_init(&bars->empty[s], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&bars->tfull[i], 1); mbar_init(&bars->tempty[i], 2 * EW); }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  cluster_sync_all();               // the other CTA runs, and both CTAs' barriers exist before anything crosses over
  if (warp == 1) tmem_alloc_pair(&bars->tmem_base, TMEM_COLS);   // with the other CTA's warp 1
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (each CTA its own halves)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, last_par = 0;
      bool ok = true;
      // MN: both operands stored [K][M or N] (the weight gradients): this CTA's 128 rows of M (or N) are
      // two boxes of 64 (M or N) x 64 (K) at 8 KB strides, as in gemm_tc_kernel's MN-major stages
      auto load_a = [&](int st, int kb, int mb) {
        const uint32_t fb = cluster_addr(smem_u32(&bars->full[st]), 0);
        const int m0 = mb * 2 * BM + static_cast<int>(rank) * BM;
        if (MN) {
#pragma unroll
          for (int i = 0; i < BM / 64; ++i) tma_load_2d_pair(sA + st * P_A_BYTES + i * 8192, &tmA, fb, m0 + 64 * i, kb * BK);
        } else {
          tma_load_2d_pair(sA + st * P_A_BYTES, &tmA, fb, kb * BK, m0);
        }
      };
      auto load_b = [&](int st, int kb, int nb) {
        const uint32_t fb = cluster_addr(smem_u32(&bars->full[st]), 0);
        const int n0 = nb * BN + static_cast<int>(rank) * (BN / 2);
        if (MN) {
#pragma unroll
          for (int i = 0; i < BN / 128; ++i) tma_load_2d_pair(sB + st * P_B_BYTES + i * 8192, &tmB, fb, n0 + 64 * i, kb * BK);
        } else {
          tma_load_2d_pair(sB + st * P_B_BYTES, &tmB, fb, kb * BK, n0);
        }
      };
      int pre = 0;
      SegIter it = make_seg_iter_of(SK, KS, num_tiles, KB, args.ksplit, npairs, pair);
      if (args.b_const) {
        SegIter it0 = it;
        int tile0, kb00, kb10;
        if (it0.template next<KS>(tile0, kb00, kb10)) {
          int mb0, nb0;
          tile_coords(tile0, MB, NB, args.m_fastest, mb0, nb0);
          pre = (kb10 - kb00) < P_STAGES ? (kb10 - kb00) : P_STAGES;
          for (int i = 0; i < pre; ++i) {
            if (leader) mbar_arrive_expect_tx(&bars->full[i], 2 * P_STAGE_BYTES);
            load_b(i, kb00 + i, nb0);
          }
        }
      }
      pdl_wait();
      int tile, kb0, kb1;
      while (ok && it.template next<KS>(tile, kb0, kb1)) {
        int mb, nb;
        tile_coords(tile, MB, NB, args.m_fastest, mb, nb);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (pre > 0) {
            --pre;
            load_a(stage, kb, mb);
          } else {
            if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, args.err)) { ok = false; break; }
            if (leader) mbar_arrive_expect_tx(&bars->full[stage], 2 * P_STAGE_BYTES);
            load_a(stage, kb, mb);
            load_b(stage, kb, nb);
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == P_STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // the copies this CTA issued have landed once the pair's MMAs have read them (or the wait ran out)
      for (int s = 0; s < P_STAGES; ++s)
        if (issued & (1u << s)) mbar_wait_drain(&bars->empty[s], (last_par >> s) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (even CTA; whole warp, one elected lane issues)
    if (leader) {
      const uint32_t idesc = idesc_bf16_f32(2 * BM, BN, MN) | (MN ? (1u << 15) : 0u);   // bit 15: A MN-major
      const uint64_t da0 = smem_desc(smem_u32(sA), MN ? 8192 : 16, 1024, SWZ_128B);
      const uint64_t db0 = smem_desc(smem_u32(sB), MN ? 8192 : 16, 1024, SWZ_128B);
      constexpr uint64_t kstep = MN ? (16 * 128) >> 4 : 2;    // one K step of 16, in 16-byte units
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      SegIter it = make_seg_iter_of(SK, KS, num_tiles, KB, args.ksplit, npairs, pair);
      int tile, kb0, kb1;
      while (ok && it.template next<KS>(tile, kb0, kb1)) {
        if (!mbar_wait_warp(&bars->tempty[acc], acc_phase ^ 1u, abort_flag, args.err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_warp(&bars->full[stage], phase, abort_flag, args.err)) { ok = false; break; }
          tc_fence_after();
          const uint64_t da = da0 + static_cast<uint64_t>((stage * P_A_BYTES) >> 4);
          const uint64_t db = db0 + static_cast<uint64_t>((stage * P_B_BYTES) >> 4);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc_mma_pair_warp(d_tmem, da + kstep * k, db + kstep * k, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
          tc_commit_pair_both_warp(&bars->empty[stage]);
          if (++stage == P_STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit_pair_both_warp(&bars->tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      tc_commit_pair_warp(&bars->drain);
      mbar_wait_drain(&bars->drain, 0);
    }
  } else {
    // ------------------------------------------------ epilogue warps (each CTA its 128 rows)
    const int ew = warp - 2;                         // 0 .. EW-1
    const int sub = warp & 3;                        // TMEM lane quarter this warp may read
    const int c2a = (ew / 4) * CF::CHUNKS;           // its first 64-column chunk of the tile
    const int row = sub * 32 + lane;
    uint8_t* my_stage = sE + ew * EPI_BUF;
    float* my_bias = sBias + ew * BN;
    pdl_wait();
    int acc = 0;
    uint32_t acc_phase = 0;
    SegIter it = make_seg_iter_of(SK, KS, num_tiles, KB, args.ksplit, npairs, pair);
    int tile, kb0, kb1;
    while (it.template next<KS>(tile, kb0, kb1)) {
      int mb, nb;
      tile_coords(tile, MB, NB, args.m_fastest, mb, nb);
      const bool writer = kb0 > 0;
      const bool owner = kb0 == 0 && kb1 < KB;
      if (args.bias != nullptr && !writer) {
        const int nbase = nb * BN + lane * (BN / 32);
#pragma unroll
        for (int i = 0; i < BN / 32; ++i)
          my_bias[lane * (BN / 32) + i] = (nbase + i < args.N) ? __ldg(args.bias + nbase + i) : 0.0f;
        __syncwarp();
      }
      if (!mbar_wait(&bars->tfull[acc], acc_phase, abort_flag, args.err)) break;
      tc_fence_after();
      const int m0 = mb * 2 * BM + static_cast<int>(rank) * BM + sub * 32;   // this warp's first output row
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + static_cast<uint32_t>(acc * BN);
      // the accumulator is read: one arrival of this warp on the even CTA's barrier
      auto release_acc = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(cluster_addr(smem_u32(&bars->tempty[acc]), 0));
      };
      if (SK && writer) {
        float4* pw = reinterpret_cast<float4*>(args.sk_part) + ((size_t)blockIdx.x * 4 + sub) * (BN / 64) * 16 * 32 + lane;
#pragma unroll 1
        for (int c2 = 0; c2 < BN / 64; ++c2) {
          uint32_t r[64];
          tmem_ld_32x32b_x64(tbase + c2 * 64, r);
          tmem_ld_wait();
          if (c2 == BN / 64 - 1) release_acc();
#pragma unroll
          for (int q = 0; q < 16; ++q)
            pw[(c2 * 16 + q) * 32] = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                                 __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(args.sk_flag + blockIdx.x * 4 + sub, 1);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
        continue;
      }
      const float4* ppart = nullptr;
      if (SK && owner) {
        const int fi = (blockIdx.x + 2) * 4 + sub;
        int* flag = args.sk_wait_flag != nullptr ? const_cast<int*>(args.sk_wait_flag) + fi : args.sk_flag + fi;
        const long long limit = args.wait_limit > 0 ? args.wait_limit : kWaitLimitCycles;
        bool seen = ld_acquire_gpu(flag) != 0;
        if (!seen) {
          const long long t0 = clock64();
          while (!(seen = (ld_acquire_gpu(flag) != 0))) {
            if (*abort_flag || clock64() - t0 > limit) break;
          }
        }
        if (!__all_sync(0xffffffffu, seen)) {
          if (lane == 0) { record_error(args.err, GPT_DEV_ETIMEOUT); *abort_flag = 1; }
        } else if (lane == 0) {
          *flag = 0;
        }
        ppart = reinterpret_cast<const float4*>(args.sk_part) + ((size_t)(blockIdx.x + 2) * 4 + sub) * (BN / 64) * 16 * 32 + lane;
      }
#pragma unroll 1
      for (int c2 = c2a; c2 < c2a + CF::CHUNKS; ++c2) {
        uint32_t r[64];
        tmem_ld_32x32b_x64(tbase + c2 * 64, r);
        tmem_ld_wait();
        if (c2 == c2a + CF::CHUNKS - 1) release_acc();
        if (SK && ppart != nullptr) {
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float4 p4 = ppart[(c2 * 16 + q) * 32];
            r[4 * q + 0] = __float_as_uint(__uint_as_float(r[4 * q + 0]) + p4.x);
            r[4 * q + 1] = __float_as_uint(__uint_as_float(r[4 * q + 1]) + p4.y);
            r[4 * q + 2] = __float_as_uint(__uint_as_float(r[4 * q + 2]) + p4.z);
            r[4 * q + 3] = __float_as_uint(__uint_as_float(r[4 * q + 3]) + p4.w);
          }
        }
        constexpr int CW = (EPI == EPI_BIAS_RESID || EPI == EPI_F32_OUT) ? 32 : 64;   // columns per 128-byte row
#pragma unroll
        for (int h = 0; h < 64 / CW; ++h) {
          const int c = c2 * (64 / CW) + h;            // chunk of CW columns within the tile
          const int n0 = nb * BN + c * CW;
          if (n0 >= args.N) continue;
          uint32_t w[32];
          finish_chunk<EPI, CW>(args, r + h * CW, args.bias != nullptr ? my_bias + c * CW : nullptr, w);
          if (lane == 0) bulk_wait_read<0>();          // the previous store has read the box
          __syncwarp();
          stage_row(my_stage, lane, w);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (EPI == EPI_BIAS_RESID) tma_reduce_add_2d(&tmC, my_stage, n0, m0);   // x += tile, in L2
            else tma_store_2d(&tmC, my_stage, n0, m0);
            bulk_commit();
          }
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_all();
  }

  // Neither CTA leaves while the pair's MMAs, copies or arrivals may still touch it, and the TMEM is
  // freed by both CTAs' warps 1 together while both are still running.
  __syncwarp();
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
  cluster_sync_all();
}

template <int EPI, int MODE, int EW, bool MN = false>
cudaError_t launch_pair_inst(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, const GemmArgs& a,
                             int pairs, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<EPI, MODE, EW, MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               PairCfg<EW>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(PairCfg<EW>::THREADS);
  cfg.dynamicSmemBytes = PairCfg<EW>::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<EPI, MODE, EW, MN>, tmA, tmB, tmC, a);
}

template <int EPI, int MODE, bool MN = false>
cudaError_t launch_inst(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, const CUtensorMap& tmC2,
                        const GemmArgs& a, int grid, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<EPI, MODE, MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Layout<EPI>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_k(gemm_tc_kernel<EPI, MODE, MN>, dim3(grid), dim3(THREADS), Layout<EPI>::SMEM, s, tmA, tmB, tmC, tmC2,
                  a);
}

template <int EPI>
cudaError_t launch_one(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, const CUtensorMap& tmC2,
                       const GemmArgs& a, int grid_limit, cudaStream_t s) {
  const int MB = (a.M + BM - 1) / BM;
  const int NB = (a.N + BN - 1) / BN;
  const int tiles = MB * NB;
  const int grid = tiles < grid_limit ? tiles : grid_limit;
  if (grid <= 0) return cudaSuccess;
  constexpr bool kSplit = EPI == EPI_BIAS_OUT || EPI == EPI_BIAS_GELU_OUT || EPI == EPI_BIAS_RESID || EPI == EPI_F32_OUT;
  if (a.mn_major) {                   // weight gradients: both operands MN-major
    if constexpr (EPI == EPI_BIAS_RESID) {
      if (a.bias != nullptr) return cudaErrorInvalidValue;
      if (a.ksplit > 1) {
        if (a.ksplit > (a.K + BK - 1) / BK) return cudaErrorInvalidValue;
        const long long units = static_cast<long long>(tiles) * a.ksplit;
        const int g2 = units < grid_limit ? static_cast<int>(units) : grid_limit;
        return launch_inst<EPI, 2, true>(tmA, tmB, tmC, tmC2, a, g2, s);
      }
      if (a.sk_part != nullptr && a.sk_flag != nullptr && gemm_tc_stream_k(a.M, a.N, a.K, EPI, grid_limit))
        return launch_inst<EPI, 1, true>(tmA, tmB, tmC, tmC2, a, grid, s);
      return launch_inst<EPI, 0, true>(tmA, tmB, tmC, tmC2, a, grid, s);
    } else {
      return cudaErrorInvalidValue;
    }
  }
  if (a.ksplit > 1) {                 // split-K: (tile, K slice) units, reduce-add of each partial
    if constexpr (EPI == EPI_BIAS_RESID) {
      if (a.bias != nullptr || a.ksplit > (a.K + BK - 1) / BK) return cudaErrorInvalidValue;
      const long long units = static_cast<long long>(tiles) * a.ksplit;
      const int g2 = units < grid_limit ? static_cast<int>(units) : grid_limit;
      return launch_inst<EPI, 2>(tmA, tmB, tmC, tmC2, a, g2, s);
    } else {
      return cudaErrorInvalidValue;
    }
  }
  if constexpr (kSplit) {
    if (a.sk_part != nullptr && a.sk_flag != nullptr && gemm_tc_stream_k(a.M, a.N, a.K, EPI, grid_limit))
      return launch_inst<EPI, 1>(tmA, tmB, tmC, tmC2, a, grid, s);
  }
  return launch_inst<EPI, 0>(tmA, tmB, tmC, tmC2, a, grid, s);
}

}  // namespace

int gemm_tc_bn() { return BN; }

// Stream-K only where whole tiles would leave a partly idle last wave, and only
// for long K (at least kSplitMinKB K blocks): with shorter tiles the idle part of
// the last wave is smaller than the cost of splitting (measured on GB300).
constexpr int kSplitMinKB = 24;
bool gemm_tc_stream_k(int M, int N, int K, int epi, int grid_limit) {
  if (epi != EPI_BIAS_OUT && epi != EPI_BIAS_GELU_OUT && epi != EPI_BIAS_RESID && epi != EPI_F32_OUT) return false;
  const long long tiles = static_cast<long long>((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int KB = (K + BK - 1) / BK;
  return KB >= kSplitMinKB && grid_limit > 0 && tiles > grid_limit && tiles % grid_limit != 0;
}
// Slots 0 .. grid + 1: a CTA pair's partial goes from slot blockIdx.x + 2 to blockIdx.x.
size_t gemm_sk_part_floats(int grid) { return static_cast<size_t>(grid + 2) * BM * BN; }
size_t gemm_sk_flag_ints(int grid) { return static_cast<size_t>(grid + 2) * 4; }

int gemm_pair_capacity() {
  static int cap = -1;
  if (cap < 0) {
    int n = 0;
    if (cudaFuncSetAttribute(gemm_pair_kernel<EPI_BIAS_RESID, 1, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PairCfg<4>::SMEM) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2);
      cfg.blockDim = dim3(PairCfg<4>::THREADS);
      cfg.dynamicSmemBytes = PairCfg<4>::SMEM;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<EPI_BIAS_RESID, 1, 4>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();                    // a refused query leaves no error behind
    cap = n;
  }
  return cap;
}

bool pair_split(int tiles, int KB, int cap) { return KB >= kSplitMinKB && tiles > cap && tiles % cap != 0; }

bool gemm_pair_stream_k(int M, int N, int K, int max_pairs) {
  const int cap0 = gemm_pair_capacity();
  const int cap = cap0 < max_pairs ? cap0 : max_pairs;
  const int tiles = ((M + 2 * BM - 1) / (2 * BM)) * ((N + BN - 1) / BN);
  return cap > 0 && pair_split(tiles, (K + BK - 1) / BK, cap);
}

template <int EPI>
cudaError_t launch_pair_epi(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, const GemmArgs& a,
                            int max_pairs, cudaStream_t s) {
  if (a.mn_major && (EPI != EPI_BIAS_RESID || a.bias != nullptr)) return cudaErrorInvalidValue;
  const int cap0 = gemm_pair_capacity();
  const int cap = cap0 < max_pairs ? cap0 : max_pairs;
  if (cap <= 0) return cudaErrorNotSupported;
  const int MB = (a.M + 2 * BM - 1) / (2 * BM);
  const int NB = (a.N + BN - 1) / BN;
  const int tiles = MB * NB;
  if (tiles == 0) return cudaSuccess;
  const int KB = (a.K + BK - 1) / BK;
  if constexpr (EPI == EPI_BIAS_GELU_OUT) {   // eight epilogue warps, whole tiles only
    if (a.ksplit > 1) return cudaErrorInvalidValue;
    return launch_pair_inst<EPI, 0, 8>(tmA, tmB, tmC, a, tiles < cap ? tiles : cap, s);
  } else {
    if (a.ksplit > 1) {                    // split-K: (pair tile, K slice) units, each reduce-added
      if (EPI != EPI_BIAS_RESID || a.bias != nullptr || a.ksplit > KB) return cudaErrorInvalidValue;
      const long long units = static_cast<long long>(tiles) * a.ksplit;
      const int pairs = units < cap ? static_cast<int>(units) : cap;
      if constexpr (EPI == EPI_BIAS_RESID) {
        if (a.mn_major) return launch_pair_inst<EPI, 2, 4, true>(tmA, tmB, tmC, a, pairs, s);
      }
      return launch_pair_inst<EPI, 2, 4>(tmA, tmB, tmC, a, pairs, s);
    }
    if constexpr (EPI == EPI_BIAS_RESID) {
      if (a.mn_major) {
        if (a.sk_part != nullptr && a.sk_flag != nullptr && pair_split(tiles, KB, cap))
          return launch_pair_inst<EPI, 1, 4, true>(tmA, tmB, tmC, a, cap, s);
        return launch_pair_inst<EPI, 0, 4, true>(tmA, tmB, tmC, a, tiles < cap ? tiles : cap, s);
      }
    }
    if (a.sk_part != nullptr && a.sk_flag != nullptr && pair_split(tiles, KB, cap))
      return launch_pair_inst<EPI, 1, 4>(tmA, tmB, tmC, a, cap, s);
    return launch_pair_inst<EPI, 0, 4>(tmA, tmB, tmC, a, tiles < cap ? tiles : cap, s);
  }
}

cudaError_t launch_gemm_pair(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, const GemmArgs& a,
                             int epi, int max_pairs, cudaStream_t s) {
  switch (epi) {
    case EPI_BIAS_RESID: return launch_pair_epi<EPI_BIAS_RESID>(tmA, tmB, tmC, a, max_pairs, s);
    case EPI_F32_OUT: return launch_pair_epi<EPI_F32_OUT>(tmA, tmB, tmC, a, max_pairs, s);
    case EPI_BIAS_OUT: return launch_pair_epi<EPI_BIAS_OUT>(tmA, tmB, tmC, a, max_pairs, s);
    case EPI_BIAS_GELU_OUT: return launch_pair_epi<EPI_BIAS_GELU_OUT>(tmA, tmB, tmC, a, max_pairs, s);
    default: return cudaErrorInvalidValue;
  }
}
int gemm_tc_num_ntiles(int N) { return (N + BN - 1) / BN; }

cudaError_t launch_gemm_tc2(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                            const CUtensorMap& tmC2, const GemmArgs& a, int epi, int grid_limit, cudaStream_t s) {
  switch (epi) {
    case EPI_BIAS_OUT: return launch_one<EPI_BIAS_OUT>(tmA, tmB, tmC, tmC2, a, grid_limit, s);
    case EPI_BIAS_GELU_OUT: return launch_one<EPI_BIAS_GELU_OUT>(tmA, tmB, tmC, tmC2, a, grid_limit, s);
    case EPI_BIAS_RESID: return launch_one<EPI_BIAS_RESID>(tmA, tmB, tmC, tmC2, a, grid_limit, s);
    case EPI_F32: return launch_one<EPI_F32>(tmA, tmB, tmC, tmC2, a, grid_limit, s);
    case EPI_CE: return launch_one<EPI_CE>(tmA, tmB, tmC, tmC2, a, grid_limit, s);
    case EPI_CE_GRAD: return launch_one<EPI_CE_GRAD>(tmA, tmB, tmC, tmC2, a, grid_limit, s);
    case EPI_F32_OUT: return launch_one<EPI_F32_OUT>(tmA, tmB, tmC, tmC2, a, grid_limit, s);
    case EPI_GELU_GRAD: return launch_one<EPI_GELU_GRAD>(tmA, tmB, tmC, tmC2, a, grid_limit, s);
    case EPI_BIAS_GELU_UOUT: return launch_one<EPI_BIAS_GELU_UOUT>(tmA, tmB, tmC, tmC2, a, grid_limit, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_tc(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, const GemmArgs& a,
                           int epi, int grid_limit, cudaStream_t s) {
  if (epi == EPI_BIAS_GELU_UOUT) return cudaErrorInvalidValue;   // needs the second map
  return launch_gemm_tc2(tmA, tmB, tmC, tmC, a, epi, grid_limit, s);
}

}  // namespace gptgb
