// Causal flash-style self-attention on tcgen05 for sm_103a.
//
// Computes, per (batch b, head h), y = softmax(Q K^T / sqrt(D) + M) U with
// M = -inf for key s > query t ("第 25 章 从小 GPT 到 GPT-2" §25.2; "预训练一个
// Mini GPT" 第2步-第3步), reading Q, K, U straight out of the fused c_attn
// output qkv[B, T, 3C] (no head-split copy: the TMA coordinates pick the head's
// D columns) and writing the merged heads y[B, T, C].
//
// One CTA owns one 128-row query tile of one (b, h) and walks the key tiles
// 0..qtile (tiles above the diagonal are never touched; only the diagonal tile
// is masked). The softmax is the online (running max / running sum) form, the
// FlashAttention method named in "GPT-1 学习笔记" §10.2, so the T x T scores
// never reach memory.
//   S_j  = Q K_j^T      tcgen05.mma M=128 N=128 K=D   -> TMEM columns [0, 128)
//   PV_j = P_j U_j      tcgen05.mma M=128 N=D   K=128 -> TMEM columns [128, 128+D)
// P_j is written by the softmax threads to shared memory as bf16 in the
// 128-byte-swizzled K-major layout; U_j is consumed MN-major straight from its
// TMA tile. The running output O stays in registers (one row per thread).
// Warp roles (192 threads, two CTAs per SM):
//   warp 0      TMA producer: Q once, then K_j and U_j into a two-stage ring
//   warp 1      TMEM allocator and MMA issuer
//   warps 2-5   softmax / output: thread = query row (TMEM lane)
#include "common.cuh"
#include "kernels.h"

#include <math.h>

namespace gptgb {

namespace {

constexpr int BQ = kAttnBQ;       // query rows per tile
constexpr int BKV = 128;          // keys per tile
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 256;
constexpr int P_BYTES = BQ * BKV * 2;   // two 128-byte-swizzled blocks of 64 keys
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct AttnCfg {
  static constexpr int ROWB = D * 2;                               // bytes per row of a Q/K/U tile
  static constexpr uint32_t SWZ = (ROWB == 128) ? SWZ_128B : SWZ_64B;
  static constexpr int TILE = BQ * ROWB;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = TILE;                                 // two stages
  static constexpr int OFF_U = 3 * TILE;                             // two stages
  static constexpr int OFF_P = 5 * TILE;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int SMEM = OFF_BAR + 256;
  static_assert(D == 32 || D == 64, "head width");
  static_assert((OFF_P % 1024) == 0, "P must sit on a 1024-byte boundary");
};

struct __align__(8) AttnBars {
  uint64_t q_full;
  uint64_t kv_full[2];
  uint64_t kv_empty[2];
  uint64_t s_full;
  uint64_t p_full;
  uint64_t o_full;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > 200000000ull) return;
  }
}

template <int D>
__device__ __forceinline__ void issue_s(uint32_t tS, uint32_t q_addr, uint32_t k_addr) {
  using Cfg = AttnCfg<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(BQ, BKV, false);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    // K-major operands: a K step of 16 bf16 is 32 bytes along the swizzled row
    const uint64_t ad = smem_desc(q_addr + k * 32, 16, 8 * Cfg::ROWB, Cfg::SWZ);
    const uint64_t bd = smem_desc(k_addr + k * 32, 16, 8 * Cfg::ROWB, Cfg::SWZ);
    tc_mma_bf16(tS, ad, bd, idesc, k > 0 ? 1u : 0u);
  }
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t p_addr, uint32_t u_addr) {
  using Cfg = AttnCfg<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(BQ, D, true);     // U is MN-major (D contiguous)
#pragma unroll
  for (int kk = 0; kk < BKV / 16; ++kk) {
    const uint64_t ad = smem_desc(p_addr + (kk >> 2) * (BQ * 128) + (kk & 3) * 32, 16, 1024, SWZ_128B);
    // 16 keys = 16 rows of the U tile; 8-row groups are 8*ROWB apart
    const uint64_t bd = smem_desc(u_addr + kk * 16 * Cfg::ROWB, Cfg::TILE, 8 * Cfg::ROWB, Cfg::SWZ);
    tc_mma_bf16(tO, ad, bd, idesc, kk > 0 ? 1u : 0u);
  }
}

template <int D>
__global__ void __launch_bounds__(THREADS, 2)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm, __nv_bfloat16* __restrict__ y, int B, int T,
                   int H, int n_qtiles, float scale_log2, int* err) {
  using Cfg = AttnCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  AttnBars* bars = reinterpret_cast<AttnBars*>(smem_raw + Cfg::OFF_BAR);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((smem_u32(smem_raw) & 1023u) != 0) {           // the swizzle atoms need 1024-byte alignment
    if (threadIdx.x == 0) record_error(err, GPT_DEV_EALIGN);
    return;
  }
  uint8_t* sQ = smem_raw + Cfg::OFF_Q;
  uint8_t* sK = smem_raw + Cfg::OFF_K;
  uint8_t* sU = smem_raw + Cfg::OFF_U;
  uint8_t* sP = smem_raw + Cfg::OFF_P;
  volatile int* abort_flag = &bars->abort_flag;

  const int BH = B * H;
  const int qt = n_qtiles - 1 - static_cast<int>(blockIdx.x) / BH;   // longest rows first
  const int bh = static_cast<int>(blockIdx.x) % BH;
  const int b = bh / H;
  const int h = bh % H;
  const int C = H * D;
  const int q0 = qt * BQ;
  const int n_kv = qt + 1;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < 2; ++i) { mbar_init(&bars->kv_full[i], 1); mbar_init(&bars->kv_empty[i], 1); }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_full, 4);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&tm);
  if (warp == 1) tmem_alloc(&bars->tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  const uint32_t tS = tmem_base;
  const uint32_t tO = tmem_base + 128;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t issued = 0, last_par = 0;
      mbar_arrive_expect_tx(&bars->q_full, Cfg::TILE);
      tma_load_3d(sQ, &tm, &bars->q_full, h * D, q0, b);
      for (int j = 0; j < n_kv; ++j) {
        const int s = j & 1;
        const uint32_t use_par = static_cast<uint32_t>(j >> 1) & 1u;
        if (!mbar_wait(&bars->kv_empty[s], use_par ^ 1u, abort_flag, err)) break;
        mbar_arrive_expect_tx(&bars->kv_full[s], 2 * Cfg::TILE);
        tma_load_3d(sK + s * Cfg::TILE, &tm, &bars->kv_full[s], C + h * D, j * BKV, b);
        tma_load_3d(sU + s * Cfg::TILE, &tm, &bars->kv_full[s], 2 * C + h * D, j * BKV, b);
        issued |= 1u << s;
        last_par = (last_par & ~(1u << s)) | (use_par << s);
      }
      wait_drain(&bars->q_full, 0);
      for (int s = 0; s < 2; ++s)
        if (issued & (1u << s)) wait_drain(&bars->kv_full[s], (last_par >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t q_addr = smem_u32(sQ);
      bool ok = mbar_wait(&bars->q_full, 0, abort_flag, err) &&
                mbar_wait(&bars->kv_full[0], 0, abort_flag, err);
      if (ok) {
        tc_fence_after();
        issue_s<D>(tS, q_addr, smem_u32(sK));
        tc_commit(&bars->s_full);
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        const int s = j & 1;
        if (!mbar_wait(&bars->p_full, static_cast<uint32_t>(j) & 1u, abort_flag, err)) break;
        tc_fence_after();
        issue_pv<D>(tO, smem_u32(sP), smem_u32(sU + s * Cfg::TILE));
        tc_commit(&bars->o_full);
        tc_commit(&bars->kv_empty[s]);
        if (j + 1 < n_kv) {
          const int s1 = (j + 1) & 1;
          if (!mbar_wait(&bars->kv_full[s1], static_cast<uint32_t>((j + 1) >> 1) & 1u, abort_flag, err)) break;
          tc_fence_after();
          issue_s<D>(tS, q_addr, smem_u32(sK + s1 * Cfg::TILE));
          tc_commit(&bars->s_full);
        }
      }
      tc_commit(&bars->drain);
      wait_drain(&bars->drain, 0);
    }
  } else {
    // ------------------------------------------------ softmax and output
    const int sub = warp & 3;
    const int r = sub * 32 + lane;           // query row within the tile = TMEM lane
    const int t = q0 + r;                    // query position
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    float o[D];
#pragma unroll
    for (int i = 0; i < D; ++i) o[i] = 0.0f;
    float m = -INFINITY;                     // running max of the log2-scaled scores
    float l = 0.0f;                          // running sum of 2^(s - m)
    bool ok = true;
    uint8_t* prow = sP + (r >> 3) * 1024 + (r & 7) * 128;

    for (int j = 0; j < n_kv; ++j) {
      if (!mbar_wait(&bars->s_full, static_cast<uint32_t>(j) & 1u, abort_flag, err)) { ok = false; break; }
      tc_fence_after();
      const bool diag = (j == n_kv - 1);
      const int k0 = j * BKV;
      // pass 1: row maximum of this tile (allowed keys only)
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < BKV / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tS + lane_off + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float sv = __uint_as_float(v[i]) * scale_log2;
          if (!diag || (k0 + c * 32 + i) <= t) mx = fmaxf(mx, sv);
        }
      }
      const float m_new = fmaxf(m, mx);
      // fold in the previous tile's P U (scaled to the previous max)
      if (j > 0) {
        if (!mbar_wait(&bars->o_full, static_cast<uint32_t>(j - 1) & 1u, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tO + lane_off + c * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[c * 32 + i] += __uint_as_float(v[i]);
        }
      }
      const float alpha = ex2_approx(m - m_new);      // m = -inf on the first tile: alpha = 0
#pragma unroll
      for (int i = 0; i < D; ++i) o[i] *= alpha;
      l *= alpha;
      // pass 2: probabilities of this tile, as bf16 into the swizzled P tile
#pragma unroll 1
      for (int c = 0; c < BKV / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tS + lane_off + c * 32, v);
        tmem_ld_wait();
        float p[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const bool allowed = !diag || (k0 + c * 32 + i) <= t;
          p[i] = allowed ? ex2_approx(fmaf(__uint_as_float(v[i]), scale_log2, -m_new)) : 0.0f;
          l += p[i];
        }
        uint8_t* blk = prow + (c >> 1) * (BQ * 128);
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) {
          const int unit = ((c & 1) * 4 + qd) ^ (r & 7);
          uint4 w;
          w.x = pack_bf16x2(p[8 * qd + 0], p[8 * qd + 1]);
          w.y = pack_bf16x2(p[8 * qd + 2], p[8 * qd + 3]);
          w.z = pack_bf16x2(p[8 * qd + 4], p[8 * qd + 5]);
          w.w = pack_bf16x2(p[8 * qd + 6], p[8 * qd + 7]);
          *reinterpret_cast<uint4*>(blk + unit * 16) = w;
        }
      }
      m = m_new;
      fence_proxy_async_smem();               // P stores -> visible to the tensor core
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);
    }
    if (ok && mbar_wait(&bars->o_full, static_cast<uint32_t>(n_kv - 1) & 1u, abort_flag, err)) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tO + lane_off + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[c * 32 + i] += __uint_as_float(v[i]);
      }
      if (t < T) {
        const float inv = 1.0f / l;
        uint4* dst = reinterpret_cast<uint4*>(y + ((size_t)b * T + t) * C + h * D);
#pragma unroll
        for (int q = 0; q < D / 8; ++q) {
          uint4 w;
          w.x = pack_bf16x2(o[8 * q + 0] * inv, o[8 * q + 1] * inv);
          w.y = pack_bf16x2(o[8 * q + 2] * inv, o[8 * q + 3] * inv);
          w.z = pack_bf16x2(o[8 * q + 4] * inv, o[8 * q + 5] * inv);
          w.w = pack_bf16x2(o[8 * q + 6] * inv, o[8 * q + 7] * inv);
          dst[q] = w;
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_d(const CUtensorMap& tm, void* y, int B, int T, int H, int* err, cudaStream_t s) {
  using Cfg = AttnCfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int n_qtiles = (T + BQ - 1) / BQ;
  const long long grid = (long long)n_qtiles * B * H;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  const float scale_log2 = kLog2e / sqrtf(static_cast<float>(D));
  attn_fwd_tc_kernel<D><<<static_cast<unsigned>(grid), THREADS, Cfg::SMEM, s>>>(
      tm, reinterpret_cast<__nv_bfloat16*>(y), B, T, H, n_qtiles, scale_log2, err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_tc(const CUtensorMap& tm_qkv, void* y, int B, int T, int H, int D, int* err,
                                cudaStream_t s) {
  if (D == 64) return launch_d<64>(tm_qkv, y, B, T, H, err, s);
  if (D == 32) return launch_d<32>(tm_qkv, y, B, T, H, err, s);
  return cudaErrorInvalidValue;
}

}  // namespace gptgb
