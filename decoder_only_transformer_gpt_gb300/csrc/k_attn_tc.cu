// Causal flash-style self-attention on tcgen05 for sm_103a.
//
// Computes, per (batch b, head h), y = softmax(Q K^T / sqrt(D) + M) U with
// M = -inf for key s > query t ("第 25 章 从小 GPT 到 GPT-2" §25.2; "预训练一个
// Mini GPT" 第2步-第3步), reading Q, K, U straight out of the fused c_attn
// output qkv[B, T, 3C] through a 3-D TMA map (the head is a column offset, no
// split or transpose copy) and writing the merged heads y[B, T, C].
//
// The softmax is the online (running max / running sum) form, the tiling +
// online-softmax method named in "GPT-1 学习笔记" §10.2, so the T x T scores
// never reach memory. Key tiles above the diagonal are never loaded; only the
// diagonal tile is masked.
//
// A work item is one (b, h) and a PAIR of adjacent 128-row query tiles A = 2p and
// B = 2p+1, which share every K/U tile load. The kernel is persistent: one CTA
// per SM walks its items (heaviest first, snake-dealt), keeping its barriers,
// TMEM and K/U ring across items so the next item's tiles load early. Two softmax groups of 4 warps (one
// per query tile; thread = query row = TMEM lane) alternate with the tensor
// core: while group A turns S_A(j) into probabilities, the tensor core runs
// group B's products, and the other way round.
//   S_g(j)  = Q_g K_j^T   tcgen05.mma M=128 N=128 K=D   -> TMEM [128g, 128g+128)
//   O_g    += P_g(j) U_j  tcgen05.mma M=128 N=D   K=128 -> TMEM [256+128g, 256+128g+D)
// O accumulates in TMEM across key tiles. The running max is updated lazily: O
// and the running sum are rescaled only when a row's max grows by more than
// 2^8 (so probabilities stay below 256), which after the first tiles is rare.
// P_g(j) is written by the softmax threads as bf16 into a 128-byte-swizzled
// K-major shared tile; U_j is consumed MN-major straight from its TMA tile.
// Warp roles (320 threads, one persistent CTA per SM):
//   warp 0      TMA producer: Q_A, Q_B once, then K_j, U_j into a four-stage ring
//   warp 1      TMEM allocator (512 columns) and MMA issuer
//   warps 2-5   softmax group A, warps 6-9 softmax group B
#include "common.cuh"
#include "kernels.h"
#include "launch.h"

#include <math.h>

namespace gptgb {

namespace {

constexpr int BQ = kAttnBQ;       // query rows per tile
constexpr int BKV = 128;          // keys per tile
constexpr int THREADS = 320;
constexpr int TMEM_COLS = 512;
constexpr int P_BYTES = BQ * BKV * 2;   // two 128-byte-swizzled blocks of 64 keys
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;    // rescale O only when the max grows by more than this
constexpr int NS = 4;                   // K/U ring depth (key tiles in flight)

template <int D>
struct AttnCfg {
  static constexpr int ROWB = D * 2;                               // bytes per row of a Q/K/U tile
  static constexpr uint32_t SWZ = (ROWB == 128) ? SWZ_128B : SWZ_64B;
  static constexpr int TILE = BQ * ROWB;
  static constexpr int OFF_Q = 0;                                    // Q_A, Q_B
  static constexpr int OFF_K = 2 * TILE;                             // NS stages
  static constexpr int OFF_U = OFF_K + NS * TILE;                    // NS stages
  static constexpr int OFF_P = OFF_U + NS * TILE;                    // P_A, P_B
  static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
  // at least 120 KB so that two CTAs (2 x 512 TMEM columns) never share an SM
  static constexpr int SMEM = (OFF_BAR + 256 > 120 * 1024) ? OFF_BAR + 256 : 120 * 1024;
  static_assert(D == 32 || D == 64, "head width");
  static_assert((OFF_P % 1024) == 0, "P must sit on a 1024-byte boundary");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct __align__(8) AttnBars {
  uint64_t q_full;
  uint64_t q_empty;
  uint64_t kv_full[NS];
  uint64_t kv_empty[NS];
  uint64_t s_full[2];       // per group
  uint64_t p_full[2];
  uint64_t o_full[2];
  uint64_t o_free[2];       // the group read its item's final O out of TMEM
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};


// The start-address field is the low 14 bits of a descriptor (address >> 4), and
// every operand here lies below 256 KB, so advancing an operand by `bytes` is a
// plain add of bytes >> 4 to its base descriptor.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

template <int D>
__device__ __forceinline__ void issue_s(uint32_t tS, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = idesc_bf16_f32(BQ, BKV, false);
#pragma unroll
  for (int k = 0; k < D / 16; ++k)          // K-major: a K step of 16 bf16 is 32 bytes along the swizzled row
    tc_mma_bf16(tS, desc_add(q_desc, k * 32), desc_add(k_desc, k * 32), idesc, k > 0 ? 1u : 0u);
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tO, uint64_t p_desc, uint64_t u_desc, bool accumulate) {
  using Cfg = AttnCfg<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(BQ, D, true);     // U is MN-major (D contiguous)
#pragma unroll
  for (int kk = 0; kk < BKV / 16; ++kk) {
    // P: 64-key swizzle blocks of BQ*128 bytes, 32 bytes per K step inside one;
    // U: 16 keys = 16 rows of ROWB bytes
    tc_mma_bf16(tO, desc_add(p_desc, (kk >> 2) * (BQ * 128) + (kk & 3) * 32),
                desc_add(u_desc, kk * 16 * Cfg::ROWB), idesc, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// Work item `it` of this CTA's sequence: items are (query-tile pair, b, h) with
// the heaviest pairs first, dealt to the CTAs in a snake order (CTA c takes
// c, 2G-1-c, 2G+c, ...) so long and short items even out across the grid.
__device__ __forceinline__ int item_of(int r, int cta, int G) {
  return (r & 1) ? r * G + (G - 1 - cta) : r * G + cta;
}

struct Item {
  int b, h, qt_a, nA, nB, n_kv;
};

__device__ __forceinline__ Item decode_item(int item, int BH, int H, int n_pairs, int n_qtiles) {
  Item w;
  const int pair = n_pairs - 1 - item / BH;
  const int bh = item % BH;
  w.b = bh / H;
  w.h = bh % H;
  w.qt_a = 2 * pair;
  w.nA = w.qt_a + 1;                                       // key tiles of query tile A
  w.nB = (w.qt_a + 1 < n_qtiles) ? w.qt_a + 2 : 0;         // of tile B (none past the sequence)
  w.n_kv = w.nB > w.nA ? w.nB : w.nA;
  return w;
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm, __nv_bfloat16* __restrict__ y, int B, int T,
                   int H, int n_qtiles, int n_pairs, float scale_log2, int* err) {
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
  const int C = H * D;
  const int n_items = n_pairs * BH;
  const int G = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);
      mbar_init(&bars->o_full[i], 1);
      mbar_init(&bars->o_free[i], 4);
    }
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
  pdl_wait();                       // qkv written by the previous kernel is now visible
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t issued = 0, last_par = 0;
      uint32_t kv_it = 0;                            // K/U tiles loaded so far (ring position)
      uint32_t q_loads = 0;                          // Q pairs loaded so far (q_full phases)
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int item = item_of(r, cta, G);
        if (item >= n_items) break;
        const Item w = decode_item(item, BH, H, n_pairs, n_qtiles);
        if (r > 0 && !mbar_wait(&bars->q_empty, static_cast<uint32_t>(r - 1) & 1u, abort_flag, err)) break;
        mbar_arrive_expect_tx(&bars->q_full, (w.nB > 0 ? 2 : 1) * Cfg::TILE);
        tma_load_3d(sQ, &tm, &bars->q_full, w.h * D, w.qt_a * BQ, w.b);
        if (w.nB > 0) tma_load_3d(sQ + Cfg::TILE, &tm, &bars->q_full, w.h * D, (w.qt_a + 1) * BQ, w.b);
        ++q_loads;
        for (int j = 0; j < w.n_kv; ++j, ++kv_it) {
          const int s = kv_it % NS;
          const uint32_t use_par = (kv_it / NS) & 1u;
          if (!mbar_wait(&bars->kv_empty[s], use_par ^ 1u, abort_flag, err)) { ok = false; break; }
          mbar_arrive_expect_tx(&bars->kv_full[s], 2 * Cfg::TILE);
          tma_load_3d(sK + s * Cfg::TILE, &tm, &bars->kv_full[s], C + w.h * D, j * BKV, w.b);
          tma_load_3d(sU + s * Cfg::TILE, &tm, &bars->kv_full[s], 2 * C + w.h * D, j * BKV, w.b);
          issued |= 1u << s;
          last_par = (last_par & ~(1u << s)) | (use_par << s);
        }
      }
      // never leave with copies in flight into this CTA's shared memory
      if (q_loads > 0) mbar_wait_drain(&bars->q_full, (q_loads - 1) & 1u);
      for (int s = 0; s < NS; ++s)
        if (issued & (1u << s)) mbar_wait_drain(&bars->kv_full[s], (last_par >> s) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      // base descriptors: Q and K K-major (8-row groups ROWB*8 apart), P K-major
      // 128-byte swizzle, U MN-major (K-direction 8-row groups ROWB*8 apart)
      const uint64_t dq0 = smem_desc(smem_u32(sQ), 16, 8 * Cfg::ROWB, Cfg::SWZ);
      const uint64_t dq[2] = {dq0, desc_add(dq0, Cfg::TILE)};
      const uint64_t dk0 = smem_desc(smem_u32(sK), 16, 8 * Cfg::ROWB, Cfg::SWZ);
      const uint64_t du0 = smem_desc(smem_u32(sU), Cfg::TILE, 8 * Cfg::ROWB, Cfg::SWZ);
      const uint64_t dp0 = smem_desc(smem_u32(sP), 16, 1024, SWZ_128B);
      uint32_t kv_it = 0;
      uint32_t gstep[2] = {0, 0};                    // group steps so far (phase of s/p/o_full)
      uint32_t gitem[2] = {0, 0};                    // items each group finished (phase of o_free)
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int item = item_of(r, cta, G);
        if (item >= n_items) break;
        const Item w = decode_item(item, BH, H, n_pairs, n_qtiles);
        const int ng[2] = {w.nA, w.nB};
        if (!mbar_wait(&bars->q_full, static_cast<uint32_t>(r) & 1u, abort_flag, err) ||
            !mbar_wait(&bars->kv_full[kv_it % NS], (kv_it / NS) & 1u, abort_flag, err)) break;
        tc_fence_after();
        for (int g = 0; g < 2; ++g) {
          if (ng[g] == 0) continue;
          issue_s<D>(tmem_base + 128 * g, dq[g], desc_add(dk0, (kv_it % NS) * Cfg::TILE));
          tc_commit(&bars->s_full[g]);
        }
        for (int j = 0; j < w.n_kv && ok; ++j) {
          const uint32_t s = (kv_it + j) % NS;
          for (int g = 0; g < 2 && ok; ++g) {
            if (j >= ng[g]) continue;
            if (!mbar_wait(&bars->p_full[g], (gstep[g] + j) & 1u, abort_flag, err)) { ok = false; break; }
            if (j == 0 && gitem[g] > 0 &&          // the previous item's O has been read out
                !mbar_wait(&bars->o_free[g], (gitem[g] - 1) & 1u, abort_flag, err)) { ok = false; break; }
            tc_fence_after();
            issue_pv<D>(tmem_base + 256 + 128 * g, desc_add(dp0, g * P_BYTES), desc_add(du0, s * Cfg::TILE), j > 0);
            tc_commit(&bars->o_full[g]);
            if (j + 1 < ng[g]) {
              const uint32_t t1 = kv_it + j + 1;
              if (!mbar_wait(&bars->kv_full[t1 % NS], (t1 / NS) & 1u, abort_flag, err)) { ok = false; break; }
              tc_fence_after();
              issue_s<D>(tmem_base + 128 * g, dq[g], desc_add(dk0, (t1 % NS) * Cfg::TILE));
              tc_commit(&bars->s_full[g]);
            }
          }
          if (ok) tc_commit(&bars->kv_empty[s]);     // K_j and U_j consumed by both groups
        }
        if (!ok) break;
        tc_commit(&bars->q_empty);                   // every S of this item has read Q
        for (int g = 0; g < 2; ++g) {
          gstep[g] += ng[g];
          gitem[g] += ng[g] > 0 ? 1u : 0u;
        }
        kv_it += w.n_kv;
      }
      tc_commit(&bars->drain);
      mbar_wait_drain(&bars->drain, 0);
    }
  } else {
    // ------------------------------------------------ softmax groups
    const int grp = (warp - 2) >> 2;
    const int sub = warp & 3;
    const int r_row = sub * 32 + lane;                 // query row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    const uint32_t tS = tmem_base + 128 * grp + lane_off;
    const uint32_t tO = tmem_base + 256 + 128 * grp + lane_off;
    uint8_t* prow = sP + grp * P_BYTES + (r_row >> 3) * 1024 + (r_row & 7) * 128;
    uint32_t gstep = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int item = item_of(r, cta, G);
      if (item >= n_items) break;
      const Item w = decode_item(item, BH, H, n_pairs, n_qtiles);
      const int n_mine = grp ? w.nB : w.nA;
      if (n_mine == 0) continue;
      const int t = (w.qt_a + grp) * BQ + r_row;      // query position
      float m_run = -INFINITY;                        // running (lazily raised) max, log2 units
      float l = 0.0f;                                 // running sum of 2^(s - m_run)
      for (int j = 0; j < n_mine; ++j) {
        const uint32_t gs = gstep + j;
        if (!mbar_wait(&bars->s_full[grp], gs & 1u, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
        const bool diag = (j == n_mine - 1);
        const int k0 = j * BKV;
        // pass 1: row maximum over the allowed keys, 64 columns per TMEM wait,
        // eight independent chains
        float mx8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = -INFINITY;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t va[32], vb[32];
          tmem_ld_32x32b_x32(tS + hf * 64, va);
          tmem_ld_32x32b_x32(tS + hf * 64 + 32, vb);
          tmem_ld_wait();
          const int kb = k0 + hf * 64;
          if (diag) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float a = (kb + i <= t) ? __uint_as_float(va[i]) : -INFINITY;
              const float bv = (kb + 32 + i <= t) ? __uint_as_float(vb[i]) : -INFINITY;
              mx8[i & 7] = fmaxf(mx8[i & 7], fmaxf(a, bv));
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              mx8[i & 7] = fmaxf(mx8[i & 7], fmaxf(__uint_as_float(va[i]), __uint_as_float(vb[i])));
          }
        }
        const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const float m_new = fmaxf(m_run, mx * scale_log2);
        const bool need = m_new > m_run + kRescaleLog2;          // always true on the first tile
        if (__any_sync(0xffffffffu, need)) {
          if (j > 0) {
            if (!mbar_wait(&bars->o_full[grp], (gs - 1) & 1u, abort_flag, err)) { ok = false; break; }
            tc_fence_after();
          }
          const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
          if (need) m_run = m_new;
          l *= alpha;
          if (j > 0) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld_32x32b_x32(tO + c * 32, o);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
              tmem_st_32x32b_x32(tO + c * 32, o);
            }
            tmem_st_wait();
          }
        }
        // P_g is rewritten below: the previous step's P U must have finished reading it
        // (for j == 0 that was waited for when the previous item's O was read out)
        if (j > 0 && !mbar_wait(&bars->o_full[grp], (gs - 1) & 1u, abort_flag, err)) { ok = false; break; }
        // pass 2: probabilities 2^(s*scale - m_run) as bf16 into the swizzled P tile
        const float neg_m = -m_run;
        float ls[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) ls[k] = 0.0f;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t va[32], vb[32];
          tmem_ld_32x32b_x32(tS + hf * 64, va);
          tmem_ld_32x32b_x32(tS + hf * 64 + 32, vb);
          tmem_ld_wait();
          const int kb = k0 + hf * 64;
          uint8_t* blk = prow + hf * (BQ * 128);            // keys [64 hf, 64 hf + 64): one swizzle block
#pragma unroll
          for (int qd = 0; qd < 8; ++qd) {
            float pv[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int col = 8 * qd + k;                     // 0..63 within the half
              const uint32_t raw = col < 32 ? va[col & 31] : vb[col & 31];
              const bool allowed = !diag || (kb + col) <= t;
              pv[k] = allowed ? ex2_approx(fmaf(__uint_as_float(raw), scale_log2, neg_m)) : 0.0f;
              ls[k] += pv[k];
            }
            const int unit = qd ^ (r_row & 7);
            uint4 wv;
            wv.x = pack_bf16x2(pv[0], pv[1]);
            wv.y = pack_bf16x2(pv[2], pv[3]);
            wv.z = pack_bf16x2(pv[4], pv[5]);
            wv.w = pack_bf16x2(pv[6], pv[7]);
            *reinterpret_cast<uint4*>(blk + unit * 16) = wv;
          }
        }
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        fence_proxy_async_smem();               // P stores -> visible to the tensor core
        tc_fence_before();                      // our TMEM loads/stores are ordered before the next MMA
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[grp]);
      }
      if (!ok) break;
      // the item's output: O / l for this row
      if (!mbar_wait(&bars->o_full[grp], (gstep + n_mine - 1) & 1u, abort_flag, err)) break;
      tc_fence_after();
      const float inv = 1.0f / l;
      uint32_t o[D];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tO + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[c * 32 + i] = v[i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_free[grp]);   // O may be overwritten by the next item
      if (t < T) {
        uint4* dst = reinterpret_cast<uint4*>(y + ((size_t)w.b * T + t) * C + w.h * D);
#pragma unroll
        for (int q = 0; q < D / 8; ++q) {
          uint4 wv;
          wv.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
          wv.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
          wv.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
          wv.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
          dst[q] = wv;
        }
      }
      gstep += n_mine;
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
  static int num_sms = 0;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::SMEM);
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int n_qtiles = (T + BQ - 1) / BQ;
  const int n_pairs = (n_qtiles + 1) / 2;
  const long long items = (long long)n_pairs * B * H;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  const float scale_log2 = kLog2e / sqrtf(static_cast<float>(D));
  return launch_k(attn_fwd_tc_kernel<D>, dim3(grid), dim3(THREADS), Cfg::SMEM, s, tm,
                  reinterpret_cast<__nv_bfloat16*>(y), B, T, H, n_qtiles, n_pairs, scale_log2, err);
}

}  // namespace

cudaError_t launch_attention_tc(const CUtensorMap& tm_qkv, void* y, int B, int T, int H, int D, int* err,
                                cudaStream_t s) {
  if (D == 64) return launch_d<64>(tm_qkv, y, B, T, H, err, s);
  if (D == 32) return launch_d<32>(tm_qkv, y, B, T, H, err, s);
  return cudaErrorInvalidValue;
}

}  // namespace gptgb

