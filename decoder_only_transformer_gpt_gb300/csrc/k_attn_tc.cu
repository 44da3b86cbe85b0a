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
// A work item is one (b, h) and one 128-row query tile; the kernel is
// persistent (one CTA per SM walks its items, heaviest first, snake-dealt) and
// keeps its barriers, TMEM and K/U ring across items. Inside an item the score
// tiles are triple-buffered so the tensor core and the softmax overlap:
//   S(j)  = Q K_j^T   tcgen05.mma M=128 N=128 K=D  -> TMEM S[j % 3] (128 columns each)
//   O_h  += P(j)_h U_j[64h:64h+64]                 -> TMEM O_h (h = 0, 1)
// The softmax reads its 64 scores of S(j) into registers and writes P(j) back
// as bf16 pairs over the first 32 columns of the same 64 (row = lane), so the
// P U MMA takes its A operand straight from tensor memory: probabilities never
// pass through shared memory. While the softmax turns S(j) into P(j), the
// tensor core already holds S(j+1) and S(j+2); once P(j) is handed over it runs
// P(j) U_j and then S(j+3) into the same buffer (one thread's MMAs execute in
// issue order, so S(j+3) overwrites P(j) only after P(j) U_j has read it), which
// leaves two softmax steps for that chain. The query tile is double-buffered
// across items, so an item's first score tiles never wait for its Q load; the
// next item's first P U waits only for the previous item's output to be read,
// which the same softmax warps do before they produce that P. U_j is consumed
// MN-major straight from its TMA tile. Two softmax threads share each query row
// (= TMEM lane): one owns keys [0, 64) of every key tile, the other keys
// [64, 128), each with its own running max, running sum and TMEM output
// accumulator. The running max is raised lazily: a half's O and sum are
// rescaled only when its max grows by more than 2^8. At the end of an item both
// threads of a row exchange their (max, sum) and each writes half of the row's
// D output columns.
// Warp roles (320 threads, one persistent CTA per SM):
//   warp 0      TMA producer: Q once per item (two buffers), then K_j, U_j into a five-stage ring
//   warp 1      TMEM allocator (512 columns) and MMA issuer (the whole warp runs
//               the loop, one elected lane issues)
//   warps 2-5   softmax, keys [0, 64) of each tile; warps 6-9 keys [64, 128)
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
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;    // rescale O only when the max grows by more than this
constexpr float kSumLimit = 65536.0f;   // off-diagonal tiles: recompute against the exact max past this sum
constexpr int NS = 5;                   // K/U ring depth (key tiles in flight)
constexpr uint32_t NSB = 3;             // score buffers: S(j+3) is issued while the softmax works on S(j+1)
// TMEM columns
constexpr uint32_t kColS = 0;           // S[k] at 128 k, k < NSB
constexpr uint32_t kColO = 128 * NSB;   // O (half h at + 64 h): 384..511

template <int D>
struct AttnCfg {
  static constexpr int ROWB = D * 2;                               // bytes per row of a Q/K/U tile
  static constexpr uint32_t SWZ = (ROWB == 128) ? SWZ_128B : SWZ_64B;
  static constexpr int TILE = BQ * ROWB;
  static constexpr int OFF_Q = 0;                                    // Q[0], Q[1]
  static constexpr int OFF_K = 2 * TILE;                             // NS stages
  static constexpr int OFF_U = OFF_K + NS * TILE;                    // NS stages
  static constexpr int OFF_ML = OFF_U + NS * TILE;                  // (max, sum) of both halves of every row
  static constexpr int OFF_BAR = OFF_ML + 2 * BQ * 8;
  // at least 120 KB so that two CTAs (2 x 512 TMEM columns) never share an SM
  static constexpr int SMEM = (OFF_BAR + 256 > 120 * 1024) ? OFF_BAR + 256 : 120 * 1024;
  static_assert(D == 32 || D == 64, "head width");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct __align__(8) AttnBars {
  uint64_t q_full[2];       // Q buffer r % 2 holds item r's query tile
  uint64_t q_empty[2];      // every S of the item that used Q buffer k has been computed
  uint64_t kv_full[NS];
  uint64_t kv_empty[NS];
  uint64_t s_full[NSB];     // score buffer b holds a new score tile
  uint64_t p_full[NSB];     // buffer b holds a tile's probabilities (8 softmax warps)
  uint64_t o_full[NSB];     // the P U of a step with buffer b has completed
  uint64_t o_free;          // the output accumulator has been read out of TMEM (8 softmax warps)
  uint64_t ml_full;         // both halves wrote their (max, sum) for the merge (8 softmax warps)
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(AttnBars) <= 256, "barrier block");

// The start-address field is the low 14 bits of a descriptor (address >> 4), and
// every operand here lies below 256 KB, so advancing an operand by `bytes` is a
// plain add of bytes >> 4 to its base descriptor.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

template <int D>
__device__ __forceinline__ void issue_s(uint32_t tS, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = idesc_bf16_f32(BQ, BKV, false);
#pragma unroll
  for (int k = 0; k < D / 16; ++k)          // K-major: a K step of 16 bf16 is 32 bytes along the swizzled row
    tc_mma_bf16_warp(tS, desc_add(q_desc, k * 32), desc_add(k_desc, k * 32), idesc, k > 0 ? 1u : 0u);
}

// O_h += P(j)_h U_h for both key halves h: P(j) lies in TMEM over the first 32
// columns of each 64-column half of its score buffer (two bf16 per column, row =
// lane), U_j is MN-major in shared memory (D contiguous per key).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tO, uint32_t tP, uint64_t u_desc, bool accumulate) {
  using Cfg = AttnCfg<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(BQ, D, true);     // U is MN-major (D contiguous)
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      // a K step of 16 keys is 8 TMEM columns of P and 16 rows of ROWB bytes of U
      tc_mma_bf16_ts_warp(tO + 64 * hf, tP + 64 * hf + 8 * kk, desc_add(u_desc, (hf * 64 + kk * 16) * Cfg::ROWB),
                          idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
  }
}

// Work item `r` of this CTA's sequence: items are (query tile, b, h) with the
// heaviest tiles first, dealt to the CTAs in a snake order (CTA c takes c,
// 2G-1-c, 2G+c, ...) so long and short items even out across the grid.
__device__ __forceinline__ int item_of(int r, int cta, int G) {
  return (r & 1) ? r * G + (G - 1 - cta) : r * G + cta;
}

struct Item {
  int b, h, qt, n;          // n: key tiles 0..qt
};

__device__ __forceinline__ Item decode_item(int item, int BH, int H, int n_qtiles) {
  Item w;
  w.qt = n_qtiles - 1 - item / BH;
  const int bh = item % BH;
  w.b = bh / H;
  w.h = bh % H;
  w.n = w.qt + 1;
  return w;
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
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
  volatile int* abort_flag = &bars->abort_flag;

  const int BH = B * H;
  const int C = H * D;
  const int n_items = n_qtiles * BH;
  const int G = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    for (uint32_t i = 0; i < NSB; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 8);
      mbar_init(&bars->o_full[i], 1);
    }
    mbar_init(&bars->o_free, 8);
    mbar_init(&bars->ml_full, 8);
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
      uint32_t q_loads = 0;                          // Q tiles loaded so far (q_full phases)
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int item = item_of(r, cta, G);
        if (item >= n_items) break;
        const Item w = decode_item(item, BH, H, n_qtiles);
        const int qb = r & 1;                        // Q buffer of this item; its previous user was item r - 2
        if (r >= 2 && !mbar_wait(&bars->q_empty[qb], static_cast<uint32_t>((r >> 1) - 1) & 1u, abort_flag, err)) break;
        mbar_arrive_expect_tx(&bars->q_full[qb], Cfg::TILE);
        tma_load_3d(sQ + qb * Cfg::TILE, &tm, &bars->q_full[qb], w.h * D, w.qt * BQ, w.b);
        ++q_loads;
        for (int j = 0; j < w.n; ++j, ++kv_it) {
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
      for (uint32_t k = q_loads > 2 ? q_loads - 2 : 0; k < q_loads; ++k)
        mbar_wait_drain(&bars->q_full[k & 1u], (k >> 1) & 1u);
      for (int s = 0; s < NS; ++s)
        if (issued & (1u << s)) mbar_wait_drain(&bars->kv_full[s], (last_par >> s) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (whole warp; one elected lane issues)
    {
      // base descriptors: Q and K K-major (8-row groups ROWB*8 apart), P K-major
      // 128-byte swizzle, U MN-major (K-direction 8-row groups ROWB*8 apart)
      const uint64_t dq0 = smem_desc(smem_u32(sQ), 16, 8 * Cfg::ROWB, Cfg::SWZ);
      const uint64_t dk0 = smem_desc(smem_u32(sK), 16, 8 * Cfg::ROWB, Cfg::SWZ);
      const uint64_t du0 = smem_desc(smem_u32(sU), Cfg::TILE, 8 * Cfg::ROWB, Cfg::SWZ);
      uint32_t kv_it = 0;                            // K/U tiles consumed so far (ring position)
      uint32_t gs = 0;                               // score tiles so far: step g uses buffers g % 2
      uint32_t items_done = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int item = item_of(r, cta, G);
        if (item >= n_items) break;
        const Item w = decode_item(item, BH, H, n_qtiles);
        const int qb = r & 1;
        if (!mbar_wait_warp(&bars->q_full[qb], static_cast<uint32_t>(r >> 1) & 1u, abort_flag, err)) break;
        const uint64_t dq = desc_add(dq0, qb * Cfg::TILE);
        const uint32_t tO = tmem_base + kColO;
        // the first two score tiles (the softmax read both buffers' previous tiles before
        // handing over the previous item's last probabilities)
        for (int jj = 0; jj < static_cast<int>(NSB) && jj < w.n; ++jj) {
          const uint32_t t = kv_it + jj;
          const uint32_t b = (gs + jj) % NSB;
          if (!mbar_wait_warp(&bars->kv_full[t % NS], (t / NS) & 1u, abort_flag, err)) { ok = false; break; }
          tc_fence_after();
          issue_s<D>(tmem_base + kColS + 128 * b, dq, desc_add(dk0, (t % NS) * Cfg::TILE));
          tc_commit_warp(&bars->s_full[b]);
        }
        for (int j = 0; j < w.n && ok; ++j) {
          const uint32_t g = gs + j;
          const uint32_t b = g % NSB;
          const uint32_t s = (kv_it + j) % NS;
          if (!mbar_wait_warp(&bars->p_full[b], (g / NSB) & 1u, abort_flag, err)) { ok = false; break; }
          // the previous item's output has been read out of the accumulator
          if (j == 0 && items_done >= 1 &&
              !mbar_wait_warp(&bars->o_free, (items_done - 1) & 1u, abort_flag, err)) { ok = false; break; }
          tc_fence_after();
          issue_pv<D>(tO, tmem_base + kColS + 128 * b, desc_add(du0, s * Cfg::TILE), j > 0);
          tc_commit_warp(&bars->o_full[b]);
          tc_commit_warp(&bars->kv_empty[s]);        // K_j and U_j are consumed
          // the score tile after next into buffer b: issued after P(j) U_j, which reads
          // P(j) out of the same columns (one thread's MMAs run in issue order)
          if (j + static_cast<int>(NSB) < w.n) {
            const uint32_t t2 = kv_it + j + NSB;
            if (!mbar_wait_warp(&bars->kv_full[t2 % NS], (t2 / NS) & 1u, abort_flag, err)) { ok = false; break; }
            tc_fence_after();
            issue_s<D>(tmem_base + kColS + 128 * b, dq, desc_add(dk0, (t2 % NS) * Cfg::TILE));
            tc_commit_warp(&bars->s_full[b]);
          }
        }
        if (!ok) break;
        tc_commit_warp(&bars->q_empty[qb]);          // every S of this item has read its Q
        gs += w.n;
        kv_it += w.n;
        ++items_done;
      }
      tc_commit_warp(&bars->drain);
      mbar_wait_drain(&bars->drain, 0);
    }
  } else {
    // ------------------------------------------------ softmax
    const int hf = (warp - 2) >> 2;                   // which 64 keys of every key tile
    const int sub = warp & 3;
    const int r_row = sub * 32 + lane;                // query row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    float2* sML = reinterpret_cast<float2*>(smem_raw + Cfg::OFF_ML);   // [2 halves][BQ rows]
    uint32_t gs = 0;
    uint32_t items_done = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int item = item_of(r, cta, G);
      if (item >= n_items) break;
      const Item w = decode_item(item, BH, H, n_qtiles);
      const int t = w.qt * BQ + r_row;                // query position
      const uint32_t tO0 = tmem_base + kColO + lane_off;              // O of keys [0, 64)
      const uint32_t tO = tO0 + 64 * hf;                                // this half's O
      float m_run = -INFINITY;                        // running (lazily raised) max, log2 units
      float l = 0.0f;                                 // running sum of 2^(s - m_run) over this half
      for (int j = 0; j < w.n; ++j) {
        const uint32_t g = gs + j;
        const uint32_t b = g % NSB;
        if (!mbar_wait_warp(&bars->s_full[b], (g / NSB) & 1u, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tS = tmem_base + kColS + 128 * b + 64 * hf + lane_off;
        const bool diag = (j == w.n - 1);
        const int kb = j * BKV + 64 * hf;             // first key of this half
        // Raise this half's running max to m_new where `need`: scale its sum and output by
        // 2^(m_run - m_new) (the output once every earlier P U has landed). Warp-uniform.
        auto raise_max = [&](bool need, float m_new) -> bool {
          if (j > 0) {                                // this half's O must hold all earlier P U
            if (!mbar_wait_warp(&bars->o_full[(g - 1) % NSB], ((g - 1) / NSB) & 1u, abort_flag, err)) return false;
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
          return true;
        };
        // Exact maximum of this half's allowed keys, eight independent chains.
        auto tile_max = [&](const uint32_t (&v)[64]) -> float {
          float mx8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) mx8[k] = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float a = (!diag || kb + i <= t) ? __uint_as_float(v[i]) : -INFINITY;
            const float bv = (!diag || kb + 32 + i <= t) ? __uint_as_float(v[32 + i]) : -INFINITY;
            mx8[i & 7] = fmax3(mx8[i & 7], a, bv);
          }
          return fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        };
        // pv = 2^(s*scale - m_run), two keys per f32x2 instruction; returns their sum
        const float2 sc2 = make_float2(scale_log2, scale_log2);
        auto probs = [&](const uint32_t (&v)[64], float (&p)[64]) -> float {
          const float2 nm2 = make_float2(-m_run, -m_run);
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            const float2 x = fma2_rn(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), sc2, nm2);
            p[i] = ex2_approx(x.x);
            p[i + 1] = ex2_approx(x.y);
          }
          if (diag) {                                 // keys after t get probability 0
#pragma unroll
            for (int i = 0; i < 64; ++i) p[i] = (kb + i <= t) ? p[i] : 0.0f;
          }
          float2 ls[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) ls[k] = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int i = 0; i < 64; i += 2) ls[(i >> 1) & 3] = add2_rn(ls[(i >> 1) & 3], make_float2(p[i], p[i + 1]));
          const float2 l2 = add2_rn(add2_rn(ls[0], ls[1]), add2_rn(ls[2], ls[3]));
          return l2.x + l2.y;
        };
        // this half's 64 scores (one 64-column TMEM load)
        uint32_t sv[64];
        tmem_ld_32x32b_x64(tS, sv);
        tmem_ld_wait();
        float pv[64];
        float lt;                                     // this tile's sum of probabilities
        if (!diag) {
          // Off the diagonal no maximum pass: the probabilities are taken against the running
          // max (for an item's first tile, against this row's first score), and only a tile
          // whose sum passes 2^16 (every probability is at most its sum, and an overflow shows
          // as an infinite sum) is recomputed against its exact maximum.
          if (j == 0) m_run = __uint_as_float(sv[0]) * scale_log2;
          lt = probs(sv, pv);
          if (__any_sync(0xffffffffu, !(lt <= kSumLimit))) {
            tmem_ld_32x32b_x64(tS, sv);               // the scores again (their registers were reused)
            tmem_ld_wait();
            const float m_new = fmaxf(m_run, tile_max(sv) * scale_log2);
            if (!raise_max(m_new > m_run + kRescaleLog2, m_new)) { ok = false; break; }
            tmem_ld_32x32b_x64(tS, sv);
            tmem_ld_wait();
            lt = probs(sv, pv);
          }
        } else {
          // the diagonal tile: exact maximum first (a fully masked half leaves -inf: nothing to raise)
          const float m_new = fmaxf(m_run, tile_max(sv) * scale_log2);
          const bool need = m_new > m_run + kRescaleLog2;
          if (__any_sync(0xffffffffu, need)) {
            if (!raise_max(need, m_new)) { ok = false; break; }
            tmem_ld_32x32b_x64(tS, sv);               // read the scores again rather than hold them
            tmem_ld_wait();
          }
          lt = probs(sv, pv);
        }
        l += lt;
        // P(j) as bf16 pairs over the first 32 columns of this half (its scores are in registers)
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(pv[2 * i], pv[2 * i + 1]);
        tmem_st_32x32b_x32(tS, pk);
        tmem_st_wait();
        tc_fence_before();                      // our TMEM reads of S and writes of P precede the next MMA
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[b]);
      }
      if (!ok) break;
      // the item's output: both threads of a row exchange (max, sum); each writes D/2 columns
      const uint32_t glast = gs + w.n - 1;
      if (!mbar_wait_warp(&bars->o_full[glast % NSB], (glast / NSB) & 1u, abort_flag, err)) break;
      tc_fence_after();
      sML[hf * BQ + r_row] = make_float2(m_run, l);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->ml_full);
      if (!mbar_wait_warp(&bars->ml_full, items_done & 1u, abort_flag, err)) break;
      const float2 other = sML[(hf ^ 1) * BQ + r_row];
      const float m0 = hf == 0 ? m_run : other.x, l0 = hf == 0 ? l : other.y;
      const float m1 = hf == 0 ? other.x : m_run, l1 = hf == 0 ? other.y : l;
      const float m = fmaxf(m0, m1);                // finite: key 0 of tile 0 is always allowed
      const float a0 = ex2_approx(m0 - m);
      const float a1 = ex2_approx(m1 - m);          // 0 when the upper half never had an allowed key
      const float inv = 1.0f / (a0 * l0 + a1 * l1);
      const float w0 = a0 * inv, w1 = a1 * inv;
      constexpr int DH = D / 2;                      // output columns per thread
      const int c0 = hf * DH;
      uint32_t v0[DH], v1[DH];
      if constexpr (DH == 32) {
        tmem_ld_32x32b_x32(tO0 + c0, v0);
        tmem_ld_32x32b_x32(tO0 + 64 + c0, v1);
      } else {
        tmem_ld_32x32b_x16(tO0 + c0, v0);
        tmem_ld_32x32b_x16(tO0 + 64 + c0, v1);
      }
      tmem_ld_wait();
      tc_fence_before();                             // the accumulator may be overwritten after this
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->o_free);
      if (t < T) {
        uint4* dst = reinterpret_cast<uint4*>(y + ((size_t)w.b * T + t) * C + w.h * D + c0);
#pragma unroll
        for (int q = 0; q < DH / 8; ++q) {
          float f[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) f[i] = w0 * __uint_as_float(v0[8 * q + i]) + w1 * __uint_as_float(v1[8 * q + i]);
          uint4 wv;
          wv.x = pack_bf16x2(f[0], f[1]);
          wv.y = pack_bf16x2(f[2], f[3]);
          wv.z = pack_bf16x2(f[4], f[5]);
          wv.w = pack_bf16x2(f[6], f[7]);
          dst[q] = wv;
        }
      }
      gs += w.n;
      ++items_done;
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
  const long long items = (long long)n_qtiles * B * H;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  const float scale_log2 = kLog2e / sqrtf(static_cast<float>(D));
  return launch_k(attn_fwd_tc_kernel<D>, dim3(grid), dim3(THREADS), Cfg::SMEM, s, tm,
                  reinterpret_cast<__nv_bfloat16*>(y), B, T, H, n_qtiles, scale_log2, err);
}

}  // namespace

cudaError_t launch_attention_tc(const CUtensorMap& tm_qkv, void* y, int B, int T, int H, int D, int* err,
                                cudaStream_t s) {
  if (D == 64) return launch_d<64>(tm_qkv, y, B, T, H, err, s);
  if (D == 32) return launch_d<32>(tm_qkv, y, B, T, H, err, s);
  return cudaErrorInvalidValue;
}

}  // namespace gptgb
