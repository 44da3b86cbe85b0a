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
// Work item: one (b, h) and a PAIR of consecutive 128-row query tiles
// (2p, 2p + 1). Both read the same stream of 128-key K/U tiles, so each K/U
// tile is loaded once for 256 query rows. Two softmax groups of four warps own
// one query tile each (group 0 tile 2p, group 1 tile 2p + 1), one thread per
// query row (= TMEM lane), and run out of phase: while one group turns its
// scores into probabilities, the tensor core runs the other group's P U and the
// next scores. Items are numbered heaviest pair first and taken from a global
// counter by each CTA's producer as it needs them (longest-first list
// scheduling over the persistent CTAs).
//
// The score tiles of both groups form ONE sequence in a fixed order: per item,
// for key tile j, group 0's (if j <= 2p) then group 1's (if the tile 2p + 1
// exists). Score number k goes to TMEM buffer k % 3 (three 128-column
// buffers). Two MMA-issuing warps walk the sequence: one waits for the
// probabilities P(k) (written by the owning group over the first 64 columns of
// buffer k % 3, two bf16 per column, released in two 64-key halves) and issues
// O_g += P(k) U_j with the A operand in tensor memory; the other issues
// S(k + 3) = Q K^T into that buffer once the P U of number k has completed. Each
// group therefore finds its next score tile issued while it still works on the
// current one.
//
// Per row, one running (lazily raised) max and sum over all keys: a tile's
// probabilities are taken against the running max without a maximum pass (for
// an item's first tile the reference is the row's first score); only when a
// half tile's sum passes 2^16 (every probability is at most the sum, and an
// overflow shows as an infinite sum) is its exact maximum taken, and the
// running output and sum are rescaled when the max grows by more than 2^8. An
// item's output is normalised, staged in shared memory and stored by TMA (one
// 32-row box per warp; rows past T are clipped by the copy) during the group's
// next tile, just before that tile's first P U overwrites the accumulator.
//
// Tensor memory (512 columns): score buffers at 0, 128, 256; O_g at 384 + 64 g.
// Warp roles (352 threads, one persistent CTA per SM):
//   warp 0      TMA producer: takes work items, loads both query tiles of an item and then
//               K_j, U_j into a four-stage ring
//   warp 1      TMEM allocator; issues the P U MMAs (the whole warp runs the loop, one elected lane issues)
//   warps 2-5   softmax group 0; warps 6-9 softmax group 1
//   warp 10     issues the score MMAs
#include "common.cuh"
#include "kernels.h"
#include "launch.h"

#include <math.h>

namespace gptgb {

namespace {

constexpr int BQ = kAttnBQ;       // query rows per tile
constexpr int BKV = 128;          // keys per tile
constexpr int THREADS = 352;
constexpr int TMEM_COLS = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;    // rescale O only when the max grows by more than this
constexpr float kSumLimit = 65536.0f;   // recompute a tile against its exact max past this sum
constexpr int NS = 4;                   // K/U ring depth; the MMA warp's look-ahead needs at least 4
constexpr int NSB = 3;                  // score buffers
constexpr uint32_t kColO = 128 * NSB;   // O_g at kColO + 64 g
constexpr int SR = 8;                   // work items announced ahead by the producer (ring slots)
constexpr int kConsumers = 10;          // warps that read each announced item: 2 MMA issuers + 8 softmax

template <int D>
struct AttnCfg {
  static constexpr int ROWB = D * 2;                               // bytes per row of a Q/K/U tile
  static constexpr uint32_t SWZ = (ROWB == 128) ? SWZ_128B : SWZ_64B;
  static constexpr int TILE = BQ * ROWB;
  static constexpr int STG = 32 * ROWB;                            // one warp's 32 output rows
  static constexpr int OFF_Q = 0;                                    // [buffer][group] query tiles
  static constexpr int OFF_K = 4 * TILE;                             // NS stages
  static constexpr int OFF_U = OFF_K + NS * TILE;                    // NS stages
  static constexpr int OFF_STG = OFF_U + NS * TILE;                  // 8 warps' output staging
  static constexpr int OFF_BAR = OFF_STG + 8 * STG;
  // at least 120 KB so that two CTAs (2 x 512 TMEM columns) never share an SM
  static constexpr int SMEM = (OFF_BAR + 512 > 120 * 1024) ? OFF_BAR + 512 : 120 * 1024;
  static_assert(D == 32 || D == 64, "head width");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct __align__(8) AttnBars {
  uint64_t q_empty[2];      // every S of the item that used Q buffer k has been computed
  uint64_t kv_full[NS];     // ring stage holds K_j, U_j (and, for an item's first tile, its query tiles)
  uint64_t kv_empty[NS];
  uint64_t s_full[2][NSB];  // score buffer b holds a new score tile of group g (that group's uses of b, in order)
  uint64_t p_full[NSB][2];  // score buffer b holds that tile's probabilities of keys [64 h, 64 h + 64) (4 warps)
  uint64_t pv_done[NSB];    // the P U that read buffer b has completed (the buffer may take new scores)
  uint64_t o_full[2][3];    // group g's P U number i (its own count) has completed: barrier i % 3
  uint64_t drain[2];        // the issuing warps' own MMAs have completed (exit)
  uint64_t sched_full[SR];  // slot r % SR holds this CTA's r-th work item (from the producer)
  uint64_t sched_empty[SR]; // every consumer warp has read the slot
  int sched_item[SR];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(AttnBars) <= 512, "barrier block");

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

// O += P_h U_h for keys [64 h, 64 h + 64) of a tile: P lies in TMEM over the first 64
// columns of its score buffer (two bf16 per column, row = lane; keys 64 h.. at column 32 h),
// U is MN-major in shared memory (D contiguous per key).
template <int D>
__device__ __forceinline__ void issue_pv_half(uint32_t tO, uint32_t tP, uint64_t u_desc, int h, bool accumulate) {
  using Cfg = AttnCfg<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(BQ, D, true);     // U is MN-major (D contiguous)
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)            // a K step of 16 keys: 8 TMEM columns of P, 16 rows of U
    tc_mma_bf16_ts_warp(tO, tP + 32 * h + 8 * kk, desc_add(u_desc, (64 * h + 16 * kk) * Cfg::ROWB), idesc,
                        (accumulate || kk > 0) ? 1u : 0u);
}

// Work items are ((b, h), query-tile pair), numbered heaviest pair first. A CTA's producer
// takes the next number from a global counter whenever it starts an item (so the work
// evens out across the CTAs the way longest-first list scheduling does) and announces it to
// the CTA's other warps through a ring of SR slots; a number >= the item count ends the list.
__device__ __forceinline__ int next_item(AttnBars* bars, int r, volatile int* abort_flag, int* err, int lane) {
  const int slot = r % SR;
  if (!mbar_wait_warp(&bars->sched_full[slot], static_cast<uint32_t>(r / SR) & 1u, abort_flag, err)) return 0x7fffffff;
  const int item = reinterpret_cast<volatile int*>(bars->sched_item)[slot];
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars->sched_empty[slot]);
  return item;
}

struct Item {
  int b, h, qt0;            // query tiles qt0 (group 0) and qt0 + 1 (group 1)
  int n0, n1;               // key tiles of each group: qt + 1, or 0 for a tile past the sequence
  int nkv;                  // key tiles the item loads: max(n0, n1)
};

__device__ __forceinline__ Item decode_item(int item, int BH, int H, int n_qtiles, int n_pairs) {
  Item w;
  const int p = n_pairs - 1 - item / BH;
  const int bh = item % BH;
  w.b = bh / H;
  w.h = bh % H;
  w.qt0 = 2 * p;
  w.n0 = w.qt0 + 1;
  w.n1 = (w.qt0 + 1 < n_qtiles) ? w.qt0 + 2 : 0;
  w.nkv = w.n1 > w.n0 ? w.n1 : w.n0;
  return w;
}

// Walks the score-tile sequence of one CTA for the MMA warp: item r, key tile j, group g,
// with the item's tile counts and the ring position of its key tile 0.
struct Cursor {
  int r, j, g, n0, n1, nkv;
  uint32_t kvb;
  bool valid;
  __device__ __forceinline__ void load(AttnBars* bars, volatile int* abort_flag, int* err, int lane, int n_items, int BH,
                                       int n_qtiles, int n_pairs) {
    const int item = next_item(bars, r, abort_flag, err, lane);
    valid = item < n_items;
    if (valid) {
      const int qt0 = 2 * (n_pairs - 1 - item / BH);
      n0 = qt0 + 1;
      n1 = (qt0 + 1 < n_qtiles) ? qt0 + 2 : 0;
      nkv = n1 > n0 ? n1 : n0;
    }
  }
  __device__ __forceinline__ void advance(AttnBars* bars, volatile int* abort_flag, int* err, int lane, int n_items,
                                          int BH, int n_qtiles, int n_pairs) {
    if (g == 0 && j < n1) { g = 1; return; }
    if (++j < nkv) { g = (j < n0) ? 0 : 1; return; }
    kvb += nkv;
    ++r;
    j = 0;
    g = 0;
    load(bars, abort_flag, err, lane, n_items, BH, n_qtiles, n_pairs);
  }
  __device__ __forceinline__ uint32_t pos() const { return kvb + j; }
  // the element is the last MMA reader of its ring position / the item's last score tile
  __device__ __forceinline__ bool last_of_pos() const { return g == 1 || j >= n1; }
  __device__ __forceinline__ bool last_of_item() const { return j == nkv - 1 && last_of_pos(); }
};

// 16-byte unit u of row r of a staging box (rows of ROWB bytes) in the TMA swizzle of that width.
template <int ROWB>
__device__ __forceinline__ int swz_unit(int r, int u) {
  return (ROWB == 128) ? (u ^ (r & 7)) : (u ^ ((r >> 1) & 3));
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ CUtensorMap tm_y, int B,
                   int T, int H, int n_qtiles, float scale_log2, int* err, int* sched, float* lse2) {
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
  const int n_pairs = (n_qtiles + 1) / 2;
  const int n_items = n_pairs * BH;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_empty[i], 1);
      for (int k = 0; k < 3; ++k) mbar_init(&bars->o_full[i][k], 1);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 2);                // K read by the score warp, U by the P U warp
    }
    for (int i = 0; i < NSB; ++i) {
      mbar_init(&bars->s_full[0][i], 1);
      mbar_init(&bars->s_full[1][i], 1);
      mbar_init(&bars->p_full[i][0], 4);
      mbar_init(&bars->p_full[i][1], 4);
      mbar_init(&bars->pv_done[i], 1);
    }
    mbar_init(&bars->drain[0], 1);
    mbar_init(&bars->drain[1], 1);
    for (int i = 0; i < SR; ++i) {
      mbar_init(&bars->sched_full[i], 1);
      mbar_init(&bars->sched_empty[i], kConsumers);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm);
    tma_prefetch_desc(&tm_y);
  }
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
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int slot = r % SR;                     // announce the CTA's r-th item
        if (r >= SR && !mbar_wait(&bars->sched_empty[slot], static_cast<uint32_t>(r / SR - 1) & 1u, abort_flag, err)) break;
        const int item = atomicAdd(sched, 1);
        reinterpret_cast<volatile int*>(bars->sched_item)[slot] = item;
        mbar_arrive(&bars->sched_full[slot]);
        if (item >= n_items) break;
        const Item w = decode_item(item, BH, H, n_qtiles, n_pairs);
        const int qb = r & 1;                        // Q buffer of this item; its previous user was item r - 2
        if (r >= 2 && !mbar_wait(&bars->q_empty[qb], static_cast<uint32_t>((r >> 1) - 1) & 1u, abort_flag, err)) break;
        for (int j = 0; j < w.nkv; ++j, ++kv_it) {
          const int s = kv_it % NS;
          const uint32_t use_par = (kv_it / NS) & 1u;
          if (!mbar_wait(&bars->kv_empty[s], use_par ^ 1u, abort_flag, err)) { ok = false; break; }
          // the item's query tiles complete on the barrier of its first K/U tile
          const int nq = (j == 0) ? (w.n1 > 0 ? 2 : 1) : 0;
          mbar_arrive_expect_tx(&bars->kv_full[s], (2 + nq) * Cfg::TILE);
          if (nq > 0) tma_load_3d(sQ + (2 * qb) * Cfg::TILE, &tm, &bars->kv_full[s], w.h * D, w.qt0 * BQ, w.b);
          if (nq > 1) tma_load_3d(sQ + (2 * qb + 1) * Cfg::TILE, &tm, &bars->kv_full[s], w.h * D, (w.qt0 + 1) * BQ, w.b);
          tma_load_3d(sK + s * Cfg::TILE, &tm, &bars->kv_full[s], C + w.h * D, j * BKV, w.b);
          tma_load_3d(sU + s * Cfg::TILE, &tm, &bars->kv_full[s], 2 * C + w.h * D, j * BKV, w.b);
          issued |= 1u << s;
          last_par = (last_par & ~(1u << s)) | (use_par << s);
        }
      }
      // never leave with copies in flight into this CTA's shared memory
      for (int s = 0; s < NS; ++s)
        if (issued & (1u << s)) mbar_wait_drain(&bars->kv_full[s], (last_par >> s) & 1u);
    }
  } else if (warp == 1 || warp == 10) {
    // ------------------------------------------------ MMA issuers (whole warp; one elected lane issues)
    // Two warps on different sub-partitions share the issue work, each walking the same
    // sequence of score numbers: warp 1 waits for P(k) and issues O_g += P(k) U_j; warp 10
    // issues S(k) = Q K_j^T into buffer k % 3 once the P U of number k - 3 (which read that
    // buffer) has completed. A ring stage is released after both the last S reading its K and
    // the last P U reading its U; S(k) lies at most three ring positions past the oldest
    // unreleased stage, so four stages never wait on each other.
    {
      const bool pv_warp = warp == 1;
      // base descriptors: Q and K K-major (8-row groups ROWB*8 apart), U MN-major (K-direction
      // 8-row groups ROWB*8 apart)
      const uint64_t dq0 = smem_desc(smem_u32(sQ), 16, 8 * Cfg::ROWB, Cfg::SWZ);
      const uint64_t dk0 = smem_desc(smem_u32(sK), 16, 8 * Cfg::ROWB, Cfg::SWZ);
      const uint64_t du0 = smem_desc(smem_u32(sU), Cfg::TILE, 8 * Cfg::ROWB, Cfg::SWZ);
      Cursor c;
      c.r = 0;
      c.j = 0;
      c.g = 0;
      c.kvb = 0;
      c.load(bars, abort_flag, err, lane, n_items, BH, n_qtiles, n_pairs);
      uint32_t b = 0;                                // buffer of number k (k % 3)
      uint32_t bits = 0;                             // phase per buffer of the barrier this warp waits on
      if (pv_warp) {
        uint32_t oi0 = 0, oi1 = 0;                   // next o_full barrier per group (P U count % 3)
        while (c.valid) {
          const uint32_t st = c.pos() % NS;
          const uint32_t tOg = tmem_base + kColO + 64 * c.g;
          // keys [0, 64) as soon as the group releases them, then keys [64, 128)
          if (!mbar_wait_warp(&bars->p_full[b][0], (bits >> b) & 1u, abort_flag, err)) break;
          tc_fence_after();
          issue_pv_half<D>(tOg, tmem_base + 128 * b, desc_add(du0, st * Cfg::TILE), 0, c.j > 0);
          if (!mbar_wait_warp(&bars->p_full[b][1], (bits >> b) & 1u, abort_flag, err)) break;
          bits ^= 1u << b;
          tc_fence_after();
          issue_pv_half<D>(tOg, tmem_base + 128 * b, desc_add(du0, st * Cfg::TILE), 1, true);
          tc_commit_warp(&bars->pv_done[b]);
          if (c.g) {
            tc_commit_warp(&bars->o_full[1][oi1]);
            oi1 = oi1 == 2 ? 0 : oi1 + 1;
          } else {
            tc_commit_warp(&bars->o_full[0][oi0]);
            oi0 = oi0 == 2 ? 0 : oi0 + 1;
          }
          if (c.last_of_pos()) tc_commit_warp(&bars->kv_empty[st]);   // U_j is consumed
          c.advance(bars, abort_flag, err, lane, n_items, BH, n_qtiles, n_pairs);
          b = b == NSB - 1 ? 0 : b + 1;
        }
      } else {
        uint32_t n = 0;                              // score number
        uint32_t waited = 0xffffffffu;               // ring position whose K/U (and Q) was last waited for
        while (c.valid) {
          if (n >= NSB) {                            // the P U that read this buffer has completed
            if (!mbar_wait_warp(&bars->pv_done[b], (bits >> b) & 1u, abort_flag, err)) break;
            bits ^= 1u << b;
          }
          const uint32_t pos = c.pos();
          const uint32_t st = pos % NS;
          if (pos != waited) {
            if (!mbar_wait_warp(&bars->kv_full[st], (pos / NS) & 1u, abort_flag, err)) break;
            waited = pos;
          }
          tc_fence_after();
          const uint32_t qb = static_cast<uint32_t>(c.r) & 1u;
          issue_s<D>(tmem_base + 128 * b, desc_add(dq0, (2 * qb + c.g) * Cfg::TILE), desc_add(dk0, st * Cfg::TILE));
          tc_commit_warp(c.g ? &bars->s_full[1][b] : &bars->s_full[0][b]);
          if (c.last_of_pos()) tc_commit_warp(&bars->kv_empty[st]);   // K_j is consumed
          if (c.last_of_item()) tc_commit_warp(&bars->q_empty[qb]);   // every S of the item has read its Q
          c.advance(bars, abort_flag, err, lane, n_items, BH, n_qtiles, n_pairs);
          b = b == NSB - 1 ? 0 : b + 1;
          ++n;
        }
      }
      uint64_t* dr = &bars->drain[pv_warp ? 0 : 1];
      tc_commit_warp(dr);
      mbar_wait_drain(dr, 0);
    }
  } else {
    // ------------------------------------------------ softmax (group g owns query tile qt0 + g)
    const int g = (warp - 2) >> 2;
    const int sub = warp & 3;
    const int r_row = sub * 32 + lane;                // query row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    const uint32_t tO = tmem_base + kColO + 64 * g + lane_off;
    uint8_t* stg = smem_raw + Cfg::OFF_STG + (warp - 2) * Cfg::STG;
    uint32_t kbase = 0;                               // score number of the item's first tile
    uint32_t tiles = 0;                               // this group's tiles so far (its P U numbering)
    uint32_t used0 = 0, used1 = 0, used2 = 0;         // this group's score tiles so far in buffers 0, 1, 2
    bool ok = true;
    const float2 sc2 = make_float2(scale_log2, scale_log2);
    // An item's output is written during the group's next tile, just before that tile's first
    // P U (which overwrites the accumulator) is released: by then the item's last P U has
    // completed, so the group never idles on it.
    bool pend = false;
    float pl = 0.0f;                                  // the pending item's running sum
    float pm = 0.0f;                                  // and its running max (log2 units)
    int pb = 0, ph = 0, pqt = 0;                      // its batch row, head and query tile
    uint32_t plast = 0;                               // its last tile (this group's numbering)
    auto write_out = [&]() -> bool {
      if (!mbar_wait_warp(&bars->o_full[g][plast % 3], (plast / 3) & 1u, abort_flag, err)) return false;
      tc_fence_after();
      const float inv = 1.0f / pl;
      uint32_t ov[D];
      if constexpr (D == 64) {
        uint32_t (&o64)[64] = *reinterpret_cast<uint32_t (*)[64]>(ov);
        tmem_ld_32x32b_x64(tO, o64);
      } else {
        uint32_t (&o32)[32] = *reinterpret_cast<uint32_t (*)[32]>(ov);
        tmem_ld_32x32b_x32(tO, o32);
      }
      tmem_ld_wait();
      tc_fence_before();                        // the accumulator may be overwritten after this
      if (lane == 0) bulk_wait_read_all();      // this warp's previous store has read its staging box
      __syncwarp();
      uint8_t* row = stg + lane * Cfg::ROWB;
#pragma unroll
      for (int u = 0; u < Cfg::ROWB / 16; ++u) {
        uint4 v;
        v.x = pack_bf16x2(__uint_as_float(ov[8 * u + 0]) * inv, __uint_as_float(ov[8 * u + 1]) * inv);
        v.y = pack_bf16x2(__uint_as_float(ov[8 * u + 2]) * inv, __uint_as_float(ov[8 * u + 3]) * inv);
        v.z = pack_bf16x2(__uint_as_float(ov[8 * u + 4]) * inv, __uint_as_float(ov[8 * u + 5]) * inv);
        v.w = pack_bf16x2(__uint_as_float(ov[8 * u + 6]) * inv, __uint_as_float(ov[8 * u + 7]) * inv);
        *reinterpret_cast<uint4*>(row + (swz_unit<Cfg::ROWB>(lane, u) << 4)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&tm_y, stg, ph * D, pqt * BQ + sub * 32, pb);
        bulk_commit();
      }
      if (lse2 != nullptr) {                      // the row's base-2 log-sum-exp of the scaled scores
        const int t = pqt * BQ + r_row;
        if (t < T) lse2[(static_cast<size_t>(pb) * H + ph) * T + t] = pm + log2f(pl);
      }
      pend = false;
      return true;
    };
    for (int r = 0; ok; ++r) {
      const int item = next_item(bars, r, abort_flag, err, lane);
      if (item >= n_items) break;
      const Item w = decode_item(item, BH, H, n_qtiles, n_pairs);
      const int n = g == 0 ? w.n0 : w.n1;
      const uint32_t knext = kbase + w.n0 + w.n1;
      if (n == 0) { kbase = knext; continue; }        // group 1 past the last query tile
      const int qt = w.qt0 + g;
      const int t = qt * BQ + r_row;                  // query position
      float mr = -INFINITY;                           // running (lazily raised) max, log2 units
      float l = 0.0f;                                 // running sum of 2^(s - mr)
      for (int j = 0; j < n && ok; ++j) {
        // this tile's score number and buffer
        const uint32_t k = kbase + (g == 0 ? j + min(j, w.n1) : j + min(j + 1, w.n0));
        const uint32_t b = k % NSB;
        const uint32_t use = b == 0 ? used0++ : (b == 1 ? used1++ : used2++);
        if (!mbar_wait_warp(&bars->s_full[g][b], use & 1u, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tS = tmem_base + 128 * b + lane_off;
        const bool diag = (j == n - 1);
        const int kb = j * BKV;                       // first key of the tile
        // pv = 2^(s*scale - mr) in place of the scores, two keys per f32x2 instruction;
        // keys after t get 0 on the diagonal; returns the sum
        auto probs = [&](uint32_t (&v)[64], int kb_half) -> float {
          const float2 nm2 = make_float2(-mr, -mr);
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            const float2 x = fma2_rn(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), sc2, nm2);
            float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
            if (diag) {
              p0 = (kb_half + i <= t) ? p0 : 0.0f;
              p1 = (kb_half + i + 1 <= t) ? p1 : 0.0f;
            }
            v[i] = __float_as_uint(p0);
            v[i + 1] = __float_as_uint(p1);
          }
          float2 ls[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) ls[q] = make_float2(0.0f, 0.0f);
#pragma unroll
          for (int i = 0; i < 64; i += 2)
            ls[(i >> 1) & 3] = add2_rn(ls[(i >> 1) & 3], make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])));
          const float2 l2 = add2_rn(add2_rn(ls[0], ls[1]), add2_rn(ls[2], ls[3]));
          return l2.x + l2.y;
        };
        // exact maximum of the allowed keys of one half, eight independent chains
        auto half_max = [&](const uint32_t (&v)[64], int kb_half) -> float {
          float mx8[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) mx8[q] = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float a = (!diag || kb_half + i <= t) ? __uint_as_float(v[i]) : -INFINITY;
            const float c = (!diag || kb_half + 32 + i <= t) ? __uint_as_float(v[32 + i]) : -INFINITY;
            mx8[i & 7] = fmax3(mx8[i & 7], a, c);
          }
          return fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        };
        // The two 64-key halves in turn. A half's probabilities are final once its sum is checked
        // (and, rarely, recomputed against a raised max); they are then stored as bf16 pairs over
        // columns [32 hf, 32 hf + 32) of the buffer, whose scores are already in registers.
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          const uint32_t tSh = tS + 64 * hf;
          const int kbh = kb + 64 * hf;
          uint32_t sv[64];
          tmem_ld_32x32b_x64(tSh, sv);
          tmem_ld_wait();
          if (j == 0 && hf == 0) mr = __uint_as_float(sv[0]) * scale_log2;   // key 0 is allowed for every row
          float lt = probs(sv, kbh);
          if (__any_sync(0xffffffffu, !(lt <= kSumLimit))) {
            // rare: this half's exact maximum, a rescale of the running output and sum (and of
            // the first half's stored probabilities) where the max grew by more than 2^8, and
            // the half again against the new reference
            tmem_ld_32x32b_x64(tSh, sv);
            tmem_ld_wait();
            const float m_new = fmaxf(mr, half_max(sv, kbh) * scale_log2);
            const bool need = m_new > mr + kRescaleLog2;
            if (__any_sync(0xffffffffu, need)) {
              const float alpha = need ? ex2_approx(mr - m_new) : 1.0f;
              if (need) mr = m_new;
              l *= alpha;
              if (j > 0) {
                // every earlier P U of the group has completed (its own numbering, barrier i % 3)
                const uint32_t last = tiles - 1;
                if (!mbar_wait_warp(&bars->o_full[g][last % 3], (last / 3) & 1u, abort_flag, err)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                  uint32_t o[32];
                  tmem_ld_32x32b_x32(tO + c * 32, o);
                  tmem_ld_wait();
#pragma unroll
                  for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                  tmem_st_32x32b_x32(tO + c * 32, o);
                }
              }
              if (hf == 1) {                          // the first half's probabilities, already stored
                tmem_st_wait();
                uint32_t q[32];
                tmem_ld_32x32b_x32(tS, q);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                  const float2 f = unpack_bf16x2(q[i]);
                  q[i] = pack_bf16x2(f.x * alpha, f.y * alpha);
                }
                tmem_st_32x32b_x32(tS, q);
              }
              tmem_st_wait();
            }
            tmem_ld_32x32b_x64(tSh, sv);
            tmem_ld_wait();
            lt = probs(sv, kbh);
          }
          l += lt;
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(__uint_as_float(sv[2 * i]), __uint_as_float(sv[2 * i + 1]));
          if (hf == 1) {
            // the previous item's output leaves the accumulator before this item's first P U
            if (j == 0 && pend && !write_out()) { ok = false; break; }
            tmem_st_wait();                           // keys [0, 64) are final: hand them to the P U warp
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->p_full[b][0]);
          }
          tmem_st_32x32b_x32(tS + 32 * hf, pk);
        }
        if (!ok) break;
        tmem_st_wait();
        tc_fence_before();                      // our TMEM reads of S and writes of P precede the next MMA
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[b][1]);
        ++tiles;
      }
      if (!ok) break;
      // the item's output is written during the group's next tile (or after the last item)
      pend = true;
      pl = l;
      pm = mr;
      pb = w.b;
      ph = w.h;
      pqt = qt;
      plast = tiles - 1;
      kbase = knext;
    }
    if (ok && pend) write_out();
    if (lane == 0) bulk_wait_all();              // stores complete before the CTA exits
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    // every CTA has taken its last number once all have arrived here: the last one resets the
    // counter for the next launch
    __threadfence();
    if (atomicAdd(sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
      sched[0] = 0;
      sched[1] = 0;
      __threadfence();
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_d(const CUtensorMap& tm, void* y, int B, int T, int H, int* err, int* sched, float* lse2,
                     cudaStream_t s) {
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
  const long long items = (long long)((n_qtiles + 1) / 2) * B * H;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  CUtensorMap tm_y;
  if (!make_tmap_attn_out(&tm_y, y, B, T, H * D, D)) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  const float scale_log2 = kLog2e / sqrtf(static_cast<float>(D));
  return launch_k(attn_fwd_tc_kernel<D>, dim3(grid), dim3(THREADS), Cfg::SMEM, s, tm, tm_y, B, T, H, n_qtiles,
                  scale_log2, err, sched, lse2);
}

}  // namespace

cudaError_t launch_attention_tc(const CUtensorMap& tm_qkv, void* y, int B, int T, int H, int D, int* err,
                                int* sched, cudaStream_t s, float* lse2) {
  if (!sched) return cudaErrorInvalidValue;
  if (D == 64) return launch_d<64>(tm_qkv, y, B, T, H, err, sched, lse2, s);
  if (D == 32) return launch_d<32>(tm_qkv, y, B, T, H, err, sched, lse2, s);
  return cudaErrorInvalidValue;
}

}  // namespace gptgb
