// Derivative of causal self-attention on tcgen05 for sm_103a.
//
// Forward ("第 25 章 从小 GPT 到 GPT-2" §25.2): S = Q K^T / sqrt(D) with s > t masked, A = softmax(S)
// per row, Y = A U. Back-propagation of the loss through it (the chain rule of these definitions, the
// training loop of "预训练一个 Mini GPT"): with A recomputed from the row's log-sum-exp (written by the
// forward) and Dsum[t] = sum_d dY[t,d] Y[t,d] (= sum_s A[t,s] dA[t,s]):
//   dA = dY U^T,  dS = A * (dA - Dsum),  dQ = dS K / sqrt(D),  dK = dS^T Q / sqrt(D),  dU = A^T dY.
//
// A work item is one (b, h) and one 128-key tile j; it walks the query tiles i = j, j + 1, .. that see
// those keys (causality), heaviest items first, taken from a global counter by each CTA's producer.
// Each query tile is taken in two halves g of 64 queries, each with its own tensor-memory buffer
// (key = TMEM lane); K_j and U_j themselves sit in tensor memory (columns [448, 448 + D)), copied there
// once per item by the output warps, so these products read only Q and dY from shared memory:
//   S^T_g  = K_j Q_{i,g}^T     M=128 keys, N=64 queries, K=D    columns [128 g, 128 g + 64)
//   dP^T_g = U_j dY_{i,g}^T    M=128, N=64, K=D                 columns [128 g + 64, 128 g + 128)
// so the tensor core works on one half while four derivative warps (one thread per key) work on the
// other: P^T = 2^(S^T log2(e)/sqrt(D) - lse2[q]), dS^T = P^T (dP^T - Dsum[q]) (zero above the diagonal
// and past T), written back as bf16 pairs over the first 32 columns of their fp32 halves, and dS^T also
// into shared memory (the MN-major A operand of the dQ product; two buffers, by query tile). Then
//   dU_j += P^T_g dY_{i,g}     A from tensor memory, B = dY rows read MN-major    columns [256, 256 + D)
//   dK_j += dS^T_g Q_{i,g}     A from tensor memory, B = Q rows read MN-major     columns [320, 320 + D)
//   dQ_i  = dS_i K_j           after both halves: A = dS (shared memory), B = K_j  columns [384, 384 + D)
// Order of issue per query tile t: [half 0 done] dU, dK of half 0, then S^T, dP^T of half 0 of the
// next tile; [half 1 done] dU, dK of half 1, dQ_t, then S^T, dP^T of half 1 of the next tile. So when
// the derivative warps see a half's scores, every earlier product (and with it every read of the
// buffers they are about to overwrite) has completed.
// Four output warps add each dQ_i tile into an fp32 [B][T][C] buffer with TMA reduce-adds (a query tile
// gets one from every key tile j <= i: no atomics on single elements) and, at the end of an item, store
// dK_j / sqrt(D) and dU_j into dqkv with TMA stores. A last kernel turns the fp32 dQ into bf16
// (x 1/sqrt(D)); the buffer is cleared before the derivative by a memset (zeroing it in that last kernel,
// right after reading each line, ran at a sixth of the copy rate). (Converting each 32-row slab inside this kernel, by the
// warp whose completed reduce-add is the slab's last as counted by a global atomic, was measured
// slower: the atomic's round trip, ~2-4k cycles after each reduce-add, held back the dQ hand-off.)
// Warp roles (320 threads, one persistent CTA per SM):
//   warp 0      producer: takes work items; K_j, U_j per item (two buffers), then Q_i, dY_i by TMA and
//               the rows' -lse2 and -Dsum (plain loads, interleaved by query pair) into a two-stage ring
//   warp 1      TMEM allocator and MMA issuer (the whole warp runs the loop, one elected lane issues)
//   warps 2-5   softmax derivative (thread = key row)
//   warps 6-9   output: K_j and U_j into tensor memory, dQ reduce-adds, dK and dU stores
#include "common.cuh"
#include "kernels.h"
#include "launch.h"

#include <math.h>

namespace gptgb {

namespace {

constexpr int BT = 128;                 // rows per key or query tile
constexpr int HQ = 64;                  // queries per half tile
constexpr int THREADS = 320;
constexpr int TMEM_COLS = 512;
constexpr int NQ = 2;                   // query-tile ring stages
constexpr int SR = 8;                   // work-item ring slots
constexpr int kConsumers = 9;           // warps that read each announced item: MMA + 4 derivative + 4 output
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kColDU = 256, kColDK = 320, kColDQ = 384;   // half g: S^T at 128 g, dP^T at 128 g + 64
constexpr uint32_t kColK = 448;         // K_j (bf16 pairs, D / 2 columns), then U_j: the item's A operands

template <int D>
struct BwdCfg {
  static constexpr int ROWB = D * 2;                              // bytes per row of a Q/K/U/dY tile
  static constexpr uint32_t SWZ = (ROWB == 128) ? SWZ_128B : SWZ_64B;
  static constexpr int TILE = BT * ROWB;
  static constexpr int OFF_K = 0;                                   // [2] item buffers
  static constexpr int OFF_U = 2 * TILE;                            // [2]
  static constexpr int OFF_Q = 4 * TILE;                            // [NQ]
  static constexpr int OFF_DY = OFF_Q + NQ * TILE;                  // [NQ]
  static constexpr int OFF_LD = OFF_DY + NQ * TILE;                 // [NQ][64 pairs] {-lse2 x2, -Dsum x2}
  static constexpr int OFF_DS = (OFF_LD + NQ * BT * 8 + 1023) / 1024 * 1024;
  static constexpr int DS_BUF = 2 * BT * 128;                       // one tile's dS: 2 atoms x 128 keys x 128 B
  static constexpr int OFF_STG = OFF_DS + 2 * DS_BUF;               // 4 output warps x 2 boxes of 4 KB
  static constexpr int OFF_BAR = OFF_STG + 4 * 8192;
  static constexpr int SMEM = OFF_BAR + 512;
  static_assert(D == 32 || D == 64, "head width");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct __align__(8) BwdBars {
  uint64_t kv_full[2], kv_empty[2];     // K_j, U_j of an item (buffer r % 2)
  uint64_t q_full[NQ], q_empty[NQ];     // Q_i, dY_i, -lse2 and -Dsum of a query tile
  uint64_t s_full[2];                   // S^T and dP^T of half g are in tensor memory
  uint64_t p_full[2];                   // the derivative warps wrote half g (4 warps)
  uint64_t dq_full;                     // the current tile's dQ product has completed
  uint64_t dq_free;                     // the output warps read it out of tensor memory (4 warps)
  uint64_t acc_full;                    // the item's dK and dU are complete
  uint64_t acc_free;                    // the output warps read them (4 warps)
  uint64_t kvt_full;                    // the item's K_j and U_j are in tensor memory (4 warps)
  uint64_t kvt_free;                    // the last product reading them has completed
  uint64_t sched_full[SR], sched_empty[SR];
  uint64_t drain;
  int sched_item[SR];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(BwdBars) <= 512, "barrier block");

__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (bytes >> 4); }

__device__ __forceinline__ int next_item(BwdBars* bars, int r, volatile int* abort_flag, int* err, int lane) {
  const int slot = r % SR;
  if (!mbar_wait_warp(&bars->sched_full[slot], static_cast<uint32_t>(r / SR) & 1u, abort_flag, err)) return 0x7fffffff;
  const int item = reinterpret_cast<volatile int*>(bars->sched_item)[slot];
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars->sched_empty[slot]);
  return item;
}

// 16-byte unit u of row r of a staging box (rows of `rowb` bytes) in the TMA swizzle of that width.
__device__ __forceinline__ int swz_unit(int rowb, int r, int u) {
  return (rowb == 128) ? (u ^ (r & 7)) : (u ^ ((r >> 1) & 3));
}

// One half tile of the softmax derivative for this thread's key row: reads S^T and dP^T (64 queries
// each) from columns [col, col + 64) and [col + 64, col + 128), writes P^T and dS^T as bf16 pairs
// over [col, col + 32) and [col + 64, col + 96), and dS^T into the row's 128-byte slot `ds_row` of a
// 64-query shared-memory atom, 32 queries at a time. ld: the half's 32 query pairs {-lse2, -lse2, -Dsum,
// -Dsum}. kMasked: keep only the queries ql (counted within the half) whose bit ql of `keep` is set.
template <bool kMasked>
__device__ __forceinline__ void derivative_half(uint32_t col, const float4* __restrict__ ld, float sl2, uint64_t keep,
                                                uint8_t* ds_row, int kr) {
  const float2 sl2v = make_float2(sl2, sl2);
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {                      // 32 queries at a time
    uint32_t sv[32], dv[32];
    tmem_ld_32x32b_x32(col + 32 * c, sv);
    tmem_ld_32x32b_x32(col + 64 + 32 * c, dv);
    tmem_ld_wait();
    uint32_t pp[16], pd[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float4 L = ld[16 * c + e];
      const float2 x = fma2_rn(make_float2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), sl2v,
                               make_float2(L.x, L.y));
      float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
      if (kMasked) {
        p0 = ((keep >> (32 * c + 2 * e)) & 1u) ? p0 : 0.0f;
        p1 = ((keep >> (32 * c + 2 * e + 1)) & 1u) ? p1 : 0.0f;
      }
      const float2 d = mul2_rn(make_float2(p0, p1),
                               add2_rn(make_float2(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1])),
                                       make_float2(L.z, L.w)));
      pp[e] = pack_bf16x2(p0, p1);
      pd[e] = pack_bf16x2(d.x, d.y);
    }
    // P^T and dS^T over columns [16 c, 16 c + 16) of their halves (already read)
    tmem_st_32x32b_x16(col + 16 * c, pp);
    tmem_st_32x32b_x16(col + 64 + 16 * c, pd);
#pragma unroll
    for (int u4 = 0; u4 < 4; ++u4) {                 // 16-byte unit u = queries [8 u, 8 u + 8) of the half
      const int u = 4 * c + u4;
      *reinterpret_cast<uint4*>(ds_row + (swz_unit(128, kr, u) << 4)) =
          make_uint4(pd[4 * u4], pd[4 * u4 + 1], pd[4 * u4 + 2], pd[4 * u4 + 3]);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(THREADS, 1)
attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_qkv, const __grid_constant__ CUtensorMap tm_dy,
                   const __grid_constant__ CUtensorMap tm_dkv, const __grid_constant__ CUtensorMap tm_dq,
                   const float* __restrict__ lse2, const float* __restrict__ dsum, int B, int T, int H, int n_qt,
                   float sl2, float rsd, int* err, int* sched) {
  using Cfg = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  BwdBars* bars = reinterpret_cast<BwdBars*>(smem_raw + Cfg::OFF_BAR);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) record_error(err, GPT_DEV_EALIGN);
    return;
  }
  volatile int* abort_flag = &bars->abort_flag;
  const int BH = B * H;
  const int C = H * D;
  const int n_items = n_qt * BH;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);
    }
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 4);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_free, 4);
    mbar_init(&bars->kvt_full, 4);
    mbar_init(&bars->kvt_free, 1);
    for (int i = 0; i < SR; ++i) {
      mbar_init(&bars->sched_full[i], 1);
      mbar_init(&bars->sched_empty[i], kConsumers);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_qkv);
    tma_prefetch_desc(&tm_dy);
    tma_prefetch_desc(&tm_dkv);
    tma_prefetch_desc(&tm_dq);
  }
  if (warp == 1) tmem_alloc(&bars->tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  pdl_wait();
  pdl_trigger();

  uint8_t* sK = smem_raw + Cfg::OFF_K;
  uint8_t* sU = smem_raw + Cfg::OFF_U;
  uint8_t* sQ = smem_raw + Cfg::OFF_Q;
  uint8_t* sDY = smem_raw + Cfg::OFF_DY;
  float* sLD = reinterpret_cast<float*>(smem_raw + Cfg::OFF_LD);
  uint8_t* sDS = smem_raw + Cfg::OFF_DS;

  if (warp == 0) {
    // ------------------------------------------------ producer (whole warp; lane 0 issues the copies)
    uint32_t qcount = 0;
    bool ok = true;
    uint32_t issued_kv = 0, par_kv = 0, issued_q = 0, par_q = 0;
    for (int r = 0; ok; ++r) {
      const int slot = r % SR;
      if (r >= SR && !mbar_wait_warp(&bars->sched_empty[slot], static_cast<uint32_t>(r / SR - 1) & 1u, abort_flag, err))
        break;
      int item = 0;
      if (lane == 0) {
        item = atomicAdd(sched, 1);
        reinterpret_cast<volatile int*>(bars->sched_item)[slot] = item;
        mbar_arrive(&bars->sched_full[slot]);
      }
      item = __shfl_sync(0xffffffffu, item, 0);
      if (item >= n_items) break;
      const int j = item / BH, bh = item - j * BH, b = bh / H, h = bh - b * H;
      const int kb = r & 1;
      if (r >= 2 && !mbar_wait_warp(&bars->kv_empty[kb], static_cast<uint32_t>((r >> 1) - 1) & 1u, abort_flag, err)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->kv_full[kb], 2 * Cfg::TILE);
        tma_load_3d(sK + kb * Cfg::TILE, &tm_qkv, &bars->kv_full[kb], C + h * D, j * BT, b);
        tma_load_3d(sU + kb * Cfg::TILE, &tm_qkv, &bars->kv_full[kb], 2 * C + h * D, j * BT, b);
      }
      issued_kv |= 1u << kb;
      par_kv = (par_kv & ~(1u << kb)) | (static_cast<uint32_t>((r >> 1) & 1) << kb);
      // the rows' -lse2 and -Dsum by query pair (plain loads; rows past T read nothing), each tile's
      // fetched one tile ahead so that their latency passes while the producer waits for a free slot
      const float* lrow = lse2 + static_cast<size_t>(bh) * T;
      const float* drow = dsum + static_cast<size_t>(bh) * T;
      float nl[BT / 32], nd[BT / 32];
      auto fetch_rows = [&](int i) {
#pragma unroll
        for (int e = 0; e < BT / 32; ++e) {
          const int t = i * BT + e * 32 + lane;
          nl[e] = t < T ? -__ldg(lrow + t) : 0.0f;
          nd[e] = t < T ? -__ldg(drow + t) : 0.0f;
        }
      };
      fetch_rows(j);
      for (int i = j; i < n_qt; ++i, ++qcount) {
        const uint32_t qs = qcount % NQ;
        if (qcount >= NQ && !mbar_wait_warp(&bars->q_empty[qs], (qcount / NQ - 1) & 1u, abort_flag, err)) { ok = false; break; }
        float* ld = sLD + qs * (2 * BT);
#pragma unroll
        for (int e = 0; e < BT / 32; ++e) {
          const int ql = e * 32 + lane;
          const int o = (ql >> 1) * 4 + (ql & 1);
          ld[o] = nl[e];
          ld[o + 2] = nd[e];
        }
        __threadfence_block();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->q_full[qs], 2 * Cfg::TILE);
          tma_load_3d(sQ + qs * Cfg::TILE, &tm_qkv, &bars->q_full[qs], h * D, i * BT, b);
          tma_load_3d(sDY + qs * Cfg::TILE, &tm_dy, &bars->q_full[qs], h * D, i * BT, b);
        }
        issued_q |= 1u << qs;
        par_q = (par_q & ~(1u << qs)) | (((qcount / NQ) & 1u) << qs);
        if (i + 1 < n_qt) fetch_rows(i + 1);
      }
    }
    // never leave with copies in flight into this CTA's shared memory
    if (lane == 0) {
      for (int k = 0; k < 2; ++k)
        if (issued_kv & (1u << k)) mbar_wait_drain(&bars->kv_full[k], (par_kv >> k) & 1u);
      for (int k = 0; k < NQ; ++k)
        if (issued_q & (1u << k)) mbar_wait_drain(&bars->q_full[k], (par_q >> k) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (whole warp; one elected lane issues)
    const uint64_t dq0 = smem_desc(smem_u32(sQ), 16, 8 * Cfg::ROWB, Cfg::SWZ);       // K-major (B of S^T)
    const uint64_t dy0 = smem_desc(smem_u32(sDY), 16, 8 * Cfg::ROWB, Cfg::SWZ);      // K-major (B of dP^T)
    const uint64_t qmn0 = smem_desc(smem_u32(sQ), Cfg::TILE, 8 * Cfg::ROWB, Cfg::SWZ);   // MN-major (B of dK)
    const uint64_t dymn0 = smem_desc(smem_u32(sDY), Cfg::TILE, 8 * Cfg::ROWB, Cfg::SWZ); // MN-major (B of dU)
    const uint64_t kmn0 = smem_desc(smem_u32(sK), Cfg::TILE, 8 * Cfg::ROWB, Cfg::SWZ);   // MN-major (B of dQ)
    // dS: MN-major A (queries contiguous): 64-query atoms 16 KB apart, 8-key groups 1 KB apart
    const uint64_t ds0 = smem_desc(smem_u32(sDS), BT * 128, 1024, SWZ_128B);
    constexpr uint32_t id_s = idesc_bf16_f32(BT, HQ, false);
    constexpr uint32_t id_acc = idesc_bf16_f32(BT, D, true);                  // B MN-major
    constexpr uint32_t id_dq = idesc_bf16_f32(BT, D, true) | (1u << 15);      // A and B MN-major
    // S^T and dP^T of half g of the query tile in ring slot qs; A = K_j, U_j from tensor memory (a K step
    // of 16 dimensions: 8 columns)
    auto issue_scores = [&](int g, uint32_t qs) {
      const uint32_t qoff = qs * Cfg::TILE + g * HQ * Cfg::ROWB;
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        tc_mma_bf16_ts_warp(tmem_base + 128 * g, tmem_base + kColK + 8 * k, desc_add(dq0, qoff + k * 32), id_s,
                            k > 0 ? 1u : 0u);
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        tc_mma_bf16_ts_warp(tmem_base + 128 * g + 64, tmem_base + kColK + D / 2 + 8 * k, desc_add(dy0, qoff + k * 32),
                            id_s, k > 0 ? 1u : 0u);
      tc_commit_warp(&bars->s_full[g]);
    };
    // dU += P^T_g dY_g and dK += dS^T_g Q_g (a K step of 16 queries: 8 TMEM columns, 16 rows of dY / Q)
    auto issue_acc = [&](int g, uint32_t qs, bool first) {
      const uint32_t qoff = qs * Cfg::TILE + g * HQ * Cfg::ROWB;
#pragma unroll
      for (int kk = 0; kk < HQ / 16; ++kk)
        tc_mma_bf16_ts_warp(tmem_base + kColDU, tmem_base + 128 * g + 8 * kk, desc_add(dymn0, qoff + kk * 16 * Cfg::ROWB),
                            id_acc, (first && kk == 0) ? 0u : 1u);
#pragma unroll
      for (int kk = 0; kk < HQ / 16; ++kk)
        tc_mma_bf16_ts_warp(tmem_base + kColDK, tmem_base + 128 * g + 64 + 8 * kk,
                            desc_add(qmn0, qoff + kk * 16 * Cfg::ROWB), id_acc, (first && kk == 0) ? 0u : 1u);
    };
    int r = 0;
    const int item0 = next_item(bars, 0, abort_flag, err, lane);
    bool ok = item0 < n_items;
    int j = ok ? item0 / BH : 0, i = j, kb = 0;
    uint32_t qcount = 0, qs = 0, tiles = 0;
    if (ok)
      ok = mbar_wait_warp(&bars->kv_full[0], 0u, abort_flag, err) && mbar_wait_warp(&bars->q_full[0], 0u, abort_flag, err) &&
           mbar_wait_warp(&bars->kvt_full, 0u, abort_flag, err);
    if (ok) {
      tc_fence_after();
      issue_scores(0, qs);
      issue_scores(1, qs);
      if (i == n_qt - 1) tc_commit_warp(&bars->kvt_free);   // the item's last reads of K_j, U_j in TMEM
    }
    while (ok) {
      const bool first = i == j, last = i == n_qt - 1;
      if (!mbar_wait_warp(&bars->p_full[0], tiles & 1u, abort_flag, err)) break;
      // the previous item's dK and dU have been read out of the accumulators
      if (first && r > 0 && !mbar_wait_warp(&bars->acc_free, static_cast<uint32_t>(r - 1) & 1u, abort_flag, err)) break;
      tc_fence_after();
      issue_acc(0, qs, first);
      // the next query tile: the same item's, or the first of the next item
      bool has_next = !last;
      int r2 = r, j2 = j, i2 = i + 1, kb2 = kb;
      if (last) {
        const int item2 = next_item(bars, r + 1, abort_flag, err, lane);
        has_next = item2 < n_items;
        if (has_next) {
          r2 = r + 1;
          j2 = item2 / BH;
          i2 = j2;
          kb2 = r2 & 1;
          if (!mbar_wait_warp(&bars->kv_full[kb2], static_cast<uint32_t>(r2 >> 1) & 1u, abort_flag, err)) break;
          if (!mbar_wait_warp(&bars->kvt_full, static_cast<uint32_t>(r2) & 1u, abort_flag, err)) break;
        }
      }
      const uint32_t qcount2 = qcount + 1, qs2 = qcount2 % NQ;
      if (has_next) {
        if (!mbar_wait_warp(&bars->q_full[qs2], (qcount2 / NQ) & 1u, abort_flag, err)) break;
        tc_fence_after();
        issue_scores(0, qs2);
      }
      if (!mbar_wait_warp(&bars->p_full[1], tiles & 1u, abort_flag, err)) break;
      tc_fence_after();
      issue_acc(1, qs, false);
      tc_commit_warp(&bars->q_empty[qs]);            // Q_i and dY_i are consumed
      if (last) tc_commit_warp(&bars->acc_full);
      if (tiles > 0 && !mbar_wait_warp(&bars->dq_free, (tiles - 1) & 1u, abort_flag, err)) break;
      tc_fence_after();
      const uint32_t dsoff = (tiles & 1u) * Cfg::DS_BUF;
#pragma unroll
      for (int kk = 0; kk < BT / 16; ++kk)           // a K step of 16 keys: 16 rows of dS and of K_j
        tc_mma_bf16_warp(tmem_base + kColDQ, desc_add(ds0, dsoff + kk * 16 * 128),
                         desc_add(kmn0, kb * Cfg::TILE + kk * 16 * Cfg::ROWB), id_dq, kk > 0 ? 1u : 0u);
      tc_commit_warp(&bars->dq_full);
      if (last) tc_commit_warp(&bars->kv_empty[kb]);   // K_j and U_j are consumed
      if (!has_next) break;
      issue_scores(1, qs2);
      if (i2 == n_qt - 1) tc_commit_warp(&bars->kvt_free);
      r = r2;
      j = j2;
      i = i2;
      kb = kb2;
      qcount = qcount2;
      qs = qs2;
      ++tiles;
    }
    tc_commit_warp(&bars->drain);
    mbar_wait_drain(&bars->drain, 0);
  } else if (warp < 6) {
    // ------------------------------------------------ softmax derivative (thread = key row)
    const int sub = warp & 3;
    const int kr = sub * 32 + lane;                  // key row within the tile = TMEM lane
    const uint32_t tb = tmem_base + (static_cast<uint32_t>(sub * 32) << 16);
    uint32_t qcount = 0, tiles = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int item = next_item(bars, r, abort_flag, err, lane);
      if (item >= n_items) break;
      const int j = item / BH;
      for (int i = j; i < n_qt; ++i, ++qcount, ++tiles) {
        const uint32_t qs = qcount % NQ;
        if (!mbar_wait_warp(&bars->q_full[qs], (qcount / NQ) & 1u, abort_flag, err)) { ok = false; break; }
        const float4* ld = reinterpret_cast<const float4*>(sLD + qs * (2 * BT));
        uint8_t* ds_row = sDS + (tiles & 1u) * Cfg::DS_BUF + kr * 128;
#pragma unroll 1                                 // rolled, like the chunk loop inside: smaller code
        for (int g = 0; g < 2; ++g) {
          if (!mbar_wait_warp(&bars->s_full[g], tiles & 1u, abort_flag, err)) { ok = false; break; }
          tc_fence_after();
          // query i BT + 64 g + ql is kept for ql <= T - 1 - (i BT + 64 g) and, on the diagonal, ql >= kr - 64 g.
          // The choice of path depends on the tile only: the TMEM loads in it are warp-wide (.aligned).
          const int hi = T - 1 - (i * BT + g * HQ);
          const int lo = (i == j) ? kr - g * HQ : 0;
          if (i == j || hi < HQ - 1) {
            // bit ql set for the kept queries lo <= ql <= hi
            const uint64_t below_hi = hi < 0 ? 0ull : (hi >= HQ - 1 ? ~0ull : (2ull << hi) - 1ull);
            const uint64_t from_lo = lo >= HQ ? 0ull : (~0ull << (lo > 0 ? lo : 0));
            derivative_half<true>(tb + 128 * g, ld + 32 * g, sl2, below_hi & from_lo, ds_row + g * (BT * 128), kr);
          } else {
            derivative_half<false>(tb + 128 * g, ld + 32 * g, sl2, ~0ull, ds_row + g * (BT * 128), kr);
          }
          tmem_st_wait();
          fence_proxy_async_smem();                  // dS in shared memory is read by the dQ product
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->p_full[g]);
        }
        if (!ok) break;
      }
    }
  } else {
    // ------------------------------------------------ output: dQ reduce-adds and conversion, dK and dU stores
    const int sub = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    uint8_t* stg = smem_raw + Cfg::OFF_STG + (warp - 6) * 8192;
    // K_j and U_j (item buffer kb) into tensor memory as the scores' A operands: this warp's 32 key rows,
    // each row's D values as bf16 pairs
    auto stage_kv = [&](int kb) {
      constexpr int ROWB = Cfg::ROWB;
      const int kr = sub * 32 + lane;
      const uint8_t* krow = sK + kb * Cfg::TILE + kr * ROWB;
      const uint8_t* urow = sU + kb * Cfg::TILE + kr * ROWB;
      uint32_t kw[D / 2], uw[D / 2];
#pragma unroll
      for (int u = 0; u < ROWB / 16; ++u) {
        const uint4 a = *reinterpret_cast<const uint4*>(krow + (swz_unit(ROWB, kr, u) << 4));
        const uint4 c = *reinterpret_cast<const uint4*>(urow + (swz_unit(ROWB, kr, u) << 4));
        kw[4 * u] = a.x; kw[4 * u + 1] = a.y; kw[4 * u + 2] = a.z; kw[4 * u + 3] = a.w;
        uw[4 * u] = c.x; uw[4 * u + 1] = c.y; uw[4 * u + 2] = c.z; uw[4 * u + 3] = c.w;
      }
      if constexpr (D == 64) {
        tmem_st_32x32b_x32(tmem_base + lane_off + kColK, kw);
        tmem_st_32x32b_x32(tmem_base + lane_off + kColK + D / 2, uw);
      } else {
        tmem_st_32x32b_x16(tmem_base + lane_off + kColK, kw);
        tmem_st_32x32b_x16(tmem_base + lane_off + kColK + D / 2, uw);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->kvt_full);
    };
    uint32_t tiles = 0;
    bool ok = true;
    int item = next_item(bars, 0, abort_flag, err, lane);
    if (item < n_items) {
      ok = mbar_wait_warp(&bars->kv_full[0], 0u, abort_flag, err);
      if (ok) stage_kv(0);
    }
    for (int r = 0; ok && item < n_items; ++r) {
      const int j = item / BH, bh = item - j * BH, b = bh / H, h = bh - b * H;
      int item_next = 0x7fffffff;
      for (int i = j; i < n_qt; ++i, ++tiles) {
        if (i == n_qt - 1) {
          // before the item's last dQ: the next item's K_j, U_j, once the item's last scores have read theirs
          item_next = next_item(bars, r + 1, abort_flag, err, lane);
          if (item_next < n_items) {
            if (!mbar_wait_warp(&bars->kvt_free, static_cast<uint32_t>(r) & 1u, abort_flag, err) ||
                !mbar_wait_warp(&bars->kv_full[(r + 1) & 1], static_cast<uint32_t>((r + 1) >> 1) & 1u, abort_flag, err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            stage_kv((r + 1) & 1);
          }
        }
        if (!mbar_wait_warp(&bars->dq_full, tiles & 1u, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
        uint32_t v[D];
        if constexpr (D == 64) {
          tmem_ld_32x32b_x64(tmem_base + kColDQ + lane_off, *reinterpret_cast<uint32_t (*)[64]>(v));
        } else {
          tmem_ld_32x32b_x32(tmem_base + kColDQ + lane_off, *reinterpret_cast<uint32_t (*)[32]>(v));
        }
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->dq_free);
        if (lane == 0) bulk_wait_read_all();         // the previous copies have read the staging boxes
        __syncwarp();
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {        // 32 fp32 columns (128 bytes) per box row
          uint8_t* box = stg + cc * 4096 + lane * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(box + (swz_unit(128, lane, u) << 4)) =
                make_uint4(v[32 * cc + 4 * u], v[32 * cc + 4 * u + 1], v[32 * cc + 4 * u + 2], v[32 * cc + 4 * u + 3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc)
            tma_reduce_add_3d(&tm_dq, stg + cc * 4096, h * D + 32 * cc, i * BT + sub * 32, b);
          bulk_commit();
        }
      }
      if (!ok) break;
      // the item's dK and dU
      if (!mbar_wait_warp(&bars->acc_full, static_cast<uint32_t>(r) & 1u, abort_flag, err)) { ok = false; break; }
      tc_fence_after();
      uint32_t kv[D], uv[D];
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t (&k32)[32] = *reinterpret_cast<uint32_t (*)[32]>(kv + 32 * cc);
        uint32_t (&u32)[32] = *reinterpret_cast<uint32_t (*)[32]>(uv + 32 * cc);
        tmem_ld_32x32b_x32(tmem_base + kColDK + lane_off + 32 * cc, k32);
        tmem_ld_32x32b_x32(tmem_base + kColDU + lane_off + 32 * cc, u32);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_free);
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
      constexpr int ROWB = Cfg::ROWB;
#pragma unroll
      for (int u = 0; u < ROWB / 16; ++u) {          // bf16 rows of D values: dK / sqrt(D) in box 0, dU in box 1
        const uint4 wk = make_uint4(pack_bf16x2(__uint_as_float(kv[8 * u]) * rsd, __uint_as_float(kv[8 * u + 1]) * rsd),
                                    pack_bf16x2(__uint_as_float(kv[8 * u + 2]) * rsd, __uint_as_float(kv[8 * u + 3]) * rsd),
                                    pack_bf16x2(__uint_as_float(kv[8 * u + 4]) * rsd, __uint_as_float(kv[8 * u + 5]) * rsd),
                                    pack_bf16x2(__uint_as_float(kv[8 * u + 6]) * rsd, __uint_as_float(kv[8 * u + 7]) * rsd));
        const uint4 wu = make_uint4(pack_bf16x2(__uint_as_float(uv[8 * u]), __uint_as_float(uv[8 * u + 1])),
                                    pack_bf16x2(__uint_as_float(uv[8 * u + 2]), __uint_as_float(uv[8 * u + 3])),
                                    pack_bf16x2(__uint_as_float(uv[8 * u + 4]), __uint_as_float(uv[8 * u + 5])),
                                    pack_bf16x2(__uint_as_float(uv[8 * u + 6]), __uint_as_float(uv[8 * u + 7])));
        *reinterpret_cast<uint4*>(stg + lane * ROWB + (swz_unit(ROWB, lane, u) << 4)) = wk;
        *reinterpret_cast<uint4*>(stg + 4096 + lane * ROWB + (swz_unit(ROWB, lane, u) << 4)) = wu;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_3d(&tm_dkv, stg, C + h * D, j * BT + sub * 32, b);
        tma_store_3d(&tm_dkv, stg + 4096, 2 * C + h * D, j * BT + sub * 32, b);
        bulk_commit();
      }
      item = item_next;
    }
    if (lane == 0) bulk_wait_all();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
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

// Dsum[(b H + h) T + t] = sum_d dY[b, t, h D + d] Y[b, t, h D + d]: one warp per row, D / 8 lanes per
// head with 16-byte loads, so each load instruction of the warp reads 512 contiguous bytes of the row.
template <int D>
__global__ void __launch_bounds__(256)
attn_bwd_dsum_kernel(const __nv_bfloat16* __restrict__ y, const __nv_bfloat16* __restrict__ dy, float* __restrict__ dsum,
                     int M, int T, int H) {
  pdl_wait();
  pdl_trigger();
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  constexpr int LPH = D / 8;
  const int C = H * D, nv = C / 8;
  const uint4* a4 = reinterpret_cast<const uint4*>(dy + static_cast<size_t>(row) * C);
  const uint4* o4 = reinterpret_cast<const uint4*>(y + static_cast<size_t>(row) * C);
  const int b = static_cast<int>(row / T), t = static_cast<int>(row - static_cast<long long>(b) * T);
  for (int v0 = 0; v0 < nv; v0 += 32) {            // nv is a multiple of LPH: a head's lanes are all in or all out
    const int v = v0 + lane;
    float acc = 0.0f;
    if (v < nv) {
      const uint4 a = __ldg(a4 + v), o = __ldg(o4 + v);
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 x = unpack_bf16x2(aw[k]), z = unpack_bf16x2(ow[k]);
        acc = fmaf(x.x, z.x, fmaf(x.y, z.y, acc));
      }
    }
#pragma unroll
    for (int o = LPH / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (v < nv && (lane % LPH) == 0) dsum[(static_cast<size_t>(b) * H + v / LPH) * T + t] = acc;
  }
}

// dqkv[m, c] (the first C columns of each 3C row) = bf16(dqacc[m, c] / sqrt(D)): four consecutive floats
// per thread and step, so each warp access covers 512 contiguous bytes.
__global__ void __launch_bounds__(256)
attn_bwd_dq_convert_kernel(const float* __restrict__ dqacc, __nv_bfloat16* __restrict__ dqkv, int M, int C, float rsd) {
  pdl_wait();
  pdl_trigger();
  const int c4n = C / 4;
  const long long n = static_cast<long long>(M) * c4n;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(e / c4n), c = static_cast<int>(e - static_cast<long long>(m) * c4n) * 4;
    const float4 a = __ldg(reinterpret_cast<const float4*>(dqacc) + e);
    *reinterpret_cast<uint2*>(dqkv + static_cast<size_t>(m) * 3 * C + c) =
        make_uint2(pack_bf16x2(a.x * rsd, a.y * rsd), pack_bf16x2(a.z * rsd, a.w * rsd));
  }
}

template <int D>
cudaError_t launch_bwd_d(const CUtensorMap& tm_qkv, const CUtensorMap& tm_dy, const CUtensorMap& tm_dkv,
                         const CUtensorMap& tm_dq, const void* y, const void* dy, const float* lse2, float* dsum,
                         float* dqacc, void* dqkv, int B, int T, int H, int* err, int* sched, cudaStream_t s) {
  using Cfg = BwdCfg<D>;
  static bool attr_set = false;
  static int num_sms = 0;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int M = B * T;
  const int n_qt = (T + BT - 1) / BT;
  const long long items = static_cast<long long>(n_qt) * B * H;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const float rsd = 1.0f / sqrtf(static_cast<float>(D));
  const float sl2 = rsd * kLog2e;
  cudaError_t e = cudaMemsetAsync(dqacc, 0, static_cast<size_t>(M) * H * D * sizeof(float), s);
  if (e != cudaSuccess) return e;
  e = launch_k(attn_bwd_dsum_kernel<D>, dim3(static_cast<unsigned>((M + 7) / 8)), dim3(256), 0, s,
                           static_cast<const __nv_bfloat16*>(y), static_cast<const __nv_bfloat16*>(dy), dsum, M, T, H);
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  e = launch_k(attn_bwd_tc_kernel<D>, dim3(grid), dim3(THREADS), static_cast<size_t>(Cfg::SMEM), s, tm_qkv, tm_dy,
               tm_dkv, tm_dq, static_cast<const float*>(lse2), static_cast<const float*>(dsum), B, T, H, n_qt, sl2, rsd,
               err, sched);
  if (e != cudaSuccess) return e;
  const long long n4 = static_cast<long long>(M) * (H * D / 4);
  const long long cblocks = (n4 + 255) / 256;
  const int cgrid = static_cast<int>(cblocks < 8LL * num_sms ? cblocks : 8LL * num_sms);
  return launch_k(attn_bwd_dq_convert_kernel, dim3(cgrid), dim3(256), 0, s, static_cast<const float*>(dqacc),
                  static_cast<__nv_bfloat16*>(dqkv), M, H * D, rsd);
}

}  // namespace

cudaError_t launch_attention_bwd_tc(const CUtensorMap& tm_qkv, const CUtensorMap& tm_dy, const CUtensorMap& tm_dkv,
                                    const CUtensorMap& tm_dq, const void* y, const void* dy, const float* lse2,
                                    float* dsum, float* dqacc, void* dqkv, int B, int T, int H, int D, int* err,
                                    int* sched, cudaStream_t s) {
  if (B <= 0 || T <= 0) return cudaSuccess;
  if (!sched || !lse2 || !dsum || !dqacc || !dqkv) return cudaErrorInvalidValue;
  if (D == 64) return launch_bwd_d<64>(tm_qkv, tm_dy, tm_dkv, tm_dq, y, dy, lse2, dsum, dqacc, dqkv, B, T, H, err, sched, s);
  if (D == 32) return launch_bwd_d<32>(tm_qkv, tm_dy, tm_dkv, tm_dq, y, dy, lse2, dsum, dqacc, dqkv, B, T, H, err, sched, s);
  return cudaErrorInvalidValue;
}

}  // namespace gptgb
