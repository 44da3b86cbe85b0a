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
// Per query tile, in tensor memory (key = TMEM lane):
//   S^T  = K_j Q_i^T      M=128 keys, N=128 queries, K=D    columns [0, 128)
//   dP^T = U_j dY_i^T     M=128, N=128, K=D                 columns [128, 256)
// Four derivative warps (one thread per key) form P^T = 2^(S^T log2(e)/sqrt(D) - lse2[q]) and
// dS^T = P^T (dP^T - Dsum[q]) (zero above the diagonal and past T), write both back as bf16 pairs over
// the first 64 columns of their fp32 tiles, and dS^T also into shared memory (as the MN-major A operand
// of the dQ product). Then
//   dU_j += P^T dY_i      A from tensor memory, B = dY_i read MN-major        columns [256, 256 + D)
//   dK_j += dS^T Q_i      A from tensor memory, B = Q_i read MN-major         columns [320, 320 + D)
//   dQ_i  = dS K_j        A = dS from shared memory (MN-major), B = K_j       columns [384, 384 + D)
// Four output warps add each dQ_i tile into an fp32 [B][T][C] buffer with TMA reduce-adds (a query tile
// gets one from every key tile it sees: no atomics on single elements, no ordering needed) and, at the
// end of an item, store dK_j / sqrt(D) and dU_j into dqkv with TMA stores. A last small kernel turns the
// fp32 dQ into bf16 (x 1/sqrt(D)) and zeroes the buffer again.
// The score tiles of the next query tile are issued after the previous tile's dQ product, so when the
// derivative warps see them, every earlier MMA (and its reads of the dS tile in shared memory) is done.
// Warp roles (320 threads, one persistent CTA per SM):
//   warp 0      producer: takes work items; K_j, U_j per item (two buffers), then Q_i, dY_i by TMA and
//               the rows' lse2 and Dsum (plain loads) into a two-stage ring
//   warp 1      TMEM allocator and MMA issuer (the whole warp runs the loop, one elected lane issues)
//   warps 2-5   softmax derivative (thread = key row)
//   warps 6-9   output: dQ reduce-adds, dK and dU stores
#include "common.cuh"
#include "kernels.h"
#include "launch.h"

#include <math.h>

namespace gptgb {

namespace {

constexpr int BT = 128;                 // rows per key or query tile
constexpr int THREADS = 320;
constexpr int TMEM_COLS = 512;
constexpr int NQ = 2;                   // query-tile ring stages
constexpr int SR = 8;                   // work-item ring slots
constexpr int kConsumers = 9;           // warps that read each announced item: MMA + 4 derivative + 4 output
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kColS = 0, kColDP = 128, kColDU = 256, kColDK = 320, kColDQ = 384;

template <int D>
struct BwdCfg {
  static constexpr int ROWB = D * 2;                              // bytes per row of a Q/K/U/dY tile
  static constexpr uint32_t SWZ = (ROWB == 128) ? SWZ_128B : SWZ_64B;
  static constexpr int TILE = BT * ROWB;
  static constexpr int OFF_K = 0;                                   // [2] item buffers
  static constexpr int OFF_U = 2 * TILE;                            // [2]
  static constexpr int OFF_Q = 4 * TILE;                            // [NQ]
  static constexpr int OFF_DY = OFF_Q + NQ * TILE;                  // [NQ]
  static constexpr int OFF_LSE = OFF_DY + NQ * TILE;                // [NQ][128] fp32
  static constexpr int OFF_DSUM = OFF_LSE + NQ * BT * 4;            // [NQ][128] fp32
  static constexpr int OFF_DS = (OFF_DSUM + NQ * BT * 4 + 1023) / 1024 * 1024;   // dS: 2 atoms x 128 rows x 128 B
  static constexpr int DS_BYTES = 2 * BT * 128;
  static constexpr int OFF_STG = OFF_DS + DS_BYTES;                 // 4 output warps x 2 boxes of 4 KB
  static constexpr int OFF_BAR = OFF_STG + 4 * 8192;
  static constexpr int SMEM = (OFF_BAR + 512 > 120 * 1024) ? OFF_BAR + 512 : 120 * 1024;
  static_assert(D == 32 || D == 64, "head width");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct __align__(8) BwdBars {
  uint64_t kv_full[2], kv_empty[2];     // K_j, U_j of an item (buffer r % 2)
  uint64_t q_full[NQ], q_empty[NQ];     // Q_i, dY_i, lse2 and Dsum of a query tile
  uint64_t s_full;                      // S^T and dP^T of the current tile are in tensor memory
  uint64_t p_full;                      // the derivative warps wrote P^T, dS^T (4 warps)
  uint64_t dq_full;                     // the current tile's dQ product has completed
  uint64_t dq_free;                     // the output warps read it out of tensor memory (4 warps)
  uint64_t acc_full;                    // the item's dK and dU are complete
  uint64_t acc_free;                    // the output warps read them (4 warps)
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
    }
    for (int i = 0; i < NQ; ++i) {
      mbar_init(&bars->q_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->p_full, 4);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_free, 4);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_free, 4);
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
  float* sLse = reinterpret_cast<float*>(smem_raw + Cfg::OFF_LSE);
  float* sDsum = reinterpret_cast<float*>(smem_raw + Cfg::OFF_DSUM);
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
      for (int i = j; i < n_qt; ++i, ++qcount) {
        const uint32_t qs = qcount % NQ;
        if (qcount >= NQ && !mbar_wait_warp(&bars->q_empty[qs], (qcount / NQ - 1) & 1u, abort_flag, err)) { ok = false; break; }
        // the rows' log-sum-exp and Dsum (plain loads; rows past T read nothing)
        const float* lrow = lse2 + static_cast<size_t>(bh) * T;
        const float* drow = dsum + static_cast<size_t>(bh) * T;
#pragma unroll
        for (int e = 0; e < BT / 32; ++e) {
          const int t = i * BT + e * 32 + lane;
          sLse[qs * BT + e * 32 + lane] = t < T ? __ldg(lrow + t) : 0.0f;
          sDsum[qs * BT + e * 32 + lane] = t < T ? __ldg(drow + t) : 0.0f;
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
    const uint64_t dk0 = smem_desc(smem_u32(sK), 16, 8 * Cfg::ROWB, Cfg::SWZ);       // K-major (A of S^T)
    const uint64_t du0 = smem_desc(smem_u32(sU), 16, 8 * Cfg::ROWB, Cfg::SWZ);       // K-major (A of dP^T)
    const uint64_t dq0 = smem_desc(smem_u32(sQ), 16, 8 * Cfg::ROWB, Cfg::SWZ);       // K-major (B of S^T)
    const uint64_t dy0 = smem_desc(smem_u32(sDY), 16, 8 * Cfg::ROWB, Cfg::SWZ);      // K-major (B of dP^T)
    const uint64_t qmn0 = smem_desc(smem_u32(sQ), Cfg::TILE, 8 * Cfg::ROWB, Cfg::SWZ);   // MN-major (B of dK)
    const uint64_t dymn0 = smem_desc(smem_u32(sDY), Cfg::TILE, 8 * Cfg::ROWB, Cfg::SWZ); // MN-major (B of dU)
    const uint64_t kmn0 = smem_desc(smem_u32(sK), Cfg::TILE, 8 * Cfg::ROWB, Cfg::SWZ);   // MN-major (B of dQ)
    // dS: MN-major A (queries contiguous): 64-query atoms 16 KB apart, 8-key groups 1 KB apart
    const uint64_t ds0 = smem_desc(smem_u32(sDS), BT * 128, 1024, SWZ_128B);
    constexpr uint32_t id_s = idesc_bf16_f32(BT, BT, false);
    constexpr uint32_t id_acc = idesc_bf16_f32(BT, D, true);                  // B MN-major
    constexpr uint32_t id_dq = idesc_bf16_f32(BT, D, true) | (1u << 15);      // A and B MN-major
    uint32_t qcount = 0, tiles = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int item = next_item(bars, r, abort_flag, err, lane);
      if (item >= n_items) break;
      const int j = item / BH;
      const int kb = r & 1;
      if (!mbar_wait_warp(&bars->kv_full[kb], static_cast<uint32_t>(r >> 1) & 1u, abort_flag, err)) break;
      for (int i = j; i < n_qt && ok; ++i, ++qcount, ++tiles) {
        const uint32_t qs = qcount % NQ;
        if (!mbar_wait_warp(&bars->q_full[qs], (qcount / NQ) & 1u, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          tc_mma_bf16_warp(tmem_base + kColS, desc_add(dk0, kb * Cfg::TILE + k * 32), desc_add(dq0, qs * Cfg::TILE + k * 32),
                           id_s, k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          tc_mma_bf16_warp(tmem_base + kColDP, desc_add(du0, kb * Cfg::TILE + k * 32),
                           desc_add(dy0, qs * Cfg::TILE + k * 32), id_s, k > 0 ? 1u : 0u);
        tc_commit_warp(&bars->s_full);
        if (!mbar_wait_warp(&bars->p_full, tiles & 1u, abort_flag, err)) { ok = false; break; }
        // the previous item's dK and dU have been read out of the accumulators
        if (i == j && r > 0 && !mbar_wait_warp(&bars->acc_free, static_cast<uint32_t>(r - 1) & 1u, abort_flag, err)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)           // a K step of 16 queries: 8 columns of P^T, 16 rows of dY
          tc_mma_bf16_ts_warp(tmem_base + kColDU, tmem_base + kColS + 8 * kk,
                              desc_add(dymn0, qs * Cfg::TILE + kk * 16 * Cfg::ROWB), id_acc, (i > j || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
          tc_mma_bf16_ts_warp(tmem_base + kColDK, tmem_base + kColDP + 8 * kk,
                              desc_add(qmn0, qs * Cfg::TILE + kk * 16 * Cfg::ROWB), id_acc, (i > j || kk > 0) ? 1u : 0u);
        tc_commit_warp(&bars->q_empty[qs]);            // Q_i and dY_i are consumed
        if (tiles > 0 && !mbar_wait_warp(&bars->dq_free, (tiles - 1) & 1u, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)           // a K step of 16 keys: 16 rows of dS and of K_j
          tc_mma_bf16_warp(tmem_base + kColDQ, desc_add(ds0, kk * 16 * 128),
                           desc_add(kmn0, kb * Cfg::TILE + kk * 16 * Cfg::ROWB), id_dq, kk > 0 ? 1u : 0u);
        tc_commit_warp(&bars->dq_full);
        if (i == n_qt - 1) {
          tc_commit_warp(&bars->acc_full);
          tc_commit_warp(&bars->kv_empty[kb]);         // K_j and U_j are consumed
        }
      }
    }
    tc_commit_warp(&bars->drain);
    mbar_wait_drain(&bars->drain, 0);
  } else if (warp < 6) {
    // ------------------------------------------------ softmax derivative (thread = key row)
    const int sub = warp & 3;
    const int kr = sub * 32 + lane;                  // key row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    const uint32_t tS = tmem_base + kColS + lane_off;
    const uint32_t tP = tmem_base + kColDP + lane_off;
    uint8_t* ds_row = sDS + kr * 128;                // this key's row in both 64-query atoms
    uint32_t qcount = 0, tiles = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int item = next_item(bars, r, abort_flag, err, lane);
      if (item >= n_items) break;
      const int j = item / BH;
      const int key = j * BT + kr;
      for (int i = j; i < n_qt; ++i, ++qcount, ++tiles) {
        const uint32_t qs = qcount % NQ;
        if (!mbar_wait_warp(&bars->q_full[qs], (qcount / NQ) & 1u, abort_flag, err) ||
            !mbar_wait_warp(&bars->s_full, tiles & 1u, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
        const float* lse = sLse + qs * BT;
        const float* dsm = sDsum + qs * BT;
        const bool diag = i == j;
#pragma unroll 1
        for (int c = 0; c < BT / 32; ++c) {          // 32 queries at a time
          uint32_t sv[32], dv[32];
          tmem_ld_32x32b_x32(tS + 32 * c, sv);
          tmem_ld_32x32b_x32(tP + 32 * c, dv);
          tmem_ld_wait();
          uint32_t pp[16], pd[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float p2[2], d2[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int ql = 32 * c + e + h2;
              const int q = i * BT + ql;
              const bool valid = q < T && (!diag || key <= q);
              const float p = ex2_approx(fmaf(__uint_as_float(sv[e + h2]), sl2, -lse[ql]));
              p2[h2] = valid ? p : 0.0f;
              d2[h2] = valid ? p * (__uint_as_float(dv[e + h2]) - dsm[ql]) : 0.0f;
            }
            pp[e >> 1] = pack_bf16x2(p2[0], p2[1]);
            pd[e >> 1] = pack_bf16x2(d2[0], d2[1]);
          }
          // P^T and dS^T over columns [16 c, 16 c + 16) of their tiles (already read), dS^T into shared memory
          tmem_st_32x32b_x16(tS + 16 * c, pp);
          tmem_st_32x32b_x16(tP + 16 * c, pd);
          uint8_t* atom = ds_row + (c >> 1) * (BT * 128);
#pragma unroll
          for (int u4 = 0; u4 < 4; ++u4) {
            const int u = (c & 1) * 4 + u4;            // 16-byte unit (8 queries) within the 64-query atom
            *reinterpret_cast<uint4*>(atom + (swz_unit(128, kr, u) << 4)) =
                make_uint4(pd[4 * u4], pd[4 * u4 + 1], pd[4 * u4 + 2], pd[4 * u4 + 3]);
          }
        }
        tmem_st_wait();
        fence_proxy_async_smem();                    // dS in shared memory is read by the dQ product
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full);
      }
    }
  } else {
    // ------------------------------------------------ output: dQ reduce-adds, dK and dU stores
    const int sub = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    uint8_t* stg = smem_raw + Cfg::OFF_STG + (warp - 6) * 8192;
    uint32_t tiles = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int item = next_item(bars, r, abort_flag, err, lane);
      if (item >= n_items) break;
      const int j = item / BH, bh = item - j * BH, b = bh / H, h = bh - b * H;
      for (int i = j; i < n_qt; ++i, ++tiles) {
        if (!mbar_wait_warp(&bars->dq_full, tiles & 1u, abort_flag, err)) { ok = false; break; }
        tc_fence_after();
        uint32_t v[D];
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t (&v32)[32] = *reinterpret_cast<uint32_t (*)[32]>(v + 32 * cc);
          tmem_ld_32x32b_x32(tmem_base + kColDQ + lane_off + 32 * cc, v32);
        }
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->dq_free);
        if (lane == 0) bulk_wait_read_all();         // the previous stores have read the staging boxes
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
      if (!mbar_wait_warp(&bars->acc_full, static_cast<uint32_t>(r) & 1u, abort_flag, err)) break;
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

// Dsum[(b H + h) T + t] = sum_d dY[b, t, h D + d] Y[b, t, h D + d]: one thread per (row, head).
template <int D>
__global__ void __launch_bounds__(256)
attn_bwd_dsum_kernel(const __nv_bfloat16* __restrict__ y, const __nv_bfloat16* __restrict__ dy, float* __restrict__ dsum,
                     int M, int T, int H) {
  pdl_wait();
  pdl_trigger();
  const long long id = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (id >= static_cast<long long>(M) * H) return;
  const int m = static_cast<int>(id / H), h = static_cast<int>(id - static_cast<long long>(m) * H);
  const int C = H * D;
  const uint4* a4 = reinterpret_cast<const uint4*>(dy + static_cast<size_t>(m) * C + h * D);
  const uint4* o4 = reinterpret_cast<const uint4*>(y + static_cast<size_t>(m) * C + h * D);
  float acc = 0.0f;
#pragma unroll
  for (int v = 0; v < D / 8; ++v) {
    const uint4 a = __ldg(a4 + v), o = __ldg(o4 + v);
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 x = unpack_bf16x2(aw[k]), z = unpack_bf16x2(ow[k]);
      acc = fmaf(x.x, z.x, fmaf(x.y, z.y, acc));
    }
  }
  const int b = m / T, t = m - b * T;
  dsum[(static_cast<size_t>(b) * H + h) * T + t] = acc;
}

// dqkv[m, c] (the first C columns of each 3C row) = bf16(dqacc[m, c] / sqrt(D)); dqacc = 0 again.
__global__ void __launch_bounds__(256)
attn_bwd_dq_convert_kernel(float* __restrict__ dqacc, __nv_bfloat16* __restrict__ dqkv, int M, int C, float rsd) {
  pdl_wait();
  pdl_trigger();
  const long long id = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;   // 8 columns each
  const int cpr = C / 8;
  if (id >= static_cast<long long>(M) * cpr) return;
  const int m = static_cast<int>(id / cpr), c = static_cast<int>(id - static_cast<long long>(m) * cpr) * 8;
  float4* src = reinterpret_cast<float4*>(dqacc + static_cast<size_t>(m) * C + c);
  const float4 a = src[0], b = src[1];
  src[0] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  src[1] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  *reinterpret_cast<uint4*>(dqkv + static_cast<size_t>(m) * 3 * C + c) =
      make_uint4(pack_bf16x2(a.x * rsd, a.y * rsd), pack_bf16x2(a.z * rsd, a.w * rsd), pack_bf16x2(b.x * rsd, b.y * rsd),
                 pack_bf16x2(b.z * rsd, b.w * rsd));
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
  const int M = B * T, C = H * D;
  const int n_qt = (T + BT - 1) / BT;
  const long long items = static_cast<long long>(n_qt) * B * H;
  if (items <= 0) return cudaSuccess;
  if (items > 0x7fffffffLL) return cudaErrorInvalidValue;
  const float rsd = 1.0f / sqrtf(static_cast<float>(D));
  const float sl2 = rsd * kLog2e;
  const long long nd = static_cast<long long>(M) * H;
  cudaError_t e = launch_k(attn_bwd_dsum_kernel<D>, dim3(static_cast<unsigned>((nd + 255) / 256)), dim3(256), 0, s,
                           static_cast<const __nv_bfloat16*>(y), static_cast<const __nv_bfloat16*>(dy), dsum, M, T, H);
  if (e != cudaSuccess) return e;
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  e = launch_k(attn_bwd_tc_kernel<D>, dim3(grid), dim3(THREADS), Cfg::SMEM, s, tm_qkv, tm_dy, tm_dkv, tm_dq, lse2,
               static_cast<const float*>(dsum), B, T, H, n_qt, sl2, rsd, err, sched);
  if (e != cudaSuccess) return e;
  const long long nc = static_cast<long long>(M) * (C / 8);
  return launch_k(attn_bwd_dq_convert_kernel, dim3(static_cast<unsigned>((nc + 255) / 256)), dim3(256), 0, s, dqacc,
                  static_cast<__nv_bfloat16*>(dqkv), M, C, rsd);
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
