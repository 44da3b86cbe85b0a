// gpt_backward and gpt_grad: the gradient of the mean next-token cross-entropy
// with respect to every parameter of a bf16 model, the back-propagation step
// of the training loop in "预训练一个 Mini GPT" (训练循环).
//
// Sequence (M = B*T tokens; every product is a tcgen05 GEMM out = A . B^T: the
// input-gradient products read transposed copies of the weights, the
// weight-gradient products read the stored activations as MN-major operands):
//   forward + loss, keeping every block's input and activations (and c_fc's pre-activation)
//   head: dz = (softmax(z) - onehot) / M in bf16 straight from the GEMM that
//         recomputes z = h E^T (the row's log-sum-exp from the forward's loss);
//         dh = dz E; dE += dz^T h ("第 25 章" §25.4: the tied table's two uses add)
//   ln_f: dx = LN'(x_L) dh
//   per block, last to first, from its kept activations:
//         dW_mp += dx^T g, db_mp, du = (dx W_mp) gelu'(u) (one GEMM), dW_fc += du^T a2,
//         db_fc, da2 = du W_fc, LN2', dW_proj += ds1^T y, db_proj, dy = ds1 W_proj,
//         attention' -> dqkv, dW_attn += dqkv^T a1, db_attn, da1 = dqkv W_attn, LN1'
//   embedding: dE[id] += dx_0, dP[t] += dx_0.
// Weight gradients with few output tiles split K (the token axis) and add their
// partials with reduce-add stores into the zeroed fp32 gradient.
#include "launch.h"
#include "model.h"

#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <vector>

using namespace gptgb;

struct gpt_layer_grad {
  float *attn_w, *attn_b, *proj_w, *proj_b, *fc_w, *fc_b, *mp_w, *mp_b, *ln1_g, *ln1_b, *ln2_g, *ln2_b;
  CUtensorMap tg_attn_w, tg_proj_w, tg_fc_w, tg_mp_w;      // fp32 reduce-add targets
  void *attn_wT, *proj_wT, *fc_wT, *mp_wT;                  // bf16 transposed weights [in, out]
  CUtensorMap tb_attn_wT, tb_proj_wT, tb_fc_wT, tb_mp_wT;  // as B operands
  CUtensorMap tb_attn_wT_pair, tb_fc_wT_pair;                // the same with 128-row boxes (CTA pairs)
};

// One block's activations from the training forward (kept for its backward).
struct gpt_layer_act {
  float* x = nullptr;            // block input [M, C] fp32
  void *a1, *qkv, *y, *a2, *u, *g;   // bf16: ln_1 output (post-norm: x itself), c_attn out, attention
                                     // out, ln_2 output (post-norm: n), c_fc pre- and post-GELU
  float *s1, *n, *s2;            // fp32: x + attention branch; post-norm: LN1(s1), n + MLP branch
  float* lse2 = nullptr;         // the attention rows' base-2 log-sum-exp [B*H][T] (from the forward)
  CUtensorMap A_a1, A_y, A_a2, A_g;        // as GEMM A operands
  CUtensorMap K_a1, K_y, K_a2, K_g;        // as MN-major operands of the weight-gradient products
  CUtensorMap C_qkv, C_u, C_g, Q3;         // as epilogue outputs; qkv as the attention input
};

struct gpt_train {
  size_t Mx = 0;                 // token capacity (max_tokens)
  int Vp = 0;                    // V rounded up to 8 (row stride of dz and E^T)
  uint8_t* buf = nullptr;        // one allocation for everything below
  size_t grad_floats = 0;
  float* gbuf = nullptr;         // all gradients, contiguous
  float *g_wte = nullptr, *g_wpe = nullptr, *g_lnf_g = nullptr, *g_lnf_b = nullptr;
  float* g_head = nullptr;       // the untied head's gradient (nullptr when tied)
  std::vector<gpt_layer_grad> lg;
  std::vector<gpt_layer_act> la;
  CUtensorMap tg_wte, tg_head;
  void* wteT = nullptr;          // the head's matrix (E when tied) transposed: [C][Vp] bf16
  CUtensorMap tb_wteT;
  CUtensorMap tb_wteT_pair;      // the same with 128-row boxes (CTA pairs)
  bool wT_ready = false;
  // gradients of activations
  float *dx, *da;
  void *dxb, *dyb, *dqkv, *du;
  float *lse2, *dsum;
  float* dqacc = nullptr;        // fp32 [M, C] dQ accumulator of the attention derivative (scratch)
  CUtensorMap T_dy, T_dkv, T_dq; // dy, dqkv and dqacc as the attention derivative's TMA operands
  void* dz;
  // activation maps, for one (B, T)
  int mB = -1, mT = -1;
  CUtensorMap A_dz, A_dxb, A_du, A_dqkv;
  CUtensorMap K_dz, K_h, K_dxb, K_du, K_dqkv;    // MN-major operands (64-row boxes)
  CUtensorMap C_dz, C_du, C_dyb, C_da, C_dx;
  int launches = 0;
  // AdamW state (allocated by the first gpt_adamw_step): fp32 master weights and both moments, in the
  // gradients' layout, and the parameter segments
  float *master = nullptr, *m1 = nullptr, *m2 = nullptr;
  OptSeg* d_segs = nullptr;
  int nseg = 0;
  int opt_t = 0;
};

namespace gptgb {
void free_train(gpt_model* m) {
  if (!m || !m->tr) return;
  cudaFree(m->tr->master);
  cudaFree(m->tr->d_segs);
  cudaFree(m->tr->buf);
  delete m->tr;
  m->tr = nullptr;
}
}  // namespace gptgb

namespace {

int cu(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return GPT_OK;
  set_detail(what, e);
  return GPT_ECUDA;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Bump allocator over one buffer: the first pass sizes it, the second hands out pointers.
struct Carve {
  uint8_t* base = nullptr;
  size_t off = 0;
  void* take(size_t bytes) {
    off = align_up(off, 256);
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
};

int alloc_train(gpt_model* m) {
  const gpt_config& c = m->cfg;
  const size_t Mx = static_cast<size_t>(c.max_tokens), C = c.C, F = c.ffn, V = c.V, L = c.L, ctx = c.ctx;
  const size_t Vp = (V + 7) / 8 * 8;
  gpt_train* t = new gpt_train();
  t->Mx = Mx;
  t->Vp = static_cast<int>(Vp);
  t->lg.resize(L);
  t->la.resize(L);
  const size_t per_layer_grad = 3 * C * C + 3 * C + C * C + C + F * C + F + C * F + C + 4 * C;
  const size_t head_grad = c.untied_head ? V * C : 0;
  t->grad_floats = V * C + ctx * C + 2 * C + head_grad + L * per_layer_grad;
  // sizes, then one allocation
  auto layout = [&](Carve& cv) {
    t->gbuf = static_cast<float*>(cv.take(t->grad_floats * 4));
    t->wteT = cv.take(C * Vp * 2);
    for (size_t l = 0; l < L; ++l) {
      gpt_layer_grad& g = t->lg[l];
      g.attn_wT = cv.take(3 * C * C * 2);
      g.proj_wT = cv.take(C * C * 2);
      g.fc_wT = cv.take(F * C * 2);
      g.mp_wT = cv.take(C * F * 2);
    }
    const bool post = c.norm_mode != 0;
    for (size_t l = 0; l < L; ++l) {
      gpt_layer_act& q = t->la[l];
      q.x = static_cast<float*>(cv.take(Mx * C * 4));
      q.a1 = cv.take(Mx * C * 2);
      q.qkv = cv.take(Mx * 3 * C * 2);
      q.y = cv.take(Mx * C * 2);
      q.a2 = cv.take(Mx * C * 2);
      q.u = cv.take(Mx * F * 2);
      q.g = cv.take(Mx * F * 2);
      q.s1 = static_cast<float*>(cv.take(Mx * C * 4));
      q.n = post ? static_cast<float*>(cv.take(Mx * C * 4)) : nullptr;
      q.s2 = post ? static_cast<float*>(cv.take(Mx * C * 4)) : nullptr;
      q.lse2 = static_cast<float*>(cv.take(Mx * c.H * 4));
    }
    t->dx = static_cast<float*>(cv.take(Mx * C * 4));
    t->da = static_cast<float*>(cv.take(Mx * C * 4));
    t->dxb = cv.take(Mx * C * 2);
    t->dyb = cv.take(Mx * C * 2);
    t->dqkv = cv.take(Mx * 3 * C * 2);
    t->du = cv.take(Mx * F * 2);
    t->lse2 = static_cast<float*>(cv.take(Mx * c.H * 4));
    t->dsum = static_cast<float*>(cv.take(Mx * c.H * 4));
    t->dqacc = static_cast<float*>(cv.take(Mx * C * 4));
    t->dz = cv.take(Mx * Vp * 2);
  };
  Carve sizing;
  layout(sizing);
  if (cudaMalloc(&t->buf, sizing.off) != cudaSuccess) {
    cudaGetLastError();
    delete t;
    return GPT_ENOMEM;
  }
  Carve real;
  real.base = t->buf;
  layout(real);
  // gradient pointers in the order of the weights
  float* p = t->gbuf;
  auto take = [&](size_t n) { float* q = p; p += n; return q; };
  t->g_wte = take(V * C);
  t->g_wpe = take(ctx * C);
  t->g_lnf_g = take(C);
  t->g_lnf_b = take(C);
  if (head_grad) t->g_head = take(head_grad);
  for (size_t l = 0; l < L; ++l) {
    gpt_layer_grad& g = t->lg[l];
    g.ln1_g = take(C); g.ln1_b = take(C);
    g.attn_w = take(3 * C * C); g.attn_b = take(3 * C);
    g.proj_w = take(C * C); g.proj_b = take(C);
    g.ln2_g = take(C); g.ln2_b = take(C);
    g.fc_w = take(F * C); g.fc_b = take(F);
    g.mp_w = take(C * F); g.mp_b = take(C);
  }
  // fixed descriptors: gradient reduce-add targets and transposed weights
  bool ok = make_tmap_2d(&t->tg_wte, t->g_wte, 4, V, C, 32, kEpiRows) &&
            make_tmap_2d_bf16(&t->tb_wteT, t->wteT, C, V, gemm_tc_bn(), Vp) &&
            make_tmap_2d_bf16(&t->tb_wteT_pair, t->wteT, C, V, kGemmBM, Vp) &&
            (!t->g_head || make_tmap_2d(&t->tg_head, t->g_head, 4, V, C, 32, kEpiRows));
  for (size_t l = 0; l < L && ok; ++l) {
    gpt_layer_grad& g = t->lg[l];
    ok = make_tmap_2d(&g.tg_attn_w, g.attn_w, 4, 3 * C, C, 32, kEpiRows) &&
         make_tmap_2d(&g.tg_proj_w, g.proj_w, 4, C, C, 32, kEpiRows) &&
         make_tmap_2d(&g.tg_fc_w, g.fc_w, 4, F, C, 32, kEpiRows) &&
         make_tmap_2d(&g.tg_mp_w, g.mp_w, 4, C, F, 32, kEpiRows) &&
         make_tmap_2d_bf16(&g.tb_attn_wT, g.attn_wT, C, 3 * C, gemm_tc_bn()) &&
         make_tmap_2d_bf16(&g.tb_proj_wT, g.proj_wT, C, C, gemm_tc_bn()) &&
         make_tmap_2d_bf16(&g.tb_fc_wT, g.fc_wT, C, F, gemm_tc_bn()) &&
         make_tmap_2d_bf16(&g.tb_mp_wT, g.mp_wT, F, C, gemm_tc_bn()) &&
         make_tmap_2d_bf16(&g.tb_attn_wT_pair, g.attn_wT, C, 3 * C, kGemmBM) &&
         make_tmap_2d_bf16(&g.tb_fc_wT_pair, g.fc_wT, C, F, kGemmBM);
  }
  if (!ok) {
    cudaFree(t->buf);
    delete t;
    set_detail_text("backward tensor map");
    return GPT_ECUDA;
  }
  m->tr = t;
  return GPT_OK;
}

}  // namespace

namespace {

// Activation descriptors for one (B, T): A operands (128-row boxes), B operands (256-row
// boxes), epilogue outputs (bf16 64 x 32 or fp32 32 x 32 boxes) and the attention input.
int ensure_bwd_maps(gpt_model* m, gpt_train* t, int B, int T) {
  if (t->mB == B && t->mT == T) return GPT_OK;
  const gpt_config& c = m->cfg;
  const uint64_t M = static_cast<uint64_t>(B) * T, C = c.C, F = c.ffn, V = c.V, Vp = t->Vp;
  const uint32_t BA = kGemmBM, BB = gemm_tc_bn();
  const uint32_t BK = kGemmBK;
  bool ok =
      make_tmap_2d_bf16(&t->A_dz, t->dz, M, V, BA, Vp) && make_tmap_2d_bf16(&t->A_dxb, t->dxb, M, C, BA) &&
      make_tmap_2d_bf16(&t->A_du, t->du, M, F, BA) && make_tmap_2d_bf16(&t->A_dqkv, t->dqkv, M, 3 * C, BA) &&
      make_tmap_2d_bf16(&t->K_dz, t->dz, M, V, BK, Vp) && make_tmap_2d_bf16(&t->K_h, m->a, M, C, BK) &&
      make_tmap_2d_bf16(&t->K_dxb, t->dxb, M, C, BK) && make_tmap_2d_bf16(&t->K_du, t->du, M, F, BK) &&
      make_tmap_2d_bf16(&t->K_dqkv, t->dqkv, M, 3 * C, BK) &&
      make_tmap_2d(&t->C_dz, t->dz, 2, M, V, 64, kEpiRows, Vp) &&
      make_tmap_2d(&t->C_du, t->du, 2, M, F, 64, kEpiRows) && make_tmap_2d(&t->C_dyb, t->dyb, 2, M, C, 64, kEpiRows) &&
      make_tmap_2d(&t->C_da, t->da, 4, M, C, 32, kEpiRows) && make_tmap_2d(&t->C_dx, t->dx, 4, M, C, 32, kEpiRows) &&
      make_tmap_qkv(&t->T_dy, t->dyb, B, T, C, C / c.H) && make_tmap_attn_out(&t->T_dkv, t->dqkv, B, T, 3 * C, C / c.H) &&
      make_tmap_bt_f32(&t->T_dq, t->dqacc, B, T, C);
  for (size_t l = 0; l < t->la.size() && ok; ++l) {
    gpt_layer_act& q = t->la[l];
    ok = make_tmap_2d_bf16(&q.A_a1, q.a1, M, C, BA) && make_tmap_2d_bf16(&q.A_y, q.y, M, C, BA) &&
         make_tmap_2d_bf16(&q.A_a2, q.a2, M, C, BA) && make_tmap_2d_bf16(&q.A_g, q.g, M, F, BA) &&
         make_tmap_2d_bf16(&q.K_a1, q.a1, M, C, BK) && make_tmap_2d_bf16(&q.K_y, q.y, M, C, BK) &&
         make_tmap_2d_bf16(&q.K_a2, q.a2, M, C, BK) && make_tmap_2d_bf16(&q.K_g, q.g, M, F, BK) &&
         make_tmap_2d(&q.C_qkv, q.qkv, 2, M, 3 * C, 64, kEpiRows) && make_tmap_2d(&q.C_u, q.u, 2, M, F, 64, kEpiRows) &&
         make_tmap_2d(&q.C_g, q.g, 2, M, F, 64, kEpiRows) && make_tmap_qkv(&q.Q3, q.qkv, B, T, 3 * C, C / c.H);
  }
  if (!ok) {
    t->mB = t->mT = -1;
    set_detail_text("backward activation tensor map");
    return GPT_ECUDA;
  }
  t->mB = B;
  t->mT = T;
  return GPT_OK;
}

// Slices along the token axis for a weight-gradient product of `tiles` output tiles: the count whose
// (tile, slice) units fill one or two waves of the grid best, the fewest slices among equally full ones
// (a slice's partial tile costs one reduce-add of the tile), at least 4 K blocks per slice. Dealing
// about two units per CTA regardless of the wave fill left a third wave of 2 units for the 18-tile
// attention projection (306 units on 152 CTAs) and 2.4 waves for the 72-tile MLP products.
int grad_ksplit(int tiles, int KB, int grid) {
  if (tiles >= grid) return 1;
  const int ks_max = KB / 4 > 1 ? KB / 4 : 1;
  int best_ks = 1;
  double best = -1.0;
  for (int ks = 1; ks <= ks_max; ++ks) {
    const long long units = static_cast<long long>(tiles) * ks;
    if (units > 2LL * grid) break;
    const long long waves = (units + grid - 1) / grid;
    const double fill = static_cast<double>(units) / static_cast<double>(waves * grid);
    if (fill > best + 0.02) {
      best = fill;
      best_ks = ks;
    }
  }
  return best_ks;
}

// Slices along K for a long product added into an fp32 output zeroed before it (dh = dz E, K = V): the
// count, at most 8 and at least 48 K blocks per slice, whose (tile, slice) units fill the waves best, the
// fewest among equally full ones. Dealt tile by tile, the units of one wave hold the three N tiles of the
// same rows at the same K slice, so each A slice comes from DRAM once and is reused from L2; stream-K's
// contiguous ranges put those three tiles at different K offsets, and with K = V the A rows in use
// (12.9 MB per 128-row block) do not stay in L2 between them.
int long_k_split(int tiles, int KB, int grid) {
  int best_ks = 1;
  double best = -1.0;
  for (int ks = 1; ks <= 8 && KB / ks >= 48; ++ks) {
    const long long units = static_cast<long long>(tiles) * ks;
    const long long waves = (units + grid - 1) / grid;
    const double fill = static_cast<double>(units) / static_cast<double>(waves * grid);
    if (fill > best + 0.02) {
      best = fill;
      best_ks = ks;
    }
  }
  return best_ks;
}

// A weight-gradient product: out [N0, N1] fp32 += A^T B summed over the M tokens, A [M, N0] and
// B [M, N1] the activations as stored (MN-major operands, maps with 64-row boxes), split along M
// (grad_ksplit).
int grad_gemm(gpt_model* m, const CUtensorMap& A, const CUtensorMap& Bm, const CUtensorMap& out_map, float* out,
              int N0, int N1, int M, cudaStream_t s) {
  GemmArgs a{};
  a.M = N0; a.N = N1; a.K = M;
  a.out = out;
  a.ldo = N1;
  a.err = m->err;
  a.m_fastest = (N1 > N0) ? 1 : 0;
  a.mn_major = 1;
  const int KB = (M + kGemmBK - 1) / kGemmBK;
  const int pairs = pair_enabled() ? gemm_pair_capacity() : 0;
  if (pairs > 0) {                        // CTA pairs: 256 x 256 tiles, the same boxes (two per operand and CTA)
    const int grid = pairs < m->num_sms / 2 ? pairs : m->num_sms / 2;
    const int tiles = ((N0 + 2 * kGemmBM - 1) / (2 * kGemmBM)) * gemm_tc_num_ntiles(N1);
    a.ksplit = grad_ksplit(tiles, KB, grid);
    if (a.ksplit == 1) {
      a.sk_part = m->sk_part;
      a.sk_flag = m->sk_flag;
    }
    GPT_CUDA(launch_gemm_pair(A, Bm, out_map, a, EPI_BIAS_RESID, m->num_sms / 2, s));
    return GPT_OK;
  }
  const int tiles = ((N0 + kGemmBM - 1) / kGemmBM) * gemm_tc_num_ntiles(N1);
  const int ks = grad_ksplit(tiles, KB, m->num_sms);
  a.ksplit = ks;
  if (ks == 1) {                          // enough tiles: whole tiles (stream-K where it applies)
    a.sk_part = m->sk_part;
    a.sk_flag = m->sk_flag;
  }
  GPT_CUDA(launch_gemm_tc(A, Bm, out_map, a, EPI_BIAS_RESID, m->num_sms, s));
  return GPT_OK;
}

}  // namespace

namespace {

#define BW(expr)                   \
  do {                             \
    const int rc_ = (expr);        \
    if (rc_ != GPT_OK) return rc_; \
    ++t->launches;                 \
  } while (0)

// A timed step of the backward: the armed probe's events around it (as GPT_STEP in the forward).
#define BWS(step, layer, expr)                                                        \
  do {                                                                                \
    const bool hit_ = m->prof_ev0 != nullptr && m->prof_step == (step) &&             \
                      ((layer) < 0 || m->prof_layer == (layer));                      \
    if (hit_) GPT_CUDA(cudaEventRecord(m->prof_ev0, s));                              \
    BW(expr);                                                                         \
    if (hit_) {                                                                       \
      GPT_CUDA(cudaEventRecord(m->prof_ev1, s));                                      \
      ++m->probe_hits;                                                                \
    }                                                                                 \
  } while (0)

// The transposed weights the input-gradient products read: made by the first backward and
// again after each gpt_adamw_step (which changes the weights).
int prepare_weights(gpt_model* m, gpt_train* t, cudaStream_t s) {
  if (t->wT_ready) return GPT_OK;
  const gpt_config& c = m->cfg;
  const int C = c.C, F = c.ffn, V = c.V;
  BW(cu(launch_transpose_bf16(m->head, V, C, C, t->wteT, t->Vp, s), "transpose head"));
  for (int l = 0; l < c.L; ++l) {
    const gpt_layer_dev& w = m->layers[l];
    gpt_layer_grad& g = t->lg[l];
    BW(cu(launch_transpose_bf16(w.attn_w, 3 * C, C, C, g.attn_wT, 3 * C, s), "transpose attn_w"));
    BW(cu(launch_transpose_bf16(w.proj_w, C, C, C, g.proj_wT, C, s), "transpose proj_w"));
    BW(cu(launch_transpose_bf16(w.fc_w, F, C, C, g.fc_wT, F, s), "transpose fc_w"));
    BW(cu(launch_transpose_bf16(w.mp_w, C, F, F, g.mp_wT, C, s), "transpose mp_w"));
  }
  t->wT_ready = true;
  return GPT_OK;
}

// The head and ln_f: dx = d loss / d x_L (the last block's output) in t->dx.
int head_backward(gpt_model* m, gpt_train* t, const int32_t* tg, int M, cudaStream_t s) {
  const gpt_config& c = m->cfg;
  const int C = c.C, V = c.V;
  // dz = (softmax(h E^T) - onehot) / M, bf16 [M, V] (row stride Vp)
  GemmArgs a{};
  a.M = M; a.N = V; a.K = C;
  a.out = t->dz;
  a.ldo = t->Vp;
  a.targets = tg;
  a.row_nll = m->nll;
  a.ztgt = m->ztgt;
  a.scale = 1.0f / static_cast<float>(M);
  a.err = m->err;
  a.m_fastest = 1;
  a.b_const = 1;                          // the token table
  BWS(GPT_STEP_B_DZ, -1, cu(launch_gemm_tc(m->tm_a, m->tm_head, t->C_dz, a, EPI_CE_GRAD, m->num_sms, s), "head grad"));
  // dE += dz^T h (the head's share of the tied table), or the untied head's gradient
  if (t->g_head)
    BWS(GPT_STEP_B_DE, -1, grad_gemm(m, t->K_dz, t->K_h, t->tg_head, t->g_head, V, C, M, s));
  else
    BWS(GPT_STEP_B_DE, -1, grad_gemm(m, t->K_dz, t->K_h, t->tg_wte, t->g_wte, V, C, M, s));
  // dh = dz E (fp32 into da)
  GPT_CUDA(cudaMemsetAsync(t->da, 0, static_cast<size_t>(M) * C * sizeof(float), s));
  {
    GemmArgs a{};
    a.M = M; a.N = C; a.K = V;
    a.out = t->da;
    a.ldo = C;
    a.err = m->err;
    a.b_const = 1;
    const int KB = (V + kGemmBK - 1) / kGemmBK;
    const int pairs = pair_enabled() ? gemm_pair_capacity() : 0;
    if (pairs > 0) {                       // CTA pairs: 256 x 256 tiles
      const int tiles = ((M + 2 * kGemmBM - 1) / (2 * kGemmBM)) * gemm_tc_num_ntiles(C);
      a.ksplit = long_k_split(tiles, KB, pairs < m->num_sms / 2 ? pairs : m->num_sms / 2);
    } else {
      const int tiles = ((M + kGemmBM - 1) / kGemmBM) * gemm_tc_num_ntiles(C);
      a.ksplit = long_k_split(tiles, KB, m->num_sms);
    }
    if (a.ksplit == 1) {
      a.sk_part = m->sk_part;
      a.sk_flag = m->sk_flag;
    }
    if (pairs > 0)
      BWS(GPT_STEP_B_DH, -1,
          cu(launch_gemm_pair(t->A_dz, t->tb_wteT_pair, t->C_da, a, EPI_BIAS_RESID, m->num_sms / 2, s), "dh"));
    else
      BWS(GPT_STEP_B_DH, -1, cu(launch_gemm_tc(t->A_dz, t->tb_wteT, t->C_da, a, EPI_BIAS_RESID, m->num_sms, s), "dh"));
  }
  if (c.final_ln) {
    BW(cu(launch_layernorm_bwd(m->x, m->lnf_g, t->da, t->dx, 0, t->g_lnf_g, t->g_lnf_b, M, C, c.ln_eps, m->num_sms, s),
          "ln_f backward"));
  } else {
    GPT_CUDA(cudaMemcpyAsync(t->dx, t->da, static_cast<size_t>(M) * C * sizeof(float), cudaMemcpyDeviceToDevice, s));
  }
  return GPT_OK;
}

// The forward pass and loss with every block's activations kept: the kernels and their order are
// those of gpt_forward (so the loss is the same bit for bit), only the outputs go to per-block
// buffers. c_fc also runs without its GELU, for the pre-activation the derivative needs.
int train_forward(gpt_model* m, gpt_train* t, const int32_t* ids, const int32_t* tg, int B, int T, float* d_loss,
                  cudaStream_t s) {
  const gpt_config& c = m->cfg;
  const int M = B * T, C = c.C, F = c.ffn, L = c.L;
  const bool pre = c.norm_mode == 0;
  const float eps = c.ln_eps;
  const size_t MC4 = static_cast<size_t>(M) * C * sizeof(float);
  {
    int out_mode = 1;
    const float* g = nullptr;
    const float* b = nullptr;
    if (pre) {
      if (L > 0) { out_mode = 2; g = m->layers[0].ln1_g; b = m->layers[0].ln1_b; }
      else if (c.final_ln) { out_mode = 2; g = m->lnf_g; b = m->lnf_b; }
    }
    void* out = L > 0 ? t->la[0].a1 : m->a;
    BW(cu(launch_embed(ids, m->wte, m->wpe, 1, m->x, out, out_mode, 1, g, b, M, T, C, c.V, eps, m->err, s), "embed"));
  }
  for (int l = 0; l < L; ++l) {
    const gpt_layer_dev& w = m->layers[l];
    gpt_layer_act& q = t->la[l];
    void* next_a = (l + 1 < L) ? t->la[l + 1].a1 : m->a;
    GPT_CUDA(cudaMemcpyAsync(q.x, m->x, MC4, cudaMemcpyDeviceToDevice, s));
    BW(gemm_bf16_long(m, q.A_a1, w.tm_attn_w, w.tm_attn_w_pair, q.C_qkv, M, 3 * C, C, w.attn_b, q.qkv, EPI_BIAS_OUT, s));
    BW(cu(launch_attention_tc(q.Q3, q.y, B, T, c.H, C / c.H, m->err, m->attn_sched, s, q.lse2), "attention"));
    BW(gemm_bf16(m, q.A_y, w.tm_proj_w, m->tm_x_out, M, C, C, w.proj_b, m->x, EPI_BIAS_RESID, s));
    GPT_CUDA(cudaMemcpyAsync(q.s1, m->x, MC4, cudaMemcpyDeviceToDevice, s));
    if (pre) {
      BW(cu(launch_layernorm(m->x, w.ln2_g, w.ln2_b, q.a2, 1, nullptr, M, C, eps, s), "ln2"));
    } else {
      BW(cu(launch_layernorm(m->x, w.ln1_g, w.ln1_b, q.a2, 1, m->x, M, C, eps, s), "ln1"));
      GPT_CUDA(cudaMemcpyAsync(q.n, m->x, MC4, cudaMemcpyDeviceToDevice, s));
    }
    BW(gemm_bf16_gelu_u(m, q.A_a2, w.tm_fc_w, q.C_g, q.C_u, M, F, C, w.fc_b, q.g, s));   // g and u in one product
    BW(gemm_bf16_long(m, q.A_g, w.tm_mp_w, w.tm_mp_w_pair, m->tm_x_out, M, C, F, w.mp_b, m->x, EPI_BIAS_RESID, s));
    if (pre) {
      const float* g = nullptr;
      const float* b = nullptr;
      if (l + 1 < L) { g = m->layers[l + 1].ln1_g; b = m->layers[l + 1].ln1_b; }
      else if (c.final_ln) { g = m->lnf_g; b = m->lnf_b; }
      BW(cu(launch_layernorm(m->x, g, b, next_a, 1, nullptr, M, C, eps, s), "ln"));
    } else {
      GPT_CUDA(cudaMemcpyAsync(q.s2, m->x, MC4, cudaMemcpyDeviceToDevice, s));
      BW(cu(launch_layernorm(m->x, w.ln2_g, w.ln2_b, next_a, 1, m->x, M, C, eps, s), "ln2"));
    }
  }
  if (!pre && c.final_ln)
    BW(cu(launch_layernorm(m->x, m->lnf_g, m->lnf_b, m->a, 1, nullptr, M, C, eps, s), "ln_f"));
  // tied head with the cross-entropy partials, then the loss
  GemmArgs a{};
  a.M = M; a.N = c.V; a.K = C;
  a.ldo = c.V;
  a.targets = tg;
  a.pmax = m->pmax;
  a.psum = m->psum;
  a.ztgt = m->ztgt;
  a.err = m->err;
  a.m_fastest = 1;
  a.b_const = 1;
  BW(cu(launch_gemm_tc(m->tm_a, m->tm_head, m->tm_a, a, EPI_CE, m->num_sms, s), "head"));
  BW(cu(launch_ce_combine(m->pmax, m->psum, m->ztgt, tg, m->nll, m->block_sums, M, gemm_tc_num_ntiles(c.V), c.V,
                          m->err, s),
        "ce_combine"));
  if (d_loss) BW(cu(launch_mean(m->block_sums, ce_combine_blocks(M), M, d_loss, s), "mean"));
  return GPT_OK;
}

}  // namespace

namespace {

// Block l backward: on entry t->dx = d loss / d (block output), on return d loss / d x_l.
int block_backward(gpt_model* m, gpt_train* t, int l, int B, int T, cudaStream_t s) {
  const gpt_config& c = m->cfg;
  const int M = B * T, C = c.C, F = c.ffn, H = c.H;
  const bool pre = c.norm_mode == 0;
  const float eps = c.ln_eps;
  const gpt_layer_dev& w = m->layers[l];
  gpt_layer_grad& g = t->lg[l];
  const gpt_layer_act& q = t->la[l];
  const float* xl = q.x;
  if (!pre)      // x_{l+1} = LN2(s2): d loss / d s2, in place
    BW(cu(launch_layernorm_bwd(q.s2, w.ln2_g, t->dx, t->dx, 0, g.ln2_g, g.ln2_b, M, C, eps, m->num_sms, s), "ln2'"));
  // MLP: s2 = n + g W_mp^T + b_mp, g = gelu(u), u = a2 W_fc^T + b_fc
  BW(cu(launch_cast_transpose(t->dx, M, C, t->dxb, nullptr, 0, s, g.mp_b), "cast dx, db_mp"));
  BWS(GPT_STEP_B_MP_W, l, grad_gemm(m, t->K_dxb, q.K_g, g.tg_mp_w, g.mp_w, C, F, M, s));
  {                                   // du = (dx W_mp) * gelu'(u), the GELU's derivative in the epilogue
    GemmArgs a{};
    a.M = M; a.N = F; a.K = C;
    a.out = t->du;
    a.ldo = F;
    a.gelu_erf = c.gelu;
    a.aux = q.u;
    a.err = m->err;
    a.m_fastest = (F > M) ? 1 : 0;
    a.b_const = 1;
    BWS(GPT_STEP_B_DG, l, cu(launch_gemm_tc(t->A_dxb, g.tb_mp_wT, t->C_du, a, EPI_GELU_GRAD, m->num_sms, s), "dg"));
  }
  BW(cu(launch_colsum(t->du, 1, M, F, F, g.fc_b, m->num_sms, s), "db_fc"));
  BWS(GPT_STEP_B_FC_W, l, grad_gemm(m, t->K_du, q.K_a2, g.tg_fc_w, g.fc_w, F, C, M, s));
  if (pre) {
    // da2 = du W_fc; s1 -> LN2 -> a2: dx += LN2'(da2)
    BWS(GPT_STEP_B_DA2, l, gemm_bf16_long(m, t->A_du, g.tb_fc_wT, g.tb_fc_wT_pair, t->C_da, M, C, F, nullptr, t->da,
                                          EPI_F32_OUT, s));
    BW(cu(launch_layernorm_bwd(q.s1, w.ln2_g, t->da, t->dx, 1, g.ln2_g, g.ln2_b, M, C, eps, m->num_sms, s), "ln2'"));
  } else {
    // dn = ds2 + du W_fc; n = LN1(s1): d loss / d s1 in place
    BWS(GPT_STEP_B_DA2, l, gemm_bf16_long(m, t->A_du, g.tb_fc_wT, g.tb_fc_wT_pair, t->C_dx, M, C, F, nullptr, t->dx,
                                          EPI_BIAS_RESID, s));
    BW(cu(launch_layernorm_bwd(q.s1, w.ln1_g, t->dx, t->dx, 0, g.ln1_g, g.ln1_b, M, C, eps, m->num_sms, s), "ln1'"));
  }
  // attention: s1 = x + y W_proj^T + b_proj, y = attention(qkv), qkv = a1 W_attn^T + b_attn
  BW(cu(launch_cast_transpose(t->dx, M, C, t->dxb, nullptr, 0, s, g.proj_b), "cast ds1, db_proj"));
  BWS(GPT_STEP_B_PROJ_W, l, grad_gemm(m, t->K_dxb, q.K_y, g.tg_proj_w, g.proj_w, C, C, M, s));
  BWS(GPT_STEP_B_DY, l, gemm_bf16(m, t->A_dxb, g.tb_proj_wT, t->C_dyb, M, C, C, nullptr, t->dyb, EPI_BIAS_OUT, s));
  BWS(GPT_STEP_B_ATTN, l,
      cu(launch_attention_bwd_tc(q.Q3, t->T_dy, t->T_dkv, t->T_dq, q.y, t->dyb, q.lse2, t->dsum, t->dqacc, t->dqkv, B,
                                 T, H, C / H, m->err, m->attn_sched, s),
         "attention'"));
  t->launches += 2;                                          // three kernels: Dsum, the derivative, dQ to bf16
  BW(cu(launch_colsum(t->dqkv, 1, M, 3 * C, 3 * C, g.attn_b, m->num_sms, s), "db_attn"));
  BWS(GPT_STEP_B_ATTN_W, l, grad_gemm(m, t->K_dqkv, q.K_a1, g.tg_attn_w, g.attn_w, 3 * C, C, M, s));
  if (pre) {
    // da1 = dqkv W_attn; x -> LN1 -> a1: dx += LN1'(da1)
    BWS(GPT_STEP_B_DA1, l, gemm_bf16_long(m, t->A_dqkv, g.tb_attn_wT, g.tb_attn_wT_pair, t->C_da, M, C, 3 * C, nullptr,
                                          t->da, EPI_F32_OUT, s));
    BW(cu(launch_layernorm_bwd(xl, w.ln1_g, t->da, t->dx, 1, g.ln1_g, g.ln1_b, M, C, eps, m->num_sms, s), "ln1'"));
  } else {
    // a1 = x: dx += dqkv W_attn
    BWS(GPT_STEP_B_DA1, l, gemm_bf16_long(m, t->A_dqkv, g.tb_attn_wT, g.tb_attn_wT_pair, t->C_dx, M, C, 3 * C, nullptr,
                                          t->dx, EPI_BIAS_RESID, s));
  }
  return GPT_OK;
}

}  // namespace

extern "C" {

int gpt_backward(gpt_model* m, const int32_t* d_ids, const int32_t* d_targets, int32_t B, int32_t T, float* d_loss,
                 void* stream) {
  if (!m || !d_ids || !d_targets) return GPT_EINVAL;
  if (!m->bf16) return GPT_ECONFIG;
  int rc = shape_ok(m, B, T);
  if (rc != GPT_OK) return rc;
  const int M = B * T;
  if (!m->tr) {
    rc = alloc_train(m);
    if (rc != GPT_OK) return rc;
  }
  gpt_train* t = m->tr;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const gpt_config& c = m->cfg;
  t->launches = 0;
  rc = prepare_weights(m, t, s);
  if (rc != GPT_OK) return rc;
  rc = ensure_bwd_maps(m, t, B, T);
  if (rc != GPT_OK) return rc;
  GPT_CUDA(cudaMemsetAsync(t->gbuf, 0, t->grad_floats * sizeof(float), s));
  // forward and loss, keeping every block's input
  m->launches = 0;
  m->probe_hits = 0;
  rc = forward_maps(m, B, T);
  if (rc == GPT_OK) rc = train_forward(m, t, d_ids, d_targets, B, T, d_loss, s);
  if (rc == GPT_OK) rc = head_backward(m, t, d_targets, M, s);
  for (int l = c.L - 1; l >= 0 && rc == GPT_OK; --l) rc = block_backward(m, t, l, B, T, s);
  if (rc == GPT_OK) rc = cu(launch_embed_bwd(t->dx, d_ids, t->g_wte, t->g_wpe, M, T, c.C, c.V, s), "embedding'");
  m->prof_ev0 = m->prof_ev1 = nullptr;            // a probe covers one call
  m->prof_step = m->prof_layer = -1;
  if (rc != GPT_OK) return rc;
  m->launches = t->launches + 1;                 // + the embedding derivative
  return GPT_OK;
}

int gpt_grad(const gpt_model* m, int param, int layer, float** d_grad, int64_t* numel) {
  if (!m || !d_grad || !m->tr) return GPT_EINVAL;
  const gpt_config& c = m->cfg;
  const int64_t C = c.C, F = c.ffn;
  const gpt_train* t = m->tr;
  float* p = nullptr;
  int64_t n = 0;
  if (param <= GPT_P_LNF_B || param == GPT_P_HEAD) {
    switch (param) {
      case GPT_P_WTE: p = t->g_wte; n = static_cast<int64_t>(c.V) * C; break;
      case GPT_P_WPE: p = t->g_wpe; n = static_cast<int64_t>(c.ctx) * C; break;
      case GPT_P_LNF_G: p = t->g_lnf_g; n = C; break;
      case GPT_P_LNF_B: p = t->g_lnf_b; n = C; break;
      case GPT_P_HEAD:
        if (!t->g_head) return GPT_EINVAL;
        p = t->g_head; n = static_cast<int64_t>(c.V) * C; break;
      default: return GPT_EINVAL;
    }
  } else {
    if (layer < 0 || layer >= c.L) return GPT_EINVAL;
    const gpt_layer_grad& g = t->lg[layer];
    switch (param) {
      case GPT_P_LN1_G: p = g.ln1_g; n = C; break;
      case GPT_P_LN1_B: p = g.ln1_b; n = C; break;
      case GPT_P_ATTN_W: p = g.attn_w; n = 3 * C * C; break;
      case GPT_P_ATTN_B: p = g.attn_b; n = 3 * C; break;
      case GPT_P_PROJ_W: p = g.proj_w; n = C * C; break;
      case GPT_P_PROJ_B: p = g.proj_b; n = C; break;
      case GPT_P_LN2_G: p = g.ln2_g; n = C; break;
      case GPT_P_LN2_B: p = g.ln2_b; n = C; break;
      case GPT_P_FC_W: p = g.fc_w; n = F * C; break;
      case GPT_P_FC_B: p = g.fc_b; n = F; break;
      case GPT_P_MP_W: p = g.mp_w; n = C * F; break;
      case GPT_P_MP_B: p = g.mp_b; n = C; break;
      default: return GPT_EINVAL;
    }
  }
  *d_grad = p;
  if (numel) *numel = n;
  return GPT_OK;
}

}  // extern "C"

extern "C" int gpt_grad_copy(const gpt_model* m, int param, int layer, float* d_dst, void* stream) {
  if (!d_dst) return GPT_EINVAL;
  float* src = nullptr;
  int64_t n = 0;
  const int rc = gpt_grad(m, param, layer, &src, &n);
  if (rc != GPT_OK) return rc;
  GPT_CUDA(cudaMemcpyAsync(d_dst, src, static_cast<size_t>(n) * sizeof(float), cudaMemcpyDeviceToDevice,
                           reinterpret_cast<cudaStream_t>(stream)));
  return GPT_OK;
}

namespace {

// The optimiser's segment table (gradient order) and state, once.
int alloc_optimizer(gpt_model* m, gpt_train* t) {
  const gpt_config& c = m->cfg;
  const long long C = c.C, F = c.ffn;
  std::vector<OptSeg> segs;
  auto add = [&](const float* g, long long n, void* dst, bool matrix) {
    if (dst == nullptr) return;
    OptSeg sg;
    sg.off = g - t->gbuf;
    sg.n = n;
    sg.dst = dst;
    sg.bf16 = (matrix && m->bf16) ? 1 : 0;
    sg.decay = matrix ? 1 : 0;
    segs.push_back(sg);
  };
  add(t->g_wte, static_cast<long long>(c.V) * C, m->wte, true);
  add(t->g_wpe, static_cast<long long>(c.ctx) * C, m->wpe, true);
  add(t->g_lnf_g, C, m->lnf_g, false);
  add(t->g_lnf_b, C, m->lnf_b, false);
  if (t->g_head) add(t->g_head, static_cast<long long>(c.V) * C, m->head, true);
  for (int l = 0; l < c.L; ++l) {
    const gpt_layer_grad& g = t->lg[l];
    const gpt_layer_dev& w = m->layers[l];
    add(g.ln1_g, C, w.ln1_g, false);
    add(g.ln1_b, C, w.ln1_b, false);
    add(g.attn_w, 3 * C * C, w.attn_w, true);
    add(g.attn_b, 3 * C, w.attn_b, false);
    add(g.proj_w, C * C, w.proj_w, true);
    add(g.proj_b, C, w.proj_b, false);
    add(g.ln2_g, C, w.ln2_g, false);
    add(g.ln2_b, C, w.ln2_b, false);
    add(g.fc_w, F * C, w.fc_w, true);
    add(g.fc_b, F, w.fc_b, false);
    add(g.mp_w, C * F, w.mp_w, true);
    add(g.mp_b, C, w.mp_b, false);
  }
  const size_t n = t->grad_floats;
  if (cudaMalloc(&t->master, 3 * n * sizeof(float)) != cudaSuccess) {
    cudaGetLastError();
    t->master = nullptr;
    return GPT_ENOMEM;
  }
  t->m1 = t->master + n;
  t->m2 = t->m1 + n;
  if (cudaMalloc(&t->d_segs, segs.size() * sizeof(OptSeg)) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(t->master);
    t->master = nullptr;
    t->d_segs = nullptr;
    return GPT_ENOMEM;
  }
  GPT_CUDA(cudaMemcpy(t->d_segs, segs.data(), segs.size() * sizeof(OptSeg), cudaMemcpyHostToDevice));
  t->nseg = static_cast<int>(segs.size());
  return GPT_OK;
}

}  // namespace

extern "C" int gpt_adamw_step(gpt_model* m, float lr, float beta1, float beta2, float eps, float weight_decay,
                              void* stream) {
  if (!m || !m->tr) return GPT_EINVAL;
  if (!(beta1 >= 0.0f && beta1 < 1.0f && beta2 >= 0.0f && beta2 < 1.0f && eps > 0.0f)) return GPT_EINVAL;
  gpt_train* t = m->tr;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!t->master) {
    const int rc = alloc_optimizer(m, t);
    if (rc != GPT_OK) return rc;
    GPT_CUDA(cudaMemsetAsync(t->m1, 0, 2 * t->grad_floats * sizeof(float), s));
    GPT_CUDA(cudaMemsetAsync(t->master, 0, t->grad_floats * sizeof(float), s));
    GPT_CUDA(launch_master_init(t->d_segs, t->nseg, t->master, s));
  }
  t->opt_t += 1;
  const float bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(beta1), t->opt_t));
  const float bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(beta2), t->opt_t));
  GPT_CUDA(launch_adamw(t->d_segs, t->nseg, t->gbuf, t->master, t->m1, t->m2, lr, beta1, beta2, eps, weight_decay, bc1,
                        bc2, s));
  t->wT_ready = false;             // the transposed weights are made again by the next backward
  m->launches = 1;
  return GPT_OK;
}

extern "C" int gpt_master_copy(const gpt_model* m, int param, int layer, float* d_dst, void* stream) {
  if (!d_dst || !m || !m->tr || !m->tr->master) return GPT_EINVAL;
  float* g = nullptr;
  int64_t n = 0;
  const int rc = gpt_grad(m, param, layer, &g, &n);
  if (rc != GPT_OK) return rc;
  GPT_CUDA(cudaMemcpyAsync(d_dst, m->tr->master + (g - m->tr->gbuf), static_cast<size_t>(n) * sizeof(float),
                           cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream)));
  return GPT_OK;
}
