// gpt_forward, gpt_forward_host and gpt_status: the launch sequence of one
// forward pass plus loss.
//
// bf16 path, pre-norm ("第 25 章 从小 GPT 到 GPT-2" §25.1-25.4):
//   K1 embed + LN1(block 0)           x fp32, a bf16
//   per block l:
//     K3 c_attn   a . W_attn^T + b          -> qkv bf16 [M, 3C]
//     K4 attention (causal, online softmax) -> y bf16 [M, C]
//     K3 c_proj   x += y . W_proj^T + b     (residual in the epilogue)
//     K2 LN2      x -> a
//     K3 c_fc     a . W_fc^T + b, GELU      -> g bf16 [M, ffn]
//     K3 mlp.c_proj x += g . W_mp^T + b
//     K2 LN1 of block l+1, or ln_f after the last block: x -> a
//   K5 tied head with the cross-entropy epilogue: per (row, 256-column tile)
//      partial max / sum-exp and the target's logit; logits stored only if asked
//   K6 combine the partials per row -> nll; mean -> loss
// Post-norm ("GPT-1 学习笔记" §3.1-3.2): c_attn reads x itself (a = bf16 copy),
// the LayerNorms read the residual sums and write back into x, no ln_f.
#include "launch.h"
#include "model.h"

#include <cuda_runtime.h>

#include <cstdlib>
#include <vector>

using namespace gptgb;

namespace {

int cu(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return GPT_OK;
  set_detail(what, e);
  return GPT_ECUDA;
}

bool probe_hit(const gpt_model* m, int step, int layer) {
  return m->prof_ev0 != nullptr && m->prof_step == step && (layer < 0 || m->prof_layer == layer);
}

// One step = one kernel launch, optionally bracketed by the armed probe events.
// An armed probe's events around one step. Inside a graph capture the records become event-record
// nodes (external events), outside it they are plain records.
#define GPT_STEP(step, layer, expr)                                                 \
  do {                                                                              \
    const bool hit_ = probe_hit(m, (step), (layer));                                \
    const unsigned fl_ = m->capturing ? cudaEventRecordExternal : cudaEventRecordDefault; \
    if (hit_) GPT_CUDA(cudaEventRecordWithFlags(m->prof_ev0, s, fl_));              \
    const int rc_ = (expr);                                                         \
    if (rc_ != GPT_OK) return rc_;                                                  \
    ++m->launches;                                                                  \
    if (hit_) {                                                                     \
      GPT_CUDA(cudaEventRecordWithFlags(m->prof_ev1, s, fl_));                      \
      ++m->probe_hits;                                                              \
    }                                                                               \
  } while (0)

int ensure_act_maps(gpt_model* m, int B, int T) {
  if (m->cached_B == B && m->cached_T == T) return GPT_OK;
  const int M = B * T, C = m->cfg.C, F = m->cfg.ffn;
  const bool ok = make_tmap_2d_bf16(&m->tm_a, m->a, M, C, kGemmBM) &&
                  make_tmap_2d_bf16(&m->tm_y, m->y, M, C, kGemmBM) &&
                  make_tmap_2d_bf16(&m->tm_g, m->g, M, F, kGemmBM) &&
                  make_tmap_qkv(&m->tm_qkv, m->qkv, B, T, 3 * C, C / m->cfg.H) &&
                  make_tmap_2d(&m->tm_qkv_out, m->qkv, 2, M, 3 * C, 64, kEpiRows) &&
                  make_tmap_2d(&m->tm_g_out, m->g, 2, M, F, 64, kEpiRows) &&
                  make_tmap_2d(&m->tm_x_out, m->x, 4, M, C, 32, kEpiRows);
  if (!ok) {
    set_detail_text("activation tensor map");
    m->cached_B = m->cached_T = -1;
    return GPT_ECUDA;
  }
  m->cached_B = B;
  m->cached_T = T;
  return GPT_OK;
}

GemmArgs tc_args(gpt_model* m, int M, int N, int K, const float* bias, void* out) {
  GemmArgs a{};
  a.M = M; a.N = N; a.K = K;
  a.bias = bias;
  a.out = out;
  a.ldo = N;
  a.gelu_erf = m->cfg.gelu;
  a.err = m->err;
  a.m_fastest = (N > M) ? 1 : 0;        // keep the larger operand's tiles shared by co-running CTAs
  a.sk_part = m->sk_part;               // used where whole tiles would leave the last wave part-idle
  a.sk_flag = m->sk_flag;
  if (m->dbg_armed) {                   // failure-detection check: wait on flags nothing sets
    a.sk_wait_flag = m->dbg_flag;
    a.wait_limit = m->dbg_wait_limit;
  }
  a.b_const = 1;                        // every caller's B is a weight (or a transposed copy made earlier)
  return a;
}

int tc_gemm(gpt_model* m, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, int M, int N,
            int K, const float* bias, void* out, int epi, cudaStream_t s, const CUtensorMap* tmC2 = nullptr) {
  const GemmArgs a = tc_args(m, M, N, K, bias, out);
  GPT_CUDA(launch_gemm_tc2(tmA, tmB, tmC, tmC2 != nullptr ? *tmC2 : tmC, a, epi, m->num_sms, s));
  return GPT_OK;
}

// A product with a tensor-store epilogue (EPI_BIAS_RESID, EPI_F32_OUT, EPI_BIAS_OUT, EPI_BIAS_GELU_OUT) on
// CTA pairs (256 x 256 tiles, a six-stage ring of 32 KB per CTA; tmB_pair has 128-row boxes) where they
// were measured faster in the GPT-2 small step at 16,384 tokens: long K (at least 1536: mlp c_proj
// 66 -> 61 us, the input gradients through W_fc and W_attn), the QKV projection (N = 2304, bf16 out:
// 46.6 -> 44.5 us) and the GELU product c_fc (with eight epilogue warps and five stages: 60.5 -> 59.1 us;
// with four it was 64: its epilogue bounds each tile). Not the attention c_proj (32 us either way).
// Elsewhere, or where clusters of two cannot be resident, the single-CTA kernel.
constexpr int kPairMinK = 1536;
bool pair_pays(int N, int K, int epi) {
  return epi == EPI_BIAS_GELU_OUT || K >= kPairMinK || (epi == EPI_BIAS_OUT && N >= 2048);
}

int tc_gemm_long(gpt_model* m, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmB_pair,
                 const CUtensorMap& tmC, int M, int N, int K, const float* bias, void* out, int epi, cudaStream_t s) {
  if (pair_enabled() && pair_pays(N, K, epi) && gemm_pair_capacity() > 0) {
    const GemmArgs a = tc_args(m, M, N, K, bias, out);
    GPT_CUDA(launch_gemm_pair(tmA, tmB_pair, tmC, a, epi, m->num_sms / 2, s));
    return GPT_OK;
  }
  return tc_gemm(m, tmA, tmB, tmC, M, N, K, bias, out, epi, s);
}

// Layer l's key/value cache: [kv_batch][ctx][2C] bf16.
void* kv_layer(gpt_model* m, int l) {
  return m->kv + static_cast<size_t>(l) * m->kv_batch * m->cfg.ctx * 2 * m->cfg.C * 2;
}

// The LayerNorm that follows the residual add of a block (or ln_f / nothing).
// Pre-norm: a = LN(x). Post-norm: x = LN(x) and a = copy of it.
struct NextLN { const float* g; const float* b; };

int forward_bf16(gpt_model* m, const int32_t* ids, const int32_t* tg, int B, int T, float* d_loss, float* d_logits,
                 cudaStream_t s) {
  const gpt_config& c = m->cfg;
  const int M = B * T, C = c.C, F = c.ffn, L = c.L;
  const bool pre = c.norm_mode == 0;
  int rc = ensure_act_maps(m, B, T);
  if (rc != GPT_OK) return rc;

  // K1: embedding (+ the first LayerNorm of the pre-norm stack)
  {
    int out_mode = 1;
    const float* g = nullptr;
    const float* b = nullptr;
    if (pre) {
      if (L > 0) { out_mode = 2; g = m->layers[0].ln1_g; b = m->layers[0].ln1_b; }
      else if (c.final_ln) { out_mode = 2; g = m->lnf_g; b = m->lnf_b; }
    }
    GPT_STEP(GPT_STEP_EMBED, -1,
             cu(launch_embed(ids, m->wte, m->wpe, 1, m->x, m->a, out_mode, 1, g, b, M, T, C, c.V, c.ln_eps, m->err, s),
                "embed"));
  }
  for (int l = 0; l < L; ++l) {
    const gpt_layer_dev& w = m->layers[l];
    GPT_STEP(GPT_STEP_C_ATTN, l, tc_gemm_long(m, m->tm_a, w.tm_attn_w, w.tm_attn_w_pair, m->tm_qkv_out, M, 3 * C, C, w.attn_b, m->qkv, EPI_BIAS_OUT, s));
    if (m->kv_fill) {                       // prefill: keep every token's key and value
      ++m->launches;
      rc = cu(launch_kv_store(m->qkv, kv_layer(m, l), B, T, C, c.ctx, s), "kv_store");
      if (rc != GPT_OK) return rc;
    }
    GPT_STEP(GPT_STEP_ATTN, l, cu(launch_attention_tc(m->tm_qkv, m->y, B, T, c.H, C / c.H, m->err, m->attn_sched, s), "attention"));
    // the LayerNorm after each residual add: ln_2 then the next block's ln_1 or ln_f
    // (pre-norm), ln_1 then ln_2 applied to x itself (post-norm)
    NextLN mid = pre ? NextLN{w.ln2_g, w.ln2_b} : NextLN{w.ln1_g, w.ln1_b};
    NextLN out{w.ln2_g, w.ln2_b};
    if (pre) {
      out = {nullptr, nullptr};
      if (l + 1 < L) out = {m->layers[l + 1].ln1_g, m->layers[l + 1].ln1_b};
      else if (c.final_ln) out = {m->lnf_g, m->lnf_b};
    }
    GPT_STEP(GPT_STEP_C_PROJ, l, tc_gemm_long(m, m->tm_y, w.tm_proj_w, w.tm_proj_w_pair, m->tm_x_out, M, C, C, w.proj_b, m->x, EPI_BIAS_RESID, s));
    GPT_STEP(GPT_STEP_LN_MID, l,
             cu(launch_layernorm(m->x, mid.g, mid.b, m->a, 1, pre ? nullptr : m->x, M, C, c.ln_eps, s), "ln"));
    GPT_STEP(GPT_STEP_C_FC, l, tc_gemm_long(m, m->tm_a, w.tm_fc_w, w.tm_fc_w_pair, m->tm_g_out, M, F, C, w.fc_b, m->g, EPI_BIAS_GELU_OUT, s));
    GPT_STEP(GPT_STEP_MLP_PROJ, l, tc_gemm_long(m, m->tm_g, w.tm_mp_w, w.tm_mp_w_pair, m->tm_x_out, M, C, F, w.mp_b, m->x, EPI_BIAS_RESID, s));
    GPT_STEP(GPT_STEP_LN_OUT, l,
             cu(launch_layernorm(m->x, out.g, out.b, m->a, 1, pre ? nullptr : m->x, M, C, c.ln_eps, s), "ln"));
  }
  if (!pre && c.final_ln)                   // post-norm with a final LayerNorm: after the last block's ln_2
    GPT_STEP(GPT_STEP_LN_OUT, -1, cu(launch_layernorm(m->x, m->lnf_g, m->lnf_b, m->a, 1, nullptr, M, C, c.ln_eps, s), "ln"));

  // K5/K6: tied head
  if (tg) {
    GemmArgs a{};
    a.M = M; a.N = c.V; a.K = C;
    a.ldo = c.V;
    a.targets = tg;
    a.pmax = m->pmax;
    a.psum = m->psum;
    a.ztgt = m->ztgt;
    a.logits = d_logits;
    a.err = m->err;
    a.m_fastest = 1;
    a.b_const = 1;
    GPT_STEP(GPT_STEP_HEAD, -1, cu(launch_gemm_tc(m->tm_a, m->tm_head, m->tm_a, a, EPI_CE, m->num_sms, s), "head"));
    GPT_STEP(GPT_STEP_CE, -1,
             cu(launch_ce_combine(m->pmax, m->psum, m->ztgt, tg, m->nll, m->block_sums, M, gemm_tc_num_ntiles(c.V),
                                  c.V, m->err, s),
                "ce_combine"));
    if (d_loss)
      GPT_STEP(GPT_STEP_MEAN, -1, cu(launch_mean(m->block_sums, ce_combine_blocks(M), M, d_loss, s), "mean"));
  } else if (d_logits) {
    GPT_STEP(GPT_STEP_HEAD, -1, tc_gemm(m, m->tm_a, m->tm_head, m->tm_a, M, c.V, C, nullptr, d_logits, EPI_F32, s));
  }
  return GPT_OK;
}

int forward_f32(gpt_model* m, const int32_t* ids, const int32_t* tg, int B, int T, float* d_loss, float* d_logits,
                cudaStream_t s) {
  const gpt_config& c = m->cfg;
  const int M = B * T, C = c.C, F = c.ffn, L = c.L, H = c.H;
  const bool pre = c.norm_mode == 0;
  float* a = reinterpret_cast<float*>(m->a);
  float* qkv = reinterpret_cast<float*>(m->qkv);
  float* y = reinterpret_cast<float*>(m->y);
  float* g = reinterpret_cast<float*>(m->g);
  {
    int out_mode = 1;
    const float* lg = nullptr;
    const float* lb = nullptr;
    if (pre) {
      if (L > 0) { out_mode = 2; lg = m->layers[0].ln1_g; lb = m->layers[0].ln1_b; }
      else if (c.final_ln) { out_mode = 2; lg = m->lnf_g; lb = m->lnf_b; }
    }
    GPT_STEP(GPT_STEP_EMBED, -1,
             cu(launch_embed(ids, m->wte, m->wpe, 0, m->x, a, out_mode, 0, lg, lb, M, T, C, c.V, c.ln_eps, m->err, s),
                "embed"));
  }
  for (int l = 0; l < L; ++l) {
    const gpt_layer_dev& w = m->layers[l];
    GPT_STEP(GPT_STEP_C_ATTN, l,
             cu(launch_gemm_simt(a, reinterpret_cast<const float*>(w.attn_w), w.attn_b, qkv, M, 3 * C, C, 3 * C,
                                 EPI_BIAS_OUT, c.gelu, s), "gemm"));
    GPT_STEP(GPT_STEP_ATTN, l, cu(launch_attention_simt(qkv, y, B, T, H, C / H, s), "attention"));
    GPT_STEP(GPT_STEP_C_PROJ, l,
             cu(launch_gemm_simt(y, reinterpret_cast<const float*>(w.proj_w), w.proj_b, m->x, M, C, C, C,
                                 EPI_BIAS_RESID, c.gelu, s), "gemm"));
    if (pre)
      GPT_STEP(GPT_STEP_LN_MID, l, cu(launch_layernorm(m->x, w.ln2_g, w.ln2_b, a, 0, nullptr, M, C, c.ln_eps, s), "ln"));
    else
      GPT_STEP(GPT_STEP_LN_MID, l, cu(launch_layernorm(m->x, w.ln1_g, w.ln1_b, a, 0, m->x, M, C, c.ln_eps, s), "ln"));
    GPT_STEP(GPT_STEP_C_FC, l,
             cu(launch_gemm_simt(a, reinterpret_cast<const float*>(w.fc_w), w.fc_b, g, M, F, C, F,
                                 EPI_BIAS_GELU_OUT, c.gelu, s), "gemm"));
    GPT_STEP(GPT_STEP_MLP_PROJ, l,
             cu(launch_gemm_simt(g, reinterpret_cast<const float*>(w.mp_w), w.mp_b, m->x, M, C, F, C,
                                 EPI_BIAS_RESID, c.gelu, s), "gemm"));
    if (pre) {
      NextLN n{nullptr, nullptr};
      if (l + 1 < L) n = {m->layers[l + 1].ln1_g, m->layers[l + 1].ln1_b};
      else if (c.final_ln) n = {m->lnf_g, m->lnf_b};
      GPT_STEP(GPT_STEP_LN_OUT, l, cu(launch_layernorm(m->x, n.g, n.b, a, 0, nullptr, M, C, c.ln_eps, s), "ln"));
    } else {
      GPT_STEP(GPT_STEP_LN_OUT, l, cu(launch_layernorm(m->x, w.ln2_g, w.ln2_b, a, 0, m->x, M, C, c.ln_eps, s), "ln"));
    }
  }
  if (!pre && c.final_ln)                   // post-norm with a final LayerNorm: after the last block's ln_2
    GPT_STEP(GPT_STEP_LN_OUT, -1, cu(launch_layernorm(m->x, m->lnf_g, m->lnf_b, a, 0, nullptr, M, C, c.ln_eps, s), "ln"));
  if (!tg && !d_logits) return GPT_OK;
  float* z = d_logits ? d_logits : m->logits_ws;
  GPT_STEP(GPT_STEP_HEAD, -1,
           cu(launch_gemm_simt(a, reinterpret_cast<const float*>(m->head), nullptr, z, M, c.V, C, c.V, EPI_F32, 0, s),
              "head"));
  if (tg) {
    GPT_STEP(GPT_STEP_CE, -1, cu(launch_ce_rows(z, tg, m->nll, M, c.V, m->err, s), "ce_rows"));
    if (d_loss) GPT_STEP(GPT_STEP_MEAN, -1, cu(launch_mean(m->nll, M, M, d_loss, s), "mean"));
  }
  return GPT_OK;
}

int check_shape(const gpt_model* m, int B, int T) {
  if (B < 1 || T < 1) return GPT_EINVAL;
  if (T > m->cfg.ctx) return GPT_ESEQ;
  if ((int64_t)B * T > m->cfg.max_tokens) return GPT_EINVAL;
  return GPT_OK;
}

// Forward passes and decode steps are captured into CUDA graphs and replayed (GPT_GB300_NO_GRAPH=1:
// launched directly each time); the results are the same either way.
bool graphs_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("GPT_GB300_NO_GRAPH");
    return !(v && v[0] == '1');
  }();
  return on;
}

// One decode step (bf16): B new tokens at position *pos_dev, every projection a
// matrix-vector product over the B rows, attention over the cached rows.
int decode_bf16(gpt_model* m, const int32_t* ids, int B, const int* pos_dev, float* d_logits, cudaStream_t s) {
  const gpt_config& c = m->cfg;
  const int C = c.C, F = c.ffn, L = c.L, D = C / c.H;
  const bool pre = c.norm_mode == 0;
#define GPT_DEC(expr, what)                       \
  do {                                            \
    const int rc_ = cu((expr), what);             \
    if (rc_ != GPT_OK) return rc_;                \
    ++m->launches;                                \
  } while (0)
  {
    int out_mode = 1;
    const float* g = nullptr;
    const float* b = nullptr;
    if (pre) {
      if (L > 0) { out_mode = 2; g = m->layers[0].ln1_g; b = m->layers[0].ln1_b; }
      else if (c.final_ln) { out_mode = 2; g = m->lnf_g; b = m->lnf_b; }
    }
    GPT_DEC(launch_embed(ids, m->wte, m->wpe, 1, m->x, m->a, out_mode, 1, g, b, B, 1, C, c.V, c.ln_eps, m->err, s, 0,
                         pos_dev),
            "embed");
  }
  for (int l = 0; l < L; ++l) {
    const gpt_layer_dev& w = m->layers[l];
    GPT_DEC(launch_gemv(m->a, C, w.attn_w, w.attn_b, m->qkv, 3 * C, B, 3 * C, C, EPI_BIAS_OUT, c.gelu, s), "c_attn");
    GPT_DEC(launch_attention_decode(m->qkv, kv_layer(m, l), m->y, B, c.H, D, c.ctx, pos_dev, s), "attention");
    NextLN mid = pre ? NextLN{w.ln2_g, w.ln2_b} : NextLN{w.ln1_g, w.ln1_b};
    NextLN out{w.ln2_g, w.ln2_b};
    if (pre) {
      out = {nullptr, nullptr};
      if (l + 1 < L) out = {m->layers[l + 1].ln1_g, m->layers[l + 1].ln1_b};
      else if (c.final_ln) out = {m->lnf_g, m->lnf_b};
    }
    GPT_DEC(launch_gemv(m->y, C, w.proj_w, w.proj_b, m->x, C, B, C, C, EPI_BIAS_RESID, c.gelu, s), "c_proj");
    GPT_DEC(launch_layernorm(m->x, mid.g, mid.b, m->a, 1, pre ? nullptr : m->x, B, C, c.ln_eps, s), "ln");
    GPT_DEC(launch_gemv(m->a, C, w.fc_w, w.fc_b, m->g, F, B, F, C, EPI_BIAS_GELU_OUT, c.gelu, s), "c_fc");
    GPT_DEC(launch_gemv(m->g, F, w.mp_w, w.mp_b, m->x, C, B, C, F, EPI_BIAS_RESID, c.gelu, s), "mlp_proj");
    GPT_DEC(launch_layernorm(m->x, out.g, out.b, m->a, 1, pre ? nullptr : m->x, B, C, c.ln_eps, s), "ln");
  }
  if (!pre && c.final_ln)                   // post-norm with a final LayerNorm: after the last block's ln_2
    GPT_DEC(launch_layernorm(m->x, m->lnf_g, m->lnf_b, m->a, 1, nullptr, B, C, c.ln_eps, s), "ln");
  GPT_DEC(launch_gemv(m->a, C, m->head, nullptr, d_logits, c.V, B, c.V, C, EPI_F32, c.gelu, s), "head");
#undef GPT_DEC
  return GPT_OK;
}

// Point an event-record node of an executable graph at another event, through the driver entry
// point. The driver refuses this for some callers' events (those of a framework's own copy of the
// runtime, seen with PyTorch's); the caller then captures the forward again with the new events.
cudaError_t graph_exec_set_event(cudaGraphExec_t exec, cudaGraphNode_t node, cudaEvent_t ev) {
  using Fn = CUresult (*)(CUgraphExec, CUgraphNode, CUevent);
  static Fn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuGraphExecEventRecordNodeSetEvent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<Fn>(p);
  }();
  if (!fn) return cudaErrorNotSupported;
  return fn(reinterpret_cast<CUgraphExec>(exec), reinterpret_cast<CUgraphNode>(node), reinterpret_cast<CUevent>(ev)) ==
                 CUDA_SUCCESS
             ? cudaSuccess
             : cudaErrorInvalidValue;
}

// gpt_forward on the bf16 path through a CUDA graph: captured on the first call for a set of
// (pointers, B, T, armed probe) and replayed while they repeat. An armed probe's events are
// event-record nodes of the graph; a replay points them at the probe's current events.
int forward_graphed(gpt_model* m, const int32_t* ids, const int32_t* tg, int B, int T, float* d_loss,
                    float* d_logits, cudaStream_t s) {
  const bool probe = m->prof_ev0 != nullptr;
  const void* key[8] = {ids, tg, d_loss, d_logits, reinterpret_cast<const void*>(static_cast<intptr_t>(B)),
                        reinterpret_cast<const void*>(static_cast<intptr_t>(T)),
                        reinterpret_cast<const void*>(static_cast<intptr_t>(probe ? m->prof_step : -1)),
                        reinterpret_cast<const void*>(static_cast<intptr_t>(probe ? m->prof_layer : -2))};
  bool same = m->fwd_exec != nullptr;
  for (int i = 0; i < 8 && same; ++i) same = m->fwd_key[i] == key[i];
  if (same && probe && m->fwd_ev_node[0] && m->fwd_ev_node[1]) {
    // point the captured event-record nodes at this call's events; events the driver does not
    // accept there (some runtimes' own) mean a fresh capture with them instead
    same = graph_exec_set_event(m->fwd_exec, m->fwd_ev_node[0], m->prof_ev0) == cudaSuccess &&
           graph_exec_set_event(m->fwd_exec, m->fwd_ev_node[1], m->prof_ev1) == cudaSuccess;
  }
  if (!same) {
    if (m->fwd_exec) {
      GPT_CUDA(cudaStreamSynchronize(s));    // the old graph may still be running
      GPT_CUDA(cudaGraphExecDestroy(m->fwd_exec));
      m->fwd_exec = nullptr;
    }
    if (m->fwd_graph) {
      cudaGraphDestroy(m->fwd_graph);
      m->fwd_graph = nullptr;
    }
    if (!m->cap_stream) GPT_CUDA(cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking));
    GPT_CUDA(cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal));
    m->launches = 0;
    m->probe_hits = 0;
    m->capturing = true;
    const int rc = forward_bf16(m, ids, tg, B, T, d_loss, d_logits, m->cap_stream);
    m->capturing = false;
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(m->cap_stream, &g);
    if (rc != GPT_OK) {
      if (g) cudaGraphDestroy(g);
      return rc;
    }
    GPT_CUDA(e);
    m->fwd_ev_node[0] = m->fwd_ev_node[1] = nullptr;
    if (m->probe_hits > 0) {                 // find the probe's two event-record nodes
      size_t n = 0;
      GPT_CUDA(cudaGraphGetNodes(g, nullptr, &n));
      std::vector<cudaGraphNode_t> nodes(n);
      GPT_CUDA(cudaGraphGetNodes(g, nodes.data(), &n));
      for (cudaGraphNode_t nd : nodes) {
        cudaGraphNodeType ty;
        GPT_CUDA(cudaGraphNodeGetType(nd, &ty));
        if (ty != cudaGraphNodeTypeEventRecord) continue;
        cudaEvent_t ev = nullptr;
        GPT_CUDA(cudaGraphEventRecordNodeGetEvent(nd, &ev));
        if (ev == m->prof_ev0) m->fwd_ev_node[0] = nd;
        if (ev == m->prof_ev1) m->fwd_ev_node[1] = nd;
      }
    }
    const cudaError_t ei = cudaGraphInstantiate(&m->fwd_exec, g, 0);
    if (ei != cudaSuccess) {
      cudaGraphDestroy(g);
      GPT_CUDA(ei);
    }
    m->fwd_graph = g;                        // kept: its nodes name the event-record nodes
    for (int i = 0; i < 8; ++i) m->fwd_key[i] = key[i];
    m->fwd_launches = m->launches;
    m->fwd_probe_hits = m->probe_hits;
  }
  GPT_CUDA(cudaGraphLaunch(m->fwd_exec, s));
  m->launches = m->fwd_launches;
  m->probe_hits = m->fwd_probe_hits;
  return GPT_OK;
}

}  // namespace

namespace gptgb {

// The activation descriptors of the forward pass (x, a, ...) for this (B, T).
int forward_maps(gpt_model* m, int B, int T) { return ensure_act_maps(m, B, T); }

int gemm_bf16(gpt_model* m, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, int M, int N,
              int K, const float* bias, void* out, int epi, cudaStream_t s) {
  return tc_gemm(m, tmA, tmB, tmC, M, N, K, bias, out, epi, s);
}

int gemm_bf16_long(gpt_model* m, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmB_pair,
                   const CUtensorMap& tmC, int M, int N, int K, const float* bias, void* out, int epi, cudaStream_t s) {
  return tc_gemm_long(m, tmA, tmB, tmB_pair, tmC, M, N, K, bias, out, epi, s);
}

int gemm_bf16_gelu_u(gpt_model* m, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tm_g,
                     const CUtensorMap& tm_u, int M, int N, int K, const float* bias, void* g, cudaStream_t s) {
  return tc_gemm(m, tmA, tmB, tm_g, M, N, K, bias, g, EPI_BIAS_GELU_UOUT, s, &tm_u);
}

int shape_ok(const gpt_model* m, int B, int T) { return check_shape(m, B, T); }

}  // namespace gptgb

namespace {

int map_device_error(int code) {
  switch (code) {
    case GPT_DEV_OK: return GPT_OK;
    case GPT_DEV_ETOKEN:
    case GPT_DEV_ETARGET: return GPT_ETOKEN;
    default: return GPT_EDEVICE;
  }
}

}  // namespace

extern "C" {

int gpt_forward(gpt_model* m, const int32_t* d_ids, const int32_t* d_targets, int32_t B, int32_t T, float* d_loss,
                float* d_logits, void* stream) {
  if (!m || !d_ids) return GPT_EINVAL;
  int rc = check_shape(m, B, T);
  if (rc != GPT_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  m->launches = 0;
  m->probe_hits = 0;
  if (m->dbg_armed) {                        // the armed check runs once, launched directly
    rc = forward_bf16(m, d_ids, d_targets, B, T, d_loss, d_logits, s);
    m->dbg_armed = false;
  } else if (m->bf16 && graphs_enabled())
    rc = forward_graphed(m, d_ids, d_targets, B, T, d_loss, d_logits, s);
  else
    rc = m->bf16 ? forward_bf16(m, d_ids, d_targets, B, T, d_loss, d_logits, s)
                 : forward_f32(m, d_ids, d_targets, B, T, d_loss, d_logits, s);
  m->prof_ev0 = m->prof_ev1 = nullptr;       // a probe covers one forward
  m->prof_step = m->prof_layer = -1;
  return rc;
}

int gpt_prefill(gpt_model* m, const int32_t* d_ids, int32_t B, int32_t T, float* d_logits, void* stream) {
  if (!m || !d_ids) return GPT_EINVAL;
  if (!m->bf16) return GPT_ECONFIG;
  int rc = check_shape(m, B, T);
  if (rc != GPT_OK) return rc;
  if (B > m->kv_batch) return GPT_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  m->launches = 0;
  m->probe_hits = 0;
  m->kv_fill = true;
  rc = forward_bf16(m, d_ids, nullptr, B, T, nullptr, nullptr, s);
  m->kv_fill = false;
  m->prof_ev0 = m->prof_ev1 = nullptr;
  m->prof_step = m->prof_layer = -1;
  if (rc != GPT_OK || !d_logits) return rc;
  // the head on each sequence's last row only (rows T-1, 2T-1, ... of the final activations)
  const gpt_config& c = m->cfg;
  rc = cu(launch_gemv(static_cast<const uint8_t*>(m->a) + static_cast<size_t>(T - 1) * c.C * 2, T * c.C, m->head,
                      nullptr, d_logits, c.V, B, c.V, c.C, EPI_F32, c.gelu, s),
          "head");
  if (rc == GPT_OK) ++m->launches;
  return rc;
}

int gpt_decode_step(gpt_model* m, const int32_t* d_ids, int32_t B, int32_t pos, float* d_logits, void* stream) {
  if (!m || !d_ids || !d_logits) return GPT_EINVAL;
  if (!m->bf16) return GPT_ECONFIG;
  if (B < 1 || B > m->kv_batch || B > m->cfg.max_tokens) return GPT_EINVAL;
  if (pos < 0 || pos >= m->cfg.ctx) return GPT_ESEQ;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the step reads its ids and position from model memory, so one captured graph serves every step
  GPT_CUDA(cudaMemcpyAsync(m->stage_ids, d_ids, static_cast<size_t>(B) * sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
  GPT_CUDA(launch_set_int(m->dec_pos, pos, s));
  if (!graphs_enabled()) {
    m->launches = 1;
    return decode_bf16(m, m->stage_ids, B, m->dec_pos, d_logits, s);
  }
  if (!m->dec_exec || m->dec_B != B || m->dec_logits != d_logits) {
    if (m->dec_exec) {
      GPT_CUDA(cudaStreamSynchronize(s));    // the old graph may still be running
      GPT_CUDA(cudaGraphExecDestroy(m->dec_exec));
      m->dec_exec = nullptr;
    }
    if (!m->cap_stream) GPT_CUDA(cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking));
    GPT_CUDA(cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal));
    m->launches = 0;
    m->capturing = true;
    const int rc = decode_bf16(m, m->stage_ids, B, m->dec_pos, d_logits, m->cap_stream);
    m->capturing = false;
    cudaGraph_t g = nullptr;
    const cudaError_t e = cudaStreamEndCapture(m->cap_stream, &g);
    if (rc != GPT_OK) {
      if (g) cudaGraphDestroy(g);
      return rc;
    }
    GPT_CUDA(e);
    const cudaError_t ei = cudaGraphInstantiate(&m->dec_exec, g, 0);
    cudaGraphDestroy(g);
    GPT_CUDA(ei);
    m->dec_B = B;
    m->dec_logits = d_logits;
    m->dec_launches = m->launches;
  }
  GPT_CUDA(cudaGraphLaunch(m->dec_exec, s));
  m->launches = m->dec_launches + 1;
  return GPT_OK;
}

int gpt_sample(const float* d_logits, int32_t B, int32_t V, float temperature, int32_t top_k, float top_p,
               const float* d_uniform, int32_t* d_ids, void* stream) {
  if (!d_logits || !d_ids || B < 1 || V < 1 || V > kSampleMaxV) return GPT_EINVAL;
  if (temperature > 0.0f && !d_uniform) return GPT_EINVAL;
  GPT_CUDA(launch_sample(d_logits, B, V, temperature, top_k, top_p, d_uniform, d_ids,
                         reinterpret_cast<cudaStream_t>(stream)));
  return GPT_OK;
}

int gpt_time_step(gpt_model* m, int step, int layer, void* ev_start, void* ev_stop) {
  if (!m) return GPT_EINVAL;
  if (!ev_start) {
    m->prof_ev0 = m->prof_ev1 = nullptr;
    m->prof_step = m->prof_layer = -1;
    return GPT_OK;
  }
  if (!ev_stop || step < GPT_STEP_EMBED || (step > GPT_STEP_MEAN && step < GPT_STEP_B_DZ) || step > GPT_STEP_B_DA1)
    return GPT_EINVAL;
  m->prof_step = step;
  m->prof_layer = layer;
  m->prof_ev0 = reinterpret_cast<cudaEvent_t>(ev_start);
  m->prof_ev1 = reinterpret_cast<cudaEvent_t>(ev_stop);
  return GPT_OK;
}

int gpt_debug_expire_waits(gpt_model* m, int64_t limit_cycles) {
  if (!m || limit_cycles < 1) return GPT_EINVAL;
  if (!m->bf16) return GPT_ECONFIG;
  if (!m->dbg_flag) {
    const size_t bytes = gemm_sk_flag_ints(m->num_sms) * sizeof(int);
    GPT_CUDA(cudaMalloc(&m->dbg_flag, bytes));
    GPT_CUDA(cudaMemset(m->dbg_flag, 0, bytes));
  }
  m->dbg_wait_limit = limit_cycles;
  m->dbg_armed = true;
  return GPT_OK;
}

int gpt_last_launch_count(const gpt_model* m) { return m ? m->launches : 0; }

int gpt_last_probe_hits(const gpt_model* m) { return m ? m->probe_hits : 0; }

int gpt_status(gpt_model* m, void* stream) {
  if (!m) return GPT_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GPT_CUDA(cudaMemcpyAsync(m->h_pinned, m->err, sizeof(int), cudaMemcpyDeviceToHost, s));
  GPT_CUDA(cudaMemsetAsync(m->err, 0, sizeof(int), s));
  GPT_CUDA(cudaStreamSynchronize(s));
  if (m->h_pinned[0] != 0 && m->sk_flag != nullptr) {
    // a launch that gave up may have left stream-K flags set
    GPT_CUDA(cudaMemsetAsync(m->sk_flag, 0, gemm_sk_flag_ints(m->num_sms) * sizeof(int), s));
    GPT_CUDA(cudaStreamSynchronize(s));
  }
  return map_device_error(m->h_pinned[0]);
}

int gpt_forward_host(gpt_model* m, const int32_t* h_ids, const int32_t* h_targets, int32_t B, int32_t T,
                     float* h_loss, float* h_logits, void* stream) {
  if (!m || !h_ids) return GPT_EINVAL;
  if (h_targets && !h_loss) return GPT_EINVAL;
  int rc = check_shape(m, B, T);
  if (rc != GPT_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t M = static_cast<size_t>(B) * T;
  float* d_logits = nullptr;
  if (h_logits) {
    const size_t need = M * static_cast<size_t>(m->cfg.V);
    if (m->stage_logits_elems < need) {
      cudaFree(m->stage_logits);
      m->stage_logits = nullptr;
      m->stage_logits_elems = 0;
      if (cudaMalloc(&m->stage_logits, need * sizeof(float)) != cudaSuccess) return GPT_ENOMEM;
      m->stage_logits_elems = need;
    }
    d_logits = m->stage_logits;
  }
  GPT_CUDA(cudaMemcpyAsync(m->stage_ids, h_ids, M * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  if (h_targets) GPT_CUDA(cudaMemcpyAsync(m->stage_tg, h_targets, M * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  rc = gpt_forward(m, m->stage_ids, h_targets ? m->stage_tg : nullptr, B, T, h_targets ? m->stage_loss : nullptr,
                   d_logits, stream);
  if (rc != GPT_OK) return rc;
  if (h_targets) GPT_CUDA(cudaMemcpyAsync(m->h_pinned + 1, m->stage_loss, sizeof(float), cudaMemcpyDeviceToHost, s));
  if (h_logits)
    GPT_CUDA(cudaMemcpyAsync(h_logits, d_logits, M * m->cfg.V * sizeof(float), cudaMemcpyDeviceToHost, s));
  rc = gpt_status(m, stream);
  if (h_targets) *h_loss = reinterpret_cast<const float*>(m->h_pinned)[1];
  return rc;
}

}  // extern "C"
