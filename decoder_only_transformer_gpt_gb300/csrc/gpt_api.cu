// The C ABI (include/gpt.h): model creation, the forward pass that chains the
// kernels, host-buffer entry, status and teardown.
//
// The forward pass follows "第 25 章 从小 GPT 到 GPT-2" §25.1-25.4 (pre-norm
// GPT-2) and "GPT-1 学习笔记" §3.1-3.2 (post-norm GPT-1):
//   embed (+ LN1 of block 0 fused in, pre-norm)
//   per block: c_attn -> attention -> c_proj(+residual) -> LN -> c_fc(+GELU) -> mlp c_proj(+residual) -> LN
//   tied head with the fused cross-entropy epilogue -> per-row combine -> mean
#include "model.h"

#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

using namespace gptgb;

namespace {
thread_local char g_detail[512] = "";
}  // namespace

namespace gptgb {
void set_detail(const char* what, cudaError_t e) {
  std::snprintf(g_detail, sizeof(g_detail), "%s: %s", what, cudaGetErrorString(e));
}
void set_detail_text(const char* text) { std::snprintf(g_detail, sizeof(g_detail), "%s", text); }
}  // namespace gptgb

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;          // NaN
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// A bump allocator over one device allocation.
struct Carve {
  size_t off = 0;
  size_t take(size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  }
};

}  // namespace

namespace {

int validate_config(const gpt_config* c) {
  if (!c) return GPT_EINVAL;
  if (c->V <= 0 || c->C <= 0 || c->H <= 0 || c->L < 0 || c->ctx <= 0 || c->ffn <= 0 || c->max_tokens <= 0)
    return GPT_EINVAL;
  if (c->dtype != 0 && c->dtype != 1) return GPT_EINVAL;
  if (c->norm_mode != 0 && c->norm_mode != 1) return GPT_EINVAL;
  if (c->gelu != 0 && c->gelu != 1) return GPT_EINVAL;
  if (c->untied_head != 0 && c->untied_head != 1) return GPT_EINVAL;
  if (c->C % c->H != 0) return GPT_ECONFIG;
  if (c->C % 8 != 0 || c->ffn % 8 != 0) return GPT_EINVAL;
  if (c->C > 2048) return GPT_ECONFIG;
  if (c->max_tokens > (int64_t)1 << 30) return GPT_EINVAL;
  if (c->dtype == 1) {
    const int D = c->C / c->H;
    if (D != 32 && D != 64) return GPT_ECONFIG;
  }
  return GPT_OK;
}

int copy_matrix(void* dst, const float* src, size_t n, int bf16) {
  if (!src) return GPT_EINVAL;
  if (!bf16) {
    GPT_CUDA(cudaMemcpy(dst, src, n * sizeof(float), cudaMemcpyHostToDevice));
    return GPT_OK;
  }
  std::vector<uint16_t> tmp;
  try { tmp.resize(n); } catch (...) { return GPT_ENOMEM; }
  for (size_t i = 0; i < n; ++i) tmp[i] = f32_to_bf16_rne(src[i]);
  GPT_CUDA(cudaMemcpy(dst, tmp.data(), n * sizeof(uint16_t), cudaMemcpyHostToDevice));
  return GPT_OK;
}

int copy_vec(float* dst, const float* src, size_t n) {
  if (!src) return GPT_EINVAL;
  GPT_CUDA(cudaMemcpy(dst, src, n * sizeof(float), cudaMemcpyHostToDevice));
  return GPT_OK;
}

void free_model(gpt_model* m) {
  if (!m) return;
  cudaFree(m->wbuf);
  cudaFree(m->ws);
  cudaFree(m->stage_logits);
  cudaFree(m->kv);
  cudaFree(m->dec_pos);
  cudaFree(m->dbg_flag);
  gptgb::free_train(m);
  if (m->dec_exec) cudaGraphExecDestroy(m->dec_exec);
  if (m->fwd_exec) cudaGraphExecDestroy(m->fwd_exec);
  if (m->fwd_graph) cudaGraphDestroy(m->fwd_graph);
  if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
  cudaFreeHost(m->h_pinned);
  delete m;
}

}  // namespace

extern "C" {

const char* gpt_strerror(int code) {
  switch (code) {
    case GPT_OK: return "ok";
    case GPT_EINVAL: return "invalid argument (null pointer, size, or a dimension not a multiple of 8)";
    case GPT_ECONFIG: return "invalid configuration (C not divisible by H, or unsupported head width / width)";
    case GPT_ESEQ: return "sequence longer than the position table (T > ctx)";
    case GPT_ETOKEN: return "token id or target outside [0, V)";
    case GPT_ECUDA: return "CUDA call failed";
    case GPT_ENOMEM: return "out of memory";
    case GPT_EDEVICE: return "device-side failure (expired wait or misaligned shared memory)";
    case GPT_EUNSUPPORTED: return "unsupported device (needs sm_103, GB300)";
    default: return "unknown status";
  }
}

const char* gpt_last_error_detail(void) { return g_detail; }

int64_t gpt_param_count(const gpt_config* c) {
  if (!c) return -1;
  const int64_t C = c->C, F = c->ffn;
  const int64_t per_block = 4 * C + (3 * C * C + 3 * C) + (C * C + C) + (F * C + F) + (C * F + C);
  return c->L * per_block + (int64_t)c->V * C * (c->untied_head ? 2 : 1) + (int64_t)c->ctx * C +
         (c->final_ln ? 2 * C : 0);
}

int gpt_create(const gpt_config* cfg, const gpt_weights* w, gpt_model** out) {
  if (!out) return GPT_EINVAL;
  *out = nullptr;
  int rc = validate_config(cfg);
  if (rc != GPT_OK) return rc;
  if (!w || !w->wte || !w->wpe || (cfg->L > 0 && !w->layers)) return GPT_EINVAL;
  if (cfg->final_ln && (!w->lnf_g || !w->lnf_b)) return GPT_EINVAL;
  if (cfg->untied_head && !w->head) return GPT_EINVAL;

  gpt_model* m = new (std::nothrow) gpt_model();
  if (!m) return GPT_ENOMEM;
  m->cfg = *cfg;
  m->bf16 = cfg->dtype == 1;
  cudaDeviceProp prop;
  if (cudaGetDevice(&m->device) != cudaSuccess || cudaGetDeviceProperties(&prop, m->device) != cudaSuccess) {
    set_detail_text("cudaGetDevice / cudaGetDeviceProperties failed");
    free_model(m);
    return GPT_ECUDA;
  }
  m->num_sms = prop.multiProcessorCount;
  if (m->bf16 && !(prop.major == 10 && prop.minor == 3)) { free_model(m); return GPT_EUNSUPPORTED; }

  const size_t V = cfg->V, C = cfg->C, F = cfg->ffn, ctx = cfg->ctx, L = cfg->L;
  const size_t es = m->bf16 ? 2 : 4;
  // ---- weights
  Carve wc;
  const size_t o_wte = wc.take(V * C * es), o_wpe = wc.take(ctx * C * es);
  std::vector<size_t> lo(L * 12);
  for (size_t l = 0; l < L; ++l) {
    lo[l * 12 + 0] = wc.take(3 * C * C * es);
    lo[l * 12 + 1] = wc.take(C * C * es);
    lo[l * 12 + 2] = wc.take(F * C * es);
    lo[l * 12 + 3] = wc.take(C * F * es);
    lo[l * 12 + 4] = wc.take(3 * C * 4);
    lo[l * 12 + 5] = wc.take(C * 4);
    lo[l * 12 + 6] = wc.take(F * 4);
    lo[l * 12 + 7] = wc.take(C * 4);
    for (int k = 8; k < 12; ++k) lo[l * 12 + k] = wc.take(C * 4);
  }
  const size_t o_lnf = wc.take(2 * C * 4);
  const size_t o_head = cfg->untied_head ? wc.take(V * C * es) : 0;
  if (cudaMalloc(&m->wbuf, wc.off) != cudaSuccess) { free_model(m); return GPT_ENOMEM; }
  m->wte = m->wbuf + o_wte;
  m->wpe = m->wbuf + o_wpe;
  rc = copy_matrix(m->wte, w->wte, V * C, m->bf16);
  m->head = m->wte;
  if (rc == GPT_OK && cfg->untied_head) {
    m->head = m->wbuf + o_head;
    rc = copy_matrix(m->head, w->head, V * C, m->bf16);
  }
  if (rc == GPT_OK) rc = copy_matrix(m->wpe, w->wpe, ctx * C, m->bf16);
  m->layers.resize(L);
  for (size_t l = 0; l < L && rc == GPT_OK; ++l) {
    gpt_layer_dev& d = m->layers[l];
    const gpt_layer_weights& s = w->layers[l];
    d.attn_w = m->wbuf + lo[l * 12 + 0];
    d.proj_w = m->wbuf + lo[l * 12 + 1];
    d.fc_w = m->wbuf + lo[l * 12 + 2];
    d.mp_w = m->wbuf + lo[l * 12 + 3];
    d.attn_b = reinterpret_cast<float*>(m->wbuf + lo[l * 12 + 4]);
    d.proj_b = reinterpret_cast<float*>(m->wbuf + lo[l * 12 + 5]);
    d.fc_b = reinterpret_cast<float*>(m->wbuf + lo[l * 12 + 6]);
    d.mp_b = reinterpret_cast<float*>(m->wbuf + lo[l * 12 + 7]);
    d.ln1_g = reinterpret_cast<float*>(m->wbuf + lo[l * 12 + 8]);
    d.ln1_b = reinterpret_cast<float*>(m->wbuf + lo[l * 12 + 9]);
    d.ln2_g = reinterpret_cast<float*>(m->wbuf + lo[l * 12 + 10]);
    d.ln2_b = reinterpret_cast<float*>(m->wbuf + lo[l * 12 + 11]);
    rc = copy_matrix(d.attn_w, s.attn_w, 3 * C * C, m->bf16);
    if (rc == GPT_OK) rc = copy_matrix(d.proj_w, s.proj_w, C * C, m->bf16);
    if (rc == GPT_OK) rc = copy_matrix(d.fc_w, s.fc_w, F * C, m->bf16);
    if (rc == GPT_OK) rc = copy_matrix(d.mp_w, s.mp_w, C * F, m->bf16);
    if (rc == GPT_OK) rc = copy_vec(d.attn_b, s.attn_b, 3 * C);
    if (rc == GPT_OK) rc = copy_vec(d.proj_b, s.proj_b, C);
    if (rc == GPT_OK) rc = copy_vec(d.fc_b, s.fc_b, F);
    if (rc == GPT_OK) rc = copy_vec(d.mp_b, s.mp_b, C);
    if (rc == GPT_OK) rc = copy_vec(d.ln1_g, s.ln1_g, C);
    if (rc == GPT_OK) rc = copy_vec(d.ln1_b, s.ln1_b, C);
    if (rc == GPT_OK) rc = copy_vec(d.ln2_g, s.ln2_g, C);
    if (rc == GPT_OK) rc = copy_vec(d.ln2_b, s.ln2_b, C);
    if (rc == GPT_OK && m->bf16) {
      const bool ok = make_tmap_2d_bf16(&d.tm_attn_w, d.attn_w, 3 * C, C, gemm_tc_bn()) &&
                      make_tmap_2d_bf16(&d.tm_proj_w, d.proj_w, C, C, gemm_tc_bn()) &&
                      make_tmap_2d_bf16(&d.tm_fc_w, d.fc_w, F, C, gemm_tc_bn()) &&
                      make_tmap_2d_bf16(&d.tm_mp_w, d.mp_w, C, F, gemm_tc_bn()) &&
                      make_tmap_2d_bf16(&d.tm_attn_w_pair, d.attn_w, 3 * C, C, kGemmBM) &&
                      make_tmap_2d_bf16(&d.tm_proj_w_pair, d.proj_w, C, C, kGemmBM) &&
                      make_tmap_2d_bf16(&d.tm_fc_w_pair, d.fc_w, F, C, kGemmBM) &&
                      make_tmap_2d_bf16(&d.tm_mp_w_pair, d.mp_w, C, F, kGemmBM);
      if (!ok) { set_detail_text("weight tensor map"); rc = GPT_ECUDA; }
    }
  }
  if (rc == GPT_OK && cfg->final_ln) {
    m->lnf_g = reinterpret_cast<float*>(m->wbuf + o_lnf);
    m->lnf_b = m->lnf_g + C;
    rc = copy_vec(m->lnf_g, w->lnf_g, C);
    if (rc == GPT_OK) rc = copy_vec(m->lnf_b, w->lnf_b, C);
  }
  if (rc == GPT_OK && m->bf16 && !make_tmap_2d_bf16(&m->tm_wte, m->wte, V, C, gemm_tc_bn())) {
    set_detail_text("token-table tensor map");
    rc = GPT_ECUDA;
  }
  if (rc == GPT_OK && m->bf16) {
    m->tm_head = m->tm_wte;
    if (cfg->untied_head && !make_tmap_2d_bf16(&m->tm_head, m->head, V, C, gemm_tc_bn())) {
      set_detail_text("head tensor map");
      rc = GPT_ECUDA;
    }
  }
  if (rc != GPT_OK) { free_model(m); return rc; }

  // ---- workspace
  const size_t Mx = static_cast<size_t>(cfg->max_tokens);
  const size_t NB = static_cast<size_t>(gemm_tc_num_ntiles(cfg->V));
  Carve ws;
  const size_t o_x = ws.take(Mx * C * 4), o_a = ws.take(Mx * C * es), o_qkv = ws.take(Mx * 3 * C * es),
               o_y = ws.take(Mx * C * es), o_g = ws.take(Mx * F * es);
  size_t o_pmax = 0, o_psum = 0, o_ztgt = 0, o_logits = 0, o_skp = 0, o_skf = 0;
  if (m->bf16) {
    o_pmax = ws.take(NB * Mx * 4);
    o_psum = ws.take(NB * Mx * 4);
    o_ztgt = ws.take(Mx * 4);
    o_skp = ws.take(gemm_sk_part_floats(m->num_sms) * 4);
    o_skf = ws.take(gemm_sk_flag_ints(m->num_sms) * 4);
  } else {
    o_logits = ws.take(Mx * V * 4);
  }
  const size_t o_bsum = ws.take(static_cast<size_t>(ce_combine_blocks(static_cast<int>(Mx))) * 4);
  const size_t o_nll = ws.take(Mx * 4), o_err = ws.take(256), o_ids = ws.take(Mx * 4), o_tg = ws.take(Mx * 4),
               o_loss = ws.take(256);
  if (cudaMalloc(&m->ws, ws.off) != cudaSuccess) { free_model(m); return GPT_ENOMEM; }
  m->x = reinterpret_cast<float*>(m->ws + o_x);
  m->a = m->ws + o_a;
  m->qkv = m->ws + o_qkv;
  m->y = m->ws + o_y;
  m->g = m->ws + o_g;
  if (m->bf16) {
    m->pmax = reinterpret_cast<float*>(m->ws + o_pmax);
    m->psum = reinterpret_cast<float*>(m->ws + o_psum);
    m->ztgt = reinterpret_cast<float*>(m->ws + o_ztgt);
    m->sk_part = reinterpret_cast<float*>(m->ws + o_skp);
    m->sk_flag = reinterpret_cast<int*>(m->ws + o_skf);
    if (cudaMemset(m->sk_flag, 0, gemm_sk_flag_ints(m->num_sms) * 4) != cudaSuccess) {
      free_model(m);
      return GPT_ECUDA;
    }
  } else {
    m->logits_ws = reinterpret_cast<float*>(m->ws + o_logits);
  }
  m->nll = reinterpret_cast<float*>(m->ws + o_nll);
  m->block_sums = reinterpret_cast<float*>(m->ws + o_bsum);
  m->err = reinterpret_cast<int*>(m->ws + o_err);
  m->attn_sched = m->err + 16;
  m->stage_ids = reinterpret_cast<int32_t*>(m->ws + o_ids);
  m->stage_tg = reinterpret_cast<int32_t*>(m->ws + o_tg);
  m->stage_loss = reinterpret_cast<float*>(m->ws + o_loss);
  if (cudaMemset(m->err, 0, 256) != cudaSuccess) { free_model(m); return GPT_ECUDA; }
  if (cudaMallocHost(&m->h_pinned, 64) != cudaSuccess) { free_model(m); return GPT_ENOMEM; }
  *out = m;
  return GPT_OK;
}

int gpt_kv_reserve(gpt_model* m, int32_t max_batch) {
  if (!m || max_batch < 1) return GPT_EINVAL;
  if (!m->bf16) return GPT_ECONFIG;
  if (max_batch <= m->kv_batch) return GPT_OK;
  const size_t bytes = static_cast<size_t>(m->cfg.L) * max_batch * m->cfg.ctx * 2 * m->cfg.C * 2;
  if (!m->dec_pos && cudaMalloc(&m->dec_pos, sizeof(int)) != cudaSuccess) return GPT_ENOMEM;
  uint8_t* p = nullptr;
  if (bytes > 0 && cudaMalloc(&p, bytes) != cudaSuccess) return GPT_ENOMEM;
  cudaDeviceSynchronize();                  // no launch may still use the old cache
  cudaFree(m->kv);
  m->kv = p;
  m->kv_batch = max_batch;
  if (m->dec_exec) {                        // the captured step holds the old cache's address
    cudaGraphExecDestroy(m->dec_exec);
    m->dec_exec = nullptr;
  }
  return GPT_OK;
}

void gpt_destroy(gpt_model* m) {
  if (!m) return;
  cudaDeviceSynchronize();
  free_model(m);
}

}  // extern "C"
