// Internal state of a model handle (shared by the library's translation units).
#pragma once

#include "../../include/gpt.h"
#include "kernels.h"

#include <vector>

struct gpt_layer_dev {
  void *attn_w, *proj_w, *fc_w, *mp_w;                     // bf16 or fp32 [out, in]
  float *attn_b, *proj_b, *fc_b, *mp_b, *ln1_g, *ln1_b, *ln2_g, *ln2_b;
  CUtensorMap tm_attn_w, tm_proj_w, tm_fc_w, tm_mp_w;      // bf16 path only
  CUtensorMap tm_attn_w_pair, tm_proj_w_pair, tm_fc_w_pair, tm_mp_w_pair;   // 128-row boxes (launch_gemm_pair)
};

struct gpt_train;                 // backward-pass workspace and gradients (gpt_backward.cu)

struct gpt_model {
  gpt_config cfg;
  int device = 0;
  int num_sms = 0;
  int bf16 = 0;
  // weights
  uint8_t* wbuf = nullptr;
  void* wte = nullptr;
  void* wpe = nullptr;
  std::vector<gpt_layer_dev> layers;
  float* lnf_g = nullptr;
  float* lnf_b = nullptr;
  CUtensorMap tm_wte;
  void* head = nullptr;     // the head's [V, C] matrix: wte when tied, its own storage when untied
  CUtensorMap tm_head;
  // workspace
  uint8_t* ws = nullptr;
  float* x = nullptr;       // residual stream fp32 [Mx, C]
  void* a = nullptr;        // LN output / GEMM input [Mx, C] (bf16 or fp32)
  void* qkv = nullptr;      // [Mx, 3C]
  void* y = nullptr;        // attention output [Mx, C]
  void* g = nullptr;        // MLP hidden [Mx, ffn]
  float* pmax = nullptr;    // [NB, Mx]
  float* psum = nullptr;
  float* ztgt = nullptr;    // [Mx]
  float* nll = nullptr;     // [Mx]
  float* block_sums = nullptr;  // [ce_combine_blocks(Mx)] per-block sums of nll
  float* logits_ws = nullptr;   // fp32 path: [Mx, V]
  float* sk_part = nullptr;     // bf16 path: stream-K partial tiles of the block projections
  int* sk_flag = nullptr;       // and their flags (zero between launches)
  // failure-detection check (gpt_debug_expire_waits): the next bf16 forward's finishing CTAs wait on
  // these flags, which nothing sets, for at most dbg_wait_limit SM cycles
  int* dbg_flag = nullptr;
  long long dbg_wait_limit = 0;
  bool dbg_armed = false;
  // key/value cache for incremental decoding: per layer [kv_batch][ctx][2C] bf16
  uint8_t* kv = nullptr;
  int kv_batch = 0;
  bool kv_fill = false;         // the next bf16 forward also stores keys and values (prefill)
  int* dec_pos = nullptr;       // device int: the position of the decode step being run
  cudaStream_t cap_stream = nullptr;   // where a decode step is captured into a CUDA graph
  cudaGraphExec_t dec_exec = nullptr;  // the captured decode step, for dec_B rows into dec_logits
  int dec_B = 0;
  float* dec_logits = nullptr;
  int dec_launches = 0;
  // the captured forward pass, for one set of arguments and one timing probe (see gpt_forward)
  cudaGraph_t fwd_graph = nullptr;
  cudaGraphExec_t fwd_exec = nullptr;
  const void* fwd_key[8] = {};
  cudaGraphNode_t fwd_ev_node[2] = {nullptr, nullptr};   // the probe's event-record nodes
  int fwd_launches = 0;
  int fwd_probe_hits = 0;
  bool capturing = false;       // a forward or decode step is being captured into a graph
  gpt_train* tr = nullptr;      // allocated by the first gpt_backward
  int* err = nullptr;       // device error word
  int* attn_sched = nullptr;   // attention work counter (2 ints, zero between launches)
  int32_t* stage_ids = nullptr;
  int32_t* stage_tg = nullptr;
  float* stage_loss = nullptr;
  float* stage_logits = nullptr;   // lazily allocated for gpt_forward_host with logits
  size_t stage_logits_elems = 0;
  int* h_pinned = nullptr;  // [0] error word, [1] loss bits
  // activation descriptors, rebuilt when (B, T) changes
  // timing probe (gpt_time_step) and launch counter
  int prof_step = -1, prof_layer = -1;
  cudaEvent_t prof_ev0 = nullptr, prof_ev1 = nullptr;
  int launches = 0;
  int probe_hits = 0;       // launches the armed probe bracketed in the last forward
  int cached_B = -1, cached_T = -1;
  CUtensorMap tm_a, tm_y, tm_g, tm_qkv;            // GEMM A operands and the attention input
  CUtensorMap tm_qkv_out, tm_g_out, tm_x_out;      // GEMM epilogue outputs (TMA store / reduce-add)
};

namespace gptgb {
void free_train(gpt_model* m);     // releases m->tr (gpt_backward.cu)
// gpt_forward.cu: the forward pass's activation descriptors for (B, T); one tcgen05 GEMM launch
// (stream-K workspace attached); the (B, T) checks of gpt_forward.
int forward_maps(gpt_model* m, int B, int T);
int gemm_bf16(gpt_model* m, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC, int M, int N,
              int K, const float* bias, void* out, int epi, cudaStream_t s);
// c_fc of the training forward: g = gelu(a W^T + b) through tm_g and the GELU's input u through tm_u.
// A product with epi EPI_BIAS_RESID (out fp32 += A W^T + bias), EPI_F32_OUT (out fp32 = A W^T + bias),
// EPI_BIAS_OUT or EPI_BIAS_GELU_OUT (bf16 out) through tmC: on CTA pairs where they pay and can run
// (tmB_pair: W with 128-row boxes), else as gemm_bf16.
int gemm_bf16_long(gpt_model* m, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmB_pair,
                   const CUtensorMap& tmC, int M, int N, int K, const float* bias, void* out, int epi, cudaStream_t s);
int gemm_bf16_gelu_u(gpt_model* m, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tm_g,
                     const CUtensorMap& tm_u, int M, int N, int K, const float* bias, void* g, cudaStream_t s);
int shape_ok(const gpt_model* m, int B, int T);
// thread-local text of the last failing CUDA call
void set_detail(const char* what, cudaError_t e);
void set_detail_text(const char* text);
}  // namespace gptgb

#define GPT_CUDA(call)                                  \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) {                            \
      ::gptgb::set_detail(#call, e_);                   \
      return GPT_ECUDA;                                 \
    }                                                   \
  } while (0)
