// Per-step entry points (include/gpt_kernels.h): one kernel of the forward pass
// on caller-owned device buffers.
#include "../../include/gpt_kernels.h"
#include "model.h"

#include <cuda_runtime.h>

#include <mutex>

using namespace gptgb;

namespace {

int* g_err = nullptr;
std::mutex g_err_mu;

int* err_word() {
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err) {
    if (cudaMalloc(&g_err, sizeof(int)) != cudaSuccess) { g_err = nullptr; return nullptr; }
    if (cudaMemset(g_err, 0, sizeof(int)) != cudaSuccess) return nullptr;
  }
  return g_err;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

int gptk_gemm(const void* A, const void* W, const float* bias, void* out, int32_t M, int32_t N, int32_t K,
              int32_t epilogue, int32_t dtype, void* stream) {
  if (!A || !W || !out || M < 0 || N <= 0 || K <= 0) return GPT_EINVAL;
  if (epilogue < 0 || epilogue > 3) return GPT_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) return GPT_OK;
  if (dtype == 0) {
    GPT_CUDA(launch_gemm_simt(reinterpret_cast<const float*>(A), reinterpret_cast<const float*>(W), bias,
                              reinterpret_cast<float*>(out), M, N, K, N, epilogue, 0, s));
    return GPT_OK;
  }
  if (dtype != 1 || (K % 8) || (N % 8) || !aligned16(A) || !aligned16(W) || !aligned16(out)) return GPT_EINVAL;
  int* err = err_word();
  if (!err) return GPT_ENOMEM;
  CUtensorMap tmA, tmB, tmC = {};
  if (!make_tmap_2d_bf16(&tmA, A, M, K, kGemmBM) || !make_tmap_2d_bf16(&tmB, W, N, K, gemm_tc_bn())) {
    set_detail_text("gemm tensor map");
    return GPT_ECUDA;
  }
  bool ok_c = true;
  if (epilogue == GPTK_EPI_BIAS || epilogue == GPTK_EPI_BIAS_GELU) ok_c = make_tmap_2d(&tmC, out, 2, M, N, 64, kEpiRows);
  else if (epilogue == GPTK_EPI_BIAS_RESID) ok_c = make_tmap_2d(&tmC, out, 4, M, N, 32, kEpiRows);
  if (!ok_c) {
    set_detail_text("gemm output tensor map");
    return GPT_ECUDA;
  }
  GemmArgs a{};
  a.M = M; a.N = N; a.K = K;
  a.bias = bias; a.out = out; a.ldo = N;
  a.err = err;
  a.m_fastest = N > M ? 1 : 0;
  const int grid = num_sms();
  uint8_t* skws = nullptr;                 // stream-K partial tiles + flags, on the stream
  if (gemm_tc_stream_k(M, N, K, epilogue, grid)) {
    const size_t pbytes = gemm_sk_part_floats(grid) * sizeof(float);
    const size_t fbytes = gemm_sk_flag_ints(grid) * sizeof(int);
    GPT_CUDA(cudaMallocAsync(reinterpret_cast<void**>(&skws), pbytes + fbytes, s));
    a.sk_part = reinterpret_cast<float*>(skws);
    a.sk_flag = reinterpret_cast<int*>(skws + pbytes);
    const cudaError_t e = cudaMemsetAsync(a.sk_flag, 0, fbytes, s);
    if (e != cudaSuccess) {
      cudaFreeAsync(skws, s);
      set_detail("cudaMemsetAsync", e);
      return GPT_ECUDA;
    }
  }
  const cudaError_t e = launch_gemm_tc(tmA, tmB, tmC, a, epilogue, grid, s);
  if (skws) cudaFreeAsync(skws, s);
  if (e != cudaSuccess) {
    set_detail("launch_gemm_tc", e);
    return GPT_ECUDA;
  }
  return GPT_OK;
}

int gptk_gemm_pair(const void* A, const void* W, const float* bias, void* out, int32_t M, int32_t N, int32_t K,
                   int32_t epilogue, int32_t ksplit, void* stream) {
  if (!A || !W || !out || M < 0 || N <= 0 || K <= 0) return GPT_EINVAL;
  if (epilogue < GPTK_EPI_BIAS || epilogue > GPTK_EPI_F32) return GPT_EINVAL;
  if (ksplit > 1 && epilogue != GPTK_EPI_BIAS_RESID) return GPT_EINVAL;
  if ((K % 8) || (N % 8) || !aligned16(A) || !aligned16(W) || !aligned16(out)) return GPT_EINVAL;
  if (ksplit > 1 && (bias != nullptr || ksplit > (K + kGemmBK - 1) / kGemmBK)) return GPT_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) return GPT_OK;
  if (gemm_pair_capacity() <= 0) return GPT_ECONFIG;
  int* err = err_word();
  if (!err) return GPT_ENOMEM;
  CUtensorMap tmA, tmB, tmC;
  const bool bf16_out = epilogue == GPTK_EPI_BIAS || epilogue == GPTK_EPI_BIAS_GELU;
  if (!make_tmap_2d_bf16(&tmA, A, M, K, kGemmBM) || !make_tmap_2d_bf16(&tmB, W, N, K, kGemmBM) ||
      !(bf16_out ? make_tmap_2d(&tmC, out, 2, M, N, 64, kEpiRows) : make_tmap_2d(&tmC, out, 4, M, N, 32, kEpiRows))) {
    set_detail_text("gemm tensor map");
    return GPT_ECUDA;
  }
  GemmArgs a{};
  a.M = M; a.N = N; a.K = K;
  a.bias = bias; a.out = out; a.ldo = N;
  a.err = err;
  a.m_fastest = N > M ? 1 : 0;
  a.ksplit = ksplit > 1 ? ksplit : 0;
  const int grid = num_sms();
  uint8_t* skws = nullptr;                 // stream-K partial tiles + flags, on the stream
  if (ksplit <= 1 && gemm_pair_stream_k(M, N, K, grid / 2)) {
    const size_t pbytes = gemm_sk_part_floats(grid) * sizeof(float);
    const size_t fbytes = gemm_sk_flag_ints(grid) * sizeof(int);
    GPT_CUDA(cudaMallocAsync(reinterpret_cast<void**>(&skws), pbytes + fbytes, s));
    a.sk_part = reinterpret_cast<float*>(skws);
    a.sk_flag = reinterpret_cast<int*>(skws + pbytes);
    const cudaError_t e = cudaMemsetAsync(a.sk_flag, 0, fbytes, s);
    if (e != cudaSuccess) {
      cudaFreeAsync(skws, s);
      set_detail("cudaMemsetAsync", e);
      return GPT_ECUDA;
    }
  }
  const int epi = epilogue == GPTK_EPI_BIAS ? EPI_BIAS_OUT
                  : epilogue == GPTK_EPI_BIAS_GELU ? EPI_BIAS_GELU_OUT
                  : epilogue == GPTK_EPI_F32 ? EPI_F32_OUT : EPI_BIAS_RESID;
  const cudaError_t e = launch_gemm_pair(tmA, tmB, tmC, a, epi, grid / 2, s);
  if (skws) cudaFreeAsync(skws, s);
  if (e != cudaSuccess) {
    set_detail("launch_gemm_pair", e);
    return GPT_ECUDA;
  }
  return GPT_OK;
}

int gptk_attention(const void* qkv, void* y, int32_t B, int32_t T, int32_t H, int32_t D, int32_t dtype,
                   void* stream) {
  if (!qkv || !y || B < 1 || T < 1 || H < 1 || D < 1) return GPT_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == 0) {
    GPT_CUDA(launch_attention_simt(reinterpret_cast<const float*>(qkv), reinterpret_cast<float*>(y), B, T, H, D, s));
    return GPT_OK;
  }
  if (dtype != 1 || (D != 32 && D != 64) || !aligned16(qkv) || !aligned16(y)) return GPT_ECONFIG;
  int* err = err_word();
  if (!err) return GPT_ENOMEM;
  CUtensorMap tm;
  if (!make_tmap_qkv(&tm, qkv, B, T, 3 * H * D, D)) {
    set_detail_text("qkv tensor map");
    return GPT_ECUDA;
  }
  int* sched = nullptr;                    // the kernel's work counter, zeroed, on the stream
  GPT_CUDA(cudaMallocAsync(reinterpret_cast<void**>(&sched), 2 * sizeof(int), s));
  cudaError_t e = cudaMemsetAsync(sched, 0, 2 * sizeof(int), s);
  if (e == cudaSuccess) e = launch_attention_tc(tm, y, B, T, H, D, err, sched, s);
  cudaFreeAsync(sched, s);
  if (e != cudaSuccess) {
    set_detail("attention", e);
    return GPT_ECUDA;
  }
  return GPT_OK;
}

int gptk_attention_lse(const void* qkv, void* y, float* lse2, int32_t B, int32_t T, int32_t H, int32_t D,
                       void* stream) {
  if (!qkv || !y || !lse2 || B < 1 || T < 1 || H < 1 || D < 1) return GPT_EINVAL;
  if ((D != 32 && D != 64) || !aligned16(qkv) || !aligned16(y)) return GPT_ECONFIG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* err = err_word();
  if (!err) return GPT_ENOMEM;
  CUtensorMap tm;
  if (!make_tmap_qkv(&tm, qkv, B, T, 3 * H * D, D)) {
    set_detail_text("qkv tensor map");
    return GPT_ECUDA;
  }
  int* sched = nullptr;
  GPT_CUDA(cudaMallocAsync(reinterpret_cast<void**>(&sched), 2 * sizeof(int), s));
  cudaError_t e = cudaMemsetAsync(sched, 0, 2 * sizeof(int), s);
  if (e == cudaSuccess) e = launch_attention_tc(tm, y, B, T, H, D, err, sched, s, lse2);
  cudaFreeAsync(sched, s);
  if (e != cudaSuccess) {
    set_detail("attention", e);
    return GPT_ECUDA;
  }
  return GPT_OK;
}

int gptk_attention_bwd(const void* qkv, const void* y, const void* dy, const float* lse2, void* dqkv, int32_t B,
                       int32_t T, int32_t H, int32_t D, void* stream) {
  if (!qkv || !y || !dy || !lse2 || !dqkv || B < 1 || T < 1 || H < 1 || D < 1) return GPT_EINVAL;
  if ((D != 32 && D != 64) || !aligned16(qkv) || !aligned16(y) || !aligned16(dy) || !aligned16(dqkv))
    return GPT_ECONFIG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* err = err_word();
  if (!err) return GPT_ENOMEM;
  const int C = H * D;
  const size_t M = static_cast<size_t>(B) * T;
  // scratch on the stream: dQ accumulator, Dsum and the work counter (zeroed)
  const size_t acc_b = M * C * sizeof(float), dsum_b = M * H * sizeof(float), cnt_b = 2 * sizeof(int);
  uint8_t* ws = nullptr;
  GPT_CUDA(cudaMallocAsync(reinterpret_cast<void**>(&ws), acc_b + dsum_b + cnt_b, s));
  float* dqacc = reinterpret_cast<float*>(ws);
  float* dsum = reinterpret_cast<float*>(ws + acc_b);
  int* sched = reinterpret_cast<int*>(ws + acc_b + dsum_b);
  CUtensorMap tq, tdy, tdkv, tdq;
  cudaError_t e = cudaMemsetAsync(sched, 0, cnt_b, s);
  if (e == cudaSuccess &&
      !(make_tmap_qkv(&tq, qkv, B, T, 3 * C, D) && make_tmap_qkv(&tdy, dy, B, T, C, D) &&
        make_tmap_attn_out(&tdkv, dqkv, B, T, 3 * C, D) && make_tmap_bt_f32(&tdq, dqacc, B, T, C))) {
    cudaFreeAsync(ws, s);
    set_detail_text("attention derivative tensor maps");
    return GPT_ECUDA;
  }
  if (e == cudaSuccess)
    e = launch_attention_bwd_tc(tq, tdy, tdkv, tdq, y, dy, lse2, dsum, dqacc, dqkv, B, T, H, D, err, sched, s);
  cudaFreeAsync(ws, s);
  if (e != cudaSuccess) {
    set_detail("attention derivative", e);
    return GPT_ECUDA;
  }
  return GPT_OK;
}

int gptk_layernorm(const float* x, const float* g, const float* b, void* out, float* out_f32, int32_t M, int32_t C,
                   float eps, int32_t dtype, void* stream) {
  if (!x || !g || !b || !out || M < 0 || C <= 0 || (C % 8) || C > 2048) return GPT_EINVAL;
  if (dtype != 0 && dtype != 1) return GPT_EINVAL;
  GPT_CUDA(launch_layernorm(x, g, b, out, dtype, out_f32, M, C, eps, reinterpret_cast<cudaStream_t>(stream)));
  return GPT_OK;
}

int gptk_embed(const int32_t* ids, const void* wte, const void* wpe, float* x, int32_t B, int32_t T, int32_t C,
               int32_t V, int32_t dtype, void* stream) {
  if (!ids || !wte || !wpe || !x || B < 1 || T < 1 || C <= 0 || (C % 8) || C > 2048 || V < 1) return GPT_EINVAL;
  if (dtype != 0 && dtype != 1) return GPT_EINVAL;
  int* err = err_word();
  if (!err) return GPT_ENOMEM;
  GPT_CUDA(launch_embed(ids, wte, wpe, dtype, x, nullptr, 0, 0, nullptr, nullptr, B * T, T, C, V, 0.0f, err,
                        reinterpret_cast<cudaStream_t>(stream)));
  return GPT_OK;
}

int gptk_lmhead_ce(const void* h, const void* wte, const int32_t* targets, float* nll, float* logits, int32_t M,
                   int32_t V, int32_t C, int32_t dtype, void* stream) {
  if (!h || !wte || !targets || !nll || M < 0 || V < 1 || C < 1) return GPT_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M == 0) return GPT_OK;
  int* err = err_word();
  if (!err) return GPT_ENOMEM;
  if (dtype == 0) {
    float* z = logits;
    if (!z) GPT_CUDA(cudaMallocAsync(reinterpret_cast<void**>(&z), (size_t)M * V * sizeof(float), s));
    GPT_CUDA(launch_gemm_simt(reinterpret_cast<const float*>(h), reinterpret_cast<const float*>(wte), nullptr, z, M,
                              V, C, V, EPI_F32, 0, s));
    GPT_CUDA(launch_ce_rows(z, targets, nll, M, V, err, s));
    if (!logits) GPT_CUDA(cudaFreeAsync(z, s));
    return GPT_OK;
  }
  if (dtype != 1 || (C % 8) || !aligned16(h) || !aligned16(wte)) return GPT_EINVAL;
  CUtensorMap tmA, tmB;
  if (!make_tmap_2d_bf16(&tmA, h, M, C, kGemmBM) || !make_tmap_2d_bf16(&tmB, wte, V, C, gemm_tc_bn())) {
    set_detail_text("head tensor map");
    return GPT_ECUDA;
  }
  const int NB = gemm_tc_num_ntiles(V);
  float* scratch = nullptr;        // pmax [NB, M], psum [NB, M], ztgt [M]
  GPT_CUDA(cudaMallocAsync(reinterpret_cast<void**>(&scratch), ((size_t)2 * NB + 1) * M * sizeof(float), s));
  GemmArgs a{};
  a.M = M; a.N = V; a.K = C;
  a.ldo = V;
  a.targets = targets;
  a.pmax = scratch;
  a.psum = scratch + (size_t)NB * M;
  a.ztgt = scratch + (size_t)2 * NB * M;
  a.logits = logits;
  a.err = err;
  a.m_fastest = 1;
  cudaError_t e = launch_gemm_tc(tmA, tmB, tmA, a, EPI_CE, num_sms(), s);
  if (e == cudaSuccess) e = launch_ce_combine(a.pmax, a.psum, a.ztgt, targets, nll, nullptr, M, NB, V, err, s);
  cudaFreeAsync(scratch, s);
  if (e != cudaSuccess) {
    set_detail("lmhead_ce", e);
    return GPT_ECUDA;
  }
  return GPT_OK;
}

int gptk_mean(const float* nll, int32_t M, float* loss, void* stream) {
  if (!nll || !loss || M < 1) return GPT_EINVAL;
  GPT_CUDA(launch_mean(nll, M, M, loss, reinterpret_cast<cudaStream_t>(stream)));
  return GPT_OK;
}

int gptk_status(void* stream) {
  int* err = err_word();
  if (!err) return GPT_ENOMEM;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int h = 0;
  GPT_CUDA(cudaStreamSynchronize(s));
  GPT_CUDA(cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost));
  GPT_CUDA(cudaMemset(err, 0, sizeof(int)));
  if (h == GPT_DEV_OK) return GPT_OK;
  if (h == GPT_DEV_ETOKEN || h == GPT_DEV_ETARGET) return GPT_ETOKEN;
  return GPT_EDEVICE;
}

}  // extern "C"
