// gptk_lmhead_ce_noalloc: the tied-head + cross-entropy step with its scratch
// in a fixed, file-scope device array instead of memory allocated per call.
//
// Who needs it: callers that must not allocate device memory while they run,
// for example a serving loop whose memory budget was fixed at start-up, a host
// framework whose caching allocator already owns the free device memory (so a
// plain cudaMalloc can fail although the framework could still serve the
// request), or a latency-critical loop that cannot afford the implicit device
// synchronisation that cudaMalloc/cudaFree may cause. Those callers pass their
// inputs and outputs and get the same result as gptk_lmhead_ce.
//
// The scratch (per-row, per-256-column-tile partial maxima and exp-sums, plus
// the target logits) lives in g_head_scratch below. Every GPU that loads this
// library holds that array until the process exits. All calls share it and it
// keeps the last call's contents; each call overwrites every element it reads,
// so nothing needs clearing. Calls whose GPU work overlaps in time (different
// streams without ordering, or several host threads) race on the array.
#include "../../include/gpt_kernels.h"
#include "model.h"

#include <cuda_runtime.h>

#include <mutex>

using namespace gptgb;

namespace {

constexpr size_t kScratchFloats = size_t(2) * 1024 * 1024;     // 8 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) float g_head_scratch[kScratchFloats];

float* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// The device address of g_head_scratch on the current device. The host-side
// name of a __device__ array is only a stand-in, so the address is looked up
// once per device with that device current.
int scratch_address(float** out) {
  int dev = 0;
  GPT_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) {
    set_detail_text("gptk_lmhead_ce_noalloc: device index out of range");
    return GPT_EUNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    GPT_CUDA(cudaGetSymbolAddress(&p, g_head_scratch));
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return GPT_OK;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n;
}

}  // namespace

extern "C" int gptk_lmhead_ce_noalloc(const void* h, const void* wte, const int32_t* targets, float* nll,
                                      int32_t M, int32_t V, int32_t C, int32_t* d_err, void* stream) {
  if (!h || !wte || !targets || !nll || M < 0 || V < 1 || C < 1 || (C % 8)) return GPT_EINVAL;
  if ((reinterpret_cast<uintptr_t>(h) & 15u) || (reinterpret_cast<uintptr_t>(wte) & 15u)) return GPT_EINVAL;
  if (M == 0) return GPT_OK;
  const int NB = gemm_tc_num_ntiles(V);
  const size_t need = (size_t(2) * NB + 1) * size_t(M);
  if (need > kScratchFloats) {
    set_detail_text("gptk_lmhead_ce_noalloc: M * (2 * ceil(V/256) + 1) exceeds the 2,097,152-float scratch");
    return GPT_EINVAL;
  }
  float* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != GPT_OK) return rc;
  CUtensorMap tmA, tmB;
  if (!make_tmap_2d_bf16(&tmA, h, M, C, kGemmBM) || !make_tmap_2d_bf16(&tmB, wte, V, C, gemm_tc_bn())) {
    set_detail_text("gptk_lmhead_ce_noalloc: tensor map");
    return GPT_ECUDA;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GemmArgs a{};
  a.M = M; a.N = V; a.K = C;
  a.ldo = V;
  a.targets = targets;
  a.pmax = scratch;
  a.psum = scratch + size_t(NB) * M;
  a.ztgt = scratch + size_t(2) * NB * M;
  a.logits = nullptr;
  a.err = reinterpret_cast<int*>(d_err);
  a.m_fastest = 1;
  GPT_CUDA(launch_gemm_tc(tmA, tmB, tmA, a, EPI_CE, sm_count(), s));
  GPT_CUDA(launch_ce_combine(a.pmax, a.psum, a.ztgt, targets, nll, nullptr, M, NB, V, a.err, s));
  return GPT_OK;
}
