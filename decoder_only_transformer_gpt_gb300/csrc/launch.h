// Kernel launch with Programmatic Dependent Launch (host side).
//
// A kernel launched this way may start (and run its prologue: barrier set-up,
// TMEM allocation, descriptor prefetch) while the previous kernel on the stream
// is still finishing. Every kernel launched through here executes
// griddepcontrol.wait (pdl_wait) before its first global-memory access, which
// returns only once the previous grid has completed and its writes are visible,
// so results are unchanged. Set GPT_GB300_NO_PDL=1 to launch without overlap.
#pragma once

#include <cuda_runtime.h>

#include <cstdlib>
#include <utility>

namespace gptgb {

inline bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("GPT_GB300_NO_PDL");
    return !(v && v[0] == '1');
  }();
  return on;
}

// The CTA-pair (cluster of two) kernels where a product has one; GPT_GB300_NO_PAIR=1 uses the
// single-CTA kernels everywhere.
inline bool pair_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("GPT_GB300_NO_PAIR");
    return !(v && v[0] == '1');
  }();
  return on;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace gptgb
