// Shared device helpers of libspectree (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <stdlib.h>

#include <nvtx3/nvToolsExt.h>

#include "spectree.h"

#define SPEC_MAX_NODES 1024
#define SPEC_MAX_WORDS (SPEC_MAX_NODES / 64)
#define SPEC_MAX_VOCAB 131072

namespace spectree {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace spectree

// Host helpers.

// An NVTX range around one C-ABI call (named after the call), for profilers
// that show ranges; without a tool attached the calls cost a few nanoseconds.
struct SpecNvtxRange {
  explicit SpecNvtxRange(const char* name) { nvtxRangePushA(name); }
  ~SpecNvtxRange() { nvtxRangePop(); }
};
#define SPEC_NVTX_RANGE(name) SpecNvtxRange spec_nvtx_range_(name)

// Debug switch: with SPECTREE_WORKSPACE_CANARY=1 in the environment, calls
// that take a workspace first fill it with 0xFF bytes (NaN floats, all-ones
// integers), so that a read of scratch the call did not write shows up in
// the results.  Off by default; read at every call.
inline void spec_workspace_canary(void* ws, size_t bytes, cudaStream_t stream) {
  const char* e = getenv("SPECTREE_WORKSPACE_CANARY");
  if (e && e[0] == '1' && ws && bytes) cudaMemsetAsync(ws, 0xFF, bytes, stream);
}
#define SPEC_LAUNCH_CHECK()                       \
  do {                                            \
    if (cudaGetLastError() != cudaSuccess)        \
      return SPEC_ERR_CUDA;                       \
  } while (0)
