// Shared device/host helpers of libbd (CUDA, sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bd.h"

#define BD_API extern "C" __attribute__((visibility("default")))

namespace bd {

// First device-side error wins; the caller's status word starts at 0.
__device__ __forceinline__ void flag_error(int32_t *dev_status, int32_t code) {
  if (dev_status) atomicCAS(dev_status, 0, code);
}

// Programmatic dependent launch: every kernel of the library is launched so
// that it may start while the previous kernel on the stream drains.  A kernel
// calls pdl_wait() before it touches global memory that earlier stream work
// writes or reads, and pdl_trigger() once its own dependents may be scheduled.
// Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Whether any of the block_len (<= 32) tokens is still masked; one load per
// lane, so the answer costs one memory latency.  Call with the full warp.
__device__ __forceinline__ bool block_has_mask(const int32_t *tokens, int block_len) {
  const int lane = threadIdx.x & 31;
  const bool m = lane < block_len && tokens[lane] == BD_MASK;
  return __any_sync(0xffffffffu, m);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Online-softmax state of one row: running max m, running sum s of
// exp(l - m), and the lowest index attaining m.
struct MaxSumArg {
  float m;
  float s;
  int32_t idx;
};

// Merge b into a.  Deterministic: on equal maxima the lower index wins and
// both sums are kept.
__device__ __forceinline__ MaxSumArg merge(MaxSumArg a, MaxSumArg b) {
  if (b.m > a.m || (b.m == a.m && b.idx < a.idx)) {
    MaxSumArg t = a;
    a = b;
    b = t;
  }
  // a.m >= b.m now
  if (b.s > 0.f) a.s += b.s * __expf(b.m - a.m);
  return a;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launch counter behind bd_kernel_launches(); every host entry point adds
// the number of kernels it launched.
void count_launches(int n);

// Device facts of the current device (cached per device; zeros when no GPU).
struct DevInfo {
  int sms = 0;
  int major = 0;
};
DevInfo dev_info();

// TMA tensor maps over bf16 tensors with a 128-byte swizzle.  dims[0] is the
// innermost (contiguous) extent; strides_bytes[i] is the stride of dim i+1.
bool tma_available();
bool tma_encode_bf16(CUtensorMap *m, int rank, const void *base, const uint64_t *dims,
                     const uint64_t *strides_bytes, const uint32_t *box);

// Load a kernel's module and allow it the largest dynamic shared memory the
// device offers.  Done once per device before first use (kernel modules load
// lazily, and a first load inside a CUDA-graph capture is not allowed).
template <typename... KArgs>
inline bool preload_kernel(void (*kernel)(KArgs...), bool dyn_smem) {
  if (dyn_smem) {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
      return false;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) ==
           cudaSuccess;
  }
  cudaFuncAttributes attr;
  return cudaFuncGetAttributes(&attr, kernel) == cudaSuccess;
}

// Preload every kernel of the library on the current device (idempotent).
bool preload_all();
bool preload_attention_simt();
bool preload_attention_tc();
bool preload_attention_tc5();
bool preload_confidence();
bool preload_lmhead_tc();

inline bd_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

}  // namespace bd
