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

// launch_pdl for a kernel launched as clusters of `cluster` CTAs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                      size_t smem, cudaStream_t st, dim3 cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster.x;
  attr[1].val.clusterDim.y = cluster.y;
  attr[1].val.clusterDim.z = cluster.z;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
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

// State of one row under temperature sampling (Gumbel-max): the online
// softmax of z = l / temperature (max m, sum s of exp(z - m)) and the best
// perturbed key z + G seen so far (key kb, its z zb and its index idx).
struct SampleState {
  float m;
  float s;
  float kb;
  float zb;
  int32_t idx;
};

// Merge two sampling states: sums rescaled to the larger max; the larger key
// wins, equal keys keep the lower index.
__device__ __forceinline__ void merge_sample_into(float &m, float &s, float &kb, float &zb,
                                                  int &i, float bm, float bs, float bkb,
                                                  float bzb, int bi) {
  const float mm = fmaxf(m, bm);
  s = (s > 0.f ? s * __expf(m - mm) : 0.f) + (bs > 0.f ? bs * __expf(bm - mm) : 0.f);
  m = mm;
  const bool take = bkb > kb || (bkb == kb && bi < i);
  kb = take ? bkb : kb;
  zb = take ? bzb : zb;
  i = take ? bi : i;
}

__device__ __forceinline__ SampleState merge(SampleState a, const SampleState &b) {
  merge_sample_into(a.m, a.s, a.kb, a.zb, a.idx, b.m, b.s, b.kb, b.zb, b.idx);
  return a;
}

// Philox-4x64 with 10 rounds (Salmon, Moraes, Dror and Shaw, "Parallel random
// numbers: as easy as 1, 2, 3", SC'11): a round multiplies c0 and c2 by the
// two round constants into 128-bit products and mixes the halves with c1, c3
// and the key; the key steps by the two Weyl constants between rounds.
__device__ __forceinline__ void philox4x64_10(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3,
                                              uint64_t k0, uint64_t k1, uint64_t (&out)[4]) {
  constexpr uint64_t kM0 = 0xD2E7470EE14C6C93ull, kM1 = 0xCA5A826395121157ull;
  constexpr uint64_t kW0 = 0x9E3779B97F4A7C15ull, kW1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint64_t h0 = __umul64hi(kM0, c0), l0 = kM0 * c0;
    const uint64_t h1 = __umul64hi(kM1, c2), l1 = kM1 * c2;
    c0 = h1 ^ c1 ^ k0;
    c1 = l1;
    c2 = h0 ^ c3 ^ k1;
    c3 = l0;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

// The 23-bit field of position id pos in its Philox block (the block serves
// the eight positions 8k..8k+7): word (pos / 2) % 4, bits 41..63 for even pos
// and bits 9..31 for odd pos.
__device__ __forceinline__ uint32_t philox_field(const uint64_t (&w)[4], int pos) {
  const int k = (pos >> 1) & 3;
  const uint64_t word = k == 0 ? w[0] : k == 1 ? w[1] : k == 2 ? w[2] : w[3];
  return (pos & 1) ? static_cast<uint32_t>(word >> 9) & 0x7FFFFFu
                   : static_cast<uint32_t>(word >> 41);
}

// Gumbel noise G = -ln(-ln U) of U = (field + 1/2) / 2^23, a value fp32 holds
// exactly.  x = -ln U comes from the Taylor series of -ln(1 - d), d = 1 - U,
// while d < 2^-6 (four terms, relative error below 2^-26), which keeps x
// accurate near U = 1 where G is largest; elsewhere from the fast logarithm
// (absolute error about 2^-21 near U = 1/2, so relative error below 1e-4 of x
// and below 1e-4 in G).
__device__ __forceinline__ float gumbel_of_field(uint32_t field) {
  const float u = (static_cast<float>(field) + 0.5f) * 1.1920928955078125e-07f;   // 2^-23
  const float d = (static_cast<float>(0x7FFFFFu - field) + 0.5f) * 1.1920928955078125e-07f;
  const float series = d * (1.f + d * (0.5f + d * (0.33333334f + d * 0.25f)));
  const float x = d < 0.015625f ? series : -__logf(u);
  return -__logf(x);
}

// Gumbel noise of vocabulary entry v at position id pos: Philox block at
// counter (v, pos / 8, draw, 0) under key (seed, 0).
__device__ __forceinline__ float gumbel_at(int v, int pos, uint64_t seed, uint64_t draw) {
  uint64_t w[4];
  philox4x64_10(static_cast<uint64_t>(v), static_cast<uint64_t>(pos >> 3), draw, 0ull, seed, 0ull,
                w);
  return gumbel_of_field(philox_field(w, pos));
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
    cudaFuncAttributes attr;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaFuncGetAttributes(&attr, kernel) != cudaSuccess)
      return false;
    // the opt-in limit covers static and dynamic shared memory together
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                optin - (int)attr.sharedSizeBytes) == cudaSuccess;
  }
  cudaFuncAttributes attr;
  return cudaFuncGetAttributes(&attr, kernel) == cudaSuccess;
}

// Preload every kernel of the library on the current device (idempotent).
bool preload_all();
bool preload_attention_simt();
bool preload_attention_tc();
bool preload_confidence();
bool preload_lmhead_tc();
bool preload_decoder();
bool preload_attention_pair();
bool preload_truncated();
bool preload_parallel();

inline bd_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

}  // namespace bd
