// bd_confidence_commit_noalloc: the confidence/commit step with its
// workspace taken from a fixed device array instead of the caller.
//
// Why it exists: some callers cannot allocate device memory at the point
// where they run a denoise step.  Serving runtimes often forbid allocation
// while a request is in flight (cudaMalloc can synchronise the device and
// break the server's fixed memory budget); plugins hosted by another
// framework get no handle to that framework's allocator; embedded callers
// may run with every byte of device memory already handed out at start-up.  Such callers still own the inputs and the
// outputs, but they have nowhere to put the scratch space that
// bd_confidence_commit needs (masked-row list, compact copy of the masked
// rows, per-CTA partial softmax states).  This file gives them one: a
// file-scope __device__ array of kScratchBytes that every GPU which loads
// the library holds until the process exits.
//
// Rules of use (also stated in bd.h):
//  - The first call on a device looks up the array's device address with
//    cudaGetSymbolAddress while that device is current; make that first call
//    before any stream capture begins.  Later calls reuse the cached address,
//    so every call must run in the device's primary context (the one the
//    runtime API uses), and the process must not call cudaDeviceReset after
//    the first call: the array, and its address, belong to that context.
//  - Every call on a device shares the one array and leaves its contents
//    behind.  Nothing in it has to start at zero (each call writes every
//    scratch value it later reads), but two calls whose executions overlap
//    on the GPU (different streams, no ordering between them) race on it.
//  - Shapes whose workspace exceeds kScratchBytes are rejected with
//    BD_ERR_WORKSPACE before anything is launched.
//  - Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "bd_common.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;  // 8 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per
// device); nullptr when the lookup fails.
void *scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

}  // namespace

BD_API bd_status bd_confidence_commit_noalloc(bd_dtype dtype, int32_t batch, int32_t block_len,
                                              int32_t hidden, int32_t vocab,
                                              const void *hidden_states, const void *lm_head,
                                              float threshold, int32_t *tokens, float *p_max,
                                              int32_t *argmax, int32_t *n_committed,
                                              int32_t *n_masked, int32_t *dev_status,
                                              void *stream) {
  const size_t need = bd_confidence_commit_workspace(dtype, batch, block_len, hidden, vocab);
  if (need == 0) return BD_ERR_INVALID_ARG;
  if (need > kScratchBytes) return BD_ERR_WORKSPACE;
  void *scratch = scratch_for_current_device();
  if (!scratch) return BD_ERR_CUDA;
  return bd_confidence_commit(dtype, batch, block_len, hidden, vocab, hidden_states, lm_head,
                              threshold, tokens, p_max, argmax, n_committed, n_masked, scratch,
                              kScratchBytes, dev_status, stream);
}
