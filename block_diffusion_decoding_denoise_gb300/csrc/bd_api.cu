// Host entry points of libbd: block attention dispatch, KV append, status.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "bd_attention.cuh"
#include "bd_common.cuh"

namespace bd {

static std::atomic<uint64_t> g_launches{0};
// kernel forced by bd_debug_force_attention_kernel (BD_ATTN_AUTO: by shape)
static std::atomic<int> g_forced_attention{BD_ATTN_AUTO};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

__global__ void append_kv_kernel(bd_paged_kv kv, int block_len, size_t elem_bytes,
                                 const char *k_blk, const char *v_blk, int32_t *ctx_len,
                                 const int32_t *n_masked, int32_t *dev_status);

bool preload_all() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (done[dev]) return true;
  const bool ok = preload_kernel(append_kv_kernel, false) && preload_attention_simt() &&
                  preload_attention_tc() && preload_confidence() &&
                  preload_lmhead_tc() && preload_decoder() && preload_attention_pair() &&
                  preload_truncated() && preload_parallel();
  if (!ok) {
    cudaGetLastError();
    return false;
  }
  done[dev] = true;
  return true;
}

static int num_sms() {
  static int cached = 0;
  if (cached == 0) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
      cached = n;
    else
      return 148;
  }
  return cached;
}

// KV split of the fp32 and tcgen05 kernels (page-aligned slices of the keys).
// Small problems (at most about 8 pages per SM in all) get one work item per
// SM, so every SM streams a few pages at once; larger ones get about four
// items per SM, each at least 8 pages long.  (The bf16 mma.sync kernel
// partitions the tiles itself, see attn_plan_kernel.)
// At most about 8 pages per SM in all.
static bool attn_small(int batch, int hkv, int block_len, int max_ctx) {
  const long long pages =
      (long long)batch * hkv * ((max_ctx + block_len + BD_PAGE_SIZE - 1) / BD_PAGE_SIZE);
  return pages <= 8LL * num_sms();
}

// `heads` counts the segments that are split: KV heads of all sequences, or
// head pairs for the head-pair kernel.
static void choose_split(int heads, int block_len, int max_ctx, int *num_splits,
                         int *split_keys) {
  const int sms = num_sms();
  const int nkeys = max_ctx + block_len;
  const long long pages = (long long)heads * ((nkeys + BD_PAGE_SIZE - 1) / BD_PAGE_SIZE);
  int keys;
  if (pages <= 8LL * sms) {
    // small problem: about one item per SM
    int s = std::max(1, (sms + heads - 1) / heads);
    s = std::min(s, std::max(1, (nkeys + BD_PAGE_SIZE - 1) / BD_PAGE_SIZE));
    keys = (nkeys + s - 1) / s;
  } else {
    // large problem: about four items per SM, each at least 8 pages long
    int s = std::max(1, (4 * sms + heads - 1) / heads);
    s = std::min(s, std::max(1, nkeys / (8 * BD_PAGE_SIZE)));
    keys = (nkeys + s - 1) / s;
  }
  keys = (keys + BD_PAGE_SIZE - 1) / BD_PAGE_SIZE * BD_PAGE_SIZE;
  *split_keys = keys;
  *num_splits = (nkeys + keys - 1) / keys;
}

static bool attn_shape_ok(int32_t batch, int32_t block_len, int32_t hq, int32_t hkv, int32_t d,
                          int32_t max_ctx) {
  if (batch < 1 || block_len < 1 || block_len > 32 || hq < 1 || hkv < 1 || hq % hkv) return false;
  if (d != 64 && d != 128) return false;
  if (block_len * (hq / hkv) > 128) return false;
  if (max_ctx < 0 || (int64_t)max_ctx + block_len > (1 << 30)) return false;
  return true;
}

// Every attention workspace starts with the head-pair kernel's merge jobs
// (eight ints per CTA of the persistent grid, rewritten by every call); the
// other buffers of a call follow them.
static size_t attn_job_bytes(int grid) { return align_up((size_t)grid * 8 * sizeof(int), 256); }

// Workspace of the tile-range partition: the plan (mma.sync kernel), then
// partial O and (m, l) for batch * hkv + 2 grid slots of R rows (the
// head-pair kernel needs batch * hkv / 2 + grid slots of 2R rows, fewer).
static size_t attn_sk_bytes(int batch, int block_len, int hq, int hkv, int d, int grid,
                            size_t *off_plan, size_t *off_o, size_t *off_ml) {
  const size_t rows = ((size_t)batch * hkv + 2 * (size_t)grid) * block_len * (hq / hkv);
  *off_plan = attn_job_bytes(grid);
  *off_o = *off_plan + align_up((2 * (size_t)batch + 1) * sizeof(int), 256);
  *off_ml = *off_o + align_up(rows * d * sizeof(float), 256);
  return *off_ml + align_up(rows * 2 * sizeof(float), 256);
}

// Workspace of the fixed KV splits: partial O and (m, l) per (KV head, split,
// query row) of every sequence.
static size_t attn_ws_bytes(int batch, int block_len, int hq, int hkv, int d, int max_ctx,
                            int grid, int *num_splits, int *split_keys, size_t *off_o,
                            size_t *off_ml) {
  choose_split(batch * hkv, block_len, max_ctx, num_splits, split_keys);
  const size_t rows = (size_t)batch * hkv * (*num_splits) * block_len * (hq / hkv);
  *off_o = attn_job_bytes(grid);
  if (*num_splits == 1) {
    *off_ml = *off_o;
    return *off_o;
  }
  *off_ml = *off_o + align_up(rows * d * sizeof(float), 256);
  return *off_ml + align_up(rows * 2 * sizeof(float), 256);
}

// ---------------------------------------------------------------------------
// append: one CTA per sequence, 16-byte vector copies
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) append_kv_kernel(bd_paged_kv kv, int block_len,
                                                        size_t elem_bytes, const char *k_blk,
                                                        const char *v_blk, int32_t *ctx_len,
                                                        const int32_t *n_masked,
                                                        int32_t *dev_status) {
  const int b = blockIdx.x;
  pdl_trigger();
  pdl_wait();
  if (n_masked && n_masked[b] != 0) return;
  const int ctx = ctx_len[b];
  const size_t row_bytes = (size_t)kv.head_dim * elem_bytes;           // one head, one token
  const int vec_per_row = (int)(row_bytes / 16);
  const int total = block_len * kv.num_kv_heads * vec_per_row;
  if (ctx < 0 || ctx + block_len > kv.max_pages_per_seq * kv.page_size) {
    if (threadIdx.x == 0) flag_error(dev_status, BD_ERR_DEVICE_CHECK);
    return;
  }
  for (int e = threadIdx.x; e < total; e += blockDim.x) {
    const int c = e % vec_per_row;
    const int g = (e / vec_per_row) % kv.num_kv_heads;
    const int i = e / (vec_per_row * kv.num_kv_heads);
    const int pos = ctx + i;
    const int pg = kv.page_table[(size_t)b * kv.max_pages_per_seq + pos / kv.page_size];
    if (pg < 0 || pg >= kv.num_pages) {
      flag_error(dev_status, BD_ERR_DEVICE_CHECK);
      continue;
    }
    const size_t src = ((((size_t)b * block_len + i) * kv.num_kv_heads + g) * row_bytes) + c * 16;
    const size_t dst = ((((size_t)pg * kv.num_kv_heads + g) * kv.page_size + pos % kv.page_size) *
                        row_bytes) + c * 16;
    *reinterpret_cast<int4 *>(static_cast<char *>(kv.k_pool) + dst) =
        *reinterpret_cast<const int4 *>(k_blk + src);
    *reinterpret_cast<int4 *>(static_cast<char *>(kv.v_pool) + dst) =
        *reinterpret_cast<const int4 *>(v_blk + src);
  }
  __syncthreads();
  if (threadIdx.x == 0) ctx_len[b] = ctx + block_len;
}

static bool kv_ok(const bd_paged_kv *kv) {
  if (!kv || !kv->k_pool || !kv->v_pool || !kv->page_table) return false;
  if (kv->dtype != BD_F32 && kv->dtype != BD_BF16) return false;
  if (kv->page_size != BD_PAGE_SIZE || kv->num_pages < 1 || kv->num_kv_heads < 1) return false;
  if (kv->max_pages_per_seq < 1) return false;
  if (kv->head_dim != 64 && kv->head_dim != 128) return false;
  if ((reinterpret_cast<uintptr_t>(kv->k_pool) | reinterpret_cast<uintptr_t>(kv->v_pool)) & 15)
    return false;
  return true;
}

}  // namespace bd

using namespace bd;

BD_API size_t bd_block_attention_workspace(int32_t batch, int32_t block_len, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t head_dim,
                                           int32_t max_ctx) {
  if (!attn_shape_ok(batch, block_len, num_q_heads, num_kv_heads, head_dim, max_ctx)) return 0;
  preload_all();
  int ns, sk;
  size_t a, b, c;
  return std::max(attn_ws_bytes(batch, block_len, num_q_heads, num_kv_heads, head_dim, max_ctx,
                                num_sms(), &ns, &sk, &a, &b),
                  attn_sk_bytes(batch, block_len, num_q_heads, num_kv_heads, head_dim, num_sms(),
                                &a, &b, &c));
}

BD_API bd_status bd_block_attention(const bd_paged_kv *kv, const int32_t *ctx_len,
                                    const int32_t *tokens, int32_t batch, int32_t block_len,
                                    int32_t num_q_heads, int32_t max_ctx, const void *q,
                                    const void *k_blk, const void *v_blk, float softmax_scale,
                                    void *out, void *ws, size_t ws_bytes, int32_t *dev_status,
                                    void *stream) {
  if (!kv_ok(kv) || !ctx_len || !q || !k_blk || !v_blk || !out) return BD_ERR_INVALID_ARG;
  if (!attn_shape_ok(batch, block_len, num_q_heads, kv->num_kv_heads, kv->head_dim, max_ctx))
    return BD_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || isinf(softmax_scale)) return BD_ERR_INVALID_ARG;
  if (!preload_all()) return BD_ERR_CUDA;
  AttnParams p{};
  p.dtype = kv->dtype;
  p.batch = batch;
  p.block_len = block_len;
  p.hq = num_q_heads;
  p.hkv = kv->num_kv_heads;
  p.head_dim = kv->head_dim;
  p.num_pages = kv->num_pages;
  p.page_size = kv->page_size;
  p.max_pages = kv->max_pages_per_seq;
  p.max_ctx = max_ctx;
  p.scale = softmax_scale;
  p.q = q;
  p.k_blk = k_blk;
  p.v_blk = v_blk;
  p.k_pool = kv->k_pool;
  p.v_pool = kv->v_pool;
  p.page_table = kv->page_table;
  p.ctx_len = ctx_len;
  p.tokens = tokens;
  p.out = out;
  p.dev_status = dev_status;
  p.grid = num_sms();
  p.seg_heads = 1;
  // Kernel choice, by shape, for bf16: the tcgen05 head-pair kernel at
  // head_dim 128 and 64 query rows per KV head (the SDAR shapes), the
  // mma.sync kernel for other shapes; each in its cluster form on small
  // problems (a few pages per SM in all: one cluster of CTAs per segment, one
  // launch, pieces merged through L2) and in its tile-range
  // form on large ones.  SIMT for fp32.  A test may force one kernel with
  // bd_debug_force_attention_kernel.
  const int forced = g_forced_attention.load(std::memory_order_relaxed);
  const bool small = attn_small(batch, p.hkv, block_len, max_ctx);
  size_t fs_o, fs_ml, off_plan, sk_o, sk_ml;
  const size_t need = std::max(
      attn_ws_bytes(batch, block_len, num_q_heads, p.hkv, p.head_dim, max_ctx, p.grid,
                    &p.num_splits, &p.split_keys, &fs_o, &fs_ml),
      attn_sk_bytes(batch, block_len, num_q_heads, p.hkv, p.head_dim, p.grid, &off_plan, &sk_o,
                    &sk_ml));
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255)) return BD_ERR_WORKSPACE;
  char *w = static_cast<char *>(ws);
  p.jobs = reinterpret_cast<int *>(w);
  p.part_o = reinterpret_cast<float *>(w + fs_o);
  p.part_ml = reinterpret_cast<float *>(w + fs_ml);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // tile-range partials of the mma.sync and head-pair kernels; the cluster
  // forms keep one piece slot per CTA there
  p.sk_o = reinterpret_cast<float *>(w + sk_o);
  p.sk_ml = reinterpret_cast<float *>(w + sk_ml);
  if (forced == BD_ATTN_PAIR_CLUSTER || (forced == BD_ATTN_AUTO && small)) {
    const bd_status s = attention_pair_cluster(p, st);
    if (s != BD_ERR_UNSUPPORTED) return s;
  }
  if (forced == BD_ATTN_CLUSTER || (forced == BD_ATTN_AUTO && small)) {
    const bd_status s = attention_cluster(p, st);
    if (s != BD_ERR_UNSUPPORTED) return s;
  }
  if (forced == BD_ATTN_PAIR || (forced == BD_ATTN_AUTO && !small)) {
    if (attention_pair_supported(p)) return attention_pair(p, st);
  }
  if (small) {
    // fixed splits: the kernel writes its partials where the split combine reads them
    p.plan = nullptr;
    p.sk_o = p.part_o;
    p.sk_ml = p.part_ml;
  } else {
    p.plan = reinterpret_cast<int *>(w + off_plan);
  }
  if (forced != BD_ATTN_SIMT) {
    const bd_status s = attention_tc(p, st);
    if (s != BD_ERR_UNSUPPORTED) return s;
  }
  return attention_simt(p, st);
}

BD_API bd_status bd_append_block_kv(const bd_paged_kv *kv, int32_t batch, int32_t block_len,
                                    const void *k_blk, const void *v_blk, int32_t *ctx_len,
                                    const int32_t *n_masked, int32_t *dev_status, void *stream) {
  if (!kv_ok(kv) || !k_blk || !v_blk || !ctx_len) return BD_ERR_INVALID_ARG;
  if (batch < 1 || block_len < 1 || block_len > 1024) return BD_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k_blk) | reinterpret_cast<uintptr_t>(v_blk)) & 15)
    return BD_ERR_INVALID_ARG;
  if (!preload_all()) return BD_ERR_CUDA;
  const size_t elem = kv->dtype == BD_BF16 ? 2 : 4;
  const cudaError_t e = launch_pdl(append_kv_kernel, dim3(batch), dim3(256), 0,
                                   static_cast<cudaStream_t>(stream), *kv, block_len, elem,
                                   static_cast<const char *>(k_blk),
                                   static_cast<const char *>(v_blk), ctx_len, n_masked,
                                   dev_status);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

BD_API const char *bd_status_string(bd_status s) {
  switch (s) {
    case BD_OK: return "BD_OK";
    case BD_ERR_INVALID_ARG: return "BD_ERR_INVALID_ARG";
    case BD_ERR_UNSUPPORTED: return "BD_ERR_UNSUPPORTED";
    case BD_ERR_CUDA: return "BD_ERR_CUDA";
    case BD_ERR_DEVICE_CHECK: return "BD_ERR_DEVICE_CHECK";
    case BD_ERR_TIMEOUT: return "BD_ERR_TIMEOUT";
    case BD_ERR_WORKSPACE: return "BD_ERR_WORKSPACE";
  }
  return "BD_ERR_UNKNOWN";
}

BD_API int32_t bd_version(void) { return 200; }

BD_API bd_status bd_debug_force_attention_kernel(int32_t which) {
  if (which < BD_ATTN_AUTO || which > BD_ATTN_PAIR_CLUSTER) return BD_ERR_INVALID_ARG;
  g_forced_attention.store(which, std::memory_order_relaxed);
  return BD_OK;
}

BD_API uint64_t bd_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }
