// Combine steps of a denoise step split across GPUs.
//
// The path shards by sequence with no exchange at all.  Within one sequence
// two splits need one exchange each:
//   vocabulary-parallel LM head: rank r holds rows [v0_r, v1_r) of W and
//     reduces each masked position's logits over its rows to the online-
//     softmax state (max l, sum exp(l - max), lowest argmax): 12 bytes per
//     position (bd_confidence_shard).  The states of all ranks, gathered,
//     merge into the whole vocabulary's p_max and argmax exactly as the
//     per-CTA states of one GPU do (bd_commit_shards, or the host merge here);
//   KV-split attention: rank r holds a slice of every sequence's keys and
//     produces, per query row, the unnormalised output O_r = sum_j e^(s_j -
//     m_r) v_j with its max m_r and sum l_r; out = sum_r e^(m_r - M) O_r /
//     sum_r e^(m_r - M) l_r with M = max_r m_r.
// ("Rethinking Document OCR as Inverse Rendering via Diffusion Decoding",
// paper.rainbus.top summary, method steps 3-4: the attention of the block
// and the confidence of each masked position are the quantities split.)
// The host merges are plain C++ for callers that gather on the CPU (and for
// tests that run ranks as CPU processes); the device merge is a kernel.
#include <math.h>
#include <stdint.h>

#include <vector>

#include "bd_common.cuh"

namespace bd {
namespace {

// Host copy of the device merge rule (larger max wins, equal maxima keep the
// lower index, the smaller state's sum is rescaled to the larger max).
inline bd_conf_record merge_record(bd_conf_record a, bd_conf_record b) {
  if (b.m > a.m || (b.m == a.m && b.idx < a.idx)) {
    const bd_conf_record t = a;
    a = b;
    b = t;
  }
  if (b.s > 0.f) a.s += b.s * expf(b.m - a.m);
  return a;
}

// One warp per query row, lanes over head_dim (up to 8 values per lane).
template <typename T>
__global__ void __launch_bounds__(256) merge_partials_kernel(int num_shards, int64_t rows,
                                                             int head_dim, const float *m,
                                                             const float *l, const float *o,
                                                             T *out) {
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  if (row >= rows) return;
  float M = -INFINITY;
  for (int s = 0; s < num_shards; ++s) M = fmaxf(M, m[(size_t)s * rows + row]);
  float S = 0.f, acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
  for (int s = 0; s < num_shards; ++s) {
    const float ms = m[(size_t)s * rows + row];
    const float w = ms == -INFINITY ? 0.f : __expf(ms - M);
    S = fmaf(l[(size_t)s * rows + row], w, S);
    const float *src = o + ((size_t)s * rows + row) * head_dim;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int d = lane + 32 * j;
      if (d < head_dim) acc[j] = fmaf(src[d], w, acc[j]);
    }
  }
  const float inv = S > 0.f ? 1.f / S : 0.f;
  T *dst = out + (size_t)row * head_dim;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int d = lane + 32 * j;
    if (d < head_dim) dst[d] = from_f32<T>(acc[j] * inv);
  }
}

}  // namespace

bool preload_parallel() {
  return preload_kernel(merge_partials_kernel<float>, false) &&
         preload_kernel(merge_partials_kernel<__nv_bfloat16>, false);
}

}  // namespace bd

using namespace bd;

BD_API bd_status bd_merge_conf_records_host(int32_t num_shards, int64_t n,
                                            const bd_conf_record *records, bd_conf_record *out) {
  if (num_shards < 1 || n < 0 || (n > 0 && (!records || !out))) return BD_ERR_INVALID_ARG;
  for (int64_t i = 0; i < n; ++i) {
    bd_conf_record acc = records[i];
    for (int32_t s = 1; s < num_shards; ++s) acc = merge_record(acc, records[(size_t)s * n + i]);
    out[i] = acc;
  }
  return BD_OK;
}

BD_API bd_status bd_merge_attention_partials_host(int32_t num_shards, int64_t rows,
                                                  int32_t head_dim, const float *m,
                                                  const float *l, const float *o, float *out) {
  if (num_shards < 1 || rows < 0 || head_dim < 1) return BD_ERR_INVALID_ARG;
  if (rows > 0 && (!m || !l || !o || !out)) return BD_ERR_INVALID_ARG;
  std::vector<float> w((size_t)num_shards);
  for (int64_t r = 0; r < rows; ++r) {
    float M = -INFINITY;
    for (int32_t s = 0; s < num_shards; ++s) M = fmaxf(M, m[(size_t)s * rows + r]);
    float S = 0.f;
    for (int32_t s = 0; s < num_shards; ++s) {
      const float ms = m[(size_t)s * rows + r];
      w[s] = ms == -INFINITY ? 0.f : expf(ms - M);
      S += l[(size_t)s * rows + r] * w[s];
    }
    const float inv = S > 0.f ? 1.f / S : 0.f;
    for (int32_t d = 0; d < head_dim; ++d) {
      float acc = 0.f;
      for (int32_t s = 0; s < num_shards; ++s)
        acc += o[((size_t)s * rows + r) * head_dim + d] * w[s];
      out[(size_t)r * head_dim + d] = acc * inv;
    }
  }
  return BD_OK;
}

BD_API bd_status bd_merge_attention_partials(int32_t num_shards, int64_t rows, int32_t head_dim,
                                             const float *m, const float *l, const float *o,
                                             bd_dtype out_dtype, void *out, void *stream) {
  if (num_shards < 1 || rows < 1 || head_dim < 1 || head_dim > 256 || !m || !l || !o || !out)
    return BD_ERR_INVALID_ARG;
  if (out_dtype != BD_F32 && out_dtype != BD_BF16) return BD_ERR_INVALID_ARG;
  if (!preload_all()) return BD_ERR_CUDA;
  const int64_t blocks = (rows * 32 + 255) / 256;
  if (blocks > INT32_MAX) return BD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e =
      out_dtype == BD_F32
          ? launch_pdl(merge_partials_kernel<float>, dim3((unsigned)blocks), dim3(256), 0, st,
                       (int)num_shards, rows, (int)head_dim, m, l, o, static_cast<float *>(out))
          : launch_pdl(merge_partials_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256), 0,
                       st, (int)num_shards, rows, (int)head_dim, m, l, o,
                       static_cast<__nv_bfloat16 *>(out));
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}
