// Internal launch parameters of the block-attention kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bd.h"

namespace bd {

struct AttnParams {
  bd_dtype dtype;
  int batch, block_len, hq, hkv, head_dim;
  int num_pages, page_size, max_pages, max_ctx;
  int num_splits, split_keys;  // KV split: split s covers keys [s*split_keys, (s+1)*split_keys)
  float scale;
  const void *q, *k_blk, *v_blk;
  const void *k_pool, *v_pool;
  const int32_t *page_table, *ctx_len, *tokens;
  void *out;
  float *part_o;   // [batch][hkv][num_splits][R][head_dim]
  float *part_ml;  // [batch][hkv][num_splits][R][2]
  int32_t *dev_status;
  // tile-range partition of the bf16 mma.sync kernel (attn_plan_kernel):
  // tiles of sequence b = its cache pages + 1 block tile; segment (b, g) =
  // the tiles of KV head g; CTA c of `grid` takes the tiles
  // [c T / grid, (c+1) T / grid) of the concatenated segments; a piece of
  // segment s computed by CTA c writes partial slot s + c
  int grid;
  int seg_heads;   // KV heads per segment: 1 (mma.sync kernel) or 2 (head-pair kernel)
  int *plan;       // [2 batch + 1]: base_b, tiles_b per sequence, then T
  int *jobs;       // [grid][8] merge jobs of the head-pair kernel (one per CTA)
  float *sk_o;     // [batch * hkv + grid][R][head_dim]
  float *sk_ml;    // [batch * hkv + grid][R][2]
};

// CTA of the tile-range partition that holds tile t (T tiles over G CTAs).
__host__ __device__ inline int sk_cta_of(long long t, long long T, long long G) {
  return (int)(((t + 1) * G - 1) / T);
}

bd_status attention_simt(const AttnParams &p, cudaStream_t st);
bd_status attention_tc(const AttnParams &p, cudaStream_t st);
bd_status attention_cluster(const AttnParams &p, cudaStream_t st);
bd_status attention_combine(const AttnParams &p, cudaStream_t st);
bd_status attention_combine_sk(const AttnParams &p, cudaStream_t st);
bool attention_pair_supported(const AttnParams &p);
bd_status attention_pair(const AttnParams &p, cudaStream_t st);
bool attention_pair_cluster_supported(const AttnParams &p);
bd_status attention_pair_cluster(const AttnParams &p, cudaStream_t st);
cudaError_t attention_plan_launch(const AttnParams &p, cudaStream_t st);

}  // namespace bd
