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
};

bd_status attention_simt(const AttnParams &p, cudaStream_t st);
bd_status attention_tc(const AttnParams &p, cudaStream_t st);
bd_status attention_combine(const AttnParams &p, cudaStream_t st);
bool attention_tc5_supported(const AttnParams &p);
bd_status attention_tc5(const AttnParams &p, cudaStream_t st);

}  // namespace bd
