// Internal parameters of the confidence/commit kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/bd.h"
#include "bd_common.cuh"

namespace bd {

// Workspace layout of bd_confidence_commit (all offsets 256-byte aligned):
//   rows     [B*L] int32   compact list of masked positions (b*L + i)
//   row_of   [B*L] int32   position -> compact row (-1 if not masked)
//   count    [1]   int32   number of masked rows
//   partial  [P][B*L] MaxSumArg   one online-softmax state per producer and row
//   hc       [B*L][H] bf16        masked rows of h, compacted (bf16 only)
struct ConfWorkspace {
  int32_t *rows, *row_of, *count;
  MaxSumArg *partial;
  int num_partials;
  char *hc;
};

struct ConfParams {
  bd_dtype dtype;
  int batch, block_len, hidden, vocab;
  const void *h, *w;
  float threshold;
  int32_t *tokens;
  float *p_max;
  int32_t *argmax, *n_committed, *n_masked;
  int32_t *dev_status;
  ConfWorkspace ws;
};

// Number of partial states the LM-head kernel of `dtype` produces per row.
int conf_num_partials(bd_dtype dtype, int batch, int block_len, int hidden, int vocab);

bd_status lmhead_simt(const ConfParams &p, cudaStream_t st);
bool lmhead_tc_supported(const ConfParams &p);
int lmhead_tc_num_partials(int vocab);
bd_status lmhead_tc(const ConfParams &p, cudaStream_t st);

}  // namespace bd
