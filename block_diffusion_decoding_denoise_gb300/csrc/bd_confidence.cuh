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
//   partial  [B*L][P] MaxSumArg   one online-softmax state per row and producer
//                                 (SampleState when sampling); a row's P states
//                                 are contiguous, so the commit reads them coalesced
//   hc       [B*L][H] bf16        masked rows of h, compacted (bf16 only)
struct ConfWorkspace {
  int32_t *rows, *row_of, *count;
  MaxSumArg *partial;
  SampleState *spartial;  // the same memory, typed for the sampling mode
  int num_partials;
  // partial (row k, producer c) at k * row_stride + c * col_stride; 0 means the
  // default [row][producer] layout (row_stride = num_partials, col_stride = 1)
  int64_t row_stride, col_stride;
  char *hc;
};

struct ConfParams {
  bd_dtype dtype;
  int batch, block_len, hidden, vocab;
  const void *h, *w;
  float threshold;
  const float *thresholds;      // per-position thresholds [batch][block_len], or null: threshold
  int32_t *tokens;
  float *p_max;                 // greedy: p_max; sampling: probability of the draw
  int32_t *argmax, *n_committed, *n_masked;   // argmax: greedy argmax or the draw
  int32_t *dev_status;
  // sampling mode (bd_sample_commit): z = l * inv_temp, draw by Gumbel-max;
  // *offset is the device-side draw counter (read by the LM-head kernel,
  // advanced by one by the commit kernel)
  int sample;
  float inv_temp;
  uint64_t seed;
  uint64_t *offset;
  // direct rows (few positions, tensor-core path): the LM head reads all
  // batch * block_len rows of h in place, row k being position k, and no
  // compaction runs; masked or not, every row gets its partial states
  int direct;
  ConfWorkspace ws;
};

// Confidence and token of a row from its merged sampling state: the drawn
// token and its probability exp(z_token - m) / s.
__device__ __forceinline__ void finalize_sample_row(const ConfParams &p, const SampleState &st,
                                                    float &pm, int &am) {
  if (st.idx < 0 || st.idx >= p.vocab || !(st.s >= 1.f) || !(st.zb <= st.m)) {
    flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
    pm = 0.f;
    am = 0;
  } else {
    pm = __expf(st.zb - st.m) / st.s;
    am = st.idx;
  }
}

// p_max and argmax of a row from its merged online-softmax state.
__device__ __forceinline__ void finalize_row(const ConfParams &p, const MaxSumArg &st, float &pm,
                                             int &am) {
  if (st.idx < 0 || st.idx >= p.vocab || !(st.s >= 1.f)) {
    flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
    pm = 0.f;
    am = 0;
  } else {
    pm = 1.f / st.s;
    am = st.idx;
  }
}

// Commit decision of sequence b by one warp; lane i (< block_len) holds
// position i's masked flag and, when masked, its p_max and argmax.
//   S = { masked i : p_max_i >= T_i }; if S is empty and a position is masked,
//   S = { the masked i with the largest p_max, lowest i on ties }.
// T_i is the scalar threshold, or position i's entry of the per-position
// array (region thresholds); a NaN entry never qualifies.
__device__ __forceinline__ void commit_sequence_warp(const ConfParams &p, int b, bool masked,
                                                     float pm, int am) {
  const int lane = threadIdx.x & 31;
  const int L = p.block_len;
  const int pos = b * L + lane;
  const bool in = lane < L;
  const unsigned mmask = __ballot_sync(0xffffffffu, masked);
  const float thr = (p.thresholds && in) ? p.thresholds[pos] : p.threshold;
  unsigned sel = __ballot_sync(0xffffffffu, masked && pm >= thr);
  if (sel == 0u && mmask != 0u) {
    float best = masked ? pm : -INFINITY;
    int who = masked ? lane : 32;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int ow = __shfl_xor_sync(0xffffffffu, who, o);
      if (ob > best || (ob == best && ow < who)) {
        best = ob;
        who = ow;
      }
    }
    sel = 1u << who;
  }
  if (in) {
    p.p_max[pos] = masked ? pm : -1.f;
    p.argmax[pos] = masked ? am : -1;
    if ((sel >> lane) & 1u) p.tokens[pos] = am;
  }
  if (lane == 0) {
    p.n_committed[b] = __popc(sel);
    p.n_masked[b] = __popc(mmask) - __popc(sel);
  }
}

// Number of partial states the LM-head kernel of `dtype` produces per row.
int conf_num_partials(bd_dtype dtype, int batch, int block_len, int hidden, int vocab,
                      bool sample);

bd_status lmhead_simt(const ConfParams &p, cudaStream_t st);
bool lmhead_tc_supported(const ConfParams &p);
int lmhead_tc_num_partials(int vocab, int rows, bool sample);
bd_status lmhead_tc(const ConfParams &p, cudaStream_t st);

// Truncated sampling (bd_sample_commit_truncated): logits of the masked rows
// into `logits` ([batch * block_len][vocab] fp32, rows < *ws.count written),
// then one sampling state per row into ws.spartial[row] (a single partial).
bd_status trunc_logits_and_select(const ConfParams &p, float *logits, int top_k, float top_p,
                                  cudaStream_t st);
// tcgen05 projection of x [rows_max][K] (bf16) against w [V][K] (bf16) into
// out [rows_max][V] fp32 for rows < *dev_rows.
bd_status logits_tc(int rows_max, int K, int V, const void *x, const void *w, float *out,
                    const int32_t *dev_rows, int32_t *dev_status, cudaStream_t st);

}  // namespace bd
