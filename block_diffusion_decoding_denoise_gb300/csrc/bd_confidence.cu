// Vocabulary projection, confidence and threshold commit of one denoise step.
//
// "Rethinking Document OCR as Inverse Rendering via Diffusion Decoding"
// (paper.rainbus.top summary), method step 4 (a token is confirmed once its
// prediction confidence passes T = 0.95, otherwise it is denoised again) and
// step 6 (greedy settings: top-k 0, temperature 1, top-p 1).  Confidence is
// the largest softmax probability, p_max = 1 / sum_v exp(l_v - max l); the
// token is the lowest id attaining max l.  When no masked position reaches T,
// the most confident masked position is confirmed (lowest position on ties).
//
// Pipeline (one stream, no host synchronisation):
//   conf_prep_kernel     compact the still-masked positions into a row list
//   lmhead_*             per (producer, row) online max / sum-exp / argmax of
//                        h . W^T over a slice of the vocabulary; logits stay
//                        on chip (SIMT path here, tcgen05 path in
//                        bd_lmhead_tc.cu)
//   conf_commit_kernel   one warp per sequence: merge the partial states,
//                        p_max, argmax, ballot over p_max >= T, fallback, write
//
// bd_sample_commit runs the same pipeline in sampling mode: each masked
// position draws its token from softmax(l / temperature) by the Gumbel-max
// rule, its confidence is the drawn token's probability, and the commit rule
// is unchanged (the sampling reading of step 6's settings).
#include <math.h>

#include <algorithm>

#include "bd_confidence.cuh"

namespace bd {

// ---------------------------------------------------------------------------
// masked-row compaction (+ optional gather of the masked rows of h into a
// contiguous buffer).  Every CTA scans all positions (a block-wide exclusive
// scan, B*L' <= a few thousand); CTA 0 publishes the row list, and CTA c
// copies the rows whose compact index k satisfies k % gridDim.x == c.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) conf_prep_kernel(const int32_t *tokens, int n,
                                                         ConfWorkspace ws, const char *src,
                                                         int row_bytes) {
  __shared__ int warp_sums[32];
  __shared__ int carry;
  __shared__ int list_n;
  __shared__ int2 list[1024];
  pdl_trigger();
  pdl_wait();
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  for (int base = 0; base < n; base += blockDim.x) {
    if (threadIdx.x == 0) list_n = 0;
    const int pos = base + threadIdx.x;
    const int m = (pos < n && tokens[pos] == BD_MASK) ? 1 : 0;
    const unsigned bal = __ballot_sync(0xffffffffu, m);
    const int before_in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) warp_sums[warp] = __popc(bal);
    __syncthreads();
    int before = carry;
    for (int w = 0; w < warp; ++w) before += warp_sums[w];
    const int k = before + before_in_warp;
    if (blockIdx.x == 0 && pos < n) {
      ws.row_of[pos] = m ? k : -1;
      if (m) ws.rows[k] = pos;
    }
    if (src && m && (k % gridDim.x) == blockIdx.x) list[atomicAdd(&list_n, 1)] = make_int2(k, pos);
    __syncthreads();
    if (src) {  // copy this CTA's rows of the chunk, one warp per row, 16 bytes per lane
      const int vecs = row_bytes / 16;
      for (int e = warp; e < list_n; e += nwarps) {
        const int2 kp = list[e];
        const int4 *from = reinterpret_cast<const int4 *>(src + (size_t)kp.y * row_bytes);
        int4 *to = reinterpret_cast<int4 *>(ws.hc + (size_t)kp.x * row_bytes);
        for (int v = lane; v < vecs; v += 32) to[v] = from[v];
      }
    }
    if (threadIdx.x == 0) {
      int tot = 0;
      for (int w = 0; w < nwarps; ++w) tot += warp_sums[w];
      carry += tot;
    }
    __syncthreads();
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *ws.count = carry;
}

// ---------------------------------------------------------------------------
// SIMT LM head: 64 rows x 64 vocab tiles, 4x4 per thread, fp32 FMA
// ---------------------------------------------------------------------------
constexpr int kSimtRows = 64, kSimtVocab = 64, kSimtK = 16;
constexpr int kSimtChunk = 512;  // vocab entries per CTA (-> one partial per chunk)

__device__ __forceinline__ MaxSumArg shfl_xor_state(const MaxSumArg &a, int o) {
  MaxSumArg b;
  b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
  b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
  b.idx = __shfl_xor_sync(0xffffffffu, a.idx, o);
  return b;
}

__device__ __forceinline__ SampleState shfl_xor_state(const SampleState &a, int o) {
  SampleState b;
  b.m = __shfl_xor_sync(0xffffffffu, a.m, o);
  b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
  b.kb = __shfl_xor_sync(0xffffffffu, a.kb, o);
  b.zb = __shfl_xor_sync(0xffffffffu, a.zb, o);
  b.idx = __shfl_xor_sync(0xffffffffu, a.idx, o);
  return b;
}

__device__ __forceinline__ void set_empty(MaxSumArg &a) { a = MaxSumArg{-INFINITY, 0.f, 0x7fffffff}; }
__device__ __forceinline__ void set_empty(SampleState &a) {
  a = SampleState{-INFINITY, 0.f, -INFINITY, -INFINITY, 0x7fffffff};
}

template <bool kSample> struct ConfState { using type = MaxSumArg; };
template <> struct ConfState<true> { using type = SampleState; };

template <typename T, bool kSample>
__global__ void __launch_bounds__(256) lmhead_simt_kernel(ConfParams p) {
  using St = typename ConfState<kSample>::type;
  __shared__ float As[kSimtK][kSimtRows + 4];
  __shared__ float Bs[kSimtK][kSimtVocab + 4];
  __shared__ St state[kSimtRows];
  __shared__ int spos[kSimtRows];
  pdl_trigger();
  pdl_wait();
  const int count = *p.ws.count;
  const int r0 = blockIdx.y * kSimtRows;
  if (r0 >= count) return;
  uint64_t draw = 0;                       // the step's draw counter (sampling)
  if constexpr (kSample) draw = *p.offset;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int v_lo = blockIdx.x * kSimtChunk;
  const int v_hi = min(p.vocab, v_lo + kSimtChunk);
  const T *h = static_cast<const T *>(p.h);
  const T *w = static_cast<const T *>(p.w);
  const int H = p.hidden;
  if (threadIdx.x < kSimtRows) {
    set_empty(state[threadIdx.x]);
    spos[threadIdx.x] = r0 + threadIdx.x < count ? p.ws.rows[r0 + threadIdx.x] : 0;
  }

  for (int v0 = v_lo; v0 < v_hi; v0 += kSimtVocab) {
    float acc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
    for (int k0 = 0; k0 < H; k0 += kSimtK) {
      __syncthreads();
      for (int e = threadIdx.x; e < kSimtK * kSimtRows; e += blockDim.x) {
        const int rr = e / kSimtK, kk = e % kSimtK;
        const int r = r0 + rr;
        As[kk][rr] = r < count ? to_f32(h[(size_t)p.ws.rows[r] * H + k0 + kk]) : 0.f;
        const int v = v0 + rr;
        Bs[kk][rr] = v < v_hi ? to_f32(w[(size_t)v * H + k0 + kk]) : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int kk = 0; kk < kSimtK; ++kk) {
        float a[4], bv[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          a[t] = As[kk][ty * 4 + t];
          bv[t] = Bs[kk][tx * 4 + t];
        }
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(a[x], bv[y], acc[x][y]);
      }
    }
    // epilogue: reduce each row over this tile's 64 vocab entries
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      St st;
      set_empty(st);
      if constexpr (kSample) {
        const int pos = spos[ty * 4 + x];
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int v = v0 + tx * 4 + y;
          if (v < v_hi) {
            const float z = acc[x][y] * p.inv_temp;
            const float key = z + gumbel_at(v, pos, p.seed, draw);
            st = merge(st, SampleState{z, 1.f, key, z, v});
          }
        }
      } else {
#pragma unroll
        for (int y = 0; y < 4; ++y) {
          const int v = v0 + tx * 4 + y;
          if (v < v_hi && acc[x][y] > st.m) {
            st.m = acc[x][y];
            st.idx = v;
          }
        }
        if (st.idx != 0x7fffffff) {
#pragma unroll
          for (int y = 0; y < 4; ++y) {
            const int v = v0 + tx * 4 + y;
            if (v < v_hi) st.s += __expf(acc[x][y] - st.m);
          }
        }
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) st = merge(st, shfl_xor_state(st, o));
      if (tx == 0) state[ty * 4 + x] = merge(state[ty * 4 + x], st);
    }
  }
  __syncthreads();
  if (threadIdx.x < kSimtRows) {
    const int r = r0 + threadIdx.x;
    St *part;
    if constexpr (kSample) part = p.ws.spartial;
    else part = p.ws.partial;
    if (r < count) part[(size_t)r * gridDim.x + blockIdx.x] = state[threadIdx.x];   // [row][CTA]
  }
}

template <bool kSample> static cudaError_t launch_simt(const ConfParams &p, dim3 grid, cudaStream_t st) {
  return p.dtype == BD_F32
             ? launch_pdl(lmhead_simt_kernel<float, kSample>, grid, dim3(256), 0, st, p)
             : launch_pdl(lmhead_simt_kernel<__nv_bfloat16, kSample>, grid, dim3(256), 0, st, p);
}

bd_status lmhead_simt(const ConfParams &p, cudaStream_t st) {
  const int nrows = p.batch * p.block_len;
  dim3 grid((p.vocab + kSimtChunk - 1) / kSimtChunk, (nrows + kSimtRows - 1) / kSimtRows);
  const cudaError_t e = p.sample ? launch_simt<true>(p, grid, st) : launch_simt<false>(p, grid, st);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// commit: one CTA per sequence; warp i merges the partial states of position
// i (lanes stride over the producers, up to twelve loads in flight per lane
// before any is merged; the merge order is the producers' order), warp 0 then
// takes the decision
// ---------------------------------------------------------------------------
template <bool kSample>
__global__ void __launch_bounds__(1024) conf_commit_kernel(ConfParams p) {
  using St = typename ConfState<kSample>::type;
  // loads in flight per lane: 12 greedy states cover the 304 partials of a
  // two-CTAs-per-SM LM head in one round (1024 threads leave 64 registers a
  // thread, which the larger sampling states fit at 8)
  constexpr int kInFlight = kSample ? 8 : 12;
  __shared__ float s_pm[32];
  __shared__ int s_am[32];
  __shared__ int s_masked[32];
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = p.block_len;
  pdl_trigger();
  pdl_wait();
  // the LM-head kernel has read the draw counter (it completed before this
  // kernel passed the wait); advance it for the next call on the stream
  if constexpr (kSample)
    if (b == 0 && threadIdx.x == 0) *p.offset += 1;
  if (warp < L) {
    const int pos = b * L + warp;
    const int tok = p.tokens[pos];            // both loads issued together
    const int k = p.direct ? pos : p.ws.row_of[pos];
    const size_t stride = (size_t)p.batch * L;
    float pm = -1.f;
    int am = -1;
    const bool masked = tok == BD_MASK;
    if (masked && (k < 0 || (size_t)k >= stride)) {
      if (lane == 0) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
    } else if (masked) {
      St st;
      set_empty(st);
      const St *part;
      if constexpr (kSample) part = p.ws.spartial;
      else part = p.ws.partial;
      const int np = p.ws.num_partials;
      const int64_t rs = p.ws.row_stride ? p.ws.row_stride : np;
      const int64_t cs = p.ws.row_stride ? p.ws.col_stride : 1;
      for (int c0 = 0; c0 < np; c0 += 32 * kInFlight) {
        St v[kInFlight];
#pragma unroll
        for (int j = 0; j < kInFlight; ++j) {
          const int c = c0 + lane + 32 * j;
          // by default a row's partials are contiguous (coalesced)
          if (c < np) v[j] = part[(size_t)k * rs + (size_t)c * cs];
          else set_empty(v[j]);
        }
#pragma unroll
        for (int j = 0; j < kInFlight; ++j) st = merge(st, v[j]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) st = merge(st, shfl_xor_state(st, o));
      if (lane == 0) {
        if constexpr (kSample) finalize_sample_row(p, st, pm, am);
        else finalize_row(p, st, pm, am);
      }
    }
    if (lane == 0) {
      s_pm[warp] = pm;
      s_am[warp] = am;
      s_masked[warp] = masked ? 1 : 0;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  const bool masked = lane < L && s_masked[lane] != 0;
  commit_sequence_warp(p, b, masked, masked ? s_pm[lane] : -1.f, masked ? s_am[lane] : -1);
}

// Vocabulary-parallel LM head: the merged (max, sum-exp, argmax) state of
// every position over this call's vocabulary slice, the argmax shifted by the
// slice's first entry, in position order; positions already committed get
// the empty state.  One warp per position, partial loads as in the commit.
__global__ void __launch_bounds__(1024) conf_records_kernel(ConfParams p, MaxSumArg *records,
                                                            int vocab_offset) {
  constexpr int kInFlight = 12;
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = p.block_len;
  pdl_trigger();
  pdl_wait();
  if (warp >= L) return;
  const int pos = b * L + warp;
  const int tok = p.tokens[pos];
  const int k = p.direct ? pos : p.ws.row_of[pos];
  MaxSumArg st;
  set_empty(st);
  if (tok == BD_MASK) {
    if (k < 0 || k >= p.batch * L) {
      if (lane == 0) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
    } else {
      const int np = p.ws.num_partials;
      for (int c0 = 0; c0 < np; c0 += 32 * kInFlight) {
        MaxSumArg v[kInFlight];
#pragma unroll
        for (int j = 0; j < kInFlight; ++j) {
          const int c = c0 + lane + 32 * j;
          if (c < np) v[j] = p.ws.partial[(size_t)k * np + c];
          else set_empty(v[j]);
        }
#pragma unroll
        for (int j = 0; j < kInFlight; ++j) st = merge(st, v[j]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) st = merge(st, shfl_xor_state(st, o));
      if (st.idx >= 0 && st.idx < p.vocab) st.idx += vocab_offset;
    }
  }
  if (lane == 0) records[pos] = st;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
int conf_num_partials(bd_dtype dtype, int batch, int block_len, int hidden, int vocab,
                      bool sample) {
  ConfParams probe{};
  probe.dtype = dtype;
  probe.batch = batch;
  probe.block_len = block_len;
  probe.hidden = hidden;
  probe.vocab = vocab;
  if (lmhead_tc_supported(probe)) return lmhead_tc_num_partials(vocab, batch * block_len, sample);
  return (vocab + kSimtChunk - 1) / kSimtChunk;
}

bool preload_confidence() {
  return preload_kernel(conf_prep_kernel, false) &&
         preload_kernel(conf_commit_kernel<false>, false) &&
         preload_kernel(conf_records_kernel, false) &&
         preload_kernel(conf_commit_kernel<true>, false) &&
         preload_kernel(lmhead_simt_kernel<float, false>, false) &&
         preload_kernel(lmhead_simt_kernel<__nv_bfloat16, false>, false) &&
         preload_kernel(lmhead_simt_kernel<float, true>, false) &&
         preload_kernel(lmhead_simt_kernel<__nv_bfloat16, true>, false);
}

static size_t carve(const ConfParams &p, char *base, ConfWorkspace *ws) {
  const size_t n = (size_t)p.batch * p.block_len;
  const int np = conf_num_partials(p.dtype, p.batch, p.block_len, p.hidden, p.vocab, p.sample != 0);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char *ptr = base ? base + off : nullptr;
    off = align_up(off + bytes, 256);
    return ptr;
  };
  char *rows = take(n * 4), *row_of = take(n * 4), *count = take(4);
  char *part = take((size_t)np * n * (p.sample ? sizeof(SampleState) : sizeof(MaxSumArg)));
  char *hc = p.dtype == BD_BF16 ? take(n * (size_t)p.hidden * 2) : nullptr;
  if (ws) {
    ws->rows = reinterpret_cast<int32_t *>(rows);
    ws->row_of = reinterpret_cast<int32_t *>(row_of);
    ws->count = reinterpret_cast<int32_t *>(count);
    ws->partial = reinterpret_cast<MaxSumArg *>(part);
    ws->spartial = reinterpret_cast<SampleState *>(part);
    ws->num_partials = np;
    ws->hc = hc;
  }
  return off;
}

static bool conf_args_ok(bd_dtype dtype, int32_t batch, int32_t block_len, int32_t hidden,
                         int32_t vocab) {
  if (dtype != BD_F32 && dtype != BD_BF16) return false;
  if (batch < 1 || block_len < 1 || block_len > 32 || hidden < 1 || vocab < 1) return false;
  if (dtype == BD_BF16 && hidden % 64 != 0) return false;
  if (dtype == BD_F32 && hidden % 16 != 0) return false;
  if ((int64_t)batch * block_len > (1 << 20)) return false;
  return true;
}

static size_t conf_workspace(bd_dtype dtype, int32_t batch, int32_t block_len, int32_t hidden,
                             int32_t vocab, bool sample) {
  if (!conf_args_ok(dtype, batch, block_len, hidden, vocab)) return 0;
  preload_all();
  ConfParams p{};
  p.dtype = dtype;
  p.batch = batch;
  p.block_len = block_len;
  p.hidden = hidden;
  p.vocab = vocab;
  p.sample = sample ? 1 : 0;
  return carve(p, nullptr, nullptr);
}

// At most this many positions per call: the LM head reads h in place.
constexpr int kDirectRows = 64;

// Truncation of a sampled call: logits buffer after the carved workspace.
struct TruncArgs {
  int top_k;
  float top_p;
  float *logits;
};

// Shared body of bd_confidence_commit, bd_sample_commit and
// bd_sample_commit_truncated: argument checks, workspace carve, then
// prep -> LM head (or logits + truncated selection) -> commit on one stream.
// `records` (vocabulary-parallel LM head, greedy only): write every
// position's merged state over this vocabulary slice instead of committing.
static bd_status conf_run(ConfParams &p, const void *hidden_states, const void *lm_head,
                          void *ws, size_t ws_bytes, void *stream,
                          const TruncArgs *trunc_in = nullptr, MaxSumArg *records = nullptr,
                          int vocab_offset = 0) {
  if (!conf_args_ok(p.dtype, p.batch, p.block_len, p.hidden, p.vocab)) return BD_ERR_INVALID_ARG;
  if (!hidden_states || !lm_head || !p.tokens ||
      (!records && (!p.p_max || !p.argmax || !p.n_committed || !p.n_masked)))
    return BD_ERR_INVALID_ARG;
  if (!preload_all()) return BD_ERR_CUDA;
  if (isnan(p.threshold)) return BD_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(hidden_states) | reinterpret_cast<uintptr_t>(lm_head)) & 15)
    return BD_ERR_INVALID_ARG;
  p.h = hidden_states;
  p.w = lm_head;
  const size_t carved = carve(p, nullptr, nullptr);
  const size_t need =
      carved + (trunc_in ? align_up((size_t)p.batch * p.block_len * p.vocab * 4, 256) : 0);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255)) return BD_ERR_WORKSPACE;
  carve(p, static_cast<char *>(ws), &p.ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TruncArgs tr{};
  const TruncArgs *trunc = nullptr;
  if (trunc_in) {
    tr = *trunc_in;
    tr.logits = reinterpret_cast<float *>(static_cast<char *>(ws) + carved);
    trunc = &tr;
  }

  // the tensor-core paths read the masked rows from a contiguous copy, except
  // with few positions (at most kDirectRows), where the LM head reads all rows
  // in place: at that width it is bound by the W stream either way, and the
  // compaction kernel and its launch drop out of the step
  const bool tc = trunc ? p.dtype == BD_BF16 : lmhead_tc_supported(p);
  const int nrows = p.batch * p.block_len;
  p.direct = (!trunc && tc && nrows <= kDirectRows) ? 1 : 0;
  cudaError_t e;
  if (!p.direct) {
    const int prep_ctas =
        tc ? std::max(1, std::min(std::max(dev_info().sms, 1), (nrows + 7) / 8)) : 1;
    const int32_t *tok_in = p.tokens;
    const char *src = tc ? static_cast<const char *>(hidden_states) : nullptr;
    e = launch_pdl(conf_prep_kernel, dim3(prep_ctas), dim3(1024), 0, st, tok_in, nrows, p.ws, src,
                   p.hidden * 2);
    count_launches(1);
    if (e != cudaSuccess) return BD_ERR_CUDA;
  }
  bd_status s;
  if (trunc) {
    s = trunc_logits_and_select(p, trunc->logits, trunc->top_k, trunc->top_p, st);
    p.ws.num_partials = 1;                    // one sampling state per row
  } else {
    s = tc ? lmhead_tc(p, st) : lmhead_simt(p, st);
  }
  if (s != BD_OK) return s;
  if (records) {
    e = launch_pdl(conf_records_kernel, dim3(p.batch), dim3(32 * p.block_len), 0, st, p, records,
                   vocab_offset);
    count_launches(1);
    return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
  }
  e = p.sample ? launch_pdl(conf_commit_kernel<true>, dim3(p.batch), dim3(32 * p.block_len), 0,
                            st, p)
               : launch_pdl(conf_commit_kernel<false>, dim3(p.batch), dim3(32 * p.block_len), 0,
                            st, p);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

}  // namespace bd

using namespace bd;

BD_API size_t bd_confidence_commit_workspace(bd_dtype dtype, int32_t batch, int32_t block_len,
                                             int32_t hidden, int32_t vocab) {
  return conf_workspace(dtype, batch, block_len, hidden, vocab, false);
}

BD_API bd_status bd_confidence_commit(bd_dtype dtype, int32_t batch, int32_t block_len,
                                      int32_t hidden, int32_t vocab, const void *hidden_states,
                                      const void *lm_head, float threshold, int32_t *tokens,
                                      float *p_max, int32_t *argmax, int32_t *n_committed,
                                      int32_t *n_masked, void *ws, size_t ws_bytes,
                                      int32_t *dev_status, void *stream) {
  ConfParams p{};
  p.dtype = dtype;
  p.batch = batch;
  p.block_len = block_len;
  p.hidden = hidden;
  p.vocab = vocab;
  p.threshold = threshold;
  p.tokens = tokens;
  p.p_max = p_max;
  p.argmax = argmax;
  p.n_committed = n_committed;
  p.n_masked = n_masked;
  p.dev_status = dev_status;
  return conf_run(p, hidden_states, lm_head, ws, ws_bytes, stream);
}

BD_API bd_status bd_confidence_commit_regions(bd_dtype dtype, int32_t batch, int32_t block_len,
                                              int32_t hidden, int32_t vocab,
                                              const void *hidden_states, const void *lm_head,
                                              const float *thresholds, int32_t *tokens,
                                              float *p_max, int32_t *argmax,
                                              int32_t *n_committed, int32_t *n_masked, void *ws,
                                              size_t ws_bytes, int32_t *dev_status,
                                              void *stream) {
  if (!thresholds || (reinterpret_cast<uintptr_t>(thresholds) & 3)) return BD_ERR_INVALID_ARG;
  ConfParams p{};
  p.dtype = dtype;
  p.batch = batch;
  p.block_len = block_len;
  p.hidden = hidden;
  p.vocab = vocab;
  p.threshold = 0.f;
  p.thresholds = thresholds;
  p.tokens = tokens;
  p.p_max = p_max;
  p.argmax = argmax;
  p.n_committed = n_committed;
  p.n_masked = n_masked;
  p.dev_status = dev_status;
  return conf_run(p, hidden_states, lm_head, ws, ws_bytes, stream);
}

BD_API size_t bd_sample_commit_truncated_workspace(bd_dtype dtype, int32_t batch,
                                                   int32_t block_len, int32_t hidden,
                                                   int32_t vocab) {
  const size_t base = conf_workspace(dtype, batch, block_len, hidden, vocab, true);
  return base ? base + align_up((size_t)batch * block_len * vocab * 4, 256) : 0;
}

BD_API bd_status bd_sample_commit_truncated(
    bd_dtype dtype, int32_t batch, int32_t block_len, int32_t hidden, int32_t vocab,
    const void *hidden_states, const void *lm_head, float threshold, float temperature,
    int32_t top_k, float top_p, uint64_t seed, uint64_t *offset, int32_t *tokens, float *p_sel,
    int32_t *sampled, int32_t *n_committed, int32_t *n_masked, void *ws, size_t ws_bytes,
    int32_t *dev_status, void *stream) {
  if (!(temperature >= 1e-6f) || !(temperature <= 1e6f)) return BD_ERR_INVALID_ARG;
  if (!offset || (reinterpret_cast<uintptr_t>(offset) & 7)) return BD_ERR_INVALID_ARG;
  if (top_k < 0 || !(top_p > 0.f) || !(top_p <= 1.f)) return BD_ERR_INVALID_ARG;
  ConfParams p{};
  p.dtype = dtype;
  p.batch = batch;
  p.block_len = block_len;
  p.hidden = hidden;
  p.vocab = vocab;
  p.threshold = threshold;
  p.tokens = tokens;
  p.p_max = p_sel;
  p.argmax = sampled;
  p.n_committed = n_committed;
  p.n_masked = n_masked;
  p.dev_status = dev_status;
  p.sample = 1;
  p.inv_temp = 1.0f / temperature;
  p.seed = seed;
  p.offset = offset;
  if ((top_k == 0 || top_k >= vocab) && top_p == 1.f)   // nothing truncated: the fused path
    return conf_run(p, hidden_states, lm_head, ws, ws_bytes, stream);
  if (vocab > 65535 * 256) return BD_ERR_UNSUPPORTED;
  TruncArgs tr{top_k, top_p, nullptr};
  return conf_run(p, hidden_states, lm_head, ws, ws_bytes, stream, &tr);
}

BD_API size_t bd_sample_commit_workspace(bd_dtype dtype, int32_t batch, int32_t block_len,
                                         int32_t hidden, int32_t vocab) {
  return conf_workspace(dtype, batch, block_len, hidden, vocab, true);
}

BD_API bd_status bd_sample_commit(bd_dtype dtype, int32_t batch, int32_t block_len,
                                  int32_t hidden, int32_t vocab, const void *hidden_states,
                                  const void *lm_head, float threshold, float temperature,
                                  uint64_t seed, uint64_t *offset, int32_t *tokens, float *p_sel,
                                  int32_t *sampled, int32_t *n_committed, int32_t *n_masked,
                                  void *ws, size_t ws_bytes, int32_t *dev_status, void *stream) {
  if (!(temperature >= 1e-6f) || !(temperature <= 1e6f)) return BD_ERR_INVALID_ARG;
  if (!offset || (reinterpret_cast<uintptr_t>(offset) & 7)) return BD_ERR_INVALID_ARG;
  ConfParams p{};
  p.dtype = dtype;
  p.batch = batch;
  p.block_len = block_len;
  p.hidden = hidden;
  p.vocab = vocab;
  p.threshold = threshold;
  p.tokens = tokens;
  p.p_max = p_sel;
  p.argmax = sampled;
  p.n_committed = n_committed;
  p.n_masked = n_masked;
  p.dev_status = dev_status;
  p.sample = 1;
  p.inv_temp = 1.0f / temperature;
  p.seed = seed;
  p.offset = offset;
  return conf_run(p, hidden_states, lm_head, ws, ws_bytes, stream);
}

// ---------------------------------------------------------------------------
// vocabulary-parallel LM head (one vocabulary slice per GPU)
// ---------------------------------------------------------------------------
static_assert(sizeof(bd_conf_record) == sizeof(MaxSumArg), "record layout");

BD_API size_t bd_confidence_shard_workspace(bd_dtype dtype, int32_t batch, int32_t block_len,
                                            int32_t hidden, int32_t vocab_shard) {
  if (dtype != BD_BF16) return 0;
  return conf_workspace(dtype, batch, block_len, hidden, vocab_shard, false);
}

BD_API bd_status bd_confidence_shard(bd_dtype dtype, int32_t batch, int32_t block_len,
                                     int32_t hidden, int32_t vocab_shard, int32_t vocab_offset,
                                     const void *hidden_states, const void *lm_head_shard,
                                     const int32_t *tokens, bd_conf_record *records, void *ws,
                                     size_t ws_bytes, int32_t *dev_status, void *stream) {
  if (dtype != BD_BF16 || !records || vocab_offset < 0 ||
      (int64_t)vocab_offset + vocab_shard > (int64_t)1 << 31)
    return BD_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(records) & 3) return BD_ERR_INVALID_ARG;
  ConfParams p{};
  p.dtype = dtype;
  p.batch = batch;
  p.block_len = block_len;
  p.hidden = hidden;
  p.vocab = vocab_shard;
  p.tokens = const_cast<int32_t *>(tokens);
  p.dev_status = dev_status;
  return conf_run(p, hidden_states, lm_head_shard, ws, ws_bytes, stream, nullptr,
                  reinterpret_cast<MaxSumArg *>(records), vocab_offset);
}

BD_API bd_status bd_commit_shards(int32_t batch, int32_t block_len, int32_t vocab,
                                  int32_t num_shards, const bd_conf_record *records,
                                  float threshold, int32_t *tokens, float *p_max, int32_t *argmax,
                                  int32_t *n_committed, int32_t *n_masked, int32_t *dev_status,
                                  void *stream) {
  if (batch < 1 || block_len < 1 || block_len > 32 || vocab < 1 || num_shards < 1 ||
      (int64_t)batch * block_len > (1 << 20))
    return BD_ERR_INVALID_ARG;
  if (!records || !tokens || !p_max || !argmax || !n_committed || !n_masked || isnan(threshold))
    return BD_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(records) & 3) return BD_ERR_INVALID_ARG;
  if (!preload_all()) return BD_ERR_CUDA;
  ConfParams p{};
  p.dtype = BD_BF16;
  p.batch = batch;
  p.block_len = block_len;
  p.vocab = vocab;
  p.threshold = threshold;
  p.tokens = tokens;
  p.p_max = p_max;
  p.argmax = argmax;
  p.n_committed = n_committed;
  p.n_masked = n_masked;
  p.dev_status = dev_status;
  p.direct = 1;                               // records are in position order
  p.ws.partial = const_cast<MaxSumArg *>(reinterpret_cast<const MaxSumArg *>(records));
  p.ws.num_partials = num_shards;
  p.ws.row_stride = 1;                        // [shard][position]
  p.ws.col_stride = (int64_t)batch * block_len;
  const cudaError_t e = launch_pdl(conf_commit_kernel<false>, dim3(batch), dim3(32 * block_len),
                                   0, static_cast<cudaStream_t>(stream), p);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}
