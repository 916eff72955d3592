// Decoder layer stack around the block attention: token embedding, RMSNorm,
// the QKV and output projections and the residual add.
//
// "Rethinking Document OCR as Inverse Rendering via Diffusion Decoding"
// (paper.rainbus.top summary), reproduction paragraph: the diffusion decoder
// is initialised from SDAR-1.7B-Chat-b32.  The pages give no layer internals,
// so the layer computed here is the plainest reading:
//   x0 = E[token] for a confirmed position, e_mask for a masked one
//   per layer: xn = bf16(x / sqrt(mean(x^2) + eps))     (no gain)
//              [q | k | v] = bf16(xn Wqkv^T)
//              a = bf16(block attention of q over the layer's cache + k, v)
//              x = x + a Wo^T
//   optional MLP:  xn = bf16(RMSNorm(x)); [g | u] = xn Wgu^T
//                  x = x + bf16(silu(g) * u) Wdown^T      (SwiGLU, Qwen3 family)
// x is kept in fp32; everything stored between kernels except x is bf16.
//
// Kernels:
//   embed_norm_kernel  one CTA per row: gather the embedding row into fp32 x
//                      and write xn
//   proj_tc_kernel     tcgen05 split-K GEMM: output features are the MMA's M
//                      (tiles of 128 weight rows, A operand), activation rows
//                      are N (<= 256 per pass, B operand), K is split so that
//                      the grid covers the SMs.  Each CTA writes one fp32
//                      partial tile [split][row][feature]; no atomics, so the
//                      result does not depend on scheduling
//   qkv_finish_kernel  sum of the partials -> bf16 q, k, v
//   out_finish_kernel  one CTA per row: x += sum of the partials, then the
//                      next layer's xn
//   swiglu_finish_kernel  (optional MLP, bd_mlp_residual) act = bf16(silu(g) * u)
//                      from the partials of the gate/up projection; the down
//                      projection then goes through proj_tc_kernel and
//                      out_finish_kernel like the output projection
//   append_layers_kernel / ctx_bump_kernel: a finished block's K/V of every
//                      layer into the per-layer caches, then ctx += L' once
// Every mbarrier wait is bounded (1 s); on expiry the kernel records
// BD_ERR_TIMEOUT, waits (bounded) for what it issued, frees TMEM and returns.
#include <math.h>
#include <string.h>

#include <algorithm>

#include "bd_common.cuh"
#include "bd_sm100.cuh"

namespace bd {

using namespace sm100;

namespace {

// ---------------------------------------------------------------------------
// row kernels
// ---------------------------------------------------------------------------
constexpr int kRowThreads = 256;

// Sum of v over the CTA (kRowThreads threads); every thread gets the total.
__device__ __forceinline__ float block_sum(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) t += red[w];
  return t;
}

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16 *dst, float4 v) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t *>(&lo);
  u.y = *reinterpret_cast<uint32_t *>(&hi);
  *reinterpret_cast<uint2 *>(dst) = u;
}

__device__ __forceinline__ float4 load_bf16x4(const __nv_bfloat16 *src) {
  const uint2 u = *reinterpret_cast<const uint2 *>(src);
  const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
  const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
  const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
  return make_float4(a.x, a.y, b.x, b.y);
}

// xn = bf16(x * rsqrt(mean(x^2) + eps)) for the row held in `vals`
// (4 * kMaxVec values per thread, elements f = 4 * (threadIdx.x + i * 256)).
constexpr int kMaxVec = 4;   // hidden <= 4 * 4 * 256 = 4096

// The finishing kernels sum the split-K partials in split order, loading up to
// kSplitGroup of them at once so that the sum costs one memory latency per
// group instead of one per split.
constexpr int kSplitGroup = 8;

__device__ __forceinline__ void add4(float4 &a, const float4 &b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}

// acc += partial[s][off] for s = 0 .. splits - 1 (stride sstride floats), in order.
__device__ __forceinline__ void sum_splits(float4 &acc, const float *partial, size_t off,
                                           size_t sstride, int splits) {
  for (int s0 = 0; s0 < splits; s0 += kSplitGroup) {
    float4 pv[kSplitGroup];
#pragma unroll
    for (int j = 0; j < kSplitGroup; ++j)
      if (s0 + j < splits)
        pv[j] = *reinterpret_cast<const float4 *>(partial + (size_t)(s0 + j) * sstride + off);
#pragma unroll
    for (int j = 0; j < kSplitGroup; ++j)
      if (s0 + j < splits) add4(acc, pv[j]);
  }
}

__device__ __forceinline__ void write_norm(const float4 (&vals)[kMaxVec], int nvec, int hidden,
                                           float eps, __nv_bfloat16 *xn_row, float *red) {
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i)
    if (i < nvec) {
      const int f = 4 * (threadIdx.x + i * kRowThreads);
      if (f < hidden) {
        const float4 v = vals[i];
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
    }
  const float r = rsqrtf(block_sum(ss, red) / (float)hidden + eps);
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i)
    if (i < nvec) {
      const int f = 4 * (threadIdx.x + i * kRowThreads);
      if (f < hidden) {
        const float4 v = vals[i];
        store_bf16x4(xn_row + f, make_float4(v.x * r, v.y * r, v.z * r, v.w * r));
      }
    }
}

__global__ void __launch_bounds__(kRowThreads) embed_norm_kernel(
    const int32_t *tokens, int hidden, int vocab, const __nv_bfloat16 *E,
    const __nv_bfloat16 *e_mask, float eps, float *x, __nv_bfloat16 *xn, int32_t *dev_status) {
  __shared__ float red[kRowThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x;
  const int t = tokens[row];
  const __nv_bfloat16 *src = e_mask;
  if (t != BD_MASK) {
    if (t >= 0 && t < vocab) {
      src = E + (size_t)t * hidden;
    } else if (threadIdx.x == 0) {
      flag_error(dev_status, BD_ERR_DEVICE_CHECK);
    }
  }
  const int nvec = (hidden / 4 + kRowThreads - 1) / kRowThreads;
  float4 vals[kMaxVec];
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const int f = 4 * (threadIdx.x + i * kRowThreads);
    vals[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < nvec && f < hidden) {
      vals[i] = load_bf16x4(src + f);
      *reinterpret_cast<float4 *>(x + (size_t)row * hidden + f) = vals[i];
    }
  }
  write_norm(vals, nvec, hidden, eps, xn + (size_t)row * hidden, red);
}

__global__ void __launch_bounds__(kRowThreads) out_finish_kernel(const float *partial, int splits,
                                                                 int rows, int hidden, float eps,
                                                                 float *x, __nv_bfloat16 *xn) {
  __shared__ float red[kRowThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int row = blockIdx.x;
  const int nvec = (hidden / 4 + kRowThreads - 1) / kRowThreads;
  float4 vals[kMaxVec];
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const int f = 4 * (threadIdx.x + i * kRowThreads);
    vals[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < nvec && f < hidden) vals[i] = *reinterpret_cast<const float4 *>(x + (size_t)row * hidden + f);
  }
  const size_t sstride = (size_t)rows * hidden;
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const int f = 4 * (threadIdx.x + i * kRowThreads);
    if (i < nvec && f < hidden) sum_splits(vals[i], partial, (size_t)row * hidden + f, sstride, splits);
  }
#pragma unroll
  for (int i = 0; i < kMaxVec; ++i) {
    const int f = 4 * (threadIdx.x + i * kRowThreads);
    if (i < nvec && f < hidden) *reinterpret_cast<float4 *>(x + (size_t)row * hidden + f) = vals[i];
  }
  write_norm(vals, nvec, hidden, eps, xn + (size_t)row * hidden, red);
}

// q/k/v = bf16(sum of the split partials); one thread per 4 features.
__global__ void __launch_bounds__(256) qkv_finish_kernel(const float *partial, int splits, int rows,
                                                         int F, int fq, int fk, __nv_bfloat16 *q,
                                                         __nv_bfloat16 *k, __nv_bfloat16 *v) {
  pdl_trigger();
  pdl_wait();
  const size_t e = 4 * ((size_t)blockIdx.x * blockDim.x + threadIdx.x);
  if (e >= (size_t)rows * F) return;
  const int row = (int)(e / F), f = (int)(e % F);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  sum_splits(acc, partial, (size_t)row * F + f, (size_t)rows * F, splits);
  __nv_bfloat16 *dst;
  if (f < fq) dst = q + (size_t)row * fq + f;
  else if (f < fq + fk) dst = k + (size_t)row * fk + (f - fq);
  else dst = v + (size_t)row * fk + (f - fq - fk);
  store_bf16x4(dst, acc);
}

// act = bf16(silu(g) * u) from the split partials of [g | u] (gate rows
// first); one thread per 4 features of the intermediate.
__global__ void __launch_bounds__(256) swiglu_finish_kernel(const float *partial, int splits,
                                                            int rows, int inter,
                                                            __nv_bfloat16 *act) {
  pdl_trigger();
  pdl_wait();
  const size_t e = 4 * ((size_t)blockIdx.x * blockDim.x + threadIdx.x);
  if (e >= (size_t)rows * inter) return;
  const int row = (int)(e / inter), j = (int)(e % inter);
  const size_t F = 2 * (size_t)inter;
  float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
  sum_splits(g, partial, (size_t)row * F + j, (size_t)rows * F, splits);
  sum_splits(u, partial, (size_t)row * F + inter + j, (size_t)rows * F, splits);
  const auto silu = [](float x) { return x / (1.f + __expf(-x)); };
  store_bf16x4(act + (size_t)row * inter + j,
               make_float4(silu(g.x) * u.x, silu(g.y) * u.y, silu(g.z) * u.z, silu(g.w) * u.w));
}

// ---------------------------------------------------------------------------
// split-K projection GEMM on the tensor cores
// ---------------------------------------------------------------------------
constexpr int kPThreads = 192;              // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kPTileF = 128;                // output features per tile (MMA M)
constexpr int kPK = 64;                     // K elements per stage (128 bytes of bf16)
constexpr int kPMaxN = 256;                 // rows per pass (MMA N)
constexpr int kPABytes = kPTileF * 128;     // 16 KB of weights per stage
constexpr int kPMaxStages = 8;
constexpr uint32_t kPTmemCols = 256;
constexpr int kPSmemLimit = 227 * 1024;

struct ProjCtrl {
  uint64_t full[kPMaxStages];
  uint64_t empty[kPMaxStages];
  uint64_t done;
  uint32_t tmem_base;
  volatile int32_t abort;
};

struct ProjArgs {
  int rows, K, F;       // partial[s][r][f] = sum over split s's K range of x[r][k] * w[f][k]
  const int32_t *dev_rows;  // if set: only rows < min(rows, *dev_rows) are computed
  int splits, kper;     // K range of one split (a multiple of kPK)
  int box_rows;         // rows per TMA box of x (the pass width, rounded up to 16)
  int stages, stage_bytes, ctrl_off;
  float *partial;       // [splits][rows][F]
  int32_t *dev_status;
};

__global__ void __launch_bounds__(kPThreads, 1)
    proj_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_x, const ProjArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  ProjCtrl *ctrl = reinterpret_cast<ProjCtrl *>(smem + a.ctrl_off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ft = blockIdx.x, sp = blockIdx.y, pass = blockIdx.z;
  const int r0 = pass * kPMaxN;
  const int KC = a.kper / kPK;
  const int k0 = sp * a.kper;
  const int S = a.stages;
  const uint32_t tx = kPABytes + a.box_rows * 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), 1);
    }
    mbar_init(smem_u32(&ctrl->done), 1);
    ctrl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_x);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctrl->tmem_base), kPTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  pdl_trigger();
  // The weights do not depend on earlier work on the stream: the first stages'
  // weight tiles are requested before the dependency wait (their transaction
  // bytes registered without an arrival, so no stage can complete before its
  // activation tile, requested after the wait, has landed too).
  const int pre = min(S, KC);
  if (warp == 0 && lane == 0) {
    for (int kc = 0; kc < pre; ++kc) {
      const uint32_t bar = smem_u32(&ctrl->full[kc]);
      mbar_expect_tx(bar, kPABytes);
      tma_load_2d(smem_u32(smem + (size_t)kc * a.stage_bytes), &tmap_w, k0 + kc * kPK,
                  ft * kPTileF, bar);
    }
  }
  pdl_wait();   // x (and the row count) are written by the previous kernel on the stream
  const int rows = a.dev_rows ? min(a.rows, max(0, *a.dev_rows)) : a.rows;
  const int n = min(kPMaxN, rows - r0);     // rows of this pass; none: nothing to do
  const int npad = (n + 15) & ~15;

  if (n <= 0) {
    // pass beyond the row count: let the early weight copies land before leaving
    if (warp == 0 && lane == 0) {
      for (int kc = 0; kc < pre; ++kc) {
        mbar_arrive(smem_u32(&ctrl->full[kc]));
        mbar_wait(smem_u32(&ctrl->full[kc]), 0);
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int kc = 0;
      for (; kc < KC; ++kc) {
        const uint32_t s = kc % S, round = kc / S;
        if (ctrl->abort) break;
        if (round > 0 && !mbar_wait(smem_u32(&ctrl->empty[s]), (round - 1) & 1)) {
          ctrl->abort = 1;
          flag_error(a.dev_status, BD_ERR_TIMEOUT);
          break;
        }
        uint8_t *st = smem + (size_t)s * a.stage_bytes;
        const uint32_t bar = smem_u32(&ctrl->full[s]);
        if (kc < pre) {                       // weights already requested
          mbar_arrive_expect_tx(bar, tx - kPABytes);
        } else {
          mbar_arrive_expect_tx(bar, tx);
          tma_load_2d(smem_u32(st), &tmap_w, k0 + kc * kPK, ft * kPTileF, bar);
        }
        tma_load_2d(smem_u32(st + kPABytes), &tmap_x, k0 + kc * kPK, r0, bar);
      }
      if (kc < KC) {   // aborted: wait (bounded) for the copies still in flight
        for (int i = kc; i < pre; ++i) mbar_arrive(smem_u32(&ctrl->full[i]));   // weights only
        const int first = kc > S ? kc - S : 0;
        for (int i = first; i < max(kc, pre); ++i)
          mbar_wait(smem_u32(&ctrl->full[i % S]), (i / S) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kPTileF, npad);
      for (int kc = 0; kc < KC; ++kc) {
        const uint32_t s = kc % S, round = kc / S;
        if (ctrl->abort || !mbar_wait(smem_u32(&ctrl->full[s]), round & 1)) {
          ctrl->abort = 1;
          flag_error(a.dev_status, BD_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t a_base = smem_u32(smem + (size_t)s * a.stage_bytes);
        const uint32_t b_base = a_base + kPABytes;
#pragma unroll
        for (int k = 0; k < kPK / 16; ++k)
          mma_bf16(tmem, sw128_kmajor_desc(a_base + k * 32), sw128_kmajor_desc(b_base + k * 32),
                   idesc, (kc | k) != 0);
        mma_commit(smem_u32(&ctrl->empty[s]));
      }
      // fires once every MMA issued above has completed
      mma_commit(smem_u32(&ctrl->done));
      mbar_wait(smem_u32(&ctrl->done), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                   // TMEM lane quarter of this warp
    int ok = 1;
    if (lane == 0) ok = mbar_wait(smem_u32(&ctrl->done), 0) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) flag_error(a.dev_status, BD_ERR_TIMEOUT);
    if (ok && !ctrl->abort) {
      tc_fence_after();
      const int f = ft * kPTileF + 32 * q + lane;
      const bool fin = f < a.F;               // the last tile may run past F
      float *out = a.partial + (size_t)sp * a.rows * a.F + f;
      for (int c0 = 0; c0 < npad; c0 += 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(tmem + ((uint32_t)(32 * q) << 16) + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int row = r0 + c0 + j;
          if (row < rows && fin) out[(size_t)row * a.F] = __uint_as_float(r[j]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kPTmemCols);
  }
}

bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_in,
              uint32_t box_out) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t strides[1] = {inner * 2};
  const uint32_t box[2] = {box_in, box_out};
  return tma_encode_bf16(m, 2, base, dims, strides, box);
}

void proj_plan(int rows, int K, int F, ProjArgs &a, size_t *smem, bool split_k = true) {
  const int sms = std::max(1, dev_info().sms);
  const int ftiles = (F + kPTileF - 1) / kPTileF;
  const int passes = (rows + kPMaxN - 1) / kPMaxN;
  const int kchunks = K / kPK;
  const int want = split_k ? std::max(1, sms / std::max(1, ftiles * passes)) : 1;
  int splits = 1;
  for (int s = std::min(want, kchunks); s >= 1; --s)
    if (kchunks % s == 0) {
      splits = s;
      break;
    }
  a.rows = rows;
  a.K = K;
  a.F = F;
  a.dev_rows = nullptr;
  a.splits = splits;
  a.kper = K / splits;
  a.box_rows = std::min(kPMaxN, (rows + 15) & ~15);
  a.stage_bytes = (kPABytes + a.box_rows * 128 + 1023) & ~1023;
  const int fixed = (int)sizeof(ProjCtrl) + 1024;
  a.stages = std::max(1, std::min(std::min(kPMaxStages, a.kper / kPK),
                                  (kPSmemLimit - fixed) / a.stage_bytes));
  a.ctrl_off = a.stages * a.stage_bytes;
  *smem = (size_t)a.ctrl_off + sizeof(ProjCtrl) + 1024;
}

bool proj_shape_ok(int rows, int K, int F) {
  return rows >= 1 && rows <= (1 << 20) && K >= kPK && K % kPK == 0 && K <= (1 << 16) &&
         F >= kPTileF && F % kPTileF == 0 && F <= (1 << 16);
}

size_t proj_ws_bytes(int rows, int K, int F) {
  ProjArgs a;
  size_t smem;
  proj_plan(rows, K, F, a, &smem);
  return align_up((size_t)a.splits * rows * F * sizeof(float), 256);
}

// Launch the split-K GEMM into ws (fp32 partials); returns the split count.
bd_status proj_launch(int rows, int K, int F, const void *x, const void *w, void *ws,
                      int32_t *dev_status, cudaStream_t st, int *splits) {
  ProjArgs a;
  size_t smem;
  proj_plan(rows, K, F, a, &smem);
  if (smem > (size_t)kPSmemLimit) return BD_ERR_UNSUPPORTED;
  a.partial = static_cast<float *>(ws);
  a.dev_status = dev_status;
  CUtensorMap mw, mx;
  if (!make_map(&mw, w, K, F, kPK, kPTileF)) return BD_ERR_CUDA;
  if (!make_map(&mx, x, K, rows, kPK, a.box_rows)) return BD_ERR_CUDA;
  const dim3 grid(F / kPTileF, a.splits, (rows + kPMaxN - 1) / kPMaxN);
  const cudaError_t e = launch_pdl(proj_tc_kernel, grid, dim3(kPThreads), smem, st, mw, mx, a);
  count_launches(1);
  *splits = a.splits;
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

}  // namespace

// Logits of the masked rows for truncated sampling: out[r][v] = x[r] . w[v]
// (fp32) for r < *dev_rows (at most rows_max), v < V; one K pass, no split.
bd_status logits_tc(int rows_max, int K, int V, const void *x, const void *w, float *out,
                    const int32_t *dev_rows, int32_t *dev_status, cudaStream_t st) {
  if (rows_max < 1 || K < kPK || K % kPK || V < 1) return BD_ERR_UNSUPPORTED;
  ProjArgs a;
  size_t smem;
  proj_plan(rows_max, K, V, a, &smem, false);
  if (smem > (size_t)kPSmemLimit) return BD_ERR_UNSUPPORTED;
  a.partial = out;
  a.dev_rows = dev_rows;
  a.dev_status = dev_status;
  CUtensorMap mw, mx;
  if (!make_map(&mw, w, K, V, kPK, kPTileF)) return BD_ERR_CUDA;
  if (!make_map(&mx, x, K, rows_max, kPK, a.box_rows)) return BD_ERR_CUDA;
  const dim3 grid((V + kPTileF - 1) / kPTileF, 1, (rows_max + kPMaxN - 1) / kPMaxN);
  const cudaError_t e = launch_pdl(proj_tc_kernel, grid, dim3(kPThreads), smem, st, mw, mx, a);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

namespace {

bool tc_ready() {
  const DevInfo d = dev_info();
  return d.major >= 10 && d.sms > 0 && tma_available();
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// ---------------------------------------------------------------------------
// append of every layer's block K/V
// ---------------------------------------------------------------------------
constexpr int kMaxLayers = 64;

struct LayerPools {
  void *k[kMaxLayers];
  void *v[kMaxLayers];
};

__device__ __forceinline__ bool append_allowed(const int32_t *ctx_len, const int32_t *n_masked,
                                               int b, int block_len, int capacity, int *ctx) {
  if (n_masked && n_masked[b] != 0) return false;
  *ctx = ctx_len[b];
  return *ctx >= 0 && *ctx + block_len <= capacity;
}

// grid (batch, layers): copy layer blockIdx.y's block K/V of sequence blockIdx.x
__global__ void __launch_bounds__(256) append_layers_kernel(
    LayerPools pools, bd_paged_kv geom, int block_len, size_t elem_bytes, const char *k_blk,
    const char *v_blk, size_t layer_stride, const int32_t *ctx_len, const int32_t *n_masked,
    int32_t *dev_status) {
  const int b = blockIdx.x, l = blockIdx.y;
  pdl_trigger();
  pdl_wait();
  int ctx;
  const int capacity = geom.max_pages_per_seq * geom.page_size;
  if (!append_allowed(ctx_len, n_masked, b, block_len, capacity, &ctx)) {
    if (threadIdx.x == 0 && !(n_masked && n_masked[b] != 0))
      flag_error(dev_status, BD_ERR_DEVICE_CHECK);
    return;
  }
  const size_t row_bytes = (size_t)geom.head_dim * elem_bytes;
  const int vec_per_row = (int)(row_bytes / 16);
  const int total = block_len * geom.num_kv_heads * vec_per_row;
  char *kp = static_cast<char *>(pools.k[l]);
  char *vp = static_cast<char *>(pools.v[l]);
  const char *ks = k_blk + (size_t)l * layer_stride;
  const char *vs = v_blk + (size_t)l * layer_stride;
  for (int e = threadIdx.x; e < total; e += blockDim.x) {
    const int c = e % vec_per_row;
    const int g = (e / vec_per_row) % geom.num_kv_heads;
    const int i = e / (vec_per_row * geom.num_kv_heads);
    const int pos = ctx + i;
    const int pg = geom.page_table[(size_t)b * geom.max_pages_per_seq + pos / geom.page_size];
    if (pg < 0 || pg >= geom.num_pages) {
      flag_error(dev_status, BD_ERR_DEVICE_CHECK);
      continue;
    }
    const size_t src = ((((size_t)b * block_len + i) * geom.num_kv_heads + g) * row_bytes) + c * 16;
    const size_t dst = ((((size_t)pg * geom.num_kv_heads + g) * geom.page_size +
                         pos % geom.page_size) * row_bytes) + c * 16;
    *reinterpret_cast<int4 *>(kp + dst) = *reinterpret_cast<const int4 *>(ks + src);
    *reinterpret_cast<int4 *>(vp + dst) = *reinterpret_cast<const int4 *>(vs + src);
  }
}

__global__ void ctx_bump_kernel(int batch, int block_len, int capacity, int32_t *ctx_len,
                                const int32_t *n_masked) {
  pdl_trigger();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  int ctx;
  if (append_allowed(ctx_len, n_masked, b, block_len, capacity, &ctx)) ctx_len[b] = ctx + block_len;
}

bool kv_layer_ok(const bd_paged_kv &kv, const bd_paged_kv &ref) {
  if (!kv.k_pool || !kv.v_pool || !kv.page_table) return false;
  if ((reinterpret_cast<uintptr_t>(kv.k_pool) | reinterpret_cast<uintptr_t>(kv.v_pool)) & 15)
    return false;
  return kv.dtype == ref.dtype && kv.num_pages == ref.num_pages && kv.page_size == ref.page_size &&
         kv.num_kv_heads == ref.num_kv_heads && kv.head_dim == ref.head_dim &&
         kv.max_pages_per_seq == ref.max_pages_per_seq && kv.page_table == ref.page_table;
}

}  // namespace

bool preload_decoder() {
  return preload_kernel(embed_norm_kernel, false) && preload_kernel(out_finish_kernel, false) &&
         preload_kernel(qkv_finish_kernel, false) && preload_kernel(proj_tc_kernel, true) &&
         preload_kernel(append_layers_kernel, false) && preload_kernel(ctx_bump_kernel, false) &&
         preload_kernel(swiglu_finish_kernel, false);
}

}  // namespace bd

using namespace bd;

BD_API bd_status bd_embed_rmsnorm(int32_t rows, int32_t hidden, int32_t vocab,
                                  const int32_t *tokens, const void *embed,
                                  const void *mask_embed, float eps, float *x, void *xn,
                                  int32_t *dev_status, void *stream) {
  if (rows < 1 || rows > (1 << 20) || hidden < 4 || hidden % 4 != 0 ||
      hidden > 4 * kMaxVec * kRowThreads || vocab < 1)
    return BD_ERR_INVALID_ARG;
  if (!tokens || !embed || !mask_embed || !x || !xn || !(eps >= 0.f) || isinf(eps))
    return BD_ERR_INVALID_ARG;
  if (!aligned16(embed) || !aligned16(mask_embed) || !aligned16(x) || !aligned16(xn))
    return BD_ERR_INVALID_ARG;
  if (!preload_all()) return BD_ERR_CUDA;
  const cudaError_t e = launch_pdl(
      embed_norm_kernel, dim3(rows), dim3(kRowThreads), 0, static_cast<cudaStream_t>(stream),
      tokens, (int)hidden, (int)vocab, static_cast<const __nv_bfloat16 *>(embed),
      static_cast<const __nv_bfloat16 *>(mask_embed), eps, x, static_cast<__nv_bfloat16 *>(xn),
      dev_status);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

BD_API size_t bd_qkv_projection_workspace(int32_t rows, int32_t hidden, int32_t num_q_heads,
                                          int32_t num_kv_heads, int32_t head_dim) {
  if (num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1) return 0;
  const int64_t F = (int64_t)(num_q_heads + 2 * num_kv_heads) * head_dim;
  if (F > (1 << 16) || !proj_shape_ok(rows, hidden, (int)F)) return 0;
  preload_all();
  return proj_ws_bytes(rows, hidden, (int)F);
}

BD_API bd_status bd_qkv_projection(int32_t rows, int32_t hidden, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim, const void *xn,
                                   const void *w_qkv, void *q, void *k, void *v, void *ws,
                                   size_t ws_bytes, int32_t *dev_status, void *stream) {
  if (num_q_heads < 1 || num_kv_heads < 1 || head_dim < 4 || head_dim % 4 != 0)
    return BD_ERR_INVALID_ARG;
  const int64_t F = (int64_t)(num_q_heads + 2 * num_kv_heads) * head_dim;
  if (F > (1 << 16) || !proj_shape_ok(rows, hidden, (int)F)) return BD_ERR_INVALID_ARG;
  if (!xn || !w_qkv || !q || !k || !v) return BD_ERR_INVALID_ARG;
  if (!aligned16(xn) || !aligned16(w_qkv) || !aligned16(q) || !aligned16(k) || !aligned16(v))
    return BD_ERR_INVALID_ARG;
  if (!preload_all()) return BD_ERR_CUDA;
  if (!tc_ready()) return BD_ERR_UNSUPPORTED;
  const size_t need = proj_ws_bytes(rows, hidden, (int)F);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255)) return BD_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int splits = 0;
  const bd_status s = proj_launch(rows, hidden, (int)F, xn, w_qkv, ws, dev_status, st, &splits);
  if (s != BD_OK) return s;
  const int fq = num_q_heads * head_dim, fk = num_kv_heads * head_dim;
  const size_t threads = (size_t)rows * F / 4;
  const cudaError_t e = launch_pdl(
      qkv_finish_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, st,
      static_cast<const float *>(ws), splits, (int)rows, (int)F, fq, fk,
      static_cast<__nv_bfloat16 *>(q), static_cast<__nv_bfloat16 *>(k),
      static_cast<__nv_bfloat16 *>(v));
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

BD_API size_t bd_out_projection_workspace(int32_t rows, int32_t in_features, int32_t hidden) {
  if (!proj_shape_ok(rows, in_features, hidden)) return 0;
  preload_all();
  return proj_ws_bytes(rows, in_features, hidden);
}

BD_API bd_status bd_out_projection_residual(int32_t rows, int32_t in_features, int32_t hidden,
                                            const void *attn, const void *w_o, float eps,
                                            float *x, void *xn, void *ws, size_t ws_bytes,
                                            int32_t *dev_status, void *stream) {
  if (!proj_shape_ok(rows, in_features, hidden) || hidden > 4 * kMaxVec * kRowThreads)
    return BD_ERR_INVALID_ARG;
  if (!attn || !w_o || !x || !xn || !(eps >= 0.f) || isinf(eps)) return BD_ERR_INVALID_ARG;
  if (!aligned16(attn) || !aligned16(w_o) || !aligned16(x) || !aligned16(xn))
    return BD_ERR_INVALID_ARG;
  if (!preload_all()) return BD_ERR_CUDA;
  if (!tc_ready()) return BD_ERR_UNSUPPORTED;
  const size_t need = proj_ws_bytes(rows, in_features, hidden);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255)) return BD_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int splits = 0;
  const bd_status s = proj_launch(rows, in_features, hidden, attn, w_o, ws, dev_status, st,
                                  &splits);
  if (s != BD_OK) return s;
  const cudaError_t e = launch_pdl(out_finish_kernel, dim3(rows), dim3(kRowThreads), 0, st,
                                   static_cast<const float *>(ws), splits, (int)rows, (int)hidden,
                                   eps, x, static_cast<__nv_bfloat16 *>(xn));
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

// Workspace of bd_mlp_residual: the activation, then the partials of the
// larger of its two projections (they run one after the other).
static size_t mlp_ws(int rows, int hidden, int inter, size_t *act_bytes) {
  *act_bytes = align_up((size_t)rows * inter * 2, 256);
  return *act_bytes + std::max(proj_ws_bytes(rows, hidden, 2 * inter),
                               proj_ws_bytes(rows, inter, hidden));
}

static bool mlp_shape_ok(int rows, int hidden, int inter) {
  return inter >= 64 && inter % 64 == 0 && inter <= (1 << 15) &&
         proj_shape_ok(rows, hidden, 2 * inter) && proj_shape_ok(rows, inter, hidden) &&
         hidden <= 4 * kMaxVec * kRowThreads;
}

BD_API size_t bd_mlp_workspace(int32_t rows, int32_t hidden, int32_t inter) {
  if (!mlp_shape_ok(rows, hidden, inter)) return 0;
  preload_all();
  size_t act;
  return mlp_ws(rows, hidden, inter, &act);
}

BD_API bd_status bd_mlp_residual(int32_t rows, int32_t hidden, int32_t inter, const void *xn,
                                 const void *w_gate_up, const void *w_down, float eps, float *x,
                                 void *xn_out, void *ws, size_t ws_bytes, int32_t *dev_status,
                                 void *stream) {
  if (!mlp_shape_ok(rows, hidden, inter)) return BD_ERR_INVALID_ARG;
  if (!xn || !w_gate_up || !w_down || !x || !xn_out || !(eps >= 0.f) || isinf(eps))
    return BD_ERR_INVALID_ARG;
  if (!aligned16(xn) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(x) ||
      !aligned16(xn_out))
    return BD_ERR_INVALID_ARG;
  if (!preload_all()) return BD_ERR_CUDA;
  if (!tc_ready()) return BD_ERR_UNSUPPORTED;
  size_t act_bytes;
  const size_t need = mlp_ws(rows, hidden, inter, &act_bytes);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255)) return BD_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  __nv_bfloat16 *act = static_cast<__nv_bfloat16 *>(ws);
  float *part = reinterpret_cast<float *>(static_cast<char *>(ws) + act_bytes);
  int splits = 0;
  bd_status s = proj_launch(rows, hidden, 2 * inter, xn, w_gate_up, part, dev_status, st, &splits);
  if (s != BD_OK) return s;
  const size_t quads = (size_t)rows * inter / 4;
  cudaError_t e = launch_pdl(swiglu_finish_kernel, dim3((unsigned)((quads + 255) / 256)),
                             dim3(256), 0, st, (const float *)part, splits, (int)rows,
                             (int)inter, act);
  count_launches(1);
  if (e != cudaSuccess) return BD_ERR_CUDA;
  s = proj_launch(rows, inter, hidden, act, w_down, part, dev_status, st, &splits);
  if (s != BD_OK) return s;
  e = launch_pdl(out_finish_kernel, dim3(rows), dim3(kRowThreads), 0, st, (const float *)part,
                 splits, (int)rows, (int)hidden, eps, x, static_cast<__nv_bfloat16 *>(xn_out));
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

BD_API bd_status bd_append_block_kv_layers(const bd_paged_kv *kv, int32_t num_layers,
                                           int32_t batch, int32_t block_len, const void *k_blk,
                                           const void *v_blk, int32_t *ctx_len,
                                           const int32_t *n_masked, int32_t *dev_status,
                                           void *stream) {
  if (!kv || num_layers < 1 || num_layers > kMaxLayers) return BD_ERR_INVALID_ARG;
  if (batch < 1 || block_len < 1 || block_len > 1024 || !k_blk || !v_blk || !ctx_len)
    return BD_ERR_INVALID_ARG;
  const bd_paged_kv &g = kv[0];
  if (g.dtype != BD_F32 && g.dtype != BD_BF16) return BD_ERR_INVALID_ARG;
  if (g.page_size != BD_PAGE_SIZE || g.num_pages < 1 || g.num_kv_heads < 1 ||
      g.max_pages_per_seq < 1 || (g.head_dim != 64 && g.head_dim != 128))
    return BD_ERR_INVALID_ARG;
  LayerPools pools;
  memset(&pools, 0, sizeof(pools));
  for (int l = 0; l < num_layers; ++l) {
    if (!kv_layer_ok(kv[l], g)) return BD_ERR_INVALID_ARG;
    pools.k[l] = kv[l].k_pool;
    pools.v[l] = kv[l].v_pool;
  }
  if (!aligned16(k_blk) || !aligned16(v_blk)) return BD_ERR_INVALID_ARG;
  if (!preload_all()) return BD_ERR_CUDA;
  const size_t elem = g.dtype == BD_BF16 ? 2 : 4;
  const size_t layer_stride = (size_t)batch * block_len * g.num_kv_heads * g.head_dim * elem;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_pdl(append_layers_kernel, dim3(batch, num_layers), dim3(256), 0, st,
                             pools, g, (int)block_len, elem, static_cast<const char *>(k_blk),
                             static_cast<const char *>(v_blk), layer_stride,
                             (const int32_t *)ctx_len, n_masked, dev_status);
  count_launches(1);
  if (e != cudaSuccess) return BD_ERR_CUDA;
  e = launch_pdl(ctx_bump_kernel, dim3((batch + 127) / 128), dim3(128), 0, st, (int)batch,
                 (int)block_len, g.max_pages_per_seq * g.page_size, ctx_len, n_masked);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}
