// Top-k / top-p truncated sampling of the masked rows (bd_sample_commit_truncated).
//
// "Rethinking Document OCR as Inverse Rendering via Diffusion Decoding"
// (paper.rainbus.top summary), method step 6 lists the inference settings
// top-k 0, temperature 1.0, top-p 1.0.  Read as sampling with the truncations
// switched on, each masked position keeps the entries of z = l / temperature
// that survive top-k (the k largest, ties at the boundary kept) and then
// top-p on what top-k kept (the smallest run of largest entries whose
// renormalised mass reaches p, ties kept), and draws its token from the
// renormalised kept distribution by the Gumbel-max rule with the same
// counter-based noise as bd_sample_commit.
//
// Both truncations reduce to one value threshold theta per row, found
// exactly by a three-digit radix select (11, 11 and 10 bits) over the
// order-preserving integer image of z:
//   top-k: digit histograms of counts, descending, until k entries are above;
//   top-p: digit histograms of masses w = floor(exp(z - max) * 2^40) (64-bit
//          integers, so the sums do not depend on the order of the atomics),
//          descending, until the running mass reaches ceil(p * total).
// The logits of the masked rows come from the tcgen05 projection kernel
// (bf16) or logits_simt_kernel (fp32) into the workspace: truncation needs
// every row's full distribution, so in this mode, and only in it, the logits
// pass through memory (4 bytes per masked row and vocabulary entry).
//
// Kernels:
//   logits_simt_kernel   one CTA per (masked row, 256 entries): fp32 dot
//                        products against the row of h staged in smem
//   trunc_select_kernel  one CTA per masked row: max and the top-k digits,
//                        the top-p digits, then the restricted Gumbel-max draw
//                        and the kept mass; writes one sampling state per row
//                        for conf_commit_kernel
#include <math.h>

#include <algorithm>

#include "bd_confidence.cuh"

namespace bd {

namespace {

constexpr int kSelThreads = 512;
constexpr int kBins = 2048;                 // 11-bit digits
constexpr double kMassScale = 1099511627776.0;   // 2^40

// Order-preserving map of fp32 to uint32 (larger z, larger key); -0 takes the
// key of +0 so that equal values have equal keys.
__device__ __forceinline__ uint32_t ordered_key(float z) {
  uint32_t u = __float_as_uint(z);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return u == 0x7FFFFFFFu ? 0x80000000u : u;
}

__device__ __forceinline__ unsigned long long mass_of(float z, float m) {
  return static_cast<unsigned long long>(static_cast<double>(__expf(z - m)) * kMassScale);
}

__device__ __forceinline__ float block_max(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = red[0];
  for (int w = 1; w < kSelThreads / 32; ++w) t = fmaxf(t, red[w]);
  return t;
}

// The digit d of an nb-bin histogram such that the bins above d hold less
// than `need` and the bins from d up hold at least `need`; `above` gets the
// sum of the bins above d.  Every thread returns the same values.
__device__ int find_from_top(const unsigned long long *hist, int nb, unsigned long long need,
                             unsigned long long &above, unsigned long long *scan,
                             int *s_digit, unsigned long long *s_above) {
  constexpr int kPer = kBins / kSelThreads;  // bins per thread, walked from the top
  const int t = threadIdx.x;
  unsigned long long local = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = nb - 1 - (t * kPer + j);
    if (b >= 0) local += hist[b];
  }
  // inclusive scan of `local` over the threads (thread order = descending bins)
  const int warp = t >> 5, lane = t & 31;
  unsigned long long inc = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) scan[warp] = inc;
  if (t == 0) {
    *s_digit = -1;
    *s_above = 0;
  }
  __syncthreads();
  unsigned long long base = 0;
  for (int w = 0; w < warp; ++w) base += scan[w];
  const unsigned long long excl = base + inc - local;
  if (excl < need && excl + local >= need) {
    unsigned long long acc = excl;
    for (int j = 0; j < kPer; ++j) {
      const int b = nb - 1 - (t * kPer + j);
      if (b < 0) break;
      if (acc + hist[b] >= need) {
        *s_digit = b;
        *s_above = acc;
        break;
      }
      acc += hist[b];
    }
  }
  __syncthreads();
  const int d = *s_digit;
  above = *s_above;
  __syncthreads();
  return d;
}

__global__ void __launch_bounds__(kSelThreads) trunc_select_kernel(ConfParams p, const float *logits,
                                                                   int top_k, float top_p) {
  __shared__ unsigned long long hist[kBins];
  __shared__ unsigned long long scan[kSelThreads / 32];
  __shared__ float red[kSelThreads / 32];
  __shared__ int s_digit;
  __shared__ unsigned long long s_above;
  __shared__ float s_kb[kSelThreads / 32], s_zb[kSelThreads / 32], s_sum[kSelThreads / 32];
  __shared__ int s_idx[kSelThreads / 32];
  const int k = blockIdx.x, t = threadIdx.x;
  const int V = p.vocab;
  pdl_trigger();
  pdl_wait();
  if (k >= *p.ws.count) return;
  const int pos = p.ws.rows[k];
  const uint64_t draw = *p.offset;
  const float *l = logits + (size_t)k * V;
  const float it = p.inv_temp;
  constexpr int kShift[3] = {21, 10, 0};
  constexpr int kWidth[3] = {11, 11, 10};

  // max of z and the top-k digits: the first digit pass also finds the max
  float m = -INFINITY;
  uint32_t thr = 0;                           // entries with key >= thr are kept
  const bool use_k = top_k > 0 && top_k < V;
  {
    uint32_t prefix = 0, pmask = 0;
    unsigned long long need = (unsigned long long)(use_k ? top_k : 0);
    const int ndig = use_k ? 3 : 0;
    for (int v = t; v < kBins; v += kSelThreads) hist[v] = 0;
    __syncthreads();
    for (int v = t; v < V; v += kSelThreads) {
      const float z = l[v] * it;
      m = fmaxf(m, z);
      if (use_k) atomicAdd(&hist[ordered_key(z) >> kShift[0]], 1ull);
    }
    m = block_max(m, red);
    for (int d = 0; d < ndig; ++d) {
      const int nb = 1 << kWidth[d];
      if (d > 0) {
        for (int v = t; v < kBins; v += kSelThreads) hist[v] = 0;
        __syncthreads();
        for (int v = t; v < V; v += kSelThreads) {
          const uint32_t key = ordered_key(l[v] * it);
          if ((key & pmask) == prefix) atomicAdd(&hist[(key >> kShift[d]) & (nb - 1)], 1ull);
        }
      }
      __syncthreads();
      unsigned long long above;
      int dig = find_from_top(hist, nb, need, above, scan, &s_digit, &s_above);
      if (dig < 0) {                          // cannot happen for 0 < k < V
        if (t == 0) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
        dig = 0;
        above = 0;
      }
      prefix |= (uint32_t)dig << kShift[d];
      pmask |= (uint32_t)(nb - 1) << kShift[d];
      need -= above;
    }
    if (use_k) thr = prefix;
  }

  // top-p digits over the entries top-k kept, by integer mass
  if (top_p < 1.f) {
    uint32_t prefix = 0, pmask = 0;
    unsigned long long need = 0;
    for (int d = 0; d < 3; ++d) {
      const int nb = 1 << kWidth[d];
      for (int v = t; v < kBins; v += kSelThreads) hist[v] = 0;
      __syncthreads();
      for (int v = t; v < V; v += kSelThreads) {
        const float z = l[v] * it;
        const uint32_t key = ordered_key(z);
        if (key >= thr && (key & pmask) == prefix)
          atomicAdd(&hist[(key >> kShift[d]) & (nb - 1)], mass_of(z, m));
      }
      __syncthreads();
      if (d == 0) {                           // total kept mass -> the target
        unsigned long long part = 0;
        for (int b = t; b < nb; b += kSelThreads) part += hist[b];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if ((t & 31) == 0) scan[t >> 5] = part;
        __syncthreads();
        unsigned long long total = 0;
        for (int w = 0; w < kSelThreads / 32; ++w) total += scan[w];
        __syncthreads();
        need = (unsigned long long)ceil((double)top_p * (double)total);
        if (need == 0) need = 1;
      }
      unsigned long long above;
      int dig = find_from_top(hist, nb, need, above, scan, &s_digit, &s_above);
      if (dig < 0) {                          // rounding put the target past the total
        if (t == 0) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
        dig = 0;
        above = 0;
      }
      prefix |= (uint32_t)dig << kShift[d];
      pmask |= (uint32_t)(nb - 1) << kShift[d];
      need -= above;
    }
    thr = max(thr, prefix);
  }

  // restricted Gumbel-max draw and the kept mass
  float kb = -INFINITY, zb = -INFINITY, sum = 0.f;
  int idx = 0x7FFFFFFF;
  for (int v = t; v < V; v += kSelThreads) {
    const float z = l[v] * it;
    if (ordered_key(z) < thr) continue;
    const float key = z + gumbel_at(v, pos, p.seed, draw);
    if (key > kb) {                           // v ascending per thread: ties keep the lower
      kb = key;
      zb = z;
      idx = v;
    }
    sum += __expf(z - m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float okb = __shfl_xor_sync(0xffffffffu, kb, o);
    const float ozb = __shfl_xor_sync(0xffffffffu, zb, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (okb > kb || (okb == kb && oi < idx)) {
      kb = okb;
      zb = ozb;
      idx = oi;
    }
  }
  const int warp = t >> 5;
  if ((t & 31) == 0) {
    s_kb[warp] = kb;
    s_zb[warp] = zb;
    s_idx[warp] = idx;
    s_sum[warp] = sum;
  }
  __syncthreads();
  if (t == 0) {
    float S = 0.f;
    for (int w = 0; w < kSelThreads / 32; ++w) {
      S += s_sum[w];
      if (s_kb[w] > kb || (s_kb[w] == kb && s_idx[w] < idx)) {
        kb = s_kb[w];
        zb = s_zb[w];
        idx = s_idx[w];
      }
    }
    SampleState st;
    st.m = m;
    st.s = S;
    st.kb = kb;
    st.zb = zb;
    st.idx = idx < V ? idx : -1;
    p.ws.spartial[k] = st;                    // the only partial of row k
  }
}

// out[k][v] = h[row k] . W[v] in fp32, for the masked rows k < count.
template <typename T>
__global__ void __launch_bounds__(256) logits_simt_kernel(ConfParams p, float *out) {
  extern __shared__ float hrow[];
  const int k = blockIdx.x;
  pdl_trigger();
  pdl_wait();
  if (k >= *p.ws.count) return;
  const int H = p.hidden, V = p.vocab;
  const T *h = static_cast<const T *>(p.h) + (size_t)p.ws.rows[k] * H;
  for (int i = threadIdx.x; i < H; i += blockDim.x) hrow[i] = to_f32(h[i]);
  __syncthreads();
  const int v = blockIdx.y * blockDim.x + threadIdx.x;
  if (v >= V) return;
  const T *w = static_cast<const T *>(p.w) + (size_t)v * H;
  float acc = 0.f;
  for (int i = 0; i < H; ++i) acc = fmaf(hrow[i], to_f32(w[i]), acc);
  out[(size_t)k * V + v] = acc;
}

}  // namespace

bool preload_truncated() {
  return preload_kernel(trunc_select_kernel, false) &&
         preload_kernel(logits_simt_kernel<float>, false) &&
         preload_kernel(logits_simt_kernel<__nv_bfloat16>, false);
}

bd_status trunc_logits_and_select(const ConfParams &p, float *logits, int top_k, float top_p,
                                  cudaStream_t st) {
  const int rows_max = p.batch * p.block_len;
  bd_status s = BD_ERR_UNSUPPORTED;
  if (p.dtype == BD_BF16)
    s = logits_tc(rows_max, p.hidden, p.vocab, p.ws.hc, p.w, logits, p.ws.count, p.dev_status,
                  st);
  if (s == BD_ERR_UNSUPPORTED) {
    if (p.hidden > 12288) return BD_ERR_UNSUPPORTED;
    const dim3 grid(rows_max, (p.vocab + 255) / 256);
    const size_t smem = (size_t)p.hidden * sizeof(float);
    const cudaError_t e =
        p.dtype == BD_BF16
            ? launch_pdl(logits_simt_kernel<__nv_bfloat16>, grid, dim3(256), smem, st, p, logits)
            : launch_pdl(logits_simt_kernel<float>, grid, dim3(256), smem, st, p, logits);
    count_launches(1);
    s = e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
  }
  if (s != BD_OK) return s;
  const cudaError_t e = launch_pdl(trunc_select_kernel, dim3(rows_max), dim3(kSelThreads), 0, st,
                                   p, (const float *)logits, top_k, top_p);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

}  // namespace bd
