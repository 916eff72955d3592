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
//   trunc_select_kernel  one cluster of four CTAs per masked row, each on a
//                        quarter of the row, their histograms summed through
//                        the cluster's shared memory after every pass: max and
//                        the top-k digits,
//                        the top-p digits, then the restricted Gumbel-max draw
//                        and the kept mass; writes one sampling state per row
//                        for conf_commit_kernel.  With top-k, once the first
//                        digit is known, every entry at or above the boundary
//                        digit (at most 4096) is copied to shared memory and
//                        the remaining passes run there: two passes over the
//                        row instead of up to seven.  Row passes load eight
//                        values per thread before using them and count into
//                        per-warp private histograms (no contention between
//                        warps), merged after the pass.
#include <math.h>

#include <algorithm>

#include "bd_confidence.cuh"
#include "bd_sm100.cuh"

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

// exp(z - m) with the difference rounded on its own (no contraction into the
// exponent's scaling), so that the row's maximum contributes exactly 1.
__device__ __forceinline__ float rel_exp(float z, float m) { return __expf(__fsub_rn(z, m)); }

__device__ __forceinline__ unsigned long long mass_of(float z, float m) {
  return static_cast<unsigned long long>(static_cast<double>(rel_exp(z, m)) * kMassScale);
}

// Calls f(v, z_v) for this thread's entries of slice `part` of `parts` of the
// row, v ascending: loads are issued in batches of eight (float4 when the row
// is 16-byte aligned) before any of them is used, so each batch costs one
// memory latency.
template <typename F>
__device__ __forceinline__ void for_row(const float *__restrict__ l, int V, float it, int part,
                                        int parts, F &&f) {
  constexpr int kBatch = 8;
  const int t = threadIdx.x;
  if ((V & 3) == 0) {
    const float4 *__restrict__ l4 = reinterpret_cast<const float4 *>(l);
    const int lo4 = (int)((long long)part * (V >> 2) / parts);
    const int V4 = (int)((long long)(part + 1) * (V >> 2) / parts);
    for (int base = lo4 + t; base < V4; base += kSelThreads * kBatch) {
      float4 x[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = base + j * kSelThreads;
        if (i < V4) x[j] = __ldg(l4 + i);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = base + j * kSelThreads;
        if (i < V4) {
          f(4 * i, x[j].x * it);
          f(4 * i + 1, x[j].y * it);
          f(4 * i + 2, x[j].z * it);
          f(4 * i + 3, x[j].w * it);
        }
      }
    }
  } else {
    const int lo = (int)((long long)part * V / parts);
    const int hi = (int)((long long)(part + 1) * V / parts);
    for (int base = lo + t; base < hi; base += kSelThreads * kBatch) {
      float x[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = base + j * kSelThreads;
        if (i < hi) x[j] = __ldg(l + i);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = base + j * kSelThreads;
        if (i < hi) f(i, x[j] * it);
      }
    }
  }
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

// Histograms over a whole row go to private copies in shared memory, one per
// warp for counts and one per pair of warps for masses, so that warps never
// contend for a bin; priv_merge sums the copies into hist.
constexpr int kPrivWords = 32768;           // 128 KB
__device__ __forceinline__ void priv_zero(uint32_t *priv) {
  for (int i = threadIdx.x; i < kPrivWords; i += kSelThreads) priv[i] = 0u;
}

__device__ __forceinline__ void priv_merge(const uint32_t *priv, bool mass,
                                          unsigned long long *hist) {
  for (int b = threadIdx.x; b < kBins; b += kSelThreads) {
    unsigned long long s = 0;
    if (mass) {
      const unsigned long long *p64 = reinterpret_cast<const unsigned long long *>(priv);
      for (int c = 0; c < kSelThreads / 64; ++c) s += p64[c * kBins + b];
    } else {
      for (int c = 0; c < kSelThreads / 32; ++c) s += priv[c * kBins + b];
    }
    hist[b] = s;
  }
}

// Total of an nb-bin histogram (every thread gets it).
__device__ unsigned long long hist_total(const unsigned long long *hist, int nb,
                                         unsigned long long *scan) {
  const int t = threadIdx.x;
  unsigned long long part = 0;
  for (int b = t; b < nb; b += kSelThreads) part += hist[b];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if ((t & 31) == 0) scan[t >> 5] = part;
  __syncthreads();
  unsigned long long total = 0;
  for (int w = 0; w < kSelThreads / 32; ++w) total += scan[w];
  __syncthreads();
  return total;
}

// A row is split over a cluster of kSelCluster CTAs, each taking a slice.
// After every histogram pass each CTA adds up all slices' histograms from
// the cluster's shared memory into its own copy of the row's histogram
// (integer sums, so every CTA gets the same values and takes the same
// digit), and the cluster barriers on both sides keep a CTA from starting the
// next pass, which overwrites its histogram, while others still read it.
constexpr int kSelCluster = 4;

__device__ void cluster_sum_hist(const unsigned long long *hist, unsigned long long *ghist, int nb) {
  sm100::cluster_sync();                      // every slice's histogram is complete
  for (int b = threadIdx.x; b < nb; b += kSelThreads) {
    unsigned long long v[kSelCluster];
    const uint32_t a = sm100::smem_u32(&hist[b]);
#pragma unroll
    for (int q = 0; q < kSelCluster; ++q) v[q] = sm100::ld_cluster_u64(sm100::map_shared(a, q));
    unsigned long long sum = 0;
#pragma unroll
    for (int q = 0; q < kSelCluster; ++q) sum += v[q];
    ghist[b] = sum;
  }
  sm100::cluster_sync();                      // every CTA has read the others' histograms
}

constexpr int kCand = 4096;                 // entries a row's candidate list can hold
constexpr size_t kSelDynSmem = (size_t)kCand * 8 + (size_t)kPrivWords * 4;

__global__ void __launch_bounds__(kSelThreads) trunc_select_kernel(ConfParams p, const float *logits,
                                                                   int top_k, float top_p) {
  __shared__ unsigned long long hist[kBins];    // this slice's histogram
  __shared__ unsigned long long ghist[kBins];   // the row's (all slices of the cluster)
  __shared__ float s_max;
  __shared__ float s_fkb, s_fzb, s_fsum;
  __shared__ int s_fidx;
  __shared__ unsigned long long scan[kSelThreads / 32];
  __shared__ float red[kSelThreads / 32];
  __shared__ int s_digit, s_n;
  __shared__ unsigned long long s_above;
  __shared__ float s_kb[kSelThreads / 32], s_zb[kSelThreads / 32], s_sum[kSelThreads / 32];
  __shared__ int s_idx[kSelThreads / 32];
  extern __shared__ float cand_z[];           // kCand values, kCand entry ids, private hists
  int *cand_v = reinterpret_cast<int *>(cand_z + kCand);
  uint32_t *priv = reinterpret_cast<uint32_t *>(cand_v + kCand);
  uint32_t *priv_c = priv + (threadIdx.x >> 5) * kBins;       // this warp's count copy
  unsigned long long *priv_m =
      reinterpret_cast<unsigned long long *>(priv) + (threadIdx.x >> 6) * kBins;  // mass copy
  const int k = blockIdx.x / kSelCluster, t = threadIdx.x;
  const int part = (int)sm100::cluster_ctarank();
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
  const bool use_k = top_k > 0 && top_k < V;

  // pass over the row: the max, and the counts of the top-k first digit
  if (use_k) priv_zero(priv);
  __syncthreads();
  float m = -INFINITY;
  for_row(l, V, it, part, kSelCluster, [&](int, float z) {
    m = fmaxf(m, z);
    if (use_k) atomicAdd(&priv_c[ordered_key(z) >> kShift[0]], 1u);
  });
  m = block_max(m, red);
  if (t == 0) s_max = m;
  if (use_k) {
    priv_merge(priv, false, hist);
    cluster_sum_hist(hist, ghist, 1 << kWidth[0]);   // also publishes s_max
  } else {
    sm100::cluster_sync();
  }
  {                                           // the row's max over the slices
    float gm = -INFINITY;
    const uint32_t a = sm100::smem_u32(&s_max);
#pragma unroll
    for (int q = 0; q < kSelCluster; ++q) gm = fmaxf(gm, sm100::ld_cluster_f32(sm100::map_shared(a, q)));
    m = gm;
  }

  // Entries are visited either straight from the row or, when top-k leaves
  // few enough candidates (every entry whose first digit is at least the
  // boundary digit), from a list of them in shared memory.
  bool use_cand = false;
  int ncand = 0;
  uint32_t thr = 0;                           // entries with key >= thr are kept
  uint32_t prefix = 0, pmask = 0;
  unsigned long long need = 0;
  int d_next = 0;                             // next top-k digit to resolve
  if (use_k) {
    unsigned long long above;
    const int d0 = find_from_top(ghist, 1 << kWidth[0], (unsigned long long)top_k, above, scan,
                                 &s_digit, &s_above);
    if (d0 < 0) {                             // cannot happen for 0 < k < V
      if (t == 0) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
    } else {
      prefix = (uint32_t)d0 << kShift[0];
      pmask = (uint32_t)((1 << kWidth[0]) - 1) << kShift[0];
      need = (unsigned long long)top_k - above;
      d_next = 1;
      if (above + ghist[d0] <= (unsigned long long)kCand) {
        if (t == 0) s_n = 0;
        __syncthreads();
        for_row(l, V, it, part, kSelCluster, [&](int v, float z) {
          if ((ordered_key(z) >> kShift[0]) >= (uint32_t)d0) {
            const int i = atomicAdd(&s_n, 1);
            if (i < kCand) {
              cand_z[i] = z;
              cand_v[i] = v;
            }
          }
        });
        __syncthreads();
        ncand = min(s_n, kCand);
        use_cand = true;
      }
    }
  }

  // `row`: the entries come from the row (private histograms), else from the
  // short candidate list (atomics straight into hist)
  auto resolve = [&](auto &&visit, bool row) {
    auto begin_hist = [&]() {
      if (row) priv_zero(priv);
      else
        for (int b = t; b < kBins; b += kSelThreads) hist[b] = 0;
      __syncthreads();
    };
    auto end_hist = [&](bool mass, int nb) {
      __syncthreads();
      if (row) priv_merge(priv, mass, hist);
      cluster_sum_hist(hist, ghist, nb);
    };
    // remaining top-k digits
    if (use_k && d_next > 0) {
      for (int d = d_next; d < 3; ++d) {
        const int nb = 1 << kWidth[d], sh = kShift[d];
        begin_hist();
        visit([&](int, float z) {
          const uint32_t key = ordered_key(z);
          if ((key & pmask) == prefix) {
            const uint32_t bin = (key >> sh) & (nb - 1);
            if (row) atomicAdd(&priv_c[bin], 1u);
            else atomicAdd(&hist[bin], 1ull);
          }
        });
        end_hist(false, nb);
        unsigned long long above;
        int dig = find_from_top(ghist, nb, need, above, scan, &s_digit, &s_above);
        if (dig < 0) {
          if (t == 0) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
          dig = 0;
          above = 0;
        }
        prefix |= (uint32_t)dig << sh;
        pmask |= (uint32_t)(nb - 1) << sh;
        need -= above;
      }
      thr = prefix;
    }
    // top-p digits over the entries top-k kept, by integer mass
    if (top_p < 1.f) {
      uint32_t pp = 0, pm = 0;
      unsigned long long pneed = 0;
      for (int d = 0; d < 3; ++d) {
        const int nb = 1 << kWidth[d], sh = kShift[d];
        begin_hist();
        visit([&](int, float z) {
          const uint32_t key = ordered_key(z);
          if (key >= thr && (key & pm) == pp) {
            const uint32_t bin = (key >> sh) & (nb - 1);
            if (row) atomicAdd(&priv_m[bin], mass_of(z, m));
            else atomicAdd(&hist[bin], mass_of(z, m));
          }
        });
        end_hist(true, nb);
        if (d == 0) {                         // total kept mass -> the target
          pneed = (unsigned long long)ceil((double)top_p * (double)hist_total(ghist, nb, scan));
          if (pneed == 0) pneed = 1;
        }
        unsigned long long above;
        int dig = find_from_top(ghist, nb, pneed, above, scan, &s_digit, &s_above);
        if (dig < 0) {                        // rounding put the target past the total
          if (t == 0) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
          dig = 0;
          above = 0;
        }
        pp |= (uint32_t)dig << sh;
        pm |= (uint32_t)(nb - 1) << sh;
        pneed -= above;
      }
      thr = max(thr, pp);
    }
    // restricted Gumbel-max draw and the kept mass
    float kb = -INFINITY, zb = -INFINITY, sum = 0.f;
    int idx = 0x7FFFFFFF;
    visit([&](int v, float z) {
      if (ordered_key(z) < thr) return;
      const float key = z + gumbel_at(v, pos, p.seed, draw);
      if (key > kb || (key == kb && v < idx)) {
        kb = key;
        zb = z;
        idx = v;
      }
      sum += rel_exp(z, m);
    });
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
    if (t == 0) {                             // this slice's draw and kept mass
      float S = 0.f;
      for (int w = 0; w < kSelThreads / 32; ++w) {
        S += s_sum[w];
        if (s_kb[w] > kb || (s_kb[w] == kb && s_idx[w] < idx)) {
          kb = s_kb[w];
          zb = s_zb[w];
          idx = s_idx[w];
        }
      }
      s_fkb = kb;
      s_fzb = zb;
      s_fidx = idx;
      s_fsum = S;
    }
    sm100::cluster_sync();
    if (part == 0 && t == 0) {                // the row's: slices merged in order
      float S = 0.f;
      kb = -INFINITY;
      zb = -INFINITY;
      idx = 0x7FFFFFFF;
      for (int q = 0; q < kSelCluster; ++q) {
        const float qkb = sm100::ld_cluster_f32(sm100::map_shared(sm100::smem_u32(&s_fkb), q));
        const float qzb = sm100::ld_cluster_f32(sm100::map_shared(sm100::smem_u32(&s_fzb), q));
        const int qi = sm100::ld_cluster_s32(sm100::map_shared(sm100::smem_u32(&s_fidx), q));
        S += sm100::ld_cluster_f32(sm100::map_shared(sm100::smem_u32(&s_fsum), q));
        if (qkb > kb || (qkb == kb && qi < idx)) {
          kb = qkb;
          zb = qzb;
          idx = qi;
        }
      }
      SampleState st;
      st.m = m;
      st.s = S;
      st.kb = kb;
      st.zb = zb;
      st.idx = idx < V ? idx : -1;
      p.ws.spartial[k] = st;                  // the only partial of row k
    }
    sm100::cluster_sync();                    // the slices' results stay until read
  };
  if (use_cand)
    resolve([&](auto &&f) {
      for (int i = t; i < ncand; i += kSelThreads) f(cand_v[i], cand_z[i]);
    }, false);
  else
    resolve([&](auto &&f) { for_row(l, V, it, part, kSelCluster, f); }, true);
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
  return preload_kernel(trunc_select_kernel, true) &&
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
  const cudaError_t e =
      launch_pdl_cluster(trunc_select_kernel, dim3(rows_max * kSelCluster), dim3(kSelThreads),
                         kSelDynSmem, st, dim3(kSelCluster, 1, 1), p, (const float *)logits,
                         top_k, top_p);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

}  // namespace bd
