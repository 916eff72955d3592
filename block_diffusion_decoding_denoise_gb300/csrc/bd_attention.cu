// Block attention over a paged KV cache: split-KV online softmax.
//
// "Rethinking Document OCR as Inverse Rendering via Diffusion Decoding"
// (paper.rainbus.top summary), method step 3: a token of the current block
// attends fully to its own block, causally to all earlier blocks and the
// prefix, and never to later blocks.  At decode time the cache holds exactly
// the prefix and the earlier blocks, so the rule becomes "all cached keys plus
// all block keys".
//
// This file holds the generic SIMT path (fp32 or bf16 storage, fp32 math);
// it is the fp32 path of the library.  Grid: (split, kv head, sequence).  A
// CTA owns the R = block_len * (Hq/Hkv) query rows of one KV head and one
// page-aligned slice of the keys; warps own 8 rows each; lanes own one key of
// a 32-key tile for Q.K and 1/32 of head_dim for P.V.  Split partials
// (unnormalised O, running max m, running sum l) are merged by
// attn_combine_kernel.
#include <math.h>

#include <algorithm>

#include "bd_attention.cuh"
#include "bd_common.cuh"

namespace bd {

constexpr int kTileKeys = 32;
constexpr int kRowsPerWarp = 8;

template <typename T, int D>
__global__ void __launch_bounds__(512) attn_splitkv_simt_kernel(AttnParams p) {
  extern __shared__ float smem[];
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int group = p.hq / p.hkv;
  const int R = p.block_len * group;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nthreads = blockDim.x;
  pdl_trigger();
  pdl_wait();

  // skip sequences whose block is fully committed
  if (p.tokens && !block_has_mask(p.tokens + (size_t)b * p.block_len, p.block_len)) return;
  const int ctx = p.ctx_len[b];
  if (ctx < 0 || ctx > p.max_ctx || ctx > p.max_pages * p.page_size) {
    if (split == 0 && g == 0 && threadIdx.x == 0) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
    return;
  }
  const int nkeys = ctx + p.block_len;
  const int kbeg = split * p.split_keys;
  const int kend = min(nkeys, kbeg + p.split_keys);

  float *Qs = smem;                            // [R][D]
  float *Ks = Qs + R * D;                      // [32][D+1]
  float *Vs = Ks + kTileKeys * (D + 1);        // [32][D]
  const T *q = static_cast<const T *>(p.q);
  for (int idx = threadIdx.x; idx < R * D; idx += nthreads) {
    const int r = idx / D, d = idx % D;
    const int i = r / group, h = g * group + r % group;
    Qs[idx] = to_f32(q[(((size_t)b * p.block_len + i) * p.hq + h) * D + d]) * p.scale;
  }

  constexpr int DPL = D / 32;                  // head_dim elements per lane
  float acc[kRowsPerWarp][DPL];
  float mrow[kRowsPerWarp], lrow[kRowsPerWarp];
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    mrow[rr] = -INFINITY;
    lrow[rr] = 0.f;
#pragma unroll
    for (int t = 0; t < DPL; ++t) acc[rr][t] = 0.f;
  }

  const T *kpool = static_cast<const T *>(p.k_pool);
  const T *vpool = static_cast<const T *>(p.v_pool);
  const T *kblk = static_cast<const T *>(p.k_blk);
  const T *vblk = static_cast<const T *>(p.v_blk);

  for (int k0 = kbeg; k0 < kend; k0 += kTileKeys) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kTileKeys * D; idx += nthreads) {
      const int j = idx / D, d = idx % D;
      const int pos = k0 + j;
      float kv = 0.f, vv = 0.f;
      if (pos < kend) {
        if (pos < ctx) {
          const int pg = p.page_table[(size_t)b * p.max_pages + pos / p.page_size];
          if (pg >= 0 && pg < p.num_pages) {
            const size_t off = (((size_t)pg * p.hkv + g) * p.page_size + pos % p.page_size) * D + d;
            kv = to_f32(kpool[off]);
            vv = to_f32(vpool[off]);
          } else if (d == 0) {
            flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
          }
        } else {
          const size_t off = (((size_t)b * p.block_len + (pos - ctx)) * p.hkv + g) * D + d;
          kv = to_f32(kblk[off]);
          vv = to_f32(vblk[off]);
        }
      }
      Ks[j * (D + 1) + d] = kv;
      Vs[j * D + d] = vv;
    }
    __syncthreads();
    const bool valid = (k0 + lane) < kend;
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
      const int r = warp * kRowsPerWarp + rr;
      if (r >= R) break;
      const float *qr = Qs + r * D;
      const float *kr = Ks + lane * (D + 1);
      float s = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) s = fmaf(qr[d], kr[d], s);
      s = valid ? s : -INFINITY;
      float mt = s;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float mnew = fmaxf(mrow[rr], mt);
      const float corr = __expf(mrow[rr] - mnew);   // exp(-inf) = 0 on the first tile
      const float pj = valid ? __expf(s - mnew) : 0.f;
      float ps = pj;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      lrow[rr] = lrow[rr] * corr + ps;
      mrow[rr] = mnew;
#pragma unroll
      for (int t = 0; t < DPL; ++t) acc[rr][t] *= corr;
      for (int j = 0; j < kTileKeys; ++j) {
        const float pjj = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
        for (int t = 0; t < DPL; ++t) acc[rr][t] = fmaf(pjj, Vs[j * D + lane + 32 * t], acc[rr][t]);
      }
    }
  }

  // write: final output when there is one split, else the partial
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int r = warp * kRowsPerWarp + rr;
    if (r >= R) break;
    const int i = r / group, h = g * group + r % group;
    if (p.num_splits == 1) {
      T *out = static_cast<T *>(p.out);
      const float inv = lrow[rr] > 0.f ? 1.f / lrow[rr] : 0.f;
#pragma unroll
      for (int t = 0; t < DPL; ++t)
        out[(((size_t)b * p.block_len + i) * p.hq + h) * D + lane + 32 * t] =
            from_f32<T>(acc[rr][t] * inv);
    } else {
      const size_t prow = (((size_t)b * p.hkv + g) * p.num_splits + split) * R + r;
#pragma unroll
      for (int t = 0; t < DPL; ++t) p.part_o[prow * D + lane + 32 * t] = acc[rr][t];
      if (lane == 0) {
        p.part_ml[prow * 2 + 0] = mrow[rr];
        p.part_ml[prow * 2 + 1] = lrow[rr];
      }
    }
  }
}

// Merge split partials: O = sum_s O_s exp(m_s - m) / sum_s l_s exp(m_s - m).
// One warp per (sequence, KV head, query row); lanes own D/32 output columns.
template <typename T, int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnParams p) {
  constexpr int DPL = D / 32;
  const int group = p.hq / p.hkv;
  const int R = p.block_len * group;
  const int wid = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  if (wid >= p.batch * p.hkv * R) return;
  const int r = wid % R, g = (wid / R) % p.hkv, b = wid / (R * p.hkv);
  if (p.tokens && !block_has_mask(p.tokens + (size_t)b * p.block_len, p.block_len)) return;
  const int ctx = p.ctx_len[b];
  if (ctx < 0 || ctx > p.max_ctx || ctx > p.max_pages * p.page_size) return;
  const int used = (ctx + p.block_len + p.split_keys - 1) / p.split_keys;  // splits with keys
  // partials [segment][split][seg_heads * R rows]; a segment is one KV head, or
  // a pair of them for the head-pair kernel
  const int HS = p.seg_heads > 0 ? p.seg_heads : 1;
  const size_t seg = (size_t)b * (p.hkv / HS) + g / HS;
  const size_t srows = (size_t)HS * R;
  const size_t base = seg * p.num_splits * srows + (size_t)(g % HS) * R + r;
  float m = -INFINITY;
  for (int s = lane; s < used; s += 32) m = fmaxf(m, __ldcg(&p.part_ml[(base + (size_t)s * srows) * 2]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float l = 0.f, acc[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) acc[j] = 0.f;
#pragma unroll 4
  for (int s = 0; s < used; ++s) {
    const size_t pr = base + (size_t)s * srows;
    const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + pr * 2));
    const float w = __expf(ml.x - m);
    l = fmaf(ml.y, w, l);
    const float *src = p.part_o + pr * D + lane * DPL;
#pragma unroll
    for (int j = 0; j < DPL; ++j) acc[j] = fmaf(__ldcg(src + j), w, acc[j]);
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int i = r / group, h = g * group + r % group;
  T *out = static_cast<T *>(p.out) + (((size_t)b * p.block_len + i) * p.hq + h) * D + lane * DPL;
#pragma unroll
  for (int j = 0; j < DPL; ++j) out[j] = from_f32<T>(acc[j] * inv);
}

// The same merge when there are at most 32 partials per row: every load the
// row needs (the block's tokens, its ctx, the partials' (m, l) pairs and O
// rows) is issued before any of them is used, so the merge costs about one
// memory latency instead of one per group of partials.
template <typename T, int D>
__global__ void __launch_bounds__(256) attn_combine32_kernel(AttnParams p) {
  constexpr int DPL = D / 32;
  constexpr int kMax = 32;
  const int group = p.hq / p.hkv;
  const int R = p.block_len * group;
  const int wid = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  if (wid >= p.batch * p.hkv * R) return;
  const int r = wid % R, g = (wid / R) % p.hkv, b = wid / (R * p.hkv);
  const int HS = p.seg_heads > 0 ? p.seg_heads : 1;
  const size_t seg = (size_t)b * (p.hkv / HS) + g / HS;
  const size_t srows = (size_t)HS * R;
  const size_t base = seg * p.num_splits * srows + (size_t)(g % HS) * R + r;
  const int ns = p.num_splits;                // <= kMax (host-checked)
  const int tok = (p.tokens && lane < p.block_len) ? p.tokens[(size_t)b * p.block_len + lane] : 0;
  const int ctx = p.ctx_len[b];
  float2 ml = make_float2(-INFINITY, 0.f);
  if (lane < ns) ml = __ldcg(reinterpret_cast<const float2 *>(p.part_ml + (base + lane * srows) * 2));
  float v[kMax][DPL];
#pragma unroll
  for (int s = 0; s < kMax; ++s) {
    if (s < ns) {
      const float *src = p.part_o + (base + (size_t)s * srows) * D + lane * DPL;
#pragma unroll
      for (int d = 0; d < DPL; ++d) v[s][d] = __ldcg(src + d);
    }
  }
  if (p.tokens && !__any_sync(0xffffffffu, lane < p.block_len && tok == BD_MASK)) return;
  if (ctx < 0 || ctx > p.max_ctx || ctx > p.max_pages * p.page_size) return;
  const int used = min(ns, (ctx + p.block_len + p.split_keys - 1) / p.split_keys);
  float m = lane < used ? ml.x : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float w_l = lane < used ? __expf(ml.x - m) : 0.f;
  float l = lane < used ? ml.y * w_l : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  float acc[DPL];
#pragma unroll
  for (int d = 0; d < DPL; ++d) acc[d] = 0.f;
#pragma unroll
  for (int s = 0; s < kMax; ++s) {
    if (s < used) {
      const float w = __shfl_sync(0xffffffffu, w_l, s);
#pragma unroll
      for (int d = 0; d < DPL; ++d) acc[d] = fmaf(v[s][d], w, acc[d]);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int i = r / group, h = g * group + r % group;
  T *out = static_cast<T *>(p.out) + (((size_t)b * p.block_len + i) * p.hq + h) * D + lane * DPL;
#pragma unroll
  for (int d = 0; d < DPL; ++d) out[d] = from_f32<T>(acc[d] * inv);
}

// Merge the pieces of every segment cut by the tile-range partition of the
// bf16 mma.sync kernel; same arithmetic as attn_combine_kernel, slots
// segment + CTA for the CTAs between those holding the segment's first and
// last tiles (skipping CTAs with an empty range).  A segment inside one CTA
// was written by that CTA directly.
template <typename T, int D>
__global__ void __launch_bounds__(256) attn_combine_sk_kernel(AttnParams p) {
  constexpr int DPL = D / 32;
  const int group = p.hq / p.hkv;
  const int R = p.block_len * group;
  const int wid = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  if (wid >= p.batch * p.hkv * R) return;
  const int r = wid % R, g = (wid / R) % p.hkv, b = wid / (R * p.hkv);
  const int HS = p.seg_heads;                  // KV heads per segment
  const int total = p.plan[2 * p.batch];
  const int tiles = p.plan[2 * b + 1];
  if (tiles <= 0 || total <= 0) return;
  const long long seg0 = (long long)p.plan[2 * b] + (long long)(g / HS) * tiles;
  const int c0 = sk_cta_of(seg0, total, p.grid), c1 = sk_cta_of(seg0 + tiles - 1, total, p.grid);
  if (c0 == c1) return;
  // CTAs c0..c1 hold the segment's pieces, except those whose tile range is
  // empty (when there are more CTAs than tiles); a slot holds HS * R rows
  const size_t seg = (size_t)b * (p.hkv / HS) + g / HS;
  const size_t srows = (size_t)HS * R;
  const size_t rin = (size_t)(g % HS) * R + r;
  auto holds = [&](int c) {
    return ((long long)c * total) / p.grid < ((long long)(c + 1) * total) / p.grid;
  };
  float m = -INFINITY;
  for (int c = c0 + lane; c <= c1; c += 32)
    if (holds(c)) m = fmaxf(m, __ldcg(&p.sk_ml[((seg + c) * srows + rin) * 2]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float l = 0.f, acc[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) acc[j] = 0.f;
  for (int c = c0; c <= c1; ++c) {
    if (!holds(c)) continue;
    const size_t pr = (seg + c) * srows + rin;
    const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.sk_ml + pr * 2));
    const float w = __expf(ml.x - m);
    l = fmaf(ml.y, w, l);
    const float *src = p.sk_o + pr * D + lane * DPL;
#pragma unroll
    for (int j = 0; j < DPL; ++j) acc[j] = fmaf(__ldcg(src + j), w, acc[j]);
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int i = r / group, h = g * group + r % group;
  T *out = static_cast<T *>(p.out) + (((size_t)b * p.block_len + i) * p.hq + h) * D + lane * DPL;
#pragma unroll
  for (int j = 0; j < DPL; ++j) out[j] = from_f32<T>(acc[j] * inv);
}

// attn_combine_sk_kernel with one memory latency for segments cut into at
// most 32 pieces: every piece's (m, l) pair and O row are loaded before any
// is used; a segment with more pieces takes the loop of attn_combine_sk_kernel.
template <typename T, int D>
__global__ void __launch_bounds__(256) attn_combine_sk32_kernel(AttnParams p) {
  constexpr int DPL = D / 32;
  constexpr int kMax = 32;
  const int group = p.hq / p.hkv;
  const int R = p.block_len * group;
  const int wid = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  if (wid >= p.batch * p.hkv * R) return;
  const int r = wid % R, g = (wid / R) % p.hkv, b = wid / (R * p.hkv);
  const int HS = p.seg_heads;
  const int total = p.plan[2 * p.batch];
  const int tiles = p.plan[2 * b + 1];
  const int sbase = p.plan[2 * b];
  if (tiles <= 0 || total <= 0) return;
  const long long seg0 = (long long)sbase + (long long)(g / HS) * tiles;
  const int c0 = sk_cta_of(seg0, total, p.grid), c1 = sk_cta_of(seg0 + tiles - 1, total, p.grid);
  if (c0 == c1) return;
  const size_t seg = (size_t)b * (p.hkv / HS) + g / HS;
  const size_t srows = (size_t)HS * R;
  const size_t rin = (size_t)(g % HS) * R + r;
  auto holds = [&](int c) {
    return ((long long)c * total) / p.grid < ((long long)(c + 1) * total) / p.grid;
  };
  const int i = r / group, h = g * group + r % group;
  T *out = static_cast<T *>(p.out) + (((size_t)b * p.block_len + i) * p.hq + h) * D + lane * DPL;
  if (c1 - c0 + 1 > kMax) {                   // more pieces than lanes: one group at a time
    float m = -INFINITY;
    for (int c = c0 + lane; c <= c1; c += 32)
      if (holds(c)) m = fmaxf(m, __ldcg(&p.sk_ml[((seg + c) * srows + rin) * 2]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f, acc[DPL];
#pragma unroll
    for (int j = 0; j < DPL; ++j) acc[j] = 0.f;
    for (int c = c0; c <= c1; ++c) {
      if (!holds(c)) continue;
      const size_t pr = (seg + c) * srows + rin;
      const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.sk_ml + pr * 2));
      const float w = __expf(ml.x - m);
      l = fmaf(ml.y, w, l);
      const float *src = p.sk_o + pr * D + lane * DPL;
#pragma unroll
      for (int j = 0; j < DPL; ++j) acc[j] = fmaf(__ldcg(src + j), w, acc[j]);
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) out[j] = from_f32<T>(acc[j] * inv);
    return;
  }
  const int n = c1 - c0 + 1;
  const bool mine = lane < n && holds(c0 + lane);
  float2 ml = make_float2(-INFINITY, 0.f);
  if (mine) ml = __ldcg(reinterpret_cast<const float2 *>(p.sk_ml + ((seg + c0 + lane) * srows + rin) * 2));
  float v[kMax][DPL];
#pragma unroll
  for (int s = 0; s < kMax; ++s) {
    if (s < n) {
      const float *src = p.sk_o + ((seg + c0 + s) * srows + rin) * D + lane * DPL;
#pragma unroll
      for (int d = 0; d < DPL; ++d) v[s][d] = __ldcg(src + d);
    }
  }
  float m = mine ? ml.x : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float w_l = mine ? __expf(ml.x - m) : 0.f;
  float l = mine ? ml.y * w_l : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
  float acc[DPL];
#pragma unroll
  for (int d = 0; d < DPL; ++d) acc[d] = 0.f;
#pragma unroll
  for (int s = 0; s < kMax; ++s) {
    if (s < n) {
      const float w = __shfl_sync(0xffffffffu, w_l, s);
      if (w != 0.f) {                         // pieces of CTAs with an empty range weigh 0
#pragma unroll
        for (int d = 0; d < DPL; ++d) acc[d] = fmaf(v[s][d], w, acc[d]);
      }
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int d = 0; d < DPL; ++d) out[d] = from_f32<T>(acc[d] * inv);
}

bd_status attention_combine(const AttnParams &p, cudaStream_t st);

template <typename T, int D>
static bd_status launch_combine_sk(const AttnParams &p, cudaStream_t st) {
  const int R = p.block_len * (p.hq / p.hkv);
  const size_t warps = (size_t)p.batch * p.hkv * R;
  const int blocks = (int)((warps + 7) / 8);
  // the one-latency merge holds 32 partial rows per lane (about 150
  // registers): it wins while the rows fit in one wave of CTAs and latency
  // decides; with more rows the leaner loop keeps more warps per SM busy
  const bool one_wave = blocks <= std::max(1, dev_info().sms);
  const cudaError_t e =
      one_wave ? launch_pdl(attn_combine_sk32_kernel<T, D>, dim3(blocks), dim3(256), 0, st, p)
               : launch_pdl(attn_combine_sk_kernel<T, D>, dim3(blocks), dim3(256), 0, st, p);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

bd_status attention_combine_sk(const AttnParams &p, cudaStream_t st) {
  return p.head_dim == 64 ? launch_combine_sk<__nv_bfloat16, 64>(p, st)
                          : launch_combine_sk<__nv_bfloat16, 128>(p, st);
}

template <typename T, int D>
static bd_status launch_simt(const AttnParams &p, cudaStream_t st) {
  const int R = p.block_len * (p.hq / p.hkv);
  const int warps = (R + kRowsPerWarp - 1) / kRowsPerWarp;
  const size_t smem = sizeof(float) * ((size_t)R * D + kTileKeys * (D + 1) + kTileKeys * D);
  auto kern = attn_splitkv_simt_kernel<T, D>;
  dim3 grid(p.num_splits, p.hkv, p.batch);
  const cudaError_t e = launch_pdl(kern, grid, dim3(warps * 32), smem, st, p);
  count_launches(1);
  if (e != cudaSuccess) return BD_ERR_CUDA;
  return p.num_splits > 1 ? attention_combine(p, st) : BD_OK;
}

template <typename T, int D>
static bd_status launch_combine(const AttnParams &p, cudaStream_t st) {
  const int R = p.block_len * (p.hq / p.hkv);
  const size_t warps = (size_t)p.batch * p.hkv * R;
  const int blocks = (int)((warps + 7) / 8);
  // one-latency merge while it fits (see launch_combine_sk)
  const bool one_wave = blocks <= std::max(1, dev_info().sms);
  const cudaError_t e =
      p.num_splits <= 32 && one_wave
          ? launch_pdl(attn_combine32_kernel<T, D>, dim3(blocks), dim3(256), 0, st, p)
          : launch_pdl(attn_combine_kernel<T, D>, dim3(blocks), dim3(256), 0, st, p);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

bd_status attention_combine(const AttnParams &p, cudaStream_t st) {
  if (p.dtype == BD_F32)
    return p.head_dim == 64 ? launch_combine<float, 64>(p, st) : launch_combine<float, 128>(p, st);
  return p.head_dim == 64 ? launch_combine<__nv_bfloat16, 64>(p, st)
                          : launch_combine<__nv_bfloat16, 128>(p, st);
}

bool preload_attention_simt() {
  return preload_kernel(attn_splitkv_simt_kernel<float, 64>, true) &&
         preload_kernel(attn_splitkv_simt_kernel<float, 128>, true) &&
         preload_kernel(attn_splitkv_simt_kernel<__nv_bfloat16, 64>, true) &&
         preload_kernel(attn_splitkv_simt_kernel<__nv_bfloat16, 128>, true) &&
         preload_kernel(attn_combine_kernel<float, 64>, false) &&
         preload_kernel(attn_combine_kernel<float, 128>, false) &&
         preload_kernel(attn_combine_kernel<__nv_bfloat16, 64>, false) &&
         preload_kernel(attn_combine_kernel<__nv_bfloat16, 128>, false) &&
         preload_kernel(attn_combine32_kernel<float, 64>, false) &&
         preload_kernel(attn_combine32_kernel<float, 128>, false) &&
         preload_kernel(attn_combine32_kernel<__nv_bfloat16, 64>, false) &&
         preload_kernel(attn_combine32_kernel<__nv_bfloat16, 128>, false) &&
         preload_kernel(attn_combine_sk_kernel<__nv_bfloat16, 64>, false) &&
         preload_kernel(attn_combine_sk_kernel<__nv_bfloat16, 128>, false) &&
         preload_kernel(attn_combine_sk32_kernel<__nv_bfloat16, 64>, false) &&
         preload_kernel(attn_combine_sk32_kernel<__nv_bfloat16, 128>, false);
}

bd_status attention_simt(const AttnParams &p, cudaStream_t st) {
  if (p.dtype == BD_F32) {
    if (p.head_dim == 64) return launch_simt<float, 64>(p, st);
    if (p.head_dim == 128) return launch_simt<float, 128>(p, st);
  } else {
    if (p.head_dim == 64) return launch_simt<__nv_bfloat16, 64>(p, st);
    if (p.head_dim == 128) return launch_simt<__nv_bfloat16, 128>(p, st);
  }
  return BD_ERR_UNSUPPORTED;
}

}  // namespace bd
