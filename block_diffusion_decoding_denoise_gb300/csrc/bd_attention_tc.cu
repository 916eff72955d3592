// bf16 block attention on the tensor cores, K/V pages streamed by TMA.
//
// Same contract and split as attention_simt (see bd_attention.cu): CTA =
// (KV split, KV head g, sequence b) over the R = block_len * (Hq/Hkv) query
// rows that read KV head g, key positions [split * split_keys, ...) of
// [cache | block] ("Rethinking Document OCR as Inverse Rendering via Diffusion
// Decoding", paper.rainbus.top summary, method step 3: bidirectional inside
// the block, causal to every earlier block and the prefix).
//
// The cached keys arrive one 64-token page at a time: a 4-D TMA map over the
// pool [page][Hkv][64][D] fetches the page's [64][D] slab of head g (two
// 64-column boxes when D = 128) with a 128-byte swizzle, so the ldmatrix reads
// below are bank-conflict free.  The block's own keys come through a second
// map over [B][L'][Hkv][D].  Two buffers alternate: the next tile is in
// flight while the current one is consumed.
//
// Math: each warp owns 16 query rows; S = Q K^T and O += P V run on
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) with the online softmax of
// flash attention kept in registers (P never leaves the register file).  The
// cache read is the roofline here (about 64 flop per byte), so the legacy
// warp-level MMA has ample throughput.
#include <math.h>

#include "bd_attention.cuh"
#include "bd_common.cuh"
#include "bd_sm100.cuh"

namespace bd {

using namespace sm100;

namespace {

constexpr int kPageRows = 64;
constexpr int kHalfBytes = kPageRows * 128;   // one 64-column half of a 64-row tile

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *m, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Byte offset of (row, 16-byte chunk) inside a tile stored as 64-column
// halves of 128-byte rows with the 128-byte TMA swizzle.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)((chunk >> 3) * kHalfBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(256) attn_tc_kernel(const __grid_constant__ CUtensorMap mk_pool,
                                                      const __grid_constant__ CUtensorMap mv_pool,
                                                      const __grid_constant__ CUtensorMap mk_blk,
                                                      const __grid_constant__ CUtensorMap mv_blk,
                                                      const AttnParams p) {
  constexpr int NH = D / 64;                  // 64-column halves per row
  constexpr int TILE = NH * kHalfBytes;       // one K (or V) tile
  constexpr int KSTEPS = D / 16;
  constexpr int DN = D / 8;                   // 8-wide output column tiles
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *bufk[2] = {smem, smem + 2 * TILE};
  uint8_t *bufv[2] = {smem + TILE, smem + 3 * TILE};
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + 4 * TILE);

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int group = p.hq / p.hkv;
  const int R = p.block_len * group;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int L = p.block_len;

  if (p.tokens) {
    int any = 0;
    for (int i = 0; i < L; ++i) any |= (p.tokens[b * L + i] == BD_MASK);
    if (!any) return;
  }
  const int ctx = p.ctx_len[b];
  if (ctx < 0 || ctx > p.max_ctx || ctx > p.max_pages * p.page_size) {
    if (split == 0 && g == 0 && threadIdx.x == 0) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
    return;
  }
  const int kbeg = split * p.split_keys;
  const int kend = min(ctx + L, kbeg + p.split_keys);
  if (kbeg >= kend) return;                   // this split holds no key of this sequence
  const int p_first = kbeg / kPageRows;
  const int p_end = kbeg < ctx ? (min(kend, ctx) + kPageRows - 1) / kPageRows : p_first;
  const int npg = p_end - p_first;
  const int ntiles = npg + (kend > ctx ? 1 : 0);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&full[0]), 1);
    mbar_init(smem_u32(&full[1]), 1);
    fence_barrier_init();
  }
  __syncthreads();

  // page id of tile u (-1 for the block tile, -2 for a page id outside the pool)
  auto tile_page = [&](int u) -> int {
    if (u >= npg) return -1;
    const int pg = p.page_table[(size_t)b * p.max_pages + p_first + u];
    return (pg >= 0 && pg < p.num_pages) ? pg : -2;
  };
  auto issue = [&](int u) {
    const int buf = u & 1;
    const uint32_t bar = smem_u32(&full[buf]);
    const int pg = tile_page(u);
    fence_proxy_async();
    if (pg >= 0) {
      mbar_arrive_expect_tx(bar, 2 * TILE);
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        tma_load_4d(smem_u32(bufk[buf] + h * kHalfBytes), &mk_pool, 64 * h, 0, g, pg, bar);
        tma_load_4d(smem_u32(bufv[buf] + h * kHalfBytes), &mv_pool, 64 * h, 0, g, pg, bar);
      }
    } else if (pg == -1) {
      mbar_arrive_expect_tx(bar, 2 * NH * L * 128);
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        tma_load_4d(smem_u32(bufk[buf] + h * kHalfBytes), &mk_blk, 64 * h, g, 0, b, bar);
        tma_load_4d(smem_u32(bufv[buf] + h * kHalfBytes), &mv_blk, 64 * h, g, 0, b, bar);
      }
    } else {
      flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
      mbar_arrive(bar);                       // nothing to load; the tile is skipped
    }
  };
  if (threadIdx.x == 0) issue(0);

  // Q fragments of this warp's 16 rows (A operand, row-major 16x16 per k-step)
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t qa[KSTEPS][4];
  {
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
    const int r_lo = warp * 16 + gid, r_hi = r_lo + 8;
    const __nv_bfloat16 *q_lo = nullptr, *q_hi = nullptr;
    if (r_lo < R) q_lo = q + (((size_t)b * L + r_lo / group) * p.hq + g * group + r_lo % group) * D;
    if (r_hi < R) q_hi = q + (((size_t)b * L + r_hi / group) * p.hq + g * group + r_hi % group) * D;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      const int c = kk * 16 + tig * 2;
      qa[kk][0] = q_lo ? *reinterpret_cast<const uint32_t *>(q_lo + c) : 0u;
      qa[kk][1] = q_hi ? *reinterpret_cast<const uint32_t *>(q_hi + c) : 0u;
      qa[kk][2] = q_lo ? *reinterpret_cast<const uint32_t *>(q_lo + c + 8) : 0u;
      qa[kk][3] = q_hi ? *reinterpret_cast<const uint32_t *>(q_hi + c + 8) : 0u;
    }
  }

  const float sl2 = p.scale * 1.4426950408889634f;   // softmax scale in base 2
  float o[DN][4];
#pragma unroll
  for (int j = 0; j < DN; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  bool aborted = false;
  int u_stop = 0;

  for (int u = 0; u < ntiles; ++u) {
    if (threadIdx.x == 0 && u + 1 < ntiles) issue(u + 1);
    const int buf = u & 1;
    const bool ok = mbar_wait(smem_u32(&full[buf]), (u >> 1) & 1);
    if (__syncthreads_or(!ok)) {
      if (threadIdx.x == 0) flag_error(p.dev_status, BD_ERR_TIMEOUT);
      aborted = true;
      u_stop = u;
      break;
    }
    const int pg = tile_page(u);
    if (pg == -2) {                            // corrupt page id: skip the tile
      __syncthreads();
      continue;
    }
    // valid key rows [lo, hi) of this tile
    int lo = 0, hi;
    if (pg >= 0) {
      hi = min(kPageRows, ctx - (p_first + u) * kPageRows);
    } else {
      lo = max(kbeg, ctx) - ctx;
      hi = kend - ctx;
    }
    const uint32_t kbase = smem_u32(bufk[buf]);
    const uint32_t vbase = smem_u32(bufv[buf]);
    const int hi16 = (hi + 15) & ~15;
    if (hi & 15) {                             // rows past the valid ones feed P = 0: make them finite
      for (int e = threadIdx.x; e < (hi16 - hi) * NH * 8; e += blockDim.x) {
        const int row = hi + e / (NH * 8), chunk = e % (NH * 8);
        *reinterpret_cast<int4 *>(bufv[buf] + swz(row, chunk)) = make_int4(0, 0, 0, 0);
      }
      __syncthreads();
    }

    // S = Q K^T for this warp's 16 rows x 64 keys
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {
        if (16 * jp < hi) {
          const int key = 16 * jp + (lane & 7) + ((lane >> 4) << 3);
          const int chunk = 2 * kk + ((lane >> 3) & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kbase + swz(key, chunk), b0, b1, b2, b3);
          mma_16816(s[2 * jp], qa[kk], b0, b1);
          mma_16816(s[2 * jp + 1], qa[kk], b2, b3);
        }
      }
    }
    // mask, online softmax (rows gid and gid + 8 of the warp)
    float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = 8 * j + tig * 2 + (e & 1);
        if (key < lo || key >= hi) s[j][e] = -INFINITY;
        mt[e >> 1] = fmaxf(mt[e >> 1], s[j][e]);
      }
    }
    float corr[2], mneg[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mt[i] = fmaxf(mt[i], __shfl_xor_sync(0xffffffffu, mt[i], 1));
      mt[i] = fmaxf(mt[i], __shfl_xor_sync(0xffffffffu, mt[i], 2));
      const float mnew = fmaxf(m_run[i], mt[i]);
      corr[i] = exp2f((m_run[i] - mnew) * sl2);
      m_run[i] = mnew;
      mneg[i] = -mnew * sl2;
      l_run[i] *= corr[i];
    }
#pragma unroll
    for (int j = 0; j < DN; ++j) {
      o[j][0] *= corr[0];
      o[j][1] *= corr[0];
      o[j][2] *= corr[1];
      o[j][3] *= corr[1];
    }
    uint32_t pa[4][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s[j][e] = exp2f(fmaf(s[j][e], sl2, mneg[e >> 1]));
        l_run[e >> 1] += s[j][e];
      }
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      pa[kk][0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[kk][1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[kk][2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[kk][3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if (16 * kk < hi16) {
#pragma unroll
        for (int dp = 0; dp < DN / 2; ++dp) {
          const int key = 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int chunk = 2 * dp + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vbase + swz(key, chunk), b0, b1, b2, b3);
          mma_16816(o[2 * dp], pa[kk], b0, b1);
          mma_16816(o[2 * dp + 1], pa[kk], b2, b3);
        }
      }
    }
    __syncthreads();                           // buffer free for the load two tiles ahead
  }

  if (aborted) {
    // wait (bounded) for copies still in flight before the CTA's smem goes away
    if (threadIdx.x == 0)
      for (int v = u_stop; v < ntiles && v < u_stop + 2; ++v)
        mbar_wait(smem_u32(&full[v & 1]), (v >> 1) & 1);
    return;
  }

#pragma unroll
  for (int i = 0; i < 2; ++i) {
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 1);
    l_run[i] += __shfl_xor_sync(0xffffffffu, l_run[i], 2);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = warp * 16 + gid + 8 * i;
    if (r >= R) continue;
    const int qi = r / group, h = g * group + r % group;
    if (p.num_splits == 1) {
      const float inv = l_run[i] > 0.f ? 1.f / l_run[i] : 0.f;
      __nv_bfloat16 *out =
          static_cast<__nv_bfloat16 *>(p.out) + (((size_t)b * L + qi) * p.hq + h) * D;
#pragma unroll
      for (int j = 0; j < DN; ++j)
        *reinterpret_cast<uint32_t *>(out + 8 * j + tig * 2) =
            pack_bf16(o[j][2 * i] * inv, o[j][2 * i + 1] * inv);
    } else {
      const size_t prow = (((size_t)b * p.hkv + g) * p.num_splits + split) * R + r;
#pragma unroll
      for (int j = 0; j < DN; ++j)
        *reinterpret_cast<float2 *>(p.part_o + prow * D + 8 * j + tig * 2) =
            make_float2(o[j][2 * i], o[j][2 * i + 1]);
      if (tig == 0) {
        p.part_ml[prow * 2 + 0] = m_run[i] * p.scale;   // natural-log units, like the SIMT path
        p.part_ml[prow * 2 + 1] = l_run[i];
      }
    }
  }
}

template <int D>
bd_status launch(const AttnParams &p, cudaStream_t st) {
  constexpr int NH = D / 64;
  const uint64_t eb = 2;
  CUtensorMap mkp, mvp, mkb, mvb;
  const uint64_t pdims[4] = {(uint64_t)D, (uint64_t)p.page_size, (uint64_t)p.hkv,
                             (uint64_t)p.num_pages};
  const uint64_t pstr[3] = {D * eb, (uint64_t)p.page_size * D * eb,
                            (uint64_t)p.hkv * p.page_size * D * eb};
  const uint32_t pbox[4] = {64, (uint32_t)p.page_size, 1, 1};
  const uint64_t bdims[4] = {(uint64_t)D, (uint64_t)p.hkv, (uint64_t)p.block_len,
                             (uint64_t)p.batch};
  const uint64_t bstr[3] = {D * eb, (uint64_t)p.hkv * D * eb,
                            (uint64_t)p.block_len * p.hkv * D * eb};
  const uint32_t bbox[4] = {64, 1, (uint32_t)p.block_len, 1};
  if (!tma_encode_bf16(&mkp, 4, p.k_pool, pdims, pstr, pbox) ||
      !tma_encode_bf16(&mvp, 4, p.v_pool, pdims, pstr, pbox) ||
      !tma_encode_bf16(&mkb, 4, p.k_blk, bdims, bstr, bbox) ||
      !tma_encode_bf16(&mvb, 4, p.v_blk, bdims, bstr, bbox))
    return BD_ERR_CUDA;
  const int R = p.block_len * (p.hq / p.hkv);
  const int warps = (R + 15) / 16;
  const size_t smem = 4 * (size_t)NH * kHalfBytes + 64 + 1024;
  auto kern = attn_tc_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return BD_ERR_CUDA;
  dim3 grid(p.num_splits, p.hkv, p.batch);
  kern<<<grid, warps * 32, smem, st>>>(mkp, mvp, mkb, mvb, p);
  count_launches(1);
  return launch_status();
}

}  // namespace

bd_status attention_tc(const AttnParams &p, cudaStream_t st) {
  if (p.dtype != BD_BF16 || (p.head_dim != 64 && p.head_dim != 128)) return BD_ERR_UNSUPPORTED;
  if (p.page_size != kPageRows || p.block_len > 32) return BD_ERR_UNSUPPORTED;
  if (p.block_len * (p.hq / p.hkv) > 128) return BD_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(p.q) & 3) != 0) return BD_ERR_UNSUPPORTED;
  const DevInfo d = dev_info();
  if (d.major < 10 || !tma_available()) return BD_ERR_UNSUPPORTED;
  const bd_status s = p.head_dim == 64 ? launch<64>(p, st) : launch<128>(p, st);
  if (s != BD_OK || p.num_splits == 1) return s;
  return attention_combine(p, st);
}

}  // namespace bd
