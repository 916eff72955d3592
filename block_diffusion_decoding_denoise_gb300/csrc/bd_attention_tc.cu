// bf16 block attention on the tensor cores, K/V pages streamed by TMA.
//
// Same contract as attention_simt (see bd_attention.cu): the R = block_len *
// (Hq/Hkv) query rows that read KV head g attend to the keys of [cache |
// block] ("Rethinking Document OCR as Inverse Rendering via Diffusion
// Decoding", paper.rainbus.top summary, method step 3: bidirectional inside
// the block, causal to every earlier block and the prefix).
//
// Work partition (large problems): the keys of (sequence b, KV head g) form
// a segment of tiles (one per cached 64-token page, then one for the block's
// own keys); attn_plan_kernel lays the segments end to end and every CTA
// takes an equal contiguous range of tiles, so ragged batches cost no
// balance.  Small problems (a few pages per SM) skip the plan launch and deal
// fixed KV splits round-robin instead, which starts streaming sooner.  A segment
// inside one CTA's range is written as the final output; a segment cut by
// range boundaries leaves one partial per piece (slot = segment + CTA, which
// is unique because pieces are ordered along the tile line) for
// attn_combine_sk_kernel.
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

#include <algorithm>
#include <atomic>

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

// 2^x by the SFU's approximation (relative error about 2^-22; exact 0 for
// -inf), which is ample for probabilities that are rounded to bf16 next.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// Per-stage description written by the producer before it arms the stage.
struct TileMeta {
  int item;   // segment = sequence * Hkv + KV head
  int lo, hi; // valid key rows [lo, hi) of the tile
  int flags;  // kFirst | kLast | kSkip | kEnd
  int slot;   // partial slot of this piece, -1 when the piece is the whole segment
};

// Tile plan: tiles_b = ceil(ctx_b / 64) + 1 (0 for a sequence with no masked
// position or an invalid context) and base_b = (Hkv / seg_heads) *
// sum_{b' < b} tiles_b' (segments of one or two KV heads);
// plan[2b] = base_b, plan[2b + 1] = tiles_b, plan[2 batch] = the total T.
// One CTA; a block-wide scan per 1024 sequences.
__global__ void __launch_bounds__(1024) attn_plan_kernel(AttnParams p) {
  __shared__ int warp_sum[32];
  __shared__ int carry;
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int b0 = 0; b0 < p.batch; b0 += blockDim.x) {
    const int b = b0 + threadIdx.x;
    int tiles = 0;
    if (b < p.batch) {
      bool active = true;
      if (p.tokens) {
        active = false;
        const int32_t *t = p.tokens + (size_t)b * p.block_len;
        for (int i = 0; i < p.block_len; ++i) active |= t[i] == BD_MASK;
      }
      const int ctx = p.ctx_len[b];
      if (ctx < 0 || ctx > p.max_ctx || ctx > p.max_pages * p.page_size) {
        if (active) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
        active = false;
      }
      tiles = active ? (ctx + kPageRows - 1) / kPageRows + 1 : 0;
    }
    const int v = tiles * (p.hkv / p.seg_heads);
    int inc = v;                                 // inclusive scan inside the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    if (lane == 31) warp_sum[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      int w = lane < (int)(blockDim.x >> 5) ? warp_sum[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += u;
      }
      warp_sum[lane] = w;                        // inclusive over warps
    }
    __syncthreads();
    const int excl = carry + (warp > 0 ? warp_sum[warp - 1] : 0) + inc - v;
    if (b < p.batch) {
      p.plan[2 * b] = excl;
      p.plan[2 * b + 1] = tiles;
    }
    __syncthreads();
    if (threadIdx.x == 0) carry += warp_sum[31];
    __syncthreads();
  }
  if (threadIdx.x == 0) p.plan[2 * p.batch] = carry;
}
// One tile of a consumer warp: S = Q K^T over the warp's keys [max(lo, key0),
// min(hi, key0 + 8 KJ)) of the stage at bk (K, then V TILE bytes later), the
// online-softmax update of (m_run, l_run, o) and O += P V.
template <int D, int KJ>
__device__ __forceinline__ void attend_tile(uint8_t *bk, int lo, int hi, int key0, int lane,
                                            float sl2, const uint32_t (&qa)[D / 16][4],
                                            float (&o)[D / 8][4], float (&m_run)[2],
                                            float (&l_run)[2]) {
  constexpr int NH = D / 64;
  constexpr int TILE = NH * kHalfBytes;
  constexpr int KSTEPS = D / 16;
  constexpr int DN = D / 8;
  const int tig = lane & 3;
  const int w_lo = max(lo, key0), w_hi = min(hi, key0 + 8 * KJ);
  if (w_lo >= w_hi) return;
  uint8_t *bv = bk + TILE;
  const uint32_t kbase = smem_u32(bk), vbase = smem_u32(bv);
  const int hi16 = (w_hi + 15) & ~15;
  const bool zeroed = (w_hi & 15) != 0;
  if (zeroed) {                          // rows past the valid ones feed P = 0: make them finite
    for (int e = lane; e < (hi16 - w_hi) * NH * 8; e += 32) {
      const int row = w_hi + e / (NH * 8), chunk = e % (NH * 8);
      *reinterpret_cast<int4 *>(bv + swz(row, chunk)) = make_int4(0, 0, 0, 0);
    }
    __syncwarp();
  }
  // S = Q K^T for this warp's 16 rows x 8 KJ keys
  float sc[KJ][4];
#pragma unroll
  for (int j = 0; j < KJ; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
    for (int jp = 0; jp < KJ / 2; ++jp) {
      if (key0 + 16 * jp < w_hi) {
        const int key = key0 + 16 * jp + (lane & 7) + ((lane >> 4) << 3);
        const int chunk = 2 * kk + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + swz(key, chunk), b0, b1, b2, b3);
        mma_16816(sc[2 * jp], qa[kk], b0, b1);
        mma_16816(sc[2 * jp + 1], qa[kk], b2, b3);
      }
    }
  }
  float mt[2] = {-INFINITY, -INFINITY};
  if (w_lo != key0 || w_hi != key0 + 8 * KJ) {   // partial tile: mask the invalid keys
#pragma unroll
    for (int j = 0; j < KJ; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = key0 + 8 * j + tig * 2 + (e & 1);
        if (key < w_lo || key >= w_hi) sc[j][e] = -INFINITY;
      }
  }
#pragma unroll
  for (int j = 0; j < KJ; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) mt[e >> 1] = fmaxf(mt[e >> 1], sc[j][e]);
  float corr[2], mneg[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    mt[i] = fmaxf(mt[i], __shfl_xor_sync(0xffffffffu, mt[i], 1));
    mt[i] = fmaxf(mt[i], __shfl_xor_sync(0xffffffffu, mt[i], 2));
    const float mnew = fmaxf(m_run[i], mt[i]);
    corr[i] = fast_exp2((m_run[i] - mnew) * sl2);
    m_run[i] = mnew;
    mneg[i] = -mnew * sl2;
    l_run[i] *= corr[i];
  }
  // rescale only when some running max of the warp moved (a factor of
  // exactly 1 changes nothing, and after the first tiles most do not move)
  if (!__all_sync(0xffffffffu, corr[0] == 1.f && corr[1] == 1.f)) {
#pragma unroll
    for (int j = 0; j < DN; ++j) {
      o[j][0] *= corr[0];
      o[j][1] *= corr[0];
      o[j][2] *= corr[1];
      o[j][3] *= corr[1];
    }
  }
#pragma unroll
  for (int j = 0; j < KJ; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      sc[j][e] = fast_exp2(fmaf(sc[j][e], sl2, mneg[e >> 1]));
      l_run[e >> 1] += sc[j][e];
    }
  }
  uint32_t pa[KJ / 2][4];
#pragma unroll
  for (int kk = 0; kk < KJ / 2; ++kk) {
    pa[kk][0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
    pa[kk][1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
    pa[kk][2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
    pa[kk][3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
  }
#pragma unroll
  for (int kk = 0; kk < KJ / 2; ++kk) {
    if (key0 + 16 * kk < hi16) {
#pragma unroll
      for (int dp = 0; dp < DN / 2; ++dp) {
        const int key = key0 + 16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int chunk = 2 * dp + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + swz(key, chunk), b0, b1, b2, b3);
        mma_16816(o[2 * dp], pa[kk], b0, b1);
        mma_16816(o[2 * dp + 1], pa[kk], b2, b3);
      }
    }
  }
  if (zeroed) fence_proxy_async();       // our generic writes precede the next TMA fill
}

// Merge the two key halves of a row group (KH = 2): half 1 hands its state
// over through the exchange slot, half 0 folds it into its own.  Both warps
// of the row group call this once.
template <int D>
__device__ __forceinline__ void merge_key_halves(float *xchg, int rg, int kh, int lane, float sl2,
                                                 float (&o)[D / 8][4], float (&m_run)[2],
                                                 float (&l_run)[2]) {
  constexpr int DN = D / 8;
  // merge the two key halves of the row group: half 1 hands over, half 0 writes
  constexpr int F = 4 * DN + 4;        // floats per lane: o[DN][4] + m[2], l[2]
  float *xw = xchg + (size_t)rg * F * 32;
  if (kh == 1) {
#pragma unroll
    for (int j = 0; j < DN; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) xw[(j * 4 + e) * 32 + lane] = o[j][e];
    xw[(4 * DN + 0) * 32 + lane] = m_run[0];
    xw[(4 * DN + 1) * 32 + lane] = m_run[1];
    xw[(4 * DN + 2) * 32 + lane] = l_run[0];
    xw[(4 * DN + 3) * 32 + lane] = l_run[1];
  }
  named_barrier(1 + rg, 64);
  if (kh == 0) {
    float w0[2], w1[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float mo = xw[(4 * DN + i) * 32 + lane];
      const float mnew = fmaxf(m_run[i], mo);
      w0[i] = m_run[i] == -INFINITY ? 0.f : exp2f((m_run[i] - mnew) * sl2);
      w1[i] = mo == -INFINITY ? 0.f : exp2f((mo - mnew) * sl2);
      l_run[i] = l_run[i] * w0[i] + xw[(4 * DN + 2 + i) * 32 + lane] * w1[i];
      m_run[i] = mnew;
    }
#pragma unroll
    for (int j = 0; j < DN; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        o[j][e] = o[j][e] * w0[e >> 1] + xw[(j * 4 + e) * 32 + lane] * w1[e >> 1];
  }
  named_barrier(1 + rg, 64);           // exchange slot free for the next item
}

constexpr int kFirst = 1, kLast = 2, kSkip = 4, kEnd = 8;
constexpr int kMaxStages = 12;

// Persistent, warp-specialised block attention.
//   warp 0        producer: walks this CTA's tile range of the plan, and for
//                 each tile (one cached page, or the block's own keys) arms a
//                 ring stage with the tile's TMA loads and a TileMeta record
//   warps 1..NW   consumers: a row group of 16 query rows (and, with KH = 2,
//                 one half of every tile's keys) per warp; Q K^T, the online
//                 softmax and P V on each stage, release of the stage, and
//                 after a piece's last tile the output (whole segment) or the
//                 piece's partial
// A sentinel stage (kEnd) tells the consumers that the producer is done.
template <int D, int RG, int KH>
__global__ void __launch_bounds__((RG * KH + 1) * 32, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap mk_pool,
                   const __grid_constant__ CUtensorMap mv_pool,
                   const __grid_constant__ CUtensorMap mk_blk,
                   const __grid_constant__ CUtensorMap mv_blk, const AttnParams p, int S) {
  constexpr int NH = D / 64;                  // 64-column halves per row
  constexpr int TILE = NH * kHalfBytes;       // one K (or V) tile
  constexpr int KSTEPS = D / 16;
  constexpr int DN = D / 8;                   // 8-wide output column tiles
  constexpr int NW = RG * KH;                 // consumer warps
  constexpr size_t kXchgBytes = KH == 2 ? (size_t)RG * (4 * DN + 4) * 32 * 4 : 0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * 2 * TILE + kXchgBytes);
  uint64_t *empty = full + kMaxStages;
  TileMeta *meta = reinterpret_cast<TileMeta *>(empty + kMaxStages);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(meta + kMaxStages);

  const int group = p.hq / p.hkv;
  const int R = p.block_len * group;
  const int L = p.block_len;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), NW);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mk_pool);
    tma_prefetch_desc(&mv_pool);
    tma_prefetch_desc(&mk_blk);
    tma_prefetch_desc(&mv_blk);
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0;
    bool stop = false;
    // arm stage `it` (waiting for it to be free); false on timeout or abort
    auto acquire = [&](uint32_t &s_out) -> bool {
      const uint32_t s = it % S, round = it / S;
      int ok = 1;
      if (lane == 0) {
        if (*abort_flag) ok = 0;
        else if (round > 0 && !mbar_wait(smem_u32(&empty[s]), (round - 1) & 1)) {
          ok = 0;
          *abort_flag = 1;
          flag_error(p.dev_status, BD_ERR_TIMEOUT);
        }
      }
      s_out = s;
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    // Arm one tile of segment (b, g): the cached page u (keys [64u, 64u + 64)
    // of the sequence, valid up to ctx) or, for u == npg, the block's own keys
    // [klo, khi) (relative to ctx).  Lane 0 issues; returns false on abort.
    auto arm = [&](int b, int g, int u, int npg, int ctx, int klo, int khi, int seg, int slot,
                   int flags) -> bool {
      uint32_t s;
      if (!acquire(s)) return false;
      if (lane == 0) {
        const uint32_t bar = smem_u32(&full[s]);
        uint8_t *bk = smem + (size_t)s * 2 * TILE, *bv = bk + TILE;
        TileMeta m;
        m.item = seg;
        m.slot = slot;
        m.flags = flags;
        if (u < npg) {
          const int pg = p.page_table[(size_t)b * p.max_pages + u];
          m.lo = 0;
          m.hi = min(kPageRows, ctx - u * kPageRows);
          if (pg >= 0 && pg < p.num_pages) {
            meta[s] = m;
            fence_proxy_async();
            mbar_arrive_expect_tx(bar, 2 * TILE);
#pragma unroll
            for (int h = 0; h < NH; ++h) {
              tma_load_4d(smem_u32(bk + h * kHalfBytes), &mk_pool, 64 * h, 0, g, pg, bar);
              tma_load_4d(smem_u32(bv + h * kHalfBytes), &mv_pool, 64 * h, 0, g, pg, bar);
            }
          } else {
            flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
            m.flags |= kSkip;
            meta[s] = m;
            mbar_arrive(bar);
          }
        } else {
          m.lo = klo;
          m.hi = khi;
          meta[s] = m;
          fence_proxy_async();
          mbar_arrive_expect_tx(bar, 2 * NH * L * 128);
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            tma_load_4d(smem_u32(bk + h * kHalfBytes), &mk_blk, 64 * h, g, 0, b, bar);
            tma_load_4d(smem_u32(bv + h * kHalfBytes), &mv_blk, 64 * h, g, 0, b, bar);
          }
        }
      }
      __syncwarp();
      ++it;
      return true;
    };
    if (p.plan) {
      // tile-range partition: this CTA's tiles [t_begin, t_end) of the plan's T
      const int T = p.plan[2 * p.batch];
      const int c = blockIdx.x, G = gridDim.x;
      const int t_begin = (int)(((long long)c * T) / G);
      const int t_end = (int)(((long long)(c + 1) * T) / G);
      int b = 0;
      {                                          // last sequence with base <= t_begin
        int lo = 0, hi = p.batch - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (p.plan[2 * mid] <= t_begin) lo = mid;
          else hi = mid - 1;
        }
        b = lo;
      }
      for (int t = t_begin; t < t_end && !stop;) {
        while (b < p.batch - 1 && t >= p.plan[2 * b] + p.hkv * p.plan[2 * b + 1]) ++b;
        const int base = p.plan[2 * b], tiles = p.plan[2 * b + 1];
        if (tiles <= 0 || t < base || t >= base + p.hkv * tiles) {   // inconsistent plan
          if (lane == 0) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
          break;
        }
        const int g = (t - base) / tiles, u0 = (t - base) % tiles;
        const int seg0 = base + g * tiles;
        const int u1 = min(seg0 + tiles, t_end) - seg0;
        const int seg = b * p.hkv + g;
        const int slot = (u0 == 0 && u1 == tiles) ? -1 : seg + c;
        const int ctx = p.ctx_len[b];
        for (int u = u0; u < u1 && !stop; ++u)
          stop = !arm(b, g, u, tiles - 1, ctx, 0, L, seg, slot,
                      (u == u0 ? kFirst : 0) | (u == u1 - 1 ? kLast : 0));
        t = seg0 + u1;
      }
    } else {
      // KV splits (small problems): items (sequence, KV head, split) dealt
      // round-robin; split s covers keys [s * split_keys, (s + 1) * split_keys)
      const int nitems = p.batch * p.hkv * p.num_splits;
      for (int item = blockIdx.x; item < nitems && !stop; item += gridDim.x) {
        const int split = item % p.num_splits;
        const int g = (item / p.num_splits) % p.hkv;
        const int b = item / (p.num_splits * p.hkv);
        if (p.tokens && !block_has_mask(p.tokens + (size_t)b * L, L)) continue;
        const int ctx = p.ctx_len[b];
        if (ctx < 0 || ctx > p.max_ctx || ctx > p.max_pages * p.page_size) {
          if (split == 0 && g == 0 && lane == 0) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
          continue;
        }
        const int kbeg = split * p.split_keys;
        const int kend = min(ctx + L, kbeg + p.split_keys);
        if (kbeg >= kend) continue;              // no key of this sequence in this split
        const int p_first = kbeg / kPageRows;
        const int npg = (ctx + kPageRows - 1) / kPageRows;
        const int p_end = kbeg < ctx ? (min(kend, ctx) + kPageRows - 1) / kPageRows : p_first;
        const int ntiles = (p_end - p_first) + (kend > ctx ? 1 : 0);
        const int seg = b * p.hkv + g;
        const int slot = p.num_splits == 1 ? -1 : seg * p.num_splits + split;
        for (int k = 0; k < ntiles && !stop; ++k) {
          const int u = p_first + k < p_end ? p_first + k : npg;
          stop = !arm(b, g, u, npg, ctx, max(kbeg, ctx) - ctx, kend - ctx, seg, slot,
                      (k == 0 ? kFirst : 0) | (k == ntiles - 1 ? kLast : 0));
        }
      }
    }
    // sentinel: tells the consumers there is no more work
    if (!stop) {
      uint32_t s;
      if (acquire(s)) {
        if (lane == 0) {
          meta[s] = TileMeta{-1, 0, 0, kEnd, -1};
          mbar_arrive(smem_u32(&full[s]));
        }
        ++it;
      } else {
        stop = true;
      }
    }
    if (stop && lane == 0) {                   // drain copies that may still be in flight
      const uint32_t first = it > (uint32_t)S ? it - S : 0;
      for (uint32_t i = first; i < it; ++i) mbar_wait(smem_u32(&full[i % S]), (i / S) & 1);
    }
  } else {
    // ------------------------------------------------------------ consumers
    // warp cw owns rows [16 rg, 16 rg + 16) and, when KH == 2, one half of the
    // keys of every tile; the two key halves of a row group merge at item end
    const int cw = warp - 1;
    const int rg = cw % RG, kh = cw / RG;
    constexpr int KJ = 8 / KH;                 // 8-key column tiles per warp
    const int key0 = kh * 8 * KJ;              // first key of this warp within a tile
    const int gid = lane >> 2, tig = lane & 3;
    const float sl2 = p.scale * 1.4426950408889634f;   // softmax scale in base 2
    float *xchg = reinterpret_cast<float *>(smem + (size_t)S * 2 * TILE);   // key-half exchange
    uint32_t qa[KSTEPS][4];
    float o[DN][4];
    float m_run[2], l_run[2];
    int b = 0, g = 0;
    for (uint32_t it = 0;; ++it) {
      const uint32_t s = it % S;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(smem_u32(&full[s]), (it / S) & 1) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) {
          *abort_flag = 1;
          flag_error(p.dev_status, BD_ERR_TIMEOUT);
        }
        break;
      }
      TileMeta m;
      {
        const volatile int *mv = reinterpret_cast<const volatile int *>(&meta[s]);
        m.item = mv[0];
        m.lo = mv[1];
        m.hi = mv[2];
        m.flags = mv[3];
        m.slot = mv[4];
      }
      if (m.flags & kEnd) break;
      if (m.flags & kFirst) {
        g = m.item % p.hkv;
        b = m.item / p.hkv;
        const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
        const int r_lo = rg * 16 + gid, r_hi = r_lo + 8;
        const __nv_bfloat16 *q_lo = nullptr, *q_hi = nullptr;
        if (r_lo < R)
          q_lo = q + (((size_t)b * L + r_lo / group) * p.hq + g * group + r_lo % group) * D;
        if (r_hi < R)
          q_hi = q + (((size_t)b * L + r_hi / group) * p.hq + g * group + r_hi % group) * D;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
          const int c = kk * 16 + tig * 2;
          qa[kk][0] = q_lo ? *reinterpret_cast<const uint32_t *>(q_lo + c) : 0u;
          qa[kk][1] = q_hi ? *reinterpret_cast<const uint32_t *>(q_hi + c) : 0u;
          qa[kk][2] = q_lo ? *reinterpret_cast<const uint32_t *>(q_lo + c + 8) : 0u;
          qa[kk][3] = q_hi ? *reinterpret_cast<const uint32_t *>(q_hi + c + 8) : 0u;
        }
#pragma unroll
        for (int j = 0; j < DN; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
      }
      if (!(m.flags & kSkip))
        attend_tile<D, KJ>(smem + (size_t)s * 2 * TILE, m.lo, m.hi, key0, lane, sl2, qa, o, m_run,
                           l_run);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
      if (m.flags & kLast) {
        if (KH == 2) merge_key_halves<D>(xchg, rg, kh, lane, sl2, o, m_run, l_run);
        if (kh == 0) {
          float lsum[2];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            lsum[i] = l_run[i] + __shfl_xor_sync(0xffffffffu, l_run[i], 1);
            lsum[i] += __shfl_xor_sync(0xffffffffu, lsum[i], 2);
          }
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int r = rg * 16 + gid + 8 * i;
            if (r >= R) continue;
            const int qi = r / group, h = g * group + r % group;
            if (m.slot < 0) {
              const float inv = lsum[i] > 0.f ? 1.f / lsum[i] : 0.f;
              __nv_bfloat16 *out =
                  static_cast<__nv_bfloat16 *>(p.out) + (((size_t)b * L + qi) * p.hq + h) * D;
#pragma unroll
              for (int j = 0; j < DN; ++j)
                *reinterpret_cast<uint32_t *>(out + 8 * j + tig * 2) =
                    pack_bf16(o[j][2 * i] * inv, o[j][2 * i + 1] * inv);
            } else {
              const size_t prow = (size_t)m.slot * R + r;
#pragma unroll
              for (int j = 0; j < DN; ++j)
                *reinterpret_cast<float2 *>(p.sk_o + prow * D + 8 * j + tig * 2) =
                    make_float2(o[j][2 * i], o[j][2 * i + 1]);
              if (tig == 0) {
                p.sk_ml[prow * 2 + 0] = m_run[i] * p.scale;     // natural-log units
                p.sk_ml[prow * 2 + 1] = lsum[i];
              }
            }
          }
        }
      }
    }
  }
  __syncthreads();
}

// Block attention for small problems, one launch (cluster form).
//
// A cluster of C CTAs works on one segment (sequence b, KV head g).  The
// segment's tiles are numbered on a grid fixed by max_ctx: u = 0 .. Tm - 1
// with Tm = ceil(max_ctx / 64) + 1; tile u < npg = ceil(ctx / 64) is cached
// page u, tile npg is the block's own keys and later tiles are empty.  CTA
// rank r takes tiles [r Tm / C, (r + 1) Tm / C).  That range does not depend
// on ctx, so the producer issues its loads of the block's tokens, of ctx and
// of the range's page ids together (one memory latency before the first TMA),
// and the consumers load their Q rows before the first tile lands.  At the
// end every CTA writes its piece's state (m in base-2 units, l, O) to its
// slot of the workspace; after a cluster barrier CTA r merges rows
// [r R / C, (r + 1) R / C) of the C pieces from L2,
//   out = sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k,
// and writes them as bf16.  (Reading the pieces straight from the other CTAs'
// shared memory was measured slower: about 2 us per row group of 12 to 16
// remote loads per lane.)  With C == 1 the piece is the segment and is
// written as the output.
constexpr int kMaxCluster = 16;

template <int D, int RG, int KH>
__global__ void __launch_bounds__((RG * KH + 1) * 32, 1)
    attn_cluster_kernel(const __grid_constant__ CUtensorMap mk_pool,
                        const __grid_constant__ CUtensorMap mv_pool,
                        const __grid_constant__ CUtensorMap mk_blk,
                        const __grid_constant__ CUtensorMap mv_blk, const AttnParams p, int S,
                        int C, int Tm) {
  constexpr int NH = D / 64;
  constexpr int TILE = NH * kHalfBytes;
  constexpr int KSTEPS = D / 16;
  constexpr int DN = D / 8;
  constexpr int DPL = D / 32;                 // merged columns per lane
  constexpr int NW = RG * KH;
  constexpr int KJ = 8 / KH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * 2 * TILE);
  uint64_t *empty = full + kMaxStages;
  TileMeta *meta = reinterpret_cast<TileMeta *>(empty + kMaxStages);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(meta + kMaxStages);
  volatile int *active_flag = abort_flag + 1;

  const int group = p.hq / p.hkv;
  const int R = p.block_len * group;
  const int L = p.block_len;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  const int seg = blockIdx.x / C;
  const int b = seg / p.hkv, g = seg % p.hkv;
  const float sl2 = p.scale * 1.4426950408889634f;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), NW);
    }
    *abort_flag = 0;
    *active_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mk_pool);
    tma_prefetch_desc(&mv_pool);
    tma_prefetch_desc(&mk_blk);
    tma_prefetch_desc(&mv_blk);
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();

  // consumer state (warps 1..NW); warp cw owns rows [16 rg, 16 rg + 16) and,
  // when KH == 2, one half of the keys of every tile
  const int cw = warp - 1;
  const int rg = cw % RG, kh = cw / RG;
  const int key0 = kh * 8 * KJ;
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t qa[KSTEPS][4];
  float o[DN][4];
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
#pragma unroll
  for (int j = 0; j < DN; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const int u0 = (int)((long long)rank * Tm / C), u1 = (int)((long long)(rank + 1) * Tm / C);
    const int32_t *tok = p.tokens ? p.tokens + (size_t)b * L : nullptr;
    const int32_t *ptab = p.page_table + (size_t)b * p.max_pages;
    // one memory latency: the block's tokens, ctx and the first 32 page ids
    const int t = (tok && lane < L) ? tok[lane] : 0;
    const int ctx = p.ctx_len[b];
    int pid = -1;
    if (u0 + lane < u1 && u0 + lane < p.max_pages) pid = ptab[u0 + lane];
    const bool has = !tok || __any_sync(0xffffffffu, lane < L && t == BD_MASK);
    const bool ctx_ok = ctx >= 0 && ctx <= p.max_ctx && ctx <= p.max_pages * p.page_size;
    if (has && !ctx_ok && rank == 0 && lane == 0) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
    const bool active = has && ctx_ok;
    if (lane == 0) *active_flag = active ? 1 : 0;
    uint32_t it = 0;
    bool stop = false;
    auto acquire = [&](uint32_t &s_out) -> bool {
      const uint32_t s = it % S, round = it / S;
      int ok = 1;
      if (lane == 0) {
        if (*abort_flag) ok = 0;
        else if (round > 0 && !mbar_wait(smem_u32(&empty[s]), (round - 1) & 1)) {
          ok = 0;
          *abort_flag = 1;
          flag_error(p.dev_status, BD_ERR_TIMEOUT);
        }
      }
      s_out = s;
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    if (active) {
      const int npg = (ctx + kPageRows - 1) / kPageRows;
      const int last = min(u1, npg + 1);
      for (int c0 = u0; c0 < last && !stop; c0 += 32) {
        if (c0 != u0) {
          pid = -1;
          if (c0 + lane < last && c0 + lane < npg) pid = ptab[c0 + lane];
        }
        const int cend = min(c0 + 32, last);
        for (int u = c0; u < cend && !stop; ++u) {
          const int pg = __shfl_sync(0xffffffffu, pid, u - c0);
          uint32_t s;
          if (!acquire(s)) {
            stop = true;
            break;
          }
          if (lane == 0) {
            const uint32_t bar = smem_u32(&full[s]);
            uint8_t *bk = smem + (size_t)s * 2 * TILE, *bv = bk + TILE;
            TileMeta m;
            m.item = seg;
            m.slot = -1;
            m.flags = 0;
            m.lo = 0;
            if (u < npg) {
              m.hi = min(kPageRows, ctx - u * kPageRows);
              if (pg >= 0 && pg < p.num_pages) {
                meta[s] = m;
                fence_proxy_async();
                mbar_arrive_expect_tx(bar, 2 * TILE);
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                  tma_load_4d(smem_u32(bk + h * kHalfBytes), &mk_pool, 64 * h, 0, g, pg, bar);
                  tma_load_4d(smem_u32(bv + h * kHalfBytes), &mv_pool, 64 * h, 0, g, pg, bar);
                }
              } else {
                flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
                m.flags = kSkip;
                meta[s] = m;
                mbar_arrive(bar);
              }
            } else {                               // u == npg: the block's own keys
              m.hi = L;
              meta[s] = m;
              fence_proxy_async();
              mbar_arrive_expect_tx(bar, 2 * NH * L * 128);
#pragma unroll
              for (int h = 0; h < NH; ++h) {
                tma_load_4d(smem_u32(bk + h * kHalfBytes), &mk_blk, 64 * h, g, 0, b, bar);
                tma_load_4d(smem_u32(bv + h * kHalfBytes), &mv_blk, 64 * h, g, 0, b, bar);
              }
            }
          }
          __syncwarp();
          ++it;
        }
      }
    }
    if (!stop) {
      uint32_t s;
      if (acquire(s)) {
        if (lane == 0) {
          meta[s] = TileMeta{-1, 0, 0, kEnd, -1};
          mbar_arrive(smem_u32(&full[s]));
        }
        ++it;
      }
    }
    // Wait for every copy this CTA issued (each stage's last use), so that
    // the stage memory is free for the merge below; on the normal path the
    // consumers have already seen all of them land.
    if (lane == 0) {
      const uint32_t first = it > (uint32_t)S ? it - S : 0;
      for (uint32_t i = first; i < it; ++i) mbar_wait(smem_u32(&full[i % S]), (i / S) & 1);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    {
      const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q);
      const int r_lo = rg * 16 + gid, r_hi = r_lo + 8;
      const __nv_bfloat16 *q_lo = nullptr, *q_hi = nullptr;
      if (r_lo < R)
        q_lo = q + (((size_t)b * L + r_lo / group) * p.hq + g * group + r_lo % group) * D;
      if (r_hi < R)
        q_hi = q + (((size_t)b * L + r_hi / group) * p.hq + g * group + r_hi % group) * D;
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        const int c = kk * 16 + tig * 2;
        qa[kk][0] = q_lo ? *reinterpret_cast<const uint32_t *>(q_lo + c) : 0u;
        qa[kk][1] = q_hi ? *reinterpret_cast<const uint32_t *>(q_hi + c) : 0u;
        qa[kk][2] = q_lo ? *reinterpret_cast<const uint32_t *>(q_lo + c + 8) : 0u;
        qa[kk][3] = q_hi ? *reinterpret_cast<const uint32_t *>(q_hi + c + 8) : 0u;
      }
    }
    for (uint32_t it = 0;; ++it) {
      const uint32_t s = it % S;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(smem_u32(&full[s]), (it / S) & 1) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) {
          *abort_flag = 1;
          flag_error(p.dev_status, BD_ERR_TIMEOUT);
        }
        break;
      }
      const volatile int *mv = reinterpret_cast<const volatile int *>(&meta[s]);
      const int lo = mv[1], hi = mv[2], flags = mv[3];
      if (flags & kEnd) break;
      if (!(flags & kSkip))
        attend_tile<D, KJ>(smem + (size_t)s * 2 * TILE, lo, hi, key0, lane, sl2, qa, o, m_run,
                           l_run);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
  }
  __syncthreads();                             // stage memory free: the key-half exchange goes there

  // This CTA's piece: with C == 1 it is the whole segment and is written as
  // the output; otherwise O [R][D] fp32 goes to slot blockIdx.x of sk_o and
  // (m in base-2 units, l) [R][2] to sk_ml, and after a cluster barrier
  // (release/acquire at cluster scope) CTA rank r merges rows [r R / C,
  // (r + 1) R / C) of the C pieces of its cluster.
  float *xchg = reinterpret_cast<float *>(smem);
  const bool active = *active_flag != 0;
  if (warp > 0) {
    if (KH == 2) merge_key_halves<D>(xchg, rg, kh, lane, sl2, o, m_run, l_run);
    if (kh == 0) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float ls = l_run[i] + __shfl_xor_sync(0xffffffffu, l_run[i], 1);
        ls += __shfl_xor_sync(0xffffffffu, ls, 2);
        const int r = rg * 16 + gid + 8 * i;
        if (r >= R) continue;
        if (C == 1) {
          if (!active) continue;
          const float inv = ls > 0.f ? 1.f / ls : 0.f;
          const int qi = r / group, h = g * group + r % group;
          __nv_bfloat16 *out =
              static_cast<__nv_bfloat16 *>(p.out) + (((size_t)b * L + qi) * p.hq + h) * D;
#pragma unroll
          for (int j = 0; j < DN; ++j)
            *reinterpret_cast<uint32_t *>(out + 8 * j + tig * 2) =
                pack_bf16(o[j][2 * i] * inv, o[j][2 * i + 1] * inv);
        } else {
          const size_t prow = (size_t)blockIdx.x * R + r;
          if (m_run[i] != -INFINITY) {
#pragma unroll
            for (int j = 0; j < DN; ++j)
              *reinterpret_cast<float2 *>(p.sk_o + prow * D + 8 * j + tig * 2) =
                  make_float2(o[j][2 * i], o[j][2 * i + 1]);
          }
          if (tig == 0)
            *reinterpret_cast<float2 *>(p.sk_ml + prow * 2) = make_float2(m_run[i] * sl2, ls);
        }
      }
    }
  }
  if (C > 1) {
    cluster_sync();                            // every piece of the cluster is written
    if (active) {
      const size_t first = (size_t)blockIdx.x - rank;   // CTA of rank 0
      const int r_begin = (int)((long long)rank * R / C), r_end = (int)((long long)(rank + 1) * R / C);
      for (int r = r_begin + warp; r < r_end; r += NW + 1) {
        float2 ml = make_float2(-INFINITY, 0.f);
        if (lane < C)
          ml = __ldcg(reinterpret_cast<const float2 *>(p.sk_ml + ((first + lane) * R + r) * 2));
        float mx = ml.x;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float w = (lane < C && ml.x != -INFINITY) ? exp2f(ml.x - mx) : 0.f;
        float l = w * ml.y;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
        float v[kMaxCluster][DPL];
        float wk[kMaxCluster];
#pragma unroll
        for (int k = 0; k < kMaxCluster; ++k) {
          wk[k] = __shfl_sync(0xffffffffu, w, k & 31);
          const float *src = p.sk_o + ((first + k) * R + r) * D + lane * DPL;
          if (k < C && wk[k] > 0.f) {
            if constexpr (DPL == 4) {
              const float4 x = __ldcg(reinterpret_cast<const float4 *>(src));
              v[k][0] = x.x;
              v[k][1] = x.y;
              v[k][2] = x.z;
              v[k][3] = x.w;
            } else {
              const float2 x = __ldcg(reinterpret_cast<const float2 *>(src));
              v[k][0] = x.x;
              v[k][1] = x.y;
            }
          } else {
#pragma unroll
            for (int d = 0; d < DPL; ++d) v[k][d] = 0.f;
          }
        }
        float acc[DPL];
#pragma unroll
        for (int d = 0; d < DPL; ++d) acc[d] = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxCluster; ++k)
#pragma unroll
          for (int d = 0; d < DPL; ++d) acc[d] = fmaf(wk[k], v[k][d], acc[d]);
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int qi = r / group, h = g * group + r % group;
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out) +
                             (((size_t)b * L + qi) * p.hq + h) * D + lane * DPL;
        if constexpr (DPL == 4) {
          *reinterpret_cast<uint2 *>(out) =
              make_uint2(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv));
        } else {
          *reinterpret_cast<uint32_t *>(out) = pack_bf16(acc[0] * inv, acc[1] * inv);
        }
      }
    }
  }
}

// TMA maps of one call: the pool as [page][Hkv][64][D] and the block's keys
// as [B][L'][Hkv][D], each read in [64 keys][64 columns] boxes.
template <int D>
bool encode_maps(const AttnParams &p, CUtensorMap &mkp, CUtensorMap &mvp, CUtensorMap &mkb,
                 CUtensorMap &mvb) {
  const uint64_t eb = 2;
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
    return false;
  return true;
}

template <int D, int RG, int KH>
bd_status launch(const AttnParams &p, cudaStream_t st) {
  constexpr int NW = RG * KH;
  constexpr size_t kXchgBytes = KH == 2 ? (size_t)RG * (4 * (D / 8) + 4) * 32 * 4 : 0;
  constexpr int NH = D / 64;
  constexpr int TILE = NH * kHalfBytes;
  CUtensorMap mkp, mvp, mkb, mvb;
  if (!encode_maps<D>(p, mkp, mvp, mkb, mvb)) return BD_ERR_CUDA;
  const size_t ctrl = kMaxStages * (2 * sizeof(uint64_t) + sizeof(TileMeta)) + 16;
  const int S = (int)std::min<size_t>(kMaxStages,
                                      (200 * 1024 - ctrl - kXchgBytes) / (2 * TILE));
  const size_t smem = (size_t)S * 2 * TILE + kXchgBytes + ctrl + 1024;
  auto kern = attn_tc_kernel<D, RG, KH>;
  int grid = p.grid;
  if (p.plan) {
    if (attention_plan_launch(p, st) != cudaSuccess) return BD_ERR_CUDA;
  } else {
    grid = std::max(1, std::min(p.batch * p.hkv * p.num_splits, p.grid));
  }
  const cudaError_t e =
      launch_pdl(kern, dim3(grid), dim3((NW + 1) * 32), smem, st, mkp, mvp, mkb, mvb, p, S);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}


// Shared memory of attn_cluster_kernel: S stages of K and V, the control
// block, and the alignment slack; the stages also hold the key-half exchange
// at the end.
template <int D, int RG, int KH>
bool cluster_layout(int R, int *S_out, size_t *smem_out) {
  constexpr int TILE = (D / 64) * kHalfBytes;
  constexpr size_t kXchgBytes = KH == 2 ? (size_t)RG * (4 * (D / 8) + 4) * 32 * 4 : 0;
  constexpr size_t kOptin = 227 * 1024;
  const size_t ctrl = kMaxStages * (2 * sizeof(uint64_t) + sizeof(TileMeta)) + 16;
  const int S = (int)std::min<size_t>(kMaxStages, (kOptin - 1024 - ctrl) / (2 * TILE));
  if (S < 2 || kXchgBytes > (size_t)S * 2 * TILE) return false;
  *S_out = S;
  *smem_out = (size_t)S * 2 * TILE + ctrl + 1024;
  return true;
}

// Clusters of C CTAs of attn_cluster_kernel that the device holds at once
// (cached per device and C; 0 when the size cannot be launched).
template <int D, int RG, int KH>
int active_clusters(int C, size_t smem) {
  static std::atomic<int> cache[64][kMaxCluster + 1];
  static std::atomic<bool> init{false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  if (!init.exchange(true))
    for (auto &row : cache)
      for (auto &c : row) c.store(-1);
  const int hit = cache[dev][C].load();
  if (hit >= 0) return hit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3((RG * KH + 1) * 32);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attn_cluster_kernel<D, RG, KH>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[dev][C].store(n);
  return n;
}

// One cluster per segment; C as large as the SMs allow (each CTA then streams
// a few pages), reduced until all clusters of the call fit on the device at once.
template <int D, int RG, int KH>
bd_status launch_cluster(const AttnParams &p, cudaStream_t st) {
  constexpr int NW = RG * KH;
  const int R = p.block_len * (p.hq / p.hkv);
  int S;
  size_t smem;
  if (!cluster_layout<D, RG, KH>(R, &S, &smem)) return BD_ERR_UNSUPPORTED;
  const long long segs = (long long)p.batch * p.hkv;
  if (segs > (1LL << 24) || !p.sk_o || !p.sk_ml || p.grid < 1) return BD_ERR_UNSUPPORTED;
  const int sms = std::max(1, dev_info().sms);
  const int Tm = (p.max_ctx + kPageRows - 1) / kPageRows + 1;
  // pieces (C > 1) take one R-row slot of sk_o / sk_ml per CTA: segs * C <= grid
  int C = (int)std::min<long long>(std::min(kMaxCluster, Tm),
                                   std::max(1LL, std::min<long long>(sms, p.grid) / segs));
  while (C > 1 && active_clusters<D, RG, KH>(C, smem) < std::min<long long>(segs, sms / C)) --C;
  if (active_clusters<D, RG, KH>(C, smem) < 1) return BD_ERR_UNSUPPORTED;
  CUtensorMap mkp, mvp, mkb, mvb;
  if (!encode_maps<D>(p, mkp, mvp, mkb, mvb)) return BD_ERR_CUDA;
  const cudaError_t e =
      launch_pdl_cluster(attn_cluster_kernel<D, RG, KH>, dim3((unsigned)(segs * C)),
                         dim3((NW + 1) * 32), smem, st, dim3(C, 1, 1), mkp, mvp, mkb, mvb, p, S,
                         C, Tm);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}
}  // namespace

cudaError_t attention_plan_launch(const AttnParams &p, cudaStream_t st) {
  const cudaError_t e = launch_pdl(attn_plan_kernel, dim3(1), dim3(1024), 0, st, p);
  count_launches(1);
  return e;
}

// The cluster kernel may run clusters of up to 16 CTAs (beyond the portable 8).
template <int D, int RG, int KH>
static bool preload_cluster() {
  auto k = attn_cluster_kernel<D, RG, KH>;
  return preload_kernel(k, true) &&
         cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
}

bool preload_attention_tc() {
  return preload_cluster<64, 4, 2>() && preload_cluster<64, 8, 1>() &&
         preload_cluster<128, 4, 2>() && preload_cluster<128, 8, 1>() &&
         preload_kernel(attn_plan_kernel, false) && preload_kernel(attn_tc_kernel<64, 4, 2>, true) &&
         preload_kernel(attn_tc_kernel<64, 8, 1>, true) &&
         preload_kernel(attn_tc_kernel<128, 4, 2>, true) &&
         preload_kernel(attn_tc_kernel<128, 8, 1>, true);
}

// Shapes both bf16 tensor-core kernels take.
static bool tc_shape_ok(const AttnParams &p) {
  if (p.dtype != BD_BF16 || (p.head_dim != 64 && p.head_dim != 128)) return false;
  if (p.page_size != kPageRows || p.block_len > 32) return false;
  if (p.block_len * (p.hq / p.hkv) > 128) return false;
  if ((reinterpret_cast<uintptr_t>(p.q) & 3) != 0) return false;
  const DevInfo d = dev_info();
  return d.major >= 10 && tma_available();
}

bd_status attention_cluster(const AttnParams &p, cudaStream_t st) {
  if (!tc_shape_ok(p) || (reinterpret_cast<uintptr_t>(p.out) & 7) != 0) return BD_ERR_UNSUPPORTED;
  const int R = p.block_len * (p.hq / p.hkv);
  if (p.head_dim == 64)
    return R <= 64 ? launch_cluster<64, 4, 2>(p, st) : launch_cluster<64, 8, 1>(p, st);
  return R <= 64 ? launch_cluster<128, 4, 2>(p, st) : launch_cluster<128, 8, 1>(p, st);
}

bd_status attention_tc(const AttnParams &p, cudaStream_t st) {
  if (!tc_shape_ok(p)) return BD_ERR_UNSUPPORTED;
  if (p.grid < 1 || ((p.plan || p.num_splits > 1) && (!p.sk_o || !p.sk_ml)))
    return BD_ERR_UNSUPPORTED;
  if (p.plan && (long long)p.batch * p.hkv * (p.max_pages + 1) >= (1LL << 30))
    return BD_ERR_UNSUPPORTED;
  const int R = p.block_len * (p.hq / p.hkv);
  bd_status s;
  // up to 64 rows: 4 row groups x 2 key halves; up to 128 rows: 8 row groups
  if (p.head_dim == 64)
    s = R <= 64 ? launch<64, 4, 2>(p, st) : launch<64, 8, 1>(p, st);
  else
    s = R <= 64 ? launch<128, 4, 2>(p, st) : launch<128, 8, 1>(p, st);
  if (s != BD_OK) return s;
  if (p.plan) return attention_combine_sk(p, st);
  return p.num_splits > 1 ? attention_combine(p, st) : BD_OK;
}

}  // namespace bd
