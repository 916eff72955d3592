// bf16 block attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Same contract, work items and split partials as attention_tc (mma.sync):
// query rows r = i * (Hq/Hkv) + j of the current block against the cached
// keys of KV head g plus the block's own keys ("Rethinking Document OCR as
// Inverse Rendering via Diffusion Decoding", paper.rainbus.top summary,
// method step 3).  Used for head_dim 128 and at most 64 query rows per KV
// head, where the legacy warp-level MMA, not HBM, limits the mma.sync kernel.
//
// Per tile of 128 keys (two cached pages, or the block's keys):
//   MMA1  S^T[key][row]  = K[key][:] . Q[row][:]      M=128 keys, N=rows, K=D
//         (A = K tile, B = Q, both K-major in 128-byte-swizzled smem; D in TMEM)
//   softmax warps read S^T (one key per TMEM lane), reduce each row's max and
//         sum over the 128 lanes with butterflies, update the running max,
//         write P = exp(S - m) as bf16 into smem (row-major, K-major for MMA2)
//         and zero the V rows of masked keys
//   MMA2  O_t^T[d][row] = V^T[d][key] . P^T[key][row]  M=128 (D), N=rows, K=128
//         (A = the V tile read MN-major, B = P)
//   the same warps read O_t^T (one d per lane) and keep O[d][row] in registers:
//   O = O * exp(m_old - m_new) + O_t.
// Warp roles (192 threads, one CTA per SM, persistent over work items):
//   warp 0 TMA producer (Q per item, K/V per tile, two ring stages),
//   warp 1 TMEM allocator and MMA issuer (MMA1 of tile t+1 overlaps the
//   softmax of tile t), warps 2-5 softmax / accumulation.
// All waits are bounded; on expiry the kernel records BD_ERR_TIMEOUT.
#include <math.h>

#include <algorithm>

#include "bd_attention.cuh"
#include "bd_common.cuh"
#include "bd_sm100.cuh"

namespace bd {

using namespace sm100;

namespace {

constexpr int D = 128;
constexpr int kTK = 128;                    // keys per tile
constexpr int kPage = 64;
constexpr int kHalf = kTK * 128;            // one 64-column half of a 128-key tile: 16 KB
constexpr int kKV = 2 * kHalf;              // K (or V) of one stage: 32 KB
constexpr int kQHalf = 64 * 128;            // one half of Q (64 rows): 8 KB
constexpr int kPAtom = 64 * 128;            // 64 rows x 64 keys of P: 8 KB
constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;         // S^T x2 (64 cols each) + O^T x2
constexpr int kFirst = 1, kLast = 2, kSkip = 4, kEnd = 8;

struct Meta {
  int item, lo, hi, flags;
};

struct Smem {
  uint8_t k[kStages][kKV];
  uint8_t v[kStages][kKV];
  uint8_t q[2][2 * kQHalf];
  uint8_t pm[2][2 * kPAtom];
  float red[4][64];
  float m_run[64], l_run[64];
  float corr[2][64];
  Meta meta[kStages];
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], s_empty[2], p_full[2], o_full[2], o_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  volatile int abort_flag;
};

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

// MN-major 128-byte-swizzled operand (the V tile read as V^T): rows of 128 B
// hold 64 consecutive elements along M (head dim), 8-row groups along K (keys)
// are 1024 B apart, the next 64 elements along M sit one half (16 KB) further.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(kHalf >> 4) << 16;        // leading byte offset: next 64 along M
  d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: next 8 along K
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ bool barrier_or(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// tcgen05.ld of 16 fp32 columns of this warp's 32 lanes
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  tmem_ld_32x32b_x16(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// Transposing butterfly over the warp: 16 columns in, lanes 2k and 2k+1 end
// with column k reduced over the 32 lanes (max when MAX, else sum).
template <bool MAX>
__device__ __forceinline__ float bfly16(float (&x)[16], int lane) {
#pragma unroll
  for (int K = 8, off = 16; K >= 1; K >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const float send = upper ? x[k] : x[K + k];
      const float keep = upper ? x[K + k] : x[k];
      const float got = __shfl_xor_sync(0xffffffffu, send, off);
      x[k] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  const float o = __shfl_xor_sync(0xffffffffu, x[0], 1);
  return MAX ? fmaxf(x[0], o) : x[0] + o;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc5_kernel(const __grid_constant__ CUtensorMap mk_pool,
                    const __grid_constant__ CUtensorMap mv_pool,
                    const __grid_constant__ CUtensorMap mk_blk,
                    const __grid_constant__ CUtensorMap mv_blk,
                    const __grid_constant__ CUtensorMap mq, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = p.hq / p.hkv;
  const int L = p.block_len;
  const int R = L * group;
  const int npad = (R + 15) & ~15;
  const int nitems = p.batch * p.hkv * p.num_splits;
  const float sl2 = p.scale * 1.4426950408889634f;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.kv_full[s]), 1);
      mbar_init(smem_u32(&sm.kv_empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.q_full[i]), 1);
      mbar_init(smem_u32(&sm.q_empty[i]), 1);
      mbar_init(smem_u32(&sm.s_full[i]), 1);
      mbar_init(smem_u32(&sm.s_empty[i]), 4);
      mbar_init(smem_u32(&sm.p_full[i]), 4);
      mbar_init(smem_u32(&sm.o_full[i]), 1);
      mbar_init(smem_u32(&sm.o_empty[i]), 4);
    }
    mbar_init(smem_u32(&sm.mma_done), 1);
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mk_pool);
    tma_prefetch_desc(&mv_pool);
    tma_prefetch_desc(&mk_blk);
    tma_prefetch_desc(&mv_blk);
    tma_prefetch_desc(&mq);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  pdl_trigger();
  pdl_wait();

  auto fail = [&]() {
    sm.abort_flag = 1;
    flag_error(p.dev_status, BD_ERR_TIMEOUT);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0, nq = 0;
    bool stop = false;
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
      if (kbeg >= kend) continue;
      const int p_first = kbeg / kPage;
      const int p_end = kbeg < ctx ? (min(kend, ctx) + kPage - 1) / kPage : p_first;
      const int npt = (p_end - p_first + 1) / 2;   // page-pair tiles
      const int ntiles = npt + (kend > ctx ? 1 : 0);
      if (lane == 0) {
        // Q of this item (rows i * group + j), released by the MMA warp after the item
        const uint32_t qb = nq & 1;
        if (nq >= 2 && !mbar_wait(smem_u32(&sm.q_empty[qb]), ((nq >> 1) - 1) & 1)) {
          fail();
          stop = true;
        } else {
          const uint32_t bar = smem_u32(&sm.q_full[qb]);
          mbar_arrive_expect_tx(bar, 2 * R * 128);
          for (int h = 0; h < 2; ++h)
            tma_load_4d(smem_u32(sm.q[qb] + h * kQHalf), &mq, 64 * h, g * group, 0, b, bar);
        }
      }
      stop = __shfl_sync(0xffffffffu, stop ? 1 : 0, 0) != 0;
      if (stop) break;
      ++nq;
      for (int u = 0; u < ntiles; ++u, ++it) {
        const uint32_t s = it % kStages, round = it / kStages;
        int ok = 1;
        if (lane == 0) {
          if (sm.abort_flag) ok = 0;
          else if (round > 0 && !mbar_wait(smem_u32(&sm.kv_empty[s]), (round - 1) & 1)) {
            fail();
            ok = 0;
          }
          if (ok) {
            const uint32_t bar = smem_u32(&sm.kv_full[s]);
            Meta m;
            m.item = item;
            m.flags = (u == 0 ? kFirst : 0) | (u == ntiles - 1 ? kLast : 0);
            if (u < npt) {
              const int pa = p_first + 2 * u;
              const bool two = pa + 1 < p_end;
              const int ga = p.page_table[(size_t)b * p.max_pages + pa];
              const int gb = two ? p.page_table[(size_t)b * p.max_pages + pa + 1] : 0;
              m.lo = 0;
              m.hi = min(kTK, min(kend, ctx) - pa * kPage);   // the split may end after page a
              const bool good = ga >= 0 && ga < p.num_pages && gb >= 0 && gb < p.num_pages;
              if (good) {
                sm.meta[s] = m;
                fence_proxy_async();
                mbar_arrive_expect_tx(bar, (two ? 2 : 1) * 2 * 2 * kPage * 128);
                for (int h = 0; h < 2; ++h) {
                  const uint32_t kd = smem_u32(sm.k[s] + h * kHalf);
                  const uint32_t vd = smem_u32(sm.v[s] + h * kHalf);
                  tma_load_4d(kd, &mk_pool, 64 * h, 0, g, ga, bar);
                  tma_load_4d(vd, &mv_pool, 64 * h, 0, g, ga, bar);
                  if (two) {
                    tma_load_4d(kd + kPage * 128, &mk_pool, 64 * h, 0, g, gb, bar);
                    tma_load_4d(vd + kPage * 128, &mv_pool, 64 * h, 0, g, gb, bar);
                  }
                }
              } else {
                flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
                m.flags |= kSkip;
                sm.meta[s] = m;
                mbar_arrive(bar);
              }
            } else {
              m.lo = max(kbeg, ctx) - ctx;
              m.hi = kend - ctx;
              sm.meta[s] = m;
              fence_proxy_async();
              mbar_arrive_expect_tx(bar, 2 * 2 * L * 128);
              for (int h = 0; h < 2; ++h) {
                tma_load_4d(smem_u32(sm.k[s] + h * kHalf), &mk_blk, 64 * h, g, 0, b, bar);
                tma_load_4d(smem_u32(sm.v[s] + h * kHalf), &mv_blk, 64 * h, g, 0, b, bar);
              }
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          stop = true;
          break;
        }
      }
    }
    if (lane == 0) {
      if (!stop) {                             // sentinel stage: no more work
        const uint32_t s = it % kStages, round = it / kStages;
        if (round > 0 && !mbar_wait(smem_u32(&sm.kv_empty[s]), (round - 1) & 1)) {
          fail();
        } else {
          sm.meta[s] = Meta{-1, 0, 0, kEnd};
          mbar_arrive(smem_u32(&sm.kv_full[s]));
          ++it;
        }
      }
      if (sm.abort_flag) {                     // drain copies that may be in flight
        const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0;
        for (uint32_t i = first; i < it; ++i)
          mbar_wait(smem_u32(&sm.kv_full[i % kStages]), (i / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc1 = idesc_bf16_f32(kTK, npad);
      const uint32_t idesc2 = idesc_bf16_f32(D, npad) | (1u << 15);   // A (V^T) is MN-major
      uint32_t nq = 0;
      Meta cur, nxt;
      auto meta_at = [&](uint32_t t, Meta &m) -> bool {
        const uint32_t s = t % kStages;
        if (!mbar_wait(smem_u32(&sm.kv_full[s]), (t / kStages) & 1)) return false;
        const volatile int *mv = reinterpret_cast<const volatile int *>(&sm.meta[s]);
        m.item = mv[0];
        m.lo = mv[1];
        m.hi = mv[2];
        m.flags = mv[3];
        return true;
      };
      // S^T(t) = K(t) . Q^T
      auto issue_s = [&](uint32_t t, const Meta &m) -> bool {
        const uint32_t s = t % kStages, sb = t & 1, use = t >> 1;
        if (m.flags & kFirst) {
          const uint32_t qb = nq & 1;
          if (!mbar_wait(smem_u32(&sm.q_full[qb]), (nq >> 1) & 1)) return false;
        }
        if (use > 0 && !mbar_wait(smem_u32(&sm.s_empty[sb]), (use - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t kb = smem_u32(sm.k[s]), qb = smem_u32(sm.q[nq & 1]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          const uint32_t qoff = (kk >> 2) * kQHalf + (kk & 3) * 32;
          mma_bf16(tmem + sb * 64, sw128_kmajor_desc(kb + off), sw128_kmajor_desc(qb + qoff),
                   idesc1, kk > 0);
        }
        mma_commit(smem_u32(&sm.s_full[sb]));
        return true;
      };
      bool ok = meta_at(0, cur);
      if (ok && !(cur.flags & kEnd)) ok = issue_s(0, cur);
      for (uint32_t t = 0; ok && !(cur.flags & kEnd); ++t) {
        // look ahead: S of tile t+1 overlaps the softmax of tile t
        ok = meta_at(t + 1, nxt);
        if (!ok) break;
        if (cur.flags & kLast) ++nq;             // the next tile starts a new item
        if (!(nxt.flags & kEnd)) {
          ok = issue_s(t + 1, nxt);
          if (!ok) break;
        }
        if (cur.flags & kLast) --nq;
        // O^T(t) = V^T(t) . P^T(t)
        const uint32_t s = t % kStages, sb = t & 1, use = t >> 1;
        if (!mbar_wait(smem_u32(&sm.p_full[sb]), use & 1) ||
            (use > 0 && !mbar_wait(smem_u32(&sm.o_empty[sb]), (use - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t vb = smem_u32(sm.v[s]), pb = smem_u32(sm.pm[sb]);
#pragma unroll
        for (int kk = 0; kk < kTK / 16; ++kk) {
          const uint32_t voff = kk * 16 * 128;
          const uint32_t poff = (kk >> 2) * kPAtom + (kk & 3) * 32;
          mma_bf16(tmem + 128 + sb * 64, sw128_mnmajor_desc(vb + voff),
                   sw128_kmajor_desc(pb + poff), idesc2, kk > 0);
        }
        mma_commit(smem_u32(&sm.o_full[sb]));
        mma_commit(smem_u32(&sm.kv_empty[s]));
        if (cur.flags & kLast) {
          mma_commit(smem_u32(&sm.q_empty[nq & 1]));
          ++nq;
        }
        cur = nxt;
      }
      if (!ok) fail();
      mma_commit(smem_u32(&sm.mma_done));
      mbar_wait(smem_u32(&sm.mma_done), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    // Every wait is followed by an OR-barrier over the four warps, so a timeout
    // in one warp makes all four leave together (no warp is left at a barrier).
    const int ew = warp - 2;                   // 0..3
    const int q4 = warp & 3;                   // TMEM sub-partition (lanes 32 q4 ..)
    const int tid = threadIdx.x - 64;          // 0..127
    const int row_lane = 32 * q4 + lane;       // key of S^T / head-dim index of O^T
    float o[64];
    int b = 0, g = 0, split = 0;
    auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {   // true: give up
      int ok = 1;
      if (lane == 0) ok = mbar_wait(smem_u32(bar), parity) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok && lane == 0) fail();
      return barrier_or(3, 128, !ok);
    };
    for (uint32_t t = 0;; ++t) {
      const uint32_t s = t % kStages, sb = t & 1, use = t >> 1;
      if (wait_all(&sm.kv_full[s], (t / kStages) & 1)) break;
      Meta m;
      {
        const volatile int *mv = reinterpret_cast<const volatile int *>(&sm.meta[s]);
        m.item = mv[0];
        m.lo = mv[1];
        m.hi = mv[2];
        m.flags = mv[3];
      }
      if (m.flags & kEnd) break;
      if (m.flags & kFirst) {
        split = m.item % p.num_splits;
        g = (m.item / p.num_splits) % p.hkv;
        b = m.item / (p.num_splits * p.hkv);
#pragma unroll
        for (int r = 0; r < 64; ++r) o[r] = 0.f;
        if (tid < 64) {
          sm.m_run[tid] = -INFINITY;
          sm.l_run[tid] = 0.f;
        }
      }
      const bool valid = !(m.flags & kSkip) && row_lane >= m.lo && row_lane < m.hi;
      // ---- S^T row of this lane's key
      if (wait_all(&sm.s_full[sb], use & 1)) break;
      tc_fence_after();
      float x[64];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (16 * c < npad) {
          float v[16];
          ld16(tmem + ((uint32_t)(32 * q4) << 16) + sb * 64 + 16 * c, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) x[16 * c + j] = valid ? v[j] : -INFINITY;
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) x[16 * c + j] = -INFINITY;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.s_empty[sb]));
      // ---- row maxima over the 128 keys
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (16 * c < npad) {
          float t16[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) t16[j] = x[16 * c + j];
          const float mx = bfly16<true>(t16, lane);
          if ((lane & 1) == 0) sm.red[ew][16 * c + (lane >> 1)] = mx;
        }
      }
      named_barrier(1, 128);
      if (tid < npad) {
        const float mt = fmaxf(fmaxf(sm.red[0][tid], sm.red[1][tid]),
                               fmaxf(sm.red[2][tid], sm.red[3][tid]));
        const float mo = sm.m_run[tid];
        const float mn = fmaxf(mo, mt);
        sm.corr[sb][tid] = (mo == -INFINITY || mn == -INFINITY) ? 0.f : exp2f((mo - mn) * sl2);
        sm.m_run[tid] = mn;
      }
      named_barrier(2, 128);
      // ---- P = exp(S - m) (bf16, row-major for MMA2), row sums
      uint8_t *pbuf = sm.pm[sb];
      const int katom = row_lane >> 6, kin = row_lane & 63;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (16 * c < npad) {
          float t16[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int r = 16 * c + j;
            const float mr = sm.m_run[r];
            const float pv = (valid && mr != -INFINITY) ? exp2f((x[r] - mr) * sl2) : 0.f;
            const __nv_bfloat16 pb16 = __float2bfloat16_rn(pv);
            t16[j] = __bfloat162float(pb16);     // sum exactly what MMA2 multiplies
            *reinterpret_cast<__nv_bfloat16 *>(pbuf + katom * kPAtom + r * 128 +
                                               (((kin >> 3) ^ (r & 7)) << 4) + (kin & 7) * 2) =
                pb16;
          }
          const float sx = bfly16<false>(t16, lane);
          if ((lane & 1) == 0) sm.red[ew][16 * c + (lane >> 1)] = sx;
        }
      }
      if (!valid) {                              // masked key: its V row must be finite
        uint8_t *vrow = sm.v[s] + row_lane * 128;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c16 = 0; c16 < 8; ++c16)
            *reinterpret_cast<int4 *>(vrow + h * kHalf + c16 * 16) = make_int4(0, 0, 0, 0);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.p_full[sb]));
      named_barrier(1, 128);
      if (tid < npad)
        sm.l_run[tid] = sm.l_run[tid] * sm.corr[sb][tid] + sm.red[0][tid] + sm.red[1][tid] +
                        sm.red[2][tid] + sm.red[3][tid];
      // ---- O = O * corr + O_t (this lane's head-dim element d = row_lane)
      if (wait_all(&sm.o_full[sb], use & 1)) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (16 * c < npad) {
          float v[16];
          ld16(tmem + ((uint32_t)(32 * q4) << 16) + 128 + sb * 64 + 16 * c, v);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            o[16 * c + j] = o[16 * c + j] * sm.corr[sb][16 * c + j] + v[j];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.o_empty[sb]));
      if (m.flags & kLast) {
        // the OR-barrier inside the o_full wait also published l_run of this tile
        const int d = row_lane;
#pragma unroll
        for (int r = 0; r < 64; ++r) {
          if (r < R) {
            const int qi = r / group, h = g * group + r % group;
            if (p.num_splits == 1) {
              const float l = sm.l_run[r];
              static_cast<__nv_bfloat16 *>(p.out)[(((size_t)b * L + qi) * p.hq + h) * D + d] =
                  __float2bfloat16_rn(l > 0.f ? o[r] / l : 0.f);
            } else {
              const size_t prow = (((size_t)b * p.hkv + g) * p.num_splits + split) * R + r;
              p.part_o[prow * D + d] = o[r];
              if (d == 0) {
                p.part_ml[prow * 2 + 0] = sm.m_run[r] * p.scale;   // natural-log units
                p.part_ml[prow * 2 + 1] = sm.l_run[r];
              }
            }
          }
        }
        named_barrier(2, 128);                   // m_run / l_run may be reset after this
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

bool preload_attention_tc5() { return preload_kernel(attn_tc5_kernel, true); }

bool attention_tc5_supported(const AttnParams &p) {
  if (p.dtype != BD_BF16 || p.head_dim != D || p.page_size != kPage) return false;
  const int R = p.block_len * (p.hq / p.hkv);
  if (R > 64 || p.block_len > 32) return false;
  if ((reinterpret_cast<uintptr_t>(p.q) & 15) != 0) return false;
  const DevInfo dv = dev_info();
  return dv.major >= 10 && tma_available();
}

bd_status attention_tc5(const AttnParams &p, cudaStream_t st) {
  const uint64_t eb = 2;
  const int group = p.hq / p.hkv;
  CUtensorMap mkp, mvp, mkb, mvb, mq;
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
  const uint64_t qdims[4] = {(uint64_t)D, (uint64_t)p.hq, (uint64_t)p.block_len,
                             (uint64_t)p.batch};
  const uint64_t qstr[3] = {D * eb, (uint64_t)p.hq * D * eb,
                            (uint64_t)p.block_len * p.hq * D * eb};
  const uint32_t qbox[4] = {64, (uint32_t)group, (uint32_t)p.block_len, 1};
  if (!tma_encode_bf16(&mkp, 4, p.k_pool, pdims, pstr, pbox) ||
      !tma_encode_bf16(&mvp, 4, p.v_pool, pdims, pstr, pbox) ||
      !tma_encode_bf16(&mkb, 4, p.k_blk, bdims, bstr, bbox) ||
      !tma_encode_bf16(&mvb, 4, p.v_blk, bdims, bstr, bbox) ||
      !tma_encode_bf16(&mq, 4, p.q, qdims, qstr, qbox))
    return BD_ERR_CUDA;
  const size_t smem = sizeof(Smem) + 1024;
  const int nitems = p.batch * p.hkv * p.num_splits;
  const int grid = std::max(1, std::min(nitems, std::max(dev_info().sms, 1)));
  const cudaError_t e = launch_pdl(attn_tc5_kernel, dim3(grid), dim3(kThreads), smem, st, mkp,
                                   mvp, mkb, mvb, mq, p);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

}  // namespace bd
