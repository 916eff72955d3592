// bf16 block attention on the 5th-generation tensor cores, two KV heads per
// tile so that the MMA's M dimension is 128 query rows.
//
// Same contract as the other attention kernels: the R = block_len * (Hq/Hkv)
// query rows of KV head g attend to head g's keys of [cache | block]
// ("Rethinking Document OCR as Inverse Rendering via Diffusion Decoding",
// paper.rainbus.top summary, method step 3).  Used for head_dim 128 and
// R = 64, the SDAR shapes (32-token blocks, two query heads per KV head).
//
// A tile is one 64-token page (or the block's own keys) of the KV heads
// 2p and 2p + 1.  Rows 0..63 of every operand belong to head 2p, rows
// 64..127 to head 2p + 1:
//   MMA1  S[row][key]  = Q[row][:] . K[key][:]     M = 128 rows, N = 128 keys, K = D
//   softmax (one thread per query row, no shuffles): the row's 64 keys of its
//         own head, running max kept in base-2 units and moved only when a new
//         maximum exceeds it by more than 8 (then O's row is rescaled in
//         TMEM), P = exp2(s - m) as bf16 written to TMEM (the thread's own
//         lane); the other head's 64 keys of P stay zero.  For a partial
//         tile the V rows of the keys outside its valid range are zeroed
//         first (they may hold anything, and 0 * NaN is NaN)
//   MMA2  O[row][d]   += P[row][key] . V[key][d]    M = 128, N = D, K = 128 keys
//         (P read from TMEM, V from shared memory MN-major); O stays in TMEM
//         for the whole piece
// The off-diagonal halves of MMA1 and MMA2 are wasted work; the tensor pipe
// has several times the throughput this HBM-bound loop needs.
//
// Work partition: the tiles of (sequence, KV-head pair) segments are laid
// end to end (a sequence with no masked position has none), each segment
// preceded by kPieceCost places that hold no tile (the cost of starting a
// piece); CTA c of the persistent grid takes the equal range
// [c T / G, (c + 1) T / G) of the T places.  Warp 0 of
// every CTA finds its range with a warp-wide scan of the sequences' tile
// counts, so no separate plan launch precedes the kernel.  A segment inside
// one CTA's range is written as the final output.  A segment cut by range
// boundaries leaves one partial per piece (O, and the running max and sum
// per row) in slot segment + CTA, and the CTA holding the segment's first
// tile records a merge job; attn_pair_merge_kernel, launched right after,
// merges each job's pieces, 32 rows per CTA with all loads of a row block in
// flight at once.
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0     TMA producer: Q of each piece, K and V of each tile (three stages)
//   warp 1     TMEM allocator and MMA issuer: MMA1 of a tile once its K/V
//              stage has landed, MMA2 of a tile once the softmax has written
//              its P, each as soon as it is ready (the softmax of t overlaps
//              MMA2 of t - 1, and a stage is freed without waiting for the
//              next tile)
//   warps 2-5  softmax, O rescale and the output of each piece
// Every wait is bounded; on expiry the kernel records BD_ERR_TIMEOUT, stops
// issuing, waits (bounded) for its copies and MMAs, frees TMEM and returns.
#include <math.h>

#include <algorithm>
#include <atomic>

#include "bd_attention.cuh"
#include "bd_common.cuh"
#include "bd_sm100.cuh"

namespace bd {

using namespace sm100;

namespace {

constexpr int D = 128;
constexpr int kRows = 128;                  // 2 heads x 64 query rows
constexpr int kPage = 64;
constexpr int kHalf = 128 * 128;            // 128 rows x 64 columns of bf16: 16 KB
constexpr int kHeadOff = 64 * 128;          // rows of the second head: +8 KB
constexpr int kThreads = 192;
constexpr int kStages = 3;
constexpr uint32_t kTmemCols = 512;         // S x2 (128 cols each), O (128), P x2 (64 each)
constexpr uint32_t kColO = 256;
constexpr uint32_t kColP = 384;             // P buffer b at kColP + 64 b: 128 keys as bf16 pairs
constexpr float kLazy = 8.f;                // max moves only beyond 2^8
constexpr int kFirst = 1, kLast = 2, kSkip = 4, kEnd = 8;
constexpr int kJobInts = 8;                 // merge job: seg (-1: none), c1, b, hp, T
constexpr int kMaxCluster = 16;             // cluster form: CTAs per segment
constexpr int kPieceCost = 3;               // tile-range form: tiles of budget a segment
                                            // start costs the CTA that takes it (a second
                                            // piece: its Q, the drain of O, a partial);
                                            // 0-4 measured, 3 best at 8 x 16384 keys
constexpr int kPieceStride = D + 4;         // cluster form: floats per piece row in shared
                                            // memory (a thread writing its own row has no
                                            // bank conflicts)

struct Meta {
  int item, lo, hi, flags, slot;
};

struct Smem {
  uint8_t q[2][kHalf];                      // two 64-column halves of D
  uint8_t k[kStages][2][kHalf];             // [stage][half]
  uint8_t v[kStages][2][kHalf];
  Meta meta[kStages];
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t q_full, q_empty;
  uint64_t s_full[2], s_empty[2], p_full[2];
  uint64_t o_done, o_empty;
  uint64_t mma_done;
  uint32_t tmem_base;
  volatile int abort_flag;
  int pid[32];                              // page ids of the first piece's first 32 pages
  volatile int active;                      // cluster form: the segment has output to write
};

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *m, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// Whether the phase with the given parity has completed (never suspends).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Whether CTA c's tile range is non-empty (T tiles over G CTAs).
__device__ __forceinline__ bool range_nonempty(int c, long long T, long long G) {
  return ((long long)c * T) / G < ((long long)(c + 1) * T) / G;
}

// MN-major operand in the 128-byte-swizzled layout a TMA load of [key][64 d]
// boxes writes: 128-byte rows of 64 consecutive d for one key, 8-key groups
// 1024 B apart, the next 64 d one half (16 KB) further.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(kHalf >> 4) << 16;        // leading byte offset: next 64 along N (d)
  d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: next 8 along K (keys)
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, bf16 inputs, fp32 accumulator; A is M
// rows (one per TMEM lane) of K bf16 values packed two per 32-bit column.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Zero the V rows of keys outside [lo, hi) in one stage (both heads, both
// halves of D; a key's row is 128 bytes in each of the four 8 KB blocks),
// shared by the 128 softmax threads (tid 0..127); then order the writes before
// MMA2 (async proxy) reads the stage.  Kept out of line: it runs for partial
// tiles only, and the softmax loop keeps its registers.
__device__ __noinline__ void zero_v_rows(uint8_t *vs, int lo, int hi, int tid) {
  const int nlo = max(0, lo), hi0 = max(nlo, min(64, hi));
  const int nz = nlo + (64 - hi0);               // keys [0, lo) and [hi, 64)
  for (int i = tid; i < nz * 32; i += 128) {
    const int j = i >> 5, c = i & 31;            // j-th zeroed key, 16-byte chunk of its 512 bytes
    const int r = j < nlo ? j : hi0 + (j - nlo);
    *reinterpret_cast<int4 *>(vs + (c >> 4) * kHalf + ((c >> 3) & 1) * kHeadOff + r * 128 +
                              (c & 7) * 16) = make_int4(0, 0, 0, 0);
  }
  fence_proxy_async();
}

template <bool kCluster>
__global__ void __launch_bounds__(kThreads, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap mk_pool,
                     const __grid_constant__ CUtensorMap mv_pool,
                     const __grid_constant__ CUtensorMap mk_blk,
                     const __grid_constant__ CUtensorMap mv_blk,
                     const __grid_constant__ CUtensorMap mq, const AttnParams p, int C, int Tm) {
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = p.hq / p.hkv;
  const int L = p.block_len;
  const int npairs = p.hkv / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.kv_full[s]), 1);
      mbar_init(smem_u32(&sm.kv_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&sm.s_full[s]), 1);
      mbar_init(smem_u32(&sm.s_empty[s]), 4);
      mbar_init(smem_u32(&sm.p_full[s]), 4);
    }
    mbar_init(smem_u32(&sm.q_full), 1);
    mbar_init(smem_u32(&sm.q_empty), 1);
    mbar_init(smem_u32(&sm.o_done), 1);
    mbar_init(smem_u32(&sm.o_empty), 4);
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
  // cluster form: this CTA's piece (a softmax thread's row keeps its O in TMEM)
  bool have_piece = false;
  float piece_m2 = -INFINITY, piece_l = 0.f;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // tiles of sequence b: its cached pages + the block's own keys, or none
    // when it has no masked position (or an invalid context)
    auto seq_tiles = [&](int b) -> int {
      bool active = true;
      if (p.tokens) {
        active = false;
        const int32_t *tk = p.tokens + (size_t)b * L;
        for (int i = 0; i < L; ++i) active |= tk[i] == BD_MASK;
      }
      const int ctx = p.ctx_len[b];
      if (ctx < 0 || ctx > p.max_ctx || ctx > p.max_pages * p.page_size) {
        if (active) flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
        return 0;
      }
      return active ? (ctx + kPage - 1) / kPage + 1 : 0;
    };
    const int c = blockIdx.x, G = gridDim.x;
    int T = 0, t_begin = 0, t_end = 0, b_first = -1, base_first = 0, tiles_first = 0;
    // cluster form: segment (b, hp) of this cluster, this CTA's tiles
    // [cu0, clast) of it, and the page ids of the first 32 of them in sm.pid
    int cb = 0, chp = 0, cctx = 0, cnpg = 0, cu0 = 0, clast = 0;
    // page ids of sequence pid_b's pages [pid_u0, pid_u0 + 32), loaded by the
    // whole warp in one latency (the first piece's pages)
    int pid_b = -1, pid_u0 = 0;
    if constexpr (kCluster) {
      const int rank = (int)cluster_ctarank();
      const int seg = blockIdx.x / C;
      cb = seg / npairs;
      chp = seg % npairs;
      cu0 = (int)((long long)rank * Tm / C);
      const int cu1 = (int)((long long)(rank + 1) * Tm / C);
      // one memory latency: the block's tokens, ctx and the range's page ids
      const int32_t *tk = p.tokens ? p.tokens + (size_t)cb * L : nullptr;
      const int32_t *prow = p.page_table + (size_t)cb * p.max_pages;
      const int tv = (tk && lane < L) ? tk[lane] : 0;
      cctx = p.ctx_len[cb];
      const int pid = (cu0 + lane < cu1 && cu0 + lane < p.max_pages) ? prow[cu0 + lane] : -1;
      const bool has = !tk || __any_sync(0xffffffffu, lane < L && tv == BD_MASK);
      const bool ctx_ok = cctx >= 0 && cctx <= p.max_ctx && cctx <= p.max_pages * p.page_size;
      if (has && !ctx_ok && rank == 0 && chp == 0 && lane == 0)
        flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
      const bool active = has && ctx_ok;
      cnpg = active ? (cctx + kPage - 1) / kPage : 0;
      clast = active ? min(cu1, cnpg + 1) : cu0;
      sm.pid[lane] = pid;
      pid_b = cb;
      pid_u0 = cu0;
      if (lane == 0) sm.active = active ? 1 : 0;
      __syncwarp();
    }
    // the plan: every segment of tl tiles takes tl + kPieceCost places on the
    // tile line (its first kPieceCost places hold no tile), T = all places;
    // this CTA's range [t_begin, t_end) of places and the sequence holding
    // t_begin (warp-wide passes over the sequences)
    auto vlen = [](int tl) { return tl > 0 ? tl + kPieceCost : 0; };
    if constexpr (!kCluster) {
    for (int b0 = 0; b0 < p.batch; b0 += 32) {
      int v = (b0 + lane < p.batch) ? npairs * vlen(seq_tiles(b0 + lane)) : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      T += v;
    }
    t_begin = (int)(((long long)c * T) / G);
    t_end = (int)(((long long)(c + 1) * T) / G);
    if (t_begin < t_end) {
      int carry = 0;
      for (int b0 = 0; b0 < p.batch && b_first < 0; b0 += 32) {
        const int b = b0 + lane;
        const int tl = b < p.batch ? seq_tiles(b) : 0;
        const int v = npairs * vlen(tl);
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += u;
        }
        const int excl = carry + inc - v;
        const unsigned hit = __ballot_sync(0xffffffffu, v > 0 && excl <= t_begin &&
                                                            t_begin < excl + v);
        if (hit) {
          const int src = __ffs(hit) - 1;
          b_first = __shfl_sync(0xffffffffu, b, src);
          base_first = __shfl_sync(0xffffffffu, excl, src);
          tiles_first = __shfl_sync(0xffffffffu, tl, src);
        }
        carry += __shfl_sync(0xffffffffu, inc, 31);
      }
    }
    if (b_first >= 0) {
      const int u0 = max(0, (t_begin - base_first) % vlen(tiles_first) - kPieceCost);
      const int u = u0 + lane;
      sm.pid[lane] = u < tiles_first - 1 ? p.page_table[(size_t)b_first * p.max_pages + u] : -1;
      pid_b = b_first;
      pid_u0 = u0;
      __syncwarp();
    }
    }
    uint32_t it = 0, pc = 0;
    bool stop = false;
    if (lane == 0) {
      // one piece: Q of the head pair, then tiles u in [u_first, u_last) of
      // sequence b (u < npg: cached page u; u == npg: the block's own keys
      // [blo, bhi)); false once stopped
      auto emit = [&](int b, int hp, int ctx, int npg, int u_first, int u_last, int blo,
                      int bhi, int seg, int slot) -> bool {
        const int32_t *prow = p.page_table + (size_t)b * p.max_pages;
        if (pc > 0 && !mbar_wait(smem_u32(&sm.q_empty), (pc - 1) & 1)) {
          fail();
          return false;
        }
        {
          const uint32_t bar = smem_u32(&sm.q_full);
          mbar_arrive_expect_tx(bar, 2 * 2 * L * group * 128);
          for (int hs = 0; hs < 2; ++hs)
            for (int h = 0; h < 2; ++h)
              tma_load_4d(smem_u32(sm.q[h] + hs * kHeadOff), &mq, 64 * h,
                          (2 * hp + hs) * group, 0, b, bar);
        }
        ++pc;
        for (int u = u_first; u < u_last; ++u, ++it) {
          const uint32_t s = it % kStages, round = it / kStages;
          // the page id is read before the wait, so the wait covers its latency
          // (the first piece's first 32 were loaded together up front)
          const int pg = u < npg ? ((b == pid_b && u >= pid_u0 && u - pid_u0 < 32)
                                        ? sm.pid[u - pid_u0]
                                        : prow[u])
                                 : -1;
          if (sm.abort_flag) return false;
          if (round > 0 && !mbar_wait(smem_u32(&sm.kv_empty[s]), (round - 1) & 1)) {
            fail();
            return false;
          }
          const uint32_t bar = smem_u32(&sm.kv_full[s]);
          Meta m;
          m.item = seg;
          m.slot = slot;
          m.lo = 0;
          m.flags = (u == u_first ? kFirst : 0) | (u == u_last - 1 ? kLast : 0);
          if (u < npg) {
            m.hi = min(kPage, ctx - u * kPage);
            if (pg >= 0 && pg < p.num_pages) {
              sm.meta[s] = m;
              fence_proxy_async();
              mbar_arrive_expect_tx(bar, 2 * 2 * 2 * kPage * 128);
              for (int hs = 0; hs < 2; ++hs)
                for (int h = 0; h < 2; ++h) {
                  tma_load_4d(smem_u32(sm.k[s][h] + hs * kHeadOff), &mk_pool, 64 * h, 0,
                              2 * hp + hs, pg, bar);
                  tma_load_4d(smem_u32(sm.v[s][h] + hs * kHeadOff), &mv_pool, 64 * h, 0,
                              2 * hp + hs, pg, bar);
                }
            } else {
              flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
              m.flags |= kSkip;
              m.hi = 0;
              sm.meta[s] = m;
              mbar_arrive(bar);
            }
          } else {
            m.lo = blo;
            m.hi = bhi;
            sm.meta[s] = m;
            fence_proxy_async();
            mbar_arrive_expect_tx(bar, 2 * 2 * 2 * L * 128);
            for (int hs = 0; hs < 2; ++hs)
              for (int h = 0; h < 2; ++h) {
                tma_load_4d(smem_u32(sm.k[s][h] + hs * kHeadOff), &mk_blk, 64 * h,
                            2 * hp + hs, 0, b, bar);
                tma_load_4d(smem_u32(sm.v[s][h] + hs * kHeadOff), &mv_blk, 64 * h,
                            2 * hp + hs, 0, b, bar);
              }
          }
        }
        return true;
      };
      if constexpr (kCluster) {
        if (cu0 < clast)
          stop = !emit(cb, chp, cctx, cnpg, cu0, clast, 0, L, cb * npairs + chp, -1);
      } else {
      int job[4] = {-1, 0, 0, 0};
      if (b_first >= 0) {
        int b = b_first, base = base_first, tiles = tiles_first;
        for (int t = t_begin; t < t_end && !stop;) {
          while (b < p.batch - 1 && t >= base + npairs * vlen(tiles)) {
            base += npairs * vlen(tiles);
            ++b;
            tiles = seq_tiles(b);
          }
          if (tiles <= 0 || t < base || t >= base + npairs * vlen(tiles)) {
            flag_error(p.dev_status, BD_ERR_DEVICE_CHECK);
            break;
          }
          const int vl = vlen(tiles);
          const int hp = (t - base) / vl;
          const int seg0 = base + hp * vl;        // the segment's first place
          const int vend = min(seg0 + vl, t_end);
          const int u0 = max(0, t - seg0 - kPieceCost), u1 = vend - seg0 - kPieceCost;
          if (u1 > u0) {                         // the range holds tiles [u0, u1) of it
            const int seg = b * npairs + hp;
            const bool whole = u0 == 0 && u1 == tiles;
            if (!whole && u0 == 0) {             // this CTA holds the cut segment's first
              job[0] = seg;                      // tile: it records the merge job
              job[1] = sk_cta_of(seg0 + kPieceCost + tiles - 1, T, G);
              job[2] = b;
              job[3] = hp;
            }
            stop = !emit(b, hp, p.ctx_len[b], tiles - 1, u0, u1, 0, L, seg, whole ? -1 : seg + c);
          }
          t = vend;
        }
      }
      {                                        // every CTA writes its entry
        int *jd = p.jobs + (size_t)c * kJobInts;
        jd[0] = job[0];
        jd[1] = job[1];
        jd[2] = job[2];
        jd[3] = job[3];
        jd[4] = T;
      }
      }
      if (!stop) {                             // sentinel stage: no more work
        const uint32_t s = it % kStages, round = it / kStages;
        if (round > 0 && !mbar_wait(smem_u32(&sm.kv_empty[s]), (round - 1) & 1)) {
          fail();
        } else {
          sm.meta[s] = Meta{-1, 0, 0, kEnd, -1};
          mbar_arrive(smem_u32(&sm.kv_full[s]));
          ++it;
        }
      }
      if (sm.abort_flag) {                     // wait (bounded) for copies in flight
        const uint32_t first = it > (uint32_t)kStages ? it - kStages : 0;
        for (uint32_t i = first; i < it; ++i)
          mbar_wait(smem_u32(&sm.kv_full[i % kStages]), (i / kStages) & 1);
        if (pc > 0) mbar_wait(smem_u32(&sm.q_full), (pc - 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // MMA1 of tile t needs the tile's K/V stage, MMA2 of tile t the softmax's P
    // of t.  Each is issued as soon as its inputs are ready (MMA1 first when
    // both are), so a stage is released once its own MMA2 is done, without
    // waiting for the next tile to land.
    if (lane == 0) {
      const uint32_t idesc1 = idesc_bf16_f32(kRows, kRows);
      const uint32_t idesc2 = idesc_bf16_f32(kRows, D) | (1u << 16);   // B (V) MN-major
      uint32_t pc = 0;                         // pieces whose Q was consumed
      uint32_t t1 = 0, t2 = 0;                 // next tile of MMA1, of MMA2 (t2 <= t1)
      // tiles t2..t1-1 awaiting MMA2, 8 bits each at bit 8 (t % 4): the meta
      // flags (bits 0-3), piece > 0 (bit 4), parity of piece - 1 (bit 5)
      uint32_t pend = 0;
      bool ended = false, o_init = false, ok = true;
      uint32_t idle = 0;
      uint64_t idle_t0 = 0;
      while (true) {
        bool progressed = false;
        if (!ended && t1 - t2 < 4) {
          const uint32_t st = t1 % kStages, s = t1 & 1;
          if (mbar_test_wait(smem_u32(&sm.kv_full[st]), (t1 / kStages) & 1)) {
            const volatile int *mv = reinterpret_cast<const volatile int *>(&sm.meta[st]);
            const int flags = mv[3];
            const bool first = (flags & kFirst) != 0;
            if (flags & kEnd) {
              ended = true;
              progressed = true;
            } else if ((!first || mbar_test_wait(smem_u32(&sm.q_full), pc & 1)) &&
                       (t1 < 2 || mbar_test_wait(smem_u32(&sm.s_empty[s]), ((t1 >> 1) - 1) & 1))) {
              tc_fence_after();
              if (!(flags & kSkip)) {
                const uint32_t qa = smem_u32(sm.q[0]);
                const uint32_t kb = smem_u32(sm.k[st][0]);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  mma_bf16(tmem + s * 128,
                           sw128_kmajor_desc(qa + (j >> 2) * kHalf + (j & 3) * 32),
                           sw128_kmajor_desc(kb + (j >> 2) * kHalf + (j & 3) * 32), idesc1,
                           j > 0 ? 1u : 0u);
              }
              mma_commit(smem_u32(&sm.s_full[s]));
              if (flags & kLast) mma_commit(smem_u32(&sm.q_empty));   // Q free after this MMA1
              {
                const uint32_t piece = first ? pc : (pc > 0 ? pc - 1 : 0);
                const uint32_t e = (uint32_t)(flags & 15) | (piece > 0 ? 16u : 0u) |
                                   (((piece - 1) & 1u) << 5);
                const uint32_t sh = 8 * (t1 & 3);
                pend = (pend & ~(0xFFu << sh)) | (e << sh);
              }
              if (first) ++pc;
              ++t1;
              progressed = true;
            }
          }
        }
        if (t2 < t1) {
          const uint32_t e = (pend >> (8 * (t2 & 3))) & 0xFFu;
          const int flags = (int)(e & 15);
          const bool first = (flags & kFirst) != 0;
          if (mbar_test_wait(smem_u32(&sm.p_full[t2 & 1]), (t2 >> 1) & 1) &&
              (!first || !(e & 16) || mbar_test_wait(smem_u32(&sm.o_empty), (e >> 5) & 1))) {
            if (first) o_init = false;
            tc_fence_after();
            if (!(flags & kSkip)) {
              const uint32_t pt = tmem + kColP + 64 * (t2 & 1);
              const uint32_t vb = smem_u32(sm.v[t2 % kStages][0]);
#pragma unroll
              for (int j = 0; j < 8; ++j)         // 16 keys = 8 TMEM columns per step
                mma_bf16_ts(tmem + kColO, pt + 8 * j, sw128_mnmajor_desc(vb + j * 2048),
                            idesc2, (o_init || j > 0) ? 1u : 0u);
              o_init = true;
            }
            mma_commit(smem_u32(&sm.kv_empty[t2 % kStages]));
            mma_commit(smem_u32(&sm.o_done));
            ++t2;
            progressed = true;
          }
        }
        if (ended && t2 == t1) {
          mma_commit(smem_u32(&sm.s_full[t1 & 1]));   // tells the softmax warps to stop
          break;
        }
        if (progressed) {
          idle = 0;
        } else if ((++idle & 63) == 0) {       // bounded: no progress for the wait limit
          const uint64_t now = globaltimer();
          if (idle == 64) {
            idle_t0 = now;
          } else if (sm.abort_flag || now - idle_t0 > kWaitLimitNs) {
            ok = false;
            break;
          }
        }
      }
      if (!ok) fail();
      // every MMA issued above has completed once mma_done fires
      mma_commit(smem_u32(&sm.mma_done));
      mbar_wait(smem_u32(&sm.mma_done), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int q = warp & 3;                    // TMEM lane quarter of this warp
    const int row = 32 * q + lane;             // query row of the tile (0..127)
    const int hs = row >> 6;                   // which head of the pair
    const int rr = row & 63;                   // row within its head: i * group + j
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
    const float sl2 = p.scale * 1.4426950408889634f;
    float m2 = -INFINITY, l = 0.f;
    uint32_t o_seen = 0;                       // o_done phases consumed
    {                                          // the other head's keys of P stay zero
      uint32_t z[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) z[j] = 0u;
#pragma unroll
      for (int b2 = 0; b2 < 2; ++b2)
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tmem_st_32x32b_x16(lane_base + kColP + 64 * b2 + 32 * (1 - hs) + 16 * c, z);
      tmem_st_wait();
    }
    bool ok = true;
    auto wait_o = [&](uint32_t tile) -> bool {   // MMA2 of `tile` has completed
      int w = 1;
      if (lane == 0) w = mbar_wait(smem_u32(&sm.o_done), tile & 1) ? 1 : 0;
      return __shfl_sync(0xffffffffu, w, 0) != 0;
    };
    for (uint32_t t = 0;; ++t) {
      const uint32_t s = t & 1;
      int w = 1;
      if (lane == 0) w = mbar_wait(smem_u32(&sm.s_full[s]), (t >> 1) & 1) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, w, 0)) {
        ok = false;
        break;
      }
      Meta m;
      {
        const volatile int *mv = reinterpret_cast<const volatile int *>(&sm.meta[t % kStages]);
        m.item = mv[0];
        m.lo = mv[1];
        m.hi = mv[2];
        m.flags = mv[3];
        m.slot = mv[4];
      }
      if (m.flags & kEnd) break;
      if (m.flags & kFirst) {
        m2 = -INFINITY;
        l = 0.f;
      }
      tc_fence_after();
      // this row's 64 scores (its own head's keys of the tile)
      float sc[64];
      {
        uint32_t r[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          tmem_ld_32x32b_x16(lane_base + s * 128 + hs * 64 + c * 16, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) sc[c * 16 + j] = __uint_as_float(r[j]) * sl2;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.s_empty[s]));
      const int lo = m.lo, hi = (m.flags & kSkip) ? 0 : m.hi;
      const bool none = hi <= lo;              // no valid key in the tile: P = 0
      if (lo > 0 || hi < 64) {                 // partial tile: masked keys score -inf
#pragma unroll
        for (int j = 0; j < 64; ++j)
          if (j < lo || j >= hi) sc[j] = -INFINITY;
      }
      float mt4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // four short chains
#pragma unroll
      for (int j = 0; j < 64; ++j) mt4[j & 3] = fmaxf(mt4[j & 3], sc[j]);
      const float mt = fmaxf(fmaxf(mt4[0], mt4[1]), fmaxf(mt4[2], mt4[3]));
      float factor = 1.f;
      if (mt > m2) {
        if (m2 == -INFINITY) {
          m2 = mt;                             // first keys of the piece: O not yet written
        } else if (mt > m2 + kLazy) {
          factor = fast_exp2(m2 - mt);
          l *= factor;
          m2 = mt;
        }
      }
      // P row as bf16 pairs (its own head's 64 keys = 32 TMEM columns)
      uint32_t pw[32];
      if (none) {
#pragma unroll
        for (int e = 0; e < 32; ++e) pw[e] = 0u;
      } else {                                 // exp2(-inf - m2) = 0 for the masked keys
        float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p0 = fast_exp2(sc[2 * e] - m2);
          const float p1 = fast_exp2(sc[2 * e + 1] - m2);
          sum4[e & 3] += p0 + p1;
          pw[e] = pack_bf16(p0, p1);
        }
        l += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
      }
      // MMA2 of the previous tile has to be complete before O is rescaled and
      // before this tile's P overwrites the buffer MMA2 of tile t - 2 read
      if (t >= 1 && o_seen < t) {
        if (!wait_o(t - 1)) {
          ok = false;
          break;
        }
        o_seen = t;
      }
      tc_fence_after();
      {
        uint32_t h16[16];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int j = 0; j < 16; ++j) h16[j] = pw[16 * c + j];
          tmem_st_32x32b_x16(lane_base + kColP + 64 * s + 32 * hs + 16 * c, h16);
        }
      }
      if (__any_sync(0xffffffffu, factor != 1.f)) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(lane_base + kColO + c * 16, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * factor);
          tmem_st_32x32b_x16(lane_base + kColO + c * 16, r);
        }
      }
      if (!(m.flags & kSkip) && (m.lo > 0 || m.hi < 64)) {
        // A masked key has P = 0, but 0 * NaN is NaN: the V rows of the tile's
        // keys outside [lo, hi) (pool rows past the context, the rows of the
        // block tile's stage that its copy did not write) are zeroed, both
        // heads and both halves of D, before MMA2 reads the stage.
        zero_v_rows(&sm.v[t % kStages][0][0], m.lo, m.hi, threadIdx.x - 64);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.p_full[s]));
      if (m.flags & kLast) {
        if (!wait_o(t)) {
          ok = false;
          break;
        }
        o_seen = t + 1;
        tc_fence_after();
        if (kCluster && C > 1) {               // O stays in TMEM for the cluster merge
          have_piece = true;
          piece_m2 = m2;
          piece_l = l;
        } else {
        const int b = m.item / npairs, hp = m.item % npairs;
        const int g = 2 * hp + hs;
        const int qi = rr / group, h = g * group + rr % group;
        if (m.slot < 0) {
          const float inv = l > 0.f ? 1.f / l : 0.f;
          __nv_bfloat16 *out =
              static_cast<__nv_bfloat16 *>(p.out) + (((size_t)b * L + qi) * p.hq + h) * D;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t r[16];
            tmem_ld_32x32b_x16(lane_base + kColO + c * 16, r);
            tmem_ld_wait();
            uint32_t w8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              w8[e] = pack_bf16(__uint_as_float(r[2 * e]) * inv, __uint_as_float(r[2 * e + 1]) * inv);
            *reinterpret_cast<uint4 *>(out + c * 16) = make_uint4(w8[0], w8[1], w8[2], w8[3]);
            *reinterpret_cast<uint4 *>(out + c * 16 + 8) = make_uint4(w8[4], w8[5], w8[6], w8[7]);
          }
        } else {
          const size_t prow = (size_t)m.slot * kRows + row;
          float *po = p.sk_o + prow * D;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t r[16];
            tmem_ld_32x32b_x16(lane_base + kColO + c * 16, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 4; ++e)
              *reinterpret_cast<uint4 *>(po + c * 16 + 4 * e) =
                  make_uint4(r[4 * e], r[4 * e + 1], r[4 * e + 2], r[4 * e + 3]);
          }
          p.sk_ml[prow * 2 + 0] = m2 * 0.6931471805599453f;   // natural-log units
          p.sk_ml[prow * 2 + 1] = l;
        }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.o_empty));
      }
    }
    if (!ok && lane == 0) fail();
  }

  tc_fence_before();
  __syncthreads();
  if (kCluster && C > 1) {
    // Every CTA publishes its piece in its own slot of the workspace: O
    // [128][D] fp32 at sk_o and (m in base-2 units, l) [128][2] at sk_ml (a
    // CTA without tiles publishes m = -inf, l = 0 and O = 0).  The softmax
    // threads stage their rows in the K stages (free now: every copy has
    // landed and every MMA has completed), and all threads copy the piece out
    // in coalesced 16-byte stores.  After a cluster barrier (release/acquire
    // at cluster scope) CTA rank r merges rows [r 128 / C, (r + 1) 128 / C) of
    // the C pieces from L2, one item (row, 8 columns) per thread with every
    // load of the item issued before any is used.
    float *c_o = reinterpret_cast<float *>(&sm.k[0][0][0]);
    float *c_ml = c_o + kRows * kPieceStride;
    if (warp >= 2) {
      const int row = 32 * (warp & 3) + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
      float4 *dst = reinterpret_cast<float4 *>(c_o + row * kPieceStride);
      if (__any_sync(0xffffffffu, have_piece)) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(lane_base + kColO + c * 16, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[4 * c + e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                                         __uint_as_float(r[4 * e + 2]),
                                         __uint_as_float(r[4 * e + 3]));
        }
      } else {
#pragma unroll
        for (int e = 0; e < D / 4; ++e) dst[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      *reinterpret_cast<float2 *>(c_ml + 2 * row) =
          have_piece ? make_float2(piece_m2, piece_l) : make_float2(-INFINITY, 0.f);
    }
    __syncthreads();
    {
      float4 *go = reinterpret_cast<float4 *>(p.sk_o + (size_t)blockIdx.x * kRows * D);
      for (int i = threadIdx.x; i < kRows * D / 4; i += kThreads)
        go[i] = *reinterpret_cast<const float4 *>(c_o + (i / (D / 4)) * kPieceStride +
                                                  4 * (i % (D / 4)));
      float2 *gml = reinterpret_cast<float2 *>(p.sk_ml + (size_t)blockIdx.x * kRows * 2);
      for (int i = threadIdx.x; i < kRows; i += kThreads)
        gml[i] = *reinterpret_cast<const float2 *>(c_ml + 2 * i);
    }
    cluster_sync();                            // every piece of the cluster is published
    if (sm.active) {
      const int rank = (int)cluster_ctarank();
      const int seg = blockIdx.x / C, b = seg / npairs, hp = seg % npairs;
      const size_t first = (size_t)blockIdx.x - rank;   // CTA of rank 0
      const int r_begin = rank * kRows / C, r_end = (rank + 1) * kRows / C;
      for (int item = threadIdx.x; item < (r_end - r_begin) * (D / 8); item += kThreads) {
        const int r = r_begin + item / (D / 8), q = item % (D / 8);
        float2 ml[kMaxCluster];
        float4 va[kMaxCluster], vb[kMaxCluster];
#pragma unroll
        for (int k = 0; k < kMaxCluster; ++k) {
          if (k < C) {
            const size_t prow = (first + k) * kRows + r;
            ml[k] = __ldcg(reinterpret_cast<const float2 *>(p.sk_ml + prow * 2));
            const float4 *src = reinterpret_cast<const float4 *>(p.sk_o + prow * D + 8 * q);
            va[k] = __ldcg(src);
            vb[k] = __ldcg(src + 1);
          }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMaxCluster; ++k)
          if (k < C) mx = fmaxf(mx, ml[k].x);
        float lsum = 0.f;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < kMaxCluster; ++k) {
          if (k < C && ml[k].x != -INFINITY) {
            const float w = exp2f(ml[k].x - mx);
            lsum = fmaf(w, ml[k].y, lsum);
            acc[0] = fmaf(w, va[k].x, acc[0]);
            acc[1] = fmaf(w, va[k].y, acc[1]);
            acc[2] = fmaf(w, va[k].z, acc[2]);
            acc[3] = fmaf(w, va[k].w, acc[3]);
            acc[4] = fmaf(w, vb[k].x, acc[4]);
            acc[5] = fmaf(w, vb[k].y, acc[5]);
            acc[6] = fmaf(w, vb[k].z, acc[6]);
            acc[7] = fmaf(w, vb[k].w, acc[7]);
          }
        }
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        const int g = 2 * hp + (r >> 6), rr = r & 63;
        const int qi = rr / group, h = g * group + rr % group;
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out) +
                             (((size_t)b * L + qi) * p.hq + h) * D + 8 * q;
        *reinterpret_cast<uint4 *>(out) =
            make_uint4(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv),
                       pack_bf16(acc[4] * inv, acc[5] * inv), pack_bf16(acc[6] * inv, acc[7] * inv));
      }
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge of the cut segments, one wave of CTAs.  Every CTA reads the whole
// job table (one entry per attention CTA) and compacts the active jobs; work
// item (job, r) covers rows [16 r, 16 r + 16) of the job's head pair, and CTA
// i takes items i, i + gridDim.x, ...  The pieces k of a job are the partials
// of CTAs c0 .. c1 with non-empty ranges, each an unnormalised O_k with its
// running max m_k and sum l_k per row:
//   M = max_k m_k,  S = sum_k l_k e^(m_k - M),  out = sum_k e^(m_k - M) O_k / S.
// All pieces' (m, l) and the first eight pieces' O rows are loaded before any
// is used; further pieces follow eight at a time.
constexpr int kMergeRows = 16;
constexpr int kMergeThreads = 256;
constexpr int kMergeGroup = 8;
constexpr int kMergeEpt = kMergeRows * (D / 4) / kMergeThreads;   // float4 per thread
constexpr int kMergeMaxPieces = 160;        // pieces of one segment (at most the grid)

__global__ void __launch_bounds__(kMergeThreads) attn_pair_merge_kernel(const AttnParams p) {
  __shared__ int slots[kMergeMaxPieces];
  __shared__ int active[kMergeMaxPieces];
  __shared__ int4 active_job[kMergeMaxPieces];
  __shared__ int warp_off[kMergeThreads / 32 + 1];
  __shared__ int npieces;
  __shared__ long long s_T;
  __shared__ float ml_m[kMergeMaxPieces][kMergeRows], ml_l[kMergeMaxPieces][kMergeRows];
  __shared__ float wts[kMergeMaxPieces][kMergeRows];
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int group = p.hq / p.hkv, L = p.block_len;
  const long long G = p.grid;                  // CTAs of the attention kernel (<= 160)
  // the active jobs in CTA order (the same list in every CTA); each entry is
  // read whole in this one pass
  int4 myjob = make_int4(-1, 0, 0, 0);
  int myT = 0;
  if (tid < G) {
    myjob = *reinterpret_cast<const int4 *>(p.jobs + (size_t)tid * kJobInts);   // seg, c1, b, hp
    myT = p.jobs[(size_t)tid * kJobInts + 4];
  }
  const bool has = tid < G && myjob.x >= 0;
  if (tid == 0) s_T = myT;                     // every entry holds the same T
  const unsigned bal = __ballot_sync(0xffffffffu, has);
  if (lane == 0) warp_off[warp + 1] = __popc(bal);
  __syncthreads();
  if (tid == 0) {
    warp_off[0] = 0;
    for (int w = 0; w < kMergeThreads / 32; ++w) warp_off[w + 1] += warp_off[w];
  }
  __syncthreads();
  if (has) {
    const int pos = warp_off[warp] + __popc(bal & ((1u << lane) - 1));
    active[pos] = tid;
    active_job[pos] = myjob;
  }
  const int nactive = warp_off[kMergeThreads / 32];
  const int items = nactive * (kRows / kMergeRows);
  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    __syncthreads();                           // active[] written; last item's data used
    const int j = active[item / (kRows / kMergeRows)];
    const int r0 = (item % (kRows / kMergeRows)) * kMergeRows;
    const int4 job = active_job[item / (kRows / kMergeRows)];   // seg, c1, b, hp
    const int seg = job.x, c1 = job.y, b = job.z, hp = job.w;
    const long long T = s_T;
    if (T >= G) {                              // the pieces: CTAs j..c1, every range
      const int n = min(c1 - j + 1, kMergeMaxPieces);   // non-empty
      for (int k = tid; k < n; k += kMergeThreads) slots[k] = seg + j + k;
      if (tid == 0) npieces = n;
    } else if (tid == 0) {                     // the CTAs j..c1 with tiles
      int n = 0;
      for (int cc = j; cc <= c1 && n < kMergeMaxPieces; ++cc)
        if (range_nonempty(cc, T, G)) slots[n++] = seg + cc;
      npieces = n;
    }
    __syncthreads();
    const int P = npieces;
    // every (piece, row) pair's running max and sum, one load each, all at once
    for (int i = tid; i < P * kMergeRows; i += kMergeThreads) {
      const int k = i / kMergeRows, rr = i % kMergeRows;
      const float2 ml = __ldcg(reinterpret_cast<const float2 *>(
          p.sk_ml + ((size_t)slots[k] * kRows + r0 + rr) * 2));
      ml_m[k][rr] = ml.x;
      ml_l[k][rr] = ml.y;
    }
    // the first group of pieces' O, issued before the statistics are used
    float4 acc[kMergeEpt];
#pragma unroll
    for (int i = 0; i < kMergeEpt; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 v[kMergeGroup][kMergeEpt];
    auto load_group = [&](int k0) {
#pragma unroll
      for (int k = 0; k < kMergeGroup; ++k)
#pragma unroll
        for (int i = 0; i < kMergeEpt; ++i)
          v[k][i] = k0 + k < P ? __ldcg(reinterpret_cast<const float4 *>(
                                     p.sk_o + ((size_t)slots[k0 + k] * kRows + r0) * D) +
                                 tid + kMergeThreads * i)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    load_group(0);
    __syncthreads();
    // weights w_k = e^(m_k - M) / S per row (one thread per row)
    if (tid < kMergeRows) {
      float M = -INFINITY;
      for (int k = 0; k < P; ++k) M = fmaxf(M, ml_m[k][tid]);
      float S = 0.f;
      for (int k = 0; k < P; ++k) {
        const float e = __expf(ml_m[k][tid] - M);
        wts[k][tid] = e;
        S = fmaf(ml_l[k][tid], e, S);
      }
      const float inv = S > 0.f ? 1.f / S : 0.f;
      for (int k = 0; k < P; ++k) wts[k][tid] *= inv;
    }
    __syncthreads();
    for (int k0 = 0; k0 < P; k0 += kMergeGroup) {
      if (k0 > 0) load_group(k0);
#pragma unroll
      for (int k = 0; k < kMergeGroup; ++k)
#pragma unroll
        for (int i = 0; i < kMergeEpt; ++i) {
          const float w = k0 + k < P ? wts[k0 + k][(tid + kMergeThreads * i) >> 5] : 0.f;
          acc[i].x = fmaf(v[k][i].x, w, acc[i].x);
          acc[i].y = fmaf(v[k][i].y, w, acc[i].y);
          acc[i].z = fmaf(v[k][i].z, w, acc[i].z);
          acc[i].w = fmaf(v[k][i].w, w, acc[i].w);
        }
    }
#pragma unroll
    for (int i = 0; i < kMergeEpt; ++i) {
      const int e = tid + kMergeThreads * i;
      const int r = r0 + (e >> 5), d4 = e & 31;
      const int g = 2 * hp + (r >> 6), rr = r & 63;
      const int qi = rr / group, h = g * group + rr % group;
      __nv_bfloat16 *out =
          static_cast<__nv_bfloat16 *>(p.out) + (((size_t)b * L + qi) * p.hq + h) * D + 4 * d4;
      *reinterpret_cast<uint2 *>(out) =
          make_uint2(pack_bf16(acc[i].x, acc[i].y), pack_bf16(acc[i].z, acc[i].w));
    }
  }
}

}  // namespace

bool preload_attention_pair() {
  return preload_kernel(attn_pair_kernel<false>, true) &&
         preload_kernel(attn_pair_kernel<true>, true) &&
         cudaFuncSetAttribute(attn_pair_kernel<true>,
                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
         preload_kernel(attn_pair_merge_kernel, false);
}

// Shapes the head-pair kernel takes (both forms).
static bool pair_shape_ok(const AttnParams &p) {
  if (p.dtype != BD_BF16 || p.head_dim != D || p.page_size != kPage) return false;
  if (p.hkv % 2 != 0 || p.hq % p.hkv != 0) return false;
  if (p.block_len * (p.hq / p.hkv) != 64) return false;
  if ((reinterpret_cast<uintptr_t>(p.out) & 7) != 0) return false;
  const DevInfo d = dev_info();
  return d.major >= 10 && tma_available();
}

bool attention_pair_supported(const AttnParams &p) {
  if (!pair_shape_ok(p)) return false;
  if (p.grid < 1 || p.grid > kMergeMaxPieces || !p.sk_o || !p.sk_ml || !p.jobs) return false;
  return (long long)p.batch * (p.hkv / 2) * (p.max_pages + 1) < (1LL << 30);
}

// TMA maps of one call: the pool as [page][Hkv][64][D], the block's keys as
// [B][L'][Hkv][D] (both in [64 keys][64 d] boxes) and Q as [B][L'][Hq][D]
// (boxes of the group's query heads for all L' positions).
static bool pair_maps(const AttnParams &p, CUtensorMap &mkp, CUtensorMap &mvp, CUtensorMap &mkb,
                      CUtensorMap &mvb, CUtensorMap &mq) {
  const uint64_t eb = 2;
  const int group = p.hq / p.hkv;
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
  return tma_encode_bf16(&mkp, 4, p.k_pool, pdims, pstr, pbox) &&
         tma_encode_bf16(&mvp, 4, p.v_pool, pdims, pstr, pbox) &&
         tma_encode_bf16(&mkb, 4, p.k_blk, bdims, bstr, bbox) &&
         tma_encode_bf16(&mvb, 4, p.v_blk, bdims, bstr, bbox) &&
         tma_encode_bf16(&mq, 4, p.q, qdims, qstr, qbox);
}

bd_status attention_pair(const AttnParams &p0, cudaStream_t st) {
  if (!attention_pair_supported(p0)) return BD_ERR_UNSUPPORTED;
  AttnParams p = p0;
  p.seg_heads = 2;
  CUtensorMap mkp, mvp, mkb, mvb, mq;
  if (!pair_maps(p, mkp, mvp, mkb, mvb, mq)) return BD_ERR_CUDA;
  const size_t smem = sizeof(Smem) + 1024;
  cudaError_t e = launch_pdl(attn_pair_kernel<false>, dim3(p.grid), dim3(kThreads), smem, st, mkp,
                             mvp, mkb, mvb, mq, p, 1, 0);
  count_launches(1);
  if (e != cudaSuccess) return BD_ERR_CUDA;
  e = launch_pdl(attn_pair_merge_kernel, dim3(2 * p.grid), dim3(kMergeThreads), 0, st, p);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

// Clusters of C CTAs of the cluster form that the device holds at once
// (cached per device and C; 0 when that size cannot be launched).
static int pair_active_clusters(int C, size_t smem) {
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
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, attn_pair_kernel<true>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  cache[dev][C].store(n);
  return n;
}

bool attention_pair_cluster_supported(const AttnParams &p) {
  return pair_shape_ok(p) && (long long)p.batch * (p.hkv / 2) <= (1LL << 24) && p.sk_o &&
         p.sk_ml && p.grid >= 1;
}

// Cluster form: one cluster of C CTAs per (sequence, KV-head pair) segment,
// C as large as the SMs allow, reduced until all clusters fit at once.
bd_status attention_pair_cluster(const AttnParams &p0, cudaStream_t st) {
  if (!attention_pair_cluster_supported(p0)) return BD_ERR_UNSUPPORTED;
  AttnParams p = p0;
  p.seg_heads = 2;
  const size_t smem = sizeof(Smem) + 1024;
  const long long segs = (long long)p.batch * (p.hkv / 2);
  const int sms = std::max(1, dev_info().sms);
  const int Tm = (p.max_ctx + kPage - 1) / kPage + 1;
  // pieces (C > 1) take one 128-row slot of sk_o / sk_ml per CTA: segs * C <= grid
  int C = (int)std::min<long long>(std::min(kMaxCluster, Tm),
                                   std::max(1LL, std::min<long long>(sms, p.grid) / segs));
  while (C > 1 && pair_active_clusters(C, smem) < std::min<long long>(segs, sms / C)) --C;
  if (pair_active_clusters(C, smem) < 1) return BD_ERR_UNSUPPORTED;
  CUtensorMap mkp, mvp, mkb, mvb, mq;
  if (!pair_maps(p, mkp, mvp, mkb, mvb, mq)) return BD_ERR_CUDA;
  const cudaError_t e =
      launch_pdl_cluster(attn_pair_kernel<true>, dim3((unsigned)(segs * C)), dim3(kThreads), smem,
                         st, dim3(C, 1, 1), mkp, mvp, mkb, mvb, mq, p, C, Tm);
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

}  // namespace bd
