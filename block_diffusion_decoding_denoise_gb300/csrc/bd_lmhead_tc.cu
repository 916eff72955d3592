// LM head + online-softmax confidence on the 5th-generation tensor cores.
//
// Computes, for every still-masked row r of the step (the compact row list
// written by conf_prep_kernel) and every vocabulary entry v,
//     l[r, v] = h[row r] . W[v]            (bf16 x bf16 -> fp32, tcgen05.mma)
// and reduces each row to the online-softmax state (max l, sum exp(l - max),
// lowest argmax) over the vocabulary slice this CTA owns, without writing a
// logit to memory ("Rethinking Document OCR as Inverse Rendering via
// Diffusion Decoding", paper.rainbus.top summary, method step 4: confidence of
// each masked prediction).
//
// Orientation ("swap AB"): the vocabulary is the MMA's M dimension (tiles of
// 128 entries of W, A operand) and the masked rows are N (up to 128 per pass,
// B operand), so a step with only a handful of masked rows still fills the
// 128-lane tensor-core tile and the kernel streams W at HBM speed.
//
// Work: units of (pass over up to 256 masked rows, tile of 128 vocabulary
// entries), laid out pass by pass and dealt round-robin to the persistent
// CTAs, so the shares differ by at most one unit over the whole call.  Calls
// of at most 128 positions run two CTAs per SM; wider calls run CTA pairs
// (clusters of two, tcgen05.mma.cta_group::2 with M = 256: each CTA stages its
// 128 rows of W and half of the pass's rows, the even CTA issues the MMAs).
// Warp roles (320 threads):
//   warp 0     TMA producer: per 64-wide K chunk, one 128x64 box of W and
//              16x64 boxes of the compacted masked rows of h (conf_prep_kernel
//              gathers them) into a ring of smem stages (128-byte swizzle),
//              completion on the stage's "full" mbarrier
//   warp 1     TMEM allocator and MMA issuer (one thread): 4 x (M128,N,K16)
//              per stage into one of two TMEM accumulators; tcgen05.commit
//              frees the stage and, after the last K chunk, hands the
//              accumulator to the epilogue
//   warps 2-9  epilogue, two warps per TMEM lane quarter taking alternate
//              16-column chunks: tcgen05.ld 32 lanes x 16 columns; a transposing
//              butterfly over the 32 lanes reduces the 16 columns to one
//              (max, sum-exp, argmax) each; a 4-warp merge through smem; a
//              running state per row kept in registers
// Sampling mode (kSample, bd_sample_commit): the epilogue scales the logits
// by 1 / temperature, adds per-entry Gumbel noise from the counter-based
// generator (one Philox block per vocabulary entry and group of eight
// positions, shared by consecutive masked rows of the same group) and keeps
// the online softmax of z together with the best perturbed key.
// Each CTA writes one partial state per row; conf_commit_kernel (launched
// right behind, with programmatic dependent launch) merges them and commits.
// Every mbarrier wait is bounded (1 s); on expiry the kernel records
// BD_ERR_TIMEOUT, drains what it issued, frees TMEM and returns.
#include <math.h>

#include <algorithm>

#include "bd_confidence.cuh"
#include "bd_sm100.cuh"

namespace bd {

using namespace sm100;

namespace {

constexpr int kEpiWarps = 8;               // epilogue warps: two per TMEM lane quarter
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kTileV = 128;                 // vocabulary entries per tile (MMA M)
constexpr int kKChunk = 64;                 // K elements per stage (128 bytes of bf16)
constexpr int kMaxN = 256;                  // masked rows per pass (MMA N), at most
constexpr int kNarrowN = 128;               // ... in the two-CTAs-per-SM configuration
constexpr int kNarrowSmem = 112 * 1024;     // shared memory per CTA there
constexpr int kBoxRows = 16;                // rows of the compact h copy per small TMA box
constexpr int kBigBoxRows = 64;             // ... per large box (whole 64-row groups)
constexpr int kABytes = kTileV * 128;       // 16 KB of W per stage
constexpr int kMaxStages = 12;
constexpr int kSmemLimit = 227 * 1024;

struct Ctrl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  volatile int32_t abort;
};

struct LmTcArgs {
  ConfParams p;
  int stages;
  int stage_bytes;
  int num_tiles;
  int nmax;       // masked rows per pass this launch can hold (multiple of 16; of 32
                  // for a CTA pair)
  int maxn;       // rows per pass: kMaxN, or kNarrowN with two CTAs per SM
  int brows;      // rows of h per stage in this CTA: nmax, or nmax / 2 for a CTA pair
  int big_boxes;  // 1: tmap_h64 (64-row boxes) is valid
  int red_off;    // smem offsets of the merge buffer, the row positions
  int pos_off;    // (sampling only) and Ctrl
  int ctrl_off;
};

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

// Merge the online-softmax state (bm, bs, bi) into (m, s, i): larger max
// wins, equal maxima keep the lower index, sums are rescaled to the new max.
__device__ __forceinline__ void merge_into(float &m, float &s, int &i, float bm, float bs,
                                           int bi) {
  const bool take = bm > m || (bm == m && bi < i);
  const float hi_m = take ? bm : m, lo_m = take ? m : bm;
  const float hi_s = take ? bs : s, lo_s = take ? s : bs;
  s = hi_s + (lo_s > 0.f ? lo_s * __expf(lo_m - hi_m) : 0.f);
  m = hi_m;
  i = take ? bi : i;
}

// One butterfly round over lanes (lane, lane ^ off): a lane keeps K of its 2K
// states (the lower half when its `off` bit is clear) and merges in the
// partner's copy of the same K columns.
template <int K>
__device__ __forceinline__ void bfly_round(float (&m)[16], float (&s)[16], int (&id)[16], int off,
                                           int lane) {
  const bool upper = (lane & off) != 0;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const float send_m = upper ? m[k] : m[K + k];
    const float send_s = upper ? s[k] : s[K + k];
    const int send_i = upper ? id[k] : id[K + k];
    float km = upper ? m[K + k] : m[k];
    float ks = upper ? s[K + k] : s[k];
    int ki = upper ? id[K + k] : id[k];
    const float rm = __shfl_xor_sync(0xffffffffu, send_m, off);
    const float rs = __shfl_xor_sync(0xffffffffu, send_s, off);
    const int ri = __shfl_xor_sync(0xffffffffu, send_i, off);
    merge_into(km, ks, ki, rm, rs, ri);
    m[k] = km;
    s[k] = ks;
    id[k] = ki;
  }
}

// bfly_round for sampling states (online softmax of z plus the best key).
template <int K>
__device__ __forceinline__ void bfly_round_s(float (&m)[16], float (&s)[16], float (&kb)[16],
                                             float (&zb)[16], int (&id)[16], int off, int lane) {
  const bool upper = (lane & off) != 0;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const float send_m = upper ? m[k] : m[K + k];
    const float send_s = upper ? s[k] : s[K + k];
    const float send_kb = upper ? kb[k] : kb[K + k];
    const float send_zb = upper ? zb[k] : zb[K + k];
    const int send_i = upper ? id[k] : id[K + k];
    float km = upper ? m[K + k] : m[k];
    float ks = upper ? s[K + k] : s[k];
    float kkb = upper ? kb[K + k] : kb[k];
    float kzb = upper ? zb[K + k] : zb[k];
    int ki = upper ? id[K + k] : id[k];
    const float rm = __shfl_xor_sync(0xffffffffu, send_m, off);
    const float rs = __shfl_xor_sync(0xffffffffu, send_s, off);
    const float rkb = __shfl_xor_sync(0xffffffffu, send_kb, off);
    const float rzb = __shfl_xor_sync(0xffffffffu, send_zb, off);
    const int ri = __shfl_xor_sync(0xffffffffu, send_i, off);
    merge_sample_into(km, ks, kkb, kzb, ki, rm, rs, rkb, rzb, ri);
    m[k] = km;
    s[k] = ks;
    kb[k] = kkb;
    zb[k] = kzb;
    id[k] = ki;
  }
}

// 16 accumulator columns (rows c0..c0+15 of the pass) x 32 vocabulary lanes
// -> one greedy state per column, written to red[c0 .. c0+15].
__device__ __forceinline__ void reduce_chunk(const uint32_t (&r)[16], int vbase, bool valid,
                                             int lane, MaxSumArg *red) {
  // a transposing butterfly: each round halves the columns a lane keeps and
  // merges the partner's copy of them
  float m[16], sx[16];
  int id[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    m[j] = valid ? __uint_as_float(r[j]) : -INFINITY;
    sx[j] = valid ? 1.f : 0.f;
    id[j] = valid ? vbase + lane : 0x7fffffff;
  }
  bfly_round<8>(m, sx, id, 16, lane);
  bfly_round<4>(m, sx, id, 8, lane);
  bfly_round<2>(m, sx, id, 4, lane);
  bfly_round<1>(m, sx, id, 2, lane);
  {
    const float om = __shfl_xor_sync(0xffffffffu, m[0], 1);
    const float os = __shfl_xor_sync(0xffffffffu, sx[0], 1);
    const int oi = __shfl_xor_sync(0xffffffffu, id[0], 1);
    merge_into(m[0], sx[0], id[0], om, os, oi);
  }
  // lanes 2k and 2k+1 now hold column k of the 32 lanes' reduction
  if ((lane & 1) == 0) red[lane >> 1] = MaxSumArg{m[0], sx[0], id[0]};
}

// Sampling variant: z = l * inv_temp, key = z + Gumbel(v, pos).  pos[j] is
// the position id of column j; consecutive columns of one group of eight
// positions reuse one Philox block (the group test is uniform across the warp).
__device__ __forceinline__ void reduce_chunk(const uint32_t (&r)[16], int vbase, bool valid,
                                             int lane, SampleState *red, const int *pos,
                                             float inv_temp, uint64_t seed, uint64_t offset) {
  float m[16], sx[16], kb[16], zb[16];
  int id[16];
  const int v = vbase + lane;
  uint64_t w[4] = {0ull, 0ull, 0ull, 0ull};
  int prev_g = -1;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int pj = pos[j];
    const int g = pj >> 3;
    if (g != prev_g) {
      philox4x64_10(static_cast<uint64_t>(v), static_cast<uint64_t>(g), offset, 0ull, seed, 0ull,
                    w);
      prev_g = g;
    }
    const float z = __uint_as_float(r[j]) * inv_temp;
    const float key = z + gumbel_of_field(philox_field(w, pj));
    m[j] = valid ? z : -INFINITY;
    sx[j] = valid ? 1.f : 0.f;
    kb[j] = valid ? key : -INFINITY;
    zb[j] = valid ? z : -INFINITY;
    id[j] = valid ? v : 0x7fffffff;
  }
  bfly_round_s<8>(m, sx, kb, zb, id, 16, lane);
  bfly_round_s<4>(m, sx, kb, zb, id, 8, lane);
  bfly_round_s<2>(m, sx, kb, zb, id, 4, lane);
  bfly_round_s<1>(m, sx, kb, zb, id, 2, lane);
  {
    const float om = __shfl_xor_sync(0xffffffffu, m[0], 1);
    const float os = __shfl_xor_sync(0xffffffffu, sx[0], 1);
    const float okb = __shfl_xor_sync(0xffffffffu, kb[0], 1);
    const float ozb = __shfl_xor_sync(0xffffffffu, zb[0], 1);
    const int oi = __shfl_xor_sync(0xffffffffu, id[0], 1);
    merge_sample_into(m[0], sx[0], kb[0], zb[0], id[0], om, os, okb, ozb, oi);
  }
  if ((lane & 1) == 0) red[lane >> 1] = SampleState{m[0], sx[0], kb[0], zb[0], id[0]};
}

template <bool kSample> struct StateOf { using type = MaxSumArg; };
template <> struct StateOf<true> { using type = SampleState; };

template <typename St> __device__ __forceinline__ St empty_state();
template <> __device__ __forceinline__ MaxSumArg empty_state<MaxSumArg>() {
  return MaxSumArg{-INFINITY, 0.f, 0x7fffffff};
}
template <> __device__ __forceinline__ SampleState empty_state<SampleState>() {
  return SampleState{-INFINITY, 0.f, -INFINITY, -INFINITY, 0x7fffffff};
}

// kPair: the CTAs of a two-CTA cluster share each tile of 256 vocabulary
// entries (128 per CTA) through tcgen05.mma.cta_group::2 (M = 256): each CTA
// stages its 128 rows of W and half of the pass's rows of h, so each SM
// brings in a third less operand data per FLOP; the even CTA issues the MMAs
// and the odd CTA's copies and epilogue report to the even CTA's barriers.
template <bool kSample, bool kPair>
__global__ void __launch_bounds__(kThreads, kPair ? 1 : 2)   // narrow calls: two CTAs per SM
    lmhead_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                     const __grid_constant__ CUtensorMap tmap_h,
                     const __grid_constant__ CUtensorMap tmap_h64, const LmTcArgs a) {
  using St = typename StateOf<kSample>::type;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Ctrl *ctrl = reinterpret_cast<Ctrl *>(smem + a.ctrl_off);
  St *red = reinterpret_cast<St *>(smem + a.red_off);   // [2][4][nmax]
  int *spos = reinterpret_cast<int *>(smem + a.pos_off);  // [nmax], sampling only
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const ConfParams &p = a.p;

  const int G = gridDim.x, cta = blockIdx.x;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;   // 0: issues the pair's MMAs
  // Work units: (pass over the rows, vocabulary tile) pairs laid out pass by
  // pass; a CTA (or a pair) takes units unit + i * units, so every CTA's share
  // differs by at most one unit over the whole call, not one per pass.  A
  // pair's tiles are pair tiles of two 128-entry tiles (2 pt + rank here).
  const int unit = kPair ? cta >> 1 : cta, units = kPair ? G >> 1 : G;
  const int unit_tiles = kPair ? (a.num_tiles + 1) >> 1 : a.num_tiles;
  const int KC = p.hidden / kKChunk;
  const int S = a.stages;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&ctrl->full[s]), 1);
      mbar_init(smem_u32(&ctrl->empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ctrl->tfull[i]), 1);
      mbar_init(smem_u32(&ctrl->tempty[i]), kPair ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(smem_u32(&ctrl->mma_done), 1);
    ctrl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_h);
    if (a.big_boxes) tma_prefetch_desc(&tmap_h64);
  }
  if (warp == 1) {
    if (kPair) {
      tmem_alloc_pair(smem_u32(&ctrl->tmem_base), 2u * a.maxn);   // two accumulators
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&ctrl->tmem_base), 2u * a.maxn);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // a pair: both CTAs' barriers exist before either CTA's copies or MMAs signal them
  if (kPair) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  // set-up above overlaps the previous kernel; the row list is read after it
  pdl_trigger();
  pdl_wait();
  int count;
  if (p.direct) {
    // all rows, or none once every position of the call is committed (each
    // warp reads the <= 64 tokens itself)
    const int n = p.batch * p.block_len;
    const bool m0 = lane < n && p.tokens[lane] == BD_MASK;
    const bool m1 = lane + 32 < n && p.tokens[lane + 32] == BD_MASK;
    count = __ballot_sync(0xffffffffu, m0 || m1) ? n : 0;
  } else {
    count = *p.ws.count;
  }
  const int MN = a.maxn;
  const int npass = count > 0 ? (count + MN - 1) / MN : 0;   // 0: nothing masked
  const int total_units = npass * unit_tiles;
  const int my_units = total_units > unit ? (total_units - unit + units - 1) / units : 0;
  auto unit_pass = [&](int i) { return (unit + i * units) / unit_tiles; };
  auto unit_tile = [&](int i) {
    const int tp = (unit + i * units) % unit_tiles;
    return kPair ? 2 * tp + (int)rank : tp;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t w_policy = l2_policy_evict_first();   // W is read once per step
    uint32_t it = 0;
    bool stop = false;
    for (int i = 0; i < my_units && !stop; ++i) {
      const int r0 = unit_pass(i) * MN;
      const int n = min(MN, count - r0);
      const int npad = kPair ? (n + 31) & ~31 : (n + 15) & ~15;
      const int nmine = kPair ? npad >> 1 : npad;          // rows of h this CTA stages
      const int rfirst = r0 + (int)rank * nmine;
      const uint32_t tx = kABytes + nmine * 128;
      {
        const int vt = unit_tile(i);
        for (int kc = 0; kc < KC; ++kc, ++it) {
          const uint32_t s = it % S, round = it / S;
          uint8_t *st = smem + (size_t)s * a.stage_bytes;
          int ok = 1;
          if (lane == 0) {
            if (ctrl->abort) ok = 0;
            else if (round > 0 && !mbar_wait_cluster(smem_u32(&ctrl->empty[s]), (round - 1) & 1)) {
              ok = 0;
              ctrl->abort = 1;
              flag_error(p.dev_status, BD_ERR_TIMEOUT);
            }
            if (ok) {
              // a pair's copies all count on the even CTA's barrier, which
              // expects both CTAs' bytes
              const uint32_t bar = kPair ? map_shared(smem_u32(&ctrl->full[s]), 0)
                                         : smem_u32(&ctrl->full[s]);
              if (rank == 0) mbar_arrive_expect_tx(smem_u32(&ctrl->full[s]), kPair ? 2 * tx : tx);
              if (kPair)
                tma_load_2d_pair_hint(smem_u32(st), &tmap_w, kc * kKChunk, vt * kTileV, bar,
                                      w_policy);
              else
                tma_load_2d_hint(smem_u32(st), &tmap_w, kc * kKChunk, vt * kTileV, bar, w_policy);
              // whole 64-row groups in one box each (fewer, larger copies), the
              // rest of the pass in 16-row boxes
              int r = 0;
              if (a.big_boxes)
                for (; r + kBigBoxRows <= nmine; r += kBigBoxRows) {
                  if (kPair)
                    tma_load_2d_pair(smem_u32(st + kABytes + r * 128), &tmap_h64, kc * kKChunk,
                                     rfirst + r, bar);
                  else
                    tma_load_2d(smem_u32(st + kABytes + r * 128), &tmap_h64, kc * kKChunk,
                                rfirst + r, bar);
                }
              for (; r < nmine; r += kBoxRows) {
                if (kPair)
                  tma_load_2d_pair(smem_u32(st + kABytes + r * 128), &tmap_h, kc * kKChunk,
                                   rfirst + r, bar);
                else
                  tma_load_2d(smem_u32(st + kABytes + r * 128), &tmap_h, kc * kKChunk, rfirst + r,
                              bar);
              }
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            stop = true;
            break;
          }
        }
      }
    }
    // on an abort, wait (bounded) for the copies this warp may still have in
    // flight; the odd CTA of a pair cannot observe its copies (they count on
    // the even CTA's barrier), so it waits a fixed 200 us, far beyond any copy
    if (stop && lane == 0) {
      if (rank == 0) {
        const uint32_t first = it > (uint32_t)S ? it - S : 0;
        for (uint32_t i = first; i < it; ++i)
          mbar_wait_cluster(smem_u32(&ctrl->full[i % S]), (i / S) & 1);
      } else {
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 200000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      uint32_t it = 0, tg = 0;
      bool stop = false;
      for (int i = 0; i < my_units && !stop; ++i, ++tg) {
        const int n = min(MN, count - unit_pass(i) * MN);
        const int npad = kPair ? (n + 31) & ~31 : (n + 15) & ~15;
        const uint32_t idesc = idesc_bf16_f32(kPair ? 2 * kTileV : kTileV, npad);
        {
          const uint32_t acc = tg & 1, use = tg >> 1;
          if (ctrl->abort ||
              (use > 0 && !mbar_wait_cluster(smem_u32(&ctrl->tempty[acc]), (use - 1) & 1))) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + acc * MN;
          for (int kc = 0; kc < KC; ++kc, ++it) {
            const uint32_t s = it % S, round = it / S;
            if (ctrl->abort || !mbar_wait_cluster(smem_u32(&ctrl->full[s]), round & 1)) {
              stop = true;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(smem + (size_t)s * a.stage_bytes);
            const uint32_t b_base = a_base + kABytes;
#pragma unroll
            for (int k = 0; k < kKChunk / 16; ++k) {
              if (kPair)
                mma_bf16_pair(d, sw128_kmajor_desc(a_base + k * 32),
                              sw128_kmajor_desc(b_base + k * 32), idesc, (kc | k) != 0);
              else
                mma_bf16(d, sw128_kmajor_desc(a_base + k * 32), sw128_kmajor_desc(b_base + k * 32),
                         idesc, (kc | k) != 0);
            }
            if (kPair) mma_commit_pair(smem_u32(&ctrl->empty[s]), 0x3);   // both CTAs' stage
            else mma_commit(smem_u32(&ctrl->empty[s]));
          }
          if (stop) break;
          if (kPair) mma_commit_pair(smem_u32(&ctrl->tfull[acc]), 0x3);
          else mma_commit(smem_u32(&ctrl->tfull[acc]));
        }
      }
      if (stop) {
        ctrl->abort = 1;
        flag_error(p.dev_status, BD_ERR_TIMEOUT);
      }
      // every MMA this thread issued has completed once mma_done fires
      if (kPair) mma_commit_pair(smem_u32(&ctrl->mma_done), 0x1);
      else mma_commit(smem_u32(&ctrl->mma_done));
      mbar_wait(smem_u32(&ctrl->mma_done), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;                 // 0..7
    const int q = warp & 3;                  // TMEM lane quarter this warp may read
    const int slot = ew & 3;                 // merge-buffer slot (one per lane quarter)
    const int half = ew >> 2;                // the two warps of a quarter split the chunks
    const int tid_e = threadIdx.x - 64;      // 0..255: row tid_e of the pass
    uint64_t draw = 0;                       // the step's draw counter (sampling)
    if constexpr (kSample) draw = *p.offset;
    St *part;
    if constexpr (kSample) part = p.ws.spartial;
    else part = p.ws.partial;
    // this CTA's state of every row of pass q: `run`, or an empty state for a
    // pass it has no tile of
    auto write_pass = [&](int q, const St &st) {
      const int n = min(MN, count - q * MN);
      if (tid_e < n) part[(size_t)(q * MN + tid_e) * G + cta] = st;   // [row][CTA]
    };
    bool stop = false;
    int cur = -1;                            // pass of the running state
    St run = empty_state<St>();
    for (int i = 0; i < my_units; ++i) {
      const int pass = unit_pass(i);
      const uint32_t tg = (uint32_t)i;
      const int r0 = pass * MN;
      const int n = min(MN, count - r0);
      const int npad = (n + 15) & ~15;
      if (pass != cur) {
        if (cur >= 0) write_pass(cur, run);
        for (int q = cur + 1; q < pass; ++q) write_pass(q, empty_state<St>());
        cur = pass;
        run = empty_state<St>();
        if constexpr (kSample) {
          // position ids of this pass's rows (the previous pass's readers have
          // all passed the per-tile barrier below)
          for (int j = tid_e; j < npad; j += kEpiThreads)
            spos[j] = j < n ? (p.direct ? r0 + j : p.ws.rows[r0 + j]) : 0;
          named_barrier(2, kEpiThreads);
        }
      }
      {
        const int vt = unit_tile(i);
        const uint32_t acc = tg & 1, use = tg >> 1;
        int ok = 1;
        if (lane == 0) ok = mbar_wait_cluster(smem_u32(&ctrl->tfull[acc]), use & 1) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) {
          tc_fence_after();
          const int vbase = vt * kTileV + 32 * q;
          const bool valid = vbase + lane < p.vocab;
          for (int c0 = 16 * half; c0 < npad; c0 += 32) {
            uint32_t r[16];
            tmem_ld_32x32b_x16(tmem + ((uint32_t)(32 * q) << 16) + acc * MN + c0, r);
            tmem_ld_wait();
            St *dst = red + ((tg & 1) * 4 + slot) * a.nmax + c0;
            if constexpr (kSample)
              reduce_chunk(r, vbase, valid, lane, dst, spos + c0, p.inv_temp, p.seed, draw);
            else
              reduce_chunk(r, vbase, valid, lane, dst);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {                     // the pair's MMAs wait on the even CTA's barrier
            if (kPair) mbar_arrive_cluster(map_shared(smem_u32(&ctrl->tempty[acc]), 0));
            else mbar_arrive(smem_u32(&ctrl->tempty[acc]));
          }
        } else {
          ctrl->abort = 1;
          if (lane == 0) flag_error(p.dev_status, BD_ERR_TIMEOUT);
        }
        if (barrier_or(1, kEpiThreads, !ok || ctrl->abort)) {
          stop = true;
          break;
        }
        if (tid_e < npad) {
#pragma unroll
          for (int w = 0; w < 4; ++w) run = merge(run, red[((tg & 1) * 4 + w) * a.nmax + tid_e]);
        }
      }
    }
    if (!stop) {
      if (cur >= 0) write_pass(cur, run);
      for (int q = cur + 1; q < npass; ++q) write_pass(q, empty_state<St>());
    }
  }

  tc_fence_before();
  __syncthreads();
  // a pair: the even CTA's MMAs (which read the odd CTA's shared memory and
  // write its tensor memory) and all cross-CTA arrivals are done
  if (kPair) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if (kPair) tmem_dealloc_pair(tmem, 2u * a.maxn);
    else tmem_dealloc(tmem, 2u * a.maxn);
  }
}

// 2-D bf16 tensor map over a row-major [outer][inner] matrix, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_in,
              uint32_t box_out) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t strides[1] = {inner * 2};
  const uint32_t box[2] = {box_in, box_out};
  return tma_encode_bf16(m, 2, base, dims, strides, box);
}

int num_tiles(int vocab) { return (vocab + kTileV - 1) / kTileV; }

// Calls with at most kNarrowN positions run two CTAs per SM (half the TMEM
// and at most kNarrowSmem of shared memory each): one CTA's epilogue and tile
// hand-offs overlap the other's stream, and the smaller CTAs become resident
// while the previous kernel drains.  Measured at 32 rows: 134.8 -> 130.7 us
// per call alone and 6740 -> 7690 committed tokens/s in the step graphs.
// (The kernel is compiled for two CTAs per SM: at most 102 registers a thread;
// the sampling epilogue fits in 96 without spills.)
bool narrow(int rows, bool) { return rows <= kNarrowN; }

// Wider calls run as CTA pairs (cta_group::2, one CTA per SM).
bool paired(int rows, bool sample) { return !narrow(rows, sample); }

void plan(const ConfParams &p, LmTcArgs &a, size_t *smem) {
  const int rows = p.batch * p.block_len;
  const bool nar = narrow(rows, p.sample != 0);
  const bool pair = paired(rows, p.sample != 0);
  a.maxn = nar ? kNarrowN : kMaxN;
  const int nmax = std::min(a.maxn, pair ? (rows + 31) & ~31 : (rows + 15) & ~15);
  a.nmax = nmax;
  a.brows = pair ? nmax / 2 : nmax;
  a.stage_bytes = (kABytes + a.brows * 128 + 1023) & ~1023;
  const int state = p.sample ? (int)sizeof(SampleState) : (int)sizeof(MaxSumArg);
  const int red = (2 * 4 * nmax * state + 1023) & ~1023;
  const int pos = p.sample ? ((nmax * 4 + 127) & ~127) : 0;
  const int fixed = red + pos + (int)sizeof(Ctrl) + 1024;
  const int budget = nar ? kNarrowSmem : kSmemLimit;
  a.stages = std::max(2, std::min(kMaxStages, (budget - fixed) / a.stage_bytes));
  a.red_off = a.stages * a.stage_bytes;
  a.pos_off = a.red_off + red;
  a.ctrl_off = a.pos_off + pos;
  *smem = (size_t)a.ctrl_off + sizeof(Ctrl) + 1024;
}

}  // namespace

bool preload_lmhead_tc() {
  return preload_kernel(lmhead_tc_kernel<false, false>, true) &&
         preload_kernel(lmhead_tc_kernel<true, false>, true) &&
         preload_kernel(lmhead_tc_kernel<false, true>, true) &&
         preload_kernel(lmhead_tc_kernel<true, true>, true);
}

bool lmhead_tc_supported(const ConfParams &p) {
  if (p.dtype != BD_BF16 || p.hidden % kKChunk != 0 || p.hidden < kKChunk) return false;
  if ((int64_t)p.batch * p.block_len > (1 << 20)) return false;
  const DevInfo d = dev_info();
  if (d.major < 10 || d.sms <= 0) return false;
  return tma_available();
}

int lmhead_tc_num_partials(int vocab, int rows, bool sample) {
  const DevInfo d = dev_info();
  if (paired(rows, sample))   // an even number of CTAs, at most one pair per pair tile
    return std::max(2, std::min(d.sms & ~1, 2 * ((num_tiles(vocab) + 1) / 2)));
  const int ctas = narrow(rows, sample) ? 2 * d.sms : d.sms;
  return std::max(1, std::min(ctas, num_tiles(vocab)));
}

bd_status lmhead_tc(const ConfParams &p, cudaStream_t st) {
  LmTcArgs a;
  a.p = p;
  a.num_tiles = num_tiles(p.vocab);
  size_t smem;
  plan(p, a, &smem);
  if (smem > (size_t)kSmemLimit) return BD_ERR_UNSUPPORTED;
  CUtensorMap mw, mh, mh64;
  const uint64_t rows = (uint64_t)p.batch * p.block_len;
  if (!make_map(&mw, p.w, p.hidden, p.vocab, kKChunk, kTileV)) return BD_ERR_CUDA;
  const void *hsrc = p.direct ? p.h : p.ws.hc;   // rows in place, or the compact copy
  if (!make_map(&mh, hsrc, p.hidden, rows, kKChunk, kBoxRows)) return BD_ERR_CUDA;
  // the large-box map only when a whole 64-row group can exist
  a.big_boxes = rows >= (uint64_t)kBigBoxRows ? 1 : 0;
  if (a.big_boxes) {
    if (!make_map(&mh64, hsrc, p.hidden, rows, kKChunk, kBigBoxRows)) return BD_ERR_CUDA;
  } else {
    mh64 = mh;
  }
  const int grid = p.ws.num_partials;
  cudaError_t e;
  if (paired((int)rows, p.sample != 0)) {
    if (grid < 2 || grid % 2 || grid > 2 * ((a.num_tiles + 1) / 2)) return BD_ERR_INVALID_ARG;
    e = p.sample ? launch_pdl_cluster(lmhead_tc_kernel<true, true>, dim3(grid), dim3(kThreads),
                                      smem, st, dim3(2, 1, 1), mw, mh, mh64, a)
                 : launch_pdl_cluster(lmhead_tc_kernel<false, true>, dim3(grid), dim3(kThreads),
                                      smem, st, dim3(2, 1, 1), mw, mh, mh64, a);
  } else {
    if (grid < 1 || grid > a.num_tiles) return BD_ERR_INVALID_ARG;
    e = p.sample ? launch_pdl(lmhead_tc_kernel<true, false>, dim3(grid), dim3(kThreads), smem, st,
                              mw, mh, mh64, a)
                 : launch_pdl(lmhead_tc_kernel<false, false>, dim3(grid), dim3(kThreads), smem, st,
                              mw, mh, mh64, a);
  }
  count_launches(1);
  return e == cudaSuccess ? BD_OK : BD_ERR_CUDA;
}

}  // namespace bd
