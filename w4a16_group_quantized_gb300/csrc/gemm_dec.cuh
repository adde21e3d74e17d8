// w4a16_gemm for decode batches (M <= 16 tokens): the dequantized weights go straight into the A
// fragments of register-operand tensor-core MMAs (mma.sync m16n8k16, fp16 or bf16 in, fp32
// accumulate), so a weight is read once as a 4-bit code, turned into fp16 / bf16 in registers and
// consumed there.
//
// Work split: the weight tiles (128 rows each) are dealt out to thread-block clusters round-robin
// (cluster q: tiles q, q + Q, ...). The C CTAs of a cluster split every tile along K: CTA rank k
// takes the 256-wide K stages [k KS / C, (k + 1) KS / C) of it. At the end of a tile the CTAs
// reduce-scatter their fp32 partial sums through distributed shared memory: CTA j sums rows
// [j 128 / C, (j + 1) 128 / C) of the tile over all C CTAs (in a fixed order: deterministic) and
// writes them to y. Nothing waits across clusters and nothing goes through global memory but the
// weights, x and y. The cluster size is chosen per layer for the best balance (a small layer's 16
// stages per tile split 4 ways keeps 128 SMs busy on a 32-tile layer; a large layer runs whole
// tiles, C = 1).
//
// Warp roles (one CTA per SM):
//   2 producer warps take the CTA's stages in turn; lane 0 issues per stage one tensor copy of x
//                   (128-byte swizzle, zero fill outside [M, K]) and two bulk copies: 16 KB of codes
//                   and the group records the stage needs. With `early` set the first stages' weight
//                   copies are issued before the wait for the previous grid (the weights are
//                   read-only), and x after it.
//   16 consumer warps in two sets of 8 that take the stages in turn (even / odd): warp (set, slab)
//                   covers weight rows 16 slab .. 16 slab + 15 over the stage's four 64-wide K blocks.
//                   Per block a lane loads two rows' 16-code spans (one 8-byte load each), the x
//                   fragments of its token (two 16-byte loads) and issues 4 k16 steps x NB8 MMAs.
//                   With g a multiple of 64 the MMAs run on the exact integers q - z and each group's
//                   fp32 partial is scaled by its s once per row; any other g rounds (q - z) * s to
//                   fp16 per 8 codes. At a tile's end a warp stores its rows' partial sums into the
//                   shared memory of the CTA that sums them and arrives on that CTA's barrier.
//   1 reducer warp sums the partial sums of this CTA's rows of each finished tile over the cluster
//                   and writes y, while the consumers already work on the next tile.
//
// The 16 k of one MMA step are taken in a permuted order, the same on both operands (the dot
// product is unchanged): lane (g, t) holds in step p the code pairs of its rows at k = 16t + 4p, +1 and
// 16t + 4p + 2, +3 of the block and the matching x pairs, which the tile layout of w4_repack and the
// 128-byte swizzle of x serve without shuffles, register moves or bank conflicts on x.
//
// This is Marlin's register-level dequant into MMA fragments (Marlin post) carried to sm_103a, with
// TMA/mbarrier staging, clusters and distributed shared memory for the split along K.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <climits>
#include <mutex>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace w4 {
namespace {

using namespace detail;

enum DecMode { kDecG256 = 0, kDecG128 = 1, kDecG64 = 2, kDecGen = 3 };

template <int NB8, int MODE>
struct DecCfg {
  static constexpr int BN = 8 * NB8;  // tokens per tile (the MMA's N, or two of them)
  // The CTA's K range of x stays in shared memory for the whole launch, M token rows of 128 bytes per
  // 64-wide K block (512 M bytes per stage), at most kXSlice stages and kDecXRegionBytes.
  static constexpr int kXSlice = kDecXSliceMax;
  static constexpr int kCodeBytes = kSB * kTileBytes;
  // group records a 256-wide stage can touch: one when g % 256 == 0, two for g == 128, five for other
  // multiples of 64, 33 for any g
  static constexpr int kMaxRecs = MODE == kDecGen ? kStageK / 8 + 1 : MODE == kDecG64 ? 5 : MODE == kDecG128 ? 2 : 1;
  static constexpr int kStageBytes = (kCodeBytes + kMaxRecs * kRecBytes + 127) / 128 * 128;
  static constexpr int kProducers = 2;
  static constexpr int kConsumers = 16;
  static constexpr int kSetWarps = kConsumers / 2;
  static constexpr int kReducerWarp = kProducers + kConsumers;
  static constexpr int kThreads = (kReducerWarp + 1) * 32;
  // Shared memory: [x: the CTA's K range][ring: S stages of weights][partial sums a CTA receives per tile:
  // [C senders][2 sets][M tokens][128 / C rows] fp32, 1 KB per token]. The ring takes whatever x leaves
  // (S even, for the two producers, at most kMaxStages).
  static constexpr int kSmemMax = 226 * 1024;
  static constexpr int kMaxStages = 14;
  static int x_bytes(int xslice, int m) { return xslice * kSB * m * 128; }
  static int ring_stages(int xslice, int m) {
    const int s = (kSmemMax - 1024 - 1024 * m - x_bytes(xslice, m)) / kStageBytes;
    return (s > kMaxStages ? kMaxStages : s) / 2 * 2;
  }
  static int smem_bytes(int xslice, int m, int stages) {
    return 1024 + x_bytes(xslice, m) + stages * kStageBytes + 1024 * m;
  }
  static_assert(kDecXRegionBytes + 4 * kStageBytes + 1024 * BN + 1024 <= kSmemMax, "shared memory");
  static_assert(NB8 == 1 || NB8 == 2, "tokens per tile");
};

template <int OFF>
__device__ __forceinline__ uint32_t lds16_at(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1+%2];" : "=h"(v) : "r"(addr), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint32_t lds8_at(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1+%2];" : "=h"(v) : "r"(addr), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint2 lds64_at(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2+%3];" : "=r"(v.x), "=r"(v.y) : "r"(addr), "n"(OFF));
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

template <int OFF>
__device__ __forceinline__ uint4 lds128_at(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4+%5];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr), "n"(OFF));
  return v;
}

// D (+)= A . B, m16n8k16, A row-major (4 regs), B column-major (2 regs), both fp16 or both bf16, fp32 D.
template <int DT>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if (DT == kDtypeBf16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The two rows a lane serves in a slab (rows R and R + 8): dequant constants and fp32 scales.
struct SlabConsts {
  GroupConsts a, b;
  float sa, sb;
};

// Integer path: zero points of rows R, R + 8 from the record at `rec`, scales as fp32.
template <int DT>
__device__ __forceinline__ SlabConsts slab_consts_int(uint32_t rec, uint32_t zero_off, uint32_t zero_shift,
                                                      uint32_t scale_off) {
  SlabConsts c;
  c.a = group_consts<DT>(0u, (lds8_at<0>(rec + zero_off) >> zero_shift) & 0xFu);
  c.b = group_consts<DT>(0u, (lds8_at<4>(rec + zero_off) >> zero_shift) & 0xFu);
  c.sa = scale_f32<DT>(lds16_at<0>(rec + scale_off));
  c.sb = scale_f32<DT>(lds16_at<16>(rec + scale_off));
  return c;
}

// Scaled path: the full constants (scale applied in the dequant) of rows R, R + 8.
template <int DT>
__device__ __forceinline__ SlabConsts slab_consts_scaled(uint32_t rec, uint32_t zero_off, uint32_t zero_shift,
                                                         uint32_t scale_off) {
  SlabConsts c;
  c.a = group_consts<DT>(lds16_at<0>(rec + scale_off), (lds8_at<0>(rec + zero_off) >> zero_shift) & 0xFu);
  c.b = group_consts<DT>(lds16_at<16>(rec + scale_off), (lds8_at<4>(rec + zero_off) >> zero_shift) & 0xFu);
  c.sa = c.sb = 1.0f;
  return c;
}

// One 64-wide K block BB of a lane's two rows: the 8-byte spans of rows R and R + 8 (words 2t, 2t + 1,
// k = 16t .. 16t + 15 of the block) dequantized into the A fragments of 4 k16 steps, times the x
// fragments of the block's tokens. Step p takes the pairs at k = 16t + 4p, +1 (the MMA's k-slot 2t, 2t + 1)
// and 16t + 4p + 2, +3 (slot 2t + 8, 2t + 9) on both operands: the x pair of a step is then two
// consecutive registers of one 16-byte load. SCALED: the constants of words 2t (c0) and 2t + 1 (c1)
// carry the scale; else both are the block's group and the MMAs see the exact q - z.
// The x operand of a lane: rows g and 8 + g of each block (the lane's tokens), present when < M.
struct XLane {
  uint32_t a, b;  // x of the lane's first row, chunks 2t and 2t + 1 (block 0 of the stage)
  uint32_t blk;   // bytes per 64-wide block (M rows of 128 bytes)
  bool v0, v1;    // token g, 8 + g < M
};

template <int NB8, int BB, bool SCALED, int DT>
__device__ __forceinline__ void dec_block(uint32_t codes, const XLane &xl, const SlabConsts &c0,
                                          const SlabConsts &c1, float (&acc)[NB8][4]) {
  const uint2 wr = lds64_at<BB * kTileBytes>(codes);        // row R: words 2t, 2t + 1
  const uint2 ws = lds64_at<BB * kTileBytes + 128>(codes);  // row R + 8
  uint32_t r0[4], r1[4], s0[4], s1[4];
  if (SCALED) {
    dequant_word<DT>(wr.x, c0.a, r0);
    dequant_word<DT>(wr.y, c1.a, r1);
    dequant_word<DT>(ws.x, c0.b, s0);
    dequant_word<DT>(ws.y, c1.b, s1);
  } else {
    dequant_word_int<DT>(wr.x, c0.a, r0);
    dequant_word_int<DT>(wr.y, c0.a, r1);
    dequant_word_int<DT>(ws.x, c0.b, s0);
    dequant_word_int<DT>(ws.y, c0.b, s1);
  }
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb) {
    // token g + 8 nb: x chunks 2t and 2t + 1 of the block (k 16t .. 16t + 15)
    uint4 x0 = make_uint4(0u, 0u, 0u, 0u), x1 = x0;
    if (nb == 0 ? xl.v0 : xl.v1) {
      x0 = nb == 0 ? lds128_at<0>(xl.a + BB * xl.blk) : lds128_at<1024>(xl.a + BB * xl.blk);
      x1 = nb == 0 ? lds128_at<0>(xl.b + BB * xl.blk) : lds128_at<1024>(xl.b + BB * xl.blk);
    }
    {
      const uint32_t a[4] = {r0[0], s0[0], r0[1], s0[1]};
      mma16816<DT>(acc[nb], a, x0.x, x0.y);
    }
    {
      const uint32_t a[4] = {r0[2], s0[2], r0[3], s0[3]};
      mma16816<DT>(acc[nb], a, x0.z, x0.w);
    }
    {
      const uint32_t a[4] = {r1[0], s1[0], r1[1], s1[1]};
      mma16816<DT>(acc[nb], a, x1.x, x1.y);
    }
    {
      const uint32_t a[4] = {r1[2], s1[2], r1[3], s1[3]};
      mma16816<DT>(acc[nb], a, x1.z, x1.w);
    }
  }
}

template <int NB8>
__device__ __forceinline__ void zero_acc(float (&acc)[NB8][4]) {
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[nb][c] = 0.0f;
}

// tot += s * acc per row (fragment elements 0, 1: row R; 2, 3: row R + 8).
template <int NB8>
__device__ __forceinline__ void flush_scaled(float (&tot)[NB8][4], const float (&acc)[NB8][4], const SlabConsts &c) {
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb) {
    tot[nb][0] = fmaf(c.sa, acc[nb][0], tot[nb][0]);
    tot[nb][1] = fmaf(c.sa, acc[nb][1], tot[nb][1]);
    tot[nb][2] = fmaf(c.sb, acc[nb][2], tot[nb][2]);
    tot[nb][3] = fmaf(c.sb, acc[nb][3], tot[nb][3]);
  }
}

// A lane's fixed offsets within a stage.
struct LaneOffsets {
  uint32_t code, x0, x1, xblk, zero, zero_shift, scale;
  bool xv0, xv1;
};

template <int BB>
__device__ __forceinline__ bool has_block(bool full, int nbk) {
  return full || BB < nbk;
}

// One stage (up to four K blocks from k0) of a lane's two rows, accumulated into tot. FULL: all four
// blocks present (the compiler then sees straight-line code); else nbk of them.
template <int NB8, int MODE, int CODEBYTES, bool FULL, int DT>
__device__ __forceinline__ void dec_stage(const DecParams &p, int G, uint32_t stage, uint32_t xstage,
                                          const LaneOffsets &o, int k0, int nbk, int t, float (&tot)[NB8][4]) {
  const uint32_t codes = stage + o.code;
  XLane xb;
  xb.a = xstage + o.x0;
  xb.b = xstage + o.x1;
  xb.blk = o.xblk;
  xb.v0 = o.xv0;
  xb.v1 = o.xv1;
  const uint32_t recs = stage + CODEBYTES;
  if (MODE == kDecG256) {  // g % 256 == 0: the whole stage lies in one group
    const SlabConsts c = slab_consts_int<DT>(recs, o.zero, o.zero_shift, o.scale);
    float acc[NB8][4];
    zero_acc<NB8>(acc);
    dec_block<NB8, 0, false, DT>(codes, xb, c, c, acc);
    if (has_block<1>(FULL, nbk)) dec_block<NB8, 1, false, DT>(codes, xb, c, c, acc);
    if (has_block<2>(FULL, nbk)) dec_block<NB8, 2, false, DT>(codes, xb, c, c, acc);
    if (has_block<3>(FULL, nbk)) dec_block<NB8, 3, false, DT>(codes, xb, c, c, acc);
    flush_scaled<NB8>(tot, acc, c);
  } else if (MODE == kDecG128) {  // g == 128: blocks 0, 1 in the stage's first group, 2, 3 in the next
    const SlabConsts c0 = slab_consts_int<DT>(recs, o.zero, o.zero_shift, o.scale);
    float acc[NB8][4];
    zero_acc<NB8>(acc);
    dec_block<NB8, 0, false, DT>(codes, xb, c0, c0, acc);
    if (has_block<1>(FULL, nbk)) dec_block<NB8, 1, false, DT>(codes, xb, c0, c0, acc);
    flush_scaled<NB8>(tot, acc, c0);
    if (has_block<2>(FULL, nbk)) {
      const SlabConsts c1 = slab_consts_int<DT>(recs + kRecBytes, o.zero, o.zero_shift, o.scale);
      float acc1[NB8][4];
      zero_acc<NB8>(acc1);
      dec_block<NB8, 2, false, DT>(codes, xb, c1, c1, acc1);
      if (has_block<3>(FULL, nbk)) dec_block<NB8, 3, false, DT>(codes, xb, c1, c1, acc1);
      flush_scaled<NB8>(tot, acc1, c1);
    }
  } else if (MODE == kDecG64) {  // g % 64 == 0: each block lies in one group, looked up per block
    const int jlo = p.gdiv.div(k0);
#pragma unroll
    for (int bb = 0; bb < kSB; ++bb) {
      if (FULL || bb < nbk) {
        const uint32_t rec = recs + (p.gdiv.div(k0 + bb * kTK) - jlo) * kRecBytes;
        const SlabConsts c = slab_consts_int<DT>(rec, o.zero, o.zero_shift, o.scale);
        float acc[NB8][4];
        zero_acc<NB8>(acc);
        if (bb == 0) dec_block<NB8, 0, false, DT>(codes, xb, c, c, acc);
        if (bb == 1) dec_block<NB8, 1, false, DT>(codes, xb, c, c, acc);
        if (bb == 2) dec_block<NB8, 2, false, DT>(codes, xb, c, c, acc);
        if (bb == 3) dec_block<NB8, 3, false, DT>(codes, xb, c, c, acc);
        flush_scaled<NB8>(tot, acc, c);
      }
    }
  } else {  // any g (a multiple of 8): (q - z) * s per 8 codes; codes past K (zero, against zero x) take
            // the last group's record, which the stage holds
    const int jlo = p.gdiv.div(k0);
#pragma unroll
    for (int bb = 0; bb < kSB; ++bb) {
      if (FULL || bb < nbk) {
        const int kw = k0 + bb * kTK + 16 * t;
        const uint32_t r0 = recs + (min(p.gdiv.div(kw), G - 1) - jlo) * kRecBytes;
        const uint32_t r1 = recs + (min(p.gdiv.div(kw + 8), G - 1) - jlo) * kRecBytes;
        const SlabConsts c0 = slab_consts_scaled<DT>(r0, o.zero, o.zero_shift, o.scale);
        const SlabConsts c1 = slab_consts_scaled<DT>(r1, o.zero, o.zero_shift, o.scale);
        if (bb == 0) dec_block<NB8, 0, true, DT>(codes, xb, c0, c1, tot);
        if (bb == 1) dec_block<NB8, 1, true, DT>(codes, xb, c0, c1, tot);
        if (bb == 2) dec_block<NB8, 2, true, DT>(codes, xb, c0, c1, tot);
        if (bb == 3) dec_block<NB8, 3, true, DT>(codes, xb, c0, c1, tot);
      }
    }
  }
}

// Waits with a caller-given limit; on timeout raises the CTA's abort flag and the error word.
__device__ __forceinline__ bool dec_wait(uint32_t bar, uint32_t parity, bool cluster_scope, const DecParams &p,
                                         volatile uint32_t *abort_flag) {
  const uint64_t t0 = clock_cycles();
  for (;;) {
    const bool done = cluster_scope ? mbar_try_wait_cluster(bar, parity, kSuspendNs)
                                    : mbar_try_wait_sleep(bar, parity, kSuspendNs);
    if (done) return true;
    if (*abort_flag) return false;
    if (clock_cycles() - t0 > p.wait_limit) {
      *abort_flag = 1u;
      atomicOr(p.err, kDevErrTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ bool dec_warp_wait(uint32_t bar, uint32_t parity, bool cluster_scope, const DecParams &p,
                                              volatile uint32_t *abort_flag) {
  const bool ok = dec_wait(bar, parity, cluster_scope, p, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// A cluster's tiles in order (q, q + Q, ... over the problems' tiles one after another) and this
// CTA's K stages [kb, ke) of each: rank k of C takes stages [k KS / C, (k + 1) KS / C) of its tile.
struct TileWalk {
  int T;       // global tile
  int pi;      // its problem
  int t;       // tile within the problem
  int kb, ke;  // this CTA's K stages of the tile
};

// Problem pi of the launch. A launch of one problem (MULTI false) reads entry 0 at a fixed place.
template <bool MULTI>
__device__ __forceinline__ const DecProblem &prob_at(const DecParams &p, int pi) {
  return p.prob[MULTI ? pi : 0];
}

__device__ __forceinline__ TileWalk walk_start() {
  TileWalk w;
  w.T = w.t = w.pi = 0;
  w.kb = w.ke = -1;
  return w;
}

template <bool MULTI>
__device__ __forceinline__ void walk_to(const DecParams &p, int rank, int T, TileWalk &w) {
  w.T = T;
  if (!MULTI) {  // one problem: the K range is the same for every tile
    w.t = T;
    if (w.ke < 0) {
      w.kb = rank * p.prob[0].KS / p.C;
      w.ke = (rank + 1) * p.prob[0].KS / p.C;
    }
    return;
  }
  while (w.pi + 1 < p.nprob && T >= p.prob[w.pi].tile_end) ++w.pi;  // tiles only move forward
  const DecProblem &pr = p.prob[w.pi];
  w.t = T - pr.tile_begin;
  w.kb = rank * pr.KS / p.C;
  w.ke = (rank + 1) * pr.KS / p.C;
}

// Where a tile's weight stages come from, kept in registers while the producers walk the tile.
struct StageSrc {
  const uint8_t *codes;  // the tile's first code block
  const uint8_t *meta;   // the tile's first group record
  int K, KS, nb_last;    // the problem's K, K stages and blocks in its last stage
};

// The same walk, one K stage at a time (the producers' view of the CTA's stage sequence).
template <bool MULTI>
struct StageWalk {
  TileWalk w;
  StageSrc src;
  int ks;
  __device__ __forceinline__ void load_src(const DecParams &p) {
    const DecProblem &pr = prob_at<MULTI>(p, w.pi);
    src.codes = pr.codes + static_cast<int64_t>(w.t) * pr.KB * kTileBytes;
    src.meta = pr.meta + static_cast<int64_t>(w.t) * pr.G * kRecBytes;
    src.K = pr.K;
    src.KS = pr.KS;
    src.nb_last = pr.KB - kSB * (pr.KS - 1);
  }
  __device__ __forceinline__ void init(const DecParams &p, int rank, int q) {
    w = walk_start();
    walk_to<MULTI>(p, rank, q, w);
    load_src(p);
    ks = w.kb;
  }
  __device__ __forceinline__ void advance(const DecParams &p, int rank, int n) {
    if (!MULTI) {  // the next tile of the one problem: Q tiles further on
      ks += n;
      while (ks >= w.ke) {
        ks -= w.ke - w.kb;
        w.T += p.Q;
        w.t += p.Q;
        src.codes += static_cast<int64_t>(p.Q) * p.prob[0].KB * kTileBytes;
        src.meta += static_cast<int64_t>(p.Q) * p.prob[0].G * kRecBytes;
      }
      return;
    }
    for (int j = 0; j < n; ++j) {
      if (++ks >= w.ke) {
        if (w.T + p.Q >= p.tiles) {  // past the cluster's last tile: stay put (never used)
          ks = w.ke;
          continue;
        }
        walk_to<MULTI>(p, rank, w.T + p.Q, w);
        load_src(p);
        ks = w.kb;
      }
    }
  }
};

// The CTA's K range [kb, kb + nstages) of problem pr's x, stage by stage (four 64-wide K blocks of M
// token rows each, 128-byte swizzle: 16-byte chunk c of row n of a block at n * 128 + (c ^ (n % 8)) * 16),
// loaded by the 512 consumer threads with zero-filling asynchronous copies (rows >= M and k >= K read
// nothing and land as zeros): thread `tid` copies chunk tid of each stage, then arrives on every stage
// barrier of the slice (xslice of them) once its copies so far have landed, so that each load moves
// every barrier by one phase.
__device__ __forceinline__ void load_x_slice(const DecParams &p, const DecProblem &pr, uint32_t xbase, int kb,
                                             int nstages, int tid, uint64_t *x_ready) {
  const int m = p.M;  // rows per block; 32 m <= 512 chunks per stage
  const int b = tid / (8 * m);
  const int n = (tid / 8) % m;
  const int c = tid % 8;
  const bool mine = tid < 32 * m;  // thread tid copies chunk tid of every stage
  const uint32_t dst0 = xbase + b * m * 128 + n * 128 + ((c ^ (n & 7)) << 4);
  for (int st = 0; st < p.xslice; ++st) {
    if (mine && st < nstages) {
      const int k = (kb + st) * kStageK + b * kTK + 8 * c;
      const bool valid = k < pr.K;
      const uint16_t *src = valid ? pr.x + static_cast<int64_t>(n) * pr.K + k : pr.x;
      cp_async16_zfill(dst0 + st * kSB * m * 128, src, valid ? 16u : 0u);
    }
    cp_async_mbar_arrive(smem_u32(&x_ready[st]));
  }
}

// Reducer: quads a lane holds in registers between the sum and the store (up to 128 quads of 4 rows:
// every cluster size at M <= 8, C >= 4 at M <= 16).
constexpr int kRedQuads = 4;

// Quad e (token e / (rows / 4), rows 4 (e % (rows / 4)) .. + 3 of the CTA's share) summed over the
// partials of the 2 C senders (by rank, set 0 then set 1 of each: a fixed order).
__device__ __forceinline__ float4 red_quad_sum(uint32_t red_base, int e, int M, int rows_per, int C) {
  const int tok = e / (rows_per / 4);
  const int lr = 4 * (e - tok * (rows_per / 4));
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k = 0; k < 2 * C; ++k) {
    const float4 a = lds128f(red_base + ((k * M + tok) * rows_per + lr) * 4);
    v.x += a.x;
    v.y += a.y;
    v.z += a.z;
    v.w += a.w;
  }
  return v;
}

// Quad e of the tile's outputs (rows n0 + 4 (e % (rows / 4)) ..) through the problem's epilogue: one
// store of 4 outputs (2 for silu * up), vectorized when aligned.
template <int DT>
__device__ __forceinline__ void red_quad_store(const DecProblem &pr, const Epi &epi, int n0, int e, int rows_per,
                                               float4 v) {
  const int tok = e / (rows_per / 4);
  const int n = n0 + 4 * (e - tok * (rows_per / 4));
  if (n >= pr.N) return;
  if (epi.kind == kEpiSiluMul) {  // rows n, n + 1: gate, up of output n / 2 (N even)
    uint16_t *dst = pr.y + static_cast<int64_t>(tok) * epi.ld + n / 2;
    const float h0 = silu_mul(v.x, v.y), h1 = silu_mul(v.z, v.w);
    if (n + 3 < pr.N && (reinterpret_cast<uintptr_t>(dst) & 3) == 0) {
      *reinterpret_cast<uint32_t *>(dst) = out_bits2<DT>(h0, h1);
    } else {
      dst[0] = out_bits<DT>(h0);
      if (n + 3 < pr.N) dst[1] = out_bits<DT>(h1);
    }
    return;
  }
  uint16_t *dst;
  if (epi.kind == kEpiNone) {
    dst = pr.y + static_cast<int64_t>(tok) * pr.N + n;
  } else {
    int ld;
    dst = epi_row(epi, pr.y, n, &ld) + static_cast<int64_t>(tok) * ld;
  }
  if (n + 3 < pr.N && (reinterpret_cast<uintptr_t>(dst) & 7) == 0) {
    *reinterpret_cast<uint2 *>(dst) = make_uint2(out_bits2<DT>(v.x, v.y), out_bits2<DT>(v.z, v.w));
  } else {
    const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (n + c < pr.N) dst[c] = out_bits<DT>(vv[c]);
  }
}

// The reducer frees the slots of the sender at `addr` (a release: the slots' reads come first).
__device__ __forceinline__ void red_free(uint32_t addr, int C) {
  if (C > 1)
    mbar_arrive_cluster(addr);
  else
    mbar_arrive(addr);
}

// The stage's weight copies: its code blocks and the group records it touches.
template <int kCodeBytes>
__device__ __forceinline__ void issue_stage(const StageSrc &src, const FastDiv &gdiv, int ks, uint32_t stage,
                                            uint32_t bar, uint64_t pol, bool arrive) {
  const int nb = ks == src.KS - 1 ? src.nb_last : kSB;
  const int k0 = ks * kStageK;
  const int jlo = gdiv.div(k0);
  const int nrec = gdiv.div(min(k0 + nb * kTK, src.K) - 1) - jlo + 1;
  const uint32_t bytes = nb * kTileBytes + nrec * kRecBytes;
  if (arrive)
    mbar_arrive_expect_tx(bar, bytes);
  else
    mbar_expect_tx(bar, bytes);
  bulk_g2s(stage, src.codes + static_cast<int64_t>(ks) * kSB * kTileBytes, nb * kTileBytes, bar, pol);
  bulk_g2s(stage + kCodeBytes, src.meta + static_cast<int64_t>(jlo) * kRecBytes, nrec * kRecBytes, bar, pol);
}

template <int NB8, int MODE, int DT, bool MULTI>
__global__ void __launch_bounds__(DecCfg<NB8, MODE>::kThreads, 1)
    w4a16_gemm_dec_kernel(const __grid_constant__ DecParams p) {
  using Cfg = DecCfg<NB8, MODE>;
  constexpr int SMAX = Cfg::kMaxStages;
  const int S = p.S;  // ring stages (even)
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[SMAX];   // the stage's weights landed
  __shared__ __align__(8) uint64_t x_ready[Cfg::kXSlice];  // x of the CTA's k-th stage of the current problem landed
  __shared__ __align__(8) uint64_t x_free;           // the 16 consumer warps are done with the loaded x
  __shared__ __align__(8) uint64_t empty_bar[SMAX];  // the 8 warps of the stage's set are done with it
  __shared__ __align__(8) uint64_t recv_bar;      // the 16 warps of the cluster whose rows this CTA sums stored them
  __shared__ __align__(8) uint64_t free_bar;      // every CTA of the cluster summed its rows of this CTA's last partials
  __shared__ uint32_t abort_sh;

  const uint32_t x_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t smem_base = x_base + p.xslice * kSB * p.M * 128;
  const uint32_t red_base = smem_base + S * Cfg::kStageBytes;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  volatile uint32_t *abort_flag = &abort_sh;

  const int C = p.C;
  const int rank = C > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int q = static_cast<int>(blockIdx.x) / C;
  const int rounds = q < p.tiles ? (p.tiles - 1 - q) / p.Q + 1 : 0;  // tiles q, q + Q, ...
  const int rows_per = kTN / C;  // rows of each tile this CTA sums

  // the barriers, one per thread (one thread initializing them all took about a microsecond)
  {
    const int t = threadIdx.x;
    bool did = true;
    if (t < S) {
      mbar_init(smem_u32(&full_bar[t]), 1);
      mbar_init(smem_u32(&empty_bar[t]), Cfg::kSetWarps);
    } else if (t >= 64 && t < 64 + p.xslice) {
      mbar_init(smem_u32(&x_ready[t - 64]), 32 * Cfg::kConsumers);
    } else if (t == 32) {
      mbar_init(smem_u32(&x_free), Cfg::kConsumers);
      mbar_init(smem_u32(&recv_bar), 1);  // the reducer's arrival; the partial sums come as transaction bytes
      mbar_init(smem_u32(&free_bar), C);   // one arrival from each CTA's reducer
      abort_sh = 0;
    } else {
      did = false;
    }
    if (did) fence_mbar_init();
  }
  __syncwarp();
  // every CTA's barriers are initialized before any CTA of the cluster arrives on them remotely
  if (C > 1)
    cluster_sync_all();
  else
    cta_sync_all();
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp < Cfg::kProducers) {
    // ---------------------------------------------------------------- producers
    const int pw = warp;
    int nst = 0;  // the CTA's stages over all its tiles
    {
      TileWalk w = walk_start();
      for (int r = 0; r < rounds; ++r) {
        walk_to<MULTI>(p, rank, q + r * p.Q, w);
        nst += w.ke - w.kb;  // >= 1: the planner keeps C <= KS of every problem
      }
    }
    const uint64_t pol = policy_evict_first();  // each weight byte is read once
    StageWalk<MULTI> sw;
    sw.init(p, rank, q);
    sw.advance(p, rank, pw);
    int i = pw;
    if (p.early) {
      // the first stages' weights before the previous grid is waited for: the packed weights are
      // read-only to every kernel of the stream (the caller states this)
      StageWalk<MULTI> se = sw;
      for (int ie = pw; ie < nst && ie < S; ie += 2) {
        if (lane == 0)
          issue_stage<Cfg::kCodeBytes>(se.src, p.gdiv, se.ks, smem_base + (ie % S) * Cfg::kStageBytes,
                                       smem_u32(&full_bar[ie % S]), pol, false);
        se.advance(p, rank, 2);
      }
      __syncwarp();
    } else if (pw == 0 && lane == 0 && nst > 0) {
      // ask L2 for the first tile's first stages while the previous grid finishes
      const DecProblem &pr = prob_at<MULTI>(p, sw.w.pi);
      const int t = sw.w.t, kb = sw.w.kb;
      const int n0 = min(sw.w.ke - kb, S);
      const int blocks = min((kb + n0) * kSB, pr.KB) - kb * kSB;
      bulk_prefetch_l2(pr.codes + (static_cast<int64_t>(t) * pr.KB + kb * kSB) * kTileBytes, blocks * kTileBytes);
      const int jlo = p.gdiv.div(kb * kStageK);
      const int jhi = p.gdiv.div(min((kb + n0) * kStageK, pr.K) - 1);
      bulk_prefetch_l2(pr.meta + (static_cast<int64_t>(t) * pr.G + jlo) * kRecBytes, (jhi - jlo + 1) * kRecBytes);
    }
    griddep_wait();  // x may be the previous grid's output
    int s = pw, ph = 0;  // slot i % S and the parity of its use i / S (S even: this warp's slots have its parity)
    for (; i < nst; i += 2) {
      if (i >= S && !dec_warp_wait(smem_u32(&empty_bar[s]), ph ^ 1, false, p, abort_flag)) break;
      if (lane == 0) {
        const uint32_t bar = smem_u32(&full_bar[s]);
        if (p.early && i < S)
          mbar_arrive(bar);  // the weights are on their way since before the wait
        else
          issue_stage<Cfg::kCodeBytes>(sw.src, p.gdiv, sw.ks, smem_base + s * Cfg::kStageBytes, bar, pol, true);
      }
      __syncwarp();
      sw.advance(p, rank, 2);
      s += 2;
      if (s >= S) {
        s -= S;
        ph ^= 1;
      }
    }
    if (*abort_flag && lane == 0) {
      // let every weight copy this warp issued land before the CTA's shared memory goes away. Early
      // weight copies of stages the loop never reached have no arrival yet: arrive, so that their phase
      // completes once the bytes are in.
      int last = i;
      if (p.early) {
        for (int j = i; j < min(nst, S); j += 2) mbar_arrive(smem_u32(&full_bar[j % S]));
        const int n_early = min(nst, S);
        if (n_early > pw) last = max(last, pw + (n_early - 1 - pw) / 2 * 2 + 2);
      }
      for (int j = last - 2; j >= 0 && j >= last - S; j -= 2) drain_wait(smem_u32(&full_bar[j % S]), (j / S) & 1);
    }
  } else if (warp < Cfg::kReducerWarp) {
    // ---------------------------------------------------------------- consumers
    const int cw = warp - Cfg::kProducers;
    const int qs = (cw >> 2) & 1;                // stage set: stages of parity qs (two warps per SMSP)
    const int sl = (cw & 3) | ((cw >> 3) << 2);  // slab: rows 16 sl .. 16 sl + 15
    const int g = lane >> 2;
    const int t = lane & 3;
    const int R = 16 * sl + g;  // rows R and R + 8
    LaneOffsets o;
    o.code = (t >> 1) * 2048 + R * 16 + 8 * (t & 1);
    // x of token g, 128-byte swizzle: chunk c of row n sits at n * 128 + (c ^ (n % 8)) * 16 (n % 8 == g)
    o.x0 = 128 * g + (((2 * t) ^ g) << 4);
    o.x1 = 128 * g + (((2 * t + 1) ^ g) << 4);
    o.xblk = p.M * 128;
    o.xv0 = g < p.M;
    o.xv1 = 8 + g < p.M;
    o.zero = 256 + R / 2;  // (+4 for row R + 8)
    o.zero_shift = 4 * (R & 1);
    o.scale = 2 * R;  // (+16 for row R + 8)
    // this warp's rows are summed by cluster CTA j, into slot [rank][qs][token][row - j rows_per]
    const int j = (16 * sl) / rows_per;
    const uint32_t slot_local = red_base + ((rank * 2 + qs) * p.M * rows_per + (R - j * rows_per)) * 4;
    const uint32_t slot = mapa_shared(slot_local, j);
    const uint32_t recv_at_j = mapa_shared(smem_u32(&recv_bar), j);

    griddep_wait();  // x may be the previous grid's output
    float tot[NB8][4];
    zero_acc<NB8>(tot);
    bool ok = true;
    int s = qs, ph = 0;  // slot and use parity of the set's next stage (its stages are i = qs, qs + 2, ...)
    int ibase = 0;       // the CTA's stage index of the round's first stage
    int xloads = 0;      // x slices loaded so far
    int r_load = 0;      // the round of the last load
    const uint16_t *x_cur = nullptr;  // the loaded slice: problem x, its K and the first stage
    int xk_cur = -1, xkb_cur = -1;
    TileWalk w = walk_start();
    if (!MULTI) {  // one problem: the same K range of x for every tile, loaded once
      walk_to<MULTI>(p, rank, q, w);
      if (rounds > 0) {
        load_x_slice(p, p.prob[0], x_base, w.kb, w.ke - w.kb, cw * 32 + lane, x_ready);
        xloads = 1;
      }
    }
    for (int r = 0; r < rounds && ok; ++r) {
      walk_to<MULTI>(p, rank, q + r * p.Q, w);
      const DecProblem &pr = prob_at<MULTI>(p, w.pi);
      const int per_tile = w.ke - w.kb;
      const int G = pr.G;
      const int ks_short = pr.KB % kSB ? pr.KS - 1 : -1;  // the problem's short last stage, if any
      const int nb_short = pr.KB - kSB * (pr.KS - 1);
      // x of the CTA's K range of this tile, unless it is already loaded (tiles of one problem, or of
      // problems that share x and K)
      if (MULTI && (pr.x != x_cur || pr.K != xk_cur || w.kb != xkb_cur)) {
        if (xloads > 0) {
          // every phase of the last load is complete before the next load arrives on any barrier, and
          // every consumer warp is done with the loaded slice before it is overwritten
          for (int st = 0; st < p.xslice && ok; ++st)
            ok = dec_warp_wait(smem_u32(&x_ready[st]), (xloads - 1) & 1, false, p, abort_flag);
          if (!ok) break;
          if (lane == 0) mbar_arrive(smem_u32(&x_free));
          ok = dec_warp_wait(smem_u32(&x_free), (xloads - 1) & 1, false, p, abort_flag);
          if (!ok) break;
        }
        load_x_slice(p, pr, x_base, w.kb, per_tile, cw * 32 + lane, x_ready);
        ++xloads;
        r_load = r;
        x_cur = pr.x;
        xk_cur = pr.K;
        xkb_cur = w.kb;
      }
      // a warp meets each x stage of a load first in one of the two rounds after it (its set's stage
      // parity flips between rounds when per_tile is odd and repeats after that)
      const bool xchk = r - r_load < 2;
      const uint32_t xpar = (xloads - 1) & 1;
      // this set's stages of the round: local stage indices ibase .. ibase + per_tile - 1 of parity qs
      for (int i = ibase + ((qs - ibase) & 1); i < ibase + per_tile; i += 2) {
        const int st = i - ibase;  // the stage's place in the CTA's K range (its x slot)
        if (xchk) {
          ok = dec_warp_wait(smem_u32(&x_ready[st]), xpar, false, p, abort_flag);
          if (!ok) break;
        }
        ok = dec_warp_wait(smem_u32(&full_bar[s]), ph, false, p, abort_flag);
        if (!ok) break;
        const uint32_t stage = smem_base + s * Cfg::kStageBytes;
        const uint32_t xstage = x_base + st * kSB * o.xblk;
        const int ks = w.kb + st;
        if (ks != ks_short)
          dec_stage<NB8, MODE, Cfg::kCodeBytes, true, DT>(p, G, stage, xstage, o, ks * kStageK, kSB, t, tot);
        else
          dec_stage<NB8, MODE, Cfg::kCodeBytes, false, DT>(p, G, stage, xstage, o, ks * kStageK, nb_short, t, tot);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
        s += 2;
        if (s >= S) {
          s -= S;
          ph ^= 1;
        }
      }
      if (!ok) break;
      ibase += per_tile;
      // the tile's partial sums of rows R, R + 8 go to CTA j once it has summed the previous tile's
      if (r > 0 && !dec_warp_wait(smem_u32(&free_bar), (r - 1) & 1, true, p, abort_flag)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int nb = 0; nb < NB8; ++nb) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int tok = 8 * nb + 2 * t + (c & 1);
          if (tok < p.M) st_async_f32(slot + (tok * rows_per + 8 * (c >> 1)) * 4, tot[nb][c], recv_at_j);
        }
      }
      zero_acc<NB8>(tot);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // (after an abort) no copy of this thread in flight
  } else {
    // ---------------------------------------------------------------- reducer
    // sums this CTA's rows [rank rows_per, (rank + 1) rows_per) of each finished tile over the cluster's
    // CTAs and both sets, in a fixed order, and writes them through the problem's epilogue; then frees
    // the slots of every sender
    griddep_wait();  // y may still be in use by the previous grid
    const uint32_t free_at_lane = C > 1 && lane < C ? mapa_shared(smem_u32(&free_bar), lane) : smem_u32(&free_bar);
    TileWalk w = walk_start();
    for (int r = 0; r < rounds; ++r) {
      walk_to<MULTI>(p, rank, q + r * p.Q, w);
      const DecProblem &pr = prob_at<MULTI>(p, w.pi);
      const Epi epi = pr.epi;
      // this tile's partial sums for this CTA's rows: 2 sets x C CTAs x rows_per rows x M tokens x 4 bytes
      if (lane == 0) mbar_arrive_expect_tx(smem_u32(&recv_bar), 1024u * p.M + p.test_extra_tx);
      if (!dec_warp_wait(smem_u32(&recv_bar), r & 1, true, p, abort_flag)) break;
      const int n0 = w.t * kTN + rank * rows_per;
      // 4 consecutive rows per lane and step: one 16-byte load per partial, one store of 4 outputs
      // (2 for silu * up), vectorized when aligned
      const int quads = p.M * (rows_per / 4);
      const bool more = r + 1 < rounds;
      if (more && quads <= 32 * kRedQuads) {
        // a later tile follows: every quad of the lane is summed into registers first, so that the
        // release that frees the senders' slots orders only shared-memory reads, then the stores
        float4 v[kRedQuads];
#pragma unroll
        for (int j = 0; j < kRedQuads; ++j)
          if (lane + 32 * j < quads) v[j] = red_quad_sum(red_base, lane + 32 * j, p.M, rows_per, C);
        __syncwarp();
        if (lane < C) red_free(free_at_lane, C);
#pragma unroll
        for (int j = 0; j < kRedQuads; ++j)
          if (lane + 32 * j < quads) red_quad_store<DT>(pr, epi, n0, lane + 32 * j, rows_per, v[j]);
        continue;
      }
      if (epi.kind == kEpiNone) {
        const bool vec_y = pr.N % 4 == 0 && (reinterpret_cast<uintptr_t>(pr.y) & 7) == 0;
#pragma unroll 2
        for (int e = lane; e < quads; e += 32) {
          const int tok = e / (rows_per / 4);
          const int lr = 4 * (e - tok * (rows_per / 4));
          const float4 v = red_quad_sum(red_base, e, p.M, rows_per, C);
          uint16_t *dst = pr.y + static_cast<int64_t>(tok) * pr.N + n0 + lr;
          if (vec_y && n0 + lr + 3 < pr.N) {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(out_bits2<DT>(v.x, v.y), out_bits2<DT>(v.z, v.w));
          } else {
            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int c = 0; c < 4; ++c)
              if (n0 + lr + c < pr.N) dst[c] = out_bits<DT>(vv[c]);
          }
        }
      } else {
#pragma unroll 2
        for (int e = lane; e < quads; e += 32)
          red_quad_store<DT>(pr, epi, n0, e, rows_per, red_quad_sum(red_base, e, p.M, rows_per, C));
      }
      // the slots are freed for the next tile; after the last tile no CTA waits for that
      __syncwarp();
      if (lane < C && more) red_free(free_at_lane, C);
    }
  }
  // no CTA leaves while another CTA of the cluster may still store into its shared memory. On the
  // normal path every such access has completed by now: a CTA's partial sums are counted by the
  // receiver's barrier before its reducer finishes, and every arrival on a CTA's free_bar was waited
  // for by that CTA's consumers (the last tile's is not made), so the barrier needs no release
  // ordering. After an abort, remote arrivals may not have been waited for: release them.
  __syncwarp();
  if (C > 1) {
    if (__shfl_sync(0xFFFFFFFFu, *abort_flag, 0))
      cluster_sync_all();
    else
      cluster_sync_all_relaxed();
  } else {
    cta_sync_all();
  }
}

// Largest number of clusters of `c` CTAs of this kernel that can be resident at once on the current
// device (cached per device).
template <int NB8, int MODE, int DT, bool MULTI>
int max_clusters(int c, int dev) {
  using Cfg = DecCfg<NB8, MODE>;
  static int cache[64][4] = {};
  static std::mutex mu;
  const int ci = c == 1 ? 0 : c == 2 ? 1 : c == 4 ? 2 : 3;
  std::lock_guard<std::mutex> lk(mu);
  if (dev >= 0 && dev < 64 && cache[dev][ci] > 0) return cache[dev][ci];
  auto kern = w4a16_gemm_dec_kernel<NB8, MODE, DT, MULTI>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(c * 64));
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemMax;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(c);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();
    n = 0;
  }
  if (dev >= 0 && dev < 64 && n > 0) cache[dev][ci] = n;
  return n;
}

template <int NB8, int MODE, int DT, bool MULTI>
cudaError_t launch_dec_t(DecParams p, int clusters, int cluster, cudaStream_t stream) {
  using Cfg = DecCfg<NB8, MODE>;
  auto kern = w4a16_gemm_dec_kernel<NB8, MODE, DT, MULTI>;
  static uint64_t done_mask = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 64 || !(done_mask & (1ull << dev))) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemMax);
      if (e != cudaSuccess) return e;
      if (dev < 64) done_mask |= 1ull << dev;
    }
  }
  // choose the cluster size (CTAs splitting each tile along K) and the number of clusters: the fewest
  // stages for the busiest CTA (at most ceil(NT / Q) tiles of each problem per cluster), then the
  // smaller cluster
  auto fits = [&](int c) {
    for (int i = 0; i < p.nprob; ++i)
      if (c > p.prob[i].KS || !dec_x_fits(p.prob[i].KS, c, p.M)) return false;  // x range would not fit
    return true;
  };
  int C = cluster, Q = clusters;
  if (C <= 0) {
    int64_t best = INT64_MAX;
    for (int c : {1, 2, 4, 8}) {
      if (!fits(c)) continue;
      const int mc = max_clusters<NB8, MODE, DT, MULTI>(c, dev);
      if (mc < 1) continue;
      const int qq = std::min(Q > 0 ? Q : mc, p.tiles);
      int64_t work = 0;
      for (int i = 0; i < p.nprob; ++i)
        work += static_cast<int64_t>((p.prob[i].NT + qq - 1) / qq) * ((p.prob[i].KS + c - 1) / c);
      if (work < best) {
        best = work;
        C = c;
      }
    }
    if (C <= 0) C = 1;
  }
  if (!fits(C)) return cudaErrorInvalidValue;
  if (Q <= 0) {
    const int mc = max_clusters<NB8, MODE, DT, MULTI>(C, dev);
    Q = mc > 0 ? mc : 1;
  }
  Q = std::min(Q, p.tiles);
  p.C = C;
  p.Q = Q;
  p.xslice = 0;  // the longest K range of a CTA, in stages
  for (int i = 0; i < p.nprob; ++i) p.xslice = std::max(p.xslice, (p.prob[i].KS + C - 1) / C);
  p.S = Cfg::ring_stages(p.xslice, p.M);
  if (p.S < 4) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(Q * C));
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(Cfg::smem_bytes(p.xslice, p.M, p.S));
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(C);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int NB8, int DT, bool MULTI>
cudaError_t launch_dec_nb(const DecParams &p, int clusters, int cluster, cudaStream_t stream) {
  if (p.g % 256 == 0) return launch_dec_t<NB8, kDecG256, DT, MULTI>(p, clusters, cluster, stream);
  if (p.g == 128) return launch_dec_t<NB8, kDecG128, DT, MULTI>(p, clusters, cluster, stream);
  if (p.g % 64 == 0) return launch_dec_t<NB8, kDecG64, DT, MULTI>(p, clusters, cluster, stream);
  return launch_dec_t<NB8, kDecGen, DT, MULTI>(p, clusters, cluster, stream);
}

// The decode kernel for value type DT: tokens per tile (nb8 x 8) and one or several problems.
template <int DT>
cudaError_t launch_dec_dt(const DecParams &p, int nb8, int clusters, int cluster, cudaStream_t stream) {
  const bool multi = p.nprob > 1;
  if (nb8 == 1)
    return multi ? launch_dec_nb<1, DT, true>(p, clusters, cluster, stream)
                 : launch_dec_nb<1, DT, false>(p, clusters, cluster, stream);
  if (nb8 == 2)
    return multi ? launch_dec_nb<2, DT, true>(p, clusters, cluster, stream)
                 : launch_dec_nb<2, DT, false>(p, clusters, cluster, stream);
  return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace w4
