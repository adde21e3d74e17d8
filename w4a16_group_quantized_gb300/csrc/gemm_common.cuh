// Pieces shared by the GEMM kernels: the schedule (persistent CTAs over (tile, K stage) units:
// stream-K ranges or round-robin whole tiles), the one-tile weight-stream producer, the fp16 / bf16
// dequant of 8 packed codes, bounded waits and the owner-reduces finish of tiles cut between CTAs.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace w4 {
namespace detail {

constexpr int kSB = 4;           // 64-wide K blocks per stage
constexpr int kStageK = kSB * kTK;
constexpr int kMaxPieces = 8;    // CTAs that may share one output tile (the planner guarantees it)

// Division by the group size g without a divide instruction: Granlund and Montgomery, "Division by
// invariant integers using multiplication" (PLDI 1994), the round-up method with a 33-bit multiplier
// split as 2^32 + m: q = (t + ((n - t) >> s1)) >> s2 with t = umulhi(m, n), exact for all n < 2^32.
struct FastDiv {
  uint32_t m, s1, s2;
  __device__ __forceinline__ int div(int n) const {
    const uint32_t un = static_cast<uint32_t>(n);
    const uint32_t t = __umulhi(m, un);
    return static_cast<int>((t + ((un - t) >> s1)) >> s2);
  }
};

inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((uint64_t{1} << l) < d) ++l;  // l = ceil(log2 d)
  FastDiv f;
  f.m = static_cast<uint32_t>(((uint64_t{1} << 32) * ((uint64_t{1} << l) - d)) / d + 1);
  f.s1 = l < 1 ? l : 1;
  f.s2 = l < 1 ? 0 : l - 1;
  return f;
}

// Output epilogues. The fp32 sum of weight row n for token m goes to
//   kEpiNone     y[m * ld + n];
//   kEpiSiluMul  rows alternate gate, up (row 2j: gate j, row 2j + 1: up j): h[m * ld + j] =
//                silu(gate) * up, silu(v) = v / (1 + e^-v), from the two fp32 sums, rounded once;
//   kEpiQkv      rows in head groups of (r query heads, 1 key head, 1 value head) x d rows: row n of
//                group n / ((r + 2) d), head hh = n % ((r + 2) d) / d goes to q (y) column
//                (grp r + hh) d + n % d for hh < r, to k column grp d + n % d for hh == r, to v for
//                hh == r + 1; q has ld columns per token, k and v ldkv.
struct Epi {
  int kind;
  int d, r;        // kEpiQkv: head size, query heads per group
  int ld, ldkv;    // output columns per token: y (or q, or h) and k / v
  uint16_t *k, *v;
};

// Where row n of token 0 goes (kEpiNone, kEpiQkv; d a multiple of 4, so four rows from a multiple
// of 4 stay in one head) and the output's columns per token.
__device__ __forceinline__ uint16_t *epi_row(const Epi &e, uint16_t *y, int n, int *ld) {
  if (e.kind != kEpiQkv) {
    *ld = e.ld;
    return y + n;
  }
  const int span = (e.r + 2) * e.d;
  const int grp = n / span;
  const int w = n - grp * span;
  const int hh = w / e.d;
  const int c = w - hh * e.d;
  if (hh < e.r) {
    *ld = e.ld;
    return y + (grp * e.r + hh) * e.d + c;
  }
  *ld = e.ldkv;
  return (hh == e.r ? e.k : e.v) + grp * e.d + c;
}

// silu(gate) * up in fp32 with the fast exponential and division (relative error ~1e-6, far below the
// output's rounding); a very negative gate gives 1 + e^-gate = inf and a (signed) zero.
__device__ __forceinline__ float silu_mul(float gate, float up) {
  return __fdividef(gate, 1.0f + __expf(-gate)) * up;
}

// Work decomposition. A unit is one K stage of one output tile (128 weight rows, or 256 for two-tile
// units, x BN activation rows); units are numbered tile-major: u = tile * KS + ks, tile = t * MT + mt.
// CTA c owns the contiguous units [begin(c), begin(c+1)), cut at multiples of `gran` units
// (gran = 1: stream-K, any cut; gran = KS: whole tiles only); or, for whole tiles of several token
// tiles (tstride = P), the tiles c, c + P, c + 2P, ...: the CTAs running at one time then share
// weight tiles (tile t * MT + mt for consecutive mt), whose re-reads hit L2.
// Problems of one tensor-memory launch that share x and K (one-tile units only): their weight tiles
// follow one another in the launch's tile numbering, problem i holding tiles [tile0[i], tile0[i + 1]).
constexpr int kTmemGroupMax = 8;

struct Params {
  const uint8_t *codes;  // tile region of the packed weights (nprob == 1)
  const uint8_t *meta;   // group-record region of the packed weights
  uint16_t *y;           // fp16 or bf16 bits
  float *pieces;         // [P][2][BN][128] fp32 partial tiles (first and last segment of each CTA)
  uint32_t *counters;    // [tiles] arrivals per split tile
  uint32_t *err;
  int M, N, K, g, G, NT, KB, KS, MT;
  int P;                 // CTAs
  int gran;              // units per scheduling grain
  int x3d;               // x tensor map is [KB][M][64] (one copy per stage); else [M][K] (one per block)
  int tstride;           // tiles between a CTA's consecutive tiles: 1 (contiguous ranges) or P
  FastDiv gdiv;          // division by g
  int64_t grains;        // total units / gran
  uint64_t wait_limit;   // cycles a wait may take before the kernel gives up
  int test_extra_piece;  // test only: owners wait for this many pieces more than will come
  Epi epi;               // where the sums go (y: q for kEpiQkv, h for kEpiSiluMul)
  // nprob > 1: the problems of a grouped launch (codes, meta, y, N and epi above are unused)
  int nprob;
  int tile0[kTmemGroupMax + 1];
  int gN[kTmemGroupMax];
  const uint8_t *gcodes[kTmemGroupMax];
  const uint8_t *gmeta[kTmemGroupMax];
  uint16_t *gy[kTmemGroupMax];
  Epi gepi[kTmemGroupMax];
};

// The problem holding weight tile t (0 for a single problem).
__device__ __forceinline__ int tile_problem(const Params &p, int t) {
  int i = 0;
  for (int j = 1; j < p.nprob; ++j) i += t >= p.tile0[j] ? 1 : 0;
  return i;
}

// Weight tile t's problem: its packed weights and the tile's index within them.
__device__ __forceinline__ void tile_weights(const Params &p, int t, const uint8_t **codes, const uint8_t **meta,
                                             int *local_t) {
  if (p.nprob <= 1) {
    *codes = p.codes;
    *meta = p.meta;
    *local_t = t;
    return;
  }
  const int i = tile_problem(p, t);
  *codes = p.gcodes[i];
  *meta = p.gmeta[i];
  *local_t = t - p.tile0[i];
}

// Where the rows of weight tile t go: its problem (read its output, N and epilogue with the accessors
// below, from the kernel parameters where they are used) and the tile's first row within it.
struct TileOut {
  int pi;
  int row0;
};

__device__ __forceinline__ TileOut tile_out(const Params &p, int t) {
  if (p.nprob <= 1) return TileOut{0, t * kTN};
  const int i = tile_problem(p, t);
  return TileOut{i, (t - p.tile0[i]) * kTN};
}

__device__ __forceinline__ uint16_t *prob_y(const Params &p, int pi) { return p.nprob <= 1 ? p.y : p.gy[pi]; }
__device__ __forceinline__ int prob_n(const Params &p, int pi) { return p.nprob <= 1 ? p.N : p.gN[pi]; }
__device__ __forceinline__ const Epi &prob_epi(const Params &p, int pi) { return p.nprob <= 1 ? p.epi : p.gepi[pi]; }

__device__ __forceinline__ int64_t range_begin(const Params &p, int c) {
  return static_cast<int64_t>(c) * p.grains / p.P * p.gran;
}

// CTA c's first unit and its number of units (stages).
__device__ __forceinline__ void cta_units(const Params &p, int c, int64_t *u0, int *nst) {
  if (p.tstride == 1) {
    *u0 = range_begin(p, c);
    *nst = static_cast<int>(range_begin(p, c + 1) - *u0);
  } else {  // whole tiles c, c + P, ...: p.grains tiles
    *u0 = static_cast<int64_t>(c) * p.KS;
    *nst = c < p.grains ? static_cast<int>((p.grains - c + p.P - 1) / p.P) * p.KS : 0;
  }
}

// The global unit of CTA c's local unit ul (its first unit u0).
__device__ __forceinline__ int64_t unit_at(const Params &p, int c, int64_t u0, int ul) {
  if (p.tstride == 1) return u0 + ul;
  return (static_cast<int64_t>(c) + static_cast<int64_t>(ul / p.KS) * p.tstride) * p.KS + ul % p.KS;
}

// The CTA whose range holds unit u: the largest c with range_begin(c) <= u (contiguous ranges).
__device__ __forceinline__ int owner_of(const Params &p, int64_t u) {
  const int64_t v = u / p.gran;
  return static_cast<int>(((v + 1) * p.P - 1) / p.grains);
}

// K blocks in stage ks of a tile: SBK, except a shorter last stage when KB is not a multiple of SBK.
template <int SBK = kSB>
__device__ __forceinline__ int stage_blocks(const Params &p, int ks) {
  return ks == p.KS - 1 ? p.KB - SBK * (p.KS - 1) : SBK;
}

// Walks (tile, ks, t, mt) over a CTA's units (without divisions for contiguous ranges). Every step
// stays within the CTA's own units: ranges are whole tiles whenever tstride > 1.
struct StageIter {
  int tile, ks, t, mt;
  __device__ __forceinline__ void init(const Params &p, int64_t u) {
    tile = static_cast<int>(u / p.KS);
    ks = static_cast<int>(u % p.KS);
    t = tile / p.MT;
    mt = tile % p.MT;
  }
  __device__ __forceinline__ void advance(const Params &p, int step) {
    ks += step;
    while (ks >= p.KS) {
      ks -= p.KS;
      if (p.tstride == 1) {
        ++tile;
        if (++mt == p.MT) {
          mt = 0;
          ++t;
        }
      } else {
        tile += p.tstride;
        t = tile / p.MT;
        mt = tile % p.MT;
      }
    }
  }
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// Per-(row, group) dequant constants as fp16x2 pairs.
struct GroupConsts {
  uint32_t s2;    // (s, s)
  uint32_t zb2;   // fp16: (1024 + z, 1024 + z); bf16: (128 + z, 128 + z)
  uint32_t nz2;   // fp16: (-(64 + z), -(64 + z)); bf16: unused
};

template <int DT = kDtypeF16>
__device__ __forceinline__ GroupConsts group_consts(uint32_t sbits, uint32_t z) {
  GroupConsts c;
  c.s2 = sbits * 0x00010001u;
  if (DT == kDtypeBf16) {
    c.zb2 = (0x4300u + z) * 0x00010001u;        // bf16 128 + z: exponent of 128, z in the fraction
    c.nz2 = 0u;
  } else {
    c.zb2 = (0x6400u + z) * 0x00010001u;        // fp16 1024 + z: exponent of 1024, z in the fraction
    c.nz2 = (0xD400u + 16u * z) * 0x00010001u;  // fp16 -(64 + z): step of 1/16 at 64
  }
  return c;
}

// 8 codes (tile nibble order: code e at nibble 4 (e % 2) + e / 2) -> 4 registers of 16-bit pairs
// (k, k+1) holding q - z exactly.
// fp16: 0x6400 | q is 1024 + q and 0x6400 | (q << 4) is 1024 + 16 q, both exact; subtracting
// 1024 + z (or scaling by 1/16 and adding -(64 + z)) leaves the small integer q - z, exact.
// bf16 (7 fraction bits): only the low nibble of each half fits under the exponent of 128, so the
// word is shifted by 0, 4, 8 and 12 bits; 0x4300 | q is 128 + q, and subtracting 128 + z is exact.
template <int DT = kDtypeF16>
__device__ __forceinline__ void dequant_word_int(uint32_t w, const GroupConsts &c, uint32_t *o) {
  if (DT == kDtypeBf16) {
    o[0] = bsub2_rn(lop3_and_or(w, 0x000F000Fu, 0x43004300u), c.zb2);
    o[1] = bsub2_rn(lop3_and_or(w >> 4, 0x000F000Fu, 0x43004300u), c.zb2);
    o[2] = bsub2_rn(lop3_and_or(w >> 8, 0x000F000Fu, 0x43004300u), c.zb2);
    o[3] = bsub2_rn(lop3_and_or(w >> 12, 0x000F000Fu, 0x43004300u), c.zb2);
  } else {
    constexpr uint32_t kInv16x2 = 0x2C002C00u;  // (1/16, 1/16)
    const uint32_t w8 = w >> 8;
    o[0] = hsub2_rn(lop3_and_or(w, 0x000F000Fu, 0x64006400u), c.zb2);
    o[1] = hfma2_rn(lop3_and_or(w, 0x00F000F0u, 0x64006400u), kInv16x2, c.nz2);
    o[2] = hsub2_rn(lop3_and_or(w8, 0x000F000Fu, 0x64006400u), c.zb2);
    o[3] = hfma2_rn(lop3_and_or(w8, 0x00F000F0u, 0x64006400u), kInv16x2, c.nz2);
  }
}

// As dequant_word_int, then one multiply by s: each weight (q - z) * s rounded once to the type.
template <int DT = kDtypeF16>
__device__ __forceinline__ void dequant_word(uint32_t w, const GroupConsts &c, uint32_t *o) {
  dequant_word_int<DT>(w, c, o);
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = DT == kDtypeBf16 ? bmul2_rn(o[i], c.s2) : hmul2_rn(o[i], c.s2);
}

// A stored scale (fp16 or bf16 bits) as fp32, exactly.
template <int DT>
__device__ __forceinline__ float scale_f32(uint32_t bits) {
  if (DT == kDtypeBf16) return __uint_as_float(bits << 16);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}

// An fp32 sum rounded once (to nearest even) to the output type, as bits.
template <int DT>
__device__ __forceinline__ uint16_t out_bits(float v) {
  if (DT == kDtypeBf16) return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  return __half_as_ushort(__float2half_rn(v));
}

// Two of them as one 32-bit word (lo at the lower address).
template <int DT>
__device__ __forceinline__ uint32_t out_bits2(float lo, float hi) {
  return static_cast<uint32_t>(out_bits<DT>(lo)) | (static_cast<uint32_t>(out_bits<DT>(hi)) << 16);
}

// A wait whose outcome is the same for all 32 lanes: the warp then either executes the
// following .sync.aligned tcgen05 instructions together or leaves the loop together.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                          uint32_t *err, uint64_t limit) {
  const bool ok = mbar_wait(bar, parity, abort_flag, err, limit);
  return __all_sync(0xffffffffu, ok);
}

// Waits ignoring the abort flag (used only to drain in-flight copies/MMAs before exit).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = clock_cycles();
  while (!mbar_try_wait_sleep(bar, parity, kSuspendNs)) {
    if (clock_cycles() - t0 > kWaitLimitCycles) return;
  }
}

// Tiles cut between CTAs (stream-K). A cut tile's owner is the CTA holding its first K stages;
// those are always the last units of the owner's range (ranges are contiguous and the tile goes on
// past the range's end). Every other CTA holding a piece of the tile holds it in its first (or
// only) segment: it stores the piece ([TP][BN][128] fp32, slot 0 of its two) and counts itself in
// with a release add. The owner, when its own part is done, waits (bounded) until all the others
// have counted in, adds their pieces to its own partial sums in K order and writes y; it leaves the
// counter at 0. Only owners wait, and only for pieces that the other CTAs produce without waiting,
// so the schedule cannot deadlock however the CTAs are scheduled.

// The piece CTA c keeps in slot `slot` (0: its first segment, 1: its last).
template <int BN, int TP>
__device__ __forceinline__ const float *piece_of(const Params &p, int c, int slot) {
  return p.pieces + (static_cast<int64_t>(c) * 2 + slot) * TP * BN * kTN;
}

// The owner's wait for the other npieces - 1 pieces of its tile (one thread; the caller's barrier
// after it orders the other threads' piece reads). Resets the counter. False on abort or timeout.
__device__ __forceinline__ bool wait_pieces(const Params &p, int tile, int npieces, volatile uint32_t *abort_flag) {
  const uint32_t target = static_cast<uint32_t>(npieces - 1 + p.test_extra_piece);
  const uint64_t t0 = clock_cycles();
  while (ld_acquire_gpu(&p.counters[tile]) < target) {
    if (*abort_flag) return false;
    if (clock_cycles() - t0 > p.wait_limit) {
      *abort_flag = 1u;
      atomicOr(p.err, kDevErrTimeout);
      return false;
    }
    __nanosleep(100);
  }
  p.counters[tile] = 0u;  // every other piece has counted in; ready for the next call
  return true;
}

// Pieces of tile `tile` (owned by CTA `owner`): the owner's own plus the others'.
__device__ __forceinline__ int tile_pieces(const Params &p, int tile, int owner) {
  return owner_of(p, static_cast<int64_t>(tile) * p.KS + p.KS - 1) - owner + 1;
}

// The weight-stream producer. Producer warp pw (of two) fills the stages i = pw, pw + 2, ... of the
// CTA's range; the whole warp waits, lane 0 issues. A stage is [x: four BN x 64 sub-tiles][codes:
// up to four 4 KB code tiles][group records], landing on full_bar[i % S]. Before stage i reuses
// slot s = i % S it waits for the release barriers rel[e * rel_stride + s], e < nrel, of stage
// i - S. Producer 0 first asks L2 for the codes and records of the CTA's first stages, then (like
// every role that reads global memory) waits for the previous grid in the stream.
template <int BN, int S, int kStageBytes>
__device__ __forceinline__ void produce_stages(const CUtensorMap *x_map, const Params &p, int64_t u0, int nst,
                                               int pw, int lane, uint32_t smem_base, uint64_t *full_bar,
                                               uint64_t *rel, int rel_stride, int nrel,
                                               volatile uint32_t *abort_flag) {
  constexpr int kXSub = BN * 128;
  constexpr int kXBytes = kSB * kXSub;
  constexpr int kCodeBytes = kSB * kTileBytes;
  // weights read once (one token tile) stream through L2 (evict first, so x stays); with several
  // token tiles the CTA reads each weight tile again for the next token tile, so they stay cached
  const uint64_t pol_stream = p.MT == 1 ? policy_evict_first() : policy_evict_normal();
  if (pw == 0 && lane == 0 && nst > 0) {
    StageIter f;
    f.init(p, u0);
    const int n0 = min(nst, min(S, p.KS - f.ks));  // first stages, contiguous within the first tile
    const int kend = min((f.ks + n0) * kStageK, p.K);
    const int blocks = min((f.ks + n0) * kSB, p.KB) - f.ks * kSB;
    const uint8_t *codes, *meta;
    int lt;
    tile_weights(p, f.t, &codes, &meta, &lt);
    bulk_prefetch_l2(codes + (static_cast<int64_t>(lt) * p.KB + f.ks * kSB) * kTileBytes, blocks * kTileBytes);
    const int jlo = p.gdiv.div(f.ks * kStageK);
    const int jhi = p.gdiv.div(kend - 1);
    bulk_prefetch_l2(meta + (static_cast<int64_t>(lt) * p.G + jlo) * kRecBytes, (jhi - jlo + 1) * kRecBytes);
  }
  griddep_wait();
  StageIter it;
  it.init(p, u0);
  it.advance(p, pw);
  int i = pw;
  for (; i < nst; i += 2, it.advance(p, 2)) {
    const int s = i % S;
    if (i >= S) {  // the consumers are done with the stage this slot held
      const uint32_t ph = ((i / S) - 1) & 1;
      bool ok = true;
      for (int e = 0; e < nrel && ok; ++e)
        ok = warp_wait(smem_u32(&rel[e * rel_stride + s]), ph, abort_flag, p.err, p.wait_limit);
      if (!ok) break;
    }
    if (lane == 0) {
      const int nb = stage_blocks(p, it.ks);
      const int k0 = it.ks * kStageK;
      const int jlo = p.gdiv.div(k0);
      const int jhi = p.gdiv.div(min(k0 + nb * kTK, p.K) - 1);
      const int nrec = jhi - jlo + 1;
      const uint32_t stage = smem_base + s * kStageBytes;
      const uint32_t bar = smem_u32(&full_bar[s]);
      // the 3-D box always lands whole (zero fill past the last K block); the 2-D boxes per block
      const uint32_t xbytes = p.x3d ? kXBytes : nb * kXSub;
      mbar_arrive_expect_tx(bar, xbytes + nb * kTileBytes + nrec * kRecBytes);
      if (p.x3d) {
        tma_load_3d(stage, x_map, 0, it.mt * BN, it.ks * kSB, bar);
      } else {
        for (int b = 0; b < nb; ++b) tma_load_2d(stage + b * kXSub, x_map, k0 + b * kTK, it.mt * BN, bar);
      }
      const uint8_t *codes, *meta;
      int lt;
      tile_weights(p, it.t, &codes, &meta, &lt);
      bulk_g2s(stage + kXBytes, codes + (static_cast<int64_t>(lt) * p.KB + it.ks * kSB) * kTileBytes,
               nb * kTileBytes, bar, pol_stream);
      bulk_g2s(stage + kXBytes + kCodeBytes, meta + (static_cast<int64_t>(lt) * p.G + jlo) * kRecBytes,
               nrec * kRecBytes, bar, pol_stream);
    }
    __syncwarp();
  }
  if (*abort_flag && lane == 0) {
    // let every copy this warp issued land before the CTA's shared memory goes away
    for (int j = i - 2; j >= 0 && j >= i - S; j -= 2) drain_wait(smem_u32(&full_bar[j % S]), (j / S) & 1);
  }
}

// Launch with programmatic stream serialization: the launch may overlap the previous kernel's tail;
// the kernels wait for it (griddepcontrol.wait) before touching global memory it may have written.
template <typename Kernel, typename... Args>
cudaError_t launch_programmatic(Kernel kern, int ctas, int threads, int smem_bytes, cudaStream_t stream,
                                const Args &...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Parameters of the cluster decode kernel (gemm_dec.cuh): M <= 8 * nb8 tokens, one token tile, and one
// or more independent problems (same M, g and type) whose weight tiles the launch walks in order.
constexpr int kDecMaxProblems = kGroupMax;

struct DecProblem {
  const uint16_t *x;     // [M, K] activations (fp16 or bf16 bits)
  const uint8_t *codes;  // tile region of the packed weights
  const uint8_t *meta;   // group-record region of the packed weights
  uint16_t *y;           // output (q for kEpiQkv, h for kEpiSiluMul)
  Epi epi;
  int N, K, G, NT, KB, KS;
  int tile_begin, tile_end;  // the problem's tiles in the launch's tile sequence
};
static_assert(sizeof(DecProblem) % 4 == 0, "the kernel copies the table in 4-byte words");

struct DecParams {
  DecProblem prob[kDecMaxProblems];
  int nprob;
  int tiles;             // all problems' weight tiles
  uint32_t *err;
  int M, g;
  int C;                 // CTAs per cluster; each takes a contiguous K range of every tile of the cluster
  int Q;                 // clusters; cluster q takes the tiles q, q + Q, ...
  int xslice;            // 256-wide K stages of x each CTA keeps in shared memory (its longest K range)
  int S;                 // stages in the weight ring (even)
  int early;             // issue the first stages' weight copies before waiting for the previous grid
  uint32_t test_extra_tx;  // test only: the reducer expects this many bytes more than will come
  FastDiv gdiv;          // division by g
  uint64_t wait_limit;   // cycles a pipeline wait may take before the kernel gives up
};

// Launches the decode kernel with `clusters` clusters of `cluster` CTAs (0: chosen for the layer), for
// fp16 or bf16 (dtype) activations, scales and outputs (gemm_dec_f16.cu, gemm_dec_bf16.cu).
cudaError_t launch_gemm_dec_f16(const DecParams &p, int nb8, int clusters, int cluster, cudaStream_t stream);
cudaError_t launch_gemm_dec_bf16(const DecParams &p, int nb8, int clusters, int cluster, cudaStream_t stream);
inline cudaError_t launch_gemm_dec(const DecParams &p, int nb8, int dtype, int clusters, int cluster,
                                   cudaStream_t stream) {
  return dtype == kDtypeBf16 ? launch_gemm_dec_bf16(p, nb8, clusters, cluster, stream)
                             : launch_gemm_dec_f16(p, nb8, clusters, cluster, stream);
}

}  // namespace detail
}  // namespace w4
