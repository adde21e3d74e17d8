// w4a16_gemm: y[M,N] = x[M,K] . dequant(Wq)[N,K]^T on sm_103a tensor cores (M >= 9 by default; the
// register-operand decode kernel, gemm_dec.cuh, takes M <= 8).
//
// Output tiles are 128 (weight rows n) x BN (activation rows m) tiles of y^T
// ("swap-AB": the weights sit on the MMA's M = 128 side, the tokens on its N
// side, so a decode batch still fills an MMA). The kernel is persistent: one
// CTA per SM walks its units (tile, K stage) -- a contiguous range (stream-K,
// so the work is split evenly whatever the number of tiles) or whole tiles
// dealt out round-robin (gemm_common.cuh).
//
// A stage is four 64-wide K blocks of one tile, or (TP = 2: BN = 128 from
// M = 256, and below where the tile pairs are many) two K blocks of two weight
// tiles sharing one x tile: 16 KB of 4-bit
// codes, the group records they need and the x sub-tiles, moved by three
// copies (one thread can issue a bulk copy only every ~350 cycles, so copies
// are made large). Warp roles (one CTA per SM):
//   2 producer warps take the stages in turn (lane 0 issues): a TMA tensor
//                   copy of x (128-byte swizzle, zero fill outside [M, K]) and
//                   two copies (codes, group records) on the stage's mbarrier.
//   4 dequant warpgroups: group d turns A block d of every stage into fp16
//                   w = (q - z) * s in tensor memory (thread r owns weight row
//                   r; tcgen05.st), the MMA's A operand; shared memory only
//                   holds 4-bit codes. A group never waits for the MMAs of its
//                   own block, only for its tensor-memory slots to come free.
//   4 MMA warps (2 for BN = 128; lane 0 issues): warp e issues the MMAs of its
//                   block(s) of every stage into its own accumulator and commits
//                   once per stage (a thread issues a tcgen05.mma only every
//                   ~50-130 cycles, so the issue is spread over several warps).
//   1 epilogue warpgroup: adds the MMA warps' accumulators of a finished tile
//                   segment in a fixed order (TP = 1; with TP = 2 each MMA warp
//                   owns one weight tile) and writes y, or an fp32 piece when
//                   the tile was cut between CTAs.
// When g is not a multiple of 64 the dequant looks the group up per 8 codes.
//
// This is the GB300 form of the techniques the Marlin post lists (prefetch,
// activation reuse, asynchronous weight loads, dequant interleaved with the
// tensor-core work, tuned warp roles): the weight stream is a multi-stage
// TMA/mbarrier ring, each x tile is reused by all 128 weight rows, and the
// dequant warps run ahead of the asynchronous MMAs through tensor-memory slots.
//
// A tile cut between CTAs is finished by its owner, the CTA holding its first
// K stages: the others store their fp32 pieces to the workspace and count
// themselves in early in their ranges; the owner adds the pieces to its own
// partial sums in K order (deterministic) and writes y (gemm_common.cuh).
// Every wait is bounded (ptx.cuh).
#include <cuda.h>
#include <cuda_fp16.h>

#include <cstring>
#include <mutex>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace w4 {
namespace {

using namespace detail;

enum Mode { kScaleIn = 1, kGeneral = 2 };  // g % 64 == 0 (one group per K block) or any g

template <int BN, int MODE, int TP>
struct Cfg {
  // Weight tiles per unit: TP = 2 (BN = 128 only) pairs two 128-row weight tiles on each x tile (half
  // the x bytes per MMA flop, twice the stages in shared memory); a stage then spans 2 K blocks of
  // both tiles.
  static constexpr int kTP = TP;
  static constexpr int kSBK = kSB / kTP;  // K blocks per stage; kTP * kSBK = 4 A blocks per stage
  static constexpr int kXSub = BN * 128;  // x for one K block: BN rows x 64 fp16 (1024-byte multiple)
  static constexpr int kXBytes = kSBK * kXSub;
  static constexpr int kCodeBytes = kSB * kTileBytes;
  // group records one stage can touch per weight tile: g >= 64 -> at most kSBK + 1; g >= 8 -> 8 kSBK + 1
  static constexpr int kMaxRecs = MODE == kGeneral ? kSBK * kTK / 8 + 1 : kSBK * kTK / 64 + 1;
  static constexpr int kRecBoxBytes = kTP * kMaxRecs * kRecBytes;
  static constexpr int kStageBytes = (kXBytes + kCodeBytes + kRecBoxBytes + 1023) / 1024 * 1024;
  static constexpr int kSmemBudget = 224 * 1024;  // one CTA per SM
  static constexpr int kStagesRaw = kSmemBudget / kStageBytes > 8 ? 8 : kSmemBudget / kStageBytes;
  // producer warp w fills the stages i = w (mod 2): an even ring keeps each slot with one producer
  static constexpr int kStages = kStagesRaw / 2 * 2;
  // MMA warps: one per K block of a stage (a thread issues a tcgen05.mma only every ~50-130 cycles),
  // two for BN = 128, whose accumulators would not fit four times into tensor memory
  static constexpr int kIssuers = BN == 128 ? 2 : 4;
  static constexpr int kBPI = kSB / kIssuers;  // K blocks per MMA warp and stage
  // tensor-memory A slots per dequant group (32 columns each): a group runs this many stages ahead of
  // its MMA warp. Narrow tiles take a third slot and give up a second accumulator set for it.
  static constexpr int kASlots = BN <= 32 ? 3 : 2;
  static constexpr int kDStride = BN < 32 ? 32 : BN;
  static constexpr int kDBufs = (BN <= 32 && kASlots == 2) ? 2 : 1;  // accumulator sets
  static constexpr int kACol0 = kIssuers * kDBufs * kDStride;  // accumulators first, then the A slots
  static constexpr int kTmemCols = 512;
  static constexpr int kIssuerWarp0 = 2;
  static constexpr int kDqWarp0 = kIssuerWarp0 + kIssuers;
  static constexpr int kEpiWarp0 = kDqWarp0 + 4 * kSB;  // one dequant warpgroup per K block of a stage
  static constexpr int kThreads = (kEpiWarp0 + 4) * 32;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack
  static_assert(kStages >= 2, "stage ring");
  static_assert(kACol0 + kSB * kASlots * 32 <= kTmemCols, "tensor memory budget");
  // a dequant group waits on the MMA-done barrier of stage i - kASlots; the next phase of that barrier
  // (stage i - kASlots + kStages) needs the group's own arrival for that stage, so it cannot come
  // before this wait as long as the stage ring is at least as long as the A-slot ring
  static_assert(kStages >= kASlots, "stage ring at least as long as the A-slot ring");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "MMA N");
  static_assert(TP == 1 || (TP == 2 && BN == 128), "two-tile units need both accumulators of BN = 128");
};

// Writes 16 consecutive columns (activation rows m0 + c0 ..) of weight row n of a finished tile
// segment: to y (fp16, rounded once) for a whole tile, else to the CTA's fp32 piece, which is laid
// out column by column ([BN][128]) so that a warp's 32 rows make one 128-byte line per column.
// Plain outputs of 128-token tiles (16-byte aligned y, row stride a multiple of 8) go through the
// warp's staging buffer wbuf (16 tokens x kEpiStride values): written token-major, then read back 8
// consecutive rows of one token per lane and stored 16 bytes at a time, an eighth of the store
// instructions of one 2-byte store per row and token (measured 2-2.5% faster at M = 512-1024; at
// block_n <= 64 no faster than the direct stores, which those tiles keep).
constexpr int kEpiStride = 40;  // 80 bytes: 16-byte aligned rows that start on different banks

template <int BN, int DT>
__device__ __forceinline__ void emit16(const Params &p, int pi, bool whole, int n, int m0, int m_end, int c0,
                                       const float (&v)[16], float *piece, uint16_t *wbuf) {
  if (whole) {
    const Epi &epi = prob_epi(p, pi);
    const int N = prob_n(p, pi);
    uint16_t *const y = prob_y(p, pi);
    if (BN == 128 && epi.kind == kEpiNone && epi.ld % 8 == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0) {
      const int lane = static_cast<int>(threadIdx.x) & 31;
      const int nw = n - lane;  // the warp's first row (a multiple of 32)
#pragma unroll
      for (int e = 0; e < 16; ++e) wbuf[e * kEpiStride + lane] = out_bits<DT>(v[e]);
      __syncwarp();
      const int n8 = 8 * (lane & 3);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int q = 2 * (lane >> 2) + k;
        const int64_t m = m0 + c0 + q;
        if (m < m_end) {
          const uint16_t *src = wbuf + q * kEpiStride + n8;
          uint16_t *dst = y + m * epi.ld + nw + n8;
          if (nw + n8 + 8 <= N) {
            *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
          } else {
            for (int j = 0; j < 8 && nw + n8 + j < N; ++j) dst[j] = src[j];
          }
        }
      }
      __syncwarp();  // the buffer is rewritten by the next chunk
      return;
    }
    if (epi.kind == kEpiSiluMul) {
      // rows n & ~1 (even lane: gate) and n | 1 (odd lane: up) of 16 tokens: the pair swaps values and
      // splits the tokens, the even lane writes silu(gate) * up of tokens 0..7, the odd lane of 8..15
      const bool odd = n & 1;
      float gate[8], up[8];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float other = __shfl_xor_sync(0xffffffffu, v[e], 1);
        if (e < 8 && !odd) {
          gate[e] = v[e];
          up[e] = other;
        } else if (e >= 8 && odd) {
          gate[e - 8] = other;
          up[e - 8] = v[e];
        }
      }
      if (n < N) {
        uint16_t *dst = prob_y(p, pi) + n / 2;
        const int e0 = odd ? 8 : 0;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (m0 + c0 + e0 + e < m_end)
            dst[static_cast<int64_t>(m0 + c0 + e0 + e) * epi.ld] = out_bits<DT>(silu_mul(gate[e], up[e]));
      }
    } else if (n < N) {
      int ld;
      uint16_t *dst = epi_row(epi, prob_y(p, pi), n, &ld);
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (m0 + c0 + e < m_end) dst[static_cast<int64_t>(m0 + c0 + e) * ld] = out_bits<DT>(v[e]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e) __stcg(piece + (c0 + e) * kTN, v[e]);
  }
}

// The weight-stream producer for units of two weight tiles (BN = 128). A stage is [x: SBK sub-tiles
// of BN x 64][codes: tile 0's SBK blocks, then tile 1's][records: kMaxRecs per tile from the stage's
// first group], moved by three tensor copies: x as for one tile, the codes of both tiles as one box
// of the [NT][16 KB][256 B] view of the tile region, their records as one box of the [NT][G][320 B]
// view of the record region. A second tile past N, blocks past K and records past G are filled with
// zeros by the copy (zero codes under a zero scale: A = 0). Otherwise as produce_stages.
template <int BN, int S, int kStageBytes, int SBK, int kMaxRecs>
__device__ __forceinline__ void produce_stages_pair(const CUtensorMap *x_map, const CUtensorMap *code_map,
                                                    const CUtensorMap *rec_map, const Params &p, int64_t u0, int nst,
                                                    int pw, int lane, uint32_t smem_base, uint64_t *full_bar,
                                                    uint64_t *rel, int rel_stride, int nrel,
                                                    volatile uint32_t *abort_flag) {
  constexpr int kXSub = BN * 128;
  constexpr int kXBytes = SBK * kXSub;
  constexpr int kCodeBytes = 2 * SBK * kTileBytes;
  constexpr int kRecBox = 2 * kMaxRecs * kRecBytes;
  constexpr int kRowsPerBlock = kTileBytes / 256;  // 256-byte rows of the code view
  // weights read once (one token tile) stream through L2 (evict first, so x stays); with several
  // token tiles the CTA reads each weight tile again for the next token tile, so they stay cached
  const uint64_t pol_stream = p.MT == 1 ? policy_evict_first() : policy_evict_normal();
  if (pw == 0 && lane == 0 && nst > 0) {
    StageIter f;
    f.init(p, u0);
    const int n0 = min(nst, min(S, p.KS - f.ks));  // first stages, contiguous within the first unit
    const int blocks = min((f.ks + n0) * SBK, p.KB) - f.ks * SBK;
    const int kend = min((f.ks + n0) * SBK * kTK, p.K);
    const int jlo = p.gdiv.div(f.ks * SBK * kTK);
    const int jhi = p.gdiv.div(kend - 1);
    for (int te = 0; te < 2; ++te) {
      const int t = 2 * f.t + te;
      if (t < p.NT) {
        bulk_prefetch_l2(p.codes + (static_cast<int64_t>(t) * p.KB + f.ks * SBK) * kTileBytes, blocks * kTileBytes);
        bulk_prefetch_l2(p.meta + (static_cast<int64_t>(t) * p.G + jlo) * kRecBytes, (jhi - jlo + 1) * kRecBytes);
      }
    }
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
      const int nb = stage_blocks<SBK>(p, it.ks);
      const int jlo = p.gdiv.div(it.ks * SBK * kTK);
      const uint32_t stage = smem_base + s * kStageBytes;
      const uint32_t bar = smem_u32(&full_bar[s]);
      // the 3-D boxes always land whole (zero fill outside); the 2-D x boxes per block
      const uint32_t xbytes = p.x3d ? kXBytes : nb * kXSub;
      mbar_arrive_expect_tx(bar, xbytes + kCodeBytes + kRecBox);
      if (p.x3d) {
        tma_load_3d(stage, x_map, 0, it.mt * BN, it.ks * SBK, bar);
      } else {
        for (int b = 0; b < nb; ++b) tma_load_2d(stage + b * kXSub, x_map, (it.ks * SBK + b) * kTK, it.mt * BN, bar);
      }
      tma_load_3d_hint(stage + kXBytes, code_map, 0, it.ks * SBK * kRowsPerBlock, 2 * it.t, bar, pol_stream);
      tma_load_3d_hint(stage + kXBytes + kCodeBytes, rec_map, 0, jlo, 2 * it.t, bar, pol_stream);
    }
    __syncwarp();
  }
  if (*abort_flag && lane == 0) {
    // let every copy this warp issued land before the CTA's shared memory goes away
    for (int j = i - 2; j >= 0 && j >= i - S; j -= 2) drain_wait(smem_u32(&full_bar[j % S]), (j / S) & 1);
  }
}

template <int BN, int MODE, int TP, int DT>
__global__ void __launch_bounds__(Cfg<BN, MODE, TP>::kThreads, 1)
    w4a16_gemm_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap code_map,
                      const __grid_constant__ CUtensorMap rec_map, const __grid_constant__ Params p) {
  using C = Cfg<BN, MODE, TP>;
  constexpr int S = C::kStages;
  // the owner of a cut tile parks its sums ([kTP][BN][128] fp32) in the idle stage ring
  constexpr bool kOwnInSmem = C::kTP * BN * kTN * 4 <= S * C::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  // Per-stage barriers (ring index = local stage index i mod the ring size; every waiter waits on
  // every phase of the barriers it uses, in order, so no parity wait can skip a phase):
  //   full[i % S]       the stage's copies landed (producer's expect_tx + the copies' bytes)
  //   mdone[e][i % S]   the MMAs MMA warp e issued for stage i are complete (one commit per stage):
  //                     frees the stage for the producer and the A slots of MMA warp e's dequant
  //                     groups (reused two stages later)
  //   afull[e][i % 2]   the dequant groups of MMA warp e's blocks (4 warps each) stored their A operands
  //   dfull / dempty    a tile segment's accumulators are complete / read out by the epilogue
  __shared__ __align__(8) uint64_t full_bar[S];
  constexpr int I = C::kIssuers;
  constexpr int BPI = C::kBPI;
  __shared__ __align__(8) uint64_t mdone_bar[I][S];
  __shared__ __align__(8) uint64_t afull_bar[I][C::kASlots];
  __shared__ __align__(8) uint64_t dfull_bar[C::kDBufs];
  __shared__ __align__(8) uint64_t dempty_bar[C::kDBufs];
  __shared__ __align__(8) uint64_t drain_bar[I];
  __shared__ __align__(8) uint64_t fix_bar;  // the owner's copies of the other pieces of its cut tile landed
  // per epilogue warp: its output staging (128-token tiles only)
  __shared__ __align__(16) uint16_t epi_stage[4][BN == 128 ? 16 * kEpiStride : 8];
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t abort_sh;
  __shared__ int npieces_sh;      // pieces of the cut tile the epilogue's segment owns
  __shared__ int own_tile_sh;     // the cut tile the CTA's last segment owns, or -1

  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  volatile uint32_t *abort_flag = &abort_sh;

  const int cta = blockIdx.x;
  int64_t u0;
  int nst;
  cta_units(p, cta, &u0, &nst);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      for (int e = 0; e < I; ++e) mbar_init(smem_u32(&mdone_bar[e][s]), 1);
    }
    for (int e = 0; e < I; ++e) {
      for (int a = 0; a < C::kASlots; ++a) mbar_init(smem_u32(&afull_bar[e][a]), 4 * BPI);  // groups' warps
      mbar_init(smem_u32(&drain_bar[e]), 1);
    }
    for (int d = 0; d < C::kDBufs; ++d) {
      mbar_init(smem_u32(&dfull_bar[d]), I);
      mbar_init(smem_u32(&dempty_bar[d]), 4);
    }
    mbar_init(smem_u32(&fix_bar), 1);
    abort_sh = 0;
    own_tile_sh = -1;
    fence_mbar_init();
  }
  if (warp == C::kDqWarp0) {
    tmem_alloc(smem_u32(&tmem_base_sh), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&x_map);
    if (C::kTP == 2) {
      prefetch_tensormap(&code_map);
      prefetch_tensormap(&rec_map);
    }
  }
  tc_fence_before();
  __syncwarp();
  cta_sync_all();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  // Programmatic dependent launch: the next grid in the stream may start launching now (its CTAs
  // take SMs as this grid's CTAs exit). Each role waits for the previous grid before its first
  // access to global memory that grid could have written: the producer (x, weights) after it has
  // asked L2 for its first stages' weights (a prefetch only: L2 is the point of coherence), the
  // epilogue (y, workspace) before its first store. Dequant and MMA warps touch only shared and
  // tensor memory.
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp < C::kIssuerWarp0) {
    // ------------------------------------------------------------ producers
    if (C::kTP == 2)
      produce_stages_pair<BN, S, C::kStageBytes, C::kSBK, C::kMaxRecs>(&x_map, &code_map, &rec_map, p, u0, nst, warp,
                                                                       lane, smem_base, full_bar, &mdone_bar[0][0], S,
                                                                       I, abort_flag);
    else
      produce_stages<BN, S, C::kStageBytes>(&x_map, p, u0, nst, warp, lane, smem_base, full_bar, &mdone_bar[0][0], S,
                                            I, abort_flag);
  } else if (warp < C::kDqWarp0) {
    // ------------------------------------------------------------ MMA issue
    // The whole warp runs the loop and waits together; lane 0 issues the MMAs and commits.
    // blocks (A slots of dequant groups) e * BPI .. e * BPI + BPI - 1 of every stage: K blocks of the
    // stage's one tile, or (kTP = 2) all K blocks of the stage's weight tile e
    const int e = warp - C::kIssuerWarp0;
    const int b0 = C::kTP == 2 ? 0 : BPI * e;  // this warp's first K block (x sub-tile) in a stage
    constexpr uint32_t idesc = idesc_f16_f32(128, BN, DT == kDtypeBf16);
    StageIter it;
    it.init(p, u0);
    int seg = 0;          // segment (tile) index within the CTA's range
    int seg_tile = it.tile;
    int seg_freed = 0;    // segments below this one are known to be read out by the epilogue
    bool started = false; // this warp issued an MMA into the current segment's accumulator
    bool ok = true;
    for (int i = 0; i < nst; ++i, it.advance(p, 1)) {
      if (it.tile != seg_tile) {
        if (lane == 0) mma_commit(smem_u32(&dfull_bar[seg % C::kDBufs]));
        ++seg;
        seg_tile = it.tile;
        started = false;
      }
      const int nb = stage_blocks<C::kSBK>(p, it.ks);
      const bool has = b0 < nb;
      if (has && !started) {
        // before the first MMA into a reused accumulator set, the epilogue must have read it out:
        // wait for every earlier segment's release in order, so no parity wait skips a phase
        for (; ok && seg_freed <= seg - C::kDBufs; ++seg_freed)
          ok = warp_wait(smem_u32(&dempty_bar[seg_freed % C::kDBufs]), (seg_freed / C::kDBufs) & 1, abort_flag,
                         p.err, p.wait_limit);
      }
      const uint32_t dcol = tmem + ((seg % C::kDBufs) * I + e) * C::kDStride;
      // the dequant groups stored their A operands; they saw the stage land before that, which
      // orders the x tile's arrival before these MMAs
      if (ok)
        ok = warp_wait(smem_u32(&afull_bar[e][i % C::kASlots]), (i / C::kASlots) & 1, abort_flag, p.err, p.wait_limit);
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t xs = smem_base + (i % S) * C::kStageBytes;
#pragma unroll
        for (int bb = 0; bb < BPI; ++bb) {
          const int b = b0 + bb;
          if (b >= nb) break;
          const uint64_t bdesc = sw128_kmajor_desc(xs + b * C::kXSub);
          const uint32_t acol = tmem + C::kACol0 + ((BPI * e + bb) * C::kASlots + i % C::kASlots) * 32;
#pragma unroll
          for (int kk = 0; kk < kTK / 16; ++kk) {
            // A: 128 x 16 fp16 in tensor memory (8 columns per 16 K); B: 16 K-columns of the x block
            const bool fresh = kk == 0 && bb == 0 && !started;
            mma_f16_ts(dcol, acol + kk * 8, bdesc + static_cast<uint64_t>(kk * 2), idesc, fresh ? 0u : 1u);
          }
        }
        mma_commit(smem_u32(&mdone_bar[e][i % S]));
      }
      if (has) started = true;
      __syncwarp();
    }
    if (lane == 0) {
      if (ok && nst > 0) mma_commit(smem_u32(&dfull_bar[seg % C::kDBufs]));
      if (*abort_flag) {
        mma_commit(smem_u32(&drain_bar[e]));
        drain_wait(smem_u32(&drain_bar[e]), 0);
      }
    }
  } else if (warp < C::kEpiWarp0) {
    // ------------------------------------------------------------ dequant
    // Group d takes K block d of every stage: thread r turns weight row r's 64 codes into the
    // A slot (d, i % kASlots), then its warp counts itself in on MMA warp d / BPI's afull barrier. A
    // group with no block in a (short) stage still takes part in every wait and arrival.
    const int d = (warp - C::kDqWarp0) / 4;
    const int e = d / BPI;
    const int te = C::kTP == 2 ? d / C::kSBK : 0;  // weight tile of the unit
    const int b = C::kTP == 2 ? d % C::kSBK : d;   // K block of the stage
    const int lq = warp % 4;  // tensor-memory lane quarter this warp may access
    const int r = lq * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(lq * 32) << 16;
    // g % 64 == 0 and g dividing the stage's K (or the stage lying in one group): block b's group is
    // the stage's first plus the same b * 64 / g in every stage, so its record sits at a fixed place
    constexpr int kStageKHere = C::kSBK * kTK;
    const bool fixed_rec = kStageKHere % p.g == 0 || p.g % kStageKHere == 0;
    const uint32_t fixed_rec_off = kStageKHere % p.g == 0 ? (b * kTK) / p.g * kRecBytes : 0u;
    StageIter it;
    it.init(p, u0);
    for (int i = 0; i < nst; ++i, it.advance(p, 1)) {
      const int s = i % S;
      if (!warp_wait(smem_u32(&full_bar[s]), (i / S) & 1, abort_flag, p.err, p.wait_limit)) break;
      const bool have = b < stage_blocks<C::kSBK>(p, it.ks);
      // the A slot's previous stage (i - kASlots) must have gone through its MMAs
      if (i >= C::kASlots &&
          !warp_wait(smem_u32(&mdone_bar[e][(i - C::kASlots) % S]), ((i - C::kASlots) / S) & 1, abort_flag, p.err,
                     p.wait_limit))
        break;
      if (have) {
        const uint32_t stage = smem_base + s * C::kStageBytes;
        const uint32_t codes = stage + C::kXBytes + d * kTileBytes;
        const uint32_t recs = stage + C::kXBytes + C::kCodeBytes + te * C::kMaxRecs * kRecBytes;
        const uint4 w0 = lds128(codes + r * 16);
        const uint4 w1 = lds128(codes + 2048 + r * 16);
        const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        const int kfirst = (it.ks * C::kSBK + b) * kTK;
        const uint32_t acol = tmem + lane_addr + C::kACol0 + (d * C::kASlots + i % C::kASlots) * 32;
        tc_fence_after();
        if (MODE != kGeneral) {
          // g % 64 == 0: one group per block
          const uint32_t rec =
              recs + (fixed_rec ? fixed_rec_off
                                : (p.gdiv.div(kfirst) - p.gdiv.div(it.ks * kStageKHere)) * kRecBytes);
          const uint32_t z = (lds8(rec + 256 + r / 2) >> (4 * (r & 1))) & 0xFu;
          const GroupConsts gc = group_consts<DT>(lds16(rec + 2 * r), z);
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // two halves of 16 columns: fewer registers live at once
            uint32_t out[16];
#pragma unroll
            for (int ci = 0; ci < 4; ++ci) dequant_word<DT>(words[4 * h + ci], gc, &out[4 * ci]);
            tmem_st_32x32b_x16(acol + 16 * h, out);
          }
        } else {
          const int jlo = p.gdiv.div(it.ks * kStageKHere);
          int j = p.gdiv.div(kfirst);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t out[16];
#pragma unroll
            for (int ci = 0; ci < 4; ++ci) {
              const int kc = kfirst + 8 * (4 * h + ci);
              if (kc >= (j + 1) * p.g && j < p.G - 1) ++j;  // g >= 8: at most one group boundary per 8 codes
              const uint32_t rec = recs + (j - jlo) * kRecBytes;
              const uint32_t z = (lds8(rec + 256 + r / 2) >> (4 * (r & 1))) & 0xFu;
              dequant_word<DT>(words[4 * h + ci], group_consts<DT>(lds16(rec + 2 * r), z), &out[4 * ci]);
            }
            tmem_st_32x32b_x16(acol + 16 * h, out);
          }
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&afull_bar[e][i % C::kASlots]));
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int lq = warp % 4;
    const int r = lq * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(lq * 32) << 16;
    griddep_wait();  // y and the workspace may still be in use by the previous grid
    int seg = 0;
    for (int ul = 0; ul < nst; ++seg) {  // local units ul .. ul + seg_len - 1: one tile segment
      const int64_t u = unit_at(p, cta, u0, ul);
      const int tile = static_cast<int>(u / p.KS);
      const int64_t tile_u0 = static_cast<int64_t>(tile) * p.KS;
      const int ks_first = static_cast<int>(u - tile_u0);
      const int seg_len = min(nst - ul, p.KS - ks_first);
      const int ks_last = ks_first + seg_len - 1;
      const bool whole = ks_first == 0 && ks_last == p.KS - 1;
      const int t = tile / p.MT;
      const int m0 = (tile % p.MT) * BN;
      const int m_end = min(p.M, m0 + BN);
      const int db = seg % C::kDBufs;
      // kTP = 1: MMA warp e took part iff some stage of the segment has more than BPI * e K blocks
      // (only a tile's last stage can be short), and the parts are added. kTP = 2: MMA warp e's
      // accumulator is weight tile e of the unit.
      const int nparts =
          C::kTP == 2 ? 1 : (ks_first < ks_last ? I : (stage_blocks<C::kSBK>(p, ks_last) + BPI - 1) / BPI);
      // a cut tile: its owner (the segment holds the tile's first stages) waits for the other pieces
      // before the accumulators are done, so the wait overlaps its last stages; any other piece is
      // stored and counted in (gemm_common.cuh)
      const bool owner = !whole && ks_first == 0;
      bool ok = true;
      if (owner && r == 0) {
        const int np = tile_pieces(p, tile, cta);
        ok = wait_pieces(p, tile, np, abort_flag);
        npieces_sh = np;
      }
      const bool landed = warp_wait(smem_u32(&dfull_bar[db]), (seg / C::kDBufs) & 1, abort_flag, p.err, p.wait_limit);
      if (!named_bar_and(1, 128, ok && landed)) break;  // (also publishes npieces_sh)
      tc_fence_after();
      // The owner's segment is the CTA's last, so once its accumulators landed every stage of the CTA
      // has gone through its MMAs and the stage ring is idle: the other pieces are copied into it (one
      // round trip, instead of one per 16 columns when read from the epilogue's loop), all at once when
      // they fit, else (two-tile units) one weight tile's part of every piece at a time; beyond that,
      // four or more go through the shared fixup below.
      constexpr uint32_t kPartBytes = BN * kTN * 4;  // one weight tile of a piece
      constexpr uint32_t kPieceBytes = C::kTP * kPartBytes;
      const int np = owner ? npieces_sh : 1;
      const bool ring_all = np > 1 && (np - 1) * kPieceBytes <= S * C::kStageBytes;
      const bool ring_part = !ring_all && C::kTP == 2 && np > 1 && (np - 1) * kPartBytes <= S * C::kStageBytes;
      const bool ring_fix = ring_all || ring_part;
      const uint32_t ring_stride = ring_all ? kPieceBytes : kPartBytes;  // bytes between pieces in the ring
      bool fix_ok = true;
      const float *fixed = reinterpret_cast<const float *>(smem_raw + (smem_base - smem_u32(smem_raw)));
      // With four or more pieces the owner's own sums go to shared memory (the stage ring is idle:
      // every MMA is done), where all dequant and epilogue warps add the other pieces below; with
      // fewer the epilogue adds them itself (measured on the 7B decode shapes: the extra barrier and
      // round trip through shared memory cost more than the wider reduction saves below four).
      const bool shared_fix = kOwnInSmem && owner && npieces_sh >= 4 && !ring_fix;
      float *own = reinterpret_cast<float *>(smem_raw + (smem_base - smem_u32(smem_raw)));
#pragma unroll 1
      for (int te = 0; te < C::kTP; ++te) {
        if (ring_fix && (te == 0 || ring_part)) {
          // every warp takes part in each round (no warp leaves the loop early): the barrier orders the
          // previous round's reads of the ring before its next copies
          if (te > 0) fix_ok = named_bar_and(1, 128, fix_ok);
          if (fix_ok) {
            if (r == 0) {
              // the pieces' stores (acquired by the counter wait) and the ring's earlier reads before the copies
              fence_proxy_async_global();
              fence_proxy_async_shared();
              const uint32_t bytes = ring_all ? kPieceBytes : kPartBytes;
              mbar_arrive_expect_tx(smem_u32(&fix_bar), (np - 1) * bytes);
              const uint64_t pol = policy_evict_first();
              for (int pc = 1; pc < np; ++pc)
                bulk_g2s(smem_base + (pc - 1) * ring_stride,
                         piece_of<BN, C::kTP>(p, cta + pc, 0) + (ring_all ? 0 : te * BN * kTN), bytes,
                         smem_u32(&fix_bar), pol);
            }
            fix_ok = warp_wait(smem_u32(&fix_bar), te & 1, abort_flag, p.err, p.wait_limit);
            if (!fix_ok && r == 0) drain_wait(smem_u32(&fix_bar), te & 1);  // no copy in flight when the CTA leaves
          }
        }
        if (!fix_ok) continue;
        const TileOut out = tile_out(p, t * C::kTP + te);
        const int n = out.row0 + r;  // the row within its problem
        float *piece =
            p.pieces + ((static_cast<int64_t>(cta) * 2 + (seg == 0 ? 0 : 1)) * C::kTP + te) * BN * kTN + r;
#pragma unroll 1
        for (int c0 = 0; c0 < BN && m0 + c0 < m_end; c0 += 16) {
          uint32_t v[16];
          const uint32_t dbase = tmem + lane_addr + (db * I + te) * C::kDStride + c0;
          // the MMA warps' partial sums, added in a fixed order; two loads per wait
          uint32_t v2[16];
          tmem_ld_32x32b_x16(dbase, v);
          if (nparts > 1) tmem_ld_32x32b_x16(dbase + C::kDStride, v2);
          tmem_wait_ld();
          float f[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) f[q] = __uint_as_float(v[q]);
          if (nparts > 1) {
#pragma unroll
            for (int q = 0; q < 16; ++q) f[q] += __uint_as_float(v2[q]);
          }
#pragma unroll 1
          for (int e = 2; e < nparts; e += 2) {
            tmem_ld_32x32b_x16(dbase + e * C::kDStride, v);
            if (e + 1 < nparts) tmem_ld_32x32b_x16(dbase + (e + 1) * C::kDStride, v2);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 16; ++q) f[q] += __uint_as_float(v[q]);
            if (e + 1 < nparts) {
#pragma unroll
              for (int q = 0; q < 16; ++q) f[q] += __uint_as_float(v2[q]);
            }
          }
          if (shared_fix) {
#pragma unroll
            for (int q = 0; q < 16; ++q) own[(te * BN + c0 + q) * kTN + r] = f[q];
          } else {
            if (ring_fix) {  // the later pieces in K order, from their copies in the ring
#pragma unroll 1
              for (int pc = 1; pc < np; ++pc) {
                const float *src = fixed + (pc - 1) * (ring_stride / 4) + ((ring_all ? te * BN : 0) + c0) * kTN + r;
#pragma unroll
                for (int q = 0; q < 16; ++q) f[q] += src[q * kTN];
              }
            } else if (owner) {  // the epilogue adds the later pieces in K order
#pragma unroll 1
              for (int pc = 1; pc < npieces_sh; ++pc) {
                const float *src = piece_of<BN, C::kTP>(p, cta + pc, 0) + (te * BN + c0) * kTN + r;
#pragma unroll
                for (int q = 0; q < 16; ++q) f[q] += __ldcg(src + q * kTN);
              }
            }
            emit16<BN, DT>(p, out.pi, whole || owner, n, m0, m_end, c0, f, piece, epi_stage[lq]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&dempty_bar[db]));
      if (!whole && !owner) {
        // a later piece of a cut tile: the warpgroup's stores are ordered (barrier) before one
        // thread's release count
        __syncwarp();
        named_bar_sync(1, 128);
        if (r == 0) red_add_release_gpu(&p.counters[tile]);
      }
      if (shared_fix && r == 0) own_tile_sh = tile;  // (the owner's segment is the CTA's last)
      ul += seg_len;
    }
  }

  if (warp >= C::kDqWarp0) {
    // the owner's fixup: every dequant and epilogue warp is idle now; they add the later pieces to
    // the owner's sums in K order and write y
    constexpr int kFixThreads = 32 * (C::kEpiWarp0 + 4 - C::kDqWarp0);
    __syncwarp();
    named_bar_sync(3, kFixThreads);
    const int tile = own_tile_sh;
    if (tile >= 0) {
      const float *own = reinterpret_cast<const float *>(smem_raw + (smem_base - smem_u32(smem_raw)));
      const int npieces = npieces_sh;
      const int m0 = (tile % p.MT) * BN;
      const int ncols = min(p.M, m0 + BN) - m0;
      const int tid = static_cast<int>(threadIdx.x) - 32 * C::kDqWarp0;
#pragma unroll
      for (int te = 0; te < C::kTP; ++te) {
        const TileOut out = tile_out(p, (tile / p.MT) * C::kTP + te);
        const Epi &epi = prob_epi(p, out.pi);
        // silu * up takes rows in (gate, up) pairs
        const int step = epi.kind == kEpiSiluMul ? 2 : 1;
#pragma unroll 2
        for (int e = tid * step; e < ncols * kTN; e += kFixThreads * step) {
          const int o = te * BN * kTN + e;
          float acc = own[o];
#pragma unroll
          for (int pc = 1; pc < kMaxPieces; ++pc)
            if (pc < npieces) acc += __ldcg(piece_of<BN, C::kTP>(p, cta + pc, 0) + o);
          const int n = out.row0 + e % kTN;  // the row within its problem
          const int64_t m = m0 + e / kTN;
          if (n >= prob_n(p, out.pi)) continue;
          if (step == 2) {
            float up = own[o + 1];
#pragma unroll
            for (int pc = 1; pc < kMaxPieces; ++pc)
              if (pc < npieces) up += __ldcg(piece_of<BN, C::kTP>(p, cta + pc, 0) + o + 1);
            prob_y(p, out.pi)[m * epi.ld + n / 2] = out_bits<DT>(silu_mul(acc, up));
          } else {
            int ld;
            uint16_t *dst = epi_row(epi, prob_y(p, out.pi), n, &ld);
            dst[m * ld] = out_bits<DT>(acc);
          }
        }
      }
    }
  }

  // every role ends here; lanes of a warp arrive at different times (lane 0 ran the producer or
  // MMA loop), so reconverge each warp and use the non-aligned barrier before freeing tensor memory
  tc_fence_before();
  __syncwarp();
  cta_sync_all();
  if (warp == C::kDqWarp0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ----------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// x [M, K] fp16 row-major, 128-byte swizzle, zero fill outside, in one of two views:
//  3-D [K/64][M][64] (K a multiple of 64): one box {64, BN, sbk} is a whole stage, sbk BN x 64
//      sub-tiles one after another, each laid out as the MMA reads it;
//  2-D [M][K]: one box {64, BN} per K block.
bool make_x_map(CUtensorMap *map, const void *x, int64_t M, int64_t K, int bn, int sbk, bool three_d, int dtype) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const CUtensorMapDataType dt = dtype == kDtypeBf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (three_d) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kTK), static_cast<cuuint64_t>(M),
                                static_cast<cuuint64_t>(K / kTK)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, static_cast<cuuint64_t>(kTK) * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(kTK), static_cast<cuuint32_t>(bn),
                               static_cast<cuuint32_t>(sbk)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, dt, 3, const_cast<void *>(x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTK), static_cast<cuuint32_t>(bn)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void *>(x), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The packed weights as two 3-D tensors of 32-bit words for the two-tile units (no swizzle, zero fill
// outside): the tile region [NT][KB * 16][64] (a 4 KB code block is 16 rows of 256 bytes), one box
// {64, 16 sbk, 2} = sbk blocks of two consecutive tiles; the record region [NT][G][80], one box
// {80, recs, 2} = recs consecutive group records of both tiles.
bool make_weight_maps(CUtensorMap *code_map, CUtensorMap *rec_map, const void *packed, int64_t NT, int64_t KB,
                      int64_t G, int sbk, int recs) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const uint8_t *codes = static_cast<const uint8_t *>(packed);
  const uint8_t *meta = codes + NT * KB * kTileBytes;
  const cuuint32_t estr[3] = {1, 1, 1};
  {
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(KB * (kTileBytes / 256)), static_cast<cuuint64_t>(NT)};
    const cuuint64_t strides[2] = {256, static_cast<cuuint64_t>(KB * kTileBytes)};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(sbk * (kTileBytes / 256)), 2};
    if (enc(code_map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t *>(codes), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  const cuuint64_t dims[3] = {kRecBytes / 4, static_cast<cuuint64_t>(G), static_cast<cuuint64_t>(NT)};
  const cuuint64_t strides[2] = {kRecBytes, static_cast<cuuint64_t>(G * kRecBytes)};
  const cuuint32_t box[3] = {kRecBytes / 4, static_cast<cuuint32_t>(recs), 2};
  return enc(rec_map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t *>(meta), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int MODE, int TP, int DT>
cudaError_t launch_t(const CUtensorMap &map, const CUtensorMap &code_map, const CUtensorMap &rec_map, const Params &p,
                     int ctas, cudaStream_t stream) {
  using C = Cfg<BN, MODE, TP>;
  auto kern = w4a16_gemm_kernel<BN, MODE, TP, DT>;
  // the dynamic shared-memory opt-in is a per-device function attribute
  static uint64_t done_mask = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev >= 64 || !(done_mask & (1ull << dev))) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
      if (e != cudaSuccess) return e;
      if (dev < 64) done_mask |= 1ull << dev;
    }
  }
  return launch_programmatic(kern, ctas, C::kThreads, C::kSmemBytes, stream, map, code_map, rec_map, p);
}

// One group per 64-wide K block (g % 64 == 0) lets the dequant take the block's group once.
int gemm_mode(int32_t g) { return g % 64 == 0 ? kScaleIn : kGeneral; }

// Pieces of a cut tile whose owner can take the others into its idle stage ring at once (the
// epilogue's fast fixup): 1 + ring bytes / piece bytes.
template <int BN, int MODE, int TP>
constexpr int64_t ring_piece_cap_t() {
  using C = Cfg<BN, MODE, TP>;
  return 1 + static_cast<int64_t>(C::kStages) * C::kStageBytes / (static_cast<int64_t>(TP) * BN * kTN * 4);
}
int64_t ring_piece_cap(int bn, int tp, int mode) {
  const bool s = mode == kScaleIn;
  if (bn == 64) return s ? ring_piece_cap_t<64, kScaleIn, 1>() : ring_piece_cap_t<64, kGeneral, 1>();
  if (bn == 128 && tp == 2) return s ? ring_piece_cap_t<128, kScaleIn, 2>() : ring_piece_cap_t<128, kGeneral, 2>();
  if (bn == 128) return s ? ring_piece_cap_t<128, kScaleIn, 1>() : ring_piece_cap_t<128, kGeneral, 1>();
  return 1;
}

template <int DT>
cudaError_t launch_variant(int bn, int mode, int tp, const CUtensorMap &map, const CUtensorMap &code_map,
                           const CUtensorMap &rec_map, const Params &p, int ctas, cudaStream_t stream) {
  if (mode == kScaleIn) {
    if (bn == 16) return launch_t<16, kScaleIn, 1, DT>(map, code_map, rec_map, p, ctas, stream);
    if (bn == 32) return launch_t<32, kScaleIn, 1, DT>(map, code_map, rec_map, p, ctas, stream);
    if (bn == 64) return launch_t<64, kScaleIn, 1, DT>(map, code_map, rec_map, p, ctas, stream);
    if (bn == 128 && tp == 1) return launch_t<128, kScaleIn, 1, DT>(map, code_map, rec_map, p, ctas, stream);
    if (bn == 128 && tp == 2) return launch_t<128, kScaleIn, 2, DT>(map, code_map, rec_map, p, ctas, stream);
  } else {
    if (bn == 16) return launch_t<16, kGeneral, 1, DT>(map, code_map, rec_map, p, ctas, stream);
    if (bn == 32) return launch_t<32, kGeneral, 1, DT>(map, code_map, rec_map, p, ctas, stream);
    if (bn == 64) return launch_t<64, kGeneral, 1, DT>(map, code_map, rec_map, p, ctas, stream);
    if (bn == 128 && tp == 1) return launch_t<128, kGeneral, 1, DT>(map, code_map, rec_map, p, ctas, stream);
    if (bn == 128 && tp == 2) return launch_t<128, kGeneral, 2, DT>(map, code_map, rec_map, p, ctas, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool make_gemm_plan(int64_t M, int64_t N, int64_t K, int32_t g, const GemmOptions &opt, int num_sms,
                    GemmPlan *plan) {
  (void)g;
  const int block_n = opt.block_n, ctas = opt.ctas, schedule = opt.schedule;
  if (opt.kernel < kKernelAuto || opt.kernel > kKernelTmem) return false;
  if (opt.cluster != 0 && opt.cluster != 1 && opt.cluster != 2 && opt.cluster != 4 && opt.cluster != 8) return false;
  // The decode kernel: M <= 8 by default, or on request with block_n 8 or 16 and M <= block_n. Its
  // workspace is the error word alone (the split along K is reduced in distributed shared memory).
  // Each CTA keeps its K range of x in shared memory, so K may be split at most 8 ways into ranges of
  // dec_x_stages_max stages; longer K goes to the tensor-memory kernel when the choice is automatic.
  const int64_t ks_dec = cdiv(cdiv(K, kTK), kSB);
  const bool dec_fits = dec_x_fits(ks_dec, 8, M);
  // 9..16 tokens: the decode kernel (two 8-token MMA columns) where a layer has few weight tiles, the
  // tensor-memory kernel otherwise (measured on the 7B decode shapes: faster on the 32-tile o_proj and
  // down_proj at M = 9..16 and on the 96-tile qkv up to M = 12; slower on the 172-tile gate/up)
  const int64_t nt_dec = cdiv(N, kTN);
  const int sms_dec = num_sms > 0 ? num_sms : 148;
  const bool dec_mid = M > 8 && M <= 16 && (nt_dec <= 64 || (M <= 12 && nt_dec * ks_dec <= 11 * sms_dec));
  const bool dec = opt.kernel == kKernelDecode ||
                   (opt.kernel == kKernelAuto &&
                    (block_n == 8 || (block_n == 0 && (M <= 8 || dec_mid) && dec_fits)));
  if (dec) {
    const int bn = block_n == 0 ? (M <= 8 ? 8 : 16) : block_n;
    if ((bn != 8 && bn != 16) || M > bn || ctas < 0 || ctas > 65535) return false;
    const int64_t nt = cdiv(N, kTN), kb = cdiv(K, kTK), ks = cdiv(kb, kSB);
    if (nt > 0x7FFFFFFF || (opt.cluster > 1 && opt.cluster > ks)) return false;
    // clusters below this size cannot hold x
    if (!dec_x_fits(ks, 8, M) || (opt.cluster > 0 && !dec_x_fits(ks, opt.cluster, M))) return false;
    *plan = GemmPlan{};
    plan->kernel = kKernelDecode;
    plan->cluster = opt.cluster;
    plan->block_n = bn;
    plan->m_tiles = 1;
    plan->n_tiles = static_cast<int>(nt);
    plan->k_blocks = static_cast<int>(kb);
    plan->k_stages = static_cast<int>(ks);
    plan->tiles_per_unit = 1;
    plan->ctas = ctas;  // clusters (0: as many as fit)
    plan->gran = static_cast<int>(ks);
    plan->whole = opt.cluster == 1;
    plan->grains = nt;
    plan->counters_offset = 256;
    plan->pieces_offset = 256;
    plan->workspace_bytes = 256;
    return true;
  }
  if (opt.kernel == kKernelTmem && block_n == 8) return false;
  int bn = block_n;
  if (bn == 0) {
    bn = M <= 8 ? 8 : M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
    // 65..128 tokens on a layer with fewer 128-row weight tiles than SMs: two token tiles of 64
    // give twice the output tiles (cut less often) at one extra, mostly L2-served, pass over the
    // weights; measured faster on the 4096- to 12288-row 7B layers, slower on the 22016-row one.
    // The same holds with three token tiles (129..192 tokens), and with four on layers of at most 32
    // weight tiles, for K up to 16384 (at M = 129..255: 4096x4096 22% faster, 11008x4096 12-15%,
    // 8192x8192 8-10%, 10240x8192 0-3%; four token tiles on the 64- to 96-tile layers 9-14% slower,
    // and 8192x28672 12% slower than two-tile units)
    const int sms = num_sms > 0 ? num_sms : 148;
    const int64_t nt_b = cdiv(N, kTN);
    if (bn == 128 && nt_b < sms && (M <= 128 || (K <= 16384 && (M <= 192 || nt_b <= 32)))) bn = 64;
  }
  if (bn != 16 && bn != 32 && bn != 64 && bn != 128) return false;
  if (ctas < 0 || ctas > 65535 || schedule < 0 || schedule > 2) return false;
  // Units of two weight tiles and 128-wide K stages for block_n 128 from M = 256 up (two or more
  // token tiles, so each CTA holds long runs of units and a tile pair is cut at most a few times), and
  // below that where the tile pairs are many (at least 0.4 per SM): a one-tile stage with 128 tokens of
  // x (82 KB) leaves room for a ring of two, too short to hide the weight stream's latency, a pair
  // stage (50 KB) for four. Measured at M = 80..224: 22016x4096 4-15% faster, 57344x8192 26-33%,
  // 28672x8192 22%, 8192x28672 33%, 10240x8192 7%; with 32 pairs (4096-row layers) 40-110% slower, the
  // fixup of the cut pairs (two 64 KB tiles a piece) costing more than the deeper ring saves.
  // Otherwise one tile and 256-wide stages.
  const int64_t pairs = cdiv(M, 128) * cdiv(cdiv(N, kTN), 2);
  const int sms_tp = num_sms > 0 ? num_sms : 148;
  const int tp = bn == 128 && (M >= 256 || (!opt.one_tile_mid && 5 * pairs >= 2 * sms_tp)) ? 2 : 1;
  const int64_t mt = cdiv(M, bn), nt = cdiv(N, kTN), kb = cdiv(K, kTK), ks = cdiv(kb, kSB / tp);
  const int64_t tiles = mt * cdiv(nt, tp);  // output tiles of the schedule (units along K: ks each)
  const int64_t units = tiles * ks;
  if (tiles > 0x7FFFFFFF || units > (int64_t{1} << 40)) return false;
  int64_t P = ctas > 0 ? ctas : (num_sms > 0 ? num_sms : 148);
  // Fewer output tiles than SMs (64- or 128-token tiles): cut each tile into equal pieces, as many as
  // the SMs allow and the owner can take into its stage ring at once, instead of spreading all stages
  // over every SM; one piece means whole tiles. Measured on the 7B layers (M = 64: o_proj 10% faster
  // in 4 pieces, down_proj 16%; M = 64..128 qkv 18% faster as whole tiles) and the 70B layers
  // (M = 256: down_proj 14% faster in 2 pieces, o_proj 30%; qkv 8% as whole tiles).
  // Units of two weight tiles go stream-K over every SM instead, unless whole tiles keep at least 4/5 of
  // the SMs busy (70B layers: qkv M = 256 20% faster than whole tiles, down_proj M = 256 6% faster than
  // 2 pieces; o_proj M = 512 3% slower than whole tiles).
  bool fewer = false;
  if (ctas == 0 && schedule == 0 && bn >= 64 && tiles < P) {
    const int64_t pieces = std::max<int64_t>(1, std::min<int64_t>(P / tiles, ring_piece_cap(bn, tp, gemm_mode(g))));
    if (tp == 1 || tiles * 5 >= P * 4) {
      P = tp == 1 ? tiles * pieces : tiles;
      fewer = tp == 2 || pieces == 1;
    }
  }
  // whole-tile scheduling when every CTA gets many tiles (imbalance <= 1/8) or the tiles divide
  // evenly; otherwise stream-K over 256-wide K stages, which needs the partial-tile fixup
  bool whole = schedule == 2 ||
               (schedule == 0 && (fewer || tiles >= 8 * P || (tiles >= P && tiles % P == 0)));
  const int64_t gran = whole ? ks : 1;
  const int64_t grains = units / gran;
  P = std::min(P, grains);
  if (!whole) {
    // the fixup adds at most kMaxPieces pieces per tile: shrink the grid until no tile is cut into more
    // (CTA c owns units [c*U/P, (c+1)*U/P); the owner of unit u is ((u + 1) * P - 1) / U)
    auto max_pieces = [&](int64_t PP) {
      int64_t worst = 1;
      for (int64_t tt = 0; tt < tiles; ++tt) {
        const int64_t first = ((tt * ks + 1) * PP - 1) / units;
        const int64_t last = (((tt + 1) * ks) * PP - 1) / units;
        worst = std::max(worst, last - first + 1);
      }
      return worst;
    };
    while (P > 1 && max_pieces(P) > kMaxPieces) --P;
  }
  plan->kernel = kKernelTmem;
  plan->cluster = 0;
  plan->block_n = bn;
  plan->m_tiles = static_cast<int>(mt);
  plan->n_tiles = static_cast<int>(nt);
  plan->k_blocks = static_cast<int>(kb);
  plan->k_stages = static_cast<int>(ks);
  plan->tiles_per_unit = tp;
  plan->ctas = static_cast<int>(P);
  plan->gran = static_cast<int>(gran);
  plan->whole = whole;
  // whole tiles of several token tiles are dealt out round-robin, so that the CTAs running together
  // read the same weight tiles (one DRAM read, the rest L2 hits)
  plan->interleave = whole && mt > 1;
  plan->grains = grains;
  plan->counters_offset = 256;
  const size_t counters_bytes = static_cast<size_t>(cdiv(tiles * 4, 256) * 256);
  plan->pieces_offset = plan->counters_offset + counters_bytes;
  const size_t piece_bytes = whole ? 0 : static_cast<size_t>(P * 2 * tp * kTN * bn * 4);
  plan->workspace_bytes = plan->pieces_offset + piece_bytes;
  return true;
}

bool epi_valid(const EpiSpec &e, int64_t N) {
  if (e.kind == kEpiNone) return true;
  if (e.kind == kEpiSiluMul) return N % 2 == 0;
  if (e.kind != kEpiQkv) return false;
  if (e.head_dim < 4 || e.head_dim % 4 != 0 || e.q_per_group < 1 || !e.k || !e.v) return false;
  const int64_t span = static_cast<int64_t>(e.q_per_group + 2) * e.head_dim;
  return span <= N && N % span == 0;
}

namespace {

Epi make_epi(const EpiSpec &e, int64_t N) {
  Epi d{};
  d.kind = e.kind;
  d.ld = static_cast<int>(e.kind == kEpiSiluMul ? N / 2 : N);
  if (e.kind == kEpiQkv) {
    const int64_t groups = N / ((e.q_per_group + 2) * static_cast<int64_t>(e.head_dim));
    d.d = e.head_dim;
    d.r = e.q_per_group;
    d.ld = static_cast<int>(groups * e.q_per_group * e.head_dim);
    d.ldkv = static_cast<int>(groups * e.head_dim);
    d.k = static_cast<uint16_t *>(e.k);
    d.v = static_cast<uint16_t *>(e.v);
  }
  return d;
}

// One problem's entry of the decode kernel's table, its tiles from `tile_begin`.
DecProblem dec_problem(const void *x, const void *packed, void *y, int64_t N, int64_t K, int32_t g,
                       const EpiSpec &epi, int tile_begin) {
  DecProblem d{};
  const int64_t nt = cdiv(N, kTN), kb = cdiv(K, kTK);
  d.x = static_cast<const uint16_t *>(x);
  d.codes = static_cast<const uint8_t *>(packed);
  d.meta = d.codes + nt * kb * kTileBytes;
  d.y = static_cast<uint16_t *>(y);
  d.epi = make_epi(epi, N);
  d.N = static_cast<int>(N);
  d.K = static_cast<int>(K);
  d.G = static_cast<int>(cdiv(K, g));
  d.NT = static_cast<int>(nt);
  d.KB = static_cast<int>(kb);
  d.KS = static_cast<int>(cdiv(kb, kSB));
  d.tile_begin = tile_begin;
  d.tile_end = tile_begin + d.NT;
  return d;
}

DecParams dec_params(int64_t M, int32_t g, void *workspace, const GemmOptions &opt) {
  DecParams p;
  std::memset(&p, 0, sizeof(p));
  p.err = static_cast<uint32_t *>(workspace);
  p.M = static_cast<int>(M);
  p.g = g;
  p.early = opt.weights_static ? 1 : 0;
  p.gdiv = make_fastdiv(static_cast<uint32_t>(g));
  p.wait_limit = opt.wait_limit ? opt.wait_limit : kWaitLimitCycles;
  p.test_extra_tx = opt.test_timeout ? 4u : 0u;
  return p;
}

}  // namespace

// The tensor-memory launch of a validated plan over x [M, K]: builds the tensor maps and the schedule
// fields of p; the caller has filled the problem fields (codes, meta, y, N, epi and nprob, or the
// problem table). `packed` is the single problem's weights (two-tile units read them by tensor maps).
cudaError_t launch_tmem(const void *x, const void *packed, int64_t M, int64_t K, int32_t g, void *workspace,
                        const GemmPlan &plan, const GemmOptions &opt, Params &p, cudaStream_t stream,
                        bool *encode_failed) {
  CUtensorMap map;
  const int sbk = kSB / plan.tiles_per_unit;
  bool x3d = K % kTK == 0 && make_x_map(&map, x, M, K, plan.block_n, sbk, true, opt.dtype);
  if (!x3d && !make_x_map(&map, x, M, K, plan.block_n, sbk, false, opt.dtype)) {
    *encode_failed = true;
    return cudaErrorInvalidValue;
  }
  CUtensorMap code_map, rec_map;  // the weights as tensors, for units of two weight tiles
  std::memset(&code_map, 0, sizeof(code_map));
  std::memset(&rec_map, 0, sizeof(rec_map));
  if (plan.tiles_per_unit == 2) {
    const int recs = gemm_mode(g) == kGeneral ? sbk * kTK / 8 + 1 : sbk * kTK / 64 + 1;
    if (!make_weight_maps(&code_map, &rec_map, packed, plan.n_tiles, plan.k_blocks, cdiv(K, g), sbk, recs)) {
      *encode_failed = true;
      return cudaErrorInvalidValue;
    }
  }
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  p.pieces = reinterpret_cast<float *>(ws + plan.pieces_offset);
  p.counters = reinterpret_cast<uint32_t *>(ws + plan.counters_offset);
  p.err = reinterpret_cast<uint32_t *>(ws);
  p.M = static_cast<int>(M);
  p.K = static_cast<int>(K);
  p.g = g;
  p.gdiv = make_fastdiv(static_cast<uint32_t>(g));
  p.G = static_cast<int>(cdiv(K, g));
  p.NT = plan.n_tiles;
  p.KB = plan.k_blocks;
  p.KS = plan.k_stages;
  p.MT = plan.m_tiles;
  p.P = plan.ctas;
  p.gran = plan.gran;
  p.x3d = x3d ? 1 : 0;
  p.tstride = plan.interleave ? plan.ctas : 1;
  p.grains = plan.grains;
  p.wait_limit = opt.wait_limit ? opt.wait_limit : kWaitLimitCycles;
  p.test_extra_piece = opt.test_timeout ? 1 : 0;
  if (opt.dtype == kDtypeBf16)
    return launch_variant<kDtypeBf16>(plan.block_n, gemm_mode(g), plan.tiles_per_unit, map, code_map, rec_map, p,
                                      plan.ctas, stream);
  return launch_variant<kDtypeF16>(plan.block_n, gemm_mode(g), plan.tiles_per_unit, map, code_map, rec_map, p,
                                   plan.ctas, stream);
}

cudaError_t launch_gemm(const void *x, const void *packed, int64_t M, int64_t N, int64_t K, int32_t g, void *y,
                        void *workspace, const GemmPlan &plan, const GemmOptions &opt, const EpiSpec &epi,
                        cudaStream_t stream, bool *encode_failed) {
  *encode_failed = false;
  if (plan.kernel == kKernelDecode) {
    DecParams p = dec_params(M, g, workspace, opt);
    p.prob[0] = dec_problem(x, packed, y, N, K, g, epi, 0);
    p.nprob = 1;
    p.tiles = p.prob[0].NT;
    return launch_gemm_dec(p, plan.block_n / 8, opt.dtype, plan.ctas, plan.cluster, stream);
  }
  Params p;
  std::memset(&p, 0, sizeof(p));
  p.codes = static_cast<const uint8_t *>(packed);
  p.meta = p.codes + static_cast<int64_t>(plan.n_tiles) * plan.k_blocks * kTileBytes;
  p.y = static_cast<uint16_t *>(y);
  p.N = static_cast<int>(N);
  p.epi = make_epi(epi, N);
  p.nprob = 1;
  return launch_tmem(x, packed, M, K, g, workspace, plan, opt, p, stream, encode_failed);
}


bool make_group_plan(const GemmProblem *probs, int count, int64_t M, int32_t g, const GemmOptions &opt, int num_sms,
                     GroupPlan *plan) {
  if (count < 1) return false;
  *plan = GroupPlan{};
  // the decode kernel runs the whole group when it would run each problem alone; the planner's checks
  // of the options (cluster sizes, tokens per tile) apply to every problem
  bool all_dec = true;
  for (int i = 0; i < count; ++i) {
    GemmPlan pl;
    if (!make_gemm_plan(M, probs[i].N, probs[i].K, g, opt, num_sms, &pl)) return false;
    if (pl.kernel != kKernelDecode) all_dec = false;
    if (i == 0) plan->block_n = pl.block_n;
    plan->workspace_bytes = std::max(plan->workspace_bytes, pl.workspace_bytes);
  }
  // one cluster size must suit every problem of a launch (at most each one's K stages, and short
  // enough K ranges for x to fit); otherwise the problems run one launch each
  bool common = false;
  for (int c : {1, 2, 4, 8}) {
    if (opt.cluster > 0 && c != opt.cluster) continue;
    bool ok = true;
    for (int i = 0; i < count && ok; ++i) {
      const int64_t ks = cdiv(cdiv(probs[i].K, kTK), kSB);
      ok = c <= ks && dec_x_fits(ks, c, M);
    }
    common = common || ok;
  }
  plan->decode = all_dec && common;
  if (plan->decode || count > kTmemGroupMaxHost) return true;
  // the tensor-memory kernel runs problems of one x and K together when the plan for their weight
  // tiles laid one after another takes it with one-tile units (below M = 256 asked for: on the 7B
  // gate/up pair at M = 65..128 one launch of one-tile units beats a launch per problem)
  int64_t tiles = 0;
  for (int i = 0; i < count; ++i) {
    if (probs[i].x != probs[0].x || probs[i].K != probs[0].K) return true;
    tiles += cdiv(probs[i].N, kTN);
  }
  GemmPlan pl;
  GemmOptions one = opt;
  one.one_tile_mid = true;
  if (count > 1 && tiles * kTN <= 0x7FFFFFFF && make_gemm_plan(M, tiles * kTN, probs[0].K, g, one, num_sms, &pl) &&
      pl.kernel == kKernelTmem && pl.tiles_per_unit == 1) {
    plan->tmem = true;
    plan->tmem_plan = pl;
    plan->workspace_bytes = pl.workspace_bytes;
  }
  return true;
}

cudaError_t launch_gemm_grouped(const GemmProblem *probs, int count, int64_t M, int32_t g, void *workspace,
                                const GroupPlan &plan, const GemmOptions &opt, int num_sms, cudaStream_t stream,
                                bool *encode_failed) {
  *encode_failed = false;
  if (plan.decode) {
    for (int i0 = 0; i0 < count; i0 += kGroupMax) {
      const int n = std::min(count - i0, kGroupMax);
      DecParams p = dec_params(M, g, workspace, opt);
      int tiles = 0;
      for (int i = 0; i < n; ++i) {
        const GemmProblem &pr = probs[i0 + i];
        p.prob[i] = dec_problem(pr.x, pr.packed, pr.y, pr.N, pr.K, g, pr.epi, tiles);
        tiles = p.prob[i].tile_end;
      }
      p.nprob = n;
      p.tiles = tiles;
      const cudaError_t e = launch_gemm_dec(p, plan.block_n / 8, opt.dtype, opt.ctas, opt.cluster, stream);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  if (plan.tmem) {
    static_assert(kTmemGroupMaxHost == kTmemGroupMax, "group table size");
    Params p;
    std::memset(&p, 0, sizeof(p));
    p.nprob = count;
    int tiles = 0;
    for (int i = 0; i < count; ++i) {
      const GemmProblem &pr = probs[i];
      const int nt = static_cast<int>(cdiv(pr.N, kTN));
      p.tile0[i] = tiles;
      p.gN[i] = static_cast<int>(pr.N);
      p.gcodes[i] = static_cast<const uint8_t *>(pr.packed);
      p.gmeta[i] = p.gcodes[i] + static_cast<int64_t>(nt) * plan.tmem_plan.k_blocks * kTileBytes;
      p.gy[i] = static_cast<uint16_t *>(pr.y);
      p.gepi[i] = make_epi(pr.epi, pr.N);
      tiles += nt;
    }
    p.tile0[count] = tiles;
    p.N = tiles * kTN;
    return launch_tmem(probs[0].x, probs[0].packed, M, probs[0].K, g, workspace, plan.tmem_plan, opt, p, stream,
                       encode_failed);
  }
  for (int i = 0; i < count; ++i) {
    const GemmProblem &pr = probs[i];
    GemmPlan pl;
    if (!make_gemm_plan(M, pr.N, pr.K, g, opt, num_sms, &pl)) return cudaErrorInvalidValue;
    const cudaError_t e = launch_gemm(pr.x, pr.packed, M, pr.N, pr.K, g, pr.y, workspace, pl, opt, pr.epi, stream,
                                      encode_failed);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace w4
