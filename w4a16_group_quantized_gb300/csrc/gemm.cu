// w4a16_gemm: y[M,N] = x[M,K] . dequant(Wq)[N,K]^T on sm_103a tensor cores.
//
// Output tiles are 128 (weight rows n) x BN (activation rows m) tiles of y^T
// ("swap-AB": the weights sit on the MMA's M = 128 side, the tokens on its N
// side, so a batch of 1..16 tokens still fills an MMA). The kernel is
// persistent: one CTA per SM walks a contiguous range of (tile, 64-wide K
// block) units, so the work is split evenly whatever the number of tiles
// (stream-K); a tile cut between CTAs is finished by a fixup (below).
//
// Warp roles (one CTA per SM):
//   4 producer warps (lane 0) take the 64-wide K blocks in turn: per block one
//                   TMA tensor copy of the x tile (128-byte swizzle, zero fill
//                   outside [M, K]) and two bulk copies (4 KB of codes, group
//                   records), all completing on the stage's mbarrier.
//   2-4 dequant warpgroups take K blocks in turn: thread r owns weight row r;
//                   it turns the row's 64 codes into fp16 (q - z) * s and stores
//                   them into tensor memory (tcgen05.st), where they are the
//                   MMA's A operand (shared memory only ever holds 4-bit codes);
//                   then the group's first thread issues the block's MMAs into
//                   the group's own accumulator. The first group also
//                   allocates tensor memory.
//   1 epilogue warpgroup: reads a finished tile's accumulators (double-buffered
//                   for BN <= 32, so the next tile's MMAs overlap it), adds the
//                   groups' parts in a fixed order and writes y, or an fp32
//                   partial tile when the tile was cut between CTAs.
// The copies and MMAs are spread over several threads because one thread
// issues a bulk copy only every ~350 cycles and a tcgen05 op every ~100.
//
// This is the GB300 form of the techniques the Marlin post lists (prefetch,
// activation reuse, asynchronous weight loads, dequant interleaved with the
// tensor-core work, tuned warp roles): the weight stream is a multi-stage
// TMA/mbarrier ring, each x tile is reused by all 128 weight rows, and the
// dequant warps run ahead of the asynchronous MMAs through a ring of tensor-
// memory slots.
//
// Fixup of a cut tile: each CTA holding a piece writes it (fp32) to the
// workspace and counts itself in on the tile's counter; the last to arrive
// adds the pieces in K order (deterministic) and writes y. Nothing ever waits
// on another CTA. Every mbarrier wait is bounded (ptx.cuh).
#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace w4 {
namespace {

constexpr int kMaxRecs = 9;  // group records one 64-wide K block can touch (g = 8: 8 groups)
constexpr int kMaxPieces = 8;  // CTAs that may share one output tile (the planner guarantees it)

__host__ __device__ constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p *= 2;
  return p;
}

template <int BN, bool GENERAL>
struct Cfg {
  static constexpr int kXBytes = BN * 128;  // BN rows x 64 fp16
  static constexpr int kMetaBytes = GENERAL ? kMaxRecs * kRecBytes : kRecBytes;
  static constexpr int kStageBytes = (kXBytes + kTileBytes + kMetaBytes + 1023) / 1024 * 1024;
  static constexpr int kSmemBudget = 200 * 1024;  // one CTA per SM
  // One thread can issue a bulk copy only every ~350 cycles, whatever its size, so four producer
  // warps take the K blocks in turn (three copies each).
  static constexpr int kProducers = 4;
  // Dequant warpgroups: narrow (HBM-bound) tiles need four to hide each one's latency; wide
  // (tensor-bound) tiles need a K block only every 256-512 cycles and keep the registers instead.
  static constexpr int kDqGroups = BN <= 64 ? 4 : 2;
  // A producer / dequant warpgroup waits only on the stages (and tensor-memory slots) of its own K
  // blocks. An mbarrier parity wait is only sound for a waiter that sees every phase of that
  // barrier: if a ring's size were not a multiple of the number of such waiters, successive uses of
  // one stage would go to different waiters, and one that ran ahead could take the previous, still
  // landing phase for its own (bulk copies complete out of order). So the rings are multiples of 4.
  static constexpr int kStagesRaw = kSmemBudget / kStageBytes;
  static constexpr int kStages = (kStagesRaw > 16 ? 16 : kStagesRaw) / 4 * 4;
  static constexpr int kASlots = 8;    // tensor-memory slots of dequantized weights (32 columns each)
  // Each dequant warpgroup issues the MMAs of its own K blocks into its own tensor-memory
  // accumulator (the epilogue adds the groups' accumulators in a fixed order): no separate issuing
  // warp, no extra barrier hop between a block's dequant and its MMAs.
  static constexpr int kDBufs = BN <= 32 ? 2 : 1;  // accumulator sets (epilogue overlaps the next tile)
  static constexpr int kDStride = BN < 32 ? 32 : BN;
  static constexpr int kACol0 = kDBufs * kDqGroups * kDStride;
  static constexpr int kTmemCols = pow2_at_least(kACol0 + kASlots * 32);
  static constexpr int kDqWarp0 = kProducers;
  static constexpr int kEpiWarp0 = kDqWarp0 + 4 * kDqGroups;
  static constexpr int kThreads = (kEpiWarp0 + 4) * 32;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack
  static_assert(kStages >= 4 && kStages % kDqGroups == 0 && kStages % kProducers == 0,
                "stage ring: a multiple of the producers and of the dequant groups");
  static_assert(kASlots % kDqGroups == 0, "tensor-memory slot ring: a multiple of the dequant groups");
  static_assert(kTmemCols <= 512, "tensor memory budget");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "MMA N");
};

// Work decomposition. A unit is one 64-wide K block of one output tile (128 weight rows x BN
// activation rows); units are numbered tile-major: u = tile * KB + kb, tile = t * MT + mt.
// CTA c owns the contiguous units [begin(c), begin(c+1)), cut at multiples of `gran` units
// (gran = 1: stream-K, any cut; gran = KB: whole tiles only).
struct Params {
  const uint8_t *codes;  // tile region of the packed weights
  const uint8_t *meta;   // group-record region of the packed weights
  __half *y;
  float *pieces;         // [P][2][128][BN] fp32 partial tiles (first and last segment of each CTA)
  uint32_t *counters;    // [tiles] arrivals per split tile
  uint32_t *err;
  int M, N, K, g, G, NT, KB, MT;
  int P;                 // CTAs
  int gran;              // units per scheduling grain
  int64_t grains;        // total units / gran
};

__device__ __forceinline__ int64_t range_begin(const Params &p, int c) {
  return static_cast<int64_t>(c) * p.grains / p.P * p.gran;
}

// The CTA whose range holds unit u: the largest c with range_begin(c) <= u.
__device__ __forceinline__ int owner_of(const Params &p, int64_t u) {
  const int64_t v = u / p.gran;
  return static_cast<int>(((v + 1) * p.P - 1) / p.grains);
}

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
  uint32_t zb2;   // (1024 + z, 1024 + z)
  uint32_t nz2;   // (-(64 + z), -(64 + z))
};

__device__ __forceinline__ GroupConsts group_consts(uint32_t sbits, uint32_t z) {
  GroupConsts c;
  c.s2 = sbits * 0x00010001u;
  c.zb2 = (0x6400u + z) * 0x00010001u;          // fp16 1024 + z: exponent of 1024, z in the fraction
  c.nz2 = (0xD400u + 16u * z) * 0x00010001u;    // fp16 -(64 + z): step of 1/16 at 64
  return c;
}

// 8 codes (tile nibble order) -> 4 registers of fp16 pairs (k, k+1), each (q - z) * s rounded once.
// 0x6400 | q is the fp16 1024 + q and 0x6400 | (q << 4) is 1024 + 16 q, both exact; subtracting
// 1024 + z (or scaling by 1/16 and adding -(64 + z)) gives q - z exactly; one multiply by s rounds.
__device__ __forceinline__ void dequant_word(uint32_t w, const GroupConsts &c, uint32_t *o) {
  constexpr uint32_t kInv16x2 = 0x2C002C00u;  // (1/16, 1/16)
  const uint32_t w8 = w >> 8;
  const uint32_t p0 = lop3_and_or(w, 0x000F000Fu, 0x64006400u);
  const uint32_t p1 = lop3_and_or(w, 0x00F000F0u, 0x64006400u);
  const uint32_t p2 = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);
  const uint32_t p3 = lop3_and_or(w8, 0x00F000F0u, 0x64006400u);
  o[0] = hmul2_rn(hsub2_rn(p0, c.zb2), c.s2);
  o[1] = hmul2_rn(hfma2_rn(p1, kInv16x2, c.nz2), c.s2);
  o[2] = hmul2_rn(hsub2_rn(p2, c.zb2), c.s2);
  o[3] = hmul2_rn(hfma2_rn(p3, kInv16x2, c.nz2), c.s2);
}

// A wait whose outcome is the same for all 32 lanes: the warp then either executes the
// following .sync.aligned tcgen05 instructions together or leaves the loop together.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag,
                                          uint32_t *err, uint32_t max_sleep_ns = 128) {
  const bool ok = mbar_wait(bar, parity, abort_flag, err, max_sleep_ns);
  return __all_sync(0xffffffffu, ok);
}

// Waits ignoring the abort flag (used only to drain in-flight copies/MMAs before exit).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait_sleep(bar, parity, 1000000u)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

__device__ __forceinline__ void st_f32x4(float *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<float4 *>(p) = make_float4(__uint_as_float(a), __uint_as_float(b), __uint_as_float(c),
                                               __uint_as_float(d));
}

template <int BN, bool GENERAL>
__global__ void __launch_bounds__(Cfg<BN, GENERAL>::kThreads, 1)
    w4a16_gemm_kernel(const __grid_constant__ CUtensorMap x_map, const Params p) {
  using C = Cfg<BN, GENERAL>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ __align__(8) uint64_t aempty_bar[C::kASlots];
  __shared__ __align__(8) uint64_t dfull_bar[C::kDBufs];
  __shared__ __align__(8) uint64_t dempty_bar[C::kDBufs];
  __shared__ __align__(8) uint64_t drain_bar[C::kDqGroups];
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t abort_sh;
  __shared__ uint32_t last_sh;

  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  volatile uint32_t *abort_flag = &abort_sh;

  const int cta = blockIdx.x;
  const int64_t u0 = range_begin(p, cta);
  const int nu = static_cast<int>(range_begin(p, cta + 1) - u0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < C::kASlots; ++a) mbar_init(smem_u32(&aempty_bar[a]), 1);
    for (int d = 0; d < C::kDBufs; ++d) {
      mbar_init(smem_u32(&dfull_bar[d]), C::kDqGroups);
      mbar_init(smem_u32(&dempty_bar[d]), 128);
    }
    for (int w = 0; w < C::kDqGroups; ++w) mbar_init(smem_u32(&drain_bar[w]), 1);
    abort_sh = 0;
    last_sh = 0;
    fence_mbar_init();
  }
  if (warp == C::kDqWarp0) {
    tmem_alloc(smem_u32(&tmem_base_sh), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&x_map);
  tc_fence_before();
  __syncwarp();
  cta_sync_all();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp < C::kProducers) {
    // ------------------------------------------------------------ producers
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first();
      // producer warp pw loads units pw, pw + P, ...; coordinates advance without divisions:
      // u = (t * MT + mt) * KB + kb
      const int pw = warp;
      int kb = static_cast<int>((u0 + pw) % p.KB);
      const int tile0 = static_cast<int>((u0 + pw) / p.KB);
      int t = tile0 / p.MT;
      int mt = tile0 % p.MT;
      int i = pw;
      for (; i < nu; i += C::kProducers) {
        const int s = i % C::kStages;
        const uint32_t ph = (i / C::kStages) & 1;
        if (!mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1, abort_flag, p.err)) break;
        const int kfirst = kb * kTK;
        const int jlo = min(kfirst / p.g, p.G - 1);
        int nrec = 1;
        if (GENERAL) nrec = min((kfirst + kTK - 8) / p.g, p.G - 1) - jlo + 1;
        const uint32_t stage = smem_base + s * C::kStageBytes;
        const uint32_t bar = smem_u32(&full_bar[s]);
        mbar_arrive_expect_tx(bar, C::kXBytes + kTileBytes + nrec * kRecBytes);
        tma_load_2d(stage, &x_map, kfirst, mt * BN, bar);
        bulk_g2s(stage + C::kXBytes, p.codes + (static_cast<int64_t>(t) * p.KB + kb) * kTileBytes, kTileBytes, bar,
                 pol_stream);
        bulk_g2s(stage + C::kXBytes + kTileBytes, p.meta + (static_cast<int64_t>(t) * p.G + jlo) * kRecBytes,
                 nrec * kRecBytes, bar, pol_stream);
        kb += C::kProducers;
        while (kb >= p.KB) {
          kb -= p.KB;
          if (++mt == p.MT) {
            mt = 0;
            ++t;
          }
        }
      }
      if (*abort_flag) {
        // let every copy this warp issued land before the CTA's shared memory goes away
        for (int j = i - C::kProducers; j >= 0 && j >= i - C::kStages; j -= C::kProducers)
          drain_wait(smem_u32(&full_bar[j % C::kStages]), (j / C::kStages) & 1);
      }
    }
  } else if (warp < C::kEpiWarp0) {
    // ------------------------------------------------- dequant + MMA issue
    // Group dq takes K blocks i = dq, dq + kDqGroups, ...: thread r dequantizes weight row r into
    // a tensor-memory slot; after a group barrier the group's first thread issues the block's four
    // MMAs into the group's own accumulator and commits the stage and the slot. That thread also
    // keeps the group's part of the accumulator protocol: before the group's first block of a
    // segment (tile) it waits for the segment's accumulator set to be free, and it commits dfull
    // once for every segment of the CTA's range when the group is past it (a commit covers the
    // committing thread's own MMAs, so the same thread issues and commits).
    const int dq = (warp - C::kDqWarp0) / 4;
    const bool issuer = warp == C::kDqWarp0 + 4 * dq && lane == 0;
    const int lq = warp % 4;  // tensor-memory lane quarter this warp may access
    const int r = lq * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(lq * 32) << 16;
    constexpr uint32_t idesc = idesc_f16_f32(128, BN);
    const int64_t tile0 = u0 / p.KB;
    const int seg_count = static_cast<int>((u0 + nu - 1) / p.KB - tile0) + 1;
    int kb = static_cast<int>((u0 + dq) % p.KB);                  // K block of unit i
    int seg_i = static_cast<int>((u0 + dq) / p.KB - tile0);        // segment of unit i
    int prev_seg = -1;       // segment of this group's previous block
    int seg_closed = 0;      // segments below this one have had this group's dfull commit
    int seg_freed = 0;       // segments below this one are known to be read out by the epilogue
    bool issue_ok = true;    // the issuer's own waits (shared with the group at the next barrier)
    for (int i = dq; i < nu; i += C::kDqGroups) {
      const int s = i % C::kStages;
      const int a = i % C::kASlots;
      const int db = seg_i % C::kDBufs;
      bool okw = warp_wait(smem_u32(&full_bar[s]), (i / C::kStages) & 1, abort_flag, p.err);
      uint32_t out[32];
      if (okw) {
        const uint32_t codes = smem_base + s * C::kStageBytes + C::kXBytes;
        const uint32_t meta = codes + kTileBytes;
        const uint4 w0 = lds128(codes + r * 16);
        const uint4 w1 = lds128(codes + 2048 + r * 16);
        const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
        if (!GENERAL) {
          const uint32_t z = (lds8(meta + 256 + r / 2) >> (4 * (r & 1))) & 0xFu;
          const GroupConsts c = group_consts(lds16(meta + 2 * r), z);
#pragma unroll
          for (int ci = 0; ci < 8; ++ci) dequant_word(words[ci], c, &out[4 * ci]);
        } else {
          const int kfirst = kb * kTK;
          const int jlo = min(kfirst / p.g, p.G - 1);
          int j = jlo;
#pragma unroll
          for (int ci = 0; ci < 8; ++ci) {
            const int kc = kfirst + 8 * ci;
            if (kc >= (j + 1) * p.g && j < p.G - 1) ++j;  // g >= 8: at most one group boundary per 8 codes
            const uint32_t rec = meta + (j - jlo) * kRecBytes;
            const uint32_t z = (lds8(rec + 256 + r / 2) >> (4 * (r & 1))) & 0xFu;
            dequant_word(words[ci], group_consts(lds16(rec + 2 * r), z), &out[4 * ci]);
          }
        }
        // the slot's previous block (i - kASlots) is this group's too: its MMAs must be done
        okw = warp_wait(smem_u32(&aempty_bar[a]), ((i / C::kASlots) & 1) ^ 1, abort_flag, p.err);
      }
      if (okw) {
        tc_fence_after();
        tmem_st_32x32b_x32(tmem + lane_addr + C::kACol0 + a * 32, out);
        tmem_wait_st();
        tc_fence_before();
      }
      // one decision for the whole group: go on together or stop together
      if (!named_bar_and(2 + dq, 128, okw && issue_ok)) break;
      if (issuer) {
        for (; seg_closed < seg_i; ++seg_closed) mma_commit(smem_u32(&dfull_bar[seg_closed % C::kDBufs]));
        const bool first = prev_seg != seg_i;
        // before the first block of segment seg_i, the accumulator set it reuses must be read out,
        // i.e. segment seg_i - kDBufs finished. The group may have had no block in some segments:
        // wait for every segment's phase in order, so no parity wait can skip a phase.
        for (; first && issue_ok && seg_freed <= seg_i - C::kDBufs; ++seg_freed)
          issue_ok = mbar_wait(smem_u32(&dempty_bar[seg_freed % C::kDBufs]), (seg_freed / C::kDBufs) & 1,
                               abort_flag, p.err);
        if (issue_ok) {
          tc_fence_after();
          const uint64_t bdesc = sw128_kmajor_desc(smem_base + s * C::kStageBytes);
          const uint32_t dcol = tmem + (db * C::kDqGroups + dq) * C::kDStride;
#pragma unroll
          for (int kk = 0; kk < kTK / 16; ++kk) {
            // A: 128 x 16 fp16 in tensor memory (8 columns per 16 K); B: 16 K-columns of the x tile
            mma_f16_ts(dcol, tmem + C::kACol0 + a * 32 + kk * 8, bdesc + static_cast<uint64_t>(kk * 2), idesc,
                       (first && kk == 0) ? 0u : 1u);
          }
          mma_commit(smem_u32(&empty_bar[s]));
          mma_commit(smem_u32(&aempty_bar[a]));
        }
      }
      prev_seg = seg_i;
      kb += C::kDqGroups;
      while (kb >= p.KB) {
        kb -= p.KB;
        ++seg_i;
      }
    }
    if (issuer) {
      // segments after the group's last block (or all of them if it had none) still need its commit
      for (; seg_closed < seg_count; ++seg_closed) mma_commit(smem_u32(&dfull_bar[seg_closed % C::kDBufs]));
      if (*abort_flag) {
        mma_commit(smem_u32(&drain_bar[dq]));
        drain_wait(smem_u32(&drain_bar[dq]), 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int lq = warp % 4;
    const int r = lq * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(lq * 32) << 16;
    const int64_t u_end = u0 + nu;
    int seg = 0;
    for (int64_t u = u0; u < u_end; ++seg) {
      const int tile = static_cast<int>(u / p.KB);
      const int64_t tile_end = static_cast<int64_t>(tile + 1) * p.KB;
      const int64_t seg_end = min(u_end, tile_end);
      const bool whole = (u % p.KB == 0) && seg_end == tile_end;
      const int db = seg % C::kDBufs;
      // the epilogue waits a whole tile for its accumulator: sleep longer between looks
      if (!warp_wait(smem_u32(&dfull_bar[db]), (seg / C::kDBufs) & 1, abort_flag, p.err, 1024)) break;
      tc_fence_after();
      const int t = tile / p.MT;
      const int m0 = (tile % p.MT) * BN;
      const int m_end = min(p.M, m0 + BN);
      const int n = t * kTN + r;
      float *piece = p.pieces + ((static_cast<int64_t>(cta) * 2 + (seg == 0 ? 0 : 1)) * kTN + r) * BN;
      // dequant groups that took a block of this segment: all of them unless the segment is shorter
      const int i_first = static_cast<int>(u - u0);
      const int seg_len = static_cast<int>(seg_end - u);
      uint32_t contrib = 0;
      for (int j = 0; j < seg_len && j < C::kDqGroups; ++j) contrib |= 1u << ((i_first + j) % C::kDqGroups);
      const int w_first = __ffs(contrib) - 1;
#pragma unroll 1
      for (int c0 = 0; c0 < BN && m0 + c0 < m_end; c0 += 16) {
        uint32_t v[16];
        const uint32_t dbase = tmem + lane_addr + db * C::kDqGroups * C::kDStride + c0;
        tmem_ld_32x32b_x16(dbase + w_first * C::kDStride, v);
        tmem_wait_ld();
#pragma unroll 1
        for (int w = w_first + 1; w < C::kDqGroups; ++w) {  // the groups' partial sums, in a fixed order
          if (!(contrib >> w & 1u)) continue;
          uint32_t v2[16];
          tmem_ld_32x32b_x16(dbase + w * C::kDStride, v2);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) + __uint_as_float(v2[e]));
        }
        if (whole) {
          if (n < p.N) {
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (m0 + c0 + e < m_end)
                p.y[static_cast<int64_t>(m0 + c0 + e) * p.N + n] = __float2half_rn(__uint_as_float(v[e]));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 16; e += 4) st_f32x4(piece + c0 + e, v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&dempty_bar[db]));
      if (!whole) {
        // the last CTA to finish a piece of this tile adds all pieces in K order and writes y
        const int c_first = owner_of(p, static_cast<int64_t>(tile) * p.KB);
        const int c_last = owner_of(p, tile_end - 1);
        __threadfence();
        __syncwarp();
        named_bar_sync(1, 128);
        if (r == 0) {
          const uint32_t old = atomicAdd(&p.counters[tile], 1u);
          last_sh = (old == static_cast<uint32_t>(c_last - c_first)) ? 1u : 0u;
        }
        __syncwarp();
        named_bar_sync(1, 128);
        if (last_sh) {
          __threadfence();
          // all pieces' loads of a 2-column slice are in flight together, then added in K order
          const int npieces = c_last - c_first + 1;
          uint32_t slot_mask = 0;  // bit q: piece q is CTA (c_first + q)'s second slot
          for (int q = 0; q < npieces; ++q)
            if (range_begin(p, c_first + q) / p.KB != tile) slot_mask |= 1u << q;
          const float *base = p.pieces + (static_cast<int64_t>(c_first) * 2 * kTN + r) * BN;
#pragma unroll 1
          for (int c0 = 0; c0 < BN && m0 + c0 < m_end; c0 += 2) {
            float2 v[kMaxPieces];
#pragma unroll
            for (int q = 0; q < kMaxPieces; ++q)
              if (q < npieces)
                v[q] = __ldcg(reinterpret_cast<const float2 *>(base + (2 * q + (slot_mask >> q & 1u)) * kTN * BN + c0));
            float2 acc = v[0];
#pragma unroll
            for (int q = 1; q < kMaxPieces; ++q)
              if (q < npieces) {
                acc.x += v[q].x;
                acc.y += v[q].y;
              }
            if (n < p.N) {
              if (m0 + c0 < m_end) p.y[static_cast<int64_t>(m0 + c0) * p.N + n] = __float2half_rn(acc.x);
              if (m0 + c0 + 1 < m_end) p.y[static_cast<int64_t>(m0 + c0 + 1) * p.N + n] = __float2half_rn(acc.y);
            }
          }
          if (r == 0) p.counters[tile] = 0u;  // ready for the next call
        }
      }
      u = seg_end;
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

// x [M, K] fp16 row-major, boxes of 64 (K) x BN (rows), 128-byte swizzle, zero fill outside.
bool make_x_map(CUtensorMap *map, const void *x, int64_t M, int64_t K, int bn) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTK), static_cast<cuuint32_t>(bn)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(x), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool GENERAL>
cudaError_t launch_t(const CUtensorMap &map, const Params &p, int ctas, cudaStream_t stream) {
  using C = Cfg<BN, GENERAL>;
  auto kern = w4a16_gemm_kernel<BN, GENERAL>;
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
  kern<<<ctas, C::kThreads, C::kSmemBytes, stream>>>(map, p);
  return cudaGetLastError();
}

template <bool GENERAL>
cudaError_t launch_bn(int bn, const CUtensorMap &map, const Params &p, int ctas, cudaStream_t stream) {
  switch (bn) {
    case 16: return launch_t<16, GENERAL>(map, p, ctas, stream);
    case 32: return launch_t<32, GENERAL>(map, p, ctas, stream);
    case 64: return launch_t<64, GENERAL>(map, p, ctas, stream);
    case 128: return launch_t<128, GENERAL>(map, p, ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool make_gemm_plan(int64_t M, int64_t N, int64_t K, int32_t g, int block_n, int ctas, int schedule,
                    int num_sms, GemmPlan *plan) {
  (void)g;
  int bn = block_n;
  if (bn == 0) bn = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
  if (bn != 16 && bn != 32 && bn != 64 && bn != 128) return false;
  if (ctas < 0 || ctas > 65535 || schedule < 0 || schedule > 2) return false;
  const int64_t mt = cdiv(M, bn), nt = cdiv(N, kTN), kb = cdiv(K, kTK);
  const int64_t tiles = mt * nt;
  const int64_t units = tiles * kb;
  if (tiles > 0x7FFFFFFF || units > (int64_t{1} << 40)) return false;
  int64_t P = ctas > 0 ? ctas : (num_sms > 0 ? num_sms : 148);
  // whole-tile scheduling when every CTA gets many tiles (imbalance <= 1/8) or the tiles divide
  // evenly; otherwise stream-K over 64-wide K blocks, which needs the partial-tile fixup
  bool whole = schedule == 2 || (schedule == 0 && (tiles >= 8 * P || (tiles >= P && tiles % P == 0)));
  const int64_t gran = whole ? kb : 1;
  const int64_t grains = units / gran;
  P = std::min(P, grains);
  if (!whole) {
    // the fixup adds at most kMaxPieces pieces per tile: shrink the grid until no tile is cut into more
    // (CTA c owns units [c*U/P, (c+1)*U/P); the owner of unit u is ((u + 1) * P - 1) / U)
    auto max_pieces = [&](int64_t PP) {
      int64_t worst = 1;
      for (int64_t tt = 0; tt < tiles; ++tt) {
        const int64_t first = ((tt * kb + 1) * PP - 1) / units;
        const int64_t last = (((tt + 1) * kb) * PP - 1) / units;
        worst = std::max(worst, last - first + 1);
      }
      return worst;
    };
    while (P > 1 && max_pieces(P) > kMaxPieces) --P;
  }
  plan->block_n = bn;
  plan->m_tiles = static_cast<int>(mt);
  plan->n_tiles = static_cast<int>(nt);
  plan->k_blocks = static_cast<int>(kb);
  plan->ctas = static_cast<int>(P);
  plan->gran = static_cast<int>(gran);
  plan->grains = grains;
  plan->counters_offset = 256;
  const size_t counters_bytes = static_cast<size_t>(cdiv(tiles * 4, 256) * 256);
  plan->pieces_offset = plan->counters_offset + counters_bytes;
  const size_t piece_bytes = whole ? 0 : static_cast<size_t>(P * 2 * kTN * bn * 4);
  plan->workspace_bytes = plan->pieces_offset + piece_bytes;
  return true;
}

cudaError_t launch_gemm(const void *x, const void *packed, int64_t M, int64_t N, int64_t K, int32_t g, void *y,
                        void *workspace, const GemmPlan &plan, cudaStream_t stream, bool *encode_failed) {
  *encode_failed = false;
  CUtensorMap map;
  if (!make_x_map(&map, x, M, K, plan.block_n)) {
    *encode_failed = true;
    return cudaErrorInvalidValue;
  }
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  Params p;
  p.codes = static_cast<const uint8_t *>(packed);
  p.meta = p.codes + static_cast<int64_t>(plan.n_tiles) * plan.k_blocks * kTileBytes;
  p.y = static_cast<__half *>(y);
  p.pieces = reinterpret_cast<float *>(ws + plan.pieces_offset);
  p.counters = reinterpret_cast<uint32_t *>(ws + plan.counters_offset);
  p.err = reinterpret_cast<uint32_t *>(ws);
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.g = g;
  p.G = static_cast<int>(cdiv(K, g));
  p.NT = plan.n_tiles;
  p.KB = plan.k_blocks;
  p.MT = plan.m_tiles;
  p.P = plan.ctas;
  p.gran = plan.gran;
  p.grains = plan.grains;
  const bool general = (g % kTK) != 0;
  return general ? launch_bn<true>(plan.block_n, map, p, plan.ctas, stream)
                 : launch_bn<false>(plan.block_n, map, p, plan.ctas, stream);
}

}  // namespace w4
