// w4a16_gemm for decode batches (block_n 8, M <= 8): the dequantized weights go straight into the A
// fragments of register-operand tensor-core MMAs (mma.sync m16n8k16, fp16 in, fp32 accumulate),
// so a weight is loaded once as 4-bit codes, turned into fp16 in registers and consumed there:
// no shared- or tensor-memory round trip, no MMA-issuing thread, one handshake per warp and stage.
//
// Schedule, weight stream and fixup are the tensor-core kernel's (gemm_common.cuh): persistent
// stream-K over (128-row weight tile x BN-token tile, 256-wide K stage) units, two producer warps
// moving each stage's x sub-tiles (TMA, 128-byte swizzle), 16 KB of codes and the group records.
//
// Consumers: 16 warps in two sets of 8 that take the stages in turn (even / odd). Warp (q, sl) of
// set q handles weight rows 16 sl .. 16 sl + 15 (one MMA slab) over all four K blocks of its
// stages: 16 code words per thread and stage, so the per-stage costs (wait, release, addresses,
// the groups' scales and zeros) are spread over 128 weights. Per block it loads 2 rows x 2 code
// words per thread and the x fragments of the block, dequantizes and issues 4 k16 steps x BN/8
// MMAs. The tile layout of w4_repack serves these fragments directly once the 16 k of an MMA step
// are taken in a permuted order (the same order on both operands, so the dot product is
// unchanged): in step p, lane (g, t) holds the code pairs p of its row's words t and t + 4 (k =
// 8t + 2p, +1 and 32 + 8t + 2p, +1 of the block) and the matching x pairs.
//
// Scale: with g a multiple of 64 a K block lies in one group, so the MMAs run on the exact
// integers q - z (fp16) and the group's fp32 partial is scaled by s once per row (more accurate
// than rounding (q - z) * s to fp16, and 9 instead of 13 instructions per 8 weights). Any other g
// rounds (q - z) * s to fp16 per 8 codes, looking the group up per code word.
//
// At the end of a tile segment the two warps of a slab add their partials through shared memory
// (set 0 + set 1: deterministic) and write y, or an fp32 piece of a tile cut between CTAs; the
// owner of a cut tile adds the other CTAs' pieces first (gemm_common.cuh). This is the split-K-in-the-CTA, stream-K-across-CTAs decode
// path; Marlin's register-level dequant into MMA fragments (Marlin post) on sm_103a.
#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "gemm_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace w4 {
namespace {

using namespace detail;

enum RfMode { kRfScaleOut = 0, kRfGeneral = 1 };  // g % 64 == 0, or any g

template <int NB8, int MODE>
struct RfCfg {
  static constexpr int BN = 8 * NB8;  // tokens per tile
  static constexpr int kXSub = BN * 128;
  static constexpr int kXBytes = kSB * kXSub;
  static constexpr int kCodeBytes = kSB * kTileBytes;
  static constexpr int kMaxRecs = MODE == kRfGeneral ? kStageK / 8 + 1 : kStageK / 64 + 1;
  static constexpr int kStageBytes = (kXBytes + kCodeBytes + kMaxRecs * kRecBytes + 1023) / 1024 * 1024;
  static constexpr int kConsumers = 16;
  static constexpr int kConsumerWarp0 = 2;
  static constexpr int kThreads = (kConsumerWarp0 + kConsumers) * 32;
  static constexpr int kSetWarps = kConsumers / 2;  // consumer warps per stage
  // partial sums of the set-1 warps, per (slab, lane): NB8 x 4 floats
  static constexpr int kVals = 4 * NB8;
  static constexpr int kRedBytes = 8 * 32 * kVals * 4;
  static constexpr int kSmemBudget = 224 * 1024 - kRedBytes;
  static constexpr int kStagesRaw = kSmemBudget / kStageBytes > 10 ? 10 : kSmemBudget / kStageBytes;
  static constexpr int kStages = kStagesRaw / 2 * 2;  // two producers take the stages in turn
  static constexpr int kSmemBytes = kStages * kStageBytes + kRedBytes + 1024;
  static_assert(kStages >= 4, "stage ring");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(NB8 == 1 || NB8 == 2, "tokens per tile");
};

// Shared-memory loads at a register address plus a constant offset (folded into the instruction).
template <int OFF>
__device__ __forceinline__ uint32_t lds32_at(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1+%2];" : "=r"(v) : "r"(addr), "n"(OFF));
  return v;
}
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
__device__ __forceinline__ uint4 lds128_at(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4+%5];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr), "n"(OFF));
  return v;
}

// D (+)= A . B, m16n8k16, A row-major fp16 (4 regs), B column-major fp16 (2 regs), fp32 D.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                         const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint32_t component(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// The two rows a thread serves in one slab (rows R and R + 8), as dequant constants and fp32 scales.
struct SlabConsts {
  GroupConsts a, b;
  float sa, sb;
};

// Scale outside: zero points of rows R, R + 8 from the record at `rec` (scales as fp32).
__device__ __forceinline__ SlabConsts slab_consts_int(uint32_t rec, uint32_t zero_off, uint32_t zero_shift,
                                                      uint32_t scale_off) {
  SlabConsts c;
  c.a = group_consts(0u, (lds8_at<0>(rec + zero_off) >> zero_shift) & 0xFu);
  c.b = group_consts(0u, (lds8_at<4>(rec + zero_off) >> zero_shift) & 0xFu);
  c.sa = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16_at<0>(rec + scale_off))));
  c.sb = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16_at<16>(rec + scale_off))));
  return c;
}

// Full constants (scale applied in the dequant) of rows R, R + 8 from the record at `rec`.
__device__ __forceinline__ SlabConsts slab_consts_scaled(uint32_t rec, uint32_t zero_off, uint32_t zero_shift,
                                                         uint32_t scale_off) {
  SlabConsts c;
  c.a = group_consts(lds16_at<0>(rec + scale_off), (lds8_at<0>(rec + zero_off) >> zero_shift) & 0xFu);
  c.b = group_consts(lds16_at<16>(rec + scale_off), (lds8_at<4>(rec + zero_off) >> zero_shift) & 0xFu);
  c.sa = c.sb = 1.0f;
  return c;
}

// One K block (BB = 0 or 1 of the warp's K half) of one slab: 4 code words per thread (rows R and
// R + 8, words t and t + 4), dequantized into the A fragments of 4 k16 steps, times the x fragments
// of the block's BN tokens, accumulated into acc. c_lo / c_hi: the constants for the words t (k
// 8t ..) and t + 4 (k 32 + 8t ..): the same group unless g is not a multiple of 64.
template <int NB8, int BB, int XSUB, bool SCALED>
__device__ __forceinline__ void slab_block(uint32_t codes, uint32_t xa, uint32_t xb, const SlabConsts &c_lo,
                                           const SlabConsts &c_hi, float (&acc)[NB8][4]) {
  constexpr int kC = BB * kTileBytes;
  const uint32_t w_a_lo = lds32_at<kC>(codes);               // row R, word t
  const uint32_t w_b_lo = lds32_at<kC + 128>(codes);         // row R + 8, word t
  const uint32_t w_a_hi = lds32_at<kC + 2048>(codes);        // row R, word t + 4
  const uint32_t w_b_hi = lds32_at<kC + 2048 + 128>(codes);  // row R + 8, word t + 4
  uint32_t oa_lo[4], ob_lo[4], oa_hi[4], ob_hi[4];
  if (SCALED) {
    dequant_word(w_a_lo, c_lo.a, oa_lo);
    dequant_word(w_b_lo, c_lo.b, ob_lo);
    dequant_word(w_a_hi, c_hi.a, oa_hi);
    dequant_word(w_b_hi, c_hi.b, ob_hi);
  } else {
    dequant_word_int(w_a_lo, c_lo.a, oa_lo);
    dequant_word_int(w_b_lo, c_lo.b, ob_lo);
    dequant_word_int(w_a_hi, c_hi.a, oa_hi);
    dequant_word_int(w_b_hi, c_hi.b, ob_hi);
  }
#pragma unroll
  for (int nb = 0; nb < NB8; ++nb) {
    // token g + 8 nb: its x chunks t and t + 4 of the block (128-byte rows, 8 tokens per 1 KB)
    const uint4 xlo = nb == 0 ? lds128_at<BB * XSUB>(xa) : lds128_at<BB * XSUB + 1024>(xa);
    const uint4 xhi = nb == 0 ? lds128_at<BB * XSUB>(xb) : lds128_at<BB * XSUB + 1024>(xb);
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      const uint32_t a[4] = {oa_lo[pp], ob_lo[pp], oa_hi[pp], ob_hi[pp]};
      mma16816(acc[nb], a, component(xlo, pp), component(xhi, pp), acc[nb]);
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

template <int NB8, int MODE>
__global__ void __launch_bounds__(RfCfg<NB8, MODE>::kThreads, 1)
    w4a16_gemm_rf_kernel(const __grid_constant__ CUtensorMap x_map, const Params p) {
  using C = RfCfg<NB8, MODE>;
  constexpr int S = C::kStages;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[S];
  __shared__ __align__(8) uint64_t empty_bar[S];
  __shared__ __align__(8) uint64_t own_bar;  // the owner's wait for the other pieces is over
  __shared__ uint32_t abort_sh;
  __shared__ int npieces_sh;  // pieces of the cut tile the CTA's last segment owns (-1: failed)

  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  float *red = reinterpret_cast<float *>(smem_raw + (smem_base - smem_u32(smem_raw)) + S * C::kStageBytes);
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
      mbar_init(smem_u32(&empty_bar[s]), C::kSetWarps);  // one arrival per warp of the stage's set
    }
    mbar_init(smem_u32(&own_bar), 1);
    abort_sh = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&x_map);
  __syncwarp();
  cta_sync_all();
  // the next grid in the stream may start launching; every role waits for the previous grid before
  // touching global memory it may have written (the producer inside produce_stages)
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp < C::kConsumerWarp0) {
    produce_stages<BN, S, C::kStageBytes>(&x_map, p, u0, nst, warp, lane, smem_base, full_bar, empty_bar, 0, 1,
                                          abort_flag);
    // The CTA's last segment owns a cut tile when it holds the tile's first stages but not its last
    // (gemm_common.cuh). Producer 0, idle once its copies are issued, waits for the tile's other
    // pieces while the consumers finish, so the owner's epilogue does not wait.
    const int64_t ulast = u0 + nst - 1;
    const int64_t lt0 = nst > 0 ? ulast / p.KS * p.KS : 0;
    if (warp == 0 && lane == 0 && nst > 0 && lt0 >= u0 && ulast < lt0 + p.KS - 1) {
      const int tile = static_cast<int>(ulast / p.KS);
      const int np = tile_pieces(p, tile, cta);
      npieces_sh = wait_pieces(p, tile, np, abort_flag) ? np : -1;
      mbar_arrive(smem_u32(&own_bar));
    }
  } else {
    const int cw = warp - C::kConsumerWarp0;
    const int q = (cw >> 2) & 1;                 // stage set: stages of parity q (two warps per SMSP)
    const int sl = (cw & 3) | ((cw >> 3) << 2);  // slab: rows 16 sl .. 16 sl + 15
    const int g = lane >> 2;
    const int t = lane & 3;
    const int tid = cw * 32 + lane;  // 0 .. 511
    // per-thread offsets into a stage, fixed for the whole loop; the per-row / per-block / per-token
    // differences are constants folded into the loads
    const int row0 = 16 * sl + g;  // rows row0 and row0 + 8
    const uint32_t code_off = C::kXBytes + row0 * 16 + 4 * t;
    const uint32_t zero_off = 256 + row0 / 2;  // (+4 for row0 + 8)
    const uint32_t zero_shift = 4 * (row0 & 1);
    const uint32_t scale_off = 2 * row0;  // (+16 for row0 + 8)
    // x of token g, 128-byte swizzle: chunk c of row n sits at (c ^ (n % 8)) * 16 (n % 8 == g)
    const uint32_t x_off_lo = 128 * g + ((t ^ g) << 4);
    const uint32_t x_off_hi = 128 * g + (((t + 4) ^ g) << 4);
    griddep_wait();  // y and the workspace may still be in use by the previous grid

    float tot[NB8][4];
    zero_acc<NB8>(tot);
    StageIter it;
    it.init(p, u0);
    int seg = 0;
    bool ok = true;  // a failed wait is shared at the segment end, where all stop together
    for (int i = 0; i < nst;) {
      // one tile segment: local stages i .. i + seg_len - 1 hold stages ks0 .. of tile it.tile
      const int tile = it.tile;
      const int ks0 = it.ks;
      const int seg_len = min(nst - i, p.KS - ks0);
      for (int r = (q - i) & 1; r < seg_len && ok; r += 2) {
        const int ii = i + r;
        const int ks = ks0 + r;
        const int s = ii % S;
        ok = warp_wait(smem_u32(&full_bar[s]), (ii / S) & 1, abort_flag, p.err);
        if (!ok) break;
        const int nbk = stage_blocks(p, ks);  // 1 .. 4 K blocks in the stage
        const uint32_t stage = smem_base + s * C::kStageBytes;
        const uint32_t codes = stage + code_off;
        const uint32_t xa = stage + x_off_lo;
        const uint32_t xb = stage + x_off_hi;
        const uint32_t recs = stage + C::kXBytes + C::kCodeBytes;
        const int k0 = ks * kStageK;
        const int jlo = p.gdiv.div(k0);  // the stage's first group record
        if (MODE == kRfScaleOut) {
          // g >= 64: a block lies in one group and the next group starts at most one block later
          float acc[NB8][4];
          zero_acc<NB8>(acc);
          int knext = (jlo + 1) * p.g;  // K where the next group starts
          uint32_t rec = recs;
          SlabConsts c = slab_consts_int(rec, zero_off, zero_shift, scale_off);
          slab_block<NB8, 0, C::kXSub, false>(codes, xa, xb, c, c, acc);
#pragma unroll
          for (int bb = 1; bb < kSB; ++bb) {
            if (bb < nbk) {
              if (k0 + bb * kTK >= knext) {  // block bb starts a new group
                flush_scaled<NB8>(tot, acc, c);
                zero_acc<NB8>(acc);
                knext += p.g;
                rec += kRecBytes;
                c = slab_consts_int(rec, zero_off, zero_shift, scale_off);
              }
              if (bb == 1) slab_block<NB8, 1, C::kXSub, false>(codes, xa, xb, c, c, acc);
              if (bb == 2) slab_block<NB8, 2, C::kXSub, false>(codes, xa, xb, c, c, acc);
              if (bb == 3) slab_block<NB8, 3, C::kXSub, false>(codes, xa, xb, c, c, acc);
            }
          }
          flush_scaled<NB8>(tot, acc, c);
        } else {
          // codes past K (zero, against zero x) take the last group's record, which the stage holds
#pragma unroll
          for (int bb = 0; bb < kSB; ++bb) {
            if (bb < nbk) {
              const int kb0 = k0 + bb * kTK;
              const uint32_t r_lo = recs + (min(p.gdiv.div(kb0 + 8 * t), p.G - 1) - jlo) * kRecBytes;
              const uint32_t r_hi = recs + (min(p.gdiv.div(kb0 + 32 + 8 * t), p.G - 1) - jlo) * kRecBytes;
              const SlabConsts c_lo = slab_consts_scaled(r_lo, zero_off, zero_shift, scale_off);
              const SlabConsts c_hi = slab_consts_scaled(r_hi, zero_off, zero_shift, scale_off);
              if (bb == 0) slab_block<NB8, 0, C::kXSub, true>(codes, xa, xb, c_lo, c_hi, tot);
              if (bb == 1) slab_block<NB8, 1, C::kXSub, true>(codes, xa, xb, c_lo, c_hi, tot);
              if (bb == 2) slab_block<NB8, 2, C::kXSub, true>(codes, xa, xb, c_lo, c_hi, tot);
              if (bb == 3) slab_block<NB8, 3, C::kXSub, true>(codes, xa, xb, c_lo, c_hi, tot);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty_bar[s]));
      }

      // ------------------------------------------------ end of a tile segment
      // one decision for all consumer warps: go on together or stop together (never leave a warp
      // waiting at a barrier the others no longer reach)
      if (!named_bar_and(1, 32 * C::kConsumers, ok)) break;  // also: the previous partials were read
      const bool whole = ks0 == 0 && seg_len == p.KS;
      const bool owner = !whole && ks0 == 0;  // holds a cut tile's first stages (the CTA's last segment)
      // the warps of set 1 hand their partial sums to the warp of set 0 of their slab
      float *mine = red + sl * 32 * C::kVals + lane;
      if (q == 1) {
#pragma unroll
        for (int nb = 0; nb < NB8; ++nb)
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) mine[(nb * 4 + cc) * 32] = tot[nb][cc];
      }
      bool have_pieces = true;
      if (owner && tid == 0)
        have_pieces = mbar_wait(smem_u32(&own_bar), 0, abort_flag, p.err) && npieces_sh > 0;
      if (!named_bar_and(1, 32 * C::kConsumers, have_pieces)) break;
      const int npieces = owner ? npieces_sh : 1;
      if (q == 0) {
        const int m0 = (tile % p.MT) * BN;
        const int n0 = (tile / p.MT) * kTN;
        float *piece = p.pieces + (static_cast<int64_t>(cta) * 2 + (seg == 0 ? 0 : 1)) * BN * kTN;
#pragma unroll
        for (int nb = 0; nb < NB8; ++nb) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float v = tot[nb][c] + mine[(nb * 4 + c) * 32];
            const int row = row0 + 8 * (c >> 1);
            const int tok = 8 * nb + 2 * t + (c & 1);
            for (int pc = 1; pc < npieces; ++pc)  // the owner adds the later pieces in K order
              v += __ldcg(piece_of<BN, 1>(p, cta + pc, 0) + tok * kTN + row);
            if (whole || owner) {
              if (n0 + row < p.N && m0 + tok < p.M)
                p.y[static_cast<int64_t>(m0 + tok) * p.N + n0 + row] = __float2half_rn(v);
            } else {
              __stcg(piece + tok * kTN + row, v);
            }
          }
        }
      }
      if (!whole && !owner) {
        // a later piece of a cut tile: its stores are ordered (barrier) before one thread's release count
        named_bar_sync(1, 32 * C::kConsumers);
        if (tid == 0) red_add_release_gpu(&p.counters[tile]);
      }
      zero_acc<NB8>(tot);
      i += seg_len;
      it.advance(p, seg_len);
      ++seg;
    }
  }
  __syncwarp();
  cta_sync_all();
}

template <int NB8, int MODE>
cudaError_t launch_rf_t(const CUtensorMap &map, const Params &p, int ctas, cudaStream_t stream) {
  using C = RfCfg<NB8, MODE>;
  auto kern = w4a16_gemm_rf_kernel<NB8, MODE>;
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
  return launch_programmatic(kern, ctas, C::kThreads, C::kSmemBytes, stream, map, p);
}

}  // namespace

namespace detail {

cudaError_t launch_gemm_rf(const CUtensorMap &map, const Params &p, int nb8, bool general, int ctas,
                           cudaStream_t stream) {
  if (!general) {
    if (nb8 == 1) return launch_rf_t<1, kRfScaleOut>(map, p, ctas, stream);
  } else {
    if (nb8 == 1) return launch_rf_t<1, kRfGeneral>(map, p, ctas, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace detail
}  // namespace w4
