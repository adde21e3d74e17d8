// w4a16_gemm: y[M,N] = x[M,K] . dequant(Wq)[N,K]^T on sm_103a tensor cores.
//
// One CTA computes a 128 (weight rows n) x BN (activation rows m) tile of y^T
// over a range of K ("swap-AB": the weights sit on the MMA's M = 128 side, the
// tokens on its N side, so a batch of 1..16 tokens still fills an MMA).
//
// Warp roles (one CTA, 64 + 128 * kDqGroups threads):
//   warp 0, lane 0  producer: per 64-wide K block, one TMA tensor copy of the
//                   x tile (128-byte swizzle, zero fill outside [M, K]) and
//                   two bulk copies of the weight tile (4 KB of codes) and its
//                   group records, all completing on one mbarrier.
//   warp 1          allocates tensor memory; lane 0 issues tcgen05.mma.
//   warps 2..       dequant warpgroup(s): thread r owns weight row r; it turns
//                   the row's 64 codes into fp16 (q - z) * s and stores them
//                   into tensor memory (tcgen05.st), where they are the MMA's
//                   A operand; shared memory only ever holds 4-bit codes.
//                   After the K loop the same warps read the fp32 accumulator
//                   out of tensor memory and write y (or split-K partials).
//
// This is the GB300 form of the techniques the Marlin post lists (prefetch,
// activation reuse, asynchronous weight loads, dequant interleaved with the
// tensor-core work, tuned warp roles): the weight stream is a multi-stage
// TMA/mbarrier ring, each x tile is reused by all 128 weight rows, and the
// dequant warps run ahead of the asynchronous MMAs through a ring of tensor-
// memory slots.
//
// Split-K: with S > 1 the CTAs of one output tile each write fp32 partials to
// the workspace; the last CTA to arrive on the tile's counter adds them in
// split order 0..S-1 (deterministic) and writes y. Nothing ever waits on
// another CTA. Every mbarrier wait is bounded (ptx.cuh).
#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace w4 {
namespace {

constexpr int kMaxRecs = 9;  // group records one 64-wide K block can touch (g = 8: 8 groups)

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
  // Two CTAs per SM for BN <= 128 (about 110 KB of stages each), one for BN = 256.
  static constexpr int kSmemBudget = BN == 256 ? 200 * 1024 : 108 * 1024;
  static constexpr int kStagesRaw = kSmemBudget / kStageBytes;
  static constexpr int kStages = kStagesRaw > 12 ? 12 : kStagesRaw;
  static constexpr int kASlots = 4;  // tensor-memory slots of dequantized weights (32 columns each)
  static constexpr int kDCols = BN < 32 ? 32 : BN;
  static constexpr int kACol0 = kDCols;
  static constexpr int kTmemCols = pow2_at_least(kDCols + kASlots * 32);
  static constexpr int kDqGroups = 1;
  static constexpr int kThreads = 64 + 128 * kDqGroups;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;  // + alignment slack
  static_assert(kStages >= 2, "pipeline needs at least two stages");
  static_assert(kTmemCols <= 512, "tensor memory budget");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
};

struct Params {
  const uint8_t *codes;  // tile region of the packed weights
  const uint8_t *meta;   // group-record region of the packed weights
  __half *y;
  float *partials;  // [S][M][Npad]
  uint32_t *counters;
  uint32_t *err;
  int M, N, K, g, G, NT, KB, MT, S;
  int Npad;
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
                                          uint32_t *err) {
  const bool ok = mbar_wait(bar, parity, abort_flag, err);
  return __all_sync(0xffffffffu, ok);
}

// Waits ignoring the abort flag (used only to drain in-flight copies/MMAs before exit).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

template <int BN, bool GENERAL>
__global__ void __launch_bounds__(Cfg<BN, GENERAL>::kThreads, 1)
    w4a16_gemm_kernel(const __grid_constant__ CUtensorMap x_map, const Params p) {
  using C = Cfg<BN, GENERAL>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ __align__(8) uint64_t afull_bar[C::kASlots];
  __shared__ __align__(8) uint64_t aempty_bar[C::kASlots];
  __shared__ __align__(8) uint64_t acc_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ uint32_t abort_sh;
  __shared__ uint32_t last_sh;

  const uint32_t smem_base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  volatile uint32_t *abort_flag = &abort_sh;

  // tile of this CTA: m fastest, then n, then the K split
  int bid = blockIdx.x;
  const int mt = bid % p.MT;
  bid /= p.MT;
  const int t = bid % p.NT;
  const int sk = bid / p.NT;
  const int kb0 = static_cast<int>(static_cast<int64_t>(sk) * p.KB / p.S);
  const int kb1 = static_cast<int>(static_cast<int64_t>(sk + 1) * p.KB / p.S);
  const int nkb = kb1 - kb0;
  const int m0 = mt * BN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int a = 0; a < C::kASlots; ++a) {
      mbar_init(smem_u32(&afull_bar[a]), 128);
      mbar_init(smem_u32(&aempty_bar[a]), 1);
    }
    mbar_init(smem_u32(&acc_bar), 1);
    abort_sh = 0;
    last_sh = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), C::kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&x_map);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_stream = policy_evict_first();
      const uint8_t *codes = p.codes + static_cast<int64_t>(t) * p.KB * kTileBytes;
      const uint8_t *meta = p.meta + static_cast<int64_t>(t) * p.G * kRecBytes;
      int it = 0;
      for (; it < nkb; ++it) {
        const int s = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1;
        if (!mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1, abort_flag, p.err)) break;
        const int kb = kb0 + it;
        const int kfirst = kb * kTK;
        const int jlo = min(kfirst / p.g, p.G - 1);
        int nrec = 1;
        if (GENERAL) nrec = min((kfirst + kTK - 8) / p.g, p.G - 1) - jlo + 1;
        const uint32_t stage = smem_base + s * C::kStageBytes;
        const uint32_t bar = smem_u32(&full_bar[s]);
        mbar_arrive_expect_tx(bar, C::kXBytes + kTileBytes + nrec * kRecBytes);
        tma_load_2d(stage, &x_map, kfirst, m0, bar);
        bulk_g2s(stage + C::kXBytes, codes + static_cast<int64_t>(kb) * kTileBytes, kTileBytes, bar, pol_stream);
        bulk_g2s(stage + C::kXBytes + kTileBytes, meta + static_cast<int64_t>(jlo) * kRecBytes, nrec * kRecBytes,
                 bar, pol_stream);
      }
      if (*abort_flag) {
        // let every copy already issued land before the CTA's shared memory goes away
        for (int i = max(0, it - C::kStages); i < it; ++i)
          drain_wait(smem_u32(&full_bar[i % C::kStages]), (i / C::kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(128, BN);
      for (int it = 0; it < nkb; ++it) {
        const int s = it % C::kStages;
        const uint32_t ph = (it / C::kStages) & 1;
        const int a = it % C::kASlots;
        const uint32_t aph = (it / C::kASlots) & 1;
        if (!mbar_wait(smem_u32(&full_bar[s]), ph, abort_flag, p.err)) break;
        if (!mbar_wait(smem_u32(&afull_bar[a]), aph, abort_flag, p.err)) break;
        tc_fence_after();
        const uint64_t bdesc = sw128_kmajor_desc(smem_base + s * C::kStageBytes);
#pragma unroll
        for (int kk = 0; kk < kTK / 16; ++kk) {
          // A: 128 x 16 fp16 in tensor memory (8 columns per 16 K); B: 16 K-columns of the x tile (32 bytes)
          mma_f16_ts(tmem, tmem + C::kACol0 + a * 32 + kk * 8, bdesc + static_cast<uint64_t>(kk * 2), idesc,
                     (it | kk) != 0);
        }
        mma_commit(smem_u32(&empty_bar[s]));
        mma_commit(smem_u32(&aempty_bar[a]));
      }
      mma_commit(smem_u32(&acc_bar));
      if (*abort_flag) drain_wait(smem_u32(&acc_bar), 0);
    }
  } else {
    // ------------------------------------------------- dequant + epilogue
    const int dq = (warp - 2) / 4;
    const int lq = warp % 4;  // tensor-memory lane quarter this warp may access
    const int r = lq * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(lq * 32) << 16;
    for (int it = dq; it < nkb; it += C::kDqGroups) {
      const int s = it % C::kStages;
      const uint32_t ph = (it / C::kStages) & 1;
      const int a = it % C::kASlots;
      const uint32_t aph = (it / C::kASlots) & 1;
      if (!warp_wait(smem_u32(&full_bar[s]), ph, abort_flag, p.err)) break;
      const uint32_t codes = smem_base + s * C::kStageBytes + C::kXBytes;
      const uint32_t meta = codes + kTileBytes;
      const uint4 w0 = lds128(codes + r * 16);
      const uint4 w1 = lds128(codes + 2048 + r * 16);
      const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      uint32_t out[32];
      if (!warp_wait(smem_u32(&aempty_bar[a]), aph ^ 1, abort_flag, p.err)) break;
      tc_fence_after();
      if (!GENERAL) {
        const uint32_t z = (lds8(meta + 256 + r / 2) >> (4 * (r & 1))) & 0xFu;
        const GroupConsts c = group_consts(lds16(meta + 2 * r), z);
#pragma unroll
        for (int ci = 0; ci < 8; ++ci) dequant_word(words[ci], c, &out[4 * ci]);
      } else {
        const int kfirst = (kb0 + it) * kTK;
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
      tmem_st_32x32b_x32(tmem + lane_addr + C::kACol0 + a * 32, out);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&afull_bar[a]));
    }

    // ------------------------------------------------------------ epilogue
    const bool acc_ok = warp_wait(smem_u32(&acc_bar), 0, abort_flag, p.err);
    tc_fence_after();
    const int n = t * kTN + r;
    const int m_end = min(p.M, m0 + BN);
    if (__all_sync(0xffffffffu, acc_ok && !*abort_flag)) {
#pragma unroll 1
      for (int c0 = dq * 16; c0 < BN; c0 += 16 * C::kDqGroups) {
        if (m0 + c0 >= m_end) break;
        uint32_t v[16];
        tmem_ld_32x32b_x16(tmem + lane_addr + c0, v);
        tmem_wait_ld();
        if (n < p.N) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int m = m0 + c0 + i;
            if (m < m_end) {
              const float acc = __uint_as_float(v[i]);
              if (p.S == 1)
                p.y[static_cast<int64_t>(m) * p.N + n] = __float2half_rn(acc);
              else
                p.partials[(static_cast<int64_t>(sk) * p.M + m) * p.Npad + n] = acc;
            }
          }
        }
      }
    }
    if (p.S > 1) {
      // last-arriving CTA of this output tile adds the partials in split order
      __threadfence();
      named_bar_sync(1, 128 * C::kDqGroups);
      if (threadIdx.x == 64) {
        const uint32_t old = atomicAdd(&p.counters[t * p.MT + mt], 1u);
        last_sh = (old == static_cast<uint32_t>(p.S - 1)) ? 1u : 0u;
      }
      named_bar_sync(1, 128 * C::kDqGroups);
      if (last_sh) {
        __threadfence();
        if (n < p.N && !*abort_flag) {
          for (int m = m0 + dq; m < m_end; m += C::kDqGroups) {
            float acc = 0.f;
            for (int s = 0; s < p.S; ++s)
              acc += __ldcg(&p.partials[(static_cast<int64_t>(s) * p.M + m) * p.Npad + n]);
            p.y[static_cast<int64_t>(m) * p.N + n] = __float2half_rn(acc);
          }
        }
        if (threadIdx.x == 64) p.counters[t * p.MT + mt] = 0u;  // ready for the next call
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
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
    case 256: return launch_t<256, GENERAL>(map, p, ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool make_gemm_plan(int64_t M, int64_t N, int64_t K, int32_t g, int block_n, int splits, int num_sms,
                    GemmPlan *plan) {
  (void)g;
  int bn = block_n;
  if (bn == 0) bn = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
  if (bn != 16 && bn != 32 && bn != 64 && bn != 128 && bn != 256) return false;
  if (splits < 0 || splits > 64) return false;
  const int64_t mt = cdiv(M, bn), nt = cdiv(N, kTN), kb = cdiv(K, kTK);
  const int64_t tiles = mt * nt;
  int64_t S = splits;
  if (S == 0) {
    const int64_t per_sm = bn == 256 ? 1 : 2;
    const int64_t slots = static_cast<int64_t>(num_sms > 0 ? num_sms : 148) * per_sm;
    S = tiles >= slots ? 1 : slots / tiles;
    S = std::min<int64_t>(S, std::max<int64_t>(1, kb / 4));  // at least 4 K blocks per split
    S = std::min<int64_t>(S, 32);
  }
  S = std::max<int64_t>(1, std::min<int64_t>(S, kb));
  if (tiles * S > 0x7FFFFFFF) return false;
  plan->block_n = bn;
  plan->splits = static_cast<int>(S);
  plan->m_tiles = static_cast<int>(mt);
  plan->n_tiles = static_cast<int>(nt);
  plan->k_blocks = static_cast<int>(kb);
  plan->ctas = static_cast<int>(tiles * S);
  plan->counters_offset = 256;
  const size_t counters_bytes = static_cast<size_t>(cdiv(tiles * 4, 256) * 256);
  plan->partials_offset = plan->counters_offset + counters_bytes;
  const size_t partial_bytes = S > 1 ? static_cast<size_t>(S * M * nt * kTN * 4) : 0;
  plan->workspace_bytes = plan->partials_offset + partial_bytes;
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
  p.partials = reinterpret_cast<float *>(ws + plan.partials_offset);
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
  p.S = plan.splits;
  p.Npad = plan.n_tiles * kTN;
  const bool general = (g % kTK) != 0;
  return general ? launch_bn<true>(plan.block_n, map, p, plan.ctas, stream)
                 : launch_bn<false>(plan.block_n, map, p, plan.ctas, stream);
}

}  // namespace w4
