// w4_pack: fp16 or bf16 weights -> canonical 4-bit codes, scales of the same type, 4-bit zeros.
//
// Group-wise 4-bit quantization along K (lmdeploy PR #202, AWQ weights with --group_size;
// torchchat issue #1362, 'linear:int4' with a groupsize, in fp16 or bf16 precision), with a last
// group narrower than g when K % g != 0 (torchchat issue #1362, option 2). Asymmetric: the range of
// a group is [min(0, min w), max(0, max w)] and z puts zero on the code grid; symmetric: the range
// is [-max|w|, max|w|] and z = 8. All arithmetic is fp64 with explicit round-to-nearest operations,
// so the result is bit-exact and independent of contraction or fast-math settings.
//
// One warp takes the 8 consecutive groups of a row that share one zeros word: per group, the lanes
// read the weights 32 at a time (coalesced), reduce the range across the warp, and each lane turns
// its weights into codes; lanes 8i .. 8i + 7 hold the 8 codes of one uint32 word, which lane 8i
// assembles with shuffles and stores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace w4 {
namespace {

template <int DT>
__device__ __forceinline__ double to_f64(uint16_t b) {  // exact widening
  if (DT == kDtypeBf16) return static_cast<double>(__uint_as_float(static_cast<uint32_t>(b) << 16));
  return static_cast<double>(__half2float(__ushort_as_half(b)));
}

template <int DT>
__device__ __forceinline__ uint16_t from_f64_rn(double v) {  // one rounding, to nearest even
  uint16_t h;
  if (DT == kDtypeBf16)
    asm("cvt.rn.bf16.f64 %0, %1;" : "=h"(h) : "d"(v));
  else
    asm("cvt.rn.f16.f64 %0, %1;" : "=h"(h) : "d"(v));
  return h;
}

__device__ __forceinline__ double warp_min(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmin(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ double warp_max(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <int DT, bool SYM>
__global__ void pack_kernel(const uint16_t *__restrict__ W, int64_t N, int64_t K, int32_t g, int64_t G,
                            uint32_t *__restrict__ qw, uint16_t *__restrict__ scales, uint32_t *__restrict__ zeros) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int64_t Gw = (G + 7) / 8;
  const int64_t n = wid / Gw;
  const int64_t jw = wid % Gw;
  if (n >= N) return;  // whole warps leave together
  const int64_t Kw = (K + 7) / 8;
  const uint16_t *row = W + n * K;
  const uint16_t one = DT == kDtypeBf16 ? 0x3F80 : 0x3C00;
  uint32_t zword = 0;
  for (int64_t j = 8 * jw; j < min(8 * jw + 8, G); ++j) {
    const int64_t k0 = j * g;
    const int64_t k1 = min(k0 + static_cast<int64_t>(g), K);
    double lo = 0.0, hi = 0.0;  // the asymmetric range always includes zero
    for (int64_t k = k0 + lane; k < k1; k += 32) {
      const double w = to_f64<DT>(row[k]);
      lo = fmin(lo, w);
      hi = fmax(hi, w);
    }
    lo = warp_min(lo);
    hi = warp_max(hi);
    if (SYM) {
      const double amax = fmax(hi, -lo);
      lo = -amax;
      hi = amax;
    }
    const double r = __dsub_rn(hi, lo);  // exact
    uint16_t sb = one;                   // 1 for an all-zero group
    double sv = 1.0;
    uint32_t z = SYM ? 8u : 0u;
    if (r != 0.0) {
      sb = from_f64_rn<DT>(__ddiv_rn(r, 15.0));
      sv = to_f64<DT>(sb);
      if (__dmul_rn(sv, 15.0) < r) {  // exact product; one step up so that 15 s >= r
        sb = static_cast<uint16_t>(sb + 1);
        sv = to_f64<DT>(sb);
      }
      if (!SYM) {
        const double zz = rint(__ddiv_rn(-lo, sv));
        z = static_cast<uint32_t>(zz < 0.0 ? 0.0 : (zz > 15.0 ? 15.0 : zz));
      }
    }
    if (lane == 0) scales[n * G + j] = sb;
    zword |= z << (4 * (j - 8 * jw));
    // codes, 32 per pass: g is a multiple of 8, so the group owns whole words (a row's last may be
    // partial, its padding nibbles 0)
    for (int64_t kc = k0; kc < k1; kc += 32) {
      const int64_t k = kc + lane;
      uint32_t code = 0;
      if (k < k1) {
        code = z;  // an all-zero group encodes every weight as z
        if (r != 0.0) {
          const double t = rint(__ddiv_rn(to_f64<DT>(row[k]), sv)) + static_cast<double>(z);  // exact sum
          code = static_cast<uint32_t>(t < 0.0 ? 0.0 : (t > 15.0 ? 15.0 : t));
        }
      }
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) word |= __shfl_sync(0xffffffffu, code, (lane & ~7) + e) << (4 * e);
      if ((lane & 7) == 0 && kc + lane < k1) qw[n * Kw + (kc + lane) / 8] = word;
    }
  }
  if (lane == 0) zeros[n * Gw + jw] = zword;
}

}  // namespace

cudaError_t launch_pack(const void *W, int64_t N, int64_t K, int32_t g, int dtype, bool symmetric, uint32_t *qw,
                        void *scales, uint32_t *zeros, cudaStream_t stream) {
  const int64_t G = cdiv(K, g);
  const int64_t warps = N * cdiv(G, 8);
  const int block = 128;
  const int64_t blocks = cdiv(warps * 32, block);
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const auto *w = static_cast<const uint16_t *>(W);
  auto *s = static_cast<uint16_t *>(scales);
  const dim3 grid(static_cast<unsigned>(blocks));
  if (dtype == kDtypeBf16) {
    if (symmetric)
      pack_kernel<kDtypeBf16, true><<<grid, block, 0, stream>>>(w, N, K, g, G, qw, s, zeros);
    else
      pack_kernel<kDtypeBf16, false><<<grid, block, 0, stream>>>(w, N, K, g, G, qw, s, zeros);
  } else {
    if (symmetric)
      pack_kernel<kDtypeF16, true><<<grid, block, 0, stream>>>(w, N, K, g, G, qw, s, zeros);
    else
      pack_kernel<kDtypeF16, false><<<grid, block, 0, stream>>>(w, N, K, g, G, qw, s, zeros);
  }
  return cudaGetLastError();
}

}  // namespace w4
