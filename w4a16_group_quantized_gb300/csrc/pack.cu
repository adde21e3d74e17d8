// w4_pack: fp16 weights -> canonical 4-bit codes, fp16 scales, 4-bit zeros.
//
// Group-wise asymmetric 4-bit quantization along K (lmdeploy PR #202, AWQ
// weights with --group_size; torchchat issue #1362, 'linear:int4' with a
// groupsize), with a last group narrower than g when K % g != 0 (torchchat
// issue #1362, option 2). All arithmetic is fp64 with explicit round-to-
// nearest intrinsics, so the result is bit-exact and independent of
// contraction or fast-math settings.
#include <cuda_fp16.h>

#include "internal.h"

namespace w4 {
namespace {

__device__ __forceinline__ uint16_t f64_to_f16_rn(double v) {
  uint16_t h;
  asm("cvt.rn.f16.f64 %0, %1;" : "=h"(h) : "d"(v));
  return h;
}

__device__ __forceinline__ double f16_to_f64(uint16_t h) {
  return static_cast<double>(__half2float(__ushort_as_half(h)));  // exact widening
}

// One thread per (row n, group j); 8 consecutive threads share one zeros word.
// Threads are laid out over [N, Gp] with Gp = G rounded up to 8, so an
// aligned group of 8 lanes always belongs to one row.
__global__ void pack_kernel(const uint16_t *__restrict__ W, int64_t N, int64_t K, int32_t g, int64_t G,
                            int64_t Gp, uint32_t *__restrict__ qw, uint16_t *__restrict__ scales,
                            uint32_t *__restrict__ zeros) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t n = idx / Gp;
  const int64_t j = idx % Gp;
  const bool valid = n < N && j < G;
  const int64_t Kw = (K + 7) / 8;
  uint32_t z = 0;
  if (valid) {
    const int64_t k0 = j * g;
    const int64_t k1 = min(k0 + static_cast<int64_t>(g), K);
    const uint16_t *row = W + n * K;
    double lo = 0.0, hi = 0.0;  // the range always includes zero
    for (int64_t k = k0; k < k1; ++k) {
      const double w = f16_to_f64(row[k]);
      lo = w < lo ? w : lo;
      hi = w > hi ? w : hi;
    }
    const double r = __dsub_rn(hi, lo);  // exact
    uint16_t sb = 0x3C00;                // 1.0 for an all-zero group
    double sv = 1.0;
    if (r != 0.0) {
      sb = f64_to_f16_rn(__ddiv_rn(r, 15.0));
      sv = f16_to_f64(sb);
      if (__dmul_rn(sv, 15.0) < r) {  // exact product; raise s one fp16 step so that 15 s >= r
        sb = static_cast<uint16_t>(sb + 1);
        sv = f16_to_f64(sb);
      }
      const double zz = rint(__ddiv_rn(-lo, sv));
      z = static_cast<uint32_t>(zz < 0.0 ? 0.0 : (zz > 15.0 ? 15.0 : zz));
    }
    scales[n * G + j] = sb;
    // codes: g is a multiple of 8, so the group owns whole words (the row's last word may be partial)
    for (int64_t c = k0 / 8; c < (k1 + 7) / 8; ++c) {
      uint32_t word = 0;
      for (int e = 0; e < 8; ++e) {
        const int64_t k = 8 * c + e;
        if (k >= k1) break;
        uint32_t code = 0;
        if (r != 0.0) {
          const double t = rint(__ddiv_rn(f16_to_f64(row[k]), sv)) + static_cast<double>(z);  // exact sum
          code = static_cast<uint32_t>(t < 0.0 ? 0.0 : (t > 15.0 ? 15.0 : t));
        }
        word |= code << (4 * e);
      }
      qw[n * Kw + c] = word;
    }
  }
  // zeros: lane 8i collects the 8 zeros of its aligned lane group
  const int lane = threadIdx.x & 31;
  uint32_t zword = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) zword |= __shfl_sync(0xffffffffu, z, (lane & ~7) + e) << (4 * e);
  if ((lane & 7) == 0 && n < N && j < G) zeros[n * (Gp / 8) + j / 8] = zword;
}

}  // namespace

cudaError_t launch_pack(const void *W, int64_t N, int64_t K, int32_t g, uint32_t *qw, void *scales,
                        uint32_t *zeros, cudaStream_t stream) {
  const int64_t G = cdiv(K, g);
  const int64_t Gp = cdiv(G, 8) * 8;
  const int64_t threads = N * Gp;
  const int block = 256;
  const int64_t blocks = cdiv(threads, block);
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  pack_kernel<<<static_cast<unsigned>(blocks), block, 0, stream>>>(
      static_cast<const uint16_t *>(W), N, K, g, G, Gp, qw, static_cast<uint16_t *>(scales), zeros);
  return cudaGetLastError();
}

}  // namespace w4
