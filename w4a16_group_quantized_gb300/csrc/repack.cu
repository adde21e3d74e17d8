// w4_repack: canonical packed weights -> the GEMM's tile layout.
//
// The offline conversion of packed 4-bit weights into an engine's own layout
// is the converter step of lmdeploy PR #202 (AWQ checkpoint -> TurboMind
// workspace). Here the target layout is made for the sm_103a GEMM:
//  * each 128-row x 64-code tile is one contiguous 4 KB block, so a single
//    bulk copy moves one pipeline stage of weights into shared memory;
//  * inside a tile, thread r of the dequantizing warpgroup reads row r as two
//    16-byte words at h*2048 + r*16, which is free of bank conflicts;
//  * inside each 8-code word, code e sits at nibble 4*(e%2) + e/2, so that
//    masking with 0x000F000F (after a shift of 0 or 8 bits) or 0x00F000F0
//    leaves codes 2p and 2p+1 in the two fp16 halves of one register, in the
//    order the tensor memory operand wants them;
//  * per (n-tile, group) one 320-byte record holds the 128 fp16 scales and
//    128 4-bit zeros, so a stage fetches exactly the records it needs.
// Everything outside [N, K] is written as 0.
#include "internal.h"

namespace w4 {
namespace {

// canonical nibble e (code k = 8c + e) -> tile nibble 4*(e%2) + e/2
__device__ __forceinline__ uint32_t permute_nibbles(uint32_t w) {
  uint32_t out = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) out |= ((w >> (4 * e)) & 0xFu) << (4 * (4 * (e % 2) + e / 2));
  return out;
}

// One thread per 16-byte output word: (tile t, k-block b, half h, row r).
__global__ void repack_codes_kernel(const uint32_t *__restrict__ qw, int64_t N, int64_t K, int64_t KB,
                                    int64_t total, uint4 *__restrict__ out) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int r = static_cast<int>(idx % kTN);
  const int h = static_cast<int>((idx / kTN) % 2);
  const int64_t tb = idx / (2 * kTN);  // t * KB + b
  const int64_t b = tb % KB;
  const int64_t t = tb / KB;
  const int64_t n = t * kTN + r;
  const int64_t Kw = (K + 7) / 8;
  uint32_t v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t k0 = b * kTK + 32 * h + 8 * i;  // first code of this word
    uint32_t w = 0;
    if (n < N && k0 < K) {
      w = qw[n * Kw + k0 / 8];
      const int64_t valid = K - k0;  // codes at k >= K are written as 0
      if (valid < 8) w &= (1u << (4 * valid)) - 1u;
    }
    v[i] = permute_nibbles(w);
  }
  out[idx] = make_uint4(v[0], v[1], v[2], v[3]);
}

// One thread per (tile t, group j, row pair rp): two scales and one zero byte.
__global__ void repack_groups_kernel(const uint16_t *__restrict__ scales, const uint32_t *__restrict__ zeros,
                                     int64_t N, int64_t G, int64_t total, uint8_t *__restrict__ meta) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int rp = static_cast<int>(idx % (kTN / 2));
  const int64_t tj = idx / (kTN / 2);  // t * G + j
  const int64_t j = tj % G;
  const int64_t t = tj / G;
  const int64_t Gw = (G + 7) / 8;
  uint32_t s2 = 0, zb = 0;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int64_t n = t * kTN + 2 * rp + u;
    if (n < N) {
      s2 |= static_cast<uint32_t>(scales[n * G + j]) << (16 * u);
      zb |= ((zeros[n * Gw + j / 8] >> (4 * (j % 8))) & 0xFu) << (4 * u);
    }
  }
  uint8_t *rec = meta + tj * kRecBytes;
  reinterpret_cast<uint32_t *>(rec)[rp] = s2;
  rec[256 + rp] = static_cast<uint8_t>(zb);
}

}  // namespace

cudaError_t launch_repack(const uint32_t *qw, const void *scales, const uint32_t *zeros, int64_t N, int64_t K,
                          int32_t g, void *packed, cudaStream_t stream) {
  const int64_t NT = cdiv(N, kTN), KB = cdiv(K, kTK), G = cdiv(K, g);
  const int block = 256;
  const int64_t total_codes = NT * KB * 2 * kTN;
  const int64_t blocks_c = cdiv(total_codes, block);
  const int64_t total_meta = NT * G * (kTN / 2);
  const int64_t blocks_m = cdiv(total_meta, block);
  if (blocks_c > 0x7FFFFFFF || blocks_m > 0x7FFFFFFF) return cudaErrorInvalidValue;
  uint8_t *base = static_cast<uint8_t *>(packed);
  repack_codes_kernel<<<static_cast<unsigned>(blocks_c), block, 0, stream>>>(qw, N, K, KB, total_codes,
                                                                              reinterpret_cast<uint4 *>(base));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  repack_groups_kernel<<<static_cast<unsigned>(blocks_m), block, 0, stream>>>(
      static_cast<const uint16_t *>(scales), zeros, N, G, total_meta, base + NT * KB * kTileBytes);
  return cudaGetLastError();
}

}  // namespace w4
