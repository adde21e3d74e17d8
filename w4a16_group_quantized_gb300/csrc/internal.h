// Host-side declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace w4 {

// Tile layout constants (the code tiles and group records of w4_repack).
constexpr int kTN = 128;         // weight rows per tile (the MMA's M)
constexpr int kTK = 64;          // codes along K per tile (one K block)
constexpr int kTileBytes = 4096; // 128 rows x 64 codes x 4 bits
constexpr int kRecBytes = 320;   // 128 fp16 scales + 128 4-bit zeros

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

cudaError_t launch_pack(const void *W, int64_t N, int64_t K, int32_t g, uint32_t *qw, void *scales,
                        uint32_t *zeros, cudaStream_t stream);

cudaError_t launch_repack(const uint32_t *qw, const void *scales, const uint32_t *zeros, int64_t N, int64_t K,
                          int32_t g, void *packed, cudaStream_t stream);

struct GemmPlan {
  int block_n;   // activation rows per tile: 8 (decode kernel), 16, 32, 64 or 128 (tensor-memory kernel)
  int m_tiles;
  int n_tiles;
  int k_blocks;
  int k_stages;  // K stages per output tile (4 K blocks, or 2 for two-tile units; the last may be shorter)
  int tiles_per_unit;  // weight tiles per unit: 2 for block_n 128 (one x tile serves both), else 1
  int ctas;      // persistent CTAs (one per SM)
  int gran;      // K stages per scheduling grain: 1 (stream-K) or k_stages (whole tiles)
  bool whole;    // whole-tile schedule (no tile is cut between CTAs)
  bool interleave;  // whole tiles dealt out round-robin (CTA c: tiles c, c + ctas, ...), else ranges
  int64_t grains;
  size_t counters_offset;
  size_t pieces_offset;
  size_t workspace_bytes;
};

// schedule: 0 automatic, 1 stream-K, 2 whole tiles. ctas: 0 = one per SM.
// Returns false if block_n / ctas / schedule are not valid values.
bool make_gemm_plan(int64_t M, int64_t N, int64_t K, int32_t g, int block_n, int ctas, int schedule, int num_sms,
                    GemmPlan *plan);

// Launches the GEMM for a validated plan. Returns the CUDA error (cudaSuccess on success);
// *encode_failed is set when the tensor map could not be built.
cudaError_t launch_gemm(const void *x, const void *packed, int64_t M, int64_t N, int64_t K, int32_t g, void *y,
                        void *workspace, const GemmPlan &plan, cudaStream_t stream, bool *encode_failed);

}  // namespace w4
