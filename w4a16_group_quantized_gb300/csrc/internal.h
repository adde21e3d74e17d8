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

// 16-bit value types of weights, scales, activations and outputs.
constexpr int kDtypeF16 = 0;
constexpr int kDtypeBf16 = 1;

// Output epilogues (W4_EPI_* of the C ABI).
constexpr int kEpiNone = 0;
constexpr int kEpiSiluMul = 1;
constexpr int kEpiQkv = 2;

cudaError_t launch_pack(const void *W, int64_t N, int64_t K, int32_t g, int dtype, bool symmetric, uint32_t *qw,
                        void *scales, uint32_t *zeros, cudaStream_t stream);

cudaError_t launch_repack(const uint32_t *qw, const void *scales, const uint32_t *zeros, int64_t N, int64_t K,
                          int32_t g, void *packed, cudaStream_t stream);

// Which GEMM kernel runs: the register-operand decode kernel (M <= 16, gemm_dec.cuh) or the
// tensor-memory kernel (gemm.cu).
constexpr int kKernelAuto = 0;
constexpr int kKernelDecode = 1;
constexpr int kKernelTmem = 2;

// The decode kernel keeps each CTA's K range of x in shared memory: M rows of 512 bytes per 256-wide
// K stage, at most kDecXRegionBytes and kDecXSliceMax stages.
constexpr int kDecXRegionBytes = 96 * 1024;
constexpr int kDecXSliceMax = 48;
inline int64_t dec_x_stages_max(int64_t M) {
  const int64_t s = kDecXRegionBytes / (512 * M);
  return s < kDecXSliceMax ? s : kDecXSliceMax;
}
// Whether a split of KS stages among C CTAs leaves each CTA a K range of x that fits.
inline bool dec_x_fits(int64_t KS, int64_t C, int64_t M) { return (KS + C - 1) / C <= dec_x_stages_max(M); }

// Caller choices for one GEMM (zero = automatic); mirrors w4a16_options of the C ABI.
struct GemmOptions {
  int kernel = kKernelAuto;
  int block_n = 0;
  int ctas = 0;       // tensor-memory kernel: persistent CTAs; decode kernel: clusters
  int schedule = 0;   // tensor-memory kernel: 1 stream-K, 2 whole tiles
  int cluster = 0;    // decode kernel: CTAs per cluster (1, 2, 4, 8)
  bool weights_static = false;
  bool test_timeout = false;  // test only: one wait expects more than will come (runs out after wait_limit)
  uint64_t wait_limit = 0;
  int dtype = kDtypeF16;      // x, scales and y
  bool one_tile_mid = false;  // below M = 256, one-tile units only (the grouped tensor-memory launch takes no others)
};

struct GemmPlan {
  int kernel;    // kKernelDecode or kKernelTmem
  int cluster;   // decode kernel: forced cluster size (0: chosen at launch)
  int block_n;   // activation rows per tile: 8 or 16 (decode kernel), 16, 32, 64 or 128 (tensor-memory kernel)
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

// Returns false if the options are not valid values for this problem.
bool make_gemm_plan(int64_t M, int64_t N, int64_t K, int32_t g, const GemmOptions &opt, int num_sms,
                    GemmPlan *plan);

// An output epilogue as the caller gives it (w4a16_epilogue of the C ABI).
struct EpiSpec {
  int kind = kEpiNone;
  int head_dim = 0;     // kEpiQkv
  int q_per_group = 0;  // kEpiQkv
  void *k = nullptr;    // kEpiQkv
  void *v = nullptr;
};

// Whether the epilogue is valid for a problem of N weight rows.
bool epi_valid(const EpiSpec &e, int64_t N);

// Launches the GEMM for a validated plan. Returns the CUDA error (cudaSuccess on success);
// *encode_failed is set when the tensor map could not be built.
cudaError_t launch_gemm(const void *x, const void *packed, int64_t M, int64_t N, int64_t K, int32_t g, void *y,
                        void *workspace, const GemmPlan &plan, const GemmOptions &opt, const EpiSpec &epi,
                        cudaStream_t stream, bool *encode_failed);

// Several independent GEMMs of the same M, g and type (w4a16_gemm_grouped).
struct GemmProblem {
  const void *x;
  const void *packed;
  void *y;
  int64_t N, K;
  EpiSpec epi;
};

// How a group runs: with the decode kernel, all problems in launches of up to kGroupMax problems
// that walk their weight tiles in one persistent grid; with the tensor-memory kernel, problems that
// share x and K (up to kTmemGroupMax, one-tile units) in one launch over all their weight tiles
// (`tmem_plan`, made for the tiles laid one after another); otherwise one launch per problem.
constexpr int kGroupMax = 16;
constexpr int kTmemGroupMaxHost = 8;
struct GroupPlan {
  bool decode;
  bool tmem;
  int block_n;            // decode kernel: 8 or 16
  GemmPlan tmem_plan;
  size_t workspace_bytes;
};

bool make_group_plan(const GemmProblem *probs, int count, int64_t M, int32_t g, const GemmOptions &opt, int num_sms,
                     GroupPlan *plan);

cudaError_t launch_gemm_grouped(const GemmProblem *probs, int count, int64_t M, int32_t g, void *workspace,
                                const GroupPlan &plan, const GemmOptions &opt, int num_sms, cudaStream_t stream,
                                bool *encode_failed);

}  // namespace w4
