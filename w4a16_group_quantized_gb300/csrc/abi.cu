// C ABI of the library (declared in include/w4a16.h): host-side argument
// checks, workspace sizing, tiling choice and the launches. Every check runs
// before anything is enqueued; a failed check returns a status and touches
// no device state.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "internal.h"
#include "w4a16.h"

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_group(int32_t g) { return g > 0 && g % 8 == 0; }

// 2^31 - 1 bounds every index the kernels form in 32-bit arithmetic.
constexpr int64_t kMaxDim = 0x7FFFFFFF;

// Problems per w4a16_gemm_grouped call (the host list is copied once per call).
constexpr int32_t kMaxGroup = 4096;

int num_sms_current_device() {
  static int cache[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cache[dev] = sms;
  return sms;
}

int check_gemm_args(const void *x, const void *packed, int64_t M, int64_t N, int64_t K, int32_t g, void *y,
                    void *ws) {
  if (!x || !packed || !y || !ws) return W4_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || !valid_group(g)) return W4_ERR_INVALID_ARG;
  if (K % 8 != 0) return W4_ERR_UNSUPPORTED_SHAPE;  // the x row stride must be a multiple of 16 bytes
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim || M * N > (int64_t{1} << 40)) return W4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(packed, 16) || !aligned(y, 2) || !aligned(ws, 256)) return W4_ERR_MISALIGNED;
  return W4_OK;
}

// The C options struct -> the library's options (false: a field out of range).
bool to_options(const w4a16_options *o, w4::GemmOptions *out) {
  *out = w4::GemmOptions{};
  if (!o) return true;
  if (o->flags & ~(W4_FLAG_WEIGHTS_STATIC | W4_FLAG_TEST_TIMEOUT)) return false;
  if ((o->dtype != W4_DTYPE_F16 && o->dtype != W4_DTYPE_BF16) || o->reserved != 0) return false;
  out->kernel = o->kernel;
  out->block_n = o->block_n;
  out->ctas = o->ctas;
  out->schedule = o->schedule;
  out->cluster = o->cluster;
  out->weights_static = (o->flags & W4_FLAG_WEIGHTS_STATIC) != 0;
  out->test_timeout = (o->flags & W4_FLAG_TEST_TIMEOUT) != 0;
  out->wait_limit = o->wait_limit_cycles;
  out->dtype = o->dtype;
  return true;
}

// w4a16_gemm_ex's (block_n, ctas, schedule): block_n 8 is the decode kernel, whose schedule 2 runs
// whole tiles per CTA (clusters of 1) and whose ctas counts clusters.
w4::GemmOptions ex_options(int32_t block_n, int32_t ctas, int32_t schedule) {
  w4::GemmOptions o;
  o.block_n = block_n;
  o.ctas = ctas;
  if (block_n == 8) {
    o.kernel = w4::kKernelDecode;
    o.cluster = schedule == 2 ? 1 : 0;
  } else {
    o.kernel = block_n == 0 ? w4::kKernelAuto : w4::kKernelTmem;
    o.schedule = schedule;
  }
  return o;
}

int gemm_impl(const void *x, const void *packed, int64_t M, int64_t N, int64_t K, int32_t g, void *y, void *ws,
              size_t ws_bytes, const w4::GemmOptions &opt, void *stream) {
  const int rc = check_gemm_args(x, packed, M, N, K, g, y, ws);
  if (rc != W4_OK) return rc;
  w4::GemmPlan plan;
  if (!w4::make_gemm_plan(M, N, K, g, opt, num_sms_current_device(), &plan)) return W4_ERR_INVALID_ARG;
  if (ws_bytes < plan.workspace_bytes) return W4_ERR_WORKSPACE_TOO_SMALL;
  bool encode_failed = false;
  const cudaError_t e =
      w4::launch_gemm(x, packed, M, N, K, g, y, ws, plan, opt, w4::EpiSpec{}, static_cast<cudaStream_t>(stream),
                      &encode_failed);
  if (encode_failed) return W4_ERR_CUDA;
  return e == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

// The C problem list -> the library's, with every check of a single GEMM applied to each problem and
// its epilogue (outputs 2-byte aligned). Returns W4_OK or the first failing status.
int to_problems(const w4a16_problem *in, int32_t count, int64_t M, int32_t g, w4::GemmProblem *out) {
  if (!in || count < 1 || count > kMaxGroup) return W4_ERR_INVALID_ARG;
  for (int32_t i = 0; i < count; ++i) {
    const w4a16_problem &a = in[i];
    const int rc = check_gemm_args(a.x_dev, a.packed_dev, M, a.N, a.K, g, a.y_dev, reinterpret_cast<void *>(256));
    if (rc != W4_OK) return rc;
    w4::EpiSpec e;
    e.kind = a.epilogue.kind;
    e.head_dim = a.epilogue.head_dim;
    e.q_per_group = a.epilogue.q_per_group;
    e.k = a.epilogue.k_dev;
    e.v = a.epilogue.v_dev;
    if (a.epilogue.reserved != 0 || !w4::epi_valid(e, a.N)) return W4_ERR_INVALID_ARG;
    if ((e.k && !aligned(e.k, 2)) || (e.v && !aligned(e.v, 2))) return W4_ERR_MISALIGNED;
    out[i] = w4::GemmProblem{a.x_dev, a.packed_dev, a.y_dev, a.N, a.K, e};
  }
  return W4_OK;
}

size_t workspace_impl(int64_t M, int64_t N, int64_t K, int32_t g, const w4::GemmOptions &opt) {
  if (M < 1 || N < 1 || K < 1 || !valid_group(g) || M > kMaxDim || N > kMaxDim || K > kMaxDim) return 0;
  w4::GemmPlan plan;
  if (!w4::make_gemm_plan(M, N, K, g, opt, num_sms_current_device(), &plan)) return 0;
  return plan.workspace_bytes;
}

}  // namespace

extern "C" {

const char *w4_status_string(int status) {
  switch (status) {
    case W4_OK: return "W4_OK";
    case W4_ERR_INVALID_ARG: return "W4_ERR_INVALID_ARG: null pointer, non-positive size or bad group size";
    case W4_ERR_UNSUPPORTED_SHAPE: return "W4_ERR_UNSUPPORTED_SHAPE";
    case W4_ERR_MISALIGNED: return "W4_ERR_MISALIGNED";
    case W4_ERR_WORKSPACE_TOO_SMALL: return "W4_ERR_WORKSPACE_TOO_SMALL";
    case W4_ERR_CUDA: return "W4_ERR_CUDA: a CUDA call or kernel launch failed";
    case W4_ERR_TIMEOUT: return "W4_ERR_TIMEOUT: a device-side wait gave up";
    default: return "unknown w4 status";
  }
}

int w4_pack_ex(const void *W_dev, int64_t N, int64_t K, int32_t g, int32_t dtype, int32_t symmetric,
               uint32_t *qw_dev, void *scales_dev, uint32_t *zeros_dev, void *stream) {
  if (!W_dev || !qw_dev || !scales_dev || !zeros_dev) return W4_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || !valid_group(g)) return W4_ERR_INVALID_ARG;
  if ((dtype != W4_DTYPE_F16 && dtype != W4_DTYPE_BF16) || (symmetric != 0 && symmetric != 1))
    return W4_ERR_INVALID_ARG;
  if (N > kMaxDim || K > kMaxDim || N * K > (int64_t{1} << 40)) return W4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(W_dev, 2) || !aligned(qw_dev, 4) || !aligned(scales_dev, 2) || !aligned(zeros_dev, 4))
    return W4_ERR_MISALIGNED;
  const cudaError_t e = w4::launch_pack(W_dev, N, K, g, dtype, symmetric != 0, qw_dev, scales_dev, zeros_dev,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

int w4_pack(const void *W_dev, int64_t N, int64_t K, int32_t g, uint32_t *qw_dev, void *scales_dev,
            uint32_t *zeros_dev, void *stream) {
  return w4_pack_ex(W_dev, N, K, g, W4_DTYPE_F16, 0, qw_dev, scales_dev, zeros_dev, stream);
}

size_t w4_repacked_bytes(int64_t N, int64_t K, int32_t g) {
  if (N < 1 || K < 1 || !valid_group(g) || N > kMaxDim || K > kMaxDim) return 0;
  const int64_t NT = w4::cdiv(N, w4::kTN), KB = w4::cdiv(K, w4::kTK), G = w4::cdiv(K, g);
  return static_cast<size_t>(NT * KB * w4::kTileBytes + NT * G * w4::kRecBytes);
}

int w4_repack(const uint32_t *qw_dev, const void *scales_dev, const uint32_t *zeros_dev, int64_t N, int64_t K,
              int32_t g, void *packed_dev, void *stream) {
  if (!qw_dev || !scales_dev || !zeros_dev || !packed_dev) return W4_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || !valid_group(g)) return W4_ERR_INVALID_ARG;
  if (N > kMaxDim || K > kMaxDim || N * K > (int64_t{1} << 40)) return W4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(qw_dev, 4) || !aligned(scales_dev, 2) || !aligned(zeros_dev, 4) || !aligned(packed_dev, 16))
    return W4_ERR_MISALIGNED;
  const cudaError_t e =
      w4::launch_repack(qw_dev, scales_dev, zeros_dev, N, K, g, packed_dev, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

size_t w4a16_workspace_bytes_ex(int64_t M, int64_t N, int64_t K, int32_t g, int32_t block_n, int32_t ctas,
                                int32_t schedule) {
  return workspace_impl(M, N, K, g, ex_options(block_n, ctas, schedule));
}

size_t w4a16_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t g) {
  return workspace_impl(M, N, K, g, w4::GemmOptions{});
}

size_t w4a16_workspace_bytes_opts(int64_t M, int64_t N, int64_t K, int32_t g, const w4a16_options *opts) {
  w4::GemmOptions o;
  if (!to_options(opts, &o)) return 0;
  return workspace_impl(M, N, K, g, o);
}

int w4a16_gemm_plan(int64_t M, int64_t N, int64_t K, int32_t g, int32_t *block_n, int32_t *ctas,
                    int32_t *schedule) {
  if (!block_n || !ctas || !schedule) return W4_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || !valid_group(g) || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return W4_ERR_INVALID_ARG;
  w4::GemmPlan plan;
  if (!w4::make_gemm_plan(M, N, K, g, w4::GemmOptions{}, num_sms_current_device(), &plan))
    return W4_ERR_INVALID_ARG;
  *block_n = plan.block_n;
  *ctas = plan.ctas;
  *schedule = plan.whole ? 2 : 1;
  return W4_OK;
}

int w4a16_gemm(const void *x_dev, const void *packed_dev, int64_t M, int64_t N, int64_t K, int32_t g, void *y_dev,
               void *workspace_dev, size_t workspace_bytes, void *stream) {
  return gemm_impl(x_dev, packed_dev, M, N, K, g, y_dev, workspace_dev, workspace_bytes, w4::GemmOptions{}, stream);
}

int w4a16_gemm_ex(const void *x_dev, const void *packed_dev, int64_t M, int64_t N, int64_t K, int32_t g, void *y_dev,
                  void *workspace_dev, size_t workspace_bytes, int32_t block_n, int32_t ctas, int32_t schedule,
                  void *stream) {
  return gemm_impl(x_dev, packed_dev, M, N, K, g, y_dev, workspace_dev, workspace_bytes,
                   ex_options(block_n, ctas, schedule), stream);
}

int w4a16_gemm_opts(const void *x_dev, const void *packed_dev, int64_t M, int64_t N, int64_t K, int32_t g,
                    void *y_dev, void *workspace_dev, size_t workspace_bytes, const w4a16_options *opts, void *stream) {
  w4::GemmOptions o;
  if (!to_options(opts, &o)) return W4_ERR_INVALID_ARG;
  return gemm_impl(x_dev, packed_dev, M, N, K, g, y_dev, workspace_dev, workspace_bytes, o, stream);
}

size_t w4a16_grouped_workspace_bytes(const w4a16_problem *problems, int32_t count, int64_t M, int32_t g,
                                     const w4a16_options *opts) {
  w4::GemmOptions o;
  if (!to_options(opts, &o)) return 0;
  std::vector<w4::GemmProblem> probs(count > 0 && count <= kMaxGroup ? count : 0);
  if (to_problems(problems, count, M, g, probs.data()) != W4_OK) return 0;
  w4::GroupPlan plan;
  if (!w4::make_group_plan(probs.data(), count, M, g, o, num_sms_current_device(), &plan)) return 0;
  return plan.workspace_bytes;
}

int w4a16_gemm_grouped(const w4a16_problem *problems, int32_t count, int64_t M, int32_t g, void *workspace_dev,
                       size_t workspace_bytes, const w4a16_options *opts, void *stream) {
  w4::GemmOptions o;
  if (!to_options(opts, &o)) return W4_ERR_INVALID_ARG;
  if (!workspace_dev) return W4_ERR_INVALID_ARG;
  if (!aligned(workspace_dev, 256)) return W4_ERR_MISALIGNED;
  std::vector<w4::GemmProblem> probs(count > 0 && count <= kMaxGroup ? count : 0);
  const int rc = to_problems(problems, count, M, g, probs.data());
  if (rc != W4_OK) return rc;
  const int sms = num_sms_current_device();
  w4::GroupPlan plan;
  if (!w4::make_group_plan(probs.data(), count, M, g, o, sms, &plan)) return W4_ERR_INVALID_ARG;
  if (workspace_bytes < plan.workspace_bytes) return W4_ERR_WORKSPACE_TOO_SMALL;
  bool encode_failed = false;
  const cudaError_t e = w4::launch_gemm_grouped(probs.data(), count, M, g, workspace_dev, plan, o, sms,
                                                static_cast<cudaStream_t>(stream), &encode_failed);
  if (encode_failed) return W4_ERR_CUDA;
  return e == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

int w4_last_device_error(void *workspace_dev, void *stream) {
  if (!workspace_dev) return W4_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace_dev, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return W4_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return W4_ERR_CUDA;
  if (word == 0) return W4_OK;
  if (cudaMemsetAsync(workspace_dev, 0, sizeof(word), st) != cudaSuccess) return W4_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return W4_ERR_CUDA;
  return W4_ERR_TIMEOUT;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// w4a16_gemm_noalloc: w4a16_gemm with its scratch in a fixed, library-owned
// device array instead of a caller workspace (see include/w4a16.h).
// ---------------------------------------------------------------------------
namespace {

// The scratch every call shares: error word, per-tile counters and the fp32
// partial tiles of the stream-K fixup. Each GPU that loads the library keeps
// these bytes until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[W4A16_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch for the current device. In host code the
// array's name is only a host-side stand-in; the real address comes from
// cudaGetSymbolAddress with that device current, looked up once per device.
void *noalloc_scratch_address(int *status) {
  static void *addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *status = W4_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      *status = W4_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  *status = W4_OK;
  return addr[dev];
}

}  // namespace

extern "C" {

int w4a16_gemm_noalloc(const void *x_dev, const void *packed_dev, int64_t M, int64_t N, int64_t K, int32_t g,
                       void *y_dev, void *stream) {
  static_assert(W4A16_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size");
  // the usual argument checks, with an aligned non-null stand-in for the workspace argument
  int rc = check_gemm_args(x_dev, packed_dev, M, N, K, g, y_dev, reinterpret_cast<void *>(uintptr_t{256}));
  if (rc != W4_OK) return rc;
  w4::GemmPlan plan;
  const w4::GemmOptions opt;
  if (!w4::make_gemm_plan(M, N, K, g, opt, num_sms_current_device(), &plan)) return W4_ERR_INVALID_ARG;
  if (plan.workspace_bytes > W4A16_NOALLOC_SCRATCH_BYTES) return W4_ERR_WORKSPACE_TOO_SMALL;
  void *scratch = noalloc_scratch_address(&rc);
  if (rc != W4_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: the error word and the tile counters must start at zero
  if (cudaMemsetAsync(scratch, 0, plan.pieces_offset, st) != cudaSuccess) return W4_ERR_CUDA;
  bool encode_failed = false;
  const cudaError_t e =
      w4::launch_gemm(x_dev, packed_dev, M, N, K, g, y_dev, scratch, plan, opt, w4::EpiSpec{}, st, &encode_failed);
  if (encode_failed) return W4_ERR_CUDA;
  return e == cudaSuccess ? W4_OK : W4_ERR_CUDA;
}

}  // extern "C"
