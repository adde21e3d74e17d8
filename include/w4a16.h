/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) W4A16 group-quantized linear layer.
 *
 *   y[M,N] = x[M,K] . dequant(Wq)[N,K]^T,   w[n,k] = (q[n,k] - z[n,j]) * s[n,j],  j = floor(k/g)
 *
 * x and y are fp16 (or bf16), row-major. Each weight is an unsigned 4-bit
 * code q in [0,15]; every (output row n, group j of g consecutive k) has a
 * scale s of the same 16-bit type and a 4-bit zero z. When K is not a
 * multiple of g the last group is narrower than g and is handled as such:
 * nothing is padded or skipped.
 *
 * Each call's comment names the passage of the pages it follows ("Follows:");
 * calls that are plumbing of this library (sizes, status, errors) name none.
 *
 * Conventions for every call:
 *  - Pointers named *_dev are device pointers; the caller allocates and owns
 *    all buffers. The library allocates no device memory and never
 *    synchronises a stream, except w4_last_device_error (documented there).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All device work is enqueued on it and is asynchronous to the host.
 *  - Arguments are checked on the host first; a failed check returns a
 *    status and enqueues nothing. Launch failures return W4_ERR_CUDA.
 *  - The device code is built for sm_103a only.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define W4_API __attribute__((visibility("default")))
#else
#define W4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    W4_OK = 0,
    W4_ERR_INVALID_ARG = 1,        /* null pointer, non-positive size, g not a positive multiple of 8 */
    W4_ERR_UNSUPPORTED_SHAPE = 2,  /* a size the kernel does not take (e.g. K % 8 != 0 in the GEMM) */
    W4_ERR_MISALIGNED = 3,         /* a pointer not aligned as the call requires */
    W4_ERR_WORKSPACE_TOO_SMALL = 4,
    W4_ERR_CUDA = 5,               /* a CUDA runtime/driver call or kernel launch failed */
    W4_ERR_TIMEOUT = 6             /* a device-side wait gave up (read with w4_last_device_error) */
} w4_status;

/* Static, human-readable name of a status code. Never NULL. */
W4_API const char *w4_status_string(int status);

/*
 * w4_pack -- quantize fp16 weights into the canonical packed form.
 *
 * W_dev      fp16 [N, K] row-major (nn.Linear weight layout). Must be finite.
 * N, K       >= 1, any value.
 * g          group size along K, a positive multiple of 8. G = ceil(K/g).
 * qw_dev     out: uint32 [N, ceil(K/8)]; code of k = 8c + i in bits 4i..4i+3
 *            of word c of row n; padding nibbles (k >= K) are 0.
 * scales_dev out: fp16 [N, G].
 * zeros_dev  out: uint32 [N, ceil(G/8)]; zero of group j = 8c + i in bits
 *            4i..4i+3 of word c of row n; padding nibbles are 0.
 *
 * Follows: group-wise 4-bit weights with a group size -- lmdeploy PR #202
 * "Blazing fast W4A16 inference" (AWQ weights, --group_size 128) and
 * torchchat issue #1362 ('linear:int4' with 'groupsize'); a last group
 * narrower than g -- torchchat issue #1362, option 2 ("groupwise GEMM with
 * a last group that's not a full group").
 *
 * Per (n, j), over k in [j*g, min((j+1)*g, K)), in fp64:
 *   lo = min(0, min w), hi = max(0, max w), r = hi - lo;
 *   r == 0: s = 1, z = 0, q = 0;
 *   else s = fp16(r / 15) rounded to nearest-even, raised one fp16 step if
 *   15*s < r; z = clamp(rint(-lo / s), 0, 15); q = clamp(rint(w / s) + z, 0, 15)
 *   (rint = round half to even). Bit-exact and deterministic.
 * Alignment: W 2-byte, outputs 4-byte (scales 2-byte).
 */
W4_API int w4_pack(const void *W_dev, int64_t N, int64_t K, int32_t g,
            uint32_t *qw_dev, void *scales_dev, uint32_t *zeros_dev, void *stream);

/* Value types of weights, scales, activations and outputs. */
#define W4_DTYPE_F16 0
#define W4_DTYPE_BF16 1

/*
 * w4_pack_ex -- w4_pack for fp16 or bf16 weights, asymmetric or symmetric.
 *
 * dtype      W4_DTYPE_F16 or W4_DTYPE_BF16: the type of W and of the scales
 *            written (bf16: the 'bf16' precision torchchat issue #1362 runs
 *            'linear:int4' quantization with).
 * symmetric  0: the zero-point form of w4_pack. 1: z = 8 for every group and
 *            the range [-m, m], m = max|w| over the group: s is the least
 *            value of the type with 15 s >= 2 m (s = 1 for an all-zero
 *            group), q = clamp(rint(w / s) + 8, 0, 15); |w - (q - 8) s| <= s/2.
 * Other arguments, layouts and guarantees as w4_pack (the zeros buffer holds
 * 8 in every nibble for symmetric weights, so the GEMM takes them unchanged).
 * Returns W4_ERR_INVALID_ARG for another dtype or symmetric value.
 */
W4_API int w4_pack_ex(const void *W_dev, int64_t N, int64_t K, int32_t g, int32_t dtype, int32_t symmetric,
                      uint32_t *qw_dev, void *scales_dev, uint32_t *zeros_dev, void *stream);

/*
 * Size in bytes of the GEMM's tile layout for an [N, K] weight with group size g:
 *   ceil(N/128) * ceil(K/64) * 4096 + ceil(N/128) * ceil(K/g) * 320.
 * Returns 0 for invalid sizes.
 */
W4_API size_t w4_repacked_bytes(int64_t N, int64_t K, int32_t g);

/*
 * w4_repack -- canonical packed form -> the GEMM's tile layout (a permutation
 * of codes, scales and zeros; bit-exact, deterministic).
 *
 * Follows: converting canonical packed weights into the kernel's own layout
 * once, offline -- the converter step of lmdeploy PR #202 (deploy.py with
 * --model_format awq). Scales are moved as 16-bit values: fp16 and bf16
 * scales repack alike.
 *
 * Inputs as produced by w4_pack. `packed_dev` (out) has w4_repacked_bytes(N,K,g)
 * bytes, 16-byte aligned. Layout, with NT = ceil(N/128), KB = ceil(K/64):
 *  - code tiles: tile (t, b) of 4096 bytes at offset (t*KB + b)*4096 holds
 *    rows n = 128t + r (r < 128) and k = 64b .. 64b+63; the little-endian
 *    uint32 at byte h*2048 + r*16 + 4*i (h < 2, i < 4) holds the 8 codes of
 *    row n at k = 64b + 32h + 8i + e (e < 8), code e at nibble 4*(e%2) + e/2;
 *  - group records after the tiles: record (t, j) of 320 bytes at offset
 *    NT*KB*4096 + (t*G + j)*320 holds the scale of row 128t + r at byte
 *    2r and its zero in byte 256 + r/2 (low nibble for even r);
 *  - everything at n >= N or k >= K is 0.
 */
W4_API int w4_repack(const uint32_t *qw_dev, const void *scales_dev, const uint32_t *zeros_dev,
              int64_t N, int64_t K, int32_t g, void *packed_dev, void *stream);

/*
 * Bytes of device workspace w4a16_gemm needs for this problem on the current
 * device (error word, per-tile counters and fp32 partial tiles for the
 * stream-K fixup). Always >= 256. Returns 0 for invalid sizes.
 */
W4_API size_t w4a16_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t g);

/*
 * w4a16_gemm -- y = x . dequant(packed)^T.
 *
 * x_dev      fp16 [M, K] row-major, 16-byte aligned.
 * packed_dev w4_repack output for (N, K, g), 16-byte aligned.
 * y_dev      out: fp16 [M, N] row-major, 2-byte aligned.
 * workspace_dev / workspace_bytes: at least w4a16_workspace_bytes(M, N, K, g)
 *            bytes, 256-byte aligned, ZERO-FILLED BEFORE ITS FIRST USE; the
 *            kernels leave it ready for the next call. Calls sharing one
 *            workspace must not overlap on the device.
 * M >= 1, N >= 1, K >= 8 with K % 8 == 0 (the activation rows' byte stride
 * must be a multiple of 16), g a positive multiple of 8; K % g may be
 * anything (the last group is partial).
 *
 * Follows: fp16 activations times 4-bit weights on the tensor cores,
 * memory-bound at small batch and compute-bound at large batch -- the Marlin
 * post ("FP16xINT4" kernel; ideal speed-up of 4x from weight bytes alone).
 *
 * Numerics: q - z is formed exactly. The tensor-memory kernel (M >= 9 by
 * default) rounds each weight once, fp16((q - z) * s), and accumulates in
 * fp32 in tensor memory; the decode kernel (M <= 8) multiplies the exact
 * integers q - z on the tensor cores and scales each group's fp32 partial
 * sum by s when g is a multiple of 64 (else it rounds (q - z) * s once like
 * the other kernel). Pieces of a tile cut along K are added in fp32 in a
 * fixed order; y is rounded once to fp16 (nearest-even). Results are
 * deterministic run to run on one device.
 */
W4_API int w4a16_gemm(const void *x_dev, const void *packed_dev, int64_t M, int64_t N, int64_t K,
               int32_t g, void *y_dev, void *workspace_dev, size_t workspace_bytes, void *stream);

/*
 * As w4a16_gemm with the schedule forced. block_n: activation rows per output
 * tile (8, 16, 32, 64 or 128; 0 = automatic); 8 runs the decode kernel
 * (register-operand MMAs), 16..128 the tensor-memory kernel. ctas: number of persistent
 * CTAs (1..65535; 0 = one per SM). schedule: 0 = automatic, 1 = stream-K
 * (CTAs may cut a tile along K; the cut tiles are finished by a fixup through
 * the workspace), 2 = whole tiles per CTA. The workspace must be at least
 * w4a16_workspace_bytes_ex(M, N, K, g, block_n, ctas, schedule) bytes.
 * Results are identical up to fp32 summation order. For tests and tuning.
 */
W4_API int w4a16_gemm_ex(const void *x_dev, const void *packed_dev, int64_t M, int64_t N, int64_t K,
                  int32_t g, void *y_dev, void *workspace_dev, size_t workspace_bytes,
                  int32_t block_n, int32_t ctas, int32_t schedule, void *stream);
W4_API size_t w4a16_workspace_bytes_ex(int64_t M, int64_t N, int64_t K, int32_t g,
                                int32_t block_n, int32_t ctas, int32_t schedule);

/*
 * Options of w4a16_gemm_opts. Zero-initialise the struct (every zero field
 * means "automatic" / "off"), then set what you need.
 *
 * kernel     0 automatic (the decode kernel for M <= 8, else the tensor-memory
 *            kernel); 1 the decode kernel (register-operand tensor-core MMAs,
 *            M <= 16; the K range of every weight tile may be split between
 *            the CTAs of a thread-block cluster and reduced in distributed
 *            shared memory, so its workspace is the 256-byte error word
 *            alone); 2 the tensor-memory kernel (tcgen05, any M).
 * block_n    tokens per output tile, 0 automatic: decode kernel 8 or 16
 *            (M <= block_n); tensor-memory kernel 16, 32, 64 or 128.
 * ctas       0 automatic. Tensor-memory kernel: persistent CTAs (1..65535).
 *            Decode kernel: clusters (each takes the weight tiles q, q + ctas,
 *            ...).
 * schedule   tensor-memory kernel: 0 automatic, 1 stream-K (a tile may be cut
 *            along K between CTAs and finished through the workspace), 2 whole
 *            tiles per CTA.
 * cluster    decode kernel: CTAs per cluster that split each tile along K:
 *            0 automatic, 1, 2, 4 or 8 (at most the tile's number of 256-wide
 *            K stages, ceil(K / 256)).
 * flags      W4_FLAG_WEIGHTS_STATIC: the caller states that the kernel
 *            launched just before this call on `stream` does not write the
 *            packed weights (true once a model is loaded). The decode kernel
 *            then starts copying its first weight tiles before that kernel
 *            has finished; x is still read only after it.
 *            W4_FLAG_TEST_TIMEOUT (tests only): one wait of the kernel expects
 *            more than will ever come -- the decode kernel's reducer a few
 *            bytes more, the tensor-memory kernel's owner of a cut tile one
 *            piece more -- so that it runs out after wait_limit_cycles. The
 *            kernel then stops early without a fault, y is undefined and
 *            w4_last_device_error reports W4_ERR_TIMEOUT; zero the workspace
 *            before its next use.
 * wait_limit_cycles  0: about 1.5 s. A pipeline wait inside the kernels gives
 *            up after this many SM clock cycles, sets the workspace error
 *            word (W4_ERR_TIMEOUT from w4_last_device_error) and the kernel
 *            returns early.
 * dtype      W4_DTYPE_F16 (0) or W4_DTYPE_BF16: the type of x, of the packed
 *            scales (w4_pack_ex / w4_repack of bf16 scales) and of y. bf16
 *            runs the same kernels with bf16 operands (torchchat issue #1362
 *            runs 'linear:int4' under the bf16 precision): (q - z) is exact in
 *            bf16 too, products accumulate in fp32 and y is rounded once to
 *            bf16. When g is not a multiple of 64, or on the tensor-memory
 *            kernel, each weight is (q - z) * s rounded once to the type, so
 *            the error bound doubles the unit roundoff of the type: 2^-7 for
 *            bf16 against 2^-10 for fp16.
 */
#define W4_FLAG_WEIGHTS_STATIC 1u
#define W4_FLAG_TEST_TIMEOUT 2u
typedef struct {
    int32_t kernel;
    int32_t block_n;
    int32_t ctas;
    int32_t schedule;
    int32_t cluster;
    uint32_t flags;
    uint64_t wait_limit_cycles;
    int32_t dtype;
    int32_t reserved; /* 0 */
} w4a16_options;

/* w4a16_gemm with options (NULL = all automatic). The workspace must be at
 * least w4a16_workspace_bytes_opts(M, N, K, g, opts) bytes. Results are
 * identical up to fp32 summation order across options; for fixed options
 * they are deterministic run to run on one device. */
W4_API int w4a16_gemm_opts(const void *x_dev, const void *packed_dev, int64_t M, int64_t N, int64_t K,
                           int32_t g, void *y_dev, void *workspace_dev, size_t workspace_bytes,
                           const w4a16_options *opts, void *stream);
W4_API size_t w4a16_workspace_bytes_opts(int64_t M, int64_t N, int64_t K, int32_t g,
                                         const w4a16_options *opts);

/*
 * Output epilogues: where the fp32 sums of a GEMM go instead of y[m, n].
 * AutoAWQ issue #31 lists fused qkv among the operations its tests must
 * cover; these two write a fused layer's output in the form the next step
 * reads, so that no separate pass over y follows.
 *
 * W4_EPI_NONE      y [M, N], as w4a16_gemm.
 * W4_EPI_SILU_MUL  a fused gate/up projection whose weight rows alternate:
 *                  row 2j is gate row j, row 2j + 1 is up row j (interleave
 *                  the rows before packing). y [M, N / 2] receives
 *                  silu(gate) * up, silu(v) = v / (1 + e^-v), evaluated in
 *                  fp32 from the two unrounded sums and rounded once. N even.
 * W4_EPI_QKV_SPLIT a fused q/k/v projection whose weight rows come in head
 *                  groups: for each of the N / ((r + 2) d) groups, r query
 *                  heads, then one key head, then one value head, d rows
 *                  each (d = head_dim, r = q_per_group; r = 1 for multi-head
 *                  attention, r > 1 for grouped-query attention). y_dev
 *                  receives q [M, groups * r * d], k_dev and v_dev receive
 *                  k and v [M, groups * d], all row-major. head_dim a
 *                  multiple of 4; N a multiple of (r + 2) d.
 */
#define W4_EPI_NONE 0
#define W4_EPI_SILU_MUL 1
#define W4_EPI_QKV_SPLIT 2
typedef struct {
    int32_t kind;
    int32_t head_dim;     /* W4_EPI_QKV_SPLIT */
    int32_t q_per_group;  /* W4_EPI_QKV_SPLIT */
    int32_t reserved;     /* 0 */
    void *k_dev;          /* W4_EPI_QKV_SPLIT: out, 2-byte aligned */
    void *v_dev;          /* W4_EPI_QKV_SPLIT: out, 2-byte aligned */
} w4a16_epilogue;

/* One GEMM of a group: x [M, K], packed weights [N, K], output y with its
 * epilogue (a zeroed epilogue is W4_EPI_NONE). */
typedef struct {
    const void *x_dev;
    const void *packed_dev;
    void *y_dev;
    int64_t N;
    int64_t K;
    w4a16_epilogue epilogue;
} w4a16_problem;

/*
 * w4a16_gemm_grouped -- `count` (1..4096) independent GEMMs of the same M, g
 * and value type (opts->dtype), enqueued on `stream` by one call. Each
 * problem is checked as w4a16_gemm checks its arguments; the call enqueues
 * nothing unless all pass. A single GEMM with an epilogue is a group of one.
 *
 * Where every problem would run on the decode kernel alone (M <= 8 by
 * default), each launch takes up to 16 problems and walks all their weight
 * tiles in one persistent grid: the weight stream of one problem runs on
 * into the next without a launch boundary, which removes the start-up and
 * tail cost of a launch per GEMM (the bigcode-inference-benchmark roadmap,
 * issue #11, names that cost for many small GEMMs). Problems that share x
 * and K (q, k and v of one layer; gate and up) keep x in shared memory
 * across problems. Above the decode kernel's range, up to 8 problems that
 * share x (the same pointer) and K run in one tensor-memory launch over all
 * their weight tiles (scheduled as one GEMM of the tiles laid one after
 * another, one-tile units; two-tile units from M = 256 do not group).
 * Otherwise the problems run one launch each, in order.
 * Outputs must not overlap one another or any input. The workspace must be
 * at least w4a16_grouped_workspace_bytes(...) bytes, 256-byte aligned and
 * zeroed before first use, like w4a16_gemm's.
 * Returns as w4a16_gemm; W4_ERR_INVALID_ARG also for a bad epilogue.
 */
W4_API int w4a16_gemm_grouped(const w4a16_problem *problems, int32_t count, int64_t M, int32_t g,
                              void *workspace_dev, size_t workspace_bytes, const w4a16_options *opts,
                              void *stream);
W4_API size_t w4a16_grouped_workspace_bytes(const w4a16_problem *problems, int32_t count, int64_t M, int32_t g,
                                            const w4a16_options *opts);

/*
 * The schedule w4a16_gemm picks on the current device: writes block_n, the
 * number of CTAs and the schedule (1 stream-K, 2 whole tiles).
 * Returns W4_OK or an error status.
 */
W4_API int w4a16_gemm_plan(int64_t M, int64_t N, int64_t K, int32_t g,
                    int32_t *block_n, int32_t *ctas, int32_t *schedule);

/*
 * Reads and clears the device error word that GEMM kernels write into the
 * workspace. SYNCHRONISES `stream`. Returns W4_OK, W4_ERR_TIMEOUT (a
 * pipeline wait inside a kernel gave up after about a second and the kernel
 * returned early; y is then undefined, and so are the workspace's tile
 * counters: zero the whole workspace before the next GEMM uses it) or
 * W4_ERR_CUDA.
 */
W4_API int w4_last_device_error(void *workspace_dev, void *stream);

/*
 * w4a16_gemm_noalloc -- w4a16_gemm for callers that cannot allocate device
 * memory. The pages have no counterpart to this call; it exists for users of
 * this library.
 *
 * Some callers have no way to hand the GEMM a workspace: inference engines
 * that reserve all device memory when they start and give each kernel only
 * its inputs and outputs, and plug-ins running inside such engines, which see
 * their input and output tensors but no allocator. This call takes the same
 * inputs and output as w4a16_gemm (same checks, same automatic schedule, same
 * results, bit for bit) but keeps its scratch -- the error word, the per-tile
 * counters and the fp32 partial tiles of tiles split between CTAs -- in a
 * device array inside the library, W4A16_NOALLOC_SCRATCH_BYTES long. It calls
 * no cudaMalloc, cudaFree or other allocating routine.
 *
 *  - Every GPU on which the library is loaded holds that array until the
 *    process exits.
 *  - A problem is refused with W4_ERR_WORKSPACE_TOO_SMALL, before anything is
 *    enqueued, exactly when w4a16_workspace_bytes(M, N, K, g) >
 *    W4A16_NOALLOC_SCRATCH_BYTES. For example, on GB300 (152 SMs) a layer
 *    of N <= 10^6 rows fits for every M <= 32 (at most 4.8 MB of partial
 *    tiles plus 4 bytes per output tile), while M = 64 on a 4096 x 4096
 *    layer (32 tiles, each cut between 4 of 128 CTAs) needs 8.4 MB and is
 *    refused.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any
 *    stream capture begins.
 *  - All calls share the one array: calls that may overlap on the GPU (other
 *    streams, other host threads) race and give wrong results; calls on one
 *    stream are fine. Each call first clears the error word and the counters
 *    on `stream`, so the previous call's leftovers do not matter.
 *  - Device-side timeouts are not reported: there is no workspace to hand to
 *    w4_last_device_error.
 */
#define W4A16_NOALLOC_SCRATCH_BYTES (8u << 20)
W4_API int w4a16_gemm_noalloc(const void *x_dev, const void *packed_dev, int64_t M, int64_t N, int64_t K,
                       int32_t g, void *y_dev, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
