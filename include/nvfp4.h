/*
 * nvfp4.h -- C ABI of the fused NVFP4 linear layer for B300 (sm_103a).
 *
 * The operation: a block-scaled 4-bit (NVFP4) GEMM whose trailing small op is applied in
 * the GEMM epilogue, so each output tile is written to HBM once. Source of the method:
 * page "How fal made Ideogram V4 6x faster" (news.ditty.ir summary of fal's sub-second
 * Ideogram V4 post) -- paragraph "first step: run the transformer in NVFP4", the
 * epilogue-fusion paragraph (RMSNorm with head_dim 256), and the gated-SiLU snippet
 * "C = A @ B; output = SiLU(C[:, :N//2]) * C[:, N//2:]" with B's columns paired at
 * weight-packing time.
 *
 * NVFP4 tensor format used by every call:
 *   codes  : uint8 [rows, K/2], row-major, two 4-bit E2M1 codes per byte, element 2j in the
 *            low nibble of byte j (values +-{0, .5, 1, 1.5, 2, 3, 4, 6}; bit 3 = sign).
 *   scales : one unsigned E4M3 code per 16 contiguous K-elements of a row, stored in the
 *            tiled layout the tensor cores read (see nvfp4_scale_offset): tiles of 128 rows
 *            x 4 blocks = 512 bytes, K-tiles fastest, rows padded to a multiple of 128 with
 *            zero bytes. Size: nvfp4_scales_bytes(rows, K).
 *   tensor scale : one fp32 ts = amax(|x|) / (6 * 448); value = e2m1 * e4m3 * ts.
 *
 * Conventions for every entry point:
 *   - Pointers named x, w, codes, scales, bias, gamma, out, workspace, device_error and the
 *     fp32 tensor-scale pointers are DEVICE pointers owned by the caller; the library never
 *     allocates, frees or keeps them.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream)
 *     and return right after the launch; nothing synchronizes except
 *     nvfp4_get_device_error.
 *   - Host-side checks run before anything is launched; a failed check returns a non-zero
 *     status and launches nothing. A launch failure returns NVFP4_ERR_LAUNCH.
 *   - Every pointer a call reads or writes must be memory of the CURRENT device (cudaMalloc'd
 *     there, or managed memory associated with it). Host memory (pageable or pinned) and
 *     another GPU's memory reached through unified addressing are refused with
 *     NVFP4_ERR_ARG before anything is launched: no kernel of the library, and no TMA tensor
 *     map it encodes, ever covers another device's memory.
 *   - Device-side waits are bounded in time. A wait that runs out writes
 *     NVFP4_ERR_TIMEOUT into *device_error (when device_error is not NULL), frees its
 *     on-chip resources and ends the kernel; the output is then undefined.
 *   - Non-finite inputs (inf, NaN) are outside the format; their results are undefined.
 *   - Requires a compute capability 10.3 GPU (B300); others get NVFP4_ERR_DEVICE.
 *   - One device per process: each kernel's launch attributes (its shared-memory size) and
 *     occupancy figures are set up once, with the device current at the first call; calls
 *     on another device of the same process are not supported (run one process per GPU).
 *   - The FP8 and attention calls below follow the same conventions.
 */
#ifndef NVFP4_H_
#define NVFP4_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define NVFP4_API __attribute__((visibility("default")))
#else
#define NVFP4_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *nvfp4_stream_t;

typedef enum nvfp4_status {
  NVFP4_OK = 0,
  NVFP4_ERR_NULL = 1,     /* a required pointer is NULL */
  NVFP4_ERR_SHAPE = 2,    /* a size or shape rule is broken (see each call) */
  NVFP4_ERR_ALIGN = 3,    /* a pointer or leading dimension breaks a 16-byte rule */
  NVFP4_ERR_DEVICE = 4,   /* no current CUDA device, or it is not compute capability 10.3 */
  NVFP4_ERR_LAUNCH = 5,   /* a CUDA launch or runtime call failed */
  NVFP4_ERR_TIMEOUT = 6,  /* device-side: a bounded wait ran out (read via device_error) */
  NVFP4_ERR_ARG = 7       /* an enum or scalar argument is out of range */
} nvfp4_status;

typedef enum nvfp4_epilogue {
  NVFP4_EPI_BIAS = 0,          /* y = alpha * acc + bias[n] */
  NVFP4_EPI_HEAD_RMSNORM = 1,  /* bias, then per-head RMSNorm on columns [0, norm_cols) */
  NVFP4_EPI_GATED_SILU = 2     /* y[:, j] = SiLU(g_j) * u_j over interleaved (gate, up) pairs */
} nvfp4_epilogue;

typedef enum nvfp4_out_dtype {
  NVFP4_OUT_BF16 = 0,  /* round to nearest even */
  NVFP4_OUT_FP32 = 1
} nvfp4_out_dtype;

/* Bytes of a tiled scale buffer for `rows` rows of K elements (K % 64 == 0):
 * ceil(rows / 128) * (K / 64) * 512. Returns 0 for rows <= 0 or a bad K. */
NVFP4_API size_t nvfp4_scales_bytes(int64_t rows, int64_t K);

/* Byte offset, inside the tiled scale buffer, of the E4M3 scale of row `row` and 16-element
 * block `kblock` (0 <= kblock < K/16):
 *   ((row / 128) * (K / 64) + kblock / 4) * 512 + (row % 32) * 16 + ((row / 32) % 4) * 4
 *   + kblock % 4
 * This is the 1-D block-scale layout Blackwell tensor cores read (128 rows x 4 scales per
 * 512-byte tile). Returns -1 for out-of-range arguments. */
NVFP4_API int64_t nvfp4_scale_offset(int64_t row, int64_t kblock, int64_t K);

/* Bytes of scratch `workspace` that nvfp4_quantize / nvfp4_pack_weights need (16).
 * nvfp4_quantize expects the workspace zero-filled before its first use and leaves it
 * zero-filled again (its amax word and CTA counters), so allocate and zero it once and
 * reuse it; nvfp4_pack_weights also leaves it zero-filled. Calls that use the same
 * workspace must not overlap on the GPU. After a call that reported a device-side time-out
 * (a NaN tensor_scale, see nvfp4_quantize) zero it again before reuse. */
NVFP4_API size_t nvfp4_workspace_bytes(void);

/*
 * nvfp4_quantize -- bf16 activations -> NVFP4 (the quantizer that feeds the GEMM).
 *
 *   x        bf16 [M, K] with row stride ldx elements (ldx >= K, ldx % 8 == 0, x 16-byte
 *            aligned).
 *   codes    out, uint8 [M, K/2] contiguous (16-byte aligned).
 *   scales   out, nvfp4_scales_bytes(M, K) bytes, tiled layout; padding rows are written 0.
 *   tensor_scale     out, fp32 [1]: the ts used.
 *   tensor_scale_in  optional fp32 [1] device pointer. NULL: ts = amax(|x|) / 2688 of this
 *            x (dynamic per call; costs one extra read of x). Non-NULL: that static ts is
 *            used and x is read once.
 *   workspace  >= nvfp4_workspace_bytes() device bytes, 16-byte aligned, zero-filled
 *            before its first use and then reused (see nvfp4_workspace_bytes); may be NULL
 *            when tensor_scale_in is given.
 * Dynamic scale and 16-byte aligned rows, when at least a quarter of each CTA's rows fit in
 * 200 KB of shared memory (one CTA per SM; M * K up to about 14.8M elements entirely, the
 * down-projection input [4608, 12288] a quarter): one cooperative launch reads x, keeps
 * those rows in shared memory, reduces the amax, meets the other CTAs at a grid-wide barrier
 * on the workspace words and quantizes, reading only the rows not kept a second time.
 * Otherwise two launches: an amax pass over x (skipped for a static scale), then the
 * quantize pass, which walks x backwards so that what the amax pass read last is still in
 * L2. Codes and scales are identical either way.
 * If a device-side wait of the single launch runs out of time (NVFP4_WAIT_TIMEOUT_NS,
 * default 2 s; it cannot under a cooperative launch unless the GPU misbehaves), tensor_scale
 * is written NaN, no codes are written, and the workspace must be zeroed before reuse.
 * Per block of 16: s = E4M3(bamax / fp32(6 ts)) (nearest even, saturating at 448);
 * d = fp32(dec(s) ts); if d < 2^-126 the block stores scale 0 and codes +0; otherwise each
 * element is coded E2M1(fp32(x * fp32(1/d))) (nearest even, saturating at 6; a negative
 * value that rounds to 0 keeps its sign, code 0x8). ts <= 0 zeroes everything.
 * Rules: M >= 0, K > 0, K % 64 == 0, M * K < 2^34. M == 0 launches nothing and returns
 * NVFP4_OK after the shape checks (the pointers may then be NULL).
 */
NVFP4_API nvfp4_status nvfp4_quantize(const void *x, int64_t M, int64_t K, int64_t ldx,
                            uint8_t *codes, uint8_t *scales, float *tensor_scale,
                            const float *tensor_scale_in, void *workspace,
                            nvfp4_stream_t stream);

/*
 * nvfp4_pack_weights -- offline packing of a linear layer's weight W [K, N] (y = x @ W).
 *
 *   w        bf16 [K, N] row-major (16-byte aligned, N % 8 == 0).
 *   gated_interleave  0: packed row n = column n of W.
 *            1: the gated-SiLU pairing from the page's packing sentence: packed row 2j =
 *            gate column j, packed row 2j+1 = up column N/2 + j (N even).
 *   codes    out, uint8 [N, K/2] (K-major: W transposed), 16-byte aligned.
 *   scales   out, nvfp4_scales_bytes(N, K) bytes, tiled layout.
 *   tensor_scale  out, fp32 [1]: ts = amax(|W|) / 2688.
 *   workspace  >= nvfp4_workspace_bytes() device bytes.
 * Quantization rules are those of nvfp4_quantize, applied to the rows of the packed W^T.
 * Rules: K > 0, K % 64 == 0, N > 0, N % 8 == 0.
 */
NVFP4_API nvfp4_status nvfp4_pack_weights(const void *w, int64_t K, int64_t N, int gated_interleave,
                                uint8_t *codes, uint8_t *scales, float *tensor_scale,
                                void *workspace, nvfp4_stream_t stream);

/*
 * nvfp4_gemm -- block-scaled FP4 GEMM with a fused epilogue.
 *
 *   acc[m, n] = sum over 16-blocks kb of sA[m,kb] sB[n,kb] sum_{k in kb} qA[m,k] qB[n,k]
 *   z[m, n]   = alpha * acc[m, n] + bias[n],   alpha = (*a_ts) * (*b_ts)   (fp32)
 *
 *   a_codes/a_scales/a_ts  activations A [M, K] as written by nvfp4_quantize.
 *   b_codes/b_scales/b_ts  weights B [N, K] (K-major) as written by nvfp4_pack_weights.
 *   epi  NVFP4_EPI_BIAS:         y = z, out [M, N].
 *        NVFP4_EPI_HEAD_RMSNORM: columns n < norm_cols, in heads of head_dim columns:
 *                                y = z * rsqrt(mean_head(z^2) + eps) * gamma[n];
 *                                other columns y = z. out [M, N].
 *        NVFP4_EPI_GATED_SILU:   B packed with gated_interleave = 1; for j < N/2,
 *                                g = z[:, 2j], u = z[:, 2j+1],
 *                                y[:, j] = g / (1 + exp(-g)) * u. out [M, N/2].
 *   bias   fp32, NULL for none. Indexed by ORIGINAL output column: length N; for the gated
 *          epilogue bias[j] belongs to gate column j and bias[N/2 + j] to up column j.
 *   gamma  fp32 [norm_cols], required for HEAD_RMSNORM, ignored otherwise.
 *   head_dim  HEAD_RMSNORM: one of 32, 64, 128, 256. norm_cols % head_dim == 0,
 *          0 <= norm_cols <= N.
 *   out    16-byte aligned; row stride ldo elements (ldo >= output width; ldo % 8 == 0
 *          for BF16, % 4 for FP32).
 *   device_error  optional int [1]: receives NVFP4_ERR_TIMEOUT if a device wait runs out;
 *          the caller zeroes it. NULL: device timeouts are not reported.
 * Rules: M >= 0, N > 0, N % 32 == 0, K > 0, K % 64 == 0, M * K < 2^34 and N * K < 2^34 (the
 * operand bounds of nvfp4_quantize and nvfp4_pack_weights), ceil(M / 256) * ceil(N / 256) <
 * 2^31 (256 x 256 output tiles), all code and scale pointers 16-byte aligned. Shapes outside
 * these return NVFP4_ERR_SHAPE. M == 0 launches nothing and returns NVFP4_OK after the shape
 * and enum checks (the pointers may then be NULL).
 */
NVFP4_API nvfp4_status nvfp4_gemm(const uint8_t *a_codes, const uint8_t *a_scales, const float *a_ts,
                        const uint8_t *b_codes, const uint8_t *b_scales, const float *b_ts,
                        int64_t M, int64_t N, int64_t K, nvfp4_epilogue epi,
                        const float *bias, const float *gamma, int head_dim,
                        int64_t norm_cols, float eps, nvfp4_out_dtype out_dtype, void *out,
                        int64_t ldo, int *device_error, nvfp4_stream_t stream);

/*
 * nvfp4_gemm_nvfp4_out -- the same GEMM and epilogue, writing the output as NVFP4 for the
 * next layer instead of bf16/fp32: no bf16 round trip through HBM between two FP4 layers
 * (page "How fal made Ideogram V4 6x faster", NVFP4 paragraph: a 4-bit matmul only pays off
 * when the bytes around it shrink too, so the quantize of a layer's output belongs in the
 * producing kernel).
 *
 *   out_tensor_scale  fp32 [1] device: the output's STATIC tensor scale ts_out (a dynamic
 *          scale would need the whole output's amax before the first block is coded; a
 *          caller can use, e.g., a calibrated value or the previous step's amax / 2688).
 *   out_codes   uint8 [M, W/2] contiguous, W = output width (N, or N/2 for GATED_SILU).
 *   out_scales  nvfp4_scales_bytes(M, W) bytes, tiled layout; padding rows written 0.
 * Each output value is first rounded to bf16 exactly as the bf16 output mode stores it, then
 * the 16-blocks along a row are quantized as nvfp4_quantize does with tensor_scale_in =
 * out_tensor_scale: the codes and scales are identical to nvfp4_gemm(..., NVFP4_OUT_BF16)
 * followed by nvfp4_quantize(y, static ts), and feed nvfp4_gemm as its A operand (K = W).
 * Rules: those of nvfp4_gemm, plus W % 64 == 0; out_codes and out_scales 16-byte aligned.
 */
NVFP4_API nvfp4_status nvfp4_gemm_nvfp4_out(const uint8_t *a_codes, const uint8_t *a_scales,
                        const float *a_ts, const uint8_t *b_codes, const uint8_t *b_scales,
                        const float *b_ts, int64_t M, int64_t N, int64_t K, nvfp4_epilogue epi,
                        const float *bias, const float *gamma, int head_dim, int64_t norm_cols,
                        float eps, const float *out_tensor_scale, uint8_t *out_codes,
                        uint8_t *out_scales, int *device_error, nvfp4_stream_t stream);

/*
 * FP8 variant -- E4M3 operands with one fp32 scale per tensor, the same fused GEMM and
 * epilogues, for layers kept at higher precision than NVFP4. Pages "WaveSpeedAI x
 * DataCrunch: FLUX real-time image inference on B200" (BF16/FP8 mixed precision through
 * Blackwell's Transformer Engine) and "FLUX.1-dev inference optimization with LoRAs" (FP8
 * quantization: lossy, the best speed/memory trade-off); neither fixes the scheme, which is:
 *   ts = amax / 448 (448 = largest E4M3 value), fp32 IEEE division;
 *   code = E4M3(fp32(x * fp32(1 / ts))), round to nearest even, saturating at +-448, sign
 *   kept (a negative value that rounds to zero is 0x80);
 *   a tensor with ts < 2^-126 (all zeros, or 1 / ts not finite) is stored as codes 0x00.
 * Workspaces, streams, device errors and status codes are those of the NVFP4 calls.
 */

/*
 * fp8_quantize -- x bf16 [M, K] (row stride ldx elements) -> codes uint8 [M, K] (contiguous,
 * element k of row m at byte m * K + k), *tensor_scale = ts used (fp32, device).
 *   tensor_scale_in  NULL: dynamic ts = amax(|x|) / 448 (two launches: amax, then encode;
 *          `workspace` (nvfp4_workspace_bytes(), zero on first use) is left zeroed);
 *          else a static fp32 ts on the device and `workspace` may be NULL.
 * Rules: M >= 0 (M == 0 does nothing), K > 0, K % 64 == 0, ldx >= K, ldx % 8 == 0; x, codes,
 * workspace 16-byte aligned, tensor_scale 4-byte aligned. Non-finite inputs: undefined.
 */
NVFP4_API nvfp4_status fp8_quantize(const void *x, int64_t M, int64_t K, int64_t ldx, uint8_t *codes,
                                    float *tensor_scale, const float *tensor_scale_in, void *workspace,
                                    nvfp4_stream_t stream);

/*
 * fp8_pack_weights -- W bf16 [K, N] (row-major, x @ W) -> codes uint8 [N, K] (K-major: packed
 * row p holds the K values of output column n(p)), *tensor_scale = amax(|W|) / 448.
 *   gated_interleave  1: packed row 2j = column j (gate), 2j+1 = column N/2 + j (up), the
 *          pairing of the gated-SiLU epilogue; 0: row p = column p.
 * Rules: K % 64 == 0, N % 8 == 0, K / 64 <= 65535; w, codes, workspace 16-byte aligned.
 */
NVFP4_API nvfp4_status fp8_pack_weights(const void *w, int64_t K, int64_t N, int gated_interleave, uint8_t *codes,
                                        float *tensor_scale, void *workspace, nvfp4_stream_t stream);

/*
 * fp8_gemm -- y = epilogue(a_ts * b_ts * (A B^T) + bias) with E4M3 A [M, K] and B [N, K] (codes
 * from fp8_quantize and fp8_pack_weights), fp32 accumulation on the tensor cores
 * (tcgen05.mma kind::f8f6f4); epilogue, bias, gamma, head_dim, norm_cols, eps, out_dtype,
 * out, ldo, device_error and the rules are those of nvfp4_gemm (K % 64 == 0; a_codes, b_codes
 * 16-byte aligned).
 */
NVFP4_API nvfp4_status fp8_gemm(const uint8_t *a_codes, const float *a_ts, const uint8_t *b_codes,
                                const float *b_ts, int64_t M, int64_t N, int64_t K, nvfp4_epilogue epi,
                                const float *bias, const float *gamma, int head_dim, int64_t norm_cols,
                                float eps, nvfp4_out_dtype out_dtype, void *out, int64_t ldo,
                                int *device_error, nvfp4_stream_t stream);

/*
 * Attention -- the DiT block's other large op, between the QKV projection and the output
 * projection (page "How fal made Ideogram V4 6x faster": a pass costs the sum of its layers).
 * Scaled dot-product attention per head, no mask, bf16 in and out, fp32 softmax and
 * accumulation on the tensor cores (tcgen05.mma kind::f16):
 *   out[m, h*D + d] = sum_j softmax_j(q_m . k_j / sqrt(D)) v_j[d],   D = head_dim = 256,
 * with q_m = qkv[m, h*D .. h*D + D), k_j = qkv[j, H + h*D ..), v_j = qkv[j, 2H + h*D ..),
 * H = heads * D: the layout the QKV GEMM writes (Q | K | V, heads side by side in each).
 * The probabilities are rounded to bf16 before they multiply V (as FlashAttention kernels
 * do), so results match exact attention to about 2^-9 relative, not bit for bit.
 */

/* Bytes of the attention_fwd workspace (V transposed, bf16 [heads * 256, round_up(M, 8)]);
 * 0 for M <= 0 or heads <= 0. */
NVFP4_API size_t attention_workspace_bytes(int64_t M, int heads);

/*
 * attention_fwd -- qkv bf16 [M, ld_qkv >= 3 * heads * 256] -> out bf16 [M, ldo >= heads * 256].
 * workspace: attention_workspace_bytes(M, heads) bytes of device memory (contents need not
 * be initialised; overwritten). Two launches on `stream`: the V transpose, then the attention
 * kernel (one CTA per 128 queries and head).
 * Rules: head_dim == 256 (else NVFP4_ERR_ARG); 1 <= heads <= 256; M >= 0 (M == 0 does
 * nothing); ld_qkv and ldo multiples of 8; qkv, workspace, out 16-byte aligned.
 * device_error: as for nvfp4_gemm (a bounded wait that expired writes NVFP4_ERR_TIMEOUT).
 */
NVFP4_API nvfp4_status attention_fwd(const void *qkv, int64_t M, int64_t ld_qkv, int heads, int head_dim,
                                     void *workspace, void *out, int64_t ldo, int *device_error,
                                     nvfp4_stream_t stream);

/* Synchronizes `stream`, copies *device_error to *code, then zeroes the device word.
 * Returns NVFP4_ERR_NULL for NULL pointers, NVFP4_ERR_LAUNCH if a CUDA call fails. */
NVFP4_API nvfp4_status nvfp4_get_device_error(int *device_error, int *code, nvfp4_stream_t stream);

/* Static, human-readable name of a status code ("NVFP4_OK", ...). Never NULL. */
NVFP4_API const char *nvfp4_status_string(nvfp4_status status);

/*
 * nvfp4_debug_wait_timeout -- exercises the bounded device wait.
 * Launches one small kernel that waits on an on-chip barrier that nothing ever completes,
 * for at most timeout_ns nanoseconds (1 <= timeout_ns <= 10^10), then writes
 * NVFP4_ERR_TIMEOUT into *device_error and returns normally; the CUDA context stays usable.
 * Used by the tests of the error path; it computes nothing.
 */
NVFP4_API nvfp4_status nvfp4_debug_wait_timeout(int *device_error, int64_t timeout_ns,
                                      nvfp4_stream_t stream);

/*
 * Debug build -- the same library compiled with -DNVFP4_DEBUG (libnvfp4_debug.so, built beside
 * libnvfp4.so). Its kernels check the indices of their stores (and of the few loads whose
 * index is computed): output rows and columns against M and the output width, the
 * 16-byte alignment of every TMA store's first coordinate, code and scale offsets against
 * the buffers' sizes, shared-memory offsets against the rows a CTA holds, bias indices against
 * N. A failed check skips that access and is counted on the device; nothing traps, so the
 * context stays usable. Release builds compile the checks out.
 */

/* 1 if this library was built with the index checks, 0 otherwise. Needs no GPU. */
NVFP4_API int nvfp4_debug_build(void);

/* Synchronizes the device, writes to *count the number of index checks that failed in the
 * library's kernels since the last call (always 0 in a release build), and clears it. */
NVFP4_API nvfp4_status nvfp4_debug_index_failures(int64_t *count);

/* Instruction kinds of nvfp4_debug_mma_rate. */
typedef enum nvfp4_probe_kind {
  NVFP4_PROBE_NVFP4 = 0,  /* tcgen05.mma kind::mxf4nvf4.block_scale.block16, K = 64 */
  NVFP4_PROBE_FP8 = 1,    /* tcgen05.mma kind::f8f6f4 (E4M3 x E4M3), K = 32 */
  NVFP4_PROBE_BF16 = 2    /* tcgen05.mma kind::f16 (BF16 x BF16), K = 16 */
} nvfp4_probe_kind;

/*
 * nvfp4_debug_mma_rate -- measures the rate at which this device's tensor pipe retires one
 * tcgen05.mma instruction kind and shape, the ceiling of any GEMM built from it (the fused
 * GEMM above issues NVFP4 at cta_group 2, N = 256).
 * Launches `ctas` CTAs (cta_group 1: M = 128 on one SM each) or `ctas` CTA pairs (cta_group
 * 2: M = 256 across two SMs), one per SM; one thread of each (of each pair's leader) issues
 * `iters` back-to-back instructions on zero operands held in shared memory (128-byte
 * swizzled, K-major, 32 bytes of each row per instruction; NVFP4 block scales in TMEM) into
 * a TMEM accumulator. It computes nothing useful.
 *   out  device int64 [2 * ctas], zero-filled by the caller: out[2c] = SM cycles and
 *        out[2c + 1] = nanoseconds from the first issue to the completion of the last
 *        instruction, for CTA (pair) c; -1 if a device wait ran out.
 * FLOP per instruction: 2 * M * n * K.
 * Rules: kind one of nvfp4_probe_kind; cta_group 1 or 2; n in {64, 128, 192, 256};
 * 1 <= iters <= 4,000,000; 1 <= ctas <= SM count (cta_group 1) or SM count / 2 (cta_group 2).
 */
NVFP4_API nvfp4_status nvfp4_debug_mma_rate(nvfp4_probe_kind kind, int cta_group, int n, int64_t iters,
                                            int ctas, int64_t *out, int *device_error,
                                            nvfp4_stream_t stream);

/*
 * nvfp4_quantize_noalloc -- nvfp4_quantize (dynamic tensor scale) without a workspace
 * argument, for callers that cannot allocate device memory. The pages have no counterpart:
 * this is a packaging of the quantizer, not part of the method.
 *
 * Who needs it: a host framework's plugin interface that hands a kernel its inputs and
 * outputs but no scratch buffer; a serving process that reserves all device memory in its
 * own pool at start-up and forbids allocations afterwards; a latency-critical loop that
 * must not call cudaMalloc/cudaFree, because those can synchronize the device or fail for
 * lack of memory in the middle of a request.
 *
 * Arguments, checks and results are those of nvfp4_quantize with tensor_scale_in = NULL;
 * every check runs first, so a refused call touches neither the scratch nor the stream.
 * The scratch (the quantizer's 16 workspace bytes: the amax word, two grid-barrier counters
 * and a failure flag) is a fixed 256-byte array inside the library, resident on every GPU
 * that loads it until the process exits; a need above 256 bytes would be refused with
 * NVFP4_ERR_SHAPE. Nothing is allocated: no cudaMalloc, cudaFree or allocating library
 * routine is called. The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it; make that first call
 * before any stream capture. Every call shares the array and zeroes the 16 bytes it uses on
 * `stream` before the quantizer runs, so calls that overlap on the GPU (different streams,
 * or different host threads) race: serialize them.
 */
NVFP4_API nvfp4_status nvfp4_quantize_noalloc(const void *x, int64_t M, int64_t K, int64_t ldx,
                                              uint8_t *codes, uint8_t *scales,
                                              float *tensor_scale, nvfp4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H_ */
