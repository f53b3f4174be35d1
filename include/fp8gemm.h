/*
 * fp8gemm — FP8 (E4M3) GEMM library for one GB300 GPU (sm_103a).
 *
 *   C[M,N] = (sA . A[M,K]) (sB . B[N,K])^T
 *
 * E4M3 operands ("fn" variant: max 448, no infinities, NaN = S.1111.111),
 * fp32 accumulation in tensor memory, bf16 or fp32 output.  Three GEMM entry
 * points: per-tensor scales, 1x32 block scales along K, and the grouped (MoE)
 * form of the block-scaled GEMM.  Plus the operand quantiser that produces the
 * codes and scales these entry points consume.
 *
 * Sources for the operation (page titles, sections):
 *   [JAX-BW]  "Optimizing FP8 GEMM kernels in JAX with Triton for Blackwell
 *             GPUs: TMA async loads and warp-level primitives" — format and
 *             parameter paragraph (E4M3, 32-wide microscaling blocks, 128x128
 *             TMA tiles, multicast of the shared operand), GEMM pseudo-kernel
 *             (fp32 accumulate, down-converting store), MoE paragraph (grouped
 *             GEMM over experts).
 *   [TRITON-FP8] "Triton FP8 CUTLASS-named kernel benchmarking" — parameter
 *             list (torch.float8_e4m3fn), monitoring checklist (2*M*N*K FLOPs).
 *   [TUT-12]  "Triton tutorial ch. 12: Hopper / Blackwell architecture
 *             features" — 12.2.3 (TMA alignment rules), 12.6.1-12.6.2 (TMEM,
 *             tcgen05, MXFP8 micro-scaling), 12.7 (grouped raster order of a
 *             persistent matmul), 12.8 Q3 (TMEM column budget).
 *
 * Conventions shared by every entry point
 *   - All data pointers are DEVICE pointers owned by the caller.  The library
 *     keeps no reference after the call returns.
 *   - Calls are asynchronous on `stream` (stream order only).  Host-side
 *     argument checks are synchronous: a call that fails them launches nothing
 *     and returns the error.  Errors found on the device (a bad scale value,
 *     inconsistent group counts, an internal wait that timed out) are recorded
 *     in a per-device status word read by fp8_gemm_status().
 *   - Row-major, densely packed: A[M,K] (row stride K), B[N,K] (row stride K),
 *     C[M,N] (row stride N).  "K-contiguous B" means C = A B^T.
 *   - Alignment [TUT-12 12.2.3]: every pointer 16-byte aligned, K % 16 == 0,
 *     N * sizeof(out element) % 16 == 0.  Violations return FP8G_ERR_ALIGNMENT.
 *   - M, N, K >= 1 (grouped: total_rows >= 0).  M and N need not be multiples
 *     of the tile; out-of-range rows/columns are neither read past the end nor
 *     written.
 *   - Thread safety: calls from several host threads, on any streams, are safe.
 *   - Device memory: fp8_gemm and fp8g_quantize_e4m3 allocate nothing.  The
 *     block-scaled entry points repack the fp32 scales into the tensor core's
 *     UE8M0 layout in a temporary of about (rows of A + rows of B) * K/32
 *     bytes, taken from a library-owned memory pool with
 *     cudaMallocFromPoolAsync on `stream` and returned with cudaFreeAsync on
 *     `stream` (stream-ordered, so calls on different streams never share
 *     it).  Shapes with few output tiles (split-K, or one CTA per 128 x 128
 *     tile: see fp8g_gemm_plan) and grouped calls on 128 x 128 tiles (see
 *     fp8g_grouped_plan: BM = 128) skip the temporary: the GEMM converts the
 *     scales itself.  The library also holds one status word per device (a
 *     static device variable) and a host-side tensor-map cache.
 */
#ifndef FP8GEMM_H
#define FP8GEMM_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define FP8G_API __attribute__((visibility("default")))
#else
#define FP8G_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8G_OK = 0,
    FP8G_ERR_INVALID_ARG = 1,       /* null pointer, bad size, bad enum, counts inconsistent */
    FP8G_ERR_ALIGNMENT = 2,         /* pointer / row-stride alignment rule broken */
    FP8G_ERR_UNSUPPORTED_SHAPE = 3, /* K % 32 != 0 for block scales, E > 64, sizes too large */
    FP8G_ERR_SCALE_FORMAT = 4,      /* a block scale is not a positive power of two */
    FP8G_ERR_CUDA = 5,              /* a CUDA runtime/driver call failed */
    FP8G_ERR_TIMEOUT = 6,           /* a device-side wait exceeded its limit; kernel aborted */
    FP8G_ERR_DEVICE = 7             /* no usable sm_100-family device */
} fp8g_status;

typedef enum { FP8G_OUT_BF16 = 0, FP8G_OUT_F32 = 1 } fp8g_out;

/*
 * Operand element formats [JAX-BW format paragraph: E4M3 for its
 * range/precision balance, E5M2 the wider-range alternative; TUT-12 12.6.1:
 * the fifth-generation tensor core's FP4 micro-scaling formats].  E4M3
 * ("fn"): bias 7, 3 mantissa bits, no infinities, NaN = S.1111.111, largest
 * finite 448.  E5M2: bias 15, 2 mantissa bits, infinities and NaNs in the top
 * binade, largest finite 57344.  Both one code per byte.  E2M1 (FP4; with 1x32
 * power-of-two scales this is MXFP4): bias 1, 1 mantissa bit, values 0, 0.5,
 * 1, 1.5, 2, 3, 4, 6, no infinities or NaNs (the quantiser saturates to +-6
 * and writes NaN as +6); two codes per byte, element 2j in the low nibble of
 * byte j, so a row of K elements takes K/2 bytes.  A GEMM with an E2M1
 * operand needs K % 128 == 0 (else FP8G_ERR_UNSUPPORTED_SHAPE) and that
 * operand 32-byte aligned (else FP8G_ERR_ALIGNMENT), and reads half the
 * operand bytes.  E2M1 x E2M1 with 1x32 power-of-two scales on shapes that
 * take CTA pairs (see fp8g_gemm_plan: BM = 256) and K % 256 == 0 runs the
 * FP4-rate MMA (kind::mxf4); every other E2M1 call runs the FP8-rate MMA
 * (kind::f8f6f4 / mxf8f6f4).  The entry points without a format argument
 * take E4M3.
 * FP6 [TUT-12 12.6.1 hardware table, 12.6.4 stability table; with 1x32
 * power-of-two scales this is MXFP6]: E2M3 (bias 1, 3 mantissa bits, values
 * k/8 below 2, largest 7.5) and E3M2 (bias 3, 2 mantissa bits, subnormals
 * k/16, largest 28), no infinities or NaNs (the quantiser saturates and
 * writes NaN as the largest positive value, code 0x1F).  Four codes in three
 * bytes: code i of a row in bits 6i .. 6i+5 of the row read as a
 * little-endian bit string, so a row of K elements takes 3K/4 bytes.  The
 * GEMM rules of E2M1 apply (K % 128 == 0, the operand 32-byte aligned); FP6
 * runs the FP8-rate MMA and reads three quarters of the operand bytes.  Any
 * two formats may be paired.
 */
typedef enum {
    FP8G_E4M3 = 0,
    FP8G_E5M2 = 1,
    FP8G_E2M1 = 2,
    FP8G_E2M3 = 3,
    FP8G_E3M2 = 4
} fp8g_format;

/*
 * Fused-epilogue activations [TRITON-FP8 benchmark list: a bias_add_relu
 * epilogue beside the plain GEMM].  Applied per output element after the
 * per-tensor scale and an optional per-column bias, before the output
 * rounding:  out( act( fl32( fl32(alpha * acc) + bias[j] ) ) ).
 * RELU: v < 0 ? 0 : v (NaN stays NaN).  GELU: 0.5 v (1 + erf(v / sqrt 2)).
 */
typedef enum { FP8G_ACT_NONE = 0, FP8G_ACT_RELU = 1, FP8G_ACT_GELU = 2 } fp8g_act;

/* Largest expert count accepted by fp8_grouped_gemm. */
#define FP8G_MAX_EXPERTS 64

/*
 * Per-tensor-scaled GEMM [JAX-BW, GEMM pseudo-kernel; TRITON-FP8 dtype].
 *   C[i,j] = out( fl32( fl32(sA*sB) * acc_ij ) ),  acc_ij = sum_k a_ik b_jk in fp32
 * A: uint8 E4M3 codes [M,K]; B: uint8 E4M3 codes [N,K]; scale_a, scale_b: device
 * pointers to one fp32 each; C: [M,N] bf16 (RNE) or fp32 per `out`.
 * Errors: FP8G_ERR_INVALID_ARG (null pointer, M/N/K < 1, bad `out`),
 * FP8G_ERR_ALIGNMENT, FP8G_ERR_CUDA (launch failure).
 */
FP8G_API fp8g_status fp8_gemm(const void *A, const void *B, const float *scale_a, const float *scale_b,
                     void *C, int out, int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * 1x32 block-scaled GEMM [JAX-BW microscaling paragraph; TUT-12 12.6.1 MXFP8].
 *   C[i,j] = out( sum_kb sfa[i,kb] * sfb[j,kb] * sum_{k in kb} a_ik b_jk )
 * sfa: fp32 [M, K/32] row-major; sfb: fp32 [N, K/32].  Every scale must be a
 * positive power of two (2^-126 .. 2^127; NaN propagates as NaN); the tensor
 * core applies it exactly as an 8-bit exponent.  Any other value records
 * FP8G_ERR_SCALE_FORMAT in the status word (the output is then unspecified).
 * K % 32 == 0 (else FP8G_ERR_UNSUPPORTED_SHAPE).  Other rules as fp8_gemm.
 * Runs two kernels on `stream`: the scale packing (scales -> UE8M0 chunks,
 * which also performs the scale check) and the GEMM; shapes with few output
 * tiles (fewer than SMs / 2 tiles of 128 x 256: plan split > 1, or plan
 * BM = BN = 128 below 16 K steps) run the GEMM alone, which then converts and
 * checks the scales of each K step itself.
 */
FP8G_API fp8g_status fp8_gemm_blockscaled(const void *A, const void *B, const float *sfa,
                                 const float *sfb, void *C, int out, int64_t M, int64_t N,
                                 int64_t K, cudaStream_t stream);

/*
 * Allocation-free form of fp8_gemm_blockscaled (the source pages have no
 * counterpart; this is a library convenience).  For callers that cannot let
 * the library allocate device memory, e.g. code under a fixed device-memory
 * budget, behind an allocator that owns every device byte, or on a path where
 * allocation calls are not allowed.  Same arguments, results and errors as
 * fp8_gemm_blockscaled, but the repacked scale factors live in a fixed 16 MiB
 * device array that is part of the library (every GPU that loads the library
 * holds it until the process exits); no call allocates or frees memory.
 * Limit: the repacked scales, at most (ceil(M/128) + 8*ceil(N/256)) *
 * ceil(K/128) * 512 bytes, must fit in 16 MiB (M = N = K = 8192 needs
 * 10 MiB); larger shapes return FP8G_ERR_UNSUPPORTED_SHAPE without launching.
 * The first call on a device looks up the array's device address (one
 * cudaGetSymbolAddress with that device current); make that first call before
 * any stream capture.  All calls share the one array: calls whose kernels can
 * overlap on the GPU (different streams without ordering between them) race
 * and must not be issued.  Nothing in the array needs to start at zero: each
 * call rewrites the part it reads.
 */
FP8G_API fp8g_status fp8_gemm_blockscaled_noalloc(const void *A, const void *B, const float *sfa,
                                                  const float *sfb, void *C, int out, int64_t M,
                                                  int64_t N, int64_t K, cudaStream_t stream);

/*
 * Grouped (MoE) block-scaled GEMM [JAX-BW MoE paragraph].
 * Expert e owns rows [off_e, off_e + counts[e]) of A and C, off = exclusive
 * prefix sum of counts; those rows multiply B[e]:
 *   C[r, :] = blockscaled(A[r, :], B[e])   for off_e <= r < off_e + counts[e]
 * A: [total_rows, K] (rows already gathered per expert, expert-contiguous);
 * B: [E, N, K]; sfa: fp32 [total_rows, K/32]; sfb: fp32 [E, N, K/32];
 * C: [total_rows, N]; counts: DEVICE int32[E], each >= 0, summing to total_rows
 * (checked on the device: a mismatch records FP8G_ERR_INVALID_ARG and writes
 * no output).  Empty experts produce no tiles and no rows; their weights and
 * weight scales are not read (so their scales are not checked either).
 * Plans on 128 x 128 tiles (fewer rows than a wave of 128 x 256 tiles; see
 * fp8g_grouped_plan) convert the scales inside the GEMM kernel, each CTA those
 * of its own tiles; 256 x 256 tiles on CTA pairs take them repacked by a
 * packing kernel first.
 * offsets_out (nullable): device int32[E+1] receives the exclusive prefix.
 * tile_map_out (nullable): device int32[4 * max_tiles] (see fp8g_grouped_plan)
 * receives, for linear tile t, (expert, m_tile, n_tile, 0): experts in index
 * order, expert e's ceil(M_e/BM)*ceil(N/BN) tiles in the grouped raster order.
 * Entries past the actual tile count are left untouched.
 * 1 <= E <= FP8G_MAX_EXPERTS.  Other rules as fp8_gemm_blockscaled.
 */
FP8G_API fp8g_status fp8_grouped_gemm(const void *A, const void *B, const float *sfa, const float *sfb,
                             void *C, int out, const int32_t *counts, int32_t E, int64_t N,
                             int64_t K, int64_t total_rows, int32_t *offsets_out,
                             int32_t *tile_map_out, cudaStream_t stream);

/*
 * Tile configuration fp8_grouped_gemm launches for (N, K, total_rows, E):
 * tile height BM, width BN, raster group height G, and an upper bound on the
 * tile count (the capacity tile_map_out needs, in 4-int32 entries).
 * Synchronous; uses the current device's SM count (148 when no device is
 * present).  Any output pointer may be null.
 */
FP8G_API fp8g_status fp8g_grouped_plan(int64_t N, int64_t K, int64_t total_rows, int32_t E, int32_t *BM,
                              int32_t *BN, int32_t *G, int64_t *max_tiles);

/*
 * Tile configuration fp8_gemm / fp8_gemm_blockscaled launch for a shape:
 * BM, BN, raster group G, K-split factor (1 = none) and grid size in CTAs.
 * block = 0 per-tensor, 1 block-scaled.  Host-only; needs the current device
 * to size the grid (FP8G_ERR_DEVICE if none).  Any output pointer may be null.
 */
FP8G_API fp8g_status fp8g_gemm_plan(int block, int64_t M, int64_t N, int64_t K, int32_t *BM, int32_t *BN,
                           int32_t *G, int32_t *split_k, int32_t *grid);

/*
 * Operand quantiser [JAX-BW microscaling paragraph and the fine-grained
 * quantisation advice; TRITON-FP8 dtype].
 * x: device fp32 [rows, cols] row-major; q: device uint8 [rows, cols].
 * block == 0: per-tensor.  s = fl32(amax/448) over the non-NaN |x| (s = 1 if
 *   that is 0); scales: device fp32[1] receives s.
 * block == 32: 1x32 blocks along cols (cols % 32 == 0).  Each block's s is the
 *   smallest power of two with 448*s >= amax (clamped to 2^-126..2^127; 1 for
 *   an all-zero block); scales: device fp32 [rows, cols/32].
 * q = E4M3(fl32(x / s)) rounded to nearest even, saturated to +-448; NaN -> 0x7F.
 * Alignment: x 16 B, q 8 B aligned; cols % 8 == 0 for block == 0.
 * Per-tensor mode runs three kernels (amax, quantise, store s).
 */
FP8G_API fp8g_status fp8g_quantize_e4m3(const float *x, int64_t rows, int64_t cols, int32_t block,
                               uint8_t *q, float *scales, cudaStream_t stream);

/*
 * fp8g_quantize_e4m3 with the output format `fmt` (fp8g_format): with
 * FP8G_E5M2 the bound 448 becomes 57344 throughout (s = fl32(amax/57344), or
 * the smallest power of two with 57344*s >= amax; saturation to +-57344;
 * infinities saturate too; NaN -> 0x7F).  With FP8G_E2M1 the bound is 6
 * (saturation to +-6, NaN -> code 7) and q holds two codes per byte: uint8
 * [rows, cols/2].  With FP8G_E2M3 / FP8G_E3M2 the bound is 7.5 / 28
 * (saturation, NaN -> code 0x1F) and q holds four codes per three bytes:
 * uint8 [rows, 3 cols/4].  A bad `fmt` is FP8G_ERR_INVALID_ARG.
 */
FP8G_API fp8g_status fp8g_quantize(const float *x, int64_t rows, int64_t cols, int32_t block,
                          int32_t fmt, uint8_t *q, float *scales, cudaStream_t stream);

/*
 * NVFP4 quantiser [TUT-12 12.6.1: NVFP4 among the fifth-generation tensor
 * core's micro-scaling formats; the pages print no recipe, the reading taken
 * is this]: E2M1 elements, one E4M3 scale per 1x16 block along cols, one fp32
 * scale g per tensor.
 *   g = fl32(amax / 2688) over the non-NaN |x| (2688 = 6 x 448), 1 if that is 0;
 *   per block: t = fl32(amax_b / fl32(6 g)), s = E4M3(t) rounded to nearest
 *   even, saturating; d = fl32(dec(s) g); q = E2M1(fl32(x / d)) rounded to
 *   nearest even, saturating, NaN -> +6; all codes 0 when d is 0.
 * x: device fp32 or bf16 (in_dtype) [rows, cols], 16-byte aligned, finite
 * apart from NaNs; q: uint8 [rows, cols/2], two codes per byte (element 2j in
 * the low nibble), 4-byte aligned; sf: uint8 E4M3 codes [rows, cols/16]; g:
 * device fp32[1], 4-byte aligned.  cols % 16 == 0 (else
 * FP8G_ERR_UNSUPPORTED_SHAPE).  Runs three kernels (amax, quantise, g).
 */
FP8G_API fp8g_status fp8g_quantize_nvfp4(const void *x, int32_t in_dtype, int64_t rows,
                                         int64_t cols, uint8_t *q, uint8_t *sf, float *g,
                                         cudaStream_t stream);

/*
 * NVFP4 GEMM [TUT-12 12.6.1]:
 *   C[i,j] = out( act( fl32( fl32(ga gb) * sum_kb sa[i,kb] sb[j,kb] sum_{k in kb} a_ik b_jk ) + bias[j] ) )
 * over 1x16 K blocks.  A [M, K/2], B [N, K/2]: E2M1 codes two per byte, as
 * fp8g_quantize_nvfp4 writes them, 32-byte aligned; sfa [M, K/16], sfb
 * [N, K/16]: E4M3 scale codes (positive; the tensor core applies them
 * exactly), 16-byte aligned; ga, gb: device fp32[1] each (the tensors' g);
 * bias (nullable) fp32 [N]; act an fp8g_act.  K % 256 == 0 (else
 * FP8G_ERR_UNSUPPORTED_SHAPE).  Runs two kernels: the scale packing and the
 * GEMM on CTA pairs with the FP4-rate kind::mxf4nvf4 MMA (scale_vec::4X),
 * for every shape.  Parity: the tolerance of the block-scaled GEMM.
 */
FP8G_API fp8g_status fp8_gemm_nvfp4(const void *A, const void *B, const uint8_t *sfa,
                                    const uint8_t *sfb, const float *ga, const float *gb, void *C,
                                    int out, const float *bias, int32_t act, int64_t M, int64_t N,
                                    int64_t K, cudaStream_t stream);

/*
 * Grouped (MoE) NVFP4 GEMM [TUT-12 12.6.1 for the arithmetic; JAX-BW MoE
 * paragraph for the grouping]: the rows of A [total_rows, K/2] are sorted by
 * expert, counts[e] of them for expert e (device int32[E], summing to
 * total_rows, else FP8G_ERR_INVALID_ARG through the status word), and expert
 * e's rows are multiplied by its own weight B[e] [N, K/2] (B: [E, N, K/2]):
 *   C[r,j] = out( act( fl32( fl32(ga gb[e]) * sum_kb sa[r,kb] sb[e,j,kb] sum_k a_rk b_ejk ) + bias[e,j] ) )
 * sfa [total_rows, K/16], sfb [E, N, K/16]: E4M3 scale codes, 16-byte
 * aligned; ga device fp32[1] (A's g), gb device fp32[E] (each expert's g);
 * bias (nullable) fp32 [E, N]; C [total_rows, N] in expert order.  A, B
 * 32-byte aligned; K % 256 == 0; 1 <= E <= FP8G_MAX_EXPERTS; total_rows may
 * be 0 (A and C then unused, may be null).  offsets_out (nullable, device
 * int32[E+1]) receives the exclusive prefix of counts; tile_map_out
 * (nullable, device int32[4 * ((total_rows / 256 + E) * ceil(N / 256))],
 * 16-byte aligned) one entry per 256 x 256 tile: expert, row tile within the
 * expert, column tile, 0.  Runs two kernels (scale packing, GEMM on CTA
 * pairs at the FP4 rate).  Parity: the tolerance of the block-scaled GEMM,
 * per expert.
 */
FP8G_API fp8g_status fp8_grouped_gemm_nvfp4(const void *A, const void *B, const uint8_t *sfa,
                                            const uint8_t *sfb, const float *ga, const float *gb,
                                            void *C, int out, const float *bias, int32_t act,
                                            const int32_t *counts, int32_t E, int64_t N, int64_t K,
                                            int64_t total_rows, int32_t *offsets_out,
                                            int32_t *tile_map_out, cudaStream_t stream);

/*
 * `block` value of the quantisers for 1x32 blocks with the literal scale
 * s = fl32(amax / fmax) (1 when that is 0) — the "fp32 scale = block
 * amax/448" wording taken literally — and q = FP8(fl32(x / s)).  Such scales
 * are generally not powers of two: use them with
 * fp8_gemm_blockscaled_promote.
 */
#define FP8G_BLOCK32_LITERAL 33

/* Source element types of fp8g_quantize_rows. */
typedef enum { FP8G_IN_F32 = 0, FP8G_IN_BF16 = 1 } fp8g_in_dtype;

/*
 * Activation quantiser with a row gather [JAX-BW MoE paragraph: tokens routed
 * to experts; its fine-grained quantisation advice]: output row r (of n_rows)
 * is row rows[r] of x [x_rows, cols] quantised as fp8g_quantize does (rows
 * null: row r, n_rows <= x_rows).  x is fp32 or bf16 (in_dtype; bf16 is
 * widened exactly), 16-byte aligned; rows: device int32 [n_rows], 4-byte
 * aligned; q: uint8 [n_rows, cols] (E2M1: [n_rows, cols/2]); scales:
 * [n_rows, cols/32] (block 32) or
 * [1].  Gather, scale and quantisation are one pass over HBM (per-tensor:
 * two).  cols % 8 == 0 (block 32: cols % 32 == 0).  A row index outside
 * [0, x_rows) records FP8G_ERR_INVALID_ARG in the status word (detail: r) and
 * quantises zeros for that row.
 */
FP8G_API fp8g_status fp8g_quantize_rows(const void *x, int32_t in_dtype, int64_t x_rows,
                               int64_t cols, const int32_t *rows, int64_t n_rows, int32_t block,
                               int32_t fmt, uint8_t *q, float *scales, cudaStream_t stream);

/*
 * The GEMM entry points with explicit operand formats (fp8g_format each for
 * A and B, mixed allowed: the tensor core's kind::f8f6f4 and
 * kind::mxf8f6f4 MMAs take any of the three per operand; an E2M1 operand
 * is packed, two codes per byte, with the rules of fp8g_format).  Everything else as
 * fp8_gemm / fp8_gemm_blockscaled / fp8_grouped_gemm; a bad format is
 * FP8G_ERR_INVALID_ARG.  Parity: the same tolerance as for E4M3.
 */
FP8G_API fp8g_status fp8_gemm_fmt(const void *A, const void *B, const float *scale_a,
                         const float *scale_b, void *C, int out, int32_t a_fmt, int32_t b_fmt,
                         int64_t M, int64_t N, int64_t K, cudaStream_t stream);
FP8G_API fp8g_status fp8_gemm_blockscaled_fmt(const void *A, const void *B, const float *sfa,
                                     const float *sfb, void *C, int out, int32_t a_fmt,
                                     int32_t b_fmt, int64_t M, int64_t N, int64_t K,
                                     cudaStream_t stream);
FP8G_API fp8g_status fp8_grouped_gemm_fmt(const void *A, const void *B, const float *sfa,
                                 const float *sfb, void *C, int out, int32_t a_fmt, int32_t b_fmt,
                                 const int32_t *counts, int32_t E, int64_t N, int64_t K,
                                 int64_t total_rows, int32_t *offsets_out, int32_t *tile_map_out,
                                 cudaStream_t stream);

/*
 * The GEMM entry points with operand formats and a fused epilogue: `bias`
 * (nullable) is a device fp32 [N] (grouped: [E, N], expert e's row for its
 * rows of C), 4-byte aligned; `act` is an fp8g_act.  out = out(act(fl32(v +
 * bias[j]))) with v the value the plain entry point would round.  Parity:
 * |C - ref| <= L (2^-8 sum_k |sA a||sB b|) + 2^-20 (|v| + |bias|) + 1 bf16
 * ulp(|ref|), L = 1 (none, ReLU) or 1.13 (GELU, the bound of |GELU'|); the
 * 2^-20 term covers the fp32 bias add and activation.  Bad `act` or
 * formats: FP8G_ERR_INVALID_ARG.
 */
FP8G_API fp8g_status fp8_gemm_ex(const void *A, const void *B, const float *scale_a,
                        const float *scale_b, void *C, int out, int32_t a_fmt, int32_t b_fmt,
                        const float *bias, int32_t act, int64_t M, int64_t N, int64_t K,
                        cudaStream_t stream);
FP8G_API fp8g_status fp8_gemm_blockscaled_ex(const void *A, const void *B, const float *sfa,
                                    const float *sfb, void *C, int out, int32_t a_fmt,
                                    int32_t b_fmt, const float *bias, int32_t act, int64_t M,
                                    int64_t N, int64_t K, cudaStream_t stream);
/*
 * 1x32 block-scaled GEMM for arbitrary fp32 scales [JAX-BW warp
 * specialisation paragraph: the promotion warp role; the workloads' literal
 * "fp32 scale = block amax/448"].  Same C = sum_kb sfa*sfb*partial_kb as
 * fp8_gemm_blockscaled, but any finite fp32 scale (NaN and infinities
 * propagate) rather than only powers of two.  Two routes, chosen by shape:
 *   - at least a wave of 256 x 256 output tiles (fp8g_gemm_plan(0, M, N, K)
 *     BM = 256) with 1-byte operands (E4M3 / E5M2): each operand is
 *     dequantised once with its scales to TF32 (round to nearest, ties
 *     away; every value within 2^-11 of fl32(dec(q) s)) into a stream-ordered
 *     temporary of 4 (M + N) K bytes from the library's pool, then a
 *     kind::tf32 tensor-core GEMM on CTA pairs: three kernels.  Each scaled
 *     operand value must be finite in fp32.
 *   - otherwise: the tensor core computes each 32-wide K block's unscaled
 *     partial and CUDA-core warps scale and accumulate it in fp32
 *     (fma(fl32(sfa*sfb), partial, acc)): one kernel, no allocation.
 * Both lie within the block-scaled GEMM's tolerance.  Operand formats, bias
 * and activation as fp8_gemm_blockscaled_ex.  K % 128 == 0 (else
 * FP8G_ERR_UNSUPPORTED_SHAPE); sfa, sfb 16-byte aligned.
 */
FP8G_API fp8g_status fp8_gemm_blockscaled_promote(const void *A, const void *B, const float *sfa,
                                         const float *sfb, void *C, int out, int32_t a_fmt,
                                         int32_t b_fmt, const float *bias, int32_t act, int64_t M,
                                         int64_t N, int64_t K, cudaStream_t stream);

FP8G_API fp8g_status fp8_grouped_gemm_ex(const void *A, const void *B, const float *sfa,
                                const float *sfb, void *C, int out, int32_t a_fmt, int32_t b_fmt,
                                const float *bias, int32_t act, const int32_t *counts, int32_t E,
                                int64_t N, int64_t K, int64_t total_rows, int32_t *offsets_out,
                                int32_t *tile_map_out, cudaStream_t stream);

/*
 * fp8_grouped_gemm_ex whose output rows are scattered [JAX-BW MoE paragraph:
 * expert outputs return to token order]: routed row r (expert order) is
 * stored to row c_row_of[r] of C [c_rows, N] (device int32 [total_rows],
 * 4-byte aligned; null: row r, c_rows = total_rows).  Rows of C that no
 * routed row names are not written; two routed rows naming one row of C
 * race (the caller's responsibility).  An index outside [0, c_rows) records
 * FP8G_ERR_INVALID_ARG (detail: r) and that row is not stored.
 */
FP8G_API fp8g_status fp8_grouped_gemm_scatter(const void *A, const void *B, const float *sfa,
                                     const float *sfb, void *C, int out, int32_t a_fmt,
                                     int32_t b_fmt, const float *bias, int32_t act,
                                     const int32_t *counts, int32_t E, int64_t N, int64_t K,
                                     int64_t total_rows, const int32_t *c_row_of, int64_t c_rows,
                                     int32_t *offsets_out, int32_t *tile_map_out,
                                     cudaStream_t stream);

/* `flags` of fp8_grouped_gemm_quant. */
#define FP8G_QUANT_FUSED 1

/*
 * Grouped (MoE) GEMM from unquantised activations [JAX-BW MoE paragraph:
 * tokens routed to experts; its fine-grained (1x32) quantisation advice
 * against FP8 underflow].  The result equals
 *   fp8g_quantize_rows(X, x_dtype, x_rows, K, rows, total_rows, 32, FP8G_E4M3,
 *                      qa, sfa)
 *   fp8_grouped_gemm_scatter(qa, B, sfa, sfb, C, out, FP8G_E4M3, b_fmt, bias,
 *                            act, counts, E, N, K, total_rows, c_row_of,
 *                            c_rows, offsets_out, tile_map_out)
 * bit for bit: routed row r (expert order) is source row rows[r] of X
 * [x_rows, K] (rows null: row r, total_rows <= x_rows), quantised to E4M3
 * with one power-of-two scale per 1x32 block, then multiplied by its
 * expert's B[e].  flags 0: the two steps run as two kernels (plus the
 * packing of the scales), the codes in qa_out / sfa_out or, when those are
 * null, in a stream-ordered temporary from the library's pool.
 * flags FP8G_QUANT_FUSED, when the grouped plan runs one CTA per 128-row
 * tile (fp8g_grouped_plan BM = 128: few routed rows, e.g. decoding): the
 * quantisation runs inside the GEMM kernel, each CTA quantising the tile of A
 * it multiplies from X into shared memory, so the codes never go through
 * memory (other plans: as flags 0).  On GB300 the two kernels are faster:
 * every CTA of a row tile re-reads that tile's bf16 rows, 56 times for
 * N = 14336, and those loads wait behind the weights streaming through the
 * memory system (decode-shaped MoE: 176 against 72 us per call).
 * X: fp32 or bf16 (x_dtype, FP8G_IN_*), 16-byte aligned; rows: device int32
 * [total_rows], 4-byte aligned; qa_out (nullable) uint8 [total_rows, K] and
 * sfa_out (nullable) fp32 [total_rows, K/32], both or neither, 16-byte
 * aligned: they receive the codes and scales (when the counts are valid).
 * K % 32 == 0; flags 0 or FP8G_QUANT_FUSED.  Other arguments and rules as
 * fp8_grouped_gemm_scatter.  A source row outside [0, x_rows) records
 * FP8G_ERR_INVALID_ARG (detail: the routed row) and that row quantises as
 * zeros.  Parity: the quantiser's codes and scales bit-exact, the GEMM
 * within the block-scaled tolerance.
 */
FP8G_API fp8g_status fp8_grouped_gemm_quant(const void *X, int32_t x_dtype, int64_t x_rows,
                                           const int32_t *rows, const void *B, const float *sfb,
                                           void *C, int out, int32_t b_fmt, const float *bias,
                                           int32_t act, const int32_t *counts, int32_t E,
                                           int64_t N, int64_t K, int64_t total_rows,
                                           const int32_t *c_row_of, int64_t c_rows,
                                           uint8_t *qa_out, float *sfa_out, int32_t *offsets_out,
                                           int32_t *tile_map_out, int32_t flags,
                                           cudaStream_t stream);

/*
 * Synchronises `stream`, then returns and clears the current device's status
 * word (FP8G_OK if no kernel recorded an error since the last call).
 * `detail` (nullable) receives a kernel-specific code for the first error
 * (for a timeout: role * 256 + pipeline stage).
 */
FP8G_API fp8g_status fp8_gemm_status(cudaStream_t stream, int32_t *detail);

/*
 * Kernel timing (the source pages have no counterpart; for benchmarks).
 * fp8g_kernel_timing_begin(n) creates n pairs of CUDA events on the current
 * device; each following GEMM call (any GEMM entry point, any stream or host
 * thread) records pair i on its stream immediately before launching its GEMM
 * kernel and immediately after, for its first n calls (i = 0, 1, ...).
 * fp8g_kernel_timing_end(ms, cap, count) waits for the recorded calls,
 * writes their GEMM-kernel durations in milliseconds (without the scale
 * packing that block calls launch first) to ms[0 .. *count), frees the events
 * and turns the recording off.  Recording costs each call two stream
 * operations and keeps the GEMM's prologue from overlapping the packing
 * kernel, so measure throughput with the recording off.
 * Errors: FP8G_ERR_INVALID_ARG (n outside 1 .. 2^20, begin while on, end
 * while off), FP8G_ERR_CUDA.
 */
FP8G_API fp8g_status fp8g_kernel_timing_begin(int32_t n);
FP8G_API fp8g_status fp8g_kernel_timing_end(float *ms, int32_t cap, int32_t *count);

/*
 * Diagnostic (the source pages have no counterpart): launches a one-warp
 * kernel that makes one mbarrier wait complete and then waits, with the same
 * bounded-wait code as the GEMM kernels, on a barrier that nothing arrives at.
 * After timeout_us microseconds (1 .. 10^7) that wait gives up and records
 * FP8G_ERR_TIMEOUT with detail 0xDEAD in the status word, and the kernel
 * returns.  Read it with fp8_gemm_status.  Shows on a live GPU that a wait
 * which cannot complete ends in a host-visible error, not a hang.
 */
FP8G_API fp8g_status fp8g_wait_selftest(uint32_t timeout_us, cudaStream_t stream);

/* Static English description of a status code. */
FP8G_API const char *fp8g_status_string(fp8g_status status);

/*
 * Device-side wait limit in milliseconds for kernels launched after this call
 * (default 2000, or the FP8G_WAIT_TIMEOUT_MS environment variable at load).
 * 0 restores the default.
 */
FP8G_API void fp8g_set_wait_timeout_ms(uint32_t ms);

/* Drops the host tensor-map cache and releases the memory the scale-packing
 * pool holds (pending stream-ordered frees are honoured).  Safe to call at
 * any time. */
FP8G_API void fp8g_shutdown(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
FP8G_API int fp8g_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8GEMM_H */
