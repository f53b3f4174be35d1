// Internal declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "fp8gemm.h"

namespace fp8g {

// Tile geometry of the GEMM kernels.  BM = 128 rows (the single-CTA tcgen05
// M), BK = 128 E4M3 values = 128 bytes per row, which is exactly one 128-byte
// swizzle span ("TMA block 128x128, 128-byte aligned" in the parameter
// paragraph of the JAX/Blackwell FP8 GEMM page).
constexpr int kBM = 128;
constexpr int kBK = 128;
constexpr int kRasterG = 16;  // grouped raster band height (GROUP_M)

enum Mode : int { kModeTensor = 0, kModeBlock = 1, kModeGrouped = 2 };

// Everything a GEMM kernel needs besides its tensor maps.
struct GemmParams {
    int64_t M;           // rows of A and C (grouped: total rows)
    int64_t N;           // rows of B, columns of C
    int64_t K;
    int32_t num_kb;      // ceil(K / kBK)
    int32_t npm, npn;    // tile grid (non-grouped)
    int64_t T;           // tile count (non-grouped)
    int32_t split;       // K-split factor (cluster size along K), 1 = none
    int32_t kb_per_split;
    const float *sa;     // per-tensor: &sA ; block: sfa [M, sfc]
    const float *sb;     // per-tensor: &sB ; block: sfb [N, sfc] (grouped [E, N, sfc])
    int64_t sfc;         // K / 32
    void *C;
    const int32_t *counts;
    int32_t E;
    int32_t *offsets_out;
    int32_t *tile_map_out;
    unsigned int *status;  // [0] = first error code, [1] = detail
    uint64_t timeout_ns;
    const uint8_t *sfa_pk; // block modes: packed UE8M0 scale chunks of A and B
    const uint8_t *sfb_pk;
    int32_t n_rtA, n_rtB;  // 128-row tiles per K group in the packed arrays
    uint32_t ab_fmt;       // operand formats as MMA instruction-descriptor bits (A: 7-9, B: 10-12)
    // Packed operands (E2M1 two codes per byte, FP6 four codes per three
    // bytes): their tile loads deliver the packed byte count, not the tile's
    // shared-memory footprint (16 codes widened to 16 bytes), so each stage
    // expects that many fewer transaction bytes: gap8 eighths of the operand's
    // tile (E2M1 4, FP6 2, FP8 0).
    int32_t a_gap8, b_gap8;
    // E2M1 x E2M1 block-scaled on CTA pairs at the FP4 rate (kind::mxf4):
    // operands loaded as dense bytes, 256 K elements per stage, num_kb = K /
    // 256, the packed scale arrays holding 2 * num_kb chunks per row tile.
    int32_t f4;               // 1: MXFP4 (kind::mxf4); 2: NVFP4 (kind::mxf4nvf4, 1x16 E4M3
                              // scales); 3: TF32 operands (kind::tf32, per-tensor mode, alpha 1)
    const float *ga, *gb;     // NVFP4: the tensors' fp32 scales (epilogue alpha = fl32(ga gb))
    int32_t st32;             // epilogue: 32-byte stores (C 32-byte aligned, rows multiples of 32 B)
    const float *bias;     // fused epilogue: fp32 [N] (grouped [E, N]) or null
    int32_t act;           // fused epilogue activation: FP8G_ACT_*
    const int32_t *c_row_of;  // grouped scatter: row of C for routed row r (null: r)
    int64_t c_rows;           // rows of C when scattering
    // Fused activation quantiser (grouped GEMM on single CTAs): A is not read
    // from memory; each stage's 128 x 128 tile of A is quantised in the kernel
    // (E4M3, 1x32 power-of-two scales) from routed row r = source row
    // xq_rows[r] (null: r) of xq [xq_src_rows, K] (fp32, or bf16 if xq_bf16).
    // qa_out [rows, K] / sfa_out [rows, K/32] (nullable) receive the codes and
    // scales, written by the CTAs of the first column of tiles.
    const void *xq;
    int32_t xq_bf16;
    const int32_t *xq_rows;
    int64_t xq_src_rows;
    uint8_t *qa_out;
    float *sfa_out;
};

// TMA descriptors of one launch: E4M3 operands and, for block-scaled CTA
// pairs, the packed scale arrays viewed as rows of 512 bytes (unused ones
// repeat A's).
struct GemmMaps {
    CUtensorMap A, B, SA, SB;
};

struct KernelChoice {
    int BM;      // output tile rows (256 for a CTA pair)
    int BN;      // output tile columns
    int b_rows;  // rows of B per TMA box (a CTA pair loads half of BN each)
    int split;   // K-split cluster size (1 = none)
    int grid;    // CTAs launched
    int cluster; // CTAs per cluster
    bool pair;   // tcgen05 cta_group::2 kernel (gemm_pair.cu)
    bool inl;    // block-scaled single CTAs converting their own scales (no packing kernel)
};

// gemm.cu
cudaError_t launch_gemm(int mode, bool out_f32, const GemmMaps &maps, const GemmParams &p,
                        const KernelChoice &kc, cudaStream_t stream);
KernelChoice choose_kernel(int mode, int64_t M, int64_t N, int64_t K, int num_sms);

// selftest.cu: one warp, one wait that runs out after timeout_ns
cudaError_t launch_wait_selftest(unsigned int *status, uint64_t timeout_ns, cudaStream_t s);

// gemm_promote.cu: arbitrary fp32 1x32 scales (maps.SA / maps.SB: the fp32
// scale arrays, box 4 x 128); grid CTAs over 128 x 128 tiles.
cudaError_t launch_gemm_promote(bool out_f32, const GemmMaps &maps, const GemmParams &p, int grid,
                                cudaStream_t stream);

// gemm_pair.cu (per-tensor and block-scaled, CTA pairs)
cudaError_t launch_gemm_pair(int mode, bool out_f32, const GemmMaps &maps, const GemmParams &p,
                             int grid, cudaStream_t stream);


// api.cu: checks done by the caller; scratch == nullptr takes the packed
// scale temporary from the library pool, otherwise uses [scratch,
// scratch + scratch_bytes) (FP8G_ERR_UNSUPPORTED_SHAPE if it is too small).
// a_fmt, b_fmt: operand formats (FP8G_E4M3 / FP8G_E5M2).
// fq (grouped mode only, single-CTA plan): the fused activation quantiser's
// source (GemmParams::xq ..); A and sa are then not read.
struct FusedQuant {
    const void *x;
    int32_t bf16;
    const int32_t *rows;
    int64_t src_rows;
    uint8_t *qa_out;
    float *sfa_out;
};
fp8g_status run_gemm(int mode, const void *A, const void *B, const float *sa, const float *sb,
                     void *C, int out, int64_t M, int64_t N, int64_t K, const int32_t *counts,
                     int32_t E, int32_t *offsets_out, int32_t *tile_map_out, cudaStream_t stream,
                     void *scratch, size_t scratch_bytes, int a_fmt = 0, int b_fmt = 0,
                     const float *bias = nullptr, int act = 0, const int32_t *c_row_of = nullptr,
                     int64_t c_rows = 0, const FusedQuant *fq = nullptr);

// api.cu: the host-side argument checks of the 1x32 block-scaled GEMM, in the
// order fp8_gemm_blockscaled applies them (shared by its allocation-free
// form, so both return the same status for the same bad arguments); and the
// current device's usability (an sm_103 device, status word and tensor-map
// encoder set up), FP8G_OK or the status a GEMM call would return.
fp8g_status check_blockscaled_args(const void *A, const void *B, const float *sfa,
                                  const float *sfb, const void *C, int out, int64_t M, int64_t N,
                                  int64_t K);
fp8g_status device_ready();

// scales.cu: fp32 1x32 scales -> packed UE8M0 chunks.  One launch packs
// two operands (nz = 0 skips one): src [nz][z_rows][sfc] (rows_total valid
// rows per z), dst chunks ((z * n_kg + kg) * n_rt + rt) * 512; counts != null
// numbers A's row tiles per expert.
// Launch with programmatic stream serialization: the kernel may begin while
// the previous one on the stream finishes; it calls grid_dep_wait before any
// global memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_programmatic(void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t s,
                                Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

struct PackArgs {
    const float *src;
    int64_t rows_total, z_rows;
    int32_t n_rt, nz;
    uint8_t *dst;
    const int32_t *counts;
    int32_t rep;  // B of single-CTA 256-wide tiles: 4 KB per (z, kg, 256-row tile), replicated for tcgen05.cp 128x256b
    const int32_t *zskip = nullptr;  // grouped B: matrices z with zskip[z] <= 0 (experts without rows) are skipped
};
// NVFP4: E4M3 scale codes [rows, K/16] -> the same 512-byte chunks, a K group
// being 64 wide (4 blocks of 16, one MMA's word), the four groups of a
// 256-wide stage adjacent per 128-row tile; rows past the operand 1.0.  A
// with expert-local row tiles when counts is set (E experts); B as z_b
// matrices of rows_b rows.
cudaError_t launch_pack_nvfp4(const uint8_t *sfa, int64_t rows_a, int32_t n_rt_a, uint8_t *dst_a,
                              const int32_t *counts, const uint8_t *sfb, int64_t rows_b,
                              int32_t n_rt_b, int32_t z_b, uint8_t *dst_b, int32_t n_kg,
                              int64_t sfc, int32_t E, cudaStream_t s);
size_t packed_scale_bytes(int32_t n_kg, int32_t n_rt, int32_t z);
cudaError_t launch_pack_scales(const PackArgs &a, const PackArgs &b, int64_t sfc, int32_t n_kg,
                               int32_t E, unsigned int *status, cudaStream_t s);

// quant.cu: A [rows, K] FP8 codes (fmt FP8G_E4M3 / FP8G_E5M2) with fp32 1x32
// scales s [rows, K/32] -> out [rows, K] fp32 = TF32(fl32(dec(a) s)) (round to
// nearest, ties away: exact TF32 values).
cudaError_t launch_dequant_tf32(const uint8_t *a, const float *s, int64_t rows, int64_t K, int fmt,
                                float *out, int num_sms, cudaStream_t stream);
// quant.cu: output row r quantises source row rows[r] (rows null: row r) of
// x [x_rows, cols] (fp32, or bf16 if in_bf16); block 0 per-tensor or 32; fmt
// FP8G_E4M3 / FP8G_E5M2.  Bad row indices record FP8G_ERR_INVALID_ARG.
// block FP8G_BLOCK32_LITERAL: 1x32 blocks with s = fl32(amax / fmax).
cudaError_t launch_quantize_nvfp4(const void *x, int in_bf16, int64_t rows, int64_t cols,
                                  uint8_t *q, uint8_t *sf, float *g, unsigned int *status,
                                  int num_sms, cudaStream_t s);
cudaError_t launch_quantize_rows(const void *x, int in_bf16, int64_t x_rows, int64_t cols,
                                 const int32_t *rows, int64_t n_rows, int32_t block, int fmt,
                                 uint8_t *q, float *scales, unsigned int *status, int num_sms,
                                 cudaStream_t s);

}  // namespace fp8g
