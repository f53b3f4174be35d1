// Persistent, warp-specialised FP8 (E4M3) GEMM for sm_103a.
//
//   C = (sA A)(sB B)^T,  A[M,K], B[N,K] row-major, fp32 accumulation in tensor
//   memory, bf16 or fp32 output.  Three modes: per-tensor scales, 1x32 block
//   scales along K (applied by the block-scaled tensor-core MMA), and the
//   grouped (MoE) form of the block-scaled GEMM.  Operands E4M3 or any other
//   kind::f8f6f4 element (E5M2, E2M3, E3M2, E2M1; the packed ones load
//   through the 4- and 6-bit tile types), one format per operand.
//
// Design (GB300-native; the pages' Triton/Pallas kernels are prior art only):
//   - one CTA per SM, persistent over output tiles in the grouped raster order
//     (persistent matmul and GROUP_M swizzle: Triton tutorial ch. 12, 12.7);
//   - warp 0: TMA producer filling a STAGES-deep shared-memory ring, one
//     mbarrier pair (full / empty) per stage with expect_tx byte accounting
//     (12.2.1 and 12.3.1 of the tutorial; "one warp loads with TMA" in the
//     warp-specialisation paragraph of the JAX/Blackwell FP8 GEMM page);
//   - warp 1: a single thread issues tcgen05.mma (kind::f8f6f4, or
//     kind::mxf8f6f4.block_scale with UE8M0 scale factors read from tensor
//     memory) into an fp32 accumulator in tensor memory (12.6.1-12.6.2);
//   - block modes: the producer also bulk-copies each stage's scale factors,
//     pre-packed as UE8M0 bytes in the layout tcgen05.cp reads (scales.cu),
//     into the stage (split-K: epilogue warps convert them in place); warp 2
//     copies them shared -> tensor memory and commits them to the stage's
//     "scales ready" barrier, which the MMA thread waits on;
//   - warps 4..19: epilogue; each warp drains its 32-lane quarter of the
//     accumulator (tcgen05.ld), releases it, scales / rounds and stores.
//
// Tensor-memory budget (Triton tutorial ch. 12, 12.8 Q3): a 128 x 256 fp32
// accumulator is 256 columns.  Per-tensor mode double-buffers it (512 columns);
// block mode keeps one accumulator plus one scale-factor slot per stage and
// overlaps the epilogue by releasing the accumulator as soon as it has been
// copied into registers.
//
// Every wait is bounded (globaltimer); on expiry the CTA records
// FP8G_ERR_TIMEOUT in the status word, all roles leave their loops, in-flight
// copies and MMAs are drained with bounded waits, and tensor memory is freed.
#include <cuda_bf16.h>

#include <atomic>

#include "internal.h"
#include "ptx.cuh"
#include "kernel_common.cuh"
#include "quant_math.cuh"

namespace fp8g {

namespace {

constexpr int kThreads = 640;  // 20 warps
constexpr int kMaxSplit = 4;   // K-split cluster size (clusters of <= 4 CTAs co-schedule)
// Few-tile shapes with fewer K steps than this run one CTA per 128 x 128 tile
// instead of splitting K (the split-K exchange costs more than it saves);
// block-scaled ones convert their scales in the kernel as split-K does
constexpr int kMinSplitKb = 16;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 16;
// Block-scaled split-K: the epilogue warps convert the fp32 block scales (128
// rows of A, 128 of B) of every K step into the stage's UE8M0 chunk, kSfWarps
// warps per operand.
constexpr int kSfWarps = 8;

// Split-K (SPLITC): the ring of a split-K CTA, then its receive region for
// the peers' partial blocks: (S - 1) x 128 rows x (128 / S) columns of fp32,
// at most 48 KB (S <= 4).
constexpr int kSplitStages = 5;
constexpr int kRecvBytes = 48 * 1024;

template <int MODE, int BN, int NUM_ACC, int STAGES, bool SPLITC = false>
struct Cfg {
    static constexpr bool kBlock = MODE != kModeTensor;
    static constexpr int A_BYTES = kBM * kBK;
    static constexpr int B_BYTES = BN * kBK;
    // Packed UE8M0 scales per stage (4 K blocks per row): A's 128 rows (512 B,
    // one replicating 32x128b copy); B's rows: 128 -> 512 B the same way,
    // 256 -> 4 KB already replicated over the four lane quarters (one
    // 128x256b copy, issued by the scale-copy warp).
    static constexpr bool kRepB = kBlock && BN == 256;
    static constexpr int SFB_BYTES = kBlock ? (kRepB ? 4096 : BN * 4) : 0;
    static constexpr int CHUNK_BYTES = kBlock ? kBM * 4 + SFB_BYTES : 0;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SF = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_RECV = OFF_SF + STAGES * CHUNK_BYTES;
    static constexpr int OFF_BAR = OFF_RECV + (SPLITC ? kRecvBytes : 0);
    // full[S], empty[S], acc_full[NA], acc_empty[NA], drain, split-K receive,
    // drain of the scale-copy thread, scales ready[S]
    static constexpr int NUM_BARS = 3 * STAGES + 2 * NUM_ACC + 3;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_GROUP = OFF_MISC + 16;
    static constexpr int GROUP_BYTES = 3 * (FP8G_MAX_EXPERTS + 1) * 4;
    static constexpr int SMEM_USED = OFF_GROUP + GROUP_BYTES;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment
    static constexpr uint32_t TX_BYTES = A_BYTES + B_BYTES + CHUNK_BYTES;
    static constexpr int ACC_COLS = NUM_ACC * BN;
    static constexpr int SF_COLS = kBlock ? (kRepB ? 16 : kBM / 32 + BN / 32) : 0;
    static constexpr int SFB_COL = kRepB ? 8 : kBM / 32;  // B's scale columns in a slot
    static constexpr int SF_COL0 = ACC_COLS;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int CW = BN / 4;  // accumulator columns per epilogue warp

    static_assert(ACC_COLS + STAGES * SF_COLS <= 512, "tensor memory over budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory over the per-CTA limit");
    static_assert(BN % 128 == 0 && BN <= 256, "BN must be 128 or 256");
    static_assert(CW % 32 == 0, "epilogue chunk must be a multiple of 32 columns");
    static_assert(OFF_SF % 16 == 0 && CHUNK_BYTES % 16 == 0, "bulk-copy alignment");
};

struct Tile {
    int32_t row0, row_end, n0, e, pm, pn;
    int32_t rtA;  // 128-row tile of A in the packed scale layout
};

template <int MODE, int BN>
__device__ __forceinline__ Tile get_tile(int32_t t, const GemmParams &p, const int32_t *row_off,
                                         const int32_t *tile_off, const int32_t *rt_off) {
    Tile ti;
    if constexpr (MODE == kModeGrouped) {
        int e = 0;
        while (tile_off[e + 1] <= t) ++e;
        const int32_t Me = row_off[e + 1] - row_off[e];
        const int32_t npm_e = (Me + kBM - 1) / kBM;
        raster(t - tile_off[e], npm_e, p.npn, kRasterG, ti.pm, ti.pn);
        ti.row0 = row_off[e] + ti.pm * kBM;
        ti.row_end = row_off[e + 1];
        ti.e = e;
        ti.rtA = rt_off[e] + ti.pm;
    } else {
        raster(t, p.npm, p.npn, kRasterG, ti.pm, ti.pn);
        ti.row0 = ti.pm * kBM;
        ti.row_end = (int32_t)p.M;
        ti.e = 0;
        ti.rtA = ti.pm;
    }
    ti.n0 = ti.pn * BN;
    return ti;
}

// Block-scaled kernels that convert their own scales (split-K, single CTAs on
// few tiles, grouped single CTAs), epilogue warp ew (of 2 kSfWarps): writes
// the UE8M0 chunk (the layout of scales.cu: byte 16 d + 4 w + j = row 32 w +
// d, K block j; A's 128 rows, then B's) of each of the tile's K steps into the ring, after
// the stage's empty barrier, and counts one arrival per warp and stage on its
// full barrier.  Warps 0..7 take A's rows, 8..15 B's, 16 rows each.  K steps
// go in windows of 8: lane (i, s) = (lane / 8, lane % 8) reads the 16 bytes of
// step s for rows 4 j + i (j < 4) of the warp's 16, so eight lanes read one
// row's 128 contiguous bytes and every load of a window is in flight at once.
// (One row per lane and a step per load, each warp load touched 32 lines.)
// sf_fetch issues a window's loads, sf_put converts and stores them.  Rows
// past the operand and K blocks past K/32 get code 127; a scale that is not a
// positive normal power of two sets `bad`.
struct SfWindow {
    uint32_t v[4][4];  // this lane's step: 4 fp32 scales of each of its 4 rows
};

__device__ __forceinline__ void sf_fetch(const GemmParams &p, const Tile &ti, int kb_begin, int n,
                                         int w0, int ew, SfWindow &f) {
    const int lane = threadIdx.x & 31;
    const bool isB = ew >= kSfWarps;
    const int sl = lane & 7;
    const int r0 = (ew % kSfWarps) * 16 + (lane >> 3);
    const int64_t g0 = (isB ? (int64_t)ti.n0 : (int64_t)ti.row0) + r0;  // row of j = 0
    const int64_t left = (isB ? p.N : (int64_t)ti.row_end) - g0;     // rows from it on
    const bool live = w0 + sl < n;
    const int64_t k0 = (int64_t)(kb_begin + w0 + sl) * 4;  // this lane's first scale column
    // grouped: B's scales are E matrices of N rows (ti.e = 0 otherwise)
    const int64_t gz = isB ? (int64_t)ti.e * p.N + g0 : g0;
    const float *row = (isB ? p.sb : p.sa) + (live && left > 0 ? gz * p.sfc + k0 : 0);
    const int64_t step = 4 * p.sfc;  // four rows on
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const bool valid = live && 4 * j < left;
        const float *src = row + (valid ? j * step : 0);
        if ((p.sfc & 3) == 0) {
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (valid) x = __ldg(reinterpret_cast<const uint4 *>(src));
            f.v[j][0] = x.x;
            f.v[j][1] = x.y;
            f.v[j][2] = x.z;
            f.v[j][3] = x.w;
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                f.v[j][q] = (valid && k0 + q < p.sfc) ? __float_as_uint(__ldg(src + q)) : 0u;
        }
    }
}

// UE8M0 codes of four fp32 scales in one word (byte q: scale q): their
// exponent fields, which is ue8m0_code's result for every input (a NaN's
// exponent field is 0xFF).  ue8m0_code's checks run only when some scale is
// not a positive normal power of two (a set sign or mantissa bit, an
// exponent field 0 or 0xFF).
__device__ __forceinline__ uint32_t ue8m0_word(const uint32_t (&x)[4], bool &bad) {
    const uint32_t w = __byte_perm(__byte_perm(x[0] << 1, x[1] << 1, 0x0073u),
                                   __byte_perm(x[2] << 1, x[3] << 1, 0x0073u), 0x5410u);
    if ((((x[0] | x[1] | x[2] | x[3]) & 0x807FFFFFu) | __vcmpeq4(w, 0u) | __vcmpeq4(w, ~0u)) != 0u) {
#pragma unroll
        for (int q = 0; q < 4; ++q) (void)ue8m0_code(x[q], bad);
    }
    return w;
}

// Returns false when the CTA is aborting.  With fresh = true (the first window
// of a CTA's first tile: its first STAGES stages were never used) those
// stages are filled without waiting and published with one proxy fence.
template <int STAGES>
__device__ __forceinline__ bool sf_put(const GemmParams &p, const Tile &ti, int kb_begin, int n,
                                       int w0, uint32_t it, int ew, const SfWindow &f,
                                       uint32_t sf_base, uint32_t chunk_bytes, uint64_t *bars,
                                       volatile int *abort_flag, bool &bad, bool fresh) {
    const int lane = threadIdx.x & 31;
    const bool isB = ew >= kSfWarps;
    const int sl = lane & 7;
    const int r0 = (ew % kSfWarps) * 16 + (lane >> 3);
    const int64_t left = (isB ? p.N : (int64_t)ti.row_end) -
                         ((isB ? (int64_t)ti.n0 : (int64_t)ti.row0) + r0);
    const uint32_t half = isB ? kBM * 4u : 0u;
    const bool live = w0 + sl < n;
    const int64_t k0 = (int64_t)(kb_begin + w0 + sl) * 4;
    const bool whole = k0 + 4 <= p.sfc;  // no K block of this step past K / 32
    uint32_t word[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        word[j] = 0x7F7F7F7Fu;
        if (live && 4 * j < left) {
            if (whole) {
                word[j] = ue8m0_word(f.v[j], bad);
            } else {
                word[j] = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    word[j] |= (k0 + q < p.sfc ? ue8m0_code(f.v[j][q], bad) : 127u) << (8 * q);
            }
        }
    }
    auto put = [&](uint32_t stage) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t r = (uint32_t)(r0 + 4 * j);
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(sf_base + stage * chunk_bytes + half +
                                                         16u * (r & 31u) + 4u * (r >> 5)),
                         "r"(word[j])
                         : "memory");
        }
    };
    const int steps = n - w0 < 8 ? n - w0 : 8;
    int t0 = 0;
    if (fresh) {
        t0 = steps < STAGES ? steps : STAGES;
        if (sl < t0) put((it + (uint32_t)sl) % STAGES);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane < t0) ptx::mbar_arrive(ptx::smem_addr(&bars[(it + (uint32_t)lane) % STAGES]));
    }
    for (int t = t0; t < steps; ++t) {  // warp-uniform
        const uint32_t gi = it + (uint32_t)(w0 + t);
        const uint32_t stage = gi % STAGES, phase = (gi / STAGES) & 1u;
        if (!wait_bar_warp(ptx::smem_addr(&bars[STAGES + stage]), phase ^ 1u, abort_flag, p,
                           5 * 256 + stage))
            return false;
        if (sl == t) put(stage);
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&bars[stage]));
    }
    return true;
}

// Fused activation quantiser (grouped GEMM, single CTA; epilogue warp ew of
// 16): quantises this CTA's 128-row tile of A for K step kb into ring stage
// it % STAGES, from the routed rows' source activations: E4M3 codes with one
// power-of-two scale per 1x32 block, by the arithmetic of fp8g_quantize_rows
// (quant_math.cuh), so the codes and scales equal that quantiser's bit for
// bit.  Thread (ew, lane) takes row 8 ew + lane / 4 and the stage's 32-wide K
// block lane % 4.  The codes go to the stage's A tile in the 128-byte-swizzle
// K-major layout the TMA load would have written (16-byte chunk c of row r at
// (c ^ (r % 8)) * 16 within the row's 128 bytes, 8-row groups of 1 KB), the
// scales' UE8M0 codes to the stage's A chunk (byte 16 d + 4 w + j = row 32 w +
// d, block j).  Rows past the expert and blocks past K: zeros, code 127
// (scale 1), as the TMA zero fill and the scale packer give.  A source row
// outside [0, xq_src_rows) records FP8G_ERR_INVALID_ARG (detail: the routed
// row) and reads as zeros.  With qa_out set, the CTAs of tile column 0 also
// store the codes and fp32 scales of their rows.
//
// Two halves, so that a warp's loads for the next K step are in flight while
// it converts and stores this one (one step at a time, each warp waited a
// whole memory round trip per step): fq_fetch issues the loads (kept in their
// source form), fq_put converts, waits for the stage and stores.
template <bool BF16>
struct FqIn {
    uint4 u[BF16 ? 4 : 8];  // the block's 32 values: bf16 (4 words) or fp32 (8)
    bool live;              // a routed row's block whose source row exists
};

// Routed row and first K of this lane's block of K step kb; whether the block
// belongs to a routed row (and to K).
__device__ __forceinline__ bool fq_block(const GemmParams &p, const Tile &ti, int kb, int ew,
                                         int64_t &grow, int64_t &k0) {
    const int lane = threadIdx.x & 31;
    grow = (int64_t)ti.row0 + ew * 8 + (lane >> 2);
    k0 = (int64_t)kb * kBK + 32 * (lane & 3);
    return grow < ti.row_end && k0 < p.K;
}

// This lane's source row of tile ti (one index load per tile; the same for
// every K step): -1 for rows past the expert; a source row outside
// [0, xq_src_rows) records FP8G_ERR_INVALID_ARG (detail: the routed row) and
// gives -1.
__device__ __forceinline__ int64_t fq_source(const GemmParams &p, const Tile &ti, int ew) {
    const int lane = threadIdx.x & 31;
    const int64_t grow = (int64_t)ti.row0 + ew * 8 + (lane >> 2);
    if (grow >= ti.row_end) return -1;
    const int64_t src = p.xq_rows != nullptr ? (int64_t)__ldg(p.xq_rows + grow) : grow;
    if (src < 0 || src >= p.xq_src_rows) {
        if ((lane & 3) == 0) record_error(p, FP8G_ERR_INVALID_ARG, (unsigned)grow);
        return -1;
    }
    return src;
}

template <bool BF16>
__device__ __forceinline__ FqIn<BF16> fq_fetch(const GemmParams &p, int64_t src, int kb) {
    FqIn<BF16> in;
    const int64_t k0 = (int64_t)kb * kBK + 32 * (threadIdx.x & 3);
    in.live = src >= 0 && k0 < p.K;
    const uint4 *x = reinterpret_cast<const uint4 *>(
        static_cast<const uint8_t *>(p.xq) + ((in.live ? src : 0) * p.K + k0) * (BF16 ? 2 : 4));
#pragma unroll
    for (int i = 0; i < (BF16 ? 4 : 8); ++i)
        in.u[i] = in.live ? __ldg(x + i) : make_uint4(0u, 0u, 0u, 0u);
    return in;
}

template <int STAGES, bool BF16>
__device__ __forceinline__ bool fq_put(const GemmParams &p, const FqIn<BF16> &in, const Tile &ti,
                                       int kb, uint32_t it, int ew, uint32_t a_base,
                                       uint32_t a_bytes, uint32_t sf_base, uint32_t chunk_bytes,
                                       uint64_t *bars, volatile int *abort_flag) {
    const int lane = threadIdx.x & 31;
    int64_t grow, k0;
    const bool in_tile = fq_block(p, ti, kb, ew, grow, k0);
    const uint32_t stage = it % STAGES, phase = (it / STAGES) & 1u;
    const int r = ew * 8 + (lane >> 2);
    const int j = lane & 3;
    // values 8q .. 8q + 7 of the block as fp32 (widened again where used, so
    // that the 32 values never occupy 32 registers at once)
    auto group = [&](int q, float4 &a, float4 &b) {
        if constexpr (BF16) {
            bf16x8_to_f32(in.u[q], a, b);
        } else {
            const uint4 x = in.u[2 * q], y = in.u[2 * q + 1];
            a = make_float4(__uint_as_float(x.x), __uint_as_float(x.y), __uint_as_float(x.z),
                            __uint_as_float(x.w));
            b = make_float4(__uint_as_float(y.x), __uint_as_float(y.y), __uint_as_float(y.z),
                            __uint_as_float(y.w));
        }
    };
    float am = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float4 a, b;
        group(q, a, b);
        am = fmaxf(am, absmax8(a, b));
    }
    const float s = in.live ? pow2_scale<0>(am) : 1.0f;
    uint2 o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        float4 a, b;
        group(q, a, b);
        o[q] = quant8_pow2<0>(a, b, s);
    }
    const uint4 c0 = make_uint4(o[0].x, o[0].y, o[1].x, o[1].y);
    const uint4 c1 = make_uint4(o[2].x, o[2].y, o[3].x, o[3].y);
    if (p.qa_out != nullptr && ti.pn == 0 && in_tile) {
        uint4 *dq = reinterpret_cast<uint4 *>(p.qa_out + grow * p.K + k0);
        dq[0] = c0;
        dq[1] = c1;
        p.sfa_out[grow * p.sfc + k0 / 32] = s;
    }
    // the row's scale word: block j's code in byte j (the four lanes of the row)
    uint32_t word = ((__float_as_uint(s) >> 23) & 0xFFu) << (8 * j);
    word |= __shfl_xor_sync(0xffffffffu, word, 1);
    word |= __shfl_xor_sync(0xffffffffu, word, 2);
    if (!wait_bar_warp(ptx::smem_addr(&bars[STAGES + stage]), phase ^ 1u, abort_flag, p,
                       6 * 256 + stage))
        return false;
    const uint32_t row_base = a_base + stage * a_bytes + (uint32_t)(r >> 3) * 1024u +
                              (uint32_t)(r & 7) * 128u;
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                     row_base + ((uint32_t)((2 * j) ^ (r & 7)) << 4)),
                 "r"(c0.x), "r"(c0.y), "r"(c0.z), "r"(c0.w)
                 : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                     row_base + ((uint32_t)((2 * j + 1) ^ (r & 7)) << 4)),
                 "r"(c1.x), "r"(c1.y), "r"(c1.z), "r"(c1.w)
                 : "memory");
    if (j == 0)
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(sf_base + stage * chunk_bytes +
                                                       16u * (uint32_t)(r & 31) +
                                                       4u * (uint32_t)(r >> 5)),
                     "r"(word)
                     : "memory");
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&bars[stage]));
    return true;
}

// SPLIT: the CTAs of one cluster share an output tile, each taking a
// contiguous range of K blocks; CTA o of the cluster owns columns
// [o 128 / S, (o + 1) 128 / S) of the tile.  As soon as its accumulator is in
// registers, each epilogue warp (32 rows x 32 columns) stages the block in
// its CTA's idle operand ring and pushes it with one bulk copy into the
// owner's receive region (slot: sender, row quarter, column group), counted
// in bytes on the owner's receive barrier; the owner's warps wait for every
// peer's block of their rows, add them to their own partial in rank order (a
// fixed order, so results do not depend on timing) and store.  Blocks are row-major
// 32 x 32 fp32, 16-byte chunks XOR-swizzled by row (lane = row: conflict-free).
// (Sending the blocks straight from registers with 16-byte st.async remote
// stores instead was slower on GB300: 14.8 against 13.2 us per 128 x 4096 x
// 4096 call, the stores alone taking ~2.5 us to issue.)
// FQ (grouped, single CTA): the epilogue warps also quantise A in the kernel
// (fq_fetch / fq_put) from fp32 (FQ = 1) or bf16 (FQ = 2) activations; the
// producer loads only B and B's scale chunk.
template <int MODE, int BN, int NUM_ACC, int STAGES, bool OUT_F32, bool SPLIT, int FQ = 0,
          bool INL = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmParams p) {
    using C_ = Cfg<MODE, BN, NUM_ACC, STAGES, SPLIT>;
    static_assert(!SPLIT || (BN == 128 && C_::CW == 32 && STAGES * C_::A_BYTES >= kEpiWarps * 4096),
                  "split-K: 32 x 32 blocks per epilogue warp, staged in the A ring");
    // split-K tiles are few: the kernel converts its own scale chunks instead
    // of reading chunks that a packing kernel wrote
    // INL: few-tile block-scaled shapes with short K on single CTAs (one tile
    // each) convert their scales the same way
    constexpr bool kInlineSF = (SPLIT || INL) && C_::kBlock;
    static_assert(!INL || (!SPLIT && (MODE == kModeBlock || MODE == kModeGrouped) && FQ == 0),
                  "inline scales, single CTAs");
    static_assert(!kInlineSF || (BN == kBM && kEpiWarps == 2 * kSfWarps), "inline scale layout");
    static_assert(!SPLIT || MODE != kModeGrouped, "split-K: non-grouped only");
    static_assert(!FQ || (MODE == kModeGrouped && !SPLIT && kEpiWarps * 8 == kBM),
                  "fused quantiser: grouped single-CTA kernel, 8 rows per epilogue warp");
    constexpr uint32_t kTxBytes = kInlineSF ? C_::A_BYTES + C_::B_BYTES
                                  : FQ      ? C_::B_BYTES + C_::SFB_BYTES
                                            : C_::TX_BYTES;
    const uint32_t tx_bytes = kTxBytes - (FQ ? 0u : C_::A_BYTES / 8 * (uint32_t)p.a_gap8) -
                              C_::B_BYTES / 8 * (uint32_t)p.b_gap8;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte-swizzled TMA tiles need 1024-byte alignment in the shared window
    const uint32_t raw_base = ptx::smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C_::OFF_BAR);
    auto bar_full = [&](int s) { return ptx::smem_addr(&bars[s]); };
    auto bar_empty = [&](int s) { return ptx::smem_addr(&bars[STAGES + s]); };
    auto bar_accf = [&](int a) { return ptx::smem_addr(&bars[2 * STAGES + a]); };
    auto bar_acce = [&](int a) { return ptx::smem_addr(&bars[2 * STAGES + NUM_ACC + a]); };
    const uint32_t bar_drain = ptx::smem_addr(&bars[2 * STAGES + 2 * NUM_ACC]);
    const uint32_t bar_recv = ptx::smem_addr(&bars[2 * STAGES + 2 * NUM_ACC + 1]);
    const uint32_t bar_drain_sf = ptx::smem_addr(&bars[2 * STAGES + 2 * NUM_ACC + 2]);
    auto bar_sfr = [&](int s) { return ptx::smem_addr(&bars[2 * STAGES + 2 * NUM_ACC + 3 + s]); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C_::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C_::OFF_MISC + 4);
    int32_t *row_off = reinterpret_cast<int32_t *>(smem + C_::OFF_GROUP);
    int32_t *tile_off = row_off + (FP8G_MAX_EXPERTS + 1);
    int32_t *rt_off = tile_off + (FP8G_MAX_EXPERTS + 1);

    // ------------------------------------------------------------ setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(bar_full(s), kInlineSF ? 1 + 2 * kSfWarps : FQ ? 1 + kEpiWarps : 1);
            ptx::mbar_init(bar_empty(s), 1);
            ptx::mbar_init(bar_sfr(s), 1);
        }
        for (int a = 0; a < NUM_ACC; ++a) {
            ptx::mbar_init(bar_accf(a), 1);
            ptx::mbar_init(bar_acce(a), kEpiWarps);
        }
        ptx::mbar_init(bar_drain, 1);
        ptx::mbar_init(bar_recv, 1);
        ptx::mbar_init(bar_drain_sf, 1);
        if constexpr (SPLIT)  // the peers' blocks of this CTA's columns (one tile per cluster)
            ptx::mbar_arrive_expect_tx(bar_recv, (uint32_t)((p.split - 1) * kBM * (BN / p.split) * 4));
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C_::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    // Split-K: every CTA's receive barrier initialised before any peer's push
    if constexpr (SPLIT) ptx::cluster_arrive_release();
    // Non-grouped kernels need nothing from global memory before their roles
    // start: they publish the barriers and the tensor-memory slot here, so
    // that every role begins the moment the dependency wait returns (the
    // first run of each role's code per launch is slow, ~0.25 us per stretch
    // of new code on GB300, and a block-wide barrier after the wait made
    // every role wait for the slowest).
    constexpr bool kEarlySync = MODE != kModeGrouped;
    if constexpr (kEarlySync) {
        ptx::tc_fence_before();
        __syncthreads();
        if constexpr (SPLIT) ptx::cluster_wait();
        ptx::tc_fence_after();
    }
    // Everything above touched only shared / tensor memory and kernel
    // parameters; global memory (which the previous kernel on the stream may
    // still be writing, or reading) is accessed only after this wait.  The
    // next kernel may begin its own prologue.
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();
    int32_t T = (int32_t)p.T;
    // Block scales converted in the kernel (split-K, single CTAs on few
    // tiles): the epilogue warps convert the first window of the first tile's
    // K steps right away, in one stretch of code, ahead of the operand loads.
    // (Grouped kernels know their tiles only after the prefix sums below.)
    bool sf_ok0 = true;
    if constexpr (kInlineSF && MODE != kModeGrouped) {
        const int32_t t0 = SPLIT ? (int32_t)ptx::cluster_id_x() : (int32_t)blockIdx.x;
        if (warp >= kEpiWarp0 && t0 < T) {
            const int rank = SPLIT ? (int)ptx::cluster_rank() : 0;
            const int split = SPLIT ? p.split : 1;
            const Tile ti = get_tile<MODE, BN>(t0, p, nullptr, nullptr, nullptr);
            const int kb0 = rank * p.num_kb / split;
            const int n = (rank + 1) * p.num_kb / split - kb0;
            SfWindow f;
            bool bad = false;
            sf_fetch(p, ti, kb0, n, 0, warp - kEpiWarp0, f);
            sf_ok0 = sf_put<STAGES>(p, ti, kb0, n, 0, 0u, warp - kEpiWarp0, f,
                                    sbase + C_::OFF_SF, C_::CHUNK_BYTES, bars, abort_flag, bad,
                                    true);
            if (__any_sync(0xffffffffu, bad) && lane == 0) record_error(p, FP8G_ERR_SCALE_FORMAT, 0);
        }
    }
    if constexpr (!kEarlySync) {
        if constexpr (MODE == kModeGrouped) grouped_prefix(p, kBM, row_off, tile_off, rt_off);
        ptx::tc_fence_before();
        __syncthreads();
        ptx::tc_fence_after();
        if constexpr (MODE == kModeGrouped) T = tile_off[p.E];
    }
    const uint32_t tmem_base = *tmem_slot;

    // work of this CTA: tiles t_first, t_first + t_step, ...; K blocks [kb_begin, kb_end)
    int32_t t_first = blockIdx.x, t_step = gridDim.x;
    int kb_begin = 0, kb_end = p.num_kb;
    if constexpr (SPLIT) {
        const int rank = (int)ptx::cluster_rank();
        t_first = (int32_t)ptx::cluster_id_x();
        t_step = (int32_t)ptx::num_clusters_x();
        kb_begin = rank * p.num_kb / p.split;
        kb_end = (rank + 1) * p.num_kb / p.split;
    }

    // ------------------------------------------------------------ roles
    if (warp == 0) {
        // ===== TMA producer: A, B (and the packed scale chunks) per stage =====
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            for (int32_t t = t_first; t < T; t += t_step) {
                const Tile ti = get_tile<MODE, BN>(t, p, row_off, tile_off, rt_off);
                if constexpr (MODE == kModeGrouped) {
                    if (p.tile_map_out != nullptr) {
                        int4 v = make_int4(ti.e, ti.pm, ti.pn, 0);
                        *reinterpret_cast<int4 *>(p.tile_map_out + 4 * (int64_t)t) = v;
                    }
                }
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!wait_bar(bar_empty(stage), phase ^ 1u, abort_flag, p, 0 * 256 + stage))
                        goto roles_done;
                    const uint32_t fb = bar_full(stage);
                    ptx::mbar_arrive_expect_tx(fb, tx_bytes);
                    if constexpr (!FQ)
                        ptx::tma_load_2d(sbase + C_::OFF_A + stage * C_::A_BYTES, &tmA, fb,
                                         kb * kBK, ti.row0);
                    if constexpr (MODE == kModeGrouped)
                        ptx::tma_load_3d(sbase + C_::OFF_B + stage * C_::B_BYTES, &tmB, fb,
                                         kb * kBK, ti.n0, ti.e);
                    else
                        ptx::tma_load_2d(sbase + C_::OFF_B + stage * C_::B_BYTES, &tmB, fb,
                                         kb * kBK, ti.n0);
                    if constexpr (C_::kBlock && !kInlineSF) {
                        const uint32_t dst = sbase + C_::OFF_SF + stage * C_::CHUNK_BYTES;
                        const uint8_t *sa_src =
                            p.sfa_pk + ((int64_t)kb * p.n_rtA + ti.rtA) * 512;
                        const uint8_t *sb_src =
                            p.sfb_pk +
                            (((int64_t)ti.e * p.num_kb + kb) * p.n_rtB + ti.n0 / kBM) * 512;
                        if constexpr (!FQ) ptx::bulk_load(dst, sa_src, kBM * 4, fb);
                        if constexpr (C_::kRepB) {
                            const uint8_t *sb_rep =
                                p.sfb_pk +
                                (((int64_t)ti.e * p.num_kb + kb) * (p.n_rtB / 2) + ti.n0 / 256) *
                                    4096;
                            ptx::bulk_load(dst + kBM * 4, sb_rep, C_::SFB_BYTES, fb);
                        } else {
                            ptx::bulk_load(dst + kBM * 4, sb_src, BN * 4, fb);
                        }
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ===== MMA issuer =====
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int32_t lt = 0;
            for (int32_t t = t_first; t < T; t += t_step, ++lt) {
                const int acc = lt % NUM_ACC;
                const uint32_t acc_par = (uint32_t)((lt / NUM_ACC) & 1);
                if (!wait_bar(bar_acce(acc), acc_par ^ 1u, abort_flag, p, 1 * 256 + 64 + acc))
                    goto roles_done;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    // block modes: data and scale factors in place (the
                    // scale-copy thread waited for "full" and committed its copies)
                    const uint32_t rb = C_::kBlock ? bar_sfr(stage) : bar_full(stage);
                    if (!wait_bar(rb, phase, abort_flag, p, 1 * 256 + stage)) goto roles_done;
                    ptx::tc_fence_after();
                    const uint32_t a0 = sbase + C_::OFF_A + stage * C_::A_BYTES;
                    const uint32_t b0 = sbase + C_::OFF_B + stage * C_::B_BYTES;
                    if constexpr (C_::kBlock) {
                        const uint32_t sf_tmem = tmem_base + C_::SF_COL0 + stage * C_::SF_COLS;
#pragma unroll
                        for (int k = 0; k < kBK / 32; ++k)
                            ptx::mma_mxf8(d_tmem, ptx::desc_kmajor_sw128(a0 + k * 32),
                                          ptx::desc_kmajor_sw128(b0 + k * 32),
                                          ptx::idesc_mxf8(kBM, BN, (uint32_t)k) | p.ab_fmt, sf_tmem,
                                          sf_tmem + C_::SFB_COL,
                                          (kb != kb_begin || k != 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int k = 0; k < kBK / 32; ++k)
                            ptx::mma_f8(d_tmem, ptx::desc_kmajor_sw128(a0 + k * 32),
                                        ptx::desc_kmajor_sw128(b0 + k * 32),
                                        ptx::idesc_f8(kBM, BN) | p.ab_fmt,
                                        (kb != kb_begin || k != 0) ? 1u : 0u);
                    }
                    ptx::tc_commit(bar_empty(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                ptx::tc_commit(bar_accf(acc));
            }
        }
    } else if (warp == 2 && C_::kBlock) {
        // ===== scale-factor copies shared -> tensor memory (block modes) =====
        // Issued from the MMA thread, each copy stalls the MMA stream; from
        // their own thread they overlap the previous stages' MMAs.  A stage's
        // tensor-memory slot is rewritten only after "full" of its next use,
        // i.e. after the producer saw the MMAs that read it complete.
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            for (int32_t t = t_first; t < T; t += t_step) {
                for (int kb = kb_begin; kb < kb_end; ++kb) {
                    if (!wait_bar(bar_full(stage), phase, abort_flag, p, 2 * 256 + stage))
                        goto roles_done;
                    ptx::tc_fence_after();
                    const uint32_t sf_tmem = tmem_base + C_::SF_COL0 + stage * C_::SF_COLS;
                    const uint32_t sfa_s = sbase + C_::OFF_SF + stage * C_::CHUNK_BYTES;
                    ptx::tc_cp_32x128b_warpx4(sf_tmem, ptx::desc_sf_chunk(sfa_s));
                    if constexpr (C_::kRepB)
                        ptx::tc_cp_128x256b(sf_tmem + C_::SFB_COL,
                                            ptx::desc_sf_128x256b(sfa_s + kBM * 4));
                    else
                        ptx::tc_cp_32x128b_warpx4(sf_tmem + C_::SFB_COL,
                                                  ptx::desc_sf_chunk(sfa_s + kBM * 4));
                    ptx::tc_commit(bar_sfr(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (FQ != 0 && warp >= kEpiWarp0) {
        // ===== fused quantiser + epilogue =====
        // Each warp quantises its 8 rows of A for every K step (fq_fetch /
        // fq_put) and drains / stores the previous tile's accumulator once
        // the first min(STAGES - 1, num_kb) steps of the next tile are
        // quantised: those steps wait only for the previous tile's MMAs, and
        // a tile's first MMA waits only for the drain of the tile NUM_ACC
        // before it, which came earlier, so neither order can deadlock.
        const int ew = warp - kEpiWarp0;
        const int q = warp & 3;
        const int col0 = (ew >> 2) * C_::CW;
        int32_t ltd = 0;  // tiles drained
        uint32_t it = 0;  // K steps quantised (the ring's stage counter)
        Tile prev{};
        bool have_prev = false;
        auto drain_store = [&](const Tile &ti) -> bool {
            const int acc = ltd % NUM_ACC;
            if (!wait_bar_warp(bar_accf(acc), (uint32_t)((ltd / NUM_ACC) & 1), abort_flag, p,
                               3 * 256 + acc, 128))
                return false;
            ptx::tc_fence_after();
            uint32_t r[C_::CW / 32][32];
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN + col0;
#pragma unroll
            for (int c = 0; c < C_::CW / 32; ++c) ptx::tmem_ld_32x32b_x32(taddr + c * 32, r[c]);
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_acce(acc));
            ++ltd;
            const int64_t arow = (int64_t)ti.row0 + q * 32 + lane;          // routed row
            const int64_t row = arow < ti.row_end ? out_row(p, arow) : -1;  // row of C
            if (row >= 0) {
                const int64_t ncol0 = (int64_t)ti.n0 + col0;
                if (p.bias != nullptr || p.act != FP8G_ACT_NONE) {
                    const float *brow = p.bias != nullptr ? p.bias + (int64_t)ti.e * p.N : nullptr;
#pragma unroll
                    for (int c = 0; c < C_::CW / 32; ++c)
                        epi32(r[c], 1.0f, brow, p.act, ncol0 + c * 32, p.N);
                }
#pragma unroll
                for (int c = 0; c < C_::CW / 32; ++c)
                    store_row32<OUT_F32>(p.C, row, p.N, ncol0 + c * 32, r[c], 1.0f, p.st32 != 0);
            }
            return true;
        };
        // K steps in order over this CTA's tiles; the loads of the next step
        // are issued before the current one is converted, except across a
        // drain (no loads held in registers beside the accumulator)
        {
            constexpr bool BF = FQ == 2;
            // bf16: one step of loads in flight ahead (16 registers); fp32
            // (32 registers per step) fetches each step just before its use
            constexpr bool kAhead = BF;
            FqIn<BF> nxt;
            bool have_nxt = false;
            int64_t src_next = -1;  // the next tile's source row, once fetched ahead
            for (int32_t t = t_first; t < T; t += t_step) {
                const Tile ti = get_tile<MODE, BN>(t, p, row_off, tile_off, rt_off);
                const int64_t src = have_nxt ? src_next : fq_source(p, ti, ew);
                const int pre = p.num_kb < STAGES - 1 ? p.num_kb : STAGES - 1;
                for (int kb = 0; kb <= p.num_kb; ++kb) {
                    if (kb == pre && have_prev) {
                        if (!drain_store(prev)) goto roles_done;
                        have_prev = false;
                    }
                    if (kb == p.num_kb) break;
                    if (!have_nxt) nxt = fq_fetch<BF>(p, src, kb);
                    const FqIn<BF> cur = nxt;
                    have_nxt = false;
                    if constexpr (kAhead) {
                        if (kb + 1 < p.num_kb) {
                            if (!(kb + 1 == pre && have_prev)) {
                                nxt = fq_fetch<BF>(p, src, kb + 1);
                                have_nxt = true;
                            }
                        } else if (t + t_step < T) {  // the next tile's first step: no drain before it
                            src_next = fq_source(
                                p, get_tile<MODE, BN>(t + t_step, p, row_off, tile_off, rt_off), ew);
                            nxt = fq_fetch<BF>(p, src_next, 0);
                            have_nxt = true;
                        }
                    }
                    if (!fq_put<STAGES, BF>(p, cur, ti, kb, it, ew, sbase + C_::OFF_A, C_::A_BYTES,
                                            sbase + C_::OFF_SF, C_::CHUNK_BYTES, bars, abort_flag))
                        goto roles_done;
                    ++it;
                }
                prev = ti;
                have_prev = true;
            }
        }
        if (have_prev) (void)drain_store(prev);
    } else if (kInlineSF && MODE == kModeGrouped && warp >= kEpiWarp0) {
        // ===== grouped: scale conversion + epilogue =====
        // Each warp converts its 16 rows' scales for every K step of this
        // CTA's tiles (windows of 8 steps: sf_fetch / sf_put), and drains /
        // stores the previous tile's accumulator once the next tile's first
        // window is in the ring.  Converting a step waits only for the MMAs of
        // earlier steps (its ring slot), and a tile's MMAs wait only for the
        // drain of the tile NUM_ACC before it, which came earlier, so this
        // order cannot deadlock.  The next window's loads are issued before the
        // current one is converted, so they are in flight across a drain too.
        const int ew = warp - kEpiWarp0;
        const int q = warp & 3;
        const int col0 = (ew >> 2) * C_::CW;
        const int n = p.num_kb;
        int32_t ltd = 0;  // tiles drained
        uint32_t it = 0;  // K steps converted before the current tile (the ring's counter)
        bool bad = false;
        Tile prev{};
        bool have_prev = false;
        auto drain_store = [&](const Tile &ti) -> bool {
            const int acc = ltd % NUM_ACC;
            if (!wait_bar_warp(bar_accf(acc), (uint32_t)((ltd / NUM_ACC) & 1), abort_flag, p,
                               3 * 256 + acc, 128))
                return false;
            ptx::tc_fence_after();
            uint32_t r[C_::CW / 32][32];
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN + col0;
#pragma unroll
            for (int c = 0; c < C_::CW / 32; ++c) ptx::tmem_ld_32x32b_x32(taddr + c * 32, r[c]);
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_acce(acc));
            ++ltd;
            const int64_t arow = (int64_t)ti.row0 + q * 32 + lane;          // routed row
            const int64_t row = arow < ti.row_end ? out_row(p, arow) : -1;  // row of C
            if (row >= 0) {
                const int64_t ncol0 = (int64_t)ti.n0 + col0;
                if (p.bias != nullptr || p.act != FP8G_ACT_NONE) {
                    const float *brow = p.bias != nullptr ? p.bias + (int64_t)ti.e * p.N : nullptr;
#pragma unroll
                    for (int c = 0; c < C_::CW / 32; ++c)
                        epi32(r[c], 1.0f, brow, p.act, ncol0 + c * 32, p.N);
                }
#pragma unroll
                for (int c = 0; c < C_::CW / 32; ++c)
                    store_row32<OUT_F32>(p.C, row, p.N, ncol0 + c * 32, r[c], 1.0f, p.st32 != 0);
            }
            return true;
        };
        SfWindow f;
        Tile ti{};
        if (t_first < T) {
            ti = get_tile<MODE, BN>(t_first, p, row_off, tile_off, rt_off);
            sf_fetch(p, ti, 0, n, 0, ew, f);
        }
        for (int32_t t = t_first; t < T; t += t_step) {
            Tile tn = ti;  // the tile of the next window
            for (int w0 = 0; w0 < n; w0 += 8) {
                const SfWindow cur = f;
                int wn = w0 + 8;
                bool more = true;
                if (wn >= n) {
                    wn = 0;
                    more = t + t_step < T;
                    if (more) tn = get_tile<MODE, BN>(t + t_step, p, row_off, tile_off, rt_off);
                }
                if (more) sf_fetch(p, tn, 0, n, wn, ew, f);
                if (!sf_put<STAGES>(p, ti, 0, n, w0, it, ew, cur, sbase + C_::OFF_SF,
                                    C_::CHUNK_BYTES, bars, abort_flag, bad, it == 0 && w0 == 0))
                    goto roles_done;
                if (w0 == 0 && have_prev) {
                    if (!drain_store(prev)) goto roles_done;
                    have_prev = false;
                }
            }
            it += (uint32_t)n;
            prev = ti;
            have_prev = true;
            ti = tn;
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0) record_error(p, FP8G_ERR_SCALE_FORMAT, 0);
        if (have_prev) (void)drain_store(prev);
    } else if (warp >= kEpiWarp0) {
        // ===== epilogue =====
        const int ew = warp - kEpiWarp0;
        const int q = warp & 3;           // tensor-memory lane quarter of this warp
        const int col0 = (ew >> 2) * C_::CW;
        float alpha = 1.0f;
        if constexpr (MODE == kModeTensor) alpha = __fmul_rn(p.sa[0], p.sb[0]);
        int32_t lt = 0;
        uint32_t it = 0;  // K steps of this CTA so far (the ring's stage counter)
        for (int32_t t = t_first; t < T; t += t_step, ++lt) {
            const Tile ti = get_tile<MODE, BN>(t, p, row_off, tile_off, rt_off);
            if constexpr (kInlineSF) {
                const int n = kb_end - kb_begin;
                bool bad = false, ok = lt > 0 || sf_ok0;
                // (the first tile's first window was converted after the dependency wait)
                for (int w0 = lt == 0 ? 8 : 0; w0 < n && ok; w0 += 8) {
                    SfWindow f;
                    sf_fetch(p, ti, kb_begin, n, w0, ew, f);
                    ok = sf_put<STAGES>(p, ti, kb_begin, n, w0, it, ew, f, sbase + C_::OFF_SF,
                                        C_::CHUNK_BYTES, bars, abort_flag, bad, false);
                }
                if (__any_sync(0xffffffffu, bad) && lane == 0)
                    record_error(p, FP8G_ERR_SCALE_FORMAT, 0);
                if (!ok) break;
                it += (uint32_t)n;
            }
            const int acc = lt % NUM_ACC;
            const uint32_t acc_par = (uint32_t)((lt / NUM_ACC) & 1);
            if (!wait_bar_warp(bar_accf(acc), acc_par, abort_flag, p, 3 * 256 + acc, 128)) break;
            ptx::tc_fence_after();
            uint32_t r[C_::CW / 32][32];
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN + col0;
#pragma unroll
            for (int c = 0; c < C_::CW / 32; ++c) ptx::tmem_ld_32x32b_x32(taddr + c * 32, r[c]);
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_acce(acc));

            if constexpr (SPLIT) {
                const int S = p.split;
                const int rank = (int)ptx::cluster_rank();
                const int cg = ew >> 2;                  // this warp's 32 columns of the 128
                const int owner = cg * S / 4;            // CTA that sums these columns
                const int cgi = cg - owner * (4 / S);    // 32-column group within its slice
                auto chunk = [&](uint32_t blk, int v) {  // 16-byte chunk v of row `lane`
                    return blk + (uint32_t)lane * 128u + ((uint32_t)(v ^ (lane & 7)) << 4);
                };
                if (owner != rank) {
                    // the ring is idle (every MMA, hence every operand read, completed)
                    const uint32_t blk = sbase + C_::OFF_A + (uint32_t)ew * 4096u;
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(chunk(blk, v)),
                                     "r"(r[0][4 * v]), "r"(r[0][4 * v + 1]), "r"(r[0][4 * v + 2]),
                                     "r"(r[0][4 * v + 3])
                                     : "memory");
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int slot = rank < owner ? rank : rank - 1;
                        const uint32_t dst = sbase + C_::OFF_RECV +
                                             (uint32_t)(((slot * 4 + q) * (4 / S) + cgi) * 4096);
                        ptx::bulk_push(ptx::map_shared(dst, (uint32_t)owner), blk, 4096u,
                                       ptx::map_shared(bar_recv, (uint32_t)owner));
                    }
                    continue;
                }
                // own columns: every peer's block of these rows, then the sum in a
                // fixed order: this CTA's partial, then the peers' in rank order
                if (!wait_bar_landed_warp(bar_recv, 0, abort_flag, p, 4 * 256)) break;
                for (int sl = 0; sl < S - 1; ++sl) {
                    const uint32_t blk = sbase + C_::OFF_RECV +
                                         (uint32_t)(((sl * 4 + q) * (4 / S) + cgi) * 4096);
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        float x0, x1, x2, x3;
                        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                     : "=f"(x0), "=f"(x1), "=f"(x2), "=f"(x3)
                                     : "r"(chunk(blk, v))
                                     : "memory");
                        r[0][4 * v] = __float_as_uint(__fadd_rn(__uint_as_float(r[0][4 * v]), x0));
                        r[0][4 * v + 1] = __float_as_uint(__fadd_rn(__uint_as_float(r[0][4 * v + 1]), x1));
                        r[0][4 * v + 2] = __float_as_uint(__fadd_rn(__uint_as_float(r[0][4 * v + 2]), x2));
                        r[0][4 * v + 3] = __float_as_uint(__fadd_rn(__uint_as_float(r[0][4 * v + 3]), x3));
                    }
                }
            }
            const int64_t arow = (int64_t)ti.row0 + q * 32 + lane;  // routed row
            const int64_t row = arow < ti.row_end ? out_row(p, arow) : -1;  // row of C
            if (row >= 0) {
                const int64_t ncol0 = (int64_t)ti.n0 + col0;
                float a_t = alpha;  // scale left for the stores below
                if (p.bias != nullptr || p.act != FP8G_ACT_NONE) {
                    const float *brow = p.bias != nullptr ? p.bias + (int64_t)ti.e * p.N : nullptr;
#pragma unroll
                    for (int c = 0; c < C_::CW / 32; ++c)
                        epi32(r[c], alpha, brow, p.act, ncol0 + c * 32, p.N);
                    a_t = 1.0f;
                }
#pragma unroll
                for (int c = 0; c < C_::CW / 32; ++c)
                    store_row32<OUT_F32>(p.C, row, p.N, ncol0 + c * 32, r[c], a_t, p.st32 != 0);
            }
        }
    }

roles_done:
    __syncwarp();
    __syncthreads();
    if (*abort_flag) {
        // Drain: wait (bounded) for this CTA's MMAs, then give in-flight TMA
        // copies a bounded grace period before shared memory is released.
        if ((warp == 1 || (warp == 2 && C_::kBlock)) && lane == 0) {
            const uint32_t db = warp == 1 ? bar_drain : bar_drain_sf;
            ptx::tc_commit(db);
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(db, 0) && ptx::globaltimer() - t0 < p.timeout_ns) {
            }
        }
        const uint64_t t0 = ptx::globaltimer();
        while (ptx::globaltimer() - t0 < 200000ull) {
        }
        __syncthreads();
    }
    if constexpr (SPLIT) {
        // A CTA leaves only when every CTA of the cluster has received all its
        // blocks (each CTA arrives after its own receive barrier completed or
        // gave up), i.e. when no copy reads or writes its shared memory.
        ptx::cluster_arrive_relaxed();
        ptx::cluster_wait();
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C_::TMEM_COLS);
    }
}

template <int MODE, int BN, int NUM_ACC, int STAGES, bool OUT_F32, bool SPLIT, int FQ = 0,
          bool INL = false>
cudaError_t launch_one(const GemmMaps &maps, const GemmParams &p, const KernelChoice &kc,
                       cudaStream_t stream) {
    using C_ = Cfg<MODE, BN, NUM_ACC, STAGES, SPLIT>;
    auto kern = gemm_kernel<MODE, BN, NUM_ACC, STAGES, OUT_F32, SPLIT, FQ, INL>;
    // The shared-memory opt-in is per device; the flag races benignly (the
    // attribute set is idempotent).
    static unsigned long long attr_done = 0ull;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if ((attr_done & bit) == 0ull) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C_::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done |= bit;
    }
    // Programmatic dependent launch: the prologue (barrier init, tensor-memory
    // allocation, descriptor prefetch) overlaps the previous kernel's tail;
    // the kernel waits (griddepcontrol.wait) before touching global memory.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)kc.grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C_::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int n = 1;
    if constexpr (SPLIT) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)kc.split;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, maps.A, maps.B, p);
}

// Clusters of `S` split-K CTAs that can be resident at once on the current
// device (cudaOccupancyMaxActiveClusters; cached per device).  Clusters are
// placed inside one GPC, so the count is not SMs / S: on GB300 (152 SMs) with
// these ~200 KB CTAs, 76 pairs fit but only 36 clusters of four.  A grid of
// more clusters would run the rest as a second wave.  0 if unknown.
int max_split_clusters(int S) {
    static std::atomic<int> cache[64][kMaxSplit + 1];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || S < 1 || S > kMaxSplit)
        return 0;
    int v = cache[dev][S].load(std::memory_order_relaxed);
    if (v > 0) return v;
    using C_ = Cfg<kModeBlock, 128, 1, kSplitStages, true>;  // the larger split-K footprint
    auto kern = gemm_kernel<kModeBlock, 128, 1, kSplitStages, false, true>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C_::SMEM_BYTES) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(S * 64), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = C_::SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
        cudaGetLastError();  // clear
        return 0;
    }
    cache[dev][S].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace

KernelChoice choose_kernel(int mode, int64_t M, int64_t N, int64_t K, int num_sms) {
    KernelChoice kc;
    kc.BM = kBM;
    kc.BN = 256;
    kc.b_rows = 256;
    kc.split = 1;
    kc.cluster = 1;
    kc.pair = false;
    kc.inl = false;
    if (mode == kModeGrouped) {
        // at least a wave of 128 x 256 tiles (counting rows as one problem):
        // 256 x 256 tiles on CTA pairs inside each expert
        const int64_t est = (M / kBM) * ((N + 255) / 256);
        if (est >= num_sms && num_sms >= 2) {
            kc.BM = 256;
            kc.b_rows = 128;
            kc.cluster = 2;
            kc.pair = true;
            kc.grid = 2 * (num_sms / 2);
        } else {
            // Less than a wave: 128 x 128 tiles, twice as many, so the last
            // wave idles half as long (each expert's rows are padded to whole
            // tiles, so the tile count exceeds the estimate: decode-shaped
            // MoE, 256 routed rows over 3 experts, N = 14336: 168 tiles of
            // 128 x 256 on 148 SMs are two waves, the second 14% full).  The
            // kernel converts its own block scales (no packing kernel, whose
            // pass over the used experts' fp32 scales would precede it; a
            // fused-quantiser call packs B's scales all the same)
            kc.BN = 128;
            kc.b_rows = 128;
            kc.inl = true;
            kc.grid = num_sms;
        }
        return kc;
    }
    const int64_t num_kb = (K + kBK - 1) / kBK;
    const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + kc.BN - 1) / kc.BN);
    // Few output tiles: 128-wide tiles, K split over a cluster of S CTAs per
    // tile (S a power of two <= kMaxSplit and <= the K blocks, S * tiles <= SMs,
    // and every cluster resident at once).
    if (tiles * 2 <= num_sms && num_kb >= kMinSplitKb) {
        const int64_t tiles128 = ((M + kBM - 1) / kBM) * ((N + 127) / 128);
        int S = 1;
        while (S * 2 <= kMaxSplit && S * 2 <= num_kb && tiles128 * S * 2 <= num_sms) {
            const int cap = max_split_clusters(S * 2);
            if (cap > 0 && tiles128 > cap) break;
            S *= 2;
        }
        if (S >= 2) {
            kc.BN = 128;
            kc.b_rows = 128;
            kc.split = S;
            kc.cluster = S;
            kc.grid = (int)(tiles128 * S);
            return kc;
        }
    }
    if (tiles * 2 <= num_sms) {
        // few tiles, short K: one CTA per 128 x 128 tile, two accumulators;
        // block-scaled: scales converted in the kernel (no packing kernel)
        kc.BN = 128;
        kc.b_rows = 128;
        kc.inl = mode == kModeBlock;
        const int64_t t128 = ((M + kBM - 1) / kBM) * ((N + 127) / 128);
        kc.grid = (int)(t128 < num_sms ? t128 : num_sms);
        return kc;
    }
    // At least a wave of tiles: 256 x 256 tiles on CTA pairs.
    if (tiles >= num_sms) {
        const int64_t pairs = ((M + 255) / 256) * ((N + 255) / 256);
        const int64_t clusters = pairs < num_sms / 2 ? pairs : num_sms / 2;
        kc.BM = 256;
        kc.b_rows = 128;
        kc.cluster = 2;
        kc.pair = true;
        kc.grid = (int)(2 * clusters);
        return kc;
    }
    kc.grid = (int)(tiles < num_sms ? tiles : num_sms);
    if (kc.grid < 1) kc.grid = 1;
    return kc;
}

cudaError_t launch_gemm(int mode, bool out_f32, const GemmMaps &maps, const GemmParams &p,
                        const KernelChoice &kc, cudaStream_t stream) {
    const bool split = kc.split > 1;
    if (kc.pair && p.xq != nullptr) return cudaErrorInvalidValue;
    if (kc.pair) return launch_gemm_pair(mode, out_f32, maps, p, kc.grid, stream);
    if (mode == kModeTensor) {
        if (split)
            return out_f32 ? launch_one<kModeTensor, 128, 1, kSplitStages, true, true>(maps, p, kc, stream)
                           : launch_one<kModeTensor, 128, 1, kSplitStages, false, true>(maps, p, kc, stream);
        if (kc.BN == 128)  // few tiles, short K
            return out_f32 ? launch_one<kModeTensor, 128, 2, 6, true, false>(maps, p, kc, stream)
                           : launch_one<kModeTensor, 128, 2, 6, false, false>(maps, p, kc, stream);
        return out_f32 ? launch_one<kModeTensor, 256, 2, 4, true, false>(maps, p, kc, stream)
                       : launch_one<kModeTensor, 256, 2, 4, false, false>(maps, p, kc, stream);
    } else if (mode == kModeBlock) {
        if (split)
            return out_f32 ? launch_one<kModeBlock, 128, 1, kSplitStages, true, true>(maps, p, kc, stream)
                           : launch_one<kModeBlock, 128, 1, kSplitStages, false, true>(maps, p, kc, stream);
        if (kc.inl)  // few tiles, short K
            return out_f32 ? launch_one<kModeBlock, 128, 2, 6, true, false, 0, true>(maps, p, kc, stream)
                           : launch_one<kModeBlock, 128, 2, 6, false, false, 0, true>(maps, p, kc, stream);
        return out_f32 ? launch_one<kModeBlock, 256, 1, 4, true, false>(maps, p, kc, stream)
                       : launch_one<kModeBlock, 256, 1, 4, false, false>(maps, p, kc, stream);
    } else if (p.xq != nullptr) {
        // fused activation quantiser (single CTAs, 128 x 128 tiles)
        if (kc.pair || split || kc.BN != 128) return cudaErrorInvalidValue;
        if (p.xq_bf16)
            return out_f32 ? launch_one<kModeGrouped, 128, 2, 6, true, false, 2>(maps, p, kc, stream)
                           : launch_one<kModeGrouped, 128, 2, 6, false, false, 2>(maps, p, kc, stream);
        return out_f32 ? launch_one<kModeGrouped, 128, 2, 6, true, false, 1>(maps, p, kc, stream)
                       : launch_one<kModeGrouped, 128, 2, 6, false, false, 1>(maps, p, kc, stream);
    } else {
        // 128 x 128 tiles, two 128-column accumulators: the epilogue of a tile
        // overlaps the next tile's MMAs; the kernel converts its own scales
        if (kc.BN != 128 || !kc.inl) return cudaErrorInvalidValue;
        return out_f32 ? launch_one<kModeGrouped, 128, 2, 6, true, false, 0, true>(maps, p, kc, stream)
                       : launch_one<kModeGrouped, 128, 2, 6, false, false, 0, true>(maps, p, kc, stream);
    }
}

}  // namespace fp8g
