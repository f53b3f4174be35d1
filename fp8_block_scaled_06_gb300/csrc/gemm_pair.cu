// FP8 / FP6 / FP4 GEMMs on CTA pairs (tcgen05 cta_group::2), sm_103a:
// per-tensor, block-scaled and grouped, any E4M3 / E5M2 / E2M3 / E3M2 / E2M1
// operand pairing on the FP8-rate MMA; MXFP4 and NVFP4 on the FP4-rate MMAs.
//
// Why: the single-CTA kernel stages 48 KB per 128-wide K step for a 128x256
// output tile, so four stages fill shared memory and cannot hide the refill
// latency (measured tensor-pipe activity 64%).  A cluster of two CTAs
// computes a 256x256 tile with one MMA stream: each CTA loads its own 128 rows
// of A and 128 rows (one half) of B, 32 KB per K step, so each SM holds six
// stages (seven per-tensor, without scale chunks) and the same MMA work per
// SM needs two thirds of the bytes.
//
// Roles (640 threads per CTA, as in the single-CTA kernel):
//   warp 0   both CTAs: TMA producer for the CTA's own halves; both complete
//            on the even CTA's full barrier (TMA cta_group::2)
//   warp 1   even CTA: the single MMA-issuing thread (M = 256, N = 256)
//   warp 2   even CTA, block modes: copies each stage's scale factors shared
//            -> tensor memory and commits them to the stage's "scales ready"
//            barrier, which the MMA thread waits on instead of "full".  Issued
//            from the MMA thread, each copy stalled the MMA stream (~6-7% per
//            copy instruction); from their own warp the copies overlap the
//            previous stages' MMAs (8192^3: 395 -> 363 us).
//   warp 3   even CTA, NVFP4 only: a second scale-copy warp (half the K
//            groups; both commit to "scales ready")
//   warps 4-19 both CTAs: epilogue of the CTA's 128 accumulator rows; the
//            accumulator release is counted on the even CTA's barrier
// The MMA thread's commits go to both CTAs' barriers (multicast), so each
// producer learns when a stage is free and each epilogue when its rows are
// final.  Persistent over 256x256 tiles in the grouped raster order.  Every
// wait is bounded; tensor memory (512 columns: two accumulators per-tensor,
// one accumulator plus per-stage scale factors block-scaled; an accumulator
// is released as soon as it is in registers) is allocated and freed by both
// CTAs together.
//
// F4 = 1 (E2M1 x E2M1 with 1x32 power-of-two scales, i.e. MXFP4, at the FP4
// rate): kind::mxf4 reads dense 4-bit operands, so the packed codes are
// loaded as plain bytes and a 128-byte swizzled row of a stage holds 256 K
// elements; each of the four MMAs per stage takes K = 64 (32 bytes, the same
// descriptor step as FP8) with two scale bytes per row.  A stage therefore
// carries two 128-wide K groups of packed scales (3 KB: A's two chunks, B's
// two pairs of chunks), copied to a second set of scale columns.
// F4 = 2 (NVFP4: 1x16 E4M3 block scales, kind::mxf4nvf4 scale_vec::4X): the
// same operand stages, but each MMA reads four scale bytes per row, so a stage
// carries four 64-wide K groups of scales (6 KB, loaded as two copies: the
// packing keeps a stage's groups adjacent); tensor memory then holds 12 scale
// columns per group (48 per stage), which leaves room for 5 stages.  The
// output is scaled by the product of the two fp32 tensor scales, per expert
// on the grouped GEMM (each expert's B has its own).
// F4 = 3 (per-tensor mode, TF32): fp32 operands (32 K values per 128-byte
// row of a stage) through kind::tf32 MMAs, alpha = 1: the literal-scale GEMM
// after its operands were dequantised with their fp32 block scales.
#include <cuda_bf16.h>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace fp8g {

namespace {

constexpr int kThreads = 640;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 16;
constexpr int kPairBN = 256;                 // output tile: 256 x 256 per pair
constexpr int kA = kBM * kBK;                // 16 KB: this CTA's 128 rows of A
constexpr int kB = (kPairBN / 2) * kBK;      // 16 KB: this CTA's half of B

// Block-scaled pairs: each CTA's tensor memory holds the scale factors of
// its own 128 rows of A but of all 256 rows (both halves) of the tile's B,
// and tcgen05.cp.cta_group::2 copies each CTA's shared memory into its own
// tensor memory.  (Established on GB300 by the exact scale-layout test: with
// only the CTA's own half of B's scales the results are wrong.)  Per K step
// three 32x128b.warpx4 copies (each replicated over the four lane quarters by
// the copy): A's 128 rows, B's rows 0-127 and 128-255, from 1.5 KB of packed
// chunks.  Issued by their own warp the copies overlap the MMAs, so three
// small copies beat one 128x256b copy from a pre-replicated 4 KB source
// (which saved copy instructions when the MMA thread issued them).
constexpr int kSfaBytes = 512;
constexpr int kSfbBytes = 1024;  // B's two 128-row chunks

template <int MODE, int F4>
struct PairCfg {
    static constexpr bool kBlock = MODE != kModeTensor;
    static_assert(kBlock || F4 == 0 || F4 == 3, "FP4-rate MMAs are block-scaled");
    static_assert(F4 != 3 || !kBlock, "TF32 operands carry their scales (per-tensor mode)");
    static constexpr int STAGES = F4 == 2 ? 5 : kBlock ? 6 : 7;
    // K groups of packed scales per stage: 128-wide (FP8, MXFP4) or 64-wide (NVFP4)
    static constexpr int G = F4 == 2 ? 4 : F4 == 1 ? 2 : 1;
    static constexpr int CHUNK = kBlock ? G * (kSfaBytes + kSfbBytes) : 0;  // packed scales per stage
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * kA;
    static constexpr int OFF_SF = OFF_B + STAGES * kB;
    static constexpr int OFF_BAR = OFF_SF + STAGES * CHUNK;
    // Accumulators: per-tensor double-buffers the 256-column accumulator (the
    // next tile's MMAs never wait for the epilogue); block modes keep one and
    // use the other columns for the scale factors of each stage.
    static constexpr int NUM_ACC = kBlock ? 1 : 2;
    // Scale-copy issuers: one warp, two for NVFP4 (12 copies per stage are
    // more than one thread issues in a stage's time; measured 8192^3: 3955 ->
    // 5610 TFLOPS without them)
    static constexpr int SF_WARPS = F4 == 2 ? 2 : 1;
    // full, (spare), empty [S]; acc_full, acc_empty [NUM_ACC]; drain (MMA
    // thread), drain (scale-copy threads) [SF_WARPS], scales ready [S]
    static constexpr int NUM_BARS = 4 * STAGES + 2 * NUM_ACC + 1 + SF_WARPS;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_GROUP = OFF_MISC + 16;  // row_off, tile_off, rt_off [E + 1]
    static constexpr int SMEM_BYTES = OFF_GROUP + 3 * (FP8G_MAX_EXPERTS + 1) * 4 + 1024;
    static constexpr uint32_t TX = kA + kB + CHUNK;            // bytes per CTA per stage
    // Scale columns of K group g of a stage: A's at g SFG .. + 3, B's 256 rows
    // at g SFG + SFB .. + 7 (FP8 / MXFP4: A 0-3, B 8-15, the second group 16
    // later; NVFP4: packed 12 per group)
    static constexpr int SFG = F4 == 2 ? 12 : 16;
    static constexpr int SFB = F4 == 2 ? 4 : 8;
    static constexpr int SF_COLS = kBlock ? G * SFG : 0;
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(SMEM_BYTES <= 232448, "shared memory over the per-CTA limit");
    static_assert(256 + STAGES * SF_COLS <= (int)TMEM_COLS || !kBlock, "tensor memory over budget");
    static_assert(OFF_SF % 128 == 0 && CHUNK % 128 == 0, "TMA destination alignment");
};
constexpr int kCW = kPairBN / 4;  // columns per epilogue warp


// Bounded wait with cluster-scope acquire (barriers remote CTAs arrive on).
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity,
                                                 volatile int *abort_flag, const GemmParams &p,
                                                 unsigned detail) {
    if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (ptx::mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            record_error(p, FP8G_ERR_TIMEOUT, detail);
            return false;
        }
    }
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t caddr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(caddr) : "memory");
    return v;
}

// One 256 x 256 output tile of a pair: rows [row0, row0 + 256) (the odd CTA
// takes the second 128), valid below row_end; columns [pn * 256, + 256);
// expert e; A's packed scale tiles from rtA0.
struct PairTile {
    int32_t row0, row_end, pm, pn, e, rtA0;
};

template <int MODE>
__device__ __forceinline__ PairTile pair_tile(int32_t t, const GemmParams &p, const int32_t *row_off,
                                              const int32_t *tile_off, const int32_t *rt_off) {
    PairTile ti;
    if constexpr (MODE == kModeGrouped) {
        int e = 0;
        while (tile_off[e + 1] <= t) ++e;
        const int32_t Me = row_off[e + 1] - row_off[e];
        raster(t - tile_off[e], (Me + 2 * kBM - 1) / (2 * kBM), p.npn, kRasterG, ti.pm, ti.pn);
        ti.row0 = row_off[e] + ti.pm * 2 * kBM;
        ti.row_end = row_off[e + 1];
        ti.e = e;
        ti.rtA0 = rt_off[e] + 2 * ti.pm;
    } else {
        raster(t, p.npm, p.npn, kRasterG, ti.pm, ti.pn);
        ti.row0 = ti.pm * 2 * kBM;
        ti.row_end = (int32_t)p.M;
        ti.e = 0;
        ti.rtA0 = 2 * ti.pm;
    }
    return ti;
}

template <int MODE, bool OUT_F32, int F4>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmSA,
                     const __grid_constant__ CUtensorMap tmSB, const GemmParams p) {
    using PC = PairCfg<MODE, F4>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = ptx::smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_rank();
    const bool leader = rank == 0;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + PC::OFF_BAR);
    auto bar_full = [&](int s) { return ptx::smem_addr(&bars[s]); };
    auto bar_peer = [&](int s) { return ptx::smem_addr(&bars[PC::STAGES + s]); };
    auto bar_empty = [&](int s) { return ptx::smem_addr(&bars[2 * PC::STAGES + s]); };
    auto bar_accf = [&](int a) { return ptx::smem_addr(&bars[3 * PC::STAGES + a]); };
    auto bar_acce = [&](int a) { return ptx::smem_addr(&bars[3 * PC::STAGES + PC::NUM_ACC + a]); };
    const uint32_t bar_drain = ptx::smem_addr(&bars[3 * PC::STAGES + 2 * PC::NUM_ACC]);
    auto bar_drain_sf = [&](int w) {
        return ptx::smem_addr(&bars[3 * PC::STAGES + 2 * PC::NUM_ACC + 1 + w]);
    };
    auto bar_sfr = [&](int s) {
        return ptx::smem_addr(&bars[3 * PC::STAGES + 2 * PC::NUM_ACC + 1 + PC::SF_WARPS + s]);
    };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + PC::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + PC::OFF_MISC + 4);
    int32_t *row_off = reinterpret_cast<int32_t *>(smem + PC::OFF_GROUP);
    int32_t *tile_off = row_off + (FP8G_MAX_EXPERTS + 1);
    int32_t *rt_off = tile_off + (FP8G_MAX_EXPERTS + 1);

    // ------------------------------------------------------------ setup
    if (threadIdx.x == 0) {
        for (int s = 0; s < PC::STAGES; ++s) {
            ptx::mbar_init(bar_full(s), 1);
            ptx::mbar_init(bar_peer(s), 1);
            ptx::mbar_init(bar_empty(s), 1);
            ptx::mbar_init(bar_sfr(s), PC::SF_WARPS);
        }
        for (int a = 0; a < PC::NUM_ACC; ++a) {
            ptx::mbar_init(bar_accf(a), 1);
            ptx::mbar_init(bar_acce(a), 2 * kEpiWarps);
        }
        ptx::mbar_init(bar_drain, 1);
        for (int w = 0; w < PC::SF_WARPS; ++w) ptx::mbar_init(bar_drain_sf(w), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        if constexpr (PC::kBlock) {
            ptx::prefetch_tmap(&tmSA);
            ptx::prefetch_tmap(&tmSB);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), PC::TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();  // both CTAs' barriers and tensor memory exist
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (threadIdx.x == 0) {
        // both CTAs must see the same accumulator columns
        const uint32_t other = ld_cluster_u32(ptx::map_shared(ptx::smem_addr(tmem_slot), rank ^ 1u));
        if (other != tmem_base) {
            record_error(p, FP8G_ERR_DEVICE, 0xA11Cu);
            *abort_flag = 1;
        }
    }
    ptx::grid_dep_wait();  // global memory only after the previous kernel
    ptx::grid_dep_launch();
    __syncthreads();
    const bool run = !*abort_flag;
    int32_t T = (int32_t)p.T;
    if constexpr (MODE == kModeGrouped) {
        grouped_prefix(p, 2 * kBM, row_off, tile_off, rt_off);
        T = tile_off[p.E];
    }
    const int32_t t_first = (int32_t)ptx::cluster_id_x();
    const int32_t t_step = (int32_t)ptx::num_clusters_x();

    if (run && warp == 0) {
        // ===== TMA producer (both CTAs): own 128 rows of A, own half of B =====
        // Both CTAs' copies complete on the even CTA's full barrier (TMA
        // cta_group::2), which expects both halves; the odd CTA does not arrive.
        if (lane == 0) {
            // F4 loads dense bytes; otherwise a packed (E2M1, FP6) operand's
            // tile load counts only its packed bytes
            const uint32_t tx_bytes =
                F4 ? PC::TX
                   : PC::TX - kA / 8 * (uint32_t)p.a_gap8 - kB / 8 * (uint32_t)p.b_gap8;
            const int32_t num_kg = PC::G * p.num_kb;  // K groups of the packed scales
            uint32_t stage = 0, phase = 0;
            for (int32_t t = t_first; t < T; t += t_step) {
                const PairTile ti = pair_tile<MODE>(t, p, row_off, tile_off, rt_off);
                const int32_t row0 = ti.row0 + (int32_t)rank * kBM;
                const int32_t nb0 = ti.pn * kPairBN + (int32_t)rank * (kPairBN / 2);
                if constexpr (MODE == kModeGrouped) {
                    if (leader && p.tile_map_out != nullptr)
                        *reinterpret_cast<int4 *>(p.tile_map_out + 4 * (int64_t)t) =
                            make_int4(ti.e, ti.pm, ti.pn, 0);
                }
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar(bar_empty(stage), phase ^ 1u, abort_flag, p, 0 * 256 + stage))
                        goto roles_done;
                    const uint32_t fb = leader ? bar_full(stage) : ptx::map_shared(bar_full(stage), 0);
                    if (leader) ptx::mbar_arrive_expect_tx(fb, 2 * tx_bytes);
                    // first K element of the stage: a 128-byte row holds 128 one-byte
                    // elements, or 32 fp32 ones (TF32)
                    const int32_t kx = F4 == 3 ? kb * (kBK / 4) : kb * kBK;
                    ptx::tma_load_2d_pair(sbase + PC::OFF_A + stage * kA, &tmA, fb, kx, row0);
                    if constexpr (MODE == kModeGrouped)
                        ptx::tma_load_3d_pair(sbase + PC::OFF_B + stage * kB, &tmB, fb, kx, nb0,
                                              ti.e);
                    else
                        ptx::tma_load_2d_pair(sbase + PC::OFF_B + stage * kB, &tmB, fb, kx, nb0);
                    if constexpr (PC::kBlock) {
                        // packed UE8M0 chunks (512-byte rows of the packed arrays):
                        // this CTA's 128 rows of A; the tile's 256 rows of B
                        // (G > 1: K groups G kb .. G kb + G - 1, A's chunks first,
                        // then B's pairs)
                        const uint32_t dst = sbase + PC::OFF_SF + stage * PC::CHUNK;
                        constexpr int G = PC::G;
                        if constexpr (F4 == 2) {
                            // NVFP4 chunks: a stage's 4 groups adjacent per 128-row
                            // tile: A's 4 chunks (2 KB), B's two tiles x 4 (4 KB)
                            ptx::tma_load_2d_pair(dst, &tmSA, fb, 0,
                                                  (kb * p.n_rtA + ti.rtA0 + (int32_t)rank) * 4);
                            // (B: expert e's chunks follow e whole matrices)
                            ptx::tma_load_2d_pair(dst + G * kSfaBytes, &tmSB, fb, 0,
                                                  ((ti.e * p.num_kb + kb) * p.n_rtB + 2 * ti.pn) * 4);
                        } else
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            const int32_t kg = G * kb + g;
                            ptx::tma_load_2d_pair(dst + g * kSfaBytes, &tmSA, fb, 0,
                                                  kg * p.n_rtA + ti.rtA0 + (int32_t)rank);
                            // B's chunks of pair tile pn: 128-row tiles 2 pn and 2 pn + 1
                            ptx::tma_load_2d_pair(dst + G * kSfaBytes + g * kSfbBytes, &tmSB, fb, 0,
                                                  (ti.e * num_kg + kg) * p.n_rtB + 2 * ti.pn);
                        }
                    }
                    if (++stage == PC::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (run && warp == 1 && leader) {
        // ===== MMA issuer (even CTA): 256 x 256 x 32 per instruction =====
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int32_t lt = 0;
            const uint32_t idesc = F4 == 3 ? ptx::idesc_tf32(2 * kBM, kPairBN)
                                           : ptx::idesc_f8(2 * kBM, kPairBN) | p.ab_fmt;
            for (int32_t t = t_first; t < T; t += t_step, ++lt) {
                const int acc = lt % PC::NUM_ACC;
                const uint32_t acc_par = (uint32_t)((lt / PC::NUM_ACC) & 1);
                const uint32_t d_tmem = tmem_base + acc * kPairBN;
                if (!wait_bar_cluster(bar_acce(acc), acc_par ^ 1u, abort_flag, p,
                                      1 * 256 + 64))
                    goto roles_done;
                ptx::tc_fence_after();
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    // block modes: data and scale factors in place (the
                    // scale-copy thread waited for "full" and committed its copies)
                    const uint32_t rb = PC::kBlock ? bar_sfr(stage) : bar_full(stage);
                    if (!wait_bar(rb, phase, abort_flag, p, 1 * 256 + stage)) goto roles_done;
                    ptx::tc_fence_after();
                    const uint32_t a0 = sbase + PC::OFF_A + stage * kA;
                    const uint32_t b0 = sbase + PC::OFF_B + stage * kB;
                    if constexpr (F4 == 2) {
                        // MMA k: K elements 64k .. 64k + 63 = K group k's four
                        // 16-wide scale blocks (the whole word, sf_id 0)
                        const uint32_t sf = tmem_base + 256 + stage * PC::SF_COLS;
#pragma unroll
                        for (int k = 0; k < kBK / 32; ++k) {
                            const uint32_t sfk = sf + PC::SFG * k;
                            ptx::mma_nvf4_pair(d_tmem, ptx::desc_kmajor_sw128(a0 + k * 32),
                                               ptx::desc_kmajor_sw128(b0 + k * 32),
                                               ptx::idesc_nvf4(2 * kBM, kPairBN), sfk,
                                               sfk + PC::SFB, (kb | k) != 0 ? 1u : 0u);
                        }
                    } else if constexpr (F4 == 1) {
                        // MMA k: K elements 64k .. 64k + 63 = scale blocks 2k, 2k + 1,
                        // in K group k / 2 (columns + 16 (k / 2)), bytes 2 (k % 2), + 1
                        const uint32_t sf = tmem_base + 256 + stage * PC::SF_COLS;
#pragma unroll
                        for (int k = 0; k < kBK / 32; ++k) {
                            const uint32_t sfk = sf + 16 * (k >> 1);
                            ptx::mma_mxf4_pair(d_tmem, ptx::desc_kmajor_sw128(a0 + k * 32),
                                               ptx::desc_kmajor_sw128(b0 + k * 32),
                                               ptx::idesc_mxf4(2 * kBM, kPairBN, 2u * (k & 1)),
                                               sfk, sfk + 8, (kb | k) != 0 ? 1u : 0u);
                        }
                    } else if constexpr (PC::kBlock) {
                        const uint32_t sf = tmem_base + 256 + stage * PC::SF_COLS;
#pragma unroll
                        for (int k = 0; k < kBK / 32; ++k)
                            ptx::mma_mxf8_pair(d_tmem, ptx::desc_kmajor_sw128(a0 + k * 32),
                                               ptx::desc_kmajor_sw128(b0 + k * 32),
                                               ptx::idesc_mxf8(2 * kBM, kPairBN, (uint32_t)k) | p.ab_fmt, sf,
                                               sf + 8, (kb | k) != 0 ? 1u : 0u);
                    } else if constexpr (F4 == 3) {
                        // TF32: 32 fp32 K values per 128-byte row, four K = 8 MMAs
#pragma unroll
                        for (int k = 0; k < kBK / 32; ++k)
                            ptx::mma_tf32_pair(d_tmem, ptx::desc_kmajor_sw128(a0 + k * 32),
                                               ptx::desc_kmajor_sw128(b0 + k * 32), idesc,
                                               (kb | k) != 0 ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int k = 0; k < kBK / 32; ++k)
                            ptx::mma_f8_pair(d_tmem, ptx::desc_kmajor_sw128(a0 + k * 32),
                                             ptx::desc_kmajor_sw128(b0 + k * 32), idesc,
                                             (kb | k) != 0 ? 1u : 0u);
                    }
                    ptx::tc_commit_pair_mc(bar_empty(stage), 0x3);
                    if (++stage == PC::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                ptx::tc_commit_pair_mc(bar_accf(acc), 0x3);
            }
        }
    } else if (run && warp >= 2 && warp < 2 + PC::SF_WARPS && leader && PC::kBlock) {
        // ===== scale-factor copies (even CTA, block modes) =====
        // Tensor-memory slot of a stage is rewritten only after "full" of its
        // next use, i.e. after the producer saw the MMAs that read it complete.
        // With two issuing warps, warp 2 + h copies K groups h G/2 .. and both
        // commit to the stage's "scales ready" barrier (arrival count 2).
        const int h = warp - 2;
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            for (int32_t t = t_first; t < T; t += t_step) {
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar(bar_full(stage), phase, abort_flag, p, 2 * 256 + stage))
                        goto roles_done;
                    ptx::tc_fence_after();
                    const uint32_t sf = tmem_base + 256 + stage * PC::SF_COLS;
                    const uint32_t cs = sbase + PC::OFF_SF + stage * PC::CHUNK;
                    constexpr int G = PC::G;
                    constexpr int GW = G / PC::SF_WARPS;  // groups per issuing warp
#pragma unroll
                    for (int gi = 0; gi < GW; ++gi) {
                        const int g = h * GW + gi;
                        // K group g: A's rows to columns SFG g + 0-3; B's rows
                        // 0-127 to SFG g + SFB + 0-3, rows 128-255 to the next
                        // four (each replicated over the lane quarters by the copy).
                        // Source chunks: B's rows 0-127 / 128-255 of group g at
                        // g * 1 KB and + 512 (NVFP4: g * 512 and 2 KB + g * 512)
                        const uint32_t sfg = sf + PC::SFG * g;
                        const uint32_t cb = cs + G * kSfaBytes;
                        const uint32_t b0 = F4 == 2 ? cb + g * 512 : cb + g * kSfbBytes;
                        const uint32_t b1 = F4 == 2 ? cb + G * 512 + g * 512 : b0 + 512;
                        ptx::tc_cp_32x128b_warpx4_pair(sfg, ptx::desc_sf_chunk(cs + g * kSfaBytes));
                        ptx::tc_cp_32x128b_warpx4_pair(sfg + PC::SFB, ptx::desc_sf_chunk(b0));
                        ptx::tc_cp_32x128b_warpx4_pair(sfg + PC::SFB + 4, ptx::desc_sf_chunk(b1));
                    }
                    ptx::tc_commit_pair_mc(bar_sfr(stage), 0x1);
                    if (++stage == PC::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (run && warp >= kEpiWarp0) {
        // ===== epilogue (both CTAs): this CTA's 128 rows of the 256 x 256 tile =====
        const int ew = warp - kEpiWarp0;
        const int q = warp & 3;
        const int col0 = (ew >> 2) * kCW;
        float alpha = 1.0f;
        // (TF32 operands already carry their scales)
        if constexpr (MODE == kModeTensor && F4 != 3) alpha = __fmul_rn(p.sa[0], p.sb[0]);
        if constexpr (F4 == 2) alpha = __fmul_rn(p.ga[0], p.gb[0]);  // NVFP4 tensor scales
        int32_t lt = 0;
        for (int32_t t = t_first; t < T; t += t_step, ++lt) {
            const PairTile ti = pair_tile<MODE>(t, p, row_off, tile_off, rt_off);
            const int acc = lt % PC::NUM_ACC;
            const uint32_t acc_par = (uint32_t)((lt / PC::NUM_ACC) & 1);
            // no back-off between polls: the next tile's first MMA waits for
            // this drain (8192^3 block-scaled kernel: 384 -> 380 us)
            if (!wait_bar_warp(bar_accf(acc), acc_par, abort_flag, p, 3 * 256 + acc, 0)) break;
            ptx::tc_fence_after();
            uint32_t r[kCW / 32][32];
            const uint32_t taddr =
                tmem_base + ((uint32_t)(q * 32) << 16) + acc * kPairBN + col0;
#pragma unroll
            for (int c = 0; c < kCW / 32; ++c) ptx::tmem_ld_32x32b_x32(taddr + c * 32, r[c]);
            ptx::tmem_ld_wait();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(ptx::map_shared(bar_acce(acc), 0));

            const int64_t arow = (int64_t)ti.row0 + rank * kBM + q * 32 + lane;  // routed row
            const int64_t row = arow < ti.row_end ? out_row(p, arow) : -1;       // row of C
            const int64_t ncol0 = (int64_t)ti.pn * kPairBN + col0;
            // NVFP4 grouped: each expert's B carries its own tensor scale
            float alpha_e = alpha;
            if constexpr (F4 == 2 && MODE == kModeGrouped) alpha_e = __fmul_rn(p.ga[0], p.gb[ti.e]);
            float a_t = alpha_e;  // scale left for the stores below
            if (p.bias != nullptr || p.act != FP8G_ACT_NONE) {
                // every lane (rows past the output too: they are not stored)
                const float *brow = p.bias != nullptr ? p.bias + (int64_t)ti.e * p.N : nullptr;
#pragma unroll
                for (int c = 0; c < kCW / 32; ++c)
                    epi32(r[c], alpha_e, brow, p.act, ncol0 + c * 32, p.N);
                a_t = 1.0f;
            }
            // FP4-rate tiles end twice as often: their stores go out as whole
            // 128-byte row segments (measured 8192^3: +1.8%; on the FP8-rate
            // tiles the shuffles cost more than the coalescing saves, -0.5%)
            if ((F4 == 1 || F4 == 2) && p.st32) {
                store_rows64<OUT_F32>(p.C, row, p.N, ncol0, r, a_t, lane);  // whole warp
            } else if (row >= 0) {
#pragma unroll
                for (int c = 0; c < kCW / 32; ++c)
                    store_row32<OUT_F32>(p.C, row, p.N, ncol0 + c * 32, r[c], a_t, p.st32 != 0);
            }
        }
    }

roles_done:
    __syncwarp();
    __syncthreads();
    if (*abort_flag) {
        // drain the tensor-core work each issuing thread may have in flight
        if (leader && (warp == 1 || (warp >= 2 && warp < 2 + PC::SF_WARPS && PC::kBlock)) &&
            lane == 0) {
            const uint32_t db = warp == 1 ? bar_drain : bar_drain_sf(warp - 2);
            ptx::tc_commit_pair(db);
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(db, 0) && ptx::globaltimer() - t0 < p.timeout_ns) {
            }
        }
        const uint64_t t0 = ptx::globaltimer();
        while (ptx::globaltimer() - t0 < 200000ull) {
        }
        __syncthreads();
    }
    // Neither CTA frees tensor memory (collectively) or leaves while the other
    // may still arrive on its barriers or its MMAs still run.
    ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, PC::TMEM_COLS);
    }
}

template <int MODE, bool OUT_F32, int F4 = 0>
cudaError_t launch_pair(const GemmMaps &maps, const GemmParams &p, int grid, cudaStream_t stream) {
    using PC = PairCfg<MODE, F4>;
    auto kern = gemm_pair_kernel<MODE, OUT_F32, F4>;
    static unsigned long long attr_done = 0ull;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if ((attr_done & bit) == 0ull) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PC::SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done |= bit;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = PC::SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, maps.A, maps.B, maps.SA, maps.SB, p);
}

}  // namespace

cudaError_t launch_gemm_pair(int mode, bool out_f32, const GemmMaps &maps, const GemmParams &p,
                             int grid, cudaStream_t stream) {
    if (p.f4 == 2 && mode == kModeBlock)
        return out_f32 ? launch_pair<kModeBlock, true, 2>(maps, p, grid, stream)
                       : launch_pair<kModeBlock, false, 2>(maps, p, grid, stream);
    if (p.f4 == 2 && mode == kModeGrouped)
        return out_f32 ? launch_pair<kModeGrouped, true, 2>(maps, p, grid, stream)
                       : launch_pair<kModeGrouped, false, 2>(maps, p, grid, stream);
    if (p.f4 == 1 && mode == kModeBlock)
        return out_f32 ? launch_pair<kModeBlock, true, 1>(maps, p, grid, stream)
                       : launch_pair<kModeBlock, false, 1>(maps, p, grid, stream);
    if (p.f4 == 1 && mode == kModeGrouped)
        return out_f32 ? launch_pair<kModeGrouped, true, 1>(maps, p, grid, stream)
                       : launch_pair<kModeGrouped, false, 1>(maps, p, grid, stream);
    if (p.f4 == 3 && mode == kModeTensor)
        return out_f32 ? launch_pair<kModeTensor, true, 3>(maps, p, grid, stream)
                       : launch_pair<kModeTensor, false, 3>(maps, p, grid, stream);
    if (p.f4) return cudaErrorInvalidValue;
    if (mode == kModeBlock)
        return out_f32 ? launch_pair<kModeBlock, true>(maps, p, grid, stream)
                       : launch_pair<kModeBlock, false>(maps, p, grid, stream);
    if (mode == kModeGrouped)
        return out_f32 ? launch_pair<kModeGrouped, true>(maps, p, grid, stream)
                       : launch_pair<kModeGrouped, false>(maps, p, grid, stream);
    return out_f32 ? launch_pair<kModeTensor, true>(maps, p, grid, stream)
                   : launch_pair<kModeTensor, false>(maps, p, grid, stream);
}

}  // namespace fp8g
