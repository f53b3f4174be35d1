// FP8 GEMM with arbitrary fp32 1x32 block scales, sm_103a.
//
//   C[i,j] = out( sum_kb sfa[i,kb] * sfb[j,kb] * P_kb[i,j] ),
//   P_kb[i,j] = sum_{k in kb} a_ik b_jk      (32-wide K blocks)
//
// The block-scaled MMA applies only 8-bit power-of-two exponents, so scales
// such as the literal fp32 quotient amax/448 ("fp32 scale = block amax/448")
// cannot ride on it.  Here the tensor core computes each K block's unscaled
// partial P_kb (one kind::f8f6f4 MMA, K = 32, written fresh into one of
// kPBufs tensor-memory buffers) and CUDA-core "promotion" warps scale and
// accumulate it in fp32 registers:  acc += fl32(sa * sb) * P_kb  (fma).  This
// is the promotion warp role of the warp-specialisation paragraph of the
// JAX/Blackwell FP8 page; its ceiling is the promotion arithmetic (two fp32
// operations per output element per K block), well below the MXFP8 path.
//
// Roles (640 threads): warp 0 TMA producer (A 128x128, B 128x128 codes and
// both operands' fp32 scales for the stage's 4 K blocks, one full barrier),
// warp 1 MMA issue, warps 4-19 promotion + epilogue (warp w: TMEM lane
// quarter w & 3, 32 columns (w - 4) >> 2).  A stage is free once its MMAs
// completed (commit) and all 16 promotion warps read its scales.  Every wait
// is bounded; tensor memory is freed on every exit path.
#include <cuda_bf16.h>

#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace fp8g {

namespace {

constexpr int kPThreads = 640;
constexpr int kPEpi0 = 4;
constexpr int kPEpiWarps = 16;
constexpr int kPBN = 128;
constexpr int kPStages = 6;
constexpr int kPBufs = 4;                   // partial-product buffers (128 columns each)
constexpr int kPA = kBM * kBK;              // 16 KB of A codes
constexpr int kPB = kPBN * kBK;             // 16 KB of B codes
constexpr int kPSA = kBM * 4 * 4;           // 2 KB: A's 128 rows x 4 K blocks, fp32
constexpr int kPSB = kPBN * 4 * 4;          // 2 KB: B's 128 rows x 4 K blocks
constexpr int kPStage = kPA + kPB + kPSA + kPSB;
constexpr int kPOffBar = kPStages * kPStage;
// full[S], empty[S], pfull[NB], pempty[NB], drain
constexpr int kPNumBars = 2 * kPStages + 2 * kPBufs + 1;
// per promotion warp: its 32 columns' B scales of the current stage,
// transposed to [K block][column] so a K block's 32 values are contiguous
constexpr int kPOffT = (kPOffBar + kPNumBars * 8 + 15) / 16 * 16;  // float4 reads
constexpr int kPOffMisc = kPOffT + kPEpiWarps * 4 * 32 * 4;
constexpr int kPSmem = kPOffMisc + 16 + 1024;  // + slack for 1024-byte alignment
constexpr uint32_t kPTmemCols = kPBufs * kPBN;
static_assert(kPSmem <= 232448, "shared memory over the per-CTA limit");
static_assert(kPStage % 1024 == 0, "swizzled tiles need 1024-byte aligned stages");
static_assert(kPTmemCols <= 512, "tensor memory over budget");
static_assert(kPOffT % 16 == 0 && kPOffMisc % 16 == 0, "16-byte aligned scratch");

template <bool OUT_F32>
__global__ void __launch_bounds__(kPThreads, 1)
    gemm_promote_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSA,
                        const __grid_constant__ CUtensorMap tmSB, const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = ptx::smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kPOffBar);
    auto bar_full = [&](int s) { return ptx::smem_addr(&bars[s]); };
    auto bar_empty = [&](int s) { return ptx::smem_addr(&bars[kPStages + s]); };
    auto bar_pfull = [&](int b) { return ptx::smem_addr(&bars[2 * kPStages + b]); };
    auto bar_pempty = [&](int b) { return ptx::smem_addr(&bars[2 * kPStages + kPBufs + b]); };
    const uint32_t bar_drain = ptx::smem_addr(&bars[2 * kPStages + 2 * kPBufs]);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kPOffMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kPOffMisc + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            ptx::mbar_init(bar_full(s), 1);
            ptx::mbar_init(bar_empty(s), 1 + kPEpiWarps);
        }
        for (int b = 0; b < kPBufs; ++b) {
            ptx::mbar_init(bar_pfull(b), 1);
            ptx::mbar_init(bar_pempty(b), kPEpiWarps);
        }
        ptx::mbar_init(bar_drain, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        ptx::prefetch_tmap(&tmSA);
        ptx::prefetch_tmap(&tmSB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kPTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::grid_dep_wait();  // global memory only after the previous kernel
    ptx::grid_dep_launch();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int32_t T = (int32_t)p.T;

    if (warp == 0) {
        // ===== TMA producer =====
        if (lane == 0) {
            const uint32_t tx_bytes =
                kPStage - kPA / 8 * (uint32_t)p.a_gap8 - kPB / 8 * (uint32_t)p.b_gap8;
            uint32_t stage = 0, phase = 0;
            for (int32_t t = blockIdx.x; t < T; t += gridDim.x) {
                int32_t pm, pn;
                raster(t, p.npm, p.npn, kRasterG, pm, pn);
                const int32_t row0 = pm * kBM, n0 = pn * kPBN;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar(bar_empty(stage), phase ^ 1u, abort_flag, p, 0 * 256 + stage))
                        goto roles_done;
                    const uint32_t fb = bar_full(stage);
                    const uint32_t st = sbase + stage * kPStage;
                    ptx::mbar_arrive_expect_tx(fb, tx_bytes);
                    ptx::tma_load_2d(st, &tmA, fb, kb * kBK, row0);
                    ptx::tma_load_2d(st + kPA, &tmB, fb, kb * kBK, n0);
                    ptx::tma_load_2d(st + kPA + kPB, &tmSA, fb, kb * 4, row0);
                    ptx::tma_load_2d(st + kPA + kPB + kPSA, &tmSB, fb, kb * 4, n0);
                    if (++stage == kPStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ===== MMA issue: one K = 32 MMA per K block, into a fresh buffer =====
        if (lane == 0) {
            const uint32_t idesc = ptx::idesc_f8(kBM, kPBN) | p.ab_fmt;
            uint32_t stage = 0, phase = 0, g = 0;
            for (int32_t t = blockIdx.x; t < T; t += gridDim.x) {
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bar(bar_full(stage), phase, abort_flag, p, 1 * 256 + stage))
                        goto roles_done;
                    ptx::tc_fence_after();
                    const uint32_t a0 = sbase + stage * kPStage;
                    const uint32_t b0 = a0 + kPA;
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k, ++g) {
                        const uint32_t buf = g % kPBufs;
                        if (!wait_bar(bar_pempty(buf), ((g / kPBufs) & 1u) ^ 1u, abort_flag, p,
                                      1 * 256 + 64 + buf))
                            goto roles_done;
                        ptx::tc_fence_after();
                        ptx::mma_f8(tmem_base + buf * kPBN, ptx::desc_kmajor_sw128(a0 + k * 32),
                                    ptx::desc_kmajor_sw128(b0 + k * 32), idesc, 0u);
                        ptx::tc_commit(bar_pfull(buf));
                    }
                    ptx::tc_commit(bar_empty(stage));
                    if (++stage == kPStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp >= kPEpi0) {
        // ===== promotion and epilogue =====
        const int ew = warp - kPEpi0;
        const int q = warp & 3;             // tensor-memory lane quarter: rows 32 q ..
        const int col0 = (ew >> 2) * 32;    // 32 columns of the 128
        const int r = q * 32 + lane;        // row in the tile
        float *sbt = reinterpret_cast<float *>(smem + kPOffT) + ew * 4 * 32;
        uint32_t stage = 0, phase = 0, g = 0;
        for (int32_t t = blockIdx.x; t < T; t += gridDim.x) {
            int32_t pm, pn;
            raster(t, p.npm, p.npn, kRasterG, pm, pn);
            float acc[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) acc[c] = 0.0f;
            bool ok = true;
            for (int kb = 0; kb < p.num_kb && ok; ++kb) {
                if (!wait_bar_warp(bar_full(stage), phase, abort_flag, p, 3 * 256 + stage)) {
                    ok = false;
                    break;
                }
                const float *sa_s = reinterpret_cast<const float *>(smem + stage * kPStage + kPA + kPB);
                const float *sb_s = sa_s + kBM * 4;
                {
                    // lane l: column col0 + l's 4 K blocks -> sbt[k][l]
                    const float4 v = *reinterpret_cast<const float4 *>(sb_s + (col0 + lane) * 4);
                    __syncwarp();  // the previous stage's reads of sbt are done
                    sbt[0 * 32 + lane] = v.x;
                    sbt[1 * 32 + lane] = v.y;
                    sbt[2 * 32 + lane] = v.z;
                    sbt[3 * 32 + lane] = v.w;
                    __syncwarp();
                }
#pragma unroll 1
                for (int k = 0; k < kBK / 32; ++k, ++g) {
                    const uint32_t buf = g % kPBufs;
                    if (!wait_bar_warp(bar_pfull(buf), (g / kPBufs) & 1u, abort_flag, p,
                                       3 * 256 + 64 + buf)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    uint32_t pv[32];
                    ptx::tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + buf * kPBN + col0,
                                            pv);
                    ptx::tmem_ld_wait();
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar_pempty(buf));
                    const float sa = sa_s[r * 4 + k];
                    const float4 *sbk = reinterpret_cast<const float4 *>(sbt + k * 32);
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 sb = sbk[c4];  // the same address in every lane: broadcast
                        acc[4 * c4 + 0] = __fmaf_rn(__fmul_rn(sa, sb.x), __uint_as_float(pv[4 * c4 + 0]),
                                                    acc[4 * c4 + 0]);
                        acc[4 * c4 + 1] = __fmaf_rn(__fmul_rn(sa, sb.y), __uint_as_float(pv[4 * c4 + 1]),
                                                    acc[4 * c4 + 1]);
                        acc[4 * c4 + 2] = __fmaf_rn(__fmul_rn(sa, sb.z), __uint_as_float(pv[4 * c4 + 2]),
                                                    acc[4 * c4 + 2]);
                        acc[4 * c4 + 3] = __fmaf_rn(__fmul_rn(sa, sb.w), __uint_as_float(pv[4 * c4 + 3]),
                                                    acc[4 * c4 + 3]);
                    }
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar_empty(stage));
                if (++stage == kPStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            // ----- store: out(act(fl32(acc + bias))) -----
            const int64_t row = (int64_t)pm * kBM + r;
            const int64_t ncol0 = (int64_t)pn * kPBN + col0;
            if (row < p.M) {
                if (p.bias != nullptr || p.act != FP8G_ACT_NONE) {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (ncol0 + c < p.N) acc[c] = epi1(acc[c], p.bias, p.act, ncol0 + c);
                }
                if constexpr (OUT_F32) {
                    float *out = reinterpret_cast<float *>(p.C) + row * p.N + ncol0;
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        if (ncol0 + v * 4 < p.N)
                            *reinterpret_cast<float4 *>(out + v * 4) =
                                make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
                } else {
                    __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(p.C) + row * p.N + ncol0;
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        if (ncol0 + v * 8 < p.N) {
                            uint32_t pk[4];
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                __nv_bfloat162 b2 =
                                    __floats2bfloat162_rn(acc[8 * v + 2 * h], acc[8 * v + 2 * h + 1]);
                                pk[h] = *reinterpret_cast<uint32_t *>(&b2);
                            }
                            *reinterpret_cast<uint4 *>(out + v * 8) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        }
                }
            }
        }
    }

roles_done:
    __syncwarp();
    __syncthreads();
    if (*abort_flag) {
        // Drain: wait (bounded) for this CTA's MMAs, then give in-flight TMA
        // copies a bounded grace period before shared memory is released.
        if (warp == 1 && lane == 0) {
            ptx::tc_commit(bar_drain);
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(bar_drain, 0) && ptx::globaltimer() - t0 < p.timeout_ns) {
            }
        }
        const uint64_t t0 = ptx::globaltimer();
        while (ptx::globaltimer() - t0 < 200000ull) {
        }
        __syncthreads();
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, kPTmemCols);
    }
}

template <bool OUT_F32>
cudaError_t launch_promote_t(const GemmMaps &maps, const GemmParams &p, int grid,
                             cudaStream_t stream) {
    auto kern = gemm_promote_kernel<OUT_F32>;
    static unsigned long long attr_done = 0ull;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if ((attr_done & bit) == 0ull) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
        if (e != cudaSuccess) return e;
        attr_done |= bit;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kPThreads, 1, 1);
    cfg.dynamicSmemBytes = kPSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, maps.A, maps.B, maps.SA, maps.SB, p);
}

}  // namespace

cudaError_t launch_gemm_promote(bool out_f32, const GemmMaps &maps, const GemmParams &p, int grid,
                                cudaStream_t stream) {
    return out_f32 ? launch_promote_t<true>(maps, p, grid, stream)
                   : launch_promote_t<false>(maps, p, grid, stream);
}

}  // namespace fp8g
