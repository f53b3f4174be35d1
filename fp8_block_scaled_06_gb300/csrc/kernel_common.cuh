// Device helpers shared by the GEMM kernels: the grouped raster order of
// output tiles and the bounded mbarrier waits with their error reporting.
#pragma once
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fp8g {

// Grouped raster order: bands of G tile-rows; inside a band walk down one
// tile-column, then move to the next column.  (Tile counts fit in 31 bits.)
__device__ __forceinline__ void raster(int32_t t, int32_t npm, int32_t npn, int32_t G, int32_t &pm,
                                       int32_t &pn) {
    const int32_t band = G * npn;
    const int32_t grp = t / band;
    const int32_t first = grp * G;
    const int32_t height = min(npm - first, G);
    const int32_t in_band = t - grp * band;
    pm = first + in_band % height;
    pn = in_band / height;
}

// UE8M0 code of an fp32 block scale: a positive power of two's code is its
// exponent field (lossless).  A NaN scale gives the NaN code 0xFF; any other
// scale that is not a positive normal power of two sets `bad`.
__device__ __forceinline__ uint32_t ue8m0_code(uint32_t bits, bool &bad) {
    const uint32_t ex = (bits >> 23) & 0xFFu;
    const uint32_t man = bits & 0x7FFFFFu;
    if (ex == 0xFFu && man != 0u) return 0xFFu;
    if ((bits >> 31) != 0u || man != 0u || ex == 0u || ex == 0xFFu) bad = true;
    return ex;
}

__device__ __forceinline__ void record_error(const GemmParams &p, unsigned code, unsigned detail) {
    if (atomicCAS(&p.status[0], 0u, code) == 0u) atomicExch(&p.status[1], detail);
}

// Bounded wait on an mbarrier phase.  Returns false when this CTA is aborting
// (another role timed out) or when this wait itself exceeded the limit.
// sleep_ns > 0 backs off between polls (for roles that wait a whole tile).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         const GemmParams &p, unsigned detail,
                                         uint32_t sleep_ns = 0) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            record_error(p, FP8G_ERR_TIMEOUT, detail);
            return false;
        }
        if (sleep_ns) __nanosleep(sleep_ns);
    }
}

// Bounded wait that does not give up when the CTA is aborting: for copies
// that other CTAs make into this CTA's shared memory, which must have landed
// before the CTA may exit.  Returns false only when the limit expired.
__device__ __forceinline__ bool wait_bar_landed(uint32_t bar, uint32_t parity,
                                                volatile int *abort_flag, const GemmParams &p,
                                                unsigned detail) {
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            record_error(p, FP8G_ERR_TIMEOUT, detail);
            return false;
        }
    }
    return true;
}

// Warp-uniform bounded wait: lane 0 waits, the outcome is broadcast, and the
// warp re-converges before any .sync.aligned tcgen05 instruction follows.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity,
                                              volatile int *abort_flag, const GemmParams &p,
                                              unsigned detail, uint32_t sleep_ns = 0) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort_flag, p, detail, sleep_ns) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

__device__ __forceinline__ bool wait_bar_landed_warp(uint32_t bar, uint32_t parity,
                                                     volatile int *abort_flag,
                                                     const GemmParams &p, unsigned detail) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = wait_bar_landed(bar, parity, abort_flag, p, detail) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

// Row of C that routed row `row` is stored to: c_row_of[row] when scattering
// (grouped GEMM), else `row`.  An index outside [0, c_rows) records
// FP8G_ERR_INVALID_ARG (detail: row) and returns -1 (the row is not stored).
__device__ __forceinline__ int64_t out_row(const GemmParams &p, int64_t row) {
    if (p.c_row_of == nullptr) return row;
    const int64_t c = __ldg(p.c_row_of + row);
    if (c < 0 || c >= p.c_rows) {
        record_error(p, FP8G_ERR_INVALID_ARG, (unsigned)row);
        return -1;
    }
    return c;
}

// Fused epilogue on one output value of column `col`:
//   v = act(fl32(v + bias[col]))   (bias row may be null; act FP8G_ACT_*)
// applied after the per-tensor scale and before the output rounding.  ReLU
// keeps NaN (v < 0 ? 0 : v); GELU is the erf form 0.5 v (1 + erf(v / sqrt 2)).
__device__ __forceinline__ float epi1(float v, const float *brow, int act, int64_t col) {
    if (brow != nullptr) v = __fadd_rn(v, __ldg(brow + col));
    if (act == FP8G_ACT_RELU) {
        v = v < 0.0f ? 0.0f : v;
    } else if (act == FP8G_ACT_GELU) {
        v = 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
    }
    return v;
}

// The fused epilogue in place on 32 consecutive accumulator columns
// [col0, col0 + 32) held as fp32 bit patterns (columns >= N are skipped; they
// are never stored): r = act(fl32(fl32(alpha * r) + bias)).
__device__ __forceinline__ void epi32(uint32_t (&r)[32], float alpha, const float *brow, int act,
                                      int64_t col0, int64_t N) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
        if (col0 + i < N)
            r[i] = __float_as_uint(epi1(__fmul_rn(alpha, __uint_as_float(r[i])), brow, act, col0 + i));
}

// Grouped GEMM problem list, computed by every CTA from the device counts:
// row_off[e] = first row of expert e (exclusive prefix of counts), tile_off[e]
// = first output tile of expert e (experts in index order, ceil(M_e/bm) *
// npn tiles each), rt_off[e] = first 128-row tile of expert e in the packed
// scale layout of A.  Negative counts or a sum other than total_rows record
// FP8G_ERR_INVALID_ARG (once, CTA 0) and give zero tiles.  CTA 0 also writes
// offsets_out.  Call with all threads; ends with __syncthreads.
__device__ __forceinline__ void grouped_prefix(const GemmParams &p, int bm, int32_t *row_off,
                                               int32_t *tile_off, int32_t *rt_off) {
    if (threadIdx.x < FP8G_MAX_EXPERTS)
        tile_off[threadIdx.x] = threadIdx.x < p.E ? p.counts[threadIdx.x] : 0;
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t r = 0, tt = 0;
        bool bad = false;
        int32_t cnt[FP8G_MAX_EXPERTS];
        for (int e = 0; e < p.E; ++e) {
            cnt[e] = tile_off[e];
            if (cnt[e] < 0) bad = true;
        }
        row_off[0] = 0;
        for (int e = 0; e < p.E; ++e) {
            const int32_t c = max(cnt[e], 0);
            r += c;
            row_off[e + 1] = (int32_t)(r < (int64_t)INT32_MAX ? r : (int64_t)INT32_MAX);
        }
        if (bad || r != p.M) {
            bad = true;
            if (blockIdx.x == 0) record_error(p, FP8G_ERR_INVALID_ARG, 1);
        }
        tile_off[0] = 0;
        rt_off[0] = 0;
        for (int e = 0; e < p.E; ++e) {
            const int64_t Me = bad ? 0 : (row_off[e + 1] - row_off[e]);
            tt += ((Me + bm - 1) / bm) * (int64_t)p.npn;
            tile_off[e + 1] = (int32_t)tt;
            // packed scale row tiles of A: counted as the packing kernel does
            rt_off[e + 1] = rt_off[e] + (max(cnt[e], 0) + kBM - 1) / kBM;
        }
        if (blockIdx.x == 0 && p.offsets_out != nullptr)
            for (int e = 0; e <= p.E; ++e) p.offsets_out[e] = row_off[e];
    }
    __syncthreads();
}

// Columns ncol .. ncol + 31 of row `row` of C (row stride N) from 32 fp32
// accumulator words times a_t, bf16 (RNE) or fp32, none at or past column N
// (N is a multiple of 8 / 4 elements and ncol of 32, so every store is
// whole).  wide: 32-byte stores, each a whole L2 sector (C 32-byte aligned,
// rows a multiple of 32 bytes); otherwise 16-byte stores.  With one row per
// lane a warp's store touches 32 rows: 16-byte stores leave every sector
// half-written and double the L2 write requests, which the concurrent TMA
// operand loads of the next tile then queue behind.
template <bool OUT_F32>
__device__ __forceinline__ void store_row32(void *C, int64_t row, int64_t N, int64_t ncol,
                                            const uint32_t (&r)[32], float a_t, bool wide) {
    if constexpr (OUT_F32) {
        float *out = reinterpret_cast<float *>(C) + row * N + ncol;
        uint32_t o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__fmul_rn(a_t, __uint_as_float(r[i])));
        if (wide) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
                if (ncol + v * 8 < N) ptx::st_global_v8(out + v * 8, o + 8 * v);
        } else {
#pragma unroll
            for (int v = 0; v < 8; ++v)
                if (ncol + v * 4 < N)
                    *reinterpret_cast<uint4 *>(out + v * 4) =
                        make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
        }
    } else {
        __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(C) + row * N + ncol;
        uint32_t pk[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
            const float lo = __fmul_rn(a_t, __uint_as_float(r[2 * h]));
            const float hi = __fmul_rn(a_t, __uint_as_float(r[2 * h + 1]));
            __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
            pk[h] = *reinterpret_cast<uint32_t *>(&b2);
        }
        if (wide) {
#pragma unroll
            for (int v = 0; v < 2; ++v)
                if (ncol + v * 16 < N) ptx::st_global_v8(out + v * 16, pk + 8 * v);
        } else {
#pragma unroll
            for (int v = 0; v < 4; ++v)
                if (ncol + v * 8 < N)
                    *reinterpret_cast<uint4 *>(out + v * 8) =
                        make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
    }
}

// Quad transpose of 32-byte chunks: lane 4q + p holds the 4 chunks (8 words
// each, w[8c .. 8c + 7]) of one row segment; afterwards slot t holds chunk p
// of lane 4q + t's segment.  Two xor-shuffle exchanges of the off-diagonal
// halves: 2 x 2 blocks of chunks with lane ^ 2, then single chunks with
// lane ^ 1.
__device__ __forceinline__ void quad_transpose(uint32_t (&w)[32], int lane) {
    const bool hi = (lane & 2) != 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const uint32_t send = hi ? w[j] : w[16 + j];
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 2);
        if (hi)
            w[j] = recv;
        else
            w[16 + j] = recv;
    }
    const bool odd = (lane & 1) != 0;
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t send = odd ? w[16 * k + i] : w[16 * k + 8 + i];
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
            if (odd)
                w[16 * k + i] = recv;
            else
                w[16 * k + 8 + i] = recv;
        }
}

// Whole warp: lane L's 128-byte row segment (w, 32 words) goes to seg (null:
// a row past the output, nothing stored; 32-byte aligned).  After
// quad_transpose, store step t has lane 4q + p write chunk p of lane
// 4q + t's segment, so each store instruction writes eight whole 128-byte
// segments instead of 32 sectors of 32 different rows.  chunk_ok: chunk p of
// every segment lies inside the row (the same columns for every row).
__device__ __forceinline__ void store_seg128(uint8_t *seg, uint32_t (&w)[32], int lane,
                                             bool chunk_ok) {
    quad_transpose(w, lane);
    const int p = lane & 3;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        uint8_t *dst = reinterpret_cast<uint8_t *>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(seg), (lane & ~3) | t));
        if (dst != nullptr && chunk_ok) ptx::st_global_v8(dst + 32 * p, w + 8 * t);
    }
}

// Whole warp, one row per lane (row < 0: past the output): columns
// ncol .. ncol + 63 of C from 64 fp32 accumulator words (r[0], r[1]) times
// a_t, as 128-byte segments through store_seg128 (bf16: one segment, fp32:
// two).  C 32-byte aligned with rows a multiple of 32 bytes; ncol a multiple
// of 64; columns at or past N (a multiple of 16 / 8) are not written.
template <bool OUT_F32>
__device__ __forceinline__ void store_rows64(void *C, int64_t row, int64_t N, int64_t ncol,
                                             const uint32_t (&r)[2][32], float a_t, int lane) {
    const int p = lane & 3;
    if constexpr (OUT_F32) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
                w[i] = __float_as_uint(__fmul_rn(a_t, __uint_as_float(r[c][i])));
            uint8_t *seg = row >= 0 ? reinterpret_cast<uint8_t *>(
                                          reinterpret_cast<float *>(C) + row * N + ncol + 32 * c)
                                    : nullptr;
            store_seg128(seg, w, lane, ncol + 32 * c + 8 * p < N);
        }
    } else {
        uint32_t w[32];
#pragma unroll
        for (int h = 0; h < 32; ++h) {
            const uint32_t *src = r[h >> 4];
            const float lo = __fmul_rn(a_t, __uint_as_float(src[(2 * h) & 31]));
            const float hi = __fmul_rn(a_t, __uint_as_float(src[(2 * h + 1) & 31]));
            __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
            w[h] = *reinterpret_cast<uint32_t *>(&b2);
        }
        uint8_t *seg = row >= 0 ? reinterpret_cast<uint8_t *>(
                                      reinterpret_cast<__nv_bfloat16 *>(C) + row * N + ncol)
                                : nullptr;
        store_seg128(seg, w, lane, ncol + 16 * p < N);
    }
}

}  // namespace fp8g
