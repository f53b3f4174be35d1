// Operand quantiser: fp32 -> FP8 / FP4 codes + fp32 scales (data preparation
// for the GEMM entry points).  Formats: E4M3 (largest finite fmax = 448) and
// E5M2 (fmax = 57344), the two FP8 formats of the format paragraph of
// "Optimizing FP8 GEMM kernels in JAX with Triton for Blackwell GPUs", and
// E2M1 (fmax = 6, two codes per byte, the first in the low nibble), the FP4
// element of the micro-scaling formats of the Triton tutorial ch. 12, 12.6.1,
// and the FP6 elements E2M3 (fmax = 7.5) and E3M2 (fmax = 28), the tensor
// core's FP6 types of that page's 12.6.1 table (four codes per three bytes,
// code i in bits 6i .. 6i+5 of a little-endian bit string).
//
// Per-tensor: s = fl32(amax / fmax) over the non-NaN |x| (1 if that is 0).
// 1x32 block along the contiguous axis: s = the smallest power of two with
// fmax s >= block amax, so every |x / s| <= fmax and the scale is exactly an
// 8-bit exponent (UE8M0) — the microscaling form of the parameter paragraph of
// the same page and the MXFP8 micro-scaling of the Triton tutorial ch. 12,
// 12.6.1; its "fine-grained quantisation" advice against FP8 underflow is the
// reason for the block form.  q = FP8(fl32(x / s)), round to nearest even,
// saturating (cvt ... satfinite), NaN -> 0x7F (a NaN code in both FP8
// formats; E2M1 has none and takes +6, FP6 its largest value, code 0x1F).
//
// The source is fp32 or bf16 (activations; widened exactly), and the output
// rows may gather source rows through an index list (the routing step of the
// MoE paragraph of the JAX/Blackwell page: tokens copied into expert order),
// so that gather, scale and quantisation take one pass over HBM.
//
// NVFP4 (the other FP4 micro-scaling format of 12.6.1): E2M1 codes, one E4M3
// scale per 1x16 block and an fp32 scale per tensor (quant_nvfp4_kernel; the
// recipe is stated there).
//
// HBM-bound elementwise kernels: 16-byte loads, 8-byte (E2M1: 4-byte; FP6:
// three 2-byte) stores, a grid of a few CTAs per SM striding over the output.
#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8g {

namespace {

// Store the codes of group g (values 8g .. 8g+7 of the output): 8 bytes
// (FP8), 4 bytes (E2M1) or 6 bytes (FP6: the eight six-bit codes as a 48-bit
// little-endian string) at g times that size.
template <int FMT>
__device__ __forceinline__ void store8(uint8_t *q, int64_t g, uint2 o) {
    if constexpr (FMT == 2) {
        reinterpret_cast<uint32_t *>(q)[g] = o.x | (o.y << 16);
    } else if constexpr (FMT >= 3) {
        uint64_t v = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v |= (uint64_t)((o.x >> (8 * i)) & 0x3Fu) << (6 * i);
            v |= (uint64_t)((o.y >> (8 * i)) & 0x3Fu) << (24 + 6 * i);
        }
        uint16_t *p = reinterpret_cast<uint16_t *>(q + 6 * g);  // 2-byte aligned
        p[0] = (uint16_t)v;
        p[1] = (uint16_t)(v >> 16);
        p[2] = (uint16_t)(v >> 32);
    } else {
        reinterpret_cast<uint2 *>(q)[g] = o;
    }
}

// 8 values -> their codes (first four in .x), for store8.
template <int FMT>
__device__ __forceinline__ uint2 quant8(const float4 a, const float4 b, float s) {
    uint2 o;
    o.x = fp8x4<FMT>(__fdiv_rn(a.x, s), __fdiv_rn(a.y, s), __fdiv_rn(a.z, s), __fdiv_rn(a.w, s));
    o.y = fp8x4<FMT>(__fdiv_rn(b.x, s), __fdiv_rn(b.y, s), __fdiv_rn(b.z, s), __fdiv_rn(b.w, s));
    return o;
}

// Output row r reads source row rows[r] (rows == null: row r).  A source row
// outside [0, x_rows) records FP8G_ERR_INVALID_ARG (detail: r) and reads as
// zeros; nothing outside the source is read.
struct RowMap {
    const void *x;
    const int32_t *rows;
    int64_t x_rows, cols;
    unsigned int *status;
};

__device__ __forceinline__ int64_t src_row(const RowMap &m, int64_t r, bool &ok) {
    const int64_t s = m.rows != nullptr ? (int64_t)__ldg(m.rows + r) : r;
    ok = s >= 0 && s < m.x_rows;
    return ok ? s : 0;
}

__device__ __forceinline__ void bad_row(const RowMap &m, int64_t r) {
    if (atomicCAS(&m.status[0], 0u, (unsigned)FP8G_ERR_INVALID_ARG) == 0u)
        atomicExch(&m.status[1], (unsigned)r);
}

// Work layout: CTAs stride over output rows; within a row the CTA's threads
// take groups of 8 consecutive values (g and g + blockDim.x per pass, both
// loads issued before either is used).  A 1x32 block is 4 consecutive groups,
// held by 4 consecutive lanes (blockDim.x and cols / 8 are multiples of 4), so
// its amax is two shuffles; lanes past the row's end stay in the pass
// (inactive) until the whole warp is done, so the shuffles always see all 32
// lanes.  (Measured on 8192 x 8192: one warp per row with 4-8 groups in
// flight per lane was 10-30% slower.)
constexpr int kQThreads = 256;

// LITERAL: s = fl32(amax / fmax) (1 when that is 0) and q = FP8(fl32(x / s)),
// instead of the power-of-two scale.
template <int FMT, bool BF16, bool LITERAL>
__global__ void __launch_bounds__(kQThreads) quant_block32_kernel(RowMap m, int64_t n_rows,
                                                                 uint8_t *__restrict__ q,
                                                                 float *__restrict__ scales) {
    // launched programmatically: global memory only after the previous kernel
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();  // a GEMM's scale packing may be placed now
    constexpr int U = 2;  // groups per thread and pass
    const int64_t gpr = m.cols / 8;  // groups of 8 per row
    const int64_t wbase = threadIdx.x & ~31;
    for (int64_t r = blockIdx.x; r < n_rows; r += gridDim.x) {
        bool ok;
        const int64_t sr = src_row(m, r, ok);
        if (!ok && threadIdx.x == 0) bad_row(m, r);
        const int64_t in0 = sr * m.cols, out0 = r * gpr;
        for (int64_t c0 = wbase; c0 < gpr; c0 += U * kQThreads) {
            float4 a[U], b[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (threadIdx.x & 31) + u * kQThreads;
                a[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                b[u] = a[u];
                if (ok && c < gpr) load8<BF16>(m.x, in0 + c * 8, a[u], b[u]);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + (threadIdx.x & 31) + u * kQThreads;
                float am = absmax8(a[u], b[u]);
                am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
                am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
                float sc;
                if constexpr (LITERAL) {
                    sc = __fdiv_rn(am, Fp8Fmt<FMT>::kMax);
                    if (sc == 0.0f) sc = 1.0f;
                } else {
                    sc = pow2_scale<FMT>(am);
                }
                if (c < gpr) {
                    store8<FMT>(q, out0 + c,
                                LITERAL ? quant8<FMT>(a[u], b[u], sc)
                                        : quant8_pow2<FMT>(a[u], b[u], sc));
                    if ((c & 3) == 0) scales[(out0 + c) >> 2] = sc;
                }
            }
        }
    }
}

template <bool BF16>
__global__ void __launch_bounds__(kQThreads) amax_kernel(RowMap m, int64_t n_rows,
                                                        unsigned int *__restrict__ out) {
    const int64_t gpr = m.cols / 8;
    float am = 0.0f;
    for (int64_t r = blockIdx.x; r < n_rows; r += gridDim.x) {
        bool ok;
        const int64_t sr = src_row(m, r, ok);
        if (!ok) {
            if (threadIdx.x == 0) bad_row(m, r);
            continue;  // block-uniform
        }
        for (int64_t c = threadIdx.x; c < gpr; c += kQThreads) {
            float4 a, b;
            load8<BF16>(m.x, sr * m.cols + c * 8, a, b);
            am = fmaxf(am, absmax8(a, b));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    // non-negative floats order like their bit patterns
    if ((threadIdx.x & 31) == 0) atomicMax(out, __float_as_uint(am));
}

template <int FMT>
__device__ __forceinline__ float tensor_scale(const float *amax_slot) {
    const float amax = *amax_slot;
    float s = __fdiv_rn(amax, Fp8Fmt<FMT>::kMax);
    if (s == 0.0f) s = 1.0f;
    return s;
}

// the scale slot still holds amax
template <int FMT, bool BF16>
__global__ void __launch_bounds__(kQThreads) quant_tensor_kernel(RowMap m, int64_t n_rows,
                                                                uint8_t *__restrict__ q,
                                                                const float *__restrict__ amax_slot) {
    const float s = tensor_scale<FMT>(amax_slot);
    const int64_t gpr = m.cols / 8;
    for (int64_t r = blockIdx.x; r < n_rows; r += gridDim.x) {
        bool ok;
        const int64_t sr = src_row(m, r, ok);
        for (int64_t c = threadIdx.x; c < gpr; c += kQThreads) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (ok) load8<BF16>(m.x, sr * m.cols + c * 8, a, b);
            store8<FMT>(q, r * gpr + c, quant8<FMT>(a, b, s));
        }
    }
}

template <int FMT>
__global__ void finish_scale_kernel(float *slot) { *slot = tensor_scale<FMT>(slot); }

// ---------------------------------------------------------------- NVFP4
// E4M3 value of a non-negative code (0x7F: NaN), from its bit fields.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    if (c == 0x7Fu) return __int_as_float(0x7FC00000);
    return e == 0 ? (float)m * 0.001953125f : __int_as_float((int)((e + 120u) << 23 | m << 20));
}

// g = fl32(amax / 2688) (2688 = 6 x 448), 1 when that is 0.
__device__ __forceinline__ float nvfp4_g(const float *amax_slot) {
    float g = __fdiv_rn(*amax_slot, 2688.0f);
    if (g == 0.0f) g = 1.0f;
    return g;
}

// NVFP4: a 1x16 block is two groups of 8 held by two consecutive lanes.  Per
// block t = fl32(amax_b / fl32(6 g)), s = E4M3(t) (RNE, saturating), d =
// fl32(dec(s) g), codes E2M1(fl32(x / d)) (all 0 when d is not positive).
// q: two codes per byte [rows, cols/2]; sf: one E4M3 code per block
// [rows, cols/16]; the slot still holds the tensor's amax.
template <bool BF16>
__global__ void __launch_bounds__(kQThreads) quant_nvfp4_kernel(RowMap m, int64_t n_rows,
                                                               uint8_t *__restrict__ q,
                                                               uint8_t *__restrict__ sf,
                                                               const float *amax_slot) {
    const float g = nvfp4_g(amax_slot);
    const float g6 = __fmul_rn(6.0f, g);
    const int64_t gpr = m.cols / 8;  // groups of 8 per row
    const int64_t wbase = threadIdx.x & ~31;
    for (int64_t r = blockIdx.x; r < n_rows; r += gridDim.x) {
        bool ok;
        const int64_t sr = src_row(m, r, ok);
        const int64_t in0 = sr * m.cols, out0 = r * gpr;
        for (int64_t c0 = wbase; c0 < gpr; c0 += kQThreads) {
            const int64_t c = c0 + (threadIdx.x & 31);
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (ok && c < gpr) load8<BF16>(m.x, in0 + c * 8, a, b);
            float am = absmax8(a, b);
            am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
            uint16_t sc;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(sc) : "f"(0.0f), "f"(__fdiv_rn(am, g6)));
            const uint32_t s = sc & 0xFFu;
            const float d = __fmul_rn(e4m3_value(s), g);
            uint2 o = make_uint2(0u, 0u);
            if (d > 0.0f) o = quant8<2>(a, b, d);
            if (c < gpr) {
                store8<2>(q, out0 + c, o);
                if ((c & 1) == 0) sf[(out0 + c) >> 1] = (uint8_t)s;
            }
        }
    }
}

__global__ void finish_nvfp4_kernel(float *slot) { *slot = nvfp4_g(slot); }

// ------------------------------------------------- literal scales -> TF32
// Value of an FP8 code from its bit fields: E4M3 (bias 7, subnormals m 2^-9,
// S.1111.111 NaN) or E5M2 (bias 15, subnormals m 2^-16, exponent 31: inf for
// m = 0, else NaN).
template <int FMT>
__device__ __forceinline__ float fp8_value(uint32_t c) {
    const uint32_t sign = (c & 0x80u) << 24;
    if constexpr (FMT == 0) {
        const uint32_t e = (c >> 3) & 15u, m = c & 7u;
        if (e == 15u && m == 7u) return __uint_as_float(sign | 0x7FC00000u);
        if (e == 0u) return __uint_as_float(sign | __float_as_uint((float)m * 0.001953125f));
        return __uint_as_float(sign | (e + 120u) << 23 | m << 20);
    } else {
        const uint32_t e = (c >> 2) & 31u, m = c & 3u;
        if (e == 31u) return __uint_as_float(sign | (m == 0u ? 0x7F800000u : 0x7FC00000u));
        if (e == 0u) return __uint_as_float(sign | __float_as_uint((float)m * 1.52587890625e-5f));
        return __uint_as_float(sign | (e + 112u) << 23 | m << 21);
    }
}

__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// out = TF32(fl32(dec(a) s)) for 8 consecutive codes per thread (one 8-byte
// load, two 16-byte stores; the 8 share one 1x32 block scale).  HBM-bound.
template <int FMT>
__global__ void __launch_bounds__(256) dequant_tf32_kernel(const uint8_t *__restrict__ a,
                                                          const float *__restrict__ s,
                                                          int64_t rows, int64_t K,
                                                          float *__restrict__ out) {
    const int64_t gpr = K / 8;  // groups of 8 per row
    const int64_t n = rows * gpr;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < n;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = g / gpr, c = g - r * gpr;
        const uint2 q = __ldg(reinterpret_cast<const uint2 *>(a) + g);
        const float sc = __ldg(s + r * (K / 32) + c / 4);
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t code = ((i < 4 ? q.x : q.y) >> (8 * (i & 3))) & 0xFFu;
            v[i] = to_tf32(__fmul_rn(fp8_value<FMT>(code), sc));
        }
        float4 *o = reinterpret_cast<float4 *>(out) + 2 * g;
        o[0] = make_float4(v[0], v[1], v[2], v[3]);
        o[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
}

}  // namespace

namespace {

template <int FMT, bool BF16>
cudaError_t launch_rows(const RowMap &m, int64_t n_rows, int32_t block, uint8_t *q, float *scales,
                        int num_sms, cudaStream_t s) {
    if (n_rows == 0 || m.cols == 0) return cudaSuccess;
    const int64_t cap = (int64_t)num_sms * 8;  // 8 CTAs of 256 threads per SM
    const unsigned blocks = (unsigned)(n_rows < cap ? n_rows : cap);
    if (block == 32)
        return launch_programmatic(quant_block32_kernel<FMT, BF16, false>, dim3(blocks),
                                   dim3(kQThreads), s, m, n_rows, q, scales);
    if (block == FP8G_BLOCK32_LITERAL)
        return launch_programmatic(quant_block32_kernel<FMT, BF16, true>, dim3(blocks),
                                   dim3(kQThreads), s, m, n_rows, q, scales);
    cudaError_t e = cudaMemsetAsync(scales, 0, sizeof(float), s);
    if (e != cudaSuccess) return e;
    amax_kernel<BF16><<<blocks, kQThreads, 0, s>>>(m, n_rows, reinterpret_cast<unsigned int *>(scales));
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    quant_tensor_kernel<FMT, BF16><<<blocks, kQThreads, 0, s>>>(m, n_rows, q, scales);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    finish_scale_kernel<FMT><<<1, 1, 0, s>>>(scales);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_nvfp4(const void *x, int in_bf16, int64_t rows, int64_t cols,
                                  uint8_t *q, uint8_t *sf, float *g, unsigned int *status,
                                  int num_sms, cudaStream_t s) {
    const RowMap m{x, nullptr, rows, cols, status};
    const int64_t cap = (int64_t)num_sms * 8;
    const unsigned blocks = (unsigned)(rows < cap ? rows : cap);
    cudaError_t e = cudaMemsetAsync(g, 0, sizeof(float), s);
    if (e != cudaSuccess) return e;
    if (in_bf16) {
        amax_kernel<true><<<blocks, kQThreads, 0, s>>>(m, rows, reinterpret_cast<unsigned int *>(g));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        quant_nvfp4_kernel<true><<<blocks, kQThreads, 0, s>>>(m, rows, q, sf, g);
    } else {
        amax_kernel<false><<<blocks, kQThreads, 0, s>>>(m, rows, reinterpret_cast<unsigned int *>(g));
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        quant_nvfp4_kernel<false><<<blocks, kQThreads, 0, s>>>(m, rows, q, sf, g);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    finish_nvfp4_kernel<<<1, 1, 0, s>>>(g);
    return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const void *x, int in_bf16, int64_t x_rows, int64_t cols,
                                 const int32_t *rows, int64_t n_rows, int32_t block, int fmt,
                                 uint8_t *q, float *scales, unsigned int *status, int num_sms,
                                 cudaStream_t s) {
    const RowMap m{x, rows, x_rows, cols, status};
    if (fmt == 3)
        return in_bf16 ? launch_rows<3, true>(m, n_rows, block, q, scales, num_sms, s)
                       : launch_rows<3, false>(m, n_rows, block, q, scales, num_sms, s);
    if (fmt == 4)
        return in_bf16 ? launch_rows<4, true>(m, n_rows, block, q, scales, num_sms, s)
                       : launch_rows<4, false>(m, n_rows, block, q, scales, num_sms, s);
    if (fmt == 2)
        return in_bf16 ? launch_rows<2, true>(m, n_rows, block, q, scales, num_sms, s)
                       : launch_rows<2, false>(m, n_rows, block, q, scales, num_sms, s);
    if (fmt == 1)
        return in_bf16 ? launch_rows<1, true>(m, n_rows, block, q, scales, num_sms, s)
                       : launch_rows<1, false>(m, n_rows, block, q, scales, num_sms, s);
    return in_bf16 ? launch_rows<0, true>(m, n_rows, block, q, scales, num_sms, s)
                   : launch_rows<0, false>(m, n_rows, block, q, scales, num_sms, s);
}

cudaError_t launch_dequant_tf32(const uint8_t *a, const float *s, int64_t rows, int64_t K, int fmt,
                                float *out, int num_sms, cudaStream_t stream) {
    const int64_t n = rows * (K / 8);
    if (n == 0) return cudaSuccess;
    const int64_t cap = (int64_t)num_sms * 8;
    const int64_t want = (n + 255) / 256;
    const unsigned blocks = (unsigned)(want < cap ? want : cap);
    if (fmt == FP8G_E5M2)
        dequant_tf32_kernel<1><<<blocks, 256, 0, stream>>>(a, s, rows, K, out);
    else
        dequant_tf32_kernel<0><<<blocks, 256, 0, stream>>>(a, s, rows, K, out);
    return cudaGetLastError();
}

}  // namespace fp8g
