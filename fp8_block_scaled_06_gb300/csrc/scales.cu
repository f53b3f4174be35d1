// Scale-factor packing: fp32 1x32 block scales -> UE8M0 bytes in the layout
// the tensor core's scale-factor copy reads (tcgen05.cp 32x128b.warpx4).
//
// The block-scaled MMA (kind::mxf8f6f4, "MXFP8 micro-scaling" of the Triton
// tutorial ch. 12, 12.6.1) applies one 8-bit power-of-two exponent per row
// and 32-wide K block.  A positive power of two's UE8M0 code is exactly its
// fp32 exponent field, so packing is lossless for the scales the API accepts.
//
// Packed layout, per operand: chunks of 512 bytes, one per (K group of 4
// blocks = one 128-wide K stage of the GEMM, tile of 128 rows):
//   chunk(z, kg, rt) at byte ((z * n_kg + kg) * n_rt + rt) * 512
//   byte 16 d + 4 w + j = code(row 128 rt + 32 w + d, K block 4 kg + j)
// so one GEMM stage reads its A chunk (512 B) and its B chunks (BN/128 x 512
// B, adjacent) with 1-D bulk copies.  Rows past the operand and K blocks past
// K/32 get code 127 (scale 1.0; the operand data there is zero).
//
// Grouped A: row tiles are expert-local (an expert's rows start a new tile),
// numbered in expert order, like the GEMM's tile list.
//
// HBM-bound: one launch packs both operands.  A block takes one 128-row tile
// and 8 K groups: it reads the tile's 128-byte row segments coalesced (8
// threads per row, 16 bytes each, all loads issued before any is used),
// converts them to code words in shared memory, and writes whole 16-byte
// groups of the output (4 rows' words of one K group).
#include "internal.h"
#include "ptx.cuh"
#include "kernel_common.cuh"

namespace fp8g {

namespace {


constexpr int kKgPerBlock = 8;
constexpr int kThreadsPack = 128;
constexpr int kRowsPerPass = kThreadsPack / kKgPerBlock;  // 16

struct PackJob {
    const float *src;
    int64_t rows_total, z_rows;
    int32_t n_rt, nz;
    uint8_t *dst;
    const int32_t *counts;  // grouped A: expert-local row tiles
    int32_t rep;            // replicated 256-row layout (B of 256-wide tiles)
    const int32_t *zskip;   // grouped B: matrix z of an expert without rows is not packed
};

// blockIdx.z < a.nz packs operand a (z = blockIdx.z), the rest operand b.
__global__ void __launch_bounds__(kThreadsPack) pack_scales_kernel(PackJob a, PackJob b, int64_t sfc,
                                                                  int32_t n_kg, int32_t E,
                                                                  unsigned int *status) {
    __shared__ int32_t row_off[FP8G_MAX_EXPERTS + 1];
    __shared__ int32_t rt_off[FP8G_MAX_EXPERTS + 1];
    __shared__ uint32_t words[kKgPerBlock][kBM];  // code word of (K group, row of the tile)
    // Launched programmatically: the blocks may be placed while the previous
    // kernel on the stream still runs (the last wave of a GEMM leaves SMs
    // idle), but touch global memory only after it completed.
    ptx::grid_dep_wait();
    ptx::grid_dep_launch();  // the GEMM may start its prologue now
    const bool first = (int)blockIdx.z < a.nz;
    const PackJob &j = first ? a : b;
    const int z = first ? (int)blockIdx.z : (int)blockIdx.z - a.nz;
    const int rt = blockIdx.y;
    if (rt >= j.n_rt) return;  // block-uniform
    // (no tile of the GEMM reads an empty expert's chunks; its scales are
    // neither packed nor checked)
    if (j.zskip != nullptr && j.zskip[z] <= 0) return;
    int64_t base, limit;
    if (j.counts != nullptr) {
        if (threadIdx.x == 0) {
            int64_t ro = 0, to = 0;
            row_off[0] = 0;
            rt_off[0] = 0;
            for (int e = 0; e < E; ++e) {
                const int32_t c = max(j.counts[e], 0);
                ro += c;
                to += (c + kBM - 1) / kBM;
                row_off[e + 1] = (int32_t)(ro < (int64_t)INT32_MAX ? ro : (int64_t)INT32_MAX);
                rt_off[e + 1] = (int32_t)to;
            }
        }
        __syncthreads();
        if (rt >= rt_off[E]) {
            base = 0;
            limit = 0;  // padding tile past the last expert
        } else {
            int e = 0;
            while (rt_off[e + 1] <= rt) ++e;
            base = (int64_t)row_off[e] + (int64_t)(rt - rt_off[e]) * kBM;
            limit = row_off[e + 1];
        }
    } else {
        base = (int64_t)rt * kBM;
        limit = j.rows_total;
    }
    if (limit > j.rows_total) limit = j.rows_total;
    const int kg0 = blockIdx.x * kKgPerBlock;
    const int sub = threadIdx.x % kKgPerBlock;  // K group of this thread's loads
    const int kg = kg0 + sub;
    const int64_t k0 = (int64_t)kg * 4;
    const bool vec = (sfc % 4) == 0;
    const float *zsrc = j.src + (int64_t)z * j.z_rows * sfc;
    // all loads first (independent): rows threadIdx.x / 8 + 16 p
    uint32_t v[kBM / kRowsPerPass][4];
#pragma unroll
    for (int pss = 0; pss < kBM / kRowsPerPass; ++pss) {
        const int64_t row = base + pss * kRowsPerPass + threadIdx.x / kKgPerBlock;
        const bool in = row < limit && kg < n_kg;
        const float *srow = zsrc + (in ? row : 0) * sfc;
        if (vec) {
            uint4 f = make_uint4(0u, 0u, 0u, 0u);
            if (in) f = __ldg(reinterpret_cast<const uint4 *>(srow + k0));
            v[pss][0] = f.x;
            v[pss][1] = f.y;
            v[pss][2] = f.z;
            v[pss][3] = f.w;
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                v[pss][q] = (in && k0 + q < sfc) ? __float_as_uint(__ldg(srow + k0 + q)) : 0u;
        }
    }
    bool bad = false;
#pragma unroll
    for (int pss = 0; pss < kBM / kRowsPerPass; ++pss) {
        const int r = pss * kRowsPerPass + threadIdx.x / kKgPerBlock;
        uint32_t word = 0x7F7F7F7Fu;  // rows past the operand: scale 1
        if (base + r < limit) {
            word = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t c = (k0 + q < sfc) ? ue8m0_code(v[pss][q], bad) : 127u;
                word |= c << (8 * q);
            }
        }
        words[sub][r] = word;
    }
    __syncthreads();
    // 16-byte output groups: the words of rows d, 32 + d, 64 + d, 96 + d of one
    // K group (byte 16 d + 4 w of a chunk is row 32 w + d)
    // per z: n_kg x n_rt chunks of 512 B, or (replicated) n_kg x n_rt / 2 blocks of 4 KB
    uint8_t *zdst = j.dst + (int64_t)z * n_kg * j.n_rt * (j.rep ? 2048 : 512);
    const int nk = n_kg - kg0 < kKgPerBlock ? n_kg - kg0 : kKgPerBlock;
    if (j.rep) {
        // 4 KB per (z, K group, 256-row tile): the 128-lane x 32-byte source of
        // one tcgen05.cp 128x256b; lane L = 32 q + d holds rows 32 w + d of
        // both 128-row halves h (bytes 128 h + 4 w of its 32), identical for
        // the four lane quarters q; 16-byte core rows, lane groups of 8 every
        // 256 bytes.
        const int h = rt & 1;
        for (int i = threadIdx.x; i < nk * kBM; i += kThreadsPack) {
            const int g = i / kBM, L = i % kBM, d = L & 31;
            const uint4 o = make_uint4(words[g][d], words[g][32 + d], words[g][64 + d], words[g][96 + d]);
            uint8_t *out = zdst + ((int64_t)(kg0 + g) * (j.n_rt / 2) + (rt >> 1)) * 4096 +
                           (L >> 3) * 256 + (L & 7) * 16 + h * 128;
            *reinterpret_cast<uint4 *>(out) = o;
        }
    } else {
        for (int i = threadIdx.x; i < nk * 32; i += kThreadsPack) {
            const int g = i / 32, d = i % 32;
            const uint4 o = make_uint4(words[g][d], words[g][32 + d], words[g][64 + d], words[g][96 + d]);
            *reinterpret_cast<uint4 *>(zdst + ((int64_t)(kg0 + g) * j.n_rt + rt) * 512 + 16 * d) = o;
        }
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0)
        if (atomicCAS(&status[0], 0u, (unsigned)FP8G_ERR_SCALE_FORMAT) == 0u)
            atomicExch(&status[1], 0u);
}

// NVFP4 scale codes -> chunks.  A block takes one 128-row tile and 8
// 64-wide K groups of one operand (blockIdx.z: 0 A, z >= 1 B's matrix z - 1):
// thread t loads row t / 2's four codes words of K groups kg0 + 4 (t % 2) ..
// + 3 (16 bytes), the words go through shared memory, and warp g stores K
// group kg0 + g's whole chunk (32 x 16 bytes: datapath d holds rows d,
// 32 + d, 64 + d, 96 + d).  Chunk order: the four K groups of one 256-wide
// GEMM stage are adjacent, chunk(z, kg, rt) at
// (z * n_kg * n_rt + (kg / 4 * n_rt + rt) * 4 + kg % 4) * 512, so a stage's
// scales of one 128-row tile are one 2 KB load.  Grouped A (counts set): row
// tiles are expert-local, numbered in expert order as the GEMM numbers them.
// Rows past the operand or the expert: 1.0 (0x38).  n_kg is a multiple of 4
// (K % 256 == 0).
struct PackNv {
    const uint8_t *src;
    int64_t rows;
    int32_t n_rt;
    uint8_t *dst;
    const int32_t *counts;  // A of the grouped GEMM, else null
};

__global__ void __launch_bounds__(256) pack_nvfp4_kernel(PackNv a, PackNv b, int32_t n_kg,
                                                        int64_t sfc, int32_t E) {
    __shared__ uint32_t words[8][kBM];
    __shared__ int64_t base_lim[2];
    ptx::grid_dep_wait();    // global memory only after the previous kernel (launched
    ptx::grid_dep_launch();  // programmatically); the GEMM may start its prologue now
    const PackNv &j = blockIdx.z == 0 ? a : b;
    const int rt = blockIdx.y;
    if (rt >= j.n_rt) return;  // block-uniform
    // grouped: an expert without rows has no tile, its B chunks are not packed
    if (blockIdx.z > 0 && a.counts != nullptr && a.counts[blockIdx.z - 1] <= 0) return;
    const int64_t z = blockIdx.z == 0 ? 0 : (int64_t)blockIdx.z - 1;
    const uint8_t *src = j.src + z * j.rows * sfc;
    uint8_t *dst = j.dst + z * n_kg * j.n_rt * 512;
    int64_t base = (int64_t)rt * kBM, limit = j.rows;
    if (j.counts != nullptr) {
        if (threadIdx.x == 0) {
            // this tile's expert: the first whose tiles end past rt
            int64_t ro = 0, to = 0, b0 = 0, lim = 0;
            for (int e = 0; e < E; ++e) {
                const int64_t c = j.counts[e] > 0 ? j.counts[e] : 0;
                const int64_t nt = (c + kBM - 1) / kBM;
                if (rt >= to && rt < to + nt) {
                    b0 = ro + (rt - to) * kBM;
                    lim = ro + c;
                }
                ro += c;
                to += nt;
            }
            base_lim[0] = b0;
            base_lim[1] = lim;  // 0 for padding tiles past the last expert
        }
        __syncthreads();
        base = base_lim[0];
        limit = base_lim[1] < j.rows ? base_lim[1] : j.rows;
    }
    const int kg0 = blockIdx.x * 8;
    {
        const int r = threadIdx.x >> 1, hh = threadIdx.x & 1;
        const int64_t row = base + r;
        const int k = kg0 + 4 * hh;
        uint4 w = make_uint4(0x38383838u, 0x38383838u, 0x38383838u, 0x38383838u);
        if (row < limit && k < n_kg)
            w = __ldg(reinterpret_cast<const uint4 *>(src + row * sfc) + k / 4);
        words[4 * hh + 0][r] = w.x;
        words[4 * hh + 1][r] = w.y;
        words[4 * hh + 2][r] = w.z;
        words[4 * hh + 3][r] = w.w;
    }
    __syncthreads();
    const int g = threadIdx.x >> 5, d = threadIdx.x & 31;
    const int kg = kg0 + g;
    if (kg < n_kg) {
        const uint4 o = make_uint4(words[g][d], words[g][32 + d], words[g][64 + d], words[g][96 + d]);
        *reinterpret_cast<uint4 *>(dst + (((int64_t)(kg >> 2) * j.n_rt + rt) * 4 + (kg & 3)) * 512 +
                                   16 * d) = o;
    }
}

}  // namespace

cudaError_t launch_pack_nvfp4(const uint8_t *sfa, int64_t rows_a, int32_t n_rt_a, uint8_t *dst_a,
                              const int32_t *counts, const uint8_t *sfb, int64_t rows_b,
                              int32_t n_rt_b, int32_t z_b, uint8_t *dst_b, int32_t n_kg,
                              int64_t sfc, int32_t E, cudaStream_t s) {
    const int ny = n_rt_a > n_rt_b ? n_rt_a : n_rt_b;
    if (n_kg <= 0 || ny <= 0 || z_b < 1) return cudaSuccess;
    const PackNv ja{sfa, rows_a, n_rt_a, dst_a, counts};
    const PackNv jb{sfb, rows_b, n_rt_b, dst_b, nullptr};
    const dim3 grid((unsigned)((n_kg + 7) / 8), (unsigned)ny, (unsigned)(1 + z_b));
    return launch_programmatic(pack_nvfp4_kernel, grid, dim3(256), s, ja, jb, n_kg, sfc, E);
}

size_t packed_scale_bytes(int32_t n_kg, int32_t n_rt, int32_t z) {
    return (size_t)z * (size_t)n_kg * (size_t)n_rt * 512u;
}

cudaError_t launch_pack_scales(const PackArgs &a, const PackArgs &b, int64_t sfc, int32_t n_kg,
                               int32_t E, unsigned int *status, cudaStream_t s) {
    if (n_kg <= 0) return cudaSuccess;
    PackJob ja{a.src, a.rows_total, a.z_rows, a.n_rt, a.nz, a.dst, a.counts, a.rep, a.zskip};
    PackJob jb{b.src, b.rows_total, b.z_rows, b.n_rt, b.nz, b.dst, b.counts, b.rep, b.zskip};
    const int nz = ja.nz + jb.nz;
    const int ny = ja.n_rt > jb.n_rt ? ja.n_rt : jb.n_rt;
    if (nz <= 0 || ny <= 0) return cudaSuccess;
    dim3 grid((unsigned)((n_kg + kKgPerBlock - 1) / kKgPerBlock), (unsigned)ny, (unsigned)nz);
    return launch_programmatic(pack_scales_kernel, grid, dim3(kThreadsPack), s, ja, jb, sfc, n_kg,
                               E, status);
}

}  // namespace fp8g
