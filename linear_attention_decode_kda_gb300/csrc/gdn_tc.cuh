// tcgen05 (5th-generation tensor core) helpers for sm_100 / sm_103a, inline PTX.
//
// Conventions used by every caller:
//   * cta_group::1, M = 128: row r of the accumulator D lives in TMEM lane r,
//     fp32 column c in TMEM column (d_col + c).  Warp w of the CTA reaches the
//     32 lanes 32 * (w % 4) .. 32 * (w % 4) + 31 with tcgen05.ld / st.
//   * Operands A (M x K) and B (N x K) are 16-bit (fp16 or bf16), K-major, in the canonical
//     no-swizzle layout of 8 x 8 "core matrices" (8 rows x 16 bytes, stored as
//     128 contiguous bytes).  Core matrix (row group g, K group q) of an
//     operand with `kdim` columns sits at byte ((g * (kdim / 8)) + q) * 128, so
//     the stride between K groups (leading byte offset) is 128 bytes and the
//     stride between row groups (stride byte offset) is kdim * 16 bytes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace gdn {
namespace tc {

// Byte offset of 16-bit element (r, k) of a K-major canonical operand with kdim columns.
__host__ __device__ __forceinline__ uint32_t op_offset(int r, int k, int kdim)
{
    return static_cast<uint32_t>((((r >> 3) * (kdim >> 3)) + (k >> 3)) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// Shared-memory matrix descriptor (no swizzle) for the K group pair starting at
// element column k0 of an operand at shared address `base` with kdim columns.
__device__ __forceinline__ uint64_t op_desc(uint32_t base, int k0, int kdim)
{
    const uint32_t start = base + static_cast<uint32_t>(k0 >> 3) * 128;
    const uint64_t lbo = 128, sbo = static_cast<uint64_t>(kdim) * 16;
    uint64_t d = 0;
    d |= static_cast<uint64_t>((start & 0x3FFFF) >> 4);   // bits 0-13: start address
    d |= ((lbo >> 4) & 0x3FFF) << 16;                       // bits 16-29: leading byte offset
    d |= ((sbo >> 4) & 0x3FFF) << 32;                       // bits 32-45: stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                    // bits 46-48: descriptor version 1
    return d;                                               // base offset 0, no swizzle
}

// Descriptor of a K-major no-swizzle operand laid out with any strides: `lbo`
// bytes between core matrices adjacent in K, `sbo` bytes between 8-row groups
// (op_desc is this with lbo = 128 and sbo = kdim * 16).
__device__ __forceinline__ uint64_t op_desc_strided(uint32_t start, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((start & 0x3FFFF) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    return d;
}

// Descriptor of a K-major operand in the 128-byte swizzled layout that a TMA box
// of 64 16-bit elements x R rows with CU_TENSOR_MAP_SWIZZLE_128B writes (1024-byte
// aligned): rows of 128 bytes, 8-row groups 1024 bytes apart (SBO), the 16-byte
// chunks of row r permuted by r % 8.  The K step k0 (a multiple of 16 elements,
// below 64) advances the start address by 2 k0 bytes inside the 128-byte row.
__device__ __forceinline__ uint64_t op_desc_sw128(uint32_t base, int k0)
{
    const uint32_t start = base + static_cast<uint32_t>(k0) * 2;
    uint64_t d = 0;
    d |= static_cast<uint64_t>((start & 0x3FFFF) >> 4);  // bits 0-13: start address
    d |= static_cast<uint64_t>(1) << 16;                   // bits 16-29: leading offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;           // bits 32-45: stride byte offset
    d |= static_cast<uint64_t>(1) << 46;                   // bits 46-48: descriptor version 1
    d |= static_cast<uint64_t>(2) << 61;                   // bits 61-63: 128-byte swizzle
    return d;
}

// Byte offset of 16-bit element (r, k) of a K-major operand with `rows` rows in the
// 128-byte swizzled layout (1024-byte aligned base): K splits into atoms of 64
// elements, atom a holding every row at a * rows * 128; inside an atom rows are
// 128 bytes, 8-row groups 1024 bytes apart, and the 16-byte chunk c of row r sits
// at chunk position c ^ (r % 8) -- the layout a TMA box with
// CU_TENSOR_MAP_SWIZZLE_128B writes, and what op_desc_sw128 describes.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int r, int k, int rows)
{
    const int kk = k & 63;
    return static_cast<uint32_t>((k >> 6) * rows * 128 + (r >> 3) * 1024 + (r & 7) * 128 +
                                 ((((kk >> 3) ^ (r & 7)) & 7) << 4) + (kk & 7) * 2);
}

// Instruction descriptor of kind::f16: fp16 (or bf16) A and B, fp32 D, both K-major.
__host__ __device__ __forceinline__ uint32_t idesc_f16(int M, int N, bool negate_a, bool bf16 = false)
{
    uint32_t d = 0;
    d |= 1u << 4;                                    // D format: fp32
    if (bf16) d |= (1u << 7) | (1u << 10);           // A, B format: bf16 (0 = fp16)
    if (negate_a) d |= 1u << 13;                     // negate A
    d |= static_cast<uint32_t>(N >> 3) << 17;        // N / 8
    d |= static_cast<uint32_t>(M >> 4) << 24;        // M / 16
    return d;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// One warp allocates `ncols` TMEM columns; the address lands in *slot (shared).
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// D[tmem] (+)= A * B^T over one K step of 16; issued by a single thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0)
        : "memory");
}

// D[tmem] (+)= A * B^T with A in TMEM: row m of A in lane m, its 16-bit K values two
// to a 32-bit column (K-step k0 at column k0 / 2); B from shared memory.
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0)
        : "memory");
}

// Arrives on the mbarrier when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 lanes x 16 consecutive fp32 columns: this thread gets columns col .. col+15 of its lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 8 consecutive fp32 columns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 16 consecutive 32-bit columns, raw words (no wait).
__device__ __forceinline__ void tmem_st16u_nowait(uint32_t taddr, const uint32_t (&w)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
        "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&w)[16])
{
    tmem_st16u_nowait(taddr, w);
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Tensor-core operands are fp16 (11 significant bits); precision-critical ones
// are kept as hi + lo pairs (x ~ hi + lo) and multiplied as hi*hi + hi*lo + lo*hi.
__device__ __forceinline__ void put_split(unsigned char *hi, unsigned char *lo, uint32_t off, float v)
{
    const __half h = __float2half_rn(v);
    *reinterpret_cast<__half *>(hi + off) = h;
    *reinterpret_cast<__half *>(lo + off) = __float2half_rn(v - __half2float(h));
}

// 8 consecutive K values of one row of a K-major operand (offset 16-byte aligned),
// as one 128-bit store per half of the split (lo may be null: a plain fp16 operand).
__device__ __forceinline__ void put_row8(unsigned char *hi, unsigned char *lo, uint32_t off, const float *v)
{
    __half2 h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half a = __float2half_rn(v[2 * i]), b = __float2half_rn(v[2 * i + 1]);
        h[i] = __halves2half2(a, b);
        l[i] = __floats2half2_rn(v[2 * i] - __half2float(a), v[2 * i + 1] - __half2float(b));
    }
    *reinterpret_cast<uint4 *>(hi + off) = *reinterpret_cast<const uint4 *>(h);
    if (lo) *reinterpret_cast<uint4 *>(lo + off) = *reinterpret_cast<const uint4 *>(l);
}

// D (+)= A B^T over K in steps of 16 (single thread).
__device__ __forceinline__ void mma_chain(uint32_t d, uint32_t a, uint32_t b, int kdim,
                                          uint32_t idesc, bool acc)
{
    for (int k0 = 0; k0 < kdim; k0 += 16)
        mma_f16(d, op_desc(a, k0, kdim), op_desc(b, k0, kdim), idesc, acc || k0 > 0);
}

// D (+)= (A_hi + A_lo)(B_hi + B_lo)^T without the lo*lo term.
__device__ __forceinline__ void mma_split(uint32_t d, uint32_t ah, uint32_t al, uint32_t bh,
                                          uint32_t bl, int kdim, uint32_t idesc, bool acc)
{
    mma_chain(d, ah, bh, kdim, idesc, acc);
    mma_chain(d, ah, bl, kdim, idesc, true);
    mma_chain(d, al, bh, kdim, idesc, true);
}

// TMEM address of (lane, column) for the warp's lane quadrant.
__device__ __forceinline__ uint32_t taddr(uint32_t base, int lane_base, int col)
{
    return base + (static_cast<uint32_t>(lane_base) << 16) + static_cast<uint32_t>(col);
}

}  // namespace tc
}  // namespace gdn
