// Chunked prefill of Gated DeltaNet (one decay per head), d_k = d_v = 128, bf16
// rows, 64-token chunks, every dense product on tcgen05, no workspace.
//
// The form is the chunked WY/UT recurrence of "llama.cpp PR #84" (the chunked
// KDA prefill, here with the per-head decay of Gated DeltaNet).  Inside a chunk
// of n <= 64 tokens with start state S0, G_t is the log-decay summed from the
// chunk's first token through t (every exponent below is <= 0), q^, k^ the
// L2-normalised rows (q^ scaled), and
//   A[t][s] = beta_t (k^_t . k^_s) e^{G_t - G_s}   (s < t),   T = (I + A)^-1
//   W = T diag(beta e^G) K^,   U = T diag(beta) V,   V_new = U - W S0
//   O = diag(e^G) Q^ S0 + M V_new,   M[t][s] = (q^_t . k^_s) e^{G_t - G_s}  (s <= t)
//   S = e^{G_last} S0 + (diag(e^{G_last - G}) K^)^T V_new
// T sequential steps of "Thirty tiny kernels per layer" and this form agree up to
// rounding.
//
// Layout of the work.  One CTA of 16 warps owns one (sequence, value head) and
// walks its chunks; value heads sharing a qk head form a thread-block cluster so
// the shared q/k conv window is written back only after every CTA of the group
// has read it.  Everything is computed transposed so that each product has
// M = 128 rows (the head dimension) in TMEM lanes:
//   Gram    [K; Q] K^T                      K-raw and Q-raw rows (128 x 64)
//   W^T   = K^T T1^T,   T1 = T diag(beta e^G rk)
//   U^T   = V^T T2^T,   T2 = T diag(beta)
//   V_new^T = U^T - S0^T W^T                (accumulated onto U^T, A negated)
//   P^T   = S0^T Q^T                        (scaled by e^{G_t} rq_t when read)
//   OV^T  = V_new^T M^T
//   S^T   = e^{G_last} S^T + (V_new diag(e^{G_last - G} rk))^T K
// The norms rk, rq and every per-token factor are folded into these small
// matrices and the read-back, so q, k and v enter the tensor core unscaled.
// S^T is an fp32 accumulator in TMEM; its fp16 copy (hi + lo) is the A operand
// of the two S0 products straight from TMEM.  Every other operand is a K-major
// shared-memory operand, stored as fp16 hi + lo pairs (x ~ hi + lo, about 22
// significant bits) and multiplied as hi*hi + hi*lo + lo*hi.
//
// Per chunk the CTA runs: conv + SiLU of the 64 q/k/v rows (warps 0-11, while
// warps 12-15 finish the previous chunk's output and rebuild the fp16 state),
// the Gram product, A, the blocked inverse T, the W and U products, the W and M
// operands, the two S0 products, the V_new operands, then the output and state
// products.  The next chunk's input rows arrive by TMA while this one runs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"
#include "gdn_device.cuh"
#include "gdn_internal.h"
#include "gdn_prefill.h"
#include "gdn_tc.cuh"
#include "gdn_tmap.h"

namespace gdn {
namespace {

using namespace dev;

constexpr int D = 128;       // d_k = d_v
constexpr int CK = 64;       // chunk length
constexpr int NT = 512;      // threads: 16 warps
constexpr int NCONV = 384;   // conv threads (warps 0-11)
constexpr int RAWR = CK + 3; // input rows a chunk reads: its 64 and the 3 before

// Dynamic shared memory (bytes from a 1024-byte aligned base).
// [K; Q]: rows 0-63 K, 64-127 Q, 128-byte swizzled K-major (two atoms of 64 channels).
constexpr uint32_t S_KQH = 0, S_KQL = 32768;
// K^T and V^T: [128 channels][64 tokens] canonical K-major with 8-row groups 1040
// bytes apart (16 bytes of padding spread the conv threads' stores over the banks).
constexpr uint32_t TSBO = 1040;
constexpr uint32_t T_BYTES = 16 * TSBO;
constexpr uint32_t S_KTH = 65536, S_KTL = S_KTH + T_BYTES, S_VTH = S_KTL + T_BYTES,
                   S_VTL = S_VTH + T_BYTES;
constexpr uint32_t S_RAW = ((S_VTL + T_BYTES + 1023) / 1024) * 1024;  // q, k, v boxes [67][128] bf16
constexpr uint32_t RAW_BOX = RAWR * D * 2;
constexpr uint32_t S_Z = ((S_RAW + 3 * RAW_BOX + 1023) / 1024) * 1024;  // z box [64][128] bf16
constexpr uint32_t S_WIN = S_Z + CK * D * 2;                            // fp32 window [3][384]
constexpr uint32_t SMEM_USED = S_WIN + 3 * NCONV * 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base
static_assert(SMEM_BYTES <= 232448, "shared memory per block");
// Reused regions.  The K rows of [K; Q] are dead after the Gram product: they take
// T1, T2 (canonical [64][64], 8 KB each), then W (swizzled [64][128], two atoms).
constexpr uint32_t KP0 = S_KQH, KP1 = S_KQH + 16384, KP2 = S_KQL, KP3 = S_KQL + 16384;
// M (canonical [64][64]) takes V^T's place after the U product.
constexpr uint32_t S_MH = S_VTH, S_ML = S_VTH + 8192;
// V_new and V_new diag(d) (canonical [128][64], 16 KB each) take [K; Q] after the S0 products.
constexpr uint32_t S_VNH = S_KQH, S_VNL = S_KQH + 16384, S_VDH = S_KQL, S_VDL = S_KQL + 16384;
// fp32 scratch of the inverse inside the raw-row region (free between the conv and
// the next chunk's copy): A and T [64][65], the block products [3][16][17].
constexpr int FS = CK + 1;
constexpr uint32_t S_AF = S_RAW, S_TF = S_AF + CK * FS * 4, S_RF = S_TF + CK * FS * 4;
static_assert(S_RF + 3 * 16 * 17 * 4 <= S_RAW + 3 * RAW_BOX, "inverse scratch");
static_assert(S_ML + 8192 <= S_VTH + T_BYTES, "M operand");

// TMEM columns.
constexpr uint32_t TM_S = 0;     // 128: S^T fp32
constexpr uint32_t TM_SH = 128;  // 64: S^T fp16 hi, two to a column
constexpr uint32_t TM_SL = 192;  // 64: S^T fp16 lo
constexpr uint32_t TM_G = 256;   // 64: Gram, then S0^T Q^T
constexpr uint32_t TM_W = 320;   // 64: W^T
constexpr uint32_t TM_U = 384;   // 64: U^T, then V_new^T
constexpr uint32_t TM_OV = 448;  // 64: V_new^T M^T

__device__ unsigned int g_c64_error;  // bit 0: a bounded mbarrier wait gave up

struct C64Shared {
    float G2[CK];        // cumulative log2-decay inside the chunk
    float bt[CK];        // beta (0 past the chunk's end)
    float nq[CK], nk[CK];  // |q|^2, |k|^2 of the raw rows
    float rk[CK];        // 1 / |k|
    float rq[CK];        // q_scale / |q|
    float f1[CK];        // beta_s e^{G_s} rk_s
    float ds[CK];        // e^{G_last - G_s} rk_s
    float cq[CK];        // e^{G_t} rq_t
    float osq[4][CK];    // per TMEM quadrant: partial sums of o^2
    float rinv[CK];
    float egl;           // e^{G_last}
    uint64_t raw_full, z_full, mma_bar;
    uint32_t tmem;
};

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// fp16 hi + lo of a pair of values, each packed two to a 32-bit word (first in the low half).
__device__ __forceinline__ void split2(float a, float b, uint32_t &hi, uint32_t &lo)
{
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// v[k]: this lane's partial for item k of 8.  Returns the warp-wide sum of item
// 4 * bit4(lane) + 2 * bit3(lane) + bit2(lane), in every lane.
__device__ __forceinline__ float reduce8(const float (&v)[8], int lane)
{
    float a[4], b[2];
    bool up = (lane & 16) != 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float send = up ? v[k] : v[k + 4], keep = up ? v[k + 4] : v[k];
        a[k] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    up = (lane & 8) != 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const float send = up ? a[k] : a[k + 2], keep = up ? a[k + 2] : a[k];
        b[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    up = (lane & 4) != 0;
    float c = (up ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, up ? b[0] : b[1], 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    return c;
}

// After the call lane l holds the warp-wide sum of v[l].
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane)
{
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
            const float send = up ? v[j] : v[j + w];
            const float keep = up ? v[j + w] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    return v[0];
}

// Byte offset of element (r, k) of a canonical K-major operand whose 8-row groups
// are `sbo` bytes apart (16-byte core-matrix rows, K groups 128 bytes apart).
__device__ __forceinline__ uint32_t cano(int r, int k, uint32_t sbo)
{
    return static_cast<uint32_t>(r >> 3) * sbo + static_cast<uint32_t>(k >> 3) * 128 +
           static_cast<uint32_t>(r & 7) * 16 + static_cast<uint32_t>(k & 7) * 2;
}

// 8 values of row r, K columns k0 .. k0 + 7 (k0 % 8 == 0), as hi and lo 16-byte stores.
__device__ __forceinline__ void put8(unsigned char *hi, unsigned char *lo, uint32_t off, const float *v)
{
    uint4 h, l;
    split2(v[0], v[1], h.x, l.x);
    split2(v[2], v[3], h.y, l.y);
    split2(v[4], v[5], h.z, l.z);
    split2(v[6], v[7], h.w, l.w);
    *reinterpret_cast<uint4 *>(hi + off) = h;
    *reinterpret_cast<uint4 *>(lo + off) = l;
}

// Writes the fp16 hi / lo copy of S^T columns i0 .. i0 + 31 of this thread's lane.
__device__ __forceinline__ void put_s16(uint32_t tm, int lb, int i0, const float (&s)[32])
{
    uint32_t h[16], l[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) split2(s[2 * k], s[2 * k + 1], h[k], l[k]);
    tc::tmem_st16u_nowait(tc::taddr(tm, lb, TM_SH + i0 / 2), h);
    tc::tmem_st16u_nowait(tc::taddr(tm, lb, TM_SL + i0 / 2), l);
}

__device__ __forceinline__ uint64_t cdesc(uint32_t base, int k0, uint32_t sbo)
{
    return tc::op_desc_strided(base + static_cast<uint32_t>(k0 >> 3) * 128, 128, sbo);
}

// D (+)= (A_hi + A_lo)(B_hi + B_lo)^T without lo*lo, both operands canonical K-major.
__device__ __forceinline__ void mma3c(uint32_t d, uint32_t ah, uint32_t al, uint32_t asbo, uint32_t bh,
                                      uint32_t bl, uint32_t bsbo, int kdim, uint32_t idesc, bool acc)
{
    for (int k0 = 0; k0 < kdim; k0 += 16) {
        const uint64_t dah = cdesc(ah, k0, asbo), dal = cdesc(al, k0, asbo);
        const uint64_t dbh = cdesc(bh, k0, bsbo), dbl = cdesc(bl, k0, bsbo);
        tc::mma_f16(d, dah, dbh, idesc, acc || k0 > 0);
        tc::mma_f16(d, dah, dbl, idesc, true);
        tc::mma_f16(d, dal, dbh, idesc, true);
    }
}

__device__ __forceinline__ void publish()
{
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
}

__device__ __forceinline__ void bar_epi()  // warps 12-15
{
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

__global__ void __launch_bounds__(NT, 1)
c64_prefill_kernel(const StepArgs a, const __grid_constant__ CUtensorMap tm_qkv,
                   const __grid_constant__ CUtensorMap tm_z)
{
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    __shared__ __align__(16) C64Shared ps;
    unsigned char *sm = sm_raw + ((1024u - (tc::smem_u32(sm_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, part = warp >> 2, lb = 32 * quad;
    const int h = blockIdx.x, b = blockIdx.y, hq = h / a.group;
    const int T = a.T, C = a.C, H = a.H_v;
    const bool clustered = a.group > 1;
    const bool qk_owner = (h % a.group) == 0;
    const size_t head = static_cast<size_t>(b) * H + h;
    const int chq = hq * D, chk = a.H_qk * D + hq * D, chv = 2 * a.H_qk * D + h * D;
    float *win = reinterpret_cast<float *>(sm + S_WIN);
    float *Af = reinterpret_cast<float *>(sm + S_AF);
    float *Tf = reinterpret_cast<float *>(sm + S_TF);
    float *Rf = reinterpret_cast<float *>(sm + S_RF);

    if (warp == 0) tc::tmem_alloc(&ps.tmem, 512);
    if (tid == 0) {
        mbar_init(&ps.raw_full, 1);
        mbar_init(&ps.z_full, 1);
        mbar_init(&ps.mma_bar, 1);
        fence_mbar_init();
        prefetch_tensormap(&tm_qkv);
        prefetch_tensormap(&tm_z);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = ps.tmem;
    pdl_wait();
    // Dependents launch only once this grid has passed its own dependency wait.
    pdl_launch_dependents();

    // this chunk's q, k, v rows and the 3 before them: three [67][128] boxes of [B*T, C]
    auto issue_raw = [&](int c0) {
        mbar_expect_tx(&ps.raw_full, 3 * RAW_BOX);
        const int row = b * T + c0 - 3;  // rows before the tensor read as zero
        tma_load_2d(sm + S_RAW, &tm_qkv, chq, row, &ps.raw_full);
        tma_load_2d(sm + S_RAW + RAW_BOX, &tm_qkv, chk, row, &ps.raw_full);
        tma_load_2d(sm + S_RAW + 2 * RAW_BOX, &tm_qkv, chv, row, &ps.raw_full);
    };
    if (tid == 0) issue_raw(0);

    // the kept conv window (fp32; the first chunk's 3 earlier rows) and the initial state
    if (tid < NCONV) {
        const int ten = tid >> 7, c = tid & 127;
        const int ch = (ten == 0 ? chq : ten == 1 ? chk : chv) + c;
#pragma unroll
        for (int r = 0; r < 3; ++r) win[r * NCONV + tid] = a.conv_in[(static_cast<size_t>(b) * 3 + r) * C + ch];
    }
    {   // S[i][j] -> TMEM S^T (lane j, column i) and its fp16 copy; this warp takes rows 32 part ..
        const float *Sg = a.state_in + head * D * D;
        float s[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) s[k] = Sg[(32 * part + k) * D + lb + lane];
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) w[k] = __float_as_uint(s[k]);
        tc::tmem_st16u_nowait(tc::taddr(tm, lb, TM_S + 32 * part), w);
#pragma unroll
        for (int k = 0; k < 16; ++k) w[k] = __float_as_uint(s[16 + k]);
        tc::tmem_st16u_nowait(tc::taddr(tm, lb, TM_S + 32 * part + 16), w);
        put_s16(tm, lb, 32 * part, s);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    if (clustered) cluster_arrive_relaxed();  // this CTA has read the shared q/k window

    // conv threads: tensor ten (0 q, 1 k, 2 v), channels 4 lane .. 4 lane + 3, token
    // blocks 2 (warp % 4) and 2 (warp % 4) + 1 of every chunk
    const int ten = warp >> 2;
    float4 cw[4];
    if (warp < 12) {
        const int ch0 = (ten == 0 ? chq : ten == 1 ? chk : chv) + 4 * lane;
#pragma unroll
        for (int c = 0; c < 4; ++c) cw[c] = reinterpret_cast<const float4 *>(a.conv_w)[ch0 + c];
    }

    // gate logits of the next chunk: warp 12, tokens 2 lane and 2 lane + 1
    const float A_h = expf(a.A_log[h]);
    const float dt_h = a.dt_bias[h];
    float fx[2] = {0.f, 0.f}, bx[2] = {0.f, 0.f};
    auto load_gates = [&](int c0) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = c0 + 2 * lane + u;
            if (t < T) {
                const size_t e = (static_cast<size_t>(b) * T + t) * H + h;
                fx[u] = ld_in(a.f, e, 1);
                bx[u] = ld_in(a.beta, e, 1);
            }
        }
    };
    if (warp == 12) load_gates(0);
    const float nw = a.norm_w[lb + lane];  // output-norm weight of this lane's column

    bool ok = true;
    uint32_t mma_ph = 0;
    auto mma_wait = [&]() {
        if (ok) ok = mbar_wait_bounded(&ps.mma_bar, mma_ph);
        mma_ph ^= 1u;
        tc::fence_after_sync();
    };
    const uint32_t smb = tc::smem_u32(sm);
    const uint32_t id64 = tc::idesc_f16(128, 64, false), id64n = tc::idesc_f16(128, 64, true),
                   id128 = tc::idesc_f16(128, 128, false);

    // The output of chunk (cp, np) from TMEM: o = P^T e^{G_t} rq_t + OV^T, the gated
    // RMSNorm over the 128 columns, y stored.  Warps 12-15 (lane = column j).
    auto epilogue = [&](int cp, int np, int it) {
        if (ok) ok = mbar_wait_bounded(&ps.z_full, static_cast<uint32_t>(it & 1));
        const int j = lb + lane;
        const unsigned char *zs = sm + S_Z;
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
            float o[32], v[32];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float p16[16], ov16[16];
                tc::tmem_ld16(tc::taddr(tm, lb, TM_G + 32 * hf + 16 * q), p16);
                tc::tmem_ld16(tc::taddr(tm, lb, TM_OV + 32 * hf + 16 * q), ov16);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float x = fmaf(p16[k], ps.cq[32 * hf + 16 * q + k], ov16[k]);
                    o[16 * q + k] = x;
                    v[16 * q + k] = x * x;
                }
            }
            const float sq = reduce_scatter32(v, lane);
            ps.osq[quad][32 * hf + lane] = sq;
            bar_epi();
            if (warp == 12) {
                const int t = 32 * hf + lane;
                const float m = (ps.osq[0][t] + ps.osq[1][t] + ps.osq[2][t] + ps.osq[3][t]) * (1.0f / D);
                ps.rinv[t] = rsqrtf(m + a.eps_norm);
            }
            bar_epi();
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const int t = 32 * hf + k;
                if (t < np) {
                    const float zz = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(zs + (t * D + j) * 2));
                    const float gz = a.sig_gate ? sigmoid_fast(zz) : silu_fast(zz);
                    const float y = o[k] * ps.rinv[t] * nw * gz;
                    const size_t idx = ((static_cast<size_t>(b) * T + cp + t) * H + h) * D + j;
                    if (a.out_bf16)
                        reinterpret_cast<__nv_bfloat16 *>(a.out)[idx] = __float2bfloat16_rn(y);
                    else
                        reinterpret_cast<float *>(a.out)[idx] = y;
                }
            }
        }
        fence_proxy_async_smem();  // the z stage is read: the next copy may land there
    };

    int cp = 0, np = 0;
#pragma unroll 1
    for (int c0 = 0, it = 0; c0 < T; c0 += CK, ++it) {
        const int n = min(CK, T - c0);

        if (warp < 12) {
            // ---- conv + SiLU of two 8-token blocks; q -> Q rows, k -> K rows and K^T, v -> V^T
            if (ok) ok = mbar_wait_bounded(&ps.raw_full, static_cast<uint32_t>(it & 1));
            const unsigned char *raw = sm + S_RAW + ten * RAW_BOX;
#pragma unroll 1
            for (int blk = 0; blk < 2; ++blk) {
                const int tb = 2 * quad + blk;  // token block: tokens 8 tb .. 8 tb + 7
                float xw[3][4];
#pragma unroll
                for (int r = 0; r < 3; ++r) {
                    if (c0 == 0 && tb == 0) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) xw[r][c] = win[r * NCONV + ten * 128 + 4 * lane + c];
                    } else {
                        const uint2 u = *reinterpret_cast<const uint2 *>(raw + ((8 * tb + r) * D + 4 * lane) * 2);
                        xw[r][0] = __uint_as_float(u.x << 16);
                        xw[r][1] = __uint_as_float(u.x & 0xffff0000u);
                        xw[r][2] = __uint_as_float(u.y << 16);
                        xw[r][3] = __uint_as_float(u.y & 0xffff0000u);
                    }
                }
                uint32_t hn[8][2], ln[8][2];
                float nrm[8];
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const int t = 8 * tb + rr;
                    const uint2 u = *reinterpret_cast<const uint2 *>(raw + ((t + 3) * D + 4 * lane) * 2);
                    float x[4];
                    x[0] = __uint_as_float(u.x << 16);
                    x[1] = __uint_as_float(u.x & 0xffff0000u);
                    x[2] = __uint_as_float(u.y << 16);
                    x[3] = __uint_as_float(u.y & 0xffff0000u);
                    float y[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float acc = cw[c].x * xw[0][c];
                        acc = fmaf(cw[c].y, xw[1][c], acc);
                        acc = fmaf(cw[c].z, xw[2][c], acc);
                        acc = fmaf(cw[c].w, x[c], acc);
                        y[c] = t < n ? silu_fast(acc) : 0.f;
                        xw[0][c] = xw[1][c];
                        xw[1][c] = xw[2][c];
                        xw[2][c] = x[c];
                    }
                    nrm[rr] = y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3];
                    split2(y[0], y[1], hn[rr][0], ln[rr][0]);
                    split2(y[2], y[3], hn[rr][1], ln[rr][1]);
                    if (ten < 2) {  // row t (k) or 64 + t (q) of [K; Q], 4 channels = 8 bytes
                        const int R = ten == 0 ? 64 + t : t;
                        const uint32_t off = (lane >> 4) * 16384 + (R >> 3) * 1024 + (R & 7) * 128 +
                                             (((((lane & 15) >> 1) ^ (R & 7)) & 7) << 4) + (lane & 1) * 8;
                        *reinterpret_cast<uint2 *>(sm + S_KQH + off) = make_uint2(hn[rr][0], hn[rr][1]);
                        *reinterpret_cast<uint2 *>(sm + S_KQL + off) = make_uint2(ln[rr][0], ln[rr][1]);
                    }
                }
                if (ten >= 1) {  // K^T / V^T rows 4 lane + c: the block's 8 tokens, 16 bytes
                    unsigned char *th = sm + (ten == 1 ? S_KTH : S_VTH);
                    unsigned char *tl = sm + (ten == 1 ? S_KTL : S_VTL);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t sel = (c & 1) ? 0x7632u : 0x5410u;
                        uint4 vh, vl;
                        vh.x = __byte_perm(hn[0][c >> 1], hn[1][c >> 1], sel);
                        vh.y = __byte_perm(hn[2][c >> 1], hn[3][c >> 1], sel);
                        vh.z = __byte_perm(hn[4][c >> 1], hn[5][c >> 1], sel);
                        vh.w = __byte_perm(hn[6][c >> 1], hn[7][c >> 1], sel);
                        vl.x = __byte_perm(ln[0][c >> 1], ln[1][c >> 1], sel);
                        vl.y = __byte_perm(ln[2][c >> 1], ln[3][c >> 1], sel);
                        vl.z = __byte_perm(ln[4][c >> 1], ln[5][c >> 1], sel);
                        vl.w = __byte_perm(ln[6][c >> 1], ln[7][c >> 1], sel);
                        const uint32_t off = cano(4 * lane + c, 8 * tb, TSBO);
                        *reinterpret_cast<uint4 *>(th + off) = vh;
                        *reinterpret_cast<uint4 *>(tl + off) = vl;
                    }
                }
                if (ten < 2) {
                    const float tot = reduce8(nrm, lane);
                    if ((lane & 3) == 0) {
                        const int t = 8 * tb + ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
                        (ten == 0 ? ps.nq : ps.nk)[t] = tot;
                    }
                }
            }
        } else {
            // ---- gates of this chunk (warp 12), then the previous chunk's output and
            // the fp16 copy of the state it left (warps 12-15)
            if (warp == 12) {
                float g[2], bb[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const bool in = 2 * lane + u < n;
                    g[u] = in ? -A_h * softplus_fast(fx[u] + dt_h) : 0.f;
                    bb[u] = in ? sigmoid_fast(bx[u]) : 0.f;
                }
                if (c0 + CK < T) load_gates(c0 + CK);
                const float pair = g[0] + g[1];
                float sc = pair;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, sc, off);
                    if (lane >= off) sc += y;
                }
                ps.G2[2 * lane] = (sc - g[1]) * kLog2e;
                ps.G2[2 * lane + 1] = sc * kLog2e;
                ps.bt[2 * lane] = bb[0];
                ps.bt[2 * lane + 1] = bb[1];
            }
            if (it > 0) {
#pragma unroll 1
                for (int i0 = 0; i0 < D; i0 += 32) {
                    float s[32], s16[16];
                    tc::tmem_ld16(tc::taddr(tm, lb, TM_S + i0), s16);
#pragma unroll
                    for (int k = 0; k < 16; ++k) s[k] = s16[k];
                    tc::tmem_ld16(tc::taddr(tm, lb, TM_S + i0 + 16), s16);
#pragma unroll
                    for (int k = 0; k < 16; ++k) s[16 + k] = s16[k];
                    put_s16(tm, lb, i0, s);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                epilogue(cp, np, it - 1);
            }
        }
        publish();  // B1: conv operands written, previous output read

        // ---- Gram product [K; Q] K^T (hi.hi + hi.lo + lo.hi); the z rows of this chunk
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll 1
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t at = (ks >> 2) * 16384;
                const int k0 = (ks & 3) * 16;
                const uint64_t ah = tc::op_desc_sw128(smb + S_KQH + at, k0);
                const uint64_t al = tc::op_desc_sw128(smb + S_KQL + at, k0);
                tc::mma_f16(tm + TM_G, ah, ah, id64, ks > 0);  // B = rows 0-63 (K) of the same atom
                tc::mma_f16(tm + TM_G, ah, al, id64, true);
                tc::mma_f16(tm + TM_G, al, ah, id64, true);
            }
            tc::mma_commit(&ps.mma_bar);
            mbar_expect_tx(&ps.z_full, CK * D * 2);
            tma_load_3d(sm + S_Z, &tm_z, 0, h, b * T + c0, &ps.z_full);
        }
        // per-token factors of this chunk
        if (tid < CK) {
            const int t = tid;
            const bool in = t < n;
            const float rk = in ? rsqrtf(ps.nk[t] + a.eps_l2) : 0.f;
            const float rq = in ? a.q_scale * rsqrtf(ps.nq[t] + a.eps_l2) : 0.f;
            const float G2t = ps.G2[t], G2l = ps.G2[n - 1];
            ps.rk[t] = rk;
            ps.rq[t] = rq;
            ps.f1[t] = ps.bt[t] * ex2(G2t) * rk;
            ps.ds[t] = in ? ex2(G2l - G2t) * rk : 0.f;
            ps.cq[t] = ex2(G2t) * rq;
            if (t == 0) ps.egl = ex2(G2l);
        }
        __syncthreads();
        mma_wait();

        // ---- A = beta_t rk_t rk_s (k.k) e^{G_t - G_s} (s < t): lanes 0-63 hold K rows
        if (quad < 2) {
            const int t = lb + lane;
            float v[16];
            tc::tmem_ld16(tc::taddr(tm, lb, TM_G + 16 * part), v);
            const float bt = ps.bt[t] * ps.rk[t], G2t = ps.G2[t];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int s = 16 * part + k;
                Af[t * FS + s] = (s < t && t < n) ? bt * ps.rk[s] * v[k] * ex2(G2t - ps.G2[s]) : 0.f;
            }
        }
        __syncthreads();

        // ---- T = (I + A)^-1: four 16 x 16 diagonal blocks by forward substitution,
        // then the blocks below the diagonal, one block diagonal at a time
        if (tid < CK) {
            const int bi = tid >> 4, c = tid & 15, o = 16 * bi;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m)
                    if (m >= c) acc = fmaf(Af[(o + r) * FS + o + m], x[m], acc);
                x[r] = r < c ? 0.f : (r == c ? 1.f : -acc);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Tf[(o + r) * FS + o + c] = x[r];
        }
        __syncthreads();
#pragma unroll 1
        for (int dd = 1; dd < 4; ++dd) {
            const int ne = (4 - dd) * 256;
            for (int e = tid; e < ne; e += NT) {  // R = sum_m A_im T_mj
                const int blk = e >> 8, i = dd + blk, j = blk, r = (e >> 4) & 15, c = e & 15;
                float acc = 0.f;
                for (int m = j; m < i; ++m)
#pragma unroll
                    for (int x = 0; x < 16; ++x)
                        acc = fmaf(Af[(16 * i + r) * FS + 16 * m + x], Tf[(16 * m + x) * FS + 16 * j + c], acc);
                Rf[(blk * 16 + r) * 17 + c] = acc;
            }
            __syncthreads();
            for (int e = tid; e < ne; e += NT) {  // T_ij = -T_ii R
                const int blk = e >> 8, i = dd + blk, j = blk, r = (e >> 4) & 15, c = e & 15;
                float acc = 0.f;
#pragma unroll
                for (int x = 0; x < 16; ++x) acc = fmaf(Tf[(16 * i + r) * FS + 16 * i + x], Rf[(blk * 16 + x) * 17 + c], acc);
                Tf[(16 * i + r) * FS + 16 * j + c] = -acc;
            }
            __syncthreads();
        }

        // ---- T1 = T diag(beta e^G rk), T2 = T diag(beta): canonical [64 t][64 s]
        {
            const int t = tid & 63, s0 = 8 * (tid >> 6);
            float v1[8], v2[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int s = s0 + k;
                const float x = s <= t ? Tf[t * FS + s] : 0.f;
                v1[k] = x * ps.f1[s];
                v2[k] = x * ps.bt[s];
            }
            const uint32_t off = cano(t, s0, 1024);
            put8(sm + KP0, sm + KP2, off, v1);
            put8(sm + KP1, sm + KP3, off, v2);
        }
        publish();  // B3

        // ---- W^T = K^T T1^T, U^T = V^T T2^T
        if (tid == 0) {
            tc::fence_after_sync();
            mma3c(tm + TM_W, smb + S_KTH, smb + S_KTL, TSBO, smb + KP0, smb + KP2, 1024, CK, id64, false);
            mma3c(tm + TM_U, smb + S_VTH, smb + S_VTL, TSBO, smb + KP1, smb + KP3, 1024, CK, id64, false);
            tc::mma_commit(&ps.mma_bar);
        }
        mma_wait();
        if (tid == 0 && c0 + CK < T) issue_raw(c0 + CK);  // the raw region is free again

        // ---- W operand [t][i] (swizzled, 64 rows) from W^T; M operand [t][s]
        {
            const int i = lb + lane;
            float w[16];
            tc::tmem_ld16(tc::taddr(tm, lb, TM_W + 16 * part), w);
            unsigned char *wh = sm + (i < 64 ? KP0 : KP1), *wl = sm + (i < 64 ? KP2 : KP3);
            const int ii = i & 63;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int t = 16 * part + k;
                const uint32_t off = (t >> 3) * 1024 + (t & 7) * 128 + ((((ii >> 3) ^ (t & 7)) & 7) << 4) + (ii & 7) * 2;
                const __half hv = __float2half_rn(w[k]);
                *reinterpret_cast<__half *>(wh + off) = hv;
                *reinterpret_cast<__half *>(wl + off) = __float2half_rn(w[k] - __half2float(hv));
            }
        }
        if (quad >= 2) {
            const int t = lb + lane - 64;
            float v[16];
            tc::tmem_ld16(tc::taddr(tm, lb, TM_G + 16 * part), v);
            const float rq = ps.rq[t], G2t = ps.G2[t];
            float m[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int s = 16 * part + k;
                m[k] = (s <= t && t < n) ? rq * ps.rk[s] * v[k] * ex2(G2t - ps.G2[s]) : 0.f;
            }
            put8(sm + S_MH, sm + S_ML, cano(t, 16 * part, 1024), m);
            put8(sm + S_MH, sm + S_ML, cano(t, 16 * part + 8, 1024), m + 8);
        }
        publish();  // B4

        // ---- V_new^T = U^T - S0^T W^T;  P^T = S0^T Q^T   (A = S0^T from TMEM)
        if (tid == 0) {
            tc::fence_after_sync();
#pragma unroll 1
            for (int ks = 0; ks < 8; ++ks) {
                const int k0 = (ks & 3) * 16;
                const uint32_t ash = tm + TM_SH + 8 * ks, asl = tm + TM_SL + 8 * ks;
                const uint64_t wh = tc::op_desc_sw128(smb + ((ks >> 2) ? KP1 : KP0), k0);
                const uint64_t wl = tc::op_desc_sw128(smb + ((ks >> 2) ? KP3 : KP2), k0);
                tc::mma_f16_ta(tm + TM_U, ash, wh, id64n, true);
                tc::mma_f16_ta(tm + TM_U, ash, wl, id64n, true);
                tc::mma_f16_ta(tm + TM_U, asl, wh, id64n, true);
                const uint32_t at = (ks >> 2) * 16384 + 8192;  // rows 64-127 (Q) of the atom
                const uint64_t qh = tc::op_desc_sw128(smb + S_KQH + at, k0);
                const uint64_t ql = tc::op_desc_sw128(smb + S_KQL + at, k0);
                tc::mma_f16_ta(tm + TM_G, ash, qh, id64, ks > 0);
                tc::mma_f16_ta(tm + TM_G, ash, ql, id64, true);
                tc::mma_f16_ta(tm + TM_G, asl, qh, id64, true);
            }
            tc::mma_commit(&ps.mma_bar);
        }
        mma_wait();

        // ---- V_new and V_new diag(e^{G_last - G} rk) operands [j][s]; S^T <- e^{G_last} S^T
        {
            const int j = lb + lane;
            float v[16], vd[16];
            tc::tmem_ld16(tc::taddr(tm, lb, TM_U + 16 * part), v);
#pragma unroll
            for (int k = 0; k < 16; ++k) vd[k] = v[k] * ps.ds[16 * part + k];
            put8(sm + S_VNH, sm + S_VNL, cano(j, 16 * part, 1024), v);
            put8(sm + S_VNH, sm + S_VNL, cano(j, 16 * part + 8, 1024), v + 8);
            put8(sm + S_VDH, sm + S_VDL, cano(j, 16 * part, 1024), vd);
            put8(sm + S_VDH, sm + S_VDL, cano(j, 16 * part + 8, 1024), vd + 8);
            const float gl = ps.egl;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float s[16];
                tc::tmem_ld16(tc::taddr(tm, lb, TM_S + 32 * part + 16 * q), s);
#pragma unroll
                for (int k = 0; k < 16; ++k) s[k] *= gl;
                tc::tmem_st16(tc::taddr(tm, lb, TM_S + 32 * part + 16 * q), s);
            }
        }
        publish();  // B5

        // ---- OV^T = V_new^T M^T;  S^T += (V_new diag(d))^T K
        if (tid == 0) {
            tc::fence_after_sync();
            mma3c(tm + TM_OV, smb + S_VNH, smb + S_VNL, 1024, smb + S_MH, smb + S_ML, 1024, CK, id64, false);
            mma3c(tm + TM_S, smb + S_VDH, smb + S_VDL, 1024, smb + S_KTH, smb + S_KTL, TSBO, CK, id128, true);
            tc::mma_commit(&ps.mma_bar);
        }
        mma_wait();
        cp = c0;
        np = n;
    }

    // the last chunk's output, the final state and the conv window
    const int nchunks = (T + CK - 1) / CK;
    if (warp >= 12) epilogue(cp, np, nchunks - 1);
    {
        float *So = a.state_out + head * D * D;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float s[16];
            tc::tmem_ld16(tc::taddr(tm, lb, TM_S + 32 * part + 16 * q), s);
#pragma unroll
            for (int k = 0; k < 16; ++k) So[(32 * part + 16 * q + k) * D + lb + lane] = s[k];
        }
    }
    if (clustered) cluster_wait_acquire();  // every CTA of the group has read the q/k window
    if (tid < NCONV) {
        const int tn = tid >> 7, c = tid & 127;
        if (tn == 2 || qk_owner) {
            const int ch = (tn == 0 ? chq : tn == 1 ? chk : chv) + c;
            float v[3];
#pragma unroll
            for (int r = 0; r < 3; ++r) {
                const int tau = T - 3 + r;
                v[r] = tau >= 0 ? ld_in(a.qkv, (static_cast<size_t>(b) * T + tau) * C + ch, 1)
                                : win[(3 + tau) * NCONV + tid];
            }
#pragma unroll
            for (int r = 0; r < 3; ++r) a.conv_out[(static_cast<size_t>(b) * 3 + r) * C + ch] = v[r];
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, 512);
    if (!ok && lane == 0) atomicOr(&g_c64_error, 1u);
}

}  // namespace

bool c64_shape(const gdn_shape_t &s)
{
    const int group = s.H_v / s.H_qk;
    const size_t C = 2 * static_cast<size_t>(s.H_qk) * s.d_k + static_cast<size_t>(s.H_v) * s.d_v;
    return s.gate_mode == GDN_GATE_PER_HEAD && s.d_k == D && s.d_v == D && s.in_dtype == GDN_BF16 &&
           s.chunk == CK && s.conv_K == 4 && group <= 8 && (C * 2) % 16 == 0 &&
           static_cast<long long>(s.B) * s.T < (1LL << 31) - 2 * CK;
}

bool c64_pointers_ok(const StepArgs &a)
{
    return (reinterpret_cast<uintptr_t>(a.qkv) & 15u) == 0 && (reinterpret_cast<uintptr_t>(a.z) & 15u) == 0;
}

cudaError_t launch_c64(const StepArgs &a, cudaStream_t stream)
{
    static bool attr_set[64];  // per device; benign race: every writer sets the same value
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(c64_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    CUtensorMap tq, tz;
    const uint64_t rows = static_cast<uint64_t>(a.B) * a.T;
    {   // qkv as [B*T rows][C channels] bf16, boxes of 67 rows x 128 channels
        const uint64_t dim[2] = {static_cast<uint64_t>(a.C), rows};
        const uint64_t stride[1] = {static_cast<uint64_t>(a.C) * 2};
        const uint32_t box[2] = {D, RAWR};
        if (!encode_tiled(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.qkv, dim, stride, box))
            return cudaErrorInvalidValue;
    }
    {   // z as [B*T][H_v][128] bf16, boxes of 64 tokens x 1 head x 128 channels
        const uint64_t dim[3] = {D, static_cast<uint64_t>(a.H_v), rows};
        const uint64_t stride[2] = {D * 2, static_cast<uint64_t>(a.H_v) * D * 2};
        const uint32_t box[3] = {D, 1, CK};
        if (!encode_tiled(&tz, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.z, dim, stride, box))
            return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.H_v, a.B, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    int n = 0;
    if (a.group > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = a.group;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, c64_prefill_kernel, a, tq, tz);
}

unsigned int take_c64_error()
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_c64_error, sizeof(v)) != cudaSuccess) return ~0u;
    if (v && cudaMemcpyToSymbol(g_c64_error, &zero, sizeof(zero)) != cudaSuccess) return ~0u;
    return v;
}

}  // namespace gdn
