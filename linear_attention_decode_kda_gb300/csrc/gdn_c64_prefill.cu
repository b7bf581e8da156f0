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
constexpr int NCONV = 384;   // q, k, v channels of one value head
constexpr int RAWR = CK + 3; // input rows a chunk reads: its 64 and the 3 before

// Dynamic shared memory (bytes from a 1024-byte aligned base).  Operands are K-major
// in the canonical no-swizzle layout: 8 x 16-byte core matrices, LBO bytes between
// neighbours along K, SBO bytes between 8-row groups.
// [K; Q]: rows 0-63 K, 64-127 Q, 128 channels; LBO 144 spreads the conv threads'
// stores of one token row over all banks.
constexpr uint32_t QLBO = 144, QSBO = 16 * QLBO, Q_BYTES = 16 * QSBO;
constexpr uint32_t S_KQH = 0, S_KQL = Q_BYTES;
// K^T and V^T: [128 channels][64 tokens]; SBO 1040 spreads the stores of 8-token rows.
constexpr uint32_t TSBO = 1040, T_BYTES = 16 * TSBO;
constexpr uint32_t S_KTH = 2 * Q_BYTES, S_KTL = S_KTH + T_BYTES, S_VTH = S_KTL + T_BYTES,
                   S_VTL = S_VTH + T_BYTES;
constexpr uint32_t S_RAW = ((S_VTL + T_BYTES + 1023) / 1024) * 1024;  // q, k, v boxes [67][128] bf16
constexpr uint32_t RAW_BOX = RAWR * D * 2;
constexpr uint32_t S_Z = ((S_RAW + 3 * RAW_BOX + 1023) / 1024) * 1024;  // z box [64][128] bf16
constexpr uint32_t S_WIN = S_Z + CK * D * 2;                            // fp32 window [3][384]
constexpr uint32_t SMEM_USED = S_WIN + 3 * NCONV * 4;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for aligning the base
static_assert(SMEM_BYTES + 4096 <= 232448, "shared memory per block");
// Reused regions.  The K rows of [K; Q] are dead after the Gram product: they take
// T1 and T2 ([64][64], SBO 1024, 8 KB each), then W (the [W; Q] operand of the S0 product).
constexpr uint32_t S_T1H = S_KQH, S_T2H = S_KQH + 8192, S_T1L = S_KQL, S_T2L = S_KQL + 8192;
static_assert(8192 + 8192 <= 8 * QSBO, "T1 and T2 inside the K rows");
// M ([64][64], SBO 1024) takes V^T's place after the U product.
constexpr uint32_t S_MH = S_VTH, S_ML = S_VTH + 8192;
static_assert(S_ML + 8192 <= S_VTH + T_BYTES, "M operand");
// fp32 scratch of the inverse inside the raw-row region (free between the conv and
// the next chunk's copy): A and T [64][68], the block products [3][16][20] (rows
// 16-byte aligned for 128-bit loads).
constexpr int FS = CK + 4, RS = 20;
constexpr uint32_t S_AF = S_RAW, S_TF = S_AF + CK * FS * 4, S_RF = S_TF + CK * FS * 4;
static_assert(S_RF + 3 * 16 * RS * 4 <= S_RAW + 3 * RAW_BOX, "inverse scratch");

// TMEM columns.
constexpr uint32_t TM_S = 0;     // 128: S^T fp32
constexpr uint32_t TM_SH = 128;  // 64: S0^T fp16 hi, two to a column (A of the S0 product) ...
constexpr uint32_t TM_SL = 192;  // 64: ... and lo; after that product:
constexpr uint32_t TM_VNH = 128, TM_VNL = 160, TM_VDH = 192, TM_VDL = 224;  // V_new, V_new diag(d)
constexpr uint32_t TM_X1 = 256;  // 64: W^T, then V_new^T M^T (OV)
constexpr uint32_t TM_U = 320;   // 64: U^T
constexpr uint32_t TM_X3 = 384;  // 64: Gram, then S0^T W^T (PW)
constexpr uint32_t TM_PQ = 448;  // 64: S0^T Q^T (written with PW as one N = 128 product)

__device__ unsigned int g_c64_error;  // bit 0: a bounded mbarrier wait gave up

struct C64Shared {
    float G2[CK];          // cumulative log2-decay inside the chunk
    float bt[CK];          // beta (0 past the chunk's end)
    float nqp[2][CK], nkp[2][CK];  // |q|^2, |k|^2 of the raw rows, per half of the channels
    float rk[CK];          // 1 / |k|
    float rq[CK];          // q_scale / |q|
    float f1[CK];          // beta_s e^{G_s} rk_s
    float ds[CK];          // e^{G_last - G_s} rk_s
    float cq[2][CK];       // e^{G_t} rq_t, by chunk parity
    float osq[4][CK];      // per TMEM quadrant: partial sums of o^2
    float rinv[CK];
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

// Byte offset of element (r, k) of a canonical K-major operand.
__device__ __forceinline__ uint32_t cano(int r, int k, uint32_t lbo, uint32_t sbo)
{
    return static_cast<uint32_t>(r >> 3) * sbo + static_cast<uint32_t>(k >> 3) * lbo +
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

__device__ __forceinline__ void tmem_st8u_nowait(uint32_t taddr, const uint32_t (&w)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Descriptor of the K step at column k0 of a canonical operand.
__device__ __forceinline__ uint64_t cdesc(uint32_t base, int k0, uint32_t lbo, uint32_t sbo)
{
    return tc::op_desc_strided(base + static_cast<uint32_t>(k0 >> 3) * lbo, lbo, sbo);
}

// D (+)= (A_hi + A_lo)(B_hi + B_lo)^T without lo*lo, both operands canonical in shared memory.
__device__ __forceinline__ void mma3c(uint32_t d, uint32_t ah, uint32_t al, uint32_t asbo, uint32_t bh,
                                      uint32_t bl, uint32_t bsbo, int kdim, uint32_t idesc, bool acc)
{
    for (int k0 = 0; k0 < kdim; k0 += 16) {
        const uint64_t dah = cdesc(ah, k0, 128, asbo), dal = cdesc(al, k0, 128, asbo);
        const uint64_t dbh = cdesc(bh, k0, 128, bsbo), dbl = cdesc(bl, k0, 128, bsbo);
        tc::mma_f16(d, dah, dbh, idesc, acc || k0 > 0);
        tc::mma_f16(d, dah, dbl, idesc, true);
        tc::mma_f16(d, dal, dbh, idesc, true);
    }
}

// The same with A in TMEM (hi at column ah, lo at al; K step k0 at column + k0 / 2).
__device__ __forceinline__ void mma3t(uint32_t d, uint32_t ah, uint32_t al, uint32_t bh, uint32_t bl,
                                      uint32_t blbo, uint32_t bsbo, int kdim, uint32_t idesc, bool acc)
{
    for (int k0 = 0; k0 < kdim; k0 += 16) {
        const uint64_t dbh = cdesc(bh, k0, blbo, bsbo), dbl = cdesc(bl, k0, blbo, bsbo);
        tc::mma_f16_ta(d, ah + k0 / 2, dbh, idesc, acc || k0 > 0);
        tc::mma_f16_ta(d, ah + k0 / 2, dbl, idesc, true);
        tc::mma_f16_ta(d, al + k0 / 2, dbh, idesc, true);
    }
}

__device__ __forceinline__ void publish()
{
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
}

__device__ __forceinline__ void bar_a() { asm volatile("bar.sync 1, 256;" ::: "memory"); }  // warps 0-7
__device__ __forceinline__ void bar_b() { asm volatile("bar.sync 2, 256;" ::: "memory"); }  // warps 8-15

__global__ void __launch_bounds__(NT, 1)
c64_prefill_kernel(const StepArgs a, const __grid_constant__ CUtensorMap tm_qkv,
                   const __grid_constant__ CUtensorMap tm_z)
{
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    __shared__ __align__(16) C64Shared ps;
    unsigned char *sm = sm_raw + ((1024u - (tc::smem_u32(sm_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, part = warp >> 2, lb = 32 * quad;
    const bool grp_a = warp < 8;  // warps 0-7: Gram, A, inverse; 8-15: state copy, output
    const int h = blockIdx.x, b = blockIdx.y, hq = h / a.group;
    const int T = a.T, Ts = a.Ts, C = a.C, H = a.H_v;
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
        const int row = b * Ts + c0 - 3;  // rows before the tensor read as zero
        tma_load_2d(sm + S_RAW, &tm_qkv, chq, row, &ps.raw_full);
        tma_load_2d(sm + S_RAW + RAW_BOX, &tm_qkv, chk, row, &ps.raw_full);
        tma_load_2d(sm + S_RAW + 2 * RAW_BOX, &tm_qkv, chv, row, &ps.raw_full);
    };
    if (tid == 0) issue_raw(0);

    // the kept conv window (fp32; the first chunk's 3 earlier rows) and the initial state
    if (tid < NCONV) {
        const int tn = tid >> 7, c = tid & 127;
        const int ch = (tn == 0 ? chq : tn == 1 ? chk : chv) + c;
#pragma unroll
        for (int r = 0; r < 3; ++r) win[r * NCONV + tid] = a.conv_in[(static_cast<size_t>(b) * 3 + r) * C + ch];
    }
    {   // S[i][j] -> TMEM S^T (lane j, column i); this warp takes rows 32 part .. 32 part + 31
        const float *Sg = a.state_in + head * D * D;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) w[k] = __float_as_uint(Sg[(32 * part + 16 * q + k) * D + lb + lane]);
            tc::tmem_st16u_nowait(tc::taddr(tm, lb, TM_S + 32 * part + 16 * q), w);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    if (clustered) cluster_arrive_relaxed();  // this CTA has read the shared q/k window

    // conv: every warp takes tokens 8 tb .. 8 tb + 7 and channels 64 hf + 2 lane, + 1
    // of q, k and v
    const int hf = (warp >> 3) & 1, tb = warp & 7;
    float4 cw[3][2];
#pragma unroll
    for (int tn = 0; tn < 3; ++tn) {
        const int ch0 = (tn == 0 ? chq : tn == 1 ? chk : chv) + 64 * hf + 2 * lane;
        cw[tn][0] = reinterpret_cast<const float4 *>(a.conv_w)[ch0];
        cw[tn][1] = reinterpret_cast<const float4 *>(a.conv_w)[ch0 + 1];
    }

    // gate logits of the next chunk: warp 15, tokens 2 lane and 2 lane + 1
    const float A_h = expf(a.A_log[h]);
    const float dt_h = a.dt_bias[h];
    float fx[2] = {0.f, 0.f}, bx[2] = {0.f, 0.f};
    auto load_gates = [&](int c0) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int t = c0 + 2 * lane + u;
            if (t < T) {
                const size_t e = (static_cast<size_t>(b) * Ts + t) * H + h;
                fx[u] = ld_in(a.f, e, 1);
                bx[u] = ld_in(a.beta, e, 1);
            }
        }
    };
    if (warp == 15) load_gates(0);
    const float nw = a.norm_w[lb + lane];  // output-norm weight of this lane's column

    bool ok = true;
    uint32_t mma_ph = 0;
    auto mma_wait = [&](bool wait) {
        if (wait && ok) ok = mbar_wait_suspend_bounded(&ps.mma_bar, mma_ph);
        mma_ph ^= 1u;
        tc::fence_after_sync();
    };
    const uint32_t smb = tc::smem_u32(sm);
    const uint32_t id64 = tc::idesc_f16(128, 64, false), id128 = tc::idesc_f16(128, 128, false);

    // The output of chunk (cp, np) from TMEM: o = PQ e^{G_t} rq_t + OV, the gated
    // RMSNorm over the 128 columns, y stored.  Warps 8-15: lane = column j, tokens
    // 32 th .. 32 th + 31.
    auto epilogue = [&](int cp, int np, int it) {
        if (ok) ok = mbar_wait_suspend_bounded(&ps.z_full, static_cast<uint32_t>(it & 1));
        const int j = lb + lane, th = part & 1;
        const float *cq = ps.cq[it & 1];
        float o[32], v[32];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float p16[16], ov16[16];
            tc::tmem_ld16(tc::taddr(tm, lb, TM_PQ + 32 * th + 16 * q), p16);
            tc::tmem_ld16(tc::taddr(tm, lb, TM_X1 + 32 * th + 16 * q), ov16);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float x = fmaf(p16[k], cq[32 * th + 16 * q + k], ov16[k]);
                o[16 * q + k] = x;
                v[16 * q + k] = x * x;
            }
        }
        ps.osq[quad][32 * th + lane] = reduce_scatter32(v, lane);
        bar_b();
        if (tid < 256 + CK) {
            const int t = tid - 256;
            const float m = (ps.osq[0][t] + ps.osq[1][t] + ps.osq[2][t] + ps.osq[3][t]) * (1.0f / D);
            ps.rinv[t] = rsqrtf(m + a.eps_norm);
        }
        bar_b();
        // y = o rinv w gate(z) for the 32 tokens, then the stores (row stride H * D)
        const unsigned char *zs = sm + S_Z + (32 * th * D + j) * 2;
        const bool sig = a.sig_gate != 0;
#pragma unroll
        for (int k4 = 0; k4 < 32; k4 += 4) {
            const float4 r4 = *reinterpret_cast<const float4 *>(&ps.rinv[32 * th + k4]);
            const float rv[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float zz = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(zs + (k4 + k) * D * 2));
                const float e = __expf(-zz);
                const float gz = __fdividef(sig ? 1.0f : zz, 1.0f + e);
                o[k4 + k] *= rv[k] * nw * gz;
            }
        }
        const size_t row0 = (static_cast<size_t>(b) * Ts + cp + 32 * th) * H + h;
        const int nk = min(32, np - 32 * th);  // tokens of this half inside the chunk
        if (a.out_bf16) {
            __nv_bfloat16 *yo = reinterpret_cast<__nv_bfloat16 *>(a.out) + row0 * D + j;
#pragma unroll
            for (int k = 0; k < 32; ++k)
                if (k < nk) yo[static_cast<size_t>(k) * H * D] = __float2bfloat16_rn(o[k]);
        } else {
            float *yo = reinterpret_cast<float *>(a.out) + row0 * D + j;
#pragma unroll
            for (int k = 0; k < 32; ++k)
                if (k < nk) yo[static_cast<size_t>(k) * H * D] = o[k];
        }
        fence_proxy_async_smem();  // the z stage is read: the next copy may land there
    };

    int cp = 0, np = 0;
#pragma unroll 1
    for (int c0 = 0, it = 0; c0 < T; c0 += CK, ++it) {
        const int n = min(CK, T - c0);

        // ---- gates of this chunk (warp 15)
        if (warp == 15) {
            float g[2], bb[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const bool in = 2 * lane + u < n;
                g[u] = in ? -A_h * softplus_fast(fx[u] + dt_h) : 0.f;
                bb[u] = in ? sigmoid_fast(bx[u]) : 0.f;
            }
            if (c0 + CK < T) load_gates(c0 + CK);
            float sc = g[0] + g[1];
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

        // ---- conv + SiLU: q -> Q rows, k -> K rows and K^T, v -> V^T (all warps)
        if (ok) ok = mbar_wait_suspend_bounded(&ps.raw_full, static_cast<uint32_t>(it & 1));
#pragma unroll
        for (int tn = 0; tn < 3; ++tn) {
            const unsigned char *raw = sm + S_RAW + tn * RAW_BOX;
            const int cl = 64 * hf + 2 * lane;  // first of this lane's two channels in the tensor
            float xw[3][2];
#pragma unroll
            for (int r = 0; r < 3; ++r) {
                if (c0 == 0 && tb == 0) {
                    xw[r][0] = win[r * NCONV + tn * 128 + cl];
                    xw[r][1] = win[r * NCONV + tn * 128 + cl + 1];
                } else {
                    const uint32_t u = *reinterpret_cast<const uint32_t *>(raw + ((8 * tb + r) * D + cl) * 2);
                    xw[r][0] = __uint_as_float(u << 16);
                    xw[r][1] = __uint_as_float(u & 0xffff0000u);
                }
            }
            uint32_t hn[8], ln[8];
            float nrm[8];
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const int t = 8 * tb + rr;
                const uint32_t u = *reinterpret_cast<const uint32_t *>(raw + ((t + 3) * D + cl) * 2);
                const float x0 = __uint_as_float(u << 16), x1 = __uint_as_float(u & 0xffff0000u);
                float acc0 = cw[tn][0].x * xw[0][0], acc1 = cw[tn][1].x * xw[0][1];
                acc0 = fmaf(cw[tn][0].y, xw[1][0], acc0);
                acc1 = fmaf(cw[tn][1].y, xw[1][1], acc1);
                acc0 = fmaf(cw[tn][0].z, xw[2][0], acc0);
                acc1 = fmaf(cw[tn][1].z, xw[2][1], acc1);
                acc0 = fmaf(cw[tn][0].w, x0, acc0);
                acc1 = fmaf(cw[tn][1].w, x1, acc1);
                const float y0 = t < n ? silu_fast(acc0) : 0.f, y1 = t < n ? silu_fast(acc1) : 0.f;
                xw[0][0] = xw[1][0]; xw[1][0] = xw[2][0]; xw[2][0] = x0;
                xw[0][1] = xw[1][1]; xw[1][1] = xw[2][1]; xw[2][1] = x1;
                nrm[rr] = y0 * y0 + y1 * y1;
                split2(y0, y1, hn[rr], ln[rr]);
                if (tn < 2) {  // row t (k) or 64 + t (q) of [K; Q]
                    const uint32_t off = cano(tn == 0 ? 64 + t : t, cl, QLBO, QSBO);
                    *reinterpret_cast<uint32_t *>(sm + S_KQH + off) = hn[rr];
                    *reinterpret_cast<uint32_t *>(sm + S_KQL + off) = ln[rr];
                }
            }
            if (tn >= 1) {  // K^T / V^T rows cl, cl + 1: the block's 8 tokens, 16 bytes each
                unsigned char *th = sm + (tn == 1 ? S_KTH : S_VTH);
                unsigned char *tl = sm + (tn == 1 ? S_KTL : S_VTL);
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    const uint32_t sel = cc ? 0x7632u : 0x5410u;
                    const uint4 vh = make_uint4(__byte_perm(hn[0], hn[1], sel), __byte_perm(hn[2], hn[3], sel),
                                                __byte_perm(hn[4], hn[5], sel), __byte_perm(hn[6], hn[7], sel));
                    const uint4 vl = make_uint4(__byte_perm(ln[0], ln[1], sel), __byte_perm(ln[2], ln[3], sel),
                                                __byte_perm(ln[4], ln[5], sel), __byte_perm(ln[6], ln[7], sel));
                    const uint32_t off = cano(cl + cc, 8 * tb, 128, TSBO);
                    *reinterpret_cast<uint4 *>(th + off) = vh;
                    *reinterpret_cast<uint4 *>(tl + off) = vl;
                }
            }
            if (tn < 2) {
                const float tot = reduce8(nrm, lane);
                if ((lane & 3) == 0) {
                    const int t = 8 * tb + ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
                    (tn == 0 ? ps.nqp : ps.nkp)[hf][t] = tot;
                }
            }
        }
        publish();  // B1: the conv operands, the gates and the norms are written

        if (grp_a) {
            // ---- warps 0-7: the Gram product [K; Q] K^T (hi.hi + hi.lo + lo.hi), the
            // per-token factors, A, and T = (I + A)^-1
            if (tid == 0) {
                tc::fence_after_sync();
#pragma unroll 1
                for (int k0 = 0; k0 < D; k0 += 16) {
                    const uint64_t ah = cdesc(smb + S_KQH, k0, QLBO, QSBO), al = cdesc(smb + S_KQL, k0, QLBO, QSBO);
                    tc::mma_f16(tm + TM_X3, ah, ah, id64, k0 > 0);  // B = rows 0-63 (K)
                    tc::mma_f16(tm + TM_X3, ah, al, id64, true);
                    tc::mma_f16(tm + TM_X3, al, ah, id64, true);
                }
                tc::mma_commit(&ps.mma_bar);
            }
            if (tid < CK) {
                const int t = tid;
                const bool in = t < n;
                const float rk = in ? rsqrtf(ps.nkp[0][t] + ps.nkp[1][t] + a.eps_l2) : 0.f;
                const float rq = in ? a.q_scale * rsqrtf(ps.nqp[0][t] + ps.nqp[1][t] + a.eps_l2) : 0.f;
                const float G2t = ps.G2[t], G2l = ps.G2[n - 1];
                ps.rk[t] = rk;
                ps.rq[t] = rq;
                ps.f1[t] = ps.bt[t] * ex2(G2t) * rk;
                ps.ds[t] = in ? ex2(G2l - G2t) * rk : 0.f;
                ps.cq[it & 1][t] = ex2(G2t) * rq;
            }
            bar_a();
            mma_wait(true);
            // A = beta_t rk_t rk_s (k.k) e^{G_t - G_s} (s < t): lanes 0-63 hold the K rows
            if (quad < 2) {
                const int t = lb + lane;
                const float bt = ps.bt[t] * ps.rk[t], G2t = ps.G2[t];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    float v[16];
                    tc::tmem_ld16(tc::taddr(tm, lb, TM_X3 + 32 * part + 16 * q), v);
#pragma unroll
                    for (int k4 = 0; k4 < 16; k4 += 4) {
                        float e[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int s = 32 * part + 16 * q + k4 + k;
                            e[k] = (s < t && t < n) ? bt * ps.rk[s] * v[k4 + k] * ex2(G2t - ps.G2[s]) : 0.f;
                        }
                        *reinterpret_cast<float4 *>(Af + t * FS + 32 * part + 16 * q + k4) = make_float4(e[0], e[1], e[2], e[3]);
                    }
                }
            }
            bar_a();
            // four 16 x 16 diagonal blocks by forward substitution (x[m] = 0 for m < c)
            if (tid < CK) {
                const int bi = tid >> 4, c = tid & 15, o = 16 * bi;
                float x[16], ar[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
#pragma unroll
                    for (int m4 = 0; m4 < r; m4 += 4) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(Af + (o + r) * FS + o + m4);
                        ar[m4] = a4.x; ar[m4 + 1] = a4.y; ar[m4 + 2] = a4.z; ar[m4 + 3] = a4.w;
                    }
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int m = 0; m < r; ++m) acc[m & 3] = fmaf(ar[m], x[m], acc[m & 3]);
                    x[r] = r < c ? 0.f : (r == c ? 1.f : -((acc[0] + acc[1]) + (acc[2] + acc[3])));
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Tf[(o + r) * FS + o + c] = x[r];
            }
            bar_a();
            // the blocks below the diagonal, one block diagonal at a time:
            // T_ij = -T_ii sum_{m=j}^{i-1} A_im T_mj; a thread takes 4 columns of one row
#pragma unroll 1
            for (int dd = 1; dd < 4; ++dd) {
                const int blk = tid >> 6, i = dd + blk, j = blk, r = (tid >> 2) & 15, c4 = 4 * (tid & 3);
                const bool act = blk < 4 - dd;
                if (act) {
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int m = j; m < i; ++m)
#pragma unroll
                        for (int x4 = 0; x4 < 16; x4 += 4) {
                            const float4 a4 = *reinterpret_cast<const float4 *>(Af + (16 * i + r) * FS + 16 * m + x4);
                            const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                            for (int xx = 0; xx < 4; ++xx) {
                                const float4 t4 = *reinterpret_cast<const float4 *>(Tf + (16 * m + x4 + xx) * FS + 16 * j + c4);
                                acc.x = fmaf(av[xx], t4.x, acc.x);
                                acc.y = fmaf(av[xx], t4.y, acc.y);
                                acc.z = fmaf(av[xx], t4.z, acc.z);
                                acc.w = fmaf(av[xx], t4.w, acc.w);
                            }
                        }
                    *reinterpret_cast<float4 *>(Rf + (blk * 16 + r) * RS + c4) = acc;
                }
                bar_a();
                if (act) {
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int x4 = 0; x4 < 16; x4 += 4) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(Tf + (16 * i + r) * FS + 16 * i + x4);
                        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                        for (int xx = 0; xx < 4; ++xx) {
                            const float4 r4 = *reinterpret_cast<const float4 *>(Rf + (blk * 16 + x4 + xx) * RS + c4);
                            acc.x = fmaf(av[xx], r4.x, acc.x);
                            acc.y = fmaf(av[xx], r4.y, acc.y);
                            acc.z = fmaf(av[xx], r4.z, acc.z);
                            acc.w = fmaf(av[xx], r4.w, acc.w);
                        }
                    }
                    *reinterpret_cast<float4 *>(Tf + (16 * i + r) * FS + 16 * j + c4) =
                        make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
                }
                bar_a();
            }
        } else {
            // ---- warps 8-15: the fp16 copy of the state this chunk starts from (A of its
            // S0 product), the state scaled by e^{G_last} for its update, and the previous
            // chunk's output
            mma_wait(false);
            const float gl = ex2(ps.G2[n - 1]);
            const int c0s = 64 * (part & 1);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float s[16];
                tc::tmem_ld16(tc::taddr(tm, lb, TM_S + c0s + 16 * q), s);
                uint32_t hw[8], lw[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) split2(s[2 * k], s[2 * k + 1], hw[k], lw[k]);
                tmem_st8u_nowait(tc::taddr(tm, lb, TM_SH + c0s / 2 + 8 * q), hw);
                tmem_st8u_nowait(tc::taddr(tm, lb, TM_SL + c0s / 2 + 8 * q), lw);
#pragma unroll
                for (int k = 0; k < 16; ++k) s[k] *= gl;
                tc::tmem_st16(tc::taddr(tm, lb, TM_S + c0s + 16 * q), s);
            }
            if (it > 0) epilogue(cp, np, it - 1);
        }
        publish();  // B2
        if (tid == 0) {  // the previous output has read the z stage: this chunk's rows
            mbar_expect_tx(&ps.z_full, CK * D * 2);
            tma_load_3d(sm + S_Z, &tm_z, 0, h, b * Ts + c0, &ps.z_full);
        }

        // ---- T1 = T diag(beta e^G rk), T2 = T diag(beta): [64 t][64 s] into the K rows
        {
            const int t = tid & 63, s0 = 8 * (tid >> 6);
            float v1[8], v2[8];
            const float4 ta = *reinterpret_cast<const float4 *>(Tf + t * FS + s0);
            const float4 tb4 = *reinterpret_cast<const float4 *>(Tf + t * FS + s0 + 4);
            const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb4.x, tb4.y, tb4.z, tb4.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int s = s0 + k;
                const float x = s <= t ? tv[k] : 0.f;
                v1[k] = x * ps.f1[s];
                v2[k] = x * ps.bt[s];
            }
            const uint32_t off = cano(t, s0, 128, 1024);
            put8(sm + S_T1H, sm + S_T1L, off, v1);
            put8(sm + S_T2H, sm + S_T2L, off, v2);
        }
        publish();  // B3

        // ---- W^T = K^T T1^T, U^T = V^T T2^T
        if (tid == 0) {
            tc::fence_after_sync();
            mma3c(tm + TM_X1, smb + S_KTH, smb + S_KTL, TSBO, smb + S_T1H, smb + S_T1L, 1024, CK, id64, false);
            mma3c(tm + TM_U, smb + S_VTH, smb + S_VTL, TSBO, smb + S_T2H, smb + S_T2L, 1024, CK, id64, false);
            tc::mma_commit(&ps.mma_bar);
        }
        mma_wait(true);
        if (tid == 0 && c0 + CK < T) issue_raw(c0 + CK);  // the raw region is free again

        // ---- W operand: rows 0-63 of [W; Q] from W^T (lane = channel i);
        // M operand [t][s] from the Gram's Q rows (lanes 64-127)
        {
            const int i = lb + lane;
            float w[16];
            tc::tmem_ld16(tc::taddr(tm, lb, TM_X1 + 16 * part), w);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const uint32_t off = cano(16 * part + k, i, QLBO, QSBO);
                const __half hv = __float2half_rn(w[k]);
                *reinterpret_cast<__half *>(sm + S_KQH + off) = hv;
                *reinterpret_cast<__half *>(sm + S_KQL + off) = __float2half_rn(w[k] - __half2float(hv));
            }
        }
        if (quad >= 2) {
            const int t = lb + lane - 64;
            float v[16];
            tc::tmem_ld16(tc::taddr(tm, lb, TM_X3 + 16 * part), v);
            const float rq = ps.rq[t], G2t = ps.G2[t];
            float m[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int s = 16 * part + k;
                m[k] = (s <= t && t < n) ? rq * ps.rk[s] * v[k] * ex2(G2t - ps.G2[s]) : 0.f;
            }
            put8(sm + S_MH, sm + S_ML, cano(t, 16 * part, 128, 1024), m);
            put8(sm + S_MH, sm + S_ML, cano(t, 16 * part + 8, 128, 1024), m + 8);
        }
        publish();  // B4

        // ---- [PW | PQ] = S0^T [W; Q]^T, one N = 128 product with A = S0^T from TMEM
        if (tid == 0) {
            tc::fence_after_sync();
            mma3t(tm + TM_X3, tm + TM_SH, tm + TM_SL, smb + S_KQH, smb + S_KQL, QLBO, QSBO, D, id128, false);
            tc::mma_commit(&ps.mma_bar);
        }
        mma_wait(true);

        // ---- V_new = U - PW and V_new diag(e^{G_last - G} rk), fp16 hi / lo, into TMEM
        {
            float u[16], pw[16];
            tc::tmem_ld16(tc::taddr(tm, lb, TM_U + 16 * part), u);
            tc::tmem_ld16(tc::taddr(tm, lb, TM_X3 + 16 * part), pw);
            uint32_t nh[8], nl[8], dh[8], dl[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float v0 = u[2 * k] - pw[2 * k], v1 = u[2 * k + 1] - pw[2 * k + 1];
                split2(v0, v1, nh[k], nl[k]);
                split2(v0 * ps.ds[16 * part + 2 * k], v1 * ps.ds[16 * part + 2 * k + 1], dh[k], dl[k]);
            }
            tmem_st8u_nowait(tc::taddr(tm, lb, TM_VNH + 8 * part), nh);
            tmem_st8u_nowait(tc::taddr(tm, lb, TM_VNL + 8 * part), nl);
            tmem_st8u_nowait(tc::taddr(tm, lb, TM_VDH + 8 * part), dh);
            tmem_st8u_nowait(tc::taddr(tm, lb, TM_VDL + 8 * part), dl);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        tc::fence_before_sync();
        __syncthreads();  // B5

        // ---- OV = V_new^T M^T;  S^T += (V_new diag(d))^T K
        if (tid == 0) {
            tc::fence_after_sync();
            mma3t(tm + TM_X1, tm + TM_VNH, tm + TM_VNL, smb + S_MH, smb + S_ML, 128, 1024, CK, id64, false);
            mma3t(tm + TM_S, tm + TM_VDH, tm + TM_VDL, smb + S_KTH, smb + S_KTL, 128, TSBO, CK, id128, true);
            tc::mma_commit(&ps.mma_bar);
        }
        mma_wait(true);
        cp = c0;
        np = n;
    }

    // the last chunk's output, the final state and the conv window
    const int nchunks = (T + CK - 1) / CK;
    if (!grp_a) epilogue(cp, np, nchunks - 1);
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
                v[r] = tau >= 0 ? ld_in(a.qkv, (static_cast<size_t>(b) * Ts + tau) * C + ch, 1)
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
    const uint64_t rows = static_cast<uint64_t>(a.B) * a.Ts;
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
