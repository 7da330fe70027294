// chunk_tc.cu -- chunked forward of the gated delta rule on the tensor cores
// (tcgen05 + tensor memory + TMA), bf16 inputs, dk = 128, dv % 128 == 0.
//
// "Gated Delta Networks: Improving Mamba2 with Delta Rule", §3.3, split into the
// two kernels its structure suggests:
//
// ut_tc_kernel -- one CTA per (chunk, head), all chunks in parallel (the
//   chunk-local UT transform, with the prologue folded in).  Per chunk of
//   C = 64 row-stacked tokens:
//     prologue   b_r = sum_{i<=r} g_i (chunk-local, base 2 internally);
//                rk_r = 1/||k_r||, rq_r = scale/||q_r||
//     P1 (MMA)   G = [K; Q] K^T                               (128 x 64, fp32)
//     masks      L_ri   = beta_r e^{b_r-b_i} rk_r rk_i G_ri,   i <  r   (the system)
//                Aqk_ri = e^{b_r-b_i} rq_r rk_i G_(64+r)i,     i <= r   (Q K^T o Gamma)
//     solve      T = (I + L)^{-1} (16x16 diagonal blocks by forward substitution,
//                then the block rule for the 16->32 and 32->64 merges)
//                T' = T diag(beta),  T'' = T diag(beta e^b rk)
//     P2 (MMA)   W~^T = K^T T''^T   (W<- of the pages for the normalised keys)
//   and writes T', W~^T, Aqk (bf16, already in the 128-B-swizzled tile layout
//   the recurrence kernel's MMAs read) plus the per-row factors
//   fq_r = e^{b_r} rq_r, fk_r = e^{b_C - b_r} rk_r and e^{b_C} to the workspace.
//
// recur_tc_kernel -- one CTA per (sequence, head, 128-row slice of S), the
//   sequential inter-chunk recurrence with the fp32 state resident in tensor
//   memory for the whole sequence:
//     a1, a2     V_new^T = V^T T'^T - S W~^T                  ((U~ - W<- S^T)^T)
//     c2         S <- e^{b_C} S + (V_new^T diag(fk)) K         (K-> folded into V_new)
//     b, c1      O^T = diag-scaled (S Q^T) + V_new^T Aqk^T     (O = Q<- S^T + Aqk V_new)
//
// All gate ratios are exp(b_r - b_i) with i <= r (never 1/gamma), so heavy
// decay cannot overflow.  The output mask is the decay mask Gamma
// ("【论文解读】Gated Delta Network", §二(一)2(3)).  Every wait is bounded
// (globaltimer); a timeout records kDevErrTimeout in the workspace header,
// raises a CTA-wide abort flag, and all roles unwind to the common exit, where
// tensor memory is released.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr uint32_t LDL = 68;           // fp32 row pitch of T (16-B aligned rows for vector loads)
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s: legitimate waits are microseconds

// Per (chunk, head) block of the workspace written by ut_tc_kernel.
// All tiles are 128-B-swizzled rows of 64 bf16 (8 KB per 64 rows).
// T' is carried as a bf16 hi + lo pair (the two K-major B tiles of a1, back to back); the
// operands of the c product (Aqk^T, K->, and V_new^T in the recurrence) are fp16, whose 11
// significand bits keep the intra-chunk products accurate where they nearly cancel (nearly
// parallel keys with beta close to 2).
constexpr uint32_t PB_TP = 0;          // T'_hi [64 r][64 i] bf16, then T'_lo  (K-major B of a1)
constexpr uint32_t PB_W = 16384;       // W~    [d-block][64 r][64 d]  x 2    (K-major B of a2), bf16
constexpr uint32_t PB_AQT = 32768;     // Aqk^T [64 i][64 r] fp16             (MN-major B of c)
constexpr uint32_t PB_KT = 40960;      // K->   [d-block][64 r][64 d]  x 2    (MN-major B of c), fp16
constexpr uint32_t PB_SC = 57344;      // fq[64], e^{b_C}, range flag, 2 x 0 (fp32)
constexpr uint32_t kPrepBlock = 57856;
// With the block prologue fused in, the chunk-local kernel also leaves the convolved Q tile
// (both 64-wide d-blocks, in the TMA box layout) for the recurrence.
constexpr uint32_t PB_QC = kPrepBlock;
constexpr uint32_t kPrepBlockFused = kPrepBlock + 16384;
constexpr uint32_t kWsHeader = 1024;   // device error word + padding

// ---- ut_tc_kernel shared memory
constexpr int kThreadsUt = 160;        // warp 0: TMA, MMA, TMEM; warps 1-4: 128 "prep" threads
constexpr uint32_t U_QK = 0;           // [K kb0][Q kb0][K kb1][Q kb1], 8 KB each
// Once the Gram product has read Q, its two tiles are reused:
constexpr uint32_t U_TPP = 8192;       // T'' (bf16, 8 KB): A of the W~ product; its padding rows
                                       // 64-127 read the K tile behind it (results not used)
constexpr uint32_t U_MT = 24576;       // solve scratch (4 KB), then
constexpr uint32_t U_TPL = 24576;      // T''_lo (bf16, 8 KB): T'' - T''_hi; its padding rows read U_A
constexpr uint32_t U_A = 32768;        // L, then T, in place: fp32 [64][LDL]
constexpr uint32_t U_SC = U_A + 64 * LDL * 4;     // b, beta, rk, rq, cw, ecol, cq[3], misc, fk  [11][64] fp32
constexpr uint32_t U_BAR = U_SC + 11 * 64 * 4;
constexpr uint32_t U_MISC = U_BAR + 8 * 8;
constexpr uint32_t kSmemUt = U_MISC + 64 + 1024;
static_assert(U_A % 16 == 0 && U_SC % 16 == 0, "alignment");
static_assert(4 * (kSmemUt + 1024) <= 233472, "four UT CTAs per SM");

// ---- recur_tc_kernel shared memory.  Operands are staged by lifetime:
//   "early" stages (2): T' and V (a1), [W~ | Q] interleaved (the merged a2 product)
//   "late"  stages (2): [Aqk^T | K->] (even chunks) or [K-> | Aqk^T] (odd chunks) for the
//                       merged c product; afterwards the chunk's output staging tile
//   the bf16 state (A of a2) and the bf16 V_new^T (A of c), and a ring of per-chunk factors.
constexpr int kThreadsRc = 448;        // warp 0: loads, TMEM; warp 1: MMA; warps 2-9: state; 10-13: outputs
                                       // (and, with the block prologue fused in, the V convolution)
constexpr int kEarly = 2, kLate = 2, kScSlots = 4;
constexpr uint32_t E_TP = 0, E_V = 16384, E_WQ = 32768, kEarlyBytes = 65536;
constexpr uint32_t kLateBytes = 24576;
constexpr uint32_t R_EARLY = 0;
constexpr uint32_t R_LATE = R_EARLY + kEarly * kEarlyBytes;
constexpr uint32_t R_SBF = R_LATE + kLate * kLateBytes;   // S bf16, [d-block][128 j][64 d] x 2
constexpr uint32_t R_X = R_SBF + 32768;                   // V_new^T bf16, [128 j][64 r]
constexpr uint32_t R_SCR = R_X + 16384;                   // factor ring: kScSlots x kScStride
constexpr uint32_t kScBytes = 272;                        // fq[64], e^{b_C}, range flag (+ pad)
constexpr uint32_t kScStride = 288;
constexpr uint32_t R_BAR = R_SCR + kScSlots * kScStride;
constexpr uint32_t R_MISC = R_BAR + 32 * 8;
constexpr uint32_t kSmemRc = R_MISC + 64 + 1024;
static_assert(kEarlyBytes % 1024 == 0 && kLateBytes % 1024 == 0 && kSmemRc <= 232448, "recurrence smem");
constexpr uint32_t kEarlyTxA = 16384 + 16384;          // T' (hi, lo) and V
constexpr uint32_t kEarlyTxB = 32768;                  // W~ and Q
constexpr uint32_t kLateTx = 24576;                     // Aqk^T and K->

// recurrence tensor-memory columns (512).  The two output accumulators alternate by
// chunk parity so the output warps may drain one while the next chunk runs:
//   even chunk: a2 -> [D1_0 | D2A_0] (0..127),   c -> [D2B_0 | S] (128..319)
//   odd  chunk: a2 -> [D1_1 | D2A_1] (384..511), c -> [S | D2B_1] (192..383)
constexpr uint32_t TM_S = 192;
__device__ __forceinline__ uint32_t tm_d1(int c) { return (c & 1) ? 384u : 0u; }
__device__ __forceinline__ uint32_t tm_d2a(int c) { return (c & 1) ? 448u : 64u; }
__device__ __forceinline__ uint32_t tm_d2b(int c) { return (c & 1) ? 320u : 128u; }
__device__ __forceinline__ uint32_t tm_c(int c) { return (c & 1) ? 192u : 128u; }

// The early ring's two halves fill and drain separately: A (T', V) is read only by a1 and may be
// refilled as soon as a1 completes; B ([W~ | Q]) is read by a2.
enum : int { RB_EF = 0, RB_EE = 2, RB_LF = 4, RB_LE = 6, RB_SCF = 8, RB_SCE = 12,   // rings (EF/EE: half A)
             RB_D1 = 16, RB_X = 17, RB_S = 18, RB_SP = 19, RB_D2 = 20,
             RB_D2O = 21, RB_OFREE = 23,                                         // [2] by parity
             RB_FIN = 25, RB_VC = 26,                    // RB_VC [2]: V convolved (early slot)
             RB_EFB = 28, RB_EEB = 30, RB_COUNT = 32 };  // early ring, half B
enum : int { UB_QK = 0, UB_P1 = 1, UB_TRDY = 2, UB_P2 = 3, UB_FIN = 4, UB_CONV = 5, UB_COUNT = 6 };

// Development-only phase timestamps (SM clock) of the first CTA; compiled out
// of the library unless GDN_KERNEL_TRACE is defined.
#ifdef GDN_KERNEL_TRACE
long long *g_trace_buffer = nullptr;
// UT kernel: up to 48 phase stamps of CTA (slot 0, head 0) in rows 13-15 of role 3
#define GDN_UTR(trace, ev)                                                                          \
    do {                                                                                             \
        if ((trace) && blockIdx.x == 0 && blockIdx.y == 0) (trace)[(3 * 16 + 13) * 16 + (ev)] = clock64(); \
    } while (0)
#define GDN_TR(trace, role, c, ev)                                                                   \
    do {                                                                                             \
        if ((trace) && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (c) < 16)            \
            (trace)[((role) * 16 + (c)) * 16 + (ev)] = clock64();                                    \
    } while (0)
#else
#define GDN_TR(trace, role, c, ev) do { } while (0)
#define GDN_UTR(trace, ev) do { } while (0)
#endif

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag, unsigned *err,
                                         uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicExch(err, kDevErrTimeout);
            return false;
        }
    }
}

// Spinning variant for the latency-critical hand-offs of the recurrence: a
// sleeping try_wait can wake up late, which adds directly to the serial chain.
__device__ __forceinline__ bool wait_spin(uint32_t bar, uint32_t parity, volatile int *abort_flag, unsigned *err)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 256; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicExch(err, kDevErrTimeout);
            return false;
        }
    }
}

// Named barrier over `count` threads that also ORs a predicate across them,
// so a whole group leaves a loop at the same point.
__device__ __forceinline__ bool group_sync_or(int id, int count, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(count) : "memory");
    return r != 0;
}

__device__ __forceinline__ void group_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(float a, float b)
{
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Largest magnitude an fp16 operand may carry before it would round to infinity.
constexpr float kF16Max = 65504.f;

__device__ __forceinline__ float2 unpack_bf16(uint32_t u)
{
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(v);
}

__device__ __forceinline__ uint32_t to_tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// fp32 A fragments of one 16-row strip of X (m16n8k8 layout) for the k-steps
// 8ks >= kbeg: X(r, k) = X0[r * xp + k].
template <int KS>
__device__ __forceinline__ void load_a_f32(float (&fa)[KS][4], const float *X0, int xp, int kbeg, int g, int t)
{
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const int k0 = 8 * ks;
        if (k0 < kbeg) continue;
        fa[ks][0] = X0[g * xp + k0 + t];
        fa[ks][1] = X0[(g + 8) * xp + k0 + t];
        fa[ks][2] = X0[g * xp + k0 + t + 4];
        fa[ks][3] = X0[(g + 8) * xp + k0 + t + 4];
    }
}

// x = hi + lo with hi, lo both tf32 (x - hi is exact in fp32), about 22 bits together.
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo)
{
    hi = to_tf32(x);
    lo = to_tf32(x - __uint_as_float(hi));
}

// acc (16 x 8) += X Y over the k-steps 8ks >= kbeg, X given as fp32 fragments,
// Y(k, n) = Y0[k * yp + n], as three tf32 products (X_lo Y_hi + X_hi Y_lo + X_hi Y_hi): the
// lo x lo term is below fp32 rounding, so the result has fp32 accuracy.  The solve's merges need
// it: with nearly parallel keys and beta close to 2 the entries of T alternate in sign and a
// single tf32 pass loses about three decimal digits of the intra-chunk products.
template <int KS>
__device__ __forceinline__ void mma_a_3xtf32(float (&acc)[4], const float (&fa)[KS][4], const float *Y0, int yp,
                                             int kbeg, int g, int t)
{
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const int k0 = 8 * ks;
        if (k0 < kbeg) continue;
        uint32_t ah[4], al[4], bh0, bl0, bh1, bl1;
#pragma unroll
        for (int e = 0; e < 4; ++e) split_tf32(fa[ks][e], ah[e], al[e]);
        split_tf32(Y0[(k0 + t) * yp + g], bh0, bl0);
        split_tf32(Y0[(k0 + t + 4) * yp + g], bh1, bl1);
        mma_tf32(acc, al, bh0, bh1);
        mma_tf32(acc, ah, bl0, bl1);
        mma_tf32(acc, ah, bh0, bh1);
    }
}

// Store a 16 x 8 accumulator tile, scaled by sg, to Z0[r * zp + n].
__device__ __forceinline__ void store_16x8(const float (&acc)[4], float *Z0, int zp, float sg, int g, int t)
{
    *reinterpret_cast<float2 *>(Z0 + g * zp + 2 * t) = make_float2(sg * acc[0], sg * acc[1]);
    *reinterpret_cast<float2 *>(Z0 + (g + 8) * zp + 2 * t) = make_float2(sg * acc[2], sg * acc[3]);
}

// In place: A (64 x 64, pitch LDL) holds the strictly lower L on entry (zeros
// elsewhere) and T = (I + L)^{-1} on exit; 128 threads (4 warps, `warp` 0-3),
// Mt >= 4 x 256 floats of scratch.  Block rule
//   [A 0; C B]^{-1} = [A^-1 0; -B^-1 (C A^-1)  B^-1]
// in three steps with one barrier after each:
//   (i)   warp w inverts the unit-lower 16 x 16 diagonal block w by forward
//         substitution, one column per lane, the column in registers;
//   (ii)  the 16 -> 32 merges of blocks (0,1) and (2,3), warp w taking the
//         8-column half (w & 1) of merge (w >> 1);
//   (iii) the 32 -> 64 merge, warp w taking columns 8w..8w+7.
// The off-diagonal blocks of L that (ii) and (iii) overwrite are read into
// registers before the first barrier, and each warp's two products touch only
// its own columns of C A^-1, so no other synchronisation is needed.
__device__ __forceinline__ void solve_in_place(float *__restrict__ A, float *__restrict__ Mt, int warp, int lane,
                                               long long *trace)
{
    (void)trace;
    const bool stamp = warp == 3 && lane == 0;
    const int g = lane >> 2, t = lane & 3;
    const int m2 = warp >> 1, h2 = warp & 1, a2 = 32 * m2, b2 = a2 + 16, n2 = a2 + 8 * h2;   // step (ii)
    const int n3 = 8 * warp;                                                               // step (iii)
    float c2[2][4], c3[2][4][4];
    // C of step (ii): L rows b2.., columns a2..; A^-1 is lower triangular, so
    // k-steps below this warp's first column contribute nothing
    load_a_f32<2>(c2, A + b2 * LDL + a2, LDL, 8 * h2, g, t);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) load_a_f32<4>(c3[mt], A + (32 + 16 * mt) * LDL, LDL, n3, g, t);
    {   // (i) diagonal block `warp`, column c of its inverse
        const int o = 16 * warp, c = lane & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
            const float *row = A + (o + r) * LDL + o;
            float acc = 0.f;
#pragma unroll
            for (int i4 = 0; i4 < r; i4 += 4) {
                const float4 l4 = *reinterpret_cast<const float4 *>(row + i4);
                acc = fmaf(l4.x, x[i4], acc);
                if (i4 + 1 < r) acc = fmaf(l4.y, x[i4 + 1], acc);
                if (i4 + 2 < r) acc = fmaf(l4.z, x[i4 + 2], acc);
                if (i4 + 3 < r) acc = fmaf(l4.w, x[i4 + 3], acc);
            }
            if (r > c) x[r] = -acc;
        }
        if (stamp) GDN_UTR(trace, 9);
        group_sync(1, 128);   // every warp has read its L fragments and diagonal rows
        if (stamp) GDN_UTR(trace, 10);
        if (lane < 16) {
#pragma unroll
            for (int r = 0; r < 16; ++r) A[(o + r) * LDL + o + c] = x[r];
        }
    }
    group_sync(1, 128);
    if (stamp) GDN_UTR(trace, 11);
    float *M = Mt + warp * 256;   // this warp's C A^-1 columns: up to 32 x 8, pitch 8
    {   // (ii)
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        mma_a_3xtf32<2>(acc, c2, A + a2 * LDL + n2, LDL, 8 * h2, g, t);
        store_16x8(acc, M, 8, 1.f, g, t);
        __syncwarp();
        float acc2[4] = {0.f, 0.f, 0.f, 0.f};
        float tb[2][4];
        load_a_f32<2>(tb, A + b2 * LDL + b2, LDL, 0, g, t);
        mma_a_3xtf32<2>(acc2, tb, M, 8, 0, g, t);
        store_16x8(acc2, A + b2 * LDL + n2, LDL, -1.f, g, t);
    }
    if (stamp) GDN_UTR(trace, 12);
    group_sync(1, 128);
    if (stamp) GDN_UTR(trace, 13);
    {   // (iii)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            mma_a_3xtf32<4>(acc, c3[mt], A + n3, LDL, n3, g, t);
            store_16x8(acc, M + 16 * mt * 8, 8, 1.f, g, t);
        }
        __syncwarp();
        {   // rows 32-47: B^-1 is lower triangular, k < 16
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            float tb[2][4];
            load_a_f32<2>(tb, A + 32 * LDL + 32, LDL, 0, g, t);
            mma_a_3xtf32<2>(acc, tb, M, 8, 0, g, t);
            store_16x8(acc, A + 32 * LDL + n3, LDL, -1.f, g, t);
        }
        {   // rows 48-63
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            float tb[4][4];
            load_a_f32<4>(tb, A + 48 * LDL + 32, LDL, 0, g, t);
            mma_a_3xtf32<4>(acc, tb, M, 8, 0, g, t);
            store_16x8(acc, A + 48 * LDL + n3, LDL, -1.f, g, t);
        }
    }
    if (stamp) GDN_UTR(trace, 14);
    group_sync(1, 128);
    if (stamp) GDN_UTR(trace, 15);
}

// ===========================================================================
// chunk-local UT transform
// ===========================================================================
// The block prologue, when it is fused into the chunked forward ("Gated Delta Networks: Improving
// Mamba2 with Delta Rule", §3.4 "Token mixing block", Fig. 1): q, k, v = SiLU(short causal
// depthwise convolution of the projections), g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b).
// The arithmetic is written exactly as in prologue.cu, so the fused call reproduces
// gdn_prologue followed by gdn_chunk_fwd bit for bit.
struct ConvParams {
    const __nv_bfloat16 *xq, *xk, *xv;         // raw projections [rows, H, d] (halo rows are read here)
    const float *wq, *wk, *wv;                 // filters [H, d, K]
    const float *a, *b, *A_log, *dt_bias;      // gate projections [rows, H]; per-head parameters [H]
    const __nv_bfloat16 *state_in;             // [N, K-1, H, 2 dk + dv] or null (zeros)
    __nv_bfloat16 *state_out;                  // same layout, or null
};

__device__ __forceinline__ float conv_silu(float z) { return __fdividef(z, 1.f + __expf(-z)); }
__device__ __forceinline__ float gate_softplus(float z) { return z > 20.f ? z : log1pf(expf(z)); }

struct UtParams {
    const float *g, *beta;
    uint8_t *blocks;
    size_t block_bytes;
    unsigned *err;
    Geometry gm;
    float scale;
    int l2;
    long long *trace;
    ConvParams cv;      // used when the kernel is instantiated with a convolution width KC > 0
};

// KC = 0: q, k, g, beta are the operator's inputs.  KC = 1..4: they are made here from the raw
// projections by the block prologue with a convolution of width KC.
template <int KC>
__global__ void __launch_bounds__(kThreadsUt, 4)
ut_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk, const UtParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the first CTA clears the call's device error word (a timeout anywhere
    // is at least kWaitLimitNs later)
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) *p.err = kDevErrNone;
    const int64_t slot = blockIdx.x;
    const int h = blockIdx.y;
    const Geometry gm = p.gm;
    int n, c, rows;
    int64_t tok0c;
    if (!slot_to_chunk(gm, slot, n, c, tok0c, rows)) return;
    const int H = gm.H;
    uint32_t *tmem_sh = reinterpret_cast<uint32_t *>(sm + U_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + U_MISC + 4);
    volatile int *range_flag = reinterpret_cast<volatile int *>(sm + U_MISC + 8);
    auto bar = [&](int i) -> uint32_t { return sb + U_BAR + 8u * (uint32_t)i; };
    uint8_t *blk = p.blocks + ((size_t)slot * H + h) * p.block_bytes;

    if (tid == 0) {
        for (int i = 0; i < UB_COUNT; ++i) mbar_init(bar(i), 1);
        *abort_flag = 0;
        *range_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_sh, 128);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = *tmem_sh;
    const uint32_t TP1 = 0, TP2 = 0;   // the W~ product reuses the Gram columns once they are read

    if (warp == 0) {
        if (lane == 0) {
            const int z = (int)tok0c;
            mbar_expect_tx(bar(UB_QK), 32768);
            tma_load_3d(sb + U_QK, &tmk, 0, h, z, bar(UB_QK));
            tma_load_3d(sb + U_QK + 8192, &tmq, 0, h, z, bar(UB_QK));
            tma_load_3d(sb + U_QK + 16384, &tmk, 64, h, z, bar(UB_QK));
            tma_load_3d(sb + U_QK + 24576, &tmq, 64, h, z, bar(UB_QK));
            bool tiles = wait_bar(bar(UB_QK), 0, abort_flag, p.err);
            if (KC > 0 && tiles) tiles = wait_bar(bar(UB_CONV), 0, abort_flag, p.err);   // convolved in place
            if (tiles) {
                fence_after_sync();
                const uint32_t id_p1 = idesc_bf16(128, 128, false, false);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {   // G = [K; Q] [K; Q]^T  (rows 0-63: K K^T | K Q^T)
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_ss(tb + TP1, smem_desc(sb + U_QK + off, 16, 1024), smem_desc(sb + U_QK + off, 16, 1024),
                           id_p1, ks > 0);
                }
                commit(bar(UB_P1));
                if (wait_bar(bar(UB_TRDY), 0, abort_flag, p.err)) {
                    fence_after_sync();
                    const uint32_t id_p2 = idesc_bf16(128, 128, false, true);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)   // [W~; 0] = [T''_hi; 0] K + [T''_lo; 0] K  (rows 0-63 are W~)
                        mma_ss(tb + TP2, smem_desc(sb + ((ks < 4) ? U_TPP : U_TPL) + (ks & 3) * 32, 16, 1024),
                               smem_desc(sb + U_QK + (ks & 3) * 2048, 16384, 1024), id_p2, ks > 0);
                    commit(bar(UB_P2));
                }
            }
            if (*abort_flag) mbar_wait(bar(UB_QK), 0, 10000000ull);   // the tile copy must land before exit
            commit(bar(UB_FIN));
            mbar_wait(bar(UB_FIN), 0, kWaitLimitNs);
        }
        __syncwarp();
    } else {
        const int prow = 32 * (warp & 3) + lane;   // tensor-memory lane of this thread
        float *Am = reinterpret_cast<float *>(sm + U_A);
        float *Mt = reinterpret_cast<float *>(sm + U_MT);
        float *sc = reinterpret_cast<float *>(sm + U_SC);
        float *bsum = sc, *bet = sc + 64, *rk = sc + 128, *rq = sc + 192, *cw = sc + 256, *ecol = sc + 320;
        float *cq = sc + 384;   // [3][64]: e^{b_m - b_p} rq_m for the block ends p = 15, 31, 47
        float *fkt = sc + 640;  // fk_r = e^{b_C - b_r} rk_r
        const uint32_t lane_base = tb + ((uint32_t)(32 * (warp & 3)) << 16);
        const uint8_t *st = sm + U_QK;
        if (prow == 0) GDN_UTR(p.trace, 0);
        do {
            // (1) gates: chunk-local cumulative log-gate in base 2, beta
            {
                const int r = prow & 63;
                const int64_t t = (tok0c + r) * H + h;
                float x = 0.f;
                if (prow < 64) {
                    if (KC > 0) {
                        x = (r < rows) ? -expf(p.cv.A_log[h]) * gate_softplus(p.cv.a[t] + p.cv.dt_bias[h]) * kLog2e : 0.f;
                    } else {
                        x = (r < rows) ? p.g[t] * kLog2e : 0.f;
                    }
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float y = __shfl_up_sync(0xffffffffu, x, o);
                        if (lane >= o) x += y;
                    }
                    if (lane == 31) sc[576 + (prow >> 5)] = x;
                } else {
                    if (KC > 0) bet[r] = (r < rows) ? 1.f / (1.f + expf(-p.cv.b[t])) : 0.f;
                    else bet[r] = (r < rows) ? p.beta[t] : 0.f;
                }
                group_sync(1, 128);
                if (prow < 64) bsum[prow] = x + ((prow >= 32) ? sc[576] : 0.f);
                group_sync(1, 128);
            }
            if constexpr (KC > 0) {
                // (1b) block prologue on the raw Q and K tiles, in place: thread p takes the channel
                //      pair 2(p % 64), 2(p % 64) + 1 of Q (p < 64) or K over the chunk's 64 rows, with
                //      the KC - 1 inputs before each row in registers (the previous chunk's last rows,
                //      or the carried convolution state before a sequence's first chunk)
                bool okc = wait_bar(bar(UB_QK), 0, abort_flag, p.err);
                if (okc) {
                    const bool isq = prow < 64;
                    const int dk = gm.dk, Cw = 2 * dk + gm.dv;
                    const int c0 = 2 * (prow & 63);
                    uint8_t *tile = sm + U_QK + (isq ? 8192 : 0) + (c0 >> 6) * 16384;
                    const __nv_bfloat16 *xg = isq ? p.cv.xq : p.cv.xk;
                    const float *wf = isq ? p.cv.wq : p.cv.wk;
                    const int chan = (isq ? 0 : dk) + c0;   // channel in the [q | k | v] state axis
                    float2 wt[KC];
#pragma unroll
                    for (int j = 0; j < KC; ++j)
                        wt[j] = make_float2(wf[((int64_t)h * dk + c0) * KC + j], wf[((int64_t)h * dk + c0 + 1) * KC + j]);
                    constexpr int KH = KC > 1 ? KC - 1 : 1;
                    float2 hist[KH];   // hist[m]: the input KC-1-m rows before the current one
#pragma unroll
                    for (int m = 0; m < KC - 1; ++m) {
                        if (c > 0)
                            hist[m] = unpack_bf16(*reinterpret_cast<const uint32_t *>(
                                xg + (tok0c - (KC - 1) + m) * H * dk + (int64_t)h * dk + c0));
                        else if (p.cv.state_in)
                            hist[m] = unpack_bf16(*reinterpret_cast<const uint32_t *>(
                                p.cv.state_in + (((int64_t)n * (KC - 1) + m) * H + h) * Cw + chan));
                        else
                            hist[m] = make_float2(0.f, 0.f);
                    }
                    int64_t s0;
                    int len;
                    seq_span(gm, n, s0, len);
                    const bool last = (int64_t)c * kChunk + rows == len;
                    float2 snap[KH];   // the KC-1 inputs up to the chunk's last row (the carried state)
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        // the 32 raw rows first (their loads overlap), then filter and store in place
                        uint32_t raw[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            raw[i] = *reinterpret_cast<const uint32_t *>(tile + sw128_offset(32 * half + i, c0 & 63));
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int tr = 32 * half + i;
                            const float2 xt = unpack_bf16(raw[i]);
                            float2 z = make_float2(wt[KC - 1].x * xt.x, wt[KC - 1].y * xt.y);
#pragma unroll
                            for (int j = 0; j < KC - 1; ++j) {
                                z.x += wt[j].x * hist[j].x;
                                z.y += wt[j].y * hist[j].y;
                            }
                            *reinterpret_cast<uint32_t *>(tile + sw128_offset(tr, c0 & 63)) =
                                pack_bf16(conv_silu(z.x), conv_silu(z.y));
#pragma unroll
                            for (int m = 0; m + 1 < KC - 1; ++m) hist[m] = hist[m + 1];
                            if (KC > 1) hist[KH - 1] = xt;
                            if (tr == rows - 1)
#pragma unroll
                                for (int m = 0; m < KH; ++m) snap[m] = hist[m];
                        }
                    }
                    if (last && p.cv.state_out)   // the sequence's last KC-1 inputs, oldest first
#pragma unroll
                        for (int m = 0; m < KC - 1; ++m)
                            *reinterpret_cast<uint32_t *>(p.cv.state_out + (((int64_t)n * (KC - 1) + m) * H + h) * Cw + chan) =
                                pack_bf16(snap[m].x, snap[m].y);
                }
                fence_proxy_async();
                if (group_sync_or(2, 128, !okc || *abort_flag)) break;
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) {   // the convolved Q tile (2 x 8 KB) for the recurrence
                    const int u = prow + 128 * k2, q = u >> 9, o = (u & 511) * 16;
                    *reinterpret_cast<uint4 *>(blk + PB_QC + q * 8192 + o) =
                        *reinterpret_cast<const uint4 *>(sm + U_QK + 8192 + q * 16384 + o);
                }
                if (prow == 0) mbar_arrive(bar(UB_CONV));
            }
            // (2) inverse norms from the diagonal of the Gram product: thread p reads
            //     G_pp (= ||k_p||^2 or ||q_{p-64}||^2, fp32 sums of exact bf16 products)
            //     from column p of its own tensor-memory lane
            if (prow == 0) GDN_UTR(p.trace, 1);
            bool ok = wait_bar(bar(UB_P1), 0, abort_flag, p.err);
            ok = ok && wait_bar(bar(UB_QK), 0, abort_flag, p.err);   // (already complete) the K tile for K->
            if (prow == 0) GDN_UTR(p.trace, 2);
            fence_after_sync();
            {
                const int r = prow & 63;
                const bool isq = prow >= 64;
                uint32_t d[32];
                tmem_ld16(lane_base + TP1 + 32 * (warp & 3), *reinterpret_cast<uint32_t(*)[16]>(d));
                tmem_ld16(lane_base + TP1 + 32 * (warp & 3) + 16, *reinterpret_cast<uint32_t(*)[16]>(d + 16));
                tmem_wait_ld();
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 32; ++e) ss = (e == lane) ? __uint_as_float(d[e]) : ss;
                float inv = p.l2 ? 1.f / sqrtf(ss + kL2Eps) : 1.f;
                if (isq) inv *= p.scale;
                inv = (r < rows) ? inv : 0.f;
                // column factors of the masks: decay of column i to the end of its
                // 16-block (off-diagonal blocks, where e^{b_r - b_i} = e^{b_r - b_p} e^{b_p - b_i}
                // with both factors <= 1) and e^{b_i} rk_i (for T'');  for the query
                // columns m, e^{b_m - b_p} rq_m for the block ends p = 15, 31, 47
                if (!isq) {
                    rk[r] = inv;
                    cw[r] = exp2f(bsum[r | 15] - bsum[r]) * inv;
                    ecol[r] = exp2f(bsum[r]) * inv;
                    fkt[r] = (r < rows) ? exp2f(bsum[63] - bsum[r]) * inv : 0.f;
                } else {
                    rq[r] = inv;
#pragma unroll
                    for (int I = 0; I < 3; ++I) cq[I * 64 + r] = (r > I * 16 + 15) ? exp2f(bsum[r] - bsum[I * 16 + 15]) * inv : 0.f;
                }
            }
            if (group_sync_or(2, 128, !ok || *abort_flag)) break;

            // (3) masks from the Gram rows of K: lane i holds k_i . k_m and k_i . q_m.
            //     L_im  = beta_i e^{b_i - b_m} rk_i rk_m (k_i . k_m),    m <  i   (into A)
            //     AqkT_im = e^{b_m - b_i} rq_m rk_i (k_i . q_m),          m >= i   (to the workspace)
            //   Rows 64-127 (Q rows) are not needed; their threads write K-> meanwhile.
            if (prow == 0) GDN_UTR(p.trace, 3);
            if (prow == 0) GDN_UTR(p.trace, 4);
            if (prow < 64) {
                // Thread i (TMEM lane i) holds row i of K [K; Q]^T.  Warp quarter wq covers
                // rows 32wq..32wq+31 (16-blocks 2wq, 2wq+1): the "near" column blocks 2wq and
                // 2wq+1 take the exact factor e^{+-(b_i - b_m)} per entry (masked by a select),
                // the far blocks the factorised one, so every branch is uniform over the warp.
                const int i = prow, I = i >> 4, wq = warp & 3;
                const float bi = bsum[i];
                float amax = 0.f;   // largest |Aqk| this thread converts to fp16
                uint32_t u[64];
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld16(lane_base + TP1 + q * 16, *reinterpret_cast<uint32_t(*)[16]>(u + q * 16));
                tmem_wait_ld();
                if (prow == 0) GDN_UTR(p.trace, 5);
                {   // L row i, columns m < i: beta_i e^{b_i - b_m} rk_i rk_m G_im
                    const float f = bet[i] * rk[i];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float v[16];
                        if (q < 2 * wq) {
                            const float fu = f * exp2f(bi - bsum[q * 16 + 15]);
#pragma unroll
                            for (int e4 = 0; e4 < 16; e4 += 4) {
                                const float4 c4 = *reinterpret_cast<const float4 *>(cw + q * 16 + e4);
                                v[e4 + 0] = fu * c4.x * __uint_as_float(u[q * 16 + e4 + 0]);
                                v[e4 + 1] = fu * c4.y * __uint_as_float(u[q * 16 + e4 + 1]);
                                v[e4 + 2] = fu * c4.z * __uint_as_float(u[q * 16 + e4 + 2]);
                                v[e4 + 3] = fu * c4.w * __uint_as_float(u[q * 16 + e4 + 3]);
                            }
                        } else if (q <= 2 * wq + 1) {
#pragma unroll
                            for (int e4 = 0; e4 < 16; e4 += 4) {
                                const float4 b4 = *reinterpret_cast<const float4 *>(bsum + q * 16 + e4);
                                const float4 r4 = *reinterpret_cast<const float4 *>(rk + q * 16 + e4);
                                const float bb[4] = {b4.x, b4.y, b4.z, b4.w}, rr[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int m = q * 16 + e4 + e;
                                    const float x = f * rr[e] * __uint_as_float(u[m]) * exp2f(bi - bb[e]);
                                    v[e4 + e] = (m < i) ? x : 0.f;
                                }
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] = 0.f;
                        }
                        float4 *dst = reinterpret_cast<float4 *>(Am + i * LDL + q * 16);
#pragma unroll
                        for (int e = 0; e < 4; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                    }
                }
                if (prow == 0) GDN_UTR(p.trace, 6);
                // Aqk^T row i, columns m >= i: e^{b_m - b_i} rq_m rk_i G_(i, 64+m); far blocks
                // as e^{b_m - b_p} e^{b_p - b_i} with p the end of i's 16-block
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    tmem_ld16(lane_base + TP1 + 64 + q * 16, *reinterpret_cast<uint32_t(*)[16]>(u + q * 16));
                tmem_wait_ld();
                if (prow == 0) GDN_UTR(p.trace, 7);
                {
                    const float fi = rk[i];
                    const float fw = fi * exp2f(bsum[i | 15] - bi);   // rk_i e^{b_p - b_i}
                    const float *cqi = cq + (I < 3 ? I : 2) * 64;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float v[16];
                        if (q > 2 * wq + 1) {
#pragma unroll
                            for (int e4 = 0; e4 < 16; e4 += 4) {
                                const float4 c4 = *reinterpret_cast<const float4 *>(cqi + q * 16 + e4);
                                v[e4 + 0] = fw * c4.x * __uint_as_float(u[q * 16 + e4 + 0]);
                                v[e4 + 1] = fw * c4.y * __uint_as_float(u[q * 16 + e4 + 1]);
                                v[e4 + 2] = fw * c4.z * __uint_as_float(u[q * 16 + e4 + 2]);
                                v[e4 + 3] = fw * c4.w * __uint_as_float(u[q * 16 + e4 + 3]);
                            }
                        } else if (q >= 2 * wq) {
#pragma unroll
                            for (int e4 = 0; e4 < 16; e4 += 4) {
                                const float4 b4 = *reinterpret_cast<const float4 *>(bsum + q * 16 + e4);
                                const float4 r4 = *reinterpret_cast<const float4 *>(rq + q * 16 + e4);
                                const float bb[4] = {b4.x, b4.y, b4.z, b4.w}, rr[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int m = q * 16 + e4 + e;
                                    const float x = fi * rr[e] * __uint_as_float(u[m]) * exp2f(bb[e] - bi);
                                    v[e4 + e] = (m >= i) ? x : 0.f;
                                }
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) v[e] = 0.f;
                        }
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                amax = fmaxf(amax, fmaxf(fabsf(v[hh * 8 + 2 * e]), fabsf(v[hh * 8 + 2 * e + 1])));
                                w[e] = pack_f16(v[hh * 8 + 2 * e], v[hh * 8 + 2 * e + 1]);
                            }
                            *reinterpret_cast<uint4 *>(sm + U_TPP + sw128_offset(i, q * 16 + hh * 8)) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                if (amax > kF16Max) *range_flag = 1;
                if (prow == 0) GDN_UTR(p.trace, 22);
            } else {   // K-> = diag(fk) K in the K tile's own layout; 16-B chunk u of the two
                       // 8-KB tiles per step, so a warp writes 512 contiguous bytes
                const int t = prow - 64;
                float kmax = 0.f;   // largest |K->| this thread converts to fp16
#pragma unroll 4
                for (int k2 = 0; k2 < 16; ++k2) {
                    const int u = t + 64 * k2, kb = u >> 9, r = (u >> 3) & 63, pc = u & 7;
                    const float fk = fkt[r];
                    const uint4 uu = *reinterpret_cast<const uint4 *>(st + kb * 16384 + r * 128 + pc * 16);
                    const uint32_t w[4] = {uu.x, uu.y, uu.z, uu.w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = unpack_bf16(w[e]);
                        kmax = fmaxf(kmax, fmaxf(fabsf(x.x * fk), fabsf(x.y * fk)));
                        o[e] = pack_f16(x.x * fk, x.y * fk);
                    }
                    *reinterpret_cast<uint4 *>(blk + PB_KT + kb * 8192 + r * 128 + pc * 16) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                if (kmax > kF16Max) *range_flag = 1;
                if (prow == 64) GDN_UTR(p.trace, 23);
            }
            fence_before_sync();
            if (group_sync_or(2, 128, !ok || *abort_flag)) break;
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2) {   // Aqk^T: staging tile -> workspace, 512 B per warp store
                const int o = 16 * (prow + 128 * k2);
                *reinterpret_cast<uint4 *>(blk + PB_AQT + o) = *reinterpret_cast<const uint4 *>(sm + U_TPP + o);
            }
            if (prow == 0) GDN_UTR(p.trace, 8);

            // (4) T = (I + L)^{-1} in place;  T' -> workspace,  T'' -> shared memory
            solve_in_place(Am, Mt, (warp + 3) & 3, lane, p.trace);
            if (prow == 0) GDN_UTR(p.trace, 16);
            {   // 16-B chunk u = (row r, physical chunk pc) per step: consecutive threads write
                // consecutive bytes of T' (and of T''); columns ib..ib+7 of row r
#pragma unroll
                for (int k2 = 0; k2 < 4; ++k2) {
                    const int u = prow + 128 * k2, r = u >> 3, pc = u & 7, ib = 8 * (pc ^ (r & 7));
                    const float4 t0 = *reinterpret_cast<const float4 *>(Am + r * LDL + ib);
                    const float4 t1 = *reinterpret_cast<const float4 *>(Am + r * LDL + ib + 4);
                    const float4 b0 = *reinterpret_cast<const float4 *>(bet + ib);
                    const float4 b1 = *reinterpret_cast<const float4 *>(bet + ib + 4);
                    const float4 e0 = *reinterpret_cast<const float4 *>(ecol + ib);
                    const float4 e1 = *reinterpret_cast<const float4 *>(ecol + ib + 4);
                    const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
                    const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                    const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
                    uint32_t w1[4], w1l[4], w2[4], w3[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float p0 = tv[2 * e] * bv[2 * e], p1 = tv[2 * e + 1] * bv[2 * e + 1];
                        w1[e] = pack_bf16(p0, p1);   // T' = T'_hi + T'_lo, each bf16
                        const float2 h1 = unpack_bf16(w1[e]);
                        w1l[e] = pack_bf16(p0 - h1.x, p1 - h1.y);
                        // T'' as a sum of two bf16 terms: W~ = T'' K can cancel heavily (nearly
                        // parallel keys), so its operand carries ~16 bits
                        const float q0 = p0 * ev[2 * e], q1 = p1 * ev[2 * e + 1];
                        w2[e] = pack_bf16(q0, q1);
                        const float2 h2 = unpack_bf16(w2[e]);
                        w3[e] = pack_bf16(q0 - h2.x, q1 - h2.y);
                    }
                    const uint32_t off = (uint32_t)(r * 128 + pc * 16);   // = sw128_offset(r, ib)
                    *reinterpret_cast<uint4 *>(blk + PB_TP + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
                    *reinterpret_cast<uint4 *>(blk + PB_TP + 8192 + off) = make_uint4(w1l[0], w1l[1], w1l[2], w1l[3]);
                    *reinterpret_cast<uint4 *>(sm + U_TPP + off) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
                    *reinterpret_cast<uint4 *>(sm + U_TPL + off) = make_uint4(w3[0], w3[1], w3[2], w3[3]);
                }
            }
            fence_proxy_async();
            if (group_sync_or(2, 128, !ok || *abort_flag)) break;
            if (prow == 0) mbar_arrive(bar(UB_TRDY));
            if (prow == 0) GDN_UTR(p.trace, 17);

            // (5) W~^T and the per-row factors to the workspace
            {
                const int r = prow & 63;
                const float bC = bsum[63];
                if (prow < 64) {
                    reinterpret_cast<float *>(blk + PB_SC)[r] = (r < rows) ? exp2f(bsum[r]) * rq[r] : 0.f;
                } else if (r < 4) {   // [65]: 1 if an fp16 operand of this block overflowed
                    reinterpret_cast<float *>(blk + PB_SC)[64 + r] =
                        (r == 0) ? exp2f(bC) : ((r == 1 && *range_flag) ? 1.f : 0.f);
                }
            }
            if (prow == 0) GDN_UTR(p.trace, 18);
            ok = wait_bar(bar(UB_P2), 0, abort_flag, p.err);
            if (prow == 0) GDN_UTR(p.trace, 19);
            fence_after_sync();
            if (prow < 64) {   // row r of W~ (128 d) -> staging [d-block][64 r][64 d] in the dead T area
                uint8_t *wst = sm + U_A;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    uint32_t u[16];
                    tmem_ld16(lane_base + TP2 + q * 16, u);
                    tmem_wait_ld();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack_bf16(__uint_as_float(u[hh * 8 + 2 * e]), __uint_as_float(u[hh * 8 + 2 * e + 1]));
                        const int d = q * 16 + hh * 8;
                        *reinterpret_cast<uint4 *>(wst + (d >> 6) * 8192 + sw128_offset(prow, d & 63)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            if (group_sync_or(2, 128, !ok || *abort_flag)) break;
#pragma unroll
            for (int k2 = 0; k2 < 8; ++k2) {   // W~: staging -> workspace, 512 B per warp store
                const int o = 16 * (prow + 128 * k2);
                *reinterpret_cast<uint4 *>(blk + PB_W + o) = *reinterpret_cast<const uint4 *>(sm + U_A + o);
            }
            fence_before_sync();
        } while (false);
    }
    if (tid == 32) GDN_UTR(p.trace, 20);
    fence_before_sync();
    __syncthreads();
    if (tid == 32) GDN_UTR(p.trace, 21);
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tb, 128);
    }
}

// ===========================================================================
// inter-chunk recurrence
// ===========================================================================
struct RcParams {
    const float *init_state;
    const uint8_t *blocks;
    size_t block_bytes;
    __nv_bfloat16 *out;
    float *final_state;
    unsigned *err;
    Geometry gm;
    long long *trace;
    ConvParams cv;      // KC > 0: the raw V tile is convolved in place, Q comes convolved from the workspace
    // For the backward pass: when save_s is set, the state at every chunk start (fp32, transposed:
    // [128][dv], S^T) and V_new (fp32 [64][dv]) go to per (slot, head) blocks save_stride floats
    // apart; out may then be null.
    float *save_s, *save_vn;
    int64_t save_stride;
};

// SAVE (the backward's forward scan): the chunk-start states and V_new go to p.save_s and p.save_vn,
// and the outputs are not written.
template <int KC, bool SAVE = false>
__global__ void __launch_bounds__(kThreadsRc, 1)
recur_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmv, const RcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * 128;
    // The backward's reverse scan does not read what this saving instance writes: it may start on
    // the free SMs once every CTA of this grid is resident (programmatic dependent launch; without
    // a programmatic dependent this is a no-op).
    if constexpr (SAVE)
        if (tid == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const Geometry gm = p.gm;
    const int H = gm.H, dv = gm.dv;
    int64_t tok0;
    int len;
    seq_span(gm, n, tok0, len);
    const int nch = ceil_div(len, kChunk);
    const int64_t slot0 = slot_base(gm, n);
    uint32_t *tmem_sh = reinterpret_cast<uint32_t *>(sm + R_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + R_MISC + 4);
    auto bar = [&](int i) -> uint32_t { return sb + R_BAR + 8u * (uint32_t)i; };
    auto early = [&](int c) -> uint32_t { return R_EARLY + (uint32_t)(c % kEarly) * kEarlyBytes; };
    auto late = [&](int c) -> uint32_t { return R_LATE + (uint32_t)(c % kLate) * kLateBytes; };

    if (tid == 0) {
        for (int i = 0; i < RB_COUNT; ++i) mbar_init(bar(i), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tmem_sh, 512);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tb = *tmem_sh;
    const uint32_t lane_base = tb + ((uint32_t)(32 * (warp & 3)) << 16);

    if (warp == 0) {
        // ------------------------------------------------------------ loads
        // lane 0: early ring half A (T', V); lane 3: half B (W~ | Q); lane 1: factor ring;
        // lane 2: late ring (Aqk^T, K->)
        if (lane < 4 && nch > 0) {
            if (lane == 0) { prefetch_tmap(&tmq); prefetch_tmap(&tmv); }
            const int slots = (lane == 0 || lane == 3) ? kEarly : (lane == 1 ? kScSlots : kLate);
            const int fbar = lane == 0 ? RB_EF : (lane == 1 ? RB_SCF : (lane == 2 ? RB_LF : RB_EFB));
            const int ebar = lane == 0 ? RB_EE : (lane == 1 ? RB_SCE : (lane == 2 ? RB_LE : RB_EEB));
            int last = -1;
            for (int c = 0; c < nch; ++c) {
                const int s = c % slots;
                if (c >= slots && !wait_bar(bar(ebar + s), ((c / slots) - 1) & 1, abort_flag, p.err)) break;
                const int z = (int)(tok0 + (int64_t)c * kChunk);
                const uint8_t *blk = p.blocks + ((size_t)(slot0 + c) * H + h) * p.block_bytes;
                const uint32_t fb = bar(fbar + s);
                if (lane == 0) {
                    const uint32_t base = sb + early(c);
                    mbar_expect_tx(fb, kEarlyTxA);
                    bulk_load(base + E_TP, blk + PB_TP, 16384, fb);                 // T'_hi, T'_lo
                    tma_load_3d(base + E_V, &tmv, j0, h, z, fb);
                    tma_load_3d(base + E_V + 8192, &tmv, j0 + 64, h, z, fb);
                } else if (lane == 3) {
                    const uint32_t base = sb + early(c);
                    mbar_expect_tx(fb, kEarlyTxB);
                    bulk_load(base + E_WQ, blk + PB_W, 8192, fb);                 // W~ d 0-63   -> rows 0-63
                    bulk_load(base + E_WQ + 16384, blk + PB_W + 8192, 8192, fb);  // W~ d 64-127
                    if (KC > 0) {   // the convolved Q left by the chunk-local kernel
                        bulk_load(base + E_WQ + 8192, blk + PB_QC, 8192, fb);
                        bulk_load(base + E_WQ + 24576, blk + PB_QC + 8192, 8192, fb);
                    } else {
                        tma_load_3d(base + E_WQ + 8192, &tmq, 0, h, z, fb);       // Q  d 0-63   -> rows 64-127
                        tma_load_3d(base + E_WQ + 24576, &tmq, 64, h, z, fb);     // Q  d 64-127
                    }
                } else if (lane == 1) {
                    mbar_expect_tx(fb, kScBytes);
                    bulk_load(sb + R_SCR + s * kScStride, blk + PB_SC, kScBytes, fb);
                } else {
                    const uint32_t base = sb + late(c);
                    mbar_expect_tx(fb, kLateTx);
                    if ((c & 1) == 0) {
                        bulk_load(base, blk + PB_AQT, kLateTx, fb);          // [Aqk^T | K->]
                    } else {
                        bulk_load(base, blk + PB_KT, 16384, fb);             // [K-> | Aqk^T]
                        bulk_load(base + 16384, blk + PB_AQT, 8192, fb);
                    }
                }
                last = c;
            }
            if (*abort_flag)   // let the copies in flight land before the CTA exits
                for (int c = (last >= slots ? last - slots + 1 : 0); c <= last; ++c)
                    mbar_wait(bar(fbar + c % slots), (c / slots) & 1, 10000000ull);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        // Per chunk three products (20 instructions):
        //   a1 : D1       = V^T T'_hi^T + V^T T'_lo^T       (N = 64,  K = 2 x 64)
        //   a2 : D1|D2A  -= S [W~ ; Q]^T                   (N = 128, K = 128)  V_new^T and -S Q^T
        //   c  : D2B|S   += V_new^T [Aqk^T | K->]           (N = 192, K = 64)   outputs and state
        // D2A and D2B (one pair per chunk parity) are re-zeroed by the output warps.
        if (lane == 0 && nch > 0) {
            const uint32_t id_a1 = idesc_bf16(128, 64, true, false);
            const uint32_t id_a2 = idesc_bf16(128, 128, false, false, true);   // negated B
            const uint32_t id_c = idesc_f16(128, 192, false, true);          // fp16 operands
            auto issue_a1 = [&](int c) -> bool {
                const uint32_t eb = sb + early(c);
                if (!wait_spin(bar(RB_EF + c % kEarly), (c / kEarly) & 1, abort_flag, p.err)) return false;
                if (KC > 0 && !wait_spin(bar(RB_VC + c % kEarly), (c / kEarly) & 1, abort_flag, p.err)) return false;
                fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)   // K-steps 0-3 against T'_hi, 4-7 against T'_lo
                    mma_ss(tb + tm_d1(c), smem_desc(eb + E_V + (ks & 3) * 2048, 8192, 1024),
                           smem_desc(eb + E_TP + (ks >> 2) * 8192 + (ks & 3) * 32, 16, 1024), id_a1, ks > 0);
                commit(bar(RB_EE + c % kEarly));   // half A may be refilled once a1 has read it
                return true;
            };
            auto issue_a2 = [&](int c) -> bool {
                const uint32_t eb = sb + early(c);
                if (!wait_spin(bar(RB_OFREE + (c & 1)), (c >> 1) & 1, abort_flag, p.err)) return false;
                if (!wait_spin(bar(RB_S), c & 1, abort_flag, p.err)) return false;
                if (!wait_spin(bar(RB_EFB + c % kEarly), (c / kEarly) & 1, abort_flag, p.err)) return false;
                GDN_TR(p.trace, 1, c, 0);
                fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_ss(tb + tm_d1(c), smem_desc(sb + R_SBF + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024),
                           smem_desc(eb + E_WQ + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024), id_a2, 1);
                commit(bar(RB_D1));
                commit(bar(RB_EEB + c % kEarly));
                GDN_TR(p.trace, 1, c, 4);
                return true;
            };
            bool ok = issue_a1(0) && issue_a2(0);
            for (int c = 0; c < nch && ok; ++c) {
                const uint32_t lb = sb + late(c);
                if (!wait_spin(bar(RB_LF + c % kLate), (c / kLate) & 1, abort_flag, p.err)) break;
                GDN_TR(p.trace, 1, c, 2);
                if (!wait_spin(bar(RB_X), c & 1, abort_flag, p.err)) break;
                GDN_TR(p.trace, 1, c, 3);
                if (!wait_spin(bar(RB_SP), c & 1, abort_flag, p.err)) break;   // state pre-decayed
                GDN_TR(p.trace, 1, c, 1);
                fence_after_sync();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tb + tm_c(c), smem_desc(sb + R_X + ks * 32, 16, 1024), smem_desc(lb + ks * 2048, 8192, 1024),
                           id_c, 1);
                commit(bar(RB_D2));
                commit(bar(RB_D2O + (c & 1)));
                if (c + 1 < nch && !(ok = issue_a1(c + 1) && issue_a2(c + 1))) break;
            }
            commit(bar(RB_FIN));   // every MMA must complete before tensor memory is released
            mbar_wait(bar(RB_FIN), 0, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp < 10) {
        // ------------------------------------------------------------ state epilogue (warps 2-9)
        // Each tensor-memory lane (row j of S) is served by two threads: half 0 owns
        // the first half of every row's columns, half 1 the second.  Per chunk:
        //   X : V_new^T -> bf16 shared tile (A of the merged c product)
        //   S : S -> bf16 shared tile (A of the next a2), then S <- e^{b_C} S (gates the next c)
        const int j = 32 * (warp & 3) + lane;
        const int hf = warp >= 6 ? 1 : 0;
        const bool leader = (warp == 2 && lane == 0);
        const size_t srow = (((size_t)n * H + h) * (size_t)dv + (size_t)(j0 + j)) * 128;
        auto gsync = [&](bool bad) -> bool { return group_sync_or(1, 256, bad); };
        auto gwait = [&](int b, uint32_t parity) -> bool {
            bool ok = true;
            if (leader) ok = wait_spin(bar(b), parity, abort_flag, p.err);
            return !gsync(!ok);
        };
        // the state at the start of chunk c: this thread's 64 entries of row j0 + j, stored transposed
        // (column d of the state at d dv), so that a warp's 32 rows of one column are one 128-B line
        auto save_state = [&](int c, const uint32_t (&sv)[64]) {
            float *dst = p.save_s + ((slot0 + c) * H + h) * p.save_stride + (size_t)(hf * 64) * dv + j0 + j;
#pragma unroll
            for (int e = 0; e < 64; ++e) dst[(size_t)e * dv] = __uint_as_float(sv[e]);
        };
        // 64 fp32 state entries (this thread's half of row j) -> the bf16 A tile of a2
        auto put_sbf = [&](const uint32_t (&sv)[64]) {
            uint8_t *row = sm + R_SBF + hf * 16384;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint4 w;
                w.x = pack_bf16(__uint_as_float(sv[ch * 8 + 0]), __uint_as_float(sv[ch * 8 + 1]));
                w.y = pack_bf16(__uint_as_float(sv[ch * 8 + 2]), __uint_as_float(sv[ch * 8 + 3]));
                w.z = pack_bf16(__uint_as_float(sv[ch * 8 + 4]), __uint_as_float(sv[ch * 8 + 5]));
                w.w = pack_bf16(__uint_as_float(sv[ch * 8 + 6]), __uint_as_float(sv[ch * 8 + 7]));
                *reinterpret_cast<uint4 *>(row + sw128_offset(j, ch * 8)) = w;
            }
        };
        if (nch == 0) {
            if (p.final_state)
                for (int d = hf * 64; d < hf * 64 + 64; d += 4) {
                    float4 v4 = p.init_state ? *reinterpret_cast<const float4 *>(p.init_state + srow + d)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                    *reinterpret_cast<float4 *>(p.final_state + srow + d) = v4;
                }
        } else do {
            {   // initial state: this thread's 64 entries of row j.  The bf16 copy (A of the
                // first a2) goes out before the first factor slot is waited for; the
                // pre-decayed fp32 state (gating the first c) after it.
                uint32_t sv[64];
#pragma unroll
                for (int e = 0; e < 64; e += 4) {
                    float4 v4 = p.init_state ? *reinterpret_cast<const float4 *>(p.init_state + srow + hf * 64 + e)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                    sv[e] = __float_as_uint(v4.x); sv[e + 1] = __float_as_uint(v4.y);
                    sv[e + 2] = __float_as_uint(v4.z); sv[e + 3] = __float_as_uint(v4.w);
                }
                put_sbf(sv);
                if constexpr (SAVE) save_state(0, sv);
                fence_proxy_async();
                if (gsync(*abort_flag)) break;
                if (leader) mbar_arrive(bar(RB_S));
                if (!gwait(RB_SCF, 0)) break;
                const float e0 = reinterpret_cast<const float *>(sm + R_SCR)[64];
#pragma unroll
                for (int e = 0; e < 64; ++e) sv[e] = __float_as_uint(e0 * __uint_as_float(sv[e]));
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    tmem_st16(lane_base + TM_S + hf * 64 + q * 16, *reinterpret_cast<uint32_t(*)[16]>(sv + q * 16));
                tmem_wait_st();
            }
            fence_before_sync();
            if (gsync(*abort_flag)) break;
            if (leader) mbar_arrive(bar(RB_SP));
            for (int c = 0; c < nch; ++c) {
                // ---- X: this thread's 32 tokens of V_new^T row j
                if (!gwait(RB_D1, c & 1)) break;
                if (leader) GDN_TR(p.trace, 2, c, 0);
                fence_after_sync();
                {
                    uint32_t a[32];
                    tmem_ld16(lane_base + tm_d1(c) + hf * 32, *reinterpret_cast<uint32_t(*)[16]>(a));
                    tmem_ld16(lane_base + tm_d1(c) + hf * 32 + 16, *reinterpret_cast<uint32_t(*)[16]>(a + 16));
                    tmem_wait_ld();
                    float xmax = 0.f;
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        uint4 w;
#pragma unroll
                        for (int e = 0; e < 8; ++e) xmax = fmaxf(xmax, fabsf(__uint_as_float(a[ch * 8 + e])));
                        w.x = pack_f16(__uint_as_float(a[ch * 8 + 0]), __uint_as_float(a[ch * 8 + 1]));
                        w.y = pack_f16(__uint_as_float(a[ch * 8 + 2]), __uint_as_float(a[ch * 8 + 3]));
                        w.z = pack_f16(__uint_as_float(a[ch * 8 + 4]), __uint_as_float(a[ch * 8 + 5]));
                        w.w = pack_f16(__uint_as_float(a[ch * 8 + 6]), __uint_as_float(a[ch * 8 + 7]));
                        *reinterpret_cast<uint4 *>(sm + R_X + sw128_offset(j, hf * 32 + ch * 8)) = w;
                    }
                    if (xmax > kF16Max) atomicExch(p.err, kDevErrRange);
                    if constexpr (SAVE) {   // V_new[t][j0 + j] for this thread's 32 tokens (a warp stores 128 B a token)
                        float *dst = p.save_vn + ((slot0 + c) * H + h) * p.save_stride + (size_t)(hf * 32) * dv + j0 + j;
#pragma unroll
                        for (int t = 0; t < 32; ++t) dst[(size_t)t * dv] = __uint_as_float(a[t]);
                    }
                }
                fence_proxy_async();
                fence_before_sync();
                if (gsync(*abort_flag)) break;
                if (leader) mbar_arrive(bar(RB_X));
                if (leader) GDN_TR(p.trace, 2, c, 4);
                // ---- S: this thread's 64 entries of row j
                if (!gwait(RB_D2, c & 1)) break;
                if (leader) GDN_TR(p.trace, 2, c, 1);
                fence_after_sync();
                if (c + 1 < nch) {
                    const int s1 = (c + 1) % kScSlots;
                    if (!gwait(RB_SCF + s1, ((c + 1) / kScSlots) & 1)) break;
                    const float e1 = reinterpret_cast<const float *>(sm + R_SCR + s1 * kScStride)[64];
                    uint32_t sv[64];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tmem_ld16(lane_base + TM_S + hf * 64 + q * 16, *reinterpret_cast<uint32_t(*)[16]>(sv + q * 16));
                    tmem_wait_ld();
                    put_sbf(sv);
                    fence_proxy_async();
                    if (gsync(*abort_flag)) break;
                    if (leader) mbar_arrive(bar(RB_S));   // the bf16 state is ready: the next a2 may start
                    if constexpr (SAVE) save_state(c + 1, sv);
                    if (leader) GDN_TR(p.trace, 2, c, 2);
#pragma unroll
                    for (int e = 0; e < 64; ++e) sv[e] = __float_as_uint(e1 * __uint_as_float(sv[e]));
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tmem_st16(lane_base + TM_S + hf * 64 + q * 16, *reinterpret_cast<uint32_t(*)[16]>(sv + q * 16));
                    tmem_wait_st();
                    fence_before_sync();
                    if (gsync(*abort_flag)) break;
                    if (leader) mbar_arrive(bar(RB_SP));  // the fp32 state is pre-decayed for the next c
                    if (leader) GDN_TR(p.trace, 2, c, 5);
                } else if (p.final_state) {   // one tensor-memory round trip, then 16-B stores
                    uint32_t u[64];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tmem_ld16(lane_base + TM_S + hf * 64 + q * 16, *reinterpret_cast<uint32_t(*)[16]>(u + q * 16));
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 64; e += 4)
                        *reinterpret_cast<float4 *>(p.final_state + srow + hf * 64 + e) =
                            make_float4(__uint_as_float(u[e]), __uint_as_float(u[e + 1]),
                                        __uint_as_float(u[e + 2]), __uint_as_float(u[e + 3]));
                }
            }
        } while (false);
    } else {
        // ------------------------------------------------------------ output epilogue (warps 10-13)
        // O = fq . (Q S^T) + Aqk V_new = D2B - fq . D2A; the chunk-parity accumulators are
        // re-zeroed for the chunk after next, then O goes through a [64 r][128 j] bf16 staging
        // tile (in the chunk's late stage, whose operands the finished c product no longer
        // needs) to coalesced 16-B stores.
        const int j = 32 * (warp & 3) + lane;   // output column j0 + j
        const bool leader = (warp == 10 && lane == 0);
        auto osync = [&](bool bad) -> bool { return group_sync_or(2, 128, bad); };
        auto zero_d2 = [&](int c) {
            uint32_t z[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) z[e] = 0u;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                tmem_st16(lane_base + tm_d2a(c) + q * 16, z);
                tmem_st16(lane_base + tm_d2b(c) + q * 16, z);
            }
            tmem_wait_st();
        };
        zero_d2(0);
        zero_d2(1);
        fence_before_sync();
        if (!osync(*abort_flag) && leader && nch > 0) {   // phase 0 of each parity: zero accumulators
            mbar_arrive(bar(RB_OFREE));
            mbar_arrive(bar(RB_OFREE + 1));
        }
        // With the block prologue fused in, these warps also turn each landed raw V tile into
        // SiLU(short convolution) in place (bf16, exactly as the block prologue writes v), two
        // chunks ahead of its a1 product.  Thread j takes the channel pair j0 + 2(j % 64),
        // j0 + 2(j % 64) + 1 over rows 32(j / 64) .. 32(j / 64) + 31.
        const int cpr = 2 * (j & 63), chalf = j >> 6;
        const int Cw = 2 * gm.dk + dv, vchan = 2 * gm.dk + j0 + cpr;
        constexpr int KH = KC > 1 ? KC - 1 : 1;
        float2 wv[KC > 0 ? KC : 1];
#pragma unroll
        for (int jj = 0; jj < KC; ++jj)
            wv[jj] = make_float2(p.cv.wv[((int64_t)h * dv + j0 + cpr) * KC + jj],
                                 p.cv.wv[((int64_t)h * dv + j0 + cpr + 1) * KC + jj]);
        // raw input of this thread's channel pair at token position pos of sequence n (the carried
        // state before the sequence's first token)
        auto raw_v = [&](int64_t pos) -> float2 {
            if (pos >= tok0)
                return unpack_bf16(*reinterpret_cast<const uint32_t *>(p.cv.xv + pos * H * dv + (int64_t)h * dv + j0 + cpr));
            if (p.cv.state_in)
                return unpack_bf16(*reinterpret_cast<const uint32_t *>(
                    p.cv.state_in + (((int64_t)n * (KC - 1) + (KC - 1) + (pos - tok0)) * H + h) * Cw + vchan));
            return make_float2(0.f, 0.f);
        };
        auto convert_v = [&](int cc) -> bool {
          if constexpr (KC > 0) {
            const int s = cc % kEarly;
            bool okv = true;
            if (leader) okv = wait_bar(bar(RB_EF + s), (cc / kEarly) & 1, abort_flag, p.err);
            if (osync(!okv)) return false;
            uint8_t *tile = sm + early(cc) + E_V + (cpr >> 6) * 8192;
            float2 hist[KH];
            uint32_t raw[32];
#pragma unroll
            for (int m = 0; m < KC - 1; ++m)   // the KC-1 inputs before the thread's first row
                hist[m] = chalf ? unpack_bf16(*reinterpret_cast<const uint32_t *>(
                                      tile + sw128_offset(32 - (KC - 1) + m, cpr & 63)))
                                : raw_v(tok0 + (int64_t)cc * kChunk - (KC - 1) + m);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                raw[i] = *reinterpret_cast<const uint32_t *>(tile + sw128_offset(32 * chalf + i, cpr & 63));
            if (osync(*abort_flag)) return false;   // every raw row is read before any is overwritten
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float2 xt = unpack_bf16(raw[i]);
                float2 z = make_float2(wv[KC - 1].x * xt.x, wv[KC - 1].y * xt.y);
#pragma unroll
                for (int jj = 0; jj < KC - 1; ++jj) {
                    z.x += wv[jj].x * hist[jj].x;
                    z.y += wv[jj].y * hist[jj].y;
                }
                *reinterpret_cast<uint32_t *>(tile + sw128_offset(32 * chalf + i, cpr & 63)) =
                    pack_bf16(conv_silu(z.x), conv_silu(z.y));
#pragma unroll
                for (int m = 0; m + 1 < KC - 1; ++m) hist[m] = hist[m + 1];
                if (KC > 1) hist[KH - 1] = xt;
            }
            if (cc == nch - 1 && chalf == 0 && p.cv.state_out)   // the sequence's last KC-1 inputs
#pragma unroll
                for (int m = 0; m < KC - 1; ++m) {
                    const float2 x = raw_v(tok0 + len - (KC - 1) + m);
                    *reinterpret_cast<uint32_t *>(p.cv.state_out + (((int64_t)n * (KC - 1) + m) * H + h) * Cw + vchan) =
                        pack_bf16(x.x, x.y);
                }
            fence_proxy_async();
            if (osync(*abort_flag)) return false;
            if (leader) mbar_arrive(bar(RB_VC + s));
          }
            return true;
        };
        bool nch_out_abort = false;
        if constexpr (KC > 0) {
            if (nch == 0 && p.cv.state_out) {
                // an empty sequence carries its convolution state through unchanged (this CTA's v
                // channels; the CTA of the first v slice also takes q and k)
                const int64_t base = ((int64_t)n * (KC - 1) * H + h) * Cw;
                for (int e = j; e < 64 + (j0 == 0 ? gm.dk : 0); e += 128) {   // channel pairs
                    const int ch = e < 64 ? vchan - 2 * (j & 63) + 2 * e : 2 * (e - 64);
#pragma unroll
                    for (int m = 0; m < KC - 1; ++m) {
                        const int64_t o = base + (int64_t)m * H * Cw + ch;
                        *reinterpret_cast<uint32_t *>(p.cv.state_out + o) =
                            p.cv.state_in ? *reinterpret_cast<const uint32_t *>(p.cv.state_in + o) : 0u;
                    }
                }
            }
            bool okc = true;
            for (int cc = 0; cc < 2 && cc < nch && okc; ++cc) okc = convert_v(cc);
            if (!okc) nch_out_abort = true;
        }
        for (int c = 0; c < nch && !nch_out_abort; ++c) {
            const float *fq = reinterpret_cast<const float *>(sm + R_SCR + (c % kScSlots) * kScStride);
            bool ok = true;
            if (leader) {
                ok = wait_spin(bar(RB_SCF + c % kScSlots), (c / kScSlots) & 1, abort_flag, p.err);
                ok = ok && wait_spin(bar(RB_D2O + (c & 1)), (c >> 1) & 1, abort_flag, p.err);
            }
            if (osync(!ok)) break;
            if (leader && fq[65] != 0.f) atomicExch(p.err, kDevErrRange);   // flagged by the chunk-local kernel
            if (leader) GDN_TR(p.trace, 0, c, 0);
            fence_after_sync();
            uint8_t *stg = sm + late(c);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t a[16], b[16];
                tmem_ld16(lane_base + tm_d2a(c) + q * 16, a);
                tmem_ld16(lane_base + tm_d2b(c) + q * 16, b);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int r = q * 16 + e;
                    *reinterpret_cast<__nv_bfloat16 *>(stg + (r * 128 + j) * 2) =
                        __float2bfloat16_rn(__uint_as_float(b[e]) - fq[r] * __uint_as_float(a[e]));
                }
            }
            zero_d2(c);
            fence_before_sync();
            if (osync(*abort_flag)) break;
            if (leader && c + 2 < nch) mbar_arrive(bar(RB_OFREE + (c & 1)));   // drained and re-zeroed
            if (leader) GDN_TR(p.trace, 0, c, 1);
            const int rows = min(kChunk, len - c * kChunk);
            __nv_bfloat16 *obase = p.out + (size_t)(tok0 + (int64_t)c * kChunk) * H * dv + (size_t)h * dv + j0;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int idx = it * 128 + j, r = idx >> 4, ch = idx & 15;
                if (!SAVE && r < rows)
                    *reinterpret_cast<uint4 *>(obase + (size_t)r * H * dv + ch * 8) =
                        *reinterpret_cast<const uint4 *>(stg + r * 256 + ch * 16);
            }
            if (osync(*abort_flag)) break;
            if (leader) {
                mbar_arrive(bar(RB_LE + c % kLate));       // the late stage may be refilled
                mbar_arrive(bar(RB_SCE + c % kScSlots));   // and the factor slot
            }
            if (leader) GDN_TR(p.trace, 0, c, 2);
            if (KC > 0 && c + 2 < nch && !convert_v(c + 2)) break;
        }
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tb, 512);
    }
}

// ===========================================================================
// self-test of the bounded wait
// ===========================================================================
// One CTA waits, through the same bounded wait as the kernels above, on an mbarrier
// phase that nothing completes.  The wait gives up after limit_ns, records
// kDevErrTimeout in the error word and raises the CTA's abort flag, and every thread
// leaves; nothing faults and the context stays usable.
__global__ void __launch_bounds__(128)
wait_selftest_kernel(unsigned *err, uint64_t limit_ns)
{
    __shared__ uint64_t barrier_word;
    __shared__ int abort_word;
    const uint32_t b = smem_u32(&barrier_word);
    volatile int *abort_flag = &abort_word;
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) wait_bar(b, 0, abort_flag, err, limit_ns);   // no arrival ever comes
    __syncthreads();
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// [rows, H, d] bf16 viewed as a 3-D tensor (d innermost); box 64 x 1 x 64, 128-B swizzle.
bool make_tmap(CUtensorMap *m, const void *base, int d, int H, int64_t rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

#ifdef GDN_KERNEL_TRACE
extern "C" void gdn_debug_set_trace(long long *buf) { g_trace_buffer = buf; }
#endif

bool chunk_tc_supported(int dt, int dk, int dv, int64_t tokens)
{
    return dt == 1 && dk == 128 && dv % 128 == 0 && tokens > 0 && tokens < ((int64_t)1 << 31);
}

cudaError_t launch_wait_selftest(unsigned *err, uint64_t limit_ns, cudaStream_t st)
{
    wait_selftest_kernel<<<1, 128, 0, st>>>(err, limit_ns);
    return cudaGetLastError();
}

size_t chunk_tc_workspace_bytes(int64_t slots, int H, bool fused)
{
    return kWsHeader + (size_t)slots * H * (fused ? kPrepBlockFused : kPrepBlock);
}

namespace {

template <int KC>
cudaError_t launch_pair(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const UtParams &up,
                        const RcParams &rp, const Geometry &gm, int64_t slots, cudaStream_t st)
{
    cudaError_t e = cudaFuncSetAttribute(ut_tc_kernel<KC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemUt);
    if (e != cudaSuccess) return e;
    ut_tc_kernel<KC><<<dim3((unsigned)slots, gm.H), kThreadsUt, kSmemUt, st>>>(tq, tk, up);
    if constexpr (KC == 0) {
        if (rp.save_s) {
            e = cudaFuncSetAttribute(recur_tc_kernel<0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemRc);
            if (e != cudaSuccess) return e;
            recur_tc_kernel<0, true><<<dim3(gm.N, gm.H, gm.dv / 128), kThreadsRc, kSmemRc, st>>>(tq, tv, rp);
            return cudaGetLastError();
        }
    }
    e = cudaFuncSetAttribute(recur_tc_kernel<KC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemRc);
    if (e != cudaSuccess) return e;
    recur_tc_kernel<KC><<<dim3(gm.N, gm.H, gm.dv / 128), kThreadsRc, kSmemRc, st>>>(tq, tv, rp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t st)
{
    const int64_t rows = (int64_t)a.gm.B * a.gm.T;
    const PrologueArgs *f = a.fuse;
    CUtensorMap tq, tk, tv;
    if (!make_tmap(&tq, f ? f->xq : a.q, a.gm.dk, a.gm.H, rows) || !make_tmap(&tk, f ? f->xk : a.k, a.gm.dk, a.gm.H, rows) ||
        !make_tmap(&tv, f ? f->xv : a.v, a.gm.dv, a.gm.H, rows))
        return cudaErrorInvalidValue;
    long long *trace = nullptr;
#ifdef GDN_KERNEL_TRACE
    trace = g_trace_buffer;
#endif
    uint8_t *blocks = a.blocks ? reinterpret_cast<uint8_t *>(a.blocks) : reinterpret_cast<uint8_t *>(a.workspace) + kWsHeader;
    unsigned *err = reinterpret_cast<unsigned *>(a.workspace);
    ConvParams cv{};
    if (f) {
        cv.xq = reinterpret_cast<const __nv_bfloat16 *>(f->xq);
        cv.xk = reinterpret_cast<const __nv_bfloat16 *>(f->xk);
        cv.xv = reinterpret_cast<const __nv_bfloat16 *>(f->xv);
        cv.wq = f->wq; cv.wk = f->wk; cv.wv = f->wv;
        cv.a = f->a; cv.b = f->b; cv.A_log = f->A_log; cv.dt_bias = f->dt_bias;
        cv.state_in = reinterpret_cast<const __nv_bfloat16 *>(f->state_in);
        cv.state_out = reinterpret_cast<__nv_bfloat16 *>(f->state_out);
    }
    const size_t block_bytes = a.blocks ? a.block_stride : (f ? kPrepBlockFused : kPrepBlock);

    UtParams up;
    up.g = a.g; up.beta = a.beta; up.blocks = blocks; up.block_bytes = block_bytes; up.err = err; up.gm = a.gm;
    up.scale = a.scale; up.l2 = a.l2; up.trace = trace; up.cv = cv;
    RcParams rp;
    rp.init_state = a.init_state; rp.blocks = blocks; rp.block_bytes = block_bytes;
    rp.out = reinterpret_cast<__nv_bfloat16 *>(a.out);
    rp.final_state = a.final_state; rp.err = err; rp.gm = a.gm; rp.trace = trace; rp.cv = cv;
    rp.save_s = a.save_s; rp.save_vn = a.save_vn; rp.save_stride = a.save_stride;
    switch (f ? f->K : 0) {
        case 0: return launch_pair<0>(tq, tk, tv, up, rp, a.gm, a.slots, st);
        case 1: return launch_pair<1>(tq, tk, tv, up, rp, a.gm, a.slots, st);
        case 2: return launch_pair<2>(tq, tk, tv, up, rp, a.gm, a.slots, st);
        case 3: return launch_pair<3>(tq, tk, tv, up, rp, a.gm, a.slots, st);
        case 4: return launch_pair<4>(tq, tk, tv, up, rp, a.gm, a.slots, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gdn
