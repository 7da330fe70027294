// chunk_tc.cu -- fused chunked forward of the gated delta rule on the tensor
// cores (tcgen05 + tensor memory + TMA), bf16 inputs, dk = 128, dv % 128 == 0.
//
// One CTA per (sequence, head, 128-row slice of S) runs every step of
// "Gated Delta Networks: Improving Mamba2 with Delta Rule", §3.3 for its
// sequence, chunk after chunk, with the fp32 state S resident in tensor
// memory for the whole sequence.  Per chunk of C = 64 tokens (row-stacked):
//
//   prologue   b_r = sum_{i<=r} g_i; rk_r = 1/||k_r||, rq_r = scale/||q_r||
//   P1 (MMA)   G = [K; Q] K^T                              (128 x 64, fp32)
//   Gram mask  L_ri  = beta_r e^{b_r-b_i} rk_r rk_i G_ri,   i < r   (system)
//              Aqk_ri = e^{b_r-b_i} rq_r rk_i G_(64+r)i,    i <= r  (Q K^T o Gamma)
//   solve      T = (I + L)^{-1}  (blocked: 16x16 diagonal blocks by forward
//              substitution, then two levels of block merges)
//              T'  = T diag(beta),  T'' = T diag(beta e^b rk)
//   P2 (MMA)   W~^T = K^T T''^T     (W~ = W<- of the pages, normalised keys)
//   a1, a2     V_new^T = V^T T'^T - S W~^T                 (U~ - W<- S^T)^T
//   b, c1      O^T = S Q<-^T + V_new^T Aqk^T,   Q<- = diag(e^b rq) Q
//   c2         S  <- e^{b_C} S + V_new^T K->,   K-> = diag(e^{b_C-b} rk) K
//
// All gate ratios are exp(b_r - b_i) with i <= r (never 1/gamma), so heavy
// decay cannot overflow.  The output mask is the decay mask Gamma
// ("【论文解读】Gated Delta Network", §二(一)2(3)).
//
// Warp roles (320 threads):
//   warp 0      TMA producer (q/k/v tiles, 128-B swizzle) and TMEM allocator
//   warp 1      single-thread tcgen05.mma issuer
//   warps 2-5   "prep": prologue, Gram masking, solve, operand preparation for
//               chunk c+1 while the chain runs chunk c
//   warps 6-9   "chain": tensor-memory epilogues of the recurrence (row j of
//               S per thread), output stores, final state
// Every wait is bounded (globaltimer); a timeout records GDN device error
// kDevErrTimeout in the workspace header, raises a CTA-wide abort flag, and
// all roles unwind to the common exit, where tensor memory is released.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {
namespace {

using namespace umma;

constexpr int kThreadsTc = 320;
constexpr uint32_t kQKStage = 32768;   // [K kb0][Q kb0][K kb1][Q kb1], 8 KB each (64 rows x 128 B)
constexpr uint32_t kVStage = 16384;    // [V cols 0-63][V cols 64-127]
constexpr uint32_t LDA = 65;           // fp32 row pitch of L (conflict-free row-per-thread writes)
constexpr uint32_t LDL = 68;           // fp32 row pitch of T (16-B aligned rows for vector loads)
constexpr float kLog2e = 1.4426950408889634f;

constexpr uint32_t OFF_QK = 0;
constexpr uint32_t OFF_V = OFF_QK + 3 * kQKStage;
constexpr uint32_t OFF_TP = OFF_V + 2 * kVStage;      // T'   bf16 [64 r][64 i] K-major
constexpr uint32_t OFF_TPP = OFF_TP + 8192;           // T''  bf16 [64 r][64 i] K-major
constexpr uint32_t OFF_WT = OFF_TPP + 8192;           // W~^T bf16 [128 d][64 r] (MN-major B)
constexpr uint32_t OFF_AQK = OFF_WT + 16384;          // Aqk  bf16 [64 r][64 i] x 2 buffers
constexpr uint32_t OFF_LF = OFF_AQK + 16384;          // L    fp32 [64][LDA]
constexpr uint32_t OFF_TF = OFF_LF + 64 * LDA * 4;    // T    fp32 [64][LDL]
constexpr uint32_t OFF_MT = OFF_TF + 64 * LDL * 4;    // merge temp fp32 [32][33]
constexpr uint32_t OFF_SC = OFF_MT + 32 * 33 * 4;     // per stage: b, beta, rk, rq, spare [5][64] fp32
constexpr uint32_t OFF_BAR = OFF_SC + 3 * 5 * 64 * 4;
constexpr int kNumBars = 32;
constexpr uint32_t OFF_MISC = OFF_BAR + kNumBars * 8;
constexpr uint32_t kSmemTc = OFF_MISC + 64 + 1024;    // + slack for 1024-B alignment
static_assert(kSmemTc <= 232448, "shared memory budget exceeded");
static_assert(OFF_LF % 16 == 0 && OFF_TF % 16 == 0 && OFF_MT % 16 == 0 && OFF_SC % 16 == 0, "alignment");

// tensor-memory columns (512 allocated)
constexpr uint32_t TM_S = 0;      // fp32 state, 128 columns
constexpr uint32_t TM_SBF = 128;  // bf16 state (A operand), 64 columns
constexpr uint32_t TM_D1 = 192;   // V_new^T accumulator, 64
constexpr uint32_t TM_D2 = 256;   // O^T accumulator, 64
constexpr uint32_t TM_X1 = 320;   // V_new^T bf16 (A operand), 32
constexpr uint32_t TM_P1 = 384;   // [K;Q] K^T accumulator, 64
constexpr uint32_t TM_P2 = 448;   // W~^T accumulator, 64

// mbarriers
enum : int {
    B_QKF = 0,      // [3] q/k tile landed
    B_QKE = 3,      // [3] q/k stage free (chain done with K-> and Q<-)
    B_VF = 6,       // [2] v tile landed
    B_VE = 8,       // [2] v stage free
    B_P1 = 10,      // P1 accumulator ready
    B_P2 = 11,      // P2 accumulator ready
    B_TRDY = 12,    // T', T'' written
    B_PREP = 13,    // all chain operands of the chunk ready
    B_TWFREE = 14,  // T' and W~^T of the previous chunk consumed
    B_AQKF = 15,    // [2] Aqk buffer consumed
    B_D1 = 17,      // V_new^T accumulated
    B_D2 = 18,      // O^T and the state update accumulated
    B_X = 19,       // V_new^T bf16 written to tensor memory (and D1 drained)
    B_S = 20,       // bf16 state written, fp32 state pre-decayed (and D2 drained)
    B_GATE = 21,    // [3] cumulative gates of a stage written
    B_FIN = 24      // final drain of the MMA pipe
};

constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s: legitimate waits are microseconds

struct TcParams {
    const float *g, *beta, *init_state;
    __nv_bfloat16 *out;
    float *final_state;
    unsigned *err;
    Geometry gm;
    float scale;
    int l2;
#ifdef GDN_KERNEL_TRACE
    long long *trace;
#endif
};

// Development-only phase timestamps (SM clock) of the first CTA; compiled out
// of the library unless GDN_KERNEL_TRACE is defined.
#ifdef GDN_KERNEL_TRACE
#define GDN_TR(role, c, ev)                                                                          \
    do {                                                                                             \
        if (p.trace && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (c) < 16)            \
            p.trace[((role) * 16 + (c)) * 16 + (ev)] = clock64();                                    \
    } while (0)
#else
#define GDN_TR(role, c, ev) do { } while (0)
#endif

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag, unsigned *err)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
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

__device__ __forceinline__ float2 unpack_bf16(uint32_t u)
{
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(v);
}

// Sum of squares of the 64 bf16 of one 128-B row segment (row index r, used
// only to visit the 16-B chunks in an order that spreads consecutive rows
// over all shared-memory banks).
__device__ __forceinline__ float row_sumsq(const uint8_t *row, int r)
{
    float ss = 0.f;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const uint4 u = *reinterpret_cast<const uint4 *>(row + ((ch ^ r) & 7) * 16);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16(w[e]);
            ss += f.x * f.x + f.y * f.y;
        }
    }
    return ss;
}

// Multiply the 64 bf16 of one 128-B row segment by f, in place (chunk order as above).
__device__ __forceinline__ void row_scale(uint8_t *row, int r, float f)
{
#pragma unroll
    for (int ch0 = 0; ch0 < 8; ++ch0) {
        const int ch = (ch0 ^ r) & 7;
        uint4 u = *reinterpret_cast<uint4 *>(row + ch * 16);
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 x = unpack_bf16(w[e]);
            w[e] = pack_bf16(x.x * f, x.y * f);
        }
        *reinterpret_cast<uint4 *>(row + ch * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// T = (I + L)^{-1} for a strictly lower 64x64 L (row pitch LDA; T pitch LDL), 128 threads.
// 16x16 diagonal blocks by forward substitution (one thread per column),
// then the block rule [A 0; C B]^{-1} = [A^-1 0; -B^-1 C A^-1  B^-1] for the
// 16->32 and 32->64 merges.
__device__ __forceinline__ void solve_unit_lower(const float *__restrict__ Lf, float *__restrict__ Tf,
                                                 float *__restrict__ Mt, int pid)
{
    for (int e = pid; e < 64 * (int)LDL; e += 128) Tf[e] = 0.f;
    group_sync(1, 128);
    if (pid < 64) {
        const int base = (pid >> 4) * 16, cc = pid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < r; ++i) acc += Lf[(base + r) * LDA + base + i] * x[i];
            x[r] = (r == cc) ? 1.f : ((r < cc) ? 0.f : -acc);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Tf[(base + r) * LDL + base + cc] = x[r];
    }
    group_sync(1, 128);
    {   // 16 -> 32 merges: blocks (a0 = 0, b0 = 16) and (a0 = 32, b0 = 48)
        const int m = pid >> 6, q = pid & 63, r = q >> 2, cg = (q & 3) * 4;
        const int a0 = m * 32, b0 = a0 + 16;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float l = Lf[(b0 + r) * LDA + a0 + i];
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[c] += l * Tf[(a0 + i) * LDL + a0 + cg + c];
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) Mt[m * 272 + r * 17 + cg + c] = acc[c];
        group_sync(1, 128);
        float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float t = Tf[(b0 + r) * LDL + b0 + i];
#pragma unroll
            for (int c = 0; c < 4; ++c) o[c] += t * Mt[m * 272 + i * 17 + cg + c];
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) Tf[(b0 + r) * LDL + a0 + cg + c] = -o[c];
    }
    group_sync(1, 128);
    {   // 32 -> 64 merge
        const int r = pid >> 2, cg = (pid & 3) * 8;
        float acc[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = 0.f;
#pragma unroll 8
        for (int i = 0; i < 32; ++i) {
            const float l = Lf[(32 + r) * LDA + i];
            const float4 t0 = *reinterpret_cast<const float4 *>(Tf + i * LDL + cg);
            const float4 t1 = *reinterpret_cast<const float4 *>(Tf + i * LDL + cg + 4);
            acc[0] += l * t0.x; acc[1] += l * t0.y; acc[2] += l * t0.z; acc[3] += l * t0.w;
            acc[4] += l * t1.x; acc[5] += l * t1.y; acc[6] += l * t1.z; acc[7] += l * t1.w;
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) Mt[r * 33 + cg + c] = acc[c];
        group_sync(1, 128);
        float o[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) o[c] = 0.f;
#pragma unroll 8
        for (int i = 0; i < 32; ++i) {
            const float t = Tf[(32 + r) * LDL + 32 + i];
#pragma unroll
            for (int c = 0; c < 8; ++c) o[c] += t * Mt[i * 33 + cg + c];
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) Tf[(32 + r) * LDL + cg + c] = -o[c];
    }
    group_sync(1, 128);
}

__global__ void __launch_bounds__(kThreadsTc, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv, const TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * 128;
    const Geometry gm = p.gm;
    const int H = gm.H, dv = gm.dv;
    int64_t tok0;
    int len;
    seq_span(gm, n, tok0, len);
    const int nch = ceil_div(len, kChunk);
    uint32_t *tmem_sh = reinterpret_cast<uint32_t *>(sm + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_MISC + 4);
    float *sc_all = reinterpret_cast<float *>(sm + OFF_SC);
    auto bar = [&](int i) -> uint32_t { return sb + OFF_BAR + 8u * (uint32_t)i; };

    // the first CTA clears the call's device error word; any timeout is at
    // least kWaitLimitNs later, long after this store
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && tid == 0) *p.err = kDevErrNone;
    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
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
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && nch > 0) {
            prefetch_tmap(&tmq);
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmv);
            int last_qk = -1, last_v = -1;
            for (int c = 0; c < nch; ++c) {
                const int s = c % 3, sv = c & 1;
                const int z = (int)(tok0 + (int64_t)c * kChunk);
                if (c >= 3 && !wait_bar(bar(B_QKE + s), ((c / 3) - 1) & 1, abort_flag, p.err)) break;
                const uint32_t st = sb + OFF_QK + s * kQKStage;
                GDN_TR(3, c, 0);
                mbar_expect_tx(bar(B_QKF + s), kQKStage);
                tma_load_3d(st, &tmk, 0, h, z, bar(B_QKF + s));
                tma_load_3d(st + 8192, &tmq, 0, h, z, bar(B_QKF + s));
                tma_load_3d(st + 16384, &tmk, 64, h, z, bar(B_QKF + s));
                tma_load_3d(st + 24576, &tmq, 64, h, z, bar(B_QKF + s));
                last_qk = c;
                if (c >= 2 && !wait_bar(bar(B_VE + sv), ((c >> 1) - 1) & 1, abort_flag, p.err)) break;
                const uint32_t vt = sb + OFF_V + sv * kVStage;
                mbar_expect_tx(bar(B_VF + sv), kVStage);
                tma_load_3d(vt, &tmv, j0, h, z, bar(B_VF + sv));
                tma_load_3d(vt + 8192, &tmv, j0 + 64, h, z, bar(B_VF + sv));
                last_v = c;
            }
            if (*abort_flag) {
                // let the copies still in flight land before the CTA exits
                for (int c = (last_qk > 1 ? last_qk - 2 : 0); c <= last_qk; ++c)
                    mbar_wait(bar(B_QKF + c % 3), (c / 3) & 1, 10000000ull);
                for (int c = (last_v > 0 ? last_v - 1 : 0); c <= last_v; ++c)
                    mbar_wait(bar(B_VF + (c & 1)), (c >> 1) & 1, 10000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && nch > 0) {
            const uint32_t id_p1 = idesc_bf16(128, 64, false, false);
            const uint32_t id_p2 = idesc_bf16(128, 64, true, false);
            const uint32_t id_a1 = idesc_bf16(128, 64, true, false);
            const uint32_t id_a2 = idesc_bf16(128, 64, false, true, true);   // negated B: -S W~^T
            const uint32_t id_b = idesc_bf16(128, 64, false, false);
            const uint32_t id_c1 = idesc_bf16(128, 64, false, false);
            const uint32_t id_c2 = idesc_bf16(128, 128, false, true);
            auto stage = [&](int c) -> uint32_t { return sb + OFF_QK + (uint32_t)(c % 3) * kQKStage; };
            auto issue_p1 = [&](int c) {       // G = [K; Q] K^T
                const uint32_t st = stage(c);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
                    mma_ss(tb + TM_P1, smem_desc(st + off, 16, 1024), smem_desc(st + off, 16, 1024), id_p1, ks > 0);
                }
                commit(bar(B_P1));
            };
            auto issue_p2 = [&](int c) {       // W~^T = K^T T''^T
                const uint32_t st = stage(c);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_ss(tb + TM_P2, smem_desc(st + ks * 2048, 16384, 1024),
                           smem_desc(sb + OFF_TPP + ks * 32, 16, 1024), id_p2, ks > 0);
                commit(bar(B_P2));
            };
            bool ok = wait_bar(bar(B_QKF), 0, abort_flag, p.err);
            if (ok) issue_p1(0);
            ok = ok && wait_bar(bar(B_TRDY), 0, abort_flag, p.err);
            if (ok) { fence_after_sync(); issue_p2(0); }
            for (int c = 0; c < nch && ok; ++c) {
                if (!wait_bar(bar(B_PREP), c & 1, abort_flag, p.err)) break;
                GDN_TR(1, c, 0);
                fence_after_sync();
                if (c + 1 < nch) {
                    if (!wait_bar(bar(B_QKF + (c + 1) % 3), ((c + 1) / 3) & 1, abort_flag, p.err)) break;
                    issue_p1(c + 1);
                }
                if (!wait_bar(bar(B_VF + (c & 1)), (c >> 1) & 1, abort_flag, p.err)) break;
                if (c > 0 && !wait_bar(bar(B_X), (c - 1) & 1, abort_flag, p.err)) break;   // D1 drained
                GDN_TR(1, c, 1);
                fence_after_sync();
                {   // a1: D1 = V^T T'^T
                    const uint32_t vt = sb + OFF_V + (uint32_t)(c & 1) * kVStage;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_ss(tb + TM_D1, smem_desc(vt + ks * 2048, 8192, 1024),
                               smem_desc(sb + OFF_TP + ks * 32, 16, 1024), id_a1, ks > 0);
                }
                if (!wait_bar(bar(B_S), c & 1, abort_flag, p.err)) break;
                GDN_TR(1, c, 2);
                fence_after_sync();
                {   // a2: D1 -= S W~^T
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        mma_ts(tb + TM_D1, tb + TM_SBF + ks * 8, smem_desc(sb + OFF_WT + ks * 2048, 16384, 1024),
                               id_a2, 1);
                    commit(bar(B_D1));
                    commit(bar(B_TWFREE));
                }
                // the chain's second half and the next chunk's P2, whichever is ready first
                bool need_c = true, need_p2 = (c + 1 < nch);
                const uint64_t t0 = globaltimer_ns();
                while (need_c || need_p2) {
                    bool idle = true;
                    if (need_c && mbar_try_wait(bar(B_X), c & 1)) {
                        // (the chain epilogue drained D2 of the previous chunk before arriving here)
                        fence_after_sync();
                        const uint32_t st = stage(c);
                        const uint32_t aq = sb + OFF_AQK + (uint32_t)(c & 1) * 8192;
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {   // b: D2 = S Q<-^T
                            const uint32_t off = 8192 + (ks >> 2) * 16384 + (ks & 3) * 32;
                            mma_ts(tb + TM_D2, tb + TM_SBF + ks * 8, smem_desc(st + off, 16, 1024), id_b, ks > 0);
                        }
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)   // c1: D2 += V_new^T Aqk^T
                            mma_ts(tb + TM_D2, tb + TM_X1 + ks * 8, smem_desc(aq + ks * 32, 16, 1024), id_c1, 1);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)   // c2: S += V_new^T K->
                            mma_ts(tb + TM_S, tb + TM_X1 + ks * 8, smem_desc(st + ks * 2048, 16384, 1024), id_c2, 1);
                        commit(bar(B_D2));
                        commit(bar(B_QKE + c % 3));
                        commit(bar(B_AQKF + (c & 1)));
                        need_c = false;
                        idle = false;
                        GDN_TR(1, c, 3);
                    }
                    if (need_p2 && mbar_try_wait(bar(B_TRDY), (c + 1) & 1)) {
                        fence_after_sync();
                        issue_p2(c + 1);
                        need_p2 = false;
                        idle = false;
                        GDN_TR(1, c, 4);
                    }
                    if (idle) __nanosleep(32);
                    if (*abort_flag) { ok = false; break; }
                    if (globaltimer_ns() - t0 > kWaitLimitNs) {
                        *abort_flag = 1;
                        atomicExch(p.err, kDevErrTimeout);
                        ok = false;
                        break;
                    }
                }
            }
            // every MMA issued above must complete before tensor memory is released
            commit(bar(B_FIN));
            mbar_wait(bar(B_FIN), 0, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------------ prep group
        const int prow = 32 * (warp & 3) + lane;   // tensor-memory lane of this thread
        float *Lf = reinterpret_cast<float *>(sm + OFF_LF);
        float *Tf = reinterpret_cast<float *>(sm + OFF_TF);
        float *Mt = reinterpret_cast<float *>(sm + OFF_MT);
        // rows 0-63 carry g, rows 64-127 carry beta; the next chunk's values
        // are loaded one iteration ahead to hide the global-memory latency
        auto load_gate = [&](int c) -> float {
            const int r = prow & 63;
            const int rows_c = min(kChunk, len - c * kChunk);
            if (r >= rows_c) return 0.f;
            const int64_t t = (tok0 + (int64_t)c * kChunk + r) * H + h;
            return prow < 64 ? p.g[t] : p.beta[t];
        };
        float gnext = (nch > 0) ? load_gate(0) : 0.f;
        for (int c = 0; c < nch; ++c) {
            const float gcur = gnext;
            if (c + 1 < nch) gnext = load_gate(c + 1);
            const int s = c % 3;
            const int rows = min(kChunk, len - c * kChunk);
            float *sc = sc_all + s * 5 * 64;
            const float *bsum = sc, *bet = sc + 64, *rk = sc + 128, *rq = sc + 192;
            uint8_t *st = sm + OFF_QK + s * kQKStage;
            if (prow == 0) GDN_TR(0, c, 0);

            // (1) gates: chunk-local cumulative log-gate (base 2), beta
            float x = 0.f;
            if (prow < 64) {
                x = gcur * kLog2e;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                if (lane == 31) Mt[prow >> 5] = x;
            } else {
                sc[prow] = gcur;   // beta (0 on padded rows)
            }
            group_sync(1, 128);
            if (prow < 64) sc[prow] = x + ((prow >= 32) ? Mt[0] : 0.f);
            group_sync(1, 128);
            if (prow == 0) mbar_arrive(bar(B_GATE + s));
            if (prow == 0) GDN_TR(0, c, 1);

            // (2) inverse norms from the landed tiles
            bool ok = wait_bar(bar(B_QKF + s), (c / 3) & 1, abort_flag, p.err);
            if (prow == 0) GDN_TR(0, c, 2);
            {
                const int r = prow & 63;
                const bool isq = prow >= 64;
                const uint8_t *row = st + (isq ? 8192 : 0) + r * 128;
                const float ss = row_sumsq(row, r) + row_sumsq(row + 16384, r);
                float inv = p.l2 ? 1.f / sqrtf(ss + kL2Eps) : 1.f;
                if (isq) inv *= p.scale;
                sc[(isq ? 192 : 128) + r] = (r < rows) ? inv : 0.f;
            }
            if (group_sync_or(2 + 0, 128, !ok || *abort_flag)) break;
            if (prow == 0) GDN_TR(0, c, 3);

            // (3) Gram masking: L (rows 0-63) and Aqk (rows 64-127)
            ok = wait_bar(bar(B_P1), c & 1, abort_flag, p.err);
            if (prow == 0) GDN_TR(0, c, 4);
            fence_after_sync();
            {
                float G[64];
                uint32_t u[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    tmem_ld16(lane_base + TM_P1 + q * 16, u);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) G[q * 16 + e] = __uint_as_float(u[e]);
                }
                if (prow < 64) {
                    const int r = prow;
                    const float br = bsum[r], f = bet[r] * rk[r];
                    float *Lr = Lf + r * LDA;
#pragma unroll
                    for (int i = 0; i < 64; ++i) Lr[i] = (i < r) ? f * exp2f(br - bsum[i]) * rk[i] * G[i] : 0.f;
                } else {
                    const int r = prow - 64;
                    if (c >= 2) ok = ok && wait_bar(bar(B_AQKF + (c & 1)), ((c - 2) >> 1) & 1, abort_flag, p.err);
                    uint8_t *aq = sm + OFF_AQK + (c & 1) * 8192;
                    const float br = bsum[r], f = rq[r];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int i0 = ch * 8 + 2 * e;
                            const float a0 = (i0 <= r) ? f * exp2f(br - bsum[i0]) * rk[i0] * G[i0] : 0.f;
                            const float a1 = (i0 + 1 <= r) ? f * exp2f(br - bsum[i0 + 1]) * rk[i0 + 1] * G[i0 + 1] : 0.f;
                            w[e] = pack_bf16(a0, a1);
                        }
                        *reinterpret_cast<uint4 *>(aq + sw128_offset(r, ch * 8)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            fence_before_sync();
            fence_proxy_async();
            if (group_sync_or(2, 128, !ok || *abort_flag)) break;

            // (4) T = (I + L)^{-1};  T' = T diag(beta),  T'' = T diag(beta e^b rk)
            if (prow == 0) GDN_TR(0, c, 5);
            solve_unit_lower(Lf, Tf, Mt, prow);
            if (prow == 0) GDN_TR(0, c, 6);
            if (c >= 1) ok = wait_bar(bar(B_TWFREE), (c - 1) & 1, abort_flag, p.err);
            if (prow == 0) GDN_TR(0, c, 7);
            {
                const int r = prow >> 1, i0 = (prow & 1) * 32;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t w1[4], w2[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = i0 + ch * 8 + 2 * e;
                        const float t0 = Tf[r * LDL + i], t1 = Tf[r * LDL + i + 1];
                        const float p0 = t0 * bet[i], p1 = t1 * bet[i + 1];
                        w1[e] = pack_bf16(p0, p1);
                        w2[e] = pack_bf16(p0 * exp2f(bsum[i]) * rk[i], p1 * exp2f(bsum[i + 1]) * rk[i + 1]);
                    }
                    const uint32_t off = sw128_offset(r, i0 + ch * 8);
                    *reinterpret_cast<uint4 *>(sm + OFF_TP + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
                    *reinterpret_cast<uint4 *>(sm + OFF_TPP + off) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
                }
            }
            fence_proxy_async();
            if (group_sync_or(2, 128, !ok || *abort_flag)) break;
            if (prow == 0) mbar_arrive(bar(B_TRDY));
            if (prow == 0) GDN_TR(0, c, 8);

            // (5) W~^T to shared memory; K -> K->, Q -> Q<- in place
            ok = wait_bar(bar(B_P2), c & 1, abort_flag, p.err);
            if (prow == 0) GDN_TR(0, c, 9);
            fence_after_sync();
            {
                uint32_t u[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    tmem_ld16(lane_base + TM_P2 + q * 16, u);
                    tmem_wait_ld();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack_bf16(__uint_as_float(u[hh * 8 + 2 * e]), __uint_as_float(u[hh * 8 + 2 * e + 1]));
                        *reinterpret_cast<uint4 *>(sm + OFF_WT + sw128_offset(prow, q * 16 + hh * 8)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                const int r = prow >> 1, kb = prow & 1;
                const float bC = bsum[63];
                const float fk = (r < rows) ? exp2f(bC - bsum[r]) * rk[r] : 0.f;
                const float fq = (r < rows) ? exp2f(bsum[r]) * rq[r] : 0.f;
                row_scale(st + kb * 16384 + r * 128, r, fk);
                row_scale(st + 8192 + kb * 16384 + r * 128, r, fq);
            }
            fence_before_sync();
            fence_proxy_async();
            if (group_sync_or(2, 128, !ok || *abort_flag)) break;
            if (prow == 0) mbar_arrive(bar(B_PREP));
            if (prow == 0) GDN_TR(0, c, 10);
        }
    } else {
        // ------------------------------------------------------------ chain epilogue
        const int j = 32 * (warp & 3) + lane;   // row of S within the slice
        const size_t srow = (((size_t)n * H + h) * (size_t)dv + (size_t)(j0 + j)) * 128;
        if (nch == 0) {
            if (p.final_state)
                for (int d = 0; d < 128; d += 4) {
                    float4 v4 = p.init_state ? *reinterpret_cast<const float4 *>(p.init_state + srow + d)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                    *reinterpret_cast<float4 *>(p.final_state + srow + d) = v4;
                }
        } else {
            bool ok = wait_bar(bar(B_GATE), 0, abort_flag, p.err);
            {
                const float e0 = exp2f(sc_all[63]);
#pragma unroll
                for (int q2 = 0; q2 < 4; ++q2) {   // 32 state entries per pass
                    float v[32];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        float4 v4 = p.init_state ? *reinterpret_cast<const float4 *>(p.init_state + srow + q2 * 32 + e)
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                        v[e] = v4.x; v[e + 1] = v4.y; v[e + 2] = v4.z; v[e + 3] = v4.w;
                    }
                    uint32_t pk[16], sc0[16], sc1[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        pk[e] = pack_bf16(v[2 * e], v[2 * e + 1]);
                        sc0[e] = __float_as_uint(e0 * v[e]);
                        sc1[e] = __float_as_uint(e0 * v[16 + e]);
                    }
                    tmem_st16(lane_base + TM_SBF + q2 * 16, pk);
                    tmem_st16(lane_base + TM_S + q2 * 32, sc0);
                    tmem_st16(lane_base + TM_S + q2 * 32 + 16, sc1);
                }
                tmem_wait_st();
            }
            fence_before_sync();
            if (!group_sync_or(3, 128, !ok || *abort_flag) && j == 0) mbar_arrive(bar(B_S));
            for (int c = 0; c < nch; ++c) {
                const int rows = min(kChunk, len - c * kChunk);
                const int64_t z0 = tok0 + (int64_t)c * kChunk;
                // V_new^T -> bf16 A operand
                ok = wait_bar(bar(B_D1), c & 1, abort_flag, p.err);
                if (j == 0) GDN_TR(2, c, 0);
                fence_after_sync();
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    uint32_t a[16], b[16], pk[16];
                    tmem_ld16(lane_base + TM_D1 + q2 * 32, a);
                    tmem_ld16(lane_base + TM_D1 + q2 * 32 + 16, b);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        pk[e] = pack_bf16(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
                        pk[8 + e] = pack_bf16(__uint_as_float(b[2 * e]), __uint_as_float(b[2 * e + 1]));
                    }
                    tmem_st16(lane_base + TM_X1 + q2 * 16, pk);
                }
                tmem_wait_st();
                fence_before_sync();
                if (group_sync_or(3, 128, !ok || *abort_flag)) break;
                if (j == 0) mbar_arrive(bar(B_X));
                if (j == 0) GDN_TR(2, c, 1);
                // next state first (it gates the next chunk), then the outputs
                ok = wait_bar(bar(B_D2), c & 1, abort_flag, p.err);
                if (j == 0) GDN_TR(2, c, 2);
                fence_after_sync();
                if (c + 1 < nch) {
                    const int s1 = (c + 1) % 3;
                    ok = ok && wait_bar(bar(B_GATE + s1), ((c + 1) / 3) & 1, abort_flag, p.err);
                    if (j == 0) GDN_TR(2, c, 3);
                    const float e1 = exp2f(sc_all[s1 * 5 * 64 + 63]);
#pragma unroll
                    for (int q2 = 0; q2 < 4; ++q2) {
                        uint32_t a[16], b[16], pk[16];
                        tmem_ld16(lane_base + TM_S + q2 * 32, a);
                        tmem_ld16(lane_base + TM_S + q2 * 32 + 16, b);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            pk[e] = pack_bf16(__uint_as_float(a[2 * e]), __uint_as_float(a[2 * e + 1]));
                            pk[8 + e] = pack_bf16(__uint_as_float(b[2 * e]), __uint_as_float(b[2 * e + 1]));
                        }
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            a[e] = __float_as_uint(e1 * __uint_as_float(a[e]));
                            b[e] = __float_as_uint(e1 * __uint_as_float(b[e]));
                        }
                        tmem_st16(lane_base + TM_SBF + q2 * 16, pk);
                        tmem_st16(lane_base + TM_S + q2 * 32, a);
                        tmem_st16(lane_base + TM_S + q2 * 32 + 16, b);
                    }
                    tmem_wait_st();
                    fence_before_sync();
                    if (group_sync_or(3, 128, !ok || *abort_flag)) break;
                    if (j == 0) mbar_arrive(bar(B_S));
                    if (j == 0) GDN_TR(2, c, 4);
                } else if (p.final_state && ok) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        uint32_t u[16];
                        tmem_ld16(lane_base + TM_S + q * 16, u);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; e += 4)
                            *reinterpret_cast<float4 *>(p.final_state + srow + q * 16 + e) =
                                make_float4(__uint_as_float(u[e]), __uint_as_float(u[e + 1]),
                                            __uint_as_float(u[e + 2]), __uint_as_float(u[e + 3]));
                    }
                }
                // O^T (row j = output column j0 + j) through a [64 r][128 j] bf16 staging
                // tile in this chunk's V stage (a1 has long completed), then 16-B stores
                {
                    uint8_t *stg = sm + OFF_V + (uint32_t)(c & 1) * kVStage;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t u[16];
                        tmem_ld16(lane_base + TM_D2 + q * 16, u);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            *reinterpret_cast<__nv_bfloat16 *>(stg + ((q * 16 + e) * 128 + j) * 2) =
                                __float2bfloat16_rn(__uint_as_float(u[e]));
                    }
                    fence_before_sync();
                    if (group_sync_or(3, 128, !ok || *abort_flag)) break;
                    __nv_bfloat16 *obase = p.out + (size_t)z0 * H * dv + (size_t)h * dv + j0;
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int idx = it * 128 + j, r = idx >> 4, ch = idx & 15;
                        if (r < rows)
                            *reinterpret_cast<uint4 *>(obase + (size_t)r * H * dv + ch * 8) =
                                *reinterpret_cast<const uint4 *>(stg + r * 256 + ch * 16);
                    }
                    if (group_sync_or(3, 128, !ok || *abort_flag)) break;
                    if (j == 0) mbar_arrive(bar(B_VE + (c & 1)));   // the V stage may be refilled
                    if (j == 0) GDN_TR(2, c, 5);
                }
            }
        }
    }

    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        tmem_dealloc(tb, 512);
    }
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

#ifdef GDN_KERNEL_TRACE
long long *g_trace_buffer = nullptr;
#endif

}  // namespace

#ifdef GDN_KERNEL_TRACE
extern "C" void gdn_debug_set_trace(long long *buf) { g_trace_buffer = buf; }
#endif

bool chunk_tc_supported(int dt, int dk, int dv, int64_t tokens)
{
    return dt == 1 && dk == 128 && dv % 128 == 0 && tokens > 0 && tokens < ((int64_t)1 << 31);
}

cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t st)
{
    const int64_t rows = (int64_t)a.gm.B * a.gm.T;
    CUtensorMap tq, tk, tv;
    if (!make_tmap(&tq, a.q, a.gm.dk, a.gm.H, rows) || !make_tmap(&tk, a.k, a.gm.dk, a.gm.H, rows) ||
        !make_tmap(&tv, a.v, a.gm.dv, a.gm.H, rows))
        return cudaErrorInvalidValue;
    TcParams p;
    p.g = a.g;
    p.beta = a.beta;
    p.init_state = a.init_state;
    p.out = reinterpret_cast<__nv_bfloat16 *>(a.out);
    p.final_state = a.final_state;
    p.err = reinterpret_cast<unsigned *>(a.workspace);
    p.gm = a.gm;
    p.scale = a.scale;
    p.l2 = a.l2;
#ifdef GDN_KERNEL_TRACE
    p.trace = g_trace_buffer;
#endif
    cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTc);
    if (e != cudaSuccess) return e;
    dim3 grid(a.gm.N, a.gm.H, a.gm.dv / 128);
    chunk_tc_kernel<<<grid, kThreadsTc, kSmemTc, st>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace gdn
