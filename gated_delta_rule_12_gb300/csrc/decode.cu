// decode.cu -- decode steps of the gated delta rule (one or a few tokens per call).
//
// "Gated DeltaNet：先忘一点，再按误差更新记忆", "为什么再加一个遗忘门？":
//     Sbar = alpha S,   S <- Sbar + beta (v - Sbar k) k^T,   o = S q.
// Row j of S evolves independently given k, q, v_j, alpha, beta:
//     p_j  = alpha (S k)_j
//     e_j  = beta (v_j - p_j)
//     S'_j = alpha S_j + e_j k^T
//     o_j  = S'_j q = alpha (S q)_j + e_j (k . q)
// so one pass reads each row once, reduces (S k)_j and (S q)_j together,
// and writes the row once: the state is read and written exactly once per
// step, which is the HBM floor of this step.
//
// Work split: a "group" is R consecutive rows of one (sequence, head) state
// (R * dk * 4 bytes).  Warps stride over all groups of the call, so the load
// is balanced whatever N*H is.  Each lane holds dk/32 consecutive entries of
// a row (16-byte vector loads when dk >= 128).
//
// Several tokens per call ("Decode 递归": the ordered composition of steps):
// the group's rows stay in registers while the T tokens of the call are
// applied in order, so the state is still read once and written once per call
// however many tokens it carries.  Token t of sequence n, head h is at
// ((n T + t) H + h) of the token-major inputs; T = 1 is the single step.
#include "common.cuh"
#include "kernels.h"

namespace gdn {

template <int V>
struct FVec;
template <> struct FVec<2> { using type = float2; };
template <> struct FVec<4> { using type = float4; };

template <int VEC>
__device__ __forceinline__ void load_row(const float *p, float (&x)[VEC])
{
    if constexpr (VEC == 2) {
        float2 t = __ldcs(reinterpret_cast<const float2 *>(p));
        x[0] = t.x; x[1] = t.y;
    } else {
#pragma unroll
        for (int i = 0; i < VEC; i += 4) {
            float4 t = __ldcs(reinterpret_cast<const float4 *>(p + i));
            x[i] = t.x; x[i + 1] = t.y; x[i + 2] = t.z; x[i + 3] = t.w;
        }
    }
}

template <int VEC>
__device__ __forceinline__ void store_row(float *p, const float (&x)[VEC])
{
    if constexpr (VEC == 2) {
        __stcs(reinterpret_cast<float2 *>(p), make_float2(x[0], x[1]));
    } else {
#pragma unroll
        for (int i = 0; i < VEC; i += 4)
            __stcs(reinterpret_cast<float4 *>(p + i), make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]));
    }
}

// Sums of eight per-lane partials x[0..7] (one per row) over the warp, reduced
// together: three exchange stages halve the rows a lane carries (xor 16, 8, 4),
// two more finish the sum (xor 2, 1).  Afterwards lane l holds the total of
// row l >> 2 (9 shuffles for 8 rows instead of 5 per row).
__device__ __forceinline__ float warp_sum8_transposed(const float (&x)[8], int lane)
{
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float w4[4], w2[2];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w4[i] = (b4 ? x[i + 4] : x[i]) + __shfl_xor_sync(0xffffffffu, b4 ? x[i] : x[i + 4], 16);
#pragma unroll
    for (int i = 0; i < 2; ++i)
        w2[i] = (b3 ? w4[i + 2] : w4[i]) + __shfl_xor_sync(0xffffffffu, b3 ? w4[i] : w4[i + 2], 8);
    float w = (b2 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? w2[0] : w2[1], 4);
    w += __shfl_xor_sync(0xffffffffu, w, 2);
    w += __shfl_xor_sync(0xffffffffu, w, 1);
    return w;
}

// MULTI = false compiles the single-token step as straight-line code.
template <typename T, int DK, bool MULTI>
__global__ void __launch_bounds__(256)
decode_kernel(float *__restrict__ state, const T *__restrict__ q, const T *__restrict__ k,
              const T *__restrict__ v, const float *__restrict__ g, const float *__restrict__ beta,
              T *__restrict__ out, int NH, int H, int ntok, int dv, float scale, int l2)
{
    constexpr int R = 8;           // rows of S per warp group
    constexpr int VEC = DK / 32;   // entries of a row per lane
    const int lane = threadIdx.x & 31;
    const int myrow = lane >> 2;   // the row whose reductions this lane ends up holding
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int groups_per_head = dv / R;
    const int64_t total = (int64_t)NH * groups_per_head;
    const int nt = MULTI ? ntok : 1;

    for (int64_t grp = warp0; grp < total; grp += nwarps) {
        const int64_t nh = grp / groups_per_head;
        const int j0 = (int)(grp % groups_per_head) * R;
        float *S = state + ((size_t)nh * dv + j0) * DK + lane * VEC;

        float s[R][VEC];
#pragma unroll
        for (int r = 0; r < R; ++r) load_row<VEC>(S + (size_t)r * DK, s[r]);

        const int64_t n = MULTI ? nh / H : nh, h = MULTI ? nh % H : 0;
#pragma unroll 1
        for (int t = 0; t < nt; ++t) {
            const int64_t tok = MULTI ? (n * ntok + t) * H + h : nh;   // token-head index
            // normalised key and scaled, normalised query of this token
            float kv[VEC], qv[VEC];
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                kv[i] = to_f32(k[tok * DK + lane * VEC + i]);
                qv[i] = to_f32(q[tok * DK + lane * VEC + i]);
                sk += kv[i] * kv[i];
                sq += qv[i] * qv[i];
            }
            const float vj = to_f32(v[tok * dv + j0 + myrow]);
            const float alpha = expf(g[tok]);
            const float b = beta[tok];
            float rk = 1.f, rq = scale;
            if (l2) {
                sk = warp_sum(sk);
                sq = warp_sum(sq);
                rk = 1.f / sqrtf(sk + kL2Eps);
                rq = scale / sqrtf(sq + kL2Eps);
            }
            float kq = 0.f;
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                kv[i] *= rk;
                qv[i] *= rq;
                kq += kv[i] * qv[i];
            }
            kq = warp_sum(kq);

            float pk[R], pq[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                pk[r] = 0.f;
                pq[r] = 0.f;
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    pk[r] += s[r][i] * kv[i];
                    pq[r] += s[r][i] * qv[i];
                }
            }
            const float pkm = warp_sum8_transposed(pk, lane);   // (S k) of row myrow
            const float pqm = warp_sum8_transposed(pq, lane);   // (S q) of row myrow
            const float em = b * (vj - alpha * pkm);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float e = __shfl_sync(0xffffffffu, em, 4 * r);
#pragma unroll
                for (int i = 0; i < VEC; ++i) s[r][i] = alpha * s[r][i] + e * kv[i];
            }
            if ((lane & 3) == 0) out[tok * dv + j0 + myrow] = from_f32<T>(alpha * pqm + em * kq);
        }
#pragma unroll
        for (int r = 0; r < R; ++r) store_row<VEC>(S + (size_t)r * DK, s[r]);
    }
}

// Several tokens per call with the per-token work that does not depend on the state -- loading
// and normalising k and q, k . q, alpha and beta -- done once per token for a run of GPW row
// groups of one (sequence, head), instead of once per group.  Each group then runs exactly the
// arithmetic of decode_kernel (same operations in the same order), so the results are bit for
// bit those of NT single steps.  NT <= 4 tokens, DK <= 128 (the token vectors stay in registers).
template <typename T, int DK, int NT, int GPW>
__global__ void __launch_bounds__(256, 3)
decode_multi_kernel(float *__restrict__ state, const T *__restrict__ q, const T *__restrict__ k,
                    const T *__restrict__ v, const float *__restrict__ g, const float *__restrict__ beta,
                    T *__restrict__ out, int NH, int H, int dv, float scale, int l2)
{
    constexpr int R = 8;           // rows of S per group
    constexpr int VEC = DK / 32;   // entries of a row per lane
    // the run's normalised keys and queries, each lane's own VEC entries (shared memory keeps them
    // out of the registers that hold the state rows)
    __shared__ __align__(16) float tkq[8][NT][2][DK];
    __shared__ float tsc[8][NT][4];   // per token: k . q, alpha, beta
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int myrow = lane >> 2;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int groups_per_head = dv / R;
    const int runs_per_head = (groups_per_head + GPW - 1) / GPW;
    const int64_t total = (int64_t)NH * runs_per_head;

    for (int64_t run = warp0; run < total; run += nwarps) {
        const int64_t nh = run / runs_per_head;
        const int g0 = (int)(run % runs_per_head) * GPW;
        const int64_t n = nh / H, h = nh % H;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int64_t tok = (n * NT + t) * H + h;
            float kv[VEC], qv[VEC];
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                kv[i] = to_f32(k[tok * DK + lane * VEC + i]);
                qv[i] = to_f32(q[tok * DK + lane * VEC + i]);
                sk += kv[i] * kv[i];
                sq += qv[i] * qv[i];
            }
            const float alpha_t = expf(g[tok]);
            const float beta_t = beta[tok];
            float rk = 1.f, rq = scale;
            if (l2) {
                sk = warp_sum(sk);
                sq = warp_sum(sq);
                rk = 1.f / sqrtf(sk + kL2Eps);
                rq = scale / sqrtf(sq + kL2Eps);
            }
            float kqt = 0.f;
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                kv[i] *= rk;
                qv[i] *= rq;
                kqt += kv[i] * qv[i];
                tkq[wib][t][0][lane * VEC + i] = kv[i];
                tkq[wib][t][1][lane * VEC + i] = qv[i];
            }
            kqt = warp_sum(kqt);
            if (lane == 0) {
                tsc[wib][t][0] = kqt;
                tsc[wib][t][1] = alpha_t;
                tsc[wib][t][2] = beta_t;
            }
        }
        __syncwarp();
#pragma unroll 1
        for (int gi = g0; gi < g0 + GPW && gi < groups_per_head; ++gi) {
            const int j0 = gi * R;
            float *S = state + ((size_t)nh * dv + j0) * DK + lane * VEC;
            float s[R][VEC];
#pragma unroll
            for (int r = 0; r < R; ++r) load_row<VEC>(S + (size_t)r * DK, s[r]);
#pragma unroll 1
            for (int t = 0; t < NT; ++t) {
                const int64_t tok = (n * NT + t) * H + h;
                const float vj = to_f32(v[tok * dv + j0 + myrow]);
                const float kqt = tsc[wib][t][0], alpha_t = tsc[wib][t][1], beta_t = tsc[wib][t][2];
                float kv[VEC], qv[VEC];
#pragma unroll
                for (int i = 0; i < VEC; ++i) {
                    kv[i] = tkq[wib][t][0][lane * VEC + i];
                    qv[i] = tkq[wib][t][1][lane * VEC + i];
                }
                float pk[R], pq[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    pk[r] = 0.f;
                    pq[r] = 0.f;
#pragma unroll
                    for (int i = 0; i < VEC; ++i) {
                        pk[r] += s[r][i] * kv[i];
                        pq[r] += s[r][i] * qv[i];
                    }
                }
                const float pkm = warp_sum8_transposed(pk, lane);
                const float pqm = warp_sum8_transposed(pq, lane);
                const float em = beta_t * (vj - alpha_t * pkm);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const float e = __shfl_sync(0xffffffffu, em, 4 * r);
#pragma unroll
                    for (int i = 0; i < VEC; ++i) s[r][i] = alpha_t * s[r][i] + e * kv[i];
                }
                if ((lane & 3) == 0) out[tok * dv + j0 + myrow] = from_f32<T>(alpha_t * pqm + em * kqt);
            }
#pragma unroll
            for (int r = 0; r < R; ++r) store_row<VEC>(S + (size_t)r * DK, s[r]);
        }
        __syncwarp();   // the buffer is rewritten by the next run's tokens
    }
}

template <typename T, int DK, int NT>
static cudaError_t launch_decode_multi_kernel(const DecodeArgs &a, cudaStream_t st)
{
    constexpr int GPW = 4;   // row groups per warp run (32 rows)
    const int NH = a.N * a.H;
    const int64_t runs = (int64_t)NH * ((a.dv / 8 + GPW - 1) / GPW);
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_multi_kernel<T, DK, NT, GPW>, 256, 0);
    if (per_sm < 1) per_sm = 1;
    int64_t blocks = (runs + 7) / 8;
    const int64_t cap = (int64_t)sms * per_sm;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    decode_multi_kernel<T, DK, NT, GPW><<<(unsigned)blocks, 256, 0, st>>>(
        a.state, (const T *)a.q, (const T *)a.k, (const T *)a.v, a.g, a.beta, (T *)a.out, NH, a.H, a.dv,
        a.scale, a.l2);
    return cudaGetLastError();
}

template <typename T, int DK, bool MULTI>
static cudaError_t launch_decode_kernel(const DecodeArgs &a, cudaStream_t st)
{
    const int NH = a.N * a.H;
    const int64_t groups = (int64_t)NH * (a.dv / 8);
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<T, DK, MULTI>, 256, 0);
    if (per_sm < 1) per_sm = 1;
    int64_t blocks = (groups + 7) / 8;
    const int64_t cap = (int64_t)sms * per_sm;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    decode_kernel<T, DK, MULTI><<<(unsigned)blocks, 256, 0, st>>>(
        a.state, (const T *)a.q, (const T *)a.k, (const T *)a.v, a.g, a.beta, (T *)a.out, NH, a.H, a.ntok,
        a.dv, a.scale, a.l2);
    return cudaGetLastError();
}

template <typename T, int DK>
static cudaError_t launch_decode_typed(const DecodeArgs &a, cudaStream_t st)
{
    if constexpr (DK <= 128) {
        switch (a.ntok) {
            case 2: return launch_decode_multi_kernel<T, DK, 2>(a, st);
            case 3: return launch_decode_multi_kernel<T, DK, 3>(a, st);
            case 4: return launch_decode_multi_kernel<T, DK, 4>(a, st);
            default: break;
        }
    }
    return a.ntok > 1 ? launch_decode_kernel<T, DK, true>(a, st) : launch_decode_kernel<T, DK, false>(a, st);
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st)
{
    if (a.dt == 0) {
        switch (a.dk) {
            case 64: return launch_decode_typed<float, 64>(a, st);
            case 128: return launch_decode_typed<float, 128>(a, st);
            default: return launch_decode_typed<float, 256>(a, st);
        }
    }
    switch (a.dk) {
        case 64: return launch_decode_typed<__nv_bfloat16, 64>(a, st);
        case 128: return launch_decode_typed<__nv_bfloat16, 128>(a, st);
        default: return launch_decode_typed<__nv_bfloat16, 256>(a, st);
    }
}

}  // namespace gdn
