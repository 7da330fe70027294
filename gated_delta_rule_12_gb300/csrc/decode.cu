// decode.cu -- single-token decode step of the gated delta rule.
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

template <typename T, int DK, int R>
__global__ void __launch_bounds__(256)
decode_kernel(float *__restrict__ state, const T *__restrict__ q, const T *__restrict__ k,
              const T *__restrict__ v, const float *__restrict__ g, const float *__restrict__ beta,
              T *__restrict__ out, int NH, int dv, float scale, int l2)
{
    constexpr int VEC = DK / 32;   // entries of a row per lane
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int groups_per_head = dv / R;
    const int64_t total = (int64_t)NH * groups_per_head;

    for (int64_t grp = warp0; grp < total; grp += nwarps) {
        const int64_t nh = grp / groups_per_head;
        const int j0 = (int)(grp % groups_per_head) * R;
        float *S = state + ((size_t)nh * dv + j0) * DK + lane * VEC;

        float s[R][VEC];
#pragma unroll
        for (int r = 0; r < R; ++r) load_row<VEC>(S + (size_t)r * DK, s[r]);

        // normalised key and scaled, normalised query for this head
        float kv[VEC], qv[VEC];
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
            kv[i] = to_f32(k[nh * DK + lane * VEC + i]);
            qv[i] = to_f32(q[nh * DK + lane * VEC + i]);
            sk += kv[i] * kv[i];
            sq += qv[i] * qv[i];
        }
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
        const float alpha = expf(g[nh]);
        const float b = beta[nh];

        float ov = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float pk = 0.f, pq = 0.f;
#pragma unroll
            for (int i = 0; i < VEC; ++i) {
                pk += s[r][i] * kv[i];
                pq += s[r][i] * qv[i];
            }
            pk = warp_sum(pk);
            pq = warp_sum(pq);
            const float vj = to_f32(v[nh * dv + j0 + r]);
            const float e = b * (vj - alpha * pk);
#pragma unroll
            for (int i = 0; i < VEC; ++i) s[r][i] = alpha * s[r][i] + e * kv[i];
            const float o = alpha * pq + e * kq;
            if (lane == r) ov = o;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) store_row<VEC>(S + (size_t)r * DK, s[r]);
        if (lane < R) out[nh * dv + j0 + lane] = from_f32<T>(ov);
    }
}

template <typename T, int DK>
static cudaError_t launch_decode_typed(const DecodeArgs &a, cudaStream_t st)
{
    constexpr int R = 8;
    const int NH = a.N * a.H;
    const int64_t groups = (int64_t)NH * (a.dv / R);
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int per_sm = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<T, DK, R>, 256, 0);
    if (per_sm < 1) per_sm = 1;
    int64_t blocks = (groups + 7) / 8;
    const int64_t cap = (int64_t)sms * per_sm;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    decode_kernel<T, DK, R><<<(unsigned)blocks, 256, 0, st>>>(
        a.state, (const T *)a.q, (const T *)a.k, (const T *)a.v, a.g, a.beta, (T *)a.out, NH, a.dv,
        a.scale, a.l2);
    return cudaGetLastError();
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
