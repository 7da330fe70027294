// chunk_simt.cu -- chunked forward pass on the CUDA cores (fp32 arithmetic).
//
// Three kernels, one per step of the chunkwise algorithm of "Gated Delta
// Networks: Improving Mamba2 with Delta Rule", §3.3:
//   prologue_kernel   per chunk: b_r = sum_{i<=r} g_i (chunk-local log of
//                     gamma^r), inverse L2 norms of q and k (scale folded into q)
//   ut_simt_kernel    per chunk: the UT transform; solves
//                     [I + strictLower(diag(beta)(Gamma o K K^T))] X = [diag(beta e^b) K | diag(beta) V]
//                     by forward substitution, X = [W<- | U~]
//   recur_simt_kernel per (sequence, head, 32-row slice of S): the sequential
//                     chunk recurrence with the decay mask Gamma in the
//                     output term ("【论文解读】Gated Delta Network", §二(一)2(4)).
// Every ratio gamma_r / gamma_i is formed as exp(b_r - b_i) with i <= r, so
// no factor above 1 is ever built, whatever the decay.
// This path serves fp32 inputs (where tensor-core rounding would exceed the
// fp32 tolerance) and head sizes the tensor-core path does not cover.
#include "common.cuh"
#include "kernels.h"

namespace gdn {

// ---------------------------------------------------------------------------
// K1: prologue
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256)
prologue_kernel(const T *__restrict__ q, const T *__restrict__ k, const float *__restrict__ g,
                Geometry gm, float scale, int l2, float *__restrict__ bcum,
                float *__restrict__ rq, float *__restrict__ rk, unsigned *__restrict__ err_word)
{
    const int64_t slot = blockIdx.x;
    // the first kernel of a call clears the device error word of the workspace
    if (slot == 0 && blockIdx.y == 0 && threadIdx.x == 0) *err_word = kDevErrNone;
    const int h = blockIdx.y;
    int n, c, rows;
    int64_t tok0;
    if (!slot_to_chunk(gm, slot, n, c, tok0, rows)) return;
    const size_t base = ((size_t)slot * gm.H + h) * kChunk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (int r = warp; r < kChunk; r += 8) {
        float iq = 0.f, ik = 0.f;
        if (r < rows) {
            if (l2) {
                const int64_t th = (tok0 + r) * gm.H + h;
                const T *qr = q + th * gm.dk;
                const T *kr = k + th * gm.dk;
                float sq = 0.f, sk = 0.f;
                for (int d = lane; d < gm.dk; d += 32) {
                    float a = to_f32(qr[d]), b = to_f32(kr[d]);
                    sq += a * a;
                    sk += b * b;
                }
                sq = warp_sum(sq);
                sk = warp_sum(sk);
                iq = scale / sqrtf(sq + kL2Eps);
                ik = 1.f / sqrtf(sk + kL2Eps);
            } else {
                iq = scale;
                ik = 1.f;
            }
        }
        if (lane == 0) {
            rq[base + r] = iq;
            rk[base + r] = ik;
        }
    }

    // inclusive scan of g over the chunk (padded rows add 0)
    __shared__ float carry;
    if (threadIdx.x < kChunk) {
        const int r = threadIdx.x;
        float x = (r < rows) ? g[(tok0 + r) * gm.H + h] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            float y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (r == 31) carry = x;
        __syncwarp();
        // make the first warp's total visible to the second
        asm volatile("bar.sync 1, 64;");
        if (r >= 32) x += carry;
        bcum[base + r] = x;
    }
}

// ---------------------------------------------------------------------------
// K2: UT transform on the CUDA cores
// ---------------------------------------------------------------------------
template <typename T, int DK>
__global__ void __launch_bounds__(256)
ut_simt_kernel(const T *__restrict__ k, const T *__restrict__ v, const float *__restrict__ beta,
               Geometry gm, const float *__restrict__ bcum, const float *__restrict__ rk,
               float *__restrict__ Wout, float *__restrict__ Uout)
{
    extern __shared__ float smem[];
    constexpr int P = DK + 4;               // row pitch of K: 16-B rows for the tiled Gram product
    float *Ks = smem;                       // [64][DK+4]
    float *A = Ks + kChunk * P;             // [64][65]  strictly lower system matrix
    float *bs = A + kChunk * 65;            // [64]
    float *bt = bs + kChunk;                // [64]   beta (0 on padded rows)

    const int64_t slot = blockIdx.x;
    const int h = blockIdx.y;
    int n, c, rows;
    int64_t tok0;
    if (!slot_to_chunk(gm, slot, n, c, tok0, rows)) return;
    const int dv = gm.dv;
    const size_t base = ((size_t)slot * gm.H + h) * kChunk;
    const int tid = threadIdx.x;

    if (tid < kChunk) {
        bs[tid] = bcum[base + tid];
        bt[tid] = (tid < rows) ? beta[(tok0 + tid) * gm.H + h] : 0.f;
    }
    for (int e = tid; e < kChunk * DK; e += blockDim.x) {
        const int r = e / DK, d = e % DK;
        float x = 0.f;
        if (r < rows) x = to_f32(k[((tok0 + r) * gm.H + h) * DK + d]) * rk[base + r];
        Ks[r * P + d] = x;
    }
    __syncthreads();
    {   // K K^T, a 4 x 4 tile of rows r0.., columns i0.. per thread, 16-B loads along d
        const int r0 = 4 * (tid >> 4), i0 = 4 * (tid & 15);
        float acc[4][4] = {};
        if (i0 < r0 + 3) {
#pragma unroll 4
            for (int d = 0; d < DK; d += 4) {
                float4 kr[4], ki[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    kr[u] = *reinterpret_cast<const float4 *>(Ks + (r0 + u) * P + d);
                    ki[u] = *reinterpret_cast<const float4 *>(Ks + (i0 + u) * P + d);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        acc[u][v] += kr[u].x * ki[v].x + kr[u].y * ki[v].y + kr[u].z * ki[v].z + kr[u].w * ki[v].w;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const int r = r0 + u, i = i0 + v;
                A[r * 65 + i] = (i < r) ? bt[r] * expf(bs[r] - bs[i]) * acc[u][v] : 0.f;
            }
    }
    __syncthreads();

    float *Wd = Wout + base * DK;
    float *Ud = Uout + base * dv;
    for (int col = tid; col < DK + dv; col += blockDim.x) {
        float x[kChunk];
        if (col < DK) {
#pragma unroll
            for (int r = 0; r < kChunk; ++r) x[r] = bt[r] * expf(bs[r]) * Ks[r * P + col];
        } else {
            const int j = col - DK;
#pragma unroll
            for (int r = 0; r < kChunk; ++r)
                x[r] = (r < rows) ? bt[r] * to_f32(v[((tok0 + r) * gm.H + h) * dv + j]) : 0.f;
        }
        // forward substitution, column-oriented: once x_i is final it is taken out of every later
        // row, so the updates of one step are independent (a chain of 63 steps, not of 2016 FMAs)
#pragma unroll
        for (int i = 0; i < kChunk - 1; ++i) {
            const float xi = x[i];
#pragma unroll
            for (int r = i + 1; r < kChunk; ++r) x[r] -= A[r * 65 + i] * xi;
        }
        if (col < DK) {
#pragma unroll
            for (int r = 0; r < kChunk; ++r) Wd[r * DK + col] = x[r];
        } else {
#pragma unroll
            for (int r = 0; r < kChunk; ++r) Ud[r * dv + (col - DK)] = x[r];
        }
    }
}

// ---------------------------------------------------------------------------
// K3: inter-chunk recurrence on the CUDA cores, 32 rows of S per block
// ---------------------------------------------------------------------------
constexpr int kRowsSimt = 32;

// At DK = 256 the three 64 x DK tiles would not fit in shared memory together: W<- is then read
// from the workspace directly (each value is a broadcast to the 32 threads of a warp).
template <int DK>
constexpr bool ws_in_smem() { return DK <= 128; }

template <int DK>
__host__ __device__ constexpr size_t recur_simt_smem_floats()
{
    return (size_t)kChunk * DK           /* Qs  */
         + (size_t)kChunk * (DK + 1)     /* Ks  */
         + (ws_in_smem<DK>() ? (size_t)kChunk * DK : 0)   /* Ws  */
         + (size_t)kChunk * kRowsSimt    /* Us  */
         + (size_t)kRowsSimt * (DK + 1)  /* Ss  */
         + (size_t)kChunk * kRowsSimt    /* Vn  */
         + (size_t)kChunk * 65           /* Aqk */
         + 3 * kChunk;                   /* bs, eb (e^{b_r}), ed (e^{b_C-b_r}) */
}

template <typename T, int DK>
__global__ void __launch_bounds__(256)
recur_simt_kernel(const T *__restrict__ q, const T *__restrict__ k,
                  const float *__restrict__ init_state, T *__restrict__ out,
                  float *__restrict__ final_state, Geometry gm,
                  const float *__restrict__ bcum, const float *__restrict__ rq,
                  const float *__restrict__ rk, const float *__restrict__ Wg,
                  const float *__restrict__ Ug, unsigned *__restrict__ err_word)
{
    if (err_word && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
        *err_word = kDevErrNone;
    extern __shared__ float smem[];
    float *Qs = smem;
    float *Ks = Qs + kChunk * DK;
    float *Ws = Ks + kChunk * (DK + 1);
    float *Us = Ws + (ws_in_smem<DK>() ? kChunk * DK : 0);
    float *Ss = Us + kChunk * kRowsSimt;
    float *Vn = Ss + kRowsSimt * (DK + 1);
    float *Aqk = Vn + kChunk * kRowsSimt;
    float *bs = Aqk + kChunk * 65;
    float *eb = bs + kChunk;
    float *ed = eb + kChunk;

    const int n = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * kRowsSimt;
    const int tid = threadIdx.x;
    const int H = gm.H, dv = gm.dv;
    int64_t tok0;
    int len;
    seq_span(gm, n, tok0, len);
    const int64_t sbase = slot_base(gm, n);
    const size_t st_off = ((size_t)n * H + h) * (size_t)dv * DK;

    for (int e = tid; e < kRowsSimt * DK; e += blockDim.x) {
        const int j = e / DK, d = e % DK;
        Ss[j * (DK + 1) + d] = init_state ? init_state[st_off + (size_t)(j0 + j) * DK + d] : 0.f;
    }

    const int nchunks = ceil_div(len, kChunk);
    for (int c = 0; c < nchunks; ++c) {
        const int64_t slot = sbase + c;
        const size_t base = ((size_t)slot * H + h) * kChunk;
        const int rows = min(kChunk, len - c * kChunk);
        const int64_t t0 = tok0 + (int64_t)c * kChunk;
        __syncthreads();   // previous chunk finished with every buffer
        if (tid < kChunk) {
            const float b = bcum[base + tid];
            bs[tid] = b;
            eb[tid] = expf(b);
        }
        for (int e = tid; e < kChunk * DK; e += blockDim.x) {
            const int r = e / DK, d = e % DK;
            float xq = 0.f, xk = 0.f;
            if (r < rows) {
                const size_t gi = ((size_t)(t0 + r) * H + h) * DK + d;
                xq = to_f32(q[gi]) * rq[base + r];
                xk = to_f32(k[gi]) * rk[base + r];
            }
            Qs[r * DK + d] = xq;
            Ks[r * (DK + 1) + d] = xk;
            if (ws_in_smem<DK>()) Ws[r * DK + d] = Wg[base * DK + (size_t)r * DK + d];
        }
        for (int e = tid; e < kChunk * kRowsSimt; e += blockDim.x) {
            const int r = e / kRowsSimt, j = e % kRowsSimt;
            Us[e] = Ug[base * dv + (size_t)r * dv + j0 + j];
        }
        __syncthreads();
        if (tid < kChunk) ed[tid] = expf(bs[kChunk - 1] - bs[tid]);
        // V_new = U~ - W<- S^T ;  Aqk = (Q K^T) o Gamma
        {
            const int j = tid & 31;
            for (int r = tid >> 5; r < kChunk; r += 8) {
                const float *wr = ws_in_smem<DK>() ? Ws + r * DK : Wg + base * DK + (size_t)r * DK;
                float acc = 0.f;
#pragma unroll 8
                for (int d = 0; d < DK; ++d) acc += (ws_in_smem<DK>() ? wr[d] : __ldg(wr + d)) * Ss[j * (DK + 1) + d];
                Vn[r * kRowsSimt + j] = Us[r * kRowsSimt + j] - acc;
            }
        }
        for (int e = tid; e < kChunk * kChunk; e += blockDim.x) {
            const int r = e / kChunk, i = e % kChunk;
            float val = 0.f;
            if (i <= r) {
                float acc = 0.f;
#pragma unroll 8
                for (int d = 0; d < DK; ++d) acc += Qs[r * DK + d] * Ks[i * (DK + 1) + d];
                val = acc * expf(bs[r] - bs[i]);
            }
            Aqk[r * 65 + i] = val;
        }
        __syncthreads();
        // O = Q<- S^T + Aqk V_new
        {
            const int j = tid & 31;
            for (int r = tid >> 5; r < rows; r += 8) {
                float acc = 0.f;
#pragma unroll 8
                for (int d = 0; d < DK; ++d) acc += Qs[r * DK + d] * Ss[j * (DK + 1) + d];
                float o = eb[r] * acc;
                for (int i = 0; i <= r; ++i) o += Aqk[r * 65 + i] * Vn[i * kRowsSimt + j];
                out[((size_t)(t0 + r) * H + h) * dv + j0 + j] = from_f32<T>(o);
            }
        }
        __syncthreads();
        // S <- gamma^C S + V_new^T K->
        {
            const float gC = eb[kChunk - 1];
            for (int e = tid; e < kRowsSimt * DK; e += blockDim.x) {
                const int j = e / DK, d = e % DK;
                float acc = gC * Ss[j * (DK + 1) + d];
#pragma unroll 8
                for (int r = 0; r < kChunk; ++r) acc += Vn[r * kRowsSimt + j] * ed[r] * Ks[r * (DK + 1) + d];
                Ss[j * (DK + 1) + d] = acc;
            }
        }
    }
    __syncthreads();
    if (final_state) {
        for (int e = tid; e < kRowsSimt * DK; e += blockDim.x) {
            const int j = e / DK, d = e % DK;
            final_state[st_off + (size_t)(j0 + j) * DK + d] = Ss[j * (DK + 1) + d];
        }
    }
}

// ---------------------------------------------------------------------------
// K3, register-tiled (dk <= 128): the same recurrence with each thread computing
// a small tile of every product from 16-B shared-memory loads along the
// contraction (rows padded to DK + 4 floats, so the rows a warp reads start in
// different banks): about one 16-B load per eight FMAs instead of two 4-B loads
// per FMA in the kernel above, which is bound by shared-memory traffic.
//   (a) V_new = U~ - W<- S^T            64 x 32, thread tile 4 r x 2 j
//   (b) Aqk = (Q K^T) o Gamma           64 x 64 lower, thread tile 4 r x 4 i
//   (c) O = e^b (Q S^T) + Aqk V_new     64 x 32, thread tile 4 r x 2 j
//   (d) S <- e^{b_C} S + (ed o V_new)^T K->   32 x DK, thread tile 2 j x DK/16 d
// ---------------------------------------------------------------------------
template <int DK>
__host__ __device__ constexpr size_t recur_tiled_smem_floats()
{
    return (size_t)kChunk * (DK + 4) * 3       /* Q, K, W rows            */
         + (size_t)kRowsSimt * (DK + 4)        /* S rows                  */
         + (size_t)kChunk * 36 * 3             /* U, V_new, ed o V_new    */
         + (size_t)kChunk * 68                 /* Aqk rows                */
         + 3 * kChunk;                         /* b, e^b, e^{b_C - b}     */
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

template <typename T, int DK>
__global__ void __launch_bounds__(256)
recur_simt_tiled_kernel(const T *__restrict__ q, const T *__restrict__ k,
                        const float *__restrict__ init_state, T *__restrict__ out,
                        float *__restrict__ final_state, Geometry gm,
                        const float *__restrict__ bcum, const float *__restrict__ rq,
                        const float *__restrict__ rk, const float *__restrict__ Wg,
                        const float *__restrict__ Ug, unsigned *__restrict__ err_word)
{
    static_assert(DK == 64 || DK == 128, "tiled path: dk 64 or 128");
    constexpr int P = DK + 4, PV = 36, PA = 68, DT = DK / 16;   // pitches; d per thread in (d)
    if (err_word && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
        *err_word = kDevErrNone;
    extern __shared__ float smem[];
    float *Qs = smem, *Ks = Qs + kChunk * P, *Ws = Ks + kChunk * P, *Ss = Ws + kChunk * P;
    float *Us = Ss + kRowsSimt * P, *Vn = Us + kChunk * PV, *Ve = Vn + kChunk * PV;
    float *Aq = Ve + kChunk * PV, *bs = Aq + kChunk * PA, *eb = bs + kChunk, *ed = eb + kChunk;

    const int n = blockIdx.x, h = blockIdx.y, j0 = blockIdx.z * kRowsSimt;
    const int tid = threadIdx.x;
    const int H = gm.H, dv = gm.dv;
    int64_t tok0;
    int len;
    seq_span(gm, n, tok0, len);
    const int64_t sbase = slot_base(gm, n);
    const size_t st_off = ((size_t)n * H + h) * (size_t)dv * DK;
    // thread tiles
    const int tr = tid >> 4, tc = tid & 15;          // (a), (b), (c): rows 4 tr..; columns by tc
    const int r0 = 4 * tr, ja = 2 * tc, ia = 4 * tc;
    const int jd = 2 * (tid >> 4), dd = DT * (tid & 15);   // (d): rows jd, jd + 1 of S, columns dd..

    for (int e = tid; e < kRowsSimt * DK; e += 256) {
        const int j = e / DK, d = e % DK;
        Ss[j * P + d] = init_state ? init_state[st_off + (size_t)(j0 + j) * DK + d] : 0.f;
    }
    const int nchunks = ceil_div(len, kChunk);
    for (int c = 0; c < nchunks; ++c) {
        const int64_t slot = sbase + c;
        const size_t base = ((size_t)slot * H + h) * kChunk;
        const int rows = min(kChunk, len - c * kChunk);
        const int64_t t0 = tok0 + (int64_t)c * kChunk;
        __syncthreads();   // the previous chunk is done with every buffer
        if (tid < kChunk) {
            const float b = bcum[base + tid];
            bs[tid] = b;
            eb[tid] = expf(b);
        }
        for (int e = tid; e < kChunk * DK; e += 256) {
            const int r = e / DK, d = e % DK;
            float xq = 0.f, xk = 0.f;
            if (r < rows) {
                const size_t gi = ((size_t)(t0 + r) * H + h) * DK + d;
                xq = to_f32(q[gi]) * rq[base + r];
                xk = to_f32(k[gi]) * rk[base + r];
            }
            Qs[r * P + d] = xq;
            Ks[r * P + d] = xk;
            Ws[r * P + d] = Wg[base * DK + (size_t)r * DK + d];
        }
        for (int e = tid; e < kChunk * kRowsSimt; e += 256) {
            const int r = e / kRowsSimt, j = e % kRowsSimt;
            Us[r * PV + j] = Ug[base * dv + (size_t)r * dv + j0 + j];
        }
        __syncthreads();
        if (tid < kChunk) ed[tid] = expf(bs[kChunk - 1] - bs[tid]);
        {   // (a) V_new and (b) Aqk
            float va[4][2] = {}, qs[4][2] = {};
#pragma unroll 4
            for (int d = 0; d < DK; d += 4) {
                const float4 s0 = ld4(Ss + ja * P + d), s1 = ld4(Ss + (ja + 1) * P + d);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 w = ld4(Ws + (r0 + u) * P + d), x = ld4(Qs + (r0 + u) * P + d);
                    va[u][0] += w.x * s0.x + w.y * s0.y + w.z * s0.z + w.w * s0.w;
                    va[u][1] += w.x * s1.x + w.y * s1.y + w.z * s1.z + w.w * s1.w;
                    qs[u][0] += x.x * s0.x + x.y * s0.y + x.z * s0.z + x.w * s0.w;
                    qs[u][1] += x.x * s1.x + x.y * s1.y + x.z * s1.z + x.w * s1.w;
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                Vn[(r0 + u) * PV + ja] = Us[(r0 + u) * PV + ja] - va[u][0];
                Vn[(r0 + u) * PV + ja + 1] = Us[(r0 + u) * PV + ja + 1] - va[u][1];
            }
            float ac[4][4] = {};
            if (ia <= r0 + 3) {
#pragma unroll 4
                for (int d = 0; d < DK; d += 4) {
                    float4 kk[4];
#pragma unroll
                    for (int v = 0; v < 4; ++v) kk[v] = ld4(Ks + (ia + v) * P + d);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4 x = ld4(Qs + (r0 + u) * P + d);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            ac[u][v] += x.x * kk[v].x + x.y * kk[v].y + x.z * kk[v].z + x.w * kk[v].w;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int r = r0 + u, i = ia + v;
                    Aq[r * PA + i] = (i <= r) ? ac[u][v] * expf(bs[r] - bs[i]) : 0.f;
                }
            __syncthreads();
            // (c) O = e^b (Q S^T) + Aqk V_new
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                qs[u][0] *= eb[r0 + u];
                qs[u][1] *= eb[r0 + u];
            }
            for (int i = 0; i <= r0; i += 4) {
                const float2 v0 = *reinterpret_cast<const float2 *>(Vn + i * PV + ja);
                const float2 v1 = *reinterpret_cast<const float2 *>(Vn + (i + 1) * PV + ja);
                const float2 v2 = *reinterpret_cast<const float2 *>(Vn + (i + 2) * PV + ja);
                const float2 v3 = *reinterpret_cast<const float2 *>(Vn + (i + 3) * PV + ja);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 a = ld4(Aq + (r0 + u) * PA + i);
                    qs[u][0] += a.x * v0.x + a.y * v1.x + a.z * v2.x + a.w * v3.x;
                    qs[u][1] += a.x * v0.y + a.y * v1.y + a.z * v2.y + a.w * v3.y;
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int r = r0 + u;
                if (r < rows) {
                    T *o = out + ((size_t)(t0 + r) * H + h) * dv + j0 + ja;
                    o[0] = from_f32<T>(qs[u][0]);
                    o[1] = from_f32<T>(qs[u][1]);
                }
            }
        }
        // (d) S <- e^{b_C} S + (ed o V_new)^T K->, after every thread has read S for (a) and (c)
        for (int e = tid; e < kChunk * kRowsSimt; e += 256) {
            const int r = e / kRowsSimt, j = e % kRowsSimt;
            Ve[r * PV + j] = ed[r] * Vn[r * PV + j];
        }
        __syncthreads();
        {
            const float gC = eb[kChunk - 1];
            float sacc[2][DT];
#pragma unroll
            for (int v = 0; v < DT; ++v) {
                sacc[0][v] = gC * Ss[jd * P + dd + v];
                sacc[1][v] = gC * Ss[(jd + 1) * P + dd + v];
            }
#pragma unroll 4
            for (int r = 0; r < kChunk; ++r) {
                const float2 x = *reinterpret_cast<const float2 *>(Ve + r * PV + jd);
#pragma unroll
                for (int v4 = 0; v4 < DT; v4 += 4) {
                    const float4 kk = ld4(Ks + r * P + dd + v4);
                    sacc[0][v4] += x.x * kk.x; sacc[0][v4 + 1] += x.x * kk.y;
                    sacc[0][v4 + 2] += x.x * kk.z; sacc[0][v4 + 3] += x.x * kk.w;
                    sacc[1][v4] += x.y * kk.x; sacc[1][v4 + 1] += x.y * kk.y;
                    sacc[1][v4 + 2] += x.y * kk.z; sacc[1][v4 + 3] += x.y * kk.w;
                }
            }
#pragma unroll
            for (int v = 0; v < DT; ++v) {
                Ss[jd * P + dd + v] = sacc[0][v];
                Ss[(jd + 1) * P + dd + v] = sacc[1][v];
            }
        }
    }
    __syncthreads();
    if (final_state) {
        for (int e = tid; e < kRowsSimt * DK; e += 256) {
            const int j = e / DK, d = e % DK;
            final_state[st_off + (size_t)(j0 + j) * DK + d] = Ss[j * P + d];
        }
    }
}

// ---------------------------------------------------------------------------
// launcher
// ---------------------------------------------------------------------------
template <typename T, int DK>
static cudaError_t launch_simt_typed(const ChunkArgs &a, cudaStream_t st)
{
    const ChunkWorkspace L = chunk_workspace_layout(a.slots, a.gm.H, DK, a.gm.dv);
    char *ws = (char *)a.workspace;
    float *bcum = (float *)(ws + L.bcum), *rq = (float *)(ws + L.rq), *rk = (float *)(ws + L.rk);
    float *W = (float *)(ws + L.W), *U = (float *)(ws + L.U);
    const T *q = (const T *)a.q, *k = (const T *)a.k, *v = (const T *)a.v;
    unsigned *err = (unsigned *)(ws + L.hdr);

    if (a.slots > 0) {
        dim3 grid1((unsigned)a.slots, a.gm.H);
        prologue_kernel<T><<<grid1, 256, 0, st>>>(q, k, a.g, a.gm, a.scale, a.l2, bcum, rq, rk, err);
        const size_t sm2 = sizeof(float) * ((size_t)kChunk * (DK + 4) + kChunk * 65 + 2 * kChunk);
        cudaFuncSetAttribute(ut_simt_kernel<T, DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2);
        ut_simt_kernel<T, DK><<<grid1, 256, sm2, st>>>(k, v, a.beta, a.gm, bcum, rk, W, U);
    }
    dim3 grid3(a.gm.N, a.gm.H, a.gm.dv / kRowsSimt);
    if constexpr (DK <= 128) {
        const size_t sm3 = sizeof(float) * recur_tiled_smem_floats<DK>();
        cudaFuncSetAttribute(recur_simt_tiled_kernel<T, DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3);
        recur_simt_tiled_kernel<T, DK><<<grid3, 256, sm3, st>>>(q, k, a.init_state, (T *)a.out, a.final_state,
                                                                a.gm, bcum, rq, rk, W, U,
                                                                a.slots > 0 ? nullptr : err);
    } else {
        const size_t sm3 = sizeof(float) * recur_simt_smem_floats<DK>();
        cudaFuncSetAttribute(recur_simt_kernel<T, DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm3);
        recur_simt_kernel<T, DK><<<grid3, 256, sm3, st>>>(q, k, a.init_state, (T *)a.out, a.final_state,
                                                          a.gm, bcum, rq, rk, W, U,
                                                          a.slots > 0 ? nullptr : err);
    }
    return cudaGetLastError();
}

cudaError_t launch_chunk_simt(const ChunkArgs &a, cudaStream_t st)
{
    if (a.dt == 0) {
        if (a.gm.dk == 64) return launch_simt_typed<float, 64>(a, st);
        if (a.gm.dk == 256) return launch_simt_typed<float, 256>(a, st);
        return launch_simt_typed<float, 128>(a, st);
    }
    if (a.gm.dk == 64) return launch_simt_typed<__nv_bfloat16, 64>(a, st);
    if (a.gm.dk == 256) return launch_simt_typed<__nv_bfloat16, 256>(a, st);
    return launch_simt_typed<__nv_bfloat16, 128>(a, st);
}

}  // namespace gdn
