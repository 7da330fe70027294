// chunk_bwd.cu -- backward pass of the chunked gated delta rule.
//
// "Gated Delta Networks: Improving Mamba2 with Delta Rule", §3.3 (the chunkwise
// form; the training forward whose gradients these are).  Per chunk, with
// q^ = scale q / |q|, k^ = k / |k| (when normalising), b the chunk-local
// cumulative log-gate, gam = e^b, gC = e^{b_last}, Gamma_ri = e^{b_r - b_i} (i <= r):
//     L = strictLower(diag(beta)(Gamma o K^K^T)),  T = (I + L)^{-1}
//     U = T diag(beta) V,   W = T diag(beta gam) K^,   A = (Q^ K^T) o Gamma
//     V_new = U - W S^T,    O = diag(gam) Q^ S^T + A V_new
//     S' = gC S + V_new^T diag(gC / gam) K^
// Reverse mode, chunk by chunk from the last one, with dS' the gradient of the
// state after the chunk:
//     dV_new = Kd dS'^T + A^T dO                     (Kd = diag(gC/gam) K^, Qd = diag(gam) Q^)
//     dS     = gC dS' + dO^T Qd - dV_new^T W          (the gradient of the state before it)
// and, in parallel over chunks, the local gradients through A, Qd, Kd, U, W, T, L,
// Gamma and the gates (see bwd_local_kernel), then through the normalisations.
//
// Four fp32 kernels (fp32 inputs, other head sizes):
//   bwd_prep_kernel      per chunk: q^, k^, b, T, U, W, A, Qd, Kd, the unmasked K^K^T and
//                        Q^K^T, and the reverse scan's state-independent A^T dO and dO^T Qd
//   bwd_fwd_scan_kernel  per (sequence, head, 32 state rows): the state at every chunk start
//                        and V_new
//   bwd_bwd_scan_kernel  the same units in reverse: dS' per chunk, dV_new, dS_0
//   bwd_local_kernel     per chunk: dq, dk, dv, dg, dbeta
// Their intermediates are fp32 and their products go through one block-level GEMM (block_gemm)
// on the tensor cores with fp32 accuracy (three tf32 products per pair).  For bf16 inputs with
// dk = 128 and dv a multiple of 128 the forward scan is the tensor-core chunked forward (its
// saving instance); with dk = dv = 128 the other three steps run on the tcgen05 tensor cores
// too (bwd_prep_tc_kernel, bwd_scan_tc_kernel beside the forward scan, bwd_local_tc_kernel),
// each fp32 intermediate entering a product as a bf16 (high, low) pair.
#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int kBT = 256;   // threads per block of every backward kernel

// ---------------------------------------------------------------------------
// per (slot, head) fp32 workspace block
// ---------------------------------------------------------------------------
struct BwdLayout {   // float offsets within one block (under 2^31 for every supported head size)
    int qh, kh, qd, kd, b, t, u, w, a, kk, qk, ado, doq, s, vn, dvn, dsn, dqh, dkh, dw, total;
};

__host__ __device__ inline BwdLayout bwd_layout(int dk, int dv)
{
    BwdLayout L;
    int o = 0;
    L.qh = o;  o += 64 * dk;
    L.kh = o;  o += 64 * dk;
    L.qd = o;  o += 64 * dk;             // diag(gam) Q^
    L.kd = o;  o += 64 * dk;             // diag(gC / gam) K^
    L.b = o;   o += 64;
    L.t = o;   o += 64 * 64;
    L.u = o;   o += 64 * dv;
    L.w = o;   o += 64 * dk;
    L.a = o;   o += 64 * 64;
    L.kk = o;  o += 64 * 64;             // K^ K^T and Q^ K^T before masking
    L.qk = o;  o += 64 * 64;
    L.ado = o; o += 64 * dv;             // A^T dO   (the state-independent part of dV_new)
    L.doq = o; o += dv * dk;             // dO^T Qd  (the state-independent part of dS)
    L.s = o;   o += dv * dk;
    L.vn = o;  o += 64 * dv;
    L.dvn = o; o += 64 * dv;
    L.dsn = o; o += dv * dk;
    L.dqh = o; o += 64 * dk;             // scratch of bwd_local_kernel
    L.dkh = o; o += 64 * dk;
    L.dw = o;  o += 64 * dk;
    L.total = o;
    return L;
}

// ---------------------------------------------------------------------------
// block GEMM: out(i, j, sum_k A(i, k) B(k, j)) for i < M <= 16 MT, j < N <= 16 NT,
// all kBT threads of the block.  A and B are read through functors; AK / BK say
// whether consecutive k are contiguous in memory (then the tile loads run along k),
// so the staging loads coalesce.  Each 16-wide k-tile is staged in shared memory
// (pitch MR + 4 and NR + 4, which makes the fragment loads below conflict-free) and
// multiplied on the tensor cores: mma.sync m16n8k8 in tf32, each operand split into
// a tf32 head and a tf32 tail and the three products head*head + head*tail +
// tail*head accumulated in fp32, which keeps fp32 accuracy (the tail*tail term is
// below fp32 rounding).  The 8 warps tile the output as (MR / 16) x (8 / (MR / 16))
// blocks of 16 rows.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t tf32_of(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo)
{
    hi = tf32_of(x);
    lo = tf32_of(x - __uint_as_float(hi));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2])
{
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// shared staging of block_gemm: up to 16 x (128 + 4) floats for A and for B
constexpr int kStage = 16 * (128 + 4);

// NRS > 0: fo also returns NRS per-element contributions (a float2) to row sums,
// which are reduced in registers and across the 4 lanes that share a row, then added
// to rs0[i] (and rs1[i]) with one shared-memory atomic per row and warp.
template <int MT, int NT, bool AK, bool BK, int NRS = 0, class FA, class FB, class FO>
__device__ __forceinline__ void block_gemm(int M, int N, int K, FA fa, FB fb, FO fo, float *sA, float *sB,
                                           float *rs0 = nullptr, float *rs1 = nullptr)
{
    constexpr int MR = 16 * MT, NR = 16 * NT, MRP = MR + 4, NRP = NR + 4;
    static_assert(16 * MRP <= kStage && 16 * NRP <= kStage, "staging size");
    constexpr int WM = MR / 16, WN = 8 / WM;          // warps along M and N
    static_assert(WM * WN == kBT / 32 && NR % (8 * WN) == 0, "warp tiling");
    constexpr int NTW = NR / WN / 8;                  // n8 tiles per warp
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int m0 = 16 * (warp % WM), n0 = (NR / WN) * (warp / WM);
    float acc[NTW][4];
#pragma unroll
    for (int n = 0; n < NTW; ++n)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[n][q] = 0.f;
    static_assert((16 * MR) % kBT == 0 && (16 * NR) % kBT == 0, "tile sizes");
    constexpr int EA = 16 * MR / kBT, EB = 16 * NR / kBT;   // tile elements per thread
    float va[EA], vb[EB];
    // the loads of a k-tile are all issued before any is stored, and the next tile's
    // loads are in flight while the current one is multiplied
    auto load = [&](int k0) {
#pragma unroll
        for (int u = 0; u < EA; ++u) {
            const int e = tid + u * kBT;
            const int kk = AK ? (e & 15) : (e / MR), i = AK ? (e >> 4) : (e % MR);
            va[u] = (i < M && k0 + kk < K) ? fa(i, k0 + kk) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < EB; ++u) {
            const int e = tid + u * kBT;
            const int kk = BK ? (e & 15) : (e / NR), j = BK ? (e >> 4) : (e % NR);
            vb[u] = (j < N && k0 + kk < K) ? fb(k0 + kk, j) : 0.f;
        }
    };
    auto store = [&]() {
#pragma unroll
        for (int u = 0; u < EA; ++u) {
            const int e = tid + u * kBT;
            const int kk = AK ? (e & 15) : (e / MR), i = AK ? (e >> 4) : (e % MR);
            sA[kk * MRP + i] = va[u];
        }
#pragma unroll
        for (int u = 0; u < EB; ++u) {
            const int e = tid + u * kBT;
            const int kk = BK ? (e & 15) : (e / NR), j = BK ? (e >> 4) : (e % NR);
            sB[kk * NRP + j] = vb[u];
        }
    };
    load(0);
    store();
    __syncthreads();
    for (int k0 = 0; k0 < K; k0 += 16) {
        const bool more = k0 + 16 < K;
        if (more) load(k0 + 16);
#pragma unroll
        for (int ks = 0; ks < 16; ks += 8) {
            uint32_t ah[4], al[4];
            split_tf32(sA[(ks + t) * MRP + m0 + g], ah[0], al[0]);
            split_tf32(sA[(ks + t) * MRP + m0 + g + 8], ah[1], al[1]);
            split_tf32(sA[(ks + t + 4) * MRP + m0 + g], ah[2], al[2]);
            split_tf32(sA[(ks + t + 4) * MRP + m0 + g + 8], ah[3], al[3]);
#pragma unroll
            for (int n = 0; n < NTW; ++n) {
                uint32_t bh[2], bl[2];
                split_tf32(sB[(ks + t) * NRP + n0 + 8 * n + g], bh[0], bl[0]);
                split_tf32(sB[(ks + t + 4) * NRP + n0 + 8 * n + g], bh[1], bl[1]);
                mma_tf32(acc[n], al, bh);
                mma_tf32(acc[n], ah, bl);
                mma_tf32(acc[n], ah, bh);
            }
        }
        __syncthreads();
        if (more) {
            store();
            __syncthreads();
        }
    }
    float rsum[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int n = 0; n < NTW; ++n)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = m0 + g + 8 * (q >> 1), j = n0 + 8 * n + 2 * t + (q & 1);
            if (i < M && j < N) {
                if constexpr (NRS > 0) {
                    const float2 c = fo(i, j, acc[n][q]);
                    rsum[q >> 1][0] += c.x;
                    rsum[q >> 1][1] += c.y;
                } else {
                    fo(i, j, acc[n][q]);
                }
            }
        }
    if constexpr (NRS > 0) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int s = 0; s < NRS; ++s) {
                float v = rsum[hh][s];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                rsum[hh][s] = v;
            }
        if (t == 0)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = m0 + g + 8 * hh;
                if (i < M) {
                    atomicAdd(&rs0[i], rsum[hh][0]);
                    if constexpr (NRS > 1) atomicAdd(&rs1[i], rsum[hh][1]);
                }
            }
    }
}

// block_gemm over column blocks of 128 (N up to 256): fb and fo see global column indices.
template <int MT, bool AK, bool BK, int NRS = 0, class FA, class FB, class FO>
__device__ __forceinline__ void block_gemm_cols(int M, int N, int K, FA fa, FB fb, FO fo, float *sA, float *sB,
                                                float *rs0 = nullptr, float *rs1 = nullptr)
{
    for (int j0 = 0; j0 < N; j0 += 128) {
        block_gemm<MT, 8, AK, BK, NRS>(
            M, min(N - j0, 128), K, fa, [&](int k, int j) { return fb(k, j0 + j); },
            [&](int i, int j, float x) { return fo(i, j0 + j, x); }, sA, sB, rs0, rs1);
    }   // block_gemm ends with a barrier after its last shared reads, so the next block may restage
}

// The chunk (sequence n, chunk c) of `slot` and its token range; false if none.
__device__ __forceinline__ bool chunk_of(const Geometry &gm, int64_t slot, int &n, int &c, int64_t &tok0, int &rows)
{
    return slot_to_chunk(gm, slot, n, c, tok0, rows);
}

struct BwdParams {
    const void *q, *k, *v, *dout;   // dtype dt
    const float *g, *beta, *init_state, *dfinal;
    void *dq, *dk, *dv;             // dtype dt
    float *dg, *dbeta, *dinit;
    float *ws;                      // per (slot, head) blocks of BwdLayout
    int need_u;                     // U~ is only read by the CUDA-core forward scan
    int s_t;                        // the chunk-start states are stored transposed, [dk][dv] (they come
                                    // from the tensor-core forward scan)
    unsigned *err;                  // device error word (the workspace's first word)
    Geometry gm;
    float scale;
    int l2;
};

template <typename T>
__device__ __forceinline__ float ld(const void *p, int64_t i) { return to_f32(reinterpret_cast<const T *>(p)[i]); }

// ---------------------------------------------------------------------------
// bwd_prep_kernel: per (slot, head) -- q^, k^, b, T = (I + L)^{-1}, U, W, A, Qd, Kd,
// K^K^T and Q^K^T unmasked, A^T dO and dO^T Qd
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kBT, 2)
bwd_prep_kernel(const BwdParams p)
{
    extern __shared__ float smb[];
    const Geometry gm = p.gm;
    const int H = gm.H, dk = gm.dk, dv = gm.dv, h = blockIdx.y, tid = threadIdx.x;
    const int64_t slot = blockIdx.x;
    int n, c, rows;
    int64_t tok0;
    if (!chunk_of(gm, slot, n, c, tok0, rows)) return;
    const BwdLayout LY = bwd_layout(dk, dv);
    float *blk = p.ws + (slot * H + h) * LY.total;
    float *sA = smb, *sB = sA + kStage;
    float *sL = sB + kStage;             // [64][65]: L
    float *sT = sL + 64 * 65;            // [64][65]: T = (I + L)^{-1}
    float *sb = sT + 64 * 65, *sbe = sb + 64, *sgam = sbe + 64, *sfk = sgam + 64;   // b, beta, gam, gC / gam

    // gates: chunk-local cumulative log-gate (padding rows: g = 0, beta = 0), a warp scan
    // over each half of the chunk, then the first half's total added to the second
    if (tid < 64) {
        const int64_t th = (tok0 + tid) * H + h;
        float x = tid < rows ? p.g[th] : 0.f;
        const int lane = tid & 31;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        sb[tid] = x;
        sbe[tid] = tid < rows ? p.beta[th] : 0.f;
    }
    __syncthreads();
    if (tid >= 32 && tid < 64) sb[tid] += sb[31];
    __syncthreads();
    if (tid < 64) {
        sgam[tid] = expf(sb[tid]);
        sfk[tid] = expf(sb[63] - sb[tid]);
        blk[LY.b + tid] = sb[tid];
    }
    // normalised q^ (scaled) and k^: one warp per row, rows tid>>5 + 8 i
    for (int r = tid >> 5; r < 64; r += kBT / 32) {
        const int lane = tid & 31;
        const int64_t th = (tok0 + r) * H + h;
        float sq = 0.f, sk = 0.f;
        for (int d = lane; d < dk; d += 32) {
            const float qv = r < rows ? ld<T>(p.q, th * dk + d) : 0.f, kv = r < rows ? ld<T>(p.k, th * dk + d) : 0.f;
            sq += qv * qv;
            sk += kv * kv;
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        const float rq = (p.l2 ? rsqrtf(sq + kL2Eps) : 1.f) * p.scale, rk = p.l2 ? rsqrtf(sk + kL2Eps) : 1.f;
        for (int d = lane; d < dk; d += 32) {
            blk[LY.qh + r * dk + d] = r < rows ? ld<T>(p.q, th * dk + d) * rq : 0.f;
            blk[LY.kh + r * dk + d] = r < rows ? ld<T>(p.k, th * dk + d) * rk : 0.f;
        }
    }
    __syncthreads();
    const float *qh = blk + LY.qh, *kh = blk + LY.kh;
    for (int e = tid; e < 64 * dk; e += kBT) {
        const int r = e / dk;
        blk[LY.qd + e] = sgam[r] * qh[e];
        blk[LY.kd + e] = sfk[r] * kh[e];
    }
    // KK = K^ K^T -> L (strictly lower, beta_r Gamma_ri KK_ri) into sL;  A = (Q^ K^T) o Gamma
    block_gemm<4, 4, true, true>(64, 64, dk, [&](int i, int k) { return kh[i * dk + k]; },
                                 [&](int k, int j) { return kh[j * dk + k]; },
                                 [&](int i, int j, float x) {
                                     sL[i * 65 + j] = j < i ? sbe[i] * expf(sb[i] - sb[j]) * x : 0.f;
                                     blk[LY.kk + i * 64 + j] = x;
                                 }, sA, sB);
    block_gemm<4, 4, true, true>(64, 64, dk, [&](int i, int k) { return qh[i * dk + k]; },
                                 [&](int k, int j) { return kh[j * dk + k]; },
                                 [&](int i, int j, float x) {
                                     blk[LY.a + i * 64 + j] = j <= i ? expf(sb[i] - sb[j]) * x : 0.f;
                                     blk[LY.qk + i * 64 + j] = x;
                                 }, sA, sB);
    __syncthreads();
    // T = (I + L)^{-1} by the block rule [A 0; C B]^{-1} = [A^-1 0; -B^-1 C A^-1  B^-1]:
    // the four 16 x 16 diagonal blocks by forward substitution (thread tid < 64 owns column
    // tid & 15 of block tid >> 4, in registers), then the 16 -> 32 and 32 -> 64 merges
    // as two small products each, X = C A^-1 into scratch, then -B^-1 X
    for (int e = tid; e < 64 * 64; e += kBT) {   // blocks above the diagonal
        const int r = e >> 6, c = e & 63;
        if ((c >> 4) > (r >> 4)) sT[r * 65 + c] = 0.f;
    }
    if (tid < 64) {
        const int b0 = 16 * (tid >> 4), c = tid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = r == c ? 1.f : 0.f;
#pragma unroll
            for (int i = 0; i < r; ++i) acc -= sL[(b0 + r) * 65 + b0 + i] * x[i];
            x[r] = acc;   // zero above the diagonal (r < c), since then every x[i] is zero
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(b0 + r) * 65 + b0 + c] = x[r];
    }
    __syncthreads();
    auto merge = [&](int n, int a0, int b0, float *X, int e0, int estep) {
        // block [b0, b0 + n) x [a0, a0 + n) of T from the diagonal blocks at a0 and b0
        for (int e = e0; e < n * n; e += estep) {
            const int r = e / n, c = e % n;
            float acc = 0.f;
            for (int i = c; i < n; ++i) acc += sL[(b0 + r) * 65 + a0 + i] * sT[(a0 + i) * 65 + a0 + c];
            X[e] = acc;
        }
        __syncthreads();
        for (int e = e0; e < n * n; e += estep) {
            const int r = e / n, c = e % n;
            float acc = 0.f;
            for (int i = 0; i <= r; ++i) acc += sT[(b0 + r) * 65 + b0 + i] * X[i * n + c];
            sT[(b0 + r) * 65 + a0 + c] = -acc;
        }
        __syncthreads();
    };
    merge(16, 32 * (tid >> 7), 32 * (tid >> 7) + 16, sA + 256 * (tid >> 7), tid & 127, 128);   // 16 -> 32, two at once
    merge(32, 0, 32, sA, tid, kBT);                                                            // 32 -> 64
    for (int e = tid; e < 64 * 64; e += kBT) blk[LY.t + e] = sT[(e >> 6) * 65 + (e & 63)];
    const float *Tm = sT;   // pitch 65 below
    // U = T diag(beta) V,  W = T diag(beta gam) K^
    if (p.need_u)
        block_gemm_cols<4, true, false>(64, dv, 64, [&](int i, int k) { return Tm[i * 65 + k]; },
                                        [&](int k, int j) {
                                            return k < rows ? sbe[k] * ld<T>(p.v, ((tok0 + k) * H + h) * dv + j) : 0.f;
                                        },
                                        [&](int i, int j, float x) { blk[LY.u + i * dv + j] = x; }, sA, sB);
    block_gemm_cols<4, true, false>(64, dk, 64, [&](int i, int k) { return Tm[i * 65 + k]; },
                                    [&](int k, int j) { return sbe[k] * sgam[k] * kh[k * dk + j]; },
                                    [&](int i, int j, float x) { blk[LY.w + i * dk + j] = x; }, sA, sB);
    // the state-independent parts of the reverse scan's two products: A^T dO and dO^T Qd
    const float *Ag = blk + LY.a, *qd = blk + LY.qd;
    auto dOf = [&](int r, int j) { return r < rows ? ld<T>(p.dout, ((tok0 + r) * H + h) * dv + j) : 0.f; };
    block_gemm_cols<4, false, false>(64, dv, 64, [&](int r, int i) { return Ag[i * 64 + r]; },
                                     [&](int i, int j) { return dOf(i, j); },
                                     [&](int r, int j, float x) { blk[LY.ado + r * dv + j] = x; }, sA, sB);
    for (int j0 = 0; j0 < dv; j0 += 64)
        block_gemm_cols<4, false, false>(min(64, dv - j0), dk, 64, [&](int i, int r) { return dOf(r, j0 + i); },
                                         [&](int r, int d) { return qd[r * dk + d]; },
                                         [&](int i, int d, float x) { blk[LY.doq + (int64_t)(j0 + i) * dk + d] = x; },
                                         sA, sB);
}

// ---------------------------------------------------------------------------
// bwd_fwd_scan_kernel: per (sequence, head, 32 rows of the state) -- the state at
// every chunk start (S_c, saved) and V_new = U - W S_c^T (saved), then
// S_{c+1} = gC S_c + V_new^T Kd.  State rows evolve independently, so each block
// owns 32 of them, in shared memory.
// ---------------------------------------------------------------------------
constexpr int kScanRows = 32;

__global__ void __launch_bounds__(kBT)
bwd_fwd_scan_kernel(const BwdParams p)
{
    extern __shared__ float smb[];
    const Geometry gm = p.gm;
    const int H = gm.H, dk = gm.dk, dv = gm.dv, n = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int j0 = blockIdx.z * kScanRows;
    const BwdLayout LY = bwd_layout(dk, dv);
    float *sA = smb, *sB = sA + kStage, *S = sB + kStage;   // S [32][dk]: rows j0 .. j0 + 31
    const int64_t SZ = (int64_t)kScanRows * dk, so = (int64_t)j0 * dk;
    for (int64_t e = tid; e < SZ; e += kBT)
        S[e] = p.init_state ? p.init_state[((int64_t)n * H + h) * dv * dk + so + e] : 0.f;
    int64_t tok0;
    int len;
    seq_span(gm, n, tok0, len);
    const int nch = ceil_div(len, kChunk);
    const int64_t slot0 = slot_base(gm, n);
    __syncthreads();
    for (int c = 0; c < nch; ++c) {
        float *blk = p.ws + ((slot0 + c) * H + h) * LY.total;
        const float *b = blk + LY.b, *W = blk + LY.w, *U = blk + LY.u, *kd = blk + LY.kd;
        for (int64_t e = tid; e < SZ; e += kBT) blk[LY.s + so + e] = S[e];
        float *vn = blk + LY.vn;
        block_gemm<4, 2, true, true>(64, kScanRows, dk, [&](int i, int k) { return W[i * dk + k]; },
                                     [&](int k, int j) { return S[j * dk + k]; },
                                     [&](int i, int j, float x) {
                                         vn[i * dv + j0 + j] = U[i * dv + j0 + j] - x;
                                     }, sA, sB);
        __syncthreads();
        const float gC = expf(b[63]);
        block_gemm_cols<2, false, false>(kScanRows, dk, 64, [&](int i, int r) { return vn[r * dv + j0 + i]; },
                                       [&](int r, int d) { return kd[r * dk + d]; },
                                       [&](int i, int d, float x) {
                                           float &s_ = S[(int64_t)i * dk + d];
                                           s_ = gC * s_ + x;
                                       }, sA, sB);
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// bwd_bwd_scan_kernel: per (sequence, head, 32 state rows), chunks in reverse --
// dS' (saved per chunk), dV_new = Kd dS'^T + A^T dO (saved),
// dS = gC dS' + dO^T Qd - dV_new^T W; the gradient of the initial state at the end.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kBT)
bwd_bwd_scan_kernel(const BwdParams p)
{
    extern __shared__ float smb[];
    const Geometry gm = p.gm;
    const int H = gm.H, dk = gm.dk, dv = gm.dv, n = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int j0 = blockIdx.z * kScanRows;
    const BwdLayout LY = bwd_layout(dk, dv);
    float *sA = smb, *sB = sA + kStage, *dS = sB + kStage;   // dS [32][dk]
    const int64_t SZ = (int64_t)kScanRows * dk, so = (int64_t)j0 * dk;
    for (int64_t e = tid; e < SZ; e += kBT)
        dS[e] = p.dfinal ? p.dfinal[((int64_t)n * H + h) * dv * dk + so + e] : 0.f;
    int64_t tok0;
    int len;
    seq_span(gm, n, tok0, len);
    const int nch = ceil_div(len, kChunk);
    const int64_t slot0 = slot_base(gm, n);
    __syncthreads();
    for (int c = nch - 1; c >= 0; --c) {
        float *blk = p.ws + ((slot0 + c) * H + h) * LY.total;
        const float *b = blk + LY.b, *W = blk + LY.w, *kd = blk + LY.kd, *ado = blk + LY.ado, *doq = blk + LY.doq;
        for (int64_t e = tid; e < SZ; e += kBT) blk[LY.dsn + so + e] = dS[e];
        float *dvn = blk + LY.dvn;
        // dV_new = Kd dS'^T + A^T dO  (columns j0 .. j0 + 31; A^T dO comes from the prep kernel)
        block_gemm<4, 2, true, true>(64, kScanRows, dk, [&](int r, int k) { return kd[r * dk + k]; },
                                     [&](int k, int j) { return dS[(int64_t)j * dk + k]; },
                                     [&](int r, int j, float x) { dvn[r * dv + j0 + j] = x + ado[r * dv + j0 + j]; },
                                     sA, sB);
        __syncthreads();
        // dS <- gC dS' + dO^T Qd - dV_new^T W  (dO^T Qd comes from the prep kernel)
        const float gC = expf(b[63]);
        block_gemm_cols<2, false, false>(kScanRows, dk, 64, [&](int i, int k) { return -dvn[k * dv + j0 + i]; },
                                       [&](int k, int d) { return W[k * dk + d]; },
                                       [&](int i, int d, float x) {
                                           float &s_ = dS[(int64_t)i * dk + d];
                                           s_ = gC * s_ + doq[(int64_t)(j0 + i) * dk + d] + x;
                                       }, sA, sB);
        __syncthreads();
    }
    if (p.dinit)
        for (int64_t e = tid; e < SZ; e += kBT) p.dinit[((int64_t)n * H + h) * dv * dk + so + e] = dS[e];
}

// ---------------------------------------------------------------------------
// bwd_local_kernel: per (slot, head) -- the gradients of the chunk's inputs given
// S (state at the chunk start), V_new, dV_new and dS' (gradient after the chunk):
//   dQd = dO S,  dKd = V_new dS',  dW = -dV_new S,  dA = tril(dO V_new^T)
//   dV = diag(beta) T^T dV_new,  T^T dW -> dK, dbeta, dgam
//   dT = dV_new (diag(beta) V)^T + dW (diag(beta gam) K^)^T,  dL = strictLower(-T^T dT T^T)
//   through L = diag(beta)(Gamma o K^K^T) and A = (Q^K^T) o Gamma: dQ^, dK^, dbeta, dGamma
//   db from Gamma, gam, gC/gam and gC (= e^{b_last}), dg = reverse cumsum of db,
//   then dq, dk through the normalisations.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kBT, 2)
bwd_local_kernel(const BwdParams p)
{
    extern __shared__ float smb[];
    const Geometry gm = p.gm;
    const int H = gm.H, dk = gm.dk, dv = gm.dv, h = blockIdx.y, tid = threadIdx.x;
    const int64_t slot = blockIdx.x;
    int n, c, rows;
    int64_t tok0;
    if (!chunk_of(gm, slot, n, c, tok0, rows)) return;
    const BwdLayout LY = bwd_layout(dk, dv);
    float *blk = p.ws + (slot * H + h) * LY.total;
    float *sA = smb, *sB = sA + kStage;
    float *sDA = sB + kStage, *sDT = sDA + 4096, *sX = sDT + 4096, *sGG = sX + 4096;
    float *sDL = sDT;   // dT is dead once X = T^T dT is formed
    float *sb = sGG + 4096, *sbe = sb + 64, *sgam = sbe + 64, *sdgam = sgam + 64, *sdkdf = sdgam + 64,
          *sdbeta = sdkdf + 64, *st = sdbeta + 64, *sfk = st + 64, *sred = sfk + 64;   // sred [kBT]
    const float *qh = blk + LY.qh, *kh = blk + LY.kh, *Tm = blk + LY.t, *S = blk + LY.s, *Vn = blk + LY.vn,
                *dVn = blk + LY.dvn, *dSn = blk + LY.dsn;
    float *dQ = blk + LY.dqh, *dK = blk + LY.dkh, *dW = blk + LY.dw;
    if (tid < 64) {
        sb[tid] = blk[LY.b + tid];
        sbe[tid] = tid < rows ? p.beta[(tok0 + tid) * H + h] : 0.f;
        sgam[tid] = expf(sb[tid]);
        sdgam[tid] = 0.f;
        sdkdf[tid] = 0.f;
        sdbeta[tid] = 0.f;
    }
    __syncthreads();
    if (tid < 64) sfk[tid] = expf(sb[63] - sb[tid]);   // gC / gam
    const float gC = expf(sb[63]);
    auto dOf = [&](int r, int j) { return r < rows ? ld<T>(p.dout, ((tok0 + r) * H + h) * dv + j) : 0.f; };
    auto Vf = [&](int r, int j) { return r < rows ? ld<T>(p.v, ((tok0 + r) * H + h) * dv + j) : 0.f; };
    auto Gam = [&](int r, int i) { return i <= r ? expf(sb[r] - sb[i]) : 0.f; };

    // dQd = dO S  ->  dQ = gam dQd,  dgam += Q^ . dQd
    block_gemm_cols<4, true, false, 1>(64, dk, dv, [&](int r, int j) { return dOf(r, j); },
                                       [&](int j, int d) { return p.s_t ? S[(int64_t)d * dv + j] : S[(int64_t)j * dk + d]; },
                                       [&](int r, int d, float x) {
                                           dQ[r * dk + d] = sgam[r] * x;
                                           return make_float2(qh[r * dk + d] * x, 0.f);
                                       }, sA, sB, sdgam);
    // dKd = V_new dS'  ->  dK = (gC / gam) dKd,  dkdf += K^ . dKd
    block_gemm_cols<4, true, false, 1>(64, dk, dv, [&](int r, int j) { return Vn[r * dv + j]; },
                                       [&](int j, int d) { return dSn[(int64_t)j * dk + d]; },
                                       [&](int r, int d, float x) {
                                           dK[r * dk + d] = sfk[r] * x;
                                           return make_float2(kh[r * dk + d] * x, 0.f);
                                       }, sA, sB, sdkdf);
    // dW = -dV_new S
    block_gemm_cols<4, true, false>(64, dk, dv, [&](int r, int j) { return dVn[r * dv + j]; },
                                    [&](int j, int d) { return p.s_t ? S[(int64_t)d * dv + j] : S[(int64_t)j * dk + d]; },
                                    [&](int r, int d, float x) { dW[r * dk + d] = -x; }, sA, sB);
    // dA = tril(dO V_new^T) (diagonal included)
    block_gemm<4, 4, true, true>(64, 64, dv, [&](int r, int j) { return dOf(r, j); },
                                 [&](int j, int i) { return Vn[i * dv + j]; },
                                 [&](int r, int i, float x) { sDA[r * 64 + i] = i <= r ? x : 0.f; }, sA, sB);
    __syncthreads();
    // T^T dV_new -> dv = beta T^T dV_new,  dbeta += (T^T dV_new) . V
    block_gemm_cols<4, false, false, 1>(64, dv, 64, [&](int i, int r) { return Tm[r * 64 + i]; },
                                        [&](int r, int j) { return dVn[r * dv + j]; },
                                        [&](int i, int j, float x) {
                                            float c = 0.f;
                                            if (i < rows) {
                                                reinterpret_cast<T *>(p.dv)[((tok0 + i) * H + h) * dv + j] =
                                                    from_f32<T>(sbe[i] * x);
                                                c = x * Vf(i, j);
                                            }
                                            return make_float2(c, 0.f);
                                        }, sA, sB, sdbeta);
    // T^T dW -> dK += beta gam T^T dW,  dbeta += gam (T^T dW) . K^,  dgam += beta (T^T dW) . K^
    block_gemm_cols<4, false, false, 2>(64, dk, 64, [&](int i, int r) { return Tm[r * 64 + i]; },
                                        [&](int r, int d) { return dW[r * dk + d]; },
                                        [&](int i, int d, float x) {
                                            dK[i * dk + d] += sbe[i] * sgam[i] * x;
                                            const float t = x * kh[i * dk + d];
                                            return make_float2(sgam[i] * t, sbe[i] * t);
                                        }, sA, sB, sdbeta, sdgam);
    // dT = dV_new (diag(beta) V)^T + dW (diag(beta gam) K^)^T
    block_gemm<4, 4, true, true>(64, 64, dv + dk,
                                 [&](int i, int k) { return k < dv ? dVn[i * dv + k] : dW[i * dk + k - dv]; },
                                 [&](int k, int j) {
                                     return k < dv ? sbe[j] * Vf(j, k) : sbe[j] * sgam[j] * kh[j * dk + k - dv];
                                 },
                                 [&](int i, int j, float x) { sDT[i * 64 + j] = x; }, sA, sB);
    __syncthreads();
    // X = T^T dT;  dL = strictLower(-X T^T)
    block_gemm<4, 4, false, false>(64, 64, 64, [&](int i, int r) { return Tm[r * 64 + i]; },
                                   [&](int r, int j) { return sDT[r * 64 + j]; },
                                   [&](int i, int j, float x) { sX[i * 64 + j] = x; }, sA, sB);
    __syncthreads();
    block_gemm<4, 4, true, true>(64, 64, 64, [&](int i, int r) { return sX[i * 64 + r]; },
                                 [&](int r, int j) { return Tm[j * 64 + r]; },
                                 [&](int i, int j, float x) { sDL[i * 64 + j] = j < i ? -x : 0.f; }, sA, sB);
    __syncthreads();
    // One pass over the 64 x 64 entries, with K^K^T and Q^K^T as the prep kernel formed them:
    //   GG = Gamma o dGamma = Gamma o (dL beta_r KK + dA QK),  dbeta_r += sum_{i<r} dL Gamma KK,
    //   then dA -> dA o Gamma and dL -> M = dL o beta_r Gamma.
    // Warp w takes rows 8w .. 8w + 7, lane l columns l and l + 32 of each.
    static_assert(kBT == 256, "eight warps of eight rows");
    {
        const float *KK = blk + LY.kk, *QK = blk + LY.qk;
        const int warp = tid >> 5, lane = tid & 31;
        for (int rr = 0; rr < 8; ++rr) {
            const int r = warp * 8 + rr;
            float db = 0.f;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int i = lane + 32 * h2, e = r * 64 + i;
                const float G = Gam(r, i), dl = sDL[e], da = sDA[e], kk = KK[e];
                sGG[e] = G * (dl * sbe[r] * kk + da * QK[e]);
                if (i < r) db += dl * G * kk;
                sDA[e] = da * G;
                sDL[e] = dl * sbe[r] * G;
            }
            db = warp_sum(db);
            if (lane == 0) sdbeta[r] += db;
        }
    }
    __syncthreads();
    // dQ += (dA o Gamma) K^;   dK += (dA o Gamma)^T Q^ + M K^ + M^T K^
    block_gemm_cols<4, true, false>(64, dk, 64, [&](int r, int i) { return sDA[r * 64 + i]; },
                                    [&](int i, int d) { return kh[i * dk + d]; },
                                    [&](int r, int d, float x) { dQ[r * dk + d] += x; }, sA, sB);
    block_gemm_cols<4, false, false>(64, dk, 192,
                                    [&](int i, int k) {
                                        return k < 64 ? sDA[k * 64 + i]
                                                      : (k < 128 ? sDL[i * 64 + k - 64] : sDL[(k - 128) * 64 + i]);
                                    },
                                    [&](int k, int d) { return k < 64 ? qh[k * dk + d] : kh[(k & 63) * dk + d]; },
                                    [&](int i, int d, float x) { dK[i * dk + d] += x; }, sA, sB);
    // dgC = <dS', S>
    float part = 0.f;
    for (int64_t e = tid; e < (int64_t)dv * dk; e += kBT)   // e = j dk + d
        part += dSn[e] * (p.s_t ? S[(e % dk) * dv + e / dk] : S[e]);
    sred[tid] = part;
    __syncthreads();
    for (int off = kBT / 2; off > 0; off >>= 1) {
        if (tid < off) sred[tid] += sred[tid + off];
        __syncthreads();
    }
    const float dgC = sred[0];
    // db_r, then dg = reverse cumsum within the chunk
    if (tid < 64) {
        const int r = tid;
        float dbr = 0.f;
        for (int i = 0; i < 64; ++i) dbr += sGG[r * 64 + i] - sGG[i * 64 + r];
        const float t = sdkdf[r] * sfk[r];
        st[r] = t;
        sb[r] = dbr + sdgam[r] * sgam[r] - t;   // sb is no longer needed as b
    }
    __syncthreads();
    if (tid == 0) {
        float tsum = 0.f;
        for (int r = 0; r < 64; ++r) tsum += st[r];
        sb[63] += tsum + dgC * gC;
        float acc = 0.f;
        for (int r = 63; r >= 0; --r) { acc += sb[r]; sb[r] = acc; }
    }
    __syncthreads();
    if (tid < rows) {
        const int64_t th = (tok0 + tid) * H + h;
        p.dg[th] = sb[tid];
        p.dbeta[th] = sdbeta[tid];
    }
    // dq, dk through the normalisations (and scale on q): one warp per row
    for (int r = tid >> 5; r < rows; r += kBT / 32) {
        const int lane = tid & 31;
        const int64_t th = (tok0 + r) * H + h;
        float sq = 0.f, sk = 0.f, qd = 0.f, kd = 0.f;
        for (int d = lane; d < dk; d += 32) {
            const float qv = ld<T>(p.q, th * dk + d), kv = ld<T>(p.k, th * dk + d);
            sq += qv * qv; sk += kv * kv;
            qd += qv * dQ[r * dk + d]; kd += kv * dK[r * dk + d];
        }
        sq = warp_sum(sq); sk = warp_sum(sk); qd = warp_sum(qd); kd = warp_sum(kd);
        const float rq = p.l2 ? rsqrtf(sq + kL2Eps) : 1.f, rk = p.l2 ? rsqrtf(sk + kL2Eps) : 1.f;
        for (int d = lane; d < dk; d += 32) {
            const float qv = ld<T>(p.q, th * dk + d), kv = ld<T>(p.k, th * dk + d);
            const float gq = p.l2 ? p.scale * (rq * dQ[r * dk + d] - rq * rq * rq * qd * qv) : p.scale * dQ[r * dk + d];
            const float gk = p.l2 ? rk * dK[r * dk + d] - rk * rk * rk * kd * kv : dK[r * dk + d];
            reinterpret_cast<T *>(p.dq)[th * dk + d] = from_f32<T>(gq);
            reinterpret_cast<T *>(p.dk)[th * dk + d] = from_f32<T>(gk);
        }
    }
}

// ===========================================================================
// bwd_local_tc_kernel: the products of bwd_local_kernel on the tcgen05 tensor
// cores, for bf16 inputs with dk = dv = 128.  Every operand is staged once into
// shared memory as 128-B-swizzled bf16 tiles -- an fp32 intermediate x as the pair
// hi = bf16(x), lo = bf16(x - hi) (about 16 significand bits), a bf16 input as it
// is -- and serves every product that reads it, as a K-major or an MN-major
// operand.  One thread issues hi*hi + hi*lo + lo*hi (two products when one side is
// an exact bf16 input) into fp32 accumulators in tensor memory; the epilogues and
// the elementwise steps are those of bwd_local_kernel.  The MMAs are M = 128 with
// the chunk's 64 rows in lanes 0-63 (the rows behind a 64-row tile only feed lanes
// 64-127, which are never read); warps 0, 1 (columns 0-63 of a row) and 4, 5
// (columns 64-127) read them back.
// ===========================================================================
namespace lt {
using umma::smem_desc;
using umma::idesc_bf16;
using umma::mma_ss;
using umma::sw128_offset;

// shared memory, bytes from the 1024-aligned base.  Tiles are [64-column block][rows][128 B].
constexpr uint32_t DO = 0;                   // dO [64 r][128 j] bf16; then dT (hi, lo); then M (hi, lo)
constexpr uint32_t VNH = 16384, VNL = 32768; // V_new [64 r][128 j] hi, lo; then K^ [64 i][128 d] hi, lo
constexpr uint32_t DVH = 49152, DVL = 65536; // dV_new [64 r][128 j] hi, lo; then dA' (hi, lo) at DVH
constexpr uint32_t BH = 81920, BL = 114688;  // S^T, then dS'^T [128 d][128 j] hi, lo; then dW hi, lo (BH, BH + 16K),
                                             // V [64 j][128 c] bf16 (BL), X (hi, lo) (BL + 16K); then Q^ (BH, BH + 16K)
constexpr uint32_t TT = 147456;              // T [64 r][64 i] hi, lo (8 KB each)
constexpr uint32_t FA = 163840, FB = 180224; // fp32 [64][64]: dA, then dA o Gamma;  dT, then dL, then M
constexpr uint32_t VEC = 196608;             // per-row vectors, 16 x 64 floats
constexpr uint32_t MISC = VEC + 16 * 64 * 4; // mbarrier, tensor-memory base, abort flag
constexpr uint32_t kSmem = MISC + 64 + 1024;
static_assert(kSmem <= 232448, "local kernel shared memory");
constexpr uint64_t kWaitNs = 1000000000ull;

__device__ __forceinline__ void split_pair(float x, float y, uint32_t &hi, uint32_t &lo)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// 8 consecutive floats of row r, columns 8 c8 .. 8 c8 + 7, into the hi and lo tiles of R rows
__device__ __forceinline__ void put8(uint8_t *hi, uint8_t *lo, int R, int r, int c8, const float (&v)[8])
{
    uint4 h, l;
    split_pair(v[0], v[1], h.x, l.x);
    split_pair(v[2], v[3], h.y, l.y);
    split_pair(v[4], v[5], h.z, l.z);
    split_pair(v[6], v[7], h.w, l.w);
    const uint32_t o = (uint32_t)(c8 >> 3) * (uint32_t)R * 128u + sw128_offset((uint32_t)r, (uint32_t)(c8 & 7) * 8u);
    *reinterpret_cast<uint4 *>(hi + o) = h;
    *reinterpret_cast<uint4 *>(lo + o) = l;
}

// fp32 [R][C] (row stride ld floats, 16-B aligned rows) -> hi, lo tiles; rows >= valid are zero.
// Each thread takes R C / (8 kBT) chunks of 8 columns and issues all their loads before the first
// conversion, so the staging waits on one memory latency, not one per chunk.
template <int R, int C>
__device__ __noinline__ void stage_f32(uint8_t *hi, uint8_t *lo, const float *src, int ld, int valid)
{
    constexpr int per_row = C / 8, NI = R * per_row / kBT;
    static_assert(NI * kBT == R * per_row, "whole chunks per thread");
    float4 a[NI], b[NI];
#pragma unroll
    for (int u = 0; u < NI; ++u) {
        const int id = threadIdx.x + u * kBT, r = id / per_row, c8 = id % per_row;
        if (r < valid) {
            a[u] = *reinterpret_cast<const float4 *>(src + (int64_t)r * ld + 8 * c8);
            b[u] = *reinterpret_cast<const float4 *>(src + (int64_t)r * ld + 8 * c8 + 4);
        } else {
            a[u] = b[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
#pragma unroll
    for (int u = 0; u < NI; ++u) {
        const int id = threadIdx.x + u * kBT, r = id / per_row, c8 = id % per_row;
        const float v[8] = {a[u].x, a[u].y, a[u].z, a[u].w, b[u].x, b[u].y, b[u].z, b[u].w};
        put8(hi, lo, R, r, c8, v);
    }
}

// bf16 (high, low) tile pairs of BYTES bytes each, stored high then low in the layout of the tiles at
// hi and lo: pairs_load issues this thread's 16-B pieces (consecutive threads take consecutive pieces,
// so the loads coalesce) and pairs_store_dot later writes them over the tiles, returning this thread's
// part of sum(new * old), each entry read as high + low (about 16 significand bits).  Split so that the
// loads can be in flight while the products that still read the old tiles finish.
template <int BYTES>
struct PairPieces {
    static constexpr int NI = BYTES / 16 / kBT;
    static_assert(NI * 16 * kBT == BYTES, "whole pieces per thread");
    uint4 nh[NI], nl[NI];
};
template <int BYTES>
__device__ __forceinline__ void pairs_load(PairPieces<BYTES> &pp, const uint8_t *src)
{
#pragma unroll
    for (int u = 0; u < PairPieces<BYTES>::NI; ++u) {
        const uint32_t o = (threadIdx.x + u * kBT) * 16u;
        pp.nh[u] = *reinterpret_cast<const uint4 *>(src + o);
        pp.nl[u] = *reinterpret_cast<const uint4 *>(src + BYTES + o);
    }
}
template <int BYTES>
__device__ __forceinline__ float pairs_store_dot(uint8_t *hi, uint8_t *lo, const PairPieces<BYTES> &pp)
{
    float dot = 0.f;
#pragma unroll
    for (int u = 0; u < PairPieces<BYTES>::NI; ++u) {
        const uint32_t o = (threadIdx.x + u * kBT) * 16u;
        const uint4 oh = *reinterpret_cast<const uint4 *>(hi + o), ol = *reinterpret_cast<const uint4 *>(lo + o);
        const uint32_t ohw[4] = {oh.x, oh.y, oh.z, oh.w}, olw[4] = {ol.x, ol.y, ol.z, ol.w};
        const uint32_t nhw[4] = {pp.nh[u].x, pp.nh[u].y, pp.nh[u].z, pp.nh[u].w};
        const uint32_t nlw[4] = {pp.nl[u].x, pp.nl[u].y, pp.nl[u].z, pp.nl[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ohw[e]));
            const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&olw[e]));
            const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&nhw[e]));
            const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&nlw[e]));
            dot += (x.x + y.x) * (a.x + b.x) + (x.y + y.y) * (a.y + b.y);
        }
        *reinterpret_cast<uint4 *>(hi + o) = pp.nh[u];
        *reinterpret_cast<uint4 *>(lo + o) = pp.nl[u];
    }
    return dot;
}

// bf16 [R][C] (row stride ld elements) -> one tile; rows >= valid are zero (loads batched as above)
template <int R, int C>
__device__ __noinline__ void stage_bf16(uint8_t *dst, const __nv_bfloat16 *src, int64_t ld, int valid)
{
    constexpr int per_row = C / 8, NI = R * per_row / kBT;
    static_assert(NI * kBT == R * per_row, "whole chunks per thread");
    uint4 w[NI];
#pragma unroll
    for (int u = 0; u < NI; ++u) {
        const int id = threadIdx.x + u * kBT, r = id / per_row, c8 = id % per_row;
        w[u] = r < valid ? *reinterpret_cast<const uint4 *>(src + r * ld + 8 * c8) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < NI; ++u) {
        const int id = threadIdx.x + u * kBT, r = id / per_row, c8 = id % per_row;
        const uint32_t o = (uint32_t)(c8 >> 3) * (uint32_t)R * 128u + sw128_offset((uint32_t)r, (uint32_t)(c8 & 7) * 8u);
        *reinterpret_cast<uint4 *>(dst + o) = w[u];
    }
}

// An fp32 [R][C] block (row stride ld, rows >= valid zero) or a bf16 [R][C] block held in registers
// between its loads and its staging into tiles (the layouts of stage_f32 and stage_bf16), so that the
// loads can be in flight while earlier work finishes.
template <int R, int C>
struct F32Block {
    static constexpr int per_row = C / 8, NI = R * per_row / kBT;
    static_assert(NI * kBT == R * per_row, "whole chunks per thread");
    float4 a[NI], b[NI];
};
template <int R, int C>
__device__ __forceinline__ void f32_load(F32Block<R, C> &t, const float *src, int ld, int valid)
{
#pragma unroll
    for (int u = 0; u < F32Block<R, C>::NI; ++u) {
        const int id = threadIdx.x + u * kBT, r = id / F32Block<R, C>::per_row, c8 = id % F32Block<R, C>::per_row;
        if (r < valid) {
            t.a[u] = *reinterpret_cast<const float4 *>(src + (int64_t)r * ld + 8 * c8);
            t.b[u] = *reinterpret_cast<const float4 *>(src + (int64_t)r * ld + 8 * c8 + 4);
        } else {
            t.a[u] = t.b[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
}
template <int R, int C>
__device__ __forceinline__ void f32_put(uint8_t *hi, uint8_t *lo, const F32Block<R, C> &t)
{
#pragma unroll
    for (int u = 0; u < F32Block<R, C>::NI; ++u) {
        const int id = threadIdx.x + u * kBT, r = id / F32Block<R, C>::per_row, c8 = id % F32Block<R, C>::per_row;
        const float v[8] = {t.a[u].x, t.a[u].y, t.a[u].z, t.a[u].w, t.b[u].x, t.b[u].y, t.b[u].z, t.b[u].w};
        put8(hi, lo, R, r, c8, v);
    }
}
template <int R, int C>
struct Bf16Block {
    static constexpr int per_row = C / 8, NI = R * per_row / kBT;
    static_assert(NI * kBT == R * per_row, "whole chunks per thread");
    uint4 w[NI];
};
template <int R, int C>
__device__ __forceinline__ void bf16_load(Bf16Block<R, C> &t, const __nv_bfloat16 *src, int64_t ld, int valid)
{
#pragma unroll
    for (int u = 0; u < Bf16Block<R, C>::NI; ++u) {
        const int id = threadIdx.x + u * kBT, r = id / Bf16Block<R, C>::per_row, c8 = id % Bf16Block<R, C>::per_row;
        t.w[u] = r < valid ? *reinterpret_cast<const uint4 *>(src + r * ld + 8 * c8) : make_uint4(0u, 0u, 0u, 0u);
    }
}
template <int R, int C>
__device__ __forceinline__ void bf16_put(uint8_t *dst, const Bf16Block<R, C> &t)
{
#pragma unroll
    for (int u = 0; u < Bf16Block<R, C>::NI; ++u) {
        const int id = threadIdx.x + u * kBT, r = id / Bf16Block<R, C>::per_row, c8 = id % Bf16Block<R, C>::per_row;
        const uint32_t o = (uint32_t)(c8 >> 3) * (uint32_t)R * 128u + sw128_offset((uint32_t)r, (uint32_t)(c8 & 7) * 8u);
        *reinterpret_cast<uint4 *>(dst + o) = t.w[u];
    }
}

// K-step ks (16 elements of K) of a tile of R rows read as a K-major operand (K along the columns)
__device__ __forceinline__ uint64_t kmaj(uint32_t base, int R, int ks)
{
    return smem_desc(base + (uint32_t)(ks >> 2) * (uint32_t)R * 128u + (uint32_t)(ks & 3) * 32u, 16, 1024);
}
// K-step ks of a tile of R rows read as an MN-major operand (K along the rows)
__device__ __forceinline__ uint64_t mnmaj(uint32_t base, int R, int ks)
{
    return smem_desc(base + (uint32_t)ks * 2048u, (uint32_t)R * 128u, 1024);
}
}  // namespace lt

template <typename T>
__global__ void __launch_bounds__(kBT, 1)
bwd_local_tc_kernel(const BwdParams p)
{
    using namespace lt;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb0 = umma::smem_u32(sm);
    const Geometry gm = p.gm;
    constexpr int DK = 128, DV = 128;
    const int H = gm.H, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t slot = blockIdx.x;
    int n, c, rows;
    int64_t tok0;
    if (!chunk_of(gm, slot, n, c, tok0, rows)) return;
    const BwdLayout LY = bwd_layout(DK, DV);
    float *blk = p.ws + (slot * H + h) * LY.total;
    const float *qh = blk + LY.qh, *kh = blk + LY.kh, *Tm = blk + LY.t, *S = blk + LY.s, *Vn = blk + LY.vn,
                *dVn = blk + LY.dvn, *dSn = blk + LY.dsn;
    // dQ^ and dK^ accumulate in the scratch fields transposed, [d][r]: a warp's 32 rows of one column
    // are then one 128-B line
    float *dQt = blk + LY.dqh, *dKt = blk + LY.dkh;
    float *sDA = reinterpret_cast<float *>(sm + FA), *sDT = reinterpret_cast<float *>(sm + FB), *sDL = sDT;
    float *vec = reinterpret_cast<float *>(sm + VEC);
    float *sb = vec, *sbe = vec + 64, *sgam = vec + 128, *sfk = vec + 192, *sdgam = vec + 256, *sdkdf = vec + 320,
          *sdbeta = vec + 384, *st = vec + 448, *sgrow = vec + 512, *sgcol = vec + 576, *sred = vec + 640;   // sred [256]
    const uint32_t bar = sb0 + MISC, cbar = sb0 + MISC + 16;   // MMA commits; bulk copies
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sm + MISC + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + MISC + 12);
    const __nv_bfloat16 *dO = reinterpret_cast<const __nv_bfloat16 *>(p.dout) + (tok0 * H + h) * DV;
    const __nv_bfloat16 *Vraw = reinterpret_cast<const __nv_bfloat16 *>(p.v) + (tok0 * H + h) * DV;
    const int64_t tstride = (int64_t)H * DV;   // elements between tokens of dO and v

    if (tid == 0) {
        umma::mbar_init(bar, 1);
        umma::mbar_init(cbar, 1);
        *abort_flag = 0;
        umma::fence_mbar_init();
    }
    if (warp == 0) umma::tmem_alloc(tmem_holder, 512);
    if (tid < 64) {
        sb[tid] = blk[LY.b + tid];
        sbe[tid] = tid < rows ? p.beta[(tok0 + tid) * H + h] : 0.f;
        sgam[tid] = expf(sb[tid]);
        sdgam[tid] = 0.f;
        sdkdf[tid] = 0.f;
        sdbeta[tid] = 0.f;
        sgcol[tid] = 0.f;
    }
    // phase 1 operands
    stage_bf16<64, DV>(sm + DO, dO, tstride, rows);
    stage_f32<64, DV>(sm + VNH, sm + VNL, Vn, DV, 64);
    stage_f32<64, DV>(sm + DVH, sm + DVL, dVn, DV, 64);
    stage_f32<DK, DV>(sm + BH, sm + BL, S, DV, DK);   // S^T [d][j]
    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tm = *tmem_holder;
    if (tid < 64) sfk[tid] = expf(sb[63] - sb[tid]);   // gC / gam
    const float gC = expf(sb[63]);
    uint32_t phase = 0;
    // bounded wait for the MMAs committed so far; the outcome is the same for every thread
    auto wait_all = [&]() -> bool {
        bool ok = umma::mbar_wait(bar, phase, kWaitNs);
        if (!ok) {
            *abort_flag = 1;
            atomicExch(p.err, kDevErrTimeout);
        }
        phase ^= 1u;
        const bool bad = __syncthreads_or(!ok || *abort_flag);
        umma::fence_after_sync();
        return !bad;
    };
    uint32_t cphase = 0;
    auto wait_copies = [&]() -> bool {
        bool ok2 = umma::mbar_wait(cbar, cphase, kWaitNs);
        if (!ok2) {
            *abort_flag = 1;
            atomicExch(p.err, kDevErrTimeout);
        }
        cphase ^= 1u;
        return !__syncthreads_or(!ok2 || *abort_flag);
    };
    // one product: nks K-steps, A and B descriptors for (step, lo) via functors; a_exact/b_exact skip lo terms
    auto mma = [&](uint32_t dcol, int N, bool a_mn, bool b_mn, int nks, auto ad, auto bd, bool a_exact, bool b_exact) {
        const uint32_t id = idesc_bf16(128, N, a_mn, b_mn);
#pragma unroll 1
        for (int ks = 0; ks < nks; ++ks) {
            const uint64_t ah = ad(ks, 0), bh = bd(ks, 0);
            mma_ss(tm + dcol, ah, bh, id, ks > 0 ? 1u : 0u);
            if (!b_exact) mma_ss(tm + dcol, ah, bd(ks, 1), id, 1u);
            if (!a_exact) mma_ss(tm + dcol, ad(ks, 1), bh, id, 1u);
        }
    };
    // the calling warp's tensor-memory lanes (rows 0-63 are read by warps 0, 1, 4 and 5), its column half
    const int q4 = warp & 3, half = warp >> 2, row = 32 * q4 + lane;
    const bool reader = q4 < 2;
    auto f = [](uint32_t u) { return __uint_as_float(u); };
    // the calling warp's tensor-memory row, n32 groups of 32 columns from col, fn(u, first column of the
    // group) per group.  The group loop stays rolled: this kernel runs each phase once per CTA, and
    // straight-line epilogues were bound by instruction fetch.
    auto row_groups = [&](uint32_t col, int n32, auto fn) {
        const uint32_t a = tm + ((uint32_t)(32 * q4) << 16) + col;
#pragma unroll 1
        for (int g = 0; g < n32; ++g) {
            uint32_t u[32];
            umma::tmem_ld16(a + 32 * g, *reinterpret_cast<uint32_t(*)[16]>(u));
            umma::tmem_ld16(a + 32 * g + 16, *reinterpret_cast<uint32_t(*)[16]>(u + 16));
            umma::tmem_wait_ld();
            fn(u, 32 * g);
        }
    };
    const uint32_t C1a = 0, C1b = 128, C3 = 256, C4 = 384;

    // ---- phase 1: dQd = dO S, dW' = dV_new S, dA = dO V_new^T; then dKd = V_new dS'
    // (S and dS' are staged transposed, [d][j], as the forward scan and the reverse scan store them:
    // B operands with K = j along the rows' 128 B)
    if (tid == 0) {
        mma(C1a, 128, false, false, 8, [&](int ks, int) { return kmaj(sb0 + DO, 64, ks); },
            [&](int ks, int lo) { return kmaj(sb0 + (lo ? BL : BH), 128, ks); }, true, false);
        mma(C1b, 128, false, false, 8, [&](int ks, int lo) { return kmaj(sb0 + (lo ? DVL : DVH), 64, ks); },
            [&](int ks, int lo) { return kmaj(sb0 + (lo ? BL : BH), 128, ks); }, false, false);
        mma(C4, 64, false, false, 8, [&](int ks, int) { return kmaj(sb0 + DO, 64, ks); },
            [&](int ks, int lo) { return kmaj(sb0 + (lo ? VNL : VNH), 64, ks); }, true, false);
        umma::commit(bar);
    }
    // dS' (saved by the reverse scan as bf16 high and low tiles): loads in flight while the products run
    PairPieces<DV * DK * 2> dsp;
    float4 qpre[16];         // a reader's 64 entries of its q^ row, for the dQd epilogue
    F32Block<64, 64> nT;     // the phase-2 operands T, K^ and V, loaded during the next product
    F32Block<64, DK> nK;
    Bf16Block<64, DV> nV;
    pairs_load(dsp, reinterpret_cast<const uint8_t *>(dSn));
    if (reader) {
#pragma unroll
        for (int e = 0; e < 16; ++e) qpre[e] = *reinterpret_cast<const float4 *>(qh + row * DK + 64 * half + 4 * e);
    }
    bool ok = wait_all();
    if (ok) {
        // dS' over S; dgC = <dS', S> on the way
        sred[tid] = pairs_store_dot(sm + BH, sm + BL, dsp);
        umma::fence_proxy_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        if (tid == 0) {
            mma(C3, 128, false, false, 8, [&](int ks, int lo) { return kmaj(sb0 + (lo ? VNL : VNH), 64, ks); },
                [&](int ks, int lo) { return kmaj(sb0 + (lo ? BL : BH), 128, ks); }, false, false);
            umma::commit(bar);
        }
        // while it runs: dQ = gam dQd (dgam += Q^ . dQd) and dA, from columns this warp's half owns
        if (reader) {
            float acc = 0.f;
            const float g = sgam[row];
            const uint32_t a1 = tm + ((uint32_t)(32 * q4) << 16) + C1a + 64 * half;
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {   // unrolled: the prefetched q^ entries stay in registers
                uint32_t u[32];
                umma::tmem_ld16(a1 + 32 * gg, *reinterpret_cast<uint32_t(*)[16]>(u));
                umma::tmem_ld16(a1 + 32 * gg + 16, *reinterpret_cast<uint32_t(*)[16]>(u + 16));
                umma::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const int d = 64 * half + 32 * gg + e;
                    const float4 qv = qpre[(32 * gg + e) >> 2];
                    acc += qv.x * f(u[e]) + qv.y * f(u[e + 1]) + qv.z * f(u[e + 2]) + qv.w * f(u[e + 3]);
#pragma unroll
                    for (int x = 0; x < 4; ++x) dQt[(d + x) * 64 + row] = g * f(u[e + x]);
                }
            }
            atomicAdd(&sdgam[row], acc);
            row_groups(C4 + 32 * half, 1, [&](const uint32_t (&u)[32], int) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int i = 32 * half + e;
                    sDA[row * 64 + i] = i <= row ? f(u[e]) : 0.f;
                }
            });
        }
        f32_load(nT, Tm, 64, 64);
        f32_load(nK, kh, DK, 64);
        bf16_load(nV, Vraw, tstride, rows);
        ok = wait_all();
    }
    if (ok) {
        // phase 2 operands (loaded above): T, K^ (over V_new, which the V_new dS' product has read) and V
        // (bf16, over dS' lo)
        f32_put(sm + TT, sm + TT + 8192, nT);
        f32_put(sm + VNH, sm + VNL, nK);
        bf16_put(sm + BL, nV);
        __syncthreads();
        // dK = fk dKd (dkdf += K^ . dKd, K^ read from its tiles); dW = -dW' into its tiles over dS'
        if (reader) {
            float acc = 0.f;
            const float fk = sfk[row];
            row_groups(C3 + 64 * half, 2, [&](const uint32_t (&u)[32], int b) {
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    const int d = 64 * half + b + e;
                    const uint32_t o = (uint32_t)(d >> 6) * 8192u + sw128_offset((uint32_t)row, (uint32_t)(d & 63));
                    const uint4 kh4 = *reinterpret_cast<const uint4 *>(sm + VNH + o);
                    const uint4 kl4 = *reinterpret_cast<const uint4 *>(sm + VNL + o);
                    const uint32_t hw[4] = {kh4.x, kh4.y, kh4.z, kh4.w}, lw[4] = {kl4.x, kl4.y, kl4.z, kl4.w};
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const float2 ka = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hw[x]));
                        const float2 kc = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&lw[x]));
                        acc += (ka.x + kc.x) * f(u[e + 2 * x]) + (ka.y + kc.y) * f(u[e + 2 * x + 1]);
                    }
#pragma unroll
                    for (int x = 0; x < 8; ++x) dKt[(d + x) * 64 + row] = fk * f(u[e + x]);
                }
            });
            atomicAdd(&sdkdf[row], acc);
            row_groups(C1b + 64 * half, 2, [&](const uint32_t (&u)[32], int b) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = -f(u[8 * q + e]);
                    put8(sm + BH, sm + BH + 16384, 64, row, 8 * half + b / 8 + q, v);
                }
            });
        }
    }
    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    if (*abort_flag) goto done;
    {
        // ---- phase 2: T^T dV_new, T^T dW, dV_new V^T, dW K^^T
        const uint32_t C5a = 0, C5b = 128, C6a = 256, C6b = 320;
        if (tid == 0) {
            mma(C5a, 128, true, true, 4, [&](int ks, int lo) { return mnmaj(sb0 + TT + (lo ? 8192u : 0u), 64, ks); },
                [&](int ks, int lo) { return mnmaj(sb0 + (lo ? DVL : DVH), 64, ks); }, false, false);
            mma(C5b, 128, true, true, 4, [&](int ks, int lo) { return mnmaj(sb0 + TT + (lo ? 8192u : 0u), 64, ks); },
                [&](int ks, int lo) { return mnmaj(sb0 + BH + (lo ? 16384u : 0u), 64, ks); }, false, false);
            mma(C6a, 64, false, false, 8, [&](int ks, int lo) { return kmaj(sb0 + (lo ? DVL : DVH), 64, ks); },
                [&](int ks, int) { return kmaj(sb0 + BL, 64, ks); }, false, true);
            mma(C6b, 64, false, false, 8, [&](int ks, int lo) { return kmaj(sb0 + BH + (lo ? 16384u : 0u), 64, ks); },
                [&](int ks, int lo) { return kmaj(sb0 + (lo ? VNL : VNH), 64, ks); }, false, false);
            umma::commit(bar);
        }
        if (!wait_all()) goto done;
        if (reader) {
            const int i = row;
            // dv = beta T^T dV_new,  dbeta += (T^T dV_new) . V: dv row i into a bf16 [64][136] staging tile
            // over dV_new (copied out coalesced below; the 8-element pad spreads a warp's rows over the banks)
            float db = 0.f;
            __nv_bfloat16 *dvs = reinterpret_cast<__nv_bfloat16 *>(sm + DVH) + i * (DV + 8) + 64 * half;
            row_groups(C5a + 64 * half, 2, [&](const uint32_t (&u)[32], int b) {
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int j = 64 * half + b + e;
                    *reinterpret_cast<__nv_bfloat162 *>(dvs + b + e) =
                        __floats2bfloat162_rn(sbe[i] * f(u[e]), sbe[i] * f(u[e + 1]));
                    const __nv_bfloat162 vb = *reinterpret_cast<const __nv_bfloat162 *>(
                        sm + BL + (uint32_t)(j >> 6) * 8192u + sw128_offset((uint32_t)i, (uint32_t)(j & 63)));
                    const float2 v2 = __bfloat1622float2(vb);
                    db += f(u[e]) * v2.x + f(u[e + 1]) * v2.y;
                }
            });
            // dK += beta gam T^T dW,  dbeta += gam (T^T dW) . K^,  dgam += beta (T^T dW) . K^
            float tk = 0.f;
            const float bg = sbe[i] * sgam[i];
            row_groups(C5b + 64 * half, 2, [&](const uint32_t (&u)[32], int b) {
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    const int d = 64 * half + b + e;
                    // K^ row i, columns d .. d + 7, from its staged tiles as high + low
                    const uint32_t o = (uint32_t)(d >> 6) * 8192u + sw128_offset((uint32_t)i, (uint32_t)(d & 63));
                    const uint4 kh4 = *reinterpret_cast<const uint4 *>(sm + VNH + o);
                    const uint4 kl4 = *reinterpret_cast<const uint4 *>(sm + VNL + o);
                    const uint32_t hw[4] = {kh4.x, kh4.y, kh4.z, kh4.w}, lw[4] = {kl4.x, kl4.y, kl4.z, kl4.w};
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&hw[x]));
                        const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&lw[x]));
                        tk += f(u[e + 2 * x]) * (a.x + c.x) + f(u[e + 2 * x + 1]) * (a.y + c.y);
                    }
#pragma unroll
                    for (int x = 0; x < 8; ++x) dKt[(d + x) * 64 + i] += bg * f(u[e + x]);
                }
            });
            atomicAdd(&sdbeta[i], db + sgam[i] * tk);
            atomicAdd(&sdgam[i], sbe[i] * tk);
            // dT = dV_new (diag(beta) V)^T + dW (diag(beta gam) K^)^T, columns j of this warp's half
            {
                uint32_t u[32], w[32];
                const uint32_t a = tm + ((uint32_t)(32 * q4) << 16);
                umma::tmem_ld16(a + C6a + 32 * half, *reinterpret_cast<uint32_t(*)[16]>(u));
                umma::tmem_ld16(a + C6a + 32 * half + 16, *reinterpret_cast<uint32_t(*)[16]>(u + 16));
                umma::tmem_ld16(a + C6b + 32 * half, *reinterpret_cast<uint32_t(*)[16]>(w));
                umma::tmem_ld16(a + C6b + 32 * half + 16, *reinterpret_cast<uint32_t(*)[16]>(w + 16));
                umma::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int j = 32 * half + e;
                    sDT[i * 64 + j] = sbe[j] * f(u[e]) + sbe[j] * sgam[j] * f(w[e]);
                }
            }
        }
        umma::fence_before_sync();
        __syncthreads();
        if (tid == 0) {   // K^K^T, Q^K^T for the 64 x 64 pass: bulk copies into the dead dW tiles
            umma::mbar_expect_tx(cbar, 32768);
            umma::bulk_load(sb0 + BH, blk + LY.kk, 16384, cbar);
            umma::bulk_load(sb0 + BH + 16384, blk + LY.qk, 16384, cbar);
        }
        {   // dv: the staged rows out in 16-B pieces, a warp covering two rows
            const __nv_bfloat16 *dvs = reinterpret_cast<const __nv_bfloat16 *>(sm + DVH);
            T *dvo = reinterpret_cast<T *>(p.dv) + (tok0 * H + h) * DV;
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
                const int id = tid + u4 * kBT, r = id >> 4, c8 = id & 15;
                if (r < rows)
                    *reinterpret_cast<uint4 *>(dvo + (int64_t)r * H * DV + 8 * c8) =
                        *reinterpret_cast<const uint4 *>(dvs + r * (DV + 8) + 8 * c8);
            }
        }
        __syncthreads();
        // ---- phase 3: X = T^T dT, then dL = strictLower(-X T^T)
        stage_f32<64, 64>(sm + DO, sm + DO + 8192, sDT, 64, 64);
        umma::fence_proxy_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        const uint32_t C7 = 0, C8 = 64;
        if (tid == 0) {
            mma(C7, 64, true, true, 4, [&](int ks, int lo) { return mnmaj(sb0 + TT + (lo ? 8192u : 0u), 64, ks); },
                [&](int ks, int lo) { return mnmaj(sb0 + DO + (lo ? 8192u : 0u), 64, ks); }, false, false);
            umma::commit(bar);
        }
        F32Block<64, DK> nQ;   // Q^ for phase 4, loaded while phase 3 runs
        f32_load(nQ, qh, DK, 64);
        if (!wait_all()) goto done;
        if (reader)   // X row i, this warp's 32 columns -> X tiles (K-major [i][r])
            row_groups(C7 + 32 * half, 1, [&](const uint32_t (&u)[32], int) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = f(u[8 * q + e]);
                    put8(sm + BL + 16384, sm + BL + 16384 + 8192, 64, row, 4 * half + q, v);
                }
            });
        umma::fence_proxy_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        if (tid == 0) {
            mma(C8, 64, false, false, 4, [&](int ks, int lo) { return kmaj(sb0 + BL + 16384 + (lo ? 8192u : 0u), 64, ks); },
                [&](int ks, int lo) { return kmaj(sb0 + TT + (lo ? 8192u : 0u), 64, ks); }, false, false);
            umma::commit(bar);
        }
        if (!wait_all()) goto done;
        if (reader)
            row_groups(C8 + 32 * half, 1, [&](const uint32_t (&u)[32], int) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int j = 32 * half + e;
                    sDL[row * 64 + j] = j < row ? -f(u[e]) : 0.f;
                }
            });
        __syncthreads();
        // ---- the 64 x 64 pass (as bwd_local_kernel): GG's row and column sums, dbeta, dA o Gamma, M
        {
            if (!wait_copies()) goto done;
            const float *KK = reinterpret_cast<const float *>(sm + BH), *QK = reinterpret_cast<const float *>(sm + BH + 16384);
            float gcol[2] = {0.f, 0.f};
#pragma unroll 1
            for (int rr = 0; rr < 8; ++rr) {
                const int r = warp * 8 + rr;
                float db = 0.f, grow = 0.f;
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int i = lane + 32 * h2, e = r * 64 + i;
                    const float G = i <= r ? expf(sb[r] - sb[i]) : 0.f, dl = sDL[e], da = sDA[e], kk = KK[e];
                    const float gg = G * (dl * sbe[r] * kk + da * QK[e]);
                    grow += gg;
                    gcol[h2] += gg;
                    if (i < r) db += dl * G * kk;
                    sDA[e] = da * G;
                    sDL[e] = dl * sbe[r] * G;
                }
                db = warp_sum(db);
                grow = warp_sum(grow);
                if (lane == 0) {
                    sdbeta[r] += db;
                    sgrow[r] = grow;
                }
            }
            atomicAdd(&sgcol[lane], gcol[0]);
            atomicAdd(&sgcol[lane + 32], gcol[1]);
        }
        __syncthreads();
        // ---- phase 4: [dQ-part; dK-part] = [dA o Gamma; M + M^T] K^ (one product, all 128 rows), then
        // dK-part += (dA o Gamma)^T Q^.  The stacked A tile sits at DVH (high) and DVL (low).
        stage_f32<64, 64>(sm + DVH, sm + DVL, sDA, 64, 64);   // rows 0-63: dA o Gamma [r][i]
#pragma unroll
        for (int u = 0; u < 2; ++u) {   // rows 64-127: M + M^T (M is symmetric in its use: d(K^K^T) = M)
            const int id = tid + u * kBT, r = id >> 3, c8 = id & 7;
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = sDL[r * 64 + 8 * c8 + e] + sDL[(8 * c8 + e) * 64 + r];
            put8(sm + DVH + 8192, sm + DVL + 8192, 64, r, c8, v);
        }
        f32_put(sm + BH, sm + BH + 16384, nQ);                       // Q^ over K^K^T and Q^K^T
        umma::fence_proxy_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        const uint32_t C9 = 0, C10 = 128;
        if (tid == 0) {
            // K^ [i][d] as MN-major B (K = i), at VNH / VNL
            mma(C9, 128, false, true, 4, [&](int ks, int lo) { return kmaj(sb0 + (lo ? DVL : DVH), 128, ks); },
                [&](int ks, int lo) { return mnmaj(sb0 + (lo ? VNL : VNH), 64, ks); }, false, false);
            // (dA o Gamma)^T Q^: A MN-major from rows 0-63 of the stacked tile (M = i, K = r)
            mma(C10, 128, true, true, 4, [&](int ks, int lo) { return mnmaj(sb0 + (lo ? DVL : DVH), 64, ks); },
                [&](int ks, int lo) { return mnmaj(sb0 + BH + (lo ? 16384u : 0u), 64, ks); }, false, false);
            umma::commit(bar);
        }
        if (warp == 0) {   // q and k rows of the chunk for the normalisation: bulk copies over T and the dA staging
            if (lane == 0) umma::mbar_expect_tx(cbar, (uint32_t)(2 * rows * DK * 2));
            __syncwarp();
            for (int r = lane; r < rows; r += 32) {
                const int64_t th = (tok0 + r) * H + h;
                umma::bulk_load(sb0 + TT + (uint32_t)r * 256u, reinterpret_cast<const T *>(p.q) + th * DK, 256, cbar);
                umma::bulk_load(sb0 + FA + (uint32_t)r * 256u, reinterpret_cast<const T *>(p.k) + th * DK, 256, cbar);
            }
        }
        float pq[64];   // this reader's dQ^ scratch entries, loaded while the products run
        if (reader) {
#pragma unroll
            for (int e = 0; e < 64; ++e) pq[e] = dQt[(64 * half + e) * 64 + row];
        }
        if (!wait_all()) goto done;
        // the finished dQ and dK rows, fp32 [64][132] each (33 KB: VNH .. DVH + 1 KB and BH .. BL + 1 KB; a
        // 4-float pad so the rows a warp reads start in different banks), over tiles no product reads any more
        float *fQ = reinterpret_cast<float *>(sm + VNH), *fK = reinterpret_cast<float *>(sm + BH);
        constexpr int PF = DK + 4;
        const uint32_t a0 = tm + ((uint32_t)(32 * q4) << 16);
        if (!reader) {   // rows 64-127 of C9 (the (M + M^T) K^ part of dK) into fK first
            const int r = row - 64;
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                const int d0 = 64 * half + 32 * g;
                uint32_t u[32];
                umma::tmem_ld16(a0 + C9 + d0, *reinterpret_cast<uint32_t(*)[16]>(u));
                umma::tmem_ld16(a0 + C9 + d0 + 16, *reinterpret_cast<uint32_t(*)[16]>(u + 16));
                umma::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(fK + r * PF + d0 + e) = make_float4(f(u[e]), f(u[e + 1]), f(u[e + 2]), f(u[e + 3]));
            }
        }
        __syncthreads();
        if (reader) {
            // columns [64 half, 64 half + 64) of C9 (dQ, with the prefetched scratch), then the same
            // columns of C10 (dK, added to the part already in fK)
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const int d0 = 64 * half + 32 * g;
                uint32_t u[32];
                umma::tmem_ld16(a0 + C9 + d0, *reinterpret_cast<uint32_t(*)[16]>(u));
                umma::tmem_ld16(a0 + C9 + d0 + 16, *reinterpret_cast<uint32_t(*)[16]>(u + 16));
                umma::tmem_wait_ld();
                float *dst = fQ + row * PF + d0;
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(dst + e) =
                        make_float4(pq[32 * g + e] + f(u[e]), pq[32 * g + e + 1] + f(u[e + 1]),
                                    pq[32 * g + e + 2] + f(u[e + 2]), pq[32 * g + e + 3] + f(u[e + 3]));
            }
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                const int d0 = 64 * half + 32 * g;
                uint32_t u[32];
                umma::tmem_ld16(a0 + C10 + d0, *reinterpret_cast<uint32_t(*)[16]>(u));
                umma::tmem_ld16(a0 + C10 + d0 + 16, *reinterpret_cast<uint32_t(*)[16]>(u + 16));
                umma::tmem_wait_ld();
                const float *src = dKt + d0 * 64 + row;
                float *dst = fK + row * PF + d0;
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    float4 a = *reinterpret_cast<const float4 *>(dst + e);
                    a.x += src[e * 64] + f(u[e]);
                    a.y += src[(e + 1) * 64] + f(u[e + 1]);
                    a.z += src[(e + 2) * 64] + f(u[e + 2]);
                    a.w += src[(e + 3) * 64] + f(u[e + 3]);
                    *reinterpret_cast<float4 *>(dst + e) = a;
                }
            }
        }
        __syncthreads();
        for (int off = kBT / 2; off > 0; off >>= 1) {
            if (tid < off) sred[tid] += sred[tid + off];
            __syncthreads();
        }
        const float dgC = sred[0];
        if (tid < 64) {
            const int r = tid;
            const float t = sdkdf[r] * sfk[r];
            st[r] = t;
            sb[r] = sgrow[r] - sgcol[r] + sdgam[r] * sgam[r] - t;   // sb is no longer needed as b
        }
        __syncthreads();
        if (tid == 0) {
            float tsum = 0.f;
            for (int r = 0; r < 64; ++r) tsum += st[r];
            sb[63] += tsum + dgC * gC;
            float acc = 0.f;
            for (int r = 63; r >= 0; --r) { acc += sb[r]; sb[r] = acc; }
        }
        __syncthreads();
        if (tid < rows) {
            const int64_t th = (tok0 + tid) * H + h;
            p.dg[th] = sb[tid];
            p.dbeta[th] = sdbeta[tid];
        }
        // dq, dk through the normalisations (and scale on q): one warp per row, the row loop rolled
        if (!wait_copies()) goto done;
        {
            const T *sq_rows = reinterpret_cast<const T *>(sm + TT), *sk_rows = reinterpret_cast<const T *>(sm + FA);
#pragma unroll 1
            for (int r = warp; r < rows; r += 8) {
                const int64_t th = (tok0 + r) * H + h;
                float qv[4], kv[4], fq[4], fk[4];
                float sq = 0.f, sk = 0.f, qd = 0.f, kd = 0.f;
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int d = lane + 32 * x;
                    qv[x] = to_f32(sq_rows[r * DK + d]);
                    kv[x] = to_f32(sk_rows[r * DK + d]);
                    fq[x] = fQ[r * PF + d];
                    fk[x] = fK[r * PF + d];
                    sq += qv[x] * qv[x]; sk += kv[x] * kv[x];
                    qd += qv[x] * fq[x]; kd += kv[x] * fk[x];
                }
                sq = warp_sum(sq); sk = warp_sum(sk); qd = warp_sum(qd); kd = warp_sum(kd);
                const float rq = p.l2 ? rsqrtf(sq + kL2Eps) : 1.f, rk = p.l2 ? rsqrtf(sk + kL2Eps) : 1.f;
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const int d = lane + 32 * x;
                    const float gq = p.l2 ? p.scale * (rq * fq[x] - rq * rq * rq * qd * qv[x]) : p.scale * fq[x];
                    const float gk = p.l2 ? rk * fk[x] - rk * rk * rk * kd * kv[x] : fk[x];
                    reinterpret_cast<T *>(p.dq)[th * DK + d] = from_f32<T>(gq);
                    reinterpret_cast<T *>(p.dk)[th * DK + d] = from_f32<T>(gk);
                }
            }
        }
    }
done:
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    if (warp == 0) umma::tmem_dealloc(tm, 512);
}

// ---------------------------------------------------------------------------
// bwd_scan_tc_kernel: the reverse scan on the tensor cores, for bf16 inputs with dk = 128 and dv a
// multiple of 128.  One CTA per (sequence, head, 128 state rows), chunks in reverse:
//   save dS' (the gradient of the state after the chunk);
//   dV_new^T = dS' Kd^T + (A^T dO)^T            (saved as dV_new);
//   dS = gC dS' + dO^T Qd - dV_new^T W.
// dS stays in registers, one state row per thread and half of its columns (the rows and columns a
// warp reads from tensor memory).  Each product reads dS', Kd, -dV_new^T and W from shared memory
// as bf16 (high, low) pairs and sums high.high + high.low + low.high in the fp32 accumulator.  Kd and
// W arrive as ready tile pairs (written so by bwd_prep_tc_kernel): the next chunk's copy is issued as
// soon as the product that reads the tiles has finished.  dS' is saved by two bulk copies of its staged tiles (the
// local kernel reads it back in that form), and dO^T Qd is read in its transposed layout, so every
// global access of the chain is coalesced.
// ---------------------------------------------------------------------------
// This grid may run beside the saving forward scan launched before it (programmatic dependent
// launch): it reads nothing that scan writes, and waits for that grid to complete (and its writes
// to be visible) before it exits, so that the kernels after it see both.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

namespace rs {
constexpr uint32_t SAH = 0, SAL = 32768;        // dS'^T [128 d][128 j] high, low (A, MN-major)
constexpr uint32_t KDH = 65536, KDL = 81920;    // Kd [64 r][128 d]
constexpr uint32_t WH = 98304, WL = 114688;     // W [64 r][128 d]
constexpr uint32_t VAH = 131072, VAL = 147456;  // -dV_new^T [128 j][64 r]
constexpr uint32_t MISC = 163840;               // mbarriers (MMA, Kd copy, W copy), tensor-memory base, abort flag
constexpr uint32_t kSmem = MISC + 64 + 1024;
constexpr int kRows = 128;                      // state rows per CTA

}  // namespace rs

template <typename T>
__global__ void __launch_bounds__(kBT, 1)
bwd_scan_tc_kernel(const BwdParams p)
{
    using namespace rs;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb0 = umma::smem_u32(sm);
    const Geometry gm = p.gm;
    constexpr int DK = 128;
    const int H = gm.H, dv = gm.dv, n = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5,
              lane = tid & 31;
    const int j0 = 0;   // dv = 128: one CTA per (sequence, head)
    const int q4 = warp & 3, half = warp >> 2, j = 32 * q4 + lane;   // this thread's state row and column half
    const BwdLayout LY = bwd_layout(DK, dv);
    int64_t tok0;
    int len;
    seq_span(gm, n, tok0, len);
    const int nch = ceil_div(len, kChunk);
    const int64_t slot0 = slot_base(gm, n);
    const int64_t soff = (((int64_t)n * H + h) * dv + j0 + j) * DK + 64 * half;   // in a [N][H][dv][dk] state

    float dS[64];
#pragma unroll
    for (int e = 0; e < 64; e += 4) {
        const float4 x = p.dfinal ? *reinterpret_cast<const float4 *>(p.dfinal + soff + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        dS[e] = x.x; dS[e + 1] = x.y; dS[e + 2] = x.z; dS[e + 3] = x.w;
    }
    if (nch == 0) {   // an empty sequence: the state gradient passes through
        if (p.dinit)
#pragma unroll
            for (int e = 0; e < 64; e += 4)
                *reinterpret_cast<float4 *>(p.dinit + soff + e) = make_float4(dS[e], dS[e + 1], dS[e + 2], dS[e + 3]);
        grid_dep_wait();
        return;
    }
    const uint32_t bar = sb0 + MISC, kbar = sb0 + MISC + 16, wbar = sb0 + MISC + 24;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sm + MISC + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + MISC + 12);
    // the Kd and W tile pairs of one chunk: 32 KB each, contiguous in the workspace and here
    auto copy_kd = [&](int cc) {
        umma::mbar_expect_tx(kbar, 32768);
        umma::bulk_load(sb0 + KDH, p.ws + ((slot0 + cc) * H + h) * LY.total + LY.kd, 32768, kbar);
    };
    auto copy_w = [&](int cc) {
        umma::mbar_expect_tx(wbar, 32768);
        umma::bulk_load(sb0 + WH, p.ws + ((slot0 + cc) * H + h) * LY.total + LY.w, 32768, wbar);
    };
    if (tid == 0) {
        umma::mbar_init(bar, 1);
        umma::mbar_init(kbar, 1);
        umma::mbar_init(wbar, 1);
        *abort_flag = 0;
        umma::fence_mbar_init();
        copy_kd(nch - 1);
        copy_w(nch - 1);
    }
    if (warp == 0) umma::tmem_alloc(tmem_holder, 256);
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tm = *tmem_holder;
    uint32_t kph = 0, wph = 0;
    bool kpend = true, wpend = true;   // copies in flight
    const uint32_t D1 = 0, D2 = 128;   // dV_new^T [128 j][64 r];  dO^T Qd - dV_new^T W [128 j][128 d]
    const uint32_t trow = tm + ((uint32_t)(32 * q4) << 16);
    uint32_t phase = 0;
    auto wait_mma = [&]() -> bool {   // bounded; the outcome is the same for every thread
        const bool ok = umma::mbar_wait(bar, phase, lt::kWaitNs);
        if (!ok) {
            *abort_flag = 1;
            atomicExch(p.err, kDevErrTimeout);
        }
        phase ^= 1u;
        const bool bad = __syncthreads_or(!ok || *abort_flag);
        umma::fence_after_sync();
        return !bad;
    };
    auto mma3 = [&](uint32_t dcol, int N, bool a_mn, bool b_mn, int nks, auto ad, auto bd) {
        const uint32_t id = umma::idesc_bf16(128, N, a_mn, b_mn);
        for (int ks = 0; ks < nks; ++ks) {
            const uint64_t ah = ad(ks, 0), bh = bd(ks, 0);
            umma::mma_ss(tm + dcol, ah, bh, id, ks > 0 ? 1u : 0u);
            umma::mma_ss(tm + dcol, ah, bd(ks, 1), id, 1u);
            umma::mma_ss(tm + dcol, ad(ks, 1), bh, id, 1u);
        }
    };
    auto f = [](uint32_t u) { return __uint_as_float(u); };
    // bounded wait for a tile copy by every thread; false (for all of them) after a timeout
    auto wait_copy = [&](uint32_t b, uint32_t &ph, bool &pend) -> bool {
        const bool ok1 = umma::mbar_wait(b, ph, lt::kWaitNs);
        if (!ok1) {
            *abort_flag = 1;
            atomicExch(p.err, kDevErrTimeout);
        }
        ph ^= 1u;
        pend = false;
        return ok1;
    };

    bool ok = true;
    for (int c = nch - 1; c >= 0 && ok; --c) {
        float *blk = p.ws + ((slot0 + c) * H + h) * LY.total;
        {   // dS' staged transposed for the first product (and saved from there): column j of rows d;
            // a warp's 32 lanes write 64 contiguous bytes of one row
            const uint32_t cb = (uint32_t)(j >> 6) * 16384u;
#pragma unroll
            for (int e = 0; e < 64; ++e) {
                const __nv_bfloat16 hb = __float2bfloat16_rn(dS[e]);
                const __nv_bfloat16 lb = __float2bfloat16_rn(dS[e] - __bfloat162float(hb));
                const uint32_t o = cb + umma::sw128_offset((uint32_t)(64 * half + e), (uint32_t)(j & 63));
                *reinterpret_cast<__nv_bfloat16 *>(sm + SAH + o) = hb;
                *reinterpret_cast<__nv_bfloat16 *>(sm + SAL + o) = lb;
            }
        }
        wait_copy(kbar, kph, kpend);   // this chunk's Kd
        umma::fence_proxy_async();
        umma::fence_before_sync();
        if (__syncthreads_or(*abort_flag)) { ok = false; break; }
        umma::fence_after_sync();
        if (tid == 0) {   // dS' Kd^T: A from the [128 d][128 j] tiles (MN-major), B [64 r][128 d] K-major
            mma3(D1, 64, true, false, 8, [&](int ks, int lo) { return lt::mnmaj(sb0 + (lo ? SAL : SAH), kRows, ks); },
                 [&](int ks, int lo) { return lt::kmaj(sb0 + (lo ? KDL : KDH), 64, ks); });
            umma::commit(bar);
            // dS' for the local kernel: its high and low tiles as they are ([d][j]), 32 KB each
            uint8_t *dsn = reinterpret_cast<uint8_t *>(blk + LY.dsn);
            umma::bulk_store(dsn, sb0 + SAH, 32768);
            umma::bulk_store(dsn + 32768, sb0 + SAL, 32768);
            umma::bulk_commit();
        }
        // while it runs: this thread's 32 entries of A^T dO
        float ado[32];
        {
            const float *a0 = blk + LY.ado + j0 + j + (int64_t)(32 * half) * dv;
#pragma unroll
            for (int e = 0; e < 32; ++e) ado[e] = a0[(int64_t)e * dv];
        }
        if (!(ok = wait_mma())) break;
        if (tid == 0 && c > 0) {   // the first product is done with Kd: the next chunk's comes in
            copy_kd(c - 1);
            kpend = true;
        }
        {   // dV_new^T = dS' Kd^T + (A^T dO)^T: saved as dV_new [r][j], staged negated as A [128 j][64 r]
            uint32_t u[32];
            umma::tmem_ld16(trow + D1 + 32 * half, *reinterpret_cast<uint32_t(*)[16]>(u));
            umma::tmem_ld16(trow + D1 + 32 * half + 16, *reinterpret_cast<uint32_t(*)[16]>(u + 16));
            umma::tmem_wait_ld();
            float *dvn = blk + LY.dvn + j0 + j + (int64_t)(32 * half) * dv;
            float x[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                x[e] = f(u[e]) + ado[e];
                dvn[(int64_t)e * dv] = x[e];
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float v[8] = {-x[8 * q], -x[8 * q + 1], -x[8 * q + 2], -x[8 * q + 3],
                                    -x[8 * q + 4], -x[8 * q + 5], -x[8 * q + 6], -x[8 * q + 7]};
                lt::put8(sm + VAH, sm + VAL, kRows, j, 4 * half + q, v);
            }
        }
        wait_copy(wbar, wph, wpend);   // this chunk's W
        umma::fence_proxy_async();
        umma::fence_before_sync();
        if (__syncthreads_or(*abort_flag)) { ok = false; break; }
        umma::fence_after_sync();
        if (tid == 0) {   // -dV_new^T W: A [128 j][64 r] K-major, B [64 r][128 d] MN-major
            mma3(D2, 128, false, true, 4, [&](int ks, int lo) { return lt::kmaj(sb0 + (lo ? VAL : VAH), kRows, ks); },
                 [&](int ks, int lo) { return lt::mnmaj(sb0 + (lo ? WL : WH), 64, ks); });
            umma::commit(bar);
        }
        // while it runs: this thread's part of dO^T Qd (stored [d][j]) and the chunk's decay
        float dq[64];
        {
            const float *d0 = blk + LY.doq + (int64_t)(64 * half) * dv + j0 + j;
#pragma unroll
            for (int e = 0; e < 64; ++e) dq[e] = d0[(int64_t)e * dv];
        }
        const float gC = expf(blk[LY.b + 63]);
        if (tid == 0) umma::bulk_wait_read();   // dS' tiles read out before the next chunk restages them
        if (!(ok = wait_mma())) break;
        if (tid == 0 && c > 0) {   // the second product is done with W: the next chunk's comes in
            copy_w(c - 1);
            wpend = true;
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {   // dS = gC dS' + dO^T Qd - dV_new^T W
            uint32_t u[32];
            umma::tmem_ld16(trow + D2 + 64 * half + 32 * i, *reinterpret_cast<uint32_t(*)[16]>(u));
            umma::tmem_ld16(trow + D2 + 64 * half + 32 * i + 16, *reinterpret_cast<uint32_t(*)[16]>(u + 16));
            umma::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) dS[32 * i + e] = gC * dS[32 * i + e] + dq[32 * i + e] + f(u[e]);
        }
    }
    if (ok && p.dinit)
#pragma unroll
        for (int e = 0; e < 64; e += 4)
            *reinterpret_cast<float4 *>(p.dinit + soff + e) = make_float4(dS[e], dS[e + 1], dS[e + 2], dS[e + 3]);
    if (tid == 0) {   // copies still in flight after an abort: bounded waits before the CTA leaves
        if (kpend) umma::mbar_wait(kbar, kph, lt::kWaitNs);
        if (wpend) umma::mbar_wait(wbar, wph, lt::kWaitNs);
        umma::bulk_wait_all();
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    if (warp == 0) umma::tmem_dealloc(tm, 256);
    grid_dep_wait();
}

// ---------------------------------------------------------------------------
// bwd_prep_tc_kernel: the prep step on the tensor cores, for bf16 inputs with dk = dv = 128.  One CTA
// per (slot, head), two per SM.  The products, each accumulated in fp32 in tensor memory:
//   G = [K; Q] K^T on the raw bf16 rows: exact products, one MMA per K-step; the norms and the
//     scale are applied afterwards, giving K^K^T and Q^K^T;
//   W = (T diag(beta gam / |k|)) K, with that left factor as a bf16 (high, low) pair;
//   A^T dO, with A = (Q^K^T) o Gamma as a pair;
//   dO^T Qd = (diag(gam scale / |q|) dO)^T Q, with the scaled dO as a pair.
// T = (I + L)^{-1} by the block rule on the CUDA cores, as in bwd_prep_kernel (L kept transposed).
// Kd and W are written as bf16 (high, low) tile pairs, [2 column blocks][64 rows][128 B] each, the
// layout the tensor-core reverse scan copies straight into its operand tiles.
// ---------------------------------------------------------------------------
namespace pp {
// Products with M = 128 whose A has 64 rows read 64 more rows past the tile (their results are not
// read back); the map keeps every such over-read inside this CTA's tiles.
constexpr uint32_t KQ = 0;                    // [K; Q]: [2 column blocks][128 rows][128 B] bf16
constexpr uint32_t DOT = 32768;               // dO [2][64 rows][128 B] bf16
constexpr uint32_t LT = 49152;                // L^T fp32 [64][64]; then A (high, low) [64 q][64 k]
constexpr uint32_t TD = 65536;                // merge scratch; then T diag(beta gam / |k|) (high, low) [64 i][64 r]
constexpr uint32_t ST = 81920;                // T fp32 [64][65]
constexpr uint32_t SD = 65536;                // diag(gam scale / |q|) dO (high, low) [2][64 r][128 B], over TD and T
constexpr uint32_t VEC = 98560;               // per-row vectors, 8 x 64 floats
constexpr uint32_t MISC = VEC + 8 * 64 * 4;   // mbarrier, tensor-memory base, abort flag
constexpr uint32_t kSmem = MISC + 64 + 1024;
static_assert(TD + 16384 <= ST && ST + 64 * 65 * 4 <= VEC && SD + 32768 <= VEC, "prep tile map");
static_assert(TD + 8192 + 16384 <= ST + 64 * 65 * 4, "rows 64-127 of the low TD tile lie inside T");
static_assert(LT + 8192 + 16384 <= TD + 16384, "the second M block of the low A tile lies inside TD");

__device__ __forceinline__ void unpack8(const uint4 &w, float (&v)[8])
{
    const uint32_t x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x[e]));
        v[2 * e] = f2.x;
        v[2 * e + 1] = f2.y;
    }
}
__device__ __forceinline__ void split8(const float (&v)[8], uint4 &hi, uint4 &lo)
{
    lt::split_pair(v[0], v[1], hi.x, lo.x);
    lt::split_pair(v[2], v[3], hi.y, lo.y);
    lt::split_pair(v[4], v[5], hi.z, lo.z);
    lt::split_pair(v[6], v[7], hi.w, lo.w);
}
}  // namespace pp

__global__ void __launch_bounds__(kBT, 2)
bwd_prep_tc_kernel(const BwdParams p)
{
    using namespace pp;
    using umma::sw128_offset;
    extern __shared__ uint8_t smraw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    const uint32_t sb0 = umma::smem_u32(sm);
    const Geometry gm = p.gm;
    constexpr int DK = 128;
    const int H = gm.H, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t slot = blockIdx.x;
    int n, c, rows;
    int64_t tok0;
    if (!chunk_of(gm, slot, n, c, tok0, rows)) return;
    const BwdLayout LY = bwd_layout(DK, DK);
    float *blk = p.ws + (slot * H + h) * LY.total;
    float *vec = reinterpret_cast<float *>(sm + VEC);
    float *sb = vec, *sbe = vec + 64, *sgam = vec + 128, *sfk = vec + 192, *snk = vec + 256, *snq = vec + 320,
          *scoef = vec + 384;
    float *sLT = reinterpret_cast<float *>(sm + LT), *sT = reinterpret_cast<float *>(sm + ST);
    const uint32_t bar = sb0 + MISC;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sm + MISC + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + MISC + 12);
    const int64_t tstride = (int64_t)H * DK;   // elements between tokens of q, k and dO
    const __nv_bfloat16 *qg = reinterpret_cast<const __nv_bfloat16 *>(p.q) + (tok0 * H + h) * DK;
    const __nv_bfloat16 *kg = reinterpret_cast<const __nv_bfloat16 *>(p.k) + (tok0 * H + h) * DK;
    const __nv_bfloat16 *dog = reinterpret_cast<const __nv_bfloat16 *>(p.dout) + (tok0 * H + h) * DK;

    if (tid == 0) {
        umma::mbar_init(bar, 1);
        *abort_flag = 0;
        umma::fence_mbar_init();
    }
    if (warp == 0) umma::tmem_alloc(tmem_holder, 256);
    // gates: chunk-local cumulative log-gate (padding rows: g = 0, beta = 0), a warp scan per half
    if (tid < 64) {
        const int64_t th = (tok0 + tid) * H + h;
        float x = tid < rows ? p.g[th] : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        sb[tid] = x;
        sbe[tid] = tid < rows ? p.beta[th] : 0.f;
    }
    {   // K, Q and dO rows into their tiles (rows past the sequence are zero): 12 16-B pieces a thread
        uint4 w[12];
#pragma unroll
        for (int u = 0; u < 12; ++u) {
            const int id = tid + u * kBT, m = id >> 10, r = (id >> 4) & 63, c8 = id & 15;
            const __nv_bfloat16 *src = m == 0 ? kg : (m == 1 ? qg : dog);
            w[u] = r < rows ? *reinterpret_cast<const uint4 *>(src + r * tstride + 8 * c8) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 12; ++u) {
            const int id = tid + u * kBT, m = id >> 10, r = (id >> 4) & 63, c8 = id & 15;
            const uint32_t o = m < 2 ? (uint32_t)(c8 >> 3) * 16384u + sw128_offset((uint32_t)(64 * m + r), (uint32_t)(c8 & 7) * 8u)
                                     : DOT + (uint32_t)(c8 >> 3) * 8192u + sw128_offset((uint32_t)r, (uint32_t)(c8 & 7) * 8u);
            *reinterpret_cast<uint4 *>(sm + o) = w[u];
        }
    }
    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tm = *tmem_holder;
    uint32_t phase = 0;
    auto wait_mma = [&]() -> bool {   // bounded; the outcome is the same for every thread
        const bool ok = umma::mbar_wait(bar, phase, lt::kWaitNs);
        if (!ok) {
            *abort_flag = 1;
            atomicExch(p.err, kDevErrTimeout);
        }
        phase ^= 1u;
        const bool bad = __syncthreads_or(!ok || *abort_flag);
        umma::fence_after_sync();
        return !bad;
    };
    // nks K-steps into dcol; the low half of A joins unless a_exact, of B unless b_exact
    auto mma = [&](uint32_t dcol, int N, bool a_mn, bool b_mn, int nks, auto ad, auto bd, bool a_exact, bool b_exact) {
        const uint32_t id = umma::idesc_bf16(128, N, a_mn, b_mn);
#pragma unroll 1
        for (int ks = 0; ks < nks; ++ks) {
            const uint64_t ah = ad(ks, 0), bh = bd(ks, 0);
            umma::mma_ss(tm + dcol, ah, bh, id, ks > 0 ? 1u : 0u);
            if (!b_exact) umma::mma_ss(tm + dcol, ah, bd(ks, 1), id, 1u);
            if (!a_exact) umma::mma_ss(tm + dcol, ad(ks, 1), bh, id, 1u);
        }
    };
    auto f = [](uint32_t u) { return __uint_as_float(u); };
    const int q4 = warp & 3, hh = warp >> 2, R = 32 * q4 + lane;   // tensor-memory lane (row) and column half
    const uint32_t trow = tm + ((uint32_t)(32 * q4) << 16);
    const uint32_t DG = 0, DW = 0, DA = 128, DQ = 0;   // columns: G; then W and A^T dO; then dO^T Qd
    auto ld32 = [&](uint32_t col, uint32_t (&u)[32]) {
        umma::tmem_ld16(trow + col, *reinterpret_cast<uint32_t(*)[16]>(u));
        umma::tmem_ld16(trow + col + 16, *reinterpret_cast<uint32_t(*)[16]>(u + 16));
        umma::tmem_wait_ld();
    };

    if (tid == 0) {   // G = [K; Q] K^T: A all 128 rows of [K; Q], B its first 64 (both K-major)
        mma(DG, 64, false, false, 8, [&](int ks, int) { return lt::kmaj(sb0 + KQ, 128, ks); },
            [&](int ks, int) { return lt::kmaj(sb0 + KQ, 128, ks); }, true, true);
        umma::commit(bar);
    }
    if (tid >= 32 && tid < 64) sb[tid] += sb[31];
    {   // norms: four threads a row, each a quarter of its columns, from the staged tiles
        const int r = tid >> 2, qq = tid & 3;
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int c8 = 4 * qq + cc;
            const uint32_t o = (uint32_t)(c8 >> 3) * 16384u + sw128_offset((uint32_t)r, (uint32_t)(c8 & 7) * 8u);
            float kv[8], qv[8];
            unpack8(*reinterpret_cast<const uint4 *>(sm + o), kv);
            unpack8(*reinterpret_cast<const uint4 *>(sm + o + 8192u), qv);   // row 64 + r
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                sk += kv[e] * kv[e];
                sq += qv[e] * qv[e];
            }
        }
        sk += __shfl_xor_sync(0xffffffffu, sk, 1);
        sk += __shfl_xor_sync(0xffffffffu, sk, 2);
        sq += __shfl_xor_sync(0xffffffffu, sq, 1);
        sq += __shfl_xor_sync(0xffffffffu, sq, 2);
        if (qq == 0) {
            snk[r] = p.l2 ? rsqrtf(sk + kL2Eps) : 1.f;
            snq[r] = (p.l2 ? rsqrtf(sq + kL2Eps) : 1.f) * p.scale;
        }
    }
    __syncthreads();
    if (tid < 64) {
        sgam[tid] = expf(sb[tid]);
        sfk[tid] = expf(sb[63] - sb[tid]);
        scoef[tid] = sbe[tid] * sgam[tid] * snk[tid];
        blk[LY.b + tid] = sb[tid];
    }
    __syncthreads();
    if (!wait_mma()) goto done;
    {   // K^K^T (rows 0-63) and Q^K^T (rows 64-127), this thread's 32 columns
        uint32_t u[32];
        ld32(DG + 32 * hh, u);
        if (R < 64) {
            const int i = R;
            const float ni = snk[i], bi = sbe[i], gi = sb[i];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int j = 32 * hh + e;
                const float x = f(u[e]) * ni * snk[j];
                blk[LY.kk + j * 64 + i] = x;   // symmetric: row j, column i is this row's entry j (coalesced)
                sLT[j * 64 + i] = j < i ? bi * expf(gi - sb[j]) * x : 0.f;
            }
        } else {
            const int q = R - 64;
            const float nq = snq[q];
            float *dst = blk + LY.qk + q * 64 + 32 * hh;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const int j = 32 * hh + e;
                *reinterpret_cast<float4 *>(dst + e) =
                    make_float4(f(u[e]) * nq * snk[j], f(u[e + 1]) * nq * snk[j + 1], f(u[e + 2]) * nq * snk[j + 2],
                                f(u[e + 3]) * nq * snk[j + 3]);
            }
        }
    }
    __syncthreads();
    // T = (I + L)^{-1} by the block rule (as bwd_prep_kernel), L read from its transpose
    for (int e = tid; e < 64 * 64; e += kBT) {
        const int r = e >> 6, cc = e & 63;
        if ((cc >> 4) > (r >> 4)) sT[r * 65 + cc] = 0.f;
    }
    if (tid < 64) {
        const int b0 = 16 * (tid >> 4), cc = tid & 15;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = r == cc ? 1.f : 0.f;
#pragma unroll
            for (int i = 0; i < r; ++i) acc -= sLT[(b0 + i) * 64 + b0 + r] * x[i];
            x[r] = acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(b0 + r) * 65 + b0 + cc] = x[r];
    }
    __syncthreads();
    {
        auto merge = [&](int nn, int a0, int b0, float *X, int e0, int estep) {
            for (int e = e0; e < nn * nn; e += estep) {
                const int r = e / nn, cc = e % nn;
                float acc = 0.f;
                for (int i = cc; i < nn; ++i) acc += sLT[(a0 + i) * 64 + b0 + r] * sT[(a0 + i) * 65 + a0 + cc];
                X[e] = acc;
            }
            __syncthreads();
            for (int e = e0; e < nn * nn; e += estep) {
                const int r = e / nn, cc = e % nn;
                float acc = 0.f;
                for (int i = 0; i <= r; ++i) acc += sT[(b0 + r) * 65 + b0 + i] * X[i * nn + cc];
                sT[(b0 + r) * 65 + a0 + cc] = -acc;
            }
            __syncthreads();
        };
        float *X = reinterpret_cast<float *>(sm + TD);
        merge(16, 32 * (tid >> 7), 32 * (tid >> 7) + 16, X + 256 * (tid >> 7), tid & 127, 128);   // 16 -> 32, two at once
        merge(32, 0, 32, X, tid, kBT);                                                            // 32 -> 64
    }
    for (int e = tid; e < 64 * 64; e += kBT) blk[LY.t + e] = sT[(e >> 6) * 65 + (e & 63)];
    // T diag(beta gam / |k|) as a pair (A of the W product, K-major [i][r])
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int id = tid + u * kBT, i = id >> 3, c8 = id & 7;
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = sT[i * 65 + 8 * c8 + e] * scoef[8 * c8 + e];
        lt::put8(sm + TD, sm + TD + 8192, 64, i, c8, v);
    }
    if (q4 >= 2) {   // A = (Q^K^T) o Gamma (lower, diagonal included) as a pair, [q][k], over L^T
        const int q = R - 64;
        uint32_t u[32];
        ld32(DG + 32 * hh, u);
        const float nq = snq[q], gq = sb[q];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int j = 32 * hh + 8 * cc + e;
                v[e] = j <= q ? expf(gq - sb[j]) * f(u[8 * cc + e]) * nq * snk[j] : 0.f;
            }
            lt::put8(sm + LT, sm + LT + 8192, 64, q, 4 * hh + cc, v);
        }
    }
    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    if (tid == 0) {
        // W = TD K: A [64 i][64 r] K-major (rows 64-127 of the product are not read), B = K [r][d] MN-major
        mma(DW, 128, false, true, 4, [&](int ks, int lo) { return lt::kmaj(sb0 + TD + (lo ? 8192u : 0u), 64, ks); },
            [&](int ks, int) { return lt::mnmaj(sb0 + KQ, 128, ks); }, false, true);
        // A^T dO: A MN-major from the [q][k] tile (M = k), B = dO [q][j] MN-major
        mma(DA, 128, true, true, 4, [&](int ks, int lo) { return lt::mnmaj(sb0 + LT + (lo ? 8192u : 0u), 64, ks); },
            [&](int ks, int) { return lt::mnmaj(sb0 + DOT, 64, ks); }, false, true);
        umma::commit(bar);
    }
    // while they run: q^, k^ (fp32) and Kd = diag(gC / gam / |k|) K as a pair of tiles, from the staged rows
#pragma unroll 1
    for (int u = 0; u < 4; ++u) {
        const int id = tid + u * kBT, r = id >> 4, c8 = id & 15;
        const uint32_t o = (uint32_t)(c8 >> 3) * 16384u + sw128_offset((uint32_t)r, (uint32_t)(c8 & 7) * 8u);
        float kv[8], qv[8];
        unpack8(*reinterpret_cast<const uint4 *>(sm + o), kv);
        unpack8(*reinterpret_cast<const uint4 *>(sm + o + 8192u), qv);
        const float rk = snk[r], rq = snq[r], fk = sfk[r] * rk;
        float *qo = blk + LY.qh + r * DK + 8 * c8, *ko = blk + LY.kh + r * DK + 8 * c8;
        *reinterpret_cast<float4 *>(qo) = make_float4(qv[0] * rq, qv[1] * rq, qv[2] * rq, qv[3] * rq);
        *reinterpret_cast<float4 *>(qo + 4) = make_float4(qv[4] * rq, qv[5] * rq, qv[6] * rq, qv[7] * rq);
        *reinterpret_cast<float4 *>(ko) = make_float4(kv[0] * rk, kv[1] * rk, kv[2] * rk, kv[3] * rk);
        *reinterpret_cast<float4 *>(ko + 4) = make_float4(kv[4] * rk, kv[5] * rk, kv[6] * rk, kv[7] * rk);
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = fk * kv[e];
        uint4 hi, lo;
        split8(v, hi, lo);
        uint8_t *kt = reinterpret_cast<uint8_t *>(blk + LY.kd) + (c8 >> 3) * 8192 + sw128_offset((uint32_t)r, (uint32_t)(c8 & 7) * 8u);
        *reinterpret_cast<uint4 *>(kt) = hi;
        *reinterpret_cast<uint4 *>(kt + 16384) = lo;
    }
    if (!wait_mma()) goto done;
    if (q4 < 2) {   // rows 0-63: W as a pair of tiles [r][d], and A^T dO [k][j] (fp32)
        const int i = R;
        uint8_t *wt = reinterpret_cast<uint8_t *>(blk + LY.w);
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
            const int d0 = 64 * hh + 32 * g;
            uint32_t u[32];
            ld32(DW + d0, u);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = f(u[8 * cc + e]);
                uint4 hi, lo;
                split8(v, hi, lo);
                const int d = d0 + 8 * cc;
                uint8_t *dst = wt + (d >> 6) * 8192 + sw128_offset((uint32_t)i, (uint32_t)(d & 63));
                *reinterpret_cast<uint4 *>(dst) = hi;
                *reinterpret_cast<uint4 *>(dst + 16384) = lo;
            }
            ld32(DA + d0, u);
            float *ado = blk + LY.ado + i * DK + d0;
#pragma unroll
            for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4 *>(ado + e) = make_float4(f(u[e]), f(u[e + 1]), f(u[e + 2]), f(u[e + 3]));
        }
    }
    // diag(gam scale / |q|) dO as a pair [r][j] (A of dO^T Qd), over T and TD (their products are done)
#pragma unroll 1
    for (int u = 0; u < 4; ++u) {
        const int id = tid + u * kBT, r = id >> 4, c8 = id & 15;
        const uint32_t o = (uint32_t)(c8 >> 3) * 8192u + sw128_offset((uint32_t)r, (uint32_t)(c8 & 7) * 8u);
        float v[8];
        unpack8(*reinterpret_cast<const uint4 *>(sm + DOT + o), v);
        const float sr = sgam[r] * snq[r];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] *= sr;
        uint4 hi, lo;
        split8(v, hi, lo);
        *reinterpret_cast<uint4 *>(sm + SD + o) = hi;
        *reinterpret_cast<uint4 *>(sm + SD + 16384 + o) = lo;
    }
    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    if (tid == 0) {   // dO^T Qd: A MN-major from the scaled dO [r][j] (M = j), B = Q [r][d] MN-major
        mma(DQ, 128, true, true, 4, [&](int ks, int lo) { return lt::mnmaj(sb0 + SD + (lo ? 16384u : 0u), 64, ks); },
            [&](int ks, int) { return lt::mnmaj(sb0 + KQ + 8192, 128, ks); }, false, true);
        umma::commit(bar);
    }
    if (!wait_mma()) goto done;
    {   // dO^T Qd, all 128 rows j, stored transposed ([d][j]: a warp's rows of one column are one line)
        float *dq = blk + LY.doq;
#pragma unroll 1
        for (int g = 0; g < 2; ++g) {
            const int d0 = 64 * hh + 32 * g;
            uint32_t u[32];
            ld32(DQ + d0, u);
#pragma unroll
            for (int e = 0; e < 32; ++e) dq[(d0 + e) * 128 + R] = f(u[e]);
        }
    }
done:
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    if (warp == 0) umma::tmem_dealloc(tm, 256);
}

template <typename T>
cudaError_t launch_bwd_typed(const BwdArgs &a, cudaStream_t st)
{
    BwdParams p;
    p.q = a.q; p.k = a.k; p.v = a.v; p.dout = a.dout; p.g = a.g; p.beta = a.beta;
    p.init_state = a.init_state; p.dfinal = a.dfinal;
    p.dq = a.dq; p.dk = a.dk; p.dv = a.dv; p.dg = a.dg; p.dbeta = a.dbeta; p.dinit = a.dinit;
    p.ws = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(a.workspace) + 256);
    p.err = reinterpret_cast<unsigned *>(a.workspace);
    const bool tc_scan = a.dt == 1 && chunk_tc_supported(1, a.gm.dk, a.gm.dv, (int64_t)a.gm.B * a.gm.T);
    // bf16 with dk = dv = 128: the tensor-core prep, reverse scan and local kernels, which store dO^T Qd
    // transposed ([dk][dv]) and dS', Kd and W as bf16 (high, low) tiles (implies tc_scan)
    const bool tc_local = a.dt == 1 && a.gm.dk == 128 && a.gm.dv == 128;
    p.need_u = tc_scan ? 0 : 1;
    p.s_t = tc_scan ? 1 : 0;
    p.gm = a.gm; p.scale = a.scale; p.l2 = a.l2;
    const size_t stage = 2 * (size_t)kStage * sizeof(float);
    const size_t sm_prep = stage + sizeof(float) * (2 * 64 * 65 + 4 * 64);
    const size_t sm_scan = stage + sizeof(float) * (size_t)kScanRows * a.gm.dk;
    const size_t sm_local = stage + sizeof(float) * (4 * 4096 + 8 * 64 + kBT);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(bwd_prep_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_prep)))
        return e;
    if ((e = cudaFuncSetAttribute(bwd_fwd_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_scan)))
        return e;
    if ((e = cudaFuncSetAttribute(bwd_bwd_scan_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_scan)))
        return e;
    if ((e = cudaFuncSetAttribute(bwd_local_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm_local)))
        return e;
    if (a.slots > 0) {
        if (tc_local) {
            if ((e = cudaFuncSetAttribute(bwd_prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pp::kSmem)))
                return e;
            bwd_prep_tc_kernel<<<dim3((unsigned)a.slots, a.gm.H), kBT, pp::kSmem, st>>>(p);
        } else {
            bwd_prep_kernel<T><<<dim3((unsigned)a.slots, a.gm.H), kBT, sm_prep, st>>>(p);
        }
    }
    const dim3 sgrid(a.gm.N, a.gm.H, a.gm.dv / kScanRows);
    if (tc_scan) {
        // The forward scan on the tensor cores: the chunked forward itself, saving the state at every
        // chunk start and V_new into their workspace fields.  Its chunk-local blocks (57.8 KB each) sit
        // in the local kernel's scratch fields (dq^, dk^, dW: 96 KB at dk = 128), free until then.
        const BwdLayout LY = bwd_layout(a.gm.dk, a.gm.dv);
        ChunkArgs f;
        f.q = a.q; f.k = a.k; f.v = a.v; f.g = a.g; f.beta = a.beta; f.init_state = a.init_state;
        f.out = nullptr; f.final_state = nullptr; f.gm = a.gm; f.slots = a.slots; f.dt = 1;
        f.scale = a.scale; f.l2 = a.l2; f.workspace = a.workspace;
        f.blocks = p.ws + LY.dqh;
        f.block_stride = (size_t)LY.total * sizeof(float);
        f.save_s = p.ws + LY.s;
        f.save_vn = p.ws + LY.vn;
        f.save_stride = LY.total;
        if ((e = launch_chunk_tc(f, st))) return e;
    } else {
        bwd_fwd_scan_kernel<<<sgrid, kBT, sm_scan, st>>>(p);
    }
    if (tc_local) {
        if ((e = cudaFuncSetAttribute(bwd_scan_tc_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)rs::kSmem)))
            return e;
        // beside the saving forward scan: it may start once that grid's CTAs are all resident
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(a.gm.N, a.gm.H);
        cfg.blockDim = dim3(kBT);
        cfg.dynamicSmemBytes = rs::kSmem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, bwd_scan_tc_kernel<T>, p))) return e;
    } else {
        bwd_bwd_scan_kernel<T><<<sgrid, kBT, sm_scan, st>>>(p);
    }
    if (a.slots > 0) {
        if (tc_local) {
            if ((e = cudaFuncSetAttribute(bwd_local_tc_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)lt::kSmem)))
                return e;
            bwd_local_tc_kernel<T><<<dim3((unsigned)a.slots, a.gm.H), kBT, lt::kSmem, st>>>(p);
        } else {
            bwd_local_kernel<T><<<dim3((unsigned)a.slots, a.gm.H), kBT, sm_local, st>>>(p);
        }
    }
    return cudaGetLastError();
}

}  // namespace

size_t chunk_bwd_workspace_bytes(int64_t slots, int H, int dk, int dv)
{
    return 256 + (size_t)slots * H * bwd_layout(dk, dv).total * sizeof(float);
}

cudaError_t launch_chunk_bwd(const BwdArgs &a, cudaStream_t st)
{
    return a.dt == 1 ? launch_bwd_typed<__nv_bfloat16>(a, st) : launch_bwd_typed<float>(a, st);
}

}  // namespace gdn
