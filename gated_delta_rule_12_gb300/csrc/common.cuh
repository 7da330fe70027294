// common.cuh -- shared device helpers of the gated delta rule kernels.
//
// Chunk-slot addressing.  A chunk is 64 consecutive tokens of one sequence;
// chunks never cross a sequence boundary, so a sequence of `len` tokens has
// ceil(len / 64) chunks and the last one may be partial.  Per-chunk
// intermediates live in "slots" of the workspace:
//   equal-length batch:   slot(n, c) = n * ceil(T / 64) + c
//   packed varlen:        slot(n, c) = floor(cu[n] / 64) + n + c
// The varlen map is injective because sequence n owns at most
// floor(cu[n+1]/64) - floor(cu[n]/64) + 1 chunks, and it needs at most
// floor(T / 64) + N + 1 slots, a bound the host computes without reading
// cu_seqlens back from the device.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kChunk = 64;
constexpr float kL2Eps = 1e-6f;

// Device error word codes (first 4 bytes of the workspace header).
constexpr unsigned kDevErrNone = 0u;
constexpr unsigned kDevErrTimeout = 1u;
constexpr unsigned kDevErrRange = 2u;   // a tensor-core operand exceeded the fp16 range

struct Geometry {
    int B, T, H, dk, dv, N;
    const int32_t *cu;   // device, may be null
    int nct;             // chunks per row when cu == null
};

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

__host__ inline int64_t num_slots(int B, int T, int N, bool varlen)
{
    if (varlen) return (int64_t)(T / kChunk) + N + 1;
    return (int64_t)B * ceil_div(T, kChunk);
}

// First token (index into the flattened B*T token axis) and length of sequence n.
__device__ __forceinline__ void seq_span(const Geometry &gm, int n, int64_t &tok0, int &len)
{
    if (gm.cu) {
        int a = __ldg(gm.cu + n), b = __ldg(gm.cu + n + 1);
        tok0 = a;
        len = b - a;
    } else {
        tok0 = (int64_t)n * gm.T;
        len = gm.T;
    }
}

__device__ __forceinline__ int64_t slot_base(const Geometry &gm, int n)
{
    if (gm.cu) return (int64_t)(__ldg(gm.cu + n) / kChunk) + n;
    return (int64_t)n * gm.nct;
}

// Map a slot to (sequence, chunk).  Returns false for a slot no chunk uses.
__device__ __forceinline__ bool slot_to_chunk(const Geometry &gm, int64_t slot, int &n, int &c,
                                              int64_t &tok0, int &rows)
{
    int len;
    if (gm.cu) {
        // largest n with slot_base(n) <= slot (slot_base is strictly increasing)
        int lo = 0, hi = gm.N - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (slot_base(gm, mid) <= slot) lo = mid; else hi = mid - 1;
        }
        n = lo;
        int64_t base = slot_base(gm, n);
        if (slot < base) return false;
        c = (int)(slot - base);
    } else {
        n = (int)(slot / gm.nct);
        c = (int)(slot % gm.nct);
    }
    int64_t s0;
    seq_span(gm, n, s0, len);
    if ((int64_t)c * kChunk >= len) return false;
    tok0 = s0 + (int64_t)c * kChunk;
    rows = min(kChunk, len - c * kChunk);
    return true;
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Workspace layout of the chunked forward pass (byte offsets, 256-aligned).
struct ChunkWorkspace {
    size_t hdr;      // 256 B: device error word
    size_t bcum;     // float [slots][H][64]   chunk-local cumulative log-gate b_r
    size_t rq;       // float [slots][H][64]   scale / ||q_r|| (or scale)
    size_t rk;       // float [slots][H][64]   1 / ||k_r||   (or 1)
    size_t W;        // float [slots][H][64][dk]  W<- = T diag(beta e^b) K
    size_t U;        // float [slots][H][64][dv]  U~  = T diag(beta) V
    size_t total;
};

__host__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ inline ChunkWorkspace chunk_workspace_layout(int64_t slots, int H, int dk, int dv)
{
    ChunkWorkspace w;
    size_t off = 0;
    w.hdr = off;  off += 256;
    size_t per = (size_t)slots * H * kChunk * sizeof(float);
    w.bcum = off; off = align256(off + per);
    w.rq = off;   off = align256(off + per);
    w.rk = off;   off = align256(off + per);
    w.W = off;    off = align256(off + per * dk);
    w.U = off;    off = align256(off + per * dv);
    w.total = off;
    return w;
}

}  // namespace gdn
