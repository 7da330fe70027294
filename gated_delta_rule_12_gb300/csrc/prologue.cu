// prologue.cu -- the block prologue feeding the gated delta rule.
//
// "Gated Delta Networks: Improving Mamba2 with Delta Rule", §3.4 "Token mixing
// block" and Fig. 1: q, k, v come from their linear projections through a short
// causal convolution and SiLU (q and k are L2-normalised afterwards, which the
// chunked forward and decode do themselves); alpha comes from a linear
// projection in Mamba2's parameterisation and beta from one through a sigmoid:
//     y_t   = silu( sum_{j<K} w[j] x_{t-K+1+j} )      (depthwise, per channel)
//     g_t   = log alpha_t = -exp(A_log) softplus(a_t + dt_bias)
//     beta_t = sigmoid(b_t)
// Tap K-1 multiplies the current token; before a sequence's first token the
// history is the caller's convolution state (its K-1 previous inputs, oldest
// first) or zero, and the state after its last token is written back.
//
// One pass: every raw projection element is read once from HBM (the K-1-token
// halo of a strip comes from L2) and q, k, v, g, beta are written once.  A
// thread owns two consecutive channels of one head over a strip of kStrip
// tokens: it issues the loads of the whole strip first, then runs the filter
// with the K-1 previous inputs of its channels in registers.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

constexpr int kStrip = 64;
constexpr int kThreads = 128;

// two consecutive channels as floats
template <typename T>
__device__ __forceinline__ float2 load2(const T *p)
{
    if constexpr (sizeof(T) == 2) return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
    else return *reinterpret_cast<const float2 *>(p);
}

template <typename T>
__device__ __forceinline__ void store2(T *p, float2 v)
{
    if constexpr (sizeof(T) == 2) *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(v.x, v.y);
    else *reinterpret_cast<float2 *>(p) = v;
}

// SiLU with the fast exponential and division intrinsics: relative error a few fp32 ulps,
// far below the single rounding to the output dtype that follows
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + __expf(-z)); }

__device__ __forceinline__ float softplus(float z) { return z > 20.f ? z : log1pf(expf(z)); }

// One thread per item (strip of kStrip tokens, head h, channel pair cp), the channel pair
// fastest, so a warp's loads and stores of one token are 32 consecutive pairs: channels
// 2 cp, 2 cp + 1 of the concatenated [q | k | v] channel axis of head h.
template <typename T, int K>
__global__ void __launch_bounds__(kThreads)
block_prologue_kernel(const PrologueArgs p)
{
    constexpr int KH = K > 1 ? K - 1 : 1;   // history registers (unused when K == 1)
    const int H = p.H, dk = p.dk, dv = p.dv, Cw = 2 * dk + dv, G = Cw / 2;
    const int64_t BT = (int64_t)p.B * p.T;
    int64_t strips = (BT + kStrip - 1) / kStrip;
    if (strips < 1) strips = 1;
    const int64_t item = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int cp = (int)(item % G);
    const int h = (int)((item / G) % H);
    const int64_t strip = item / ((int64_t)G * H);
    if (strip >= strips) return;
    const int64_t t0 = strip * kStrip, t1 = min(t0 + kStrip, BT);

    // gates of the strip's token-heads, one token per channel-pair thread
    for (int r = cp; r < kStrip && t0 + r < BT; r += G) {
        const int64_t i = (t0 + r) * H + h;
        p.g[i] = -expf(p.A_log[h]) * softplus(p.a[i] + p.dt_bias[h]);
        p.beta[i] = 1.f / (1.f + expf(-p.b[i]));
    }

    const int c0 = 2 * cp;
    const T *x;
    T *y;
    const float *w;
    int d, ch;
    if (c0 < dk) { x = (const T *)p.xq; y = (T *)p.q; w = p.wq; d = dk; ch = c0; }
    else if (c0 < 2 * dk) { x = (const T *)p.xk; y = (T *)p.k; w = p.wk; d = dk; ch = c0 - dk; }
    else { x = (const T *)p.xv; y = (T *)p.v; w = p.wv; d = dv; ch = c0 - 2 * dk; }
    const int64_t xs = (int64_t)H * d;                  // token stride of x and y
    const int64_t xo = (int64_t)h * d + ch;             // offset of this thread's channels in a token
    const T *sin = (const T *)p.state_in;
    T *sout = (T *)p.state_out;
    const int64_t ss = (int64_t)H * Cw;                 // token stride of the convolution state
    const int64_t so = (int64_t)h * Cw + c0;

    // sequences without tokens carry their history through unchanged
    if (strip == 0 && sout && K > 1)
        for (int n = 0; n < p.N; ++n) {
            const int64_t len = p.cu ? (int64_t)p.cu[n + 1] - p.cu[n] : (int64_t)p.T;
            if (len != 0) continue;
            for (int m = 0; m < K - 1; ++m) {
                const float2 hv = sin ? load2(sin + ((int64_t)n * (K - 1) + m) * ss + so) : make_float2(0.f, 0.f);
                store2(sout + ((int64_t)n * (K - 1) + m) * ss + so, hv);
            }
        }
    if (t0 >= BT) return;

    float2 wt[K];   // the two channels' filters
#pragma unroll
    for (int j = 0; j < K; ++j)
        wt[j] = make_float2(w[((int64_t)h * d + ch) * K + j], w[((int64_t)h * d + ch + 1) * K + j]);

    // the sequence holding token t0
    int n;
    int64_t start, end;
    if (p.cu) {
        int lo = 0, hi = p.N;   // last n with cu[n] <= t0 (then cu[n + 1] > t0)
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.cu[mid] <= t0) lo = mid; else hi = mid;
        }
        n = lo;
        start = p.cu[n];
        end = p.cu[n + 1];
    } else {
        n = (int)(t0 / p.T);
        start = (int64_t)n * p.T;
        end = start + p.T;
    }
    float2 hist[KH];   // hist[m]: the input K-1-m tokens back
    auto load_history = [&](int64_t t) {
#pragma unroll
        for (int m = 0; m < K - 1; ++m) {
            const int64_t pos = t - (K - 1) + m;
            if (pos >= start) hist[m] = load2(x + pos * xs + xo);
            else if (sin) hist[m] = load2(sin + ((int64_t)n * (K - 1) + (K - 1) + (pos - start)) * ss + so);
            else hist[m] = make_float2(0.f, 0.f);
        }
    };
    load_history(t0);
    auto step = [&](float2 xt, int64_t t) {
        float2 z = make_float2(wt[K - 1].x * xt.x, wt[K - 1].y * xt.y);
#pragma unroll
        for (int j = 0; j < K - 1; ++j) {
            z.x += wt[j].x * hist[j].x;
            z.y += wt[j].y * hist[j].y;
        }
        store2(y + t * xs + xo, make_float2(silu(z.x), silu(z.y)));
#pragma unroll
        for (int m = 0; m + 1 < K - 1; ++m) hist[m] = hist[m + 1];
        if (K > 1) hist[KH - 1] = xt;
    };
    auto put_state = [&]() {
        if (sout)
#pragma unroll
            for (int m = 0; m < K - 1; ++m) store2(sout + ((int64_t)n * (K - 1) + m) * ss + so, hist[m]);
    };
    if (t0 + kStrip <= end && t1 == t0 + kStrip) {
        // the whole strip inside one sequence: issue all its loads, then filter
        float2 raw[kStrip];
#pragma unroll
        for (int u = 0; u < kStrip; ++u) raw[u] = load2(x + (t0 + u) * xs + xo);
#pragma unroll
        for (int u = 0; u < kStrip; ++u) step(raw[u], t0 + u);
        if (t1 == end) put_state();
    } else {
        // a ragged strip or one crossing sequence boundaries: token by token
#pragma unroll 1
        for (int64_t t = t0; t < t1; ++t) {
            if (t >= end) {   // next sequence (skipping empty ones): fresh history
                while (t >= end) {
                    ++n;
                    start = p.cu ? (int64_t)p.cu[n] : (int64_t)n * p.T;
                    end = p.cu ? (int64_t)p.cu[n + 1] : start + p.T;
                }
                load_history(t);
            }
            step(load2(x + t * xs + xo), t);
            if (t == end - 1) put_state();
        }
    }
}

template <typename T>
cudaError_t launch_typed(const PrologueArgs &a, cudaStream_t st)
{
    const int64_t BT = (int64_t)a.B * a.T;
    int64_t strips = (BT + kStrip - 1) / kStrip;
    if (strips < 1) strips = 1;   // the empty-sequence states are still carried
    const int64_t items = strips * a.H * ((2 * a.dk + a.dv) / 2);
    const unsigned blocks = (unsigned)((items + kThreads - 1) / kThreads);
    switch (a.K) {
        case 1: block_prologue_kernel<T, 1><<<blocks, kThreads, 0, st>>>(a); break;
        case 2: block_prologue_kernel<T, 2><<<blocks, kThreads, 0, st>>>(a); break;
        case 3: block_prologue_kernel<T, 3><<<blocks, kThreads, 0, st>>>(a); break;
        default: block_prologue_kernel<T, 4><<<blocks, kThreads, 0, st>>>(a); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prologue(const PrologueArgs &a, cudaStream_t st)
{
    return a.dt == 1 ? launch_typed<__nv_bfloat16>(a, st) : launch_typed<float>(a, st);
}

}  // namespace gdn
