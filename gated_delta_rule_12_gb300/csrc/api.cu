// api.cu -- the C ABI of libgdn.so (declared in include/gdn.h).
//
// Host-side validation happens first and synchronously; only then is work
// enqueued on the caller's stream.  Nothing here allocates device memory,
// synchronises the device (except gdn_check_device_error) or keeps state
// between calls.
#include <stdint.h>
#include <string.h>

#include "../../include/gdn.h"
#include "common.cuh"
#include "kernels.h"

using namespace gdn;

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned_to(const void *p, unsigned a) { return ((uintptr_t)p & (uintptr_t)(a - 1)) == 0; }

bool chunk_dims_supported(int dk, int dv)
{
    return (dk == 64 || dk == 128 || dk == 256) && dv >= 32 && dv <= 256 && dv % 32 == 0;
}

// the backward kernels are built and tested for dk in {64, 128}
bool bwd_dims_supported(int dk, int dv) { return (dk == 64 || dk == 128 || dk == 256) && dv >= 32 && dv <= 256 && dv % 32 == 0; }

}  // namespace

extern "C" {

const char *gdn_status_string(gdn_status s)
{
    switch (s) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
        case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
        case GDN_ERR_DEVICE_TIMEOUT: return "GDN_ERR_DEVICE_TIMEOUT";
        case GDN_ERR_RANGE: return "GDN_ERR_RANGE";
    }
    return "GDN_UNKNOWN_STATUS";
}

size_t gdn_chunk_fwd_workspace_size(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv,
                                    int32_t num_seqs, gdn_dtype dt)
{
    if (B < 1 || T < 0 || H < 1 || num_seqs < 0) return 0;
    if (dt != GDN_F32 && dt != GDN_BF16) return 0;
    if (!chunk_dims_supported(dk, dv)) return 0;
    const bool varlen = num_seqs > 0;
    if (varlen && B != 1) return 0;
    const int64_t slots = num_slots(B, T, varlen ? num_seqs : B, varlen);
    if (chunk_tc_supported(dt == GDN_BF16 ? 1 : 0, dk, dv, (int64_t)B * T))
        return chunk_tc_workspace_bytes(slots, H);
    return chunk_workspace_layout(slots, H, dk, dv).total;
}

int32_t gdn_chunk_fwd_kernel_count(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv,
                                   int32_t num_seqs, gdn_dtype dt)
{
    if (gdn_chunk_fwd_workspace_size(B, T, H, dk, dv, num_seqs, dt) == 0) return 0;
    const int64_t tokens = (int64_t)B * T;
    if (chunk_tc_supported(dt == GDN_BF16 ? 1 : 0, dk, dv, tokens)) return 2;   // UT + recurrence
    return tokens > 0 ? 3 : 1;   // prologue + UT + recurrence, or the state copy alone
}

gdn_status gdn_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                         const float *beta, const float *init_state, const int32_t *cu_seqlens,
                         int32_t num_seqs, void *out, float *final_state, int32_t B, int32_t T,
                         int32_t H, int32_t dk, int32_t dv, gdn_dtype dt, float scale,
                         int32_t use_qk_l2norm, int32_t chunk_size, void *workspace,
                         size_t workspace_bytes, void *stream)
{
    if (B < 1 || T < 0 || H < 1 || dk < 1 || dv < 1) return GDN_ERR_INVALID_ARG;
    if (dt != GDN_F32 && dt != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (chunk_size != kChunk) return GDN_ERR_UNSUPPORTED;
    if (!chunk_dims_supported(dk, dv)) return GDN_ERR_UNSUPPORTED;
    const bool varlen = cu_seqlens != nullptr;
    if (varlen && (B != 1 || num_seqs < 1)) return GDN_ERR_INVALID_ARG;
    if (!varlen && num_seqs != 0 && num_seqs != B) return GDN_ERR_INVALID_ARG;
    const int N = varlen ? num_seqs : B;
    const bool have_tokens = (int64_t)B * T > 0;
    if (have_tokens && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_INVALID_ARG;
    const void *ptrs16[] = {q, k, v, init_state, out, final_state};
    for (const void *p : ptrs16)
        if (p && !aligned16(p)) return GDN_ERR_INVALID_ARG;
    const void *ptrs4[] = {g, beta, cu_seqlens};
    for (const void *p : ptrs4)
        if (p && !aligned_to(p, 4)) return GDN_ERR_INVALID_ARG;
    if (!workspace) return GDN_ERR_WORKSPACE;
    if (((uintptr_t)workspace & 255u) != 0) return GDN_ERR_WORKSPACE;
    const size_t need = gdn_chunk_fwd_workspace_size(B, T, H, dk, dv, varlen ? num_seqs : 0, dt);
    if (need == 0) return GDN_ERR_INVALID_ARG;
    if (workspace_bytes < need) return GDN_ERR_WORKSPACE;

    ChunkArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.init_state = init_state;
    a.out = out; a.final_state = final_state;
    a.gm.B = B; a.gm.T = T; a.gm.H = H; a.gm.dk = dk; a.gm.dv = dv; a.gm.N = N;
    a.gm.cu = cu_seqlens;
    a.gm.nct = ceil_div(T, kChunk);
    a.slots = have_tokens ? num_slots(B, T, N, varlen) : 0;
    a.dt = (dt == GDN_BF16) ? 1 : 0;
    a.scale = scale;
    a.l2 = use_qk_l2norm ? 1 : 0;
    a.workspace = workspace;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = chunk_tc_supported(a.dt, dk, dv, (int64_t)B * T) ? launch_chunk_tc(a, st)
                                                                     : launch_chunk_simt(a, st);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

size_t gdn_chunk_bwd_workspace_size(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv,
                                    int32_t num_seqs, gdn_dtype dt)
{
    if (B < 1 || T < 0 || H < 1 || num_seqs < 0) return 0;
    if (dt != GDN_F32 && dt != GDN_BF16) return 0;
    if (!bwd_dims_supported(dk, dv)) return 0;
    const bool varlen = num_seqs > 0;
    if (varlen && B != 1) return 0;
    return chunk_bwd_workspace_bytes(num_slots(B, T, varlen ? num_seqs : B, varlen), H, dk, dv);
}

gdn_status gdn_chunk_bwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                         const float *init_state, const int32_t *cu_seqlens, int32_t num_seqs,
                         const void *dout, const float *dfinal_state,
                         void *dq, void *dk_, void *dv_, float *dg, float *dbeta, float *dinit_state,
                         int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, gdn_dtype dt, float scale,
                         int32_t use_qk_l2norm, int32_t chunk_size, void *workspace, size_t workspace_bytes,
                         void *stream)
{
    if (B < 1 || T < 0 || H < 1 || dk < 1 || dv < 1) return GDN_ERR_INVALID_ARG;
    if (dt != GDN_F32 && dt != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (chunk_size != kChunk) return GDN_ERR_UNSUPPORTED;
    if (!bwd_dims_supported(dk, dv)) return GDN_ERR_UNSUPPORTED;
    const bool varlen = cu_seqlens != nullptr;
    if (varlen && (B != 1 || num_seqs < 1)) return GDN_ERR_INVALID_ARG;
    if (!varlen && num_seqs != 0 && num_seqs != B) return GDN_ERR_INVALID_ARG;
    const int N = varlen ? num_seqs : B;
    const bool have_tokens = (int64_t)B * T > 0;
    if (have_tokens && (!q || !k || !v || !g || !beta || !dout || !dq || !dk_ || !dv_ || !dg || !dbeta))
        return GDN_ERR_INVALID_ARG;
    const void *ptrs16[] = {q, k, v, init_state, dout, dfinal_state, dq, dk_, dv_, dinit_state};
    for (const void *p : ptrs16)
        if (p && !aligned16(p)) return GDN_ERR_INVALID_ARG;
    const void *ptrs4[] = {g, beta, cu_seqlens, dg, dbeta};
    for (const void *p : ptrs4)
        if (p && !aligned_to(p, 4)) return GDN_ERR_INVALID_ARG;
    if (!workspace || ((uintptr_t)workspace & 255u) != 0) return GDN_ERR_WORKSPACE;
    const size_t need = gdn_chunk_bwd_workspace_size(B, T, H, dk, dv, varlen ? num_seqs : 0, dt);
    if (need == 0) return GDN_ERR_INVALID_ARG;
    if (workspace_bytes < need) return GDN_ERR_WORKSPACE;

    BwdArgs a;
    a.q = q; a.k = k; a.v = v; a.dout = dout; a.g = g; a.beta = beta;
    a.init_state = init_state; a.dfinal = dfinal_state;
    a.dq = dq; a.dk = dk_; a.dv = dv_; a.dg = dg; a.dbeta = dbeta; a.dinit = dinit_state;
    a.gm.B = B; a.gm.T = T; a.gm.H = H; a.gm.dk = dk; a.gm.dv = dv; a.gm.N = N;
    a.gm.cu = cu_seqlens;
    a.gm.nct = ceil_div(T, kChunk);
    a.slots = have_tokens ? num_slots(B, T, N, varlen) : 0;
    a.dt = (dt == GDN_BF16) ? 1 : 0;
    a.scale = scale;
    a.l2 = use_qk_l2norm ? 1 : 0;
    a.workspace = workspace;
    cudaError_t e = launch_chunk_bwd(a, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

static gdn_status decode_common(float *state, const void *q, const void *k, const void *v, const float *g,
                                const float *beta, void *out, int32_t N, int32_t T, int32_t H, int32_t dk,
                                int32_t dv, gdn_dtype dt, float scale, int32_t use_qk_l2norm, void *stream)
{
    if (N < 0 || T < 0 || H < 1 || dk < 1 || dv < 1) return GDN_ERR_INVALID_ARG;
    if (dt != GDN_F32 && dt != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (!(dk == 64 || dk == 128 || dk == 256) || dv % 8 != 0) return GDN_ERR_UNSUPPORTED;
    if (N == 0 || T == 0) return GDN_OK;
    if ((int64_t)N * T * H * (dk > dv ? dk : dv) >= ((int64_t)1 << 62)) return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {state, q, k, v, g, beta, out};
    for (const void *p : ptrs)
        if (!p) return GDN_ERR_INVALID_ARG;
    const unsigned esz = (dt == GDN_BF16) ? 2u : 4u;
    if (!aligned16(state) || !aligned_to(q, esz) || !aligned_to(k, esz) || !aligned_to(v, esz) ||
        !aligned_to(out, esz) || !aligned_to(g, 4) || !aligned_to(beta, 4))
        return GDN_ERR_INVALID_ARG;
    DecodeArgs a;
    a.state = state; a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.out = out;
    a.N = N; a.H = H; a.dk = dk; a.dv = dv; a.dt = (dt == GDN_BF16) ? 1 : 0;
    a.ntok = T;
    a.scale = scale; a.l2 = use_qk_l2norm ? 1 : 0;
    cudaError_t e = launch_decode(a, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_decode_step(float *state, const void *q, const void *k, const void *v,
                           const float *g, const float *beta, void *out, int32_t N, int32_t H,
                           int32_t dk, int32_t dv, gdn_dtype dt, float scale,
                           int32_t use_qk_l2norm, void *stream)
{
    return decode_common(state, q, k, v, g, beta, out, N, 1, H, dk, dv, dt, scale, use_qk_l2norm, stream);
}

gdn_status gdn_decode_multi(float *state, const void *q, const void *k, const void *v,
                            const float *g, const float *beta, void *out, int32_t N, int32_t T,
                            int32_t H, int32_t dk, int32_t dv, gdn_dtype dt, float scale,
                            int32_t use_qk_l2norm, void *stream)
{
    return decode_common(state, q, k, v, g, beta, out, N, T, H, dk, dv, dt, scale, use_qk_l2norm, stream);
}

gdn_status gdn_prologue(const void *xq, const void *xk, const void *xv, const float *wq, const float *wk,
                        const float *wv, const float *a, const float *b, const float *A_log,
                        const float *dt_bias, const void *conv_state_in, void *conv_state_out,
                        const int32_t *cu_seqlens, int32_t num_seqs, void *q, void *k, void *v, float *g,
                        float *beta, int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv, int32_t K,
                        gdn_dtype dt, void *stream)
{
    if (B < 1 || T < 0 || H < 1 || dk < 1 || dv < 1) return GDN_ERR_INVALID_ARG;
    if (dt != GDN_F32 && dt != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (K < 1 || K > 4 || dk % 8 != 0 || dv % 8 != 0 || dk > 256 || dv > 256) return GDN_ERR_UNSUPPORTED;
    const bool varlen = cu_seqlens != nullptr;
    if (varlen && (B != 1 || num_seqs < 1)) return GDN_ERR_INVALID_ARG;
    if (!varlen && num_seqs != 0 && num_seqs != B) return GDN_ERR_INVALID_ARG;
    const int N = varlen ? num_seqs : B;
    if ((int64_t)B * T * H >= ((int64_t)1 << 40)) return GDN_ERR_INVALID_ARG;
    const bool have_tokens = (int64_t)B * T > 0;
    if (have_tokens) {
        const void *need[] = {xq, xk, xv, wq, wk, wv, a, b, A_log, dt_bias, q, k, v, g, beta};
        for (const void *p : need)
            if (!p) return GDN_ERR_INVALID_ARG;
    }
    const void *al16[] = {xq, xk, xv, q, k, v, conv_state_in, conv_state_out};
    for (const void *p : al16)
        if (p && !aligned16(p)) return GDN_ERR_INVALID_ARG;
    const void *al4[] = {wq, wk, wv, a, b, A_log, dt_bias, g, beta, cu_seqlens};
    for (const void *p : al4)
        if (p && !aligned_to(p, 4)) return GDN_ERR_INVALID_ARG;
    if (conv_state_in && conv_state_out && K > 1) {   // the two state buffers must not overlap
        const size_t bytes = (size_t)N * (K - 1) * H * (2 * dk + dv) * (dt == GDN_BF16 ? 2 : 4);
        const uintptr_t i0 = (uintptr_t)conv_state_in, o0 = (uintptr_t)conv_state_out;
        if (i0 < o0 + bytes && o0 < i0 + bytes) return GDN_ERR_INVALID_ARG;
    }
    if (!have_tokens && !conv_state_out) return GDN_OK;
    PrologueArgs pa;
    pa.xq = xq; pa.xk = xk; pa.xv = xv; pa.wq = wq; pa.wk = wk; pa.wv = wv;
    pa.a = a; pa.b = b; pa.A_log = A_log; pa.dt_bias = dt_bias;
    pa.state_in = K > 1 ? conv_state_in : nullptr;
    pa.state_out = K > 1 ? conv_state_out : nullptr;
    pa.cu = cu_seqlens;
    pa.q = q; pa.k = k; pa.v = v; pa.g = g; pa.beta = beta;
    pa.B = B; pa.T = T; pa.H = H; pa.dk = dk; pa.dv = dv; pa.N = N; pa.K = K;
    pa.dt = (dt == GDN_BF16) ? 1 : 0;
    cudaError_t e = launch_prologue(pa, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_selftest_wait_timeout(void *workspace, uint32_t limit_us, void *stream)
{
    if (!workspace || ((uintptr_t)workspace & 255u) != 0) return GDN_ERR_INVALID_ARG;
    if (limit_us < 1 || limit_us > 1000000u) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(workspace, 0, sizeof(unsigned), st) != cudaSuccess) return GDN_ERR_CUDA;
    cudaError_t e = launch_wait_selftest(reinterpret_cast<unsigned *>(workspace), (uint64_t)limit_us * 1000u, st);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

size_t gdn_prologue_chunk_fwd_workspace_size(int32_t B, int32_t T, int32_t H, int32_t dk, int32_t dv,
                                             int32_t num_seqs, gdn_dtype dt)
{
    if (B < 1 || T < 0 || H < 1 || num_seqs < 0) return 0;
    if (dt != GDN_BF16 || !chunk_tc_supported(1, dk, dv, 1)) return 0;
    const bool varlen = num_seqs > 0;
    if (varlen && B != 1) return 0;
    const int64_t slots = (int64_t)B * T > 0 ? num_slots(B, T, varlen ? num_seqs : B, varlen) : 0;
    return chunk_tc_workspace_bytes(slots, H, true);
}

gdn_status gdn_prologue_chunk_fwd(const void *xq, const void *xk, const void *xv, const float *wq,
                                  const float *wk, const float *wv, const float *a, const float *b,
                                  const float *A_log, const float *dt_bias, const void *conv_state_in,
                                  void *conv_state_out, const float *init_state, const int32_t *cu_seqlens,
                                  int32_t num_seqs, void *out, float *final_state, int32_t B, int32_t T,
                                  int32_t H, int32_t dk, int32_t dv, int32_t K, gdn_dtype dt, float scale,
                                  int32_t use_qk_l2norm, int32_t chunk_size, void *workspace,
                                  size_t workspace_bytes, void *stream)
{
    if (B < 1 || T < 0 || H < 1 || dk < 1 || dv < 1) return GDN_ERR_INVALID_ARG;
    if (dt != GDN_F32 && dt != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (chunk_size != kChunk) return GDN_ERR_UNSUPPORTED;
    if (dt != GDN_BF16 || !chunk_tc_supported(1, dk, dv, 1) || K < 1 || K > 4) return GDN_ERR_UNSUPPORTED;
    const bool varlen = cu_seqlens != nullptr;
    if (varlen && (B != 1 || num_seqs < 1)) return GDN_ERR_INVALID_ARG;
    if (!varlen && num_seqs != 0 && num_seqs != B) return GDN_ERR_INVALID_ARG;
    const int N = varlen ? num_seqs : B;
    const int64_t tokens = (int64_t)B * T;
    if (tokens >= ((int64_t)1 << 31)) return GDN_ERR_INVALID_ARG;
    const bool have_tokens = tokens > 0;
    if (have_tokens) {
        const void *need[] = {xq, xk, xv, wq, wk, wv, a, b, A_log, dt_bias, out};
        for (const void *p : need)
            if (!p) return GDN_ERR_INVALID_ARG;
    }
    const void *al16[] = {xq, xk, xv, out, init_state, final_state, conv_state_in, conv_state_out};
    for (const void *p : al16)
        if (p && !aligned16(p)) return GDN_ERR_INVALID_ARG;
    const void *al4[] = {wq, wk, wv, a, b, A_log, dt_bias, cu_seqlens};
    for (const void *p : al4)
        if (p && !aligned_to(p, 4)) return GDN_ERR_INVALID_ARG;
    if (conv_state_in && conv_state_out && K > 1) {   // the two state buffers must not overlap
        const size_t bytes = (size_t)N * (K - 1) * H * (2 * dk + dv) * 2;
        const uintptr_t i0 = (uintptr_t)conv_state_in, o0 = (uintptr_t)conv_state_out;
        if (i0 < o0 + bytes && o0 < i0 + bytes) return GDN_ERR_INVALID_ARG;
    }
    if (!workspace || ((uintptr_t)workspace & 255u) != 0) return GDN_ERR_WORKSPACE;
    const size_t need = gdn_prologue_chunk_fwd_workspace_size(B, T, H, dk, dv, varlen ? num_seqs : 0, dt);
    if (need == 0) return GDN_ERR_INVALID_ARG;
    if (workspace_bytes < need) return GDN_ERR_WORKSPACE;

    PrologueArgs pa;
    pa.xq = xq; pa.xk = xk; pa.xv = xv; pa.wq = wq; pa.wk = wk; pa.wv = wv;
    pa.a = a; pa.b = b; pa.A_log = A_log; pa.dt_bias = dt_bias;
    pa.state_in = K > 1 ? conv_state_in : nullptr;
    pa.state_out = K > 1 ? conv_state_out : nullptr;
    pa.cu = cu_seqlens;
    pa.q = nullptr; pa.k = nullptr; pa.v = nullptr; pa.g = nullptr; pa.beta = nullptr;
    pa.B = B; pa.T = T; pa.H = H; pa.dk = dk; pa.dv = dv; pa.N = N; pa.K = K;
    pa.dt = 1;
    ChunkArgs ca;
    ca.q = nullptr; ca.k = nullptr; ca.v = nullptr; ca.g = nullptr; ca.beta = nullptr;
    ca.init_state = init_state; ca.out = out; ca.final_state = final_state;
    ca.gm.B = B; ca.gm.T = T; ca.gm.H = H; ca.gm.dk = dk; ca.gm.dv = dv; ca.gm.N = N;
    ca.gm.cu = cu_seqlens;
    ca.gm.nct = ceil_div(T, kChunk);
    ca.slots = have_tokens ? num_slots(B, T, N, varlen) : 0;
    ca.dt = 1;
    ca.scale = scale;
    ca.l2 = use_qk_l2norm ? 1 : 0;
    ca.workspace = workspace;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e;
    if (!have_tokens) {
        // nothing to transform: the states pass through (the prologue kernel carries the
        // convolution state of empty sequences; the CUDA-core path copies init to final)
        e = pa.state_out ? launch_prologue(pa, st) : cudaSuccess;
        if (e == cudaSuccess) e = launch_chunk_simt(ca, st);
    } else {
        ca.fuse = &pa;
        e = launch_chunk_tc(ca, st);
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

gdn_status gdn_check_device_error(void *workspace, void *stream)
{
    if (!workspace || ((uintptr_t)workspace & 255u) != 0) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    unsigned word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ERR_CUDA;
    if (word == kDevErrNone) return GDN_OK;
    if (cudaMemsetAsync(workspace, 0, sizeof(word), st) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ERR_CUDA;
    if (word == kDevErrTimeout) return GDN_ERR_DEVICE_TIMEOUT;
    if (word == kDevErrRange) return GDN_ERR_RANGE;
    return GDN_ERR_CUDA;
}

}  // extern "C"
