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

bool chunk_dims_supported(int dk, int dv) { return (dk == 64 || dk == 128) && dv >= 32 && dv <= 256 && dv % 32 == 0; }

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
    return word == kDevErrTimeout ? GDN_ERR_DEVICE_TIMEOUT : GDN_ERR_CUDA;
}

}  // extern "C"
