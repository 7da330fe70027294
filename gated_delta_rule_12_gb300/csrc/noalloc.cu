// noalloc.cu -- gdn_chunk_fwd_noalloc: the chunked forward pass for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they run the operator: plugin hosts and serving runtimes that
// plan every device byte up front and forbid allocation on the request path,
// and bindings that have no device allocator of their own.  They also cannot
// hand the library a workspace.  For them this entry point runs the CUDA-core
// chunked forward kernels (prologue, UT transform, recurrence) with their
// scratch in a fixed array that is part of this library's device image.
//
// The array:
//   - is kNoAllocScratchBytes (32 MiB) per GPU, allocated by the CUDA runtime
//     when the library's device code is loaded on a GPU and held by every GPU
//     that loads it until the process exits;
//   - is shared by every call on that GPU and keeps the previous call's
//     contents; the only part that must start at zero (the device error word
//     in its first 256 bytes) is cleared by the first kernel of every call,
//     and every other byte a kernel reads is written earlier in the same call;
//   - is one buffer per GPU, so calls that overlap on the GPU (different
//     streams, or different host threads) race on it: callers must order them.
// Host code cannot use the array's name as a device address (it names a
// host-side stand-in), so every call looks the address up with
// cudaGetSymbolAddress while the call's device is current.  A device reset
// (cudaDeviceReset) unloads the module and the array may come back at another
// address; looking it up on every call keeps the address current.  While the
// caller's stream is being captured into a graph the lookup is skipped and the
// address found by the last call on that device outside a capture is used, so
// at least one call on each device (after any device reset) must come before
// a capture.
#include <mutex>
#include <stdint.h>

#include "../../include/gdn.h"
#include "common.cuh"
#include "kernels.h"

using namespace gdn;

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)GDN_NOALLOC_SCRATCH_BYTES;
static_assert(kNoAllocScratchBytes == (32u << 20), "header and array disagree on the scratch size");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices];   // last looked-up device address of g_noalloc_scratch, per device

// The device address of the scratch array on the current device.  Outside a
// stream capture it is looked up afresh (cudaGetSymbolAddress, which neither
// allocates nor enqueues work), so it follows a device reset; during a capture
// of `stream` the last address found on this device is reused.  Returns nullptr
// on failure.
void *scratch_on_current_device(cudaStream_t stream, cudaError_t *err)
{
    int dev = -1;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) { *err = cudaErrorInvalidDevice; return nullptr; }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    *err = cudaStreamIsCapturing(stream, &cs);
    if (*err != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (cs == cudaStreamCaptureStatusNone || !g_scratch_addr[dev]) {
        void *p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (*err != cudaSuccess || !p) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

bool aligned_to(const void *p, unsigned a) { return ((uintptr_t)p & (uintptr_t)(a - 1)) == 0; }

}  // namespace

extern "C" gdn_status gdn_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *g,
                                            const float *beta, const float *init_state,
                                            const int32_t *cu_seqlens, int32_t num_seqs, void *out,
                                            float *final_state, int32_t B, int32_t T, int32_t H, int32_t dk,
                                            int32_t dv, gdn_dtype dt, float scale, int32_t use_qk_l2norm,
                                            int32_t chunk_size, void *stream)
{
    if (B < 1 || T < 0 || H < 1 || dk < 1 || dv < 1) return GDN_ERR_INVALID_ARG;
    if (dt != GDN_F32 && dt != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (chunk_size != kChunk) return GDN_ERR_UNSUPPORTED;
    if (!((dk == 64 || dk == 128 || dk == 256) && dv >= 32 && dv <= 256 && dv % 32 == 0)) return GDN_ERR_UNSUPPORTED;
    const bool varlen = cu_seqlens != nullptr;
    if (varlen && (B != 1 || num_seqs < 1)) return GDN_ERR_INVALID_ARG;
    if (!varlen && num_seqs != 0 && num_seqs != B) return GDN_ERR_INVALID_ARG;
    const int N = varlen ? num_seqs : B;
    const bool have_tokens = (int64_t)B * T > 0;
    if (have_tokens && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_INVALID_ARG;
    const void *ptrs16[] = {q, k, v, init_state, out, final_state};
    for (const void *p : ptrs16)
        if (p && !aligned_to(p, 16)) return GDN_ERR_INVALID_ARG;
    const void *ptrs4[] = {g, beta, cu_seqlens};
    for (const void *p : ptrs4)
        if (p && !aligned_to(p, 4)) return GDN_ERR_INVALID_ARG;

    const int64_t slots = have_tokens ? num_slots(B, T, N, varlen) : 0;
    const size_t need = chunk_workspace_layout(slots, H, dk, dv).total;
    if (need > kNoAllocScratchBytes) return GDN_ERR_WORKSPACE;   // problem too large for the fixed array

    cudaError_t e = cudaSuccess;
    void *scratch = scratch_on_current_device((cudaStream_t)stream, &e);
    if (!scratch) return GDN_ERR_CUDA;

    ChunkArgs a;
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.init_state = init_state;
    a.out = out; a.final_state = final_state;
    a.gm.B = B; a.gm.T = T; a.gm.H = H; a.gm.dk = dk; a.gm.dv = dv; a.gm.N = N;
    a.gm.cu = cu_seqlens;
    a.gm.nct = ceil_div(T, kChunk);
    a.slots = slots;
    a.dt = (dt == GDN_BF16) ? 1 : 0;
    a.scale = scale;
    a.l2 = use_qk_l2norm ? 1 : 0;
    a.workspace = scratch;
    e = launch_chunk_simt(a, (cudaStream_t)stream);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
