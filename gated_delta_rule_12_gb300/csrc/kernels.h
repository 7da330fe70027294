// kernels.h -- internal launcher interface between the C ABI (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace gdn {

struct PrologueArgs;

struct ChunkArgs {
    const void *q, *k, *v;
    const float *g, *beta, *init_state;
    void *out;
    float *final_state;
    Geometry gm;
    int64_t slots;
    int dt;          // 0 = fp32, 1 = bf16
    float scale;
    int l2;
    void *workspace;
    const PrologueArgs *fuse = nullptr;   // non-null: q, k, v, g, beta are made from these projections
    // Tensor-core path, for the backward pass: chunk-local blocks at blocks + (slot * H + h) * block_stride
    // (instead of after the workspace header), and the chunk-start states and V_new saved (see RcParams).
    void *blocks = nullptr;
    size_t block_stride = 0;
    float *save_s = nullptr, *save_vn = nullptr;
    int64_t save_stride = 0;
};

struct DecodeArgs {
    float *state;
    const void *q, *k, *v;
    const float *g, *beta;
    void *out;
    int N, H, dk, dv, dt;
    int ntok;        // tokens per sequence in this call (1 = single step)
    float scale;
    int l2;
};

struct PrologueArgs {
    const void *xq, *xk, *xv;                 // raw projections [B, T, H, dk|dk|dv], dtype dt
    const float *wq, *wk, *wv;                // convolution filters [H, d, K]
    const float *a, *b, *A_log, *dt_bias;     // gate projections [B, T, H]; per-head parameters [H]
    const void *state_in;                     // [N, K-1, H, 2 dk + dv] dtype dt, or null
    void *state_out;                          // same layout, or null
    const int32_t *cu;                        // [N + 1] or null
    void *q, *k, *v;                          // outputs [B, T, H, dk|dk|dv], dtype dt
    float *g, *beta;                          // outputs [B, T, H]
    int B, T, H, dk, dv, N, K, dt;
};

struct BwdArgs {
    const void *q, *k, *v, *dout;            // dtype dt
    const float *g, *beta, *init_state, *dfinal;
    void *dq, *dk, *dv;                      // dtype dt
    float *dg, *dbeta, *dinit;
    Geometry gm;
    int64_t slots;
    int dt;
    float scale;
    int l2;
    void *workspace;
};

cudaError_t launch_chunk_simt(const ChunkArgs &a, cudaStream_t st);
cudaError_t launch_chunk_bwd(const BwdArgs &a, cudaStream_t st);
size_t chunk_bwd_workspace_bytes(int64_t slots, int H, int dk, int dv);
cudaError_t launch_prologue(const PrologueArgs &a, cudaStream_t st);
bool chunk_tc_supported(int dt, int dk, int dv, int64_t tokens);
size_t chunk_tc_workspace_bytes(int64_t slots, int H, bool fused = false);
cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t st);
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st);
// one CTA whose bounded wait on a never-completed mbarrier phase gives up after limit_ns
cudaError_t launch_wait_selftest(unsigned *err, uint64_t limit_ns, cudaStream_t st);

}  // namespace gdn
