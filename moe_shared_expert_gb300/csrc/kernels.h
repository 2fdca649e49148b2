// Internal launch interfaces between the C-ABI layer (api.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace mse {

// ---------------------------------------------------------------- generic path
// C[m, n] = sum_k A[m, k] * B[n, k] for one group g = blockIdx.z, with A, B, out
// advanced by g * {a,b,o}_gstride elements.  Any shape, any alignment.
enum SimtMode : int {
    SIMT_SWIGLU = 0,   // out bf16 = bf16(silu(A.B^T) * (A.B2^T))
    SIMT_BF16 = 1,     // out bf16
    SIMT_F32 = 2,      // out fp32
    SIMT_MERGED = 3,   // out bf16 to logical (out) and/or rank-major (out_rm)
};

struct SimtGemmArgs {
    const uint16_t *A; int64_t lda; int64_t a_gstride;
    const uint16_t *B; int64_t ldb; int64_t b_gstride;
    const uint16_t *B2;               // SWIGLU only: up rows, same ldb/b_gstride
    int64_t M, N, K;
    int groups;
    void *out; int64_t ldo; int64_t o_gstride;
    uint16_t *out_rm;                 // MERGED only (nullable)
    int64_t q_dim, kv_dim; int tp;    // MERGED only
    int mode;
};
cudaError_t launch_simt_gemm(const SimtGemmArgs &a, cudaStream_t s);

// ---------------------------------------------------------------- elementwise
// pdl: launched with programmatic dependent launch (waits for its predecessor in-kernel)
cudaError_t launch_shard_sum(const void *partials, int dtype_f32, int n_parts, int64_t plane, uint16_t *out,
                             int sm_count, bool pdl, cudaStream_t s);
cudaError_t launch_reorder(const uint16_t *rm, uint16_t *logical, int64_t T, int64_t q_dim, int64_t kv_dim, int tp,
                           bool pdl, cudaStream_t s);
cudaError_t launch_wait_selftest(uint64_t limit_ns, uint32_t *err, cudaStream_t s);
// Copy of activations from host (device-mapped) to device memory, with programmatic
// dependent launch; `early`: the source is read before waiting for the previous kernel.
cudaError_t launch_copy_in(const void *src, void *dst, int64_t bytes, bool early, int sm_count, cudaStream_t s);

}  // namespace mse
