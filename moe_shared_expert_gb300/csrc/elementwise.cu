// HBM-bound elementwise kernels: the sum of shard partials and the
// rank-major -> logical reorder of the merged latent projection; plus the
// bounded-wait self test.
#include "common.cuh"
#include "kernels.h"

namespace mse {
namespace {

// out[e] = bf16( sum_{r ascending} p[r*plane + e] ), fp32 accumulate, 8 bf16 per thread-step.
__global__ void __launch_bounds__(256) shard_sum_bf16_vec(const uint4 *__restrict__ p, int n_parts, int64_t plane8,
                                                          uint4 *__restrict__ out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < plane8;
         i += (int64_t)gridDim.x * blockDim.x) {
        float acc[8] = {};
        for (int r = 0; r < n_parts; ++r) {
            const uint4 v = __ldcs(p + r * plane8 + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                acc[2 * k] += __uint_as_float(w[k] << 16);
                acc[2 * k + 1] += __uint_as_float(w[k] & 0xFFFF0000u);
            }
        }
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            o[k] = (uint32_t)f32_to_bf16_bits(acc[2 * k]) | ((uint32_t)f32_to_bf16_bits(acc[2 * k + 1]) << 16);
        out[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__global__ void __launch_bounds__(256) shard_sum_f32_vec(const float4 *__restrict__ p, int n_parts, int64_t plane4,
                                                         uint2 *__restrict__ out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < plane4;
         i += (int64_t)gridDim.x * blockDim.x) {
        float acc[4] = {};
        for (int r = 0; r < n_parts; ++r) {
            const float4 v = __ldcs(p + r * plane4 + i);
            acc[0] += v.x; acc[1] += v.y; acc[2] += v.z; acc[3] += v.w;
        }
        out[i] = make_uint2((uint32_t)f32_to_bf16_bits(acc[0]) | ((uint32_t)f32_to_bf16_bits(acc[1]) << 16),
                            (uint32_t)f32_to_bf16_bits(acc[2]) | ((uint32_t)f32_to_bf16_bits(acc[3]) << 16));
    }
}

__global__ void __launch_bounds__(256) shard_sum_scalar(const void *__restrict__ p, int is_f32, int n_parts,
                                                        int64_t plane, uint16_t *__restrict__ out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < plane;
         i += (int64_t)gridDim.x * blockDim.x) {
        float acc = 0.f;
        for (int r = 0; r < n_parts; ++r)
            acc += is_f32 ? static_cast<const float *>(p)[r * plane + i]
                          : bf16_bits_to_f32(static_cast<const uint16_t *>(p)[r * plane + i]);
        out[i] = f32_to_bf16_bits(acc);
    }
}

// logical[t, c] = rank_major[t, gathered(c)]; one thread per output word.
__global__ void __launch_bounds__(256) reorder_kernel(const uint16_t *__restrict__ rm, uint16_t *__restrict__ lo,
                                                      int64_t T, int64_t C, int64_t q_dim, int64_t qs, int64_t ks) {
    const int64_t total = T * C, w = qs + ks;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = e / C, c = e % C;
        int64_t g;
        if (c < q_dim) {
            g = (c / qs) * w + (c % qs);
        } else {
            const int64_t c2 = c - q_dim;
            g = (c2 / ks) * w + qs + (c2 % ks);
        }
        lo[e] = rm[t * C + g];
    }
}

// One CTA waits on a barrier that nothing arrives on, bounded by limit_ns.
__global__ void wait_selftest_kernel(uint64_t limit_ns, uint32_t *err) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(smem_u32(&bar), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, limit_ns, err);
    __syncthreads();
}

}  // namespace

cudaError_t launch_shard_sum(const void *partials, int dtype_f32, int n_parts, int64_t plane, uint16_t *out,
                             int sm_count, cudaStream_t s) {
    if (plane <= 0) return cudaSuccess;
    const int blocks_cap = sm_count * 8;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(partials), oa = reinterpret_cast<uintptr_t>(out);
    if (!dtype_f32 && plane % 8 == 0 && pa % 16 == 0 && oa % 16 == 0) {
        const int64_t n = plane / 8;
        const int blocks = (int)std::min<int64_t>((n + 255) / 256, blocks_cap);
        shard_sum_bf16_vec<<<blocks, 256, 0, s>>>(static_cast<const uint4 *>(partials), n_parts, n,
                                                  reinterpret_cast<uint4 *>(out));
    } else if (dtype_f32 && plane % 4 == 0 && pa % 16 == 0 && oa % 8 == 0) {
        const int64_t n = plane / 4;
        const int blocks = (int)std::min<int64_t>((n + 255) / 256, blocks_cap);
        shard_sum_f32_vec<<<blocks, 256, 0, s>>>(static_cast<const float4 *>(partials), n_parts, n,
                                                 reinterpret_cast<uint2 *>(out));
    } else {
        const int blocks = (int)std::min<int64_t>((plane + 255) / 256, blocks_cap);
        shard_sum_scalar<<<blocks, 256, 0, s>>>(partials, dtype_f32, n_parts, plane, out);
    }
    return cudaGetLastError();
}

cudaError_t launch_reorder(const uint16_t *rm, uint16_t *logical, int64_t T, int64_t q_dim, int64_t kv_dim, int tp,
                           cudaStream_t s) {
    const int64_t C = q_dim + kv_dim, total = T * C;
    if (total <= 0) return cudaSuccess;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, 4096);
    reorder_kernel<<<blocks, 256, 0, s>>>(rm, logical, T, C, q_dim, q_dim / tp, kv_dim / tp);
    return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, uint32_t *err, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, err);
    return cudaGetLastError();
}

}  // namespace mse
