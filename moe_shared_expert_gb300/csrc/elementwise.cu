// HBM-bound elementwise kernels: the sum of shard partials and the
// rank-major -> logical reorder of the merged latent projection; plus the
// bounded-wait self test.
#include "common.cuh"
#include "kernels.h"

namespace mse {
namespace {

// out[e] = bf16( sum_{r ascending} p[r*plane + e] ), fp32 accumulate, 8 bf16 per thread-step.
// The parts' loads are requested in batches of kPartBatch before any is summed, so a
// thread waits for one DRAM round trip per batch, not one per part.
constexpr int kPartBatch = 8;

__global__ void __launch_bounds__(256) shard_sum_bf16_vec(const uint4 *__restrict__ p, int n_parts, int64_t plane8,
                                                          uint4 *__restrict__ out) {
    pdl_launch_dependents();   // the next kernel may start fetching its weights
    pdl_wait();                // inputs written by the previous kernel
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < plane8;
         i += (int64_t)gridDim.x * blockDim.x) {
        float acc[8] = {};
        for (int r0 = 0; r0 < n_parts; r0 += kPartBatch) {
            uint4 v[kPartBatch];
#pragma unroll
            for (int b = 0; b < kPartBatch; ++b)
                if (r0 + b < n_parts) v[b] = __ldcs(p + (int64_t)(r0 + b) * plane8 + i);
#pragma unroll
            for (int b = 0; b < kPartBatch; ++b) {
                if (r0 + b < n_parts) {
                    const uint32_t w[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        acc[2 * k] += __uint_as_float(w[k] << 16);
                        acc[2 * k + 1] += __uint_as_float(w[k] & 0xFFFF0000u);
                    }
                }
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
    pdl_launch_dependents();   // the next kernel may start fetching its weights
    pdl_wait();                // inputs written by the previous kernel
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < plane4;
         i += (int64_t)gridDim.x * blockDim.x) {
        float acc[4] = {};
        for (int r0 = 0; r0 < n_parts; r0 += kPartBatch) {
            float4 v[kPartBatch];
#pragma unroll
            for (int b = 0; b < kPartBatch; ++b)
                if (r0 + b < n_parts) v[b] = __ldcs(p + (int64_t)(r0 + b) * plane4 + i);
#pragma unroll
            for (int b = 0; b < kPartBatch; ++b) {
                if (r0 + b < n_parts) {
                    acc[0] += v[b].x; acc[1] += v[b].y; acc[2] += v[b].z; acc[3] += v[b].w;
                }
            }
        }
        out[i] = make_uint2((uint32_t)f32_to_bf16_bits(acc[0]) | ((uint32_t)f32_to_bf16_bits(acc[1]) << 16),
                            (uint32_t)f32_to_bf16_bits(acc[2]) | ((uint32_t)f32_to_bf16_bits(acc[3]) << 16));
    }
}

__global__ void __launch_bounds__(256) shard_sum_scalar(const void *__restrict__ p, int is_f32, int n_parts,
                                                        int64_t plane, uint16_t *__restrict__ out) {
    pdl_launch_dependents();   // the next kernel may start fetching its weights
    pdl_wait();                // inputs written by the previous kernel
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
    pdl_launch_dependents();   // the next kernel may start fetching its weights
    pdl_wait();                // inputs written by the previous kernel
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

// Copy of activations from host memory (device-mapped) to device memory, launched with
// programmatic dependent launch.  It waits for the previous kernel before writing (the
// destination may still be read by it).  With `early`, each thread reads its first
// kCopyPer 16-byte words before that wait (the caller knows that the previous work on
// the stream does not write the source); else it reads after the wait too.
constexpr int kCopyPer = 4;

__global__ void __launch_bounds__(256) copy_in_vec(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int64_t n,
                                                   int early) {
    pdl_launch_dependents();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint4 v[kCopyPer];
    if (early) {
#pragma unroll
        for (int k = 0; k < kCopyPer; ++k)
            if (i0 + k * stride < n) v[k] = src[i0 + k * stride];
    }
    pdl_wait();
    if (!early) {
#pragma unroll
        for (int k = 0; k < kCopyPer; ++k)
            if (i0 + k * stride < n) v[k] = src[i0 + k * stride];
    }
#pragma unroll
    for (int k = 0; k < kCopyPer; ++k)
        if (i0 + k * stride < n) dst[i0 + k * stride] = v[k];
    for (int64_t i = i0 + kCopyPer * stride; i < n; i += stride) dst[i] = src[i];
}

__global__ void __launch_bounds__(256) copy_in_bytes(const unsigned char *__restrict__ src,
                                                     unsigned char *__restrict__ dst, int64_t n) {
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
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

// Launch with programmatic dependent launch when `pdl` (the kernels wait for their
// predecessor before reading and let their successor start early).
template <typename... KArgs, typename... Args>
cudaError_t launch_ew(void (*kern)(KArgs...), int blocks, bool pdl, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

cudaError_t launch_shard_sum(const void *partials, int dtype_f32, int n_parts, int64_t plane, uint16_t *out,
                             int sm_count, bool pdl, cudaStream_t s) {
    if (plane <= 0) return cudaSuccess;
    const int blocks_cap = sm_count * 8;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(partials), oa = reinterpret_cast<uintptr_t>(out);
    if (!dtype_f32 && plane % 8 == 0 && pa % 16 == 0 && oa % 16 == 0) {
        const int64_t n = plane / 8;
        const int blocks = (int)std::min<int64_t>((n + 255) / 256, blocks_cap);
        return launch_ew(shard_sum_bf16_vec, blocks, pdl, s, static_cast<const uint4 *>(partials), n_parts, n,
                         reinterpret_cast<uint4 *>(out));
    } else if (dtype_f32 && plane % 4 == 0 && pa % 16 == 0 && oa % 8 == 0) {
        const int64_t n = plane / 4;
        const int blocks = (int)std::min<int64_t>((n + 255) / 256, blocks_cap);
        return launch_ew(shard_sum_f32_vec, blocks, pdl, s, static_cast<const float4 *>(partials), n_parts, n,
                         reinterpret_cast<uint2 *>(out));
    }
    const int blocks = (int)std::min<int64_t>((plane + 255) / 256, blocks_cap);
    return launch_ew(shard_sum_scalar, blocks, pdl, s, partials, dtype_f32, n_parts, plane, out);
}

cudaError_t launch_reorder(const uint16_t *rm, uint16_t *logical, int64_t T, int64_t q_dim, int64_t kv_dim, int tp,
                           bool pdl, cudaStream_t s) {
    const int64_t C = q_dim + kv_dim, total = T * C;
    if (total <= 0) return cudaSuccess;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, 4096);
    return launch_ew(reorder_kernel, blocks, pdl, s, rm, logical, T, C, q_dim, q_dim / tp, kv_dim / tp);
}

cudaError_t launch_copy_in(const void *src, void *dst, int64_t bytes, bool early, int sm_count, cudaStream_t s) {
    if (bytes <= 0) return cudaSuccess;
    const uintptr_t a = reinterpret_cast<uintptr_t>(src), b = reinterpret_cast<uintptr_t>(dst);
    if (a % 16 == 0 && b % 16 == 0 && bytes % 16 == 0) {
        const int64_t n = bytes / 16;
        const int per = 256 * kCopyPer;
        const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((n + per - 1) / per, (int64_t)sm_count * 4));
        return launch_ew(copy_in_vec, blocks, true, s, static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n,
                         early ? 1 : 0);
    }
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((bytes + 255) / 256, (int64_t)sm_count * 4));
    return launch_ew(copy_in_bytes, blocks, true, s, static_cast<const unsigned char *>(src),
                     static_cast<unsigned char *>(dst), bytes);
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, uint32_t *err, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns, err);
    return cudaGetLastError();
}

}  // namespace mse
