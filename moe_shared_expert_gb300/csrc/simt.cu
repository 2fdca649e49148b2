// Generic CUDA-core kernels: a shared-memory tiled bf16 GEMM with fp32
// accumulation and the three epilogues of the library.  They serve every shape
// and alignment (e.g. the tiny tp=4 / hidden 16 / intermediate 12 case, whose
// 3-wide shard slices break the 16-byte TMA stride rule) and act as the
// independent CUDA cross-check of the tensor-core kernels.
#include "common.cuh"
#include "kernels.h"

namespace mse {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

__device__ __forceinline__ int64_t logical_to_gathered(int64_t c, int64_t q_dim, int64_t kv_dim, int tp) {
    // logical column c of [q_a | kv_a] -> its column in the rank-major gather
    const int64_t qs = q_dim / tp, ks = kv_dim / tp, w = qs + ks;
    if (c < q_dim) return (c / qs) * w + (c % qs);
    const int64_t c2 = c - q_dim;
    return (c2 / ks) * w + qs + (c2 % ks);
}

template <bool kSwiglu>
__global__ void __launch_bounds__(NT) simt_gemm_kernel(SimtGemmArgs a) {
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    __shared__ float B2s[kSwiglu ? BK : 1][BN + 4];

    const int g = blockIdx.z;
    const uint16_t *A = a.A + g * a.a_gstride;
    const uint16_t *B = a.B + g * a.b_gstride;
    const uint16_t *B2 = kSwiglu ? a.B2 + g * a.b_gstride : nullptr;
    const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;

    float acc[4][4] = {};
    float acc2[4][4] = {};

    for (int64_t k0 = 0; k0 < a.K; k0 += BK) {
#pragma unroll
        for (int i = 0; i < (BM * BK) / NT; ++i) {
            const int e = tid + i * NT, r = e / BK, k = e % BK;
            const int64_t gm = m0 + r, gk = k0 + k;
            As[k][r] = (gm < a.M && gk < a.K) ? bf16_bits_to_f32(A[gm * a.lda + gk]) : 0.f;
            const int64_t gn = n0 + r;
            const bool okb = (gn < a.N && gk < a.K);
            Bs[k][r] = okb ? bf16_bits_to_f32(B[gn * a.ldb + gk]) : 0.f;
            if (kSwiglu) B2s[k][r] = okb ? bf16_bits_to_f32(B2[gn * a.ldb + gk]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < BK; ++k) {
            float av[4], bv[4], b2v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                av[i] = As[k][ty * 4 + i];
                bv[i] = Bs[k][tx * 4 + i];
                if (kSwiglu) b2v[i] = B2s[k][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
                    if (kSwiglu) acc2[i][j] = fmaf(av[i], b2v[j], acc2[i][j]);
                }
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + ty * 4 + i;
        if (m >= a.M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t n = n0 + tx * 4 + j;
            if (n >= a.N) continue;
            const int64_t o = g * a.o_gstride + m * a.ldo + n;
            if (kSwiglu) {
                static_cast<uint16_t *>(a.out)[o] = f32_to_bf16_bits(silu_f32(acc[i][j]) * acc2[i][j]);
            } else if (a.mode == SIMT_F32) {
                static_cast<float *>(a.out)[o] = acc[i][j];
            } else if (a.mode == SIMT_BF16) {
                static_cast<uint16_t *>(a.out)[o] = f32_to_bf16_bits(acc[i][j]);
            } else {  // SIMT_MERGED
                const uint16_t v = f32_to_bf16_bits(acc[i][j]);
                if (a.out) static_cast<uint16_t *>(a.out)[o] = v;
                if (a.out_rm) a.out_rm[m * a.ldo + logical_to_gathered(n, a.q_dim, a.kv_dim, a.tp)] = v;
            }
        }
    }
}

}  // namespace

cudaError_t launch_simt_gemm(const SimtGemmArgs &a, cudaStream_t s) {
    if (a.M <= 0 || a.N <= 0 || a.groups <= 0) return cudaSuccess;
    dim3 grid((unsigned)((a.N + BN - 1) / BN), (unsigned)((a.M + BM - 1) / BM), (unsigned)a.groups);
    if (a.mode == SIMT_SWIGLU)
        simt_gemm_kernel<true><<<grid, NT, 0, s>>>(a);
    else
        simt_gemm_kernel<false><<<grid, NT, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace mse
