// mlp_swiglu_forward_static_scratch: the replicated shared-expert MLP for callers
// that cannot allocate device memory.  Its scratch (the bf16 intermediate h, the
// fp32 split-K partial tiles and the tile counters) lives in a fixed file-scope
// device array instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "mse.h"

namespace mse {
// defined in api.cu
void mlp_workspace_counter_range(int64_t T, int64_t H, int64_t I, size_t workspace_bytes, size_t *off,
                                 size_t *bytes);
}  // namespace mse

namespace {

// 32 MiB: enough for the decode-size shared-expert layer (T <= 64 tokens at
// hidden 7168 / intermediate 6144 needs 30.8 MiB: h, the split-K partial tiles of
// the three passes and the sync words).  Every device that loads the library holds this
// array until the process exits.
constexpr size_t kStaticScratchBytes = (size_t)32 << 20;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];   // device address of the array, per device
bool g_checked[kMaxDevices];         // compute capability read for this device
bool g_supported[kMaxDevices];       // compute capability 10.3 (the only code this library holds)

}  // namespace

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

extern "C" {

MSE_API mse_status mlp_swiglu_forward_static_scratch(const mse_bf16 *x, int64_t T, int64_t H, int64_t I,
                                                     const mse_bf16 *w_gate_up, const mse_bf16 *w_down, mse_bf16 *y,
                                                     int64_t y_capacity, void *stream) {
    if (!x || !w_gate_up || !w_down || !y || T <= 0 || H <= 0 || I <= 0) return MSE_ERR_INVALID_ARG;
    if (y_capacity < T * H) return MSE_ERR_GEOMETRY;
    const size_t need = mlp_swiglu_workspace_bytes(T, H, I);
    if (need == 0 || need > kStaticScratchBytes) return MSE_ERR_WORKSPACE;   // beyond the fixed maximum

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MSE_ERR_UNSUPPORTED_DEVICE;
    }
    void *scratch = nullptr;
    {
        // Set-up, once per device, with that device current: the array's name is
        // only a host-side stand-in, so its device address is looked up here.  The
        // device is checked first: on a device without sm_103a code the lookup would
        // fail (or load the module) instead of reporting the unsupported device.
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_checked[dev]) {
            int major = 0, minor = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
                cudaGetLastError();
                return MSE_ERR_CUDA;
            }
            g_supported[dev] = major == 10 && minor == 3;
            g_checked[dev] = true;
        }
        if (!g_supported[dev]) return MSE_ERR_UNSUPPORTED_DEVICE;
        if (!g_scratch_addr[dev]) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
                cudaGetLastError();
                return MSE_ERR_CUDA;
            }
            g_scratch_addr[dev] = p;
        }
        scratch = g_scratch_addr[dev];
    }
    // The array keeps the previous call's contents: the tile counters must start at zero.
    size_t off = 0, bytes = 0;
    mse::mlp_workspace_counter_range(T, H, I, kStaticScratchBytes, &off, &bytes);
    if (bytes > 0 &&
        cudaMemsetAsync(static_cast<unsigned char *>(scratch) + off, 0, bytes, static_cast<cudaStream_t>(stream)) !=
            cudaSuccess) {
        cudaGetLastError();
        return MSE_ERR_CUDA;
    }
    return mlp_swiglu_forward(x, T, H, I, w_gate_up, w_down, y, y_capacity, scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
