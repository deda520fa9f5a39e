// Status strings, the per-device error word and small device queries.
#include "common.cuh"

#include <mutex>
#include <set>
#include <utility>

namespace {

// One error word per device: a kernel that meets bad data in device memory
// ORs a PK_DEVERR_* bit here and skips the access instead of faulting.
__device__ unsigned int g_error_word;

constexpr int kMaxDevices = 64;
unsigned int *g_error_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];
std::mutex g_mu;
std::set<std::pair<int, const void *>> g_smem_attr_done;   // (device, kernel) pairs already raised

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

}  // namespace

namespace pk {

unsigned int *error_word_ptr() {
    int dev = current_device();
    if (dev < 0) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_error_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_error_ptr[dev] = static_cast<unsigned int *>(p);
    }
    return g_error_ptr[dev];
}

int sm_count() {
    int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

cudaError_t set_max_dynamic_smem(const void *func, int bytes) {
    const int dev = current_device();
    if (dev < 0) {
        cudaGetLastError();
        return cudaErrorNoDevice;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_smem_attr_done.count({dev, func})) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    g_smem_attr_done.insert({dev, func});
    return cudaSuccess;
}

}  // namespace pk

extern "C" const char *pk_status_string(int status) {
    switch (status) {
        case PK_OK: return "ok";
        case PK_ERR_NULL: return "a required pointer is NULL";
        case PK_ERR_SHAPE: return "sizes are inconsistent or out of range";
        case PK_ERR_UNSUPPORTED: return "head_dim, block_size or group size not supported";
        case PK_ERR_WORKSPACE: return "workspace missing or too small";
        case PK_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
        case PK_ERR_ALIGNMENT: return "a device pointer is not 16-byte aligned";
        case PK_ERR_NO_DEVICE: return "no usable CUDA device";
        case PK_ERR_NO_BLOCKS: return "no free block left in the pool";
        case PK_ERR_UNKNOWN_SEQUENCE: return "no sequence with that id";
        case PK_ERR_SEQUENCE_EXISTS: return "a sequence with that id already exists";
        case PK_ERR_HOST_MEMORY: return "a host allocation failed";
        default: return "unknown status";
    }
}

extern "C" int pk_version(void) { return (1 << 16) | 0; }

extern "C" int pk_get_device_error(unsigned int *code_out, pk_stream_t stream) {
    if (!code_out) return PK_ERR_NULL;
    *code_out = 0;
    unsigned int *p = pk::error_word_ptr();
    if (!p) return PK_ERR_NO_DEVICE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned int v = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PK_ERR_CUDA;
    if (cudaMemcpyAsync(&v, p, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return PK_ERR_CUDA;
    if (cudaMemsetAsync(p, 0, sizeof(v), s) != cudaSuccess) return PK_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PK_ERR_CUDA;
    *code_out = v;
    return PK_OK;
}
