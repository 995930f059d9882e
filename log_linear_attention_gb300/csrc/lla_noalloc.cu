// lla_forward_noalloc: the prefill for callers that cannot allocate GPU memory.
//
// Some callers run where cudaMalloc is off limits: inside a host that owns every
// device allocation itself (a pre-sized arena), in code paths that must not grow
// the process's GPU footprint after start-up, or under allocators that forbid
// foreign allocations. For them the forward's scratch (inter-chunk states) lives
// in the fixed array below, which every GPU that loads this library holds until
// the process exits. The caller still passes its own inputs and output.
#include <mutex>

#include "../../include/lla.h"
#include "lla_internal.cuh"

// Scratch shared by every lla_forward_noalloc call on a device.
static __device__ __align__(256) unsigned char lla_noalloc_scratch[LLA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices];

// Device address of this device's scratch array, looked up once per device with
// that device current. In host code the array's name is only a host-side stand-in.
void* scratch_address(int dev) {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, lla_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int lla_forward_noalloc(const void* q, const void* k, const void* v, const float* log_a,
                                   const float* lambda, void* out, int B, int H, int T, int dk, int dv, int chunk,
                                   void* stream, int dtype) {
    const size_t need = lla_forward_workspace_size(B, H, T, dk, dv, chunk, dtype);
    if (need == 0) {
        // invalid sizes: let the regular validation report which argument is wrong
        return lla_forward_ws(q, k, v, log_a, lambda, out, B, H, T, dk, dv, chunk, stream, dtype, nullptr, 0);
    }
    if (need > LLA_NOALLOC_SCRATCH_BYTES) return LLA_ERR_NOMEM;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LLA_ERR_CUDA;
    void* scratch = scratch_address(dev);
    if (!scratch) return LLA_ERR_CUDA;
    return lla_forward_ws(q, k, v, log_a, lambda, out, B, H, T, dk, dv, chunk, stream, dtype, scratch,
                          LLA_NOALLOC_SCRATCH_BYTES);
}
