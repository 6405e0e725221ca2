// noalloc.cu -- conv_bwd_data_run_noalloc: the tensor-core dgrad for callers
// that must not allocate device memory.
//
// Who needs it: code that runs inside a host framework which owns every byte
// of device memory through its own pool (a plugin or custom-op host, an
// inference server with a fixed arena), and latency-critical loops that may
// not call cudaMalloc because it can synchronise the device or fail under
// memory pressure at an unpredictable moment.  Such callers can pass their
// inputs and output, but cannot give the library the small device buffer
// that conv_bwd_data_create allocates for the kernel's status word.
//
// What replaces the allocation: the status word of the tensor-core kernel
// (its only scratch memory; every other byte it touches is an input or the
// output) lives in a file-scope __device__ array of a fixed size that every
// GPU loading this library holds until the process exits.  Every call shares
// that array and it keeps the last call's contents, so each call clears the
// status word on the caller's stream before launching; calls whose kernels
// overlap on the GPU (different streams, or different threads without
// ordering) race on the array and may report each other's status.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/conv_bwd_data.h"
#include "internal.h"

namespace cbd {
conv_bwd_status plan_create_borrowed_status(const conv_bwd_desc *desc, int32_t *status, conv_bwd_plan *out);
int32_t plan_path_of(conv_bwd_plan p);
}  // namespace cbd

namespace {

// Maximum scratch of the no-allocation entry point.  The tensor-core kernel
// needs kStatusBytes of it (one 32-bit status word, padded to 16 bytes).
constexpr size_t kStaticScratchBytes = 256;
constexpr size_t kStatusBytes = 16;
static_assert(kStatusBytes <= kStaticScratchBytes, "static scratch too small for the status word");

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, never a device address, so the
// address is looked up once per device, with that device current.
cudaError_t scratch_address(int dev, void **addr) {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" conv_bwd_status conv_bwd_data_run_noalloc(const conv_bwd_desc *desc, const void *dy, const void *w,
                                                     void *dx, void *stream, int32_t *device_status) {
    if (!desc || !dy || !w || !dx) return CONV_BWD_ERR_INVALID_ARG;
    if (device_status) *device_status = 0;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return CONV_BWD_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return CONV_BWD_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (scratch_address(dev, &scratch) != cudaSuccess) {
        cudaGetLastError();
        return CONV_BWD_ERR_CUDA;
    }
    conv_bwd_plan plan = nullptr;
    conv_bwd_status st = cbd::plan_create_borrowed_status(desc, static_cast<int32_t *>(scratch), &plan);
    if (st != CONV_BWD_OK) return st;
    // Only the tensor-core kernel (bf16 NHWC/KYXC, C/G >= 64) has this variant.
    if (cbd::plan_path_of(plan) != CONV_BWD_PATH_TCGEN05 || kStatusBytes > kStaticScratchBytes) {
        conv_bwd_data_destroy(plan);
        return CONV_BWD_ERR_UNSUPPORTED;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The array keeps the previous call's contents: the status word must start at zero.
    if (cudaMemsetAsync(scratch, 0, kStatusBytes, s) != cudaSuccess) {
        conv_bwd_data_destroy(plan);
        return CONV_BWD_ERR_CUDA;
    }
    st = conv_bwd_data_run(plan, dy, w, dx, stream);
    conv_bwd_data_destroy(plan);  // host memory only; kernel arguments were passed by value
    if (st != CONV_BWD_OK || !device_status) return st;
    int32_t h = 0;
    if (cudaMemcpyAsync(&h, scratch, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return CONV_BWD_ERR_CUDA;
    }
    *device_status = h;
    if (h == 0) return CONV_BWD_OK;
    return (h & 0xF00) == 0x200 ? CONV_BWD_ERR_DEVICE_FAULT : CONV_BWD_ERR_DEVICE_TIMEOUT;
}
