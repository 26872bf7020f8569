// ds41_common.cu - host-side error reporting and the device status word.
#include <mutex>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "ds41_common.cuh"

namespace ds41 {

static thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_check(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return DS41_OK;
    return fail(DS41_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int launch_check(const char* what) { return cuda_check(cudaGetLastError(), what); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One status word per device.  Kernels get its device address as an argument;
// the address is looked up once per device (with that device current).
static __device__ unsigned int g_status_word;
static constexpr int kMaxDevices = 64;
static unsigned int* g_status_ptr[kMaxDevices];
static std::mutex g_status_mu;

int status_word(unsigned int** out) {
    int dev = 0;
    int rc = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
    if (rc) return rc;
    if (dev < 0 || dev >= kMaxDevices) return fail(DS41_E_CUDA, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        rc = cuda_check(cudaGetSymbolAddress(&p, g_status_word), "cudaGetSymbolAddress(status)");
        if (rc) return rc;
        g_status_ptr[dev] = static_cast<unsigned int*>(p);
    }
    *out = g_status_ptr[dev];
    return DS41_OK;
}

}  // namespace ds41

extern "C" const char* ds41_last_error(void) { return ds41::g_msg; }

extern "C" int ds41_device_status(int32_t* status, int reset) {
    if (!status) return ds41::fail(DS41_E_ARG, "ds41_device_status: status is NULL");
    unsigned int* p = nullptr;
    int rc = ds41::status_word(&p);
    if (rc) return rc;
    unsigned int v = 0;
    rc = ds41::cuda_check(cudaDeviceSynchronize(), "ds41_device_status: synchronize");
    if (rc) return rc;
    rc = ds41::cuda_check(cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost),
                          "ds41_device_status: read");
    if (rc) return rc;
    *status = (int32_t)v;
    if (reset) {
        rc = ds41::cuda_check(cudaMemset(p, 0, sizeof v), "ds41_device_status: reset");
        if (rc) return rc;
        rc = ds41::cuda_check(cudaDeviceSynchronize(), "ds41_device_status: synchronize");
    }
    return rc;
}
