// mp_gemm_noalloc: the GEMM of mp_gemm for callers that must not allocate
// device memory.
//
// Some callers cannot call cudaMalloc at all, or cannot afford to:
//   - plugin interfaces of inference runtimes that own every byte of device
//     memory and hand a plugin only its inputs and outputs;
//   - processes that reserve (nearly) all device memory up front for their
//     own pool, so that a late cudaMalloc fails;
//   - latency-critical loops, where cudaMalloc and cudaFree may synchronize
//     the device and stall the whole pipeline.
// mp_gemm needs an mp_handle, and mp_init allocates the handle's split-K
// workspace, tile counters, status word and staging area with cudaMalloc.
// This entry point needs no handle: its scratch is one fixed array that is
// part of the library image (kScratchBytes below, about 48 MiB).  Its device
// memory is committed when the library's device code is loaded on a GPU: at
// the first call on that device under CUDA's default lazy module loading (or
// when the library loads, with CUDA_MODULE_LOADING=EAGER), and it is held
// until the process exits.  A caller that reserves nearly all device memory
// up front should make one call first.
//
// Layout of the array: split-K partials (16 MiB of fp32), tile counters (4096
// x 32 bit), the device status word, and a 32 MiB staging area for operands
// whose rows are not 16-byte aligned.
//
// Every call shares the array and finds it as the previous call left it: the
// tile counters a call uses are cleared on the call's stream before its
// kernel runs.  Two calls whose kernels overlap on the GPU (different streams,
// or several host threads) race on the array and give wrong results; issue
// them on one stream.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "mp_internal.h"

namespace {

constexpr size_t kPartialBytes = size_t(16) << 20;
constexpr size_t kCounterCount = 4096;
constexpr size_t kCounterBytes = kCounterCount * sizeof(unsigned int);
constexpr size_t kStatusBytes = 256;
constexpr size_t kStagingBytes = size_t(32) << 20;
constexpr size_t kScratchBytes = kPartialBytes + kCounterBytes + kStatusBytes + kStagingBytes;

// The fixed scratch.  In host code `g_scratch` only names the symbol; its
// device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct PerDevice {
    bool ready = false;
    mp_handle_s handle;  // planner state; no plan cache, so no host allocation either
    unsigned int* counters = nullptr;
};

PerDevice g_devices[mp::kMaxFixedDevices];
std::mutex g_setup_mu;

// First call on a device (with that device current): find the array's device
// address, clear the counters and status word, and point the library's device
// state at the array.  This first call synchronizes with a cudaMemset.
mp_status setup(int device, PerDevice** out) {
    if (device < 0 || device >= mp::kMaxFixedDevices) return MP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    PerDevice& d = g_devices[device];
    if (!d.ready) {
        void* base = nullptr;
        if (cudaGetSymbolAddress(&base, g_scratch) != cudaSuccess || base == nullptr) return MP_ERR_CUDA;
        uint8_t* p = static_cast<uint8_t*>(base);
        float* partials = reinterpret_cast<float*>(p);
        unsigned int* counters = reinterpret_cast<unsigned int*>(p + kPartialBytes);
        int* status = reinterpret_cast<int*>(p + kPartialBytes + kCounterBytes);
        uint8_t* staging = p + kPartialBytes + kCounterBytes + kStatusBytes;
        if (cudaMemset(counters, 0, kCounterBytes + kStatusBytes) != cudaSuccess) return MP_ERR_CUDA;
        mp_status st = mp::device_attach_fixed(&d.handle, device, partials, (int64_t)(kPartialBytes / sizeof(float)),
                                               counters, (int64_t)kCounterCount, status, staging,
                                               (int64_t)kStagingBytes);
        if (st != MP_OK) return st;
        mp::default_gb300_kernels(d.handle.hw, d.handle.kernels, &d.handle.num_kernels);
        mp::drop_unavailable_kernels(&d.handle);
        d.counters = counters;
        d.ready = true;
    }
    *out = &d;
    return MP_OK;
}

}  // namespace

extern "C" mp_status mp_gemm_noalloc(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                                     int64_t ldb, const float* C, int64_t ldc, float* D, int64_t ldd, float alpha,
                                     float beta, mp_stream stream) {
    mp::GemmArgs a{1, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, D, ldd, 0, alpha, beta, stream};
    mp_status st = mp::validate_args(a);
    if (st != MP_OK) return st;
    if (M == 0 || N == 0) return MP_OK;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return MP_ERR_CUDA;
    PerDevice* d = nullptr;
    st = setup(device, &d);
    if (st != MP_OK) return st;
    mp_plan_info plan;
    st = mp::plan_shape(&d->handle, 1, M, N, K, &plan);  // split-K bounded by the 16 MiB of partials
    if (st != MP_OK) return st;
    // Reject plans beyond the fixed scratch (the planner keeps partials within
    // it; the counters are checked here).
    int64_t counters = 0;
    for (int i = 0; i < plan.num_regions; i++) {
        const mp_region_info& r = plan.region[i];
        if (r.splits > 1) counters += ((r.m_ext + r.um - 1) / r.um) * ((r.n_ext + r.un - 1) / r.un);
    }
    if (counters > (int64_t)kCounterCount || plan.workspace_bytes > (int64_t)kPartialBytes) return MP_ERR_UNSUPPORTED;
    // The counters this launch uses must start at zero, whatever an earlier
    // (possibly aborted) call left there.
    if (counters > 0 && cudaMemsetAsync(d->counters, 0, (size_t)counters * sizeof(unsigned int),
                                        (cudaStream_t)stream) != cudaSuccess)
        return MP_ERR_CUDA;
    // Operands needing more than the 32 MiB staging area give MP_ERR_UNSUPPORTED here.
    return mp::device_run(&d->handle, plan, a);
}

// The fixed status word of the current device: a kernel of mp_gemm_noalloc
// that gave up on a bounded wait left a nonzero code there.  Synchronize
// `stream`, read the word, and on a nonzero code clear it and the tile
// counters (an aborted split may leave them mid-count).  Copies and memsets
// only: nothing is allocated.
extern "C" mp_status mp_check_noalloc(mp_stream stream) {
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return MP_ERR_CUDA;
    if (device < 0 || device >= mp::kMaxFixedDevices) return MP_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        if (!g_devices[device].ready) return MP_OK;  // nothing has run on this device
    }
    return mp_check(&g_devices[device].handle, stream);
}

// Test hook for the bounded waits of mp_gemm_noalloc on the current device
// (the same modes as mp_inject_wait_timeout).  Sets the device up first when
// no call has done so yet.
extern "C" mp_status mp_noalloc_inject_wait_timeout(int32_t enable, int64_t limit_ns) {
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return MP_ERR_CUDA;
    PerDevice* d = nullptr;
    mp_status st = setup(device, &d);
    if (st != MP_OK) return st;
    return mp_inject_wait_timeout(&d->handle, enable, limit_ns);
}
