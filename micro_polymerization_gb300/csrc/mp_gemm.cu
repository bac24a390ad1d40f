// Host side of the persistent GEMM: tensor maps, device state, the plan's
// region table and the launch.  The kernel itself is in mp_kernel.cuh.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "mp_internal.h"
#include "mp_kernel.cuh"
#include "mp_b2b.cuh"
#include "mp_conv.cuh"
#include "mp_grouped.cuh"

namespace mp {
namespace dev {

// One operand to stage: a (batch x rows x cols) bf16 matrix whose rows are
// not 16-byte aligned, copied with rows padded to ld_dst (a multiple of 8
// elements, zero-filled) so that TMA can address it.
struct RepackJob {
    const uint16_t* src;
    long long ld_src, stride_src;
    uint16_t* dst;
    long long ld_dst, stride_dst;
    int rows, cols, batch;
};

// Up to two operands (A and B of one GEMM) in one launch: 16 bytes of the
// destination per thread and step, the first operand's chunks first.  Chunk
// indices stay below 2^31 (the staging area bounds them), so the index
// arithmetic is 32-bit.  The source is read in aligned 32-bit words: a row
// that starts 2 bytes past a word boundary takes each output pair from the
// high half of one word and the low half of the next.  Only words that hold
// at least one element of the row are read.
__global__ void k_repack_bf16(const RepackJob j0, const RepackJob j1, int njobs) {
    // Launched as a programmatic dependent: wait until the previous kernel
    // on the stream (which may still read the staging area) has finished;
    // the GEMM that reads this copy may start its own set-up meanwhile.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t c0 = (uint32_t)(j0.ld_dst / 8), c1 = njobs > 1 ? (uint32_t)(j1.ld_dst / 8) : 1u;
    const uint32_t t0 = (uint32_t)j0.batch * (uint32_t)j0.rows * c0;
    const uint32_t total = t0 + (njobs > 1 ? (uint32_t)j1.batch * (uint32_t)j1.rows * c1 : 0u);
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const bool second = i >= t0;
        const RepackJob& j = second ? j1 : j0;
        const uint32_t chunks = second ? c1 : c0;
        const uint32_t k = second ? i - t0 : i;
        const uint32_t rb = k / chunks;
        const uint32_t ch = k - rb * chunks;
        uint32_t b = 0, r = rb;
        if (j.batch > 1) {
            b = rb / (uint32_t)j.rows;
            r = rb - b * (uint32_t)j.rows;
        }
        const uint16_t* srow = j.src + (long long)b * j.stride_src + (long long)r * j.ld_src;
        const int e0 = (int)ch * 8;
        const int nvalid = min(8, j.cols - e0);  // >= 1: the padding never fills a whole chunk
        const bool odd = (reinterpret_cast<uintptr_t>(srow) & 2u) != 0;
        const uint32_t* wp =
            reinterpret_cast<const uint32_t*>(reinterpret_cast<uintptr_t>(srow) & ~uintptr_t(3)) + e0 / 2;
        uint32_t o[4];
        if (!odd) {
            // word k holds elements e0 + 2k (low half) and e0 + 2k + 1
#pragma unroll
            for (int q = 0; q < 4; q++) o[q] = 2 * q < nvalid ? __ldg(wp + q) : 0u;
        } else {
            // word k holds elements e0 + 2k - 1 (low half) and e0 + 2k
            uint32_t x[5];
#pragma unroll
            for (int q = 0; q < 5; q++) x[q] = 2 * q <= nvalid ? __ldg(wp + q) : 0u;
#pragma unroll
            for (int q = 0; q < 4; q++) o[q] = (x[q] >> 16) | (x[q + 1] << 16);
        }
#pragma unroll
        for (int q = 0; q < 4; q++) {
            if (2 * q >= nvalid) o[q] = 0u;
            else if (2 * q + 1 >= nvalid) o[q] &= 0xffffu;
        }
        *reinterpret_cast<uint4*>(j.dst + (long long)b * j.stride_dst + (long long)r * j.ld_dst + e0) =
            make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace dev

namespace {

dev::RepackJob repack_job(const void* src, long long ld_src, long long stride_src, uint16_t* dst, long long ld_dst,
                          long long stride_dst, int rows, int cols, int batch) {
    return dev::RepackJob{reinterpret_cast<const uint16_t*>(src), ld_src, stride_src, dst, ld_dst, stride_dst,
                          rows, cols, batch};
}

// One repack launch for `n` (1 or 2) operands, as a programmatic dependent of
// the previous kernel.
cudaError_t launch_repack(cudaStream_t stream, const dev::RepackJob* jobs, int n) {
    long long chunks = 0;
    for (int i = 0; i < n; i++) chunks += (long long)jobs[i].batch * jobs[i].rows * (jobs[i].ld_dst / 8);
    if (chunks >= (1ll << 31)) return cudaErrorInvalidValue;  // 32-bit chunk indices
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::max<long long>(1, std::min<long long>((chunks + 255) / 256, 4096)));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dev::k_repack_bf16, jobs[0], n > 1 ? jobs[1] : jobs[0], n);
}

}  // namespace

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

// Encoded tensor maps keyed by every input of the encoding: dynamic-shape
// callers reuse buffers (weights always, activations often), so most calls
// find their maps here instead of re-encoding them.
struct TmKey {
    uint64_t ptr;
    uint64_t dims[4];
    uint64_t strides[3];
    uint32_t box[4];
    uint32_t dtype, rank;
    bool operator==(const TmKey& o) const { return std::memcmp(this, &o, sizeof(TmKey)) == 0; }
};

struct alignas(128) TmEntry {
    CUtensorMap map;
    TmKey key;
    bool valid;
};

constexpr int kTmCacheEntries = 256;

struct DeviceState {
    int device = -1;
    int num_sms = 0;
    float* ws = nullptr;
    unsigned int* cnt = nullptr;
    int* err = nullptr;
    uint8_t* staging = nullptr;
    int64_t staging_bytes = 0;
    EncodeTiledFn encode = nullptr;
    bool log = false;
    int inject_timeout = 0;
    int64_t num_counters = kMaxCounters;  // split-K tile counters at `cnt`
    uint64_t wait_limit_ns = 1000000000ull;  // 1 s
    // Tensor-map cache (only for handles, which serve one host thread).
    TmEntry* tm_cache = nullptr;
    // Clusters of two CTAs of k_poly_gemm that can be resident at once (0:
    // paired launches disabled).
    int max_pairs = 0;
};

// The dynamic shared memory of every instantiation of the persistent kernel.
bool set_kernel_smem() {
    return set_poly_gemm_smem<0>() && set_poly_gemm_smem<8>() && set_poly_gemm_smem<16>() && set_poly_gemm_smem<32>() &&
           set_poly_gemm_smem_act_f32() &&
           set_poly_gemm_smem_bf16() && b2b::set_smem() &&
           conv::set_smem() && grp::set_smem();
}

// Split-K on chip: for S = 2..16, the CTAs that clusters of S CTAs of the
// one-CTA kernel can keep resident (queried once; sizes past 8 need the
// non-portable cluster attribute).  MP_CSPLIT=0 disables it.
void query_cluster_split(mp_handle h, int num_sms) {
    h->cluster_split_max = 0;
    for (int S = 0; S <= 16; S++) h->cluster_ctas[S] = 0;
    if (const char* v = std::getenv("MP_CSPLIT"))
        if (std::atoi(v) == 0) return;
    const bool big =
        cudaFuncSetAttribute(dev::k_poly_gemm<1, 0>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    if (!big) (void)cudaGetLastError();
    for (int S = 2; S <= (big ? 16 : 8); S++) {
        cudaLaunchConfig_t oc = {};
        oc.gridDim = dim3((unsigned)(S * ((num_sms + S - 1) / S)));
        oc.blockDim = dim3(dev::kThreads);
        oc.dynamicSmemBytes = dev::kSmemBytes;
        cudaLaunchAttribute ca[1];
        ca[0].id = cudaLaunchAttributeClusterDimension;
        ca[0].val.clusterDim.x = (unsigned)S;
        ca[0].val.clusterDim.y = 1;
        ca[0].val.clusterDim.z = 1;
        oc.attrs = ca;
        oc.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, dev::k_poly_gemm<1, 0>, &oc) != cudaSuccess) {
            (void)cudaGetLastError();
            continue;
        }
        if (n > 0) {
            h->cluster_ctas[S] = n * S;
            h->cluster_split_max = S;
        }
    }
}

// Resident two-CTA clusters of the persistent kernel (0 if the query fails).
int query_max_pairs(int num_sms) {
    // MP_PAIR=0 leaves pair micro-kernels out of the handle's set.
    if (const char* v = std::getenv("MP_PAIR"))
        if (std::atoi(v) == 0) return 0;
    cudaLaunchConfig_t oc = {};
    oc.gridDim = dim3((unsigned)(2 * ((num_sms + 1) / 2)));
    oc.blockDim = dim3(dev::kThreads);
    oc.dynamicSmemBytes = dev::kSmemBytes;
    cudaLaunchAttribute ca[1];
    ca[0].id = cudaLaunchAttributeClusterDimension;
    ca[0].val.clusterDim.x = 2;
    ca[0].val.clusterDim.y = 1;
    ca[0].val.clusterDim.z = 1;
    oc.attrs = ca;
    oc.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, dev::k_poly_gemm<2, 0>, &oc) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

namespace {

struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        ok = cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

// Tiled map, interleave none, 128-byte swizzle (or `swz`), zero fill,
// element strides 1.
bool encode_tiled(DeviceState* s, CUtensorMap* m, CUtensorMapDataType dt, uint32_t rank, const void* ptr,
                  const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                  CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    TmKey key;
    std::memset(&key, 0, sizeof key);
    key.ptr = (uint64_t)(uintptr_t)ptr;
    key.dtype = (uint32_t)dt | ((uint32_t)swz << 8);
    key.rank = rank;
    for (uint32_t i = 0; i < rank; i++) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
        if (i + 1 < rank) key.strides[i] = strides[i];
    }
    TmEntry* e = nullptr;
    if (s->tm_cache) {
        uint64_t h = key.ptr * 0x9E3779B97F4A7C15ull;
        for (uint32_t i = 0; i < rank; i++) h ^= (key.dims[i] + 0x632BE59BD9B4E019ull * (i + 1)) * 0xC2B2AE3D27D4EB4Full;
        h ^= ((uint64_t)key.box[0] << 32 | key.box[1]) * 0x165667B19E3779F9ull ^ (uint64_t)key.box[2] << 7 ^ dt ^
             (uint64_t)rank << 3;
        for (uint32_t i = 0; i + 1 < rank; i++) h ^= key.strides[i] * (0x27D4EB2F165667C5ull + i);
        h ^= h >> 31;
        e = &s->tm_cache[h % kTmCacheEntries];
        if (e->valid && e->key == key) {
            std::memcpy(m, &e->map, sizeof(CUtensorMap));
            return true;
        }
    }
    cuuint64_t d[5];
    cuuint64_t st[4];
    cuuint32_t bx[5], es[5];
    for (uint32_t i = 0; i < rank; i++) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    CUresult r = s->encode(m, dt, rank, const_cast<void*>(ptr), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    if (e) {
        std::memcpy(&e->map, m, sizeof(CUtensorMap));
        e->key = key;
        e->valid = true;
    }
    return true;
}

bool encode_3d(DeviceState* s, CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
               CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    const uint64_t dims[3] = {d0, d1, d2};
    const uint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const uint32_t box[3] = {box0, box1, 1};
    return encode_tiled(s, m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ptr, dims, strides, box, swz);
}

// fp32 output view [d2][d1][d0] for bulk tensor stores, box {box0, box1, 1}.
bool encode_3d_f32(DeviceState* s, CUtensorMap* m, void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1) {
    const uint64_t dims[3] = {d0, d1, d2};
    const uint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const uint32_t box[3] = {box0, box1, 1};
    return encode_tiled(s, m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box);
}

// fp32 output view with the 64-byte swizzle (boxes of 16 fp32 columns).
bool encode_3d_f32_sw64(DeviceState* s, CUtensorMap* m, void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                        uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1) {
    const uint64_t dims[3] = {d0, d1, d2};
    const uint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const uint32_t box[3] = {box0, box1, 1};
    return encode_tiled(s, m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

bool encode_4d(DeviceState* s, CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t d3, uint64_t s1, uint64_t s2, uint64_t s3, uint32_t box0, uint32_t box1, uint32_t box2) {
    const uint64_t dims[4] = {d0, d1, d2, d3};
    const uint64_t strides[3] = {s1, s2, s3};
    const uint32_t box[4] = {box0, box1, box2, 1};
    return encode_tiled(s, m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ptr, dims, strides, box);
}

bool tma_ok(const void* p, int64_t ld, int64_t batch, int64_t stride) {
    if (((uintptr_t)p & 15u) != 0) return false;
    if ((ld * 2) % 16 != 0) return false;
    if (batch > 1 && stride != 0 && (stride * 2) % 16 != 0) return false;
    return true;
}

void log_plan(const mp_plan_info& plan, const GemmArgs& a, int grid, int pair) {
    std::fprintf(stderr,
                 "[mp] batch=%lld M=%lld N=%lld K=%lld pattern=%d regions=%d tasks=%lld grid=%d cluster=%d cost=%.2fus\n",
                 (long long)a.batch, (long long)a.M, (long long)a.N, (long long)a.K, plan.pattern,
                 plan.num_regions, (long long)plan.total_tasks, grid, pair, plan.cost_us);
    for (int i = 0; i < plan.num_regions; i++) {
        const mp_region_info& r = plan.region[i];
        std::fprintf(stderr, "[mp]   R%d [%lld+%lld, %lld+%lld] kernel=%d (%dx%d%s) splits=%d f_num=%d waves=%lld pipe=%.2fus\n",
                     i, (long long)r.m0, (long long)r.m_ext, (long long)r.n0, (long long)r.n_ext, r.kernel, r.um,
                     r.un, r.swap ? " swapped" : "", r.splits, r.f_num, (long long)r.f_wave, r.f_pipe_us);
    }
}

}  // namespace

mp_status device_init(mp_handle h, int device) {
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) return MP_ERR_UNSUPPORTED;
    if (device >= count) return MP_ERR_INVALID_ARG;
    DeviceGuard g(device);
    if (!g.ok) return MP_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MP_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return MP_ERR_UNSUPPORTED;  // sm_103 only

    DeviceState* s = new DeviceState();
    h->dev = s;
    s->device = device;
    s->num_sms = prop.multiProcessorCount;
    s->log = std::getenv("MP_LOG") != nullptr;
    if (const char* v = std::getenv("MP_STAGING_BYTES")) s->staging_bytes = std::atoll(v);
    if (s->staging_bytes <= 0) s->staging_bytes = kDefaultStagingBytes;

    h->hw.num_pe = prop.multiProcessorCount;
    h->hw.warps_per_wave = prop.multiProcessorCount * kModelWarpsPerTask;
    h->hw.local_mem_bytes = (int64_t)prop.sharedMemPerBlockOptin;
    h->hw.shared_mem_bytes = (int64_t)prop.l2CacheSize;
    h->hw.hbm_gbs = 6684.0;    // measured STREAM-style copy on GB300
    h->hw.l2_gbs = 20000.0;    // L2 -> SM operand rate assumed by the model
    h->hw.mma_tflops = 1974.0; // measured dense bf16 on GB300

    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return MP_ERR_CUDA;
    s->encode = reinterpret_cast<EncodeTiledFn>(fn);
    if (!std::getenv("MP_NO_TMAP_CACHE")) s->tm_cache = new TmEntry[kTmCacheEntries]();

    if (cudaMalloc(&s->ws, sizeof(float) * (size_t)h->workspace_floats) != cudaSuccess) return MP_ERR_NO_MEMORY;
    if (cudaMalloc(&s->cnt, sizeof(unsigned) * (size_t)kMaxCounters) != cudaSuccess) return MP_ERR_NO_MEMORY;
    if (cudaMalloc(&s->err, sizeof(int)) != cudaSuccess) return MP_ERR_NO_MEMORY;
    if (cudaMalloc(&s->staging, (size_t)s->staging_bytes) != cudaSuccess) return MP_ERR_NO_MEMORY;
    if (cudaMemset(s->cnt, 0, sizeof(unsigned) * (size_t)kMaxCounters) != cudaSuccess) return MP_ERR_CUDA;
    if (cudaMemset(s->err, 0, sizeof(int)) != cudaSuccess) return MP_ERR_CUDA;
    if (!set_kernel_smem()) return MP_ERR_CUDA;
    s->max_pairs = query_max_pairs(s->num_sms);
    query_cluster_split(h, s->num_sms);
    if (cudaDeviceSynchronize() != cudaSuccess) return MP_ERR_CUDA;
    return MP_OK;
}

// Device state for the no-allocation entry point: the same kernels run over
// memory the caller of this function already owns (a fixed array of the
// library image), so nothing is allocated here.  One state per device,
// kept in static storage; call with `device` current.
mp_status device_attach_fixed(mp_handle h, int device, float* ws, int64_t ws_floats, unsigned int* cnt,
                              int64_t num_counters, int* err, uint8_t* staging, int64_t staging_bytes) {
    static DeviceState fixed_states[kMaxFixedDevices];
    if (device < 0 || device >= kMaxFixedDevices) return MP_ERR_UNSUPPORTED;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MP_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return MP_ERR_UNSUPPORTED;  // sm_103 only
    DeviceState* s = &fixed_states[device];
    s->device = device;
    s->num_sms = prop.multiProcessorCount;
    s->ws = ws;
    s->cnt = cnt;
    s->num_counters = num_counters;
    s->err = err;
    s->staging = staging;
    s->staging_bytes = staging_bytes;
    s->log = std::getenv("MP_LOG") != nullptr;
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return MP_ERR_CUDA;
    s->encode = reinterpret_cast<EncodeTiledFn>(fn);
    if (!set_kernel_smem()) return MP_ERR_CUDA;
    s->max_pairs = query_max_pairs(s->num_sms);
    query_cluster_split(h, s->num_sms);
    h->host_only = false;
    h->device = device;
    h->hw.num_pe = prop.multiProcessorCount;
    h->hw.warps_per_wave = prop.multiProcessorCount * kModelWarpsPerTask;
    h->hw.local_mem_bytes = (int64_t)prop.sharedMemPerBlockOptin;
    h->hw.shared_mem_bytes = (int64_t)prop.l2CacheSize;
    h->hw.hbm_gbs = 6684.0;
    h->hw.l2_gbs = 20000.0;
    h->hw.mma_tflops = 1974.0;
    h->workspace_floats = ws_floats;
    h->dev = s;
    return MP_OK;
}

void device_destroy(mp_handle h) {
    DeviceState* s = h->dev;
    if (!s) return;
    {
        DeviceGuard g(s->device);
        cudaDeviceSynchronize();
        cudaFree(s->ws);
        cudaFree(s->cnt);
        cudaFree(s->err);
        cudaFree(s->staging);
    }
    delete[] s->tm_cache;
    delete s;
    h->dev = nullptr;
}

mp_status device_check(mp_handle h, void* stream) {
    DeviceState* s = h->dev;
    if (!s) return MP_ERR_UNSUPPORTED;
    DeviceGuard g(s->device);
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MP_ERR_CUDA;
    int e = 0;
    if (cudaMemcpy(&e, s->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MP_ERR_CUDA;
    if (e != 0) {
        // An aborted launch may leave split-K counters mid-count: clear them.
        cudaMemset(s->err, 0, sizeof(int));
        cudaMemset(s->cnt, 0, sizeof(unsigned) * (size_t)s->num_counters);
        if (cudaDeviceSynchronize() != cudaSuccess) return MP_ERR_CUDA;
        return MP_ERR_DEVICE_TIMEOUT;
    }
    return MP_OK;
}

mp_status device_run(mp_handle h, const mp_plan_info& plan, const GemmArgs& a) {
    DeviceState* s = h->dev;
    if (!s) return MP_ERR_UNSUPPORTED;
    cudaStream_t stream = (cudaStream_t)a.stream;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return MP_ERR_CUDA;
    DeviceGuard g(s->device);  // no-op when already current

    dev::Params p;
    std::memset(&p, 0, sizeof(p));
    const int64_t batch = a.batch, M = a.M, N = a.N, K = a.K;

    // ---- CTA pairs: the plan's regions are all pair tiles or none ----------
    const int pair = plan.num_regions > 0 && plan.region[0].pair ? 1 : 0;
    if (pair && s->max_pairs <= 0) return MP_ERR_UNSUPPORTED;
    // ---- split-K on chip: every region split S ways, one task per CTA in
    // clusters of S, each partial fitting the idle operand ring ------------
    int csplit = 0;
    if (!pair && plan.num_regions > 0 && K > 0) {
        const int S = plan.region[0].splits;
        bool ok = S >= 2 && S <= h->cluster_split_max && S <= 8;  // past 8 measured no cheaper
        int64_t tasks = 0;
        for (int i = 0; i < plan.num_regions && ok; i++) {
            const mp_region_info& r = plan.region[i];
            const int64_t bn = r.swap ? r.um : r.un;
            const int64_t R = r.swap ? bn : 128, L = r.swap ? 128 : bn;
            ok = r.splits == S && R * (L + 4) * 4 <= dev::kRingBytes;
            tasks += cdiv(r.m_ext, r.um) * cdiv(r.n_ext, r.un) * batch * S;
        }
        if (ok && tasks <= mp::cluster_split_room(h, S)) csplit = S;
    }
    p.csplit = csplit;
    p.pair = pair;

    // ---- operands: TMA views, repacked when rows are not 16-byte aligned ----
    const void* A = a.A;
    const void* B = a.B;
    int64_t lda = a.lda, ldb = a.ldb, sA = a.strideA, sB = a.strideB;
    int64_t bA = (batch > 1 && a.strideA != 0) ? batch : 1;
    int64_t bB = (batch > 1 && a.strideB != 0) ? batch : 1;
    if (K > 0) {
        int64_t used = 0;
        dev::RepackJob jobs[2];
        int njobs = 0;
        if (!tma_ok(A, lda, batch, sA)) {
            const int64_t ld2 = round_up(K, 8), st2 = M * ld2;
            const int64_t bytes = round_up(2 * bA * st2, 256);
            if (used + bytes > s->staging_bytes) return MP_ERR_UNSUPPORTED;
            uint16_t* dst = reinterpret_cast<uint16_t*>(s->staging + used);
            jobs[njobs++] = repack_job(A, lda, sA, dst, ld2, st2, (int)M, (int)K, (int)bA);
            A = dst;
            lda = ld2;
            sA = st2;
            used += bytes;
        }
        if (!tma_ok(B, ldb, batch, sB)) {
            const int64_t ld2 = round_up(N, 8), st2 = K * ld2;
            const int64_t bytes = round_up(2 * bB * st2, 256);
            if (used + bytes > s->staging_bytes) return MP_ERR_UNSUPPORTED;
            uint16_t* dst = reinterpret_cast<uint16_t*>(s->staging + used);
            jobs[njobs++] = repack_job(B, ldb, sB, dst, ld2, st2, (int)K, (int)N, (int)bB);
            B = dst;
            ldb = ld2;
            sB = st2;
            used += bytes;
        }
        // Both operands' copies in one launch.
        if (njobs > 0 && launch_repack(stream, jobs, njobs) != cudaSuccess) return MP_ERR_CUDA;
        // Box shapes the plan's regions use: rows per A box of swapped tiles
        // (the smallest swapped bn divides the others: all are powers of 2),
        // and the numbers of 64-column blocks a B copy covers.
        int as_rows = 128;
        bool need_b4[4] = {false, false, false, false};
        bool need_bs = false;
        for (int i = 0; i < plan.num_regions; i++) {
            const mp_region_info& r = plan.region[i];
            if (r.swap) {
                as_rows = std::min(as_rows, (int)r.um);
                need_b4[1] = true;
            } else if (r.pair && r.un == 192) {
                need_bs = true;  // 96-column halves: 32-column boxes, 64-byte swizzle
            } else if (r.un >= 64 && r.un <= 256) {
                const int nblk = (int)(r.un / 64);
                if (r.pair) {  // each CTA of a pair holds half of the blocks
                    need_b4[nblk / 2 - 1] = true;
                } else {
                    need_b4[nblk - 1] = true;
                }
            }
        }
        p.as_rows = as_rows;
        const uint64_t a_s2 = bA > 1 ? (uint64_t)sA * 2 : (uint64_t)round_up(M * lda * 2, 16);
        const uint64_t b_s2 = bB > 1 ? (uint64_t)sB * 2 : (uint64_t)round_up(K * ldb * 2, 16);
        if (!encode_3d(s, &p.tmA, A, K, M, bA, lda * 2, a_s2, 64, 128) ||
            !encode_3d(s, &p.tmAs, A, K, M, bA, lda * 2, a_s2, 64, (uint32_t)as_rows) ||
            !encode_3d(s, &p.tmB, B, N, K, bB, ldb * 2, b_s2, 64, 64))
            return MP_ERR_CUDA;
        if (need_bs) {
            if (!encode_3d(s, &p.tmBs, B, N, K, bB, ldb * 2, b_s2, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B))
                return MP_ERR_CUDA;
            p.bs_ok = 1;
        }
        // Whole-tile B copies: B as [batch][N/64][K][64] (block stride 128 B).
        // Only full 64-column blocks are addressable, so nothing past a row
        // end is ever read; tiles reaching past the last full block load per
        // block.  If a view cannot be encoded, every tile loads per block.
        p.nb_full = (int)(N / 64);
        for (int j = 0; j < 4 && p.nb_full > 0; j++) {
            if (!need_b4[j]) continue;
            if (!encode_4d(s, &p.tmB4[j], B, 64, (uint64_t)K, (uint64_t)p.nb_full, (uint64_t)bB,
                           (uint64_t)ldb * 2, 128, b_s2, 64, 64, (uint32_t)(j + 1))) {
                p.nb_full = 0;
                p.b4_mask = 0;
                break;
            }
            p.b4_mask |= 1 << j;
        }
    } else {
        // K == 0: no operand is read; the maps only have to be well formed.
        p.as_rows = 16;
        p.nb_full = 0;
        if (!encode_3d(s, &p.tmA, s->staging, 64, 128, 1, 128, 128 * 128, 64, 128) ||
            !encode_3d(s, &p.tmAs, s->staging, 64, 128, 1, 128, 128 * 128, 64, 16) ||
            !encode_3d(s, &p.tmB, s->staging, 64, 128, 1, 128, 128 * 128, 64, 64))
            return MP_ERR_CUDA;
    }
    p.a_bstep = bA > 1 ? 1 : 0;
    p.b_bstep = bB > 1 ? 1 : 0;

    p.C = a.beta != 0.0f ? a.C : nullptr;
    // Bulk tensor stores of D for normal tiles when D's rows allow a tensor
    // map (16-byte aligned base, row pitch and batch pitch).  Rows and columns
    // past M and N are clipped by the map; region cuts fall on tile
    // boundaries, so no tile reaches another region.  C (beta != 0) is read
    // by the epilogue threads and fused before the store.
    // Epilogue variant: activation on alpha*acc + beta*C, and fp32 or bf16 D.
    p.act = a.epilogue & 0xff;
    p.out_bf16 = (a.epilogue & MP_EPI_OUT_BF16) ? 1 : 0;
    const int64_t de = p.out_bf16 ? 2 : 4;  // bytes per element of D
    p.tma_d = 0;
    if (((uintptr_t)a.D & 15u) == 0 && (a.ldd * de) % 16 == 0 && (batch == 1 || (a.strideD * de) % 16 == 0)) {
        const uint64_t d_s2 = batch > 1 ? (uint64_t)(a.strideD * de) : (uint64_t)round_up(M * a.ldd * de, 16);
        // fp32: slabs of 32 x 32; bf16: slabs of 64 columns x 32 rows (128-byte rows either way).
        if (p.out_bf16 ? encode_3d(s, &p.tmD, a.D, (uint64_t)N, (uint64_t)M, (uint64_t)batch,
                                   (uint64_t)(a.ldd * 2), d_s2, 64, 32)
                       : encode_3d_f32(s, &p.tmD, a.D, (uint64_t)N, (uint64_t)M, (uint64_t)batch,
                                       (uint64_t)a.ldd * 4, d_s2, 32, 32))
            p.tma_d = 1;
    }
    // Four consecutive elements per store: 16 bytes (fp32) or 8 bytes (bf16).
    p.vec_d = (((uintptr_t)a.D & (uintptr_t)(4 * de - 1)) == 0 && a.ldd % 4 == 0 &&
               (batch == 1 || a.strideD % 4 == 0))
                  ? 1
                  : 0;
    p.vec_c = (p.C && ((uintptr_t)a.C & 15u) == 0 && a.ldc % 4 == 0 && (batch == 1 || a.strideC % 4 == 0)) ? 1 : 0;
    p.D = a.D;
    p.ldc = a.ldc;
    p.ldd = a.ldd;
    p.strideC = a.strideC;
    p.strideD = a.strideD;
    p.alpha = a.alpha;
    p.beta = a.beta;
    p.num_kb = (int)cdiv(K, kUk);
    p.ws = s->ws;
    p.cnt = s->cnt;
    p.err = s->err;
    p.inject_timeout = s->inject_timeout;
    s->inject_timeout = 0;
    p.wait_limit_ns = s->wait_limit_ns;

    // ---- regions -> device work list ----------------------------------------
    int64_t units = 0, ws_floats = 0, counters = 0;
    p.num_regions = plan.num_regions;
    for (int i = 0; i < plan.num_regions; i++) {
        const mp_region_info& r = plan.region[i];
        dev::Region& d = p.reg[i];
        const int bn = r.swap ? r.um : r.un;
        if (r.uk != kUk || bn < 16 || bn > kMaxBn || bn % 16 != 0 || (r.pair != 0) != (pair != 0) ||
            (!r.swap && !r.pair && (r.um != 128 || bn % 64 != 0)) || (r.swap && (r.un != 128 || r.pair)) ||
            (r.pair && (r.um != 256 || (bn != 128 && bn != 192 && bn != 256) || r.splits != 1)))
            return MP_ERR_PLAN;
        d.m0 = (int)r.m0;
        d.n0 = (int)r.n0;
        d.m_end = (int)(r.m0 + r.m_ext);
        d.n_end = (int)(r.n0 + r.n_ext);
        d.tiles_m = (int)cdiv(r.m_ext, r.um);  // pairs: rows of 256-row tile pairs
        d.tiles_n = (int)cdiv(r.n_ext, r.un);
        {
            // When one problem's operands do not stay in L2 across waves,
            // order tiles so that a wave of `slots` tiles covers G rows x
            // slots/G columns; A and B bytes per wave balance at
            // G = sqrt(slots * un / um).
            const int64_t slots = pair ? s->max_pairs : s->num_sms;
            const double operand_bytes = 2.0 * (double)(M * K + K * N);
            int grp = 1;
            if ((int64_t)d.tiles_m * d.tiles_n > slots && operand_bytes > 0.6 * (double)h->hw.shared_mem_bytes) {
                grp = (int)std::lround(std::sqrt((double)slots * (double)r.un / (double)r.um));
                grp = std::max(1, std::min(grp, d.tiles_m));
            }
            d.group = grp;
        }
        d.bn = bn;
        d.swap = r.swap;
        d.splits = r.splits;
        d.kb_per_split = K > 0 ? (int)cdiv(p.num_kb, r.splits) : 0;
        if (K > 0 && cdiv(p.num_kb, d.kb_per_split) != r.splits) return MP_ERR_PLAN;
        const int64_t tiles = (int64_t)d.tiles_m * d.tiles_n * batch;
        d.unit_begin = (int)units;
        d.units = (int)(tiles * r.splits);
        units += tiles * r.splits;
        d.ws_begin = ws_floats;
        d.cnt_begin = (int)counters;
        if (r.splits > 1 && !csplit) {
            const int64_t rows = tiles * r.splits * 128;
            if (!r.swap && ws_floats + rows * bn <= h->workspace_floats &&
                encode_3d_f32(s, &p.tmW[i], s->ws + ws_floats, (uint64_t)bn, (uint64_t)rows, 1,
                              (uint64_t)bn * 4, (uint64_t)round_up(rows * bn * 4, 16), 32, 32))
                p.w_mask |= 1 << i;
            ws_floats += rows * bn;
            counters += tiles;
        }
    }
    if (units >= ((int64_t)1 << 31) || ws_floats > h->workspace_floats || counters > kMaxCounters)
        return MP_ERR_PLAN;
    p.total_units = (int)units;
    if (units == 0) return MP_OK;

    // Ring depth: stages sized for the widest Y tile of this plan.
    int bn_max = 16;
    for (int i = 0; i < p.num_regions; i++) bn_max = std::max(bn_max, p.reg[i].bn);
    // The single MMA-issuing thread pays a fixed cost per stage (barrier
    // check, fence, commit: about 350 cycles measured on GB300) on top of
    // about 70 cycles per MMA; two K steps per stage halve that cost per MMA
    // wherever the ring still holds at least three stages.  Measured on CTA
    // pairs with a 3072-deep K loop: 256 x 128 units 17.8 -> 12.9 us, 256 x 192
    // 17.8 -> 16.6 us; 256 x 256 within 3% either way.
    p.sub_bytes = dev::kXBytes + (pair ? bn_max / 2 : bn_max) * 128;  // a pair's CTA holds half of B
    p.kg = (3 * 2 * p.sub_bytes <= dev::kRingBytes) ? 2 : 1;
    p.stage_bytes = p.kg * p.sub_bytes;
    p.num_stages = std::min(dev::kMaxStages, dev::kRingBytes / p.stage_bytes);

    const int grid = pair     ? 2 * (int)std::min<int64_t>(units, s->max_pairs)
                     : csplit ? (int)units  // one task per CTA, a multiple of S
                              : (int)std::min<int64_t>(units, s->num_sms);
    if (s->log) log_plan(plan, a, grid, pair ? 2 : csplit);
    // One CTA per SM; launched as a programmatic dependent of the previous
    // kernel on the stream so that its set-up overlaps that kernel's tail.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(dev::kThreads);
    cfg.dynamicSmemBytes = dev::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = pair ? 2 : (csplit ? (unsigned)csplit : 1u);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (pair || csplit) ? 2 : 1;
    // One instantiation per epilogue: the activation in bits 0-1, a bf16 D in
    // bit 2 (the occupancy queries above hold for all of them: the same
    // threads, shared memory and launch bounds).
    const int epi = p.act | (p.out_bf16 ? 4 : 0);
    // Lean instantiations when the plan needs none of the paths they leave
    // out.  EPI bit 3 (any epilogue): no split, no swapped region, 16-byte
    // aligned D, beta = 0.  For the plain epilogue also bit 4 (no split, no
    // swapped region) and bit 5 (every region split, none swapped).
    bool nsns = !csplit;  // no split, no swapped region
    for (int i = 0; i < plan.num_regions && nsns; i++)
        nsns = plan.region[i].splits == 1 && !plan.region[i].swap;
    const bool lean = nsns && p.tma_d && p.beta == 0.0f;
    // L2 prefetch of each CTA's first three K steps before the dependency
    // wait, for one-CTA plans with no split, no swapped region and beta = 0.
    // Measured on GB300 in streams of different GEMMs with cold operands:
    // +1.5% on the dynamic-sequence step, +2.3% dynamic resolution, +1.3%
    // merged QKV, +2.5% the batched merge; deeper prefetches gained less
    // (six steps lost 0.5%).  Split and beta*C plans lost 0.9-1.5% with it,
    // and a GEMM repeated on operands already in L2 pays up to 0.14 us.
    p.l2_pf = (nsns && !pair && p.beta == 0.0f) ? kL2PrefetchSteps : 0;
    bool split_only = epi == 0 && !pair && plan.num_regions > 0;
    for (int i = 0; i < plan.num_regions && split_only; i++)
        split_only = plan.region[i].splits > 1 && !plan.region[i].swap;
    const int epi_l = lean ? (epi | 8) : epi;
    const cudaError_t e = epi == 0 ? (lean ? launch_poly_gemm<8>(cfg, pair, p)
                                      : nsns ? launch_poly_gemm<16>(cfg, pair, p)
                                      : split_only ? launch_poly_gemm<32>(cfg, false, p)
                                                   : launch_poly_gemm<0>(cfg, pair, p))
                          : p.out_bf16 ? launch_poly_gemm_bf16(cfg, pair, epi_l, p)
                                       : launch_poly_gemm_act_f32(cfg, pair, epi_l, p);
    if (e != cudaSuccess) return MP_ERR_CUDA;
    return MP_OK;
}

// A device that cannot hold two-CTA clusters of the kernel (or MP_PAIR=0)
// keeps no pair micro-kernels in its set.
void drop_unavailable_kernels(mp_handle h) {
    if (!h || !h->dev || h->dev->max_pairs > 0) return;
    int32_t n = 0;
    for (int32_t k = 0; k < h->num_kernels; k++)
        if (!h->kernels[k].pair) h->kernels[n++] = h->kernels[k];
    h->num_kernels = n;
}

// ---------------------------------------------------------------------------
// Back-to-back GEMMs: tensor maps and the launch of k_b2b_gemm
// ---------------------------------------------------------------------------
namespace {

// The bf16 operands of one launch whose base or row pitch TMA cannot address
// (at most three) are redirected to copies in the staging area with rows
// padded to a multiple of 8 elements; the copies go out two per launch.
struct StageOperand {
    const void** P;
    int64_t* ld;
    int64_t rows, cols;
};

mp_status stage_unaligned(DeviceState* s, cudaStream_t stream, const StageOperand* ops, int n, int64_t& used) {
    dev::RepackJob jobs[3];
    int nj = 0;
    for (int i = 0; i < n; i++) {
        const StageOperand& o = ops[i];
        if (tma_ok(*o.P, *o.ld, 1, 0)) continue;
        const int64_t ld2 = round_up(o.cols, 8);
        const int64_t bytes = round_up(2 * o.rows * ld2, 256);
        if (used + bytes > s->staging_bytes || nj == 3) return MP_ERR_UNSUPPORTED;
        uint16_t* dst = reinterpret_cast<uint16_t*>(s->staging + used);
        jobs[nj++] = repack_job(*o.P, *o.ld, 0, dst, ld2, 0, (int)o.rows, (int)o.cols, 1);
        *o.P = dst;
        *o.ld = ld2;
        used += bytes;
    }
    // The copy kernel takes two operands per launch.
    for (int i = 0; i < nj; i += 2)
        if (launch_repack(stream, jobs + i, std::min(2, nj - i)) != cudaSuccess) return MP_ERR_CUDA;
    return MP_OK;
}

}  // namespace

mp_status device_run_b2b(mp_handle h, const mp_b2b_plan& pl, const B2BArgs& a) {
    DeviceState* s = h->dev;
    if (!s) return MP_ERR_UNSUPPORTED;
    DeviceGuard g(s->device);
    b2b::Params p;
    std::memset(&p, 0, sizeof(p));
    const int64_t M = a.M, N0 = a.N0, N1 = a.N1, K0 = a.N0 > 0 ? a.K0 : 0;
    cudaStream_t stream = (cudaStream_t)a.stream;
    const void *A0 = a.A0, *W0 = a.W0, *W1 = a.W1;
    int64_t lda0 = a.lda0, ldw0 = a.ldw0, ldw1 = a.ldw1, used = 0;
    {
        StageOperand ops[3];
        int n = 0;
        if (K0 > 0) {
            ops[n++] = StageOperand{&A0, &lda0, M, K0};
            ops[n++] = StageOperand{&W0, &ldw0, K0, N0};
        }
        if (N0 > 0) ops[n++] = StageOperand{&W1, &ldw1, N0, N1};
        const mp_status st = stage_unaligned(s, stream, ops, n, used);
        if (st != MP_OK) return st;
    }
    if (K0 > 0) {
        if (!encode_3d(s, &p.tmA0, A0, K0, M, 1, lda0 * 2, round_up(M * lda0 * 2, 16), 64, 128) ||
            !encode_3d(s, &p.tmW0, W0, N0, K0, 1, ldw0 * 2, round_up(K0 * ldw0 * 2, 16), 64, 64))
            return MP_ERR_CUDA;
    }
    if (N0 > 0) {
        if (!encode_3d(s, &p.tmW1, W1, N1, N0, 1, ldw1 * 2, round_up(N0 * ldw1 * 2, 16), 64, 64))
            return MP_ERR_CUDA;
    }
    p.tma_d = (((uintptr_t)a.D1 & 15u) == 0 && (a.ldd1 * 4) % 16 == 0) ? 1 : 0;
    if (p.tma_d &&
        !encode_3d_f32_sw64(s, &p.tmD1, a.D1, N1, M, 1, a.ldd1 * 4, round_up(M * a.ldd1 * 4, 16), 16, 32))
        return MP_ERR_CUDA;
    p.C0 = a.C0;
    p.C1 = a.C1;
    p.D1 = a.D1;
    p.ldc0 = a.ldc0;
    p.ldc1 = a.ldc1;
    p.ldd1 = a.ldd1;
    p.M = (int)M;
    p.N0 = (int)N0;
    p.N1 = (int)N1;
    p.K0 = (int)K0;
    p.n0p = pl.n0p;
    p.bn1 = pl.bn1;
    p.chunks = pl.chunks;
    p.mblocks = pl.mblocks;
    p.cpg = pl.cpg;
    p.units = pl.units;
    p.num_stages = pl.num_stages;
    p.stage_bytes = pl.stage_bytes;
    p.alpha0 = a.alpha0;
    p.beta0 = a.beta0;
    p.alpha1 = a.alpha1;
    p.beta1 = a.beta1;
    p.act0 = a.act0;
    p.vec_c0 = (a.C0 && ((uintptr_t)a.C0 & 15u) == 0 && a.ldc0 % 4 == 0) ? 1 : 0;
    p.vec_c1 = (a.C1 && ((uintptr_t)a.C1 & 15u) == 0 && a.ldc1 % 4 == 0) ? 1 : 0;
    p.err = s->err;
    p.wait_limit_ns = s->wait_limit_ns;
    p.inject_timeout = s->inject_timeout;
    s->inject_timeout = 0;
    // L2 prefetch of each CTA's first K steps of A0 and W0 before the
    // dependency wait, as in the GEMM kernel.  Measured on GB300 (beta0 =
    // beta1 = 0): b2b_1x1 0.786 -> 0.752 ms per step, b2b_adapter 0.959 ->
    // 0.944 ms.  Pairs that read C0 or C1 are left without it, as the GEMM's
    // beta*C plans are.
    p.l2_pf = (a.beta0 == 0.0f && a.beta1 == 0.0f) ? kL2PrefetchSteps : 0;
    if (s->log)
        std::fprintf(stderr, "[mp] b2b M=%lld N0=%lld N1=%lld K0=%lld bn1=%d cpg=%d units=%d grid=%d stages=%d\n",
                     (long long)M, (long long)N0, (long long)N1, (long long)K0, pl.bn1, pl.cpg, pl.units, pl.grid,
                     pl.num_stages);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3(b2b::kThreads);
    cfg.dynamicSmemBytes = (size_t)pl.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (b2b::launch(cfg, p) != cudaSuccess) return MP_ERR_CUDA;
    return MP_OK;
}

// The two-launch form of a back-to-back pair: the first GEMM with the
// activation and a bf16 D (the rounding D0 gets on chip) into the handle's
// scratch buffer, then the second GEMM reading it.  Both launches go to the
// same stream, so the second reads D0 after the first has written it.
mp_status device_run_b2b_two(mp_handle h, const B2BArgs& a) {
    DeviceState* s = h->dev;
    if (!s) return MP_ERR_UNSUPPORTED;
    DeviceGuard g(s->device);
    const int64_t ld0 = round_up(std::max<int64_t>(a.N0, 1), 8);
    const int64_t bytes = round_up(a.M * ld0 * 2, 256);
    // D0 (bf16, rows of ld0) lives at the end of the handle's staging area,
    // allocated at mp_init, so that this form allocates nothing; the two
    // launches stage their unaligned operands in the part before it.  D0 may
    // take at most half of the area.
    const int64_t full = s->staging_bytes;
    if (bytes > full / 2) return MP_ERR_UNSUPPORTED;
    void* d0 = s->staging + (full - bytes);
    s->staging_bytes = full - bytes;
    mp_status st = MP_OK;
    if (a.N0 > 0) {
        GemmArgs g0{1, a.M, a.N0, a.K0, a.A0, a.lda0, 0, a.W0, a.ldw0, 0, a.C0, a.ldc0, 0,
                    static_cast<float*>(d0), ld0, 0, a.alpha0, a.beta0, a.stream,
                    a.act0 | MP_EPI_OUT_BF16};
        mp_plan_info p0;
        if ((st = validate_args(g0)) != MP_OK || (st = plan_shape(h, 1, a.M, a.N0, a.K0, &p0)) != MP_OK ||
            (st = device_run(h, p0, g0)) != MP_OK) {
            s->staging_bytes = full;
            return st;
        }
    }
    GemmArgs g1{1, a.M, a.N1, a.N0, d0, ld0, 0, a.W1, a.ldw1, 0, a.C1, a.ldc1, 0, a.D1, a.ldd1, 0,
                a.alpha1, a.beta1, a.stream, 0};
    mp_plan_info p1;
    if ((st = validate_args(g1)) == MP_OK && (st = plan_shape(h, 1, a.M, a.N1, a.N0, &p1)) == MP_OK)
        st = device_run(h, p1, g1);
    s->staging_bytes = full;
    return st;
}

// ---------------------------------------------------------------------------
// Implicit-GEMM convolution: tensor maps and the launch of k_conv_igemm
// ---------------------------------------------------------------------------
mp_status device_run_conv(mp_handle h, const mp_conv_plan& pl, const ConvArgs& a) {
    DeviceState* s = h->dev;
    if (!s) return MP_ERR_UNSUPPORTED;
    DeviceGuard g(s->device);
    conv::Params p;
    std::memset(&p, 0, sizeof(p));
    cudaStream_t stream = (cudaStream_t)a.stream;
    const int64_t N = a.N, H = a.H, W = a.W, C = a.C, K = a.K, R = a.R, S = a.S;
    const int64_t P = H + 2 * a.pad_h - R + 1, Q = W + 2 * a.pad_w - S + 1;
    if (C > 0) {
        // X as [N*H*W] rows of C channels and F as [R*S*C] rows of K: copied
        // with padded rows when TMA cannot address them.
        const void* X = a.X;
        const void* F = a.F;
        int64_t ldx = C, ldf = K, used = 0;
        const StageOperand ops[2] = {{&X, &ldx, N * H * W, C}, {&F, &ldf, R * S * C, K}};
        const mp_status st = stage_unaligned(s, stream, ops, 2, used);
        if (st != MP_OK) return st;
        const uint64_t xd[4] = {(uint64_t)C, (uint64_t)W, (uint64_t)H, (uint64_t)N};
        const uint64_t xs[3] = {(uint64_t)ldx * 2, (uint64_t)(W * ldx * 2), (uint64_t)(H * W * ldx * 2)};
        const uint32_t xb[4] = {64, (uint32_t)pl.wb, (uint32_t)pl.hb, (uint32_t)pl.nb};
        if (!encode_tiled(s, &p.tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, X, xd, xs, xb) ||
            !encode_3d(s, &p.tmF, F, K, R * S * C, 1, ldf * 2, round_up(R * S * C * ldf * 2, 16), 64, 64))
            return MP_ERR_CUDA;
    }
    const bool d_aligned = ((uintptr_t)a.D & 15u) == 0 && (a.ldd * 4) % 16 == 0;
    auto pow2 = [](int v) { return v > 0 && (v & (v - 1)) == 0; };
    const bool pow2_box = pow2(pl.wb) && pow2(pl.hb) && pow2(pl.nb) && pl.wb * pl.hb * pl.nb == 128;
    p.tma_d = d_aligned && pow2_box ? 1 : 0;
    p.vec_d = d_aligned ? 1 : 0;
    p.box_rows = pl.wb * pl.hb * pl.nb;
    p.bw = pl.wb >= 32 ? 32 : pl.wb;
    p.bh = pl.wb >= 32 ? 1 : (pl.wb * pl.hb >= 32 ? 32 / pl.wb : pl.hb);
    p.bnn = 32 / (p.bw * p.bh);
    if (p.tma_d) {
        const uint64_t dd[4] = {(uint64_t)K, (uint64_t)Q, (uint64_t)P, (uint64_t)N};
        const uint64_t ds[3] = {(uint64_t)a.ldd * 4, (uint64_t)(Q * a.ldd * 4), (uint64_t)(P * Q * a.ldd * 4)};
        const uint32_t db[4] = {32, (uint32_t)p.bw, (uint32_t)p.bh, (uint32_t)p.bnn};
        if (!encode_tiled(s, &p.tmD, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.D, dd, ds, db)) return MP_ERR_CUDA;
    }
    p.Cin = a.Cin;
    p.D = a.D;
    p.ldc = a.ldc;
    p.ldd = a.ldd;
    p.N = (int)N;
    p.H = (int)H;
    p.W = (int)W;
    p.C = (int)C;
    p.K = (int)K;
    p.R = (int)R;
    p.S = (int)S;
    p.pad_h = (int)a.pad_h;
    p.pad_w = (int)a.pad_w;
    p.P = (int)P;
    p.Q = (int)Q;
    p.wb = pl.wb;
    p.hb = pl.hb;
    p.nb = pl.nb;
    p.tiles_q = pl.tiles_q;
    p.tiles_p = pl.tiles_p;
    p.tiles_n = pl.tiles_n;
    p.tiles_k = pl.tiles_k;
    p.bn = pl.bn;
    p.cblocks = (int)cdiv(C, 64);
    p.ksteps = pl.ksteps;
    p.tiles = pl.tiles;
    p.splits = pl.splits;
    p.units = pl.units;
    p.ws = s->ws;
    if (pl.splits > 1 && (int64_t)pl.tiles * pl.splits * 128 * pl.bn > h->workspace_floats) return MP_ERR_PLAN;
    p.num_stages = pl.num_stages;
    p.stage_bytes = pl.stage_bytes;
    p.alpha = a.alpha;
    p.beta = a.beta;
    p.vec_c = (a.Cin && ((uintptr_t)a.Cin & 15u) == 0 && a.ldc % 4 == 0) ? 1 : 0;
    p.err = s->err;
    p.wait_limit_ns = s->wait_limit_ns;
    p.inject_timeout = s->inject_timeout;
    s->inject_timeout = 0;
    // L2 prefetch of each CTA's first K steps before the dependency wait, as
    // in the GEMM kernel.  Measured on GB300 on the dynamic-resolution layers
    // (beta = 0): +1.3% with it on every plan, +0.6% on unsplit plans only.
    // beta*Cin layers are left without it, as the GEMM's beta*C plans are.
    p.l2_pf = a.beta == 0.0f ? kL2PrefetchSteps : 0;
    if (s->log)
        std::fprintf(stderr, "[mp] conv N=%lld H=%lld W=%lld C=%lld K=%lld RxS=%lldx%lld tile %dx%dx%d bn=%d splits=%d units=%d\n",
                     (long long)N, (long long)H, (long long)W, (long long)C, (long long)K, (long long)R, (long long)S,
                     pl.wb, pl.hb, pl.nb, pl.bn, pl.splits, pl.units);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.grid);
    cfg.blockDim = dim3(conv::kThreads);
    cfg.dynamicSmemBytes = (size_t)pl.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (conv::launch(cfg, p) != cudaSuccess) return MP_ERR_CUDA;
    if (pl.splits > 1 && conv::launch_reduce(stream, p) != cudaSuccess) return MP_ERR_CUDA;
    return MP_OK;
}

// ---------------------------------------------------------------------------
// Grouped GEMM: per-problem tensor maps in the kernel parameters, one launch
// per 48 problems
// ---------------------------------------------------------------------------
mp_status device_run_grouped(mp_handle h, const mp_grouped_plan& pl, int32_t count, const mp_gemm_problem* probs,
                             void* stream_ptr) {
    DeviceState* s = h->dev;
    if (!s) return MP_ERR_UNSUPPORTED;
    DeviceGuard g(s->device);
    cudaStream_t stream = (cudaStream_t)stream_ptr;
    static_assert(sizeof(grp::Params) <= 32764, "the problem table must fit the kernel parameters");
    grp::Params* p = new (std::nothrow) grp::Params;
    if (!p) return MP_ERR_NO_MEMORY;
    int64_t used = 0;  // staging bytes taken by repacked operands (the whole group's)
    mp_status st = MP_OK;
    for (int32_t first = 0; first < count && st == MP_OK; first += grp::kMaxGroup) {
        std::memset(p, 0, sizeof(*p));
        const int32_t n = std::min<int32_t>(grp::kMaxGroup, count - first);
        int units = 0;
        for (int32_t j = 0; j < n && st == MP_OK; j++) {
            const mp_gemm_problem& a = probs[first + j];
            grp::Problem& q = p->prob[j];
            const void* A = a.A;
            const void* B = a.B;
            int64_t lda = a.lda, ldb = a.ldb;
            if (a.K > 0) {
                const StageOperand ops[2] = {{&A, &lda, a.M, a.K}, {&B, &ldb, a.K, a.N}};
                if ((st = stage_unaligned(s, stream, ops, 2, used)) != MP_OK) break;
                if (!encode_3d(s, &q.tmA, A, a.K, a.M, 1, lda * 2, round_up(a.M * lda * 2, 16), 64, 128) ||
                    !encode_3d(s, &q.tmB, B, a.N, a.K, 1, ldb * 2, round_up(a.K * ldb * 2, 16), 64, 64)) {
                    st = MP_ERR_CUDA;
                    break;
                }
            }
            q.tma_d = (((uintptr_t)a.D & 15u) == 0 && (a.ldd * 4) % 16 == 0) ? 1 : 0;
            if (q.tma_d &&
                !encode_3d_f32(s, &q.tmD, a.D, a.N, a.M, 1, a.ldd * 4, round_up(a.M * a.ldd * 4, 16), 32, 32)) {
                st = MP_ERR_CUDA;
                break;
            }
            q.C = a.C;
            q.D = a.D;
            q.ldc = a.ldc;
            q.ldd = a.ldd;
            q.M = (int)a.M;
            q.N = (int)a.N;
            q.K = (int)a.K;
            q.tiles_n = (int)cdiv(a.N, pl.bn);
            q.tile0 = units;
            q.alpha = a.alpha;
            q.beta = a.beta;
            q.vec_c = (a.C && ((uintptr_t)a.C & 15u) == 0 && a.ldc % 4 == 0) ? 1 : 0;
            units += (int)(cdiv(a.M, 128) * q.tiles_n);
        }
        if (st != MP_OK) break;
        p->count = n;
        p->units = units;
        p->bn = pl.bn;
        p->num_stages = pl.num_stages;
        p->stage_bytes = pl.stage_bytes;
        p->err = s->err;
        p->wait_limit_ns = s->wait_limit_ns;
        p->inject_timeout = s->inject_timeout;
        s->inject_timeout = 0;
        // L2 prefetch of each CTA's first K steps before the dependency wait,
        // as in the GEMM kernel (the kernel leaves out problems that read
        // C).  Measured on GB300 on the 48-problem expert group: 0.0817 ->
        // 0.0812 ms per call.
        p->l2_pf = kL2PrefetchSteps;
        if (s->log)
            std::fprintf(stderr, "[mp] grouped problems=%d bn=%d units=%d\n", n, pl.bn, units);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)std::min<int64_t>(units, s->num_sms));
        cfg.blockDim = dim3(grp::kThreads);
        cfg.dynamicSmemBytes = (size_t)pl.smem_bytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (grp::launch(cfg, *p) != cudaSuccess) st = MP_ERR_CUDA;
    }
    delete p;
    return st;
}

}  // namespace mp

// Test hook for the bounded waits: the next launch withholds one stage (1),
// or makes the ring-staged split-K sums wait for bytes that never come (2),
// so that a bounded wait runs out after `limit_ns`; mp_check then reports
// MP_ERR_DEVICE_TIMEOUT.  limit_ns == 0 keeps the current limit.
extern "C" mp_status mp_inject_wait_timeout(mp_handle h, int32_t enable, int64_t limit_ns) {
    if (!h || !h->dev || limit_ns < 0 || enable < 0 || enable > 2) return MP_ERR_INVALID_ARG;
    h->dev->inject_timeout = enable;
    if (limit_ns > 0) h->dev->wait_limit_ns = (uint64_t)limit_ns;
    return MP_OK;
}
