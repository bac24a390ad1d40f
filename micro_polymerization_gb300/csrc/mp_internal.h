// Internal declarations shared by the host planner, the C ABI and the launch
// code.  Nothing here is exported.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <vector>

#include "mp.h"  // include/ is on the compiler's include path

namespace mp {

// Micro-kernel geometry fixed by the device code: UMMA M = 128 rows of
// accumulator lanes, one 128-byte swizzle row of bf16 (64 elements) per K step.
constexpr int kUmmaM = 128;
constexpr int kUk = 64;
constexpr int kMaxBn = 256;
// K steps of A and B a one-CTA launch prefetches into L2 before waiting for
// the previous kernel on the stream (plans that qualify: mp_gemm.cu).
constexpr int kL2PrefetchSteps = 3;
// Warps per task in the wave model of the GB300 kernel set (one CTA per SM,
// so warps_per_wave = SMs * kModelWarpsPerTask gives one task slot per SM).
constexpr int kModelWarpsPerTask = 6;

// Limits of the device-side bookkeeping (allocated once per handle).
constexpr int64_t kMaxCounters = 1 << 16;          // split-K tile counters
constexpr int64_t kDefaultWorkspaceFloats = 16ll << 20;  // 64 MiB of fp32 partials
constexpr int64_t kDefaultStagingBytes = 1ll << 30;      // repack area for unaligned operands
constexpr int kMaxFixedDevices = 64;                      // devices served by the no-allocation entry point

// Split-K reduction cost beyond g_predict(f_num), per task: sync_us plus
// bytes_factor passes of the tile's fp32 partial at one PE's share of L2
// bandwidth.  Through L2: park the partial, a counter round trip, sum 1/S of
// every partial.  On chip (clusters of S <= 8 CTAs): two cluster barriers and
// the sum through distributed shared memory, with terms per S (measured on
// GB300 the sum costs more at S = 2 and 3, where each CTA sums and stores a
// larger slice).  Defaults fitted on GB300 from timestamped kernel copies; a
// calibration table's "split" lines replace them with measured values.
constexpr int kClusterSplitMaxS = 8;
constexpr double kDefaultSplitSyncUs[2] = {4.0, 2.5};        // [0] through L2, [1] on chip
constexpr double kDefaultSplitBytesFactor[2] = {4.0, 1.0};

struct PlanKey {
    int64_t batch, M, N, K;
    bool operator==(const PlanKey& o) const {
        return batch == o.batch && M == o.M && N == o.N && K == o.K;
    }
};

struct PlanCacheEntry {
    PlanKey key{-1, -1, -1, -1};
    mp_plan_info plan{};
};

struct DeviceState;  // defined in the CUDA translation unit

}  // namespace mp

struct mp_handle_s {
    bool host_only = true;
    int device = -1;
    mp_hw hw{};
    mp_kernel_desc kernels[MP_MAX_KERNELS]{};
    int32_t num_kernels = 0;

    // Test / ablation hooks (mp_force_plan, mp_set_plan_mode).
    int32_t force_kernel = -1;
    int32_t force_splits = 0;
    int32_t plan_mode = MP_PLAN_MIKPOLY;
    int32_t b2b_mode = MP_B2B_AUTO;

    // Plan cache: shapes repeat in dynamic workloads; a hit skips the search.
    std::vector<mp::PlanCacheEntry> cache;
    int64_t workspace_floats = mp::kDefaultWorkspaceFloats;

    // Split-K on chip (clusters of S CTAs reduce through distributed shared
    // memory): the largest S a cluster can hold (0: none), and per S the
    // CTAs such clusters can keep resident at once.
    int32_t cluster_split_max = 0;
    int32_t cluster_ctas[17] = {};

    // true once a calibration table has set a micro-kernel's g_predict (the
    // GEMM estimates then include each launch's fixed costs).
    bool calibrated = false;

    // Split-K cost model (mp_set_split_model): index 0 through L2, index S
    // (2..8) on chip in clusters of S CTAs; index 1 is unused.
    double split_sync_us[mp::kClusterSplitMaxS + 1];
    double split_bytes_factor[mp::kClusterSplitMaxS + 1];
    mp_handle_s() {
        for (int s = 0; s <= mp::kClusterSplitMaxS; s++) {
            split_sync_us[s] = mp::kDefaultSplitSyncUs[s == 0 ? 0 : 1];
            split_bytes_factor[s] = mp::kDefaultSplitBytesFactor[s == 0 ? 0 : 1];
        }
    }

    mp::DeviceState* dev = nullptr;
};

namespace mp {

// Tasks a split-K launch on chip (clusters of S CTAs) may have: the clusters
// the device keeps resident, less one for odd S.  Measured on GB300 in a
// stream of different GEMMs, clusters of 3 and 5 that took every cluster slot
// cost 3-5 us more than with one slot free (odd clusters straddle the
// two-SM TPCs, and the last ones wait until the previous kernel's CTAs leave
// the SMs they need); at full occupancy clusters of 2, 4, 6 and 8 did not,
// and back to back, one shape after itself, none did.
inline int64_t cluster_split_room(const mp_handle_s* h, int S) {
    const int64_t cap = h->cluster_ctas[S];
    return (S & 1) ? (cap > S ? cap - S : 0) : cap;
}

// Planner (mp_planner.cpp).
mp_status plan_shape(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K,
                     mp_plan_info* out);
void clear_plan_cache(mp_handle h);
// Every candidate strategy of the search space, sorted by cost (mp_enumerate_plans).
mp_status enumerate_plans(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K,
                          std::vector<mp_plan_info>* out);
mp_status evaluate_plan(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K,
                        mp_plan_info* p);
void default_gb300_kernels(const mp_hw& hw, mp_kernel_desc* out, int32_t* n);
// Checks that the regions of a plan tile the M x N output exactly once and
// satisfy the device code's alignment rules.  Returns MP_OK or MP_ERR_PLAN.
mp_status validate_plan(const mp_plan_info& p, int64_t M, int64_t N, int64_t K);

// Device side (mp_gemm.cu).
mp_status device_init(mp_handle h, int device);
void device_destroy(mp_handle h);
struct GemmArgs {
    int64_t batch, M, N, K;
    const void* A; int64_t lda, strideA;
    const void* B; int64_t ldb, strideB;
    const float* C; int64_t ldc, strideC;
    float* D; int64_t ldd, strideD;
    float alpha, beta;
    void* stream;
    int32_t epilogue = 0;  // mp_gemm_ex's epilogue word (activation, bf16 D)
};
mp_status device_run(mp_handle h, const mp_plan_info& plan, const GemmArgs& a);
mp_status device_check(mp_handle h, void* stream);
// Remove micro-kernels the handle's device cannot run (CTA pairs).
void drop_unavailable_kernels(mp_handle h);
mp_status device_attach_fixed(mp_handle h, int device, float* ws, int64_t ws_floats, unsigned int* cnt,
                              int64_t num_counters, int* err, uint8_t* staging, int64_t staging_bytes);
// Argument rules of mp_gemm (mp_api.cpp).
mp_status validate_args(const GemmArgs& a);

// Back-to-back GEMMs (mp_gemm_b2b): planner (mp_planner.cpp) and launch
// (mp_gemm.cu).
struct B2BArgs {
    int64_t M, N0, N1, K0;
    const void* A0; int64_t lda0;
    const void* W0; int64_t ldw0;
    const float* C0; int64_t ldc0;
    const void* W1; int64_t ldw1;
    const float* C1; int64_t ldc1;
    float* D1; int64_t ldd1;
    float alpha0, beta0, alpha1, beta1;
    int32_t act0;
    void* stream;
};
mp_status plan_b2b(const mp_hw& hw, int64_t M, int64_t N0, int64_t N1, int64_t K0, mp_b2b_plan* out);
mp_status device_run_b2b(mp_handle h, const mp_b2b_plan& plan, const B2BArgs& a);
// The same pair as two launches through a bf16 scratch buffer for D0.
mp_status device_run_b2b_two(mp_handle h, const B2BArgs& a);

// Implicit-GEMM convolution (mp_conv2d): planner (mp_planner.cpp) and launch
// (mp_gemm.cu).
struct ConvArgs {
    int64_t N, H, W, C, K, R, S, pad_h, pad_w;
    const void* X;
    const void* F;
    const float* Cin; int64_t ldc;
    float* D; int64_t ldd;
    float alpha, beta;
    void* stream;
};
mp_status plan_conv(const mp_hw& hw, int64_t ws_floats, int64_t N, int64_t H, int64_t W, int64_t C, int64_t K,
                    int64_t R, int64_t S, int64_t pad_h, int64_t pad_w, mp_conv_plan* out);
mp_status device_run_conv(mp_handle h, const mp_conv_plan& plan, const ConvArgs& a);

// Grouped GEMM (mp_gemm_grouped): planner (mp_planner.cpp) and launches
// (mp_gemm.cu).  `probs` holds only non-empty problems.
mp_status plan_grouped(const mp_hw& hw, int32_t count, const mp_gemm_problem* probs, mp_grouped_plan* out);
mp_status device_run_grouped(mp_handle h, const mp_grouped_plan& plan, int32_t count, const mp_gemm_problem* probs,
                             void* stream);

}  // namespace mp
