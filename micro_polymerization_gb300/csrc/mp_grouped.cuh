// Grouped GEMM: up to kMaxGroup independent problems of different shapes in
// one launch, D_i = alpha_i * A_i B_i + beta_i * C_i.  The BladeDISC v0.2.0
// notes merge GEMMs to fill the machine and to launch fewer kernels, for
// same-shape problems (a batched GEMM); a group drops that condition.  In
// the terms of the MikPoly summary each problem's output is a region of one
// polymerized program: every problem is cut into 128 x bn tiles of the one
// micro-kernel the plan picks, and the persistent CTAs walk all tiles of all
// problems.
//
// The problem table travels in the kernel parameters (tensor maps included,
// so TMA reads them from parameter space, as in the other kernels): nothing
// is copied to the device before the launch.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace mp {
namespace grp {

constexpr int kMaxGroup = 48;                   // problems per launch (kernel parameters <= 32 KB)
constexpr int kThreads = 224;                   // warps 0, 6 TMA, warp 1 MMA + TMEM, warps 2..5 epilogue
constexpr int kMaxStages = 8;
constexpr int kEpiSlabBytes = 2 * 32 * 32 * 4;  // two 32 x 32 fp32 slabs per epilogue warp
constexpr int kSmemLimit = 232448;

struct alignas(128) Problem {
    CUtensorMap tmA;  // A [M][K] bf16, box {64, 128}
    CUtensorMap tmB;  // B [K][N] bf16, box {64, 64}
    CUtensorMap tmD;  // D [M][N] fp32, box {32, 32} (bulk stores, when tma_d)
    const float* C;
    float* D;
    long long ldc, ldd;
    int M, N, K;
    int tiles_n;      // ceil(N / bn)
    int tile0;        // first unit of this problem (prefix sum of tiles)
    float alpha, beta;
    int tma_d, vec_c;
};

struct alignas(128) Params {
    Problem prob[kMaxGroup];
    int count;
    int units;        // tiles of all problems
    int bn;           // output columns per tile (64, 128 or 256)
    int num_stages, stage_bytes;
    int* err;
    unsigned long long wait_limit_ns;
    int inject_timeout;  // test hook: producer warp 0 withholds its first stage
    // K steps of A and B the first epilogue warp prefetches into L2 for its
    // CTA's first tile (when that problem reads no C) before waiting for the
    // previous kernel (0: none).
    int l2_pf;
};

inline int smem_bytes(int num_stages, int stage_bytes) {
    return num_stages * stage_bytes + 4 * kEpiSlabBytes + 1024 + 1024;
}

cudaError_t launch(const cudaLaunchConfig_t& cfg, const Params& p);
bool set_smem();

}  // namespace grp
}  // namespace mp
