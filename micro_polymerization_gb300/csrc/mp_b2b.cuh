// Back-to-back GEMMs in one persistent kernel (BOLT summary, "Persistent
// kernel (GEMM/Conv) fusion"):
//   D0 = act0(alpha0 * A0 W0 + beta0 * C0)      (kept on chip, bf16)
//   D1 = alpha1 * D0 W1 + beta1 * C1
// The summary's key property is threadblock residence: the thread block that
// produces a block of D0 rows also consumes it as the A operand of the second
// GEMM, from its own shared memory, so D0 never goes to global memory.  That
// needs every column of D0 in the block: N0 <= 256 (one TMEM accumulator).
//
// Work unit: 128 rows of M x a group of `cpg` consecutive chunks of bn1
// columns of D1 (unit u: row block u / groups, group u % groups).  A unit computes its 128 x N0 block of D0 once (first GEMM
// into TMEM, epilogue warps convert it into the second GEMM's K-major
// 128-byte-swizzled operand in shared memory), then each chunk of D1 (second
// GEMM into TMEM, epilogue to global memory).  Several groups of one row
// block recompute D0 when that fills more SMs (the host's cost model picks
// the grouping).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace mp {
namespace b2b {

constexpr int kThreads = 224;               // warps 0, 6 TMA, warp 1 MMA + TMEM, warps 2..5 epilogue
constexpr int kMaxStages = 8;
constexpr int kEpiSlabBytes = 2 * 32 * 16 * 4;  // two 32 x 16 fp32 boxes per epilogue warp
constexpr int kSmemLimit = 232448;          // dynamic shared memory per CTA (227 KB)

struct alignas(128) Params {
    CUtensorMap tmA0;  // A0 [M][K0] bf16, box {64, 128}
    CUtensorMap tmW0;  // W0 [K0][N0] bf16, box {64, 64}
    CUtensorMap tmW1;  // W1 [N0][N1] bf16, box {64, 64}
    CUtensorMap tmD1;  // D1 [M][N1] fp32, box {16, 32}, 64-byte swizzle (bulk stores, when tma_d)
    const float* C0;
    const float* C1;
    float* D1;
    long long ldc0, ldc1, ldd1;
    int M, N0, N1, K0;  // K0 is 0 when N0 is 0 (no first GEMM)
    int n0p;            // N0 rounded up to 64: the first GEMM's N, the second's K
    int bn1;            // D1 columns per chunk (64..256)
    int chunks;         // ceil(N1 / bn1)
    int mblocks;        // ceil(M / 128)
    int cpg;            // chunks per work unit
    int units;          // mblocks * ceil(chunks / cpg)
    int num_stages, stage_bytes;
    float alpha0, beta0, alpha1, beta1;
    int act0;            // activation on D0: 0 none, 1 ReLU, 2 GELU
    int tma_d;           // D1 rows 16-byte aligned: bulk tensor stores
    int vec_c0, vec_c1;  // C rows allow 16-byte loads
    int* err;            // the handle's status word
    unsigned long long wait_limit_ns;
    int inject_timeout;  // test hook: producer warp 0 withholds its first stage
    // K steps of A0 and W0 the first epilogue warp prefetches into L2 for its
    // CTA's first unit before waiting for the previous kernel (0: none).
    int l2_pf;
};

// Dynamic shared memory of a launch: operand ring, D0 operand (128 rows of
// n0p bf16), epilogue slabs, barriers, and 1 KB for the alignment of the base.
inline int smem_bytes(int num_stages, int stage_bytes, int n0p) {
    return num_stages * stage_bytes + n0p * 256 + 4 * kEpiSlabBytes + 1024 + 1024;
}

cudaError_t launch(const cudaLaunchConfig_t& cfg, const Params& p);
bool set_smem();

}  // namespace b2b
}  // namespace mp
