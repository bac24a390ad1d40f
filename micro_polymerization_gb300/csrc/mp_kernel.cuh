// Device side: one persistent kernel that runs a whole polymerization plan.
//
// Each CTA (one per SM) walks the plan's work units -- (region, tile, split)
// triples -- in a static round-robin.  Every unit is a pipeline task in the
// sense of the MikPoly summary, section 3 ("micro-kernel performance
// model"): its K loop is serial on one PE and runs in three stages,
//   (1) load the operand tiles into the PE's local memory  -> TMA producer warp
//   (2) run the micro-kernel on them                       -> tcgen05.mma issuer
//   (3) write the result back                              -> epilogue warps
// overlapped through an mbarrier ring of shared-memory stages and two TMEM
// accumulator buffers.  Offsets and loop counts of the fixed-size
// micro-kernels arrive as run-time scalars (MikPoly summary, section 4).  The
// epilogue applies D = alpha*acc + beta*C (BOLT summary, persistent kernel
// fusion) with masking at the region edges, so any (M, N, K) runs in one
// launch without per-shape compilation.
//
// Micro-kernel forms (both with a 128-lane fp32 accumulator in TMEM):
//   normal:  acc[128 x bn] = A_tile[128 x K] * B_tile[K x bn]
//            A is K-major (row-major A), B is MN-major (row-major B).
//   swapped: acc[128 x bn] = B_tile^T[128 x K] * A_tile^T[K x bn], i.e. the
//            transpose of a bn x 128 block of D, for short M: the UMMA M runs
//            over N and bn (16..128) over M.
// Operand tiles use the 128-byte swizzle: one swizzle row holds 64 bf16, so
// a stage carries 64 elements of K.
//
// Warp roles (192 threads):  warp 0 = TMA producer, warp 1 = TMEM owner and
// MMA issuer, warps 2..5 = epilogue (warp w reads TMEM lanes 32*(w%4)..+31).
// Every wait is bounded: on expiry the CTA records an error code in the
// handle's status word, tells its other roles to stop, waits (bounded) for
// its own copies and MMAs in flight, frees TMEM and returns.
#pragma once

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

namespace mp {
namespace dev {

// Shared-memory ring: each stage holds one X tile (16 KB) and one Y tile of
// the plan's widest micro-kernel (bn x 64 bf16), so narrow plans get more
// stages in flight: 4 at bn = 256, 6 at 128, 8 at 64, 10 at 16.
constexpr int kXBytes = 128 * 64 * 2;   // 128 rows (or 128 columns of B^T) x 64 K, bf16
constexpr int kRingBytes = 4 * (kXBytes + 256 * 64 * 2);
constexpr int kMaxStages = 12;
constexpr int kThreads = 224;           // 7 warps: producer, MMA, 4 epilogue, producer
constexpr int kProducer2Warp = 6;
constexpr int kTmemCols = 512;          // two accumulator buffers of 256 columns
constexpr int kAccStride = 256;
// Epilogue staging, 8 KB per epilogue warp: two 32 x 32 fp32 slabs for bulk
// tensor stores of D (the 16-column transposes use the first 2 KB).
constexpr int kEpiWarpBytes = 2 * 32 * 32 * 4;
constexpr int kStageBytesEpi = 4 * kEpiWarpBytes;
constexpr int kBarBytes = 1024;  // mbarriers, flags and the region table
constexpr int kSmemBytes = kRingBytes + kStageBytesEpi + kBarBytes + 1024;

// Error codes written to the status word (first writer wins).
constexpr int kErrWaitEmpty = 1;
constexpr int kErrWaitFull = 2;
constexpr int kErrWaitAccEmpty = 3;
constexpr int kErrWaitAccFull = 4;
constexpr int kErrDrain = 5;
constexpr int kErrWaitSplits = 6;

struct Region {
    int m0, n0, m_end, n_end;   // region bounds in D
    int tiles_m, tiles_n;
    int bn;                     // UMMA N (normal: columns of D; swapped: rows of D)
    int swap;
    int splits, kb_per_split;
    int unit_begin, units;
    long long ws_begin;         // first fp32 of this region's split-K partials
    int cnt_begin;              // first tile counter
    // Tile order: groups of `group` tile rows, column by column inside a
    // group, so that the tiles in flight at once share their rows of A and
    // columns of B in L2 (1: row by row).
    int group;
};

struct alignas(128) Params {
    CUtensorMap tmA;     // A viewed as [batch][M][K] bf16, box {64 (K), 128 rows}
    CUtensorMap tmAs;    // same tensor, box {64 (K), as_rows rows}: A of swapped tiles
    CUtensorMap tmB;     // B viewed as [batch][K][N] bf16, box {64 (N), 64 rows of K}
    // B viewed as [batch][N/64 full blocks][K][64]: box {64, 64 (K), j+1 blocks}
    // fetches j+1 adjacent 64-column blocks in one copy (encoded when used).
    CUtensorMap tmB4[4];
    // B with the 64-byte swizzle, box {32 (N), 64 rows of K}: the 96-column
    // halves of 256 x 192 pair tiles, in atoms of 32 columns (encoded when used).
    CUtensorMap tmBs;
    int bs_ok;           // 1: tmBs is encoded
    int nb_full;         // floor(N / 64): blocks tmB4 may address
    int b4_mask;         // bit j: tmB4[j] is encoded (prefetched at set-up)
    int as_rows;         // rows per A box of swapped tiles (divides every swapped bn)
    const float* C;
    float* D;
    long long ldc, ldd, strideC, strideD;
    float alpha, beta;
    int num_kb;          // ceil(K / 64)
    int a_bstep, b_bstep;
    int total_units;
    int num_regions;
    int inject_timeout;  // test hook: 1 withholds the first stage of the first unit; 2 makes the
                         // ring-staged split-K sums wait for 16 bytes that never come
    int vec_c, vec_d;    // C / D rows allow 16-byte (fp32 D) or 8-byte (bf16 D) vector access
    int act;             // activation on alpha*acc + beta*C: 0 none, 1 ReLU, 2 GELU (erf form)
    int out_bf16;        // 1: D is bf16 (round to nearest even), else fp32
    CUtensorMap tmD;     // D viewed as [batch][M][N] fp32, box {32 (N), 32 rows}, 128-byte swizzle
    // Split-K partials of region i viewed as [tiles*splits*128 rows][bn] fp32,
    // box {32, 32}, 128-byte swizzle (encoded for split regions of normal tiles).
    CUtensorMap tmW[MP_MAX_REGIONS];
    int w_mask;          // bit i: tmW[i] is encoded
    int tma_d;           // 1: normal tiles store D through tmD (beta == 0, rows 16-byte aligned)
    int num_stages;      // shared-memory ring depth for this plan
    int sub_bytes;       // one 64-deep K step: 16 KB X tile + the widest Y tile of the plan
    int kg;              // K steps per ring stage (1 or 2): one full/empty barrier pair per stage
    int stage_bytes;     // kg * sub_bytes
    // S > 1: split-K on chip.  Clusters of S CTAs, one task each (unit =
    // tile * S + split = blockIdx.x); each CTA leaves its partial in its
    // shared memory and the cluster reduces it through distributed shared
    // memory at the end of the kernel.
    int csplit;
    // 1: clusters of two CTAs; a work unit is two vertically adjacent tiles
    // (rank r takes tile row 2 t + r) that share their B tile, each CTA
    // multicasting half of B's 64-column blocks into both shared memories.
    int pair;
    // One-CTA launches: the first epilogue warp prefetches into L2 the first
    // l2_pf K steps of A and B of its CTA's first unit before waiting for the
    // previous kernel (0: no prefetch).
    int l2_pf;
    unsigned long long wait_limit_ns;
    Region reg[MP_MAX_REGIONS];
    float* ws;
    unsigned int* cnt;
    int* err;
};

struct Work {
    int b, split, splits;
    int m_t0, n_t0, m_end, n_end;
    int bn, swap;
    int kb0, kb1;
    long long ws_tile;   // split 0 of this tile's partials
    int cnt;
    int r;               // region index
    int ws_row;          // first row of this split's partial in the region's [rows][bn] view
};

// `regs` is the shared-memory copy of p.reg made during set-up.
// In paired launches `u` counts tile pairs and `rank` picks the pair's tile.
__device__ __forceinline__ Work decode(const Params& p, const Region* regs, int u, int rank) {
    int r = 0;
#pragma unroll
    for (int i = 1; i < MP_MAX_REGIONS; i++)
        if (i < p.num_regions && u >= regs[i].unit_begin) r = i;
    const Region& g = regs[r];
    const int local = u - g.unit_begin;
    const int tiles = g.tiles_m * g.tiles_n;
    const int per_b = tiles * g.splits;
    Work w;
    w.b = local / per_b;
    const int rem = local - w.b * per_b;
    const int tile = rem / g.splits;
    w.split = rem - tile * g.splits;
    w.splits = g.splits;
    int tm, tn;
    if (g.group > 1) {
        const int per_group = g.group * g.tiles_n;
        const int gi = tile / per_group;
        const int first = gi * g.group;
        const int rows = min(g.tiles_m - first, g.group);
        const int in = tile - gi * per_group;
        tn = in / rows;
        tm = first + (in - tn * rows);
    } else {
        tm = tile / g.tiles_n;
        tn = tile - tm * g.tiles_n;
    }
    w.swap = g.swap;
    w.bn = g.bn;
    if (!g.swap) {
        w.m_t0 = g.m0 + (p.pair ? 2 * tm + rank : tm) * 128;
        w.n_t0 = g.n0 + tn * g.bn;
    } else {
        w.m_t0 = g.m0 + tm * g.bn;
        w.n_t0 = g.n0 + tn * 128;
    }
    w.m_end = g.m_end;
    w.n_end = g.n_end;
    w.kb0 = w.split * g.kb_per_split;
    w.kb1 = min(w.kb0 + g.kb_per_split, p.num_kb);
    const long long tile_id = (long long)w.b * tiles + tile;
    w.ws_tile = g.ws_begin + tile_id * g.splits * (128ll * g.bn);
    w.cnt = g.cnt_begin + (int)tile_id;
    w.r = r;
    w.ws_row = (int)((tile_id * g.splits + w.split) * 128);
    return w;
}

// ---------------------------------------------------------------------------
// PTX wrappers (PTX ISA: mbarrier, cp.async.bulk.tensor, tcgen05)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Untiled bulk copy global -> shared memory (both 16-byte aligned, `bytes` a
// multiple of 16), completing `bytes` transactions on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of parity `parity` of `bar` to complete, for at most
// `limit_ns`.  With `honor_abort`, also give up as soon as another role of
// the CTA has aborted.  On expiry, raise the CTA's abort flag and record
// `code` in the status word.
static __device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* err, int code, uint64_t limit_ns, bool honor_abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (honor_abort && *abort_flag) return false;
        if (globaltimer() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicCAS(err, 0, code);
            return false;
        }
    }
}

// Non-blocking probe of a phase (mbarrier.test_wait never suspends).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Inline fast path: one non-blocking probe, then the bounded slow path.
__device__ __forceinline__ bool wait_fast(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* err,
                                          int code, uint64_t limit_ns) {
    if (mbar_test_wait(bar, parity)) return true;
    return wait_bounded(bar, parity, abort_flag, err, code, limit_ns, true);
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                            int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                            int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// Copies of the odd CTA of a pair: the box lands in this CTA's shared memory
// and completes its bytes on the even CTA's barrier (`bar`, a cluster address
// from mapa), where that CTA's MMA issuer waits for both halves.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                                 int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0,
                                                 int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster: arrive (release) and wait (acquire).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bulk tensor store of a shared-memory box to global memory (bulk-group
// completion); rows and columns outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most one bulk group of this thread is still reading shared memory.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Every bulk store this thread issued has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Generic-proxy writes to shared memory become visible to the async proxy (TMA).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 prefetch of one tensor box (the coordinates a load of the same box
// would take); nothing reaches shared memory and nothing is waited for.
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
}

// TMEM allocation.  CG = 1: one warp of the CTA; CG = 2: one warp of each
// CTA of the pair, together (both receive the same address).  A kernel uses
// one CTA group for all its tcgen05 operations.
template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    if constexpr (CG == 1)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                     : "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_relinquish() {
    if constexpr (CG == 1)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    if constexpr (CG == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], bf16 inputs, fp32 accumulate.
// CG = 2: issued by the even CTA of a pair for both; each CTA holds its half
// of A's rows and of B's columns at the same shared-memory offsets, and
// receives its half of D's rows at the same TMEM address.
template <int CG = 1>
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    if constexpr (CG == 1)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Arrive (once) on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Pair version: arrive, once every tcgen05 operation issued so far by this
// thread has completed, on the barrier at `bar`'s offset in every CTA of
// `mask` (cluster ranks).
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(mask)
        : "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// 16 bytes of another CTA's shared memory (address from mapa).
__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t cluster_addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(cluster_addr)
                 : "memory");
    return v;
}

// Arrive on a barrier of another CTA of the cluster (address from mapa).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// 16 consecutive accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    // The wait names the registers so that no use is scheduled above it.
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                   "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, and the swizzle
// mode (2: 128-byte, 4: 64-byte).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz = 2) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)swz << 61;
    return d;
}

// K-major operand: rows of 64 bf16 (128 B) with 8-row swizzle atoms 1024 B
// apart; one UMMA K step (16 elements) advances 32 B inside the row.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kstep) {
    return smem_desc(tile + 32u * kstep, 16u, 1024u);
}

// MN-major operand: atoms of 64 MN elements x 8 K rows (1024 B); K groups of
// 8 rows 1024 B apart, 64-wide MN blocks 8192 B apart (one TMA box each); one
// UMMA K step (16 rows) advances 2048 B.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int kstep) {
    return smem_desc(tile + 2048u * kstep, 8192u, 1024u);
}

// MN-major operand with the 64-byte swizzle: atoms of 32 MN elements x 8 K
// rows (512 B); K groups of 8 rows 512 B apart, 32-wide MN blocks 4096 B
// apart (one TMA box each); one UMMA K step (16 rows) advances 1024 B.
__device__ __forceinline__ uint64_t desc_mnmajor64(uint32_t tile, int kstep) {
    return smem_desc(tile + 1024u * kstep, 4096u, 512u, 4u);
}

// Instruction descriptor, kind::f16: fp32 D, bf16 A and B, M = m (128, or
// 256 for a CTA pair), N = n.
__device__ __forceinline__ uint32_t idesc_bf16(int n, bool a_mn, bool b_mn, int m = 128) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// ---------------------------------------------------------------------------
// Epilogue store of 16 accumulator columns of one TMEM lane
// ---------------------------------------------------------------------------
// Epilogue variants are compile-time: EPI bits 0-1 name the activation (0
// none, 1 ReLU, 2 GELU), bit 2 a bf16 D.  Each EPI is its own instantiation
// of the kernel, so the plain alpha/beta epilogue (EPI 0) keeps its registers
// and instruction stream and a variant carries only its own code.
template <int EPI>
__host__ __device__ constexpr int epi_act() {
    return EPI & 3;
}
template <int EPI>
__host__ __device__ constexpr bool epi_bf16() {
    return (EPI & 4) != 0;
}

// GELU(x) = x Phi(x), Phi(x) = (1 + erf(x / sqrt 2)) / 2.  erfc on z >= 0 is
// Hastings' rational approximation (Abramowitz and Stegun, Handbook of
// Mathematical Functions, formula 7.1.26; |error in erf| <= 1.5e-7):
//   erfc(z) ~ t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2),  t = 1 / (1 + p z),
// one reciprocal and one exponential, so that the activation costs a few
// instructions per element of the epilogue.  Phi takes erfc for x < 0 and
// 1 - erfc/2 for x >= 0, so the negative tail keeps its relative accuracy.
__device__ __forceinline__ float gelu_f32(float x) {
    const float z = fabsf(x) * 0.70710678118654752f;
    const float t = __fdividef(1.0f, fmaf(0.3275911f, z, 1.0f));
    float y = fmaf(t, 1.061405429f, -1.453152027f);
    y = fmaf(t, y, 1.421413741f);
    y = fmaf(t, y, -0.284496736f);
    y = fmaf(t, y, 0.254829592f);
    const float half_erfc = 0.5f * t * y * __expf(-z * z);
    return x * (x >= 0.0f ? 1.0f - half_erfc : half_erfc);
}

// The activation of the epilogue, applied to alpha*acc + beta*C.
template <int EPI>
__device__ __forceinline__ float act_fn(float x) {
    if constexpr (epi_act<EPI>() == 0) return x;
    if constexpr (epi_act<EPI>() == 1) return fmaxf(x, 0.0f);
    return gelu_f32(x);
}

// D is addressed in bytes: an element is 4 bytes (fp32), or 2 in the bf16-D
// instantiations, and row pointers advance by ldd elements of that size.
template <int EPI>
__device__ __forceinline__ int d_esize(const Params&) {
    return epi_bf16<EPI>() ? 2 : 4;
}
template <int EPI>
__device__ __forceinline__ uint8_t* d_ptr(const Params& p, long long off) {
    return reinterpret_cast<uint8_t*>(p.D) + off * d_esize<EPI>(p);
}

// One output element at byte address `d` of D (fp32 or bf16).
template <int EPI>
__device__ __forceinline__ void put_out(const Params& p, uint8_t* d, float x) {
    if constexpr (epi_bf16<EPI>())
        *reinterpret_cast<__nv_bfloat16*>(d) = __float2bfloat16_rn(x);
    else
        *reinterpret_cast<float*>(d) = x;
}

// Four consecutive elements (16-byte fp32 or 8-byte bf16 store; the caller
// has checked the alignment).
template <int EPI>
__device__ __forceinline__ void put_out4(const Params& p, uint8_t* d, float x0, float x1, float x2, float x3) {
    if constexpr (epi_bf16<EPI>()) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(x0, x1), hi = __floats2bfloat162_rn(x2, x3);
        uint2 u;
        u.x = *reinterpret_cast<const uint32_t*>(&lo);
        u.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(d) = u;
    } else {
        *reinterpret_cast<float4*>(d) = make_float4(x0, x1, x2, x3);
    }
}

// Swapped tile: TMEM lane tl is column n_t0 + tl of D, and the 16 values
// are rows m_t0 + c .. + 15 (a warp's stores of one row cover 128
// contiguous bytes).  All 16 values of C are loaded before the first store:
// C may be D itself (in place), so a load after a store could not be moved
// ahead of it and the loads would wait for each other; each element of D
// depends only on its own element of C, so reading them all first gives the
// same result.
template <int EPI>
__device__ __forceinline__ void store16(const Params& p, const Work& w, int tl, int c, const float* v) {
    const float alpha = p.alpha, beta = p.beta;
    const int n = w.n_t0 + tl;
    if (n >= w.n_end) return;
    uint8_t* bd = d_ptr<EPI>(p, (long long)w.b * p.strideD + n);
    const long long ldd_b = p.ldd * d_esize<EPI>(p);
    const long long bc = (long long)w.b * p.strideC + n;
    float cv[16];
    if (beta != 0.0f) {
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const int m = w.m_t0 + c + j;
            cv[j] = m < w.m_end ? p.C[bc + (long long)m * p.ldc] : 0.0f;
        }
    }
#pragma unroll
    for (int j = 0; j < 16; j++) {
        const int m = w.m_t0 + c + j;
        if (m < w.m_end) {
            float r = alpha * v[j];
            if (beta != 0.0f) r = fmaf(beta, cv[j], r);
            put_out<EPI>(p, bd + (long long)m * ldd_b, act_fn<EPI>(r));
        }
    }
}

// Four consecutive columns n..n+3 of row m of D (vector access when allowed).
// Same arithmetic as store16: alpha*acc, then fma with beta*C.
template <int EPI>
__device__ __forceinline__ void store4(const Params& p, const Work& w, int m, int n, float4 x) {
    if (n >= w.n_end) return;
    const float alpha = p.alpha, beta = p.beta;
    uint8_t* d = d_ptr<EPI>(p, (long long)w.b * p.strideD + (long long)m * p.ldd + n);
    const float* cp = p.C + (long long)w.b * p.strideC + (long long)m * p.ldc + n;
    float o[4] = {alpha * x.x, alpha * x.y, alpha * x.z, alpha * x.w};
    if (p.vec_d && n + 3 < w.n_end) {
        if (beta != 0.0f) {
            float4 cv;
            if (p.vec_c) {
                cv = *reinterpret_cast<const float4*>(cp);
            } else {
                cv = make_float4(cp[0], cp[1], cp[2], cp[3]);
            }
            o[0] = fmaf(beta, cv.x, o[0]);
            o[1] = fmaf(beta, cv.y, o[1]);
            o[2] = fmaf(beta, cv.z, o[2]);
            o[3] = fmaf(beta, cv.w, o[3]);
        }
        put_out4<EPI>(p, d, act_fn<EPI>(o[0]), act_fn<EPI>(o[1]), act_fn<EPI>(o[2]), act_fn<EPI>(o[3]));
    } else {
#pragma unroll
        for (int e = 0; e < 4; e++) {
            if (n + e < w.n_end) {
                float r = o[e];
                if (beta != 0.0f) r = fmaf(beta, cp[e], r);
                put_out<EPI>(p, d + e * d_esize<EPI>(p), act_fn<EPI>(r));
            }
        }
    }
}

// Write accumulator columns [c, c+16) of this thread's TMEM lane to D.
//   normal tiles (lane = row of D): the warp's 32 x 16 block is staged in
//   shared memory -- rows of 64 B, 16-byte groups XOR-swizzled so that both
//   the row-wise writes and the transposed reads are free of bank conflicts
//   -- and read back so that each store instruction covers 8 rows x 64
//   contiguous bytes instead of 32 scattered rows.
//   swapped tiles (lane = column of D): each store already covers 32
//   consecutive columns of one row.
// Transpose a warp's 32 x 16 block (lane = row, v = its 16 columns) through
// `stage` and hand it back as (row r, column group g, 4 values) so that the
// 32 lanes of one call cover 8 rows x 4 groups.
template <class Sink>
__device__ __forceinline__ void transpose16(int lane, const float* v, float4* stage, Sink sink) {
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int i = 0; i < 4; i++)
        stage[lane * 4 + (i ^ sw)] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    __syncwarp();
    const int g = lane & 3;
#pragma unroll
    for (int it = 0; it < 4; it++) {
        const int r = it * 8 + (lane >> 2);
        sink(r, g, stage[r * 4 + (g ^ ((r >> 1) & 3))]);
    }
    __syncwarp();
}

// beta * C for a normal tile's 32-column chunk c: lane = column n_t0 + c +
// lane, cv[r] = row m_t0 + 32 q + r (0 outside the region).  All 32 loads are
// issued before any is used, and the caller issues them before the chunk's
// TMEM load: one memory round trip per chunk.
__device__ __forceinline__ void load_c_cols(const Params& p, const Work& w, int q, int lane, int c, float* cv) {
    const int n = w.n_t0 + c + lane;
    const int mb = w.m_t0 + q * 32;
    const int rows = min(32, w.m_end - mb);
    const float* cr = p.C + (long long)w.b * p.strideC + (long long)mb * p.ldc + n;
    const bool in_n = n < w.n_end;
#pragma unroll
    for (int r = 0; r < 32; r++) {
        cv[r] = (in_n && r < rows) ? *cr : 0.0f;
        cr += p.ldc;
    }
}

// Normal tile whose D rows are not 16-byte aligned (no tensor map; any
// alignment): the warp's 32 rows x 32 columns go through its shared-memory
// slab (128-byte swizzle, conflict-free both ways) and come back one row at
// a time with lane = column, so that every store instruction covers 128
// contiguous bytes of one row of D.  cv: the chunk's beta * C operand
// (load_c_cols), unused when beta == 0.  Same arithmetic as the other paths.
template <int EPI>
__device__ __forceinline__ void emit32_rows(const Params& p, const Work& w, int q, int lane, int c, const float* v,
                                            const float* cv, uint8_t* slab) {
    const float a = p.alpha, bt = p.beta;
    const int n = w.n_t0 + c + lane;
    const bool in_n = n < w.n_end;
    const int mb = w.m_t0 + q * 32;
    const int rows = min(32, w.m_end - mb);
    __syncwarp();  // the previous chunk's reads of the slab are done
    uint8_t* row = slab + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; j++)
        *reinterpret_cast<float4*>(row + ((j ^ (lane & 7)) << 4)) =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    __syncwarp();
    const uint8_t* src = slab + (lane & 3) * 4;
    uint8_t* dp = d_ptr<EPI>(p, (long long)w.b * p.strideD + (long long)mb * p.ldd + n);
    const long long ldd_b = p.ldd * d_esize<EPI>(p);
#pragma unroll
    for (int r = 0; r < 32; r++) {
        if (r >= rows) break;
        const float x = *reinterpret_cast<const float*>(src + r * 128 + (((lane >> 2) ^ (r & 7)) << 4));
        if (in_n) {
            float o = a * x;
            if (bt != 0.0f) o = fmaf(bt, cv[r], o);
            put_out<EPI>(p, dp, act_fn<EPI>(o));
        }
        dp += ldd_b;
    }
}

// L2 prefetch of the C rows a normal tile's epilogue will read (thread =
// row of the tile, any alignment), issued before the accumulator is ready.
__device__ __forceinline__ void prefetch_c_tile_row(const Params& p, const Work& w, int m) {
    if (m >= w.m_end) return;
    const float* cr = p.C + (long long)w.b * p.strideC + (long long)m * p.ldc + w.n_t0;
    const int cols = min(w.bn, w.n_end - w.n_t0);
    for (int c = 0; c < cols + 31; c += 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(cr + min(c, cols - 1)));
}

template <int EPI>
__device__ __forceinline__ void emit16(const Params& p, const Work& w, int q, int lane, int c, const float* v,
                                       float4* stage) {
    if ((EPI & 24) == 0 && w.swap) {  // the lean instantiations have no swapped tiles
        store16<EPI>(p, w, q * 32 + lane, c, v);
        return;
    }
    transpose16(lane, v, stage, [&](int r, int g, float4 x) {
        const int m = w.m_t0 + q * 32 + r;
        if (m < w.m_end) store4<EPI>(p, w, m, w.n_t0 + c + 4 * g, x);
    });
}

// Normal tile, beta == 0: write alpha * (32 accumulator columns of this
// lane's row) into a 32 x 32 fp32 slab with the 128-byte swizzle (16-byte
// group j of row r at r*128 + ((j ^ (r & 7)) << 4): conflict-free, and the
// layout a swizzled tensor store expects), then one lane stores the slab to
// D(m0 .. m0+31, n0 .. n0+31) with a bulk tensor copy.  Two slabs alternate;
// before a slab is rewritten, the store that last read it must have finished
// reading.
// C for the same 32 x 32 block, one row per lane (zero outside the region);
// issued before the TMEM load of the chunk so that both latencies overlap.
template <int W>
__device__ __forceinline__ void load_c(const Params& p, const Work& w, int lane, int m0, int n0, float* c) {
    const int m = m0 + lane;
    if (m < w.m_end) {
        const float* cr = p.C + (long long)w.b * p.strideC + (long long)m * p.ldc + n0;
        if (p.vec_c && n0 + W <= w.n_end) {
#pragma unroll
            for (int j = 0; j < W / 4; j++) {
                const float4 x = __ldg(reinterpret_cast<const float4*>(cr) + j);
                c[4 * j] = x.x;
                c[4 * j + 1] = x.y;
                c[4 * j + 2] = x.z;
                c[4 * j + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < W; j++) c[j] = n0 + j < w.n_end ? __ldg(cr + j) : 0.0f;
        }
    } else {
#pragma unroll
        for (int j = 0; j < W; j++) c[j] = 0.0f;
    }
}

__device__ __forceinline__ void load_c32(const Params& p, const Work& w, int lane, int m0, int n0, float* c) {
    load_c<32>(p, w, lane, m0, n0, c);
}

// Swapped tile: ask L2 for the block of C its epilogue will read before the
// accumulator is ready.  Warp quarter q stores D columns n_t0 + 32 q .. + 31
// (one 128-byte line of a row); lane l asks for rows l, l + 32, ... of the
// tile's w.bn rows.
__device__ __forceinline__ void prefetch_c_swapped(const Params& p, const Work& w, int q, int lane) {
    const int n = w.n_t0 + 32 * q;
    if (n >= w.n_end) return;
    const float* cb = p.C + (long long)w.b * p.strideC + n;
    for (int r = lane; r < w.bn && w.m_t0 + r < w.m_end; r += 32)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(cb + (long long)(w.m_t0 + r) * p.ldc));
}

// Ask L2 for this lane's row of C over the whole tile (one 128-byte line per
// 32 columns) before the accumulator is ready.
__device__ __forceinline__ void prefetch_c_row(const Params& p, const Work& w, int m) {
    if (m >= w.m_end) return;
    const float* cr = p.C + (long long)w.b * p.strideC + (long long)m * p.ldc + w.n_t0;
    for (int c = 0; c < w.bn && w.n_t0 + c < w.n_end; c += 32)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(cr + c));
}

template <int EPI>
__device__ __forceinline__ void emit32_tma(const Params& p, const Work& w, int lane, int m0, int n0,
                                           const float* v, const float* c, uint8_t* slab, uint32_t slab_s) {
    if (lane == 0) bulk_wait_read_1();
    __syncwarp();
    const float a = p.alpha, bt = p.beta;
    uint8_t* row = slab + lane * 128;
    if (epi_act<EPI>() == 0 && ((EPI & 8) != 0 || bt == 0.0f)) {
#pragma unroll
        for (int j = 0; j < 8; j++)
            *reinterpret_cast<float4*>(row + ((j ^ (lane & 7)) << 4)) =
                make_float4(a * v[4 * j], a * v[4 * j + 1], a * v[4 * j + 2], a * v[4 * j + 3]);
    } else {
        // Same arithmetic as the other epilogue paths: fma(beta, C, alpha*acc),
        // then the activation.
#pragma unroll
        for (int j = 0; j < 8; j++) {
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                o[e] = a * v[4 * j + e];
                if ((EPI & 8) == 0 && (EPI == 0 || bt != 0.0f))  // EPI 0 (not lean): bt != 0 here
                    o[e] = fmaf(bt, c[4 * j + e], o[e]);
                o[e] = act_fn<EPI>(o[e]);
            }
            *reinterpret_cast<float4*>(row + ((j ^ (lane & 7)) << 4)) = make_float4(o[0], o[1], o[2], o[3]);
        }
    }
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_3d(&p.tmD, slab_s, n0, m0, w.b);
        bulk_commit_group();
    }
}

// Split-K partials are kept "D-row-major" per tile: a buffer of R rows x L
// columns where element (r, l) belongs to D(m_t0 + r, n_t0 + l).  Normal
// tiles: R = 128 (TMEM lanes), L = bn.  Swapped tiles: R = bn (TMEM
// columns), L = 128 (TMEM lanes).
__device__ __forceinline__ void park16(const Work& w, int q, int lane, int c, const float* v, float4* stage,
                                       float* part) {
    if (w.swap) {
        // lane = column l of the buffer, v = rows c..c+15: 128 B per store.
#pragma unroll
        for (int j = 0; j < 16; j++) __stcg(part + (c + j) * 128 + q * 32 + lane, v[j]);
        return;
    }
    transpose16(lane, v, stage, [&](int r, int g, float4 x) {
        __stcg(reinterpret_cast<float4*>(part + (q * 32 + r) * w.bn + c + 4 * g), x);
    });
}

// Rows [r0, r1) of a split tile: sum the S partials in split order and write
// D.  Consecutive threads take consecutive 16-byte groups of a row.
template <int EPI>
__device__ __forceinline__ void reduce_rows(const Params& p, const Work& w, const float* tile_ws, int r0, int r1,
                                            int tid) {
    const int L = w.swap ? 128 : w.bn;
    const int L4 = L / 4;
    const long long part_floats = 128ll * w.bn;
    if (!p.vec_d) {
        // D rows not 16-byte aligned: one column per thread, consecutive
        // threads on consecutive columns (every store covers 128 contiguous
        // bytes); the same split order per output.
        const int tot = (r1 - r0) * L;
        const float alpha = p.alpha, beta = p.beta;
        for (int i = tid; i < tot; i += 128) {
            const int rr = r0 + i / L, l = i - (i / L) * L;
            const float* src = tile_ws + (long long)rr * L + l;
            float acc = 0.0f;
            int s = 0;
            for (; s + 8 <= w.splits; s += 8) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; e++) x[e] = __ldcg(src + (s + e) * part_floats);
#pragma unroll
                for (int e = 0; e < 8; e++) acc += x[e];
            }
            for (; s < w.splits; s++) acc += __ldcg(src + s * part_floats);
            const int m = w.m_t0 + rr, n = w.n_t0 + l;
            if (m < w.m_end && n < w.n_end) {
                float o = alpha * acc;
                if (beta != 0.0f) o = fmaf(beta, p.C[(long long)w.b * p.strideC + (long long)m * p.ldc + n], o);
                put_out<EPI>(p, d_ptr<EPI>(p, (long long)w.b * p.strideD + (long long)m * p.ldd + n),
                             act_fn<EPI>(o));
            }
        }
        return;
    }
    const int total = (r1 - r0) * L4;
    const long long step4 = part_floats / 4;
    // Each thread takes two outputs at a time and keeps 2 x 8 loads in
    // flight; every output still adds its partials in split order.
    for (int i0 = tid; i0 < total; i0 += 256) {
        const int i1 = i0 + 128;
        const bool two = i1 < total;
        const float4* src0 = reinterpret_cast<const float4*>(tile_ws + (long long)(r0 + i0 / L4) * L) + (i0 % L4);
        const float4* src1 =
            two ? reinterpret_cast<const float4*>(tile_ws + (long long)(r0 + i1 / L4) * L) + (i1 % L4) : src0;
        float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
        int s = 0;
        for (; s + 8 <= w.splits; s += 8) {
            float4 x0[8], x1[8];
#pragma unroll
            for (int e = 0; e < 8; e++) {
                x0[e] = __ldcg(src0 + (s + e) * step4);
                x1[e] = __ldcg(src1 + (s + e) * step4);
            }
#pragma unroll
            for (int e = 0; e < 8; e++) {
                a0.x += x0[e].x; a0.y += x0[e].y; a0.z += x0[e].z; a0.w += x0[e].w;
                a1.x += x1[e].x; a1.y += x1[e].y; a1.z += x1[e].z; a1.w += x1[e].w;
            }
        }
        for (; s < w.splits; s++) {
            const float4 x0 = __ldcg(src0 + s * step4);
            const float4 x1 = __ldcg(src1 + s * step4);
            a0.x += x0.x; a0.y += x0.y; a0.z += x0.z; a0.w += x0.w;
            a1.x += x1.x; a1.y += x1.y; a1.z += x1.z; a1.w += x1.w;
        }
        const int m0 = w.m_t0 + r0 + i0 / L4;
        if (m0 < w.m_end) store4<EPI>(p, w, m0, w.n_t0 + 4 * (i0 % L4), a0);
        if (two) {
            const int m1 = w.m_t0 + r0 + i1 / L4;
            if (m1 < w.m_end) store4<EPI>(p, w, m1, w.n_t0 + 4 * (i1 % L4), a1);
        }
    }
}

// o[0..3] = alpha * sum + beta * C at D[m][n..n+3] (columns past the region
// clipped): activation, then the store.
template <int EPI>
__device__ __forceinline__ void put4_clipped(const Params& p, const Work& w, int m, int n, const float* o) {
    if (n >= w.n_end) return;
    uint8_t* d = d_ptr<EPI>(p, (long long)w.b * p.strideD + (long long)m * p.ldd + n);
    if (p.vec_d && n + 3 < w.n_end) {
        put_out4<EPI>(p, d, act_fn<EPI>(o[0]), act_fn<EPI>(o[1]), act_fn<EPI>(o[2]), act_fn<EPI>(o[3]));
    } else {
#pragma unroll
        for (int e = 0; e < 4; e++)
            if (n + e < w.n_end) put_out<EPI>(p, d + e * d_esize<EPI>(p), act_fn<EPI>(o[e]));
    }
}

// Shared memory the ring reduction needs for rows [r0, r1) of a split tile:
// the S partial slices, and C's rows when they are copied too.
__device__ __forceinline__ bool ring_c_rows(const Params& p, const Work& w) {
    const int L = w.swap ? 128 : w.bn;
    return p.beta != 0.0f && p.vec_c && w.n_t0 + L <= w.n_end;
}
__device__ __forceinline__ uint32_t ring_reduce_bytes(const Params& p, const Work& w, int r0, int r1) {
    const uint32_t slice = (uint32_t)(r1 - r0) * (uint32_t)(w.swap ? 128 : w.bn) * 4u;
    return slice * (uint32_t)(w.splits + (ring_c_rows(p, w) ? 1 : 0));
}

// Rows [r0, r1) of a split tile, when the operand ring is idle (every MMA of
// this CTA has completed): one warp bulk-copies the S partial slices (each
// (r1 - r0) x L contiguous floats) and, where C's rows lie whole inside D
// and are 16-byte aligned, those rows of C into the ring under one mbarrier;
// then the 128 epilogue threads add the partials in split order from shared
// memory (the same order, hence the same bits, as reduce_rows) and write D.
// Only one memory round trip, instead of one per group of outputs.  Returns
// false when the wait for the copies gave up (the status word is set).
template <int EPI>
__device__ __forceinline__ bool reduce_rows_ring(const Params& p, const Work& w, const float* tile_ws, int r0,
                                                 int r1, int tid, uint32_t ring, const uint8_t* ring_g,
                                                 uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                 uint64_t limit) {
    const int L = w.swap ? 128 : w.bn;
    const int L4 = L / 4;
    const int S = w.splits;
    const long long part_floats = 128ll * w.bn;
    const int rows = r1 - r0;
    const uint32_t slice = (uint32_t)rows * (uint32_t)L * 4u;
    const bool c_ring = ring_c_rows(p, w);
    const int rows_c = c_ring ? max(0, min(r1, w.m_end - w.m_t0) - r0) : 0;
    const uint32_t c_off = (uint32_t)S * slice;
    if (tid < 32) {
        // (Test hook 2: expect 16 bytes more than are copied, so that the
        // bounded wait below runs out.)
        if (tid == 0)
            mbar_arrive_expect_tx(bar, (uint32_t)S * slice + (uint32_t)rows_c * (uint32_t)L * 4u +
                                           (p.inject_timeout == 2 ? 16u : 0u));
        __syncwarp();
        for (int s = tid; s < S; s += 32)
            bulk_load(ring + (uint32_t)s * slice, tile_ws + s * part_floats + (long long)r0 * L, slice, bar);
        const float* c0 = p.C + (long long)w.b * p.strideC + (long long)(w.m_t0 + r0) * p.ldc + w.n_t0;
        for (int r = tid; r < rows_c; r += 32)
            bulk_load(ring + c_off + (uint32_t)(r * L * 4), c0 + (long long)r * p.ldc, (uint32_t)L * 4u, bar);
    }
    int ok = 1;
    if ((tid & 31) == 0) ok = wait_bounded(bar, parity, abort_flag, p.err, kErrWaitSplits, limit, true) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) {
        // Let this CTA's copies land before it leaves.
        if (tid == 0) wait_bounded(bar, parity, abort_flag, p.err, kErrDrain, limit, false);
        __syncwarp();
        return false;
    }
    const float* sm = reinterpret_cast<const float*>(ring_g);
    const float alpha = p.alpha, beta = p.beta;
    const int total = rows * L4;
    for (int i = tid; i < total; i += 128) {
        const int rr = i / L4, g = i - rr * L4;
        const int m = w.m_t0 + r0 + rr;
        if (m >= w.m_end) continue;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < S; sp++) {
            const float4 x = *reinterpret_cast<const float4*>(sm + (size_t)sp * (slice / 4) + rr * L + 4 * g);
            a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
        }
        float o[4] = {alpha * a.x, alpha * a.y, alpha * a.z, alpha * a.w};
        const int n = w.n_t0 + 4 * g;
        if (beta != 0.0f) {
            if (c_ring) {
                const float4 cv = *reinterpret_cast<const float4*>(sm + c_off / 4 + rr * L + 4 * g);
                o[0] = fmaf(beta, cv.x, o[0]);
                o[1] = fmaf(beta, cv.y, o[1]);
                o[2] = fmaf(beta, cv.z, o[2]);
                o[3] = fmaf(beta, cv.w, o[3]);
            } else {
                const float* cp = p.C + (long long)w.b * p.strideC + (long long)m * p.ldc + n;
#pragma unroll
                for (int e = 0; e < 4; e++)
                    if (n + e < w.n_end) o[e] = fmaf(beta, cp[e], o[e]);
            }
        }
        put4_clipped<EPI>(p, w, m, n, o);
    }
    return true;
}

// Wait until the previous kernel on the stream (programmatic dependent
// launch) has completed and its memory operations are visible; returns at
// once when there is none.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Split-K on chip: every split of a tile runs on one CTA of a cluster of S
// and has left its fp32 partial in its own shared memory at `part_s`, as R
// rows x L columns of the tile in D-row-major order with a row pitch of L + 4
// floats.  After a cluster barrier, this CTA sums rows [R r / S, R (r+1) / S)
// over the S partials in split order (the same order, hence the same bits, as
// the global-memory reduction) and writes D.  All threads of the CTA take part.
template <int EPI>
__device__ __forceinline__ void csplit_reduce(const Params& p, const Work& w, uint32_t part_s) {
    const int S = w.splits, r = w.split;
    const int R = w.swap ? w.bn : 128, L = w.swap ? 128 : w.bn, P = L + 4;
    const int r0 = (int)((long long)R * r / S), r1 = (int)((long long)R * (r + 1) / S);
    const int L4 = L / 4;
    const int total = (r1 - r0) * L4;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int row = r0 + i / L4, g = i - (i / L4) * L4;
        const uint32_t off = part_s + (uint32_t)((row * P + 4 * g) * 4);
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        int sp = 0;
        for (; sp + 8 <= S; sp += 8) {
            float4 x[8];
#pragma unroll
            for (int e = 0; e < 8; e++) x[e] = ld_dsmem_v4(mapa_shared(off, (uint32_t)(sp + e)));
#pragma unroll
            for (int e = 0; e < 8; e++) {
                a.x += x[e].x; a.y += x[e].y; a.z += x[e].z; a.w += x[e].w;
            }
        }
        for (; sp < S; sp++) {
            const float4 x = ld_dsmem_v4(mapa_shared(off, (uint32_t)sp));
            a.x += x.x; a.y += x.y; a.z += x.z; a.w += x.w;
        }
        const int m = w.m_t0 + row;
        if (m < w.m_end) store4<EPI>(p, w, m, w.n_t0 + 4 * g, a);
    }
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const unsigned int* ptr) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

// ---------------------------------------------------------------------------
// The persistent kernel
// ---------------------------------------------------------------------------
// CG = 1: one CTA per tile.  CG = 2: clusters of two CTAs on 256-row tile
// pairs with the pair MMA (the even CTA issues for both; see umma_bf16).
template <int CG, int EPI>
__global__ void __launch_bounds__(kThreads, 1) k_poly_gemm(const __grid_constant__ Params p) {
    constexpr bool kPair = CG == 2;
    // Lean instantiations (the launch picks them; the paths they cannot
    // take are folded away).  EPI bit 4: plans with no split and no swapped
    // region.  Bit 3: the same with 16-byte aligned D and beta = 0 as well.
    constexpr bool kLean = (EPI & 8) != 0;
    constexpr bool kPlain = (EPI & 24) != 0;
    // EPI bit 5: plans whose regions are all split and none swapped.
    constexpr bool kSplitOnly = (EPI & 32) != 0;
    constexpr bool kNoSwap = kPlain || kSplitOnly;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t ring0 = base;
    const uint32_t epi0 = base + kRingBytes;
    const uint32_t bar0 = epi0 + kStageBytesEpi;
    uint64_t* bars = reinterpret_cast<uint64_t*>(gbase + (bar0 - base));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 6);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* s_last = reinterpret_cast<volatile int*>(tmem_slot + 2);
    volatile int* epi_abort = reinterpret_cast<volatile int*>(tmem_slot + 3);
    // Region table copy: 512 bytes into the 1 KB barrier area (barriers and
    // flags use the first ~250 bytes).
    static_assert(sizeof(Region) * MP_MAX_REGIONS <= kBarBytes - 512, "region table does not fit");
    static_assert((2 * kMaxStages + 6) * 8 + 16 <= 512, "barriers do not fit");
    Region* regs_s = reinterpret_cast<Region*>(gbase + (bar0 - base) + 512);

    const int nst = p.num_stages;
    const uint32_t stage_bytes = (uint32_t)p.stage_bytes;  // kg sub-stages of (X tile, then Y tile)
    const uint32_t sub_bytes = (uint32_t)p.sub_bytes;
    const int kg = p.kg;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
    auto accf = [&](int b) { return bar0 + 8u * (2 * kMaxStages + b); };
    auto acce = [&](int b) { return bar0 + 8u * (2 * kMaxStages + 2 + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * kMaxStages + 4);
    const uint32_t red_bar = bar0 + 8u * (2 * kMaxStages + 5);  // split-K sums staged in the idle ring
    const uint64_t limit = p.wait_limit_ns;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Pairs: a cluster of two CTAs works through tile pairs; rank 0 (the
    // leader) waits for both CTAs' operands and issues the MMAs; its commits
    // reach the barriers of both.
    const int rank = kPair ? (int)cluster_ctarank() : 0;
    const bool leader = rank == 0;
    const int u0 = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int ustep = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(accf(b), 1);
            // The leader's accumulator is free once the epilogues of both
            // CTAs have read their halves.
            mbar_init(acce(b), kPair ? 8 : 4);
        }
        mbar_init(done_bar, 1);
        mbar_init(red_bar, 1);
        *abort_flag = 0;
        *s_last = 0;
        *epi_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // Fetch every descriptor this launch uses while the previous kernel
        // on the stream may still be running.
        tma_prefetch_map(&p.tmA);
        tma_prefetch_map(&p.tmAs);
        tma_prefetch_map(&p.tmB);
        for (int j = 0; j < 4; j++)
            if (p.b4_mask & (1 << j)) tma_prefetch_map(&p.tmB4[j]);
        if (p.tma_d) tma_prefetch_map(&p.tmD);
        if (p.bs_ok) tma_prefetch_map(&p.tmBs);
        for (int i = 0; i < MP_MAX_REGIONS; i++)
            if (p.w_mask & (1 << i)) tma_prefetch_map(&p.tmW[i]);
    }
    // The region table goes to shared memory during set-up (ordinary member
    // reads of the parameter), so that work-unit decoding after the
    // dependency wait reads shared memory instead of cold parameter lines.
    if (threadIdx.x < MP_MAX_REGIONS) regs_s[threadIdx.x] = p.reg[threadIdx.x];
    if (warp == 1) {
        tmem_alloc<CG>(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish<CG>();
    }
    __syncthreads();
    // Pairs: each CTA's copies, commits and arrivals also target the other's
    // barriers, so both finish initialising them before either starts.
    if (kPair) cluster_sync();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Programmatic dependent launch: set-up, work decoding and the first slot
    // probes may overlap the previous kernel on this stream.  Each thread that
    // touches global memory (the producers before their first copy, the
    // epilogue before anything else) first waits until that kernel has
    // finished and its writes are visible; every thread waits once more
    // before exit, so this grid never completes ahead of its predecessor.
    // The next kernel may start its own set-up on SMs as they free up.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0 || warp == kProducer2Warp) {
        // ------------------------------ TMA producers (two warps) -------------
        // Issuing a stage (probe the slot, copies, expect-tx) costs several
        // hundred cycles of dependent latency, so two warps take alternate
        // stages of the CTA's global stage sequence g: a stage holds kg
        // consecutive 64-deep K steps of one unit (fewer at the unit's end);
        // stage g uses ring slot g % nst, phase (g / nst) & 1, and belongs to
        // warp 0 when g is even.  Within a warp, lane 0 probes the slot and
        // arms it; each K step's copies (one to five boxes) go out from
        // different lanes in one instruction, before the expect-tx for the
        // whole stage (the transaction count may run negative until then; the
        // phase cannot complete without the arrive).
        //   normal tile:  lane 0 -> A box (128 rows), lanes 1.. -> B
        //   swapped tile: lane 0.. -> B^T (128 columns), lanes 2.. -> A
        // B comes in one box of all the tile's 64-column blocks when they
        // are all full; a tile that reaches past the last full block loads
        // its blocks one by one (zero-filled beyond N).
        const uint32_t pid = warp == 0 ? 0u : 1u;
        uint32_t g = 0;
        uint32_t armed_mask = 0, armed_ph = 0;
        bool withhold = pid == 0 && p.inject_timeout == 1;
        bool dep_done = false;
        for (int u = u0; u < p.total_units; u += ustep) {
            const Work w = decode(p, regs_s, u, rank);
            const int ab = w.b * p.a_bstep, bb = w.b * p.b_bstep;
            const int blk0 = w.n_t0 >> 6;
            const int nblk = (!kNoSwap && w.swap) ? 2 : (w.bn >> 6);
            const bool whole_b = blk0 + nblk <= p.nb_full;
            for (int kb = w.kb0; kb < w.kb1; kb += kg, ++g) {
                if ((g & 1u) != pid) continue;
                const int stage = (int)(g % (uint32_t)nst);
                const uint32_t ph = (g / (uint32_t)nst) & 1u;
                int ok = 1;
                if (lane == 0) ok = wait_fast(empty(stage), ph ^ 1u, abort_flag, p.err, kErrWaitEmpty, limit) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, ok, 0)) goto producer_out;
                if (!dep_done) {
                    grid_dep_wait();
                    dep_done = true;
                }
                if (!withhold) {
                    // Pairs: the odd CTA's copies complete on the leader's barrier.
                    const uint32_t fb = (kPair && !leader) ? mapa_shared(full(stage), 0) : full(stage);
                    const int nsub = min(kg, w.kb1 - kb);
                    for (int j = 0; j < nsub; j++) {
                    const uint32_t xs = ring0 + stage * stage_bytes + j * sub_bytes, ys = xs + kXBytes;
                    const int kc = (kb + j) * 64;
                    if (kNoSwap || !w.swap) {
                        if constexpr (kPair) {
                            // This CTA's 128 rows of A and its half of B's
                            // 64-column blocks (rank r: blocks [r h, r h + h)).
                            const int h = nblk >> 1, first = rank * h;
                            if (w.bn == 192) {
                                // 96 columns per CTA: three 32-column boxes
                                // (64-byte swizzle) from lanes 1..3.
                                const int x = w.n_t0 + 96 * rank + 32 * (lane - 1);
                                if (leader) {
                                    if (lane == 0) tma_load_3d(xs, &p.tmA, fb, kc, w.m_t0, ab);
                                    else if (lane <= 3) tma_load_3d(ys + (lane - 1) * 4096, &p.tmBs, fb, x, kc, bb);
                                } else {
                                    if (lane == 0) tma_load_3d_pair(xs, &p.tmA, fb, kc, w.m_t0, ab);
                                    else if (lane <= 3) tma_load_3d_pair(ys + (lane - 1) * 4096, &p.tmBs, fb, x, kc, bb);
                                }
                            } else if (leader) {
                                if (lane == 0) tma_load_3d(xs, &p.tmA, fb, kc, w.m_t0, ab);
                                if (whole_b) {
                                    if (lane == 1) tma_load_4d(ys, &p.tmB4[h - 1], fb, 0, kc, blk0 + first, bb);
                                } else if (lane >= 1 && lane <= h) {
                                    const int c = first + lane - 1;
                                    tma_load_3d(ys + (lane - 1) * 8192, &p.tmB, fb, w.n_t0 + 64 * c, kc, bb);
                                }
                            } else {
                                if (lane == 0) tma_load_3d_pair(xs, &p.tmA, fb, kc, w.m_t0, ab);
                                if (whole_b) {
                                    if (lane == 1) tma_load_4d_pair(ys, &p.tmB4[h - 1], fb, 0, kc, blk0 + first, bb);
                                } else if (lane >= 1 && lane <= h) {
                                    const int c = first + lane - 1;
                                    tma_load_3d_pair(ys + (lane - 1) * 8192, &p.tmB, fb, w.n_t0 + 64 * c, kc, bb);
                                }
                            }
                        } else {
                        if (lane == 0) tma_load_3d(xs, &p.tmA, fb, kc, w.m_t0, ab);
                        if (whole_b) {
                            if (lane == 1) tma_load_4d(ys, &p.tmB4[nblk - 1], fb, 0, kc, blk0, bb);
                        } else if (lane >= 1 && lane <= nblk) {
                            const int c = lane - 1;
                            tma_load_3d(ys + c * 8192, &p.tmB, fb, w.n_t0 + 64 * c, kc, bb);
                        }
                        }
                    } else {
                        if (whole_b) {
                            if (lane == 0) tma_load_4d(xs, &p.tmB4[1], fb, 0, kc, blk0, bb);
                        } else if (lane < 2) {
                            tma_load_3d(xs + lane * 8192, &p.tmB, fb, w.n_t0 + 64 * lane, kc, bb);
                        }
                        const int na = w.bn / p.as_rows;
                        if (lane >= 2 && lane < 2 + na) {
                            const int c = lane - 2;
                            tma_load_3d(ys + c * p.as_rows * 128, &p.tmAs, fb, kc, w.m_t0 + c * p.as_rows, ab);
                        }
                    }
                    }
                    __syncwarp();
                    // The leader arms its barrier for both CTAs' bytes (A rows
                    // and B halves of each); the odd CTA arms nothing.
                    if (!kPair || leader) {
                        const uint32_t bytes = kPair ? 2u * (kXBytes + (w.bn >> 1) * 128) : kXBytes + w.bn * 128;
                        if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)nsub * bytes);
                        armed_mask |= 1u << stage;
                        armed_ph = (armed_ph & ~(1u << stage)) | (ph << stage);
                    }
                }
                withhold = false;
            }
        }
    producer_out:
        if (lane == 0 && *abort_flag) {
            // Let every copy this warp started land before the CTA exits.
            for (int s = 0; s < nst; s++)
                if (armed_mask & (1u << s))
                    wait_bounded(full(s), (armed_ph >> s) & 1u, abort_flag, p.err, kErrDrain, limit, false);
        } else if (kPair && pid == 0 && lane == 0) {
            // Pairs: the leader's MMA commits reach this CTA's empty barriers
            // too; wait until the last use of every slot has been released,
            // so that nothing arrives here after exit.
            for (uint32_t s = 0; s < (uint32_t)nst && s < g; s++) {
                const uint32_t k = (g - 1u - s) / (uint32_t)nst;
                wait_bounded(empty((int)s), k & 1u, abort_flag, p.err, kErrDrain, limit, true);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer (lane 0) --------------------
        // One thread waits, issues every MMA and every commit, so that each
        // commit tracks exactly this thread's MMAs.  Pairs: the leader's
        // thread issues for both CTAs; the odd CTA's MMA warp only holds TMEM.
        if (lane == 0 && (!kPair || leader)) {
        int stage = 0;
        uint32_t ph = 0;
        int acc = 0;
        uint32_t aph = 0;
        for (int u = u0; u < p.total_units; u += ustep) {
            const Work w = decode(p, regs_s, u, rank);
            bool ok = wait_fast(acce(acc), aph ^ 1u, abort_flag, p.err, kErrWaitAccEmpty, limit);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * kAccStride);
            const uint32_t idesc =
                (!kNoSwap && w.swap) ? idesc_bf16(w.bn, true, false) : idesc_bf16(w.bn, false, true, kPair ? 256 : 128);
            // Descriptors of stage 0, K step 0.  Every later stage and K step
            // only moves the start address (bits 0..13, in 16-byte units;
            // shared addresses stay below 2^18, so the sums never carry out of
            // the field): one 64-bit add per operand.
            const bool swp = !kNoSwap && w.swap;
            const uint64_t dx0 = swp ? desc_mnmajor(ring0, 0) : desc_kmajor(ring0, 0);
            // Pairs of 192-wide tiles hold B with the 64-byte swizzle.
            const bool b64 = kPair && w.bn == 192;
            const uint64_t dy0 = swp ? desc_kmajor(ring0 + kXBytes, 0)
                                 : b64  ? desc_mnmajor64(ring0 + kXBytes, 0)
                                        : desc_mnmajor(ring0 + kXBytes, 0);
            const uint32_t kx = swp ? (2048u >> 4) : (32u >> 4);
            const uint32_t ky = swp ? (32u >> 4) : b64 ? (1024u >> 4) : (2048u >> 4);
            const uint32_t sstep = stage_bytes >> 4, jstep = sub_bytes >> 4;
            // One wait and one commit per stage of kg (1 or 2) K steps.
            for (int kb = w.kb0; kb < w.kb1; kb += kg) {
                ok = wait_fast(full(stage), ph, abort_flag, p.err, kErrWaitFull, limit);
                if (!ok) break;
                tc_fence_after();
                uint64_t ax = dx0 + (uint64_t)(stage * sstep);
                uint64_t by = dy0 + (uint64_t)(stage * sstep);
                umma_bf16<CG>(d, ax, by, idesc, kb > w.kb0 ? 1u : 0u);
                umma_bf16<CG>(d, ax + kx, by + ky, idesc, 1u);
                umma_bf16<CG>(d, ax + 2 * kx, by + 2 * ky, idesc, 1u);
                umma_bf16<CG>(d, ax + 3 * kx, by + 3 * ky, idesc, 1u);
                if (kg > 1 && kb + 1 < w.kb1) {
                    ax += jstep;
                    by += jstep;
                    umma_bf16<CG>(d, ax, by, idesc, 1u);
                    umma_bf16<CG>(d, ax + kx, by + ky, idesc, 1u);
                    umma_bf16<CG>(d, ax + 2 * kx, by + 2 * ky, idesc, 1u);
                    umma_bf16<CG>(d, ax + 3 * kx, by + 3 * ky, idesc, 1u);
                }
                if constexpr (kPair)
                    umma_commit_pair(empty(stage), (uint16_t)3);  // the slot of both CTAs
                else
                    umma_commit(empty(stage));
                if (++stage == nst) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            if constexpr (kPair)
                umma_commit_pair(accf(acc), (uint16_t)3);  // both CTAs' epilogues
            else
                umma_commit(accf(acc));
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
        // Every MMA this thread issued has completed once `done_bar` flips.
        if constexpr (kPair)
            umma_commit_pair(done_bar, (uint16_t)1);
        else
            umma_commit(done_bar);
        wait_bounded(done_bar, 0, abort_flag, p.err, kErrDrain, limit, false);
        }
    } else {
        // ------------------------------ epilogue (128 threads) ----------------
        // While the previous kernel may still run, warm L2 with the leading K
        // steps of this CTA's first unit (one K step per lane, the boxes the
        // producers will load).  A prefetch hands no data to the SM, so it
        // may precede the dependency wait; the producers' own copies follow it.
        if constexpr (!kPair) {
            if (warp == 2 && p.l2_pf > 0 && u0 < p.total_units) {
                const Work w = decode(p, regs_s, u0, 0);
                if (kNoSwap || !w.swap) {
                    const int nk = min(p.l2_pf, w.kb1 - w.kb0);
                    const int ab = w.b * p.a_bstep, bb = w.b * p.b_bstep;
                    const int blk0 = w.n_t0 >> 6, nblk = w.bn >> 6;
                    const bool whole_b = blk0 + nblk <= p.nb_full;
                    for (int j = lane; j < nk; j += 32) {
                        const int kc = (w.kb0 + j) * 64;
                        tma_prefetch_l2_3d(&p.tmA, kc, w.m_t0, ab);
                        if (whole_b)
                            tma_prefetch_l2_4d(&p.tmB4[nblk - 1], 0, kc, blk0, bb);
                        else  // the blocks that start inside N
                            for (int c = 0; c < nblk && w.n_t0 + 64 * c < w.n_end; c++)
                                tma_prefetch_l2_3d(&p.tmB, w.n_t0 + 64 * c, kc, bb);
                    }
                }
            }
        }
        // The same for the C block of that unit's epilogue, when beta*C is
        // read (one-CTA plans; later units ask for theirs after the wait).
        bool c_early = false;
        if constexpr (!kLean && !kSplitOnly && !kPair) {
            if (p.beta != 0.0f && u0 < p.total_units) {
                const Work w = decode(p, regs_s, u0, 0);
                if (kPlain || w.splits == 1) {
                    const int q = warp & 3;
                    if (!kPlain && w.swap)
                        prefetch_c_swapped(p, w, q, lane);
                    else if (p.tma_d)
                        prefetch_c_row(p, w, w.m_t0 + q * 32 + lane);
                    else
                        prefetch_c_tile_row(p, w, w.m_t0 + q * 32 + lane);
                    c_early = true;
                }
            }
        }
        grid_dep_wait();
        // The accumulator buffer goes back to the MMA issuer: the leader's
        // barrier, from both CTAs of a pair.
        auto release_acc = [&](int b) {
            if (kPair && !leader)
                mbar_arrive_remote(mapa_shared(acce(b), 0));
            else
                mbar_arrive(acce(b));
        };
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        uint8_t* epi_g = gbase + (epi0 - base) + (warp - 2) * kEpiWarpBytes;
        const uint32_t epi_s = epi0 + (uint32_t)((warp - 2) * kEpiWarpBytes);
        float4* stage = reinterpret_cast<float4*>(epi_g);
        uint32_t slab = 0;  // running slab index of this warp's bulk stores
        int acc = 0;
        uint32_t aph = 0;
        uint32_t red_ph = 0;  // phase of red_bar
        for (int u = u0; u < p.total_units; u += ustep) {
            const Work w = decode(p, regs_s, u, rank);
            if (!kLean && !kSplitOnly && p.beta != 0.0f && (kPlain || w.splits == 1) && !(c_early && u == u0)) {
                if (!kPlain && w.swap)
                    prefetch_c_swapped(p, w, q, lane);
                else if (p.tma_d)
                    prefetch_c_row(p, w, w.m_t0 + q * 32 + lane);
                else
                    prefetch_c_tile_row(p, w, w.m_t0 + q * 32 + lane);
            }
            int ok = 1;
            if (lane == 0)
                ok = wait_bounded(accf(acc), aph, abort_flag, p.err, kErrWaitAccFull, limit, true) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            // The four epilogue warps decide together whether to stop, so that
            // none of them is left alone at a later named barrier.  The flag
            // is written only before the first barrier and read between the
            // two, so no warp can see another iteration's value.
            if (!ok && lane == 0) *epi_abort = 1;
            named_bar_sync(1, 128);
            const int stop = *epi_abort;
            named_bar_sync(1, 128);
            if (stop) break;
            tc_fence_after();
            const uint32_t t = tmem + (uint32_t)(acc * kAccStride) + ((uint32_t)(q * 32) << 16);
            const bool has_k = w.kb1 > w.kb0;
            if (!kSplitOnly && epi_bf16<EPI>() && (kLean || (w.splits == 1 && p.tma_d && !w.swap))) {
                // bf16 D: 64-column chunks, so that a lane's row of the slab is
                // 128 bytes (the 128-byte swizzle); two TMEM loads per chunk.
                const bool with_c = !kLean && p.beta != 0.0f;
                const float a = p.alpha, bt = p.beta;
                for (int c = 0; c < w.bn; c += 64) {
                    const int m0 = w.m_t0 + q * 32, n0 = w.n_t0 + c;
                    const bool do_store = m0 < w.m_end && n0 < w.n_end;  // the same for the whole warp
                    const uint32_t off = (slab & 1u) * 4096u;
                    if (do_store) {
                        if (lane == 0) bulk_wait_read_1();
                        __syncwarp();
                    }
                    uint8_t* row = epi_g + off + lane * 128;
#pragma unroll 1
                    for (int qq = 0; qq < 4; qq++) {  // 16 columns = 32 bytes of bf16 at a time
                        float cv[16];
                        if (with_c) load_c<16>(p, w, lane, m0, n0 + 16 * qq, cv);
                        float v[16];
                        if (has_k) {
                            tmem_ld16(t + c + 16 * qq, v);
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; j++) v[j] = 0.0f;
                        }
                        uint32_t pk[8];
#pragma unroll
                        for (int j = 0; j < 8; j++) {
                            float x0 = a * v[2 * j], x1 = a * v[2 * j + 1];
                            if (with_c) {
                                x0 = fmaf(bt, cv[2 * j], x0);
                                x1 = fmaf(bt, cv[2 * j + 1], x1);
                            }
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(act_fn<EPI>(x0), act_fn<EPI>(x1));
                            pk[j] = *reinterpret_cast<const uint32_t*>(&b2);
                        }
                        if (do_store) {
#pragma unroll
                            for (int j = 0; j < 2; j++)
                                *reinterpret_cast<uint4*>(row + (((2 * qq + j) ^ (lane & 7)) << 4)) =
                                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                        }
                    }
                    if (do_store) {
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_3d(&p.tmD, epi_s + off, n0, m0, w.b);
                            bulk_commit_group();
                        }
                        ++slab;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_acc(acc);
            } else if ((kLean && !epi_bf16<EPI>()) ||
                       (!kSplitOnly && !epi_bf16<EPI>() && (kPlain || (w.splits == 1 && !w.swap)) && p.tma_d)) {
                const bool with_c = !kLean && p.beta != 0.0f;
                for (int c = 0; c < w.bn; c += 32) {
                    const int m0 = w.m_t0 + q * 32, n0 = w.n_t0 + c;
                    float cv[32];
                    if (with_c) load_c32(p, w, lane, m0, n0, cv);
                    float v[32];
                    if (has_k) {
                        tmem_ld32(t + c, v);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j++) v[j] = 0.0f;
                    }
                    // A slab wholly past the region's last row or column has
                    // nothing to store (and no store group, so the slab
                    // alternation is kept by counting only real stores).
                    if (m0 < w.m_end && n0 < w.n_end) {
                        const uint32_t off = (slab & 1u) * 4096u;
                        emit32_tma<EPI>(p, w, lane, m0, n0, v, cv, epi_g + off, epi_s + off);
                        ++slab;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_acc(acc);
            } else if (!kSplitOnly && (kPlain || (w.splits == 1 && !w.swap)) && p.beta != 0.0f) {
                // Unaligned D with beta * C (measured: faster than the
                // transposed stores below once C has to be read).
                // The slab area may still be read by an earlier tile's bulk stores.
                if (lane == 0) bulk_wait_read_all();
                for (int c = 0; c < w.bn; c += 32) {
                    float cv[32];
                    load_c_cols(p, w, q, lane, c, cv);
                    float v[32];
                    if (has_k) {
                        tmem_ld32(t + c, v);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; j++) v[j] = 0.0f;
                    }
                    emit32_rows<EPI>(p, w, q, lane, c, v, cv, epi_g);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_acc(acc);
            } else if (!kSplitOnly && (kPlain || w.splits == 1)) {
                for (int c = 0; c < w.bn; c += 16) {
                    float v[16];
                    if (has_k) {
                        tmem_ld16(t + c, v);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; j++) v[j] = 0.0f;
                    }
                    emit16<EPI>(p, w, q, lane, c, v, stage);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release_acc(acc);
            } else {
                // Split-K: park this split's partial (D-row-major per tile),
                // free the TMEM buffer, wait until every split of the tile
                // has parked, then sum this split's 1/S slice of the tile's
                // rows over all partials, in split order, and write D.
                float* part = p.ws + w.ws_tile + (long long)w.split * (128ll * w.bn);
                if (p.csplit) {
                    // On chip: the partial goes to this CTA's shared memory
                    // (the ring is idle: one task per CTA, all MMAs done); the
                    // cluster sums it at the end of the kernel.
                    float* ps = reinterpret_cast<float*>(gbase);
                    const int P = ((!kNoSwap && w.swap) ? 128 : w.bn) + 4;
                    if (kNoSwap || !w.swap) {
                        float* prow = ps + (q * 32 + lane) * P;
                        for (int c = 0; c < w.bn; c += 32) {
                            float v[32];
                            if (has_k) {
                                tmem_ld32(t + c, v);
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; j++) v[j] = 0.0f;
                            }
#pragma unroll
                            for (int j = 0; j < 8; j++)
                                *reinterpret_cast<float4*>(prow + c + 4 * j) =
                                    make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        }
                    } else {
                        float* pcol = ps + q * 32 + lane;
                        for (int c = 0; c < w.bn; c += 16) {
                            float v[16];
                            if (has_k) {
                                tmem_ld16(t + c, v);
                            } else {
#pragma unroll
                                for (int j = 0; j < 16; j++) v[j] = 0.0f;
                            }
#pragma unroll
                            for (int j = 0; j < 16; j++) pcol[(c + j) * P] = v[j];
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) release_acc(acc);
                } else if (!kNoSwap && w.swap) {
                    // lane = buffer column: every store covers 128 contiguous bytes.
                    for (int c = 0; c < w.bn; c += 16) {
                        float v[16];
                        tmem_ld16(t + c, v);
                        park16(w, q, lane, c, v, stage, part);
                    }
                } else if (p.w_mask & (1 << w.r)) {
                    // Bulk tensor stores of 32 x 32 slabs into the region's
                    // row-major partial view; the stores must have landed
                    // (not just left shared memory) before the tile counter
                    // announces this split.
                    for (int c = 0; c < w.bn; c += 32) {
                        float v[32];
                        tmem_ld32(t + c, v);
                        const uint32_t off = (slab & 1u) * 4096u;
                        if (lane == 0) bulk_wait_read_1();
                        __syncwarp();
                        uint8_t* row = epi_g + off + lane * 128;
#pragma unroll
                        for (int j = 0; j < 8; j++)
                            *reinterpret_cast<float4*>(row + ((j ^ (lane & 7)) << 4)) =
                                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        fence_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_3d(&p.tmW[w.r], epi_s + off, c, w.ws_row + q * 32, 0);
                            bulk_commit_group();
                        }
                        ++slab;
                    }
                    if (lane == 0) {
                        bulk_wait_all();
                        asm volatile("fence.proxy.async.global;" ::: "memory");
                    }
                    __syncwarp();
                } else {
                    // lane = buffer row: 32 columns are 128 contiguous bytes of it.
                    float* prow = part + (long long)(q * 32 + lane) * w.bn;
                    for (int c = 0; c < w.bn; c += 32) {
                        float v[32];
                        tmem_ld32(t + c, v);
#pragma unroll
                        for (int j = 0; j < 8; j++)
                            __stcg(reinterpret_cast<float4*>(prow + c) + j,
                                   make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
                    }
                }
                if (!p.csplit) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) release_acc(acc);  // TMEM buffer free for the next unit
                    __threadfence();
                    named_bar_sync(1, 128);
                    if (threadIdx.x == 64) {
                        unsigned int* cnt = p.cnt + w.cnt;
                        atomicAdd(cnt, 1u);
                        // Bounded wait for the other splits.  They are consecutive
                        // work units on distinct CTAs, so none of them waits on
                        // this CTA's later work.
                        int arrived = ld_acquire_u32(cnt) >= (unsigned)w.splits;
                        if (!arrived) {
                            const uint64_t t0 = globaltimer();
                            while (!(arrived = ld_acquire_u32(cnt) >= (unsigned)w.splits)) {
                                if (*abort_flag) break;
                                if (globaltimer() - t0 > limit) {
                                    *abort_flag = 1;
                                    atomicCAS(p.err, 0, kErrWaitSplits);
                                    break;
                                }
                                __nanosleep(64);
                            }
                        }
                        *s_last = arrived;
                    }
                    named_bar_sync(1, 128);
                    const int arrived = *s_last;
                    named_bar_sync(1, 128);
                    bool reduced = true;
                    if (arrived) {
                        __threadfence();
                        const int R = w.swap ? w.bn : 128;
                        const int r0 = (int)((long long)R * w.split / w.splits);
                        const int r1 = (int)((long long)R * (w.split + 1) / w.splits);
                        // The ring is idle once this is the CTA's last unit:
                        // every copy it loaded has been consumed by MMAs that
                        // have completed.
                        if (r1 > r0 && u + ustep >= p.total_units &&
                            ring_reduce_bytes(p, w, r0, r1) <= (uint32_t)kRingBytes) {
                            // The partials were written by other CTAs' generic or
                            // bulk stores; the copies read them through the async proxy.
                            asm volatile("fence.proxy.async.global;" ::: "memory");
                            reduced = reduce_rows_ring<EPI>(p, w, p.ws + w.ws_tile, r0, r1, threadIdx.x - 64,
                                                            ring0, gbase, red_bar, red_ph, abort_flag, limit);
                            red_ph ^= 1u;
                        } else {
                            reduce_rows<EPI>(p, w, p.ws + w.ws_tile, r0, r1, threadIdx.x - 64);
                        }
                        named_bar_sync(1, 128);
                    }
                    if (arrived && reduced) {
                        if (threadIdx.x == 64) {
                            // The last split to leave resets the counter for the next launch.
                            const unsigned old = atomicAdd(p.cnt + w.cnt, 1u);
                            if (old == 2u * (unsigned)w.splits - 1u) p.cnt[w.cnt] = 0u;
                        }
                    } else if (lane == 0) {
                        *epi_abort = 1;  // stop at the next unit (the flag is read between its barriers)
                    }
                }
            }
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
        // Bulk stores still in flight must finish before the CTA exits.
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    grid_dep_wait();
    __syncthreads();
    if constexpr (!kPair && !kPlain) {
        if (p.csplit) {
            // Every partial of this CTA's tile is now in its cluster's shared
            // memory; sum this CTA's slice; leave only when no CTA of the
            // cluster still reads this one's partial.
            cluster_sync();
            if ((int)blockIdx.x < p.total_units) csplit_reduce<EPI>(p, decode(p, regs_s, (int)blockIdx.x, 0), ring0);
            cluster_sync();
        }
    }
    if constexpr (kPair) {
        // After an abort, copies or commits of the peer may still be in
        // flight towards this CTA: give them time to land (they need
        // microseconds) before the pair leaves together.
        if (threadIdx.x == 0 && *abort_flag) {
            const uint64_t t0 = globaltimer();
            while (globaltimer() - t0 < 100000ull) __nanosleep(1000);
        }
        __syncthreads();
        cluster_sync();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<CG>(tmem, kTmemCols);
    }
}

}  // namespace dev

// Launch and attribute helpers for one epilogue instantiation (EPI: bits 0-1
// the activation, bit 2 a bf16 D; 0 is the plain alpha/beta epilogue).
template <int EPI>
inline cudaError_t launch_poly_gemm(const cudaLaunchConfig_t& cfg, bool pair, const dev::Params& p) {
    return pair ? cudaLaunchKernelEx(&cfg, dev::k_poly_gemm<2, EPI>, p)
                : cudaLaunchKernelEx(&cfg, dev::k_poly_gemm<1, EPI>, p);
}
template <int EPI>
inline bool set_poly_gemm_smem() {
    const auto a = cudaFuncAttributeMaxDynamicSharedMemorySize;
    return cudaFuncSetAttribute(dev::k_poly_gemm<1, EPI>, a, dev::kSmemBytes) == cudaSuccess &&
           cudaFuncSetAttribute(dev::k_poly_gemm<2, EPI>, a, dev::kSmemBytes) == cudaSuccess;
}

// The epilogue-variant instantiations live in their own translation units
// (compiled in parallel): fp32 D with an activation, and bf16 D.
cudaError_t launch_poly_gemm_act_f32(const cudaLaunchConfig_t& cfg, bool pair, int epi, const dev::Params& p);
bool set_poly_gemm_smem_act_f32();
cudaError_t launch_poly_gemm_bf16(const cudaLaunchConfig_t& cfg, bool pair, int epi, const dev::Params& p);
bool set_poly_gemm_smem_bf16();

}  // namespace mp
