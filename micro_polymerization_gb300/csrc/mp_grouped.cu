// The grouped GEMM kernel (see mp_grouped.cuh for the operation).
//
// Roles (224 threads), as in the GEMM kernel: warps 0 and 6 issue the TMA
// copies of alternate stages, lane 0 of warp 1 every tcgen05.mma and commit,
// warps 2..5 the epilogue (warp w reads TMEM lanes 32*(w%4)..+31: those 32
// rows of the tile).  A unit is one 128 x bn tile of one problem; its K loop
// runs in 64-deep steps, one ring stage each (A box 128 x 64, then bn/64 B
// boxes 64 x 64 of that problem).  Two 256-column TMEM accumulators alternate
// over the CTA's units.  Every wait is bounded (1 s by default), with the
// abort protocol of the other kernels.

#include "mp_kernel.cuh"
#include "mp_grouped.cuh"

namespace mp {
namespace grp {

using namespace mp::dev;

struct Tile {
    int i;       // problem
    int m0, n0;  // tile origin in the problem's D
    int nk;      // K steps
};

// Unit u -> (problem, tile): the last problem whose first unit is <= u (at
// most kMaxGroup problems, a short scan of the table in parameter space).
__device__ __forceinline__ Tile decode(const Params& p, int u) {
    int i = 0;
    while (i + 1 < p.count && p.prob[i + 1].tile0 <= u) ++i;
    const Problem& q = p.prob[i];
    const int t = u - q.tile0;
    return Tile{i, (t / q.tiles_n) * 128, (t % q.tiles_n) * p.bn, (q.K + 63) >> 6};
}

// The tile's epilogue for this warp's 32 rows: alpha*acc + beta*C, 32
// columns at a time, through the warp's two slabs and bulk tensor stores
// (clipped at the problem's edges), or plain stores when D's rows are not
// 16-byte aligned.
__device__ __forceinline__ void epilogue(const Problem& q, const Tile& t, int bn, uint32_t tacc, int wq, int lane,
                                         uint8_t* slab, uint32_t slab_s, uint32_t& slab_seq) {
    const int m_w = t.m0 + 32 * wq;
    if (m_w >= q.M) return;
    const int row = m_w + lane;
    const bool row_ok = row < q.M;
    const bool has_k = t.nk > 0;
    for (int c = 0; c < bn; c += 32) {
        const int n0 = t.n0 + c;
        if (n0 >= q.N) break;
        float v[32];
        if (has_k) {
            tmem_ld32(tacc + (uint32_t)c, v);
        } else {  // K == 0: no MMA wrote the accumulator
#pragma unroll
            for (int j = 0; j < 32; j++) v[j] = 0.0f;
        }
        float o[32];
#pragma unroll
        for (int j = 0; j < 32; j++) o[j] = q.alpha * v[j];
        if (q.beta != 0.0f && row_ok) {
            const float* cr = q.C + (long long)row * q.ldc + n0;
            if (q.vec_c && n0 + 32 <= q.N) {
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const float4 x = __ldg(reinterpret_cast<const float4*>(cr) + j);
                    o[4 * j] = fmaf(q.beta, x.x, o[4 * j]);
                    o[4 * j + 1] = fmaf(q.beta, x.y, o[4 * j + 1]);
                    o[4 * j + 2] = fmaf(q.beta, x.z, o[4 * j + 2]);
                    o[4 * j + 3] = fmaf(q.beta, x.w, o[4 * j + 3]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; j++)
                    if (n0 + j < q.N) o[j] = fmaf(q.beta, __ldg(cr + j), o[j]);
            }
        }
        if (q.tma_d) {
            const uint32_t buf = (slab_seq & 1u) * 4096u;
            if (lane == 0) bulk_wait_read_1();  // this slab's previous store has read it
            __syncwarp();
            uint8_t* line = slab + buf + lane * 128;
#pragma unroll
            for (int j = 0; j < 8; j++)
                *reinterpret_cast<float4*>(line + ((j ^ (lane & 7)) << 4)) =
                    make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_3d(&q.tmD, slab_s + buf, n0, m_w, 0);
                bulk_commit_group();
            }
            ++slab_seq;
        } else if (row_ok) {
            float* dr = q.D + (long long)row * q.ldd + n0;
#pragma unroll
            for (int j = 0; j < 32; j++)
                if (n0 + j < q.N) dr[j] = o[j];
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) k_gemm_grouped(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const int nst = p.num_stages;
    const uint32_t sb = (uint32_t)p.stage_bytes;  // 16 KB of A + bn x 128 B of B: a multiple of 8 KB
    const uint32_t ring0 = base;
    const uint32_t epi0 = ring0 + (uint32_t)nst * sb;
    const uint32_t bar0 = epi0 + 4u * kEpiSlabBytes;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
    auto accf = [&](int b) { return bar0 + 8u * (2 * kMaxStages + b); };
    auto acce = [&](int b) { return bar0 + 8u * (2 * kMaxStages + 2 + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * kMaxStages + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar0 - base) + 8 * (2 * kMaxStages + 5));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint64_t limit = p.wait_limit_ns;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nbox = p.bn >> 6;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(accf(b), 1);
            mbar_init(acce(b), 4);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_slot), 512);
        tmem_relinquish<1>();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Programmatic dependent launch, as in the GEMM kernel: the set-up above
    // may overlap the previous kernel on the stream; every role that touches
    // global memory first waits until that kernel has finished (its writes
    // visible), and every thread waits once more before exit.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0 || warp == 6) {
        grid_dep_wait();
        // ------------------------------ TMA producers (two warps) -------------
        // Stage g of the CTA's sequence belongs to warp 0 when g is even, to
        // warp 6 when it is odd.
        const uint32_t pid = warp == 0 ? 0u : 1u;
        uint32_t g = 0, armed_mask = 0, armed_ph = 0;
        // Test hook (failure detection): warp 0 leaves its first stage empty,
        // so the MMA issuer's bounded wait on it runs out.
        bool withhold = pid == 0 && p.inject_timeout != 0;
        for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
            const Tile t = decode(p, u);
            const Problem& q = p.prob[t.i];
            for (int kb = 0; kb < t.nk; kb++, g++) {
                if ((g & 1u) != pid) continue;
                const int stage = (int)(g % (uint32_t)nst);
                const uint32_t ph = (g / (uint32_t)nst) & 1u;
                int ok = 1;
                if (lane == 0) ok = wait_fast(empty(stage), ph ^ 1u, abort_flag, p.err, kErrWaitEmpty, limit) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, ok, 0)) goto producer_out;
                if (withhold) {  // neither copies nor an arrive: the stage never completes
                    withhold = false;
                    continue;
                }
                const uint32_t st = ring0 + (uint32_t)stage * sb;
                if (lane == 0)
                    tma_load_3d(st, &q.tmA, full(stage), kb * 64, t.m0, 0);
                else if (lane <= nbox)
                    tma_load_3d(st + 16384u + (uint32_t)(lane - 1) * 8192u, &q.tmB, full(stage), t.n0 + 64 * (lane - 1),
                                kb * 64, 0);
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(full(stage), 16384u + (uint32_t)p.bn * 128u);
                armed_mask |= 1u << stage;
                armed_ph = (armed_ph & ~(1u << stage)) | (ph << stage);
            }
        }
    producer_out:
        if (lane == 0 && *abort_flag) {
            for (int s = 0; s < nst; s++)
                if (armed_mask & (1u << s))
                    wait_bounded(full(s), (armed_ph >> s) & 1u, abort_flag, p.err, kErrDrain, limit, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer (lane 0) --------------------
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            const uint32_t idesc = idesc_bf16(p.bn, false, true);
            bool ok = true;
            for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
                const int nk = decode(p, u).nk;
                ok = wait_fast(acce(acc), aph ^ 1u, abort_flag, p.err, kErrWaitAccEmpty, limit);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * 256);
                for (int kb = 0; kb < nk; kb++) {
                    ok = wait_fast(full(stage), ph, abort_flag, p.err, kErrWaitFull, limit);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t st = ring0 + (uint32_t)stage * sb;
                    const uint64_t da = desc_kmajor(st, 0), db = desc_mnmajor(st + 16384u, 0);
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        umma_bf16<1>(d, da + 2u * j, db + 128u * j, idesc, (kb | j) ? 1u : 0u);
                    umma_commit(empty(stage));
                    if (++stage == nst) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(accf(acc));
                acc ^= 1;
                if (acc == 0) aph ^= 1u;
            }
            umma_commit(done_bar);
            wait_bounded(done_bar, 0, abort_flag, p.err, kErrDrain, limit, false);
        }
        __syncwarp();
    } else {
        // ------------------------------ epilogue (128 threads) ----------------
        // While the previous kernel may still run, warm L2 with the leading K
        // steps of this CTA's first tile (one K step per lane: the A box and
        // the B boxes that start inside N), unless that problem reads C.  A
        // prefetch hands no data to the SM, so it may precede the wait.
        if (warp == 2 && p.l2_pf > 0 && (int)blockIdx.x < p.units) {
            const Tile t = decode(p, (int)blockIdx.x);
            const Problem& q = p.prob[t.i];
            if (q.beta == 0.0f) {
                const int nk = min(p.l2_pf, t.nk);
                for (int j = lane; j < nk; j += 32) {
                    tma_prefetch_l2_3d(&q.tmA, j * 64, t.m0, 0);
                    for (int b = 0; b < nbox && t.n0 + 64 * b < q.N; b++)
                        tma_prefetch_l2_3d(&q.tmB, t.n0 + 64 * b, j * 64, 0);
                }
            }
        }
        grid_dep_wait();
        const int wq = warp & 3;
        uint8_t* slab = gbase + (epi0 - base) + wq * kEpiSlabBytes;
        const uint32_t slab_s = epi0 + (uint32_t)(wq * kEpiSlabBytes);
        const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
        int acc = 0;
        uint32_t aph = 0, slab_seq = 0;
        for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
            const Tile t = decode(p, u);
            int w = 1;
            if (lane == 0) w = wait_fast(accf(acc), aph, abort_flag, p.err, kErrWaitAccFull, limit) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, w, 0)) break;
            tc_fence_after();
            epilogue(p.prob[t.i], t, p.bn, tmem + (uint32_t)(acc * 256) + lane_off, wq, lane, slab, slab_s, slab_seq);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce(acc));
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }
    grid_dep_wait();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<1>(tmem, 512);
    }
}

cudaError_t launch(const cudaLaunchConfig_t& cfg, const Params& p) {
    return cudaLaunchKernelEx(&cfg, k_gemm_grouped, p);
}

bool set_smem() {
    return cudaFuncSetAttribute(k_gemm_grouped, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) ==
           cudaSuccess;
}

}  // namespace grp
}  // namespace mp
