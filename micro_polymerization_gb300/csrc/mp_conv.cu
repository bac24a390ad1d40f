// The implicit-GEMM convolution kernel (see mp_conv.cuh for the operation
// and the tiling).
//
// Roles (224 threads), as in the GEMM kernel: warps 0 and 6 issue the TMA
// copies of alternate stages (issuing a stage -- probe the slot, the copies,
// the expect-tx -- is several hundred cycles of dependent latency, longer
// than the MMAs of a narrow stage), lane 0 of warp 1 every tcgen05.mma and
// commit, warps 2..5 the epilogue (warp w reads TMEM lanes 32*(w%4)..+31:
// those 32 pixels of the tile).  A
// work unit is one output tile; its K loop runs over filter taps and blocks
// of 64 input channels, one ring stage per step (the A box from X, the
// tile's 64-column boxes of the filter).  Two 256-column TMEM accumulators
// alternate over the CTA's units, so a unit's epilogue overlaps the next
// unit's K loop.  Every wait is bounded (1 s by default), with the same
// abort protocol as the other kernels.

#include "mp_kernel.cuh"
#include "mp_conv.cuh"

namespace mp {
namespace conv {

using namespace mp::dev;

// Bulk tensor store of a shared-memory box to a 4-D view of global memory
// (bulk-group completion); elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

struct Tile {
    int n0, p0, q0, k0;
};

__device__ __forceinline__ Tile decode_tile(const Params& p, int t) {
    // Units run channel tile fastest, so the units that read one box of X
    // (and its halo) run side by side.
    const int kt = t % p.tiles_k;
    int m = t / p.tiles_k;
    const int tq = m % p.tiles_q;
    m /= p.tiles_q;
    const int tp = m % p.tiles_p;
    const int tn = m / p.tiles_p;
    return Tile{tn * p.nb, tp * p.hb, tq * p.wb, kt * p.bn};
}

// K steps [kb0, kb1) of split `sp`: the tile's ksteps cut into equal slices.
__device__ __forceinline__ void split_range(const Params& p, int sp, int& kb0, int& kb1) {
    kb0 = (int)((long long)p.ksteps * sp / p.splits);
    kb1 = (int)((long long)p.ksteps * (sp + 1) / p.splits);
}

// Pixel of tile row `row` (w fastest, then h, then image).
__device__ __forceinline__ void tile_pixel(const Params& p, const Tile& t, int row, int& n, int& ph, int& qw) {
    qw = t.q0 + row % p.wb;
    ph = t.p0 + (row / p.wb) % p.hb;
    n = t.n0 + row / (p.wb * p.hb);
}

// One tile's epilogue for this warp's 32 pixels: alpha*acc + beta*Cin, 32
// channels at a time, through the warp's two slabs and 4-D bulk tensor
// stores (clipped at the edges of D), or plain stores when D's pixel rows
// are not 16-byte aligned.
__device__ __forceinline__ void conv_epilogue(const Params& p, const Tile& t, uint32_t tacc, bool has_k, int q,
                                              int lane, uint8_t* slab, uint32_t slab_s, uint32_t& slab_seq) {
    int n_w, p_w, q_w;  // the warp's first pixel: the origin of its store box
    tile_pixel(p, t, 32 * q, n_w, p_w, q_w);
    if (n_w >= p.N || p_w >= p.P || q_w >= p.Q) return;  // the whole box is outside D
    int n_l, p_l, q_l;
    tile_pixel(p, t, 32 * q + lane, n_l, p_l, q_l);
    const bool px_ok = 32 * q + lane < p.box_rows && n_l < p.N && p_l < p.P && q_l < p.Q;
    const long long pix = ((long long)n_l * p.P + p_l) * p.Q + q_l;
    const float a = p.alpha, b = p.beta;
    for (int c = 0; c < p.bn; c += 32) {
        const int k0 = t.k0 + c;
        if (k0 >= p.K) break;
        float v[32];
        if (has_k) {
            tmem_ld32(tacc + (uint32_t)c, v);
        } else {  // C == 0: no MMA wrote the accumulator
#pragma unroll
            for (int j = 0; j < 32; j++) v[j] = 0.0f;
        }
        float o[32];
#pragma unroll
        for (int j = 0; j < 32; j++) o[j] = a * v[j];
        if (b != 0.0f && px_ok) {
            const float* cr = p.Cin + pix * p.ldc + k0;
            if (p.vec_c && k0 + 32 <= p.K) {
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const float4 x = __ldg(reinterpret_cast<const float4*>(cr) + j);
                    o[4 * j] = fmaf(b, x.x, o[4 * j]);
                    o[4 * j + 1] = fmaf(b, x.y, o[4 * j + 1]);
                    o[4 * j + 2] = fmaf(b, x.z, o[4 * j + 2]);
                    o[4 * j + 3] = fmaf(b, x.w, o[4 * j + 3]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; j++)
                    if (k0 + j < p.K) o[j] = fmaf(b, __ldg(cr + j), o[j]);
            }
        }
        if (p.tma_d) {
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
                tma_store_4d(&p.tmD, slab_s + buf, k0, q_w, p_w, n_w);
                bulk_commit_group();
            }
            ++slab_seq;
        } else if (px_ok) {
            float* dr = p.D + pix * p.ldd + k0;
            if (p.vec_d && k0 + 32 <= p.K) {
#pragma unroll
                for (int j = 0; j < 8; j++)
                    reinterpret_cast<float4*>(dr)[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 32; j++)
                    if (k0 + j < p.K) dr[j] = o[j];
            }
        }
    }
}

// Split-K: this warp's 32 rows of the raw fp32 accumulator into the
// workspace slot of (tile, split), row-major [128][bn], 16-byte stores.
__device__ __forceinline__ void conv_partial(const Params& p, int tile, int sp, uint32_t tacc, bool has_k, int q,
                                             int lane) {
    float* row = p.ws + (((long long)tile * p.splits + sp) * 128 + 32 * q + lane) * p.bn;
    for (int c = 0; c < p.bn; c += 32) {
        float v[32];
        if (has_k) {
            tmem_ld32(tacc + (uint32_t)c, v);
        } else {
#pragma unroll
            for (int j = 0; j < 32; j++) v[j] = 0.0f;
        }
#pragma unroll
        for (int j = 0; j < 8; j++)
            *reinterpret_cast<float4*>(row + c + 4 * j) = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
}

__global__ void __launch_bounds__(kThreads, 1) k_conv_igemm(const __grid_constant__ Params p) {
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
    const int nbox = p.bn >> 6;  // 64-column boxes of the filter per stage

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
        if (p.ksteps > 0) {  // C == 0 leaves the operand maps unencoded
            tma_prefetch_map(&p.tmX);
            tma_prefetch_map(&p.tmF);
        }
        if (p.tma_d) tma_prefetch_map(&p.tmD);
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
    // visible), and every thread waits once more before exit.  The next
    // kernel (the split-K reduction) may start its own set-up early.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0 || warp == 6) {
        grid_dep_wait();
        // ------------------------------ TMA producers (two warps) -------------
        // Stage g of the CTA's sequence uses ring slot g % nst and belongs to
        // warp 0 when g is even, to warp 6 when it is odd.
        const uint32_t pid = warp == 0 ? 0u : 1u;
        uint32_t g = 0, armed_mask = 0, armed_ph = 0;
        // Test hook (failure detection): warp 0 leaves its first stage empty,
        // so the MMA issuer's bounded wait on it runs out.
        bool withhold = pid == 0 && p.inject_timeout != 0;
        for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
            const Tile t = decode_tile(p, u / p.splits);
            int kb0, kb1;
            split_range(p, u % p.splits, kb0, kb1);
            for (int kb = kb0; kb < kb1; kb++, g++) {
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
                const int tap = kb / p.cblocks, cb = kb - tap * p.cblocks;
                const int r = tap / p.S, s = tap - r * p.S;
                const uint32_t st = ring0 + (uint32_t)stage * sb;
                if (lane == 0)
                    tma_load_4d(st, &p.tmX, full(stage), cb * 64, t.q0 + s - p.pad_w, t.p0 + r - p.pad_h, t.n0);
                else if (lane <= nbox)
                    tma_load_3d(st + 16384u + (uint32_t)(lane - 1) * 8192u, &p.tmF, full(stage), t.k0 + 64 * (lane - 1),
                                tap * p.C + cb * 64, 0);
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(full(stage), (uint32_t)(p.box_rows + p.bn) * 128u);
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
                int kb0, kb1;
                split_range(p, u % p.splits, kb0, kb1);
                ok = wait_fast(acce(acc), aph ^ 1u, abort_flag, p.err, kErrWaitAccEmpty, limit);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * 256);
                for (int kb = kb0; kb < kb1; kb++) {
                    ok = wait_fast(full(stage), ph, abort_flag, p.err, kErrWaitFull, limit);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t st = ring0 + (uint32_t)stage * sb;
                    const uint64_t da = desc_kmajor(st, 0), db = desc_mnmajor(st + 16384u, 0);
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        umma_bf16<1>(d, da + 2u * j, db + 128u * j, idesc, (kb > kb0 || j) ? 1u : 0u);
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
        // steps of this CTA's first unit (one K step per lane): the X box and
        // the filter boxes its producers will load.  A prefetch hands no data
        // to the SM, so it may precede the dependency wait.  Its coordinates
        // are clamped into X, and filter boxes past K are left out: every
        // prefetch starts inside its tensor.
        if (warp == 2 && p.l2_pf > 0 && p.ksteps > 0 && (int)blockIdx.x < p.units) {
            const Tile t = decode_tile(p, (int)blockIdx.x / p.splits);
            int kb0, kb1;
            split_range(p, (int)blockIdx.x % p.splits, kb0, kb1);
            const int nk = min(p.l2_pf, kb1 - kb0);
            for (int j = lane; j < nk; j += 32) {
                const int kb = kb0 + j;
                const int tap = kb / p.cblocks, cb = kb - tap * p.cblocks;
                const int r = tap / p.S, s = tap - r * p.S;
                const int qx = min(max(t.q0 + s - p.pad_w, 0), p.W - 1);
                const int py = min(max(t.p0 + r - p.pad_h, 0), p.H - 1);
                tma_prefetch_l2_4d(&p.tmX, cb * 64, qx, py, t.n0);
                for (int b = 0; b < nbox && t.k0 + 64 * b < p.K; b++)
                    tma_prefetch_l2_3d(&p.tmF, t.k0 + 64 * b, tap * p.C + cb * 64, 0);
            }
        }
        grid_dep_wait();
        const int q = warp & 3;
        uint8_t* slab = gbase + (epi0 - base) + q * kEpiSlabBytes;
        const uint32_t slab_s = epi0 + (uint32_t)(q * kEpiSlabBytes);
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        int acc = 0;
        uint32_t aph = 0, slab_seq = 0;
        for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
            const int tile = u / p.splits, sp = u % p.splits;
            int kb0, kb1;
            split_range(p, sp, kb0, kb1);
            int w = 1;
            if (lane == 0) w = wait_fast(accf(acc), aph, abort_flag, p.err, kErrWaitAccFull, limit) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, w, 0)) break;
            tc_fence_after();
            const uint32_t tacc = tmem + (uint32_t)(acc * 256) + lane_off;
            if (p.splits > 1)
                conv_partial(p, tile, sp, tacc, kb1 > kb0, q, lane);
            else
                conv_epilogue(p, decode_tile(p, tile), tacc, kb1 > kb0, q, lane, slab, slab_s, slab_seq);
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

// Split-K reduction: thread i handles 4 channels of one tile row; the splits
// are summed in order, then the epilogue arithmetic of the one-pass path.
__global__ void __launch_bounds__(256) k_conv_reduce(const __grid_constant__ Params p) {
    // Launched as a programmatic dependent of the convolution kernel: wait
    // until it has finished and its partials are visible.
    grid_dep_wait();
    const int groups = p.bn >> 2;
    const long long total = (long long)p.tiles * 128 * groups;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int g4 = (int)(i % groups);
        const long long tr = i / groups;
        const int row = (int)(tr % 128);
        const int tile = (int)(tr / 128);
        const Tile t = decode_tile(p, tile);
        int n, ph, qw;
        tile_pixel(p, t, row, n, ph, qw);
        const int k = t.k0 + 4 * g4;
        if (row >= p.box_rows || n >= p.N || ph >= p.P || qw >= p.Q || k >= p.K) continue;
        const float* src = p.ws + ((long long)tile * p.splits * 128 + row) * p.bn + 4 * g4;
        float4 acc = __ldcg(reinterpret_cast<const float4*>(src));
        for (int s = 1; s < p.splits; s++) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(src + (long long)s * 128 * p.bn));
            acc.x += x.x;
            acc.y += x.y;
            acc.z += x.z;
            acc.w += x.w;
        }
        const long long pix = ((long long)n * p.P + ph) * p.Q + qw;
        float o[4] = {p.alpha * acc.x, p.alpha * acc.y, p.alpha * acc.z, p.alpha * acc.w};
#pragma unroll
        for (int e = 0; e < 4; e++) {
            if (k + e >= p.K) break;
            if (p.beta != 0.0f) o[e] = fmaf(p.beta, __ldg(p.Cin + pix * p.ldc + k + e), o[e]);
            p.D[pix * p.ldd + k + e] = o[e];
        }
    }
}

cudaError_t launch_reduce(cudaStream_t stream, const Params& p) {
    const long long total = (long long)p.tiles * 128 * (p.bn >> 2);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min<long long>((total + 255) / 256, 152LL * 8));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_conv_reduce, p);
}

cudaError_t launch(const cudaLaunchConfig_t& cfg, const Params& p) {
    return cudaLaunchKernelEx(&cfg, k_conv_igemm, p);
}

bool set_smem() {
    return cudaFuncSetAttribute(k_conv_igemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) ==
           cudaSuccess;
}

}  // namespace conv
}  // namespace mp
