// The fused back-to-back GEMM kernel (see mp_b2b.cuh for the operation and
// the work decomposition).
//
// Roles (224 threads): warps 0 and 6 issue the TMA copies of alternate ring
// stages, lane 0 of warp 1 issues every tcgen05.mma and commit, warps 2..5
// run the epilogues (warp w reads TMEM lanes 32*(w%4)..+31, i.e. those rows
// of the tile).  One ring of
// shared-memory stages carries, per work unit, the first GEMM's K steps (an
// A0 box of 128 x 64 and the 64 x n0p W0 boxes) and then, per chunk of D1,
// the second GEMM's K steps (64 x bn1 W1 boxes).  Two TMEM accumulators of
// 256 columns alternate over the sequence D0, D1 chunk, D1 chunk, ...
//
// Hand-over of D0: the epilogue warps read the first GEMM's accumulator,
// apply alpha0, beta0*C0 and the activation, round to bf16 and write the
// 128 x n0p block into shared memory in the layout a TMA load of a K-major
// A tile would give (64-column atoms of 128 rows x 128 bytes, 16-byte chunks
// swizzled by row % 8).  Each writer fences its stores into the async proxy
// and the four warps arrive on `d0full`; the MMA issuer waits for it before
// the first MMA of the second GEMM.  The next unit's D0 overwrites the block
// only after the epilogue has drained the unit's last D1 chunk, whose commit
// follows every MMA that read the block.
//
// Every wait is bounded (1 s by default): on expiry the CTA records an error
// code in the handle's status word, the other roles stop, the producer waits
// (bounded) for its copies in flight, the MMA issuer for its MMAs, and the
// CTA frees TMEM and returns.

#include "mp_kernel.cuh"
#include "mp_b2b.cuh"

namespace mp {
namespace b2b {

using namespace mp::dev;

constexpr int kErrWaitD0 = 7;  // the MMA issuer gave up waiting for D0 in shared memory

// 64 consecutive accumulator columns of this thread's TMEM lane, one load
// and one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* v) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
        "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]),
                   "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]),
                   "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]),
                   "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]),
                   "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
                 :
                 : "memory");
#pragma unroll
    for (int i = 0; i < 64; i++) v[i] = __uint_as_float(r[i]);
}

// Columns [c, c + 64) of this lane's row of the D0 block (one swizzle atom):
// alpha0*acc + beta0*C0, the activation, bf16, into the K-major operand.
template <int ACT>
__device__ __forceinline__ void d0_atom(const Params& p, uint32_t t, bool has_k, int row, int r, int c,
                                        uint8_t* d0g) {
    float v[64];
    if (has_k) {
        tmem_ld64(t + (uint32_t)c, v);
    } else {
#pragma unroll
        for (int j = 0; j < 64; j++) v[j] = 0.0f;
    }
    const float a = p.alpha0, b = p.beta0;
    const bool row_ok = row < p.M;
    uint8_t* line = d0g + (c >> 6) * 16384 + r * 128;
#pragma unroll
    for (int h = 0; h < 2; h++) {  // 32 columns = four 16-byte chunks of bf16 at a time
        float cv[32];
        if (b != 0.0f) {
            const int cc = c + 32 * h;
            const float* cr = p.C0 + (long long)row * p.ldc0 + cc;
            if (row_ok && p.vec_c0 && cc + 32 <= p.N0) {
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const float4 x = __ldg(reinterpret_cast<const float4*>(cr) + j);
                    cv[4 * j] = x.x;
                    cv[4 * j + 1] = x.y;
                    cv[4 * j + 2] = x.z;
                    cv[4 * j + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; j++) cv[j] = (row_ok && cc + j < p.N0) ? __ldg(cr + j) : 0.0f;
            }
        }
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; j++) {
            float x0 = a * v[32 * h + 2 * j], x1 = a * v[32 * h + 2 * j + 1];
            if (b != 0.0f) {
                x0 = fmaf(b, cv[2 * j], x0);
                x1 = fmaf(b, cv[2 * j + 1], x1);
            }
            const __nv_bfloat162 hv = __floats2bfloat162_rn(act_fn<ACT>(x0), act_fn<ACT>(x1));
            pk[j] = *reinterpret_cast<const uint32_t*>(&hv);
        }
#pragma unroll
        for (int i = 0; i < 4; i++)
            *reinterpret_cast<uint4*>(line + (((4 * h + i) ^ (r & 7)) << 4)) =
                make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
    }
}

template <int ACT>
__device__ __forceinline__ void d0_block(const Params& p, uint32_t t, bool has_k, int row, int r, uint8_t* d0g) {
    for (int c = 0; c < p.n0p; c += 64) d0_atom<ACT>(p, t, has_k, row, r, c, d0g);
}

// One chunk of D1 for this warp's 32 rows: alpha1*acc + beta1*C1, 64 columns
// of TMEM at a time, stored as 32 x 16 boxes through the warp's two
// slabs in turn (bulk tensor stores clip rows and columns past the edge; a
// slab is rewritten once its previous store has read it, while the other
// slab's store may still be in flight), or with plain stores when D1's rows
// are not 16-byte aligned.  `slab_seq` counts this warp's stores.
__device__ __forceinline__ void d1_chunk(const Params& p, uint32_t t, bool has_k, int m_w, int lane, int n_base,
                                         uint8_t* slab, uint32_t slab_s, uint32_t& slab_seq) {
    if (m_w >= p.M) return;  // the whole warp is past the last row
    const int row = m_w + lane;
    const bool row_ok = row < p.M;
    const float a = p.alpha1, b = p.beta1;
    for (int c = 0; c < p.bn1; c += 64) {  // one TMEM round trip per 64 columns
        if (n_base + c >= p.N1) break;
        float v[64];
        if (has_k) {
            tmem_ld64(t + (uint32_t)c, v);
        } else {
#pragma unroll
            for (int j = 0; j < 64; j++) v[j] = 0.0f;
        }
#pragma unroll
        for (int h = 0; h < 2; h++) {
            const int n0 = n_base + c + 32 * h;
            if (n0 >= p.N1) break;
            float o[32];
#pragma unroll
            for (int j = 0; j < 32; j++) o[j] = a * v[32 * h + j];
            if (b != 0.0f) {
                const float* cr = p.C1 + (long long)row * p.ldc1 + n0;
                if (row_ok && p.vec_c1 && n0 + 32 <= p.N1) {
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
                        if (row_ok && n0 + j < p.N1) o[j] = fmaf(b, __ldg(cr + j), o[j]);
                }
            }
            if (p.tma_d) {
#pragma unroll
                for (int hh = 0; hh < 2; hh++) {
                    const int nh = n0 + 16 * hh;
                    if (nh >= p.N1) break;
                    const uint32_t buf = (slab_seq & 1u) * 2048u;
                    if (lane == 0) bulk_wait_read_1();  // this slab's previous store has read it
                    __syncwarp();
                    // 64-byte rows, 64-byte swizzle: chunk j of row `lane` at j ^ ((lane >> 1) & 3).
                    uint8_t* line = slab + buf + lane * 64;
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        *reinterpret_cast<float4*>(line + ((j ^ ((lane >> 1) & 3)) << 4)) =
                            make_float4(o[16 * hh + 4 * j], o[16 * hh + 4 * j + 1], o[16 * hh + 4 * j + 2],
                                        o[16 * hh + 4 * j + 3]);
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&p.tmD1, slab_s + buf, nh, m_w, 0);
                        bulk_commit_group();
                    }
                    ++slab_seq;
                }
            } else if (row_ok) {
                float* dr = p.D1 + (long long)row * p.ldd1 + n0;
#pragma unroll
                for (int j = 0; j < 32; j++)
                    if (n0 + j < p.N1) dr[j] = o[j];
            }
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1) k_b2b_gemm(const __grid_constant__ Params p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const int nst = p.num_stages;
    const uint32_t sb = (uint32_t)p.stage_bytes;  // a multiple of 8 KB
    const uint32_t ring0 = base;
    const uint32_t d0s = ring0 + (uint32_t)nst * sb;      // 1 KB aligned: the swizzle atoms
    const uint32_t epi0 = d0s + (uint32_t)p.n0p * 256u;   // 128 rows x n0p bf16
    const uint32_t bar0 = epi0 + 4u * kEpiSlabBytes;
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
    auto accf = [&](int b) { return bar0 + 8u * (2 * kMaxStages + b); };
    auto acce = [&](int b) { return bar0 + 8u * (2 * kMaxStages + 2 + b); };
    const uint32_t d0full = bar0 + 8u * (2 * kMaxStages + 4);
    const uint32_t done_bar = bar0 + 8u * (2 * kMaxStages + 5);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar0 - base) + 8 * (2 * kMaxStages + 6));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint64_t limit = p.wait_limit_ns;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nk0 = (p.K0 + 63) >> 6;  // first GEMM: K steps of 64
    const int nk1 = p.n0p >> 6;        // second GEMM: K = n0p
    // Units are numbered row block by row block, so the units that share a
    // block of A0 (and recompute its D0) run side by side and read it from L2.
    const int groups = (p.chunks + p.cpg - 1) / p.cpg;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; s++) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(accf(b), 1);
            mbar_init(acce(b), 4);
        }
        mbar_init(d0full, 4);
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (nk0 > 0) {
            tma_prefetch_map(&p.tmA0);
            tma_prefetch_map(&p.tmW0);
        }
        if (nk1 > 0) tma_prefetch_map(&p.tmW1);
        if (p.tma_d) tma_prefetch_map(&p.tmD1);
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
        // Lane 0 probes the slot; the copies of one stage go out from
        // different lanes (A0 from lane 0 and W0 boxes from lanes 1..; or the
        // W1 boxes from lanes 0..), then lane 0 arms the stage with its bytes
        // (full boxes: TMA fills out-of-range elements with zeros and still
        // counts them).
        const uint32_t pid = warp == 0 ? 0u : 1u;
        uint32_t g = 0, armed_mask = 0, armed_ph = 0;
        // Test hook (failure detection): warp 0 leaves its first stage empty,
        // so the MMA issuer's bounded wait on it runs out.
        bool withhold = pid == 0 && p.inject_timeout != 0;
        for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
            const int mb = u / groups, grp = u % groups;
            const int m0 = mb * 128;
            const int c0 = grp * p.cpg, c1 = min(p.chunks, c0 + p.cpg);
            const int steps = nk0 + (c1 - c0) * nk1;
            for (int i = 0; i < steps; i++, g++) {
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
                uint32_t bytes;
                if (i < nk0) {
                    const int kc = i * 64;
                    if (lane == 0)
                        tma_load_3d(st, &p.tmA0, full(stage), kc, m0, 0);
                    else if (lane <= nk1)
                        tma_load_3d(st + 16384u + (uint32_t)(lane - 1) * 8192u, &p.tmW0, full(stage), 64 * (lane - 1),
                                    kc, 0);
                    bytes = 16384u + (uint32_t)p.n0p * 128u;
                } else {
                    const int j = i - nk0, c = c0 + j / nk1, kk = j % nk1;
                    if (lane < (p.bn1 >> 6))
                        tma_load_3d(st + (uint32_t)lane * 8192u, &p.tmW1, full(stage), c * p.bn1 + 64 * lane, kk * 64,
                                    0);
                    bytes = (uint32_t)p.bn1 * 128u;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_expect_tx(full(stage), bytes);
                armed_mask |= 1u << stage;
                armed_ph = (armed_ph & ~(1u << stage)) | (ph << stage);
            }
        }
    producer_out:
        if (lane == 0 && *abort_flag) {
            // Let every copy this warp started land before the CTA exits.
            for (int s = 0; s < nst; s++)
                if (armed_mask & (1u << s))
                    wait_bounded(full(s), (armed_ph >> s) & 1u, abort_flag, p.err, kErrDrain, limit, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer (lane 0) --------------------
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t ph = 0, aph = 0, uc = 0;
            const uint32_t id0 = idesc_bf16(p.n0p > 0 ? p.n0p : 64, false, true);
            const uint32_t id1 = idesc_bf16(p.bn1, false, true);
            bool ok = true;
            for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x, uc++) {
                const int grp = u % groups;
                const int c0 = grp * p.cpg, c1 = min(p.chunks, c0 + p.cpg);
                // First GEMM: D0 accumulator.
                ok = wait_fast(acce(acc), aph ^ 1u, abort_flag, p.err, kErrWaitAccEmpty, limit);
                if (!ok) break;
                tc_fence_after();
                uint32_t d = tmem + (uint32_t)(acc * 256);
                for (int kb = 0; kb < nk0; kb++) {
                    ok = wait_fast(full(stage), ph, abort_flag, p.err, kErrWaitFull, limit);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t st = ring0 + (uint32_t)stage * sb;
                    const uint64_t da = desc_kmajor(st, 0), db = desc_mnmajor(st + 16384u, 0);
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        umma_bf16<1>(d, da + 2u * j, db + 128u * j, id0, (kb | j) ? 1u : 0u);
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
                // Second GEMM, chunk by chunk, once D0 is in shared memory.
                ok = wait_fast(d0full, uc & 1u, abort_flag, p.err, kErrWaitD0, limit);
                if (!ok) break;
                tc_fence_after();
                for (int c = c0; c < c1; c++) {
                    ok = wait_fast(acce(acc), aph ^ 1u, abort_flag, p.err, kErrWaitAccEmpty, limit);
                    if (!ok) break;
                    tc_fence_after();
                    d = tmem + (uint32_t)(acc * 256);
                    for (int kk = 0; kk < nk1; kk++) {
                        ok = wait_fast(full(stage), ph, abort_flag, p.err, kErrWaitFull, limit);
                        if (!ok) break;
                        tc_fence_after();
                        const uint64_t da = desc_kmajor(d0s + (uint32_t)kk * 16384u, 0);
                        const uint64_t db = desc_mnmajor(ring0 + (uint32_t)stage * sb, 0);
#pragma unroll
                        for (int j = 0; j < 4; j++)
                            umma_bf16<1>(d, da + 2u * j, db + 128u * j, id1, (kk | j) ? 1u : 0u);
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
            }
            // Every MMA this thread issued has completed once `done_bar` flips.
            umma_commit(done_bar);
            wait_bounded(done_bar, 0, abort_flag, p.err, kErrDrain, limit, false);
        }
        __syncwarp();
    } else {
        // ------------------------------ epilogue (128 threads) ----------------
        // While the previous kernel may still run, warm L2 with the first
        // GEMM's leading K steps of this CTA's first unit (one K step per
        // lane: the A0 box and the W0 boxes that start inside N0).  A
        // prefetch hands no data to the SM, so it may precede the wait.
        if (warp == 2 && p.l2_pf > 0 && nk0 > 0 && (int)blockIdx.x < p.units) {
            const int m0 = ((int)blockIdx.x / groups) * 128;
            const int nk = min(p.l2_pf, nk0);
            for (int j = lane; j < nk; j += 32) {
                tma_prefetch_l2_3d(&p.tmA0, j * 64, m0, 0);
                for (int b = 0; b < nk1 && 64 * b < p.N0; b++) tma_prefetch_l2_3d(&p.tmW0, 64 * b, j * 64, 0);
            }
        }
        grid_dep_wait();
        const int q = warp & 3;  // TMEM lane quarter = rows 32q..32q+31 of the tile
        uint8_t* slab = gbase + (epi0 - base) + q * kEpiSlabBytes;
        const uint32_t slab_s = epi0 + (uint32_t)(q * kEpiSlabBytes);
        uint8_t* d0g = gbase + (d0s - base);
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const bool has_k0 = nk0 > 0, has_k1 = nk1 > 0;
        int acc = 0;
        uint32_t aph = 0, slab_seq = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
            const int mb = u / groups, grp = u % groups;
            const int m0 = mb * 128;
            const int c0 = grp * p.cpg, c1 = min(p.chunks, c0 + p.cpg);
            int w = 1;
            if (lane == 0) w = wait_fast(accf(acc), aph, abort_flag, p.err, kErrWaitAccFull, limit) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, w, 0)) break;
            tc_fence_after();
            const uint32_t t0 = tmem + (uint32_t)(acc * 256) + lane_off;
            const int r = 32 * q + lane;
            if (p.act0 == 1)
                d0_block<1>(p, t0, has_k0, m0 + r, r, d0g);
            else if (p.act0 == 2)
                d0_block<2>(p, t0, has_k0, m0 + r, r, d0g);
            else
                d0_block<0>(p, t0, has_k0, m0 + r, r, d0g);
            fence_async_smem();  // this thread's D0 stores, into the async proxy
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(acce(acc));
                mbar_arrive(d0full);
            }
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
            for (int c = c0; c < c1; c++) {
                if (lane == 0) w = wait_fast(accf(acc), aph, abort_flag, p.err, kErrWaitAccFull, limit) ? 1 : 0;
                if (!__shfl_sync(0xffffffffu, w, 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t t1 = tmem + (uint32_t)(acc * 256) + lane_off;
                d1_chunk(p, t1, has_k1, m0 + 32 * q, lane, c * p.bn1, slab, slab_s, slab_seq);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce(acc));
                acc ^= 1;
                if (acc == 0) aph ^= 1u;
            }
        }
        if (lane == 0) bulk_wait_all();  // the stores have finished before the CTA exits
        __syncwarp();
    }
    grid_dep_wait();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<1>(tmem, 512);
    }
}

cudaError_t launch(const cudaLaunchConfig_t& cfg, const Params& p) { return cudaLaunchKernelEx(&cfg, k_b2b_gemm, p); }

bool set_smem() {
    return cudaFuncSetAttribute(k_b2b_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit) == cudaSuccess;
}

}  // namespace b2b
}  // namespace mp
