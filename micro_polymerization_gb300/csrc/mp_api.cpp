// The C ABI: handle lifecycle, argument checking and dispatch to the planner
// and the device code.  Every entry point returns an mp_status; nothing here
// throws across the boundary or falls back to host arithmetic.
#include <cerrno>
#include <cstdio>
#include <dlfcn.h>
#include <string>
#include <cstdlib>
#include <cstring>
#include <new>

#include <algorithm>
#include <climits>

#include <vector>

#include "mp_internal.h"

namespace {

constexpr int64_t kMaxDim = (int64_t)1 << 31;  // sizes and offsets fit int32 on the device

double env_double(const char* name, double dflt) {
    const char* v = std::getenv(name);
    if (!v || !*v) return dflt;
    char* end = nullptr;
    double x = std::strtod(v, &end);
    return (end && end != v && x > 0) ? x : dflt;
}

// Calibration table: "um un uk swap fixed_us per_step_us [tail_us]" per
// micro-kernel (a line without tail_us keeps the kernel's tail), and
// "split on_chip sync_us bytes_factor [S]" for the split-K reduction (on_chip
// 0: through L2; 1: on chip, for cluster size S or, without S, every size).
// One split-K cost entry (see mp_set_split_model); false if out of range.
bool set_split_model(mp_handle h, int on_chip, int S, double sync_us, double factor) {
    if (!(sync_us >= 0) || !(factor >= 0)) return false;
    if (on_chip == 0 && S == 0) {
        h->split_sync_us[0] = sync_us;
        h->split_bytes_factor[0] = factor;
        return true;
    }
    if (on_chip != 1 || (S != 0 && (S < 2 || S > mp::kClusterSplitMaxS))) return false;
    for (int s = 2; s <= mp::kClusterSplitMaxS; s++) {
        if (S == 0 || s == S) {
            h->split_sync_us[s] = sync_us;
            h->split_bytes_factor[s] = factor;
        }
    }
    return true;
}

// Returns false when the file cannot be opened.
bool load_calibration(mp_handle h, const char* path) {
    if (!path || !*path) return false;
    FILE* f = std::fopen(path, "r");
    if (!f) return false;
    char line[512];
    while (std::fgets(line, sizeof line, f)) {
        char* hash = std::strchr(line, '#');
        if (hash) *hash = 0;
        int on_chip, S = 0;
        double sync_us, factor;
        const int sg = std::sscanf(line, " split %d %lf %lf %d", &on_chip, &sync_us, &factor, &S);
        if (sg >= 3) {
            if (sg == 3) S = 0;
            set_split_model(h, on_chip, S, sync_us, factor);
            continue;
        }
        int um, un, uk, swap;
        double fixed, step, tail = -1.0;
        const int got = std::sscanf(line, "%d %d %d %d %lf %lf %lf", &um, &un, &uk, &swap, &fixed, &step, &tail);
        if (got < 6) continue;
        if (!(fixed >= 0) || !(step > 0)) continue;
        for (int k = 0; k < h->num_kernels; k++) {
            mp_kernel_desc& d = h->kernels[k];
            if (d.um == um && d.un == un && d.uk == uk && d.swap == swap) {
                d.fixed_us = fixed;
                d.per_step_us = step;
                if (got == 7 && tail >= 0) d.tail_us = tail;
                h->calibrated = true;
            }
        }
    }
    std::fclose(f);
    mp::clear_plan_cache(h);
    return true;
}

// The measured table shipped with the library: the library is
// <package>/_lib/libmp.so and the table <package>/calib/gb300.txt.  Empty if
// the library's own path cannot be found.
std::string shipped_calibration() {
    Dl_info info;
    if (!dladdr(reinterpret_cast<void*>(&mp_init), &info) || !info.dli_fname) return {};
    std::string p = info.dli_fname;
    for (int up = 0; up < 2; up++) {
        const size_t cut = p.find_last_of('/');
        if (cut == std::string::npos) return {};
        p.resize(cut);
    }
    return p + "/calib/gb300.txt";
}

mp_handle new_handle() {
    mp_handle h = new (std::nothrow) mp_handle_s();
    if (!h) return nullptr;
    // MP_PLAN_CACHE=0: no plan cache, so that every call runs the search.
    const char* pc = std::getenv("MP_PLAN_CACHE");
    try {
        if (!(pc && pc[0] == '0')) h->cache.resize(4096);
    } catch (...) {
        delete h;
        return nullptr;
    }
    return h;
}

// Byte extent [lo, hi) of a row-major matrix block.
struct Span {
    uintptr_t lo, hi;
};

Span span_of(const void* p, int64_t rows, int64_t cols, int64_t ld, int64_t elem, int64_t batch,
             int64_t stride) {
    uintptr_t lo = (uintptr_t)p;
    int64_t last = (rows - 1) * ld + cols;  // elements from the first to one past the last
    if (batch > 1) last += (batch - 1) * stride;
    return Span{lo, lo + (uintptr_t)(last * elem)};
}

bool overlap(const Span& a, const Span& b) { return a.lo < b.hi && b.lo < a.hi; }

mp_status check_args(const mp::GemmArgs& a) {
    const int64_t batch = a.batch, M = a.M, N = a.N, K = a.K;
    if (batch < 0 || M < 0 || N < 0 || K < 0) return MP_ERR_INVALID_ARG;
    if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim || batch >= kMaxDim) return MP_ERR_INVALID_ARG;
    const int act = a.epilogue & 0xff;
    const bool d_bf16 = (a.epilogue & MP_EPI_OUT_BF16) != 0;
    if ((a.epilogue & ~(0xff | MP_EPI_OUT_BF16)) != 0 || act > MP_ACT_GELU) return MP_ERR_INVALID_ARG;
    if (batch == 0 || M == 0 || N == 0) return MP_OK;
    const int64_t d_elem = d_bf16 ? 2 : 4;
    if (!a.D) return MP_ERR_INVALID_ARG;
    if (a.ldd < (N > 1 ? N : 1)) return MP_ERR_INVALID_ARG;
    if (((uintptr_t)a.D & (uintptr_t)(d_elem - 1)) != 0) return MP_ERR_INVALID_ARG;
    if (a.strideA < 0 || a.strideB < 0 || a.strideC < 0 || a.strideD < 0) return MP_ERR_INVALID_ARG;
    if (K > 0) {
        if (!a.A || !a.B) return MP_ERR_INVALID_ARG;
        if (a.lda < K || a.ldb < (N > 1 ? N : 1)) return MP_ERR_INVALID_ARG;
        if (((uintptr_t)a.A & 1) != 0 || ((uintptr_t)a.B & 1) != 0) return MP_ERR_INVALID_ARG;
    }
    const bool read_c = a.beta != 0.0f;
    if (read_c) {
        if (!a.C || a.ldc < (N > 1 ? N : 1)) return MP_ERR_INVALID_ARG;
        if (((uintptr_t)a.C & 3) != 0) return MP_ERR_INVALID_ARG;
    }
    // Distinct problems of a batch must write disjoint D blocks.
    if (batch > 1 && a.strideD < (M - 1) * a.ldd + N) return MP_ERR_INVALID_ARG;
    const Span d = span_of(a.D, M, N, a.ldd, d_elem, batch, a.strideD);
    if (K > 0) {
        if (overlap(d, span_of(a.A, M, K, a.lda, 2, batch, a.strideA))) return MP_ERR_INVALID_ARG;
        if (overlap(d, span_of(a.B, K, N, a.ldb, 2, batch, a.strideB))) return MP_ERR_INVALID_ARG;
    }
    if (read_c) {
        // In place needs C and D of one type: fp32 D only.
        const bool in_place =
            !d_bf16 && a.C == a.D && a.ldc == a.ldd && (batch == 1 || a.strideC == a.strideD);
        if (!in_place && overlap(d, span_of(a.C, M, N, a.ldc, 4, batch, a.strideC)))
            return MP_ERR_INVALID_ARG;
    }
    return MP_OK;
}

// Argument rules of mp_gemm_b2b (include/mp.h).
mp_status check_b2b(const mp::B2BArgs& a) {
    const int64_t M = a.M, N0 = a.N0, N1 = a.N1, K0 = a.K0;
    if (M < 0 || N0 < 0 || N1 < 0 || K0 < 0) return MP_ERR_INVALID_ARG;
    if (M >= kMaxDim || N0 >= kMaxDim || N1 >= kMaxDim || K0 >= kMaxDim) return MP_ERR_INVALID_ARG;
    if (a.act0 < MP_ACT_NONE || a.act0 > MP_ACT_GELU) return MP_ERR_INVALID_ARG;
    if (M == 0 || N1 == 0) return MP_OK;
    auto one = [](int64_t n) { return n > 1 ? n : (int64_t)1; };
    if (!a.D1 || a.ldd1 < one(N1) || ((uintptr_t)a.D1 & 3) != 0) return MP_ERR_INVALID_ARG;
    const bool first = N0 > 0 && K0 > 0, read_c0 = N0 > 0 && a.beta0 != 0.0f, second = N0 > 0;
    const bool read_c1 = a.beta1 != 0.0f;
    if (first) {
        if (!a.A0 || !a.W0 || a.lda0 < K0 || a.ldw0 < one(N0)) return MP_ERR_INVALID_ARG;
        if (((uintptr_t)a.A0 & 1) != 0 || ((uintptr_t)a.W0 & 1) != 0) return MP_ERR_INVALID_ARG;
    }
    if (read_c0 && (!a.C0 || a.ldc0 < one(N0) || ((uintptr_t)a.C0 & 3) != 0)) return MP_ERR_INVALID_ARG;
    if (second && (!a.W1 || a.ldw1 < one(N1) || ((uintptr_t)a.W1 & 1) != 0)) return MP_ERR_INVALID_ARG;
    if (read_c1 && (!a.C1 || a.ldc1 < one(N1) || ((uintptr_t)a.C1 & 3) != 0)) return MP_ERR_INVALID_ARG;
    const Span d = span_of(a.D1, M, N1, a.ldd1, 4, 1, 0);
    if (first && (overlap(d, span_of(a.A0, M, K0, a.lda0, 2, 1, 0)) || overlap(d, span_of(a.W0, K0, N0, a.ldw0, 2, 1, 0))))
        return MP_ERR_INVALID_ARG;
    if (read_c0 && overlap(d, span_of(a.C0, M, N0, a.ldc0, 4, 1, 0))) return MP_ERR_INVALID_ARG;
    if (second && overlap(d, span_of(a.W1, N0, N1, a.ldw1, 2, 1, 0))) return MP_ERR_INVALID_ARG;
    if (read_c1 && !(a.C1 == a.D1 && a.ldc1 == a.ldd1) && overlap(d, span_of(a.C1, M, N1, a.ldc1, 4, 1, 0)))
        return MP_ERR_INVALID_ARG;
    return MP_OK;
}

// Argument rules of mp_conv2d (include/mp.h).
mp_status check_conv(const mp::ConvArgs& a) {
    if (a.N < 0 || a.H < 0 || a.W < 0 || a.C < 0 || a.K < 0 || a.R < 1 || a.S < 1 || a.pad_h < 0 || a.pad_w < 0)
        return MP_ERR_INVALID_ARG;
    for (int64_t v : {a.N, a.H, a.W, a.C, a.K, a.R, a.S, a.pad_h, a.pad_w})
        if (v >= kMaxDim) return MP_ERR_INVALID_ARG;
    const int64_t P = a.H + 2 * a.pad_h - a.R + 1, Q = a.W + 2 * a.pad_w - a.S + 1;
    if (a.N == 0 || a.K == 0 || P <= 0 || Q <= 0) return MP_OK;
    if (a.N * a.H * a.W >= kMaxDim || a.N * P * Q >= kMaxDim || a.R * a.S * (a.C + 63) >= kMaxDim)
        return MP_ERR_INVALID_ARG;
    if (!a.D || a.ldd < a.K || ((uintptr_t)a.D & 3) != 0) return MP_ERR_INVALID_ARG;
    const bool reads_x = a.C > 0, read_c = a.beta != 0.0f;
    if (reads_x && (!a.X || !a.F || ((uintptr_t)a.X & 1) != 0 || ((uintptr_t)a.F & 1) != 0)) return MP_ERR_INVALID_ARG;
    if (read_c && (!a.Cin || a.ldc < a.K || ((uintptr_t)a.Cin & 3) != 0)) return MP_ERR_INVALID_ARG;
    const Span d = span_of(a.D, a.N * P * Q, a.K, a.ldd, 4, 1, 0);
    if (reads_x && (overlap(d, span_of(a.X, a.N * a.H * a.W, a.C, a.C, 2, 1, 0)) ||
                    overlap(d, span_of(a.F, a.R * a.S * a.C, a.K, a.K, 2, 1, 0))))
        return MP_ERR_INVALID_ARG;
    if (read_c && !(a.Cin == a.D && a.ldc == a.ldd) && overlap(d, span_of(a.Cin, a.N * P * Q, a.K, a.ldc, 4, 1, 0)))
        return MP_ERR_INVALID_ARG;
    return MP_OK;
}

// The fused plan and the form mp_gemm_b2b runs.  The fused kernel costs its
// own estimate plus 2.0 us (launch, fill and drain, which its model leaves
// out).  The two-launch form costs the GEMM planner's estimates of both GEMMs
// plus what they leave out, which depends on the GEMM model:
//   - measured table (the default): less 1.5 us (the second launch's set-up
//     overlaps the first), plus D0's write and read (4 M N0 bytes) at
//     1.87 TB/s, which a single GEMM's estimate does not see.  Fitted on GB300
//     to every problem of the two fused-pair workloads (128 problems), each
//     timed in both forms on cold operands: rms error of the two-launch
//     estimate 0.46 us, of the fused one 0.91 us.  Fused unless two launches
//     are predicted faster by more than 5%.
//   - analytic model (no launch costs in the GEMM estimates): plus 7.7 us,
//     fitted to the same two workloads' step times; fused unless two launches
//     are predicted faster by more than 10%.
// N0 > 256 (a D0 row too wide for one accumulator) always runs as two
// launches.
constexpr double kB2BFusedFixedUs = 2.0;
constexpr double kB2BTwoLaunchFixedUs[2] = {7.7, -1.5};     // analytic, measured
constexpr double kB2BD0RoundTripGBs = 1870.0;               // measured table only
constexpr double kB2BMargin[2] = {1.10, 1.05};

mp_status plan_b2b_mode(mp_handle h, int64_t M, int64_t N0, int64_t N1, int64_t K0, mp_b2b_plan* out) {
    mp_status st = mp::plan_b2b(h->hw, M, N0, N1, K0, out);
    const bool wide = st == MP_ERR_UNSUPPORTED && N0 > 256;
    if (wide) {
        if (h->b2b_mode == MP_B2B_FUSED) return MP_ERR_UNSUPPORTED;
        std::memset(out, 0, sizeof(*out));
    } else if (st != MP_OK) {
        return st;
    }
    mp_plan_info p0, p1;
    const int64_t k0 = N0 > 0 ? K0 : 0;
    const int cal = h->calibrated ? 1 : 0;
    double two = kB2BTwoLaunchFixedUs[cal];
    if (cal) two += 4.0 * (double)M * (double)N0 / (kB2BD0RoundTripGBs * 1e3);
    if (N0 > 0) {
        if ((st = mp::plan_shape(h, 1, M, N0, k0, &p0)) != MP_OK) return st;
        two += p0.cost_us;
    }
    if ((st = mp::plan_shape(h, 1, M, N1, N0, &p1)) != MP_OK) return st;
    two += p1.cost_us;
    out->two_launch_cost_us = two;
    if (wide)
        out->mode = MP_B2B_TWO_LAUNCH;
    else if (h->b2b_mode != MP_B2B_AUTO)
        out->mode = h->b2b_mode;
    else
        out->mode = (out->cost_us + kB2BFusedFixedUs <= kB2BMargin[cal] * two) ? MP_B2B_FUSED : MP_B2B_TWO_LAUNCH;
    return MP_OK;
}

mp_status run(mp_handle h, const mp::GemmArgs& a) {
    if (!h) return MP_ERR_INVALID_ARG;
    mp_status st = check_args(a);
    if (st != MP_OK) return st;
    if (a.batch == 0 || a.M == 0 || a.N == 0) return MP_OK;
    if (h->host_only) return MP_ERR_UNSUPPORTED;
    mp_plan_info plan;
    st = mp::plan_shape(h, a.batch, a.M, a.N, a.K, &plan);
    if (st != MP_OK) return st;
    return mp::device_run(h, plan, a);
}

}  // namespace

mp_status mp::validate_args(const mp::GemmArgs& a) { return check_args(a); }

extern "C" {

mp_status mp_init(mp_handle* out, int device, const char* calib_path) {
    if (!out) return MP_ERR_INVALID_ARG;
    *out = nullptr;
    if (device < 0) return MP_ERR_INVALID_ARG;
    mp_handle h = new_handle();
    if (!h) return MP_ERR_NO_MEMORY;
    h->host_only = false;
    h->device = device;
    mp_status st = mp::device_init(h, device);  // fills H and allocates device state
    if (st != MP_OK) {
        mp::device_destroy(h);
        delete h;
        return st;
    }
    h->hw.hbm_gbs = env_double("MP_HBM_GBS", h->hw.hbm_gbs);
    h->hw.l2_gbs = env_double("MP_L2_GBS", h->hw.l2_gbs);
    h->hw.mma_tflops = env_double("MP_MMA_TFLOPS", h->hw.mma_tflops);
    mp::default_gb300_kernels(h->hw, h->kernels, &h->num_kernels);
    mp::drop_unavailable_kernels(h);
    if (calib_path) {
        load_calibration(h, calib_path);  // "" keeps the analytic model
    } else {
        const std::string shipped = shipped_calibration();
        if (!shipped.empty()) load_calibration(h, shipped.c_str());
    }
    *out = h;
    return MP_OK;
}

mp_status mp_init_host(mp_handle* out, const mp_hw* hw, const mp_kernel_desc* kernels,
                       int32_t num_kernels) {
    if (!out) return MP_ERR_INVALID_ARG;
    *out = nullptr;
    if (!hw || hw->num_pe < 1 || hw->warps_per_wave < 1) return MP_ERR_INVALID_ARG;
    if (num_kernels < 0 || num_kernels > MP_MAX_KERNELS || (num_kernels > 0 && !kernels))
        return MP_ERR_INVALID_ARG;
    for (int32_t k = 0; k < num_kernels; k++) {
        const mp_kernel_desc& d = kernels[k];
        if (d.um < 1 || d.un < 1 || d.uk < 1 || d.warps < 1 || d.fixed_us < 0 || d.per_step_us < 0 ||
            !(d.tail_us >= 0))
            return MP_ERR_INVALID_ARG;
    }
    mp_handle h = new_handle();
    if (!h) return MP_ERR_NO_MEMORY;
    h->hw = *hw;
    if (num_kernels == 0) {
        mp::default_gb300_kernels(h->hw, h->kernels, &h->num_kernels);
    } else {
        std::memcpy(h->kernels, kernels, sizeof(mp_kernel_desc) * (size_t)num_kernels);
        h->num_kernels = num_kernels;
    }
    *out = h;
    return MP_OK;
}

mp_status mp_destroy(mp_handle h) {
    if (!h) return MP_OK;
    mp::device_destroy(h);
    delete h;
    return MP_OK;
}

mp_status mp_plan(mp_handle h, int64_t M, int64_t N, int64_t K, mp_plan_info* out) {
    return mp_plan_batched(h, 1, M, N, K, out);
}

mp_status mp_plan_batched(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K,
                          mp_plan_info* out) {
    if (!h) return MP_ERR_INVALID_ARG;
    if (batch < 0 || M < 0 || N < 0 || K < 0) return MP_ERR_INVALID_ARG;
    if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim || batch >= kMaxDim) return MP_ERR_INVALID_ARG;
    mp_plan_info tmp;
    return mp::plan_shape(h, batch, M, N, K, out ? out : &tmp);
}

mp_status mp_plan_many(mp_handle h, int32_t count, const int64_t* mnk, mp_plan_info* out) {
    if (!h || count < 0 || (count > 0 && !mnk)) return MP_ERR_INVALID_ARG;
    mp_plan_info tmp;
    for (int32_t i = 0; i < count; i++) {
        const int64_t M = mnk[3 * i], N = mnk[3 * i + 1], K = mnk[3 * i + 2];
        if (M < 0 || N < 0 || K < 0 || M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return MP_ERR_INVALID_ARG;
        const mp_status st = mp::plan_shape(h, 1, M, N, K, out ? out + i : &tmp);
        if (st != MP_OK) return st;
    }
    return MP_OK;
}

mp_status mp_evaluate_plan(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K,
                           mp_plan_info* inout) {
    return mp::evaluate_plan(h, batch, M, N, K, inout);
}

mp_status mp_gemm(mp_handle h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                  const void* B, int64_t ldb, const float* C, int64_t ldc, float* D, int64_t ldd,
                  float alpha, float beta, mp_stream stream) {
    mp::GemmArgs a{1, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, D, ldd, 0, alpha, beta, stream};
    return run(h, a);
}

mp_status mp_gemm_ex(mp_handle h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                     int64_t ldb, const float* C, int64_t ldc, void* D, int64_t ldd, float alpha, float beta,
                     int32_t epilogue, mp_stream stream) {
    mp::GemmArgs a{1, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, static_cast<float*>(D), ldd, 0, alpha, beta, stream,
                   epilogue};
    return run(h, a);
}

mp_status mp_gemm_batched(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K,
                          const void* A, int64_t lda, int64_t strideA, const void* B, int64_t ldb,
                          int64_t strideB, const float* C, int64_t ldc, int64_t strideC, float* D,
                          int64_t ldd, int64_t strideD, float alpha, float beta, mp_stream stream) {
    mp::GemmArgs a{batch, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC,
                   D, ldd, strideD, alpha, beta, stream};
    return run(h, a);
}

mp_status mp_enumerate_plans(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K, mp_plan_info* out,
                             int32_t capacity, int32_t* count) {
    if (!h || !count || capacity < 0 || (capacity > 0 && !out)) return MP_ERR_INVALID_ARG;
    if (batch < 1 || M < 1 || N < 1 || K < 0) return MP_ERR_INVALID_ARG;
    if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim || batch >= kMaxDim) return MP_ERR_INVALID_ARG;
    std::vector<mp_plan_info> all;
    mp_status st;
    try {
        st = mp::enumerate_plans(h, batch, M, N, K, &all);
    } catch (...) {
        return MP_ERR_NO_MEMORY;
    }
    if (st != MP_OK) return st;
    *count = (int32_t)std::min<size_t>(all.size(), (size_t)INT32_MAX);
    const size_t n = std::min<size_t>(all.size(), (size_t)capacity);
    if (n) std::memcpy(out, all.data(), sizeof(mp_plan_info) * n);
    return MP_OK;
}

mp_status mp_gemm_with_plan(mp_handle h, const mp_plan_info* plan, int64_t M, int64_t N, int64_t K, const void* A,
                            int64_t lda, const void* B, int64_t ldb, const float* C, int64_t ldc, float* D,
                            int64_t ldd, float alpha, float beta, mp_stream stream) {
    if (!h || !plan) return MP_ERR_INVALID_ARG;
    mp::GemmArgs a{1, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, D, ldd, 0, alpha, beta, stream};
    mp_status st = check_args(a);
    if (st != MP_OK) return st;
    if (M == 0 || N == 0) return MP_OK;
    if (h->host_only) return MP_ERR_UNSUPPORTED;
    mp_plan_info p = *plan;
    st = mp::evaluate_plan(h, 1, M, N, K, &p);  // checks the tiling and refills every derived field
    if (st != MP_OK) return st == MP_ERR_INVALID_ARG ? MP_ERR_PLAN : st;
    return mp::device_run(h, p, a);
}

mp_status mp_set_plan_mode(mp_handle h, int32_t mode) {
    if (!h || (mode != MP_PLAN_MIKPOLY && mode != MP_PLAN_WAVE && mode != MP_PLAN_PIPE)) return MP_ERR_INVALID_ARG;
    h->plan_mode = mode;
    mp::clear_plan_cache(h);
    return MP_OK;
}

mp_status mp_gemm_b2b(mp_handle h, int64_t M, int64_t N0, int64_t N1, int64_t K0, const void* A0, int64_t lda0,
                      const void* W0, int64_t ldw0, const float* C0, int64_t ldc0, const void* W1, int64_t ldw1,
                      const float* C1, int64_t ldc1, float* D1, int64_t ldd1, float alpha0, float beta0,
                      float alpha1, float beta1, int32_t act0, mp_stream stream) {
    if (!h) return MP_ERR_INVALID_ARG;
    const mp::B2BArgs a{M, N0, N1, K0, A0, lda0, W0, ldw0, C0, ldc0, W1, ldw1, C1, ldc1, D1, ldd1,
                        alpha0, beta0, alpha1, beta1, act0, stream};
    mp_status st = check_b2b(a);
    if (st != MP_OK) return st;
    if (M == 0 || N1 == 0) return MP_OK;
    if (h->host_only) return MP_ERR_UNSUPPORTED;
    mp_b2b_plan plan;
    st = plan_b2b_mode(h, M, N0, N1, K0, &plan);
    if (st != MP_OK) return st;
    return plan.mode == MP_B2B_TWO_LAUNCH ? mp::device_run_b2b_two(h, a) : mp::device_run_b2b(h, plan, a);
}

mp_status mp_plan_b2b(mp_handle h, int64_t M, int64_t N0, int64_t N1, int64_t K0, mp_b2b_plan* out) {
    if (!h || !out) return MP_ERR_INVALID_ARG;
    return plan_b2b_mode(h, M, N0, N1, K0, out);
}

mp_status mp_set_b2b_mode(mp_handle h, int32_t mode) {
    if (!h || mode < MP_B2B_AUTO || mode > MP_B2B_TWO_LAUNCH) return MP_ERR_INVALID_ARG;
    h->b2b_mode = mode;
    return MP_OK;
}

mp_status mp_conv2d(mp_handle h, int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R, int64_t S,
                    int64_t pad_h, int64_t pad_w, const void* X, const void* F, const float* Cin, int64_t ldc,
                    float* D, int64_t ldd, float alpha, float beta, mp_stream stream) {
    if (!h) return MP_ERR_INVALID_ARG;
    const mp::ConvArgs a{N, H, W, C, K, R, S, pad_h, pad_w, X, F, Cin, ldc, D, ldd, alpha, beta, stream};
    mp_status st = check_conv(a);
    if (st != MP_OK) return st;
    const int64_t P = H + 2 * pad_h - R + 1, Q = W + 2 * pad_w - S + 1;
    if (N == 0 || K == 0 || P <= 0 || Q <= 0) return MP_OK;
    if (h->host_only) return MP_ERR_UNSUPPORTED;
    mp_conv_plan plan;
    st = mp::plan_conv(h->hw, h->workspace_floats, N, H, W, C, K, R, S, pad_h, pad_w, &plan);
    if (st != MP_OK) return st;
    return mp::device_run_conv(h, plan, a);
}

mp_status mp_plan_conv(mp_handle h, int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R, int64_t S,
                       int64_t pad_h, int64_t pad_w, mp_conv_plan* out) {
    if (!h || !out) return MP_ERR_INVALID_ARG;
    return mp::plan_conv(h->hw, h->workspace_floats, N, H, W, C, K, R, S, pad_h, pad_w, out);
}

}  // extern "C"

namespace {

mp::GemmArgs problem_args(const mp_gemm_problem& q) {
    return mp::GemmArgs{1, q.M, q.N, q.K, q.A, q.lda, 0, q.B, q.ldb, 0, q.C, q.ldc, 0, q.D, q.ldd, 0,
                        q.alpha, q.beta, nullptr};
}

// Each problem by mp_gemm's rules; no output overlaps another problem's
// operands or output.  Fills `live` with the non-empty problems.
mp_status check_group(int32_t count, const mp_gemm_problem* probs, std::vector<mp_gemm_problem>& live) {
    if (count < 0 || count > 4096 || (count > 0 && !probs)) return MP_ERR_INVALID_ARG;
    for (int32_t i = 0; i < count; i++) {
        const mp_status st = check_args(problem_args(probs[i]));
        if (st != MP_OK) return st;
        if (probs[i].M > 0 && probs[i].N > 0) live.push_back(probs[i]);
    }
    const size_t n = live.size();
    for (size_t i = 0; i < n; i++) {
        const mp_gemm_problem& a = live[i];
        const Span d = span_of(a.D, a.M, a.N, a.ldd, 4, 1, 0);
        for (size_t j = 0; j < n; j++) {
            if (j == i) continue;
            const mp_gemm_problem& b = live[j];
            if (overlap(d, span_of(b.D, b.M, b.N, b.ldd, 4, 1, 0))) return MP_ERR_INVALID_ARG;
            if (b.K > 0 && (overlap(d, span_of(b.A, b.M, b.K, b.lda, 2, 1, 0)) ||
                            overlap(d, span_of(b.B, b.K, b.N, b.ldb, 2, 1, 0))))
                return MP_ERR_INVALID_ARG;
            if (b.beta != 0.0f && overlap(d, span_of(b.C, b.M, b.N, b.ldc, 4, 1, 0))) return MP_ERR_INVALID_ARG;
        }
    }
    return MP_OK;
}

}  // namespace

extern "C" {

mp_status mp_gemm_grouped(mp_handle h, int32_t count, const mp_gemm_problem* problems, mp_stream stream) {
    if (!h) return MP_ERR_INVALID_ARG;
    std::vector<mp_gemm_problem> live;
    mp_status st = check_group(count, problems, live);
    if (st != MP_OK) return st;
    if (live.empty()) return MP_OK;
    if (h->host_only) return MP_ERR_UNSUPPORTED;
    mp_grouped_plan plan;
    st = mp::plan_grouped(h->hw, (int32_t)live.size(), live.data(), &plan);
    if (st != MP_OK) return st;
    return mp::device_run_grouped(h, plan, (int32_t)live.size(), live.data(), stream);
}

mp_status mp_plan_grouped(mp_handle h, int32_t count, const mp_gemm_problem* problems, mp_grouped_plan* out) {
    if (!h || !out) return MP_ERR_INVALID_ARG;
    std::vector<mp_gemm_problem> live;
    mp_status st = check_group(count, problems, live);
    if (st != MP_OK) return st;
    return mp::plan_grouped(h->hw, (int32_t)live.size(), live.data(), out);
}

mp_status mp_check(mp_handle h, mp_stream stream) {
    if (!h) return MP_ERR_INVALID_ARG;
    if (h->host_only) return MP_OK;
    return mp::device_check(h, stream);
}

mp_status mp_force_plan(mp_handle h, int32_t kernel, int32_t splits) {
    if (!h) return MP_ERR_INVALID_ARG;
    if (kernel < -1 || kernel >= h->num_kernels || splits < 0) return MP_ERR_INVALID_ARG;
    h->force_kernel = kernel;
    h->force_splits = splits;
    mp::clear_plan_cache(h);
    return MP_OK;
}

mp_status mp_get_hw(mp_handle h, mp_hw* hw, mp_kernel_desc* kernels, int32_t* num_kernels) {
    if (!h) return MP_ERR_INVALID_ARG;
    if (hw) *hw = h->hw;
    if (kernels) std::memcpy(kernels, h->kernels, sizeof(mp_kernel_desc) * (size_t)h->num_kernels);
    if (num_kernels) *num_kernels = h->num_kernels;
    return MP_OK;
}

mp_status mp_set_kernel_model(mp_handle h, int32_t k, double fixed_us, double per_step_us, double tail_us) {
    if (!h || k < 0 || k >= h->num_kernels || !(fixed_us >= 0) || !(per_step_us > 0) || !(tail_us >= 0))
        return MP_ERR_INVALID_ARG;
    h->kernels[k].fixed_us = fixed_us;
    h->kernels[k].per_step_us = per_step_us;
    h->kernels[k].tail_us = tail_us;
    h->calibrated = true;
    mp::clear_plan_cache(h);
    return MP_OK;
}

mp_status mp_load_calibration(mp_handle h, const char* path) {
    if (!h || !path) return MP_ERR_INVALID_ARG;
    return load_calibration(h, path) ? MP_OK : MP_ERR_INVALID_ARG;
}

mp_status mp_set_split_model(mp_handle h, int32_t on_chip, int32_t S, double sync_us, double bytes_factor) {
    if (!h || !set_split_model(h, on_chip, S, sync_us, bytes_factor)) return MP_ERR_INVALID_ARG;
    mp::clear_plan_cache(h);
    return MP_OK;
}

mp_status mp_get_split_model(mp_handle h, int32_t on_chip, int32_t S, double* sync_us, double* bytes_factor) {
    if (!h) return MP_ERR_INVALID_ARG;
    int i;
    if (on_chip == 0 && S == 0)
        i = 0;
    else if (on_chip == 1 && S >= 2 && S <= mp::kClusterSplitMaxS)
        i = S;
    else
        return MP_ERR_INVALID_ARG;
    if (sync_us) *sync_us = h->split_sync_us[i];
    if (bytes_factor) *bytes_factor = h->split_bytes_factor[i];
    return MP_OK;
}

const char* mp_status_string(mp_status s) {
    switch (s) {
        case MP_OK: return "ok";
        case MP_ERR_INVALID_ARG: return "invalid argument";
        case MP_ERR_UNSUPPORTED: return "unsupported";
        case MP_ERR_CUDA: return "CUDA error";
        case MP_ERR_PLAN: return "no valid plan";
        case MP_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case MP_ERR_NO_MEMORY: return "out of memory";
    }
    return "unknown status";
}

}  // extern "C"
