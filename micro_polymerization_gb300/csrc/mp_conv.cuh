// Implicit-GEMM 2-D convolution (stride 1, zero padding), NHWC:
//   D[n,p,q,k] = alpha * sum_{r,s,c} X[n, p+r-pad_h, q+s-pad_w, c] * F[r,s,c,k]
//              + beta * Cin[n,p,q,k]
// The MikPoly summary (section 5) runs convolutions as GEMMs over the im2col
// matrix [N*P*Q, R*S*C].  Here that matrix is never built: the TMA producer
// loads each 128 x 64 A tile straight from X.
//
// An output tile is a box of wb x hb x nb output pixels (a rectangle of one
// image, or the same rectangle of several small images), at most 128 of them
// (the UMMA's rows), by bn output channels.  Power-of-two sides with product
// 128 let each epilogue warp store its 32 pixels as one box; sides that
// divide a small image exactly (5 x 5 x 5, 3 x 9 x 4, ...) waste fewer MMA
// rows, and their pixels are stored one by one.  Rows past wb*hb*nb hold
// whatever the stage held before; their accumulator rows are never read.  For filter tap (r, s) and channels
// [c0, c0+64), the A tile is the 4-D box {64 channels, wb, hb, nb} of X at
// (c0, q0+s-pad_w, p0+r-pad_h, n0): in shared memory 128 rows of 64 bf16
// with the 128-byte swizzle, row = pixel (w fastest, then h, then n), the
// layout a GEMM A tile has.  TMA fills coordinates outside X (the padding,
// and the box's overhang past the image) with zeros.  The B tile is rows
// tap*C + c0 .. +63 of F as a [R*S*C] x K matrix; when C is not a multiple
// of 64, rows past the tap's C meet zero A channels, so they add nothing.
// The epilogue stores each warp's 32 pixels as a 4-D box of D, clipped at
// the edges.  Layers with few tiles and long K loops split K: a tile's
// splits run side by side, each writes its raw fp32 partial to a workspace,
// and a second kernel sums the partials in split order (so the result does
// not depend on timing) before alpha, beta*Cin and the store.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace mp {
namespace conv {

constexpr int kThreads = 224;                  // warps 0, 6 TMA, warp 1 MMA + TMEM, warps 2..5 epilogue
constexpr int kMaxStages = 8;
constexpr int kEpiSlabBytes = 2 * 32 * 32 * 4;  // two 32-pixel x 32-channel fp32 slabs per epilogue warp
constexpr int kSmemLimit = 232448;             // dynamic shared memory per CTA (227 KB)

struct alignas(128) Params {
    CUtensorMap tmX;  // X as {C, W, H, N} bf16, box {64, wb, hb, nb}
    CUtensorMap tmF;  // F as {K, R*S*C, 1} bf16, box {64, 64, 1}
    CUtensorMap tmD;  // D as {K, Q, P, N} fp32, box {32, bw, bh, bnn} (bulk stores, when tma_d)
    const float* Cin;
    float* D;
    float* ws;           // split-K partials: [tile][split][128 rows][bn] fp32
    long long ldc, ldd;  // elements from one output pixel to the next in Cin and D
    int N, H, W, C, K, R, S, pad_h, pad_w, P, Q;
    int wb, hb, nb;     // output pixels per tile along Q, P and images
    int box_rows;       // wb * hb * nb <= 128: the A box's rows; the tile's later rows are unused
    int bw, bh, bnn;    // one warp's 32 pixels: the first 32 rows of the tile's order
    int tiles_q, tiles_p, tiles_n, tiles_k;
    int bn;             // output channels per tile (64, 128 or 256)
    int cblocks;        // ceil(C / 64)
    int ksteps;         // R * S * cblocks
    int tiles;          // tiles_n * tiles_p * tiles_q * tiles_k
    int splits;         // K slices per tile (split-K); > 1: partials go to `ws`
    int units;          // tiles * splits
    int num_stages, stage_bytes;
    float alpha, beta;
    int tma_d;          // bulk tensor stores (D 16-byte aligned, ldd % 4 == 0, power-of-two box sides)
    int vec_d;          // D rows allow 16-byte stores
    int vec_c;          // Cin rows allow 16-byte loads
    int* err;           // the handle's status word
    unsigned long long wait_limit_ns;
    int inject_timeout;  // test hook: producer warp 0 withholds its first stage
    // K steps of X and F the first epilogue warp prefetches into L2 for its
    // CTA's first unit before waiting for the previous kernel (0: none).
    int l2_pf;
};

inline int smem_bytes(int num_stages, int stage_bytes) {
    return num_stages * stage_bytes + 4 * kEpiSlabBytes + 1024 + 1024;
}

cudaError_t launch(const cudaLaunchConfig_t& cfg, const Params& p);
// Split-K: sum each tile's partials in split order, then alpha, beta*Cin and
// the store of the tile's pixels (one thread per 4 channels of a tile row).
cudaError_t launch_reduce(cudaStream_t stream, const Params& p);
bool set_smem();

}  // namespace conv
}  // namespace mp
