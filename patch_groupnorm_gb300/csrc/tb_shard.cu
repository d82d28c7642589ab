// tb_shard.cu -- the copy a rank makes before a row-sharded stitch.
//
// Page "Add tiled VAE parallelism & extended model support" (xDiT DistVAE
// PR #14), the halo-exchange commits: when the tile rows of a tiled decode
// are shared out among ranks, each rank needs, before it can blend its first
// tile row, the rows of the tile row above that its band cross-fades with --
// the last e_y rows of every tile of the previous rank's last tile row --
// and the ranks exchange such neighbour rows point to point.  Only raw rows
// travel: blends rewrite the first rows of a tile, never the rows it lends
// to the tile below (bands apart), and the horizontal blend of those rows
// with their left neighbours is recomputed by the receiving rank's stitch.
//
// halo_pack_kernel gathers those rows of every tile of one tile row into one
// dense buffer, so the exchange is a single message per rank boundary.  It
// moves chunks of `VB` bytes (the widest power of two up to 16 dividing every
// row, offset and address).
#include "tb_internal.h"

namespace tb {
namespace {

template <int VB>
struct Vec;
template <>
struct Vec<16> {
    using T = uint4;
};
template <>
struct Vec<8> {
    using T = uint2;
};
template <>
struct Vec<4> {
    using T = uint32_t;
};
template <>
struct Vec<2> {
    using T = uint16_t;
};
template <>
struct Vec<1> {
    using T = uint8_t;
};

// CTA (b, q) copies band rows [b * per_cta, (b + 1) * per_cta) of band q;
// a band row is one of the `e` rows of one (plane, frame), `width` chunks
// long at the same place in the source tile and in the band.  Threads lie
// across a row (bdx of them) and over `HALO_BLOCK / bdx` rows at a time, so
// each thread divides once per row, and issues HALO_INFLIGHT loads before
// its stores.
constexpr int HALO_INFLIGHT = 4;

template <int VB>
__global__ void __launch_bounds__(HALO_BLOCK) halo_pack_kernel(const __grid_constant__ HaloPackParams p) {
    using T = typename Vec<VB>::T;
    const int q = blockIdx.y;
    const uint32_t w = (uint32_t)p.width[q];
    const uint32_t e = (uint32_t)p.e;
    const uint32_t L = (uint32_t)p.rows[q];
    const int64_t nrows = p.n[q] / w;                      // band rows of band q
    const int64_t r0 = (int64_t)blockIdx.x * p.per_cta;
    const int64_t r1 = r0 + p.per_cta < nrows ? r0 + p.per_cta : nrows;
    const uint32_t bdx = w < (uint32_t)HALO_BLOCK ? w : (uint32_t)HALO_BLOCK;
    const uint32_t bdy = HALO_BLOCK / bdx;
    const uint32_t tx = threadIdx.x % bdx, ty = threadIdx.x / bdx;
    if (ty >= bdy) return;
    const T* src = reinterpret_cast<const T*>(p.src[q]);
    T* dst = reinterpret_cast<T*>(p.dst) + p.dst_off[q];
    const int64_t src_bytes = nrows / e * (int64_t)L * w * VB;  // bounds-checked build
    for (int64_t r = r0 + ty; r < r1; r += bdy) {
        const int64_t fp = r / e;                            // (plane, frame)
        const int64_t row = r - fp * e;
        const T* srow = src + ((uint64_t)fp * L + (L - e + row)) * w;
        T* drow = dst + (uint64_t)r * w;
        for (uint32_t x0 = tx; x0 < w; x0 += bdx * HALO_INFLIGHT) {
            T v[HALO_INFLIGHT];
#pragma unroll
            for (int u = 0; u < HALO_INFLIGHT; ++u) {
                const uint32_t x = x0 + u * bdx;
                if (x < w && in_bounds(srow + x, VB, src, src_bytes, p.status)) v[u] = __ldcs(srow + x);
            }
#pragma unroll
            for (int u = 0; u < HALO_INFLIGHT; ++u) {
                const uint32_t x = x0 + u * bdx;
                if (x < w && in_bounds(drow + x, VB, p.dst, p.dst_total * VB, p.status)) __stcs(drow + x, v[u]);
            }
        }
    }
}

}  // namespace

cudaError_t launch_halo_pack(const HaloPackParams& p, int vec_bytes, int64_t ranges, cudaStream_t s) {
    void (*fn)(const HaloPackParams);
    switch (vec_bytes) {
        case 16: fn = halo_pack_kernel<16>; break;
        case 8: fn = halo_pack_kernel<8>; break;
        case 4: fn = halo_pack_kernel<4>; break;
        case 2: fn = halo_pack_kernel<2>; break;
        default: fn = halo_pack_kernel<1>; break;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ranges, (unsigned)p.ntiles, 1);
    cfg.blockDim = dim3(HALO_BLOCK, 1, 1);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace tb
