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
// row, offset and address); CTA (b, q) copies the b-th range of band q.
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

template <int VB>
__global__ void __launch_bounds__(HALO_BLOCK) halo_pack_kernel(const __grid_constant__ HaloPackParams p) {
    using T = typename Vec<VB>::T;
    const int q = blockIdx.y;
    const int64_t n = p.n[q];
    const int64_t c0 = (int64_t)blockIdx.x * p.per_cta;
    const int64_t c1 = c0 + p.per_cta < n ? c0 + p.per_cta : n;
    const uint64_t w = (uint64_t)p.width[q];
    const uint64_t e = (uint64_t)p.e;
    const uint64_t L = (uint64_t)p.rows[q];
    const T* src = reinterpret_cast<const T*>(p.src[q]);
    T* dst = reinterpret_cast<T*>(p.dst) + p.dst_off[q];
    const int64_t src_bytes = n / (int64_t)e * (int64_t)L * VB;  // bounds-checked build
    for (int64_t c = c0 + threadIdx.x; c < c1; c += HALO_BLOCK) {
        const uint64_t r = (uint64_t)c / w;      // (plane, frame, band row), flattened
        const uint64_t x = (uint64_t)c - r * w;
        const uint64_t fp = r / e;               // (plane, frame)
        const uint64_t row = r - fp * e;
        const T* at = src + (fp * L + (L - e + row)) * w + x;
        if (in_bounds(at, VB, src, src_bytes, p.status) &&
            in_bounds(dst + c, VB, p.dst, p.dst_total * VB, p.status))
            dst[c] = __ldcs(at);
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
