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

// CTA (b, q) copies chunks [b * per_cta, (b + 1) * per_cta) of band q, in
// the band's own order ((plane, frame), band row, column).  A thread divides
// twice to find its first chunk's (plane and frame, band row, column), then
// steps HALO_BLOCK chunks at a time by additions, and keeps HALO_INFLIGHT
// loads in flight before it stores them.
constexpr int HALO_INFLIGHT = 8;

template <int VB>
__global__ void __launch_bounds__(HALO_BLOCK) halo_pack_kernel(const __grid_constant__ HaloPackParams p) {
    using T = typename Vec<VB>::T;
    const int q = blockIdx.y;
    const int64_t n = p.n[q];
    int64_t c = (int64_t)blockIdx.x * p.per_cta + threadIdx.x;
    const int64_t c1 = (int64_t)blockIdx.x * p.per_cta + p.per_cta < n ? (int64_t)blockIdx.x * p.per_cta + p.per_cta : n;
    if (c >= c1) return;
    const uint32_t w = (uint32_t)p.width[q];
    const uint32_t e = (uint32_t)p.e;
    const uint32_t L = (uint32_t)p.rows[q];
    const uint64_t r = (uint64_t)c / w;            // (plane, frame, band row)
    uint32_t x = (uint32_t)((uint64_t)c - r * w);
    uint64_t fp = r / e;                            // (plane, frame)
    uint32_t brow = (uint32_t)(r - fp * e);
    const uint32_t rstep = HALO_BLOCK / w, xstep = HALO_BLOCK % w;
    const T* src = reinterpret_cast<const T*>(p.src[q]);
    T* dst = reinterpret_cast<T*>(p.dst) + p.dst_off[q];
    const int64_t src_bytes = n / (int64_t)(e * w) * (int64_t)L * w * VB;  // bounds-checked build
    while (c < c1) {
        T v[HALO_INFLIGHT];
        int64_t at[HALO_INFLIGHT];
#pragma unroll
        for (int u = 0; u < HALO_INFLIGHT; ++u) {
            at[u] = -1;
            if (c < c1) {
                const T* s = src + (fp * L + (L - e + brow)) * w + x;
                if (in_bounds(s, VB, src, src_bytes, p.status)) {
                    v[u] = __ldcs(s);
                    at[u] = c;
                }
            }
            c += HALO_BLOCK;
            x += xstep;
            uint32_t dr = rstep;
            if (x >= w) {
                x -= w;
                ++dr;
            }
            brow += dr;
            while (brow >= e) {
                brow -= e;
                ++fp;
            }
        }
#pragma unroll
        for (int u = 0; u < HALO_INFLIGHT; ++u)
            if (at[u] >= 0 && in_bounds(dst + at[u], VB, p.dst, p.dst_total * VB, p.status)) __stcs(dst + at[u], v[u]);
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
