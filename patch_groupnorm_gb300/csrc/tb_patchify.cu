// tb_patchify.cu -- the ragged Patchify split and the patch gather for sm_103a.
//
// What is moved (page "Add tiled VAE parallelism & extended model support",
// xDiT DistVAE PR #14, the commits on Patchify's bands and on
// gather_patches): a tensor viewed as [outer, extent, inner] is cut along
// its middle axis into P bands of whole multiples of the VAE's scale factor,
// the first ranks taking one band more; the gather puts the bands back in
// rank order, reading each from a buffer that may be padded along the axis
// to the longest band (the equal-shape buffers of an all-gather).
//
// How.  Both directions are one batched strided copy: band p is `outer`
// runs of run[p] contiguous chunks, at pitch ppitch[p] in its patch buffer
// and at pitch wpitch, offset woff[p], in the whole tensor.  A chunk is the
// widest power of two <= 16 bytes that divides every run, pitch, offset and
// base pointer, so a chunk never straddles a run and every access is an
// aligned vector access.  Each patch's chunks, counted in patch order, are
// cut into the same number of CTA-sized ranges; CTA b takes range b / P of
// patch b % P, so neighbouring CTAs copy the same outer slices of different
// bands and a DRAM sector shared by two bands is fetched while it is still
// in L2.  A thread keeps eight chunk loads in flight before it stores, and
// walks its chunks 256 at a time with (outer, run) position updates that
// need no division.
#include <cstdint>

#include "tb_internal.h"

namespace tb {
namespace {

template <int V>
struct Chunk;
template <>
struct Chunk<16> {
    using T = uint4;
};
template <>
struct Chunk<8> {
    using T = uint2;
};
template <>
struct Chunk<4> {
    using T = unsigned int;
};
template <>
struct Chunk<2> {
    using T = unsigned short;
};
template <>
struct Chunk<1> {
    using T = unsigned char;
};

constexpr int PF_INFLIGHT = 8;  // chunk loads issued before the first store

template <int V, bool TO_PATCHES>
__global__ void __launch_bounds__(PF_BLOCK) patch_copy_kernel(const __grid_constant__ PatchCopyParams p) {
    using T = typename Chunk<V>::T;
    const int pi = (int)(blockIdx.x % (unsigned)p.P);
    const int64_t range = blockIdx.x / (unsigned)p.P;
    const int64_t n = p.n[pi];
    const int64_t c0 = range * p.per_cta[pi];
    if (c0 >= n) return;
    const int64_t c1 = c0 + p.per_cta[pi] < n ? c0 + p.per_cta[pi] : n;
    const int run = p.run[pi];
    int64_t c = c0 + threadIdx.x;
    int32_t o = (int32_t)(c / run);
    int32_t r = (int32_t)(c - (int64_t)o * run);
    const int32_t so = p.step_o[pi], sr = p.step_r[pi];
    const int64_t ppitch = p.ppitch[pi], wpitch = p.wpitch, woff = p.woff[pi];
    T* const pb = static_cast<T*>(p.patch[pi]);
    T* const wb = static_cast<T*>(p.whole);
    const int64_t pbytes = p.outer * ppitch * V, wbytes = p.outer * wpitch * V;  // bounds-checked build
    // The previous kernel on the stream (launched with programmatic
    // serialisation) may still be writing what this one reads.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    while (c < c1) {
        T v[PF_INFLIGHT];
        T* dst[PF_INFLIGHT];
#pragma unroll
        for (int u = 0; u < PF_INFLIGHT; ++u) {
            dst[u] = nullptr;
            if (c < c1) {
                T* const at_patch = pb + ((int64_t)o * ppitch + r);
                T* const at_whole = wb + ((int64_t)o * wpitch + woff + r);
                if (!in_bounds(at_patch, V, pb, pbytes, p.status) || !in_bounds(at_whole, V, wb, wbytes, p.status)) {
                    // skipped (bounds-checked build only)
                } else if (TO_PATCHES) {
                    v[u] = __ldg(at_whole);
                    dst[u] = at_patch;
                } else {
                    v[u] = __ldg(at_patch);
                    dst[u] = at_whole;
                }
            }
            c += PF_BLOCK;
            o += so;
            r += sr;
            if (r >= run) {
                r -= run;
                ++o;
            }
        }
#pragma unroll
        for (int u = 0; u < PF_INFLIGHT; ++u)
            if (dst[u] != nullptr) __stcs(dst[u], v[u]);
    }
}

template <int V>
void (*pick(bool to_patches))(const PatchCopyParams) {
    return to_patches ? patch_copy_kernel<V, true> : patch_copy_kernel<V, false>;
}

}  // namespace

cudaError_t launch_patch_copy(const PatchCopyParams& p, int vec, bool to_patches, int64_t grid, cudaStream_t s) {
    void (*fn)(const PatchCopyParams);
    switch (vec) {
        case 16: fn = pick<16>(to_patches); break;
        case 8: fn = pick<8>(to_patches); break;
        case 4: fn = pick<4>(to_patches); break;
        case 2: fn = pick<2>(to_patches); break;
        default: fn = pick<1>(to_patches); break;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(PF_BLOCK, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol.wait
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace tb
