// tb_stitch.cu -- single-pass tile stitch kernels for sm_103a.
//
// What is computed (page "[Proposal] Vectorize tiled VAE blending while
// preserving rounding and CUDA graph replay", "Proposed scope"): the output
// of diffusers' tiled-decode recurrence -- tiles visited in row-major order,
// each cross-faded in place along time (blend_t), height (blend_v) and width
// (blend_h) with its already-blended predecessor on that axis, then cropped
// to row_limit and concatenated -- bit for bit, including the per-product
// rounding to the storage type.
//
// How.  Blends only rewrite the first e(n) slices of a tile, and (with bands
// that do not reach each other) the slices a tile lends to its successor are
// never rewritten by its own band.  So the final value of an output element
// in tile (k, i, j) at local (ct, cy, cx) depends on at most 2^d raw tile
// elements: for each axis a whose band contains the element, its neighbour
// n_a - 1 at local coordinate L_a(n_a - 1) - e_a(n_a) + c_a.  Label the raw
// values by delta in {0,1}^d (delta_a = 1: the neighbour along a).  The
// recurrence's final value of node delta is
//     F(delta) = raw(delta), then for a in (t, y, x) with delta_a = 0 and the
//                element inside axis a's band:
//                F(delta) <- blend(F(delta + e_a), F(delta), c_a)
// evaluated in order of decreasing popcount; the output is F(0).  Each blend
// is rnd(rnd(P * u) + rnd(Q * w)) with P the neighbour, Q the current value,
// (w, u) = ((float)(c/e), (float)(1 - c/e)) from double quotients, fp32
// products and sum, and rnd() round-to-nearest-even into the storage type.
// The explicit _rn intrinsics (and -fmad=false for this file) keep every
// product and sum separately rounded, as the rounding contract requires.
//
// Data movement.  One thread owns one 16-byte chunk (8 x 16-bit or 4 x fp32
// elements) per output row, or one element where the geometry is not
// 16-byte aligned.  Its chunk's column placement -- tile column, band
// membership, neighbour column -- is fixed for every row it visits, so it is
// resolved once per thread.  Rows are spread over a persistent grid;
// everything about a row is uniform across the threads that share it.  Each
// output element is written once with a 128-bit streaming store, each tile
// element is read once with a 128-bit streaming load: the kernel moves the
// algorithmic minimum, all tile bytes plus all output bytes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tb_internal.h"

namespace tb {
namespace {

// ---------------------------------------------------------------------------
// storage traits
// ---------------------------------------------------------------------------

template <int DT>
struct Elt;

template <>
struct Elt<F32> {
    static constexpr int BYTES = 4;
};
template <>
struct Elt<F16> {
    static constexpr int BYTES = 2;
    __device__ __forceinline__ static void unpack(uint32_t v, float& lo, float& hi) {
        __half2 h = *reinterpret_cast<const __half2*>(&v);
        float2 f = __half22float2(h);
        lo = f.x;
        hi = f.y;
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
};
template <>
struct Elt<BF16> {
    static constexpr int BYTES = 2;
    __device__ __forceinline__ static void unpack(uint32_t v, float& lo, float& hi) {
        lo = __uint_as_float(v << 16);
        hi = __uint_as_float(v & 0xffff0000u);
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
};

// A chunk: VEC elements held in 32-bit words (16 bytes when vectorised).
template <int DT, int VEC>
struct Chunk {
    static constexpr int WORDS = (VEC * Elt<DT>::BYTES + 3) / 4;
    uint32_t w[WORDS];
};

template <int DT, int VEC>
__device__ __forceinline__ Chunk<DT, VEC> load_chunk(const void* base, int64_t chunk_index) {
    Chunk<DT, VEC> c;
    if constexpr (VEC * Elt<DT>::BYTES == 16) {
        uint4 v = __ldcs(reinterpret_cast<const uint4*>(base) + chunk_index);
        c.w[0] = v.x;
        c.w[1] = v.y;
        c.w[2] = v.z;
        c.w[3] = v.w;
    } else if constexpr (Elt<DT>::BYTES == 4) {
        c.w[0] = __ldcs(reinterpret_cast<const unsigned int*>(base) + chunk_index);
    } else {
        c.w[0] = __ldcs(reinterpret_cast<const unsigned short*>(base) + chunk_index);
    }
    return c;
}

template <int DT, int VEC>
__device__ __forceinline__ void store_chunk(void* base, int64_t chunk_index, const Chunk<DT, VEC>& c) {
    if constexpr (VEC * Elt<DT>::BYTES == 16) {
        __stcs(reinterpret_cast<uint4*>(base) + chunk_index, make_uint4(c.w[0], c.w[1], c.w[2], c.w[3]));
    } else if constexpr (Elt<DT>::BYTES == 4) {
        __stcs(reinterpret_cast<unsigned int*>(base) + chunk_index, c.w[0]);
    } else {
        __stcs(reinterpret_cast<unsigned short*>(base) + chunk_index, (unsigned short)(c.w[0] & 0xffffu));
    }
}

// blend(P, Q) lane by lane: rnd(rnd(P * u[l]) + rnd(Q * w[l])).
// Coefficients are read through `cw(l)` / `cu(l)`.
template <int DT, int VEC, class CW, class CU>
__device__ __forceinline__ Chunk<DT, VEC> blend(const Chunk<DT, VEC>& P, const Chunk<DT, VEC>& Q, CW cw, CU cu) {
    Chunk<DT, VEC> R;
    if constexpr (Elt<DT>::BYTES == 4) {
#pragma unroll
        for (int q = 0; q < Chunk<DT, VEC>::WORDS; ++q) {
            const float pa = __fmul_rn(__uint_as_float(P.w[q]), cu(q));
            const float qb = __fmul_rn(__uint_as_float(Q.w[q]), cw(q));
            R.w[q] = __float_as_uint(__fadd_rn(pa, qb));
        }
    } else if constexpr (VEC == 1) {
        float a, b, ra, rb, dummy;
        Elt<DT>::unpack(P.w[0], a, dummy);
        Elt<DT>::unpack(Q.w[0], b, dummy);
        Elt<DT>::unpack(Elt<DT>::pack(__fmul_rn(a, cu(0)), 0.f), ra, dummy);
        Elt<DT>::unpack(Elt<DT>::pack(__fmul_rn(b, cw(0)), 0.f), rb, dummy);
        R.w[0] = Elt<DT>::pack(__fadd_rn(ra, rb), 0.f) & 0xffffu;
    } else {
#pragma unroll
        for (int q = 0; q < Chunk<DT, VEC>::WORDS; ++q) {
            float a0, a1, b0, b1;
            Elt<DT>::unpack(P.w[q], a0, a1);
            Elt<DT>::unpack(Q.w[q], b0, b1);
            const uint32_t pa = Elt<DT>::pack(__fmul_rn(a0, cu(2 * q)), __fmul_rn(a1, cu(2 * q + 1)));
            const uint32_t qb = Elt<DT>::pack(__fmul_rn(b0, cw(2 * q)), __fmul_rn(b1, cw(2 * q + 1)));
            float ra0, ra1, rb0, rb1;
            Elt<DT>::unpack(pa, ra0, ra1);
            Elt<DT>::unpack(qb, rb0, rb1);
            R.w[q] = Elt<DT>::pack(__fadd_rn(ra0, rb0), __fadd_rn(ra1, rb1));
        }
    }
    return R;
}

__host__ __device__ constexpr int popc3(int m) { return (m & 1) + ((m >> 1) & 1) + ((m >> 2) & 1); }

// Evaluate the DAG of nodes m subset of NEED (bit 2: time, bit 1: height,
// bit 0: width) in order of decreasing popcount; F[0] ends as the output.
template <int NDIM, int NEED, int DT, int VEC, class XW, class XU>
__device__ __forceinline__ void eval_nodes(Chunk<DT, VEC> (&F)[NDIM == 3 ? 8 : 4], float wt, float ut, float wy,
                                           float uy, XW xw, XU xu) {
    constexpr int NN = NDIM == 3 ? 8 : 4;
#pragma unroll
    for (int pc = 3; pc >= 0; --pc) {
#pragma unroll
        for (int m = NN - 1; m >= 0; --m) {
            if ((m & ~NEED) != 0 || popc3(m) != pc) continue;
            Chunk<DT, VEC> cur = F[m];
            if constexpr (NDIM == 3) {
                if ((NEED & 4) && !(m & 4))
                    cur = blend<DT, VEC>(F[(m | 4) & (NN - 1)], cur, [&](int) { return wt; }, [&](int) { return ut; });
            }
            if ((NEED & 2) && !(m & 2))
                cur = blend<DT, VEC>(F[m | 2], cur, [&](int) { return wy; }, [&](int) { return uy; });
            if ((NEED & 1) && !(m & 1)) cur = blend<DT, VEC>(F[m | 1], cur, xw, xu);
            F[m] = cur;
        }
    }
}

// Index of the tile whose output range [off[n], off[n+1]) holds v.
template <int MAXA>
__device__ __forceinline__ int find_tile(const StitchAxis<MAXA>& a, int v) {
    int lo = 0, hi = a.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.off[mid] <= v)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

template <int NDIM, int DT, int VEC, int KX, int MAXA, int MAXT, int MAXC>
__global__ void __launch_bounds__(512) stitch_kernel(const __grid_constant__ StitchParams<MAXA, MAXT, MAXC> p) {
    constexpr int NN = NDIM == 3 ? 8 : 4;
    using C = Chunk<DT, VEC>;
    extern __shared__ float2 s_coef[];

    // coefficient tables into shared memory (lane-varying width coefficients
    // would serialise on the constant bank)
    const int ncoef = p.ncoef;
    for (int q = threadIdx.x; q < ncoef; q += blockDim.x) s_coef[q] = p.coef[q];
    __syncthreads();

    const auto& AT = p.ax[0];
    const auto& AY = p.ax[1];
    const auto& AX = p.ax[2];
    const int nx = AX.n, ny = AY.n;
    const int xs = threadIdx.x % p.xt;
    const int rs = threadIdx.x / p.xt;
    const uint32_t nseg = (uint32_t)p.nseg, OH = (uint32_t)p.OH, OT = (uint32_t)p.OT;
    const int64_t OW = p.OW;

    // this thread's chunks in the current row segment
    int cur_seg = -1;
    int xj[KX], xcx[KX], xcxn[KX], xcoef[KX], xout[KX];
    bool xband[KX], xvalid[KX];

    for (int64_t vrow = (int64_t)blockIdx.x * p.rp + rs; vrow < p.nvrows; vrow += (int64_t)gridDim.x * p.rp) {
        const uint32_t vr = (uint32_t)vrow;
        const uint32_t seg = vr % nseg;
        const uint32_t row = vr / nseg;
        if ((int)seg != cur_seg) {
            cur_seg = (int)seg;
#pragma unroll
            for (int k = 0; k < KX; ++k) {
                const int x0 = ((int)seg * p.seg_chunks + xs + k * p.xt) * VEC;
                xvalid[k] = x0 < OW;
                const int x = xvalid[k] ? x0 : 0;
                const int j = find_tile(AX, x);
                const int cx = x - AX.off[j];
                xj[k] = j;
                xcx[k] = cx;
                xout[k] = x;
                xband[k] = j > 0 && cx < AX.blend[j];
                xcxn[k] = xband[k] ? AX.ext[j - 1] - AX.blend[j] + cx : 0;
                xcoef[k] = xband[k] ? AX.coef[j] + cx : 0;
            }
        }
        // the row: (plane, t, y)
        const uint32_t y = row % OH;
        const uint32_t r2 = row / OH;
        const uint32_t t = NDIM == 3 ? r2 % OT : 0u;
        const uint32_t plane = NDIM == 3 ? r2 / OT : r2;

        const int i = find_tile(AY, (int)y);
        const int cy = (int)y - AY.off[i];
        const bool by = i > 0 && cy < AY.blend[i];
        const int cyn = by ? AY.ext[i - 1] - AY.blend[i] + cy : 0;
        float wy = 0.f, uy = 0.f;
        if (by) {
            const float2 c = s_coef[AY.coef[i] + cy];
            wy = c.x;
            uy = c.y;
        }
        int kk = 0, ct = 0, ctn = 0;
        bool bt = false;
        float wt = 0.f, ut = 0.f;
        if constexpr (NDIM == 3) {
            kk = find_tile(AT, (int)t);
            ct = (int)t - AT.off[kk];
            bt = kk > 0 && ct < AT.blend[kk];
            ctn = bt ? AT.ext[kk - 1] - AT.blend[kk] + ct : 0;
            if (bt) {
                const float2 c = s_coef[AT.coef[kk] + ct];
                wt = c.x;
                ut = c.y;
            }
        }
        // per (dt, dy) node: tile row index and element offset of the row
        // start inside that tile, in units of the tile's row length
        int64_t rbase[2][2];
        int tbase[2][2];
#pragma unroll
        for (int dt = 0; dt < 2; ++dt) {
#pragma unroll
            for (int dy = 0; dy < 2; ++dy) {
                const bool use = (dt == 0 || bt) && (dy == 0 || by) && (NDIM == 3 || dt == 0);
                const int kq = use ? kk - dt : 0;
                const int iq = use ? i - dy : 0;
                const int64_t Lt = NDIM == 3 ? AT.ext[kq] : 1;
                const int lt = dt ? ctn : ct;
                const int ly = dy ? cyn : cy;
                rbase[dt][dy] = ((int64_t)plane * Lt + lt) * AY.ext[iq] + ly;
                tbase[dt][dy] = (kq * ny + iq) * nx;
            }
        }
        const int64_t obase = (((int64_t)plane * (NDIM == 3 ? OT : 1u) + t) * OH + y) * OW;

        // issue every load of this row before any arithmetic
        C F[KX][NN];
        int need[KX];
#pragma unroll
        for (int k = 0; k < KX; ++k) {
            need[k] = (bt ? 4 : 0) | (by ? 2 : 0) | (xband[k] ? 1 : 0);
            if (!xvalid[k]) need[k] = -1;
#pragma unroll
            for (int m = 0; m < NN; ++m) {
                if (need[k] >= 0 && (m & ~need[k]) == 0) {
                    const int dt = (m >> 2) & 1, dy = (m >> 1) & 1, dx = m & 1;
                    const int jq = xj[k] - dx;
                    const int lx = dx ? xcxn[k] : xcx[k];
                    const int64_t e = rbase[dt][dy] * AX.ext[jq] + lx;
                    F[k][m] = load_chunk<DT, VEC>(p.tiles[tbase[dt][dy] + jq], (int64_t)((uint64_t)e / VEC));
                }
            }
        }
#pragma unroll
        for (int k = 0; k < KX; ++k) {
            if (need[k] < 0) continue;
            const int cb = xcoef[k];
            auto xw = [&](int l) { return s_coef[cb + l].x; };
            auto xu = [&](int l) { return s_coef[cb + l].y; };
            switch (need[k]) {
                case 0: break;
                case 1: eval_nodes<NDIM, 1, DT, VEC>(F[k], wt, ut, wy, uy, xw, xu); break;
                case 2: eval_nodes<NDIM, 2, DT, VEC>(F[k], wt, ut, wy, uy, xw, xu); break;
                case 3: eval_nodes<NDIM, 3, DT, VEC>(F[k], wt, ut, wy, uy, xw, xu); break;
                default:
                    if constexpr (NDIM == 3) {
                        switch (need[k]) {
                            case 4: eval_nodes<NDIM, 4, DT, VEC>(F[k], wt, ut, wy, uy, xw, xu); break;
                            case 5: eval_nodes<NDIM, 5, DT, VEC>(F[k], wt, ut, wy, uy, xw, xu); break;
                            case 6: eval_nodes<NDIM, 6, DT, VEC>(F[k], wt, ut, wy, uy, xw, xu); break;
                            case 7: eval_nodes<NDIM, 7, DT, VEC>(F[k], wt, ut, wy, uy, xw, xu); break;
                        }
                    }
                    break;
            }
            store_chunk<DT, VEC>(p.out, (int64_t)((uint64_t)(obase + xout[k]) / VEC), F[k][0]);
        }
    }
}

template <int MAXA, int MAXT, int MAXC>
using KernelFn = void (*)(const StitchParams<MAXA, MAXT, MAXC>);

template <int NDIM, int DT, int MAXA, int MAXT, int MAXC>
KernelFn<MAXA, MAXT, MAXC> pick_vec(int vec, int kx) {
    constexpr int V = 16 / Elt<DT>::BYTES;
    if (vec == 1) {
        return kx == 2 ? stitch_kernel<NDIM, DT, 1, 2, MAXA, MAXT, MAXC>
                       : stitch_kernel<NDIM, DT, 1, 1, MAXA, MAXT, MAXC>;
    }
    return kx == 2 ? stitch_kernel<NDIM, DT, V, 2, MAXA, MAXT, MAXC> : stitch_kernel<NDIM, DT, V, 1, MAXA, MAXT, MAXC>;
}

template <int MAXA, int MAXT, int MAXC>
KernelFn<MAXA, MAXT, MAXC> pick(const StitchLaunch& l) {
    if (l.ndim == 3) {
        switch (l.dtype) {
            case F32: return pick_vec<3, F32, MAXA, MAXT, MAXC>(l.vec, l.kx);
            case F16: return pick_vec<3, F16, MAXA, MAXT, MAXC>(l.vec, l.kx);
            default: return pick_vec<3, BF16, MAXA, MAXT, MAXC>(l.vec, l.kx);
        }
    }
    switch (l.dtype) {
        case F32: return pick_vec<2, F32, MAXA, MAXT, MAXC>(l.vec, l.kx);
        case F16: return pick_vec<2, F16, MAXA, MAXT, MAXC>(l.vec, l.kx);
        default: return pick_vec<2, BF16, MAXA, MAXT, MAXC>(l.vec, l.kx);
    }
}

template <int MAXA, int MAXT, int MAXC>
cudaError_t launch(const StitchParams<MAXA, MAXT, MAXC>& p, const StitchLaunch& l, cudaStream_t s) {
    auto fn = pick<MAXA, MAXT, MAXC>(l);
    const size_t smem = sizeof(float2) * (size_t)p.ncoef;
    fn<<<l.grid, l.block, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_stitch_small(const StitchParamsSmall& p, const StitchLaunch& l, cudaStream_t s) {
    return launch(p, l, s);
}

cudaError_t launch_stitch_large(const StitchParamsLarge& p, const StitchLaunch& l, cudaStream_t s) {
    return launch(p, l, s);
}

int stitch_kernel_max_ctas_per_sm(const StitchLaunch& l, bool large) {
    int n = 0;
    cudaError_t e;
    if (large) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, pick<LARGE_MAXA, LARGE_MAXT, LARGE_MAXC>(l), l.block,
                                                          sizeof(float2) * LARGE_MAXC);
    } else {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, pick<SMALL_MAXA, SMALL_MAXT, SMALL_MAXC>(l), l.block,
                                                          sizeof(float2) * SMALL_MAXC);
    }
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    return n > 0 ? n : 1;
}

}  // namespace tb
