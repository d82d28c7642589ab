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
// product and sum separately rounded, as the rounding contract requires
// (see blend() for why the narrow-type sums may use packed adds).
//
// Data movement.  The kept part of every tile splits into at most 2^d
// rectangular boxes by band membership (interior, width band, height band,
// corner; times the time band in 3D).  Inside a box every element needs the
// same set of source tiles, so one CTA takes one piece of one box (a run of
// rows of the box's frame-major (frame, row) space, for one (batch, channel)
// plane) and runs a path compiled for exactly that set: no per-element band
// tests and no divergence.  Pieces of heavier boxes are shorter, and every
// tile's heaviest pieces are dispatched first.  Threads are laid out 2D over
// the box: a thread keeps its columns -- and so its width coefficients -- for
// every row it visits, and each row costs one multiply-add per source
// address.  On the 16-byte path each thread streams the source chunks of its
// coming rows into its own ring of shared-memory slots with cp.async (no
// registers held by loads in flight) and reads each node's value right before
// its blend; stores are 128-bit streaming stores.  Each output element is
// written once and each tile element read once: the kernel moves the
// algorithmic minimum, all tile bytes plus all output bytes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tb_internal.h"

// Rows whose loads are issued together on the element path, by box kind
// (copy / one band / two bands / three).
#ifndef TB_STITCH_UR_COPY
#define TB_STITCH_UR_COPY 4
#endif
#ifndef TB_STITCH_UR_ONE
#define TB_STITCH_UR_ONE 2
#endif
#ifndef TB_STITCH_UR_TWO
#define TB_STITCH_UR_TWO 1
#endif
#ifndef TB_STITCH_UR_THREE
#define TB_STITCH_UR_THREE 1
#endif
// Programmatic dependent launch: the kernel's parameter-only prologue may
// overlap the previous kernel in the stream; it waits for that kernel before
// its first global-memory access.
#ifndef TB_STITCH_PDL
#define TB_STITCH_PDL 1
#endif
#ifndef TB_STITCH_MIN_CTAS_2D
#define TB_STITCH_MIN_CTAS_2D 4
#endif
#ifndef TB_STITCH_MIN_CTAS_3D
#define TB_STITCH_MIN_CTAS_3D 3
#endif

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
    // a + b rounded once to fp16, lane by lane
    __device__ __forceinline__ static uint32_t add2(uint32_t a, uint32_t b) {
        uint32_t r;
        asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
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
    // a + b rounded once to bf16, lane by lane
    __device__ __forceinline__ static uint32_t add2(uint32_t a, uint32_t b) {
        uint32_t r;
        asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
        return r;
    }
};

// A chunk: VEC elements held in 32-bit words (16 bytes when vectorised).
template <int DT, int VEC>
struct Chunk {
    static constexpr int WORDS = (VEC * Elt<DT>::BYTES + 3) / 4;
    uint32_t w[WORDS];
};

// Chunk at element offset `e` of `base` (16-byte aligned when VEC * size is 16).
template <int DT, int VEC>
__device__ __forceinline__ Chunk<DT, VEC> load_chunk(const void* base, int64_t e) {
    Chunk<DT, VEC> c;
    const char* p = reinterpret_cast<const char*>(base) + e * Elt<DT>::BYTES;
    if constexpr (VEC * Elt<DT>::BYTES == 16) {
        uint4 v = __ldcs(reinterpret_cast<const uint4*>(p));
        c.w[0] = v.x;
        c.w[1] = v.y;
        c.w[2] = v.z;
        c.w[3] = v.w;
    } else if constexpr (Elt<DT>::BYTES == 4) {
        c.w[0] = __ldcs(reinterpret_cast<const unsigned int*>(p));
    } else {
        c.w[0] = __ldcs(reinterpret_cast<const unsigned short*>(p));
    }
    return c;
}

template <int DT, int VEC>
__device__ __forceinline__ void store_chunk(void* base, int64_t e, const Chunk<DT, VEC>& c) {
    char* p = reinterpret_cast<char*>(base) + e * Elt<DT>::BYTES;
    if constexpr (VEC * Elt<DT>::BYTES == 16) {
        __stcs(reinterpret_cast<uint4*>(p), make_uint4(c.w[0], c.w[1], c.w[2], c.w[3]));
    } else if constexpr (Elt<DT>::BYTES == 4) {
        __stcs(reinterpret_cast<unsigned int*>(p), c.w[0]);
    } else {
        __stcs(reinterpret_cast<unsigned short*>(p), (unsigned short)(c.w[0] & 0xffffu));
    }
}

// Two IEEE fp32 products, round-to-nearest, in one packed instruction
// (per lane identical to __fmul_rn).
__device__ __forceinline__ void mul2_rn(float a0, float a1, float b0, float b1, float& r0, float& r1) {
    asm("{\n\t.reg .b64 x, y, z;\n\t"
        "mov.b64 x, {%2, %3};\n\t"
        "mov.b64 y, {%4, %5};\n\t"
        "mul.rn.f32x2 z, x, y;\n\t"
        "mov.b64 {%0, %1}, z;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// blend(P, Q) lane by lane: rnd(rnd(P * u[l]) + rnd(Q * w[l])).
// Coefficients are read through `cw(l)` / `cu(l)`.
//
// For fp16 / bf16 the two rounded products are added with one packed
// add.rn.{f16,bf16}x2.  That equals the contract's fp32 add followed by
// rounding: the fp32 sum of two fp16 (bf16) values is exact unless their
// exponents differ by more than 13 (16); then the smaller one lies far below
// half an ulp of the larger, and both routes return the larger.
template <int DT, int VEC, class CW, class CU>
__device__ __forceinline__ Chunk<DT, VEC> blend(const Chunk<DT, VEC>& P, const Chunk<DT, VEC>& Q, CW cw, CU cu) {
    Chunk<DT, VEC> R;
    if constexpr (Elt<DT>::BYTES == 4) {
        // fp32: scalar products and sum (a packed product feeding a packed
        // add could be fused into one rounding)
#pragma unroll
        for (int q = 0; q < Chunk<DT, VEC>::WORDS; ++q) {
            const float pa = __fmul_rn(__uint_as_float(P.w[q]), cu(q));
            const float qb = __fmul_rn(__uint_as_float(Q.w[q]), cw(q));
            R.w[q] = __float_as_uint(__fadd_rn(pa, qb));
        }
    } else if constexpr (VEC == 1) {
        float a, b, dummy;
        Elt<DT>::unpack(P.w[0], a, dummy);
        Elt<DT>::unpack(Q.w[0], b, dummy);
        const uint32_t pa = Elt<DT>::pack(__fmul_rn(a, cu(0)), 0.f);
        const uint32_t qb = Elt<DT>::pack(__fmul_rn(b, cw(0)), 0.f);
        R.w[0] = Elt<DT>::add2(pa, qb) & 0xffffu;
    } else {
#pragma unroll
        for (int q = 0; q < Chunk<DT, VEC>::WORDS; ++q) {
            float a0, a1, b0, b1, pa0, pa1, qb0, qb1;
            Elt<DT>::unpack(P.w[q], a0, a1);
            Elt<DT>::unpack(Q.w[q], b0, b1);
            mul2_rn(a0, a1, cu(2 * q), cu(2 * q + 1), pa0, pa1);
            mul2_rn(b0, b1, cw(2 * q), cw(2 * q + 1), qb0, qb1);
            R.w[q] = Elt<DT>::add2(Elt<DT>::pack(pa0, pa1), Elt<DT>::pack(qb0, qb1));
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

// Per-CTA description of its box piece.  A box is `nt` frames x `nyb` rows x
// `width` chunks of the tile's kept part, starting at frame t0, row y0,
// column x0 (tile-local); a piece is the rows [rbeg, rend) of the box in
// frame-major order (row r is frame t0 + r / nyb, row y0 + r % nyb).
struct Piece {
    int64_t plane;       // (batch, channel) plane
    int k, i, j;         // tile
    int need;            // box bits: 4 time band, 2 height band, 1 width band
    int t0, y0, nyb;     // box origin and rows per frame
    int rbeg, rend;      // flattened rows of this piece
    int x0, width;       // first column (elements) and width (chunks)
    int bdx, bdy, cpt;   // thread layout
};

// Source node m of the box: its tile, and the byte address of the box
// origin (frame t0, row y0) at column cx.
template <int NDIM, int DT, int MAXA, int MAXT, int MAXC>
__device__ __forceinline__ const char* node_origin(const StitchParams<MAXA, MAXT, MAXC>& p, const Piece& pc, int m,
                                                   int cx) {
    const auto& AT = p.ax[0];
    const auto& AY = p.ax[1];
    const auto& AX = p.ax[2];
    const int dt = (m >> 2) & 1, dy = (m >> 1) & 1, dx = m & 1;
    const int kq = pc.k - dt, iq = pc.i - dy, jq = pc.j - dx;
    const int64_t Lt = NDIM == 3 ? AT.ext[kq] : 1;
    const int64_t Ly = AY.ext[iq];
    const int64_t Lx = AX.ext[jq];
    const int lt = NDIM == 3 ? (dt ? AT.ext[pc.k - 1] - AT.blend[pc.k] + pc.t0 : pc.t0) : 0;
    const int ly = (dy ? AY.ext[pc.i - 1] - AY.blend[pc.i] : 0) + pc.y0;
    const int lx = dx ? AX.ext[pc.j - 1] - AX.blend[pc.j] + cx : cx;
    return reinterpret_cast<const char*>(p.tiles[(kq * AY.n + iq) * AX.n + jq]) +
           (((pc.plane * Lt + lt) * Ly + ly) * Lx + lx) * Elt<DT>::BYTES;
}

// The tile node m of the box reads, as a byte range, for the bounds-checked
// build (empty otherwise); the node's tile indices are checked too.
struct Span {
#if TB_DEBUG_BOUNDS
    const char* base;
    int64_t size;
#endif
};

template <int NDIM, int DT, int MAXA, int MAXT, int MAXC>
__device__ __forceinline__ Span node_span(const StitchParams<MAXA, MAXT, MAXC>& p, const Piece& pc, int m) {
    Span sp;
#if TB_DEBUG_BOUNDS
    const auto& AT = p.ax[0];
    const auto& AY = p.ax[1];
    const auto& AX = p.ax[2];
    const int kq = pc.k - ((m >> 2) & 1), iq = pc.i - ((m >> 1) & 1), jq = pc.j - (m & 1);
    const bool ok = kq >= 0 && kq < (NDIM == 3 ? AT.n : 1) && iq >= 0 && iq < AY.n && jq >= 0 && jq < AX.n;
    if (!index_ok(ok, p.status)) {
        sp.base = nullptr;
        sp.size = 0;
        return sp;
    }
    sp.base = reinterpret_cast<const char*>(p.tiles[(kq * AY.n + iq) * AX.n + jq]);
    sp.size = p.planes * (NDIM == 3 ? AT.ext[kq] : 1) * (int64_t)AY.ext[iq] * AX.ext[jq] * Elt<DT>::BYTES;
#else
    (void)p, (void)pc, (void)m;
#endif
    return sp;
}

template <int DT, int MAXA, int MAXT, int MAXC>
__device__ __forceinline__ Span out_span(const StitchParams<MAXA, MAXT, MAXC>& p) {
    Span sp;
#if TB_DEBUG_BOUNDS
    sp.base = reinterpret_cast<const char*>(p.out);
    sp.size = p.planes * p.OT * (int64_t)p.OH * p.OW * Elt<DT>::BYTES;
#else
    (void)p;
#endif
    return sp;
}

__device__ __forceinline__ bool span_ok(const Span& sp, const void* a, int64_t bytes, uint32_t* status) {
#if TB_DEBUG_BOUNDS
    return in_bounds(a, bytes, sp.base, sp.size, status);
#else
    (void)sp, (void)a, (void)bytes, (void)status;
    return true;
#endif
}

// Byte pitches of one frame and one row in the source tiles: row pitch by
// width-neighbour bit dx, frame pitch by (dy, dx).
struct Pitches {
    int32_t row[2];
    int32_t frame[2][2];
    int32_t orow, oframe;  // output
};

template <int DT, int MAXA, int MAXT, int MAXC>
__device__ __forceinline__ Pitches make_pitches(const StitchParams<MAXA, MAXT, MAXC>& p, const Piece& pc) {
    const auto& AY = p.ax[1];
    const auto& AX = p.ax[2];
    Pitches q;
    for (int dx = 0; dx < 2; ++dx) {
        const int jq = pc.j - dx >= 0 ? pc.j - dx : 0;
        q.row[dx] = AX.ext[jq] * Elt<DT>::BYTES;
        for (int dy = 0; dy < 2; ++dy) {
            const int iq = pc.i - dy >= 0 ? pc.i - dy : 0;
            q.frame[dy][dx] = AY.ext[iq] * AX.ext[jq] * Elt<DT>::BYTES;
        }
    }
    q.orow = p.OW * Elt<DT>::BYTES;
    q.oframe = p.OH * p.OW * Elt<DT>::BYTES;
    return q;
}

template <int NDIM, int DT, int MAXA, int MAXT, int MAXC>
__device__ __forceinline__ char* out_origin(const StitchParams<MAXA, MAXT, MAXC>& p, const Piece& pc, int cx) {
    const auto& AT = p.ax[0];
    const auto& AY = p.ax[1];
    const auto& AX = p.ax[2];
    const int64_t ot = NDIM == 3 ? AT.off[pc.k] + pc.t0 : 0;
    return reinterpret_cast<char*>(p.out) +
           (((pc.plane * p.OT + ot) * p.OH + AY.off[pc.i] + pc.y0) * (int64_t)p.OW + AX.off[pc.j] + cx) *
               Elt<DT>::BYTES;
}

// A thread's position in the box: frame and row relative to the box origin
// (a 2D box has one frame).
template <int NDIM>
struct RowPos {
    int ft, fy;
    __device__ __forceinline__ void set(int r, int nyb) {
        if constexpr (NDIM == 3) {
            ft = r / nyb;
            fy = r - ft * nyb;
        } else {
            ft = 0;
            fy = r;
        }
    }
    __device__ __forceinline__ void advance(int by, int nyb) {
        fy += by;
        if constexpr (NDIM == 3) {
            while (fy >= nyb) {
                fy -= nyb;
                ++ft;
            }
        }
    }
    // byte offset of this position for frame / row pitches
    __device__ __forceinline__ int64_t off(int32_t frame_pitch, int32_t row_pitch) const {
        if constexpr (NDIM == 3) return (int64_t)ft * frame_pitch + (int64_t)fy * row_pitch;
        return (int64_t)fy * row_pitch;
    }
};

// One box, compiled for its set of source tiles NEED (element path).  Rows
// are processed UR at a time: all their loads first, then the arithmetic.
template <int NDIM, int NEED, int UR, int DT, int VEC, int MAXA, int MAXT, int MAXC>
__device__ __forceinline__ void run_box(const StitchParams<MAXA, MAXT, MAXC>& p, const Piece& pc,
                                        const float* s_xw, const float* s_xu, const float* s_yw, const float* s_yu,
                                        const float* s_tw, const float* s_tu) {
    constexpr int NN = NDIM == 3 ? 8 : 4;
    using C = Chunk<DT, VEC>;
    const int tx = threadIdx.x % pc.bdx;
    const int ty = threadIdx.x / pc.bdx;
    if (ty >= pc.bdy) return;
    const Pitches pt = make_pitches<DT>(p, pc);
    for (int q = 0; q < pc.cpt; ++q) {
        const int c = tx + q * pc.bdx;
        if (c >= pc.width) break;
        const int cx = pc.x0 + c * VEC;
        float xw[VEC], xu[VEC];
        if constexpr ((NEED & 1) != 0) {
#pragma unroll
            for (int l = 0; l < VEC; ++l) {
                xw[l] = s_xw[cx + l];
                xu[l] = s_xu[cx + l];
            }
        }
        const char* org[NN];
        Span span[NN];
#pragma unroll
        for (int m = 0; m < NN; ++m)
            if ((m & ~NEED) == 0) {
                org[m] = node_origin<NDIM, DT>(p, pc, m, cx);
                span[m] = node_span<NDIM, DT>(p, pc, m);
            }
        char* oorg = out_origin<NDIM, DT>(p, pc, cx);
        const Span ospan = out_span<DT>(p);
        for (int r = pc.rbeg + ty; r < pc.rend; r += UR * pc.bdy) {
            C F[UR][NN];
            RowPos<NDIM> pos[UR];
#pragma unroll
            for (int u = 0; u < UR; ++u) {
                const int ru = r + u * pc.bdy;
                pos[u].set(ru, pc.nyb);
                if (ru < pc.rend) {
#pragma unroll
                    for (int m = 0; m < NN; ++m) {
                        if ((m & ~NEED) != 0) continue;
                        const int dy = (m >> 1) & 1, dx = m & 1;
                        const char* at = org[m] + pos[u].off(pt.frame[dy][dx], pt.row[dx]);
                        if (span_ok(span[m], at, VEC * Elt<DT>::BYTES, p.status)) F[u][m] = load_chunk<DT, VEC>(at, 0);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < UR; ++u) {
                const int ru = r + u * pc.bdy;
                if (ru < pc.rend) {
                    if constexpr (NEED != 0) {
                        float wy = 0.f, uy = 0.f, wt = 0.f, ut = 0.f;
                        if constexpr ((NEED & 2) != 0) {
                            wy = s_yw[pc.y0 + pos[u].fy];
                            uy = s_yu[pc.y0 + pos[u].fy];
                        }
                        if constexpr ((NEED & 4) != 0) {
                            wt = s_tw[pc.t0 + pos[u].ft];
                            ut = s_tu[pc.t0 + pos[u].ft];
                        }
                        eval_nodes<NDIM, NEED, DT, VEC>(F[u], wt, ut, wy, uy, [&](int l) { return xw[l]; },
                                                        [&](int l) { return xu[l]; });
                    }
                    char* const ot = oorg + pos[u].off(pt.oframe, pt.orow);
                    if (span_ok(ospan, ot, VEC * Elt<DT>::BYTES, p.status)) store_chunk<DT, VEC>(ot, 0, F[u][0]);
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// 16-byte path: a per-thread cp.async pipeline through shared memory
// ---------------------------------------------------------------------------


__host__ __device__ constexpr int nodes_of(int need) { return 1 << popc3(need); }
__host__ __device__ constexpr int stages_of(int need) {
    return STITCH_SLOTS / nodes_of(need) >= 2 ? STITCH_SLOTS / nodes_of(need) : 1;
}
// Position of node m among the nodes of NEED (masks that are subsets of NEED,
// in increasing order).
__host__ __device__ constexpr int node_rank(int need, int m) {
    int r = 0;
    for (int x = 0; x < m; ++x)
        if ((x & ~need) == 0) ++r;
    return r;
}

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* gptr) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(saddr), "l"(gptr) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

template <int DT, int VEC>
__device__ __forceinline__ Chunk<DT, VEC> lds_chunk(uint32_t saddr) {
    Chunk<DT, VEC> c;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(c.w[0]), "=r"(c.w[1]), "=r"(c.w[2]), "=r"(c.w[3])
                 : "r"(saddr));
    return c;
}

// Final value of node m (and, recursively, of the nodes it blends with) for
// the row held in `stage`: the raw value comes from the thread's staging
// slot right before it is used, which keeps the set of live values small.
template <int NDIM, int NEED, int M, int DT, int VEC>
struct NodeEval {
    template <class Ctx>
    __device__ __forceinline__ static void run(Ctx& ctx, Chunk<DT, VEC> (&F)[NDIM == 3 ? 8 : 4]) {
        Chunk<DT, VEC> cur = lds_chunk<DT, VEC>(ctx.slot(node_rank(NEED, M)));
        if constexpr (NDIM == 3 && (NEED & 4) && !(M & 4))
            cur = blend<DT, VEC>(F[M | 4], cur, [&](int) { return ctx.wt; }, [&](int) { return ctx.ut; });
        if constexpr ((NEED & 2) && !(M & 2))
            cur = blend<DT, VEC>(F[M | 2], cur, [&](int) { return ctx.wy; }, [&](int) { return ctx.uy; });
        if constexpr ((NEED & 1) && !(M & 1))
            cur = blend<DT, VEC>(F[M | 1], cur, [&](int l) { return ctx.xw[l]; }, [&](int l) { return ctx.xu[l]; });
        F[M] = cur;
    }
};

template <int NDIM, int NEED, int PC, int M, int DT, int VEC>
struct PassEval {  // nodes of popcount PC, from mask M downwards
    template <class Ctx>
    __device__ __forceinline__ static void run(Ctx& ctx, Chunk<DT, VEC> (&F)[NDIM == 3 ? 8 : 4]) {
        if constexpr (M >= 0) {
            if constexpr ((M & ~NEED) == 0 && popc3(M) == PC) NodeEval<NDIM, NEED, M, DT, VEC>::run(ctx, F);
            PassEval<NDIM, NEED, PC, M - 1, DT, VEC>::run(ctx, F);
        }
    }
};

template <int NDIM, int NEED, int PC, int DT, int VEC>
struct DagEval {  // popcount PC down to 0
    template <class Ctx>
    __device__ __forceinline__ static void run(Ctx& ctx, Chunk<DT, VEC> (&F)[NDIM == 3 ? 8 : 4]) {
        if constexpr (PC >= 0) {
            PassEval<NDIM, NEED, PC, (NDIM == 3 ? 7 : 3), DT, VEC>::run(ctx, F);
            DagEval<NDIM, NEED, PC - 1, DT, VEC>::run(ctx, F);
        }
    }
};

template <int VEC>
struct RowCtx {
    uint32_t base;      // this thread's slot 0 of the current stage
    uint32_t stride;    // bytes between a thread's consecutive slots
    float wt, ut, wy, uy;
    float xw[VEC], xu[VEC];
    __device__ __forceinline__ uint32_t slot(int rank) const { return base + (uint32_t)rank * stride; }
};

template <int NDIM, int NEED, int DT, int VEC, int MAXA, int MAXT, int MAXC>
__device__ __forceinline__ void run_box_pipe(const StitchParams<MAXA, MAXT, MAXC>& p, const Piece& pc,
                                             const float* s_xw, const float* s_xu, const float* s_yw,
                                             const float* s_yu, const float* s_tw, const float* s_tu,
                                             uint32_t s_slots) {
    constexpr int NN = NDIM == 3 ? 8 : 4;
    constexpr int NU = nodes_of(NEED);
    constexpr int S = stages_of(NEED);
    using C = Chunk<DT, VEC>;
    const int tx = threadIdx.x % pc.bdx;
    const int ty = threadIdx.x / pc.bdx;
    if (ty >= pc.bdy) return;
    // slot (stage st, node rank n) of this thread: [st][n][thread] x 16 bytes,
    // so a warp's 16-byte accesses to one slot are contiguous
    const uint32_t slot_stride = (uint32_t)STITCH_BLOCK * 16u;
    const uint32_t my_slot0 = s_slots + (uint32_t)threadIdx.x * 16u;
    const Pitches pt = make_pitches<DT>(p, pc);
    RowCtx<VEC> ctx;
    ctx.stride = slot_stride;
    for (int q = 0; q < pc.cpt; ++q) {
        const int c = tx + q * pc.bdx;
        if (c >= pc.width) break;
        const int cx = pc.x0 + c * VEC;
        if constexpr ((NEED & 1) != 0) {
#pragma unroll
            for (int l = 0; l < VEC; ++l) {
                ctx.xw[l] = s_xw[cx + l];
                ctx.xu[l] = s_xu[cx + l];
            }
        }
        const char* org[NU];
        Span span[NU];
#pragma unroll
        for (int m = 0; m < NN; ++m)
            if ((m & ~NEED) == 0) {
                org[node_rank(NEED, m)] = node_origin<NDIM, DT>(p, pc, m, cx);
                span[node_rank(NEED, m)] = node_span<NDIM, DT>(p, pc, m);
            }
        char* oorg = out_origin<NDIM, DT>(p, pc, cx);
        const Span ospan = out_span<DT>(p);

        const int r0 = pc.rbeg + ty;
        const int nrows = r0 < pc.rend ? (pc.rend - r0 + pc.bdy - 1) / pc.bdy : 0;
        RowPos<NDIM> ipos, cpos;  // the row being fetched, the row being computed
        ipos.set(r0, pc.nyb);
        cpos = ipos;
        auto issue = [&](int m) {  // the fetch row into stage m % S
            const uint32_t st = my_slot0 + (uint32_t)((m % S) * NU) * slot_stride;
#pragma unroll
            for (int mm = 0; mm < NN; ++mm) {
                if ((mm & ~NEED) != 0) continue;
                const int dy = (mm >> 1) & 1, dx = mm & 1;
                const int n = node_rank(NEED, mm);
                const char* at = org[n] + ipos.off(pt.frame[dy][dx], pt.row[dx]);
                if (span_ok(span[n], at, 16, p.status)) cp_async16(st + (uint32_t)n * slot_stride, at);
            }
            ipos.advance(pc.bdy, pc.nyb);
        };
#pragma unroll
        for (int m = 0; m < S - 1; ++m) {
            if (m < nrows) issue(m);
            cp_async_commit();
        }
        for (int m = 0; m < nrows; ++m) {
            if (m + S - 1 < nrows) issue(m + S - 1);
            cp_async_commit();
            cp_async_wait<S - 1>();
            ctx.base = my_slot0 + (uint32_t)((m % S) * NU) * slot_stride;
            if constexpr ((NEED & 2) != 0) {
                ctx.wy = s_yw[pc.y0 + cpos.fy];
                ctx.uy = s_yu[pc.y0 + cpos.fy];
            }
            if constexpr ((NEED & 4) != 0) {
                ctx.wt = s_tw[pc.t0 + cpos.ft];
                ctx.ut = s_tu[pc.t0 + cpos.ft];
            }
            C F[NN];
            DagEval<NDIM, NEED, 3, DT, VEC>::run(ctx, F);
            char* const ot = oorg + cpos.off(pt.oframe, pt.orow);
            if (span_ok(ospan, ot, 16, p.status)) store_chunk<DT, VEC>(ot, 0, F[0]);
            cpos.advance(pc.bdy, pc.nyb);
        }
        cp_async_wait<0>();
    }
}

template <int NDIM, int DT, int VEC, int MAXA, int MAXT, int MAXC>
__global__ void __launch_bounds__(STITCH_BLOCK, (NDIM == 3 ? TB_STITCH_MIN_CTAS_3D : TB_STITCH_MIN_CTAS_2D))
    stitch_kernel(const __grid_constant__ StitchParams<MAXA, MAXT, MAXC> p) {
    pdl_trigger_dependents();
    extern __shared__ __align__(16) unsigned char s_dyn[];
    const auto& AT = p.ax[0];
    const auto& AY = p.ax[1];
    const auto& AX = p.ax[2];

    // which tile, which box, which rows.  Pieces are ranked within their
    // tile, heaviest first, and the blocks run rank by rank, so the GPU
    // dispatches every tile's longest pieces before any short one.  With
    // the one-dimensional grid (p.nrank > 0) only pieces that exist get a
    // block: rank r holds, plane by plane, the tiles of tile_order that have
    // more than r pieces; otherwise blockIdx.x runs over (plane, tile) with
    // the tile fastest and blockIdx.y over the ranks.
    Piece pc;
    const int ntiles = AX.n * AY.n * (NDIM == 3 ? AT.n : 1);
    int tile, piece;
    if (p.nrank > 0) {
        const int b = (int)blockIdx.x;
        int lo = 0, hi = p.nrank;  // rank_start[lo] <= b < rank_start[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.rank_start[mid] <= b) lo = mid;
            else hi = mid;
        }
        const unsigned idx = (unsigned)(b - p.rank_start[lo]);
        const unsigned per_plane = (unsigned)((p.rank_start[lo + 1] - p.rank_start[lo]) / p.planes);
        const unsigned q = idx / per_plane;
        pc.plane = (int64_t)q;
        tile = p.tile_order[idx - q * per_plane];
        piece = lo;
        if (!index_ok(tile >= 0 && tile < ntiles && pc.plane < p.planes, p.status)) return;
    } else {
        tile = (int)(blockIdx.x % (unsigned)ntiles);
        pc.plane = (int64_t)(blockIdx.x / (unsigned)ntiles);
        piece = (int)blockIdx.y;
    }
    pc.j = tile % AX.n;
    pc.i = (tile / AX.n) % AY.n;
    pc.k = NDIM == 3 ? tile / (AX.n * AY.n) : 0;
    const int Kt = NDIM == 3 ? AT.off[pc.k + 1] - AT.off[pc.k] : 1;
    const int Ky = AY.off[pc.i + 1] - AY.off[pc.i];
    const int Kx = AX.off[pc.j + 1] - AX.off[pc.j];
    const int ebt = (NDIM == 3 && pc.k > 0) ? min(AT.blend[pc.k], Kt) : 0;
    const int eby = pc.i > 0 ? min(AY.blend[pc.i], Ky) : 0;
    const int ebx = pc.j > 0 ? min(AX.blend[pc.j], Kx) : 0;
    pc.need = -1;
    constexpr int NB = NDIM == 3 ? 8 : 4;
    for (int b = NB - 1; b >= 0; --b) {  // same order as tile_pieces()
        const BoxShape s = box_shape(b, Kt, Ky, Kx, ebt, eby, ebx, VEC);
        if (s.nt <= 0 || s.ny <= 0 || s.width <= 0) continue;
        const int R = box_piece_rows(b, s.width, p.rows_per_thread);
        const int np = (s.nt * s.ny + R - 1) / R;
        if (piece < np) {
            pc.need = b;
            pc.t0 = s.t0;
            pc.y0 = s.y0;
            pc.nyb = s.ny;
            pc.rbeg = piece * R;
            pc.rend = min(s.nt * s.ny, pc.rbeg + R);
            pc.x0 = s.x0;
            pc.width = s.width;
            box_layout(s.width, pc.bdx, pc.bdy, pc.cpt);
            break;
        }
        piece -= np;
    }
    if (pc.need < 0) return;  // this tile has fewer pieces than the grid row

    // shared memory: the vector path's staging slots, then band coefficients
    unsigned char* s_stage = s_dyn;
    float* s_coef = reinterpret_cast<float*>(s_dyn + (VEC * Elt<DT>::BYTES == 16 ? STITCH_SLOTS * STITCH_BLOCK * 16 : 0));
    float* s_xw = s_coef;
    float* s_xu = s_xw + ebx;
    float* s_yw = s_xu + ebx;
    float* s_yu = s_yw + eby;
    float* s_tw = s_yu + eby;
    float* s_tu = s_tw + ebt;
    if (pc.need & 1)
        for (int c = threadIdx.x; c < ebx; c += blockDim.x) {
            const float2 v = p.coef[AX.coef[pc.j] + c];
            s_xw[c] = v.x;
            s_xu[c] = v.y;
        }
    if (pc.need & 2)
        for (int c = threadIdx.x; c < eby; c += blockDim.x) {
            const float2 v = p.coef[AY.coef[pc.i] + c];
            s_yw[c] = v.x;
            s_yu[c] = v.y;
        }
    if (pc.need & 4)
        for (int c = threadIdx.x; c < ebt; c += blockDim.x) {
            const float2 v = p.coef[AT.coef[pc.k] + c];
            s_tw[c] = v.x;
            s_tu[c] = v.y;
        }
    __syncthreads();
#if TB_STITCH_PDL
    // everything above read kernel parameters only; from here on the tiles
    // and the output are touched, so the preceding grid must be complete
    asm volatile("griddepcontrol.wait;" ::: "memory");
#endif

#define TB_BOX_ARGS p, pc, s_xw, s_xu, s_yw, s_yu, s_tw, s_tu
    if constexpr (VEC * Elt<DT>::BYTES == 16) {
        const uint32_t s_slots = (uint32_t)__cvta_generic_to_shared(s_stage);
        switch (pc.need) {
            case 0: run_box_pipe<NDIM, 0, DT, VEC>(TB_BOX_ARGS, s_slots); break;
            case 1: run_box_pipe<NDIM, 1, DT, VEC>(TB_BOX_ARGS, s_slots); break;
            case 2: run_box_pipe<NDIM, 2, DT, VEC>(TB_BOX_ARGS, s_slots); break;
            case 3: run_box_pipe<NDIM, 3, DT, VEC>(TB_BOX_ARGS, s_slots); break;
            default:
                if constexpr (NDIM == 3) {
                    switch (pc.need) {
                        case 4: run_box_pipe<NDIM, 4, DT, VEC>(TB_BOX_ARGS, s_slots); break;
                        case 5: run_box_pipe<NDIM, 5, DT, VEC>(TB_BOX_ARGS, s_slots); break;
                        case 6: run_box_pipe<NDIM, 6, DT, VEC>(TB_BOX_ARGS, s_slots); break;
                        case 7: run_box_pipe<NDIM, 7, DT, VEC>(TB_BOX_ARGS, s_slots); break;
                    }
                }
                break;
        }
    } else {
        switch (pc.need) {
            case 0: run_box<NDIM, 0, TB_STITCH_UR_COPY, DT, VEC>(TB_BOX_ARGS); break;
            case 1: run_box<NDIM, 1, TB_STITCH_UR_ONE, DT, VEC>(TB_BOX_ARGS); break;
            case 2: run_box<NDIM, 2, TB_STITCH_UR_ONE, DT, VEC>(TB_BOX_ARGS); break;
            case 3: run_box<NDIM, 3, TB_STITCH_UR_TWO, DT, VEC>(TB_BOX_ARGS); break;
            default:
                if constexpr (NDIM == 3) {
                    switch (pc.need) {
                        case 4: run_box<NDIM, 4, TB_STITCH_UR_ONE, DT, VEC>(TB_BOX_ARGS); break;
                        case 5: run_box<NDIM, 5, TB_STITCH_UR_TWO, DT, VEC>(TB_BOX_ARGS); break;
                        case 6: run_box<NDIM, 6, TB_STITCH_UR_TWO, DT, VEC>(TB_BOX_ARGS); break;
                        case 7: run_box<NDIM, 7, TB_STITCH_UR_THREE, DT, VEC>(TB_BOX_ARGS); break;
                    }
                }
                break;
        }
    }
#undef TB_BOX_ARGS
}

// ---------------------------------------------------------------------------
// TMA path: a CTA stages every source rectangle of its piece with tensor
// copies that complete on one mbarrier, so the piece costs one memory latency
// however many rows it has; the closed form is then evaluated from shared
// memory exactly as on the ring path.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(phase)
        : "memory");
    return ok != 0;
}
// One box [wb columns, rb rows] of a [planes][L_t][L_y][L_x] tile at
// (x, y, t, plane) into shared memory; completes `bar`'s transaction count.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int t, int plane,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(t), "r"(plane), "r"(bar)
        : "memory");
}

// A piece waits for its copies at most this long (nanoseconds of the
// global timer), then reports DEV_WAIT_TIMEOUT and gives up.
#ifndef TB_TMA_WAIT_NS
#define TB_TMA_WAIT_NS 1000000000ull
#endif
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

struct TmaPiece {
    int64_t plane;
    int k, i, j;      // tile
    int t, y, x;      // tile-local frame, first row, first column (elements)
    int rows, wc;     // valid rows, width in chunks
};

template <int NDIM, int NEED, int DT>
__device__ __forceinline__ void run_box_tma(const StitchTmaParams& tp, const TmaPiece& pc, const float* s_xw,
                                            const float* s_xu, const float* s_yw, const float* s_yu,
                                            const float* s_tw, const float* s_tu, uint32_t bar, uint32_t s_data) {
    constexpr int VEC = 16 / Elt<DT>::BYTES;
    constexpr int NN = NDIM == 3 ? 8 : 4;
    constexpr int NU = nodes_of(NEED);
    using C = Chunk<DT, VEC>;
    const auto& p = tp.g;
    const auto& AT = p.ax[0];
    const auto& AY = p.ax[1];
    const auto& AX = p.ax[2];
    const int cpb = tp.wb / VEC;                          // chunks per TMA box row
    const int nblk = (pc.wc + cpb - 1) / cpb;             // TMA boxes per source row block
    const uint32_t box_bytes = (uint32_t)tp.rb * (uint32_t)tp.wb * Elt<DT>::BYTES;
    const uint32_t node_bytes = (uint32_t)nblk * box_bytes;

    // warp 0 arms the barrier and issues every copy: node n, box bk
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) mbar_expect_tx(bar, (uint32_t)NU * node_bytes);
        __syncwarp();
        for (int q = threadIdx.x; q < NU * nblk; q += 32) {
            const int n = q / nblk, bk = q - n * nblk;
            int m = 0;  // the n-th subset of NEED in increasing order
#pragma unroll
            for (int mm = 0, r = 0; mm < NN; ++mm)
                if ((mm & ~NEED) == 0) {
                    if (r == n) m = mm;
                    ++r;
                }
            const int dt = (m >> 2) & 1, dy = (m >> 1) & 1, dx = m & 1;
            const int tile = ((pc.k - dt) * AY.n + (pc.i - dy)) * AX.n + (pc.j - dx);
            const int xs = (dx ? AX.ext[pc.j - 1] - AX.blend[pc.j] : 0) + pc.x + bk * tp.wb;
            const int ys = (dy ? AY.ext[pc.i - 1] - AY.blend[pc.i] : 0) + pc.y;
            const int ts = NDIM == 3 ? (dt ? AT.ext[pc.k - 1] - AT.blend[pc.k] : 0) + pc.t : 0;
            tma_load_4d(s_data + (uint32_t)n * node_bytes + (uint32_t)bk * box_bytes, &tp.maps[tile], xs, ys, ts,
                        (int)pc.plane, bar);
        }
    }
    bool ready = mbar_try_wait(bar, 0);
    if (!ready) {
        const uint64_t t0 = global_ns();
        while (!(ready = mbar_try_wait(bar, 0)) && global_ns() - t0 < TB_TMA_WAIT_NS) {
        }
    }
    if (!ready) {
        if (threadIdx.x == 0 && tp.status != nullptr) atomicCAS(tp.status, (uint32_t)DEV_OK, (uint32_t)DEV_WAIT_TIMEOUT);
        return;
    }

    int bdx, bdy, cpt;
    box_layout(pc.wc, bdx, bdy, cpt);
    const int tx = threadIdx.x % bdx;
    const int ty = threadIdx.x / bdx;
    if (ty >= bdy) return;
    RowCtx<VEC> ctx;
    ctx.stride = node_bytes;
    if constexpr ((NEED & 4) != 0) {
        ctx.wt = s_tw[pc.t];
        ctx.ut = s_tu[pc.t];
    }
    const int64_t orow = (int64_t)p.OW * Elt<DT>::BYTES;
    const Span ospan = out_span<DT>(p);
    char* const obase = reinterpret_cast<char*>(p.out) +
                        ((((pc.plane * p.OT + (NDIM == 3 ? AT.off[pc.k] + pc.t : 0)) * p.OH + AY.off[pc.i] + pc.y) *
                              (int64_t)p.OW +
                          AX.off[pc.j] + pc.x) *
                         Elt<DT>::BYTES);
    for (int q = 0; q < cpt; ++q) {
        const int cc = tx + q * bdx;
        if (cc >= pc.wc) break;
        const int col = pc.x + cc * VEC;
        if constexpr ((NEED & 1) != 0) {
#pragma unroll
            for (int l = 0; l < VEC; ++l) {
                ctx.xw[l] = s_xw[col + l];
                ctx.xu[l] = s_xu[col + l];
            }
        }
        const int blk = cc / cpb;
        const uint32_t cbase = s_data + (uint32_t)blk * box_bytes + (uint32_t)(cc - blk * cpb) * 16u;
        for (int r = ty; r < pc.rows; r += bdy) {
            ctx.base = cbase + (uint32_t)r * (uint32_t)tp.wb * Elt<DT>::BYTES;
            if constexpr ((NEED & 2) != 0) {
                ctx.wy = s_yw[pc.y + r];
                ctx.uy = s_yu[pc.y + r];
            }
            C F[NN];
            DagEval<NDIM, NEED, 3, DT, VEC>::run(ctx, F);
            char* const ot = obase + r * orow + cc * 16;
            if (span_ok(ospan, ot, 16, p.status)) store_chunk<DT, VEC>(ot, 0, F[0]);
        }
    }
}

#ifndef TB_TMA_MIN_CTAS
#define TB_TMA_MIN_CTAS 1
#endif
#ifndef TB_TMA_PREFETCH
#define TB_TMA_PREFETCH 1
#endif

template <int NDIM, int DT>
__global__ void __launch_bounds__(STITCH_BLOCK, TB_TMA_MIN_CTAS)
    stitch_tma_kernel(const __grid_constant__ StitchTmaParams tp) {
    pdl_trigger_dependents();
    constexpr int VEC = 16 / Elt<DT>::BYTES;
    extern __shared__ __align__(128) unsigned char s_dyn[];
    const auto& p = tp.g;
    const auto& AT = p.ax[0];
    const auto& AY = p.ax[1];
    const auto& AX = p.ax[2];

    // which tile and plane (blockIdx.x, tile fastest), which piece (blockIdx.y)
    TmaPiece pc;
    const int ntiles = AX.n * AY.n * (NDIM == 3 ? AT.n : 1);
    const int tile = (int)(blockIdx.x % (unsigned)ntiles);
    pc.plane = (int64_t)(blockIdx.x / (unsigned)ntiles);
    pc.j = tile % AX.n;
    pc.i = (tile / AX.n) % AY.n;
    pc.k = NDIM == 3 ? tile / (AX.n * AY.n) : 0;
    const int Kt = NDIM == 3 ? AT.off[pc.k + 1] - AT.off[pc.k] : 1;
    const int Ky = AY.off[pc.i + 1] - AY.off[pc.i];
    const int Kx = AX.off[pc.j + 1] - AX.off[pc.j];
    const int ebt = (NDIM == 3 && pc.k > 0) ? min(AT.blend[pc.k], Kt) : 0;
    const int eby = pc.i > 0 ? min(AY.blend[pc.i], Ky) : 0;
    const int ebx = pc.j > 0 ? min(AX.blend[pc.j], Kx) : 0;
    int piece = blockIdx.y;
    int need = -1;
    constexpr int NB = NDIM == 3 ? 8 : 4;
    for (int b = NB - 1; b >= 0; --b) {  // same order as tma_tile_pieces()
        const BoxShape s = box_shape(b, Kt, Ky, Kx, ebt, eby, ebx, VEC);
        if (s.nt <= 0 || s.ny <= 0 || s.width <= 0) continue;
        const int np = tma_box_pieces(s, tp.rb, tp.wpc);
        if (piece < np) {
            const int ncb = (s.width + tp.wpc - 1) / tp.wpc;
            const int nrb = (s.ny + tp.rb - 1) / tp.rb;
            const int cb = piece % ncb;
            const int rest = piece / ncb;
            const int rbk = rest % nrb;
            need = b;
            pc.t = s.t0 + rest / nrb;
            pc.y = s.y0 + rbk * tp.rb;
            pc.rows = min(tp.rb, s.ny - rbk * tp.rb);
            pc.x = s.x0 + cb * tp.wpc * VEC;
            pc.wc = min(tp.wpc, s.width - cb * tp.wpc);
            break;
        }
        piece -= np;
    }
    if (need < 0) return;  // this tile has fewer pieces than the grid row
#if TB_TMA_PREFETCH
    // the tensor maps of the (up to 2^d) source tiles, ahead of their copies
    if (threadIdx.x < (1 << NDIM)) {
        const int m = threadIdx.x;
        const int dt = (m >> 2) & 1, dy = (m >> 1) & 1, dx = m & 1;
        if ((m & ~need) == 0) {
            const CUtensorMap* map = &tp.maps[((pc.k - dt) * AY.n + (pc.i - dy)) * AX.n + (pc.j - dx)];
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
        }
    }
#endif

    // shared memory: mbarrier, band coefficients, then the staged sources
    const uint32_t s_raw = (uint32_t)__cvta_generic_to_shared(s_dyn);
    const uint32_t s_base = (s_raw + 127u) & ~127u;
    const uint32_t bar = s_base;
    float* s_coef = reinterpret_cast<float*>(s_dyn + (s_base - s_raw) + 128);
    float* s_xw = s_coef;
    float* s_xu = s_xw + ebx;
    float* s_yw = s_xu + ebx;
    float* s_yu = s_yw + eby;
    float* s_tw = s_yu + eby;
    float* s_tu = s_tw + ebt;
    const uint32_t coef_bytes = (uint32_t)(2 * (ebx + eby + ebt)) * 4u;
    const uint32_t s_data = (s_base + 128u + coef_bytes + 127u) & ~127u;
    if (need & 1)
        for (int c = threadIdx.x; c < ebx; c += blockDim.x) {
            const float2 v = p.coef[AX.coef[pc.j] + c];
            s_xw[c] = v.x;
            s_xu[c] = v.y;
        }
    if (need & 2)
        for (int c = threadIdx.x; c < eby; c += blockDim.x) {
            const float2 v = p.coef[AY.coef[pc.i] + c];
            s_yw[c] = v.x;
            s_yu[c] = v.y;
        }
    if (need & 4)
        for (int c = threadIdx.x; c < ebt; c += blockDim.x) {
            const float2 v = p.coef[AT.coef[pc.k] + c];
            s_tw[c] = v.x;
            s_tu[c] = v.y;
        }
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    // everything above read kernel parameters only; the tiles and the output
    // may belong to the preceding grid
    asm volatile("griddepcontrol.wait;" ::: "memory");

#define TB_TMA_ARGS tp, pc, s_xw, s_xu, s_yw, s_yu, s_tw, s_tu, bar, s_data
    switch (need) {
        case 0: run_box_tma<NDIM, 0, DT>(TB_TMA_ARGS); break;
        case 1: run_box_tma<NDIM, 1, DT>(TB_TMA_ARGS); break;
        case 2: run_box_tma<NDIM, 2, DT>(TB_TMA_ARGS); break;
        case 3: run_box_tma<NDIM, 3, DT>(TB_TMA_ARGS); break;
        default:
            if constexpr (NDIM == 3) {
                switch (need) {
                    case 4: run_box_tma<NDIM, 4, DT>(TB_TMA_ARGS); break;
                    case 5: run_box_tma<NDIM, 5, DT>(TB_TMA_ARGS); break;
                    case 6: run_box_tma<NDIM, 6, DT>(TB_TMA_ARGS); break;
                    case 7: run_box_tma<NDIM, 7, DT>(TB_TMA_ARGS); break;
                }
            }
            break;
    }
#undef TB_TMA_ARGS
}

template <int MAXA, int MAXT, int MAXC>
using KernelFn = void (*)(const StitchParams<MAXA, MAXT, MAXC>);

template <int NDIM, int DT, int MAXA, int MAXT, int MAXC>
KernelFn<MAXA, MAXT, MAXC> pick_vec(int vec) {
    constexpr int V = 16 / Elt<DT>::BYTES;
    return vec == 1 ? stitch_kernel<NDIM, DT, 1, MAXA, MAXT, MAXC> : stitch_kernel<NDIM, DT, V, MAXA, MAXT, MAXC>;
}

template <int MAXA, int MAXT, int MAXC>
KernelFn<MAXA, MAXT, MAXC> pick(const StitchLaunch& l) {
    if (l.ndim == 3) {
        switch (l.dtype) {
            case F32: return pick_vec<3, F32, MAXA, MAXT, MAXC>(l.vec);
            case F16: return pick_vec<3, F16, MAXA, MAXT, MAXC>(l.vec);
            default: return pick_vec<3, BF16, MAXA, MAXT, MAXC>(l.vec);
        }
    }
    switch (l.dtype) {
        case F32: return pick_vec<2, F32, MAXA, MAXT, MAXC>(l.vec);
        case F16: return pick_vec<2, F16, MAXA, MAXT, MAXC>(l.vec);
        default: return pick_vec<2, BF16, MAXA, MAXT, MAXC>(l.vec);
    }
}

template <int MAXA, int MAXT, int MAXC>
cudaError_t launch(const StitchParams<MAXA, MAXT, MAXC>& p, const StitchLaunch& l, cudaStream_t s) {
    auto fn = pick<MAXA, MAXT, MAXC>(l);
    if (l.smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, l.smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(l.grid_x, l.grid_y, l.grid_z);
    cfg.blockDim = dim3(STITCH_BLOCK, 1, 1);
    cfg.dynamicSmemBytes = (size_t)l.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = TB_STITCH_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace

cudaError_t launch_stitch_small(const StitchParamsSmall& p, const StitchLaunch& l, cudaStream_t s) {
    return launch(p, l, s);
}

cudaError_t launch_stitch_large(const StitchParamsLarge& p, const StitchLaunch& l, cudaStream_t s) {
    return launch(p, l, s);
}

cudaError_t launch_stitch_tma(const StitchTmaParams& p, const StitchLaunch& l, cudaStream_t s) {
    void (*fn)(const StitchTmaParams);
    if (l.ndim == 3) {
        fn = l.dtype == F32 ? stitch_tma_kernel<3, F32> : l.dtype == F16 ? stitch_tma_kernel<3, F16>
                                                                        : stitch_tma_kernel<3, BF16>;
    } else {
        fn = l.dtype == F32 ? stitch_tma_kernel<2, F32> : l.dtype == F16 ? stitch_tma_kernel<2, F16>
                                                                        : stitch_tma_kernel<2, BF16>;
    }
    if (l.smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, l.smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(l.grid_x, l.grid_y, l.grid_z);
    cfg.blockDim = dim3(STITCH_BLOCK, 1, 1);
    cfg.dynamicSmemBytes = (size_t)l.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace tb
