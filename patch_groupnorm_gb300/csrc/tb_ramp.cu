// tb_ramp.cu -- normalised-ramp tile stitch for sm_103a.
//
// What is computed (page "Studio: size seam-free VAE tiles from measured
// peaks", unsloth PR #12764, commit "Decode this VAE in 32-latent tiles ..."):
// equally sized tiles overlap; a tile has no weight within `zero` samples of
// an edge it shares with another tile and its weight then rises linearly to
// 1 over `ramp` samples; the weights are normalised to 1 at every sample.
// Output = sum over covering tiles of w_y * w_x * x, divided by the sum of
// the weights -- computed in fp32 and rounded once into the storage type.
//
// How.  The weight of a tile factorises over the axes and so does the
// normaliser, so the normalised weight of tile (a, b) is wy_a * wx_b with
// wy, wx normalised per axis.  The host cuts each axis into segments over
// which the set of tiles with positive weight is constant (at 16-byte chunk
// granularity along the width); the canvas then splits into rectangles with
// a fixed number of source tiles.  A CTA takes a run of rows of one
// rectangle, the rows of all (batch, channel) planes laid end to end so that
// rectangles only a few rows high (latent-space tiles) still fill a CTA, and
// runs a path compiled for its (height cover, width cover) in {1, 2, 3}^2; a
// rectangle covered by one tile is an exact copy (w / w = 1).  Loads stream
// through a per-thread cp.async ring in shared memory, as in the recurrence
// stitch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tb_internal.h"

namespace tb {
namespace {

template <int DT>
struct RElt;
template <>
struct RElt<F32> {
    static constexpr int BYTES = 4;
    __device__ __forceinline__ static void unpack2(uint32_t v, float& lo, float&) { lo = __uint_as_float(v); }
};
template <>
struct RElt<F16> {
    static constexpr int BYTES = 2;
    __device__ __forceinline__ static void unpack2(uint32_t v, float& lo, float& hi) {
        float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
        lo = f.x;
        hi = f.y;
    }
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
};
template <>
struct RElt<BF16> {
    static constexpr int BYTES = 2;
    __device__ __forceinline__ static void unpack2(uint32_t v, float& lo, float& hi) {
        lo = __uint_as_float(v << 16);
        hi = __uint_as_float(v & 0xffff0000u);
    }
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
};

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* gptr) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(saddr), "l"(gptr) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds16(uint32_t saddr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr));
    return v;
}

// Weight of a tile of extent T at tile-local position q, with ramps on the
// shared edges (lo: an edge at the start, hi: an edge at the end).
__device__ __forceinline__ float ramp_weight(int q, int T, bool lo, bool hi, int zero, float inv_ramp) {
    float w = 1.f;
    if (lo) w *= fminf(1.f, fmaxf(0.f, (float)(q - zero) * inv_ramp));
    if (hi) w *= fminf(1.f, fmaxf(0.f, (float)((T - 1 - q) - zero) * inv_ramp));
    return w;
}

// 16-byte chunk -> floats
template <int DT, int VEC>
__device__ __forceinline__ void unpack_chunk(const uint4& v, float (&x)[VEC]) {
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    if constexpr (RElt<DT>::BYTES == 4) {
#pragma unroll
        for (int q = 0; q < 4; ++q) x[q] = __uint_as_float(wd[q]);
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) RElt<DT>::unpack2(wd[q], x[2 * q], x[2 * q + 1]);
    }
}
// floats -> storage, rounded once (element path: the value sits in .x)
template <int DT, int VEC>
__device__ __forceinline__ uint4 acc_pack(const float (&a)[VEC]) {
    if constexpr (VEC == 1) {
        if constexpr (RElt<DT>::BYTES == 4) return make_uint4(__float_as_uint(a[0]), 0, 0, 0);
        else return make_uint4(RElt<DT>::pack2(a[0], 0.f) & 0xffffu, 0, 0, 0);
    } else if constexpr (RElt<DT>::BYTES == 4) {
        return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]), __float_as_uint(a[3]));
    } else {
        return make_uint4(RElt<DT>::pack2(a[0], a[1]), RElt<DT>::pack2(a[2], a[3]), RElt<DT>::pack2(a[4], a[5]),
                          RElt<DT>::pack2(a[6], a[7]));
    }
}

template <int DT>
__device__ __forceinline__ uint32_t load_elem(const char* p) {
    if constexpr (RElt<DT>::BYTES == 4) return __ldcs(reinterpret_cast<const unsigned int*>(p));
    else return __ldcs(reinterpret_cast<const unsigned short*>(p));
}
template <int DT>
__device__ __forceinline__ float elem_value(uint32_t v) {
    float lo, hi = 0.f;
    RElt<DT>::unpack2(v, lo, hi);
    return lo;
}
template <int DT>
__device__ __forceinline__ void store_elem(char* p, uint32_t v) {
    if constexpr (RElt<DT>::BYTES == 4) __stcs(reinterpret_cast<unsigned int*>(p), v);
    else __stcs(reinterpret_cast<unsigned short*>(p), (unsigned short)(v & 0xffffu));
}

constexpr int RAMP_BLOCK = 256;
constexpr int RAMP_SLOTS = 9;  // per thread, 16 bytes each

template <int NA>
__device__ __forceinline__ float axis_w(const RampAxisK& A, int seg, int a, int pos) {
    const int t = A.seg_tile[seg][a];
    return ramp_weight(pos - A.org[t], A.T, t > 0, t < A.n - 1, A.zero, A.inv_ramp);
}

// Position of a row in the flattened (plane, row) space of one rectangle,
// stepped `bdy` rows at a time without division.
struct FlatRow {
    int plane, yl;
    __device__ __forceinline__ void advance(int sq, int sr, int len) {
        plane += sq;
        yl += sr;
        if (yl >= len) {
            yl -= len;
            ++plane;
        }
    }
};

template <int CY, int CX, int DT, int VEC>
__device__ __forceinline__ void run_rect(const RampParams& p, int sy, int sx, int fbeg, int fend, uint32_t s_ring) {
    constexpr int NU = CY * CX;
    constexpr int S = RAMP_SLOTS / NU >= 2 ? RAMP_SLOTS / NU : 1;
    const RampAxisK& AY = p.ay;
    const RampAxisK& AX = p.ax;
    const int width = AX.seg_len[sx] / VEC;  // chunks
    const int bdx = width < RAMP_BLOCK ? width : RAMP_BLOCK;
    const int bdy = RAMP_BLOCK / bdx;
    const int tx = threadIdx.x % bdx;
    const int ty = threadIdx.x / bdx;
    if (ty >= bdy) return;
    const uint32_t slot_stride = RAMP_BLOCK * 16u;
    const uint32_t my_slot = s_ring + threadIdx.x * 16u;
    for (int c = tx; c < width; c += bdx) {
        const int x0 = AX.seg_start[sx] + c * VEC;
        // normalised width weights of this chunk's lanes
        float wx[CX][VEC];
        if constexpr (CX > 1) {
#pragma unroll
            for (int l = 0; l < VEC; ++l) {
                float sum = 0.f;
#pragma unroll
                for (int b = 0; b < CX; ++b) {
                    wx[b][l] = axis_w<CX>(AX, sx, b, x0 + l);
                    sum += wx[b][l];
                }
                const float inv = 1.0f / sum;
#pragma unroll
                for (int b = 0; b < CX; ++b) wx[b][l] *= inv;
            }
        }
        // sources: tile (Y.tile[a], X.tile[b]) at plane 0, canvas row y0
        const int y0 = AY.seg_start[sy];
        const char* src[NU];
        const char* tbase[NU];  // the bounds-checked build's source ranges
        const int32_t pitch = AX.T * RElt<DT>::BYTES;
        const int64_t tplane = (int64_t)AY.T * AX.T * RElt<DT>::BYTES;
        const int64_t tbytes = p.planes * tplane;
        const int64_t obytes = p.planes * (int64_t)AY.out * AX.out * RElt<DT>::BYTES;
#pragma unroll
        for (int a = 0; a < CY; ++a)
#pragma unroll
            for (int b = 0; b < CX; ++b) {
                const int ti = AY.seg_tile[sy][a], tj = AX.seg_tile[sx][b];
                index_ok(ti >= 0 && ti < AY.n && tj >= 0 && tj < AX.n, p.status);
                tbase[a * CX + b] = reinterpret_cast<const char*>(p.tiles[ti * AX.n + tj]);
                // element (plane, y0 + yl - oy, x0 - ox) of tile (ti, tj) is
                // src + plane * tplane + yl * pitch
                src[a * CX + b] = reinterpret_cast<const char*>(p.tiles[ti * AX.n + tj]) +
                                  ((int64_t)(y0 - AY.org[ti]) * AX.T + (x0 - AX.org[tj])) * RElt<DT>::BYTES;
            }
        char* dst = reinterpret_cast<char*>(p.out) + ((int64_t)y0 * AX.out + x0) * RElt<DT>::BYTES;
        const int32_t opitch = AX.out * RElt<DT>::BYTES;
        const int64_t oplane = (int64_t)AY.out * AX.out * RElt<DT>::BYTES;

        const int len = AY.seg_len[sy];
        const int sq = bdy / len, sr = bdy % len;
        const int r0 = fbeg + ty;
        const int nrows = r0 < fend ? (fend - r0 + bdy - 1) / bdy : 0;
        const FlatRow first = {r0 / len, r0 % len};
        // combine the CY x CX source values of one row; x_ab(l) reads them
        auto combine = [&](int y, auto x_ab) {
            float wy[CY];
            if constexpr (CY > 1) {
                float sum = 0.f;
#pragma unroll
                for (int a = 0; a < CY; ++a) {
                    wy[a] = axis_w<CY>(AY, sy, a, y);
                    sum += wy[a];
                }
                const float inv = 1.0f / sum;
#pragma unroll
                for (int a = 0; a < CY; ++a) wy[a] *= inv;
            } else {
                wy[0] = 1.f;
            }
            float acc[VEC];
#pragma unroll
            for (int l = 0; l < VEC; ++l) acc[l] = 0.f;
#pragma unroll
            for (int a = 0; a < CY; ++a)
#pragma unroll
                for (int b = 0; b < CX; ++b) {
                    float x[VEC];
                    x_ab(a, b, x);
#pragma unroll
                    for (int l = 0; l < VEC; ++l) {
                        const float wgt = CX > 1 ? wy[a] * wx[b][l] : wy[a];
                        acc[l] = fmaf(wgt, x[l], acc[l]);
                    }
                }
            return acc_pack<DT, VEC>(acc);
        };
        if constexpr (VEC * RElt<DT>::BYTES == 16) {
            FlatRow ahead = first;  // the next row to issue
            auto issue = [&](int m) {
                const int64_t off = ahead.plane * tplane + (int64_t)ahead.yl * pitch;
                const uint32_t st = my_slot + (uint32_t)((m % S) * NU) * slot_stride;
#pragma unroll
                for (int n = 0; n < NU; ++n)
                    if (in_bounds(src[n] + off, 16, tbase[n], tbytes, p.status))
                        cp_async16(st + (uint32_t)n * slot_stride, src[n] + off);
                ahead.advance(sq, sr, len);
            };
#pragma unroll
            for (int m = 0; m < S - 1; ++m) {
                if (m < nrows) issue(m);
                cp_async_commit();
            }
            FlatRow at = first;
            for (int m = 0; m < nrows; ++m) {
                if (m + S - 1 < nrows) issue(m + S - 1);
                cp_async_commit();
                cp_async_wait<S - 1>();
                const uint32_t st = my_slot + (uint32_t)((m % S) * NU) * slot_stride;
                uint4 o;
                if constexpr (NU == 1) {
                    o = lds16(st);  // one tile: its normalised weight is exactly 1
                } else {
                    o = combine(y0 + at.yl, [&](int a, int b, float (&x)[VEC]) {
                        const uint4 v = lds16(st + (uint32_t)(a * CX + b) * slot_stride);
                        unpack_chunk<DT, VEC>(v, x);
                    });
                }
                char* const ot = dst + at.plane * oplane + (int64_t)at.yl * opitch;
                if (in_bounds(ot, 16, p.out, obytes, p.status)) __stcs(reinterpret_cast<uint4*>(ot), o);
                at.advance(sq, sr, len);
            }
            cp_async_wait<0>();
        } else {
            // element path (unaligned geometry): plain loads, one row at a time
            FlatRow at = first;
            for (int m = 0; m < nrows; ++m) {
                const int64_t off = at.plane * tplane + (int64_t)at.yl * pitch;
                char* const o_at = dst + at.plane * oplane + (int64_t)at.yl * opitch;
                const bool store_ok = in_bounds(o_at, RElt<DT>::BYTES, p.out, obytes, p.status);
                if constexpr (NU == 1) {
                    if (store_ok && in_bounds(src[0] + off, RElt<DT>::BYTES, tbase[0], tbytes, p.status))
                        store_elem<DT>(o_at, load_elem<DT>(src[0] + off));
                } else {
                    const uint4 o = combine(y0 + at.yl, [&](int a, int b, float (&x)[VEC]) {
                        const char* at_src = src[a * CX + b] + off;
                        x[0] = in_bounds(at_src, RElt<DT>::BYTES, tbase[a * CX + b], tbytes, p.status)
                                   ? elem_value<DT>(load_elem<DT>(at_src))
                                   : 0.f;
                    });
                    if (store_ok) store_elem<DT>(o_at, o.x);
                }
                at.advance(sq, sr, len);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// 16-byte path: weights precomputed per CTA, lane pairs in packed fp32
// ---------------------------------------------------------------------------

// Rows of a rectangle whose normalised height weights, and 16-byte columns
// whose normalised width weights, one CTA tabulates in shared memory (larger
// multi-cover rectangles compute them per row or per column).
constexpr int RAMP_WY_CAP = 256;
constexpr int RAMP_WX_CAP = 64;

using u64 = unsigned long long;
__device__ __forceinline__ u64 pk2(float lo, float hi) {
    u64 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void upk2(u64 v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
    u64 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
    u64 r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// A 16-byte chunk as fp32 lane pairs (element 2w in the low half).
template <int DT>
__device__ __forceinline__ void chunk_pairs(const uint4& v, u64 (&x)[RElt<DT>::BYTES == 4 ? 2 : 4]) {
    if constexpr (RElt<DT>::BYTES == 4) {
        x[0] = pk2(__uint_as_float(v.x), __uint_as_float(v.y));
        x[1] = pk2(__uint_as_float(v.z), __uint_as_float(v.w));
    } else {
        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float lo, hi;
            RElt<DT>::unpack2(wd[q], lo, hi);
            x[q] = pk2(lo, hi);
        }
    }
}
template <int DT>
__device__ __forceinline__ uint4 pairs_chunk(const u64 (&a)[RElt<DT>::BYTES == 4 ? 2 : 4]) {
    if constexpr (RElt<DT>::BYTES == 4) {
        float f0, f1, f2, f3;
        upk2(a[0], f0, f1);
        upk2(a[1], f2, f3);
        return make_uint4(__float_as_uint(f0), __float_as_uint(f1), __float_as_uint(f2), __float_as_uint(f3));
    } else {
        uint32_t wd[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float lo, hi;
            upk2(a[q], lo, hi);
            wd[q] = RElt<DT>::pack2(lo, hi);
        }
        return make_uint4(wd[0], wd[1], wd[2], wd[3]);
    }
}

// Position of a row in a rectangle's flattened (plane, row) space, with the
// byte offset of that row in a source tile and in the output, stepped `bdy`
// rows at a time with additions only.
struct RowCursor {
    int plane, yl;
    int64_t src, dst;
};

template <int CY, int CX, int DT>
__device__ __forceinline__ void run_rect_vec(const RampParams& p, int sy, int sx, int fbeg, int fend,
                                             uint32_t s_ring, const float* s_wy, bool wy_table, const float* s_wx,
                                             bool wx_table) {
    constexpr int VEC = 16 / RElt<DT>::BYTES;
    constexpr int NP = RElt<DT>::BYTES == 4 ? 2 : 4;  // lane pairs per chunk
    constexpr int NU = CY * CX;
    constexpr int S = RAMP_SLOTS / NU >= 2 ? RAMP_SLOTS / NU : 1;
    const RampAxisK& AY = p.ay;
    const RampAxisK& AX = p.ax;
    const int width = AX.seg_len[sx] / VEC;  // chunks
    const int bdx = width < RAMP_BLOCK ? width : RAMP_BLOCK;
    const int bdy = RAMP_BLOCK / bdx;
    const int tx = threadIdx.x % bdx;
    const int ty = threadIdx.x / bdx;
    if (ty >= bdy) return;
    const uint32_t slot_stride = RAMP_BLOCK * 16u;
    const uint32_t my_slot = s_ring + threadIdx.x * 16u;
    const int y0 = AY.seg_start[sy];
    const int len = AY.seg_len[sy];
    const int32_t pitch = AX.T * RElt<DT>::BYTES;
    const int64_t tplane = (int64_t)AY.T * AX.T * RElt<DT>::BYTES;
    const int32_t opitch = AX.out * RElt<DT>::BYTES;
    const int64_t oplane = (int64_t)AY.out * AX.out * RElt<DT>::BYTES;
    const int64_t tbytes = p.planes * tplane;                        // bounds-checked build
    const int64_t obytes = p.planes * oplane;
    const int sq = bdy / len, sr = bdy % len;
    const int64_t src_step = sq * tplane + (int64_t)sr * pitch, src_wrap = tplane - (int64_t)len * pitch;
    const int64_t dst_step = sq * oplane + (int64_t)sr * opitch, dst_wrap = oplane - (int64_t)len * opitch;
    auto advance = [&](RowCursor& c) {
        c.plane += sq;
        c.yl += sr;
        c.src += src_step;
        c.dst += dst_step;
        if (c.yl >= len) {
            c.yl -= len;
            ++c.plane;
            c.src += src_wrap;
            c.dst += dst_wrap;
        }
    };
    const int r0 = fbeg + ty;
    const int nrows = r0 < fend ? (fend - r0 + bdy - 1) / bdy : 0;
    RowCursor first;
    first.plane = r0 / len;
    first.yl = r0 - first.plane * len;
    first.src = first.plane * tplane + (int64_t)first.yl * pitch;
    first.dst = first.plane * oplane + (int64_t)first.yl * opitch;

    for (int c = tx; c < width; c += bdx) {
        const int x0 = AX.seg_start[sx] + c * VEC;
        // normalised width weights of this chunk's lanes, as lane pairs
        u64 wxp[CX][NP];
        if constexpr (CX > 1) {
            float wx[CX][VEC];
            if (wx_table) {
#pragma unroll
                for (int l = 0; l < VEC; ++l)
#pragma unroll
                    for (int b = 0; b < CX; ++b) wx[b][l] = s_wx[(c * VEC + l) * CX + b];
            } else {
#pragma unroll
                for (int l = 0; l < VEC; ++l) {
                    float sum = 0.f;
#pragma unroll
                    for (int b = 0; b < CX; ++b) {
                        wx[b][l] = axis_w<CX>(AX, sx, b, x0 + l);
                        sum += wx[b][l];
                    }
                    const float inv = 1.0f / sum;
#pragma unroll
                    for (int b = 0; b < CX; ++b) wx[b][l] *= inv;
                }
            }
#pragma unroll
            for (int b = 0; b < CX; ++b)
#pragma unroll
                for (int w = 0; w < NP; ++w) wxp[b][w] = pk2(wx[b][2 * w], wx[b][2 * w + 1]);
        }
        const char* src[NU];
        const char* tbase[NU];
#pragma unroll
        for (int a = 0; a < CY; ++a)
#pragma unroll
            for (int b = 0; b < CX; ++b) {
                const int ti = AY.seg_tile[sy][a], tj = AX.seg_tile[sx][b];
                index_ok(ti >= 0 && ti < AY.n && tj >= 0 && tj < AX.n, p.status);
                tbase[a * CX + b] = reinterpret_cast<const char*>(p.tiles[ti * AX.n + tj]);
                src[a * CX + b] = tbase[a * CX + b] +
                                  ((int64_t)(y0 - AY.org[ti]) * AX.T + (x0 - AX.org[tj])) * RElt<DT>::BYTES;
            }
        char* const dst = reinterpret_cast<char*>(p.out) + ((int64_t)y0 * AX.out + x0) * RElt<DT>::BYTES;

        RowCursor ahead = first;  // the next row to fetch
        auto issue = [&](int m) {
            const uint32_t st = my_slot + (uint32_t)((m % S) * NU) * slot_stride;
#pragma unroll
            for (int n = 0; n < NU; ++n)
                if (in_bounds(src[n] + ahead.src, 16, tbase[n], tbytes, p.status))
                    cp_async16(st + (uint32_t)n * slot_stride, src[n] + ahead.src);
            advance(ahead);
        };
#pragma unroll
        for (int m = 0; m < S - 1; ++m) {
            if (m < nrows) issue(m);
            cp_async_commit();
        }
        RowCursor at = first;
        for (int m = 0; m < nrows; ++m) {
            if (m + S - 1 < nrows) issue(m + S - 1);
            cp_async_commit();
            cp_async_wait<S - 1>();
            const uint32_t st = my_slot + (uint32_t)((m % S) * NU) * slot_stride;
            uint4 o;
            if constexpr (NU == 1) {
                o = lds16(st);  // one tile: its normalised weight is exactly 1
            } else {
                float wy[CY];
                if constexpr (CY > 1) {
                    if (wy_table) {
#pragma unroll
                        for (int a = 0; a < CY; ++a) wy[a] = s_wy[at.yl * CY + a];
                    } else {
                        float sum = 0.f;
#pragma unroll
                        for (int a = 0; a < CY; ++a) {
                            wy[a] = axis_w<CY>(AY, sy, a, y0 + at.yl);
                            sum += wy[a];
                        }
                        const float inv = 1.0f / sum;
#pragma unroll
                        for (int a = 0; a < CY; ++a) wy[a] *= inv;
                    }
                }
                // sum over a of wy[a] * (sum over b of wx[b] * x_ab), lane pairs
                u64 acc[NP];
#pragma unroll
                for (int a = 0; a < CY; ++a) {
                    u64 inner[NP];
#pragma unroll
                    for (int b = 0; b < CX; ++b) {
                        u64 x[NP];
                        chunk_pairs<DT>(lds16(st + (uint32_t)(a * CX + b) * slot_stride), x);
#pragma unroll
                        for (int w = 0; w < NP; ++w) {
                            if constexpr (CX == 1) inner[w] = x[w];
                            else inner[w] = b == 0 ? mul2(x[w], wxp[0][w]) : fma2(x[w], wxp[b][w], inner[w]);
                        }
                    }
                    if constexpr (CY == 1) {
#pragma unroll
                        for (int w = 0; w < NP; ++w) acc[w] = inner[w];
                    } else {
                        const u64 wyp = pk2(wy[a], wy[a]);
#pragma unroll
                        for (int w = 0; w < NP; ++w) acc[w] = a == 0 ? mul2(inner[w], wyp) : fma2(inner[w], wyp, acc[w]);
                    }
                }
                o = pairs_chunk<DT>(acc);
            }
            char* const ot = dst + at.dst;
            if (in_bounds(ot, 16, p.out, obytes, p.status)) __stcs(reinterpret_cast<uint4*>(ot), o);
            advance(at);
        }
        cp_async_wait<0>();
    }
}

#ifndef TB_RAMP_MIN_CTAS_2
#define TB_RAMP_MIN_CTAS_2 4
#endif

// MAXC = 2: the rectangles covered by at most 2 x 2 tiles; MAXC = 3: those
// with 3 tiles along an axis (a separate, larger kernel launched only when
// such rectangles exist, so the common one keeps fewer registers and less
// code).
template <int DT, int VEC, int MAXC>
__global__ void __launch_bounds__(RAMP_BLOCK, MAXC == 2 ? TB_RAMP_MIN_CTAS_2 : 3)
    ramp_kernel(const __grid_constant__ RampParams p) {
    extern __shared__ __align__(16) unsigned char s_ring[];
    __shared__ float s_wy[RAMP_WY_CAP * RAMP_MAXCOVER];
    __shared__ float s_wx[RAMP_WX_CAP * 8 * RAMP_MAXCOVER];
    // A piece is a run of rows of one rectangle, in the rectangle's (plane,
    // row) space flattened over all planes.  blockIdx.y is the piece index and
    // blockIdx.x the rectangle, so the CTAs launched first cover every
    // rectangle, i.e. whole rows of the canvas; rectangles with fewer pieces
    // leave their trailing CTAs empty.  The rectangles are numbered group by
    // group of equal (height cover, width cover), so that CTAs dispatched
    // together mostly run one code path (fewer instruction-cache misses).
    int sy, sx;
    {
        constexpr int NG = MAXC == 2 ? 4 : 5;
        constexpr int groups[2][5] = {{0, 1, 3, 4, 0}, {2, 5, 6, 7, 8}};
        int idx = (int)blockIdx.x, g = -1;
#pragma unroll
        for (int q = 0; q < NG; ++q) {
            const int gq = groups[MAXC - 2][q];
            const int cnt = p.ycnt[gq / RAMP_MAXCOVER] * p.xcnt[gq % RAMP_MAXCOVER];
            if (g < 0) {
                if (idx < cnt) g = gq;
                else idx -= cnt;
            }
        }
        if (g < 0) return;
        const int gy = g / RAMP_MAXCOVER, gx = g - gy * RAMP_MAXCOVER;
        const int iy = idx / p.xcnt[gx];
        sy = p.yseg[gy][iy];
        sx = p.xseg[gx][idx - iy * p.xcnt[gx]];
    }
    const int rem = (int)blockIdx.y;
    const int flat = (int)p.planes * p.ay.seg_len[sy];
    const int fbeg = rem * p.rows_per_piece[sx];
    if (fbeg >= flat) return;
    const int fend = min(flat, fbeg + p.rows_per_piece[sx]);
    const int cy = p.ay.seg_n[sy], cx = p.ax.seg_n[sx];
    // the rectangle's normalised height weights (parameters only)
    const int len = p.ay.seg_len[sy];
    const bool wy_table = cy > 1 && len <= RAMP_WY_CAP;
    const int wcols = p.ax.seg_len[sx];  // samples
    const bool wx_table = cx > 1 && wcols <= RAMP_WX_CAP * VEC;
    if constexpr (VEC * RElt<DT>::BYTES == 16) {
        if (wx_table) {
            const int x0 = p.ax.seg_start[sx];
            for (int xl = threadIdx.x; xl < wcols; xl += RAMP_BLOCK) {
                float w[RAMP_MAXCOVER], sum = 0.f;
                for (int b = 0; b < cx; ++b) {
                    w[b] = axis_w<1>(p.ax, sx, b, x0 + xl);
                    sum += w[b];
                }
                const float inv = 1.0f / sum;
                for (int b = 0; b < cx; ++b) s_wx[xl * cx + b] = w[b] * inv;
            }
        }
        if (wy_table) {
            const int y0 = p.ay.seg_start[sy];
            for (int yl = threadIdx.x; yl < len; yl += RAMP_BLOCK) {
                float w[RAMP_MAXCOVER], sum = 0.f;
                for (int a = 0; a < cy; ++a) {
                    w[a] = axis_w<1>(p.ay, sy, a, y0 + yl);
                    sum += w[a];
                }
                const float inv = 1.0f / sum;
                for (int a = 0; a < cy; ++a) s_wy[yl * cy + a] = w[a] * inv;
            }
        }
        if (wy_table || wx_table) __syncthreads();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t ring = (uint32_t)__cvta_generic_to_shared(s_ring);
    if constexpr (VEC * RElt<DT>::BYTES == 16) {
#define TB_RECT(CY_, CX_) run_rect_vec<CY_, CX_, DT>(p, sy, sx, fbeg, fend, ring, s_wy, wy_table, s_wx, wx_table)
        if constexpr (MAXC == 2) {
            switch (cy * 4 + cx) {
                case 5: TB_RECT(1, 1); break;
                case 6: TB_RECT(1, 2); break;
                case 9: TB_RECT(2, 1); break;
                case 10: TB_RECT(2, 2); break;
                default: break;
            }
        } else {
            switch (cy * 4 + cx) {
                case 7: TB_RECT(1, 3); break;
                case 11: TB_RECT(2, 3); break;
                case 13: TB_RECT(3, 1); break;
                case 14: TB_RECT(3, 2); break;
                case 15: TB_RECT(3, 3); break;
                default: break;
            }
        }
#undef TB_RECT
    } else {
#define TB_RECT(CY_, CX_) run_rect<CY_, CX_, DT, VEC>(p, sy, sx, fbeg, fend, ring)
        if constexpr (MAXC == 2) {
            switch (cy * 4 + cx) {
                case 5: TB_RECT(1, 1); break;
                case 6: TB_RECT(1, 2); break;
                case 9: TB_RECT(2, 1); break;
                case 10: TB_RECT(2, 2); break;
                default: break;
            }
        } else {
            switch (cy * 4 + cx) {
                case 7: TB_RECT(1, 3); break;
                case 11: TB_RECT(2, 3); break;
                case 13: TB_RECT(3, 1); break;
                case 14: TB_RECT(3, 2); break;
                case 15: TB_RECT(3, 3); break;
                default: break;
            }
        }
#undef TB_RECT
    }
}

}  // namespace

int ramp_block() { return RAMP_BLOCK; }
int ramp_smem() { return RAMP_SLOTS * RAMP_BLOCK * 16; }

cudaError_t launch_ramp(const RampParams& p, int dtype, int vec, int grid_small, int grid_large, int grid_y,
                        cudaStream_t s) {
    for (int big = 0; big < 2; ++big) {
        const int grid_x = big ? grid_large : grid_small;
        if (grid_x <= 0) continue;
        void (*fn)(const RampParams);
        if (big) {
            switch (dtype) {
                case F32: fn = vec > 1 ? ramp_kernel<F32, 4, 3> : ramp_kernel<F32, 1, 3>; break;
                case F16: fn = vec > 1 ? ramp_kernel<F16, 8, 3> : ramp_kernel<F16, 1, 3>; break;
                default: fn = vec > 1 ? ramp_kernel<BF16, 8, 3> : ramp_kernel<BF16, 1, 3>; break;
            }
        } else {
            switch (dtype) {
                case F32: fn = vec > 1 ? ramp_kernel<F32, 4, 2> : ramp_kernel<F32, 1, 2>; break;
                case F16: fn = vec > 1 ? ramp_kernel<F16, 8, 2> : ramp_kernel<F16, 1, 2>; break;
                default: fn = vec > 1 ? ramp_kernel<BF16, 8, 2> : ramp_kernel<BF16, 1, 2>; break;
            }
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid_x, (unsigned)grid_y, 1);
        cfg.blockDim = dim3(RAMP_BLOCK, 1, 1);
        cfg.dynamicSmemBytes = vec > 1 ? (size_t)ramp_smem() : 0;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol.wait
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, fn, p);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace tb
