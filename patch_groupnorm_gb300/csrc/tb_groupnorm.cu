// tb_groupnorm.cu -- patch-parallel GroupNorm (+ SiLU) kernels for sm_103a.
//
// What is computed (page "Add tiled VAE parallelism & extended model
// support", xDiT DistVAE PR #14, the PatchGroupNorm commits): a GroupNorm
// over an activation split into P patches must equal GroupNorm of the whole
// tensor -- the group mean pooled over all patches and the biased variance
// (divided by the count) about that pooled mean -- followed by the affine
// and, in the decoder blocks, SiLU.
//
// The page's implementation meets across ranks twice per norm (one
// all_reduce for the count and the sums, a second for the squares about the
// pooled mean, because folding the second into the first would change the
// estimator).  Here every patch is resident on one GPU, and each patch's
// statistics travel as (count, mean, M2) -- the sum of squared deviations
// about the patch's own mean.  Chan's pairwise update combines such triples
// exactly (up to rounding) into the pooled mean and the M2 about it, so one
// pass over the data suffices and the combination needs no second reduction:
//     n = nA + nB,  d = meanB - meanA,
//     mean = meanA + d * nB / n,  M2 = M2A + M2B + d^2 * nA * nB / n.
//
// gn_stats_kernel: each (patch, sample, group) unit's elements are cut into
// `parts` contiguous parts (1 .. TB_GN_PARTS, chosen on the host from the
// sizes and the SM count), one CTA per part; every part's statistics go to
// their own record and the unit's remaining records get count 0, so the
// records describe themselves (the apply step merges every record with
// elements, whatever split produced it).  Each thread streams 16-byte chunks through a
// ring of cp.async slots, seven ahead (range checks only in the last groups
// of its run).  For fp16 / bf16 it sums x - K and
// (x - K)^2 over groups of 8 chunks (64 elements) on packed fp32 pairs, K
// being the group's first element -- differences and squares of 16-bit
// values are nearly always exact in fp32, and the shift keeps
// M2 = S2 - S1^2 / m from cancelling -- and folds each group into its
// running triple with Chan's update; fp32 chunks are folded one by one after
// their own mean and M2 are computed directly.  Warps merge with shuffles and
// then through shared memory, in a fixed order (deterministic results).
// Earlier versions merged the CTAs of a unit in a thread-block cluster over
// distributed shared memory into one record; the cluster's scheduling and
// barriers cost about 1 us per launch (measured), more than the extra
// records cost the apply step.
//
// Both kernels are launched with programmatic stream serialisation: their
// parameter-only prologue may overlap the preceding kernel, and they execute
// griddepcontrol.wait before touching global memory.
//
// gn_apply_kernel: one CTA per segment of one channel row.  The CTA issues
// its data loads, then each warp combines the R * TB_GN_PARTS records of the
// row's group (pooled_stats; R record sets, one per patch of the whole
// tensor, possibly gathered from other ranks) into a = rstd * gamma[c] and
// b = beta[c] - mean * a; the elements become
// y = silu(x * a + b), rounded once into the storage type.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tb_internal.h"

namespace tb {
namespace {

#ifndef TB_GN_STATS_BLOCK
#define TB_GN_STATS_BLOCK 256
#endif
#ifndef TB_GN_STATS_SLOTS
#define TB_GN_STATS_SLOTS 8
#endif
constexpr int STATS_BLOCK = TB_GN_STATS_BLOCK;
constexpr int STATS_SLOTS = TB_GN_STATS_SLOTS;  // cp.async ring slots per thread (16 bytes each)
#ifndef TB_GN_STATS_GROUP
#define TB_GN_STATS_GROUP 8
#endif
constexpr int STATS_GROUP = TB_GN_STATS_GROUP;  // 16-bit chunks per shifted-sum group
constexpr int APPLY_BLOCK = 128;
#ifndef TB_GN_APPLY_CPT
#define TB_GN_APPLY_CPT 16
#endif
constexpr int APPLY_CPT = TB_GN_APPLY_CPT;  // 16-byte chunks per thread per segment

template <int DT>
struct GElt;
template <>
struct GElt<F32> {
    static constexpr int BYTES = 4;
    __device__ __forceinline__ static float to_f(uint32_t v) { return __uint_as_float(v); }
};
template <>
struct GElt<F16> {
    static constexpr int BYTES = 2;
    __device__ __forceinline__ static void unpack(uint32_t v, float& lo, float& hi) {
        float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
        lo = f.x;
        hi = f.y;
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ __forceinline__ static float to_f(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)v)); }
};
template <>
struct GElt<BF16> {
    static constexpr int BYTES = 2;
    __device__ __forceinline__ static void unpack(uint32_t v, float& lo, float& hi) {
        lo = __uint_as_float(v << 16);
        hi = __uint_as_float(v & 0xffff0000u);
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    __device__ __forceinline__ static float to_f(uint32_t v) { return __uint_as_float(v << 16); }
};

// Elements of one 16-byte chunk as floats.
template <int DT>
__device__ __forceinline__ void chunk_to_floats(const uint4& v, float (&x)[16 / GElt<DT>::BYTES]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    if constexpr (GElt<DT>::BYTES == 4) {
#pragma unroll
        for (int q = 0; q < 4; ++q) x[q] = __uint_as_float(w[q]);
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) GElt<DT>::unpack(w[q], x[2 * q], x[2 * q + 1]);
    }
}

// Scalar element load (unaligned paths).
template <int DT>
__device__ __forceinline__ float load_scalar(const void* base, int64_t i) {
    if constexpr (GElt<DT>::BYTES == 4) {
        return __ldcs(reinterpret_cast<const float*>(base) + i);
    } else {
        return GElt<DT>::to_f(__ldcs(reinterpret_cast<const unsigned short*>(base) + i));
    }
}

struct Stat {
    float n, mean, m2;
};

// Chan's pairwise combination of two (count, mean, M2) triples.
__device__ __forceinline__ Stat chan(const Stat& a, const Stat& b) {
    if (b.n == 0.f) return a;
    if (a.n == 0.f) return b;
    const float n = a.n + b.n;
    const float r = b.n / n;
    const float d = b.mean - a.mean;
    Stat s;
    s.n = n;
    s.mean = fmaf(d, r, a.mean);
    s.m2 = a.m2 + b.m2 + d * d * a.n * r;
    return s;
}

// (count, mean, M2) of a block of K elements, computed directly.
template <int K>
__device__ __forceinline__ Stat block_stat(const float (&x)[K]) {
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < K; ++q) s += x[q];
    const float mean = s * (1.0f / K);
    float m2 = 0.f;
#pragma unroll
    for (int q = 0; q < K; ++q) {
        const float d = x[q] - mean;
        m2 = fmaf(d, d, m2);
    }
    return Stat{(float)K, mean, m2};
}

__device__ __forceinline__ Stat shfl_down_stat(const Stat& s, int delta) {
    return Stat{__shfl_down_sync(0xffffffffu, s.n, delta), __shfl_down_sync(0xffffffffu, s.mean, delta),
                __shfl_down_sync(0xffffffffu, s.m2, delta)};
}

__device__ __forceinline__ Stat warp_reduce(Stat s) {
#pragma unroll
    for (int delta = 16; delta >= 1; delta >>= 1) s = chan(s, shfl_down_stat(s, delta));
    return s;  // valid in lane 0
}

// Chan's update with an approximate quotient, for a thread's own running
// merge of equal-sized blocks (the counts are exact; the ratio's last-bit
// error is far below the statistics' tolerance).
__device__ __forceinline__ Stat chan_fast(const Stat& a, const Stat& b) {
    const float n = a.n + b.n;
    const float r = __fdividef(b.n, n);
    const float d = b.mean - a.mean;
    Stat s;
    s.n = n;
    s.mean = fmaf(d, r, a.mean);
    s.m2 = a.m2 + b.m2 + d * d * a.n * r;
    return s;
}

// Shifted sums of the two 16-bit lanes of word v, on packed fp32 pairs:
// s1 += x - K, s2 += (x - K)^2 (k2 holds K in both lanes).
template <int DT>
__device__ __forceinline__ void shifted_acc(uint32_t v, unsigned long long k2, unsigned long long& s1,
                                            unsigned long long& s2) {
    if constexpr (DT == BF16) {
        asm("{\n\t.reg .b32 lo, hi;\n\t.reg .b64 x, d;\n\t"
            "shl.b32 lo, %2, 16;\n\t"
            "and.b32 hi, %2, 0xffff0000;\n\t"
            "mov.b64 x, {lo, hi};\n\t"
            "sub.rn.f32x2 d, x, %3;\n\t"
            "add.rn.f32x2 %0, %0, d;\n\t"
            "fma.rn.f32x2 %1, d, d, %1;\n\t}"
            : "+l"(s1), "+l"(s2)
            : "r"(v), "l"(k2));
    } else {
        asm("{\n\t.reg .b16 hl, hh;\n\t.reg .b32 lo, hi;\n\t.reg .b64 x, d;\n\t"
            "mov.b32 {hl, hh}, %2;\n\t"
            "cvt.f32.f16 lo, hl;\n\t"
            "cvt.f32.f16 hi, hh;\n\t"
            "mov.b64 x, {lo, hi};\n\t"
            "sub.rn.f32x2 d, x, %3;\n\t"
            "add.rn.f32x2 %0, %0, d;\n\t"
            "fma.rn.f32x2 %1, d, d, %1;\n\t}"
            : "+l"(s1), "+l"(s2)
            : "r"(v), "l"(k2));
    }
}

__device__ __forceinline__ float lane_sum(unsigned long long v) {
    return __uint_as_float((uint32_t)v) + __uint_as_float((uint32_t)(v >> 32));
}

// (count, mean, M2) of a group of m elements from its shifted sums about K:
// mean = K + s1 / m, M2 = s2 - s1^2 / m.  K is the group's first element,
// so the shift removes the group's offset and the subtraction loses little.
__device__ __forceinline__ Stat shifted_stat(unsigned long long s1, unsigned long long s2, float K, float m) {
    const float a = lane_sum(s1), b = lane_sum(s2);
    const float q = __fdividef(a, m);
    return Stat{m, K + q, fmaxf(0.f, fmaf(-a, q, b))};
}

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

// Groups whose chunks and fetches ahead are all in range skip the range
// checks (0: every group checks, as the tail of a thread's run does).
#ifndef TB_GN_FAST_GROUPS
#define TB_GN_FAST_GROUPS 1
#endif

// The shifted sums of the group of chunks k0 .. k0 + STATS_GROUP - 1 from the
// thread's cp.async ring (the group starts on ring slot 0), each chunk
// fetching the one STATS_SLOTS - 1 ahead at `next`.  CHECKED: only the chunks
// below cnt, and only the fetches below cnt (the tail of a thread's run);
// otherwise the whole group and all its fetches are known to be in range.
// One 16-byte chunk of the unit [unit, unit + nv) into a ring slot; the
// bounds-checked build checks the address first.
__device__ __forceinline__ void stats_fetch(uint32_t dst, const uint4* at, const uint4* unit, int64_t nv,
                                            uint32_t* status) {
    if (in_bounds(at, 16, unit, nv * 16, status)) cp_async16(dst, at);
}

template <int DT, bool CHECKED>
__device__ __forceinline__ void stats_group(uint32_t ring, const uint4*& next, int k0, int cnt, unsigned long long& s1,
                                            unsigned long long& s2, unsigned long long& k2, float& K,
                                            const uint4* unit, int64_t nv, uint32_t* status) {
    constexpr uint32_t SLOT = STATS_BLOCK * 16u;
#pragma unroll
    for (int u = 0; u < STATS_GROUP; ++u) {
        if (!CHECKED || k0 + u < cnt) {
            if (!CHECKED || k0 + u + STATS_SLOTS - 1 < cnt)
                stats_fetch(ring + ((u + STATS_SLOTS - 1) % STATS_SLOTS) * SLOT, next, unit, nv, status);
            next += STATS_BLOCK;
            cp_async_commit();
            cp_async_wait<STATS_SLOTS - 1>();
            const uint4 v = lds16(ring + (u % STATS_SLOTS) * SLOT);
            if (u == 0) {
                K = GElt<DT>::to_f(v.x);
                const unsigned long long kb = __float_as_uint(K);
                k2 = kb | (kb << 32);
                s1 = 0;
                s2 = 0;
            }
            shifted_acc<DT>(v.x, k2, s1, s2);
            shifted_acc<DT>(v.y, k2, s1, s2);
            shifted_acc<DT>(v.z, k2, s1, s2);
            shifted_acc<DT>(v.w, k2, s1, s2);
        }
    }
}

template <int DT, bool VECTOR>
__global__ void __launch_bounds__(STATS_BLOCK) gn_stats_kernel(const __grid_constant__ GnStatsParams p) {
    constexpr int VEC = 16 / GElt<DT>::BYTES;
    extern __shared__ __align__(16) unsigned char s_ring[];  // STATS_SLOTS x STATS_BLOCK x 16 bytes
    __shared__ Stat s_warp[STATS_BLOCK / 32];

    const unsigned parts = (unsigned)p.parts;
    const unsigned unit = blockIdx.x / parts;
    const int rank = (int)(blockIdx.x - unit * parts);
    const unsigned NG = (unsigned)p.N * (unsigned)p.G;
    const unsigned pp = unit / NG;
    const unsigned rem = unit - pp * NG;
    const unsigned n = rem / (unsigned)p.G;
    const unsigned g = rem - n * (unsigned)p.G;
    const int64_t S = p.spatial[pp];
    const int64_t cg_ = p.C / p.G;
    const int64_t len = cg_ * S;
    const int64_t start = ((int64_t)n * p.C + (int64_t)g * cg_) * S;
    const char* base = reinterpret_cast<const char*>(p.patches[pp]) + start * GElt<DT>::BYTES;

    // parameters only above; the patches may be written by the preceding grid
    asm volatile("griddepcontrol.wait;" ::: "memory");

    Stat acc{0.f, 0.f, 0.f};
    if constexpr (VECTOR) {
        // len and start are multiples of VEC: whole 16-byte chunks.  Each
        // thread streams its chunks through its own ring of STATS_SLOTS
        // shared-memory slots with cp.async, STATS_SLOTS - 1 chunks ahead.
        const int64_t nv = len / VEC;
        const int64_t v0 = nv * rank / parts, v1 = nv * (rank + 1) / parts;
        const uint4* src = reinterpret_cast<const uint4*>(base);
        const int64_t first = v0 + threadIdx.x;
        const int cnt = first < v1 ? (int)((v1 - first + STATS_BLOCK - 1) / STATS_BLOCK) : 0;
        const uint32_t ring = (uint32_t)__cvta_generic_to_shared(s_ring) + threadIdx.x * 16u;
        constexpr uint32_t SLOT = STATS_BLOCK * 16u;
#pragma unroll
        for (int k = 0; k < STATS_SLOTS - 1; ++k) {
            if (k < cnt) stats_fetch(ring + k * SLOT, src + first + (int64_t)k * STATS_BLOCK, src, nv, p.status);
            cp_async_commit();
        }
        if constexpr (GElt<DT>::BYTES == 2) {
            // Groups of STATS_GROUP chunks: shifted sums about the group's
            // first element on packed fp32 pairs (3 packed operations per
            // element pair), then one Chan merge per group.
            // The loop runs one group per iteration, unrolled: a group starts
            // on ring slot 0, so every slot index is a constant, and the
            // address of the chunk fetched ahead steps by a constant.
            static_assert(STATS_GROUP % STATS_SLOTS == 0, "a group must start on ring slot 0");
            unsigned long long s1 = 0, s2 = 0, k2 = 0;
            float K = 0.f;
            const uint4* next = src + first + (int64_t)(STATS_SLOTS - 1) * STATS_BLOCK;  // chunk k + SLOTS - 1
            for (int k0 = 0; k0 < cnt; k0 += STATS_GROUP) {
                if (TB_GN_FAST_GROUPS && k0 + STATS_GROUP + STATS_SLOTS - 1 <= cnt) {
                    // a whole group whose fetches ahead are all in range: no checks
                    stats_group<DT, false>(ring, next, k0, cnt, s1, s2, k2, K, src, nv, p.status);
                    acc = chan_fast(acc, shifted_stat(s1, s2, K, (float)(STATS_GROUP * VEC)));
                    continue;
                }
                const int m = min(STATS_GROUP, cnt - k0);
                stats_group<DT, true>(ring, next, k0, cnt, s1, s2, k2, K, src, nv, p.status);
                // merging into the empty triple of the first group is exact
                acc = chan_fast(acc, shifted_stat(s1, s2, K, (float)(m * VEC)));
            }
        } else {
            for (int k = 0; k < cnt; ++k) {
                const int ahead = k + STATS_SLOTS - 1;
                if (ahead < cnt)
                    stats_fetch(ring + (ahead % STATS_SLOTS) * SLOT, src + first + (int64_t)ahead * STATS_BLOCK, src,
                                nv, p.status);
                cp_async_commit();
                cp_async_wait<STATS_SLOTS - 1>();
                float x[VEC];
                chunk_to_floats<DT>(lds16(ring + (k % STATS_SLOTS) * SLOT), x);
                acc = k == 0 ? block_stat<VEC>(x) : chan_fast(acc, block_stat<VEC>(x));
            }
        }
        cp_async_wait<0>();
    } else {
        const int64_t e0 = len * rank / parts, e1 = len * (rank + 1) / parts;
        for (int64_t e = e0 + threadIdx.x; e < e1; e += STATS_BLOCK) {
            if (!index_ok(e >= 0 && e < len, p.status)) continue;
            const float x = load_scalar<DT>(base, e);
            acc = chan(acc, Stat{1.f, x, 0.f});
        }
    }

    // warp, then CTA (fixed order); the part's record, and the empty records
    // of parts no CTA takes (records rank + j * parts, j >= 1: together the
    // CTAs of a unit write all TB_GN_PARTS of its records)
    acc = warp_reduce(acc);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) s_warp[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        Stat t = s_warp[0];
#pragma unroll
        for (int w = 1; w < STATS_BLOCK / 32; ++w) t = chan(t, s_warp[w]);
        int64_t count;
        if constexpr (VECTOR) {
            const int64_t nv = len / VEC;
            count = (nv * (rank + 1) / parts - nv * rank / parts) * VEC;
        } else {
            count = len * (rank + 1) / parts - len * rank / parts;
        }
        if (!index_ok(unit < (unsigned)p.P * NG && rank < TB_GN_PARTS, p.status)) return;
        GnPartial* const rec = p.partials + (int64_t)unit * TB_GN_PARTS;
        GnPartial out;
        out.n = count;
        out.mean = count > 0 ? t.mean : 0.f;
        out.m2 = count > 0 ? t.m2 : 0.f;
        rec[rank] = out;
        const GnPartial none = {0, 0.f, 0.f};
        for (int k = rank + (int)parts; k < TB_GN_PARTS; k += (int)parts) rec[k] = none;
    }
}

// Pooled (mean, rstd) of group g of sample n from the part records, computed
// by one warp.  `partials` holds R record sets of [N][G][TB_GN_PARTS] (the
// sets of one or more statistics calls, e.g. gathered from every rank), and
// every record describes itself: records with count 0 hold no elements and
// are skipped, whichever call wrote them and however it split its units.
// Each record (count c, mean m, M2) adds c, c * (m - K) and
// M2 + c * (m - K)^2 to three sums taken about K, the mean of the first
// record with elements (so the sums do not cancel); then
//     mean = K + S1 / n,   M2 = S2 - S1^2 / n   (Chan's combination, summed),
// and the variance is M2 / n, biased.  Counts are summed exactly in 64 bits
// and converted to fp32 once.  Lane 0 holds the result.
__device__ __forceinline__ void pooled_stats(const GnApplyParams& p, int64_t n, int64_t g, float& mean, float& rstd) {
    const int lane = threadIdx.x & 31;
    const int total = p.R * TB_GN_PARTS;
    const int64_t set_stride = p.N * p.G * TB_GN_PARTS;  // records between consecutive sets
    const GnPartial* const unit0 = p.partials + (n * p.G + g) * TB_GN_PARTS;
    auto record = [&](int q, long long& c, float& m, float& m2) {
        const int r = q / TB_GN_PARTS, k = q - r * TB_GN_PARTS;
        const GnPartial* const at = unit0 + r * set_stride + k;
        if (!in_bounds(at, sizeof(GnPartial), p.partials, (int64_t)p.R * set_stride * (int64_t)sizeof(GnPartial),
                       p.status)) {
            c = 0;
            m = m2 = 0.f;
            return;
        }
        const longlong2 raw = __ldg(reinterpret_cast<const longlong2*>(at));
        c = raw.x;
        m = __int_as_float((int)(raw.y & 0xffffffffLL));
        m2 = __int_as_float((int)(raw.y >> 32));
    };
    // the first 32 records stay in registers (all of them when R <= 4)
    long long c0 = 0;
    float m0 = 0.f, v0 = 0.f;
    if (lane < total) record(lane, c0, m0, v0);
    float K = 0.f;
    unsigned has = __ballot_sync(0xffffffffu, c0 > 0);
    if (has != 0u) {
        K = __shfl_sync(0xffffffffu, m0, __ffs(has) - 1);
    } else {
        for (int base = 32; base < total; base += 32) {
            long long c = 0;
            float m = 0.f, m2 = 0.f;
            if (base + lane < total) record(base + lane, c, m, m2);
            has = __ballot_sync(0xffffffffu, c > 0);
            if (has != 0u) {
                K = __shfl_sync(0xffffffffu, m, __ffs(has) - 1);
                break;
            }
        }
    }
    long long sn = 0;
    float s1 = 0.f, s2 = 0.f;
    auto add = [&](long long c, float m, float m2) {
        if (c > 0) {
            const float cf = (float)c;
            const float d = m - K;
            sn += c;
            s1 = fmaf(cf, d, s1);
            s2 += fmaf(cf * d, d, m2);
        }
    };
    add(c0, m0, v0);
    for (int q = lane + 32; q < total; q += 32) {
        long long c;
        float m, m2;
        record(q, c, m, m2);
        add(c, m, m2);
    }
#pragma unroll
    for (int delta = 16; delta >= 1; delta >>= 1) {  // fixed order: deterministic
        sn += __shfl_down_sync(0xffffffffu, sn, delta);
        s1 += __shfl_down_sync(0xffffffffu, s1, delta);
        s2 += __shfl_down_sync(0xffffffffu, s2, delta);
    }
    const float nf = (float)sn;
    const float q1 = sn > 0 ? s1 / nf : 0.f;
    const float var = sn > 0 ? fmaxf(0.f, fmaf(-s1, q1, s2) / nf) : 0.f;  // biased: divide by the count
    mean = K + q1;
    rstd = 1.0f / sqrtf(var + p.eps);
}

// (a, b) with y = x * a + b for channel c.
template <int DT>
__device__ __forceinline__ float2 channel_affine(const GnApplyParams& p, int64_t n, int64_t g, int64_t c);

template <int DT>
__device__ __forceinline__ float load_param(const void* ptr, int64_t c, float dflt) {
    if (ptr == nullptr) return dflt;
    if constexpr (GElt<DT>::BYTES == 4) {
        return __ldg(reinterpret_cast<const float*>(ptr) + c);
    } else {
        return GElt<DT>::to_f(__ldg(reinterpret_cast<const unsigned short*>(ptr) + c));
    }
}

template <int DT>
__device__ __forceinline__ float2 channel_affine(const GnApplyParams& p, int64_t n, int64_t g, int64_t c) {
    // every warp combines the records itself: a few loads and shuffles,
    // cheaper than a CTA barrier (measured)
    float mean, rstd;
    pooled_stats(p, n, g, mean, rstd);
    mean = __shfl_sync(0xffffffffu, mean, 0);
    rstd = __shfl_sync(0xffffffffu, rstd, 0);
    const bool c_ok = index_ok(c >= 0 && c < p.C, p.status);
    const float a = rstd * (c_ok ? load_param<DT>(p.gamma, c, 1.f) : 1.f);
    return make_float2(a, (c_ok ? load_param<DT>(p.beta, c, 0.f) : 0.f) - mean * a);
}

// silu(z) = z / (1 + e^-z), with e^-z = 2^(-z log2 e) and the reciprocal
// from the approximate special-function unit (relative errors ~2^-22, far
// inside the output tolerances).  Flushing subnormals there is harmless:
// e^-z is subnormal only for z > 87, where 1 + e^-z rounds to 1, and the
// reciprocal only for z < -87, where silu(z) lies below 1e-35.
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_ftz(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int SILU>
__device__ __forceinline__ float act(float x, float a, float b) {
    const float z = fmaf(x, a, b);
    if constexpr (SILU) {
        return z * rcp_ftz(1.0f + ex2_ftz(z * -1.4426950408889634f));
    } else {
        return z;
    }
}

// act() on a pair of elements: the fp32 operations in packed pairs
// (fma/mul/add.rn.f32x2 round each lane exactly as the scalar instructions
// do, so the results are the same bits), the special-function ops per lane.
#ifndef TB_GN_APPLY_PACKED
#define TB_GN_APPLY_PACKED 1
#endif
__device__ __forceinline__ unsigned long long pack2f(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2f(unsigned long long v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
template <int SILU>
__device__ __forceinline__ void act2(float& lo, float& hi, unsigned long long a2, unsigned long long b2) {
    if constexpr (!TB_GN_APPLY_PACKED) {
        float a, b, a1, b1;
        unpack2f(a2, a, a1);
        unpack2f(b2, b, b1);
        lo = act<SILU>(lo, a, b);
        hi = act<SILU>(hi, a1, b1);
        return;
    }
    unsigned long long z;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(z) : "l"(pack2f(lo, hi)), "l"(a2), "l"(b2));
    if constexpr (SILU) {
        unsigned long long t, d, y;
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(t) : "l"(z), "l"(pack2f(-1.4426950408889634f, -1.4426950408889634f)));
        float tl, th;
        unpack2f(t, tl, th);
        asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(pack2f(ex2_ftz(tl), ex2_ftz(th))), "l"(pack2f(1.0f, 1.0f)));
        float dl, dh;
        unpack2f(d, dl, dh);
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y) : "l"(z), "l"(pack2f(rcp_ftz(dl), rcp_ftz(dh))));
        z = y;
    }
    unpack2f(z, lo, hi);
}

template <int DT, bool VECTOR, int SILU>
__global__ void __launch_bounds__(APPLY_BLOCK) gn_apply_kernel(const __grid_constant__ GnApplyParams p) {
    constexpr int VEC = VECTOR ? 16 / GElt<DT>::BYTES : 1;
    const int64_t item = blockIdx.x;
    int pp = 0;
    while (pp + 1 < p.P && p.item_start[pp + 1] <= item) ++pp;
    // item counts, rows and channels fit 32 bits (the host checks the grid)
    const unsigned local = (unsigned)(item - p.item_start[pp]);
    const unsigned nseg = (unsigned)p.nseg[pp];
    const unsigned row = local / nseg;  // n * C + c
    const int64_t seg = local - row * nseg;
    const int64_t S = p.spatial[pp];
    const unsigned C32 = (unsigned)p.C;
    const int64_t c = row % C32;
    const int64_t n = row / C32;
    const int64_t g = (unsigned)c / (C32 / (unsigned)p.G);
    const int64_t e_begin = seg * p.seg;
    const int64_t e_end = min(S, e_begin + p.seg);
    const int64_t row_start = (int64_t)row * S;
    // parameters only above; patches and partials come from preceding grids
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // the patch's and its output's extent, for the bounds-checked build
    const int64_t pbytes = p.N * p.C * S * GElt<DT>::BYTES;
    if constexpr (VECTOR) {
        // S and every row start are multiples of VEC; issue the data loads first
        const uint4* src = reinterpret_cast<const uint4*>(p.patches[pp]) + (row_start + e_begin) / VEC;
        uint4* dst = reinterpret_cast<uint4*>(p.outs[pp]) + (row_start + e_begin) / VEC;
        const int nchunk = (int)((e_end - e_begin) / VEC);
        uint4 v[APPLY_CPT];
#pragma unroll
        for (int q = 0; q < APPLY_CPT; ++q) {
            const int idx = threadIdx.x + q * APPLY_BLOCK;
            if (idx < nchunk) {
                if (in_bounds(src + idx, 16, p.patches[pp], pbytes, p.status)) v[q] = __ldcs(src + idx);
                else v[q] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        const float2 ab = channel_affine<DT>(p, n, g, c);
        const unsigned long long a2 = pack2f(ab.x, ab.x), b2 = pack2f(ab.y, ab.y);
#pragma unroll
        for (int q = 0; q < APPLY_CPT; ++q) {
            const int idx = threadIdx.x + q * APPLY_BLOCK;
            if (idx >= nchunk) continue;
            uint4 o;
            if constexpr (GElt<DT>::BYTES == 4) {
                float x0 = __uint_as_float(v[q].x), x1 = __uint_as_float(v[q].y);
                float x2 = __uint_as_float(v[q].z), x3 = __uint_as_float(v[q].w);
                act2<SILU>(x0, x1, a2, b2);
                act2<SILU>(x2, x3, a2, b2);
                o = make_uint4(__float_as_uint(x0), __float_as_uint(x1), __float_as_uint(x2), __float_as_uint(x3));
            } else {
                uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float lo, hi;
                    GElt<DT>::unpack(w[k], lo, hi);
                    act2<SILU>(lo, hi, a2, b2);
                    w[k] = GElt<DT>::pack(lo, hi);
                }
                o = make_uint4(w[0], w[1], w[2], w[3]);
            }
            if (in_bounds(dst + idx, 16, p.outs[pp], pbytes, p.status)) __stcs(dst + idx, o);
        }
    } else {
        const float2 ab = channel_affine<DT>(p, n, g, c);
        const float a = ab.x, b = ab.y;
        const void* src = p.patches[pp];
        void* dst = p.outs[pp];
        for (int64_t e = e_begin + threadIdx.x; e < e_end; e += APPLY_BLOCK) {
            if (!index_ok(row_start + e >= 0 && (row_start + e) * GElt<DT>::BYTES < pbytes, p.status)) continue;
            const float y = act<SILU>(load_scalar<DT>(src, row_start + e), a, b);
            if constexpr (GElt<DT>::BYTES == 4) {
                __stcs(reinterpret_cast<float*>(dst) + row_start + e, y);
            } else {
                __stcs(reinterpret_cast<unsigned short*>(dst) + row_start + e,
                       (unsigned short)(GElt<DT>::pack(y, 0.f) & 0xffffu));
            }
        }
    }
}

template <int DT>
void (*stats_fn(bool aligned))(const GnStatsParams) {
    return aligned ? gn_stats_kernel<DT, true> : gn_stats_kernel<DT, false>;
}

size_t stats_smem(bool aligned) { return aligned ? (size_t)STATS_SLOTS * STATS_BLOCK * 16 : 0; }

template <int DT>
cudaError_t stats_dt(const GnStatsParams& p, int64_t units, cudaStream_t s) {
    void (*fn)(const GnStatsParams) = stats_fn<DT>(p.aligned != 0);
    if (stats_smem(p.aligned != 0) > 40 * 1024) {  // with the static shared memory, past the 48 KB default
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)stats_smem(p.aligned != 0));
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(units * p.parts), 1, 1);
    cfg.blockDim = dim3(STATS_BLOCK, 1, 1);
    cfg.dynamicSmemBytes = stats_smem(p.aligned != 0);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol.wait
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

template <int DT>
cudaError_t apply_dt(const GnApplyParams& p, int64_t items, cudaStream_t s) {
    void (*fn)(const GnApplyParams);
    if (p.aligned) {
        fn = p.silu ? gn_apply_kernel<DT, true, 1> : gn_apply_kernel<DT, true, 0>;
    } else {
        fn = p.silu ? gn_apply_kernel<DT, false, 1> : gn_apply_kernel<DT, false, 0>;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)items, 1, 1);
    cfg.blockDim = dim3(APPLY_BLOCK, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see griddepcontrol.wait
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace

int gn_apply_segment(int dtype, bool aligned) {
    const int bytes = dtype == F32 ? 4 : 2;
    return APPLY_BLOCK * (aligned ? APPLY_CPT * (16 / bytes) : APPLY_CPT);
}

cudaError_t launch_gn_stats(const GnStatsParams& p, int dtype, int64_t units, cudaStream_t s) {
    switch (dtype) {
        case F32: return stats_dt<F32>(p, units, s);
        case F16: return stats_dt<F16>(p, units, s);
        default: return stats_dt<BF16>(p, units, s);
    }
}

cudaError_t launch_gn_apply(const GnApplyParams& p, int dtype, int64_t items, cudaStream_t s) {
    switch (dtype) {
        case F32: return apply_dt<F32>(p, items, s);
        case F16: return apply_dt<F16>(p, items, s);
        default: return apply_dt<BF16>(p, items, s);
    }
}

}  // namespace tb
