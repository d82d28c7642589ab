// tb_internal.h -- structures shared by libtileblend's host layer and its
// CUDA kernels (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tb {

enum Dtype : int32_t { F32 = 0, F16 = 1, BF16 = 2 };

// ---------------------------------------------------------------------------
// Stitch
// ---------------------------------------------------------------------------

// Geometry of one grid axis as the kernel sees it.  Entries past `n` are 0.
template <int MAXA>
struct StitchAxis {
    int32_t n;               // tile count
    int32_t ext[MAXA];       // L(n): tile extent
    int32_t blend[MAXA];     // e(n): clamped blend extent against tile n-1 (e(0) = 0)
    int32_t coef[MAXA];      // first entry of e(n)'s coefficients in the table
    int32_t off[MAXA + 1];   // O(n): output offset of tile n's kept part; off[n] = output extent
};

// Everything a stitch launch needs, passed by value (__grid_constant__).
// Capacities come in two classes so that small grids launch with small
// parameter blocks.
template <int MAXA, int MAXT, int MAXC>
struct StitchParams {
    const void* tiles[MAXT];   // row-major over (k, i, j)
    void* out;                 // [planes, OT, OH, OW]
    int64_t planes;            // B * C
    int64_t nvrows;            // virtual rows = planes * OT * OH * nseg
    int32_t OT, OH, OW;        // output extents
    int32_t nseg;              // row segments per output row (width split across virtual rows)
    int32_t seg_chunks;        // chunks per segment (= XT * KX)
    int32_t xt;                // threads per virtual row
    int32_t rp;                // virtual rows per CTA pass (blockDim = xt * rp)
    int32_t ncoef;             // used entries of coef[]
    StitchAxis<MAXA> ax[3];    // t, y, x
    float2 coef[MAXC];         // (w, u) = ((float)(c/e), (float)(1 - c/e)) per distinct e, c < e
};

constexpr int SMALL_MAXA = 16, SMALL_MAXT = 256, SMALL_MAXC = 640;
constexpr int LARGE_MAXA = 64, LARGE_MAXT = 1024, LARGE_MAXC = 2048;

using StitchParamsSmall = StitchParams<SMALL_MAXA, SMALL_MAXT, SMALL_MAXC>;
using StitchParamsLarge = StitchParams<LARGE_MAXA, LARGE_MAXT, LARGE_MAXC>;

static_assert(sizeof(StitchParamsLarge) <= 32000, "kernel parameter block too large");

// Launch configuration picked by the host.
struct StitchLaunch {
    int ndim;       // 2 or 3
    int dtype;      // Dtype
    int vec;        // elements per chunk: 16 bytes / sizeof(dtype), or 1
    int kx;         // chunks per thread per virtual row
    int grid;       // CTAs
    int block;      // threads per CTA
};

// Implemented in tb_stitch.cu.
cudaError_t launch_stitch_small(const StitchParamsSmall& p, const StitchLaunch& l, cudaStream_t s);
cudaError_t launch_stitch_large(const StitchParamsLarge& p, const StitchLaunch& l, cudaStream_t s);
int stitch_kernel_max_ctas_per_sm(const StitchLaunch& l, bool large);

// ---------------------------------------------------------------------------
// PatchGroupNorm
// ---------------------------------------------------------------------------

constexpr int GN_MAXP = 64;

struct GnPartial {  // layout-identical to tb_gn_partial
    int64_t n;
    float mean;
    float m2;
};
static_assert(sizeof(GnPartial) == 16, "partial must be 16 bytes");

struct GnStatsParams {
    const void* patches[GN_MAXP];
    int64_t spatial[GN_MAXP];     // elements per channel in patch p
    GnPartial* partials;          // [P][N][G]
    int64_t N, C;
    int32_t P, G;
    int32_t cs;                   // CTAs per (p, n, g) unit (cluster size)
    int32_t aligned;              // every unit start and length is a multiple of the vector width
};

struct GnApplyParams {
    const void* patches[GN_MAXP];
    void* outs[GN_MAXP];
    int64_t spatial[GN_MAXP];
    int64_t item_start[GN_MAXP + 1];  // first work item of patch p (prefix sums)
    int64_t nseg[GN_MAXP];            // segments per channel row of patch p
    const GnPartial* partials;
    const void* gamma;                // [C] or null
    const void* beta;                 // [C] or null
    int64_t N, C;
    int32_t P, G;
    int32_t seg;                      // elements per segment
    float eps;
    int32_t silu;
    int32_t aligned;                  // every channel row start is 16-byte aligned
};

// Elements per apply work item (one CTA): depends on the element size and
// on whether the 16-byte vector path is taken.
int gn_apply_segment(int dtype, bool aligned);

// Records a CUDA error for tb_last_cuda_error() (defined in tb_host.cpp).
void record_cuda_error(cudaError_t e);

cudaError_t launch_gn_stats(const GnStatsParams& p, int dtype, int64_t units, cudaStream_t s);
cudaError_t launch_gn_apply(const GnApplyParams& p, int dtype, int64_t items, cudaStream_t s);

}  // namespace tb
