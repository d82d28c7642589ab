// tb_internal.h -- structures shared by libtileblend's host layer and its
// CUDA kernels (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "tileblend.h"

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
// Piece ranks the one-dimensional stitch grid can index (more: two-dimensional grid).
constexpr int STITCH_MAXR = 128;

template <int MAXA, int MAXT, int MAXC>
struct StitchParams {
    const void* tiles[MAXT];   // row-major over (k, i, j)
    void* out;                 // [planes, OT, OH, OW]
    int64_t planes;            // B * C
    int32_t OT, OH, OW;        // output extents
    uint32_t* status;          // device status word (bounds-checked build), or null
    int32_t ncoef;             // used entries of coef[]
    int32_t rows_per_thread;   // work per thread in a box piece (tuning)
    StitchAxis<MAXA> ax[3];    // t, y, x
    float2 coef[MAXC];         // (w, u) = ((float)(c/e), (float)(1 - c/e)) per distinct e, c < e
    // One-dimensional grid of the pieces that exist (nrank > 0): block b is
    // piece rank r of some (plane, tile) where rank_start[r] <= b <
    // rank_start[r + 1]; within rank r the blocks run over planes, and within
    // a plane over the first (rank_start[r + 1] - rank_start[r]) / planes
    // entries of tile_order (the tiles sorted by piece count, most first, so
    // the tiles with a piece of rank r come first).  nrank = 0: the grid is
    // (planes x tiles, pieces of the largest tile), blocks past a tile's
    // pieces exit at once.
    int32_t nrank;
    int32_t rank_start[STITCH_MAXR + 1];
    int16_t tile_order[MAXT];
};

constexpr int SMALL_MAXA = 16, SMALL_MAXT = 256, SMALL_MAXC = 640;
constexpr int LARGE_MAXA = 64, LARGE_MAXT = 1024, LARGE_MAXC = 2048;

using StitchParamsSmall = StitchParams<SMALL_MAXA, SMALL_MAXT, SMALL_MAXC>;
using StitchParamsLarge = StitchParams<LARGE_MAXA, LARGE_MAXT, LARGE_MAXC>;

static_assert(sizeof(StitchParamsLarge) <= 32000, "kernel parameter block too large");

constexpr int STITCH_BLOCK = 256;
// 16-byte staging slots per thread on the stitch's vector path (rows in
// flight x source nodes).
#ifndef TB_STITCH_SLOTS
#define TB_STITCH_SLOTS 8
#endif
constexpr int STITCH_SLOTS = TB_STITCH_SLOTS;

// The kept part of a tile splits into up to 2^d boxes by band membership:
// box b has bit 2 set if it lies in the tile's time band, bit 1 in its
// height band, bit 0 in its width band.  Inside a box every element is
// computed from the same set of source tiles.  `eb*` are the band extents
// clamped to the kept extents; widths are in chunks of `vec` elements.
struct BoxShape {
    int t0, nt, y0, ny, x0, width;
};

__host__ __device__ inline BoxShape box_shape(int b, int Kt, int Ky, int Kx, int ebt, int eby, int ebx, int vec) {
    BoxShape s;
    s.t0 = (b & 4) ? 0 : ebt;
    s.nt = (b & 4) ? ebt : Kt - ebt;
    s.y0 = (b & 2) ? 0 : eby;
    s.ny = (b & 2) ? eby : Ky - eby;
    s.x0 = (b & 1) ? 0 : ebx;
    const int nx = (b & 1) ? ebx : Kx - ebx;
    s.width = nx / vec;
    return s;
}

#ifndef TB_DEBUG_BOUNDS
#define TB_DEBUG_BOUNDS 0
#endif

#ifdef __CUDACC__
// The bounds-checked build (TB_DEBUG_BOUNDS=1) checks every computed address
// before it is read or written: true if the `bytes` at `addr` lie inside
// [base, base + size); otherwise the first such finding is recorded in the
// device status word (DEV_OUT_OF_BOUNDS, no trap) and the caller skips the
// access.  In the product build the check compiles away.
__device__ __forceinline__ bool in_bounds(const void* addr, int64_t bytes, const void* base, int64_t size,
                                          uint32_t* status) {
#if TB_DEBUG_BOUNDS
    const char* a = static_cast<const char*>(addr);
    const char* b = static_cast<const char*>(base);
    if (base != nullptr && a >= b && bytes >= 0 && a + bytes <= b + size) return true;
    if (status != nullptr) atomicCAS(status, 0u, 2u);
    return false;
#else
    (void)addr, (void)bytes, (void)base, (void)size, (void)status;
    return true;
#endif
}
// Records DEV_OUT_OF_BOUNDS when `ok` is false (bounds-checked build only).
__device__ __forceinline__ bool index_ok(bool ok, uint32_t* status) {
#if TB_DEBUG_BOUNDS
    if (!ok && status != nullptr) atomicCAS(status, 0u, 2u);
    return ok;
#else
    (void)status;
    return true;
#endif
}

// Every kernel is launched with programmatic stream serialisation and runs
// griddepcontrol.wait before its first global-memory access.  Triggering at
// the start of each CTA lets the next kernel in the stream launch as soon as
// every CTA of this grid has started (so it never takes a slot this grid
// still needs); its CTAs run their parameter-only prologue and then wait for
// this grid to complete and its writes to become visible.  Only the stitch
// triggers: its grids run many waves, and the next grid fills the SMs as the
// last wave drains (small stitches 12-18% faster back to back).  The
// GroupNorm statistics grid is one wave spread evenly over the SMs, and a
// grid placed early, while its predecessor drains, lands unevenly (measured
// up to 2x slower); so no kernel that may precede it in a sharded decode --
// the Patchify copy, the GroupNorm kernels themselves -- triggers, and the
// ramp stitch measured no gain from it.
#ifndef TB_PDL_TRIGGER
#define TB_PDL_TRIGGER 1
#endif
__device__ __forceinline__ void pdl_trigger_dependents() {
#if TB_PDL_TRIGGER
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}
#endif

// Thread layout of a CTA on a box `width` chunks wide: bdx threads across,
// bdy rows at a time, each thread covering cpt columns.
__host__ __device__ inline void box_layout(int width, int& bdx, int& bdy, int& cpt) {
    bdx = width < STITCH_BLOCK ? width : STITCH_BLOCK;
    if (bdx < 1) bdx = 1;
    bdy = STITCH_BLOCK / bdx;
    cpt = (width + bdx - 1) / bdx;
}

// Rows of box b one CTA processes (a "piece").  A box costs about one load
// and one blend more per element for every band it lies in, so heavier boxes
// get proportionally fewer rows per thread: pieces then take similar time.
__host__ __device__ inline int box_piece_rows(int b, int width, int rows_per_thread) {
    int bdx, bdy, cpt;
    box_layout(width, bdx, bdy, cpt);
    const int bands = (b & 1) + ((b >> 1) & 1) + ((b >> 2) & 1);
    const int per = (rows_per_thread >> bands) / cpt;
    return bdy * (per > 1 ? per : 1);
}

// Pieces of one tile: for every non-empty box, one piece per run of
// box_piece_rows() rows of its (frame, row) space flattened frame-major.  Boxes are enumerated from the most bands to
// the fewest, so the longest pieces are dispatched first.
__host__ __device__ inline int tile_pieces(int ndim, int Kt, int Ky, int Kx, int ebt, int eby, int ebx, int vec,
                                           int rows_per_thread) {
    int total = 0;
    const int nb = ndim == 3 ? 8 : 4;
    for (int b = nb - 1; b >= 0; --b) {
        const BoxShape s = box_shape(b, Kt, Ky, Kx, ebt, eby, ebx, vec);
        if (s.nt <= 0 || s.ny <= 0 || s.width <= 0) continue;
        const int R = box_piece_rows(b, s.width, rows_per_thread);
        total += (s.nt * s.ny + R - 1) / R;  // frames x rows, flattened
    }
    return total;
}

// Launch configuration picked by the host.
struct StitchLaunch {
    int ndim;       // 2 or 3
    int dtype;      // Dtype
    int vec;        // elements per chunk: 16 bytes / sizeof(dtype), or 1
    int grid_x;     // planes * tiles (tile fastest)
    int grid_y;     // pieces per tile (max over tiles)
    int grid_z;     // 1
    int smem;       // bytes of coefficient staging
};

// Implemented in tb_stitch.cu.
cudaError_t launch_stitch_small(const StitchParamsSmall& p, const StitchLaunch& l, cudaStream_t s);
cudaError_t launch_stitch_large(const StitchParamsLarge& p, const StitchLaunch& l, cudaStream_t s);

// ---------------------------------------------------------------------------
// Stitch, TMA path: each CTA stages every source rectangle of its piece into
// shared memory with tensor copies (one mbarrier, one memory latency), then
// evaluates the same closed form from shared memory.
// ---------------------------------------------------------------------------

constexpr int TMA_MAXT = 128;            // tiles (one tensor map each)
#ifndef TB_TMA_SMEM_BUDGET
#define TB_TMA_SMEM_BUDGET (64 * 1024)
#endif
constexpr int TMA_SMEM_BUDGET = TB_TMA_SMEM_BUDGET;

// A piece of box b (BoxShape s): one frame, `rb` rows, `wpc` chunks of
// columns.  Pieces are numbered column block fastest, then row block, then
// frame.
__host__ __device__ inline int tma_box_pieces(const BoxShape& s, int rb, int wpc) {
    return s.nt * ((s.ny + rb - 1) / rb) * ((s.width + wpc - 1) / wpc);
}

__host__ __device__ inline int tma_tile_pieces(int ndim, int Kt, int Ky, int Kx, int ebt, int eby, int ebx, int vec,
                                               int rb, int wpc) {
    int total = 0;
    const int nb = ndim == 3 ? 8 : 4;
    for (int b = nb - 1; b >= 0; --b) {
        const BoxShape s = box_shape(b, Kt, Ky, Kx, ebt, eby, ebx, vec);
        if (s.nt <= 0 || s.ny <= 0 || s.width <= 0) continue;
        total += tma_box_pieces(s, rb, wpc);
    }
    return total;
}

// Parameters of a TMA-path launch: one tensor map per source tile, viewing
// it as [planes][L_t][L_y][L_x] with a box of `wb` columns x `rb` rows, and
// the geometry of the ring path's parameters (their tile pointers unused).
struct alignas(128) StitchTmaParams {
    CUtensorMap maps[TMA_MAXT];
    StitchParamsSmall g;
    uint32_t* status;    // device status word (may be null)
    int32_t rb;          // rows per piece (= TMA box rows)
    int32_t wb;          // TMA box columns (elements)
    int32_t wpc;         // piece width in 16-byte chunks (a multiple of wb's)
    int32_t node_bytes;  // shared-memory bytes of one source rectangle
};
static_assert(sizeof(StitchTmaParams) <= 32000, "kernel parameter block too large");

cudaError_t launch_stitch_tma(const StitchTmaParams& p, const StitchLaunch& l, cudaStream_t s);

// Device status word: 0, or the first problem a kernel reported.
enum DeviceStatus : uint32_t { DEV_OK = 0, DEV_WAIT_TIMEOUT = 1, DEV_OUT_OF_BOUNDS = 2 };
static_assert(DEV_OK == TB_DEV_OK && DEV_WAIT_TIMEOUT == TB_DEV_WAIT_TIMEOUT &&
                  DEV_OUT_OF_BOUNDS == TB_DEV_OUT_OF_BOUNDS,
              "status codes differ from the header");
// Its device address in the current context (null if it cannot be looked up).
uint32_t* device_status_word();
// Process-unique id (+1) of the calling thread's current CUDA context; 0 if
// none is bound yet.  Device addresses of the library's static device arrays
// are cached per context id: a device reset replaces the context and module.
unsigned long long current_context_id();

// ---------------------------------------------------------------------------
// Normalised-ramp stitch
// ---------------------------------------------------------------------------

constexpr int RAMP_MAXA = 64;              // tiles per axis
constexpr int RAMP_MAXSEG = 2 * RAMP_MAXA + 1;
constexpr int RAMP_MAXCOVER = 3;           // tiles with positive weight at one position

// One axis as the ramp kernel sees it: the tiles, and the axis cut into
// segments over which the set of tiles with positive weight is constant.
struct RampAxisK {
    int32_t n, T, out, zero;
    float inv_ramp;
    int32_t org[RAMP_MAXA];
    int32_t nseg;
    int32_t seg_start[RAMP_MAXSEG];
    int32_t seg_len[RAMP_MAXSEG];
    int32_t seg_n[RAMP_MAXSEG];
    int8_t seg_tile[RAMP_MAXSEG][RAMP_MAXCOVER];
};

struct RampParams {
    const void* tiles[1024];
    void* out;
    uint32_t* status;   // device status word (bounds-checked build), or null
    int64_t planes;
    RampAxisK ay, ax;
    int32_t rows_per_piece[RAMP_MAXSEG];  // flattened (plane, row) rows per piece, by width segment
    // Rectangles in grid order grouped by (height cover, width cover): the
    // segments of each axis listed by cover count, and where each of the 9
    // groups starts among the grid's first coordinate.
    int16_t yseg[RAMP_MAXCOVER][RAMP_MAXSEG];
    int16_t xseg[RAMP_MAXCOVER][RAMP_MAXSEG];
    int32_t ycnt[RAMP_MAXCOVER], xcnt[RAMP_MAXCOVER];
    int32_t group_start[RAMP_MAXCOVER * RAMP_MAXCOVER + 1];
};
static_assert(sizeof(RampParams) <= 32000, "kernel parameter block too large");

int ramp_block();
int ramp_smem();
// Launches the rectangles of at most 2 x 2 tiles (grid_small of them) and,
// if any, those with 3 tiles along an axis (grid_large).
cudaError_t launch_ramp(const RampParams& p, int dtype, int vec, int grid_small, int grid_large, int grid_y,
                        cudaStream_t s);

// ---------------------------------------------------------------------------
// Patchify split / patch gather
// ---------------------------------------------------------------------------

constexpr int PF_MAXP = 64;
constexpr int PF_BLOCK = 256;          // threads per CTA
constexpr int PF_CTA_BYTES = 32768;    // bytes one CTA moves at most

// The whole tensor viewed as [outer, extent, inner]; patch p holds rows
// [start_p, start_p + size_p) of every outer slice.  All offsets below are
// in chunks of `vec` bytes (a power of two that divides every run, pitch,
// offset and base address).  Position (o, r) of patch p -- outer slice o,
// chunk r of its run -- is chunk o * ppitch[p] + r of the patch buffer and
// chunk o * wpitch + woff[p] + r of the whole tensor.
struct PatchCopyParams {
    void* patch[PF_MAXP];
    void* whole;
    int64_t n[PF_MAXP];        // chunks of patch p: outer * run[p]
    int64_t per_cta[PF_MAXP];  // chunks one CTA of patch p copies
    int64_t woff[PF_MAXP];     // run start inside an outer slice of the whole
    int64_t ppitch[PF_MAXP];   // chunks per outer slice of the patch buffer
    int32_t run[PF_MAXP];      // chunks per outer slice of band p (>= 1 if n > 0)
    int32_t step_o[PF_MAXP];   // PF_BLOCK / run[p]
    int32_t step_r[PF_MAXP];   // PF_BLOCK % run[p]
    int64_t wpitch;            // chunks per outer slice of the whole
    int64_t outer;             // outer slices
    uint32_t* status;          // device status word (bounds-checked build), or null
    int32_t P;
};
static_assert(sizeof(PatchCopyParams) <= 32000, "kernel parameter block too large");

// to_patches: whole -> patches (the split), else patches -> whole (the gather).
cudaError_t launch_patch_copy(const PatchCopyParams& p, int vec, bool to_patches, int64_t grid, cudaStream_t s);

// ---------------------------------------------------------------------------
// Row-sharded stitch: packing the band a rank sends to its successor
// ---------------------------------------------------------------------------

constexpr int HALO_MAXT = 512;      // tiles in one tile row (all frame tiles x width tiles)
constexpr int HALO_BLOCK = 256;

// Band q is the last `e` rows of every frame of every plane of source tile
// q, packed densely: [planes][frames_q][e][width_q] chunks at chunk dst_off[q]
// of the halo buffer.  Offsets and sizes are in chunks of the launch's width.
struct HaloPackParams {
    const void* src[HALO_MAXT];
    int64_t dst_off[HALO_MAXT];
    int64_t n[HALO_MAXT];          // chunks of band q
    int32_t rows[HALO_MAXT];       // rows per frame of source tile q
    int32_t width[HALO_MAXT];      // chunks per row of source tile q
    void* dst;
    int64_t per_cta;               // chunks one CTA copies
    int64_t dst_total;             // chunks of the whole halo buffer
    uint32_t* status;              // device status word (bounds-checked build), or null
    int32_t e;                     // band rows
    int32_t ntiles;
};
static_assert(sizeof(HaloPackParams) <= 32000, "kernel parameter block too large");

cudaError_t launch_halo_pack(const HaloPackParams& p, int vec_bytes, int64_t ranges, cudaStream_t s);

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

static_assert(TB_GN_PARTS >= 1 && TB_GN_PARTS <= 32 && (TB_GN_PARTS & (TB_GN_PARTS - 1)) == 0,
              "records per unit must be a power of two");

struct GnStatsParams {
    const void* patches[GN_MAXP];
    int64_t spatial[GN_MAXP];     // elements per channel in patch p
    GnPartial* partials;          // [P][N][G][TB_GN_PARTS]
    int64_t N, C;
    int32_t P, G;
    int32_t parts;                // CTAs per (p, n, g) unit: 1 .. TB_GN_PARTS
    int32_t aligned;              // every unit start and length is a multiple of the vector width
    uint32_t* status;             // bounds-checked build: device status word (else null)
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
    int32_t R;                        // record sets in `partials`: [R][N][G][TB_GN_PARTS]
    float eps;
    int32_t silu;
    int32_t aligned;                  // every channel row start is 16-byte aligned
    uint32_t* status;                 // bounds-checked build: device status word (else null)
};

// Elements per apply work item (one CTA): depends on the element size and
// on whether the 16-byte vector path is taken.
int gn_apply_segment(int dtype, bool aligned);

// Records a CUDA error for tb_last_cuda_error() (defined in tb_host.cpp).
void record_cuda_error(cudaError_t e);

cudaError_t launch_gn_stats(const GnStatsParams& p, int dtype, int64_t units, cudaStream_t s);
cudaError_t launch_gn_apply(const GnApplyParams& p, int dtype, int64_t items, cudaStream_t s);

}  // namespace tb
