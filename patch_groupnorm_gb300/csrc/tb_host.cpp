// tb_host.cpp -- libtileblend's C ABI: argument validation, tile-grid
// geometry, blend coefficient tables, launch configuration.
//
// Geometry follows the stock tiled decode (page "Studio: size seam-free VAE
// tiles from measured peaks", commit "Decode this VAE in 32-latent tiles
// ...": 256 px tiles with a 192 px stride and a 64 px blend at 16x; page
// "[Proposal] Vectorize tiled VAE blending ...", "Proposed scope": clamped
// blend extents):
//     stride = int(latent_tile * (1 - overlap))
//     origins = range(0, latent_extent, stride)
//     L(n) = min(latent_tile, latent_extent - origin) * scale
//     blend_extent = int(latent_tile * scale * overlap),  row_limit = tile - blend_extent
//     e(n) = min(L(n-1), L(n), blend_extent),  K(n) = min(L(n), row_limit)
// The blend coefficients are the Python-double quotients c/e and 1 - c/e
// narrowed to fp32 (the same page divides in float64 so that on-device
// coefficients equal Python's), computed here once per distinct e.
#include <algorithm>
#include <vector>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "tb_internal.h"
#include "tileblend.h"

#define TB_API extern "C" __attribute__((visibility("default")))

// Output rows per thread in one stitch work piece.
#ifndef TB_STITCH_ROWS_PER_THREAD
#define TB_STITCH_ROWS_PER_THREAD 16
#endif
#ifndef TB_STITCH_ROWS_PER_THREAD_3D
#define TB_STITCH_ROWS_PER_THREAD_3D 64
#endif
// Ramp stitch pieces: rows per thread start at the maximum and halve while
// the grid has fewer than this many pieces per SM.
#ifndef TB_RAMP_PIECES_PER_SM
#define TB_RAMP_PIECES_PER_SM 3
#endif
#ifndef TB_RAMP_MAX_ROWS_PER_THREAD
#define TB_RAMP_MAX_ROWS_PER_THREAD 16
#endif
// Stitch grid: 1 launches one block per existing piece (a one-dimensional
// grid, ranks in the kernel parameters), 0 the (planes x tiles, pieces of the
// largest tile) grid whose surplus blocks exit at once.
#ifndef TB_STITCH_FLAT_GRID
#define TB_STITCH_FLAT_GRID 1
#endif
// Stitch path for aligned grids of up to 128 tiles: 1 stages each piece's
// sources with tensor copies (TMA), 0 always streams them through the
// per-thread cp.async rings.
#ifndef TB_STITCH_TMA
#define TB_STITCH_TMA 0
#endif
// L2 promotion of the TMA path's copies (CUtensorMapL2promotion: 0 none,
// 1 64 B, 2 128 B, 3 256 B).
#ifndef TB_TMA_L2_PROMOTION
#define TB_TMA_L2_PROMOTION 3
#endif
// Rows of a TMA-path piece for 2-byte types (4-byte types take half).
#ifndef TB_STITCH_TMA_ROWS
#define TB_STITCH_TMA_ROWS 32
#endif
// Grids sized to one wave: a stitch small enough to run in a few waves takes
// the rows per thread that fill one wave of TB_STITCH_WAVE_CTAS CTAs per SM
// best; the GroupNorm statistics take the part count that fills one wave of
// TB_GN_WAVE_CTAS CTAs per SM best.  A lone launch then has no partial last
// wave.  0 keeps the fixed choices.
#ifndef TB_STITCH_WAVE_FIT
#define TB_STITCH_WAVE_FIT 0
#endif
#ifndef TB_STITCH_WAVE_CTAS
#define TB_STITCH_WAVE_CTAS 4
#endif
#ifndef TB_GN_WAVE_FIT
#define TB_GN_WAVE_FIT 0
#endif
#ifndef TB_GN_WAVE_CTAS
#define TB_GN_WAVE_CTAS 5
#endif
// CTAs per GroupNorm statistics unit (a power of two dividing TB_GN_PARTS);
// 0 picks it from the sizes and the SM count.
#ifndef TB_GN_FORCE_PARTS
#define TB_GN_FORCE_PARTS 0
#endif

static_assert(tb::RAMP_MAXCOVER == TB_RAMP_MAX_COVER, "ramp cover limit differs from the header");

namespace {

thread_local int g_last_cuda_error = 0;

tb_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return TB_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// geometry
// ---------------------------------------------------------------------------

struct Axis {
    int32_t n = 0;
    int64_t stride = 0;
    int32_t ext[TB_MAX_TILES_PER_AXIS] = {};
    int32_t blend[TB_MAX_TILES_PER_AXIS] = {};
    int32_t kept[TB_MAX_TILES_PER_AXIS] = {};
    int32_t blend_extent = 0;
    int32_t row_limit = 0;
    int64_t out = 0;
};

// Validates `a` and derives its grid.  *n_total receives the tile count even
// when it exceeds TB_MAX_TILES_PER_AXIS (then TB_ERR_UNSUPPORTED).
tb_status derive_axis(const tb_axis* a, Axis& g, int64_t* n_total) {
    if (a == nullptr) return TB_ERR_NULL;
    if (a->latent_extent < 0 || a->latent_tile < 1 || a->scale < 1) return TB_ERR_GEOMETRY;
    if (!(a->overlap >= 0.0 && a->overlap < 1.0)) return TB_ERR_GEOMETRY;
    const double tile_px = (double)a->latent_tile * (double)a->scale;
    if (tile_px > 2147483647.0) return TB_ERR_GEOMETRY;
    const int64_t stride = (int64_t)((double)a->latent_tile * (1.0 - a->overlap));
    if (stride < 1) return TB_ERR_GEOMETRY;
    const int64_t be = a->blend_extent < 0 ? (int64_t)((double)((int64_t)a->latent_tile * a->scale) * a->overlap)
                                           : (int64_t)a->blend_extent;
    const int64_t rl = a->row_limit <= 0 ? (int64_t)a->latent_tile * a->scale - be : (int64_t)a->row_limit;
    if (rl < 1 || be > 2147483647LL || rl > 2147483647LL) return TB_ERR_GEOMETRY;
    const int64_t n = a->latent_extent == 0 ? 0 : ((int64_t)a->latent_extent + stride - 1) / stride;
    if (n_total) *n_total = n;
    if (n > TB_MAX_TILES_PER_AXIS) return TB_ERR_UNSUPPORTED;
    g.n = (int32_t)n;
    g.stride = stride;
    g.blend_extent = (int32_t)be;
    g.row_limit = (int32_t)rl;
    g.out = 0;
    for (int64_t k = 0; k < n; ++k) {
        const int64_t origin = k * stride;
        const int64_t lat = std::min<int64_t>(a->latent_tile, a->latent_extent - origin);
        const int64_t L = lat * a->scale;
        if (L > 2147483647LL) return TB_ERR_GEOMETRY;
        g.ext[k] = (int32_t)L;
        g.blend[k] = k == 0 ? 0 : (int32_t)std::min<int64_t>(std::min<int64_t>(g.ext[k - 1], L), be);
        g.kept[k] = (int32_t)std::min<int64_t>(L, rl);
        g.out += g.kept[k];
    }
    if (g.out > 2147483647LL) return TB_ERR_GEOMETRY;
    return TB_OK;
}

// Bands that reach each other (a middle tile's lent rows rewritten by its
// own band) fall outside the closed form the kernels evaluate.
bool bands_apart(const Axis& g) {
    for (int k = 1; k + 1 < g.n; ++k)
        if ((int64_t)g.ext[k] < (int64_t)g.blend[k] + g.blend[k + 1]) return false;
    return true;
}

// ---------------------------------------------------------------------------
// device facts, cached per device (no allocation)
// ---------------------------------------------------------------------------

constexpr int MAX_DEVICES = 64;
std::atomic<int> g_sm_count[MAX_DEVICES] = {};  // 0: not looked up yet

tb_status device_sms(int* sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev >= 0 && dev < MAX_DEVICES) {
        const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
        if (cached > 0) {
            *sms = cached;
            return TB_OK;
        }
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev >= 0 && dev < MAX_DEVICES) g_sm_count[dev].store(n, std::memory_order_relaxed);
    *sms = n;
    return TB_OK;
}

int elem_bytes(tb_dtype d) { return d == TB_F32 ? 4 : 2; }

// The status word the bounds-checked build's kernels report to (null in the
// product build, whose kernels make no checks).
uint32_t* debug_status() {
#if TB_DEBUG_BOUNDS
    return tb::device_status_word();
#else
    return nullptr;
#endif
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// ---------------------------------------------------------------------------
// stitch
// ---------------------------------------------------------------------------

// ---------------------------------------------------------------------------
// stitch, TMA path
// ---------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, reached through the runtime (no driver
// library is linked); null if unavailable.
EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Tile shape of the TMA path: `rb` rows per piece (= TMA box rows), TMA box
// `wbc` chunks wide, pieces at most `wpc` chunks wide, and the shared memory
// the widest piece's sources take.
struct TmaShape {
    int rb = 0, wbc = 0, wpc = 0;
    int64_t smem = 0;
};

// Picks the TMA tile shape for the grid's boxes: the cheapest by a rough cost
// (bytes staged, including rows and columns read past a box's edge, plus a
// per-copy and a per-CTA charge) among shapes whose pieces fit the shared
// memory budget.  False if no shape fits.
bool pick_tma_shape(const Axis (&g)[3], int ndim, int vec, int eb, TmaShape& out) {
    struct Box {
        int nodes, nt, ny, w;
    };
    Box boxes[4 * 8 * 8];  // distinct box shapes suffice for the cost; cap below
    int nbx = 0;
    int64_t weight[4 * 8 * 8];
    for (int k = 0; k < g[0].n; ++k)
        for (int i = 0; i < g[1].n; ++i)
            for (int j = 0; j < g[2].n; ++j) {
                const int ebt = (ndim == 3 && k > 0) ? std::min(g[0].blend[k], g[0].kept[k]) : 0;
                const int eby = i > 0 ? std::min(g[1].blend[i], g[1].kept[i]) : 0;
                const int ebx = j > 0 ? std::min(g[2].blend[j], g[2].kept[j]) : 0;
                for (int b = (ndim == 3 ? 7 : 3); b >= 0; --b) {
                    const tb::BoxShape sh = tb::box_shape(b, g[0].kept[k], g[1].kept[i], g[2].kept[j], ebt, eby,
                                                          ebx, vec);
                    if (sh.nt <= 0 || sh.ny <= 0 || sh.width <= 0) continue;
                    const Box bx{1 << ((b & 1) + ((b >> 1) & 1) + ((b >> 2) & 1)), sh.nt, sh.ny, sh.width};
                    int f = 0;
                    while (f < nbx && !(boxes[f].nodes == bx.nodes && boxes[f].nt == bx.nt &&
                                        boxes[f].ny == bx.ny && boxes[f].w == bx.w))
                        ++f;
                    if (f == nbx) {
                        if (nbx == (int)(sizeof(boxes) / sizeof(boxes[0]))) return false;
                        boxes[nbx] = bx;
                        weight[nbx] = 0;
                        ++nbx;
                    }
                    ++weight[f];
                }
            }
    const int base_rows = std::max(8, TB_STITCH_TMA_ROWS * 2 / eb);
    const int rows_c[] = {base_rows, base_rows / 2, base_rows * 3 / 4, base_rows * 5 / 4, base_rows * 3 / 2};
    const int max_wbc = 256 * eb / 16;  // a TMA box is at most 256 elements wide
    bool found = false;
    double best = 0.0;
    for (int rb : rows_c) {
        if (rb < 8 || rb % 8 != 0 || rb > 256) continue;
        for (int wbc = std::max(1, 64 / 16); wbc <= max_wbc; ++wbc) {  // boxes of at least 64 bytes per row
            int maxw = 0;
            for (int f = 0; f < nbx; ++f) maxw = std::max(maxw, boxes[f].w);
            // widest piece (a multiple of the box width) whose sources fit
            int wpc = ((maxw + wbc - 1) / wbc) * wbc;
            int64_t smem = 0;
            while (wpc >= wbc) {
                smem = 0;
                for (int f = 0; f < nbx; ++f) {
                    const int wp = std::min(boxes[f].w, wpc);
                    smem = std::max<int64_t>(smem, (int64_t)boxes[f].nodes * rb * ((wp + wbc - 1) / wbc) * wbc * 16);
                }
                if (smem <= tb::TMA_SMEM_BUDGET) break;
                wpc -= wbc;
            }
            if (wpc < wbc) continue;
            double cost = 0.0;
            for (int f = 0; f < nbx; ++f) {
                const Box& bx = boxes[f];
                const int64_t rblk = (bx.ny + rb - 1) / rb, cblk = (bx.w + wpc - 1) / wpc;
                const int64_t pieces = (int64_t)bx.nt * rblk * cblk;
                int64_t copies = 0, staged = 0;
                for (int64_t c = 0; c < cblk; ++c) {
                    const int wp = (int)std::min<int64_t>(wpc, bx.w - c * wpc);
                    const int nb = (wp + wbc - 1) / wbc;
                    copies += nb;
                    staged += (int64_t)nb * wbc * 16 * rb;
                }
                cost += (double)weight[f] * bx.nt * rblk * bx.nodes * (staged + 512.0 * copies) +
                        (double)weight[f] * pieces * 8192.0;
            }
            if (!found || cost < best) {
                found = true;
                best = cost;
                out.rb = rb;
                out.wbc = wbc;
                out.wpc = wpc;
                out.smem = smem;
            }
        }
    }
    return found;
}

// Launches the TMA path for an aligned grid; *launched stays false when the
// grid does not suit it (then the ring path runs).
tb_status try_launch_tma(const tb::StitchParamsSmall& prm, const Axis (&g)[3], int ndim, tb_dtype dtype, int vec,
                         int64_t planes, const void* const* tiles, cudaStream_t stream, bool* launched) {
    *launched = false;
    const int ntiles = g[0].n * g[1].n * g[2].n;
    if (!TB_STITCH_TMA || vec == 1 || ntiles > tb::TMA_MAXT) return TB_OK;
    if (planes > 2147483647LL) return TB_OK;
    EncodeTiledFn encode = encode_tiled();
    if (encode == nullptr) return TB_OK;
    const int eb = elem_bytes(dtype);
    TmaShape sh;
    if (!pick_tma_shape(g, ndim, vec, eb, sh)) return TB_OK;
    static thread_local tb::StitchTmaParams tp;  // 24 KB: kept off the stack
    std::memset(&tp, 0, sizeof(tp));
    tp.g = prm;
    tp.rb = sh.rb;
    tp.wb = sh.wbc * vec;
    tp.wpc = sh.wpc;
    tp.status = tb::device_status_word();
    const CUtensorMapDataType dt = dtype == TB_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dtype == TB_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    int max_pieces = 0;
    for (int k = 0; k < g[0].n; ++k)
        for (int i = 0; i < g[1].n; ++i)
            for (int j = 0; j < g[2].n; ++j) {
                const int q = (k * g[1].n + i) * g[2].n + j;
                const cuuint64_t dims[4] = {(cuuint64_t)g[2].ext[j], (cuuint64_t)g[1].ext[i],
                                            (cuuint64_t)g[0].ext[k], (cuuint64_t)planes};
                const cuuint64_t strides[3] = {(cuuint64_t)g[2].ext[j] * eb, (cuuint64_t)g[1].ext[i] * g[2].ext[j] * eb,
                                               (cuuint64_t)g[0].ext[k] * g[1].ext[i] * g[2].ext[j] * eb};
                const cuuint32_t box[4] = {(cuuint32_t)tp.wb, (cuuint32_t)tp.rb, 1, 1};
                const cuuint32_t estr[4] = {1, 1, 1, 1};
                if (encode(&tp.maps[q], dt, 4, const_cast<void*>(tiles[q]), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           (CUtensorMapL2promotion)TB_TMA_L2_PROMOTION, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
                    CUDA_SUCCESS)
                    return TB_OK;
                const int ebt = (ndim == 3 && k > 0) ? std::min(g[0].blend[k], g[0].kept[k]) : 0;
                const int eby = i > 0 ? std::min(g[1].blend[i], g[1].kept[i]) : 0;
                const int ebx = j > 0 ? std::min(g[2].blend[j], g[2].kept[j]) : 0;
                max_pieces = std::max(max_pieces, tb::tma_tile_pieces(ndim, g[0].kept[k], g[1].kept[i],
                                                                      g[2].kept[j], ebt, eby, ebx, vec, sh.rb,
                                                                      sh.wpc));
            }
    if (max_pieces == 0 || max_pieces > 65535 || (int64_t)ntiles * planes > 2147483647LL) return TB_OK;
    int max_ebx = 0, max_eby = 0, max_ebt = 0;
    for (int j = 1; j < g[2].n; ++j) max_ebx = std::max(max_ebx, std::min(g[2].blend[j], g[2].kept[j]));
    for (int i = 1; i < g[1].n; ++i) max_eby = std::max(max_eby, std::min(g[1].blend[i], g[1].kept[i]));
    for (int k = 1; ndim == 3 && k < g[0].n; ++k) max_ebt = std::max(max_ebt, std::min(g[0].blend[k], g[0].kept[k]));
    const int64_t coef = (int64_t)(2 * (max_ebx + max_eby + max_ebt)) * 4;
#ifdef TB_TMA_SMEM_CAP
    if (sh.smem > TB_TMA_SMEM_CAP) return TB_OK;
#endif
    tb::StitchLaunch l{};
    l.ndim = ndim;
    l.dtype = (int)dtype;
    l.vec = vec;
    l.grid_x = (int)(ntiles * planes);
    l.grid_y = max_pieces;
    l.grid_z = 1;
    const int64_t smem = 128 + 128 + ((coef + 127) / 128) * 128 + sh.smem;  // alignment slack, mbarrier
    if (smem > 200 * 1024) return TB_OK;
    l.smem = (int)smem;
    cudaError_t e = tb::launch_stitch_tma(tp, l, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    *launched = true;
    return TB_OK;
}

template <class P>
tb_status fill_and_launch(P& prm, const Axis (&g)[3], int ndim, tb_dtype dtype, int64_t planes,
                          const void* const* tiles, void* out, cudaStream_t stream, bool large) {
    constexpr int MAXA = sizeof(prm.ax[0].ext) / sizeof(int32_t);
    constexpr int MAXC = sizeof(prm.coef) / sizeof(float2);
    std::memset(&prm, 0, sizeof(prm));
    // coefficient tables, one per distinct clamped blend extent
    int32_t distinct_e[3 * TB_MAX_TILES_PER_AXIS];
    int32_t distinct_off[3 * TB_MAX_TILES_PER_AXIS];
    int nd = 0, ncoef = 0;
    for (int a = 0; a < 3; ++a) {
        auto& ax = prm.ax[a];
        ax.n = g[a].n;
        int32_t acc = 0;
        for (int k = 0; k < g[a].n; ++k) {
            ax.ext[k] = g[a].ext[k];
            ax.blend[k] = g[a].blend[k];
            ax.off[k] = acc;
            acc += g[a].kept[k];
            const int32_t e = g[a].blend[k];
            ax.coef[k] = 0;
            if (e <= 0) continue;
            int f = 0;
            while (f < nd && distinct_e[f] != e) ++f;
            if (f == nd) {
                if (ncoef + e > MAXC) return TB_ERR_UNSUPPORTED;
                distinct_e[nd] = e;
                distinct_off[nd] = ncoef;
                for (int32_t c = 0; c < e; ++c) {
                    const double q = (double)c / (double)e;
                    prm.coef[ncoef + c] = make_float2((float)q, (float)(1.0 - (double)c / (double)e));
                }
                ncoef += e;
                ++nd;
            }
            ax.coef[k] = distinct_off[f];
        }
        ax.off[g[a].n] = acc;
    }
    (void)MAXA;
    prm.ncoef = ncoef;
    const int ntiles = g[0].n * g[1].n * g[2].n;
    for (int q = 0; q < ntiles; ++q) prm.tiles[q] = tiles[q];
    prm.out = out;
    prm.status = debug_status();
    prm.planes = planes;
    prm.OT = (int32_t)g[0].out;
    prm.OH = (int32_t)g[1].out;
    prm.OW = (int32_t)g[2].out;

    // 16-byte chunks where the width geometry and every pointer allow it
    const int eb = elem_bytes(dtype);
    int vec = 16 / eb;
    bool ok = (prm.OW % vec == 0) && aligned16(out);
    for (int k = 0; ok && k < g[2].n; ++k)
        ok = g[2].ext[k] % vec == 0 && g[2].kept[k] % vec == 0 && g[2].blend[k] % vec == 0;
    for (int q = 0; ok && q < ntiles; ++q) ok = aligned16(tiles[q]);
    if (!ok) vec = 1;

    tb::StitchLaunch l{};
    l.ndim = ndim;
    l.dtype = (int)dtype;
    l.vec = vec;
    // Pieces per tile; the grid's second extent is the largest count.
    int rpt = ndim == 3 ? TB_STITCH_ROWS_PER_THREAD_3D : TB_STITCH_ROWS_PER_THREAD;
    std::vector<int> np(ntiles);  // pieces of tile (k, i, j), row-major, for the last count
    auto count = [&](int r, int& max_p, int64_t& total) {
        max_p = 0;
        total = 0;
        for (int k = 0; k < g[0].n; ++k)
            for (int i = 0; i < g[1].n; ++i)
                for (int j = 0; j < g[2].n; ++j) {
                    const int ebt = (ndim == 3 && k > 0) ? std::min(g[0].blend[k], g[0].kept[k]) : 0;
                    const int eby = i > 0 ? std::min(g[1].blend[i], g[1].kept[i]) : 0;
                    const int ebx = j > 0 ? std::min(g[2].blend[j], g[2].kept[j]) : 0;
                    const int n = tb::tile_pieces(ndim, g[0].kept[k], g[1].kept[i], g[2].kept[j], ebt, eby, ebx,
                                                  vec, r);
                    np[(k * g[1].n + i) * g[2].n + j] = n;
                    max_p = std::max(max_p, n);
                    total += n;
                }
        total *= planes;
    };
    int max_pieces = 0;
    int64_t total_pieces = 0;
    count(rpt, max_pieces, total_pieces);
    if (TB_STITCH_WAVE_FIT && ndim == 2) {
        int sms = 0;
        if (device_sms(&sms) == TB_OK && sms > 0) {
            const int64_t wave = (int64_t)sms * TB_STITCH_WAVE_CTAS;
            if (total_pieces < 3 * wave) {
                // the rows per thread whose piece count comes closest to one
                // wave without passing it
                int best = rpt;
                int64_t best_n = total_pieces <= wave ? total_pieces : -1;
                for (int r = 8; r <= 40; r += 2) {
                    int mp = 0;
                    int64_t n = 0;
                    count(r, mp, n);
                    if (n <= wave && n > best_n) {
                        best = r;
                        best_n = n;
                    }
                }
                rpt = best;
                count(rpt, max_pieces, total_pieces);  // the counts (and np) of the chosen rows
            }
        }
    }
    int max_ebx = 0, max_eby = 0;
    for (int j = 1; j < g[2].n; ++j) max_ebx = std::max(max_ebx, std::min(g[2].blend[j], g[2].kept[j]));
    for (int i = 1; i < g[1].n; ++i) max_eby = std::max(max_eby, std::min(g[1].blend[i], g[1].kept[i]));
    prm.rows_per_thread = rpt;
    if (max_pieces == 0) return TB_OK;
    if ((int64_t)ntiles * planes > 2147483647LL || max_pieces > 65535) return TB_ERR_UNSUPPORTED;
    l.grid_x = (int)(ntiles * planes);
    l.grid_y = max_pieces;
    l.grid_z = 1;
    // One block per existing piece where the two-dimensional grid would not
    // fit the GPU at once: there its blocks without a piece hold slots that
    // real pieces wait for (the wide 1600 x 2048 image, 900 blocks: 13.0 µs
    // two-dimensional, 12.1 µs one-dimensional, one launch under ncu).
    // Within one resident wave every block starts at once and the
    // two-dimensional order measured faster (1024² fp32, 432 blocks: 8.6 µs
    // against 9.2 µs).  The ranks must fit the table.  Order: the tiles
    // sorted by piece count (most first, ties in tile order), and for every
    // rank r the blocks of the tiles with more than r pieces, plane by plane.
    prm.nrank = 0;
    int sms_now = 0;
    const bool over_a_wave = device_sms(&sms_now) == TB_OK &&
                             (int64_t)ntiles * planes * max_pieces > (int64_t)sms_now * (ndim == 3 ? 3 : 4);
    if (TB_STITCH_FLAT_GRID && over_a_wave && max_pieces <= tb::STITCH_MAXR && total_pieces <= 2147483647LL) {
        std::vector<int> order(ntiles);
        for (int t = 0; t < ntiles; ++t) order[t] = t;
        std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return np[a] > np[b]; });
        for (int t = 0; t < ntiles; ++t) prm.tile_order[t] = (int16_t)order[t];
        int64_t start = 0;
        int tiles_left = ntiles;
        for (int r = 0; r < max_pieces; ++r) {
            while (tiles_left > 0 && np[order[tiles_left - 1]] <= r) --tiles_left;
            prm.rank_start[r] = (int32_t)start;
            start += (int64_t)tiles_left * planes;
        }
        prm.rank_start[max_pieces] = (int32_t)start;
        if (start != total_pieces) return TB_ERR_UNSUPPORTED;  // the two counts must agree
        prm.nrank = max_pieces;
        l.grid_x = (int)start;
        l.grid_y = 1;
    }
    // vector path: STITCH_SLOTS staging slots of 16 bytes per thread, then coefficients
    int max_ebt = 0;
    for (int k = 1; ndim == 3 && k < g[0].n; ++k) max_ebt = std::max(max_ebt, std::min(g[0].blend[k], g[0].kept[k]));
    l.smem = (vec > 1 ? tb::STITCH_SLOTS * tb::STITCH_BLOCK * 16 : 0) +
             (int)(sizeof(float) * 2 * (size_t)(max_ebx + max_eby + max_ebt));
    // byte pitches of a frame of any tile and of the output fit 32 bits
    for (int i = 0; i < g[1].n; ++i)
        for (int j = 0; j < g[2].n; ++j)
            if ((int64_t)g[1].ext[i] * g[2].ext[j] * eb > 2147483647LL) return TB_ERR_UNSUPPORTED;
    if ((int64_t)prm.OH * prm.OW * eb > 2147483647LL) return TB_ERR_UNSUPPORTED;
    if (l.smem > 200 * 1024) return TB_ERR_UNSUPPORTED;
    (void)large;

    cudaError_t e;
    if constexpr (sizeof(P) == sizeof(tb::StitchParamsLarge)) {
        e = tb::launch_stitch_large(prm, l, stream);
    } else {
        bool launched = false;
        tb_status st = try_launch_tma(prm, g, ndim, dtype, vec, planes, tiles, stream, &launched);
        if (st != TB_OK || launched) return st;
        e = tb::launch_stitch_small(prm, l, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return TB_OK;
}

// Tile rows (axis 1, height) or frame tiles (axis 0, time) [begin, end),
// stitched by one rank of a sharded stitch; `halo` holds the packed band of
// tile begin - 1 along that axis.
struct Shard {
    int axis;
    int32_t row_begin, row_end;
    const void* halo;
};

// The local height axis of a shard: its tile rows, preceded (when its first
// row blends with the row above) by a halo row of extent e_y(row_begin) that
// holds exactly the rows of the row above that the band reads, keeps nothing
// and blends with nothing.  With that extent the kernel's neighbour row
// L(n-1) - e(n) + c is band row c, and the plane pitch is the band's.
bool shard_axis(const Axis& g, int32_t row_begin, int32_t row_end, Axis& l, bool* halo) {
    if (row_begin < 0 || row_end < row_begin || row_end > g.n) return false;
    *halo = row_begin > 0 && row_end > row_begin && g.blend[row_begin] > 0;
    l = Axis{};
    l.stride = g.stride;
    l.blend_extent = g.blend_extent;
    l.row_limit = g.row_limit;
    int n = 0;
    if (*halo) {
        l.ext[n] = g.blend[row_begin];
        l.blend[n] = 0;
        l.kept[n] = 0;
        ++n;
    }
    for (int i = row_begin; i < row_end; ++i, ++n) {
        l.ext[n] = g.ext[i];
        l.blend[n] = (n == 0) ? 0 : g.blend[i];
        l.kept[n] = g.kept[i];
        l.out += g.kept[i];
    }
    l.n = n;
    return true;
}

tb_status stitch_common(int ndim, const void* const* tiles, tb_dtype dtype, int64_t B, int64_t C,
                        const tb_axis* at, const tb_axis* ay, const tb_axis* ax, void* out, int64_t out_t,
                        int64_t out_h, int64_t out_w, void* stream, const Shard* shard = nullptr) {
    if (dtype != TB_F32 && dtype != TB_F16 && dtype != TB_BF16) return TB_ERR_DTYPE;
    if (B < 0 || C < 0 || out_t < 0 || out_h < 0 || out_w < 0) return TB_ERR_SHAPE;
    if (B > 0 && C > INT64_MAX / B) return TB_ERR_SHAPE;
    Axis g[3];
    int64_t ntot = 0;
    if (ndim == 3) {
        tb_status s = derive_axis(at, g[0], &ntot);
        if (s != TB_OK) return s;
    } else {
        g[0].n = 1;
        g[0].ext[0] = 1;
        g[0].kept[0] = 1;
        g[0].blend[0] = 0;
        g[0].out = 1;
    }
    tb_status s = derive_axis(ay, g[1], &ntot);
    if (s != TB_OK) return s;
    s = derive_axis(ax, g[2], &ntot);
    if (s != TB_OK) return s;
    for (int a = 0; a < 3; ++a)
        if (!bands_apart(g[a])) return TB_ERR_UNSUPPORTED;
    // a shard stitches its own tile rows, with the band of the row above as
    // a halo row that is read but not written
    bool halo = false;
    const void* table[TB_MAX_TILES];
    if (shard != nullptr) {
        const int A = shard->axis;  // 0: frame tiles, 1: tile rows
        Axis l;
        if (!shard_axis(g[A], shard->row_begin, shard->row_end, l, &halo)) return TB_ERR_SHAPE;
        const int32_t in = shard->row_end - shard->row_begin;
        const int h = halo ? 1 : 0;
        const int nt = A == 0 ? in + h : g[0].n, ny = A == 1 ? in + h : g[1].n;
        if ((int64_t)nt * ny * g[2].n > TB_MAX_TILES) return TB_ERR_UNSUPPORTED;
        if (halo && shard->halo == nullptr && B * C > 0) return TB_ERR_NULL;
        if (tiles == nullptr && in > 0 && B * C > 0) return TB_ERR_NULL;
        const int eb = elem_bytes(dtype);
        const char* hp = reinterpret_cast<const char*>(shard->halo);
        const int ny_in = A == 1 ? in : g[1].n;  // rows of the caller's own tiles
        int q = 0;
        for (int k = 0; k < nt; ++k)
            for (int i = 0; i < ny; ++i)
                for (int j = 0; j < g[2].n; ++j) {
                    if (halo && ((A == 0 && k == 0) || (A == 1 && i == 0))) {
                        // the halo tiles lie in the band in the order visited here
                        table[q++] = hp;
                        const int64_t lt = A == 0 ? l.ext[0] : g[0].ext[k];
                        const int64_t ly = A == 1 ? l.ext[0] : g[1].ext[i];
                        hp += B * C * lt * ly * g[2].ext[j] * eb;
                    } else {
                        const int kin = A == 0 ? k - h : k, iin = A == 1 ? i - h : i;
                        table[q++] = tiles[((int64_t)kin * ny_in + iin) * g[2].n + j];
                    }
                }
        g[A] = l;
        tiles = table;
    }
    if ((ndim == 3 && out_t != g[0].out) || out_h != g[1].out || out_w != g[2].out) return TB_ERR_SHAPE;
    const int64_t planes = B * C;
    const int64_t ntiles = (int64_t)g[0].n * g[1].n * g[2].n;
    if (planes == 0 || ntiles == 0 || g[0].out == 0 || g[1].out == 0) return TB_OK;  // nothing to write
    if (B > 0 && planes / B != C) return TB_ERR_SHAPE;
    if (tiles == nullptr || out == nullptr) return TB_ERR_NULL;
    if (ntiles > TB_MAX_TILES) return TB_ERR_UNSUPPORTED;
    for (int64_t q = 0; q < ntiles; ++q)
        if (tiles[q] == nullptr) return TB_ERR_NULL;
    // every tile's element count must fit the kernel's 64-bit offsets (always)
    // and the output row count its 32-bit row arithmetic (checked at launch)
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const bool small = g[0].n <= tb::SMALL_MAXA && g[1].n <= tb::SMALL_MAXA && g[2].n <= tb::SMALL_MAXA &&
                       ntiles <= tb::SMALL_MAXT;
    if (small) {
        tb::StitchParamsSmall prm;
        tb_status r = fill_and_launch(prm, g, ndim, dtype, planes, tiles, out, st, false);
        if (r != TB_ERR_UNSUPPORTED) return r;
    }
    tb::StitchParamsLarge prm_l;
    return fill_and_launch(prm_l, g, ndim, dtype, planes, tiles, out, st, true);
}

// ---------------------------------------------------------------------------
// PatchGroupNorm
// ---------------------------------------------------------------------------

tb_status gn_validate(const void* const* patches, int32_t P, tb_dtype dtype, int64_t N, int64_t C,
                      const int64_t* spatial, int32_t G, const void* partials) {
    if (dtype != TB_F32 && dtype != TB_F16 && dtype != TB_BF16) return TB_ERR_DTYPE;
    if (P < 1 || N < 0 || C < 0 || G < 1) return TB_ERR_SHAPE;
    if (C % G != 0) return TB_ERR_SHAPE;
    if (P > tb::GN_MAXP) return TB_ERR_UNSUPPORTED;
    if (spatial == nullptr || patches == nullptr) return TB_ERR_NULL;
    for (int p = 0; p < P; ++p) {
        if (spatial[p] < 0) return TB_ERR_SHAPE;
        if (N > 0 && C > 0 && spatial[p] > 0 && patches[p] == nullptr) return TB_ERR_NULL;
        // element counts must stay well inside int64
        if (spatial[p] > 0 && N > 0 && C > 0 && (double)N * (double)C * (double)spatial[p] > 9.0e18)
            return TB_ERR_SHAPE;
    }
    if (N > 0 && C > 0 && partials == nullptr) return TB_ERR_NULL;
    if ((double)P * (double)N * (double)G * TB_GN_PARTS > 2.0e9) return TB_ERR_UNSUPPORTED;
    return TB_OK;
}

// CTAs per GroupNorm statistics unit (each writes one of the unit's
// TB_GN_PARTS records; the rest get count 0): 1, 2, 4 or 8, about two CTAs
// per SM in all, each streaming >= 16 KB.  Measured on GB300: more, shorter
// CTAs per unit lose more to their fixed costs than they gain.  Only the
// statistics call uses it: the records describe themselves, so the apply
// step reads every record and needs no agreement with this choice.
tb_status gn_parts(int32_t P, int64_t N, int64_t C, const int64_t* spatial, int32_t G, tb_dtype dtype, int* parts) {
    int64_t max_len = 0;
    for (int p = 0; p < P; ++p) max_len = std::max(max_len, (C / G) * spatial[p]);
    const int64_t units = (int64_t)P * N * G;
    const int64_t bytes = max_len * elem_bytes(dtype);
    int sms = 0;
    tb_status s = device_sms(&sms);
    if (s != TB_OK) return s;
    int64_t want = units > 0 ? (2LL * sms + units / 2) / units : 1;
    want = std::min<int64_t>(want, bytes / 16384);
    int k = 1;
    while (k * 2 <= TB_GN_PARTS && k * 2 <= want) k *= 2;
    if (TB_GN_WAVE_FIT && units > 0) {
        // as many parts as keep the grid within one wave, each >= 16 KB
        const int64_t fit = std::min<int64_t>((int64_t)TB_GN_WAVE_CTAS * sms / units, bytes / 16384);
        k = (int)std::max<int64_t>(1, std::min<int64_t>(TB_GN_PARTS, fit));
    }
    if (TB_GN_FORCE_PARTS > 0) k = TB_GN_FORCE_PARTS;
    *parts = k;
    return TB_OK;
}

// The apply step over R record sets (R = P for the plain two-call path).
tb_status gn_apply(const void* const* patches, void* const* outs, int32_t P, tb_dtype dtype, int64_t N, int64_t C,
                   const int64_t* spatial, int32_t G, const tb_gn_partial* partials, int32_t R, const void* gamma,
                   const void* beta, float eps, int32_t silu, void* stream) {
    tb_status s = gn_validate(patches, P, dtype, N, C, spatial, G, partials);
    if (s != TB_OK) return s;
    if (R < 1) return TB_ERR_SHAPE;
    if ((double)R * (double)N * (double)G * TB_GN_PARTS > 2.0e9 || R > 65536) return TB_ERR_UNSUPPORTED;
    if (!(eps >= 0.0f) || std::isinf(eps)) return TB_ERR_SHAPE;
    if (outs == nullptr) return TB_ERR_NULL;
    if (N == 0 || C == 0) return TB_OK;
    for (int p = 0; p < P; ++p)
        if (spatial[p] > 0 && outs[p] == nullptr) return TB_ERR_NULL;
    tb::GnApplyParams prm;
    std::memset(&prm, 0, sizeof(prm));
    const int vec = 16 / elem_bytes(dtype);
    bool aligned = true;
    for (int p = 0; p < P; ++p) {
        if (spatial[p] > 0 && (spatial[p] % vec != 0 || !aligned16(patches[p]) || !aligned16(outs[p])))
            aligned = false;
    }
    const int64_t seg = tb::gn_apply_segment((int)dtype, aligned);
    int64_t items = 0;
    for (int p = 0; p < P; ++p) {
        prm.patches[p] = patches[p];
        prm.outs[p] = outs[p];
        prm.spatial[p] = spatial[p];
        prm.item_start[p] = items;
        prm.nseg[p] = spatial[p] > 0 ? (spatial[p] + seg - 1) / seg : 1;
        if (spatial[p] > 0) items += N * C * prm.nseg[p];
    }
    prm.item_start[P] = items;  // a patch with no elements owns an empty item range
    if (items == 0) return TB_OK;
    if (items > 2147483647LL) return TB_ERR_UNSUPPORTED;
    prm.partials = reinterpret_cast<const tb::GnPartial*>(partials);
    prm.gamma = gamma;
    prm.beta = beta;
    prm.N = N;
    prm.C = C;
    prm.P = P;
    prm.G = G;
    prm.seg = (int32_t)seg;
    prm.R = R;
    prm.eps = eps;
    prm.silu = silu ? 1 : 0;
    prm.aligned = aligned ? 1 : 0;
    prm.status = debug_status();
    cudaError_t e = tb::launch_gn_apply(prm, (int)dtype, items, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return TB_OK;
}

// ---------------------------------------------------------------------------
// Patchify split / patch gather
// ---------------------------------------------------------------------------

tb_status band_layout(int64_t extent, int32_t factor, int32_t P, int64_t* starts, int64_t* sizes) {
    if (extent < 0 || factor < 1 || P < 1) return TB_ERR_SHAPE;
    if (extent % factor != 0) return TB_ERR_SHAPE;
    if (P > tb::PF_MAXP) return TB_ERR_UNSUPPORTED;
    const int64_t bands = extent / factor, each = bands / P, extra = bands % P;
    int64_t at = 0;
    for (int p = 0; p < P; ++p) {
        const int64_t size = (each + (p < extra ? 1 : 0)) * factor;
        if (starts) starts[p] = at;
        if (sizes) sizes[p] = size;
        at += size;
    }
    return TB_OK;
}

// The tensor of `shape` seen as [outer, extent, inner] around `axis`.
tb_status split_view(int32_t ndim, const int64_t* shape, int32_t axis, int64_t& outer, int64_t& extent,
                     int64_t& inner) {
    if (shape == nullptr) return TB_ERR_NULL;
    if (ndim < 1 || ndim > 8 || axis < 0 || axis >= ndim) return TB_ERR_SHAPE;
    double total = 1.0;
    outer = 1;
    inner = 1;
    for (int d = 0; d < ndim; ++d) {
        if (shape[d] < 0) return TB_ERR_SHAPE;
        total *= (double)shape[d];
        if (d < axis) outer *= shape[d];
        if (d > axis) inner *= shape[d];
        if (total > 1.0e18) return TB_ERR_SHAPE;
    }
    extent = shape[axis];
    return TB_OK;
}

// One launch copying the P bands between the whole tensor and the patches.
tb_status patch_copy(bool to_patches, void* whole, void* const* patches, int32_t P, const int64_t* starts,
                     const int64_t* sizes, int eb, int64_t outer, int64_t extent, int64_t inner, int64_t slot,
                     void* stream) {
    int64_t largest = 0;
    for (int p = 0; p < P; ++p) largest = std::max(largest, sizes[p]);
    if (slot < 0 || (slot > 0 && slot < largest)) return TB_ERR_SHAPE;
    if (outer == 0 || inner == 0 || extent == 0) return TB_OK;
    if (whole == nullptr) return TB_ERR_NULL;
    for (int p = 0; p < P; ++p)
        if (sizes[p] > 0 && patches[p] == nullptr) return TB_ERR_NULL;
    // widest chunk dividing every run, pitch, offset and base address
    int vec = 16;
    auto fit = [&vec](uint64_t q) {
        while (vec > 1 && q % (uint64_t)vec != 0) vec >>= 1;
    };
    fit((uint64_t)(extent * inner * eb));
    fit((uint64_t)reinterpret_cast<uintptr_t>(whole));
    for (int p = 0; p < P; ++p) {
        if (sizes[p] == 0) continue;
        fit((uint64_t)(sizes[p] * inner * eb));
        fit((uint64_t)(starts[p] * inner * eb));
        fit((uint64_t)((slot > 0 ? slot : sizes[p]) * inner * eb));
        fit((uint64_t)reinterpret_cast<uintptr_t>(patches[p]));
    }
    // element counts in chunks (a chunk narrower than an element only for
    // a base address that is not aligned to the element)
    auto chunks = [&](int64_t elems) { return elems * eb / vec; };
    if (outer + tb::PF_BLOCK >= 2147483647LL) return TB_ERR_UNSUPPORTED;
    tb::PatchCopyParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.whole = whole;
    prm.wpitch = chunks(extent * inner);
    prm.outer = outer;
    prm.status = debug_status();
    prm.P = P;
    const int64_t cta_chunks = tb::PF_CTA_BYTES / vec;
    int64_t ranges = 1;
    for (int p = 0; p < P; ++p) {
        const int64_t run = chunks(sizes[p] * inner);
        if (run >= 2147483647LL) return TB_ERR_UNSUPPORTED;
        prm.patch[p] = patches[p];
        prm.n[p] = outer * run;
        prm.run[p] = (int32_t)std::max<int64_t>(run, 1);
        prm.step_o[p] = tb::PF_BLOCK / prm.run[p];
        prm.step_r[p] = tb::PF_BLOCK % prm.run[p];
        prm.woff[p] = chunks(starts[p] * inner);
        prm.ppitch[p] = chunks((slot > 0 ? slot : sizes[p]) * inner);
        ranges = std::max(ranges, (prm.n[p] + cta_chunks - 1) / cta_chunks);
    }
    for (int p = 0; p < P; ++p) prm.per_cta[p] = std::max<int64_t>(1, (prm.n[p] + ranges - 1) / ranges);
    const int64_t grid = ranges * P;
    if (grid > 2147483647LL) return TB_ERR_UNSUPPORTED;
    cudaError_t e = tb::launch_patch_copy(prm, vec, to_patches, grid, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return TB_OK;
}

}  // namespace

void tb::record_cuda_error(cudaError_t e) { g_last_cuda_error = (int)e; }

// ---------------------------------------------------------------------------
// normalised-ramp stitch
// ---------------------------------------------------------------------------

// Weight of tile n (of N, extent T) at tile-local position q.
double ramp_w(int n, int N, int T, int q, int zero, int ramp) {
    double w = 1.0;
    if (n > 0) w *= std::min(1.0, std::max(0.0, (double)(q - zero) / ramp));
    if (n < N - 1) w *= std::min(1.0, std::max(0.0, (double)((T - 1 - q) - zero) / ramp));
    return w;
}

// Validates one axis and cuts it into segments of constant positive-weight
// tile sets, positions grouped `gran` at a time.
tb_status ramp_axis(const tb_ramp_axis* a, int gran, tb::RampAxisK& k) {
    if (a == nullptr || a->origins == nullptr) return TB_ERR_NULL;
    const int N = a->n_tiles, T = a->tile_extent, out = a->out_extent;
    if (N < 1 || T < 1 || out < 1 || a->zero < 0 || a->ramp < 1) return TB_ERR_GEOMETRY;
    if (N > tb::RAMP_MAXA) return TB_ERR_UNSUPPORTED;
    if (a->origins[0] != 0 || a->origins[N - 1] + T != out) return TB_ERR_GEOMETRY;
    for (int n = 1; n < N; ++n)
        if (a->origins[n] <= a->origins[n - 1] || a->origins[n] > out - T) return TB_ERR_GEOMETRY;
    k.n = N;
    k.T = T;
    k.out = out;
    k.zero = a->zero;
    k.inv_ramp = (float)(1.0 / a->ramp);
    for (int n = 0; n < N; ++n) k.org[n] = (int32_t)a->origins[n];
    k.nseg = 0;
    int cur[tb::RAMP_MAXCOVER] = {-1, -1, -1}, ncur = -1;
    for (int p0 = 0; p0 < out; p0 += gran) {
        // tiles with positive weight at any of positions p0 .. p0 + gran - 1
        int set[tb::RAMP_MAXCOVER], ns = 0;
        for (int n = 0; n < N; ++n) {
            bool pos = false;
            for (int p = p0; p < p0 + gran && p < out; ++p) {
                const int q = p - (int)a->origins[n];
                if (q >= 0 && q < T && ramp_w(n, N, T, q, a->zero, a->ramp) > 0.0) pos = true;
            }
            if (!pos) continue;
            if (ns == tb::RAMP_MAXCOVER) return TB_ERR_UNSUPPORTED;
            set[ns++] = n;
        }
        // every single position must have some positive weight
        for (int p = p0; p < p0 + gran && p < out; ++p) {
            double sum = 0.0;
            for (int e = 0; e < ns; ++e) {
                const int q = p - (int)a->origins[set[e]];
                if (q >= 0 && q < T) sum += ramp_w(set[e], N, T, q, a->zero, a->ramp);
            }
            if (!(sum > 0.0)) return TB_ERR_GEOMETRY;
        }
        bool same = ns == ncur;
        for (int e = 0; same && e < ns; ++e) same = set[e] == cur[e];
        if (!same) {
            if (k.nseg == tb::RAMP_MAXSEG) return TB_ERR_UNSUPPORTED;
            k.seg_start[k.nseg] = p0;
            k.seg_len[k.nseg] = 0;
            k.seg_n[k.nseg] = ns;
            for (int e = 0; e < tb::RAMP_MAXCOVER; ++e) k.seg_tile[k.nseg][e] = (int8_t)(e < ns ? set[e] : 0);
            ++k.nseg;
            ncur = ns;
            for (int e = 0; e < ns; ++e) cur[e] = set[e];
        }
        k.seg_len[k.nseg - 1] += std::min(gran, out - p0);
    }
    return TB_OK;
}

// ===========================================================================
// C ABI
// ===========================================================================

TB_API size_t tb_version(void) { return 10000 * 0 + 100 * 3 + 0; }

TB_API const char* tb_status_string(tb_status s) {
    switch (s) {
        case TB_OK: return "ok";
        case TB_ERR_NULL: return "a required pointer is NULL";
        case TB_ERR_DTYPE: return "unknown dtype";
        case TB_ERR_SHAPE: return "sizes are inconsistent";
        case TB_ERR_GEOMETRY: return "tile-grid geometry out of range";
        case TB_ERR_UNSUPPORTED: return "request outside what the kernels handle";
        case TB_ERR_CUDA: return "the CUDA runtime refused the launch";
    }
    return "unknown status";
}

TB_API int tb_last_cuda_error(void) { return g_last_cuda_error; }

TB_API tb_status tb_axis_layout(const tb_axis* a, int32_t cap, int32_t* n_tiles, int64_t* origins, int32_t* extents,
                                int32_t* blends, int32_t* kept, int64_t* out_extent) {
    if (a == nullptr || n_tiles == nullptr) return TB_ERR_NULL;
    Axis g;
    int64_t ntot = 0;
    tb_status s = derive_axis(a, g, &ntot);
    if (s == TB_ERR_UNSUPPORTED) {
        *n_tiles = (int32_t)std::min<int64_t>(ntot, 2147483647LL);
        return s;
    }
    if (s != TB_OK) return s;
    *n_tiles = g.n;
    for (int k = 0; k < g.n && k < cap; ++k) {
        if (origins) origins[k] = (int64_t)k * g.stride * a->scale;
        if (extents) extents[k] = g.ext[k];
        if (blends) blends[k] = g.blend[k];
        if (kept) kept[k] = g.kept[k];
    }
    if (out_extent) *out_extent = g.out;
    return TB_OK;
}

TB_API tb_status tb_stitch2d(const void* const* tiles, tb_dtype dtype, int64_t B, int64_t C, const tb_axis* ay,
                             const tb_axis* ax, void* out, int64_t out_h, int64_t out_w, void* stream) {
    return stitch_common(2, tiles, dtype, B, C, nullptr, ay, ax, out, 1, out_h, out_w, stream);
}

TB_API tb_status tb_stitch3d(const void* const* tiles, tb_dtype dtype, int64_t B, int64_t C, const tb_axis* at,
                             const tb_axis* ay, const tb_axis* ax, void* out, int64_t out_t, int64_t out_h,
                             int64_t out_w, void* stream) {
    if (at == nullptr) return TB_ERR_NULL;
    return stitch_common(3, tiles, dtype, B, C, at, ay, ax, out, out_t, out_h, out_w, stream);
}

// The three axes of a 2D (at == NULL) or 3D grid, validated.
tb_status grid_axes(const tb_axis* at, const tb_axis* ay, const tb_axis* ax, Axis (&g)[3]) {
    int64_t ntot = 0;
    if (at != nullptr) {
        tb_status s = derive_axis(at, g[0], &ntot);
        if (s != TB_OK) return s;
    } else {
        g[0].n = 1;
        g[0].ext[0] = 1;
        g[0].kept[0] = 1;
        g[0].blend[0] = 0;
        g[0].out = 1;
    }
    tb_status s = derive_axis(ay, g[1], &ntot);
    if (s != TB_OK) return s;
    return derive_axis(ax, g[2], &ntot);
}

// Elements of the packed band of `e` slices along `axis` (0: frames, 1: rows)
// of every tile of one tile row (or frame tile), all planes.
int64_t band_elems(const Axis (&g)[3], int axis, int64_t planes, int32_t e) {
    int64_t frames = 0, rows = 0, width = 0;
    for (int k = 0; k < g[0].n; ++k) frames += g[0].ext[k];
    for (int i = 0; i < g[1].n; ++i) rows += g[1].ext[i];
    for (int j = 0; j < g[2].n; ++j) width += g[2].ext[j];
    return axis == 0 ? planes * (int64_t)e * rows * width : planes * frames * (int64_t)e * width;
}

tb_status shard_layout(int axis, const tb_axis* at, const tb_axis* ay, const tb_axis* ax, int64_t B, int64_t C,
                       int32_t world, int32_t rank, tb_shard_layout* out) {
    if (ay == nullptr || ax == nullptr || out == nullptr || (axis == 0 && at == nullptr)) return TB_ERR_NULL;
    if (B < 0 || C < 0 || world < 1 || rank < 0 || rank >= world) return TB_ERR_SHAPE;
    if (B > 0 && C > INT64_MAX / B) return TB_ERR_SHAPE;
    Axis g[3];
    tb_status s = grid_axes(at, ay, ax, g);
    if (s != TB_OK) return s;
    const Axis& a = g[axis];
    // tiles along the axis shared out in rank order, the first ranks one more
    const int32_t n = a.n, each = n / world, extra = n % world;
    const int32_t begin = rank * each + std::min(rank, extra);
    const int32_t end = begin + each + (rank < extra ? 1 : 0);
    tb_shard_layout l{};
    l.row_begin = begin;
    l.row_end = end;
    for (int i = 0; i < begin; ++i) l.out_row_begin += a.kept[i];
    for (int i = begin; i < end; ++i) l.out_rows += a.kept[i];
    const int64_t planes = B * C;
    if (end > begin && begin > 0 && a.blend[begin] > 0) {
        l.halo_rows = a.blend[begin];
        l.halo_elems = band_elems(g, axis, planes, l.halo_rows);
    }
    if (end > begin && end < n && a.blend[end] > 0) l.send_elems = band_elems(g, axis, planes, a.blend[end]);
    *out = l;
    return TB_OK;
}

// Packs the last e(index + 1) slices along `axis` of every tile of tile row
// (axis 1) or frame tile (axis 0) `index`: tiles are the n_t x n_x tiles of
// the row (k-major) or the n_y x n_x tiles of the frame tile (i-major).
tb_status halo_pack(int axis, const void* const* tiles, tb_dtype dtype, int64_t B, int64_t C, const tb_axis* at,
                    const tb_axis* ay, const tb_axis* ax, int32_t index, void* halo, void* stream) {
    if (dtype != TB_F32 && dtype != TB_F16 && dtype != TB_BF16) return TB_ERR_DTYPE;
    if (ay == nullptr || ax == nullptr || (axis == 0 && at == nullptr)) return TB_ERR_NULL;
    if (B < 0 || C < 0) return TB_ERR_SHAPE;
    if (B > 0 && C > INT64_MAX / B) return TB_ERR_SHAPE;
    Axis g[3];
    tb_status s = grid_axes(at, ay, ax, g);
    if (s != TB_OK) return s;
    if (index < 0 || index + 1 >= g[axis].n) return TB_ERR_SHAPE;
    const int32_t e = g[axis].blend[index + 1];
    const int64_t planes = B * C;
    if (e == 0 || planes == 0) return TB_OK;
    const int nouter = axis == 0 ? g[1].n : g[0].n;  // tiles of the row / frame tile: nouter x n_x
    const int64_t ntiles = (int64_t)nouter * g[2].n;
    if (ntiles > tb::HALO_MAXT) return TB_ERR_UNSUPPORTED;
    if (tiles == nullptr || halo == nullptr) return TB_ERR_NULL;
    for (int64_t q = 0; q < ntiles; ++q)
        if (tiles[q] == nullptr) return TB_ERR_NULL;
    const int eb = elem_bytes(dtype);
    // widest chunk dividing every slice, band offset and address
    int vb = 16;
    auto fit = [&vb](uint64_t v) {
        while (vb > 1 && v % (uint64_t)vb != 0) vb >>= 1;
    };
    fit((uint64_t)reinterpret_cast<uintptr_t>(halo));
    for (int o = 0; o < nouter; ++o)
        for (int j = 0; j < g[2].n; ++j)
            fit((uint64_t)(axis == 0 ? (int64_t)g[1].ext[o] * g[2].ext[j] : (int64_t)g[2].ext[j]) * eb);
    for (int64_t q = 0; q < ntiles; ++q) fit((uint64_t)reinterpret_cast<uintptr_t>(tiles[q]));
    tb::HaloPackParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.dst = halo;
    prm.status = debug_status();
    prm.e = e;
    prm.ntiles = (int32_t)ntiles;
    // a tile is [planes][outer slices][slices along the axis][slice], so a
    // band is the last e slices of each (plane, outer slice)
    int64_t off = 0, most = 0;
    for (int o = 0; o < nouter; ++o)
        for (int j = 0; j < g[2].n; ++j) {
            const int64_t q = (int64_t)o * g[2].n + j;
            const int64_t slices = axis == 0 ? g[0].ext[index] : g[1].ext[index];
            const int64_t outer = axis == 0 ? 1 : g[0].ext[o];
            const int64_t w = (axis == 0 ? (int64_t)g[1].ext[o] * g[2].ext[j] : (int64_t)g[2].ext[j]) * eb / vb;
            if (w > 2147483647LL || slices > 2147483647LL || planes * outer * slices * w > (INT64_MAX >> 1))
                return TB_ERR_UNSUPPORTED;
            prm.src[q] = tiles[q];
            prm.rows[q] = (int32_t)slices;
            prm.width[q] = (int32_t)w;
            prm.n[q] = planes * outer * e * w;
            prm.dst_off[q] = off;
            off += prm.n[q];
            most = std::max(most, prm.n[q]);
        }
    prm.dst_total = off;
    // chunks per CTA: 8 rounds of 256 threads, 32 KB of 16-byte chunks
    const int64_t cta = (int64_t)tb::HALO_BLOCK * 8;
    prm.per_cta = cta;
    const int64_t ranges = (most + cta - 1) / cta;
    if (ranges > 2147483647LL) return TB_ERR_UNSUPPORTED;
    cudaError_t e2 = tb::launch_halo_pack(prm, vb, ranges, reinterpret_cast<cudaStream_t>(stream));
    if (e2 != cudaSuccess) return cuda_fail(e2);
    return TB_OK;
}

TB_API tb_status tb_stitch_shard_layout(const tb_axis* at, const tb_axis* ay, const tb_axis* ax, int64_t B, int64_t C,
                                        int32_t world, int32_t rank, tb_shard_layout* out) {
    return shard_layout(1, at, ay, ax, B, C, world, rank, out);
}

TB_API tb_status tb_stitch_shard_frames_layout(const tb_axis* at, const tb_axis* ay, const tb_axis* ax, int64_t B,
                                               int64_t C, int32_t world, int32_t rank, tb_shard_layout* out) {
    return shard_layout(0, at, ay, ax, B, C, world, rank, out);
}

TB_API tb_status tb_stitch_halo_pack(const void* const* tiles, tb_dtype dtype, int64_t B, int64_t C,
                                     const tb_axis* at, const tb_axis* ay, const tb_axis* ax, int32_t row, void* halo,
                                     void* stream) {
    return halo_pack(1, tiles, dtype, B, C, at, ay, ax, row, halo, stream);
}

TB_API tb_status tb_stitch_halo_pack_frames(const void* const* tiles, tb_dtype dtype, int64_t B, int64_t C,
                                            const tb_axis* at, const tb_axis* ay, const tb_axis* ax,
                                            int32_t frame_tile, void* halo, void* stream) {
    return halo_pack(0, tiles, dtype, B, C, at, ay, ax, frame_tile, halo, stream);
}

TB_API tb_status tb_stitch2d_shard(const void* const* tiles, const void* halo, tb_dtype dtype, int64_t B, int64_t C,
                                   const tb_axis* ay, const tb_axis* ax, int32_t row_begin, int32_t row_end,
                                   void* out, int64_t out_rows, int64_t out_w, void* stream) {
    const Shard sh{1, row_begin, row_end, halo};
    return stitch_common(2, tiles, dtype, B, C, nullptr, ay, ax, out, 1, out_rows, out_w, stream, &sh);
}

TB_API tb_status tb_stitch3d_shard(const void* const* tiles, const void* halo, tb_dtype dtype, int64_t B, int64_t C,
                                   const tb_axis* at, const tb_axis* ay, const tb_axis* ax, int32_t row_begin,
                                   int32_t row_end, void* out, int64_t out_t, int64_t out_rows, int64_t out_w,
                                   void* stream) {
    if (at == nullptr) return TB_ERR_NULL;
    const Shard sh{1, row_begin, row_end, halo};
    return stitch_common(3, tiles, dtype, B, C, at, ay, ax, out, out_t, out_rows, out_w, stream, &sh);
}

TB_API tb_status tb_stitch3d_shard_frames(const void* const* tiles, const void* halo, tb_dtype dtype, int64_t B,
                                          int64_t C, const tb_axis* at, const tb_axis* ay, const tb_axis* ax,
                                          int32_t frame_begin, int32_t frame_end, void* out, int64_t out_frames,
                                          int64_t out_h, int64_t out_w, void* stream) {
    if (at == nullptr) return TB_ERR_NULL;
    const Shard sh{0, frame_begin, frame_end, halo};
    return stitch_common(3, tiles, dtype, B, C, at, ay, ax, out, out_frames, out_h, out_w, stream, &sh);
}

TB_API tb_status tb_ramp_axis_spread(int32_t latent_extent, int32_t latent_tile, int32_t n_tiles, int32_t scale,
                                     int32_t zero_latents, int32_t ramp_latents, int64_t* origins,
                                     tb_ramp_axis* axis) {
    if (origins == nullptr || axis == nullptr) return TB_ERR_NULL;
    if (n_tiles < 1 || scale < 1 || latent_tile < 1 || latent_tile > latent_extent || zero_latents < 0 ||
        ramp_latents < 1)
        return TB_ERR_GEOMETRY;
    if (n_tiles > TB_MAX_TILES_PER_AXIS) return TB_ERR_UNSUPPORTED;
    if ((int64_t)latent_extent * scale > 2147483647LL || (int64_t)zero_latents * scale > 2147483647LL ||
        (int64_t)ramp_latents * scale > 2147483647LL)
        return TB_ERR_UNSUPPORTED;
    if (n_tiles == 1 && latent_tile != latent_extent) return TB_ERR_GEOMETRY;
    const int64_t span = (int64_t)latent_extent - latent_tile;
    int64_t prev = 0;
    for (int n = 0; n < n_tiles; ++n) {
        const int64_t lat = n_tiles == 1 ? 0 : (int64_t)n * span / (n_tiles - 1);
        if (n > 0 && lat - prev > latent_tile) return TB_ERR_GEOMETRY;
        origins[n] = lat * scale;
        prev = lat;
    }
    axis->n_tiles = n_tiles;
    axis->tile_extent = latent_tile * scale;
    axis->out_extent = latent_extent * scale;
    axis->zero = zero_latents * scale;
    axis->ramp = ramp_latents * scale;
    axis->origins = origins;
    return TB_OK;
}

TB_API tb_status tb_stitch2d_ramp(const void* const* tiles, tb_dtype dtype, int64_t B, int64_t C,
                                  const tb_ramp_axis* ay, const tb_ramp_axis* ax, void* out, void* stream) {
    if (dtype != TB_F32 && dtype != TB_F16 && dtype != TB_BF16) return TB_ERR_DTYPE;
    if (B < 0 || C < 0) return TB_ERR_SHAPE;
    if (ay == nullptr || ax == nullptr) return TB_ERR_NULL;
    const int eb = elem_bytes(dtype);
    const int64_t planes = B * C;
    if (B > 0 && planes / B != C) return TB_ERR_SHAPE;
    // 16-byte chunks along the width when the layout and every pointer allow
    int vec = 16 / eb;
    bool ok = ax->tile_extent % vec == 0 && ax->out_extent % vec == 0 && ax->origins != nullptr;
    for (int n = 0; ok && n < ax->n_tiles && n < tb::RAMP_MAXA; ++n) ok = ax->origins[n] % vec == 0;
    tb::RampParams prm;
    std::memset(&prm, 0, sizeof(prm));
    tb_status st = ramp_axis(ay, 1, prm.ay);
    if (st != TB_OK) return st;
    st = ramp_axis(ax, 1, prm.ax);  // validates the width axis element by element
    if (st != TB_OK) return st;
    const int64_t ntiles = (int64_t)ay->n_tiles * ax->n_tiles;
    if (ntiles > TB_MAX_TILES) return TB_ERR_UNSUPPORTED;
    if (planes == 0) return TB_OK;
    if (tiles == nullptr || out == nullptr) return TB_ERR_NULL;
    for (int64_t q = 0; q < ntiles; ++q)
        if (tiles[q] == nullptr) return TB_ERR_NULL;
    if ((int64_t)ay->tile_extent * ax->tile_extent * eb > 2147483647LL ||
        (int64_t)ax->out_extent * eb > 2147483647LL)
        return TB_ERR_UNSUPPORTED;
    ok = ok && aligned16(out);
    for (int64_t q = 0; ok && q < ntiles; ++q) ok = aligned16(tiles[q]);
    if (ok) {
        st = ramp_axis(ax, vec, prm.ax);  // chunk-granular width segments
        if (st == TB_ERR_UNSUPPORTED) ok = false;
        else if (st != TB_OK) return st;
    }
    if (!ok) {
        vec = 1;
        st = ramp_axis(ax, 1, prm.ax);
        if (st != TB_OK) return st;
    }
    for (int64_t q = 0; q < ntiles; ++q) prm.tiles[q] = tiles[q];
    prm.out = out;
    prm.status = debug_status();
    prm.planes = planes;
    // rectangles grouped by cover counts, so CTAs dispatched together mostly
    // run the same code path
    for (int sy = 0; sy < prm.ay.nseg; ++sy) {
        const int c = prm.ay.seg_n[sy] - 1;
        prm.yseg[c][prm.ycnt[c]++] = (int16_t)sy;
    }
    for (int sx = 0; sx < prm.ax.nseg; ++sx) {
        const int c = prm.ax.seg_n[sx] - 1;
        prm.xseg[c][prm.xcnt[c]++] = (int16_t)sx;
    }
    prm.group_start[0] = 0;
    for (int g = 0; g < tb::RAMP_MAXCOVER * tb::RAMP_MAXCOVER; ++g)
        prm.group_start[g + 1] =
            prm.group_start[g] + prm.ycnt[g / tb::RAMP_MAXCOVER] * prm.xcnt[g % tb::RAMP_MAXCOVER];
    // A piece is a run of rows of one rectangle with every plane's rows laid
    // end to end, so rectangles a few rows high still fill whole CTAs.  Rows
    // per thread start at TB_RAMP_MAX_ROWS_PER_THREAD and halve (down to 2)
    // while there are fewer than TB_RAMP_PIECES_PER_SM pieces per SM.  The
    // grid is (rectangle, piece index).
    if (planes * ay->out_extent > 2147483647LL - 4LL * tb::ramp_block()) return TB_ERR_UNSUPPORTED;
    int sms = 0;
    st = device_sms(&sms);
    if (st != TB_OK) return st;
    int64_t max_pieces = 1;
    for (int rpt = TB_RAMP_MAX_ROWS_PER_THREAD;; rpt /= 2) {
        for (int sx = 0; sx < prm.ax.nseg; ++sx) {
            const int width = prm.ax.seg_len[sx] / vec;
            const int bdx = std::max(1, std::min(width, tb::ramp_block()));
            prm.rows_per_piece[sx] = (tb::ramp_block() / bdx) * rpt;
        }
        int64_t total = 0;
        max_pieces = 1;
        for (int sy = 0; sy < prm.ay.nseg; ++sy) {
            const int64_t flat = planes * prm.ay.seg_len[sy];
            for (int sx = 0; sx < prm.ax.nseg; ++sx) {
                const int64_t n = (flat + prm.rows_per_piece[sx] - 1) / prm.rows_per_piece[sx];
                total += n;
                max_pieces = std::max(max_pieces, n);
            }
        }
        if (total >= (int64_t)TB_RAMP_PIECES_PER_SM * sms || rpt <= 2) break;
    }
    if (max_pieces > 65535) return TB_ERR_UNSUPPORTED;
    int small = 0;
    for (int g : {0, 1, 3, 4}) small += prm.ycnt[g / tb::RAMP_MAXCOVER] * prm.xcnt[g % tb::RAMP_MAXCOVER];
    cudaError_t e = tb::launch_ramp(prm, (int)dtype, vec, small, prm.ay.nseg * prm.ax.nseg - small, (int)max_pieces,
                                    reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return TB_OK;
}

TB_API tb_status tb_patch_gn_stats(const void* const* patches, int32_t P, tb_dtype dtype, int64_t N, int64_t C,
                                   const int64_t* spatial, int32_t G, tb_gn_partial* partials, void* stream) {
    tb_status s = gn_validate(patches, P, dtype, N, C, spatial, G, partials);
    if (s != TB_OK) return s;
    if (N == 0 || C == 0) return TB_OK;
    tb::GnStatsParams prm;
    std::memset(&prm, 0, sizeof(prm));
    const int vec = 16 / elem_bytes(dtype);
    const int64_t cg = C / G;
    bool aligned = true;
    for (int p = 0; p < P; ++p) {
        prm.patches[p] = patches[p];
        prm.spatial[p] = spatial[p];
        const int64_t len = cg * spatial[p];
        if (spatial[p] > 0 && (!aligned16(patches[p]) || len % vec != 0)) aligned = false;
    }
    prm.partials = reinterpret_cast<tb::GnPartial*>(partials);
    prm.N = N;
    prm.C = C;
    prm.P = P;
    prm.G = G;
    prm.aligned = aligned ? 1 : 0;
    prm.status = debug_status();
    const int64_t units = (int64_t)P * N * G;
    int parts = 1;
    s = gn_parts(P, N, C, spatial, G, dtype, &parts);
    if (s != TB_OK) return s;
    prm.parts = parts;
    if (units * parts > 2147483647LL) return TB_ERR_UNSUPPORTED;
    cudaError_t e = tb::launch_gn_stats(prm, (int)dtype, units, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return TB_OK;
}

TB_API tb_status tb_patch_gn_apply(const void* const* patches, void* const* outs, int32_t P, tb_dtype dtype, int64_t N,
                                   int64_t C, const int64_t* spatial, int32_t G, const tb_gn_partial* partials,
                                   const void* gamma, const void* beta, float eps, int32_t silu, void* stream) {
    return gn_apply(patches, outs, P, dtype, N, C, spatial, G, partials, P, gamma, beta, eps, silu, stream);
}

TB_API tb_status tb_patch_gn_apply_gathered(const void* const* patches, void* const* outs, int32_t P, tb_dtype dtype,
                                            int64_t N, int64_t C, const int64_t* spatial, int32_t G,
                                            const tb_gn_partial* partials, int32_t R, const void* gamma,
                                            const void* beta, float eps, int32_t silu, void* stream) {
    return gn_apply(patches, outs, P, dtype, N, C, spatial, G, partials, R, gamma, beta, eps, silu, stream);
}

TB_API tb_status tb_patchify_layout(int64_t extent, int32_t factor, int32_t P, int64_t* starts, int64_t* sizes) {
    return band_layout(extent, factor, P, starts, sizes);
}

TB_API tb_status tb_patchify(const void* x, tb_dtype dtype, int32_t ndim, const int64_t* shape, int32_t axis,
                             int32_t factor, int32_t P, int64_t slot, void* const* patches, void* stream) {
    if (dtype != TB_F32 && dtype != TB_F16 && dtype != TB_BF16) return TB_ERR_DTYPE;
    int64_t outer, extent, inner;
    tb_status s = split_view(ndim, shape, axis, outer, extent, inner);
    if (s != TB_OK) return s;
    int64_t starts[tb::PF_MAXP], sizes[tb::PF_MAXP];
    s = band_layout(extent, factor, P, starts, sizes);
    if (s != TB_OK) return s;
    if (patches == nullptr) return TB_ERR_NULL;
    return patch_copy(true, const_cast<void*>(x), patches, P, starts, sizes, elem_bytes(dtype), outer, extent, inner,
                      slot, stream);
}

TB_API tb_status tb_gather_patches(const void* const* patches, int32_t P, const int64_t* sizes, tb_dtype dtype,
                                   int32_t ndim, const int64_t* shape, int32_t axis, int64_t slot, void* out,
                                   void* stream) {
    if (dtype != TB_F32 && dtype != TB_F16 && dtype != TB_BF16) return TB_ERR_DTYPE;
    int64_t outer, extent, inner;
    tb_status s = split_view(ndim, shape, axis, outer, extent, inner);
    if (s != TB_OK) return s;
    if (P < 1) return TB_ERR_SHAPE;
    if (P > tb::PF_MAXP) return TB_ERR_UNSUPPORTED;
    if (sizes == nullptr || patches == nullptr) return TB_ERR_NULL;
    int64_t starts[tb::PF_MAXP], at = 0;
    for (int p = 0; p < P; ++p) {
        if (sizes[p] < 0 || sizes[p] > extent - at) return TB_ERR_SHAPE;
        starts[p] = at;
        at += sizes[p];
    }
    if (at != extent) return TB_ERR_SHAPE;
    return patch_copy(false, out, const_cast<void* const*>(patches), P, starts, sizes, elem_bytes(dtype), outer, extent,
                      inner, slot, stream);
}
