/*
 * tileblend.h -- C ABI of libtileblend: tiled-VAE tile stitching and
 * patch-parallel GroupNorm on NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (web pages, cited by title and section):
 *   [VTB] "[Proposal] Vectorize tiled VAE blending while preserving rounding
 *         and CUDA graph replay" (diffusers issue #14722), "Proposed scope".
 *   [STU] "Studio: size seam-free VAE tiles from measured peaks" (unsloth PR
 *         #12764), commit "Decode this VAE in 32-latent tiles ...".
 *   [DVA] "Add tiled VAE parallelism & extended model support" (xDiT
 *         DistVAE PR #14), the PatchGroupNorm commits and the commits on
 *         Patchify's ragged bands and on gather_patches.
 *
 * Conventions shared by every call
 *   - Plain C types only.  Device pointers point to memory the caller
 *     allocated on the current CUDA device; host pointers (pointer tables,
 *     size arrays, geometry structs) are read before the call returns and may
 *     be freed right after it.
 *   - The library allocates no device, pinned or managed memory: all of it
 *     is the caller's.  Its only state is a small host-side cache of device
 *     facts (SM count, kernel occupancy) filled on first use per device.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream) and runs asynchronously; a TB_OK return
 *     means the launch was accepted, not that the kernel finished.  Errors
 *     raised later by the kernel surface on the caller's next synchronising
 *     CUDA call.
 *   - Every argument is validated on the host before anything is launched;
 *     an invalid call returns an error status and launches nothing.  No call
 *     aborts, throws or prints.
 *   - Tensors are dense, contiguous, row-major (last dimension fastest).
 *   - Kernel parameters are passed by value.  Captured into a CUDA graph
 *     and replayed with new tensor contents at the same addresses (tested):
 *     tb_stitch2d, tb_stitch3d, tb_stitch2d_ramp, tb_patchify,
 *     tb_gather_patches, tb_stitch_halo_pack with tb_stitch2d_shard,
 *     tb_stitch_halo_pack_frames with tb_stitch3d_shard_frames, and
 *     tb_patch_gn_stats with tb_patch_gn_apply and with
 *     tb_patch_gn_apply_gathered.
 */
#ifndef TILEBLEND_H
#define TILEBLEND_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TB_OK = 0,
    TB_ERR_NULL = 1,        /* a required pointer is NULL */
    TB_ERR_DTYPE = 2,       /* unknown dtype */
    TB_ERR_SHAPE = 3,       /* sizes inconsistent with each other or the geometry */
    TB_ERR_GEOMETRY = 4,    /* tb_axis parameters out of range */
    TB_ERR_UNSUPPORTED = 5, /* valid request outside what the kernels handle (see each call) */
    TB_ERR_CUDA = 6         /* the CUDA runtime refused the launch; see tb_last_cuda_error() */
} tb_status;

typedef enum {
    TB_F32 = 0,  /* IEEE binary32 */
    TB_F16 = 1,  /* IEEE binary16 */
    TB_BF16 = 2  /* bfloat16 (upper half of binary32) */
} tb_dtype;

/*
 * One axis of a tile grid, in the parameters the pages use [VTB], [STU]:
 *   latent_extent  extent of the latent along this axis (latents; frames for
 *                  a temporal axis given with scale 1)
 *   latent_tile    tile size in latents
 *   overlap        overlap factor in [0, 1)
 *   scale          decoded samples per latent along this axis (>= 1)
 *   blend_extent   samples cross-faded between neighbours; < 0 derives the
 *                  stock value int(latent_tile * scale * overlap)
 *   row_limit      samples each tile keeps; <= 0 derives the stock value
 *                  latent_tile * scale - blend_extent
 * Derived grid (the stock tiled decode): stride = int(latent_tile *
 * (1 - overlap)); tile origins range(0, latent_extent, stride); tile n has
 * extent L(n) = min(latent_tile, latent_extent - origin) * scale samples;
 * the blend between tiles n-1 and n is clamped to e(n) = min(L(n-1), L(n),
 * blend_extent); tile n keeps K(n) = min(L(n), row_limit) samples and the
 * output extent is the sum of K(n).
 */
typedef struct {
    int32_t latent_extent;
    int32_t latent_tile;
    double overlap;
    int32_t scale;
    int32_t blend_extent;
    int32_t row_limit;
} tb_axis;

/*
 * Partial GroupNorm statistics [DVA] of one part of the elements of one
 * (patch, sample, group): element count, the part's own mean, and the sum of
 * squared deviations about that mean.  16 bytes, no padding.  Each
 * (patch, sample, group) has TB_GN_PARTS records; the statistics kernel cuts
 * its elements into up to that many contiguous parts (how many depends on
 * the sizes and the GPU) and gives the unused records count 0.  A record
 * describes itself: the apply step reads all TB_GN_PARTS records of every
 * unit and merges those with a nonzero count, so record sets from different
 * statistics calls (other patch counts, other GPUs, other ranks) combine
 * freely.
 */
typedef struct {
    int64_t n;
    float mean;
    float m2;
} tb_gn_partial;

/* Partial-statistics records per (patch, sample, group). */
#define TB_GN_PARTS 8

/* Largest tile count per axis, and per grid, the stitch calls accept. */
#define TB_MAX_TILES_PER_AXIS 64
#define TB_MAX_TILES 1024

/* Library version as 10000 * major + 100 * minor + patch. */
size_t tb_version(void);

/* Static, human-readable name of a status code (never NULL). */
const char* tb_status_string(tb_status status);

/* The cudaError_t value behind the last TB_ERR_CUDA returned on the calling
 * thread (0 if none). */
int tb_last_cuda_error(void);

/*
 * tb_axis_layout -- the derived geometry of one axis (host only, no GPU).
 *   a            axis parameters (see tb_axis)
 *   cap          capacity of each output array
 *   n_tiles      out: number of tiles along the axis
 *   origins      out, may be NULL: tile n's origin in decoded samples,
 *                n * stride * scale, for n < min(n_tiles, cap)
 *   extents      out, may be NULL: L(n) for n < min(n_tiles, cap)
 *   blends       out, may be NULL: e(n), with e(0) = 0
 *   kept         out, may be NULL: K(n)
 *   out_extent   out, may be NULL: sum of K(n)
 * Returns TB_ERR_GEOMETRY for latent_extent < 0, latent_tile < 1, scale < 1,
 * an overlap outside [0, 1) or one that leaves a zero stride, or a derived
 * row_limit < 1; TB_ERR_UNSUPPORTED if the axis has more than
 * TB_MAX_TILES_PER_AXIS tiles (n_tiles is still written).
 */
tb_status tb_axis_layout(const tb_axis* a, int32_t cap, int32_t* n_tiles, int64_t* origins, int32_t* extents,
                         int32_t* blends, int32_t* kept, int64_t* out_extent);

/*
 * tb_stitch2d -- stitch a 2D grid of decoded tiles into one image [VTB]:
 * the result of visiting the tiles in row-major order, cross-fading each
 * tile's first e_y(i) rows with the already-blended tile above (blend_v),
 * then its first e_x(j) columns with the already-blended tile to its left
 * (blend_h), in place, each blend
 *     b[c] = rnd(rnd(a[L_a - e + c] * (float)(1 - c/e)) + rnd(b[c] * (float)(c/e)))
 * with the quotients taken in double, the products and the sum in fp32 and
 * rnd() round-to-nearest-even into the storage dtype; then cropping every
 * tile to K_y(i) x K_x(j) and concatenating.  The output equals that
 * sequence bit for bit.  Each output element is computed in one pass from
 * at most 4 tiles (the closed form of the recurrence).
 *
 *   tiles     host array of n_y * n_x device pointers, row-major (i, j);
 *             tile (i, j) is [B, C, L_y(i), L_x(j)] of `dtype`.  Read only:
 *             unlike the pages' loops, tiles are NOT modified.
 *   dtype     storage type of tiles and output
 *   B, C      batch and channels (>= 0; 0 launches nothing)
 *   ay, ax    height and width axes of the grid
 *   out       device pointer, [B, C, out_h, out_w]; must not overlap a tile
 *   out_h/w   must equal the sum of kept extents of ay / ax
 * Errors: TB_ERR_NULL (tiles, a tile, out, ay or ax NULL with work to do),
 * TB_ERR_SHAPE (out_h/out_w mismatch, negative sizes), TB_ERR_GEOMETRY,
 * TB_ERR_UNSUPPORTED (more than TB_MAX_TILES tiles, or blend bands that
 * reach each other: every middle tile n must have L(n) >= e(n) + e(n+1) --
 * true of whole middle tiles whenever overlap <= 1/2), TB_ERR_CUDA.
 */
tb_status tb_stitch2d(const void* const* tiles, tb_dtype dtype, int64_t B, int64_t C, const tb_axis* ay,
                      const tb_axis* ax, void* out, int64_t out_h, int64_t out_w, void* stream);

/*
 * tb_stitch3d -- stitch a 3D grid of decoded video tiles [VTB]: as
 * tb_stitch2d with a leading frame axis; tiles are visited in row-major
 * order over (k, i, j) and each tile is blended along time (blend_t, against
 * the already-blended tile k-1), then height (blend_v), then width
 * (blend_h); crop to K_t x K_y x K_x and concatenate.  Each output element
 * is computed from at most 8 tiles.
 *
 *   tiles     host array of n_t * n_y * n_x device pointers, row-major
 *             (k, i, j); tile (k, i, j) is [B, C, L_t(k), L_y(i), L_x(j)]
 *   at        frame axis (typically scale 1: latent_extent in frames)
 *   out       [B, C, out_t, out_h, out_w]
 * Errors as tb_stitch2d.
 */
tb_status tb_stitch3d(const void* const* tiles, tb_dtype dtype, int64_t B, int64_t C, const tb_axis* at,
                      const tb_axis* ay, const tb_axis* ax, void* out, int64_t out_t, int64_t out_h,
                      int64_t out_w, void* stream);

/*
 * Row-sharded stitch [DVA], the halo-exchange commits: the tile rows of the
 * height axis are shared out among `world` ranks, each rank decodes and
 * stitches its own rows, and before stitching, rank r receives from rank
 * r - 1 the raw rows its first tile row blends with: the last e_y(row_begin)
 * rows of every tile of rank r - 1's last tile row (one message per rank
 * boundary).  The ranks' outputs, concatenated in rank order along the
 * height, equal the unsharded stitch bit for bit.
 *
 * tb_shard_layout describes one rank's share:
 *   row_begin, row_end  tile rows [row_begin, row_end) of the height axis,
 *                       shared out in rank order as evenly as they go, the
 *                       first ranks one row more (empty past the row count)
 *   out_row_begin       first output row the rank writes
 *   out_rows            output rows it writes (sum of its rows' kept extents)
 *   halo_rows           rows of the band it receives: e_y(row_begin), or 0
 *                       when it needs none (first rank, empty share, or no
 *                       blend between the two rows)
 *   halo_elems          elements of that band (every frame tile and width
 *                       tile of row row_begin - 1, every plane): the size of
 *                       the message it receives
 *   send_elems          elements of the band it sends to rank + 1, or 0
 */
typedef struct {
    int32_t row_begin;
    int32_t row_end;
    int64_t out_row_begin;
    int64_t out_rows;
    int32_t halo_rows;
    int64_t halo_elems;
    int64_t send_elems;
} tb_shard_layout;

/*
 * tb_stitch_shard_layout -- rank `rank`'s share of a row-sharded stitch of
 * the grid (at, ay, ax) (at NULL for a 2D grid) with B x C planes (host only,
 * no GPU).
 * Errors: TB_ERR_NULL (ay, ax or out NULL), TB_ERR_SHAPE (negative sizes,
 * world < 1, rank outside [0, world)), TB_ERR_GEOMETRY, TB_ERR_UNSUPPORTED
 * (as tb_axis_layout).
 */
tb_status tb_stitch_shard_layout(const tb_axis* at, const tb_axis* ay, const tb_axis* ax, int64_t B, int64_t C,
                                 int32_t world, int32_t rank, tb_shard_layout* out);

/*
 * tb_stitch_halo_pack -- the band a rank sends to its successor: the last
 * e_y(row + 1) rows (raw, as decoded) of every tile of tile row `row`, packed
 * into one dense device buffer, tile by tile in row-major (k, j) order,
 * each [B, C, L_t(k), e_y(row + 1), L_x(j)] (L_t = 1 for a 2D grid).
 *
 *   tiles   host array of the device pointers of tile row `row`: n_x tiles
 *           (2D, at NULL), or n_t * n_x tiles row-major over (k, j) (3D)
 *   row     0 .. n_y - 2
 *   halo    device buffer of send_elems elements of `dtype` (see
 *           tb_shard_layout); must not overlap a tile
 * Nothing is launched when e_y(row + 1) is 0.
 * Errors: TB_ERR_NULL, TB_ERR_DTYPE, TB_ERR_SHAPE (row out of range,
 * negative sizes), TB_ERR_GEOMETRY, TB_ERR_UNSUPPORTED (more than 512 tiles
 * in the row), TB_ERR_CUDA.
 */
tb_status tb_stitch_halo_pack(const void* const* tiles, tb_dtype dtype, int64_t B, int64_t C, const tb_axis* at,
                              const tb_axis* ay, const tb_axis* ax, int32_t row, void* halo, void* stream);

/*
 * tb_stitch2d_shard -- rows [row_begin, row_end) of the tile grid stitched
 * as tb_stitch2d would stitch them in the whole grid: the output rows
 * [out_row_begin, out_row_begin + out_rows) of the full image, written to
 * `out` ([B, C, out_rows, out_w]).
 *
 *   tiles     host array of (row_end - row_begin) * n_x device pointers,
 *             row-major; tile (i, j) of the grid is entry
 *             (i - row_begin) * n_x + j
 *   halo      device pointer to the band tb_stitch_halo_pack made of row
 *             row_begin - 1, received from the rank before; required when
 *             row_begin > 0 and e_y(row_begin) > 0, else ignored
 *   out_rows  the sum of the kept extents of rows [row_begin, row_end)
 * Errors as tb_stitch2d, plus TB_ERR_SHAPE for a row range outside
 * [0, n_y] or out_rows that does not match it.
 */
tb_status tb_stitch2d_shard(const void* const* tiles, const void* halo, tb_dtype dtype, int64_t B, int64_t C,
                            const tb_axis* ay, const tb_axis* ax, int32_t row_begin, int32_t row_end, void* out,
                            int64_t out_rows, int64_t out_w, void* stream);

/*
 * tb_stitch3d_shard -- as tb_stitch2d_shard for a video grid, sharded along
 * the height: tiles holds n_t * (row_end - row_begin) * n_x pointers,
 * row-major over (k, i - row_begin, j); `halo` the 3D band of row
 * row_begin - 1; `out` is [B, C, out_t, out_rows, out_w].
 */
tb_status tb_stitch3d_shard(const void* const* tiles, const void* halo, tb_dtype dtype, int64_t B, int64_t C,
                            const tb_axis* at, const tb_axis* ay, const tb_axis* ax, int32_t row_begin,
                            int32_t row_end, void* out, int64_t out_t, int64_t out_rows, int64_t out_w,
                            void* stream);

/*
 * Frame-sharded video stitch: the same partition along the time axis of a 3D
 * grid.  The frame tiles are dealt to the ranks; before stitching, rank r
 * receives the raw last e_t(frame_begin) frames of every tile of rank
 * r - 1's last frame tile.  The ranks' outputs, concatenated along the
 * frames, equal tb_stitch3d bit for bit.
 *
 * tb_stitch_shard_frames_layout -- as tb_stitch_shard_layout, with the
 * fields counting frame tiles and output frames (row_begin/row_end: frame
 * tiles; out_row_begin/out_rows: output frames; halo_rows: e_t(frame_begin));
 * `at` is required.
 */
tb_status tb_stitch_shard_frames_layout(const tb_axis* at, const tb_axis* ay, const tb_axis* ax, int64_t B,
                                        int64_t C, int32_t world, int32_t rank, tb_shard_layout* out);

/*
 * tb_stitch_halo_pack_frames -- the band a rank sends to its successor along
 * the time axis: the last e_t(frame_tile + 1) frames of every tile of frame
 * tile `frame_tile`, packed tile by tile in row-major (i, j) order, each
 * [B, C, e_t(frame_tile + 1), L_y(i), L_x(j)].
 *   tiles       host array of the n_y * n_x device pointers of the frame
 *               tile, row-major (i, j)
 *   frame_tile  0 .. n_t - 2
 *   halo        device buffer of send_elems elements (see
 *               tb_stitch_shard_frames_layout)
 * Errors as tb_stitch_halo_pack.
 */
tb_status tb_stitch_halo_pack_frames(const void* const* tiles, tb_dtype dtype, int64_t B, int64_t C,
                                     const tb_axis* at, const tb_axis* ay, const tb_axis* ax, int32_t frame_tile,
                                     void* halo, void* stream);

/*
 * tb_stitch3d_shard_frames -- frame tiles [frame_begin, frame_end) of a video
 * grid stitched as tb_stitch3d would stitch them in the whole grid, into
 * `out` ([B, C, out_frames, out_h, out_w]: the output frames
 * [out_row_begin, out_row_begin + out_frames) of the full video).
 *   tiles   host array of (frame_end - frame_begin) * n_y * n_x device
 *           pointers, row-major over (k - frame_begin, i, j)
 *   halo    the band tb_stitch_halo_pack_frames made of frame tile
 *           frame_begin - 1; required when frame_begin > 0 and
 *           e_t(frame_begin) > 0, else ignored
 * Errors as tb_stitch3d, plus TB_ERR_SHAPE for a frame range outside
 * [0, n_t] or out_frames that does not match it.
 */
tb_status tb_stitch3d_shard_frames(const void* const* tiles, const void* halo, tb_dtype dtype, int64_t B, int64_t C,
                                   const tb_axis* at, const tb_axis* ay, const tb_axis* ax, int32_t frame_begin,
                                   int32_t frame_end, void* out, int64_t out_frames, int64_t out_h, int64_t out_w,
                                   void* stream);

/*
 * One axis of a normalised-ramp tile layout [STU]: n_tiles tiles of one
 * extent, placed by the caller (a planner spreads them so the first starts at
 * 0 and the last ends at out_extent).
 *   n_tiles      1 .. TB_MAX_TILES_PER_AXIS
 *   tile_extent  samples per tile (>= 1)
 *   out_extent   samples of the canvas
 *   zero         samples of zero weight next to an edge shared with another
 *                tile (4 latents * scale on the page)
 *   ramp         samples over which the weight then rises to 1 (8 latents *
 *                scale on the page; >= 1)
 *   origins      host array of n_tiles origins in samples, strictly
 *                ascending, origins[0] == 0, origins[n-1] + tile_extent ==
 *                out_extent
 * A tile's weight at distance d (samples) from a shared edge is
 * clamp((d - zero) / ramp, 0, 1); edges of the canvas carry no ramp.
 */
typedef struct {
    int32_t n_tiles;
    int32_t tile_extent;
    int32_t out_extent;
    int32_t zero;
    int32_t ramp;
    const int64_t* origins;
} tb_ramp_axis;

/*
 * tb_ramp_axis_spread -- one axis of a normalised-ramp layout as the Studio
 * planner lays it out [STU], commit "Decode this VAE in 32-latent tiles
 * ...": n_tiles tiles of latent_tile latents spread so the first starts at 0
 * and the last ends at the canvas edge, tile n at
 *     floor(n * (latent_extent - latent_tile) / (n_tiles - 1))  latents
 * (the page does not say how the spread rounds; flooring is the reading
 * taken), decoded at `scale` samples per latent, with a zero band of
 * zero_latents and a ramp of ramp_latents latents (4 and 8 on the page).
 * Host only.
 *   origins  out: host array of n_tiles entries, the origins in samples
 *   axis     out: the tb_ramp_axis for tb_stitch2d_ramp; axis->origins
 *            points to `origins`
 * Errors: TB_ERR_NULL; TB_ERR_GEOMETRY for n_tiles < 1, scale < 1,
 * latent_tile outside [1, latent_extent], a single tile that is not the
 * whole canvas, neighbouring origins further apart than a tile (samples
 * no tile covers), zero_latents < 0 or ramp_latents < 1;
 * TB_ERR_UNSUPPORTED for more than TB_MAX_TILES_PER_AXIS tiles or sizes
 * past 2^31 samples.
 */
tb_status tb_ramp_axis_spread(int32_t latent_extent, int32_t latent_tile, int32_t n_tiles, int32_t scale,
                              int32_t zero_latents, int32_t ramp_latents, int64_t* origins, tb_ramp_axis* axis);

/* Most tiles with positive weight at one position of a ramp axis. */
#define TB_RAMP_MAX_COVER 3

/*
 * tb_stitch2d_ramp -- stitch a 2D grid of equally sized overlapping tiles by
 * the normalised-ramp blend [STU]: every output sample is the average of the
 * tiles covering it, weighted by the product of each tile's ramps along both
 * axes, out = sum(w * x) / sum(w), computed in fp32 and rounded once into the
 * storage type.  Used for decoded tiles (scale = the VAE's) and for latent
 * tiles of a tiled encode (scale 1).
 *
 *   tiles     host array of ay->n_tiles * ax->n_tiles device pointers,
 *             row-major; every tile is [B, C, ay->tile_extent, ax->tile_extent]
 *   out       device [B, C, ay->out_extent, ax->out_extent]; must not
 *             overlap a tile
 * Errors: TB_ERR_NULL, TB_ERR_DTYPE, TB_ERR_SHAPE (negative sizes),
 * TB_ERR_GEOMETRY (origins out of order, not covering the canvas, or a
 * sample with no positive weight), TB_ERR_UNSUPPORTED (more than
 * TB_RAMP_MAX_COVER tiles with positive weight at one position, more than
 * TB_MAX_TILES tiles), TB_ERR_CUDA.
 */
tb_status tb_stitch2d_ramp(const void* const* tiles, tb_dtype dtype, int64_t B, int64_t C, const tb_ramp_axis* ay,
                           const tb_ramp_axis* ax, void* out, void* stream);

/*
 * tb_patch_gn_stats -- per-patch GroupNorm partial statistics [DVA].
 * An activation [N, C, *spatial] is split along one spatial axis into P
 * patches (the ranks' shards in the pages' patch-parallel decode); patch p is
 * [N, C, *spatial_p], contiguous, with spatial[p] elements per channel.
 * Channel c belongs to group c / (C / G).  The C/G channels of group g in
 * sample n of patch p are one run of elements; it is cut into up to
 * TB_GN_PARTS contiguous parts and part k's statistics go to
 *   partials[((p * N + n) * G + g) * TB_GN_PARTS + k]
 *     = { count, mean, sum (x - mean)^2 }
 * (fp32 accumulation, deterministic: the same inputs on the same GPU give
 * the same bits).  Records of unused parts get count 0.
 *
 *   patches   host array of P device pointers
 *   P         number of patches (1 = plain, unsharded GroupNorm)
 *   dtype     element type of the patches
 *   N, C      samples and channels; C % G == 0
 *   spatial   host array of P element counts per channel (>= 0)
 *   G         number of groups (>= 1)
 *   partials  device array of P * N * G * TB_GN_PARTS tb_gn_partial,
 *             written fully
 * Errors: TB_ERR_NULL, TB_ERR_SHAPE (C % G != 0, negative sizes, P < 1),
 * TB_ERR_UNSUPPORTED (P > 64, or P * N * G * TB_GN_PARTS above 2e9),
 * TB_ERR_CUDA.
 */
tb_status tb_patch_gn_stats(const void* const* patches, int32_t P, tb_dtype dtype, int64_t N, int64_t C,
                            const int64_t* spatial, int32_t G, tb_gn_partial* partials, void* stream);

/*
 * tb_patch_gn_apply -- combine the partials of all P patches (all their
 * parts) into the pooled group mean and the biased variance about it
 * (divided by the total count, no Bessel correction) [DVA], then normalise,
 * apply the per-channel affine and optionally SiLU:
 *     z = (x - mean) / sqrt(var + eps) * gamma[c] + beta[c]
 *     y = silu ? z / (1 + exp(-z)) : z,   rounded once into dtype.
 * The result equals GroupNorm (+ SiLU) of the unsharded tensor.
 *
 *   patches   host array of P device pointers (as tb_patch_gn_stats)
 *   outs      host array of P device pointers, same shapes; outs[p] may
 *             equal patches[p] (in place), other overlaps are not allowed
 *   partials  device array of P * N * G * TB_GN_PARTS records written by
 *             tb_patch_gn_stats for these patches (by one call over all P,
 *             or by several calls whose record sets lie back to back in
 *             patch order); every record is read and those with count 0
 *             are skipped
 *   gamma     device [C] of dtype, or NULL for 1
 *   beta      device [C] of dtype, or NULL for 0
 *   eps       added to the variance (> 0 recommended; >= 0 required)
 *   silu      nonzero applies SiLU
 * Equivalent to tb_patch_gn_apply_gathered with R = P.
 * Errors as tb_patch_gn_stats, plus TB_ERR_SHAPE for eps < 0 or NaN.
 */
tb_status tb_patch_gn_apply(const void* const* patches, void* const* outs, int32_t P, tb_dtype dtype, int64_t N,
                            int64_t C, const int64_t* spatial, int32_t G, const tb_gn_partial* partials,
                            const void* gamma, const void* beta, float eps, int32_t silu, void* stream);

/*
 * tb_patch_gn_apply_gathered -- the apply step of a sharded PatchGroupNorm
 * [DVA]: each rank holds only its own patch(es), has run tb_patch_gn_stats
 * on them, and has gathered every rank's records (one all-gather of
 * N * G * TB_GN_PARTS records per patch, in place of the page's two
 * all-reduces per norm).  This call pools the statistics of all R record
 * sets and normalises the P local patches with them.
 *
 *   patches, outs, P, dtype, N, C, spatial, G, gamma, beta, eps, silu
 *             as tb_patch_gn_apply, describing only the local patches
 *   partials  device array of R record sets of [N][G][TB_GN_PARTS] records,
 *             back to back: the records of every patch of the whole tensor
 *             (the local ones included), in any order
 *   R         record sets in `partials` (>= 1; the total patch count)
 * The pooled mean and variance are those of every element described by the
 * records; the call cannot check that they describe the same tensor as the
 * local patches.
 * Errors as tb_patch_gn_apply, plus TB_ERR_SHAPE for R < 1 and
 * TB_ERR_UNSUPPORTED for R > 65536 or R * N * G * TB_GN_PARTS above 2e9.
 */
tb_status tb_patch_gn_apply_gathered(const void* const* patches, void* const* outs, int32_t P, tb_dtype dtype,
                                     int64_t N, int64_t C, const int64_t* spatial, int32_t G,
                                     const tb_gn_partial* partials, int32_t R, const void* gamma, const void* beta,
                                     float eps, int32_t silu, void* stream);

/*
 * tb_device_status -- the library's device-side status word on the current
 * device.  Kernels never trap: a kernel that cannot complete a piece of work
 * (a wait for its tensor copies that exceeds about one second; in a build
 * with bounds checks, an index outside its tile or output) records a code
 * and skips that work.  The first code recorded stays until cleared.
 *   code    out: 0 (TB_DEV_OK) or the first code recorded
 *   clear   nonzero resets the word to 0 after reading it
 * Synchronises with the device (a blocking copy from the word).  Errors:
 * TB_ERR_NULL, TB_ERR_CUDA.
 */
#define TB_DEV_OK 0u
#define TB_DEV_WAIT_TIMEOUT 1u
#define TB_DEV_OUT_OF_BOUNDS 2u
tb_status tb_device_status(uint32_t* code, int32_t clear);

/* Most patches (ranks) one Patchify split or patch gather handles. */
#define TB_MAX_PATCHES 64

/*
 * tb_patchify_layout -- the ranks' bands of one axis (host only, no GPU)
 * [DVA], Patchify: the axis is cut into bands of `factor` positions (the
 * factor by which the VAE narrows or widens it), the bands are shared out
 * in rank order as evenly as they go, and when they do not divide evenly the
 * first ranks get one band more.  No position is invented or dropped.
 *   extent   positions along the axis; a whole number of bands (>= 0)
 *   factor   positions per band (>= 1)
 *   P        ranks (1 .. TB_MAX_PATCHES)
 *   starts   out, may be NULL: P offsets of the bands along the axis
 *   sizes    out, may be NULL: P band extents (multiples of factor; 0 for
 *            ranks past the band count)
 * Errors: TB_ERR_SHAPE (extent < 0, factor < 1, P < 1, extent not a
 * multiple of factor), TB_ERR_UNSUPPORTED (P > TB_MAX_PATCHES).
 */
tb_status tb_patchify_layout(int64_t extent, int32_t factor, int32_t P, int64_t* starts, int64_t* sizes);

/*
 * tb_patchify -- cut a tensor into the P ranks' patches along `axis` by the
 * bands of tb_patchify_layout [DVA], one device copy for all of them.
 *
 *   x        device pointer, dense row-major tensor of `shape`
 *   dtype    element type (only its size matters: the copy is bit exact)
 *   ndim     1 .. 8;  shape: host array of ndim extents (>= 0)
 *   axis     0 .. ndim-1, the split axis; shape[axis] must be a whole
 *            number of bands
 *   factor   band extent (>= 1);  P: ranks (1 .. TB_MAX_PATCHES)
 *   slot     0: patch p is the dense tensor of `shape` with shape[axis]
 *            replaced by sizes[p].  > 0: every patch buffer holds `slot`
 *            positions along the axis (slot >= the largest band), as the
 *            equal-shape buffers of a collective all-gather; band p fills
 *            the first sizes[p] of them and the rest are left untouched
 *   patches  host array of P device pointers (a pointer of an empty patch
 *            may be NULL); no patch may overlap x or another patch
 * Errors: TB_ERR_NULL, TB_ERR_DTYPE, TB_ERR_SHAPE (ndim, axis, negative
 * extents, a partial band, 0 < slot < largest band, slot < 0),
 * TB_ERR_UNSUPPORTED (P > TB_MAX_PATCHES, more than 2^31 - 1 rows before
 * the axis or elements in one row of a patch), TB_ERR_CUDA.
 */
tb_status tb_patchify(const void* x, tb_dtype dtype, int32_t ndim, const int64_t* shape, int32_t axis,
                      int32_t factor, int32_t P, int64_t slot, void* const* patches, void* stream);

/*
 * tb_gather_patches -- reassemble the tensor from the P ranks' patches
 * [DVA], gather_patches: the sizes along `axis` are given (the exchange
 * of sizes that comes first on the page), each patch is read without its
 * padding, and the patches are concatenated in rank order.  One device copy.
 *
 *   patches  host array of P device pointers (NULL allowed for size 0)
 *   P        1 .. TB_MAX_PATCHES
 *   sizes    host array of P extents along the axis (>= 0), summing to
 *            shape[axis]; any sizes, not only tb_patchify_layout's
 *   dtype, ndim, axis   as tb_patchify; shape: the gathered tensor
 *   slot     0: dense patches; > 0: every patch buffer has `slot`
 *            positions along the axis and only the first sizes[p] are read
 *   out      device pointer to the gathered tensor; must not overlap a patch
 * Errors as tb_patchify (TB_ERR_SHAPE also when the sizes do not sum to
 * shape[axis]).
 */
tb_status tb_gather_patches(const void* const* patches, int32_t P, const int64_t* sizes, tb_dtype dtype, int32_t ndim,
                            const int64_t* shape, int32_t axis, int64_t slot, void* out, void* stream);

/*
 * tb_patch_group_norm_noalloc -- PatchGroupNorm (statistics, then pooled
 * normalisation, affine and optional SiLU) for callers that cannot allocate
 * device memory.  The pages have no counterpart: it exists for this
 * library's users.
 *
 * Some callers may not call cudaMalloc at all: code embedded in a host
 * framework that owns every device allocation through its own memory pool,
 * or code on a latency-critical path where an allocation (which can
 * synchronise the device) is not allowed.  Such a caller still owns the
 * inputs and outputs, but cannot provide the partials buffer that
 * tb_patch_gn_stats / tb_patch_gn_apply exchange.  This call keeps those
 * partials in a fixed scratch array compiled into the library instead
 * (TB_NOALLOC_MAX_PARTIALS records of 16 bytes, 1 MiB, held on every GPU
 * that loads the library until the process exits) and allocates nothing.
 * That holds the records of P * N * G <= TB_NOALLOC_MAX_PARTIALS /
 * TB_GN_PARTS = 8192 (patch, sample, group) triples.
 *
 * Arguments and results are those of tb_patch_gn_apply, minus `partials`.
 * The result equals tb_patch_gn_stats followed by tb_patch_gn_apply.
 *
 *   - P * N * G * TB_GN_PARTS larger than TB_NOALLOC_MAX_PARTIALS returns
 *     TB_ERR_UNSUPPORTED and launches nothing.
 *   - The first call on each device looks up the scratch array's device
 *     address (cudaGetSymbolAddress, with that device current).  The
 *     address belongs to the device's CUDA context: after cudaDeviceReset
 *     (or any other teardown of the context) the next call finds a new
 *     context id and looks the address up again.
 *   - Every call uses the same scratch array.  Each call writes every record
 *     it reads before reading it, so nothing needs clearing, but two calls
 *     whose work overlaps on the GPU (different streams, or different host
 *     threads, without ordering between them) race on the array and may give
 *     wrong results.  Order such calls on one stream.
 * Errors as tb_patch_gn_apply; TB_ERR_CUDA also if the address lookup fails.
 */
#define TB_NOALLOC_MAX_PARTIALS 65536
tb_status tb_patch_group_norm_noalloc(const void* const* patches, void* const* outs, int32_t P, tb_dtype dtype,
                                      int64_t N, int64_t C, const int64_t* spatial, int32_t G, const void* gamma,
                                      const void* beta, float eps, int32_t silu, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TILEBLEND_H */
