/*
 * oracle/stitch.c -- CPU oracle for tiled-VAE tile stitching.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link or call this file.  Only the test
 * suite, the package smoke check and the benchmark's CPU-baseline leg use it.
 * It shares no code, header or table with the CUDA library.
 *
 * What it computes: diffusers' tiled decode as described on the page
 * "[Proposal] Vectorize tiled VAE blending while preserving rounding and CUDA
 * graph replay" (diffusers issue #14722, "Proposed scope"): every tile is
 * visited in row-major order; a tile is first cross-faded with the already
 * blended tile before it in time (blend_t), then with the already blended
 * tile above it (blend_v), then with the already blended tile to its left
 * (blend_h).  Blending happens in place, so later tiles see blended
 * neighbours.  Each blend clamps its extent to
 *     e = min(extent of the neighbour, extent of the tile, blend_extent)
 * and rewrites the first e slices of the tile as
 *     b[c] = a[La - e + c] * (1 - c/e) + b[c] * (c/e),   c = 0 .. e-1.
 * Afterwards every tile is cropped to its first row_limit slices per axis
 * and the crops are concatenated.
 *
 * Rounding (the same page, same section: each product is rounded on its
 * own, and the coefficients come from double-precision division so that
 * they equal Python's float quotients): the two coefficients are computed
 * in double precision and used as fp32 scalars;
 * each product is one fp32 multiply rounded to the storage type; the sum of
 * the two rounded products is one fp32 add rounded to the storage type.
 * Round-to-nearest-even into fp16 and bf16 is written out below from the
 * IEEE-754 definition.  A fourth storage mode, ORC_F64, keeps everything in
 * double with double coefficients and no narrowing, so that the recurrence
 * can be checked against its algebraic closed form.
 *
 * The oracle makes no assumption about how far a blend band reaches: it runs
 * the literal recurrence on private copies of the tiles.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -shared -fPIC (contraction of a
 * multiply and an add into one fused operation would change the rounding).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_F64 = 3 };

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary formats                                                   */
/* ------------------------------------------------------------------------ */

/* A binary floating-point format: precision p (significand bits including
 * the implicit one), exponent field width, and exponent bias (= emax). */
typedef struct {
    int prec;
    int ebits;
    int bias;
} orc_format;

static const orc_format FMT_F16 = {11, 5, 15};
static const orc_format FMT_BF16 = {8, 8, 127};

static int bit_length_u64(uint64_t v) {
    int n = 0;
    while (v) {
        ++n;
        v >>= 1;
    }
    return n;
}

/*
 * Round the exact finite value (-1)^sign * mant * 2^exp2 to the nearest
 * member of `f`, ties to the member whose last significand bit is 0, and
 * return its bit pattern.  Values beyond the largest finite member after
 * rounding become infinity; values below half the smallest subnormal become
 * a signed zero.
 */
static uint32_t round_exact_to_format(int sign, uint64_t mant, int exp2, orc_format f) {
    const uint32_t sign_bit = (uint32_t)sign << (f.ebits + f.prec - 1);
    if (mant == 0) return sign_bit;
    const int emin = 1 - f.bias;
    const int emax = f.bias;
    /* exponent of the leading bit: |x| in [2^E, 2^(E+1)) */
    const int E = exp2 + bit_length_u64(mant) - 1;
    /* spacing of the format's members around |x|: 2^qe */
    int qe = (E > emin ? E : emin) - (f.prec - 1);
    const int shift = qe - exp2;
    uint64_t n;
    if (shift <= 0) {
        n = mant << (-shift); /* exact: |x| is already a multiple of 2^qe */
    } else if (shift >= 64) {
        n = 0; /* |x| < 2^63 * 2^exp2 <= 2^(qe-1): below half a spacing */
    } else {
        n = mant >> shift;
        const uint64_t rem = mant & ((UINT64_C(1) << shift) - 1);
        const uint64_t half = UINT64_C(1) << (shift - 1);
        if (rem > half || (rem == half && (n & 1))) n += 1;
    }
    /* |result| = n * 2^qe */
    const uint64_t hidden = UINT64_C(1) << (f.prec - 1);
    if (n == 0) return sign_bit;
    if (n < hidden) {
        /* subnormal: exponent field 0, qe is the subnormal spacing */
        return sign_bit | (uint32_t)n;
    }
    if (n == (hidden << 1)) { /* rounding carried into the next binade */
        n = hidden;
        qe += 1;
    }
    const int biased = qe + (f.prec - 1) + f.bias;
    if (biased > 2 * emax) { /* overflow to infinity */
        return sign_bit | (((UINT32_C(1) << f.ebits) - 1) << (f.prec - 1));
    }
    return sign_bit | ((uint32_t)biased << (f.prec - 1)) | (uint32_t)(n - hidden);
}

static uint32_t nan_of_format(int sign, orc_format f) {
    const uint32_t sign_bit = (uint32_t)sign << (f.ebits + f.prec - 1);
    const uint32_t exp_all = ((UINT32_C(1) << f.ebits) - 1) << (f.prec - 1);
    return sign_bit | exp_all | (UINT32_C(1) << (f.prec - 2)); /* quiet NaN */
}

static uint32_t inf_of_format(int sign, orc_format f) {
    const uint32_t sign_bit = (uint32_t)sign << (f.ebits + f.prec - 1);
    return sign_bit | (((UINT32_C(1) << f.ebits) - 1) << (f.prec - 1));
}

/* Round a binary32 value, given by its bits, into format f. */
static uint32_t round_f32_bits(uint32_t bits, orc_format f) {
    const int sign = (int)(bits >> 31);
    const uint32_t be = (bits >> 23) & 0xFFu;
    const uint32_t frac = bits & 0x7FFFFFu;
    if (be == 0xFFu) return frac ? nan_of_format(sign, f) : inf_of_format(sign, f);
    if (be == 0) return round_exact_to_format(sign, frac, -149, f);
    return round_exact_to_format(sign, (uint64_t)frac | (UINT64_C(1) << 23), (int)be - 150, f);
}

/* Round a binary64 value, given by its bits, into format f (one rounding). */
static uint32_t round_f64_bits(uint64_t bits, orc_format f) {
    const int sign = (int)(bits >> 63);
    const uint32_t be = (uint32_t)((bits >> 52) & 0x7FFu);
    const uint64_t frac = bits & ((UINT64_C(1) << 52) - 1);
    if (be == 0x7FFu) return frac ? nan_of_format(sign, f) : inf_of_format(sign, f);
    if (be == 0) return round_exact_to_format(sign, frac, -1074, f);
    return round_exact_to_format(sign, frac | (UINT64_C(1) << 52), (int)be - 1075, f);
}

/* Exact value of a member of format f, given by its bits, as a double. */
static double decode_format(uint32_t bits, orc_format f) {
    const int sign = (int)(bits >> (f.ebits + f.prec - 1)) & 1;
    const uint32_t be = (bits >> (f.prec - 1)) & ((UINT32_C(1) << f.ebits) - 1);
    const uint32_t frac = bits & ((UINT32_C(1) << (f.prec - 1)) - 1);
    double v;
    if (be == (UINT32_C(1) << f.ebits) - 1) {
        v = frac ? NAN : INFINITY;
    } else if (be == 0) {
        v = ldexp((double)frac, 1 - f.bias - (f.prec - 1));
    } else {
        v = ldexp((double)(frac | (UINT32_C(1) << (f.prec - 1))), (int)be - f.bias - (f.prec - 1));
    }
    return sign ? -v : v;
}

static uint32_t f32_bits(float x) {
    uint32_t b;
    memcpy(&b, &x, 4);
    return b;
}

static uint64_t f64_bits(double x) {
    uint64_t b;
    memcpy(&b, &x, 8);
    return b;
}

/* Exported conversion entry points (used by the oracle's own pins and by the
 * GroupNorm oracle's final rounding). */
uint16_t orc_f32_to_f16(float x) { return (uint16_t)round_f32_bits(f32_bits(x), FMT_F16); }
uint16_t orc_f32_to_bf16(float x) { return (uint16_t)round_f32_bits(f32_bits(x), FMT_BF16); }
uint16_t orc_f64_to_f16(double x) { return (uint16_t)round_f64_bits(f64_bits(x), FMT_F16); }
uint16_t orc_f64_to_bf16(double x) { return (uint16_t)round_f64_bits(f64_bits(x), FMT_BF16); }
double orc_f16_value(uint16_t b) { return decode_format(b, FMT_F16); }
double orc_bf16_value(uint16_t b) { return decode_format(b, FMT_BF16); }

void orc_f32_to_f16_array(const float* x, uint16_t* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = orc_f32_to_f16(x[i]);
}
void orc_f32_to_bf16_array(const float* x, uint16_t* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = orc_f32_to_bf16(x[i]);
}
void orc_f64_to_f16_array(const double* x, uint16_t* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = orc_f64_to_f16(x[i]);
}
void orc_f64_to_bf16_array(const double* x, uint16_t* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = orc_f64_to_bf16(x[i]);
}
void orc_f16_to_f64_array(const uint16_t* x, double* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = orc_f16_value(x[i]);
}
void orc_bf16_to_f64_array(const uint16_t* x, double* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = orc_bf16_value(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Storage access                                                            */
/* ------------------------------------------------------------------------ */

static size_t elem_size(int dt) {
    switch (dt) {
        case ORC_F32: return 4;
        case ORC_F16: return 2;
        case ORC_BF16: return 2;
        case ORC_F64: return 8;
    }
    return 0;
}

/* The stored value at index i, widened exactly to float (narrow types). */
static float load_narrow(int dt, const void* base, int64_t i) {
    switch (dt) {
        case ORC_F32: return ((const float*)base)[i];
        case ORC_F16: return (float)orc_f16_value(((const uint16_t*)base)[i]);
        default: return (float)orc_bf16_value(((const uint16_t*)base)[i]);
    }
}

/* rnd_S: round an fp32 value into the storage type and return it widened. */
static float round_to_storage(int dt, float x) {
    switch (dt) {
        case ORC_F32: return x;
        case ORC_F16: return (float)orc_f16_value(orc_f32_to_f16(x));
        default: return (float)orc_bf16_value(orc_f32_to_bf16(x));
    }
}

static void store_narrow(int dt, void* base, int64_t i, float x_representable) {
    switch (dt) {
        case ORC_F32: ((float*)base)[i] = x_representable; break;
        case ORC_F16: ((uint16_t*)base)[i] = orc_f32_to_f16(x_representable); break;
        default: ((uint16_t*)base)[i] = orc_f32_to_bf16(x_representable); break;
    }
}

/*
 * One element of one blend: b[ib] <- a[ia] * (1 - c/e) + b[ib] * (c/e).
 * The coefficients are Python-double quotients; for the narrow storage types
 * they enter the arithmetic as fp32 scalars.
 */
static void blend_element(int dt, const void* a, int64_t ia, void* b, int64_t ib, int c, int e) {
    const double w_d = (double)c / (double)e;
    const double u_d = 1.0 - (double)c / (double)e;
    if (dt == ORC_F64) {
        const double pa = ((const double*)a)[ia] * u_d;
        const double pb = ((double*)b)[ib] * w_d;
        ((double*)b)[ib] = pa + pb;
        return;
    }
    const float u = (float)u_d;
    const float w = (float)w_d;
    const float pa = round_to_storage(dt, load_narrow(dt, a, ia) * u);
    const float pb = round_to_storage(dt, load_narrow(dt, b, ib) * w);
    const float s = round_to_storage(dt, pa + pb);
    store_narrow(dt, b, ib, s);
}

/* ------------------------------------------------------------------------ */
/* The tiled-decode stitch                                                   */
/* ------------------------------------------------------------------------ */

/* A tile of shape [B, C, Lt, Ly, Lx], contiguous. */
typedef struct {
    void* data;
    int64_t Lt, Ly, Lx;
} orc_tile;

static int64_t tile_index(const orc_tile* t, int64_t plane, int64_t ct, int64_t cy, int64_t cx) {
    return ((plane * t->Lt + ct) * t->Ly + cy) * t->Lx + cx;
}

static int64_t min3(int64_t a, int64_t b, int64_t c) {
    int64_t m = a < b ? a : b;
    return m < c ? m : c;
}

/* blend_t: cross-fade the first e frames of b with the last e frames of a. */
static void blend_t(int dt, int64_t planes, const orc_tile* a, orc_tile* b, int64_t blend_extent) {
    const int64_t e = min3(a->Lt, b->Lt, blend_extent);
    for (int64_t c = 0; c < e; ++c)
        for (int64_t p = 0; p < planes; ++p)
            for (int64_t y = 0; y < b->Ly; ++y)
                for (int64_t x = 0; x < b->Lx; ++x)
                    blend_element(dt, a->data, tile_index(a, p, a->Lt - e + c, y, x), b->data,
                                  tile_index(b, p, c, y, x), (int)c, (int)e);
}

/* blend_v: cross-fade the first e rows of b with the last e rows of a. */
static void blend_v(int dt, int64_t planes, const orc_tile* a, orc_tile* b, int64_t blend_extent) {
    const int64_t e = min3(a->Ly, b->Ly, blend_extent);
    for (int64_t c = 0; c < e; ++c)
        for (int64_t p = 0; p < planes; ++p)
            for (int64_t t = 0; t < b->Lt; ++t)
                for (int64_t x = 0; x < b->Lx; ++x)
                    blend_element(dt, a->data, tile_index(a, p, t, a->Ly - e + c, x), b->data,
                                  tile_index(b, p, t, c, x), (int)c, (int)e);
}

/* blend_h: cross-fade the first e columns of b with the last e columns of a. */
static void blend_h(int dt, int64_t planes, const orc_tile* a, orc_tile* b, int64_t blend_extent) {
    const int64_t e = min3(a->Lx, b->Lx, blend_extent);
    for (int64_t c = 0; c < e; ++c)
        for (int64_t p = 0; p < planes; ++p)
            for (int64_t t = 0; t < b->Lt; ++t)
                for (int64_t y = 0; y < b->Ly; ++y)
                    blend_element(dt, a->data, tile_index(a, p, t, y, a->Lx - e + c), b->data,
                                  tile_index(b, p, t, y, c), (int)c, (int)e);
}

/*
 * orc_stitch -- run the tiled-decode blend recurrence, crop and concatenate.
 *
 *   dt          storage type (ORC_F32, ORC_F16, ORC_BF16, ORC_F64)
 *   planes      B * C (batch times channels; the blend treats them alike)
 *   ntiles[3]   tile counts along t, y, x (a 2D grid passes ntiles[0] = 1)
 *   ext_t/y/x   tile extents along each axis, ntiles[a] entries each
 *   blend[3]    blend_extent along t, y, x
 *   limit[3]    row_limit along t, y, x (a tile keeps min(extent, limit))
 *   tiles       ntiles[0]*ntiles[1]*ntiles[2] host pointers, row-major over
 *               (k, i, j); tile (k,i,j) is [planes, ext_t[k], ext_y[i], ext_x[j]]
 *   out         [planes, sum kept_t, sum kept_y, sum kept_x], written fully
 *
 * Returns 0 on success, -1 if memory for the private copies runs out.
 * The input tiles are not modified.
 */
int orc_stitch(int dt, int64_t planes, const int32_t* ntiles, const int32_t* ext_t,
               const int32_t* ext_y, const int32_t* ext_x, const int32_t* blend,
               const int32_t* limit, const void* const* tiles, void* out) {
    const int64_t nt = ntiles[0], ny = ntiles[1], nx = ntiles[2];
    const int64_t ntot = nt * ny * nx;
    const size_t es = elem_size(dt);
    orc_tile* buf = (orc_tile*)calloc((size_t)(ntot > 0 ? ntot : 1), sizeof(orc_tile));
    if (!buf) return -1;
    int rc = 0;
    /* private copies: the recurrence mutates tiles in place */
    for (int64_t k = 0; k < nt && rc == 0; ++k)
        for (int64_t i = 0; i < ny && rc == 0; ++i)
            for (int64_t j = 0; j < nx; ++j) {
                orc_tile* t = &buf[(k * ny + i) * nx + j];
                t->Lt = ext_t[k];
                t->Ly = ext_y[i];
                t->Lx = ext_x[j];
                const size_t bytes = (size_t)(planes * t->Lt * t->Ly * t->Lx) * es;
                t->data = malloc(bytes > 0 ? bytes : 1);
                if (!t->data) {
                    rc = -1;
                    break;
                }
                memcpy(t->data, tiles[(k * ny + i) * nx + j], bytes);
            }
    if (rc == 0) {
        /* the recurrence, row-major over tiles */
        for (int64_t k = 0; k < nt; ++k)
            for (int64_t i = 0; i < ny; ++i)
                for (int64_t j = 0; j < nx; ++j) {
                    orc_tile* cur = &buf[(k * ny + i) * nx + j];
                    if (k > 0) blend_t(dt, planes, &buf[((k - 1) * ny + i) * nx + j], cur, blend[0]);
                    if (i > 0) blend_v(dt, planes, &buf[(k * ny + (i - 1)) * nx + j], cur, blend[1]);
                    if (j > 0) blend_h(dt, planes, &buf[(k * ny + i) * nx + (j - 1)], cur, blend[2]);
                }
        /* crop every tile to row_limit per axis and concatenate */
        int64_t OT = 0, OH = 0, OW = 0;
        for (int64_t k = 0; k < nt; ++k) OT += ext_t[k] < limit[0] ? ext_t[k] : limit[0];
        for (int64_t i = 0; i < ny; ++i) OH += ext_y[i] < limit[1] ? ext_y[i] : limit[1];
        for (int64_t j = 0; j < nx; ++j) OW += ext_x[j] < limit[2] ? ext_x[j] : limit[2];
        int64_t ot = 0;
        for (int64_t k = 0; k < nt; ++k) {
            const int64_t kt = ext_t[k] < limit[0] ? ext_t[k] : limit[0];
            int64_t oy = 0;
            for (int64_t i = 0; i < ny; ++i) {
                const int64_t ky = ext_y[i] < limit[1] ? ext_y[i] : limit[1];
                int64_t ox = 0;
                for (int64_t j = 0; j < nx; ++j) {
                    const int64_t kx = ext_x[j] < limit[2] ? ext_x[j] : limit[2];
                    const orc_tile* t = &buf[(k * ny + i) * nx + j];
                    for (int64_t p = 0; p < planes; ++p)
                        for (int64_t ct = 0; ct < kt; ++ct)
                            for (int64_t cy = 0; cy < ky; ++cy) {
                                const int64_t dst = ((p * OT + ot + ct) * OH + oy + cy) * OW + ox;
                                const int64_t src = tile_index(t, p, ct, cy, 0);
                                memcpy((char*)out + (size_t)dst * es, (const char*)t->data + (size_t)src * es,
                                       (size_t)kx * es);
                            }
                    ox += kx;
                }
                oy += ky;
            }
            ot += kt;
        }
    }
    for (int64_t n = 0; n < ntot; ++n) free(buf[n].data);
    free(buf);
    return rc;
}
