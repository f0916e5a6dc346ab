/*
 * vqx oracle: TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, obviously correct CPU statement of what the GPU library
 * computes for one frame pair (a reference and a distorted luma plane):
 * the float_psnr noise sum, MSE and PSNR, and the float_moment mean and mean
 * square of both planes.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this code; the GPU library never does, and
 * the two share no source, header, table or helper.
 *
 * What is followed (vmafx ADR pages):
 *  - "ADR-1440: float_psnr_hip adds its squared differences as integers and
 *    returns the CPU's score bit for bit", section Context: the CPU extractor
 *    scales both planes to the 8-bit range (a sample over 2^(bpc - 8)) in
 *    float, takes the per-pixel difference and its square in float, and
 *    keeps a double running total over the frame, one row after another.
 *    Its Consequences section shows that the score is capped (there is an
 *    option to lift the cap) and places MSE 16570 under 6 dB, which only
 *    holds with a peak of 255.
 *  - "ADR-1447: float_moment_hip adds the float squares the CPU adds, and is
 *    bit-identical while the CPU's own sum is exact", section Context: the
 *    same scaling (scalers 1, 4, 16, 256 for 8, 10, 12, 16 bits), then one
 *    double total of the scaled samples and one of their float squares per
 *    plane, each divided by the number of pixels at the end.
 *
 * Readings where the pages are silent:
 *  - the row-by-row accumulation is one double accumulator walked in raster order;
 *  - MSE = noise / (w * h); PSNR = 10 log10(255^2 / MSE);
 *  - the PSNR cap is 6 * bpc + 12 dB (60, 72, 84, 108), applied as a min; the
 *    uncapped value is +inf when MSE = 0;
 *  - samples are unsigned, one byte at 8 bits and two little-endian bytes
 *    otherwise; frame f of a batch starts f * h * stride bytes after the base.
 *
 * The exact-integer function (vqx_oracle_units_frame) is the plain definition
 * of the raw sums the GPU library also reports: the sum over pixels of the
 * float square of the raw difference converted to an integer, the sum of raw
 * samples and the sum of the float squares of raw samples.  ADR-1440
 * (Decision) and ADR-1447 (Decision) state that these integers, divided by
 * scaler^2 (or scaler), are the CPU's terms and sums.
 *
 * The integer psnr (vqx_oracle_int_psnr_frame) and the psnr_hvs plane sum
 * (vqx_oracle_hvs_plane) are stated beside them, with their own readings.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -fno-tree-vectorize.
 * Contraction must stay off: the pages' CPU reference is a strict build.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define VQX_ORACLE_OK 0
#define VQX_ORACLE_EINVAL (-1)

/* One frame's results, CPU definition. */
typedef struct {
    double noise;         /* sum of float squares of scaled differences */
    double mse;           /* noise / (w * h) */
    double psnr;          /* min(psnr_uncapped, cap) */
    double psnr_uncapped; /* 10 log10(255^2 / mse), +inf when mse == 0 */
    double ref_mean, ref_meansq, dist_mean, dist_meansq;
} vqx_oracle_scores;

/* One frame's exact integer sums, raw sample units. */
typedef struct {
    uint64_t noise_units; /* sum of (uint) float(D * D), D = r - d */
    uint64_t ref_sum, dist_sum;
    uint64_t ref_sumsq, dist_sumsq; /* sum of (uint) float(s * s) */
} vqx_oracle_units;

static int valid_bpc(int bpc) { return bpc == 8 || bpc == 10 || bpc == 12 || bpc == 16; }

/* Sample x of the row starting at byte address row; bpc 8 is one byte, the
 * others are two bytes, little-endian (memcpy: rows need not be aligned). */
static unsigned sample_at(const unsigned char *row, int x, int bpc) {
    if (bpc == 8) return row[x];
    uint16_t v;
    memcpy(&v, row + 2 * (size_t)x, sizeof v);
    return v;
}

double vqx_oracle_psnr_cap(int bpc) { return 6.0 * bpc + 12.0; }

/* float_psnr (ADR-1440, Context): scaled samples, float difference, float
 * square, one double running sum over the rows in order. */
static double psnr_noise(const unsigned char *ref, const unsigned char *dist, int w, int h,
                         size_t stride, int bpc) {
    const float scaler = (float)(1u << (bpc - 8));
    double noise = 0.0;
    for (int y = 0; y < h; y++) {
        const unsigned char *rrow = ref + (size_t)y * stride;
        const unsigned char *drow = dist + (size_t)y * stride;
        for (int x = 0; x < w; x++) {
            float r = (float)sample_at(rrow, x, bpc) / scaler;
            float d = (float)sample_at(drow, x, bpc) / scaler;
            float e = r - d;
            float sq = e * e;
            noise += (double)sq;
        }
    }
    return noise;
}

/* float_moment (ADR-1447, Context): picture_copy() scaling, then one double
 * per output: the samples, and the float squares of the samples. */
static void plane_moments(const unsigned char *plane, int w, int h, size_t stride, int bpc,
                          double *mean, double *meansq) {
    const float scaler = (float)(1u << (bpc - 8));
    double sum = 0.0, sum2 = 0.0;
    for (int y = 0; y < h; y++) {
        const unsigned char *row = plane + (size_t)y * stride;
        for (int x = 0; x < w; x++) {
            float pic = (float)sample_at(row, x, bpc) / scaler;
            sum += (double)pic;
            const float term = pic * pic;
            sum2 += (double)term;
        }
    }
    const double n = (double)w * (double)h;
    *mean = sum / n;
    *meansq = sum2 / n;
}

int vqx_oracle_scores_frame(const void *ref, const void *dist, int w, int h, size_t stride,
                            int bpc, vqx_oracle_scores *out) {
    if (!ref || !dist || !out || w <= 0 || h <= 0 || !valid_bpc(bpc)) return VQX_ORACLE_EINVAL;
    if (stride < (size_t)w * (bpc == 8 ? 1u : 2u)) return VQX_ORACLE_EINVAL;
    const unsigned char *r = (const unsigned char *)ref;
    const unsigned char *d = (const unsigned char *)dist;

    out->noise = psnr_noise(r, d, w, h, stride, bpc);
    out->mse = out->noise / ((double)w * (double)h);
    out->psnr_uncapped = 10.0 * log10(255.0 * 255.0 / out->mse);
    const double cap = vqx_oracle_psnr_cap(bpc);
    out->psnr = out->psnr_uncapped < cap ? out->psnr_uncapped : cap;

    plane_moments(r, w, h, stride, bpc, &out->ref_mean, &out->ref_meansq);
    plane_moments(d, w, h, stride, bpc, &out->dist_mean, &out->dist_meansq);
    return VQX_ORACLE_OK;
}

/* Exact integer sums of the same terms, raw units (unit 1/scaler^2 for the
 * squares, 1/scaler for the samples).  The square is one float product of
 * the raw values, rounded to nearest even by the FPU, then converted: the
 * product of two integers below 2^16 is an integer below 2^32. */
int vqx_oracle_units_frame(const void *ref, const void *dist, int w, int h, size_t stride,
                           int bpc, vqx_oracle_units *out) {
    if (!ref || !dist || !out || w <= 0 || h <= 0 || !valid_bpc(bpc)) return VQX_ORACLE_EINVAL;
    if (stride < (size_t)w * (bpc == 8 ? 1u : 2u)) return VQX_ORACLE_EINVAL;
    const unsigned char *rp = (const unsigned char *)ref;
    const unsigned char *dp = (const unsigned char *)dist;
    uint64_t noise = 0, rs = 0, ds = 0, rss = 0, dss = 0;
    for (int y = 0; y < h; y++) {
        const unsigned char *rrow = rp + (size_t)y * stride;
        const unsigned char *drow = dp + (size_t)y * stride;
        for (int x = 0; x < w; x++) {
            unsigned r = sample_at(rrow, x, bpc);
            unsigned d = sample_at(drow, x, bpc);
            float diff = (float)r - (float)d;
            float dsq = diff * diff;
            noise += (uint64_t)dsq;
            float rsq = (float)r * (float)r;
            float dsq2 = (float)d * (float)d;
            rs += r;
            ds += d;
            rss += (uint64_t)rsq;
            dss += (uint64_t)dsq2;
        }
    }
    out->noise_units = noise;
    out->ref_sum = rs;
    out->dist_sum = ds;
    out->ref_sumsq = rss;
    out->dist_sumsq = dss;
    return VQX_ORACLE_OK;
}

/*
 * Integer psnr, the integer sibling of float_psnr.  "ADR-1440: float_psnr_hip
 * adds its squared differences as integers ..." (Alternatives) names its HIP
 * twin, psnr_hip, as keeping one uint64 per frame; the pages give no formula
 * beyond that.  Readings taken:
 *  - SSE = the sum over pixels of (r - d)^2, raw samples at their own depth,
 *    in uint64 (exact: at most 2^25 (2^16 - 1)^2 < 2^57);
 *  - MSE = SSE / (w * h), one double division of the converted SSE;
 *  - PSNR = 10 log10(peak^2 / MSE), peak = 2^bpc - 1 (the largest sample),
 *    capped as float_psnr is; +inf uncapped when the SSE is 0.
 */
typedef struct {
    uint64_t sse;
    double mse, psnr, psnr_uncapped;
} vqx_oracle_int_psnr;

int vqx_oracle_int_psnr_frame(const void *ref, const void *dist, int w, int h, size_t stride,
                              int bpc, vqx_oracle_int_psnr *out) {
    if (!ref || !dist || !out || w <= 0 || h <= 0 || !valid_bpc(bpc)) return VQX_ORACLE_EINVAL;
    if (stride < (size_t)w * (bpc == 8 ? 1u : 2u)) return VQX_ORACLE_EINVAL;
    const unsigned char *rp = (const unsigned char *)ref;
    const unsigned char *dp = (const unsigned char *)dist;
    uint64_t sse = 0;
    for (int y = 0; y < h; y++) {
        const unsigned char *rrow = rp + (size_t)y * stride;
        const unsigned char *drow = dp + (size_t)y * stride;
        for (int x = 0; x < w; x++) {
            const int64_t e = (int64_t)sample_at(rrow, x, bpc) - (int64_t)sample_at(drow, x, bpc);
            sse += (uint64_t)(e * e);
        }
    }
    out->sse = sse;
    out->mse = (double)sse / ((double)w * (double)h);
    const double peak = (double)((1u << bpc) - 1);
    out->psnr_uncapped = 10.0 * log10(peak * peak / out->mse);
    const double cap = vqx_oracle_psnr_cap(bpc);
    out->psnr = out->psnr_uncapped < cap ? out->psnr_uncapped : cap;
    return VQX_ORACLE_OK;
}

int vqx_oracle_int_psnr_batch(const void *ref, const void *dist, int w, int h, size_t stride,
                              int bpc, int n_frames, vqx_oracle_int_psnr *out) {
    if (n_frames < 0 || (n_frames > 0 && !out)) return VQX_ORACLE_EINVAL;
    const size_t pitch = (size_t)h * stride;
    for (int f = 0; f < n_frames; f++) {
        const int rc = vqx_oracle_int_psnr_frame((const unsigned char *)ref + (size_t)f * pitch,
                                                 (const unsigned char *)dist + (size_t)f * pitch,
                                                 w, h, stride, bpc, &out[f]);
        if (rc != VQX_ORACLE_OK) return rc;
    }
    return VQX_ORACLE_OK;
}

/* A batch of frames laid out as the GPU library takes them: frame f of each
 * plane starts f * h * stride bytes after its base.  Frames are independent. */
int vqx_oracle_batch(const void *ref, const void *dist, int w, int h, size_t stride, int bpc,
                     int n_frames, vqx_oracle_scores *scores, vqx_oracle_units *units) {
    if (n_frames < 0) return VQX_ORACLE_EINVAL;
    const size_t pitch = (size_t)h * stride;
    for (int f = 0; f < n_frames; f++) {
        const unsigned char *r = (const unsigned char *)ref + (size_t)f * pitch;
        const unsigned char *d = (const unsigned char *)dist + (size_t)f * pitch;
        int rc = VQX_ORACLE_OK;
        if (scores) rc = vqx_oracle_scores_frame(r, d, w, h, stride, bpc, &scores[f]);
        if (rc == VQX_ORACLE_OK && units)
            rc = vqx_oracle_units_frame(r, d, w, h, stride, bpc, &units[f]);
        if (rc != VQX_ORACLE_OK) return rc;
    }
    return VQX_ORACLE_OK;
}

/* psnr_hvs plane score, summation step.
 *
 * "ADR-1397: GPU psnr_hvs twins reproduce the CPU's running float sum bit for
 * bit", sections Context and Decision ("Sum on the host"): every masked
 * coefficient error of a plane (64 per 8x8 block, the block's values in row
 * order, blocks in raster order) is added, one after another, into a single
 * float that starts at zero; the total is then divided, in float, by the
 * number of terms and by the squared sample maximum.  The strict build of the
 * CPU reference means every addition and division is one IEEE single
 * operation, rounded to nearest even, subnormals kept.
 *
 * The terms themselves (transform, CSF and masking) are not on the pages;
 * here they are the input.  Readings taken:
 *  - the two divisions happen in the order the page names them: first by the
 *    term count converted to float, then by the squared maximum;
 *  - the squared maximum is the float product of (2^bpc - 1) with itself.
 */
int vqx_oracle_hvs_plane(const float *terms, int64_t n_terms, int bpc, float *sum, float *score) {
    if (!terms || !sum || !score || n_terms < 1 || !valid_bpc(bpc)) return VQX_ORACLE_EINVAL;
    float s = 0.0f;
    for (int64_t i = 0; i < n_terms; i++) s = s + terms[i];
    const float peak = (float)((1u << bpc) - 1u);
    float q = s / (float)n_terms;
    q = q / (peak * peak);
    *sum = s;
    *score = q;
    return VQX_ORACLE_OK;
}

/* n_planes planes of n_terms terms, plane p starting p * pitch floats after
 * the base.  Planes are independent. */
int vqx_oracle_hvs_batch(const float *terms, int64_t n_terms, int64_t pitch, int n_planes, int bpc,
                         float *sums, float *scores) {
    if (n_planes < 0 || pitch < n_terms || (n_planes > 0 && (!sums || !scores)))
        return VQX_ORACLE_EINVAL;
    for (int p = 0; p < n_planes; p++) {
        const int rc = vqx_oracle_hvs_plane(terms + (size_t)p * (size_t)pitch, n_terms, bpc,
                                            &sums[p], &scores[p]);
        if (rc != VQX_ORACLE_OK) return rc;
    }
    return VQX_ORACLE_OK;
}
