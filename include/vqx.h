/*
 * vqx: exact per-frame PSNR-noise and moment statistics of luma plane pairs
 * on one NVIDIA GB300 (sm_103a).  C ABI.
 *
 * What is computed, per frame pair (a reference plane r and a distorted plane
 * d of w x h samples at bpc bits, scaler S = 2^(bpc - 8), N = w * h):
 *
 *   float_psnr  ("ADR-1440: float_psnr_hip adds its squared differences as
 *               integers and returns the CPU's score bit for bit", Context and
 *               Decision): noise = sum over pixels of the float square of the
 *               float difference of the scaled samples, mse = noise / N,
 *               psnr = 10 log10(255^2 / mse), capped.
 *   float_moment ("ADR-1447: float_moment_hip adds the float squares the CPU
 *               adds, and is bit-identical while the CPU's own sum is exact",
 *               Context and Decision): mean = sum(s / S) / N and
 *               meansq = sum(float(s/S * s/S)) / N for both planes.
 *
 * How: every per-pixel term is formed in fp32 exactly as the CPU forms it
 * (one round-to-nearest-even product, no contraction) and is an integer in
 * units of 1/S^2 (1/S for the plain samples), so the library adds the terms
 * as integers, exactly and in any order, on the device, and converts the
 * integer sums to the scores on the host in double.  The scores are
 * therefore bit-identical to the CPU's wherever the CPU's double sum stays
 * under 2^53 units, where a double holds it exactly (always up to 12 bits,
 * and at 16 bits for frames of at most 2^21 pixels); beyond that they are
 * the exact sum rounded once, within the bound derived in ADR-1447
 * (Decision).
 *
 * Sample layout (all entry points): bpc 8 = one byte per sample; bpc 10, 12
 * and 16 = one little-endian uint16 per sample (the low bpc bits; a sample
 * of 2^bpc or more is an error, VQX_ERANGE).  Row y of frame f starts
 * f * height * stride + y * stride bytes after the plane's base pointer;
 * both planes use the same stride and the same frame pitch (with
 * vqx_planes_stats each plane descriptor gives its own, and a frame pitch).
 * Planes of uint16 samples must be 2-byte aligned (base and stride).
 *
 * Entry points:
 *   vqx_plane_stats            device planes, blocking
 *   vqx_plane_stats_submit / _finish   the same in two halves (pipelining)
 *   vqx_planes_stats           several planes of every frame (Y, Cb, Cr)
 *   vqx_plane_stats_host       planes in host memory (copies overlapped)
 *   vqx_plane_stats_ordered (+ _submit / _finish)   doubles equal to the CPU's
 *                              also past 2^53 units
 *   vqx_plane_stats_noalloc    no allocation at call time (fixed scratch)
 *   vqx_plane_int_psnr (+ _submit / _finish)   the integer psnr
 *   vqx_plane_scores (+ _submit / _finish)     the fused statistics and the
 *                              integer psnr from one read of the planes
 *   vqx_psnr_hvs_sum (+ _submit / _finish)     psnr_hvs plane sums of given
 *                              terms, the CPU's sequential float sum
 *   vqx_psnr_cap, vqx_status_string, vqx_last_cuda_error,
 *   vqx_profile_enable / vqx_profile_read      helpers and counters
 */
#ifndef VQX_H
#define VQX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *vqx_stream_t;

/* Status codes: 0 on success, negative on failure. */
#define VQX_OK 0
#define VQX_EINVAL (-1)  /* null pointer, size <= 0, stride too short,
                            misaligned uint16 plane, frame over 2^25 pixels */
#define VQX_EBPC (-2)    /* bpc not one of 8, 10, 12, 16 */
#define VQX_ERANGE (-3)  /* a sample >= 2^bpc was read (results are still
                            written; the frames concerned carry
                            VQX_FLAG_RANGE) */
#define VQX_ECUDA (-4)   /* a CUDA runtime call failed; see
                            vqx_last_cuda_error() */
#define VQX_ENOMEM (-5)  /* device or pinned host memory could not be had */
#define VQX_ETIMEOUT (-6) /* a wait inside a kernel gave up after about a
                             second (a copy that never completed); the
                             frames concerned carry VQX_FLAG_TIMEOUT and their
                             sums are incomplete.  The CUDA context stays
                             usable. */

/* Largest frame accepted, in pixels (w * h).  With terms below 2^24 (bit
 * depths up to 12) a frame of this size keeps the exact noise sum within
 * 49 bits, 2^24 * 2^25, the width ADR-1440 (Context) gives for the CPU's
 * exact sums. */
#define VQX_MAX_FRAME_PIXELS (1u << 25)

/* vqx_frame_stats.flags */
#define VQX_FLAG_RANGE 1u   /* the frame holds a sample >= 2^bpc */
#define VQX_FLAG_TIMEOUT 2u /* a device-side wait for this frame timed out */

/* Results for one frame pair.  The integer fields are the exact sums on the
 * device (the accumulators a debug mode would show); the doubles are concluded
 * from them. */
typedef struct {
    uint64_t noise_units;     /* sum of float(D * D), D = r - d raw; unit 1/S^2 */
    uint64_t ref_sum;         /* sum of r; unit 1/S */
    uint64_t dist_sum;        /* sum of d; unit 1/S */
    uint64_t ref_sumsq;       /* sum of float(r * r); unit 1/S^2 */
    uint64_t dist_sumsq;      /* sum of float(d * d); unit 1/S^2 */
    uint32_t flags;           /* VQX_FLAG_* */
    uint32_t reserved;
    double noise;             /* noise_units / S^2 */
    double mse;               /* noise / N (the 8-bit scale) */
    double psnr;              /* min(psnr_uncapped, vqx_psnr_cap(bpc)) */
    double psnr_uncapped;     /* 10 log10(255^2 / mse); +inf when mse == 0 */
    double ref_mean, ref_meansq;   /* (ref_sum / S) / N, (ref_sumsq / S^2) / N */
    double dist_mean, dist_meansq; /* the same for the distorted plane */
} vqx_frame_stats;

/*
 * vqx_plane_stats: the fused pass over device-resident planes.
 *
 *   ref, dist  device pointers (caller-owned, read only, not retained) to
 *              n_frames frames laid out as above.
 *   width, height  samples per row, rows per frame (>= 1; w * h at most
 *              VQX_MAX_FRAME_PIXELS).
 *   stride     bytes from one row to the next (>= width * bytes per sample).
 *   bpc        8, 10, 12 or 16.
 *   n_frames   frames in the batch (0 is an empty batch: returns VQX_OK and
 *              touches nothing).
 *   stream     the CUDA stream the work is ordered on; it must belong to the
 *              current device.  The call waits for the stream before it
 *              returns (out is filled on return).
 *   out        host array of n_frames records (caller-owned).
 *
 * The library owns only short-lived memory: a stream-ordered device
 * workspace from its own memory pool and a pinned host record buffer, both
 * reused across calls.  No device memory is cleared before use: every device
 * buffer is written before it is read.  Calls on different streams or
 * threads may run concurrently.  Returns VQX_OK or a negative status; on an
 * argument error nothing is launched and out is untouched.
 */
int vqx_plane_stats(const void *ref, const void *dist, int width, int height, size_t stride,
                    int bpc, int n_frames, vqx_stream_t stream, vqx_frame_stats *out);

/*
 * vqx_plane_stats_submit / vqx_plane_stats_finish: vqx_plane_stats in two
 * halves, so that a caller can enqueue the next batch before it concludes
 * this one (the device then runs the next batch's kernels while the host
 * waits on and concludes this one).
 *
 * vqx_plane_stats_submit takes the arguments of vqx_plane_stats without
 * `out`, plus flags (0 or VQX_SUBMIT_PLANES_READY), checks them (same status
 * codes, and VQX_EINVAL for an unknown flag; on an error nothing is enqueued
 * and *pending is set to NULL), enqueues the batch's kernels on `stream` and
 * returns without waiting.  *pending receives a library-owned handle, NULL
 * for an empty batch.  ref and dist must stay valid and unchanged until
 * vqx_plane_stats_finish on that handle has returned.
 *
 * The batch's main kernel is a programmatic dependent of the kernel before it
 * on the stream: it is set up while that kernel finishes, and by default
 * waits for it to complete before reading the planes.  VQX_SUBMIT_PLANES_READY
 * tells it not to wait before reading (it still waits before writing
 * anything): pass it when no kernel ahead on the stream that lets its
 * dependents start early (programmatic dependent launch) is still writing
 * these planes, for instance when the planes were written before the batch
 * ahead was enqueued.  Consecutive batches then overlap one's end with the
 * next one's start.  Results are the same either way.
 *
 * vqx_plane_stats_finish waits for the batch, writes its n_frames records to
 * out (host array, caller-owned) exactly as vqx_plane_stats would and
 * returns that call's status; it releases the handle whatever it returns.
 * Every handle must be finished exactly once, from any thread, in any order;
 * a NULL handle (an empty batch) returns VQX_OK and touches nothing.  Device
 * times (vqx_profile_enable) are recorded if profiling was enabled on the
 * submitting thread and counted on the finishing thread.
 */
typedef struct vqx_pending vqx_pending;

#define VQX_SUBMIT_PLANES_READY 1u

int vqx_plane_stats_submit(const void *ref, const void *dist, int width, int height,
                           size_t stride, int bpc, int n_frames, vqx_stream_t stream,
                           unsigned flags, vqx_pending **pending);

int vqx_plane_stats_finish(vqx_pending *pending, vqx_frame_stats *out);

/*
 * Several planes of each frame in one call (Y, Cb, Cr of 4:2:0 or 4:2:2
 * video, at most VQX_MAX_PLANES).  Each plane has its own size, row pitch and
 * frame pitch, so the planes may live in separate buffers or interleaved in
 * one buffer per frame.
 */
#define VQX_MAX_PLANES 4

typedef struct {
    const void *ref;    /* device pointer: this plane of frame 0 of the reference */
    const void *dist;   /* the same plane of frame 0 of the distorted video */
    int width, height;  /* samples per row, rows (>= 1; w * h <= VQX_MAX_FRAME_PIXELS) */
    size_t stride;      /* bytes from one row to the next (>= width * bytes per sample) */
    size_t frame_pitch; /* bytes from this plane of frame f to that of f + 1; 0 means
                           height * stride; otherwise at least height * stride */
} vqx_plane_desc;

/*
 * vqx_planes_stats: vqx_plane_stats for every plane of every frame; out is a
 * host array of n_frames * n_planes records, the record of plane p of frame
 * f at out[f * n_planes + p].  Status codes as for vqx_plane_stats
 * (VQX_EINVAL also for n_planes outside 1 .. VQX_MAX_PLANES or a frame pitch
 * below height * stride, or odd, at 10 to 16 bits); nothing is launched on
 * an argument error.  Synchronous on return.
 */
int vqx_planes_stats(const vqx_plane_desc *planes, int n_planes, int bpc, int n_frames,
                    vqx_stream_t stream, vqx_frame_stats *out);

/* The same in two halves, as vqx_plane_stats_submit / _finish (flags, the
 * planes' lifetime and the handle's rules alike); the descriptors themselves
 * are read during the submit only. */
int vqx_planes_stats_submit(const vqx_plane_desc *planes, int n_planes, int bpc, int n_frames,
                            vqx_stream_t stream, unsigned flags, vqx_pending **pending);

int vqx_planes_stats_finish(vqx_pending *pending, vqx_frame_stats *out);

/*
 * Integer psnr of one frame pair: the integer sibling of float_psnr.
 * "ADR-1440: float_psnr_hip adds its squared differences as integers ..."
 * (Alternatives) names psnr_hip as keeping one uint64 per frame; the pages
 * give no more of it, so the conclusion below is a stated reading.
 */
typedef struct {
    uint64_t sse;         /* sum over pixels of (r - d)^2, raw samples, exact */
    uint32_t flags;       /* VQX_FLAG_* as in vqx_frame_stats */
    uint32_t reserved;    /* 0 */
    double mse;           /* sse / (width * height), at the samples' own scale */
    double psnr;          /* min(psnr_uncapped, vqx_psnr_cap(bpc)) */
    double psnr_uncapped; /* 10 log10((2^bpc - 1)^2 / mse); +inf when sse == 0 */
} vqx_int_psnr_stats;     /* 40 bytes */

/*
 * vqx_plane_int_psnr: the integer psnr of every frame of a batch of
 * device-resident planes.  Arguments, layout, ownership and status codes as
 * for vqx_plane_stats, with out an array of n_frames vqx_int_psnr_stats.  The
 * SSE is exact at every depth (at most 2^25 * (2^16 - 1)^2 < 2^57); mse is
 * its one correctly rounded division by the pixel count.
 */
int vqx_plane_int_psnr(const void *ref, const void *dist, int width, int height, size_t stride,
                       int bpc, int n_frames, vqx_stream_t stream, vqx_int_psnr_stats *out);

/* The same in two halves, as vqx_plane_stats_submit / _finish (a handle
 * from one pair is not accepted by the other: VQX_EINVAL, handle released). */
int vqx_plane_int_psnr_submit(const void *ref, const void *dist, int width, int height,
                              size_t stride, int bpc, int n_frames, vqx_stream_t stream,
                              unsigned flags, vqx_pending **pending);

int vqx_plane_int_psnr_finish(vqx_pending *pending, vqx_int_psnr_stats *out);

/*
 * vqx_plane_scores: float_psnr, float_moment and the integer psnr of every
 * frame from one read of the planes.  "ADR-1440: float_psnr_hip adds its
 * squared differences as integers ..." (Alternatives) sets psnr_hip's one
 * uint64 per frame beside float_psnr's integer sums; both are sums over the
 * same sample pairs, so one pass forms both.
 *
 * out receives exactly what vqx_plane_stats returns, int_out exactly what
 * vqx_plane_int_psnr returns (both host arrays of n_frames records,
 * caller-owned; int_out may not be NULL when n_frames > 0).  Up to 12 bits
 * the SSE is the noise sum itself (the float squares are the integer
 * squares there); at 16 bits the fused kernel also adds up, exactly, the
 * rounding error of every float noise square (one fused multiply-add a
 * pixel), and SSE = noise sum - the sum of those errors.  Arguments, layout,
 * ownership and status codes (one status for both arrays) as for
 * vqx_plane_stats; synchronous on return.
 */
int vqx_plane_scores(const void *ref, const void *dist, int width, int height, size_t stride,
                     int bpc, int n_frames, vqx_stream_t stream, vqx_frame_stats *out,
                     vqx_int_psnr_stats *int_out);

/* The same in two halves, as vqx_plane_stats_submit / _finish (flags, the
 * planes' lifetime and the handle's rules alike; a handle of another pair is
 * refused with VQX_EINVAL and released, and so is a NULL out or int_out). */
int vqx_plane_scores_submit(const void *ref, const void *dist, int width, int height,
                            size_t stride, int bpc, int n_frames, vqx_stream_t stream,
                            unsigned flags, vqx_pending **pending);

int vqx_plane_scores_finish(vqx_pending *pending, vqx_frame_stats *out,
                            vqx_int_psnr_stats *int_out);

/*
 * vqx_plane_stats_host: the same results for planes in host memory.  The
 * frames are copied to the device in chunks on an internal copy stream while
 * earlier chunks are reduced on `stream` (copy and compute overlap); pinned
 * host memory (cudaHostAlloc / cudaHostRegister) gives asynchronous copies,
 * pageable memory works but copies synchronously.  Arguments as for
 * vqx_plane_stats, with ref and dist host pointers.
 */
int vqx_plane_stats_host(const void *ref, const void *dist, int width, int height,
                         size_t stride, int bpc, int n_frames, vqx_stream_t stream,
                         vqx_frame_stats *out);

/*
 * vqx_plane_stats_ordered: vqx_plane_stats, bit-identical to the CPU
 * extractors also where their double sums pass 2^53 units.
 *
 * Past 2^53 units the CPU's running double sum rounds at every add, so its
 * value depends on the order of the terms; vqx_plane_stats returns the exact
 * sum rounded once, within the bound of "ADR-1447: float_moment_hip adds the
 * float squares the CPU adds ..." (Decision).  This entry point replays the
 * CPU's raster-order sequence of roundings on the device (ADR-1447,
 * Alternatives, names that replay as the way to be bit-identical for every
 * frame), so noise, mse, psnr, psnr_uncapped, ref_meansq and dist_meansq
 * equal the CPU's doubles for every frame.  The integer fields stay the exact
 * sums.  Only 16-bit frames of more than 2^21 pixels can pass 2^53 units;
 * for the others the call is vqx_plane_stats.  For those it runs four
 * kernels of its own instead (block sums of every sequence, their
 * classification, transfer tables of the blocks that need them, and one walk
 * per frame and sum), which read the planes once plus again for the blocks
 * that are tabulated or replayed.  Arguments and status codes as for
 * vqx_plane_stats, plus VQX_EINVAL for more than 65535 frames in such a
 * batch.
 */
int vqx_plane_stats_ordered(const void *ref, const void *dist, int width, int height,
                            size_t stride, int bpc, int n_frames, vqx_stream_t stream,
                            vqx_frame_stats *out);

/* The same in two halves, as vqx_plane_stats_submit / _finish (flags, the
 * planes' lifetime and the handle's rules alike).  A batch's device
 * workspace is held until its handle is finished. */
int vqx_plane_stats_ordered_submit(const void *ref, const void *dist, int width, int height,
                                   size_t stride, int bpc, int n_frames, vqx_stream_t stream,
                                   unsigned flags, vqx_pending **pending);

int vqx_plane_stats_ordered_finish(vqx_pending *pending, vqx_frame_stats *out);

/* The PSNR cap in dB for a bit depth (6 * bpc + 12: 60, 72, 84, 108), or a
 * NaN for an unsupported bpc.  ADR-1440 (Consequences) shows that a cap
 * exists but does not print its value; this value is a stated choice. */
double vqx_psnr_cap(int bpc);

/* A static, human-readable description of a status code. */
const char *vqx_status_string(int status);

/* The cudaError_t of the last failed CUDA call made by this thread inside
 * the library (0 if none). */
int vqx_last_cuda_error(void);

/* Per-thread counters of the library's work.  Calls, kernel launches and
 * bytes read are always counted.  Device times are measured only while
 * enabled: a vqx_plane_stats or vqx_plane_int_psnr batch (submitted on a
 * thread with profiling on; counted on the thread that finishes it) then
 * records CUDA events on the caller's stream around its fused kernel and
 * its per-frame kernel, and vqx_plane_stats_ordered around its block-sum
 * kernel (counted as its stage-1 launch).  vqx_profile_read returns the
 * totals since the last reset. */
typedef struct {
    uint64_t calls;            /* successful calls */
    uint64_t kernel_launches;  /* library kernels launched by those calls */
    uint64_t stage1_launches;  /* of which fused load/reduce launches */
    double stage1_ms;          /* device time of the fused launches (enabled only) */
    double stage2_ms;          /* device time of the per-frame sums (enabled only) */
    uint64_t stage1_bytes;     /* plane bytes the fused launches read */
} vqx_profile;

void vqx_profile_enable(int enable);
void vqx_profile_read(vqx_profile *out, int reset);

/*
 * Records held by the static scratch of vqx_plane_stats_noalloc: 65536
 * records of 64 bytes (4 MiB of device memory on every GPU the library's
 * device code is loaded on, held until the process exits).
 */
#define VQX_NOALLOC_MAX_RECORDS 65536

/*
 * vqx_plane_stats_noalloc: vqx_plane_stats for callers that cannot allocate.
 * (An addition of this library, with no counterpart in the pages it follows.)
 *
 * Some callers must not allocate memory once they run: a real-time video
 * pipeline whose frame deadline cannot absorb a device or pinned allocation
 * (these can take driver locks or wait for the device), or a host
 * application that hands all of the GPU's memory to its own allocator and
 * lets no library take memory behind its back.  Its calls allocate nothing:
 * its scratch is a fixed-size array in the library's device memory, and the
 * per-frame sums are copied straight into `out`.
 *
 * That array is reserved when the library's device code is loaded on a
 * device: with CUDA's default lazy module loading, during the first call on
 * that device that needs it (of this entry point, or of any other vqx entry
 * point), or when the CUDA context is created if the process runs with
 * CUDA_MODULE_LOADING=EAGER.  A caller whose own allocator takes all of the
 * GPU's memory should therefore make one call of this entry point (any
 * valid batch) before its allocator takes the memory; later calls then have
 * nothing to reserve.
 *
 * Arguments, results and status codes are those of vqx_plane_stats.  The
 * batch may hold at most VQX_NOALLOC_MAX_RECORDS / 2 frames; a larger
 * n_frames is rejected with VQX_EINVAL before anything runs.  Large frames
 * may be split into fewer segments than vqx_plane_stats uses, so a batch of
 * many frames can run somewhat slower; the results are identical.
 *
 * The first call on each device (with that device current) also looks up the
 * scratch array's device address and sets the kernels' attributes.  Every
 * call ends by copying the sums into `out` (pageable host memory) and
 * waiting for `stream`: it is synchronous, and it cannot be captured into a
 * CUDA graph.  Make the first call before any other thread begins a stream
 * capture in global mode, which the set-up's calls would disturb.  Every
 * call uses the same scratch array, which keeps the last
 * call's contents; nothing in it needs to start at zero, because every
 * record is written before it is read.  Two calls whose work overlaps on the
 * GPU (calls on different streams, or from different threads, at the same
 * time) use the same scratch and race: serialise them, or use
 * vqx_plane_stats.
 */
int vqx_plane_stats_noalloc(const void *ref, const void *dist, int width, int height,
                            size_t stride, int bpc, int n_frames, vqx_stream_t stream,
                            vqx_frame_stats *out);

/*
 * psnr_hvs plane sum ("ADR-1397: GPU psnr_hvs twins reproduce the CPU's
 * running float sum bit for bit", Context and Decision).
 *
 * The CPU adds a plane's terms, the masked coefficient errors (64 per 8x8
 * block, a block's values in row order, blocks in raster order), one after
 * another into a single float that starts at zero, then divides that sum in
 * float by the number of terms and then by the float square of the sample
 * maximum 2^bpc - 1 (the plane score).  vqx_psnr_hvs_sum returns both, the
 * sum equal bit for bit to that sequential float sum, computed on the device
 * from transfer tables of runs of additions instead of a sequential pass.
 * The terms are the input: their transform, CSF and masking are not part of
 * this call.
 *
 * terms: device memory, float32; plane p's n_terms terms start
 *   p * plane_pitch floats after `terms`.  4-byte aligned.  A 16-byte aligned
 *   base with plane_pitch a multiple of 4 (and at least 32 terms) takes the
 *   fast path, a persistent pipeline of tensor-map copies; any other layout
 *   takes one CTA per node with plain loads, which is slower.  Read only, not
 *   retained after the call.
 * Every term must be a non-negative float below 2^95 (-0 counts as 0).  A
 *   plane holding anything else (a negative value, NaN, infinity, 2^95 or
 *   more) gets VQX_FLAG_RANGE and NaN sum and score; the call fills every
 *   record and then returns VQX_ERANGE.
 * n_terms: 1 .. 2^31 - 1; plane_pitch >= n_terms; n_planes >= 0 (0 does
 *   nothing); bpc: 8, 10, 12 or 16 (the score's peak); n_planes times
 *   ceil(n_terms / 8192) at most 2^31 - 1.
 * out: host memory for n_planes records.  Synchronous, like
 *   vqx_plane_stats.  The _submit / _finish pair splits it in two as
 *   vqx_plane_stats_submit / _finish do, with the same rules; flags is 0 or
 *   VQX_SUBMIT_PLANES_READY, which here means that the terms are ready (the
 *   batch's first kernel is a programmatic dependent of the kernel ahead and
 *   then reads the terms without waiting for it).  A submitted batch holds
 *   its device workspace (about 1 % of its terms' size) until finished.
 * Errors: VQX_EINVAL, VQX_EBPC, VQX_ERANGE, VQX_ENOMEM, VQX_ECUDA.
 */
typedef struct {
    float sum;                /* the sequential float sum of the plane's terms */
    float score;              /* (sum / n_terms) / peak^2, each step in float */
    uint32_t flags;           /* VQX_FLAG_RANGE: a term outside [0, 2^95) */
    uint32_t replayed_leaves; /* leaves of 1024 terms the device walked run by
                                 run rather than from their tables (where the
                                 sum crosses a power of two): diagnostic */
} vqx_hvs_plane;

int vqx_psnr_hvs_sum(const float *terms, int64_t n_terms, int64_t plane_pitch, int n_planes,
                     int bpc, vqx_stream_t stream, vqx_hvs_plane *out);

int vqx_psnr_hvs_sum_submit(const float *terms, int64_t n_terms, int64_t plane_pitch,
                            int n_planes, int bpc, vqx_stream_t stream, unsigned flags,
                            vqx_pending **pending);

int vqx_psnr_hvs_sum_finish(vqx_pending *pending, vqx_hvs_plane *out);

#ifdef __cplusplus
}
#endif

#endif /* VQX_H */
