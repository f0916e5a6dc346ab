// Host side of the C ABI declared in include/vqx.h.
//
// A call validates its arguments, plans the launch (layout path and how many
// segments each frame is split into, so that the grid is a whole number of
// resident waves on this GPU), takes a stream-ordered workspace for the
// per-CTA records from a library-owned memory pool, launches the fused
// stage-1 kernel and the per-frame stage-2 kernel, waits for the stream and
// concludes the scores from the exact integer sums in double on the host.
//
// The conclusion ("ADR-1440: float_psnr_hip adds its squared differences as
// integers ...", Decision: the host puts the integer sums together in double
// and divides by scaler^2; "ADR-1447: float_moment_hip adds the float squares
// the CPU adds ...", Decision: the two final divisions) is compiled with
// contraction off, and uses only divisions, one product by 10 and log10.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "vqx.h"
#include "vqx_kernels.cuh"
#include "vqx_hvs.cuh"
#include "vqx_ordered.cuh"

namespace {

using vqx::Partial;
using vqx::u64;

thread_local int t_last_cuda_error = 0;

int cuda_status(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return e == cudaErrorMemoryAllocation ? VQX_ENOMEM : VQX_ECUDA;
}

// ------------------------------------------------------------------ paths
// kDense: frames of contiguous, 16-byte aligned rows (1-D bulk copies);
// kRows: padded rows of whole 16-byte vectors, at least kRowsMinBytes long,
// on 16-byte aligned bases and pitch (1-D bulk copies of row pieces);
// kTiles: other rows on 16-byte aligned bases and pitch (tensor-map boxes);
// kRowsScalar: anything else (sample loads);
// kFrames: many dense frames of at most kFramesMaxVecs vectors (a warp per
// frame, plain 16-byte loads).  Measured: 64x64 16-bit frames (512 vectors)
// stream at 0.70 of the copy bandwidth this way from about 1200 frames on,
// 0.38 through the TMA pipeline, whose unit ends dominate such frames; from
// 128x128 16-bit (2048 vectors) and for every 8-bit size tried the pipeline
// is faster.
enum Path { kDense = 0, kTiles = 1, kRowsScalar = 2, kRows = 3, kFrames = 4, kPaths = 5 };
constexpr uint32_t kFramesMaxVecs = 1024;  // 16 KB of each plane
constexpr size_t kRowsMinBytes = 512;

// What a call computes: the fused statistics, the integer psnr, or both from
// one read (kScores).  Up to 12 bits the integer psnr's SSE is the fused
// pass's noise sum (its squares are exact), so only 16 bits has kernel
// variants of its own: the SSE alone, and the fused statistics carrying the
// SSE as well.
enum Kind { kStats = 0, kIntPsnr = 1, kPlanes = 2, kOrdered = 3, kHvs = 4, kScores = 5 };
// fused 8, 10, 12, 16 bits; integer psnr 16 bits; fused with the SSE, 16 bits
constexpr int kVariants = 6;

int variant_index(int bpc, int kind) {  // kPlanes runs the fused statistics
    if (kind == kIntPsnr && bpc == 16) return 4;
    if (kind == kScores && bpc == 16) return 5;
    return bpc == 8 ? 0 : bpc == 10 ? 1 : bpc == 12 ? 2 : 3;
}

// Kernel, CTA size and dynamic shared memory of each stage-1 variant.
struct Stage1Shape {
    const void *fn;
    int threads;
    size_t smem;
};

template <int BPC, class Src, class Acc>
constexpr auto stream_kernel() {
    return vqx::fused_stream_tma<BPC, vqx::kTmaWarps, vqx::kTmaStageVecs, vqx::kTmaStages, Src, Acc>;
}

template <int BPC, class Acc>
Stage1Shape stage1_shape(int path) {
    switch (path) {
    case kDense:
        return {(const void *)stream_kernel<BPC, vqx::DenseSource, Acc>(), vqx::kTmaThreads,
                vqx::kTmaSmem};
    case kTiles:
        return {(const void *)stream_kernel<BPC, vqx::TileSource, Acc>(), vqx::kTmaThreads,
                vqx::kTmaSmem};
    case kRows:
        return {(const void *)stream_kernel<BPC, vqx::RowSource, Acc>(), vqx::kTmaThreads,
                vqx::kTmaSmem};
    case kFrames:
        return {(const void *)vqx::fused_frames<BPC, Acc>, 32 * vqx::kFrameWarps, 0};
    default: return {(const void *)vqx::fused_rows<BPC, Acc>, vqx::kThreads, 0};
    }
}

// cuTensorMapEncodeTiled, found through the runtime (no link against the
// driver library), once per process.
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

cudaError_t encode_fn(PFN_cuTensorMapEncodeTiled_v12000 *out) {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && (q != cudaDriverEntryPointSuccess || fn == nullptr))
            g_encode_err = cudaErrorNotSupported;
        g_encode_tiled = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    });
    *out = g_encode_tiled;
    return g_encode_err;
}

// A width x height x frames tensor of elem_bytes-byte elements starting at
// base, rows `stride` bytes apart and frames frame_pitch bytes apart, read
// in bx x by x 1 boxes.
cudaError_t encode_planes(CUtensorMap *tm, const void *base, int elem_bytes, int width, int height,
                          size_t stride, size_t frame_pitch, int frames, int bx, int by) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    cudaError_t e = encode_fn(&enc);
    if (e != cudaSuccess) return e;
    const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)height, (cuuint64_t)frames};
    const cuuint64_t strides[2] = {(cuuint64_t)stride, (cuuint64_t)frame_pitch};
    const cuuint32_t box[3] = {(cuuint32_t)bx, (cuuint32_t)by, 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    const CUtensorMapDataType type = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                     : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                     : elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                                                       : CU_TENSOR_MAP_DATA_TYPE_INT64;
    const CUresult r = enc(tm, type,
                           3, const_cast<void *>(base), dims, strides, box, elem,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// psnr_hvs terms as a 32 x rows x planes tensor of floats (rows of 128
// bytes, planes pitch floats apart), read in 32 x 256 x 1 boxes with the
// 128-byte swizzle.  Only full rows are in the tensor.
cudaError_t encode_hvs(CUtensorMap *tm, const float *terms, long long rows, long long pitch,
                       int planes) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
    cudaError_t e = encode_fn(&enc);
    if (e != cudaSuccess) return e;
    const cuuint64_t dims[3] = {32, (cuuint64_t)rows, (cuuint64_t)planes};
    // one plane: its pitch is never stepped over, so any valid stride does
    // (a pitch of 2^38 floats or more would not encode)
    const cuuint64_t strides[2] = {128, planes > 1 ? (cuuint64_t)pitch * 4 : (cuuint64_t)rows * 128};
    const cuuint32_t box[3] = {32, (cuuint32_t)vqx::kHvsNodeRows, 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(terms), dims,
                           strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

Stage1Shape stage1_shape(int path, int variant) {
    switch (variant) {
    case 0: return stage1_shape<8, vqx::TermSums<8>>(path);
    case 1: return stage1_shape<10, vqx::TermSums<10>>(path);
    case 2: return stage1_shape<12, vqx::TermSums<12>>(path);
    case 3: return stage1_shape<16, vqx::TermSums<16>>(path);
    case 4: return stage1_shape<16, vqx::SseSums16>(path);
    default: return stage1_shape<16, vqx::TermSums16Sse>(path);
    }
}

// Per device: allow the dense kernels their shared-memory ring and count
// the CTAs of each variant that fit on one SM.
cudaError_t prepare_stage1(int (&resident)[kPaths][kVariants]) {
    for (int p = 0; p < kPaths; p++)
        for (int b = 0; b < kVariants; b++) {
            const Stage1Shape sh = stage1_shape(p, b);
            cudaError_t e = cudaSuccess;
            if (sh.smem > 48 * 1024)
                e = cudaFuncSetAttribute(sh.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sh.smem);
            if (e != cudaSuccess) return e;
            int n = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sh.fn, sh.threads, sh.smem);
            if (e != cudaSuccess) return e;
            resident[p][b] = n > 0 ? n : 1;
        }
    return cudaSuccess;
}

// ------------------------------------------------------------------ device state
// Per-device state, made once: SM count, resident CTAs per SM of every
// stage-1 variant, the library's stream-ordered memory pool (memory stays
// in the pool between calls, so a call allocates nothing from the driver
// once warm) and a copy stream for the host-memory entry point.
struct DeviceCtx {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int sms = 0;
    int resident[kPaths][kVariants] = {};
    cudaMemPool_t pool = nullptr;
    cudaStream_t copy_stream = nullptr;
    std::atomic<uint32_t> hvs_epoch{0};  // tags of the psnr_hvs look-back words
    int hvs_tma_resident = 0;            // hvs_tables_tma CTAs per SM (0: not used here)
};

constexpr int kMaxDevices = 64;
DeviceCtx g_dev[kMaxDevices];

cudaError_t init_device(DeviceCtx &c, int dev) {
    cudaError_t e = cudaDeviceGetAttribute(&c.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if ((e = prepare_stage1(c.resident)) != cudaSuccess) return e;
    e = cudaFuncSetAttribute(vqx::hvs_tables, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)vqx::kHvsTablesSmem);
    if (e != cudaSuccess) return e;
    // The pipelined psnr_hvs kernel takes all the shared memory a CTA may
    // have; on a device that offers less it is not used (hvs_tables is).
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    const bool hvs_tma = (size_t)optin >= vqx::kHvsTmaSmem;
    if (hvs_tma) {
        e = cudaFuncSetAttribute(vqx::hvs_tables_tma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)vqx::kHvsTmaSmem);
        if (e != cudaSuccess) return e;
    }
    // The walk (one warp, no shared memory) runs beside the next batch's
    // tables kernel: keep the SMs it sits on configured for the tables'
    // shared memory, so that their CTAs are not held back until it ends.
    e = cudaFuncSetAttribute(vqx::hvs_walk, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (hvs_tma) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&c.hvs_tma_resident, vqx::hvs_tables_tma,
                                                          vqx::kHvsTmaThreads, vqx::kHvsTmaSmem);
        if (e != cudaSuccess) return e;
    }

    cudaMemPoolProps props;
    memset(&props, 0, sizeof props);
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    e = cudaMemPoolCreate(&c.pool, &props);
    if (e != cudaSuccess) return e;
    uint64_t keep = UINT64_MAX;  // never hand memory back between calls
    e = cudaMemPoolSetAttribute(c.pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) return e;
    return cudaStreamCreateWithFlags(&c.copy_stream, cudaStreamNonBlocking);
}

int device_ctx(DeviceCtx **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return VQX_EINVAL;
    DeviceCtx &c = g_dev[dev];
    std::call_once(c.once, [&] { c.err = init_device(c, dev); });
    if (c.err != cudaSuccess) return cuda_status(c.err);
    *out = &c;
    return VQX_OK;
}

// ------------------------------------------------------------------ pinned records
// Pinned, device-mapped host buffers that stage 2 writes the per-frame sums
// into.  A call takes one from the free list and returns it afterwards, so
// concurrent calls never share one.
struct PinnedBuf {
    void *host = nullptr;
    void *dev = nullptr;
    size_t cap = 0;
};
std::mutex g_pinned_mu;
std::vector<PinnedBuf> g_pinned_free;

int acquire_pinned(size_t bytes, PinnedBuf *out) {
    {
        std::lock_guard<std::mutex> lk(g_pinned_mu);
        for (size_t i = 0; i < g_pinned_free.size(); i++)
            if (g_pinned_free[i].cap >= bytes) {
                *out = g_pinned_free[i];
                g_pinned_free.erase(g_pinned_free.begin() + (long)i);
                return VQX_OK;
            }
    }
    size_t cap = 4096;
    while (cap < bytes) cap *= 2;
    PinnedBuf b;
    cudaError_t e = cudaHostAlloc(&b.host, cap, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) return cuda_status(e);
    e = cudaHostGetDevicePointer(&b.dev, b.host, 0);
    if (e != cudaSuccess) {
        cudaFreeHost(b.host);
        return cuda_status(e);
    }
    b.cap = cap;
    *out = b;
    return VQX_OK;
}

void release_pinned(const PinnedBuf &b) {
    std::lock_guard<std::mutex> lk(g_pinned_mu);
    g_pinned_free.push_back(b);
}

// ------------------------------------------------------------------ profiling
struct Profiler {
    bool on = false;
    vqx_profile totals = {};
};
thread_local Profiler t_prof;

// ------------------------------------------------------------------ pending batches
}  // namespace

// A batch enqueued by vqx_plane_stats_submit: its pinned record buffer, the
// event recorded after its last kernel and, when profiling, timing events.
// Handles are kept on a per-device free list, events and all.
struct vqx_pending {
    PinnedBuf rec;
    cudaEvent_t done = nullptr;
    cudaEvent_t ev[3] = {};
    bool timed = false;
    DeviceCtx *ctx = nullptr;
    int kind = 0;  // Kind: what the batch computes
    int n_frames = 0, bpc = 0, width = 0, height = 0;
    int n_planes = 1;                                    // kPlanes: the planes' sizes
    int pw[VQX_MAX_PLANES] = {}, ph[VQX_MAX_PLANES] = {};
    long long n_terms = 0;  // kHvs: terms per plane (n_frames counts the planes)
    void *ws = nullptr;     // kOrdered: the workspace, held until finished
};

namespace {

std::mutex g_pending_mu;
std::vector<vqx_pending *> g_pending_free[kMaxDevices];

int acquire_pending(DeviceCtx *ctx, bool timed, vqx_pending **out) {
    const size_t d = (size_t)(ctx - g_dev);
    vqx_pending *p = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_pending_mu);
        if (!g_pending_free[d].empty()) {
            p = g_pending_free[d].back();
            g_pending_free[d].pop_back();
        }
    }
    if (!p) {
        p = new (std::nothrow) vqx_pending;
        if (!p) return VQX_ENOMEM;
        p->ctx = ctx;
        const cudaError_t e = cudaEventCreateWithFlags(&p->done, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            delete p;
            return cuda_status(e);
        }
    }
    p->timed = false;
    if (timed) {
        p->timed = true;
        for (auto &e : p->ev)
            if (!e && cudaEventCreate(&e) != cudaSuccess) p->timed = false;
    }
    *out = p;
    return VQX_OK;
}

void release_pending(vqx_pending *p) {
    std::lock_guard<std::mutex> lk(g_pending_mu);
    g_pending_free[(size_t)(p->ctx - g_dev)].push_back(p);
}

// ------------------------------------------------------------------ validation
int bytes_per_sample(int bpc) { return bpc == 8 ? 1 : 2; }

int validate(const void *ref, const void *dist, int width, int height, size_t stride, int bpc,
             int n_frames, const vqx_frame_stats *out) {
    if (bpc != 8 && bpc != 10 && bpc != 12 && bpc != 16) return VQX_EBPC;
    if (n_frames < 0) return VQX_EINVAL;
    if (n_frames == 0) return VQX_OK;
    if (!ref || !dist || !out) return VQX_EINVAL;
    if (width <= 0 || height <= 0) return VQX_EINVAL;
    if ((uint64_t)width * (uint64_t)height > VQX_MAX_FRAME_PIXELS) return VQX_EINVAL;
    const size_t bps = (size_t)bytes_per_sample(bpc);
    if (stride < (size_t)width * bps) return VQX_EINVAL;
    if (bps == 2 && (((uintptr_t)ref | (uintptr_t)dist | (uintptr_t)stride) & 1u)) return VQX_EINVAL;
    // the whole batch must be addressable
    const unsigned __int128 span = (unsigned __int128)n_frames * (unsigned __int128)height * stride;
    if (span > (unsigned __int128)(SIZE_MAX / 2)) return VQX_EINVAL;
    return VQX_OK;
}

// One plane of vqx_planes_stats: as validate, with its own frame pitch.
int validate_plane(const vqx_plane_desc &d, int bpc, int n_frames, size_t *pitch) {
    int rc = validate(d.ref, d.dist, d.width, d.height, d.stride, bpc, n_frames,
                      reinterpret_cast<const vqx_frame_stats *>(&d));
    if (rc != VQX_OK) return rc;
    const size_t min_pitch = (size_t)d.height * d.stride;
    const size_t fp = d.frame_pitch ? d.frame_pitch : min_pitch;
    if (fp < min_pitch) return VQX_EINVAL;
    if (bytes_per_sample(bpc) == 2 && (fp & 1u)) return VQX_EINVAL;
    const unsigned __int128 span = (unsigned __int128)fp * (unsigned __int128)n_frames;
    if (span > (unsigned __int128)(SIZE_MAX / 2)) return VQX_EINVAL;
    *pitch = fp;
    return VQX_OK;
}

// ------------------------------------------------------------------ plan
struct Plan {
    int path = kDense;
    int bpc = 8;
    int variant = 0;         // variant_index(bpc, kind)
    int segs = 1;
    int rec_per_unit = 1;    // records a unit writes (one per consumer warp, or one)
    long long resident = 1;  // CTAs of this variant resident on the whole GPU
    uint32_t work = 0;      // 16-byte vectors (dense) or rows per frame
    uint32_t seg_work = 0;  // per segment
    size_t frame_pitch = 0;
    size_t stride = 0;
    int width = 0, height = 0;
    int tile_elem = 0, tile_bx = 0, tile_by = 0;  // kTiles: element bytes, box
};

// The box of the tile path for rows of row_bytes bytes: the element is the
// widest of 8, 4, 2 or 1 bytes that divides a row; a box line is a whole
// number of 16-byte vectors and at most 256 elements, and a box at most one
// pipeline stage, and at most max_by rows (so that a small batch still
// splits into enough bands to keep every CTA busy).  Among those the box with
// the least work per frame wins, counting the zero fill past the last column
// and row as work, with a fixed cost per stage and per box line (a box of
// short lines copies measurably slower than one of long lines with some fill).
void choose_box(size_t row_bytes, int height, long long max_by, int *elem, int *bx, int *by) {
    int eb = 8;
    while (row_bytes % (size_t)eb) eb /= 2;
    const long long row_elems = (long long)(row_bytes / (size_t)eb);
    const long long cap = (long long)vqx::kTmaStageVecs * 16;
    const long long kStageCost = 128, kLineCost = 64;  // in vectors' worth of work
    long long best = -1;
    for (int x = 16 / eb; x <= 256; x += 16 / eb) {
        long long y = cap / ((long long)x * eb);
        if (y > 256) y = 256;
        if (y > height) y = height;
        if (y > max_by) y = max_by;
        const long long vecs = (long long)x * y * eb / 16;
        const long long cost = ((row_elems + x - 1) / x) * ((height + y - 1) / y) * (vecs + kStageCost + y * kLineCost);
        if (best < 0 || cost <= best) {  // ties: the longer line
            best = cost;
            *bx = x;
            *by = (int)y;
        }
    }
    *elem = eb;
}

// Segments per frame.  The frames x segments units run in waves of the
// resident CTAs, and a unit takes a whole number of pipeline stages, so a
// launch lasts about waves x (stages per unit + kUnitCost) stage times; the
// segment count with the fewest wins (ties: fewer units).  unit(s) gives the
// segment work, the segment count and the stages per unit for s segments
// asked for (whole bands can give fewer).  max_segs bounds s.
constexpr double kUnitCost = 0.35;  // a unit's end, in stage times (measured)

struct UnitShape {
    uint32_t seg_work;
    long long segs, stages;
};

template <class UnitFn>
UnitShape choose_segs(long long frames, long long max_segs, long long resident, UnitFn unit) {
    if (max_segs < 1) max_segs = 1;
    // More than eight waves buys no better fill; it only shrinks the units.
    const long long eight_waves = (8 * resident + frames - 1) / frames;
    if (max_segs > eight_waves) max_segs = eight_waves;
    while (max_segs > 1 && frames * max_segs > (1ll << 30)) max_segs /= 2;
    UnitShape best = unit(1);
    double best_t = -1.0;
    for (long long s = 1; s <= max_segs; s++) {
        const UnitShape u = unit(s);
        const long long waves = (frames * u.segs + resident - 1) / resident;
        const double t = (double)waves * ((double)u.stages + kUnitCost);
        if (best_t < 0 || t < best_t - 1e-9) {
            best = u;
            best_t = t;
        }
    }
    return best;
}

// max_records: at most this many stage-1 records per frame (a caller with a
// fixed scratch); units then write one record each, and if need be the
// frames get fewer segments.  frame_pitch: bytes from one frame to the next
// (0: height * stride, frames back to back).
Plan make_plan(const DeviceCtx &c, const void *ref, const void *dist, int width, int height,
               size_t stride, int bpc, long long frames_per_launch, int kind = kStats,
               long long max_records = 1ll << 40, size_t frame_pitch = 0) {
    Plan p;
    p.bpc = bpc;
    p.variant = variant_index(bpc, kind);
    p.width = width;
    p.height = height;
    p.stride = stride;
    p.frame_pitch = frame_pitch ? frame_pitch : (size_t)height * stride;
    const size_t row_bytes = (size_t)width * (size_t)bytes_per_sample(bpc);
    const bool aligned = (((uintptr_t)ref | (uintptr_t)dist) & 15u) == 0;
    const size_t frame_bytes = row_bytes * (size_t)height;
    if (aligned && stride == row_bytes && p.frame_pitch == frame_bytes && (frame_bytes & 15u) == 0) {
        p.path = kDense;
        p.work = (uint32_t)(frame_bytes >> 4);
        // many small frames (8 or more per SM): a warp per frame
        if (p.work <= kFramesMaxVecs && frames_per_launch >= 8ll * c.sms) p.path = kFrames;
    } else {
        // copies need 16-byte aligned rows; very narrow ones take the sample path
        const bool pitched = aligned && ((stride | p.frame_pitch) & 15u) == 0;
        p.path = pitched && (row_bytes & 15u) == 0 && row_bytes >= kRowsMinBytes ? kRows
                 : pitched && width >= 64                                         ? kTiles
                                                                                  : kRowsScalar;
        p.work = (uint32_t)height;
    }
    p.resident = (long long)c.sms * c.resident[p.path][p.variant];
    if (p.path == kFrames) {  // one record per frame, written by its warp
        p.segs = 1;
        p.seg_work = p.work;
        p.rec_per_unit = 1;
        return p;
    }
    if (p.path == kTiles) {
        // rows per CTA were the batch spread over every resident CTA
        long long max_by = (long long)height * frames_per_launch / (p.resident > 0 ? p.resident : 1);
        if (max_by < 1) max_by = 1;
        choose_box(row_bytes, height, max_by, &p.tile_elem, &p.tile_bx, &p.tile_by);
    }
    // Stage counts per unit: a dense or row-piece unit is cut into stages of
    // SV vectors, a tile unit into bands of boxes (segments of whole bands), a
    // scalar row unit into rows, one per warp (8 warps).
    const uint32_t sv = (uint32_t)vqx::kTmaStageVecs;
    const uint32_t band = p.path == kTiles ? (uint32_t)p.tile_by : 1u;
    const uint32_t tiles_x =
        p.path == kTiles ? (uint32_t)((row_bytes / (size_t)p.tile_elem + p.tile_bx - 1) / p.tile_bx) : 1u;
    const uint64_t row_vecs = row_bytes / 16;
    const uint32_t work = p.work;
    auto unit = [&](long long asked) {
        UnitShape u;
        u.seg_work = (uint32_t)((work + asked - 1) / asked);
        u.seg_work = (u.seg_work + band - 1) / band * band;
        u.segs = (work + u.seg_work - 1) / u.seg_work;
        switch (p.path) {
        case kDense: u.stages = (u.seg_work + sv - 1) / sv; break;
        case kRows: u.stages = (long long)(((uint64_t)u.seg_work * row_vecs + sv - 1) / sv); break;
        case kTiles: u.stages = (long long)(u.seg_work / band) * tiles_x; break;
        default: u.stages = (u.seg_work + 7) / 8; break;
        }
        return u;
    };
    // at least half a stage (dense), a band (tiles) or a row per unit
    long long max_segs = p.path == kDense ? (long long)(2 * (uint64_t)work / sv) : (long long)(work / band);
    p.rec_per_unit = p.path == kRowsScalar ? 1 : vqx::kTmaWarps;
    UnitShape u = choose_segs(frames_per_launch, max_segs, p.resident, unit);
    if (u.segs * p.rec_per_unit > max_records) {
        p.rec_per_unit = 1;
        if (u.segs > max_records) u = choose_segs(frames_per_launch, max_records, p.resident, unit);
    }
    p.segs = (int)u.segs;
    p.seg_work = u.seg_work;
    return p;
}

template <int BPC, class Acc>
cudaError_t launch_tiles(cudaLaunchConfig_t &cfg, const Plan &p, const unsigned char *ref,
                         const unsigned char *dist, int frame0, int frames, int units,
                         Partial *partials, bool planes_ready) {
    vqx::TileSource src;
    memset(&src, 0, sizeof src);
    const size_t first = (size_t)frame0 * p.frame_pitch;
    const int row_elems = (int)((size_t)p.width * bytes_per_sample(BPC) / (size_t)p.tile_elem);
    cudaError_t e = encode_planes(&src.tref, ref + first, p.tile_elem, row_elems, p.height, p.stride,
                                  p.frame_pitch, frames, p.tile_bx, p.tile_by);
    if (e == cudaSuccess)
        e = encode_planes(&src.tdist, dist + first, p.tile_elem, row_elems, p.height, p.stride,
                          p.frame_pitch, frames, p.tile_bx, p.tile_by);
    if (e != cudaSuccess) return e;
    src.width = row_elems;
    src.height = p.height;
    src.seg_rows = (int)p.seg_work;
    src.segs = p.segs;
    src.frame0 = frame0;
    src.bx = p.tile_bx;
    src.by = p.tile_by;
    src.box_vecs = (uint32_t)((size_t)p.tile_bx * p.tile_by * p.tile_elem / 16);
    return cudaLaunchKernelEx(&cfg, stream_kernel<BPC, vqx::TileSource, Acc>(), src, units,
                              (int)(p.rec_per_unit > 1), (int)planes_ready, partials);
}

template <int BPC, class Acc>
cudaError_t launch_stage1_bpc(const Plan &p, const unsigned char *ref, const unsigned char *dist,
                              int frame0, int frames, Partial *partials, cudaStream_t st,
                              bool overlap, bool planes_ready) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    const long long units = (long long)frames * p.segs;
    cfg.stream = st;
    if (p.path == kFrames) {
        // no programmatic dependency here: fused_frames stores without waiting
        const long long need = ((long long)frames + vqx::kFrameWarps - 1) / vqx::kFrameWarps;
        cfg.gridDim = dim3((unsigned)(need < p.resident ? need : p.resident));
        cfg.blockDim = dim3(32 * vqx::kFrameWarps);
        return cudaLaunchKernelEx(&cfg, vqx::fused_frames<BPC, Acc>, ref, dist, p.frame_pitch, p.work,
                                  frames, frame0, partials);
    }
    if (p.path == kRowsScalar) {
        cfg.gridDim = dim3((unsigned)units);
        cfg.blockDim = dim3(vqx::kThreads);
        return cudaLaunchKernelEx(&cfg, vqx::fused_rows<BPC, Acc>, ref, dist, p.frame_pitch,
                                  p.stride, p.width, p.height, (int)p.seg_work, p.segs, frame0,
                                  partials);
    }
    // persistent: at most the resident CTAs, each walking several units
    cfg.gridDim = dim3((unsigned)(units < p.resident ? units : p.resident));
    cfg.blockDim = dim3(vqx::kTmaThreads);
    cfg.dynamicSmemBytes = vqx::kTmaSmem;
    cudaLaunchAttribute attr[1];
    if (overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (p.path == kDense) {
        vqx::DenseSource src;
        src.ref = ref;
        src.dist = dist;
        src.frame_pitch = p.frame_pitch;
        src.frame_vecs = p.work;
        src.seg_vecs = p.seg_work;
        src.segs = p.segs;
        src.frame0 = frame0;
        return cudaLaunchKernelEx(&cfg, stream_kernel<BPC, vqx::DenseSource, Acc>(), src, (int)units,
                                  (int)(p.rec_per_unit > 1), (int)planes_ready, partials);
    }
    if (p.path == kRows) {
        vqx::RowSource src;
        src.ref = ref;
        src.dist = dist;
        src.frame_pitch = p.frame_pitch;
        src.stride = p.stride;
        src.row_vecs = (uint32_t)((size_t)p.width * bytes_per_sample(BPC) / 16);
        src.height = p.height;
        src.seg_rows = (int)p.seg_work;
        src.segs = p.segs;
        src.frame0 = frame0;
        return cudaLaunchKernelEx(&cfg, stream_kernel<BPC, vqx::RowSource, Acc>(), src, (int)units,
                                  (int)(p.rec_per_unit > 1), (int)planes_ready, partials);
    }
    return launch_tiles<BPC, Acc>(cfg, p, ref, dist, frame0, frames, (int)units, partials,
                                  planes_ready);
}

// overlap: launch the persistent kernels as programmatic dependents of the
// kernel before them on the stream, so that their CTAs are set up while that
// kernel finishes; they wait for it before their first load (unless
// planes_ready) and before their first store.
cudaError_t launch_stage1(const Plan &p, const void *ref, const void *dist, int frame0,
                          int frames, Partial *partials, cudaStream_t st, bool overlap = false,
                          bool planes_ready = false) {
    const unsigned char *r = (const unsigned char *)ref;
    const unsigned char *d = (const unsigned char *)dist;
    switch (p.variant) {
    case 0: return launch_stage1_bpc<8, vqx::TermSums<8>>(p, r, d, frame0, frames, partials, st, overlap,
                                                       planes_ready);
    case 1: return launch_stage1_bpc<10, vqx::TermSums<10>>(p, r, d, frame0, frames, partials, st, overlap,
                                                       planes_ready);
    case 2: return launch_stage1_bpc<12, vqx::TermSums<12>>(p, r, d, frame0, frames, partials, st, overlap,
                                                       planes_ready);
    case 3: return launch_stage1_bpc<16, vqx::TermSums<16>>(p, r, d, frame0, frames, partials, st, overlap,
                                                       planes_ready);
    case 4: return launch_stage1_bpc<16, vqx::SseSums16>(p, r, d, frame0, frames, partials, st, overlap,
                                                       planes_ready);
    default: return launch_stage1_bpc<16, vqx::TermSums16Sse>(p, r, d, frame0, frames, partials, st,
                                                              overlap, planes_ready);
    }
}

cudaError_t launch_stage2(const Plan &p, int n_frames, const Partial *partials, Partial *out,
                          cudaStream_t st) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)n_frames);
    cfg.blockDim = dim3(vqx::kSumThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, vqx::frame_sums, partials, p.segs * p.rec_per_unit, out);
}

// Bytes of the stage-1 records of n_frames frames.
size_t records_bytes(const Plan &p, long long n_frames) {
    return (size_t)n_frames * (size_t)p.segs * (size_t)p.rec_per_unit * sizeof(Partial);
}

// ------------------------------------------------------------------ conclusion
// The flags of a record: a sample at or above 2^bpc, a device wait that
// timed out.
uint32_t record_flags(const Partial &s, int bpc) {
    uint32_t flags = ((s.v[5] & 0xffffffffull) >> bpc) != 0 ? VQX_FLAG_RANGE : 0u;
    if (s.v[5] & vqx::kErrTimeout) flags |= VQX_FLAG_TIMEOUT;
    return flags;
}

// cpu, when given, holds the CPU's sequential double sums (noise, reference
// squares, distorted squares) in units, replayed on the device; otherwise
// the exact integer sums are rounded once.
void conclude(const Partial &s, int bpc, int width, int height, vqx_frame_stats *o,
              const u64 *cpu = nullptr) {
    const double S = (double)(1u << (bpc - 8));
    const double S2 = S * S;
    const double n = (double)width * (double)height;
    o->noise_units = s.v[0];
    o->ref_sum = s.v[1];
    o->dist_sum = s.v[2];
    o->ref_sumsq = s.v[3];
    o->dist_sumsq = s.v[4];
    o->flags = record_flags(s, bpc);
    o->reserved = 0;
    o->noise = (double)(cpu ? cpu[0] : s.v[0]) / S2;
    o->mse = o->noise / n;
    o->psnr_uncapped = 10.0 * log10(255.0 * 255.0 / o->mse);
    const double cap = vqx_psnr_cap(bpc);
    o->psnr = o->psnr_uncapped < cap ? o->psnr_uncapped : cap;
    o->ref_mean = ((double)s.v[1] / S) / n;
    o->ref_meansq = ((double)(cpu ? cpu[1] : s.v[3]) / S2) / n;
    o->dist_mean = ((double)s.v[2] / S) / n;
    o->dist_meansq = ((double)(cpu ? cpu[2] : s.v[4]) / S2) / n;
}

// The call's status from the frames' flags: a timed-out device wait first
// (its sums are incomplete), then an out-of-range sample.
int merge_status_flags(int rc, uint32_t flags) {
    if (flags & VQX_FLAG_TIMEOUT) return VQX_ETIMEOUT;
    if ((flags & VQX_FLAG_RANGE) && rc == VQX_OK) return VQX_ERANGE;
    return rc;
}

int merge_status(int rc, const vqx_frame_stats &f) { return merge_status_flags(rc, f.flags); }

// Integer psnr of one frame from its record: the exact SSE is word 0 plus
// word 6 (the integer-psnr kernel's sum and 0 at 16 bits; the fused pass's
// noise sum and 0 up to 12 bits, where the float squares are the integer
// squares; the float noise sum and the exact difference to the SSE from the
// fused pass that carries it).  MSE = SSE / N, one division; PSNR =
// 10 log10(peak^2 / MSE), peak = 2^bpc - 1, capped as float_psnr is.
void conclude_int_psnr(const Partial &s, int bpc, int width, int height, vqx_int_psnr_stats *o) {
    const u64 sse = s.v[0] + s.v[6];
    o->sse = sse;
    o->flags = record_flags(s, bpc);
    o->reserved = 0;
    o->mse = (double)sse / ((double)width * (double)height);
    const double peak = (double)((1u << bpc) - 1);
    o->psnr_uncapped = 10.0 * log10(peak * peak / o->mse);
    const double cap = vqx_psnr_cap(bpc);
    o->psnr = o->psnr_uncapped < cap ? o->psnr_uncapped : cap;
}

int conclude_all(const Partial *sums, int n_frames, int bpc, int width, int height,
                 vqx_frame_stats *out) {
    int rc = VQX_OK;
    for (int f = 0; f < n_frames; f++) {
        conclude(sums[f], bpc, width, height, &out[f]);
        rc = merge_status(rc, out[f]);
    }
    return rc;
}

// Bytes the fused kernel reads for a batch (both planes, each sample once).
uint64_t plane_bytes(int width, int height, int bpc, int n_frames) {
    return 2ull * (uint64_t)width * (uint64_t)height * (uint64_t)bytes_per_sample(bpc) *
           (uint64_t)n_frames;
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

double vqx_psnr_cap(int bpc) {
    if (bpc != 8 && bpc != 10 && bpc != 12 && bpc != 16) return NAN;
    return 6.0 * bpc + 12.0;
}

const char *vqx_status_string(int status) {
    switch (status) {
    case VQX_OK: return "ok";
    case VQX_EINVAL: return "invalid argument";
    case VQX_EBPC: return "unsupported bit depth (8, 10, 12 or 16)";
    case VQX_ERANGE: return "a sample is out of range for the bit depth";
    case VQX_ECUDA: return "CUDA runtime error";
    case VQX_ENOMEM: return "out of memory";
    case VQX_ETIMEOUT: return "a device-side wait timed out (results incomplete)";
    default: return "unknown status";
    }
}

int vqx_last_cuda_error(void) { return t_last_cuda_error; }

void vqx_profile_enable(int enable) { t_prof.on = enable != 0; }

void vqx_profile_read(vqx_profile *out, int reset) {
    if (out) *out = t_prof.totals;
    if (reset) t_prof.totals = vqx_profile{};
}

}  // extern "C"

namespace {

// The plane score of "ADR-1397: GPU psnr_hvs twins reproduce the CPU's
// running float sum bit for bit" (Decision): the sum divided in float by the
// term count, then by the float square of the largest sample (compiled with
// contraction off; every operation is one IEEE single operation).
void conclude_hvs(const vqx::HvsOut &w, int bpc, long long n_terms, vqx_hvs_plane *o) {
    o->flags = w.flags & (VQX_FLAG_RANGE | VQX_FLAG_TIMEOUT);
    o->replayed_leaves = w.replayed_leaves;
    if (o->flags & (VQX_FLAG_RANGE | VQX_FLAG_TIMEOUT)) {
        o->sum = o->score = std::nanf("");
        return;
    }
    float sum;
    memcpy(&sum, &w.sum_bits, sizeof sum);
    const float peak = (float)((1u << bpc) - 1u);
    float q = sum / (float)n_terms;
    q = q / (peak * peak);
    o->sum = sum;
    o->score = q;
}

int submit_impl(const void *ref, const void *dist, int width, int height, size_t stride, int bpc,
                int n_frames, vqx_stream_t stream, int kind, unsigned flags, vqx_pending **pending) {
    if (flags & ~VQX_SUBMIT_PLANES_READY) return VQX_EINVAL;
    if (!pending) return VQX_EINVAL;
    *pending = nullptr;
    // out is checked by vqx_plane_stats_finish; any non-null pointer passes here
    int rc = validate(ref, dist, width, height, stride, bpc, n_frames,
                      reinterpret_cast<const vqx_frame_stats *>(pending));
    if (rc != VQX_OK || n_frames == 0) return rc;
    DeviceCtx *ctx = nullptr;
    if ((rc = device_ctx(&ctx)) != VQX_OK) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    const Plan plan = make_plan(*ctx, ref, dist, width, height, stride, bpc, n_frames, kind);

    vqx_pending *p = nullptr;
    if ((rc = acquire_pending(ctx, t_prof.on, &p)) != VQX_OK) return rc;
    if ((rc = acquire_pinned((size_t)n_frames * sizeof(Partial), &p->rec)) != VQX_OK) {
        release_pending(p);
        return rc;
    }
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, records_bytes(plan, n_frames), ctx->pool, st);
    if (e != cudaSuccess) {
        release_pinned(p->rec);
        release_pending(p);
        return cuda_status(e);
    }
    Partial *partials = (Partial *)ws;
    if (p->timed) cudaEventRecord(p->ev[0], st);
    e = launch_stage1(plan, ref, dist, 0, n_frames, partials, st, true,
                      (flags & VQX_SUBMIT_PLANES_READY) != 0);
    if (e == cudaSuccess && p->timed) cudaEventRecord(p->ev[1], st);
    if (e == cudaSuccess) e = launch_stage2(plan, n_frames, partials, (Partial *)p->rec.dev, st);
    if (e == cudaSuccess && p->timed) cudaEventRecord(p->ev[2], st);
    const cudaError_t ef = cudaFreeAsync(ws, st);
    if (e == cudaSuccess) e = ef;
    if (e == cudaSuccess) e = cudaEventRecord(p->done, st);
    if (e != cudaSuccess) {
        // whatever was enqueued finishes before the record buffer is reused
        cudaStreamSynchronize(st);
        release_pinned(p->rec);
        release_pending(p);
        return cuda_status(e);
    }
    p->kind = kind;
    p->n_planes = 1;
    p->n_frames = n_frames;
    p->bpc = bpc;
    p->width = width;
    p->height = height;
    *pending = p;
    return VQX_OK;
}

// Waits for a batch, concludes it into out (vqx_frame_stats or
// vqx_int_psnr_stats records, as kind says; kScores: both, into out and
// out2) and releases the handle.
int finish_impl(vqx_pending *p, int kind, void *out, void *out2 = nullptr) {
    if (!p) return VQX_OK;
    int rc = VQX_OK;
    const cudaError_t e = cudaEventSynchronize(p->done);
    if (e != cudaSuccess) {
        rc = cuda_status(e);
    } else if (!out || p->kind != kind || (kind == kScores && !out2)) {
        rc = VQX_EINVAL;
    } else {
        t_prof.totals.calls++;
        t_prof.totals.kernel_launches += kind == kOrdered ? 4 : 2 * (uint64_t)p->n_planes;
        t_prof.totals.stage1_launches += (uint64_t)p->n_planes;
        if (kind == kHvs)
            t_prof.totals.stage1_bytes += 4ull * (uint64_t)p->n_terms * (uint64_t)p->n_frames;
        else if (kind == kPlanes)
            for (int q = 0; q < p->n_planes; q++)
                t_prof.totals.stage1_bytes += plane_bytes(p->pw[q], p->ph[q], p->bpc, p->n_frames);
        else
            t_prof.totals.stage1_bytes += plane_bytes(p->width, p->height, p->bpc, p->n_frames);
        if (p->timed) {
            float a = 0.f, b = 0.f;
            cudaEventElapsedTime(&a, p->ev[0], p->ev[1]);
            cudaEventElapsedTime(&b, p->ev[1], p->ev[2]);
            t_prof.totals.stage1_ms += a;
            t_prof.totals.stage2_ms += b;
        }
        const Partial *sums = (const Partial *)p->rec.host;
        if (kind == kOrdered) {
            const u64 *w = (const u64 *)p->rec.host;
            for (int f = 0; f < p->n_frames; f++) {
                const u64 *o = w + (size_t)f * vqx::kOrdOut;
                Partial s_f;
                s_f.v[0] = o[3];  // exact noise units
                s_f.v[1] = o[6];  // sample sums
                s_f.v[2] = o[7];
                s_f.v[3] = o[4];  // exact squares
                s_f.v[4] = o[5];
                s_f.v[5] = 0;  // 16 bits: no sample out of range; no device wait to time out
                s_f.v[6] = s_f.v[7] = 0;
                vqx_frame_stats &r = ((vqx_frame_stats *)out)[f];
                conclude(s_f, p->bpc, p->width, p->height, &r, o);
                rc = merge_status(rc, r);
            }
        } else if (kind == kHvs) {
            const vqx::HvsOut *w = (const vqx::HvsOut *)p->rec.host;
            vqx_hvs_plane *o = (vqx_hvs_plane *)out;
            for (int q = 0; q < p->n_frames; q++) {
                conclude_hvs(w[q], p->bpc, p->n_terms, &o[q]);
                rc = merge_status_flags(rc, o[q].flags);
            }
        } else if (kind == kStats) {
            rc = conclude_all(sums, p->n_frames, p->bpc, p->width, p->height, (vqx_frame_stats *)out);
        } else if (kind == kScores) {
            rc = conclude_all(sums, p->n_frames, p->bpc, p->width, p->height, (vqx_frame_stats *)out);
            vqx_int_psnr_stats *o = (vqx_int_psnr_stats *)out2;
            for (int f = 0; f < p->n_frames; f++)
                conclude_int_psnr(sums[f], p->bpc, p->width, p->height, &o[f]);
        } else if (kind == kPlanes) {
            vqx_frame_stats *o = (vqx_frame_stats *)out;
            for (int q = 0; q < p->n_planes; q++)
                for (int f = 0; f < p->n_frames; f++) {
                    vqx_frame_stats &r = o[(size_t)f * p->n_planes + q];
                    conclude(sums[(size_t)q * p->n_frames + f], p->bpc, p->pw[q], p->ph[q], &r);
                    rc = merge_status(rc, r);
                }
        } else {
            vqx_int_psnr_stats *o = (vqx_int_psnr_stats *)out;
            for (int f = 0; f < p->n_frames; f++) {
                conclude_int_psnr(sums[f], p->bpc, p->width, p->height, &o[f]);
                rc = merge_status_flags(rc, o[f].flags);
            }
        }
    }
    if (p->ws) {
        // the batch is over (its event completed, or the wait failed and the
        // context is gone): the workspace goes back to the pool
        cudaFreeAsync(p->ws, p->ctx->copy_stream);
        p->ws = nullptr;
    }
    release_pinned(p->rec);
    release_pending(p);
    return rc;
}

}  // namespace

extern "C" {

int vqx_plane_stats_submit(const void *ref, const void *dist, int width, int height,
                           size_t stride, int bpc, int n_frames, vqx_stream_t stream,
                           unsigned flags, vqx_pending **pending) {
    return submit_impl(ref, dist, width, height, stride, bpc, n_frames, stream, kStats, flags,
                       pending);
}

int vqx_plane_stats_finish(vqx_pending *pending, vqx_frame_stats *out) {
    return finish_impl(pending, kStats, out);
}

int vqx_plane_int_psnr_submit(const void *ref, const void *dist, int width, int height,
                              size_t stride, int bpc, int n_frames, vqx_stream_t stream,
                              unsigned flags, vqx_pending **pending) {
    return submit_impl(ref, dist, width, height, stride, bpc, n_frames, stream, kIntPsnr, flags,
                       pending);
}

int vqx_plane_int_psnr_finish(vqx_pending *pending, vqx_int_psnr_stats *out) {
    return finish_impl(pending, kIntPsnr, out);
}

int vqx_plane_scores_submit(const void *ref, const void *dist, int width, int height,
                            size_t stride, int bpc, int n_frames, vqx_stream_t stream,
                            unsigned flags, vqx_pending **pending) {
    return submit_impl(ref, dist, width, height, stride, bpc, n_frames, stream, kScores, flags,
                       pending);
}

int vqx_plane_scores_finish(vqx_pending *pending, vqx_frame_stats *out,
                            vqx_int_psnr_stats *int_out) {
    return finish_impl(pending, kScores, out, int_out);
}

int vqx_plane_scores(const void *ref, const void *dist, int width, int height, size_t stride,
                     int bpc, int n_frames, vqx_stream_t stream, vqx_frame_stats *out,
                     vqx_int_psnr_stats *int_out) {
    int rc = validate(ref, dist, width, height, stride, bpc, n_frames, out);
    if (rc != VQX_OK || n_frames == 0) return rc;
    if (!int_out) return VQX_EINVAL;
    vqx_pending *p = nullptr;
    rc = submit_impl(ref, dist, width, height, stride, bpc, n_frames, stream, kScores, 0u, &p);
    if (rc != VQX_OK) return rc;
    return finish_impl(p, kScores, out, int_out);
}

int vqx_plane_int_psnr(const void *ref, const void *dist, int width, int height, size_t stride,
                       int bpc, int n_frames, vqx_stream_t stream, vqx_int_psnr_stats *out) {
    int rc = validate(ref, dist, width, height, stride, bpc, n_frames,
                      reinterpret_cast<const vqx_frame_stats *>(out));
    if (rc != VQX_OK || n_frames == 0) return rc;
    vqx_pending *p = nullptr;
    rc = submit_impl(ref, dist, width, height, stride, bpc, n_frames, stream, kIntPsnr, 0u, &p);
    if (rc != VQX_OK) return rc;
    return finish_impl(p, kIntPsnr, out);
}


int vqx_plane_stats(const void *ref, const void *dist, int width, int height, size_t stride,
                    int bpc, int n_frames, vqx_stream_t stream, vqx_frame_stats *out) {
    int rc = validate(ref, dist, width, height, stride, bpc, n_frames, out);
    if (rc != VQX_OK || n_frames == 0) return rc;
    vqx_pending *p = nullptr;
    rc = vqx_plane_stats_submit(ref, dist, width, height, stride, bpc, n_frames, stream, 0u, &p);
    if (rc != VQX_OK) return rc;
    return vqx_plane_stats_finish(p, out);
}

int vqx_planes_stats_submit(const vqx_plane_desc *planes, int n_planes, int bpc, int n_frames,
                           vqx_stream_t stream, unsigned flags, vqx_pending **pending) {
    if (!pending) return VQX_EINVAL;
    *pending = nullptr;
    if (flags & ~VQX_SUBMIT_PLANES_READY) return VQX_EINVAL;
    if (!planes || n_planes < 1 || n_planes > VQX_MAX_PLANES) return VQX_EINVAL;
    if (bpc != 8 && bpc != 10 && bpc != 12 && bpc != 16) return VQX_EBPC;
    if (n_frames < 0) return VQX_EINVAL;
    if (n_frames == 0) return VQX_OK;
    size_t pitch[VQX_MAX_PLANES];
    for (int p = 0; p < n_planes; p++) {
        const int rc = validate_plane(planes[p], bpc, n_frames, &pitch[p]);
        if (rc != VQX_OK) return rc;
    }
    DeviceCtx *ctx = nullptr;
    int rc = device_ctx(&ctx);
    if (rc != VQX_OK) return rc;
    cudaStream_t st = (cudaStream_t)stream;

    Plan plan[VQX_MAX_PLANES];
    size_t off[VQX_MAX_PLANES + 1] = {0};  // record offsets of the planes, in records
    for (int p = 0; p < n_planes; p++) {
        const vqx_plane_desc &d = planes[p];
        plan[p] = make_plan(*ctx, d.ref, d.dist, d.width, d.height, d.stride, bpc, n_frames, kPlanes,
                            1ll << 40, pitch[p]);
        off[p + 1] = off[p] + records_bytes(plan[p], n_frames) / sizeof(Partial);
    }
    vqx_pending *pd = nullptr;
    if ((rc = acquire_pending(ctx, t_prof.on, &pd)) != VQX_OK) return rc;
    if ((rc = acquire_pinned((size_t)n_planes * n_frames * sizeof(Partial), &pd->rec)) != VQX_OK) {
        release_pending(pd);
        return rc;
    }
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, off[n_planes] * sizeof(Partial), ctx->pool, st);
    if (e != cudaSuccess) {
        release_pinned(pd->rec);
        release_pending(pd);
        return cuda_status(e);
    }
    Partial *partials = (Partial *)ws;
    const bool ready = (flags & VQX_SUBMIT_PLANES_READY) != 0;
    if (pd->timed) cudaEventRecord(pd->ev[0], st);
    for (int p = 0; e == cudaSuccess && p < n_planes; p++)
        e = launch_stage1(plan[p], planes[p].ref, planes[p].dist, 0, n_frames, partials + off[p], st,
                          true, ready);
    if (e == cudaSuccess && pd->timed) cudaEventRecord(pd->ev[1], st);
    for (int p = 0; e == cudaSuccess && p < n_planes; p++)
        e = launch_stage2(plan[p], n_frames, partials + off[p],
                          (Partial *)pd->rec.dev + (size_t)p * n_frames, st);
    if (e == cudaSuccess && pd->timed) cudaEventRecord(pd->ev[2], st);
    const cudaError_t ef = cudaFreeAsync(ws, st);
    if (e == cudaSuccess) e = ef;
    if (e == cudaSuccess) e = cudaEventRecord(pd->done, st);
    if (e != cudaSuccess) {
        cudaStreamSynchronize(st);  // whatever was enqueued finishes first
        release_pinned(pd->rec);
        release_pending(pd);
        return cuda_status(e);
    }
    pd->kind = kPlanes;
    pd->n_frames = n_frames;
    pd->bpc = bpc;
    pd->n_planes = n_planes;
    for (int p = 0; p < n_planes; p++) {
        pd->pw[p] = planes[p].width;
        pd->ph[p] = planes[p].height;
    }
    *pending = pd;
    return VQX_OK;
}

int vqx_planes_stats_finish(vqx_pending *pending, vqx_frame_stats *out) {
    return finish_impl(pending, kPlanes, out);
}

int vqx_planes_stats(const vqx_plane_desc *planes, int n_planes, int bpc, int n_frames,
                    vqx_stream_t stream, vqx_frame_stats *out) {
    if (n_frames > 0 && !out) return VQX_EINVAL;
    vqx_pending *p = nullptr;
    const int rc = vqx_planes_stats_submit(planes, n_planes, bpc, n_frames, stream, 0u, &p);
    if (rc != VQX_OK || !p) return rc;
    return finish_impl(p, kPlanes, out);
}

int vqx_plane_stats_host(const void *ref, const void *dist, int width, int height,
                         size_t stride, int bpc, int n_frames, vqx_stream_t stream,
                         vqx_frame_stats *out) {
    int rc = validate(ref, dist, width, height, stride, bpc, n_frames, out);
    if (rc != VQX_OK || n_frames == 0) return rc;
    DeviceCtx *ctx = nullptr;
    if ((rc = device_ctx(&ctx)) != VQX_OK) return rc;
    cudaStream_t st = (cudaStream_t)stream;

    // Device copies of the planes keep the host byte layout but start on a
    // 256-byte boundary.  The last row of the last frame may end before the
    // frame pitch does: copy only the bytes that exist.
    const size_t pitch = (size_t)height * stride;
    const size_t row_bytes = (size_t)width * (size_t)bytes_per_sample(bpc);
    const size_t batch_bytes = (size_t)(n_frames - 1) * pitch + (size_t)(height - 1) * stride + row_bytes;
    const size_t plane_alloc = (batch_bytes + 255) & ~(size_t)255;

    // Chunks of frames: copy chunk k+1 while chunk k is reduced.
    int chunk = n_frames;
    const size_t target = (size_t)64 << 20;  // about 64 MB of each plane per chunk
    if (pitch > 0 && (size_t)n_frames * pitch > target) {
        chunk = (int)(target / pitch);
        if (chunk < 1) chunk = 1;
    }
    const int n_chunks = (n_frames + chunk - 1) / chunk;

    // Plan with the device copies' alignment (256-byte aligned bases).
    const Plan plan = make_plan(*ctx, (const void *)(uintptr_t)256, (const void *)(uintptr_t)256,
                                width, height, stride, bpc, chunk);

    PinnedBuf rec;
    if ((rc = acquire_pinned((size_t)n_frames * sizeof(Partial), &rec)) != VQX_OK) return rc;
    void *ws = nullptr;
    const size_t part_bytes = (records_bytes(plan, n_frames) + 255) & ~(size_t)255;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, 2 * plane_alloc + part_bytes + 256, ctx->pool, st);
    if (e != cudaSuccess) {
        release_pinned(rec);
        return cuda_status(e);
    }
    unsigned char *dr = (unsigned char *)(((uintptr_t)ws + 255) & ~(uintptr_t)255);
    unsigned char *dd = dr + plane_alloc;
    Partial *partials = (Partial *)(dd + plane_alloc);

    std::vector<cudaEvent_t> evs;
    cudaEvent_t ready = nullptr;
    e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(ready, st);  // the workspace exists from here
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->copy_stream, ready, 0);
    for (int k = 0; e == cudaSuccess && k < n_chunks; k++) {
        const int f0 = k * chunk;
        const int nf = (f0 + chunk <= n_frames) ? chunk : n_frames - f0;
        const size_t off = (size_t)f0 * pitch;
        const size_t bytes = (size_t)(nf - 1) * pitch + (size_t)(height - 1) * stride + row_bytes;
        e = cudaMemcpyAsync(dr + off, (const unsigned char *)ref + off, bytes,
                            cudaMemcpyHostToDevice, ctx->copy_stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dd + off, (const unsigned char *)dist + off, bytes,
                                cudaMemcpyHostToDevice, ctx->copy_stream);
        cudaEvent_t ev = nullptr;
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e == cudaSuccess) {
            evs.push_back(ev);
            e = cudaEventRecord(ev, ctx->copy_stream);
        }
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev, 0);
        if (e == cudaSuccess) e = launch_stage1(plan, dr, dd, f0, nf, partials, st);
    }
    if (e == cudaSuccess) e = launch_stage2(plan, n_frames, partials, (Partial *)rec.dev, st);
    // Every copy issued into the workspace must be over before the workspace
    // is freed, also when the loop stopped early on an error: wait for the
    // copy stream on the host (all copies are queued by now, so this costs
    // nothing), then free in the compute stream's order.
    const cudaError_t ec = cudaStreamSynchronize(ctx->copy_stream);
    if (e == cudaSuccess) e = ec;
    const cudaError_t ef = cudaFreeAsync(ws, st);
    const cudaError_t es = cudaStreamSynchronize(st);
    for (cudaEvent_t ev : evs) cudaEventDestroy(ev);
    if (ready) cudaEventDestroy(ready);
    if (e == cudaSuccess) e = ef != cudaSuccess ? ef : es;
    if (e != cudaSuccess) {
        release_pinned(rec);
        return cuda_status(e);
    }
    t_prof.totals.calls++;
    t_prof.totals.kernel_launches += (uint64_t)n_chunks + 1;
    t_prof.totals.stage1_launches += (uint64_t)n_chunks;
    t_prof.totals.stage1_bytes += plane_bytes(width, height, bpc, n_frames);
    rc = conclude_all((const Partial *)rec.host, n_frames, bpc, width, height, out);
    release_pinned(rec);
    return rc;
}

}  // extern "C"

// ====================================================================== CPU-order replay
extern "C" int vqx_plane_stats_ordered_submit(const void *ref, const void *dist, int width,
                                              int height, size_t stride, int bpc, int n_frames,
                                              vqx_stream_t stream, unsigned flags,
                                              vqx_pending **pending) {
    if (!pending) return VQX_EINVAL;
    *pending = nullptr;
    if (flags & ~VQX_SUBMIT_PLANES_READY) return VQX_EINVAL;
    int rc = validate(ref, dist, width, height, stride, bpc, n_frames,
                      reinterpret_cast<const vqx_frame_stats *>(pending));
    if (rc != VQX_OK || n_frames == 0) return rc;
    const uint64_t pixels = (uint64_t)width * (uint64_t)height;
    // Below 16 bits, or up to 2^21 pixels, no CPU sum can reach 2^53 units:
    // the exact sums are the CPU's sums.
    if (bpc != 16 || pixels <= (1u << 21))
        return submit_impl(ref, dist, width, height, stride, bpc, n_frames, stream, kStats, flags,
                           pending);
    if (n_frames > 65535) return VQX_EINVAL;
    // The replay kernels produce every integer sum as well (the blocks' exact
    // sums), so the plain pass is not run here.
    DeviceCtx *ctx = nullptr;
    if ((rc = device_ctx(&ctx)) != VQX_OK) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    const int nb = (int)((pixels + vqx::kOrdBlock - 1) / vqx::kOrdBlock);
    const size_t cells = (size_t)n_frames * vqx::kOrdSeqs * nb;
    const size_t sums_b = cells * sizeof(u64), cls_b = cells * sizeof(int),
                 tab_b = cells * sizeof(vqx::OrdTable), ors_b = cells * sizeof(uint32_t),
                 work_b = cells * sizeof(vqx::OrdWork),
                 ssum_b = (size_t)n_frames * nb * 2 * sizeof(uint32_t);
    vqx_pending *pd = nullptr;
    if ((rc = acquire_pending(ctx, t_prof.on, &pd)) != VQX_OK) return rc;
    if ((rc = acquire_pinned((size_t)n_frames * vqx::kOrdOut * sizeof(u64), &pd->rec)) != VQX_OK) {
        release_pending(pd);
        return rc;
    }
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, sums_b + cls_b + tab_b + ors_b + work_b + ssum_b + 256,
                                            ctx->pool, st);
    if (e != cudaSuccess) {
        release_pinned(pd->rec);
        release_pending(pd);
        return cuda_status(e);
    }
    // sums and tables (8-byte aligned), then the 4-byte arrays
    u64 *sums = (u64 *)ws;
    vqx::OrdTable *tables = (vqx::OrdTable *)((unsigned char *)ws + sums_b);
    int *cls = (int *)((unsigned char *)ws + sums_b + tab_b);
    uint32_t *ors = (uint32_t *)((unsigned char *)ws + sums_b + tab_b + cls_b);
    vqx::OrdWork *work = (vqx::OrdWork *)((unsigned char *)ws + sums_b + tab_b + cls_b + ors_b);
    uint32_t *ssums = (uint32_t *)((unsigned char *)ws + sums_b + tab_b + cls_b + ors_b + work_b);
    int *n_work = (int *)((unsigned char *)ws + sums_b + tab_b + cls_b + ors_b + work_b + ssum_b);
    vqx::OrdPlanes g;
    g.ref = (const unsigned char *)ref;
    g.dist = (const unsigned char *)dist;
    g.frame_pitch = (size_t)height * stride;
    g.stride = stride;
    g.width = width;
    g.pixels = (uint32_t)pixels;
    g.nb = nb;
    g.dense = stride == (size_t)width * 2 && (pixels & 7u) == 0 &&
              (((uintptr_t)ref | (uintptr_t)dist) & 15u) == 0;
    // The block sums are a programmatic dependent of the kernel ahead (the
    // batch ahead's walk, when batches follow each other): they start while
    // it runs and write only this batch's workspace.
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((nb + vqx::kSumWarps - 1) / vqx::kSumWarps, n_frames);
    cfg.blockDim = dim3(32 * vqx::kSumWarps);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int ready = (flags & VQX_SUBMIT_PLANES_READY) ? 1 : 0;
    if (pd->timed) cudaEventRecord(pd->ev[0], st);
    e = cudaLaunchKernelEx(&cfg, vqx::ordered_block_sums, g, sums, ors, ssums, n_work, ready);
    if (e == cudaSuccess && pd->timed) cudaEventRecord(pd->ev[1], st);
    // The kernels after it are programmatic dependents too, each waiting
    // for the one ahead before it reads: their CTAs are in place when it
    // ends, and the next batch's block sums start during this batch's
    // classification, tables and walk.
    if (e == cudaSuccess) {
        cfg.gridDim = dim3(n_frames, vqx::kOrdSeqs);
        cfg.blockDim = dim3(vqx::kClassThreads);
        e = cudaLaunchKernelEx(&cfg, vqx::ordered_classify, (const u64 *)sums, (const uint32_t *)ors,
                               (const uint32_t *)ssums, nb, cls, work, n_work, (u64 *)pd->rec.dev);
    }
    if (e == cudaSuccess) {
        // a fixed grid of warps takes the tabulated blocks from the list
        const size_t jobs_max = (cells + vqx::kTableWarps - 1) / vqx::kTableWarps;
        cfg.gridDim = dim3((unsigned)(jobs_max < (size_t)ctx->sms * 6 ? jobs_max : (size_t)ctx->sms * 6));
        cfg.blockDim = dim3(32 * vqx::kTableWarps);
        e = cudaLaunchKernelEx(&cfg, vqx::ordered_tables, g, (const int *)cls, (const vqx::OrdWork *)work,
                               (const int *)n_work, tables);
    }
    if (e == cudaSuccess) {
        cfg.gridDim = dim3(n_frames, vqx::kOrdSeqs);
        cfg.blockDim = dim3(32);
        e = cudaLaunchKernelEx(&cfg, vqx::ordered_walk, g, (const u64 *)sums, (const uint32_t *)ors,
                               (const int *)cls, (const vqx::OrdTable *)tables, (u64 *)pd->rec.dev);
    }
    if (e == cudaSuccess && pd->timed) cudaEventRecord(pd->ev[2], st);
    if (e == cudaSuccess) e = cudaEventRecord(pd->done, st);
    if (e != cudaSuccess) {
        cudaStreamSynchronize(st);  // whatever was enqueued finishes first
        cudaFreeAsync(ws, st);
        cudaStreamSynchronize(st);
        release_pinned(pd->rec);
        release_pending(pd);
        return cuda_status(e);
    }
    pd->kind = kOrdered;
    pd->n_planes = 1;
    pd->n_frames = n_frames;
    pd->bpc = bpc;
    pd->width = width;
    pd->height = height;
    pd->ws = ws;
    *pending = pd;
    return VQX_OK;
}

extern "C" int vqx_plane_stats_ordered_finish(vqx_pending *pending, vqx_frame_stats *out) {
    // a batch that needed no replay was submitted as a plain one
    return finish_impl(pending, pending && pending->kind == kStats ? kStats : kOrdered, out);
}

extern "C" int vqx_plane_stats_ordered(const void *ref, const void *dist, int width, int height,
                                       size_t stride, int bpc, int n_frames, vqx_stream_t stream,
                                       vqx_frame_stats *out) {
    int rc = validate(ref, dist, width, height, stride, bpc, n_frames, out);
    if (rc != VQX_OK || n_frames == 0) return rc;
    vqx_pending *p = nullptr;
    rc = vqx_plane_stats_ordered_submit(ref, dist, width, height, stride, bpc, n_frames, stream, 0u, &p);
    if (rc != VQX_OK) return rc;
    return vqx_plane_stats_ordered_finish(p, out);
}

// ====================================================================== no-allocation variant
// vqx_plane_stats_noalloc runs the same two kernels as vqx_plane_stats, but
// its scratch (the per-CTA records and the per-frame sums) is the file-scope
// array below instead of memory taken from a pool, and the per-frame sums are
// copied into the caller's own output array instead of a pinned buffer.  It
// therefore never allocates: not at set-up, not per call.
static __device__ __align__(256) vqx::Partial g_noalloc_scratch[VQX_NOALLOC_MAX_RECORDS];

namespace {

// Per-device set-up, done by the first call on each device with that device
// current: the scratch array's device address (in host code the array's name
// is only a host-side stand-in, so kernels must be given this address), the
// SM count and the resident CTAs of each stage-1 variant for planning.
struct NoAllocCtx {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    Partial *scratch = nullptr;
    DeviceCtx planning;  // only sms and resident are filled in
};
NoAllocCtx g_noalloc[kMaxDevices];

cudaError_t init_noalloc(NoAllocCtx &c, int dev) {
    cudaError_t e = cudaGetSymbolAddress((void **)&c.scratch, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (c.scratch == nullptr) return cudaErrorInvalidSymbol;
    e = cudaDeviceGetAttribute(&c.planning.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    return prepare_stage1(c.planning.resident);
}

}  // namespace

extern "C" int vqx_plane_stats_noalloc(const void *ref, const void *dist, int width, int height,
                                       size_t stride, int bpc, int n_frames, vqx_stream_t stream,
                                       vqx_frame_stats *out) {
    int rc = validate(ref, dist, width, height, stride, bpc, n_frames, out);
    if (rc != VQX_OK || n_frames == 0) return rc;
    // one record per frame for the sums plus at least one per frame for stage 1
    if ((long long)n_frames * 2 > (long long)VQX_NOALLOC_MAX_RECORDS) return VQX_EINVAL;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= kMaxDevices) return VQX_EINVAL;
    NoAllocCtx &c = g_noalloc[dev];
    std::call_once(c.once, [&] { c.err = init_noalloc(c, dev); });
    if (c.err != cudaSuccess) return cuda_status(c.err);

    const long long room = (long long)VQX_NOALLOC_MAX_RECORDS / n_frames - 1;  // >= 1
    const Plan plan =
        make_plan(c.planning, ref, dist, width, height, stride, bpc, n_frames, kStats, room);
    Partial *partials = c.scratch;
    Partial *sums = c.scratch + (size_t)n_frames * plan.segs * plan.rec_per_unit;
    cudaStream_t st = (cudaStream_t)stream;
    // Every record is written before it is read, so the scratch needs no
    // clearing between calls.
    e = launch_stage1(plan, ref, dist, 0, n_frames, partials, st);
    if (e == cudaSuccess) e = launch_stage2(plan, n_frames, partials, sums, st);
    // The sums (64 bytes a frame) land in the front of the caller's array,
    // which has 112 bytes a frame; they are concluded in place below.
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(out, sums, (size_t)n_frames * sizeof(Partial), cudaMemcpyDeviceToHost, st);
    const cudaError_t es = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = es;
    if (e != cudaSuccess) return cuda_status(e);
    // Last frame first: record f starts at byte 112 f, at or after the sums of
    // every frame below f, so no sums are overwritten before they are read.
    // That holds only while a record is at least as large as a frame's sums.
    static_assert(sizeof(vqx_frame_stats) >= sizeof(Partial),
                  "in-place conclusion needs records at least as large as the sums");
    rc = VQX_OK;
    for (int f = n_frames - 1; f >= 0; f--) {
        Partial s_f;
        memcpy(&s_f, (const unsigned char *)out + (size_t)f * sizeof(Partial), sizeof s_f);
        conclude(s_f, bpc, width, height, &out[f]);
        rc = merge_status(rc, out[f]);
    }
    return rc;
}

// ====================================================================== psnr_hvs plane sum
namespace {

int validate_hvs(const float *terms, int64_t n_terms, int64_t plane_pitch, int n_planes, int bpc) {
    if (bpc != 8 && bpc != 10 && bpc != 12 && bpc != 16) return VQX_EBPC;
    if (n_planes < 0) return VQX_EINVAL;
    if (n_planes == 0) return VQX_OK;
    if (!terms || ((uintptr_t)terms & 3u) != 0) return VQX_EINVAL;
    if (n_terms < 1 || n_terms > 0x7FFFFFFFll || plane_pitch < n_terms) return VQX_EINVAL;
    const long long nodes = (n_terms + vqx::kHvsNode - 1) / vqx::kHvsNode;
    if ((long long)n_planes * nodes > 0x7FFFFFFFll) return VQX_EINVAL;
    return VQX_OK;
}

}  // namespace

extern "C" int vqx_psnr_hvs_sum_submit(const float *terms, int64_t n_terms, int64_t plane_pitch,
                                       int n_planes, int bpc, vqx_stream_t stream, unsigned flags,
                                       vqx_pending **pending) {
    if (!pending) return VQX_EINVAL;
    *pending = nullptr;
    if (flags & ~VQX_SUBMIT_PLANES_READY) return VQX_EINVAL;
    int rc = validate_hvs(terms, n_terms, plane_pitch, n_planes, bpc);
    if (rc != VQX_OK || n_planes == 0) return rc;
    DeviceCtx *ctx = nullptr;
    if ((rc = device_ctx(&ctx)) != VQX_OK) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    vqx::HvsArgs a;
    a.terms = terms;
    a.n_terms = n_terms;
    a.pitch = plane_pitch;
    a.n_planes = n_planes;
    a.n_leaves = (int)((n_terms + vqx::kHvsLeaf - 1) / vqx::kHvsLeaf);
    a.n_nodes = (a.n_leaves + vqx::kHvsLeaves - 1) / vqx::kHvsLeaves;
    a.vec = ((uintptr_t)terms & 15u) == 0 && (plane_pitch & 3) == 0;
    a.terms_ready = (flags & VQX_SUBMIT_PLANES_READY) ? 1 : 0;
    uint32_t ep = 0;
    while (ep == 0) ep = (ctx->hvs_epoch.fetch_add(1u) + 1u) & vqx::kHvsEpochMask;
    a.epoch = ep;
    const size_t recs = (size_t)n_planes * ((size_t)a.n_leaves + (size_t)a.n_nodes);
    const size_t rec_b = recs * sizeof(vqx::HvsRec);
    const size_t status_b = (size_t)n_planes * a.n_nodes * sizeof(u64);

    vqx_pending *pd = nullptr;
    if ((rc = acquire_pending(ctx, t_prof.on, &pd)) != VQX_OK) return rc;
    if ((rc = acquire_pinned((size_t)n_planes * sizeof(vqx::HvsOut), &pd->rec)) != VQX_OK) {
        release_pending(pd);
        return rc;
    }
    void *ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, rec_b + status_b, ctx->pool, st);
    if (e != cudaSuccess) {
        release_pinned(pd->rec);
        release_pending(pd);
        return cuda_status(e);
    }
    // records (16-byte aligned), then the look-back words; nothing needs
    // clearing (the words carry this call's epoch)
    a.leaves = (vqx::HvsRec *)ws;
    a.nodes = a.leaves + (size_t)n_planes * a.n_leaves;
    a.status = (u64 *)((unsigned char *)ws + rec_b);
    // The tables are a programmatic dependent of the kernel ahead (the batch
    // ahead's walk, when batches follow each other): they start while it
    // runs and write only this call's workspace, which is held until finish
    // so that no later call is given the same memory while this one may run.
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)((size_t)n_planes * a.n_nodes));
    cfg.blockDim = dim3(vqx::kHvsThreads);
    cfg.dynamicSmemBytes = vqx::kHvsTablesSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // Planes of 16-byte aligned terms with a pitch of whole vectors and at
    // least one full row of 32 terms stream through the persistent TMA
    // pipeline; anything else takes one CTA per node.
    const long long rows_full = n_terms / 32;
    const bool tma = a.vec && rows_full >= 1 && ctx->hvs_tma_resident > 0;
    CUtensorMap tm;
    vqx::HvsTmaArgs ta;
    ta.rows_full = rows_full;
    ta.tail = (int)(n_terms % 32);
    if (tma) {
        e = encode_hvs(&tm, terms, rows_full, plane_pitch, n_planes);
        const long long total = (long long)n_planes * a.n_nodes;
        const long long grid = (long long)ctx->hvs_tma_resident * ctx->sms;
        cfg.gridDim = dim3((unsigned)(total < grid ? total : grid));
        cfg.blockDim = dim3(vqx::kHvsTmaThreads);
        cfg.dynamicSmemBytes = vqx::kHvsTmaSmem;
    }
    if (e == cudaSuccess && pd->timed) e = cudaEventRecord(pd->ev[0], st);
    if (e == cudaSuccess)
        e = tma ? cudaLaunchKernelEx(&cfg, vqx::hvs_tables_tma, tm, a, ta)
                : cudaLaunchKernelEx(&cfg, vqx::hvs_tables, a);
    if (e == cudaSuccess && pd->timed) e = cudaEventRecord(pd->ev[1], st);
    if (e == cudaSuccess) {
        // a programmatic dependent of the tables: its warps are in place when
        // they end (a walk warp fits beside a tables CTA)
        cfg.gridDim = dim3((unsigned)n_planes);
        cfg.blockDim = dim3(32);
        cfg.dynamicSmemBytes = 0;
        e = cudaLaunchKernelEx(&cfg, vqx::hvs_walk, a, (vqx::HvsOut *)pd->rec.dev);
    }
    if (e == cudaSuccess && pd->timed) e = cudaEventRecord(pd->ev[2], st);
    if (e == cudaSuccess) e = cudaEventRecord(pd->done, st);
    if (e != cudaSuccess) {
        cudaStreamSynchronize(st);  // whatever was enqueued finishes first
        cudaFreeAsync(ws, st);
        cudaStreamSynchronize(st);
        release_pinned(pd->rec);
        release_pending(pd);
        return cuda_status(e);
    }
    pd->kind = kHvs;
    pd->n_planes = 1;
    pd->n_frames = n_planes;
    pd->bpc = bpc;
    pd->width = pd->height = 0;
    pd->n_terms = n_terms;
    pd->ws = ws;
    *pending = pd;
    return VQX_OK;
}

extern "C" int vqx_psnr_hvs_sum_finish(vqx_pending *pending, vqx_hvs_plane *out) {
    return finish_impl(pending, kHvs, out);
}

extern "C" int vqx_psnr_hvs_sum(const float *terms, int64_t n_terms, int64_t plane_pitch,
                                int n_planes, int bpc, vqx_stream_t stream, vqx_hvs_plane *out) {
    int rc = validate_hvs(terms, n_terms, plane_pitch, n_planes, bpc);
    if (rc != VQX_OK || n_planes == 0) return rc;
    if (!out) return VQX_EINVAL;
    vqx_pending *p = nullptr;
    if ((rc = vqx_psnr_hvs_sum_submit(terms, n_terms, plane_pitch, n_planes, bpc, stream, 0u, &p)) !=
        VQX_OK)
        return rc;
    return vqx_psnr_hvs_sum_finish(p, out);
}
