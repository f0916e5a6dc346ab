// Device side of the fused PSNR-noise + moment reduction (sm_103a).
//
// Stage 1 (fused_dense / fused_rows): one pass over both planes.  Each CTA
// owns one (frame, segment) unit, streams its samples with 16-byte
// non-allocating loads, forms the per-pixel terms and adds them as integers;
// warp shuffles and a shared-memory step reduce the CTA to one Partial record,
// which it *writes* (no atomics, nothing to clear beforehand).
//
// Stage 2 (frame_sums): one CTA per frame adds the frame's Partial records
// (integers, so the order is irrelevant and the result deterministic) and
// writes the frame's sums straight into pinned, mapped host memory.  It is
// launched with programmatic dependent launch and waits on the grid
// dependency, so its launch latency hides under stage 1's tail.
//
// Per-pixel terms ("ADR-1440: float_psnr_hip adds its squared differences as
// integers ...", Decision; "ADR-1447: float_moment_hip adds the float squares
// the CPU adds ...", Decision): with r, d raw samples,
//   noise term  float(float(r) - float(d))^2 rounded to nearest even, an
//               integer below 2^32 equal to the CPU's term times S^2;
//   moments     r, d, and float(r * r), float(d * d) (one RNE product each).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace vqx {

typedef unsigned long long u64;

// One CTA's sums: noise, ref sum, dist sum, ref sum of squares, dist sum of
// squares, and the OR of every sample read (for the range check).
struct Partial {
    u64 v[6];
};

constexpr int kThreads = 256;      // stage-1 CTA size
constexpr int kSumThreads = 128;   // stage-2 CTA size
constexpr int kUnroll = 2;         // 16-byte vectors per plane in flight per thread

// ---------------------------------------------------------------- loads
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

template <int BPC>
__device__ __forceinline__ uint32_t ld_sample(const unsigned char *row, int x) {
    if constexpr (BPC == 8) {
        return __ldg(row + x);
    } else {
        return __ldg(reinterpret_cast<const unsigned short *>(row) + x);
    }
}

// ---------------------------------------------------------------- PDL
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- terms
// The per-pixel arithmetic, literally: both samples converted to fp32, the
// difference and the squares taken with explicit round-to-nearest-even
// operations (never contracted into an FMA), the integer-valued products
// converted back to integers and added into 64-bit sums.
template <int BPC>
struct TermSums {
    u64 noise = 0, rs = 0, ds = 0, rss = 0, dss = 0;
    uint32_t orv = 0;

    __device__ __forceinline__ void sample(uint32_t r, uint32_t d) {
        const float fr = __uint2float_rn(r);
        const float fd = __uint2float_rn(d);
        const float diff = __fsub_rn(fr, fd);
        noise += __float2uint_rn(__fmul_rn(diff, diff));
        rss += __float2uint_rn(__fmul_rn(fr, fr));
        dss += __float2uint_rn(__fmul_rn(fd, fd));
        rs += r;
        ds += d;
        if constexpr (BPC == 10 || BPC == 12) orv |= r | d;
    }

    __device__ __forceinline__ void word(uint32_t a, uint32_t b) {
        if constexpr (BPC == 8) {
#pragma unroll
            for (int k = 0; k < 4; k++) sample((a >> (8 * k)) & 0xffu, (b >> (8 * k)) & 0xffu);
        } else {
            sample(a & 0xffffu, b & 0xffffu);
            sample(a >> 16, b >> 16);
        }
    }

    __device__ __forceinline__ void vec(const uint4 &a, const uint4 &b) {
        word(a.x, b.x);
        word(a.y, b.y);
        word(a.z, b.z);
        word(a.w, b.w);
    }

    __device__ __forceinline__ void flush() {}

    __device__ __forceinline__ void totals(u64 (&t)[6]) const {
        t[0] = noise;
        t[1] = rs;
        t[2] = ds;
        t[3] = rss;
        t[4] = dss;
        t[5] = orv;
    }
};

// ---------------------------------------------------------------- reduction
// Warp shuffles, then one value per warp through shared memory, then warp 0.
// Integer sums: exact and independent of the order.
template <int NT>
__device__ __forceinline__ void block_reduce_store(u64 (&t)[6], u64 *dst) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int k = 0; k < 5; k++) t[k] += __shfl_xor_sync(0xffffffffu, t[k], o);
        t[5] |= __shfl_xor_sync(0xffffffffu, t[5], o);
    }
    constexpr int kWarps = NT / 32;
    __shared__ u64 s[kWarps][6];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < 6; k++) s[warp][k] = t[k];
    }
    __syncthreads();
    if (warp == 0) {
        u64 y[6];
#pragma unroll
        for (int k = 0; k < 6; k++) y[k] = lane < kWarps ? s[lane][k] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
            for (int k = 0; k < 5; k++) y[k] += __shfl_xor_sync(0xffffffffu, y[k], o);
            y[5] |= __shfl_xor_sync(0xffffffffu, y[5], o);
        }
        u64 mine = 0;
#pragma unroll
        for (int k = 0; k < 6; k++)
            if (lane == k) mine = y[k];
        if (lane < 6) dst[lane] = mine;
    }
}

// ---------------------------------------------------------------- stage 1
// Dense layout: each frame of each plane is frame_vecs contiguous 16-byte
// vectors (16-byte aligned, rows packed).  Unit u of the grid is frame
// frame0 + u / segs, vectors [s * seg_vecs, min((s + 1) * seg_vecs,
// frame_vecs)) with s = u % segs.
template <int BPC>
__global__ void __launch_bounds__(kThreads)
    fused_dense(const unsigned char *__restrict__ ref, const unsigned char *__restrict__ dist,
                size_t frame_pitch, uint32_t frame_vecs, uint32_t seg_vecs, int segs, int frame0,
                Partial *__restrict__ partials) {
    allow_dependent_launch();
    const int unit = blockIdx.x;
    const int f = frame0 + unit / segs;
    const int s = unit - (unit / segs) * segs;
    const uint32_t v0 = (uint32_t)s * seg_vecs;
    const uint32_t v1 = min(v0 + seg_vecs, frame_vecs);
    const uint4 *R = reinterpret_cast<const uint4 *>(ref + (size_t)f * frame_pitch);
    const uint4 *D = reinterpret_cast<const uint4 *>(dist + (size_t)f * frame_pitch);

    TermSums<BPC> acc;
    uint32_t v = v0 + threadIdx.x;
    for (; v + (kUnroll - 1) * kThreads < v1; v += kUnroll * kThreads) {
        uint4 a[kUnroll], b[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; u++) {
            a[u] = ld_stream16(R + v + u * kThreads);
            b[u] = ld_stream16(D + v + u * kThreads);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; u++) acc.vec(a[u], b[u]);
        acc.flush();
    }
    for (; v < v1; v += kThreads) {
        acc.vec(ld_stream16(R + v), ld_stream16(D + v));
        acc.flush();
    }
    u64 t[6];
    acc.totals(t);
    block_reduce_store<kThreads>(t, partials[(size_t)f * segs + s].v);
}

// Any layout: unit u is frame frame0 + u / segs, rows [s * seg_rows,
// min((s + 1) * seg_rows, height)).  A warp walks one row at a time.  With
// VEC, rows start 16-byte aligned and are read as 16-byte vectors plus a
// scalar tail; without, every sample is read on its own.
template <int BPC, bool VEC>
__global__ void __launch_bounds__(kThreads)
    fused_rows(const unsigned char *__restrict__ ref, const unsigned char *__restrict__ dist,
               size_t frame_pitch, size_t stride, int width, int height, int seg_rows, int segs,
               int frame0, Partial *__restrict__ partials) {
    allow_dependent_launch();
    constexpr int kBps = BPC == 8 ? 1 : 2;
    const int unit = blockIdx.x;
    const int f = frame0 + unit / segs;
    const int s = unit - (unit / segs) * segs;
    const int y0 = s * seg_rows;
    const int y1 = min(y0 + seg_rows, height);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned char *rf = ref + (size_t)f * frame_pitch;
    const unsigned char *df = dist + (size_t)f * frame_pitch;

    TermSums<BPC> acc;
    for (int y = y0 + warp; y < y1; y += kThreads / 32) {
        const unsigned char *rr = rf + (size_t)y * stride;
        const unsigned char *dr = df + (size_t)y * stride;
        int x0 = 0;
        if constexpr (VEC) {
            const int nvec = (width * kBps) >> 4;
            for (int c = lane; c < nvec; c += 32) {
                acc.vec(ld_stream16(rr + 16 * (size_t)c), ld_stream16(dr + 16 * (size_t)c));
                acc.flush();
            }
            x0 = nvec * (16 / kBps);
        }
        for (int x = x0 + lane; x < width; x += 32) {
            acc.sample(ld_sample<BPC>(rr, x), ld_sample<BPC>(dr, x));
            acc.flush();
        }
    }
    u64 t[6];
    acc.totals(t);
    block_reduce_store<kThreads>(t, partials[(size_t)f * segs + s].v);
}

// ---------------------------------------------------------------- stage 2
// One CTA per frame: the frame's segs Partial records, added in a fixed
// order, written to out[frame] (pinned host memory mapped into the device).
__global__ void __launch_bounds__(kSumThreads)
    frame_sums(const Partial *__restrict__ partials, int segs, Partial *__restrict__ out) {
    grid_dependency_wait();
    const int f = blockIdx.x;
    u64 t[6] = {0, 0, 0, 0, 0, 0};
    for (int s = threadIdx.x; s < segs; s += kSumThreads) {
        const Partial &p = partials[(size_t)f * segs + s];
#pragma unroll
        for (int k = 0; k < 5; k++) t[k] += p.v[k];
        t[5] |= p.v[5];
    }
    block_reduce_store<kSumThreads>(t, out[f].v);
}

}  // namespace vqx
