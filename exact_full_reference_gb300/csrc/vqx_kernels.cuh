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
// All sums are integers: exact, so the order of additions is free.
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
// Per-thread accumulators.  Each forms, for every pixel, exactly the terms
// listed at the top of this file, and adds them exactly, but without any
// integer <-> float conversion instruction: those run on the SM's narrow XU
// pipe, and with five of them per pixel the literal form was bound by that
// pipe at about half the HBM bandwidth.  Each specialisation states why its
// value is the literal one.
//
// vec() takes 16 bytes of each plane, sample() one sample of each; flush()
// folds the bounded 32-bit / fp32 runs into 64-bit sums and must be called at
// least once per kFlushVecs vec() or sample() calls; totals() returns
// {noise, ref sum, dist sum, ref sum of squares, dist sum of squares, OR of
// samples} in raw units.

// vec() / sample() calls a thread may make between two flush() calls.
constexpr uint32_t kFlushVecs = 2048;

// An fp32 holding an integer of magnitude below 2^22, as an int, by an add:
// x + 1.5 * 2^23 lies in [2^23, 2^24), where the ulp is 1, so that sum is
// exact and its significand field is x + 2^22.
__device__ __forceinline__ int small_float_to_int(float x) {
    return (int)(__float_as_uint(__fadd_rn(x, 12582912.0f)) - 0x4B400000u);
}

template <int BPC>
struct TermSums;

// 8 bits.  Every square is below 2^16 < 2^24, so the float square of a
// difference or of a sample is the integer square.  Four samples share a
// 32-bit word; dp4a adds four byte products at once:
//   sum r, sum d        dp4a(w, 0x01010101)
//   sum r^2, d^2, r*d   dp4a(wr, wr), dp4a(wd, wd), dp4a(wr, wd)
// and sum D^2 = sum r^2 + sum d^2 - 2 sum r*d.  A dp4a adds at most
// 4 * 255^2 = 260100, so 32-bit runs of 2048 vectors (8192 words) stay below
// 2^31.
template <>
struct TermSums<8> {
    u64 sr = 0, sd = 0, srr = 0, sdd = 0, srd = 0;
    uint32_t r_ = 0, d_ = 0, rr_ = 0, dd_ = 0, rd_ = 0;

    __device__ __forceinline__ void word(uint32_t a, uint32_t b) {
        r_ = __dp4a(a, 0x01010101u, r_);
        d_ = __dp4a(b, 0x01010101u, d_);
        rr_ = __dp4a(a, a, rr_);
        dd_ = __dp4a(b, b, dd_);
        rd_ = __dp4a(a, b, rd_);
    }
    __device__ __forceinline__ void vec(const uint4 &a, const uint4 &b) {
        word(a.x, b.x);
        word(a.y, b.y);
        word(a.z, b.z);
        word(a.w, b.w);
    }
    __device__ __forceinline__ void sample(uint32_t r, uint32_t d) {
        r_ += r;
        d_ += d;
        rr_ += r * r;
        dd_ += d * d;
        rd_ += r * d;
    }
    __device__ __forceinline__ void flush() {
        sr += r_;
        sd += d_;
        srr += rr_;
        sdd += dd_;
        srd += rd_;
        r_ = d_ = rr_ = dd_ = rd_ = 0;
    }
    __device__ __forceinline__ void totals(u64 (&t)[6]) {
        flush();
        t[0] = srr + sdd - 2 * srd;
        t[1] = sr;
        t[2] = sd;
        t[3] = srr;
        t[4] = sdd;
        t[5] = 0;
    }
};

// 10 and 12 bits.  A valid sample is below 2^12, so |D| and s are below
// 2^12, their squares below 2^24, and the float squares are the integer
// squares ("ADR-1440 ...", Decision: up to 12 bits the square is exact).
// Squares and products are added with 32x32->64-bit multiply-adds; the sums
// of samples with dp2a (two 16-bit halves at once).  The OR of all samples
// flags values of 2^bpc or more, for which the library reports VQX_ERANGE.
template <int BPC>
struct TermSums {
    static_assert(BPC == 10 || BPC == 12, "8 and 16 bits have their own forms");
    u64 sr = 0, sd = 0, rr = 0, dd = 0, rd = 0;
    uint32_t r_ = 0, d_ = 0, orv = 0;

    __device__ __forceinline__ void pixel(uint32_t r, uint32_t d) {
        rr += (u64)r * r;
        dd += (u64)d * d;
        rd += (u64)r * d;
    }
    __device__ __forceinline__ void word(uint32_t a, uint32_t b) {
        orv |= a | b;
        r_ = __dp2a_lo(a, 0x01010101u, r_);
        d_ = __dp2a_lo(b, 0x01010101u, d_);
        pixel(a & 0xffffu, b & 0xffffu);
        pixel(a >> 16, b >> 16);
    }
    __device__ __forceinline__ void vec(const uint4 &a, const uint4 &b) {
        word(a.x, b.x);
        word(a.y, b.y);
        word(a.z, b.z);
        word(a.w, b.w);
    }
    __device__ __forceinline__ void sample(uint32_t r, uint32_t d) {
        orv |= r | d;
        r_ += r;
        d_ += d;
        pixel(r, d);
    }
    __device__ __forceinline__ void flush() {
        sr += r_;
        sd += d_;
        r_ = d_ = 0;
    }
    __device__ __forceinline__ void totals(u64 (&t)[6]) {
        flush();
        t[0] = rr + dd - 2 * rd;
        t[1] = sr;
        t[2] = sd;
        t[3] = rr;
        t[4] = dd;
        t[5] = (orv & 0xffffu) | (orv >> 16);  // word() ORs two samples per word
    }
};

// 16 bits.  Here the float square rounds (D^2 and s^2 reach 2^32), so the
// terms are the fp32 products, computed as such, and their sum is split as
//   sum fl(x*x) = sum x^2 - sum e,   e = x*x - fl(x*x),
// with both parts exact:
// - Floats without conversion: with K = 0x4B000000 (the bits of 2^23), the
//   bits K | s are the float 2^23 + s exactly (s < 2^16), so
//   (2^23 + r) - (2^23 + d) = r - d = D and (2^23 + s) - 2^23 = s are exact
//   fp32 subtractions.  fl(D*D) and fl(s*s) are single round-to-nearest-even
//   products (__fmul_rn), the CPU's terms.
// - e = fma(x, x, -fl(x*x)) is exact: the fused operation rounds the exact
//   x*x - fl(x*x), an integer of magnitude at most 128 (half an ulp below
//   2^32), which fp32 holds.  Runs of at most 2048 vectors (16384 pixels)
//   keep the fp32 sums of e below 2^21 in magnitude, hence exact.
// - sum x^2: the bit patterns K + s are integers, so 32x32->64-bit
//   multiply-adds give B_rr = sum (K + r)^2, B_dd and B_rd = sum (K + r)(K + d)
//   modulo 2^64, and
//     sum r^2 = B_rr - n K^2 - 2 K sum r,   sum r d = B_rd - n K^2 - K (sum r + sum d)
//   hold modulo 2^64; the true values are below 2^57, so they are exact.
//   sum D^2 = sum r^2 + sum d^2 - 2 sum r d.
// The products fl(x*x) are formed with __fmul_rn and the residuals with an
// explicit __fmaf_rn; nothing else is fused (the file is built with
// --fmad=false).
template <>
struct TermSums<16> {
    static constexpr uint32_t kBias = 0x4B000000u;
    u64 brr = 0, bdd = 0, brd = 0, sr = 0, sd = 0;
    long long en = 0, er = 0, ed = 0;
    uint32_t r_ = 0, d_ = 0, n = 0;
    float en_ = 0.f, er_ = 0.f, ed_ = 0.f;

    __device__ __forceinline__ void pixel(uint32_t br, uint32_t bd) {
        const float xr = __uint_as_float(br);
        const float xd = __uint_as_float(bd);
        const float diff = __fsub_rn(xr, xd);
        const float t = __fmul_rn(diff, diff);
        en_ = __fadd_rn(en_, __fmaf_rn(diff, diff, -t));
        const float fr = __fsub_rn(xr, 8388608.0f);
        const float fd = __fsub_rn(xd, 8388608.0f);
        const float qr = __fmul_rn(fr, fr);
        const float qd = __fmul_rn(fd, fd);
        er_ = __fadd_rn(er_, __fmaf_rn(fr, fr, -qr));
        ed_ = __fadd_rn(ed_, __fmaf_rn(fd, fd, -qd));
        brr += (u64)br * br;
        bdd += (u64)bd * bd;
        brd += (u64)br * bd;
    }
    __device__ __forceinline__ void word(uint32_t a, uint32_t b) {
        r_ = __dp2a_lo(a, 0x01010101u, r_);
        d_ = __dp2a_lo(b, 0x01010101u, d_);
        pixel((a & 0xffffu) | kBias, (b & 0xffffu) | kBias);
        pixel(__byte_perm(a, kBias, 0x7632), __byte_perm(b, kBias, 0x7632));
    }
    __device__ __forceinline__ void vec(const uint4 &a, const uint4 &b) {
        word(a.x, b.x);
        word(a.y, b.y);
        word(a.z, b.z);
        word(a.w, b.w);
        n += 8;
    }
    __device__ __forceinline__ void sample(uint32_t r, uint32_t d) {
        r_ += r;
        d_ += d;
        pixel(r | kBias, d | kBias);
        n += 1;
    }
    __device__ __forceinline__ void flush() {
        sr += r_;
        sd += d_;
        r_ = d_ = 0;
        en += small_float_to_int(en_);
        er += small_float_to_int(er_);
        ed += small_float_to_int(ed_);
        en_ = er_ = ed_ = 0.f;
    }
    __device__ __forceinline__ void totals(u64 (&t)[6]) {
        flush();
        const u64 K = kBias, K2 = K * K, N = n;
        const u64 rr = brr - N * K2 - 2 * K * sr;
        const u64 dd = bdd - N * K2 - 2 * K * sd;
        const u64 rd = brd - N * K2 - K * (sr + sd);
        t[0] = rr + dd - 2 * rd - (u64)en;
        t[1] = sr;
        t[2] = sd;
        t[3] = rr - (u64)er;
        t[4] = dd - (u64)ed;
        t[5] = 0;
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
    while (v < v1) {
        // at most kFlushVecs vectors per thread before the next flush
        const uint32_t stop = min(v1, v + kFlushVecs * kThreads);
        for (; v + (kUnroll - 1) * kThreads < stop; v += kUnroll * kThreads) {
            uint4 a[kUnroll], b[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; u++) {
                a[u] = ld_stream16(R + v + u * kThreads);
                b[u] = ld_stream16(D + v + u * kThreads);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; u++) acc.vec(a[u], b[u]);
        }
        for (; v < stop; v += kThreads) acc.vec(ld_stream16(R + v), ld_stream16(D + v));
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
            for (int c = lane; c < nvec;) {
                const int stop = min(nvec, c + (int)kFlushVecs * 32);
                for (; c < stop; c += 32)
                    acc.vec(ld_stream16(rr + 16 * (size_t)c), ld_stream16(dr + 16 * (size_t)c));
                acc.flush();
            }
            x0 = nvec * (16 / kBps);
        }
        for (int x = x0 + lane; x < width;) {
            const int stop = min(width, x + (int)kFlushVecs * 32);
            for (; x < stop; x += 32) acc.sample(ld_sample<BPC>(rr, x), ld_sample<BPC>(dr, x));
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
