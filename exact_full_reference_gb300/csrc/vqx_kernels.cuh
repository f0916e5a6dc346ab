// Device side of the fused PSNR-noise + moment reduction (sm_103a).
//
// Stage 1 (fused_stream_tma / fused_rows): one pass over both planes, in
// (frame, segment) units.  Planes with 16-byte aligned rows stream through a
// persistent TMA pipeline (1-D bulk copies for dense frames, 3-D tensor-map
// tiles for padded rows, into a shared-memory ring, with an mbarrier
// hand-off to consumer warps); other layouts are read row by row.  The per-pixel terms are formed and added as
// integers; warp shuffles and a shared-memory step reduce each unit to one
// Partial record, which is *written* (no atomics, nothing to clear
// beforehand).
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

#include <cuda.h>  // CUtensorMap (a plain struct; nothing from the driver library is linked)
#include <cuda_runtime.h>

#include <cstdint>

namespace vqx {

typedef unsigned long long u64;

// One record of sums (a warp's, a CTA's, a unit's or a frame's), 64 bytes:
//   v[0] noise         sum of float(D * D)
//   v[1], v[2]         sums of the reference and distorted samples
//   v[3], v[4]         sums of float(r * r), float(d * d)
//   v[5]               OR of every sample read (the range check), plus
//                      kErrTimeout when a device wait gave up
//   v[6]               the exact sum of D * D minus v[0], modulo 2^64 (the
//                      integer psnr's SSE is v[0] + v[6]); 0 wherever the
//                      float squares are exact or the accumulator does not
//                      form it
//   v[7]               0
// The accumulators' totals() fill the same eight words; every word but v[5]
// is a sum, v[5] an OR.  Records are 16-byte aligned (read as pairs of
// words).
struct __align__(16) Partial {
    u64 v[8];
};
static_assert(sizeof(Partial) == 64, "a record is 64 bytes");
constexpr int kWords = 8;

constexpr int kThreads = 256;     // CTA size of the strided-layout stage-1 kernel
constexpr int kSumThreads = 128;  // stage-2 CTA size

// Shape of the stage-1 TMA pipeline (fused_stream_tma): consumer
// warps, 16-byte vectors per plane per stage, stages in the ring.  Chosen by
// measurement on GB300 over 8-, 10-, 12- and 16-bit batches of 3840x2160 and
// 1920x1080 frames (two large stages beat three or more smaller ones: fewer
// hand-offs per byte); two CTAs (96 KB of ring each) are resident per SM.
constexpr int kTmaWarps = 16;
constexpr int kTmaStageVecs = 1536;
constexpr int kTmaStages = 2;
constexpr int kTmaThreads = (kTmaWarps + 1) * 32;
constexpr size_t kTmaSmem = (size_t)kTmaStages * 2 * kTmaStageVecs * 16;

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

// ---------------------------------------------------------------- TMA + mbarriers
// Bulk copies (cp.async.bulk, the TMA engine's 1-D form) from global to shared
// memory, completed on an mbarrier by transaction bytes.  Every wait on an
// mbarrier is bounded: after about a second (kWaitCycles SM clock cycles) it
// gives up, and the kernel marks its record with kErrTimeout (the host then
// reports VQX_ETIMEOUT) instead of spinning forever.
constexpr long long kWaitCycles = 2000000000ll;
constexpr u64 kErrTimeout = 1ull << 63;  // in Partial::v[5]

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait until the phase of parity `parity` has completed; false after `limit`
// SM clock cycles without completion.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          long long limit = kWaitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (clock64() - t0 > limit) return false;
    }
}
// bytes (a multiple of 16) from 16-byte aligned global src to 16-byte
// aligned shared dst, completing `bytes` transactions on mbarrier bar.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// A 3-D tile of the tensor map tm at element coordinates (x, y, z) into
// shared dst, completing its bytes on mbarrier bar.  x must be a multiple of
// 16 bytes' worth of elements; parts of the box outside the tensor are
// filled with zeros.
__device__ __forceinline__ void tensor_g2s_3d(uint32_t dst, const CUtensorMap *tm, int x, int y,
                                              int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
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
// least once per TermSums::kFlushVecs vec() or sample() calls; totals() returns
// {noise, ref sum, dist sum, ref sum of squares, dist sum of squares, OR of
// samples} in raw units.


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
    static constexpr uint32_t kFlushVecs = 2048;
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
    __device__ __forceinline__ void totals(u64 (&t)[kWords]) {
        flush();
        t[0] = srr + sdd - 2 * srd;
        t[1] = sr;
        t[2] = sd;
        t[3] = srr;
        t[4] = sdd;
        t[5] = t[6] = t[7] = 0;
    }
};

// 10 and 12 bits.  A valid sample is below 2^12, so |D| and s are below
// 2^12, their squares below 2^24, and the float squares are the integer
// squares ("ADR-1440 ...", Decision: below 13 bits no float square rounds).
// Squares and products are added with 32x32->64-bit multiply-adds; the sums
// of samples with dp2a (two 16-bit halves at once).  The OR of all samples
// flags values of 2^bpc or more, for which the library reports VQX_ERANGE.
template <int BPC>
struct TermSums {
    static_assert(BPC == 10 || BPC == 12, "8 and 16 bits have their own forms");
    static constexpr uint32_t kFlushVecs = 2048;
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
    __device__ __forceinline__ void totals(u64 (&t)[kWords]) {
        flush();
        t[0] = rr + dd - 2 * rd;
        t[1] = sr;
        t[2] = sd;
        t[3] = rr;
        t[4] = dd;
        t[5] = (orv & 0xffffu) | (orv >> 16);  // word() ORs two samples per word
        t[6] = t[7] = 0;
    }
};

// Two fp32 lanes in one 64-bit register, lane 0 in the low half.  Blackwell's
// packed fp32 instructions (add/sub/fma .rn.f32x2) apply the scalar IEEE
// operation with round to nearest even to each lane, so every lane's result
// is the one the scalar instruction gives; they halve the issue slots.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_pack(uint32_t lo, uint32_t hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(f32x2 v, uint32_t &lo, uint32_t &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 f2_sub(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// fl(a * a) per lane, as one fused multiply-add with a +0 addend: a single
// round-to-nearest-even of the exact square (+0 adds nothing to a product
// that is +0 or positive).  Not a plain mul.rn.f32x2: the back end was found
// to fuse a packed multiply into the packed add or subtract that consumes it
// (which would add the unrounded square) even with contraction disabled; an
// fma result has nothing left to fuse, and the +0 addend keeps it from being
// rewritten as a plain multiply.
__device__ __forceinline__ f32x2 f2_square(f32x2 a) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %1, %2;" : "=l"(d) : "l"(a), "l"(0ull));
    return d;
}
// fl(a * b + c) per lane: one rounding of the exact a * b + c.
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Exact integer sum of pairs of integer-valued fp32 terms in [0, 2^32),
// without a conversion instruction and without accumulating in floating
// point.  Each term x is split by two exact fp32 additions into
//   h = x rounded to a multiple of 2^16      (x + 1.5*2^39 lies in
//       [2^39, 2^40), where the ulp is 2^16, so that sum is x rounded to a
//       multiple of 2^16, plus 1.5*2^39, and its bits are
//       bits(1.5*2^39) + h / 2^16)
//   l = x - h, an integer of magnitude at most 2^15 (exact)
//                                        (l + 1.5*2^23 lies in [2^23, 2^24),
//       where the ulp is 1: its bits are bits(1.5*2^23) + l)
// and the two bit patterns of both lanes are added as 32-bit integers.  Over
// n terms the sums are n*bits(1.5*2^39) + sum(h)/2^16 and
// n*bits(1.5*2^23) + sum(l), taken modulo 2^32; with at most kMaxTerms
// terms between drains, sum(h)/2^16 < 2^32 and |sum(l)| < 2^31, so the
// true values come back exactly, and sum(x) = 2^16 * sum(h)/2^16 + sum(l).
struct SplitSum2 {
    static constexpr uint32_t kMaxTerms = 32768;  // terms (both lanes) per drain
    static constexpr uint32_t kHiBits = 0x53400000u;  // 1.5 * 2^39
    static constexpr uint32_t kLoBits = 0x4B400000u;  // 1.5 * 2^23
    uint32_t hi = 0, lo = 0, n = 0;

    __device__ __forceinline__ void add(f32x2 x) {
        const f32x2 c_hi = ((f32x2)kHiBits << 32) | kHiBits;
        const f32x2 c_lo = ((f32x2)kLoBits << 32) | kLoBits;
        const f32x2 hb = f2_add(x, c_hi);                      // bits: kHiBits + h/2^16
        const f32x2 lb = f2_add(f2_sub(x, f2_sub(hb, c_hi)), c_lo);  // bits: kLoBits + l
        uint32_t h0, h1, l0, l1;
        f2_unpack(hb, h0, h1);
        f2_unpack(lb, l0, l1);
        hi += h0 + h1;
        lo += l0 + l1;
        n += 2;
    }
    __device__ __forceinline__ u64 drain() {
        const u64 units = (u64)(uint32_t)(hi - n * kHiBits);
        const long long rest = (long long)(int32_t)(lo - n * kLoBits);
        hi = lo = n = 0;
        return units * 65536 + (u64)rest;
    }
};

// 16 bits.  Here the float square rounds (D^2 and s^2 reach 2^32), so the
// terms are the fp32 products, computed as such, two pixels at a time:
// - Floats without conversion: with K = 0x4B000000 (the bits of 2^23), the
//   bits K | s are the float 2^23 + s exactly (s < 2^16), so
//   (2^23 + r) - (2^23 + d) = r - d = D and (2^23 + s) - 2^23 = s are exact
//   fp32 subtractions.
// - fl(D*D), fl(r*r), fl(d*d): one round-to-nearest-even product each (the
//   CPU's terms), integers below 2^32 (f2_square).
// - The reference plane's square stream is split into exact 16-bit parts by
//   a SplitSum2 (fp32 additions) and added as integers, drained into a 64-bit
//   integer at least every kFlushVecs vectors (8 terms each).  The noise and
//   the distorted plane's square streams are converted (exactly: the values
//   are integers below 2^32) with F2I, which runs on the XU pipe, and added in
//   64-bit integers on the ALU pipe.  None of these streams is accumulated
//   in floating point.  The work is spread over the FMA, ALU and XU pipes so that none of
//   them limits the pass (two conversions a pixel keep the XU pipe, a quarter
//   as wide, below its own limit at full HBM bandwidth).
// - Sums of samples: dp2a adds the two 16-bit halves of a word.
// With kSse the same pass also forms the exact sum of D * D (the integer
// psnr's SSE), from the rounding error of each noise square: with D exact in
// fp32 and q = fl(D * D), the fused multiply-add fl(-D * D + q) is exact
// (q - D * D is the rounding error of a product, itself a float: an integer
// of magnitude at most 128, half an ulp of 2^32), so
//   SSE = sum of q - sum of (q - D * D) = noise - sum of the errors.
// The errors are added per lane in fp32, which is exact while the running sum
// stays below 2^24 in magnitude: a run between flushes holds at most
// 4 * kFlushVecs = 8192 terms a lane, so at most 2^20.  Per pixel pair: the
// difference negated by flipping both sign bits (ALU pipe: the FMA pipe is
// the busier one here), one packed fma and one packed add; no further
// conversion.
template <bool kSse>
struct Sums16 {
    static constexpr uint32_t kBias = 0x4B000000u;
    static constexpr uint32_t kFlushVecs = 2048;
    static_assert(8 * kFlushVecs <= SplitSum2::kMaxTerms, "SplitSum2 run bound");
    static_assert(4 * kFlushVecs * 128 <= (1u << 24), "fp32 error sums stay exact");
    static constexpr f32x2 kSigns = 0x8000000080000000ull;  // -x of both lanes: x ^ kSigns
    SplitSum2 rsq_;
    u64 noise = 0, rss = 0, dss = 0, sr = 0, sd = 0;
    long long err = 0;  // sum of fl(D * D) - D * D (kSse)
    f32x2 err_ = 0;     // the current run of it, two fp32 lanes
    uint32_t r_ = 0, d_ = 0;

    __device__ __forceinline__ void pair(f32x2 xr, f32x2 xd) {
        const f32x2 two23 = ((f32x2)kBias << 32) | kBias;
        uint32_t t0, t1;
        const f32x2 diff = f2_sub(xr, xd);
        const f32x2 sq = f2_square(diff);
        f2_unpack(sq, t0, t1);
        noise += (u64)__float2uint_rn(__uint_as_float(t0)) + __float2uint_rn(__uint_as_float(t1));
        if constexpr (kSse) err_ = f2_add(err_, f2_fma(diff ^ kSigns, diff, sq));
        const f32x2 fr = f2_sub(xr, two23);
        rsq_.add(f2_square(fr));
        uint32_t q0, q1;
        f2_unpack(f2_square(f2_sub(xd, two23)), q0, q1);
        dss += (u64)__float2uint_rn(__uint_as_float(q0)) + __float2uint_rn(__uint_as_float(q1));
    }
    __device__ __forceinline__ void word(uint32_t a, uint32_t b) {
        r_ = __dp2a_lo(a, 0x01010101u, r_);
        d_ = __dp2a_lo(b, 0x01010101u, d_);
        pair(f2_pack((a & 0xffffu) | kBias, __byte_perm(a, kBias, 0x7632)),
             f2_pack((b & 0xffffu) | kBias, __byte_perm(b, kBias, 0x7632)));
    }
    __device__ __forceinline__ void vec(const uint4 &a, const uint4 &b) {
        word(a.x, b.x);
        word(a.y, b.y);
        word(a.z, b.z);
        word(a.w, b.w);
    }
    // One pixel in lane 0; lane 1 holds the sample 0, whose terms are 0.
    __device__ __forceinline__ void sample(uint32_t r, uint32_t d) {
        r_ += r;
        d_ += d;
        pair(f2_pack(r | kBias, kBias), f2_pack(d | kBias, kBias));
    }
    __device__ __forceinline__ void flush() {
        sr += r_;
        sd += d_;
        r_ = d_ = 0;
        rss += rsq_.drain();
        if constexpr (kSse) {
            uint32_t e0, e1;
            f2_unpack(err_, e0, e1);
            err += (long long)small_float_to_int(__uint_as_float(e0)) +
                   small_float_to_int(__uint_as_float(e1));
            err_ = 0;
        }
    }
    __device__ __forceinline__ void totals(u64 (&t)[kWords]) {
        flush();
        t[0] = noise;
        t[1] = sr;
        t[2] = sd;
        t[3] = rss;
        t[4] = dss;
        t[5] = 0;
        t[6] = (u64)(-err);  // SSE - noise
        t[7] = 0;
    }
};

template <>
struct TermSums<16> : Sums16<false> {};

// The 16-bit form that also carries the integer psnr's SSE (record word 6).
struct TermSums16Sse : Sums16<true> {};

// Integer psnr at 16 bits: the exact sum of (r - d)^2 (each below 2^32) in a
// 64-bit integer.  Per 32-bit word one packed absolute difference gives the
// two |r - d|, each squared and added by a 64-bit integer multiply-add.  (Up
// to 12 bits the noise terms of TermSums are these squares already: a square
// below 2^24 is exact in fp32.)  Slots 1..5 of the record stay 0.
struct SseSums16 {
    static constexpr uint32_t kFlushVecs = 1u << 20;  // nothing to flush
    u64 sse = 0;

    __device__ __forceinline__ void word(uint32_t a, uint32_t b) {
        const uint32_t d = __vabsdiffu2(a, b);
        const uint32_t lo = d & 0xffffu, hi = d >> 16;
        sse += (u64)lo * lo;
        sse += (u64)hi * hi;
    }
    __device__ __forceinline__ void vec(const uint4 &a, const uint4 &b) {
        word(a.x, b.x);
        word(a.y, b.y);
        word(a.z, b.z);
        word(a.w, b.w);
    }
    __device__ __forceinline__ void sample(uint32_t r, uint32_t d) {
        const uint32_t e = r > d ? r - d : d - r;
        sse += (u64)e * e;
    }
    __device__ __forceinline__ void flush() {}
    __device__ __forceinline__ void totals(u64 (&t)[kWords]) {
        t[0] = sse;
        t[1] = t[2] = t[3] = t[4] = t[5] = t[6] = t[7] = 0;
    }
};

// ---------------------------------------------------------------- reduction
// Warp shuffles, then one value per warp through shared memory, then warp 0:
// words 0..4, 6 and 7 of a record are added, word 5 ORed.  Integer sums:
// exact and independent of the order.
__device__ __forceinline__ u64 combine(int k, u64 a, u64 b) { return k == 5 ? (a | b) : a + b; }

template <int NT>
__device__ __forceinline__ void block_reduce_store(u64 (&t)[kWords], u64 *dst) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int k = 0; k < kWords; k++) t[k] = combine(k, t[k], __shfl_xor_sync(0xffffffffu, t[k], o));
    }
    constexpr int kWarps = NT / 32;
    __shared__ u64 s[kWarps][kWords];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kWords; k++) s[warp][k] = t[k];
    }
    __syncthreads();
    if (warp == 0) {
        u64 y[kWords];
#pragma unroll
        for (int k = 0; k < kWords; k++) y[k] = lane < kWarps ? s[lane][k] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
            for (int k = 0; k < kWords; k++) y[k] = combine(k, y[k], __shfl_xor_sync(0xffffffffu, y[k], o));
        }
        u64 mine = 0;
#pragma unroll
        for (int k = 0; k < kWords; k++)
            if (lane == k) mine = y[k];
        if (lane < kWords) dst[lane] = mine;
    }
}

// ---------------------------------------------------------------- stage 1
// Any layout (the path of rows that are not 16-byte aligned): unit u is
// frame frame0 + u / segs, rows [s * seg_rows, min((s + 1) * seg_rows,
// height)).  A warp walks one row at a time, every sample read on its own.
template <int BPC, class Acc = TermSums<BPC>>
__global__ void __launch_bounds__(kThreads)
    fused_rows(const unsigned char *__restrict__ ref, const unsigned char *__restrict__ dist,
               size_t frame_pitch, size_t stride, int width, int height, int seg_rows, int segs,
               int frame0, Partial *__restrict__ partials) {
    allow_dependent_launch();
    const int unit = blockIdx.x;
    const int f = frame0 + unit / segs;
    const int s = unit - (unit / segs) * segs;
    const int y0 = s * seg_rows;
    const int y1 = min(y0 + seg_rows, height);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned char *rf = ref + (size_t)f * frame_pitch;
    const unsigned char *df = dist + (size_t)f * frame_pitch;

    Acc acc;
    for (int y = y0 + warp; y < y1; y += kThreads / 32) {
        const unsigned char *rr = rf + (size_t)y * stride;
        const unsigned char *dr = df + (size_t)y * stride;
        for (int x = lane; x < width;) {
            const int stop = min(width, x + (int)Acc::kFlushVecs * 32);
            for (; x < stop; x += 32) acc.sample(ld_sample<BPC>(rr, x), ld_sample<BPC>(dr, x));
            acc.flush();
        }
    }
    u64 t[kWords];
    acc.totals(t);
    block_reduce_store<kThreads>(t, partials[(size_t)f * segs + s].v);
}

// Named barrier 1 over the consumer warps only (barrier 0 is __syncthreads).
template <int NCW>
__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(NCW * 32) : "memory");
}

// A warp's totals, reduced and spread over its lanes: the sums (words 0..4
// and 6 of a record) added, word 5 ORed.  The sums take a reduce-scatter over
// eight slots (words 0..4, word 6 and two zeros): at each of the first three
// halvings a lane sends its partner the half of its slots the partner keeps,
// so 18 shuffles do the work of 30 (six sums, five halvings each).  Afterwards lane L holds the sum of slot
// (L >> 2) & 7 (in all four lanes of its group); the OR of word 5 (two 32-bit
// warp reductions) is in every lane.  Word 7 is 0 in every accumulator.
struct WarpTotals {
    u64 sum;    // slot (lane >> 2) & 7
    u64 flags;  // OR of word 5
};

__device__ __forceinline__ WarpTotals warp_reduce_scatter(const u64 (&t)[kWords]) {
    const int lane = threadIdx.x & 31;
    WarpTotals w;
    w.flags = ((u64)__reduce_or_sync(0xffffffffu, (uint32_t)(t[5] >> 32)) << 32) |
              __reduce_or_sync(0xffffffffu, (uint32_t)t[5]);
    const bool up16 = lane & 16, up8 = lane & 8, up4 = lane & 4;
    u64 a[4];  // lanes below 16: slots 0..3; from 16: slots 4..7 = t[4], t[6], 0, 0
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const u64 lo = t[i], hi = i == 0 ? t[4] : i == 1 ? t[6] : 0ull;
        a[i] = (up16 ? hi : lo) + __shfl_xor_sync(0xffffffffu, up16 ? lo : hi, 16);
    }
    u64 b[2];
#pragma unroll
    for (int i = 0; i < 2; i++)
        b[i] = (up8 ? a[2 + i] : a[i]) + __shfl_xor_sync(0xffffffffu, up8 ? a[i] : a[2 + i], 8);
    u64 c = (up4 ? b[1] : b[0]) + __shfl_xor_sync(0xffffffffu, up4 ? b[0] : b[1], 4);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    w.sum = c;
    return w;
}

// The record word a lane group of warp_reduce_scatter writes, and its value:
// slots 0..4 are words 0..4, slot 5 is word 6, slot 6 carries the OR (word
// 5), slot 7 the zero sum (word 7).
__device__ __forceinline__ int slot_word(int slot) { return slot == 5 ? 6 : slot == 6 ? 5 : slot; }
__device__ __forceinline__ u64 slot_value(int slot, const WarpTotals &w) {
    return slot == 6 ? w.flags : w.sum;
}

// One warp's totals to one record (lanes 0, 4, .., 28 store a word each).
// No other warp takes part, so no warp waits at the end of a unit.
__device__ __forceinline__ void warp_reduce_store(const u64 (&t)[kWords], u64 *dst) {
    const WarpTotals w = warp_reduce_scatter(t);
    const int lane = threadIdx.x & 31, slot = (lane >> 2) & 7;
    if ((lane & 3) == 0) dst[slot_word(slot)] = slot_value(slot, w);
}

// The consumer warps' totals reduced to one record: each warp's totals
// through shared memory (warp_reduce_scatter), then lanes 0..7 of warp 0 add
// (or OR) one word each over the warps.  Only consumer threads take part
// (named barrier 1), so the producer lane keeps streaming meanwhile.
template <int NCW>
__device__ __forceinline__ void consumer_reduce_store(const u64 (&t)[kWords], u64 (*scratch)[kWords],
                                                      u64 *dst) {
    const WarpTotals w = warp_reduce_scatter(t);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, slot = (lane >> 2) & 7;
    if ((lane & 3) == 0) scratch[warp][slot_word(slot)] = slot_value(slot, w);
    consumer_sync<NCW>();
    if (warp == 0 && lane < kWords) {
        u64 y = 0;
        for (int k = 0; k < NCW; k++) y = combine(lane, y, scratch[k][lane]);
        dst[lane] = y;
    }
    consumer_sync<NCW>();  // scratch is reused by the next unit
}

// Many small dense frames: each warp takes whole frames (frame frame0 + k
// for k its warp index, then every total-warps-th), reads each one as
// frame_vecs contiguous 16-byte vectors of each plane, and writes the frame's
// single record itself, partials[frame].  No shared memory and no block
// barrier: a frame's end costs one warp's reduction, where a frame split
// across a whole CTA costs sixteen.
constexpr int kFrameWarps = 8;  // warps per CTA of fused_frames

template <int BPC, class Acc = TermSums<BPC>>
__global__ void __launch_bounds__(32 * kFrameWarps)
    fused_frames(const unsigned char *__restrict__ ref, const unsigned char *__restrict__ dist,
                 size_t frame_pitch, uint32_t frame_vecs, int frames, int frame0,
                 Partial *__restrict__ partials) {
    allow_dependent_launch();
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * kFrameWarps;
    for (int k = blockIdx.x * kFrameWarps + (threadIdx.x >> 5); k < frames; k += warps) {
        const int f = frame0 + k;
        const unsigned char *r = ref + (size_t)f * frame_pitch;
        const unsigned char *d = dist + (size_t)f * frame_pitch;
        Acc acc;
        for (uint32_t c = lane; c < frame_vecs;) {
            const uint32_t stop = min(frame_vecs, c + Acc::kFlushVecs * 32);
#pragma unroll 4
            for (; c < stop; c += 32) acc.vec(ld_stream16(r + 16 * (size_t)c), ld_stream16(d + 16 * (size_t)c));
            acc.flush();
        }
        u64 t[kWords];
        acc.totals(t);
        warp_reduce_store(t, partials[f].v);
    }
}

// Where the persistent pipeline's stages come from.  A source maps a unit
// (a (frame, segment) pair) to its stages and issues a stage's two copies
// (reference and distorted plane), arming the stage's full mbarrier with the
// bytes they will deliver.
//
// DenseSource: each frame of each plane is frame_vecs contiguous, 16-byte
// aligned 16-byte vectors.  Unit u is frame frame0 + u / segs, vectors
// [s * seg_vecs, min((s + 1) * seg_vecs, frame_vecs)), s = u % segs, moved
// with 1-D bulk copies of up to SV vectors.
struct DenseSource {
    const unsigned char *ref, *dist;
    size_t frame_pitch;
    uint32_t frame_vecs, seg_vecs;
    int segs, frame0;

    struct Unit {
        const unsigned char *r, *d;
        uint32_t nvec;
        size_t record;
    };
    __device__ __forceinline__ Unit unit(int u) const {
        const int f = frame0 + u / segs, sg = u % segs;
        const uint32_t v0 = min((uint32_t)sg * seg_vecs, frame_vecs);
        Unit x;
        x.nvec = min(v0 + seg_vecs, frame_vecs) - v0;
        x.r = ref + (size_t)f * frame_pitch + (size_t)v0 * 16;
        x.d = dist + (size_t)f * frame_pitch + (size_t)v0 * 16;
        x.record = (size_t)f * segs + sg;
        return x;
    }
    template <int SV>
    __device__ __forceinline__ uint32_t stages(const Unit &x) const {
        return (x.nvec + SV - 1) / SV;
    }
    template <int SV>
    __device__ __forceinline__ uint32_t count(const Unit &x, uint32_t j) const {
        return min((uint32_t)SV, x.nvec - j * SV);
    }
    template <int SV>
    __device__ __forceinline__ void load(const Unit &x, uint32_t j, uint32_t dst_r, uint32_t dst_d,
                                         uint32_t bar) const {
        const uint32_t bytes = count<SV>(x, j) * 16;
        mbar_arrive_expect_tx(bar, 2 * bytes);
        bulk_g2s(dst_r, x.r + (size_t)j * SV * 16, bytes, bar);
        bulk_g2s(dst_d, x.d + (size_t)j * SV * 16, bytes, bar);
    }
};

// RowSource: rows that are a whole number of 16-byte vectors, 16-byte aligned
// bases and row pitch (padded rows).  Unit u is frame frame0 + u / segs, rows
// [s * seg_rows, min((s + 1) * seg_rows, height)); its rows, laid end to end,
// are cut into stages of SV vectors exactly as a dense frame is, each stage
// filled by one bulk copy per row piece it holds (a stage of 24 KB takes four
// or five pieces of a 7680-byte row).
struct RowSource {
    const unsigned char *ref, *dist;
    size_t frame_pitch, stride;
    uint32_t row_vecs;
    int height, seg_rows, segs, frame0;

    struct Unit {
        const unsigned char *r, *d;
        uint32_t nvec;
        size_t record;
    };
    __device__ __forceinline__ Unit unit(int u) const {
        const int f = frame0 + u / segs, sg = u % segs;
        const int y0 = min(sg * seg_rows, height);
        Unit x;
        x.nvec = (uint32_t)(min(y0 + seg_rows, height) - y0) * row_vecs;
        x.r = ref + (size_t)f * frame_pitch + (size_t)y0 * stride;
        x.d = dist + (size_t)f * frame_pitch + (size_t)y0 * stride;
        x.record = (size_t)f * segs + sg;
        return x;
    }
    template <int SV>
    __device__ __forceinline__ uint32_t stages(const Unit &x) const {
        return (x.nvec + SV - 1) / SV;
    }
    template <int SV>
    __device__ __forceinline__ uint32_t count(const Unit &x, uint32_t j) const {
        return min((uint32_t)SV, x.nvec - j * SV);
    }
    template <int SV>
    __device__ __forceinline__ void load(const Unit &x, uint32_t j, uint32_t dst_r, uint32_t dst_d,
                                         uint32_t bar) const {
        const uint32_t v0 = j * SV, end = v0 + count<SV>(x, j);
        mbar_arrive_expect_tx(bar, 2 * (end - v0) * 16);
        for (uint32_t v = v0; v < end;) {
            const uint32_t row = v / row_vecs, col = v - row * row_vecs;
            const uint32_t n = min(row_vecs - col, end - v);
            const size_t off = (size_t)row * stride + (size_t)col * 16;
            bulk_g2s(dst_r + (v - v0) * 16, x.r + off, n * 16, bar);
            bulk_g2s(dst_d + (v - v0) * 16, x.d + off, n * 16, bar);
            v += n;
        }
    }
};

// TileSource: any layout whose bases and row pitch are 16-byte aligned,
// through two 3-D tensor maps (width x height x frames elements of 1 to 8
// bytes, with the row and frame pitches in bytes; the kernel never looks at
// the element type, so the host picks the widest one that divides a row).
// Unit u is frame frame0 + u / segs, rows [s * seg_rows, min((s + 1) *
// seg_rows, height)), seg_rows a multiple of by; its stages are the bx x by
// boxes covering those rows, left to right, top to bottom, each box_vecs
// 16-byte vectors (at most one stage).  Parts of a box past the last column
// or row are filled with zeros by the copy, and zero samples in both planes
// add nothing to any sum.
struct TileSource {
    CUtensorMap tref, tdist;
    int width, height, seg_rows, segs, frame0;
    int bx, by;
    uint32_t box_vecs;

    struct Unit {
        int z, y0, tiles_x;
        uint32_t n;
        size_t record;
    };
    __device__ __forceinline__ Unit unit(int u) const {
        Unit x;
        x.z = u / segs;
        const int sg = u % segs;
        x.y0 = sg * seg_rows;
        const int rows = max(0, min(x.y0 + seg_rows, height) - x.y0);
        x.tiles_x = (width + bx - 1) / bx;
        x.n = (uint32_t)(((rows + by - 1) / by) * x.tiles_x);
        x.record = (size_t)(frame0 + x.z) * segs + sg;
        return x;
    }
    template <int SV>
    __device__ __forceinline__ uint32_t stages(const Unit &x) const {
        return x.n;
    }
    template <int SV>
    __device__ __forceinline__ uint32_t count(const Unit &, uint32_t) const {
        return box_vecs;
    }
    template <int SV>
    __device__ __forceinline__ void load(const Unit &x, uint32_t j, uint32_t dst_r, uint32_t dst_d,
                                         uint32_t bar) const {
        const int ty = x.y0 + (int)(j / x.tiles_x) * by;
        const int tx = (int)(j % x.tiles_x) * bx;
        mbar_arrive_expect_tx(bar, 2 * box_vecs * 16);
        tensor_g2s_3d(dst_r, &tref, tx, ty, x.z, bar);
        tensor_g2s_3d(dst_d, &tdist, tx, ty, x.z, bar);
    }
};

// The persistent TMA pipeline.  CTA b takes units b, b + gridDim.x, ... in
// order.  One producer lane (warp NCW) streams them, stage by stage (SV
// 16-byte vectors of each plane), into a ring of STAGES shared-memory buffers;
// NCW consumer warps wait for a stage's "full" mbarrier, fold it through
// TermSums from shared memory and release it on its "empty" mbarrier (one
// arrive per warp) for the producer to refill.  Loads stay in flight while
// the consumers compute, without holding registers, and the ring does not
// drain between units: at the end of a unit only the consumers meet, to
// reduce and write its record.
//
// Ring phases: the CTA's k-th stage (counted across its units) goes to buffer
// k % STAGES; its full barrier completes phase k / STAGES, and the producer
// refills the buffer for stage k only after the empty barrier completed
// phase k / STAGES - 1 (stage k - STAGES released).  A wait that times out
// sets kErrTimeout in the waiting thread; from then on that warp waits for
// nothing, still writes (flagged) records for its remaining units, and the
// producer waits (bounded) for the copies it issued before the CTA exits.
//
// planes_ready: the caller guarantees that no kernel ahead of this one on the
// stream is still writing the planes when it lets this one start, so the
// producer streams without waiting for it (record stores still wait).
//
// Records: with warp_records every consumer warp writes its own record of
// each unit (record r of the source becomes records r * NCW .. r * NCW +
// NCW - 1) and ends a unit without waiting for the others; otherwise the
// consumers reduce to one record per unit through shared memory.
template <int BPC, int NCW, int SV, int STAGES, class Src, class Acc = TermSums<BPC>>
__global__ void __launch_bounds__((NCW + 1) * 32)
    fused_stream_tma(const __grid_constant__ Src src, int units, int warp_records,
                     int planes_ready, Partial *__restrict__ partials) {
    constexpr uint32_t kStageBytes = SV * 16;  // per plane
    constexpr uint32_t kPerThread = SV / (NCW * 32);
    static_assert(SV % (NCW * 32) == 0, "a full stage gives every consumer thread equal work");
    static_assert(kPerThread <= Acc::kFlushVecs, "flush at least once per stage");
    constexpr uint32_t kStagesPerFlush = Acc::kFlushVecs / kPerThread;
    extern __shared__ __align__(128) unsigned char ring[];  // [STAGES][2][kStageBytes]
    __shared__ __align__(8) u64 full[STAGES], empty[STAGES];
    __shared__ u64 red[NCW][kWords];

    allow_dependent_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring0 = smem_u32(ring);
    const uint32_t full0 = smem_u32(full), empty0 = smem_u32(empty);
    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; i++) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, NCW);
        }
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == NCW) {
        if (lane != 0) return;
        // Launched as a programmatic dependent, this grid may be resident
        // before the kernel ahead of it on the stream has finished: read
        // nothing it may still be writing (returns at once otherwise),
        // unless the caller declared the planes complete already.
        if (!planes_ready) grid_dependency_wait();
        bool ok = true;
        uint32_t k = 0;
        for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
            const typename Src::Unit x = src.unit(u);
            const uint32_t n = src.template stages<SV>(x);
            for (uint32_t j = 0; j < n; j++, k++) {
                const uint32_t st = k % STAGES;
                if (k >= STAGES && !mbar_wait(empty0 + 8 * st, ((k / STAGES) - 1) & 1)) {
                    ok = false;
                    break;
                }
                src.template load<SV>(x, j, ring0 + (2 * st) * kStageBytes,
                                      ring0 + (2 * st + 1) * kStageBytes, full0 + 8 * st);
            }
        }
        // The last copies must have landed before the CTA (and its shared
        // memory) goes away; stages k - STAGES .. k - 1 were issued last.
        for (uint32_t q = k > STAGES ? k - STAGES : 0; q < k; q++)
            mbar_wait(full0 + 8 * (q % STAGES), (q / STAGES) & 1);
        return;
    }

    u64 err = 0;
    uint32_t k = 0;
    bool waited = false;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const typename Src::Unit x = src.unit(u);
        const uint32_t n = src.template stages<SV>(x);
        Acc acc;
        uint32_t since_flush = 0;
        for (uint32_t j = 0; j < n; j++, k++) {
            if (err) continue;  // a wait of this warp timed out: skip, write flagged records
            const uint32_t st = k % STAGES;
            // every lane's wait is bounded; the warp then decides together,
            // so that no lane leaves while others reach __syncwarp
            if (!__all_sync(0xffffffffu, mbar_wait(full0 + 8 * st, (k / STAGES) & 1))) {
                err = kErrTimeout;
                continue;
            }
            const uint4 *a = reinterpret_cast<const uint4 *>(ring + (2 * st) * kStageBytes);
            const uint4 *b = reinterpret_cast<const uint4 *>(ring + (2 * st + 1) * kStageBytes);
            const uint32_t cnt = src.template count<SV>(x, j);
            if (cnt == SV) {
#pragma unroll
                for (uint32_t q = 0; q < kPerThread; q++) {
                    const uint32_t i = threadIdx.x + q * NCW * 32;
                    acc.vec(a[i], b[i]);
                }
            } else {
                for (uint32_t i = threadIdx.x; i < cnt; i += NCW * 32) acc.vec(a[i], b[i]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * st);
            if (++since_flush == kStagesPerFlush) {
                acc.flush();
                since_flush = 0;
            }
        }
        u64 t[kWords];
        acc.totals(t);
        t[5] |= err;
        // The same before the first record store (the kernel ahead may still
        // read records from this memory).
        if (!waited) {
            grid_dependency_wait();
            waited = true;
        }
        if (warp_records)
            warp_reduce_store(t, partials[x.record * NCW + warp].v);
        else
            consumer_reduce_store<NCW>(t, red, partials[x.record].v);
    }
}

// ---------------------------------------------------------------- stage 2
// One CTA per frame: the frame's per_frame Partial records, added in a
// fixed order, written to out[frame] (pinned host memory mapped into the
// device).
__global__ void __launch_bounds__(kSumThreads)
    frame_sums(const Partial *__restrict__ partials, int per_frame, Partial *__restrict__ out) {
    allow_dependent_launch();  // the next batch's stage 1 may start on free SMs
    grid_dependency_wait();
    const int f = blockIdx.x;
    u64 t[kWords] = {0, 0, 0, 0, 0, 0, 0, 0};
    // Records go through L2: stage 1 lets this kernel start before it ends,
    // and the read-only data path needs data unchanged for the reader's whole
    // run.  Two records a thread are loaded at a time; this also keeps the
    // kernel above 40 registers, so that its CTAs do not fit beside two
    // running stage-1 CTAs while they wait: at 32 registers they did, and
    // pipelined steps took 1-4 % longer (the next batch's stage-1 CTAs
    // found the SMs they sat on short of registers).
    const Partial *base = partials + (size_t)f * per_frame;
    int s = threadIdx.x;
    for (; s + kSumThreads < per_frame; s += 2 * kSumThreads) {
        ulonglong2 v[2][kWords / 2];
#pragma unroll
        for (int r = 0; r < 2; r++)
#pragma unroll
            for (int k = 0; k < kWords / 2; k++)
                v[r][k] = __ldcg(reinterpret_cast<const ulonglong2 *>(base + s + r * kSumThreads) + k);
#pragma unroll
        for (int r = 0; r < 2; r++)
#pragma unroll
            for (int k = 0; k < kWords / 2; k++) {
                t[2 * k] = combine(2 * k, t[2 * k], v[r][k].x);
                t[2 * k + 1] = combine(2 * k + 1, t[2 * k + 1], v[r][k].y);
            }
    }
    for (; s < per_frame; s += kSumThreads) {
        const ulonglong2 *p = reinterpret_cast<const ulonglong2 *>(base + s);
#pragma unroll
        for (int k = 0; k < kWords / 2; k++) {
            const ulonglong2 v = __ldcg(p + k);
            t[2 * k] = combine(2 * k, t[2 * k], v.x);
            t[2 * k + 1] = combine(2 * k + 1, t[2 * k + 1], v.y);
        }
    }
    block_reduce_store<kSumThreads>(t, out[f].v);
}

}  // namespace vqx
