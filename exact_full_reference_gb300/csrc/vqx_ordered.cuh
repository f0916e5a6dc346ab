// Replay of the CPU's sequential double sums past 2^53 units (16-bit only).
//
// The CPU adds each frame's terms (the float squares of the differences, and
// of each plane's samples) one after another, in raster order, into a double
// ("ADR-1440: float_psnr_hip adds its squared differences as integers ...",
// Context; "ADR-1447: float_moment_hip adds the float squares the CPU adds
// ...", Context).  Below 2^53 units those sums are exact; beyond, every add
// rounds, and the result depends on the order.  ADR-1447 (Alternatives)
// names this replay as the way to be bit-identical everywhere.  The terms
// are integers below 2^32 and the running sum S never decreases, so:
//
// - While S stays in one binade [2^(52+k), 2^(53+k)) (ulp u = 2^k), S is a
//   multiple of u, and S + t rounds to S + (t - r) or S + (t - r) + u with
//   r = t mod u: down if r < u/2, up if r > u/2, and on a tie towards the
//   multiple of 2u.  So one add is a function of one bit, the parity
//   p = (S / u) mod 2, returning the rounding error and the new parity; a
//   block of adds composes to such a function: its transfer table
//   (E[p], p'[p]) for p = 0, 1.
// - Blocks are runs of kOrdBlock raster pixels.  From the blocks' exact sums
//   and their prefix P, a block is classified: all prefixes below 2^53
//   (exact: S += T), inside one binade even allowing for the accumulated
//   rounding error (|S - P| < 2^28, since at most 2^25 adds round, each by at
//   most 8 units) (tabulated), or near a boundary (replayed term by term in
//   double arithmetic).
// - One walk per frame and sum applies the blocks in order.
//
// Kernels: ordered_block_sums -> ordered_classify -> ordered_tables ->
// ordered_walk.  The terms are recomputed from the planes: an fp32 subtract
// and square (each rounded to nearest even, never fused), then the exact
// integer conversion.  Dense frames (contiguous rows, 16-byte aligned) are
// read as 16-byte vectors and their samples turned into floats without a
// conversion instruction (the bits 0x4B000000 | s are the float 2^23 + s);
// other layouts are read sample by sample.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "vqx_kernels.cuh"

namespace vqx {

constexpr int kOrdBlock = 4096;   // raster pixels per block
constexpr int kOrdSeqs = 3;       // 0: noise, 1: reference squares, 2: distorted squares
constexpr int kOrdExact = -1;     // block class: every prefix below 2^53
constexpr int kOrdReplay = 99;    // block class: replay term by term
constexpr int kOrdLane = kOrdBlock / 32;  // terms per lane in ordered_tables
constexpr u64 kTwo53 = 1ull << 53;
constexpr u64 kOrdMargin = 1ull << 28;

struct OrdTable {
    long long e[2];  // rounding error of the block for input parity 0, 1
    int p[2];        // output parity for input parity 0, 1
};



// Where a plane pair's frames are: frame f of each plane starts f *
// frame_pitch bytes after its base, rows stride bytes apart; the pixels of a
// frame are numbered in raster order and cut into nb blocks of kOrdBlock.
// dense: rows contiguous (stride = 2 width), bases 16-byte aligned and the
// pixel count a multiple of 8, so that block b of frame f is the bytes
// [2 b kOrdBlock, 2 (b kOrdBlock + len)) of the frame, whole 16-byte vectors.
struct OrdPlanes {
    const unsigned char *ref, *dist;
    size_t frame_pitch, stride;
    int width;
    uint32_t pixels;
    int nb;
    int dense;
};

__device__ __forceinline__ uint32_t ord_len(const OrdPlanes &g, int b) {
    return min((uint32_t)kOrdBlock, g.pixels - (uint32_t)b * kOrdBlock);
}

// The float of a 16-bit sample without a conversion: (2^23 + s) - 2^23.
__device__ __forceinline__ float ord_float(uint32_t s) {
    return __fsub_rn(__uint_as_float(0x4B000000u | s), 8388608.0f);
}

// The three terms of one pixel: fl(fl(r) - fl(d))^2, fl(r * r), fl(d * d),
// each an integer below 2^32.
__device__ __forceinline__ void ord_terms(uint32_t r, uint32_t d, uint32_t (&t)[kOrdSeqs]) {
    const float fr = ord_float(r), fd = ord_float(d);
    const float diff = __fsub_rn(fr, fd);
    t[0] = __float2uint_rn(__fmul_rn(diff, diff));
    t[1] = __float2uint_rn(__fmul_rn(fr, fr));
    t[2] = __float2uint_rn(__fmul_rn(fd, fd));
}

__device__ __forceinline__ uint32_t ord_term(int q, uint32_t r, uint32_t d) {
    uint32_t t[kOrdSeqs];
    ord_terms(r, d, t);
    return t[q];
}

// Plane loads go through L2 (ld.global.cg), not the read-only data path:
// these kernels are programmatic dependents of the kernel ahead, so they
// may start while a kernel that writes the planes is still running (the
// caller's, when it lets its dependents start early), and the read-only path
// needs data unchanged for the reading kernel's whole run.
__device__ __forceinline__ uint4 ord_ld16(const unsigned char *p) {
    return __ldcg(reinterpret_cast<const uint4 *>(p));
}

// Calls fn(j, r, d) for every pixel j of block b of frame f, the lanes
// (threads) of the calling group sharing the work: nthreads of them, this
// one tid.  Dense frames go 16-byte vector by vector (8 pixels, j in raster
// order), others row segment by row segment (coalesced within a row).
template <class Fn>
__device__ __forceinline__ void ord_block_pixels(const OrdPlanes &g, int f, int b, int tid,
                                                 int nthreads, Fn fn) {
    const uint32_t i0 = (uint32_t)b * kOrdBlock, len = ord_len(g, b);
    const unsigned char *rf = g.ref + (size_t)f * g.frame_pitch;
    const unsigned char *df = g.dist + (size_t)f * g.frame_pitch;
    if (g.dense) {
        const unsigned char *rb = rf + 2 * (size_t)i0, *db = df + 2 * (size_t)i0;
        for (uint32_t v = tid; v < len / 8; v += nthreads) {
            const uint4 a = ord_ld16(rb + 16 * (size_t)v), c = ord_ld16(db + 16 * (size_t)v);
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int w = 0; w < 4; w++) {
                fn(8 * v + 2 * w, aw[w] & 0xffffu, cw[w] & 0xffffu);
                fn(8 * v + 2 * w + 1, aw[w] >> 16, cw[w] >> 16);
            }
        }
        return;
    }
    uint32_t y = i0 / (uint32_t)g.width, x = i0 - y * (uint32_t)g.width;
    for (uint32_t j0 = 0; j0 < len;) {
        const uint32_t n = min((uint32_t)g.width - x, len - j0);
        const unsigned short *rr = reinterpret_cast<const unsigned short *>(rf + (size_t)y * g.stride) + x;
        const unsigned short *dr = reinterpret_cast<const unsigned short *>(df + (size_t)y * g.stride) + x;
        for (uint32_t k = tid; k < n; k += nthreads)
            fn(j0 + k, (uint32_t)__ldcg(rr + k), (uint32_t)__ldcg(dr + k));
        j0 += n;
        y++;
        x = 0;
    }
}

// Grid (blocks per frame / kSumWarps, frames), one warp per block: the exact
// sums of the three term sequences over each block, sums[(f * nb + b) * 3 +
// q], the OR of each sequence's terms (at least of their low 16 bits),
// ors[same index] (a block whose terms are all multiples of the ulp it works
// at adds without rounding), and the sums of the block's reference and
// distorted samples, ssums[(f * nb + b) * 2 + 0, 1] (below 4096 * 2^16 =
// 2^28).
// Dense frames, two pixels of a 32-bit word at a time: the samples' floats
// from their bits, the three products as packed fp32 pairs (each lane one
// round-to-nearest-even product, fma with +0 so that nothing fuses); the noise
// and distorted squares converted to integers (F2I) and added in 64 bits, the
// reference squares split by exact fp32 additions into a multiple of 2^16 and
// a remainder of magnitude at most 2^15 whose bit patterns are added as
// 32-bit integers (SplitSum2's form), so that the conversions, which run on
// the SM's narrow XU pipe and bound this pass at three a pixel, are two.  The
// remainder's bit pattern ends in the square's low 16 bits (the multiple of
// 2^16 adds nothing there), so ORing the patterns gives the OR of the
// reference squares' low 16 bits: all that the replay tests of it (ulps up to
// 2^4, as every sum stays below 2^57).  The samples are summed by a two-way
// dot product.
struct OrdWordSums {
    u64 t[kOrdSeqs] = {0, 0, 0};
    uint32_t o[kOrdSeqs] = {0, 0, 0};
    uint32_t hi = 0, lo = 0, n = 0;  // reference squares as split bit patterns
    uint32_t sr = 0, sd = 0;

    __device__ __forceinline__ void word(uint32_t a, uint32_t b) {
        constexpr uint32_t kBias = 0x4B000000u;
        const f32x2 two23 = ((f32x2)kBias << 32) | kBias;
        const f32x2 c_hi = ((f32x2)SplitSum2::kHiBits << 32) | SplitSum2::kHiBits;
        const f32x2 c_lo = ((f32x2)SplitSum2::kLoBits << 32) | SplitSum2::kLoBits;
        const f32x2 xr = f2_pack((a & 0xffffu) | kBias, __byte_perm(a, kBias, 0x7632));
        const f32x2 xd = f2_pack((b & 0xffffu) | kBias, __byte_perm(b, kBias, 0x7632));
        uint32_t v[2][2];
        f2_unpack(f2_square(f2_sub(xr, xd)), v[0][0], v[0][1]);
        f2_unpack(f2_square(f2_sub(xd, two23)), v[1][0], v[1][1]);
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const int q = i == 0 ? 0 : 2;
            const uint32_t x0 = __float2uint_rn(__uint_as_float(v[i][0]));
            const uint32_t x1 = __float2uint_rn(__uint_as_float(v[i][1]));
            t[q] += (u64)x0 + x1;
            o[q] |= x0 | x1;
        }
        const f32x2 rsq = f2_square(f2_sub(xr, two23));
        const f32x2 hb = f2_add(rsq, c_hi);                            // kHiBits + h / 2^16
        const f32x2 lb = f2_add(f2_sub(rsq, f2_sub(hb, c_hi)), c_lo);  // kLoBits + l
        uint32_t h0, h1, l0, l1;
        f2_unpack(hb, h0, h1);
        f2_unpack(lb, l0, l1);
        hi += h0 + h1;
        lo += l0 + l1;
        o[1] |= l0 | l1;
        n += 2;
        sr = __dp2a_lo(a, 0x01010101u, sr);
        sd = __dp2a_lo(b, 0x01010101u, sd);
    }
    // the exact sum of sequence q (at most 2^15 split terms, far inside
    // SplitSum2's bound)
    __device__ __forceinline__ u64 total(int q) const {
        if (q != 1) return t[q];
        const u64 units = (u64)(uint32_t)(hi - n * SplitSum2::kHiBits);
        const long long rest = (long long)(int32_t)(lo - n * SplitSum2::kLoBits);
        return t[1] + units * 65536 + (u64)rest;
    }
};

// A warp's sums of one block to the block's records: the three exact
// sums, their ORs and the two sample sums (see ordered_block_sums).
__device__ __forceinline__ void ord_store_block(const OrdWordSums &w, int f, int b, int nb, int lane,
                                                u64 *__restrict__ sums, uint32_t *__restrict__ ors,
                                                uint32_t *__restrict__ ssums) {
    u64 tot[kOrdSeqs];
#pragma unroll
    for (int q = 0; q < kOrdSeqs; q++) tot[q] = w.total(q);
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1)
#pragma unroll
        for (int q = 0; q < kOrdSeqs; q++) tot[q] += __shfl_xor_sync(0xffffffffu, tot[q], sh);
    uint32_t o[kOrdSeqs];
#pragma unroll
    for (int q = 0; q < kOrdSeqs; q++) o[q] = __reduce_or_sync(0xffffffffu, w.o[q]);
    const uint32_t sr = __reduce_add_sync(0xffffffffu, w.sr), sd = __reduce_add_sync(0xffffffffu, w.sd);
    const size_t slot = ((size_t)f * nb + b) * kOrdSeqs;
    if (lane < kOrdSeqs) {
        sums[slot + lane] = lane == 0 ? tot[0] : lane == 1 ? tot[1] : tot[2];
        ors[slot + lane] = lane == 0 ? o[0] : lane == 1 ? o[1] : o[2];
    } else if (lane < kOrdSeqs + 2) {
        ssums[((size_t)f * nb + b) * 2 + (lane - kOrdSeqs)] = lane == kOrdSeqs ? sr : sd;
    }
}

constexpr int kSumWarps = 4;  // blocks (one per warp) per CTA of ordered_block_sums

//
// Launched as a programmatic dependent of the batch ahead, the kernel writes
// only its own batch's workspace (which the batch ahead does not hold) and,
// unless planes_ready, waits for the kernel ahead before reading the planes.
// It also zeroes the work-list count that ordered_classify appends to.
__global__ void __launch_bounds__(32 * kSumWarps, 10)
    ordered_block_sums(const OrdPlanes g, u64 *__restrict__ sums, uint32_t *__restrict__ ors,
                       uint32_t *__restrict__ ssums, int *__restrict__ n_work, int planes_ready) {
    allow_dependent_launch();  // this batch's classification may be scheduled now
    if (!planes_ready) grid_dependency_wait();
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *n_work = 0;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kSumWarps + (threadIdx.x >> 5), f = blockIdx.y;
    if (b >= g.nb) return;
    OrdWordSums w;
    if (g.dense) {
        const uint32_t len = ord_len(g, b);
        const size_t off = (size_t)f * g.frame_pitch + 2 * (size_t)b * kOrdBlock;
        const unsigned char *rb = g.ref + off, *db = g.dist + off;
#pragma unroll 8
        for (uint32_t v = lane; v < len / 8; v += 32) {
            const uint4 x = ord_ld16(rb + 16 * (size_t)v), y = ord_ld16(db + 16 * (size_t)v);
            w.word(x.x, y.x);
            w.word(x.y, y.y);
            w.word(x.z, y.z);
            w.word(x.w, y.w);
        }
    } else {
        ord_block_pixels(g, f, b, lane, 32, [&](uint32_t, uint32_t r, uint32_t d) {
            uint32_t x[kOrdSeqs];
            ord_terms(r, d, x);
#pragma unroll
            for (int q = 0; q < kOrdSeqs; q++) {
                w.t[q] += x[q];
                w.o[q] |= x[q];
            }
            w.sr += r;
            w.sd += d;
        });
    }
    ord_store_block(w, f, b, g.nb, lane, sums, ors, ssums);
}

__device__ __forceinline__ int binade_of(u64 x) { return 63 - __clzll((long long)x); }

// A tabulated block to compute: frame, sequence, block.
struct OrdWork {
    int f, q, b;
};

// Loads of what a kernel ahead on the stream wrote.  The classification,
// tables and walk are launched as programmatic dependents, before the kernels
// ahead have ended; the read-only data path needs data unchanged for the
// reading kernel's whole run, so these loads go through L2 instead.
__device__ __forceinline__ OrdWork ld_work(const OrdWork *p) {
    return OrdWork{__ldcg(&p->f), __ldcg(&p->q), __ldcg(&p->b)};
}
__device__ __forceinline__ OrdTable ld_table(const OrdTable *p) {
    OrdTable t;
    t.e[0] = __ldcg(&p->e[0]);
    t.e[1] = __ldcg(&p->e[1]);
    const int2 v = __ldcg(reinterpret_cast<const int2 *>(p->p));
    t.p[0] = v.x;
    t.p[1] = v.y;
    return t;
}

constexpr int kOrdBatch = 8;  // chunks of 32 blocks loaded at once by the one-warp kernels
constexpr int kOrdOut = 8;    // words per frame of the ordered kernels' output

// Grid (frames, 3), kClassThreads threads: prefix sums over the blocks of
// one sequence and the class of every block, cls[(f * 3 + q) * nb + b]; the
// q = 0 CTA also adds the blocks' sample sums into out[f * kOrdOut + 6, 7].
// Thread t takes a run of consecutive blocks; the runs' sums are scanned
// across the CTA (warp scans, then the warps' totals), and each thread walks
// its run from its exclusive prefix.  A single-binade block whose terms are
// all multiples of the binade's ulp is exact.  Every tabulated block is
// appended to work (count in *n_work, which starts at 0).
constexpr int kClassThreads = 512;

__global__ void __launch_bounds__(kClassThreads)
    ordered_classify(const u64 *__restrict__ sums, const uint32_t *__restrict__ ors,
                     const uint32_t *__restrict__ ssums, int nb, int *__restrict__ cls,
                     OrdWork *__restrict__ work, int *__restrict__ n_work, u64 *__restrict__ out) {
    allow_dependent_launch();
    grid_dependency_wait();  // the block sums are complete
    constexpr int kWarps = kClassThreads / 32;
    const int f = blockIdx.x, q = blockIdx.y, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int per = (nb + kClassThreads - 1) / kClassThreads;
    const int b0 = min(t * per, nb), b1 = min(b0 + per, nb);
    const size_t row = (size_t)f * nb;
    u64 mine = 0, sr = 0, sd = 0;
    for (int b = b0; b < b1; b++) {
        mine += __ldcg(sums + (row + b) * kOrdSeqs + q);
        if (q == 0) {
            sr += __ldcg(ssums + (row + b) * 2);
            sd += __ldcg(ssums + (row + b) * 2 + 1);
        }
    }
    // exclusive prefix of this thread's run
    u64 incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const u64 v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    __shared__ u64 wsum[kWarps];
    __shared__ int wcount[kWarps];
    __shared__ int wbase[kWarps];
    __shared__ u64 s2[kWarps][2];
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    u64 before = 0;
    for (int w = 0; w < warp; w++) before += wsum[w];
    u64 P = before + incl - mine;
    // classify the run, counting the tabulated blocks
    int ntab = 0;
    for (int b = b0; b < b1; b++) {
        const size_t in = (row + b) * kOrdSeqs + q;
        const u64 T = __ldcg(sums + in), P1 = P + T;
        int c = kOrdReplay;
        if (P1 < kTwo53) {
            c = kOrdExact;
        } else if (P >= kTwo53 + kOrdMargin && binade_of(P - kOrdMargin) == binade_of(P1 + kOrdMargin)) {
            c = binade_of(P) - 52;
            // the running sum is a multiple of 2^c here; so are the terms?
            if ((__ldcg(ors + in) & ((1u << c) - 1)) == 0) c = kOrdExact;
        }
        cls[((size_t)f * kOrdSeqs + q) * nb + b] = c;
        ntab += c != kOrdExact && c != kOrdReplay;
        P = P1;
    }
    // places in the work list: a scan of the counts, one atomic per CTA
    int cincl = ntab;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, cincl, o);
        if (lane >= o) cincl += v;
    }
    if (lane == 31) wcount[warp] = cincl;
    if (q == 0) {
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) {
            sr += __shfl_xor_sync(0xffffffffu, sr, sh);
            sd += __shfl_xor_sync(0xffffffffu, sd, sh);
        }
        if (lane == 0) {
            s2[warp][0] = sr;
            s2[warp][1] = sd;
        }
    }
    __syncthreads();
    if (t == 0) {
        int total = 0;
        for (int w = 0; w < kWarps; w++) {
            wbase[w] = total;
            total += wcount[w];
        }
        const int first = total ? atomicAdd(n_work, total) : 0;
        for (int w = 0; w < kWarps; w++) wbase[w] += first;
        if (q == 0) {
            u64 a = 0, d = 0;
            for (int w = 0; w < kWarps; w++) {
                a += s2[w][0];
                d += s2[w][1];
            }
            out[(size_t)f * kOrdOut + 6] = a;
            out[(size_t)f * kOrdOut + 7] = d;
        }
    }
    __syncthreads();
    int slot = wbase[warp] + cincl - ntab;
    for (int b = b0; b < b1 && ntab; b++) {
        const int c = cls[((size_t)f * kOrdSeqs + q) * nb + b];
        if (c != kOrdExact && c != kOrdReplay) work[slot++] = OrdWork{f, q, b};
    }
}

// One add of term t to a sum whose ulp is 2^k and parity p: returns the
// rounding error (result - (sum + t)) and updates p.
__device__ __forceinline__ int ord_step(uint32_t t, int k, int &p) {
    const uint32_t u = 1u << k, r = t & (u - 1), half = u >> 1, q = t >> k;
    const int qp = (int)(q & 1u);
    const bool up = r > half || (r == half && ((p + qp) & 1));
    p = (p + qp + (up ? 1 : 0)) & 1;
    return up ? (int)(u - r) : -(int)r;
}

// A block's effect at one ulp 2^k, for input parity 0 and 1: the rounding
// error and the output parity.  compose(g, h) is g, then h.
struct OrdFn {
    long long e0, e1;
    int p0, p1;
};

__device__ __forceinline__ OrdFn ord_compose(const OrdFn &g, const OrdFn &h) {
    OrdFn c;
    c.e0 = g.e0 + (g.p0 ? h.e1 : h.e0);
    c.p0 = g.p0 ? h.p1 : h.p0;
    c.e1 = g.e1 + (g.p1 ? h.e1 : h.e0);
    c.p1 = g.p1 ? h.p1 : h.p0;
    return c;
}

// Inclusive scan of the lanes' functions in lane order (lane l ends with
// f_0, then f_1, .., then f_l).
__device__ __forceinline__ OrdFn ord_scan(OrdFn fn, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        OrdFn g;
        g.e0 = __shfl_up_sync(0xffffffffu, fn.e0, o);
        g.e1 = __shfl_up_sync(0xffffffffu, fn.e1, o);
        g.p0 = __shfl_up_sync(0xffffffffu, fn.p0, o);
        g.p1 = __shfl_up_sync(0xffffffffu, fn.p1, o);
        if (lane >= o) fn = ord_compose(g, fn);
    }
    return fn;
}

constexpr int kTableWarps = 2;  // warps per CTA in ordered_tables (33 KB of staged terms)

// Fixed grid of kTableWarps-warp CTAs: each warp takes tabulated blocks from
// the work list and writes their transfer tables.  The block's terms are
// staged in the warp's shared memory with one pad word every kOrdLane
// words, so that lane l reading its run [l * kOrdLane, (l + 1) * kOrdLane)
// hits a different bank than the others; each lane folds its run for both
// input parities and a warp scan composes the runs.
__global__ void __launch_bounds__(32 * kTableWarps)
    ordered_tables(const OrdPlanes g, const int *__restrict__ cls, const OrdWork *__restrict__ work,
                   const int *__restrict__ n_work, OrdTable *__restrict__ tables) {
    allow_dependent_launch();
    grid_dependency_wait();  // the classification is complete
    __shared__ uint32_t terms_all[kTableWarps][kOrdBlock + kOrdBlock / kOrdLane];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    uint32_t *terms = terms_all[wib];
    const int n = __ldcg(n_work);
    for (int w = blockIdx.x * kTableWarps + wib; w < n; w += gridDim.x * kTableWarps) {
        const OrdWork job = ld_work(work + w);
        const size_t slot = ((size_t)job.f * kOrdSeqs + job.q) * g.nb + job.b;
        const int k = __ldcg(cls + slot);
        const uint32_t len = ord_len(g, job.b);
        ord_block_pixels(g, job.f, job.b, lane, 32, [&](uint32_t j, uint32_t r, uint32_t d) {
            terms[j + j / kOrdLane] = ord_term(job.q, r, d);
        });
        __syncwarp();
        OrdFn fn{0, 0, 0, 1};
        const uint32_t j0 = (uint32_t)lane * kOrdLane;
        for (uint32_t j = j0; j < j0 + kOrdLane && j < len; j++) {
            const uint32_t t = terms[j + j / kOrdLane];
            fn.e0 += ord_step(t, k, fn.p0);
            fn.e1 += ord_step(t, k, fn.p1);
        }
        fn = ord_scan(fn, lane);
        if (lane == 31) {
            OrdTable tb;
            tb.e[0] = fn.e0;
            tb.e[1] = fn.e1;
            tb.p[0] = fn.p0;
            tb.p[1] = fn.p1;
            tables[slot] = tb;
        }
        __syncwarp();  // terms is rewritten by the next job
    }
}

// One add of t to S (an integer below 2^58 that a double holds exactly), as
// the CPU's double add does it: the exact integer sum rounded to 53
// significant bits, to nearest with ties to even.
__device__ __forceinline__ u64 ord_add_rne(u64 S, uint32_t t) {
    u64 x = S + t;
    const int nbits = 64 - __clzll((long long)x);
    if (nbits <= 53) return x;
    const int sh = nbits - 53;
    const u64 ulp = 1ull << sh, r = x & (ulp - 1), half = ulp >> 1;
    x -= r;
    if (r > half || (r == half && ((x >> sh) & 1))) x += ulp;
    return x;
}

// A replayed block (its len terms staged in shared memory, seen by the whole
// warp) added to S.  Lane l takes the run [l kOrdLane, (l + 1) kOrdLane):
// its exact sum and, from S and the runs before it, its class as in
// ordered_classify (exact below 2^53; inside one binade with the margin;
// otherwise crossing a boundary).  A single-binade run folds its function
// of the parity at that binade's ulp; then the runs are applied in order, a
// crossing run (at most a few in a frame) term by term.
__device__ u64 ord_replay_block(u64 S, const uint32_t *terms, uint32_t len, int lane) {
    const uint32_t j0 = (uint32_t)lane * kOrdLane, j1 = min(j0 + (uint32_t)kOrdLane, len);
    u64 R = 0;
    for (uint32_t j = j0; j < j1; j++) R += terms[j];
    u64 incl = R;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const u64 v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    const u64 a = S + (incl - R), a1 = a + R;
    int c = kOrdReplay;
    if (a1 < kTwo53)
        c = kOrdExact;
    else if (a >= kTwo53 + kOrdMargin && binade_of(a - kOrdMargin) == binade_of(a1 + kOrdMargin))
        c = binade_of(a) - 52;
    OrdFn fn{0, 0, 0, 1};
    if (c != kOrdExact && c != kOrdReplay)
        for (uint32_t j = j0; j < j1; j++) {
            fn.e0 += ord_step(terms[j], c, fn.p0);
            fn.e1 += ord_step(terms[j], c, fn.p1);
        }
    for (int l = 0; l < 32; l++) {
        const int cl = __shfl_sync(0xffffffffu, c, l);
        const u64 Rl = __shfl_sync(0xffffffffu, R, l);
        if (cl == kOrdExact) {
            S += Rl;
        } else if (cl != kOrdReplay) {
            const long long e0 = __shfl_sync(0xffffffffu, fn.e0, l);
            const long long e1 = __shfl_sync(0xffffffffu, fn.e1, l);
            S += Rl + (u64)(((S >> cl) & 1) ? e1 : e0);
        } else {
            if (lane == 0) {
                const uint32_t k1 = min((uint32_t)(l + 1) * kOrdLane, len);
                for (uint32_t j = (uint32_t)l * kOrdLane; j < k1; j++) S = ord_add_rne(S, terms[j]);
            }
            S = __shfl_sync(0xffffffffu, S, 0);
        }
    }
    return S;
}

// Grid (frames, 3), one warp: the walk.  Every lane carries the CPU's
// running sum S (an integer below 2^57, exact in a double and in 64 bits)
// through the blocks, 32 at a time, one per lane (kOrdBatch chunks loaded at
// once):
// - a chunk of exact blocks adds its exact sum;
// - a chunk of blocks that all work at one ulp 2^k (tabulated at k, or exact
//   with a sum that is a multiple of 2^k) composes the blocks' functions of
//   the parity (S / 2^k) mod 2 by a warp scan and applies the result once;
// - any other chunk goes block by block: exact and tabulated blocks as
//   above; a block near a boundary adds exactly when the running sum and all
//   of its terms are multiples of the largest ulp it can reach, and is
//   otherwise replayed (ord_replay_block).
// out[f * kOrdOut + q] = S, out[f * kOrdOut + 3 + q] = the exact sum of the
// sequence.
__global__ void __launch_bounds__(32)
    ordered_walk(const OrdPlanes g, const u64 *__restrict__ sums, const uint32_t *__restrict__ ors,
                 const int *__restrict__ cls, const OrdTable *__restrict__ tables,
                 u64 *__restrict__ out) {
    allow_dependent_launch();  // the next batch's block sums may start on free SMs
    grid_dependency_wait();    // the tables are complete
    const int f = blockIdx.x, q = blockIdx.y, lane = threadIdx.x;
    __shared__ uint32_t terms[kOrdBlock];
    const int nb = g.nb;
    u64 S = 0, exact = 0;
    for (int cb = 0; cb < nb; cb += 32 * kOrdBatch) {
        int cB[kOrdBatch];
        u64 TB[kOrdBatch];
        uint32_t oB[kOrdBatch];
        OrdTable tbB[kOrdBatch];
#pragma unroll
        for (int u = 0; u < kOrdBatch; u++) {  // all loads first, then the chunks in order
            const int b = cb + 32 * u + lane;
            const bool valid = b < nb;
            const size_t slot = ((size_t)f * kOrdSeqs + q) * nb + b;
            const size_t in = ((size_t)f * nb + b) * kOrdSeqs + q;
            cB[u] = valid ? __ldcg(cls + slot) : kOrdExact;
            TB[u] = valid ? __ldcg(sums + in) : 0;
            oB[u] = valid ? __ldcg(ors + in) : 0;
            tbB[u] = OrdTable{{0, 0}, {0, 1}};
            if (valid && cB[u] != kOrdExact && cB[u] != kOrdReplay) tbB[u] = ld_table(tables + slot);
        }
#pragma unroll
        for (int u = 0; u < kOrdBatch; u++) {
            const int c0 = cb + 32 * u;
            if (c0 >= nb) break;
            const int c = cB[u];
            const u64 T = TB[u];
            const bool tab = c != kOrdExact && c != kOrdReplay;
            u64 sumT = T;
#pragma unroll
            for (int sh = 16; sh > 0; sh >>= 1) sumT += __shfl_xor_sync(0xffffffffu, sumT, sh);
            exact += sumT;
            if (__all_sync(0xffffffffu, c == kOrdExact)) {
                S += sumT;
                continue;
            }
            const int kmin = __reduce_min_sync(0xffffffffu, tab ? c : 1000);
            const int kmax = __reduce_max_sync(0xffffffffu, tab ? c : -1);
            const bool fits = c != kOrdReplay && (tab || (T & ((1ull << kmin) - 1)) == 0);
            if (kmin == kmax && __all_sync(0xffffffffu, fits)) {
                const int k = kmin;
                OrdFn fn;
                if (tab) {
                    fn = OrdFn{tbB[u].e[0], tbB[u].e[1], tbB[u].p[0], tbB[u].p[1]};
                } else {  // exact, a multiple of 2^k: the parity flips with bit k of T
                    const int t1 = (int)((T >> k) & 1);
                    fn = OrdFn{0, 0, t1, t1 ^ 1};
                }
                fn = ord_scan(fn, lane);
                const long long e0 = __shfl_sync(0xffffffffu, fn.e0, 31);
                const long long e1 = __shfl_sync(0xffffffffu, fn.e1, 31);
                S += sumT + (u64)(((S >> k) & 1) ? e1 : e0);
                continue;
            }
            // block by block (every lane follows the same steps)
            const int n = min(32, nb - c0);
            for (int i = 0; i < n; i++) {
                const int ci = __shfl_sync(0xffffffffu, c, i);
                const u64 Ti = __shfl_sync(0xffffffffu, T, i);
                if (ci == kOrdExact) {
                    S += Ti;
                } else if (ci != kOrdReplay) {
                    const long long e0 = __shfl_sync(0xffffffffu, tbB[u].e[0], i);
                    const long long e1 = __shfl_sync(0xffffffffu, tbB[u].e[1], i);
                    S += Ti + (u64)(((S >> ci) & 1) ? e1 : e0);
                } else {
                    const uint32_t oi = __shfl_sync(0xffffffffu, oB[u], i);
                    const u64 top = S + Ti + kOrdMargin;
                    const int kneed = top < kTwo53 ? 0 : binade_of(top) - 52;
                    const u64 mask = (1ull << kneed) - 1;
                    if (((S | (u64)oi) & mask) == 0) {
                        S += Ti;
                    } else {
                        const int bb = c0 + i;
                        const uint32_t len = ord_len(g, bb);
                        ord_block_pixels(g, f, bb, lane, 32, [&](uint32_t j, uint32_t r, uint32_t d) {
                            terms[j] = ord_term(q, r, d);
                        });
                        __syncwarp();
                        S = ord_replay_block(S, terms, len, lane);
                        __syncwarp();  // terms is rewritten by the next replayed block
                    }
                }
            }
        }
    }
    if (lane == 0) {
        out[(size_t)f * kOrdOut + q] = S;
        out[(size_t)f * kOrdOut + 3 + q] = exact;
    }
}

}  // namespace vqx
