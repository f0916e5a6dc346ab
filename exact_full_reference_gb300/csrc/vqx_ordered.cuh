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
// ordered_walk.  The terms are recomputed from the planes in the literal
// form (fp32 subtract and square, then the exact integer conversion).
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

__device__ __forceinline__ uint32_t ord_term(int q, uint32_t r, uint32_t d) {
    const float fr = __uint2float_rn(r), fd = __uint2float_rn(d);
    if (q == 0) {
        const float diff = __fsub_rn(fr, fd);
        return __float2uint_rn(__fmul_rn(diff, diff));
    }
    const float x = q == 1 ? fr : fd;
    return __float2uint_rn(__fmul_rn(x, x));
}

// Calls fn(j, r, d) for the raster pixels [i0, i0 + len) of frame f, j the
// offset in the block; the CTA's threads share the work row segment by row
// segment (coalesced within a row).
template <class Fn>
__device__ __forceinline__ void ord_block_pixels(const unsigned char *ref, const unsigned char *dist,
                                                 size_t frame_pitch, size_t stride, int width,
                                                 int f, uint32_t i0, uint32_t len, Fn fn) {
    uint32_t y = i0 / (uint32_t)width, x = i0 - y * (uint32_t)width;
    for (uint32_t j0 = 0; j0 < len;) {
        const uint32_t n = min((uint32_t)width - x, len - j0);
        const unsigned short *rr = reinterpret_cast<const unsigned short *>(
                                       ref + (size_t)f * frame_pitch + (size_t)y * stride) + x;
        const unsigned short *dr = reinterpret_cast<const unsigned short *>(
                                       dist + (size_t)f * frame_pitch + (size_t)y * stride) + x;
        for (uint32_t k = threadIdx.x; k < n; k += blockDim.x) fn(j0 + k, (uint32_t)rr[k], (uint32_t)dr[k]);
        j0 += n;
        y++;
        x = 0;
    }
}

// Grid (blocks per frame, frames), 128 threads: the exact sums of the three
// term sequences over each block, sums[(f * nb + b) * 3 + q], and the OR of
// each sequence's terms, ors[same index] (a block whose terms are all
// multiples of the ulp it works at adds without rounding).
__global__ void __launch_bounds__(128)
    ordered_block_sums(const unsigned char *__restrict__ ref, const unsigned char *__restrict__ dist,
                       size_t frame_pitch, size_t stride, int width, uint32_t pixels, int nb,
                       u64 *__restrict__ sums, uint32_t *__restrict__ ors) {
    const int b = blockIdx.x, f = blockIdx.y;
    const uint32_t i0 = (uint32_t)b * kOrdBlock;
    const uint32_t len = min((uint32_t)kOrdBlock, pixels - i0);
    u64 t[kOrdSeqs] = {0, 0, 0};
    uint32_t o[kOrdSeqs] = {0, 0, 0};
    ord_block_pixels(ref, dist, frame_pitch, stride, width, f, i0, len,
                     [&](uint32_t, uint32_t r, uint32_t d) {
#pragma unroll
                         for (int q = 0; q < kOrdSeqs; q++) {
                             const uint32_t x = ord_term(q, r, d);
                             t[q] += x;
                             o[q] |= x;
                         }
                     });
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1)
#pragma unroll
        for (int q = 0; q < kOrdSeqs; q++) {
            t[q] += __shfl_xor_sync(0xffffffffu, t[q], sh);
            o[q] |= __shfl_xor_sync(0xffffffffu, o[q], sh);
        }
    __shared__ u64 ts[4][kOrdSeqs];
    __shared__ uint32_t os[4][kOrdSeqs];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0)
        for (int q = 0; q < kOrdSeqs; q++) {
            ts[warp][q] = t[q];
            os[warp][q] = o[q];
        }
    __syncthreads();
    if (threadIdx.x < kOrdSeqs) {
        const int q = threadIdx.x;
        const size_t slot = ((size_t)f * nb + b) * kOrdSeqs + q;
        sums[slot] = ts[0][q] + ts[1][q] + ts[2][q] + ts[3][q];
        ors[slot] = os[0][q] | os[1][q] | os[2][q] | os[3][q];
    }
}

__device__ __forceinline__ int binade_of(u64 x) { return 63 - __clzll((long long)x); }

// Grid (frames, 3), one warp: prefix sums over the blocks of one sequence
// and the class of every block, cls[(f * 3 + q) * nb + b].  A single-binade
// block whose terms are all multiples of the binade's ulp is exact.
__global__ void __launch_bounds__(32)
    ordered_classify(const u64 *__restrict__ sums, const uint32_t *__restrict__ ors, int nb,
                     int *__restrict__ cls) {
    const int f = blockIdx.x, q = blockIdx.y, lane = threadIdx.x;
    const int per = (nb + 31) / 32;
    const int b0 = min(lane * per, nb), b1 = min(b0 + per, nb);
    u64 mine = 0;
    for (int b = b0; b < b1; b++) mine += sums[((size_t)f * nb + b) * 3 + q];
    u64 incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const u64 v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    u64 P = incl - mine;  // exclusive prefix of this lane's first block
    for (int b = b0; b < b1; b++) {
        const u64 T = sums[((size_t)f * nb + b) * 3 + q];
        const u64 P1 = P + T;
        int c;
        if (P1 < kTwo53) {
            c = kOrdExact;
        } else if (P >= kTwo53 + kOrdMargin && binade_of(P - kOrdMargin) == binade_of(P1 + kOrdMargin)) {
            c = binade_of(P) - 52;
            // the running sum is a multiple of 2^c here; so are the terms?
            if ((ors[((size_t)f * nb + b) * 3 + q] & ((1u << c) - 1)) == 0) c = kOrdExact;
        } else {
            c = kOrdReplay;
        }
        cls[((size_t)f * kOrdSeqs + q) * nb + b] = c;
        P = P1;
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

// Grid (blocks per frame, frames, 3), one warp: the transfer table of each
// single-binade block.  The block's terms are staged in shared memory with
// one pad word every kOrdLane words, so that lane l reading its run
// [l * kOrdLane, (l + 1) * kOrdLane) hits a different bank than the others.
__global__ void __launch_bounds__(32)
    ordered_tables(const unsigned char *__restrict__ ref, const unsigned char *__restrict__ dist,
                   size_t frame_pitch, size_t stride, int width, uint32_t pixels, int nb,
                   const int *__restrict__ cls, OrdTable *__restrict__ tables) {
    const int b = blockIdx.x, f = blockIdx.y, q = blockIdx.z, lane = threadIdx.x;
    const size_t slot = ((size_t)f * kOrdSeqs + q) * nb + b;
    const int k = cls[slot];
    if (k == kOrdExact || k == kOrdReplay) return;
    __shared__ uint32_t terms[kOrdBlock + kOrdBlock / kOrdLane];
    const uint32_t i0 = (uint32_t)b * kOrdBlock;
    const uint32_t len = min((uint32_t)kOrdBlock, pixels - i0);
    ord_block_pixels(ref, dist, frame_pitch, stride, width, f, i0, len,
                     [&](uint32_t j, uint32_t r, uint32_t d) { terms[j + j / kOrdLane] = ord_term(q, r, d); });
    __syncwarp();
    // this lane's run, for both input parities
    long long e0 = 0, e1 = 0;
    int p0 = 0, p1 = 1;
    const uint32_t j0 = (uint32_t)lane * kOrdLane;
    for (uint32_t j = j0; j < j0 + kOrdLane && j < len; j++) {
        const uint32_t t = terms[j + j / kOrdLane];
        e0 += ord_step(t, k, p0);
        e1 += ord_step(t, k, p1);
    }
    // compose the lanes' functions in lane order
    long long E0 = 0, E1 = 0;
    int P0 = 0, P1 = 1;
    for (int l = 0; l < 32; l++) {
        const long long le0 = __shfl_sync(0xffffffffu, e0, l), le1 = __shfl_sync(0xffffffffu, e1, l);
        const int lp0 = __shfl_sync(0xffffffffu, p0, l), lp1 = __shfl_sync(0xffffffffu, p1, l);
        E0 += P0 ? le1 : le0;
        P0 = P0 ? lp1 : lp0;
        E1 += P1 ? le1 : le0;
        P1 = P1 ? lp1 : lp0;
    }
    if (lane == 0) {
        OrdTable tb;
        tb.e[0] = E0;
        tb.e[1] = E1;
        tb.p[0] = P0;
        tb.p[1] = P1;
        tables[slot] = tb;
    }
}

// Grid (frames, 3), one warp: the walk.  Lane 0 carries the CPU's running
// sum S (an integer below 2^57, exact in a double and in 64 bits) through the
// blocks; block metadata is staged in shared memory a chunk at a time, and a
// replayed block's terms are computed by the warp, then added one by one
// with double-precision round-to-nearest-even adds.  out[f * 3 + q] = S.
__global__ void __launch_bounds__(32)
    ordered_walk(const unsigned char *__restrict__ ref, const unsigned char *__restrict__ dist,
                 size_t frame_pitch, size_t stride, int width, uint32_t pixels, int nb,
                 const u64 *__restrict__ sums, const uint32_t *__restrict__ ors,
                 const int *__restrict__ cls, const OrdTable *__restrict__ tables,
                 u64 *__restrict__ out) {
    const int f = blockIdx.x, q = blockIdx.y, lane = threadIdx.x;
    constexpr int kChunk = 128;
    __shared__ int c_s[kChunk];
    __shared__ u64 t_s[kChunk];
    __shared__ OrdTable tb_s[kChunk];
    __shared__ uint32_t terms[kOrdBlock];
    __shared__ uint32_t o_s[kChunk];
    __shared__ int replay_list[kChunk];
    __shared__ int n_replay;
    __shared__ int do_replay;
    u64 S = 0;
    for (int c0 = 0; c0 < nb; c0 += kChunk) {
        const int n = min(kChunk, nb - c0);
        for (int i = lane; i < n; i += 32) {
            const size_t slot = ((size_t)f * kOrdSeqs + q) * nb + c0 + i;
            c_s[i] = cls[slot];
            t_s[i] = sums[((size_t)f * nb + c0 + i) * 3 + q];
            o_s[i] = ors[((size_t)f * nb + c0 + i) * 3 + q];
            if (c_s[i] != kOrdExact && c_s[i] != kOrdReplay) tb_s[i] = tables[slot];
        }
        __syncwarp();
        if (lane == 0) {
            int m = 0;
            for (int i = 0; i < n; i++)
                if (c_s[i] == kOrdReplay) replay_list[m++] = i;
            n_replay = m;
        }
        __syncwarp();
        // walk the chunk; stop at each replayed block to stage its terms
        int i = 0;
        for (int rix = 0; rix <= n_replay; rix++) {
            const int stop = rix < n_replay ? replay_list[rix] : n;
            if (lane == 0) {
                for (; i < stop; i++) {
                    if (c_s[i] == kOrdExact) {
                        S += t_s[i];
                    } else {
                        const int k = c_s[i];
                        const int p = (int)((S >> k) & 1);
                        S += t_s[i] + (u64)tb_s[i].e[p];
                    }
                }
            }
            // A block near a boundary adds exactly when the running sum and all
            // of its terms are multiples of the largest ulp it can reach.
            if (lane == 0 && rix < n_replay) {
                const u64 top = S + t_s[stop] + kOrdMargin;
                const int kneed = top < kTwo53 ? 0 : binade_of(top) - 52;
                const u64 mask = (1ull << kneed) - 1;
                do_replay = ((S | (u64)o_s[stop]) & mask) != 0;
                if (!do_replay) {
                    S += t_s[stop];
                    i = stop + 1;
                }
            }
            __syncwarp();
            if (rix < n_replay && do_replay) {
                const int b = c0 + stop;
                const uint32_t i0 = (uint32_t)b * kOrdBlock;
                const uint32_t len = min((uint32_t)kOrdBlock, pixels - i0);
                ord_block_pixels(ref, dist, frame_pitch, stride, width, f, i0, len,
                                 [&](uint32_t j, uint32_t r, uint32_t d) { terms[j] = ord_term(q, r, d); });
                __syncwarp();
                if (lane == 0) {
                    double s = (double)S;
                    for (uint32_t j = 0; j < len; j++) s = __dadd_rn(s, (double)terms[j]);
                    S = (u64)s;
                    i = stop + 1;
                }
            }
            __syncwarp();  // do_replay and terms are rewritten next iteration
        }
        __syncwarp();
    }
    if (lane == 0) out[(size_t)f * kOrdSeqs + q] = S;
}

}  // namespace vqx
