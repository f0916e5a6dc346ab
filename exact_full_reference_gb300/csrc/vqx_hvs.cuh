// psnr_hvs plane sum: the CPU's running float sum of a plane's terms,
// reproduced on the device.
//
// "ADR-1397: GPU psnr_hvs twins reproduce the CPU's running float sum bit for
// bit" (Context, Decision): the CPU adds every masked coefficient error of a
// plane, one after another, into one float, so the rounding of each addition
// depends on the sum so far.  The page's twin stores the terms and adds them
// on the host; its Alternatives leave an order-preserving device reduction as
// the open design.  This is one.
//
// - The terms are non-negative, so the running sum s never decreases.  While
//   s stays in one binade b (the floats of biased exponent b; for b = 1 also
//   the subnormals, which share its ulp), s = m u with u = 2^(b - 150), and
//   fl(s + t) = (m + k) u, k being t / u rounded to nearest with a tie going
//   to the even m + k.  The increment depends on s only through the parity of
//   m, so a run of additions is a function of one bit: (K[p], p'[p]) for
//   p = 0, 1, its transfer.  In float bits m u is the word ((b - 1) << 23) + m,
//   so a state is its own bit pattern, its parity is bit 0, and applying K is
//   an integer add to the bits, valid while they stay at or below
//   (b + 1) << 23 (the top of the binade, 2^(b - 126), is reached exactly).
// - A run's transfer for binade b comes from performing its additions (the
//   float add, round to nearest even, subnormals kept) from the representative
//   state m = 2^23 + p (m = p for b = 1), the smallest state of its parity:
//   from any larger state of the same parity that stays in the binade every
//   addition rounds the same way.  A run that leaves the binade from there has
//   no transfer for b.
// - The binade a run starts in is guessed from the sum of the terms before it
//   (the float sum stays within a few per cent of it).  A node keeps
//   transfers for two candidate binades, a leaf for one, or for two where its
//   estimate lies close below a power of two.  Runs are leaves of kHvsLeaf
//   terms (a warp, kHvsLane per lane) and nodes of kHvsLeaves leaves (a CTA).
// - One warp per plane walks: windows of 32 nodes, composed by a warp scan and
//   applied to the state; a node without a transfer for the state's binade, or
//   one that would leave it, is walked leaf by leaf, and such a leaf lane by
//   lane: the lanes' runs for the state's binade are composed, and the lane
//   whose run would leave the binade adds its terms one by one with float adds
//   from the true state.
// Correctness does not depend on the guess: a wrong guess only sends more of
// the walk down to single terms.
//
// The prefix the guess needs comes from a decoupled look-back (Merrill and
// Garland, "Single-pass Parallel Prefix Scan with Decoupled Look-back", 2016)
// across the CTAs of one launch: each CTA takes its node in block order,
// publishes the node's sum, then adds its predecessors' published sums.  Its
// wait is bounded; a CTA that gives up guesses from what it has.  The CTA
// reads its node once, coalesced, into shared memory (summing and checking
// the terms on the way); after the look-back each lane takes its own run
// from there.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "vqx_kernels.cuh"

namespace vqx {

constexpr int kHvsLane = 32;                     // terms per lane
constexpr int kHvsLeaf = 32 * kHvsLane;          // terms per leaf (a warp)
constexpr int kHvsLeaves = 8;                    // leaves per node (warps per CTA)
constexpr int kHvsNode = kHvsLeaf * kHvsLeaves;  // terms per node
constexpr int kHvsThreads = 32 * kHvsLeaves;
// A leaf in shared memory: its 256 vectors of 4 terms, vector q at q + q / 8
// (16 bytes of padding after every 128), so that both the coalesced writes
// and each lane's reads of its own run of 8 vectors are free of bank
// conflicts.
constexpr int kHvsLeafVecs = kHvsLeaf / 4;
constexpr int kHvsLeafSlots = kHvsLeafVecs + kHvsLeafVecs / 8;
constexpr size_t kHvsTablesSmem = (size_t)kHvsLeaves * kHvsLeafSlots * sizeof(float4);
// Windows of 32 node records the walk holds in registers at once (and as
// many loading behind them).
constexpr int kHvsWalkWindows = 2;

// A transfer word is K itself.  The parity after a run needs no bit of its
// own: from a state of parity p the run ends at m + K, whose parity is that
// of p + K.  K <= 2^24 is a transfer; kHvsBad (2^24 + 1) means "none".  The
// sum of two words stays far below 2^32, so min(sum, kHvsBad) keeps "none"
// absorbing under composition, and a state plus kHvsBad always lies above
// the top of the state's binade, so hvs_take never applies it.
constexpr uint32_t kHvsBad = (1u << 24) + 1u;
// Terms must lie in [0, 2^95) (-0 allowed): then no plane of up to 2^31 terms
// can reach 2^127, as the float sum is below twice the exact sum.
constexpr uint32_t kHvsTermLimit = 0x6F000000u;

// Flags of a node record (the walk reports the range flag for the plane).
constexpr uint32_t kHvsFlagRange = 1u;
constexpr uint32_t kHvsFlagTimeout = 2u;  // a bounded wait gave up: no result
constexpr uint32_t kHvsFlagGuess = 4u;  // a look-back gave up (guesses only)

// Look-back status words: the call's epoch in bits 34-63, the state in bits
// 32-33, float bits in the low half.  Nothing clears them between calls: a
// word of another epoch reads as empty.
constexpr u64 kHvsAgg = 1ull << 32;
constexpr u64 kHvsPrefix = 2ull << 32;
constexpr uint32_t kHvsEpochMask = (1u << 30) - 1u;
constexpr long long kHvsLookbackCycles = 20000000ll;  // about 10 ms

struct HvsFn {
    uint32_t k0, k1;  // transfer words for input parity 0 and 1
};

// Two candidate binades b and b + 1 of a run.
struct __align__(16) HvsRec {
    uint4 k;  // (b: k0, k1), (b + 1: k0, k1)
    uint32_t b;
    uint32_t pad[3];
};

struct HvsArgs {
    const float *terms;
    long long n_terms;  // per plane
    long long pitch;    // floats from one plane to the next
    int n_planes;
    int n_leaves, n_nodes;  // per plane
    int vec;                // 16-byte loads (base 16-byte aligned, pitch % 4 == 0)
    int terms_ready;        // the terms were written before the launch ahead started
    uint32_t epoch;         // this call's tag of its status words (1 .. 2^30 - 1)
    HvsRec *leaves;         // [plane][leaf]
    HvsRec *nodes;          // [plane][node]; pad[0] holds the node's flags
    u64 *status;            // [plane][node]
};

// What the walk leaves per plane.
struct HvsOut {
    uint32_t sum_bits;
    uint32_t flags;
    uint32_t replayed_leaves;  // leaves walked lane by lane
    uint32_t replayed_runs;    // lane runs added term by term
};

__device__ __forceinline__ HvsFn hvs_identity() { return {0u, 0u}; }

// "a then b": a.k0 starts from an even state and ends odd iff a.k0 is odd;
// a.k1 starts odd and ends odd iff a.k1 is even.
__device__ __forceinline__ HvsFn hvs_compose(HvsFn a, HvsFn b) {
    const uint32_t n0 = (a.k0 & 1u) ? b.k1 : b.k0;
    const uint32_t n1 = (a.k1 & 1u) ? b.k0 : b.k1;
    return {min(a.k0 + n0, kHvsBad), min(a.k1 + n1, kHvsBad)};
}

// Word of a run that took the representative state s to e, lim being the
// top of the binade: none if e left the binade (or, for terms outside the
// domain, fell below s).
__device__ __forceinline__ uint32_t hvs_word(uint32_t e, uint32_t s, uint32_t lim) {
    return e <= lim ? min(e - s, kHvsBad) : kHvsBad;
}

// Binade of a state (float bits): 1 for zero and the subnormals.
__device__ __forceinline__ uint32_t hvs_binade(uint32_t s) { return max(s >> 23, 1u); }

// Lower candidate binade for a run whose preceding terms add up to about x:
// the binade of x (1 - 1/64), so that a float sum up to 1.6 % below the
// estimate still has a transfer (and, with the next binade as the second
// candidate, one up to twice as far above).
__device__ __forceinline__ uint32_t hvs_guess(float x) {
    return hvs_binade(__float_as_uint(__fmul_rn(x, 0.984375f)));
}

__device__ __forceinline__ bool hvs_bad_term(float t) {
    const uint32_t u = __float_as_uint(t);
    return u >= kHvsTermLimit && u != 0x80000000u;
}

// Representative state of binade b (1 <= b <= 253) for parity 0: the
// smallest even state, 2^23 in the significand (0 for b = 1).
__device__ __forceinline__ uint32_t hvs_rep(uint32_t b) {
    return ((b - 1u) << 23) + (b == 1u ? 0u : (1u << 23));
}

// Transfer of adding t[0..kHvsLane) for binade b, found by adding them from
// the two representative states.
__device__ __forceinline__ HvsFn hvs_run_fn(const float (&t)[kHvsLane], uint32_t b) {
    const uint32_t s0 = hvs_rep(b);
    float x0 = __uint_as_float(s0), x1 = __uint_as_float(s0 + 1u);
#pragma unroll
    for (int i = 0; i < kHvsLane; i++) {
        x0 = __fadd_rn(x0, t[i]);
        x1 = __fadd_rn(x1, t[i]);
    }
    const uint32_t lim = (b + 1u) << 23;
    return {hvs_word(__float_as_uint(x0), s0, lim), hvs_word(__float_as_uint(x1), s0 + 1u, lim)};
}

// The same for a lane's run held in shared memory (its 8 vectors at
// run[0..8) of a padded leaf).
__device__ __forceinline__ HvsFn hvs_run_fn_smem(const float4 *run, uint32_t b) {
    const uint32_t s0 = hvs_rep(b);
    float x0 = __uint_as_float(s0), x1 = __uint_as_float(s0 + 1u);
#pragma unroll
    for (int i = 0; i < kHvsLane / 4; i++) {
        const float4 v = run[i];
        x0 = __fadd_rn(x0, v.x);
        x1 = __fadd_rn(x1, v.x);
        x0 = __fadd_rn(x0, v.y);
        x1 = __fadd_rn(x1, v.y);
        x0 = __fadd_rn(x0, v.z);
        x1 = __fadd_rn(x1, v.z);
        x0 = __fadd_rn(x0, v.w);
        x1 = __fadd_rn(x1, v.w);
    }
    const uint32_t lim = (b + 1u) << 23;
    return {hvs_word(__float_as_uint(x0), s0, lim), hvs_word(__float_as_uint(x1), s0 + 1u, lim)};
}

// Transfers of a lane's run in shared memory for binades b and b + 1.
__device__ __forceinline__ void hvs_run_fns2(const float4 *run, uint32_t b, HvsFn &fb, HvsFn &fb1) {
    const uint32_t s0 = hvs_rep(b);
    const uint32_t u0 = hvs_rep(b + 1u);
    float x0 = __uint_as_float(s0), x1 = __uint_as_float(s0 + 1u);
    float y0 = __uint_as_float(u0), y1 = __uint_as_float(u0 + 1u);
#pragma unroll
    for (int i = 0; i < kHvsLane / 4; i++) {
        const float4 v = run[i];
        const float t[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int c = 0; c < 4; c++) {
            x0 = __fadd_rn(x0, t[c]);
            x1 = __fadd_rn(x1, t[c]);
            y0 = __fadd_rn(y0, t[c]);
            y1 = __fadd_rn(y1, t[c]);
        }
    }
    const uint32_t lim = (b + 1u) << 23, lim1 = (b + 2u) << 23;
    fb = {hvs_word(__float_as_uint(x0), s0, lim), hvs_word(__float_as_uint(x1), s0 + 1u, lim)};
    fb1 = {hvs_word(__float_as_uint(y0), u0, lim1), hvs_word(__float_as_uint(y1), u0 + 1u, lim1)};
}

// Ordered reduction: lane 0 gets lanes 0..kLanes-1 composed in lane order
// (kLanes a power of two; the other lanes' values are not used).
template <int kLanes = 32>
__device__ __forceinline__ HvsFn hvs_reduce(HvsFn f) {
#pragma unroll
    for (int off = 1; off < kLanes; off <<= 1) {
        HvsFn o;
        o.k0 = __shfl_down_sync(0xffffffffu, f.k0, off);
        o.k1 = __shfl_down_sync(0xffffffffu, f.k1, off);
        f = hvs_compose(f, o);
    }
    return f;
}

// Inclusive scan: lane j gets lanes 0..j composed in order.
__device__ __forceinline__ HvsFn hvs_scan(HvsFn f, int lane) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        HvsFn o;
        o.k0 = __shfl_up_sync(0xffffffffu, f.k0, off);
        o.k1 = __shfl_up_sync(0xffffffffu, f.k1, off);
        if (lane >= off) f = hvs_compose(o, f);
    }
    return f;
}

__device__ __forceinline__ HvsFn hvs_select(const HvsRec &r, uint32_t b) {
    if (b == r.b) return {r.k.x, r.k.y};
    if (b == r.b + 1u) return {r.k.z, r.k.w};
    return {kHvsBad, kHvsBad};
}

// Apply the scanned transfers of a window to the state s (uniform across the
// warp): the lanes below `valid` that keep s in its binade form a prefix; s
// moves past them and their count is returned.
__device__ __forceinline__ int hvs_take(HvsFn scanned, int valid, int lane, uint32_t &s) {
    const uint32_t lim = (hvs_binade(s) + 1u) << 23;
    const uint32_t w = (s & 1u) ? scanned.k1 : scanned.k0;
    const bool ok = lane < valid && s + w <= lim;
    const int took = __popc(__ballot_sync(0xffffffffu, ok));
    if (took > 0) s += __shfl_sync(0xffffffffu, w, took - 1);
    return took;
}

// The lane's kHvsLane terms starting at p, with `avail` of them inside the
// plane; the rest read as +0, which adds nothing.  Terms are read through
// L2 (ld.global.cg) everywhere in these kernels, never through the read-only
// data path: the kernels are programmatic dependents of the kernel ahead and
// may start while a kernel that wrote the terms (the caller's, when it lets
// its dependents start early) is still running.
__device__ __forceinline__ void hvs_load(const float *p, long long avail, bool vec,
                                         float (&t)[kHvsLane]) {
    if (vec && avail >= kHvsLane) {
        const float4 *q = reinterpret_cast<const float4 *>(p);
#pragma unroll
        for (int i = 0; i < kHvsLane / 4; i++) {
            const float4 v = __ldcg(q + i);
            t[4 * i] = v.x;
            t[4 * i + 1] = v.y;
            t[4 * i + 2] = v.z;
            t[4 * i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < kHvsLane; i++) t[i] = i < avail ? __ldcg(p + i) : 0.0f;
    }
}

// A status word carries everything it means (state and value in one 64-bit
// word, written and read whole), so relaxed accesses at GPU scope suffice.
__device__ __forceinline__ void st_relaxed_u64(u64 *p, u64 v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ u64 ld_relaxed_u64(const u64 *p) {
    u64 v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

// Sum of the nodes before `node` of one plane (warp-wide; status = the
// plane's status words, tag = the call's epoch in place).  Returns false if
// it gave up waiting.
__device__ __forceinline__ bool hvs_lookback(const u64 *status, int node, int lane, u64 tag,
                                             float &excl) {
    excl = 0.0f;
    int j = node - 1;
    const long long t0 = clock64();
    while (j >= 0) {
        const int idx = j - lane;
        u64 w = 0;
        unsigned pre = 0;
        for (;;) {
            if (idx >= 0 && (w >> 34) != (tag >> 34)) w = ld_relaxed_u64(status + idx);
            const bool mine = idx >= 0 && (w >> 34) == (tag >> 34);
            // needed: every lane up to the nearest published prefix (or all)
            pre = __ballot_sync(0xffffffffu, mine && (w & (3ull << 32)) == kHvsPrefix);
            const unsigned empty = __ballot_sync(0xffffffffu, idx >= 0 && !mine);
            const unsigned need = pre ? ((pre & (0u - pre)) - 1u) : 0xffffffffu;
            if ((empty & need) == 0) break;
            if (clock64() - t0 > kHvsLookbackCycles) return false;
            __nanosleep(32);
        }
        const int stop = pre ? __ffs(pre) - 1 : 32;
        const float v = (idx >= 0 && lane <= stop) ? __uint_as_float((uint32_t)w) : 0.0f;
        excl = __fadd_rn(excl, warp_sum_f(v));
        if (pre) return true;
        j -= 32;
    }
    return true;
}

// One CTA per node: loads the node's terms once, checks them, publishes the
// node's sum, learns the sum before it, and writes the transfers of its
// leaves and of itself for their candidate binades.  Launched as a
// programmatic dependent of the kernel ahead (the previous call's walk): it
// touches only this call's workspace, and reads the terms after that kernel
// has finished unless they were ready before it started.
__global__ void __launch_bounds__(kHvsThreads, 6) hvs_tables(HvsArgs a) {
    allow_dependent_launch();  // the walk may be scheduled now (it waits for this kernel)
    extern __shared__ float4 s_terms[];  // kHvsLeaves leaves, kHvsLeafSlots each
    __shared__ float s_leaf_sum[kHvsLeaves];
    __shared__ float s_excl;
    __shared__ unsigned s_flags;
    __shared__ HvsRec s_leaf[kHvsLeaves];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (!a.terms_ready) grid_dependency_wait();
    // CTAs start in block order, and blocks go round the planes (block t:
    // plane t mod n_planes, node t / n_planes), so that a plane has few nodes
    // in flight at a time and a look-back seldom needs more than one window.
    // (Were the order ever different, only the guesses would suffer.)
    const unsigned g = blockIdx.x;
    const int plane = (int)(g % (unsigned)a.n_planes), node = (int)(g / (unsigned)a.n_planes);
    const u64 tag = (u64)a.epoch << 34;
    const float *pt = a.terms + (size_t)plane * (size_t)a.pitch;
    const long long leaf = (long long)node * kHvsLeaves + warp;
    const float *lb = pt + leaf * kHvsLeaf;
    const long long avail = a.n_terms - leaf * kHvsLeaf;

    // The leaf is read once, coalesced, into shared memory, with its sum (an
    // estimate only, in two packed float pairs) and the largest term bits on
    // the way.  Every term in the domain has bits below kHvsTermLimit except
    // -0; a larger maximum (a term outside the domain, or a -0) sends the
    // lane to the exact check of its terms.
    float4 *sl = s_terms + (size_t)warp * kHvsLeafSlots;
    float ls;
    bool bad = false;
    if (a.vec && avail >= kHvsLeaf) {
        f32x2 acc_a = 0ull, acc_b = 0ull;
        uint32_t mx = 0u;
#pragma unroll
        for (int k = 0; k < kHvsLeafVecs / 32; k++) {
            const int q = lane + 32 * k;
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(lb) + q);
            sl[q + (q >> 3)] = v;
            const uint32_t ux = __float_as_uint(v.x), uy = __float_as_uint(v.y);
            const uint32_t uz = __float_as_uint(v.z), uw = __float_as_uint(v.w);
            acc_a = f2_add(acc_a, f2_pack(ux, uy));
            acc_b = f2_add(acc_b, f2_pack(uz, uw));
            mx = max(mx, max(max(ux, uy), max(uz, uw)));
        }
        uint32_t a0, a1, b0, b1;
        f2_unpack(acc_a, a0, a1);
        f2_unpack(acc_b, b0, b1);
        ls = __fadd_rn(__fadd_rn(__uint_as_float(a0), __uint_as_float(a1)),
                       __fadd_rn(__uint_as_float(b0), __uint_as_float(b1)));
        if (mx >= kHvsTermLimit) {
#pragma unroll 1
            for (int k = 0; k < kHvsLeafVecs / 32; k++) {
                const int q = lane + 32 * k;
                const float4 v = sl[q + (q >> 3)];
                bad |= hvs_bad_term(v.x) | hvs_bad_term(v.y) | hvs_bad_term(v.z) |
                       hvs_bad_term(v.w);
            }
        }
    } else {
        ls = 0.0f;
        float *sf = reinterpret_cast<float *>(sl);
        for (int k = 0; k < kHvsLeaf / 32; k++) {
            const int i = lane + 32 * k;
            const float v = i < avail ? __ldcg(lb + i) : 0.0f;
            const int q = i >> 2;
            sf[4 * (q + (q >> 3)) + (i & 3)] = v;
            ls = __fadd_rn(ls, v);
            bad |= hvs_bad_term(v);
        }
    }
    ls = warp_sum_f(ls);
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) s_leaf_sum[warp] = ls;
    if (threadIdx.x == 0) s_flags = 0u;
    __syncthreads();
    if (bad && lane == 0) atomicOr(&s_flags, kHvsFlagRange);

    if (warp == 0) {
        const float node_sum = warp_sum_f(lane < kHvsLeaves ? s_leaf_sum[lane] : 0.0f);
        u64 *st = a.status + (size_t)plane * (size_t)a.n_nodes;
        float excl = 0.0f;
        if (node == 0) {
            if (lane == 0) st_relaxed_u64(st, tag | kHvsPrefix | __float_as_uint(node_sum));
        } else {
            if (lane == 0) st_relaxed_u64(st + node, tag | kHvsAgg | __float_as_uint(node_sum));
            const bool ok = hvs_lookback(st, node, lane, tag, excl);
            if (lane == 0) {
                if (!ok) atomicOr(&s_flags, kHvsFlagGuess);
                st_relaxed_u64(st + node,
                               tag | kHvsPrefix | __float_as_uint(__fadd_rn(excl, node_sum)));
            }
        }
        if (lane == 0) s_excl = excl;
    }
    __syncthreads();

    // Second pass: each lane's run of kHvsLane terms, for the binade of this
    // leaf's estimate and, where the estimate lies within 1/16 of the top of
    // that binade, for the next one as well (a float sum running that far
    // ahead of its estimate is only walked more slowly, never wrongly).
    float lp = s_excl;
    for (int j = 0; j < warp; j++) lp = __fadd_rn(lp, s_leaf_sum[j]);
    const uint32_t bl = hvs_guess(lp);
    const bool two = hvs_binade(__float_as_uint(__fmul_rn(lp, 1.0625f))) != bl;  // warp-uniform
    const float4 *run = sl + 9 * lane;  // vectors 8 lane .. 8 lane + 7
    HvsFn f0, f1;
    if (two) {
        hvs_run_fns2(run, bl, f0, f1);
        f0 = hvs_reduce(f0);
        f1 = hvs_reduce(f1);
    } else {
        f0 = hvs_reduce(hvs_run_fn_smem(run, bl));
        f1 = {kHvsBad, kHvsBad};
    }
    if (lane == 0) {
        HvsRec r;
        r.k = make_uint4(f0.k0, f0.k1, f1.k0, f1.k1);
        r.b = bl;
        r.pad[0] = r.pad[1] = r.pad[2] = 0;
        s_leaf[warp] = r;
        if (leaf < a.n_leaves) a.leaves[(size_t)plane * (size_t)a.n_leaves + (size_t)leaf] = r;
    }
    __syncthreads();

    if (warp == 0) {
        const uint32_t bn = hvs_guess(s_excl);
        const long long nl = (long long)a.n_leaves - (long long)node * kHvsLeaves;
        const bool in = lane < kHvsLeaves && lane < nl;
        const HvsFn g0 = hvs_reduce<kHvsLeaves>(in ? hvs_select(s_leaf[lane & (kHvsLeaves - 1)], bn)
                                                   : hvs_identity());
        const HvsFn g1 = hvs_reduce<kHvsLeaves>(
            in ? hvs_select(s_leaf[lane & (kHvsLeaves - 1)], bn + 1u) : hvs_identity());
        if (lane == 0) {
            HvsRec r;
            r.k = make_uint4(g0.k0, g0.k1, g1.k0, g1.k1);
            r.b = bn;
            r.pad[0] = s_flags;
            r.pad[1] = r.pad[2] = 0;
            a.nodes[(size_t)plane * (size_t)a.n_nodes + (size_t)node] = r;
        }
    }
}

// ---------------------------------------------------------------- persistent form
// hvs_tables_tma: the same tables for planes whose terms are 16-byte aligned
// with a pitch of whole vectors (at least 32 terms), as a persistent
// pipeline.  CTA c takes nodes g = c, c + gridDim.x, ... (g in the launch
// order of hvs_tables: plane g mod n_planes, node g / n_planes).
// - A producer lane streams each node (256 rows of 32 terms, one box of a
//   tensor map over full rows, zero-filled past a plane's last full row)
//   into a ring of kHvsTmaStages shared-memory buffers, 128-byte swizzled:
//   chunk c (16 bytes) of row r lies at chunk c ^ (r mod 8), so a lane
//   reading its own row (its run) and eight lanes reading eight rows hit
//   eight different bank groups.
// - Summer warp w sums leaf w (rows 32 w .. 32 w + 31) of every node as soon
//   as it lands (any order) and checks its terms; the last of the eight adds
//   the leaf sums and publishes the node's sum at once (its status word).
// - kHvsTmaLookback look-back warps take nodes in turn, once a node is
//   summed: the look-back of hvs_tables gives its prefix estimate, and its
//   inclusive prefix is published.
// - Table warp w of set j (two sets of eight, taking even and odd nodes, so
//   that each warp's chain of dependent additions and shuffles has two
//   nodes' time) then tabulates each lane's run of leaf w in order and
//   writes the leaf's record.
// - Once its eight warps are past a named barrier, warp 0 of the set
//   releases the buffer (keeping the node's flags and estimate) and then
//   composes the node's record from the leaf records.
// The summers run up to kHvsTmaStages nodes ahead of the table warps, so the
// look-back's latency hides behind the ring instead of stalling it.
// Terms of a plane's last, partial row (fewer than 32) are not in any box:
// the lane whose run they are reads them itself.
// Stage k of a CTA uses buffer k mod kHvsTmaStages; each of its mbarriers
// (full: bytes landed; sums: the eight leaf sums written; excl: the prefix
// estimate written; empty: the buffer read, the record's inputs kept) completes
// one phase per use, parity (k / kHvsTmaStages) & 1.  Every wait is
// bounded; a warp whose wait gives up waits for nothing more, and every node
// record written after it carries kHvsFlagTimeout.  Seven stages of 32 KB
// and the control block fill the 227 KB a CTA may have, so the ring must
// start at the window's first byte: a CTA that finds its shared memory
// elsewhere (not 1024-byte aligned) marks its nodes' records with
// kHvsFlagTimeout and does nothing else.
constexpr int kHvsTmaStages = 7;
constexpr int kHvsTmaLookback = 2;
constexpr int kHvsTmaTableSets = 2;                           // table warps 0 .. 15
constexpr int kHvsTmaSummer0 = kHvsTmaTableSets * kHvsLeaves;  // summers 16 .. 23
constexpr int kHvsTmaSummers = kHvsLeaves;                     // one leaf each
constexpr int kHvsTmaProducer = kHvsTmaSummer0 + kHvsTmaSummers;
constexpr int kHvsTmaThreads = (kHvsTmaProducer + 1 + kHvsTmaLookback) * 32;
static_assert(kHvsTmaLookback <= kHvsTmaStages, "a look-back warp's previous node bounds its wait");
constexpr uint32_t kHvsNodeBytes = kHvsNode * 4;
constexpr int kHvsNodeRows = kHvsNode / 32;

// The kernel's shared memory, all of it dynamic: the ring (1024-byte aligned
// for the 128-byte swizzle, at the start of the CTA's window), then this
// control block.  Per stage: its mbarriers and what its node's roles pass
// on; the leaf records per table set, in two slots used by the set's nodes
// in turn.
struct HvsTmaShared {
    u64 full[kHvsTmaStages], empty[kHvsTmaStages], sums[kHvsTmaStages], exclb[kHvsTmaStages];
    float leaf_sum[kHvsTmaStages][kHvsLeaves];
    float excl[kHvsTmaStages];
    unsigned flags[kHvsTmaStages], summed[kHvsTmaStages];
    float node_sum[kHvsTmaStages];
    unsigned err;
    HvsRec leaf[kHvsTmaTableSets][2][kHvsLeaves];
};
constexpr size_t kHvsTmaRing = (size_t)kHvsTmaStages * kHvsNodeBytes;
constexpr size_t kHvsTmaSmem = kHvsTmaRing + sizeof(HvsTmaShared);

struct HvsTmaArgs {
    long long rows_full;  // full rows of 32 terms per plane
    int tail;             // terms in the partial row (0 .. 31)
};

// bar.sync on named barrier id (1 .. 15) for `threads` threads (whole warps).
__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// The nodes a CTA takes, g = blockIdx.x + k gridDim.x for k = k0, k0 + s, ...,
// as (plane g mod n_planes, node g / n_planes), stepped without a division
// per node (g < 2^31: the host bounds n_planes times the node count).
struct HvsNodeIter {
    int plane, node, dplane, dnode, n_planes;
    __device__ __forceinline__ HvsNodeIter(int k0, int s, int n_planes_) : n_planes(n_planes_) {
        const unsigned P = (unsigned)n_planes_;
        const unsigned g = blockIdx.x + (unsigned)k0 * gridDim.x, step = (unsigned)s * gridDim.x;
        plane = (int)(g % P);
        node = (int)(g / P);
        dplane = (int)(step % P);
        dnode = (int)(step / P);
    }
    __device__ __forceinline__ void next() {
        plane += dplane;
        node += dnode;
        if (plane >= n_planes) {
            plane -= n_planes;
            node++;
        }
    }
};

// A wait that sleeps: try_wait with a suspend-time hint lets the thread be
// suspended until the phase completes (or the hint runs out) instead of
// polling, so the warps that wait (for data, for a prefix, for a free
// buffer) leave the issue slots to the warps that compute.  Bounded like
// mbar_wait: false after `limit` SM clock cycles.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity,
                                                long long limit = kWaitCycles) {
    const long long t0 = clock64();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "r"(1000000u)
            : "memory");
        if (ok) return true;
        if (clock64() - t0 > limit) return false;
    }
}

__global__ void __launch_bounds__(kHvsTmaThreads, 1)
    hvs_tables_tma(const __grid_constant__ CUtensorMap tm, HvsArgs a, HvsTmaArgs t) {
    allow_dependent_launch();  // the walk may be scheduled now (it waits for this kernel)
    constexpr int S = kHvsTmaStages;
    extern __shared__ __align__(1024) unsigned char hvs_raw[];
    unsigned char *ring = hvs_raw;
    HvsTmaShared *ctl = reinterpret_cast<HvsTmaShared *>(hvs_raw + kHvsTmaRing);
    float(*const s_leaf_sum)[kHvsLeaves] = ctl->leaf_sum;
    float *const s_excl = ctl->excl;
    unsigned *const s_flags = ctl->flags;
    unsigned *const s_summed = ctl->summed;
    float *const s_node_sum = ctl->node_sum;
    unsigned &s_err = ctl->err;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring0 = smem_u32(hvs_raw);
    const uint32_t full0 = smem_u32(ctl->full), empty0 = smem_u32(ctl->empty);
    const uint32_t sums0 = smem_u32(ctl->sums), excl0 = smem_u32(ctl->exclb);

    const long long total = (long long)a.n_planes * a.n_nodes;
    const int nk = total > (long long)blockIdx.x
                       ? (int)((total - 1 - (long long)blockIdx.x) / gridDim.x + 1)
                       : 0;
    const u64 tag = (u64)a.epoch << 34;
    if (ring0 & 1023u) {
        // no room to align the ring: this CTA's nodes are reported, not summed
        HvsNodeIter it(0, 1, a.n_planes);
        for (int k = 0; k < nk; k++, it.next())
            if (threadIdx.x == 0) {
                HvsRec r;
                r.k = make_uint4(kHvsBad, kHvsBad, kHvsBad, kHvsBad);
                r.b = 1u;
                r.pad[0] = kHvsFlagTimeout;
                r.pad[1] = r.pad[2] = 0;
                a.nodes[(size_t)it.plane * (size_t)a.n_nodes + (size_t)it.node] = r;
            }
        return;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; i++) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
            mbar_init(sums0 + 8 * i, kHvsTmaSummers);
            mbar_init(excl0 + 8 * i, 1);
            s_flags[i] = 0u;
            s_summed[i] = 0u;
        }
        s_err = 0u;
        mbar_fence_init();
    }
    __syncthreads();

    if (warp == kHvsTmaProducer) {
        if (lane != 0) return;
        if (!a.terms_ready) grid_dependency_wait();
        int k = 0;
        HvsNodeIter it(0, 1, a.n_planes);
        for (; k < nk; k++, it.next()) {
            const int st = k % S;
            if (k >= S && !mbar_wait_sleep(empty0 + 8 * st, ((k / S) - 1) & 1)) {
                s_err = 1u;
                break;
            }
            mbar_arrive_expect_tx(full0 + 8 * st, kHvsNodeBytes);
            tensor_g2s_3d(ring0 + (uint32_t)st * kHvsNodeBytes, &tm, 0, it.node * kHvsNodeRows,
                          it.plane, full0 + 8 * st);
        }
        // the copies in flight land before the CTA (and its shared memory) ends
        for (int q = k > S ? k - S : 0; q < k; q++) mbar_wait_sleep(full0 + 8 * (q % S), (q / S) & 1);
        return;
    }

    if (warp > kHvsTmaProducer) {
        bool err = false;
        const int k0 = warp - kHvsTmaProducer - 1;
        HvsNodeIter it(k0, kHvsTmaLookback, a.n_planes);
        for (int k = k0; k < nk; k += kHvsTmaLookback, it.next()) {
            const int st = k % S;
            const uint32_t par = (k / S) & 1;
            if (!err && !__all_sync(0xffffffffu, mbar_wait_sleep(sums0 + 8 * st, par))) {
                err = true;
                if (lane == 0) s_err = 1u;
            }
            const int plane = it.plane, node = it.node;
            float excl = 0.0f;
            if (!err && node > 0) {
                // the node's own sum was published by the summers already
                u64 *stw = a.status + (size_t)plane * (size_t)a.n_nodes;
                const bool ok = hvs_lookback(stw, node, lane, tag, excl);
                if (lane == 0) {
                    if (!ok) atomicOr(&s_flags[st], kHvsFlagGuess);
                    st_relaxed_u64(stw + node,
                                   tag | kHvsPrefix | __float_as_uint(__fadd_rn(excl, s_node_sum[st])));
                }
            }
            if (lane == 0) {
                s_excl[st] = excl;
                mbar_arrive(excl0 + 8 * st);
            }
        }
        return;
    }

    // table warps (0 ..): leaf lw = warp mod 8 of set warp / 8; summers
    // (kHvsTmaSummer0 ..): leaf lw
    const bool summer = warp >= kHvsTmaSummer0;
    const int lw = summer ? warp - kHvsTmaSummer0 : warp % kHvsLeaves;
    bool err = false;
    const float *const planes = a.terms;
    auto pass1 = [&](int k, int plane, int node) {
        const int st = k % S;
        if (!err && !__all_sync(0xffffffffu, mbar_wait_sleep(full0 + 8 * st, (k / S) & 1))) {
            err = true;
            if (lane == 0) s_err = 1u;
        }
        bool bad = false;
        {
            const int leafw = lw;
            float ls = 0.0f;
            if (!err) {
                const float4 *lf = reinterpret_cast<const float4 *>(
                    ring + (size_t)st * kHvsNodeBytes + (size_t)leafw * kHvsLeaf * 4);
                f32x2 acc_a = 0ull, acc_b = 0ull;
                uint32_t mx = 0u;
#pragma unroll
                for (int i = 0; i < kHvsLeafVecs / 32; i++) {
                    const float4 v = lf[lane + 32 * i];
                    const uint32_t ux = __float_as_uint(v.x), uy = __float_as_uint(v.y);
                    const uint32_t uz = __float_as_uint(v.z), uw = __float_as_uint(v.w);
                    acc_a = f2_add(acc_a, f2_pack(ux, uy));
                    acc_b = f2_add(acc_b, f2_pack(uz, uw));
                    mx = __vimax3_u32(mx, ux, uy);
                    mx = __vimax3_u32(mx, uz, uw);
                }
                uint32_t a0, a1, b0, b1;
                f2_unpack(acc_a, a0, a1);
                f2_unpack(acc_b, b0, b1);
                ls = __fadd_rn(__fadd_rn(__uint_as_float(a0), __uint_as_float(a1)),
                               __fadd_rn(__uint_as_float(b0), __uint_as_float(b1)));
                if (mx >= kHvsTermLimit) {
#pragma unroll 1
                    for (int i = 0; i < kHvsLeafVecs / 32; i++) {
                        const float4 v = lf[lane + 32 * i];
                        bad |= hvs_bad_term(v.x) | hvs_bad_term(v.y) | hvs_bad_term(v.z) |
                               hvs_bad_term(v.w);
                    }
                }
                // the partial row, if it is one of this leaf's rows
                const long long row0 = (long long)node * kHvsNodeRows + (long long)leafw * 32;
                if (t.tail && t.rows_full >= row0 && t.rows_full < row0 + 32 && lane < t.tail) {
                    const float v = __ldcg(planes + (size_t)plane * (size_t)a.pitch +
                                          (size_t)t.rows_full * 32 + lane);
                    ls = __fadd_rn(ls, v);
                    bad |= hvs_bad_term(v);
                }
            }
            ls = warp_sum_f(ls);
            if (lane == 0) s_leaf_sum[st][leafw] = ls;
        }
        bad = __any_sync(0xffffffffu, bad);
        unsigned last = 0u;
        if (lane == 0) {
            if (bad) atomicOr(&s_flags[st], kHvsFlagRange);
            __threadfence_block();
            last = atomicAdd(&s_summed[st], 1u) == kHvsTmaSummers - 1 ? 1u : 0u;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            // the last warp: node sum, published as this node's aggregate
            // (the inclusive prefix for a plane's first node)
            __threadfence_block();
            float node_sum = s_leaf_sum[st][lane & (kHvsLeaves - 1)];
#pragma unroll
            for (int off = kHvsLeaves / 2; off > 0; off >>= 1)
                node_sum = __fadd_rn(node_sum, __shfl_xor_sync(0xffffffffu, node_sum, off));
            if (lane == 0) {
                s_node_sum[st] = node_sum;
                s_summed[st] = 0u;
                if (!err) {
                    u64 *stw = a.status + (size_t)plane * (size_t)a.n_nodes + node;
                    st_relaxed_u64(stw, tag | (node == 0 ? kHvsPrefix : kHvsAgg) |
                                            __float_as_uint(node_sum));
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(sums0 + 8 * st);
    };

    auto pass2 = [&](int k, int plane, int node) {
        const int st = k % S;
        if (!err && !__all_sync(0xffffffffu, mbar_wait_sleep(full0 + 8 * st, (k / S) & 1) &&
                                                 mbar_wait_sleep(excl0 + 8 * st, (k / S) & 1))) {
            err = true;
            if (lane == 0) s_err = 1u;
        }
        const long long leaf = (long long)node * kHvsLeaves + lw;
        HvsFn f0 = {kHvsBad, kHvsBad}, f1 = {kHvsBad, kHvsBad};
        uint32_t bl = 1u;
        if (!err) {
            float lp = s_excl[st];
            for (int j = 0; j < lw; j++) lp = __fadd_rn(lp, s_leaf_sum[st][j]);
            bl = hvs_guess(lp);
            const bool two = hvs_binade(__float_as_uint(__fmul_rn(lp, 1.0625f))) != bl;
            const long long row = (long long)node * kHvsNodeRows + (long long)lw * 32 + lane;
            float tv[kHvsLane];
            if (row == t.rows_full && t.tail) {
                // the partial row: its terms from the plane, zeros past its end
                const float *src = planes + (size_t)plane * (size_t)a.pitch + (size_t)row * 32;
#pragma unroll
                for (int i = 0; i < kHvsLane; i++) tv[i] = i < t.tail ? __ldcg(src + i) : 0.0f;
            } else {
                const float4 *rw = reinterpret_cast<const float4 *>(
                    ring + (size_t)st * kHvsNodeBytes + (size_t)(lw * 32 + lane) * 128);
                const int sw = lane & 7;
#pragma unroll
                for (int c = 0; c < kHvsLane / 4; c++) {
                    const float4 v = rw[c ^ sw];
                    tv[4 * c] = v.x;
                    tv[4 * c + 1] = v.y;
                    tv[4 * c + 2] = v.z;
                    tv[4 * c + 3] = v.w;
                }
            }
            if (two) {
                f0 = hvs_reduce(hvs_run_fn(tv, bl));
                f1 = hvs_reduce(hvs_run_fn(tv, bl + 1u));
            } else {
                f0 = hvs_reduce(hvs_run_fn(tv, bl));
            }
        }
        HvsRec *const set_leaf = ctl->leaf[warp / kHvsLeaves][(k >> 1) & 1];
        if (lane == 0) {
            HvsRec r;
            r.k = make_uint4(f0.k0, f0.k1, f1.k0, f1.k1);
            r.b = bl;
            r.pad[0] = r.pad[1] = r.pad[2] = 0;
            set_leaf[lw] = r;
            if (leaf < a.n_leaves) a.leaves[(size_t)plane * (size_t)a.n_leaves + (size_t)leaf] = r;
            if (err) s_err = 1u;
        }
        // the set's eight warps meet (their reads of the buffer are done);
        // its warp 0 frees the buffer, keeping what the node's record needs
        // (the flags, which the next use of the stage sets afresh, and the
        // prefix estimate), then composes the record from the leaf records
        // (their slot is rewritten only by this set's node after next, which
        // its warps reach past the next named barrier, after warp 0 is back)
        named_barrier(1 + warp / kHvsLeaves, 32 * kHvsLeaves);
        if (lw == 0) {
            const float ex = s_excl[st];
            const HvsRec lr = set_leaf[lane & (kHvsLeaves - 1)];
            uint32_t fl = 0u;
            if (lane == 0) {
                fl = s_flags[st] | ((err || s_err) ? kHvsFlagTimeout : 0u);
                s_flags[st] = 0u;
                mbar_arrive(empty0 + 8 * st);
            }
            const uint32_t bn = hvs_guess(ex);
            const long long nl = (long long)a.n_leaves - (long long)node * kHvsLeaves;
            const bool in = lane < kHvsLeaves && lane < nl;
            const HvsFn g0 = hvs_reduce<kHvsLeaves>(in ? hvs_select(lr, bn) : hvs_identity());
            const HvsFn g1 = hvs_reduce<kHvsLeaves>(in ? hvs_select(lr, bn + 1u) : hvs_identity());
            if (lane == 0) {
                HvsRec r;
                r.k = make_uint4(g0.k0, g0.k1, g1.k0, g1.k1);
                r.b = bn;
                r.pad[0] = fl;
                r.pad[1] = r.pad[2] = 0;
                a.nodes[(size_t)plane * (size_t)a.n_nodes + (size_t)node] = r;
            }
        }
    };

    if (summer) {
        HvsNodeIter it(0, 1, a.n_planes);
        for (int k = 0; k < nk; k++, it.next()) pass1(k, it.plane, it.node);
    } else {
        const int set = warp / kHvsLeaves;
        HvsNodeIter it(set, kHvsTmaTableSets, a.n_planes);
        for (int k = set; k < nk; k += kHvsTmaTableSets, it.next()) pass2(k, it.plane, it.node);
    }
}

// A record as the walk keeps it: its four transfer words, and its binade
// and flags in one word (binade in the low 16 bits).  Records are read
// through L2: the walk is launched as a programmatic dependent, before the
// tables kernel that writes them has ended, and the read-only data path
// needs data unchanged for the reading kernel's whole run (read through it,
// the walk saw records of an earlier call in about one test in twelve).
struct HvsWalkRec {
    uint4 k;
    uint32_t bf;
};

__device__ __forceinline__ HvsWalkRec hvs_walk_rec(const HvsRec *p, bool in) {
    HvsWalkRec r;
    if (in) {
        r.k = __ldcg(reinterpret_cast<const uint4 *>(p));
        const uint2 w = __ldcg(reinterpret_cast<const uint2 *>(&p->b));
        r.bf = w.x | (w.y << 16);
    } else {
        r.k = make_uint4(kHvsBad, kHvsBad, kHvsBad, kHvsBad);
        r.bf = 0u;
    }
    return r;
}

__device__ __forceinline__ HvsFn hvs_select_w(const HvsWalkRec &r, uint32_t b) {
    const uint32_t rb = r.bf & 0xffffu;
    if (b == rb) return {r.k.x, r.k.y};
    if (b == rb + 1u) return {r.k.z, r.k.w};
    return {kHvsBad, kHvsBad};
}

// One leaf, lane by lane, from state s.
__device__ __forceinline__ void hvs_walk_leaf(const HvsArgs &a, const float *pt, long long leaf,
                                              int lane, uint32_t &s, uint32_t &runs) {
    const long long first = leaf * kHvsLeaf + (long long)lane * kHvsLane;
    float t[kHvsLane];
    hvs_load(pt + first, a.n_terms - first, a.vec != 0, t);
    int start = 0;
    while (start < 32) {
        const HvsFn f = lane >= start ? hvs_run_fn(t, hvs_binade(s)) : hvs_identity();
        const int took = hvs_take(hvs_scan(f, lane), 32, lane, s);
        if (took >= 32) break;
        // lane `took` leaves the binade: its terms one by one, as the CPU adds them
        uint32_t ns = s;
        if (lane == took) {
            float x = __uint_as_float(s);
#pragma unroll
            for (int i = 0; i < kHvsLane; i++) x = __fadd_rn(x, t[i]);
            ns = __float_as_uint(x);
        }
        s = __shfl_sync(0xffffffffu, ns, took);
        runs++;
        start = took + 1;
    }
}

// The terms of node `node` of a plane into L2 (the warp's lanes share the
// lines; none past the plane's terms).
__device__ __forceinline__ void hvs_prefetch_terms(const HvsArgs &a, const float *pt, int node, int lane) {
    const long long t0 = (long long)node * kHvsNode;
#pragma unroll
    for (int i = 0; i < kHvsNode / 32 / 32; i++) {
        const long long t = t0 + ((long long)i * 32 + lane) * 32;
        if (t < a.n_terms) asm volatile("prefetch.global.L2 [%0];" ::"l"(pt + t));
    }
}

// Node `node` of a plane, leaf by leaf (its leaf records read once), and a
// leaf whose run leaves the state's binade lane by lane.
__device__ __forceinline__ void hvs_walk_node(const HvsArgs &a, const float *pt, const HvsRec *leaves,
                                              int node, int lane, uint32_t &s, HvsOut &o) {
    const long long l0 = (long long)node * kHvsLeaves;
    const int nl = (int)min((long long)kHvsLeaves, (long long)a.n_leaves - l0);
    const HvsWalkRec lr = hvs_walk_rec(leaves + l0 + lane, lane < nl);
    hvs_prefetch_terms(a, pt, node, lane);  // for the leaf walked lane by lane, if any
    int lf = 0;
    while (lf < nl) {
        const uint32_t b = hvs_binade(s);
        const HvsFn g = lane >= lf && lane < nl ? hvs_select_w(lr, b) : hvs_identity();
        lf = hvs_take(hvs_scan(g, lane), nl, lane, s);
        if (lf < nl) {
            hvs_walk_leaf(a, pt, l0 + lf, lane, s, o.replayed_runs);
            o.replayed_leaves++;
            lf++;
        }
    }
}

// One warp per plane: the walk over nodes, leaves and terms.  Writes the
// plane's result (into host-mapped memory).  A node whose terms were not all
// in [0, 2^95) ends the plane's walk before any of its terms are used: the
// plane's sum is NaN and its flags say why.
// The node records go through registers in blocks of kHvsWalkWindows
// windows of 32, the next block loading while this one is walked.  A window
// is scanned from the first node not yet taken (the nodes before it count as
// the identity), so a node walked leaf by leaf costs no reload of its
// window; such a node's terms are prefetched into L2 as soon as it is met.
// At most 80 registers a thread (the launch bound): a warp's registers come
// from one of the SM's four sub-partitions, and beside a CTA of the next
// call's hvs_tables_tma (27 warps of 72 registers) the least loaded one has
// 2,560 left.  A walk that needs more waits for SMs the tables kernel holds,
// and the tables CTAs it displaces start late (measured: pipelined steps
// 244 -> 287 us at 98 registers).
__global__ void __launch_bounds__(32, 24) hvs_walk(HvsArgs a, HvsOut *out) {
    allow_dependent_launch();  // the next call's tables may start on free SMs
    grid_dependency_wait();    // this call's tables are complete
    constexpr int W = kHvsWalkWindows;
    const int plane = blockIdx.x, lane = threadIdx.x;
    HvsOut o;
    o.flags = 0;
    o.replayed_leaves = 0;
    o.replayed_runs = 0;
    const float *pt = a.terms + (size_t)plane * (size_t)a.pitch;
    const HvsRec *nodes = a.nodes + (size_t)plane * (size_t)a.n_nodes;
    const HvsRec *leaves = a.leaves + (size_t)plane * (size_t)a.n_leaves;
    uint32_t s = 0u;  // the running sum, as float bits
    bool stop = false;
    HvsWalkRec cur[W], nxt[W];
#pragma unroll
    for (int j = 0; j < W; j++) {
        const int i = 32 * j + lane, i2 = 32 * (W + j) + lane;
        cur[j] = hvs_walk_rec(nodes + i, i < a.n_nodes);
        nxt[j] = hvs_walk_rec(nodes + i2, i2 < a.n_nodes);
    }
    for (int base = 0; base < a.n_nodes && !stop; base += 32 * W) {
#pragma unroll
        for (int j = 0; j < W; j++) {
            const int ws = base + 32 * j;
            if (stop || ws >= a.n_nodes) break;
            const int cnt = min(32, a.n_nodes - ws);
            const uint32_t fl = __reduce_or_sync(0xffffffffu, lane < cnt ? cur[j].bf >> 16 : 0u);
            o.flags |= fl & kHvsFlagGuess;
            if (fl & (kHvsFlagRange | kHvsFlagTimeout)) {
                o.flags |= fl & (kHvsFlagRange | kHvsFlagTimeout);
                stop = true;
                break;
            }
            int off = 0;
            while (off < cnt) {
                const uint32_t b = hvs_binade(s);
                const HvsFn f = lane >= off && lane < cnt ? hvs_select_w(cur[j], b) : hvs_identity();
                const int took = hvs_take(hvs_scan(f, lane), cnt, lane, s);
                if (took >= cnt) break;
                hvs_walk_node(a, pt, leaves, ws + took, lane, s, o);
                off = took + 1;
            }
        }
#pragma unroll
        for (int j = 0; j < W; j++) {
            const int i = base + 32 * (2 * W + j) + lane;
            cur[j] = nxt[j];
            nxt[j] = hvs_walk_rec(nodes + i, i < a.n_nodes);
        }
    }
    if (lane == 0) {
        o.sum_bits = (o.flags & (kHvsFlagRange | kHvsFlagTimeout)) ? 0x7FC00000u : s;
        out[plane] = o;
    }
}

}  // namespace vqx
