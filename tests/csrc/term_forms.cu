// GPU test library (not part of the product): runs the library's per-thread
// accumulators (vqx::TermSums<BPC> and vqx::TermSums16Sse from
// vqx_kernels.cuh) against the literal per-pixel form of the terms on the
// same device, so that every (reference, distorted) sample pair of a bit
// depth can be checked.
//
// The literal form is the arithmetic the pages describe, written out with
// conversion instructions: each sample converted to fp32, the difference and
// the squares taken as single round-to-nearest-even operations, the integer-
// valued results converted back and added in 64 bits ("ADR-1440: float_psnr_hip
// adds its squared differences as integers ...", Decision; "ADR-1447:
// float_moment_hip adds the float squares the CPU adds ...", Decision).
#include <cuda_runtime.h>

#include <cstdint>

#include "vqx_kernels.cuh"

using vqx::u64;

namespace {

// Record words (vqx::Partial): 0..4 the five sums, 5 the OR of the samples,
// 6 the exact SSE minus word 0 (modulo 2^64), 7 zero.
constexpr int kW = vqx::kWords;

struct LiteralSums {
    u64 t[kW] = {0, 0, 0, 0, 0, 0, 0, 0};
    __device__ void sample(uint32_t r, uint32_t d) {
        const float fr = __uint2float_rn(r), fd = __uint2float_rn(d);
        const float diff = __fsub_rn(fr, fd);
        const u64 q = __float2uint_rn(__fmul_rn(diff, diff));
        t[0] += q;
        t[1] += r;
        t[2] += d;
        t[3] += __float2uint_rn(__fmul_rn(fr, fr));
        t[4] += __float2uint_rn(__fmul_rn(fd, fd));
        t[5] |= r | d;
        const long long e = (long long)r - (long long)d;
        t[6] += (u64)(e * e) - q;  // the integer square, minus the float one
    }
};

template <int BPC>
__device__ uint32_t pack_word(uint32_t s0, uint32_t s1, uint32_t s2, uint32_t s3) {
    if constexpr (BPC == 8) return s0 | (s1 << 8) | (s2 << 16) | (s3 << 24);
    return s0 | (s1 << 16);
}

// Thread i takes the reference value r = i (i < 2^bpc) against every
// distorted value d in [0, 2^bpc), fed through vec() in 16-byte groups (and,
// with use_samples, through sample() instead), flushing every kFlushVecs
// calls.  fast[8 i + k] and lit[8 i + k] receive the two sets of totals.
template <int BPC, class Acc>
__global__ void exhaustive(u64 *fast, u64 *lit, int use_samples) {
    const uint32_t top = 1u << BPC;
    const uint32_t r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= top) return;
    constexpr uint32_t per_vec = BPC == 8 ? 16 : 8;
    Acc acc;
    LiteralSums ref;
    uint32_t calls = 0;
    for (uint32_t d0 = 0; d0 < top; d0 += per_vec) {
        if (use_samples) {
            for (uint32_t k = 0; k < per_vec; k++) {
                acc.sample(r, d0 + k);
                if (++calls == Acc::kFlushVecs) { acc.flush(); calls = 0; }
            }
        } else {
            uint32_t a[4], b[4];
            for (int w = 0; w < 4; w++) {
                const uint32_t base = d0 + w * (per_vec / 4);
                if constexpr (BPC == 8) {
                    a[w] = pack_word<8>(r, r, r, r);
                    b[w] = pack_word<8>(base, base + 1, base + 2, base + 3);
                } else {
                    a[w] = pack_word<BPC>(r, r, 0, 0);
                    b[w] = pack_word<BPC>(base, base + 1, 0, 0);
                }
            }
            acc.vec(make_uint4(a[0], a[1], a[2], a[3]), make_uint4(b[0], b[1], b[2], b[3]));
            if (++calls == Acc::kFlushVecs) { acc.flush(); calls = 0; }
        }
        for (uint32_t k = 0; k < per_vec; k++) ref.sample(r, d0 + k);
    }
    u64 t[kW];
    acc.totals(t);
    for (int k = 0; k < kW; k++) {
        fast[kW * (size_t)r + k] = t[k];
        lit[kW * (size_t)r + k] = ref.t[k];
    }
}

// Thread i folds n_vec 16-byte vector pairs of a stream (ref words A, dist
// words B, vector v = i + k * threads) through vec(), flushing every
// kFlushVecs calls, and the same samples through the literal form.
template <int BPC, class Acc>
__global__ void stream(const uint4 *A, const uint4 *B, uint32_t n_vec, uint32_t threads, u64 *fast,
                       u64 *lit) {
    const uint32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= threads) return;
    Acc acc;
    LiteralSums ref;
    uint32_t calls = 0;
    for (uint32_t k = 0; k < n_vec; k++) {
        const uint4 a = A[(size_t)k * threads + i], b = B[(size_t)k * threads + i];
        acc.vec(a, b);
        if (++calls == Acc::kFlushVecs) { acc.flush(); calls = 0; }
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
        for (int w = 0; w < 4; w++) {
            if constexpr (BPC == 8) {
                for (int j = 0; j < 4; j++) ref.sample((wa[w] >> (8 * j)) & 0xffu, (wb[w] >> (8 * j)) & 0xffu);
            } else {
                ref.sample(wa[w] & 0xffffu, wb[w] & 0xffffu);
                ref.sample(wa[w] >> 16, wb[w] >> 16);
            }
        }
    }
    u64 t[kW];
    acc.totals(t);
    for (int k = 0; k < kW; k++) {
        fast[kW * (size_t)i + k] = t[k];
        lit[kW * (size_t)i + k] = ref.t[k];
    }
}

template <int BPC, class Acc = vqx::TermSums<BPC>>
cudaError_t launch_exhaustive(u64 *fast, u64 *lit, int use_samples) {
    const uint32_t top = 1u << BPC;
    exhaustive<BPC, Acc><<<(top + 127) / 128, 128>>>(fast, lit, use_samples);
    return cudaGetLastError();
}

template <int BPC, class Acc = vqx::TermSums<BPC>>
cudaError_t launch_stream(const uint4 *A, const uint4 *B, uint32_t n_vec, uint32_t threads, u64 *fast,
                          u64 *lit) {
    stream<BPC, Acc><<<(threads + 127) / 128, 128>>>(A, B, n_vec, threads, fast, lit);
    return cudaGetLastError();
}

// One thread initialises an mbarrier that expects one arrival, then waits
// for it with the library's bounded wait and a limit of `limit` cycles.
// Nothing ever arrives, so the wait must give up and return false; out[0]
// receives 1 if it did, out[1] the cycles it waited.
__global__ void wait_runs_out(long long limit, long long *out) {
    __shared__ __align__(8) u64 bar;
    const uint32_t a = vqx::smem_u32(&bar);
    vqx::mbar_init(a, 1);
    vqx::mbar_fence_init();
    const long long t0 = clock64();
    const bool done = vqx::mbar_wait(a, 0, limit);
    out[1] = clock64() - t0;
    out[0] = done ? 0 : 1;
}

}  // namespace

extern "C" {

// Bounded-wait check: returns a cudaError_t; out_host[0] = 1 when the wait
// gave up, out_host[1] = cycles waited.
int vqx_test_wait_timeout(long long limit, long long *out_host) {
    long long *o = nullptr;
    cudaError_t e = cudaMalloc(&o, 2 * sizeof(long long));
    if (e == cudaSuccess) {
        wait_runs_out<<<1, 1>>>(limit, o);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(out_host, o, 2 * sizeof(long long), cudaMemcpyDeviceToHost);
    cudaFree(o);
    return (int)e;
}

// Exhaustive check for one bit depth: fast/lit are host arrays of 8 * 2^bpc
// uint64.  sse: at 16 bits, the accumulator that also carries the SSE.
// Returns a cudaError_t (0 on success).
int vqx_test_exhaustive(int bpc, int use_samples, int sse, unsigned long long *fast_host,
                        unsigned long long *lit_host) {
    const size_t n = (size_t)kW * ((size_t)1 << bpc);
    u64 *f = nullptr, *l = nullptr;
    cudaError_t e = cudaMalloc(&f, n * 8);
    if (e == cudaSuccess) e = cudaMalloc(&l, n * 8);
    if (e == cudaSuccess) {
        switch (bpc) {
        case 8: e = launch_exhaustive<8>(f, l, use_samples); break;
        case 10: e = launch_exhaustive<10>(f, l, use_samples); break;
        case 12: e = launch_exhaustive<12>(f, l, use_samples); break;
        case 16:
            e = sse ? launch_exhaustive<16, vqx::TermSums16Sse>(f, l, use_samples)
                    : launch_exhaustive<16>(f, l, use_samples);
            break;
        default: e = cudaErrorInvalidValue;
        }
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(fast_host, f, n * 8, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(lit_host, l, n * 8, cudaMemcpyDeviceToHost);
    cudaFree(f);
    cudaFree(l);
    return (int)e;
}

// Stream check: a_host/b_host hold n_vec * threads 16-byte vectors each;
// fast/lit receive 8 * threads uint64.  sse as for vqx_test_exhaustive.
int vqx_test_stream(int bpc, int sse, const void *a_host, const void *b_host, unsigned n_vec,
                    unsigned threads, unsigned long long *fast_host, unsigned long long *lit_host) {
    const size_t bytes = (size_t)n_vec * threads * 16, n = (size_t)kW * (size_t)threads;
    void *a = nullptr, *b = nullptr;
    u64 *f = nullptr, *l = nullptr;
    cudaError_t e = cudaMalloc(&a, bytes);
    if (e == cudaSuccess) e = cudaMalloc(&b, bytes);
    if (e == cudaSuccess) e = cudaMalloc(&f, n * 8);
    if (e == cudaSuccess) e = cudaMalloc(&l, n * 8);
    if (e == cudaSuccess) e = cudaMemcpy(a, a_host, bytes, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(b, b_host, bytes, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) {
        const uint4 *A = (const uint4 *)a, *B = (const uint4 *)b;
        switch (bpc) {
        case 8: e = launch_stream<8>(A, B, n_vec, threads, f, l); break;
        case 10: e = launch_stream<10>(A, B, n_vec, threads, f, l); break;
        case 12: e = launch_stream<12>(A, B, n_vec, threads, f, l); break;
        case 16:
            e = sse ? launch_stream<16, vqx::TermSums16Sse>(A, B, n_vec, threads, f, l)
                    : launch_stream<16>(A, B, n_vec, threads, f, l);
            break;
        default: e = cudaErrorInvalidValue;
        }
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(fast_host, f, n * 8, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(lit_host, l, n * 8, cudaMemcpyDeviceToHost);
    cudaFree(a);
    cudaFree(b);
    cudaFree(f);
    cudaFree(l);
    return (int)e;
}

}  // extern "C"
