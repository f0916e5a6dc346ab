/* A plain C user of the vqx C ABI: no Python, no PyTorch.
 *
 * Usage: abi_client <planes.bin> <width> <height> <bpc> <n_frames>
 * planes.bin holds the reference frames, then the distorted frames, dense
 * (row pitch width * bytes per sample).  The client copies them to the
 * device with the CUDA runtime, calls vqx_plane_stats and vqx_plane_int_psnr
 * on the default stream, and prints one line per frame: the five exact sums
 * and the flags in decimal, then the bit patterns of the eight doubles and of
 * the integer psnr's SSE and three doubles in hexadecimal, so that the caller
 * can compare them exactly.  It also checks that argument errors come back as
 * status codes with their strings.  Exit status: 0 when every call behaved,
 * 1 otherwise.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "vqx.h"

static uint64_t bits(double x) {
    uint64_t u;
    memcpy(&u, &x, sizeof u);
    return u;
}

int main(int argc, char **argv) {
    if (argc != 6) {
        fprintf(stderr, "usage: %s planes.bin width height bpc n_frames\n", argv[0]);
        return 1;
    }
    const int width = atoi(argv[2]), height = atoi(argv[3]), bpc = atoi(argv[4]),
              n = atoi(argv[5]);
    const size_t bps = bpc == 8 ? 1 : 2;
    const size_t stride = (size_t)width * bps;
    const size_t plane_bytes = stride * (size_t)height * (size_t)n;
    unsigned char *host = (unsigned char *)malloc(2 * plane_bytes);
    FILE *f = fopen(argv[1], "rb");
    if (!host || !f || fread(host, 1, 2 * plane_bytes, f) != 2 * plane_bytes) {
        fprintf(stderr, "cannot read %s\n", argv[1]);
        return 1;
    }
    fclose(f);

    void *ref = NULL, *dist = NULL;
    if (cudaMalloc(&ref, plane_bytes) != cudaSuccess || cudaMalloc(&dist, plane_bytes) != cudaSuccess ||
        cudaMemcpy(ref, host, plane_bytes, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(dist, host + plane_bytes, plane_bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
        fprintf(stderr, "CUDA setup failed\n");
        return 1;
    }

    vqx_frame_stats *st = (vqx_frame_stats *)calloc((size_t)n, sizeof *st);
    vqx_int_psnr_stats *ip = (vqx_int_psnr_stats *)calloc((size_t)n, sizeof *ip);
    int rc = vqx_plane_stats(ref, dist, width, height, stride, bpc, n, NULL, st);
    if (rc != VQX_OK) {
        fprintf(stderr, "vqx_plane_stats: %s\n", vqx_status_string(rc));
        return 1;
    }
    rc = vqx_plane_int_psnr(ref, dist, width, height, stride, bpc, n, NULL, ip);
    if (rc != VQX_OK) {
        fprintf(stderr, "vqx_plane_int_psnr: %s\n", vqx_status_string(rc));
        return 1;
    }
    for (int i = 0; i < n; i++) {
        const vqx_frame_stats *s = &st[i];
        printf("frame %d %llu %llu %llu %llu %llu %u", i, (unsigned long long)s->noise_units,
               (unsigned long long)s->ref_sum, (unsigned long long)s->dist_sum,
               (unsigned long long)s->ref_sumsq, (unsigned long long)s->dist_sumsq, s->flags);
        const double d[8] = {s->noise,    s->mse,        s->psnr,      s->psnr_uncapped,
                             s->ref_mean, s->ref_meansq, s->dist_mean, s->dist_meansq};
        for (int k = 0; k < 8; k++) printf(" %016llx", (unsigned long long)bits(d[k]));
        printf(" %llu %016llx %016llx %016llx\n", (unsigned long long)ip[i].sse,
               (unsigned long long)bits(ip[i].mse), (unsigned long long)bits(ip[i].psnr),
               (unsigned long long)bits(ip[i].psnr_uncapped));
    }

    /* argument errors: status codes, nothing launched */
    int ok = 1;
    ok &= vqx_plane_stats(ref, dist, width, height, stride, 9, n, NULL, st) == VQX_EBPC;
    ok &= vqx_plane_stats(NULL, dist, width, height, stride, bpc, n, NULL, st) == VQX_EINVAL;
    ok &= vqx_plane_stats(ref, dist, width, height, stride - 1, bpc, n, NULL, st) == VQX_EINVAL;
    ok &= strlen(vqx_status_string(VQX_EBPC)) > 0 && strlen(vqx_status_string(VQX_OK)) > 0;
    printf("errors %s cap %.17g\n", ok ? "ok" : "wrong", vqx_psnr_cap(bpc));

    cudaFree(ref);
    cudaFree(dist);
    free(st);
    free(ip);
    free(host);
    return ok ? 0 : 1;
}
