/*
 * A plain C consumer of libmsda (include/msda.h): no Python, no C++.
 *
 * On a constant value map c, the forward's output is c times the sum, over
 * samples, of the attention weight times the share of the bilinear tent that
 * falls inside the map; for samples whose four corners are all inside, that
 * is c * sum A.  This program samples two levels strictly inside, with
 * weights summing to 1 per (query, head), so every output channel must equal
 * c.  It also checks that a bad call is rejected with a message.
 * Exit status 0 on success.
 */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "msda.h"

#define N 1
#define LQ 5
#define M 2
#define D 8
#define L 2
#define K 3

int main(void)
{
    const int64_t shapes[2 * L] = {4, 6, 2, 3};     /* (H, W) of each level */
    const int64_t starts[L] = {0, 24};
    const int S = 24 + 6;
    const float c = 0.75f;
    size_t nval = (size_t)N * S * M * D, nsmp = (size_t)N * LQ * M * L * K, nout = (size_t)N * LQ * M * D;
    float *hv = malloc(nval * 4), *hloc = malloc(nsmp * 2 * 4), *hA = malloc(nsmp * 4), *hout = malloc(nout * 4);
    for (size_t i = 0; i < nval; ++i) hv[i] = c;
    for (size_t s = 0; s < nsmp; ++s) {
        /* inside: pixel coordinates in [0.2, 0.8] of the first cell of each level */
        int l = (int)((s / K) % L);
        double W = (double)shapes[2 * l + 1], H = (double)shapes[2 * l];
        double fx = 0.2 + 0.6 * (double)(s % 7) / 6.0, fy = 0.2 + 0.6 * (double)(s % 5) / 4.0;
        hloc[2 * s] = (float)((fx + 0.5) / W);
        hloc[2 * s + 1] = (float)((fy + 0.5) / H);
        hA[s] = 1.0f / (L * K);
    }
    float *dv, *dloc, *dA, *dout;
    if (cudaMalloc((void **)&dv, nval * 4) || cudaMalloc((void **)&dloc, nsmp * 8) || cudaMalloc((void **)&dA, nsmp * 4) ||
        cudaMalloc((void **)&dout, nout * 4)) {
        fprintf(stderr, "cudaMalloc failed\n");
        return 2;
    }
    cudaMemcpy(dv, hv, nval * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(dloc, hloc, nsmp * 8, cudaMemcpyHostToDevice);
    cudaMemcpy(dA, hA, nsmp * 4, cudaMemcpyHostToDevice);

    msda_problem p = {N, S, M, D, LQ, L, K, MSDA_F32, 0u, 0};
    msda_status st = msda_forward(&p, dv, shapes, starts, dloc, dA, dout, NULL);
    if (st != MSDA_OK) {
        fprintf(stderr, "msda_forward: %s: %s\n", msda_status_string(st), msda_last_error());
        return 1;
    }
    cudaMemcpy(hout, dout, nout * 4, cudaMemcpyDeviceToHost);
    double worst = 0.0;
    for (size_t i = 0; i < nout; ++i) worst = fmax(worst, fabs((double)hout[i] - c));
    /* a head_dim the kernels do not support is rejected before any launch */
    msda_problem bad = p;
    bad.head_dim = 12;
    st = msda_forward(&bad, dv, shapes, starts, dloc, dA, dout, NULL);
    int rejected = st == MSDA_ERR_UNSUPPORTED && msda_last_error()[0] != 0;
    printf("max |out - c| = %.3g, bad call rejected: %d (%s)\n", worst, rejected, msda_last_error());
    cudaFree(dv);
    cudaFree(dloc);
    cudaFree(dA);
    cudaFree(dout);
    free(hv);
    free(hloc);
    free(hA);
    free(hout);
    return (worst <= 1e-6 && rejected) ? 0 : 1;
}
