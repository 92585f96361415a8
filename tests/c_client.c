/*
 * A plain C client of libsdp.so: no Python, no framework types. It reads
 * Q, K, V (16-bit patterns) from a file, runs one forward entry point through
 * the C ABI on device buffers it allocates itself, and writes O and LSE back.
 *
 * usage: c_client <in.bin> <out.bin> B Hq Hkv Sq Skv D dtype scale [mode [n_splits]]
 * mode:    fwd (default, sdp_fwd), causal (sdp_fwd_causal), splitkv
 *          (sdp_fwd_splitkv with n_splits, 0 = automatic, and the workspace the
 *          library asks for) or noalloc (sdp_fwd_noalloc, status read with
 *          sdp_fwd_noalloc_status)
 * in.bin:  Q | K | V as raw 16-bit patterns, [B,Hq,Sq,D] then [B,Hkv,Skv,D] twice
 * out.bin: O (16-bit, [B,Hq,Sq,D]) | LSE (fp32, [B,Hq,Sq])
 * Exit status 0 on success; on an error prints the library's message.
 */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "sdp.h"

static int fail(const char *what, int code)
{
    fprintf(stderr, "%s failed: %d (%s)\n", what, code, code <= 0 ? sdp_strerror(code) : "cuda");
    return 1;
}

int main(int argc, char **argv)
{
    if (argc < 11 || argc > 13) {
        fprintf(stderr, "usage: %s in.bin out.bin B Hq Hkv Sq Skv D dtype scale [mode [n_splits]]\n", argv[0]);
        return 2;
    }
    const char *mode = argc > 11 ? argv[11] : "fwd";
    const int n_splits = argc > 12 ? atoi(argv[12]) : 0;
    const int B = atoi(argv[3]), Hq = atoi(argv[4]), Hkv = atoi(argv[5]), Sq = atoi(argv[6]), Skv = atoi(argv[7]);
    const int D = atoi(argv[8]), dtype = atoi(argv[9]);
    const float scale = (float)atof(argv[10]);
    const size_t nq = (size_t)B * Hq * Sq * D, nkv = (size_t)B * Hkv * Skv * D, nl = (size_t)B * Hq * Sq;

    uint16_t *h_in = malloc(2 * (nq + 2 * nkv));
    uint16_t *h_o = malloc(2 * nq);
    float *h_l = malloc(4 * nl);
    FILE *f = fopen(argv[1], "rb");
    if (!f || !h_in || !h_o || !h_l || fread(h_in, 2, nq + 2 * nkv, f) != nq + 2 * nkv)
        return fail("reading the input", 1);
    fclose(f);

    void *q, *k, *v, *o;
    float *lse;
    if (cudaMalloc(&q, 2 * nq) || cudaMalloc(&k, 2 * nkv) || cudaMalloc(&v, 2 * nkv) || cudaMalloc(&o, 2 * nq) ||
        cudaMalloc((void **)&lse, 4 * nl))
        return fail("cudaMalloc", 1);
    if (cudaMemcpy(q, h_in, 2 * nq, cudaMemcpyHostToDevice) ||
        cudaMemcpy(k, h_in + nq, 2 * nkv, cudaMemcpyHostToDevice) ||
        cudaMemcpy(v, h_in + nq + nkv, 2 * nkv, cudaMemcpyHostToDevice))
        return fail("cudaMemcpy to the device", 1);

    int rc;
    void *ws = NULL;
    if (strcmp(mode, "fwd") == 0) {
        rc = sdp_fwd(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, scale, dtype, NULL);
    } else if (strcmp(mode, "causal") == 0) {
        rc = sdp_fwd_causal(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, scale, dtype, NULL);
    } else if (strcmp(mode, "splitkv") == 0) {
        const long long need = sdp_fwd_splitkv_workspace_bytes(B, Hq, Hkv, Sq, Skv, D, dtype, n_splits);
        if (need < 0)
            return fail("sdp_fwd_splitkv_workspace_bytes", (int)need);
        if (need > 0 && cudaMalloc(&ws, (size_t)need))
            return fail("cudaMalloc (workspace)", 1);
        rc = sdp_fwd_splitkv(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, scale, dtype, n_splits, ws,
                             (unsigned long long)need, NULL);
    } else if (strcmp(mode, "noalloc") == 0) {
        rc = sdp_fwd_noalloc(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, scale, dtype, NULL);
    } else {
        fprintf(stderr, "unknown mode %s\n", mode);
        return 2;
    }
    if (rc != SDP_OK)
        return fail(mode, rc);
    rc = strcmp(mode, "noalloc") == 0 ? sdp_fwd_noalloc_status(NULL) : sdp_poll_status(NULL);
    if (rc != SDP_OK)
        return fail("status", rc);

    if (cudaMemcpy(h_o, o, 2 * nq, cudaMemcpyDeviceToHost) || cudaMemcpy(h_l, lse, 4 * nl, cudaMemcpyDeviceToHost))
        return fail("cudaMemcpy to the host", 1);
    f = fopen(argv[2], "wb");
    if (!f || fwrite(h_o, 2, nq, f) != nq || fwrite(h_l, 4, nl, f) != nl)
        return fail("writing the output", 1);
    fclose(f);
    cudaFree(q);
    cudaFree(k);
    cudaFree(v);
    cudaFree(o);
    cudaFree(lse);
    if (ws)
        cudaFree(ws);
    sdp_shutdown();
    free(h_in);
    free(h_o);
    free(h_l);
    printf("ok version %d\n", sdp_version());
    return 0;
}
