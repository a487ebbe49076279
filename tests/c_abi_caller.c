/*
 * A plain C99 caller of libgqa_decode.so through include/gqa_decode.h, with no
 * Python between the caller and the library (tests/test_c_abi_program.py
 * compiles and runs it).
 *
 *   c_abi_caller plan
 *       host-only calls: the plan of a Llama-shaped layer, argument errors,
 *       status strings; prints one "name value" pair per line.
 *   c_abi_caller run IN OUT
 *       IN: int32 B, sq, H, G, D, Tmax; float scale; then q [B,sq,H,D] and
 *       k, v [B,G,Tmax,D] as bf16 bits, seq_lens [B] int32. Copies them to
 *       the device on a stream of its own, calls gqa_decode, and writes OUT:
 *       out [B,sq,H,D] bf16 bits, then lse [B,sq,H] float.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "gqa_decode.h"

static int plan_mode(void) {
    gqa_decode_plan_t pl;
    const int st = gqa_decode_plan(16, 1, 32, 8, 128, 4096, 152, &pl);
    printf("plan_status %d\n", st);
    printf("plan_row_tiles %d\n", pl.row_tiles);
    printf("plan_tile_tokens %d\n", pl.tile_tokens);
    printf("plan_max_tiles %lld\n", pl.max_tiles);
    printf("head_ratio %d\n", gqa_decode_plan(1, 1, 30, 8, 128, 64, 152, &pl));
    printf("bad_head_dim %d\n", gqa_decode_plan(1, 1, 8, 8, 96, 64, 152, &pl));
    printf("null_pointers %d\n", gqa_decode(NULL, NULL, NULL, NULL, 1.0f, NULL, NULL, 1, 1, 8, 8, 128, 64, 0));
    printf("strerror_ok %s\n", gqa_decode_strerror(GQA_OK) != NULL ? "yes" : "no");
    return 0;
}

#define CHECK(call)                                                        \
    do {                                                                   \
        cudaError_t e_ = (call);                                           \
        if (e_ != cudaSuccess) {                                           \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));  \
            return 3;                                                      \
        }                                                                  \
    } while (0)

static int read_all(FILE* f, void* p, size_t bytes) { return fread(p, 1, bytes, f) == bytes ? 0 : 1; }

static int run_mode(const char* in_path, const char* out_path) {
    FILE* f = fopen(in_path, "rb");
    if (!f) return 2;
    int32_t hdr[6];
    float scale;
    if (read_all(f, hdr, sizeof hdr) || read_all(f, &scale, sizeof scale)) return 2;
    const int B = hdr[0], sq = hdr[1], H = hdr[2], G = hdr[3], D = hdr[4], Tmax = hdr[5];
    const size_t nq = (size_t)B * sq * H * D, nk = (size_t)B * G * Tmax * D, nl = (size_t)B * sq * H;
    uint16_t* hq = (uint16_t*)malloc(nq * 2);
    uint16_t* hk = (uint16_t*)malloc(nk * 2);
    uint16_t* hv = (uint16_t*)malloc(nk * 2);
    int32_t* hl = (int32_t*)malloc((size_t)B * 4);
    uint16_t* ho = (uint16_t*)malloc(nq * 2);
    float* hlse = (float*)malloc(nl * 4);
    if (!hq || !hk || !hv || !hl || !ho || !hlse) return 2;
    if (read_all(f, hq, nq * 2) || read_all(f, hk, nk * 2) || read_all(f, hv, nk * 2) ||
        read_all(f, hl, (size_t)B * 4))
        return 2;
    fclose(f);

    void *dq, *dk, *dv, *dl, *dout, *dlse;
    cudaStream_t s;
    CHECK(cudaStreamCreate(&s));
    CHECK(cudaMalloc(&dq, nq * 2));
    CHECK(cudaMalloc(&dk, nk * 2));
    CHECK(cudaMalloc(&dv, nk * 2));
    CHECK(cudaMalloc(&dl, (size_t)B * 4));
    CHECK(cudaMalloc(&dout, nq * 2));
    CHECK(cudaMalloc(&dlse, nl * 4));
    CHECK(cudaMemcpyAsync(dq, hq, nq * 2, cudaMemcpyHostToDevice, s));
    CHECK(cudaMemcpyAsync(dk, hk, nk * 2, cudaMemcpyHostToDevice, s));
    CHECK(cudaMemcpyAsync(dv, hv, nk * 2, cudaMemcpyHostToDevice, s));
    CHECK(cudaMemcpyAsync(dl, hl, (size_t)B * 4, cudaMemcpyHostToDevice, s));
    const int st = gqa_decode(dq, dk, dv, (const int32_t*)dl, scale, dout, (float*)dlse, B, sq, H, G, D, Tmax, s);
    if (st != GQA_OK) {
        fprintf(stderr, "gqa_decode: %s\n", gqa_decode_strerror(st));
        return 4;
    }
    CHECK(cudaMemcpyAsync(ho, dout, nq * 2, cudaMemcpyDeviceToHost, s));
    CHECK(cudaMemcpyAsync(hlse, dlse, nl * 4, cudaMemcpyDeviceToHost, s));
    CHECK(cudaStreamSynchronize(s));
    const int dev = gqa_decode_check_error(s);
    if (dev != GQA_OK) {
        fprintf(stderr, "device status: %s\n", gqa_decode_strerror(dev));
        return 5;
    }
    FILE* o = fopen(out_path, "wb");
    if (!o || fwrite(ho, 2, nq, o) != nq || fwrite(hlse, 4, nl, o) != nl) return 2;
    fclose(o);
    cudaFree(dq);
    cudaFree(dk);
    cudaFree(dv);
    cudaFree(dl);
    cudaFree(dout);
    cudaFree(dlse);
    cudaStreamDestroy(s);
    free(hq);
    free(hk);
    free(hv);
    free(hl);
    free(ho);
    free(hlse);
    printf("ok\n");
    return 0;
}

int main(int argc, char** argv) {
    if (argc == 2 && argv[1][0] == 'p') return plan_mode();
    if (argc == 4 && argv[1][0] == 'r') return run_mode(argv[2], argv[3]);
    fprintf(stderr, "usage: %s plan | run IN OUT\n", argv[0]);
    return 1;
}
