/*
 * The C boundary used from C: one decode step (pa_append_kv, then pa_decode;
 * and the same step as one pa_append_decode call on a copy of the pools)
 * and a verification step for the newest two tokens of every sequence
 * (pa_decode_multi, then the same rows through pa_prefill's tensor-core
 * kernel), the PagedEviction page scores of the appended pools
 * (pa_page_scores) and two copy-on-write block copies (pa_copy_blocks) on
 * device memory from cudaMalloc, with no Python or
 * PyTorch involved, checked against the fp64 oracle (linked from oracle/ as
 * test infrastructure). Inputs are deterministic (an integer hash), the pools hold
 * NaN in every slot past each sequence, and the tables name a shuffled set of
 * physical blocks with -1 past each sequence.
 *
 * Exit status 0 when the appended and the copied pools match the oracle's bit
 * for bit, every attention output is within the bf16 tolerance (1.5e-2
 * absolute), the page scores within 1e-4 relative and the victims equal.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "pa.h"

/* The oracle's C entry points (oracle/oracle.cpp). */
int oracle_decode(const void* q, const void* kpool, const void* vpool, const int32_t* table,
                  int max_blocks, const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int bs,
                  int num_blocks, float scale, int dtype, double* out, const int32_t* pairs,
                  int npairs, int nthreads);
int oracle_append(const void* k_new, const void* v_new, void* kpool, void* vpool,
                  const int32_t* table, int max_blocks, const int32_t* cache_lens, int B, int Hkv,
                  int D, int bs, int num_blocks, int elem_bytes);
int oracle_prefill(const void* q, const void* kpool, const void* vpool, const int32_t* table,
                   int max_blocks, const int32_t* seq_lens, const int32_t* q_start, int B, int Hq,
                   int Hkv, int D, int bs, int num_blocks, float scale, int dtype, double* out,
                   int nthreads);
int oracle_page_scores(const void* kpool, const void* vpool, const int32_t* table, int max_blocks,
                       const int32_t* seq_lens, int B, int Hkv, int D, int bs, int num_blocks,
                       int dtype, double* scores, int32_t* victims);
int oracle_copy_blocks(void* kpool, void* vpool, const int32_t* src, const int32_t* dst, int n,
                       int num_blocks, int64_t block_bytes);

enum { B = 3, HQ = 8, HKV = 2, D = 128, BS = 16, MAXB = 20, SPARE = 5 };
static const int kLens[B] = {1, 37, 300}; /* tokens after the append */

static uint32_t hash32(uint32_t x) {
    x ^= x >> 16; x *= 0x7feb352dU; x ^= x >> 15; x *= 0x846ca68bU; x ^= x >> 16;
    return x;
}

/* A value in [-1, 1) as bf16 bits (round to nearest even). */
static uint16_t bf16_of(uint32_t key) {
    float f = (float)((double)(hash32(key) >> 8) / 8388608.0 - 1.0);
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

static float f32_of_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

#define CHECK_CUDA(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
    fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_)); return 2; } } while (0)
#define CHECK_PA(x) do { pa_status s_ = (x); if (s_ != PA_OK) { \
    fprintf(stderr, "%s: %s\n", #x, pa_status_str(s_)); return 3; } } while (0)

int main(void) {
    int used = 0;
    for (int b = 0; b < B; ++b) used += (kLens[b] + BS - 1) / BS;
    const int NB = used + SPARE;
    const size_t pool_elems = (size_t)NB * HKV * BS * D;

    /* Shuffled physical blocks, consumed in order; -1 past each sequence. */
    int32_t* perm = malloc(sizeof(int32_t) * NB);
    for (int i = 0; i < NB; ++i) perm[i] = i;
    for (int i = NB - 1; i > 0; --i) {
        const int j = (int)(hash32(0xB10C0000u + (uint32_t)i) % (uint32_t)(i + 1));
        const int32_t t = perm[i]; perm[i] = perm[j]; perm[j] = t;
    }
    int32_t table[B * MAXB];
    int32_t seq_lens[B], cache_lens[B];
    int next = 0;
    for (int b = 0; b < B; ++b) {
        const int nb = (kLens[b] + BS - 1) / BS;
        for (int p = 0; p < MAXB; ++p) table[b * MAXB + p] = p < nb ? perm[next++] : -1;
        seq_lens[b] = kLens[b];
        cache_lens[b] = kLens[b] - 1;
    }

    /* Pools: hashed values, NaN in every slot past each sequence's cached tokens. */
    uint16_t* kpool = malloc(pool_elems * 2);
    uint16_t* vpool = malloc(pool_elems * 2);
    for (size_t i = 0; i < pool_elems; ++i) {
        kpool[i] = bf16_of(0x10000000u + (uint32_t)i);
        vpool[i] = bf16_of(0x20000000u + (uint32_t)i);
    }
    for (int b = 0; b < B; ++b)
        for (int t = cache_lens[b]; t < (kLens[b] + BS - 1) / BS * BS; ++t) {
            const int blk = table[b * MAXB + t / BS];
            for (int h = 0; h < HKV; ++h)
                for (int d = 0; d < D; ++d) {
                    const size_t i = (((size_t)blk * HKV + h) * BS + t % BS) * D + d;
                    kpool[i] = vpool[i] = 0x7FC0; /* NaN */
                }
        }
    uint16_t q[B * HQ * D], k_new[B * HKV * D], v_new[B * HKV * D];
    for (int i = 0; i < B * HQ * D; ++i) q[i] = bf16_of(0x30000000u + (uint32_t)i);
    for (int i = 0; i < B * HKV * D; ++i) {
        k_new[i] = bf16_of(0x40000000u + (uint32_t)i);
        v_new[i] = bf16_of(0x50000000u + (uint32_t)i);
    }

    void *dk, *dv, *dq, *dkn, *dvn, *dout;
    int32_t *dtab, *dsl, *dcl;
    CHECK_CUDA(cudaMalloc(&dk, pool_elems * 2));
    CHECK_CUDA(cudaMalloc(&dv, pool_elems * 2));
    CHECK_CUDA(cudaMalloc(&dq, sizeof q));
    CHECK_CUDA(cudaMalloc(&dkn, sizeof k_new));
    CHECK_CUDA(cudaMalloc(&dvn, sizeof v_new));
    CHECK_CUDA(cudaMalloc(&dout, (size_t)B * HQ * D * 2));
    CHECK_CUDA(cudaMalloc((void**)&dtab, sizeof table));
    CHECK_CUDA(cudaMalloc((void**)&dsl, sizeof seq_lens));
    CHECK_CUDA(cudaMalloc((void**)&dcl, sizeof cache_lens));
    CHECK_CUDA(cudaMemcpy(dk, kpool, pool_elems * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dv, vpool, pool_elems * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dq, q, sizeof q, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dkn, k_new, sizeof k_new, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dvn, v_new, sizeof v_new, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dtab, table, sizeof table, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dsl, seq_lens, sizeof seq_lens, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dcl, cache_lens, sizeof cache_lens, cudaMemcpyHostToDevice));

    /* A second copy of the pools for the same step in one call. */
    void *dk2, *dv2, *dout3;
    CHECK_CUDA(cudaMalloc(&dk2, pool_elems * 2));
    CHECK_CUDA(cudaMalloc(&dv2, pool_elems * 2));
    CHECK_CUDA(cudaMalloc(&dout3, (size_t)B * HQ * D * 2));
    CHECK_CUDA(cudaMemcpy(dk2, kpool, pool_elems * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dv2, vpool, pool_elems * 2, cudaMemcpyHostToDevice));

    const float scale = 1.0f / sqrtf((float)D);
    pa_plan* plan = NULL;
    CHECK_PA(pa_append_kv(dkn, dvn, dk, dv, dtab, MAXB, dcl, B, HKV, D, BS, NB, PA_BF16, NULL));
    CHECK_PA(pa_decode(dq, dk, dv, dtab, MAXB, dsl, B, HQ, HKV, D, BS, NB, MAXB * BS, scale, PA_BF16,
                       dout, PA_BF16, &plan, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    int derr = -1, aerr = -1;
    CHECK_PA(pa_last_device_error(plan, &derr));
    CHECK_PA(pa_last_device_error(NULL, &aerr));

    uint16_t* kgot = malloc(pool_elems * 2);
    uint16_t* vgot = malloc(pool_elems * 2);
    uint16_t out[B * HQ * D];
    CHECK_CUDA(cudaMemcpy(kgot, dk, pool_elems * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(vgot, dv, pool_elems * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(out, dout, sizeof out, cudaMemcpyDeviceToHost));

    /* The same step as one call: the append at seq_lens - 1 inside the decode. */
    pa_plan* plan3 = NULL;
    CHECK_PA(pa_append_decode(dq, dkn, dvn, dk2, dv2, dtab, MAXB, dsl, B, HQ, HKV, D, BS, NB,
                              MAXB * BS, scale, PA_BF16, dout3, PA_BF16, &plan3, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    int ferr = -1;
    CHECK_PA(pa_last_device_error(plan3, &ferr));
    CHECK_PA(pa_free(plan3));
    uint16_t* k3 = malloc(pool_elems * 2);
    uint16_t* v3 = malloc(pool_elems * 2);
    uint16_t out3[B * HQ * D];
    CHECK_CUDA(cudaMemcpy(k3, dk2, pool_elems * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(v3, dv2, pool_elems * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(out3, dout3, sizeof out3, cudaMemcpyDeviceToHost));
    const int fused_same = memcmp(k3, kgot, pool_elems * 2) == 0 &&
                           memcmp(v3, vgot, pool_elems * 2) == 0 &&
                           memcmp(out3, out, sizeof out) == 0;

    /* Verification step: the newest min(2, L_b) tokens of each sequence. */
    int32_t q_start[B + 1];
    q_start[0] = 0;
    for (int b = 0; b < B; ++b) q_start[b + 1] = q_start[b] + (kLens[b] < 2 ? kLens[b] : 2);
    const int T = q_start[B];
    uint16_t q2[2 * B * HQ * D];
    for (int i = 0; i < T * HQ * D; ++i) q2[i] = bf16_of(0x60000000u + (uint32_t)i);
    void *dq2, *dout2;
    int32_t* dqs;
    CHECK_CUDA(cudaMalloc(&dq2, (size_t)T * HQ * D * 2));
    CHECK_CUDA(cudaMalloc(&dout2, (size_t)T * HQ * D * 2));
    CHECK_CUDA(cudaMalloc((void**)&dqs, sizeof q_start));
    CHECK_CUDA(cudaMemcpy(dq2, q2, (size_t)T * HQ * D * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dqs, q_start, sizeof q_start, cudaMemcpyHostToDevice));
    CHECK_PA(pa_decode_multi(dq2, dqs, T, 2, dk, dv, dtab, MAXB, dsl, B, HQ, HKV, D, BS, NB,
                             MAXB * BS, scale, PA_BF16, dout2, PA_BF16, &plan, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    int merr = -1;
    CHECK_PA(pa_last_device_error(plan, &merr));
    uint16_t out2[2 * B * HQ * D];
    CHECK_CUDA(cudaMemcpy(out2, dout2, (size_t)T * HQ * D * 2, cudaMemcpyDeviceToHost));
    CHECK_PA(pa_free(plan));

    /* The same rows through pa_prefill (no plan; the library-wide error word). */
    void* dout4;
    CHECK_CUDA(cudaMalloc(&dout4, (size_t)T * HQ * D * 2));
    CHECK_PA(pa_prefill(dq2, dqs, T, dk, dv, dtab, MAXB, dsl, B, HQ, HKV, D, BS, NB, 2, MAXB * BS,
                        scale, PA_BF16, dout4, PA_BF16, NULL, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    int perr = -1;
    CHECK_PA(pa_last_device_error(NULL, &perr));
    uint16_t out4[2 * B * HQ * D];
    CHECK_CUDA(cudaMemcpy(out4, dout4, (size_t)T * HQ * D * 2, cudaMemcpyDeviceToHost));

    /* PagedEviction page scores over the appended pools. */
    float* dsc;
    int32_t* dvi;
    int* dserr;
    CHECK_CUDA(cudaMalloc((void**)&dsc, sizeof(float) * B * MAXB));
    CHECK_CUDA(cudaMalloc((void**)&dvi, sizeof(int32_t) * B));
    CHECK_CUDA(cudaMalloc((void**)&dserr, sizeof(int)));
    CHECK_CUDA(cudaMemset(dsc, 0, sizeof(float) * B * MAXB));
    CHECK_CUDA(cudaMemset(dserr, 0, sizeof(int)));
    CHECK_PA(pa_page_scores(dk, dv, dtab, MAXB, dsl, B, HKV, D, BS, NB, MAXB * BS, PA_BF16, dsc, dvi,
                            dserr, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    float sc[B * MAXB];
    int32_t vi[B];
    int serr = -1;
    CHECK_CUDA(cudaMemcpy(sc, dsc, sizeof sc, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(vi, dvi, sizeof vi, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(&serr, dserr, sizeof serr, cudaMemcpyDeviceToHost));

    /* The oracle: append on the host pools, then fp64 attention. */
    if (oracle_append(k_new, v_new, kpool, vpool, table, MAXB, cache_lens, B, HKV, D, BS, NB, 2) != 0)
        return 4;
    double ref[B * HQ * D];
    if (oracle_decode(q, kpool, vpool, table, MAXB, seq_lens, B, HQ, HKV, D, BS, NB, scale, 1, ref,
                      NULL, 0, 4) != 0)
        return 4;
    double ref2[2 * B * HQ * D];
    if (oracle_prefill(q2, kpool, vpool, table, MAXB, seq_lens, q_start, B, HQ, HKV, D, BS, NB,
                       scale, 1, ref2, 4) != 0)
        return 4;
    const int pools_equal = memcmp(kgot, kpool, pool_elems * 2) == 0 &&
                            memcmp(vgot, vpool, pool_elems * 2) == 0;
    double rsc[B * MAXB];
    int32_t rvi[B];
    if (oracle_page_scores(kpool, vpool, table, MAXB, seq_lens, B, HKV, D, BS, NB, 1, rsc, rvi) != 0)
        return 4;
    double worst_sc = 0.0; /* relative */
    int victims_equal = 1, scores_ok = 1;
    for (int b = 0; b < B; ++b) {
        victims_equal &= vi[b] == rvi[b];
        for (int p = 0; p < (kLens[b] + BS - 1) / BS; ++p) {
            const double r = rsc[b * MAXB + p], e = fabs((double)sc[b * MAXB + p] - r) / fabs(r);
            scores_ok &= e <= 1e-4; /* false for NaN */
            if (e > worst_sc) worst_sc = e;
        }
    }

    /* Copy on write: two blocks of sequence 2 into two free blocks. */
    int32_t csrc[2] = {table[2 * MAXB], table[2 * MAXB + 1]};
    int32_t cdst[2] = {perm[used], perm[used + 1]};
    int32_t *dcs, *dcd;
    CHECK_CUDA(cudaMalloc((void**)&dcs, sizeof csrc));
    CHECK_CUDA(cudaMalloc((void**)&dcd, sizeof cdst));
    CHECK_CUDA(cudaMemcpy(dcs, csrc, sizeof csrc, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dcd, cdst, sizeof cdst, cudaMemcpyHostToDevice));
    CHECK_PA(pa_copy_blocks(dk, dv, dcs, dcd, 2, HKV, D, BS, NB, PA_BF16, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    int cerr = -1;
    CHECK_PA(pa_last_device_error(NULL, &cerr));
    CHECK_CUDA(cudaMemcpy(kgot, dk, pool_elems * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(vgot, dv, pool_elems * 2, cudaMemcpyDeviceToHost));
    if (oracle_copy_blocks(kpool, vpool, csrc, cdst, 2, NB, (int64_t)HKV * BS * D * 2) != 0) return 4;
    const int copies_equal = memcmp(kgot, kpool, pool_elems * 2) == 0 &&
                             memcmp(vgot, vpool, pool_elems * 2) == 0;
    double worst = 0.0;
    int finite = 1;
    for (int i = 0; i < B * HQ * D; ++i) {
        const double g = (double)f32_of_bf16(out[i]);
        finite &= isfinite(g) != 0;
        const double e = fabs(g - ref[i]);
        if (e > worst) worst = e;
    }
    double worst2 = 0.0, worst3 = 0.0;
    for (int i = 0; i < T * HQ * D; ++i) {
        const double g = (double)f32_of_bf16(out2[i]), g4 = (double)f32_of_bf16(out4[i]);
        finite &= isfinite(g) != 0 && isfinite(g4) != 0;
        const double e = fabs(g - ref2[i]), e4 = fabs(g4 - ref2[i]);
        if (e > worst2) worst2 = e;
        if (e4 > worst3) worst3 = e4;
    }
    printf("device errors %d/%d/%d/%d/%d/%d/%d, pools equal %d, one-call step identical %d, "
           "finite %d, max abs error %.3e / %.3e / %.3e, page scores rel %.3e, victims equal %d, "
           "copies equal %d\n", derr, aerr, merr, ferr, perr, serr, cerr, pools_equal, fused_same,
           finite, worst, worst2, worst3, worst_sc, victims_equal, copies_equal);
    return (derr == 0 && aerr == 0 && merr == 0 && ferr == 0 && perr == 0 && serr == 0 &&
            cerr == 0 && pools_equal && fused_same && finite && worst <= 1.5e-2 &&
            worst2 <= 1.5e-2 && worst3 <= 1.5e-2 && scores_ok && victims_equal &&
            copies_equal)
               ? 0
               : 1;
}
