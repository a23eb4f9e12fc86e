/*
 * decode_step.c -- one decode step through the C ABI of libpagedkv, from
 * plain C99: no Python, no torch.
 *
 * It builds a small paged KV cache on CUDA device 0 (five sequences of 1 to
 * 1500 tokens, 16 query heads over 4 KV heads, head_dim 128, 16-token blocks
 * in a shuffled pool), then on one stream:
 *   paged_decode_plan            how much workspace the automatic split needs;
 *   paged_decode_workspace_clear zero the new workspace's arrival counters;
 *   paged_decode_step_ex         append each sequence's newest K/V and attend,
 *                                in one kernel (PKV_APPEND_NEWEST: token b is
 *                                sequence b's newest token);
 *   paged_kv_get_error           read the device error word.
 * Inputs and results go to the file named by argv[1], so that a checker can
 * recompute the step independently (layout at write_all below).
 *
 * Build from the repository root once the library is built:
 *   cc -std=c99 -O2 -I include -I /usr/local/cuda/include \
 *      paged_kv_cache_213_gb300/examples/decode_step.c \
 *      -L paged_kv_cache_213_gb300/_build -lpagedkv \
 *      -L /usr/local/cuda/lib64 -lcudart \
 *      -Wl,-rpath,$PWD/paged_kv_cache_213_gb300/_build -o decode_step
 *   ./decode_step step.bin
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "pagedkv.h"

enum { B = 5, H = 16, HK = 4, D = 128, BS = 16, SPARE_BLOCKS = 7, MAX_LEN = 1500 };
enum { MB = (MAX_LEN + BS - 1) / BS }; /* block-table width */
static const int kLens[B] = {1, 16, 17, 300, MAX_LEN};

/* 64-bit linear congruential generator (Knuth's MMIX constants). */
static uint64_t g_state = 20261203u;
static uint32_t next_u32(void) {
    g_state = g_state * 6364136223846793005ull + 1442695040888963407ull;
    return (uint32_t)(g_state >> 32);
}

/* A random binary16 bit pattern of magnitude in [2^-4, 2): sign, biased
 * exponent 11..15, any mantissa. */
static uint16_t random_half(void) {
    const uint32_t r = next_u32();
    const uint32_t sign = r >> 31;
    const uint32_t expo = 11u + (r >> 16) % 5u;
    const uint32_t mant = r & 0x3ffu;
    return (uint16_t)((sign << 15) | (expo << 10) | mant);
}

static void fill_halves(uint16_t *p, size_t n) {
    for (size_t i = 0; i < n; ++i) p[i] = random_half();
}

#define CUDA_OK(call)                                                              \
    do {                                                                           \
        const cudaError_t e_ = (call);                                             \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));            \
            exit(1);                                                               \
        }                                                                          \
    } while (0)

#define PKV_OK_OR_DIE(call)                                                        \
    do {                                                                           \
        const int s_ = (call);                                                     \
        if (s_ != PKV_OK) {                                                        \
            fprintf(stderr, "%s: %s\n", #call, paged_kv_status_string(s_));        \
            exit(1);                                                               \
        }                                                                          \
    } while (0)

static void *to_device(const void *host, size_t bytes) {
    void *dev = NULL;
    CUDA_OK(cudaMalloc(&dev, bytes));
    CUDA_OK(cudaMemcpy(dev, host, bytes, cudaMemcpyHostToDevice));
    return dev;
}

static void write_block(FILE *f, const void *p, size_t bytes) {
    if (fwrite(p, 1, bytes, f) != bytes) {
        fprintf(stderr, "short write\n");
        exit(1);
    }
}

int main(int argc, char **argv) {
    if (argc != 2) {
        fprintf(stderr, "usage: %s OUTPUT_FILE\n", argv[0]);
        return 2;
    }
    /* block tables: the pool's blocks in shuffled order, handed out in turn */
    int used = 0;
    for (int b = 0; b < B; ++b) used += (kLens[b] + BS - 1) / BS;
    const int num_blocks = used + SPARE_BLOCKS;
    int *perm = malloc(sizeof(int) * (size_t)num_blocks);
    if (!perm) return 1;
    for (int i = 0; i < num_blocks; ++i) perm[i] = i;
    for (int i = num_blocks - 1; i > 0; --i) { /* Fisher-Yates */
        const int j = (int)(next_u32() % (uint32_t)(i + 1));
        const int t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
    }
    int32_t tables[B * MB];
    int32_t lens[B];
    int64_t slots[B];
    for (int b = 0, next = 0; b < B; ++b) {
        lens[b] = kLens[b];
        const int nb = (kLens[b] + BS - 1) / BS;
        for (int i = 0; i < MB; ++i)  /* entries past the length are never read */
            tables[b * MB + i] = i < nb ? perm[next + i] : INT32_MAX;
        next += nb;
        const int t = kLens[b] - 1; /* the newest token: it is appended this step */
        slots[b] = (int64_t)tables[b * MB + t / BS] * BS + t % BS;
    }
    free(perm);

    const size_t cache_n = (size_t)num_blocks * HK * BS * D;
    uint16_t *k_cache = malloc(cache_n * 2), *v_cache = malloc(cache_n * 2);
    if (!k_cache || !v_cache) return 1;
    uint16_t q[B * H * D], k_new[B * HK * D], v_new[B * HK * D];
    fill_halves(k_cache, cache_n);
    fill_halves(v_cache, cache_n);
    fill_halves(q, B * H * D);
    fill_halves(k_new, B * HK * D);
    fill_halves(v_new, B * HK * D);

    CUDA_OK(cudaSetDevice(0));
    cudaStream_t stream;
    CUDA_OK(cudaStreamCreate(&stream));
    void *d_kc = to_device(k_cache, cache_n * 2), *d_vc = to_device(v_cache, cache_n * 2);
    void *d_q = to_device(q, sizeof q), *d_kn = to_device(k_new, sizeof k_new);
    void *d_vn = to_device(v_new, sizeof v_new);
    int32_t *d_bt = to_device(tables, sizeof tables);
    int32_t *d_cl = to_device(lens, sizeof lens);
    int64_t *d_sm = to_device(slots, sizeof slots);
    void *d_out = NULL;
    float *d_lse = NULL;
    int32_t *d_err = NULL;
    CUDA_OK(cudaMalloc(&d_out, sizeof(uint16_t) * B * H * D));
    CUDA_OK(cudaMalloc((void **)&d_lse, sizeof(float) * B * H));
    CUDA_OK(cudaMalloc((void **)&d_err, sizeof(int32_t)));
    CUDA_OK(cudaMemset(d_err, 0, sizeof(int32_t)));

    int partition = -1;
    size_t ws_bytes = 0;
    PKV_OK_OR_DIE(paged_decode_plan(B, H, HK, D, BS, MB, MAX_LEN, 0, &partition, &ws_bytes));
    void *d_ws = NULL;
    if (ws_bytes > 0) CUDA_OK(cudaMalloc(&d_ws, ws_bytes));
    PKV_OK_OR_DIE(paged_decode_workspace_clear(d_ws, ws_bytes, stream));
    const float scale = 1.0f / sqrtf((float)D);
    PKV_OK_OR_DIE(paged_decode_step_ex(d_kn, d_vn, d_sm, B, d_out, d_q, d_kc, d_vc, d_bt, d_cl,
                                       B, MB, num_blocks, scale, H, HK, D, BS, MAX_LEN, 0, d_ws,
                                       ws_bytes, d_lse, d_err, stream, PKV_APPEND_NEWEST));
    int32_t bits = -1;
    const int status = paged_kv_get_error(d_err, stream, &bits);
    if (status != PKV_OK && status != PKV_ERR_INDEX) PKV_OK_OR_DIE(status);

    uint16_t out[B * H * D];
    float lse[B * H];
    CUDA_OK(cudaMemcpy(out, d_out, sizeof out, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(lse, d_lse, sizeof lse, cudaMemcpyDeviceToHost));

    /* write_all: int32 header {B, H, HK, D, BS, num_blocks, MB, partition,
     * error bits}, then context_lens int32[B], block_tables int32[B][MB],
     * slot_mapping int64[B], q fp16[B][H][D], k_new and v_new fp16[B][HK][D],
     * k_cache and v_cache before the step fp16[num_blocks][HK][BS][D],
     * out fp16[B][H][D], lse fp32[B][H]. */
    FILE *f = fopen(argv[1], "wb");
    if (!f) {
        perror(argv[1]);
        return 1;
    }
    const int32_t header[9] = {B, H, HK, D, BS, num_blocks, MB, partition, bits};
    write_block(f, header, sizeof header);
    write_block(f, lens, sizeof lens);
    write_block(f, tables, sizeof tables);
    write_block(f, slots, sizeof slots);
    write_block(f, q, sizeof q);
    write_block(f, k_new, sizeof k_new);
    write_block(f, v_new, sizeof v_new);
    write_block(f, k_cache, cache_n * 2);
    write_block(f, v_cache, cache_n * 2);
    write_block(f, out, sizeof out);
    write_block(f, lse, sizeof lse);
    fclose(f);

    cudaFree(d_kc);
    cudaFree(d_vc);
    cudaFree(d_q);
    cudaFree(d_kn);
    cudaFree(d_vn);
    cudaFree(d_bt);
    cudaFree(d_cl);
    cudaFree(d_sm);
    cudaFree(d_out);
    cudaFree(d_lse);
    cudaFree(d_err);
    cudaFree(d_ws);
    cudaStreamDestroy(stream);
    free(k_cache);
    free(v_cache);
    printf("decode step: partition_tokens %d, workspace %zu bytes, error bits %d\n", partition,
           ws_bytes, (int)bits);
    return bits == 0 ? 0 : 1;
}
