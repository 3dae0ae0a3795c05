/*
 * A plain C caller of librope_qk.so: the usage the header documents, compiled with gcc
 * and linked with -lrope_qk -lcudart, no Python anywhere.
 *
 *     rope_c_caller <input file> <output file>
 *
 * Input (little-endian): int32 T, n_q_heads, n_kv_heads, head_dim, n_seqs; float64
 * theta; int32 cu_seqlens[n_seqs + 1]; bf16 Q[T][n_q_heads][head_dim]; bf16
 * K[T][n_kv_heads][head_dim].
 *
 * It allocates device memory with cudaMalloc, copies each buffer in with one
 * cudaMemcpyAsync, builds a cos/sin cache of the longest sample's rows, runs the
 * forward rotation in place with the cache (rope_qk_fwd) and copies Q and K out, then
 * the backward rotation in place without a cache (rope_qk_bwd, cos/sin evaluated on
 * the fly) on the rotated Q and K and copies them out again.  Output: bf16 fwd Q, fwd
 * K, bwd Q, bwd K, one after the other.  Exit status 0 on success; a library status is
 * printed with rope_strerror.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "rope_qk.h"

#define CUDA_OK(call)                                                              \
    do {                                                                           \
        cudaError_t e_ = (call);                                                   \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));            \
            return 2;                                                              \
        }                                                                          \
    } while (0)

#define ROPE_OK_OR_FAIL(call)                                                      \
    do {                                                                           \
        int st_ = (call);                                                          \
        if (st_ != ROPE_OK) {                                                      \
            fprintf(stderr, "%s: %s\n", #call, rope_strerror(st_));                \
            return 3;                                                              \
        }                                                                          \
    } while (0)

static int read_exact(FILE *f, void *p, size_t n)
{
    return fread(p, 1, n, f) == n ? 0 : -1;
}

int main(int argc, char **argv)
{
    if (argc != 3) {
        fprintf(stderr, "usage: %s <input> <output>\n", argv[0]);
        return 1;
    }
    FILE *in = fopen(argv[1], "rb");
    if (in == NULL) return 1;
    int32_t hdr[5];
    double theta;
    if (read_exact(in, hdr, sizeof hdr) || read_exact(in, &theta, sizeof theta)) return 1;
    const int32_t T = hdr[0], hq = hdr[1], hkv = hdr[2], d = hdr[3], n = hdr[4];
    if (T < 0 || hq < 1 || hkv < 1 || n < 0) return 1;
    const size_t cu_bytes = (size_t)(n + 1) * sizeof(int32_t);
    const size_t q_bytes = (size_t)T * hq * d * 2, k_bytes = (size_t)T * hkv * d * 2;
    int32_t *cu = malloc(cu_bytes);
    unsigned char *q = malloc(q_bytes), *k = malloc(k_bytes);
    if (!cu || !q || !k) return 1;
    if (read_exact(in, cu, cu_bytes) || read_exact(in, q, q_bytes) || read_exact(in, k, k_bytes)) return 1;
    fclose(in);
    int32_t max_len = 1;
    for (int32_t s = 0; s < n; ++s)
        if (cu[s + 1] - cu[s] > max_len) max_len = cu[s + 1] - cu[s];

    printf("rope_qk ABI %d (header %d)\n", rope_qk_abi_version(), ROPE_QK_ABI_VERSION);
    if (rope_qk_abi_version() != ROPE_QK_ABI_VERSION) return 4;

    cudaStream_t stream;
    CUDA_OK(cudaStreamCreate(&stream));
    void *dq, *dk, *dcu;
    float *cache_data;
    CUDA_OK(cudaMalloc(&dq, q_bytes));
    CUDA_OK(cudaMalloc(&dk, k_bytes));
    CUDA_OK(cudaMalloc(&dcu, cu_bytes));
    CUDA_OK(cudaMalloc((void **)&cache_data, (size_t)rope_cos_sin_cache_bytes(max_len, d)));
    CUDA_OK(cudaMemcpyAsync(dq, q, q_bytes, cudaMemcpyHostToDevice, stream));
    CUDA_OK(cudaMemcpyAsync(dk, k, k_bytes, cudaMemcpyHostToDevice, stream));
    CUDA_OK(cudaMemcpyAsync(dcu, cu, cu_bytes, cudaMemcpyHostToDevice, stream));

    /* once per (theta, head_dim): the cache and its descriptor */
    rope_cos_sin_cache cache;
    ROPE_OK_OR_FAIL(rope_cos_sin_cache_build(&cache, cache_data, max_len, d, theta, 1.0, stream));

    /* forward, in place, reading cos/sin from the cache */
    ROPE_OK_OR_FAIL(rope_qk_fwd(dq, dk, dcu, n, T, hq, hkv, d, theta, 1, NULL, NULL, &cache, stream));
    FILE *out = fopen(argv[2], "wb");
    if (out == NULL) return 1;
    CUDA_OK(cudaMemcpyAsync(q, dq, q_bytes, cudaMemcpyDeviceToHost, stream));
    CUDA_OK(cudaMemcpyAsync(k, dk, k_bytes, cudaMemcpyDeviceToHost, stream));
    CUDA_OK(cudaStreamSynchronize(stream));
    fwrite(q, 1, q_bytes, out);
    fwrite(k, 1, k_bytes, out);

    /* backward (transpose rotation), in place, cos/sin evaluated on the fly */
    ROPE_OK_OR_FAIL(rope_qk_bwd(dq, dk, dcu, n, T, hq, hkv, d, theta, 1, NULL, NULL, NULL, stream));
    CUDA_OK(cudaMemcpyAsync(q, dq, q_bytes, cudaMemcpyDeviceToHost, stream));
    CUDA_OK(cudaMemcpyAsync(k, dk, k_bytes, cudaMemcpyDeviceToHost, stream));
    CUDA_OK(cudaStreamSynchronize(stream));
    fwrite(q, 1, q_bytes, out);
    fwrite(k, 1, k_bytes, out);
    fclose(out);

    /* a cache built for another theta is refused */
    const int st = rope_qk_fwd(dq, dk, dcu, n, T, hq, hkv, d, theta * 2.0, 1, NULL, NULL, &cache, stream);
    printf("mismatched cache: %s\n", rope_strerror(st));
    if (st != ROPE_ERR_CACHE) return 5;

    CUDA_OK(cudaFree(dq));
    CUDA_OK(cudaFree(dk));
    CUDA_OK(cudaFree(dcu));
    CUDA_OK(cudaFree(cache_data));
    CUDA_OK(cudaStreamDestroy(stream));
    free(cu);
    free(q);
    free(k);
    printf("ok\n");
    return 0;
}
