/*
 * A C user of liblce: loads H, W (bf16 bits) and targets from binary files,
 * calls lce_forward_backward through the C ABI on device memory it allocates
 * itself, reads the device status word, and writes loss, dH and dW back to
 * files. No Python, no torch; the test that runs it compares the outputs with
 * the fp64 oracle.
 *
 * usage: lce_client DIR N d V ignore_index
 *   DIR/H.bin  N*d uint16 (bf16)   DIR/W.bin  V*d uint16   DIR/t.bin  N int64
 *   -> DIR/loss.bin float32, DIR/dH.bin N*d uint16, DIR/dW.bin V*d float32
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "lce.h"

static void *load(const char *dir, const char *name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) return NULL;
    void *p = malloc(bytes);
    if (p && fread(p, 1, bytes, f) != bytes) {
        free(p);
        p = NULL;
    }
    fclose(f);
    return p;
}

static int save(const char *dir, const char *name, const void *p, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "wb");
    if (!f) return 1;
    int bad = fwrite(p, 1, bytes, f) != bytes;
    fclose(f);
    return bad;
}

#define CK(x)                                                         \
    do {                                                              \
        cudaError_t e_ = (x);                                         \
        if (e_ != cudaSuccess) {                                      \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));  \
            return 2;                                                 \
        }                                                             \
    } while (0)

int main(int argc, char **argv) {
    if (argc != 6) {
        fprintf(stderr, "usage: %s DIR N d V ignore_index\n", argv[0]);
        return 2;
    }
    const char *dir = argv[1];
    const int64_t N = atoll(argv[2]), d = atoll(argv[3]), V = atoll(argv[4]), ignore = atoll(argv[5]);
    const size_t hb = (size_t)N * d * 2, wb = (size_t)V * d * 2, tb = (size_t)N * 8;
    void *H = load(dir, "H.bin", hb), *W = load(dir, "W.bin", wb), *t = load(dir, "t.bin", tb);
    if (!H || !W || !t) {
        fprintf(stderr, "cannot read inputs\n");
        return 2;
    }
    void *dH_dev, *H_dev, *W_dev, *t_dev;
    float *dW_dev, *loss_dev;
    CK(cudaMalloc(&H_dev, hb));
    CK(cudaMalloc(&W_dev, wb));
    CK(cudaMalloc(&t_dev, tb));
    CK(cudaMalloc(&dH_dev, hb));
    CK(cudaMalloc((void **)&dW_dev, (size_t)V * d * 4));
    CK(cudaMalloc((void **)&loss_dev, 4));
    CK(cudaMemcpy(H_dev, H, hb, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(W_dev, W, wb, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(t_dev, t, tb, cudaMemcpyHostToDevice));

    lce_status_t s = lce_forward_backward(H_dev, W_dev, (const int64_t *)t_dev, ignore, N, d, V, loss_dev, dH_dev,
                                          dW_dev, NULL);
    if (s != LCE_OK) {
        fprintf(stderr, "lce_forward_backward: %s\n", lce_status_string(s));
        return 1;
    }
    int32_t bits = 0;
    s = lce_get_device_status(NULL, &bits);
    if (s != LCE_OK) {
        fprintf(stderr, "device status: %s (bits %d)\n", lce_status_string(s), bits);
        return 1;
    }
    float loss = 0.f;
    void *dH = malloc(hb), *dW = malloc((size_t)V * d * 4);
    CK(cudaMemcpy(&loss, loss_dev, 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(dH, dH_dev, hb, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(dW, dW_dev, (size_t)V * d * 4, cudaMemcpyDeviceToHost));
    if (save(dir, "loss.bin", &loss, 4) || save(dir, "dH.bin", dH, hb) || save(dir, "dW.bin", dW, (size_t)V * d * 4))
        return 2;
    printf("loss %.7f launches %lld version %d\n", loss, (long long)lce_launch_count(), lce_version());
    return 0;
}
