/* Test program (not part of the library): a plain C caller of libzero.
 *
 * Only include/zero.h, libzero.so and the CUDA runtime: it lays out a buffer,
 * allocates every device buffer itself (cudaMalloc), loads the fp32 master and
 * the 16-bit gradient replicas from files, initialises the step state and the
 * 16-bit parameters, runs `steps` whole steps with zero_step (ZeRO-2, bf16, no
 * clipping: the fused path) and writes the resulting master, m, v, every
 * parameter replica and the 96-byte state to files, for the test to compare
 * with the oracle.
 *
 * usage: c_step DIR N_D N_TENSORS NUMEL... STEPS
 *   DIR/master.bin   Psi_pad fp32 values (zero padding)
 *   DIR/grads.bin    N_D x Psi_pad 16-bit gradients, rank-major (one set, used every step)
 * writes DIR/out_master.bin, out_m.bin, out_v.bin (flat order), out_params.bin
 * (N_D x Psi_pad), out_state.bin. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "zero.h"

#define CK(x)                                                                          \
    do {                                                                               \
        cudaError_t e_ = (x);                                                          \
        if (e_ != cudaSuccess) {                                                       \
            fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
            return 2;                                                                  \
        }                                                                              \
    } while (0)
#define ZK(x)                                                                         \
    do {                                                                              \
        zero_status_t s_ = (x);                                                       \
        if (s_ != ZERO_OK) {                                                          \
            fprintf(stderr, "%s:%d status %d: %s\n", __FILE__, __LINE__, (int)s_,     \
                    zero_last_error());                                               \
            return 3;                                                                 \
        }                                                                             \
    } while (0)

static int read_file(const char* dir, const char* name, void* dst, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "rb");
    if (!f) return 1;
    size_t n = fread(dst, 1, bytes, f);
    fclose(f);
    return n == bytes ? 0 : 1;
}

static int write_file(const char* dir, const char* name, const void* src, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "wb");
    if (!f) return 1;
    size_t n = fwrite(src, 1, bytes, f);
    fclose(f);
    return n == bytes ? 0 : 1;
}

int main(int argc, char** argv) {
    if (argc < 5) return 1;
    const char* dir = argv[1];
    const int nd = atoi(argv[2]);
    const int nt = atoi(argv[3]);
    if (nd < 1 || nd > ZERO_MAX_RANKS || nt < 1 || argc != 5 + nt) return 1;
    int64_t* numels = (int64_t*)malloc(sizeof(int64_t) * (size_t)nt);
    for (int t = 0; t < nt; ++t) numels[t] = atoll(argv[4 + t]);
    const int steps = atoi(argv[4 + nt]);

    zero_layout* L = NULL;
    ZK(zero_layout_init(numels, nt, NULL, nd, 2, 0, 0, ZERO_BF16, &L));
    zero_layout_info info;
    ZK(zero_layout_query(L, &info));
    const int64_t P = info.psi_pad, S = info.shard_len;

    /* device buffers: one allocation per kind, rank-major rows (rows stay 256-byte aligned) */
    float *master, *m, *v;
    uint16_t *grads, *params;
    void *workspace, *state;
    CK(cudaMalloc((void**)&master, sizeof(float) * (size_t)(nd * S)));
    CK(cudaMalloc((void**)&m, sizeof(float) * (size_t)(nd * S)));
    CK(cudaMalloc((void**)&v, sizeof(float) * (size_t)(nd * S)));
    CK(cudaMalloc((void**)&grads, sizeof(uint16_t) * (size_t)(nd * P)));
    CK(cudaMalloc((void**)&params, sizeof(uint16_t) * (size_t)(nd * P)));
    CK(cudaMalloc(&workspace, (size_t)info.workspace_bytes));
    CK(cudaMalloc(&state, sizeof(zero_step_state)));
    CK(cudaMemset(m, 0, sizeof(float) * (size_t)(nd * S)));
    CK(cudaMemset(v, 0, sizeof(float) * (size_t)(nd * S)));

    /* inputs: rank r's shard of the flat master is flat range [r*S, (r+1)*S) (one unit) */
    float* hm = (float*)malloc(sizeof(float) * (size_t)P);
    uint16_t* hg = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(nd * P));
    if (read_file(dir, "master.bin", hm, sizeof(float) * (size_t)P)) return 4;
    if (read_file(dir, "grads.bin", hg, sizeof(uint16_t) * (size_t)(nd * P))) return 4;
    CK(cudaMemcpy(master, hm, sizeof(float) * (size_t)P, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(grads, hg, sizeof(uint16_t) * (size_t)(nd * P), cudaMemcpyHostToDevice));

    const void* grad_rows[ZERO_MAX_RANKS];
    float *master_rows[ZERO_MAX_RANKS], *m_rows[ZERO_MAX_RANKS], *v_rows[ZERO_MAX_RANKS];
    void* param_rows[ZERO_MAX_RANKS];
    for (int r = 0; r < nd; ++r) {
        grad_rows[r] = grads + (size_t)r * (size_t)P;
        master_rows[r] = master + (size_t)r * (size_t)S;
        m_rows[r] = m + (size_t)r * (size_t)S;
        v_rows[r] = v + (size_t)r * (size_t)S;
        param_rows[r] = params + (size_t)r * (size_t)P;
    }
    zero_adamw_hp hp = {1e-3, 1e-8, 0.01};
    ZK(zero_state_init((zero_step_state*)state, 0.9, 0.999, 1.0f, 0, 2000, NULL));
    ZK(zero_cast_params(L, (const float* const*)master_rows, param_rows, ZERO_OUT_FULL_REPLICAS, NULL));

    zero_step_args a;
    memset(&a, 0, sizeof a);
    a.hp = &hp;
    a.max_norm = 0.0;
    a.fused = 1;
    a.per_bucket = 1;
    a.grad_replicas = grad_rows;
    a.master = master_rows;
    a.m = m_rows;
    a.v = v_rows;
    a.param16_full = param_rows;
    a.state = (zero_step_state*)state;
    a.workspace = workspace;
    for (int s = 0; s < steps; ++s) ZK(zero_step(L, &a, NULL));
    CK(cudaDeviceSynchronize());

    float* out = (float*)malloc(sizeof(float) * (size_t)P);
    float* bufs[3] = {master, m, v};
    const char* names[3] = {"out_master.bin", "out_m.bin", "out_v.bin"};
    for (int k = 0; k < 3; ++k) {
        CK(cudaMemcpy(out, bufs[k], sizeof(float) * (size_t)P, cudaMemcpyDeviceToHost));
        if (write_file(dir, names[k], out, sizeof(float) * (size_t)P)) return 5;
    }
    CK(cudaMemcpy(hg, params, sizeof(uint16_t) * (size_t)(nd * P), cudaMemcpyDeviceToHost));
    if (write_file(dir, "out_params.bin", hg, sizeof(uint16_t) * (size_t)(nd * P))) return 5;
    zero_step_state st;
    CK(cudaMemcpy(&st, state, sizeof st, cudaMemcpyDeviceToHost));
    if (write_file(dir, "out_state.bin", &st, sizeof st)) return 5;
    printf("c_step ok: t=%d norm=%.9e launches=%lld\n", st.t, st.grad_norm, (long long)zero_launch_count(0));
    zero_layout_destroy(L);
    cudaFree(master);
    cudaFree(m);
    cudaFree(v);
    cudaFree(grads);
    cudaFree(params);
    cudaFree(workspace);
    cudaFree(state);
    free(numels);
    free(hm);
    free(hg);
    free(out);
    return 0;
}
