/*
 * A plain C99 consumer of the vt_attn C ABI (include/vt_attn.h), built with gcc and linked
 * against libvt_attn.so by tests/test_c_abi.py.
 *
 * Without VT_WITH_CUDA it checks, on any machine, that the documented argument errors come
 * back before anything touches a GPU.  With VT_WITH_CUDA (a GPU machine) it also runs one
 * forward on device memory from the CUDA runtime and checks the closed form V == 1 => O == 1
 * (the softmax weights of every row sum to one; bf16 rounding of P and O keeps each output
 * within 2^-7 of 1).
 *
 * Exit status 0 on success; on failure a message on stderr and a non-zero status.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "vt_attn.h"

#ifdef VT_WITH_CUDA
#include <cuda_runtime_api.h>
#endif

static int failures = 0;

static void expect(const char *what, vt_status got, vt_status want) {
    if (got != want) {
        fprintf(stderr, "%s: got %d (%s), want %d\n", what, (int)got, vt_status_str(got), (int)want);
        ++failures;
    }
}

/* Argument checks: none of these reaches a launch. */
static void host_checks(void) {
    /* distinct, 16-byte aligned addresses that are never dereferenced */
    void *q = (void *)(uintptr_t)0x100000, *k = (void *)(uintptr_t)0x200000;
    void *v = (void *)(uintptr_t)0x300000, *o = (void *)(uintptr_t)0x400000;
    expect("S_k = 0", vt_attn_fwd(q, k, v, o, 1, 1, 4, 0, 8, 8, 0.5f, 0, VT_BF16, NULL), VT_ERR_INVALID_ARG);
    expect("D_qk > 128", vt_attn_fwd(q, k, v, o, 1, 1, 4, 4, 129, 8, 0.5f, 0, VT_BF16, NULL), VT_ERR_UNSUPPORTED);
    expect("misaligned Q", vt_attn_fwd((char *)q + 8, k, v, o, 1, 1, 4, 4, 8, 8, 0.5f, 0, VT_BF16, NULL),
           VT_ERR_MISALIGNED);
    expect("O overlaps Q", vt_attn_fwd(q, k, v, (char *)q + 32, 1, 1, 4, 4, 8, 8, 0.5f, 1, VT_BF16, NULL),
           VT_ERR_INVALID_ARG);
    expect("empty problem", vt_attn_fwd(q, k, v, o, 0, 1, 4, 4, 8, 8, 0.5f, 0, VT_F32, NULL), VT_OK);
    {
        const int64_t st[3] = {4 * 4 * 8, 4 * 8, 8};
        const int64_t skv[3] = {2 * 4 * 8, 4 * 8, 8};
        vt_attn_mask m;
        memset(&m, 0, sizeof m);
        m.kind = VT_MASK_WINDOW;
        m.window = 0; /* a window kind needs window >= 1 */
        expect("window 0", vt_attn_fwd_general(q, st, k, skv, v, skv, o, st, NULL, 1, 4, 2, 4, 4, 8, 8, 0.5f, VT_BF16,
                                               &m, 1, NULL, 0, NULL, NULL),
               VT_ERR_INVALID_ARG);
        m.window = 2;
        expect("H not a multiple of H_kv", vt_attn_fwd_general(q, st, k, skv, v, skv, o, st, NULL, 1, 4, 3, 4, 4, 8, 8,
                                                               0.5f, VT_BF16, &m, 1, NULL, 0, NULL, NULL),
               VT_ERR_INVALID_ARG);
    }
    if (vt_attn_splitkv_workspace_size(2, 3, 5, 8, 1) != 0) {
        fprintf(stderr, "workspace size for n_split = 1 should be 0\n");
        ++failures;
    }
    if (strcmp(vt_status_str(VT_OK), "VT_OK") != 0) {
        fprintf(stderr, "vt_status_str(VT_OK) = %s\n", vt_status_str(VT_OK));
        ++failures;
    }
}

#ifdef VT_WITH_CUDA
/* bf16 bits of a float, round to nearest even (inputs here are finite) */
static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

static float from_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static void gpu_ones(void) {
    enum { B = 2, H = 3, S_Q = 300, S_K = 333, D = 64 };
    const size_t nq = (size_t)B * H * S_Q * D, nk = (size_t)B * H * S_K * D;
    static uint16_t hq[(size_t)B * H * S_Q * D], hk[(size_t)B * H * S_K * D], hv[(size_t)B * H * S_K * D];
    static uint16_t ho[(size_t)B * H * S_Q * D];
    uint32_t x = 12345u;
    for (size_t i = 0; i < nq; ++i) {
        x = x * 1664525u + 1013904223u;
        hq[i] = to_bf16(((float)(x >> 8) / 16777216.0f) * 4.0f - 2.0f);
    }
    for (size_t i = 0; i < nk; ++i) {
        x = x * 1664525u + 1013904223u;
        hk[i] = to_bf16(((float)(x >> 8) / 16777216.0f) * 4.0f - 2.0f);
        hv[i] = to_bf16(1.0f);
    }
    void *dq = NULL, *dk = NULL, *dv = NULL, *dO = NULL;
    if (cudaMalloc(&dq, nq * 2) || cudaMalloc(&dk, nk * 2) || cudaMalloc(&dv, nk * 2) || cudaMalloc(&dO, nq * 2)) {
        fprintf(stderr, "cudaMalloc failed\n");
        ++failures;
        return;
    }
    cudaMemcpy(dq, hq, nq * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(dk, hk, nk * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(dv, hv, nk * 2, cudaMemcpyHostToDevice);
    for (int causal = 0; causal < 2; ++causal) {
        expect("vt_attn_fwd", vt_attn_fwd(dq, dk, dv, dO, B, H, S_Q, S_K, D, D, 0.125f, causal, VT_BF16, NULL), VT_OK);
        expect("device status", vt_last_device_status(NULL), VT_OK);
        cudaMemcpy(ho, dO, nq * 2, cudaMemcpyDeviceToHost);
        for (size_t i = 0; i < nq; ++i) {
            const float d = from_bf16(ho[i]) - 1.0f;
            if (d > 1.0f / 128 || d < -1.0f / 128) {
                fprintf(stderr, "causal=%d: O[%zu] = %g, want 1\n", causal, i, (double)from_bf16(ho[i]));
                ++failures;
                break;
            }
        }
    }
    cudaFree(dq);
    cudaFree(dk);
    cudaFree(dv);
    cudaFree(dO);
}
#endif

int main(void) {
    host_checks();
#ifdef VT_WITH_CUDA
    gpu_ones();
#endif
    if (failures) {
        fprintf(stderr, "%d check(s) failed\n", failures);
        return 1;
    }
    return 0;
}
