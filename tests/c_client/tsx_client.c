/* A plain C client of libtsx: the C ABI used without Python.
 *
 * It checks, through include/tsx.h alone:
 *   1. host-side errors come back as status codes with a message (NULL
 *      plan, unknown dtype, zero box, unknown op);
 *   2. tsx_plan_query plans without a GPU;
 *   3. on a GPU, an fp32 fma over a ragged [rows, cols] tensor equals the C
 *      library's fmaf element by element (fmaf rounds a * b + c once, as
 *      the operation is defined), and the plan's status stays TSX_OK;
 *   4. tsx_ewise_noalloc gives the same bits, and so does the launch shape
 *      tsx_plan_tune keeps;
 *   5. row sums of small integers are exact.
 *
 * Usage: tsx_client [--no-gpu].  Prints one line per check and exits 0 when
 * every check passed. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "tsx.h"

static int failures = 0;

static void check(int ok, const char* what)
{
    printf("%s %s\n", ok ? "ok  " : "FAIL", what);
    if (!ok)
        failures++;
}

/* SplitMix64, for reproducible inputs */
static uint64_t mix(uint64_t x)
{
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

static float uniform(uint64_t i, float lo, float hi)
{
    return lo + (hi - lo) * (float)(mix(i) >> 40) * (1.0f / 16777216.0f);
}

static void host_checks(void)
{
    tsx_plan_info info;
    check(tsx_plan_status(NULL) == TSX_ERR_INVALID && strlen(tsx_last_error()) > 0, "NULL plan is an error");
    check(tsx_ewise(NULL, TSX_ADD, NULL, NULL, NULL, NULL, NULL) == TSX_ERR_INVALID, "tsx_ewise on NULL plan");
    check(tsx_plan_query((tsx_dtype)7, 16, 16, 8, 16, 2, TSX_TMA, TSX_COPY, &info) != TSX_OK, "unknown dtype");
    check(tsx_plan_query(TSX_F32, 16, 16, 0, 16, 2, TSX_TMA, TSX_COPY, &info) == TSX_ERR_UNSUPPORTED, "zero box");
    check(tsx_plan_query(TSX_F32, 16, 16, 8, 16, 2, TSX_TMA, (tsx_op)9, &info) == TSX_ERR_INVALID, "unknown op");
    check(tsx_plan_query(TSX_F32, 128, 1 << 20, 8, 128, 4, TSX_TMA, TSX_FMA, &info) == TSX_OK &&
              info.loads_per_operand == 4 && info.tx_bytes == 12288,
          "query: 8x128 fp32 fma tile = 4 loads per operand, expect_tx 12288");
}

static void gpu_checks(void)
{
    const int64_t rows = 37, cols = 1000;   /* ragged against an 8x128 tile */
    const size_t n = (size_t)(rows * cols), bytes = n * sizeof(float);
    float *h[4], *d[4];
    for (int k = 0; k < 4; ++k) {
        h[k] = (float*)malloc(bytes);
        if (cudaMalloc((void**)&d[k], bytes) != cudaSuccess) {
            check(0, "cudaMalloc");
            return;
        }
    }
    for (size_t i = 0; i < n; ++i) {
        h[0][i] = uniform(3 * i, -2.f, 2.f);
        h[1][i] = uniform(3 * i + 1, -2.f, 2.f);
        h[2][i] = uniform(3 * i + 2, -2.f, 2.f);
    }
    for (int k = 0; k < 3; ++k)
        cudaMemcpy(d[k], h[k], bytes, cudaMemcpyHostToDevice);
    tsx_plan_t plan = tsx_plan_create(TSX_F32, rows, cols, 8, 128, 4, TSX_TMA);
    check(plan != NULL, "tsx_plan_create");
    if (!plan)
        return;
    check(tsx_ewise(plan, TSX_FMA, d[0], d[1], d[2], d[3], NULL) == TSX_OK, "tsx_ewise fma");
    check(tsx_ewise(plan, TSX_FMA, d[0], NULL, d[2], d[3], NULL) == TSX_ERR_INVALID, "fma without b is an error");
    cudaDeviceSynchronize();
    check(tsx_plan_status(plan) == TSX_OK, "device status");
    cudaMemcpy(h[3], d[3], bytes, cudaMemcpyDeviceToHost);
    size_t bad = 0;
    for (size_t i = 0; i < n; ++i) {
        const float want = fmaf(h[0][i], h[1][i], h[2][i]);
        if (memcmp(&want, &h[3][i], sizeof want) != 0)
            bad++;
    }
    check(bad == 0, "fma equals fmaf bit for bit");

    /* the allocation-free entry point gives the same bits */
    float* h_na = (float*)malloc(bytes);
    int status = -100;
    check(tsx_ewise_noalloc(TSX_F32, rows, cols, 8, 128, 4, TSX_TMA, TSX_FMA, d[0], d[1], d[2], d[3], NULL,
                            &status) == TSX_OK && status == TSX_OK,
          "tsx_ewise_noalloc");
    cudaMemcpy(h_na, d[3], bytes, cudaMemcpyDeviceToHost);
    check(memcmp(h_na, h[3], bytes) == 0, "noalloc equals tsx_ewise bit for bit");

    /* the launch shape tsx_plan_tune keeps gives the same bits */
    tsx_plan_info chosen;
    memset(&chosen, 0, sizeof chosen);
    cudaMemset(d[3], 0xA5, bytes);
    check(tsx_plan_tune(plan, TSX_FMA, d[0], d[1], d[2], d[3], NULL, 2, &chosen) == TSX_OK && chosen.ctas_per_sm >= 1,
          "tsx_plan_tune");
    cudaMemset(d[3], 0x5A, bytes);
    check(tsx_ewise(plan, TSX_FMA, d[0], d[1], d[2], d[3], NULL) == TSX_OK, "tsx_ewise after tuning");
    cudaMemcpy(h_na, d[3], bytes, cudaMemcpyDeviceToHost);
    check(memcmp(h_na, h[3], bytes) == 0, "tuned launch equals the planner's bit for bit");
    check(tsx_plan_tune(plan, TSX_FMA, d[3], d[1], d[2], d[3], NULL, 2, NULL) == TSX_ERR_INVALID,
          "tuning with out aliasing an input is an error");
    free(h_na);

    /* row sums of small integers are exact in fp32 whatever the order */
    for (size_t i = 0; i < n; ++i)
        h[0][i] = (float)((int)(mix(7 * i) % 129) - 64);
    cudaMemcpy(d[0], h[0], bytes, cudaMemcpyHostToDevice);
    float* d_sums = NULL;
    float h_sums[37];
    cudaMalloc((void**)&d_sums, sizeof h_sums);
    check(tsx_reduce_rows(plan, TSX_COPY, d[0], NULL, NULL, d_sums, NULL) == TSX_OK, "tsx_reduce_rows");
    cudaDeviceSynchronize();
    check(tsx_plan_status(plan) == TSX_OK, "device status after row sums");
    cudaMemcpy(h_sums, d_sums, sizeof h_sums, cudaMemcpyDeviceToHost);
    int exact = 1;
    for (int64_t r = 0; r < rows; ++r) {
        double want = 0;
        for (int64_t c = 0; c < cols; ++c)
            want += h[0][r * cols + c];
        exact &= (double)h_sums[r] == want;
    }
    check(exact, "integer row sums exact");
    cudaFree(d_sums);
    tsx_plan_destroy(plan);
    tsx_plan_destroy(NULL);
    for (int k = 0; k < 4; ++k) {
        cudaFree(d[k]);
        free(h[k]);
    }
}

int main(int argc, char** argv)
{
    host_checks();
    if (!(argc > 1 && strcmp(argv[1], "--no-gpu") == 0))
        gpu_checks();
    printf("%d failure(s)\n", failures);
    return failures ? 1 : 0;
}
