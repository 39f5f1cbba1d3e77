/*
 * Oracle (test infrastructure only): fp32 router logits of a dropless MoE layer.
 *
 * Source: "Accelerating dropless MoE training in JAX with NVIDIA Transformer
 * Engine", introduction: a learned router scores every expert for every
 * token and the Top-K experts are activated;
 * section "What are the challenges of MoE training?": the router is a learned
 * component.  The page fixes no arithmetic for the scores; the layer this
 * oracle checks takes fp32 logits, so the score is defined here as the fp32
 * dot product of the token with the expert's router column, accumulated in
 * index order with one fused multiply-add per term (one rounding per term),
 * followed by one fp32 addition of the expert's bias:
 *
 *     acc_0 = 0;  acc_{i+1} = fma(x[t,i], Wr[i,e], acc_i)  for i = 0..d-1
 *     L[t,e] = acc_d + bias[e]
 *
 * Every rounding step is fixed by that definition, so any correct
 * implementation of it produces the same bits.  Plain C, no vector
 * intrinsics; OpenMP only splits the tokens between threads.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (see oracle/build.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

void oracle_router_logits_fp32(const float *x, const float *Wr, const float *bias,
                               int64_t T, int64_t d, int64_t E, float *L, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        float *acc = L + t * E; /* the token's E accumulators live in its output row */
        for (int64_t e = 0; e < E; ++e) acc[e] = 0.0f;
        for (int64_t i = 0; i < d; ++i) {
            const float xi = x[t * d + i];
            const float *wrow = Wr + i * E;
            for (int64_t e = 0; e < E; ++e) acc[e] = fmaf(xi, wrow[e], acc[e]);
        }
        if (bias)
            for (int64_t e = 0; e < E; ++e) acc[e] = acc[e] + bias[e];
    }
}
