/*
 * Canonical float32 lightning-indexer score.  TEST INFRASTRUCTURE ONLY: part of
 * the CPU oracle; no product code links or includes this file.
 *
 * DeepSeek-V4 report (cnblogs translation), §2.3.1 "lightning indexer":
 * score_j = sum_h w_h * ReLU(q_h . kI_j).  The pages fix no summation order;
 * to make float32 selections reproducible the order is fixed here:
 *   acc_h = 0; for d in 0..d_I-1: acc_h = fma(q[h][d], k[j][d], acc_h)
 *   r_h   = acc_h > 0 ? acc_h : +0
 *   s     = 0; for h in 0..H_I-1: s = fma(w[h], r_h, s)
 * Compiled with -ffp-contract=off so the compiler adds no contraction of its
 * own; every rounding is an explicit fmaf.
 */
#include <math.h>
#include <stdint.h>

void oracle_index_scores_f32(const float* q, const float* w, const float* k,
                             int64_t heads, int64_t dim, int64_t n, float* out) {
    for (int64_t j = 0; j < n; ++j) {
        const float* kj = k + j * dim;
        float s = 0.0f;
        for (int64_t h = 0; h < heads; ++h) {
            const float* qh = q + h * dim;
            float acc = 0.0f;
            for (int64_t d = 0; d < dim; ++d) acc = fmaf(qh[d], kj[d], acc);
            float r = acc > 0.0f ? acc : 0.0f;
            s = fmaf(w[h], r, s);
        }
        out[j] = s;
    }
}
