/*
 * Oracle for masked grouped-query attention: plain fp64 loops, no tiling,
 * no online softmax, no reordering beyond the definition.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links or calls this
 * file; only the test suite, the package's smoke check and the benchmark's
 * CPU-baseline leg do. It shares no code with the CUDA library.
 *
 * What it computes (definition of scaled-dot-product attention with grouped
 * KV heads under a boolean mask):
 *   - VoxCPM page, "Upstream-identical practice", attention bullet: SDPA with
 *     enable_gqa on contiguous tensors; bidirectional in the local module;
 *     decode over a static cache under an explicit boolean mask, where slots
 *     past the current length are masked and add exact zeros.
 *   - OmniVoice page, "Upstream-identical practice", attention-mask bullet:
 *     a full 4D boolean mask, not causal, with the KV heads repeated.
 *   - OmniVoice page, "Memory & speed", packed_guidance paragraph: two
 *     sequences side by side in one row under a block-diagonal mask, each
 *     block computing what it computes alone.
 *
 * For batch b, query head h, query i, with KV head g = h / (Hq / Hkv):
 *   s_j = scale * sum_d q[b,h,i,d] * k[b,g,j,d]      for allowed (b,i,j)
 *   s_j = -inf                                        otherwise (masked_fill)
 *   m = max_j s_j,  p_j = exp(s_j - m),  l = sum_j p_j
 *   out[b,h,i,:] = sum_j p_j v[b,g,j,:] / l,   lse[b,h,i] = m + log(l)
 * A query row with no allowed key gives out = 0 and lse = -inf (the pages are
 * silent; SDPA would give NaN there).
 *
 * allowed(b,i,j) is the AND of whichever mask forms are given:
 *   bits   : bit (j % 32) of word bits[(b*Lq + i)*W + j/32], W = ceil(Lk/32),
 *            least-significant bit first; 1 = may attend (SDPA bool polarity);
 *   kv_len : j < kv_len[b];
 *   seg    : seg_q[b*Lq + i] == seg_k[b*Lk + j] and that id is >= 0;
 *   causal : j <= i + (Lk - Lq)  (VoxCPM page, "Upstream-identical practice",
 *            attention bullet: causal attention at prefill; the query rows
 *            are taken to be the last Lq of the Lk positions, which for
 *            Lq == Lk is the usual lower triangle).
 * With no mask form given every key is allowed.
 *
 * Layout: q [B][Hq][Lq][D], k and v [B][Hkv][Lk][D], out [B][Hq][Lq][D],
 * lse [B][Hq][Lq], all contiguous fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int key_allowed(int b, int i, int j, int Lq, int Lk,
                       const uint32_t *bits, const int32_t *kv_len,
                       const int32_t *seg_q, const int32_t *seg_k, int causal) {
    if (causal && j > i + (Lk - Lq)) return 0;
    if (bits) {
        long W = (Lk + 31) / 32;
        uint32_t word = bits[((long)b * Lq + i) * W + j / 32];
        if (((word >> (j % 32)) & 1u) == 0u) return 0;
    }
    if (kv_len) {
        if (j >= kv_len[b]) return 0;
    }
    if (seg_q && seg_k) {
        int32_t a = seg_q[(long)b * Lq + i];
        int32_t c = seg_k[(long)b * Lk + j];
        if (a < 0 || a != c) return 0;
    }
    return 1;
}

/* Returns the number of OpenMP threads used (1 without OpenMP), or -1 on a
 * shape error. nthreads <= 0 means "all the cores OpenMP sees". */
int mgqa_oracle_attention(const double *q, const double *k, const double *v,
                          int B, int Hq, int Hkv, int Lq, int Lk, int D,
                          const uint32_t *bits, const int32_t *kv_len,
                          const int32_t *seg_q, const int32_t *seg_k,
                          int causal, double scale, double *out, double *lse, int nthreads) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Lq < 0 || Lk < 0 || D <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    if ((seg_q == NULL) != (seg_k == NULL)) return -1;
    int used = 1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    used = omp_get_max_threads();
#else
    (void)nthreads;
#endif
    const int n_rep = Hq / Hkv;
    const long rows = (long)B * Hq * Lq;

#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (Lk > 0 ? Lk : 1));
        double *acc = (double *)malloc(sizeof(double) * D);
#pragma omp for schedule(static)
        for (long r = 0; r < rows; ++r) {
            const int i = (int)(r % Lq);
            const int h = (int)((r / Lq) % Hq);
            const int b = (int)(r / ((long)Lq * Hq));
            const int g = h / n_rep;
            const double *qi = q + r * D;
            const double *kg = k + ((long)b * Hkv + g) * (long)Lk * D;
            const double *vg = v + ((long)b * Hkv + g) * (long)Lk * D;

            double m = -INFINITY;
            for (int j = 0; j < Lk; ++j) {
                if (key_allowed(b, i, j, Lq, Lk, bits, kv_len, seg_q, seg_k, causal)) {
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += qi[d] * kg[(long)j * D + d];
                    s[j] = scale * dot;
                } else {
                    s[j] = -INFINITY;
                }
                if (s[j] > m) m = s[j];
            }
            double *o = out + r * D;
            if (m == -INFINITY) {
                for (int d = 0; d < D; ++d) o[d] = 0.0;
                if (lse) lse[r] = -INFINITY;
                continue;
            }
            double l = 0.0;
            for (int d = 0; d < D; ++d) acc[d] = 0.0;
            for (int j = 0; j < Lk; ++j) {
                double p = exp(s[j] - m); /* exp(-inf) == 0 exactly */
                l += p;
                for (int d = 0; d < D; ++d) acc[d] += p * vg[(long)j * D + d];
            }
            for (int d = 0; d < D; ++d) o[d] = acc[d] / l;
            if (lse) lse[r] = m + log(l);
        }
        free(s);
        free(acc);
    }
    return used;
}
