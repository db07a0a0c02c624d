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
 *
 * The file also holds mgqa_oracle_rope (rotary position embedding), defined
 * and cited where it is written, below.
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

/*
 * Rotary position embedding (RoPE), in place on x [B][H][L][D] (fp64 values
 * of the 16- or 32-bit input):
 *   - F5-TTS page, module table and "Upstream-identical practice": the DiT
 *     rotates interleaved feature pairs, on its first pe_attn_head heads only;
 *   - OmniVoice page, "Parity results" (the shared Qwen decoder keeps the
 *     inverse frequencies in fp32) and VoxCPM page, "Upstream-identical
 *     practice", precision bullet (the LongRoPE table is built in fp32): the
 *     language models rotate with an fp32
 *     inverse-frequency table (LongRoPE: a table built in fp32);
 *   - OmniVoice page, "Memory & speed", packed_guidance paragraph: under
 *     packing every sequence's positions start at 0 (so positions are an
 *     input, not the row index).
 * For batch b, head h < heads, position index l, pair i < rot_dim/2:
 *   theta = fl32( (float)pos[b,l] * inv_freq[i] )      (one fp32 product)
 *   (a, c) = (x[.., e0], x[.., e1]) with (e0, e1) = (2i, 2i+1) if interleaved,
 *                                                   (i, i + rot_dim/2) otherwise
 *   x[.., e0] = a cos(theta) - c sin(theta);  x[.., e1] = a sin(theta) + c cos(theta)
 * cos and sin of theta in fp64. Features >= rot_dim and heads >= `heads` are
 * untouched. positions == NULL means pos[b,l] = l. Returns 0, or -1 on bad
 * sizes.
 */
int mgqa_oracle_rope(double *x, int B, int H, int L, int D, const int32_t *positions,
                     const float *inv_freq, int rot_dim, int heads, int interleaved) {
    if (B < 0 || H <= 0 || L < 0 || D <= 0 || rot_dim < 0 || rot_dim > D || (rot_dim & 1) ||
        heads < 0 || heads > H)
        return -1;
    const int half = rot_dim / 2;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < heads; ++h)
            for (int l = 0; l < L; ++l) {
                const int32_t p = positions ? positions[(long)b * L + l] : l;
                double *row = x + (((long)b * H + h) * L + l) * D;
                for (int i = 0; i < half; ++i) {
                    volatile float theta = (float)p * inv_freq[i];
                    const double t = (double)theta;
                    const double cs = cos(t), sn = sin(t);
                    const int e0 = interleaved ? 2 * i : i;
                    const int e1 = interleaved ? 2 * i + 1 : i + half;
                    const double a = row[e0], c = row[e1];
                    row[e0] = a * cs - c * sn;
                    row[e1] = a * sn + c * cs;
                }
            }
    return 0;
}

/*
 * RMS normalisation of every head vector before the rotation (OmniVoice page,
 * "Parity results": the shared Qwen decoder normalises q and k separately,
 * as transformers does, before applying the rotary embedding):
 *   y[d] = x[d] / sqrt(mean_d(x^2) + eps) * w[d]
 * over the head dim D of every row of x [B][H][L][D] (fp64 values), in place,
 * for heads h < `heads` only. Returns 0, or -1 on bad sizes.
 */
int mgqa_oracle_rms_norm(double *x, int B, int H, int L, int D, const float *w, double eps,
                         int heads) {
    if (B < 0 || H <= 0 || L < 0 || D <= 0 || heads < 0 || heads > H || eps < 0.0) return -1;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < heads; ++h)
            for (int l = 0; l < L; ++l) {
                double *row = x + (((long)b * H + h) * L + l) * D;
                double ss = 0.0;
                for (int d = 0; d < D; ++d) ss += row[d] * row[d];
                const double r = 1.0 / sqrt(ss / D + eps);
                for (int d = 0; d < D; ++d) row[d] = row[d] * r * (double)w[d];
            }
    return 0;
}
