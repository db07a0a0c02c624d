// One-query attention over a static KV cache, split over a fixed set of CTAs
// per (request, KV-head group) and merged by log-sum-exp in the same launch.
//
// Passages: VoxCPM page, "Upstream-identical practice", attention bullet
// (decode against the static cache under an explicit boolean mask; slots past
// the current length are masked and add exact zeros) and "Memory & speed",
// attention_span paragraph (attend only to the filled blocks of the 8192-slot
// cache instead of all of it).
//
// Design: kDecodeSplits CTAs serve one (request b, head group hg) -- the NREP
// query heads of one KV head. The cache is cut into 128-slot chunks of
// absolute positions; CTA x owns chunks x, x+S, x+2S, ... (S = kDecodeSplits).
//   1. One thread per slot tests every mask form; warp ballots give the CTA's
//      allowed-slot bitmap, which is compacted into a dense list. Masked slots
//      are never read, empty chunks cost nothing.
//   2. The allowed K and V rows are gathered with 16-byte asynchronous copies
//      (consecutive threads on one row, so each row is one coalesced read)
//      into dense shared-memory rows, up to CAP rows per batch.
//   3. Scores: D/8 (bf16) lanes share a row, 16 bytes each, NREP dot products
//      per lane, butterfly-summed; per-head batch softmax (one warp a head);
//      P.V by one thread per (head, pair of dims) over the dense rows; batches
//      fold into a running (m, l, o) in ascending slot order.
//   4. Every CTA writes its partial (m, l, o) to the workspace and takes a
//      ticket; the last of the S CTAs merges the S partials in ascending x and
//      resets the ticket.
// The chunk-to-CTA assignment and every summation order depend only on the
// set of allowed slots, so a full-cache bitmask and the equivalent filled
// length give bit-identical outputs.
#include <cfloat>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mgqa {
namespace {

struct DecodeParams {
  const void *q, *k, *v;
  void *out;
  int64_t qs_b, qs_h, ks_b, ks_h, ks_l, vs_b, vs_h, vs_l, os_b, os_h;
  const uint32_t *bits;
  int64_t ms_b;
  const int32_t *kv_len, *seg_q, *seg_k;
  // fused append: this step's K/V rows go to slot kv_len[b] first
  const void *k_new, *v_new;
  int64_t kn_b, kn_h, vn_b, vn_h;
  int32_t *kv_len_out;
  int append;
  float scale_log2;
  float *lse;
  int32_t *err;
  int B, Hq, Hkv, Lk, n_rep, nch;
  float2 *ws_ml;      // [B][Hq][S]    (m in log2 units, l)
  float *ws_o;        // [B][Hq][S][D] unnormalised partial outputs
  unsigned *ws_tick;  // [B][Hq]
};

constexpr int kThreads = 256;
constexpr int C = kDecodeChunk;
constexpr int S = kDecodeSplits;
constexpr int kMaxCI = (kDecodeMaxLk / kDecodeChunk + S - 1) / S;  // chunks per CTA

template <typename T, int D>
constexpr int cap_rows() {  // dense K/V rows per batch: K and V <= 32 KB each
  return (32768 / (D * (int)sizeof(T))) < 256 ? (32768 / (D * (int)sizeof(T))) : 256;
}

// bf16 and fp16 run the two products on the tensor cores (mma.sync m16n8k16,
// the NREP query heads padded to 16 rows); fp32 stays on the CUDA cores.
// (A causal mask needs nothing here: the single query is the last position.)
template <typename T>
constexpr bool use_mma() {
  return sizeof(T) == 2;
}

template <typename T, int D, int NREP>
struct DecodeSmem {
  static constexpr int CAP = cap_rows<T, D>();
  static constexpr int RS = use_mma<T>() ? D + 8 : D;  // padded rows: conflict-free fragments
  static constexpr int SROWS = use_mma<T>() ? 1 : CAP;
  static constexpr int WG = use_mma<T>() ? kThreads / 32 : 1;
  alignas(128) T k[CAP][RS];
  alignas(128) T v[CAP][RS];
  float q[NREP][D];
  float s[NREP][SROWS];
  float wm[WG][NREP], wl[WG][NREP];  // per-warp (m, l) for the final in-CTA merge
  float wo[WG][NREP][D];             // per-warp unnormalised O
  uint32_t words[kMaxCI][C / 32];
  uint16_t slot[kMaxCI * C];
  int chunk_base[kMaxCI];
  float fo[NREP], fb[NREP];
  int n_all;
  int is_last;
};

template <typename T, int D, int NREP>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const __grid_constant__ DecodeParams p) {
  using Sm = DecodeSmem<T, D, NREP>;
  constexpr int CAP = Sm::CAP;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto &sm = *reinterpret_cast<Sm *>(smem_raw);

  const int x = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) allow_dependents();
  grid_dependency_wait();  // everything below may read what the previous kernel wrote
  const int h0 = hg * NREP;
  const int g = h0 / p.n_rep;
  const int nci = x < p.nch ? (p.nch - x + S - 1) / S : 0;
  // q does not depend on the mask: its loads fly together with kv_len's
  const T *qb = static_cast<const T *>(p.q) + (int64_t)b * p.qs_b;
  constexpr int QPT = (NREP * D + kThreads - 1) / kThreads;
  float qv[QPT];
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int i = tid + u * kThreads;
    qv[u] = i < NREP * D ? to_float(qb[(int64_t)(h0 + i / D) * p.qs_h + i % D]) : 0.f;
  }
  int kvl = load_kv_len(p.kv_len, b, p.Lk, p.err, x == 0 && hg == 0 && tid == 0);
  // append: the new row sits at slot `pos`, and the step attends to it too;
  // a full cache (kv_len == Lk) is an error and appends nothing
  int pos = -1;
  if (p.append) {
    if (kvl < p.Lk) {
      pos = kvl;
      kvl += 1;
    } else if (x == 0 && hg == 0 && tid == 0) {
      report_error(p.err, MGQA_ERR_INVALID_ARG);
    }
    if (p.kv_len_out && x == 0 && hg == 0 && tid == 0) p.kv_len_out[b] = kvl;
  }
  const int segq = p.seg_q ? __ldg(p.seg_q + b) : 0;

  // 1. allowed-slot bitmap of this CTA's chunks (two chunks per pass)
  auto allowed = [&](int i, int t) {
    const int j = (x + S * i) * C + t;
    bool a = i < nci && j < p.Lk && j < kvl;
    if (a && p.bits) a = (__ldg(p.bits + (int64_t)b * p.ms_b + (j >> 5)) >> (j & 31)) & 1u;
    if (a && p.seg_q) a = segq >= 0 && __ldg(p.seg_k + (int64_t)b * p.Lk + j) == segq;
    return a;
  };
  for (int i0 = 0; i0 < nci; i0 += kThreads / C) {
    const int i = i0 + tid / C, t = tid % C;
    const uint32_t word = __ballot_sync(0xffffffffu, allowed(i, t));
    if (lane == 0 && i < nci) sm.words[i][t >> 5] = word;
  }
  __syncthreads();
  if (tid == 0) {
    int base = 0;
    for (int i = 0; i < nci; ++i) {
      sm.chunk_base[i] = base;
#pragma unroll
      for (int w = 0; w < C / 32; ++w) base += __popc(sm.words[i][w]);
    }
    sm.n_all = base;
  }
  __syncthreads();
  // dense list of allowed slots, ascending
  for (int i0 = 0; i0 < nci; i0 += kThreads / C) {
    const int i = i0 + tid / C, t = tid % C;
    if (i < nci) {
      const uint32_t wd = sm.words[i][t >> 5];
      if ((wd >> (t & 31)) & 1u) {
        int rank = sm.chunk_base[i] + __popc(wd & ((1u << (t & 31)) - 1u));
        for (int w = 0; w < (t >> 5); ++w) rank += __popc(sm.words[i][w]);
        sm.slot[rank] = (uint16_t)(i * C + t);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int i = tid + u * kThreads;
    if (i < NREP * D) sm.q[i / D][i % D] = qv[u];
  }
  __syncthreads();
  const int n_all = sm.n_all;

  // 2-3. batches of dense rows
  constexpr int EPL = 16 / sizeof(T);  // elements per 16-byte lane load
  constexpr int G = D / EPL;           // lanes per row
  constexpr int SPW = 32 / G;          // rows per warp pass
  constexpr int ROWS_W = CAP / (kThreads / 32);
  static_assert(G <= 32 && ROWS_W % SPW == 0, "lane layout");
  constexpr int ITEMS = (NREP * D / 2 + kThreads - 1) / kThreads;  // (head, dim pair) per thread
  float o[ITEMS][2];
#pragma unroll
  for (int u = 0; u < ITEMS; ++u) o[u][0] = o[u][1] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // meaningful in warp r < NREP
  const bool ok = true;
  const int e = lane % G, sub = lane / G;
  // tensor-core path: Q as the A fragment (heads gq < NREP; rows gq+8 are padding)
  constexpr int RW = CAP / (kThreads / 32);  // dense rows per warp per batch
  constexpr int NT8 = RW / 8;
  const int gq = lane >> 2, tq = lane & 3;
  uint32_t qa[use_mma<T>() ? D / 16 : 1][2];
  float ow[use_mma<T>() ? D / 8 : 1][4];
  float wm_run = -INFINITY, wl_run = 0.f;
  if constexpr (use_mma<T>()) {
    static_assert(RW % 16 == 0, "rows per warp");
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = qa[kk][1] = 0u;
      if (gq < NREP) {
        qa[kk][0] = pack2<T>(sm.q[gq][kk * 16 + 2 * tq], sm.q[gq][kk * 16 + 2 * tq + 1]);
        qa[kk][1] = pack2<T>(sm.q[gq][kk * 16 + 2 * tq + 8], sm.q[gq][kk * 16 + 2 * tq + 9]);
      }
    }
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) ow[dt][0] = ow[dt][1] = ow[dt][2] = ow[dt][3] = 0.f;
  }
  const T *kg = static_cast<const T *>(p.k) + (int64_t)b * p.ks_b + (int64_t)g * p.ks_h;
  const T *vg = static_cast<const T *>(p.v) + (int64_t)b * p.vs_b + (int64_t)g * p.vs_h;
  for (int bs = 0; bs < n_all; bs += CAP) {
    const int nb = min(CAP, n_all - bs);
    // gather the allowed rows: 16-byte pieces, consecutive threads on one row
    constexpr int PPR = D * sizeof(T) / 16;  // pieces per row
    for (int idx = tid; idx < nb * PPR; idx += kThreads) {
      const int kk = idx / PPR, part = idx % PPR;
      const int loc = sm.slot[bs + kk];
      const int64_t j = (int64_t)(x + S * (loc / C)) * C + loc % C;
      if (!MGQA_DCHECK(j < p.Lk && g < p.Hkv, p.err)) continue;
      const T *ksrc = kg + j * p.ks_l, *vsrc = vg + j * p.vs_l;
      if (j == pos) {  // the appended row: read it from the step's input
        ksrc = static_cast<const T *>(p.k_new) + (int64_t)b * p.kn_b + (int64_t)g * p.kn_h;
        vsrc = static_cast<const T *>(p.v_new) + (int64_t)b * p.vn_b + (int64_t)g * p.vn_h;
      }
      cp_async16(reinterpret_cast<char *>(&sm.k[kk][0]) + part * 16,
                 reinterpret_cast<const char *>(ksrc) + part * 16);
      cp_async16(reinterpret_cast<char *>(&sm.v[kk][0]) + part * 16,
                 reinterpret_cast<const char *>(vsrc) + part * 16);
    }
    if constexpr (use_mma<T>()) {
      // rows past nb in the last 16-row group feed the P.V MMA with P = 0:
      // keep them finite
      const int tail = min(CAP, (nb + 15) & ~15) - nb;
      for (int idx = tid; idx < tail * (D / 8); idx += kThreads)
        *reinterpret_cast<uint4 *>(&sm.v[nb + idx / (D / 8)][(idx % (D / 8)) * 8]) =
            make_uint4(0u, 0u, 0u, 0u);
    }
    cp_async_wait_all();
    __syncthreads();

    if constexpr (use_mma<T>()) {
      // warp w owns dense rows [w*RW, w*RW + RW) of the batch and keeps its
      // own running (m, l, O) for head gq; warps merge after the last batch
      const int r0 = warp * RW;
      if (r0 < nb) {
        const int n8 = min(NT8, (nb - r0 + 7) / 8);    // row tiles holding a valid row
        const int n16 = min(RW / 16, (nb - r0 + 15) / 16);
        float c[NT8][4];
#pragma unroll
        for (int nt = 0; nt < NT8; ++nt) {
          c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
          if (nt >= n8) continue;  // warp-uniform
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const T *kr = &sm.k[r0 + nt * 8 + gq][kk * 16 + 2 * tq];
            mma_16816<T>(c[nt], qa[kk][0], 0u, qa[kk][1], 0u,
                           *reinterpret_cast<const uint32_t *>(kr),
                           *reinterpret_cast<const uint32_t *>(kr + 8));
          }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int row = r0 + nt * 8 + 2 * tq + h;
            c[nt][h] = row < nb ? c[nt][h] * p.scale_log2 : -INFINITY;
            mx = fmaxf(mx, c[nt][h]);
          }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(wm_run, mx);
        const float f = (wm_run == -INFINITY) ? 0.f : exp2f(wm_run - m_new);
        float ps = 0.f;
        uint32_t pa[NT8];
#pragma unroll
        for (int nt = 0; nt < NT8; ++nt) {
          const float p0 = exp2f(c[nt][0] - m_new), p1 = exp2f(c[nt][1] - m_new);
          ps += p0 + p1;
          pa[nt] = pack2<T>(p0, p1);
        }
        ps += __shfl_xor_sync(0xffffffffu, ps, 1);
        ps += __shfl_xor_sync(0xffffffffu, ps, 2);
        wl_run = wl_run * f + ps;
        wm_run = m_new;
#pragma unroll
        for (int dt = 0; dt < D / 8; ++dt) {
          ow[dt][0] *= f;
          ow[dt][1] *= f;
        }
#pragma unroll
        for (int ks = 0; ks < RW / 16; ++ks) {
          if (ks >= n16) break;  // warp-uniform; rows up to the next 16 are zero-filled
#pragma unroll
          for (int dt = 0; dt < D / 8; ++dt) {
            uint32_t b0, b1;
            ldmatrix_x2_trans(b0, b1, &sm.v[r0 + ks * 16 + (lane & 15)][dt * 8]);
            mma_16816<T>(ow[dt], pa[2 * ks], 0u, pa[2 * ks + 1], 0u, b0, b1);
          }
        }
      }
    } else {
    // scores (log2 units)
      {
        float qr[NREP][EPL];
  #pragma unroll
        for (int r = 0; r < NREP; ++r)
  #pragma unroll
          for (int i = 0; i < EPL; ++i) qr[r][i] = sm.q[r][e * EPL + i];
        for (int it = 0; it < ROWS_W / SPW; ++it) {
          const int row_first = warp * ROWS_W + it * SPW;
          if (row_first >= nb) break;  // warp-uniform
          const int row = row_first + sub;
          const bool valid = row < nb;
          float acc[NREP];
  #pragma unroll
          for (int r = 0; r < NREP; ++r) acc[r] = 0.f;
          if (valid) {
            const uint4 u = *reinterpret_cast<const uint4 *>(&sm.k[row][e * EPL]);
            float kf[EPL];
            unpack16_t<T>(u, kf);
  #pragma unroll
            for (int r = 0; r < NREP; ++r)
  #pragma unroll
              for (int i = 0; i < EPL; ++i) acc[r] = fmaf(qr[r][i], kf[i], acc[r]);
          }
  #pragma unroll
          for (int off = G / 2; off > 0; off >>= 1)
  #pragma unroll
            for (int r = 0; r < NREP; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
          if (e == 0 && valid) {
  #pragma unroll
            for (int r = 0; r < NREP; ++r) sm.s[r][row] = acc[r] * p.scale_log2;
          }
        }
      }
      __syncthreads();
      // per-head batch softmax, folded into the running (m, l)
      if (warp < NREP) {
        const int r = warp;
        float mb = -INFINITY;
        for (int i = lane; i < nb; i += 32) mb = fmaxf(mb, sm.s[r][i]);
  #pragma unroll
        for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
        float lb = 0.f;
        for (int i = lane; i < nb; i += 32) {
          const float pr = exp2f(sm.s[r][i] - mb);
          sm.s[r][i] = pr;
          lb += pr;
        }
  #pragma unroll
        for (int off = 16; off > 0; off >>= 1) lb += __shfl_xor_sync(0xffffffffu, lb, off);
        const float m_new = fmaxf(m_run, mb);
        const float f_old = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
        const float f_b = exp2f(mb - m_new);
        l_run = l_run * f_old + lb * f_b;
        m_run = m_new;
        if (lane == 0) {
          sm.fo[r] = f_old;
          sm.fb[r] = f_b;
        }
      }
      __syncthreads();
      // P.V over the dense rows, ascending
  #pragma unroll
      for (int u = 0; u < ITEMS; ++u) {
        const int idx = tid + u * kThreads;
        if (idx < NREP * D / 2) {
          const int r = idx / (D / 2), dp = idx % (D / 2);
          float a0 = 0.f, a1 = 0.f;
  #pragma unroll 4
          for (int kk = 0; kk < nb; ++kk) {
            const float pr = sm.s[r][kk];
            float v0, v1;
            if constexpr (sizeof(T) == 2) {
              const __nv_bfloat162 vv = *reinterpret_cast<const __nv_bfloat162 *>(&sm.v[kk][2 * dp]);
              v0 = __low2float(vv);
              v1 = __high2float(vv);
            } else {
              const float2 vv = *reinterpret_cast<const float2 *>(&sm.v[kk][2 * dp]);
              v0 = vv.x;
              v1 = vv.y;
            }
            a0 = fmaf(pr, v0, a0);
            a1 = fmaf(pr, v1, a1);
          }
          o[u][0] = o[u][0] * sm.fo[r] + a0 * sm.fb[r];
          o[u][1] = o[u][1] * sm.fo[r] + a1 * sm.fb[r];
        }
      }
    }
    __syncthreads();  // the next batch overwrites k, v and s
  }

  if constexpr (use_mma<T>()) {
    // in-CTA merge of the warps' (m, l, O), ascending warp order
    if (gq < NREP) {
      if (tq == 0) {
        sm.wm[warp][gq] = wm_run;
        sm.wl[warp][gq] = wl_run;
      }
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) {
        sm.wo[warp][gq][dt * 8 + 2 * tq] = ow[dt][0];
        sm.wo[warp][gq][dt * 8 + 2 * tq + 1] = ow[dt][1];
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) {
      const int idx = tid + u * kThreads;
      if (idx < NREP * D / 2) {
        const int r = idx / (D / 2), dp = idx % (D / 2);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) M = fmaxf(M, sm.wm[w][r]);
        float a0 = 0.f, a1 = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kThreads / 32; ++w) {
            if (sm.wm[w][r] == -INFINITY) continue;
            const float wt = exp2f(sm.wm[w][r] - M);
            a0 = fmaf(sm.wo[w][r][2 * dp], wt, a0);
            a1 = fmaf(sm.wo[w][r][2 * dp + 1], wt, a1);
          }
        }
        o[u][0] = a0;
        o[u][1] = a1;
      }
    }
    if (warp < NREP) {
      const int r = warp;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kThreads / 32; ++w) M = fmaxf(M, sm.wm[w][r]);
      float L = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w)
          if (sm.wm[w][r] != -INFINITY) L = fmaf(sm.wl[w][r], exp2f(sm.wm[w][r] - M), L);
      }
      m_run = M;
      l_run = L;
    }
  }

  // append: the CTA owning slot pos stores the new row into the cache (once
  // per KV head: only its first head group); no other CTA of this step reads
  // that slot from the cache
  if (pos >= 0 && (pos / C) % S == x && h0 % p.n_rep == 0) {
    constexpr int PPR = D * sizeof(T) / 16;
    const char *kn = static_cast<const char *>(p.k_new) +
                     ((int64_t)b * p.kn_b + (int64_t)g * p.kn_h) * sizeof(T);
    const char *vn = static_cast<const char *>(p.v_new) +
                     ((int64_t)b * p.vn_b + (int64_t)g * p.vn_h) * sizeof(T);
    char *kd = const_cast<char *>(reinterpret_cast<const char *>(kg + (int64_t)pos * p.ks_l));
    char *vd = const_cast<char *>(reinterpret_cast<const char *>(vg + (int64_t)pos * p.vs_l));
    for (int part = tid; part < 2 * PPR; part += kThreads) {
      if (part < PPR)
        reinterpret_cast<uint4 *>(kd)[part] = reinterpret_cast<const uint4 *>(kn)[part];
      else
        reinterpret_cast<uint4 *>(vd)[part - PPR] = reinterpret_cast<const uint4 *>(vn)[part - PPR];
    }
  }

  // 4. partial of this CTA; the last of the S CTAs merges all of them
  const int64_t hrow0 = ((int64_t)b * p.Hq + h0) * S;  // ws row of (head h0, split 0)
#pragma unroll
  for (int u = 0; u < ITEMS; ++u) {
    const int idx = tid + u * kThreads;
    if (idx < NREP * D / 2) {
      const int r = idx / (D / 2), dp = idx % (D / 2);
      reinterpret_cast<float2 *>(p.ws_o + (hrow0 + (int64_t)r * S + x) * D)[dp] =
          make_float2(o[u][0], o[u][1]);
    }
  }
  if (warp < NREP && lane == 0)
    p.ws_ml[hrow0 + (int64_t)warp * S + x] =
        (ok && m_run != -INFINITY) ? make_float2(m_run, l_run) : make_float2(-INFINITY, 0.f);
  __syncthreads();
  unsigned *tick = p.ws_tick + (int64_t)b * p.Hq + h0;
  if (tid == 0) {
    unsigned t;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(t) : "l"(tick) : "memory");
    sm.is_last = (t == (unsigned)(S - 1));
  }
  __syncthreads();
  if (!sm.is_last) return;

#pragma unroll
  for (int u = 0; u < ITEMS; ++u) {
    const int idx = tid + u * kThreads;
    if (idx < NREP * D / 2) {
      const int r = idx / (D / 2), dp = idx % (D / 2);
      const int64_t hr = hrow0 + (int64_t)r * S;
      // every split wrote its partial this call (empty ones: m = -inf, zeros),
      // so all loads go out in one round
      float2 ml[S], ov[S];
#pragma unroll
      for (int xx = 0; xx < S; ++xx) {
        ml[xx] = __ldcg(&p.ws_ml[hr + xx]);
        ov[xx] = __ldcg(reinterpret_cast<const float2 *>(p.ws_o + (hr + xx) * D) + dp);
      }
      float M = -INFINITY;
#pragma unroll
      for (int xx = 0; xx < S; ++xx) M = fmaxf(M, ml[xx].x);
      float L = 0.f, o0 = 0.f, o1 = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int xx = 0; xx < S; ++xx) {
          if (ml[xx].x == -INFINITY) continue;
          const float w = exp2f(ml[xx].x - M);
          L = fmaf(ml[xx].y, w, L);
          o0 = fmaf(ov[xx].x, w, o0);
          o1 = fmaf(ov[xx].y, w, o1);
        }
      }
      const float inv = (L > 0.f) ? 1.f / L : 0.f;
      T *orow = static_cast<T *>(p.out) + (int64_t)b * p.os_b + (int64_t)(h0 + r) * p.os_h;
      orow[2 * dp] = from_float<T>(o0 * inv);
      orow[2 * dp + 1] = from_float<T>(o1 * inv);
      if (dp == 0 && p.lse)
        p.lse[(int64_t)b * p.Hq + h0 + r] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
  }
  if (tid == 0) *tick = 0u;
}

template <typename T, int D, int NREP>
mgqa_status launch_t(const DecodeParams &p, cudaStream_t s) {
  auto kern = decode_kernel<T, D, NREP>;
  const size_t smem = sizeof(DecodeSmem<T, D, NREP>);
  static std::atomic<uint64_t> attr_done{0};
  const mgqa_status st = ensure_smem_attr(kern, (int)smem, attr_done, "decode kernel");
  if (st != MGQA_OK) return st;
  dim3 grid(S, p.Hq / NREP, p.B);
  const cudaError_t e = launch_pdl(kern, grid, dim3(kThreads), smem, s, p);
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return MGQA_OK;
}

template <typename T, int D>
mgqa_status launch_nrep(const DecodeParams &p, int hpc, cudaStream_t s) {
  switch (hpc) {
    case 1: return launch_t<T, D, 1>(p, s);
    case 2: return launch_t<T, D, 2>(p, s);
    case 4: return launch_t<T, D, 4>(p, s);
    case 8: return launch_t<T, D, 8>(p, s);
    default: return fail(MGQA_ERR_UNSUPPORTED, "decode: heads per CTA %d", hpc);
  }
}

struct WsLayout {
  size_t ml, o, tick, total;
};

WsLayout ws_layout(const mgqa_args &a) {
  const size_t rows = (size_t)a.B * a.Hq * S;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  WsLayout w;
  w.ml = 0;
  w.o = up(rows * sizeof(float2));
  w.tick = w.o + up(rows * a.D * sizeof(float));
  w.total = w.tick + up((size_t)a.B * a.Hq * sizeof(unsigned));
  return w;
}

}  // namespace

int decode_heads_per_cta(int n_rep) {
  for (int h : {8, 4, 2, 1})
    if (n_rep % h == 0) return h;
  return 1;
}

size_t decode_workspace_bytes(const mgqa_args &a) { return ws_layout(a).total; }

mgqa_status launch_decode(const mgqa_args &a, void *ws, size_t ws_bytes, cudaStream_t s) {
  return launch_decode_append(a, nullptr, nullptr, nullptr, nullptr, nullptr, ws, ws_bytes, s);
}

mgqa_status launch_decode_append(const mgqa_args &a, const void *k_new, const void *v_new,
                                 const int64_t *k_new_stride, const int64_t *v_new_stride,
                                 int32_t *kv_len_out, void *ws, size_t ws_bytes, cudaStream_t s) {
  const WsLayout L = ws_layout(a);
  if (ws_bytes < L.total) return fail(MGQA_ERR_INVALID_ARG, "decode workspace too small");
  DecodeParams p{};
  p.q = a.q; p.k = a.k; p.v = a.v; p.out = a.out;
  p.qs_b = a.q_stride[0]; p.qs_h = a.q_stride[1];
  p.ks_b = a.k_stride[0]; p.ks_h = a.k_stride[1]; p.ks_l = a.k_stride[2];
  p.vs_b = a.v_stride[0]; p.vs_h = a.v_stride[1]; p.vs_l = a.v_stride[2];
  p.os_b = a.o_stride[0]; p.os_h = a.o_stride[1];
  p.bits = a.mask_bits; p.ms_b = a.mask_stride_b;
  p.kv_len = a.kv_len; p.seg_q = a.seg_q; p.seg_k = a.seg_k;
  p.scale_log2 = a.scale * kLog2e;
  p.lse = a.lse; p.err = a.dev_error;
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv; p.Lk = a.Lk; p.n_rep = a.Hq / a.Hkv;
  p.nch = (a.Lk + kDecodeChunk - 1) / kDecodeChunk;
  char *base = static_cast<char *>(ws);
  p.ws_ml = reinterpret_cast<float2 *>(base + L.ml);
  p.ws_o = reinterpret_cast<float *>(base + L.o);
  p.ws_tick = reinterpret_cast<unsigned *>(base + L.tick);
  p.append = k_new != nullptr;
  if (p.append) {
    p.k_new = k_new;
    p.v_new = v_new;
    p.kn_b = k_new_stride[0]; p.kn_h = k_new_stride[1];
    p.vn_b = v_new_stride[0]; p.vn_h = v_new_stride[1];
    p.kv_len_out = kv_len_out;
  }
  const int hpc = decode_heads_per_cta(p.n_rep);
  if (a.dtype == MGQA_BF16) {
    if (a.D == 64) return launch_nrep<__nv_bfloat16, 64>(p, hpc, s);
    if (a.D == 128) return launch_nrep<__nv_bfloat16, 128>(p, hpc, s);
  } else if (a.dtype == MGQA_FP16) {
    if (a.D == 64) return launch_nrep<__half, 64>(p, hpc, s);
    if (a.D == 128) return launch_nrep<__half, 128>(p, hpc, s);
  } else {
    if (a.D == 64) return launch_nrep<float, 64>(p, hpc, s);
    if (a.D == 128) return launch_nrep<float, 128>(p, hpc, s);
  }
  return fail(MGQA_ERR_UNSUPPORTED, "decode: head dim %d", a.D);
}

}  // namespace mgqa

// ---- decode with library-owned scratch -------------------------------------
// For callers that cannot hand the library any device memory of its own: the
// partial results and merge tickets of a call live in one fixed array that
// every GPU loading this library keeps until the process exits.

namespace mgqa {
namespace {

constexpr size_t kStaticScratchBytes = (size_t)MGQA_DECODE_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];  // device address of g_static_scratch, per device

// Device address of the scratch array on the current device. The first call
// on a device looks it up (with that device current) and caches it.
mgqa_status static_scratch(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(MGQA_ERR_CUDA, "no usable current CUDA device");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_static_scratch);
    if (e != cudaSuccess || addr == nullptr)
      return fail(MGQA_ERR_CUDA, "cudaGetSymbolAddress of the decode scratch failed: %s",
                  cudaGetErrorString(e));
    g_scratch_addr[dev] = addr;
  }
  *out = g_scratch_addr[dev];
  return MGQA_OK;
}

}  // namespace
}  // namespace mgqa

extern "C" mgqa_status masked_gqa_attn_decode_static(const mgqa_args *args, cudaStream_t stream) {
  const size_t need = masked_gqa_attn_decode_workspace_size(args);
  if (need == 0) return masked_gqa_attn_decode(args, nullptr, 0, stream);  // reports the bad argument
  if (need > mgqa::kStaticScratchBytes)
    return mgqa::fail(MGQA_ERR_UNSUPPORTED,
                      "this decode needs %zu bytes of scratch; the library's fixed scratch holds %zu "
                      "(pass a workspace to masked_gqa_attn_decode instead)",
                      need, mgqa::kStaticScratchBytes);
  void *ws = nullptr;
  const mgqa_status st = mgqa::static_scratch(&ws);
  if (st != MGQA_OK) return st;
  // The merge tickets must start at zero. Their place in the array depends on
  // the shape, so a call after one of another shape could find leftovers
  // there: clear them on the caller's stream before every launch.
  const mgqa::WsLayout lay = mgqa::ws_layout(*args);
  if (cudaMemsetAsync(static_cast<char *>(ws) + lay.tick, 0, lay.total - lay.tick, stream) !=
      cudaSuccess)
    return mgqa::fail(MGQA_ERR_CUDA, "clearing the decode scratch tickets failed");
  return masked_gqa_attn_decode(args, ws, mgqa::kStaticScratchBytes, stream);
}
