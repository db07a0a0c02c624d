// One-query attention over a static KV cache: the splits of a (request,
// KV-head group) form a thread-block cluster and merge their partial results
// through distributed shared memory, inside one launch.
//
// Passages: VoxCPM page, "Upstream-identical practice", attention bullet
// (decode against the static cache under an explicit boolean mask; slots past
// the current length are masked and add exact zeros) and "Memory & speed",
// attention_span paragraph (attend only to the filled blocks of the 8192-slot
// cache instead of all of it).
//
// Design: NS = G * SC CTAs serve one (request b, head group hg) -- the NREP
// query heads of one KV head -- as G clusters of SC CTAs (SC = 16, or 8 where
// the device cannot co-schedule 16; G = 1 unless the cache is long and the
// grid small). The cache is cut into 64-slot chunks of absolute positions;
// split x owns chunks x, x + NS, x + 2 NS, ...
//   1. Every input of the mask test (kv_len, the split's mask words, segment
//      ids) and q are loaded at once. One thread per slot then tests every mask
//      form; warp ballots give the allowed-slot words, compacted into a dense
//      ascending list. Masked slots are never read; empty chunks cost nothing.
//   2. The allowed K and V rows are gathered with 16-byte asynchronous copies
//      (consecutive threads on one row) into padded shared-memory rows, two
//      batches of CAPB rows in flight: batch n + 2 is issued as soon as batch
//      n has been consumed.
//   3. bf16 / fp16: both products on the tensor cores (mma.sync m16n8k16, the
//      <= 8 query heads padded to 16 rows); each compute warp keeps a running
//      (m, l, O) over its 16 rows of every batch, and the warps merge in
//      ascending order. fp32: CUDA cores, per-head batch softmax.
//   4. The CTA's partial (m, l, O) stays in its shared memory. After a cluster
//      barrier, cluster rank r merges a 1/SC slice of the NREP x D outputs by
//      reading the SC partials through distributed shared memory in ascending
//      rank, and writes them (G = 1). With G > 1 each cluster's merged partial
//      goes to the caller's workspace instead, and the last CTA to take a
//      ticket merges the G partials in ascending cluster order.
// The chunk-to-split assignment and every summation order depend only on the
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
  int G;              // clusters per (request, head group)
  float2 *ws_ml;      // G > 1: [B][Hq][G] (m in log2 units, l) of each cluster
  float *ws_o;        // G > 1: [B][Hq][G][D] unnormalised cluster outputs
  unsigned *ws_tick;  // G > 1: [B][Hq / NREP] arrival tickets
};

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int C = kDecodeChunk;

// bf16 and fp16 run the two products on the tensor cores; fp32 on the CUDA cores.
// (A causal mask needs nothing here: the single query is the last position.)
template <typename T>
constexpr bool use_mma() {
  return sizeof(T) == 2;
}

template <typename T, int D, int NREP, int SC>
struct DecodeSmem {
  static constexpr bool kMma = use_mma<T>();
  // dense K/V rows per batch buffer (two buffers): 16 KB of K per buffer for
  // the 16-bit types at D = 64, 8 KB otherwise
  static constexpr int CAPB = kMma ? (D == 64 ? 128 : 64) : (D == 64 ? 64 : 32);
  static constexpr int RS = kMma ? D + 8 : D;  // padded rows: conflict-free fragments
  static constexpr int CW = kMma ? CAPB / 16 : kWarps;  // compute warps (16 rows each)
  static constexpr int kMaxCI = kDecodeMaxLk / C / SC;  // chunks of one split (G = 1)
  struct Rows {
    alignas(128) T k[2][CAPB][RS];
    alignas(128) T v[2][CAPB][RS];
  };
  struct WarpParts {  // per-warp (m, l, O) for the in-CTA merge (after the last batch)
    float o[CW][NREP][D];
    float m[CW][NREP], l[CW][NREP];
  };
  union {
    Rows r;
    WarpParts w;
  } u;
  float q[NREP][D];
  float s[NREP][kMma ? 1 : CAPB];  // fp32 path: one batch's scores / weights
  float fo[NREP], fb[NREP];
  // this CTA's partial, read by the cluster merge
  float pm[NREP], pl[NREP];
  float po[NREP][D];
  uint32_t words[kMaxCI][C / 32];  // mask words (bits form), then allowed-slot words
  int base[kMaxCI];                // dense index of each chunk's first allowed slot
  uint16_t slot[kMaxCI * C];       // dense list: chunk-local slot index (i * C + t)
  int n_all;
  int is_last;
};

// 16-byte pieces of the allowed rows [r0, r0 + nb) of the dense list into
// buffer `buf`; the appended row is read from the step's input.
template <typename T, int D, int NREP, int SC>
MGQA_DEV void gather_batch(DecodeSmem<T, D, NREP, SC> &sm, const DecodeParams &p, int buf, int r0,
                           int nb, const T *kg, const T *vg, int split, int NS, int b, int g,
                           int pos) {
  using Sm = DecodeSmem<T, D, NREP, SC>;
  constexpr int PPR = D * sizeof(T) / 16;  // pieces per row
  const int tid = threadIdx.x;
  for (int idx = tid; idx < nb * PPR; idx += kThreads) {
    const int kk = idx / PPR, part = idx % PPR;
    const int loc = sm.slot[r0 + kk];
    const int64_t j = (int64_t)(split + NS * (loc / C)) * C + loc % C;
    if (!MGQA_DCHECK(j < p.Lk && g < p.Hkv, p.err)) continue;
    const T *ksrc = kg + j * p.ks_l, *vsrc = vg + j * p.vs_l;
    if (j == pos) {  // the appended row: read it from the step's input
      ksrc = static_cast<const T *>(p.k_new) + (int64_t)b * p.kn_b + (int64_t)g * p.kn_h;
      vsrc = static_cast<const T *>(p.v_new) + (int64_t)b * p.vn_b + (int64_t)g * p.vn_h;
    }
    cp_async16(reinterpret_cast<char *>(&sm.u.r.k[buf][kk][0]) + part * 16,
               reinterpret_cast<const char *>(ksrc) + part * 16);
    cp_async16(reinterpret_cast<char *>(&sm.u.r.v[buf][kk][0]) + part * 16,
               reinterpret_cast<const char *>(vsrc) + part * 16);
  }
  if constexpr (Sm::kMma) {
    // rows past nb in the last 16-row group feed the P.V MMA with P = 0: keep
    // them finite (the buffer may hold anything)
    const int tail = min(Sm::CAPB, (nb + 15) & ~15) - nb;
    for (int idx = tid; idx < tail * (D / 8); idx += kThreads)
      *reinterpret_cast<uint4 *>(&sm.u.r.v[buf][nb + idx / (D / 8)][(idx % (D / 8)) * 8]) =
          make_uint4(0u, 0u, 0u, 0u);
  }
}

template <typename T, int D, int NREP, int SC>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const __grid_constant__ DecodeParams p) {
  using Sm = DecodeSmem<T, D, NREP, SC>;
  constexpr int CAPB = Sm::CAPB;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto &sm = *reinterpret_cast<Sm *>(smem_raw);

  const int split = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int rank = split % SC;  // the CTA's rank in its (SC, 1, 1) cluster
  const int cl = split / SC;    // the cluster's index among the G of this (b, hg)
  const int NS = SC * p.G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) allow_dependents();
  grid_dependency_wait();  // everything below may read what the previous kernel wrote
  const int h0 = hg * NREP;
  const int g = h0 / p.n_rep;
  const int nci = split < p.nch ? (p.nch - split + NS - 1) / NS : 0;  // my chunks

  // ---- 1. every load the mask test and the products need, issued together
  const int kvl_raw = p.kv_len ? __ldg(p.kv_len + b) : p.Lk;
  const T *qb = static_cast<const T *>(p.q) + (int64_t)b * p.qs_b;
  constexpr int QPT = (NREP * D + kThreads - 1) / kThreads;
  float qv[QPT];
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int i = tid + u * kThreads;
    qv[u] = i < NREP * D ? to_float(qb[(int64_t)(h0 + i / D) * p.qs_h + i % D]) : 0.f;
  }
  if (p.bits) {
    const int W = (p.Lk + 31) >> 5;
    for (int w = tid; w < 2 * nci; w += kThreads) {
      const int word = ((split + NS * (w >> 1)) * C >> 5) + (w & 1);
      sm.words[w >> 1][w & 1] = word < W ? __ldg(p.bits + (int64_t)b * p.ms_b + word) : 0u;
    }
  }
  const int segq = p.seg_q ? __ldg(p.seg_q + b) : 0;
  constexpr int kPasses = (Sm::kMaxCI * C + kThreads - 1) / kThreads;
  int segk[kPasses];
  if (p.seg_k) {
#pragma unroll
    for (int ps = 0; ps < kPasses; ++ps) {
      const int i = ps * (kThreads / C) + tid / C, t = tid % C;
      const int j = (split + NS * i) * C + t;
      segk[ps] = (i < nci && j < p.Lk) ? __ldg(p.seg_k + (int64_t)b * p.Lk + j) : -1;
    }
  }
  int kvl = kvl_raw;
  if (kvl < 0 || kvl > p.Lk) {
    if (split == 0 && hg == 0 && tid == 0) report_error(p.err, MGQA_ERR_INVALID_ARG);
    kvl = kvl < 0 ? 0 : p.Lk;
  }
  // append: the new row sits at slot `pos`, and the step attends to it too;
  // a full cache (kv_len == Lk) is an error and appends nothing
  int pos = -1;
  if (p.append) {
    if (kvl < p.Lk) {
      pos = kvl;
      kvl += 1;
    } else if (split == 0 && hg == 0 && tid == 0) {
      report_error(p.err, MGQA_ERR_INVALID_ARG);
    }
    if (p.kv_len_out && split == 0 && hg == 0 && tid == 0) p.kv_len_out[b] = kvl;
  }
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int i = tid + u * kThreads;
    if (i < NREP * D) sm.q[i / D][i % D] = qv[u];
  }
  __syncthreads();  // mask words

  // allowed-slot words (one thread per slot, ballots); the chunk counts
#pragma unroll
  for (int ps = 0; ps < kPasses; ++ps) {
    const int i = ps * (kThreads / C) + tid / C, t = tid % C;
    if (ps * (kThreads / C) >= nci) break;  // CTA-uniform
    const int j = (split + NS * i) * C + t;
    bool a = i < nci && j < p.Lk && j < kvl;
    if (p.bits && i < nci) a = a && ((sm.words[i][t >> 5] >> (t & 31)) & 1u);
    if (p.seg_k) a = a && segq >= 0 && segk[ps] == segq;
    const uint32_t word = __ballot_sync(0xffffffffu, a);
    __syncwarp();  // every lane has read its mask word before lane 0 overwrites it
    if (lane == 0 && i < nci) sm.words[i][t >> 5] = word;
  }
  __syncthreads();
  // prefix of the chunk counts (one warp; nci <= kMaxCI <= 64)
  if (warp == 0) {
    int run = 0;
    for (int c0 = 0; c0 < nci; c0 += 32) {
      const int i = c0 + lane;
      const int cnt = i < nci ? __popc(sm.words[i][0]) + __popc(sm.words[i][1]) : 0;
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (i < nci) sm.base[i] = run + incl - cnt;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) sm.n_all = run;
  }
  __syncthreads();
  // dense list of allowed slots, ascending
  for (int ps = 0; ps * (kThreads / C) < nci; ++ps) {
    const int i = ps * (kThreads / C) + tid / C, t = tid % C;
    if (i < nci) {
      const uint32_t wd = sm.words[i][t >> 5];
      if ((wd >> (t & 31)) & 1u) {
        const int rk = sm.base[i] + (t >= 32 ? __popc(sm.words[i][0]) : 0) +
                       __popc(wd & ((1u << (t & 31)) - 1u));
        sm.slot[rk] = (uint16_t)(i * C + t);
      }
    }
  }
  __syncthreads();
  const int n_all = sm.n_all;
  const int nbatch = (n_all + CAPB - 1) / CAPB;

  // ---- 2-3. batches of dense rows, two in flight
  const T *kg = static_cast<const T *>(p.k) + (int64_t)b * p.ks_b + (int64_t)g * p.ks_h;
  const T *vg = static_cast<const T *>(p.v) + (int64_t)b * p.vs_b + (int64_t)g * p.vs_h;
  for (int bt = 0; bt < 2 && bt < nbatch; ++bt) {
    gather_batch<T, D, NREP, SC>(sm, p, bt, bt * CAPB, min(CAPB, n_all - bt * CAPB), kg, vg, split,
                                 NS, b, g, pos);
    cp_async_commit();
  }

  constexpr int EPL = 16 / sizeof(T);  // elements per 16-byte lane load (fp32 path)
  constexpr int GL = D / EPL;          // lanes per row
  constexpr int SPW = 32 / GL;         // rows per warp pass
  constexpr int ROWS_W = CAPB / kWarps;
  static_assert(GL <= 32 && (Sm::kMma || ROWS_W % SPW == 0), "lane layout");
  constexpr int ITEMS = (NREP * D / 2 + kThreads - 1) / kThreads;  // (head, dim pair) per thread
  float o[ITEMS][2];
#pragma unroll
  for (int u = 0; u < ITEMS; ++u) o[u][0] = o[u][1] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // meaningful in warp r < NREP
  const int e = lane % GL, sub = lane / GL;
  // tensor-core path: Q as the A fragment (heads gq < NREP; rows gq + 8 are padding)
  constexpr int RW = 16;  // dense rows per compute warp per batch
  const int gq = lane >> 2, tq = lane & 3;
  uint32_t qa[Sm::kMma ? D / 16 : 1][2];
  float ow[Sm::kMma ? D / 8 : 1][4];
  float wm_run = -INFINITY, wl_run = 0.f;
  if constexpr (Sm::kMma) {
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

  for (int bt = 0; bt < nbatch; ++bt) {
    const int buf = bt & 1;
    const int nb = min(CAPB, n_all - bt * CAPB);
    if (bt + 1 < nbatch) cp_async_wait<1>(); else cp_async_wait<0>();
    __syncthreads();  // batch bt landed for every thread

    if constexpr (Sm::kMma) {
      // warp w owns dense rows [w*16, w*16 + 16) of the batch and keeps its
      // own running (m, l, O) for head gq; warps merge after the last batch
      const int r0 = warp * RW;
      if (warp < Sm::CW && r0 < nb) {
        const int n8 = min(2, (nb - r0 + 7) / 8);  // 8-row tiles holding a valid row
        float c[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
          if (nt >= n8) continue;  // warp-uniform
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const T *kr = &sm.u.r.k[buf][r0 + nt * 8 + gq][kk * 16 + 2 * tq];
            mma_16816<T>(c[nt], qa[kk][0], 0u, qa[kk][1], 0u,
                         *reinterpret_cast<const uint32_t *>(kr),
                         *reinterpret_cast<const uint32_t *>(kr + 8));
          }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
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
        uint32_t pa[2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
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
        for (int dt = 0; dt < D / 8; ++dt) {
          uint32_t b0, b1;
          ldmatrix_x2_trans(b0, b1, &sm.u.r.v[buf][r0 + (lane & 15)][dt * 8]);
          mma_16816<T>(ow[dt], pa[0], 0u, pa[1], 0u, b0, b1);
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
            const uint4 uu = *reinterpret_cast<const uint4 *>(&sm.u.r.k[buf][row][e * EPL]);
            float kf[EPL];
            unpack16_t<T>(uu, kf);
#pragma unroll
            for (int r = 0; r < NREP; ++r)
#pragma unroll
              for (int i = 0; i < EPL; ++i) acc[r] = fmaf(qr[r][i], kf[i], acc[r]);
          }
#pragma unroll
          for (int off = GL / 2; off > 0; off >>= 1)
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
            const float2 vv = *reinterpret_cast<const float2 *>(&sm.u.r.v[buf][kk][2 * dp]);
            a0 = fmaf(pr, vv.x, a0);
            a1 = fmaf(pr, vv.y, a1);
          }
          o[u][0] = o[u][0] * sm.fo[r] + a0 * sm.fb[r];
          o[u][1] = o[u][1] * sm.fo[r] + a1 * sm.fb[r];
        }
      }
    }
    __syncthreads();  // buffer `buf` (and the scores) are free again
    if (bt + 2 < nbatch) {
      gather_batch<T, D, NREP, SC>(sm, p, buf, (bt + 2) * CAPB, min(CAPB, n_all - (bt + 2) * CAPB),
                                   kg, vg, split, NS, b, g, pos);
      cp_async_commit();
    }
  }

  if constexpr (Sm::kMma) {
    // in-CTA merge of the compute warps' (m, l, O), ascending warp order (the
    // row buffers are free: every batch has been consumed)
    if (warp < Sm::CW && gq < NREP) {
      if (tq == 0) {
        sm.u.w.m[warp][gq] = wm_run;
        sm.u.w.l[warp][gq] = wl_run;
      }
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) {
        sm.u.w.o[warp][gq][dt * 8 + 2 * tq] = ow[dt][0];
        sm.u.w.o[warp][gq][dt * 8 + 2 * tq + 1] = ow[dt][1];
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
        for (int w = 0; w < Sm::CW; ++w) M = fmaxf(M, sm.u.w.m[w][r]);
        float a0 = 0.f, a1 = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < Sm::CW; ++w) {
            if (sm.u.w.m[w][r] == -INFINITY) continue;
            const float wt = exp2f(sm.u.w.m[w][r] - M);
            a0 = fmaf(sm.u.w.o[w][r][2 * dp], wt, a0);
            a1 = fmaf(sm.u.w.o[w][r][2 * dp + 1], wt, a1);
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
      for (int w = 0; w < Sm::CW; ++w) M = fmaxf(M, sm.u.w.m[w][r]);
      float L = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < Sm::CW; ++w)
          if (sm.u.w.m[w][r] != -INFINITY) L = fmaf(sm.u.w.l[w][r], exp2f(sm.u.w.m[w][r] - M), L);
      }
      m_run = M;
      l_run = L;
    }
  }

  // append: the CTA owning slot pos stores the new row into the cache (once
  // per KV head: only its first head group); no CTA of this step reads that
  // slot from the cache
  if (pos >= 0 && (pos / C) % NS == split && h0 % p.n_rep == 0) {
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

  // ---- 4. this CTA's partial into its shared memory; cluster merge
#pragma unroll
  for (int u = 0; u < ITEMS; ++u) {
    const int idx = tid + u * kThreads;
    if (idx < NREP * D / 2) {
      const int r = idx / (D / 2), dp = idx % (D / 2);
      sm.po[r][2 * dp] = o[u][0];
      sm.po[r][2 * dp + 1] = o[u][1];
    }
  }
  if (warp < NREP && lane == 0) {
    sm.pm[warp] = m_run;
    sm.pl[warp] = (m_run == -INFINITY) ? 0.f : l_run;
  }
  cluster_sync();  // every CTA's partial is visible cluster-wide
  constexpr int PER = NREP * D / SC;  // outputs merged by each CTA of the cluster
  static_assert(PER >= 1 && PER <= kThreads, "merge slice");
  const int64_t hrow = (int64_t)b * p.Hq + h0;  // output row of head h0
  if (tid < PER) {
    const int oi = rank * PER + tid;
    const int h = oi / D, d = oi % D;
    float mv[SC], lv[SC], ov[SC];
#pragma unroll
    for (int xx = 0; xx < SC; ++xx) {  // all loads in flight at once
      mv[xx] = ld_cluster_f32(cluster_map(&sm.pm[h], xx));
      lv[xx] = ld_cluster_f32(cluster_map(&sm.pl[h], xx));
      ov[xx] = ld_cluster_f32(cluster_map(&sm.po[h][d], xx));
    }
    float M = -INFINITY;
#pragma unroll
    for (int xx = 0; xx < SC; ++xx) M = fmaxf(M, mv[xx]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int xx = 0; xx < SC; ++xx) {
        if (mv[xx] == -INFINITY) continue;
        const float w = exp2f(mv[xx] - M);
        L = fmaf(lv[xx], w, L);
        acc = fmaf(ov[xx], w, acc);
      }
    }
    if (p.G == 1) {
      T *orow = static_cast<T *>(p.out) + (int64_t)b * p.os_b + (int64_t)(h0 + h) * p.os_h;
      orow[d] = from_float<T>(L > 0.f ? acc / L : 0.f);
      if (d == 0 && p.lse) p.lse[hrow + h] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
    } else {
      const int64_t wr = (hrow + h) * p.G + cl;
      p.ws_o[wr * D + d] = acc;
      if (d == 0) p.ws_ml[wr] = make_float2(M, L);
      __threadfence();  // visible GPU-wide before this CTA takes its ticket
    }
  }
  cluster_sync();  // no CTA leaves while another may still read its shared memory
  if (p.G == 1) return;

  // G > 1: the last of the NS CTAs merges the G cluster partials
  __syncthreads();
  unsigned *tick = p.ws_tick + (int64_t)b * (p.Hq / NREP) + hg;
  if (tid == 0) {
    unsigned t;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(t) : "l"(tick) : "memory");
    sm.is_last = (t == (unsigned)(NS - 1));
  }
  __syncthreads();
  if (!sm.is_last) return;
  for (int oi = tid; oi < NREP * D; oi += kThreads) {
    const int h = oi / D, d = oi % D;
    const int64_t wr0 = (hrow + h) * p.G;
    float M = -INFINITY;
    for (int c2 = 0; c2 < p.G; ++c2) M = fmaxf(M, __ldcg(&p.ws_ml[wr0 + c2].x));
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
      for (int c2 = 0; c2 < p.G; ++c2) {
        const float2 ml = __ldcg(&p.ws_ml[wr0 + c2]);
        if (ml.x == -INFINITY) continue;
        const float w = exp2f(ml.x - M);
        L = fmaf(ml.y, w, L);
        acc = fmaf(__ldcg(&p.ws_o[(wr0 + c2) * D + d]), w, acc);
      }
    }
    T *orow = static_cast<T *>(p.out) + (int64_t)b * p.os_b + (int64_t)(h0 + h) * p.os_h;
    orow[d] = from_float<T>(L > 0.f ? acc / L : 0.f);
    if (d == 0 && p.lse) p.lse[hrow + h] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
  if (tid == 0) *tick = 0u;
}

// Cluster size the device can co-schedule for this kernel: 16 (non-portable)
// when at least one such cluster fits, else 8. Decided once per device.
template <typename T, int D, int NREP>
int cluster_size_for_device() {
  static std::atomic<uint64_t> known{0}, is16{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 8;
  const uint64_t bit = 1ull << dev;
  if (known.load(std::memory_order_acquire) & bit)
    return (is16.load(std::memory_order_relaxed) & bit) ? 16 : 8;
  auto kern = decode_kernel<T, D, NREP, 16>;
  const size_t smem = sizeof(DecodeSmem<T, D, NREP, 16>);
  int n = 0;
  bool ok16 = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                  cudaSuccess &&
              cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) ==
                  cudaSuccess;
  if (ok16) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16, 1, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ok16 = cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0;
  }
  if (!ok16) (void)cudaGetLastError();  // a refused query leaves no error behind
  if (ok16) is16.fetch_or(bit, std::memory_order_relaxed);
  known.fetch_or(bit, std::memory_order_release);
  return ok16 ? 16 : 8;
}

template <typename T, int D, int NREP, int SC>
mgqa_status launch_t(const DecodeParams &p, cudaStream_t s) {
  auto kern = decode_kernel<T, D, NREP, SC>;
  const size_t smem = sizeof(DecodeSmem<T, D, NREP, SC>);
  static std::atomic<uint64_t> attr_done{0};
  const mgqa_status st = ensure_smem_attr(kern, (int)smem, attr_done, "decode kernel");
  if (st != MGQA_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(SC * p.G, p.Hq / NREP, p.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = SC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return MGQA_OK;
}

template <typename T, int D, int NREP>
mgqa_status launch_sc(const DecodeParams &p, cudaStream_t s) {
  if (cluster_size_for_device<T, D, NREP>() == 16) return launch_t<T, D, NREP, 16>(p, s);
  return launch_t<T, D, NREP, 8>(p, s);
}

template <typename T, int D>
mgqa_status launch_nrep(const DecodeParams &p, int hpc, cudaStream_t s) {
  switch (hpc) {
    case 1: return launch_sc<T, D, 1>(p, s);
    case 2: return launch_sc<T, D, 2>(p, s);
    case 4: return launch_sc<T, D, 4>(p, s);
    case 8: return launch_sc<T, D, 8>(p, s);
    default: return fail(MGQA_ERR_UNSUPPORTED, "decode: heads per CTA %d", hpc);
  }
}

}  // namespace

// Clusters per (request, head group). One cluster of 16 reads at most 2048
// rows per CTA of a 32768-slot cache; more clusters pay only when the grid
// would otherwise leave most SMs idle and each CTA would gather over 1024 rows.
int decode_clusters_per_group(const mgqa_args &a, int hpc) {
  const int nch = (a.Lk + kDecodeChunk - 1) / kDecodeChunk;
  const int64_t groups = (int64_t)a.B * (a.Hq / hpc);
  int G = 1;
  while (G < 8 && groups <= (int64_t)(kDecodeTicketBytes / sizeof(unsigned)) &&
         groups * kDecodeCluster * (2 * G) <= 2 * 152 &&
         (int64_t)((nch + kDecodeCluster * G - 1) / (kDecodeCluster * G)) * kDecodeChunk > 1024)
    G *= 2;
  return G;
}

// The workspace holds the merge tickets and cluster partials of G > 1 calls;
// a G = 1 call (the usual one) leaves it untouched. The tickets sit in a fixed
// region at offset 0 that nothing else ever writes and every call returns to
// zero, so a workspace zeroed once serves later calls of any shape.
DecodeWsLayout decode_ws_layout(const mgqa_args &a) {
  const int hpc = decode_heads_per_cta(a.Hq / a.Hkv);
  const int G = decode_clusters_per_group(a, hpc);
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  DecodeWsLayout w;
  w.G = G;
  w.tick = 0;
  w.ml = kDecodeTicketBytes;
  if (G == 1) {
    w.o = w.total = w.ml;
    return w;
  }
  const size_t rows = (size_t)a.B * a.Hq * G;
  w.o = w.ml + up(rows * sizeof(float2));
  w.total = w.o + up(rows * a.D * sizeof(float));
  return w;
}

int decode_heads_per_cta(int n_rep) {
  for (int h : {8, 4, 2, 1})
    if (n_rep % h == 0) return h;
  return 1;
}

size_t decode_workspace_bytes(const mgqa_args &a) { return decode_ws_layout(a).total; }

mgqa_status launch_decode(const mgqa_args &a, void *ws, size_t ws_bytes, cudaStream_t s) {
  return launch_decode_append(a, nullptr, nullptr, nullptr, nullptr, nullptr, ws, ws_bytes, s);
}

mgqa_status launch_decode_append(const mgqa_args &a, const void *k_new, const void *v_new,
                                 const int64_t *k_new_stride, const int64_t *v_new_stride,
                                 int32_t *kv_len_out, void *ws, size_t ws_bytes, cudaStream_t s) {
  const DecodeWsLayout L = decode_ws_layout(a);
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
  const int hpc = decode_heads_per_cta(p.n_rep);
  p.G = L.G;
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
// cluster partials and merge tickets of a call live in one fixed array that
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
  // The merge tickets must start at zero. The array is zero when the library
  // loads and every call returns its tickets to zero, but a call cut short
  // (its process or context lost mid-kernel) would not: calls that merge
  // through the array clear the ticket region on the caller's stream first
  // (calls that merge inside one cluster never touch the array).
  const mgqa::DecodeWsLayout lay = mgqa::decode_ws_layout(*args);
  if (lay.G > 1 &&
      cudaMemsetAsync(static_cast<char *>(ws) + lay.tick, 0, mgqa::kDecodeTicketBytes, stream) !=
          cudaSuccess)
    return mgqa::fail(MGQA_ERR_CUDA, "clearing the decode scratch tickets failed");
  return masked_gqa_attn_decode(args, ws, mgqa::kStaticScratchBytes, stream);
}
