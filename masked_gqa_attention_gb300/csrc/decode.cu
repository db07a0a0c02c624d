// One-query attention over a static KV cache (split over fixed chunks of
// absolute cache slots, merged by log-sum-exp in the same launch).
//
// Passages: VoxCPM page, "Upstream-identical practice", attention bullet
// (decode against the static cache under an explicit boolean mask; slots past
// the current length are masked and add exact zeros) and "Memory & speed",
// attention_span paragraph (attend only to the filled blocks of the 8192-slot
// cache instead of all of it).
//
// Design: CTA (chunk c, head group hg, batch b) owns cache slots
// [c*C, c*C + C) for the NREP query heads of one KV head.
//   1. Each thread tests one slot against every mask form; a warp ballot
//      gives the chunk's allowed-slot bitmap. An empty chunk reads no K/V.
//   2. Every allowed slot's K row and V row is fetched with one untiled bulk
//      copy each (TMA engine) into shared memory; masked slots are never read.
//   3. Scores: D/8 (bf16) lanes share a slot, each holding 16 bytes of the
//      row; NREP dot products per lane, butterfly-summed across the lanes.
//   4. Per head: chunk max, exp2, sum (one warp per head).
//   5. P.V: one thread per (head, pair of dims) walks the chunk's allowed
//      slots in ascending order.
//   6. The partial (m, l, o) goes to the workspace; the CTA that takes the
//      last ticket of (b, hg) merges all chunks in ascending chunk order and
//      resets the ticket. Empty chunks publish m = -inf and are skipped.
// All sums run in a fixed order, so the bits depend only on which slots are
// allowed: a full-cache bitmask and the equivalent filled length agree bit
// for bit.
#include <cfloat>
#include <cmath>

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
  float scale_log2;
  float *lse;
  int32_t *err;
  int B, Hq, Hkv, Lk, n_rep, nch;
  float2 *ws_ml;      // [B][Hq][nch]   (m in log2 units, l)
  float *ws_o;        // [B][Hq][nch][D] unnormalised partial outputs
  unsigned *ws_tick;  // [B][Hq/NREP]
};

constexpr int kThreads = 256;

template <typename T, int D, int NREP, int C>
struct DecodeSmem {
  alignas(128) T k[C][D];
  alignas(128) T v[C][D];
  float q[NREP][D];
  float s[NREP][C];
  uint32_t allowed[C / 32];
  float2 ml[NREP];
  uint64_t bar;
  int n_allowed;
  int is_last;
};

template <typename T, int D, int NREP, int C>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const __grid_constant__ DecodeParams p) {
  static_assert(C % 32 == 0 && C <= kThreads, "chunk size");
  extern __shared__ __align__(128) unsigned char smem_raw[];
  auto &sm = *reinterpret_cast<DecodeSmem<T, D, NREP, C> *>(smem_raw);

  const int c = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h0 = hg * NREP;
  const int g = h0 / p.n_rep;
  const int j0 = c * C;
  const int64_t row0 = ((int64_t)b * p.Hq + h0) * p.nch + c;  // ws row of head h0

  // 1. allowed-slot bitmap of this chunk
  const int kvl = load_kv_len(p.kv_len, b, p.Lk, p.err, c == 0 && hg == 0 && tid == 0);
  bool a = false;
  const int j = j0 + tid;
  if (tid < C && j < p.Lk) {
    a = true;
    if (p.bits) a = (__ldg(p.bits + (int64_t)b * p.ms_b + (j >> 5)) >> (j & 31)) & 1u;
    if (p.kv_len) a = a && (j < kvl);
    if (p.seg_q) {
      const int sq = __ldg(p.seg_q + b);
      a = a && sq >= 0 && __ldg(p.seg_k + (int64_t)b * p.Lk + j) == sq;
    }
  }
  const uint32_t word = __ballot_sync(0xffffffffu, a);
  if (lane == 0 && warp < C / 32) sm.allowed[warp] = word;
  if (tid == 0) {
    mbar_init(&sm.bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    int n = 0;
#pragma unroll
    for (int w = 0; w < C / 32; ++w) n += __popc(sm.allowed[w]);
    sm.n_allowed = n;
    if (n > 0) mbar_arrive_expect_tx(&sm.bar, (uint32_t)(n * 2 * D * sizeof(T)));
  }
  __syncthreads();
  const int n_allowed = sm.n_allowed;

  if (n_allowed > 0) {
    // 2. fetch exactly the allowed K/V rows
    if (a) {
      const T *kr = static_cast<const T *>(p.k) + (int64_t)b * p.ks_b + (int64_t)g * p.ks_h +
                    (int64_t)j * p.ks_l;
      const T *vr = static_cast<const T *>(p.v) + (int64_t)b * p.vs_b + (int64_t)g * p.vs_h +
                    (int64_t)j * p.vs_l;
      bulk_g2s(&sm.k[tid][0], kr, D * sizeof(T), &sm.bar);
      bulk_g2s(&sm.v[tid][0], vr, D * sizeof(T), &sm.bar);
    }
    const T *qb = static_cast<const T *>(p.q) + (int64_t)b * p.qs_b;
    for (int i = tid; i < NREP * D; i += kThreads) {
      const int r = i / D, d = i % D;
      sm.q[r][d] = to_float(qb[(int64_t)(h0 + r) * p.qs_h + d]);
    }
    __syncthreads();
    const bool ok = mbar_wait(&sm.bar, 0, p.err);

    // 3. scores (log2 units)
    constexpr int EPL = 16 / sizeof(T);  // elements per 16-byte lane load
    constexpr int G = D / EPL;           // lanes per slot
    constexpr int SPW = 32 / G;          // slots per warp pass
    constexpr int SLOTS_W = C / (kThreads / 32);
    static_assert(G <= 32 && SLOTS_W % SPW == 0, "lane layout");
    const int e = lane % G, sub = lane / G;
    float qr[NREP][EPL];
#pragma unroll
    for (int r = 0; r < NREP; ++r)
#pragma unroll
      for (int i = 0; i < EPL; ++i) qr[r][i] = sm.q[r][e * EPL + i];
#pragma unroll 2
    for (int it = 0; it < SLOTS_W / SPW; ++it) {
      const int sl = warp * SLOTS_W + it * SPW + sub;
      const bool al = ok && ((sm.allowed[sl >> 5] >> (sl & 31)) & 1u);
      float acc[NREP];
#pragma unroll
      for (int r = 0; r < NREP; ++r) acc[r] = 0.f;
      if (al) {
        const uint4 u = *reinterpret_cast<const uint4 *>(&sm.k[sl][e * EPL]);
        float kf[EPL];
        unpack16(u, kf);
#pragma unroll
        for (int r = 0; r < NREP; ++r)
#pragma unroll
          for (int i = 0; i < EPL; ++i) acc[r] = fmaf(qr[r][i], kf[i], acc[r]);
      }
#pragma unroll
      for (int off = G / 2; off > 0; off >>= 1)
#pragma unroll
        for (int r = 0; r < NREP; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
      if (e == 0) {
#pragma unroll
        for (int r = 0; r < NREP; ++r) sm.s[r][sl] = al ? acc[r] * p.scale_log2 : -INFINITY;
      }
    }
    __syncthreads();

    // 4. per-head chunk max and sum
    for (int r = warp; r < NREP; r += kThreads / 32) {
      float m = -INFINITY;
#pragma unroll
      for (int i = lane; i < C; i += 32) m = fmaxf(m, sm.s[r][i]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      float l = 0.f;
#pragma unroll
      for (int i = lane; i < C; i += 32) {
        const float x = sm.s[r][i];
        const float pr = (x == -INFINITY) ? 0.f : exp2f(x - m);
        sm.s[r][i] = pr;
        l += pr;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
      if (lane == 0) sm.ml[r] = make_float2(m, l);
    }
    __syncthreads();

    // 5. P.V over the allowed slots, ascending
    for (int idx = tid; idx < NREP * D / 2; idx += kThreads) {
      const int r = idx / (D / 2), dp = idx % (D / 2);
      float o0 = 0.f, o1 = 0.f;
      for (int w = 0; w < C / 32; ++w) {
        uint32_t bitsw = ok ? sm.allowed[w] : 0u;
        while (bitsw) {
          const int sl = w * 32 + __ffs(bitsw) - 1;
          bitsw &= bitsw - 1;
          const float pr = sm.s[r][sl];
          float v0, v1;
          if constexpr (sizeof(T) == 2) {
            const __nv_bfloat162 vv = *reinterpret_cast<const __nv_bfloat162 *>(&sm.v[sl][2 * dp]);
            v0 = __low2float(vv);
            v1 = __high2float(vv);
          } else {
            const float2 vv = *reinterpret_cast<const float2 *>(&sm.v[sl][2 * dp]);
            v0 = vv.x;
            v1 = vv.y;
          }
          o0 = fmaf(pr, v0, o0);
          o1 = fmaf(pr, v1, o1);
        }
      }
      reinterpret_cast<float2 *>(p.ws_o + (row0 + (int64_t)r * p.nch) * D)[dp] =
          make_float2(o0, o1);
    }
    if (tid < NREP) p.ws_ml[row0 + (int64_t)tid * p.nch] = ok ? sm.ml[tid] : make_float2(-INFINITY, 0.f);
  } else {
    if (tid < NREP) p.ws_ml[row0 + (int64_t)tid * p.nch] = make_float2(-INFINITY, 0.f);
  }

  // 6. ticket; the last CTA of (b, hg) merges every chunk
  __threadfence();
  __syncthreads();
  unsigned *tick = p.ws_tick + (int64_t)b * (p.Hq / NREP) + hg;
  if (tid == 0) {
    const unsigned t = atomicAdd(tick, 1u);
    sm.is_last = (t == (unsigned)(gridDim.x - 1));
    __threadfence();
  }
  __syncthreads();
  if (!sm.is_last) return;

  for (int idx = tid; idx < NREP * D / 2; idx += kThreads) {
    const int r = idx / (D / 2), dp = idx % (D / 2);
    const int64_t hrow = ((int64_t)b * p.Hq + h0 + r) * p.nch;
    float M = -INFINITY;
    for (int cc = 0; cc < p.nch; ++cc) M = fmaxf(M, __ldcg(&p.ws_ml[hrow + cc]).x);
    float L = 0.f, o0 = 0.f, o1 = 0.f;
    if (M != -INFINITY) {
      for (int cc = 0; cc < p.nch; ++cc) {
        const float2 ml = __ldcg(&p.ws_ml[hrow + cc]);
        if (ml.x == -INFINITY) continue;
        const float w = exp2f(ml.x - M);
        const float2 o = __ldcg(reinterpret_cast<const float2 *>(p.ws_o + (hrow + cc) * D) + dp);
        L = fmaf(ml.y, w, L);
        o0 = fmaf(o.x, w, o0);
        o1 = fmaf(o.y, w, o1);
      }
    }
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
    T *orow = static_cast<T *>(p.out) + (int64_t)b * p.os_b + (int64_t)(h0 + r) * p.os_h;
    orow[2 * dp] = from_float<T>(o0 * inv);
    orow[2 * dp + 1] = from_float<T>(o1 * inv);
    if (dp == 0 && p.lse)
      p.lse[(int64_t)b * p.Hq + h0 + r] = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
  if (tid == 0) *tick = 0u;
}

template <typename T, int D, int NREP>
mgqa_status launch_t(const DecodeParams &p, cudaStream_t s) {
  constexpr int C = kDecodeChunk;
  auto kern = decode_kernel<T, D, NREP, C>;
  const size_t smem = sizeof(DecodeSmem<T, D, NREP, C>);
  static bool attr_set = false;  // per process; the attribute is per function
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return fail(MGQA_ERR_CUDA, "cudaFuncSetAttribute failed for the decode kernel");
    attr_set = true;
  }
  dim3 grid(p.nch, p.Hq / NREP, p.B);
  kern<<<grid, kThreads, smem, s>>>(p);
  const cudaError_t e = cudaGetLastError();
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
  const int nch = (a.Lk + kDecodeChunk - 1) / kDecodeChunk;
  const size_t rows = (size_t)a.B * a.Hq * nch;
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
  const int hpc = decode_heads_per_cta(p.n_rep);
  if (a.dtype == MGQA_BF16) {
    if (a.D == 64) return launch_nrep<__nv_bfloat16, 64>(p, hpc, s);
    if (a.D == 128) return launch_nrep<__nv_bfloat16, 128>(p, hpc, s);
  } else {
    if (a.D == 64) return launch_nrep<float, 64>(p, hpc, s);
    if (a.D == 128) return launch_nrep<float, 128>(p, hpc, s);
  }
  return fail(MGQA_ERR_UNSUPPORTED, "decode: head dim %d", a.D);
}

}  // namespace mgqa
