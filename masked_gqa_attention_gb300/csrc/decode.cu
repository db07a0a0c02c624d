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
//   6. The partial (m, l, o) goes to the workspace. Every non-empty CTA also
//      knows which chunks of its row are non-empty (a bitmap built from the
//      mask words or the length, one word per thread), so empty CTAs exit at
//      once; the non-empty CTA that takes the last ticket of (b, hg) merges
//      the non-empty chunks in ascending order (loads issued in parallel) and
//      resets the ticket. With segment ids the bitmap would cost a scan of the
//      whole row, so there every CTA takes a ticket and empty chunks publish
//      m = -inf instead.
// All sums run in a fixed order, so the bits depend only on which slots are
// allowed: a full-cache bitmask and the equivalent filled length agree bit
// for bit.
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
  float scale_log2;
  float *lse;
  int32_t *err;
  int B, Hq, Hkv, Lk, n_rep, nch;
  float2 *ws_ml;      // [B][Hq][nch]   (m in log2 units, l)
  float *ws_o;        // [B][Hq][nch][D] unnormalised partial outputs
  unsigned *ws_tick;  // [B][Hq/NREP]
};

constexpr int kThreads = 256;
constexpr int kMaxChunks = kDecodeMaxLk / kDecodeChunk;

template <typename T, int D, int NREP, int C>
struct DecodeSmem {
  alignas(128) T k[C][D];
  alignas(128) T v[C][D];
  float q[NREP][D];
  float s[NREP][C];
  uint32_t allowed[C / 32];
  float2 ml[NREP];
  uint32_t chunk_ne[kMaxChunks / 32];  // non-empty chunks of this (b, head group)
  float w[NREP][kMaxChunks];           // merge: per-chunk m, then weights 2^(m_c - M)
  float lval[NREP][kMaxChunks];        // merge: per-chunk l
  int nz[kMaxChunks];                  // merge: non-empty chunk indices, ascending
  float inv_l[NREP];
  uint64_t bar;
  int n_allowed;
  int n_ne;
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
  const bool by_seg = p.seg_q != nullptr;
  const bool mine_ne = __syncthreads_or(a);
  // an empty chunk reads nothing and publishes nothing; chunk 0 stays to write
  // the output of a row that has no allowed slot at all
  if (!mine_ne && !by_seg && c != 0) return;

  // which chunks of this row hold an allowed slot (identical in every CTA)
  if (!by_seg) {
    for (int base = 0; base < p.nch; base += kThreads) {
      const int cc = base + tid;
      const int jb = cc * C;
      bool ne = cc < p.nch && jb < min(p.Lk, kvl);
      if (ne && p.bits) {
        uint32_t any = 0u;
#pragma unroll
        for (int w = 0; w < C / 32; ++w) {
          const int jw = jb + 32 * w;
          const int lim = min(p.Lk, kvl) - jw;
          if (lim > 0) {
            const uint32_t valid = lim >= 32 ? 0xffffffffu : ((1u << lim) - 1u);
            any |= __ldg(p.bits + (int64_t)b * p.ms_b + (jw >> 5)) & valid;
          }
        }
        ne = any != 0u;
      }
      const uint32_t bal = __ballot_sync(0xffffffffu, ne);
      if (lane == 0 && base + warp * 32 < p.nch) sm.chunk_ne[cc >> 5] = bal;
    }
  }
  __syncthreads();
  if (!mine_ne && !by_seg) {  // chunk 0, empty
    bool row_empty = true;
    for (int w = 0; w < (p.nch + 31) / 32; ++w) row_empty = row_empty && sm.chunk_ne[w] == 0u;
    if (row_empty) {
      for (int idx = tid; idx < NREP * D; idx += kThreads) {
        const int r = idx / D, d = idx % D;
        T *orow = static_cast<T *>(p.out) + (int64_t)b * p.os_b + (int64_t)(h0 + r) * p.os_h;
        orow[d] = from_float<T>(0.f);
        if (d == 0 && p.lse) p.lse[(int64_t)b * p.Hq + h0 + r] = -INFINITY;
      }
    }
    return;
  }
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

  // 6. ticket; the last non-empty CTA of (b, hg) merges the non-empty chunks
  __syncthreads();
  unsigned *tick = p.ws_tick + (int64_t)b * (p.Hq / NREP) + hg;
  if (tid == 0) {
    int n_ne = p.nch;
    if (!by_seg) {
      n_ne = 0;
      for (int w = 0; w < (p.nch + 31) / 32; ++w) n_ne += __popc(sm.chunk_ne[w]);
    }
    unsigned t;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(t) : "l"(tick) : "memory");
    sm.is_last = (t == (unsigned)(n_ne - 1));
  }
  __syncthreads();
  if (!sm.is_last) return;

  // non-empty chunk list, ascending
  if (warp == 0) {
    int count = 0;
    for (int base = 0; base < p.nch; base += 32) {
      const int cc = base + lane;
      bool ne = false;
      if (cc < p.nch) {
        if (by_seg) ne = __ldcg(&p.ws_ml[((int64_t)b * p.Hq + h0) * p.nch + cc]).x != -INFINITY;
        else ne = (sm.chunk_ne[cc >> 5] >> (cc & 31)) & 1u;
      }
      const uint32_t bal = __ballot_sync(0xffffffffu, ne);
      if (ne) sm.nz[count + __popc(bal & ((1u << lane) - 1u))] = cc;
      count += __popc(bal);
    }
    if (lane == 0) sm.n_ne = count;
  }
  __syncthreads();
  const int nnz = sm.n_ne;
  for (int idx = tid; idx < NREP * nnz; idx += kThreads) {
    const int r = idx / nnz, k = idx % nnz;
    const float2 ml = __ldcg(&p.ws_ml[((int64_t)b * p.Hq + h0 + r) * p.nch + sm.nz[k]]);
    sm.w[r][k] = ml.x;
    sm.lval[r][k] = ml.y;
  }
  __syncthreads();
  for (int r = warp; r < NREP; r += kThreads / 32) {
    float M = -INFINITY;
    for (int k = lane; k < nnz; k += 32) M = fmaxf(M, sm.w[r][k]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    for (int k = lane; k < nnz; k += 32) {
      const float m = sm.w[r][k];
      const float wgt = (m == -INFINITY) ? 0.f : exp2f(m - M);
      L = fmaf(sm.lval[r][k], wgt, L);
      sm.w[r][k] = wgt;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane == 0) {
      sm.inv_l[r] = (L > 0.f) ? 1.f / L : 0.f;
      sm.ml[r] = make_float2(M, L);
    }
  }
  __syncthreads();
  for (int idx = tid; idx < NREP * D / 2; idx += kThreads) {
    const int r = idx / (D / 2), dp = idx % (D / 2);
    const int64_t hrow = ((int64_t)b * p.Hq + h0 + r) * p.nch;
    float o0 = 0.f, o1 = 0.f;
    int k = 0;
    for (; k + 4 <= nnz; k += 4) {
      float2 o[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        o[u] = __ldcg(reinterpret_cast<const float2 *>(p.ws_o + (hrow + sm.nz[k + u]) * D) + dp);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        o0 = fmaf(o[u].x, sm.w[r][k + u], o0);
        o1 = fmaf(o[u].y, sm.w[r][k + u], o1);
      }
    }
    for (; k < nnz; ++k) {
      const float2 o = __ldcg(reinterpret_cast<const float2 *>(p.ws_o + (hrow + sm.nz[k]) * D) + dp);
      o0 = fmaf(o.x, sm.w[r][k], o0);
      o1 = fmaf(o.y, sm.w[r][k], o1);
    }
    const float inv = sm.inv_l[r];
    T *orow = static_cast<T *>(p.out) + (int64_t)b * p.os_b + (int64_t)(h0 + r) * p.os_h;
    orow[2 * dp] = from_float<T>(o0 * inv);
    orow[2 * dp + 1] = from_float<T>(o1 * inv);
    if (dp == 0 && p.lse) {
      const float2 ML = sm.ml[r];
      p.lse[(int64_t)b * p.Hq + h0 + r] = (ML.y > 0.f) ? (ML.x + log2f(ML.y)) * kLn2 : -INFINITY;
    }
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
