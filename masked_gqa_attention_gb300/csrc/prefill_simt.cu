// Full-sequence masked GQA attention on the CUDA cores, fp32 arithmetic.
// Serves fp32 inputs, where tensor-core tf32 (10-bit mantissa) cannot meet a
// 1e-5 relative bound.
//
// Passages: VoxCPM page, "Upstream-identical practice", attention bullet
// (SDPA with enable_gqa, bidirectional, explicit boolean mask); OmniVoice
// page, "Upstream-identical practice", attention-mask bullet (4D boolean
// mask, not causal, KV heads repeated) and "Memory & speed", packed_guidance
// paragraph (block-diagonal mask).
//
// CTA = 32 query rows of one query head; four threads per row, each owning a
// quarter of the head dim. Keys advance in tiles of 64, double-buffered in
// shared memory (tile j+1 is fetched by asynchronous copies while tile j is
// computed); a tile no row of the CTA may attend to is not computed. The 64
// scores of a row are formed from 16-byte shared-memory reads (the quarters
// summed with two shuffles), masked to -inf, and folded into a running (max,
// sum, O) with one rescale per tile.
// (Two threads per row and 4-byte reads measured 24.9 us on the tiny case:
// every row re-reads the whole tile, so the shared-memory load instructions
// were the limit.)
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace mgqa {
namespace {

struct SimtParams {
  const void *q, *k, *v;
  void *out;
  int64_t qs[3], ks[3], vs[3], os[3];
  MaskView mask;
  float scale_log2;
  float *lse;
  int32_t *err;
  int B, Hq, Hkv, Lq, Lk, n_rep;
};

constexpr int kRows = 32;
constexpr int kKeys = 64;
constexpr int kTpr = 4;  // threads per row
constexpr int kThreads = kTpr * kRows;
// Shared-memory row of a K or V tile: the four quarters of the head dim, each
// followed by 4 floats of padding, so the four threads of a row read four
// different bank groups.
template <int D> __host__ __device__ constexpr int row_floats() { return kTpr * (D / kTpr + 4); }

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
prefill_simt_kernel(const __grid_constant__ SimtParams p) {
  extern __shared__ __align__(16) float sh[];
  constexpr int DH = D / kTpr;  // head-dim elements per thread
  constexpr int RF = row_floats<D>();

  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / p.n_rep;
  const int tid = threadIdx.x;
  const int row = tid / kTpr, part = tid % kTpr;
  const int i = qt * kRows + row;
  const bool row_ok = i < p.Lq;
  const int ic = row_ok ? i : p.Lq - 1;

  const int kvl = load_kv_len(p.mask.kv_len, b, p.Lk, p.err, qt == 0 && h == 0 && tid == 0);
  const int segq = p.mask.seg_q ? __ldg(p.mask.seg_q + (int64_t)b * p.Lq + ic) : 0;

  float q[DH], o[DH];
  const T *qrow = static_cast<const T *>(p.q) + b * p.qs[0] + h * p.qs[1] + (int64_t)ic * p.qs[2];
#pragma unroll
  for (int d = 0; d < DH; ++d) {
    q[d] = to_float(qrow[part * DH + d]) * p.scale_log2;
    o[d] = 0.f;
  }
  float m = -INFINITY, l = 0.f;

  const T *kb = static_cast<const T *>(p.k) + b * p.ks[0] + g * p.ks[1];
  const T *vb = static_cast<const T *>(p.v) + b * p.vs[0] + g * p.vs[1];

  // K and V tiles in two shared-memory buffers: tile j+1's rows are fetched
  // (16-byte asynchronous copies) and its mask words loaded while tile j is
  // computed
  auto buf_k = [&](int bf) { return sh + bf * 2 * kKeys * RF; };
  auto buf_v = [&](int bf) { return sh + bf * 2 * kKeys * RF + kKeys * RF; };
  auto fetch = [&](int j0, int bf) {
    constexpr int PV = kKeys * D / 4 / kThreads;  // 16-byte pieces of K (and of V) per thread
    float *kd = buf_k(bf), *vd = buf_v(bf);
#pragma unroll
    for (int u = 0; u < PV; ++u) {
      const int e = (tid + u * kThreads) * 4;
      const int jj = e / D, d = e % D, j = j0 + jj;
      const int off = jj * RF + (d / DH) * (DH + 4) + d % DH;
      if (j < p.Lk) {  // rows are 16-byte aligned: the ABI's stride rule
        cp_async16(kd + off, kb + (int64_t)j * p.ks[2] + d);
        cp_async16(vd + off, vb + (int64_t)j * p.vs[2] + d);
      } else {
        *reinterpret_cast<float4 *>(kd + off) = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(vd + off) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    cp_async_commit();
  };
  auto mask_words = [&](int j0, uint32_t (&mw)[kKeys / 32]) {
#pragma unroll
    for (int w = 0; w < kKeys / 32; ++w)
      mw[w] = row_ok ? mask_word(p.mask, b, ic, j0 + 32 * w, p.Lk, p.Lq, kvl, segq) : 0u;
  };

  uint32_t mw[kKeys / 32] = {0u, 0u};
  if (p.Lk > 0) {
    fetch(0, 0);
    mask_words(0, mw);
  }
  for (int j0 = 0, bf = 0; j0 < p.Lk; j0 += kKeys, bf ^= 1) {
    const int jn = j0 + kKeys;
    uint32_t mwn[kKeys / 32] = {0u, 0u};
    if (jn < p.Lk) {
      fetch(jn, bf ^ 1);  // that buffer's last reader passed the barrier ending the previous tile
      mask_words(jn, mwn);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    uint32_t any = 0;
#pragma unroll
    for (int w = 0; w < kKeys / 32; ++w) any |= mw[w];
    // (also the barrier after which every thread's copies of this tile are visible)
    if (__syncthreads_or(any != 0u)) {  // an empty tile is fetched ahead but never computed
      const float *ks = buf_k(bf), *vs = buf_v(bf);
      float s[kKeys];
      float mt = -INFINITY;
#pragma unroll
      for (int jj = 0; jj < kKeys; ++jj) {
        const float4 *kr = reinterpret_cast<const float4 *>(ks + jj * RF + part * (DH + 4));
        float acc = 0.f;
#pragma unroll
        for (int d4 = 0; d4 < DH / 4; ++d4) {
          const float4 kv = kr[d4];
          acc = fmaf(q[4 * d4], kv.x, acc);
          acc = fmaf(q[4 * d4 + 1], kv.y, acc);
          acc = fmaf(q[4 * d4 + 2], kv.z, acc);
          acc = fmaf(q[4 * d4 + 3], kv.w, acc);
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        const bool al = (mw[jj >> 5] >> (jj & 31)) & 1u;
        s[jj] = al ? acc : -INFINITY;
        mt = fmaxf(mt, s[jj]);
      }
      const float m_new = fmaxf(m, mt);
      if (m_new != -INFINITY) {
        const float corr = exp2f(m - m_new);  // m == -inf gives 0
        l *= corr;
#pragma unroll
        for (int d = 0; d < DH; ++d) o[d] *= corr;
#pragma unroll
        for (int jj = 0; jj < kKeys; ++jj) {
          const float pj = exp2f(s[jj] - m_new);  // masked: exp2(-inf) = 0
          l += pj;
          const float4 *vr = reinterpret_cast<const float4 *>(vs + jj * RF + part * (DH + 4));
#pragma unroll
          for (int d4 = 0; d4 < DH / 4; ++d4) {
            const float4 vv = vr[d4];
            o[4 * d4] = fmaf(pj, vv.x, o[4 * d4]);
            o[4 * d4 + 1] = fmaf(pj, vv.y, o[4 * d4 + 1]);
            o[4 * d4 + 2] = fmaf(pj, vv.z, o[4 * d4 + 2]);
            o[4 * d4 + 3] = fmaf(pj, vv.w, o[4 * d4 + 3]);
          }
        }
        m = m_new;
      }
    }
    __syncthreads();  // this buffer is refilled two tiles later
#pragma unroll
    for (int w = 0; w < kKeys / 32; ++w) mw[w] = mwn[w];
  }

  if (row_ok) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T *orow = static_cast<T *>(p.out) + b * p.os[0] + h * p.os[1] + (int64_t)i * p.os[2];
#pragma unroll
    for (int d = 0; d < DH; ++d) orow[part * DH + d] = from_float<T>(o[d] * inv);
    if (p.lse && part == 0)
      p.lse[((int64_t)b * p.Hq + h) * p.Lq + i] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
  }
}

template <typename T, int D>
mgqa_status launch_t(const SimtParams &p, cudaStream_t s) {
  auto kern = prefill_simt_kernel<T, D>;
  const size_t smem = 2 * 2 * kKeys * row_floats<D>() * sizeof(float);  // two K/V buffers
  static std::atomic<uint64_t> attr_done{0};
  const mgqa_status st = ensure_smem_attr(kern, (int)smem, attr_done, "fp32 prefill kernel");
  if (st != MGQA_OK) return st;
  dim3 grid((p.Lq + kRows - 1) / kRows, p.Hq, p.B);
  kern<<<grid, kThreads, smem, s>>>(p);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
  return MGQA_OK;
}

}  // namespace

mgqa_status launch_prefill_simt(const mgqa_args &a, cudaStream_t s) {
  SimtParams p{};
  p.q = a.q; p.k = a.k; p.v = a.v; p.out = a.out;
  for (int t = 0; t < 3; ++t) {
    p.qs[t] = a.q_stride[t]; p.ks[t] = a.k_stride[t];
    p.vs[t] = a.v_stride[t]; p.os[t] = a.o_stride[t];
  }
  p.mask = MaskView{a.mask_bits, a.mask_stride_b, a.mask_stride_q, a.kv_len, a.seg_q, a.seg_k,
                    a.causal != 0, a.Lk - a.Lq};
  p.scale_log2 = a.scale * kLog2e;
  p.lse = a.lse; p.err = a.dev_error;
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv; p.Lq = a.Lq; p.Lk = a.Lk; p.n_rep = a.Hq / a.Hkv;
  if (a.dtype == MGQA_FP32) {
    if (a.D == 64) return launch_t<float, 64>(p, s);
    if (a.D == 128) return launch_t<float, 128>(p, s);
  }
  return fail(MGQA_ERR_UNSUPPORTED, "prefill: head dim %d", a.D);
}

}  // namespace mgqa
