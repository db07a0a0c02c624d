// Rotary position embedding, in place, on q or k.
//
// Passages: F5-TTS page, module table and "Upstream-identical practice"
// (interleaved feature pairs, x-transformers; only the first pe_attn_head
// heads rotate); OmniVoice page, "Parity results" (the inverse-frequency table stays fp32) and
// VoxCPM page, "Upstream-identical practice", precision bullet (LongRoPE table
// built in fp32); OmniVoice page, "Memory & speed", packed_guidance paragraph
// (positions restart at 0 for each packed sequence).
//
// Rows of 16-byte vectors take rope_vec_kernel (below); any other layout the
// per-pair kernel: one thread per (row b, position l, pair i) forms
// theta = fl32(pos * f_i) once, takes its sine and cosine (positions reach
// thousands of radians: the shared reduced-argument sine and cosine of
// common.cuh) and rotates pair i of every rotated head at (b, l). Both are
// launched with programmatic dependent launch and read nothing before the
// grid-dependency wait (the vector and norm kernels only issue L2 prefetch
// hints for their data there, which overlap the previous kernel's tail).
// Consecutive threads take consecutive pairs, so each warp reads and writes
// whole runs of a row (interleaved: one contiguous run; half-split: two).
// The pairs of kHeadBatch heads are loaded before any is stored, so their
// loads are in flight together (a store could alias a later head's load, so
// the compiler would not hoist the loads by itself); interleaved 16-bit pairs
// move as one 32-bit word when the rows allow it.
// With a norm weight (OmniVoice page, "Parity results": the Qwen decoder
// normalises q and k separately before the rotation) one warp takes each
// rotated head vector: RMS normalisation over all D features, then the
// rotation of the first rot_dim. Both paths use the shared helpers of
// common.cuh, so the fused attention paths give the same bits.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace mgqa {
namespace {

struct RopeParams {
  void *x;
  int64_t s_b, s_h, s_l;
  const int32_t *positions;
  const float *inv_freq;
  int B, L, D, half, heads, interleaved;
  const float *norm_w;  // [D] or null
  float eps;
};

constexpr int kRopeThreads = 256;
constexpr int kHeadBatch = 8;

// the pair (x[e0], x[e1]) of one row as floats, and back
template <typename T, bool PAIRED>
MGQA_DEV void load_pair(const T *r, int e0, int e1, float &a, float &c) {
  if constexpr (PAIRED) {
    const uint32_t w = *reinterpret_cast<const uint32_t *>(r + e0);  // e1 == e0 + 1
    const T *t = reinterpret_cast<const T *>(&w);
    a = to_float(t[0]);
    c = to_float(t[1]);
  } else {
    a = to_float(r[e0]);
    c = to_float(r[e1]);
  }
}
template <typename T, bool PAIRED>
MGQA_DEV void store_pair(T *r, int e0, int e1, float a, float c) {
  if constexpr (PAIRED) {
    *reinterpret_cast<uint32_t *>(r + e0) = pack2<T>(a, c);
  } else {
    r[e0] = from_float<T>(a);
    r[e1] = from_float<T>(c);
  }
}

template <typename T, bool PAIRED>
MGQA_DEV void rope_body(const RopeParams &p, int64_t blk) {
  const int64_t idx = blk * kRopeThreads + threadIdx.x;
  const int64_t total = (int64_t)p.B * p.L * p.half;
  if (idx >= total) return;
  const int i = (int)(idx % p.half);
  const int64_t bl = idx / p.half;
  const int l = (int)(bl % p.L), b = (int)(bl / p.L);
  allow_dependents();
  grid_dependency_wait();
  const int pos = p.positions ? __ldg(p.positions + bl) : l;
  float sn, cs;
  rope_sincos(rope_theta(pos, __ldg(p.inv_freq + i)), sn, cs);
  const int e0 = p.interleaved ? 2 * i : i;
  const int e1 = p.interleaved ? 2 * i + 1 : i + p.half;
  T *row = static_cast<T *>(p.x) + (int64_t)b * p.s_b + (int64_t)l * p.s_l;
  for (int h0 = 0; h0 < p.heads; h0 += kHeadBatch) {
    float a[kHeadBatch], c[kHeadBatch];
#pragma unroll
    for (int u = 0; u < kHeadBatch; ++u)
      if (h0 + u < p.heads)
        load_pair<T, PAIRED>(row + (int64_t)(h0 + u) * p.s_h, e0, e1, a[u], c[u]);
#pragma unroll
    for (int u = 0; u < kHeadBatch; ++u)
      if (h0 + u < p.heads) {
        float y0, y1;
        rope_rotate(a[u], c[u], cs, sn, y0, y1);
        store_pair<T, PAIRED>(row + (int64_t)(h0 + u) * p.s_h, e0, e1, y0, y1);
      }
  }
}

// Rows of 16-byte vectors (the x pointer and every stride 16-byte aligned,
// the rotated span whole vectors): one thread per (row b, position l, group
// of kVecHeads heads, vector of pairs). It takes the sines and cosines of its
// pairs once, loads its vectors of every head in the group (half-split: the
// first-half vector and its second-half partner) before storing any, and
// moves 16 bytes per access; the arithmetic is the scalar kernel's.
constexpr int kVecHeads = 4;

template <typename T> MGQA_DEV void vec_to_float(const uint4 &u, float (&f)[16 / sizeof(T)]) {
  unpack16_t<T>(u, f);
}
template <typename T> MGQA_DEV uint4 vec_from_float(const float (&f)[16 / sizeof(T)]) {
  if constexpr (sizeof(T) == 4) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  } else {
    return make_uint4(pack2<T>(f[0], f[1]), pack2<T>(f[2], f[3]), pack2<T>(f[4], f[5]),
                      pack2<T>(f[6], f[7]));
  }
}

template <typename T, bool INTER>
MGQA_DEV void rope_vec_body(const RopeParams &p, int64_t blk) {
  constexpr int EPV = 16 / sizeof(T);          // elements per vector
  constexpr int PPV = INTER ? EPV / 2 : EPV;   // pairs per vector (half-split: with its partner)
  const int nvec = INTER ? 2 * p.half / EPV : p.half / EPV;
  const int ngrp = (p.heads + kVecHeads - 1) / kVecHeads;
  const int64_t idx = blk * kRopeThreads + threadIdx.x;
  if (idx >= (int64_t)p.B * p.L * ngrp * nvec) return;
  const int v = (int)(idx % nvec);
  const int64_t r = idx / nvec;
  const int grp = (int)(r % ngrp);
  const int64_t bl = r / ngrp;
  const int l = (int)(bl % p.L), b = (int)(bl / p.L);
  allow_dependents();
  const int i0 = v * PPV;              // first pair of this vector
  const int e0 = INTER ? 2 * i0 : i0;  // first element of the vector
  T *row = static_cast<T *>(p.x) + (int64_t)b * p.s_b + (int64_t)l * p.s_l;
  // hints toward the L2 before the wait (the L2 is the point of coherence,
  // so a later write by the previous kernel still wins)
#pragma unroll
  for (int u = 0; u < kVecHeads; ++u) {
    const int h = grp * kVecHeads + u;
    if (h < p.heads) {
      prefetch_l2(row + (int64_t)h * p.s_h + e0);
      if (!INTER) prefetch_l2(row + (int64_t)h * p.s_h + e0 + p.half);
    }
  }
  grid_dependency_wait();  // x, positions and the table may come from the previous kernel
  const int pos = p.positions ? __ldg(p.positions + bl) : l;
  float sn[PPV], cs[PPV];
#pragma unroll
  for (int j = 0; j < PPV; ++j) rope_sincos(rope_theta(pos, __ldg(p.inv_freq + i0 + j)), sn[j], cs[j]);
  uint4 va[kVecHeads], vb[kVecHeads];
#pragma unroll
  for (int u = 0; u < kVecHeads; ++u) {
    const int h = grp * kVecHeads + u;
    if (h < p.heads) {
      const T *hr = row + (int64_t)h * p.s_h + e0;
      va[u] = *reinterpret_cast<const uint4 *>(hr);
      if (!INTER) vb[u] = *reinterpret_cast<const uint4 *>(hr + p.half);
    }
  }
#pragma unroll
  for (int u = 0; u < kVecHeads; ++u) {
    const int h = grp * kVecHeads + u;
    if (h >= p.heads) continue;
    T *hr = row + (int64_t)h * p.s_h + e0;
    float a[EPV];
    vec_to_float<T>(va[u], a);
    if constexpr (INTER) {
#pragma unroll
      for (int j = 0; j < PPV; ++j) rope_rotate(a[2 * j], a[2 * j + 1], cs[j], sn[j], a[2 * j], a[2 * j + 1]);
      *reinterpret_cast<uint4 *>(hr) = vec_from_float<T>(a);
    } else {
      float c[EPV];
      vec_to_float<T>(vb[u], c);
#pragma unroll
      for (int j = 0; j < PPV; ++j) rope_rotate(a[j], c[j], cs[j], sn[j], a[j], c[j]);
      *reinterpret_cast<uint4 *>(hr) = vec_from_float<T>(a);
      *reinterpret_cast<uint4 *>(hr + p.half) = vec_from_float<T>(c);
    }
  }
}

// One warp per rotated head vector (b, l, h < heads): RMS normalisation over
// the D features, then the rotation of the first rot_dim; D <= 256.
constexpr int kNormWarps = 8;
template <typename T>
MGQA_DEV void rope_norm_body(const RopeParams &p, int64_t blk) {
  __shared__ float rowbuf[kNormWarps][256];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int64_t task = blk * kNormWarps + wl;  // (b, l, h) with h fastest
  if (task >= (int64_t)p.B * p.L * p.heads) return;             // warp-uniform
  const int h = (int)(task % p.heads);
  const int64_t bl = task / p.heads;
  const int l = (int)(bl % p.L), b = (int)(bl / p.L);
  T *row = static_cast<T *>(p.x) + (int64_t)b * p.s_b + (int64_t)h * p.s_h + (int64_t)l * p.s_l;
  float *buf = rowbuf[wl];
  allow_dependents();
  if (lane * 128 < p.D * (int)sizeof(T))  // the row toward the L2 (a hint) before the wait
    prefetch_l2(reinterpret_cast<const char *>(row) + lane * 128);
  grid_dependency_wait();
  float part = 0.f;
  for (int d = lane, k = 0; d < p.D; d += 32, ++k) {
    const float x = to_float(row[d]);
    buf[d] = x;
    part = rms_partial_add(part, x, k == 0);
  }
  const float r = rms_scale(rms_butterfly_warp(part), p.D, p.eps);
  for (int d = lane; d < p.D; d += 32) buf[d] = rms_apply(buf[d], r, __ldg(p.norm_w + d));
  __syncwarp();
  const int pos = p.positions ? __ldg(p.positions + bl) : l;
  for (int i = lane; i < p.half; i += 32) {
    const int e0 = p.interleaved ? 2 * i : i;
    const int e1 = p.interleaved ? 2 * i + 1 : i + p.half;
    float sn, cs, y0, y1;
    rope_sincos(rope_theta(pos, __ldg(p.inv_freq + i)), sn, cs);
    rope_rotate(buf[e0], buf[e1], cs, sn, y0, y1);
    row[e0] = from_float<T>(y0);
    row[e1] = from_float<T>(y1);
  }
  for (int d = 2 * p.half + lane; d < p.D; d += 32) row[d] = from_float<T>(buf[d]);
}

// Every kernel rotates one tensor (p1 unused, nb0 = the grid) or two in one
// launch: blocks below nb0 take p0, the rest p1 (q and k of one layer).
template <typename T, bool PAIRED>
__global__ void __launch_bounds__(kRopeThreads)
rope_kernel(const __grid_constant__ RopeParams p0, const __grid_constant__ RopeParams p1, unsigned nb0) {
  if (blockIdx.x < nb0) rope_body<T, PAIRED>(p0, blockIdx.x);
  else rope_body<T, PAIRED>(p1, blockIdx.x - nb0);
}
template <typename T, bool INTER>
__global__ void __launch_bounds__(kRopeThreads)
rope_vec_kernel(const __grid_constant__ RopeParams p0, const __grid_constant__ RopeParams p1, unsigned nb0) {
  if (blockIdx.x < nb0) rope_vec_body<T, INTER>(p0, blockIdx.x);
  else rope_vec_body<T, INTER>(p1, blockIdx.x - nb0);
}
template <typename T>
__global__ void __launch_bounds__(32 * kNormWarps)
rope_norm_kernel(const __grid_constant__ RopeParams p0, const __grid_constant__ RopeParams p1, unsigned nb0) {
  if (blockIdx.x < nb0) rope_norm_body<T>(p0, blockIdx.x);
  else rope_norm_body<T>(p1, blockIdx.x - nb0);
}

// The kernel a tensor takes, and its grid.
enum class RopeKind { kNorm, kVecInter, kVecHalf, kScalarPaired, kScalar };
struct RopePlan {
  RopeKind kind;
  int64_t blocks;
};

template <typename T>
RopePlan plan_t(const RopeParams &p) {
  if (p.norm_w) {
    const int64_t tasks = (int64_t)p.B * p.L * p.heads;
    return {RopeKind::kNorm, (tasks + kNormWarps - 1) / kNormWarps};
  }
  // 16-byte vectors: aligned rows and a rotated span of whole vectors
  constexpr int EPV = 16 / (int)sizeof(T);
  const bool vec = (reinterpret_cast<uintptr_t>(p.x) % 16) == 0 && p.s_b % EPV == 0 &&
                   p.s_h % EPV == 0 && p.s_l % EPV == 0 &&
                   (p.interleaved ? (2 * p.half) % EPV == 0 : p.half % EPV == 0);
  if (vec) {
    const int64_t nvec = p.interleaved ? 2 * p.half / EPV : p.half / EPV;
    const int64_t vtotal = (int64_t)p.B * p.L * ((p.heads + kVecHeads - 1) / kVecHeads) * nvec;
    return {p.interleaved ? RopeKind::kVecInter : RopeKind::kVecHalf,
            (vtotal + kRopeThreads - 1) / kRopeThreads};
  }
  const int64_t total = (int64_t)p.B * p.L * p.half;
  // interleaved 16-bit pairs as 32-bit words: every row start 4-byte aligned
  const bool paired = sizeof(T) == 2 && p.interleaved &&
                      (reinterpret_cast<uintptr_t>(p.x) % 4) == 0 && p.s_b % 2 == 0 &&
                      p.s_h % 2 == 0 && p.s_l % 2 == 0;
  return {paired ? RopeKind::kScalarPaired : RopeKind::kScalar, (total + kRopeThreads - 1) / kRopeThreads};
}

// One launch of kind k over grid blocks, the first nb0 of them for p0.
template <typename T>
mgqa_status launch_kind(RopeKind k, const RopeParams &p0, const RopeParams &p1, int64_t nb0,
                        int64_t blocks, cudaStream_t s) {
  if (blocks > 0x7fffffffLL) return fail(MGQA_ERR_UNSUPPORTED, "rope: too many rows");
  const dim3 grid((unsigned)blocks);
  const unsigned n0 = (unsigned)nb0;
  cudaError_t e = cudaSuccess;
  switch (k) {
    case RopeKind::kNorm:
      e = launch_pdl(rope_norm_kernel<T>, grid, dim3(32 * kNormWarps), 0, s, p0, p1, n0);
      break;
    case RopeKind::kVecInter:
      e = launch_pdl(rope_vec_kernel<T, true>, grid, dim3(kRopeThreads), 0, s, p0, p1, n0);
      break;
    case RopeKind::kVecHalf:
      e = launch_pdl(rope_vec_kernel<T, false>, grid, dim3(kRopeThreads), 0, s, p0, p1, n0);
      break;
    case RopeKind::kScalarPaired:
      e = launch_pdl(rope_kernel<T, sizeof(T) == 2>, grid, dim3(kRopeThreads), 0, s, p0, p1, n0);
      break;
    case RopeKind::kScalar:
      e = launch_pdl(rope_kernel<T, false>, grid, dim3(kRopeThreads), 0, s, p0, p1, n0);
      break;
  }
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "rope launch: %s", cudaGetErrorString(e));
  return MGQA_OK;
}

template <typename T>
mgqa_status launch_t(const RopeParams &p, cudaStream_t s) {
  const RopePlan pl = plan_t<T>(p);
  return launch_kind<T>(pl.kind, p, p, pl.blocks, pl.blocks, s);
}

// Two tensors: one launch when they take the same kernel and their elements
// do not overlap (overlapping ones are rotated one after the other, as two
// calls would), else one launch each.
template <typename T>
mgqa_status launch_pair_t(const RopeParams &p0, const RopeParams &p1, bool disjoint, cudaStream_t s) {
  const RopePlan a = plan_t<T>(p0), b = plan_t<T>(p1);
  if (disjoint && a.kind == b.kind) return launch_kind<T>(a.kind, p0, p1, a.blocks, a.blocks + b.blocks, s);
  const mgqa_status st = launch_kind<T>(a.kind, p0, p0, a.blocks, a.blocks, s);
  if (st != MGQA_OK) return st;
  return launch_kind<T>(b.kind, p1, p1, b.blocks, b.blocks, s);
}

}  // namespace
}  // namespace mgqa

namespace mgqa {
namespace {

// Host-side checks of one tensor's arguments; fills p.
mgqa_status rope_params(const mgqa_rope_args *a, RopeParams &p, const char *what) {
  if (!a) return fail(MGQA_ERR_INVALID_ARG, "%s: args is null", what);
  if (a->dtype != MGQA_BF16 && a->dtype != MGQA_FP16 && a->dtype != MGQA_FP32)
    return fail(MGQA_ERR_INVALID_ARG, "%s: unknown dtype", what);
  if (a->B < 1 || a->H < 1 || a->L < 1 || a->D < 2)
    return fail(MGQA_ERR_INVALID_ARG, "%s: B, H, L must be >= 1 and D >= 2", what);
  if (a->rot_dim < 2 || a->rot_dim > a->D || (a->rot_dim & 1))
    return fail(MGQA_ERR_INVALID_ARG, "%s: rot_dim must be even and in [2, D]", what);
  if (a->heads < 1 || a->heads > a->H)
    return fail(MGQA_ERR_INVALID_ARG, "%s: heads must be in [1, H]", what);
  if (!a->x || !a->inv_freq) return fail(MGQA_ERR_INVALID_ARG, "%s: x or inv_freq is null", what);
  if (a->norm_weight && (a->D > 256 || !(a->norm_eps >= 0.f) || !std::isfinite(a->norm_eps) ||
                         reinterpret_cast<uintptr_t>(a->norm_weight) % 4 != 0))
    return fail(MGQA_ERR_INVALID_ARG, "%s: the norm needs D <= 256, a finite eps >= 0 and an "
                                      "aligned fp32 weight", what);
  const size_t es = a->dtype == MGQA_FP32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(a->x) % es != 0 ||
      reinterpret_cast<uintptr_t>(a->inv_freq) % 4 != 0 ||
      (a->positions && reinterpret_cast<uintptr_t>(a->positions) % 4 != 0))
    return fail(MGQA_ERR_INVALID_ARG, "%s: misaligned pointer", what);
  // a zero stride over a dimension of extent > 1 would rotate shared elements
  // more than once (or from two threads at once)
  const int ext[3] = {a->B, a->H, a->L};
  for (int t = 0; t < 3; ++t)
    if (a->x_stride[t] < 0 || (a->x_stride[t] == 0 && ext[t] > 1))
      return fail(MGQA_ERR_INVALID_ARG, "%s: stride %d must be positive", what, t);
  p = RopeParams{};
  p.x = a->x;
  p.s_b = a->x_stride[0]; p.s_h = a->x_stride[1]; p.s_l = a->x_stride[2];
  p.positions = a->positions;
  p.inv_freq = a->inv_freq;
  p.B = a->B; p.L = a->L; p.D = a->D; p.half = a->rot_dim / 2; p.heads = a->heads;
  p.interleaved = a->interleaved != 0;
  p.norm_w = a->norm_weight;
  p.eps = a->norm_eps;
  return MGQA_OK;
}

// [first, last] byte addresses of the elements a tensor's view spans
void rope_span(const mgqa_rope_args *a, uintptr_t &lo, uintptr_t &hi) {
  const size_t es = a->dtype == MGQA_FP32 ? 4 : 2;
  const int64_t last = (int64_t)(a->B - 1) * a->x_stride[0] + (int64_t)(a->H - 1) * a->x_stride[1] +
                       (int64_t)(a->L - 1) * a->x_stride[2] + (a->D - 1);
  lo = reinterpret_cast<uintptr_t>(a->x);
  hi = lo + (uintptr_t)last * es + (es - 1);
}

}  // namespace
}  // namespace mgqa

extern "C" MGQA_API mgqa_status masked_gqa_rope(const mgqa_rope_args *a, cudaStream_t stream) {
  using namespace mgqa;
  clear_error_detail();
  RopeParams p;
  const mgqa_status st = rope_params(a, p, "rope");
  if (st != MGQA_OK) return st;
  if (a->dtype == MGQA_BF16) return launch_t<__nv_bfloat16>(p, stream);
  if (a->dtype == MGQA_FP16) return launch_t<__half>(p, stream);
  return launch_t<float>(p, stream);
}

extern "C" MGQA_API mgqa_status masked_gqa_rope_pair(const mgqa_rope_args *q, const mgqa_rope_args *k,
                                                     cudaStream_t stream) {
  using namespace mgqa;
  clear_error_detail();
  RopeParams pq, pk;
  mgqa_status st = rope_params(q, pq, "rope pair (q)");
  if (st != MGQA_OK) return st;
  st = rope_params(k, pk, "rope pair (k)");
  if (st != MGQA_OK) return st;
  if (q->dtype != k->dtype) return fail(MGQA_ERR_INVALID_ARG, "rope pair: q and k dtypes differ");
  uintptr_t q0, q1, k0, k1;
  rope_span(q, q0, q1);
  rope_span(k, k0, k1);
  const bool disjoint = q1 < k0 || k1 < q0;
  if (q->dtype == MGQA_BF16) return launch_pair_t<__nv_bfloat16>(pq, pk, disjoint, stream);
  if (q->dtype == MGQA_FP16) return launch_pair_t<__half>(pq, pk, disjoint, stream);
  return launch_pair_t<float>(pq, pk, disjoint, stream);
}
