// Device helpers shared by the kernels of the masked GQA attention library.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/masked_gqa_attn.h"

#define MGQA_DEV __device__ __forceinline__

namespace mgqa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Record the first device-side error code (later ones are dropped).
MGQA_DEV void report_error(int32_t *err, int32_t code) {
  if (err) atomicCAS(err, 0, code);
}

// Bounds and alignment checks of the debug library (built with MGQA_DEBUG):
// a failed check records MGQA_ERR_DEVICE_CHECK and the caller skips the
// access. In the product library every check is the constant true.
#ifdef MGQA_DEBUG
MGQA_DEV bool dcheck(bool ok, int32_t *err) {
  if (!ok) report_error(err, MGQA_ERR_DEVICE_CHECK);
  return ok;
}
#define MGQA_DCHECK(cond, err) (::mgqa::dcheck((cond), (err)))
#else
#define MGQA_DCHECK(cond, err) true
#endif

// Longest a pipeline wait spins before it reports MGQA_ERR_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

MGQA_DEV float to_float(float x) { return x; }
MGQA_DEV float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
MGQA_DEV float to_float(__half x) { return __half2float(x); }

template <typename T> MGQA_DEV T from_float(float x);
template <> MGQA_DEV float from_float<float>(float x) { return x; }
template <> MGQA_DEV __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <> MGQA_DEV __half from_float<__half>(float x) { return __float2half_rn(x); }

// Two floats rounded to a packed pair of 16-bit values (low half = lo).
template <typename T> MGQA_DEV uint32_t pack2(float lo, float hi);
template <> MGQA_DEV uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
template <> MGQA_DEV uint32_t pack2<__half>(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// Unpack 16 bytes into float lanes: 8 bf16 / 8 fp16 or 4 fp32 values.
MGQA_DEV void unpack16(const uint4 &u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
template <typename T> MGQA_DEV void unpack16_t(const uint4 &u, float (&f)[8]);
template <> MGQA_DEV void unpack16_t<__nv_bfloat16>(const uint4 &u, float (&f)[8]) { unpack16(u, f); }
template <> MGQA_DEV void unpack16_t<__half>(const uint4 &u, float (&f)[8]) {
  const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __half22float2(h[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}
template <typename T> MGQA_DEV void unpack16_t(const uint4 &u, float (&f)[4]);
template <> MGQA_DEV void unpack16_t<float>(const uint4 &u, float (&f)[4]) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}
MGQA_DEV void unpack16(const uint4 &u, float (&f)[4]) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}

// kv_len[b] clamped to [0, Lk]; out-of-range values are reported once.
MGQA_DEV int load_kv_len(const int32_t *kv_len, int b, int Lk, int32_t *err, bool report) {
  if (!kv_len) return Lk;
  int n = __ldg(kv_len + b);
  if (n < 0 || n > Lk) {
    if (report) report_error(err, MGQA_ERR_INVALID_ARG);
    n = n < 0 ? 0 : Lk;
  }
  return n;
}

// ---- rotary embedding and RMS normalisation ---------------------------------
// Every kernel that normalises or rotates a head vector uses these, with
// every step rounded once, so a fused path gives the same bits as the
// standalone kernel followed by attention.

// theta = fl32(position * inv_freq)
MGQA_DEV float rope_theta(int pos, float f) { return __fmul_rn((float)pos, f); }

// sin and cos of theta (|theta| < 2^22): Cody-Waite argument reduction
// (W. J. Cody and W. Waite, Software Manual for the Elementary Functions,
// 1980) by 2 pi, written as a float head and a float tail of its value, with
// one rounding per fused multiply-add, to r in about [-pi, pi]; then the
// MUFU sine and cosine of r. Error: at most about 5e-7 (the unit's 2^-21.4 on
// [-pi, pi] plus half an ulp of pi from the reduction); short and branch-free,
// so kernels can unroll it over a row.
MGQA_DEV void rope_sincos(float theta, float &sn, float &cs) {
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  constexpr float kHi = (float)kTwoPi;
  constexpr float kLo = (float)(kTwoPi - (double)kHi);
  constexpr float kInv = (float)(1.0 / kTwoPi);
  const float k = rintf(__fmul_rn(theta, kInv));
  const float r = __fmaf_rn(-k, kLo, __fmaf_rn(-k, kHi, theta));
  sn = __sinf(r);
  cs = __cosf(r);
}

// (a, c) -> (a cos - c sin, a sin + c cos)
MGQA_DEV void rope_rotate(float a, float c, float cs, float sn, float &x0, float &x1) {
  x0 = __fsub_rn(__fmul_rn(a, cs), __fmul_rn(c, sn));
  x1 = __fadd_rn(__fmul_rn(a, sn), __fmul_rn(c, cs));
}

// The sum of squares of a head vector in one fixed order: lane partial l
// accumulates x_d^2 for d = l, l + 32, l + 64, ... (a product, then fused
// multiply-adds), and the 32 partials combine as an xor butterfly with
// offsets 16, 8, 4, 2, 1.
MGQA_DEV float rms_partial_add(float p, float x, bool first) {
  return first ? __fmul_rn(x, x) : __fmaf_rn(x, x, p);
}
MGQA_DEV float rms_butterfly_warp(float p) {  // every lane of the warp takes part
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, o));
  return p;
}
// The same sum for a row held by one thread: the partials of lanes l and
// l + 16 are formed and combined at once (the butterfly's first step), then
// the remaining steps run on 16 values.
template <int D>
MGQA_DEV float rms_sum_row(const float (&x)[D]) {
  static_assert(D % 32 == 0, "row of whole lanes");
  float p[16];
#pragma unroll
  for (int l = 0; l < 16; ++l) {
    float a = 0.f, c = 0.f;
#pragma unroll
    for (int d = l, k = 0; d < D; d += 32, ++k) {
      a = rms_partial_add(a, x[d], k == 0);
      c = rms_partial_add(c, x[d + 16], k == 0);
    }
    p[l] = __fadd_rn(a, c);
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1)
#pragma unroll
    for (int l = 0; l < o; ++l) p[l] = __fadd_rn(p[l], p[l + o]);
  return p[0];
}
// 1 / sqrt(ss / D + eps)
MGQA_DEV float rms_scale(float ss, int D, float eps) {
  return __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)D), eps)));
}
MGQA_DEV float rms_apply(float x, float r, float w) { return __fmul_rn(__fmul_rn(x, r), w); }

// ---- mask forms -----------------------------------------------------------

// The mask forms of one call; any pointer may be null (form absent).
struct MaskView {
  const uint32_t *bits;  // words, row (b, i) at b*sb + i*sq
  int64_t sb, sq;
  const int32_t *kv_len;  // [B]
  const int32_t *seg_q;   // [B][Lq]
  const int32_t *seg_k;   // [B][Lk]
  int causal;             // key j only for query i with j <= i + coff
  int coff;               // Lk - Lq
};

// Bits t = 0..31 of the result: may query i of row b attend to key jbase + t?
// jbase is a multiple of 32. kvl is the (clamped) kv_len of row b, segq the
// query's segment id (ignored without segment ids). Keys >= Lk are never
// allowed. Segment ids are read from global memory (cached).
MGQA_DEV uint32_t mask_word(const MaskView &m, int b, int i, int jbase, int Lk, int Lq, int kvl,
                            int segq) {
  if (jbase >= Lk) return 0u;
  int lim = min(Lk, kvl) - jbase;
  if (m.causal) lim = min(lim, i + m.coff + 1 - jbase);
  uint32_t w = lim >= 32 ? 0xffffffffu : (lim <= 0 ? 0u : ((1u << lim) - 1u));
  if (m.bits && w) w &= __ldg(m.bits + (int64_t)b * m.sb + (int64_t)i * m.sq + (jbase >> 5));
  if (m.seg_q && w) {
    if (segq < 0) return 0u;
    const int32_t *sk = m.seg_k + (int64_t)b * Lk + jbase;
    uint32_t sw = 0u;
    const int n = min(32, Lk - jbase);
    for (int t = 0; t < n; ++t) sw |= (uint32_t)(__ldg(sk + t) == segq) << t;
    w &= sw;
  }
  return w;
}

// Named CTA barriers (ids 1..15; id 0 is __syncthreads).
MGQA_DEV void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel in the stream is still
// running. Everything before grid_dependency_wait() must not touch global
// memory the previous kernel writes or reads; after it, that kernel has
// completed and its writes are visible. allow_dependents() lets the next
// kernel in the stream start its own set-up early.
MGQA_DEV void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MGQA_DEV void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// A hint that brings the line of p into the L2 (and its page translation
// into the SM's TLBs). Nothing is read into the SM and the L2 is the point
// of coherence, so it may precede grid_dependency_wait().
MGQA_DEV void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// ---- mbarrier / bulk-copy primitives (PTX) --------------------------------

MGQA_DEV uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MGQA_DEV void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

MGQA_DEV void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

MGQA_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

MGQA_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}


MGQA_DEV void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

MGQA_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

MGQA_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Non-blocking probe of an mbarrier phase (cheaper than try_wait when the
// phase has already completed, the common case on a pipeline's fast path).
MGQA_DEV bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// 2^x on the MUFU unit (approximate, flushes denormals; 2^-inf = 0).
MGQA_DEV float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait on an mbarrier phase: gives up after ~`limit_ns` of wall time
// (measured with the global timer), records MGQA_ERR_TIMEOUT and returns
// false. Never spins forever.
MGQA_DEV bool mbar_wait(uint64_t *bar, uint32_t parity, int32_t *err,
                        uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_test_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++n & 255u) == 0u) {
      if (globaltimer_ns() - t0 > limit_ns) {
        report_error(err, MGQA_ERR_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

// mbar_wait for a phase completed by other CTAs of the cluster (their
// st.async bytes): acquires at cluster scope.
MGQA_DEV bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, int32_t *err, uint64_t limit_ns) {
  auto try_wait = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0u;
  };
  uint64_t t0 = 0;
  for (uint32_t n = 0; !try_wait(); ++n) {
    if (n == 0u) t0 = globaltimer_ns();
    if ((n & 255u) == 255u && globaltimer_ns() - t0 > limit_ns) {
      report_error(err, MGQA_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// ---- thread-block clusters (distributed shared memory) ---------------------

// Barrier over every thread of the cluster. The arrive releases this thread's
// earlier shared-memory writes and the wait acquires the other CTAs' ones, so
// after it each CTA may read what the others stored before they arrived. All
// threads of every CTA of the cluster must execute it (the cluster's CTAs are
// co-scheduled, so it cannot wait for a CTA that never started).
MGQA_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of that barrier, for a wait placed long after the arrive:
// the arrive releases this thread's earlier writes (an mbarrier's
// initialisation included), the wait returns once every thread of the
// cluster arrived. Both by all threads of every CTA.
MGQA_DEV void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
MGQA_DEV void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Store two floats into shared memory of a CTA of the cluster (`addr` and
// the mbarrier `bar` both in that CTA, as cluster_map addresses); 8 bytes of
// completion are counted on `bar`, which releases them at cluster scope.
MGQA_DEV void st_async_f32x2(uint32_t addr, float a, float b, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
                   addr),
               "f"(a), "f"(b), "r"(bar)
               : "memory");
}

// Address, in the cluster's shared window, of `p` (a variable of this CTA's
// shared memory) in the CTA of cluster rank `rank`.
MGQA_DEV uint32_t cluster_map(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
MGQA_DEV float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Bulk copy of `bytes` (a multiple of 16) from global to this CTA's shared
// memory, both addresses 16-byte aligned; completion is counted in bytes on
// the mbarrier `bar` (armed by an arrive.expect_tx of the phase's total).
MGQA_DEV void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 16-byte asynchronous copy global -> shared through the L1-bypassing path;
// both addresses 16-byte aligned. Completion: cp_async_wait_all().
MGQA_DEV void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
MGQA_DEV void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
// Close the group of this thread's copies issued since the last commit.
MGQA_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's committed groups are still in flight.
template <int N> MGQA_DEV void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// D (16x8 fp32) += A (16x16, row) * B (16x8, col), both bf16 or both fp16:
// register fragments of the warp-wide mma.sync shape m16n8k16.
template <typename T>
MGQA_DEV void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                        uint32_t b0, uint32_t b1) {
  if constexpr (sizeof(T) == 2 && __is_same(T, __half)) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// Two transposed 8x8 bf16 tiles from shared memory; lane i (0..15) gives the
// address of row i (rows 8..15 form the second tile).
MGQA_DEV void ldmatrix_x2_trans(uint32_t &b0, uint32_t &b1, const void *row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(b0), "=r"(b1)
               : "r"(smem_u32(row)));
}

// Four 8x8 16-bit tiles from shared memory; lane i gives the address of row
// i % 8 of tile i / 8. Lane t receives row t / 4, elements 2 (t % 4) and
// 2 (t % 4) + 1 of each tile (the .trans form: of each tile's transpose).
MGQA_DEV void ldmatrix_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3, const void *row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(row)));
}
MGQA_DEV void ldmatrix_x4_trans(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3,
                                const void *row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(row)));
}

// Transpose of an 8x8 16-bit matrix held as a warp fragment (lane t: row
// t / 4, elements 2 (t % 4) and 2 (t % 4) + 1, low half first).
MGQA_DEV uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

}  // namespace mgqa
