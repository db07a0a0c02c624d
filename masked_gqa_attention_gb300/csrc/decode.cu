// One-query attention over a static KV cache: a cluster of 16 CTAs per
// (request, KV-head group), whose partial results are merged on chip in the
// same launch.
//
// Passages: VoxCPM page, "Upstream-identical practice", attention bullet
// (decode against the static cache under an explicit boolean mask; slots past
// the current length are masked and add exact zeros) and "Memory & speed",
// attention_span paragraph (attend only to the filled blocks of the 8192-slot
// cache instead of all of it).
//
// Design: the S = 16 CTAs of one cluster serve one (request b, head group hg)
// -- the NREP query heads of one KV head. The cache is cut into 64-slot chunks
// of absolute positions; CTA x (its rank in the cluster) owns chunks x, x + S,
// x + 2S, ...  A call is a short chain of dependent steps, each kept to one
// memory round trip or one barrier:
//   1. Every input of the mask test (kv_len, the CTA's mask words, segment
//      ids) and q are loaded together. Each warp tests the slots of its
//      chunks (one lane per slot, ballots) and stores the allowed-slot words.
//   2. The non-empty chunks, in ascending order, fill batches of CAPR rows at
//      fixed positions (row = chunk position in the batch * 64 + slot). Each
//      chunk arrives as TMA tensor boxes of 64 rows (128-byte swizzled for the
//      16-bit types, so the fragment loads are conflict-free), issued by one
//      lane per chunk, one mbarrier per batch. Masked rows then get a zero V
//      row in shared memory, so they add exact zeros (a chunk past the filled
//      length is never fetched; only the masked tail of a partly filled chunk
//      is read and discarded); the row a fused append adds is written in from
//      the step's input.
//   3. bf16 / fp16: S^T = K q^T and O^T += V^T P^T on the tensor cores
//      (mma.sync m16n8k16), the cache rows on the M side and the <= 8 heads on
//      the N side, so no product carries padding rows; only fetched chunk
//      slots are computed. All warps share one running maximum per head
//      (exchanged once per batch), so the in-CTA merge of the warps' outputs
//      is a plain sum. fp32: CUDA cores, per-head batch softmax.
//   4. CTA x owns 1/S of the (head, feature) outputs. Every CTA stores its
//      partial (m, l) and the matching slice of its unnormalised O into each
//      owner's shared memory (st.async, counted in bytes on the owner's
//      mbarrier); each owner merges the S partials of its slice in ascending
//      split order and writes them. No global workspace, no ticket.
// The chunk-to-CTA assignment, the batch layout and every summation order
// depend only on the set of allowed slots, so a full-cache bitmask and the
// equivalent filled length give bit-identical outputs.
#include <cfloat>
#include <cmath>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

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
  FusedRope rope;  // applied to q and the appended row (inv_freq null: none)
};

// 4 warps a CTA, 3 CTAs an SM (<= 75 KB of shared memory each): the 16-CTA
// clusters of the static-cache workloads then all fit on the GPU at once.
constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int C = kDecodeChunk;
constexpr int S = kDecodeSplits;              // CTAs of a cluster
constexpr int kMaxCI = kDecodeMaxLk / C / S;  // chunks per CTA (32)
constexpr int kCPW = kMaxCI / kWarps;         // chunks per warp in the mask test
static_assert(kMaxCI <= 32, "one ballot covers the CTA's chunks");

// Debug library only (MGQA_DEBUG): a per-CTA timeline of the kernel's phases
// (SM clock at each phase boundary, the global timer at entry and exit, the
// SM id), read with mgqa_debug_decode_timeline.
#ifdef MGQA_DEBUG
constexpr int kTlCtas = 512, kTlStamps = 16;
__device__ unsigned long long g_dec_tl[kTlCtas][kTlStamps];
MGQA_DEV void dec_stamp(int k) {
  const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  if (threadIdx.x == 0 && cta < (unsigned)kTlCtas) {
    g_dec_tl[cta][k] = clock64();
    if (k == 0) {
      g_dec_tl[cta][13] = globaltimer_ns();
      unsigned sm;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
      g_dec_tl[cta][15] = sm;
    }
    if (k == 7) g_dec_tl[cta][14] = globaltimer_ns();
  }
}
#else
MGQA_DEV void dec_stamp(int) {}
#endif

// bf16 and fp16 run the two products on the tensor cores; fp32 on the CUDA cores.
// (A causal mask needs nothing here: the single query is the last position.)
template <typename T>
constexpr bool use_mma() {
  return sizeof(T) == 2;
}

// Shared memory of one decode CTA. K and V of a batch are CPB chunk slots of
// KB TMA boxes (64 rows each): 16-bit rows are 128-byte swizzled boxes of 64
// columns, fp32 rows plain boxes of D columns.
template <typename T, int D, int NREP>
struct DecodeSmem {
  static constexpr bool kMma = use_mma<T>();
  static constexpr int KB = kMma ? D / 64 : 1;                 // boxes per row
  static constexpr int BOXB = kMma ? 64 * 128 : 64 * D * 4;    // bytes of one box
  static constexpr int CHB = KB * BOXB;                        // bytes of one chunk slot
  static constexpr int CPB = 32768 / CHB;                      // chunks per batch: 32 KB of K
  static constexpr int CAPR = CPB * C;                         // positional rows per batch
  static constexpr int RPW = CAPR / kWarps;                    // rows per warp (fp32 path)
  static_assert(RPW >= 16 && CAPR % (16 * kWarps) == 0, "batch layout");
  static constexpr int DP = D + 4;                             // per-warp O row pitch (floats)
  static constexpr int WOB = kWarps * NREP * DP * 4;           // per-warp O (after the last batch)
  static_assert(WOB <= 2 * CPB * CHB, "per-warp O fits in the K and V buffers");
  static constexpr int E = NREP * D / S;                       // outputs each CTA merges
  static_assert(E >= 2 && E % 2 == 0, "whole feature pairs per CTA");
  // The fused rotation's rows (and the fp32 path's q): for the 16-bit types in
  // the K buffer, which nothing else uses before the first batch's copies.
  struct Rot {
    float q[NREP][D];
    float knew[D];
    float2 cs[D / 2];
    float invf[D / 2];   // the rotation's inverse frequencies
    float qw[D], kw[D];  // the q / k norm weights
  };
  static_assert((int)sizeof(Rot) <= CPB * CHB, "rotation rows fit in the K buffer");
  // byte offsets (the base is 1024-byte aligned)
  static constexpr int k_off = 0;
  static constexpr int v_off = CPB * CHB;
  static constexpr int misc_off = 2 * CPB * CHB;
  template <int ROTB>
  struct MiscT {
    alignas(16) unsigned char rot[ROTB];  // the rotation rows, when they live here
    float s[NREP][kMma ? 1 : CAPR];   // fp32 path: one batch's scores / weights
    float fo[NREP], fb[NREP];         // fp32 path
    float wmax[kWarps][NREP], wsum[kWarps][NREP];
    float mrun[NREP], lrun[NREP];     // running (m, l) per head (l: fp32 path)
    uint32_t words[kMaxCI][2];        // allowed-slot words of the CTA's chunks
    alignas(16) T newk[D], newv[D];   // the row a fused append adds
    alignas(16) T qh[kMma ? NREP : 1][D + 8];  // q as loaded (rows padded: conflict-free fragments)
    float2 rx_ml[S][NREP];            // every split's (m, l) of each head
    alignas(8) float rx_o[S][E];      // every split's partial O of this CTA's outputs
    alignas(8) uint64_t bar;          // one phase per batch
    alignas(8) uint64_t rx_bar;       // the partials of this CTA's outputs
  };
  // The rotation rows live in this fixed region when the CTA still fits
  // three to an SM with them there (<= 75 KB); then the first batch's copies
  // go out before the rotation and land while it runs. Otherwise (the 16-bit
  // types at D = 128) they use the K buffer, free until those copies.
  static constexpr bool kRotMisc =
      !kMma || misc_off + (int)sizeof(MiscT<(int)sizeof(Rot)>) + 1024 <= 75 * 1024;
  using Misc = MiscT<kRotMisc ? (int)sizeof(Rot) : 16>;
  static constexpr int total = misc_off + (int)sizeof(Misc) + 1024;  // + alignment slack
  // byte address of 16-byte segment `seg` of positional row r (16-bit types)
  static MGQA_DEV uint32_t seg_off(int r, int seg) {
    const int r64 = r % C;
    return (r / C) * CHB + (seg / 8) * BOXB + r64 * 128 + (((seg % 8) ^ (r64 & 7)) << 4);
  }
  // byte address of row r (fp32: plain rows)
  static MGQA_DEV uint32_t row_off(int r) { return (r / C) * CHB + (r % C) * (D * 4); }
};

template <typename T, int D, int NREP>
__global__ void __launch_bounds__(kThreads, 3)
decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ DecodeParams p) {
  using Sm = DecodeSmem<T, D, NREP>;
  constexpr int CAPR = Sm::CAPR, CPB = Sm::CPB, RPW = Sm::RPW, E = Sm::E;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char *kbuf = smem + Sm::k_off, *vbuf = smem + Sm::v_off;
  auto &sm = *reinterpret_cast<typename Sm::Misc *>(smem + Sm::misc_off);
  auto &rot = *reinterpret_cast<typename Sm::Rot *>(Sm::kRotMisc ? sm.rot : kbuf);
  float(*wo)[NREP][Sm::DP] = reinterpret_cast<float(*)[NREP][Sm::DP]>(kbuf);  // K, V: after the last batch

  const int x = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;  // x: rank in the cluster
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  dec_stamp(0);
  if (tid == 0) {
    mbar_init(&sm.bar, 1);  // thread 0 arms each batch once
    mbar_init(&sm.rx_bar, 1);
    // every split delivers this CTA's slice of its partial: (m, l) of each
    // head and E floats of O
    mbar_arrive_expect_tx(&sm.rx_bar, (uint32_t)(S * (E * 4 + NREP * 8)));
    fence_mbarrier_init();
    tc::prefetch_tensormap(&tm_k);
    tc::prefetch_tensormap(&tm_v);
    allow_dependents();
  }
  // the receive barriers: armed in every CTA before any split delivers
  cluster_arrive();
#ifdef MGQA_DEBUG
  {
    uint32_t rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    if (tid == 0) MGQA_DCHECK(rank == (uint32_t)x, p.err);
  }
#endif
  const int h0 = hg * NREP;
  const int g = h0 / p.n_rep;
  {
    // before the grid-dependency wait, hints that move the lines this CTA
    // reads first toward the L2 (nothing enters the SM; the L2 is the point
    // of coherence, so a later write by the previous kernel still wins): q's
    // rows, kv_len, the mask words and segment ids of every chunk of mine,
    // and the K and V rows of my first chunk, which most calls fetch
    const int64_t r0 = (int64_t)x * C;
    if (tid < NREP)
      prefetch_l2(static_cast<const char *>(p.q) + ((int64_t)b * p.qs_b + (int64_t)(h0 + tid) * p.qs_h) * sizeof(T));
    if (tid == NREP && p.kv_len) prefetch_l2(p.kv_len + b);
    const int nci0 = x < p.nch ? (p.nch - x + S - 1) / S : 0;
    for (int i = tid; i < nci0; i += kThreads) {
      const int64_t j0 = (int64_t)(x + S * i) * C;
      if (p.bits) prefetch_l2(p.bits + (int64_t)b * p.ms_b + (j0 >> 5));
      if (p.seg_k) {
        prefetch_l2(p.seg_k + (int64_t)b * p.Lk + j0);
        if (j0 + 32 < p.Lk) prefetch_l2(p.seg_k + (int64_t)b * p.Lk + j0 + 32);
      }
    }
    constexpr int LPR = (D * (int)sizeof(T) + 127) / 128;  // 128-byte lines per row
    for (int u = tid; u < 2 * C * LPR && r0 < p.Lk; u += kThreads) {
      const int kv = u / (C * LPR), rr = (u / LPR) % C, ln = u % LPR;
      if (r0 + rr < p.Lk) {
        const char *base = static_cast<const char *>(kv ? p.v : p.k);
        const int64_t off = kv ? (int64_t)b * p.vs_b + (int64_t)g * p.vs_h + (r0 + rr) * p.vs_l
                               : (int64_t)b * p.ks_b + (int64_t)g * p.ks_h + (r0 + rr) * p.ks_l;
        prefetch_l2(base + off * sizeof(T) + ln * 128);
      }
    }
  }
  grid_dependency_wait();  // everything below may read what the previous kernel wrote
  dec_stamp(1);
  const int nci = x < p.nch ? (p.nch - x + S - 1) / S : 0;  // my chunks
  const int gq = lane >> 2, tq = lane & 3;                   // mma fragment coordinates

  // ---- 1. every load the mask test and the products need, issued together
  const int kvl_raw = p.kv_len ? __ldg(p.kv_len + b) : p.Lk;
  const T *qb = static_cast<const T *>(p.q) + (int64_t)b * p.qs_b;
  const bool rope = p.rope.inv_freq != nullptr;
  constexpr int SEGS = D * (int)sizeof(T) / 16;  // 16-byte segments of a row
  static_assert(2 * SEGS <= kThreads && (!use_mma<T>() || NREP * SEGS <= kThreads),
                "one thread per row segment");
  // q (and a fused rotation's tables) land in shared memory within this
  // round trip: every thread issues its few independent loads at once (a
  // load first used later could otherwise be scheduled next to its use)
  if constexpr (use_mma<T>()) {
    if (tid < NREP * SEGS) {
      const int h = tid / SEGS, sg = tid % SEGS;
      reinterpret_cast<uint4 *>(sm.qh[h])[sg] =
          reinterpret_cast<const uint4 *>(qb + (int64_t)(h0 + h) * p.qs_h)[sg];
    }
  } else {
    constexpr int QV = NREP * D / 4;  // float4 pieces of the CTA's q rows
#pragma unroll
    for (int u = 0; u < (QV + kThreads - 1) / kThreads; ++u) {
      const int i = tid + u * kThreads;
      if (i < QV) {
        const int h = i / (D / 4), c = i % (D / 4);
        reinterpret_cast<float4 *>(rot.q[h])[c] =
            reinterpret_cast<const float4 *>(qb + (int64_t)(h0 + h) * p.qs_h)[c];
      }
    }
  }
  int rope_pos = -1;  // the step's position when given explicitly
  if (rope) {
    static_assert(D <= kThreads, "one thread per feature");
    if (tid < p.rope.half) rot.invf[tid] = __ldg(p.rope.inv_freq + tid);
    if (tid < D && p.rope.q_norm) rot.qw[tid] = __ldg(p.rope.q_norm + tid);
    if (tid < D && p.rope.k_norm) rot.kw[tid] = __ldg(p.rope.k_norm + tid);
    if (p.rope.positions) rope_pos = __ldg(p.rope.positions + b);
  }
  uint32_t wbits[kCPW][2];
  int segk[kCPW][2];
  const int segq = p.seg_q ? __ldg(p.seg_q + b) : 0;
#pragma unroll
  for (int u = 0; u < kCPW; ++u) {
    const int i = warp + u * kWarps;
    const int j0 = (x + S * i) * C;
    wbits[u][0] = wbits[u][1] = 0xffffffffu;
    segk[u][0] = segk[u][1] = segq;
    if (i < nci) {
      if (p.bits) {
        const int W = (p.Lk + 31) >> 5;
        const uint32_t *mrow = p.bits + (int64_t)b * p.ms_b + (j0 >> 5);
        wbits[u][0] = __ldg(mrow);
        wbits[u][1] = ((j0 >> 5) + 1 < W) ? __ldg(mrow + 1) : 0u;
      }
      if (p.seg_k) {
        const int32_t *sk = p.seg_k + (int64_t)b * p.Lk + j0;
        segk[u][0] = (j0 + lane < p.Lk) ? __ldg(sk + lane) : -1;
        segk[u][1] = (j0 + 32 + lane < p.Lk) ? __ldg(sk + 32 + lane) : -1;
      }
    }
  }
  const T *kg = static_cast<const T *>(p.k) + (int64_t)b * p.ks_b + (int64_t)g * p.ks_h;
  const T *vg = static_cast<const T *>(p.v) + (int64_t)b * p.vs_b + (int64_t)g * p.vs_h;
  const T *kn = p.append ? static_cast<const T *>(p.k_new) + (int64_t)b * p.kn_b + (int64_t)g * p.kn_h
                         : nullptr;
  const T *vn = p.append ? static_cast<const T *>(p.v_new) + (int64_t)b * p.vn_b + (int64_t)g * p.vn_h
                         : nullptr;
  if (p.append && tid < 2 * SEGS) {  // the appended row, wherever it lands
    const uint4 *src = reinterpret_cast<const uint4 *>(tid < SEGS ? kn : vn);
    reinterpret_cast<uint4 *>(tid < SEGS ? sm.newk : sm.newv)[tid % SEGS] = src[tid % SEGS];
  }
  if (tid < NREP) {
    sm.mrun[tid] = -INFINITY;
    sm.lrun[tid] = 0.f;
  }
  int kvl = kvl_raw;
  if (kvl < 0 || kvl > p.Lk) {
    if (x == 0 && hg == 0 && tid == 0) report_error(p.err, MGQA_ERR_INVALID_ARG);
    kvl = kvl < 0 ? 0 : p.Lk;
  }
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
  // allowed-slot words: lane = slot within each 32-slot half of a chunk
#pragma unroll
  for (int u = 0; u < kCPW; ++u) {
    const int i = warp + u * kWarps;
    if (i < nci) {  // warp-uniform
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int j = (x + S * i) * C + hh * 32 + lane;
        bool a = j < p.Lk && j < kvl && ((wbits[u][hh] >> lane) & 1u);
        if (p.seg_k) a = a && segq >= 0 && segk[u][hh] == segq;
        const uint32_t w = __ballot_sync(0xffffffffu, a);
        if (lane == 0) sm.words[i][hh] = w;
      }
    }
  }
  __syncthreads();
  dec_stamp(2);
  uint32_t qa[use_mma<T>() ? D / 16 : 1][2];  // q as the B operand (column gq: head gq)
  if constexpr (use_mma<T>()) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = qa[kk][1] = 0u;
      if (gq < NREP && !rope) {
        qa[kk][0] = *reinterpret_cast<const uint32_t *>(&sm.qh[gq][kk * 16 + 2 * tq]);
        qa[kk][1] = *reinterpret_cast<const uint32_t *>(&sm.qh[gq][kk * 16 + 2 * tq + 8]);
      }
    }
  }
  // the non-empty chunks in ascending order: bit i set for chunk i (every warp
  // forms the same mask)
  const uint32_t nem = __ballot_sync(0xffffffffu, lane < nci && (sm.words[lane][0] | sm.words[lane][1]));
  const int n_ne = __popc(nem);
  const int nbatch = (n_ne + CPB - 1) / CPB;

  // rank of chunk `lane` among the non-empty chunks (-1: empty, or not mine)
  const int my_rank = ((nem >> lane) & 1u) ? __popc(nem & ((1u << lane) - 1u)) : -1;
  // allowed-slot words of the chunk in batch position cs of batch bt (0: none);
  // cs is the same for the whole warp
  auto chunk_words = [&](int bt, int cs, int &chunk) -> uint2 {
    const uint32_t m = __ballot_sync(0xffffffffu, my_rank == bt * CPB + cs);
    if (!m) {
      chunk = -1;
      return make_uint2(0u, 0u);
    }
    chunk = __ffs(m) - 1;
    return make_uint2(sm.words[chunk][0], sm.words[chunk][1]);
  };

  // ---- 2. gather: lane i of warp 0 holds chunk i; the chunk of rank
  // bt * CPB + cs goes to chunk slot cs, after lane 0 armed the batch's bytes
  auto issue_batch = [&](int bt) {
    const int nbc = min(CPB, n_ne - bt * CPB);  // chunks in this batch
    if (warp == 0) {
      if (lane == 0) mbar_arrive_expect_tx(&sm.bar, (uint32_t)(nbc * 2 * Sm::CHB));
      if (bt == 0) dec_stamp(12);
      __syncwarp();
      const int cs = my_rank - bt * CPB;
      if (my_rank >= 0 && cs >= 0 && cs < nbc) {
        const int row = (x + S * lane) * C;
        if (MGQA_DCHECK(row < p.Lk && g < p.Hkv, p.err)) {
#pragma unroll
          for (int bx = 0; bx < Sm::KB; ++bx) {
            tc::tma_load_4d(kbuf + cs * Sm::CHB + bx * Sm::BOXB, &tm_k, bx * 64, row, g, b, &sm.bar);
            tc::tma_load_4d(vbuf + cs * Sm::CHB + bx * Sm::BOXB, &tm_v, bx * 64, row, g, b, &sm.bar);
          }
        }
      }
    }
    if (bt == 0) dec_stamp(3);
  };
  // the first batch goes out now unless the rotation rows still need the K buffer
  const bool early = !rope || Sm::kRotMisc;
  if (early && nbatch > 0) issue_batch(0);
  if (rope) {
    // the step's query rows and new key row, normalised and rotated at the new
    // token's position with the arithmetic of the standalone kernel
    const int npos = p.rope.positions ? rope_pos : (pos >= 0 ? pos : kvl);
    const bool krow = p.append && g < p.rope.k_heads;
    if constexpr (use_mma<T>())
      for (int i = tid; i < NREP * D; i += kThreads) rot.q[i / D][i % D] = to_float(sm.qh[i / D][i % D]);
    if (krow)
      for (int d = tid; d < D; d += kThreads) rot.knew[d] = to_float(sm.newk[d]);
    for (int i = tid; i < p.rope.half; i += kThreads) {
      float sn, cs;
      rope_sincos(rope_theta(npos, rot.invf[i]), sn, cs);
      rot.cs[i] = make_float2(cs, sn);
    }
    __syncthreads();
    // eight lanes per row (all NREP + 1 rows in one round): the RMS norm,
    // then the rotation and one rounding to the I/O type (q stays a float
    // holding it). Lane sl of a row forms the canonical lane partials sl,
    // sl + 8, sl + 16, sl + 24 (x_d^2 over d = l mod 32) and combines them as
    // the xor butterfly's first two steps (16, then 8) would; the steps 4, 2,
    // 1 stay inside the eight lanes -- the standalone kernel's sum, bit for bit.
    static_assert(NREP + 1 <= 4 * kWarps, "one eight-lane group per row");
    {
      const int task = warp * 4 + (lane >> 3), sl = lane & 7;
      const bool is_k = task == NREP;
      const bool active = task <= NREP && (is_k ? krow : h0 + task < p.rope.q_heads);
      float *row = is_k ? rot.knew : rot.q[task < NREP ? task : 0];
      const float *wn = is_k ? (p.rope.k_norm ? rot.kw : nullptr) : (p.rope.q_norm ? rot.qw : nullptr);
      if (p.rope.q_norm || p.rope.k_norm) {  // uniform: the shuffles run in whole warps
        const bool normed = active && wn;
        float pl[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          pl[j] = 0.f;
#pragma unroll
          for (int k = 0; k < D / 32; ++k)
            pl[j] = normed ? rms_partial_add(pl[j], row[sl + 8 * j + 32 * k], k == 0) : 0.f;
        }
        float v = __fadd_rn(__fadd_rn(pl[0], pl[2]), __fadd_rn(pl[1], pl[3]));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
        const float rs = rms_scale(v, D, p.rope.eps);
        if (normed)
          for (int d = sl; d < D; d += 8) row[d] = rms_apply(row[d], rs, wn[d]);
      }
      __syncwarp();
      if (active) {
        for (int i = sl; i < D / 2; i += 8) {
          if (i < p.rope.half) {
            const int e0 = p.rope.interleaved ? 2 * i : i;
            const int e1 = p.rope.interleaved ? 2 * i + 1 : i + p.rope.half;
            float y0, y1;
            rope_rotate(row[e0], row[e1], rot.cs[i].x, rot.cs[i].y, y0, y1);
            if (is_k) {
              sm.newk[e0] = from_float<T>(y0);
              sm.newk[e1] = from_float<T>(y1);
            } else {
              row[e0] = to_float(from_float<T>(y0));
              row[e1] = to_float(from_float<T>(y1));
            }
          } else if (wn) {  // features past rot_dim keep their normalised value
            for (int d = 2 * p.rope.half + (i - p.rope.half); d < D; d += D / 2 - p.rope.half) {
              if (is_k) sm.newk[d] = from_float<T>(row[d]);
              else row[d] = to_float(from_float<T>(row[d]));
            }
          }
        }
      }
    }
    __syncthreads();
    if constexpr (use_mma<T>()) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        if (gq < NREP) {
          qa[kk][0] = pack2<T>(rot.q[gq][kk * 16 + 2 * tq], rot.q[gq][kk * 16 + 2 * tq + 1]);
          qa[kk][1] = pack2<T>(rot.q[gq][kk * 16 + 2 * tq + 8], rot.q[gq][kk * 16 + 2 * tq + 9]);
        }
      if constexpr (!Sm::kRotMisc) {
        // the rotation rows live in the K buffer: ordered before the copies
        // that will overwrite it
        fence_proxy_async_smem();
        __syncthreads();
      }
    }
  }
  // running state: mma path -- every lane holds the shared maximum of heads
  // 2 tq and 2 tq + 1, its rows' part of their l and its fragment of O^T
  // (rows: features, columns: heads); fp32 path -- per head in shared memory
  float m_run[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};
  float ot[use_mma<T>() ? D / 16 : 1][4];
  if constexpr (use_mma<T>()) {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) ot[mt][0] = ot[mt][1] = ot[mt][2] = ot[mt][3] = 0.f;
  }
  constexpr int ITEMS = (NREP * D / 2 + kThreads - 1) / kThreads;  // (head, feature pair) per thread
  float o[ITEMS][2];
#pragma unroll
  for (int u = 0; u < ITEMS; ++u) o[u][0] = o[u][1] = 0.f;
  bool ok = true;
  int failed_bt = -1;

  for (int bt = 0; bt < nbatch; ++bt) {
    const int nbc = min(CPB, n_ne - bt * CPB);  // chunks in this batch
    if (bt > 0 || !early) issue_batch(bt);
    ok = ok && mbar_wait(&sm.bar, bt & 1, p.err);
    ok = __syncthreads_and(ok);  // the batch landed, for every thread
    if (bt == 0) dec_stamp(4);
    if (!ok) {
      failed_bt = bt;
      break;
    }
    // masked rows: a zero V row (exact zeros through the product); the row a
    // fused append adds: the step's input. The mma path reads only the rows
    // of fetched chunk slots, so a batch of whole chunks without the new row
    // needs no pass (the same decision in every warp: one ballot over the
    // chunk lanes).
    const uint32_t fixm = __ballot_sync(
        0xffffffffu, my_rank >= bt * CPB && my_rank < bt * CPB + nbc &&
                         ((sm.words[lane][0] & sm.words[lane][1]) != 0xffffffffu ||
                          (pos >= 0 && (pos / C) % S == x && (pos / C) / S == lane)));
    if (fixm != 0u || (!use_mma<T>() && nbc < CPB)) {
      const int lim = use_mma<T>() ? nbc * C : CAPR;
      for (int r0 = warp * 32; r0 < lim; r0 += kThreads) {  // warp-uniform: 32 rows of one chunk slot
        const int r = r0 + lane;
        int chunk = -1;
        const uint2 w2 = chunk_words(bt, r / C, chunk);
        const bool allowed = ((((r % C) < 32) ? w2.x : w2.y) >> (r % 32)) & 1u;
        const bool is_new = allowed && pos >= 0 && (x + S * chunk) * C + (r % C) == pos;
        if (!allowed || is_new) {
#pragma unroll
          for (int sg = 0; sg < SEGS; ++sg) {
            const uint4 kz = is_new ? reinterpret_cast<const uint4 *>(sm.newk)[sg] : make_uint4(0u, 0u, 0u, 0u);
            const uint4 vz = is_new ? reinterpret_cast<const uint4 *>(sm.newv)[sg] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t off = use_mma<T>() ? Sm::seg_off(r, sg) : Sm::row_off(r) + sg * 16;
            if (is_new) *reinterpret_cast<uint4 *>(kbuf + off) = kz;
            *reinterpret_cast<uint4 *>(vbuf + off) = vz;
          }
          fence_proxy_async_smem();  // ordered before a later batch's TMA into this row
        }
      }
      __syncthreads();
    }
    if (bt == 0) dec_stamp(9);

    // ---- 3. the batch's products
    if constexpr (use_mma<T>()) {
      // S^T = K q^T and O^T += V^T P^T: the cache rows are the M side of the
      // score product (16 per mma, no padding rows) and the heads its N side
      // (8, padded with zero q columns); P^T becomes the B operand of the
      // second product by an in-register transpose of its two 8 x 8 halves.
      // Warp w takes the 16-row groups w, w + kWarps, ... of the fetched
      // slots: nbc groups for every warp, so the loops below are unrolled for
      // each batch size and their groups overlap.
      const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: tile, row within it
      auto products = [&](auto njc) {
        constexpr int NJ = decltype(njc)::value;
        float sc[NJ][4];  // (row gq | gq + 8) x (head 2 tq | 2 tq + 1), log2 units
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const int gi = warp + j * kWarps;
          int chunk;
          const uint2 w2 = chunk_words(bt, gi * 16 / C, chunk);
          // two accumulators (even / odd k steps) halve the dependent chain
          float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          const int krow = gi * 16 + (mi & 1) * 8 + rr;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(a0, a1, a2, a3, kbuf + Sm::seg_off(krow, 2 * kk + (mi >> 1)));
            mma_16816<T>(acc[kk & 1], a0, a1, a2, a3, qa[kk][0], qa[kk][1]);
          }
          const int s0 = (gi * 16) % C + gq, s1 = s0 + 8;  // slots within the chunk
          const bool al0 = ((s0 < 32 ? w2.x : w2.y) >> (s0 % 32)) & 1u;
          const bool al1 = ((s1 < 32 ? w2.x : w2.y) >> (s1 % 32)) & 1u;
          sc[j][0] = al0 ? (acc[0][0] + acc[1][0]) * p.scale_log2 : -INFINITY;
          sc[j][1] = al0 ? (acc[0][1] + acc[1][1]) * p.scale_log2 : -INFINITY;
          sc[j][2] = al1 ? (acc[0][2] + acc[1][2]) * p.scale_log2 : -INFINITY;
          sc[j][3] = al1 ? (acc[0][3] + acc[1][3]) * p.scale_log2 : -INFINITY;
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          mx0 = fmaxf(mx0, fmaxf(sc[j][0], sc[j][2]));
          mx1 = fmaxf(mx1, fmaxf(sc[j][1], sc[j][3]));
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        if (bt == 0) dec_stamp(11);
        if (gq == 0) {
          if (2 * tq < NREP) sm.wmax[warp][2 * tq] = mx0;
          if (2 * tq + 1 < NREP) sm.wmax[warp][2 * tq + 1] = mx1;
        }
        __syncthreads();
        if (bt == 0) dec_stamp(10);
        // finite: the batch holds an allowed row (padding heads use 0)
        float m_new[2], f[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * tq + e;
          float mb = -INFINITY;
          if (h < NREP) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) mb = fmaxf(mb, sm.wmax[w][h]);
          }
          m_new[e] = h < NREP ? fmaxf(m_run[e], mb) : 0.f;
          f[e] = (m_run[e] == -INFINITY) ? 0.f : fast_exp2(m_run[e] - m_new[e]);
          m_run[e] = m_new[e];
          l_part[e] *= f[e];
        }
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          ot[mt][0] *= f[0];
          ot[mt][1] *= f[1];
          ot[mt][2] *= f[0];
          ot[mt][3] *= f[1];
        }
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
          const int gi = warp + j * kWarps;
          const float p0 = fast_exp2(sc[j][0] - m_new[0]), p1 = fast_exp2(sc[j][1] - m_new[1]);
          const float p2 = fast_exp2(sc[j][2] - m_new[0]), p3 = fast_exp2(sc[j][3] - m_new[1]);
          l_part[0] += p0 + p2;
          l_part[1] += p1 + p3;
          // P^T (heads x rows) as the B operand: rows 0..7 of the group, then 8..15
          const uint32_t b0 = movmatrix_trans(pack2<T>(p0, p1));
          const uint32_t b1 = movmatrix_trans(pack2<T>(p2, p3));
          const int vrow = gi * 16 + (mi >> 1) * 8 + rr;
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4_trans(a0, a1, a2, a3, vbuf + Sm::seg_off(vrow, 2 * mt + (mi & 1)));
            mma_16816<T>(ot[mt], a0, a1, a2, a3, b0, b1);
          }
        }
      };
      // groups per warp: nbc (warp w's groups w + j kWarps lie in chunk slot j)
      static_assert(C / 16 == kWarps && CPB <= 4, "one group per warp per chunk slot");
      switch (nbc) {
        case 1: products(std::integral_constant<int, 1>()); break;
        case 2: if constexpr (CPB >= 2) products(std::integral_constant<int, 2>()); break;
        case 3: if constexpr (CPB >= 3) products(std::integral_constant<int, 3>()); break;
        default: if constexpr (CPB >= 4) products(std::integral_constant<int, 4>()); break;
      }
    } else {
      int chunk_w = -1;
      const uint2 ww = chunk_words(bt, (warp * RPW) / C, chunk_w);  // a warp's rows share a chunk
      auto row_allowed = [&](int row) {
        return (((row % C) < 32 ? ww.x : ww.y) >> (row % 32)) & 1u;
      };
      // scores (log2 units): GL lanes share a row, 16 bytes each
      constexpr int EPL = 16 / sizeof(T), GL = D / EPL, SPW = 32 / GL;
      static_assert(GL <= 32 && RPW % SPW == 0, "lane layout");
      const int e = lane % GL, sub = lane / GL;
      {
        float qr[NREP][EPL];
#pragma unroll
        for (int r = 0; r < NREP; ++r)
#pragma unroll
          for (int i = 0; i < EPL; ++i) qr[r][i] = rot.q[r][e * EPL + i];
        for (int it = 0; it < RPW / SPW; ++it) {
          const int row = warp * RPW + it * SPW + sub;
          float acc[NREP];
#pragma unroll
          for (int r = 0; r < NREP; ++r) acc[r] = 0.f;
          const uint4 uu = *reinterpret_cast<const uint4 *>(kbuf + Sm::row_off(row) + e * 16);
          float kf[EPL];
          unpack16_t<T>(uu, kf);
#pragma unroll
          for (int r = 0; r < NREP; ++r)
#pragma unroll
            for (int i = 0; i < EPL; ++i) acc[r] = fmaf(qr[r][i], kf[i], acc[r]);
#pragma unroll
          for (int off = GL / 2; off > 0; off >>= 1)
#pragma unroll
            for (int r = 0; r < NREP; ++r) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
          if (e == 0) {
            const bool al = row_allowed(row);
#pragma unroll
            for (int r = 0; r < NREP; ++r) sm.s[r][row] = al ? acc[r] * p.scale_log2 : -INFINITY;
          }
        }
      }
      __syncthreads();
      // per-head batch softmax, folded into the running (m, l)
      for (int r = warp; r < NREP; r += kWarps) {  // warp-uniform
        const float m_h = sm.mrun[r], l_h = sm.lrun[r];
        float mb = -INFINITY;
        for (int i = lane; i < CAPR; i += 32) mb = fmaxf(mb, sm.s[r][i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
        float lb = 0.f;
        for (int i = lane; i < CAPR; i += 32) {
          const float pr = exp2f(sm.s[r][i] - mb);
          sm.s[r][i] = pr;
          lb += pr;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) lb += __shfl_xor_sync(0xffffffffu, lb, off);
        const float m_new = fmaxf(m_h, mb);
        const float f_old = (m_h == -INFINITY) ? 0.f : exp2f(m_h - m_new);
        const float f_b = exp2f(mb - m_new);
        __syncwarp();
        if (lane == 0) {
          sm.fo[r] = f_old;
          sm.fb[r] = f_b;
          sm.mrun[r] = m_new;
          sm.lrun[r] = l_h * f_old + lb * f_b;
        }
      }
      __syncthreads();
      // P.V over the batch's rows, ascending
#pragma unroll
      for (int u = 0; u < ITEMS; ++u) {
        const int idx = tid + u * kThreads;
        if (idx < NREP * D / 2) {
          const int r = idx / (D / 2), dp = idx % (D / 2);
          float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
          for (int kk = 0; kk < CAPR; ++kk) {
            const float pr = sm.s[r][kk];
            const float2 vv = *reinterpret_cast<const float2 *>(vbuf + Sm::row_off(kk) + dp * 8);
            a0 = fmaf(pr, vv.x, a0);
            a1 = fmaf(pr, vv.y, a1);
          }
          o[u][0] = o[u][0] * sm.fo[r] + a0 * sm.fb[r];
          o[u][1] = o[u][1] * sm.fo[r] + a1 * sm.fb[r];
        }
      }
    }
    __syncthreads();  // the batch buffers (and the exchange slots) are free again
  }
  if (failed_bt >= 0) {
    // a batch's copies did not arrive in time: let them land (bounded) before
    // the buffers are reused or the CTA exits
    mbar_wait(&sm.bar, failed_bt & 1, p.err);
    __syncthreads();
  }
  dec_stamp(5);

  // in-CTA merge: every warp used the same maximum, so O and l are sums;
  // warps past the first batch's groups never held a row
  const int nact = use_mma<T>() ? min(kWarps, min(CPB, n_ne) * (C / 16)) : 0;
  if constexpr (use_mma<T>()) {
    float l0 = l_part[0], l1 = l_part[1];
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    const int h0l = 2 * tq, h1l = 2 * tq + 1;
    if (gq == 0 && warp == 0) {
      if (h0l < NREP) sm.mrun[h0l] = m_run[0];
      if (h1l < NREP) sm.mrun[h1l] = m_run[1];
    }
    if (warp < nact) {  // warp-uniform
      if (gq == 0) {
        if (h0l < NREP) sm.wsum[warp][h0l] = l0;
        if (h1l < NREP) sm.wsum[warp][h1l] = l1;
      }
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        if (h0l < NREP) {
          wo[warp][h0l][mt * 16 + gq] = ot[mt][0];
          wo[warp][h0l][mt * 16 + gq + 8] = ot[mt][2];
        }
        if (h1l < NREP) {
          wo[warp][h1l][mt * 16 + gq] = ot[mt][1];
          wo[warp][h1l][mt * 16 + gq + 8] = ot[mt][3];
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < ITEMS; ++u) {
      const int idx = tid + u * kThreads;
      if (idx < NREP * D / 2) {
        const int r = idx / (D / 2), dp = idx % (D / 2);
        float a0 = 0.f, a1 = 0.f;
        for (int w = 0; w < nact; ++w) {
          const float2 v2 = *reinterpret_cast<const float2 *>(&wo[w][r][2 * dp]);
          a0 += v2.x;
          a1 += v2.y;
        }
        o[u][0] = a0;
        o[u][1] = a1;
      }
    }
  }
  dec_stamp(6);

  // append: the CTA owning slot pos stores the new row into the cache (once
  // per KV head: only its first head group); no CTA of this step reads that
  // slot from the cache
  if (pos >= 0 && (pos / C) % S == x && h0 % p.n_rep == 0) {
    constexpr int PPR = D * sizeof(T) / 16;
    char *kd = const_cast<char *>(reinterpret_cast<const char *>(kg + (int64_t)pos * p.ks_l));
    char *vd = const_cast<char *>(reinterpret_cast<const char *>(vg + (int64_t)pos * p.vs_l));
    // the staged rows: the step's input, normalised and rotated when fused
    for (int part = tid; part < 2 * PPR; part += kThreads) {
      if (part < PPR)
        reinterpret_cast<uint4 *>(kd)[part] = reinterpret_cast<const uint4 *>(sm.newk)[part];
      else
        reinterpret_cast<uint4 *>(vd)[part - PPR] = reinterpret_cast<const uint4 *>(sm.newv)[part - PPR];
    }
  }

  // ---- 4. every split delivers each owner its slice: output pair e (head
  // e / D, feature e % D) belongs to CTA e / E
  cluster_wait();  // every CTA of the cluster armed its receive barrier
#pragma unroll
  for (int u = 0; u < ITEMS; ++u) {
    const int idx = tid + u * kThreads;
    if (idx < NREP * D / 2) {
      const int e = 2 * idx, y = e / E;
      st_async_f32x2(cluster_map(&sm.rx_o[x][e % E], y), o[u][0], o[u][1], cluster_map(&sm.rx_bar, y));
    }
  }
  for (int t = tid; t < S * NREP; t += kThreads) {
    const int r = t / S, y = t % S;
    // this CTA's partial (m, l) of head r; m = -inf: nothing allowed (or a
    // batch that never arrived), and the owner skips the split
    const float m = sm.mrun[r];
    float l = sm.lrun[r];
    if constexpr (use_mma<T>()) {
      l = 0.f;
      for (int w = 0; w < nact; ++w) l += sm.wsum[w][r];
    }
    const bool has = ok && m != -INFINITY;
    st_async_f32x2(cluster_map(&sm.rx_ml[x][r], y), has ? m : -INFINITY, has ? l : 0.f,
                   cluster_map(&sm.rx_bar, y));
  }
  dec_stamp(7);

  // the owner's merge, in ascending split order. Its wait outlasts every
  // split's own copy waits (each batch, then the drain of a failed one), so a
  // split that gave up still delivers before the owner does.
  constexpr uint64_t kRxLimitNs = (uint64_t)(kMaxCI / CPB + 2) * kWaitLimitNs;
  if (tid < E / 2) {
    if (mbar_wait_cluster(&sm.rx_bar, 0, p.err, kRxLimitNs)) {
      const int e0 = x * E + 2 * tid;
      const int r = e0 / D, d = e0 % D;
      float Mx = -INFINITY;
#pragma unroll
      for (int xx = 0; xx < S; ++xx) Mx = fmaxf(Mx, sm.rx_ml[xx][r].x);
      float L = 0.f, o0 = 0.f, o1 = 0.f;
      if (Mx != -INFINITY) {
#pragma unroll
        for (int xx = 0; xx < S; ++xx) {
          const float2 ml = sm.rx_ml[xx][r];
          if (ml.x == -INFINITY) continue;
          const float w = exp2f(ml.x - Mx);
          L = fmaf(ml.y, w, L);
          o0 = fmaf(sm.rx_o[xx][2 * tid], w, o0);
          o1 = fmaf(sm.rx_o[xx][2 * tid + 1], w, o1);
        }
      }
      const float inv = (L > 0.f) ? 1.f / L : 0.f;
      T *orow = static_cast<T *>(p.out) + (int64_t)b * p.os_b + (int64_t)(h0 + r) * p.os_h;
      orow[d] = from_float<T>(o0 * inv);
      orow[d + 1] = from_float<T>(o1 * inv);
      if (d == 0 && p.lse)
        p.lse[(int64_t)b * p.Hq + h0 + r] = (L > 0.f) ? (Mx + log2f(L)) * kLn2 : -INFINITY;
    }
  }
  dec_stamp(8);
}

template <typename T, int D, int NREP>
mgqa_status launch_t(const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                     cudaStream_t s) {
  auto kern = decode_kernel<T, D, NREP>;
  constexpr int smem = DecodeSmem<T, D, NREP>::total;
  static std::atomic<uint64_t> attr_done{0};
  const mgqa_status st = ensure_cluster_attr(kern, smem, attr_done, "decode kernel");
  if (st != MGQA_OK) return st;
  dim3 grid(S, p.Hq / NREP, p.B);
  const cudaError_t e = launch_pdl_cluster(kern, grid, dim3(kThreads), smem, s, S, mk, mv, p);
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
  return MGQA_OK;
}

template <typename T, int D>
mgqa_status launch_nrep(const CUtensorMap &mk, const CUtensorMap &mv, const DecodeParams &p,
                        int hpc, cudaStream_t s) {
  switch (hpc) {
    case 1: return launch_t<T, D, 1>(mk, mv, p, s);
    case 2: return launch_t<T, D, 2>(mk, mv, p, s);
    case 4: return launch_t<T, D, 4>(mk, mv, p, s);
    case 8: return launch_t<T, D, 8>(mk, mv, p, s);
    default: return fail(MGQA_ERR_UNSUPPORTED, "decode: heads per CTA %d", hpc);
  }
}

}  // namespace

int decode_heads_per_cta(int n_rep) {
  for (int h : {8, 4, 2, 1})
    if (n_rep % h == 0) return h;
  return 1;
}

mgqa_status launch_decode(const mgqa_args &a, cudaStream_t s) {
  return launch_decode_append(a, nullptr, nullptr, nullptr, nullptr, nullptr, s);
}

mgqa_status launch_decode_append(const mgqa_args &a, const void *k_new, const void *v_new,
                                 const int64_t *k_new_stride, const int64_t *v_new_stride,
                                 int32_t *kv_len_out, cudaStream_t s, const FusedRope &rope) {
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
  p.rope = rope;
  p.append = k_new != nullptr;
  if (p.append) {
    p.k_new = k_new;
    p.v_new = v_new;
    p.kn_b = k_new_stride[0]; p.kn_h = k_new_stride[1];
    p.vn_b = v_new_stride[0]; p.vn_h = v_new_stride[1];
    p.kv_len_out = kv_len_out;
  }
  const int hpc = decode_heads_per_cta(p.n_rep);
  // the cache as TMA boxes of 64 slots: 64-column 128-byte-swizzled boxes for
  // the 16-bit types, whole fp32 rows otherwise
  const bool half16 = a.dtype != MGQA_FP32;
  CUtensorMap mk, mv;
  if (!make_tma_map_4d(&mk, a.dtype, a.k, a.B, a.Hkv, a.Lk, a.D, a.k_stride, half16 ? 64 : a.D,
                       kDecodeChunk, half16) ||
      !make_tma_map_4d(&mv, a.dtype, a.v, a.B, a.Hkv, a.Lk, a.D, a.v_stride, half16 ? 64 : a.D,
                       kDecodeChunk, half16))
    return fail(MGQA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the decode cache");
  if (a.dtype == MGQA_BF16) {
    if (a.D == 64) return launch_nrep<__nv_bfloat16, 64>(mk, mv, p, hpc, s);
    if (a.D == 128) return launch_nrep<__nv_bfloat16, 128>(mk, mv, p, hpc, s);
  } else if (a.dtype == MGQA_FP16) {
    if (a.D == 64) return launch_nrep<__half, 64>(mk, mv, p, hpc, s);
    if (a.D == 128) return launch_nrep<__half, 128>(mk, mv, p, hpc, s);
  } else {
    if (a.D == 64) return launch_nrep<float, 64>(mk, mv, p, hpc, s);
    if (a.D == 128) return launch_nrep<float, 128>(mk, mv, p, hpc, s);
  }
  return fail(MGQA_ERR_UNSUPPORTED, "decode: head dim %d", a.D);
}

}  // namespace mgqa

// ---- decode for callers that hand the library no device memory ------------
// The kernel merges its splits on chip, so this needs no scratch of any kind:
// it is the workspace-free form of masked_gqa_attn_decode.

extern "C" mgqa_status masked_gqa_attn_decode_static(const mgqa_args *args, cudaStream_t stream) {
  return masked_gqa_attn_decode(args, nullptr, 0, stream);
}

// ---- debug library entry point (include/masked_gqa_attn_debug.h) ------------
#ifdef MGQA_DEBUG
#include "../../include/masked_gqa_attn_debug.h"

extern "C" MGQA_API mgqa_status mgqa_debug_decode_timeline(uint64_t *out, int32_t n_ctas) {
  using namespace mgqa;
  clear_error_detail();
  if (!out || n_ctas < 0 || n_ctas > kTlCtas)
    return fail(MGQA_ERR_INVALID_ARG, "mgqa_debug_decode_timeline: bad output or count");
  cudaError_t e = cudaMemcpyFromSymbol(out, g_dec_tl, (size_t)n_ctas * kTlStamps * sizeof(uint64_t));
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "reading the timeline: %s", cudaGetErrorString(e));
  static const unsigned long long zeros[kTlCtas][kTlStamps] = {};
  e = cudaMemcpyToSymbol(g_dec_tl, zeros, sizeof(zeros));
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "clearing the timeline: %s", cudaGetErrorString(e));
  return MGQA_OK;
}
#endif  // MGQA_DEBUG
