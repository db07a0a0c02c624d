// Full-sequence masked GQA attention on the tensor cores (bf16 or fp16 in,
// fp32 accumulation): TMA-staged Q/K/V tiles, tcgen05 MMAs accumulating in tensor
// memory, a warp-specialised load / MMA / softmax pipeline, and whole-tile
// skipping wherever the mask leaves a 128x128 (query, key) tile empty.
//
// Passages: VoxCPM page, "Upstream-identical practice", attention bullet
// (SDPA with enable_gqa, bidirectional in the local DiT, explicit boolean
// mask whose masked positions add exact zeros); OmniVoice page,
// "Upstream-identical practice", attention-mask bullet (4D boolean mask, not
// causal, KV heads repeated; conditional and unconditional rows in one batch)
// and "Memory & speed", packed_guidance paragraph (both sequences in one row
// under a block-diagonal mask, so the padded half of the unconditional row is
// never computed).
//
// CTA = one 128-row query tile of NT query heads that share one KV head
// (NT = 2 when Hq/Hkv is even), so each K/V tile is fetched once for both.
//   warp 0      : TMA producer (Q once, then K and V per key tile, STAGES-deep)
//   warp 1      : allocates tensor memory and runs the MMA loop; one elected
//                 lane issues every MMA
//   warps 4..   : one softmax warpgroup per query head (thread = query row)
// With two heads (384 threads, 168 registers each at launch) the first
// warpgroup gives registers away (104) and the softmax warpgroups take them
// (200; 104 + 2 x 200 = 3 x 168 per scheduler), enough to hold a whole
// 128-column score row per thread.
// Tensor memory: S_t (128 fp32 columns) and O_t (D fp32 columns) per head;
// P_t (16-bit) overwrites the first 64 columns of S_t and is the A operand of
// the P.V MMA straight from tensor memory.
// Per key tile n and head t:
//   MMA:     S_t = Q_t K_n^T              -> s_full[t]
//   softmax: mask (partial tiles only), running max with lazy rescale of O_t
//            (only when the max grows by more than 2^8), P = exp2(x - m)
//            -> p_full[t]; every exponential is one MUFU ex2 (measured: the
//            MUFU pass beats moving part of them to an FMA-pipe polynomial,
//            whose extra instructions cost more issue slots than they save)
//   MMA:     O_t += P_t V_n               -> v_empty after both heads;
//                                             o_done[t] after the last tile
// S_t(n+1) is issued right behind O_t += P_t(n) V(n) (same issuing thread,
// executed in order), so head t needs no completion round trip between
// them; the waits for the next tile's K and V sit inside P.V groups and the
// P waits are probed ahead, so few waits fall between groups of MMAs.
// Before the pipeline, all warps classify the key tiles of this query tile
// as empty / full / partial from the mask forms; only non-empty tiles enter
// the pipeline and only partial tiles pay for per-element masking. Key tile
// 0 is loaded speculatively together with Q while the classification runs;
// when the first non-empty tile is another one, the producer lets that load
// land, raises a one-shot barrier and reloads stage 0 (the MMA warp waits
// for that barrier, then for stage 0's second phase).
// Every wait is bounded (about 2 s) and reports MGQA_ERR_TIMEOUT.
#include <climits>
#include <cmath>
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace mgqa {
namespace {

constexpr int BM = 128;       // query rows per tile
constexpr int BN = 128;       // keys per tile
constexpr int MAXKT = 2048;   // key tiles per row (Lk <= 262144)
constexpr int BOX = 16384;    // one TMA box: 128 rows x 64 bf16 (128 B, swizzled)

// Debug library only (MGQA_DEBUG): event counters, an injected producer fault
// and a settable wait limit, read and written by the mgqa_debug_* entry points.
#ifdef MGQA_DEBUG
struct DebugState {
  unsigned long long counters[4];  // see mgqa_debug_counters
  int fault_tile;                  // >= 0: the producer stops issuing at this non-empty tile
  unsigned long long wait_limit_ns;
};
__device__ DebugState g_dbg = {{0ull, 0ull, 0ull, 0ull}, -1, kWaitLimitNs};
MGQA_DEV uint64_t wait_limit() { return *(volatile unsigned long long *)&g_dbg.wait_limit_ns; }
MGQA_DEV int fault_tile() { return *(volatile int *)&g_dbg.fault_tile; }
MGQA_DEV void dbg_count(int i, unsigned long long n = 1ull) { atomicAdd(&g_dbg.counters[i], n); }
// per-CTA phase timeline (SM clock; slot 13: global timer at entry, 14: at
// the end of head 0's epilogue, 15: SM id), read with mgqa_debug_prefill_timeline
constexpr int kPreTlCtas = 1024, kPreTlStamps = 16;
__device__ unsigned long long g_pre_tl[kPreTlCtas][kPreTlStamps];
MGQA_DEV void pre_stamp(int k) {  // by the one thread that owns stamp k
  const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  if (cta >= (unsigned)kPreTlCtas) return;
  g_pre_tl[cta][k] = clock64();
  if (k == 0) {
    g_pre_tl[cta][13] = globaltimer_ns();
    unsigned sm;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
    g_pre_tl[cta][15] = sm;
  }
  if (k == 7) g_pre_tl[cta][14] = globaltimer_ns();
}
// per-tile event trace of the first CTAs (SM clock), read with
// mgqa_debug_prefill_trace: for the n-th non-empty key tile, 2t / 2t+1 = the
// MMA warp begins issuing / has committed S_t(n), 4+2t / 5+2t = the same for
// O_t += P_t(n) V(n), 8+4t = softmax t sees S_t(n) (its first warp), 9+4t =
// every warp has read it, 10+4t = the first warp's exponentials are done,
// 11+4t = every warp has handed P_t(n) over; 16 / 17 = the producer has
// issued K(n) / V(n)
constexpr int kTrCtas = 4, kTrTiles = 64, kTrEvents = 18;
__device__ unsigned long long g_pre_tr[kTrCtas][kTrTiles][kTrEvents];
MGQA_DEV unsigned long long *tr_slot(int n, int ev) {
  const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  return (cta < (unsigned)kTrCtas && n < kTrTiles) ? &g_pre_tr[cta][n][ev] : nullptr;
}
MGQA_DEV void tr_stamp(int n, int ev) {
  if (unsigned long long *s = tr_slot(n, ev)) *s = clock64();
}
MGQA_DEV void tr_stamp_max(int n, int ev) {  // the latest of several warps
  if (unsigned long long *s = tr_slot(n, ev)) atomicMax(s, (unsigned long long)clock64());
}
#else
MGQA_DEV void pre_stamp(int) {}
MGQA_DEV void tr_stamp(int, int) {}
MGQA_DEV void tr_stamp_max(int, int) {}
MGQA_DEV uint64_t wait_limit() { return kWaitLimitNs; }
MGQA_DEV int fault_tile() { return -1; }
MGQA_DEV void dbg_count(int, unsigned long long = 1ull) {}
#endif

struct TcParams {
  MaskView mask;
  int B, Hq, Hkv, Lq, Lk, n_rep, nkt;
  float scale_log2;
  void *out;
  int64_t os[3];
  const void *q, *k, *v;            // the tensors behind the maps (L2 hints only)
  int64_t qs[3], ks[3], vs[3];
  int warm;                         // the grid fits in one wave: hint the first reads early
  float *lse;
  int32_t *err;
  FusedRope rope;  // applied to the query tile in shared memory (inv_freq null: none)
};

template <int D, int NT, int STAGES>
struct Layout {
  static constexpr int KB = D / 64;  // TMA boxes per 128-row tile
  static constexpr int q_off = 0;
  static constexpr int k_off = q_off + NT * KB * BOX;
  static constexpr int v_off = k_off + STAGES * KB * BOX;
  static constexpr int bar_off = v_off + STAGES * KB * BOX;
  // barriers: q, k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[NT], p_full[NT],
  // o_done[NT], spec (the speculative tile-0 loads have landed), drain (every MMA
  // issued has completed; used when a wait gave up), q_rot[NT] (head t's query
  // tile is rotated; fused rotary embedding only)
  static constexpr int n_bars = 1 + 4 * STAGES + 3 * NT + 2 + NT;
  static constexpr int misc_off = bar_off + 8 * n_bars;
  static constexpr int tmem_slot = misc_off;        // uint32
  static constexpr int seg_slot = misc_off + 8;     // int32 x2 (min, max of seg_q)
  static constexpr int any_off = misc_off + 16;     // uint32[MAXKT/32]: tile has an allowed bit
  static constexpr int all_off = any_off + MAXKT / 8;  // uint32[MAXKT/32]: tile all allowed
  static constexpr int ne_off = all_off + MAXKT / 8;   // uint32[MAXKT/32]: tile is non-empty
  static constexpr int full_off = ne_off + MAXKT / 8;  // uint32[MAXKT/32]: tile needs no masking
  // fused rotation: the inverse frequencies and the q norm weights, staged once
  static constexpr int rope_off = (full_off + MAXKT / 8 + 15) & ~15;  // float[D / 2] then float[D]
  static constexpr int total = rope_off + (D / 2 + D) * 4;
  static constexpr int smem_bytes = total + 1024;   // slack for 1024-B alignment
  static constexpr int threads = 128 * (1 + NT);
  static constexpr int tmem_cols_used = NT * (BN + D);
  static constexpr uint32_t tmem_cols = tmem_cols_used <= 32 ? 32 : tmem_cols_used <= 64 ? 64
                                        : tmem_cols_used <= 128 ? 128
                                        : tmem_cols_used <= 256 ? 256 : 512;
  static_assert(tmem_cols_used <= 512, "tensor memory");
};

// The first non-empty key tile after `prev` (-1: the first), or nkt.
MGQA_DEV int next_tile(const uint32_t *ne, int prev, int nkt) {
  int kt = prev + 1;
  while (kt < nkt) {
    const uint32_t w = ne[kt >> 5] >> (kt & 31);
    if (w) return kt + __ffs(w) - 1;
    kt = (kt | 31) + 1;
  }
  return nkt;
}

// Allowed-key words of one query row for a partial key tile (keys k0..k0+127).
// Segment ids: each lane loads 4 of the tile's key ids (coalesced) and the
// warp builds each row's words with ballots, one round per distinct query
// segment among its 32 rows (usually one or two).
MGQA_DEV void tile_mask_words(const TcParams &p, int b, int i, bool row_ok, int k0, int kvl,
                              int segq, int lane, uint32_t (&mw)[BN / 32]) {
#pragma unroll
  for (int w = 0; w < BN / 32; ++w) {
    const int jw = k0 + 32 * w;
    int lim = min(p.Lk, kvl) - jw;
    if (p.mask.causal) lim = min(lim, i + p.mask.coff + 1 - jw);
    mw[w] = lim >= 32 ? 0xffffffffu : (lim <= 0 ? 0u : ((1u << lim) - 1u));
  }
  if (p.mask.bits) {
    const uint32_t *mrow = p.mask.bits + (int64_t)b * p.mask.sb + (int64_t)i * p.mask.sq;
    uint32_t v[BN / 32];
#pragma unroll
    for (int w = 0; w < BN / 32; ++w) v[w] = (mw[w] != 0u) ? __ldg(mrow + ((k0 >> 5) + w)) : 0u;
#pragma unroll
    for (int w = 0; w < BN / 32; ++w) mw[w] &= v[w];
  }
  if (p.mask.seg_q) {
    int sk[BN / 32];
#pragma unroll
    for (int w = 0; w < BN / 32; ++w) {
      const int j = k0 + 32 * w + lane;
      sk[w] = j < p.Lk ? __ldg(p.mask.seg_k + (int64_t)b * p.Lk + j) : -1;
    }
    const int mine = (row_ok && segq >= 0) ? segq : -1;
    uint32_t sw[BN / 32] = {0u, 0u, 0u, 0u};
    uint32_t pending = __ballot_sync(0xffffffffu, mine >= 0);
    while (pending) {
      const int x = __shfl_sync(0xffffffffu, mine, __ffs(pending) - 1);
#pragma unroll
      for (int w = 0; w < BN / 32; ++w) {
        const uint32_t bw = __ballot_sync(0xffffffffu, sk[w] == x);
        if (mine == x) sw[w] = bw;
      }
      pending &= ~__ballot_sync(0xffffffffu, mine == x);
    }
#pragma unroll
    for (int w = 0; w < BN / 32; ++w) mw[w] &= sw[w];
  }
  if (!row_ok) {
#pragma unroll
    for (int w = 0; w < BN / 32; ++w) mw[w] = 0u;
  }
}

// 16-bit value `hi` (0: low half) of a packed pair, as a float.
template <typename T> MGQA_DEV float half_of(uint32_t v, int hi);
template <> MGQA_DEV float half_of<__nv_bfloat16>(uint32_t v, int hi) {
  return __uint_as_float(hi ? (v & 0xffff0000u) : (v << 16));
}
template <> MGQA_DEV float half_of<__half>(uint32_t v, int hi) {
  return __half2float(__ushort_as_half((unsigned short)(hi ? (v >> 16) : (v & 0xffffu))));
}

// The rotary embedding's pairs of one row held as floats, in place. Every
// index is a constant (interleaved pairs stop at rp.half; half-split pairs
// have HALF as a template argument), so the row stays in registers.
template <int D, bool INTERLEAVED, int HALF>
MGQA_DEV void rope_row_pairs(float (&x)[D], const FusedRope &rp, const float *invf, int pos) {
  const int half = INTERLEAVED ? rp.half : HALF;
#pragma unroll
  for (int i = 0; i < D / 2; ++i) {
    if (i >= half) break;
    const int e0 = INTERLEAVED ? 2 * i : i;
    const int e1 = INTERLEAVED ? 2 * i + 1 : i + half;
    float sn, cs, y0, y1;
    rope_sincos(rope_theta(pos, invf[i]), sn, cs);
    rope_rotate(x[e0], x[e1], cs, sn, y0, y1);
    x[e0] = y0;
    x[e1] = y1;
  }
}

// RMS normalisation and rotary embedding of query row r of one head's tile
// in shared memory (128-byte-swizzled 64-column boxes), in place: the same
// arithmetic as the standalone rotary-embedding kernel. invf and qw are the
// frequency table and the norm weights staged in shared memory.
template <typename T, int D>
MGQA_DEV void rope_q_row(unsigned char *tile, int r, int pos, const FusedRope &rp,
                         const float *invf, const float *qw) {
  float x[D];  // the row as floats (16-bit values are exact in fp32)
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const uint4 u = *reinterpret_cast<const uint4 *>(tile + (c >> 3) * BOX + r * 128 +
                                                      (((c & 7) ^ (r & 7)) << 4));
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) x[8 * c + j] = half_of<T>(w4[j >> 1], j & 1);
  }
  if (rp.q_norm) {
    const float rs = rms_scale(rms_sum_row<D>(x), D, rp.eps);
#pragma unroll
    for (int d = 0; d < D; ++d) x[d] = rms_apply(x[d], rs, qw[d]);
  }
  // half-split widths D/2, D/4, D/8 (the host refuses others)
  if (rp.interleaved) rope_row_pairs<D, true, 0>(x, rp, invf, pos);
  else if (rp.half == D / 2) rope_row_pairs<D, false, D / 2>(x, rp, invf, pos);
  else if (rp.half == D / 4) rope_row_pairs<D, false, D / 4>(x, rp, invf, pos);
  else rope_row_pairs<D, false, D / 8>(x, rp, invf, pos);
#pragma unroll
  for (int c = 0; c < D / 8; ++c)  // one rounding to the I/O type
    *reinterpret_cast<uint4 *>(tile + (c >> 3) * BOX + r * 128 + (((c & 7) ^ (r & 7)) << 4)) =
        make_uint4(pack2<T>(x[8 * c], x[8 * c + 1]), pack2<T>(x[8 * c + 2], x[8 * c + 3]),
                   pack2<T>(x[8 * c + 4], x[8 * c + 5]), pack2<T>(x[8 * c + 6], x[8 * c + 7]));
}

// One 128-key tile of one softmax row (thread = row): the whole score row is
// read from tensor memory once (four 32-column loads, one wait); its extreme
// (8 independent accumulators) updates the running max with lazy rescale of O
// (only when it grows by more than 2^8); P = exp2(s*scale*log2e - m) goes
// back as bf16 pairs over the first 64 S columns; the row sum is added to l.
// NEG: negative scale (the max of scaled scores is the min of raw ones).
// PARTIAL: mw holds the row's allowed-key bits.
template <typename T, int D, bool NEG, bool PARTIAL>
MGQA_DEV void softmax_tile(uint32_t t_s, uint32_t t_o, const uint32_t (&mw)[BN / 32], float sl2,
                           float &m_used, float &l, int n, int tr) {
  constexpr float MV = NEG ? INFINITY : -INFINITY;
  uint32_t sr[BN];
  float mr;
  if constexpr (!PARTIAL) {
    // full tile: the loads also reduce each 32-column piece of the row
    float red[BN / 32];
#pragma unroll
    for (int c = 0; c < BN / 32; ++c)
      tc::tmem_ld32_red<!NEG>(t_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]),
                              red[c]);
    tc::tmem_wait_ld();
    if (tr >= 0) tr_stamp_max(n, (tr & 0xff) + 1);
    mr = NEG ? fminf(fminf(red[0], red[1]), fminf(red[2], red[3]))
             : fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  } else {
#pragma unroll
    for (int c = 0; c < BN / 32; ++c)
      tc::tmem_ld32(t_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
    tc::tmem_wait_ld();
    if (tr >= 0) tr_stamp_max(n, (tr & 0xff) + 1);
    float mx[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) mx[k] = MV;
#pragma unroll
    for (int j = 0; j < BN; ++j) {
      float a = __uint_as_float(sr[j]);
      if (!((mw[j >> 5] >> (j & 31)) & 1u)) a = MV;
      mx[j & 7] = NEG ? fminf(mx[j & 7], a) : fmaxf(mx[j & 7], a);
    }
#pragma unroll
    for (int k = 4; k > 0; k >>= 1)
#pragma unroll
      for (int u = 0; u < k; ++u) mx[u] = NEG ? fminf(mx[u], mx[u + k]) : fmaxf(mx[u], mx[u + k]);
    mr = mx[0];
  }
  const float m_tile = (PARTIAL && mr == MV) ? -INFINITY : mr * sl2;
  const float m_new = fmaxf(m_used, m_tile);
  bool rescale = false;
  float factor = 1.f;
  if (m_used == -INFINITY) {
    m_used = m_new;
  } else if (m_new - m_used > 8.f) {
    rescale = true;
    factor = tc::ex2(m_used - m_new);
    m_used = m_new;
    l *= factor;
  }
  if (__any_sync(0xffffffffu, rescale)) {
    // O holds every P.V issued so far: this tile's S MMA was issued after the
    // previous tile's P.V, and its completion covers that MMA.
    if ((threadIdx.x & 31) == 0) dbg_count(0);  // debug library: rescale events (per warp)
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tc::tmem_ld32(t_o + c * 32, o);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * factor);
      tc::tmem_st32(t_o + c * 32, o);
    }
    tc::tmem_wait_st();
  }
  const float mb = (m_used == -INFINITY) ? 0.f : m_used;
  const uint64_t sl2x2 = tc::pk2(sl2, sl2), nmb2 = tc::pk2(-mb, -mb);
  uint64_t acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = tc::pk2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int col = c * 32 + 2 * j;
      const uint64_t y =
          tc::fma2(tc::pk2(__uint_as_float(sr[col]), __uint_as_float(sr[col + 1])), sl2x2, nmb2);
      float y0, y1;
      tc::upk2(y, y0, y1);
      float p0 = tc::ex2(y0), p1 = tc::ex2(y1);
      if (PARTIAL) {
        if (!((mw[c] >> (2 * j)) & 1u)) p0 = 0.f;
        if (!((mw[c] >> (2 * j + 1)) & 1u)) p1 = 0.f;
      }
      acc[j & 3] = tc::add2(acc[j & 3], tc::pk2(p0, p1));
      pk[j] = pack2<T>(p0, p1);
    }
    tc::tmem_st16(t_s + c * 16, pk);
  }
  acc[0] = tc::add2(acc[0], acc[1]);
  acc[2] = tc::add2(acc[2], acc[3]);
  acc[0] = tc::add2(acc[0], acc[2]);
  float s0, s1;
  tc::upk2(acc[0], s0, s1);
  l += s0 + s1;
  if (tr >= 0 && (tr >> 8) == 0) tr_stamp(n, (tr & 0xff) + 2);
  tc::tmem_wait_st();
}

// ROPE: the query tile is normalised / rotated in shared memory first (a
// separate instantiation, so the plain kernel carries none of that code).
template <typename T, int D, int NT, int STAGES, bool ROPE>
__global__ void __launch_bounds__(128 * (1 + NT), 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const __grid_constant__ TcParams p) {
  using Lay = Layout<D, NT, STAGES>;
  constexpr int KB = Lay::KB;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::bar_off);
  uint64_t *bar_q = bars;
  uint64_t *bar_kfull = bars + 1;
  uint64_t *bar_vfull = bars + 1 + STAGES;
  uint64_t *bar_kempty = bars + 1 + 2 * STAGES;
  uint64_t *bar_vempty = bars + 1 + 3 * STAGES;
  uint64_t *bar_sfull = bars + 1 + 4 * STAGES;
  uint64_t *bar_pfull = bar_sfull + NT;
  uint64_t *bar_odone = bar_pfull + NT;
  uint64_t *bar_spec = bar_odone + NT;
  uint64_t *bar_drain = bar_spec + 1;
  uint64_t *bar_qrot = bar_drain + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lay::tmem_slot);
  int *seg_slot = reinterpret_cast<int *>(smem + Lay::seg_slot);
  uint32_t *any_bits = reinterpret_cast<uint32_t *>(smem + Lay::any_off);
  uint32_t *all_bits = reinterpret_cast<uint32_t *>(smem + Lay::all_off);
  uint32_t *ne_bits = reinterpret_cast<uint32_t *>(smem + Lay::ne_off);
  uint32_t *full_bits = reinterpret_cast<uint32_t *>(smem + Lay::full_off);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int qt = blockIdx.x, hp = blockIdx.y, b = blockIdx.z;
  const int h0 = hp * NT;
  const int g = h0 / p.n_rep;
  const int row0 = qt * BM;
  const int rows = min(BM, p.Lq - row0);

  // ---- set-up that touches no global memory (may overlap the previous kernel)
  if (tid == 0) pre_stamp(0);
  if (tid == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_kfull + s, 1);
      mbar_init(bar_vfull + s, 1);
      mbar_init(bar_kempty + s, 1);
      mbar_init(bar_vempty + s, 1);
    }
    for (int t = 0; t < NT; ++t) {
      mbar_init(bar_sfull + t, 1);
      mbar_init(bar_pfull + t, 128);
      mbar_init(bar_odone + t, 1);
    }
    mbar_init(bar_spec, 1);
    mbar_init(bar_drain, 1);
    for (int t = 0; t < NT; ++t) mbar_init(bar_qrot + t, 128);
    fence_mbarrier_init();
    tc::prefetch_tensormap(&tm_q);
    tc::prefetch_tensormap(&tm_k);
    tc::prefetch_tensormap(&tm_v);
    tc::prefetch_tensormap(&tm_o);
    allow_dependents();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, Lay::tmem_cols);
  for (int w = tid; w < (p.nkt + 31) / 32; w += blockDim.x) {
    ne_bits[w] = 0u;
    full_bits[w] = 0u;
    if (p.mask.bits) {
      any_bits[w] = 0u;
      all_bits[w] = 0xffffffffu;
    }
  }
  if (p.warm) {
    // before the grid-dependency wait, hints that move this CTA's first reads
    // toward the L2 (nothing enters the SM; the L2 is the point of coherence,
    // so a later write by the previous kernel still wins): the Q rows of its
    // heads, key tile 0's K and V rows (loaded speculatively below) and the
    // first block of its mask rows. They overlap the previous kernel's tail,
    // which only a grid of one wave waits out (later waves start after it).
    const T *qg = static_cast<const T *>(p.q);
    constexpr int LPR = D * (int)sizeof(T) / 128;  // 128-byte lines per row
    const int nq = NT * rows * LPR, nk0 = 2 * min(BN, p.Lk) * LPR;
    for (int u = tid; u < nq + nk0; u += blockDim.x) {
      if (u < nq) {
        const int t = u / (rows * LPR), rr = (u / LPR) % rows, ln = u % LPR;
        prefetch_l2(qg + ((int64_t)b * p.qs[0] + (int64_t)(h0 + t) * p.qs[1] + (int64_t)(row0 + rr) * p.qs[2]) +
                    ln * (128 / (int)sizeof(T)));
      } else {
        const int w = u - nq, kv = w / (nk0 / 2), rr = (w / LPR) % min(BN, p.Lk), ln = w % LPR;
        const T *base = static_cast<const T *>(kv ? p.v : p.k);
        const int64_t *st = kv ? p.vs : p.ks;
        prefetch_l2(base + ((int64_t)b * st[0] + (int64_t)g * st[1] + (int64_t)rr * st[2]) +
                    ln * (128 / (int)sizeof(T)));
      }
    }
    if (p.mask.bits && tid < rows)
      prefetch_l2(p.mask.bits + (int64_t)b * p.mask.sb + (int64_t)(row0 + tid) * p.mask.sq);
    // and the other inputs of the tile classification: the row's kv_len, the
    // query tile's segment ids and the row's key segment ids (32 per line)
    if (p.mask.kv_len && tid == 0) prefetch_l2(p.mask.kv_len + b);
    if (p.mask.seg_q) {
      const int nq = (rows + 31) / 32, nkl = (p.Lk + 31) / 32;
      for (int u = tid; u < nq + nkl; u += blockDim.x)
        prefetch_l2(u < nq ? p.mask.seg_q + (int64_t)b * p.Lq + row0 + 32 * u
                           : p.mask.seg_k + (int64_t)b * p.Lk + 32 * (u - nq));
    }
  }
  grid_dependency_wait();
  if (tid == 0) pre_stamp(1);
  // packed-bit mask words of the first 32-word block (1024 keys) of this
  // warp's rows, requested before anything else (the copies below move
  // 64 KB or more per CTA; these few words should not queue behind them).
  // At most 16 rows per warp (128 rows, >= 8 warps): every load in flight.
  const int mW = (p.Lk + 31) >> 5;
  auto mask_words = [&](int wb, uint32_t (&wv)[BM / 8]) {
    const int w = wb + lane;
    const int lim_k = p.Lk - 32 * w;
    const uint32_t valid = w >= mW ? 0u : (lim_k >= 32 ? 0xffffffffu : ((1u << lim_k) - 1u));
#pragma unroll
    for (int k = 0; k < BM / 8; ++k) {
      const int r = warp + k * nwarps;
      const uint32_t *mrow = p.mask.bits + (int64_t)b * p.mask.sb + (int64_t)(row0 + r) * p.mask.sq;
      wv[k] = (r < rows && w < mW) ? (__ldg(mrow + w) & valid) : valid;
    }
  };
  uint32_t wv0[BM / 8];
  if (p.mask.bits) mask_words(0, wv0);

  // ---- Q load, segment range of the query tile ----------------------------
  // (the copies go out before anything waits on a global load)
  if (tid == 0) {
    // Q does not depend on the mask: start its load before classifying, and
    // key tile 0 with it (most masks keep it; checked after classifying)
    if (row0 < p.Lq && MGQA_DCHECK(h0 + NT <= p.Hq && b < p.B, p.err)) {
      mbar_arrive_expect_tx(bar_q, NT * KB * BOX);
      for (int t = 0; t < NT; ++t)
        for (int c = 0; c < KB; ++c)
          tc::tma_load_4d(smem + Lay::q_off + (t * KB + c) * BOX, &tm_q, c * 64, row0, h0 + t, b,
                          bar_q);
    }
    if (MGQA_DCHECK(g < p.Hkv, p.err)) {
      mbar_arrive_expect_tx(bar_kfull, KB * BOX);
      for (int c = 0; c < KB; ++c)
        tc::tma_load_4d(smem + Lay::k_off + c * BOX, &tm_k, c * 64, 0, g, b, bar_kfull);
      mbar_arrive_expect_tx(bar_vfull, KB * BOX);
      for (int c = 0; c < KB; ++c)
        tc::tma_load_4d(smem + Lay::v_off + c * BOX, &tm_v, c * 64, 0, g, b, bar_vfull);
    }
  }
  const int kvl = load_kv_len(p.mask.kv_len, b, p.Lk, p.err, qt == 0 && hp == 0 && tid == 0);
  const uint64_t lim = wait_limit();
  float *rope_invf = reinterpret_cast<float *>(smem + Lay::rope_off);
  float *rope_qw = rope_invf + D / 2;
  if (ROPE && (warp == 2 || warp == 3)) {
    // the rotation's tables, once per CTA (every query row reads them); every
    // load is issued before any store
    constexpr int NT3 = (D / 2 + D + 63) / 64;
    float v[NT3];
#pragma unroll
    for (int u = 0; u < NT3; ++u) {
      const int i = tid - 64 + 64 * u;
      v[u] = 0.f;
      if (i < D / 2) v[u] = i < p.rope.half ? __ldg(p.rope.inv_freq + i) : 0.f;
      else if (i < D / 2 + D && p.rope.q_norm) v[u] = __ldg(p.rope.q_norm + (i - D / 2));
    }
#pragma unroll
    for (int u = 0; u < NT3; ++u) {
      const int i = tid - 64 + 64 * u;
      if (i < D / 2 + D) rope_invf[i] = v[u];  // rope_qw follows rope_invf
    }
  }
  if (warp == 0) {
    if (p.mask.seg_q) {
      int mn = INT_MAX, mx = INT_MIN;
      for (int r = lane; r < rows; r += 32) {
        const int s = __ldg(p.mask.seg_q + (int64_t)b * p.Lq + row0 + r);
        mn = min(mn, s);
        mx = max(mx, s);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      if (lane == 0) {
        seg_slot[0] = mn;
        seg_slot[1] = mx;
      }
    }
  }
  __syncthreads();
  if (tid == 0) pre_stamp(9);

  // ---- packed-bit mask: per-tile "some key allowed" / "all keys allowed" ---
  // Each warp reads whole mask rows (32 consecutive words per load; the first
  // block was requested right after the grid-dependency wait), folds its rows
  // per word, reduces the 4 words of a tile across lanes and merges into the
  // CTA's bitsets.
  if (p.mask.bits) {
    const int W = mW;
    for (int wb = 0; wb < W; wb += 32) {
      const int w = wb + lane;
      const int lim = p.Lk - 32 * w;
      const uint32_t valid = w >= W ? 0u : (lim >= 32 ? 0xffffffffu : ((1u << lim) - 1u));
      uint32_t o = 0u, a = 0xffffffffu;
      uint32_t wv[BM / 8];
      if (wb == 0) {
#pragma unroll
        for (int k = 0; k < BM / 8; ++k) wv[k] = wv0[k];
      } else {
        mask_words(wb, wv);
      }
#pragma unroll
      for (int k = 0; k < BM / 8; ++k) {
        o |= (warp + k * nwarps < rows) ? wv[k] : 0u;
        a &= (wv[k] == valid && valid == 0xffffffffu) ? 0xffffffffu : 0u;
      }
      // a word slot past Lk (or a ragged last word) can never make a tile full
      if (w >= W || valid != 0xffffffffu) a = 0u;
      // 4 words per tile: lanes 4m..4m+3 -> tile (wb + 4m) / 4
      // (every lane runs every shuffle: no short-circuit around a sync op)
      uint32_t t_any = o != 0u ? 1u : 0u, t_all = a != 0u ? 1u : 0u;
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        const uint32_t o_any = __shfl_xor_sync(0xffffffffu, t_any, off);
        const uint32_t o_all = __shfl_xor_sync(0xffffffffu, t_all, off);
        t_any |= o_any;
        t_all &= o_all;
      }
      const int kt = w >> 2;
      if ((lane & 3) == 0 && w < W) {
        if (t_any) atomicOr(&any_bits[kt >> 5], 1u << (kt & 31));
        if (!t_all) atomicAnd(&all_bits[kt >> 5], ~(1u << (kt & 31)));
      }
    }
    __syncthreads();
  }
  if (tid == 0) pre_stamp(11);

  // ---- classify key tiles: non-empty (ne_bits), and of those full (no masking)
  for (int kt = warp; kt < p.nkt; kt += nwarps) {
    const int k0 = kt * BN;
    bool ne = k0 < p.Lk;
    bool full = k0 + BN <= p.Lk;
    if (p.mask.kv_len) {
      ne = ne && k0 < kvl;
      full = full && k0 + BN <= kvl;
    }
    if (p.mask.causal) {  // key j for query i when j <= i + coff
      ne = ne && k0 <= row0 + rows - 1 + p.mask.coff;
      full = full && k0 + BN - 1 <= row0 + p.mask.coff;
    }
    if (p.mask.bits && ne) {
      ne = (any_bits[kt >> 5] >> (kt & 31)) & 1u;  // ne was true here
      full = full && ((all_bits[kt >> 5] >> (kt & 31)) & 1u);
    }
    if (p.mask.seg_q && ne) {
      int mn = INT_MAX, mx = INT_MIN;
#pragma unroll
      for (int i = 0; i < BN / 32; ++i) {
        const int j = k0 + lane + 32 * i;
        if (j < p.Lk) {
          const int s = __ldg(p.mask.seg_k + (int64_t)b * p.Lk + j);
          mn = min(mn, s);
          mx = max(mx, s);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      const int qmn = seg_slot[0], qmx = seg_slot[1];
      if (qmx < 0 || mx < 0 || qmx < mn || mx < qmn) ne = false;
      full = full && qmn == qmx && mn == mx && qmn == mn && qmn >= 0;
    }
    if (lane == 0 && ne) {
      atomicOr(&ne_bits[kt >> 5], 1u << (kt & 31));
      if (full) atomicOr(&full_bits[kt >> 5], 1u << (kt & 31));
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0) pre_stamp(12);
  // every warp counts the non-empty tiles itself (no list, no second barrier);
  // the roles walk the bitsets in order (next_tile)
  int nk;
  {
    int cnt = 0;
    for (int w = lane; w < (p.nkt + 31) / 32; w += 32) cnt += __popc(ne_bits[w]);
    nk = __reduce_add_sync(0xffffffffu, cnt);
  }
  if (tid == 0) pre_stamp(2);
  // speculation missed when the first non-empty tile is not tile 0: stage 0
  // then holds a stale tile 0
  const uint32_t spec_miss = (nk == 0 || (ne_bits[0] & 1u) == 0u) ? 1u : 0u;
  const uint32_t tmem = *tmem_slot;
  const uint32_t sm_base = smem_u32(smem);
  bool ok = true;

  // Each role ends in role_end(): all threads meet on named barrier 1 (the
  // register split keeps the roles' code paths apart), then warp 1 frees the
  // tensor memory.
  auto role_end = [&]() {
    tc::fence_before_sync();
    named_sync(1, Lay::threads);
  };
  if (warp == 0) {
    if constexpr (NT == 2) tc::regs_dec<104>();
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      // non-empty tiles whose K (V) load has been issued; tile 0's went out
      // speculatively unless the speculation missed, in which case stage 0
      // was armed once more than the tiles say
      int k_issued = (nk > 0 && !spec_miss) ? 1 : 0, v_issued = k_issued;
      const int extra0 = (nk == 0 || spec_miss) ? 1 : 0;
      if (nk == 0 || spec_miss) {
        // every speculative load lands before its stage is reused or the CTA exits
        ok = mbar_wait(bar_q, 0, p.err, lim) && mbar_wait(bar_kfull, 0, p.err, lim) &&
             mbar_wait(bar_vfull, 0, p.err, lim);
        mbar_arrive(bar_spec);  // tells the MMA warp that stage 0 is at its phase 1
      }
      // debug library: an injected fault stops the loads at this tile (the
      // consumers' bounded waits then give up and report MGQA_ERR_TIMEOUT)
      const int stop_at = fault_tile();
      // (an L2 prefetch of the tiles ahead of their loads measured no faster)
      int kt = -1;  // the current non-empty tile
      for (int n = 0; n < nk && ok; ++n) {
        const int st = n % STAGES, use = n / STAGES;
        kt = next_tile(ne_bits, kt, p.nkt);
        if (n == 0 && !spec_miss) continue;  // tile 0 is already on its way
        if (n == stop_at) break;
        if (!MGQA_DCHECK(kt * BN < p.Lk && g < p.Hkv, p.err)) break;
        // K(n) reuses the stage K(n-STAGES) held; it is free once the S MMAs
        // that read it completed (V is released later, after P.V)
        if (n >= STAGES && !(ok = mbar_wait(bar_kempty + st, (use - 1) & 1, p.err, lim))) break;
        mbar_arrive_expect_tx(bar_kfull + st, KB * BOX);
        k_issued = n + 1;
        tr_stamp(n, 16);
        for (int c = 0; c < KB; ++c)
          tc::tma_load_4d(smem + Lay::k_off + (st * KB + c) * BOX, &tm_k, c * 64, kt * BN, g, b,
                          bar_kfull + st);
        if (n >= STAGES && !(ok = mbar_wait(bar_vempty + st, (use - 1) & 1, p.err, lim))) break;
        mbar_arrive_expect_tx(bar_vfull + st, KB * BOX);
        v_issued = n + 1;
        tr_stamp(n, 17);
        for (int c = 0; c < KB; ++c)
          tc::tma_load_4d(smem + Lay::v_off + (st * KB + c) * BOX, &tm_v, c * 64, kt * BN, g, b,
                          bar_vfull + st);
      }
      // No copy may still be in flight when the CTA exits. Only this thread
      // arms the full barriers, so the last armed phase of each is the newest
      // one it can reach and a parity wait on it is unambiguous. On the normal
      // path the MMA warp has already seen every one of them land.
      // times a stage's barrier was armed: entries n < issued with n % STAGES == st
      auto arms = [&](int issued, int st) {
        return (st == 0 ? extra0 : 0) + (issued > st ? (issued - 1 - st) / STAGES + 1 : 0);
      };
      mbar_wait(bar_q, 0, p.err, lim);
#pragma unroll
      for (int st = 0; st < STAGES; ++st) {
        const int ka = arms(k_issued, st), va = arms(v_issued, st);
        if (ka > 0) mbar_wait(bar_kfull + st, (ka - 1) & 1, p.err, lim);
        if (va > 0) mbar_wait(bar_vfull + st, (va - 1) & 1, p.err, lim);
      }
    }
    __syncwarp();
    role_end();
  } else if (warp == 1) {
    if constexpr (NT == 2) tc::regs_dec<104>();
    // ---------------- MMA issuer ----------------
    // Issue order: S_t(0) for every head, then per key tile n and head t:
    // O_t += P_t(n) V(n) followed at once by S_t(n+1) = Q_t K(n+1)^T. The
    // tensor pipe executes one thread's MMAs in issue order, so S_t(n+1)
    // overwrites P_t(n) only after the P.V MMA has consumed it; completion of
    // S_t(n+1) (s_full) therefore also implies O_t holds P.V up to tile n.
    // The whole warp runs the loop (waits, descriptor arithmetic) so every
    // operand is warp-uniform; one elected lane issues the MMAs and commits.
    if (nk > 0) {
      const bool leader = tc::elect_one();
      constexpr bool kBf16 = !__is_same(T, __half);
      constexpr uint32_t id_s = tc::idesc_16bit(BM, BN, 0, 0, kBf16);
      constexpr uint32_t id_pv = tc::idesc_16bit(BM, D, 0, 1, kBf16);
      // Each MMA costs one descriptor add: a descriptor's address field is
      // (shared address >> 4) and every buffer lies below 256 KB, so moving
      // within a buffer is adding (byte offset >> 4) to a base descriptor.
      const uint64_t qd0 = tc::sw128_desc(sm_base + Lay::q_off, 16, 1024);
      const uint64_t kd0 = tc::sw128_desc(sm_base + Lay::k_off, 16, 1024);
      const uint64_t vd0 = tc::sw128_desc(sm_base + Lay::v_off, BOX, 1024);
      constexpr uint64_t kTileStep = (uint64_t)(KB * BOX) >> 4;
      // every lane waits; the outcome is made warp-uniform
      auto wait = [&](uint64_t *bar, uint32_t parity) {
        const bool r = ok && mbar_wait(bar, parity, p.err, lim);
        ok = __all_sync(0xffffffffu, r);
        return ok;
      };
      // S_t = Q_t K(st)^T, k-steps [k0, k1); the commits follow the last one
      auto issue_s = [&](int t, int st, int k0, int k1) {
        const uint32_t d_s = tmem + t * BN;
        const uint64_t qd = qd0 + (uint64_t)t * kTileStep, kd = kd0 + (uint64_t)st * kTileStep;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            if (kk < k0 || kk >= k1) continue;
            const uint64_t off = (uint64_t)((kk / 4) * BOX + (kk % 4) * 32) >> 4;
            tc::mma_ss(d_s, qd + off, kd + off, id_s, kk > 0 ? 1u : 0u);
          }
          if (k1 == D / 16) {
            tc::mma_commit(bar_sfull + t);
            if (t == NT - 1) tc::mma_commit(bar_kempty + st);
          }
        }
        __syncwarp();
      };
      // O_t += P_t V(st), k-steps [k0, k1)
      auto issue_pv = [&](int t, int st, int k0, int k1, bool first) {
        const uint32_t d_o = tmem + NT * BN + t * D;
        const uint32_t a_p = tmem + t * BN;
        const uint64_t vd = vd0 + (uint64_t)st * kTileStep;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            if (kk < k0 || kk >= k1) continue;
            tc::mma_ts(d_o, a_p + kk * 8, vd + (uint64_t)(kk * 2048 >> 4), id_pv,
                       (!first || kk > 0) ? 1u : 0u);
          }
        }
        __syncwarp();
      };
      // After a missed speculation stage 0's first real fill is its phase 1.
      // A parity wait cannot tell phase 1 done from phase 0 pending, nor
      // (waiting late) phase 0 done from phase 2 pending, so the producer's
      // one-shot spec barrier, raised once it saw phase 0 land, is waited
      // for first; phase 2 needs this warp's first MMAs, so it cannot pass.
      auto par = [&](int st, int use) { return (uint32_t)(use + (st == 0 ? spec_miss : 0u)) & 1u; };
      if (spec_miss) wait(bar_spec, 0);
      wait(bar_q, 0) && wait(bar_kfull, par(0, 0)) && wait(bar_vfull, par(0, 0));
      tc::fence_after_sync();
      for (int t = 0; t < NT && ok; ++t) {
        // a fused rotary embedding rewrites the query tile first
        if (ROPE && !wait(bar_qrot + t, 0)) break;
        tc::fence_after_sync();
        if (leader) tr_stamp(0, 2 * t);
        issue_s(t, 0, 0, D / 16);
        if (leader) tr_stamp(0, 2 * t + 1);
      }
      if (lane == 0) pre_stamp(3);
      // The MMA queue is shallow: an issuing thread stalls in it until the
      // pipe has nearly drained, so any wait between two groups of MMAs
      // leaves the pipe idle. The waits for the next tile's K and V therefore
      // sit in the middle of a P.V group (its first half still queued), and
      // head 0's next P is probed in the middle of head 1's S group; only the
      // P waits that cannot be known early stay between groups; head 1's P is
      // likewise probed before the last MMA of head 0's S group.
      constexpr int kHalfPV = BN / 32, kLateS = D / 16 - 1;
      bool p0_seen = false;  // P_0(n) already observed complete
      for (int n = 0; n < nk && ok; ++n) {
        const int st = n % STAGES;
        const bool has_next = n + 1 < nk;
        const int st1 = (n + 1) % STAGES, use1 = (n + 1) / STAGES;
        bool p1_seen = false;  // P_1(n) already observed complete
        for (int t = 0; t < NT && ok; ++t) {
          if (!(t == 0 ? p0_seen : p1_seen) && !wait(bar_pfull + t, n & 1)) break;
          tc::fence_after_sync();
          if (leader) tr_stamp(n, 4 + 2 * t);
          issue_pv(t, st, 0, kHalfPV, n == 0);
          if (has_next) {  // K(n+1) before head 0's S(n+1), V(n+1) before the next P.V
            if (t == 0 && !wait(bar_kfull + st1, par(st1, use1))) break;
            if (t == NT - 1 && !wait(bar_vfull + st1, par(st1, use1))) break;
            tc::fence_after_sync();
          }
          issue_pv(t, st, kHalfPV, BN / 16, n == 0);
          if (leader) {
            if (n == nk - 1 && t == NT - 1) pre_stamp(8);
            if (n == nk - 1) tc::mma_commit(bar_odone + t);  // read by the epilogue only
            if (t == NT - 1) tc::mma_commit(bar_vempty + st);
            tr_stamp(n, 5 + 2 * t);
          }
          __syncwarp();
          if (has_next) {
            if (leader) tr_stamp(n + 1, 2 * t);
            if (NT > 1 && t == NT - 1) {
              issue_s(t, st1, 0, kLateS);
              // a probe, not a wait: P_0(n+1) needs the softmax of head 0,
              // which may still be running
              p0_seen = __all_sync(0xffffffffu, mbar_test_wait(bar_pfull, (n + 1) & 1));
              issue_s(t, st1, kLateS, D / 16);
            } else if (NT > 1) {
              issue_s(t, st1, 0, kLateS);
              p1_seen = __all_sync(0xffffffffu, mbar_test_wait(bar_pfull + 1, n & 1));
              issue_s(t, st1, kLateS, D / 16);
            } else {
              issue_s(t, st1, 0, D / 16);
            }
            if (leader) tr_stamp(n + 1, 2 * t + 1);
          }
        }
      }
      // drain: the last release of every stage has landed before the CTA exits
      for (int s = 0; s < STAGES && s < nk && ok; ++s) {
        const int last_use = (nk - 1 - s) / STAGES;
        wait(bar_kempty + s, last_use & 1) && wait(bar_vempty + s, last_use & 1);
      }
      if (!ok) {
        // a wait gave up: every MMA already issued completes before the tensor
        // memory is freed (the commit arrives once they all have)
        if (leader) tc::mma_commit(bar_drain);
        __syncwarp();
        mbar_wait(bar_drain, 0, p.err, lim);
      }
    }
    __syncwarp();
    role_end();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, Lay::tmem_cols);
  } else if (warp < 4) {
    if constexpr (NT == 2) tc::regs_dec<104>();
    role_end();
  } else {
    if constexpr (NT == 2) tc::regs_inc<200>();
    // ---------------- softmax warpgroup t ----------------
    const int t = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row within the tile
    const int i = row0 + r;
    const bool row_ok = r < rows;
    const int ic = row_ok ? i : row0;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_base + t * BN;
    const uint32_t t_o = tmem + lane_base + NT * BN + t * D;
    const int segq = p.mask.seg_q ? __ldg(p.mask.seg_q + (int64_t)b * p.Lq + ic) : 0;
    if constexpr (ROPE) {
      // rotary embedding (and RMS norm) of this head's query row, in shared
      // memory, before the head's first product
      if (ok) ok = mbar_wait(bar_q, 0, p.err, lim);
      if (ok && row_ok && h0 + t < p.rope.q_heads) {
        const int pos = p.rope.positions ? __ldg(p.rope.positions + (int64_t)b * p.Lq + i) : i;
        rope_q_row<T, D>(smem + Lay::q_off + t * KB * BOX, r, pos, p.rope, rope_invf, rope_qw);
      }
      fence_proxy_async_smem();  // the tensor core reads the tile through the async proxy
      mbar_arrive(bar_qrot + t);
    }
    const bool neg = p.scale_log2 < 0.f;
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    const int tr = (lane == 0) ? ((8 + 4 * t) | (quarter << 8)) : -1;  // debug trace events
    int kt = -1;  // the current non-empty tile
    for (int n = 0; n < nk; ++n) {
      kt = next_tile(ne_bits, kt, p.nkt);
      const bool partial = !((full_bits[kt >> 5] >> (kt & 31)) & 1u);
      uint32_t mw[BN / 32] = {0u, 0u, 0u, 0u};
      if (partial) tile_mask_words(p, b, ic, row_ok, kt * BN, kvl, segq, lane, mw);
      // warp-uniform outcome: the tile pass below is made of warp-wide
      // tensor-memory loads and stores
      if (ok) ok = mbar_wait(bar_sfull + t, n & 1, p.err, lim);
      ok = __all_sync(0xffffffffu, ok);
      if (n == 0 && t == 0 && tid == 128) pre_stamp(10);
      if (tr >= 0 && quarter == 0) tr_stamp(n, 8 + 4 * t);
      if (ok) {  // after a failed wait, tensor memory is left alone
        tc::fence_after_sync();
        if (neg) {
          if (partial) softmax_tile<T, D, true, true>(t_s, t_o, mw, sl2, m_used, l, n, tr);
          else softmax_tile<T, D, true, false>(t_s, t_o, mw, sl2, m_used, l, n, tr);
        } else {
          if (partial) softmax_tile<T, D, false, true>(t_s, t_o, mw, sl2, m_used, l, n, tr);
          else softmax_tile<T, D, false, false>(t_s, t_o, mw, sl2, m_used, l, n, tr);
        }
        if (lane == 0) dbg_count(1);  // debug library: tiles processed (per warp)
        tc::fence_before_sync();
      }
      mbar_arrive(bar_pfull + t);
      if (tr >= 0) tr_stamp_max(n, 11 + 4 * t);
      if (n == 0 && t == 0 && tid == 128) pre_stamp(4);
    }
    // epilogue: O / l -> bf16, staged in this head's Q buffer (free once its
    // last S MMA completed) in the 128-byte-swizzled box layout, then written
    // by TMA tensor stores (rows past Lq are clipped by the store)
    float o_scale = 0.f;
    if (nk > 0) {
      if (ok) ok = mbar_wait(bar_odone + t, 0, p.err, lim);  // committed once, after the last P.V
      ok = __all_sync(0xffffffffu, ok);
      tc::fence_after_sync();
      o_scale = (l > 0.f) ? 1.f / l : 0.f;
      if (t == 0 && tid == 128) pre_stamp(5);
    } else if (ok) {
      ok = mbar_wait(bar_q, 0, p.err, lim);  // the Q load must land before the buffer is reused
    }
    ok = __all_sync(0xffffffffu, ok);
    uint32_t orow[D];
    if (nk > 0 && ok) {  // after a failed wait the output rows are written as zeros
#pragma unroll
      for (int c = 0; c < D / 32; ++c)
        tc::tmem_ld32(t_o + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&orow[c * 32]));
      tc::tmem_wait_ld();
    } else {
#pragma unroll
      for (int j = 0; j < D; ++j) orow[j] = 0u;
    }
    unsigned char *ob = smem + Lay::q_off + t * KB * BOX;
#pragma unroll
    for (int cc = 0; cc < D / 8; ++cc) {  // 16-byte chunks of the row
      uint32_t w4[4];
#pragma unroll
      for (int h = 0; h < 4; ++h)
        w4[h] = pack2<T>(__uint_as_float(orow[cc * 8 + 2 * h]) * o_scale,
                         __uint_as_float(orow[cc * 8 + 2 * h + 1]) * o_scale);
      const int box = cc >> 3, ch = cc & 7;
      *reinterpret_cast<uint4 *>(ob + box * BOX + r * 128 + ((ch ^ (r & 7)) << 4)) =
          make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    fence_proxy_async_smem();
    named_sync(2 + t, 128);
    if (warp == 4 + 4 * t && lane == 0 && MGQA_DCHECK(row0 < p.Lq && h0 + t < p.Hq, p.err)) {
      for (int c = 0; c < KB; ++c) tc::tma_store_4d(&tm_o, ob + c * BOX, c * 64, row0, h0 + t, b);
      tc::tma_store_commit_and_wait_read();
      if (t == 0) pre_stamp(6);
    }
    if (row_ok && p.lse)
      p.lse[((int64_t)b * p.Hq + h0 + t) * p.Lq + i] =
          (l > 0.f) ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
    if (t == 0 && tid == 128) pre_stamp(7);
    role_end();
  }
}

// ---- host side ----------------------------------------------------------------

}  // namespace

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static std::atomic<EncodeTiledFn> fn{nullptr};
  EncodeTiledFn f = fn.load(std::memory_order_acquire);
  if (!f) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<EncodeTiledFn>(ptr);
      fn.store(f, std::memory_order_release);
    }
  }
  return f;
}

bool make_tma_map_4d(CUtensorMap *m, mgqa_dtype dt, const void *base, int B, int H, int L, int D,
                     const int64_t *st, int box_x, int box_y, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const size_t es = dt == MGQA_FP32 ? 4 : 2;
  const CUtensorMapDataType t = dt == MGQA_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                : dt == MGQA_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)H, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)st[2] * es, (cuuint64_t)st[1] * es,
                                 (cuuint64_t)st[0] * es};
  const cuuint32_t box[4] = {(cuuint32_t)box_x, (cuuint32_t)box_y, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, t, 4, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// Streaming multiprocessors of the current device (0 if unknown), looked up
// once per device.
int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 0;
  cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <typename T, int D, int NT, int STAGES, bool ROPE>
mgqa_status launch_t(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                     const CUtensorMap &mo, const TcParams &p, cudaStream_t s) {
  using Lay = Layout<D, NT, STAGES>;
  auto kern = prefill_tc_kernel<T, D, NT, STAGES, ROPE>;
  static std::atomic<uint64_t> attr_done{0};
  const mgqa_status st = ensure_smem_attr(kern, Lay::smem_bytes, attr_done, "tensor-core prefill");
  if (st != MGQA_OK) return st;
  dim3 grid((p.Lq + BM - 1) / BM, p.Hq / NT, p.B);
  const cudaError_t e = launch_pdl(kern, grid, dim3(Lay::threads), Lay::smem_bytes, s, mq, mk, mv,
                                   mo, p);
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
  return MGQA_OK;
}

template <typename T, bool ROPE>
mgqa_status dispatch_d(int D, bool pair, const CUtensorMap &mq, const CUtensorMap &mk,
                       const CUtensorMap &mv, const CUtensorMap &mo, const TcParams &p,
                       cudaStream_t s) {
  if (D == 128)
    return pair ? launch_t<T, 128, 2, 2, ROPE>(mq, mk, mv, mo, p, s)
                : launch_t<T, 128, 1, 2, ROPE>(mq, mk, mv, mo, p, s);
  if (D == 64)
    return pair ? launch_t<T, 64, 2, 3, ROPE>(mq, mk, mv, mo, p, s)
                : launch_t<T, 64, 1, 3, ROPE>(mq, mk, mv, mo, p, s);
  return fail(MGQA_ERR_UNSUPPORTED, "head dim %d", D);
}

}  // namespace

mgqa_status launch_prefill_tc(const mgqa_args &a, cudaStream_t s, const FusedRope &rope) {
  if (a.dtype != MGQA_BF16 && a.dtype != MGQA_FP16)
    return fail(MGQA_ERR_UNSUPPORTED, "tensor-core prefill takes bf16 or fp16");
  const int nkt = (a.Lk + BN - 1) / BN;
  if (nkt > MAXKT) return fail(MGQA_ERR_UNSUPPORTED, "Lk > %d", MAXKT * BN);
  // 16-bit [B][H][L][D] views, boxes of 64 columns x 128 rows, 128-byte swizzle
  CUtensorMap mq, mk, mv, mo;
  if (!make_tma_map_4d(&mq, a.dtype, a.q, a.B, a.Hq, a.Lq, a.D, a.q_stride, 64, BM, true) ||
      !make_tma_map_4d(&mk, a.dtype, a.k, a.B, a.Hkv, a.Lk, a.D, a.k_stride, 64, BN, true) ||
      !make_tma_map_4d(&mv, a.dtype, a.v, a.B, a.Hkv, a.Lk, a.D, a.v_stride, 64, BN, true) ||
      !make_tma_map_4d(&mo, a.dtype, a.out, a.B, a.Hq, a.Lq, a.D, a.o_stride, 64, BM, true))
    return fail(MGQA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  TcParams p{};
  p.mask = MaskView{a.mask_bits, a.mask_stride_b, a.mask_stride_q, a.kv_len, a.seg_q, a.seg_k,
                    a.causal != 0, a.Lk - a.Lq};
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv; p.Lq = a.Lq; p.Lk = a.Lk;
  p.n_rep = a.Hq / a.Hkv; p.nkt = nkt;
  p.scale_log2 = a.scale * kLog2e;
  p.out = a.out;
  p.os[0] = a.o_stride[0]; p.os[1] = a.o_stride[1]; p.os[2] = a.o_stride[2];
  p.q = a.q; p.k = a.k; p.v = a.v;
  {
    const int sms = sm_count();
    const int64_t ctas = (int64_t)((a.Lq + BM - 1) / BM) * (a.Hq / ((a.Hq / a.Hkv) % 2 == 0 ? 2 : 1)) * a.B;
    p.warm = sms > 0 && ctas <= sms;
  }
  for (int t = 0; t < 3; ++t) {
    p.qs[t] = a.q_stride[t];
    p.ks[t] = a.k_stride[t];
    p.vs[t] = a.v_stride[t];
  }
  p.lse = a.lse; p.err = a.dev_error;
  p.rope = rope;
  const bool pair = (p.n_rep % 2) == 0;
  const bool rope_on = rope.inv_freq != nullptr;
  if (a.dtype == MGQA_BF16)
    return rope_on ? dispatch_d<__nv_bfloat16, true>(a.D, pair, mq, mk, mv, mo, p, s)
                   : dispatch_d<__nv_bfloat16, false>(a.D, pair, mq, mk, mv, mo, p, s);
  return rope_on ? dispatch_d<__half, true>(a.D, pair, mq, mk, mv, mo, p, s)
                 : dispatch_d<__half, false>(a.D, pair, mq, mk, mv, mo, p, s);
}

}  // namespace mgqa

// ---- debug library entry points (include/masked_gqa_attn_debug.h) -----------
#ifdef MGQA_DEBUG
#include "../../include/masked_gqa_attn_debug.h"

extern "C" MGQA_API mgqa_status mgqa_debug_counters(uint64_t *out, int32_t n) {
  using namespace mgqa;
  clear_error_detail();
  if (!out || n < 0 || n > MGQA_DEBUG_NUM_COUNTERS)
    return fail(MGQA_ERR_INVALID_ARG, "mgqa_debug_counters: bad output or count");
  DebugState st;
  const cudaError_t e = cudaMemcpyFromSymbol(&st, g_dbg, sizeof(st));
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "reading the debug state: %s", cudaGetErrorString(e));
  for (int i = 0; i < n; ++i) out[i] = st.counters[i];
  return MGQA_OK;
}

extern "C" MGQA_API mgqa_status mgqa_debug_prefill_timeline(uint64_t *out, int32_t n_ctas) {
  using namespace mgqa;
  clear_error_detail();
  if (!out || n_ctas < 0 || n_ctas > kPreTlCtas)
    return fail(MGQA_ERR_INVALID_ARG, "mgqa_debug_prefill_timeline: bad output or count");
  cudaError_t e = cudaMemcpyFromSymbol(out, g_pre_tl, (size_t)n_ctas * kPreTlStamps * sizeof(uint64_t));
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "reading the timeline: %s", cudaGetErrorString(e));
  static const unsigned long long zeros[kPreTlCtas][kPreTlStamps] = {};
  e = cudaMemcpyToSymbol(g_pre_tl, zeros, sizeof(zeros));
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "clearing the timeline: %s", cudaGetErrorString(e));
  return MGQA_OK;
}

extern "C" MGQA_API mgqa_status mgqa_debug_prefill_trace(uint64_t *out, int32_t n_ctas) {
  using namespace mgqa;
  clear_error_detail();
  if (!out || n_ctas < 0 || n_ctas > kTrCtas)
    return fail(MGQA_ERR_INVALID_ARG, "mgqa_debug_prefill_trace: bad output or count");
  const size_t per_cta = (size_t)kTrTiles * kTrEvents * sizeof(uint64_t);
  cudaError_t e = cudaMemcpyFromSymbol(out, g_pre_tr, (size_t)n_ctas * per_cta);
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "reading the trace: %s", cudaGetErrorString(e));
  static const unsigned long long zeros[kTrCtas][kTrTiles][kTrEvents] = {};
  e = cudaMemcpyToSymbol(g_pre_tr, zeros, sizeof(zeros));
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "clearing the trace: %s", cudaGetErrorString(e));
  return MGQA_OK;
}

extern "C" MGQA_API mgqa_status mgqa_debug_reset(void) {
  using namespace mgqa;
  clear_error_detail();
  const DebugState st = {{0ull, 0ull, 0ull, 0ull}, -1, kWaitLimitNs};
  const cudaError_t e = cudaMemcpyToSymbol(g_dbg, &st, sizeof(st));
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "writing the debug state: %s", cudaGetErrorString(e));
  return MGQA_OK;
}

extern "C" MGQA_API mgqa_status mgqa_debug_inject_prefill_stall(int32_t tile, uint64_t wait_limit_ns) {
  using namespace mgqa;
  clear_error_detail();
  if (tile == 0 || (tile > 0 && wait_limit_ns == 0))
    return fail(MGQA_ERR_INVALID_ARG, "stall tile must be >= 1 (or < 0 to clear) with a wait limit > 0");
  DebugState st;
  cudaError_t e = cudaMemcpyFromSymbol(&st, g_dbg, sizeof(st));
  if (e == cudaSuccess) {
    st.fault_tile = tile < 0 ? -1 : tile;
    st.wait_limit_ns = tile < 0 ? kWaitLimitNs : wait_limit_ns;
    e = cudaMemcpyToSymbol(g_dbg, &st, sizeof(st));
  }
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "writing the debug state: %s", cudaGetErrorString(e));
  return MGQA_OK;
}
#endif  // MGQA_DEBUG
