/*
 * masked_gqa_attn.h -- C ABI of the GB300 (sm_103a) masked grouped-query
 * attention library.
 *
 * The attention operation (the prefill and decode entry points): scaled-
 * dot-product attention with grouped KV heads under an explicit boolean mask,
 * as the engine pages use it (the rotary embedding and the packing helpers
 * further down are the steps around it):
 *   - VoxCPM page, "Upstream-identical practice", attention bullet: SDPA with
 *     enable_gqa on contiguous tensors; bidirectional in the local DiT; cache
 *     decode under an explicit boolean mask where slots past the current length
 *     are masked and contribute exact zeros;
 *   - OmniVoice page, "Upstream-identical practice", attention-mask bullet: a
 *     full 4D boolean mask, not causal, with the KV heads repeated to the query
 *     heads; the conditional and unconditional rows run as one batch;
 *   - OmniVoice page, "Memory & speed", packed_guidance paragraph: both
 *     sequences side by side in one row under a block-diagonal mask;
 *   - VoxCPM page, "Memory & speed", attention_span paragraph: attend only to
 *     the filled blocks of the 8192-slot static cache.
 *
 * For batch b, query head h, query row i, with KV head g = h / (Hq / Hkv):
 *   s_j   = scale * <q[b,h,i,:], k[b,g,j,:]>   where allowed(b,i,j), else -inf
 *   out   = sum_j softmax(s)_j * v[b,g,j,:]
 *   lse   = log(sum_j exp(s_j))                 (natural log, optional output)
 * A query row with no allowed key gets out = 0 and lse = -inf.
 *
 * allowed(b,i,j) is the AND of every mask form that is given (non-NULL):
 *   mask_bits : bit (j % 32) of word mask_bits[b*mask_stride_b + i*mask_stride_q
 *               + j/32] is 1 (least-significant bit first, 1 = may attend);
 *               the same mask applies to every head;
 *   kv_len    : j < kv_len[b]  (a per-row key length; for decode, the filled
 *               length of the static cache);
 *   seg_q/seg_k: seg_q[b*Lq + i] == seg_k[b*Lk + j] and that id is >= 0
 *               (block-diagonal packing; negative ids attend nowhere);
 *   causal    : j <= i + (Lk - Lq) when nonzero (the query rows are the last
 *               Lq of the Lk positions; for Lq == Lk the lower triangle) --
 *               VoxCPM page, "Upstream-identical practice": causal prefill.
 * With no mask form given every key is allowed (dense bidirectional).
 *
 * Ownership: every pointer is device memory owned by the caller. The library
 * allocates nothing, never synchronises, and enqueues its work on `stream`
 * only. Errors found on the host return at once and enqueue nothing; errors
 * found on the device are written to *dev_error (when given) as the first
 * mgqa_status code seen, and the affected outputs are still written.
 */
#ifndef MASKED_GQA_ATTN_H
#define MASKED_GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MGQA_ABI_VERSION 6

#if defined(__GNUC__)
#define MGQA_API __attribute__((visibility("default")))
#else
#define MGQA_API
#endif

typedef enum {
  MGQA_OK = 0,
  MGQA_ERR_INVALID_ARG = 1,  /* bad pointer, shape, stride, alignment or scale;
                                on the device: kv_len < 0 or kv_len > Lk */
  MGQA_ERR_UNSUPPORTED = 2,  /* valid request the library has no kernel for */
  MGQA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  MGQA_ERR_TIMEOUT = 4,      /* device: a bounded pipeline wait gave up */
  MGQA_ERR_DEVICE_CHECK = 5  /* device, debug library only: a bounds or alignment
                                check failed and the access was skipped */
} mgqa_status;

typedef enum {
  MGQA_BF16 = 0,  /* q/k/v/out bf16, fp32 accumulation (tensor cores) */
  MGQA_FP32 = 1,  /* q/k/v/out fp32, fp32 arithmetic throughout */
  MGQA_FP16 = 2   /* q/k/v/out fp16, fp32 accumulation (tensor cores) */
} mgqa_dtype;

typedef struct mgqa_args {
  mgqa_dtype dtype;
  int32_t B;    /* batch rows */
  int32_t Hq;   /* query heads */
  int32_t Hkv;  /* KV heads; Hq % Hkv == 0 */
  int32_t Lq;   /* query positions (decode: must be 1) */
  int32_t Lk;   /* key positions (decode: static-cache capacity, <= 32768) */
  int32_t D;    /* head dim: 64 or 128 */

  /* q [B][Hq][Lq][D], k and v [B][Hkv][Lk][D], out [B][Hq][Lq][D]. The head-dim
   * stride is 1; the three strides are (batch, head, position) in ELEMENTS.
   * Every base pointer must be 16-byte aligned and every stride a multiple of
   * 16 bytes (8 elements for bf16, 4 for fp32). */
  const void *q, *k, *v;
  void *out;
  int64_t q_stride[3], k_stride[3], v_stride[3], o_stride[3];

  /* optional mask forms, combined with AND (see above) */
  const uint32_t *mask_bits;    /* words; row (b, i) starts at b*stride_b + i*stride_q */
  int64_t mask_stride_b;        /* in 32-bit words: 0 (one mask for every batch row) or
                                   >= ceil(Lk/32) */
  int64_t mask_stride_q;        /* in 32-bit words: 0 (one row for every query: a key-
                                   padding mask stored as [B][1][W]) or >= ceil(Lk/32) */
  const int32_t *kv_len;        /* [B]; values outside [0, Lk] are a device error
                                   (clamped; the static cache is full) */
  const int32_t *seg_q;         /* [B][Lq] contiguous; given together with seg_k */
  const int32_t *seg_k;         /* [B][Lk] contiguous */

  float scale;                  /* finite softmax scale; SDPA's default is 1/sqrt(D) */
  float *lse;                   /* optional out: [B][Hq][Lq] contiguous, natural log */
  int32_t *dev_error;           /* optional: first device-side mgqa_status code */
  int32_t causal;               /* nonzero: add the causal form to the mask */
} mgqa_args;

/* Full-sequence (prefill) attention: bidirectional unless `causal` is set,
 * any of the mask forms. bf16 and fp16 run on the tensor cores (TMA-fed
 * tcgen05 MMAs accumulating in tensor memory) and skip every 128x128 (query,
 * key) tile the mask leaves empty; fp32 runs on the CUDA cores. Lq, Lk >= 1.
 * Returns MGQA_OK once the kernel is enqueued. */
MGQA_API mgqa_status masked_gqa_attn_prefill(const mgqa_args *args, cudaStream_t stream);

/* Nominal workspace size for these decode arguments: 16 for supported
 * arguments, 0 when they are invalid (a validity check). The decode kernel
 * merges its splits on chip and never reads or writes a workspace; the
 * workspace parameters below are kept so that callers written against earlier
 * versions keep working. */
MGQA_API size_t masked_gqa_attn_decode_workspace_size(const mgqa_args *args);

/* One-query (Lq == 1) attention over a static KV cache of Lk slots. The
 * cache is cut into 64-slot chunks of absolute positions, dealt round-robin
 * to the 16 CTAs of one thread-block cluster per (request, KV-head group);
 * masked slots are never read. The CTAs' partial results are exchanged
 * through the cluster's shared memory and merged in a fixed order inside the
 * same launch, so the full-cache (mask_bits) and filled-span (kv_len) forms of
 * one mask give bit-identical outputs. The launch needs 16-CTA clusters (a
 * non-portable size, available on this library's sm_103a target); a GPU
 * partition too small to hold one returns MGQA_ERR_CUDA.
 * `workspace` / `workspace_bytes` are ignored (may be NULL / 0). Calls on
 * different streams are independent: no state is shared between calls.
 * `stream` belongs to the current device. */
MGQA_API mgqa_status masked_gqa_attn_decode(const mgqa_args *args, void *workspace,
                                            size_t workspace_bytes, cudaStream_t stream);

/* One decode step fused with its cache append (VoxCPM page, "Memory & speed":
 * each patch advances the language model by one position against its static
 * cache, inside one CUDA graph per patch; when the cache is full, the step
 * errors where upstream errors). For each request b this writes the step's
 * key/value rows k_new[b][g][:], v_new[b][g][:] (element strides
 * k_new_stride = {batch, head}, same for v_new; head dim contiguous, 16-byte
 * aligned) into cache slot kv_len[b] of args->k / args->v, then attends the
 * query over slots 0 .. kv_len[b] (the new one included), and writes
 * kv_len[b] + 1 to kv_len_out[b] when kv_len_out is given (it must not alias
 * kv_len, so a captured graph can ping-pong two length buffers). args->kv_len
 * is required; packed bits and segment ids are not accepted here. A request
 * whose cache is already full (kv_len[b] == Lk) appends nothing, attends over
 * the whole cache, and sets *dev_error to MGQA_ERR_INVALID_ARG. The workspace
 * parameters are ignored, as for masked_gqa_attn_decode. */
MGQA_API mgqa_status masked_gqa_attn_decode_append(const mgqa_args *args, const void *k_new,
                                                   const void *v_new, const int64_t *k_new_stride,
                                                   const int64_t *v_new_stride,
                                                   int32_t *kv_len_out, void *workspace,
                                                   size_t workspace_bytes, cudaStream_t stream);

/* Packed-guidance helpers (OmniVoice page, "Memory & speed", packed_guidance:
 * the conditional sequence and the target part of the unconditional one side
 * by side in one row under a block-diagonal mask, positions of each starting
 * at 0). pack: packed[:, :, 0:La] = a, packed[:, :, La:La+Lb] = b for every
 * batch row and head, and, when seg is given, seg[b][0:La] = 0 and
 * seg[b][La:La+Lb] = 1 (int32 [B][La+Lb], usable as seg_q and seg_k of the
 * packed call). unpack: the inverse split of a packed output. Views are
 * [B][H][L][D] with element strides (batch, head, position), head dim
 * contiguous, 16-byte aligned; D * element size a multiple of 16 bytes.
 * Positional encodings are the caller's (applied per sequence before packing). */
MGQA_API mgqa_status masked_gqa_pack_pair(mgqa_dtype dtype, int32_t B, int32_t H, int32_t D,
                                          const void *a, const int64_t *a_stride, int32_t La,
                                          const void *b, const int64_t *b_stride, int32_t Lb,
                                          void *packed, const int64_t *packed_stride,
                                          int32_t *seg, cudaStream_t stream);
MGQA_API mgqa_status masked_gqa_unpack_pair(mgqa_dtype dtype, int32_t B, int32_t H, int32_t D,
                                            const void *packed, const int64_t *packed_stride,
                                            void *a, const int64_t *a_stride, int32_t La,
                                            void *b, const int64_t *b_stride, int32_t Lb,
                                            cudaStream_t stream);

/* masked_gqa_attn_decode without a workspace argument. No passage of the
 * engine pages has a counterpart: this entry point exists for callers that
 * cannot allocate device memory for the library, such as code running inside
 * a host framework that owns every device buffer and hands an extension only
 * its inputs and outputs, or a latency-critical per-token loop that must not
 * call the allocator. The caller passes q/k/v, out and the mask forms; the
 * kernel's scratch is on-chip shared memory of its own launch, so nothing is
 * allocated or freed (no cudaMalloc, cudaFree or allocating library routine
 * is called), nothing persists between calls and calls on different streams
 * do not interfere. `stream` must belong to the current device. */
MGQA_API mgqa_status masked_gqa_attn_decode_static(const mgqa_args *args, cudaStream_t stream);

/* Rotary position embedding, in place, on q or k before attention (the
 * attention passages above take q and k already rotated):
 *   - F5-TTS page, module table and "Upstream-identical practice": the DiT
 *     rotates interleaved feature pairs (x-transformers), on its first
 *     pe_attn_head heads only -> `interleaved`, `heads`;
 *   - OmniVoice page, "Parity results": the inverse-frequency table stays fp32; VoxCPM page,
 *     "Upstream-identical practice", precision bullet: the LongRoPE table is
 *     built in fp32 -> `inv_freq` is a caller-built fp32 table (plain, scaled
 *     or LongRoPE-rescaled frequencies alike);
 *   - OmniVoice page, "Memory & speed", packed_guidance paragraph: under
 *     packing each sequence's positions start at 0 -> `positions`.
 * For b < B, h < heads, l < L, pair i < rot_dim/2:
 *   theta = fl32((float)positions[b][l] * inv_freq[i])      (one fp32 product)
 *   (e0, e1) = (2i, 2i+1) if interleaved, else (i, i + rot_dim/2)
 *   x[e0], x[e1] <- x[e0] cos(theta) - x[e1] sin(theta),
 *                   x[e0] sin(theta) + x[e1] cos(theta)     (fp32, rounded to dtype)
 * Features >= rot_dim and heads >= `heads` are left as they are.
 * With norm_weight (OmniVoice page, "Parity results": the Qwen decoder
 * normalises q and k separately, as transformers does, before the rotation),
 * each rotated head vector is first RMS-normalised over all D features:
 *   x[d] <- x[d] / sqrt(mean_d(x^2) + norm_eps) * norm_weight[d]   (fp32)
 * and the rotation then acts on the normalised values (features >= rot_dim
 * keep their normalised value); one rounding to dtype at the end. */
typedef struct {
  mgqa_dtype dtype;             /* MGQA_BF16, MGQA_FP16 or MGQA_FP32 */
  int32_t B, H, L, D;           /* x is [B][H][L][D] */
  void *x;                      /* device, rotated in place, element-aligned */
  int64_t x_stride[3];          /* batch, head, position strides in elements; head dim contiguous */
  const int32_t *positions;     /* device [B][L] contiguous, or NULL for positions[b][l] = l */
  const float *inv_freq;        /* device [rot_dim / 2] fp32 angular frequencies */
  int32_t rot_dim;              /* even, 2 <= rot_dim <= D */
  int32_t heads;                /* 1 <= heads <= H */
  int32_t interleaved;          /* nonzero: pairs (2i, 2i+1); zero: pairs (i, i + rot_dim/2) */
  const float *norm_weight;     /* optional device [D] fp32: RMS-normalise each rotated head
                                   vector over its D features first (see below); D <= 256 */
  float norm_eps;               /* with norm_weight: finite, >= 0 */
} mgqa_rope_args;

/* Host-detectable argument errors return MGQA_ERR_INVALID_ARG (detail in
 * mgqa_last_error_detail); a failed launch returns MGQA_ERR_CUDA. Allocates
 * nothing, never synchronises; MGQA_OK once the kernel is enqueued. All
 * pointers are caller-owned device memory. */
MGQA_API mgqa_status masked_gqa_rope(const mgqa_rope_args *args, cudaStream_t stream);

/* q and k of one layer rotated by one launch: the same results, bit for bit,
 * as masked_gqa_rope(q) followed by masked_gqa_rope(k). Each tensor has its
 * own arguments (shape, strides, heads, norm weight, positions, table); both
 * must have the same dtype. When the two take different kernels (for
 * instance one with a norm weight and one without, or one with 16-byte rows
 * and one without), or their elements overlap, the call makes one launch
 * each, in that order. Errors as masked_gqa_rope (the detail names q or k);
 * nothing is enqueued when either tensor's arguments are rejected. */
MGQA_API mgqa_status masked_gqa_rope_pair(const mgqa_rope_args *q, const mgqa_rope_args *k,
                                          cudaStream_t stream);

/* The rotary embedding (and optional RMS normalisation) applied INSIDE an
 * attention call, to the query rows as they are loaded and, for the fused
 * decode step, to the appended key row -- the same arithmetic as
 * masked_gqa_rope (same bits), without its extra pass over q and k. */
typedef struct {
  const float *inv_freq;        /* device [rot_dim / 2] fp32 angular frequencies */
  const int32_t *positions;     /* optional device int32 -- prefill: [B][Lq], the query rows'
                                   positions (NULL: the query index i); decode step: [B], the
                                   new token's position (NULL: kv_len[b], its cache slot) */
  int32_t rot_dim;              /* even, 2 <= rot_dim <= D */
  int32_t interleaved;          /* nonzero: pairs (2i, 2i+1); zero: pairs (i, i + rot_dim/2) */
  int32_t q_heads;              /* query heads h < q_heads are normalised / rotated (1..Hq) */
  int32_t k_heads;              /* decode step: the appended key row of KV heads g < k_heads
                                   is normalised / rotated (0..Hkv); ignored by the prefill */
  const float *q_norm_weight;   /* optional device [D] fp32: RMS-normalise those q rows first */
  const float *k_norm_weight;   /* optional device [D] fp32: the same for the appended k row */
  float norm_eps;               /* with a norm weight: finite, >= 0 */
} mgqa_qk_rope;

/* masked_gqa_attn_prefill with `rope` applied to the query rows inside the
 * kernel (each CTA transforms its query tile in shared memory once, before
 * its first product). The keys must already be rotated (and normalised), e.g.
 * by masked_gqa_rope with the same table: the result equals masked_gqa_rope
 * on q and then masked_gqa_attn_prefill, bit for bit. bf16 and fp16 only, and
 * half-split rotations over D, D/2 or D/4 features (interleaved ones of any
 * width); MGQA_ERR_UNSUPPORTED otherwise (rotate with masked_gqa_rope). */
MGQA_API mgqa_status masked_gqa_attn_prefill_rope(const mgqa_args *args, const mgqa_qk_rope *rope,
                                                  cudaStream_t stream);

/* masked_gqa_attn_decode_append with `rope` applied inside the kernel to the
 * step's query and to its new key row before that row is attended to and
 * written into the cache (the cache keeps rotated keys), at the new token's
 * position (rope->positions[b], or kv_len[b]). Equals masked_gqa_rope on q
 * and on k_new and then masked_gqa_attn_decode_append, bit for bit. */
MGQA_API mgqa_status masked_gqa_attn_decode_append_rope(
    const mgqa_args *args, const void *k_new, const void *v_new, const int64_t *k_new_stride,
    const int64_t *v_new_stride, int32_t *kv_len_out, const mgqa_qk_rope *rope, void *workspace,
    size_t workspace_bytes, cudaStream_t stream);

/* Static description of a status code. */
MGQA_API const char *mgqa_status_string(mgqa_status status);

/* Human-readable reason for the last host-side error on the calling thread
 * ("" when none). */
MGQA_API const char *mgqa_last_error_detail(void);

/* MGQA_ABI_VERSION of the loaded library. */
MGQA_API int32_t mgqa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MASKED_GQA_ATTN_H */
