// C ABI of the masked GQA attention library: argument validation and kernel
// dispatch. Allocates nothing and never synchronises; all work is enqueued on
// the caller's stream.
#include <cmath>
#include <cstdarg>
#include <cstdio>

#include "../../include/masked_gqa_attn.h"
#include "internal.h"

namespace mgqa {

static thread_local char g_detail[256] = "";

void clear_error_detail() { g_detail[0] = '\0'; }

mgqa_status fail(mgqa_status code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
  return code;
}

namespace {

bool aligned(const void *p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

mgqa_status check_tensor(const char *name, const void *ptr, const int64_t *st, size_t esize) {
  if (!ptr) return fail(MGQA_ERR_INVALID_ARG, "%s is null", name);
  if (!aligned(ptr, 16)) return fail(MGQA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  for (int t = 0; t < 3; ++t) {
    if (st[t] < 0) return fail(MGQA_ERR_INVALID_ARG, "%s stride %d is negative", name, t);
    if ((st[t] * (int64_t)esize) % 16 != 0)
      return fail(MGQA_ERR_INVALID_ARG, "%s stride %d is not a multiple of 16 bytes", name, t);
  }
  return MGQA_OK;
}

mgqa_status validate(const mgqa_args *a, bool decode) {
  g_detail[0] = '\0';
  if (!a) return fail(MGQA_ERR_INVALID_ARG, "args is null");
  if (a->dtype != MGQA_BF16 && a->dtype != MGQA_FP32 && a->dtype != MGQA_FP16)
    return fail(MGQA_ERR_INVALID_ARG, "unknown dtype %d", (int)a->dtype);
  if (a->B < 1 || a->Hq < 1 || a->Hkv < 1 || a->Lq < 1 || a->Lk < 1)
    return fail(MGQA_ERR_INVALID_ARG, "B, Hq, Hkv, Lq, Lk must be >= 1");
  if (a->Hq % a->Hkv != 0) return fail(MGQA_ERR_INVALID_ARG, "Hq %% Hkv != 0");
  if (a->D != 64 && a->D != 128) return fail(MGQA_ERR_UNSUPPORTED, "head dim %d (64 or 128)", a->D);
  if (a->Lk > (1 << 24) || a->Lq > (1 << 24))
    return fail(MGQA_ERR_UNSUPPORTED, "sequence longer than 2^24");
  if ((int64_t)a->B * a->Hq * a->Lq > (int64_t)1 << 31)
    return fail(MGQA_ERR_UNSUPPORTED, "B*Hq*Lq too large");
  if (decode && a->Lq != 1) return fail(MGQA_ERR_INVALID_ARG, "decode needs Lq == 1");
  if (decode && a->Lk > kDecodeMaxLk)
    return fail(MGQA_ERR_UNSUPPORTED, "decode cache longer than %d slots", kDecodeMaxLk);
  if (!std::isfinite(a->scale)) return fail(MGQA_ERR_INVALID_ARG, "scale is not finite");
  const size_t es = a->dtype == MGQA_FP32 ? 4 : 2;
  mgqa_status st;
  if ((st = check_tensor("q", a->q, a->q_stride, es)) != MGQA_OK) return st;
  if ((st = check_tensor("k", a->k, a->k_stride, es)) != MGQA_OK) return st;
  if ((st = check_tensor("v", a->v, a->v_stride, es)) != MGQA_OK) return st;
  if ((st = check_tensor("out", a->out, a->o_stride, es)) != MGQA_OK) return st;
  if (a->mask_bits) {
    if (!aligned(a->mask_bits, 4)) return fail(MGQA_ERR_INVALID_ARG, "mask_bits misaligned");
    // a stride of 0 broadcasts one mask row over the queries (a key-padding
    // mask given as [B][1][W]) or one mask over the batch rows
    const int64_t W = (a->Lk + 31) / 32;
    if (a->mask_stride_b < 0 || a->mask_stride_q < 0)
      return fail(MGQA_ERR_INVALID_ARG, "negative mask stride");
    if (a->Lq > 1 && a->mask_stride_q != 0 && a->mask_stride_q < W)
      return fail(MGQA_ERR_INVALID_ARG, "mask_stride_q is neither 0 nor >= ceil(Lk/32)");
    if (a->B > 1 && a->mask_stride_b != 0 && a->mask_stride_b < W)
      return fail(MGQA_ERR_INVALID_ARG, "mask_stride_b is neither 0 nor >= ceil(Lk/32)");
  }
  if ((a->seg_q == nullptr) != (a->seg_k == nullptr))
    return fail(MGQA_ERR_INVALID_ARG, "seg_q and seg_k must be given together");
  if (a->seg_q && (!aligned(a->seg_q, 4) || !aligned(a->seg_k, 4)))
    return fail(MGQA_ERR_INVALID_ARG, "segment ids misaligned");
  if (a->kv_len && !aligned(a->kv_len, 4)) return fail(MGQA_ERR_INVALID_ARG, "kv_len misaligned");
  if (a->lse && !aligned(a->lse, 4)) return fail(MGQA_ERR_INVALID_ARG, "lse misaligned");
  if (a->dev_error && !aligned(a->dev_error, 4))
    return fail(MGQA_ERR_INVALID_ARG, "dev_error misaligned");
  return MGQA_OK;
}

// The fused rotary embedding of a call with head dim D, Hq / Hkv heads.
mgqa_status validate_rope(const mgqa_qk_rope *r, const mgqa_args &a, bool decode, FusedRope *out) {
  if (!r) return fail(MGQA_ERR_INVALID_ARG, "rope is null");
  if (!r->inv_freq || !aligned(r->inv_freq, 4))
    return fail(MGQA_ERR_INVALID_ARG, "rope: inv_freq missing or misaligned");
  if (r->rot_dim < 2 || r->rot_dim > a.D || (r->rot_dim & 1))
    return fail(MGQA_ERR_INVALID_ARG, "rope: rot_dim must be even and in [2, D]");
  if (r->q_heads < 1 || r->q_heads > a.Hq)
    return fail(MGQA_ERR_INVALID_ARG, "rope: q_heads must be in [1, Hq]");
  if (decode && (r->k_heads < 0 || r->k_heads > a.Hkv))
    return fail(MGQA_ERR_INVALID_ARG, "rope: k_heads must be in [0, Hkv]");
  if (r->positions && !aligned(r->positions, 4))
    return fail(MGQA_ERR_INVALID_ARG, "rope: positions misaligned");
  if ((r->q_norm_weight && !aligned(r->q_norm_weight, 4)) ||
      (r->k_norm_weight && !aligned(r->k_norm_weight, 4)))
    return fail(MGQA_ERR_INVALID_ARG, "rope: norm weight misaligned");
  if ((r->q_norm_weight || r->k_norm_weight) && !(std::isfinite(r->norm_eps) && r->norm_eps >= 0.f))
    return fail(MGQA_ERR_INVALID_ARG, "rope: norm_eps must be finite and >= 0");
  out->inv_freq = r->inv_freq;
  out->positions = r->positions;
  out->half = r->rot_dim / 2;
  out->interleaved = r->interleaved != 0;
  out->q_heads = r->q_heads;
  out->k_heads = decode ? r->k_heads : 0;
  out->q_norm = r->q_norm_weight;
  out->k_norm = decode ? r->k_norm_weight : nullptr;
  out->eps = r->norm_eps;
  return MGQA_OK;
}

mgqa_status validate_append(const mgqa_args *args, const void *k_new, const void *v_new,
                            const int64_t *k_new_stride, const int64_t *v_new_stride,
                            int32_t *kv_len_out) {
  mgqa_status st = validate(args, true);
  if (st != MGQA_OK) return st;
  if (!args->kv_len) return fail(MGQA_ERR_INVALID_ARG, "append needs kv_len");
  if (args->mask_bits || args->seg_q)
    return fail(MGQA_ERR_INVALID_ARG, "append takes the kv_len form only");
  if (!k_new || !v_new || !k_new_stride || !v_new_stride)
    return fail(MGQA_ERR_INVALID_ARG, "append needs k_new, v_new and their strides");
  const size_t es = args->dtype == MGQA_FP32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(k_new) % 16) || (reinterpret_cast<uintptr_t>(v_new) % 16))
    return fail(MGQA_ERR_INVALID_ARG, "k_new / v_new not 16-byte aligned");
  for (int t = 0; t < 2; ++t)
    if (k_new_stride[t] < 0 || v_new_stride[t] < 0 || (k_new_stride[t] * (int64_t)es) % 16 ||
        (v_new_stride[t] * (int64_t)es) % 16)
      return fail(MGQA_ERR_INVALID_ARG, "k_new / v_new strides must be multiples of 16 bytes");
  if (kv_len_out && kv_len_out == args->kv_len)
    return fail(MGQA_ERR_INVALID_ARG, "kv_len_out must not alias kv_len");
  if (kv_len_out && (reinterpret_cast<uintptr_t>(kv_len_out) % 4))
    return fail(MGQA_ERR_INVALID_ARG, "kv_len_out misaligned");
  return MGQA_OK;
}

}  // namespace
}  // namespace mgqa

extern "C" {

mgqa_status masked_gqa_attn_prefill(const mgqa_args *args, cudaStream_t stream) {
  mgqa_status st = mgqa::validate(args, false);
  if (st != MGQA_OK) return st;
  if (args->dtype != MGQA_FP32) return mgqa::launch_prefill_tc(*args, stream);
  return mgqa::launch_prefill_simt(*args, stream);
}

size_t masked_gqa_attn_decode_workspace_size(const mgqa_args *args) {
  if (mgqa::validate(args, true) != MGQA_OK) return 0;
  return mgqa::kDecodeWorkspaceBytes;
}

mgqa_status masked_gqa_attn_decode(const mgqa_args *args, void *workspace, size_t workspace_bytes,
                                   cudaStream_t stream) {
  (void)workspace;  // merged on chip: nothing is read or written there
  (void)workspace_bytes;
  mgqa_status st = mgqa::validate(args, true);
  if (st != MGQA_OK) return st;
  return mgqa::launch_decode(*args, stream);
}

mgqa_status masked_gqa_attn_decode_append(const mgqa_args *args, const void *k_new,
                                          const void *v_new, const int64_t *k_new_stride,
                                          const int64_t *v_new_stride, int32_t *kv_len_out,
                                          void *workspace, size_t workspace_bytes,
                                          cudaStream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  const mgqa_status st = mgqa::validate_append(args, k_new, v_new, k_new_stride, v_new_stride,
                                               kv_len_out);
  if (st != MGQA_OK) return st;
  return mgqa::launch_decode_append(*args, k_new, v_new, k_new_stride, v_new_stride, kv_len_out,
                                    stream);
}

mgqa_status masked_gqa_attn_decode_append_rope(const mgqa_args *args, const void *k_new,
                                               const void *v_new, const int64_t *k_new_stride,
                                               const int64_t *v_new_stride, int32_t *kv_len_out,
                                               const mgqa_qk_rope *rope, void *workspace,
                                               size_t workspace_bytes, cudaStream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  mgqa_status st = mgqa::validate_append(args, k_new, v_new, k_new_stride, v_new_stride,
                                         kv_len_out);
  if (st != MGQA_OK) return st;
  mgqa::FusedRope fr;
  if ((st = mgqa::validate_rope(rope, *args, true, &fr)) != MGQA_OK) return st;
  return mgqa::launch_decode_append(*args, k_new, v_new, k_new_stride, v_new_stride, kv_len_out,
                                    stream, fr);
}

mgqa_status masked_gqa_attn_prefill_rope(const mgqa_args *args, const mgqa_qk_rope *rope,
                                         cudaStream_t stream) {
  mgqa_status st = mgqa::validate(args, false);
  if (st != MGQA_OK) return st;
  if (args->dtype == MGQA_FP32)
    return mgqa::fail(MGQA_ERR_UNSUPPORTED,
                      "the fused rotary embedding runs on the bf16 / fp16 path; rotate fp32 inputs "
                      "with masked_gqa_rope");
  mgqa::FusedRope fr;
  if ((st = mgqa::validate_rope(rope, *args, false, &fr)) != MGQA_OK) return st;
  // the kernel keeps a query row in registers, which needs the pairing fixed
  // at compile time: half-split rotations over D, D/2 or D/4 features
  if (!fr.interleaved && fr.half != args->D / 2 && fr.half != args->D / 4 && fr.half != args->D / 8)
    return mgqa::fail(MGQA_ERR_UNSUPPORTED,
                      "fused prefill: half-split rotary dims must be D, D/2 or D/4 (rotate with "
                      "masked_gqa_rope for other widths)");
  return mgqa::launch_prefill_tc(*args, stream, fr);
}

const char *mgqa_status_string(mgqa_status s) {
  switch (s) {
    case MGQA_OK: return "ok";
    case MGQA_ERR_INVALID_ARG: return "invalid argument";
    case MGQA_ERR_UNSUPPORTED: return "unsupported";
    case MGQA_ERR_CUDA: return "CUDA error";
    case MGQA_ERR_TIMEOUT: return "device wait timed out";
    case MGQA_ERR_DEVICE_CHECK: return "device bounds check failed (debug library)";
  }
  return "unknown status";
}

const char *mgqa_last_error_detail(void) { return mgqa::g_detail; }

int32_t mgqa_abi_version(void) { return MGQA_ABI_VERSION; }

}  // extern "C"
