// Packed-guidance helpers: build the one-row block-diagonal input from a
// conditional and an unconditional sequence, and split a packed output back.
//
// Passage: OmniVoice page, "Memory & speed", packed_guidance paragraph: the
// conditional sequence and the unconditional one (its target part only) sit
// side by side in one row under a block-diagonal mask, positions of each
// starting at 0, instead of two rows padded to the same length.
//
// One kernel copies rows of [B][H][L][D] views: CTA (row block, h, b), each
// thread moving 16-byte pieces, so every row is one coalesced read and write.
#include "common.cuh"
#include "internal.h"

namespace mgqa {
namespace {

struct CopyRows {
  const char *src;
  char *dst;
  int64_t ss[3], ds[3];  // strides in bytes (b, h, l)
  int L, dst_off, row_bytes;
  int32_t *seg;          // optional [B][seg_len]: seg_val for rows dst_off .. dst_off+L-1
  int seg_len, seg_val;
};

constexpr int kRowsPerCta = 32;

__global__ void __launch_bounds__(256) copy_rows_kernel(const __grid_constant__ CopyRows c) {
  const int b = blockIdx.z, h = blockIdx.y;
  const int r0 = blockIdx.x * kRowsPerCta;
  const int ppr = c.row_bytes / 16;
  for (int idx = threadIdx.x; idx < kRowsPerCta * ppr; idx += blockDim.x) {
    const int r = r0 + idx / ppr, part = idx % ppr;
    if (r >= c.L) break;
    const uint4 *s = reinterpret_cast<const uint4 *>(c.src + b * c.ss[0] + h * c.ss[1] + r * c.ss[2]);
    uint4 *d = reinterpret_cast<uint4 *>(c.dst + b * c.ds[0] + h * c.ds[1] +
                                         (int64_t)(c.dst_off + r) * c.ds[2]);
    d[part] = s[part];
  }
  if (c.seg && h == 0)
    for (int r = r0 + threadIdx.x; r < min(c.L, r0 + kRowsPerCta); r += blockDim.x)
      c.seg[(int64_t)b * c.seg_len + c.dst_off + r] = c.seg_val;
}

mgqa_status copy_rows(const CopyRows &c, int B, int H, cudaStream_t s) {
  if (c.L == 0) return MGQA_OK;
  dim3 grid((c.L + kRowsPerCta - 1) / kRowsPerCta, H, B);
  copy_rows_kernel<<<grid, 256, 0, s>>>(c);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(MGQA_ERR_CUDA, "copy launch: %s", cudaGetErrorString(e));
  return MGQA_OK;
}

mgqa_status check_view(const char *name, const void *p, const int64_t *st, size_t es, int L) {
  if (!p && L > 0) return fail(MGQA_ERR_INVALID_ARG, "%s is null", name);
  if ((reinterpret_cast<uintptr_t>(p) % 16) != 0)
    return fail(MGQA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  for (int t = 0; t < 3; ++t)
    if (st[t] < 0 || (st[t] * (int64_t)es) % 16 != 0)
      return fail(MGQA_ERR_INVALID_ARG, "%s strides must be non-negative multiples of 16 bytes",
                  name);
  return MGQA_OK;
}

}  // namespace

mgqa_status pack_pair(bool unpack, mgqa_dtype dt, int B, int H, int D, const void *a,
                      const int64_t *as, int La, const void *bb, const int64_t *bs, int Lb,
                      const void *packed, const int64_t *ps, int32_t *seg, cudaStream_t s) {
  if (dt != MGQA_BF16 && dt != MGQA_FP16 && dt != MGQA_FP32)
    return fail(MGQA_ERR_INVALID_ARG, "unknown dtype");
  const size_t es = dt == MGQA_FP32 ? 4 : 2;
  if (B < 1 || H < 1 || D < 1 || La < 0 || Lb < 0 || (D * es) % 16 != 0)
    return fail(MGQA_ERR_INVALID_ARG, "bad sizes (D * element size must be a multiple of 16)");
  mgqa_status st;
  if ((st = check_view("a", a, as, es, La)) != MGQA_OK) return st;
  if ((st = check_view("b", bb, bs, es, Lb)) != MGQA_OK) return st;
  if ((st = check_view("packed", packed, ps, es, La + Lb)) != MGQA_OK) return st;
  if (seg && (reinterpret_cast<uintptr_t>(seg) % 4) != 0)
    return fail(MGQA_ERR_INVALID_ARG, "seg misaligned");
  for (int part = 0; part < 2; ++part) {
    CopyRows c{};
    const void *x = part == 0 ? a : bb;
    const int64_t *xs = part == 0 ? as : bs;
    c.L = part == 0 ? La : Lb;
    c.row_bytes = (int)(D * es);
    if (!unpack) {
      c.src = static_cast<const char *>(x);
      c.dst = static_cast<char *>(const_cast<void *>(packed));
      for (int t = 0; t < 3; ++t) { c.ss[t] = xs[t] * es; c.ds[t] = ps[t] * es; }
      c.dst_off = part == 0 ? 0 : La;
      c.seg = seg;
      c.seg_len = La + Lb;
      c.seg_val = part;
    } else {
      // read rows [off, off + L) of the packed view into x
      c.src = static_cast<const char *>(packed) + (part == 0 ? 0 : (int64_t)La * ps[2] * es);
      c.dst = static_cast<char *>(const_cast<void *>(x));
      for (int t = 0; t < 3; ++t) { c.ss[t] = ps[t] * es; c.ds[t] = xs[t] * es; }
      c.dst_off = 0;
    }
    if ((st = copy_rows(c, B, H, s)) != MGQA_OK) return st;
  }
  return MGQA_OK;
}

}  // namespace mgqa

extern "C" mgqa_status masked_gqa_pack_pair(mgqa_dtype dtype, int32_t B, int32_t H, int32_t D,
                                            const void *a, const int64_t *a_stride, int32_t La,
                                            const void *b, const int64_t *b_stride, int32_t Lb,
                                            void *packed, const int64_t *packed_stride,
                                            int32_t *seg, cudaStream_t stream) {
  if (!a_stride || !b_stride || !packed_stride)
    return mgqa::fail(MGQA_ERR_INVALID_ARG, "strides are null");
  return mgqa::pack_pair(false, dtype, B, H, D, a, a_stride, La, b, b_stride, Lb, packed,
                         packed_stride, seg, stream);
}

extern "C" mgqa_status masked_gqa_unpack_pair(mgqa_dtype dtype, int32_t B, int32_t H, int32_t D,
                                              const void *packed, const int64_t *packed_stride,
                                              void *a, const int64_t *a_stride, int32_t La,
                                              void *b, const int64_t *b_stride, int32_t Lb,
                                              cudaStream_t stream) {
  if (!a_stride || !b_stride || !packed_stride)
    return mgqa::fail(MGQA_ERR_INVALID_ARG, "strides are null");
  return mgqa::pack_pair(true, dtype, B, H, D, a, a_stride, La, b, b_stride, Lb, packed,
                         packed_stride, nullptr, stream);
}
