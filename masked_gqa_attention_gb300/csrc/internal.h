// Host-side interfaces between the C ABI (api.cu) and the kernel launchers.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/masked_gqa_attn.h"

namespace mgqa {

// Sets the thread-local detail string returned by mgqa_last_error_detail().
mgqa_status fail(mgqa_status code, const char *fmt, ...);
// Empties the calling thread's error detail (entry points call it first).
void clear_error_detail();

// Raises `kern`'s dynamic shared-memory limit to `bytes` on the current
// device the first time it launches there. The attribute belongs to a device,
// so `done` (one per kernel instantiation, owned by its launcher) keeps a bit
// per device; host threads that race here both set the same value, which is
// harmless. Devices past 63 set the attribute on every launch.
template <typename Kern>
mgqa_status ensure_smem_attr(Kern kern, int bytes, std::atomic<uint64_t> &done, const char *what) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(MGQA_ERR_CUDA, "no current CUDA device");
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return MGQA_OK;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return fail(MGQA_ERR_CUDA, "cudaFuncSetAttribute failed for the %s", what);
  if (bit) done.fetch_or(bit, std::memory_order_release);
  return MGQA_OK;
}

// ensure_smem_attr for a kernel launched in clusters of up to 16 CTAs (past
// the portable 8), spread over as many SMs as the GPU allows.
template <typename Kern>
mgqa_status ensure_cluster_attr(Kern kern, int bytes, std::atomic<uint64_t> &done, const char *what) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(MGQA_ERR_CUDA, "no current CUDA device");
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return MGQA_OK;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeClusterSchedulingPolicyPreference,
                           cudaClusterSchedulingPolicySpread) != cudaSuccess)
    return fail(MGQA_ERR_CUDA, "cudaFuncSetAttribute failed for the %s", what);
  if (bit) done.fetch_or(bit, std::memory_order_release);
  return MGQA_OK;
}

// launch_pdl in thread-block clusters of cluster_x CTAs along x.
template <typename Kern, typename... Args>
cudaError_t launch_pdl_cluster(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Launch with programmatic stream serialisation (the kernel itself calls
// grid_dependency_wait() before touching global memory).
template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Rotary embedding (and RMS normalisation) applied inside an attention
// kernel; inactive when inv_freq is null.
struct FusedRope {
  const float *inv_freq = nullptr;
  const int32_t *positions = nullptr;
  int half = 0;         // rot_dim / 2
  int interleaved = 0;
  int q_heads = 0, k_heads = 0;
  const float *q_norm = nullptr, *k_norm = nullptr;
  float eps = 0.f;
};

// Decode: the cache is cut into chunks of kDecodeChunk absolute slots; the
// kDecodeSplits CTAs (one cluster) of a (request, head group) own every
// kDecodeSplits-th chunk.
constexpr int kDecodeChunk = 64;
constexpr int kDecodeSplits = 16;
// Longest static cache the decode kernel accepts (bounds its chunk masks).
constexpr int kDecodeMaxLk = 32768;
// Nominal workspace size reported for valid decode arguments: the kernel
// merges on chip and never touches a workspace.
constexpr size_t kDecodeWorkspaceBytes = 16;
// Heads handled by one decode CTA (a divisor of Hq/Hkv, at most 8).
int decode_heads_per_cta(int n_rep);
mgqa_status launch_decode(const mgqa_args &a, cudaStream_t s);
mgqa_status launch_decode_append(const mgqa_args &a, const void *k_new, const void *v_new,
                                 const int64_t *k_new_stride, const int64_t *v_new_stride,
                                 int32_t *kv_len_out, cudaStream_t s,
                                 const FusedRope &rope = FusedRope());

// Packed-guidance row copies (pack or unpack one pair of sequences).
mgqa_status pack_pair(bool unpack, mgqa_dtype dt, int B, int H, int D, const void *a,
                      const int64_t *as, int La, const void *b, const int64_t *bs, int Lb,
                      const void *packed, const int64_t *ps, int32_t *seg, cudaStream_t s);

// 4-D tensor map over a [B][H][L][D] view with element strides st = (batch,
// head, position), for TMA boxes of box_x columns x box_y rows (128-byte
// swizzle or none). false when the driver entry point is missing or the
// encoding is refused.
bool make_tma_map_4d(CUtensorMap *m, mgqa_dtype dt, const void *base, int B, int H, int L, int D,
                     const int64_t *st, int box_x, int box_y, bool swizzle128);

// Prefill on the CUDA cores (fp32 I/O).
mgqa_status launch_prefill_simt(const mgqa_args &a, cudaStream_t s);

// Prefill on the tensor cores (bf16 / fp16 I/O): TMA + tcgen05 + TMEM.
mgqa_status launch_prefill_tc(const mgqa_args &a, cudaStream_t s,
                              const FusedRope &rope = FusedRope());

}  // namespace mgqa
