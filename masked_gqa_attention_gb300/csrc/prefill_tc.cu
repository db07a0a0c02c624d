// Placeholder until the tensor-core prefill kernel lands: bf16 prefill runs
// on the CUDA-core kernel.
#include "internal.h"

namespace mgqa {
mgqa_status launch_prefill_tc(const mgqa_args &a, cudaStream_t s) { return launch_prefill_simt(a, s); }
}  // namespace mgqa
