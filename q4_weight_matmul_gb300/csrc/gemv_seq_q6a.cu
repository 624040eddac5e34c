// The mixed Q4_K / Q6_K variants of the job-list GEMV kernel
// (gemv_seq_kernel.cuh) for batch 1-4, in a translation unit of their own.
#include "gemv_seq_kernel.cuh"

namespace q4k {
namespace seq {
Q4K_SEQ_VARIANTS_1_4(Q4K_SEQ_DEFINE, true)
}  // namespace seq
}  // namespace q4k
