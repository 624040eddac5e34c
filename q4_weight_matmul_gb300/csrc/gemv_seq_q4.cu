// The Q4_K-only variants of the job-list GEMV kernel (gemv_seq_kernel.cuh),
// one per batch size, in a translation unit of their own.
#include "gemv_seq_kernel.cuh"

namespace q4k {
namespace seq {
Q4K_SEQ_VARIANTS(Q4K_SEQ_DEFINE, false)
}  // namespace seq
}  // namespace q4k
