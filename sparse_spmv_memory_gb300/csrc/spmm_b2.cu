// spmm_b2.cu -- the small-batch SpMM kernels with 2-token x slots.
#include "spmm_kernels.cuh"

namespace nmk {
template cudaError_t launch_spmm_variant<2>(const SpmmParams&, int, int, int, cudaStream_t);
}  // namespace nmk
