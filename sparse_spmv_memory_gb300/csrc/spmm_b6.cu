// spmm_b6.cu -- the small-batch SpMM kernels with 6-token x slots.
#include "spmm_kernels.cuh"

namespace nmk {
template cudaError_t launch_spmm_variant<6>(const SpmmParams&, int, int, int, cudaStream_t);
}  // namespace nmk
