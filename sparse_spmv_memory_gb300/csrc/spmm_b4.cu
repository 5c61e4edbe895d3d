// spmm_b4.cu -- the small-batch SpMM kernels with 4-token x slots.
#include "spmm_kernels.cuh"

namespace nmk {
template cudaError_t launch_spmm_variant<4>(const SpmmParams&, int, int, int, cudaStream_t);
}  // namespace nmk
