// Row-tile and swapped kernels built for the BIAS epilog alone (no other epilog's code
// in them), one translation unit per epilog so that they compile in parallel.
#include "gemm_single.cuh"

namespace gemm_epi {

GEMM_EPI_FORWARD_INSTANCES(EPI_BIAS, bias)

}  // namespace gemm_epi
