// rows_add_rms_bf16.cu -- the row kernels of one operator (residual add + RMSNorm) for one
// storage type (bfloat16): one translation unit per pair, so they compile in
// parallel.
#include "row_kernels.cuh"

namespace nrm {

cudaError_t launch_add_rms_bf16(const RowArgs &a, const Plan &p, cudaStream_t s) {
    return launch_row<OP_ADD_RMS, __nv_bfloat16>(a, p, s);
}

}  // namespace nrm
