// rows_add_rms_f32.cu -- the row kernels of one operator (residual add + RMSNorm) for one
// storage type (binary32): one translation unit per pair, so they compile in
// parallel.
#include "row_kernels.cuh"

namespace nrm {

cudaError_t launch_add_rms_f32(const RowArgs &a, const Plan &p, cudaStream_t s) {
    return launch_row<OP_ADD_RMS, float>(a, p, s);
}

}  // namespace nrm
