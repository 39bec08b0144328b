// rows_add_rms.cu -- template instances of the row kernels for one operator
// (one translation unit per operator so they compile in parallel).
#include "row_kernels.cuh"

namespace nrm {

cudaError_t launch_add_rms(const RowArgs &a, const Plan &p, int dtype, cudaStream_t s) {
    return launch_row_dtype<OP_ADD_RMS>(a, p, dtype, s);
}

}  // namespace nrm
