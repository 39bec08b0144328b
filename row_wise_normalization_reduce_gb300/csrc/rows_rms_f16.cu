// rows_rms_f16.cu -- the row kernels of one operator (RMSNorm) for one
// storage type (binary16): one translation unit per pair, so they compile in
// parallel.
#include "row_kernels.cuh"

namespace nrm {

cudaError_t launch_rms_f16(const RowArgs &a, const Plan &p, cudaStream_t s) {
    return launch_row<OP_RMS, __half>(a, p, s);
}

}  // namespace nrm
