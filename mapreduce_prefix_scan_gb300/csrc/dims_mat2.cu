// dims_mat2.cu -- strided / contiguous / general dims-reduction kernels for
// mat2 input (one translation unit per input type, built in parallel).
#include "reduce_dims.cuh"

namespace ak {
ak_status run_dims_mat2(const DimsCall& c, const DimsPlan& p) { return dims::run_for_input<Mat2>(c, p); }
}  // namespace ak
