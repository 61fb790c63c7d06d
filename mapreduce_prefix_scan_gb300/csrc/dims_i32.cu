// dims_i32.cu -- strided / contiguous / general dims-reduction kernels for
// i32 input (one translation unit per input type, built in parallel).
#include "reduce_dims.cuh"

namespace ak {
ak_status run_dims_i32(const DimsCall& c, const DimsPlan& p) { return dims::run_for_input<int32_t>(c, p); }
}  // namespace ak
