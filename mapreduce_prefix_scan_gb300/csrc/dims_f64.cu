// dims_f64.cu -- strided / contiguous / general dims-reduction kernels for
// f64 input (one translation unit per input type, built in parallel).
#include "reduce_dims.cuh"

namespace ak {
ak_status run_dims_f64(const DimsCall& c, const DimsPlan& p) { return dims::run_for_input<double>(c, p); }
}  // namespace ak
