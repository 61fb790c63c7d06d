// dims_bf16.cu -- strided / contiguous / general dims-reduction kernels for
// bf16 input (one translation unit per input type, built in parallel).
#include "reduce_dims.cuh"

namespace ak {
ak_status run_dims_bf16(const DimsCall& c, const DimsPlan& p) { return dims::run_for_input<bf16>(c, p); }
}  // namespace ak
