// scan_mat2.cu -- scan kernels for mat2 input (one translation unit per input
// type, built in parallel).
#include "scan.cuh"

namespace ak {
ak_status run_scan_mat2(const ScanCall& c, const ScanPlan& p) { return scan::run_for_input<Mat2>(c, p); }
}  // namespace ak
