// scan_i32.cu -- scan kernels for i32 input (one translation unit per input
// type, built in parallel).
#include "scan.cuh"

namespace ak {
ak_status run_scan_i32(const ScanCall& c, const ScanPlan& p) { return scan::run_for_input<int32_t>(c, p); }
}  // namespace ak
