// scan_i64.cu -- scan kernels for i64 input (one translation unit per input
// type, built in parallel).
#include "scan.cuh"

namespace ak {
ak_status run_scan_i64(const ScanCall& c, const ScanPlan& p) { return scan::run_for_input<int64_t>(c, p); }
}  // namespace ak
