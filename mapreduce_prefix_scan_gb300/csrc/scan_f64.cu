// scan_f64.cu -- scan kernels for f64 input (one translation unit per input
// type, built in parallel).
#include "scan.cuh"

namespace ak {
ak_status run_scan_f64(const ScanCall& c, const ScanPlan& p) { return scan::run_for_input<double>(c, p); }
}  // namespace ak
