// scan_f32.cu -- scan kernels for f32 input (one translation unit per input
// type, built in parallel).
#include "scan.cuh"

namespace ak {
ak_status run_scan_f32(const ScanCall& c, const ScanPlan& p) { return scan::run_for_input<float>(c, p); }
}  // namespace ak
