// scan.cu -- host side of the scans: the plan (kernel choice, tile counts,
// workspace) and the dispatch of a call's types, operator and monoid to the
// kernels of scan.cuh.
#include <algorithm>

#include "scan.cuh"

namespace ak {

ak_status run_scan_f32(const ScanCall& c, const ScanPlan& p);
ak_status run_scan_f64(const ScanCall& c, const ScanPlan& p);
ak_status run_scan_i32(const ScanCall& c, const ScanPlan& p);
ak_status run_scan_i64(const ScanCall& c, const ScanPlan& p);
ak_status run_scan_mat2(const ScanCall& c, const ScanPlan& p);

ak_status plan_scan(int64_t inner, int64_t len, int64_t outer, ak_dtype in, ak_dtype acc, ak_dtype out, ak_op op,
                    bool no_neutral, int target_blocks, int items, const DeviceInfo& dev, ScanPlan* p,
                    bool single_pass) {
    (void)target_blocks;
    (void)dev;
    const size_t psz = partial_size(acc, no_neutral);
    const size_t asz = ak_dtype_size(acc);
    if (!psz || !asz) return AK_ERR_UNSUPPORTED;
    // the TMA tile scan takes one element type throughout: f32 / i32 / i64
    // with a neutral element, and f64 sums (whose row folds run in fixed
    // point, so that only the scan itself uses the FP64 pipe)
    const bool tma_type = in == acc && out == acc && !no_neutral &&
                          (acc == AK_F32 || acc == AK_I32 || acc == AK_I64 || (acc == AK_F64 && op == AK_OP_ADD));
    return scan::plan_sizes(inner, len, outer, asz, psz, tma_type, items, p, ak_dtype_size(in), single_pass);
}

ak_status run_scan(const ScanCall& c, const ScanPlan& plan) {
    switch (c.in) {
    case AK_F32: return run_scan_f32(c, plan);
    case AK_F64: return run_scan_f64(c, plan);
    case AK_I32: return run_scan_i32(c, plan);
    case AK_I64: return run_scan_i64(c, plan);
    case AK_MAT2_MODP: return run_scan_mat2(c, plan);
    default: return AK_ERR_UNSUPPORTED;
    }
}

}  // namespace ak
