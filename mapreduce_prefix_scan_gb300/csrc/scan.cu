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
                    bool no_neutral, int target_blocks, int items, const DeviceInfo& dev, ScanPlan* p) {
    (void)op;
    (void)target_blocks;
    (void)dev;
    const size_t psz = partial_size(acc, no_neutral);
    const size_t asz = ak_dtype_size(acc);
    if (!psz || !asz) return AK_ERR_UNSUPPORTED;
    p->state_off = kWsHeader;
    p->ws_bytes = kWsHeader;
    p->tiles = 0;
    p->tiles_per_line = 0;
    p->grid = 0;
    p->tma = false;
    p->tma_tiles_per_line = 0;
    p->tma_tiles = 0;
    p->tma_ws_bytes = 0;
    if (inner > 1) {
        p->kind = 1;
        p->block = 256;
        p->items = 1;
        return AK_OK;
    }
    p->kind = 0;
    const int it = asz >= 16 ? 8 : (asz == 8 ? 16 : 32);
    if (items != 0 && items != it) return AK_ERR_UNSUPPORTED;
    p->items = it;
    const int block = asz >= 16 ? 128 : 256;
    const int seg = asz >= 16 ? 64 : (asz == 8 ? 64 : 32);
    p->block = block;
    const int64_t tile = (int64_t)block * it;
    if (len <= tile) {
        p->kind = 2;  // every line fits one tile: no state shared between blocks
        p->tiles_per_line = 1;
        p->tiles = outer;
        return AK_OK;
    }
    const int64_t super = (int64_t)block * seg;
    p->tiles_per_line = (len + super - 1) / super;
    p->tiles = p->tiles_per_line * outer;
    p->ws_bytes = align_up(kWsHeader + (size_t)p->tiles * (16 + align_up(psz, 16)), 256);  // TileRec per super-tile
    // TMA tile scan: one element type throughout, f32 / i32 / i64 with a
    // neutral element (f64 additions run on the FP64 pipe, the matrix product
    // spends more operator work per byte, Optional partials more per combine:
    // those run faster as super-tiles, whose blocks carry more warps per SM),
    // rows of 128 bytes,
    // several tiles per line, and lines that start on a row boundary unless
    // there is only one
    const int64_t rl = 128 / (int64_t)asz;
    if (items == 0 && in == acc && out == acc && (acc == AK_F32 || acc == AK_I32 || acc == AK_I64) && !no_neutral &&
        len > scan::kWsRows * rl &&
        (outer == 1 || len % rl == 0) && len / rl < ((int64_t)1 << 31) && outer < ((int64_t)1 << 31)) {
        const int64_t rows = (len + rl - 1) / rl;
        p->tma = true;
        p->tma_tiles_per_line = (rows + scan::kWsRows - 1) / scan::kWsRows;
        p->tma_tiles = p->tma_tiles_per_line * outer;
        p->tma_ws_bytes = align_up(kWsHeader + (size_t)p->tma_tiles * (16 + align_up(psz, 16)), 256);
        p->ws_bytes = std::max(p->ws_bytes, p->tma_ws_bytes);
    }
    return AK_OK;
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
