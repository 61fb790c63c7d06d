// reduce_dims.cu -- host side of the reductions over a set of dimensions:
// shape selection, workspace plan, dispatch by input type to the kernel
// translation units (dims_*.cu), and the fill used for empty reductions.
// The kernels and their design notes are in reduce_dims.cuh.
#include <algorithm>

#include "reduce_dims.cuh"

namespace ak {

ak_status run_dims_f32(const DimsCall& c, const DimsPlan& p);
ak_status run_dims_bf16(const DimsCall& c, const DimsPlan& p);
ak_status run_dims_f64(const DimsCall& c, const DimsPlan& p);
ak_status run_dims_i32(const DimsCall& c, const DimsPlan& p);
ak_status run_dims_i64(const DimsCall& c, const DimsPlan& p);
ak_status run_dims_mat2(const DimsCall& c, const DimsPlan& p);

namespace {

using dims::kBlock;
using dims::kMinRowsPerGroup;
constexpr int kMaxCluster = 16;
constexpr int64_t kClusterAutoBytes = (int64_t)16 << 20;  // default cluster combine up to this input size
// fewest reduction rows a block of a cluster should get
constexpr int64_t R_rows_min(int row_groups) { return (int64_t)row_groups * 2; }

template <class Out>
__global__ void k_fill(Out* dst, int64_t count, Out v) {
    const int64_t i = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    if (i < count) dst[i] = v;
}

}  // namespace

// Shape selection for the strided form (see k_dims_strided). The block has
// kBlock threads; a row segment of tile_out outputs is read by tpr <= 32
// threads with vec-wide loads. The reduction is split only as far as needed
// to give the device about target_ctas blocks, and never below
// kMinRowsPerGroup rows per group.
static void select_shape(int64_t I, int64_t J, int64_t K, int esz, int vec, int sm_count, int forced,
                         bool allow_cluster, bool auto_cluster, DimsPlan* p) {
    const int64_t vecs_per_row = (I + vec - 1) / vec;
    // Enough outputs that one thread per vector of outputs already puts
    // kUnroll loads in flight on every thread slot of the device.
    const bool many_outputs = vecs_per_row * K >= (int64_t)sm_count * 2048;
    int shape = forced;
    if (shape == AK_SHAPE_AUTO) shape = (J < 32 || many_outputs) ? AK_SHAPE_THREAD : AK_SHAPE_COLUMNS;
    p->vec = vec;
    p->cluster = false;
    if (shape == AK_SHAPE_THREAD) {
        const int tpr = (int)std::min<int64_t>(kBlock, vecs_per_row);
        p->tile_out = tpr * vec;
        p->row_groups = 1;
        p->split = 1;
        p->shape = AK_SHAPE_THREAD;
        return;
    }
    // Blocks wanted: enough that one round of kUnroll 16-byte loads per thread
    // covers the whole input (latency-bound sizes), at most 8 per SM.
    const int64_t bytes = I * J * K * esz;
    const int64_t per_block = (int64_t)kBlock * dims::kUnroll * 16;
    const int64_t target = std::max<int64_t>(sm_count, std::min<int64_t>((int64_t)sm_count * 8,
                                                                         (bytes + per_block - 1) / per_block));
    auto set_tile = [&](int tpr) {
        p->tile_out = tpr * vec;
        p->row_groups = kBlock / tpr;
        return ((I + p->tile_out - 1) / p->tile_out) * K;  // output tiles
    };
    // The split blocks of an output tile combine in a thread-block cluster
    // (no workspace, no second launch) on request, and by default for
    // inputs of at most kClusterAutoBytes: there the second launch is a
    // large part of the call (3072 x 2048 bf16 back to back: 7.2 against
    // 7.8 us), while on larger inputs the smaller clusters' longer row
    // ranges cost more than the launch they save.
    const bool cluster_ok = allow_cluster || (auto_cluster && forced == AK_SHAPE_AUTO && bytes <= kClusterAutoBytes);
    if (shape == AK_SHAPE_COLUMNS && cluster_ok) {
        // Prefer a cluster split (2..16 blocks per output tile, partials
        // combined in distributed shared memory): try row segments of 32,
        // 16, 8 and 4 threads until the wanted split fits a cluster. The
        // whole grid must be resident at once (a cluster that waits for a
        // second wave doubles the time of these latency-bound sizes): one
        // round of kUnroll 16-byte rows per thread, at most 4 blocks per SM
        // (the kernel's register budget).
        const int64_t per_block_c = (int64_t)kBlock * dims::kUnroll * 16;
        const int64_t target_c = std::max<int64_t>(sm_count, std::min<int64_t>((int64_t)sm_count * 4,
                                                                               (bytes + per_block_c - 1) / per_block_c));
        for (int tpr : {32, 16, 8, 4}) {
            if (tpr > vecs_per_row && tpr != 4) continue;
            const int64_t tiles = set_tile((int)std::min<int64_t>(tpr, vecs_per_row));
            if (kBlock % p->tile_out != 0) continue;
            const int64_t want = (target_c + tiles - 1) / tiles;
            if (want <= 1) {
                p->split = 1;
                p->shape = AK_SHAPE_TILED;
                return;
            }
            if (want <= kMaxCluster) {
                int cs = 2;
                while (cs < want) cs *= 2;
                if ((int64_t)cs * R_rows_min(p->row_groups) <= J) {
                    p->split = cs;
                    p->cluster = true;
                    p->shape = AK_SHAPE_COLUMNS;
                    return;
                }
            }
        }
    }
    // Split through a workspace and a second pass (or no split: tiled).
    const int64_t tiles = set_tile((int)std::min<int64_t>(32, vecs_per_row));
    int64_t split = (target + tiles - 1) / tiles;
    const int64_t max_split = std::max<int64_t>(1, J / ((int64_t)p->row_groups * kMinRowsPerGroup));
    split = std::max<int64_t>(1, std::min<int64_t>(split, max_split));
    split = std::min<int64_t>(split, 65535);
    if (shape == AK_SHAPE_TILED) split = 1;
    if (shape == AK_SHAPE_COLUMNS && forced == AK_SHAPE_COLUMNS && split == 1 && J >= 2) split = 2;
    p->split = (int)split;
    p->shape = split > 1 ? AK_SHAPE_COLUMNS : AK_SHAPE_TILED;
}

ak_status plan_dims(const DimsCall& c, const DeviceInfo& dev, DimsPlan* p) {
    const size_t psz = partial_size(c.acc, c.no_neutral);
    const size_t esz = ak_dtype_size(c.in);
    if (!psz || !esz) return AK_ERR_UNSUPPORTED;
    p->ws_bytes = kWsHeader;
    p->split = 1;
    p->cluster = false;
    p->vec = 1;
    p->tile_out = 1;
    p->row_groups = 1;
    p->shape = AK_SHAPE_THREAD;
    if (c.general) {
        // many outputs: a thread per output; few: blocks of (output, split)
        // pairs, split until the device has a few blocks per SM
        int64_t nout = 1, nfold = 1;
        for (int d = 0; d < c.ndim; ++d) {
            if ((c.mask >> d) & 1u) nfold *= c.shape[d];
            else nout *= c.shape[d];
        }
        if (nout >= (int64_t)dev.sm_count * kBlock * 4 || nout > 65535 * 1024) return AK_OK;
        p->shape = AK_SHAPE_TILED;
        int64_t split = ((int64_t)dev.sm_count * 4 + nout - 1) / nout;
        split = std::max<int64_t>(1, std::min<int64_t>({split, (nfold + 4095) / 4096, 65535}));
        p->split = (int)split;
        if (split > 1) {
            p->shape = AK_SHAPE_COLUMNS;
            p->ws_bytes = align_up(kWsHeader + (size_t)split * nout * psz, 256);
        }
        return AK_OK;
    }
    if (c.inner == 1) {
        // contiguous reduction: split long rows when there are few outputs
        const int64_t target_warps = (int64_t)dev.sm_count * 64;
        int64_t split = (target_warps + c.outer - 1) / c.outer;
        split = std::max<int64_t>(1, std::min<int64_t>(split, c.red / 1024));
        p->split = (int)split;
        p->shape = split > 1 ? AK_SHAPE_COLUMNS : AK_SHAPE_TILED;
    } else {
        const uintptr_t addr = reinterpret_cast<uintptr_t>(c.src);
        int vec = 1;
        if (esz < 16 && addr % 16 == 0 && (c.inner * (int64_t)esz) % 16 == 0 && (c.ldj * (int64_t)esz) % 16 == 0 &&
            (c.outer == 1 || (c.ldk * (int64_t)esz) % 16 == 0))
            vec = (int)(16 / esz);
        select_shape(c.inner, c.red, c.outer, (int)esz, vec, dev.sm_count, c.forced_shape, c.allow_cluster,
                     c.auto_cluster, p);
    }
    if (p->split > 1 && !p->cluster)
        p->ws_bytes = align_up(kWsHeader + (size_t)p->split * c.inner * c.outer * psz, 256);
    return AK_OK;
}

ak_status run_reduce_dims(const DimsCall& c, const DimsPlan& plan) {
    switch (c.in) {
    case AK_F32: return run_dims_f32(c, plan);
    case AK_BF16: return run_dims_bf16(c, plan);
    case AK_F64: return run_dims_f64(c, plan);
    case AK_I32: return run_dims_i32(c, plan);
    case AK_I64: return run_dims_i64(c, plan);
    case AK_MAT2_MODP: return run_dims_mat2(c, plan);
    default: return AK_ERR_UNSUPPORTED;
    }
}

ak_status run_fill(void* dst, int64_t count, ak_dtype out, const Value16& value, cudaStream_t s) {
    if (count <= 0) return AK_OK;
    const unsigned blocks = (unsigned)((count + kBlock - 1) / kBlock);
    switch (ak_dtype_size(out)) {
    case 2: { uint16_t v; memcpy(&v, value.b, 2); k_fill<uint16_t><<<blocks, kBlock, 0, s>>>((uint16_t*)dst, count, v); break; }
    case 4: { uint32_t v; memcpy(&v, value.b, 4); k_fill<uint32_t><<<blocks, kBlock, 0, s>>>((uint32_t*)dst, count, v); break; }
    case 8: { uint64_t v; memcpy(&v, value.b, 8); k_fill<uint64_t><<<blocks, kBlock, 0, s>>>((uint64_t*)dst, count, v); break; }
    case 16: { Mat2 v; memcpy(&v, value.b, 16); k_fill<Mat2><<<blocks, kBlock, 0, s>>>((Mat2*)dst, count, v); break; }
    default: return AK_ERR_UNSUPPORTED;
    }
    ak_status st = check_launch();
    if (st == AK_OK) count_launches(1);
    return st;
}

}  // namespace ak

extern "C" ak_status ak_dims_select(int64_t inner, int64_t red_len, int64_t outer, int elem_bytes,
                                    int vec_elems, int sm_count, int forced_shape, int32_t* shape_out,
                                    int32_t* tile_outputs, int32_t* row_groups, int32_t* split) {
    if (inner < 1 || red_len < 1 || outer < 1 || elem_bytes < 1 || vec_elems < 1 || sm_count < 1 ||
        forced_shape < AK_SHAPE_AUTO || forced_shape > AK_SHAPE_COLUMNS || vec_elems * elem_bytes > 16)
        return AK_ERR_INVALID_ARG;
    ak::DimsPlan p = {};
    ak::select_shape(inner, red_len, outer, elem_bytes, vec_elems, sm_count, forced_shape, false, true, &p);
    if (shape_out) *shape_out = p.shape;
    if (tile_outputs) *tile_outputs = p.tile_out;
    if (row_groups) *row_groups = p.row_groups;
    if (split) *split = p.split;
    return AK_OK;
}
