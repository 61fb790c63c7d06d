// reduce.cu -- host side of the whole-array mapreduce: the plan (grid and
// workspace) and the dispatch of a call's types, operator, map and monoid to
// the kernels of reduce.cuh.
#include <algorithm>

#include "reduce.cuh"

namespace ak {

ak_status plan_reduce(int64_t n, ak_dtype in, ak_dtype acc, bool no_neutral, int target_blocks,
                      const DeviceInfo& dev, ReducePlan* plan) {
    const size_t psz = partial_size(acc, no_neutral);
    const size_t esz = ak_dtype_size(in);
    if (psz == 0 || esz == 0) return AK_ERR_UNSUPPORTED;
    red::plan_sizes(n, esz, psz, in == AK_MAT2_MODP, target_blocks, dev.sm_count, plan);
    return AK_OK;
}

// A fused two-source reduction: the map of two sources and the monoid.
static ak_status run_reduce2(const ReduceCall& c, const ReducePlan& plan) {
    return dispatch_types(c.in, c.acc, c.out, [&](auto ti, auto ta, auto to) -> ak_status {
        using In = typename decltype(ti)::type;
        using Acc = typename decltype(ta)::type;
        using Out = typename decltype(to)::type;
        if constexpr (is_mat2_v<Acc>) {
            return AK_ERR_UNSUPPORTED;
        } else {
            return dispatch_op<Acc>(c.op, [&](auto top) -> ak_status {
                using Op = typename decltype(top)::type;
                return dispatch_monoid<Op, Acc>(c.no_neutral, [&](auto tmo) -> ak_status {
                    using M = typename decltype(tmo)::type;
                    switch (c.map2) {
                    case AK_MAP2_MUL: return red::launch2<In, Acc, Out, Map2Mul, M>(c, plan);
                    case AK_MAP2_SQDIFF: return red::launch2<In, Acc, Out, Map2SqDiff, M>(c, plan);
                    case AK_MAP2_ABSDIFF: return red::launch2<In, Acc, Out, Map2AbsDiff, M>(c, plan);
                    default: return AK_ERR_UNSUPPORTED;
                    }
                });
            });
        }
    });
}

ak_status run_reduce(const ReduceCall& c, const ReducePlan& plan) {
    if (c.src2) return run_reduce2(c, plan);
    return dispatch_types(c.in, c.acc, c.out, [&](auto ti, auto ta, auto to) -> ak_status {
        using In = typename decltype(ti)::type;
        using Acc = typename decltype(ta)::type;
        using Out = typename decltype(to)::type;
        return dispatch_op<Acc>(c.op, [&](auto top) -> ak_status {
            using Op = typename decltype(top)::type;
            return dispatch_map<Acc>(c.f, [&](auto tm) -> ak_status {
                using Map = typename decltype(tm)::type;
                return dispatch_monoid<Op, Acc>(c.no_neutral, [&](auto tmo) -> ak_status {
                    using M = typename decltype(tmo)::type;
                    return red::launch<In, Acc, Out, Map, M>(c, plan);
                });
            });
        });
    });
}

}  // namespace ak
