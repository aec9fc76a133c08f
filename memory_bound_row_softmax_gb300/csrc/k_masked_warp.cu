// k_masked_warp.cu -- path 1 instantiations for scaled, causally masked rows
// (softmax_fwd_masked): a lane group per row reading only the kept columns.
#include "warp_launch.cuh"

namespace mbrs {

cudaError_t launch_warp_masked(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid) {
    if (threads < 32 || threads > 256 || threads % 32 != 0) return cudaErrorInvalidValue;
    return a.whole ? launch_warp_masked_whole(a, threads, group, vpt, grid)
                   : warp_detail::launch<kMaskedRows>(a, threads, group, vpt, grid);
}

}  // namespace mbrs
