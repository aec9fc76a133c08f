// k_warp.cu -- path 1 instantiations: a lane group (2..32 lanes) per row,
// rows that may start or end inside a 16-byte vector.
#include "warp_launch.cuh"

namespace mbrs {

bool warp_shape_ok(int group, int vpt) {
    if (group == 2 || group == 4 || group == 8 || group == 16) return vpt >= 1 && vpt <= 8;
    return group == 32 && vpt >= 1 && vpt <= 9;
}

cudaError_t launch_warp(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid) {
    if (threads < 32 || threads > 256 || threads % 32 != 0) return cudaErrorInvalidValue;
    return a.whole ? launch_warp_whole(a, threads, group, vpt, grid)
                   : warp_detail::launch<kPlainRows>(a, threads, group, vpt, grid);
}

}  // namespace mbrs
