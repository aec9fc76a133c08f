// k_warp_whole.cu -- path 1 instantiations for rows of whole 16-byte vectors
// (aligned rows: no edge tests in the loads and stores).
#include "warp_launch.cuh"

namespace mbrs {

cudaError_t launch_warp_whole(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid) {
    return warp_detail::launch<kWholeRows>(a, threads, group, vpt, grid);
}

}  // namespace mbrs
