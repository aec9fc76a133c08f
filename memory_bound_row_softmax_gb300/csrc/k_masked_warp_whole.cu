// k_masked_warp_whole.cu -- path 1 instantiations for scaled, causally masked
// rows of whole 16-byte vectors (no edge tests but at the kept part's end).
#include "warp_launch.cuh"

namespace mbrs {

cudaError_t launch_warp_masked_whole(const LaunchArgs &a, int threads, int group, int vpt, int64_t grid) {
    return warp_detail::launch<kMaskedWholeRows>(a, threads, group, vpt, grid);
}

}  // namespace mbrs
