// k_masked_whole.cu -- path 2 instantiations for scaled, causally masked rows
// of whole 16-byte vectors (no edge tests but at the kept part's end).
#include "cta_launch.cuh"

namespace mbrs {

cudaError_t launch_cta_masked_whole(const LaunchArgs &a, int threads, int vpt, int64_t grid) {
    return cta_detail::launch<kMaskedWholeRows>(a, threads, vpt, grid);
}

}  // namespace mbrs
