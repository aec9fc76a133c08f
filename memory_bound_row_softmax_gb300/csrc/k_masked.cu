// k_masked.cu -- path 2 instantiations for scaled, causally masked rows
// (softmax_fwd_masked): a block per row reading only the kept columns.
#include "cta_launch.cuh"

namespace mbrs {

cudaError_t launch_cta_masked(const LaunchArgs &a, int threads, int vpt, int64_t grid) {
    return a.whole ? launch_cta_masked_whole(a, threads, vpt, grid) : cta_detail::launch<kMaskedRows>(a, threads, vpt, grid);
}

}  // namespace mbrs
