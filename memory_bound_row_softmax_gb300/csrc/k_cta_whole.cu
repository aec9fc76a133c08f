// k_cta_whole.cu -- path 2 instantiations for rows of whole 16-byte vectors
// (aligned rows: no edge tests in the loads and stores).
#include "cta_launch.cuh"

namespace mbrs {

cudaError_t launch_cta_whole(const LaunchArgs &a, int threads, int vpt, int64_t grid) {
    return cta_detail::launch<kWholeRows>(a, threads, vpt, grid);
}

}  // namespace mbrs
