// k_cta.cu -- path 2 instantiations: a thread block per row, rows that may
// start or end inside a 16-byte vector.
#include "cta_launch.cuh"

namespace mbrs {

bool cta_shape_ok(int threads, int vpt) {
    const bool t = threads == 64 || threads == 128 || threads == 256 || threads == 512 || threads == 1024;
    return t && ((vpt >= 1 && vpt <= 5) || ((vpt == 6 || vpt == 8 || vpt == 10) && threads < 1024));
}

cudaError_t launch_cta(const LaunchArgs &a, int threads, int vpt, int64_t grid) {
    return a.whole ? launch_cta_whole(a, threads, vpt, grid) : cta_detail::launch<kPlainRows>(a, threads, vpt, grid);
}

}  // namespace mbrs
