// launch_grouped.cu -- the grouped-GEMM instantiations of the persistent GEMM
// kernel, in a translation unit of their own.
#include "launch.cuh"

namespace tcg {

cudaError_t launch_grouped(const KernelParams& kp, const LaunchShape& ls, bool fp8, cudaStream_t stream,
                           const char** what) {
    if (ls.cluster == 2)
        return fp8 ? launch_instance<256, true, true, 2, 0, true>(kp, ls, stream, what)
                   : launch_instance<256, false, true, 2, 0, true>(kp, ls, stream, what);
    return fp8 ? launch_instance<256, true, false, 1, 0, true>(kp, ls, stream, what)
               : launch_instance<256, false, false, 1, 0, true>(kp, ls, stream, what);
}

}  // namespace tcg
