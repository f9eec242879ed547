// launch_swapped.cu -- the transposed-output instantiations of the persistent
// GEMM kernel (one-CTA 128 x 32 / 128 x 64 tiles of D^T = B^T A^T for GEMMs
// with at most 64 rows, one or two K atoms per stage), in a translation unit
// of their own.
#include "launch.cuh"

namespace tcg {

cudaError_t launch_swapped(const KernelParams& kp, const LaunchShape& ls, int bn, int katoms, bool fp8,
                           cudaStream_t stream, const char** what) {
    if (ls.cluster == 1 && katoms == 2) {
        if (bn == 32)
            return fp8 ? launch_instance<32, true, false, 2, 0, false, true>(kp, ls, stream, what)
                       : launch_instance<32, false, false, 2, 0, false, true>(kp, ls, stream, what);
        if (bn == 64)
            return fp8 ? launch_instance<64, true, false, 2, 0, false, true>(kp, ls, stream, what)
                       : launch_instance<64, false, false, 2, 0, false, true>(kp, ls, stream, what);
    }
    if (ls.cluster == 1 && katoms == 1) {
        if (bn == 32)
            return fp8 ? launch_instance<32, true, false, 1, 0, false, true>(kp, ls, stream, what)
                       : launch_instance<32, false, false, 1, 0, false, true>(kp, ls, stream, what);
        if (bn == 64)
            return fp8 ? launch_instance<64, true, false, 1, 0, false, true>(kp, ls, stream, what)
                       : launch_instance<64, false, false, 1, 0, false, true>(kp, ls, stream, what);
    }
    *what = "transposed-output tile width";
    return cudaErrorInvalidValue;
}

}  // namespace tcg
