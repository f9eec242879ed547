// launch_narrow.cu -- the pair-tile instantiations narrower than 256: the
// wave-fitting widths (256 x 160 / 192 / 224, K-major B) and the 256 x 128
// split-K tiles of tall, narrow problems, in a translation unit of their own.
#include "launch.cuh"

namespace tcg {

cudaError_t launch_narrow_pair(const KernelParams& kp, const LaunchShape& ls, int bn, bool fp8, cudaStream_t stream,
                               const char** what) {
    if (ls.cluster == 2) {
        switch (bn) {
            case 128:
                return fp8 ? launch_instance<128, true, true, 2>(kp, ls, stream, what)
                           : launch_instance<128, false, true, 2>(kp, ls, stream, what);
            case 160:
                return fp8 ? launch_instance<160, true, true, 2>(kp, ls, stream, what)
                           : launch_instance<160, false, true, 2>(kp, ls, stream, what);
            case 192:
                return fp8 ? launch_instance<192, true, true, 2>(kp, ls, stream, what)
                           : launch_instance<192, false, true, 2>(kp, ls, stream, what);
            case 224:
                return fp8 ? launch_instance<224, true, true, 2>(kp, ls, stream, what)
                           : launch_instance<224, false, true, 2>(kp, ls, stream, what);
            default:
                break;
        }
    }
    *what = "pair tile width";
    return cudaErrorInvalidValue;
}

}  // namespace tcg
