// launch_block_scaled.cu -- the block-scaled instantiations of the persistent
// GEMM kernel (MXFP8, NVFP4, MXFP4), in a translation unit of their own.
#include "launch.cuh"

namespace tcg {

cudaError_t launch_block_scaled(const KernelParams& kp, const LaunchShape& ls, int bn, int katoms, int blk,
                                cudaStream_t stream, const char** what) {
    if (ls.cluster == 2) {
        if (blk == 2 && bn == 256)
            return katoms == 2 ? launch_instance<256, true, true, 2, 2>(kp, ls, stream, what)
                               : launch_instance<256, true, true, 1, 2>(kp, ls, stream, what);
        if (blk == 3 && bn == 192) return launch_instance<192, true, true, 2, 3>(kp, ls, stream, what);
        if (blk == 3 && bn == 256)
            return katoms == 2 ? launch_instance<256, true, true, 2, 3>(kp, ls, stream, what)
                               : launch_instance<256, true, true, 1, 3>(kp, ls, stream, what);
        if (blk == 1 && bn == 192) return launch_instance<192, true, true, 2, 1>(kp, ls, stream, what);
        if (blk == 1 && bn == 256)
            return katoms == 2 ? launch_instance<256, true, true, 2, 1>(kp, ls, stream, what)
                               : launch_instance<256, true, true, 1, 1>(kp, ls, stream, what);
    } else if (bn == 128) {
        if (blk == 2) return launch_instance<128, true, false, 1, 2>(kp, ls, stream, what);
        if (blk == 3) return launch_instance<128, true, false, 1, 3>(kp, ls, stream, what);
        if (blk == 1)
            return katoms == 2 ? launch_instance<128, true, false, 2, 1>(kp, ls, stream, what)
                               : launch_instance<128, true, false, 1, 1>(kp, ls, stream, what);
    }
    *what = "block-scaled tile shape";
    return cudaErrorInvalidValue;
}

}  // namespace tcg
