// launch.cuh -- launching one instantiation of the persistent GEMM kernel.
//
// The kernel's instantiations are spread over translation units that nvcc
// compiles in parallel: the plain operand types (tcgemm_host.cu), the
// block-scaled types (launch_block_scaled.cu), the grouped GEMM
// (launch_grouped.cu), the narrower pair tiles (launch_narrow.cu) and the
// transposed-output tiles of the operand-swapped product (launch_swapped.cu).
// Each unit launches only the instantiations it holds; the host code reaches
// the others through the functions declared below.
#pragma once

#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "gemm_kernel.cuh"

namespace tcg {

struct LaunchShape {
    int grid;     // CTAs (a multiple of cluster)
    int smem;     // dynamic shared memory bytes
    int cluster;  // 1, or 2 for CTA pairs
};

constexpr int kMaxDynamicSmem = 232448;   // 227 KiB per block

template <int BN, bool kFp8, bool kCta2, int KA, int kBlk = 0, bool kGrouped = false, bool kTrans = false>
cudaError_t set_smem_attr() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(gemm_persistent_kernel<BN, kFp8, kCta2, KA, kBlk, kGrouped, kTrans>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynamicSmem);
        if (err == cudaSuccess && kCta2)
            err = cudaFuncSetAttribute(gemm_persistent_kernel<BN, kFp8, kCta2, KA, kBlk, kGrouped, kTrans>,
                                       cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    });
    return err;
}

// One launch; on failure *what names the call that failed.
template <int BN, bool kFp8, bool kCta2, int KA, int kBlk = 0, bool kGrouped = false, bool kTrans = false>
cudaError_t launch_instance(const KernelParams& kp, const LaunchShape& ls, cudaStream_t stream, const char** what) {
    cudaError_t e = set_smem_attr<BN, kFp8, kCta2, KA, kBlk, kGrouped, kTrans>();
    if (e != cudaSuccess) {
        *what = "cudaFuncSetAttribute";
        return e;
    }
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(ls.grid, 1, 1);
    cfg.blockDim = dim3(kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = ls.smem;
    cfg.stream = stream;
    if (kCta2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    e = cudaLaunchKernelEx(&cfg, gemm_persistent_kernel<BN, kFp8, kCta2, KA, kBlk, kGrouped, kTrans>, kp);
    if (e != cudaSuccess) *what = "cudaLaunchKernelEx";
    return e;
}

// Block-scaled operands (kBlk 1 = MXFP8, 2 = NVFP4, 3 = MXFP4): pairs with
// bn 256 (1 or 2 K atoms per stage) or 192 (MXFP8 / MXFP4, 2 atoms), or one
// CTA with bn 128.  cudaErrorInvalidValue for a combination not built.
cudaError_t launch_block_scaled(const KernelParams& kp, const LaunchShape& ls, int bn, int katoms, int blk,
                                cudaStream_t stream, const char** what);

// Pair tiles narrower than 256 (2 K atoms per stage) for 16-bit or 8-bit
// operands: 256 x 128 (split K, any B layout) and the wave-fitting 256 x 160
// / 192 / 224 (K-major B).  cudaErrorInvalidValue otherwise.
cudaError_t launch_narrow_pair(const KernelParams& kp, const LaunchShape& ls, int bn, bool fp8, cudaStream_t stream,
                               const char** what);

// Transposed-output tiles 128 x bn (bn 32 or 64, one CTA, one or two K atoms
// per stage) of the operand-swapped product D^T = B^T A^T, for GEMMs with at most
// 64 rows.  cudaErrorInvalidValue otherwise.
cudaError_t launch_swapped(const KernelParams& kp, const LaunchShape& ls, int bn, int katoms, bool fp8,
                           cudaStream_t stream, const char** what);

// Grouped GEMM: 256 x 256 pairs with 2 K atoms per stage, or 128 x 256 CTAs
// with 1, for 16-bit or 8-bit operands.
cudaError_t launch_grouped(const KernelParams& kp, const LaunchShape& ls, bool fp8, cudaStream_t stream,
                           const char** what);

}  // namespace tcg
