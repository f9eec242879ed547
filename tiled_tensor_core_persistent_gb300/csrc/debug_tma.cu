// debug_tma.cu -- test-only: the round trip of one TMA load with 128-byte
// swizzling into shared memory and back, so that the host model of the
// swizzle (which the source pages do not give; the GEMM kernel's shared-memory
// descriptors assume it) can be checked against the hardware.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/tcgemm.h"
#include "ptx.cuh"

namespace {

constexpr int kMaxRows = 64;                    // 8 KiB: 64 rows of 128 bytes
constexpr long long kWaitNs = 1000000000LL;     // 1 s

// One CTA: TMA-load the whole box, wait (bounded), copy shared memory out as is.
__global__ void tma_roundtrip_kernel(const __grid_constant__ CUtensorMap map, uint8_t* dst, int rows,
                                     int* status) {
    extern __shared__ uint8_t raw[];
    uint8_t* tile = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar;
    __shared__ int landed;
    if (threadIdx.x == 0) {
        tcg::ptx::mbar_init(&bar, 1);
        tcg::ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        tcg::ptx::mbar_arrive_expect_tx(&bar, static_cast<uint32_t>(rows) * 128u);
        tcg::ptx::tma_load_2d(tile, &map, &bar, 0, 0);
        // Bounded wait; if it runs out, flag it and wait once more (also
        // bounded) so that no copy is left writing this CTA's shared memory.
        bool ok = false;
        for (int round = 0; round < 2 && !ok; ++round) {
            const uint64_t t0 = tcg::ptx::globaltimer_ns();
            while (!(ok = tcg::ptx::mbar_try_wait(tcg::ptx::smem_u32(&bar), 0))) {
                if (static_cast<long long>(tcg::ptx::globaltimer_ns() - t0) > kWaitNs) break;
            }
            if (!ok && round == 0) *status = TCG_ERR_TIMEOUT;
        }
        landed = ok ? 1 : 0;
    }
    __syncthreads();
    if (!landed) return;
    for (int i = threadIdx.x; i < rows * 128; i += blockDim.x) dst[i] = tile[i];
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

extern "C" tcg_status tcg_debug_tma_swizzle128(const void* src, int rows, void* dst, int* status, void* stream) {
    if (!src || !dst || !status || rows < 1 || rows > kMaxRows) return TCG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) || (reinterpret_cast<uintptr_t>(dst) & 15u)) return TCG_ERR_MISALIGNED;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !f)
        return TCG_ERR_LAUNCH;
    CUtensorMap map;
    const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(rows)};
    const cuuint32_t estr[2] = {1, 1};
    if (reinterpret_cast<EncodeFn>(f)(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(src), dims, strides,
                                      box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                      CU_TENSOR_MAP_L2_PROMOTION_NONE,
                                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return TCG_ERR_LAUNCH;
    tma_roundtrip_kernel<<<1, 128, 1024 + kMaxRows * 128, static_cast<cudaStream_t>(stream)>>>(
        map, static_cast<uint8_t*>(dst), rows, status);
    return cudaGetLastError() == cudaSuccess ? TCG_OK : TCG_ERR_LAUNCH;
}
