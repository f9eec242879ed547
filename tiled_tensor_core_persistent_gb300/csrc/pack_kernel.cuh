// pack_kernel.cuh -- the slow path for operands the TMA cannot address.
//
// A TMA tensor map needs a 16-byte aligned base and a row pitch that is a
// multiple of 16 bytes.  An operand stored with any other pointer or leading
// dimension (e.g. a tight bf16 row of 3001 elements) is first copied, once per
// call, into 16-byte pitched rows of the caller's workspace; the GEMM then
// streams the copy with the TMA as usual.  Of the two answers the alignment
// rule of "CUTLASS" (stanleyjacob.dev), Part II allows an unaligned tensor (a
// slower path, or a refusal), this is the slower path: one extra read and
// write of the operand at HBM bandwidth.
#pragma once

#include <cstdint>

namespace tcg {

// One matrix to pack: `rows` rows of `row_bytes` bytes each from src (row
// pitch src_pitch bytes, any alignment) to dst (row pitch dst_pitch bytes,
// every row 16-byte aligned).
struct PackJob {
    const uint8_t* src;
    long long src_pitch;
    uint8_t* dst;
    long long dst_pitch;
    long long rows;
    int row_bytes;
    int chunks;          // 16-byte chunks per destination row
    long long total;     // rows * chunks
};

// Up to two matrices (A and B) in one launch.  One thread moves one 16-byte
// chunk of a destination row: it reads the one or two aligned 16-byte source
// blocks that hold the chunk and funnel-shifts the bytes into place.  Each
// block read holds at least one byte of the chunk, so no read leaves the
// pages the operand occupies.  The last, partial chunk of a row is copied byte
// by byte.  Bytes of dst past row_bytes in each row are left as they were.
struct PackParams {
    PackJob job[2];
    int njobs;
};

__device__ __forceinline__ void pack_chunk(const PackJob& j, long long i) {
    long long r;
    int c;
    if (j.total <= 0x7fffffffLL) {
        const uint32_t ui = static_cast<uint32_t>(i), uc = static_cast<uint32_t>(j.chunks);
        r = ui / uc;
        c = static_cast<int>(ui - static_cast<uint32_t>(r) * uc);
    } else {
        r = i / j.chunks;
        c = static_cast<int>(i - r * j.chunks);
    }
    const uint8_t* s = j.src + r * j.src_pitch + static_cast<long long>(c) * 16;
    uint8_t* d = j.dst + r * j.dst_pitch + static_cast<long long>(c) * 16;
    const int n = j.row_bytes - c * 16;
    if (n >= 16) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(s);
        const int off = static_cast<int>(a & 15u);
        const uint4* blk = reinterpret_cast<const uint4*>(a - static_cast<uintptr_t>(off));
        const uint4 q0 = __ldg(blk);
        uint4 out = q0;
        if (off != 0) {
            const uint4 q1 = __ldg(blk + 1);
            const uint32_t sh = static_cast<uint32_t>(off & 3) * 8u;
            uint32_t v0, v1, v2, v3, v4;
            switch (off >> 2) {
                case 0: v0 = q0.x; v1 = q0.y; v2 = q0.z; v3 = q0.w; v4 = q1.x; break;
                case 1: v0 = q0.y; v1 = q0.z; v2 = q0.w; v3 = q1.x; v4 = q1.y; break;
                case 2: v0 = q0.z; v1 = q0.w; v2 = q1.x; v3 = q1.y; v4 = q1.z; break;
                default: v0 = q0.w; v1 = q1.x; v2 = q1.y; v3 = q1.z; v4 = q1.w; break;
            }
            out.x = __funnelshift_r(v0, v1, sh);
            out.y = __funnelshift_r(v1, v2, sh);
            out.z = __funnelshift_r(v2, v3, sh);
            out.w = __funnelshift_r(v3, v4, sh);
        }
        *reinterpret_cast<uint4*>(d) = out;
    } else {
        for (int b = 0; b < n; ++b) d[b] = s[b];
    }
}

__global__ void __launch_bounds__(256) pack_rows_kernel(const __grid_constant__ PackParams p) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long t0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (long long i = t0; i < p.job[0].total; i += stride) pack_chunk(p.job[0], i);
    if (p.njobs > 1)
        for (long long i = t0; i < p.job[1].total; i += stride) pack_chunk(p.job[1], i);
}

}  // namespace tcg
