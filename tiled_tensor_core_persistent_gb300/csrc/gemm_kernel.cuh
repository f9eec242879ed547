// gemm_kernel.cuh -- the persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   D = act(alpha * (A @ B) + beta * C + bias)      (alpha already holds sA*sB)
//
// Structure (the reference pages describe the Hopper/Ampere ancestors; this is
// the Blackwell re-design):
//   * CTA tile BM x BN over D (BM = 128 = TMEM lanes), streamed over K in
//     k-blocks of one 128-byte swizzle row ("CUTLASS", Part I tile hierarchy
//     and Part IV Stage 4 mainloop).
//   * Warp 0, one thread: TMA producer.  Per k-block it waits for a free
//     stage, arms the stage's full barrier with the byte count and issues the
//     A and B box loads (128-byte swizzled shared memory).
//   * Warp 1, one thread: MMA issuer.  Per k-block it waits for the stage,
//     issues BK/MMA_K tcgen05.mma into a TMEM accumulator, and commits the
//     stage back to the producer.  Warp 1 also owns TMEM allocation.
//   * Warps 2-5: epilogue.  TMEM -> registers (tcgen05.ld), alpha / beta*C /
//     bias / activation in fp32, cast, then each thread stores its row of
//     the chunk straight from registers (32-byte stores where D allows); a
//     ragged last chunk goes into a swizzled staging tile in shared memory
//     and out through a TMA store (out-of-range columns clipped by the
//     hardware).
//   * Two TMEM accumulators: the epilogue of tile i overlaps the mainloop of
//     tile i+1 (the idea behind the ping-pong schedule, "CUTLASS", Part V
//     deep dive on collective builder and kernel schedules).
//   * Persistent static schedule with grouped rasterisation ("CUTLASS",
//     Part IV Stage 2: swizzle the tile-to-block mapping for L2 reuse).
//   * Split-K: each (tile, split) unit writes an fp32 partial; the last unit
//     to arrive sums the partials in split order and runs the epilogue
//     ("CUTLASS", Part IV Stage 6).
//   * Every wait is bounded; on expiry the CTA records TCG_ERR_TIMEOUT in the
//     status word, drains its in-flight copies, frees TMEM and returns.
//   * The debug build (TCG_DEBUG_CHECKS defined) adds device-side checks of
//     the pipeline bookkeeping: stage, accumulator, epilogue-buffer, TMEM
//     column, partial-slot and counter indices in range, every decoded unit
//     inside the tile grid, and after every mbarrier wait that the phase
//     after the awaited one has not completed too (a consumer and a producer
//     out of step by two phases).  A failed check records TCG_ERR_CHECK with
//     its code and the block in the status word and ends the CTA the way a
//     timeout does: no trap.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace tcg {

constexpr int kBM = 128;              // rows per CTA tile = TMEM lanes
constexpr int kRowBytes = 128;        // one k-block = one 128-byte swizzle row
constexpr int kNumThreads = 192;      // 6 warps
constexpr int kEpiWarp0 = 2;          // epilogue warps 2..5
constexpr int kEpiThreads = 128;
constexpr int kEpiChunk = 32;         // columns per tcgen05.ld / TMA store box
constexpr int kEpiWarpBytes = 8192;   // per epilogue warp: 2 or 4 chunk buffers
constexpr int kEpiBytes = 4 * kEpiWarpBytes;
// Block-scaled pair tiles keep half of that (one or two buffers per warp), so
// that three stages of two K atoms fit next to it.
constexpr int kEpiWarpBytesSmall = 4096;
__host__ __device__ constexpr int epi_warp_bytes(bool small) { return small ? kEpiWarpBytesSmall : kEpiWarpBytes; }
constexpr int kStatusTimeout = 7;     // == TCG_ERR_TIMEOUT
constexpr int kStatusCheck = 8;       // == TCG_ERR_CHECK

#ifdef TCG_DEBUG_CHECKS
constexpr bool kChecks = true;
#else
constexpr bool kChecks = false;
#endif

// Codes of the debug build's checks (status word [1] after TCG_ERR_CHECK).
enum : int {
    kChkStage = 101,        // pipeline stage index outside [0, stages) or stages > 16
    kChkPhase = 102,        // the phase after an awaited mbarrier phase had completed as well
    kChkAcc = 103,          // TMEM accumulator index outside the accumulators
    kChkTmemCols = 104,     // accumulator columns outside the TMEM allocation
    kChkScaleCols = 105,    // block-scale columns outside the TMEM allocation
    kChkSlot = 106,         // split-K / Stream-K partial slot outside the workspace's slots
    kChkCounter = 107,      // tile arrival counter outside the workspace's counters
    kChkUnit = 108,         // decoded unit outside the tile grid or K range
    kChkRing = 109,         // epilogue buffer index outside the warp's ring
    kChkForced = 199        // the test knob (fault_inject = 2) failed a check on purpose
};

struct KernelParams {
    CUtensorMap tmA;
    CUtensorMap tmB;
    CUtensorMap tmD;
    CUtensorMap tmC;      // C as 32 x 32 boxes (when c_tma)
    CUtensorMap tmSFA;    // block scales as rows of 128 x 32-bit words (one 512-byte block each), pair tiles
    CUtensorMap tmSFB;
    CUtensorMap tmB2;     // B in boxes of half the rows, for the half-width tail units (K-major B)
    int M, N, K;
    int num_m_blk, num_n_blk, num_kb;
    // Work, in two phases.  Data-parallel: units [0, units_a) over tiles
    // [0, units_a / splits), each tile split into `splits` equal K ranges,
    // unit u on worker u mod workers.  Stream-K: the next sk_tiles tiles as
    // one run of sk_iters = sk_tiles * num_kb k-block iterations, worker w
    // taking iterations [w * sk_iters / workers, (w + 1) * sk_iters / workers)
    // across tile boundaries; a tile shared by several workers is finished by
    // the last of them to arrive.  (A worker is a CTA, or a CTA pair.)
    int splits, num_units, group_m;
    int units_a;
    int sk_tiles;
    long long sk_iters;
    int sk_slot_base;     // first partial slot of the Stream-K phase (2 per worker)
    int half_tail;        // last tiles run as two half-width units each (decode_unit)
    int k_serp;           // odd waves walk K downwards (work_next)
    int a_mn_major, b_mn_major;
    float alpha, beta;
    const void* C;
    long long ldc;
    int c_f32;
    const void* bias;
    int bias_f32;
    int act;
    int d_f32;
    void* D;              // row-major output, for the ragged column tail
    long long ldd;
    int d_inner_aligned;  // N * sizeof(D element) is a multiple of 16 bytes
    int d_v32;            // D's base and row pitch are multiples of 32 bytes (32-byte register stores)
    int d_tma;            // D has a TMA store map (16-byte aligned base and row pitch)
    int d_stage_all;      // every chunk of D staged in shared memory and stored by TMA (else registers -> global)
    int c_vec;            // C rows may be read with 16-byte vector loads
    int c_tma;            // C is read through tmC into the epilogue buffers
    int epi_nbuf;         // epilogue buffers per warp (2 or 4, 8 KiB in all)
    int cs_vec;           // col_scale may be read with 16-byte vector loads
    int stages;
    float* partials;      // split-K partials: [slot * ranks + rank][BN][kBM] (row fastest), slot from partial_slot()
    int* tile_counters;   // split-K arrival counters [tile * ranks + rank]
    int* status;          // [0] status, [1] where, [2] block
    int num_slots;        // partial slots in the workspace (debug-build checks)
    int num_counters;     // tile arrival counters in the workspace (debug-build checks)
    long long timeout_ns;
    int fault_inject;
    unsigned long long* stats;  // optional cycle accounting (nullptr = off), see kStat*
    uint32_t ab_fmt;            // operand format field of the instruction descriptor
    const float* row_scale;     // optional dequantisation scale per output row (M)
    const float* col_scale;     // optional dequantisation scale per output column (N)
    // Block scale factors, in 512-byte blocks of 128 rows x 4 scales: block
    // (row block rb, column block cb) at (rb * num_sfcb + cb) * 512.  Used by
    // the block-scaled kernels only.
    const uint8_t* sfa;
    const uint8_t* sfb;
    int num_sfcb;               // 4-scale column blocks per row (ceil(ceil(K / block) / 4))
    // Grouped GEMM (the kGrouped kernels): num_groups independent problems,
    // each with a complete parameter block of its own in global memory (its
    // tensor maps, sizes, pointers and tile grid); problem g owns the units
    // [group_tile0[g], group_tile0[g + 1]) of the launch.
    const KernelParams* group;
    const int* group_tile0;
    int num_groups;
};


// Cycle accounting slots (summed over CTAs) when KernelParams::stats is set.
enum : int {
    kStatMmaWaitFull = 0,     // MMA issuer waiting for loaded stages
    kStatMmaWaitAcc = 1,      // MMA issuer waiting for a free accumulator
    kStatProdWaitEmpty = 2,   // producer waiting for a free stage
    kStatEpiWaitFull = 3,     // epilogue (warp 2) waiting for a finished accumulator
    kStatEpiBusy = 4,         // epilogue (warp 2) from accumulator ready to hand-back
    kStatMmaTotal = 5,        // MMA issuer loop, first wait to last commit
    kStatCtas = 6,
    kNumStats = 8
};

// Shared-memory bookkeeping that lives after the operand stages.
struct alignas(16) SmemCtl {
    uint64_t full[16];
    uint64_t empty[16];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint64_t cbar[4][4];  // per epilogue warp, per buffer: C chunk landed
    uint32_t tmem_base;
    int abort_flag;
    int splitk_last;
    alignas(16) float bias_tile[256];  // the current tile's bias (fp32), shared by the epilogue warps
};

__device__ __forceinline__ void record_timeout(const KernelParams& p, int where) {
    if (atomicCAS(p.status, 0, kStatusTimeout) == 0) {
        p.status[1] = where;
        p.status[2] = static_cast<int>(blockIdx.x);
    }
}

// Debug build: record a failed check (TCG_ERR_CHECK, its code, the block),
// make the CTA's other roles give up at their next wait, and return false.
// Release build: always true (the condition is never evaluated for effect).
// Called by whole (converged) warps; the outcome is the warp's.
__device__ __forceinline__ bool dcheck(bool cond, const KernelParams& p, SmemCtl* ctl, int where) {
    if constexpr (kChecks) {
        if (!__all_sync(0xffffffffu, cond)) {
            if ((threadIdx.x & 31) == 0 && atomicCAS(p.status, 0, kStatusCheck) == 0) {
                p.status[1] = where;
                p.status[2] = static_cast<int>(blockIdx.x);
            }
            *reinterpret_cast<volatile int*>(&ctl->abort_flag) = 1;
            return false;
        }
    }
    return true;
}

// Debug build: after a wait on `parity` of a barrier returned, the next phase
// must still be open (its completion needs an action of the waiting role).
__device__ __forceinline__ bool dcheck_phase(uint64_t* bar, uint32_t parity, const KernelParams& p, SmemCtl* ctl) {
    if constexpr (kChecks) return dcheck(!ptx::mbar_test_wait(ptx::smem_u32(bar), parity ^ 1u), p, ctl, kChkPhase);
    return true;
}

// Bounded wait on an mbarrier phase.  Returns false (and flags the CTA) when
// the limit passes or, if honor_abort, another role of this CTA already gave
// up.  Drain waits pass honor_abort = false: they must see their own copies
// land even after an abort, and are still bounded by the limit.
static __device__ __noinline__ bool wait_phase(uint64_t* bar, uint32_t parity, const KernelParams& p,
                                        SmemCtl* ctl, int where, long long limit_ns,
                                        bool honor_abort = true) {
    const uint32_t a = ptx::smem_u32(bar);
    if (ptx::mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    uint32_t n = 0;
    while (true) {
        if (ptx::mbar_try_wait(a, parity)) return true;
        if ((++n & 31u) == 0) {
            if (honor_abort && *reinterpret_cast<volatile int*>(&ctl->abort_flag)) return false;
            if (static_cast<long long>(ptx::globaltimer_ns() - t0) > limit_ns) {
                *reinterpret_cast<volatile int*>(&ctl->abort_flag) = 1;
                record_timeout(p, where);
                return false;
            }
        }
    }
}

// The whole warp waits (converged), then agrees on the outcome.  Role warps
// run their loops with all 32 lanes and let lane 0 issue, so no lane of a
// role warp ever sits at a CTA-wide barrier while its siblings spin.
// inline_first: test the phase inline first and call the bounded wait only
// when it has not completed.  Measured on GB300 (same GPU, median of 40
// launches): the pair-tile kernels gain from it (8192^3 GELU 613.0 -> 590.4
// us, 4096^3 beta=1 102.7 -> 96.7 us), the one-CTA split-K kernel of 16 x
// 8192 x 8192 loses (39.4 -> 41.5 us), so the kernels pass kCta2.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const KernelParams& p, SmemCtl* ctl,
                                          int where, long long limit_ns, bool honor_abort = true,
                                          bool inline_first = false) {
    bool ok = inline_first && ptx::mbar_try_wait(ptx::smem_u32(bar), parity);
    if (!ok) ok = wait_phase(bar, parity, p, ctl, where, limit_ns, honor_abort);
    return __all_sync(0xffffffffu, ok);
}

// One unit of work: output tile (m_blk, n_blk), its K range [kb0, kb1) in
// k-blocks, and its place among the nsplit pieces of the tile (split).
// Data-parallel units: slot_tile = first partial slot of the tile's splits.
// Stream-K pieces: sk = 1, tl = tile index within the Stream-K run,
// w_first = first worker holding a piece of the tile.
struct Unit {
    int m_blk, n_blk, tile, split, nsplit, kb0, kb1, slot_tile;
    int sk, tl, w_first;
    int g;   // problem of a grouped GEMM (0 otherwise)
    int nh;  // 0: the whole tile; 1 / 2: its first / second half of BN / 2 columns (the tail)
    int rev; // walk the K range downwards (every other wave, when KernelParams::k_serp)
};

// A unit's first column and width.
__host__ __device__ __forceinline__ int unit_n0(const Unit& w, int bn) { return w.n_blk * bn + (w.nh == 2 ? bn / 2 : 0); }
__host__ __device__ __forceinline__ int unit_bn(const Unit& w, int bn) { return w.nh ? bn / 2 : bn; }

// Tile index -> (m_blk, n_blk) in the grouped raster order: groups of
// group_m block rows, column-major inside a group ("CUTLASS", Part IV
// Stage 2: swizzled tile order for L2 reuse).
__host__ __device__ __forceinline__ void tile_coords(const KernelParams& p, int tile, int& m_blk, int& n_blk) {
    const int span = p.group_m * p.num_n_blk;
    const int gid = tile / span;
    const int first_m = gid * p.group_m;
    const int gsz = p.num_m_blk - first_m < p.group_m ? p.num_m_blk - first_m : p.group_m;
    const int local = tile - gid * span;
    m_blk = first_m + local % gsz;
    n_blk = local / gsz;
}

// Units [units_a, units_a + 2 * half_tail) of an unsplit launch are the
// last half_tail tiles in raster order, each run as two units of half the
// tile's columns: a last wave of tiles that would fill at most half of the
// workers fills them with half tiles instead, and ends in half the time.
__host__ __device__ __forceinline__ Unit decode_unit(const KernelParams& p, int u) {
    Unit w;
    w.nh = 0;
    w.rev = 0;
    if (p.half_tail > 0 && u >= p.units_a) {
        const int hu = u - p.units_a;
        w.tile = p.units_a + hu / 2;
        w.nh = 1 + (hu & 1);
        w.split = 0;
        w.nsplit = 1;
        w.slot_tile = w.tile;
        w.sk = w.tl = w.w_first = w.g = 0;
        tile_coords(p, w.tile, w.m_blk, w.n_blk);
        w.kb0 = 0;
        w.kb1 = p.num_kb;
        return w;
    }
    w.tile = u / p.splits;
    w.split = u - w.tile * p.splits;
    w.nsplit = p.splits;
    w.slot_tile = w.tile * p.splits;
    w.sk = 0;
    w.tl = 0;
    w.w_first = 0;
    w.g = 0;
    tile_coords(p, w.tile, w.m_blk, w.n_blk);
    w.kb0 = static_cast<int>((static_cast<long long>(w.split) * p.num_kb) / w.nsplit);
    w.kb1 = static_cast<int>((static_cast<long long>(w.split + 1) * p.num_kb) / w.nsplit);
    return w;
}

// Stream-K bookkeeping: first iteration of worker w, and the worker that
// holds iteration i (the largest w with sk_begin(w) <= i).
__host__ __device__ __forceinline__ long long sk_begin(const KernelParams& p, int w, int workers) {
    return static_cast<long long>(w) * p.sk_iters / workers;
}
__host__ __device__ __forceinline__ int sk_worker_of(const KernelParams& p, long long i, int workers) {
    return static_cast<int>(((i + 1) * workers - 1) / p.sk_iters);
}

// Partial slot of piece q of the unit's tile.  Stream-K: each worker owns two
// slots, one for the piece in the tile where its range starts and one for the
// piece in the tile where it ends (the only pieces that can be partial).
__host__ __device__ __forceinline__ int partial_slot(const KernelParams& p, const Unit& w, int q, int workers) {
    if (!w.sk) return w.slot_tile + q;
    const int c = w.w_first + q;
    const bool starts_here = sk_begin(p, c, workers) >= static_cast<long long>(w.tl) * p.num_kb;
    return p.sk_slot_base + 2 * c + (starts_here ? 0 : 1);
}

// The sequence of units of one worker: its data-parallel units, then its
// Stream-K pieces.  Every role of a CTA walks the same sequence.
struct WorkIter {
    int u;             // next data-parallel unit
    long long it;      // next Stream-K iteration
    long long it_end;
    int wid, workers;
};

__host__ __device__ __forceinline__ WorkIter work_begin(const KernelParams& p, int wid, int workers) {
    WorkIter s;
    s.u = wid;
    s.wid = wid;
    s.workers = workers;
    s.it = s.it_end = 0;
    if (p.sk_tiles > 0) {
        s.it = sk_begin(p, wid, workers);
        s.it_end = sk_begin(p, wid + 1, workers);
    }
    return s;
}

__host__ __device__ __forceinline__ bool work_next(const KernelParams& p, WorkIter& s, Unit& w) {
    if (s.u < p.num_units) {
        w = decode_unit(p, s.u);
        // K-serpentine: the workers' odd waves of units walk K downwards, so a
        // wave starts on the K slabs the previous wave loaded last (most
        // likely still in L2) when it revisits the same rows of A
        w.rev = p.k_serp && ((s.u / s.workers) & 1);
        s.u += s.workers;
        return true;
    }
    if (s.it >= s.it_end) return false;
    const int tl = static_cast<int>(s.it / p.num_kb);
    w.sk = 1;
    w.tl = tl;
    w.g = 0;
    w.nh = 0;
    w.rev = 0;
    w.tile = p.units_a / p.splits + tl;
    tile_coords(p, w.tile, w.m_blk, w.n_blk);
    w.kb0 = static_cast<int>(s.it - static_cast<long long>(tl) * p.num_kb);
    const long long rest = w.kb0 + (s.it_end - s.it);
    w.kb1 = static_cast<int>(rest < p.num_kb ? rest : static_cast<long long>(p.num_kb));
    w.w_first = sk_worker_of(p, static_cast<long long>(tl) * p.num_kb, s.workers);
    const int w_last = sk_worker_of(p, static_cast<long long>(tl + 1) * p.num_kb - 1, s.workers);
    w.nsplit = w_last - w.w_first + 1;
    w.split = s.wid - w.w_first;
    w.slot_tile = 0;
    s.it += w.kb1 - w.kb0;
    return true;
}

// Grouped GEMM ("CUTLASS" page, Part V: a mixture-of-experts layer as a
// grouped GEMM, one problem per expert, of different shapes): the launch's
// units are the tiles of every problem, problem after problem; a worker takes
// every workers-th unit, finds its problem by binary search over the first
// units, and decodes the tile in that problem's own grid and raster.
template <bool kGrouped>
__device__ __forceinline__ bool next_unit(const KernelParams& p, WorkIter& s, Unit& w) {
    if constexpr (!kGrouped) {
        return work_next(p, s, w);
    } else {
        if (s.u >= p.num_units) return false;
        const int u = s.u;
        s.u += s.workers;
        int lo = 0, hi = p.num_groups - 1;   // the last problem whose first unit is <= u
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.group_tile0 + mid) <= u) lo = mid;
            else hi = mid - 1;
        }
        w = decode_unit(p.group[lo], u - __ldg(p.group_tile0 + lo));
        w.g = lo;
        return true;
    }
}

// The parameters of a unit's problem: the launch's own, or its problem's block.
template <bool kGrouped>
__device__ __forceinline__ const KernelParams& unit_params(const KernelParams& p, const Unit& w) {
    if constexpr (kGrouped) return p.group[w.g];
    else return p;
}


// erf(z) for z >= 0 by Abramowitz & Stegun, Handbook of Mathematical
// Functions, formula 7.1.26: 1 - (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5)
// exp(-z^2), t = 1 / (1 + p z), |error| <= 1.5e-7; odd extension for z < 0.
// Exact-erf GELU = 0.5 x (1 + erf(x / sqrt 2)).
__device__ __forceinline__ float gelu_erf(float x) {
    const float z = x * 0.70710678118654752f;
    const float a = fabsf(z);
    const float t = __fdividef(1.0f, fmaf(0.3275911f, a, 1.0f));
    float q = fmaf(1.061405429f, t, -1.453152027f);
    q = fmaf(q, t, 1.421413741f);
    q = fmaf(q, t, -0.284496736f);
    q = fmaf(q, t, 0.254829592f);
    q *= t;
    float e;  // exp(-a^2) = 2^(-a^2 log2 e)
    asm("ex2.approx.f32 %0, %1;" : "=f"(e) : "f"(-a * a * 1.44269504088896341f));
    const float erf_z = copysignf(fmaf(-q, e, 1.0f), z);
    const float hx = 0.5f * x;
    return fmaf(hx, erf_z, hx);
}

// The same GELU on a packed pair of fp32 values: the polynomial and the
// linear steps run as f32x2 instructions, the reciprocal and 2^x per lane.
__device__ __forceinline__ uint64_t gelu_erf2(uint64_t x) {
    constexpr uint64_t kSign = 0x8000000080000000ull;
    auto splat = [](float f) { return ptx::pack2(f, f); };
    const uint64_t z = ptx::mul2(x, splat(0.70710678118654752f));
    const uint64_t a = z & ~kSign;
    float d0, d1;
    ptx::unpack2(ptx::fma2(splat(0.3275911f), a, splat(1.0f)), d0, d1);
    const uint64_t t = ptx::pack2(ptx::rcp_approx(d0), ptx::rcp_approx(d1));
    uint64_t q = ptx::fma2(splat(1.061405429f), t, splat(-1.453152027f));
    q = ptx::fma2(q, t, splat(1.421413741f));
    q = ptx::fma2(q, t, splat(-0.284496736f));
    q = ptx::fma2(q, t, splat(0.254829592f));
    q = ptx::mul2(q, t);
    float m0, m1;
    ptx::unpack2(ptx::mul2(ptx::mul2(a, a), splat(-1.44269504088896341f)), m0, m1);
    const uint64_t e = ptx::pack2(ptx::ex2_approx(m0), ptx::ex2_approx(m1));
    const uint64_t erf_abs = ptx::fma2(q ^ kSign, e, splat(1.0f));
    const uint64_t erf_z = erf_abs | (z & kSign);
    const uint64_t hx = ptx::mul2(x, splat(0.5f));
    return ptx::fma2(hx, erf_z, hx);
}

__device__ __forceinline__ float apply_act(int act, float x) {
    if (act == 1) return x > 0.0f ? x : 0.0f;
    if (act == 2) return gelu_erf(x);
    return x;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

// Load 32 consecutive elements of a row-major bf16/f32 row, columns
// [col0, col0+32) clipped to n_valid, into fp32 registers (0 outside).
// vec: the row start is 16-byte aligned, so whole chunks use 16-byte loads.
__device__ __forceinline__ void load_row32(const void* base, int is_f32, int col0, int n_valid,
                                           float (&out)[32], bool vec = true) {
    if (is_f32) {
        const float* src = static_cast<const float*>(base) + col0;
        if (vec && col0 + 32 <= n_valid) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 v = *reinterpret_cast<const float4*>(src + 4 * q);
                out[4 * q + 0] = v.x; out[4 * q + 1] = v.y;
                out[4 * q + 2] = v.z; out[4 * q + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) out[i] = (col0 + i < n_valid) ? src[i] : 0.0f;
        }
    } else {
        const uint16_t* src = static_cast<const uint16_t*>(base) + col0;
        if (vec && col0 + 32 <= n_valid) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 v = *reinterpret_cast<const uint4*>(src + 8 * q);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    out[8 * q + 2 * h + 0] = bf16_bits_to_float(w[h] & 0xFFFFu);
                    out[8 * q + 2 * h + 1] = bf16_bits_to_float(w[h] >> 16);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                out[i] = (col0 + i < n_valid) ? bf16_bits_to_float(src[i]) : 0.0f;
        }
    }
}

// C prefetch: the raw bytes of one thread's 32-column C chunk are loaded one
// chunk ahead (and the first chunk before the accumulator is ready), so the
// load latency hides behind the TMEM read and the math.  The loads are whole
// aligned 16-byte blocks: the block holding the chunk's first byte and the
// ones after it up to the block holding its last byte (4 or 5 blocks for
// bf16, 8 or 9 for fp32; the extra block only when the row segment does not
// start on a 16-byte boundary, i.e. when ldc * sizeof(C) is not a multiple of
// 16).  Every block loaded holds at least one byte of the chunk.  Full chunks
// only; a ragged last chunk is loaded element-wise when used.
__device__ __forceinline__ uintptr_t c_chunk_addr(const KernelParams& p, int row, int col0) {
    return reinterpret_cast<uintptr_t>(p.C) +
           static_cast<uintptr_t>((static_cast<long long>(row) * p.ldc + col0) * (p.c_f32 ? 4 : 2));
}

// L2 prefetch of one thread's C row segment of a whole tile, columns
// [col0, min(col0 + ncols, N)): every 128-byte line that holds a byte of it.
// Issued a tile ahead, so the epilogue's C loads hit L2 instead of DRAM.
__device__ __forceinline__ void c_prefetch_l2(const KernelParams& p, int row, int col0, int ncols) {
    if (row >= p.M || col0 >= p.N) return;
    const int eb = p.c_f32 ? 4 : 2;
    const uintptr_t s = c_chunk_addr(p, row, col0);
    const uintptr_t e = s + static_cast<uintptr_t>(min(ncols, p.N - col0) * eb);
    for (uintptr_t a = s & ~static_cast<uintptr_t>(127); a < e; a += 128)
        ptx::prefetch_l2(reinterpret_cast<const void*>(a));
}

__device__ __forceinline__ void c_prefetch(const KernelParams& p, int row, int col0, uint4 (&q)[9]) {
    if (col0 + 32 > p.N) return;
    const uintptr_t s = c_chunk_addr(p, row, col0);
    const uint4* blk = reinterpret_cast<const uint4*>(s & ~static_cast<uintptr_t>(15));
    const bool extra = !p.c_vec && (s & 15u) != 0;
    if (p.c_f32) {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = blk[i];
        q[8] = extra ? blk[8] : make_uint4(0u, 0u, 0u, 0u);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = blk[i];
        q[4] = extra ? blk[4] : make_uint4(0u, 0u, 0u, 0u);
    }
}

// Bytes [off, off + 4 NW) of the word array w (NW + 4 words), off in 0..15:
// a shift by 2 words, then by 1 word, then a funnel shift by the byte rest,
// all branch-free so lanes with different offsets stay converged.
template <int NW>
__device__ __forceinline__ void shift_bytes(const uint32_t (&w)[NW + 4], uint32_t off, uint32_t (&o)[NW]) {
    const bool s2 = (off & 8u) != 0, s1 = (off & 4u) != 0;
    uint32_t u[NW + 2];
#pragma unroll
    for (int i = 0; i < NW + 2; ++i) u[i] = s2 ? w[i + 2] : w[i];
    uint32_t v[NW + 1];
#pragma unroll
    for (int i = 0; i < NW + 1; ++i) v[i] = s1 ? u[i + 1] : u[i];
    const uint32_t sh = (off & 3u) * 8u;
#pragma unroll
    for (int i = 0; i < NW; ++i) o[i] = __funnelshift_r(v[i], v[i + 1], sh);
}

__device__ __forceinline__ void c_values(const KernelParams& p, int row, int col0, const uint4 (&q)[9],
                                         float (&c)[32]) {
    if (col0 + 32 > p.N) {
        const char* crow = static_cast<const char*>(p.C) + static_cast<long long>(row) * p.ldc * (p.c_f32 ? 4 : 2);
        load_row32(crow, p.c_f32, col0, p.N, c, p.c_vec != 0);
        return;
    }
    if (p.c_f32) {
        uint32_t o[32];
        if (p.c_vec) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                o[4 * i + 0] = q[i].x; o[4 * i + 1] = q[i].y; o[4 * i + 2] = q[i].z; o[4 * i + 3] = q[i].w;
            }
        } else {
            uint32_t w[36];
#pragma unroll
            for (int i = 0; i < 9; ++i) {
                w[4 * i + 0] = q[i].x; w[4 * i + 1] = q[i].y; w[4 * i + 2] = q[i].z; w[4 * i + 3] = q[i].w;
            }
            shift_bytes<32>(w, static_cast<uint32_t>(c_chunk_addr(p, row, col0) & 15u), o);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) c[i] = __uint_as_float(o[i]);
    } else {
        uint32_t o[16];
        if (p.c_vec) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                o[4 * i + 0] = q[i].x; o[4 * i + 1] = q[i].y; o[4 * i + 2] = q[i].z; o[4 * i + 3] = q[i].w;
            }
        } else {
            uint32_t w[20];
#pragma unroll
            for (int i = 0; i < 5; ++i) {
                w[4 * i + 0] = q[i].x; w[4 * i + 1] = q[i].y; w[4 * i + 2] = q[i].z; w[4 * i + 3] = q[i].w;
            }
            shift_bytes<16>(w, static_cast<uint32_t>(c_chunk_addr(p, row, col0) & 15u), o);
        }
#pragma unroll
        for (int h = 0; h < 16; ++h) {
            c[2 * h + 0] = bf16_bits_to_float(o[h] & 0xFFFFu);
            c[2 * h + 1] = bf16_bits_to_float(o[h] >> 16);
        }
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// One thread's row of a C chunk that the TMA brought into an epilogue buffer
// (the same swizzled layout stage_row writes for D).
__device__ __forceinline__ void c_row_from_smem(const uint8_t* buf, int row, int c_f32, float (&c)[32]) {
    if (c_f32) {
        const uint8_t* rowp = buf + row * 128;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 q = *reinterpret_cast<const float4*>(rowp + ((k ^ (row & 7)) << 4));
            c[4 * k + 0] = q.x; c[4 * k + 1] = q.y; c[4 * k + 2] = q.z; c[4 * k + 3] = q.w;
        }
    } else {
        const uint8_t* rowp = buf + row * 64;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 q = *reinterpret_cast<const uint4*>(rowp + ((k ^ ((row >> 1) & 3)) << 4));
            const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                c[8 * k + 2 * h + 0] = bf16_bits_to_float(wv[h] & 0xFFFFu);
                c[8 * k + 2 * h + 1] = bf16_bits_to_float(wv[h] >> 16);
            }
        }
    }
}

// Wait until at most n of this thread's bulk store groups still read shared memory.
__device__ __forceinline__ void bulk_wait_read_at_most(int n) {
    if (n <= 0) ptx::bulk_wait_group_read<0>();
    else if (n == 1) ptx::bulk_wait_group_read<1>();
    else if (n == 2) ptx::bulk_wait_group_read<2>();
    else ptx::bulk_wait_group_read<3>();
}

// Write one thread's 32 results (its row of the 32 x 32 chunk) into the
// staging tile in the layout the D tensor map's swizzle expects:
//   f32 : 128-byte rows, 16-byte chunk c of row r at chunk c ^ (r & 7)
//   bf16:  64-byte rows, 16-byte chunk c of row r at chunk c ^ ((r >> 1) & 3)
__device__ __forceinline__ void stage_row(uint8_t* buf, int row, int d_f32, const float (&v)[32]) {
    if (d_f32) {
        uint8_t* rowp = buf + row * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int pc = c ^ (row & 7);
            float4 q = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            *reinterpret_cast<float4*>(rowp + pc * 16) = q;
        }
    } else {
        uint8_t* rowp = buf + row * 64;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int pc = c ^ ((row >> 1) & 3);
            uint4 q;
            q.x = pack_bf16x2(v[8 * c + 0], v[8 * c + 1]);
            q.y = pack_bf16x2(v[8 * c + 2], v[8 * c + 3]);
            q.z = pack_bf16x2(v[8 * c + 4], v[8 * c + 5]);
            q.w = pack_bf16x2(v[8 * c + 6], v[8 * c + 7]);
            *reinterpret_cast<uint4*>(rowp + pc * 16) = q;
        }
    }
}

// Store a warp's staged 32 x 32 chunk (stage_row layout) without the TMA:
// lane l writes column col0 + l of each of the 32 rows, so every store
// instruction covers one contiguous run of a row.  Used when D has no TMA map
// (unaligned base or row pitch) and for a ragged last chunk whose row end is
// not on a 16-byte boundary (the TMA store clips the inner dimension only to
// 16-byte granularity).  Rows >= M and columns >= N are skipped.
__device__ __forceinline__ void store_chunk_direct(const KernelParams& p, const uint8_t* buf, int row0, int col0,
                                                   int lane) {
    const int col = col0 + lane;
    if (col >= p.N) return;
    const int nrows = min(32, p.M - row0);
    if (p.d_f32) {
        float* dst = static_cast<float*>(p.D) + col;
        const int in_row = (lane & 3) * 4, chunk = lane >> 2;
        for (int r = 0; r < nrows; ++r) {
            const float v = *reinterpret_cast<const float*>(buf + r * 128 + ((chunk ^ (r & 7)) << 4) + in_row);
            dst[static_cast<long long>(row0 + r) * p.ldd] = v;
        }
    } else {
        uint16_t* dst = static_cast<uint16_t*>(p.D) + col;
        const int in_row = (lane & 7) * 2, chunk = lane >> 3;
        for (int r = 0; r < nrows; ++r) {
            const uint16_t v =
                *reinterpret_cast<const uint16_t*>(buf + r * 64 + ((chunk ^ ((r >> 1) & 3)) << 4) + in_row);
            dst[static_cast<long long>(row0 + r) * p.ldd] = v;
        }
    }
}

// kCta2 = false: one CTA per 128 x BN tile.
// kCta2 = true : a cluster of two CTAs per 256 x BN tile (tcgen05 cta_group::2).
//   Each CTA loads its own 128 rows of A and its own BN/2 rows of B (no
//   multicast); the TMA completions of both CTAs are counted on the even
//   (leader) CTA's full barrier; the leader's single thread issues the pair
//   MMA, whose result rows 0-127 land in the leader's TMEM and rows 128-255 in
//   the peer's; commits are multicast to the barriers of both CTAs; the peer's
//   epilogue hands accumulators back through the leader's tmem_empty barrier.
//
// kKAtoms = 128-byte K atoms per pipeline stage (1 or 2).  Two atoms put
// twice the MMAs behind each stage handshake (wait, commit), which is what
// keeps the tensor pipe busy with pair tiles.
// kBlk: block-scaled operands (1-CTA tiles with BN = 128, pairs with BN = 192
// or 256): 1 = MXFP8 (E4M3/E5M2, E8M0 per 32, kind::mxf8f6f4 1X), 2 = NVFP4
// (E2M1, unsigned E4M3 per 16, kind::mxf4nvf4 4X), 3 = MXFP4 (E2M1, E8M0 per
// 32, kind::mxf4nvf4 2X).
// FP4 operands are handled as bytes (two elements each, K counted in bytes).
// Each stage also carries the tile's scale blocks for its 128-byte K atoms
// (512 bytes per 128 rows and 4 scales: 1, 4 or 2 blocks per atom per
// operand), which the MMA thread copies to TMEM with tcgen05.cp before the
// stage's MMAs; the TMEM columns after the accumulators hold 4 columns per block.
//
// kGrouped: the launch runs a grouped GEMM (see next_unit): every role reads
// the sizes, tensor maps and epilogue pointers of each unit from its
// problem's parameter block.
//
// kTrans: the launch computes the transposed product D^T = B^T A^T of a GEMM
// with few rows (the host swaps the operands and the sizes: the kernel's M is
// D's column count and its N is D's row count).  The epilogue then writes
// element (r, c) of the kernel's tile to D[c][r] (row-major D, ld = ldd) and
// reads C the same way, the bias per kernel row (D's column), and the host
// swaps the row and column scale vectors.  One-CTA tiles only.
template <int BN, bool kFp8, bool kCta2, int kKAtoms, int kBlk = 0, bool kGrouped = false, bool kTrans = false>
__global__ void __launch_bounds__(kNumThreads, 1) gemm_persistent_kernel(const __grid_constant__ KernelParams p) {
    constexpr int kElemBytes = kFp8 ? 1 : 2;
    constexpr int kBK = kRowBytes / kElemBytes;       // K elements per 128-byte atom
    constexpr int kStageK = kKAtoms * kBK;             // K elements per pipeline stage
    constexpr int kMmaK = 32 / kElemBytes;             // K per tcgen05.mma
    constexpr int kKSteps = kBK / kMmaK;               // MMAs per atom
    constexpr int kAtom = kRowBytes / kElemBytes;      // MN elements per swizzle row
    constexpr int kBRows = kCta2 ? BN / 2 : BN;        // B rows (N) this CTA loads
    static_assert(kBRows % 8 == 0 && BN % kEpiChunk == 0, "B rows in whole 8-row swizzle groups, whole epilogue chunks");
    // MN-major B boxes are whole 128-byte MN atoms, so an MN-major B needs
    // kBRows to be a multiple of kAtom; the planner gives other widths (the
    // wave-fitting pair tiles 256 x 160 / 192 / 224) K-major B only.  8-bit
    // operands are K-major only.
    constexpr bool kBMnOk = !kFp8 && kBRows % kAtom == 0;
    constexpr int kTileM = kCta2 ? 2 * kBM : kBM;      // D rows per unit of work
    constexpr int kABytes = kKAtoms * kBM * kRowBytes;
    constexpr int kBBytes = kKAtoms * kBRows * kRowBytes;
    constexpr bool kMx = kBlk != 0;
    static_assert(!(kMx && kGrouped), "grouped GEMMs take unscaled or per-tensor-scaled operands");
    static_assert(!kTrans || (!kCta2 && !kMx && !kGrouped), "transposed output: one-CTA plain tiles");
    static_assert(!kMx || (kFp8 && (kCta2 ? (BN == 256 || BN == 192) : BN == 128)),
                  "block-scaled tiles are 8-bit 128 x 128 (one CTA) or 256 x 256 / 256 x 192 (a pair)");
    constexpr int kSfBlock = 512;                          // 128 rows x 4 scales
    constexpr int kSfPerAtom = kBlk == 2 ? 4 : (kBlk == 3 ? 2 : 1);   // scale blocks per operand per atom
    // scale blocks per atom: A's (this CTA's 128 rows) and B's (all BN columns: a pair's
    // tensor cores each need the scales of every column).  B's tile columns
    // [n0, n0 + BN) start on a multiple of 64, so two 128-row scale blocks
    // cover them for BN = 192 and 256 (kBH column blocks per scale index).
    constexpr int kBH = BN > 128 ? 2 : 1;
    constexpr int kSfA = kSfPerAtom, kSfB = kSfPerAtom * kBH;
    constexpr int kSfBytes = kMx ? (kKAtoms * (kSfA + kSfB) * kSfBlock + 1023) / 1024 * 1024 : 0;  // 1 KiB padded
    // A pair tile's 256 accumulator columns leave no room for scales next to a
    // second accumulator: block-scaled 256-wide pair tiles use one
    // accumulator; 192-wide ones keep two (2 x 192 columns + scales).
    constexpr int kAccBufs = (kMx && kCta2 && BN == 256) ? 1 : 2;
    constexpr int kStageBytes = kABytes + kBBytes + kSfBytes;
    static_assert(kStageBytes % 1024 == 0, "operand tiles stay 1024-byte aligned");
    // bytes the stage's copies deliver (the scale area's padding is not loaded)
    constexpr uint32_t kTxBytes = (kCta2 ? 2 : 1) * (kABytes + kBBytes + (kMx ? kKAtoms * (kSfA + kSfB) * kSfBlock : 0));
    // half-width tail units: plain 256-wide tiles only (B rows halve, in whole MN atoms)
    constexpr bool kHalfOk = BN == 256 && !kMx && !kGrouped && !kTrans;
    constexpr uint32_t kTxBytesHalf = (kCta2 ? 2 : 1) * (kABytes + kBBytes / 2);
    // TMEM is allocated in powers of two columns: two accumulators of BN
    constexpr uint32_t kTmemCols = kMx ? 512 : (2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512));
    constexpr int kSfCol0 = kAccBufs * BN;                 // first scale-factor column in TMEM
    static_assert(!kMx || kSfCol0 + 8 * (kSfA + kSfB) * kKAtoms <= 512, "scale columns fit in TMEM for 2 stages");

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.stages;
    uint8_t* epi_smem = smem + S * kStageBytes;
    constexpr int kRingWarp = epi_warp_bytes(kMx && kCta2 && BN == 256);   // epilogue buffers per warp
    SmemCtl* ctl = reinterpret_cast<SmemCtl*>(epi_smem + 4 * kRingWarp);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = kCta2 ? ptx::cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int first_unit = kCta2 ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int unit_stride = kCta2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(&ctl->full[s], 1);
            ptx::mbar_init(&ctl->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&ctl->tmem_full[a], 1);
            ptx::mbar_init(&ctl->tmem_empty[a], kCta2 ? 8 : 4);
        }
        ptx::mbar_init(&ctl->drain, 1);
        for (int w4 = 0; w4 < 4; ++w4)
            for (int b = 0; b < 4; ++b) ptx::mbar_init(&ctl->cbar[w4][b], 1);
        ctl->abort_flag = 0;
        ctl->splitk_last = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        if constexpr (kCta2) {
            ptx::tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
            ptx::tmem_relinquish_alloc_permit_pair();
        } else {
            ptx::tmem_alloc(&ctl->tmem_base, kTmemCols);
            ptx::tmem_relinquish_alloc_permit();
        }
    }
    ptx::tc_fence_before_sync();
    if constexpr (kCta2) ptx::cluster_sync();  // peer barriers exist before anyone signals them
    else __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = ctl->tmem_base;
    const long long limit = p.timeout_ns;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        {
            const bool issuer = lane == 0;
            if (!kGrouped && issuer && p.num_kb > 0) {
                ptx::prefetch_tensormap(&p.tmA);
                ptx::prefetch_tensormap(&p.tmB);
            }
            int cur_g = -1;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;
            long long st_wait = 0;
            bool first = true;
            bool ok = true;
            WorkIter wi = work_begin(p, first_unit, unit_stride);
            Unit w;
            while (ok && next_unit<kGrouped>(p, wi, w)) {
                const KernelParams& q = unit_params<kGrouped>(p, w);
                if (!dcheck(w.m_blk >= 0 && w.m_blk < q.num_m_blk && w.n_blk >= 0 && w.n_blk < q.num_n_blk &&
                                w.kb0 >= 0 && w.kb0 <= w.kb1 && w.kb1 <= q.num_kb, p, ctl, kChkUnit)) {
                    ok = false;
                    break;
                }
                if (kGrouped && w.g != cur_g) {
                    if (issuer) {
                        ptx::fence_tensormap_acquire(&q.tmA);
                        ptx::fence_tensormap_acquire(&q.tmB);
                    }
                    cur_g = w.g;
                }
                const int m_blk = w.m_blk, n_blk = w.n_blk, kb0 = w.kb0, kb1 = w.kb1;
                const int a_row = m_blk * kTileM + static_cast<int>(rank) * kBM;
                const bool half = kHalfOk && w.nh != 0;
                const int b_row = unit_n0(w, BN) + static_cast<int>(rank) * (half ? kBRows / 2 : kBRows);
                for (int ki = kb0; ki < kb1; ++ki) {
                    const int kb = w.rev ? kb0 + kb1 - 1 - ki : ki;
                    const long long tw = p.stats ? clock64() : 0;
                    if (!dcheck(stage >= 0 && stage < S && S <= 16, p, ctl, kChkStage)) { ok = false; break; }
                    if (!warp_wait(&ctl->empty[stage], phase ^ 1u, p, ctl, 1, limit, true, kCta2)) { ok = false; break; }
                    if (!dcheck_phase(&ctl->empty[stage], phase ^ 1u, p, ctl)) { ok = false; break; }
                    // the test knob's forced failure of the debug build (no effect otherwise)
                    if (!dcheck(!(first && p.fault_inject == 2 && blockIdx.x == 0), p, ctl, kChkForced)) {
                        ok = false;
                        break;
                    }
                    if (p.stats) st_wait += clock64() - tw;
                    const bool skip = first && p.fault_inject == 1 && blockIdx.x == 0;
                    first = false;
                    if (!skip && issuer) {
                        uint8_t* sA = smem + stage * kStageBytes;
                        uint8_t* sB = sA + kABytes;
                        uint64_t* fb = &ctl->full[stage];
                        if (leader) ptx::mbar_arrive_expect_tx(fb, half ? kTxBytesHalf : kTxBytes);
                        const uint32_t fbc = kCta2 ? ptx::map_to_cta(ptx::smem_u32(fb), 0) : 0u;
                        auto load = [&](void* dst, const CUtensorMap* map, int x, int y) {
                            if constexpr (kCta2) ptx::tma_load_2d_pair(dst, map, fbc, x, y);
                            else ptx::tma_load_2d(dst, map, fb, x, y);
                        };
                        const int k0 = kb * kStageK;
                        // K-major: one box of BK x rows per atom, atoms stacked;
                        // MN-major: one box of kAtom x kStageK per MN atom.
                        if (!p.a_mn_major) {
#pragma unroll
                            for (int at = 0; at < kKAtoms; ++at)
                                load(sA + at * kBM * kRowBytes, &q.tmA, k0 + at * kBK, a_row);
                        } else {
#pragma unroll
                            for (int h = 0; h < kBM / kAtom; ++h)
                                load(sA + h * kRowBytes * kStageK, &q.tmA, a_row + h * kAtom, k0);
                        }
                        if (!kBMnOk || !p.b_mn_major) {
                            const CUtensorMap* mb = half ? &p.tmB2 : &q.tmB;
#pragma unroll
                            for (int at = 0; at < kKAtoms; ++at)
                                load(sB + at * kBRows * kRowBytes, mb, k0 + at * kBK, b_row);
                        } else {
                            const int boxes = (half ? kBRows / 2 : kBRows) / kAtom;
#pragma unroll
                            for (int h = 0; h < kBRows / kAtom; ++h)
                                if (h < boxes) load(sB + h * kRowBytes * kStageK, &q.tmB, b_row + h * kAtom, k0);
                        }
                        if constexpr (kMx && kCta2) {
                            // scale blocks of this stage's atoms, per atom: kSfA blocks of
                            // this CTA's 128-row block of A, then kSfPerAtom blocks of each
                            // of B's two 128-column blocks (both CTAs load all of B's)
                            uint8_t* sSf = sB + kBBytes;
                            const int rb_a = m_blk * 2 + static_cast<int>(rank);
#pragma unroll
                            for (int at = 0; at < kKAtoms; ++at) {
                                const int cb = (kb * kKAtoms + at) * kSfPerAtom;
                                uint8_t* dst = sSf + at * (kSfA + kSfB) * kSfBlock;
                                load(dst, &p.tmSFA, 0, rb_a * p.num_sfcb + cb);
#pragma unroll
                                for (int h = 0; h < kBH; ++h)
                                    load(dst + (kSfA + h * kSfPerAtom) * kSfBlock, &p.tmSFB, 0,
                                         ((n_blk * BN) / 128 + h) * p.num_sfcb + cb);
                            }
                        } else if constexpr (kMx) {
                            // scale blocks of this stage's atoms: per atom kSfPerAtom blocks
                            // of A's row block, then kSfPerAtom of B's column block
                            uint8_t* sSf = sB + kBBytes;
#pragma unroll
                            for (int at = 0; at < kKAtoms; ++at) {
#pragma unroll
                                for (int sb = 0; sb < kSfPerAtom; ++sb) {
                                    // blocks past K (a last, partial atom) reuse the last one:
                                    // their elements are zero-filled by the TMA
                                    const int cb = min((kb * kKAtoms + at) * kSfPerAtom + sb, p.num_sfcb - 1);
                                    ptx::bulk_load(sSf + ((2 * at) * kSfPerAtom + sb) * kSfBlock,
                                                   p.sfa + (static_cast<size_t>(m_blk) * p.num_sfcb + cb) * kSfBlock,
                                                   kSfBlock, fb);
                                    ptx::bulk_load(sSf + ((2 * at + 1) * kSfPerAtom + sb) * kSfBlock,
                                                   p.sfb + (static_cast<size_t>(n_blk) * p.num_sfcb + cb) * kSfBlock,
                                                   kSfBlock, fb);
                                }
                            }
                        }
                    }
                    if (!skip) {
                        armed |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    }
                    __syncwarp();
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            if (p.stats && issuer) atomicAdd(p.stats + kStatProdWaitEmpty, static_cast<unsigned long long>(st_wait));
            // Drain: every stage this thread filled has landed before the CTA
            // may leave (its shared memory is the copies' destination).  The
            // leader sees its fills complete on its own full barriers; the
            // peer sees them consumed through its empty barriers.
            for (int s = 0; s < S; ++s) {
                if (!(armed & (1u << s))) continue;
                const uint32_t par = (armed_parity >> s) & 1u;
                if (leader) warp_wait(&ctl->full[s], par, p, ctl, 11, limit, false);
                else warp_wait(&ctl->empty[s], par, p, ctl, 13, limit, false);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (leader) {
            const bool issuer = lane == 0;
            // Instruction descriptor.  kind::f16 / kind::f8f6f4: D format F32 in
            // bits 4-5.  Block-scaled kinds: bits 4-5 select B's scale byte, bits
            // 29-30 A's (set per MMA below), bit 23 = E8M0 (1) or UE4M3 (0)
            // scales; the operand format of kind::mxf4nvf4 is E2M1 = 1.
            constexpr uint32_t kScaleType = (kBlk == 1 || kBlk == 3) ? (1u << 23) : 0u;
            const uint32_t ab_fmt = (kBlk == 2 || kBlk == 3) ? 1u : p.ab_fmt;
            const uint32_t idesc_full = (kMx ? kScaleType : (1u << 4)) | (ab_fmt << 7) | (ab_fmt << 10) |
                                   (static_cast<uint32_t>(p.a_mn_major) << 15) |
                                   (static_cast<uint32_t>(p.b_mn_major) << 16) |
                                   (static_cast<uint32_t>(BN >> 3) << 17) |
                                   (static_cast<uint32_t>(kTileM >> 4) << 24);
            // Descriptor geometry.  K-major: 8-row groups 1024 B apart (SBO),
            // k-step = +kMmaK*elem bytes inside the swizzle row.  MN-major:
            // swizzle-row boxes of kAtom MN elements, BK rows each (LBO apart),
            // 8-row K groups 1024 B apart (SBO), k-step = kMmaK rows.
            const uint32_t a_lbo = p.a_mn_major ? static_cast<uint32_t>(kRowBytes * kStageK) : 16u;
            const uint32_t b_lbo = p.b_mn_major ? static_cast<uint32_t>(kRowBytes * kStageK) : 16u;
            // start-address advance (16-byte units) of MMA kk within a stage
            auto a_off = [&](int kk) -> uint32_t {
                return p.a_mn_major ? static_cast<uint32_t>(kk * kMmaK * kRowBytes) >> 4
                                    : static_cast<uint32_t>((kk / kKSteps) * kBM * kRowBytes +
                                                            (kk % kKSteps) * kMmaK * kElemBytes) >> 4;
            };
            auto b_off = [&](int kk) -> uint32_t {
                return p.b_mn_major ? static_cast<uint32_t>(kk * kMmaK * kRowBytes) >> 4
                                    : static_cast<uint32_t>((kk / kKSteps) * kBRows * kRowBytes +
                                                            (kk % kKSteps) * kMmaK * kElemBytes) >> 4;
            };
            int stage = 0;
            uint32_t phase = 0;
            int t = 0;
            bool ok = true;
            bool issued_any = false;
            long long st_full = 0, st_acc = 0;
            const long long st_t0 = p.stats ? clock64() : 0;
            WorkIter wi = work_begin(p, first_unit, unit_stride);
            Unit w;
            for (; ok && next_unit<kGrouped>(p, wi, w); ++t) {
                const int kb0 = w.kb0, kb1 = w.kb1;
                const int acc = kAccBufs == 2 ? (t & 1) : 0;
                const uint32_t acc_phase = kAccBufs == 2 ? ((t >> 1) & 1) : (t & 1);
                const long long ta = p.stats ? clock64() : 0;
                if (!dcheck(acc >= 0 && acc < kAccBufs && (acc + 1) * BN <= static_cast<int>(kTmemCols), p, ctl,
                            kChkAcc)) {
                    ok = false;
                    break;
                }
                if (!warp_wait(&ctl->tmem_empty[acc], acc_phase ^ 1u, p, ctl, 2, limit, true, kCta2)) { ok = false; break; }
                if (!dcheck_phase(&ctl->tmem_empty[acc], acc_phase ^ 1u, p, ctl)) { ok = false; break; }
                if (p.stats) st_acc += clock64() - ta;
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                // a half-width tail unit: N = BN / 2 (the first BN / 2 accumulator columns)
                const uint32_t idesc = (kHalfOk && w.nh != 0)
                                           ? ((idesc_full & ~(0x3Fu << 17)) | (static_cast<uint32_t>((BN / 2) >> 3) << 17))
                                           : idesc_full;
                // (the stages arrive in the producer's K order; only the first
                // of the unit's MMAs starts a new accumulation)
                for (int ki = kb0; ki < kb1; ++ki) {
                    const long long tf = p.stats ? clock64() : 0;
                    if (!dcheck(stage >= 0 && stage < S && S <= 16, p, ctl, kChkStage)) { ok = false; break; }
                    if (!warp_wait(&ctl->full[stage], phase, p, ctl, 3, limit, true, kCta2)) { ok = false; break; }
                    if (!dcheck_phase(&ctl->full[stage], phase, p, ctl)) { ok = false; break; }
                    if (kMx && !dcheck(kSfCol0 + (stage + 1) * kKAtoms * 4 * (kSfA + kSfB) <= 512, p, ctl,
                                       kChkScaleCols)) {
                        ok = false;
                        break;
                    }
                    if (p.stats) st_full += clock64() - tf;
                    ptx::tc_fence_after_sync();
                    if (issuer) {
                    const uint32_t sA = ptx::smem_u32(smem + stage * kStageBytes);
                    const uint32_t sB = sA + kABytes;
                    const uint64_t a_desc = ptx::smem_desc_sw128(sA, a_lbo, 1024);
                    const uint64_t b_desc = ptx::smem_desc_sw128(sB, b_lbo, 1024);
                    uint32_t sf_base = 0;
                    if constexpr (kMx) {
                        // this stage's scale blocks -> TMEM, 4 columns per block, in
                        // the order they sit in shared memory (per atom: A's, then B's)
                        const uint32_t sSf = sB + static_cast<uint32_t>(kBBytes);
                        sf_base = tmem_base + static_cast<uint32_t>(kSfCol0 + stage * kKAtoms * 4 * (kSfA + kSfB));
                        // TMEM order per atom: A's blocks, then B's with the column blocks of
                        // one scale index side by side (the MMA reads column n at n / 32)
                        auto cp = [&](int smem_block, int col) {
                            const uint64_t sd = ptx::smem_desc_noswizzle_16b_rows(sSf + smem_block * kSfBlock);
                            if constexpr (kCta2) ptx::tmem_cp_32x128b_warpx4_pair(sf_base + static_cast<uint32_t>(col), sd);
                            else ptx::tmem_cp_32x128b_warpx4(sf_base + static_cast<uint32_t>(col), sd);
                        };
#pragma unroll
                        for (int at = 0; at < kKAtoms; ++at) {
                            const int blk0 = at * (kSfA + kSfB), col0 = 4 * blk0;
#pragma unroll
                            for (int sb = 0; sb < kSfA; ++sb) cp(blk0 + sb, col0 + 4 * sb);
#pragma unroll
                            for (int h = 0; h < kBH; ++h)
#pragma unroll
                                for (int sb = 0; sb < kSfPerAtom; ++sb)
                                    cp(blk0 + kSfA + h * kSfPerAtom + sb, col0 + 4 * kSfA + 4 * (sb * kBH + h));
                        }
                    }
#pragma unroll
                    for (int k = 0; k < kKAtoms * kKSteps; ++k) {
                        const uint64_t ad = a_desc + static_cast<uint64_t>(a_off(k));
                        const uint64_t bd = b_desc + static_cast<uint64_t>(b_off(k));
                        const uint32_t accum = (ki > kb0 || k > 0) ? 1u : 0u;
                        if constexpr (kMx) {
                            // MMA kk of atom `at`: its scale blocks and the byte the first
                            // of its scales sits at inside each 32-bit TMEM word
                            // (B's scales: for BN = 256 two 128-column blocks, 4 columns apart
                            // per scale-block index, as the MMA reads column n at n / 32)
                            const int at = k / kKSteps, kk = k % kKSteps;
                            const uint32_t a_blocks = sf_base + static_cast<uint32_t>(at * 4 * (kSfA + kSfB));
                            // B's tile starts (n0 % 128) / 32 columns into its first block
                            const uint32_t b_blocks = a_blocks + static_cast<uint32_t>(4 * kSfA) +
                                                      static_cast<uint32_t>(((w.n_blk * BN) & 127) >> 5);
                            uint32_t sfid = 0, a_sf = a_blocks, b_sf = b_blocks;
                            if constexpr (kBlk == 1) {          // one scale per MMA: byte kk of block 0
                                sfid = static_cast<uint32_t>(kk);
                            } else if constexpr (kBlk == 2) {   // four scales per MMA: all of block kk
                                a_sf += static_cast<uint32_t>(kk * 4);
                                b_sf += static_cast<uint32_t>(kk * 4 * kBH);
                            } else {                            // two scales per MMA: half of block kk / 2
                                a_sf += static_cast<uint32_t>((kk / 2) * 4);
                                b_sf += static_cast<uint32_t>((kk / 2) * 4 * kBH);
                                sfid = static_cast<uint32_t>((kk & 1) * 2);
                            }
                            const uint32_t id = idesc | (sfid << 4) | (sfid << 29);
                            if constexpr (kCta2) {
                                if constexpr (kBlk == 1) ptx::mma_mxf8_pair(d_tmem, ad, bd, id, a_sf, b_sf, accum);
                                else if constexpr (kBlk == 2) ptx::mma_mxf4_4x_pair(d_tmem, ad, bd, id, a_sf, b_sf, accum);
                                else ptx::mma_mxf4_2x_pair(d_tmem, ad, bd, id, a_sf, b_sf, accum);
                            } else {
                                if constexpr (kBlk == 1) ptx::mma_mxf8(d_tmem, ad, bd, id, a_sf, b_sf, accum);
                                else if constexpr (kBlk == 2) ptx::mma_mxf4_4x(d_tmem, ad, bd, id, a_sf, b_sf, accum);
                                else ptx::mma_mxf4_2x(d_tmem, ad, bd, id, a_sf, b_sf, accum);
                            }
                        } else if constexpr (kCta2) {
                            if constexpr (kFp8) ptx::mma_f8_pair(d_tmem, ad, bd, idesc, accum);
                            else ptx::mma_f16_pair(d_tmem, ad, bd, idesc, accum);
                        } else {
                            if constexpr (kFp8) ptx::mma_f8(d_tmem, ad, bd, idesc, accum);
                            else ptx::mma_f16(d_tmem, ad, bd, idesc, accum);
                        }
                    }
                    if constexpr (kCta2) ptx::mma_commit_pair(&ctl->empty[stage], 0x3);
                    else ptx::mma_commit(&ctl->empty[stage]);
                    }
                    __syncwarp();
                    issued_any = true;
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                if (!issuer) {
                } else if (kb1 > kb0) {
                    if constexpr (kCta2) ptx::mma_commit_pair(&ctl->tmem_full[acc], 0x3);
                    else ptx::mma_commit(&ctl->tmem_full[acc]);
                } else {
                    if constexpr (kCta2) {
                        ptx::mbar_arrive(&ctl->tmem_full[acc]);
                        ptx::mbar_arrive_cluster(ptx::map_to_cta(ptx::smem_u32(&ctl->tmem_full[acc]), 1));
                    } else {
                        ptx::mbar_arrive(&ctl->tmem_full[acc]);
                    }
                }
            }
            if (p.stats && issuer) {
                atomicAdd(p.stats + kStatMmaWaitFull, static_cast<unsigned long long>(st_full));
                atomicAdd(p.stats + kStatMmaWaitAcc, static_cast<unsigned long long>(st_acc));
                atomicAdd(p.stats + kStatMmaTotal, static_cast<unsigned long long>(clock64() - st_t0));
                atomicAdd(p.stats + kStatCtas, 1ull);
            }
            // Drain: all MMAs lane 0 issued complete before TMEM is freed.
            if (issued_any) {
                if (issuer) {
                    if constexpr (kCta2) ptx::mma_commit_pair(&ctl->drain, 0x1);
                    else ptx::mma_commit(&ctl->drain);
                }
                __syncwarp();
                warp_wait(&ctl->drain, 0, p, ctl, 12, limit, false);
            }
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int g = warp & 3;                 // TMEM lane group this warp may access
        const int row_in_tile = g * 32 + lane;  // this thread's accumulator row
        // Per warp, a ring of nbuf chunk buffers (8 KiB in all).  Chunk number
        // cc (counted over the whole launch) uses buffer cc mod nbuf: C's
        // 32 x 32 box lands there by TMA (when C is read), the thread reads
        // its row, then writes its D row into the same buffer for the TMA
        // store.  C boxes are requested L = nbuf / 2 chunks ahead.
        uint8_t* const ring = epi_smem + (warp - kEpiWarp0) * kRingWarp;
        const int nbuf = p.epi_nbuf;
        const int buf_bytes = kRingWarp / nbuf;
        const int lookahead = nbuf / 2;
        const uint32_t c_box_bytes = p.c_f32 ? 4096u : 2048u;
        uint64_t* const cbar = ctl->cbar[warp - kEpiWarp0];
        int cc = 0;             // chunks processed by this warp
        uint32_t cph = 0;       // phase bit of each C barrier
        int c_pending = 0;      // C boxes requested and not yet waited for
        bool mixed = false;     // a chunk was stored without the TMA: wait for every store before reuse
        const bool has_c = p.beta != 0.0f;
        const bool c_tma = has_c && p.c_tma;
        long long st_ewait = 0, st_ebusy = 0;
        const CUtensorMap* tm_c = &p.tmC;   // the current unit's C map
        int cur_g = -1;
        // Request C chunk x (columns col0, this warp's 32 rows at row0) into
        // buffer x mod nbuf, once the D store that last used it has read it
        // (n_wait = stores issued after that one).  Whole warp, converged.
        auto issue_c = [&](int x, int col0, int row0, int n_wait) {
            ptx::fence_proxy_async_smem();  // this warp's reads of the buffer come first
            __syncwarp();
            if (lane == 0) {
                bulk_wait_read_at_most(mixed ? 0 : n_wait);
                uint64_t* bar = &cbar[x & (nbuf - 1)];
                ptx::mbar_arrive_expect_tx(bar, c_box_bytes);
                ptx::tma_load_2d(ring + (x & (nbuf - 1)) * buf_bytes, tm_c, bar, col0, row0);
            }
            ++c_pending;
        };
        auto wait_c = [&](int x, bool honor_abort) -> bool {
            const int b = x & (nbuf - 1);
            bool ok = warp_wait(&cbar[b], (cph >> b) & 1u, p, ctl, 5, limit, honor_abort, kCta2);
            if (ok) ok = dcheck_phase(&cbar[b], (cph >> b) & 1u, p, ctl);
            cph ^= 1u << b;
            --c_pending;
            return ok;
        };
        int t = 0;
        WorkIter wi = work_begin(p, first_unit, unit_stride);
        Unit w;
        for (; next_unit<kGrouped>(p, wi, w); ++t) {
            const KernelParams& q = unit_params<kGrouped>(p, w);
            if (kGrouped && w.g != cur_g) {
                tm_c = &q.tmC;
                if (lane == 0) {
                    if (c_tma) ptx::fence_tensormap_acquire(&q.tmC);
                    if (q.d_tma) ptx::fence_tensormap_acquire(&q.tmD);
                }
                cur_g = w.g;
            }
            const int m_blk = w.m_blk, kb0 = w.kb0, kb1 = w.kb1, split = w.split;
            const bool split_mode = w.nsplit > 1;
            constexpr int kRanks = kCta2 ? 2 : 1;
            const int counter = w.tile * kRanks + static_cast<int>(rank);
            const int acc = kAccBufs == 2 ? (t & 1) : 0;
            const uint32_t acc_phase = kAccBufs == 2 ? ((t >> 1) & 1) : (t & 1);
            const int m0 = m_blk * kTileM + static_cast<int>(rank) * kBM;
            const int n0 = unit_n0(w, BN);
            const int ubn = unit_bn(w, BN);   // the unit's columns
            const int grow = m0 + row_in_tile;
            const bool row_ok = grow < q.M;
            const bool warp_rows_live = (m0 + g * 32) < q.M;
            const int nchunks = min(ubn / kEpiChunk, (q.N - n0 + kEpiChunk - 1) / kEpiChunk);
            uint4 cq[9];
            if (has_c && !kTrans) {
                // C rows of this tile on the first pass, then always of the next tile, into L2
                if (t == 0) c_prefetch_l2(q, grow, n0, ubn);
                WorkIter peek = wi;
                Unit nw;
                if (next_unit<kGrouped>(p, peek, nw))
                    c_prefetch_l2(unit_params<kGrouped>(p, nw), nw.m_blk * kTileM + static_cast<int>(rank) * kBM + row_in_tile,
                                  unit_n0(nw, BN), unit_bn(nw, BN));
                if (!c_tma && row_ok && !split_mode) c_prefetch(q, grow, n0, cq);
            }
            // First C boxes of a tile that is not split, before the accumulator is ready.
            if (c_tma && !split_mode && warp_rows_live)
                for (int l = 0; l < lookahead && l < nchunks; ++l)
                    issue_c(cc + l, n0 + l * kEpiChunk, m0 + g * 32, nbuf - 1 - l);
            // The tile's bias, read from global memory once per tile into shared
            // memory while the accumulator is still being computed (per chunk,
            // 32 broadcast global loads left their L2 latency exposed: 7 % of
            // the block-scaled kernels).  Barrier 2: every epilogue warp has
            // finished the previous tile's chunks before the values change;
            // barrier 1 below makes them visible.
            if (q.bias && !kTrans) {
                ptx::named_barrier_sync(2, kEpiThreads);
                for (int c = static_cast<int>(threadIdx.x) - kEpiWarp0 * 32; c < BN; c += kEpiThreads) {
                    const int col = n0 + c;
                    float bv = 0.0f;
                    if (col < q.N)
                        bv = q.bias_f32 ? static_cast<const float*>(q.bias)[col]
                                        : bf16_bits_to_float(static_cast<const uint16_t*>(q.bias)[col]);
                    ctl->bias_tile[c] = bv;
                }
            }
            const long long te = p.stats ? clock64() : 0;
            bool ok = wait_phase(&ctl->tmem_full[acc], acc_phase, p, ctl, 4, limit);
            if (ok) ok = dcheck_phase(&ctl->tmem_full[acc], acc_phase, p, ctl);
            if (ok) ok = dcheck((nbuf == 1 || nbuf == 2 || nbuf == 4) && nbuf * buf_bytes <= kRingWarp, p, ctl, kChkRing);
            const long long te1 = p.stats ? clock64() : 0;
            if (p.stats) st_ewait += te1 - te;
            // All four epilogue warps take the same branch (the split-K named
            // barriers below must be reached by all 128 threads or by none).
            ok = ptx::named_barrier_and(1, kEpiThreads, ok);
            if (!ok) break;
            ptx::tc_fence_after_sync();

            const bool have_acc = kb1 > kb0;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(g * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);

            bool finish = true;
            if (split_mode) {
                // Pass 1: this split's raw fp32 partial (valid rows only).
                // Column-major within the tile: the 32 rows of a warp form one
                // contiguous 128-byte line per column (coalesced stores/loads).
                const int own_slot = partial_slot(p, w, split, unit_stride) * kRanks + static_cast<int>(rank);
                const bool slot_ok = dcheck(own_slot >= 0 && own_slot < p.num_slots, p, ctl, kChkSlot);
                const bool counter_ok = dcheck(counter >= 0 && counter < p.num_counters, p, ctl, kChkCounter);
                float* slot = p.partials + static_cast<size_t>(own_slot) * (kBM * BN) + row_in_tile;
                if (warp_rows_live && have_acc && slot_ok) {
                    for (int j = 0; j < nchunks; ++j) {
                        uint32_t r[32];
                        ptx::tmem_load_32cols(t_row + static_cast<uint32_t>(j * kEpiChunk), r);
                        if (row_ok) {
                            float* dst = slot + static_cast<size_t>(j * kEpiChunk) * kBM;
#pragma unroll
                            for (int i = 0; i < 32; ++i) dst[i * kBM] = __uint_as_float(r[i]);
                        }
                    }
                }
                // Arrive on the tile; the last of its splits finishes it.  The
                // barrier orders every epilogue thread's partial stores before
                // one thread's acquire-release add: its release publishes this
                // CTA's partial to the GPU, and for the last arrival its acquire
                // makes the other pieces' partials (released by their own adds)
                // visible; the second barrier passes that on to every thread.
                ptx::named_barrier_sync(1, kEpiThreads);
                if (threadIdx.x == kEpiWarp0 * 32) {
                    int last = 0;
                    if (counter_ok) {
                        const int old = ptx::atomic_add_acq_rel_gpu(p.tile_counters + counter, 1);
                        last = (old == w.nsplit - 1) ? 1 : 0;
                        if (last) atomicExch(p.tile_counters + counter, 0);  // ready for the next launch
                    }
                    ctl->splitk_last = last;
                }
                ptx::named_barrier_sync(1, kEpiThreads);
                finish = ctl->splitk_last != 0;
                if (kChecks && finish) {
                    // every piece's partial slot (the finishing CTA reads them all)
                    bool slots_ok = true;
                    for (int pc = 0; pc < w.nsplit; ++pc) {
                        const int sl = partial_slot(p, w, pc, unit_stride) * kRanks + static_cast<int>(rank);
                        slots_ok = slots_ok && sl >= 0 && sl < p.num_slots;
                    }
                    if (!dcheck(slots_ok, p, ctl, kChkSlot)) finish = false;
                }
            }

            // The chunks this warp finishes, as (row group rg, column chunk j).
            // Unsplit tile: its own TMEM quadrant (rg = g), every chunk.  Split
            // tile whose four row groups all hold rows: the same, and the
            // finishing piece adds its own share from TMEM (the values it
            // also wrote as its partial, so the fixed-order sum is the same
            // whichever piece finishes).  Split tile with fewer live row
            // groups: every piece's partial is read from global memory, so
            // the (row group, chunk) items of the live rows are dealt
            // round-robin to the four epilogue warps, which then sum and
            // store in parallel.
            const int wq = warp - kEpiWarp0;
            const int live_groups = max(0, min(4, (q.M - m0 + 31) / 32));
            // (not compiled into the 256-wide pair tiles, which split K only in
            // the optional Stream-K schedules: it would cost them a register spill)
            constexpr bool kOwnQ = !(kCta2 && BN == 256);
            const bool own_q = kOwnQ && split_mode && live_groups == 4 && have_acc;
            auto item_of = [&](int k, int& rg, int& jj) -> bool {
                if (!finish) return false;
                if (!split_mode || own_q) {
                    if (!warp_rows_live || k >= nchunks) return false;
                    rg = g;
                    jj = k;
                    return true;
                }
                const int i = wq + 4 * k;
                if (i >= live_groups * nchunks) return false;
                rg = i / nchunks;
                jj = i - rg * nchunks;
                return true;
            };
            if (has_c && !c_tma && split_mode && !kTrans) {
                int rg, jj;
                if (item_of(0, rg, jj) && m0 + rg * 32 + lane < q.M) c_prefetch(q, m0 + rg * 32 + lane, n0 + jj * kEpiChunk, cq);
            }
            if (c_tma && split_mode)
                for (int l = 0; l < lookahead; ++l) {
                    int rg, jj;
                    if (!item_of(l, rg, jj)) break;
                    issue_c(cc + l, n0 + jj * kEpiChunk, m0 + rg * 32, nbuf - 1 - l);
                }
            {
                for (int k = 0;; ++k) {
                    int rg, j;
                    if (!item_of(k, rg, j)) break;
                    const int col0 = n0 + j * kEpiChunk;
                    const int grow = m0 + rg * 32 + lane;
                    const bool row_ok = grow < q.M;
                    float v[32];
                    if (!split_mode) {
                        uint32_t r[32];
                        if (have_acc) {
                            ptx::tmem_load_32cols(t_row + static_cast<uint32_t>(j * kEpiChunk), r);
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
                        }
                    } else {
                        // Fixed order over the pieces: the sum does not depend
                        // on which piece arrived last.
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
                        uint32_t own[32];
                        if constexpr (kOwnQ) {
                            if (own_q) ptx::tmem_load_32cols(t_row + static_cast<uint32_t>(j * kEpiChunk), own);
                        }
                        if (row_ok) {
                            for (int pc = 0; pc < w.nsplit; ++pc) {
                                if constexpr (kOwnQ) {
                                    if (own_q && pc == split) {
#pragma unroll
                                        for (int i = 0; i < 32; ++i) v[i] += __uint_as_float(own[i]);
                                        continue;
                                    }
                                }
                                const float* src =
                                    p.partials + (static_cast<size_t>(partial_slot(p, w, pc, unit_stride)) * kRanks + rank) * (kBM * BN) +
                                    static_cast<size_t>(j * kEpiChunk) * kBM + rg * 32 + lane;
                                float pv[32];
#pragma unroll
                                for (int i = 0; i < 32; ++i) pv[i] = __ldcg(src + i * kBM);
#pragma unroll
                                for (int i = 0; i < 32; ++i) v[i] += pv[i];
                            }
                        }
                    }
                    if (c_tma) {
                        int rg2, j2;
                        if (item_of(k + lookahead, rg2, j2))
                            issue_c(cc + lookahead, n0 + j2 * kEpiChunk, m0 + rg2 * 32, nbuf - 1 - lookahead);
                    }
                    if constexpr (kTrans) {
                        // Row grow of the kernel's tile is column grow of D; column
                        // col0 + i is row col0 + i of D.  Each store instruction of the
                        // warp covers 32 consecutive columns of one row of D.
                        if (row_ok) {
                            float rs = q.alpha;
                            if (q.row_scale) rs *= q.row_scale[grow];
                            float bv = 0.0f;
                            if (q.bias)
                                bv = q.bias_f32 ? static_cast<const float*>(q.bias)[grow]
                                                : bf16_bits_to_float(static_cast<const uint16_t*>(q.bias)[grow]);
                            const int nv = min(kEpiChunk, q.N - col0);
                            // every load first (C may be D itself, so a load after a
                            // store could not move ahead of it), then every store
                            float cs[32], cv[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const long long drow = static_cast<long long>(col0 + i);
                                cs[i] = (q.col_scale && i < nv) ? q.col_scale[col0 + i] : 1.0f;
                                cv[i] = 0.0f;
                                if (has_c && i < nv)
                                    cv[i] = q.c_f32 ? static_cast<const float*>(q.C)[drow * q.ldc + grow]
                                                    : bf16_bits_to_float(static_cast<const uint16_t*>(q.C)[drow * q.ldc + grow]);
                            }
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                if (i < nv) {
                                    float x = v[i] * rs;
                                    if (q.col_scale) x *= cs[i];
                                    if (has_c) x = fmaf(p.beta, cv[i], x);
                                    x = apply_act(p.act, x + bv);
                                    const long long drow = static_cast<long long>(col0 + i);
                                    if (p.d_f32) static_cast<float*>(q.D)[drow * q.ldd + grow] = x;
                                    else reinterpret_cast<__nv_bfloat16*>(q.D)[drow * q.ldd + grow] = __float2bfloat16_rn(x);
                                }
                            }
                        }
                        __syncwarp();
                        ++cc;
                    } else {
                        // alpha, beta*C, bias and GELU on packed pairs (f32x2)
                        uint64_t v2[16];
    #pragma unroll
                        for (int i = 0; i < 16; ++i) v2[i] = ptx::pack2(v[2 * i], v[2 * i + 1]);
                        {
                            // alpha * sA * sB, and the per-row / per-column scales
                            float rs = q.alpha;
                            if (q.row_scale && row_ok) rs *= q.row_scale[grow];
                            if (rs != 1.0f) {
                                const uint64_t al = ptx::pack2(rs, rs);
    #pragma unroll
                                for (int i = 0; i < 16; ++i) v2[i] = ptx::mul2(v2[i], al);
                            }
                            if (q.col_scale) {
                                float cs[32];
                                load_row32(q.col_scale, 1, col0, q.N, cs, q.cs_vec != 0);
    #pragma unroll
                                for (int i = 0; i < 16; ++i) v2[i] = ptx::mul2(v2[i], ptx::pack2(cs[2 * i], cs[2 * i + 1]));
                            }
                        }
                        uint8_t* const buf = ring + (cc & (nbuf - 1)) * buf_bytes;
                        if (has_c) {
                            float c[32];
                            if (c_tma) {
                                wait_c(cc, false);
                                c_row_from_smem(buf, lane, p.c_f32, c);
                            } else if (row_ok) {
                                c_values(q, grow, col0, cq, c);
                                int rg2, j2;
                                if (item_of(k + 1, rg2, j2) && m0 + rg2 * 32 + lane < q.M)
                                    c_prefetch(q, m0 + rg2 * 32 + lane, n0 + j2 * kEpiChunk, cq);
                            }
                            if (c_tma || row_ok) {
                                const uint64_t be = ptx::pack2(p.beta, p.beta);
    #pragma unroll
                                for (int i = 0; i < 16; ++i) v2[i] = ptx::fma2(be, ptx::pack2(c[2 * i], c[2 * i + 1]), v2[i]);
                            }
                        }
                        if (q.bias) {
                            // broadcast reads of the tile's bias (columns past N hold 0)
                            const float4* bt = reinterpret_cast<const float4*>(ctl->bias_tile + j * kEpiChunk);
    #pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float4 b4 = bt[i];
                                v2[2 * i] = ptx::add2(v2[2 * i], ptx::pack2(b4.x, b4.y));
                                v2[2 * i + 1] = ptx::add2(v2[2 * i + 1], ptx::pack2(b4.z, b4.w));
                            }
                        }
                        if (p.act == 2) {
    #pragma unroll
                            for (int i = 0; i < 16; ++i) v2[i] = gelu_erf2(v2[i]);
                        }
    #pragma unroll
                        for (int i = 0; i < 16; ++i) ptx::unpack2(v2[i], v[2 * i], v[2 * i + 1]);
                        if (p.act == 1) {
    #pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = apply_act(1, v[i]);
                        }
                        // Unless the host asks for every chunk to be staged for a TMA
                        // store, a whole chunk of a D whose rows start on 16-byte
                        // boundaries goes from registers straight to global memory:
                        // each thread writes its row's 64 (bf16) or 128 (f32)
                        // contiguous bytes, in 32-byte stores when D allows them.
                        // A ragged last chunk is always staged (the TMA store clips
                        // at N).
                        if (q.d_tma && col0 + kEpiChunk <= q.N && !p.d_stage_all) {
                            if (row_ok) {
                                char* rowp = static_cast<char*>(q.D) +
                                             (static_cast<long long>(grow) * q.ldd + col0) * (p.d_f32 ? 4 : 2);
                                if (q.d_v32) {
                                    // 32-byte stores: each writes whole 32-byte sectors
                                    // (col0 is a multiple of 32 elements, so rowp is
                                    // 32-byte aligned when D's base and pitch are)
                                    uint32_t w[8];
                                    if (p.d_f32) {
    #pragma unroll
                                        for (int c = 0; c < 4; ++c) {
    #pragma unroll
                                            for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(v[8 * c + i]);
                                            ptx::st_global_v8(rowp + 32 * c, w);
                                        }
                                    } else {
    #pragma unroll
                                        for (int c = 0; c < 2; ++c) {
    #pragma unroll
                                            for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(v[16 * c + 2 * i], v[16 * c + 2 * i + 1]);
                                            ptx::st_global_v8(rowp + 32 * c, w);
                                        }
                                    }
                                } else if (p.d_f32) {
    #pragma unroll
                                    for (int c = 0; c < 8; ++c)
                                        *reinterpret_cast<float4*>(rowp + 16 * c) =
                                            make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
                                } else {
    #pragma unroll
                                    for (int c = 0; c < 4; ++c) {
                                        uint4 w4;
                                        w4.x = pack_bf16x2(v[8 * c + 0], v[8 * c + 1]);
                                        w4.y = pack_bf16x2(v[8 * c + 2], v[8 * c + 3]);
                                        w4.z = pack_bf16x2(v[8 * c + 4], v[8 * c + 5]);
                                        w4.w = pack_bf16x2(v[8 * c + 6], v[8 * c + 7]);
                                        *reinterpret_cast<uint4*>(rowp + 16 * c) = w4;
                                    }
                                }
                            }
                            __syncwarp();
                            ++cc;
                            continue;
                        }
                        // The buffer is free: with C, every lane has read its C row
                        // (and the C request waited for the buffer's last store);
                        // without, once the store that used it nbuf chunks ago has read it.
                        if (!c_tma && lane == 0) bulk_wait_read_at_most(mixed ? 0 : nbuf - 1);
                        __syncwarp();
                        stage_row(buf, lane, p.d_f32, v);
                        if (q.d_tma && (col0 + kEpiChunk <= q.N || q.d_inner_aligned)) {
                            ptx::fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                ptx::tma_store_2d(&q.tmD, buf, col0, m0 + rg * 32);
                                ptx::bulk_commit_group();
                            }
                        } else {
                            __syncwarp();
                            store_chunk_direct(q, buf, m0 + rg * 32, col0, lane);
                            __syncwarp();
                            mixed = true;
                        }
                        ++cc;
                    }
                }
            }
            // Hand the accumulator back to the MMA issuer.
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (p.stats) st_ebusy += clock64() - te1;
            if (lane == 0) {
                if (kCta2 && !leader)
                    ptx::mbar_arrive_cluster(ptx::map_to_cta(ptx::smem_u32(&ctl->tmem_empty[acc]), 0));
                else
                    ptx::mbar_arrive(&ctl->tmem_empty[acc]);
            }
        }
        // C boxes still in flight (only after an abort) land before the CTA leaves.
        while (c_pending > 0) wait_c(cc++, false);
        if (lane == 0) ptx::bulk_wait_group<0>();
        if (p.stats && warp == kEpiWarp0 && lane == 0) {
            atomicAdd(p.stats + kStatEpiWaitFull, static_cast<unsigned long long>(st_ewait));
            atomicAdd(p.stats + kStatEpiBusy, static_cast<unsigned long long>(st_ebusy));
        }
    }

    ptx::tc_fence_before_sync();
    if constexpr (kCta2) ptx::cluster_sync();  // the leader's MMAs into the peer's TMEM are done
    else __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after_sync();
        if constexpr (kCta2) ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
        else ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace tcg
