// tcgemm_host.cu -- the C ABI of include/tcgemm.h: argument validation, TMA
// descriptor encoding, the launch plan and the launch.
//
// The host sequence follows "CUTLASS" (stanleyjacob.dev), Part IV Stage 1:
// size the workspace, validate the problem against what the kernel can do
// (can_implement), then run one kernel launch.  The planner plays the role of
// the collective builder's StageCountAuto (the CUTLASS/CuTe/CUDA Tile page,
// "Assembling a CUTLASS kernel": the stage count is whatever fits in shared
// memory at one CTA per SM) and of the tile scheduler (grid size, raster
// group, split-K for shapes with too few output tiles, Part III / Part IV
// Stage 2 and Stage 6).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <string>
#include <vector>

#include "../../include/tcgemm.h"
#include "gemm_kernel.cuh"
#include "launch.cuh"
#include "pack_kernel.cuh"

namespace {

thread_local std::string g_last_error;

// Test-only knobs (tcg_debug_set).
int g_fault_inject = 0;
long long g_timeout_ns = 0;
int g_force_splits = 0;
int g_force_cta2 = 0;
constexpr long long kDefaultTimeoutNs = 2000000000LL;  // 2 s

constexpr size_t kHeaderBytes = 256;  // status word + diagnostics

// Planner overrides for tuning experiments (environment, read once):
// TCG_GROUP_M = raster group in M blocks, TCG_STAGES = pipeline depth cap.
int env_int(const char* name) {
    const char* v = getenv(name);
    return v ? atoi(v) : 0;
}
const int g_env_group_m = env_int("TCG_GROUP_M");
const int g_env_stages = env_int("TCG_STAGES");
// TCG_STATS=1: accumulate per-role cycle counts into workspace bytes 64..127.
const int g_env_stats = env_int("TCG_STATS");
// TCG_KATOMS = K atoms per stage for pair tiles (1 or 2; default 2).
const int g_env_katoms = env_int("TCG_KATOMS");
// width of block-scaled pair tiles (192 or 256; 0 = the format's default)
const int g_env_mx_bn = env_int("TCG_MX_BN");
// TCG_SK: Stream-K schedule.  0 = off (data-parallel tiles, split-K for
// shapes with too few tiles); 1 = the last partial wave plus one full wave
// as one Stream-K run, the rest data-parallel; 2 = only the last partial
// wave; 3 = every tile (also replaces split-K).  Unset = the default below.
const int g_env_sk = getenv("TCG_SK") ? env_int("TCG_SK") : -1;
// TCG_NARROW=0 keeps 128/256-wide tiles for small problems (default: narrow them).
const int g_env_narrow = getenv("TCG_NARROW") ? env_int("TCG_NARROW") : 1;
// TCG_SKINNY_PAIRS=0 keeps one-CTA tiles for split-K problems with at most 128 columns.
const int g_env_skinny_pairs = getenv("TCG_SKINNY_PAIRS") ? env_int("TCG_SKINNY_PAIRS") : 1;
// TCG_SWAP=1 runs GEMMs with at most 64 rows as the transposed product (use_swap).
const int g_env_swap = env_int("TCG_SWAP");
// TCG_TMA_STORE=1 / 0: every chunk of D staged in shared memory for a TMA store,
// or whole chunks stored from registers (a ragged last chunk is always staged).
// Unset: from registers.
const int g_env_tma_store = getenv("TCG_TMA_STORE") ? env_int("TCG_TMA_STORE") : -1;
// TCG_KSERP=0: every unit walks K upwards (default: odd waves downwards, see work_next).
const int g_env_kserp = getenv("TCG_KSERP") ? env_int("TCG_KSERP") : 1;
// TCG_ST32=0: the register-store epilogue writes 16-byte pieces even where
// D allows 32-byte stores (default 1).
const int g_env_st32 = getenv("TCG_ST32") ? env_int("TCG_ST32") : 1;
// TCG_HALF_TAIL=0 never runs the last wave as half-width tiles, =2 always when it fits.
const int g_env_half_tail = getenv("TCG_HALF_TAIL") ? env_int("TCG_HALF_TAIL") : 1;
// TCG_PAIR_BN = width of 16/8-bit pair tiles (160, 192, 224 or 256) when B is
// K-major; unset = chosen by the wave model in make_plan.
const int g_env_pair_bn = env_int("TCG_PAIR_BN");

tcg_status fail_launch(const char* what, cudaError_t e) {
    char buf[512];
    snprintf(buf, sizeof buf, "%s: %s", what, cudaGetErrorString(e));
    g_last_error = buf;
    return TCG_ERR_LAUNCH;
}

int elem_bytes(tcg_dtype t) {
    switch (t) {
        case TCG_BF16: return 2;
        case TCG_F16: return 2;
        case TCG_E4M3: return 1;
        case TCG_E5M2: return 1;
        case TCG_MXE4M3: return 1;
        case TCG_MXE5M2: return 1;
        case TCG_NVFP4: return 1;  // bytes of two packed elements: FP4 sizes are converted to bytes first
        case TCG_MXFP4: return 1;
        case TCG_F32: return 4;
    }
    return 0;
}

bool is_fp4(tcg_dtype t) { return t == TCG_NVFP4 || t == TCG_MXFP4; }
bool is_mx(tcg_dtype t) { return t == TCG_MXE4M3 || t == TCG_MXE5M2 || is_fp4(t); }  // block-scaled
// K in the kernel's units: bytes for packed FP4, elements otherwise
int k_units(tcg_dtype t, int K) { return is_fp4(t) ? (K + 1) / 2 : K; }
// elements per block scale, and scale blocks (4 scales) per 128-byte K atom
int sf_group(tcg_dtype t) { return t == TCG_NVFP4 ? 16 : 32; }
int sf_blocks_per_atom(tcg_dtype t) { return t == TCG_NVFP4 ? 4 : (t == TCG_MXFP4 ? 2 : 1); }
bool is_fp8(tcg_dtype t) { return t == TCG_E4M3 || t == TCG_E5M2 || is_mx(t); }
bool is_ab_type(tcg_dtype t) { return t == TCG_BF16 || t == TCG_F16 || is_fp8(t); }

// Operand format field of the tcgen05 instruction descriptor: kind::f16
// (F16 = 0, BF16 = 1) and kind::f8f6f4 (E4M3 = 0, E5M2 = 1).
uint32_t mma_format(tcg_dtype t) { return (t == TCG_BF16 || t == TCG_E5M2 || t == TCG_MXE5M2) ? 1u : 0u; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned_to(const void* p, int bytes) { return (reinterpret_cast<uintptr_t>(p) % static_cast<uintptr_t>(bytes)) == 0; }

// A matrix the TMA can stream as stored: 16-byte aligned base and row pitch.
bool tma_addressable(const void* p, long long ld, int eb) { return aligned16(p) && (ld * eb) % 16 == 0; }

// Operand storage as rows: `outer` rows of `inner` contiguous elements.
struct Rows {
    long long inner = 0, outer = 0;
};
Rows operand_rows(int rows, int cols, tcg_layout op) {  // logical rows x cols, stored per op
    Rows r;
    r.inner = op == TCG_ROW ? cols : rows;
    r.outer = op == TCG_ROW ? rows : cols;
    return r;
}

// Leading dimension (elements) of the packed copy: rows padded to 16 bytes.
long long packed_ld(long long inner, int eb) {
    const long long q = 16 / eb;
    return std::max(q, (inner + q - 1) / q * q);
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// Workspace bytes of the packed copy of an operand the TMA cannot address (0 otherwise).
size_t pack_bytes(int rows, int cols, tcg_layout op, const void* ptr, long long ld, int eb) {
    if (rows <= 0 || cols <= 0 || tma_addressable(ptr, ld, eb)) return 0;
    const Rows r = operand_rows(rows, cols, op);
    return round256(static_cast<size_t>(r.outer) * static_cast<size_t>(packed_ld(r.inner, eb)) * eb);
}

// ------------------------------------------------------------ device info

struct DeviceInfo {
    bool valid = false;
    int major = 0, minor = 0;
    int num_sms = 0;
    int max_smem_optin = 0;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[64];

tcg_status device_info(DeviceInfo& out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_launch("cudaGetDevice", e);
    if (dev < 0 || dev >= 64) { g_last_error = "device index out of range"; return TCG_ERR_LAUNCH; }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.valid) {
        if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
                cudaSuccess)
            return fail_launch("cudaDeviceGetAttribute", e);
        d.valid = true;
    }
    out = d;
    return TCG_OK;
}

// Whether this process sees any CUDA device (asked once).  Without one,
// tcg_can_implement validates the arguments alone (the CPU tests and tools).
bool have_device() {
    static std::once_flag once;
    static bool present = false;
    std::call_once(once, [] {
        int n = 0;
        if (cudaGetDeviceCount(&n) == cudaSuccess) present = n > 0;
        else cudaGetLastError();
    });
    return present;
}

tcg_status arch_check(const DeviceInfo& dev) {
    const tcg_status st = tcg_arch_status(dev.major, dev.minor);
    if (st != TCG_OK) {
        char buf[128];
        snprintf(buf, sizeof buf, "compute capability %d.%d is not 10.3 (sm_103a)", dev.major, dev.minor);
        g_last_error = buf;
    }
    return st;
}

// Per-call checks of the scale arguments that tcg_can_implement does not see.
tcg_status check_scales(const tcg_scales& scales, tcg_dtype ab_dtype, int K) {
    if (scales.col_scale && !aligned_to(scales.col_scale, 4)) return TCG_ERR_MISALIGNED;
    if (scales.row_scale && !aligned_to(scales.row_scale, 4)) return TCG_ERR_MISALIGNED;
    if (is_mx(ab_dtype) && K > 0) {
        if (!scales.block_sfa || !scales.block_sfb) return TCG_ERR_INVALID_ARG;
        if (!aligned16(scales.block_sfa) || !aligned16(scales.block_sfb)) return TCG_ERR_MISALIGNED;
    }
    return TCG_OK;
}

// ------------------------------------------------------------- tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

tcg_status get_encoder(EncodeTiledFn& fn) {
    std::call_once(g_encode_once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(f);
    });
    if (!g_encode) { g_last_error = "cuTensorMapEncodeTiled entry point not found"; return TCG_ERR_LAUNCH; }
    fn = g_encode;
    return TCG_OK;
}

CUtensorMapDataType tma_dtype(tcg_dtype t) {
    switch (t) {
        case TCG_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        case TCG_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        case TCG_E4M3: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
        case TCG_E5M2: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
        case TCG_MXE4M3: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
        case TCG_MXE5M2: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
        case TCG_NVFP4: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
        case TCG_MXFP4: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
        default: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    }
}

// A 2-D row-major view: `inner` contiguous elements per row, `outer` rows
// ld_elems apart; boxes of box_inner x box_outer elements.
// The descriptor is a pure function of its arguments, so encoded maps are
// kept in a small process-wide cache (a call with the same pointers and
// shapes as an earlier one skips the encode).  Bounded: cleared when full.
struct MapKey {
    int dtype;
    const void* base;
    uint64_t inner, outer, ld_elems;
    uint32_t box_inner, box_outer;
    int sw;
    bool operator<(const MapKey& o) const {
        return std::tie(dtype, base, inner, outer, ld_elems, box_inner, box_outer, sw) <
               std::tie(o.dtype, o.base, o.inner, o.outer, o.ld_elems, o.box_inner, o.box_outer, o.sw);
    }
};
std::mutex g_map_mu;
std::map<MapKey, CUtensorMap> g_map_cache;
constexpr size_t kMapCacheMax = 1024;

tcg_status encode_2d(CUtensorMap* map, tcg_dtype t, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t ld_elems, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    const MapKey key{static_cast<int>(t), base, inner, outer, ld_elems, box_inner, box_outer, static_cast<int>(sw)};
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_map_cache.find(key);
        if (it != g_map_cache.end()) {
            *map = it->second;
            return TCG_OK;
        }
    }
    EncodeTiledFn fn;
    tcg_status st = get_encoder(fn);
    if (st != TCG_OK) return st;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {ld_elems * static_cast<uint64_t>(elem_bytes(t))};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, tma_dtype(t), 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[256];
        snprintf(buf, sizeof buf,
                 "cuTensorMapEncodeTiled failed (%d): dims %llu x %llu, ld %llu, box %u x %u", static_cast<int>(r),
                 (unsigned long long)inner, (unsigned long long)outer, (unsigned long long)ld_elems, box_inner,
                 box_outer);
        g_last_error = buf;
        return TCG_ERR_LAUNCH;
    }
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_map_cache.size() >= kMapCacheMax) g_map_cache.clear();
    g_map_cache.emplace(key, *map);
    return TCG_OK;
}

// --------------------------------------------------------------- planning

struct Plan {
    int bn = 256;
    int stages = 4;
    int splits = 1;
    int grid = 1;
    int units = 0;
    int group_m = 8;
    int smem = 0;
    int num_m = 0, num_n = 0, num_kb = 0;
    int cluster = 1;
    int katoms = 1;     // 128-byte K atoms per pipeline stage
    int units_a = 0;    // units of the data-parallel phase (tiles x splits)
    int sk_tiles = 0;   // tiles of the Stream-K phase (the last ones in raster order)
    int workers = 0;    // CTAs or CTA pairs
    bool swap = false;  // the transposed product D^T = B^T A^T (sizes and tiles in its frame)
    int half_tail = 0;  // last tiles run as two half-width units each (wave_fit)
};

int stage_bytes(int bn, bool cta2, int katoms, int sf_blocks = 0) {
    // block-scaled stages also hold sf_blocks 512-byte scale blocks (A's and B's) per atom
    return katoms * (tcg::kBM + (cta2 ? bn / 2 : bn)) * tcg::kRowBytes + (katoms * sf_blocks * 512 + 1023) / 1024 * 1024;
}

int fixed_smem_bytes(bool small_ring = false) {
    return 1024 /*alignment slack*/ + 4 * tcg::epi_warp_bytes(small_ring) + static_cast<int>(sizeof(tcg::SmemCtl)) + 64;
}

int max_active_pairs(int bn, bool fp8, int katoms, int smem);

// The last wave of 256-wide pair tiles, by the wave model: the modelled
// time of a launch is its waves x (tile width + a per-tile fixed cost), a
// tile's MMA time growing with width x K and the fixed cost (the accumulator
// hand-off and first loads, about two microseconds, measured as a share of
// the MMA loop on GB300) expressed in the same units, 1e5 / K columns.  Wave
// quantisation ("CUTLASS", Part IV Stage 2 and Part XI: the last, partly
// filled wave of tiles) has two remedies here, each taken only when it saves
// at least 3 % over plain 256-wide tiles:
//   * a half-width tail: when the last wave would use at most half of the
//     workers, its tiles run as two 256 x 128 units each (same kernel, no
//     partial sums), so that wave ends in half the time;
//   * a narrower tile for the whole launch (224, 192 or 160 wide; B K-major
//     only), at the price of more operand bytes per FLOP.
struct WaveFit {
    int bn = 256;
    int half_tail = 0;   // tiles of the last wave run as two half-width units
};

WaveFit wave_fit(int num_m2, int N, int K, int slots, bool narrow_ok) {
    WaveFit best;
    if (g_env_pair_bn == 160 || g_env_pair_bn == 192 || g_env_pair_bn == 224 || g_env_pair_bn == 256) {
        best.bn = narrow_ok || g_env_pair_bn == 256 ? g_env_pair_bn : 256;
        return best;
    }
    if (slots <= 0) return best;
    const double fixed = 1e5 / std::max(K, 1);
    const long long tiles = static_cast<long long>(num_m2) * ((N + 255) / 256);
    const long long full = tiles / slots, rem = tiles % slots;
    const double plain = static_cast<double>((tiles + slots - 1) / slots) * (256 + fixed);
    double best_cost = plain * 0.97;
    if (g_env_half_tail != 0 && rem > 0 && 2 * rem <= slots) {
        const double c = static_cast<double>(full) * (256 + fixed) + (128 + fixed);
        if (c < best_cost || g_env_half_tail == 2) {
            best.half_tail = static_cast<int>(rem);
            best_cost = c;
        }
    }
    if (narrow_ok) {
        for (int bn : {224, 192, 160}) {
            const long long t = static_cast<long long>(num_m2) * ((N + bn - 1) / bn);
            const double c = static_cast<double>((t + slots - 1) / slots) * (bn + fixed);
            if (c < best_cost) {
                best.bn = bn;
                best.half_tail = 0;
                best_cost = c;
            }
        }
    }
    return best;
}

// A GEMM with few rows (M <= 64 of one 128-row tile) can run as the
// transposed product D^T = B^T A^T: its 128-row tiles run over D's N columns
// and its narrow N (32 or 64) covers D's rows, so the tensor cores compute no
// padding rows and the split-K partials shrink to 128 x 32.  It needs a
// K-contiguous A (A^T becomes the kernel's K-major B) and plain operands.
// Measured on GB300 it does not pay: every such problem is bound by the
// bytes of B, which the plain plan streams as fast (16 x 8192 x 8192, bias,
// beta = 0.5: 38.9 us plain with split K 4, 43.0 - 53 us transposed in every
// split and stage configuration), so it is taken only on request
// (TCG_SWAP=1, or the test knob force_cta2 = 5).
bool use_swap(int M, int N, tcg_dtype ab, tcg_layout opA) {
    return (g_env_swap == 1 || g_force_cta2 == 5) && !is_mx(ab) && M > 0 && M <= 64 && N >= 256 &&
           opA == TCG_ROW;
}

Plan make_plan(int M, int N, int K_elems, tcg_dtype ab, const DeviceInfo& dev, int sk_override = -1,
               bool b_kmajor = true, bool swap = false) {
    Plan pl;
    pl.swap = swap;
    const int K = k_units(ab, K_elems);
    const int bk = tcg::kRowBytes / elem_bytes(ab);
    const bool mx = is_mx(ab);   // block-scaled: 128 x 128 (one CTA) or 256 x BN (a pair) tiles
    pl.bn = (N <= 128) ? 128 : 256;
    if (swap) pl.bn = N <= 32 ? 32 : 64;   // the kernel's N is D's row count
    if (mx) {
        // Pair tiles: 256 x 256 with one accumulator (the scales take the TMEM
        // columns of a second one), or 256 x 192 with two accumulators, so
        // that one tile's epilogue overlaps the next tile's MMAs (not for
        // NVFP4, whose four scale blocks per atom leave no room).  Measured
        // on 8192^3 (TFLOP/s, 256 wide vs 192 wide): MXFP8 2393 vs 2151,
        // MXFP4 3353 vs 3313 (with the epilogue's staged bias and direct
        // stores; before them MXFP4 was 3019 vs 3300), so 256 by default.
        int pbn = 256;
        if (g_env_mx_bn == 192 || g_env_mx_bn == 256) pbn = g_env_mx_bn;
        if (g_force_cta2 == 3) pbn = 256;
        if (g_force_cta2 == 4) pbn = 192;
        if (ab == TCG_NVFP4) pbn = 256;
        // pairs when there is a full wave of pair tiles, else one CTA per 128 x 128
        const int pairs = ((M + 255) / 256) * ((N + pbn - 1) / pbn);
        bool pair = M > tcg::kBM && N > 128 && pairs * 2 >= dev.num_sms && g_force_splits == 0;
        if (g_force_cta2 == 1 || g_force_cta2 >= 3) pair = N > 128 && g_force_splits <= 1;
        if (g_force_cta2 == 2) pair = false;
        pl.bn = pair ? pbn : 128;
    }
    // K atoms per stage are decided with the tile shape below; the split-K
    // heuristic works on single-atom k-blocks.
    pl.num_kb = (K + bk - 1) / bk;
    const int num_m1 = (M + tcg::kBM - 1) / tcg::kBM;
    // Short K (too short to split): narrower tiles (down to 128 x 64, one full
    // 128-byte MN atom, so an MN-major B box still fits its stage) while the
    // tiles would fill less than half of the SMs.  Measured on GB300: 512^3
    // 12.4 -> 10.3 us; for long K, split-K beats narrowing (16x8192x8192:
    // 49 vs 60 us).
    if (!mx && !swap && g_env_narrow && g_force_splits == 0 && g_force_cta2 != 1 && g_force_cta2 < 3 && pl.num_kb < 16) {
        while (pl.bn > 64 && num_m1 * ((N + pl.bn - 1) / pl.bn) * 2 < dev.num_sms) pl.bn /= 2;
    }
    const int num_n = (N + pl.bn - 1) / pl.bn;
    const int tiles1 = num_m1 * num_n;
    // Split K only when the output tiles cannot fill the machine and each
    // split keeps a useful number of k-blocks.
    int splits = 1;
    if (g_force_splits > 0) {
        splits = g_force_splits;
    } else if (tiles1 * 2 <= dev.num_sms && pl.num_kb >= 16) {
        splits = std::min(dev.num_sms / tiles1, pl.num_kb / 8);
        splits = std::max(1, std::min(splits, 16));
    }
    splits = std::max(1, std::min(splits, std::max(pl.num_kb, 1)));
    if (mx && pl.bn > 128) splits = 1;   // block-scaled pair tiles do not split K
    // 2-CTA pair tiles (256 x BN) when K is not split and there is at least
    // one full wave of pairs; they halve the operand bytes each SM streams.
    const int num_m2 = (M + 2 * tcg::kBM - 1) / (2 * tcg::kBM);
    bool cta2 = splits == 1 && pl.bn == 256 && M > tcg::kBM && num_m2 * num_n * 2 >= dev.num_sms;
    // Long K, a tall A and at most 128 output columns (e.g. 8192 x 128 x 8192):
    // 256 x 128 pair tiles with split K.  Each CTA streams its own 128 rows of
    // A and only half of B's 128 columns, so a stage holds 16 KiB of A (from
    // DRAM) and 8 KiB of B (from L2) per K atom instead of 16 + 16, and twice
    // as many bytes of A are in flight per SM.
    if (!mx && !swap && splits > 1 && pl.bn == 128 && N <= 128 && num_m2 >= 8 && g_env_skinny_pairs && g_env_katoms != 1 &&
        g_force_splits == 0 && g_force_cta2 == 0) {
        const int tiles2 = num_m2 * num_n;
        splits = std::max(1, std::min(std::min((dev.num_sms / 2) / tiles2, pl.num_kb / 8), 16));
        cta2 = splits > 1;
    }
    if (g_force_cta2 == 1 || g_force_cta2 >= 3) cta2 = splits == 1 && pl.bn == 256;
    if (mx) cta2 = pl.bn > 128;
    if (g_force_cta2 == 2 || g_force_cta2 == 5 || swap) cta2 = false;
    pl.cluster = cta2 ? 2 : 1;
    pl.katoms = cta2 ? (g_env_katoms == 1 ? 1 : 2) : (g_env_katoms == 2 && pl.bn >= 128 ? 2 : 1);
    // the transposed product's small stages: two K atoms each (16 x 8192 x 8192:
    // 43 vs 50 us with one); its pipeline then holds four
    if (swap) pl.katoms = g_env_katoms == 1 ? 1 : 2;
    // block-scaled: two K atoms per stage on pair tiles, else one.  Measured on
    // 8192^3: MXFP8 pairs 1841 -> 2199 TFLOP/s (6 x 1 atom -> 3 x 2), NVFP4
    // pairs 2217 -> 2515 (5 x 1 -> 2 x 2)
    if (mx) pl.katoms = g_env_katoms > 0 ? std::min(g_env_katoms, 2) : (cta2 ? 2 : 1);
    if (mx && is_fp4(ab) && !cta2) pl.katoms = 1;
    if (mx && pl.bn == 192) pl.katoms = 2;
    // scale blocks per stage atom: A's rows, then B's columns (a pair holds the
    // two 128-column blocks its 192 or 256 columns overlap)
    const int sfb = mx ? sf_blocks_per_atom(ab) * (1 + (pl.bn > 128 ? 2 : 1)) : 0;
    pl.num_kb = (K + pl.katoms * bk - 1) / (pl.katoms * bk);
    pl.num_m = cta2 ? num_m2 : num_m1;
    pl.num_n = num_n;
    pl.splits = splits;
    const int tiles = pl.num_m * pl.num_n;
    pl.units_a = tiles * splits;
    pl.units = pl.units_a;
    // Raster group (in M blocks): 16 pair rows (or 16 rows of one-CTA tiles).
    // With the K-serpentine order (odd waves walk K downwards, so a wave that
    // revisits a group's rows of A starts on the K slabs loaded last) the
    // 8192^3 GELU launch moves 0.98 GB of DRAM instead of 1.20 GB with 8 pair
    // rows in one K direction, at the same speed in short runs and 1.8 %
    // faster in a 1000-launch run under the power cap (1627 vs 1598 TFLOP/s,
    // 1901 vs 1876 MHz median on the same GPU): less DRAM traffic leaves
    // more power to the SMs.
    pl.group_m = 16;
    if (g_env_group_m > 0) pl.group_m = g_env_group_m;
    const bool small_ring = mx && cta2 && pl.bn == 256;   // 256-wide block-scaled pairs: half-size epilogue ring
    int stages = (dev.max_smem_optin - fixed_smem_bytes(small_ring)) / stage_bytes(pl.bn, cta2, pl.katoms, sfb);
    // (the transposed plan's small stages stream B from DRAM: deeper)
    stages = std::max(2, std::min(stages, swap ? 12 : 8));
    if (mx) {
        // TMEM: accumulators (2 x 128 or 2 x 192 columns, or one 256-column pair
        // accumulator) plus 4 columns per scale block per stage atom
        const int sf_cols = 512 - (pl.bn == 192 ? 2 * 192 : 256);
        stages = std::max(2, std::min(stages, sf_cols / (4 * sfb * pl.katoms)));
    }
    if (g_env_stages > 1) stages = std::min(stages, g_env_stages);
    pl.stages = stages;
    pl.smem = fixed_smem_bytes(small_ring) + stages * stage_bytes(pl.bn, cta2, pl.katoms, sfb);
    int slots = dev.num_sms;  // units that run at once
    if (cta2) {
        slots = max_active_pairs(pl.bn, is_fp8(ab), pl.katoms, pl.smem);
        if (slots <= 0) slots = dev.num_sms / 2;
    }
    // Stream-K: balance the k-block iterations of the last tiles over all
    // workers instead of leaving the last wave partly empty.
    const int sk_mode = sk_override >= 0 ? sk_override : (g_env_sk >= 0 ? g_env_sk : 0);
    // Otherwise a half-width tail or a narrower pair tile (wave_fit).
    if (cta2 && !mx && pl.bn == 256 && pl.splits == 1 && sk_mode == 0 && g_force_splits == 0 && pl.katoms == 2 &&
        g_force_cta2 < 3) {
        // K in bf16-equivalent elements (an 8-bit K element costs half the MMA time)
        const WaveFit wf = wave_fit(pl.num_m, N, K * elem_bytes(ab) / 2, slots, b_kmajor);
        const int bn = wf.bn;
        if (wf.half_tail > 0) {
            pl.half_tail = wf.half_tail;
            pl.units_a = pl.num_m * pl.num_n - wf.half_tail;
            pl.units = pl.units_a + 2 * wf.half_tail;
        }
        if (bn != pl.bn) {
            pl.bn = bn;
            pl.num_n = (N + bn - 1) / bn;
            stages = (dev.max_smem_optin - fixed_smem_bytes()) / stage_bytes(bn, true, pl.katoms);
            stages = std::max(2, std::min(stages, 8));
            if (g_env_stages > 1) stages = std::min(stages, g_env_stages);
            pl.stages = stages;
            pl.smem = fixed_smem_bytes() + stages * stage_bytes(bn, true, pl.katoms);
            pl.units_a = pl.units = pl.num_m * pl.num_n;
        }
    }
    if (g_force_splits == 0 && pl.num_kb > 0 && sk_mode > 0) {
        const int rem = tiles % slots;
        if (sk_mode == 3) {
            pl.sk_tiles = tiles;
        } else if (splits == 1 && rem > 0) {
            pl.sk_tiles = (sk_mode == 1 && tiles >= 2 * slots) ? rem + slots : rem;
        }
        // every worker must own at least one iteration (a piece count per
        // tile then equals the number of workers that touch it)
        if (static_cast<long long>(pl.sk_tiles) * pl.num_kb < slots) pl.sk_tiles = 0;
        if (pl.sk_tiles > 0) {
            pl.splits = 1;
            pl.units_a = tiles - pl.sk_tiles;
            pl.units = pl.units_a;
        }
    }
    pl.workers = pl.sk_tiles > 0 ? slots : std::max(1, std::min(pl.units, slots));
    pl.grid = (cta2 ? 2 : 1) * pl.workers;
    return pl;
}

// The plan tcg_gemm runs for this problem and these layouts: the transposed
// product for GEMMs with few rows (use_swap), else the plain one.
Plan plan_gemm(int M, int N, int K, tcg_dtype ab, const DeviceInfo& dev, tcg_layout opA, tcg_layout opB) {
    if (use_swap(M, N, ab, opA)) return make_plan(N, M, K, ab, dev, -1, true, true);
    return make_plan(M, N, K, ab, dev, -1, opB == TCG_COL);
}

size_t partial_slots(const Plan& pl) {
    const size_t a = pl.splits > 1 ? static_cast<size_t>(pl.units_a) : 0;
    const size_t b = pl.sk_tiles > 0 ? 2 * static_cast<size_t>(pl.workers) : 0;
    return (a + b) * static_cast<size_t>(pl.cluster);
}

bool any_split(const Plan& pl) { return pl.splits > 1 || pl.sk_tiles > 0; }

size_t partial_bytes(const Plan& pl) {
    return partial_slots(pl) * tcg::kBM * pl.bn * sizeof(float);
}

size_t counter_bytes(const Plan& pl) {
    if (!any_split(pl)) return 0;
    return (static_cast<size_t>(pl.num_m) * pl.num_n * pl.cluster * sizeof(int) + 255) / 256 * 256;
}

// Workspace of one tcg_gemm call, in the order it is laid out: the status
// header, then the split-K arrival counters and fp32 partials of its plan
// (`base`), then the packed copies of A and B that the TMA cannot address as
// stored (block-scaled operands are never packed: they must be aligned).
struct WorkspaceNeed {
    size_t base = 0, pack_a = 0, pack_b = 0;
    size_t total() const { return base + pack_a + pack_b; }
};

WorkspaceNeed workspace_need(const Plan& pl, int M, int N, int K, tcg_dtype ab, const void* A, int lda,
                             tcg_layout opA, const void* B, int ldb, tcg_layout opB) {
    WorkspaceNeed w;
    w.base = kHeaderBytes + counter_bytes(pl) + partial_bytes(pl);
    if (K > 0 && !is_mx(ab)) {
        const int eb = elem_bytes(ab);
        w.pack_a = pack_bytes(M, K, opA, A, lda, eb);
        w.pack_b = pack_bytes(K, N, opB, B, ldb, eb);
    }
    return w;
}

// Plan of a grouped GEMM: one tile shape for every problem, 256 x 256 pair
// tiles when the problems' pair tiles fill the device at least once, else
// 128 x 256 tiles on single CTAs; no split K.  `tiles` receives each
// problem's tile count.
Plan make_grouped_plan(const std::vector<tcg_problem>& probs, tcg_dtype ab, const DeviceInfo& dev,
                       std::vector<int>* tiles) {
    Plan pl;
    pl.bn = 256;
    long long pair_tiles = 0;
    for (const tcg_problem& q : probs)
        pair_tiles += static_cast<long long>((q.M + 255) / 256) * ((q.N + pl.bn - 1) / pl.bn);
    bool cta2 = pair_tiles * 2 >= dev.num_sms;
    if (g_force_cta2 == 1) cta2 = true;
    if (g_force_cta2 == 2) cta2 = false;
    pl.cluster = cta2 ? 2 : 1;
    pl.katoms = cta2 ? 2 : 1;
    pl.group_m = g_env_group_m > 0 ? g_env_group_m : (cta2 ? 8 : 16);
    int stages = (dev.max_smem_optin - fixed_smem_bytes()) / stage_bytes(pl.bn, cta2, pl.katoms);
    stages = std::max(2, std::min(stages, 8));
    if (g_env_stages > 1) stages = std::min(stages, g_env_stages);
    pl.stages = stages;
    pl.smem = fixed_smem_bytes() + stages * stage_bytes(pl.bn, cta2, pl.katoms);
    const int tile_m = cta2 ? 2 * tcg::kBM : tcg::kBM;
    long long units = 0;
    if (tiles) tiles->clear();
    for (const tcg_problem& q : probs) {
        const long long t = static_cast<long long>((q.M + tile_m - 1) / tile_m) * ((q.N + pl.bn - 1) / pl.bn);
        if (tiles) tiles->push_back(static_cast<int>(t));
        units += t;
    }
    pl.num_kb = 0;
    pl.splits = 1;
    pl.units = pl.units_a = static_cast<int>(std::min<long long>(units, 1LL << 30));
    int slots = dev.num_sms;
    if (cta2) {
        slots = max_active_pairs(pl.bn, is_fp8(ab), pl.katoms, pl.smem);
        if (slots <= 0) slots = dev.num_sms / 2;
    }
    pl.workers = std::max(1, std::min(pl.units, slots));
    pl.grid = (cta2 ? 2 : 1) * pl.workers;
    return pl;
}

size_t grouped_table_bytes(int n) {
    return (static_cast<size_t>(n) * sizeof(tcg::KernelParams) + static_cast<size_t>(n + 1) * sizeof(int) + 255) /
           256 * 256;
}

template <int BN, bool kFp8, int KA>
int active_pairs_for(int smem) {
    if (tcg::set_smem_attr<BN, kFp8, true, KA>() != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(tcg::kNumThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tcg::gemm_persistent_kernel<BN, kFp8, true, KA>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// Pairs of CTAs that fit on the device at once, per (BN, dtype, smem), cached.
int max_active_pairs(int bn, bool fp8, int katoms, int smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_tuple(dev, bn, (fp8 ? 1 : 0) + 2 * katoms, smem);
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (bn == 256 && katoms == 2) n = fp8 ? active_pairs_for<256, true, 2>(smem) : active_pairs_for<256, false, 2>(smem);
    if (bn == 256 && katoms == 1) n = fp8 ? active_pairs_for<256, true, 1>(smem) : active_pairs_for<256, false, 1>(smem);
    // narrower pairs (192-wide block-scaled, the wave-fitting widths): residency
    // is set by the shared memory, the block size and the cluster shape, which
    // the 256-wide kernel shares
    if (bn != 256) n = fp8 ? active_pairs_for<256, true, 2>(smem) : active_pairs_for<256, false, 2>(smem);
    cache[key] = n;
    return n;
}

tcg::LaunchShape launch_shape(const Plan& pl) { return tcg::LaunchShape{pl.grid, pl.smem, pl.cluster}; }

template <int BN, bool kFp8, bool kCta2, int KA>
tcg_status launch_kernel(const tcg::KernelParams& kp, const Plan& pl, cudaStream_t stream) {
    const char* what = "launch";
    const cudaError_t e = tcg::launch_instance<BN, kFp8, kCta2, KA>(kp, launch_shape(pl), stream, &what);
    return e == cudaSuccess ? TCG_OK : fail_launch(what, e);
}

}  // namespace

// =================================================================== C ABI

extern "C" {

const char* tcg_last_error(void) { return g_last_error.c_str(); }

void tcg_debug_set(int fault_inject, long long wait_timeout_ns, int force_splits, int force_cta2) {
    g_fault_inject = fault_inject;
    g_timeout_ns = wait_timeout_ns;
    g_force_splits = force_splits;
    g_force_cta2 = force_cta2;
}

tcg_status tcg_can_implement(int M, int N, int K, tcg_dtype ab_dtype, const void* A, int lda, tcg_layout opA,
                             const void* B, int ldb, tcg_layout opB, int has_c, const void* C, int ldc,
                             tcg_dtype c_dtype, const void* D, int ldd, tcg_dtype d_dtype, tcg_epilogue epi) {
    if (M < 0 || N < 0 || K < 0) return TCG_ERR_INVALID_ARG;
    if (!is_ab_type(ab_dtype)) return TCG_ERR_INVALID_ARG;
    if ((opA != TCG_ROW && opA != TCG_COL) || (opB != TCG_ROW && opB != TCG_COL)) return TCG_ERR_INVALID_ARG;
    if (d_dtype != TCG_BF16 && d_dtype != TCG_F32) return TCG_ERR_INVALID_ARG;
    if (has_c && c_dtype != TCG_BF16 && c_dtype != TCG_F32) return TCG_ERR_INVALID_ARG;
    if (epi.act != TCG_ACT_NONE && epi.act != TCG_ACT_RELU && epi.act != TCG_ACT_GELU) return TCG_ERR_INVALID_ARG;
    if (epi.bias && epi.bias_dtype != TCG_BF16 && epi.bias_dtype != TCG_F32) return TCG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return TCG_OK;
    if (!D) return TCG_ERR_INVALID_ARG;
    if (has_c && !C) return TCG_ERR_INVALID_ARG;
    if (K > 0 && (!A || !B)) return TCG_ERR_INVALID_ARG;
    // leading dimensions cover the contiguous extent
    if (K > 0) {
        if (lda < (opA == TCG_ROW ? K : M)) return TCG_ERR_INVALID_ARG;
        if (ldb < (opB == TCG_ROW ? N : K)) return TCG_ERR_INVALID_ARG;
    }
    if (ldd < N) return TCG_ERR_INVALID_ARG;
    if (has_c && ldc < N) return TCG_ERR_INVALID_ARG;
    if (is_fp8(ab_dtype) && (opA != TCG_ROW || opB != TCG_COL)) return TCG_ERR_UNSUPPORTED;
    if (is_mx(ab_dtype) && K > 0) {
        // block-scaled operands take the fast path only; FP4 rows are whole bytes
        const int per_byte = is_fp4(ab_dtype) ? 2 : 1;
        if (is_fp4(ab_dtype) && ((K % 2) || (lda % 2) || (ldb % 2))) return TCG_ERR_UNSUPPORTED;
        if (!aligned16(A) || !aligned16(B) || ((static_cast<long long>(lda) / per_byte) % 16) ||
            ((static_cast<long long>(ldb) / per_byte) % 16))
            return TCG_ERR_UNSUPPORTED;
    }
    // Every pointer aligned to its element size.  Operands and outputs whose
    // base or row pitch is not a multiple of 16 bytes are still implemented:
    // A and B through a packed copy in the workspace, C, D and bias through
    // element-wise loads and stores in the epilogue.
    const int eb = elem_bytes(ab_dtype);
    if (K > 0 && (!aligned_to(A, eb) || !aligned_to(B, eb))) return TCG_ERR_MISALIGNED;
    if (!aligned_to(D, elem_bytes(d_dtype))) return TCG_ERR_MISALIGNED;
    if (has_c && !aligned_to(C, elem_bytes(c_dtype))) return TCG_ERR_MISALIGNED;
    if (epi.bias && !aligned_to(epi.bias, elem_bytes(epi.bias_dtype))) return TCG_ERR_MISALIGNED;
    // The kernels exist for sm_103a only ("A10 CuTe, CUTLASS & CuTile", the
    // pitfalls table: check the architecture a kernel was built for before
    // running it).  Without any CUDA device only the arguments are validated.
    if (have_device()) {
        DeviceInfo dev;
        const tcg_status st = device_info(dev);
        if (st != TCG_OK) return st;
        return arch_check(dev);
    }
    return TCG_OK;
}

tcg_status tcg_arch_status(int major, int minor) {
    return (major == 10 && minor == 3) ? TCG_OK : TCG_ERR_ARCH;
}

size_t tcg_workspace_size(int M, int N, int K, tcg_dtype ab_dtype) {
    if (M < 0 || N < 0 || K < 0) return 0;
    if (!is_ab_type(ab_dtype)) return 0;
    DeviceInfo dev;
    if (device_info(dev) != TCG_OK) {
        // Without a device the split-K part cannot be sized; report the
        // largest plan this library could choose on a 1024-SM device.
        dev.num_sms = 1024;
        dev.max_smem_optin = 232448;
    }
    if (M == 0 || N == 0) return kHeaderBytes;
    // the larger of the plain plan and, for a GEMM with few rows, the transposed one
    size_t base = workspace_need(make_plan(M, N, K, ab_dtype, dev), M, N, K, ab_dtype, nullptr, 0, TCG_ROW, nullptr,
                                 0, TCG_COL).base;
    if (use_swap(M, N, ab_dtype, TCG_ROW))
        base = std::max(base, workspace_need(make_plan(N, M, K, ab_dtype, dev, -1, true, true), M, N, K, ab_dtype,
                                             nullptr, 0, TCG_ROW, nullptr, 0, TCG_COL).base);
    return base;
}

size_t tcg_workspace_size_for(int M, int N, int K, tcg_dtype ab_dtype, const void* A, int lda, tcg_layout opA,
                              const void* B, int ldb, tcg_layout opB) {
    const size_t base = tcg_workspace_size(M, N, K, ab_dtype);
    if (base == 0 || M == 0 || N == 0 || K == 0) return base;
    if ((opA != TCG_ROW && opA != TCG_COL) || (opB != TCG_ROW && opB != TCG_COL)) return 0;
    const WorkspaceNeed w = workspace_need(Plan{}, M, N, K, ab_dtype, A, lda, opA, B, ldb, opB);
    return base + w.pack_a + w.pack_b;   // base covers the plain and the transposed plan
}

tcg_status tcg_workspace_init(void* workspace, size_t bytes, void* stream) {
    if (!workspace) return TCG_ERR_WORKSPACE;
    cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_launch("cudaMemsetAsync", e);
    return TCG_OK;
}

tcg_status tcg_plan(int M, int N, int K, tcg_dtype ab_dtype, tcg_layout opA, tcg_layout opB, int out[11]) {
    if (M < 0 || N < 0 || K < 0 || !out) return TCG_ERR_INVALID_ARG;
    if ((opA != TCG_ROW && opA != TCG_COL) || (opB != TCG_ROW && opB != TCG_COL)) return TCG_ERR_INVALID_ARG;
    DeviceInfo dev;
    tcg_status st = device_info(dev);
    if (st != TCG_OK) return st;
    Plan pl = plan_gemm(M, N, K, ab_dtype, dev, opA, opB);
    const int vals[11] = {tcg::kBM, pl.bn, pl.katoms * tcg::kRowBytes / elem_bytes(ab_dtype), pl.stages, pl.splits,
                          pl.grid, pl.cluster, pl.units, pl.group_m, pl.smem, pl.swap ? 1 : 0};
    memcpy(out, vals, sizeof vals);
    return TCG_OK;
}

tcg_status tcg_gemm(int M, int N, int K, float alpha, const void* A, int lda, tcg_layout opA, const void* B,
                    int ldb, tcg_layout opB, float beta, const void* C, int ldc, tcg_dtype c_dtype, void* D,
                    int ldd, tcg_dtype d_dtype, tcg_epilogue epi, tcg_dtype ab_dtype, tcg_scales scales,
                    void* workspace, size_t workspace_bytes, void* stream_) {
    const int has_c = beta != 0.0f;
    tcg_status st = tcg_can_implement(M, N, K, ab_dtype, A, lda, opA, B, ldb, opB, has_c, C, ldc, c_dtype, D, ldd,
                                      d_dtype, epi);
    if (st != TCG_OK) return st;
    if (M == 0 || N == 0) return TCG_OK;
    DeviceInfo dev;
    if ((st = device_info(dev)) != TCG_OK) return st;
    if ((st = arch_check(dev)) != TCG_OK) return st;
    if ((st = check_scales(scales, ab_dtype, K)) != TCG_OK) return st;
    Plan pl = plan_gemm(M, N, K, ab_dtype, dev, opA, opB);
    const int eb = elem_bytes(ab_dtype);
    const WorkspaceNeed wn = workspace_need(pl, M, N, K, ab_dtype, A, lda, opA, B, ldb, opB);
    const size_t base_need = wn.base, pack_a = wn.pack_a, pack_b = wn.pack_b;
    const size_t need = wn.total();
    if (!workspace || !aligned16(workspace) || workspace_bytes < need) {
        if (pack_a + pack_b > 0) {
            char buf[200];
            snprintf(buf, sizeof buf,
                     "A or B is not 16-byte addressable: the packed copy needs a workspace of %zu bytes "
                     "(tcg_workspace_size_for)", need);
            g_last_error = buf;
        }
        return TCG_ERR_WORKSPACE;
    }
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    // Slow path for operands the TMA cannot address: pack them into 16-byte
    // pitched rows in the workspace (one launch for both), then run the GEMM
    // on the copies.
    if (pack_a + pack_b > 0) {
        tcg::PackParams pp;
        memset(&pp, 0, sizeof pp);
        long long chunks_max = 0;
        auto add_job = [&](const void*& ptr, int& ld, int rows, int cols, tcg_layout op, size_t offset) {
            const Rows r = operand_rows(rows, cols, op);
            const long long ldp = packed_ld(r.inner, eb);
            tcg::PackJob& j = pp.job[pp.njobs++];
            j.src = static_cast<const uint8_t*>(ptr);
            j.src_pitch = static_cast<long long>(ld) * eb;
            j.dst = reinterpret_cast<uint8_t*>(workspace) + offset;
            j.dst_pitch = ldp * eb;
            j.rows = r.outer;
            j.row_bytes = static_cast<int>(r.inner * eb);
            j.chunks = (j.row_bytes + 15) / 16;
            j.total = j.rows * j.chunks;
            chunks_max = std::max(chunks_max, j.total);
            ptr = j.dst;
            ld = static_cast<int>(ldp);
        };
        if (pack_a) add_job(A, lda, M, K, opA, base_need);
        if (pack_b) add_job(B, ldb, K, N, opB, base_need + pack_a);
        const int grid =
            static_cast<int>(std::max(1LL, std::min<long long>((chunks_max + 255) / 256, dev.num_sms * 8LL)));
        tcg::pack_rows_kernel<<<grid, 256, 0, stream>>>(pp);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return fail_launch("pack_rows_kernel", e);
    }

    // Packed FP4 operands are streamed as bytes: K and the leading dimensions in bytes.
    const int K_elems = K;
    if (is_fp4(ab_dtype)) {
        K /= 2;
        lda /= 2;
        ldb /= 2;
    }
    tcg::KernelParams kp;
    memset(&kp, 0, sizeof kp);
    const int bk = tcg::kRowBytes / elem_bytes(ab_dtype);
    const int atom = bk;  // MN elements per 128-byte swizzle row
    if (K > 0 && pl.swap) {
        // The transposed product: the kernel's A is B^T (N x K: rows of K when
        // B is column-major, else rows of N), its B is A^T (K x M, K-major:
        // A is row-major), in boxes of BK x BN rows.
        if (opB == TCG_COL)
            st = encode_2d(&kp.tmA, ab_dtype, B, K, N, ldb, bk, tcg::kBM, CU_TENSOR_MAP_SWIZZLE_128B);
        else
            st = encode_2d(&kp.tmA, ab_dtype, B, N, K, ldb, atom, pl.katoms * bk, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != TCG_OK) return st;
        st = encode_2d(&kp.tmB, ab_dtype, A, K, M, lda, bk, pl.bn, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != TCG_OK) return st;
    } else if (K > 0) {
        // A: K-major -> rows of K, box BK x BM; MN-major -> rows of M, box atom x BK
        if (opA == TCG_ROW)
            st = encode_2d(&kp.tmA, ab_dtype, A, K, M, lda, bk, tcg::kBM, CU_TENSOR_MAP_SWIZZLE_128B);
        else
            st = encode_2d(&kp.tmA, ab_dtype, A, M, K, lda, atom, pl.katoms * bk, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != TCG_OK) return st;
        const int b_rows = pl.cluster == 2 ? pl.bn / 2 : pl.bn;  // B rows one CTA loads
        if (opB == TCG_COL)
            st = encode_2d(&kp.tmB, ab_dtype, B, K, N, ldb, bk, b_rows, CU_TENSOR_MAP_SWIZZLE_128B);
        else
            st = encode_2d(&kp.tmB, ab_dtype, B, N, K, ldb, atom, pl.katoms * bk, CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != TCG_OK) return st;
    }
    kp.d_tma = !pl.swap && tma_addressable(D, ldd, elem_bytes(d_dtype));
    if (kp.d_tma) {
        st = encode_2d(&kp.tmD, d_dtype, D, N, M, ldd, tcg::kEpiChunk, 32,
                       d_dtype == TCG_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
        if (st != TCG_OK) return st;
    }

    kp.M = pl.swap ? N : M;
    kp.N = pl.swap ? M : N;
    kp.K = K;
    kp.num_m_blk = pl.num_m; kp.num_n_blk = pl.num_n; kp.num_kb = pl.num_kb;
    kp.splits = pl.splits; kp.num_units = pl.units; kp.group_m = pl.group_m;
    kp.units_a = pl.units_a;
    kp.sk_tiles = pl.sk_tiles;
    kp.sk_iters = static_cast<long long>(pl.sk_tiles) * pl.num_kb;
    kp.sk_slot_base = pl.splits > 1 ? pl.units_a : 0;
    kp.half_tail = pl.half_tail;
    kp.k_serp = g_env_kserp;
    if (pl.half_tail > 0 && K > 0 && opB == TCG_COL) {
        // the tail's half-width units load half of each CTA's B rows
        st = encode_2d(&kp.tmB2, ab_dtype, B, K, N, ldb, bk, (pl.cluster == 2 ? pl.bn / 2 : pl.bn) / 2,
                       CU_TENSOR_MAP_SWIZZLE_128B);
        if (st != TCG_OK) return st;
    }
    kp.a_mn_major = pl.swap ? (opB == TCG_ROW) : (opA == TCG_COL);
    kp.b_mn_major = pl.swap ? 0 : (opB == TCG_ROW);
    kp.alpha = alpha * scales.scale_a * scales.scale_b;
    kp.ab_fmt = mma_format(ab_dtype);
    // (the transposed product's rows are D's columns)
    kp.row_scale = pl.swap ? scales.col_scale : scales.row_scale;
    kp.col_scale = pl.swap ? scales.row_scale : scales.col_scale;
    kp.sfa = static_cast<const uint8_t*>(scales.block_sfa);
    kp.sfb = static_cast<const uint8_t*>(scales.block_sfb);
    kp.num_sfcb = ((K_elems + sf_group(ab_dtype) - 1) / sf_group(ab_dtype) + 3) / 4;
    if (is_mx(ab_dtype) && pl.cluster == 2 && K > 0) {
        // pair tiles load their scale blocks with the TMA: rows of 128 x 32-bit words
        // (one 512-byte block per row), boxes of the blocks of one K atom
        const uint32_t per_atom = static_cast<uint32_t>(sf_blocks_per_atom(ab_dtype));
        st = encode_2d(&kp.tmSFA, TCG_F32, scales.block_sfa, 128,
                       static_cast<uint64_t>((M + 127) / 128) * kp.num_sfcb, 128, 128, per_atom,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st != TCG_OK) return st;
        st = encode_2d(&kp.tmSFB, TCG_F32, scales.block_sfb, 128,
                       static_cast<uint64_t>((N + 127) / 128) * kp.num_sfcb, 128, 128, per_atom,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st != TCG_OK) return st;
    }
    kp.beta = beta;
    kp.C = has_c ? C : nullptr;
    kp.ldc = ldc;
    kp.c_f32 = (c_dtype == TCG_F32);
    kp.c_vec = !pl.swap && has_c && tma_addressable(C, ldc, elem_bytes(c_dtype));
    kp.c_tma = kp.c_vec;
    if (kp.c_tma) {
        st = encode_2d(&kp.tmC, c_dtype, C, N, M, ldc, tcg::kEpiChunk, 32,
                       c_dtype == TCG_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
        if (st != TCG_OK) return st;
    }
    {
        // chunk buffers per epilogue warp: 8 KiB over the larger of the C and D boxes
        const int box = 32 * 32 * std::max(elem_bytes(d_dtype), kp.c_tma ? elem_bytes(c_dtype) : 0);
        kp.epi_nbuf = tcg::epi_warp_bytes(is_mx(ab_dtype) && pl.cluster == 2 && pl.bn == 256) / box;
    }
    kp.cs_vec = !pl.swap && scales.col_scale && aligned16(scales.col_scale);
    kp.bias = epi.bias;
    kp.bias_f32 = (epi.bias_dtype == TCG_F32);
    kp.act = static_cast<int>(epi.act);
    kp.d_f32 = (d_dtype == TCG_F32);
    kp.D = D;
    kp.ldd = ldd;
    kp.d_inner_aligned = (static_cast<long long>(N) * elem_bytes(d_dtype)) % 16 == 0;
    kp.d_v32 = g_env_st32 && reinterpret_cast<uintptr_t>(D) % 32 == 0 &&
               (static_cast<long long>(ldd) * elem_bytes(d_dtype)) % 32 == 0;
    // D's store path: whole chunks from registers (32-byte stores where D's
    // base and pitch allow) by default.  Measured on GB300 against staging
    // every chunk for a TMA store (one GPU, median of 30 launches, twice
    // each): 4095 x 3001 x 1537 51.7-51.8 vs 54.0 us, 16 x 8192 x 8192
    // 40.1-40.6 vs 41.2, 8192 x 128 x 8192 43.5 vs 43.8, 4096^3 96.5-96.6 vs
    // 96.7-97.0, 8192^3 GELU 594.4-594.7 vs 595.5, e4m3 and the grouped MoE
    // within 0.2 %; the block-scaled kernels, whose epilogue is not hidden
    // behind a second accumulator, gained most from registers when they
    // moved to them (NVFP4 414.5 -> 400.2, MXFP8 479.5 -> 463.1 us).
    kp.d_stage_all = g_env_tma_store >= 0 ? g_env_tma_store : 0;
    kp.stages = pl.stages;
    char* ws = static_cast<char*>(workspace);
    kp.status = reinterpret_cast<int*>(ws);
    kp.tile_counters = any_split(pl) ? reinterpret_cast<int*>(ws + kHeaderBytes) : nullptr;
    kp.num_slots = static_cast<int>(partial_slots(pl));
    kp.num_counters = any_split(pl) ? pl.num_m * pl.num_n * pl.cluster : 0;
    kp.partials = any_split(pl) ? reinterpret_cast<float*>(ws + kHeaderBytes + counter_bytes(pl)) : nullptr;
    kp.timeout_ns = g_timeout_ns > 0 ? g_timeout_ns : kDefaultTimeoutNs;
    kp.fault_inject = g_fault_inject;
    kp.stats = g_env_stats ? reinterpret_cast<unsigned long long*>(ws + 64) : nullptr;

    const bool fp8 = is_fp8(ab_dtype);
    if (pl.swap) {
        const char* what = "launch";
        const cudaError_t e = tcg::launch_swapped(kp, launch_shape(pl), pl.bn, pl.katoms, fp8, stream, &what);
        return e == cudaSuccess ? TCG_OK : fail_launch(what, e);
    }
    if (is_mx(ab_dtype)) {
        const int blk = ab_dtype == TCG_NVFP4 ? 2 : (ab_dtype == TCG_MXFP4 ? 3 : 1);
        const char* what = "launch";
        const cudaError_t e = tcg::launch_block_scaled(kp, launch_shape(pl), pl.bn, pl.katoms, blk, stream, &what);
        return e == cudaSuccess ? TCG_OK : fail_launch(what, e);
    }
    if (pl.cluster == 2 && pl.katoms == 2 && pl.bn != 256) {
        const char* what = "launch";
        const cudaError_t e = tcg::launch_narrow_pair(kp, launch_shape(pl), pl.bn, fp8, stream, &what);
        return e == cudaSuccess ? TCG_OK : fail_launch(what, e);
    }
    if (pl.cluster == 2 && pl.katoms == 2)
        return fp8 ? launch_kernel<256, true, true, 2>(kp, pl, stream)
                   : launch_kernel<256, false, true, 2>(kp, pl, stream);
    if (pl.cluster == 2)
        return fp8 ? launch_kernel<256, true, true, 1>(kp, pl, stream)
                   : launch_kernel<256, false, true, 1>(kp, pl, stream);
    if (pl.katoms == 2) {
        if (pl.bn == 256)
            return fp8 ? launch_kernel<256, true, false, 2>(kp, pl, stream)
                       : launch_kernel<256, false, false, 2>(kp, pl, stream);
        return fp8 ? launch_kernel<128, true, false, 2>(kp, pl, stream)
                   : launch_kernel<128, false, false, 2>(kp, pl, stream);
    }
    switch (pl.bn) {
        case 256:
            return fp8 ? launch_kernel<256, true, false, 1>(kp, pl, stream)
                       : launch_kernel<256, false, false, 1>(kp, pl, stream);
        case 128:
            return fp8 ? launch_kernel<128, true, false, 1>(kp, pl, stream)
                       : launch_kernel<128, false, false, 1>(kp, pl, stream);
        default:
            return fp8 ? launch_kernel<64, true, false, 1>(kp, pl, stream)
                       : launch_kernel<64, false, false, 1>(kp, pl, stream);
    }
}

int tcg_debug_schedule(int M, int N, int K, tcg_dtype ab_dtype, int num_sms, int sk_mode, int* rows, int max_rows) {
    if (M <= 0 || N <= 0 || K <= 0 || num_sms <= 0 || !is_ab_type(ab_dtype)) return -1;
    DeviceInfo dev;
    dev.num_sms = num_sms;
    dev.max_smem_optin = 232448;
    const Plan pl = make_plan(M, N, K, ab_dtype, dev, sk_mode);
    tcg::KernelParams kp;
    memset(&kp, 0, sizeof kp);
    kp.num_m_blk = pl.num_m; kp.num_n_blk = pl.num_n; kp.num_kb = pl.num_kb;
    kp.splits = pl.splits; kp.num_units = pl.units; kp.group_m = pl.group_m;
    kp.units_a = pl.units_a;
    kp.sk_tiles = pl.sk_tiles;
    kp.sk_iters = static_cast<long long>(pl.sk_tiles) * pl.num_kb;
    kp.sk_slot_base = pl.splits > 1 ? pl.units_a : 0;
    kp.half_tail = pl.half_tail;
    int n = 0;
    for (int wid = 0; wid < pl.workers; ++wid) {
        tcg::WorkIter it = tcg::work_begin(kp, wid, pl.workers);
        tcg::Unit w;
        while (tcg::work_next(kp, it, w)) {
            if (n < max_rows && rows) {
                int* r = rows + 10 * n;
                r[0] = wid; r[1] = w.tile; r[2] = w.m_blk; r[3] = w.n_blk; r[4] = w.kb0; r[5] = w.kb1;
                r[6] = w.split; r[7] = w.nsplit;
                r[8] = w.nsplit > 1 ? tcg::partial_slot(kp, w, w.split, pl.workers) : -1;
                r[9] = w.nh;
            }
            ++n;
        }
    }
    return n;
}

tcg_status tcg_device_status(void* workspace, void* stream_) {
    if (!workspace) return TCG_ERR_WORKSPACE;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail_launch("cudaStreamSynchronize", e);
    int words[4] = {0, 0, 0, 0};
    e = cudaMemcpy(words, workspace, sizeof words, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_launch("cudaMemcpy(status)", e);
    if (words[0] != 0) {
        char buf[160];
        if (words[0] == TCG_ERR_CHECK)
            snprintf(buf, sizeof buf, "device-side check failed (check code %d, block %d)", words[1], words[2]);
        else
            snprintf(buf, sizeof buf, "device wait ran out (role/stage code %d, block %d)", words[1], words[2]);
        g_last_error = buf;
        e = cudaMemset(workspace, 0, sizeof words);
        if (e != cudaSuccess) return fail_launch("cudaMemset(status)", e);
        return static_cast<tcg_status>(words[0]);
    }
    return TCG_OK;
}

}  // extern "C"

// ------------------------------------------------- no-allocation entry point
//
// Some callers cannot allocate device memory: plugins that receive only
// input and output pointers from a host engine that owns every byte of device
// memory (and hands out no allocator or workspace), and latency-critical loops
// where cudaMalloc/cudaFree are not allowed because of their cost and implicit
// synchronisation.  tcg_gemm itself allocates nothing, but it needs a
// caller-provided workspace, which such callers cannot supply.
// tcg_gemm_noalloc runs the same GEMM with its workspace taken from this
// file-scope device array instead.  Every GPU that loads the library holds
// the array until the process exits.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB

// Device-side scratch.  In host code this name is only a stand-in for the
// symbol, never a device address: the address is taken once per device with
// cudaGetSymbolAddress and passed to the kernel.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

}  // namespace

extern "C" tcg_status tcg_gemm_noalloc(int M, int N, int K, float alpha, const void* A, int lda, tcg_layout opA,
                                       const void* B, int ldb, tcg_layout opB, float beta, const void* C, int ldc,
                                       tcg_dtype c_dtype, void* D, int ldd, tcg_dtype d_dtype, tcg_epilogue epi,
                                       tcg_dtype ab_dtype, tcg_scales scales, void* stream_) {
    const int has_c = beta != 0.0f;
    tcg_status st = tcg_can_implement(M, N, K, ab_dtype, A, lda, opA, B, ldb, opB, has_c, C, ldc, c_dtype, D, ldd,
                                      d_dtype, epi);
    if (st != TCG_OK) return st;
    if (M == 0 || N == 0) return TCG_OK;
    DeviceInfo dev;
    if ((st = device_info(dev)) != TCG_OK) return st;
    // Everything tcg_gemm would refuse is refused before the scratch is touched.
    if ((st = arch_check(dev)) != TCG_OK) return st;
    if ((st = check_scales(scales, ab_dtype, K)) != TCG_OK) return st;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return fail_launch("cudaGetDevice", e);
    if (device < 0 || device >= 64) { g_last_error = "device index out of range"; return TCG_ERR_LAUNCH; }
    void* scratch = nullptr;
    {
        // Set-up, once per device, on the first call made with that device current.
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (!g_noalloc_ptr[device]) {
            void* ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess || !ptr) return fail_launch("cudaGetSymbolAddress(scratch)", e);
            g_noalloc_ptr[device] = ptr;
        }
        scratch = g_noalloc_ptr[device];
    }
    const Plan pl = plan_gemm(M, N, K, ab_dtype, dev, opA, opB);
    const size_t need = workspace_need(pl, M, N, K, ab_dtype, A, lda, opA, B, ldb, opB).total();
    if (need > kNoAllocScratchBytes) {
        char buf[200];
        snprintf(buf, sizeof buf,
                 "tcg_gemm_noalloc: this problem needs %zu bytes of scratch, more than the %zu-byte maximum; "
                 "use tcg_gemm with a workspace",
                 need, kNoAllocScratchBytes);
        g_last_error = buf;
        return TCG_ERR_WORKSPACE;
    }
    // The array keeps the previous call's contents: the status word and the
    // split-K arrival counters must start at zero.
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    e = cudaMemsetAsync(scratch, 0, kHeaderBytes + counter_bytes(pl), stream);
    if (e != cudaSuccess) return fail_launch("cudaMemsetAsync(scratch)", e);
    return tcg_gemm(M, N, K, alpha, A, lda, opA, B, ldb, opB, beta, C, ldc, c_dtype, D, ldd, d_dtype, epi, ab_dtype,
                    scales, scratch, kNoAllocScratchBytes, stream_);
}

// =================================================================== grouped GEMM

namespace {

// The problems that produce output (M > 0 and N > 0), validated.
tcg_status grouped_validate(int G, const tcg_problem* problems, tcg_layout opA, tcg_layout opB, float beta,
                            tcg_dtype c_dtype, tcg_dtype d_dtype, tcg_epilogue epi, tcg_dtype ab_dtype,
                            std::vector<tcg_problem>* live) {
    if (G < 0 || (G > 0 && !problems)) return TCG_ERR_INVALID_ARG;
    if (is_mx(ab_dtype)) return TCG_ERR_UNSUPPORTED;
    const int has_c = beta != 0.0f;
    const int eb = elem_bytes(ab_dtype);
    live->clear();
    for (int g = 0; g < G; ++g) {
        const tcg_problem& q = problems[g];
        tcg_epilogue e = epi;
        e.bias = q.bias;
        tcg_status st = tcg_can_implement(q.M, q.N, q.K, ab_dtype, q.A, q.lda, opA, q.B, q.ldb, opB, has_c, q.C,
                                          q.ldc, c_dtype, q.D, q.ldd, d_dtype, e);
        if (st != TCG_OK) return st;
        if (q.M == 0 || q.N == 0) continue;
        if (q.K > 0 && (!tma_addressable(q.A, q.lda, eb) || !tma_addressable(q.B, q.ldb, eb)))
            return TCG_ERR_UNSUPPORTED;
        live->push_back(q);
    }
    return TCG_OK;
}

}  // namespace

extern "C" size_t tcg_grouped_workspace_size(int num_problems) {
    if (num_problems < 0) return 0;
    return kHeaderBytes + grouped_table_bytes(num_problems);
}

extern "C" tcg_status tcg_grouped_plan(int num_problems, const tcg_problem* problems, tcg_dtype ab_dtype,
                                       int out[10]) {
    if (!out || num_problems < 0 || (num_problems > 0 && !problems) || !is_ab_type(ab_dtype))
        return TCG_ERR_INVALID_ARG;
    DeviceInfo dev;
    tcg_status st = device_info(dev);
    if (st != TCG_OK) return st;
    std::vector<tcg_problem> live;
    for (int g = 0; g < num_problems; ++g)
        if (problems[g].M > 0 && problems[g].N > 0) live.push_back(problems[g]);
    const Plan pl = make_grouped_plan(live, ab_dtype, dev, nullptr);
    const int vals[10] = {tcg::kBM, pl.bn, pl.katoms * tcg::kRowBytes / elem_bytes(ab_dtype), pl.stages, pl.splits,
                          pl.grid, pl.cluster, pl.units, pl.group_m, pl.smem};
    memcpy(out, vals, sizeof vals);
    return TCG_OK;
}

extern "C" tcg_status tcg_gemm_grouped(int num_problems, const tcg_problem* problems, tcg_layout opA,
                                       tcg_layout opB, float beta, tcg_dtype c_dtype, tcg_dtype d_dtype,
                                       tcg_epilogue epi, tcg_dtype ab_dtype, void* workspace, size_t workspace_bytes,
                                       void* stream_) {
    std::vector<tcg_problem> live;
    tcg_status st = grouped_validate(num_problems, problems, opA, opB, beta, c_dtype, d_dtype, epi, ab_dtype, &live);
    if (st != TCG_OK) return st;
    if (live.empty()) return TCG_OK;
    DeviceInfo dev;
    if ((st = device_info(dev)) != TCG_OK) return st;
    if ((st = arch_check(dev)) != TCG_OK) return st;
    const int n = static_cast<int>(live.size());
    const size_t table = grouped_table_bytes(n);
    if (!workspace || !aligned16(workspace) || workspace_bytes < kHeaderBytes + table) return TCG_ERR_WORKSPACE;
    std::vector<int> tiles;
    const Plan pl = make_grouped_plan(live, ab_dtype, dev, &tiles);
    long long total = 0;
    for (int t : tiles) total += t;
    if (total > (1LL << 30)) return TCG_ERR_UNSUPPORTED;

    // Launch-wide parameters; each problem's block starts as a copy of them.
    const int has_c = beta != 0.0f;
    const int eb = elem_bytes(ab_dtype);
    bool all_c_tma = has_c;
    for (const tcg_problem& q : live) all_c_tma = all_c_tma && tma_addressable(q.C, q.ldc, elem_bytes(c_dtype));
    tcg::KernelParams base;
    memset(&base, 0, sizeof base);
    base.splits = 1;
    base.group_m = pl.group_m;
    base.a_mn_major = (opA == TCG_COL);
    base.b_mn_major = (opB == TCG_ROW);
    base.beta = beta;
    base.ab_fmt = mma_format(ab_dtype);
    base.c_f32 = (c_dtype == TCG_F32);
    base.c_tma = all_c_tma;
    base.bias_f32 = (epi.bias_dtype == TCG_F32);
    base.act = static_cast<int>(epi.act);
    base.d_f32 = (d_dtype == TCG_F32);
    base.stages = pl.stages;
    base.epi_nbuf = tcg::epi_warp_bytes(false) / (32 * 32 * std::max(elem_bytes(d_dtype), all_c_tma ? elem_bytes(c_dtype) : 0));
    char* ws = static_cast<char*>(workspace);
    base.status = reinterpret_cast<int*>(ws);
    base.timeout_ns = g_timeout_ns > 0 ? g_timeout_ns : kDefaultTimeoutNs;
    base.fault_inject = g_fault_inject;
    base.stats = g_env_stats ? reinterpret_cast<unsigned long long*>(ws + 64) : nullptr;

    std::vector<tcg::KernelParams> blocks(n);
    std::vector<int> tile0(n + 1, 0);
    const int bk = tcg::kRowBytes / eb;
    const int tile_m = pl.cluster == 2 ? 2 * tcg::kBM : tcg::kBM;
    for (int g = 0; g < n; ++g) {
        const tcg_problem& q = live[g];
        tcg::KernelParams& kp = blocks[g];
        kp = base;
        if (q.K > 0) {
            if (opA == TCG_ROW)
                st = encode_2d(&kp.tmA, ab_dtype, q.A, q.K, q.M, q.lda, bk, tcg::kBM, CU_TENSOR_MAP_SWIZZLE_128B);
            else
                st = encode_2d(&kp.tmA, ab_dtype, q.A, q.M, q.K, q.lda, bk, pl.katoms * bk, CU_TENSOR_MAP_SWIZZLE_128B);
            if (st != TCG_OK) return st;
            const int b_rows = pl.cluster == 2 ? pl.bn / 2 : pl.bn;
            if (opB == TCG_COL)
                st = encode_2d(&kp.tmB, ab_dtype, q.B, q.K, q.N, q.ldb, bk, b_rows, CU_TENSOR_MAP_SWIZZLE_128B);
            else
                st = encode_2d(&kp.tmB, ab_dtype, q.B, q.N, q.K, q.ldb, bk, pl.katoms * bk, CU_TENSOR_MAP_SWIZZLE_128B);
            if (st != TCG_OK) return st;
        }
        kp.d_tma = tma_addressable(q.D, q.ldd, elem_bytes(d_dtype));
        if (kp.d_tma) {
            st = encode_2d(&kp.tmD, d_dtype, q.D, q.N, q.M, q.ldd, tcg::kEpiChunk, 32,
                           d_dtype == TCG_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
            if (st != TCG_OK) return st;
        }
        if (all_c_tma) {
            st = encode_2d(&kp.tmC, c_dtype, q.C, q.N, q.M, q.ldc, tcg::kEpiChunk, 32,
                           c_dtype == TCG_F32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
            if (st != TCG_OK) return st;
        }
        kp.M = q.M;
        kp.N = q.N;
        kp.K = q.K;
        kp.alpha = q.alpha;
        kp.num_m_blk = (q.M + tile_m - 1) / tile_m;
        kp.num_n_blk = (q.N + pl.bn - 1) / pl.bn;
        kp.num_kb = (q.K + pl.katoms * bk - 1) / (pl.katoms * bk);
        kp.num_units = kp.units_a = tiles[g];
        kp.C = has_c ? q.C : nullptr;
        kp.ldc = q.ldc;
        kp.c_vec = has_c && tma_addressable(q.C, q.ldc, elem_bytes(c_dtype));
        kp.bias = q.bias;
        kp.D = q.D;
        kp.ldd = q.ldd;
        kp.d_inner_aligned = (static_cast<long long>(q.N) * elem_bytes(d_dtype)) % 16 == 0;
        kp.d_v32 = g_env_st32 && reinterpret_cast<uintptr_t>(q.D) % 32 == 0 &&
                   (static_cast<long long>(q.ldd) * elem_bytes(d_dtype)) % 32 == 0;
        tile0[g + 1] = tile0[g] + tiles[g];
    }
    // One table in the workspace after the status header: the problems'
    // parameter blocks, then their first units.
    std::vector<unsigned char> host(table, 0);
    memcpy(host.data(), blocks.data(), static_cast<size_t>(n) * sizeof(tcg::KernelParams));
    memcpy(host.data() + static_cast<size_t>(n) * sizeof(tcg::KernelParams), tile0.data(),
           static_cast<size_t>(n + 1) * sizeof(int));
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    cudaError_t e = cudaMemcpyAsync(ws + kHeaderBytes, host.data(), table, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return fail_launch("cudaMemcpyAsync(grouped table)", e);

    tcg::KernelParams kp = base;
    kp.num_units = kp.units_a = pl.units;
    kp.group = reinterpret_cast<const tcg::KernelParams*>(ws + kHeaderBytes);
    kp.group_tile0 = reinterpret_cast<const int*>(ws + kHeaderBytes + static_cast<size_t>(n) * sizeof(tcg::KernelParams));
    kp.num_groups = n;
    kp.M = kp.N = kp.K = 1;   // launch-wide sizes are unused; the problems carry their own
    const char* what = "launch";
    e = tcg::launch_grouped(kp, launch_shape(pl), is_fp8(ab_dtype), stream, &what);
    return e == cudaSuccess ? TCG_OK : fail_launch(what, e);
}
