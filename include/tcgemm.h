/*
 * tcgemm.h -- C ABI of the GB300 (sm_103a) tiled tensor-core persistent GEMM.
 *
 * The one operation:
 *
 *     D = act( alpha * sA * sB * (A @ B) + beta * C + bias )
 *
 * "CUTLASS" (stanleyjacob.dev), Part I: the one-GEMM identity
 * D = alpha * (A @ B) + beta * C, A M x K, B K x N, C and D M x N; Part II:
 * the LinearCombination epilogue and a fused bias / ReLU variant; Part IV
 * Stage 5: bias, GELU and a dequantisation scale fused into the epilogue;
 * Part IV Stage 1: the host sequence get_workspace_size -> can_implement ->
 * run, with a status return.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Matrices are dense, addressed by a base pointer and a leading dimension
 *   (ld, in elements).  A is the logical M x K operand, B the logical K x N
 *   operand.  TCG_ROW stores a matrix row-major (element (r,c) at r*ld + c),
 *   TCG_COL column-major (element (r,c) at c*ld + r).  C and D are always
 *   row-major M x N.
 * - All device pointers (A, B, C, D, bias, workspace) are owned by the
 *   caller, are device memory of the current CUDA device, and must stay
 *   valid until the work queued on `stream` has finished.  The library keeps
 *   only a process-wide cache of TMA descriptors and launch attributes.
 * - Alignment ("CUTLASS" page, Part II, on alignment: a tensor that breaks
 *   the alignment rules is either taken by a slower path or rejected).  Every
 *   pointer must be aligned to its element size, else TCG_ERR_MISALIGNED.
 *   The fast path wants each matrix 16-byte aligned with ld * sizeof(element)
 *   a multiple of 16 bytes (the TMA rule).  Otherwise the call still runs:
 *   A or B is first copied into 16-byte pitched rows of the workspace (size
 *   it with tcg_workspace_size_for), and C, D and bias are read and written
 *   element-wise in the epilogue.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  tcg_gemm is asynchronous: host-detectable errors return before
 *   anything is queued; device-side errors (a bounded wait that ran out) are
 *   recorded in the workspace status word and read by tcg_device_status.
 * - No CPU fallback and no library GEMM: every FLOP runs in this library's
 *   sm_103a kernels.  On any other GPU tcg_can_implement, tcg_gemm and the
 *   other GEMM entry points return TCG_ERR_ARCH.
 */
#ifndef TCGEMM_H
#define TCGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TCG_OK = 0,
    TCG_ERR_INVALID_ARG = 1,   /* negative size, NULL pointer that is needed, bad enum, ld too small */
    TCG_ERR_UNSUPPORTED = 2,   /* valid request the library does not implement (e.g. MN-major e4m3) */
    TCG_ERR_MISALIGNED = 3,    /* a pointer not aligned to its element size */
    TCG_ERR_ARCH = 4,          /* current device is not compute capability 10.3 */
    TCG_ERR_WORKSPACE = 5,     /* workspace NULL, misaligned or smaller than tcg_workspace_size_for */
    TCG_ERR_LAUNCH = 6,        /* a CUDA runtime/driver call failed (message: tcg_last_error) */
    TCG_ERR_TIMEOUT = 7,       /* a bounded device-side wait ran out (reported by tcg_device_status) */
    TCG_ERR_CHECK = 8          /* debug build only: a device-side consistency check failed (tcg_device_status) */
} tcg_status;

typedef enum { TCG_ROW = 0, TCG_COL = 1 } tcg_layout;

/* Operands A and B: BF16, F16, E4M3, E5M2, MXE4M3 or MXE5M2 (both the same).
 * C, D and bias: BF16 or F32.  E4M3 / E5M2 are the FP8 formats (e4m3 without
 * infinities).  MXE4M3 / MXE5M2 are block-scaled FP8 (the OCP Microscaling
 * formats MXFP8): E4M3 / E5M2 elements plus one E8M0 scale (2^(e - 127)) per
 * 32 consecutive K of each A row and each B column, passed in
 * tcg_scales.block_sfa / block_sfb ("CUTLASS" page, Part V: narrow formats
 * in which a few neighbouring elements share one scale). */
typedef enum {
    TCG_BF16 = 0, TCG_E4M3 = 1, TCG_F32 = 2, TCG_F16 = 3, TCG_E5M2 = 4,
    TCG_MXE4M3 = 5, TCG_MXE5M2 = 6, TCG_NVFP4 = 7, TCG_MXFP4 = 8
} tcg_dtype;
/* TCG_NVFP4 / TCG_MXFP4: the block-scaled four-bit formats (same page, Part
 * V): FP4 E2M1 elements packed two per byte (the even element of each pair in
 * the low nibble; lda / ldb count elements), with one unsigned E4M3 scale per
 * 16 consecutive K (NVFP4) or one E8M0 scale per 32 (MXFP4), passed like the
 * MX scales in tcg_scales.block_sfa / block_sfb. */

typedef enum { TCG_ACT_NONE = 0, TCG_ACT_RELU = 1, TCG_ACT_GELU = 2 } tcg_act;

/* Fused epilogue.  bias: NULL or a device vector of N elements (bias_dtype
 * TCG_BF16 or TCG_F32), added per output column before the activation.
 * act: NONE, RELU = max(x, 0), GELU = exact erf form 0.5*x*(1+erf(x/sqrt 2)). */
typedef struct {
    const void* bias;
    tcg_dtype bias_dtype;
    tcg_act act;
} tcg_epilogue;

/* Dequantisation scales (CUTLASS page, Part IV Stage 5: a per-channel scale
 * fused into the epilogue).  The raw product sum of element (i, j) is
 * multiplied by alpha * scale_a * scale_b * row_scale[i] * col_scale[j].
 * scale_a / scale_b: per-tensor (1.0 when unused).  row_scale: NULL or a
 * device vector of M fp32 values; col_scale: NULL or a device vector of N
 * fp32 values (both 4-byte aligned).  Any operand type.
 *
 * block_sfa / block_sfb: the block scales of the block-scaled operand types
 * (NULL otherwise; required for them when K > 0), device memory, 16-byte
 * aligned.  Scale (r, c) belongs to row r of A (column r of B) and to K
 * elements [g c, g c + g), g = 32 (MX types) or 16 (NVFP4).  Layout: rows
 * padded to a multiple of 128, scale columns to a multiple of 4 (padding:
 * any finite code); each block of 128 rows x 4 columns is 512 consecutive
 * bytes holding (r, c) at byte (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
 * block (row block rb, column block cb) starts at byte
 * (rb * ceil(ceil(K / g) / 4) + cb) * 512.  This is the order in which the
 * tensor cores read them, so the kernel copies each block unchanged. */
typedef struct {
    float scale_a;
    float scale_b;
    const float* row_scale;
    const float* col_scale;
    const void* block_sfa;
    const void* block_sfb;
} tcg_scales;

/*
 * tcg_can_implement -- argument validation, then the architecture check; no
 * launch.  TCG_OK also for unaligned leading dimensions (the slow path above).
 *   M, N, K        : problem size, >= 0.
 *   ab_dtype       : TCG_BF16, TCG_F16, TCG_E4M3, TCG_E5M2, TCG_MXE4M3 or
 *                    TCG_MXE5M2 (A and B share it).  The 8-bit types
 *                    require opA = TCG_ROW and opB = TCG_COL (both
 *                    K-contiguous); the block-scaled types also a 16-byte
 *                    aligned A and B whose row pitch in bytes is a multiple of
 *                    16 (else TCG_ERR_UNSUPPORTED), and for FP4 an even K.
 *   A, lda, opA    : operand A; lda >= K (ROW) or >= M (COL).
 *   B, ldb, opB    : operand B; ldb >= N (ROW) or >= K (COL).
 *   has_c, C, ldc, c_dtype : has_c != 0 when beta != 0; then C row-major,
 *                    ldc >= N, c_dtype TCG_BF16 or TCG_F32.
 *   D, ldd, d_dtype: output, row-major, ldd >= N, TCG_BF16 or TCG_F32.
 *   epi            : bias pointer (aligned to its element) / dtype / activation.
 * Returns TCG_OK or the first failing rule's code.  M == 0 or N == 0 is OK
 * on any device.  When the process sees a CUDA device, a non-empty problem
 * that passes every argument rule is then checked against the current
 * device: TCG_ERR_ARCH unless it is compute capability 10.3 (the
 * tcg_arch_status mapping; the device's attributes are read once and
 * cached).  Without any CUDA device only the arguments are checked.
 */
tcg_status tcg_can_implement(int M, int N, int K, tcg_dtype ab_dtype,
                             const void* A, int lda, tcg_layout opA,
                             const void* B, int ldb, tcg_layout opB,
                             int has_c, const void* C, int ldc, tcg_dtype c_dtype,
                             const void* D, int ldd, tcg_dtype d_dtype,
                             tcg_epilogue epi);

/*
 * tcg_arch_status -- the architecture rule on its own, for a device of
 * compute capability major.minor: TCG_OK for 10.3 (the sm_103a kernels this
 * library is built for), TCG_ERR_ARCH for anything else.  "A10 CuTe,
 * CUTLASS & CuTile" (gahan9.github.io), the pitfalls table: check the
 * architecture a kernel was compiled for before running it.  Pure function,
 * no device access.
 */
tcg_status tcg_arch_status(int major, int minor);

/*
 * tcg_workspace_size -- bytes of device workspace tcg_gemm needs for this
 * problem on the current device: a 256-byte status/counter header plus, when
 * the planner splits K (skinny shapes), fp32 partial tiles and per-tile
 * arrival counters.  The workspace must be zero-filled once when allocated
 * (tcg_workspace_init); the library leaves it in that state after every call.
 * Returns 0 only for invalid sizes.
 */
size_t tcg_workspace_size(int M, int N, int K, tcg_dtype ab_dtype);

/*
 * tcg_workspace_size_for -- tcg_workspace_size plus room for packed copies of
 * A and/or B when the TMA cannot address them as stored (base not 16-byte
 * aligned, or ld * sizeof(element) not a multiple of 16): outer x ld' elements
 * per packed operand, ld' = the contiguous extent rounded up to 16 bytes,
 * each copy 256-byte aligned.  Equal to tcg_workspace_size when both operands
 * are TMA-addressable.  Arguments as in tcg_can_implement (pointers are only
 * inspected, never dereferenced).  Returns 0 for invalid sizes or layouts.
 */
size_t tcg_workspace_size_for(int M, int N, int K, tcg_dtype ab_dtype,
                              const void* A, int lda, tcg_layout opA,
                              const void* B, int ldb, tcg_layout opB);

/* Zero-fill `bytes` of workspace on `stream` (asynchronous). */
tcg_status tcg_workspace_init(void* workspace, size_t bytes, void* stream);

/*
 * tcg_gemm -- D = act(alpha*scale_a*scale_b*(A@B) + beta*C + bias), queued on
 * `stream`.  Arguments as in tcg_can_implement; beta == 0 means C is never
 * read (C may be NULL and may hold NaN).  K == 0 gives act(beta*C + bias).
 * The result is rounded once from fp32 to d_dtype (round to nearest even).
 * When A or B is not TMA-addressable, a copy kernel first packs it into the
 * workspace on `stream` (workspace_bytes >= tcg_workspace_size_for, else
 * TCG_ERR_WORKSPACE with a message in tcg_last_error).
 * D must not overlap A, B or bias; D == C (in-place update) is allowed when
 * ldc == ldd and c_dtype == d_dtype.
 * Returns TCG_OK when the kernel was queued.
 */
tcg_status tcg_gemm(int M, int N, int K, float alpha,
                    const void* A, int lda, tcg_layout opA,
                    const void* B, int ldb, tcg_layout opB,
                    float beta, const void* C, int ldc, tcg_dtype c_dtype,
                    void* D, int ldd, tcg_dtype d_dtype,
                    tcg_epilogue epi, tcg_dtype ab_dtype, tcg_scales scales,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * tcg_device_status -- synchronises `stream`, reads the workspace status word
 * (TCG_OK, TCG_ERR_TIMEOUT, or in the debug build TCG_ERR_CHECK) written by
 * earlier tcg_gemm calls on this workspace, and clears it.  Returns
 * TCG_ERR_LAUNCH if the stream itself reports a CUDA error.
 *
 * Debug build: libtcgemm_debug.so (the same sources compiled with
 * TCG_DEBUG_CHECKS) checks the kernel's pipeline bookkeeping on the device:
 * stage, accumulator, epilogue-buffer, TMEM-column, partial-slot and counter
 * indices in range, every unit of work inside the tile grid, and after each
 * mbarrier wait that the following phase has not completed as well.  A
 * failed check ends the CTA without a trap and records TCG_ERR_CHECK with the
 * check's code and the block, which tcg_device_status returns (message in
 * tcg_last_error).
 */
tcg_status tcg_device_status(void* workspace, void* stream);

/* Human-readable text of the last TCG_ERR_LAUNCH / TCG_ERR_ARCH on this thread. */
const char* tcg_last_error(void);

/*
 * tcg_plan -- the launch plan tcg_gemm would use for these sizes, operand
 * type and A / B layouts (for tests and tools).
 * out[0..10] = {BM, BN, BK, stages, splits, grid CTAs, cluster size,
 *               units of work, raster group, dynamic smem bytes, swapped}.
 * BN of a pair tile may be 160, 192 or 224 instead of 256 when B is
 * column-major (K-contiguous) and the narrower tile fills the last wave
 * better.  swapped = 1 (only on request: TCG_SWAP=1 in the environment when
 * the library loads, or the test knob below): a GEMM with at most 64 rows and
 * a row-major A runs as the transposed product D^T = B^T A^T (written back
 * into the row-major D);
 * BM, BN, splits and units then count the transposed problem's tiles (BM
 * over D's columns, BN = 32 or 64 over D's rows).  units of work > tiles x
 * splits when the last tiles are split over K to fill the last wave.
 * Needs the current device (queries SM count and shared-memory limit).
 */
tcg_status tcg_plan(int M, int N, int K, tcg_dtype ab_dtype, tcg_layout opA, tcg_layout opB, int out[11]);

/*
 * tcg_debug_set -- TEST-ONLY knobs, process-wide.
 *   fault_inject = 1: in the next launches, CTA 0's producer skips its first
 *     stage (no loads, no arrival), so the MMA issuer's bounded wait runs out
 *     and the kernel records TCG_ERR_TIMEOUT instead of hanging.
 *   fault_inject = 2: debug build only: CTA 0's producer fails a check before
 *     its first stage (code 199), so the kernel records TCG_ERR_CHECK and
 *     ends the way a timeout does; the release build ignores it.
 *   wait_timeout_ns: limit of every bounded device-side wait (0 = default 2 s).
 *   force_splits / force_cta2: override the planner (0 = automatic).
 *     force_cta2: 1 = 2-CTA pair tiles, 2 = one-CTA tiles; for the
 *     block-scaled types 3 / 4 = pair tiles 256 / 192 wide (NVFP4: 256
 *     always; the default width is 256); 5 = one-CTA tiles, and a GEMM with
 *     at most 64 rows, a row-major A and at least 256 columns runs as the
 *     transposed product D^T = B^T A^T (see tcg_plan).
 */
void tcg_debug_set(int fault_inject, long long wait_timeout_ns, int force_splits, int force_cta2);

/*
 * tcg_debug_schedule -- TEST-ONLY, needs no GPU: the work schedule tcg_gemm
 * would run on a device with num_sms SMs.  sk_mode: -1 = the default, 0 = no
 * Stream-K, 1 = last partial wave plus one full wave as Stream-K, 2 = last
 * partial wave only, 3 = all tiles.  Writes up to max_rows rows of 10 ints,
 * one per unit of work in the order each worker runs them:
 *   {worker, tile, m_blk, n_blk, kb0, kb1, split, nsplit, partial slot, half}
 * (half: 0 for a whole tile; 1 / 2 for the first / second half of a
 * 256-wide tile's columns, when the last wave runs as half-width units)
 * (k-blocks are pipeline stages; partial slot -1 for an unsplit tile) and
 * returns the number of units (which may exceed max_rows), or -1 for
 * invalid sizes.
 */
int tcg_debug_schedule(int M, int N, int K, tcg_dtype ab_dtype, int num_sms, int sk_mode,
                       int* rows, int max_rows);

/*
 * tcg_gemm_noalloc -- the same GEMM as tcg_gemm for callers that cannot
 * allocate device memory, so cannot pass a workspace: e.g. plugins that only
 * receive input/output pointers from an engine that owns all device memory,
 * or latency-critical loops where cudaMalloc/cudaFree are not allowed.
 * The reference pages have no counterpart; this is a property of the library.
 *   Arguments: as tcg_gemm, without the workspace.  It allocates nothing.
 *   Scratch: a 32 MiB file-scope device array held by every GPU that loads
 *     the library until the process exits.  Problems whose workspace
 *     (tcg_workspace_size_for) exceeds 32 MiB return TCG_ERR_WORKSPACE with
 *     a message in tcg_last_error.
 *   Set-up: the first call on each device (with that device current) looks
 *     up the array's device address; make that first call before any stream
 *     capture.
 *   Concurrency: all calls on a device share the one array; calls that
 *     overlap on the GPU (different streams, unordered) race and give wrong
 *     results.  Each call clears the status word and split-K counters first.
 *   Device-side wait timeouts still end the kernel but are not reported (no
 *     workspace is visible to the caller).
 */
tcg_status tcg_gemm_noalloc(int M, int N, int K, float alpha,
                            const void* A, int lda, tcg_layout opA,
                            const void* B, int ldb, tcg_layout opB,
                            float beta, const void* C, int ldc, tcg_dtype c_dtype,
                            void* D, int ldd, tcg_dtype d_dtype,
                            tcg_epilogue epi, tcg_dtype ab_dtype, tcg_scales scales,
                            void* stream);

/*
 * Grouped GEMM ("CUTLASS" page, Part V, numeric-types deep dive: the experts
 * of a mixture-of-experts layer run as one grouped GEMM, one problem per
 * expert, the problems of different sizes; Part III: grouped GEMMs with
 * irregular shapes).  One launch computes, for every problem g,
 *
 *     D_g = act( alpha_g * (A_g @ B_g) + beta * C_g + bias_g )
 *
 * Each problem has its own sizes, alpha, operands, C, bias and D; the operand
 * type, the layouts of A and B, beta, the activation and the C / D / bias
 * types are shared.  Problems are independent: no output may overlap another
 * problem's inputs or output.
 *
 * tcg_problem: M, N, K >= 0 and the pointers / leading dimensions of one
 * problem, with the meaning they have in tcg_gemm.  alpha: this problem's
 * factor (for FP8 operands, alpha * scale_a * scale_b of its per-tensor
 * scales).  bias: NULL or N elements of the shared bias type.  C is read only
 * when beta != 0.
 */
typedef struct {
    int M, N, K;
    float alpha;
    const void* A;
    int lda;
    const void* B;
    int ldb;
    const void* C;
    int ldc;
    void* D;
    int ldd;
    const void* bias;
} tcg_problem;

/*
 * tcg_grouped_workspace_size -- bytes of workspace tcg_gemm_grouped needs for
 * num_problems problems: the 256-byte status header plus a table of one
 * parameter block per problem (tensor maps, sizes, pointers) and the first
 * unit of each.  Zero-fill it once (tcg_workspace_init).  0 if num_problems < 0.
 */
size_t tcg_grouped_workspace_size(int num_problems);

/*
 * tcg_gemm_grouped -- every problem of problems[0 .. num_problems) in one
 * persistent launch on `stream`: the tiles of all problems form one list of
 * units that the CTAs (or CTA pairs) take in turn.
 *   problems: host array, read during the call only.
 *   opA, opB, beta, c_dtype, d_dtype, ab_dtype: shared, as in tcg_gemm;
 *     ab_dtype BF16, F16, E4M3 or E5M2 (the block-scaled types: TCG_ERR_UNSUPPORTED).
 *   epi: bias_dtype and act shared; epi.bias is ignored (each problem has its own).
 *   Each problem must pass tcg_can_implement, and its A and B (when K > 0)
 *   must be TMA-addressable: 16-byte aligned with ld * sizeof(element) a
 *   multiple of 16 (no packed slow path here; else TCG_ERR_UNSUPPORTED).  C,
 *   D and bias may be unaligned as in tcg_gemm.  Problems with M == 0 or
 *   N == 0 are skipped; K == 0 gives act(beta * C + bias) for that problem.
 *   workspace: at least tcg_grouped_workspace_size(num_problems) bytes,
 *     16-byte aligned, else TCG_ERR_WORKSPACE.  The call copies its table
 *     there with one host-to-device copy on `stream` (so it is not meant for
 *     stream capture into a CUDA graph), and calls on one workspace must be
 *     ordered (one stream).
 * Errors: the first failing problem's tcg_can_implement code, then as
 * tcg_gemm; nothing is queued on an error.  Device-side wait timeouts are
 * read with tcg_device_status, as for tcg_gemm.
 */
tcg_status tcg_gemm_grouped(int num_problems, const tcg_problem* problems,
                            tcg_layout opA, tcg_layout opB, float beta,
                            tcg_dtype c_dtype, tcg_dtype d_dtype, tcg_epilogue epi,
                            tcg_dtype ab_dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * tcg_grouped_plan -- the launch plan tcg_gemm_grouped would use, in the
 * layout of tcg_plan (units = the tiles of all problems; splits = 1).
 * Needs the current device.
 */
tcg_status tcg_grouped_plan(int num_problems, const tcg_problem* problems, tcg_dtype ab_dtype, int out[10]);

/*
 * tcg_debug_tma_swizzle128 -- TEST-ONLY: one TMA load of a rows x 128-byte
 * tile (row-major, 128-byte rows, device memory at src) into 1024-byte-aligned
 * shared memory with 128-byte swizzling, copied back unchanged to dst (rows x
 * 128 bytes), so that a test can compare the hardware's swizzled layout (the
 * one the GEMM kernel's shared-memory descriptors assume) with a host model.
 * rows in [1, 64]; src and dst 16-byte aligned device memory; status: a device
 * int the kernel sets to TCG_ERR_TIMEOUT if the load does not land within 1 s
 * (otherwise left as it is).  Queued on stream.  TCG_ERR_INVALID_ARG for bad
 * arguments, TCG_ERR_MISALIGNED for unaligned pointers.
 */
tcg_status tcg_debug_tma_swizzle128(const void* src, int rows, void* dst, int* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TCGEMM_H */
