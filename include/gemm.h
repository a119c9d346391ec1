/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense tensor-core GEMM library.
 *
 * Both GEMMs compute C = A * B^T on one GPU:
 *   A is M x K, B is N x K, both row-major with K contiguous ("K-major");
 *   C is M x N, row-major BF16, overwritten (the *_fused calls add alpha/beta scaling,
 *   a bias and an activation in the epilogue);
 *   products are accumulated in FP32 in tensor memory and rounded to BF16
 *   (round to nearest, ties to even) once, in the epilogue.
 *
 * Sources for what is computed:
 *   gemm_bf16  -- "Achieve cuBLAS Performance on NVIDIA GB300 for HGEMM",
 *                 introduction: row-major C = A @ B^T, A: MxK, B: NxK, BF16
 *                 inputs/outputs, FP32 accumulation in tensor memory.
 *   gemm_nvfp4 -- "NVFP4 GEMM on Blackwell", section "NVFP4 Datatype": E2M1
 *                 values with one FP8 scale factor per 16 values; section
 *                 "Tensor Cores and Tensor Memory": the scales are applied by
 *                 the block-scaled tensor-core MMA (scales read from TMEM).
 *
 * Conventions shared by every entry point:
 *   - All matrix pointers are DEVICE pointers of the current CUDA device,
 *     owned by the caller; the library keeps no reference after the call.
 *   - `stream` is a cudaStream_t / CUstream handle (NULL = legacy default
 *     stream). Calls are asynchronous: they enqueue work and return; nothing
 *     is synchronised. Results are visible to later work on `stream`.
 *   - Device memory: gemm_nvfp4_pack_scales allocates nothing; nor do gemm_nvfp4_blocked,
 *     except for fewer than 32 rows (a padded copy of A; gemm_options_t.no_pad_a), and
 *     gemm_bf16, except for a few-row GEMM that splits K (see gemm_bf16 and
 *     gemm_options_t.no_split_k). gemm_nvfp4 takes a temporary workspace for the
 *     rearranged scales (and the padded A) from a library-owned, stream-ordered memory
 *     pool (see gemm_nvfp4). The library also holds one process-wide device status word
 *     (a static __device__ variable) that kernels set if a bounded internal
 *     wait expires; read it with gemm_get_device_status.
 *   - Return value: GEMM_OK (0) or a gemm_status_t code for problems found on
 *     the host before launch. Nothing is launched when an error is returned.
 *     Faults during execution surface through the stream like any CUDA error.
 *   - Thread safety: calls on different streams may be made concurrently from
 *     several host threads.
 */
#ifndef DTCP_GEMM_H
#define DTCP_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,       /* null pointer with non-empty shape, negative size, bad option */
    GEMM_ERR_UNSUPPORTED_SHAPE = 2, /* a size constraint below is violated */
    GEMM_ERR_MISALIGNED = 3,        /* a pointer is not 16-byte aligned */
    GEMM_ERR_NO_DEVICE = 4,         /* no CUDA device / runtime error querying it */
    GEMM_ERR_ARCH = 5,              /* current device is not compute capability 10.3 (sm_103) */
    GEMM_ERR_DRIVER = 6,            /* cuTensorMapEncodeTiled unavailable or rejected the operand */
    GEMM_ERR_LAUNCH = 7,            /* the kernel launch itself failed */
    GEMM_ERR_TIMEOUT = 8,           /* device side: a bounded wait inside a kernel expired */
    GEMM_ERR_OUT_OF_MEMORY = 9,     /* gemm_nvfp4 could not obtain its scale workspace */
    GEMM_ERR_SCRATCH_TOO_SMALL = 10 /* gemm_nvfp4_noalloc: the problem's rearranged scales
                                       exceed its fixed scratch array */
} gemm_status_t;

/*
 * gemm_bf16 -- C[M][N] = bf16_rne( sum_k A[m][k] * B[n][k] ), FP32 accumulation.
 *
 *   A: M x K BF16, row stride K elements.   B: N x K BF16, row stride K.
 *   C: M x N BF16, row stride N elements.
 * Constraints: M, N, K >= 0; K % 8 == 0 and N % 8 == 0 (16-byte row strides
 * for the tensor-memory-accelerator copies); A, B, C 16-byte aligned.
 * M and N need not be tile multiples: rows/columns past M/N are read as zeros
 * and never written. M == 0 or N == 0: nothing to do, returns GEMM_OK.
 * K == 0: C is set to zero (an empty sum).
 * Kernel: persistent, warp-specialised, 2-CTA (cta_group::2) tcgen05 MMA with a
 * TMA-store epilogue, one kernel launch per call: a 512 x 256 output tile per CTA pair
 * (two 128-row M-waves per CTA filling TMEM) where gemm_bf16_wide_rule selects it, else
 * a 256 x 256 tile with a double-buffered TMEM accumulator. With M <= 128 and N >= 256 it
 * computes C^T = B A^T instead (tile N 64 or 128; see gemm_options_t.no_swap_ab), and
 * such a GEMM with few tiles splits K: the FP32 partial sums are added by a second launch
 * or, for two splits, inside the one launch (workspace from the library's stream-ordered
 * pool, as for gemm_nvfp4; see no_split_k).
 */
int gemm_bf16(const void* A, const void* B, void* C, int M, int N, int K, void* stream);

/*
 * gemm_nvfp4 -- C[M][N] = bf16_rne( sum_k a(m,k) * b(n,k) ), FP32 accumulation, where
 *   a(m,k) = e2m1(A code m,k) * e4m3(SFA[m][k/16]),  b(n,k) = e2m1(B code n,k) * e4m3(SFB[n][k/16]).
 *
 *   A:   M x K/2 bytes, row-major; byte j of row m holds the E2M1 code of
 *        element 2j in bits 0-3 and of element 2j+1 in bits 4-7.
 *   B:   N x K/2 bytes, same packing.
 *   SFA: M x K/16 bytes, row-major, E4M3 (OCP E4M3FN) scale of elements
 *        16q .. 16q+15 of row m at SFA[m][q]. SFB: N x K/16 bytes, same.
 *   C:   M x N BF16, row stride N.
 * Constraints: M, N, K >= 0; K % 256 == 0 (one 128-byte swizzle row of codes
 * per pipeline stage); N % 8 == 0; ceil(M/128) + ceil(N/128) <= 65535; all
 * pointers 16-byte aligned. Ragged M / N as for gemm_bf16. K == 0 sets C to zero.
 * Scales are used as the hardware's unsigned E4M3 (UE4M3): the sign bit of a
 * scale byte must be 0; NaN scales give unspecified results.
 * Launches: one scale-packing kernel (SFA and SFB together) into a workspace of
 * gemm_nvfp4_blocked_scale_bytes(M, K) + gemm_nvfp4_blocked_scale_bytes(N, K)
 * bytes (+ up to 510 bytes of alignment), then the gemm_nvfp4_blocked kernel; with
 * 1 <= M < 32 the packing launch also copies A into 32 * K / 2 more bytes of the
 * workspace, which the GEMM reads instead of A (gemm_options_t.no_pad_a). The
 * workspace comes from a library-owned stream-ordered pool (cudaMallocFromPoolAsync)
 * and is returned to it in stream order after the GEMM, so concurrent calls on
 * different streams use different workspaces. Returns GEMM_ERR_OUT_OF_MEMORY if
 * the workspace cannot be obtained.
 */
int gemm_nvfp4(const void* A, const void* SFA, const void* B, const void* SFB, void* C,
               int M, int N, int K, void* stream);

/*
 * Blocked scale layout -- the layout in which the block-scaled tensor-core MMA reads
 * scale factors (through tcgen05.cp .32x128b.warpx4; "NVFP4 GEMM on Blackwell",
 * "Tensor Cores and Tensor Memory"). For R rows and K columns (K % 64 == 0):
 * rows are padded to a multiple of 128; block (rb, j) holds the scales of rows
 * 128rb .. 128rb+127 for K elements 64j .. 64j+63 and is 512 contiguous bytes at
 * offset (rb * K/64 + j) * 512; inside a block, the 16-byte line l (0 <= l < 32)
 * holds, in order, the 4 scale bytes (16-element groups 0..3 of the 64-K step) of
 * rows l, l+32, l+64 and l+96. Padding rows are zero. Total size:
 * gemm_nvfp4_blocked_scale_bytes(R, K) = ceil(R/128) * 128 * K/16 bytes.
 */
long long gemm_nvfp4_blocked_scale_bytes(int rows, int K);   /* -1 if K % 64 != 0 or a size < 0 */

/*
 * gemm_nvfp4_pack_scales -- rearrange row-major scales SF[rows][K/16] (device) into
 * the blocked layout at SF_blocked (device, gemm_nvfp4_blocked_scale_bytes(rows, K)
 * bytes, caller-owned). One kernel launch on `stream`. Constraints: K % 64 == 0,
 * ceil(rows/128) <= 65535, both pointers 16-byte aligned.
 */
int gemm_nvfp4_pack_scales(const void* SF, void* SF_blocked, int rows, int K, void* stream);

/*
 * gemm_nvfp4_blocked -- gemm_nvfp4 with SFA and SFB given in the blocked layout
 * (gemm_nvfp4_blocked_scale_bytes(M, K) and (N, K) bytes). Same operands, result,
 * constraints and errors as gemm_nvfp4. This is the fast path: a stage's scales for
 * 128 rows are one contiguous 2 KB block, loaded by TMA together with the codes. With
 * 1 <= M < 32 the call first copies A (one small copy kernel launched ahead of the GEMM)
 * into a 32-row buffer of 32 * K / 2 bytes from the
 * library's stream-ordered pool (returned to it in stream order after the GEMM) and the
 * GEMM reads A from there (gemm_options_t.no_pad_a = 1 reads A in place and allocates
 * nothing); GEMM_ERR_OUT_OF_MEMORY if that buffer cannot be obtained.
 */
int gemm_nvfp4_blocked(const void* A, const void* SFA_blocked, const void* B, const void* SFB_blocked, void* C,
                       int M, int N, int K, void* stream);

/*
 * gemm_nvfp4_noalloc -- gemm_nvfp4 for callers that must not let the library allocate
 * device memory. (Not from the NVFP4 page: it has no counterpart there; it exists for
 * callers of this library.)
 *
 * gemm_nvfp4 rearranges the row-major scales into the blocked layout in a workspace it
 * takes from a memory pool. Some callers cannot allow that: code running where the CUDA
 * allocator must not be entered (inside a custom allocator or memory manager, an error
 * path, a loop with hard latency limits), or applications that account for every byte of
 * device memory through their own allocator. This entry point uses instead a fixed
 * scratch array compiled into the library: GEMM_NVFP4_NOALLOC_SCRATCH_BYTES (16 MiB) of
 * device memory on every GPU that loads the library, held until the process exits.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Operands, layouts, result, constraints and errors are those of gemm_nvfp4, plus:
 *   - the problem must satisfy
 *       round_up(gemm_nvfp4_blocked_scale_bytes(M, K), 256) + gemm_nvfp4_blocked_scale_bytes(N, K)
 *         <= GEMM_NVFP4_NOALLOC_SCRATCH_BYTES
 *     (e.g. M = N = 8192 allows K up to 16384); larger problems return
 *     GEMM_ERR_SCRATCH_TOO_SMALL and launch nothing;
 *   - the first call on a device looks up the scratch array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make that first
 *     call before any stream capture;
 *   - every call on a device uses the same scratch array, which keeps the last call's
 *     contents (each call rewrites all of the part it reads, so nothing needs clearing).
 *     Calls whose work overlaps on the GPU -- on different streams without ordering
 *     between them -- race on it: order them on one stream or with events.
 *   - with 1 <= M < 32, A's rows are also copied (by the packing launch) into the array after
 *     the scales, as a 32-row buffer the GEMM reads (gemm_options_t.no_pad_a), when the
 *     array has room for it (32 * K / 2 more bytes); otherwise A is read in place.
 * Launches: one scale-packing kernel (SFA and SFB together; for few rows also the copy of
 * A) and the gemm_nvfp4_blocked kernel, on `stream`.
 */
#define GEMM_NVFP4_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
int gemm_nvfp4_noalloc(const void* A, const void* SFA, const void* B, const void* SFB, void* C,
                       int M, int N, int K, void* stream);

/* Human-readable name of a gemm_status_t value (static string, never NULL). */
const char* gemm_status_string(int status);

/*
 * gemm_get_device_status -- synchronises `stream`, then reads and clears the
 * device status word. Returns GEMM_OK if no kernel reported a problem since
 * the last call, else the code a kernel stored (GEMM_ERR_TIMEOUT). If
 * `detail` is not NULL it receives the full 32-bit word (bits 8-15: the role
 * whose wait expired, 1 = TMA producer, 2 = MMA issuer, 3 = epilogue,
 * 4 = scale-factor producer; bits 16-31: the stage or slot index).
 * Returns GEMM_ERR_NO_DEVICE if the synchronisation itself fails.
 */
int gemm_get_device_status(void* stream, uint32_t* detail);

/* ---------------------------------------------------------------------------
 * Variants and introspection (ablation studies, tests, benchmarks).
 * ------------------------------------------------------------------------- */

typedef enum {
    GEMM_KERNEL_DEFAULT = 0,        /* what gemm_bf16 / gemm_nvfp4 launch */
    GEMM_KERNEL_BF16_1CTA = 1,      /* BF16, cta_group::1, 128 x 256 tile per CTA */
    GEMM_KERNEL_BF16_2CTA = 2,      /* BF16, cta_group::2, 256 x 256 tile per CTA pair, 3 stages of
                                       128 K (8 MMAs per stage), double-buffered accumulator: the
                                       default where gemm_bf16_wide_rule does not select the wide tile */
    GEMM_KERNEL_BF16_2CTA_K64 = 3,  /* the same with 6 stages of 64 K (4 MMAs per stage) */
    GEMM_KERNEL_BF16_2CTA_WIDE = 4  /* BF16, cta_group::2, 512 x 256 tile per CTA pair: each CTA
                                       holds 256 rows as two 128-row M-waves whose accumulators
                                       fill TMEM; 4 stages of 64 K; static schedule only
                                       (clc = 1 is GEMM_ERR_INVALID_ARG) */
} gemm_kernel_t;

typedef struct {
    int kernel;          /* gemm_kernel_t; GEMM_KERNEL_DEFAULT picks the default */
    int persistent;      /* 1: grid = min(tiles, co-resident clusters); 0: one cluster per tile */
    int group_m;         /* tile-order group size along M (>= 1); 0 = chosen from the shape */
    int max_clusters;    /* cap on launched clusters for the persistent grid; 0 = no cap */
    uint32_t wait_limit_us;   /* bound on each internal wait; 0 = default (2 s) */
    uint32_t debug_flags;     /* 0 in production; 1 = make the MMA issuer wait on a barrier
                                 nobody arrives on (exercises the timeout path) */
    int no_tail_split;   /* 0: when the last wave of a persistent grid is at most half full,
                            its tiles are computed as two N-halves each; 1: never */
    int no_pdl;          /* 0: launch with programmatic stream serialization (the kernel's
                            set-up overlaps the end of the previous kernel on the stream;
                            every global access waits for that kernel); 1: plain launch */
    int no_swap_ab;      /* BF16, default kernel (fused epilogue or not): 0 = a GEMM with M <= 128
                            and N >= 256 computes C^T = B A^T, so that the few rows of A fill
                            the MMA's N dimension (64 or 128) instead of padding its 256 rows,
                            and its epilogue writes C transposed; 1 = never */
    int no_split_k;      /* swapped BF16 GEMMs with at most half as many tiles as clusters:
                            0 = split K over 2 to 8 clusters per tile (at least 4 stages of
                            128 K each; two splits only for tile N 64 with at least 48 stages);
                            the splits write FP32 partial sums to a workspace from the
                            library's stream-ordered pool (as gemm_nvfp4's); a second kernel
                            adds them and rounds to BF16, except for two splits, which run as
                            one cluster of two CTA pairs per tile whose first pair adds the
                            second pair's partials itself; with a fused epilogue, the kernel
                            that adds the partials applies it; 1 = never */
    int clc;             /* persistent grids (persistent = 1, max_clusters = 0): 0 = decided by
                            gemm_clc_rule; 1 = cluster launch control: one cluster per work item
                            is launched, and each running cluster takes the items of clusters it
                            cancels before they start (dynamic tile scheduling); 2 = never: the
                            co-resident clusters walk the items with a fixed stride */
    int no_pad_a;        /* NVFP4 with 1 <= M < 32 (gemm_nvfp4*, gemm_nvfp4_blocked*): 0 = A's M rows
                            are first copied (by the scale-packing launch, or by a small copy
                            kernel) into a 32-row buffer from the library's stream-ordered pool,
                            and the GEMM reads A from there (rows M..31 are not written; they
                            only reach C rows that are never stored). All CTA pairs reading an
                            A that spans fewer than 32 rows of codes ran measurably slower on
                            GB300 (46.1 -> 31.9 us at M = 1, N = 28672, K = 8192, blocked
                            scales); 1 = never (A read in place, no allocation) */
    unsigned long long* clock_probe; /* NULL in production. Else device memory of 4 values per CTA
                            for the GEMM kernel's launch (not the scale-packing, copy or
                            split-K reduction kernels): thread 0 of CTA b (b < clock_probe_ctas)
                            stores at [4b] %globaltimer (ns) and at [4b+1] the SM's clock64
                            when its work starts (after waiting for the previous kernel on
                            the stream), and at [4b+2], [4b+3] the same when it ends (after
                            its teardown barrier). (dclock / dtime) is the SM clock the CTA
                            ran at: nvidia-smi samples every 100 ms or so and cannot see a
                            burst of a few launches. The caller owns the buffer; a call that
                            launches several GEMMs (a K split) overwrites it */
    int clock_probe_ctas; /* CTAs the buffer holds (>= 0; CTAs beyond it store nothing); must be 0
                            when clock_probe is NULL */
} gemm_options_t;

/* gemm_bf16 with explicit options (NULL options = defaults). Same contract as gemm_bf16. */
int gemm_bf16_ex(const void* A, const void* B, void* C, int M, int N, int K, void* stream,
                 const gemm_options_t* options);

/* gemm_nvfp4 with explicit options (only persistent, group_m, max_clusters,
 * wait_limit_us, debug_flags, no_tail_split, no_pdl, clc and no_pad_a apply; kernel must
 * be GEMM_KERNEL_DEFAULT). */
int gemm_nvfp4_ex(const void* A, const void* SFA, const void* B, const void* SFB, void* C,
                  int M, int N, int K, void* stream, const gemm_options_t* options);

/* gemm_nvfp4_blocked with explicit options (as for gemm_nvfp4_ex). */
int gemm_nvfp4_blocked_ex(const void* A, const void* SFA_blocked, const void* B, const void* SFB_blocked, void* C,
                          int M, int N, int K, void* stream, const gemm_options_t* options);

/*
 * Fused epilogue ("NVFP4 GEMM on Blackwell", epilogue section: the accumulator in
 * registers is where activation, bias and alpha/beta scaling belong). Each output element,
 * while its FP32 accumulator is in registers:
 *
 *     C[i][j] = act(alpha * (A B^T)[i][j] + beta * C_old[i][j] + bias[j])
 *
 * evaluated in FP32 in that order and rounded once to BF16 (round to nearest, ties to
 * even). act is the identity, max(x, 0), or the tanh form of GELU,
 * 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
 *   alpha       scales the product.
 *   beta        scales the prior contents of C. With beta == 0, C is not read (it may
 *               hold anything, NaN included).
 *   bias        device pointer to N BF16 values (one per column), 16-byte aligned, or NULL
 *               for none. Caller-owned, read only.
 *   activation  GEMM_ACT_NONE, GEMM_ACT_RELU or GEMM_ACT_GELU_TANH; anything else is
 *               GEMM_ERR_INVALID_ARG.
 *   reserved    must be 0.
 * A NULL epilogue pointer is the identity (alpha 1, beta 0, no bias, no activation).
 * With K == 0 the product is zero and the epilogue still applies to C.
 */
typedef enum { GEMM_ACT_NONE = 0, GEMM_ACT_RELU = 1, GEMM_ACT_GELU_TANH = 2 } gemm_activation_t;

typedef struct {
    float alpha;
    float beta;
    const void* bias;
    int activation;
    int reserved;
} gemm_epilogue_t;

/* gemm_bf16_ex, gemm_nvfp4_ex and gemm_nvfp4_blocked_ex with a fused epilogue. The
 * arguments, layouts, preconditions and errors are those of the unfused calls, plus: a
 * non-NULL bias not 16-byte aligned is GEMM_ERR_MISALIGNED. */
int gemm_bf16_fused(const void* A, const void* B, void* C, int M, int N, int K, void* stream,
                    const gemm_epilogue_t* epilogue, const gemm_options_t* options);
int gemm_nvfp4_fused(const void* A, const void* SFA, const void* B, const void* SFB, void* C, int M, int N, int K,
                     void* stream, const gemm_epilogue_t* epilogue, const gemm_options_t* options);
int gemm_nvfp4_blocked_fused(const void* A, const void* SFA_blocked, const void* B, const void* SFB_blocked, void* C,
                             int M, int N, int K, void* stream, const gemm_epilogue_t* epilogue,
                             const gemm_options_t* options);

/*
 * gemm_clc_rule -- whether a persistent launch with gemm_options_t.clc = 0 schedules its
 * work items with cluster launch control (dynamic tile scheduling; "NVFP4 GEMM on
 * Blackwell", static vs dynamic tile scheduling): items = work items of the launch (tiles,
 * plus the extra halves of a split tail wave, or tiles x K splits), wave = co-resident
 * clusters, K = the GEMM's K, nvfp4 = 1 for the NVFP4 kernel, 0 for BF16. Returns 1 for a
 * BF16 launch with items > wave and K >= 16384, else 0 (a rule measured on GB300: below
 * that depth, and for NVFP4 at the depths measured, the static order, which keeps each SM
 * pair on the same position of every wave, reads far fewer bytes from DRAM);
 * -GEMM_ERR_INVALID_ARG if an argument is negative, wave is 0 or nvfp4 is not 0 or 1.
 */
int gemm_clc_rule(int items, int wave, int K, int nvfp4);

/*
 * gemm_bf16_wide_rule -- whether gemm_bf16 / gemm_bf16_fused (default kernel, static schedule,
 * not swapped) computes this problem on the 512 x 256 pair tile (GEMM_KERNEL_BF16_2CTA_WIDE)
 * rather than the 256 x 256 one, with `wave` co-resident clusters (76 on a 152-SM GB300).
 * Host evaluation, no GPU needed. The rule ("Achieve cuBLAS Performance on NVIDIA GB300 for
 * HGEMM", v7: the larger tile moves fewer bytes per FLOP; the choice by wave quantization is
 * this library's): K >= 2048, and the launch's estimated length in 256 x 256 tile-times is
 * shorter with wide tiles, each counting 2 / f of a 256 x 256 one, f = 1.03 for K < 4096 and
 * 1.06 from K = 4096 (the per-work gain measured in sustained runs); a launch of T tiles on
 * W clusters lasts floor(T / W) tile-times plus, for a partial last wave, 1 (or 0.8 when its
 * tiles run as N-halves, 2 (T mod W) <= W).
 * Returns 1 or 0; -GEMM_ERR_INVALID_ARG if a size is negative or wave <= 0.
 */
int gemm_bf16_wide_rule(int M, int N, int K, int wave);

/*
 * gemm_tile_coord -- host evaluation of the persistent tile order used by the
 * kernels (no GPU needed). The output is split into ceil(M/tile_m) x
 * ceil(N/tile_n) tiles; tile index t (0 <= t < tiles) is mapped to the block
 * coordinates (*m_blk, *n_blk). Tiles are walked M-first inside groups of
 * group_m consecutive M-blocks, group after group; the last group may be
 * shorter ("Achieve cuBLAS Performance on NVIDIA GB300 for HGEMM", v6 tile
 * swizzle). Returns GEMM_ERR_INVALID_ARG for out-of-range arguments.
 */
int gemm_tile_coord(int M, int N, int tile_m, int tile_n, int group_m, int t, int* m_blk, int* n_blk);

/*
 * gemm_choose_group_m -- the group size the library picks for a problem when
 * options->group_m is 0. Balances the bytes of A and B that the tiles of two
 * waves of co-resident clusters (concurrent_tiles each) touch, and shrinks the
 * group until that footprint fits in the L2 cache ("NVFP4 GEMM on Blackwell",
 * Production Kernel, "Supergroup Size", with the roles of M and N exchanged
 * because the groups here run along M). Two waves: each wave starts on the K
 * blocks the previous one read last, so their operands share L2. elem_bytes_x2 is twice the bytes per operand element
 * (4 for BF16, 1 for packed E2M1 plus the scale bytes counted separately:
 * pass 1 and the function adds K/16 scale bytes per row).
 */
int gemm_choose_group_m(int M, int N, int K, int tile_m, int tile_n, int elem_bytes_x2,
                        int concurrent_tiles, long long l2_bytes);

/*
 * gemm_bf16_plan -- the configuration gemm_bf16_ex / gemm_bf16_fused use for a problem
 * (host only, no GPU needed): *swap_ab = 1 when the call computes C^T = B A^T (see
 * gemm_options_t.no_swap_ab), *tile_n = the MMA N of its tiles (256; 64 or 128 when
 * swapped). options and epilogue may be NULL. Returns GEMM_ERR_INVALID_ARG for negative
 * sizes, null outputs or invalid options.
 */
int gemm_bf16_plan(int M, int N, int K, const gemm_options_t* options, const gemm_epilogue_t* epilogue, int* swap_ab,
                   int* tile_n);

/*
 * gemm_nvfp4_plan -- host evaluation of the NVFP4 configuration choice (no GPU needed):
 * *a_rows = the rows of A the GEMM kernel reads: 32 when A is first copied into a padded
 * 32-row workspace (1 <= M < 32 and options->no_pad_a == 0), else M. options may be NULL.
 * Returns GEMM_ERR_INVALID_ARG for negative sizes, a null output or invalid options.
 */
int gemm_nvfp4_plan(int M, int N, int K, const gemm_options_t* options, int* a_rows);

/* Number of kernel launches this library has issued in this process (all devices). */
unsigned long long gemm_launch_count(void);

/*
 * gemm_measure_mma_rate -- measures, on the current device, the throughput of one
 * tensor-core MMA instruction form as FLOP per SM clock: one issuing thread per CTA pair
 * (cta_group::2, M = 256) or per CTA (cta_group::1, M = 128) issues 8192 back-to-back
 * MMAs from shared memory into TMEM, timed with the SM clock (the second of two launches).
 *   kind: GEMM_MMA_BF16  -- kind::f16, BF16 operands, K = 16, M = 256, N = 256 (the BF16 GEMM);
 *         GEMM_MMA_NVFP4 -- kind::mxf4nvf4.block_scale.scale_vec::4X, E2M1 operands with
 *                           UE4M3 scales per 16 elements, K = 64, M = 256, N = 256 (the NVFP4 GEMM);
 *         GEMM_MMA_NVFP4_1CTA_N128 / _N192 / _N256 -- the same kind at M = 128 (cta_group::1);
 *         GEMM_MMA_NVFP4_PAIR_N128 -- M = 256, N = 128, one accumulator;
 *         GEMM_MMA_NVFP4_PAIR_N128_2ACC -- M = 256, N = 128, alternating between two accumulators;
 *         GEMM_MMA_MXF4_PAIR_N256 -- kind::mxf4.block_scale.scale_vec::2X (UE8M0 scales per 32
 *                           elements), K = 64, M = 256, N = 256.
 *   *flop_per_clock_per_sm: the result (2 * 128 * N * K per instruction and SM, per clock).
 * It is the ceiling a kernel made of these instructions can reach per clock; multiplied
 * by the SM count and clock it gives TFLOP/s. Synchronous: it runs on a private stream
 * and waits for it. Device memory: none beyond the library's static device arrays.
 * Errors: GEMM_ERR_INVALID_ARG (unknown kind, null pointer), device errors as for the
 * GEMMs, GEMM_ERR_TIMEOUT if the MMAs did not complete within 2 s.
 */
enum {
  GEMM_MMA_BF16 = 0,
  GEMM_MMA_NVFP4 = 1,
  GEMM_MMA_NVFP4_1CTA_N128 = 2,
  GEMM_MMA_NVFP4_1CTA_N192 = 3,
  GEMM_MMA_NVFP4_1CTA_N256 = 4,
  GEMM_MMA_NVFP4_PAIR_N128 = 5,
  GEMM_MMA_NVFP4_PAIR_N128_2ACC = 6,
  GEMM_MMA_MXF4_PAIR_N256 = 7
};
int gemm_measure_mma_rate(int kind, double* flop_per_clock_per_sm);

#ifdef __cplusplus
}
#endif

#endif /* DTCP_GEMM_H */
