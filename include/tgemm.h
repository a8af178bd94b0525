/*
 * tgemm — dense matrix multiplication C = A x B for one NVIDIA GB300 (sm_103a).
 *
 * C ABI of libtgemm.so. Every entry point takes plain sizes, pointers and a
 * CUDA stream; no C++ or framework type crosses this boundary.
 *
 * The operation is the product defined in "Tiled Matrix Multiplication in
 * CUDA", section 1 ("What matrix multiplication actually does"), and
 * "Tiled GEMM: Matrix Multiplication in CUDA", section 1:
 *
 *     C[i][j] = sum over k = 0 .. K-1 of A[i][k] * B[k][j]
 *
 * for 0 <= i < M, 0 <= j < N. All three matrices are row-major and addressed
 * by the flat index row * ld + col ("Tiled Matrix Multiplication in CUDA",
 * section 2), where ld is the leading dimension: the number of elements
 * between the starts of two consecutive rows (ld >= the row length; ld larger
 * than the row length describes a sub-matrix of a wider array). The pages'
 * square "width" is generalised to M, N, K with one leading dimension per
 * matrix, following the ragged-edge code of "Tiled GEMM: Matrix
 * Multiplication in CUDA", section 7.1.
 *
 * Common rules for the compute entry points:
 *   - A, B and C are DEVICE pointers (memory the caller allocated on the
 *     current CUDA device). The library never allocates, frees or copies the
 *     caller's buffers, and keeps no reference to them after the call.
 *   - Scratch memory. A call may need device memory of its own while it
 *     runs, for two things:
 *       (a) operands rewritten into a layout the kernels read: on the
 *           tensor paths, an operand whose rows do not start
 *           on 16-byte boundaries, repacked (rows on 128-byte boundaries);
 *           on gemm_f32, both operands repacked when their rows are off 16
 *           bytes and M >= 256, N >= 256, K >= 64; on TGEMM_TF32X3, high
 *           and low copies of A and of B transposed; on gemm_ex, storage a
 *           path cannot read (transposes);
 *       (b) the partial tiles of a last wave split along K, when the
 *           planner splits it: (tiles - whole tiles) x pieces x tile rows x
 *           tile columns x 4 bytes. gemm_f32 on 4096^3 splits 56 of its 512
 *           128 x 256 tiles into 8 pieces: 56 x 8 x 128 x 256 x 4 B = 59 MB.
 *     Such a call takes one block with cudaMallocFromPoolAsync on `stream`
 *     from a memory pool that the library creates once per device, and
 *     gives it back with cudaFreeAsync on `stream` before returning. The
 *     pool keeps the memory it has handed out (no release threshold), so
 *     once a call of a given size has run, later calls reuse the cached
 *     memory without going to the driver; it stays reserved until the
 *     process exits. A call that needs neither (a) nor (b) allocates
 *     nothing: gemm_f32, and gemm_tc TGEMM_BF16 and TGEMM_TF32, on operands
 *     with 16-byte rows whose tiles fill whole waves or whose tail is not
 *     split.
 *     gemm_scratch_bytes() returns the size a call would draw, and
 *     gemm_tc_tf32_noalloc() never allocates.
 *   - C is overwritten (there is no alpha/beta); K == 0 writes zeros to the
 *     M x N block of C; M == 0 or N == 0 is a no-op that returns TGEMM_OK.
 *   - Elements of A, B and C outside the M x K, K x N and M x N blocks (the
 *     padding between the row length and ld) are never read or written.
 *   - C must not overlap A or B; overlap is undefined behaviour.
 *   - The call is asynchronous: it validates its arguments, enqueues the work
 *     on `stream` (0 = the legacy default stream) and returns. A launch
 *     failure is reported as TGEMM_ERR_CUDA. Faults found while the kernel
 *     runs (a bounded wait that ran out) are reported later, by
 *     gemm_device_status(). Every kernel is launched with programmatic
 *     dependent launch: it may be scheduled while the previous kernel on
 *     `stream` finishes, and sets up its shared and tensor memory then, but
 *     it touches no global memory before that kernel has completed and its
 *     writes are visible -- stream order is kept. Calls may be captured in a
 *     CUDA graph (after a first call outside capture on the device).
 *   - Arguments are checked before any CUDA call is made; an invalid call
 *     returns an error code and enqueues nothing.
 *   - The calls are thread-safe for distinct streams; configuration setters
 *     (gemm_set_*) are process-wide and should be called before launching.
 */
#ifndef TGEMM_H
#define TGEMM_H

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define TGEMM_API __attribute__((visibility("default")))
#else
#define TGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
#define TGEMM_OK                    0
#define TGEMM_ERR_INVALID_ARG       1  /* negative size, ld too small, null pointer, bad in_type */
#define TGEMM_ERR_ALIGNMENT         2  /* a forced kernel or the no-alloc entry cannot read this layout */
#define TGEMM_ERR_CUDA              3  /* a CUDA runtime call or launch failed */
#define TGEMM_ERR_DEVICE_TIMEOUT    4  /* a bounded wait inside a kernel ran out (see gemm_device_status) */
#define TGEMM_ERR_UNSUPPORTED       5  /* the current device is not compute capability 10.3 (sm_103) */

/* Input element types of gemm_tc. */
#define TGEMM_TF32  1   /* A and B are float arrays; products use the TF32 tensor-core format */
#define TGEMM_BF16  2   /* A and B are bfloat16 arrays (uint16 bit patterns) */
#define TGEMM_TF32X3 3  /* A and B are float arrays; each is split into a high and a low
                           TF32 part and three tensor-core products (lo*hi + hi*lo + hi*hi)
                           give FP32-level accuracy */

/*
 * gemm_f32 — exact-FP32 product on the CUDA cores.
 *
 * Computes C = A x B with A: M x K floats (leading dimension lda >= K),
 * B: K x N floats (ldb >= N), C: M x N floats (ldc >= N). Each output is
 * accumulated in FP32 with fused multiply-adds in ascending k within a thread
 * (the phase loop over K-tiles and the inner loop inside a tile of "Tiled
 * GEMM: Matrix Multiplication in CUDA", sections 2 and 4.3-4.6). Tiles of A
 * and B are staged through shared memory; rows and columns past M, N, K read
 * as zero (section 7.1 of the same page), so any M, N, K >= 0 is accepted.
 * Any lda/ldb/ldc and 4-byte aligned pointers work; 16-byte aligned pointers
 * with ld a multiple of 4 take 16-byte vector loads. Scratch (see the common
 * rules): the two operands repacked to 16-byte rows when they are large and
 * off 16 bytes, and the partial tiles when the tiles of a partial last wave
 * are split along K; neither when the operands have 16-byte rows and the
 * 128 x 256 tiles fill whole waves of the SMs.
 *
 * Returns TGEMM_OK, TGEMM_ERR_INVALID_ARG (M, N or K negative; lda < K,
 * ldb < N or ldc < N; a null pointer when the product is not empty; a pointer
 * not 4-byte aligned), TGEMM_ERR_UNSUPPORTED or TGEMM_ERR_CUDA.
 */
TGEMM_API int gemm_f32(int M, int N, int K,
             const float* A, long lda,
             const float* B, long ldb,
             float* C, long ldc,
             cudaStream_t stream);

/*
 * gemm_tc — product on the 5th-generation tensor cores (tcgen05, TMEM
 * accumulators), FP32 output.
 *
 * Same product and layout as gemm_f32. A and B hold `in_type` elements:
 *   TGEMM_TF32: A and B are float arrays; the tensor core multiplies them in
 *               the TF32 format (10 explicit mantissa bits) and accumulates in
 *               FP32.
 *   TGEMM_BF16: A and B are bfloat16 arrays; products are exact and are
 *               accumulated in FP32.
 *   TGEMM_TF32X3: A and B are float arrays. Each element x is split into
 *               hi = x rounded to TF32 and lo = (x - hi) rounded to TF32
 *               (stream-ordered scratch: A as hi/lo copies, B transposed as
 *               hi/lo copies), and every K step accumulates
 *               lo(A)hi(B) + hi(A)lo(B) + hi(A)hi(B) in FP32; the omitted
 *               lo(A)lo(B) term is below 2^-22 of each product, so the result
 *               meets the FP32 path's accuracy at a third of the TF32 rate.
 * C is FP32 (ldc >= N, any alignment). Tiles of A and B are copied by the
 * Tensor Memory Accelerator, which needs rows that start on 16-byte
 * boundaries: an operand whose pointer or leading dimension breaks that
 * (any lda, ldb and element-aligned pointer are accepted) is first repacked
 * by an HBM-bound kernel into stream-ordered scratch with rows on 128-byte
 * boundaries. B is read as stored, K x N (MN-major: BF16 in the 128-byte
 * swizzle, TF32 in the 128-byte swizzle with 32-byte atoms). Rows and
 * columns past M, N, K read as zero. Scratch (see the common rules): the
 * repacked operands, and the partial tiles of a split last wave; operands
 * with 16-byte rows whose tail is not split allocate nothing.
 *
 * Returns TGEMM_OK, TGEMM_ERR_INVALID_ARG (as gemm_f32, a bad in_type, or
 * a pointer not aligned to its element size), TGEMM_ERR_UNSUPPORTED or
 * TGEMM_ERR_CUDA.
 */
TGEMM_API int gemm_tc(int M, int N, int K,
            const void* A, long lda,
            const void* B, long ldb,
            float* C, long ldc,
            int in_type,
            cudaStream_t stream);

/* Paths of gemm_ex and gemm_host. */
#define TGEMM_PATH_F32    0   /* gemm_f32: FP32 on the CUDA cores, A and B float */
#define TGEMM_PATH_TF32   1   /* gemm_tc TGEMM_TF32: A and B float */
#define TGEMM_PATH_BF16   2   /* gemm_tc TGEMM_BF16: A and B bfloat16 */
#define TGEMM_PATH_TF32X3 3   /* gemm_tc TGEMM_TF32X3: A and B float */

/* Storage flags of gemm_ex. */
#define TGEMM_TRANS_A 1   /* A is stored K x M (lda >= M): op(A) = A^T, i.e. A column-major */
#define TGEMM_TRANS_B 2   /* B is stored N x K (ldb >= K): op(B) = B^T, i.e. B column-major */

/*
 * gemm_ex — the product with transposed storage and the usual output rule:
 *
 *     C = alpha * op(A) * op(B) + beta * C + bias
 *
 * for the M x N block of C, with op(A) M x K and op(B) K x N: op(A) = A
 * (stored M x K, lda >= K) or, with TGEMM_TRANS_A, A stored K x M
 * (lda >= M) read transposed -- an M x K matrix kept column-major, the
 * opposite convention "Tiled Matrix Multiplication in CUDA", section 2 names;
 * op(B) likewise with TGEMM_TRANS_B (B stored N x K, ldb >= K). `bias` is
 * NULL or N floats (device memory), added to every row (the per-feature
 * bias of a feed-forward layer); C is not read when beta == 0, so it may
 * hold anything then. Each output is computed as
 *     v = alpha * acc;  if (beta != 0) v = fmaf(beta, C_old, v);  v += bias[j]
 * in FP32, acc being the path's accumulated product.
 *
 * `path` is one of TGEMM_PATH_F32 (gemm_f32's arithmetic), _TF32, _BF16,
 * _TF32X3 (gemm_tc's), with A and B of that path's element type. Storage the
 * path's kernels cannot read directly is rewritten first by HBM-bound
 * kernels into stream-ordered scratch (transposes; the tensor paths read A
 * K-major, and B either MN-major or K-major, so TRANS_B needs no copy
 * there). With
 * flags 0, alpha 1, beta 0 and no bias it is exactly gemm_f32 / gemm_tc.
 *
 * Returns TGEMM_OK, TGEMM_ERR_INVALID_ARG (as gemm_f32 with the ld rules
 * above, an unknown path or flag, a bias pointer not 4-byte aligned),
 * TGEMM_ERR_ALIGNMENT (a forced FP32 configuration cannot read the layout),
 * TGEMM_ERR_UNSUPPORTED or TGEMM_ERR_CUDA.
 */
TGEMM_API int gemm_ex(int M, int N, int K,
                      const void* A, long lda,
                      const void* B, long ldb,
                      float* C, long ldc,
                      int path, int flags,
                      float alpha, float beta, const float* bias,
                      cudaStream_t stream);

/*
 * gemm_host — the same product for operands and result in HOST memory.
 *
 * A (M x K, lda >= K), B (K x N, ldb >= N) and C (M x N floats, ldc >= N)
 * are host pointers, ideally page-locked (cudaHostAlloc / pinned), with
 * elements of the path's type; `path` is any TGEMM_PATH_*. The call stages
 * them through stream-ordered device scratch from the library's pool and
 * overlaps the transfers with the multiplication: B is copied first, A
 * follows in up to four row panels on a copy stream (on the FP32 path a
 * short first and last panel, so that the arithmetic starts early and little
 * of C is left to copy out at the end; there B goes up in two column halves
 * and the first panel is multiplied in the same halves, the left one as soon
 * as it has arrived), each panel is
 * multiplied on `stream` as soon as its rows have arrived (TF32X3 splits
 * and transposes B once for all panels and splits each panel of A as it
 * arrives), and each panel of C is copied back on a second copy
 * stream while the next panel computes. Same arithmetic and result as
 * gemm_f32 / gemm_tc on device copies of the operands.
 *
 * The call is asynchronous like cudaMemcpyAsync: it returns once the work is
 * enqueued; C is complete (and A, B may be reused) when `stream` has been
 * synchronised. Calls in flight together (on different streams) copy their
 * operands to the device in call order on one library stream and copy their
 * results back on separate library streams (four, taken in turn), so one
 * call's results do not wait for another's. With pageable host memory the
 * CUDA copies become synchronous and there is no overlap. Returns TGEMM_OK,
 * TGEMM_ERR_INVALID_ARG (as gemm_f32, or an unknown path, or an operand not
 * aligned to its element size), TGEMM_ERR_UNSUPPORTED or TGEMM_ERR_CUDA.
 */
TGEMM_API int gemm_host(int M, int N, int K,
                        const void* A, long lda,
                        const void* B, long ldb,
                        float* C, long ldc,
                        int path,
                        cudaStream_t stream);

/*
 * gemm_scratch_bytes — the device scratch, in bytes, that the call
 *     gemm_ex(M, N, K, A, lda, B, ldb, C, ldc, path, flags, 1, 0, NULL, s)
 * would draw from the library's pool on the current device (see "Scratch
 * memory" above); gemm_f32 and gemm_tc are that call with flags 0 and
 * their path. The pointers are not dereferenced: only their alignment
 * matters, as it decides which operands are repacked and how C is stored.
 * Returns the size (0 when the call allocates nothing), or a negative
 * status code (-TGEMM_ERR_INVALID_ARG for arguments the call would reject,
 * -TGEMM_ERR_ALIGNMENT, -TGEMM_ERR_UNSUPPORTED, -TGEMM_ERR_CUDA). Makes no
 * CUDA call other than reading the device's attributes.
 */
TGEMM_API long long gemm_scratch_bytes(int M, int N, int K,
                                       const void* A, long lda,
                                       const void* B, long ldb,
                                       const float* C, long ldc,
                                       int path, int flags);

/*
 * gemm_plan_name — the kernels that the call
 *     gemm_ex(M, N, K, A, lda, B, ldb, C, ldc, path, flags, 1, 0, NULL, s)
 * would launch on a device with `num_sms` SMs, under the current settings
 * (gemm_set_*), written to `buf` (at most buf_len bytes, NUL-terminated) in
 * the form gemm_last_kernel reports after the call: the pre-passes, the
 * GEMM kernel's configuration, its tail. "" when M or N is 0,
 * "empty_product" when K is 0. The pointers are not dereferenced (only their
 * alignment matters) and no CUDA call is made, so the planner's choices can
 * be checked without a GPU. Returns TGEMM_OK, TGEMM_ERR_INVALID_ARG (as
 * gemm_scratch_bytes, or num_sms < 2, or no buffer) or TGEMM_ERR_ALIGNMENT.
 */
TGEMM_API int gemm_plan_name(int M, int N, int K,
                             const void* A, long lda,
                             const void* B, long ldb,
                             const float* C, long ldc,
                             int path, int flags, int num_sms,
                             char* buf, int buf_len);

/*
 * gemm_device_status — result of the kernels' bounded waits.
 *
 * Synchronises `stream`, then returns and clears the library's device-side
 * status word on the current device: TGEMM_OK if no kernel launched since the
 * last call gave up on a wait, TGEMM_ERR_DEVICE_TIMEOUT if one did (that
 * kernel's output is then incomplete), or TGEMM_ERR_CUDA if synchronising or
 * reading the word failed. A kernel that gives up releases its tensor memory
 * and exits normally, so the CUDA context stays usable.
 */
TGEMM_API int gemm_device_status(cudaStream_t stream);

/*
 * gemm_tc_peak — diagnostic: the dense MMA rate of this device's tensor
 * cores, the denominator a tensor-core roofline can be stated against.
 *
 * Every SM (pair = 0: 128 x 256 MMAs, cta_group::1) or SM pair (pair = 1:
 * 256 x 256 MMAs, cta_group::2) issues `iters` (1 .. 1e8) MMAs of in_type
 * TGEMM_BF16 (K = 16 per MMA) or TGEMM_TF32 (K = 8) back to back, from
 * operands resident in shared memory into one tensor-memory accumulator;
 * nothing is loaded or stored. Writes *flop_per_clk_sm, the dense FLOP per
 * SM clock cycle (2*M*N*K per MMA, median over the units, measured with the
 * SM clock counter), and *tflops, the rate of all SMs over the launch's
 * device time (start-up included) at whatever clock the GPU ran. Allocates
 * and frees a small device buffer and synchronises `stream`. Returns
 * TGEMM_OK, TGEMM_ERR_INVALID_ARG, TGEMM_ERR_UNSUPPORTED, TGEMM_ERR_CUDA or
 * TGEMM_ERR_DEVICE_TIMEOUT (a bounded wait ran out).
 */
TGEMM_API int gemm_tc_peak(int in_type, int pair, long iters, double* flop_per_clk_sm,
                           double* tflops, cudaStream_t stream);

/*
 * gemm_status_string — a static, human-readable name for a status code.
 * Never returns NULL; unknown codes give "unknown tgemm status".
 */
TGEMM_API const char* gemm_status_string(int status);

/*
 * gemm_set_wait_limit_ns — upper bound, in nanoseconds, on any single wait
 * inside the tensor-core kernel (a pipeline stage, the accumulator hand-off).
 * Must be > 0; the default is 2 000 000 000 (2 s). Process-wide; applies to
 * launches made after the call. Returns TGEMM_OK or TGEMM_ERR_INVALID_ARG.
 */
TGEMM_API int gemm_set_wait_limit_ns(long long ns);

/*
 * gemm_set_debug_stall — failure-detection hook for tests. When `enable` is
 * non-zero, the next gemm_tc launches never signal the first pipeline stage
 * as loaded, so the consumer's bounded wait runs out and the kernel exits
 * through its timeout path (reporting TGEMM_ERR_DEVICE_TIMEOUT through
 * gemm_device_status). Off by default; process-wide. Returns TGEMM_OK.
 */
TGEMM_API int gemm_set_debug_stall(int enable);

/*
 * gemm_set_f32_kernel — force one FP32 kernel configuration (for tests and
 * tuning): -1 restores automatic per-shape selection; 0 .. gemm_f32_kernel_count()-1
 * selects that entry of the library's table. Process-wide. Returns TGEMM_OK
 * or TGEMM_ERR_INVALID_ARG.
 */
TGEMM_API int gemm_set_f32_kernel(int id);

/*
 * gemm_set_tc_kernel — choose the tensor-core kernel (for tests and tuning):
 * 0 forces the one-SM kernel (128 x 256 tiles), 1 the 2-SM kernel (a CTA
 * pair computing 256 x 256 tiles), 2 the 2-SM kernel with 256 x 512 tiles,
 * 3 the one-SM TF32 kernel that transposes B in shared memory (128 x 128
 * tiles; TGEMM_TF32 with B stored K x N, other products as with -1), 4 the
 * one-SM kernel with 128 x 128 tiles (B read as the 128 x 256 one-SM kernel
 * reads it); -1 (default) picks by shape: for M <= 128 the one-SM
 * kernel with 128 x 256 or 128 x 128 tiles, whichever the timing model
 * expects to finish first (the narrower tiles fill more SMs), 256 x 256
 * tiles when N <= 256, and otherwise the pair shape that a timing model of
 * the two expects to finish first (whole-tile rounds over the SM pairs, the
 * cost of a split last wave, a main-loop rate per shape and type measured
 * on this GPU, and the exposed write-out of the 256 x 512 tiles), with
 * near-ties (the wide tiles less than 3 % faster) going to 256 x 256.
 * TGEMM_TF32X3 always runs 256 x 256 pair tiles. Process-wide. Returns
 * TGEMM_OK or TGEMM_ERR_INVALID_ARG.
 */
TGEMM_API int gemm_set_tc_kernel(int mode);

/*
 * gemm_set_tc_streamk — the stream-K tail of the tensor-core kernels (for
 * tests and tuning). When a product's tiles do not fill whole rounds of the
 * SMs (one-SM kernel) or SM pairs, the tiles of the partial last round can
 * instead have their K blocks shared evenly by S of them inside the same
 * launch: each computes a share of at most one tile's length, writes the
 * partial tile of a share that does not end a tile to scratch, and the SM
 * or pair whose share ends a tile adds the partial tiles of the shares
 * before it (fixed order: deterministic) and stores the tile. In the split
 * form every tail tile is instead cut into k equal shares on k SMs or
 * pairs, which all write their partial tiles and wait for nothing, and a
 * reduction kernel launched after the GEMM kernel adds each tile's shares
 * in K order, applies the output rule and stores the tile (deterministic).
 * -1 (default) takes the form and S or k from a timing model (or no
 * sharing), 0 never shares, S > 0 shares the tail among S (clamped to the
 * SMs or pairs available and to the tail's K blocks; no sharing if that
 * leaves S at or below the tail's tile count), S <= -2 takes the split form
 * with k = -S (clamped so that k times the tail's tiles fits the SMs or
 * pairs; none below k = 2). Process-wide. Returns TGEMM_OK or
 * TGEMM_ERR_INVALID_ARG (slots < -64).
 */
TGEMM_API int gemm_set_tc_streamk(int slots);

/*
 * gemm_set_tc_a_loader — how the tensor paths read an A whose rows are 4-byte
 * but not 16-byte aligned (for tests and tuning). The Tensor Memory
 * Accelerator cannot copy such rows ("Tiled GEMM: Matrix Multiplication in
 * CUDA", section 8, hands tiles to TMA), so A is either repacked first into
 * scratch with 128-byte rows (0, and the default -1) or read in place by two
 * extra warps of the GEMM kernel with 4-byte asynchronous copies into the
 * layout TMA would have written (1; TGEMM_TF32, and TGEMM_BF16 with an even
 * lda and B stored K x N). Process-wide. Returns TGEMM_OK or
 * TGEMM_ERR_INVALID_ARG.
 */
TGEMM_API int gemm_set_tc_a_loader(int mode);

/* Number of FP32 kernel configurations gemm_set_f32_kernel accepts. */
TGEMM_API int gemm_f32_kernel_count(void);

/*
 * gemm_f32_kernel_name — static name of FP32 configuration `id`
 * (tile sizes and loader), or "" for an id out of range.
 */
TGEMM_API const char* gemm_f32_kernel_name(int id);

/*
 * gemm_last_kernel — name of the kernel(s) the most recent successful
 * gemm_f32, gemm_tc or gemm_ex call on this thread launched, in launch
 * order, joined by '+' when a call launched more than one: the pre-passes
 * (repack_a, repack_b, repack_ab -- both operands in one launch --,
 * transpose_a, transpose_b, split_a, split_b, transpose_split_a,
 * transpose_split_b), the GEMM kernel's configuration
 * name, and "splitk_reduce(split=S,tiles=T)" when T tiles of a partial last
 * wave were computed in S K-pieces each and summed by a reduction kernel
 * (FP32 path); a tensor-core kernel's name carries "(streamk:slots=S,tiles=T)"
 * when the K blocks of the T tiles of its partial last round were shared by
 * S SMs or SM pairs inside the kernel (no extra launch), and is followed by
 * "tc_split_reduce(split=k,tiles=T)" when its T tail tiles were computed in
 * k shares each and summed by the tensor paths' reduction kernel;
 * "empty_product" for K == 0, "" if nothing was launched (empty output,
 * error). Valid until the thread's next call. For tests and benchmarks.
 */
TGEMM_API const char* gemm_last_kernel(void);

/*
 * gemm_tc_tf32_noalloc — the TF32 product of gemm_tc(..., TGEMM_TF32, ...)
 * for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for the
 * library's callers. gemm_tc's TF32 path takes scratch memory from a
 * stream-ordered memory pool for operands whose rows are off 16 bytes and
 * for the partial tiles of a split last wave. Callers that
 * must not let a library allocate -- an application or plugin that reserves
 * all of its device memory at start-up and treats any later allocation as a
 * failure, or code that must not touch the device allocator while it runs
 * -- call this instead: it allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine), never splits the last wave, and, when B's
 * rows are off 16 bytes, keeps a transposed B in a fixed array of
 * TGEMM_NOALLOC_SCRATCH_FLOATS floats (16 MiB) in the library's own device
 * memory, which every device that loads the library holds until the process
 * exits.
 *
 * Arguments, layout and result are those of gemm_tc with in_type TGEMM_TF32:
 * A is M x K floats (16-byte aligned, lda >= K and a multiple of 4), B is
 * K x N floats (4-byte aligned, ldb >= N), C is M x N floats (ldc >= N).
 * B whose pointer is 16-byte aligned and ldb a multiple of 4 is read as
 * stored and the array is not touched. Otherwise B transposed goes to the
 * array with rows round_up(K, 32) floats apart
 * (128-byte rows, as gemm_tc) when N * round_up(K, 32) fits in it, else
 * round_up(K, 4) floats apart (16-byte rows; the GEMM kernel reads such rows
 * somewhat slower). The tiles of a partial last wave are never split along
 * K here (that would need more scratch). Waits inside the kernel are bounded
 * by the limit of gemm_set_wait_limit_ns, as for gemm_tc.
 *
 * Returns TGEMM_OK; TGEMM_ERR_INVALID_ARG for the argument errors of gemm_tc,
 * for K > 4194240, and, when B has to be transposed, for
 * N * round_up(K, 4) > TGEMM_NOALLOC_SCRATCH_FLOATS (the problem does not
 * fit the fixed scratch; nothing is launched);
 * TGEMM_ERR_ALIGNMENT; TGEMM_ERR_UNSUPPORTED; TGEMM_ERR_CUDA.
 *
 * The first call on each device does that device's set-up (it looks up the
 * device address of the scratch array with cudaGetSymbolAddress), so make
 * the first call on a device before any stream capture. Every call shares
 * the one array and leaves its contents behind; nothing in it has to start
 * at zero because each call writes the part it reads first. Calls whose work
 * overlaps on the GPU (on different streams or from different host threads)
 * race on the array and give wrong results: serialise them.
 */
#define TGEMM_NOALLOC_SCRATCH_FLOATS 4194304L   /* 16 MiB of floats */

TGEMM_API int gemm_tc_tf32_noalloc(int M, int N, int K,
                                   const float* A, long lda,
                                   const float* B, long ldb,
                                   float* C, long ldc,
                                   cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TGEMM_H */
