// Internal interface between the C-ABI layer (api.cu) and the kernel files.
// Not installed; callers use include/tgemm.h.
#pragma once

#include <cuda_runtime.h>
#include <cstdint>
#include <atomic>
#include <utility>

namespace tgemm {

// Programmatic dependent launch. Every kernel of the library is launched
// with the stream-serialisation attribute relaxed (launch_pdl), lets the
// next kernel in the stream launch as soon as all of its own blocks have
// started (pdl_launch_dependents, first thing in every kernel), and waits
// for the previous kernel in the stream -- its completion and the
// visibility of everything it wrote -- before its own first global-memory
// access (pdl_wait). A kernel's launch and its set-up (barrier init,
// tensor-memory allocation, tensor-map prefetch) thus overlap the previous
// kernel's last blocks, and nothing reads or writes memory early.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

#ifdef __CUDACC__
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
#endif

// Output rule of a product: C = alpha * acc + beta * C_old + bias[col]
// (C_old is not read when beta == 0; bias may be null). The default is the
// plain product C = acc.
struct Epilogue {
    float alpha = 1.0f;
    float beta = 0.0f;
    const float* bias = nullptr;
    bool simple() const { return alpha == 1.0f && beta == 0.0f && bias == nullptr; }
};

// Arguments of one product, already validated by the API layer.
// Raise kernel KERNEL's dynamic shared-memory limit to `bytes`, once per
// device (the attribute stays set for the life of the context), so that a
// launch does not pay for the call every time.
template <auto KERNEL>
cudaError_t set_smem_limit_once(int bytes) {
    static std::atomic<unsigned long long> done{0};    // bit d: set on device d
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
    return e;
}

struct GemmArgs {
    int M, N, K;
    const void* A; long lda;
    const void* B; long ldb;
    float* C;      long ldc;
    // Low parts of A and B for the split-TF32 form (same layouts as A, B).
    const void* A2 = nullptr;
    const void* B2 = nullptr;
    Epilogue ep = Epilogue();
    // Tensor paths: A's rows are only 4-byte aligned and are read by the
    // kernel's SIMT loader warps instead of TMA (a_esz: A's element size).
    bool a_loader = false;
    int a_esz = 0;
};

// ---- FP32 CUDA-core path (sgemm_f32.cu) ---------------------------------
int  f32_kernel_count();
const char* f32_kernel_name(int id);
// True if configuration `id` may read these operands (vector loaders need
// 16-byte aligned pointers and leading dimensions that are multiples of 4).
bool f32_kernel_accepts(int id, const GemmArgs& a);
// Pick a configuration for this shape and alignment.
int  f32_select(const GemmArgs& a, int num_sms);
// How configuration `id` covers this problem: tiles computed whole, and the
// tiles of a partial last wave split into K-pieces whose partial tiles need
// `scratch_bytes` of device scratch (0 when nothing is split).
struct F32Plan {
    int tiles_m, tiles_n, ktiles;
    int dp_tiles, split;
    size_t scratch_bytes;
};
F32Plan f32_plan(int id, const GemmArgs& a, int num_sms);
// Launch configuration `id` under plan `pl` (plus the split-K reduction when
// the plan splits); `scratch` holds pl.scratch_bytes. Returns a cudaError_t.
cudaError_t f32_launch(int id, const GemmArgs& a, const F32Plan& pl, float* scratch,
                       cudaStream_t s);

// ---- tcgen05 tensor-core path (gemm_tcgen05.cu) -------------------------
enum TcType { TC_TF32 = 1, TC_BF16 = 2, TC_TF32X3 = 3 };
// Tile shapes of the tensor-core kernels: 128 x 256 on one SM, 256 x 256 on
// an SM pair, 256 x 512 on an SM pair (two N = 256 MMAs per K step), and
// 128 x 128 on one SM for TF32 with B read as stored (K x N) and transposed
// in shared memory by the kernel (TC_ONE_SM_T), and 128 x 128 on one SM
// (TC_ONE_SM_N: more tiles for products with few rows).
enum TcShape { TC_ONE_SM = 0, TC_PAIR = 1, TC_PAIR_WIDE = 2, TC_ONE_SM_T = 3, TC_ONE_SM_N = 4 };
// The shape a product runs with: mode -1 = the shape a timing model expects
// to finish first, 0/1/2/4 = that TcShape (the split-TF32 form always takes
// TC_PAIR); mode 3 is taken as -1 (the caller picks TC_ONE_SM_T, which
// depends on how B is stored). streamk and tma_c as for tc_plan.
int tc_shape(int M, int N, int K, int in_type, int mode, int num_sms, int streamk,
             bool tma_c = true);
const char* tc_kernel_name(int in_type, int shape);
// Tiling of one tensor-core product: tiles of tile_rows x tile_cols over
// `slots` resident units (SMs, or SM pairs), computed whole in rounds. With
// sk_slots > 0 (stream-K), the tiles of a partial last round -- tiles
// [dp_tiles, tiles) -- are not computed whole: their K blocks are shared
// evenly by slots [0, sk_slots); a slot whose share ends a tile owns it and
// adds the partial tiles of the slots before it, which wait for nothing.
// scratch_bytes then holds sk_slots partial tiles (tc_partial_bytes) and one
// counter per tail tile; 0 without stream-K.
struct TcPlan {
    int tile_rows, tile_cols, tiles_m, tiles_n, kblocks;
    int slots, dp_tiles, sk_slots;
    int sk_split;        // the tail in the split form: equal shares, then a reduction kernel
    size_t scratch_bytes;
    double est_us;       // modelled duration, for choosing between shapes
};
size_t tc_partial_bytes(const TcPlan& pl);
// tma_c: the whole tiles can leave by TMA stores (C's base and rows 16-byte
// aligned, beta = 0); it changes only the modelled epilogue cost.
// streamk: -1 = a stream-K tail where the timing model prefers it (it needs
// scratch), 0 = never, S > 0 = a tail shared by S slots where possible.
TcPlan tc_plan(int M, int N, int K, int in_type, int shape, int num_sms, int streamk,
               bool tma_c = true);
// Launch the persistent tcgen05 kernel of TcShape `shape` under plan `pl`
// (made for the same shape); `scratch` holds pl.scratch_bytes (it may be
// null when that is 0). `encode_fn` is cuTensorMapEncodeTiled. With
// b_kmajor, a.B / a.ldb describe B transposed (N x K, K contiguous).
// TC_ONE_SM_T takes TC_TF32 with b_kmajor = 0 (B K x N, rows 16-byte
// aligned) and A read by TMA only.
cudaError_t tc_launch(const GemmArgs& a, int in_type, int b_kmajor, void* encode_fn,
                      unsigned long long wait_limit_ns, int debug_stall, int shape,
                      const TcPlan& pl, void* scratch, cudaStream_t s);
// Read and clear the tensor-core kernel's status word on the current device.
cudaError_t tc_read_and_clear_status(int* status, cudaStream_t s);
// Dense MMA rate probe: every SM (or SM pair) issues `iters` MMAs from
// resident shared memory; cycles[u] receives the SM clock cycles of unit u
// (-1 if its wait ran out) for the *units launched. `cycles` holds >= num_sms
// entries. tc_peak_flop_per_mma gives the FLOP of one of those MMAs (per
// unit).
cudaError_t tc_peak(int in_type, bool pair, long iters, int num_sms, unsigned long long wait_ns,
                    long long* cycles, int* units, cudaStream_t s);
double tc_peak_flop_per_mma(int in_type, bool pair);

// ---- tail balancing (sgemm_f32.cu) --------------------------------------
// Modelled cost (us) of computing `rem` tiles of tile_bytes in `split`
// K-pieces: the partial tiles' HBM traffic and the reduction launch.
double tail_split_cost_us(int rem, double tile_bytes, int split);
// Split of `tiles` work tiles over `slots` resident units: the first
// dp_tiles whole, the tiles of a partial last wave in `split` K-pieces of at
// least 4 K-blocks (of `ktiles`). `tile_us` is the time of one whole tile on
// one unit and `tile_bytes` the size of its FP32 partial; the split that
// saves the most time net of its scratch traffic is taken (split = 1: none).
void plan_tail_split(int tiles, int slots, int ktiles, double tile_us, double tile_bytes,
                     int& dp_tiles, int& split);

// ---- layout pre-pass (transpose_f32.cu) ---------------------------------
// Split-TF32 operands: hi = x rounded to TF32 (nearest), lo = (x - hi)
// rounded to TF32. split_rows writes hi/lo of a rows x cols matrix with
// leading dimension ld_out; transpose_split writes hi/lo of B transposed.
cudaError_t split_rows_tf32(const float* X, long ldx, float* hi, float* lo, long ld_out, int rows,
                            int cols, cudaStream_t s);
cudaError_t transpose_split_tf32(const float* B, long ldb, float* hi_t, float* lo_t, long ldt,
                                 int K, int N, cudaStream_t s);
// Bt[n][k] = B[k][n] for a K x N matrix B (ldb) into Bt (N x K, ldt >= K).
cudaError_t transpose_f32(const float* B, long ldb, float* Bt, long ldt, int K, int N,
                          cudaStream_t s);
// The same for 2-byte elements (bf16 bit patterns).
cudaError_t transpose_u16(const void* B, long ldb, void* Bt, long ldt, int K, int N,
                          cudaStream_t s);

// Copy a rows x cols matrix of `esz`-byte elements (2 or 4) from leading
// dimension ld_src to ld_dst (in elements).
cudaError_t repack_rows(const void* src, long ld_src, void* dst, long ld_dst, int rows, int cols,
                        int esz, cudaStream_t s);
// One such copy (rows or cols 0: none).
struct RepackJob {
    const void* src = nullptr;
    long ld_src = 0;
    void* dst = nullptr;
    long ld_dst = 0;
    int rows = 0, cols = 0;
};
// Two copies in one launch (A and B of one product).
cudaError_t repack_rows2(const RepackJob& a, const RepackJob& b, int esz, cudaStream_t s);

// ---- process-wide settings (api.cu) ---------------------------------------
// The bound on any single wait inside the tensor-core kernels, as last set
// by gemm_set_wait_limit_ns (default 2 s).
unsigned long long wait_limit_ns();

// ---- shared helper (sgemm_f32.cu) -----------------------------------------
// The K == 0 product: C = beta * C_old + bias (zeros for the default rule).
cudaError_t empty_product(float* C, long ldc, int M, int N, const Epilogue& ep, cudaStream_t s);

}  // namespace tgemm
