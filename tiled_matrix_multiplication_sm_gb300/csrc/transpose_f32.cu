// Out-of-place transpose of an FP32 matrix: Bt[n][k] = B[k][n].
//
// Storage a path's kernel does not read directly is rewritten here: A (or,
// on the FP32 path, B) stored transposed by gemm_ex, the split form's B
// (its high and low TF32 parts, read K-major), and the B that the
// allocation-free TF32 entry point reads K-major when B's rows are not
// 16-byte aligned.
//
// Both kernels here are pure data movement, bound by HBM bandwidth. The
// transpose reads every element once and writes it once
// (8 K N bytes); a 64 x 64 tile goes through shared memory so that
// both the reads (along a row of B) and the writes (along a row of Bt) are
// coalesced; the tile row is padded by one float so that reading it by
// columns hits 32 different banks -- the padding of "Tiled GEMM: Matrix
// Multiplication in CUDA", section 7.2, which the page recommends for
// exactly this case of transposed tile accesses.

#include "tgemm_internal.h"

#include <cstdint>

namespace tgemm {
namespace {

constexpr int TT = 64;          // tile edge
constexpr int TROWS = 4;        // thread rows: 64 x 4 = 256 threads

template <typename T>
__global__ void __launch_bounds__(TT * TROWS)
transpose_kernel(const T* __restrict__ B, long ldb, T* __restrict__ Bt, long ldt,
                 int K, int N) {
    pdl_launch_dependents();    // the next kernel may launch now
    pdl_wait();                 // the previous kernel's writes are visible
    __shared__ T tile[TT][TT + 1];
    const int tx = threadIdx.x % TT, ty = threadIdx.x / TT;
    const int n0 = blockIdx.x * TT, k0 = blockIdx.y * TT;
#pragma unroll
    for (int r = ty; r < TT; r += TROWS) {
        const int k = k0 + r, n = n0 + tx;
        tile[r][tx] = (k < K && n < N) ? B[(long)k * ldb + n] : T(0);
    }
    __syncthreads();
#pragma unroll
    for (int r = ty; r < TT; r += TROWS) {
        const int n = n0 + r, k = k0 + tx;
        if (n < N && k < K) Bt[(long)n * ldt + k] = tile[tx][r];
    }
}

// Row-by-row copy of a rows x cols matrix of `esz`-byte elements from
// leading dimension ld_src to ld_dst (both in elements). Used to give the
// tensor-memory copies rows that start on 16-byte boundaries.
// Each block copies REPACK_ROWS rows of one REPACK_COLS-wide column chunk;
// every thread issues all of its loads (REPACK_ROWS rows x 4 columns, 256
// apart) before its stores, so that 8 loads per thread are in flight. (With
// 4 rows copied one after the other, 3000 x 1537 floats moved at 3.6 TB/s.)
// One launch may copy two matrices (A and B of one product): blocks
// [0, blocks_a) copy the first, the rest the second, so the two copies share
// one launch and one tail instead of two.
constexpr int REPACK_ROWS = 2;
constexpr int REPACK_COLS = 1024;

template <typename T>
__global__ void __launch_bounds__(256)
repack_kernel(const RepackJob ja, const RepackJob jb, long blocks_a) {
    pdl_launch_dependents();    // the next kernel may launch now
    pdl_wait();                 // the previous kernel's writes are visible
    const bool first = (long)blockIdx.x < blocks_a;
    const RepackJob& j = first ? ja : jb;
    const long bid = first ? (long)blockIdx.x : (long)blockIdx.x - blocks_a;
    const long chunks = ((long)j.cols + REPACK_COLS - 1) / REPACK_COLS;
    const int rows = j.rows, cols = j.cols;
    const long ld_src = j.ld_src, ld_dst = j.ld_dst;
    const T* __restrict__ src = static_cast<const T*>(j.src);
    T* __restrict__ dst = static_cast<T*>(j.dst);
    const int r0 = (int)(bid / chunks) * REPACK_ROWS;
    const int c = (int)(bid % chunks) * REPACK_COLS + threadIdx.x;
    T v[REPACK_ROWS][4];
#pragma unroll
    for (int i = 0; i < REPACK_ROWS; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (r0 + i < rows && c + 256 * j < cols)
                v[i][j] = src[(long)(r0 + i) * ld_src + c + 256 * j];
#pragma unroll
    for (int i = 0; i < REPACK_ROWS; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (r0 + i < rows && c + 256 * j < cols)
                dst[(long)(r0 + i) * ld_dst + c + 256 * j] = v[i][j];
}

// x rounded to the TF32 format (10 explicit mantissa bits), to nearest with
// ties away from zero; the low 13 bits of the result are zero.
__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// hi = tf32(x), lo = tf32(x - hi). x - hi is exact in FP32: hi is within a
// factor of two of x, so the difference needs no rounding (Sterbenz).
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
    hi = tf32_rna(x);
    lo = tf32_rna(x - hi);
}

__global__ void __launch_bounds__(256)
split_rows_kernel(const float* __restrict__ X, long ldx, float* __restrict__ hi,
                  float* __restrict__ lo, long ld_out, int rows, int cols) {
    pdl_launch_dependents();    // the next kernel may launch now
    pdl_wait();                 // the previous kernel's writes are visible
    for (int r = blockIdx.y; r < rows; r += gridDim.y) {
        const float* s = X + (long)r * ldx;
        for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < cols; c += gridDim.x * blockDim.x) {
            float h, l;
            split_tf32(s[c], h, l);
            hi[(long)r * ld_out + c] = h;
            lo[(long)r * ld_out + c] = l;
        }
    }
}

// The same on 16-byte vectors (X's rows and the outputs' rows 16-byte
// aligned): a flat grid-stride loop over (row, vector of four columns), then
// the cols % 4 columns past the last whole vector one by one.
__global__ void __launch_bounds__(256)
split_rows_vec_kernel(const float* __restrict__ X, long ldx, float* __restrict__ hi,
                      float* __restrict__ lo, long ld_out, int rows, int cols) {
    pdl_launch_dependents();    // the next kernel may launch now
    pdl_wait();                 // the previous kernel's writes are visible
    const int vecs = cols / 4;
    const long total = (long)rows * vecs;
    for (long u = blockIdx.x * (long)blockDim.x + threadIdx.x; u < total;
         u += (long)gridDim.x * blockDim.x) {
        const int r = (int)(u / vecs), c = (int)(u % vecs) * 4;
        const float4 x = *reinterpret_cast<const float4*>(X + (long)r * ldx + c);
        float4 h, l;
        split_tf32(x.x, h.x, l.x);
        split_tf32(x.y, h.y, l.y);
        split_tf32(x.z, h.z, l.z);
        split_tf32(x.w, h.w, l.w);
        *reinterpret_cast<float4*>(hi + (long)r * ld_out + c) = h;
        *reinterpret_cast<float4*>(lo + (long)r * ld_out + c) = l;
    }
    const int tail = cols % 4;
    if (tail) {
        for (long u = blockIdx.x * (long)blockDim.x + threadIdx.x; u < (long)rows * tail;
             u += (long)gridDim.x * blockDim.x) {
            const int r = (int)(u / tail), c = vecs * 4 + (int)(u % tail);
            float h, l;
            split_tf32(X[(long)r * ldx + c], h, l);
            hi[(long)r * ld_out + c] = h;
            lo[(long)r * ld_out + c] = l;
        }
    }
}

// Transpose of B (K x N) into hi/lo parts of Bt (N x K), through a padded
// shared-memory tile as in transpose_kernel.
__global__ void __launch_bounds__(TT * TROWS)
transpose_split_kernel(const float* __restrict__ B, long ldb, float* __restrict__ hi_t,
                       float* __restrict__ lo_t, long ldt, int K, int N) {
    pdl_launch_dependents();    // the next kernel may launch now
    pdl_wait();                 // the previous kernel's writes are visible
    __shared__ float tile[TT][TT + 1];
    const int tx = threadIdx.x % TT, ty = threadIdx.x / TT;
    const int n0 = blockIdx.x * TT, k0 = blockIdx.y * TT;
#pragma unroll
    for (int r = ty; r < TT; r += TROWS) {
        const int k = k0 + r, n = n0 + tx;
        tile[r][tx] = (k < K && n < N) ? B[(long)k * ldb + n] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int r = ty; r < TT; r += TROWS) {
        const int n = n0 + r, k = k0 + tx;
        if (n < N && k < K) {
            float h, l;
            split_tf32(tile[tx][r], h, l);
            hi_t[(long)n * ldt + k] = h;
            lo_t[(long)n * ldt + k] = l;
        }
    }
}

}  // namespace

cudaError_t split_rows_tf32(const float* X, long ldx, float* hi, float* lo, long ld_out, int rows,
                            int cols, cudaStream_t s) {
    auto al16 = [](const void* q) { return reinterpret_cast<uintptr_t>(q) % 16 == 0; };
    if (al16(X) && al16(hi) && al16(lo) && ldx % 4 == 0 && ld_out % 4 == 0 && cols >= 4) {
        // 16-byte vectors: up to 4 waves of 8 blocks of 256 threads per SM.
        const long work = (long)rows * (cols / 4);
        long blocks = (work + 255) / 256;
        if (blocks > 152L * 8 * 4) blocks = 152L * 8 * 4;
        if (blocks < 1) blocks = 1;
        return launch_pdl(split_rows_vec_kernel, dim3((int)blocks), dim3(256), 0, s, X, ldx, hi, lo,
                          ld_out, rows, cols);
    }
    int gx = (cols + 255) / 256;
    if (gx > 64) gx = 64;
    if (gx < 1) gx = 1;
    int gy = rows < 16384 ? rows : 16384;
    if (gy < 1) gy = 1;
    return launch_pdl(split_rows_kernel, dim3(gx, gy), dim3(256), 0, s, X, ldx, hi, lo, ld_out, rows,
                      cols);
}

cudaError_t transpose_split_tf32(const float* B, long ldb, float* hi_t, float* lo_t, long ldt,
                                 int K, int N, cudaStream_t s) {
    dim3 grid((N + TT - 1) / TT, (K + TT - 1) / TT);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    return launch_pdl(transpose_split_kernel, grid, dim3(TT * TROWS), 0, s, B, ldb, hi_t, lo_t, ldt, K,
                      N);
}

namespace {
// Blocks of one copy: REPACK_ROWS rows by REPACK_COLS columns each.
long repack_blocks(const RepackJob& j) {
    if (j.rows <= 0 || j.cols <= 0) return 0;
    return ((long)j.rows + REPACK_ROWS - 1) / REPACK_ROWS *
           (((long)j.cols + REPACK_COLS - 1) / REPACK_COLS);
}
}  // namespace

cudaError_t repack_rows2(const RepackJob& a, const RepackJob& b, int esz, cudaStream_t s) {
    // Consecutive threads copy consecutive columns (coalesced).
    const long na = repack_blocks(a), nb = repack_blocks(b);
    if (na + nb == 0) return cudaSuccess;
    if (na + nb > 2147483647L) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)(na + nb));
    if (esz == 2) return launch_pdl(repack_kernel<unsigned short>, grid, dim3(256), 0, s, a, b, na);
    return launch_pdl(repack_kernel<float>, grid, dim3(256), 0, s, a, b, na);
}

cudaError_t repack_rows(const void* src, long ld_src, void* dst, long ld_dst, int rows, int cols,
                        int esz, cudaStream_t s) {
    return repack_rows2(RepackJob{src, ld_src, dst, ld_dst, rows, cols}, RepackJob{}, esz, s);
}

cudaError_t transpose_f32(const float* B, long ldb, float* Bt, long ldt, int K, int N,
                          cudaStream_t s) {
    dim3 grid((N + TT - 1) / TT, (K + TT - 1) / TT);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    return launch_pdl(transpose_kernel<float>, grid, dim3(TT * TROWS), 0, s, B, ldb, Bt, ldt, K, N);
}

cudaError_t transpose_u16(const void* B, long ldb, void* Bt, long ldt, int K, int N,
                          cudaStream_t s) {
    dim3 grid((N + TT - 1) / TT, (K + TT - 1) / TT);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    return launch_pdl(transpose_kernel<unsigned short>, grid, dim3(TT * TROWS), 0, s,
                      static_cast<const unsigned short*>(B), ldb, static_cast<unsigned short*>(Bt), ldt,
                      K, N);
}

}  // namespace tgemm
