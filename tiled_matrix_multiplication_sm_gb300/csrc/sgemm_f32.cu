// Exact-FP32 dense product C = A x B on the CUDA cores of sm_103a.
//
// The method is the shared-memory tiling of "Tiled GEMM: Matrix
// Multiplication in CUDA", sections 2 and 4 (and "Tiling and Blocking for
// Reuse", "the tiled version"): one thread block owns one tile of C and
// walks the K dimension in phases; each phase copies a BM x BK tile of A and
// a BK x BN tile of B into shared memory, and every thread then accumulates
// its outputs from those on-chip copies. On top of that sit the refinements
// the pages list as the next steps:
//   * register blocking ("Tiling and Blocking for Reuse", "the next level:
//     register blocking"): each thread owns a TM x TN patch of C in registers
//     and reads 128-bit fragments of A and B from shared memory;
//   * asynchronous copies and a multi-stage ring ("Tiled GEMM ...",
//     section 8): cp.async moves global memory straight into shared memory,
//     STAGES-1 phases ahead of the math, so the load of phase t+1 overlaps
//     the arithmetic of phase t;
//   * ragged edges ("Tiled GEMM ...", section 7.1): loads past M, N or K are
//     zero-filled (cp.async with a short source size), stores past M or N
//     are skipped;
//   * bank-conflict-free fragment reads (section 7.2 of the same page): A is
//     kept row-major with a 4-float pad per row, so the four rows a warp
//     reads at once fall in four different bank groups, and each quarter-warp
//     reads one 128-byte run of B.
// The two barriers of the pages (after the load, before the overwrite) become
// one __syncthreads per phase: with a ring of STAGES buffers, the barrier at
// the top of phase t both publishes tile t and retires the buffer that the
// prefetch issued right after it overwrites.
//
// Within a thread every output accumulates its products in ascending k with
// FP32 fused multiply-adds.

#include "tgemm_internal.h"

#include <cstdint>

namespace tgemm {
namespace {

// ---------------------------------------------------------------- cp.async
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte copy; `src_bytes` (0, 4, 8, 12 or 16) are read, the rest is zero.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
                 :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// 4-byte copy; `src_bytes` is 0 (write a zero) or 4.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n"
                 :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" :: "n"(N) : "memory");
}

// ------------------------------------------------------------ configuration
template <int BM_, int BN_, int BK_, int WM_, int WN_, int STAGES_, int MIN_BLOCKS_>
struct Tile {
    static constexpr int BM = BM_, BN = BN_, BK = BK_;
    static constexpr int WM = WM_, WN = WN_;
    static constexpr int STAGES = STAGES_;
    static constexpr int MIN_BLOCKS = MIN_BLOCKS_;
    static constexpr int WARPS_M = BM / WM, WARPS_N = BN / WN;
    static constexpr int THREADS = 32 * WARPS_M * WARPS_N;
    // A warp is 4 rows x 8 columns of threads.
    static constexpr int TM = WM / 4;         // rows per thread (stride 4)
    static constexpr int TN = WN / 8;         // columns per thread
    static constexpr int NG = TN / 4;         // 4-wide column groups (stride 32)
    static constexpr int ALD = BK + 4;        // padded row of the A tile (floats)
    static constexpr int BLD = BN;            // row of the B tile (floats)
    static constexpr int A_STAGE = BM * ALD;  // floats
    static constexpr int B_STAGE = BK * BLD;
    static constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;
    static_assert(WM % 4 == 0 && WN % 32 == 0 && TN % 4 == 0, "warp tile shape");
    static_assert(BK % 4 == 0, "BK must be a multiple of 4");
    static_assert((BM * BK / 4) % THREADS == 0 && (BK * BN / 4) % THREADS == 0,
                  "vector loads must divide evenly over the threads");
    static_assert((BM * BK) % THREADS == 0 && (BK * BN) % THREADS == 0,
                  "scalar loads must divide evenly over the threads");
};

// Copy the A tile (rows m0.., columns k0..) into shared memory.
template <class T, bool VEC>
__device__ __forceinline__ void load_a(float* As, const float* __restrict__ A, long lda,
                                       int M, int K, int m0, int k0, int tid) {
    if constexpr (VEC) {
        constexpr int CPR = T::BK / 4;                 // 16-byte chunks per row
        constexpr int ITERS = T::BM * CPR / T::THREADS;
#pragma unroll
        for (int it = 0; it < ITERS; ++it) {
            const int c = tid + it * T::THREADS;
            const int m = c / CPR, kc = (c % CPR) * 4;
            const int gm = m0 + m, gk = k0 + kc;
            int bytes = 0;
            if (gm < M) {
                const int left = K - gk;
                bytes = left >= 4 ? 16 : (left > 0 ? left * 4 : 0);
            }
            const float* src = bytes ? A + (long)gm * lda + gk : A;
            cp_async_16(smem_u32(As + m * T::ALD + kc), src, bytes);
        }
    } else {
        constexpr int ITERS = T::BM * T::BK / T::THREADS;
#pragma unroll
        for (int it = 0; it < ITERS; ++it) {
            const int e = tid + it * T::THREADS;
            const int m = e / T::BK, k = e % T::BK;
            const int gm = m0 + m, gk = k0 + k;
            const bool ok = gm < M && gk < K;
            const float* src = ok ? A + (long)gm * lda + gk : A;
            cp_async_4(smem_u32(As + m * T::ALD + k), src, ok ? 4 : 0);
        }
    }
}

// Copy the B tile (rows k0.., columns n0..) into shared memory.
template <class T, bool VEC>
__device__ __forceinline__ void load_b(float* Bs, const float* __restrict__ B, long ldb,
                                       int N, int K, int k0, int n0, int tid) {
    if constexpr (VEC) {
        constexpr int CPR = T::BN / 4;
        constexpr int ITERS = T::BK * CPR / T::THREADS;
#pragma unroll
        for (int it = 0; it < ITERS; ++it) {
            const int c = tid + it * T::THREADS;
            const int k = c / CPR, nc = (c % CPR) * 4;
            const int gk = k0 + k, gn = n0 + nc;
            int bytes = 0;
            if (gk < K) {
                const int left = N - gn;
                bytes = left >= 4 ? 16 : (left > 0 ? left * 4 : 0);
            }
            const float* src = bytes ? B + (long)gk * ldb + gn : B;
            cp_async_16(smem_u32(Bs + k * T::BLD + nc), src, bytes);
        }
    } else {
        constexpr int ITERS = T::BK * T::BN / T::THREADS;
#pragma unroll
        for (int it = 0; it < ITERS; ++it) {
            const int e = tid + it * T::THREADS;
            const int k = e / T::BN, n = e % T::BN;
            const int gk = k0 + k, gn = n0 + n;
            const bool ok = gk < K && gn < N;
            const float* src = ok ? B + (long)gk * ldb + gn : B;
            cp_async_4(smem_u32(Bs + k * T::BLD + n), src, ok ? 4 : 0);
        }
    }
}

template <class T, bool VA, bool VB>
__global__ void __launch_bounds__(T::THREADS, T::MIN_BLOCKS)
sgemm_kernel(const float* __restrict__ A, long lda,
             const float* __restrict__ B, long ldb,
             float* __restrict__ C, long ldc,
             int M, int N, int K, int vec_c) {
    extern __shared__ __align__(16) float smem[];
    float* As = smem;                               // [STAGES][BM][ALD]
    float* Bs = smem + T::STAGES * T::A_STAGE;      // [STAGES][BK][BLD]

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int warp_m = warp / T::WARPS_N, warp_n = warp % T::WARPS_N;
    const int ty = lane >> 3, tx = lane & 7;

    // Tile raster: walk GROUP tile-rows at a time so that blocks running
    // together share panels of A and B in L2.
    constexpr int GROUP = 8;
    const int tiles_m = (M + T::BM - 1) / T::BM;
    const int tiles_n = (N + T::BN - 1) / T::BN;
    const int pid = blockIdx.x;
    const int per_group = GROUP * tiles_n;
    const int first_m = (pid / per_group) * GROUP;
    const int group_m = min(tiles_m - first_m, GROUP);
    const int tile_m = first_m + (pid % per_group) % group_m;
    const int tile_n = (pid % per_group) / group_m;
    const int m0 = tile_m * T::BM, n0 = tile_n * T::BN;

    const int wm0 = warp_m * T::WM, wn0 = warp_n * T::WN;

    float acc[T::TM][T::TN];
#pragma unroll
    for (int i = 0; i < T::TM; ++i)
#pragma unroll
        for (int j = 0; j < T::TN; ++j) acc[i][j] = 0.0f;

    const int ktiles = (K + T::BK - 1) / T::BK;

    // Prologue: put phases 0 .. STAGES-2 in flight.
#pragma unroll
    for (int s = 0; s < T::STAGES - 1; ++s) {
        if (s < ktiles) {
            load_a<T, VA>(As + s * T::A_STAGE, A, lda, M, K, m0, s * T::BK, tid);
            load_b<T, VB>(Bs + s * T::B_STAGE, B, ldb, N, K, s * T::BK, n0, tid);
        }
        cp_async_commit();
    }

    for (int kt = 0; kt < ktiles; ++kt) {
        // Phase kt's copies are done (for this thread) ...
        cp_async_wait<T::STAGES - 2>();
        // ... and for every thread; also, everyone has finished phase kt-1,
        // whose buffer the prefetch below reuses.
        __syncthreads();

        const int pf = kt + T::STAGES - 1;
        if (pf < ktiles) {
            const int ps = pf % T::STAGES;
            load_a<T, VA>(As + ps * T::A_STAGE, A, lda, M, K, m0, pf * T::BK, tid);
            load_b<T, VB>(Bs + ps * T::B_STAGE, B, ldb, N, K, pf * T::BK, n0, tid);
        }
        cp_async_commit();

        const int st = kt % T::STAGES;
        const float* as = As + st * T::A_STAGE + (wm0 + ty) * T::ALD;
        const float* bs = Bs + st * T::B_STAGE + wn0 + tx * 4;
#pragma unroll
        for (int k4 = 0; k4 < T::BK; k4 += 4) {
            float4 a[T::TM];
#pragma unroll
            for (int i = 0; i < T::TM; ++i)
                a[i] = *reinterpret_cast<const float4*>(as + (4 * i) * T::ALD + k4);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float4 b[T::NG];
#pragma unroll
                for (int g = 0; g < T::NG; ++g)
                    b[g] = *reinterpret_cast<const float4*>(bs + (k4 + kk) * T::BLD + g * 32);
#pragma unroll
                for (int i = 0; i < T::TM; ++i) {
                    const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
#pragma unroll
                    for (int g = 0; g < T::NG; ++g) {
                        acc[i][4 * g + 0] = fmaf(av, b[g].x, acc[i][4 * g + 0]);
                        acc[i][4 * g + 1] = fmaf(av, b[g].y, acc[i][4 * g + 1]);
                        acc[i][4 * g + 2] = fmaf(av, b[g].z, acc[i][4 * g + 2]);
                        acc[i][4 * g + 3] = fmaf(av, b[g].w, acc[i][4 * g + 3]);
                    }
                }
            }
        }
    }
    cp_async_wait<0>();

    // Epilogue: one store per output (section 4.8 of the second page),
    // 16-byte stores where C allows them, skipped past M and N.
#pragma unroll
    for (int i = 0; i < T::TM; ++i) {
        const int row = m0 + wm0 + ty + 4 * i;
        if (row >= M) continue;
        float* crow = C + (long)row * ldc;
#pragma unroll
        for (int g = 0; g < T::NG; ++g) {
            const int col = n0 + wn0 + g * 32 + tx * 4;
            if (vec_c && col + 3 < N) {
                *reinterpret_cast<float4*>(crow + col) =
                    make_float4(acc[i][4 * g], acc[i][4 * g + 1], acc[i][4 * g + 2], acc[i][4 * g + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (col + j < N) crow[col + j] = acc[i][4 * g + j];
            }
        }
    }
}

__global__ void zero_fill_kernel(float* __restrict__ C, long ldc, int M, int N) {
    const long total = (long)M * N;
    for (long e = blockIdx.x * (long)blockDim.x + threadIdx.x; e < total;
         e += (long)gridDim.x * blockDim.x) {
        const long r = e / N, c = e % N;
        C[r * ldc + c] = 0.0f;
    }
}

// ------------------------------------------------------------ the table
using Big = Tile<128, 128, 16, 32, 64, 4, 2>;    // 256 threads, 8x8 per thread
using Small = Tile<64, 64, 16, 32, 32, 4, 4>;    // 128 threads, 8x4 per thread

struct Entry {
    const char* name;
    bool va, vb;
    int bm, bn;
    cudaError_t (*launch)(const GemmArgs&, cudaStream_t);
};

template <class T, bool VA, bool VB>
cudaError_t launch_cfg(const GemmArgs& a, cudaStream_t s) {
    auto kern = sgemm_kernel<T, VA, VB>;
    static_assert(T::SMEM_BYTES <= 227 * 1024, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         T::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int tiles = ((a.M + T::BM - 1) / T::BM) * ((a.N + T::BN - 1) / T::BN);
    const bool vec_c = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) && (a.ldc % 4 == 0);
    kern<<<tiles, T::THREADS, T::SMEM_BYTES, s>>>(
        static_cast<const float*>(a.A), a.lda, static_cast<const float*>(a.B), a.ldb,
        a.C, a.ldc, a.M, a.N, a.K, vec_c ? 1 : 0);
    return cudaGetLastError();
}

const Entry kTable[] = {
    {"f32_128x128x16_s4_vecA_vecB", true, true, 128, 128, launch_cfg<Big, true, true>},
    {"f32_128x128x16_s4_vecA_b4", true, false, 128, 128, launch_cfg<Big, true, false>},
    {"f32_128x128x16_s4_a4_vecB", false, true, 128, 128, launch_cfg<Big, false, true>},
    {"f32_128x128x16_s4_a4_b4", false, false, 128, 128, launch_cfg<Big, false, false>},
    {"f32_64x64x16_s4_vecA_vecB", true, true, 64, 64, launch_cfg<Small, true, true>},
    {"f32_64x64x16_s4_vecA_b4", true, false, 64, 64, launch_cfg<Small, true, false>},
    {"f32_64x64x16_s4_a4_vecB", false, true, 64, 64, launch_cfg<Small, false, true>},
    {"f32_64x64x16_s4_a4_b4", false, false, 64, 64, launch_cfg<Small, false, false>},
};
constexpr int kTableSize = sizeof(kTable) / sizeof(kTable[0]);

bool vec_ok(const void* p, long ld) {
    return reinterpret_cast<uintptr_t>(p) % 16 == 0 && ld % 4 == 0;
}

}  // namespace

int f32_kernel_count() { return kTableSize; }

const char* f32_kernel_name(int id) {
    return (id >= 0 && id < kTableSize) ? kTable[id].name : "";
}

bool f32_kernel_accepts(int id, const GemmArgs& a) {
    if (id < 0 || id >= kTableSize) return false;
    if (kTable[id].va && !vec_ok(a.A, a.lda)) return false;
    if (kTable[id].vb && !vec_ok(a.B, a.ldb)) return false;
    return true;
}

int f32_select(const GemmArgs& a, int num_sms) {
    const bool va = vec_ok(a.A, a.lda), vb = vec_ok(a.B, a.ldb);
    const long big_tiles = (long)((a.M + 127) / 128) * ((a.N + 127) / 128);
    const int base = big_tiles >= num_sms ? 0 : 4;
    const int loader = (va ? 0 : 2) + (vb ? 0 : 1);
    return base + loader;
}

cudaError_t f32_launch(int id, const GemmArgs& a, cudaStream_t s) {
    return kTable[id].launch(a, s);
}

cudaError_t zero_fill(float* C, long ldc, int M, int N, cudaStream_t s) {
    const long total = (long)M * N;
    long blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    zero_fill_kernel<<<(int)blocks, 256, 0, s>>>(C, ldc, M, N);
    return cudaGetLastError();
}

}  // namespace tgemm
