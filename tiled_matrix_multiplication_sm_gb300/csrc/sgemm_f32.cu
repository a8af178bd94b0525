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
//     register blocking"): each thread owns an 8 x 16 (default) patch of C in
//     registers and reads 128-bit fragments of A and B from shared memory;
//   * asynchronous copies and a multi-stage ring ("Tiled GEMM ...",
//     section 8): cp.async moves global memory straight into shared memory,
//     STAGES-1 phases ahead of the math, so the load of phase t+1 overlaps
//     the arithmetic of phase t;
//   * ragged edges ("Tiled GEMM ...", section 7.1): loads past M, N or K are
//     zero-filled (cp.async with a short source size), stores past M or N
//     are skipped;
//   * bank-conflict-free fragment reads (section 7.2 of the same page): A is
//     kept row-major with a 4-float pad per row, a thread's rows are 4 apart,
//     so the four rows a warp reads at once fall in four different bank
//     groups, and each quarter-warp reads one 128-byte run of B.
// The two barriers of the pages (after the load, before the overwrite) become
// one __syncthreads per phase: with a ring of STAGES buffers, the barrier at
// the top of phase t both publishes tile t and retires the buffer that the
// prefetch issued right after it overwrites.
//
// The packed variants issue Blackwell's two-wide FP32 FMA (__ffma2_rn: two
// independent round-to-nearest fused multiply-adds per instruction) on pairs
// of adjacent output columns; each lane computes exactly what fmaf computes,
// so packed and scalar kernels give identical bits.
//
// Tail balancing: no output of C depends on another ("Tiled Matrix
// Multiplication in CUDA", section 1), so neither do tiles, and when the
// tile count is not a multiple of the resident blocks, the tiles of the last
// partial wave are split along K into `split` pieces. Each piece writes its partial
// tile to scratch and splitk_reduce adds the pieces in a fixed order; the
// result is deterministic.
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
template <int BM_, int BN_, int BK_, int WM_, int WN_, int STAGES_, int MIN_BLOCKS_, bool PACKED_>
struct Tile {
    static constexpr int BM = BM_, BN = BN_, BK = BK_;
    static constexpr int WM = WM_, WN = WN_;
    static constexpr int STAGES = STAGES_;
    static constexpr int MIN_BLOCKS = MIN_BLOCKS_;
    static constexpr bool PACKED = PACKED_;
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

struct F32Params {
    const float* A;
    long lda;
    const float* B;
    long ldb;
    float* C;
    long ldc;
    int M, N, K;
    int tiles_m, tiles_n;
    int ktiles;          // ceil(K / BK)
    int dp_tiles;        // tiles [0, dp_tiles) are computed whole
    int split;           // the others in `split` K-pieces each
    float* partials;     // (tiles - dp_tiles) * split partial tiles of BM x BN
    int vec_c;           // C rows may take 16-byte stores
    // Output rule C = alpha * acc + beta * C_old + bias[col]; ep_simple when
    // it is the plain product (alpha 1, beta 0, no bias).
    float alpha, beta;
    const float* bias;
    int ep_simple;
};

// One output under the rule (C_old read only when beta != 0).
__device__ __forceinline__ float apply_epilogue(float acc, const F32Params& p, const float* c_old,
                                                int col) {
    float v = p.alpha * acc;
    if (p.beta != 0.0f) v = fmaf(p.beta, *c_old, v);
    if (p.bias != nullptr) v += p.bias[col];
    return v;
}

constexpr int GROUP_M = 8;

// Grouped raster: GROUP_M tile-rows at a time, so that blocks running
// together share panels of A and B in L2.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int& tm, int& tn) {
    const int per_group = GROUP_M * tiles_n;
    const int first_m = (t / per_group) * GROUP_M;
    const int gm = min(tiles_m - first_m, GROUP_M);
    tm = first_m + (t % per_group) % gm;
    tn = (t % per_group) / gm;
}

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

__device__ __forceinline__ float pick(const float4& v, int kk) {
    return kk == 0 ? v.x : kk == 1 ? v.y : kk == 2 ? v.z : v.w;
}

// Register accumulators of one thread: TM rows x TN columns, stored as
// pairs of adjacent columns (v[i][p] holds columns 2p and 2p+1 of row i), the
// operand shape of the two-wide FMA.
template <class T>
struct Acc {
    float2 v[T::TM][T::TN / 2];
};

// One BK-deep phase of outer products from shared memory.
template <class T>
__device__ __forceinline__ void mma_phase(Acc<T>& acc, const float* as, const float* bs) {
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
            if constexpr (T::PACKED) {
                // (a, a) pairs of this k for all rows first, then the column
                // pairs one by one, each multiplied into every row: each run
                // of TM two-wide FMAs shares its B pair. (Row by row instead,
                // with each row's pair built where it is used, measured
                // 57.4 against 58.1 TFLOP/s on 4096^3.)
                float2 a2[T::TM];
#pragma unroll
                for (int i = 0; i < T::TM; ++i) {
                    const float av = pick(a[i], kk);
                    a2[i] = make_float2(av, av);
                }
#pragma unroll
                for (int h = 0; h < T::TN / 2; ++h) {
                    const float4& bg = b[h / 2];
                    const float2 bp = (h % 2) ? make_float2(bg.z, bg.w) : make_float2(bg.x, bg.y);
#pragma unroll
                    for (int i = 0; i < T::TM; ++i) acc.v[i][h] = __ffma2_rn(a2[i], bp, acc.v[i][h]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < T::TM; ++i) {
                    const float av = pick(a[i], kk);
#pragma unroll
                    for (int g = 0; g < T::NG; ++g) {
                        acc.v[i][2 * g].x = fmaf(av, b[g].x, acc.v[i][2 * g].x);
                        acc.v[i][2 * g].y = fmaf(av, b[g].y, acc.v[i][2 * g].y);
                        acc.v[i][2 * g + 1].x = fmaf(av, b[g].z, acc.v[i][2 * g + 1].x);
                        acc.v[i][2 * g + 1].y = fmaf(av, b[g].w, acc.v[i][2 * g + 1].y);
                    }
                }
            }
        }
    }
}

template <class T, bool VA, bool VB>
__global__ void __launch_bounds__(T::THREADS, T::MIN_BLOCKS)
sgemm_kernel(const F32Params p) {
    pdl_launch_dependents();    // the next kernel may launch now
    pdl_wait();                 // the previous kernel's writes are visible
    extern __shared__ __align__(16) float smem[];
    float* As = smem;                               // [STAGES][BM][ALD]
    float* Bs = smem + T::STAGES * T::A_STAGE;      // [STAGES][BK][BLD]

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int warp_m = warp / T::WARPS_N, warp_n = warp % T::WARPS_N;
    const int ty = lane >> 3, tx = lane & 7;

    // Work item: a whole tile, or one K-piece of a tile of the last wave.
    int tile, kt_begin, kt_end;
    long piece = -1;
    if ((int)blockIdx.x < p.dp_tiles) {
        tile = blockIdx.x;
        kt_begin = 0;
        kt_end = p.ktiles;
    } else {
        piece = (long)blockIdx.x - p.dp_tiles;
        const int j = (int)(piece % p.split);
        tile = p.dp_tiles + (int)(piece / p.split);
        kt_begin = (int)((long)j * p.ktiles / p.split);
        kt_end = (int)((long)(j + 1) * p.ktiles / p.split);
    }
    int tile_m, tile_n;
    tile_coords(tile, p.tiles_m, p.tiles_n, tile_m, tile_n);
    const int m0 = tile_m * T::BM, n0 = tile_n * T::BN;
    const int wm0 = warp_m * T::WM, wn0 = warp_n * T::WN;
    const float* __restrict__ A = p.A;
    const float* __restrict__ B = p.B;
    const int M = p.M, N = p.N, K = p.K;

    Acc<T> acc;
#pragma unroll
    for (int i = 0; i < T::TM; ++i)
#pragma unroll
        for (int j = 0; j < T::TN / 2; ++j) acc.v[i][j] = make_float2(0.0f, 0.0f);

    const int nk = kt_end - kt_begin;

    // Prologue: put phases 0 .. STAGES-2 of this work item in flight.
#pragma unroll
    for (int s = 0; s < T::STAGES - 1; ++s) {
        if (s < nk) {
            const int k0 = (kt_begin + s) * T::BK;
            load_a<T, VA>(As + s * T::A_STAGE, A, p.lda, M, K, m0, k0, tid);
            load_b<T, VB>(Bs + s * T::B_STAGE, B, p.ldb, N, K, k0, n0, tid);
        }
        cp_async_commit();
    }

    for (int kt = 0; kt < nk; ++kt) {
        // Phase kt's copies are done (for this thread) ...
        cp_async_wait<T::STAGES - 2>();
        // ... and for every thread; also, everyone has finished phase kt-1,
        // whose buffer the prefetch below reuses.
        __syncthreads();

        const int pf = kt + T::STAGES - 1;
        if (pf < nk) {
            const int ps = pf % T::STAGES;
            const int k0 = (kt_begin + pf) * T::BK;
            load_a<T, VA>(As + ps * T::A_STAGE, A, p.lda, M, K, m0, k0, tid);
            load_b<T, VB>(Bs + ps * T::B_STAGE, B, p.ldb, N, K, k0, n0, tid);
        }
        cp_async_commit();

        const int st = kt % T::STAGES;
        mma_phase<T>(acc, As + st * T::A_STAGE + (wm0 + ty) * T::ALD,
                     Bs + st * T::B_STAGE + wn0 + tx * 4);
    }
    cp_async_wait<0>();

    if (piece < 0) {
        // Epilogue: one store per output (section 4.8 of the second page),
        // 16-byte stores where C allows them, skipped past M and N.
#pragma unroll
        for (int i = 0; i < T::TM; ++i) {
            const int row = m0 + wm0 + ty + 4 * i;
            if (row >= M) continue;
            float* crow = p.C + (long)row * p.ldc;
#pragma unroll
            for (int g = 0; g < T::NG; ++g) {
                const int col = n0 + wn0 + g * 32 + tx * 4;
                float4 v = make_float4(acc.v[i][2 * g].x, acc.v[i][2 * g].y,
                                       acc.v[i][2 * g + 1].x, acc.v[i][2 * g + 1].y);
                if (p.vec_c && col + 3 < N) {
                    if (!p.ep_simple) {
                        v.x = apply_epilogue(v.x, p, crow + col, col);
                        v.y = apply_epilogue(v.y, p, crow + col + 1, col + 1);
                        v.z = apply_epilogue(v.z, p, crow + col + 2, col + 2);
                        v.w = apply_epilogue(v.w, p, crow + col + 3, col + 3);
                    }
                    *reinterpret_cast<float4*>(crow + col) = v;
                } else {
                    const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (col + j < N)
                            crow[col + j] = p.ep_simple ? e[j]
                                                        : apply_epilogue(e[j], p, crow + col + j,
                                                                         col + j);
                }
            }
        }
    } else {
        // A K-piece: the whole BM x BN partial tile goes to scratch.
        float* part = p.partials + piece * (long)(T::BM * T::BN);
#pragma unroll
        for (int i = 0; i < T::TM; ++i) {
            float* prow = part + (long)(wm0 + ty + 4 * i) * T::BN;
#pragma unroll
            for (int g = 0; g < T::NG; ++g)
                *reinterpret_cast<float4*>(prow + wn0 + g * 32 + tx * 4) =
                    make_float4(acc.v[i][2 * g].x, acc.v[i][2 * g].y, acc.v[i][2 * g + 1].x,
                                acc.v[i][2 * g + 1].y);
        }
    }
}

// Sum the K-pieces of every split tile, piece 0 first, and store to C.
template <class T>
__global__ void __launch_bounds__(256)
splitk_reduce(const F32Params p) {
    pdl_launch_dependents();    // the next kernel may launch now
    pdl_wait();                 // the previous kernel's writes are visible
    constexpr int Q = T::BN / 4;                       // float4 per tile row
    const long per_tile = (long)T::BM * Q;
    const long total = (long)(p.tiles_m * p.tiles_n - p.dp_tiles) * per_tile;
    for (long u = blockIdx.x * (long)blockDim.x + threadIdx.x; u < total;
         u += (long)gridDim.x * blockDim.x) {
        const int r = (int)(u / per_tile);
        const int e = (int)(u % per_tile);
        const int row = e / Q, c4 = (e % Q) * 4;
        int tm, tn;
        tile_coords(p.dp_tiles + r, p.tiles_m, p.tiles_n, tm, tn);
        const int grow = tm * T::BM + row, gcol = tn * T::BN + c4;
        if (grow >= p.M || gcol >= p.N) continue;
        const float* src = p.partials + (long)r * p.split * (T::BM * T::BN) + row * T::BN + c4;
        constexpr long kPiece = (long)T::BM * T::BN;
        // Pieces in order; four loads in flight before their adds.
        float4 s = *reinterpret_cast<const float4*>(src);
        for (int j = 1; j < p.split; j += 4) {
            float4 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (j + q < p.split) v[q] = *reinterpret_cast<const float4*>(src + (j + q) * kPiece);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (j + q < p.split) {
                    s.x += v[q].x;
                    s.y += v[q].y;
                    s.z += v[q].z;
                    s.w += v[q].w;
                }
        }
        float* dst = p.C + (long)grow * p.ldc + gcol;
        float v[4] = {s.x, s.y, s.z, s.w};
        if (!p.ep_simple)
            for (int j = 0; j < 4 && gcol + j < p.N; ++j)
                v[j] = apply_epilogue(v[j], p, dst + j, gcol + j);
        if (p.vec_c && gcol + 3 < p.N) {
            *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
            for (int j = 0; j < 4 && gcol + j < p.N; ++j) dst[j] = v[j];
        }
    }
}

// C = beta * C_old + bias[col] (the product of an empty sum is zero).
__global__ void __launch_bounds__(256)
empty_product_kernel(float* __restrict__ C, long ldc, int M, int N, float beta,
                     const float* __restrict__ bias) {
    pdl_launch_dependents();    // the next kernel may launch now
    pdl_wait();                 // the previous kernel's writes are visible
    for (int r = blockIdx.y; r < M; r += gridDim.y) {
        float* row = C + (long)r * ldc;
        for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < N; c += gridDim.x * blockDim.x) {
            float v = beta != 0.0f ? beta * row[c] : 0.0f;
            if (bias != nullptr) v += bias[c];
            row[c] = v;
        }
    }
}

// ------------------------------------------------------------ the table
// Default: 128 x 256 block tile, 8 warps of 32 x 128, 8 x 16 outputs per
// thread in column pairs (two-wide FMA), BK = 32, 3 stages, one block per SM.
using Wide32P1 = Tile<128, 256, 32, 32, 128, 3, 1, true>;
// Alternatives kept for tile selection by measurement and for tests.
using Wide16P1 = Tile<128, 256, 16, 32, 128, 4, 1, true>;
using Big32P1 = Tile<128, 128, 32, 32, 64, 3, 1, true>;
using Big16P = Tile<128, 128, 16, 32, 64, 4, 2, true>;
using Big16 = Tile<128, 128, 16, 32, 64, 4, 2, false>;   // scalar FFMA, 8 x 8 per thread
using Small = Tile<64, 64, 16, 32, 32, 4, 4, false>;     // 128 threads, 8 x 4 per thread
// Few rows (M small, the product bound by reading B): 32 or 16-row tiles so
// that few FMAs are spent on rows past M, two blocks of 128 threads per SM.
using Skinny32 = Tile<32, 256, 32, 32, 64, 3, 2, true>;   // 8 x 8 outputs per thread
using Skinny16 = Tile<16, 256, 32, 16, 64, 3, 2, true>;   // 4 x 8 outputs per thread

struct Entry {
    const char* name;
    bool va, vb;
    int bm, bn, bk, min_blocks;
    cudaError_t (*launch)(const F32Params&, int blocks, cudaStream_t);
    cudaError_t (*reduce)(const F32Params&, cudaStream_t);
};

template <class T, bool VA, bool VB>
cudaError_t launch_cfg(const F32Params& p, int blocks, cudaStream_t s) {
    auto kern = sgemm_kernel<T, VA, VB>;
    static_assert(T::SMEM_BYTES <= 227 * 1024, "shared memory budget");
    cudaError_t e = set_smem_limit_once<sgemm_kernel<T, VA, VB>>(T::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(blocks), dim3(T::THREADS), T::SMEM_BYTES, s, p);
}

template <class T>
cudaError_t reduce_cfg(const F32Params& p, cudaStream_t s) {
    const long units = (long)(p.tiles_m * p.tiles_n - p.dp_tiles) * T::BM * (T::BN / 4);
    long blocks = (units + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    return launch_pdl(splitk_reduce<T>, dim3((int)blocks), dim3(256), 0, s, p);
}

#define TGEMM_ENTRY(name, T, VA, VB)                                                       \
    {name, VA, VB, T::BM, T::BN, T::BK, T::MIN_BLOCKS, launch_cfg<T, VA, VB>, reduce_cfg<T>}

const Entry kTable[] = {
    TGEMM_ENTRY("f32_128x256x32_s3_ffma2_vecA_vecB", Wide32P1, true, true),
    TGEMM_ENTRY("f32_128x256x32_s3_ffma2_vecA_b4", Wide32P1, true, false),
    TGEMM_ENTRY("f32_128x256x32_s3_ffma2_a4_vecB", Wide32P1, false, true),
    TGEMM_ENTRY("f32_128x256x32_s3_ffma2_a4_b4", Wide32P1, false, false),
    TGEMM_ENTRY("f32_128x256x16_s4_ffma2_vecA_vecB", Wide16P1, true, true),
    TGEMM_ENTRY("f32_128x128x32_s3_ffma2_1blk_vecA_vecB", Big32P1, true, true),
    TGEMM_ENTRY("f32_128x128x16_s4_ffma2_2blk_vecA_vecB", Big16P, true, true),
    TGEMM_ENTRY("f32_128x128x16_s4_ffma_vecA_vecB", Big16, true, true),
    TGEMM_ENTRY("f32_128x128x16_s4_ffma_a4_b4", Big16, false, false),
    TGEMM_ENTRY("f32_64x64x16_s4_ffma_vecA_vecB", Small, true, true),
    TGEMM_ENTRY("f32_64x64x16_s4_ffma_a4_b4", Small, false, false),
    TGEMM_ENTRY("f32_32x256x32_s3_ffma2_2blk_vecA_vecB", Skinny32, true, true),
    TGEMM_ENTRY("f32_16x256x32_s3_ffma2_2blk_vecA_vecB", Skinny16, true, true),
};
constexpr int kBig32 = 5;
constexpr int kSmall = 9;
constexpr int kSkinny32 = 11;
constexpr int kSkinny16 = 12;
constexpr int kTableSize = sizeof(kTable) / sizeof(kTable[0]);
static_assert(kSkinny32 < kTableSize && kSkinny16 < kTableSize, "skinny entries in the table");

bool vec_ok(const void* p, long ld) {
    return reinterpret_cast<uintptr_t>(p) % 16 == 0 && ld % 4 == 0;
}

}  // namespace

// Work split of one launch: dp_tiles whole tiles, the rest in `split`
// K-pieces each. `slots` is the number of work units resident at once. A
// split is taken only when the time it saves on the partial last wave beats
// what it costs: each piece writes a partial tile and the reduction reads it
// back (plus one more launch).
double tail_split_cost_us(int rem, double tile_bytes, int split) {
    const double hbm_bytes_per_us = 6.5e6;        // a little under the measured copy rate
    const double launch_us = 5.0;                 // the reduction kernel
    // Each piece writes a partial tile, the reduction reads them all and
    // writes the tile.
    return launch_us + rem * tile_bytes * (2.0 * split + 1.0) / hbm_bytes_per_us;
}

void plan_tail_split(int tiles, int slots, int ktiles, double tile_us, double tile_bytes,
                     int& dp_tiles, int& split) {
    dp_tiles = tiles;
    split = 1;
    const int rem = tiles % slots;
    if (rem == 0) return;
    double best_net = 0.0;
    int best_s = 1;
    for (int s = 2; s <= 16; ++s) {
        if (ktiles / s < 4) break;                 // pieces of at least 4 phases
        // Tail in units of one whole-tile time: ceil(rem*s/slots) rounds of 1/s.
        const double tail = (double)((rem * s + slots - 1) / slots) / s;
        const double gain = (1.0 - tail) * tile_us;
        const double cost = tail_split_cost_us(rem, tile_bytes, s);
        if (gain - cost > best_net) {
            best_net = gain - cost;
            best_s = s;
        }
    }
    if (best_s > 1) {
        dp_tiles = tiles - rem;
        split = best_s;
    }
}

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
    if (va && vb && a.M > 0) {
        // Few rows: the 128-row tile spends its FMAs on rows past M. Measured
        // (N 4096 and 14336, K 4096): 16-row tiles fastest up to M = 16,
        // 32-row tiles up to 96 rows, and beyond that whenever the 128-row
        // tiles would pad M by 15 % more (the 32-row tile is ~12 % slower per
        // useful row on full tiles).
        if (a.M <= 16) return kSkinny16;
        const long wide_rows = ((long)a.M + 127) / 128 * 128;
        const long skinny_rows = ((long)a.M + 31) / 32 * 32;
        if (a.M <= 96 || (a.M < 512 && wide_rows * 100 > skinny_rows * 115)) return kSkinny32;
        // Small products, where the 128 x 256 tiles cannot fill the GPU. Measured
        // (us, L2 flushed; 128 x 256 / 128 x 128 / 64 x 64 tiles): 128^3 43.6 /
        // 19.1 / 12.9, 512^3 34.5 / 24.2 / 20.1, 768^3 38.1 / 30.3 / 34.4,
        // 2048 x 2048 x 256 66.2 / 58.0 / 58.0, 256 x 256 x 4096 57.0 / 37.5 /
        // 30.4, 1024^3 59.0 / 60.6 / 73.4. While the 128 x 256 tiles fill
        // less than one wave: up to 512^3 of work, or a K at least 8 times
        // both M and N, 64 x 64 tiles; otherwise 128 x 128 tiles, except
        // for K >= 1024 with at least 32 of the 128 x 256 tiles.
        const long tiles_wide = ((long)a.M + 127) / 128 * (((long)a.N + 255) / 256);
        if (tiles_wide < num_sms) {
            const long mnk = (long)a.M * a.N * a.K;
            if (mnk <= 512L * 512 * 512 || ((long)a.K >= 8L * a.M && (long)a.K >= 8L * a.N))
                return kSmall;
            if (!(a.K >= 1024 && tiles_wide >= 32)) return kBig32;
        }
    }
    return (va ? 0 : 2) + (vb ? 0 : 1);
}

F32Plan f32_plan(int id, const GemmArgs& a, int num_sms) {
    const Entry& e = kTable[id];
    F32Plan pl;
    pl.tiles_m = (a.M + e.bm - 1) / e.bm;
    pl.tiles_n = (a.N + e.bn - 1) / e.bn;
    pl.ktiles = (a.K + e.bk - 1) / e.bk;
    // One resident block of the packed 128 x 256 tile retires ~0.39 TFLOP/s
    // (59 TFLOP/s over 152 SMs); other configurations are within 25 %.
    const double slot_flops_per_us = 0.39e6;
    const double tile_us = 2.0 * e.bm * e.bn * (double)a.K / slot_flops_per_us;
    plan_tail_split(pl.tiles_m * pl.tiles_n, num_sms * e.min_blocks, pl.ktiles, tile_us,
                    (double)e.bm * e.bn * sizeof(float), pl.dp_tiles, pl.split);
    pl.scratch_bytes = pl.split > 1
        ? (size_t)(pl.tiles_m * pl.tiles_n - pl.dp_tiles) * pl.split * e.bm * e.bn * sizeof(float)
        : 0;
    return pl;
}

cudaError_t f32_launch(int id, const GemmArgs& a, const F32Plan& pl, float* scratch,
                       cudaStream_t s) {
    const Entry& e = kTable[id];
    F32Params p;
    p.A = static_cast<const float*>(a.A);
    p.lda = a.lda;
    p.B = static_cast<const float*>(a.B);
    p.ldb = a.ldb;
    p.C = a.C;
    p.ldc = a.ldc;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.tiles_m = pl.tiles_m;
    p.tiles_n = pl.tiles_n;
    p.ktiles = pl.ktiles;
    p.dp_tiles = pl.dp_tiles;
    p.split = pl.split;
    p.partials = scratch;
    p.vec_c = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0 && a.ldc % 4 == 0) ? 1 : 0;
    p.alpha = a.ep.alpha;
    p.beta = a.ep.beta;
    p.bias = a.ep.bias;
    p.ep_simple = a.ep.simple() ? 1 : 0;
    const int tiles = pl.tiles_m * pl.tiles_n;
    const int blocks = pl.dp_tiles + (tiles - pl.dp_tiles) * (pl.split > 1 ? pl.split : 0);
    cudaError_t err = e.launch(p, blocks, s);
    if (err != cudaSuccess || pl.split <= 1) return err;
    return e.reduce(p, s);
}

// The zero product (beta = 0, no bias) on 16-byte rows: four zeros per
// store, a flat grid-stride loop over (row, vector), the N % 4 last columns
// one by one.
__global__ void __launch_bounds__(256)
zero_rows_vec_kernel(float* __restrict__ C, long ldc, int M, int N) {
    pdl_launch_dependents();    // the next kernel may launch now
    pdl_wait();                 // the previous kernel's writes are visible
    const int vecs = N / 4;
    const long total = (long)M * vecs;
    for (long u = blockIdx.x * (long)blockDim.x + threadIdx.x; u < total;
         u += (long)gridDim.x * blockDim.x) {
        const int r = (int)(u / vecs), c = (int)(u % vecs) * 4;
        *reinterpret_cast<float4*>(C + (long)r * ldc + c) = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    const int tail = N % 4;
    for (long u = blockIdx.x * (long)blockDim.x + threadIdx.x; u < (long)M * tail;
         u += (long)gridDim.x * blockDim.x)
        C[(long)(u / tail) * ldc + vecs * 4 + (int)(u % tail)] = 0.0f;
}

cudaError_t empty_product(float* C, long ldc, int M, int N, const Epilogue& ep, cudaStream_t s) {
    if (ep.beta == 0.0f && ep.bias == nullptr && reinterpret_cast<uintptr_t>(C) % 16 == 0 &&
        ldc % 4 == 0 && N >= 4) {
        long blocks = ((long)M * (N / 4) + 255) / 256;
        if (blocks > 152L * 8 * 4) blocks = 152L * 8 * 4;
        if (blocks < 1) blocks = 1;
        return launch_pdl(zero_rows_vec_kernel, dim3((int)blocks), dim3(256), 0, s, C, ldc, M, N);
    }
    int gx = (N + 255) / 256;
    if (gx > 64) gx = 64;
    if (gx < 1) gx = 1;
    const int gy = M < 16384 ? (M > 0 ? M : 1) : 16384;
    return launch_pdl(empty_product_kernel, dim3(gx, gy), dim3(256), 0, s, C, ldc, M, N, ep.beta,
                      ep.bias);
}

}  // namespace tgemm
