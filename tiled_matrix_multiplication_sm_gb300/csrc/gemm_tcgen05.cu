// Dense product C = A x B on the 5th-generation tensor cores of sm_103a
// (tcgen05 MMA, accumulators in tensor memory), TF32 or BF16 inputs, FP32
// output.
//
// It is the same tiling as "Tiled GEMM: Matrix Multiplication in CUDA",
// sections 2 and 4 -- a block owns a tile of C and walks K in phases, staging
// tiles of A and B on chip -- with each step moved to the unit that does it
// best on this chip:
//   * the cooperative load of each phase (section 4.4) is one Tensor Memory
//     Accelerator copy per operand tile ("Tiled GEMM ...", section 8, TMA),
//     into a ring of STAGES shared-memory buffers in the 128-byte swizzled
//     layout the tensor core reads without bank conflicts;
//   * the two barriers of each phase (sections 4.5 and 4.7: tile loaded
//     before it is read, read before it is overwritten) are a "full" and an
//     "empty" mbarrier per ring slot;
//   * the inner product over the tile (section 4.6) is a chain of
//     tcgen05.mma instructions issued by one thread, accumulating an FP32
//     tile in tensor memory;
//   * the write-back (section 4.8) is done by epilogue warps that read
//     tensor memory with tcgen05.ld and, where C's rows allow, hand 32 x 32
//     blocks to TMA stores.
// Three tile shapes: 128 x 256 on one SM and 256 x 256 on an SM pair
// (cta_group::2), both with two accumulators so the epilogue of one tile
// overlaps the MMAs of the next; and 256 x 512 on an SM pair, whose two
// N = 256 MMAs per K step share the staged A (less operand traffic per
// FLOP) at the price of a single accumulator that the epilogue frees in two
// halves. The grid is persistent: one block (or pair) per SM (pair) walks
// tiles in a grouped order so that blocks running together share panels of
// A and B in L2.
//
// Ragged edges (section 7.1 of the same page): the TMA unit fills rows and
// columns outside the matrices with zeros; stores past M and N are skipped
// (TMA stores clip them).
//
// Operand layouts in shared memory: A (M x K, K contiguous) is K-major. For
// BF16, B (K x N, N contiguous) is read MN-major through the instruction
// descriptor's transpose bit, so neither operand is copied. The TF32 kind
// reads B only K-major (with the MN-major bit set it produced zeros on
// sm_103a), so the TF32 path hands this kernel B already transposed
// (N x K, K contiguous) and reads it K-major like A.
//
// Every wait is bounded (a limit in nanoseconds, default 2 s). A wait that
// runs out records TGEMM_ERR_DEVICE_TIMEOUT in a device status word and
// raises a block-wide abort flag; all roles then leave their loops, wait
// (bounded) for their own copies and MMAs still in flight, free tensor
// memory and return. Nothing traps.

#include "tgemm_internal.h"

#include <cuda.h>
#include <cstdint>
#include <cstring>

namespace tgemm {

__device__ int g_tc_status;

namespace {

constexpr int kStatusTimeout = 4;      // TGEMM_ERR_DEVICE_TIMEOUT

constexpr int BM = 128;                // rows of a C tile (= MMA M)
constexpr int BN = 256;                // columns of a C tile (= MMA N)
constexpr int STAGES = 4;
constexpr int SW = 128;                // bytes in one swizzled row
constexpr int A_STAGE_BYTES = BM * SW;                 // 16 KB
constexpr int B_STAGE_BYTES = 32 * 1024;               // BK x BN elements
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int TMEM_COLS = 2 * BN;                      // two accumulators
constexpr int NUM_THREADS = 192;       // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int GROUP_M = 8;

template <int ESZ> struct Kind;
template <> struct Kind<2> {           // bf16 inputs, kind::f16
    static constexpr int BK = 64;      // K elements per stage (one 128-byte row)
    static constexpr int UMMA_K = 16;  // K per instruction
    static constexpr uint32_t FMT = 1; // BF16
};
template <> struct Kind<4> {           // fp32 storage, kind::tf32
    static constexpr int BK = 32;
    static constexpr int UMMA_K = 8;
    static constexpr uint32_t FMT = 2; // TF32
};

struct Sync {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Epilogue staging: EPI_BUFS 32 x 32 FP32 blocks per epilogue warp.
constexpr int EPI_BUFS = 1;
constexpr int EPI_WARP_BYTES = EPI_BUFS * 32 * 32 * 4;
constexpr int EPI_STAGE_BYTES = 4 * EPI_WARP_BYTES;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_STAGE_BYTES + (int)sizeof(Sync);
static_assert(SMEM_BYTES <= 227 * 1024, "one-SM kernel exceeds the shared memory of a block");

struct TcParams {
    int M, N, K;
    float* C;
    long ldc;
    int tiles_m, tiles_n, num_tiles, kblocks;
    int tile_rows;       // rows of a tile: 128 (one SM) or 256 (SM pair)
    int tile_cols;       // columns of a tile: 256, or 512 (wide SM-pair tiles)
    int dp_tiles;        // tiles [0, dp_tiles) are computed whole
    int split;           // the others in `split` K-pieces each (1: none)
    int num_units;       // dp_tiles + (num_tiles - dp_tiles) * split
    float* partials;     // one tile_rows x tile_cols partial tile per K-piece
    unsigned long long wait_limit_ns;
    int debug_stall;
    int vec_c;
    // Output rule C = alpha * acc + beta * C_old + bias[col]; ep_simple when
    // it is the plain product.
    float alpha, beta;
    const float* bias;
    int ep_simple;
    int tma_c;           // whole tiles leave through TMA stores (plain rule, 16-byte rows of C)
};

// One output under the rule (C_old read only when beta != 0).
__device__ __forceinline__ float apply_epilogue(float acc, const TcParams& p, const float* c_old,
                                                int col) {
    float v = p.alpha * acc;
    if (p.beta != 0.0f) v = fmaf(p.beta, *c_old, v);
    if (p.bias != nullptr) v += p.bias[col];
    return v;
}

// A unit of persistent work: a whole tile, or K-blocks [kb0, kb1) of a tile
// whose partial result goes to scratch (piece >= 0).
struct Unit {
    int tile, kb0, kb1;
    int piece;
};

__device__ __forceinline__ Unit decode_unit(int u, const TcParams& p) {
    Unit w;
    if (u < p.dp_tiles) {
        w.tile = u;
        w.kb0 = 0;
        w.kb1 = p.kblocks;
        w.piece = -1;
    } else {
        const int pc = u - p.dp_tiles;
        const int j = pc % p.split;
        w.tile = p.dp_tiles + pc / p.split;
        w.kb0 = (int)((long)j * p.kblocks / p.split);
        w.kb1 = (int)((long)(j + 1) * p.kblocks / p.split);
        w.piece = pc;
    }
    return w;
}

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Wait until the phase of `bar` with parity `parity` has completed. Gives up
// (returns false) when the block's abort flag is raised or, if
// `honour_abort` is false, only when `limit_ns` has passed; a wait that runs
// out raises the abort flag and records the timeout.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* abort_flag,
                                       unsigned long long limit_ns, bool honour_abort) {
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 15u) == 0) {
            if (honour_abort && *(volatile int*)abort_flag) return false;
            if (globaltimer() - t0 > limit_ns || it >= (1u << 30)) {
                *(volatile int*)abort_flag = 1;
                atomicCAS(&g_tc_status, 0, kStatusTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// TMA store of a box from shared memory (completion tracked by bulk groups).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(src) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until the shared-memory sources of all but the newest `N` of this
// thread's bulk store groups are read.
template <int N>
__device__ __forceinline__ void tma_store_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory");
}
// Wait until this thread's bulk stores are complete.
__device__ __forceinline__ void tma_store_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

// ---- CTA-pair (cluster of 2) helpers for the 2-SM kernel
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                 :: "r"(cluster_addr) : "memory");
}

// TMA load into this CTA's shared memory whose completion is counted on an
// mbarrier that may live in the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

// Arrive (once the MMAs issued so far complete) on the barrier at `bar` in
// both CTAs of the pair.
__device__ __forceinline__ void tc_commit_pair_multicast(uint32_t bar) {
    const uint16_t both = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" :: "r"(bar), "h"(both) : "memory");
}

__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}

template <int ESZ>
__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
    if constexpr (ESZ == 2) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
            :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
            :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
    }
}

template <int ESZ>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
    if constexpr (ESZ == 2) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
            :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
            :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
    }
}

// Start loading 32 consecutive accumulator columns of this thread's TMEM
// lane; the registers hold them after tmem_wait_ld.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// Wait for this thread's TMEM loads. `r` is tied to the wait, so no use of
// the loaded registers can be scheduled above it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :: "memory");
}

// 32 consecutive accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    tmem_ld32_async(taddr, r);
    tmem_wait_ld(r);
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format: start
// address, leading and stride byte offsets in 16-byte units, version 1).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFF) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= 1ull << 46;                     // descriptor version for tcgen05
    d |= 2ull << 61;                     // 128-byte swizzle
    return d;
}

// Instruction descriptor: FP32 accumulator, A K-major, B K-major or
// MN-major, M x N.
template <int ESZ, bool B_KMAJOR, int MMA_M = BM>
__host__ __device__ constexpr uint32_t instr_desc() {
    return (1u << 4)                         // D format F32
         | (Kind<ESZ>::FMT << 7)             // A format
         | (Kind<ESZ>::FMT << 10)            // B format
         | (0u << 15)                        // A: K-major
         | ((B_KMAJOR ? 0u : 1u) << 16)      // B: K-major (0) or MN-major (1)
         | ((uint32_t)(BN >> 3) << 17)
         | ((uint32_t)(MMA_M >> 4) << 24);
}

__device__ __forceinline__ void tile_coords(int t, const TcParams& p, int& mb, int& nb) {
    const int per_group = GROUP_M * p.tiles_n;
    const int first_m = (t / per_group) * GROUP_M;
    const int gm = min(p.tiles_m - first_m, GROUP_M);
    mb = first_m + (t % per_group) % gm;
    nb = (t % per_group) / gm;
}

// 32 consecutive values to a 4-byte aligned address whose first H values
// precede a 16-byte boundary: those H one by one, then 16-byte stores, then
// the (32 - H) % 4 values after the last boundary.
template <int H>
__device__ __forceinline__ void store_row32_from(float* d, const uint32_t (&r)[32]) {
#pragma unroll
    for (int j = 0; j < H; ++j) d[j] = __uint_as_float(r[j]);
#pragma unroll
    for (int j = H; j + 4 <= 32; j += 4)
        *reinterpret_cast<float4*>(d + j) =
            make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                        __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
#pragma unroll
    for (int j = 32 - (32 - H) % 4; j < 32; ++j) d[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void store_row32_peeled(float* d, const uint32_t (&r)[32]) {
    switch ((4 - (int)((reinterpret_cast<uintptr_t>(d) >> 2) & 3)) & 3) {
        case 0: store_row32_from<0>(d, r); break;
        case 1: store_row32_from<1>(d, r); break;
        case 2: store_row32_from<2>(d, r); break;
        default: store_row32_from<3>(d, r); break;
    }
}

// Epilogue of one unit for this thread's accumulator row `row_in_tile`:
// the 32-column blocks [c_begin, c_end) of the tile from TMEM (the tile's
// column 0 at address `taddr`) to C, or, for a K-piece, to its partial tile
// in scratch. Rows past M and columns past N are skipped (the reduction never
// reads them). All lanes of the warp call this together.
//
// Otherwise each thread stores its row's 32-column blocks with 16-byte
// stores, after peeling the values before the first 16-byte boundary when
// C's rows are not 16-byte aligned. (Staging each 32 x 32 block through
// shared memory to store it as 32 coalesced row segments instead measured
// 9 % slower on 3072 x 5120 x 1536 TF32 with ldc = 5121: the staging's
// shared-memory traffic competes with the MMAs' operand reads.)
__device__ __forceinline__ void store_accumulator(const TcParams& p, const Unit& w, int mb, int nb,
                                                 int row_in_tile, uint32_t taddr, float* stage,
                                                 const CUtensorMap* tmC, int c_begin, int c_end) {
    const int row = mb * p.tile_rows + row_in_tile;
    const int lane = threadIdx.x & 31;
    if (w.piece < 0 && p.tma_c) {
        // Whole tile, beta = 0: alpha and bias are applied in registers, then
        // each 32 x 32 block goes to the warp's staging buffer (EPI_BUFS of
        // them) in the 128-byte-swizzled layout of the C tensor map (row i
        // holds 128 bytes, 16-byte chunk j at j ^ (i % 8)) and leaves as one
        // TMA store, which also clips rows and columns past M and N. The next
        // block's TMEM load is in flight while a block is staged, and a
        // buffer is reused once the store issued EPI_BUFS blocks earlier has
        // read it.
        const int row0 = row - lane;
        if (row0 >= p.M) return;                        // the warp's rows are all past M
        const int n_blocks = (p.N - nb * p.tile_cols + 31) / 32;   // blocks with columns < N
        const int c_stop = c_end < n_blocks ? c_end : n_blocks;
        if (c_begin >= c_stop) return;
        uint32_t r[32], nx[32];
        tmem_ld32(taddr + (uint32_t)(c_begin * 32), r);
        for (int c = c_begin; c < c_stop; ++c) {
            const int col0 = nb * p.tile_cols + c * 32;
            const bool more = c + 1 < c_stop;
            if (more) tmem_ld32_async(taddr + (uint32_t)((c + 1) * 32), nx);
            if (!p.ep_simple) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (col0 + j < p.N)
                        r[j] = __float_as_uint(apply_epilogue(__uint_as_float(r[j]), p, nullptr,
                                                              col0 + j));
            }
            float* buf = stage + ((c - c_begin) % EPI_BUFS) * (32 * 32);
            if (lane == 0) tma_store_wait_read<EPI_BUFS - 1>();   // buf's previous store has read it
            __syncwarp();
            float4* srow = reinterpret_cast<float4*>(buf + lane * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                srow[j ^ (lane & 7)] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                   __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) tma_store_2d(tmC, col0, row0, smem_u32(buf));
            if (more) {
                tmem_wait_ld(nx);
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = nx[j];
            }
        }
        return;
    }
    float* dst;
    bool vec, ep;
    if (w.piece < 0) {
        dst = p.C + (long)row * p.ldc + (long)nb * p.tile_cols;
        vec = p.vec_c != 0;
        ep = p.ep_simple == 0;                  // a whole tile writes final outputs
    } else {
        dst = p.partials + ((long)w.piece * p.tile_rows + row_in_tile) * p.tile_cols;
        vec = true;
        ep = false;                             // partial sums: the reduction applies the rule
    }
    for (int c = c_begin; c < c_end; ++c) {
        const int col0 = nb * p.tile_cols + c * 32;
        if (col0 >= p.N) break;                     // uniform across the warp
        uint32_t r[32];
        tmem_ld32(taddr + (uint32_t)(c * 32), r);
        if (row < p.M) {
            float* d = dst + c * 32;
            if (ep) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (col0 + j < p.N)
                        r[j] = __float_as_uint(apply_epilogue(__uint_as_float(r[j]), p, d + j,
                                                              col0 + j));
            }
            if (vec && col0 + 31 < p.N) {
                store_row32_from<0>(d, r);
            } else if (col0 + 31 < p.N) {
                store_row32_peeled(d, r);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (col0 + j < p.N) d[j] = __uint_as_float(r[j]);
            }
        }
    }
}

// Sum of `n` float4 at src, src + stride, ... in that order; the loads of
// four pieces are issued before their adds, so that they are in flight
// together.
__device__ __forceinline__ float4 sum_pieces(const float* src, long stride, int n) {
    float4 s = *reinterpret_cast<const float4*>(src);
    for (int j = 1; j < n; j += 4) {
        float4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (j + q < n) v[q] = *reinterpret_cast<const float4*>(src + (j + q) * stride);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (j + q < n) {
                s.x += v[q].x;
                s.y += v[q].y;
                s.z += v[q].z;
                s.w += v[q].w;
            }
    }
    return s;
}

// Sum the K-pieces of every split tile, piece 0 first, into C.
__global__ void __launch_bounds__(256)
tc_splitk_reduce(const TcParams p) {
    const int Q = p.tile_cols / 4;                         // float4 per tile row
    const int rows = p.tile_rows < p.M ? p.tile_rows : p.M; // rows a tile can hold (M small: M)
    const long per_tile = (long)rows * Q;
    const long total = (long)(p.num_tiles - p.dp_tiles) * per_tile;
    const long piece_floats = (long)p.tile_rows * p.tile_cols;
    for (long u = blockIdx.x * (long)blockDim.x + threadIdx.x; u < total;
         u += (long)gridDim.x * blockDim.x) {
        const int r = (int)(u / per_tile);
        const int e = (int)(u % per_tile);
        const int row = e / Q, c4 = (e % Q) * 4;
        int mb, nb;
        tile_coords(p.dp_tiles + r, p, mb, nb);
        const int grow = mb * p.tile_rows + row, gcol = nb * p.tile_cols + c4;
        if (grow >= p.M || gcol >= p.N) continue;
        const float* src = p.partials + (long)r * p.split * piece_floats + (long)row * p.tile_cols + c4;
        const float4 s = sum_pieces(src, piece_floats, p.split);
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

// B_KMAJOR: B arrives transposed (N x K, K contiguous) and is read K-major;
// otherwise B is K x N (N contiguous) and is read MN-major.
template <int ESZ, bool B_KMAJOR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
               const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC,
               const TcParams p) {
    using KD = Kind<ESZ>;
    constexpr int BK = KD::BK;
    constexpr int K_STEPS = BK / KD::UMMA_K;
    constexpr int B_CHUNK_COLS = SW / ESZ;               // N columns per swizzled row
    constexpr int B_CHUNKS = BN / B_CHUNK_COLS;
    constexpr int B_CHUNK_BYTES = BK * SW;
    constexpr uint32_t A_K_STEP = KD::UMMA_K * ESZ;      // bytes along a K-major row
    constexpr uint32_t B_K_STEP = KD::UMMA_K * SW;       // rows of the MN-major tile
    static_assert(B_CHUNKS * B_CHUNK_BYTES == B_STAGE_BYTES, "B stage size");
    constexpr uint32_t IDESC = instr_desc<ESZ, B_KMAJOR>();

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    float* epi_stage = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES);
    Sync* sy = reinterpret_cast<Sync*>(smem + STAGES * STAGE_BYTES + EPI_STAGE_BYTES);
    const uint32_t a_base = smem_u32(smem);
    const uint32_t b_base = a_base + STAGES * A_STAGE_BYTES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&sy->full[s]), 1);
            mbar_init(smem_u32(&sy->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&sy->tmem_full[a]), 1);
            mbar_init(smem_u32(&sy->tmem_empty[a]), 4);      // one arrival per epilogue warp
        }
        mbar_init(smem_u32(&sy->drain), 1);
        sy->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&sy->tmem_base)), "n"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sy->tmem_base;
    const unsigned long long lim = p.wait_limit_ns;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t armed = 0, armed_parity = 0;   // per-stage fills in flight
            int g = 0;
            for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
                const Unit w = decode_unit(u, p);
                int mb, nb;
                tile_coords(w.tile, p, mb, nb);
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++g) {
                    const int s = g % STAGES;
                    const uint32_t ph = (uint32_t)(g / STAGES) & 1u;
                    if (!mbar_wait(smem_u32(&sy->empty[s]), ph ^ 1u, &sy->abort, lim, true)) goto producer_done;
                    if (p.debug_stall && g == 0) continue;     // test hook: never fill stage 0
                    const uint32_t full = smem_u32(&sy->full[s]);
                    mbar_arrive_expect_tx(full, STAGE_BYTES);
                    tma_load_2d(a_base + s * A_STAGE_BYTES, &tmA, kb * BK, mb * BM, full);
                    const uint32_t bdst = b_base + s * B_STAGE_BYTES;
                    if constexpr (B_KMAJOR) {
                        tma_load_2d(bdst, &tmB, kb * BK, nb * BN, full);
                    } else {
#pragma unroll
                        for (int c = 0; c < B_CHUNKS; ++c)
                            tma_load_2d(bdst + c * B_CHUNK_BYTES, &tmB, nb * BN + c * B_CHUNK_COLS,
                                        kb * BK, full);
                    }
                    armed |= 1u << s;
                    armed_parity = (armed_parity & ~(1u << s)) | (ph << s);
                }
            }
        producer_done:
            // Copies still in flight must land before the block may exit.
            for (int s = 0; s < STAGES; ++s)
                if (armed & (1u << s))
                    mbar_wait(smem_u32(&sy->full[s]), (armed_parity >> s) & 1u, &sy->abort, lim, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int g = 0, it = 0;
            for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++it) {
                const Unit w = decode_unit(u, p);
                const int acc = it & 1;
                const uint32_t aph = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait(smem_u32(&sy->tmem_empty[acc]), aph ^ 1u, &sy->abort, lim, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                bool ok = true;
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++g) {
                    const int s = g % STAGES;
                    const uint32_t ph = (uint32_t)(g / STAGES) & 1u;
                    if (!mbar_wait(smem_u32(&sy->full[s]), ph, &sy->abort, lim, true)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = a_base + s * A_STAGE_BYTES;
                    const uint32_t b_addr = b_base + s * B_STAGE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < K_STEPS; ++kk) {
                        const uint64_t ad = smem_desc(a_addr + kk * A_K_STEP, 16, 1024);
                        const uint64_t bd =
                            B_KMAJOR ? smem_desc(b_addr + kk * A_K_STEP, 16, 1024)
                                     : smem_desc(b_addr + kk * B_K_STEP, B_CHUNK_BYTES, 1024);
                        tc_mma<ESZ>(d_tmem, ad, bd, IDESC, (kb != w.kb0 || kk != 0) ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&sy->empty[s]));      // frees the slot when done
                }
                if (!ok) break;
                tc_commit(smem_u32(&sy->tmem_full[acc]));    // accumulator ready
            }
            // Every MMA this thread issued must finish before TMEM is freed.
            tc_commit(smem_u32(&sy->drain));
            mbar_wait(smem_u32(&sy->drain), 0, &sy->abort, lim, false);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2-5)
        const int q = warp & 3;                 // TMEM lanes 32q .. 32q+31
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        int it = 0;
        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++it) {
            const Unit w = decode_unit(u, p);
            int mb, nb;
            tile_coords(w.tile, p, mb, nb);
            const int acc = it & 1;
            const uint32_t aph = (uint32_t)(it >> 1) & 1u;
            bool ok = mbar_wait(smem_u32(&sy->tmem_full[acc]), aph, &sy->abort, lim, true);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            store_accumulator(p, w, mb, nb, q * 32 + lane, tmem_base + lane_off + (uint32_t)(acc * BN),
                              epi_stage + q * (EPI_WARP_BYTES / 4), &tmC, 0, BN / 32);
            tc_fence_before();
            __syncwarp();                               // the warp's TMEM reads are done
            if (lane == 31) mbar_arrive(smem_u32(&sy->tmem_empty[acc]));   // not the storing lane
        }
        if (lane == 0) tma_store_wait_all();    // C stores done before the block retires
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem_base), "n"(TMEM_COLS) : "memory");
    }
}

// ===================================================================
// 2-SM variant: a cluster of two CTAs on a pair of SMs computes a 256 x 256
// tile with tcgen05.mma.cta_group::2 (M = 256, N = 256). CTA r of the pair
// stages rows 128r..128r+127 of the A tile and columns 128r..128r+127 of the
// B tile; the leader CTA (r = 0) issues the MMAs for both, and each CTA's
// tensor memory receives its 128 rows of the 256 x 256 accumulator. Each SM
// thus streams half of B instead of all of it, which halves the shared-
// memory traffic of the B operand per SM: the one-SM kernel's ring is
// shared-memory-bandwidth bound at about two thirds of the tensor rate.
//
// Hand-offs:
//   full[s]     leader only: the leader's producer expects both CTAs'
//               bytes; both producers' copies complete on it.
//   empty[s]    both CTAs: arrived by the leader's commit (multicast).
//   tmem_full   both CTAs: arrived by the leader's commit (multicast).
//   tmem_empty  leader only: every epilogue warp of the pair arrives once
//               (one lane, after the warp's TMEM reads).
// Both CTAs allocate and free tensor memory jointly (cta_group::2); cluster
// barriers after set-up and before the free keep the pair in step.
//
// Wide tiles (NW = 2): the pair computes a 256 x 512 tile as two N = 256
// MMAs per K step that share the staged A, so each SM stages 128 rows of A
// and 256 columns of B per K block: a quarter less TMA traffic and an eighth
// less shared-memory traffic per FLOP than 256 x 256 tiles. The 128 x 512
// FP32 accumulator of each CTA fills its tensor memory, so there is one
// accumulator, and the MMAs of the next tile wait for the epilogue; eight
// epilogue warps (two per TMEM lane quarter, one per half of the columns)
// keep that wait short.

constexpr int P_STAGES = 6;                                // ring depth (3 for the split-TF32 form)
constexpr int P_WIDE_STAGES = 4;                           // ring depth of the wide tiles
constexpr int P_A_TILE = 128 * SW;                         // 16 KB: this CTA's 128 rows of A
constexpr int P_B_TILE = 16 * 1024;                        // this CTA's 128 columns of B
constexpr int P_BM = 256;                                  // pair tile rows (= MMA M)

// Ring geometry. X3 (the three-product split-TF32 form) stages a high and a
// low copy of each operand per K block.
template <bool X3, int NW = 1>
struct PairRing {
    static constexpr int COPIES = X3 ? 2 : 1;
    static constexpr int STAGES = X3 ? 3 : NW == 2 ? P_WIDE_STAGES : P_STAGES;
    static constexpr int A_STAGE = COPIES * P_A_TILE;
    static constexpr int B_STAGE = COPIES * NW * P_B_TILE;
    static constexpr int STAGE = A_STAGE + B_STAGE;
};
// The 16 KB after the ring keep every shared-memory address an MMA
// descriptor can reach (a descriptor walks at most one 256-column B tile
// past its start) inside the block's allocation; the epilogue warps use them
// as their 32 x 32 staging blocks.
constexpr int P_GUARD_BYTES = 16 * 1024;
// Epilogue geometry: warps, block size, and their staging blocks (two
// 4 KB blocks per warp, at least the guard).
template <int NW>
struct PairEpi {
    static constexpr int WARPS = NW == 2 ? 8 : 4;
    static constexpr int THREADS = 64 + 32 * WARPS;
    static constexpr int BYTES =
        WARPS * EPI_WARP_BYTES > P_GUARD_BYTES ? WARPS * EPI_WARP_BYTES : P_GUARD_BYTES;
};
template <bool X3, int NW>
constexpr int pair_smem_bytes() {
    return 1024 + PairRing<X3, NW>::STAGES * PairRing<X3, NW>::STAGE + PairEpi<NW>::BYTES + 256;
}
static_assert(pair_smem_bytes<false, 1>() <= 227 * 1024 && pair_smem_bytes<true, 1>() <= 227 * 1024 &&
                  pair_smem_bytes<false, 2>() <= 227 * 1024,
              "CTA-pair kernels exceed the shared memory of a block");

struct PairSync {
    uint64_t full[P_STAGES];
    uint64_t empty[P_STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(PairSync) <= 256, "pair barrier block");

// X3 (TF32 only, B K-major): A and B each arrive as a high and a low TF32
// part (tmA/tmB and tmA2/tmB2), and every K step issues three MMAs into the
// same accumulator, lo(A) hi(B) + hi(A) lo(B) + hi(A) hi(B), which carries
// the product to FP32-level accuracy (the lo x lo term is below FP32's own
// rounding).
template <int ESZ, bool B_KMAJOR, bool X3, int NW>
__global__ void __launch_bounds__(PairEpi<NW>::THREADS, 1)
tc_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ CUtensorMap tmC,
                   const TcParams p) {
    using R = PairRing<X3, NW>;
    static_assert(!X3 || (ESZ == 4 && B_KMAJOR), "the split form is TF32 with B K-major");
    static_assert(NW == 1 || (NW == 2 && !X3), "wide tiles are for the one-product forms");
    constexpr int NACC = 2 / NW;                         // accumulators in tensor memory
    using KD = Kind<ESZ>;
    constexpr int BK = KD::BK;
    constexpr int K_STEPS = BK / KD::UMMA_K;
    constexpr int B_CHUNK_COLS = SW / ESZ;               // N columns per swizzled row
    constexpr int B_CHUNKS = 128 / B_CHUNK_COLS;         // per CTA (its 128 columns)
    constexpr int B_CHUNK_BYTES = BK * SW;
    constexpr uint32_t A_K_STEP = KD::UMMA_K * ESZ;
    constexpr uint32_t B_K_STEP = KD::UMMA_K * SW;
    static_assert(B_KMAJOR || B_CHUNKS * B_CHUNK_BYTES == P_B_TILE, "B stage size");
    static_assert(!B_KMAJOR || 128 * SW == P_B_TILE, "B stage size");
    constexpr uint32_t IDESC = instr_desc<ESZ, B_KMAJOR, P_BM>();

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    PairSync* sy = reinterpret_cast<PairSync*>(smem + R::STAGES * R::STAGE + PairEpi<NW>::BYTES);
    const uint32_t a_base = smem_u32(smem);
    const uint32_t b_base = a_base + R::STAGES * R::A_STAGE;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < R::STAGES; ++s) {
            mbar_init(smem_u32(&sy->full[s]), 1);
            mbar_init(smem_u32(&sy->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&sy->tmem_full[a]), 1);
            mbar_init(smem_u32(&sy->tmem_empty[a]), 2 * PairEpi<NW>::WARPS);  // one per warp, both CTAs
        }
        if constexpr (X3) {
            asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmA2)) : "memory");
            asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmB2)) : "memory");
        }
        mbar_init(smem_u32(&sy->drain), 1);
        sy->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(&sy->tmem_base)), "n"(TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync_all();        // barriers of both CTAs initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = sy->tmem_base;
    const unsigned long long lim = p.wait_limit_ns;
    // The leader's copies of the shared hand-off barriers, as cluster addresses.
    const uint32_t full0 = map_to_rank(smem_u32(&sy->full[0]), 0);
    const uint32_t tmem_empty0 = map_to_rank(smem_u32(&sy->tmem_empty[0]), 0);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            uint32_t armed = 0, armed_parity = 0;
            int g = 0;
            for (int u = pair; u < p.num_units; u += num_pairs) {
                const Unit w = decode_unit(u, p);
                int mb, nb;
                tile_coords(w.tile, p, mb, nb);
                const int row0 = mb * P_BM + (int)rank * 128;
                const int col0 = nb * (NW * BN) + (int)rank * 128;
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++g) {
                    const int s = g % R::STAGES;
                    const uint32_t ph = (uint32_t)(g / R::STAGES) & 1u;
                    if (!mbar_wait(smem_u32(&sy->empty[s]), ph ^ 1u, &sy->abort, lim, true)) goto pair_producer_done;
                    if (p.debug_stall && g == 0) continue;     // test hook: stage 0 never filled
                    const uint32_t full = full0 + (uint32_t)(s * sizeof(uint64_t));
                    if (leader) mbar_arrive_expect_tx(smem_u32(&sy->full[s]), 2 * R::STAGE);
                    const uint32_t adst = a_base + s * R::A_STAGE;
                    tma_load_2d_pair(adst, &tmA, kb * BK, row0, full);
                    const uint32_t bdst = b_base + s * R::B_STAGE;
                    if constexpr (X3) {
                        tma_load_2d_pair(adst + P_A_TILE, &tmA2, kb * BK, row0, full);
                        tma_load_2d_pair(bdst, &tmB, kb * BK, col0, full);
                        tma_load_2d_pair(bdst + P_B_TILE, &tmB2, kb * BK, col0, full);
                    } else {
#pragma unroll
                        for (int h = 0; h < NW; ++h) {          // B tile h: columns h*256.. of the tile
                            const uint32_t bh = bdst + h * P_B_TILE;
                            const int ch = col0 + h * BN;
                            if constexpr (B_KMAJOR) {
                                tma_load_2d_pair(bh, &tmB, kb * BK, ch, full);
                            } else {
#pragma unroll
                                for (int c = 0; c < B_CHUNKS; ++c)
                                    tma_load_2d_pair(bh + c * B_CHUNK_BYTES, &tmB, ch + c * B_CHUNK_COLS,
                                                     kb * BK, full);
                            }
                        }
                    }
                    armed |= 1u << s;
                    armed_parity = (armed_parity & ~(1u << s)) | (ph << s);
                }
            }
        pair_producer_done:
            if (leader) {
                // Both CTAs' copies complete on the leader's barriers.
                for (int s = 0; s < R::STAGES; ++s)
                    if (armed & (1u << s))
                        mbar_wait(smem_u32(&sy->full[s]), (armed_parity >> s) & 1u, &sy->abort, lim, false);
            } else if (*(volatile int*)&sy->abort) {
                // After a timeout the peer cannot observe its own copies; give
                // any still in flight time to land (a copy takes microseconds).
                const unsigned long long t0 = globaltimer();
                while (globaltimer() - t0 < 2000000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (leader CTA)
        if (lane == 0 && leader) {
            int g = 0, it = 0;
            // The MMAs of ring stage s (K block kb of unit w) for B tiles [h0, h1).
            auto issue = [&](int s, int kb, const Unit& w, uint32_t d_tmem, int h0, int h1) {
                const uint32_t a_addr = a_base + s * R::A_STAGE;
                const uint32_t b_addr = b_base + s * R::B_STAGE;
#pragma unroll
                for (int kk = 0; kk < K_STEPS; ++kk) {
                    const uint32_t first = (kb != w.kb0 || kk != 0) ? 1u : 0u;
                    const uint64_t ad = smem_desc(a_addr + kk * A_K_STEP, 16, 1024);
                    if constexpr (X3) {
                        const uint64_t bd = smem_desc(b_addr + kk * A_K_STEP, 16, 1024);
                        const uint64_t ad_lo = smem_desc(a_addr + P_A_TILE + kk * A_K_STEP, 16, 1024);
                        const uint64_t bd_lo = smem_desc(b_addr + P_B_TILE + kk * A_K_STEP, 16, 1024);
                        tc_mma_pair<ESZ>(d_tmem, ad_lo, bd, IDESC, first);    // lo(A) hi(B)
                        tc_mma_pair<ESZ>(d_tmem, ad, bd_lo, IDESC, 1u);       // hi(A) lo(B)
                        tc_mma_pair<ESZ>(d_tmem, ad, bd, IDESC, 1u);          // hi(A) hi(B)
                    } else {
#pragma unroll
                        for (int h = 0; h < NW; ++h) {
                            if (h < h0 || h >= h1) continue;
                            const uint32_t bh = b_addr + h * P_B_TILE;
                            const uint64_t bdh =
                                B_KMAJOR ? smem_desc(bh + kk * A_K_STEP, 16, 1024)
                                         : smem_desc(bh + kk * B_K_STEP, B_CHUNK_BYTES, 1024);
                            tc_mma_pair<ESZ>(d_tmem + (uint32_t)(h * BN), ad, bdh, IDESC, first);
                        }
                    }
                }
            };
            for (int u = pair; u < p.num_units; u += num_pairs, ++it) {
                const Unit w = decode_unit(u, p);
                const int acc = it % NACC;
                const uint32_t aph = (uint32_t)(it / NACC) & 1u;
                if (!mbar_wait(smem_u32(&sy->tmem_empty[acc]), aph ^ 1u, &sy->abort, lim, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                bool ok = true;
                int kb = w.kb0;
                if constexpr (NW == 2) {
                    // The epilogue frees the accumulator's column halves one after
                    // the other (tmem_empty[0], then tmem_empty[1]). Run the first
                    // half's MMAs on the stages already loaded while the second
                    // half still drains, then catch up on the second half's.
                    const int held = min(R::STAGES, w.kb1 - w.kb0);
                    for (int i = 0; i < held; ++i) {
                        const int s = (g + i) % R::STAGES;
                        const uint32_t ph = (uint32_t)((g + i) / R::STAGES) & 1u;
                        if (!mbar_wait(smem_u32(&sy->full[s]), ph, &sy->abort, lim, true)) { ok = false; break; }
                        tc_fence_after();
                        issue(s, w.kb0 + i, w, d_tmem, 0, 1);
                    }
                    if (ok && !mbar_wait(smem_u32(&sy->tmem_empty[1]), aph ^ 1u, &sy->abort, lim, true))
                        ok = false;
                    if (ok) {
                        tc_fence_after();
                        for (int i = 0; i < held; ++i) {
                            const int s = (g + i) % R::STAGES;
                            issue(s, w.kb0 + i, w, d_tmem, 1, 2);
                            tc_commit_pair_multicast(smem_u32(&sy->empty[s]));   // slot free in both CTAs
                        }
                    }
                    g += held;
                    kb += held;
                }
                // Wide tiles: the last K blocks (as many as the ring holds) run
                // the first half's MMAs before the second half's, so the first
                // half is complete (tmem_full[0]) while the second still computes.
                const int tail = NW == 2 ? min(R::STAGES, w.kb1 - kb) : 0;
                for (; ok && kb < w.kb1 - tail; ++kb, ++g) {
                    const int s = g % R::STAGES;
                    const uint32_t ph = (uint32_t)(g / R::STAGES) & 1u;
                    if (!mbar_wait(smem_u32(&sy->full[s]), ph, &sy->abort, lim, true)) { ok = false; break; }
                    tc_fence_after();
                    issue(s, kb, w, d_tmem, 0, NW);
                    tc_commit_pair_multicast(smem_u32(&sy->empty[s]));   // slot free in both CTAs
                }
                if (!ok) break;
                if constexpr (NW == 2) {
                    for (int i = 0; i < tail; ++i) {
                        const int s = (g + i) % R::STAGES;
                        const uint32_t ph = (uint32_t)((g + i) / R::STAGES) & 1u;
                        if (!mbar_wait(smem_u32(&sy->full[s]), ph, &sy->abort, lim, true)) { ok = false; break; }
                        tc_fence_after();
                        issue(s, kb + i, w, d_tmem, 0, 1);
                    }
                    if (!ok) break;
                    tc_commit_pair_multicast(smem_u32(&sy->tmem_full[0]));   // first half ready in both
                    for (int i = 0; i < tail; ++i) {
                        const int s = (g + i) % R::STAGES;
                        issue(s, kb + i, w, d_tmem, 1, 2);
                        tc_commit_pair_multicast(smem_u32(&sy->empty[s]));   // slot free in both CTAs
                    }
                    g += tail;
                    kb += tail;
                    tc_commit_pair_multicast(smem_u32(&sy->tmem_full[1]));   // second half ready
                } else {
                    tc_commit_pair_multicast(smem_u32(&sy->tmem_full[acc]));  // accumulator ready in both
                }
            }
            tc_commit_pair(smem_u32(&sy->drain));
            mbar_wait(smem_u32(&sy->drain), 0, &sy->abort, lim, false);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2.., both CTAs)
        const int q = warp & 3;                              // TMEM lanes 32q .. 32q+31
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        constexpr int PARTS = PairEpi<NW>::WARPS / 4;      // warps sharing a lane quarter
        const int part = (warp - 2) >> 2;
        const int blocks = p.tile_cols / 32 / PARTS;         // 32-column blocks per warp
        int it = 0;
        for (int u = pair; u < p.num_units; u += num_pairs, ++it) {
            const Unit w = decode_unit(u, p);
            int mb, nb;
            tile_coords(w.tile, p, mb, nb);
            const int acc = it % NACC;
            const uint32_t aph = (uint32_t)(it / NACC) & 1u;
            bool ok = mbar_wait(smem_u32(&sy->tmem_full[acc]), aph, &sy->abort, lim, true);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            float* stage = reinterpret_cast<float*>(smem + R::STAGES * R::STAGE) +
                           (warp - 2) * (EPI_WARP_BYTES / 4);
            if constexpr (NW == 2) {
                // Column halves in order: each is drained once its MMAs are
                // complete (tmem_full[half]) and freed (tmem_empty[half]) as
                // soon as it has left tensor memory.
                bool ok2 = true;
                for (int half = 0; half < 2 && ok2; ++half) {
                    if (half == 1) {
                        ok2 = mbar_wait(smem_u32(&sy->tmem_full[1]), aph, &sy->abort, lim, true);
                        if (!__all_sync(0xffffffffu, ok2)) { ok2 = false; break; }
                        tc_fence_after();
                    }
                    const int c0 = half * (blocks * PARTS / 2) + part * (blocks / 2);
                    store_accumulator(p, w, mb, nb, (int)rank * 128 + q * 32 + lane,
                                      tmem_base + lane_off, stage, &tmC, c0, c0 + blocks / 2);
                    tc_fence_before();
                    __syncwarp();                       // the warp's TMEM reads are done
                    // Lane 31 arrives: lane 0 issued the warp's TMA stores,
                    // and its release-ordered arrive was measured ~0.2 us later.
                    if (lane == 31) mbar_arrive_cluster(tmem_empty0 + (uint32_t)(half * sizeof(uint64_t)));
                }
                if (!ok2) break;
            } else {
                store_accumulator(p, w, mb, nb, (int)rank * 128 + q * 32 + lane,
                                  tmem_base + lane_off + (uint32_t)(acc * BN), stage, &tmC,
                                  part * blocks, (part + 1) * blocks);
                tc_fence_before();
                __syncwarp();                           // the warp's TMEM reads are done
                if (lane == 31) mbar_arrive_cluster(tmem_empty0 + (uint32_t)(acc * sizeof(uint64_t)));
            }
        }
        if (lane == 0) tma_store_wait_all();    // C stores done before the block retires
    }

    tc_fence_before();
    cluster_sync_all();        // the leader's MMAs are drained; no copy in flight
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem_base), "n"(TMEM_COLS) : "memory");
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 2-D row-major tensor map: `cols` contiguous elements per row, `rows`
// rows `ld` elements apart; boxes of box_cols x box_rows, 128-byte swizzle.
bool encode_2d(EncodeTiledFn enc, CUtensorMap* map, const void* base, int esz, long rows,
               long cols, long ld, int box_cols, int box_rows) {
    const CUtensorMapDataType dt =
        esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * esz};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

TcParams make_params(const GemmArgs& a, const TcPlan& pl, float* partials,
                     unsigned long long wait_limit_ns, int debug_stall) {
    TcParams p;
    p.M = a.M; p.N = a.N; p.K = a.K;
    p.C = a.C; p.ldc = a.ldc;
    p.tiles_m = pl.tiles_m;
    p.tiles_n = pl.tiles_n;
    p.num_tiles = pl.tiles_m * pl.tiles_n;
    p.kblocks = pl.kblocks;
    p.tile_rows = pl.tile_rows;
    p.tile_cols = pl.tile_cols;
    p.dp_tiles = pl.dp_tiles;
    p.split = pl.split;
    p.num_units = pl.dp_tiles + (p.num_tiles - pl.dp_tiles) * pl.split;
    p.partials = partials;
    p.wait_limit_ns = wait_limit_ns;
    p.debug_stall = debug_stall;
    p.vec_c = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0 && a.ldc % 4 == 0) ? 1 : 0;
    p.alpha = a.ep.alpha;
    p.beta = a.ep.beta;
    p.bias = a.ep.bias;
    p.ep_simple = a.ep.simple() ? 1 : 0;
    p.tma_c = 0;
    return p;
}

// Tensor map over C for the TMA-store epilogue (32 x 32 boxes, 128-byte
// swizzle). Used when C's base and rows are 16-byte aligned and beta = 0;
// otherwise the epilogue stores from registers and `map` stays unused.
void encode_c(EncodeTiledFn enc, CUtensorMap* map, const GemmArgs& a, TcParams& p) {
    memset(map, 0, sizeof(*map));
    if (p.vec_c && a.ep.beta == 0.0f && a.M > 0 && a.N > 0 &&
        encode_2d(enc, map, a.C, 4, a.M, a.N, a.ldc, 32, 32))
        p.tma_c = 1;
}

cudaError_t launch_reduce(const TcParams& p, cudaStream_t s) {
    const int rows = p.tile_rows < p.M ? p.tile_rows : p.M;
    const long units = (long)(p.num_tiles - p.dp_tiles) * rows * (p.tile_cols / 4);
    long blocks = (units + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    tc_splitk_reduce<<<(int)blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

template <int ESZ, bool B_KMAJOR>
cudaError_t launch_tc(const GemmArgs& a, const TcPlan& pl, float* partials, int num_sms,
                      EncodeTiledFn enc, unsigned long long wait_limit_ns, int debug_stall,
                      cudaStream_t s) {
    constexpr int BK = Kind<ESZ>::BK;
    CUtensorMap tmA, tmB;
    if (!encode_2d(enc, &tmA, a.A, ESZ, a.M, a.K, a.lda, BK, BM)) return cudaErrorInvalidValue;
    const bool okb = B_KMAJOR ? encode_2d(enc, &tmB, a.B, ESZ, a.N, a.K, a.ldb, BK, BN)
                              : encode_2d(enc, &tmB, a.B, ESZ, a.K, a.N, a.ldb, SW / ESZ, BK);
    if (!okb) return cudaErrorInvalidValue;
    TcParams p = make_params(a, pl, partials, wait_limit_ns, debug_stall);
    CUtensorMap tmC;
    encode_c(enc, &tmC, a, p);

    auto kern = tc_gemm_kernel<ESZ, B_KMAJOR>;
    cudaError_t e = set_smem_limit_once<tc_gemm_kernel<ESZ, B_KMAJOR>>(SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int grid = p.num_units < num_sms ? p.num_units : num_sms;
    kern<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(tmA, tmB, tmC, p);
    e = cudaGetLastError();
    if (e != cudaSuccess || p.split <= 1) return e;
    return launch_reduce(p, s);
}

// The 2-SM kernel: clusters of two CTAs, one CTA per SM, persistent over
// 256 x 256 tiles (NW = 1) or 256 x 512 tiles (NW = 2).
template <int ESZ, bool B_KMAJOR, bool X3 = false, int NW = 1>
cudaError_t launch_tc_pair(const GemmArgs& a, const TcPlan& pl, float* partials, int num_sms,
                           EncodeTiledFn enc, unsigned long long wait_limit_ns, int debug_stall,
                           cudaStream_t s) {
    constexpr int BK = Kind<ESZ>::BK;
    constexpr int SMEM = pair_smem_bytes<X3, NW>();
    CUtensorMap tmA, tmB, tmA2, tmB2;
    if (!encode_2d(enc, &tmA, a.A, ESZ, a.M, a.K, a.lda, BK, 128)) return cudaErrorInvalidValue;
    const bool okb = B_KMAJOR ? encode_2d(enc, &tmB, a.B, ESZ, a.N, a.K, a.ldb, BK, 128)
                              : encode_2d(enc, &tmB, a.B, ESZ, a.K, a.N, a.ldb, SW / ESZ, BK);
    if (!okb) return cudaErrorInvalidValue;
    if constexpr (X3) {
        if (!encode_2d(enc, &tmA2, a.A2, ESZ, a.M, a.K, a.lda, BK, 128) ||
            !encode_2d(enc, &tmB2, a.B2, ESZ, a.N, a.K, a.ldb, BK, 128))
            return cudaErrorInvalidValue;
    } else {
        tmA2 = tmA;
        tmB2 = tmB;
    }
    TcParams p = make_params(a, pl, partials, wait_limit_ns, debug_stall);
    CUtensorMap tmC;
    encode_c(enc, &tmC, a, p);

    auto kern = tc_gemm_2sm_kernel<ESZ, B_KMAJOR, X3, NW>;
    cudaError_t e = set_smem_limit_once<tc_gemm_2sm_kernel<ESZ, B_KMAJOR, X3, NW>>(SMEM);
    if (e != cudaSuccess) return e;
    const int pairs = p.num_units < num_sms / 2 ? p.num_units : num_sms / 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(PairEpi<NW>::THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmA2, tmB2, tmC, p);
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e != cudaSuccess || p.split <= 1) return e;
    return launch_reduce(p, s);
}

// ===================================================================
// Dense MMA rate of the tensor cores (a diagnostic, not part of the
// product): every block -- or SM pair -- issues `iters` MMAs back to back
// from one resident shared-memory stage (zeros: the values do not change the
// rate) into one tensor-memory accumulator, and records the SM clock cycles
// from the first issue to the completion of the last. One SM: 128 x 256
// MMAs (cta_group::1); pair: 256 x 256 (cta_group::2, the leader issues).
template <int ESZ, bool PAIR>
__global__ void __launch_bounds__(128, 1)
tc_peak_kernel(long iters, unsigned long long wait_limit_ns, long long* cycles) {
    using KD = Kind<ESZ>;
    constexpr int K_STEPS = KD::BK / KD::UMMA_K;
    constexpr uint32_t K_STEP_BYTES = KD::UMMA_K * ESZ;
    constexpr int A_BYTES = 128 * SW;                    // 128 rows, one 128-byte K block
    constexpr int B_BYTES = (PAIR ? 128 : BN) * SW;      // this CTA's rows of B (K-major)
    constexpr uint32_t IDESC = instr_desc<ESZ, true, PAIR ? P_BM : BM>();
    constexpr uint32_t COLS = BN;                        // one 128 x 256 FP32 accumulator
    struct PeakSync {
        uint64_t done;
        uint32_t tmem_base;
        int abort;
    };
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    PeakSync* sy = reinterpret_cast<PeakSync*>(smem + A_BYTES + B_BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool issuer = warp == 0 && lane == 0 && (!PAIR || cluster_rank() == 0);

    uint4* z = reinterpret_cast<uint4*>(smem);
    for (int i = threadIdx.x; i < (A_BYTES + B_BYTES) / 16; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // zeros visible to the MMA
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&sy->done), 1);
        sy->abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        if constexpr (PAIR) {
            asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                         :: "r"(smem_u32(&sy->tmem_base)), "n"(COLS) : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
        } else {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                         :: "r"(smem_u32(&sy->tmem_base)), "n"(COLS) : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        }
    }
    tc_fence_before();
    if constexpr (PAIR) cluster_sync_all(); else __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sy->tmem_base;

    if (issuer) {
        const uint32_t a = smem_u32(smem), b = a + A_BYTES;
        const long long t0 = clock64();
        for (long i = 0; i < iters; ++i) {
            const uint32_t kk = (uint32_t)(i % K_STEPS) * K_STEP_BYTES;
            const uint64_t ad = smem_desc(a + kk, 16, 1024);
            const uint64_t bd = smem_desc(b + kk, 16, 1024);
            if constexpr (PAIR) tc_mma_pair<ESZ>(tmem_base, ad, bd, IDESC, i > 0 ? 1u : 0u);
            else tc_mma<ESZ>(tmem_base, ad, bd, IDESC, i > 0 ? 1u : 0u);
        }
        if constexpr (PAIR) tc_commit_pair(smem_u32(&sy->done));
        else tc_commit(smem_u32(&sy->done));
        const bool ok = mbar_wait(smem_u32(&sy->done), 0, &sy->abort, wait_limit_ns, false);
        const long long t1 = clock64();
        cycles[PAIR ? blockIdx.x / 2 : blockIdx.x] = ok ? t1 - t0 : -1;
    }
    tc_fence_before();
    if constexpr (PAIR) cluster_sync_all(); else __syncthreads();
    tc_fence_after();
    if (warp == 0) {
        if constexpr (PAIR)
            asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
                         :: "r"(tmem_base), "n"(COLS) : "memory");
        else
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                         :: "r"(tmem_base), "n"(COLS) : "memory");
    }
}

template <int ESZ, bool PAIR>
cudaError_t launch_peak(long iters, int num_sms, unsigned long long wait_ns, long long* cycles,
                        int* units, cudaStream_t s) {
    constexpr int SMEM = 1024 + 128 * SW + (PAIR ? 128 : BN) * SW + 64;
    auto kern = tc_peak_kernel<ESZ, PAIR>;
    cudaError_t e = set_smem_limit_once<tc_peak_kernel<ESZ, PAIR>>(SMEM);
    if (e != cudaSuccess) return e;
    const int blocks = PAIR ? num_sms / 2 * 2 : num_sms;
    *units = PAIR ? blocks / 2 : blocks;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks, 1, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = PAIR ? 2 : 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, iters, wait_ns, cycles);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

const char* kNames[3][3] = {
    {"tc_tf32_128x256x32_s4_persistent", "tc_tf32_2sm_256x256x32_s6_persistent",
     "tc_tf32_2sm_256x512x32_s4_persistent"},
    {"tc_bf16_128x256x64_s4_persistent", "tc_bf16_2sm_256x256x64_s6_persistent",
     "tc_bf16_2sm_256x512x64_s4_persistent"},
    {"tc_tf32x3_2sm_256x256x32_s3_persistent", "tc_tf32x3_2sm_256x256x32_s3_persistent",
     "tc_tf32x3_2sm_256x256x32_s3_persistent"},
};

}  // namespace

// Timing model of one tile on one resident unit (an SM pair, or an SM),
// fitted to measurements on the FFN and square BF16/TF32 shapes:
// the main loop runs at `tflops` per unit and a wide tile's accumulator
// write-out (128 x 512 FP32 per SM, about 6.5 us) is not hidden behind the
// next tile's MMAs; the other shapes overlap it (two accumulators).
struct TileModel {
    double main_us, epi_us;
};

TileModel tile_model(int in_type, int shape, int tile_rows, int tile_cols, int K, bool tma_c) {
    double tflops = shape == TC_ONE_SM ? 9.3 : shape == TC_PAIR ? 22.8 : 30.0;   // BF16
    if (in_type != TC_BF16) tflops *= 0.5;                                      // TF32 rate
    if (in_type == TC_TF32X3) tflops /= 3.0;                                    // three products
    TileModel m;
    m.main_us = 2.0 * tile_rows * tile_cols * (double)K / (tflops * 1e6);
    // The wide tiles' single accumulator leaves part of each epilogue exposed:
    // ~6.5 us with TMA stores, more with per-thread stores when C's rows are
    // not 16-byte aligned (8192 x 14336 x 4096 BF16 with ldc = 14337: wide
    // 660 us against narrow 603; fitted together with 4096^3 TF32 and BF16,
    // where the two shapes come within 3 %).
    m.epi_us = shape == TC_PAIR_WIDE ? (tma_c ? 6.5 : 12.0) : 0.0;
    return m;
}

TcPlan tc_plan(int M, int N, int K, int in_type, int shape, int num_sms, bool allow_split,
               bool tma_c) {
    if (in_type == TC_TF32X3) shape = TC_PAIR;   // the split form: 256 x 256 CTA-pair tiles only
    const bool pair = shape != TC_ONE_SM;
    TcPlan pl;
    pl.tile_rows = pair ? P_BM : BM;
    pl.tile_cols = shape == TC_PAIR_WIDE ? 2 * BN : BN;
    pl.tiles_m = (M + pl.tile_rows - 1) / pl.tile_rows;
    pl.tiles_n = (N + pl.tile_cols - 1) / pl.tile_cols;
    const int bk = in_type == TC_BF16 ? Kind<2>::BK : Kind<4>::BK;
    pl.kblocks = (K + bk - 1) / bk;
    const int tiles = pl.tiles_m * pl.tiles_n;
    const int slots = pair ? num_sms / 2 : num_sms;
    const TileModel tm = tile_model(in_type, shape, pl.tile_rows, pl.tile_cols, K, tma_c);
    const double tile_us = tm.main_us + tm.epi_us;
    const double tile_bytes = (double)pl.tile_rows * pl.tile_cols * sizeof(float);
    pl.dp_tiles = tiles;
    pl.split = 1;
    if (allow_split) plan_tail_split(tiles, slots, pl.kblocks, tile_us, tile_bytes, pl.dp_tiles, pl.split);
    pl.scratch_bytes = pl.split > 1 ? (size_t)(tiles - pl.dp_tiles) * pl.split * pl.tile_rows *
                                          pl.tile_cols * sizeof(float)
                                    : 0;
    // Estimated duration: whole-tile rounds, then the rounds of K-pieces (each
    // with its own epilogue) plus the cost of their partial tiles.
    if (slots <= 0 || tiles == 0) {
        pl.est_us = 0.0;
    } else if (pl.split <= 1) {
        pl.est_us = (double)((tiles + slots - 1) / slots) * tile_us;
    } else {
        const int rem = tiles - pl.dp_tiles;
        const int rounds = (rem * pl.split + slots - 1) / slots;
        pl.est_us = (double)(pl.dp_tiles / slots) * tile_us +
                    rounds * (tm.main_us / pl.split + tm.epi_us) +
                    tail_split_cost_us(rem, tile_bytes, pl.split);
    }
    return pl;
}

int tc_shape(int M, int N, int K, int in_type, int mode, int num_sms, bool allow_split,
             bool tma_c) {
    if (in_type == TC_TF32X3) return TC_PAIR;
    if (mode == 0) return TC_ONE_SM;
    if (mode == 1) return TC_PAIR;
    if (mode == 2) return TC_PAIR_WIDE;
    if (M <= BM) return TC_ONE_SM;        // a pair tile is 256 rows tall
    if (N <= BN) return TC_PAIR;
    // The shape the timing model expects to finish first; near-ties go to
    // the narrow tiles, whose epilogue is hidden.
    const TcPlan narrow = tc_plan(M, N, K, in_type, TC_PAIR, num_sms, allow_split, tma_c);
    const TcPlan wide = tc_plan(M, N, K, in_type, TC_PAIR_WIDE, num_sms, allow_split, tma_c);
    return wide.est_us < 0.97 * narrow.est_us ? TC_PAIR_WIDE : TC_PAIR;
}

const char* tc_kernel_name(int in_type, int shape) {
    const int sh = shape < 0 ? 0 : shape > 2 ? 2 : shape;
    return kNames[in_type == TC_BF16 ? 1 : in_type == TC_TF32X3 ? 2 : 0][sh];
}

cudaError_t tc_launch(const GemmArgs& a, int in_type, int b_kmajor, int num_sms, void* encode_fn,
                      unsigned long long wait_limit_ns, int debug_stall, int shape,
                      const TcPlan& pl, float* partials, cudaStream_t s) {
    auto enc = reinterpret_cast<EncodeTiledFn>(encode_fn);
    const unsigned long long w = wait_limit_ns;
    const int st = debug_stall;
    if (in_type == TC_TF32X3)       // always the CTA-pair kernel, B K-major
        return launch_tc_pair<4, true, true>(a, pl, partials, num_sms, enc, w, st, s);
    if ((shape == TC_PAIR_WIDE) != (pl.tile_cols == 2 * BN)) return cudaErrorInvalidValue;
    if (shape == TC_PAIR_WIDE) {
        if (in_type == TC_BF16)
            return b_kmajor ? launch_tc_pair<2, true, false, 2>(a, pl, partials, num_sms, enc, w, st, s)
                            : launch_tc_pair<2, false, false, 2>(a, pl, partials, num_sms, enc, w, st, s);
        if (!b_kmajor) return cudaErrorInvalidValue;    // TF32 reads B K-major only
        return launch_tc_pair<4, true, false, 2>(a, pl, partials, num_sms, enc, w, st, s);
    }
    if (shape == TC_PAIR) {
        if (in_type == TC_BF16)
            return b_kmajor ? launch_tc_pair<2, true>(a, pl, partials, num_sms, enc, w, st, s)
                            : launch_tc_pair<2, false>(a, pl, partials, num_sms, enc, w, st, s);
        return b_kmajor ? launch_tc_pair<4, true>(a, pl, partials, num_sms, enc, w, st, s)
                        : launch_tc_pair<4, false>(a, pl, partials, num_sms, enc, w, st, s);
    }
    if (in_type == TC_BF16)
        return b_kmajor ? launch_tc<2, true>(a, pl, partials, num_sms, enc, w, st, s)
                        : launch_tc<2, false>(a, pl, partials, num_sms, enc, w, st, s);
    return b_kmajor ? launch_tc<4, true>(a, pl, partials, num_sms, enc, w, st, s)
                    : launch_tc<4, false>(a, pl, partials, num_sms, enc, w, st, s);
}

cudaError_t tc_peak(int in_type, bool pair, long iters, int num_sms, unsigned long long wait_ns,
                    long long* cycles, int* units, cudaStream_t s) {
    if (in_type == TC_BF16)
        return pair ? launch_peak<2, true>(iters, num_sms, wait_ns, cycles, units, s)
                    : launch_peak<2, false>(iters, num_sms, wait_ns, cycles, units, s);
    return pair ? launch_peak<4, true>(iters, num_sms, wait_ns, cycles, units, s)
                : launch_peak<4, false>(iters, num_sms, wait_ns, cycles, units, s);
}

double tc_peak_flop_per_mma(int in_type, bool pair) {
    const int uk = in_type == TC_BF16 ? Kind<2>::UMMA_K : Kind<4>::UMMA_K;
    return 2.0 * (pair ? P_BM : BM) * BN * uk;
}

cudaError_t tc_read_and_clear_status(int* status, cudaStream_t s) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_tc_status, sizeof(int), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_tc_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return e;
        e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return e;
    }
    *status = v;
    return cudaSuccess;
}

}  // namespace tgemm
