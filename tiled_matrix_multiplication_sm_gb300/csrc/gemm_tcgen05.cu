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
// Operand layouts in shared memory: A (M x K, K contiguous) is K-major. B
// (K x N, N contiguous) is read MN-major through the instruction
// descriptor's transpose bit, so neither operand is copied: BF16 in the
// 128-byte swizzle, TF32 in the 128-byte swizzle with 32-byte atoms (with
// the plain 128-byte swizzle the TF32 kind produced zeros on sm_103a). A B
// stored transposed (N x K, K contiguous) is read K-major like A.
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

// The one-SM kernel's ring holds STAGES stages of 128 x 256 tiles (192 KB);
// with 128 x 128 tiles the same bytes hold more, shallower stages.
constexpr int ONE_SM_RING = STAGES * STAGE_BYTES;
constexpr int ONE_SM_MAX_STAGES = 6;
struct Sync {
    uint64_t full[ONE_SM_MAX_STAGES];
    uint64_t empty[ONE_SM_MAX_STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Epilogue staging: EPI_BUFS 32 x 32 FP32 blocks per epilogue warp (TMA
// stores of C). The one-SM and 256 x 256 kernels give each warp a larger
// region, EPI_REGION bytes (a multiple of 1 KB, so that the swizzled block
// at its start stays aligned to its swizzle pattern), which also holds the
// 32 row slots of 36 floats (144 bytes) of the row-copy epilogue.
constexpr int EPI_BUFS = 1;
constexpr int EPI_WARP_BYTES = EPI_BUFS * 32 * 32 * 4;
constexpr int ROW_SLOT_FLOATS = 36;
constexpr int EPI_REGION = 5 * 1024;
static_assert(32 * ROW_SLOT_FLOATS * 4 <= EPI_REGION && EPI_WARP_BYTES <= EPI_REGION,
              "epilogue region");
constexpr int EPI_STAGE_BYTES = 4 * EPI_REGION;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_STAGE_BYTES + (int)sizeof(Sync);
static_assert(SMEM_BYTES <= 227 * 1024, "one-SM kernel exceeds the shared memory of a block");

struct TcParams {
    int M, N, K;
    float* C;
    long ldc;
    int tiles_m, tiles_n, num_tiles, kblocks;
    int tile_rows;       // rows of a tile: 128 (one SM) or 256 (SM pair)
    int tile_cols;       // columns of a tile: 256, or 512 (wide SM-pair tiles)
    int num_slots;       // resident work units: SMs (one-SM kernel) or SM pairs
    int dp_tiles;        // tiles [0, dp_tiles) are computed whole, round robin over the slots
    // Stream-K tail: the K blocks of tiles [dp_tiles, num_tiles), in (tile, K
    // block) order, are shared evenly by slots [0, sk_slots); 0 = the tail
    // tiles are computed whole too.
    int sk_slots;
    long long sk_total;  // (num_tiles - dp_tiles) * kblocks
    // The split form of the tail (sk_split = 1): sk_slots is a multiple of
    // the tail's tile count, so each tile's K blocks are sk_slots / tiles
    // shares of consecutive slots; every share leaves its raw partial tile and
    // nothing waits -- a separate reduction kernel sums each tile's shares
    // in K order and stores it (no chain of hand-offs; sk_flags unused).
    int sk_split;
    float* partials;     // sk_slots partial tiles (tile_rows x tile_cols), one per slot
    unsigned* sk_flags;  // one arrival counter per tail tile, zero at launch
    int sk_arrivals;     // arrivals of one contribution (the epilogue warps of a slot)
    unsigned long long wait_limit_ns;
    int debug_stall;
    int vec_c;
    // Output rule C = alpha * acc + beta * C_old + bias[col]; ep_simple when
    // it is the plain product.
    float alpha, beta;
    const float* bias;
    int ep_simple;
    int tma_c;           // whole tiles leave through TMA stores (plain rule, 16-byte rows of C)
    int row_copy;        // C not stored by TMA but beta = 0: the row-copy epilogue
    // A read by the SIMT loader warps (rows only 4-byte aligned): base, row
    // pitch in bytes, element size.
    const void* a_ptr;
    long lda_bytes;
    int a_esz;
    // B read MN-major: columns [0, b3d_cols) are also described by a 3-D
    // tensor map (128-byte column chunks as its third dimension), so that a
    // tile's chunks arrive in one copy; 0 = no such map.
    int b3d_cols;
};

// One output under the rule (C_old read only when beta != 0).
__device__ __forceinline__ float apply_epilogue(float acc, const TcParams& p, const float* c_old,
                                                int col) {
    float v = p.alpha * acc;
    if (p.beta != 0.0f) v = fmaf(p.beta, *c_old, v);
    if (p.bias != nullptr) v += p.bias[col];
    return v;
}

// A unit of persistent work: K blocks [kb0, kb1) of one tile.
//   piece < 0:  the result goes to C -- a whole tile, or the owner's segment
//               of a tail tile;
//   piece >= 0: a contributor's segment of a tail tile: its sum goes to the
//               partial tile of slot `piece`, and the tile's counter is
//               raised once it has landed.
// fix_wait > 0: the slots before this one that share the tile (fix_wait of
// them) have contributed; the last of them, slot fix_slot, left the sum of
// all their K blocks in its partial tile (each contributor adds its
// predecessor's partial before publishing), so this unit waits until the
// counter shows all fix_wait contributions and adds that one partial tile.
struct Unit {
    int tile, kb0, kb1;
    int piece;
    int fix_slot, fix_wait;
};

// The K-block range [b, e) of the tail that slot `slot` computes.
__device__ __forceinline__ void sk_range(const TcParams& p, int slot, long long& b, long long& e) {
    b = (long long)slot * p.sk_total / p.sk_slots;
    e = (long long)(slot + 1) * p.sk_total / p.sk_slots;
}

// The slot whose tail range holds flat tail index x (0 <= x < sk_total).
__device__ __forceinline__ int sk_slot_of(const TcParams& p, long long x) {
    return (int)(((x + 1) * p.sk_slots - 1) / p.sk_total);
}

// Units of slot `slot`: its whole tiles (slot, slot + num_slots, ...), then,
// with a stream-K tail, its tail range split at a tile boundary. A range is
// never longer than one tile, so it meets at most two tiles: the end of
// tile t0 (the slot holds that tile's last K block, so it owns t0) and the
// start of tile t0 + 1 (a contribution). The contribution runs first, so the
// owners that wait on it -- always slots of higher index -- find it early.
__device__ __forceinline__ int slot_unit_count(const TcParams& p, int slot) {
    if (p.sk_slots == 0)
        return slot < p.num_tiles ? (p.num_tiles - 1 - slot) / p.num_slots + 1 : 0;
    int n = p.dp_tiles / p.num_slots;
    if (slot < p.sk_slots) {
        long long b, e;
        sk_range(p, slot, b, e);
        if (e > b) n += (b / p.kblocks == (e - 1) / p.kblocks) ? 1 : 2;
    }
    return n;
}

__device__ __forceinline__ Unit slot_unit(const TcParams& p, int slot, int i) {
    Unit w;
    w.piece = -1;
    w.fix_slot = -1;
    w.fix_wait = 0;
    const int ndp = p.sk_slots == 0 ? 1 << 30 : p.dp_tiles / p.num_slots;
    if (i < ndp) {
        w.tile = slot + i * p.num_slots;
        w.kb0 = 0;
        w.kb1 = p.kblocks;
        return w;
    }
    const long long KB = p.kblocks;
    long long b, e;
    sk_range(p, slot, b, e);
    const long long t0 = b / KB, t1 = (e - 1) / KB;
    long long t, s0, s1;
    if (t1 != t0 && i == ndp) {          // the start of tile t1: a contribution
        t = t1;
        s0 = 0;
        s1 = e - t1 * KB;
    } else {                              // the end of t0, or a range inside one tile
        t = t0;
        s0 = b - t0 * KB;
        s1 = (t1 != t0) ? KB : e - t0 * KB;
    }
    w.tile = p.dp_tiles + (int)t;
    w.kb0 = (int)s0;
    w.kb1 = (int)s1;
    if (p.sk_split) {                            // every share a piece; nothing waits
        w.piece = slot;
        return w;
    }
    if (s1 != KB) w.piece = slot;               // not the tile's end: a contribution
    const int first = sk_slot_of(p, t * KB);     // the slot holding the tile's first K block
    if (slot > first) {
        w.fix_slot = slot - 1;
        w.fix_wait = slot - first;
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

// As mbar_try, acquiring at cluster scope: for barriers that threads of the
// peer CTA arrive on with release.cluster semantics.
__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Wait until the phase of `bar` with parity `parity` has completed. Gives up
// (returns false) when the block's abort flag is raised or, if
// `honour_abort` is false, only when `limit_ns` has passed; a wait that runs
// out raises the abort flag and records the timeout.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* abort_flag,
                                       unsigned long long limit_ns, bool honour_abort,
                                       bool cluster_acquire = false) {
    auto test = [&]() { return cluster_acquire ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity); };
    if (test()) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (test()) return true;
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

// A 3-D box: B's column chunks (x: column in the chunk, y: K row, z: chunk).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
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

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 int z, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
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

// Shared-memory matrix descriptor (tcgen05 format: start address, leading
// and stride byte offsets in 16-byte units, version 1, layout type): layout
// 2 is the 128-byte swizzle, layout 1 the 128-byte swizzle with 32-byte atoms.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout = 2) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFF) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= 1ull << 46;                     // descriptor version for tcgen05
    d |= (uint64_t)layout << 61;
    return d;
}

// Descriptor of B read MN-major: chunks of 128-byte rows (SW / ESZ columns
// each, one row per K) `chunk_bytes` apart along N. BF16 takes the 128-byte
// swizzle, rows grouped by 8 (1024 bytes); TF32 takes the 128-byte swizzle
// with 32-byte atoms (the tensor map's SWIZZLE_128B_ATOM_32B: each row's four
// 32-byte pieces permuted by the row index mod 4), rows grouped by 4 (512
// bytes). The TF32 form was measured on this GPU: a 128 x 64 x 32 integer
// product through it is exact, and the other offset choices are not.
template <int ESZ>
__device__ __forceinline__ uint64_t b_mn_desc(uint32_t addr, uint32_t chunk_bytes) {
    return ESZ == 4 ? smem_desc(addr, chunk_bytes, 512, 1) : smem_desc(addr, chunk_bytes, 1024, 2);
}

// Instruction descriptor: FP32 accumulator, A K-major, B K-major or
// MN-major, M x N.
template <int ESZ, bool B_KMAJOR, int MMA_M = BM, int MMA_N = BN>
__host__ __device__ constexpr uint32_t instr_desc() {
    return (1u << 4)                         // D format F32
         | (Kind<ESZ>::FMT << 7)             // A format
         | (Kind<ESZ>::FMT << 10)            // B format
         | (0u << 15)                        // A: K-major
         | ((B_KMAJOR ? 0u : 1u) << 16)      // B: K-major (0) or MN-major (1)
         | ((uint32_t)(MMA_N >> 3) << 17)
         | ((uint32_t)(MMA_M >> 4) << 24);
}

__device__ __forceinline__ void tile_coords(int t, const TcParams& p, int& mb, int& nb) {
    const int per_group = GROUP_M * p.tiles_n;
    const int first_m = (t / per_group) * GROUP_M;
    const int gm = min(p.tiles_m - first_m, GROUP_M);
    mb = first_m + (t % per_group) % gm;
    nb = (t % per_group) / gm;
}

// ---- SIMT loader for A whose rows are only 4-byte aligned
//
// TMA copies need rows that start on 16-byte boundaries. For A without them
// (fp32 with any lda, bf16 with an even lda) A_LOADER_WARPS extra warps copy
// each CTA's 128 rows of a K block (128 bytes a row) straight from the
// caller's A with 4-byte cp.async -- lane l moves word l of a row -- into the
// same 128-byte-swizzled K-major layout a TMA copy writes (16-byte chunk j of
// row r at j ^ (r % 8)), zero-filling words past K and rows past M. Each warp
// commits one group per stage and, A_LOADER_LAG stages later, waits for it,
// fences its writes into the async proxy (the tensor core reads them) and
// arrives on the stage's full barrier, which also counts the TMA bytes of B.
constexpr int A_LOADER_WARPS = 2;
constexpr int A_LOADER_LAG = 2;       // the wide tiles' (4-stage ring whose MMA holds stages)
// Stages in flight per loader warp for a ring of NSTAGES whose MMA frees
// each stage as it consumes it: all but two.
template <int NSTAGES>
__host__ __device__ constexpr int loader_lag() { return NSTAGES - 2 > 1 ? NSTAGES - 2 : 1; }

// This warp's 64 rows (from row r0 of the CTA's 128) of K block kb.
__device__ __forceinline__ void a_loader_stage(uint32_t a_dst, const TcParams& p, int row_first,
                                               int r0, int kb) {
    const int lane = threadIdx.x & 31;
    const long kbyte = (long)kb * SW + lane * 4;              // this word's byte within a row
    const long row_bytes = (long)p.K * p.a_esz;
    const int sz = kbyte + 4 <= row_bytes ? 4 : (kbyte < row_bytes ? (int)(row_bytes - kbyte) : 0);
    const char* a = static_cast<const char*>(p.a_ptr);
    const uint32_t col = (uint32_t)(lane & 3) * 4;
    const uint32_t chunk = (uint32_t)lane >> 2;
#pragma unroll 8
    for (int r = r0; r < r0 + 64; ++r) {
        const int grow = row_first + r;
        const int n = grow < p.M ? sz : 0;
        const char* src = n ? a + (long)grow * p.lda_bytes + kbyte : a;
        const uint32_t dst = a_dst + (uint32_t)r * SW + ((chunk ^ (uint32_t)(r & 7)) << 4) + col;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" :: "r"(dst), "l"(src), "r"(n)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Signal stage s loaded (this warp's part): one arrival on the full barrier
// at `full0` + 8 s -- a shared::cta address (CLUSTER false) or, for the
// leader's barrier in a CTA pair, a shared::cluster address.
template <bool CLUSTER>
__device__ __forceinline__ void a_loader_signal(uint32_t full0, int s) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        const uint32_t bar = full0 + (uint32_t)(s * sizeof(uint64_t));
        if constexpr (CLUSTER) mbar_arrive_cluster(bar); else mbar_arrive(bar);
    }
}

// The loop of one loader warp (index lw) over the units of `slot`, in the
// producer's stage order. `rank_rows` is the CTA's first row within a tile.
template <int NSTAGES, bool CLUSTER, int LAG>
__device__ __forceinline__ void a_loader_loop(const TcParams& p, int slot, int lw, uint32_t a_base,
                                              uint32_t a_stage_bytes, uint64_t* empty,
                                              uint32_t full0, int rank_rows, int* abort_flag,
                                              unsigned long long lim) {
    const int lane = threadIdx.x & 31;
    int g = 0;
    const int nu = slot_unit_count(p, slot);
    for (int i = 0; i < nu; ++i) {
        const Unit w = slot_unit(p, slot, i);
        int mb, nb;
        tile_coords(w.tile, p, mb, nb);
        const int row_first = mb * p.tile_rows + rank_rows;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++g) {
            const int s = g % NSTAGES;
            const uint32_t ph = (uint32_t)(g / NSTAGES) & 1u;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(smem_u32(&empty[s]), ph ^ 1u, abort_flag, lim, true) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) goto loader_done;
            if (p.debug_stall && g == 0)
                asm volatile("cp.async.commit_group;" ::: "memory");   // test hook: stage 0 stays empty
            else
                a_loader_stage(a_base + (uint32_t)s * a_stage_bytes, p, row_first, lw * 64, kb);
            if (g >= LAG) {
                asm volatile("cp.async.wait_group %0;" :: "n"(LAG) : "memory");
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                const int gd = g - LAG;
                if (!(p.debug_stall && gd == 0)) a_loader_signal<CLUSTER>(full0, gd % NSTAGES);
            }
        }
    }
loader_done:
    // The stages still in flight (also after an abort, so that the
    // producer's drain of its own copies can complete).
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    for (int gd = g > LAG ? g - LAG : 0; gd < g; ++gd)
        if (!(p.debug_stall && gd == 0)) a_loader_signal<CLUSTER>(full0, gd % NSTAGES);
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

// ---- stream-K hand-off between slots (global memory)

// A contributor warp's arrival on its tile's counter, once every lane's
// stores of the partial tile are visible device-wide: each lane fences its
// own stores, then one lane arrives. All lanes of the warp call this.
__device__ __forceinline__ void sk_arrive(unsigned* flag) {
    __threadfence();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) atomicAdd(flag, 1u);
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* f) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}

// Wait (lane 0 of the warp polls; bounded) until the counter reaches
// `target`. A wait that runs out raises the block's abort flag and records
// the timeout. Returns the same value in every lane.
__device__ __noinline__ bool sk_wait(const unsigned* flag, unsigned target, int* abort_flag,
                                     unsigned long long limit_ns) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) {
        if (ld_acquire(flag) < target) {
            const unsigned long long t0 = globaltimer();
            for (uint32_t it = 1;; ++it) {
                if (ld_acquire(flag) >= target) break;
                if ((it & 15u) == 0) {
                    if (*(volatile int*)abort_flag) { ok = 0; break; }
                    if (globaltimer() - t0 > limit_ns || it >= (1u << 30)) {
                        *(volatile int*)abort_flag = 1;
                        atomicCAS(&g_tc_status, 0, kStatusTimeout);
                        ok = 0;
                        break;
                    }
                }
                __nanosleep(it < 64 ? 64 : 512);    // back off: many warps poll at once
            }
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) (void)ld_acquire(flag);          // every lane orders its loads after the counter
    return ok != 0;
}

// Partial tiles are kept as 32 x 32 blocks, each block column-major (4 KB:
// column j of the block is 32 consecutive floats, one per row), blocks in
// (slot, 32-row band, 32-column block) order. A warp then reads column j of
// a block -- one value for each of its 32 rows -- as one coalesced 128-byte
// load.
__device__ __forceinline__ long partial_block(const TcParams& p, int slot, int row_in_tile, int c) {
    return ((long)slot * (p.tile_rows / 32) + row_in_tile / 32) * (p.tile_cols / 32) + c;
}

// Start loading (coalesced, 32 independent loads) the values of this
// thread's row in column block c of the partial tile of slot `slot`.
__device__ __forceinline__ void load_partial(const TcParams& p, int slot, int row_in_tile, int c,
                                             float (&v)[32]) {
    const float* src = p.partials + partial_block(p, slot, row_in_tile, c) * 1024 + (threadIdx.x & 31);
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __ldcg(src + 32 * j);
}

__device__ __forceinline__ void add_to(uint32_t (&r)[32], const float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__fadd_rn(__uint_as_float(r[j]), v[j]));
}

// Bulk copy of `bytes` (a multiple of 16) from this thread's shared memory
// at `ssrc` to global memory at `gdst`, both 16-byte aligned.
__device__ __forceinline__ void bulk_store_row(float* gdst, uint32_t ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(gdst), "r"(ssrc), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Position q of a row-copy slot holds value q - a of the current block, or,
// for q < a, value 32 + q - a of the previous block (the carry c29..c31).
template <int Q>
__device__ __forceinline__ float slot_value(const uint32_t (&v)[32], float c29, float c30, float c31,
                                            int a) {
    auto at = [&](int i) -> float {
        return i >= 32 ? 0.0f : i >= 0 ? __uint_as_float(v[i]) : i == -1 ? c31 : i == -2 ? c30 : c29;
    };
    const float lo = (a & 1) ? at(Q - 1) : at(Q);
    const float hi = (a & 1) ? at(Q - 3) : at(Q - 2);
    return (a & 2) ? hi : lo;
}

template <int K>
__device__ __forceinline__ void write_slot_chunks(float4* slot, const uint32_t (&v)[32], float c29,
                                                  float c30, float c31, int a) {
    if constexpr (K < ROW_SLOT_FLOATS / 4) {
        slot[K] = make_float4(slot_value<4 * K>(v, c29, c30, c31, a),
                              slot_value<4 * K + 1>(v, c29, c30, c31, a),
                              slot_value<4 * K + 2>(v, c29, c30, c31, a),
                              slot_value<4 * K + 3>(v, c29, c30, c31, a));
        write_slot_chunks<K + 1>(slot, v, c29, c30, c31, a);
    }
}

// Row-copy epilogue for C that TMA cannot store (rows not 16-byte aligned,
// or N not a multiple of 4), beta = 0.
// Each lane owns one row of the warp's 32. The row's values in global
// memory start `a` floats past a 16-byte boundary (the same for every
// 32-column block, as 32 floats are 128 bytes), so each block, together
// with the last `a` values of the block before it (carried in registers),
// covers whole 16-byte chunks: the lane writes them, shifted by `a`, to its
// 144-byte slot in shared memory and one bulk copy moves them to C. Only
// the values before the first 16-byte boundary of the warp's column range,
// and after the last one (or past N), are stored one by one. This replaces
// 16-byte stores from registers whose 32 lanes hit 32 rows at once.
__device__ __forceinline__ void store_rows_copy(const TcParams& p, const Unit& w, int nb,
                                                int row, int row_in_tile, uint32_t taddr,
                                                float* stage, int c_begin, int c_end) {
    const int lane = threadIdx.x & 31;
    const bool live = row < p.M;
    float* crow = p.C + (long)row * p.ldc;
    const int a = (int)((reinterpret_cast<uintptr_t>(crow) >> 2) & 3);
    float4* slot = reinterpret_cast<float4*>(stage + lane * ROW_SLOT_FLOATS);
    const uint32_t slot_s = smem_u32(slot);
    float c29 = 0.0f, c30 = 0.0f, c31 = 0.0f;
    const bool fix = w.fix_wait > 0 && live;
    float pv[32];                                      // the partial tile's block c (fix)
    if (fix && nb * p.tile_cols + c_begin * 32 < p.N) load_partial(p, w.fix_slot, row_in_tile, c_begin, pv);
    for (int c = c_begin; c < c_end; ++c) {
        const int col0 = nb * p.tile_cols + c * 32;
        if (col0 >= p.N) break;                        // uniform across the warp
        uint32_t v[32];
        tmem_ld32(taddr + (uint32_t)(c * 32), v);
        const int nvalid = p.N - col0 < 32 ? p.N - col0 : 32;
        const bool first = c == c_begin;
        const bool last = c + 1 == c_end || col0 + 32 >= p.N;
        if (fix) {
            add_to(v, pv);
            if (!last) load_partial(p, w.fix_slot, row_in_tile, c + 1, pv);   // in flight
        }
        if (!p.ep_simple) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + j < p.N)
                    v[j] = __float_as_uint(apply_epilogue(__uint_as_float(v[j]), p, nullptr, col0 + j));
        }
        // Slot positions [4 klo, 4 khi) -- values [cs, ce) of this block --
        // leave in one copy; position q is column col0 - a + q.
        const int lo = first ? a : 0, hi = a + nvalid;
        const int klo = (lo + 3) >> 2, khi = hi >> 2;
        const int cs = 4 * klo - a;
        const int ce = khi > klo ? 4 * khi - a : cs;
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");   // the slot is free
        write_slot_chunks<0>(slot, v, c29, c30, c31, a);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        float* g0 = crow + col0 - a;                   // 16-byte aligned: position 0
        if (live && khi > klo)
            bulk_store_row(g0 + 4 * klo, slot_s + 16u * (uint32_t)klo, 16u * (uint32_t)(khi - klo));
        if (live) {
            if (!first && khi <= klo) {
                // No whole chunk at N: the values carried from the block
                // before (columns col0 - a .. col0 - 1) one by one.
#pragma unroll
                for (int q = 0; q < 3; ++q)
                    if (q < a) {
                        const int i = 32 - a + q;
                        crow[col0 - a + q] = i == 29 ? c29 : i == 30 ? c30 : c31;
                    }
            }
            if (nvalid == 32) {
                if (first) {
#pragma unroll
                    for (int j = 0; j < 3; ++j)
                        if (j < cs) crow[col0 + j] = __uint_as_float(v[j]);
                }
                if (last) {
#pragma unroll
                    for (int j = 29; j < 32; ++j)
                        if (j >= ce) crow[col0 + j] = __uint_as_float(v[j]);
                }
            } else {                                    // the block at N: the rest one by one
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < nvalid && ((first && j < cs) || j >= ce))
                        crow[col0 + j] = __uint_as_float(v[j]);
            }
        }
        c29 = __uint_as_float(v[29]);
        c30 = __uint_as_float(v[30]);
        c31 = __uint_as_float(v[31]);
    }
}

// Epilogue of one unit for this thread's accumulator row `row_in_tile`:
// the 32-column blocks [c_begin, c_end) of the tile from TMEM (the tile's
// column 0 at address `taddr`) to C -- after the contributors' partial
// tiles are added, for an owner -- or, for a contribution, to the partial
// tile of its slot. Rows past M and columns past N are skipped (no owner
// reads them). All lanes of the warp call this together.
//
// Contributions go to their slot's partial tile with coalesced stores from
// registers. Results for C whose rows are 16-byte aligned (beta = 0) leave
// through TMA stores of 32 x 32 blocks staged in shared memory. Otherwise
// each thread stores its row's 32-column blocks
// with 16-byte stores, after peeling the values before the first 16-byte
// boundary when C's rows are not 16-byte aligned. (Staging each 32 x 32
// block through shared memory to store it as 32 coalesced row segments
// instead measured 9 % slower on 3072 x 5120 x 1536 TF32 with ldc = 5121:
// the staging's shared-memory traffic competes with the MMAs' operand
// reads.)
// ROWS: the kernel's epilogue region holds row slots (p.row_copy may be set).
template <bool ROWS>
__device__ __forceinline__ void store_accumulator(const TcParams& p, const Unit& w, int mb, int nb,
                                                 int row_in_tile, uint32_t taddr, float* stage,
                                                 const CUtensorMap* tmC, int c_begin, int c_end) {
    const int row = mb * p.tile_rows + row_in_tile;
    const int lane = threadIdx.x & 31;
    if (w.piece >= 0) {
        // A contribution: each 32 x 32 block (after adding the predecessor's
        // running sum) goes to the slot's partial tile as 32 coalesced
        // 128-byte rows of the column-major block, straight from registers.
        // Warps whose rows all lie past M store nothing (no one reads them).
        if (row - lane >= p.M) return;
        const int n_blocks = (p.N - nb * p.tile_cols + 31) / 32;
        const int c_stop = c_end < n_blocks ? c_end : n_blocks;
        const bool fix = w.fix_wait > 0;
        uint32_t r[32];
        float pv[32];
        for (int c = c_begin; c < c_stop; ++c) {
            tmem_ld32(taddr + (uint32_t)(c * 32), r);
            if (fix) {               // a contribution in the middle of a tile (rare): no prefetch
                load_partial(p, w.fix_slot, row_in_tile, c, pv);
                add_to(r, pv);
            }
            float* dst = p.partials + partial_block(p, w.piece, row_in_tile, c) * 1024 + lane;
#pragma unroll
            for (int j = 0; j < 32; ++j) __stcg(dst + 32 * j, __uint_as_float(r[j]));
        }
        return;
    }
    if (p.tma_c) {
        // alpha and bias are applied in registers, then each 32 x 32 block
        // goes to the warp's staging buffer (EPI_BUFS of them) in the
        // 128-byte-swizzled layout of C's tensor map (row i holds 128 bytes,
        // 16-byte chunk j at j ^ (i % 8)) and leaves as one TMA store, which
        // also clips rows and columns past M and N. A buffer is reused once
        // the store issued EPI_BUFS blocks earlier has read it. Without a
        // running sum to add, the next block's TMEM load is in flight while a
        // block is staged; with one, the next block's partial values are.
        const int row0 = row - lane;
        if (row0 >= p.M) return;                        // the warp's rows are all past M
        const int n_blocks = (p.N - nb * p.tile_cols + 31) / 32;   // blocks with columns < N
        const int c_stop = c_end < n_blocks ? c_end : n_blocks;
        if (c_begin >= c_stop) return;
        auto stage_and_store = [&](uint32_t (&r)[32], int c) {
            const int col0 = nb * p.tile_cols + c * 32;
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
                srow[j ^ (lane & 7)] =
                    make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) tma_store_2d(tmC, col0, row0, smem_u32(buf));
        };
        uint32_t r[32];
        if (w.fix_wait > 0) {
            float pv[32];
            load_partial(p, w.fix_slot, row_in_tile, c_begin, pv);
            for (int c = c_begin; c < c_stop; ++c) {
                tmem_ld32(taddr + (uint32_t)(c * 32), r);
                add_to(r, pv);
                if (c + 1 < c_stop) load_partial(p, w.fix_slot, row_in_tile, c + 1, pv);
                stage_and_store(r, c);
            }
            return;
        }
        uint32_t nx[32];
        tmem_ld32(taddr + (uint32_t)(c_begin * 32), r);
        for (int c = c_begin; c < c_stop; ++c) {
            const bool more = c + 1 < c_stop;
            if (more) tmem_ld32_async(taddr + (uint32_t)((c + 1) * 32), nx);
            stage_and_store(r, c);
            if (more) {
                tmem_wait_ld(nx);
#pragma unroll
                for (int j = 0; j < 32; ++j) r[j] = nx[j];
            }
        }
        return;
    }
    if constexpr (ROWS) {
        if (p.row_copy) {
            store_rows_copy(p, w, nb, row, row_in_tile, taddr, stage, c_begin, c_end);
            return;
        }
    }
    float* dst = p.C + (long)row * p.ldc + (long)nb * p.tile_cols;
    const bool vec = p.vec_c != 0;
    const bool ep = p.ep_simple == 0;
    const bool fix = w.fix_wait > 0 && row < p.M;
    float pv[32];                                      // the partial tile's block c (fix)
    if (fix && nb * p.tile_cols + c_begin * 32 < p.N) load_partial(p, w.fix_slot, row_in_tile, c_begin, pv);
    for (int c = c_begin; c < c_end; ++c) {
        const int col0 = nb * p.tile_cols + c * 32;
        if (col0 >= p.N) break;                     // uniform across the warp
        uint32_t r[32];
        tmem_ld32(taddr + (uint32_t)(c * 32), r);
        if (row < p.M) {
            if (fix) {
                add_to(r, pv);
                if (c + 1 < c_end && col0 + 32 < p.N)
                    load_partial(p, w.fix_slot, row_in_tile, c + 1, pv);   // in flight
            }
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

// B_KMAJOR: B arrives transposed (N x K, K contiguous) and is read K-major;
// otherwise B is K x N (N contiguous) and is read MN-major.
// A_LOADER: A is read by the SIMT loader warps (warps 6..), not by TMA.
// TBN: tile columns (= MMA N), 256, or 128 for products whose 128 x 256
// tiles would leave SMs idle (the same ring bytes then hold 6 stages).
template <int ESZ, bool B_KMAJOR, bool A_LOADER = false, int TBN = BN>
__global__ void __launch_bounds__(NUM_THREADS + (A_LOADER ? 32 * A_LOADER_WARPS : 0), 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
               const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmB3,
               const __grid_constant__ CUtensorMap tmC,
               const TcParams p) {
    using KD = Kind<ESZ>;
    constexpr int BK = KD::BK;
    constexpr int K_STEPS = BK / KD::UMMA_K;
    constexpr int B_CHUNK_COLS = SW / ESZ;               // N columns per swizzled row
    constexpr int B_CHUNKS = TBN / B_CHUNK_COLS;
    constexpr int B_CHUNK_BYTES = BK * SW;
    constexpr int B_STG = BK * TBN * ESZ;                // B bytes of a stage
    constexpr int NST = ONE_SM_RING / (A_STAGE_BYTES + B_STG);
    constexpr int STAGES = NST;                          // ring depth of this tile width
    constexpr int TMEM_COLS = 2 * TBN;                   // two accumulators
    constexpr uint32_t A_K_STEP = KD::UMMA_K * ESZ;      // bytes along a K-major row
    static_assert(B_CHUNKS * B_CHUNK_BYTES == B_STG, "B stage size");
    // B read MN-major arrives in groups of RG_ROWS K rows, each group one
    // copy of all the tile's column chunks ([group][chunk][row]): a BF16
    // stage (64 K rows) is two copies, so the two halves of a row's bytes
    // are requested 32 rows apart rather than 64 (16 x 14336 x 4096 BF16:
    // 33.4 against 35.5 us; TF32, 32 K rows a stage, is one group).
    constexpr int RG_ROWS = 32;
    constexpr int RG_GROUPS = BK / RG_ROWS;
    constexpr uint32_t RG_CHUNK = RG_ROWS * SW;          // one chunk's rows of one group
    constexpr uint32_t RG_STEP = B_CHUNKS * RG_CHUNK;    // all chunks of one group
    static_assert(BK % RG_ROWS == 0 && RG_ROWS % KD::UMMA_K == 0 && RG_STEP * RG_GROUPS == B_STG,
                  "row groups");
    static_assert(NST <= ONE_SM_MAX_STAGES && NST * (A_STAGE_BYTES + B_STG) <= ONE_SM_RING, "ring");
    static_assert(!A_LOADER || TBN == BN, "the SIMT A loader runs with 128 x 256 tiles");
    constexpr uint32_t IDESC = instr_desc<ESZ, B_KMAJOR, BM, TBN>();
    constexpr int B_STAGE_BYTES = B_STG;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    float* epi_stage = reinterpret_cast<float*>(smem + ONE_SM_RING);
    Sync* sy = reinterpret_cast<Sync*>(smem + ONE_SM_RING + EPI_STAGE_BYTES);
    const uint32_t a_base = smem_u32(smem);
    const uint32_t b_base = a_base + STAGES * A_STAGE_BYTES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // The producer's arrival (with the TMA bytes), and each loader warp's.
            mbar_init(smem_u32(&sy->full[s]), 1 + (A_LOADER ? A_LOADER_WARPS : 0));
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
        if (!A_LOADER)
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
    // Set-up done (shared memory, barriers, tensor memory): let the next
    // kernel launch, then wait for the previous one before touching memory.
    pdl_launch_dependents();
    pdl_wait();
    const unsigned long long lim = p.wait_limit_ns;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t armed = 0, armed_parity = 0;   // per-stage fills in flight
            int g = 0;
            const int nu = slot_unit_count(p, blockIdx.x);
            for (int i = 0; i < nu; ++i) {
                const Unit w = slot_unit(p, blockIdx.x, i);
                int mb, nb;
                tile_coords(w.tile, p, mb, nb);
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++g) {
                    const int s = g % STAGES;
                    const uint32_t ph = (uint32_t)(g / STAGES) & 1u;
                    if (!mbar_wait(smem_u32(&sy->empty[s]), ph ^ 1u, &sy->abort, lim, true)) goto producer_done;
                    if (p.debug_stall && g == 0) continue;     // test hook: never fill stage 0
                    const uint32_t full = smem_u32(&sy->full[s]);
                    mbar_arrive_expect_tx(full, A_LOADER ? B_STAGE_BYTES : A_STAGE_BYTES + B_STAGE_BYTES);
                    if constexpr (!A_LOADER)
                        tma_load_2d(a_base + s * A_STAGE_BYTES, &tmA, kb * BK, mb * BM, full);
                    const uint32_t bdst = b_base + s * B_STAGE_BYTES;
                    if constexpr (B_KMAJOR) {
                        tma_load_2d(bdst, &tmB, kb * BK, nb * TBN, full);
                    } else if ((nb + 1) * TBN <= p.b3d_cols) {
#pragma unroll
                        for (int gq = 0; gq < RG_GROUPS; ++gq)
                            tma_load_3d(bdst + gq * RG_STEP, &tmB3, 0, kb * BK + gq * RG_ROWS,
                                        nb * B_CHUNKS, full);
                    } else {
#pragma unroll
                        for (int gq = 0; gq < RG_GROUPS; ++gq)
#pragma unroll
                            for (int c = 0; c < B_CHUNKS; ++c)
                                tma_load_2d(bdst + gq * RG_STEP + c * RG_CHUNK, &tmB,
                                            nb * TBN + c * B_CHUNK_COLS, kb * BK + gq * RG_ROWS, full);
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
            int g = 0;
            const int nu = slot_unit_count(p, blockIdx.x);
            for (int it = 0; it < nu; ++it) {
                const Unit w = slot_unit(p, blockIdx.x, it);
                const int acc = it & 1;
                const uint32_t aph = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait(smem_u32(&sy->tmem_empty[acc]), aph ^ 1u, &sy->abort, lim, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * TBN);
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
                                     : b_mn_desc<ESZ>(b_addr + (kk * KD::UMMA_K / RG_ROWS) * RG_STEP +
                                                          (kk * KD::UMMA_K % RG_ROWS) * SW,
                                                      RG_CHUNK);
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
    } else if (warp >= 6) {
        // ------------------------------------------------ A loader (warps 6..)
        if constexpr (A_LOADER)
            a_loader_loop<STAGES, false, loader_lag<STAGES>()>(p, blockIdx.x, warp - 6, a_base,
                                                             A_STAGE_BYTES, sy->empty,
                                         smem_u32(&sy->full[0]), 0, &sy->abort, lim);
    } else {
        // ------------------------------------------------ epilogue (warps 2-5)
        const int q = warp & 3;                 // TMEM lanes 32q .. 32q+31
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        const int nu = slot_unit_count(p, blockIdx.x);
        for (int it = 0; it < nu; ++it) {
            const Unit w = slot_unit(p, blockIdx.x, it);
            int mb, nb;
            tile_coords(w.tile, p, mb, nb);
            const int acc = it & 1;
            const uint32_t aph = (uint32_t)(it >> 1) & 1u;
            bool ok = mbar_wait(smem_u32(&sy->tmem_full[acc]), aph, &sy->abort, lim, true);
            if (!__all_sync(0xffffffffu, ok)) break;
            unsigned* flag = (p.sk_flags != nullptr && (w.fix_wait > 0 || w.piece >= 0))
                                 ? p.sk_flags + (w.tile - p.dp_tiles)
                                                              : nullptr;
            // The earlier shares of this tile must have landed before their
            // running sum is added.
            if (w.fix_wait > 0 &&
                !sk_wait(flag, (unsigned)(w.fix_wait * p.sk_arrivals), &sy->abort, lim))
                break;
            tc_fence_after();
            store_accumulator<true>(p, w, mb, nb, q * 32 + lane, tmem_base + lane_off + (uint32_t)(acc * TBN),
                              epi_stage + q * (EPI_REGION / 4), &tmC, 0, TBN / 32);
            tc_fence_before();
            __syncwarp();                               // the warp's TMEM reads are done
            if (lane == 31) mbar_arrive(smem_u32(&sy->tmem_empty[acc]));   // not the storing lane
            if (w.piece >= 0 && flag != nullptr) sk_arrive(flag);   // this warp's part has landed
        }
        tma_store_wait_all();    // every lane's C stores and row copies done before the block retires
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
// TF32 with B as the caller stores it (K x N, N contiguous), transposed in
// shared memory to be read K-major (tensor-core mode 3 only). It was built
// for products with few rows before the TF32 kind's MN-major read (the
// 128-byte swizzle with 32-byte atoms) was found; the one-SM kernel reading
// B MN-major now serves them faster. TMA lands each stage's 32 x 128
// block of B in the stage's own B slot in the MN-major layout it has in
// memory (boxes of 32 columns x 32 K rows, 128-byte swizzle) next to the
// stage's A block; both land on the stage's `landed` barrier. Two transposer
// warps then read the B block into registers (4 bytes a lane, one 128-byte
// row per warp instruction: no bank conflicts), meet at a named barrier, and
// write it back in place in the K-major 128-byte-swizzled layout (one
// 16-byte chunk a lane, eight rows per quarter-warp: no bank conflicts),
// fence the writes into the async proxy and arrive on the stage's `full`
// barrier, which the MMA issuer waits on. Tiles are 128 x 128 (a 32 x 128
// TF32 block is 16 KB: 64 floats a transposer thread), six stages of 32 KB;
// the rest -- MMA issue, two accumulators, epilogue, stream-K tail -- is the
// one-SM kernel's.
constexpr int TT_BN = 128;                         // tile columns
constexpr int TT_STAGES = 6;
constexpr int TT_B_STAGE = 32 * TT_BN * 4;         // 32 K rows x 128 columns, fp32: 16 KB
constexpr int TT_STAGE = A_STAGE_BYTES + TT_B_STAGE;
constexpr int TT_TMEM_COLS = 2 * TT_BN;            // two accumulators
constexpr int TT_THREADS = NUM_THREADS + 64;       // + two transposer warps
struct SyncT {
    uint64_t full[TT_STAGES];                      // B transposed (both transposer warps)
    uint64_t landed[TT_STAGES];                    // A and B (MN-major) landed
    uint64_t empty[TT_STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};
constexpr int TT_SMEM_BYTES = 1024 + TT_STAGES * TT_STAGE + EPI_STAGE_BYTES + (int)sizeof(SyncT);
static_assert(TT_SMEM_BYTES <= 227 * 1024, "TF32 transposing kernel exceeds the shared memory of a block");

// True on every thread of the two transposer warps (named barrier 1, 64
// threads) if `pred` holds on any of them.
__device__ __forceinline__ bool transposers_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 64, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"((uint32_t)pred) : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(TT_THREADS, 1)
tc_gemm_tf32t_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC,
                     const TcParams p) {
    constexpr int BK = Kind<4>::BK;                // 32
    constexpr int K_STEPS = BK / Kind<4>::UMMA_K;  // 4
    constexpr uint32_t K_STEP = Kind<4>::UMMA_K * 4;
    constexpr uint32_t IDESC = instr_desc<4, true, BM, TT_BN>();
    constexpr int B_BOXES = TT_BN / 32;            // MN-major boxes of 32 columns
    constexpr int B_BOX_BYTES = BK * SW;           // 32 K rows x 128 bytes

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
    float* epi_stage = reinterpret_cast<float*>(smem + TT_STAGES * TT_STAGE);
    SyncT* sy = reinterpret_cast<SyncT*>(smem + TT_STAGES * TT_STAGE + EPI_STAGE_BYTES);
    const uint32_t a_base = smem_u32(smem);
    const uint32_t b_base = a_base + TT_STAGES * A_STAGE_BYTES;
    float* b_gen = reinterpret_cast<float*>(smem + TT_STAGES * A_STAGE_BYTES);   // generic view

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < TT_STAGES; ++s) {
            mbar_init(smem_u32(&sy->full[s]), 2);            // the transposer warps
            mbar_init(smem_u32(&sy->landed[s]), 1);          // producer, with the TMA bytes
            mbar_init(smem_u32(&sy->empty[s]), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&sy->tmem_full[a]), 1);
            mbar_init(smem_u32(&sy->tmem_empty[a]), 4);
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
                     :: "r"(smem_u32(&sy->tmem_base)), "n"(TT_TMEM_COLS) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sy->tmem_base;
    // Set-up done (shared memory, barriers, tensor memory): let the next
    // kernel launch, then wait for the previous one before touching memory.
    pdl_launch_dependents();
    pdl_wait();
    const unsigned long long lim = p.wait_limit_ns;
    const int nu = slot_unit_count(p, blockIdx.x);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t armed = 0, armed_parity = 0;
            int g = 0;
            for (int i = 0; i < nu; ++i) {
                const Unit w = slot_unit(p, blockIdx.x, i);
                int mb, nb;
                tile_coords(w.tile, p, mb, nb);
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++g) {
                    const int s = g % TT_STAGES;
                    const uint32_t ph = (uint32_t)(g / TT_STAGES) & 1u;
                    if (!mbar_wait(smem_u32(&sy->empty[s]), ph ^ 1u, &sy->abort, lim, true)) goto tt_producer_done;
                    if (p.debug_stall && g == 0) continue;     // test hook: never fill stage 0
                    const uint32_t landed = smem_u32(&sy->landed[s]);
                    mbar_arrive_expect_tx(landed, TT_STAGE);
                    tma_load_2d(a_base + s * A_STAGE_BYTES, &tmA, kb * BK, mb * BM, landed);
#pragma unroll
                    for (int c = 0; c < B_BOXES; ++c)
                        tma_load_2d(b_base + s * TT_B_STAGE + c * B_BOX_BYTES, &tmB,
                                    nb * TT_BN + c * 32, kb * BK, landed);
                    armed |= 1u << s;
                    armed_parity = (armed_parity & ~(1u << s)) | (ph << s);
                }
            }
        tt_producer_done:
            // Copies still in flight must land before the block may exit.
            for (int s = 0; s < TT_STAGES; ++s)
                if (armed & (1u << s))
                    mbar_wait(smem_u32(&sy->landed[s]), (armed_parity >> s) & 1u, &sy->abort, lim, false);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int g = 0;
            for (int it = 0; it < nu; ++it) {
                const Unit w = slot_unit(p, blockIdx.x, it);
                const int acc = it & 1;
                const uint32_t aph = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait(smem_u32(&sy->tmem_empty[acc]), aph ^ 1u, &sy->abort, lim, true)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * TT_BN);
                bool ok = true;
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++g) {
                    const int s = g % TT_STAGES;
                    const uint32_t ph = (uint32_t)(g / TT_STAGES) & 1u;
                    if (!mbar_wait(smem_u32(&sy->full[s]), ph, &sy->abort, lim, true)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = a_base + s * A_STAGE_BYTES;
                    const uint32_t b_addr = b_base + s * TT_B_STAGE;
#pragma unroll
                    for (int kk = 0; kk < K_STEPS; ++kk)
                        tc_mma<4>(d_tmem, smem_desc(a_addr + kk * K_STEP, 16, 1024),
                                  smem_desc(b_addr + kk * K_STEP, 16, 1024), IDESC,
                                  (kb != w.kb0 || kk != 0) ? 1u : 0u);
                    tc_commit(smem_u32(&sy->empty[s]));
                }
                if (!ok) break;
                tc_commit(smem_u32(&sy->tmem_full[acc]));
            }
            tc_commit(smem_u32(&sy->drain));
            mbar_wait(smem_u32(&sy->drain), 0, &sy->abort, lim, false);
        }
        __syncwarp();
    } else if (warp >= 6) {
        // ------------------------------------------------ B transposers (warps 6-7)
        // Thread t owns columns n = t and t + 64 of the tile (all 32 K rows).
        const int t = threadIdx.x - 6 * 32;
        int g = 0;
        for (int i = 0; i < nu; ++i) {
            const Unit w = slot_unit(p, blockIdx.x, i);
            for (int kb = w.kb0; kb < w.kb1; ++kb, ++g) {
                const int s = g % TT_STAGES;
                const uint32_t ph = (uint32_t)(g / TT_STAGES) & 1u;
                int ok = 1;
                if (lane == 0) ok = mbar_wait(smem_u32(&sy->landed[s]), ph, &sy->abort, lim, true) ? 1 : 0;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                // Both warps leave together (they meet at named barriers): a
                // reduction over the 64 threads decides.
                if (transposers_any(!ok || *(volatile int*)&sy->abort)) goto tt_transpose_done;
                float* bs = b_gen + s * (TT_B_STAGE / 4);
                float v[2][32];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int n = t + 64 * h;
                    // MN-major: box n / 32, row k, 16-byte chunk ((n % 32) / 4) ^ (k % 8).
                    const float* box = bs + (n >> 5) * (B_BOX_BYTES / 4) + (n & 3);
                    const int cn = (n & 31) >> 2;
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[h][k] = box[k * 32 + ((cn ^ (k & 7)) << 2)];
                }
                asm volatile("bar.sync 1, 64;" ::: "memory");       // every read done
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int n = t + 64 * h;
                    // K-major: row n (128 bytes), 16-byte chunk c at c ^ (n % 8).
                    float4* row = reinterpret_cast<float4*>(bs + n * 32);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        row[c ^ (n & 7)] = make_float4(v[h][4 * c], v[h][4 * c + 1], v[h][4 * c + 2],
                                                      v[h][4 * c + 3]);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sy->full[s]));
            }
        }
    tt_transpose_done:;
    } else {
        // ------------------------------------------------ epilogue (warps 2-5)
        const int q = warp & 3;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        for (int it = 0; it < nu; ++it) {
            const Unit w = slot_unit(p, blockIdx.x, it);
            int mb, nb;
            tile_coords(w.tile, p, mb, nb);
            const int acc = it & 1;
            const uint32_t aph = (uint32_t)(it >> 1) & 1u;
            bool ok = mbar_wait(smem_u32(&sy->tmem_full[acc]), aph, &sy->abort, lim, true);
            if (!__all_sync(0xffffffffu, ok)) break;
            unsigned* flag = (p.sk_flags != nullptr && (w.fix_wait > 0 || w.piece >= 0))
                                 ? p.sk_flags + (w.tile - p.dp_tiles)
                                                              : nullptr;
            if (w.fix_wait > 0 &&
                !sk_wait(flag, (unsigned)(w.fix_wait * p.sk_arrivals), &sy->abort, lim))
                break;
            tc_fence_after();
            store_accumulator<true>(p, w, mb, nb, q * 32 + lane,
                                    tmem_base + lane_off + (uint32_t)(acc * TT_BN),
                                    epi_stage + q * (EPI_REGION / 4), &tmC, 0, TT_BN / 32);
            tc_fence_before();
            __syncwarp();
            if (lane == 31) mbar_arrive(smem_u32(&sy->tmem_empty[acc]));
            if (w.piece >= 0 && flag != nullptr) sk_arrive(flag);
        }
        tma_store_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                     :: "r"(tmem_base), "n"(TT_TMEM_COLS) : "memory");
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
    static constexpr int REGION = NW == 2 ? EPI_WARP_BYTES : EPI_REGION;   // per warp
    static constexpr int BYTES = WARPS * REGION > P_GUARD_BYTES ? WARPS * REGION : P_GUARD_BYTES;
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
// A_LOADER: A is read by the SIMT loader warps (after the epilogue warps),
// not by TMA; each CTA loads its own 128 rows.
template <int ESZ, bool B_KMAJOR, bool X3, int NW, bool A_LOADER = false>
__global__ void __launch_bounds__(PairEpi<NW>::THREADS + (A_LOADER ? 32 * A_LOADER_WARPS : 0), 1)
tc_gemm_2sm_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB2,
                   const __grid_constant__ CUtensorMap tmC,
                   const TcParams p) {
    using R = PairRing<X3, NW>;
    static_assert(!X3 || (ESZ == 4 && B_KMAJOR), "the split form is TF32 with B K-major");
    static_assert(NW == 1 || (NW == 2 && !X3), "wide tiles are for the one-product forms");
    static_assert(!(A_LOADER && X3), "the split form reads its own aligned copies of A");
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
    const int pair = blockIdx.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < R::STAGES; ++s) {
            // The leader producer's arrival (with both CTAs' TMA bytes), and
            // each loader warp's of both CTAs.
            mbar_init(smem_u32(&sy->full[s]), 1 + (A_LOADER ? 2 * A_LOADER_WARPS : 0));
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
    // Set-up done (shared memory, barriers, tensor memory): let the next
    // kernel launch, then wait for the previous one before touching memory.
    pdl_launch_dependents();
    pdl_wait();
    const unsigned long long lim = p.wait_limit_ns;
    // The leader's copies of the shared hand-off barriers, as cluster addresses.
    const uint32_t full0 = map_to_rank(smem_u32(&sy->full[0]), 0);
    const uint32_t tmem_empty0 = map_to_rank(smem_u32(&sy->tmem_empty[0]), 0);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            uint32_t armed = 0, armed_parity = 0;
            int g = 0;
            const int nu = slot_unit_count(p, pair);
            for (int i = 0; i < nu; ++i) {
                const Unit w = slot_unit(p, pair, i);
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
                    if (leader)
                        mbar_arrive_expect_tx(smem_u32(&sy->full[s]), 2 * (A_LOADER ? R::B_STAGE : R::STAGE));
                    const uint32_t adst = a_base + s * R::A_STAGE;
                    if constexpr (!A_LOADER) tma_load_2d_pair(adst, &tmA, kb * BK, row0, full);
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
                            } else if (ch + 128 <= p.b3d_cols) {   // the 3-D map (in tmB2)
                                tma_load_3d_pair(bh, &tmB2, 0, kb * BK, ch / B_CHUNK_COLS, full);
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
            // Stages the wide tiles' MMA issuer waits for before it frees one.
            // The loader warps signal a stage only A_LOADER_LAG stages after
            // they issued it (which needs a freed stage), so with them the
            // issuer may hold no more than STAGES - A_LOADER_LAG.
            constexpr int HOLD = A_LOADER ? R::STAGES - A_LOADER_LAG : R::STAGES;
            static_assert(HOLD >= 1, "stages to hold");
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
                                         : b_mn_desc<ESZ>(bh + kk * B_K_STEP, B_CHUNK_BYTES);
                            tc_mma_pair<ESZ>(d_tmem + (uint32_t)(h * BN), ad, bdh, IDESC, first);
                        }
                    }
                }
            };
            const int nu = slot_unit_count(p, pair);
            for (; it < nu; ++it) {
                const Unit w = slot_unit(p, pair, it);
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
                    const int held = min(HOLD, w.kb1 - w.kb0);
                    for (int i = 0; i < held; ++i) {
                        const int s = (g + i) % R::STAGES;
                        const uint32_t ph = (uint32_t)((g + i) / R::STAGES) & 1u;
                        if (!mbar_wait(smem_u32(&sy->full[s]), ph, &sy->abort, lim, true, A_LOADER)) { ok = false; break; }
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
                const int tail = NW == 2 ? min(HOLD, w.kb1 - kb) : 0;
                for (; ok && kb < w.kb1 - tail; ++kb, ++g) {
                    const int s = g % R::STAGES;
                    const uint32_t ph = (uint32_t)(g / R::STAGES) & 1u;
                    if (!mbar_wait(smem_u32(&sy->full[s]), ph, &sy->abort, lim, true, A_LOADER)) { ok = false; break; }
                    tc_fence_after();
                    issue(s, kb, w, d_tmem, 0, NW);
                    tc_commit_pair_multicast(smem_u32(&sy->empty[s]));   // slot free in both CTAs
                }
                if (!ok) break;
                if constexpr (NW == 2) {
                    for (int i = 0; i < tail; ++i) {
                        const int s = (g + i) % R::STAGES;
                        const uint32_t ph = (uint32_t)((g + i) / R::STAGES) & 1u;
                        if (!mbar_wait(smem_u32(&sy->full[s]), ph, &sy->abort, lim, true, A_LOADER)) { ok = false; break; }
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
    } else if (warp >= 2 + PairEpi<NW>::WARPS) {
        // ------------------------------------------------ A loader (both CTAs)
        if constexpr (A_LOADER)
            a_loader_loop<R::STAGES, true, NW == 2 ? A_LOADER_LAG : loader_lag<R::STAGES>()>(
                p, pair, warp - 2 - PairEpi<NW>::WARPS, a_base, R::A_STAGE, sy->empty, full0,
                (int)rank * 128, &sy->abort, lim);
    } else {
        // ------------------------------------------------ epilogue (warps 2.., both CTAs)
        const int q = warp & 3;                              // TMEM lanes 32q .. 32q+31
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        constexpr int PARTS = PairEpi<NW>::WARPS / 4;      // warps sharing a lane quarter
        const int part = (warp - 2) >> 2;
        const int blocks = p.tile_cols / 32 / PARTS;         // 32-column blocks per warp
        const int nu = slot_unit_count(p, pair);
        for (int it = 0; it < nu; ++it) {
            const Unit w = slot_unit(p, pair, it);
            int mb, nb;
            tile_coords(w.tile, p, mb, nb);
            const int acc = it % NACC;
            const uint32_t aph = (uint32_t)(it / NACC) & 1u;
            bool ok = mbar_wait(smem_u32(&sy->tmem_full[acc]), aph, &sy->abort, lim, true);
            if (!__all_sync(0xffffffffu, ok)) break;
            unsigned* flag = (p.sk_flags != nullptr && (w.fix_wait > 0 || w.piece >= 0))
                                 ? p.sk_flags + (w.tile - p.dp_tiles)
                                                              : nullptr;
            // The earlier shares of this tile must have landed before their
            // running sum is added.
            if (w.fix_wait > 0 &&
                !sk_wait(flag, (unsigned)(w.fix_wait * p.sk_arrivals), &sy->abort, lim))
                break;
            tc_fence_after();
            float* stage = reinterpret_cast<float*>(smem + R::STAGES * R::STAGE) +
                           (warp - 2) * (PairEpi<NW>::REGION / 4);
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
                    store_accumulator<false>(p, w, mb, nb, (int)rank * 128 + q * 32 + lane,
                                             tmem_base + lane_off, stage, &tmC, c0, c0 + blocks / 2);
                    tc_fence_before();
                    __syncwarp();                       // the warp's TMEM reads are done
                    // Lane 31 arrives: lane 0 issued the warp's TMA stores,
                    // and its release-ordered arrive was measured ~0.2 us later.
                    if (lane == 31) mbar_arrive_cluster(tmem_empty0 + (uint32_t)(half * sizeof(uint64_t)));
                }
                if (!ok2) break;
            } else {
                store_accumulator<NW == 1>(p, w, mb, nb, (int)rank * 128 + q * 32 + lane,
                                           tmem_base + lane_off + (uint32_t)(acc * BN), stage, &tmC,
                                           part * blocks, (part + 1) * blocks);
                tc_fence_before();
                __syncwarp();                           // the warp's TMEM reads are done
                if (lane == 31) mbar_arrive_cluster(tmem_empty0 + (uint32_t)(acc * sizeof(uint64_t)));
            }
            if (w.piece >= 0 && flag != nullptr) sk_arrive(flag);   // this warp's part has landed
        }
        tma_store_wait_all();    // every lane's C stores and row copies done before the block retires
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
               long cols, long ld, int box_cols, int box_rows,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    const CUtensorMapDataType dt =
        esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * esz};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The same B as a 3-D tensor: x a column within a 128-byte chunk, y the K
// row, z the chunk (whole chunks only: floor(N / chunk columns)), boxes of
// `chunks` chunks. Returns the columns it covers, 0 when it cannot be made.
long encode_b_mn3(EncodeTiledFn enc, CUtensorMap* map, const GemmArgs& a, int esz, int bk,
                  int chunks) {
    const long ch = SW / esz;
    const long nc = a.N / ch;
    if (nc < 1) return 0;
    cuuint64_t dims[3] = {(cuuint64_t)ch, (cuuint64_t)a.K, (cuuint64_t)nc};
    cuuint64_t strides[2] = {(cuuint64_t)a.ldb * esz, (cuuint64_t)SW};
    cuuint32_t box[3] = {(cuuint32_t)ch, (cuuint32_t)bk, (cuuint32_t)chunks};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUresult r = enc(map, dt, 3, const_cast<void*>(a.B), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     esz == 4 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? nc * ch : 0;
}

// B read MN-major (K x N, N contiguous) in boxes of SW / esz columns x BK
// rows, with the swizzle b_mn_desc expects for the element size.
bool encode_b_mn(EncodeTiledFn enc, CUtensorMap* map, const GemmArgs& a, int esz, int bk) {
    return encode_2d(enc, map, a.B, esz, a.K, a.N, a.ldb, SW / esz, bk,
                     esz == 4 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B);
}

TcParams make_params(const GemmArgs& a, const TcPlan& pl, void* scratch, int arrivals,
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
    p.num_slots = pl.slots;
    p.dp_tiles = pl.dp_tiles;
    p.sk_slots = pl.sk_slots;
    p.sk_total = (long long)(p.num_tiles - pl.dp_tiles) * pl.kblocks;
    p.partials = nullptr;
    p.sk_flags = nullptr;
    p.sk_split = pl.sk_split;
    p.b3d_cols = 0;
    if (pl.sk_slots > 0) {
        p.partials = static_cast<float*>(scratch);
        if (!pl.sk_split)
            p.sk_flags = reinterpret_cast<unsigned*>(static_cast<char*>(scratch) + tc_partial_bytes(pl));
    }
    p.sk_arrivals = arrivals;
    p.wait_limit_ns = wait_limit_ns;
    p.debug_stall = debug_stall;
    p.vec_c = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0 && a.ldc % 4 == 0) ? 1 : 0;
    p.alpha = a.ep.alpha;
    p.beta = a.ep.beta;
    p.bias = a.ep.bias;
    p.ep_simple = a.ep.simple() ? 1 : 0;
    p.tma_c = 0;
    p.row_copy = 0;
    p.a_ptr = a.A;
    p.lda_bytes = a.lda * (long)(a.a_esz > 0 ? a.a_esz : 4);
    p.a_esz = a.a_esz > 0 ? a.a_esz : 4;
    return p;
}

// Tensor map over C for the TMA-store epilogue (32 x 32 boxes, 128-byte
// swizzle). Used when C's base and rows are 16-byte aligned, N is a
// multiple of 4 and beta = 0; otherwise the epilogue stores from registers
// (or by row copies) and `map` stays unused. (With N % 4 != 0 a TMA store
// of the last block of a row also wrote the columns up to the next 16-byte
// boundary, past N: measured on sm_103a.)
void encode_c(EncodeTiledFn enc, CUtensorMap* map, const GemmArgs& a, TcParams& p) {
    memset(map, 0, sizeof(*map));
    if (p.vec_c && a.N % 4 == 0 && a.ep.beta == 0.0f && a.M > 0 && a.N > 0 &&
        encode_2d(enc, map, a.C, 4, a.M, a.N, a.ldc, 32, 32))
        p.tma_c = 1;
}

// The split form's reduction: C for the tail tiles from their shares'
// partial tiles. One block per 32 x 32 output block: warp w sums columns
// w, w + 8, w + 16, w + 24 of the block over the tile's shares in K order
// (lane = row: one coalesced 128-byte line per share and column of the
// column-major partial block), the block transposes them through shared
// memory, and warp w stores rows w, w + 8, .. as coalesced row segments of
// C under the output rule.
__global__ void __launch_bounds__(256)
tc_split_reduce_kernel(const TcParams p) {
    pdl_launch_dependents();    // the next kernel may launch now
    pdl_wait();                 // the GEMM kernel's partial tiles are visible
    __shared__ float blk[32][33];
    const int rb_n = p.tile_rows / 32, cb_n = p.tile_cols / 32;
    const int tail_tiles = p.num_tiles - p.dp_tiles;
    const int k = p.sk_slots / tail_tiles;                 // shares per tile
    const int idx = blockIdx.x;
    const int t = idx / (rb_n * cb_n);
    if (t >= tail_tiles) return;
    const int rb = (idx / cb_n) % rb_n, cb = idx % cb_n;
    int mb, nb;
    tile_coords(p.dp_tiles + t, p, mb, nb);
    const int row0 = mb * p.tile_rows + rb * 32, col0 = nb * p.tile_cols + cb * 32;
    if (row0 >= p.M || col0 >= p.N) return;                // uniform over the block
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    // Eight shares' loads in flight before their adds (in K order).
    float sum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int j0 = 0; j0 < k; j0 += 8) {
        float v[8][4];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float* src = p.partials + partial_block(p, t * k + j0 + u, rb * 32, cb) * 1024 + lane;
#pragma unroll
            for (int i = 0; i < 4; ++i) v[u][i] = j0 + u < k ? __ldcg(src + (w + 8 * i) * 32) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (j0 + u < k) sum[i] += v[u][i];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) blk[w + 8 * i][lane] = sum[i];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = w + 8 * i;
        const int grow = row0 + r, gcol = col0 + lane;
        if (grow < p.M && gcol < p.N) {
            float* dst = p.C + (long)grow * p.ldc + gcol;
            const float v = blk[lane][r];
            *dst = p.ep_simple ? v : apply_epilogue(v, p, dst, gcol);
        }
    }
}

// Zero the tail-tile counters of a stream-K plan, in stream order before
// the launch.
bool prepare_stream_k(const TcParams& p, cudaStream_t s) {
    if (p.sk_slots == 0 || p.sk_flags == nullptr) return true;
    return cudaMemsetAsync(p.sk_flags, 0, sizeof(unsigned) * (size_t)(p.num_tiles - p.dp_tiles),
                           s) == cudaSuccess;
}

// The split form's reduction, after the GEMM kernel in stream order.
cudaError_t launch_split_reduce(const TcParams& p, cudaStream_t s) {
    if (!p.sk_split || p.sk_slots == 0) return cudaSuccess;
    const long blocks = (long)(p.num_tiles - p.dp_tiles) * (p.tile_rows / 32) * (p.tile_cols / 32);
    if (blocks <= 0 || blocks > 2147483647L) return cudaErrorInvalidValue;
    return launch_pdl(tc_split_reduce_kernel, dim3((unsigned)blocks), dim3(256), 0, s, p);
}

// Slots (SMs or SM pairs) the grid of plan `pl` needs.
int grid_slots(const TcPlan& pl) {
    const int tiles = pl.tiles_m * pl.tiles_n;
    if (pl.sk_slots == 0) return tiles < pl.slots ? tiles : pl.slots;
    return pl.dp_tiles > 0 ? pl.slots : pl.sk_slots;
}

template <int ESZ, bool B_KMAJOR, bool A_LOADER = false, int TBN = BN>
cudaError_t launch_tc(const GemmArgs& a, const TcPlan& pl, void* scratch, EncodeTiledFn enc,
                      unsigned long long wait_limit_ns, int debug_stall, cudaStream_t s) {
    constexpr int BK = Kind<ESZ>::BK;
    CUtensorMap tmA, tmB;
    memset(&tmA, 0, sizeof(tmA));
    if (pl.tile_cols != TBN) return cudaErrorInvalidValue;
    if (!A_LOADER && !encode_2d(enc, &tmA, a.A, ESZ, a.M, a.K, a.lda, BK, BM))
        return cudaErrorInvalidValue;
    // B read MN-major comes in groups of 32 K rows (see the kernel).
    const bool okb = B_KMAJOR ? encode_2d(enc, &tmB, a.B, ESZ, a.N, a.K, a.ldb, BK, TBN)
                              : encode_b_mn(enc, &tmB, a, ESZ, 32);
    if (!okb) return cudaErrorInvalidValue;
    CUtensorMap tmB3 = tmB;
    TcParams p = make_params(a, pl, scratch, 4, wait_limit_ns, debug_stall);
    if (!B_KMAJOR) p.b3d_cols = (int)encode_b_mn3(enc, &tmB3, a, ESZ, 32, TBN / (SW / ESZ));
    CUtensorMap tmC;
    encode_c(enc, &tmC, a, p);
    p.row_copy = (!p.tma_c && a.ep.beta == 0.0f) ? 1 : 0;
    if (!prepare_stream_k(p, s)) return cudaErrorInvalidValue;

    p.a_esz = ESZ;
    p.lda_bytes = a.lda * (long)ESZ;
    auto kern = tc_gemm_kernel<ESZ, B_KMAJOR, A_LOADER, TBN>;
    cudaError_t e = set_smem_limit_once<tc_gemm_kernel<ESZ, B_KMAJOR, A_LOADER, TBN>>(SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(grid_slots(pl)), dim3(NUM_THREADS + (A_LOADER ? 32 * A_LOADER_WARPS : 0)),
                   SMEM_BYTES, s, tmA, tmB, tmB3, tmC, p);
    return e != cudaSuccess ? e : launch_split_reduce(p, s);
}

// The TF32 kernel that transposes B in shared memory: one CTA per SM,
// persistent over 128 x 128 tiles; B is K x N with 16-byte rows, read by TMA
// in boxes of 32 columns x 32 K rows.
cudaError_t launch_tc_t(const GemmArgs& a, const TcPlan& pl, void* scratch, EncodeTiledFn enc,
                        unsigned long long wait_limit_ns, int debug_stall, cudaStream_t s) {
    constexpr int BK = Kind<4>::BK;
    CUtensorMap tmA, tmB, tmC;
    if (!encode_2d(enc, &tmA, a.A, 4, a.M, a.K, a.lda, BK, BM) ||
        !encode_2d(enc, &tmB, a.B, 4, a.K, a.N, a.ldb, SW / 4, BK))
        return cudaErrorInvalidValue;
    TcParams p = make_params(a, pl, scratch, 4, wait_limit_ns, debug_stall);
    encode_c(enc, &tmC, a, p);
    p.row_copy = (!p.tma_c && a.ep.beta == 0.0f) ? 1 : 0;
    if (!prepare_stream_k(p, s)) return cudaErrorInvalidValue;
    cudaError_t e = set_smem_limit_once<tc_gemm_tf32t_kernel>(TT_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = launch_pdl(tc_gemm_tf32t_kernel, dim3(grid_slots(pl)), dim3(TT_THREADS), TT_SMEM_BYTES, s,
                   tmA, tmB, tmC, p);
    return e != cudaSuccess ? e : launch_split_reduce(p, s);
}

// The 2-SM kernel: clusters of two CTAs, one CTA per SM, persistent over
// 256 x 256 tiles (NW = 1) or 256 x 512 tiles (NW = 2).
template <int ESZ, bool B_KMAJOR, bool X3 = false, int NW = 1, bool A_LOADER = false>
cudaError_t launch_tc_pair(const GemmArgs& a, const TcPlan& pl, void* scratch, EncodeTiledFn enc,
                           unsigned long long wait_limit_ns, int debug_stall, cudaStream_t s) {
    constexpr int BK = Kind<ESZ>::BK;
    constexpr int SMEM = pair_smem_bytes<X3, NW>();
    CUtensorMap tmA, tmB, tmA2, tmB2;
    memset(&tmA, 0, sizeof(tmA));
    if (!A_LOADER && !encode_2d(enc, &tmA, a.A, ESZ, a.M, a.K, a.lda, BK, 128))
        return cudaErrorInvalidValue;
    const bool okb = B_KMAJOR ? encode_2d(enc, &tmB, a.B, ESZ, a.N, a.K, a.ldb, BK, 128)
                              : encode_b_mn(enc, &tmB, a, ESZ, BK);
    if (!okb) return cudaErrorInvalidValue;
    if constexpr (X3) {
        if (!encode_2d(enc, &tmA2, a.A2, ESZ, a.M, a.K, a.lda, BK, 128) ||
            !encode_2d(enc, &tmB2, a.B2, ESZ, a.N, a.K, a.ldb, BK, 128))
            return cudaErrorInvalidValue;
    } else {
        tmA2 = tmA;
        tmB2 = tmB;
    }
    TcParams p = make_params(a, pl, scratch, 2 * PairEpi<NW>::WARPS, wait_limit_ns, debug_stall);
    if (!X3 && !B_KMAJOR)    // the 3-D map of B rides in tmB2 (unused by the one-product forms)
        p.b3d_cols = (int)encode_b_mn3(enc, &tmB2, a, ESZ, BK, 128 / (SW / ESZ));
    CUtensorMap tmC;
    encode_c(enc, &tmC, a, p);
    // The wide tiles' epilogue region has no room for row slots.
    p.row_copy = (NW == 1 && !p.tma_c && a.ep.beta == 0.0f) ? 1 : 0;
    if (!prepare_stream_k(p, s)) return cudaErrorInvalidValue;

    p.a_esz = ESZ;
    p.lda_bytes = a.lda * (long)ESZ;
    auto kern = tc_gemm_2sm_kernel<ESZ, B_KMAJOR, X3, NW, A_LOADER>;
    cudaError_t e = set_smem_limit_once<tc_gemm_2sm_kernel<ESZ, B_KMAJOR, X3, NW, A_LOADER>>(SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * grid_slots(pl), 1, 1);
    cfg.blockDim = dim3(PairEpi<NW>::THREADS + (A_LOADER ? 32 * A_LOADER_WARPS : 0), 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see launch_pdl
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmA2, tmB2, tmC, p);
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    return e != cudaSuccess ? e : launch_split_reduce(p, s);
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
    // Set-up done (shared memory, barriers, tensor memory): let the next
    // kernel launch, then wait for the previous one before touching memory.
    pdl_launch_dependents();
    pdl_wait();

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
    // One row of tiles (b_stream): each tile streams b_bytes of B from
    // memory once, at most sm_rate bytes/us per SM and, all SMs together, at
    // most kStreamRate: measured 47 GB/s per SM for the one-SM kernel with
    // 128 x 256 tiles (32 KB of B a ring stage), 40 GB/s with 128 x 128
    // tiles (16 KB a stage: TF32 16 x 14336 x 4096 on 112 SMs ran 55.9 us
    // whole against 52.4 on 128 x 256 tiles shared by 112 SMs), 26 GB/s for
    // the B-transposing TF32 kernel (in-kernel timestamps), and 5.0-5.2 TB/s
    // for all SMs together (16 x 28672 x 4096 BF16 on 112 SMs: 45.7 us).
    double b_bytes, sm_rate;
    // Main-loop time of `frac` of a tile with n SMs streaming at once.
    double share_us(double frac, int n) const {
        double us = frac * main_us;
        if (b_bytes > 0.0) {
            const double rate = sm_rate < kStreamRate / n ? sm_rate : kStreamRate / n;
            if (frac * b_bytes / rate > us) us = frac * b_bytes / rate;
        }
        return us;
    }
    static constexpr double kStreamRate = 5.0e6;     // bytes per us, all SMs
};

// b_stream: one row of tiles (M <= tile rows), so every tile streams its
// panel of B from memory exactly once; the main loop then takes at least
// the panel's bytes at one SM's share of the rate measured for such reads
// (about 3.3 TB/s over 152 SMs on 16 x 14336 x 4096, TF32 and BF16).
TileModel tile_model(int in_type, int shape, int tile_rows, int tile_cols, int K, bool tma_c,
                     bool b_stream) {
    double tflops = (shape == TC_ONE_SM || shape == TC_ONE_SM_T || shape == TC_ONE_SM_N) ? 9.3
                  : shape == TC_PAIR ? 22.8 : 30.0;                            // BF16
    // TF32: half the BF16 rate, and on the 256 x 256 pair tiles less again --
    // their operand bytes per FLOP double and the shared-memory feed limits
    // them (3072 x 5120 x 1536: ~9.6 TFLOP/s per pair measured on those
    // tiles against ~11 on the 256 x 512 tiles).
    if (in_type != TC_BF16) tflops *= shape == TC_PAIR ? 0.42 : 0.5;
    if (in_type == TC_TF32X3) tflops /= 3.0;                                    // three products
    TileModel m;
    m.main_us = 2.0 * tile_rows * tile_cols * (double)K / (tflops * 1e6);
    m.b_bytes = b_stream ? (double)tile_cols * K * (in_type == TC_BF16 ? 2 : 4) : 0.0;
    m.sm_rate = shape == TC_ONE_SM_T ? 26e3 : shape == TC_ONE_SM_N ? 40e3 : 47e3;
    // The wide tiles' single accumulator leaves part of each epilogue exposed:
    // ~6.5 us with TMA stores, more with per-thread stores when C's rows are
    // not 16-byte aligned (8192 x 14336 x 4096 BF16 with ldc = 14337: wide
    // 660 us against narrow 603; fitted together with 4096^3 TF32 and BF16,
    // where the two shapes come within 3 %).
    m.epi_us = shape == TC_PAIR_WIDE ? (tma_c ? 6.5 : 12.0) : 0.0;
    return m;
}

size_t tc_partial_bytes(const TcPlan& pl) {
    return ((size_t)pl.sk_slots * pl.tile_rows * pl.tile_cols * sizeof(float) + 255) & ~(size_t)255;
}

// Whole-tile rounds over the slots; when the last round is partial and
// `streamk` allows it, its tiles' K blocks may instead be shared by S slots
// (stream-K, S between the tail's tile count and the slot count), each slot
// computing an even share of at most one tile's length. The model charges a
// share its main-loop time, one write-out hand-off per extra share of a tile
// and the zeroing of the counters; S = the one with the lowest estimate, or
// no sharing if that is not faster than the partial round itself.
// streamk: -1 = that choice, 0 = never share, S > 0 = share among S slots
// where the tail allows it (tests and tuning).
TcPlan tc_plan(int M, int N, int K, int in_type, int shape, int num_sms, int streamk,
               bool tma_c) {
    if (in_type == TC_TF32X3) shape = TC_PAIR;   // the split form: 256 x 256 CTA-pair tiles only
    const bool pair = shape == TC_PAIR || shape == TC_PAIR_WIDE;
    TcPlan pl;
    pl.tile_rows = pair ? P_BM : BM;
    pl.tile_cols = shape == TC_PAIR_WIDE ? 2 * BN
                 : (shape == TC_ONE_SM_T || shape == TC_ONE_SM_N) ? TT_BN : BN;
    pl.tiles_m = (M + pl.tile_rows - 1) / pl.tile_rows;
    pl.tiles_n = (N + pl.tile_cols - 1) / pl.tile_cols;
    const int bk = in_type == TC_BF16 ? Kind<2>::BK : Kind<4>::BK;
    pl.kblocks = (K + bk - 1) / bk;
    const int tiles = pl.tiles_m * pl.tiles_n;
    const int slots = pair ? num_sms / 2 : num_sms;
    pl.slots = slots > 0 ? slots : 1;
    pl.dp_tiles = tiles;
    pl.sk_slots = 0;
    pl.sk_split = 0;
    pl.scratch_bytes = 0;
    pl.est_us = 0.0;
    if (slots <= 0 || tiles == 0) return pl;
    const TileModel tm = tile_model(in_type, shape, pl.tile_rows, pl.tile_cols, K, tma_c,
                                    pl.tiles_m == 1);
    // Whole-tile rounds: full ones over all slots, then the partial one.
    const int rem = tiles % slots;
    const int full = tiles / slots;
    const double tile_us = tm.share_us(1.0, slots) + tm.epi_us;
    pl.est_us = full * tile_us + (rem > 0 ? tm.share_us(1.0, rem) + tm.epi_us : 0.0);
    if (streamk == 0 || rem == 0) return pl;
    const long long T = (long long)rem * pl.kblocks;
    // The split form: each tail tile in k equal shares of consecutive slots,
    // summed in K order by a reduction kernel; k <= -streamk when forced.
    auto set_split = [&](int k) {
        pl.dp_tiles = tiles - rem;
        pl.sk_slots = k * rem;
        pl.sk_split = 1;
        pl.scratch_bytes = tc_partial_bytes(pl);
    };
    if (streamk < -1) {
        int k = -streamk;
        if (k * rem > slots) k = slots / rem;
        if (k > pl.kblocks) k = pl.kblocks;
        if (k >= 2) set_split(k);
        return pl;
    }
    if (streamk > 0) {
        // Forced width (tests and tuning), kept where the tail allows it: more
        // slots than tail tiles, every share at least one K block.
        long long S = streamk;
        if (S > slots) S = slots;
        if (S > T) S = T;
        if (S <= rem) return pl;
        pl.dp_tiles = tiles - rem;
        pl.sk_slots = (int)S;
        pl.scratch_bytes = tc_partial_bytes(pl) + (((size_t)rem * sizeof(unsigned) + 255) & ~(size_t)255);
        return pl;
    }
    if (pl.kblocks < 8) return pl;
    // A share ends with its write-out, and the shares of one tile hand their
    // running sum on one after the other, so the tail pays one write-out per
    // extra share of a tile on top of its main loop. Measured per hand-off
    // (in-kernel timestamps): ~8 us for the 256 x 512 tiles (128 x 512 FP32
    // per SM leaving all SMs at once), ~3-4 us for the one-SM tiles; the
    // 256 x 256 pair tiles are charged 8 as well (3000 x 5001 x 1537 TF32
    // with the last round's 12 tiles shared by 24 pairs, one hand-off each:
    // 120.5 us against 117.5 computed whole).
    const double hop_us = pair ? 8.0 : 4.0;
    const double memset_us = 2.0;
    double best = pl.est_us;
    int best_s = 0;
    for (int S = rem + 1; S <= slots && (long long)S * 4 <= T; ++S) {
        const long long len = (T + S - 1) / S;                 // K blocks of the longest share
        const double main_us = tm.share_us((double)len / pl.kblocks, S);
        // Shares meeting one tile: exactly S / rem when the shares divide the
        // tiles evenly, else at most one more than S / rem rounded up.
        const int per_tile = S % rem == 0 ? S / rem : (S + rem - 1) / rem + 1;
        const double est = full * tile_us + main_us + tm.epi_us + (per_tile - 1) * hop_us + memset_us;
        if (est < best && est < 0.98 * pl.est_us) {            // a clear gain only
            best = est;
            best_s = S;
        }
    }
    // The split form, for the pair tiles (whose hand-offs cost most): its
    // shares run side by side and the reduction kernel reads every share's
    // partial tile once (about 5 TB/s) after a launch gap.
    int best_k = 0;
    if (pair && slots / rem >= 2 && pl.kblocks >= 8) {
        const int k = slots / rem < pl.kblocks / 4 ? slots / rem : pl.kblocks / 4;
        if (k >= 2) {
            const double tile_bytes = (double)pl.tile_rows * pl.tile_cols * 4;
            const double reduce_us = 3.0 + (k + 1.0) * rem * tile_bytes / 5e6;
            const long long len = (pl.kblocks + k - 1) / k;
            const double est = full * tile_us + tm.share_us((double)len / pl.kblocks, k * rem) +
                               tm.epi_us + reduce_us;
            if (est < 0.98 * best) {                           // a clear gain over the rest
                best = est;
                best_k = k;
            }
        }
    }
    if (best_k > 0) {
        set_split(best_k);
        pl.est_us = best;
        return pl;
    }
    if (best_s > 0) {
        pl.dp_tiles = tiles - rem;
        pl.sk_slots = best_s;
        pl.est_us = best;
        pl.scratch_bytes = tc_partial_bytes(pl) + (((size_t)rem * sizeof(unsigned) + 255) & ~(size_t)255);
    }
    return pl;
}

int tc_shape(int M, int N, int K, int in_type, int mode, int num_sms, int streamk,
             bool tma_c) {
    if (in_type == TC_TF32X3) return TC_PAIR;
    if (mode == 0) return TC_ONE_SM;
    if (mode == 1) return TC_PAIR;
    if (mode == 2) return TC_PAIR_WIDE;
    if (mode == 4) return TC_ONE_SM_N;
    if (M <= BM) {                        // a pair tile is 256 rows tall (mode 3: as -1)
        // One row of 128 x 256 tiles, or of 128 x 128 tiles, which fill more
        // SMs without sharing tiles (16 x 14336 x 4096 BF16: 112 tiles on
        // 112 SMs, no stream-K hand-off or counter zeroing).
        const TcPlan wide1 = tc_plan(M, N, K, in_type, TC_ONE_SM, num_sms, streamk, tma_c);
        const TcPlan narrow1 = tc_plan(M, N, K, in_type, TC_ONE_SM_N, num_sms, streamk, tma_c);
        return narrow1.est_us < 0.97 * wide1.est_us ? TC_ONE_SM_N : TC_ONE_SM;
    }
    if (N <= BN) return TC_PAIR;
    // The shape the timing model expects to finish first; near-ties go to
    // the narrow tiles, whose epilogue is hidden.
    const TcPlan narrow = tc_plan(M, N, K, in_type, TC_PAIR, num_sms, streamk, tma_c);
    const TcPlan wide = tc_plan(M, N, K, in_type, TC_PAIR_WIDE, num_sms, streamk, tma_c);
    return wide.est_us < 0.97 * narrow.est_us ? TC_PAIR_WIDE : TC_PAIR;
}

const char* tc_kernel_name(int in_type, int shape) {
    if (shape == TC_ONE_SM_T && in_type == TC_TF32) return "tc_tf32_128x128x32_s6_btrans_persistent";
    if (shape == TC_ONE_SM_N && in_type == TC_TF32) return "tc_tf32_128x128x32_s6_persistent";
    if (shape == TC_ONE_SM_N && in_type == TC_BF16) return "tc_bf16_128x128x64_s6_persistent";
    const int sh = shape < 0 ? 0 : shape > 2 ? 2 : shape;
    return kNames[in_type == TC_BF16 ? 1 : in_type == TC_TF32X3 ? 2 : 0][sh];
}

cudaError_t tc_launch(const GemmArgs& a, int in_type, int b_kmajor, void* encode_fn,
                      unsigned long long wait_limit_ns, int debug_stall, int shape,
                      const TcPlan& pl, void* scratch, cudaStream_t s) {
    auto enc = reinterpret_cast<EncodeTiledFn>(encode_fn);
    const unsigned long long w = wait_limit_ns;
    const int st = debug_stall;
    if (pl.sk_slots > 0 && scratch == nullptr) return cudaErrorInvalidValue;
    if (in_type == TC_TF32X3)       // always the CTA-pair kernel, B K-major
        return a.a_loader ? cudaErrorInvalidValue
                          : launch_tc_pair<4, true, true>(a, pl, scratch, enc, w, st, s);
    if (shape == TC_ONE_SM_N) {
        if (a.a_loader || pl.tile_cols != TT_BN || in_type == TC_TF32X3) return cudaErrorInvalidValue;
        if (in_type == TC_BF16)
            return b_kmajor ? launch_tc<2, true, false, TT_BN>(a, pl, scratch, enc, w, st, s)
                            : launch_tc<2, false, false, TT_BN>(a, pl, scratch, enc, w, st, s);
        return b_kmajor ? launch_tc<4, true, false, TT_BN>(a, pl, scratch, enc, w, st, s)
                        : launch_tc<4, false, false, TT_BN>(a, pl, scratch, enc, w, st, s);
    }
    if (shape == TC_ONE_SM_T) {
        if (in_type != TC_TF32 || b_kmajor || a.a_loader || pl.tile_cols != TT_BN)
            return cudaErrorInvalidValue;
        return launch_tc_t(a, pl, scratch, enc, w, st, s);
    }
    if (pl.tile_cols == TT_BN && pl.tile_rows == BM) return cudaErrorInvalidValue;
    if ((shape == TC_PAIR_WIDE) != (pl.tile_cols == 2 * BN)) return cudaErrorInvalidValue;
    if (a.a_loader) {
        // A read by the loader warps: TF32 (B either way) and BF16 with B MN-major.
        if (in_type == TC_BF16 && b_kmajor) return cudaErrorInvalidValue;
        const int form = in_type == TC_BF16 ? 0 : (b_kmajor ? 1 : 2);
        if (shape == TC_PAIR_WIDE)
            return form == 0 ? launch_tc_pair<2, false, false, 2, true>(a, pl, scratch, enc, w, st, s)
                 : form == 1 ? launch_tc_pair<4, true, false, 2, true>(a, pl, scratch, enc, w, st, s)
                             : launch_tc_pair<4, false, false, 2, true>(a, pl, scratch, enc, w, st, s);
        if (shape == TC_PAIR)
            return form == 0 ? launch_tc_pair<2, false, false, 1, true>(a, pl, scratch, enc, w, st, s)
                 : form == 1 ? launch_tc_pair<4, true, false, 1, true>(a, pl, scratch, enc, w, st, s)
                             : launch_tc_pair<4, false, false, 1, true>(a, pl, scratch, enc, w, st, s);
        return form == 0 ? launch_tc<2, false, true>(a, pl, scratch, enc, w, st, s)
             : form == 1 ? launch_tc<4, true, true>(a, pl, scratch, enc, w, st, s)
                         : launch_tc<4, false, true>(a, pl, scratch, enc, w, st, s);
    }
    if (shape == TC_PAIR_WIDE) {
        if (in_type == TC_BF16)
            return b_kmajor ? launch_tc_pair<2, true, false, 2>(a, pl, scratch, enc, w, st, s)
                            : launch_tc_pair<2, false, false, 2>(a, pl, scratch, enc, w, st, s);
        return b_kmajor ? launch_tc_pair<4, true, false, 2>(a, pl, scratch, enc, w, st, s)
                        : launch_tc_pair<4, false, false, 2>(a, pl, scratch, enc, w, st, s);
    }
    if (shape == TC_PAIR) {
        if (in_type == TC_BF16)
            return b_kmajor ? launch_tc_pair<2, true>(a, pl, scratch, enc, w, st, s)
                            : launch_tc_pair<2, false>(a, pl, scratch, enc, w, st, s);
        return b_kmajor ? launch_tc_pair<4, true>(a, pl, scratch, enc, w, st, s)
                        : launch_tc_pair<4, false>(a, pl, scratch, enc, w, st, s);
    }
    if (in_type == TC_BF16)
        return b_kmajor ? launch_tc<2, true>(a, pl, scratch, enc, w, st, s)
                        : launch_tc<2, false>(a, pl, scratch, enc, w, st, s);
    return b_kmajor ? launch_tc<4, true>(a, pl, scratch, enc, w, st, s)
                    : launch_tc<4, false>(a, pl, scratch, enc, w, st, s);
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
