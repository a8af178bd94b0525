// C ABI of libtgemm.so: argument checks, kernel selection and launch.
// The declarations and the contract of every entry point are in
// include/tgemm.h.

#include "../../include/tgemm.h"
#include "tgemm_internal.h"

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

namespace {

constexpr int kMaxDevices = 64;
constexpr int kCopyOutStreams = 4;      // result streams of gemm_host, taken in turn
constexpr int kMaxPanels = 4;           // row panels of one gemm_host call

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    bool pool_ready = false;
    cudaMemPool_t pool = nullptr;   // stream-ordered scratch (see scratch_pool)
    cudaStream_t copy_in = nullptr; // host-operand pipeline of gemm_host
    cudaStream_t copy_out[kCopyOutStreams] = {};
    unsigned next_out = 0;
};

std::mutex g_mutex;
DeviceInfo g_devices[kMaxDevices];
void* g_encode_fn = nullptr;
bool g_encode_looked_up = false;

std::atomic<long long> g_wait_limit_ns{2000000000LL};
std::atomic<int> g_debug_stall{0};
std::atomic<int> g_forced_f32{-1};
std::atomic<int> g_tc_mode{-1};
std::atomic<int> g_tc_streamk{-1};
std::atomic<int> g_tc_a_loader{-1};
thread_local const char* g_last_kernel = "";
thread_local char g_last_kernel_buf[160];

// Device properties of the current device, looked up once per device.
int current_device_info(DeviceInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TGEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TGEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TGEMM_ERR_CUDA;
        // The library carries sm_103a code only.
        d.supported = (major == 10 && minor == 3);
        d.num_sms = sms;
        d.ready = true;
    }
    *out = d;
    return d.supported ? TGEMM_OK : TGEMM_ERR_UNSUPPORTED;
}

// The library's stream-ordered scratch pool on device `dev`. Freed blocks
// stay cached in the pool (no release threshold), so repeated calls do not
// go back to the driver.
cudaMemPool_t scratch_pool(int dev) {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (!d.pool_ready) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return nullptr;
        unsigned long long keep = ~0ull;
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        d.pool = pool;
        d.pool_ready = true;
    }
    return d.pool;
}

// The copy streams of one gemm_host call on device `dev` (created once):
// the operands of every call go to the device on one stream, in call order;
// each call's results come back on the next of kCopyOutStreams streams, so
// calls in flight together return their results independently.
bool copy_streams(int dev, cudaStream_t* in, cudaStream_t* out) {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_devices[dev];
    if (d.copy_in == nullptr) {
        cudaStream_t made[1 + kCopyOutStreams] = {};
        for (int i = 0; i <= kCopyOutStreams; ++i)
            if (cudaStreamCreateWithFlags(&made[i], cudaStreamNonBlocking) != cudaSuccess) {
                for (int j = 0; j < i; ++j) cudaStreamDestroy(made[j]);
                return false;
            }
        d.copy_in = made[0];
        for (int i = 0; i < kCopyOutStreams; ++i) d.copy_out[i] = made[1 + i];
    }
    *in = d.copy_in;
    *out = d.copy_out[d.next_out++ % kCopyOutStreams];
    return true;
}

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

// Row panels of gemm_host, on multiples of 256 rows; one panel below 1024
// rows. When the arithmetic takes longer than the transfers (`compute_bound`,
// the FP32 path): a 256-row first panel (the arithmetic starts as soon as B
// and those rows have arrived), a last panel of 256 to 511 rows (little of C
// is left to copy out once the arithmetic ends) and, between them, one panel
// (M < 2048) or two of >= 768 rows. Otherwise (tensor paths, bound by the
// CPU-GPU link): 2 or 4 equal panels, so that results start to leave early.
// Returns the panel count; bounds[i] is the first row of panel i and
// bounds[count] = M.
int host_panels(int M, bool compute_bound, long bounds[kMaxPanels + 1]) {
    bounds[0] = 0;
    if (M < 1024) {
        bounds[1] = M;
        return 1;
    }
    if (!compute_bound) {
        const int n = M >= 2048 ? 4 : 2;
        for (int i = 1; i < n; ++i) bounds[i] = (long)M * i / n / 256 * 256;
        bounds[n] = M;
        return n;
    }
    const long last = (long)(M - 256) / 256 * 256;
    const int middle = M < 2048 ? 1 : 2;
    for (int i = 0; i < middle; ++i)
        bounds[1 + i] = 256 + (last - 256) * i / middle / 256 * 256;
    bounds[1 + middle] = last;
    bounds[2 + middle] = M;
    return 2 + middle;
}

void* encode_fn() {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode_looked_up) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_fn = fn;
        g_encode_looked_up = true;
    }
    return g_encode_fn;
}

// Checks common to both paths. Returns TGEMM_OK, or an error, or -1 for
// "valid and empty: nothing to do".
int check_common(int M, int N, int K, const void* A, long lda, const void* B, long ldb,
                 const float* C, long ldc) {
    if (M < 0 || N < 0 || K < 0) return TGEMM_ERR_INVALID_ARG;
    if (lda < K || ldb < N || ldc < N) return TGEMM_ERR_INVALID_ARG;
    if (lda < 0 || ldb < 0 || ldc < 0) return TGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return -1;
    if (C == nullptr) return TGEMM_ERR_INVALID_ARG;
    if (K > 0 && (A == nullptr || B == nullptr)) return TGEMM_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(C) % 4 != 0) return TGEMM_ERR_INVALID_ARG;
    return TGEMM_OK;
}

}  // namespace

namespace tgemm {
unsigned long long wait_limit_ns() { return (unsigned long long)g_wait_limit_ns.load(); }
}  // namespace tgemm

namespace {

// One product request: C = alpha * op(A) op(B) + beta * C + bias, on `path`.
struct Request {
    int M, N, K;
    const void* A;
    long lda;
    const void* B;
    long ldb;
    float* C;
    long ldc;
    int path;            // TGEMM_PATH_*
    int flags;           // TGEMM_TRANS_A | TGEMM_TRANS_B
    tgemm::Epilogue ep;
};

// Scratch carving: consecutive 256-byte-aligned pieces of one pool block.
struct Carve {
    size_t used = 0;
    size_t take(size_t bytes) {
        const size_t at = used;
        used += align256(bytes);
        return at;
    }
};

// What has to be produced before the GEMM kernel, per operand.
enum Prep { NONE, TRANSPOSE, REPACK, SPLIT, TRANSPOSE_SPLIT };

// How one valid, non-empty (K > 0) request runs: the pre-passes, the
// layout the GEMM kernel reads, the kernel's plan and the pool scratch the
// call draws (`scratch` bytes in one block, carved at the offsets below).
struct ProductPlan {
    Prep prep_a = NONE, prep_b = NONE;
    long ldk = 0, ldn = 0;       // scratch row pitches for rows of length K and N
    long ld_a = 0, ld_b = 0;     // leading dimensions the GEMM kernel reads
    bool b_kmajor = false;       // tensor paths: B read K-major (N x K)
    bool a_loader = false;       // tensor paths: A (rows 4-byte aligned) read by loader warps
    size_t a_off = 0, a2_off = 0, b_off = 0, b2_off = 0, p_off = 0;
    size_t part_bytes = 0;       // partial tiles of a split last wave
    size_t scratch = 0;          // total pool scratch of the call (0: none)
    int f32_id = 0;
    tgemm::F32Plan fplan{};
    tgemm::TcPlan tplan{};
    int shape = tgemm::TC_ONE_SM;
};

// Argument checks of a request. Returns TGEMM_OK, an error code, or -1 for
// a valid request with nothing to compute (M or N is 0).
int check_request(const Request& r) {
    const bool ta = (r.flags & TGEMM_TRANS_A) != 0, tb = (r.flags & TGEMM_TRANS_B) != 0;
    const int M = r.M, N = r.N, K = r.K;
    if (M < 0 || N < 0 || K < 0) return TGEMM_ERR_INVALID_ARG;
    if (r.lda < (ta ? M : K) || r.ldb < (tb ? K : N) || r.ldc < N) return TGEMM_ERR_INVALID_ARG;
    if (r.lda < 0 || r.ldb < 0) return TGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return -1;
    if (r.C == nullptr || reinterpret_cast<uintptr_t>(r.C) % 4 != 0) return TGEMM_ERR_INVALID_ARG;
    if (r.ep.bias != nullptr && reinterpret_cast<uintptr_t>(r.ep.bias) % 4 != 0)
        return TGEMM_ERR_INVALID_ARG;
    const size_t esz = r.path == TGEMM_PATH_BF16 ? 2 : 4;
    if (K > 0) {
        if (r.A == nullptr || r.B == nullptr) return TGEMM_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(r.A) % esz != 0 || reinterpret_cast<uintptr_t>(r.B) % esz != 0)
            return TGEMM_ERR_INVALID_ARG;
    }
    return TGEMM_OK;
}

// TF32 with B stored K x N: the kernel that transposes B in shared memory
// (128 x 128 tiles). Taken only when forced (tensor-core mode 3): the other
// kernels read such a B MN-major as stored.
bool tf32_in_kernel_transpose(int mode) {
    return mode == 3;
}

// Plan a checked request with K > 0 on a device with dev.num_sms SMs.
int plan_product(const Request& r, const DeviceInfo& dev, ProductPlan& pp) {
    const bool ta = (r.flags & TGEMM_TRANS_A) != 0, tb = (r.flags & TGEMM_TRANS_B) != 0;
    const int M = r.M, N = r.N, K = r.K;
    const int path = r.path;
    const size_t esz = path == TGEMM_PATH_BF16 ? 2 : 4;
    auto aligned16 = [&](const void* p, long ld) {
        return reinterpret_cast<uintptr_t>(p) % 16 == 0 && (ld * (long)esz) % 16 == 0;
    };
    // Scratch rows start on 128-byte boundaries: a TMA box whose rows are
    // only 16-byte aligned straddles an extra 32-byte sector per row, and
    // the TF32 kernel measured 16 % slower on such operands (row pitch
    // 6160 bytes against 6144 or 6272).
    const long per128 = (long)(128 / esz);
    pp.ldk = (K + per128 - 1) / per128 * per128;   // rows of length K
    pp.ldn = (N + per128 - 1) / per128 * per128;   // rows of length N
    const bool f32 = path == TGEMM_PATH_F32;
    const bool tf32 = path == TGEMM_PATH_TF32;
    const bool x3 = path == TGEMM_PATH_TF32X3;
    const bool bf16 = path == TGEMM_PATH_BF16;
    // What has to be produced before the GEMM kernel:
    //   A: M x K K-major. Transposed storage -> transpose (all paths);
    //      X3 -> hi/lo split; tensor paths with rows off 16 bytes -> repack.
    //   B: F32: K x N row-major (transposed storage -> transpose).
    //      BF16, TF32: K x N read MN-major, or N x K K-major when stored
    //      transposed; rows off 16 bytes -> repack. X3: hi/lo of the N x K
    //      form.
    if (x3) {
        pp.prep_a = ta ? TRANSPOSE_SPLIT : SPLIT;
        pp.prep_b = tb ? SPLIT : TRANSPOSE_SPLIT;
    } else if (f32) {
        // Rows off 16 bytes can be read with 4-byte copies, at about a
        // quarter of the throughput; for large products it is cheaper to
        // repack them first (8 (MK + KN) bytes of HBM traffic, ~2 % of the
        // GEMM at M = 3000, N = 5001) and run the 16-byte loaders.
        // (A forced configuration reads the caller's layout as given.)
        const bool big = g_forced_f32.load() < 0 && M >= 256 && N >= 256 && K >= 64;
        pp.prep_a = ta ? TRANSPOSE : (big && !aligned16(r.A, r.lda) ? REPACK : NONE);
        pp.prep_b = tb ? TRANSPOSE : (big && !aligned16(r.B, r.ldb) ? REPACK : NONE);
    } else {
        pp.prep_a = ta ? TRANSPOSE : (aligned16(r.A, r.lda) ? NONE : REPACK);
        if (tf32 && !tb && tf32_in_kernel_transpose(g_tc_mode.load()))
            pp.shape = tgemm::TC_ONE_SM_T;
        const bool b_t = pp.shape == tgemm::TC_ONE_SM_T;
        pp.prep_b = aligned16(r.B, r.ldb) ? NONE : REPACK;
        // A whose rows are 4-byte but not 16-byte aligned: repacked, or read
        // in place by the GEMM kernel's loader warps (TF32 with B either way,
        // and BF16 with B read MN-major). The repack is the default: measured faster.
        const bool rows4 = reinterpret_cast<uintptr_t>(r.A) % 4 == 0 && (r.lda * (long)esz) % 4 == 0;
        if (pp.prep_a == REPACK && rows4 && ((tf32 && !b_t) || (bf16 && !tb)) &&
            g_tc_a_loader.load() == 1) {
            pp.prep_a = NONE;
            pp.a_loader = true;
        }
    }
    // Tensor paths: B read K-major when stored transposed (and always by the
    // split form), otherwise MN-major as stored.
    pp.b_kmajor = tb || x3;
    // Layout the GEMM reads: A M x K (ld_a), B K x N or N x K (ld_b).
    pp.ld_a = pp.prep_a == NONE ? r.lda : pp.ldk;
    pp.ld_b = pp.prep_b == NONE ? r.ldb : ((f32 || !pp.b_kmajor) ? pp.ldn : pp.ldk);
    Carve cv;
    pp.a_off = pp.prep_a == NONE ? 0 : cv.take((size_t)M * pp.ldk * esz);
    pp.a2_off = x3 ? cv.take((size_t)M * pp.ldk * esz) : 0;
    // Rows of the B the GEMM reads: K (F32, BF16 MN-major) or N (K-major).
    const size_t b_rows = (f32 || !pp.b_kmajor) ? (size_t)K : (size_t)N;
    pp.b_off = pp.prep_b == NONE ? 0 : cv.take(b_rows * (size_t)pp.ld_b * esz);
    pp.b2_off = x3 ? cv.take((size_t)N * pp.ldk * esz) : 0;

    tgemm::GemmArgs probe{M, N, K, r.A, pp.ld_a, r.B, pp.ld_b, r.C, r.ldc};
    if (f32) {
        // Operands the kernel will read: the caller's, or 16-byte-row scratch.
        probe.A = pp.prep_a == NONE ? r.A : nullptr;
        probe.B = pp.prep_b == NONE ? r.B : nullptr;
        tgemm::GemmArgs chk = probe;
        if (chk.A == nullptr) chk.A = reinterpret_cast<const void*>(256);   // scratch: aligned
        if (chk.B == nullptr) chk.B = reinterpret_cast<const void*>(256);
        const int forced = g_forced_f32.load();
        if (forced >= 0) {
            if (!tgemm::f32_kernel_accepts(forced, chk)) return TGEMM_ERR_ALIGNMENT;
            pp.f32_id = forced;
        } else {
            pp.f32_id = tgemm::f32_select(chk, dev.num_sms);
        }
        pp.fplan = tgemm::f32_plan(pp.f32_id, probe, dev.num_sms);
    } else {
        // Whole tiles leave by TMA stores when C's base and rows are 16-byte
        // aligned and beta = 0 (the model charges the wide tiles more otherwise).
        const bool tma_c = reinterpret_cast<uintptr_t>(r.C) % 16 == 0 && r.ldc % 4 == 0 &&
                           N % 4 == 0 && r.ep.beta == 0.0f;
        const int sk = g_tc_streamk.load();
        if (pp.shape != tgemm::TC_ONE_SM_T)
            pp.shape = tgemm::tc_shape(M, N, K, path, g_tc_mode.load(), dev.num_sms, sk, tma_c);
        // The SIMT A loader runs with the 128 x 256 one-SM tiles.
        if (pp.a_loader && pp.shape == tgemm::TC_ONE_SM_N) pp.shape = tgemm::TC_ONE_SM;
        pp.tplan = tgemm::tc_plan(M, N, K, path, pp.shape, dev.num_sms, sk, tma_c);
    }
    pp.part_bytes = f32 ? pp.fplan.scratch_bytes : pp.tplan.scratch_bytes;
    pp.p_off = pp.part_bytes ? cv.take(pp.part_bytes) : 0;
    pp.scratch = cv.used;
    return TGEMM_OK;
}

// The kernels a planned product launches, as gemm_last_kernel reports them:
// the pre-passes, the GEMM kernel's configuration and its tail.
void product_name(const ProductPlan& pp, int path, char* out, size_t n) {
    std::string s;
    const bool repack_both = pp.prep_a == REPACK && pp.prep_b == REPACK;
    if (repack_both) s += "repack_ab+";
    static const char* const kA[] = {"", "transpose_a+", "repack_a+", "split_a+", "transpose_split_a+"};
    static const char* const kB[] = {"", "transpose_b+", "repack_b+", "split_b+", "transpose_split_b+"};
    if (!repack_both) {
        s += kA[pp.prep_a];
        s += kB[pp.prep_b];
    }
    char tail[96] = "";
    if (path == TGEMM_PATH_F32) {
        s += tgemm::f32_kernel_name(pp.f32_id);
        if (pp.fplan.split > 1)
            snprintf(tail, sizeof(tail), "+splitk_reduce(split=%d,tiles=%d)", pp.fplan.split,
                     pp.fplan.tiles_m * pp.fplan.tiles_n - pp.fplan.dp_tiles);
    } else {
        s += tgemm::tc_kernel_name(path, pp.shape);
        if (pp.a_loader) strncat(tail, "(a_loader)", sizeof(tail) - strlen(tail) - 1);
        const int tail_tiles = pp.tplan.tiles_m * pp.tplan.tiles_n - pp.tplan.dp_tiles;
        if (pp.tplan.sk_slots > 0 && pp.tplan.sk_split)
            snprintf(tail + strlen(tail), sizeof(tail) - strlen(tail),
                     "+tc_split_reduce(split=%d,tiles=%d)", pp.tplan.sk_slots / tail_tiles, tail_tiles);
        else if (pp.tplan.sk_slots > 0)
            snprintf(tail + strlen(tail), sizeof(tail) - strlen(tail), "(streamk:slots=%d,tiles=%d)",
                     pp.tplan.sk_slots, tail_tiles);
    }
    s += tail;
    snprintf(out, n, "%s", s.c_str());
}

int run_product(const Request& r, cudaStream_t stream) {
    g_last_kernel = "";
    int st = check_request(r);
    if (st == -1) return TGEMM_OK;
    if (st != TGEMM_OK) return st;
    const int M = r.M, N = r.N, K = r.K;
    const int path = r.path;
    const size_t esz = path == TGEMM_PATH_BF16 ? 2 : 4;

    DeviceInfo dev;
    st = current_device_info(&dev);
    if (st != TGEMM_OK) return st;

    if (K == 0) {
        if (tgemm::empty_product(r.C, r.ldc, M, N, r.ep, stream) != cudaSuccess)
            return TGEMM_ERR_CUDA;
        g_last_kernel = "empty_product";
        return TGEMM_OK;
    }

    ProductPlan pp;
    st = plan_product(r, dev, pp);
    if (st != TGEMM_OK) return st;
    const bool f32 = path == TGEMM_PATH_F32;
    const bool bf16 = path == TGEMM_PATH_BF16;
    const long ldk = pp.ldk, ldn = pp.ldn;

    void* enc = nullptr;
    if (!f32) {
        enc = encode_fn();
        if (enc == nullptr) return TGEMM_ERR_CUDA;
    }
    void* ws = nullptr;
    if (pp.scratch > 0) {
        int devno = 0;
        if (cudaGetDevice(&devno) != cudaSuccess) return TGEMM_ERR_CUDA;
        cudaMemPool_t pool = scratch_pool(devno);
        if (pool == nullptr) return TGEMM_ERR_CUDA;
        if (cudaMallocFromPoolAsync(&ws, pp.scratch, pool, stream) != cudaSuccess)
            return TGEMM_ERR_CUDA;
    }
    char* base = static_cast<char*>(ws);

    // ---- pre-passes
    int rc = TGEMM_OK;
    auto ok = [&](cudaError_t e) {
        if (e != cudaSuccess && rc == TGEMM_OK) rc = TGEMM_ERR_CUDA;
    };
    tgemm::GemmArgs a{M, N, K, r.A, pp.ld_a, r.B, pp.ld_b, r.C, r.ldc};
    a.ep = r.ep;
    a.a_loader = pp.a_loader;
    a.a_esz = (int)esz;
    const size_t a_off = pp.a_off, a2_off = pp.a2_off, b_off = pp.b_off, b2_off = pp.b2_off;
    // Both operands' rows off 16 bytes: one launch repacks A and B.
    const bool repack_both = pp.prep_a == REPACK && pp.prep_b == REPACK;
    if (repack_both) {
        a.A = base + a_off;
        a.B = base + b_off;
        const tgemm::RepackJob ja{r.A, r.lda, base + a_off, ldk, M, K};
        const tgemm::RepackJob jb = pp.b_kmajor
                                        ? tgemm::RepackJob{r.B, r.ldb, base + b_off, ldk, N, K}
                                        : tgemm::RepackJob{r.B, r.ldb, base + b_off, ldn, K, N};
        ok(tgemm::repack_rows2(ja, jb, (int)esz, stream));
    }
    switch (repack_both ? NONE : pp.prep_a) {
        case TRANSPOSE:
            a.A = base + a_off;
            ok(bf16 ? tgemm::transpose_u16(r.A, r.lda, base + a_off, ldk, K, M, stream)
                    : tgemm::transpose_f32(static_cast<const float*>(r.A), r.lda,
                                           reinterpret_cast<float*>(base + a_off), ldk, K, M,
                                           stream));
            break;
        case REPACK:
            a.A = base + a_off;
            ok(tgemm::repack_rows(r.A, r.lda, base + a_off, ldk, M, K, (int)esz, stream));
            break;
        case SPLIT:
            a.A = base + a_off;
            a.A2 = base + a2_off;
            ok(tgemm::split_rows_tf32(static_cast<const float*>(r.A), r.lda,
                                      reinterpret_cast<float*>(base + a_off),
                                      reinterpret_cast<float*>(base + a2_off), ldk, M, K, stream));
            break;
        case TRANSPOSE_SPLIT:
            a.A = base + a_off;
            a.A2 = base + a2_off;
            ok(tgemm::transpose_split_tf32(static_cast<const float*>(r.A), r.lda,
                                           reinterpret_cast<float*>(base + a_off),
                                           reinterpret_cast<float*>(base + a2_off), ldk, K, M,
                                           stream));
            break;
        default:
            break;
    }
    switch (repack_both ? NONE : pp.prep_b) {
        case TRANSPOSE:     // FP32 only: stored N x K -> K x N
            a.B = base + b_off;
            ok(tgemm::transpose_f32(static_cast<const float*>(r.B), r.ldb,
                                    reinterpret_cast<float*>(base + b_off), ldn, N, K, stream));
            break;
        case REPACK:
            a.B = base + b_off;
            if (pp.b_kmajor)
                ok(tgemm::repack_rows(r.B, r.ldb, base + b_off, ldk, N, K, (int)esz, stream));
            else
                ok(tgemm::repack_rows(r.B, r.ldb, base + b_off, ldn, K, N, (int)esz, stream));
            break;
        case SPLIT:     // stored N x K
            a.B = base + b_off;
            a.B2 = base + b2_off;
            ok(tgemm::split_rows_tf32(static_cast<const float*>(r.B), r.ldb,
                                      reinterpret_cast<float*>(base + b_off),
                                      reinterpret_cast<float*>(base + b2_off), ldk, N, K, stream));
            break;
        case TRANSPOSE_SPLIT:    // stored K x N
            a.B = base + b_off;
            a.B2 = base + b2_off;
            ok(tgemm::transpose_split_tf32(static_cast<const float*>(r.B), r.ldb,
                                           reinterpret_cast<float*>(base + b_off),
                                           reinterpret_cast<float*>(base + b2_off), ldk, K, N,
                                           stream));
            break;
        default:
            break;
    }

    // ---- the product
    float* partials = pp.part_bytes ? reinterpret_cast<float*>(base + pp.p_off) : nullptr;
    if (rc == TGEMM_OK) {
        if (f32)
            ok(tgemm::f32_launch(pp.f32_id, a, pp.fplan, partials, stream));
        else
            ok(tgemm::tc_launch(a, path, pp.b_kmajor ? 1 : 0, enc,
                                (unsigned long long)g_wait_limit_ns.load(), g_debug_stall.load(),
                                pp.shape, pp.tplan, partials, stream));
    }
    if (ws != nullptr && cudaFreeAsync(ws, stream) != cudaSuccess && rc == TGEMM_OK)
        rc = TGEMM_ERR_CUDA;
    if (rc == TGEMM_OK) {
        product_name(pp, path, g_last_kernel_buf, sizeof(g_last_kernel_buf));
        g_last_kernel = g_last_kernel_buf;
    }
    return rc;
}

}  // namespace

extern "C" {

int gemm_f32(int M, int N, int K, const float* A, long lda, const float* B, long ldb,
             float* C, long ldc, cudaStream_t stream) {
    Request r{M, N, K, A, lda, B, ldb, C, ldc, TGEMM_PATH_F32, 0, tgemm::Epilogue()};
    return run_product(r, stream);
}

int gemm_tc(int M, int N, int K, const void* A, long lda, const void* B, long ldb,
            float* C, long ldc, int in_type, cudaStream_t stream) {
    g_last_kernel = "";
    if (in_type != TGEMM_TF32 && in_type != TGEMM_BF16 && in_type != TGEMM_TF32X3)
        return TGEMM_ERR_INVALID_ARG;
    // The input-type codes are the path codes of the tensor paths.
    Request r{M, N, K, A, lda, B, ldb, C, ldc, in_type, 0, tgemm::Epilogue()};
    return run_product(r, stream);
}

int gemm_ex(int M, int N, int K, const void* A, long lda, const void* B, long ldb, float* C,
            long ldc, int path, int flags, float alpha, float beta, const float* bias,
            cudaStream_t stream) {
    g_last_kernel = "";
    if (path < TGEMM_PATH_F32 || path > TGEMM_PATH_TF32X3) return TGEMM_ERR_INVALID_ARG;
    if ((flags & ~(TGEMM_TRANS_A | TGEMM_TRANS_B)) != 0) return TGEMM_ERR_INVALID_ARG;
    tgemm::Epilogue ep;
    ep.alpha = alpha;
    ep.beta = beta;
    ep.bias = bias;
    Request r{M, N, K, A, lda, B, ldb, C, ldc, path, flags, ep};
    return run_product(r, stream);
}

int gemm_host(int M, int N, int K, const void* A, long lda, const void* B, long ldb, float* C,
              long ldc, int path, cudaStream_t stream) {
    g_last_kernel = "";
    if (path < TGEMM_PATH_F32 || path > TGEMM_PATH_TF32X3) return TGEMM_ERR_INVALID_ARG;
    int st = check_common(M, N, K, A, lda, B, ldb, C, ldc);
    if (st == -1) return TGEMM_OK;
    if (st != TGEMM_OK) return st;
    const size_t esz = path == TGEMM_PATH_BF16 ? 2 : 4;
    if (K > 0 && (reinterpret_cast<uintptr_t>(A) % esz != 0 ||
                  reinterpret_cast<uintptr_t>(B) % esz != 0))
        return TGEMM_ERR_INVALID_ARG;

    DeviceInfo dev;
    st = current_device_info(&dev);
    if (st != TGEMM_OK) return st;
    int devno = 0;
    if (cudaGetDevice(&devno) != cudaSuccess) return TGEMM_ERR_CUDA;
    cudaStream_t s_in, s_out;
    if (!copy_streams(devno, &s_in, &s_out)) return TGEMM_ERR_CUDA;
    cudaMemPool_t pool = scratch_pool(devno);
    if (pool == nullptr) return TGEMM_ERR_CUDA;

    // Device copies with 128-byte rows (16 bytes is what every loader and TMA
    // copy takes; 128 keeps TMA boxes on whole sectors).
    const long per128 = (long)(128 / esz);
    const long lda_d = (K + per128 - 1) / per128 * per128;
    const long ldb_d = (N + per128 - 1) / per128 * per128;
    const long ldc_d = (N + 31) / 32 * 32;

    // Row panels: each panel is multiplied on `stream` as soon as its rows
    // of A have arrived, and its rows of C leave while the next panel
    // computes. (Panels on streams of their own finish together, as the
    // blocks of concurrent kernels interleave, and C then leaves only at the
    // end: measured slower.) FP32 4096^3 from pinned memory: 2.90 ms with
    // short first and last panels, 3.13 ms with four equal ones.
    long bounds[kMaxPanels + 1];
    const int panels = host_panels(M, path == TGEMM_PATH_F32, bounds);
    // FP32 (compute-bound): B goes up in two column halves, and the first
    // panel is multiplied in the same halves, its left half as soon as B's
    // left columns and the panel's rows have arrived. nh: the left half's
    // width, a multiple of 256 columns (0: B in one piece).
    const long nh = (path == TGEMM_PATH_F32 && panels > 1 && K > 0) ? (long)(N / 2) / 256 * 256 : 0;

    // Plans and scratch: one pool block for A, B, C, B's high and low parts
    // transposed and the high and low parts of A (TF32X3), partials. BF16 and
    // TF32 read the device copy of B MN-major as uploaded.
    const bool tc = path != TGEMM_PATH_F32;
    const bool x3 = path == TGEMM_PATH_TF32X3;
    const int in_type = path == TGEMM_PATH_BF16 ? TGEMM_BF16 : x3 ? TGEMM_TF32X3 : TGEMM_TF32;
    const long ldt = (K + 31) / 32 * 32;
    const size_t bt_bytes = align256((size_t)N * ldt * 4);
    const size_t a_bytes = align256((size_t)M * lda_d * esz);
    size_t off_b = a_bytes;
    size_t off_c = off_b + align256((size_t)K * ldb_d * esz);
    size_t off_t = off_c + align256((size_t)M * ldc_d * 4);
    size_t off_a2 = off_t + (x3 ? 2 * bt_bytes : 0);
    size_t off_p = off_a2 + (x3 ? 2 * a_bytes : 0);
    int f32_id[kMaxPanels] = {}, f32_id_right = 0;
    tgemm::F32Plan f32_plan[kMaxPanels], f32_plan_right;
    size_t part_off_right = 0;
    tgemm::TcPlan tc_plan[kMaxPanels];
    int shape[kMaxPanels] = {};
    size_t part_off[kMaxPanels];
    size_t total = off_p;
    for (int i = 0; i < panels; ++i) {
        const int rows = (int)(bounds[i + 1] - bounds[i]);
        part_off[i] = total;
        if (K == 0) continue;
        if (tc) {
            const int sk = g_tc_streamk.load();
            shape[i] = tgemm::tc_shape(rows, N, K, in_type, g_tc_mode.load(), dev.num_sms, sk);
            tc_plan[i] = tgemm::tc_plan(rows, N, K, in_type, shape[i], dev.num_sms, sk);
            total += align256(tc_plan[i].scratch_bytes);
        } else {
            // Device operands are 16-byte aligned: the vector loaders apply.
            const int forced = g_forced_f32.load();
            auto plan = [&](int cols, int& id, tgemm::F32Plan& pl) {
                tgemm::GemmArgs pa{rows, cols, K, nullptr, lda_d, nullptr, ldb_d, nullptr, ldc_d};
                tgemm::GemmArgs chk = pa;
                chk.A = chk.B = reinterpret_cast<const void*>(256);   // scratch: 16-byte aligned
                id = forced >= 0 ? forced : tgemm::f32_select(chk, dev.num_sms);
                pl = tgemm::f32_plan(id, pa, dev.num_sms);
                total += align256(pl.scratch_bytes);
            };
            if (i == 0 && nh > 0) {
                plan((int)nh, f32_id[0], f32_plan[0]);
                part_off_right = total;
                plan(N - (int)nh, f32_id_right, f32_plan_right);
            } else {
                plan(N, f32_id[i], f32_plan[i]);
            }
        }
    }
    void* ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, total, pool, stream) != cudaSuccess) return TGEMM_ERR_CUDA;
    char* base = static_cast<char*>(ws);
    char* Ad = base;
    char* Bd = base + off_b;
    float* Cd = reinterpret_cast<float*>(base + off_c);
    float* Bt = reinterpret_cast<float*>(base + off_t);
    float* Bt_lo = reinterpret_cast<float*>(base + off_t + bt_bytes);    // TF32X3
    float* A_hi = reinterpret_cast<float*>(base + off_a2);               // TF32X3
    float* A_lo = reinterpret_cast<float*>(base + off_a2 + a_bytes);

    const int nev = 2 * panels + 4;
    cudaEvent_t ev[2 * kMaxPanels + 4];
    for (int i = 0; i < nev; ++i)
        if (cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
            cudaFreeAsync(ws, stream);
            return TGEMM_ERR_CUDA;
        }
    cudaEvent_t ev_ready = ev[0], ev_b = ev[1], ev_out = ev[2], ev_b_left = ev[3];
    cudaEvent_t* ev_a = ev + 4;
    cudaEvent_t* ev_c = ev + 4 + panels;
    int rc = TGEMM_OK;
    auto ok = [&](cudaError_t e) {
        if (e != cudaSuccess && rc == TGEMM_OK) rc = TGEMM_ERR_CUDA;
        return e == cudaSuccess;
    };
    const unsigned long long limit = (unsigned long long)g_wait_limit_ns.load();
    const int stall = g_debug_stall.load();
    void* enc = tc ? encode_fn() : nullptr;
    if (tc && enc == nullptr) rc = TGEMM_ERR_CUDA;

    // The scratch block is valid on `stream` from here on.
    ok(cudaEventRecord(ev_ready, stream));
    ok(cudaStreamWaitEvent(s_in, ev_ready, 0));
    ok(cudaStreamWaitEvent(s_out, ev_ready, 0));
    // Upload order: B (or B's left columns), then each panel of A, B's
    // right columns right after the first panel.
    const long n_first = nh > 0 ? nh : N;
    if (K > 0)
        ok(cudaMemcpy2DAsync(Bd, ldb_d * esz, B, ldb * esz, n_first * esz, K,
                             cudaMemcpyHostToDevice, s_in));
    ok(cudaEventRecord(ev_b_left, s_in));
    if (nh == 0) ok(cudaEventRecord(ev_b, s_in));
    for (int i = 0; i < panels; ++i) {
        const long r0 = bounds[i], rows = bounds[i + 1] - bounds[i];
        if (K > 0)
            ok(cudaMemcpy2DAsync(Ad + r0 * lda_d * esz, lda_d * esz,
                                 static_cast<const char*>(A) + r0 * lda * esz, lda * esz, K * esz,
                                 rows, cudaMemcpyHostToDevice, s_in));
        ok(cudaEventRecord(ev_a[i], s_in));
        if (i == 0 && nh > 0) {
            ok(cudaMemcpy2DAsync(Bd + nh * esz, ldb_d * esz,
                                 static_cast<const char*>(B) + nh * esz, ldb * esz,
                                 (N - nh) * esz, K, cudaMemcpyHostToDevice, s_in));
            ok(cudaEventRecord(ev_b, s_in));
        }
    }
    ok(cudaStreamWaitEvent(stream, nh > 0 ? ev_b_left : ev_b, 0));
    if (rc == TGEMM_OK && x3 && K > 0)
        ok(tgemm::transpose_split_tf32(reinterpret_cast<const float*>(Bd), ldb_d, Bt, Bt_lo, ldt,
                                       K, N, stream));
    const char* name = "";
    for (int i = 0; i < panels && rc == TGEMM_OK; ++i) {
        const long r0 = bounds[i];
        const int rows = (int)(bounds[i + 1] - bounds[i]);
        ok(cudaStreamWaitEvent(stream, ev_a[i], 0));
        float* Cp = Cd + r0 * ldc_d;
        float* part = reinterpret_cast<float*>(base + part_off[i]);
        if (K == 0) {
            ok(tgemm::empty_product(Cp, ldc_d, rows, N, tgemm::Epilogue(), stream));
            name = "empty_product";
        } else if (x3) {
            // This panel's rows of A split into high and low TF32 parts.
            const float* Ap = reinterpret_cast<const float*>(Ad + r0 * lda_d * esz);
            ok(tgemm::split_rows_tf32(Ap, lda_d, A_hi + r0 * lda_d, A_lo + r0 * lda_d, lda_d,
                                      rows, K, stream));
            tgemm::GemmArgs pa{rows, N, K, A_hi + r0 * lda_d, lda_d, Bt, ldt, Cp, ldc_d};
            pa.A2 = A_lo + r0 * lda_d;
            pa.B2 = Bt_lo;
            ok(tgemm::tc_launch(pa, in_type, 1, enc, limit, stall, shape[i],
                                tc_plan[i], part, stream));
            name = tgemm::tc_kernel_name(in_type, shape[i]);
        } else if (tc) {
            tgemm::GemmArgs pa{rows, N, K, Ad + r0 * lda_d * esz, lda_d, Bd, ldb_d, Cp, ldc_d};
            ok(tgemm::tc_launch(pa, in_type, 0, enc, limit, stall, shape[i],
                                tc_plan[i], part, stream));
            name = tgemm::tc_kernel_name(in_type, shape[i]);
        } else if (i == 0 && nh > 0) {
            // The first panel in B's two column halves.
            tgemm::GemmArgs left{rows, (int)nh, K, Ad, lda_d, Bd, ldb_d, Cp, ldc_d};
            ok(tgemm::f32_launch(f32_id[0], left, f32_plan[0], part, stream));
            ok(cudaStreamWaitEvent(stream, ev_b, 0));
            tgemm::GemmArgs right{rows, N - (int)nh, K, Ad, lda_d, Bd + nh * esz, ldb_d,
                                  Cp + nh, ldc_d};
            ok(tgemm::f32_launch(f32_id_right, right, f32_plan_right,
                                 reinterpret_cast<float*>(base + part_off_right), stream));
            name = tgemm::f32_kernel_name(f32_id_right);
        } else {
            tgemm::GemmArgs pa{rows, N, K, Ad + r0 * lda_d * esz, lda_d, Bd, ldb_d, Cp, ldc_d};
            ok(tgemm::f32_launch(f32_id[i], pa, f32_plan[i], part, stream));
            name = tgemm::f32_kernel_name(f32_id[i]);
        }
        ok(cudaEventRecord(ev_c[i], stream));
    }
    for (int i = 0; i < panels && rc == TGEMM_OK; ++i) {
        const long r0 = bounds[i], rows = bounds[i + 1] - bounds[i];
        ok(cudaStreamWaitEvent(s_out, ev_c[i], 0));
        ok(cudaMemcpy2DAsync(C + r0 * ldc, ldc * sizeof(float), Cd + r0 * ldc_d,
                             ldc_d * sizeof(float), N * sizeof(float), rows,
                             cudaMemcpyDeviceToHost, s_out));
    }
    ok(cudaEventRecord(ev_out, s_out));
    // Whatever happened above, the caller's stream orders after every copy
    // before the scratch goes back to the pool.
    cudaStreamWaitEvent(stream, ev_out, 0);
    cudaStreamWaitEvent(stream, ev_b, 0);
    for (int i = 0; i < panels; ++i) cudaStreamWaitEvent(stream, ev_a[i], 0);
    if (cudaFreeAsync(ws, stream) != cudaSuccess && rc == TGEMM_OK) rc = TGEMM_ERR_CUDA;
    for (int i = 0; i < nev; ++i) cudaEventDestroy(ev[i]);
    if (rc == TGEMM_OK) {
        snprintf(g_last_kernel_buf, sizeof(g_last_kernel_buf), "host_pipeline(panels=%d)+%s%s",
                 panels,
                 K == 0 || !x3 ? "" : "transpose_split_b+split_a+",
                 name);
        g_last_kernel = g_last_kernel_buf;
    }
    return rc;
}

long long gemm_scratch_bytes(int M, int N, int K, const void* A, long lda, const void* B,
                             long ldb, const float* C, long ldc, int path, int flags) {
    if (path < TGEMM_PATH_F32 || path > TGEMM_PATH_TF32X3) return -TGEMM_ERR_INVALID_ARG;
    if ((flags & ~(TGEMM_TRANS_A | TGEMM_TRANS_B)) != 0) return -TGEMM_ERR_INVALID_ARG;
    Request r{M, N, K, A, lda, B, ldb, const_cast<float*>(C), ldc, path, flags, tgemm::Epilogue()};
    int st = check_request(r);
    if (st == -1) return 0;
    if (st != TGEMM_OK) return -st;
    DeviceInfo dev;
    st = current_device_info(&dev);
    if (st != TGEMM_OK) return -st;
    if (K == 0) return 0;
    ProductPlan pp;
    st = plan_product(r, dev, pp);
    if (st != TGEMM_OK) return -st;
    return (long long)pp.scratch;
}

int gemm_plan_name(int M, int N, int K, const void* A, long lda, const void* B, long ldb,
                   const float* C, long ldc, int path, int flags, int num_sms, char* buf,
                   int buf_len) {
    if (buf == nullptr || buf_len < 1 || num_sms < 2) return TGEMM_ERR_INVALID_ARG;
    buf[0] = '\0';
    if (path < TGEMM_PATH_F32 || path > TGEMM_PATH_TF32X3) return TGEMM_ERR_INVALID_ARG;
    if ((flags & ~(TGEMM_TRANS_A | TGEMM_TRANS_B)) != 0) return TGEMM_ERR_INVALID_ARG;
    Request r{M, N, K, A, lda, B, ldb, const_cast<float*>(C), ldc, path, flags, tgemm::Epilogue()};
    int st = check_request(r);
    if (st == -1) return TGEMM_OK;                  // nothing to compute
    if (st != TGEMM_OK) return st;
    if (K == 0) {
        snprintf(buf, (size_t)buf_len, "empty_product");
        return TGEMM_OK;
    }
    DeviceInfo dev;                                 // the planner reads only the SM count
    dev.num_sms = num_sms;
    ProductPlan pp;
    st = plan_product(r, dev, pp);
    if (st != TGEMM_OK) return st;
    product_name(pp, path, buf, (size_t)buf_len);
    return TGEMM_OK;
}

int gemm_device_status(cudaStream_t stream) {
    DeviceInfo dev;
    int st = current_device_info(&dev);
    if (st != TGEMM_OK) return st;
    int v = 0;
    if (tgemm::tc_read_and_clear_status(&v, stream) != cudaSuccess) return TGEMM_ERR_CUDA;
    return v == 0 ? TGEMM_OK : TGEMM_ERR_DEVICE_TIMEOUT;
}

int gemm_tc_peak(int in_type, int pair, long iters, double* flop_per_clk_sm, double* tflops,
                 cudaStream_t stream) {
    if (in_type != TGEMM_TF32 && in_type != TGEMM_BF16) return TGEMM_ERR_INVALID_ARG;
    if (pair != 0 && pair != 1) return TGEMM_ERR_INVALID_ARG;
    if (iters < 1 || iters > 100000000L || flop_per_clk_sm == nullptr || tflops == nullptr)
        return TGEMM_ERR_INVALID_ARG;
    DeviceInfo dev;
    int st = current_device_info(&dev);
    if (st != TGEMM_OK) return st;
    long long* cycles = nullptr;
    if (cudaMalloc(&cycles, sizeof(long long) * (size_t)dev.num_sms) != cudaSuccess)
        return TGEMM_ERR_CUDA;
    std::vector<long long> host((size_t)dev.num_sms, -1);
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    int units = 0;
    int rc = TGEMM_OK;
    float ms = 0.0f;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess ||
        cudaEventRecord(e0, stream) != cudaSuccess ||
        tgemm::tc_peak(in_type, pair != 0, iters, dev.num_sms,
                       (unsigned long long)g_wait_limit_ns.load(), cycles, &units,
                       stream) != cudaSuccess ||
        cudaEventRecord(e1, stream) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess ||
        cudaMemcpy(host.data(), cycles, sizeof(long long) * (size_t)units,
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        rc = TGEMM_ERR_CUDA;
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaFree(cycles);
    if (rc != TGEMM_OK) return rc;
    int status = 0;
    if (tgemm::tc_read_and_clear_status(&status, stream) != cudaSuccess) return TGEMM_ERR_CUDA;
    host.resize((size_t)units);
    for (long long c : host)
        if (c <= 0 || status != 0) return TGEMM_ERR_DEVICE_TIMEOUT;
    std::sort(host.begin(), host.end());
    const double median = (double)host[host.size() / 2];
    const double per_unit = tgemm::tc_peak_flop_per_mma(in_type, pair != 0) * (double)iters;
    *flop_per_clk_sm = per_unit / median / (pair ? 2.0 : 1.0);
    *tflops = per_unit * units / (ms * 1e-3) / 1e12;
    return TGEMM_OK;
}

const char* gemm_status_string(int status) {
    switch (status) {
        case TGEMM_OK: return "ok";
        case TGEMM_ERR_INVALID_ARG: return "invalid argument";
        case TGEMM_ERR_ALIGNMENT: return "misaligned operand (16-byte pointers and ld needed)";
        case TGEMM_ERR_CUDA: return "CUDA error";
        case TGEMM_ERR_DEVICE_TIMEOUT: return "a kernel wait timed out";
        case TGEMM_ERR_UNSUPPORTED: return "unsupported device (sm_103 required)";
        default: return "unknown tgemm status";
    }
}

int gemm_set_wait_limit_ns(long long ns) {
    if (ns <= 0) return TGEMM_ERR_INVALID_ARG;
    g_wait_limit_ns.store(ns);
    return TGEMM_OK;
}

int gemm_set_debug_stall(int enable) {
    g_debug_stall.store(enable ? 1 : 0);
    return TGEMM_OK;
}

int gemm_set_f32_kernel(int id) {
    if (id < -1 || id >= tgemm::f32_kernel_count()) return TGEMM_ERR_INVALID_ARG;
    g_forced_f32.store(id);
    return TGEMM_OK;
}

int gemm_set_tc_kernel(int mode) {
    if (mode < -1 || mode > 4) return TGEMM_ERR_INVALID_ARG;
    g_tc_mode.store(mode);
    return TGEMM_OK;
}

int gemm_set_tc_a_loader(int mode) {
    if (mode < -1 || mode > 1) return TGEMM_ERR_INVALID_ARG;
    g_tc_a_loader.store(mode);
    return TGEMM_OK;
}

int gemm_set_tc_streamk(int slots) {
    if (slots < -64) return TGEMM_ERR_INVALID_ARG;
    g_tc_streamk.store(slots);
    return TGEMM_OK;
}

int gemm_f32_kernel_count(void) { return tgemm::f32_kernel_count(); }

const char* gemm_f32_kernel_name(int id) { return tgemm::f32_kernel_name(id); }

const char* gemm_last_kernel(void) { return g_last_kernel; }

}  // extern "C"
