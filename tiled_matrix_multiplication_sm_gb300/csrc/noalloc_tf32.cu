// gemm_tc_tf32_noalloc: the TF32 tensor-core product for callers that must
// not allocate device memory.
//
// gemm_tc with TGEMM_TF32 draws scratch memory from a stream-ordered memory
// pool when an operand's rows are not 16-byte aligned (a repacked copy) and
// when the last wave of tiles is split (partial tiles). Some callers cannot
// let a library allocate:
// an application or plugin that reserves all of its device memory up front
// and treats any later allocation as a failure, or code that must not touch
// the device allocator while it runs. This entry point gives them the same
// product with the scratch in a fixed array in the library's own device
// memory (TGEMM_NOALLOC_SCRATCH_FLOATS floats, 16 MiB). Every device that
// loads the library holds that array until the process exits.
//
// With B's rows 16-byte aligned it runs gemm_tc's TF32 kernel alone, B read
// as stored (MN-major), and touches no scratch. Otherwise B is first
// transposed into the array and read K-major; the transposed rows are
// round_up(K, 32) floats apart (128 bytes, as gemm_tc's scratch: the TF32
// kernel ran 16 % slower on rows only 16 bytes aligned) when N of them fit
// the array, else round_up(K, 4) floats apart (16 bytes, the least the
// tensor-memory copies accept). The last wave is never split.
// Nothing in the scratch has to start at zero: each call writes the N x K
// block it reads before reading it, and the padding columns are never read.
// All calls share the one array, so calls whose work overlaps on the GPU
// (different streams, or different host threads) race on it and give wrong
// results; serialise them.

#include "../../include/tgemm.h"
#include "tgemm_internal.h"

#include <cstdint>
#include <mutex>

namespace {

static __device__ __align__(256) float g_noalloc_scratch[TGEMM_NOALLOC_SCRATCH_FLOATS];

constexpr int kMaxDevices = 64;
// The transpose pre-pass covers K in 64-row tiles on a grid of at most
// 65535 tile rows.
constexpr long kMaxK = 65535L * 64;

struct Device {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    float* scratch = nullptr;   // device address of g_noalloc_scratch
};

std::mutex g_mutex;
Device g_devices[kMaxDevices];
void* g_encode = nullptr;
bool g_encode_done = false;

// Set-up, once per device, with that device current: device attributes and
// the device address of the scratch array. The array's name is a host-side
// stand-in in host code; only the address from cudaGetSymbolAddress may be
// handed to a kernel.
int device_setup(Device* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TGEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TGEMM_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    Device& d = g_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return TGEMM_ERR_CUDA;
        d.supported = (major == 10 && minor == 3);
        d.num_sms = sms;
        if (d.supported) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
                return TGEMM_ERR_CUDA;
            d.scratch = static_cast<float*>(p);
        }
        d.ready = true;
    }
    *out = d;
    return d.supported ? TGEMM_OK : TGEMM_ERR_UNSUPPORTED;
}

void* encoder() {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode_done) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = fn;
        g_encode_done = true;
    }
    return g_encode;
}

}  // namespace

extern "C" int gemm_tc_tf32_noalloc(int M, int N, int K, const float* A, long lda,
                                    const float* B, long ldb, float* C, long ldc,
                                    cudaStream_t stream) {
    if (M < 0 || N < 0 || K < 0) return TGEMM_ERR_INVALID_ARG;
    if (lda < K || ldb < N || ldc < N || lda < 0 || ldb < 0 || ldc < 0) return TGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return TGEMM_OK;
    if (C == nullptr || reinterpret_cast<uintptr_t>(C) % 4 != 0) return TGEMM_ERR_INVALID_ARG;
    if (K > 0 && (A == nullptr || B == nullptr)) return TGEMM_ERR_INVALID_ARG;
    if ((long)K > kMaxK) return TGEMM_ERR_INVALID_ARG;
    // B with 16-byte rows is read as stored; otherwise transposed into the
    // array, 128-byte rows when they fit, else 16-byte rows.
    const bool b_direct = reinterpret_cast<uintptr_t>(B) % 16 == 0 && (ldb * 4) % 16 == 0;
    long ldt = ((long)K + 31) / 32 * 32;
    if ((long long)N * ldt > (long long)TGEMM_NOALLOC_SCRATCH_FLOATS) ldt = ((long)K + 3) / 4 * 4;
    if (!b_direct && (ldt <= 0 || (long long)N * ldt > (long long)TGEMM_NOALLOC_SCRATCH_FLOATS))
        return TGEMM_ERR_INVALID_ARG;
    if (K > 0 && (reinterpret_cast<uintptr_t>(A) % 16 != 0 || reinterpret_cast<uintptr_t>(B) % 4 != 0 ||
                  (lda * 4) % 16 != 0))
        return TGEMM_ERR_ALIGNMENT;

    Device d;
    int st = device_setup(&d);
    if (st != TGEMM_OK) return st;
    if (K == 0)
        return tgemm::empty_product(C, ldc, M, N, tgemm::Epilogue(), stream) == cudaSuccess
                   ? TGEMM_OK : TGEMM_ERR_CUDA;
    void* enc = encoder();
    if (enc == nullptr) return TGEMM_ERR_CUDA;
    if (!b_direct && tgemm::transpose_f32(B, ldb, d.scratch, ldt, K, N, stream) != cudaSuccess)
        return TGEMM_ERR_CUDA;
    tgemm::GemmArgs a{M, N, K, A, lda, b_direct ? B : d.scratch, b_direct ? ldb : ldt, C, ldc};
    const bool tma_c = reinterpret_cast<uintptr_t>(C) % 16 == 0 && ldc % 4 == 0 && N % 4 == 0;
    const int shape = tgemm::tc_shape(M, N, K, tgemm::TC_TF32, -1, d.num_sms, 0, tma_c);
    // No stream-K tail: its partial tiles would need more scratch.
    const tgemm::TcPlan plan =
        tgemm::tc_plan(M, N, K, tgemm::TC_TF32, shape, d.num_sms, 0, tma_c);
    if (tgemm::tc_launch(a, tgemm::TC_TF32, b_direct ? 0 : 1, enc, tgemm::wait_limit_ns(), 0, shape,
                         plan, nullptr, stream) != cudaSuccess)
        return TGEMM_ERR_CUDA;
    return TGEMM_OK;
}
