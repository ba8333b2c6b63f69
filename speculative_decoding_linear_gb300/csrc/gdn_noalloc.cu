// gdn_noalloc.cu -- tree verification that needs no caller-allocated workspace.
//
// gdn_tree_verify takes a workspace that the caller allocates.  Some callers
// cannot call cudaMalloc: code that runs inside a host framework which owns
// all device memory through its own pool and forbids raw allocations, and
// latency-critical decode loops in which an allocation (and the device
// synchronization that cudaMalloc/cudaFree may imply) is not acceptable.
// gdn_tree_verify_noalloc serves them: it runs the same kernels with the
// workspace placed in a fixed scratch array that lives in this library.
//
// The scratch is a file-scope __device__ array, so every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits.  In host
// code its name is only a stand-in, not a device address; the address is
// looked up once per device (with that device current) by the first call on
// that device.  All calls on a device share the array and it keeps the last
// call's contents; the kernels rewrite every entry they later read, so
// nothing needs clearing between calls.  Calls whose kernels overlap on the
// GPU (for example on two streams at once) race on the array.  Shapes that
// run the single-kernel tensor-core verifier (bf16 q/k, d_k = d_v = 256) use
// no workspace, so the array's size bounds only the other shapes.
#include <mutex>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr size_t kNoAllocScratchBytes = 32ull << 20;   // 32 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64];   // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device (looked up once).
void* scratch_address(int* status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *status = GDN_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            *status = GDN_ERR_CUDA;
            return nullptr;
        }
        g_scratch_ptr[dev] = p;
    }
    *status = GDN_OK;
    return g_scratch_ptr[dev];
}

bool ok16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dim_ok(int d) { return d >= 16 && d <= kMaxDim && d % 16 == 0; }

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" int gdn_tree_verify_noalloc(const void* q, const void* k, const void* v, int dtype,
                                       const float* alpha, const float* beta, const int32_t* parent_idx,
                                       const float* S0, float* out, void* factors, int B, int N, int H,
                                       int dk, int dv, cudaStream_t stream) {
    if (B < 1 || H < 1 || N < 1 || N > kMaxNodes || !dim_ok(dk) || !dim_ok(dv) ||
        (long long)B * H * N > 0x7fffffffLL)
        return GDN_ERR_ARG;
    if (dtype != GDN_DTYPE_BF16 && dtype != GDN_DTYPE_F32) return GDN_ERR_ARG;
    if (!ok16(q) || !ok16(k) || !ok16(v) || !ok16(alpha) || !ok16(beta) || !ok16(parent_idx) ||
        !ok16(S0) || !ok16(out) || !ok16(factors))
        return GDN_ERR_ARG;
    const size_t fbytes = factor_layout(B, N, H, dk, dv, dtype).total;
    const size_t obytes = (size_t)B * N * H * dv * 4;
    const char* o = reinterpret_cast<const char*>(out);
    const char* f = static_cast<const char*>(factors);
    if (o < f + fbytes && f < o + obytes) return GDN_ERR_ARG;
    VerifyArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.alpha = alpha;
    a.beta = beta;
    a.parent = parent_idx;
    a.S = const_cast<float*>(S0);
    a.out = out;
    a.f = factors_view(factors, B, N, H, dk, dv, dtype);
    a.ws = nullptr;
    a.B = B;
    a.N = N;
    a.H = H;
    a.dk = dk;
    a.dv = dv;
    a.commit = CommitSrc{nullptr, nullptr, nullptr, nullptr, 0, nullptr, 0};
    // Only the kernels that pass tables through the workspace are bounded by the
    // scratch array; the single-kernel verifier runs at any B * H.
    const bool uses_ws = tree_verify_uses_workspace(a, dtype);
    if (uses_ws && (size_t)B * H * ws_layout(N).record > kNoAllocScratchBytes) return GDN_ERR_CAPACITY;

    int st = GDN_OK;
    a.err = current_error_word(&st);
    if (a.err == nullptr) return st;
    if (uses_ws) {
        a.ws = static_cast<char*>(scratch_address(&st));
        if (a.ws == nullptr) return st;
    }
    a.overlap = launch_overlap_enabled();
    return launch_tree_verify(a, dtype, stream) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
