// gdn_api.cu -- extern "C" entry points of libgdnspec.so (declared in
// include/gdnspec.h): argument validation, buffer views, dispatch, and the
// per-device error word that kernels write instead of trapping.
#include <atomic>
#include <mutex>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

// First device-side error since the last gdn_last_error, and the wait limit; one
// block per device.
__device__ ErrorBlock g_error_block = {0, 0, kDefaultWaitLimitNs};

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices];
int g_dev_ok[kMaxDevices];       // 0 unknown, 1 sm_103, -1 other
std::mutex g_mu;
std::atomic<int> g_overlap{0};   // gdn_set_launch_overlap

// Address of this device's error word (host-side handle), or nullptr.
int dev_setup(int* status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *status = GDN_ERR_CUDA;
        return -1;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_dev_ok[dev] == 0) {
        cudaDeviceProp p;
        if (cudaGetDeviceProperties(&p, dev) != cudaSuccess) {
            *status = GDN_ERR_CUDA;
            return -1;
        }
        g_dev_ok[dev] = (p.major == 10 && p.minor == 3) ? 1 : -1;
        if (g_dev_ok[dev] == 1) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_error_block) != cudaSuccess) {
                g_dev_ok[dev] = 0;
                *status = GDN_ERR_CUDA;
                return -1;
            }
            g_err_ptr[dev] = static_cast<int*>(ptr);
        }
    }
    if (g_dev_ok[dev] != 1) {
        *status = GDN_ERR_DEVICE;
        return -1;
    }
    *status = GDN_OK;
    return dev;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dim_ok(int d) { return d >= 16 && d <= kMaxDim && d % 16 == 0; }
bool dtype_ok(int t) { return t == GDN_DTYPE_BF16 || t == GDN_DTYPE_F32; }

bool shape_ok(int B, int N, int H, int dk, int dv) {
    if (B < 1 || H < 1 || N < 1 || N > kMaxNodes || !dim_ok(dk) || !dim_ok(dv)) return false;
    return (long long)B * H * N <= 0x7fffffffLL && (long long)B * H <= 0x7fffffffLL;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const char* x = static_cast<const char*>(a);
    const char* y = static_cast<const char*>(b);
    return x < y + nb && y < x + na;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

CommitSrc commit_src(const void* factors, const int32_t* path, int Lmax, int B, int N, int H, int dk,
                     int dv, int dtype) {
    Factors f = factors_view(const_cast<void*>(factors), B, N, H, dk, dv, dtype);
    return CommitSrc{f.delta, f.key, f.g, f.parent, N, path, Lmax};
}

int verify_common(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                  const float* beta, const int32_t* parent, bool chain, float* S, float* out,
                  void* factors, void* workspace, int B, int N, int H, int dk, int dv,
                  const void* prev_factors, int N_prev, const int32_t* prev_path, int Lmax,
                  cudaStream_t stream, bool linear = false) {
    if (!shape_ok(B, N, H, dk, dv) || !dtype_ok(dtype)) return GDN_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(alpha) || !aligned16(beta) ||
        !aligned16(S) || !aligned16(out) || !aligned16(factors))
        return GDN_ERR_ARG;
    if (!chain && (!aligned16(parent) || !aligned16(workspace))) return GDN_ERR_ARG;
    const bool fused = prev_factors != nullptr || prev_path != nullptr;
    if (fused) {
        if (!aligned16(prev_factors) || !aligned16(prev_path) || Lmax < 1 || Lmax > kMaxPath ||
            N_prev < 1 || N_prev > kMaxNodes)
            return GDN_ERR_ARG;
        const size_t nf = factor_layout(B, N, H, dk, dv, dtype).total;
        const size_t np = factor_layout(B, N_prev, H, dk, dv, dtype).total;
        if (overlap(factors, nf, prev_factors, np)) return GDN_ERR_ARG;
    }
    const size_t fbytes = factor_layout(B, N, H, dk, dv, dtype).total;
    const size_t obytes = (size_t)B * N * H * dv * 4;
    if (overlap(out, obytes, factors, fbytes)) return GDN_ERR_ARG;
    int st;
    const int dev = dev_setup(&st);
    if (dev < 0) return st;

    VerifyArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.alpha = alpha;
    a.beta = beta;
    a.parent = parent;
    a.S = S;
    a.out = out;
    a.f = factors_view(factors, B, N, H, dk, dv, dtype);
    a.ws = static_cast<char*>(workspace);
    a.B = B;
    a.N = N;
    a.H = H;
    a.dk = dk;
    a.dv = dv;
    a.commit = fused ? commit_src(prev_factors, prev_path, Lmax, B, N_prev, H, dk, dv, dtype)
                     : CommitSrc{nullptr, nullptr, nullptr, nullptr, 0, nullptr, 0};
    a.err = g_err_ptr[dev];
    a.overlap = g_overlap.load() != 0;
    a.linear = linear;
    return from_cuda(chain ? launch_chain_verify(a, dtype, stream) : launch_tree_verify(a, dtype, stream));
}

}  // namespace

// Accessors for the library's other translation units.
int* current_error_word(int* status) {
    const int dev = dev_setup(status);
    return dev < 0 ? nullptr : g_err_ptr[dev];
}

bool launch_overlap_enabled() { return g_overlap.load() != 0; }

}  // namespace gdn

using namespace gdn;

extern "C" {

int gdn_factors_bytes(int B, int N, int H, int dk, int dv, int dtype, size_t* bytes) {
    if (bytes == nullptr || !shape_ok(B, N, H, dk, dv) || !dtype_ok(dtype)) return GDN_ERR_ARG;
    *bytes = factor_layout(B, N, H, dk, dv, dtype).total;
    return GDN_OK;
}

int gdn_workspace_bytes(int B, int N, int H, int dk, int dv, size_t* bytes) {
    if (bytes == nullptr || !shape_ok(B, N, H, dk, dv)) return GDN_ERR_ARG;
    *bytes = (size_t)B * H * ws_layout(N).record;
    return GDN_OK;
}

int gdn_tree_mask(const int32_t* parent_idx, int B, int N, uint64_t* mask, int32_t* depth,
                  cudaStream_t stream) {
    if (B < 1 || N < 1 || N > kMaxNodes || !aligned16(parent_idx) || !aligned16(mask) ||
        !aligned16(depth))
        return GDN_ERR_ARG;
    int st;
    const int dev = dev_setup(&st);
    if (dev < 0) return st;
    return from_cuda(launch_tree_mask(parent_idx, B, N, mask, depth, g_err_ptr[dev], stream));
}

int gdn_tree_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                    const float* beta, const int32_t* parent_idx, const float* S0, float* out,
                    void* factors, void* workspace, int B, int N, int H, int dk, int dv,
                    cudaStream_t stream) {
    return verify_common(q, k, v, dtype, alpha, beta, parent_idx, false, const_cast<float*>(S0), out,
                         factors, workspace, B, N, H, dk, dv, nullptr, 0, nullptr, 0, stream);
}

int gdn_chain_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                     const float* beta, const float* S0, float* out, void* factors, int B, int N,
                     int H, int dk, int dv, cudaStream_t stream) {
    return verify_common(q, k, v, dtype, alpha, beta, nullptr, true, const_cast<float*>(S0), out,
                         factors, nullptr, B, N, H, dk, dv, nullptr, 0, nullptr, 0, stream);
}

int gdn_commit(const float* S0, const void* factors, const int32_t* accepted_path, int Lmax,
               float* S_new, int B, int N, int H, int dk, int dv, int dtype, cudaStream_t stream) {
    if (!shape_ok(B, N, H, dk, dv) || !dtype_ok(dtype) || Lmax < 1 || Lmax > kMaxPath) return GDN_ERR_ARG;
    if (!aligned16(S0) || !aligned16(factors) || !aligned16(accepted_path) || !aligned16(S_new))
        return GDN_ERR_ARG;
    const size_t sbytes = (size_t)B * H * dv * dk * 4;
    if (S_new != S0 && overlap(S0, sbytes, S_new, sbytes)) return GDN_ERR_ARG;
    int st;
    const int dev = dev_setup(&st);
    if (dev < 0) return st;
    CommitArgs a;
    a.S0 = S0;
    a.S_new = S_new;
    a.src = commit_src(factors, accepted_path, Lmax, B, N, H, dk, dv, dtype);
    a.B = B;
    a.H = H;
    a.dk = dk;
    a.dv = dv;
    a.err = g_err_ptr[dev];
    a.overlap = g_overlap.load() != 0;
    return from_cuda(launch_commit(a, dtype, stream));
}

int gdn_commit_tree_verify(float* S, const void* prev_factors, int N_prev, const int32_t* prev_path,
                           int Lmax, const void* q, const void* k, const void* v, int dtype,
                           const float* alpha, const float* beta, const int32_t* parent_idx,
                           float* out, void* factors, void* workspace, int B, int N, int H,
                           int dk, int dv, cudaStream_t stream) {
    if (prev_factors == nullptr || prev_path == nullptr) return GDN_ERR_ARG;
    return verify_common(q, k, v, dtype, alpha, beta, parent_idx, false, S, out, factors, workspace,
                         B, N, H, dk, dv, prev_factors, N_prev, prev_path, Lmax, stream);
}

int gdn_commit_chain_verify(float* S, const void* prev_factors, int N_prev,
                            const int32_t* prev_path, int Lmax, const void* q, const void* k,
                            const void* v, int dtype, const float* alpha, const float* beta,
                            float* out, void* factors, int B, int N, int H, int dk, int dv,
                            cudaStream_t stream) {
    if (prev_factors == nullptr || prev_path == nullptr) return GDN_ERR_ARG;
    return verify_common(q, k, v, dtype, alpha, beta, nullptr, true, S, out, factors, nullptr, B, N,
                         H, dk, dv, prev_factors, N_prev, prev_path, Lmax, stream);
}

int gdn_linear_tree_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                           const float* beta, const int32_t* parent_idx, const float* S0, float* out,
                           void* factors, void* workspace, int B, int N, int H, int dk, int dv,
                           cudaStream_t stream) {
    return verify_common(q, k, v, dtype, alpha, beta, parent_idx, false, const_cast<float*>(S0), out,
                         factors, workspace, B, N, H, dk, dv, nullptr, 0, nullptr, 0, stream, true);
}

int gdn_set_launch_overlap(int enable) {
    return g_overlap.exchange(enable != 0 ? 1 : 0);
}

int gdn_last_error(cudaStream_t stream) {
    int st;
    const int dev = dev_setup(&st);
    if (dev < 0) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GDN_ERR_CUDA;
    int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_error_block, sizeof(int)) != cudaSuccess) return GDN_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_error_block, &zero, sizeof(int)) != cudaSuccess) return GDN_ERR_CUDA;
    }
    return word;
}

int gdn_set_wait_limit_ns(unsigned long long ns) {
    if (ns < 1000ull || ns > 60000000000ull) return GDN_ERR_ARG;
    int st;
    if (dev_setup(&st) < 0) return st;
    return cudaMemcpyToSymbol(g_error_block, &ns, sizeof(ns), offsetof(ErrorBlock, wait_limit_ns)) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_CUDA;
}

const char* gdn_strerror(int code) {
    switch (code) {
        case GDN_OK: return "ok";
        case GDN_ERR_ARG: return "invalid argument (shape, null or misaligned pointer, overlap)";
        case GDN_ERR_TREE: return "invalid parent_idx (parent >= node or < -1)";
        case GDN_ERR_PATH: return "invalid accepted path (not a root-first parent chain)";
        case GDN_ERR_TIMEOUT: return "a bounded device wait ran out";
        case GDN_ERR_CUDA: return "CUDA runtime error";
        case GDN_ERR_DEVICE: return "current device is not an sm_103 GPU";
        case GDN_ERR_CAPACITY:
            return "request exceeds a fixed on-device capacity (gdn_tree_verify_noalloc's scratch array)";
        default: return "unknown status";
    }
}

}  // extern "C"
