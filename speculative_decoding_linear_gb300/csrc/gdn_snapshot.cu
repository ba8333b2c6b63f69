// gdn_snapshot.cu -- the full-state snapshot baseline of state management.
//
// The review of SpecLA (pith.science 7ERME3HB), Figure 11 ("state-management
// latency"), sets the factor-buffer commit against keeping the state of every
// draft node and against replaying the accepted tokens.  This file is the
// snapshot side, on the same tensors as the verifier:
//
//   snapshot verify  node t's state S_t = alpha_t S_p + delta_t k_t^T, with
//                    delta_t = beta_t (v_t - alpha_t S_p k_t), from its parent's
//                    stored state S_p (S0 above a root); S_t is stored in
//                    S_nodes[t] and o_t = S_t q_t written.  One launch per node
//                    index t covers node t of every (sequence, head);
//                    topological order means the parent's state is ready.
//   snapshot commit  S_new = S_nodes[a], a the last accepted node (S0 when the
//                    path is empty), after checking the path against the tree.
//
// A CTA owns 16 state rows of one (sequence, head): each of its 8 warps two
// rows, each lane d_k / 32 columns in two interleaved float4 groups.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kSThreads = 256;
constexpr int kSRows = 16;

struct SnapArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;
    const float* beta;
    const int32_t* parent;
    const float* S0;        // [B][H][dv][dk]
    float* S_nodes;         // [N][B][H][dv][dk]
    float* out;             // [B][N][H][dv]
    int t, B, N, H, dk, dv;
    int* err;
};

template <typename T>
__global__ void __launch_bounds__(kSThreads) snapshot_step_kernel(SnapArgs a) {
    const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = a.t, dk = a.dk, dv = a.dv;
    griddep_wait();
    int p = a.parent[(size_t)b * a.N + t];
    if (p >= t || p < -1) {
        if (threadIdx.x == 0 && blockIdx.y == 0) set_error(a.err, GDN_ERR_TREE);
        return;
    }
    const size_t st = (size_t)dv * dk;
    const float* Sp = p >= 0 ? a.S_nodes + (((size_t)p * a.B + b) * a.H + h) * st : a.S0 + ((size_t)b * a.H + h) * st;
    float* St = a.S_nodes + (((size_t)t * a.B + b) * a.H + h) * st;
    const size_t node = ((size_t)b * a.N + t) * a.H + h;
    const T* kk = static_cast<const T*>(a.k) + node * dk;
    const T* qq = static_cast<const T*>(a.q) + node * dk;
    const float al = a.alpha[node], be = a.beta[node];
    float4 kv[2], qv[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int i = 4 * lane + 128 * j;
        kv[j] = i < dk ? ld4<T>(kk, i) : make_float4(0.f, 0.f, 0.f, 0.f);
        qv[j] = i < dk ? ld4<T>(qq, i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int rr = 0; rr < kSRows / (kSThreads / 32); ++rr) {
        const int r = blockIdx.y * kSRows + warp * (kSRows / (kSThreads / 32)) + rr;
        if (r >= dv) break;
        float4 x[2];
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = 4 * lane + 128 * j;
            x[j] = i < dk ? *reinterpret_cast<const float4*>(Sp + (size_t)r * dk + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            s += x[j].x * kv[j].x + x[j].y * kv[j].y + x[j].z * kv[j].z + x[j].w * kv[j].w;
        }
        s = warp_sum(s);
        const float d = be * (ld_elem<T>(static_cast<const T*>(a.v), node * dv + r) - al * s);
        float o = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int i = 4 * lane + 128 * j;
            if (i < dk) {
                const float4 y = make_float4(fmaf(al, x[j].x, d * kv[j].x), fmaf(al, x[j].y, d * kv[j].y),
                                             fmaf(al, x[j].z, d * kv[j].z), fmaf(al, x[j].w, d * kv[j].w));
                *reinterpret_cast<float4*>(St + (size_t)r * dk + i) = y;
                o += y.x * qv[j].x + y.y * qv[j].y + y.z * qv[j].z + y.w * qv[j].w;
            }
        }
        o = warp_sum(o);
        if (lane == 0) a.out[node * dv + r] = o;
    }
    griddep_launch();
}

struct SnapCommitArgs {
    const float* S_nodes;
    const float* S0;
    const int32_t* parent;
    const int32_t* path;
    int Lmax;
    float* S_new;
    int B, N, H, dk, dv;
    int* err;
};

__global__ void __launch_bounds__(kSThreads) snapshot_commit_kernel(SnapCommitArgs a) {
    __shared__ int s_nodes[kMaxPath];
    __shared__ int s_L;
    const int bh = blockIdx.x, b = bh / a.H;
    const int v0 = blockIdx.y * kSRows, rows = min(kSRows, a.dv - v0);
    griddep_wait();
    if (threadIdx.x < 32) {
        const int L = path_chain_setup(a.path + (size_t)b * a.Lmax, a.Lmax, a.parent + (size_t)b * a.N, a.N, s_nodes);
        if (threadIdx.x == 0) {
            s_L = L;
            if (L < 0 && blockIdx.y == 0 && bh % a.H == 0) set_error(a.err, GDN_ERR_PATH);
        }
    }
    __syncthreads();
    const int L = s_L;
    if (L < 0) return;                                   // S_new untouched
    const size_t st = (size_t)a.dv * a.dk, off = ((size_t)bh * a.dv + v0) * a.dk;
    const float* src = L > 0 ? a.S_nodes + (size_t)s_nodes[L - 1] * a.B * a.H * st + off : a.S0 + off;
    float* dst = a.S_new + off;
    if (src == dst) return;
    for (int i = threadIdx.x; i < rows * a.dk / 4; i += kSThreads)
        reinterpret_cast<float4*>(dst)[i] = reinterpret_cast<const float4*>(src)[i];
    griddep_launch();
}

bool ok16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool shape_ok(int B, int N, int H, int dk, int dv) {
    auto dim_ok = [](int d) { return d >= 16 && d <= kMaxDim && d % 16 == 0; };
    return B >= 1 && H >= 1 && N >= 1 && N <= kMaxNodes && dim_ok(dk) && dim_ok(dv) &&
           (long long)N * B * H * dv * dk < (1LL << 40);
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" int gdn_snapshot_tree_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                                        const float* beta, const int32_t* parent_idx, const float* S0, float* out,
                                        float* S_nodes, int B, int N, int H, int dk, int dv, cudaStream_t stream) {
    if (!shape_ok(B, N, H, dk, dv) || (dtype != GDN_DTYPE_BF16 && dtype != GDN_DTYPE_F32)) return GDN_ERR_ARG;
    if (!ok16(q) || !ok16(k) || !ok16(v) || !ok16(alpha) || !ok16(beta) || !ok16(parent_idx) || !ok16(S0) ||
        !ok16(out) || !ok16(S_nodes))
        return GDN_ERR_ARG;
    int st = GDN_OK;
    int* err = current_error_word(&st);
    if (err == nullptr) return st;
    SnapArgs a{q, k, v, alpha, beta, parent_idx, S0, S_nodes, out, 0, B, N, H, dk, dv, err};
    const dim3 grid(B * H, (dv + kSRows - 1) / kSRows);
    for (int t = 0; t < N; ++t) {
        a.t = t;
        const cudaError_t e = dtype == GDN_DTYPE_F32
                                  ? launch_kernel(snapshot_step_kernel<float>, grid, dim3(kSThreads), 0, stream, false, a)
                                  : launch_kernel(snapshot_step_kernel<__nv_bfloat16>, grid, dim3(kSThreads), 0, stream,
                                                  false, a);
        if (e != cudaSuccess) return GDN_ERR_CUDA;
    }
    return GDN_OK;
}

extern "C" int gdn_snapshot_commit(const float* S_nodes, const float* S0, const int32_t* parent_idx,
                                   const int32_t* accepted_path, int Lmax, float* S_new, int B, int N, int H, int dk,
                                   int dv, cudaStream_t stream) {
    if (!shape_ok(B, N, H, dk, dv) || Lmax < 1 || Lmax > kMaxPath) return GDN_ERR_ARG;
    if (!ok16(S_nodes) || !ok16(S0) || !ok16(parent_idx) || !ok16(accepted_path) || !ok16(S_new)) return GDN_ERR_ARG;
    const size_t sb = (size_t)B * H * dv * dk * 4;
    const char* x = reinterpret_cast<const char*>(S0);
    const char* y = reinterpret_cast<const char*>(S_new);
    if (x != y && x < y + sb && y < x + sb) return GDN_ERR_ARG;   // in place or disjoint
    int st = GDN_OK;
    int* err = current_error_word(&st);
    if (err == nullptr) return st;
    SnapCommitArgs a{S_nodes, S0, parent_idx, accepted_path, Lmax, S_new, B, N, H, dk, dv, err};
    return launch_kernel(snapshot_commit_kernel, dim3(B * H, (dv + kSRows - 1) / kSRows), dim3(kSThreads), 0, stream,
                         false, a) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_CUDA;
}
