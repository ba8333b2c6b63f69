// gdn_commit.cu -- accepted-path commit from buffered factors.
//
// Review of SpecLA (pith.science 7ERME3HB), Referee Report summary:
// "accepted-state recovery via buffered per-token factors".  With the factor
// record (delta, k, g) of every verified node, the state after accepting the
// root-first path ending at node a is a rank-L update of the committed state:
//
//     S_a = e^{g_a} S0 + sum_{j on path(a)} e^{g_a - g_j} delta_j k_j^T
//
// (unrolling S_t = alpha_t S_parent + delta_t k_t^T along the path).  The
// kernel is a pure stream over S: read 4 B and write 4 B per state element,
// L <= 64 FMAs each from on-chip coefficients.  One CTA owns kRows rows of one
// (sequence, head) state; threads own 16-byte column quads (coalesced).
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kRows = 16;
constexpr int kThreads = 256;

template <typename KT>
__global__ void __launch_bounds__(kThreads) commit_kernel(CommitArgs a) {
    __shared__ int s_nodes[kMaxPath];
    __shared__ float s_coef[kMaxPath];
    __shared__ float s_cd[kMaxPath * kRows];
    __shared__ float s_ega;
    __shared__ int s_L;

    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int v0 = blockIdx.y * kRows;
    const int rows = min(kRows, a.dv - v0);
    const CommitSrc& c = a.src;

    if (threadIdx.x < 32) {
        const int L = commit_path_setup(c, b, h, a.H, s_nodes, s_coef, &s_ega);
        if (threadIdx.x == 0) {
            s_L = L;
            if (L < 0) set_error(a.err, GDN_ERR_PATH);
        }
    }
    __syncthreads();
    const int L = s_L;
    if (L < 0) return;

    const float* delta_bh = c.delta + (size_t)bh * c.N * a.dv;
    for (int i = threadIdx.x; i < L * kRows; i += kThreads) {
        const int j = i / kRows, r = i % kRows;
        s_cd[i] = r < rows ? s_coef[j] * delta_bh[(size_t)s_nodes[j] * a.dv + v0 + r] : 0.f;
    }
    __syncthreads();

    const KT* key_bh = static_cast<const KT*>(c.key) + (size_t)bh * c.N * a.dk;
    const int quads = a.dk / 4;
    const size_t base = ((size_t)bh * a.dv + v0) * a.dk;
    for (int i = threadIdx.x; i < rows * quads; i += kThreads) {
        const int r = i / quads, cc = (i % quads) * 4;
        const size_t off = base + (size_t)r * a.dk + cc;
        const float4 s = *reinterpret_cast<const float4*>(a.S0 + off);
        const float4 o = commit_quad<KT>(s, s_ega, L, s_nodes, s_cd + r, kRows, key_bh, a.dk, cc);
        *reinterpret_cast<float4*>(a.S_new + off) = o;
    }
}

}  // namespace

cudaError_t launch_commit(const CommitArgs& a, int dtype, cudaStream_t s) {
    dim3 grid(a.B * a.H, (a.dv + kRows - 1) / kRows);
    if (dtype == GDN_DTYPE_F32)
        commit_kernel<float><<<grid, kThreads, 0, s>>>(a);
    else
        commit_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn
