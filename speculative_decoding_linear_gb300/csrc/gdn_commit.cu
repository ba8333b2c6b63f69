// gdn_commit.cu -- accepted-path commit from buffered factors.
//
// Review of SpecLA (pith.science 7ERME3HB), Referee Report summary: the state
// after the accepted tokens is rebuilt from the small records kept per draft
// node, with no snapshot and no replay.  With the factor record (delta, k, g)
// of every verified node, the state after accepting the
// root-first path ending at node a is a rank-L update of the committed state:
//
//     S_a = e^{g_a} S0 + sum_{j on path(a)} e^{g_a - g_j} delta_j k_j^T
//
// (unrolling S_t = alpha_t S_parent + delta_t k_t^T along the path).  The
// kernel is a pure stream over S: read 4 B and write 4 B per state element,
// L FMAs each from on-chip coefficients.  One CTA owns kRows rows of one
// (sequence, head) state; threads own 16-byte column quads (coalesced).  The
// state loads are issued first, the path's factor rows are staged with
// cp.async meanwhile, and all writes come after the programmatic wait.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kRows = 16;
constexpr int kThreads = 256;
constexpr int kItems = kRows * (kMaxDim / 4) / kThreads;   // float4 per thread (d_k = 256)

struct CommitSmem {
    int key, cd, coef, nodes, misc, total;
    __host__ __device__ CommitSmem(int dk, int Lcap, int esz) {
        int off = 0;
        auto take = [&](int bytes) { int o = off; off += (bytes + 15) / 16 * 16; return o; };
        key = take(Lcap * dk * esz);
        cd = take(Lcap * kRows * 4);
        coef = take(kMaxPath * 4);
        nodes = take(kMaxPath * 4);
        misc = take(16);
        total = off;
    }
};

template <typename KT>
__global__ void __launch_bounds__(kThreads) commit_kernel(CommitArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const CommitSrc& c = a.src;
    const CommitSmem Ly(a.dk, c.Lmax, (int)sizeof(KT));
    KT* s_key = reinterpret_cast<KT*>(smem + Ly.key);
    float* s_cd = reinterpret_cast<float*>(smem + Ly.cd);
    float* s_coef = reinterpret_cast<float*>(smem + Ly.coef);
    int* s_nodes = reinterpret_cast<int*>(smem + Ly.nodes);
    float* s_ega = reinterpret_cast<float*>(smem + Ly.misc);
    int* s_L = reinterpret_cast<int*>(smem + Ly.misc + 4);

    const int bh = blockIdx.x, tid = threadIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int v0 = blockIdx.y * kRows;
    const int rows = min(kRows, a.dv - v0);
    const int quads = a.dk / 4;
    const size_t base = ((size_t)bh * a.dv + v0) * a.dk;

    float4 x[kItems];
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        const int i = tid + j * kThreads;
        const int r = i / quads;
        x[j] = (r < rows) ? *reinterpret_cast<const float4*>(a.S0 + base + (size_t)i * 4)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid < 32) {
        const int L = commit_path_setup(c, b, h, a.H, s_nodes, s_coef, s_ega);
        if (tid == 0) {
            *s_L = L;
            if (L < 0) set_error(a.err, GDN_ERR_PATH);
        }
    }
    __syncthreads();
    const int L = *s_L;
    if (L < 0) return;
    const KT* key_bh = static_cast<const KT*>(c.key) + (size_t)bh * c.N * a.dk;
    for (int i = 0; i < L; ++i)
        cp_async_block(s_key + (size_t)i * a.dk, key_bh + (size_t)s_nodes[i] * a.dk,
                       a.dk * (int)sizeof(KT), tid, kThreads);
    const float* delta_bh = c.delta + (size_t)bh * c.N * a.dv;
    for (int i = tid; i < L * kRows; i += kThreads) {
        const int j = i / kRows, r = i % kRows;
        s_cd[i] = r < rows ? s_coef[j] * delta_bh[(size_t)s_nodes[j] * a.dv + v0 + r] : 0.f;
    }
    cp_async_wait_all();
    __syncthreads();
    const float ega = *s_ega;
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        const int i = tid + j * kThreads;
        const int r = i / quads, cc = (i % quads) * 4;
        if (r < rows) x[j] = commit_quad<KT>(x[j], ega, L, s_cd + r, kRows, s_key, a.dk, cc);
    }
    griddep_wait();
    griddep_launch();
#pragma unroll
    for (int j = 0; j < kItems; ++j) {
        const int i = tid + j * kThreads;
        if (i / quads < rows) *reinterpret_cast<float4*>(a.S_new + base + (size_t)i * 4) = x[j];
    }
}

}  // namespace

cudaError_t launch_commit(const CommitArgs& a, int dtype, cudaStream_t s) {
    static bool attr_f[64], attr_b[64];
    const CommitSmem Ly(a.dk, a.src.Lmax, dtype == GDN_DTYPE_F32 ? 4 : 2);
    dim3 grid(a.B * a.H, (a.dv + kRows - 1) / kRows);
    if (dtype == GDN_DTYPE_F32) {
        cudaError_t e = ensure_smem(commit_kernel<float>, Ly.total, attr_f);
        if (e != cudaSuccess) return e;
        return launch_kernel(commit_kernel<float>, grid, dim3(kThreads), Ly.total, s, a.overlap, a);
    }
    cudaError_t e = ensure_smem(commit_kernel<__nv_bfloat16>, Ly.total, attr_b);
    if (e != cudaSuccess) return e;
    return launch_kernel(commit_kernel<__nv_bfloat16>, grid, dim3(kThreads), Ly.total, s, a.overlap, a);
}

}  // namespace gdn
