// gdn_prune.cu -- confidence-guided pruning of draft trees before verification.
//
// Review of SpecLA (pith.science 7ERME3HB) names confidence-guided tree pruning
// with a tree margin tau_tree and a draft budget (Referee Report, comment on
// Section 6.1) without defining them.  The rule here, per sequence:
//   score(t) = logp_t + score(parent(t))          (root first, fp32)
//   t survives if score(t) >= fl(max_{siblings s} score(s) - tau) and its
//   parent survives; of the survivors, the `budget` best scores are kept (ties
//   to the lower index) -- an ancestor-closed set, since log-probabilities are
//   <= 0; the kept nodes are renumbered in their original order.
// One CTA (64 threads) per sequence; every step is a level-synchronous or an
// O(N) scan over at most 64 nodes in shared memory.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

struct PruneArgs {
    const int32_t* parent;     // [B][N]
    const float* logp;         // [B][N]
    float tau;
    int budget;
    int32_t* new_index;        // [B][N]
    int32_t* new_parent;       // [B][N], rows past n_kept set to -1
    int32_t* n_kept;           // [B]
    int B, N;
    int* err;
};

__global__ void __launch_bounds__(kMaxNodes) prune_kernel(PruneArgs a) {
    __shared__ int par[kMaxNodes], depth[kMaxNodes], alive[kMaxNodes], keep[kMaxNodes], idx[kMaxNodes];
    __shared__ float sc[kMaxNodes], lp[kMaxNodes];
    __shared__ int s_bad, s_maxdepth;
    const int b = blockIdx.x, t = threadIdx.x, N = a.N;
    griddep_wait();
    griddep_launch();
    if (t == 0) {
        s_bad = 0;
        s_maxdepth = 0;
    }
    __syncthreads();
    if (t < N) {
        par[t] = a.parent[(size_t)b * N + t];
        lp[t] = a.logp[(size_t)b * N + t];
        if (par[t] < -1 || par[t] >= t) s_bad = 1;
    }
    __syncthreads();
    if (s_bad) {
        if (t == 0) set_error(a.err, GDN_ERR_TREE);
        return;
    }
    if (t < N) {
        int d = 0;
        for (int u = par[t]; u >= 0; u = par[u]) ++d;
        depth[t] = d;
        atomicMax(&s_maxdepth, d);
    }
    __syncthreads();
    const int md = s_maxdepth;
    for (int d = 0; d <= md; ++d) {                 // scores, root first
        if (t < N && depth[t] == d) sc[t] = lp[t] + (par[t] >= 0 ? sc[par[t]] : 0.f);
        __syncthreads();
    }
    bool ok = false;
    if (t < N) {
        float best = sc[t];
        for (int u = 0; u < N; ++u)
            if (par[u] == par[t]) best = fmaxf(best, sc[u]);
        ok = sc[t] >= best - a.tau;
    }
    for (int d = 0; d <= md; ++d) {                 // margin survivors, closed under ancestors
        if (t < N && depth[t] == d) alive[t] = ok && (par[t] < 0 || alive[par[t]]);
        __syncthreads();
    }
    if (t < N) {
        int rank = 0;
        if (alive[t])
            for (int u = 0; u < N; ++u)
                rank += alive[u] && (sc[u] > sc[t] || (sc[u] == sc[t] && u < t));
        keep[t] = alive[t] && rank < a.budget;
    }
    __syncthreads();
    if (t < N) {
        int i = 0;
        for (int u = 0; u < t; ++u) i += keep[u];
        idx[t] = keep[t] ? i : -1;
    }
    __syncthreads();
    if (t < N) {
        a.new_index[(size_t)b * N + t] = idx[t];
        a.new_parent[(size_t)b * N + t] = -1;
    }
    __syncthreads();
    if (t < N && keep[t]) a.new_parent[(size_t)b * N + idx[t]] = par[t] >= 0 ? idx[par[t]] : -1;
    if (t == 0) {
        int n = 0;
        for (int u = 0; u < N; ++u) n += keep[u];
        a.n_kept[b] = n;
    }
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" int gdn_prune_tree(const int32_t* parent_idx, const float* logp, float tau, int budget,
                              int32_t* new_index, int32_t* new_parent, int32_t* n_kept, int B, int N,
                              cudaStream_t stream) {
    auto ok16 = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (B < 1 || N < 1 || N > kMaxNodes || budget < 0 || tau != tau) return GDN_ERR_ARG;
    if (!ok16(parent_idx) || !ok16(logp) || !ok16(new_index) || !ok16(new_parent) || !ok16(n_kept))
        return GDN_ERR_ARG;
    int st = GDN_OK;
    int* err = current_error_word(&st);
    if (err == nullptr) return st;
    const PruneArgs a{parent_idx, logp, tau, budget, new_index, new_parent, n_kept, B, N, err};
    return launch_kernel(prune_kernel, dim3(B), dim3(kMaxNodes), 0, stream, false, a) == cudaSuccess ? GDN_OK
                                                                                                 : GDN_ERR_CUDA;
}
