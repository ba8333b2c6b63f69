// gdn_replay.cu -- the replay baselines that tree verification and the
// factor-buffer commit replace (review of SpecLA, pith.science 7ERME3HB:
// "Core claim" compares the tree verifier against replaying every
// root-to-leaf path, and accepted-state recovery from buffered factors
// against replaying the accepted tokens).
//
//   replay verify  every leaf's root-to-leaf path is run token by token with
//                  the gated delta rule from S0, writing o_t for each node on
//                  it; nodes shared by several leaves are recomputed by each
//   replay commit  the accepted path is run token by token from S0 and the
//                  final state is written to S_new
//
// One CTA holds kRows rows of one (sequence, head) state in registers (each
// warp RPW rows, each lane d_k/32 interleaved columns), like the chain kernel,
// and replays one leaf's path (or the accepted path) from its S0 rows, the
// path's tokens staged in shared memory eight at a time.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kWarps = 4;
constexpr int kRPW = 4;
constexpr int kRows = kWarps * kRPW;
constexpr int kEPL = kMaxDim / 32;
constexpr int kChunk = 8;          // path tokens staged in shared memory at a time

struct ReplayArgs {
    const void* q;             // nullptr in commit mode
    const void* k;
    const void* v;
    const float* alpha;
    const float* beta;
    const int32_t* parent;
    const float* S0;
    float* out;                // verify mode: [B][N][H][dv]
    const int32_t* path;       // commit mode: [B][Lmax]; nullptr in verify mode
    int Lmax;
    float* S_new;              // commit mode
    int B, N, H, dk, dv;
    int* err;
};

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) replay_kernel(ReplayArgs a) {
    __shared__ int s_par[kMaxNodes];
    __shared__ int s_path[kMaxNodes];
    __shared__ int s_len;
    const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int N = a.N, dk = a.dk, dv = a.dv;
    const int v0 = blockIdx.y * kRows;
    const bool commit = a.path != nullptr;
    griddep_wait();
    griddep_launch();

    __shared__ int s_leaves[kMaxNodes];
    __shared__ int s_nl;
    __shared__ int s_haschild[kMaxNodes];
    if (tid < kMaxNodes) s_haschild[tid] = 0;
    if (tid < N) s_par[tid] = a.parent[(size_t)b * N + tid];
    __syncthreads();
    bool bad = false;
    if (tid < N) {
        const int p = s_par[tid];
        bad = p < -1 || p >= tid;
        if (!bad && p >= 0) s_haschild[p] = 1;
    }
    bad = __syncthreads_or(bad);
    if (warp == 0) {                           // leaves in ascending order, compacted by ballots
        int nl = 0;
        if (commit) {
            nl = 1;
        } else if (!bad) {
            for (int c = 0; c < N; c += 32) {
                const int t = c + lane;
                const bool leaf = t < N && s_haschild[t] == 0;
                const unsigned m = __ballot_sync(0xffffffffu, leaf);
                if (leaf) s_leaves[nl + __popc(m & ((1u << lane) - 1u))] = t;
                nl += __popc(m);
            }
        } else if (lane == 0) {
            set_error(a.err, GDN_ERR_TREE);
        }
        if (lane == 0) s_nl = nl;
    }
    __syncthreads();
    const int nl = s_nl;

    float S[kRPW][kEPL];
    const T* qg = static_cast<const T*>(a.q);
    const T* kg = static_cast<const T*>(a.k);
    const T* vg = static_cast<const T*>(a.v);
    // the path's tokens are staged kChunk at a time: k and q rows by cp.async,
    // this CTA's v entries, alpha and beta
    __shared__ __align__(16) unsigned char s_tok[kChunk * 2 * kMaxDim * 4];
    __shared__ float s_v[kChunk][kRows];
    __shared__ float s_al[kChunk], s_be[kChunk];
    T* tok = reinterpret_cast<T*>(s_tok);
    const int rowb = dk * (int)sizeof(T);
    for (int li = blockIdx.z; li < nl; li += gridDim.z) {
    __syncthreads();                           // the previous path is consumed
    if (tid == 0) {
        int len = 0;
        if (commit) {
            const int32_t* p = a.path + (size_t)b * a.Lmax;
            int prev = -1;
            for (; len < a.Lmax && p[len] >= 0; ++len) {
                const int t = p[len];
                if (t >= N || s_par[t] != prev) {
                    set_error(a.err, GDN_ERR_PATH);
                    len = -1;
                    break;
                }
                s_path[len] = t;
                prev = t;
            }
        } else {
            int n = 0;
            for (int t = s_leaves[li]; t >= 0; t = s_par[t]) ++n;
            int i = n;
            for (int t = s_leaves[li]; t >= 0; t = s_par[t]) s_path[--i] = t;
            len = n;
        }
        s_len = len;
    }
    __syncthreads();
    const int len = s_len;
    if (len < 0) return;
#pragma unroll
    for (int rr = 0; rr < kRPW; ++rr) {
        const int r = v0 + warp * kRPW + rr;
        const float* row = a.S0 + ((size_t)bh * dv + r) * dk;
#pragma unroll
        for (int e = 0; e < kEPL; ++e) {
            const int c = lane + 32 * e;
            S[rr][e] = (r < dv && c < dk) ? row[c] : 0.f;
        }
    }
    for (int c0 = 0; c0 < len; c0 += kChunk) {
        const int n = min(kChunk, len - c0);
        __syncthreads();                       // the previous chunk is consumed
        for (int i = 0; i < n; ++i) {
            const size_t gi = ((size_t)b * N + s_path[c0 + i]) * a.H + h;
            cp_async_block(tok + (size_t)(2 * i) * dk, kg + gi * dk, rowb, tid, kWarps * 32);
            if (!commit) cp_async_block(tok + (size_t)(2 * i + 1) * dk, qg + gi * dk, rowb, tid, kWarps * 32);
        }
        for (int idx = tid; idx < n * kRows; idx += kWarps * 32) {
            const int i = idx / kRows, r = idx % kRows;
            const size_t gi = ((size_t)b * N + s_path[c0 + i]) * a.H + h;
            s_v[i][r] = v0 + r < dv ? ld_elem<T>(vg, gi * dv + v0 + r) : 0.f;
        }
        if (tid < n) {
            const size_t gi = ((size_t)b * N + s_path[c0 + tid]) * a.H + h;
            s_al[tid] = a.alpha[gi];
            s_be[tid] = a.beta[gi];
        }
        cp_async_wait_all();
        __syncthreads();
        for (int i = 0; i < n; ++i) {
            const int t = s_path[c0 + i];
            float kt[kEPL], qt[kEPL];
            float kq = 0.f;
#pragma unroll
            for (int e = 0; e < kEPL; ++e) {
                const int c = lane + 32 * e;
                kt[e] = c < dk ? ld_elem<T>(tok, (size_t)(2 * i) * dk + c) : 0.f;
                qt[e] = (!commit && c < dk) ? ld_elem<T>(tok, (size_t)(2 * i + 1) * dk + c) : 0.f;
                kq = fmaf(kt[e], qt[e], kq);
            }
            float sk[kRPW], sq[kRPW];
#pragma unroll
            for (int rr = 0; rr < kRPW; ++rr) {
                float x = 0.f, y = 0.f;
#pragma unroll
                for (int e = 0; e < kEPL; ++e) {
                    x = fmaf(S[rr][e], kt[e], x);
                    y = fmaf(S[rr][e], qt[e], y);
                }
                sk[rr] = x;
                sq[rr] = y;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                kq += __shfl_xor_sync(0xffffffffu, kq, o);
#pragma unroll
                for (int rr = 0; rr < kRPW; ++rr) {
                    sk[rr] += __shfl_xor_sync(0xffffffffu, sk[rr], o);
                    sq[rr] += __shfl_xor_sync(0xffffffffu, sq[rr], o);
                }
            }
            const float al = s_al[i], be = s_be[i];
#pragma unroll
            for (int rr = 0; rr < kRPW; ++rr) {
                const int rl = warp * kRPW + rr, r = v0 + rl;
                const float dlt = be * (s_v[i][rl] - al * sk[rr]);
#pragma unroll
                for (int e = 0; e < kEPL; ++e) S[rr][e] = fmaf(al, S[rr][e], dlt * kt[e]);
                if (!commit && lane == 0 && r < dv)
                    a.out[(((size_t)b * N + t) * a.H + h) * dv + r] = fmaf(al, sq[rr], dlt * kq);
            }
        }
    }
    }
    if (commit) {
#pragma unroll
        for (int rr = 0; rr < kRPW; ++rr) {
            const int r = v0 + warp * kRPW + rr;
            float* row = a.S_new + ((size_t)bh * dv + r) * dk;
#pragma unroll
            for (int e = 0; e < kEPL; ++e) {
                const int c = lane + 32 * e;
                if (r < dv && c < dk) row[c] = S[rr][e];
            }
        }
    }
}

bool ok16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool shape_ok(int B, int N, int H, int dk, int dv) {
    auto dim_ok = [](int d) { return d >= 16 && d <= kMaxDim && d % 16 == 0; };
    return B >= 1 && H >= 1 && N >= 1 && N <= kMaxNodes && dim_ok(dk) && dim_ok(dv) && (long long)B * H < 65536LL * 32768;
}

cudaError_t launch_replay(const ReplayArgs& a, int dtype, cudaStream_t s) {
    // verify: one leaf per CTA along z (CTAs past the tree's leaf count exit at once)
    dim3 grid(a.B * a.H, (a.dv + kRows - 1) / kRows, a.path != nullptr ? 1 : a.N);
    return dtype == GDN_DTYPE_F32 ? launch_kernel(replay_kernel<float>, grid, dim3(kWarps * 32), 0, s, false, a)
                                  : launch_kernel(replay_kernel<__nv_bfloat16>, grid, dim3(kWarps * 32), 0, s, false, a);
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" int gdn_replay_tree_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                                      const float* beta, const int32_t* parent_idx, const float* S0, float* out, int B,
                                      int N, int H, int dk, int dv, cudaStream_t stream) {
    if (!shape_ok(B, N, H, dk, dv) || (dtype != GDN_DTYPE_BF16 && dtype != GDN_DTYPE_F32)) return GDN_ERR_ARG;
    if (!ok16(q) || !ok16(k) || !ok16(v) || !ok16(alpha) || !ok16(beta) || !ok16(parent_idx) || !ok16(S0) || !ok16(out))
        return GDN_ERR_ARG;
    int st = GDN_OK;
    int* err = current_error_word(&st);
    if (err == nullptr) return st;
    ReplayArgs a{q, k, v, alpha, beta, parent_idx, S0, out, nullptr, 0, nullptr, B, N, H, dk, dv, err};
    return launch_replay(a, dtype, stream) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" int gdn_replay_commit(const void* k, const void* v, int dtype, const float* alpha, const float* beta,
                                 const int32_t* parent_idx, const float* S0, const int32_t* accepted_path, int Lmax,
                                 float* S_new, int B, int N, int H, int dk, int dv, cudaStream_t stream) {
    if (!shape_ok(B, N, H, dk, dv) || (dtype != GDN_DTYPE_BF16 && dtype != GDN_DTYPE_F32)) return GDN_ERR_ARG;
    if (Lmax < 1 || Lmax > kMaxNodes) return GDN_ERR_ARG;
    if (!ok16(k) || !ok16(v) || !ok16(alpha) || !ok16(beta) || !ok16(parent_idx) || !ok16(S0) ||
        !ok16(accepted_path) || !ok16(S_new))
        return GDN_ERR_ARG;
    const size_t sb = (size_t)B * H * dv * dk * 4;
    const char* x = reinterpret_cast<const char*>(S0);
    const char* y = reinterpret_cast<const char*>(S_new);
    if (x != y && x < y + sb && y < x + sb) return GDN_ERR_ARG;   // in place or disjoint
    int st = GDN_OK;
    int* err = current_error_word(&st);
    if (err == nullptr) return st;
    ReplayArgs a{nullptr, k, v, alpha, beta, parent_idx, S0, nullptr, accepted_path, Lmax, S_new, B, N, H, dk, dv, err};
    return launch_replay(a, dtype, stream) == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
