// gdn_hybrid.cu -- chain-decomposed tree verification: serial within chains,
// parallel across the chains that are ready.
//
// Review of SpecLA (pith.science 7ERME3HB): "What carries the argument" names
// serial chains with the state split along d_v, beside the factorized tree
// form, and the Referee Report's Fig. 6 discussion contrasts them on deep,
// narrow trees.  Here the tree is cut into chains: a chain starts at a root or
// at a child of a node with two or more children, and follows only-children
// down to a leaf or a branching node.  Chains whose parent chain is done run
// concurrently, one per warp; inside a chain the gated delta rule runs token by
// token on the state rows held in registers,
//
//     delta_t = beta_t (v_t - alpha_t S k_t),  S <- alpha_t S + delta_t k_t^T,
//     o_t = S q_t,
//
// and a chain that ends at a branching node leaves its state rows in a slot
// for the chains below it.  Every node is computed once, as in the tree
// verifier, and the factor record (delta, k, g, parent) is the same, so
// gdn_commit applies to it unchanged.
//
// One CTA owns kRows rows of one (sequence, head) state; its warps take the
// chains of one level of the chain tree at a time.  A branch state is live
// from the level whose chain writes it to the end of the next level, whose
// chains start from it, so slots are reused level by level, lowest free slot
// first.  The first kSmemSlots slots are in shared memory; the rest spill to
// the caller's workspace, sized for the most branching nodes an N-node tree
// can have, (N - 1) / 2, so every valid tree runs.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kWarps = 4;
constexpr int kRows = 8;             // state rows per CTA; every warp holds all of them for its chain
constexpr int kEPL = kMaxDim / 32;   // state columns per lane
constexpr int kSmemSlots = 8;        // branch-state slots in shared memory (two CTAs per SM at d_k = 256)
constexpr int kChunk = 8;            // chain tokens staged per warp at a time

// a node with >= 2 children uses >= 2 of the N - 1 possible child links, so an
// N-node forest has at most (N - 1) / 2 branching nodes
__host__ __device__ inline int spill_slots(int N) { return max(0, (N - 1) / 2 - kSmemSlots); }

// dynamic smem: branch-state slots [kSmemSlots][kRows][dk] fp32, then per warp
// a token chunk [kChunk][k | q][dk] of the input type
struct HybridSmem {
    int branch, tok, total;
    __host__ __device__ HybridSmem(int dk, int esz)
        : branch(0), tok(kSmemSlots * kRows * dk * 4), total(tok + kWarps * kChunk * 2 * dk * esz) {}
};

// workspace: per CTA (bh, blockIdx.y) spill_slots(N) slots of [kRows][dk] fp32
size_t hybrid_ws_bytes(int B, int N, int H, int dk, int dv) {
    return (size_t)B * H * ((dv + kRows - 1) / kRows) * spill_slots(N) * kRows * dk * sizeof(float);
}

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) hybrid_kernel(VerifyArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const HybridSmem Ls(a.dk, (int)sizeof(T));
    float* s_branch = reinterpret_cast<float*>(smem + Ls.branch);
    __shared__ float s_v[kWarps][kChunk][kRows];
    __shared__ float s_al[kWarps][kChunk], s_be[kWarps][kChunk];
    __shared__ int s_par[kMaxNodes], s_nch[kMaxNodes], s_only[kMaxNodes], s_slot[kMaxNodes];
    __shared__ int s_chain_of[kMaxNodes], s_nodes[kMaxNodes];
    __shared__ int s_coff[kMaxNodes + 1], s_clevel[kMaxNodes], s_order[kMaxNodes], s_loff[kMaxNodes + 2];
    __shared__ float s_g[kMaxNodes];
    __shared__ int s_nc, s_nlev, s_fail;
    const int bh = blockIdx.x, b = bh / a.H, h = bh % a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int N = a.N, dk = a.dk, dv = a.dv;
    const int v0 = blockIdx.y * kRows;

    // this layer's rows into L2 while the previous kernel finishes (read after the wait)
    if (tid < N) {
        const size_t rt = ((size_t)b * N + tid) * a.H + h;
        prefetch_l2(static_cast<const T*>(a.q) + rt * dk, dk * (int)sizeof(T));
        prefetch_l2(static_cast<const T*>(a.k) + rt * dk, dk * (int)sizeof(T));
    }
    griddep_wait();
    griddep_launch();

    if (tid < N) {
        s_par[tid] = a.parent[(size_t)b * N + tid];
        s_nch[tid] = 0;
        s_only[tid] = -1;
    }
    __syncthreads();
    if (tid == 0) {
        // chain decomposition (N <= 64 nodes, one thread)
        int fail = 0;
        for (int t = 0; t < N; ++t) {
            const int p = s_par[t];
            if (p < -1 || p >= t) fail = GDN_ERR_TREE;
            else if (p >= 0) {
                ++s_nch[p];
                s_only[p] = t;
            }
        }
        int nc = 0, off = 0, nlev = 0;
        if (!fail) {
            for (int t = 0; t < N; ++t) {
                const int p = s_par[t];
                if (p >= 0 && s_nch[p] < 2) continue;     // continues its parent's chain
                const int c = nc++;
                s_coff[c] = off;
                s_clevel[c] = p < 0 ? 0 : s_clevel[s_chain_of[p]] + 1;
                nlev = max(nlev, s_clevel[c] + 1);
                for (int u = t;; u = s_only[u]) {
                    s_nodes[off++] = u;
                    s_chain_of[u] = c;
                    if (s_nch[u] != 1) break;
                }
            }
            s_coff[nc] = off;
            // chains ordered by level (counting sort)
            for (int l = 0; l <= nlev; ++l) s_loff[l] = 0;
            for (int c = 0; c < nc; ++c) ++s_loff[s_clevel[c] + 1];
            for (int l = 0; l < nlev; ++l) s_loff[l + 1] += s_loff[l];
            int fill[kMaxNodes + 1];
            for (int l = 0; l <= nlev; ++l) fill[l] = s_loff[l];
            for (int c = 0; c < nc; ++c) s_order[fill[s_clevel[c]]++] = c;
            // slots of the branch states: those written at level l are read at level l + 1, so
            // they are taken while the level l - 1 ones are still held and freed after level l + 1
            const int nslots = kSmemSlots + spill_slots(N);
            unsigned long long busy = 0ull;
            for (int t = 0; t < N; ++t) s_slot[t] = -1;
            for (int l = 0; l < nlev && !fail; ++l) {
                for (int ci = s_loff[l]; ci < s_loff[l + 1]; ++ci) {
                    const int u = s_nodes[s_coff[s_order[ci] + 1] - 1];
                    if (s_nch[u] < 2) continue;
                    const int sl = __ffsll((long long)~busy) - 1;
                    if (sl < 0 || sl >= nslots) {             // cannot happen for a valid tree
                        fail = GDN_ERR_CAPACITY;
                        break;
                    }
                    busy |= 1ull << sl;
                    s_slot[u] = sl;
                }
                if (l >= 1)
                    for (int ci = s_loff[l - 1]; ci < s_loff[l]; ++ci) {
                        const int u = s_nodes[s_coff[s_order[ci] + 1] - 1];
                        if (s_slot[u] >= 0) busy &= ~(1ull << s_slot[u]);
                    }
            }
        }
        s_nc = nc;
        s_nlev = nlev;
        s_fail = fail;
        if (fail) set_error(a.err, fail);
    }
    __syncthreads();
    if (s_fail) return;

    const T* qg = static_cast<const T*>(a.q);
    const T* kg = static_cast<const T*>(a.k);
    const T* vg = static_cast<const T*>(a.v);
    T* tok = reinterpret_cast<T*>(smem + Ls.tok) + (size_t)warp * kChunk * 2 * dk;
    const int rowb = dk * (int)sizeof(T);
    // slot i: shared memory below kSmemSlots, else this CTA's part of the workspace
    float* const spill = reinterpret_cast<float*>(a.ws) +
                         ((size_t)bh * gridDim.y + blockIdx.y) * spill_slots(N) * kRows * dk;
    auto slot_rows = [&](int i) -> float* {
        return i < kSmemSlots ? s_branch + (size_t)i * kRows * dk : spill + (size_t)(i - kSmemSlots) * kRows * dk;
    };

    for (int lvl = 0; lvl < s_nlev; ++lvl) {
        for (int ci = s_loff[lvl] + warp; ci < s_loff[lvl + 1]; ci += kWarps) {
            const int c = s_order[ci];
            const int first = s_nodes[s_coff[c]], len = s_coff[c + 1] - s_coff[c];
            const int p = s_par[first];
            float S[kRows][kEPL];
            if (p < 0) {
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    const float* row = a.S + ((size_t)bh * dv + v0 + r) * dk;
#pragma unroll
                    for (int e = 0; e < kEPL; ++e) {
                        const int cc = lane + 32 * e;
                        S[r][e] = (v0 + r < dv && cc < dk) ? row[cc] : 0.f;
                    }
                }
            } else {
                const float* st = slot_rows(s_slot[p]);
#pragma unroll
                for (int r = 0; r < kRows; ++r)
#pragma unroll
                    for (int e = 0; e < kEPL; ++e) {
                        const int cc = lane + 32 * e;
                        S[r][e] = cc < dk ? st[r * dk + cc] : 0.f;
                    }
            }
            float g = p < 0 ? 0.f : s_g[p];
            for (int c0 = 0; c0 < len; c0 += kChunk) {
                const int n = min(kChunk, len - c0);
                __syncwarp();                              // the previous chunk is consumed
                for (int i = 0; i < n; ++i) {
                    const size_t gi = ((size_t)b * N + s_nodes[s_coff[c] + c0 + i]) * a.H + h;
                    for (int o = lane * 16; o < rowb; o += 32 * 16) {
                        cp_async16(reinterpret_cast<char*>(tok + (size_t)(2 * i) * dk) + o,
                                   reinterpret_cast<const char*>(kg + gi * dk) + o);
                        cp_async16(reinterpret_cast<char*>(tok + (size_t)(2 * i + 1) * dk) + o,
                                   reinterpret_cast<const char*>(qg + gi * dk) + o);
                    }
                }
                for (int idx = lane; idx < n * kRows; idx += 32) {
                    const int i = idx / kRows, r = idx % kRows;
                    const size_t gi = ((size_t)b * N + s_nodes[s_coff[c] + c0 + i]) * a.H + h;
                    s_v[warp][i][r] = v0 + r < dv ? ld_elem<T>(vg, gi * dv + v0 + r) : 0.f;
                }
                if (lane < n) {
                    const size_t gi = ((size_t)b * N + s_nodes[s_coff[c] + c0 + lane]) * a.H + h;
                    s_al[warp][lane] = a.alpha[gi];
                    s_be[warp][lane] = a.beta[gi];
                }
                cp_async_wait_all();
                __syncwarp();
                for (int i = 0; i < n; ++i) {
                    const int t = s_nodes[s_coff[c] + c0 + i];
                    float kt[kEPL], qt[kEPL];
                    float kq = 0.f;
#pragma unroll
                    for (int e = 0; e < kEPL; ++e) {
                        const int cc = lane + 32 * e;
                        kt[e] = cc < dk ? ld_elem<T>(tok, (size_t)(2 * i) * dk + cc) : 0.f;
                        qt[e] = cc < dk ? ld_elem<T>(tok, (size_t)(2 * i + 1) * dk + cc) : 0.f;
                        kq = fmaf(kt[e], qt[e], kq);
                    }
                    float sk[kRows], sq[kRows];
#pragma unroll
                    for (int r = 0; r < kRows; ++r) {
                        float x = 0.f, y = 0.f;
#pragma unroll
                        for (int e = 0; e < kEPL; ++e) {
                            x = fmaf(S[r][e], kt[e], x);
                            y = fmaf(S[r][e], qt[e], y);
                        }
                        sk[r] = x;
                        sq[r] = y;
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        kq += __shfl_xor_sync(0xffffffffu, kq, o);
#pragma unroll
                        for (int r = 0; r < kRows; ++r) {
                            sk[r] += __shfl_xor_sync(0xffffffffu, sk[r], o);
                            sq[r] += __shfl_xor_sync(0xffffffffu, sq[r], o);
                        }
                    }
                    const float al = s_al[warp][i], be = s_be[warp][i];
                    g += logf(al);
                    float outv = 0.f, d_lane = 0.f;
#pragma unroll
                    for (int r = 0; r < kRows; ++r) {
                        const float dlt = be * (s_v[warp][i][r] - al * sk[r]);
#pragma unroll
                        for (int e = 0; e < kEPL; ++e) S[r][e] = fmaf(al, S[r][e], dlt * kt[e]);
                        const float o = fmaf(al, sq[r], dlt * kq);
                        if (lane == r) {
                            outv = o;
                            d_lane = dlt;
                        }
                    }
                    if (lane < kRows && v0 + lane < dv) {
                        a.out[(((size_t)b * N + t) * a.H + h) * dv + v0 + lane] = outv;
                        a.f.delta[((size_t)bh * N + t) * dv + v0 + lane] = d_lane;
                    }
                    if (lane == 0) s_g[t] = g;
                }
            }
            const int last = s_nodes[s_coff[c + 1] - 1];
            if (s_slot[last] >= 0) {                  // branching node: rows for the chains below
                float* st = slot_rows(s_slot[last]);
#pragma unroll
                for (int r = 0; r < kRows; ++r)
#pragma unroll
                    for (int e = 0; e < kEPL; ++e) {
                        const int cc = lane + 32 * e;
                        if (cc < dk) st[r * dk + cc] = S[r][e];
                    }
            }
            __syncwarp();
        }
        __syncthreads();
    }

    // rest of the factor record: g, keys and parents, spread over the CTAs of this (b, h)
    if (blockIdx.y == 0 && tid < N) a.f.g[(size_t)bh * N + tid] = s_g[tid];
    if (blockIdx.y == 0 && h == 0 && tid < N) a.f.parent[(size_t)b * N + tid] = s_par[tid];
    T* key_out = static_cast<T*>(a.f.key);
    for (int t = blockIdx.y; t < N; t += gridDim.y) {
        const size_t gi = ((size_t)b * N + t) * a.H + h;
        for (int c = tid; c < dk; c += kWarps * 32) key_out[((size_t)bh * N + t) * dk + c] = kg[gi * dk + c];
    }
}

template <typename T>
cudaError_t launch_hybrid_t(const VerifyArgs& a, cudaStream_t s) {
    static int attr_set[64];    // dynamic shared memory opted into, per device (the kernel also has static)
    const HybridSmem L(a.dk, (int)sizeof(T));
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (L.total > 48 * 1024 && attr_set[dev] < L.total) {
        e = cudaFuncSetAttribute(hybrid_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
        if (e != cudaSuccess) return e;
        attr_set[dev] = L.total;
    }
    dim3 grid(a.B * a.H, (a.dv + kRows - 1) / kRows);
    return launch_kernel(hybrid_kernel<T>, grid, dim3(kWarps * 32), L.total, s, a.overlap, a);
}

}  // namespace

}  // namespace gdn

using namespace gdn;

extern "C" int gdn_hybrid_workspace_bytes(int B, int N, int H, int dk, int dv, size_t* bytes) {
    auto dim_ok = [](int d) { return d >= 16 && d <= kMaxDim && d % 16 == 0; };
    if (bytes == nullptr || B < 1 || H < 1 || N < 1 || N > kMaxNodes || !dim_ok(dk) || !dim_ok(dv) ||
        (long long)B * H > 0x7fffffffLL)
        return GDN_ERR_ARG;
    *bytes = hybrid_ws_bytes(B, N, H, dk, dv);
    return GDN_OK;
}

extern "C" int gdn_hybrid_tree_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                                      const float* beta, const int32_t* parent_idx, const float* S0, float* out,
                                      void* factors, void* workspace, int B, int N, int H, int dk, int dv,
                                      cudaStream_t stream) {
    auto ok16 = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    auto dim_ok = [](int d) { return d >= 16 && d <= kMaxDim && d % 16 == 0; };
    if (B < 1 || H < 1 || N < 1 || N > kMaxNodes || !dim_ok(dk) || !dim_ok(dv) || (long long)B * H > 0x7fffffffLL)
        return GDN_ERR_ARG;
    if (dtype != GDN_DTYPE_BF16 && dtype != GDN_DTYPE_F32) return GDN_ERR_ARG;
    if (!ok16(q) || !ok16(k) || !ok16(v) || !ok16(alpha) || !ok16(beta) || !ok16(parent_idx) || !ok16(S0) ||
        !ok16(out) || !ok16(factors))
        return GDN_ERR_ARG;
    const size_t wbytes = hybrid_ws_bytes(B, N, H, dk, dv);
    if (wbytes > 0 && !ok16(workspace)) return GDN_ERR_ARG;
    const size_t fbytes = factor_layout(B, N, H, dk, dv, dtype).total;
    const size_t obytes = (size_t)B * N * H * dv * 4;
    const char* o = reinterpret_cast<const char*>(out);
    const char* f = static_cast<const char*>(factors);
    const char* w = static_cast<const char*>(workspace);
    if (o < f + fbytes && f < o + obytes) return GDN_ERR_ARG;
    if (wbytes > 0 && ((o < w + wbytes && w < o + obytes) || (f < w + wbytes && w < f + fbytes))) return GDN_ERR_ARG;
    int st = GDN_OK;
    int* err = current_error_word(&st);
    if (err == nullptr) return st;
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
    a.ws = wbytes > 0 ? static_cast<char*>(workspace) : nullptr;
    a.B = B;
    a.N = N;
    a.H = H;
    a.dk = dk;
    a.dv = dv;
    a.commit = CommitSrc{nullptr, nullptr, nullptr, nullptr, 0, nullptr, 0};
    a.err = err;
    a.overlap = launch_overlap_enabled();
    a.tc = false;
    const cudaError_t e = dtype == GDN_DTYPE_F32 ? launch_hybrid_t<float>(a, stream)
                                                 : launch_hybrid_t<__nv_bfloat16>(a, stream);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
