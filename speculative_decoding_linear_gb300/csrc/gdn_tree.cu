// gdn_tree.cu -- tree-masked factorized verification (SIMT path).
//
// Review of SpecLA (pith.science 7ERME3HB), "Core claim": A_tree = M_tree (.)
// (K_b K_a^T), T_tree = solve_tril(I - A_tree), O = Qhat S0^T - Attn (W S0^T)
// + Attn U.  Per (sequence b, head h), with g_t the cumulative log gate along
// path(t) and anc(t) the strict ancestors of t:
//
//   A[t,j]    = beta_t e^{g_t - g_j} (k_t . k_j),  j in anc(t)     (0 elsewhere)
//   Attn[t,j] =        e^{g_t - g_j} (q_t . k_j),  j in path(t)
//   T         = (I + A)^-1        (unit lower triangular, nonzero only on the
//                                  inclusive ancestor mask)
//   R         = diag(beta) (V - diag(e^g) K S0^T)
//   Delta     = T R               (= U - W S0^T with U = T diag(beta) V,
//                                  W = T diag(beta e^g) K)
//   O         = diag(e^g) Q S0^T + Attn Delta = diag(e^g) Q S0^T + (Attn T) R
//
// Because T and Attn T live on the ancestor mask, row t of Delta and O needs
// only the <= depth(t)+1 rows of R on path(t): the "N x N" products are short
// gathers along each node's path.
//
// Two kernels:
//   tree_prep_kernel      one CTA per (b, h): ancestor masks, gates, the masked
//                         Gram entries, T by depth levels, P = Attn T; writes
//                         the workspace record and the factor record's g,
//                         parent and key sections.
//   tree_contract_kernel  one CTA per (b, h, 32 rows of d_v): streams the S0
//                         tile (applying a pending commit first when fused),
//                         forms Y = [Q; K] S0_tile^T, then R, Delta and O.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

// ---------------------------------------------------------------------------
// ancestor mask + depth (gdn_tree_mask)
// ---------------------------------------------------------------------------
__global__ void tree_mask_kernel(const int32_t* parent, int N, uint64_t* mask, int32_t* depth,
                                 int* err) {
    __shared__ int s_par[kMaxNodes];
    const int b = blockIdx.x, t = threadIdx.x;
    int p = -1;
    bool bad = false;
    if (t < N) {
        p = parent[(size_t)b * N + t];
        bad = p < -1 || p >= t;
        s_par[t] = p;
    }
    if (__syncthreads_or(bad)) {
        if (t == 0) set_error(err, GDN_ERR_TREE);
        return;
    }
    if (t < N) {
        uint64_t m = 0;
        int d = 0;
        for (int j = p; j >= 0; j = s_par[j]) {
            m |= 1ull << j;
            ++d;
        }
        mask[(size_t)b * N + t] = m;
        depth[(size_t)b * N + t] = d;
    }
}

// ---------------------------------------------------------------------------
// per-(b, h) prologue
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 256;
constexpr int kLd = kMaxNodes + 1;   // padded row stride of the N x N tables in smem

struct PrepSmem {
    float A[kMaxNodes * kLd];
    float At[kMaxNodes * kLd];       // Attn
    float T[kMaxNodes * kLd];
    uint64_t anc[kMaxNodes];         // strict ancestors
    float la[kMaxNodes];             // log alpha_t
    float g[kMaxNodes];
    float beta[kMaxNodes];
    int par[kMaxNodes];
    int depth[kMaxNodes];
    int maxdepth;
};

template <typename T>
__global__ void __launch_bounds__(kPrepThreads) tree_prep_kernel(VerifyArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    PrepSmem& s = *reinterpret_cast<PrepSmem*>(smem_raw);
    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int N = a.N, tid = threadIdx.x;
    const WsLayout wl = ws_layout(N);
    char* rec = a.ws + (size_t)bh * wl.record;

    // 1. parents, validated
    bool bad = false;
    if (tid < N) {
        const int p = a.parent[(size_t)b * N + tid];
        bad = p < -1 || p >= tid;
        s.par[tid] = p;
        const size_t gi = ((size_t)b * N + tid) * a.H + h;
        s.la[tid] = logf(a.alpha[gi]);
        s.beta[tid] = a.beta[gi];
    }
    if (tid == 0) s.maxdepth = 0;
    for (int i = tid; i < kMaxNodes * kLd; i += kPrepThreads) s.A[i] = s.At[i] = s.T[i] = 0.f;
    if (__syncthreads_or(bad)) {
        if (tid == 0) {
            set_error(a.err, GDN_ERR_TREE);
            *reinterpret_cast<uint64_t*>(rec + wl.anc) = ~0ull;   // record marked invalid
        }
        return;
    }

    // 2. strict ancestor masks, depths, cumulative log gates (ascending = root first)
    if (tid < N) {
        uint64_t m = 0;
        int d = 0;
        for (int j = s.par[tid]; j >= 0; j = s.par[j]) {
            m |= 1ull << j;
            ++d;
        }
        s.anc[tid] = m;
        s.depth[tid] = d;
        atomicMax(&s.maxdepth, d);
        float gs = 0.f;
        for (uint64_t r = m; r; r &= r - 1) gs += s.la[__ffsll((long long)r) - 1];
        s.g[tid] = gs + s.la[tid];
    }
    __syncthreads();

    // 3. masked Gram entries; one warp per row t, lanes split d_k
    const int warp = tid >> 5, lane = tid & 31;
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    T* key_out = static_cast<T*>(a.f.key);
    for (int t = warp; t < N; t += kPrepThreads / 32) {
        const size_t rt = ((size_t)b * N + t) * a.H + h;
        float kt[kMaxDim / 32], qt[kMaxDim / 32];
#pragma unroll
        for (int e = 0; e < kMaxDim / 32; ++e) {
            const int c = lane + 32 * e;
            const bool in = c < a.dk;
            kt[e] = in ? ld_elem<T>(k, rt * a.dk + c) : 0.f;
            qt[e] = in ? ld_elem<T>(q, rt * a.dk + c) : 0.f;
            if (in) st_elem<T>(key_out, ((size_t)bh * N + t) * a.dk + c, kt[e]);
        }
        const float gt = s.g[t], bt = s.beta[t];
        uint64_t path = s.anc[t] | (1ull << t);
        for (; path; path &= path - 1) {
            const int j = __ffsll((long long)path) - 1;
            const size_t rj = ((size_t)b * N + j) * a.H + h;
            float pkk = 0.f, pqk = 0.f;
#pragma unroll
            for (int e = 0; e < kMaxDim / 32; ++e) {
                const int c = lane + 32 * e;
                const float kj = c < a.dk ? ld_elem<T>(k, rj * a.dk + c) : 0.f;
                pkk = fmaf(kt[e], kj, pkk);
                pqk = fmaf(qt[e], kj, pqk);
            }
            pkk = warp_sum(pkk);
            pqk = warp_sum(pqk);
            if (lane == 0) {
                const float gam = expf(gt - s.g[j]);
                s.At[t * kLd + j] = gam * pqk;
                if (j != t) s.A[t * kLd + j] = bt * gam * pkk;
            }
        }
    }
    __syncthreads();

    // 4. T = (I + A)^-1 by depth levels: row t needs only rows of its ancestors
    for (int d = 0; d <= s.maxdepth; ++d) {
        for (int i = tid; i < N * N; i += kPrepThreads) {
            const int t = i / N, c = i % N;
            if (s.depth[t] != d) continue;
            const uint64_t an = s.anc[t];
            if (c != t && !((an >> c) & 1ull)) continue;
            float x = c == t ? 1.f : 0.f;
            for (uint64_t r = an; r; r &= r - 1) {
                const int j = __ffsll((long long)r) - 1;
                x = fmaf(-s.A[t * kLd + j], s.T[j * kLd + c], x);
            }
            s.T[t * kLd + c] = x;
        }
        __syncthreads();
    }

    // 5. P = Attn T (support on path(t)); write the workspace record
    float* wT = reinterpret_cast<float*>(rec + wl.T);
    float* wP = reinterpret_cast<float*>(rec + wl.P);
    for (int i = tid; i < N * N; i += kPrepThreads) {
        const int t = i / N, c = i % N;
        const uint64_t path = s.anc[t] | (1ull << t);
        float x = 0.f;
        if ((path >> c) & 1ull) {
            for (uint64_t r = path; r; r &= r - 1) {
                const int j = __ffsll((long long)r) - 1;
                x = fmaf(s.At[t * kLd + j], s.T[j * kLd + c], x);
            }
        }
        wP[i] = x;
        wT[i] = s.T[t * kLd + c];
    }
    if (tid < N) {
        reinterpret_cast<float*>(rec + wl.eg)[tid] = expf(s.g[tid]);
        reinterpret_cast<float*>(rec + wl.bt)[tid] = s.beta[tid];
        reinterpret_cast<uint64_t*>(rec + wl.anc)[tid] = s.anc[tid] | (1ull << tid);
        a.f.g[(size_t)bh * N + tid] = s.g[tid];
        if (h == 0) a.f.parent[(size_t)b * N + tid] = s.par[tid];
    }
}

// ---------------------------------------------------------------------------
// contraction + epilogue (SIMT)
// ---------------------------------------------------------------------------
constexpr int kVT = 32;          // state rows per CTA
constexpr int kKC = 32;          // d_k chunk staged in smem
constexpr int kCThreads = 256;
constexpr int kRowGroups = kCThreads / 32;
constexpr int kMaxRowsPerThread = 2 * kMaxNodes / kRowGroups;   // 16

struct ContractSmem {
    float S[kVT * (kMaxDim + 1)];            // state tile, padded rows
    float qk[kKC * (2 * kMaxNodes + 1)];     // [c][r] (row stride 2N+1): r < N -> q_r, else k_{r-N}
    float YQ[kMaxNodes * (kVT + 1)];
    float R[kMaxNodes * (kVT + 1)];
    float cd[kMaxPath * kVT];                // fused commit: e^{g_a-g_j} delta_j[row]
    float coef[kMaxPath];
    int nodes[kMaxPath];
    float ega;
    int L;
};

template <typename T>
__global__ void __launch_bounds__(kCThreads) tree_contract_kernel(VerifyArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ContractSmem& s = *reinterpret_cast<ContractSmem*>(smem_raw);
    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int N = a.N, dk = a.dk, dv = a.dv, tid = threadIdx.x;
    const int v0 = blockIdx.y * kVT;
    const int rows = min(kVT, dv - v0);
    const WsLayout wl = ws_layout(N);
    const char* rec = a.ws + (size_t)bh * wl.record;
    const uint64_t* anc = reinterpret_cast<const uint64_t*>(rec + wl.anc);
    const int ldS = dk + 1;

    if (anc[0] == ~0ull) return;    // prologue rejected this tree (error already recorded)

    // 1. pending commit (fused path)
    const bool fused = a.commit.path != nullptr;
    if (fused) {
        if (tid < 32) {
            const int L = commit_path_setup(a.commit, b, h, a.H, s.nodes, s.coef, &s.ega);
            if (tid == 0) {
                s.L = L;
                if (L < 0) set_error(a.err, GDN_ERR_PATH);
            }
        }
        __syncthreads();
        if (s.L < 0) return;
        const float* dl = a.commit.delta + (size_t)bh * a.commit.N * dv;
        for (int i = tid; i < s.L * kVT; i += kCThreads) {
            const int j = i / kVT, r = i % kVT;
            s.cd[i] = r < rows ? s.coef[j] * dl[(size_t)s.nodes[j] * dv + v0 + r] : 0.f;
        }
        __syncthreads();
    }

    // 2. state tile -> smem (committed and written back once when fused)
    const int quads = dk / 4;
    const size_t sbase = ((size_t)bh * dv + v0) * dk;
    const T* ckey = fused ? static_cast<const T*>(a.commit.key) + (size_t)bh * a.commit.N * dk : nullptr;
    for (int i = tid; i < rows * quads; i += kCThreads) {
        const int r = i / quads, c = (i % quads) * 4;
        const size_t off = sbase + (size_t)r * dk + c;
        float4 x = *reinterpret_cast<const float4*>(a.S + off);
        if (fused) {
            x = commit_quad<T>(x, s.ega, s.L, s.nodes, s.cd + r, kVT, ckey, dk, c);
            *reinterpret_cast<float4*>(a.S + off) = x;
        }
        float* d = s.S + r * ldS + c;
        d[0] = x.x;
        d[1] = x.y;
        d[2] = x.z;
        d[3] = x.w;
    }

    // 3. Y = [Q; K] S_tile^T : thread (row group rg, lane = tile row v)
    const int rg = tid >> 5, lane = tid & 31;
    const int nr = 2 * N;
    const int ldq = nr + 1;
    float acc[kMaxRowsPerThread];
#pragma unroll
    for (int i = 0; i < kMaxRowsPerThread; ++i) acc[i] = 0.f;
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    for (int c0 = 0; c0 < dk; c0 += kKC) {
        __syncthreads();
        for (int i = tid; i < nr * kKC; i += kCThreads) {
            const int r = i / kKC, c = i % kKC;
            const int t = r < N ? r : r - N;
            const size_t row = ((size_t)b * N + t) * a.H + h;
            const float x = c0 + c < dk ? ld_elem<T>(r < N ? q : k, row * dk + c0 + c) : 0.f;
            s.qk[c * ldq + r] = x;
        }
        __syncthreads();
        if (lane < rows) {
            const int cn = min(kKC, dk - c0);
            for (int c = 0; c < cn; ++c) {
                const float sv = s.S[lane * ldS + c0 + c];
                const float* col = s.qk + c * ldq;
#pragma unroll
                for (int i = 0; i < kMaxRowsPerThread; ++i) {
                    const int r = rg + kRowGroups * i;
                    if (r < nr) acc[i] = fmaf(col[r], sv, acc[i]);
                }
            }
        }
    }
    __syncthreads();

    // 4. Y_Q -> smem; R = beta (v - e^g Y_K) -> smem
    const float* eg = reinterpret_cast<const float*>(rec + wl.eg);
    const float* bt = reinterpret_cast<const float*>(rec + wl.bt);
    const T* vv = static_cast<const T*>(a.v);
    if (lane < rows) {
#pragma unroll
        for (int i = 0; i < kMaxRowsPerThread; ++i) {
            const int r = rg + kRowGroups * i;
            if (r < N) {
                s.YQ[r * (kVT + 1) + lane] = acc[i];
            } else if (r < nr) {
                const int t = r - N;
                const float vt = ld_elem<T>(vv, (((size_t)b * N + t) * a.H + h) * dv + v0 + lane);
                s.R[t * (kVT + 1) + lane] = bt[t] * (vt - eg[t] * acc[i]);
            }
        }
    }
    __syncthreads();

    // 5. Delta_t = sum_{j in path(t)} T[t,j] R_j ; O_t = e^{g_t} YQ_t + sum_j P[t,j] R_j
    const float* wT = reinterpret_cast<const float*>(rec + wl.T);
    const float* wP = reinterpret_cast<const float*>(rec + wl.P);
    for (int t = rg; t < N; t += kRowGroups) {
        if (lane >= rows) continue;
        float d = 0.f, o = 0.f;
        for (uint64_t m = anc[t]; m; m &= m - 1) {
            const int j = __ffsll((long long)m) - 1;
            const float rj = s.R[j * (kVT + 1) + lane];
            d = fmaf(wT[t * N + j], rj, d);
            o = fmaf(wP[t * N + j], rj, o);
        }
        o = fmaf(eg[t], s.YQ[t * (kVT + 1) + lane], o);
        a.out[(((size_t)b * N + t) * a.H + h) * dv + v0 + lane] = o;
        a.f.delta[((size_t)bh * N + t) * dv + v0 + lane] = d;
    }
}

}  // namespace

cudaError_t launch_tree_mask(const int32_t* parent, int B, int N, uint64_t* mask, int32_t* depth,
                             int* err, cudaStream_t s) {
    tree_mask_kernel<<<B, kMaxNodes, 0, s>>>(parent, N, mask, depth, err);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_tree_t(const VerifyArgs& a, cudaStream_t s) {
    const int prep_smem = (int)sizeof(PrepSmem);
    const int con_smem = (int)sizeof(ContractSmem);
    static bool attr_set[64];   // per device: opt in to > 48 KiB dynamic smem once
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(tree_prep_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, prep_smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(tree_contract_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, con_smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    tree_prep_kernel<T><<<a.B * a.H, kPrepThreads, prep_smem, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 grid(a.B * a.H, (a.dv + kVT - 1) / kVT);
    tree_contract_kernel<T><<<grid, kCThreads, con_smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_tree_verify(const VerifyArgs& a, int dtype, cudaStream_t s) {
    return dtype == GDN_DTYPE_F32 ? launch_tree_t<float>(a, s) : launch_tree_t<__nv_bfloat16>(a, s);
}

}  // namespace gdn
