// gdn_tree.cu -- tree-masked factorized verification: mask, prologue, SIMT contraction.
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
// Kernels here:
//   tree_mask_kernel      ancestor bitmask + depth (gdn_tree_mask).
//   tree_prep_kernel      one CTA per (b, h): stages Q and K with cp.async,
//                         ancestor masks, gates, masked Gram entries (8 lanes
//                         per (node, ancestor) pair), each node's row of T by
//                         back-substitution along its own path, P = Attn T;
//                         writes dense fp32 T and P to the workspace and the
//                         factor record's g, parent and keys.
//   tree_contract_kernel  SIMT contraction for any d_k/d_v/dtype: one CTA per
//                         (b, h, 32 state rows); streams the state tile
//                         (committing a pending path first when fused), forms
//                         Y = [Q; K] S_tile^T, then R, Delta and O.
//                         (gdn_tree_tc.cu holds the tensor-core versions of
//                         both kernels, used for bf16 inputs with d_k = 256.)
#include "gdn_internal.cuh"
#include "gdn_prep_common.cuh"

namespace gdn {
namespace {

template <typename T>
struct Chunk;   // 16-byte chunk of q/k elements
template <>
struct Chunk<__nv_bfloat16> {
    __device__ static float dot(uint4 a, uint4 b) {
        const uint32_t x[4] = {a.x, a.y, a.z, a.w}, y[4] = {b.x, b.y, b.z, b.w};
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            s = fmaf(__uint_as_float(x[i] << 16), __uint_as_float(y[i] << 16), s);
            s = fmaf(__uint_as_float(x[i] & 0xffff0000u), __uint_as_float(y[i] & 0xffff0000u), s);
        }
        return s;
    }
};
template <>
struct Chunk<float> {
    __device__ static float dot(uint4 a, uint4 b) {
        float s = __uint_as_float(a.x) * __uint_as_float(b.x);
        s = fmaf(__uint_as_float(a.y), __uint_as_float(b.y), s);
        s = fmaf(__uint_as_float(a.z), __uint_as_float(b.z), s);
        return fmaf(__uint_as_float(a.w), __uint_as_float(b.w), s);
    }
};

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

struct PrepLayout {
    int qs, ks, A, At, T, pairs, plist, par, anc, la, g, beta, depth, off, misc, total, ld;
    __host__ __device__ PrepLayout(int N, int dk, int esz) {
        int o = 0;
        auto take = [&](int bytes) { int r = o; o += (bytes + 15) / 16 * 16; return r; };
        ld = N + 1;
        qs = take(N * dk * esz);
        ks = take(N * dk * esz);
        A = take(N * ld * 4);
        At = take(N * ld * 4);
        T = take(N * ld * 4);
        pairs = take(N * (N + 1) / 2 * 2);
        plist = take(N * 64);
        par = take(N * 4);
        anc = take(N * 8);
        la = take(N * 4);
        g = take(N * 4);
        beta = take(N * 4);
        depth = take(N * 4);
        off = take((N + 1) * 4);
        misc = take(16);
        total = o;
    }
};

template <typename T>
__global__ void __launch_bounds__(kPrepThreads) tree_prep_kernel(VerifyArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int N = a.N, dk = a.dk, tid = threadIdx.x;
    const PrepLayout Ly(N, dk, (int)sizeof(T));
    T* Qs = reinterpret_cast<T*>(smem + Ly.qs);
    T* Ks = reinterpret_cast<T*>(smem + Ly.ks);
    float* sA = reinterpret_cast<float*>(smem + Ly.A);
    float* sAt = reinterpret_cast<float*>(smem + Ly.At);
    float* sT = reinterpret_cast<float*>(smem + Ly.T);
    uint16_t* pairs = reinterpret_cast<uint16_t*>(smem + Ly.pairs);
    uint8_t* plist = reinterpret_cast<uint8_t*>(smem + Ly.plist);
    int* par = reinterpret_cast<int*>(smem + Ly.par);
    uint64_t* anc = reinterpret_cast<uint64_t*>(smem + Ly.anc);
    float* la = reinterpret_cast<float*>(smem + Ly.la);
    float* sg = reinterpret_cast<float*>(smem + Ly.g);
    float* sbeta = reinterpret_cast<float*>(smem + Ly.beta);
    int* sdepth = reinterpret_cast<int*>(smem + Ly.depth);
    int* off = reinterpret_cast<int*>(smem + Ly.off);
    const int ld = Ly.ld;

    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const WsLayout wl = ws_layout(N);
    char* rec = a.ws + (size_t)bh * wl.record;

    // This layer's inputs may come from the previous kernel on the stream.
    griddep_wait();
    griddep_launch();

    // 1. stage Q, K rows (cp.async) and the per-node scalars
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const int rowb = dk * (int)sizeof(T);
    for (int t = 0; t < N; ++t) {
        const size_t rt = (((size_t)b * N + t) * a.H + h) * dk;
        cp_async_block(Qs + (size_t)t * dk, q + rt, rowb, tid, kPrepThreads);
        cp_async_block(Ks + (size_t)t * dk, k + rt, rowb, tid, kPrepThreads);
    }
    bool bad = false;
    if (tid < N) {
        const int p = a.parent[(size_t)b * N + tid];
        bad = p < -1 || p >= tid;
        par[tid] = p;
        const size_t gi = ((size_t)b * N + tid) * a.H + h;
        la[tid] = logf(a.alpha[gi]);
        sbeta[tid] = a.beta[gi];
    }
    cp_async_wait_all();
    if (__syncthreads_or(bad)) {
        if (tid == 0) {
            set_error(a.err, GDN_ERR_TREE);
            *reinterpret_cast<uint64_t*>(rec + wl.anc) = ~0ull;   // record marked invalid
        }
        return;
    }

    // 2. masks, depths, gates; 3. (t, j on path(t)) pairs
    prep::node_meta(tid, N, par, la, anc, sdepth, sg, plist);
    __syncthreads();
    prep::pair_list(tid, N, sdepth, anc, off, pairs);

    // 4. masked Gram entries: 8 lanes per pair, 16-byte chunks interleaved across the group
    const int warp = tid >> 5, lane = tid & 31;
    const int npairs = off[N];
    const int grp = lane >> 3, gl = lane & 7;
    const int nchunk = rowb / 16;
    for (int base = warp * 4; base < npairs; base += (kPrepThreads / 32) * 4) {
        const int p = base + grp;
        const bool valid = p < npairs;
        const int pr = valid ? pairs[p] : 0;
        const int t = pr >> 8, j = pr & 255;
        float pkk = 0.f, pqk = 0.f;
        if (valid) {
            const uint4* kt = reinterpret_cast<const uint4*>(Ks + (size_t)t * dk);
            const uint4* qt = reinterpret_cast<const uint4*>(Qs + (size_t)t * dk);
            const uint4* kj = reinterpret_cast<const uint4*>(Ks + (size_t)j * dk);
            for (int c = gl; c < nchunk; c += 8) {
                const uint4 x = kj[c];
                pkk += Chunk<T>::dot(kt[c], x);
                pqk += Chunk<T>::dot(qt[c], x);
            }
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) {
            pkk += __shfl_xor_sync(0xffffffffu, pkk, o);
            pqk += __shfl_xor_sync(0xffffffffu, pqk, o);
        }
        if (valid && gl == 0) prep::gram_entry(t, j, pkk, pqk, ld, sg, sbeta, sA, sAt, !a.linear);
    }
    __syncthreads();

    // 5-6. rows of T, then P over A; workspace and factor records
    prep::solve_rows(tid, N, ld, sdepth, plist, sA, sAt, sT);
    prep::write_dense(tid, kPrepThreads, N, ld, anc, sA, sT, reinterpret_cast<float*>(rec + wl.T),
                      reinterpret_cast<float*>(rec + wl.P));
    prep::write_meta(tid, N, b, h, bh, rec, wl, sg, sbeta, anc, par, a.f);
    uint4* key_out = reinterpret_cast<uint4*>(static_cast<T*>(a.f.key) + (size_t)bh * N * dk);
    const uint4* ksrc = reinterpret_cast<const uint4*>(Ks);
    for (int i = tid; i < N * nchunk; i += kPrepThreads) key_out[i] = ksrc[i];
}

// ---------------------------------------------------------------------------
// contraction + epilogue (SIMT)
// ---------------------------------------------------------------------------
constexpr int kVT = 32;          // state rows per CTA
constexpr int kCThreads = 256;
constexpr int kRowGroups = kCThreads / 32;
constexpr int kMaxRowsPerThread = 2 * kMaxNodes / kRowGroups;   // 16

struct ContractLayout {
    int S, qk, YQ, R, T, P, eg, bt, anc, cd, key, coef, nodes, misc, total;
    __host__ __device__ ContractLayout(int N, int dk, int Lcap, int esz) {
        int o = 0;
        auto take = [&](int bytes) { int r = o; o += (bytes + 15) / 16 * 16; return r; };
        S = take(kVT * (dk + 4) * 4);    // rows padded by 16 bytes: float4 reads spread over banks
        qk = take(2 * N * dk * esz);     // [Q rows; K rows] in the input element type
        YQ = take(N * (kVT + 1) * 4);
        R = take(N * (kVT + 1) * 4);
        T = take(N * N * 4);
        P = take(N * N * 4);
        eg = take(N * 4);
        bt = take(N * 4);
        anc = take(N * 8);
        cd = take(Lcap * kVT * 4);
        key = take(Lcap * dk * esz);
        coef = take(kMaxPath * 4);
        nodes = take(kMaxPath * 4);
        misc = take(16);
        total = o;
    }
};

template <typename T>
__global__ void __launch_bounds__(kCThreads) tree_contract_kernel(VerifyArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int N = a.N, dk = a.dk, dv = a.dv, tid = threadIdx.x;
    const bool fused = a.commit.path != nullptr;
    const ContractLayout Ly(N, dk, fused ? a.commit.Lmax : 0, (int)sizeof(T));
    float* sS = reinterpret_cast<float*>(smem + Ly.S);
    float* sYQ = reinterpret_cast<float*>(smem + Ly.YQ);
    float* sR = reinterpret_cast<float*>(smem + Ly.R);
    float* sT = reinterpret_cast<float*>(smem + Ly.T);
    float* sP = reinterpret_cast<float*>(smem + Ly.P);
    float* seg = reinterpret_cast<float*>(smem + Ly.eg);
    float* sbt = reinterpret_cast<float*>(smem + Ly.bt);
    uint64_t* sanc = reinterpret_cast<uint64_t*>(smem + Ly.anc);
    float* scd = reinterpret_cast<float*>(smem + Ly.cd);
    T* skey = reinterpret_cast<T*>(smem + Ly.key);
    float* scoef = reinterpret_cast<float*>(smem + Ly.coef);
    int* snodes = reinterpret_cast<int*>(smem + Ly.nodes);
    float* sega = reinterpret_cast<float*>(smem + Ly.misc);
    int* sL = reinterpret_cast<int*>(smem + Ly.misc + 4);

    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int v0 = blockIdx.y * kVT;
    const int rows = min(kVT, dv - v0);
    const int ldS = dk + 4;
    const WsLayout wl = ws_layout(N);
    const char* rec = a.ws + (size_t)bh * wl.record;

    // 1. state tile -> smem and the pending commit (reads only: overlaps the prologue kernel)
    const int quads = dk / 4;
    const size_t sbase = ((size_t)bh * dv + v0) * dk;
    for (int i = tid; i < rows * quads; i += kCThreads) {
        const int r = i / quads, c = (i % quads) * 4;
        cp_async16(sS + r * ldS + c, a.S + sbase + (size_t)r * dk + c);
    }
    if (fused) {
        if (tid < 32) {
            const int L = commit_path_setup(a.commit, b, h, a.H, snodes, scoef, sega);
            if (tid == 0) {
                *sL = L;
                if (L < 0) set_error(a.err, GDN_ERR_PATH);
            }
        }
        __syncthreads();
        const int L = *sL;
        if (L < 0) return;
        const float* dl = a.commit.delta + (size_t)bh * a.commit.N * dv;
        const T* key_bh = static_cast<const T*>(a.commit.key) + (size_t)bh * a.commit.N * dk;
        for (int i = 0; i < L; ++i)
            cp_async_block(skey + (size_t)i * dk, key_bh + (size_t)snodes[i] * dk, dk * (int)sizeof(T),
                           tid, kCThreads);
        for (int i = tid; i < L * kVT; i += kCThreads) {
            const int j = i / kVT, r = i % kVT;
            scd[i] = r < rows ? scoef[j] * dl[(size_t)snodes[j] * dv + v0 + r] : 0.f;
        }
        cp_async_wait_all();
        __syncthreads();
        const float ega = *sega;
        for (int i = tid; i < rows * quads; i += kCThreads) {
            const int r = i / quads, c = (i % quads) * 4;
            float4* d = reinterpret_cast<float4*>(sS + r * ldS + c);
            *d = commit_quad<T>(*d, ega, L, scd + r, kVT, skey, dk, c);
        }
    }

    // 2. wait for the prologue kernel; stage its tables; write the committed tile
    griddep_wait();
    griddep_launch();
    if (*reinterpret_cast<const uint64_t*>(rec + wl.anc) == ~0ull) return;   // tree rejected
    cp_async_block(sT, rec + wl.T, (int)ws_table_bytes(N), tid, kCThreads);
    cp_async_block(sP, rec + wl.P, (int)ws_table_bytes(N), tid, kCThreads);
    for (int t = tid; t < N; t += kCThreads) {
        seg[t] = reinterpret_cast<const float*>(rec + wl.eg)[t];
        sbt[t] = reinterpret_cast<const float*>(rec + wl.bt)[t];
        sanc[t] = reinterpret_cast<const uint64_t*>(rec + wl.anc)[t];
    }
    __syncthreads();
    if (fused) {
        for (int i = tid; i < rows * quads; i += kCThreads) {
            const int r = i / quads, c = (i % quads) * 4;
            *reinterpret_cast<float4*>(a.S + sbase + (size_t)r * dk + c) =
                *reinterpret_cast<const float4*>(sS + r * ldS + c);
        }
    }

    // 3. Y = [Q; K] S_tile^T : thread (row group rg, lane = tile row v); [Q; K] rows
    //    staged once with cp.async, consumed 8 columns at a time
    const int rg = tid >> 5, lane = tid & 31;
    const int nr = 2 * N;
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    T* sQK = reinterpret_cast<T*>(smem + Ly.qk);
    const int rowb = dk * (int)sizeof(T);
    for (int r = 0; r < nr; ++r) {
        const int t = r < N ? r : r - N;
        const size_t row = ((size_t)b * N + t) * a.H + h;
        cp_async_block(sQK + (size_t)r * dk, (r < N ? q : k) + row * dk, rowb, tid, kCThreads);
    }
    cp_async_wait_all();
    __syncthreads();
    float acc[kMaxRowsPerThread];
#pragma unroll
    for (int i = 0; i < kMaxRowsPerThread; ++i) acc[i] = 0.f;
    if (lane < rows) {
        const float* srow = sS + lane * ldS;
        for (int c = 0; c < dk; c += 8) {
            const float4 s0 = *reinterpret_cast<const float4*>(srow + c);
            const float4 s1 = *reinterpret_cast<const float4*>(srow + c + 4);
#pragma unroll
            for (int i = 0; i < kMaxRowsPerThread; ++i) {
                const int r = rg + kRowGroups * i;
                if (r < nr) {
                    float x[8];
                    ld8<T>(sQK + (size_t)r * dk + c, x);
                    float a0 = acc[i];
                    a0 = fmaf(x[0], s0.x, a0);
                    a0 = fmaf(x[1], s0.y, a0);
                    a0 = fmaf(x[2], s0.z, a0);
                    a0 = fmaf(x[3], s0.w, a0);
                    a0 = fmaf(x[4], s1.x, a0);
                    a0 = fmaf(x[5], s1.y, a0);
                    a0 = fmaf(x[6], s1.z, a0);
                    acc[i] = fmaf(x[7], s1.w, a0);
                }
            }
        }
    }
    __syncthreads();

    // 4. Y_Q -> smem; R = beta (v - e^g Y_K) -> smem
    const T* vv = static_cast<const T*>(a.v);
    if (lane < rows) {
#pragma unroll
        for (int i = 0; i < kMaxRowsPerThread; ++i) {
            const int r = rg + kRowGroups * i;
            if (r < N) {
                sYQ[r * (kVT + 1) + lane] = acc[i];
            } else if (r < nr) {
                const int t = r - N;
                const float vt = ld_elem<T>(vv, (((size_t)b * N + t) * a.H + h) * dv + v0 + lane);
                sR[t * (kVT + 1) + lane] = sbt[t] * (a.linear ? vt : vt - seg[t] * acc[i]);
            }
        }
    }
    __syncthreads();

    // 5. Delta_t = sum_{j in path(t)} T[t,j] R_j ; O_t = e^{g_t} YQ_t + sum_j P[t,j] R_j
    for (int t = rg; t < N; t += kRowGroups) {
        if (lane >= rows) continue;
        float d = 0.f, o = 0.f;
        for (uint64_t m = sanc[t]; m; m &= m - 1) {
            const int j = __ffsll((long long)m) - 1;
            const float rj = sR[j * (kVT + 1) + lane];
            d = fmaf(sT[t * N + j], rj, d);
            o = fmaf(sP[t * N + j], rj, o);
        }
        o = fmaf(seg[t], sYQ[t * (kVT + 1) + lane], o);
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
cudaError_t launch_tree_prep(const VerifyArgs& a, cudaStream_t s) {
    static bool attr[64];
    const PrepLayout Ly(a.N, a.dk, (int)sizeof(T));
    cudaError_t e = ensure_smem(tree_prep_kernel<T>, Ly.total, attr);
    if (e != cudaSuccess) return e;
    return launch_kernel(tree_prep_kernel<T>, dim3(a.B * a.H), dim3(kPrepThreads), Ly.total, s,
                         a.overlap, a);
}

template <typename T>
cudaError_t launch_tree_contract_simt(const VerifyArgs& a, cudaStream_t s) {
    static bool attr[64];
    const ContractLayout Ly(a.N, a.dk, a.commit.path ? a.commit.Lmax : 0, (int)sizeof(T));
    cudaError_t e = ensure_smem(tree_contract_kernel<T>, Ly.total, attr);
    if (e != cudaSuccess) return e;
    dim3 grid(a.B * a.H, (a.dv + kVT - 1) / kVT);
    // always a programmatic dependent of the prologue kernel launched just before it
    return launch_kernel(tree_contract_kernel<T>, grid, dim3(kCThreads), Ly.total, s, true, a);
}

// The SIMT contraction alone for fp32 q/k/v, after a prologue of the caller's
// that has written the workspace records (it reads them, and q/k/v, only after
// its programmatic wait).
cudaError_t launch_tree_contract_simt_f32(const VerifyArgs& a, cudaStream_t s) {
    return launch_tree_contract_simt<float>(a, s);
}

// Mirrors the dispatch of launch_tree_verify below: only the single-kernel
// tensor-core verifier leaves the workspace untouched.
bool tree_verify_uses_workspace(const VerifyArgs& a, int dtype) {
    const bool tc = dtype == GDN_DTYPE_F32 ? a.split[0] != nullptr && tc_contract_eligible(a) : tc_contract_eligible(a);
    return !tc || tc_uses_workspace(a);
}

cudaError_t launch_tree_verify(const VerifyArgs& args, int dtype, cudaStream_t s) {
    VerifyArgs a = args;
    cudaError_t e;
    if (dtype == GDN_DTYPE_F32) {
        if (a.split[0] != nullptr && tc_contract_eligible(a)) {   // fp32 q/k with bf16 hi/lo terms
            a.tc = true;
            return launch_tree_tc(a, s);
        }
        a.tc = false;
        e = launch_tree_prep<float>(a, s);
        if (e != cudaSuccess) return e;
        return launch_tree_contract_simt<float>(a, s);
    }
    a.tc = tc_contract_eligible(a);
    if (a.tc) return launch_tree_tc(a, s);
    e = launch_tree_prep<__nv_bfloat16>(a, s);
    if (e != cudaSuccess) return e;
    return launch_tree_contract_simt<__nv_bfloat16>(a, s);
}

}  // namespace gdn
