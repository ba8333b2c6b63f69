// gdn_gla.cu -- gated linear attention (one gate per key channel) over a draft
// tree, with its own factor record and commit.
//
// The review of SpecLA (pith.science 7ERME3HB), editorial analysis, names GLA
// beside DeltaNet and Mamba as recurrences whose per-token factor records the
// same verify / commit runtime carries.  With S stored d_v x d_k (row = value
// index) the recurrence along a node's root-to-node path is
//
//   S_t = S_parent(t) diag(alpha_t) + beta_t v_t k_t^T,   o_t = S_t q_t,
//
// alpha_t in (0, 1]^{d_k}.  With g_t = sum_{j on path(t)} log alpha_j (a d_k
// vector) it unrolls to S_t = S0 diag(e^{g_t}) + sum_{j on path(t)} delta_j
// (k_j (.) e^{g_t - g_j})^T, delta_j = beta_j v_j, so
//
//   o_t = S0 qhat_t + sum_{j on path(t)} Attn[t, j] delta_j,
//   qhat_t = e^{g_t} (.) q_t,   Attn[t, j] = sum_c q_t[c] k_j[c] e^{g_t[c] - g_j[c]}.
//
// Nothing here needs a solve (no erasure: T = I), so verification is the
// scalar-gate verifier's contraction with the per-channel gates moved into its
// inputs: a prologue kernel (one CTA per (sequence, head)) builds g, qhat and
// the masked Attn table -- each entry from the gate difference g_t - g_j <= 0
// of an ancestor pair, never from e^{-g_j} alone, which overflows on deep
// paths -- and writes the workspace records that the contraction kernels read
// (e^g := 1, beta, the masks, [T; P] = [I; Attn]); then the tensor-core
// contraction (d_k = 256, d_v a multiple of 128: qhat as bf16 hi + lo terms)
// or the SIMT one (other shapes: fp32 qhat) forms Y = S0 qhat^T, R = beta v and
// [Delta | P R] in linear mode.  The commit is its own streaming kernel:
//
//   S_a = S0 diag(e^{g_a}) + sum_{j on path(a)} delta_j (k_j (.) e^{g_a - g_j})^T.
#include "gdn_internal.cuh"
#include "gdn_prep_common.cuh"

namespace gdn {
namespace {

// The decays e^{g} and e^{g_t - g_j} (g <= 0) as 2^(x log2 e) through exp2f:
// measured cheaper than expf in the prologue's inner loop, and within a few ulp.
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kGThreads = 1024;
constexpr int kGcThreads = 256;
constexpr int kGcRows = 16;      // state rows per commit CTA

// GLA factor record: delta fp32 [B][H][N][dv] | key dtype [B][H][N][dk] |
// g fp32 [B][H][N][dk] | parent int32 [B][N], each section 256-byte aligned.
struct GlaFactorLayout {
    size_t delta, key, g, parent, total;
    GlaFactorLayout(int B, int N, int H, int dk, int dv, int dtype) {
        const size_t BHN = (size_t)B * H * N;
        delta = 0;
        key = align_up(delta + BHN * dv * 4, kSectionAlign);
        g = align_up(key + BHN * dk * elem_bytes(dtype), kSectionAlign);
        parent = align_up(g + BHN * dk * 4, kSectionAlign);
        total = align_up(parent + (size_t)B * N * 4, kSectionAlign);
    }
};

// Workspace: the verifier's per-(sequence, head) records, then qhat (bf16 hi
// and lo terms, or fp32: 4 bytes per element either way) [B][N][H][dk], then
// fp32 v [B][N][H][dv] (used when v arrives as bf16).
struct GlaWsLayout {
    size_t recs, qhat, v32, total;
    GlaWsLayout(int B, int N, int H, int dk, int dv) {
        recs = 0;
        qhat = align_up((size_t)B * H * ws_layout(N).record, kSectionAlign);
        v32 = align_up(qhat + (size_t)B * N * H * dk * 4, kSectionAlign);
        total = align_up(v32 + (size_t)B * N * H * dv * 4, kSectionAlign);
    }
};

struct GlaArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;        // [B][N][H][dk]
    const float* beta;         // [B][N][H]
    const int32_t* parent;     // [B][N]
    void* key;                 // record: key copy
    float* g;                  // record: per-channel log gates
    int32_t* par_out;          // record: parents
    char* recs;                // workspace records
    void* qhat;
    float* v32;                // nullptr: v is already fp32
    int B, N, H, dk, dv;
    int* err;
};

// Dynamic shared memory of the prologue: g [N][dk], Attn and T [N][N + 1], then
// (bf16 inputs) the tree's q and k rows [N][dk] each.
inline size_t gla_prep_smem(int N, int dk, int esz) {
    return ((size_t)N * dk + 2 * (size_t)N * (N + 1)) * 4 + (esz == 2 ? 2 * (size_t)N * dk * 2 : 0);
}

template <typename T, bool kTc>
__global__ void __launch_bounds__(kGThreads) gla_prep_kernel(GlaArgs a) {
    extern __shared__ __align__(16) float gsm[];
    __shared__ int par[kMaxNodes], depth[kMaxNodes], off[kMaxNodes + 1];
    __shared__ uint64_t anc[kMaxNodes];
    __shared__ uint8_t plist[kMaxNodes * 64];
    __shared__ float la0[kMaxNodes], g0[kMaxNodes];   // node_meta's scalar-gate slots (zero gates)
    __shared__ uint16_t pairs[kMaxNodes * kMaxNodes];
    __shared__ int s_bad, s_maxd;
    const int N = a.N, H = a.H, dk = a.dk, dv = a.dv, ld = N + 1;
    const int bh = blockIdx.x, b = bh / H, h = bh % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float* sg = gsm;                       // g, per node and key channel
    float* sP = sg + (size_t)N * dk;       // Attn on the inclusive mask
    float* sT = sP + (size_t)N * ld;       // identity on the inclusive mask
    const WsLayout wl = ws_layout(N);
    char* rec = a.recs + (size_t)bh * wl.record;
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    griddep_wait();
    griddep_launch();     // the contraction only streams the state before its own wait

    if (tid == 0) {
        s_bad = 0;
        s_maxd = 0;
    }
    __syncthreads();
    if (tid < N) {
        const int p = a.parent[(size_t)b * N + tid];
        par[tid] = p;
        la0[tid] = 0.f;
        if (p < -1 || p >= tid) s_bad = 1;
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            set_error(a.err, GDN_ERR_TREE);
            *reinterpret_cast<uint64_t*>(rec + wl.anc) = ~0ull;   // the contraction skips this record
        }
        return;
    }
    prep::node_meta(tid, N, par, la0, anc, depth, g0, plist);
    if (tid < N) atomicMax(&s_maxd, depth[tid]);
    __syncthreads();

    // The tree's q and k rows into shared memory (bf16 inputs) by async copies, and
    // log alpha for every (node, channel) in one pass with all loads independent.
    constexpr bool kStage = sizeof(T) == 2;
    T* sq = reinterpret_cast<T*>(sT + (size_t)N * ld);
    T* sk = sq + (size_t)N * dk;
    if (kStage) {
        const int chunks = dk * (int)sizeof(T) / 16;          // 16-byte chunks per row
        for (int i = tid; i < 2 * N * chunks; i += kGThreads) {
            const int r = i / chunks, cc = i - r * chunks;
            const int t = r < N ? r : r - N;
            const T* src = (r < N ? q : k) + (((size_t)b * N + t) * H + h) * dk;
            cp_async16((r < N ? sq + t * dk : sk + t * dk) + cc * (16 / (int)sizeof(T)), src + cc * (16 / (int)sizeof(T)));
        }
    }
    const int dk4 = dk / 4;                                  // d_k is a multiple of 16
    for (int i = tid; i < N * dk4; i += kGThreads) {         // four channels per load, all in flight
        const int t = i / dk4, c = 4 * (i - t * dk4);
        const float4 al = *reinterpret_cast<const float4*>(a.alpha + (((size_t)b * N + t) * H + h) * dk + c);
        *reinterpret_cast<float4*>(sg + t * dk + c) = make_float4(logf(al.x), logf(al.y), logf(al.z), logf(al.w));
    }
    cp_async_wait_all();
    __syncthreads();

    // g_t[c] = g_parent(t)[c] + log alpha_t[c], one tree level at a time (a node's parent
    // is one level up, so it is final when the node's level is reached)
    float4* sg4 = reinterpret_cast<float4*>(sg);
    constexpr int kItems = kMaxNodes * (kMaxDim / 4) / kGThreads;   // (node, channel quad) items per thread
    int it_i[kItems], it_p[kItems], it_d[kItems];                  // item, its parent's item, its depth
#pragma unroll
    for (int e = 0; e < kItems; ++e) {
        const int i = tid + e * kGThreads, t = i / dk4;
        const bool in = i < N * dk4;
        it_i[e] = i;
        it_d[e] = in ? depth[t] : -1;
        it_p[e] = in && par[t] >= 0 ? par[t] * dk4 + (i - t * dk4) : 0;
    }
#pragma unroll 1
    for (int lvl = 1; lvl <= s_maxd; ++lvl) {
#pragma unroll
        for (int e = 0; e < kItems; ++e) {
            if (it_d[e] == lvl) {
                float4 x = sg4[it_i[e]];
                const float4 pg = sg4[it_p[e]];
                x.x += pg.x;
                x.y += pg.y;
                x.z += pg.z;
                x.w += pg.w;
                sg4[it_i[e]] = x;
            }
        }
        __syncthreads();
    }
    // the record's g and key copy and qhat_t[c] = q_t[c] e^{g_t[c]}, every (node, channel)
    __nv_bfloat16* qh = static_cast<__nv_bfloat16*>(a.qhat);
    __nv_bfloat16* ql = qh + (size_t)a.B * N * H * dk;
    for (int i = tid; i < N * dk4; i += kGThreads) {         // four channels per thread and store
        const int t = i / dk4, c = 4 * (i - t * dk4);
        const size_t src = (((size_t)b * N + t) * H + h) * dk + c;
        const size_t dst = ((size_t)bh * N + t) * dk + c;
        const float4 gt = sg4[t * dk4 + c / 4];
        *reinterpret_cast<float4*>(a.g + dst) = gt;
        const T* kp = kStage ? sk + t * dk + c : k + src;
        const T* qp = kStage ? sq + t * dk + c : q + src;
        if constexpr (sizeof(T) == 2)
            *reinterpret_cast<uint2*>(static_cast<T*>(a.key) + dst) = *reinterpret_cast<const uint2*>(kp);
        else
            *reinterpret_cast<float4*>(static_cast<T*>(a.key) + dst) = *reinterpret_cast<const float4*>(kp);
        const float4 qv = ld4<T>(qp, 0);
        const float x[4] = {qv.x * exp2f(gt.x * kLog2e), qv.y * exp2f(gt.y * kLog2e), qv.z * exp2f(gt.z * kLog2e),
                            qv.w * exp2f(gt.w * kLog2e)};
        if (kTc) {   // hi = bf16(x), lo = bf16(x - hi), two channels per conversion
            const __nv_bfloat162 h01 = __floats2bfloat162_rn(x[0], x[1]), h23 = __floats2bfloat162_rn(x[2], x[3]);
            const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
            const __nv_bfloat162 l01 = __floats2bfloat162_rn(x[0] - f01.x, x[1] - f01.y);
            const __nv_bfloat162 l23 = __floats2bfloat162_rn(x[2] - f23.x, x[3] - f23.y);
            *reinterpret_cast<uint2*>(qh + src) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
            *reinterpret_cast<uint2*>(ql + src) =
                make_uint2(*reinterpret_cast<const uint32_t*>(&l01), *reinterpret_cast<const uint32_t*>(&l23));
        } else {
            *reinterpret_cast<float4*>(static_cast<float*>(a.qhat) + src) = make_float4(x[0], x[1], x[2], x[3]);
        }
    }
    if (a.v32 != nullptr)
        for (int i = tid; i < N * (dv / 4); i += kGThreads) {    // four values per thread
            const int t = i / (dv / 4), c = 4 * (i - t * (dv / 4));
            const size_t o = (((size_t)b * N + t) * H + h) * dv + c;
            *reinterpret_cast<float4*>(a.v32 + o) = ld4<T>(static_cast<const T*>(a.v), o);
        }
    if (h == 0 && tid < N) a.par_out[(size_t)b * N + tid] = par[tid];
    __syncthreads();

    // Attn[t, j] = sum_c q_t[c] k_j[c] e^{g_t[c] - g_j[c]} on the inclusive mask; T = I there
    prep::pair_list(tid, N, depth, anc, off, pairs);
    const int npairs = off[N];
    // Each warp takes a contiguous run of the (node-major) pair list, so that it keeps its
    // lanes' q_t and g_t channels in registers while t stays the same.
    const int per_warp = (npairs + kGThreads / 32 - 1) / (kGThreads / 32);
    const int pend = min(npairs, (warp + 1) * per_warp);
    int cur_t = -1;
    float qr[kMaxDim / 32], gr[kMaxDim / 32];             // channel lane + 32 i of q_t and g_t
#pragma unroll 1
    for (int pi = warp * per_warp; pi < pend; ++pi) {
        const int t = pairs[pi] >> 8, j = pairs[pi] & 255;
        if (t != cur_t) {
            cur_t = t;
            const T* qt = kStage ? sq + t * dk : q + (((size_t)b * N + t) * H + h) * dk;
            const float* gt = sg + t * dk;
#pragma unroll
            for (int i = 0; i < kMaxDim / 32; ++i) {
                const int c = lane + 32 * i;
                qr[i] = c < dk ? ld_elem<T>(qt, c) : 0.f;
                gr[i] = c < dk ? gt[c] : 0.f;
            }
        }
        const T* kj = kStage ? sk + j * dk : k + (((size_t)b * N + j) * H + h) * dk;
        const float* gj = sg + j * dk;
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxDim / 32; i += 2) {           // d_k <= 256: at most 8 channels per lane
            const int c0 = lane + 32 * i, c1 = c0 + 32;
            if (c0 < dk) s0 = fmaf(qr[i] * ld_elem<T>(kj, c0), exp2f((gr[i] - gj[c0]) * kLog2e), s0);
            if (c1 < dk) s1 = fmaf(qr[i + 1] * ld_elem<T>(kj, c1), exp2f((gr[i + 1] - gj[c1]) * kLog2e), s1);
        }
        const float s = warp_sum(s0 + s1);
        if (lane == 0) {
            sP[t * ld + j] = s;
            sT[t * ld + j] = j == t ? 1.f : 0.f;
        }
    }
    __syncthreads();
    // workspace record: the gates live in qhat and Attn, so e^g := 1
    if (tid < N) {
        reinterpret_cast<float*>(rec + wl.eg)[tid] = 1.f;
        reinterpret_cast<float*>(rec + wl.bt)[tid] = a.beta[((size_t)b * N + tid) * H + h];
        reinterpret_cast<uint64_t*>(rec + wl.anc)[tid] = anc[tid] | (1ull << tid);
    }
    if (kTc)
        prep::write_operand(tid, kGThreads, N, ld, anc, sP, sT, reinterpret_cast<unsigned char*>(rec + wl.op));
    else
        prep::write_dense(tid, kGThreads, N, ld, anc, sP, sT, reinterpret_cast<float*>(rec + wl.T),
                          reinterpret_cast<float*>(rec + wl.P));
}

// ---------------------------------------------------------------------------
// commit
// ---------------------------------------------------------------------------
struct GlaCommitArgs {
    const float* S0;
    float* S_new;
    const float* delta;
    const void* key;
    const float* g;
    const int32_t* parent;
    const int32_t* path;
    int Lmax, B, N, H, dk, dv;
    int* err;
};

// Dynamic shared memory of the commit: e^{g_a} [dk], w [Lmax][dk], delta [Lmax][16].
inline size_t gla_commit_smem(int Lmax, int dk) { return ((size_t)dk + (size_t)Lmax * dk + (size_t)Lmax * kGcRows) * 4; }

// One CTA per (sequence, head, 16 state rows):
//   S_new[v, c] = S0[v, c] e^{g_a[c]} + sum_i delta_i[v] w_i[c],  w_i[c] = k_i[c] e^{g_a[c] - g_i[c]}.
template <typename T>
__global__ void __launch_bounds__(kGcThreads) gla_commit_kernel(GlaCommitArgs a) {
    extern __shared__ __align__(16) float csm[];
    __shared__ int s_nodes[kMaxPath];
    __shared__ int s_L;
    const int bh = blockIdx.x, b = bh / a.H;
    const int v0 = blockIdx.y * kGcRows, rows = min(kGcRows, a.dv - v0);
    const int tid = threadIdx.x, dk = a.dk, N = a.N;
    griddep_wait();
    griddep_launch();
    if (tid < 32) {
        const int L = path_chain_setup(a.path + (size_t)b * a.Lmax, a.Lmax, a.parent + (size_t)b * N, N, s_nodes);
        if (tid == 0) {
            s_L = L;
            if (L < 0 && blockIdx.y == 0 && bh % a.H == 0) set_error(a.err, GDN_ERR_PATH);
        }
    }
    __syncthreads();
    const int L = s_L;
    if (L < 0) return;                                   // S_new untouched
    const size_t sb = ((size_t)bh * a.dv + v0) * dk;
    const int quads = dk / 4;
    if (L == 0) {                                        // nothing accepted: S_new = S0
        if (a.S_new != a.S0)
            for (int i = tid; i < rows * quads; i += kGcThreads)
                reinterpret_cast<float4*>(a.S_new + sb)[i] = reinterpret_cast<const float4*>(a.S0 + sb)[i];
        return;
    }
    float* ea = csm;
    float* w = ea + dk;
    float* dl = w + (size_t)L * dk;
    const float* ga = a.g + ((size_t)bh * N + s_nodes[L - 1]) * dk;
    for (int c = tid; c < dk; c += kGcThreads) ea[c] = expf(ga[c]);
    for (int i = tid; i < L * dk; i += kGcThreads) {
        const int j = i / dk, c = i - j * dk;
        const size_t o = ((size_t)bh * N + s_nodes[j]) * dk + c;
        w[i] = ld_elem<T>(static_cast<const T*>(a.key), o) * expf(ga[c] - a.g[o]);
    }
    for (int i = tid; i < L * kGcRows; i += kGcThreads) {
        const int j = i / kGcRows, r = i - j * kGcRows;
        dl[i] = r < rows ? a.delta[((size_t)bh * N + s_nodes[j]) * a.dv + v0 + r] : 0.f;
    }
    __syncthreads();
    for (int i = tid; i < rows * quads; i += kGcThreads) {
        const int r = i / quads, c = 4 * (i - r * quads);
        const float4 s = reinterpret_cast<const float4*>(a.S0 + sb + (size_t)r * dk)[c / 4];
        float4 o = make_float4(s.x * ea[c], s.y * ea[c + 1], s.z * ea[c + 2], s.w * ea[c + 3]);
#pragma unroll 1
        for (int j = 0; j < L; ++j) {
            const float d = dl[j * kGcRows + r];
            const float4 wj = *reinterpret_cast<const float4*>(w + (size_t)j * dk + c);
            o.x = fmaf(d, wj.x, o.x);
            o.y = fmaf(d, wj.y, o.y);
            o.z = fmaf(d, wj.z, o.z);
            o.w = fmaf(d, wj.w, o.w);
        }
        reinterpret_cast<float4*>(a.S_new + sb + (size_t)r * dk)[c / 4] = o;
    }
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dim_ok(int d) { return d >= 16 && d <= kMaxDim && d % 16 == 0; }
bool shape_ok(int B, int N, int H, int dk, int dv) {
    return B >= 1 && H >= 1 && N >= 1 && N <= kMaxNodes && dim_ok(dk) && dim_ok(dv) &&
           (long long)B * H * N * (dk > dv ? dk : dv) <= 0x7fffffffLL;
}
bool overlaps(const void* x, size_t nx, const void* y, size_t ny) {
    const char* a = static_cast<const char*>(x);
    const char* b = static_cast<const char*>(y);
    return a < b + ny && b < a + nx;
}

// Opt a kernel into the largest dynamic shared memory its static part leaves,
// once per device (these kernels' static part alone can take the dynamic part
// past the default 48 KB).
template <typename K>
cudaError_t opt_in_smem(K kernel, bool* done_per_device) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (done_per_device[dev]) return cudaSuccess;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024 - (int)fa.sharedSizeBytes);
    if (e == cudaSuccess) done_per_device[dev] = true;
    return e;
}

template <typename T, bool kTc>
cudaError_t launch_gla_prep(const GlaArgs& g, cudaStream_t s) {
    static bool attr[64];
    const size_t smem = gla_prep_smem(g.N, g.dk, (int)sizeof(T));
    cudaError_t e = opt_in_smem(gla_prep_kernel<T, kTc>, attr);
    if (e != cudaSuccess) return e;
    return launch_kernel(gla_prep_kernel<T, kTc>, dim3(g.B * g.H), dim3(kGThreads), smem, s, false, g);
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" int gdn_gla_factors_bytes(int B, int N, int H, int dk, int dv, int dtype, size_t* bytes) {
    if (bytes == nullptr || !shape_ok(B, N, H, dk, dv) || (dtype != GDN_DTYPE_BF16 && dtype != GDN_DTYPE_F32))
        return GDN_ERR_ARG;
    *bytes = GlaFactorLayout(B, N, H, dk, dv, dtype).total;
    return GDN_OK;
}

extern "C" int gdn_gla_workspace_bytes(int B, int N, int H, int dk, int dv, size_t* bytes) {
    if (bytes == nullptr || !shape_ok(B, N, H, dk, dv)) return GDN_ERR_ARG;
    *bytes = GlaWsLayout(B, N, H, dk, dv).total;
    return GDN_OK;
}

extern "C" int gdn_gla_tree_verify(const void* q, const void* k, const void* v, int dtype, const float* alpha,
                                   const float* beta, const int32_t* parent_idx, const float* S0, float* out,
                                   void* factors, void* workspace, int B, int N, int H, int dk, int dv,
                                   cudaStream_t stream) {
    if (!shape_ok(B, N, H, dk, dv) || (dtype != GDN_DTYPE_BF16 && dtype != GDN_DTYPE_F32)) return GDN_ERR_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(alpha) || !aligned16(beta) ||
        !aligned16(parent_idx) || !aligned16(S0) || !aligned16(out) || !aligned16(factors) || !aligned16(workspace))
        return GDN_ERR_ARG;
    const GlaFactorLayout FL(B, N, H, dk, dv, dtype);
    const GlaWsLayout WL(B, N, H, dk, dv);
    const size_t obytes = (size_t)B * N * H * dv * 4;
    if (overlaps(out, obytes, factors, FL.total) || overlaps(out, obytes, workspace, WL.total) ||
        overlaps(factors, FL.total, workspace, WL.total))
        return GDN_ERR_ARG;
    int st = GDN_OK;
    int* err = current_error_word(&st);
    if (err == nullptr) return st;

    char* f = static_cast<char*>(factors);
    char* ws = static_cast<char*>(workspace);
    GlaArgs g;
    g.q = q;
    g.k = k;
    g.v = v;
    g.alpha = alpha;
    g.beta = beta;
    g.parent = parent_idx;
    g.key = f + FL.key;
    g.g = reinterpret_cast<float*>(f + FL.g);
    g.par_out = reinterpret_cast<int32_t*>(f + FL.parent);
    g.recs = ws + WL.recs;
    g.qhat = ws + WL.qhat;
    g.v32 = dtype == GDN_DTYPE_BF16 ? reinterpret_cast<float*>(ws + WL.v32) : nullptr;
    g.B = B;
    g.N = N;
    g.H = H;
    g.dk = dk;
    g.dv = dv;
    g.err = err;

    // the contraction in linear mode: R = beta v, Delta = T R = R, O = Y_Q + (Attn) R
    VerifyArgs va;
    va.q = g.qhat;
    va.k = g.qhat;                     // its Y_K is not used in linear mode
    va.v = g.v32 != nullptr ? static_cast<const void*>(g.v32) : v;
    va.alpha = alpha;
    va.beta = beta;
    va.parent = parent_idx;
    va.S = const_cast<float*>(S0);
    va.out = out;
    va.f = Factors{reinterpret_cast<float*>(f + FL.delta), f + FL.key, nullptr, nullptr, N};
    va.ws = g.recs;
    va.B = B;
    va.N = N;
    va.H = H;
    va.dk = dk;
    va.dv = dv;
    va.commit = CommitSrc{nullptr, nullptr, nullptr, nullptr, 0, nullptr, 0};
    va.err = err;
    va.overlap = false;
    va.linear = true;
    va.tc = tc_contract_eligible(va);
    cudaError_t e;
    if (va.tc) {
        __nv_bfloat16* qh = static_cast<__nv_bfloat16*>(g.qhat);
        __nv_bfloat16* ql = qh + (size_t)B * N * H * dk;
        va.split[0] = qh;
        va.split[1] = qh;
        va.split[2] = ql;
        va.split[3] = ql;
        e = dtype == GDN_DTYPE_BF16 ? launch_gla_prep<__nv_bfloat16, true>(g, stream) : launch_gla_prep<float, true>(g, stream);
        if (e != cudaSuccess) return GDN_ERR_CUDA;
        // the contraction reads qhat before its programmatic wait: a plain launch after the prologue
        e = launch_tc_contract_only(va, false, stream);
    } else {
        e = dtype == GDN_DTYPE_BF16 ? launch_gla_prep<__nv_bfloat16, false>(g, stream)
                                    : launch_gla_prep<float, false>(g, stream);
        if (e != cudaSuccess) return GDN_ERR_CUDA;
        e = launch_tree_contract_simt_f32(va, stream);
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" int gdn_gla_commit(const float* S0, const void* factors, const int32_t* accepted_path, int Lmax,
                              float* S_new, int B, int N, int H, int dk, int dv, int dtype, cudaStream_t stream) {
    if (!shape_ok(B, N, H, dk, dv) || (dtype != GDN_DTYPE_BF16 && dtype != GDN_DTYPE_F32) || Lmax < 1 ||
        Lmax > kMaxPath)
        return GDN_ERR_ARG;
    if (!aligned16(S0) || !aligned16(factors) || !aligned16(accepted_path) || !aligned16(S_new)) return GDN_ERR_ARG;
    const size_t sbytes = (size_t)B * H * dv * dk * 4;
    const GlaFactorLayout FL(B, N, H, dk, dv, dtype);
    if (S_new != S0 && overlaps(S0, sbytes, S_new, sbytes)) return GDN_ERR_ARG;
    if (overlaps(S_new, sbytes, factors, FL.total)) return GDN_ERR_ARG;
    int st = GDN_OK;
    int* err = current_error_word(&st);
    if (err == nullptr) return st;
    const char* f = static_cast<const char*>(factors);
    GlaCommitArgs a;
    a.S0 = S0;
    a.S_new = S_new;
    a.delta = reinterpret_cast<const float*>(f + FL.delta);
    a.key = f + FL.key;
    a.g = reinterpret_cast<const float*>(f + FL.g);
    a.parent = reinterpret_cast<const int32_t*>(f + FL.parent);
    a.path = accepted_path;
    a.Lmax = Lmax;
    a.B = B;
    a.N = N;
    a.H = H;
    a.dk = dk;
    a.dv = dv;
    a.err = err;
    const size_t smem = gla_commit_smem(Lmax, dk);
    static bool attr_b[64], attr_f[64];
    const dim3 grid(B * H, (dv + kGcRows - 1) / kGcRows);
    cudaError_t e;
    if (dtype == GDN_DTYPE_BF16) {
        e = opt_in_smem(gla_commit_kernel<__nv_bfloat16>, attr_b);
        if (e == cudaSuccess)
            e = launch_kernel(gla_commit_kernel<__nv_bfloat16>, grid, dim3(kGcThreads), smem, stream, false, a);
    } else {
        e = opt_in_smem(gla_commit_kernel<float>, attr_f);
        if (e == cudaSuccess) e = launch_kernel(gla_commit_kernel<float>, grid, dim3(kGcThreads), smem, stream, false, a);
    }
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
