// gdn_internal.cuh -- layouts, argument blocks and device helpers shared by
// the kernels of libgdnspec.so.  Not part of the public ABI (include/gdnspec.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdnspec.h"

namespace gdn {

constexpr int kMaxNodes = 64;     // draft nodes per tree (one uint64 ancestor mask per node)
constexpr int kMaxDim = 256;      // d_k, d_v upper bound
constexpr int kMaxPath = 64;      // accepted path capacity (Lmax)
constexpr size_t kSectionAlign = 256;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline int elem_bytes(int dtype) { return dtype == GDN_DTYPE_F32 ? 4 : 2; }

// ---------------------------------------------------------------------------
// factor buffer: delta fp32 [B][H][N][dv] | key dtype [B][H][N][dk] |
//                g fp32 [B][H][N] | parent int32 [B][N]
// ---------------------------------------------------------------------------
struct FactorLayout {
    size_t delta, key, g, parent, total;
};

inline FactorLayout factor_layout(int B, int N, int H, int dk, int dv, int dtype) {
    FactorLayout L;
    const size_t BHN = (size_t)B * H * N;
    L.delta = 0;
    L.key = align_up(L.delta + BHN * dv * 4, kSectionAlign);
    L.g = align_up(L.key + BHN * dk * elem_bytes(dtype), kSectionAlign);
    L.parent = align_up(L.g + BHN * 4, kSectionAlign);
    L.total = align_up(L.parent + (size_t)B * N * 4, kSectionAlign);
    return L;
}

// Device view of one factor buffer.
struct Factors {
    float* delta;       // [B][H][N][dv]
    void* key;          // [B][H][N][dk], q/k/v element type
    float* g;           // [B][H][N]
    int32_t* parent;    // [B][N]
    int N;
};

inline Factors factors_view(void* base, int B, int N, int H, int dk, int dv, int dtype) {
    FactorLayout L = factor_layout(B, N, H, dk, dv, dtype);
    char* p = static_cast<char*>(base);
    return Factors{reinterpret_cast<float*>(p + L.delta), p + L.key,
                   reinterpret_cast<float*>(p + L.g), reinterpret_cast<int32_t*>(p + L.parent), N};
}

// ---------------------------------------------------------------------------
// tree workspace, one record per (b, h):
//   T  fp32 [N][N]  (I + A)^-1, A = strict-ancestor masked beta_t e^{g_t-g_j} k_t.k_j
//   P  fp32 [N][N]  Attn T, Attn = inclusive masked e^{g_t-g_j} q_t.k_j
//   eg fp32 [N]     e^{g_t}
//   bt fp32 [N]     beta_t
//   anc u64 [N]     inclusive ancestor mask (path(t) as bits)
// ---------------------------------------------------------------------------
struct WsLayout {
    size_t T, P, op, eg, bt, anc, record;
};

// Every section starts on a 16-byte boundary and is padded to a multiple of
// 16 bytes, so kernels may stage whole sections with 16-byte async copies.
__host__ __device__ inline size_t ws_table_bytes(int N) { return align_up((size_t)N * N * 4, 16); }

// The tensor-core contraction's second MMA operand [T; P]: 128 rows (T rows
// 0..63, P rows 64..127) x 64 columns, bf16 hi then lo, each 16 KiB in the
// 128-byte-swizzled K-major shared-memory layout.  It shares storage with the
// fp32 T and P tables (a call uses one form or the other).
constexpr size_t kTcOperandBytes = 2 * 128 * 128;

__host__ __device__ inline WsLayout ws_layout(int N) {
    WsLayout L;
    L.T = 0;
    L.P = L.T + ws_table_bytes(N);
    L.op = 0;
    const size_t tab = 2 * ws_table_bytes(N) > kTcOperandBytes ? 2 * ws_table_bytes(N) : kTcOperandBytes;
    L.eg = tab;
    L.bt = L.eg + align_up((size_t)N * 4, 16);
    L.anc = L.bt + align_up((size_t)N * 4, 16);
    L.record = align_up(L.anc + (size_t)N * 8, kSectionAlign);
    return L;
}

// ---------------------------------------------------------------------------
// argument blocks
// ---------------------------------------------------------------------------
struct CommitSrc {             // accepted path into a previous tree (fused or standalone commit)
    const float* delta;        // prev factors
    const void* key;
    const float* g;
    const int32_t* parent;
    int N;                     // previous tree size
    const int32_t* path;       // [B][Lmax]
    int Lmax;
};

struct VerifyArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* alpha;
    const float* beta;
    const int32_t* parent;     // nullptr for the chain path
    float* S;                  // state (read; read-modify-write when commit.path != nullptr)
    float* out;
    Factors f;                 // new factors
    char* ws;                  // tree workspace
    int B, N, H, dk, dv;
    CommitSrc commit;          // commit.path == nullptr: no fused commit
    int* err;
    bool overlap;              // launch the call's first kernel as a programmatic dependent
    bool tc;                   // the tensor-core contraction runs: prologue writes its operand form
    // fp32 q/k on the tensor-core path: bf16 q_hi, k_hi, q_lo, k_lo with x = hi + lo to
    // ~2^-16 (same layout as q/k); all nullptr otherwise
    const void* split[4] = {nullptr, nullptr, nullptr, nullptr};
    // decay-gated linear attention instead of the gated delta rule: S_t = alpha_t S_p +
    // beta_t v_t k_t^T (no erasure), i.e. A = 0, T = I and delta_t = beta_t v_t
    bool linear = false;
    // the factor record's keys were written by the producer of q/k (the layer's conv
    // kernel): the single-kernel verifier neither copies nor reads the fp32 keys
    bool keys_done = false;
    // first (sequence, head) of the launch: the single-kernel verifier may cover the B*H pairs
    // in two launches (whole waves of one CTA per pair, then the rest as two CTAs per pair)
    int bh_base = 0;
};

struct CommitArgs {
    const float* S0;
    float* S_new;
    CommitSrc src;
    int B, H, dk, dv;
    int* err;
    bool overlap;
};

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void set_error(int* err, int code) { atomicCAS(err, 0, code); }

// The per-device error block: the error word, then (8 bytes on) the limit of
// every bounded device wait in nanoseconds (gdn_set_wait_limit_ns, default one
// second).  Waits read it only once their first poll has failed.
struct ErrorBlock {
    int code;
    int pad;
    unsigned long long wait_limit_ns;
};
constexpr unsigned long long kDefaultWaitLimitNs = 1000000000ull;
__device__ __forceinline__ unsigned long long wait_limit_ns(const int* err) {
    return *reinterpret_cast<const volatile unsigned long long*>(reinterpret_cast<const char*>(err) +
                                                                 offsetof(ErrorBlock, wait_limit_ns));
}

template <typename T>
__device__ __forceinline__ float ld_elem(const T* p, size_t i);
template <>
__device__ __forceinline__ float ld_elem<float>(const float* p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld_elem<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}

template <typename T>
__device__ __forceinline__ void st_elem(T* p, size_t i, float x);
template <>
__device__ __forceinline__ void st_elem<float>(float* p, size_t i, float x) { p[i] = x; }
template <>
__device__ __forceinline__ void st_elem<__nv_bfloat16>(__nv_bfloat16* p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// Packed fp32 pairs: two independent round-to-nearest operations per instruction,
// the same results as two fmaf / products.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long ra, rb, rc, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    unsigned long long ra, rb, rd;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
    float2 d;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
    return d;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Accepted-path check by one full warp: the -1 padded path row must be a
// root-first parent chain of the tree with parents `par` (N entries).  Returns L,
// or -1 if invalid; fills s_nodes[0 .. L).
__device__ inline int path_chain_setup(const int32_t* row, int Lmax, const int32_t* par, int N, int* s_nodes) {
    const int lane = threadIdx.x & 31;
    int n[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) n[s] = lane + 32 * s < Lmax ? row[lane + 32 * s] : -1;
    const unsigned long long nn = (unsigned long long)__ballot_sync(0xffffffffu, n[0] >= 0) |
                                  ((unsigned long long)__ballot_sync(0xffffffffu, n[1] >= 0) << 32);
    const int L = (~nn == 0ull) ? 64 : __ffsll((long long)~nn) - 1;
    bool bad = n[0] < -1 || n[1] < -1 || n[0] >= N || n[1] >= N || nn != (L == 64 ? ~0ull : (1ull << L) - 1ull);
    const int up0 = __shfl_up_sync(0xffffffffu, n[0], 1), up1 = __shfl_up_sync(0xffffffffu, n[1], 1);
    const int last0 = __shfl_sync(0xffffffffu, n[0], 31);
    if (!bad && lane < L) bad = par[n[0]] != (lane == 0 ? -1 : up0);
    if (!bad && lane + 32 < L) bad = par[n[1]] != (lane == 0 ? last0 : up1);
    if (__any_sync(0xffffffffu, bad)) return -1;
    if (lane < L) s_nodes[lane] = n[0];
    if (lane + 32 < L) s_nodes[lane + 32] = n[1];
    return L;
}

// Accepted-path setup, executed by ONE full warp.  Validates the -1 padded,
// root-first path row against the previous tree's parents and fills
//   s_nodes[i]  accepted node i (root first), i < L
//   s_coef[i]   e^{g_a - g_{node i}}, a = last accepted node
//   *s_ega      e^{g_a} (1 when L == 0)
// Returns L (0..Lmax) or -1 if the path is invalid.  The path row, the previous
// tree's parent row and head h's g row (N <= 64 entries each) are read in one
// round trip and looked up per accepted node with shuffles, so the setup costs
// one global-memory latency rather than three dependent ones.
__device__ inline int commit_path_setup(const CommitSrc& c, int b, int h, int H, int* s_nodes,
                                        float* s_coef, float* s_ega) {
    const int lane = threadIdx.x & 31;
    const int32_t* row = c.path + (size_t)b * c.Lmax;
    const int32_t* par = c.parent + (size_t)b * c.N;
    const float* g = c.g + (size_t)(b * H + h) * c.N;
    int n[2], p[2], prev[2];
    float gr[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int i = lane + 32 * s;
        n[s] = i < c.Lmax ? row[i] : -1;
        p[s] = i < c.N ? par[i] : -1;
        gr[s] = i < c.N ? g[i] : 0.f;
    }
    const unsigned nn0 = __ballot_sync(0xffffffffu, n[0] >= 0);
    const unsigned nn1 = __ballot_sync(0xffffffffu, n[1] >= 0);
    const unsigned long long nn = (unsigned long long)nn0 | ((unsigned long long)nn1 << 32);
    const int L = (~nn == 0ull) ? 64 : __ffsll((long long)~nn) - 1;
    bool bad = (n[0] < -1) || (n[1] < -1) || (n[0] >= c.N) || (n[1] >= c.N);
    bad = bad || (nn != (L == 64 ? ~0ull : ((1ull << L) - 1ull)));
    prev[0] = __shfl_up_sync(0xffffffffu, n[0], 1);
    prev[1] = __shfl_up_sync(0xffffffffu, n[1], 1);
    const int carry = __shfl_sync(0xffffffffu, n[0], 31);
    if (lane == 0) {
        prev[0] = -1;
        prev[1] = carry;
    }
    // parent and g of this lane's path entries: entry n of a row sits in lane n & 31 of half n >> 5
    int pn[2];
    float gn[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int src = n[s] & 31;
        const int p0 = __shfl_sync(0xffffffffu, p[0], src), p1 = __shfl_sync(0xffffffffu, p[1], src);
        const float g0 = __shfl_sync(0xffffffffu, gr[0], src), g1 = __shfl_sync(0xffffffffu, gr[1], src);
        pn[s] = n[s] < 32 ? p0 : p1;
        gn[s] = n[s] < 32 ? g0 : g1;
        const int i = lane + 32 * s;
        if (i < L && !bad && n[s] >= 0 && n[s] < c.N && pn[s] != prev[s]) bad = true;
    }
    if (__any_sync(0xffffffffu, bad)) return -1;
    float ga = 0.f;
    if (L > 0) ga = __shfl_sync(0xffffffffu, L - 1 < 32 ? gn[0] : gn[1], (L - 1) & 31);
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int i = lane + 32 * s;
        if (i < L) {
            s_nodes[i] = n[s];
            s_coef[i] = expf(ga - gn[s]);
        }
    }
    if (lane == 0) *s_ega = L > 0 ? expf(ga) : 1.f;
    return L;
}

// ---------------------------------------------------------------------------
// launchers (one per kernel family); each returns the launch status
// ---------------------------------------------------------------------------
cudaError_t launch_tree_mask(const int32_t* parent, int B, int N, uint64_t* mask, int32_t* depth,
                             int* err, cudaStream_t s);
cudaError_t launch_tree_verify(const VerifyArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_chain_verify(const VerifyArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_commit(const CommitArgs& a, int dtype, cudaStream_t s);
// error word of the current device (nullptr and a status on failure) and the
// launch-overlap switch (gdn_api.cu)
int* current_error_word(int* status);
bool launch_overlap_enabled();
// tensor-core prologue + contraction of the tree verifier (gdn_tree_tc.cu)
bool tc_contract_eligible(const VerifyArgs& a);
// Whether launch_tree_tc takes the two-kernel form (which passes the tables
// through the workspace) rather than the single-kernel verifier.
bool tc_uses_workspace(const VerifyArgs& a);
// Whether launch_tree_verify(a, dtype, .) reads or writes a.ws at all.
bool tree_verify_uses_workspace(const VerifyArgs& a, int dtype);
cudaError_t launch_tree_tc(const VerifyArgs& a, cudaStream_t s);
// the contraction kernels alone, after a caller's own prologue (gdn_gla.cu)
cudaError_t launch_tc_contract_only(const VerifyArgs& a, bool programmatic, cudaStream_t s);
cudaError_t launch_tree_contract_simt_f32(const VerifyArgs& a, cudaStream_t s);

}  // namespace gdn

namespace gdn {

// Four consecutive elements starting at p[i] (i a multiple of 4) widened to fp32.
template <typename T>
__device__ __forceinline__ float4 ld4(const T* p, size_t i);
template <>
__device__ __forceinline__ float4 ld4<float>(const float* p, size_t i) {
    return *reinterpret_cast<const float4*>(p + i);
}
template <>
__device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
    const uint2 u = *reinterpret_cast<const uint2*>(p + i);
    float4 r;
    r.x = __uint_as_float(u.x << 16);
    r.y = __uint_as_float(u.x & 0xffff0000u);
    r.z = __uint_as_float(u.y << 16);
    r.w = __uint_as_float(u.y & 0xffff0000u);
    return r;
}

// Eight consecutive elements starting at p[i] (16-byte aligned) widened to fp32.
template <typename T>
__device__ __forceinline__ void ld8(const T* p, float (&x)[8]);
template <>
__device__ __forceinline__ void ld8<float>(const float* p, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0];
    const float4 b = reinterpret_cast<const float4*>(p)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <>
__device__ __forceinline__ void ld8<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// One committed quad of a state row:
//   s' = e^{g_a} s + sum_i cd[i] k_i[c..c+3],  cd[i] = e^{g_a - g_i} delta_i[row]
// with the accepted path's keys staged as rows keys[i][0..dk).  Every commit
// (standalone or fused into a verify) uses this order of operations, so they
// all give identical bits.
template <typename KT>
__device__ __forceinline__ float4 commit_quad(float4 s, float ega, int L, const float* cd,
                                              int cd_stride, const KT* keys, int dk, int c) {
    float4 a;
    a.x = ega * s.x;
    a.y = ega * s.y;
    a.z = ega * s.z;
    a.w = ega * s.w;
#pragma unroll 1
    for (int i = 0; i < L; ++i) {
        const float w = cd[i * cd_stride];
        const float4 kq = ld4<KT>(keys, (size_t)i * dk + c);
        a.x = fmaf(w, kq.x, a.x);
        a.y = fmaf(w, kq.y, a.y);
        a.z = fmaf(w, kq.z, a.z);
        a.w = fmaf(w, kq.w, a.w);
    }
    return a;
}

}  // namespace gdn

namespace gdn {

// ---------------------------------------------------------------------------
// async staging, programmatic dependent launch, launch helper
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy that bypasses registers (both addresses 16-byte aligned).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Cooperative copy of `bytes` (a multiple of 16) with cp.async.
__device__ __forceinline__ void cp_async_block(void* smem, const void* gmem, int bytes, int tid, int nthr) {
    char* d = static_cast<char*>(smem);
    const char* s = static_cast<const char*>(gmem);
#pragma unroll 1
    for (int o = tid * 16; o < bytes; o += nthr * 16) cp_async16(d + o, s + o);
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// serialization attribute may start before its predecessor on the stream has
// finished; griddep_wait() blocks until the predecessor has completed and its
// writes are visible (a no-op for normally launched kernels).  Every kernel of
// this library calls griddep_launch() only after its own griddep_wait(), so a
// kernel's pre-wait section always sees the writes of every kernel launched
// two or more positions earlier on the stream.
// Warm L2 with `bytes` (a multiple of 16, 16-byte aligned) at `src`; no data
// reaches the thread.  L2 is the point of coherence, so a prefetch issued
// before griddep_wait never makes a later load see stale data.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}
// The same for the one L2 line holding `p` (no alignment or size rule).
__device__ __forceinline__ void prefetch_line_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p) : "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, bool programmatic, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device).
template <typename K>
inline cudaError_t ensure_smem(K kernel, size_t bytes, bool* done_per_device) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (bytes > 48 * 1024 && !done_per_device[dev]) {
        cudaFuncAttributes fa;                  // the opt-in limit covers static shared memory too
        e = cudaFuncGetAttributes(&fa, kernel);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 227 * 1024 - (int)fa.sharedSizeBytes);
        if (e != cudaSuccess) return e;
        done_per_device[dev] = true;
    }
    return cudaSuccess;
}

}  // namespace gdn
