// gdn_tree_tc.cu -- tensor-core (tcgen05) tree verifier: for d_v = 256 one
// kernel per call (tree_fused_tc_kernel, further below), otherwise a prologue
// kernel and a contraction kernel over 128-row tiles (described here).
//
// Same mathematics as the SIMT contraction in gdn_tree.cu (review of SpecLA,
// pith.science 7ERME3HB, "Core claim": O = Qhat S0^T - Attn (W S0^T) + Attn U):
//
//   Y = S_tile [Q; K]^T          (the dense part: 4 N d_k d_v FLOP per (b, h))
//   R_t   = beta_t (v_t - e^{g_t} Y_K[:, t])
//   Delta_t = sum_{j in path(t)} T[t,j] R_j
//   O_t     = e^{g_t} Y_Q[:, t] + sum_{j in path(t)} P[t,j] R_j
//
// One CTA owns 128 state rows of one (sequence b, head h) -- the MMA's M --
// and all draft nodes: rows 0..63 of the B operand are the queries of nodes
// 0..63, rows 64..127 their keys (MMA N = 128), so TMEM lane v holds, for state
// row v, every node's Y_Q and Y_K.  d_k is walked in four 64-wide slabs (one
// 128-byte swizzle atom of bf16):
//
//   * the fp32 state slab is loaded to registers (one slab ahead), the
//     pending commit is applied there (fused path), the committed slab is
//     written back, and each value is split into bf16 hi + lo (hi = bf16(x),
//     lo = bf16(x - hi), |x - hi - lo| <= 2^-16 |x|) and stored to shared
//     memory in the 128-byte-swizzled K-major layout;
//   * the query/key slab arrives by TMA (3-D tensor map, 128-byte swizzle);
//   * one thread issues 8 MMAs (4 K-steps x {hi, lo}) of kind::f16 with
//     bf16 operands into one fp32 accumulator in TMEM and commits them to an
//     mbarrier that frees the stage; two stages alternate.
//
// bf16 q/k times the two-term state is exact to ~2^-16 relative per product,
// with fp32 accumulation: far inside the 2e-3 x RMS budget.
//
// Epilogue, also on the tensor core: warps 0-3 read Y_K (TMEM columns 64..127)
// and write R as bf16 hi + lo rows of a second A operand; the prologue kernel
// has already written [T; P] (bf16 hi + lo, swizzled) into the workspace, and
// one bulk copy brings it in.  Twelve MMAs (4 K-steps x {hi.hi, hi.lo, lo.hi})
// give [T R | P R] in TMEM columns 128..255; warps 0-3 store Delta = T R and
// warps 4-7 store O = e^g Y_Q + P R.
//
// Every mbarrier wait is bounded (about one second, then GDN_ERR_TIMEOUT is
// recorded and the CTA skips ahead to its teardown); TMEM is always freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn_internal.cuh"
#include "gdn_prep_common.cuh"
#include "gdn_tc_ptx.cuh"

namespace gdn {
namespace {
using namespace tc;

constexpr int kThreads = 256;
constexpr int kTileV = 128;        // state rows per CTA (MMA M)
constexpr int kSlab = 64;          // d_k per slab
constexpr int kDk = 256;           // d_k handled by this kernel
constexpr int kSlabs = kDk / kSlab;
constexpr int kNodeRows = 64;      // B operand: Q rows 0..63, K rows 64..127 (MMA N = 128)
constexpr int kBufBytes = kTileV * 128;        // one 128-row x 128-byte operand buffer (16 KiB)
// Operand buffers.  bf16 q/k: two stages [A_hi, A_lo, B] (96 KiB).  fp32 q/k
// (hi + lo terms): two A stages [A_hi, A_lo] and one B buffer [B_hi, B_lo]
// (96 KiB), so that two CTAs fit on an SM; slabs take turns in the B buffer.
__host__ __device__ constexpr int a_off(bool split, int st) { return st * (split ? 2 : 3) * kBufBytes; }
__host__ __device__ constexpr int b_off(bool split, int st) {
    return split ? 4 * kBufBytes : st * 3 * kBufBytes + 2 * kBufBytes;
}
__host__ __device__ constexpr int operand_bytes(bool) { return 6 * kBufBytes; }
constexpr uint32_t kTmemCols = 256;     // Y in columns 0..127, [Delta | P R] in 128..255
constexpr int kMaxTcPath = 16;
constexpr uint32_t kIdesc = idesc_bf16(128, 128);   // D fp32, A/B bf16 K-major, M = N = 128

struct TcLayout {
    // offsets from the 1024-aligned base
    int cd, key, coef, nodes, bars, misc, egbt, total;
    __host__ __device__ TcLayout(int Lcap, bool split) {
        int o = operand_bytes(split);
        auto take = [&](int bytes) { int r = o; o += (bytes + 15) / 16 * 16; return r; };
        cd = take(Lcap * kTileV * 4);
        key = take(Lcap * kDk * (split ? 4 : 2));
        coef = take(kMaxPath * 4);
        nodes = take(kMaxPath * 4);
        bars = take(64);
        misc = take(16);
        egbt = take(2 * kNodeRows * 4);
        total = o + 1024;   // slack for aligning the base to 1024 bytes
    }
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// One state slab (this thread's 8 float4 of a 128 x 64 fp32 block) and its
// conversion to the bf16 hi/lo A-operand buffers of one stage.
__device__ __forceinline__ void load_slab(float4 (&x)[8], const float* S, size_t srow0, int rbase, int col) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        x[j] = *reinterpret_cast<const float4*>(S + srow0 + (size_t)(rbase + 16 * j) * kDk + col);
}

// S <- e^{g_a} S + sum_i cd_i[row] k_i[col..col+3], path node outermost (one key
// quad per node serves the thread's 8 rows); per element the same order of
// operations as commit_quad, so the result is bit-identical to gdn_commit.
template <typename KT>
__device__ __forceinline__ void commit_slab(float4 (&x)[8], float ega, int L, const float* s_cd,
                                            const KT* s_key, int rbase, int col) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        x[j].x *= ega;
        x[j].y *= ega;
        x[j].z *= ega;
        x[j].w *= ega;
    }
    for (int i = 0; i < L; ++i) {
        const float4 kq = ld4<KT>(s_key, (size_t)i * kDk + col);
        const float* cdi = s_cd + i * kTileV + rbase;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float w = cdi[16 * j];
            x[j].x = fmaf(w, kq.x, x[j].x);
            x[j].y = fmaf(w, kq.y, x[j].y);
            x[j].z = fmaf(w, kq.z, x[j].z);
            x[j].w = fmaf(w, kq.w, x[j].w);
        }
    }
}

__device__ __forceinline__ void store_slab(const float4 (&x)[8], float* S, size_t srow0, int rbase, int col) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float4*>(S + srow0 + (size_t)(rbase + 16 * j) * kDk + col) = x[j];
}

// hi = bf16(x), lo = bf16(x - hi), stored to the stage's swizzled K-major buffers.
__device__ __forceinline__ void convert_slab(const float4 (&x)[8], unsigned char* ahi, int rbase, int c4) {
    unsigned char* alo = ahi + kBufBytes;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int r = rbase + 16 * j;
        const float4 v = x[j];
        const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y);
        const __nv_bfloat162 h23 = __floats2bfloat162_rn(v.z, v.w);
        const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
        uint2 hi, lo;
        hi.x = *reinterpret_cast<const uint32_t*>(&h01);
        hi.y = *reinterpret_cast<const uint32_t*>(&h23);
        lo.x = pack_bf16(v.x - f01.x, v.y - f01.y);
        lo.y = pack_bf16(v.z - f23.x, v.w - f23.y);
        const uint32_t off = sw128_quad(r, c4);
        *reinterpret_cast<uint2*>(ahi + off) = hi;
        *reinterpret_cast<uint2*>(alo + off) = lo;
    }
}

// Four K-steps of one slab into the Y accumulator: state hi and lo terms times
// bf16 q/k, plus state hi times the lo term of fp32 q/k (the lo.lo product,
// ~2^-16 of the hi.lo ones, is dropped).
template <bool kSplit>
__device__ __forceinline__ void issue_slab_mma(uint32_t tmem, uint32_t a_s, uint32_t bsm, bool first) {
    const uint32_t a_hi = a_s, a_lo = a_s + kBufBytes;
#pragma unroll
    for (int kk = 0; kk < kSlab / 16; ++kk) {
        const uint64_t bd = sw128_desc(bsm + kk * 32);
        mma_bf16(tmem, sw128_desc(a_hi + kk * 32), bd, kIdesc, (!first || kk > 0) ? 1u : 0u);
        mma_bf16(tmem, sw128_desc(a_lo + kk * 32), bd, kIdesc, 1u);
        if (kSplit) mma_bf16(tmem, sw128_desc(a_hi + kk * 32), sw128_desc(bsm + kBufBytes + kk * 32), kIdesc, 1u);
    }
}

template <bool kSplit>
__device__ __forceinline__ void issue_qk_tma(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmQl,
                                             const CUtensorMap* tmKl, uint32_t bsm, int ks, int h, int row0,
                                             uint32_t bar) {
    mbar_expect_tx(bar, (kSplit ? 4 : 2) * kNodeRows * 128);
    tma_load_3d(bsm, tmQ, ks * kSlab, h, row0, bar);
    tma_load_3d(bsm + kNodeRows * 128, tmK, ks * kSlab, h, row0, bar);
    if (kSplit) {
        tma_load_3d(bsm + kBufBytes, tmQl, ks * kSlab, h, row0, bar);
        tma_load_3d(bsm + kBufBytes + kNodeRows * 128, tmKl, ks * kSlab, h, row0, bar);
    }
}

template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 2)
    tree_contract_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmQl, const __grid_constant__ CUtensorMap tmKl,
                            VerifyArgs a) {
    using KT = typename std::conditional<kSplit, float, __nv_bfloat16>::type;   // key / v element type
    constexpr uint32_t kA0 = a_off(kSplit, 0), kA1 = a_off(kSplit, 1);
    constexpr uint32_t kB0 = b_off(kSplit, 0), kB1 = b_off(kSplit, 1);   // the same buffer for fp32 q/k
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    unsigned char* base = smem_raw + (base_s - raw_s);
    const bool fused = a.commit.path != nullptr;
    const TcLayout Ly(fused ? a.commit.Lmax : 0, kSplit);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int N = a.N, dv = a.dv;
    const int v0 = blockIdx.y * kTileV;

    float* s_cd = reinterpret_cast<float*>(base + Ly.cd);
    KT* s_key = reinterpret_cast<KT*>(base + Ly.key);
    float* s_coef = reinterpret_cast<float*>(base + Ly.coef);
    int* s_nodes = reinterpret_cast<int*>(base + Ly.nodes);
    const uint32_t bar_tma0 = base_s + Ly.bars, bar_mma0 = base_s + Ly.bars + 16;
    const uint32_t bar_op = base_s + Ly.bars + 32, bar_e = base_s + Ly.bars + 40, bar_eg = base_s + Ly.bars + 48;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(base + Ly.misc);
    float* s_ega = reinterpret_cast<float*>(base + Ly.misc + 4);
    int* s_flag = reinterpret_cast<int*>(base + Ly.misc + 8);   // path length, or -1: skip the CTA
    float* seg = reinterpret_cast<float*>(base + Ly.egbt);
    float* sbt = seg + kNodeRows;
    const uint32_t a0_s = base_s + kA0, a1_s = base_s + kA1, b0_s = base_s + kB0, b1_s = base_s + kB1;

    if (tid == 0) {
        mbar_init(bar_tma0, 1);
        mbar_init(bar_tma0 + 8, 1);
        mbar_init(bar_mma0, 1);
        mbar_init(bar_mma0 + 8, 1);
        mbar_init(bar_op, 1);
        mbar_init(bar_e, 1);
        mbar_init(bar_eg, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        fence_proxy_async_smem();
        *s_flag = 0;
        *s_ega = 1.f;
    }
    if (warp == 1) tmem_alloc(smem_u32(s_tmem), kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    // ---- 1. before the wait: the state tile (the whole HBM stream of this CTA) and
    // Y = S [Q; K]^T.  Only this call's prologue kernel runs before the wait
    // releases (it starts this kernel after its own wait), and it touches neither
    // S, the previous factors nor q/k/v; every kernel before it has completed.
    // So the committed state may be written, and q/k read, here.
    if (tid == 0) {
        issue_qk_tma<kSplit>(&tmQ, &tmK, &tmQl, &tmKl, b0_s, 0, h, b * N, bar_tma0);
        if (!kSplit) issue_qk_tma<kSplit>(&tmQ, &tmK, &tmQl, &tmKl, b1_s, 1, h, b * N, bar_tma0 + 8);
    }
    const size_t srow0 = ((size_t)bh * dv + v0) * kDk;
    const int c4 = tid & 15;         // column quad within a slab
    const int rbase = tid >> 4;      // rows rbase + 16 j, j = 0..7
    if (tid < 8) bulk_prefetch_l2(a.S + srow0 + (size_t)tid * 16 * kDk, 16 * kDk * 4);
    float4 x0[8], x1[8];
    load_slab(x0, a.S, srow0, rbase, 4 * c4);
    if (fused) {
        if (warp == 2) {
            const int L = commit_path_setup(a.commit, b, h, a.H, s_nodes, s_coef, s_ega);
            if (lane == 0) {
                *s_flag = L;
                if (L < 0) set_error(a.err, GDN_ERR_PATH);
            }
        }
        __syncthreads();
        const int L = *s_flag;
        if (L > 0) {
            const KT* key_bh = static_cast<const KT*>(a.commit.key) + (size_t)bh * a.commit.N * kDk;
            for (int i = 0; i < L; ++i)
                cp_async_block(s_key + (size_t)i * kDk, key_bh + (size_t)s_nodes[i] * kDk, kDk * (int)sizeof(KT),
                               tid, kThreads);
            const float* dl = a.commit.delta + (size_t)bh * a.commit.N * dv;
            for (int i = tid; i < L * kTileV; i += kThreads) {
                const int j = i / kTileV, r = i % kTileV;
                s_cd[i] = s_coef[j] * dl[(size_t)s_nodes[j] * dv + v0 + r];
            }
            cp_async_wait_all();
        }
    }
    __syncthreads();
    const int L = fused ? *s_flag : 0;
    const bool commit_ok = L >= 0;
    const float ega = *s_ega;
    // slabs 0 and 1 -> stage buffers; committed slabs 2 and 3 stay in registers
    float4 x2[8], x3[8];
    load_slab(x1, a.S, srow0, rbase, kSlab + 4 * c4);
    if (fused && commit_ok) {
        commit_slab(x0, ega, L, s_cd, s_key, rbase, 4 * c4);
        store_slab(x0, a.S, srow0, rbase, 4 * c4);
    }
    convert_slab(x0, base + kA0, rbase, c4);
    load_slab(x2, a.S, srow0, rbase, 2 * kSlab + 4 * c4);
    if (fused && commit_ok) {
        commit_slab(x1, ega, L, s_cd, s_key, rbase, kSlab + 4 * c4);
        store_slab(x1, a.S, srow0, rbase, kSlab + 4 * c4);
    }
    convert_slab(x1, base + kA1, rbase, c4);
    load_slab(x3, a.S, srow0, rbase, 3 * kSlab + 4 * c4);
    if (fused && commit_ok) {
        commit_slab(x2, ega, L, s_cd, s_key, rbase, 2 * kSlab + 4 * c4);
        store_slab(x2, a.S, srow0, rbase, 2 * kSlab + 4 * c4);
        commit_slab(x3, ega, L, s_cd, s_key, rbase, 3 * kSlab + 4 * c4);
        store_slab(x3, a.S, srow0, rbase, 3 * kSlab + 4 * c4);
    }
    fence_proxy_async_smem();
    __syncthreads();

    // Y slabs 0 and 1 (their q/k copies were issued at the start; both must land
    // before the CTA may exit), then slabs 2 and 3 through the freed stages
    bool ok = commit_ok;
    if (tid == 0) {
        const bool l0 = mbar_wait(bar_tma0, 0, a.err);
        if (ok && l0) {
            tc_fence_after();
            issue_slab_mma<kSplit>(tmem, a0_s, b0_s, true);
            mma_commit(bar_mma0);
        }
        bool l1 = true;
        if (kSplit) {                  // slab 1 takes the B buffer once slab 0's MMAs are done
            l1 = ok && l0 && mbar_wait(bar_mma0, 0, a.err);
            if (l1) issue_qk_tma<kSplit>(&tmQ, &tmK, &tmQl, &tmKl, b1_s, 1, h, b * N, bar_tma0 + 8);
        }
        l1 = l1 && mbar_wait(bar_tma0 + 8, 0, a.err);
        if (ok && l0 && l1) {
            tc_fence_after();
            issue_slab_mma<kSplit>(tmem, a1_s, b1_s, false);
            mma_commit(bar_mma0 + 8);
        }
        ok = ok && l0 && l1;
    }
    ok = __syncthreads_and(ok);
    if (ok) {
        ok = mbar_wait(bar_mma0, 0, a.err);
        if (kSplit) ok = mbar_wait(bar_mma0 + 8, 0, a.err) && ok;   // B is free once slab 1 is done
        if (tid == 0 && ok) issue_qk_tma<kSplit>(&tmQ, &tmK, &tmQl, &tmKl, b0_s, 2, h, b * N, bar_tma0);
        convert_slab(x2, base + kA0, rbase, c4);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0 && ok) {
            ok = mbar_wait(bar_tma0, 1, a.err);
            if (ok) {
                tc_fence_after();
                issue_slab_mma<kSplit>(tmem, a0_s, b0_s, false);
                mma_commit(bar_mma0);
            }
        }
        ok = mbar_wait(bar_mma0 + 8, 0, a.err) && ok;
        if (kSplit) ok = mbar_wait(bar_mma0, 1, a.err) && ok;       // B is free once slab 2 is done
        if (tid == 0 && ok) issue_qk_tma<kSplit>(&tmQ, &tmK, &tmQl, &tmKl, b1_s, 3, h, b * N, bar_tma0 + 8);
        convert_slab(x3, base + kA1, rbase, c4);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0 && ok) {
            ok = mbar_wait(bar_tma0 + 8, 1, a.err);
            if (ok) {
                tc_fence_after();
                issue_slab_mma<kSplit>(tmem, a1_s, b1_s, false);
                mma_commit(bar_mma0 + 8);
            }
        }
    }
    const bool y_issued = __syncthreads_and(ok);

    // ---- 2. wait for the prologue kernel's outputs ----
    griddep_wait();
    griddep_launch();
    const WsLayout wl = ws_layout(N);
    const char* rec = a.ws + (size_t)bh * wl.record;
    const bool run = y_issued && *reinterpret_cast<const uint64_t*>(rec + wl.anc) != ~0ull;
    ok = y_issued;

    if (y_issued) {                               // the Y MMAs are in flight: wait for them in any case
        if (tid == 0 && run) {
            mbar_expect_tx(bar_eg, 2 * kNodeRows * 4);
            bulk_copy_g2s(smem_u32(seg), rec + wl.eg, kNodeRows * 4, bar_eg);
            bulk_copy_g2s(smem_u32(sbt), rec + wl.bt, kNodeRows * 4, bar_eg);
        }
        // Stage 0 is free once slab 2 is done: the [T; P] operand (bf16 hi, lo) into its
        // A buffers and this tile's v rows into its B buffer, by bulk copies.
        ok = mbar_wait(bar_mma0, 1, a.err);
        if (kSplit) ok = ok && mbar_wait(bar_mma0 + 8, 1, a.err);   // the v rows go into the one B buffer
        const uint32_t op_s = a0_s;                                    // B2: hi, then lo (16 KiB each)
        const uint32_t r_s = a1_s;                                     // A2: R hi, then lo
        const uint32_t v_s = b0_s;                                     // v rows: [t][128]
        if (ok && run && warp == 0) {
            if (lane == 0) {
                mbar_expect_tx(bar_op, (uint32_t)(kTcOperandBytes + N * kTileV * (int)sizeof(KT)));
                bulk_copy_g2s(op_s, rec + wl.op, (uint32_t)kTcOperandBytes, bar_op);
            }
            __syncwarp();
            const KT* vv = static_cast<const KT*>(a.v);
            for (int t = lane; t < N; t += 32)
                bulk_copy_g2s(v_s + t * kTileV * (int)sizeof(KT), vv + (((size_t)b * N + t) * a.H + h) * dv + v0,
                              kTileV * (int)sizeof(KT), bar_op);
        }
        if (ok) ok = mbar_wait(bar_mma0 + 8, 1, a.err);                // Y complete
        ok = ok && run;
        if (ok) ok = mbar_wait(bar_op, 0, a.err);                      // operand and v rows landed
        if (ok) ok = mbar_wait(bar_eg, 0, a.err);                      // e^g and beta landed
        ok = __syncthreads_and(ok);
        tc_fence_after();

        const int v = 32 * (warp & 3) + lane;            // state row of this thread (TMEM lane)
        const uint32_t t_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        const KT* vsm = reinterpret_cast<const KT*>(base + kB0);        // v rows: [t][128]
        if (ok) {
            // R[v, t] = beta_t (v_t[v] - e^{g_t} Y_K[v, t]) (0 for t >= N) as bf16 hi + lo rows of
            // the second MMA's A operand (row v, 64 columns t); warps 0-3 take t < 32, warps 4-7 the rest
            unsigned char* rhi = base + kA1;
            unsigned char* rlo = rhi + kBufBytes;
            const int c = warp >> 2;
            float yk[32];
            tmem_ld32(t_lane + kNodeRows + 32 * c, yk);
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i0 = 8 * q8 + 2 * e, i1 = i0 + 1;
                    const int t0 = 32 * c + i0, t1 = t0 + 1;
                    const float ek0 = a.linear ? 0.f : seg[t0] * yk[i0], ek1 = a.linear ? 0.f : seg[t1] * yk[i1];
                    const float r0 = t0 < N ? sbt[t0] * (to_f32(vsm[t0 * kTileV + v]) - ek0) : 0.f;
                    const float r1 = t1 < N ? sbt[t1] * (to_f32(vsm[t1 * kTileV + v]) - ek1) : 0.f;
                    const __nv_bfloat162 hh = __floats2bfloat162_rn(r0, r1);
                    const float2 hf = __bfloat1622float2(hh);
                    const __nv_bfloat162 ll = __floats2bfloat162_rn(r0 - hf.x, r1 - hf.y);
                    hi[e] = *reinterpret_cast<const uint32_t*>(&hh);
                    lo[e] = *reinterpret_cast<const uint32_t*>(&ll);
                }
                const int cc = 4 * c + q8;                           // 16-byte chunk = 8 nodes
                const uint32_t off = (uint32_t)(v * 128 + ((cc ^ (v & 7)) << 4));
                *reinterpret_cast<uint4*>(rhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(rlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && ok) {
            // [Delta | P R] (v, t) = sum_j R[v, j] [T; P](t, j): three bf16 terms (hi.hi, hi.lo, lo.hi)
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kNodeRows / 16; ++kk) {
                const uint64_t ahi = sw128_desc(r_s + kk * 32), alo = sw128_desc(r_s + kBufBytes + kk * 32);
                const uint64_t bhi = sw128_desc(op_s + kk * 32), blo = sw128_desc(op_s + kBufBytes + kk * 32);
                mma_bf16(tmem + 128, ahi, bhi, kIdesc, kk > 0 ? 1u : 0u);
                mma_bf16(tmem + 128, ahi, blo, kIdesc, 1u);
                mma_bf16(tmem + 128, alo, bhi, kIdesc, 1u);
            }
            mma_commit(bar_e);
        }
        if (ok) ok = mbar_wait(bar_e, 0, a.err);
        tc_fence_after();
        if (ok && warp < 4) {
            // Delta_t[v] = (T R)[v, t]
#pragma unroll
            for (int c = 0; c < kNodeRows / 32; ++c) {
                if (32 * c >= N) break;
                float d[32];
                tmem_ld32(t_lane + 128 + 32 * c, d);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int t = 32 * c + i;
                    if (t < N) a.f.delta[((size_t)bh * N + t) * dv + v0 + v] = d[i];
                }
            }
        } else if (ok) {
            // O_t[v] = e^{g_t} Y_Q[v, t] + (P R)[v, t]
#pragma unroll
            for (int c = 0; c < kNodeRows / 32; ++c) {
                if (32 * c >= N) break;
                float yq[32], pr[32];
                tmem_ld32(t_lane + 32 * c, yq);
                tmem_ld32(t_lane + 192 + 32 * c, pr);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int t = 32 * c + i;
                    if (t < N) a.out[(((size_t)b * N + t) * a.H + h) * dv + v0 + v] = fmaf(seg[t], yq[i], pr[i]);
                }
            }
        }
    }

    // ---- teardown: TMEM is always released ----
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// prologue on the tensor core: masked Gram from one MMA
// ---------------------------------------------------------------------------
constexpr int kPrepThreads = 256;
constexpr uint32_t kPrepTmemCols = 64;
constexpr uint32_t kGramIdesc = idesc_bf16(128, 64);   // [Q; K] (128 rows) x K^T (64 keys)

struct PrepTcLayout {
    // offsets from the 1024-aligned base; the first 64 KiB hold [Q; K] as four
    // 64-column slabs (rows 0..63 queries, 64..127 keys), 128-byte swizzled.
    // Once the Gram MMA has consumed them and the keys are copied out, the
    // A, Attn and T tables reuse that space.
    int G, A, At, T, plist, par, anc, la, g, beta, depth, bars, misc, total, ld;
    __host__ __device__ PrepTcLayout(int N, bool split) {
        ld = N + 1;
        int o = 0;
        auto take = [&](int bytes) { int r = o; o += (bytes + 15) / 16 * 16; return r; };
        A = take(N * ld * 4);
        At = take(N * ld * 4);
        T = take(N * ld * 4);
        o = kSlabs * kBufBytes;   // [Q; K]: four slabs, or for fp32 q/k two (hi, lo) slab pairs in turn
        G = take(128 * 65 * 4);          // Gram rows: q_t.k_j (rows 0..63), k_t.k_j (rows 64..127)
        plist = take(N * 64);
        par = take(N * 4);
        anc = take(N * 8);
        la = take(N * 4);
        g = take(N * 4);
        beta = take(N * 4);
        depth = take(N * 4);
        bars = take(48);
        misc = take(16);
        total = o + 1024;
    }
};

// One CTA per (sequence b, head h).  Q and K of the tree arrive by TMA in the
// MMA's swizzled layout; one tcgen05 MMA (M = 128 [Q; K] rows, N = 64 keys,
// K = 256) gives every q_t.k_j and k_t.k_j in TMEM (bf16 products are exact in
// fp32, accumulation in fp32); the masked entries, the per-node solves and
// the outputs follow as in the SIMT prologue.  Writes the tensor-core operand
// form of [T; P].
// At most 128 registers per thread, so that a prologue CTA and a contraction
// CTA (of the previous or the same call) fit on one SM together.
template <bool kSplit>
__global__ void __launch_bounds__(kPrepThreads, 2)
    tree_prep_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmQl, const __grid_constant__ CUtensorMap tmKl,
                        VerifyArgs a) {
    constexpr uint32_t kPair = 2 * kBufBytes;           // fp32 q/k: one slab's hi and lo terms (32 KiB)
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    unsigned char* base = smem_raw + (base_s - raw_s);
    const int N = a.N, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const PrepTcLayout Ly(N, kSplit);
    const int ld = Ly.ld;
    float* sG = reinterpret_cast<float*>(base + Ly.G);
    float* sA = reinterpret_cast<float*>(base + Ly.A);
    float* sAt = reinterpret_cast<float*>(base + Ly.At);
    float* sT = reinterpret_cast<float*>(base + Ly.T);
    uint8_t* plist = reinterpret_cast<uint8_t*>(base + Ly.plist);
    int* par = reinterpret_cast<int*>(base + Ly.par);
    uint64_t* anc = reinterpret_cast<uint64_t*>(base + Ly.anc);
    float* la = reinterpret_cast<float*>(base + Ly.la);
    float* sg = reinterpret_cast<float*>(base + Ly.g);
    float* sbeta = reinterpret_cast<float*>(base + Ly.beta);
    int* sdepth = reinterpret_cast<int*>(base + Ly.depth);
    const uint32_t bar_tma = base_s + Ly.bars, bar_mma = base_s + Ly.bars + 8;
    const uint32_t bar_tma1 = base_s + Ly.bars + 16, bar_free0 = base_s + Ly.bars + 24,
                   bar_free1 = base_s + Ly.bars + 32;    // fp32 q/k: second slab buffer
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(base + Ly.misc);

    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const WsLayout wl = ws_layout(N);
    char* rec = a.ws + (size_t)bh * wl.record;

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_tma1, 1);
        mbar_init(bar_free0, 1);
        mbar_init(bar_free1, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        fence_proxy_async_smem();
    }
    if (warp == 1) tmem_alloc(smem_u32(s_tmem), kPrepTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    // This layer's q/k/v rows into L2 while the previous kernel on the stream
    // finishes; its inputs may come from that kernel, so they are read only
    // after the wait.
    if (tid < N) {
        const size_t rt = ((size_t)b * N + tid) * a.H + h;
        const uint32_t esz = kSplit ? 4u : 2u;
        if (kSplit) {
            for (int i = 0; i < 4; ++i) prefetch_l2(static_cast<const __nv_bfloat16*>(a.split[i]) + rt * kDk, kDk * 2);
            prefetch_l2(static_cast<const float*>(a.k) + rt * kDk, kDk * 4);
            prefetch_l2(static_cast<const float*>(a.v) + rt * a.dv, (uint32_t)a.dv * 4);
        } else {
            prefetch_l2(static_cast<const __nv_bfloat16*>(a.q) + rt * kDk, kDk * esz);
            prefetch_l2(static_cast<const __nv_bfloat16*>(a.k) + rt * kDk, kDk * esz);
            prefetch_l2(static_cast<const __nv_bfloat16*>(a.v) + rt * a.dv, (uint32_t)a.dv * esz);
        }
    }
    griddep_wait();
    griddep_launch();

    // fp32 q/k: slab sl's hi and lo terms into pair buffer j (hi at +0, lo at +16 KiB)
    auto load_pair = [&](int sl, int j, uint32_t bar) {
        const uint32_t dst = base_s + j * kPair;
        mbar_expect_tx(bar, 2 * 2 * kNodeRows * 128);
        tma_load_3d(dst, &tmQ, sl * kSlab, h, b * N, bar);
        tma_load_3d(dst + kNodeRows * 128, &tmK, sl * kSlab, h, b * N, bar);
        tma_load_3d(dst + kBufBytes, &tmQl, sl * kSlab, h, b * N, bar);
        tma_load_3d(dst + kBufBytes + kNodeRows * 128, &tmKl, sl * kSlab, h, b * N, bar);
    };
    if (tid == 0) {
        if (kSplit) {
            load_pair(0, 0, bar_tma);
            load_pair(1, 1, bar_tma1);
        } else {
            mbar_expect_tx(bar_tma, (uint32_t)(kSlabs * 2 * kNodeRows * 128));
#pragma unroll
            for (int sl = 0; sl < kSlabs; ++sl) {
                tma_load_3d(base_s + sl * kBufBytes, &tmQ, sl * kSlab, h, b * N, bar_tma);
                tma_load_3d(base_s + sl * kBufBytes + kNodeRows * 128, &tmK, sl * kSlab, h, b * N, bar_tma);
            }
        }
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
    bad = __syncthreads_or(bad);
    bool ok = mbar_wait(bar_tma, 0, a.err);       // the copies land even if the tree is rejected
    if (kSplit) ok = mbar_wait(bar_tma1, 0, a.err) && ok;
    if (bad && tid == 0) {
        set_error(a.err, GDN_ERR_TREE);
        *reinterpret_cast<uint64_t*>(rec + wl.anc) = ~0ull;   // record marked invalid
    }
    if (!bad) {
        if (tid == 128 && ok) {                  // a warp with no per-node work issues the Gram MMA
            tc_fence_after();
            if (kSplit) {
                // hi.hi, hi.lo and lo.hi terms, two slabs at a time through the two pair buffers
                auto pair_mma = [&](int sl, int j) {
#pragma unroll
                    for (int kk = 0; kk < kSlab / 16; ++kk) {
                        const uint32_t q_s = base_s + j * kPair + kk * 32, l_s = q_s + kBufBytes;
                        mma_bf16(tmem, sw128_desc(q_s), sw128_desc(q_s + kNodeRows * 128), kGramIdesc,
                                 (sl > 0 || kk > 0) ? 1u : 0u);
                        mma_bf16(tmem, sw128_desc(q_s), sw128_desc(l_s + kNodeRows * 128), kGramIdesc, 1u);
                        mma_bf16(tmem, sw128_desc(l_s), sw128_desc(q_s + kNodeRows * 128), kGramIdesc, 1u);
                    }
                };
                pair_mma(0, 0);
                mma_commit(bar_free0);
                pair_mma(1, 1);
                mma_commit(bar_free1);
                bool l2 = mbar_wait(bar_free0, 0, a.err);
                if (l2) load_pair(2, 0, bar_tma);
                bool l3 = mbar_wait(bar_free1, 0, a.err);
                if (l3) load_pair(3, 1, bar_tma1);
                l2 = l2 && mbar_wait(bar_tma, 1, a.err);
                if (l2) {
                    tc_fence_after();
                    pair_mma(2, 0);
                }
                l3 = l3 && mbar_wait(bar_tma1, 1, a.err);
                if (l3) {
                    tc_fence_after();
                    pair_mma(3, 1);
                }
                if (l2 && l3) mma_commit(bar_mma);   // a lost copy leaves bar_mma open: the wait below times out
            } else {
#pragma unroll
                for (int sl = 0; sl < kSlabs; ++sl)
#pragma unroll
                    for (int kk = 0; kk < kSlab / 16; ++kk) {
                        const uint32_t q_s = base_s + sl * kBufBytes + kk * 32;
                        mma_bf16(tmem, sw128_desc(q_s), sw128_desc(q_s + kNodeRows * 128), kGramIdesc,
                                 (sl > 0 || kk > 0) ? 1u : 0u);
                    }
                mma_commit(bar_mma);
            }
        }
        if (tid < N) {
            prep::node_meta(tid, N, par, la, anc, sdepth, sg, plist);
        } else if (kSplit) {
            // fp32 keys into the factor record, from the fp32 inputs
            float* key_out = static_cast<float*>(a.f.key) + (size_t)bh * N * kDk;
            const float* kin = static_cast<const float*>(a.k);
            for (int item = tid - N; item < N * (kDk / 4); item += kPrepThreads - N) {
                const int t = item / (kDk / 4), c4 = item % (kDk / 4);
                *reinterpret_cast<float4*>(key_out + (size_t)t * kDk + 4 * c4) =
                    *reinterpret_cast<const float4*>(kin + (((size_t)b * N + t) * a.H + h) * kDk + 4 * c4);
            }
        } else {
            // keys into the factor record, unswizzled from the K half of the operand
            __nv_bfloat16* key_out = static_cast<__nv_bfloat16*>(a.f.key) + (size_t)bh * N * kDk;
            for (int item = tid - N; item < N * kSlabs * 8; item += kPrepThreads - N) {
                const int t = item / (kSlabs * 8), sl = (item / 8) % kSlabs, cc = item % 8;
                const uint4 x = *reinterpret_cast<const uint4*>(base + sl * kBufBytes + (kNodeRows + t) * 128 +
                                                                ((cc ^ (t & 7)) << 4));
                *reinterpret_cast<uint4*>(key_out + (size_t)t * kDk + sl * kSlab + cc * 8) = x;
            }
        }
        ok = mbar_wait(bar_mma, 0, a.err) && ok;
        tc_fence_after();
        if (ok && warp < 4) {                     // TMEM lane = operand row
            const uint32_t t_lane = tmem + ((uint32_t)(32 * warp) << 16);
            const int r = 32 * warp + lane;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float gr[32];
                tmem_ld32(t_lane + 32 * c, gr);
#pragma unroll
                for (int i = 0; i < 32; ++i) sG[r * 65 + 32 * c + i] = gr[i];
            }
        }
        __syncthreads();                          // [Q; K] consumed: A, Attn, T reuse its space
        if (tid < N)
            prep::gram_row(tid, sdepth[tid], plist, sG + tid * 65, sG + (kNodeRows + tid) * 65, ld, sg, sbeta,
                           sA, sAt, !a.linear);
        __syncthreads();
        prep::solve_rows_fast(tid, N, ld, sdepth, plist, sA, sAt, sT);
        prep::write_operand(tid, kPrepThreads, N, ld, anc, sA, sT, reinterpret_cast<unsigned char*>(rec + wl.op));
        prep::write_meta(tid, N, b, h, bh, rec, wl, sg, sbeta, anc, par, a.f);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kPrepTmemCols);
    }
}

// ---------------------------------------------------------------------------
// the whole call in one kernel: one CTA per (sequence, head), d_v = 256
// ---------------------------------------------------------------------------
// A CTA owns its (sequence, head)'s whole state (two 128-row MMA tiles, u = 0,
// 1) and runs the prologue itself, so a call is a single launch:
//   before the wait: one warp reads the pending commit's accepted path,
//     parents and gates in one round trip and brings the path's key and delta
//     rows in by bulk copies, while every thread has state slabs 0 and 1 in
//     flight; those two slabs are committed in registers, written back and
//     turned into bf16 hi/lo operand stages; slabs 2 and 3 are only brought
//     into L2;
//   after the wait: q/k slabs by TMA; per slab the Y MMAs of both tiles and
//     the Gram MMA ([Q; K] K^T: M = 128 rows, N = 64 keys) on the same operand
//     buffer, issued by lane 0 of warp 4; slabs 2 and 3 are read from L2,
//     committed and written back while the first MMAs run, and take the stages
//     over once slabs 0 and 1 are consumed -- by the other fifteen warps (warps
//     8-15 take warp 4's share), which arrive at a named barrier per slab that
//     only the issuer waits on; the node metadata meanwhile;
//   then warps 0-7 turn the Gram rows into the A and Attn tables and solve T
//     and P, while warps 8-15 form R of both tiles from Y_K, v and the gates;
//     all sixteen warps then write the [T; P] operand; one MMA group per tile gives [Delta | P R]
//     (committed per tile); warps 8-15 copy the keys into the factor record
//     while it runs; every warp stores Delta or O rows.
// TMEM, 512 columns: Y of tile u in 128u .. 128u+127 ([Y_Q | Y_K]); the Gram
// in 256 .. 319 until it is read; [Delta | P R] of tile u in 256+128u .. +127.
constexpr int kFThreads = 512;
constexpr int kFRows = 256;                          // state rows per CTA (= d_v)
constexpr uint32_t kFTmemCols = 512;
constexpr int kFAStage = 4 * kBufBytes;              // one slab of both tiles: [hi 0, lo 0, hi 1, lo 1]
constexpr uint32_t kFGramIdesc = idesc_bf16(128, 64);
constexpr int kFSmemLimit = 227 * 1024;
constexpr int kFIssuerWarp = 4;                      // lane 0 issues the TMA copies and the MMAs; the
                                                     // other lanes wait at __syncwarp, not on mbarriers

struct FusedLayout {
    // offsets from the 1024-aligned base.  The operand region holds two A
    // stages and nB q/k buffers during Y, then R (both tiles), the A / Attn / T
    // tables and the [T; P] operand.
    int nB, bsz, ops, R, A, At, T, op;
    int vs, cd, key, nodes, coef, par, la, g, beta, eg, bk, depth, anc, plist, bars, misc, total;
    __host__ __device__ FusedLayout(int N, int Lcap, bool split) {
        bsz = (split ? 2 : 1) * kBufBytes;
        build(N, Lcap, split, 2);
        if (total > kFSmemLimit) build(N, Lcap, split, 1);
    }
    __host__ __device__ void build(int N, int Lcap, bool split, int nb) {
        nB = nb;
        ops = 2 * kFAStage + nb * bsz;
        int o = 0;
        auto take = [&](int bytes) { int r = o; o += (bytes + 15) / 16 * 16; return r; };
        R = take(2 * 2 * kBufBytes);
        A = take(N * (N + 1) * 4);
        At = take(N * (N + 1) * 4);
        T = take(N * (N + 1) * 4);
        o = (o + 1023) / 1024 * 1024;
        op = take((int)kTcOperandBytes);
        if (o > ops) {   // cannot happen for N <= 64; flagged as too large
            total = 1 << 30;
            return;
        }
        o = ops;
        vs = take(split ? 0 : N * kFRows * 2);      // bf16 v rows [t][256], copied after the wait
        cd = take(Lcap * kFRows * 4);
        key = take(Lcap * kDk * (split ? 4 : 2));
        nodes = take(kMaxPath * 4);
        coef = take(kMaxPath * 4);
        par = take(kMaxNodes * 4);
        la = take(kMaxNodes * 4);
        g = take(kMaxNodes * 4);
        beta = take(kMaxNodes * 4);
        eg = take(kMaxNodes * 4);
        bk = take(kMaxNodes * 8);
        depth = take(kMaxNodes * 4);
        anc = take(kMaxNodes * 8);
        plist = take(kMaxNodes * 64);
        bars = take(16 * 8);
        misc = take(32);
        total = o + 1024;   // slack for aligning the base to 1024 bytes
    }
};

// Named barrier `id` of `count` threads: arrive without waiting (the arrival
// orders this thread's earlier shared-memory writes before the barrier completes),
// or wait for it to complete.
__device__ __forceinline__ void named_barrier_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}

// L2 cache policy of the state stream: the state is read and written once per
// call, so its lines go first (the call's inputs and the kernel stay resident).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
    return p;
}

// Rows rbase + kRS j (j = 0 .. J-1) of a CTA's state slab.  With the default
// kRS = 32 and J = 4 per 128-row tile, j < 4 lie in its tile 0, j >= 4 in tile 1.
template <int J, int kRS = 32>
__device__ __forceinline__ void f_load_slab(float4 (&x)[8], const float* S, size_t srow0, int rbase, int col,
                                            uint64_t pol) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const float* p = S + srow0 + (size_t)(rbase + kRS * j) * kDk + col;
        asm volatile("ld.global.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;\n"
                     : "=f"(x[j].x), "=f"(x[j].y), "=f"(x[j].z), "=f"(x[j].w)
                     : "l"(p), "l"(pol));
    }
}
template <int J, int kRS = 32>
__device__ __forceinline__ void f_store_slab(const float4 (&x)[8], float* S, size_t srow0, int rbase, int col,
                                             uint64_t pol) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
        float* p = S + srow0 + (size_t)(rbase + kRS * j) * kDk + col;
        asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;\n" ::"l"(p), "f"(x[j].x),
                     "f"(x[j].y), "f"(x[j].z), "f"(x[j].w), "l"(pol)
                     : "memory");
    }
}
// Same arithmetic order per element as commit_slab (and gdn_commit), in packed
// fp32 pairs (each lane one correctly rounded product or fma, so the bits are
// those of the scalar form).  s_cd rows are the (sequence, head)'s 256 state
// rows; cd_row0 is this thread's first.
template <int J, typename KT, int kRS = 32>
__device__ __forceinline__ void f_commit_slab(float4 (&x)[8], float ega, int L, const float* s_cd,
                                              const KT* s_key, int cd_row0, int col) {
    const float2 e2 = make_float2(ega, ega);
    float2 lo[J], hi[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        lo[j] = fmul2(make_float2(x[j].x, x[j].y), e2);
        hi[j] = fmul2(make_float2(x[j].z, x[j].w), e2);
    }
#pragma unroll 1
    for (int i = 0; i < L; ++i) {
        const float4 kq = ld4<KT>(s_key, (size_t)i * kDk + col);
        const float2 k01 = make_float2(kq.x, kq.y), k23 = make_float2(kq.z, kq.w);
        const float* cdi = s_cd + i * kFRows + cd_row0;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const float w = cdi[kRS * j];
            const float2 w2 = make_float2(w, w);
            lo[j] = ffma2(w2, k01, lo[j]);
            hi[j] = ffma2(w2, k23, hi[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < J; ++j) x[j] = make_float4(lo[j].x, lo[j].y, hi[j].x, hi[j].y);
}
// hi/lo split into one A stage ([tile 0 hi, tile 0 lo, tile 1 hi, tile 1 lo]).
template <int J>
__device__ __forceinline__ void f_convert_slab(const float4 (&x)[8], unsigned char* stage, int rbase, int c4) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
        unsigned char* ahi = stage + (j >> 2) * 2 * kBufBytes;
        unsigned char* alo = ahi + kBufBytes;
        const int r = rbase + 32 * (j & 3);
        const float4 v = x[j];
        const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y);
        const __nv_bfloat162 h23 = __floats2bfloat162_rn(v.z, v.w);
        const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
        uint2 hi, lo;
        hi.x = *reinterpret_cast<const uint32_t*>(&h01);
        hi.y = *reinterpret_cast<const uint32_t*>(&h23);
        lo.x = pack_bf16(v.x - f01.x, v.y - f01.y);
        lo.y = pack_bf16(v.z - f23.x, v.w - f23.y);
        const uint32_t off = sw128_quad(r, c4);
        *reinterpret_cast<uint2*>(ahi + off) = hi;
        *reinterpret_cast<uint2*>(alo + off) = lo;
    }
}

// Y of the CTA's kT tiles and the Gram for one slab (one thread issues).  Not inlined:
// the fused kernel runs each of its code paths once per CTA, so its size in
// the instruction cache matters more than a call.
template <bool kSplit, int kT>
__device__ __noinline__ void f_issue_slab(uint32_t tmem, uint32_t a_stage, uint32_t bsm, bool first) {
    issue_slab_mma<kSplit>(tmem, a_stage, bsm, first);
    if (kT == 2) issue_slab_mma<kSplit>(tmem + 128, a_stage + 2 * kBufBytes, bsm, first);
#pragma unroll
    for (int kk = 0; kk < kSlab / 16; ++kk) {
        const uint32_t q_s = bsm + kk * 32;
        const uint64_t a_hi = sw128_desc(q_s), k_hi = sw128_desc(q_s + kNodeRows * 128);
        mma_bf16(tmem + 256, a_hi, k_hi, kFGramIdesc, (!first || kk > 0) ? 1u : 0u);
        if (kSplit) {
            const uint32_t l_s = q_s + kBufBytes;
            mma_bf16(tmem + 256, a_hi, sw128_desc(l_s + kNodeRows * 128), kFGramIdesc, 1u);
            mma_bf16(tmem + 256, sw128_desc(l_s), k_hi, kFGramIdesc, 1u);
        }
    }
}

// kT = 2: the CTA owns all 256 state rows of its (sequence, head); kT = 1: rows
// 128 y .. 128 y + 127 (y = blockIdx.y), the N x N prologue repeated by both CTAs
// of a (sequence, head) -- for small batches, where the two CTAs still fit in one
// wave and each then carries half the MMAs, R rows and stores.
template <bool kSplit, int kT>
__global__ void __launch_bounds__(kFThreads, 1)
    tree_fused_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmQl, const __grid_constant__ CUtensorMap tmKl,
                         VerifyArgs a) {
    using KT = typename std::conditional<kSplit, float, __nv_bfloat16>::type;   // key / v element type
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw_s = smem_u32(smem_raw);
    const uint32_t base_s = (raw_s + 1023u) & ~1023u;
    unsigned char* base = smem_raw + (base_s - raw_s);
    const bool fused = a.commit.path != nullptr;
    const int N = a.N, H = a.H, ld = N + 1;
    const FusedLayout Ly(N, fused ? a.commit.Lmax : 0, kSplit);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = a.bh_base + (int)blockIdx.x, b = bh / H, h = bh % H;
    const int row0 = kT == 1 ? 128 * (int)blockIdx.y : 0;    // the CTA's first state row
    const bool lead = row0 == 0;                            // writes the per-(b, h) factor parts
    constexpr int kJ = 4 * kT;                              // state rows per thread and slab

    float* s_cd = reinterpret_cast<float*>(base + Ly.cd);
    KT* s_key = reinterpret_cast<KT*>(base + Ly.key);
    int* s_nodes = reinterpret_cast<int*>(base + Ly.nodes);
    float* s_coef = reinterpret_cast<float*>(base + Ly.coef);
    int* par = reinterpret_cast<int*>(base + Ly.par);
    float* la = reinterpret_cast<float*>(base + Ly.la);
    float* sg = reinterpret_cast<float*>(base + Ly.g);
    float* sbeta = reinterpret_cast<float*>(base + Ly.beta);
    float* seg = reinterpret_cast<float*>(base + Ly.eg);
    float2* sbk = reinterpret_cast<float2*>(base + Ly.bk);       // (beta_t, beta_t e^{g_t}) for R, 0 past N
    int* sdepth = reinterpret_cast<int*>(base + Ly.depth);
    uint64_t* anc = reinterpret_cast<uint64_t*>(base + Ly.anc);
    uint8_t* plist = reinterpret_cast<uint8_t*>(base + Ly.plist);
    float* sA = reinterpret_cast<float*>(base + Ly.A);
    float* sAt = reinterpret_cast<float*>(base + Ly.At);
    float* sT = reinterpret_cast<float*>(base + Ly.T);
    const uint32_t bars = base_s + Ly.bars;
    const uint32_t bar_e = bars + 64;                         // bars + 8 s: slab s copied; + 32 + 8 s: its MMAs done
    const uint32_t bar_v = bars + 72;                         // v rows landed (bf16 inputs)
    const uint32_t bar_c = bars + 80;                         // the commit's key and delta rows landed
    const uint32_t bar_e2 = bars + 88;                        // the second MMA of tile 1 done (kT = 2)
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(base + Ly.misc);
    int* s_flag = reinterpret_cast<int*>(base + Ly.misc + 4);    // path length, or -1: skip the CTA
    float* s_ega = reinterpret_cast<float*>(base + Ly.misc + 8);
    int* s_vcopy = reinterpret_cast<int*>(base + Ly.misc + 12);  // the v-row copies were issued
    int* s_qkmask = reinterpret_cast<int*>(base + Ly.misc + 16); // bit s: the q/k copy of slab s was issued
    int* s_fail = reinterpret_cast<int*>(base + Ly.misc + 20);   // a worker's wait gave up in a slab step
    const uint32_t stage0 = base_s, stage1 = base_s + kFAStage, bbase = base_s + 2 * kFAStage;
    const int nB = Ly.nB;
    auto bbuf = [&](int s) { return bbase + (nB == 2 ? (uint32_t)((s & 1) * Ly.bsz) : 0u); };
    // After the wait the issuer warp holds no state rows: the J elements of each of its
    // threads in slabs 2 and 3 are taken by threads 256 .. 256 + 32 J - 1 (warps 8-15),
    // one each, so that the issuer's MMA issue and its waits never hold up the stage
    // that the next slab's barrier waits for.
    const bool helper = tid >= 256 && tid < 256 + 32 * kJ;
    const int hx = tid - 256, hw = hx & 31, hj = hx >> 5;              // issuer lane, element
    const int h_rb = (32 * kFIssuerWarp + hw) >> 4, h_c4 = hw & 15;     // its rbase and column quad
    const int h_row = h_rb + 32 * hj;                                   // the element's state row
    const uint32_t vrows_s = base_s + Ly.vs;

    if (fused && warp == 2 && lane < 6) {   // the pending commit's path, parent and g rows, first of all
        const int r = lane >> 1, half = lane & 1;
        const char* row = r == 0   ? reinterpret_cast<const char*>(a.commit.path + (size_t)b * a.commit.Lmax)
                          : r == 1 ? reinterpret_cast<const char*>(a.commit.parent + (size_t)b * a.commit.N)
                                   : reinterpret_cast<const char*>(a.commit.g + (size_t)bh * a.commit.N);
        const int bytes = 4 * (r == 0 ? a.commit.Lmax : a.commit.N);
        if (128 * half < bytes) prefetch_line_l2(row + 128 * half);
    }
    if (tid == 0) {
        for (int i = 0; i < 12; ++i) mbar_init(bars + 8 * i, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        fence_proxy_async_smem();
        *s_flag = 0;
        *s_ega = 1.f;
        *s_vcopy = 0;
        *s_qkmask = 0;
        *s_fail = 0;
    }
    if (warp == 1) tmem_alloc(smem_u32(s_tmem), kFTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    // ---- 1. before the wait: the state stream (it only reads the state and the
    // previous factors, which the previous call on the stream does not touch) ----
    const size_t srow0 = ((size_t)bh * kFRows + row0) * kDk;
    const int c4 = tid & 15;          // column quad within a slab
    const int rbase = tid >> 4;       // rows rbase + 32 j
    if (fused && warp == 2) {
        // the path, then its key and delta rows by bulk copies issued from this warp
        const int L = commit_path_setup(a.commit, b, h, H, s_nodes, s_coef, s_ega);
        if (lane == 0) {
            *s_flag = L;
            if (L < 0) set_error(a.err, GDN_ERR_PATH);
        }
        if (L > 0) {
            const KT* key_bh = static_cast<const KT*>(a.commit.key) + (size_t)bh * a.commit.N * kDk;
            const float* dl = a.commit.delta + (size_t)bh * a.commit.N * kFRows;
            constexpr uint32_t kKeyBytes = kDk * sizeof(KT), kCdBytes = kFRows * 4;
            if (lane == 0) mbar_expect_tx(bar_c, (uint32_t)L * (kKeyBytes + kCdBytes));
            __syncwarp();
            for (int j = lane; j < L; j += 32) {     // s_nodes[j] was written by this lane
                const int nd = s_nodes[j];
                bulk_copy_g2s(smem_u32(s_key) + (uint32_t)j * kKeyBytes, key_bh + (size_t)nd * kDk, kKeyBytes,
                              bar_c);
                bulk_copy_g2s(smem_u32(s_cd + (size_t)j * kFRows), dl + (size_t)nd * kFRows, kCdBytes, bar_c);
            }
        }
    }
    const uint64_t pol_first = l2_policy_evict_first();
    float4 cur[8], nxt[8];             // slabs 0 and 1 in flight during the commit setup
    f_load_slab<kJ>(cur, a.S, srow0, rbase, 4 * c4, pol_first);
    f_load_slab<kJ>(nxt, a.S, srow0, rbase, kSlab + 4 * c4, pol_first);
    bool landed = true;
    if (fused) {
        __syncthreads();
        const int L = *s_flag;
        if (L > 0) {
            landed = mbar_wait(bar_c, 0, a.err);
            if (landed)
                for (int i = tid; i < L * kFRows; i += kFThreads) s_cd[i] *= s_coef[i / kFRows];
        }
    }
    landed = __syncthreads_and(landed);
    if (tid < 128 * kT) bulk_prefetch_l2(a.S + srow0 + (size_t)tid * kDk + 2 * kSlab, 2 * kSlab * 4);
    const int L = fused ? *s_flag : 0;
    bool ok = L >= 0 && landed;
    // This call's q/k/v rows are not prefetched into L2 before the wait: with all CTAs
    // streaming their state, the prefetch cost more than the copies after the wait gained.
    const float ega = *s_ega;
    if (ok) {
        // slabs 0 and 1: commit, write back, into the operand stages.  Slabs 2 and 3
        // only go to L2 here: they are committed and written back after the wait,
        // while the first MMAs run, so that the state writes of all CTAs do not
        // crowd into this phase, which every CTA of the call runs at the same time.
#pragma unroll 1
        for (int sl = 0; sl < 2; ++sl) {
            if (fused) {
                f_commit_slab<kJ>(cur, ega, L, s_cd, s_key, row0 + rbase, sl * kSlab + 4 * c4);
                f_store_slab<kJ>(cur, a.S, srow0, rbase, sl * kSlab + 4 * c4, pol_first);
            }
            f_convert_slab<kJ>(cur, base + sl * kFAStage, rbase, c4);
#pragma unroll
            for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
        }
        fence_proxy_async_smem();
        __syncthreads();       // every thread's part of stages 0 and 1 is in place before the first MMA
    }

    // ---- 2. this call's inputs ----
    griddep_wait();
    griddep_launch();
    float4 ecur[8], enxt[8];           // a helper's element of the issuer's rows in slabs 2 and 3 ([0] only)
    if (ok) {
        // this thread's part of slabs 2 and 3 as they were before the commit (L2)
        // (slab 3's loads only once the thread has committed slab 2, so that they do not compete
        // with slab 2's)
        if (warp != kFIssuerWarp) f_load_slab<kJ>(cur, a.S, srow0, rbase, 2 * kSlab + 4 * c4, pol_first);
        if (helper) f_load_slab<1>(ecur, a.S, srow0, h_row, 2 * kSlab + 4 * h_c4, pol_first);
        if (warp == kFIssuerWarp && lane == 0) {
            issue_qk_tma<kSplit>(&tmQ, &tmK, &tmQl, &tmKl, bbuf(0), 0, h, b * N, bars);
            if (nB == 2) issue_qk_tma<kSplit>(&tmQ, &tmK, &tmQl, &tmKl, bbuf(1), 1, h, b * N, bars + 8);
            *s_qkmask = nB == 2 ? 0x3 : 0x1;
        }
        if (!kSplit && warp == kFIssuerWarp + 1) {   // this (sequence, head)'s v rows, one node per lane
            if (lane == 0) {
                mbar_expect_tx(bar_v, (uint32_t)(N * kFRows * 2));
                *s_vcopy = 1;
            }
            __syncwarp();
            for (int t = lane; t < N; t += 32)
                bulk_copy_g2s(vrows_s + t * kFRows * 2,
                              static_cast<const KT*>(a.v) + (((size_t)b * N + t) * H + h) * kFRows, kFRows * 2, bar_v);
        }
        // parents and gates: loads issued now, used once the Y MMAs are under way
        int p_in = 0;
        float al_in = 1.f, be_in = 0.f;
        if (tid < N) {
            const size_t gi = ((size_t)b * N + tid) * H + h;
            p_in = a.parent[(size_t)b * N + tid];
            al_in = a.alpha[gi];
            be_in = a.beta[gi];
        }

        // ---- 3. Y of both tiles and the Gram, slab by slab.  Slab s: (s >= 2) its
        // state part into the stage slab s - 2 has freed, after which the workers
        // arrive at named barrier s and go on; lane 0 of the issuer warp waits there,
        // issues the slab's MMAs once its q/k copy has landed, then the copy into the
        // q/k buffer that the MMAs of slab s + 1 - nB free ----
#pragma unroll 1
        for (int sl = 0; sl < kSlabs; ++sl) {
            if (sl >= 2) {
                unsigned char* stage = base + (sl & 1) * kFAStage;
                if (warp != kFIssuerWarp) {
                    if (fused && ok) {             // commit slab sl and write it back
                        f_commit_slab<kJ>(cur, ega, L, s_cd, s_key, row0 + rbase, sl * kSlab + 4 * c4);
                        f_store_slab<kJ>(cur, a.S, srow0, rbase, sl * kSlab + 4 * c4, pol_first);
                        if (helper) {
                            f_commit_slab<1>(ecur, ega, L, s_cd, s_key, row0 + h_row, sl * kSlab + 4 * h_c4);
                            f_store_slab<1>(ecur, a.S, srow0, h_row, sl * kSlab + 4 * h_c4, pol_first);
                        }
                    }
                    if (sl == 2) {                 // slab 3 only now, behind slab 2's loads
                        f_load_slab<kJ>(nxt, a.S, srow0, rbase, 3 * kSlab + 4 * c4, pol_first);
                        if (helper) f_load_slab<1>(enxt, a.S, srow0, h_row, 3 * kSlab + 4 * h_c4, pol_first);
                    }
                    ok = ok && mbar_wait(bars + 32 + 8 * (sl - 2), 0, a.err);
                    if (ok) {
                        f_convert_slab<kJ>(cur, stage, rbase, c4);
                        if (helper)
                            f_convert_slab<1>(ecur, stage + (hj >> 2) * 2 * kBufBytes, h_rb + 32 * (hj & 3), h_c4);
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
                    ecur[0] = enxt[0];
                    fence_proxy_async_smem();
                    if (!ok) *s_fail = 1;
                    named_barrier_arrive(sl, kFThreads);
                } else {
                    named_barrier_sync(sl, kFThreads);
                    ok = ok && *s_fail == 0;
                }
            }
            if (ok && warp == kFIssuerWarp) {
                if (lane == 0) {
                    bool l = mbar_wait(bars + 8 * sl, 0, a.err);
                    if (l) {
                        tc_fence_after();
                        f_issue_slab<kSplit, kT>(tmem, (sl & 1) ? stage1 : stage0, bbuf(sl), sl == 0);
                        mma_commit(bars + 32 + 8 * sl);
                    }
                    const int sn = sl + nB;                             // next copy into bbuf(sl)
                    if (sn < kSlabs) {
                        l = l && mbar_wait(bars + 32 + 8 * sl, 0, a.err);
                        if (l) {
                            issue_qk_tma<kSplit>(&tmQ, &tmK, &tmQl, &tmKl, bbuf(sn), sn, h, b * N, bars + 8 * sn);
                            *s_qkmask |= 1 << sn;
                        }
                    }
                }
                __syncwarp();
            }
        }
        // fp32 v rows (read in place by R) into L2 while the last slab's MMAs and the tables run
        if (kSplit && ok && tid < N)
            bulk_prefetch_l2(static_cast<const KT*>(a.v) + (((size_t)b * N + tid) * H + h) * kFRows + row0,
                             (uint32_t)(128 * kT * sizeof(KT)));
        // node metadata while the last slab's MMAs run
        bool bad = false;
        if (tid < N) {
            bad = p_in < -1 || p_in >= tid;
            par[tid] = p_in;
            la[tid] = logf(al_in);
            sbeta[tid] = be_in;
        }
        if (tid >= N && tid < kMaxNodes) sbk[tid] = make_float2(0.f, 0.f);
        bad = __syncthreads_or(bad);
        if (bad) {
            if (tid == 0) set_error(a.err, GDN_ERR_TREE);
        } else if (tid < N) {
            prep::node_meta(tid, N, par, la, anc, sdepth, sg, plist);
            seg[tid] = expf(sg[tid]);
            sbk[tid] = make_float2(sbeta[tid], a.linear ? 0.f : sbeta[tid] * seg[tid]);
            if (lead) {
                a.f.g[(size_t)bh * N + tid] = sg[tid];
                if (h == 0) a.f.parent[(size_t)b * N + tid] = par[tid];
            }
        }
        if (ok) ok = mbar_wait(bars + 56, 0, a.err);              // Y and the Gram complete
        ok = __syncthreads_and(ok) && !bad;
        tc_fence_after();

        // ---- 4. warps 0-7: tables, T, P and the [T; P] operand; warps 8-15: R ----
        if (ok) {
            if (warp < 8) {
                // raw Gram rows into the tables, in place of the entries gram_row turns into
                // A and Attn: TMEM lane r < 64 holds q_r . k_j, lane 64 + r holds k_r . k_j;
                // warps w and w + 4 read the same lanes, columns 0..31 and 32..63
                const int t = tid & 63;
                float* row = ((tid & 127) < 64 ? sAt : sA) + t * ld;
                const uint32_t t_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 256;
                const int c = 32 * (warp >> 2);
                if (c < N) {                         // one 32-column load (a single wait)
                    float gr[32];
                    tmem_ld32(t_lane + c, gr);
                    if (t < N) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (c + i < N) row[c + i] = gr[i];
                    }
                }
            }
            if (tid < 256) {
                prep::group_sync(256);
                if ((tid >> 2) < N)          // four threads per node, path entries strided by four
                    prep::gram_row_part(tid >> 2, tid & 3, 4, sdepth[tid >> 2], plist, sAt + (tid >> 2) * ld,
                                        sA + (tid >> 2) * ld, ld, sg, sbeta, sA, sAt, !a.linear);
                prep::group_sync(256);
                prep::solve_rows_fast<9>(tid, N, ld, sdepth, plist, sA, sAt, sT, 256);
                // T and P are in place: warps 8-15, done with R by now, take half of the operand
                named_barrier_arrive(5, kFThreads);
                prep::write_operand(tid, kFThreads, N, ld, anc, sA, sT, base + Ly.op);
            } else {
                // R[v, t] = beta_t (v_t[v] - e^{g_t} Y_K[v, t]) (0 for t >= N) of tile u as bf16
                // hi + lo rows of the second MMA's A operand (row v, 64 columns t).  kT = 2:
                // warps 8-11 tile 0, 12-15 tile 1; kT = 1: they split the nodes of tile 0.
                const int u = kT == 2 ? (warp - 8) >> 2 : 0;
                const int tbeg = kT == 2 ? 0 : 32 * ((warp - 8) >> 2), tend = kT == 2 ? kNodeRows : tbeg + 32;
                const int v = 32 * (warp & 3) + lane;               // row within the tile = TMEM lane
                const uint32_t t_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 128 * u + kNodeRows;
                unsigned char* rhi = base + Ly.R + u * 2 * kBufBytes;
                unsigned char* rlo = rhi + kBufBytes;
                // one 16-byte chunk of R (8 nodes from t0) from Y_K, the gates and v
                auto r_chunk = [&](int t0, const float (&yk)[8], const float (&vt)[8]) {
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float r[2];
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const float2 c = sbk[t0 + 2 * e + q];   // zeros past N, where v is 0 too
                            r[q] = fmaf(-c.y, yk[2 * e + q], c.x * vt[2 * e + q]);
                        }
                        const __nv_bfloat162 hh = __floats2bfloat162_rn(r[0], r[1]);
                        const float2 hf = __bfloat1622float2(hh);
                        const __nv_bfloat162 ll = __floats2bfloat162_rn(r[0] - hf.x, r[1] - hf.y);
                        hi[e] = *reinterpret_cast<const uint32_t*>(&hh);
                        lo[e] = *reinterpret_cast<const uint32_t*>(&ll);
                    }
                    const int cc = t0 >> 3;
                    const uint32_t off = (uint32_t)(v * 128 + ((cc ^ (v & 7)) << 4));
                    *reinterpret_cast<uint4*>(rhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(rlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                };
                if constexpr (kSplit) {
                    // fp32 v from global memory, a 32-node chunk's loads in flight together
                    const KT* vin =
                        static_cast<const KT*>(a.v) + ((size_t)b * N * H + h) * kFRows + row0 + 128 * u + v;
#pragma unroll 1
                    for (int c = tbeg / 32; c < tend / 32; ++c) {
                        float vt[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            vt[i] = 32 * c + i < N ? vin[(size_t)(32 * c + i) * H * kFRows] : 0.f;
                        float yk32[32];
                        tmem_ld32(t_lane + 32 * c, yk32);
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8) {
                            float yk[8], v8[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                yk[i] = yk32[8 * q8 + i];
                                v8[i] = vt[8 * q8 + i];
                            }
                            r_chunk(32 * c + 8 * q8, yk, v8);
                        }
                    }
                } else {
                    // bf16 v rows staged in shared memory
                    const KT* vsm = reinterpret_cast<const KT*>(base + (vrows_s - base_s)) + row0 + 128 * u + v;
                    const bool vok = mbar_wait(bar_v, 0, a.err);
#pragma unroll 1
                    for (int c0 = tbeg; c0 < tend; c0 += 32) {      // 32 nodes per TMEM load
                        float yk32[32];
                        tmem_ld32(t_lane + c0, yk32);
#pragma unroll
                        for (int q8 = 0; q8 < 4; ++q8) {
                            const int t0 = c0 + 8 * q8;
                            float yk[8], v8[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                yk[i] = yk32[8 * q8 + i];
                                v8[i] = t0 + i < N && vok ? to_f32(vsm[(t0 + i) * kFRows]) : 0.f;
                            }
                            r_chunk(t0, yk, v8);
                        }
                    }
                }
                named_barrier_sync(5, kFThreads);     // the tables' T and P rows
                prep::write_operand(tid, kFThreads, N, ld, anc, sA, sT, base + Ly.op);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // keys into the factor record (warps 8-15, while the second MMA runs)
        if (ok && tid >= 256) {
            // four 16-byte loads in flight per thread
            constexpr int kVec = 16 / (int)sizeof(KT), kRow = kDk / kVec, kBatch = 4;
            const KT* kin = static_cast<const KT*>(a.k);
            KT* kout = static_cast<KT*>(a.f.key) + (size_t)bh * N * kDk;
            const int items = lead && !a.keys_done ? N * kRow : 0;
#pragma unroll 1
            for (int i0 = tid - 256; i0 < items; i0 += kBatch * (kFThreads - 256)) {
                uint4 x[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int item = i0 + u * (kFThreads - 256), t = item / kRow, c = item % kRow;
                    if (item < items)
                        x[u] = *reinterpret_cast<const uint4*>(kin + (((size_t)b * N + t) * H + h) * kDk + c * kVec);
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int item = i0 + u * (kFThreads - 256), t = item / kRow, c = item % kRow;
                    if (item < items) *reinterpret_cast<uint4*>(kout + (size_t)t * kDk + c * kVec) = x[u];
                }
            }
        }

        // ---- 5. [Delta | P R] = R [T; P]^T per tile: three bf16 terms (hi.hi, hi.lo, lo.hi) ----
        if (ok && warp == kFIssuerWarp) {
            if (lane == 0) {
            tc_fence_after();
            const uint32_t op_s = base_s + Ly.op;
#pragma unroll 1
            for (int u = 0; u < kT; ++u) {
                const uint32_t r_s = base_s + Ly.R + u * 2 * kBufBytes;
#pragma unroll
                for (int kk = 0; kk < kNodeRows / 16; ++kk) {
                    const uint64_t ahi = sw128_desc(r_s + kk * 32), alo = sw128_desc(r_s + kBufBytes + kk * 32);
                    const uint64_t bhi = sw128_desc(op_s + kk * 32), blo = sw128_desc(op_s + kBufBytes + kk * 32);
                    const uint32_t d = tmem + 256 + 128 * u;
                    mma_bf16(d, ahi, bhi, kIdesc, kk > 0 ? 1u : 0u);
                    mma_bf16(d, ahi, blo, kIdesc, 1u);
                    mma_bf16(d, alo, bhi, kIdesc, 1u);
                }
                mma_commit(u == 0 ? bar_e : bar_e2);   // tile 0's stores start while tile 1's MMAs run
            }
            }
            __syncwarp();
        }
        if (ok) ok = mbar_wait(kT == 2 && warp >= 8 ? bar_e2 : bar_e, 0, a.err);
        tc_fence_after();
        if (ok) {
            if constexpr (kT == 2) {
                // warp w: tile w >> 3, nodes 32 ((w >> 2) & 1) .. +31, first their Delta rows, then
                // their O rows, so that every warp carries the same share of reads and stores
                const int u = warp >> 3, t0 = 32 * ((warp >> 2) & 1);
                const int row = 128 * u + 32 * (warp & 3) + lane;
                const uint32_t t_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
                if (t0 < N) {
                    const int tend = min(N, t0 + 32);
                    {
                        float x[32];
                        tmem_ld32(t_lane + 256 + 128 * u + t0, x);            // T R
                        float* dst = a.f.delta + (size_t)bh * N * kFRows + row;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (t0 + i < tend) dst[(size_t)(t0 + i) * kFRows] = x[i];
                    }
                    float x[32], yq[32];
                    tmem_ld32(t_lane + 256 + 128 * u + kNodeRows + t0, x);   // P R
                    tmem_ld32(t_lane + 128 * u + t0, yq);                    // Y_Q
                    float* dst = a.out + ((size_t)b * N * H + h) * kFRows + row;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (t0 + i < tend) dst[(size_t)(t0 + i) * H * kFRows] = fmaf(seg[t0 + i], yq[i], x[i]);
                }
            } else {
                // kT = 1: warps 0-3 / 8-11 Delta of nodes 0..31 / 32..63, warps 4-7 / 12-15 O
                const int tbeg = 32 * (warp >> 3), tend = min(N, tbeg + 32);
                const int row = row0 + 32 * (warp & 3) + lane;
                const bool is_o = ((warp >> 2) & 1) != 0;
                const uint32_t t_lane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
                const uint32_t src = t_lane + 256 + (is_o ? kNodeRows : 0);   // T R or P R
                float* dst = is_o ? a.out + ((size_t)b * N * H + h) * kFRows + row : a.f.delta + (size_t)bh * N * kFRows + row;
                const size_t dstep = is_o ? (size_t)H * kFRows : (size_t)kFRows;
                if (tbeg < tend) {                                  // one chunk of 32 nodes
                    float x[32], yq[32];
                    tmem_ld32(src + tbeg, x);
                    if (is_o) tmem_ld32(t_lane + tbeg, yq);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int t = tbeg + i;
                        if (t < tend) dst[(size_t)t * dstep] = is_o ? fmaf(seg[t], yq[i], x[i]) : x[i];
                    }
                }
            }
        }
    }

    // ---- teardown: every copy into shared memory has landed; TMEM is always released ----
    if (tid == 0) {
        if (!kSplit && *s_vcopy) mbar_wait(bar_v, 0, a.err);
        for (int s = 0; s < kSlabs; ++s)      // done already unless a wait gave up on the way
            if ((*s_qkmask >> s) & 1) mbar_wait(bars + 8 * s, 0, a.err);
    }
    if (!landed && tid == 0) mbar_wait(bar_c, 0, a.err);    // the commit copies, before the CTA's memory goes
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kFTmemCols);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// q or k [B][N][H][256] bf16 viewed as 3-D (d_k, H, B*N); box = one 64-wide
// slab of 64 consecutive nodes of one head.
bool make_qk_map(CUtensorMap* m, const void* ptr, int B, int N, int H) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kDk, (cuuint64_t)H, (cuuint64_t)B * N};
    const cuuint64_t strides[2] = {(cuuint64_t)kDk * 2, (cuuint64_t)H * kDk * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kSlab, 1u, (cuuint32_t)kNodeRows};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// bf16 inputs, d_k = 256, d_v a multiple of 128 and accepted paths of at most
// 16 nodes; otherwise the SIMT kernel.
bool tc_contract_eligible(const VerifyArgs& a) {
    if (a.dk != kDk || a.dv % kTileV != 0) return false;
    if (a.commit.path != nullptr && a.commit.Lmax > kMaxTcPath) return false;
    return encode_fn() != nullptr;
}

template <bool kSplit>
cudaError_t launch_tree_tc_impl(const VerifyArgs& a, cudaStream_t s) {
    static bool attr_p[64], attr_c[64];
    CUtensorMap tq, tk, tql, tkl;
    const void* qh = kSplit ? a.split[0] : a.q;
    const void* kh = kSplit ? a.split[1] : a.k;
    if (!make_qk_map(&tq, qh, a.B, a.N, a.H) || !make_qk_map(&tk, kh, a.B, a.N, a.H)) return cudaErrorInvalidValue;
    if (kSplit) {
        if (!make_qk_map(&tql, a.split[2], a.B, a.N, a.H) || !make_qk_map(&tkl, a.split[3], a.B, a.N, a.H))
            return cudaErrorInvalidValue;
    } else {
        tql = tq;
        tkl = tk;
    }
    const PrepTcLayout Lp(a.N, kSplit);
    cudaError_t e = ensure_smem(tree_prep_tc_kernel<kSplit>, Lp.total, attr_p);
    if (e != cudaSuccess) return e;
    e = launch_kernel(tree_prep_tc_kernel<kSplit>, dim3(a.B * a.H), dim3(kPrepThreads), Lp.total, s, a.overlap, tq, tk,
                      tql, tkl, a);
    if (e != cudaSuccess) return e;
    const TcLayout Ly(a.commit.path ? a.commit.Lmax : 0, kSplit);
    e = ensure_smem(tree_contract_tc_kernel<kSplit>, Ly.total, attr_c);
    if (e != cudaSuccess) return e;
    dim3 grid(a.B * a.H, a.dv / kTileV);
    // always a programmatic dependent of the prologue kernel launched just before it
    return launch_kernel(tree_contract_tc_kernel<kSplit>, grid, dim3(kThreads), Ly.total, s, true, tq, tk, tql, tkl,
                         a);
}

// The contraction kernel alone (kSplit: fp32 q/k as bf16 hi/lo terms in a.split),
// after a prologue of the caller's that has written the workspace records.  It
// issues its q/k copies before its programmatic wait, so `programmatic` may be
// true only when the q/k terms were written two or more launches earlier.
cudaError_t launch_tc_contract_only(const VerifyArgs& a, bool programmatic, cudaStream_t s) {
    static bool attr_c[64];
    CUtensorMap tq, tk, tql, tkl;
    if (!make_qk_map(&tq, a.split[0], a.B, a.N, a.H) || !make_qk_map(&tk, a.split[1], a.B, a.N, a.H) ||
        !make_qk_map(&tql, a.split[2], a.B, a.N, a.H) || !make_qk_map(&tkl, a.split[3], a.B, a.N, a.H))
        return cudaErrorInvalidValue;
    const TcLayout Ly(a.commit.path ? a.commit.Lmax : 0, true);
    cudaError_t e = ensure_smem(tree_contract_tc_kernel<true>, Ly.total, attr_c);
    if (e != cudaSuccess) return e;
    return launch_kernel(tree_contract_tc_kernel<true>, dim3(a.B * a.H, a.dv / kTileV), dim3(kThreads), Ly.total,
                         s, programmatic, tq, tk, tql, tkl, a);
}

// d_v = 256 with the layout within the shared-memory limit: the single-kernel path.
bool fused_eligible(const VerifyArgs& a, bool split) {
    if (a.dk != kDk || a.dv != kFRows || a.N > kMaxNodes) return false;
    const FusedLayout L(a.N, a.commit.path ? a.commit.Lmax : 0, split);
    return L.total <= kFSmemLimit;
}

bool tc_uses_workspace(const VerifyArgs& a) { return !fused_eligible(a, a.split[0] != nullptr); }

template <bool kSplit, int kT>
cudaError_t launch_tree_fused_impl(const VerifyArgs& a, cudaStream_t s, int npairs = -1, bool programmatic = false) {
    static bool attr[64];
    CUtensorMap tq, tk, tql, tkl;
    const void* qh = kSplit ? a.split[0] : a.q;
    const void* kh = kSplit ? a.split[1] : a.k;
    if (!make_qk_map(&tq, qh, a.B, a.N, a.H) || !make_qk_map(&tk, kh, a.B, a.N, a.H)) return cudaErrorInvalidValue;
    if (kSplit) {
        if (!make_qk_map(&tql, a.split[2], a.B, a.N, a.H) || !make_qk_map(&tkl, a.split[3], a.B, a.N, a.H))
            return cudaErrorInvalidValue;
    } else {
        tql = tq;
        tkl = tk;
    }
    const FusedLayout L(a.N, a.commit.path ? a.commit.Lmax : 0, kSplit);
    cudaError_t e = ensure_smem(tree_fused_tc_kernel<kSplit, kT>, L.total, attr);
    if (e != cudaSuccess) return e;
    const int n = npairs < 0 ? a.B * a.H : npairs;
    return launch_kernel(tree_fused_tc_kernel<kSplit, kT>, dim3(n, 2 / kT), dim3(kFThreads), L.total, s,
                         a.overlap || programmatic, tq, tk, tql, tkl, a);
}

// bf16 q/k (or fp32 q/k with their bf16 hi/lo terms in `split`) with the
// tensor-core kernels: one fused kernel for d_v = 256, otherwise the prologue
// and the contraction kernel.  See launch_tree_verify.
cudaError_t launch_tree_tc(const VerifyArgs& a, cudaStream_t s) {
    const bool split = a.split[0] != nullptr;
    if (fused_eligible(a, split)) {
        // one 128-row tile per CTA while two CTAs per (sequence, head) fit in one wave of SMs
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cudaErrorInvalidValue;
        const long long pairs = (long long)a.B * a.H;
        if (2 * pairs <= sms)
            return split ? launch_tree_fused_impl<true, 1>(a, s) : launch_tree_fused_impl<false, 1>(a, s);
        // Whole waves of one CTA per pair, then -- when the rest fit one wave as two CTAs per
        // pair -- the rest as a second launch of half-tile CTAs, a programmatic dependent of the
        // first: it covers other pairs, and what it touches before its wait (its pairs' state and
        // the previous factors) the first launch does not.  The last wave then holds shorter CTAs
        // than a partial wave of whole-pair ones.
        const long long full = pairs / sms * sms, rest = pairs - full;
        if (rest == 0 || 2 * rest > sms)
            return split ? launch_tree_fused_impl<true, 2>(a, s) : launch_tree_fused_impl<false, 2>(a, s);
        cudaError_t e = split ? launch_tree_fused_impl<true, 2>(a, s, (int)full)
                              : launch_tree_fused_impl<false, 2>(a, s, (int)full);
        if (e != cudaSuccess) return e;
        VerifyArgs r = a;
        r.bh_base = (int)full;
        return split ? launch_tree_fused_impl<true, 1>(r, s, (int)rest, true)
                     : launch_tree_fused_impl<false, 1>(r, s, (int)rest, true);
    }
    return split ? launch_tree_tc_impl<true>(a, s) : launch_tree_tc_impl<false>(a, s);
}

}  // namespace gdn
