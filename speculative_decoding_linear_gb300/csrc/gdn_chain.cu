// gdn_chain.cu -- chain verification with the state resident on chip.
//
// Review of SpecLA (pith.science 7ERME3HB), "What carries the argument": a
// serial chain with the state split into tiles along d_v.  For a chain draft
// (node t hangs under t-1) every row of S evolves independently:
//
//     s = S_row . k_t,  u = S_row . q_t            (one pass over the row)
//     delta_t = beta_t (v_t[row] - alpha_t s)
//     o_t[row] = S_t,row . q_t = alpha_t u + delta_t (k_t . q_t)
//     S_row <- alpha_t S_row + delta_t k_t^T
//
// so the state is tiled along d_v: one CTA holds kRows rows of one (sequence,
// head) state in registers (each warp owns RPW rows, each lane d_k/32
// interleaved columns) and runs the N tokens serially without ever writing an
// intermediate state.
//
// Order of work inside a CTA:
//   1. state rows -> registers and the pending commit's factor rows -> smem;
//   2. the commit, applied in registers (1 and 2 only read memory, so with
//      launch overlap enabled they may run while the previous kernel on the
//      stream finishes);
//   3. griddep_wait; committed rows written back once; this layer's
//      q/k/v/alpha/beta staged with cp.async;
//   4. the serial chain; outputs and the factor record.
#include "gdn_internal.cuh"
#include "gdn_tc_ptx.cuh"

namespace gdn {
namespace {

constexpr int kWarps = 4;
constexpr int kEPL = kMaxDim / 32;   // state columns per lane

template <int RPW>
struct ChainGeom {
    static constexpr int kRows = kWarps * RPW;
};

// dynamic smem layout (byte offsets), all 16-byte aligned
struct ChainSmem {
    int qk, key, v, gate, o, d, cd, coef, nodes, misc, total;
    __host__ __device__ ChainSmem(int N, int dk, int Lcap, int rows, int esz) {
        int off = 0;
        auto take = [&](int bytes) { int o = off; off += (bytes + 15) / 16 * 16; return o; };
        qk = take(N * 2 * dk * esz);     // [t][k | q][dk], input element type
        key = take(Lcap * dk * esz);     // commit path keys
        v = take(N * rows * esz);        // [t][row]
        gate = take(N * 16);             // [t][alpha, beta, k_t . q_t, -]
        o = take(N * rows * 4);
        d = take(N * rows * 4);
        cd = take(Lcap * rows * 4);      // e^{g_a - g_j} delta_j[row]
        coef = take(kMaxPath * 4);
        nodes = take(kMaxPath * 4);
        misc = take(16);                 // ega, L
        total = off;
    }
};

// Reduce-scatter over the warp: M values per lane (M a power of two, <= 32) are
// summed over all 32 lanes; lane l returns the total of value l / (32 / M).  Each
// halving step sends half of the remaining values to the partner lane, so the M
// sums take M - 1 + log2(32 / M) shuffles instead of 5 M.
template <int M>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[M], int lane) {
    int s = 16;
#pragma unroll
    for (int m = M; m > 1; m >>= 1, s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < m / 2; ++i) {
            const float keep = up ? v[m / 2 + i] : v[i];
            const float send = up ? v[i] : v[m / 2 + i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    float x = v[0];
#pragma unroll
    for (; s > 0; s >>= 1) x += __shfl_xor_sync(0xffffffffu, x, s);
    return x;
}

template <typename T, int RPW>
__global__ void __launch_bounds__(kWarps * 32) chain_kernel(VerifyArgs a) {
    constexpr int kRows = ChainGeom<RPW>::kRows;
    extern __shared__ __align__(16) unsigned char smem[];
    const int Lcap = a.commit.path ? a.commit.Lmax : 0;
    const ChainSmem L(a.N, a.dk, Lcap, kRows, (int)sizeof(T));
    T* s_qk = reinterpret_cast<T*>(smem + L.qk);
    T* s_key = reinterpret_cast<T*>(smem + L.key);
    T* s_v = reinterpret_cast<T*>(smem + L.v);
    float* s_gate = reinterpret_cast<float*>(smem + L.gate);
    float* s_o = reinterpret_cast<float*>(smem + L.o);
    float* s_d = reinterpret_cast<float*>(smem + L.d);
    float* s_cd = reinterpret_cast<float*>(smem + L.cd);
    float* s_coef = reinterpret_cast<float*>(smem + L.coef);
    int* s_nodes = reinterpret_cast<int*>(smem + L.nodes);
    float* s_ega = reinterpret_cast<float*>(smem + L.misc);
    int* s_L = reinterpret_cast<int*>(smem + L.misc + 4);

    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int N = a.N, dk = a.dk, dv = a.dv, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int v0 = blockIdx.y * kRows;
    const int rows = min(kRows, dv - v0);
    const bool fused = a.commit.path != nullptr;
    __shared__ __align__(8) uint64_t s_bar;    // this layer's q/k rows: one bulk copy per row
    const uint32_t bar = smem_u32(&s_bar);
    if (tid == 0) {
        tc::mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    // 1. state rows -> registers (loads in flight while the commit is set up).  Lane
    // `lane` holds columns c0 .. c0+7 of each of its warp's rows, c0 = 8 lane (all
    // of them or none: d_k is a multiple of 16), so every access is a vector access.
    const int c0 = 8 * lane;
    const bool lane_on = c0 < dk;
    float S[RPW][kEPL];
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
        const int r = warp * RPW + rr;
        if (r < rows && lane_on) {
            ld8<float>(a.S + ((size_t)bh * dv + v0 + r) * dk + c0, S[rr]);
        } else {
#pragma unroll
            for (int e = 0; e < kEPL; ++e) S[rr][e] = 0.f;
        }
    }
    int nL = 0;
    if (fused) {
        if (warp == 0) {
            const int Lp = commit_path_setup(a.commit, b, h, a.H, s_nodes, s_coef, s_ega);
            if (lane == 0) {
                *s_L = Lp;
                if (Lp < 0) set_error(a.err, GDN_ERR_PATH);
            }
        }
        __syncthreads();
        nL = *s_L;
        if (nL < 0) return;
        const float* dl = a.commit.delta + (size_t)bh * a.commit.N * dv;
        const T* key_bh = static_cast<const T*>(a.commit.key) + (size_t)bh * a.commit.N * dk;
#pragma unroll 1
        for (int i = 0; i < nL; ++i)
            cp_async_block(s_key + (size_t)i * dk, key_bh + (size_t)s_nodes[i] * dk, dk * (int)sizeof(T),
                           tid, kWarps * 32);
#pragma unroll 1
        for (int i = tid; i < nL * kRows; i += kWarps * 32) {
            const int j = i / kRows, r = i % kRows;
            s_cd[i] = r < rows ? s_coef[j] * dl[(size_t)s_nodes[j] * dv + v0 + r] : 0.f;
        }
        cp_async_wait_all();
        __syncthreads();
        // 2. commit in registers (same arithmetic order as gdn_commit)
        const float ega = *s_ega;
        if (lane_on) {
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
                for (int e = 0; e < kEPL; ++e) S[rr][e] *= ega;
#pragma unroll 1
            for (int i = 0; i < nL; ++i) {
                float kv[kEPL];
                ld8<T>(s_key + (size_t)i * dk + c0, kv);
#pragma unroll
                for (int rr = 0; rr < RPW; ++rr) {
                    const float w = s_cd[i * kRows + warp * RPW + rr];
#pragma unroll
                    for (int e = 0; e < kEPL; ++e) S[rr][e] = fmaf(w, kv[e], S[rr][e]);
                }
            }
        }
    }

    // This layer's q/k/v rows into L2 while the previous kernel finishes (the
    // CTAs of one (sequence, head) split the tokens between them).
    if (tid == 0) {
        const int rowq = dk * (int)sizeof(T), rowv = dv * (int)sizeof(T);
#pragma unroll 1
        for (int t = blockIdx.y; t < N; t += gridDim.y) {
            const size_t rt = ((size_t)b * N + t) * a.H + h;
            prefetch_l2(static_cast<const T*>(a.q) + rt * dk, rowq);
            prefetch_l2(static_cast<const T*>(a.k) + rt * dk, rowq);
            prefetch_l2(static_cast<const T*>(a.v) + rt * dv, rowv);
        }
    }
    if (tid < N) {
        const size_t gi = ((size_t)b * N + tid) * a.H + h;
        prefetch_line_l2(a.alpha + gi);
        prefetch_line_l2(a.beta + gi);
    }

    // Everything above only read memory.  Writes and this layer's inputs come
    // after the programmatic wait.
    griddep_wait();
    griddep_launch();
    // 3. this layer's draft inputs: v, alpha, beta loads issued first (one item per
    // thread when N * kRows <= 128), then the q/k row copies (one token per lane of
    // warp 0), then the committed rows' stores, then the values into shared memory
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* vv = static_cast<const T*>(a.v);
    const int rowb = dk * (int)sizeof(T);
    const bool one_pass = N * kRows <= kWarps * 32;
    float v_reg = 0.f, al_reg = 0.f, be_reg = 0.f;
    if (one_pass) {
        if (tid < N * kRows && tid % kRows < rows)
            v_reg = ld_elem<T>(vv, (((size_t)b * N + tid / kRows) * a.H + h) * dv + v0 + tid % kRows);
        if (tid < N) {
            const size_t gi = ((size_t)b * N + tid) * a.H + h;
            al_reg = a.alpha[gi];
            be_reg = a.beta[gi];
        }
    }
    if (warp == 0) {
        if (lane == 0) tc::mbar_expect_tx(bar, (uint32_t)(2 * N * rowb));
        __syncwarp();
#pragma unroll 1
        for (int t = lane; t < N; t += 32) {
            const size_t rt = (((size_t)b * N + t) * a.H + h) * dk;
            tc::bulk_copy_g2s(smem_u32(s_qk + (size_t)(2 * t) * dk), k + rt, rowb, bar);
            tc::bulk_copy_g2s(smem_u32(s_qk + (size_t)(2 * t + 1) * dk), q + rt, rowb, bar);
        }
    }
    if (fused) {    // committed rows written back once
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            const int r = warp * RPW + rr;
            if (r < rows && lane_on) {
                float4* row = reinterpret_cast<float4*>(a.S + ((size_t)bh * dv + v0 + r) * dk + c0);
                row[0] = make_float4(S[rr][0], S[rr][1], S[rr][2], S[rr][3]);
                row[1] = make_float4(S[rr][4], S[rr][5], S[rr][6], S[rr][7]);
            }
        }
    }
    if (one_pass) {
        if (tid < N * kRows) s_v[tid] = v_reg;
        if (tid < N) {
            s_gate[4 * tid] = al_reg;
            s_gate[4 * tid + 1] = be_reg;
        }
    } else {
#pragma unroll 1
        for (int i = tid; i < N * kRows; i += kWarps * 32) {
            const int t = i / kRows, r = i % kRows;
            s_v[i] = r < rows ? ld_elem<T>(vv, (((size_t)b * N + t) * a.H + h) * dv + v0 + r) : 0.f;
        }
#pragma unroll 1
        for (int t = tid; t < N; t += kWarps * 32) {
            const size_t gi = ((size_t)b * N + t) * a.H + h;
            s_gate[4 * t] = a.alpha[gi];
            s_gate[4 * t + 1] = a.beta[gi];
        }
    }

    const bool landed = tc::mbar_wait(bar, 0, a.err);
    // k_t . q_t rides along in the token loop's reduction (below) when the 2 RPW
    // row sums leave room in a power-of-two value count; otherwise every token's is
    // formed here (the warps take turns)
    constexpr bool kFoldKq = RPW == 2 || RPW == 4;
    if (!kFoldKq && __all_sync(0xffffffffu, landed)) {
#pragma unroll 1
        for (int t = warp; t < N; t += kWarps) {
            float kt[kEPL], qt[kEPL];
            float kq = 0.f;
            if (lane_on) {
                ld8<T>(s_qk + (size_t)(2 * t) * dk + c0, kt);
                ld8<T>(s_qk + (size_t)(2 * t + 1) * dk + c0, qt);
#pragma unroll
                for (int e = 0; e < kEPL; ++e) kq = fmaf(kt[e], qt[e], kq);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
            if (lane == 0) s_gate[4 * t + 2] = kq;
        }
    }
    if (!__syncthreads_and(landed)) return;    // a bounded wait ran out (recorded in the error word)

    // 4. serial chain.  Per token the warp sums 2 RPW dot products (S_row . k_t and
    // S_row . q_t of its RPW rows) and k_t . q_t with one
    // reduce-scatter butterfly; afterwards lane l holds value l / kGroup.  The lanes
    // holding S_row . k_t form delta_t of their row and broadcast it; the lanes
    // holding S_row . q_t form o_t.  Unrolled by 2
    // so that the next tokens' shared-memory loads are issued ahead.
    constexpr int kVals = kFoldKq ? 4 * RPW : 2 * RPW;
    constexpr int kGroup = 32 / kVals;
    const int held = lane / kGroup;                 // value index held after the reduction
    const int rr_held = held % RPW;
    const int r_held = warp * RPW + rr_held;        // its state row
    const bool holds_q = held >= RPW && held < 2 * RPW && lane % kGroup == 0 && r_held < rows;
#pragma unroll 2
    for (int t = 0; t < N; ++t) {
        float kt[kEPL], qt[kEPL];
        if (lane_on) {
            ld8<T>(s_qk + (size_t)(2 * t) * dk + c0, kt);
            ld8<T>(s_qk + (size_t)(2 * t + 1) * dk + c0, qt);
        } else {
#pragma unroll
            for (int e = 0; e < kEPL; ++e) kt[e] = qt[e] = 0.f;
        }
        float val[kVals];
#pragma unroll
        for (int i = 2 * RPW; i < kVals; ++i) val[i] = 0.f;
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
            float x = 0.f, y = 0.f;
#pragma unroll
            for (int e = 0; e < kEPL; ++e) {
                x = fmaf(S[rr][e], kt[e], x);
                y = fmaf(S[rr][e], qt[e], y);
            }
            val[rr] = x;
            val[RPW + rr] = y;
        }
        if (kFoldKq) {
#pragma unroll
            for (int e = 0; e < kEPL; ++e) val[2 * RPW] = fmaf(kt[e], qt[e], val[2 * RPW]);
        }
        const float tot = warp_reduce_scatter<kVals>(val, lane);
        const float4 gt = *reinterpret_cast<const float4*>(s_gate + 4 * t);   // alpha, beta, k.q
        const float al = gt.x, be = gt.y;
        const float kq = kFoldKq ? __shfl_sync(0xffffffffu, tot, 2 * RPW * kGroup) : gt.z;
        const float vt = r_held < rows ? ld_elem<T>(s_v, (size_t)t * kRows + r_held) : 0.f;
        const float dl = be * (a.linear ? vt : vt - al * tot);             // meaningful where held < RPW
        float dlt[RPW];
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) dlt[rr] = __shfl_sync(0xffffffffu, dl, rr * kGroup);
        if (holds_q) {
            float d = dlt[0];
#pragma unroll
            for (int rr = 1; rr < RPW; ++rr)
                if (rr_held == rr) d = dlt[rr];
            s_o[t * kRows + r_held] = fmaf(al, tot, d * kq);
            s_d[t * kRows + r_held] = d;
        }
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
            for (int e = 0; e < kEPL; ++e) S[rr][e] = fmaf(al, S[rr][e], dlt[rr] * kt[e]);
    }
    __syncthreads();

    // outputs and factors (coalesced along d_v)
#pragma unroll 1
    for (int i = tid; i < N * kRows; i += kWarps * 32) {
        const int t = i / kRows, r = i % kRows;
        if (r >= rows) continue;
        a.out[(((size_t)b * N + t) * a.H + h) * dv + v0 + r] = s_o[i];
        a.f.delta[((size_t)bh * N + t) * dv + v0 + r] = s_d[i];
    }
    // key copy (from smem), gates and parents: spread over the CTAs of this (b, h)
    T* key_out = static_cast<T*>(a.f.key);
    const int vecs = rowb / 16;
#pragma unroll 1
    for (int t = blockIdx.y; t < N; t += gridDim.y) {
        const uint4* src = reinterpret_cast<const uint4*>(s_qk + (size_t)(2 * t) * dk);
        uint4* dst = reinterpret_cast<uint4*>(key_out + ((size_t)bh * N + t) * dk);
#pragma unroll 1
        for (int i = tid; i < vecs; i += kWarps * 32) dst[i] = src[i];
    }
    if (blockIdx.y == 0 && warp == 0) {
        // g_t = sum_{i <= t} log alpha_i : warp scan over chunks of 32 nodes
        float carry = 0.f;
#pragma unroll 1
        for (int t0 = 0; t0 < N; t0 += 32) {
            const int t = t0 + lane;
            float x = t < N ? logf(s_gate[4 * t]) : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            x += carry;
            if (t < N) {
                a.f.g[(size_t)bh * N + t] = x;
                if (h == 0) a.f.parent[(size_t)b * N + t] = t - 1;
            }
            carry = __shfl_sync(0xffffffffu, x, 31);
        }
    }
}

template <typename T, int RPW>
cudaError_t launch_chain_t(const VerifyArgs& a, cudaStream_t s) {
    static bool attr[64];
    constexpr int kRows = ChainGeom<RPW>::kRows;
    const ChainSmem L(a.N, a.dk, a.commit.path ? a.commit.Lmax : 0, kRows, (int)sizeof(T));
    cudaError_t e = ensure_smem(chain_kernel<T, RPW>, L.total, attr);
    if (e != cudaSuccess) return e;
    dim3 grid(a.B * a.H, (a.dv + kRows - 1) / kRows);
    return launch_kernel(chain_kernel<T, RPW>, grid, dim3(kWarps * 32), L.total, s, a.overlap, a);
}

// ---------------------------------------------------------------------------
// d_k = 256: eight lanes per state row
// ---------------------------------------------------------------------------
// The per-token step above is bound by its five-level butterfly with one warp
// per SM sub-partition.  With d_k = 256 a row can be spread over 8 lanes (32
// contiguous columns each) instead: a warp holds 4 rows, a CTA 16, and a token
// costs a three-level butterfly after which every lane of the row's group holds
// S_row . k_t, S_row . q_t and k_t . q_t, so delta_t needs no broadcast.  A
// lane's 32 columns are interleaved with its group's (4 at a time) so that the
// shared-memory reads of a group cover contiguous bytes; the four row groups of
// a warp read the same k/q words (broadcast), widened to fp32 in registers.
// Packed fp32 pairs: ffma2 / fmul2 (gdn_internal.cuh).

constexpr int kG8Rows = 16;            // state rows per CTA
constexpr int kG8Cols = 32;            // state columns per lane (8 groups of 4)

struct G8Smem {
    int qk, key, v, gate, o, d, cd, coef, nodes, misc, total;
    __host__ __device__ G8Smem(int N, int Lcap, int esz) {
        int off = 0;
        auto take = [&](int bytes) { int o = off; off += (bytes + 15) / 16 * 16; return o; };
        qk = take(N * 2 * kMaxDim * esz);                  // rows as copied: [t][k | q][256]
        key = take(Lcap * kMaxDim * esz);
        v = take(N * kG8Rows * esz);
        gate = take(N * 16);                               // [t][alpha, beta, -, -]
        o = take(N * kG8Rows * 4);
        d = take(N * kG8Rows * 4);
        cd = take(Lcap * kG8Rows * 4);
        coef = take(kMaxPath * 4);
        nodes = take(kMaxPath * 4);
        misc = take(16);
        total = off;
    }
};

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) chain_g8_kernel(VerifyArgs a) {
    constexpr int kRows = kG8Rows;
    extern __shared__ __align__(16) unsigned char smem[];
    const int Lcap = a.commit.path ? a.commit.Lmax : 0;
    const G8Smem L(a.N, Lcap, (int)sizeof(T));
    T* s_qk = reinterpret_cast<T*>(smem + L.qk);
    T* s_key = reinterpret_cast<T*>(smem + L.key);
    T* s_v = reinterpret_cast<T*>(smem + L.v);
    float* s_gate = reinterpret_cast<float*>(smem + L.gate);
    float* s_o = reinterpret_cast<float*>(smem + L.o);
    float* s_d = reinterpret_cast<float*>(smem + L.d);
    float* s_cd = reinterpret_cast<float*>(smem + L.cd);
    float* s_coef = reinterpret_cast<float*>(smem + L.coef);
    int* s_nodes = reinterpret_cast<int*>(smem + L.nodes);
    float* s_ega = reinterpret_cast<float*>(smem + L.misc);
    int* s_L = reinterpret_cast<int*>(smem + L.misc + 4);

    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int N = a.N, dv = a.dv, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int r = warp * 4 + (lane >> 3);      // this lane's state row within the CTA
    // Columns 32 m + cb + u (m = 0..7, u = 0..3), cb = 4 (lane & 7): the row's 8 lanes
    // read 128 contiguous bytes per 16-byte load (no bank conflicts); S[4 m + u].
    const int cb = 4 * (lane & 7);
    const int v0 = blockIdx.y * kRows;
    const int rows = min(kRows, dv - v0);
    const bool row_on = r < rows;
    const bool fused = a.commit.path != nullptr;
    __shared__ __align__(8) uint64_t s_bar;
    const uint32_t bar = smem_u32(&s_bar);
    if (tid == 0) {
        tc::mbar_init(bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    // 1. this lane's 32 columns of its state row
    float2 S[kG8Cols / 2];                     // column pairs, for the packed fp32 arithmetic
    const float* srow = a.S + ((size_t)bh * dv + v0 + r) * kMaxDim + cb;
#pragma unroll
    for (int e = 0; e < kG8Cols; e += 4) {
        const float4 x = row_on ? *reinterpret_cast<const float4*>(srow + 8 * e) : make_float4(0.f, 0.f, 0.f, 0.f);
        S[e / 2] = make_float2(x.x, x.y);
        S[e / 2 + 1] = make_float2(x.z, x.w);
    }
    if (fused) {
        if (warp == 0) {
            const int Lp = commit_path_setup(a.commit, b, h, a.H, s_nodes, s_coef, s_ega);
            if (lane == 0) {
                *s_L = Lp;
                if (Lp < 0) set_error(a.err, GDN_ERR_PATH);
            }
        }
        __syncthreads();
        const int nL = *s_L;
        if (nL < 0) return;
        const float* dl = a.commit.delta + (size_t)bh * a.commit.N * dv;
        const T* key_bh = static_cast<const T*>(a.commit.key) + (size_t)bh * a.commit.N * kMaxDim;
#pragma unroll 1
        for (int i = 0; i < nL; ++i)
            cp_async_block(s_key + (size_t)i * kMaxDim, key_bh + (size_t)s_nodes[i] * kMaxDim,
                           kMaxDim * (int)sizeof(T), tid, kWarps * 32);
#pragma unroll 1
        for (int i = tid; i < nL * kRows; i += kWarps * 32) {
            const int j = i / kRows, rr = i % kRows;
            s_cd[i] = rr < rows ? s_coef[j] * dl[(size_t)s_nodes[j] * dv + v0 + rr] : 0.f;
        }
        cp_async_wait_all();
        __syncthreads();
        // 2. commit in registers (same arithmetic order as gdn_commit)
        const float ega = *s_ega;
        const float2 ega2 = make_float2(ega, ega);
#pragma unroll
        for (int i = 0; i < kG8Cols / 2; ++i) S[i] = fmul2(S[i], ega2);
#pragma unroll 1
        for (int i = 0; i < nL; ++i) {
            const float w = s_cd[i * kRows + r];
            const float2 w2 = make_float2(w, w);
#pragma unroll
            for (int e = 0; e < kG8Cols; e += 4) {
                const float4 kv = ld4<T>(s_key, (size_t)i * kMaxDim + cb + 8 * e);
                S[e / 2] = ffma2(w2, make_float2(kv.x, kv.y), S[e / 2]);
                S[e / 2 + 1] = ffma2(w2, make_float2(kv.z, kv.w), S[e / 2 + 1]);
            }
        }
    }

    // This layer's q/k/v rows and gates into L2 while the previous kernel finishes.
    if (tid == 0) {
        const int rowq = kMaxDim * (int)sizeof(T), rowv = dv * (int)sizeof(T);
#pragma unroll 1
        for (int t = blockIdx.y; t < N; t += gridDim.y) {
            const size_t rt = ((size_t)b * N + t) * a.H + h;
            prefetch_l2(static_cast<const T*>(a.q) + rt * kMaxDim, rowq);
            prefetch_l2(static_cast<const T*>(a.k) + rt * kMaxDim, rowq);
            prefetch_l2(static_cast<const T*>(a.v) + rt * dv, rowv);
        }
    }
    if (tid < N) {
        const size_t gi = ((size_t)b * N + tid) * a.H + h;
        prefetch_line_l2(a.alpha + gi);
        prefetch_line_l2(a.beta + gi);
    }

    // Everything above only read memory.
    griddep_wait();
    griddep_launch();
    // 3. this layer's draft inputs (as in chain_kernel)
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* vv = static_cast<const T*>(a.v);
    const int rowb = kMaxDim * (int)sizeof(T);
    const bool one_pass = N * kRows <= kWarps * 32;
    float v_reg = 0.f, al_reg = 0.f, be_reg = 0.f;
    if (one_pass) {
        if (tid < N * kRows && tid % kRows < rows)
            v_reg = ld_elem<T>(vv, (((size_t)b * N + tid / kRows) * a.H + h) * dv + v0 + tid % kRows);
        if (tid < N) {
            const size_t gi = ((size_t)b * N + tid) * a.H + h;
            al_reg = a.alpha[gi];
            be_reg = a.beta[gi];
        }
    }
    if (warp == 0) {
        if (lane == 0) tc::mbar_expect_tx(bar, (uint32_t)(2 * N * rowb));
        __syncwarp();
#pragma unroll 1
        for (int t = lane; t < N; t += 32) {
            const size_t rt = (((size_t)b * N + t) * a.H + h) * kMaxDim;
            tc::bulk_copy_g2s(smem_u32(s_qk + (size_t)(2 * t) * kMaxDim), k + rt, rowb, bar);
            tc::bulk_copy_g2s(smem_u32(s_qk + (size_t)(2 * t + 1) * kMaxDim), q + rt, rowb, bar);
        }
    }
    if (fused && row_on) {    // committed row part written back once
        float* wrow = a.S + ((size_t)bh * dv + v0 + r) * kMaxDim + cb;
#pragma unroll
        for (int e = 0; e < kG8Cols; e += 4)
            *reinterpret_cast<float4*>(wrow + 8 * e) = make_float4(S[e / 2].x, S[e / 2].y, S[e / 2 + 1].x, S[e / 2 + 1].y);
    }
    if (one_pass) {
        if (tid < N * kRows) st_elem<T>(s_v, tid, v_reg);
        if (tid < N) {
            s_gate[4 * tid] = al_reg;
            s_gate[4 * tid + 1] = be_reg;
        }
    } else {
#pragma unroll 1
        for (int i = tid; i < N * kRows; i += kWarps * 32) {
            const int t = i / kRows, rr = i % kRows;
            st_elem<T>(s_v, i, rr < rows ? ld_elem<T>(vv, (((size_t)b * N + t) * a.H + h) * dv + v0 + rr) : 0.f);
        }
#pragma unroll 1
        for (int t = tid; t < N; t += kWarps * 32) {
            const size_t gi = ((size_t)b * N + t) * a.H + h;
            s_gate[4 * t] = a.alpha[gi];
            s_gate[4 * t + 1] = a.beta[gi];
        }
    }
    const bool landed = tc::mbar_wait(bar, 0, a.err);
    if (!__syncthreads_and(landed)) return;    // a bounded wait ran out (recorded in the error word)

    // 4. serial chain: per token three partial-sum dot products over the lane's 32
    // columns, a three-level butterfly over the row's 8 lanes, the update
#pragma unroll 2
    for (int t = 0; t < N; ++t) {
        const T* kr = s_qk + (size_t)(2 * t) * kMaxDim + cb;
        const T* qr = kr + kMaxDim;
        float2 kt[kG8Cols / 2];
        float2 xa = make_float2(0.f, 0.f), xb = xa, ya = xa, yb = xa, za = xa, zb = xa;
#pragma unroll
        for (int e = 0; e < kG8Cols; e += 4) {
            const float4 kv = ld4<T>(kr, 8 * e);
            const float4 qv = ld4<T>(qr, 8 * e);
            const float2 k01 = make_float2(kv.x, kv.y), k23 = make_float2(kv.z, kv.w);
            const float2 q01 = make_float2(qv.x, qv.y), q23 = make_float2(qv.z, qv.w);
            kt[e / 2] = k01;
            kt[e / 2 + 1] = k23;
            xa = ffma2(S[e / 2], k01, xa);
            xb = ffma2(S[e / 2 + 1], k23, xb);
            ya = ffma2(S[e / 2], q01, ya);
            yb = ffma2(S[e / 2 + 1], q23, yb);
            za = ffma2(k01, q01, za);
            zb = ffma2(k23, q23, zb);
        }
        float sk = (xa.x + xa.y) + (xb.x + xb.y);
        float sq = (ya.x + ya.y) + (yb.x + yb.y);
        float kq = (za.x + za.y) + (zb.x + zb.y);
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            sk += __shfl_xor_sync(0xffffffffu, sk, o);
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
            kq += __shfl_xor_sync(0xffffffffu, kq, o);
        }
        const float2 gt = *reinterpret_cast<const float2*>(s_gate + 4 * t);   // alpha, beta
        const float al = gt.x, be = gt.y;
        const float vt = row_on ? ld_elem<T>(s_v, (size_t)t * kRows + r) : 0.f;
        const float dlt = be * (a.linear ? vt : vt - al * sk);
        if ((lane & 7) == 0 && row_on) {
            s_o[t * kRows + r] = fmaf(al, sq, dlt * kq);
            s_d[t * kRows + r] = dlt;
        }
        const float2 al2 = make_float2(al, al), dlt2 = make_float2(dlt, dlt);
#pragma unroll
        for (int i = 0; i < kG8Cols / 2; ++i) S[i] = ffma2(al2, S[i], fmul2(dlt2, kt[i]));
    }
    __syncthreads();

    // outputs and factors (coalesced along d_v)
#pragma unroll 1
    for (int i = tid; i < N * kRows; i += kWarps * 32) {
        const int t = i / kRows, rr = i % kRows;
        if (rr >= rows) continue;
        a.out[(((size_t)b * N + t) * a.H + h) * dv + v0 + rr] = s_o[i];
        a.f.delta[((size_t)bh * N + t) * dv + v0 + rr] = s_d[i];
    }
    // key copy (the rows as copied), gates and parents: spread over the CTAs of this (b, h)
    T* key_out = static_cast<T*>(a.f.key);
    const int vecs = rowb / 16;
#pragma unroll 1
    for (int t = blockIdx.y; t < N; t += gridDim.y) {
        const uint4* src = reinterpret_cast<const uint4*>(s_qk + (size_t)(2 * t) * kMaxDim);
        uint4* dst = reinterpret_cast<uint4*>(key_out + ((size_t)bh * N + t) * kMaxDim);
#pragma unroll 1
        for (int i = tid; i < vecs; i += kWarps * 32) dst[i] = src[i];
    }
    if (blockIdx.y == 0 && warp == 0) {
        float carry = 0.f;
#pragma unroll 1
        for (int t0 = 0; t0 < N; t0 += 32) {
            const int t = t0 + lane;
            float x = t < N ? logf(s_gate[4 * t]) : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            x += carry;
            if (t < N) {
                a.f.g[(size_t)bh * N + t] = x;
                if (h == 0) a.f.parent[(size_t)b * N + t] = t - 1;
            }
            carry = __shfl_sync(0xffffffffu, x, 31);
        }
    }
}

template <typename T>
cudaError_t launch_chain_g8(const VerifyArgs& a, cudaStream_t s) {
    static bool attr[64];
    const G8Smem L(a.N, a.commit.path ? a.commit.Lmax : 0, (int)sizeof(T));
    cudaError_t e = ensure_smem(chain_g8_kernel<T>, L.total, attr);
    if (e != cudaSuccess) return e;
    dim3 grid(a.B * a.H, (a.dv + kG8Rows - 1) / kG8Rows);
    return launch_kernel(chain_g8_kernel<T>, grid, dim3(kWarps * 32), L.total, s, a.overlap, a);
}

template <typename T>
cudaError_t launch_chain_dt(const VerifyArgs& a, cudaStream_t s) {
    if (a.dk == kMaxDim) return launch_chain_g8<T>(a, s);
    // Small problems: 8-row CTAs so that more SMs stream the state.
    const long long ctas16 = (long long)a.B * a.H * ((a.dv + 15) / 16);
    return ctas16 < 2 * 152 ? launch_chain_t<T, 2>(a, s) : launch_chain_t<T, 4>(a, s);
}

}  // namespace

cudaError_t launch_chain_verify(const VerifyArgs& a, int dtype, cudaStream_t s) {
    return dtype == GDN_DTYPE_F32 ? launch_chain_dt<float>(a, s) : launch_chain_dt<__nv_bfloat16>(a, s);
}

}  // namespace gdn
