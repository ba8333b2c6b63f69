// gdn_prep_common.cuh -- per-(sequence, head) steps of the tree verifier's
// prologue shared by its SIMT and tensor-core variants (review of SpecLA,
// pith.science 7ERME3HB, "Core claim": the tree mask M_tree, the masked Gram
// A_tree = M_tree (.) (K_b K_a^T) and T_tree = solve_tril(I - A_tree)).
//
// Tables live in shared memory as N x ld fp32 (ld = N + 1), and only entries
// on the inclusive ancestor mask are ever written or read:
//   A[t, j]    = beta_t e^{g_t - g_j} (k_t . k_j),  j strict ancestor of t
//   Attn[t, j] =        e^{g_t - g_j} (q_t . k_j),  j on path(t)
//   T          = (I + A)^-1 (rows by back-substitution along each node's path)
//   P          = Attn T (written over A once T is done)
#pragma once

#include "gdn_internal.cuh"

namespace gdn {
namespace prep {

// Strict-ancestor masks, depths and cumulative log gates; threads t < N.
// par, la (log alpha) must be in shared memory.  Ascending bit order walks the
// path from the root, so g_t sums log alpha root first.
__device__ __forceinline__ void node_meta(int tid, int N, const int* par, const float* la, uint64_t* anc,
                                          int* depth, float* g) {
    if (tid < N) {
        uint64_t m = 0;
        int d = 0;
        for (int j = par[tid]; j >= 0; j = par[j]) {
            m |= 1ull << j;
            ++d;
        }
        anc[tid] = m;
        depth[tid] = d;
        float gs = 0.f;
        for (uint64_t r = m; r; r &= r - 1) gs += la[__ffsll((long long)r) - 1];
        g[tid] = gs + la[tid];
    }
}

// (t, j on path(t)) pairs, t-major, j ascending: off[t] = first pair of t,
// off[N] = count.  Call with every thread; contains block barriers.
__device__ __forceinline__ void pair_list(int tid, int N, const int* depth, const uint64_t* anc, int* off,
                                          uint16_t* pairs) {
    const int warp = tid >> 5, lane = tid & 31;
    if (warp == 0) {
        int carry = 0;
        for (int t0 = 0; t0 < N; t0 += 32) {
            const int t = t0 + lane;
            int x = t < N ? depth[t] + 1 : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (t < N) off[t + 1] = carry + x;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) off[0] = 0;
    }
    __syncthreads();
    if (tid < N) {
        int o = off[tid];
        for (uint64_t r = anc[tid]; r; r &= r - 1)
            pairs[o++] = (uint16_t)((tid << 8) | (__ffsll((long long)r) - 1));
        pairs[o] = (uint16_t)((tid << 8) | tid);
    }
    __syncthreads();
}

// A and Attn entries of pair (t, j) from the raw dot products k_t.k_j and q_t.k_j.
__device__ __forceinline__ void gram_entry(int t, int j, float kk, float qk, int ld, const float* g,
                                           const float* beta, float* sA, float* sAt) {
    const float gam = expf(g[t] - g[j]);
    sAt[t * ld + j] = gam * qk;
    if (j != t) sA[t * ld + j] = beta[t] * gam * kk;
}

// Rows of T = (I + A)^-1, then P = Attn T over A.  The principal block of
// I + A on path(t) is closed (ancestors of path nodes are on the path), so
// row t of T is the last row of that block's inverse: x_t = 1 and, walking up
// the path, x_k = -sum_{i on path(t) below k} x_i A[i, k].  Then
// P[t, c] = sum_{j on path(t) at or below c} Attn[t, j] T[j, c].  One thread
// per node, no level barriers.  Call with every thread; contains barriers.
__device__ __forceinline__ void solve_rows(int tid, int N, int ld, const uint64_t* anc, float* sA,
                                           const float* sAt, float* sT) {
    if (tid < N) {
        const int t = tid;
        const uint64_t path = anc[t] | (1ull << t);
        float* row = sT + t * ld;
        row[t] = 1.f;
        for (uint64_t up = anc[t]; up;) {
            const int kk = 63 - __clzll((long long)up);          // deepest remaining ancestor
            up &= ~(1ull << kk);
            float x = 0.f;
            for (uint64_t below = path & ~((2ull << kk) - 1ull); below; below &= below - 1) {
                const int i = __ffsll((long long)below) - 1;
                x = fmaf(row[i], sA[i * ld + kk], x);
            }
            row[kk] = -x;
        }
    }
    __syncthreads();
    if (tid < N) {
        const int t = tid;
        const uint64_t path = anc[t] | (1ull << t);
        for (uint64_t cs = path; cs; cs &= cs - 1) {
            const int c = __ffsll((long long)cs) - 1;
            float x = 0.f;
            for (uint64_t js = path & ~((1ull << c) - 1ull); js; js &= js - 1) {
                const int j = __ffsll((long long)js) - 1;
                x = fmaf(sAt[t * ld + j], sT[j * ld + c], x);
            }
            sA[t * ld + c] = x;   // A is no longer read: step one finished behind the barrier
        }
    }
    __syncthreads();
}

// [T; P] as the tensor-core contraction's second MMA operand: 128 rows (T rows
// 0..63, P rows 64..127) x 64 columns, bf16 hi then lo (16 KiB each), rows of
// 128 bytes with 16-byte chunks XOR-swizzled by (row & 7); zeros off the
// ancestor mask and beyond N.
__device__ __forceinline__ void write_operand(int tid, int nthreads, int N, int ld, const uint64_t* anc,
                                              const float* sP, const float* sT, unsigned char* op) {
    for (int item = tid; item < 128 * 8; item += nthreads) {
        const int r = item >> 3, cc = item & 7;
        const int t = r & 63;
        const float* src = r >= 64 ? sP : sT;
        const uint64_t path = t < N ? (anc[t] | (1ull << t)) : 0ull;
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j0 = 8 * cc + 2 * e, j1 = j0 + 1;
            const float x0 = ((path >> j0) & 1ull) ? src[t * ld + j0] : 0.f;
            const float x1 = ((path >> j1) & 1ull) ? src[t * ld + j1] : 0.f;
            const __nv_bfloat162 hh = __floats2bfloat162_rn(x0, x1);
            const float2 hf = __bfloat1622float2(hh);
            const __nv_bfloat162 ll = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
            hi[e] = *reinterpret_cast<const uint32_t*>(&hh);
            lo[e] = *reinterpret_cast<const uint32_t*>(&ll);
        }
        const uint32_t off = (uint32_t)(r * 128 + ((cc ^ (r & 7)) << 4));
        *reinterpret_cast<uint4*>(op + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(op + kTcOperandBytes / 2 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// Dense fp32 T and P rows (zeros off the mask) for the SIMT contraction.
__device__ __forceinline__ void write_dense(int tid, int nthreads, int N, int ld, const uint64_t* anc,
                                            const float* sP, const float* sT, float* wT, float* wP) {
    for (int i = tid; i < N * N; i += nthreads) {
        const int t = i / N, c = i % N;
        const bool on = ((anc[t] | (1ull << t)) >> c) & 1ull;
        wT[i] = on ? sT[t * ld + c] : 0.f;
        wP[i] = on ? sP[t * ld + c] : 0.f;
    }
}

// e^g, beta and the inclusive masks into the workspace record; g and parents
// into the factor record.  Threads t < N.
__device__ __forceinline__ void write_meta(int tid, int N, int b, int h, int bh, char* rec, const WsLayout& wl,
                                           const float* g, const float* beta, const uint64_t* anc,
                                           const int* par, const Factors& f) {
    if (tid < N) {
        reinterpret_cast<float*>(rec + wl.eg)[tid] = expf(g[tid]);
        reinterpret_cast<float*>(rec + wl.bt)[tid] = beta[tid];
        reinterpret_cast<uint64_t*>(rec + wl.anc)[tid] = anc[tid] | (1ull << tid);
        f.g[(size_t)bh * N + tid] = g[tid];
        if (h == 0) f.parent[(size_t)b * N + tid] = par[tid];
    }
}

}  // namespace prep
}  // namespace gdn
