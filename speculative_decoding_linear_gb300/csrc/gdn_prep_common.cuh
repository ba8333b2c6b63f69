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

// Strict-ancestor masks, depths, cumulative log gates and root-first path
// lists (plist[t * 64 + i] = i-th node of path(t), i = 0..depth(t)); threads
// t < N.  par, la (log alpha) must be in shared memory.  Ascending bit order
// walks the path from the root, so g_t sums log alpha root first.
__device__ __forceinline__ void node_meta(int tid, int N, const int* par, const float* la, uint64_t* anc,
                                          int* depth, float* g, uint8_t* plist) {
    if (tid < N) {
        uint64_t m = 0;
        int d = 0;
#pragma unroll 1
        for (int j = par[tid]; j >= 0; j = par[j]) {
            m |= 1ull << j;
            ++d;
        }
        anc[tid] = m;
        depth[tid] = d;
        uint8_t* pl = plist + tid * 64;
        float gs = 0.f;
        int i = 0;
#pragma unroll 1
        for (uint64_t r = m; r; r &= r - 1) {
            const int j = __ffsll((long long)r) - 1;
            gs += la[j];
            pl[i++] = (uint8_t)j;
        }
        pl[i] = (uint8_t)tid;
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
#pragma unroll 1
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
#pragma unroll 1
        for (uint64_t r = anc[tid]; r; r &= r - 1)
            pairs[o++] = (uint16_t)((tid << 8) | (__ffsll((long long)r) - 1));
        pairs[o] = (uint16_t)((tid << 8) | tid);
    }
    __syncthreads();
}

// A and Attn entries of pair (t, j) from the raw dot products k_t.k_j and q_t.k_j.
// A is zero without the delta rule's erasure (decay-gated linear attention).
__device__ __forceinline__ void gram_entry(int t, int j, float kk, float qk, int ld, const float* g,
                                           const float* beta, float* sA, float* sAt, bool delta_rule = true) {
    const float gam = expf(g[t] - g[j]);
    sAt[t * ld + j] = gam * qk;
    if (j != t) sA[t * ld + j] = delta_rule ? beta[t] * gam * kk : 0.f;
}

// Rows of T = (I + A)^-1, then P = Attn T over A.  The principal block of
// I + A on path(t) is closed (ancestors of path nodes are on the path), so
// row t of T is the last row of that block's inverse: with the path
// p_0 (root) .. p_m = t, x_m = 1 and x_k = -sum_{i > k} x_i A[p_i, p_k]
// (k = m-1 .. 0).  Then P[t, p_k] = sum_{i >= k} Attn[t, p_i] T[p_i, p_k].
// One thread per node, counted loops over the path list (independent loads),
// no level barriers.  Call with every thread; contains barriers.
__device__ __forceinline__ void solve_rows(int tid, int N, int ld, const int* depth, const uint8_t* plist,
                                           float* sA, const float* sAt, float* sT) {
    if (tid < N) {
        const int t = tid, m = depth[t];
        const uint8_t* p = plist + t * 64;
        float* row = sT + t * ld;
        row[t] = 1.f;
#pragma unroll 1
        for (int k = m - 1; k >= 0; --k) {
            const int pk = p[k];
            float x0 = 0.f, x1 = 0.f;
            int i = k + 1;
            for (; i + 1 <= m; i += 2) {
                const int a0 = p[i], a1 = p[i + 1];
                x0 = fmaf(row[a0], sA[a0 * ld + pk], x0);
                x1 = fmaf(row[a1], sA[a1 * ld + pk], x1);
            }
            if (i <= m) x0 = fmaf(row[p[i]], sA[p[i] * ld + pk], x0);
            row[pk] = -(x0 + x1);
        }
    }
    __syncthreads();
    if (tid < N) {
        const int t = tid, m = depth[t];
        const uint8_t* p = plist + t * 64;
#pragma unroll 1
        for (int k = 0; k <= m; ++k) {
            const int pk = p[k];
            float x0 = 0.f, x1 = 0.f;
            int i = k;
            for (; i + 1 <= m; i += 2) {
                const int a0 = p[i], a1 = p[i + 1];
                x0 = fmaf(sAt[t * ld + a0], sT[a0 * ld + pk], x0);
                x1 = fmaf(sAt[t * ld + a1], sT[a1 * ld + pk], x1);
            }
            if (i <= m) x0 = fmaf(sAt[t * ld + p[i]], sT[p[i] * ld + pk], x0);
            sA[t * ld + pk] = x0 + x1;   // A is no longer read: step one finished behind the barrier
        }
    }
    __syncthreads();
}

// Row t's A and Attn entries from its Gram rows: qk[j] = q_t.k_j, kk[j] = k_t.k_j
// (row pointers into a Gram table), for j on path(t).  One thread per node.
__device__ __forceinline__ void gram_row(int t, int m, const uint8_t* plist, const float* qk, const float* kk,
                                         int ld, const float* g, const float* beta, float* sA, float* sAt,
                                         bool delta_rule = true) {
    const uint8_t* p = plist + t * 64;
    const float gt = g[t], bt = beta[t];
#pragma unroll 1
    for (int i = 0; i <= m; ++i) {
        const int j = p[i];
        const float gam = expf(gt - g[j]);
        sAt[t * ld + j] = gam * qk[j];
        if (j != t) sA[t * ld + j] = delta_rule ? bt * gam * kk[j] : 0.f;
    }
}

// gram_row's entries i = part, part + nparts, ... of row t's path: several threads
// share one node's row.
__device__ __forceinline__ void gram_row_part(int t, int part, int nparts, int m, const uint8_t* plist,
                                              const float* qk, const float* kk, int ld, const float* g,
                                              const float* beta, float* sA, float* sAt, bool delta_rule = true) {
    const uint8_t* p = plist + t * 64;
    const float gt = g[t], bt = beta[t];
#pragma unroll 1
    for (int i = part; i <= m; i += nparts) {
        const int j = p[i];
        const float gam = expf(gt - g[j]);
        sAt[t * ld + j] = gam * qk[j];
        if (j != t) sA[t * ld + j] = delta_rule ? bt * gam * kk[j] : 0.f;
    }
}

// solve_rows with the path held in registers: q_0 = t, q_1 = parent, ..., q_m
// = root.  Row t of T: x_0 = 1, x_i = -sum_{j < i} x_j A[q_j, q_i]; row t of
// P: P[t, q_i] = sum_{j <= i} Attn[t, q_j] T[q_j, q_i].  Fully unrolled for
// depth < kRegDepth (independent shared-memory loads; the code grows as
// kRegDepth^2), the generic loops of solve_rows otherwise.  Call with every
// thread of the block, or with `group` > 0 with the first `group` threads,
// which then synchronise on named barrier 1 only; contains barriers.
__device__ __forceinline__ void group_sync(int group) {
    if (group == 0)
        __syncthreads();
    else
        asm volatile("bar.sync 1, %0;\n" ::"r"(group) : "memory");
}

template <int kRegDepth = 12>
__device__ __forceinline__ void solve_rows_fast(int tid, int N, int ld, const int* depth, const uint8_t* plist,
                                                float* sA, const float* sAt, float* sT, int group = 0) {
    const int t = tid;
    const int m = tid < N ? depth[t] : 0;
    const bool fast = tid < N && m < kRegDepth;
    int q[kRegDepth];
    float x[kRegDepth];
    if (fast) {
        const uint8_t* p = plist + t * 64;
#pragma unroll
        for (int i = 0; i < kRegDepth; ++i) q[i] = i <= m ? p[m - i] : t;
        x[0] = 1.f;
#pragma unroll
        for (int i = 1; i < kRegDepth; ++i) {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int j = 0; j < i; j += 2) {
                s0 = fmaf(x[j], sA[q[j] * ld + q[i]], s0);
                if (j + 1 < i) s1 = fmaf(x[j + 1], sA[q[j + 1] * ld + q[i]], s1);
            }
            x[i] = i <= m ? -(s0 + s1) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kRegDepth; ++i)
            if (i <= m) sT[t * ld + q[i]] = x[i];
    } else if (tid < N) {
        const uint8_t* p = plist + t * 64;
        float* row = sT + t * ld;
        row[t] = 1.f;
#pragma unroll 1
        for (int k = m - 1; k >= 0; --k) {
            const int pk = p[k];
            float x0 = 0.f;
#pragma unroll 1
            for (int i = k + 1; i <= m; ++i) x0 = fmaf(row[p[i]], sA[p[i] * ld + pk], x0);
            row[pk] = -x0;
        }
    }
    group_sync(group);
    if (fast) {
        // every entry of the row first, then the stores: a store to sA between them would
        // keep the next entry's sT loads (which the compiler must assume may alias it) behind it
        float at[kRegDepth], pr[kRegDepth];
#pragma unroll
        for (int j = 0; j < kRegDepth; ++j) at[j] = j <= m ? sAt[t * ld + q[j]] : 0.f;
#pragma unroll
        for (int i = 0; i < kRegDepth; ++i) {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int j = 0; j <= i; j += 2) {
                s0 = fmaf(at[j], sT[q[j] * ld + q[i]], s0);
                if (j + 1 <= i) s1 = fmaf(at[j + 1], sT[q[j + 1] * ld + q[i]], s1);
            }
            pr[i] = s0 + s1;
        }
#pragma unroll
        for (int i = 0; i < kRegDepth; ++i)
            if (i <= m) sA[t * ld + q[i]] = pr[i];
    } else if (tid < N) {
        const uint8_t* p = plist + t * 64;
#pragma unroll 1
        for (int k = 0; k <= m; ++k) {
            const int pk = p[k];
            float x0 = 0.f;
#pragma unroll 1
            for (int i = k; i <= m; ++i) x0 = fmaf(sAt[t * ld + p[i]], sT[p[i] * ld + pk], x0);
            sA[t * ld + pk] = x0;
        }
    }
    group_sync(group);
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
