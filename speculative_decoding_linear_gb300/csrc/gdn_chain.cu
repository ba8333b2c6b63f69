// gdn_chain.cu -- chain verification with the state resident on chip.
//
// Review of SpecLA (pith.science 7ERME3HB), "What carries the argument":
// "V-dimension tiling for the serial chain path".  For a chain draft (node t
// hangs under t-1) every row of S evolves independently:
//
//     s = S_row . k_t,  u = S_row . q_t            (one pass over the row)
//     delta_t = beta_t (v_t[row] - alpha_t s)
//     o_t[row] = S_t,row . q_t = alpha_t u + delta_t (k_t . q_t)
//     S_row <- alpha_t S_row + delta_t k_t^T
//
// so the state is tiled along d_v: one CTA holds kRowsPerCta rows of one
// (sequence, head) state in registers (one warp per kRowsPerWarp rows, each
// lane holding d_k/32 columns) and runs the N tokens serially without ever
// writing intermediate states.  When fused with a pending commit, the rows are
// first committed (same arithmetic as the standalone commit) and written back
// once.  The kernel emits the same factor record as the tree verifier.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = 4;
constexpr int kRowsPerCta = kWarps * kRowsPerWarp;   // 16
constexpr int kEPL = kMaxDim / 32;                   // columns per lane

struct ChainSmem {
    float o[kMaxNodes * kRowsPerCta];
    float d[kMaxNodes * kRowsPerCta];
    float v[kMaxNodes * kRowsPerCta];
    float alpha[kMaxNodes];
    float beta[kMaxNodes];
    float cd[kMaxPath * kRowsPerCta];
    float coef[kMaxPath];
    int nodes[kMaxPath];
    float ega;
    int L;
};

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) chain_kernel(VerifyArgs a) {
    __shared__ ChainSmem s;
    const int bh = blockIdx.x;
    const int b = bh / a.H, h = bh % a.H;
    const int N = a.N, dk = a.dk, dv = a.dv, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int v0 = blockIdx.y * kRowsPerCta;
    const int rows = min(kRowsPerCta, dv - v0);
    const T* q = static_cast<const T*>(a.q);
    const T* k = static_cast<const T*>(a.k);
    const T* vv = static_cast<const T*>(a.v);

    // gates and values of this CTA's rows
    for (int t = tid; t < N; t += kWarps * 32) {
        const size_t gi = ((size_t)b * N + t) * a.H + h;
        s.alpha[t] = a.alpha[gi];
        s.beta[t] = a.beta[gi];
    }
    for (int i = tid; i < N * kRowsPerCta; i += kWarps * 32) {
        const int t = i / kRowsPerCta, r = i % kRowsPerCta;
        s.v[i] = r < rows ? ld_elem<T>(vv, (((size_t)b * N + t) * a.H + h) * dv + v0 + r) : 0.f;
    }
    const bool fused = a.commit.path != nullptr;
    if (fused) {
        if (warp == 0) {
            const int L = commit_path_setup(a.commit, b, h, a.H, s.nodes, s.coef, &s.ega);
            if (lane == 0) {
                s.L = L;
                if (L < 0) set_error(a.err, GDN_ERR_PATH);
            }
        }
        __syncthreads();
        if (s.L < 0) return;
        const float* dl = a.commit.delta + (size_t)bh * a.commit.N * dv;
        for (int i = tid; i < s.L * kRowsPerCta; i += kWarps * 32) {
            const int j = i / kRowsPerCta, r = i % kRowsPerCta;
            s.cd[i] = r < rows ? s.coef[j] * dl[(size_t)s.nodes[j] * dv + v0 + r] : 0.f;
        }
    }
    __syncthreads();

    // state rows -> registers (committed and written back once when fused)
    float S[kRowsPerWarp][kEPL];
    const T* ckey = fused ? static_cast<const T*>(a.commit.key) + (size_t)bh * a.commit.N * dk : nullptr;
#pragma unroll
    for (int rr = 0; rr < kRowsPerWarp; ++rr) {
        const int r = warp * kRowsPerWarp + rr;
        const size_t row = ((size_t)bh * dv + v0 + r) * dk;
#pragma unroll
        for (int e = 0; e < kEPL; ++e) {
            const int c = lane + 32 * e;
            float x = 0.f;
            if (r < rows && c < dk) {
                x = a.S[row + c];
                if (fused) {
                    float acc = s.ega * x;
                    for (int i = 0; i < s.L; ++i)
                        acc = fmaf(s.cd[i * kRowsPerCta + r],
                                   ld_elem<T>(ckey, (size_t)s.nodes[i] * dk + c), acc);
                    x = acc;
                    a.S[row + c] = x;
                }
            }
            S[rr][e] = x;
        }
    }

    // serial chain
    for (int t = 0; t < N; ++t) {
        const size_t rt = (((size_t)b * N + t) * a.H + h) * dk;
        float kt[kEPL], qt[kEPL];
        float kq = 0.f;
#pragma unroll
        for (int e = 0; e < kEPL; ++e) {
            const int c = lane + 32 * e;
            kt[e] = c < dk ? ld_elem<T>(k, rt + c) : 0.f;
            qt[e] = c < dk ? ld_elem<T>(q, rt + c) : 0.f;
            kq = fmaf(kt[e], qt[e], kq);
        }
        kq = warp_sum(kq);
        const float al = s.alpha[t], be = s.beta[t];
        float sk[kRowsPerWarp], sq[kRowsPerWarp];
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
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
#pragma unroll
            for (int rr = 0; rr < kRowsPerWarp; ++rr) {
                sk[rr] += __shfl_xor_sync(0xffffffffu, sk[rr], o);
                sq[rr] += __shfl_xor_sync(0xffffffffu, sq[rr], o);
            }
        }
#pragma unroll
        for (int rr = 0; rr < kRowsPerWarp; ++rr) {
            const int r = warp * kRowsPerWarp + rr;
            const float dlt = be * (s.v[t * kRowsPerCta + r] - al * sk[rr]);
            const float o = fmaf(al, sq[rr], dlt * kq);
#pragma unroll
            for (int e = 0; e < kEPL; ++e) S[rr][e] = fmaf(al, S[rr][e], dlt * kt[e]);
            if (lane == 0) {
                s.o[t * kRowsPerCta + r] = o;
                s.d[t * kRowsPerCta + r] = dlt;
            }
        }
    }
    __syncthreads();

    // outputs and factors (coalesced along d_v)
    for (int i = tid; i < N * kRowsPerCta; i += kWarps * 32) {
        const int t = i / kRowsPerCta, r = i % kRowsPerCta;
        if (r >= rows) continue;
        a.out[(((size_t)b * N + t) * a.H + h) * dv + v0 + r] = s.o[i];
        a.f.delta[((size_t)bh * N + t) * dv + v0 + r] = s.d[i];
    }
    // key copy, gates and parents: spread over the CTAs of this (b, h)
    T* key_out = static_cast<T*>(a.f.key);
    for (int t = blockIdx.y; t < N; t += gridDim.y) {
        const size_t rt = (((size_t)b * N + t) * a.H + h) * dk;
        for (int c = tid; c < dk; c += kWarps * 32)
            key_out[((size_t)bh * N + t) * dk + c] = k[rt + c];
    }
    if (blockIdx.y == 0 && warp == 0) {
        // g_t = sum_{i <= t} log alpha_i : warp scan over chunks of 32 nodes
        float carry = 0.f;
        for (int t0 = 0; t0 < N; t0 += 32) {
            const int t = t0 + lane;
            float x = t < N ? logf(s.alpha[t]) : 0.f;
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

}  // namespace

cudaError_t launch_chain_verify(const VerifyArgs& a, int dtype, cudaStream_t s) {
    dim3 grid(a.B * a.H, (a.dv + kRowsPerCta - 1) / kRowsPerCta);
    if (dtype == GDN_DTYPE_F32)
        chain_kernel<float><<<grid, kWarps * 32, 0, s>>>(a);
    else
        chain_kernel<__nv_bfloat16><<<grid, kWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace gdn
