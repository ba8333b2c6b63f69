// gdn_layer.cuh -- internal declarations for the full GDN layer decode step
// (projections, ancestor-window convolution, gates, tree verification with
// the fused commit, output gate and output projection).
#pragma once

#include "gdn_internal.cuh"

namespace gdn {

constexpr int kConvTaps = 4;      // four-tap depthwise conv over each node's window

// C[M x Nc] (fp32, row stride ldc elements) = sum_s A_s[M x K] B[Nc x K]^T with
// bf16 row-major operands (K contiguous; A rows lda elements apart, B rows K).
// nA = 1, or 2 for an fp32 left operand carried as two bf16 terms (hi + lo).
// K must be a multiple of 64, lda a multiple of 8; operands 16-byte aligned.
cudaError_t launch_gemm_bf16(const void* A0, const void* A1, int nA, long long lda, const void* B, float* C,
                             long long ldc, int M, int Nc, int K, int* err, cudaStream_t s);

// Sizes of the layer's record (kept until the next step's commit) and workspace.
struct LayerLayout {
    int B, N, H, hidden, dk, dv;
    int rows;          // projection outputs per token: q | k | v | z | a | b
    int conv_ch;       // convolution channels: q | k | v
    long long ldy;     // row stride of the projection output (elements, multiple of 4)
    // record
    size_t y_off, fac_off, record_bytes;
    // workspace
    size_t q_off, k_off, v_off, alpha_off, beta_off, o_off, split_off[4], yhi_off, ylo_off, tws_off,
        workspace_bytes;
};

LayerLayout layer_layout(int B, int N, int H, int hidden, int dk, int dv);

}  // namespace gdn
