// grouped_gemm.cuh -- host-side interface of the tcgen05 GroupedGEMMs.
//
// "A GroupedGEMM runs the matrix products of several experts in one kernel"
// (MegaScale-MoE research digest, glossary and §3.3).  One persistent kernel
// per matmul family handles every expert: the per-expert row ranges come from
// the device-resident `offsets` array, so no count ever travels to the host.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

struct GemmProblem {
  int E;                    // experts
  const int32_t* offsets;   // [E+1] expert row ranges in the permuted order (device)
  int rows;                 // T*k permuted rows
  int h, f;                 // hidden size, expert width
  int* status;              // device status word
  int num_sms;              // persistent grid size
};

// A = X W1, B = X W3, H = silu(A) * B for the rows of each expert.
// X: x_perm [rows, h]; W1, W3: [E, h, f]; outputs [rows, f] bf16.
cudaError_t gemm_fc1_fwd(const GemmProblem& p, const void* x_perm, const void* W1,
                         const void* W3, void* A, void* B, void* H, cudaStream_t s);
// O = H W2 for the rows of each expert.  H: [rows, f]; W2: [E, f, h]; O: [rows, h].
cudaError_t gemm_fc2_fwd(const GemmProblem& p, const void* H, const void* W2, void* O,
                         cudaStream_t s);
// dH = dO W2^T, fused with the SwiGLU backward: dA = dH * B * s (1 + A (1 - s)),
// dB = dH * silu(A).  dO: [rows, h]; A, B, dA, dB: [rows, f] bf16.  With
// ab_amax [rows, gemm_col_tiles(f)], also the amax of |dA|, |dB| (fp32, before
// the bf16 store) over each 256-column tile of a row.
cudaError_t gemm_fc2_dgrad(const GemmProblem& p, const void* dO, const void* W2,
                           const void* A, const void* B, void* dA, void* dB, cudaStream_t s,
                           float* ab_amax = nullptr);
// The same matmul for selective activation rematerialisation, where neither H
// nor O was kept: the A operand is the ungated dy_perm [rows, h], and with
// u = dy_perm W2^T, g = gate_rows[row] and H = silu(A) * B rebuilt here:
//   dA, dB from dH = g u;  gH = g H (bf16 [rows, f]);
//   dg_part[row, nt] = sum of H u over n-tile nt (fp32 [rows, gemm_col_tiles(f)]).
cudaError_t gemm_fc2_dgrad_sar(const GemmProblem& p, const void* dy_perm, const void* W2,
                               const void* A, const void* B, const float* gate_rows, void* dA,
                               void* dB, void* gH, float* dg_part, cudaStream_t s);
// FP8 forward (e4m3 codes, per-row and per-column float32 scales; h and f
// multiples of 128):
//   A = sx * s1 * (Xq W1q), B = sx * s3 * (Xq W3q), H = silu(A) * B   (bf16 out)
//   Xq [rows, h]; W13q [E, 2f, h] with 128-row groups alternating W1 and W3
//   columns; s1, s3 [E, f]; sx [rows].
//   h_amax [rows, gemm_fc1_col_tiles(f)]: amax of |H| (fp32, before the bf16
//   store) over each 128-column tile of a row.
cudaError_t gemm_fc1_fwd_fp8(const GemmProblem& p, const void* Xq, const float* sx,
                             const void* W13q, const float* s1, const float* s3, void* A, void* B,
                             void* H, float* h_amax, cudaStream_t s);
int gemm_fc1_col_tiles(int f);
//   O = sh * s2 * (Hq W2q): Hq [rows, f]; W2q [E, h, f]; s2 [E, h]; sh [rows].
cudaError_t gemm_fc2_fwd_fp8(const GemmProblem& p, const void* Hq, const float* sh,
                             const void* W2q, const float* s2, void* O, cudaStream_t s);
// FP8 FC1 data gradient:
//   dX = sab * s13r * (dAq W1r^T + dBq W3r^T), fp32 [rows, h]; dAq, dBq
//   [rows, f], W1r, W3r [E, h, f] e4m3, s13r [E, h], sab [rows].
cudaError_t gemm_fc1_dgrad_fp8(const GemmProblem& p, const void* dAq, const void* dBq,
                               const float* sab, const void* W1r, const void* W3r,
                               const float* s13r, float* dX, cudaStream_t s);
// Output-column tiles of the M-grouped matmuls for n columns.
int gemm_col_tiles(int n);
// dX_perm = dA W1^T + dB W3^T (K = 2f), fp32 [rows, h].
cudaError_t gemm_fc1_dgrad(const GemmProblem& p, const void* dA, const void* dB,
                           const void* W1, const void* W3, float* dX, cudaStream_t s);
// dW2[e] = H_e^T dO_e, ragged K = rows of e.  fp32 [E, f, h].
cudaError_t gemm_fc2_wgrad(const GemmProblem& p, const void* H, const void* dO, float* dW2,
                           cudaStream_t s);
// dW1[e] = X_e^T dA_e, dW3[e] = X_e^T dB_e.  fp32 [E, h, f].
cudaError_t gemm_fc1_wgrad(const GemmProblem& p, const void* x_perm, const void* dA,
                           const void* dB, float* dW1, float* dW3, cudaStream_t s);

// Kernel names, in launch order of a layer, for the measurement hook.
extern const char* const kGemmNames[6];
extern const char* const kGemmSarDgradName;

}  // namespace moe
