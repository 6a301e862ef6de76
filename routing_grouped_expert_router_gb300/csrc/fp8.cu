// fp8.cu -- e4m3 quantisation for the FP8 expert forward.
//
// FP8 training with per-token quantisation instead of per-tensor (MegaScale-
// MoE review §三 创新点 "FP8训练优化"; digest §3.4: per-token scales on the FP8
// path).  The scales:
//   activations (x_perm, H): one float32 scale per row,      s = amax / 448
//   expert weights:          one per output column of each expert (amax over
//                            the contraction dimension),     s = amax / 448
// with s = 1 for an all-zero row or column, and q = e4m3(v / s): the division
// in IEEE float32, the conversion round-to-nearest-even with saturation
// (cuda_fp8.h, __NV_SATFINITE).  The matmul consumes the codes and rescales
// its fp32 sums by s_row * s_col.
//
// The weights are written transposed, K-major (the contraction dimension
// contiguous), because that is the operand layout the FP8 GroupedGEMM loads:
//   W13q [E, 2f, h]: for each expert, 128-row groups alternating W1 and W3
//                    columns (group 2j = W1 columns 128j..128j+127, group
//                    2j+1 = the same W3 columns), so one 256-row B tile holds
//                    matching W1 and W3 columns;
//   W2q  [E, h, f].
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.cuh"

namespace moe {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float scale_of(float amax) {
  return amax > 0.f ? __fdiv_rn(amax, kE4M3Max) : 1.0f;
}

// Two values -> two e4m3 codes (low byte = first value).
__device__ __forceinline__ uint32_t q2(float a, float b, float s) {
  const float2 v = make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s));
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3));
}

// Row p of the output quantises row src(p) of `in` (idx[p] / div when idx is
// given, else p).  A warp per row: one pass for the amax, one to quantise (the
// row is then in L1 or L2).  Rows p >= *nvalid (when nvalid is given) are
// skipped.
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint4* __restrict__ in,
                                                         const int32_t* __restrict__ idx, int div,
                                                         long long rows, long long src_rows,
                                                         const int32_t* __restrict__ nvalid,
                                                         int n8, uint2* __restrict__ q,
                                                         float* __restrict__ scale) {
  const int lane = threadIdx.x & 31;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  if (nvalid) {
    const long long nv = __ldg(nvalid);
    rows = nv < rows ? (nv < 0 ? 0 : nv) : rows;
  }
  for (long long p = gw; p < rows; p += nw) {
    long long src = idx ? __ldg(idx + p) / div : p;
    src = src < 0 ? 0 : (src >= src_rows ? src_rows - 1 : src);
    const uint4* r = in + src * n8;
    float amax = 0.f;
    for (int c = lane; c < n8; c += 32) {
      const uint4 w = __ldg(r + c);
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(u[j])), fabsf(bf16_hi(u[j]))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
    const float s = scale_of(amax);
    if (lane == 0) scale[p] = s;
    uint2* out = q + p * n8;
    for (int c = lane; c < n8; c += 32) {
      const uint4 w = __ldg(r + c);
      const uint32_t lo = q2(bf16_lo(w.x), bf16_hi(w.x), s) | (q2(bf16_lo(w.y), bf16_hi(w.y), s) << 16);
      const uint32_t hi = q2(bf16_lo(w.z), bf16_hi(w.z), s) | (q2(bf16_lo(w.w), bf16_hi(w.w), s) << 16);
      out[c] = make_uint2(lo, hi);
    }
  }
}

// Expert weights W [E, K, N] bf16 (N contiguous) -> per-(e, n) scales and
// K-major codes: output row of column n of expert e is
//   e * rows_per_e + (n / 128) * group_stride + slot * 128 + n % 128,
// row length K bytes.  A block takes 64 columns of one expert: pass 1 reduces
// their amax over K, pass 2 moves 64 x 64 tiles through shared memory,
// quantising and transposing them.
constexpr int kQcCols = 64;
constexpr int kQcRows = 64;

__global__ void __launch_bounds__(256) quant_cols_kernel(const uint16_t* __restrict__ W, int K,
                                                         int N, int rows_per_e, int group_stride,
                                                         int slot, uint8_t* __restrict__ q,
                                                         float* __restrict__ scale) {
  __shared__ float part[4][kQcCols];
  __shared__ float s_col[kQcCols];
  __shared__ uint16_t tile[kQcRows][kQcCols + 2];
  const int e = blockIdx.y;
  const int n0 = blockIdx.x * kQcCols;
  const int t = threadIdx.x;
  const uint16_t* We = W + static_cast<size_t>(e) * K * N;

  // pass 1: amax of each column (4 row groups per column, then combined)
  {
    const int c = t & (kQcCols - 1);
    const int g = t >> 6;
    float amax = 0.f;
    if (n0 + c < N)
      for (int k = g; k < K; k += 4)
        amax = fmaxf(amax, fabsf(__uint_as_float(static_cast<uint32_t>(
                               __ldg(We + static_cast<size_t>(k) * N + n0 + c)) << 16)));
    part[g][c] = amax;
  }
  __syncthreads();
  if (t < kQcCols) {
    const float amax = fmaxf(fmaxf(part[0][t], part[1][t]), fmaxf(part[2][t], part[3][t]));
    const float s = scale_of(amax);
    s_col[t] = s;
    if (n0 + t < N) scale[static_cast<size_t>(e) * N + n0 + t] = s;
  }
  __syncthreads();

  // pass 2: 64 x 64 tiles, quantised and written K-major
  for (int k0 = 0; k0 < K; k0 += kQcRows) {
    for (int i = t; i < kQcRows * kQcCols; i += 256) {
      const int r = i / kQcCols;
      const int c = i % kQcCols;
      tile[r][c] = (k0 + r < K && n0 + c < N) ? __ldg(We + static_cast<size_t>(k0 + r) * N + n0 + c)
                                             : static_cast<uint16_t>(0);
    }
    __syncthreads();
    // thread -> (column c, 16-row segment g): 16 codes, one 16-byte store
    const int c = t >> 2;
    const int g = t & 3;
    const int n = n0 + c;
    if (n < N && k0 + g * 16 < K) {
      const float s = s_col[c];
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = g * 16 + 4 * j;
        const float v0 = __uint_as_float(static_cast<uint32_t>(tile[r + 0][c]) << 16);
        const float v1 = __uint_as_float(static_cast<uint32_t>(tile[r + 1][c]) << 16);
        const float v2 = __uint_as_float(static_cast<uint32_t>(tile[r + 2][c]) << 16);
        const float v3 = __uint_as_float(static_cast<uint32_t>(tile[r + 3][c]) << 16);
        w[j] = q2(v0, v1, s) | (q2(v2, v3, s) << 16);
      }
      const size_t orow = static_cast<size_t>(e) * rows_per_e + (n / 128) * group_stride +
                          slot * 128 + n % 128;
      *reinterpret_cast<uint4*>(q + orow * K + k0 + g * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();
  }
}

int grid_rows(long long rows, int num_sms) {
  const long long warps = rows;
  long long blocks = (warps + 7) / 8;
  const long long cap = static_cast<long long>(num_sms) * 16;
  return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_quant_rows(const uint16_t* in, const int32_t* idx, int div, long long rows,
                              long long src_rows, int n, uint8_t* q, float* scale, int num_sms,
                              cudaStream_t s, const int32_t* nvalid) {
  if (rows == 0 || src_rows == 0) return cudaSuccess;
  quant_rows_kernel<<<grid_rows(rows, num_sms), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(in), idx, div, rows, src_rows, nvalid, n / 8,
      reinterpret_cast<uint2*>(q), scale);
  return launched();
}

cudaError_t launch_quant_cols(const uint16_t* W, int E, int K, int N, int rows_per_e,
                              int group_stride, int slot, uint8_t* q, float* scale,
                              cudaStream_t s) {
  if (E == 0 || K == 0 || N == 0) return cudaSuccess;
  const dim3 grid((N + kQcCols - 1) / kQcCols, E);
  quant_cols_kernel<<<grid, 256, 0, s>>>(W, K, N, rows_per_e, group_stride, slot, q, scale);
  return launched();
}

}  // namespace moe
