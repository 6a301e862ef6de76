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
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

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
// row is then in L1 or L2).  With amax_part, the row's amax is instead the
// bf16 rounding of the largest of its nt fp32 partial maxima (the same value,
// since rounding to nearest is monotone and symmetric) and the row is read
// once.  With copy, the quantising pass also writes the bf16 row to copy[p]
// (the permute of the same rows, fused).  With in1/q1, row src of in1 is
// quantised into q1 with the same scale, the amax taken over both rows.  Rows
// p >= *nvalid (when nvalid is given) are skipped.  A source index outside
// [0, src_rows) is recorded in *status and quantised as a zero row.
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint4* __restrict__ in,
                                                         const int32_t* __restrict__ idx, int div,
                                                         long long rows, long long src_rows,
                                                         const int32_t* __restrict__ nvalid,
                                                         int n8, uint2* __restrict__ q,
                                                         float* __restrict__ scale,
                                                         const float* __restrict__ amax_part,
                                                         int nt, uint4* __restrict__ copy,
                                                         const uint4* __restrict__ in1,
                                                         uint2* __restrict__ q1,
                                                         int* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  if (nvalid) {
    const long long nv = __ldg(nvalid);
    rows = nv < rows ? (nv < 0 ? 0 : nv) : rows;
  }
  for (long long p = gw; p < rows; p += nw) {
    const long long src = idx ? __ldg(idx + p) / div : p;
    if (src < 0 || src >= src_rows) {
      if (lane == 0) {
        report_bad_index(status);
        scale[p] = 1.f;
      }
      for (int c = lane; c < n8; c += 32) {
        q[p * n8 + c] = make_uint2(0, 0);
        if (copy) copy[p * n8 + c] = make_uint4(0, 0, 0, 0);
        if (q1) q1[p * n8 + c] = make_uint2(0, 0);
      }
      continue;
    }
    const uint4* r = in + src * n8;
    const uint4* r1 = in1 ? in1 + src * n8 : nullptr;
    float amax = 0.f;
    if (amax_part) {
      for (int i = lane; i < nt; i += 32) amax = fmaxf(amax, __ldg(amax_part + p * nt + i));
    } else {
      for (int c = lane; c < n8; c += 32) {
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          if (which == 1 && !r1) break;
          const uint4 w = __ldg((which ? r1 : r) + c);
          const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int j = 0; j < 4; ++j)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(u[j])), fabsf(bf16_hi(u[j]))));
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
    if (amax_part) amax = __bfloat162float(__float2bfloat16_rn(amax));
    const float s = scale_of(amax);
    if (lane == 0) scale[p] = s;
    uint2* out = q + p * n8;
    uint4* cp = copy ? copy + p * n8 : nullptr;
    for (int c = lane; c < n8; c += 32) {
      const uint4 w = __ldg(r + c);
      if (cp) cp[c] = w;
      const uint32_t lo = q2(bf16_lo(w.x), bf16_hi(w.x), s) | (q2(bf16_lo(w.y), bf16_hi(w.y), s) << 16);
      const uint32_t hi = q2(bf16_lo(w.z), bf16_hi(w.z), s) | (q2(bf16_lo(w.w), bf16_hi(w.w), s) << 16);
      out[c] = make_uint2(lo, hi);
      if (r1) {
        const uint4 w1 = __ldg(r1 + c);
        const uint32_t lo1 =
            q2(bf16_lo(w1.x), bf16_hi(w1.x), s) | (q2(bf16_lo(w1.y), bf16_hi(w1.y), s) << 16);
        const uint32_t hi1 =
            q2(bf16_lo(w1.z), bf16_hi(w1.z), s) | (q2(bf16_lo(w1.w), bf16_hi(w1.w), s) << 16);
        q1[p * n8 + c] = make_uint2(lo1, hi1);
      }
    }
  }
}

// The same operation as quant_rows_kernel with a 256-thread block per row (or
// row pair), the whole row held in registers: NPT 16-byte pieces per thread and
// row, every load issued before any arithmetic, the amax a block reduction.
// The row is read from memory once whatever the amax source, and a block has
// its full row (28 KB for 14336 bf16 values, twice that for a pair) in flight
// at once; the warp-per-row kernel kept one 16-byte load per lane in flight
// and read two-pass rows twice from DRAM.  The codes and scales are the same
// (the amax is a max, whatever the order).
constexpr int kQrThreads = 256;
constexpr int kQrMaxNpt = 8;  // rows up to 8 * 256 * 8 = 16384 values

template <int NPT, bool PAIR>
__global__ void __launch_bounds__(kQrThreads) quant_rows_reg_kernel(
    const uint4* __restrict__ in, const int32_t* __restrict__ idx, int div, long long rows,
    long long src_rows, const int32_t* __restrict__ nvalid, int n8, uint2* __restrict__ q,
    float* __restrict__ scale, const float* __restrict__ amax_part, int nt,
    uint4* __restrict__ copy, const uint4* __restrict__ in1, uint2* __restrict__ q1,
    int* __restrict__ status) {
  __shared__ float red[kQrThreads / 32];
  const int t = threadIdx.x;
  const int lane = t & 31;
  if (nvalid) {
    const long long nv = __ldg(nvalid);
    rows = nv < rows ? (nv < 0 ? 0 : nv) : rows;
  }
  for (long long p = blockIdx.x; p < rows; p += gridDim.x) {
    const long long src = idx ? __ldg(idx + p) / div : p;
    if (src < 0 || src >= src_rows) {  // block-uniform: the whole block skips the row
      if (t == 0) {
        report_bad_index(status);
        scale[p] = 1.f;
      }
      for (int c = t; c < n8; c += kQrThreads) {
        q[p * n8 + c] = make_uint2(0, 0);
        if (copy) copy[p * n8 + c] = make_uint4(0, 0, 0, 0);
        if (PAIR) q1[p * n8 + c] = make_uint2(0, 0);
      }
      continue;
    }
    const uint4* r = in + src * n8;
    const uint4* r1 = PAIR ? in1 + src * n8 : nullptr;
    uint4 v[NPT];
    uint4 v1[PAIR ? NPT : 1];
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const int c = t + kQrThreads * j;
      v[j] = c < n8 ? __ldg(r + c) : make_uint4(0, 0, 0, 0);
      if constexpr (PAIR) v1[j] = c < n8 ? __ldg(r1 + c) : make_uint4(0, 0, 0, 0);
    }
    float amax = 0.f;
    if (amax_part) {
      for (int i = t; i < nt; i += kQrThreads) amax = fmaxf(amax, __ldg(amax_part + p * nt + i));
    } else {
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(u[i])), fabsf(bf16_hi(u[i]))));
        if constexpr (PAIR) {
          const uint32_t u1[4] = {v1[j].x, v1[j].y, v1[j].z, v1[j].w};
#pragma unroll
          for (int i = 0; i < 4; ++i)
            amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(u1[i])), fabsf(bf16_hi(u1[i]))));
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
    if (lane == 0) red[t >> 5] = amax;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kQrThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    if (amax_part) amax = __bfloat162float(__float2bfloat16_rn(amax));
    const float s = scale_of(amax);
    if (t == 0) scale[p] = s;
    uint2* out = q + p * n8;
    uint4* cp = copy ? copy + p * n8 : nullptr;
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const int c = t + kQrThreads * j;
      if (c < n8) {
        const uint4 w = v[j];
        if (cp) cp[c] = w;
        out[c] = make_uint2(q2(bf16_lo(w.x), bf16_hi(w.x), s) | (q2(bf16_lo(w.y), bf16_hi(w.y), s) << 16),
                            q2(bf16_lo(w.z), bf16_hi(w.z), s) | (q2(bf16_lo(w.w), bf16_hi(w.w), s) << 16));
        if constexpr (PAIR) {
          const uint4 w1 = v1[j];
          q1[p * n8 + c] =
              make_uint2(q2(bf16_lo(w1.x), bf16_hi(w1.x), s) | (q2(bf16_lo(w1.y), bf16_hi(w1.y), s) << 16),
                         q2(bf16_lo(w1.z), bf16_hi(w1.z), s) | (q2(bf16_lo(w1.w), bf16_hi(w1.w), s) << 16));
        }
      }
    }
    __syncthreads();  // red is rewritten by the next row
  }
}

// Expert weights W [E, K, N] bf16 (N contiguous) -> per-(e, n) scales and
// K-major codes: output row of column n of expert e is
//   e * rows_per_e + (n / 128) * group_stride + slot * 128 + n % 128,
// row length K bytes.
//
// A persistent grid of two 512-thread blocks per SM walks slabs of QC columns
// (64 or 32) of one expert.  Pass 1 reads the slab with 16-byte loads (QC / 8
// threads per row segment, 4096 / QC rows at a time) and reduces each
// column's amax; pass 2 reads the slab again, in chunks of 16 * QC / 4 rows
// staged in shared memory, and writes each column's codes as 32-byte runs of
// its K-major output row (lane -> column, warp -> 32-row segment).  The next
// chunk's loads are issued before the current chunk is written.  Pass 2's
// read hits L2 when the slabs in flight (two per SM, K x 2 QC bytes each) fit
// in it, which narrower slabs make more likely.
constexpr int kQcThreads = 512;

template <int QC>
struct QcShape {
  static constexpr int TPR = QC / 8;                  // threads per row segment
  static constexpr int RSTEP = kQcThreads / TPR;      // rows per load step
  static constexpr int SEGS = QC == 64 ? 8 : 16;      // 32-row segments per chunk
  static constexpr int CHUNK = 32 * SEGS;             // rows per pass-2 chunk
  static constexpr int LOADS = CHUNK / RSTEP;         // 16-byte loads per thread per chunk
  static constexpr int PITCH = QC + 8;                // bf16 per staged row
  static constexpr int RED = RSTEP * (QC + 1) * 4;    // pass-1 reduction bytes
  static constexpr int TILE = CHUNK * PITCH * 2;      // pass-2 staging bytes
  static constexpr int SMEM = RED > TILE ? RED : TILE;
  static_assert(QC == 64 || QC == 32, "slab width");
  static_assert(kQcThreads / 32 == SEGS * (QC / 32), "one warp per (segment, 32 columns)");
};

template <int QC>
__global__ void __launch_bounds__(kQcThreads, 2) quant_cols_kernel(
    const uint16_t* __restrict__ W, int E, int K, int N, int rows_per_e, int group_stride,
    int slot, uint8_t* __restrict__ q, float* __restrict__ scale) {
  using S = QcShape<QC>;
  // pass 1 uses it as float [RSTEP][QC + 1], pass 2 as bf16 [CHUNK][PITCH]
  __shared__ __align__(16) uint8_t smem[S::SMEM];
  __shared__ float s_col[QC];
  float* red = reinterpret_cast<float*>(smem);
  uint16_t* tile = reinterpret_cast<uint16_t*>(smem);
  const int t = threadIdx.x;
  const int c8 = t % S::TPR;  // 8-column group of the loads
  const int rg = t / S::TPR;  // row within a load step
  const int warp = t >> 5;
  const int lane = t & 31;
  const int nslab = (N + QC - 1) / QC;
  for (int slab = blockIdx.x; slab < E * nslab; slab += gridDim.x) {
    const int e = slab / nslab;
    const int n0 = (slab - e * nslab) * QC;
    const uint16_t* We = W + static_cast<size_t>(e) * K * N + n0 + 8 * c8;
    const bool col_ok = n0 + 8 * c8 < N;  // N is a multiple of 8: whole groups

    // ---- pass 1: column amax
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = 0.f;
    if (col_ok) {
#pragma unroll 8
      for (int k = rg; k < K; k += S::RSTEP) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(We + static_cast<size_t>(k) * N));
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          m[2 * j] = fmaxf(m[2 * j], fabsf(bf16_lo(u[j])));
          m[2 * j + 1] = fmaxf(m[2 * j + 1], fabsf(bf16_hi(u[j])));
        }
      }
    }
    __syncthreads();  // the previous slab's pass 2 is done with the buffer
#pragma unroll
    for (int i = 0; i < 8; ++i) red[rg * (QC + 1) + 8 * c8 + i] = m[i];
    __syncthreads();
    if (t < QC) {
      float a = 0.f;
      for (int r = 0; r < S::RSTEP; ++r) a = fmaxf(a, red[r * (QC + 1) + t]);
      const float sc = scale_of(a);
      s_col[t] = sc;
      if (n0 + t < N) scale[static_cast<size_t>(e) * N + n0 + t] = sc;
    }
    __syncthreads();

    // ---- pass 2: quantise and transpose, CHUNK rows at a time
    const int wc = lane + 32 * (warp % (QC / 32));  // column of the slab
    const int seg = warp / (QC / 32);               // 32-row segment of the chunk
    const int n = n0 + wc;
    const float sc = s_col[wc];
    const size_t orow = static_cast<size_t>(e) * rows_per_e + (n / 128) * group_stride +
                        slot * 128 + n % 128;
    uint4 v[S::LOADS];
    auto load_chunk = [&](int k0) {
#pragma unroll
      for (int j = 0; j < S::LOADS; ++j) {
        const int k = k0 + S::RSTEP * j + rg;
        v[j] = (col_ok && k < K)
                   ? __ldg(reinterpret_cast<const uint4*>(We + static_cast<size_t>(k) * N))
                   : make_uint4(0, 0, 0, 0);
      }
    };
    load_chunk(0);
    for (int k0 = 0; k0 < K; k0 += S::CHUNK) {
#pragma unroll
      for (int j = 0; j < S::LOADS; ++j)
        *reinterpret_cast<uint4*>(tile + (S::RSTEP * j + rg) * S::PITCH + 8 * c8) = v[j];
      __syncthreads();
      if (k0 + S::CHUNK < K) load_chunk(k0 + S::CHUNK);  // in flight during the writes
      const int kk = k0 + 32 * seg;
      if (n < N && kk < K) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint16_t* col = tile + (32 * seg + 4 * i) * S::PITCH + wc;
          const float x0 = __uint_as_float(static_cast<uint32_t>(col[0]) << 16);
          const float x1 = __uint_as_float(static_cast<uint32_t>(col[S::PITCH]) << 16);
          const float x2 = __uint_as_float(static_cast<uint32_t>(col[2 * S::PITCH]) << 16);
          const float x3 = __uint_as_float(static_cast<uint32_t>(col[3 * S::PITCH]) << 16);
          w[i] = q2(x0, x1, sc) | (q2(x2, x3, sc) << 16);
        }
        uint4* dst = reinterpret_cast<uint4*>(q + orow * K + kk);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
      __syncthreads();
    }
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
                              cudaStream_t s, const int32_t* nvalid, const float* amax_part,
                              int nt, uint16_t* copy, const uint16_t* in1, uint8_t* q1,
                              int* status) {
  if (rows == 0) return cudaSuccess;
  const int n8 = n / 8;
  const int need = (n8 + kQrThreads - 1) / kQrThreads;
  if (need <= kQrMaxNpt) {
    const int npt = need <= 2 ? need : (need <= 4 ? 4 : (need <= 7 ? 7 : 8));
    const long long cap = static_cast<long long>(num_sms) * 8;
    const int grid = static_cast<int>(rows < cap ? rows : cap);
    const uint4* i4 = reinterpret_cast<const uint4*>(in);
    const uint4* i14 = reinterpret_cast<const uint4*>(in1);
    uint2* q2p = reinterpret_cast<uint2*>(q);
    uint2* q12p = reinterpret_cast<uint2*>(q1);
    uint4* c4 = reinterpret_cast<uint4*>(copy);
#define MOE_QR(NPT_)                                                                         \
  if (npt == NPT_) {                                                                        \
    if (in1)                                                                                \
      quant_rows_reg_kernel<NPT_, true><<<grid, kQrThreads, 0, s>>>(                        \
          i4, idx, div, rows, src_rows, nvalid, n8, q2p, scale, amax_part, nt, c4, i14, q12p, \
          status);                                                                          \
    else                                                                                    \
      quant_rows_reg_kernel<NPT_, false><<<grid, kQrThreads, 0, s>>>(                       \
          i4, idx, div, rows, src_rows, nvalid, n8, q2p, scale, amax_part, nt, c4, i14, q12p, \
          status);                                                                          \
    return launched();                                                                      \
  }
    MOE_QR(1) MOE_QR(2) MOE_QR(4) MOE_QR(7) MOE_QR(8)
#undef MOE_QR
  }
  quant_rows_kernel<<<grid_rows(rows, num_sms), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(in), idx, div, rows, src_rows, nvalid, n / 8,
      reinterpret_cast<uint2*>(q), scale, amax_part, nt, reinterpret_cast<uint4*>(copy),
      reinterpret_cast<const uint4*>(in1), reinterpret_cast<uint2*>(q1), status);
  return launched();
}

// Slab width of the weight quantiser.  Measured on GB300 (Mixtral-8x7B-shaped
// weights, E = 8): W2 (K = 14336) took 0.59-0.60 ms with 32-column slabs
// against 0.64 with 64; W1 and W3 (K = 4096) took 0.52 with 64 against 0.56
// with 32.  MOE_QC_COLS=32 or =64 forces one width (for measurement).
int qc_cols(int K) {
  static const int forced = [] {
    const char* e = getenv("MOE_QC_COLS");
    return e ? atoi(e) : 0;
  }();
  if (forced == 32 || forced == 64) return forced;
  return K > 8192 ? 32 : 64;
}

cudaError_t launch_quant_cols(const uint16_t* W, int E, int K, int N, int rows_per_e,
                              int group_stride, int slot, uint8_t* q, float* scale, int num_sms,
                              cudaStream_t s) {
  if (E == 0 || K == 0 || N == 0) return cudaSuccess;
  const int qc = qc_cols(K);
  const int slabs = E * ((N + qc - 1) / qc);
  const int grid = slabs < 2 * num_sms ? slabs : 2 * num_sms;  // two blocks per SM
  if (qc == 32)
    quant_cols_kernel<32><<<grid, kQcThreads, 0, s>>>(W, E, K, N, rows_per_e, group_stride,
                                                      slot, q, scale);
  else
    quant_cols_kernel<64><<<grid, kQcThreads, 0, s>>>(W, E, K, N, rows_per_e, group_stride,
                                                      slot, q, scale);
  return launched();
}

}  // namespace moe
