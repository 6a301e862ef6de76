// kernels.cuh -- launchers of the memory-bound and FP32 kernels of the layer:
// router, dispatch (histogram, scan, stable scatter), row moves, combine and
// the router/token backward.  All are deterministic and use no atomics on the
// data path (an index error is recorded with one compare-and-swap).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

// Kernels launched so far by the calling host thread.  Every launcher calls
// launched() right after each of its kernel launches: it counts the launch
// and returns cudaGetLastError().
long long kernel_launches();
cudaError_t launched();
// Test hook: the n-th launch from now on this thread reports
// cudaErrorLaunchFailure from launched() (the kernel itself runs); n <= 0 clears.
void fail_launch_after(int n);

// The code a kernel records in its status word when an index it reads from
// device memory (an expert id, a permutation entry) is outside its range.
// The kernel skips that element (a zero row, a slot that adds nothing, an
// assignment that is not placed) instead of reading or writing out of bounds.
// The first error sticks: the word changes only while it is still 0.
constexpr int kStatusDeviceIndex = 6;
#ifdef __CUDACC__
__device__ __forceinline__ void report_bad_index(int* status) {
  if (status) atomicCAS(status, 0, kStatusDeviceIndex);
}
#endif

// Status word of the calls that take no workspace (moe_combine,
// moe_unpermute): one int per device, in this library's device memory.
// Returns its device address for the current device (NULL if the lookup
// fails); the first call on a device looks the address up.
int* nows_status_word();

// cudaFuncSetAttribute(kern, MaxDynamicSharedMemorySize, bytes) on the
// current device, done once per (kernel, device) and size.  Launch settings
// are per device, so a process that drives several GPUs sets them on each;
// safe to call from several host threads.
cudaError_t set_smem_once(const void* kern, int bytes);

constexpr int kDispatchChunk = 1024;  // assignments per dispatch block
constexpr int kRouterMaxE = 64;

inline int dispatch_blocks(long long assignments) {
  return static_cast<int>((assignments + kDispatchChunk - 1) / kDispatchChunk);
}

// Router + softmax + top-k + renormalisation.  `partial` is scratch of
// router_partial_bytes(T, h, E) bytes (may be NULL when that is 0).
size_t router_partial_bytes(int T, int h, int E);
cudaError_t launch_router(const uint16_t* x, const float* Wg, const float* b, int T, int h, int E,
                          int k, int32_t* topk_idx, float* gates, float* partial, int num_sms,
                          cudaStream_t s);

// Which assignments dispatch keeps: experts [e_lo, e_lo + count) and at most
// `capacity` per expert (in assignment order).  Dropless: {0, E, INT_MAX}.
struct DispatchSel {
  int e_lo;
  int count;
  int capacity;
};

// Per-block expert counts [nblk, count] of the assignments.
cudaError_t launch_dispatch_hist(const int32_t* topk_idx, long long n, int E,
                                 const DispatchSel& sel, int32_t* blk_counts, cudaStream_t s,
                                 int* status = nullptr);
// counts [count] (kept), offsets [count + 1] and block rank bases [nblk, count].
cudaError_t launch_dispatch_scan(const int32_t* blk_counts, int nblk, const DispatchSel& sel,
                                 int32_t* counts, int32_t* offsets, int32_t* bases,
                                 cudaStream_t s);
// perm_dst[a] (-1 when dropped), perm_src[p] from bases, offsets and in-block ranks.
cudaError_t launch_dispatch_scatter(const int32_t* topk_idx, long long n, int E,
                                    const DispatchSel& sel, const int32_t* bases,
                                    const int32_t* offsets, int32_t* perm_src, int32_t* perm_dst,
                                    cudaStream_t s, int* status = nullptr);

// out[p] = in[idx[p] / div] for p < rows (bf16 rows of h elements), and only
// for p < *nvalid when nvalid is given; idx < 0 gives a zero row.  `in` has
// src_rows rows; a source index past them gives a zero row and records
// kStatusDeviceIndex in *status.  With gsrc and gdst, also
// gdst[p] = gsrc[idx[p]] (0 where the row is zero).
cudaError_t launch_gather_rows(const uint16_t* in, const int32_t* idx, int div, long long rows,
                               long long src_rows, int h, uint16_t* out, int num_sms,
                               cudaStream_t s, const int32_t* nvalid = nullptr,
                               const float* gsrc = nullptr, float* gdst = nullptr,
                               int* status = nullptr);
// e4m3 quantisation (fp8.cu).  Rows: q[p] = e4m3(in[src] / scale[p]) with
// scale[p] = amax(|in[src]|) / 448 (1 for a zero row), src = idx[p] / div (p
// when idx is NULL), for p < rows (and p < *nvalid when given); n elements per
// row, q row stride n bytes.
// With amax_part [rows, nt] (fp32 partial maxima of |row|), the amax is taken
// from it, rounded to bf16, and the row is read once.  With copy, the bf16
// source rows are also written to copy [rows, n] (a fused permute).  With in1
// and q1, the same rows of in1 are quantised into q1 with a shared per-row
// scale (amax over both rows).
cudaError_t launch_quant_rows(const uint16_t* in, const int32_t* idx, int div, long long rows,
                              long long src_rows, int n, uint8_t* q, float* scale, int num_sms,
                              cudaStream_t s, const int32_t* nvalid = nullptr,
                              const float* amax_part = nullptr, int nt = 0,
                              uint16_t* copy = nullptr, const uint16_t* in1 = nullptr,
                              uint8_t* q1 = nullptr, int* status = nullptr);
// Columns of expert weights W [E, K, N]: scale[e, n] = amax_k |W[e, k, n]| / 448;
// codes written K-major to row e * rows_per_e + (n / 128) * group_stride +
// slot * 128 + n % 128 of q (K bytes per row).
cudaError_t launch_quant_cols(const uint16_t* W, int E, int K, int N, int rows_per_e,
                              int group_stride, int slot, uint8_t* q, float* scale, int num_sms,
                              cudaStream_t s);
// One bounded mbarrier wait that cannot complete: records status 5 after limit_ns.
cudaError_t launch_wait_timeout_probe(int* status, unsigned long long limit_ns, cudaStream_t s);
// dg[perm_src[p]] = sum_{i < nt} part[p * nt + i] for p < *nvalid (fixed order).
cudaError_t launch_dg_reduce(const float* part, int nt, const int32_t* perm_src, long long rows,
                             const int32_t* nvalid, float* dg, int num_sms, cudaStream_t s,
                             int* status = nullptr);

// y[t] = sum_j g[t,j] O[perm_dst[t*k+j]].
cudaError_t launch_combine(const uint16_t* O, const float* gates, const int32_t* perm_dst, int T,
                           int k, int h, uint16_t* y, int num_sms, cudaStream_t s,
                           int* status = nullptr);

// dO[p] = bf16(g[a] dy[t]), dg[a] = <dy[t], O[p]> with a = perm_src[p], t = a / k.
cudaError_t launch_bwd_prep(const uint16_t* dy, const uint16_t* O, const float* gates,
                            const int32_t* perm_src, long long rows, int k, int h, uint16_t* dO,
                            float* dg, int num_sms, cudaStream_t s,
                            const int32_t* nvalid = nullptr, int* status = nullptr);

// WgT[e][i] = Wg[i][e].
cudaError_t launch_transpose_wg(const float* Wg, int h, int E, float* WgT, cudaStream_t s);

// dl (dense [T, E]) and dx[t] = sum_j dX_perm[perm_dst[t*k+j]] + sum_j dl_j WgT[e_j].
cudaError_t launch_token_grad(const float* dX_perm, const int32_t* perm_dst,
                              const int32_t* topk_idx, const float* gates, const float* dg,
                              const float* WgT, int T, int k, int h, int E, float* dl,
                              uint16_t* dx, int num_sms, cudaStream_t s, int* status = nullptr);

// Expert offsets handed in by the caller: records kStatusDeviceIndex in
// *status unless 0 = offsets[0] <= offsets[1] <= ... <= offsets[E] <= rows.
// (The matmuls clamp them into that shape either way.)
cudaError_t launch_check_offsets(const int32_t* offsets, int E, long long rows, int* status,
                                 cudaStream_t s);

// dWg = x^T dl via fixed-order partial sums over token chunks (`partial`
// holds wgrad_router_chunks(T, h, E) * h * E floats).
int wgrad_router_chunks(int T, int h, int E);
cudaError_t launch_router_wgrad(const uint16_t* x, const float* dl, int T, int h, int E,
                                float* partial, float* dWg, cudaStream_t s);

}  // namespace moe
