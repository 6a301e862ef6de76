// kernels.cu -- router, dispatch, row-move, combine and router-backward kernels.
//
// Everything here is HBM- or FP32-bound; none of it uses tensor cores.  Every
// reduction has a fixed order and no kernel uses atomics, so results are
// bitwise reproducible run to run.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <type_traits>
#include <utility>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {
thread_local long long g_launches = 0;
thread_local long long g_fail_at = -1;  // launch count that reports a failure (test hook)
}  // namespace

long long kernel_launches() { return g_launches; }

void fail_launch_after(int n) { g_fail_at = n > 0 ? g_launches + n : -1; }

cudaError_t launched() {
  ++g_launches;
  const cudaError_t e = cudaGetLastError();
  if (g_fail_at >= 0 && g_launches == g_fail_at) {
    g_fail_at = -1;
    return e != cudaSuccess ? e : cudaErrorLaunchFailure;
  }
  return e;
}
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4& q, float* v) {
  v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x);
  v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
  v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z);
  v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  return make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Blocks of `threads` threads of `kern` that fit on one SM at once, looked up
// once per (kernel, device).
int resident_blocks(const void* kern, int threads) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find({kern, dev});
  if (it != cache.end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, 0) != cudaSuccess || n < 1)
    n = 1;
  cache[{kern, dev}] = n;
  return n;
}

int grid_for(long long warps_needed, int num_sms, int warps_per_block, int blocks_per_sm) {
  long long blocks = (warps_needed + warps_per_block - 1) / warps_per_block;
  long long cap = static_cast<long long>(num_sms) * blocks_per_sm;
  if (blocks > cap) blocks = cap;
  return blocks < 1 ? 1 : static_cast<int>(blocks);
}

// ------------------------------------------------------------------ router
// E <= 8: router_a1_kernel holds all of Wg in shared memory (h <= 4096) and
// routes every token in one launch; for longer h, router_a_kernel stages one
// chunk of the router weights per block.  E > 8: router_c_kernel, a tiled
// fp32 GEMM split over h.  Split launches write fp32 partial logits
// [chunk][T][EP] that router_select_warp_kernel adds in chunk order.

// top-k of l[0..E) (descending, ties to the lower id) and renormalised gates
// exp(l_j - l_top) / sum over the selected.
template <int EP>
__device__ __forceinline__ void select_topk(const float (&l)[EP], int E, int k, int32_t* idx_out,
                                            float* gate_out) {
  uint64_t taken = 0;
  float sel_l[8];
  int sel_e[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= k) break;
    int best = -1;
    float bv = 0.f;
#pragma unroll
    for (int e = 0; e < EP; ++e) {
      if (e < E && !((taken >> e) & 1ull) && (best < 0 || l[e] > bv)) {
        best = e;
        bv = l[e];
      }
    }
    if (best < 0) {  // only when logits are NaN: keep the index in range
      best = 0;
      while (best < E - 1 && ((taken >> best) & 1ull)) ++best;
      bv = l[0];
    }
    taken |= 1ull << best;
    sel_e[j] = best;
    sel_l[j] = bv;
  }
  float sj[8];
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= k) break;
    sj[j] = expf(sel_l[j] - sel_l[0]);
    sum += sj[j];
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j >= k) break;
    idx_out[j] = sel_e[j];
    gate_out[j] = sj[j] / sum;
  }
}

// ---- E <= 8: lanes split the columns (8-element slices); each lane keeps
// all 8 partial logits of TOK tokens and reads its rows of the weights as
// conflict-free 16-byte loads from a padded layout (lane l's eight rows are
// one block + 16 bytes).  Within a slice the weights are stored by column
// pair, expert, column: a bf16x2 word of x (two adjacent columns) and the two
// weights of one expert for those columns form the operands of one packed
// fp32x2 FMA, which keeps separate sums for even and odd columns (added at
// the end).  x streams through a ring of NSTAGE shared-memory stages filled
// with cp.async (256 columns of the block's tokens each; every warp copies
// and reads only its own tokens' rows, so a stage needs no block barrier), so
// several steps of loads are in flight without holding registers.  A
// butterfly gives every lane the full logits.
constexpr int kRouterAThreads = 384;
constexpr int kRouterATok = 4;                      // tokens per warp
constexpr int kRouterATile = kRouterAThreads / 32 * kRouterATok;  // tokens per block tile
constexpr int kRouterACh = 2048;                    // columns per weight chunk
constexpr int kRouterASlice = 8 * 8 + 4;
constexpr int kRouterAStage = kRouterATile * 256;   // bf16 per x stage (24 KiB)
constexpr int kRouterANStage = 3;
constexpr int kRouterASmem =
    (kRouterACh / 8) * kRouterASlice * 4 + kRouterANStage * kRouterAStage * 2;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kRouterAThreads, 1) router_a_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ Wg, const float* __restrict__ b,
    int T, int h, int E, int k, int nch, int32_t* __restrict__ topk_idx,
    float* __restrict__ gates, float* __restrict__ partial) {
  constexpr int EP = 8, TOK = kRouterATok, TILE = kRouterATile, CH = kRouterACh;
  constexpr int SLICE = kRouterASlice, NST = kRouterANStage;
  extern __shared__ float sw[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(sw + (CH / 8) * SLICE);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int c = blockIdx.x % nch;
  const int sub = blockIdx.x / nch;
  const int bpc = gridDim.x / nch;
  const int c0 = c * CH;
  const int rows = min(CH, h - c0);
  const int nsteps = (rows + 255) / 256;  // 256-column steps of a tile
  // this block's tiles, flattened with their steps into one stream of stages
  const int ntiles = (T + TILE - 1) / TILE;
  const int my_tiles = sub < ntiles ? (ntiles - sub + bpc - 1) / bpc : 0;
  const int total = my_tiles * nsteps;
  auto issue = [&](int g) {  // stage g -> ring slot g % NST
    if (g < total) {
      const int t0 = (sub + (g / nsteps) * bpc) * TILE;
      const int cs = (g % nsteps) * 256;
      const uint32_t base = smem_addr(xs + (g % NST) * kRouterAStage);
      // each warp copies (and later reads) only its own TOK tokens' rows
#pragma unroll
      for (int i = 0; i < TOK; ++i) {
        const int tok = warp * TOK + i;
        const int t = t0 + tok;
        const bool ok = t < T && cs + 8 * lane < rows;
        const uint16_t* src = ok ? x + static_cast<size_t>(t) * h + c0 + cs + 8 * lane : x;
        cp_async16(base + (tok * 256 + 8 * lane) * 2, src, ok);
      }
    }
    cp_async_commit();  // an empty group keeps the group count uniform
  };
#pragma unroll
  for (int g = 0; g < NST - 1; ++g) issue(g);
  // the weights are staged while the first x stages are in flight
  if (E == EP) {
    // a column pair per thread: two 32-byte rows in, four interleaved float4 out
    for (int lr = 2 * threadIdx.x; lr < rows; lr += 2 * kRouterAThreads) {
      const float4* src = reinterpret_cast<const float4*>(Wg + static_cast<size_t>(c0 + lr) * EP);
      const float4 a0 = __ldg(src), a1 = __ldg(src + 1), b0 = __ldg(src + 2), b1 = __ldg(src + 3);
      float4* dst = reinterpret_cast<float4*>(sw + (lr >> 3) * SLICE + ((lr & 7) >> 1) * (2 * EP));
      dst[0] = make_float4(a0.x, b0.x, a0.y, b0.y);
      dst[1] = make_float4(a0.z, b0.z, a0.w, b0.w);
      dst[2] = make_float4(a1.x, b1.x, a1.y, b1.y);
      dst[3] = make_float4(a1.z, b1.z, a1.w, b1.w);
    }
  } else {
    for (int q = threadIdx.x; q < rows * EP; q += kRouterAThreads) {
      const int lr = q / EP;
      const int e = q - lr * EP;
      sw[(lr >> 3) * SLICE + ((lr & 7) >> 1) * (2 * EP) + 2 * e + (lr & 1)] =
          (e < E) ? __ldg(Wg + static_cast<size_t>(c0 + lr) * E + e) : 0.f;
    }
  }
  __syncthreads();  // weights staged

  float2 acc2[TOK][EP];  // (even-column, odd-column) partial sums
  for (int g = 0; g < total; ++g) {
    issue(g + NST - 1);
    cp_async_wait<NST - 1>();
    __syncwarp();  // stage g landed for every lane's copies (the warp's own rows)
    const int step = g % nsteps;
    if (step == 0) {
#pragma unroll
      for (int u = 0; u < TOK; ++u)
#pragma unroll
        for (int e = 0; e < EP; ++e) acc2[u][e] = make_float2(0.f, 0.f);
    }
    const int lc = step * 256 + 8 * lane;
    if (lc < rows) {
      const uint16_t* xt = xs + (g % NST) * kRouterAStage + (warp * TOK) * 256 + 8 * lane;
      uint4 xq[TOK];
#pragma unroll
      for (int u = 0; u < TOK; ++u) xq[u] = *reinterpret_cast<const uint4*>(xt + u * 256);
      const float4* wb = reinterpret_cast<const float4*>(sw + (lc >> 3) * SLICE);
#pragma unroll
      for (int j2 = 0; j2 < 4; ++j2) {  // column pairs of the lane's slice
        float2 xp[TOK];                 // (column 2 j2, column 2 j2 + 1) of each token
#pragma unroll
        for (int u = 0; u < TOK; ++u) {
          const uint32_t w = j2 == 0 ? xq[u].x : j2 == 1 ? xq[u].y : j2 == 2 ? xq[u].z : xq[u].w;
          xp[u] = make_float2(bf16_lo(w), bf16_hi(w));
        }
#pragma unroll
        for (int e2 = 0; e2 < EP / 2; ++e2) {  // the same columns' weights of experts 2 e2, 2 e2 + 1
          const float4 w4 = wb[j2 * (EP / 2) + e2];
          const float2 wa = make_float2(w4.x, w4.y);
          const float2 wc = make_float2(w4.z, w4.w);
#pragma unroll
          for (int u = 0; u < TOK; ++u) {
            acc2[u][2 * e2] = __ffma2_rn(xp[u], wa, acc2[u][2 * e2]);
            acc2[u][2 * e2 + 1] = __ffma2_rn(xp[u], wc, acc2[u][2 * e2 + 1]);
          }
        }
      }
    }
    __syncwarp();  // every lane is done with slot g before it is refilled
    if (step == nsteps - 1) {
      float acc[TOK][EP];
#pragma unroll
      for (int u = 0; u < TOK; ++u)
#pragma unroll
        for (int e = 0; e < EP; ++e) {
          acc[u][e] = acc2[u][e].x + acc2[u][e].y;
#pragma unroll
          for (int off = 16; off > 0; off >>= 1)
            acc[u][e] += __shfl_xor_sync(kFull, acc[u][e], off);
        }
      const int tw = (sub + (g / nsteps) * bpc) * TILE + warp * TOK;
#pragma unroll
      for (int u = 0; u < TOK; ++u) {
        const int t = tw + u;
        if (lane != u || t >= T) continue;
        if (nch == 1) {
          float l[EP];
#pragma unroll
          for (int e = 0; e < EP; ++e) l[e] = (e < E) ? acc[u][e] + (b ? __ldg(b + e) : 0.f) : 0.f;
          select_topk<EP>(l, E, k, topk_idx + static_cast<size_t>(t) * k,
                          gates + static_cast<size_t>(t) * k);
        } else {
          float4* dst = reinterpret_cast<float4*>(partial + (static_cast<size_t>(c) * T + t) * EP);
          dst[0] = make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
          dst[1] = make_float4(acc[u][4], acc[u][5], acc[u][6], acc[u][7]);
        }
      }
    }
  }
  cp_async_wait<0>();
}

// ---- E <= 8 with the whole of Wg in shared memory (h <= kRouterA1MaxH): one
// launch routes every token, with no partial logits and no select kernel.
// Work items are TOK tokens, dealt round-robin to all warps of the grid; TOK
// is picked at launch so that T / TOK items spread evenly over the warps.
// Within an item the lanes split the columns (8 per lane per 256-column
// step) and keep all TOK x 8 partial logits, as in router_a_kernel: a bf16x2
// word of x and two weights of one expert feed one packed fp32x2 FMA.  Each
// warp streams its item's x through its own ring of NST cp.async stages, so
// it needs warp-level syncs only.  At the end of an item a reduce-scatter
// over the lanes (5 exchange rounds on halving halves, 62 shuffles instead of
// 320 for a full butterfly) leaves lane l with sums 2l and 2l + 1 of the
// TOK x 8 (token, expert) logits; they meet in shared memory, where lane u
// selects token u's top-k.
constexpr int kRouterA1Step = 256;  // columns per stage
constexpr int kRouterA1MaxH = 4096;
constexpr size_t router_a1_smem(int h, int tok, int warps, int nst) {
  return static_cast<size_t>((h + 7) / 8) * kRouterASlice * 4 +
         static_cast<size_t>(warps) * nst * tok * kRouterA1Step * 2 +
         static_cast<size_t>(warps) * 64 * 4;
}

template <int TOK, int WARPS, int NSTAGE>
__global__ void __launch_bounds__(WARPS * 32, 1) router_a1_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ Wg, const float* __restrict__ b,
    int T, int h, int E, int k, int32_t* __restrict__ topk_idx, float* __restrict__ gates) {
  constexpr int kRouterA1Warps = WARPS, kRouterA1Threads = WARPS * 32;
  constexpr int EP = 8, SLICE = kRouterASlice, NST = NSTAGE, SC = kRouterA1Step;
  constexpr int XSTAGE = TOK * SC;  // bf16 per stage of one warp
  extern __shared__ float sw[];
  const int nslice = (h + 7) / 8;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint16_t* xs = reinterpret_cast<uint16_t*>(sw + nslice * SLICE) + warp * NST * XSTAGE;
  float* lg = sw + nslice * SLICE + kRouterA1Warps * NST * XSTAGE / 2 + warp * 64;

  const int nsteps = (h + SC - 1) / SC;
  const int nitems = (T + TOK - 1) / TOK;
  const int gw = blockIdx.x * kRouterA1Warps + warp;
  const int nw = gridDim.x * kRouterA1Warps;
  const int my_items = gw < nitems ? (nitems - gw + nw - 1) / nw : 0;
  const int total = my_items * nsteps;

  // the warp's stream of (item, step) stages; slot g % NST
  int is_item = gw, is_step = 0, is_slot = 0;
  auto issue = [&](int g) {
    if (g < total) {
      const int t0 = is_item * TOK;
      const int c = is_step * SC + 8 * lane;
      const uint32_t base = smem_addr(xs + is_slot * XSTAGE + 8 * lane);
#pragma unroll
      for (int i = 0; i < TOK; ++i) {
        const bool ok = t0 + i < T && c < h;
        const uint16_t* src = ok ? x + static_cast<size_t>(t0 + i) * h + c : x;
        cp_async16(base + i * SC * 2, src, ok);
      }
      if (++is_step == nsteps) {
        is_step = 0;
        is_item += nw;
      }
      if (++is_slot == NST) is_slot = 0;
    }
    cp_async_commit();  // an empty group keeps the group count uniform
  };
#pragma unroll
  for (int g = 0; g < NST - 1; ++g) issue(g);
  // the weights are staged while the first x stages are in flight
  if (E == EP) {
    for (int lr = 2 * threadIdx.x; lr < h; lr += 2 * kRouterA1Threads) {
      const float4* src = reinterpret_cast<const float4*>(Wg + static_cast<size_t>(lr) * EP);
      const float4 a0 = __ldg(src), a1 = __ldg(src + 1), b0 = __ldg(src + 2), b1 = __ldg(src + 3);
      float4* dst = reinterpret_cast<float4*>(sw + (lr >> 3) * SLICE + ((lr & 7) >> 1) * (2 * EP));
      dst[0] = make_float4(a0.x, b0.x, a0.y, b0.y);
      dst[1] = make_float4(a0.z, b0.z, a0.w, b0.w);
      dst[2] = make_float4(a1.x, b1.x, a1.y, b1.y);
      dst[3] = make_float4(a1.z, b1.z, a1.w, b1.w);
    }
  } else {
    for (int q = threadIdx.x; q < h * EP; q += kRouterA1Threads) {
      const int lr = q / EP;
      const int e = q - lr * EP;
      sw[(lr >> 3) * SLICE + ((lr & 7) >> 1) * (2 * EP) + 2 * e + (lr & 1)] =
          (e < E) ? __ldg(Wg + static_cast<size_t>(lr) * E + e) : 0.f;
    }
  }
  __syncthreads();  // weights staged

  float2 acc2[TOK][EP];  // (even-column, odd-column) partial sums
  int item = gw, step = 0, slot = 0;
  for (int g = 0; g < total; ++g) {
    issue(g + NST - 1);
    cp_async_wait<NST - 1>();
    __syncwarp();  // stage g landed for every lane's copies (the warp's own rows)
    if (step == 0) {
#pragma unroll
      for (int u = 0; u < TOK; ++u)
#pragma unroll
        for (int e = 0; e < EP; ++e) acc2[u][e] = make_float2(0.f, 0.f);
    }
    const int lc = step * SC + 8 * lane;
    if (lc < h) {
      const uint16_t* xt = xs + slot * XSTAGE + 8 * lane;
      uint4 xq[TOK];
#pragma unroll
      for (int u = 0; u < TOK; ++u) xq[u] = *reinterpret_cast<const uint4*>(xt + u * SC);
      const float4* wb = reinterpret_cast<const float4*>(sw + (lc >> 3) * SLICE);
#pragma unroll
      for (int j2 = 0; j2 < 4; ++j2) {
        float2 xp[TOK];
#pragma unroll
        for (int u = 0; u < TOK; ++u) {
          const uint32_t w = j2 == 0 ? xq[u].x : j2 == 1 ? xq[u].y : j2 == 2 ? xq[u].z : xq[u].w;
          xp[u] = make_float2(bf16_lo(w), bf16_hi(w));
        }
#pragma unroll
        for (int e2 = 0; e2 < EP / 2; ++e2) {
          const float4 w4 = wb[j2 * (EP / 2) + e2];
          const float2 wa = make_float2(w4.x, w4.y);
          const float2 wc = make_float2(w4.z, w4.w);
#pragma unroll
          for (int u = 0; u < TOK; ++u) {
            acc2[u][2 * e2] = __ffma2_rn(xp[u], wa, acc2[u][2 * e2]);
            acc2[u][2 * e2 + 1] = __ffma2_rn(xp[u], wc, acc2[u][2 * e2 + 1]);
          }
        }
      }
    }
    __syncwarp();  // every lane is done with the slot before it is refilled
    if (++slot == NST) slot = 0;
    if (++step == nsteps) {
      // reduce-scatter of v[u * 8 + e] (u < TOK, e < 8; zero-padded to 64)
      float v[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) v[i] = (i / EP < TOK) ? acc2[i / EP][i % EP].x + acc2[i / EP][i % EP].y : 0.f;
#pragma unroll
      for (int sft = 16, n = 64; sft >= 1; sft >>= 1, n >>= 1) {
        const bool upper = (lane & sft) != 0;
        const int half = n / 2;
#pragma unroll
        for (int i = 0; i < half; ++i) {
          const float keep = upper ? v[half + i] : v[i];
          const float give = upper ? v[i] : v[half + i];
          v[i] = keep + __shfl_xor_sync(kFull, give, sft);
        }
      }
      lg[2 * lane] = v[0];  // sums 2 lane and 2 lane + 1
      lg[2 * lane + 1] = v[1];
      __syncwarp();
      const int t = item * TOK + lane;
      if (lane < TOK && t < T) {
        float l[EP];
#pragma unroll
        for (int e = 0; e < EP; ++e)
          l[e] = (e < E) ? lg[lane * EP + e] + (b ? __ldg(b + e) : 0.f) : 0.f;
        select_topk<EP>(l, E, k, topk_idx + static_cast<size_t>(t) * k,
                        gates + static_cast<size_t>(t) * k);
      }
      __syncwarp();  // the scratch is read before the next item overwrites it
      step = 0;
      item += nw;
    }
  }
  cp_async_wait<0>();
}

// ---- E > 8, tiled: the logits are a skinny fp32 GEMM of x [T, h] (bf16) and
// Wg [h, EP], register-blocked on the CUDA cores.  A block computes BM tokens
// x EP experts over one chunk of h; each thread an 8-token x 8-expert tile:
// tokens tm + TMT u (u < 8; interleaved, so the rows a warp reads sit in
// different banks) and experts 8 tn .. 8 tn + 7.  The chunk runs in steps of
// BK = 32 columns through a 2-stage cp.async ring holding the x tile
// [BM][BK] bf16 (rows padded by 16 bytes) and the Wg tile [BK][EP] fp32.  Per
// 8 columns a thread reads its tokens' x as 8 16-byte loads and, per column,
// its experts' weights as 2 16-byte loads: 24 shared-memory loads feed 512
// FMAs.  Each (token, expert) sum runs over the chunk's columns in order; the
// chunks' partial logits [chunk][T][EP] are added in chunk order by
// router_select_warp_kernel.
template <int EP>
struct RouterC {
  static constexpr int TN = EP / 8;                     // threads along the experts
  static constexpr int THREADS = EP == 16 ? 128 : 256;
  static constexpr int TMT = THREADS / TN;              // threads along the tokens
  static constexpr int BM = TMT * 8;                    // tokens per block
  static constexpr int BK = 32;                         // columns per step
  static constexpr int MINB = 2;                        // blocks per SM
  static constexpr int XP = BK + 8;                     // padded x row (bf16)
  static constexpr int XSTAGE = BM * XP;                // bf16 per x stage
  static constexpr int WSTAGE = BK * EP;                // fp32 per Wg stage
  static constexpr int SMEM = 2 * (XSTAGE * 2 + WSTAGE * 4);
};

template <int EP>
__global__ void __launch_bounds__(RouterC<EP>::THREADS, RouterC<EP>::MINB) router_c_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ Wg, int T, int h, int E, int nch,
    float* __restrict__ partial) {
  using S = RouterC<EP>;
  constexpr int BM = S::BM, BK = S::BK, XP = S::XP, TMT = S::TMT, NT = S::THREADS;
  extern __shared__ float sc[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(sc);           // [2][BM][XP]
  float* ws = sc + S::XSTAGE;                                // [2][BK][EP] (after 2 x stages)
  const int tid = threadIdx.x;
  const int tn = tid % S::TN;
  const int tm = tid / S::TN;
  const int c = blockIdx.x % nch;
  const int t0 = (blockIdx.x / nch) * BM;
  // chunk c: BK-column steps [c S / nch, (c + 1) S / nch) of the S = ceil(h / BK)
  const int S_all = (h + BK - 1) / BK;
  const int s0 = static_cast<int>(static_cast<long long>(c) * S_all / nch);
  const int s1 = static_cast<int>(static_cast<long long>(c + 1) * S_all / nch);
  const int k0 = s0 * BK;
  const int kend = min(h, s1 * BK);
  const int nsteps = s1 - s0;

  auto issue = [&](int st) {
    if (st < nsteps) {
      const int kc = k0 + st * BK;
      const int slot = st & 1;
      const uint32_t xb = smem_addr(xs + slot * S::XSTAGE);
      // x tile: BM rows x BK / 8 pieces of 16 bytes
      for (int q = tid; q < BM * (BK / 8); q += NT) {
        const int r = q / (BK / 8), p8 = q % (BK / 8);
        const int t = t0 + r, col = kc + 8 * p8;
        const bool ok = t < T && col < kend;
        const uint16_t* src = ok ? x + static_cast<size_t>(t) * h + col : x;
        cp_async16(xb + (r * XP + 8 * p8) * 2, src, ok);
      }
      // Wg tile: BK rows x EP fp32 (experts past E read as 0)
      if (E % 4 == 0) {
        const uint32_t wb = smem_addr(ws + slot * S::WSTAGE);
        for (int q = tid; q < BK * (EP / 4); q += NT) {
          const int r = q / (EP / 4), e4 = q % (EP / 4);
          const int row = kc + r;
          const bool ok = row < kend && 4 * e4 < E;
          const float* src = ok ? Wg + static_cast<size_t>(row) * E + 4 * e4 : Wg;
          cp_async16(wb + (r * EP + 4 * e4) * 4, src, ok);
        }
      } else {
        // rows of E floats are not 16-byte aligned: plain loads and stores
        // (the slot was last read two steps ago, before the step's barrier)
        float* wd = ws + slot * S::WSTAGE;
        for (int q = tid; q < BK * EP; q += NT) {
          const int r = q / EP, e = q % EP;
          const int row = kc + r;
          wd[q] = (row < kend && e < E) ? __ldg(Wg + static_cast<size_t>(row) * E + e) : 0.f;
        }
      }
    }
    cp_async_commit();
  };

  float acc[8][8];
#pragma unroll
  for (int u = 0; u < 8; ++u)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[u][j] = 0.f;

  issue(0);
  for (int st = 0; st < nsteps; ++st) {
    issue(st + 1);
    cp_async_wait<1>();
    __syncthreads();  // stage st is in shared memory for every thread
    const uint16_t* xt = xs + (st & 1) * S::XSTAGE;
    const float* wt = ws + (st & 1) * S::WSTAGE + 8 * tn;
#pragma unroll
    for (int k8 = 0; k8 < BK / 8; ++k8) {
      uint4 xq[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        xq[u] = *reinterpret_cast<const uint4*>(xt + (tm + TMT * u) * XP + 8 * k8);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const float4 w0 = *reinterpret_cast<const float4*>(wt + (8 * k8 + kk) * EP);
        const float4 w1 = *reinterpret_cast<const float4*>(wt + (8 * k8 + kk) * EP + 4);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t q = kk < 2 ? xq[u].x : kk < 4 ? xq[u].y : kk < 6 ? xq[u].z : xq[u].w;
          const float xv = (kk & 1) ? bf16_hi(q) : bf16_lo(q);
          acc[u][0] = fmaf(xv, w0.x, acc[u][0]);
          acc[u][1] = fmaf(xv, w0.y, acc[u][1]);
          acc[u][2] = fmaf(xv, w0.z, acc[u][2]);
          acc[u][3] = fmaf(xv, w0.w, acc[u][3]);
          acc[u][4] = fmaf(xv, w1.x, acc[u][4]);
          acc[u][5] = fmaf(xv, w1.y, acc[u][5]);
          acc[u][6] = fmaf(xv, w1.z, acc[u][6]);
          acc[u][7] = fmaf(xv, w1.w, acc[u][7]);
        }
      }
    }
    __syncthreads();  // every thread is done with stage st before it is refilled
  }
  cp_async_wait<0>();
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int t = t0 + tm + TMT * u;
    if (t >= T) continue;
    float4* dst = reinterpret_cast<float4*>(partial + (static_cast<size_t>(c) * T + t) * EP + 8 * tn);
    dst[0] = make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
    dst[1] = make_float4(acc[u][4], acc[u][5], acc[u][6], acc[u][7]);
  }
}

template <int EP>
cudaError_t router_c_launch(const uint16_t* x, const float* Wg, int T, int h, int E, int nch,
                            float* partial, cudaStream_t s);

// Chunks of h for a split-K launch of `tiles` output tiles over S k-steps:
// the count with the shortest makespan on a 152-SM GPU at blocks_per_sm blocks per SM,
// modelled as (waves of blocks) x (steps per chunk + 2 steps of prologue and
// epilogue).  A function of the shape only (the workspace is sized from it).
int split_k_chunks(long long tiles, int S, int max_chunks = 32, int blocks_per_sm = 2) {
  const long long slots = static_cast<long long>(blocks_per_sm) * 152;
  int best = 1;
  double best_t = -1.0;
  for (int n = 1; n <= max_chunks && n <= S; ++n) {
    const long long waves = (tiles * n + slots - 1) / slots;
    const double t = static_cast<double>(waves) * (static_cast<double>(S) / n + 2.0);
    if (best_t < 0 || t < best_t - 1e-9) {
      best_t = t;
      best = n;
    }
  }
  return best;
}

template <int EP>
int router_c_nch(int T, int h) {
  const long long tiles = (T + RouterC<EP>::BM - 1) / RouterC<EP>::BM;
  return split_k_chunks(tiles, (h + RouterC<EP>::BK - 1) / RouterC<EP>::BK, 32, RouterC<EP>::MINB);
}

// Warp per token: the logits of token t are the chunks' partials summed in
// chunk order (lane l holds experts l and l + 32), plus b.  The top-k is k
// rounds of a warp arg-max (larger logit first, the lower expert id on ties;
// NaN counts as the smallest value), then lane 0 forms the renormalised gates
// exactly as select_topk does.  The same values as the thread-per-token
// kernel, with the whole warp reading each token's partials.
template <int EP>
__global__ void __launch_bounds__(256) router_select_warp_kernel(
    const float* __restrict__ partial, int nch, const float* __restrict__ b, int T, int E, int k,
    int32_t* __restrict__ topk_idx, float* __restrict__ gates) {
  constexpr int PER = (EP + 31) / 32;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int t = gw; t < T; t += nw) {
    float l[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) l[i] = 0.f;
    for (int c = 0; c < nch; ++c) {
      const float* src = partial + (static_cast<size_t>(c) * T + t) * EP;
#pragma unroll
      for (int i = 0; i < PER; ++i)
        if (lane + 32 * i < EP) l[i] += __ldg(src + lane + 32 * i);
    }
    bool live[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane + 32 * i;
      live[i] = e < E;
      if (live[i] && b) l[i] += __ldg(b + e);
    }
    float sel_l[8];
    int sel_e[8];
    for (int j = 0; j < k; ++j) {
      // this lane's best live candidate
      float bv = -INFINITY;
      int be = 1 << 30;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const float v = isnan(l[i]) ? -INFINITY : l[i];
        const int e = lane + 32 * i;
        if (live[i] && (v > bv || (v == bv && e < be))) {
          bv = v;
          be = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(kFull, bv, off);
        const int oe = __shfl_xor_sync(kFull, be, off);
        if (ov > bv || (ov == bv && oe < be)) {
          bv = ov;
          be = oe;
        }
      }
#pragma unroll
      for (int i = 0; i < PER; ++i)
        if (lane + 32 * i == be) live[i] = false;
      sel_e[j < 8 ? j : 7] = be;
      // the logit itself (NaN kept as NaN, as select_topk would give)
      const int owner = be & 31;
      float lv = 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i)
        if (32 * i <= be && be < 32 * i + 32) lv = l[i];
      sel_l[j < 8 ? j : 7] = __shfl_sync(kFull, lv, owner);
    }
    if (lane == 0) {
      float sj[8];
      float sum = 0.f;
      for (int j = 0; j < k; ++j) {
        sj[j] = expf(sel_l[j] - sel_l[0]);
        sum += sj[j];
      }
      for (int j = 0; j < k; ++j) {
        topk_idx[static_cast<size_t>(t) * k + j] = sel_e[j];
        gates[static_cast<size_t>(t) * k + j] = sj[j] / sum;
      }
    }
  }
}

int router_padded_e(int E) { return E <= 8 ? 8 : E <= 16 ? 16 : E <= 32 ? 32 : 64; }

int router_c_chunks(int T, int h, int ep) {
  return ep == 16 ? router_c_nch<16>(T, h) : ep == 32 ? router_c_nch<32>(T, h) : router_c_nch<64>(T, h);
}


int router_chunks(int T, int h, int E) {
  const int ep = router_padded_e(E);
  if (ep == 8 && h <= kRouterA1MaxH) return 1;  // router_a1_kernel holds all of Wg
  if (ep == 8) return (h + kRouterACh - 1) / kRouterACh;
  return router_c_chunks(T, h, ep);
}

// router_a1_kernel<TOK>: the TOK whose items spread most evenly over the
// grid's warps (fewest token slots on the busiest warp; ties to the larger
// TOK), within the shared-memory limit.
template <int TOK, int WARPS, int NST>
cudaError_t router_a1_launch(const uint16_t* x, const float* Wg, const float* b, int T, int h,
                             int E, int k, int32_t* idx, float* gates, int blocks,
                             cudaStream_t s) {
  const size_t smem = router_a1_smem(h, TOK, WARPS, NST);
  const cudaError_t e = set_smem_once(
      reinterpret_cast<const void*>(router_a1_kernel<TOK, WARPS, NST>), static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  router_a1_kernel<TOK, WARPS, NST><<<blocks, WARPS * 32, smem, s>>>(x, Wg, b, T, h, E, k, idx,
                                                                     gates);
  return launched();
}

// Warps per block and x stages per warp of router_a1_kernel: 8 warps with 3
// stages, or 12 warps (TOK = 4) with MOE_ROUTER_A1=12 for measurement.
void router_a1_shape(int& warps, int& nst) {
  static const int v = [] {
    const char* e = getenv("MOE_ROUTER_A1");
    return (e && e[0] == '1' && e[1] == '2') ? 1 : 0;
  }();
  warps = v == 1 ? 12 : 8;
  nst = 3;
}

cudaError_t router_a1_dispatch(const uint16_t* x, const float* Wg, const float* b, int T, int h,
                               int E, int k, int32_t* idx, float* gates, int num_sms,
                               cudaStream_t s) {
  int warps = 8, nst = 3;
  router_a1_shape(warps, nst);
  const long long nw = static_cast<long long>(num_sms) * warps;
  int best = 4;
  long long best_slots = -1;
  // more warps leave fewer registers a thread: TOK = 4 only (no spills)
  const int tok_max = warps == 8 ? 7 : 4;
  for (int tok = 4; tok <= tok_max; ++tok) {
    if (router_a1_smem(h, tok, warps, nst) > 232448) continue;
    const long long items = (T + tok - 1) / tok;
    const long long slots = (items + nw - 1) / nw * tok;
    if (best_slots < 0 || slots <= best_slots) {
      best = tok;
      best_slots = slots;
    }
  }
  // blocks: enough warps for the items, at most one block per SM
  const long long items = (T + best - 1) / best;
  int blocks = static_cast<int>((items + warps - 1) / warps);
  if (blocks > num_sms) blocks = num_sms;
#define MOE_A1(W, N)                                                                         \
  switch (best) {                                                                            \
    case 4: return router_a1_launch<4, W, N>(x, Wg, b, T, h, E, k, idx, gates, blocks, s);  \
    case 5: return router_a1_launch<5, W, N>(x, Wg, b, T, h, E, k, idx, gates, blocks, s);  \
    case 6: return router_a1_launch<6, W, N>(x, Wg, b, T, h, E, k, idx, gates, blocks, s);  \
    default: return router_a1_launch<7, W, N>(x, Wg, b, T, h, E, k, idx, gates, blocks, s); \
  }
  if (warps == 12) return router_a1_launch<4, 12, 3>(x, Wg, b, T, h, E, k, idx, gates, blocks, s);
  MOE_A1(8, 3)
#undef MOE_A1
}

template <int EP>
cudaError_t router_c_launch(const uint16_t* x, const float* Wg, int T, int h, int E, int nch,
                            float* partial, cudaStream_t s) {
  using S = RouterC<EP>;
  const cudaError_t e = set_smem_once(reinterpret_cast<const void*>(router_c_kernel<EP>), S::SMEM);
  if (e != cudaSuccess) return e;
  const long long tiles = (T + S::BM - 1) / S::BM;
  router_c_kernel<EP><<<static_cast<int>(tiles * nch), S::THREADS, S::SMEM, s>>>(x, Wg, T, h, E,
                                                                                 nch, partial);
  return launched();
}

template <int EP>
cudaError_t router_select_launch(const float* partial, int nch, const float* b, int T, int E,
                                 int k, int32_t* idx, float* gates, int num_sms, cudaStream_t s) {
  const int grid = grid_for(T, num_sms, 8, 16);
  router_select_warp_kernel<EP><<<grid, 256, 0, s>>>(partial, nch, b, T, E, k, idx, gates);
  return launched();
}

// ---------------------------------------------------------------- dispatch
// A block takes kDispatchChunk consecutive assignments in four rounds of 256.
// Within a round a warp groups equal experts with __match_any_sync; the
// group's lowest lane records the group size.  The stable rank of an
// assignment among its expert's assignments is then
//   bases[block][e] (earlier blocks) + running[e] (earlier rounds)
//   + sizes of earlier warps (this round) + lanes below it in its own group.
// An assignment is kept when its expert lies in the local range
// [e_lo, e_lo + EL) and its rank is below `cap`; kept ones go to permuted row
// offsets[e] + rank, the others get perm_dst = -1.  An expert id outside
// [0, E) is recorded in *status and the assignment is not placed.
constexpr int kDispThreads = 256;
constexpr int kDispWarps = kDispThreads / 32;
constexpr int kDispMaxE = 256;

template <bool WRITE>
__global__ void __launch_bounds__(kDispThreads) dispatch_kernel(
    const int32_t* __restrict__ topk_idx, long long n, int E, int e_lo, int EL, int cap,
    int32_t* __restrict__ blk_counts, const int32_t* __restrict__ bases,
    const int32_t* __restrict__ offsets, int32_t* __restrict__ perm_src,
    int32_t* __restrict__ perm_dst, int* __restrict__ status) {
  __shared__ int running[kDispMaxE];
  __shared__ int wc[kDispWarps][kDispMaxE];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const long long base = static_cast<long long>(blockIdx.x) * kDispatchChunk;
  for (int e = tid; e < EL; e += kDispThreads) running[e] = 0;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int r = 0; r < kDispatchChunk / kDispThreads; ++r) {
    for (int i = tid; i < kDispWarps * EL; i += kDispThreads) wc[i / EL][i % EL] = 0;
    __syncthreads();
    const long long a = base + r * kDispThreads + tid;
    const bool valid = a < n;
    int le = -1;  // local expert, -1 = not placed
    if (valid) {
      const int e = __ldg(topk_idx + a);
      if (e < 0 || e >= E) {
        // an expert id out of range: reported (once, by the histogram pass)
        // and not placed
        if (!WRITE) report_bad_index(status);
      } else {
        le = (e >= e_lo && e < e_lo + EL) ? e - e_lo : -1;
      }
    }
    const unsigned grp = __match_any_sync(kFull, le);
    const int lrank = __popc(grp & lt_mask);
    if (le >= 0 && lrank == 0) wc[warp][le] = __popc(grp);
    __syncthreads();
    if (valid && WRITE) {
      int dst = -1;
      if (le >= 0) {
        int rank = __ldg(bases + static_cast<size_t>(blockIdx.x) * EL + le) + running[le] + lrank;
        for (int w = 0; w < warp; ++w) rank += wc[w][le];
        if (rank < cap) dst = __ldg(offsets + le) + rank;
      }
      perm_dst[a] = dst;
      if (dst >= 0) perm_src[dst] = static_cast<int32_t>(a);
    }
    __syncthreads();
    for (int ee = tid; ee < EL; ee += kDispThreads) {
      int add = 0;
      for (int w = 0; w < kDispWarps; ++w) add += wc[w][ee];
      running[ee] += add;
    }
  }
  if (!WRITE) {
    __syncthreads();
    for (int e = tid; e < EL; e += kDispThreads)
      blk_counts[static_cast<size_t>(blockIdx.x) * EL + e] = running[e];
  }
}

// counts[e] = min(assignments of e, cap); offsets = exclusive scan of counts;
// bases[b][e] = assignments of e in blocks before b (ranks, not rows).
__global__ void __launch_bounds__(256) dispatch_scan_kernel(const int32_t* __restrict__ blk_counts,
                                                            int nblk, int EL, int cap,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ bases) {
  __shared__ int tot[kDispMaxE + 1];
  for (int e = threadIdx.x; e < EL; e += blockDim.x) {
    int s = 0;
    for (int bk = 0; bk < nblk; ++bk) {
      bases[static_cast<size_t>(bk) * EL + e] = s;
      s += blk_counts[static_cast<size_t>(bk) * EL + e];
    }
    s = s < cap ? s : cap;
    tot[e] = s;
    counts[e] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int e = 0; e < EL; ++e) {
      offsets[e] = run;
      run += tot[e];
    }
    offsets[EL] = run;
  }
}

// --------------------------------------------------------------- row moves
// Warp per row, 16-byte pieces.
// Rows p < *nvalid (all `rows` when nvalid is NULL); a negative index gives a
// zero row, and so does a source index past src_rows (recorded in *status).
// With gsrc/gdst, also gdst[p] = gsrc[idx[p]] (a value per row).
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ in,
                                                          const int32_t* __restrict__ idx, int div,
                                                          long long rows, long long src_rows,
                                                          const int32_t* __restrict__ nvalid,
                                                          int h8, uint4* __restrict__ out,
                                                          const float* __restrict__ gsrc,
                                                          float* __restrict__ gdst,
                                                          int* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  if (nvalid) {
    const long long nv = __ldg(nvalid);
    rows = nv < rows ? (nv < 0 ? 0 : nv) : rows;
  }
  for (long long p = gw; p < rows; p += nw) {
    const long long i = __ldg(idx + p);
    uint4* d = out + p * h8;
    const long long src = i / div;
    const bool bad = i >= 0 && src >= src_rows;
    if (bad && lane == 0) report_bad_index(status);
    if (gdst && lane == 0) gdst[p] = (i < 0 || bad) ? 0.f : __ldg(gsrc + i);
    if (i < 0 || bad) {
      for (int c = lane; c < h8; c += 32) d[c] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* s = in + src * h8;
#pragma unroll 4
    for (int c = lane; c < h8; c += 32) d[c] = __ldg(s + c);
  }
}

// y[t] = sum_j g[t,j] * O[perm_dst[t*k+j]], fp32 in slot order.  K = k.
// A row index past T*k is recorded in *status and its slot adds nothing.
template <int K>
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ O,
                                                      const float* __restrict__ gates,
                                                      const int32_t* __restrict__ perm_dst, int T,
                                                      int h8, uint4* __restrict__ y,
                                                      int* __restrict__ status) {
  constexpr int k = K;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  for (int t = gw; t < T; t += nw) {
    long long rows[K];
    bool kept[K];
    float g[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      {
        const long long r = __ldg(perm_dst + static_cast<size_t>(t) * k + j);
        const bool bad = r >= static_cast<long long>(T) * k;
        if (bad && lane == 0) report_bad_index(status);
        // a dropped slot (r < 0) adds nothing and reads no row
        kept[j] = r >= 0 && !bad;
        rows[j] = kept[j] ? r : 0;
        g[j] = kept[j] ? __ldg(gates + static_cast<size_t>(t) * k + j) : 0.f;
      }
    }
    // four 16-byte pieces per lane per step: 4 * k loads in flight
    for (int c0 = lane; c0 < h8; c0 += 128) {
      uint4 q[4][K];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + 32 * u;
#pragma unroll
        for (int j = 0; j < K; ++j)
          q[u][j] = (c < h8 && kept[j]) ? __ldg(O + rows[j] * h8 + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + 32 * u;
        if (c >= h8) break;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < K; ++j) {
          float v[8];
          unpack8(q[u][j], v);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] = fmaf(g[j], v[i], acc[i]);
        }
        y[static_cast<size_t>(t) * h8 + c] = pack8(acc);
      }
    }
  }
}

// dO[p] = bf16(g[a] * dy[t]); dg[a] = <dy[t], O[p]>.  An assignment index
// outside [0, rows) is recorded in *status; that row's dO is zero.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint4* __restrict__ dy,
                                                       const uint4* __restrict__ O,
                                                       const float* __restrict__ gates,
                                                       const int32_t* __restrict__ perm_src,
                                                       long long rows,
                                                       const int32_t* __restrict__ nvalid, int k,
                                                       int h8, uint4* __restrict__ dO,
                                                       float* __restrict__ dg,
                                                       int* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const long long total = rows;
  if (nvalid) {
    const long long nv = __ldg(nvalid);
    rows = nv < rows ? (nv < 0 ? 0 : nv) : rows;
  }
  for (long long p = gw; p < rows; p += nw) {
    const int a = __ldg(perm_src + p);
    if (a < 0 || a >= total) {
      if (lane == 0) report_bad_index(status);
      for (int c = lane; c < h8; c += 32) dO[p * h8 + c] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const long long t = a / k;
    const float g = __ldg(gates + a);
    float dot = 0.f;
    for (int c = lane; c < h8; c += 32) {
      float d[8], o[8];
      unpack8(__ldg(dy + t * h8 + c), d);
      unpack8(__ldg(O + p * h8 + c), o);
      float s[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        dot = fmaf(d[i], o[i], dot);
        s[i] = g * d[i];
      }
      dO[p * h8 + c] = pack8(s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(kFull, dot, off);
    if (lane == 0) dg[a] = dot;
  }
}

// dg[perm_src[p]] = sum over nt of part[p, nt], in nt order, for p < *nvalid.
__global__ void __launch_bounds__(256) dg_reduce_kernel(const float* __restrict__ part, int nt,
                                                        const int32_t* __restrict__ perm_src,
                                                        long long rows,
                                                        const int32_t* __restrict__ nvalid,
                                                        float* __restrict__ dg,
                                                        int* __restrict__ status) {
  const long long nv = __ldg(nvalid);
  const long long n = nv < rows ? (nv < 0 ? 0 : nv) : rows;
  for (long long p = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; p < n;
       p += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float* q = part + p * nt;
    float s = 0.f;
    for (int i = 0; i < nt; ++i) s += __ldg(q + i);
    const long long a = __ldg(perm_src + p);
    if (a < 0 || a >= rows) {
      report_bad_index(status);
      continue;
    }
    dg[a] = s;
  }
}

__global__ void transpose_wg_kernel(const float* __restrict__ Wg, int h, int E,
                                    float* __restrict__ WgT) {
  const long long n = static_cast<long long>(h) * E;
  for (long long q = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; q < n;
       q += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long e = q / h;
    const long long i = q - e * h;
    WgT[q] = Wg[i * E + e];
  }
}

// Router backward per token + dx (K = k).  A work item is one token and a
// piece of its row: NSTEP steps of 32 lanes x U 16-byte pieces; U pieces per
// lane per step keep 2 * U * K fp32 loads of dX_perm in flight.  For K <= 2
// an item is two steps, so that the grid's warps finish together (a warp per
// token left some warps one token longer than the rest); for K >= 3 the item
// is the whole row, because there the per-item work (K permutation entries,
// gates and dg, the k x k router gradient) measured slower when repeated per
// piece.  Every item recomputes its token's router gradient; the first item
// of a token writes its dl row.
template <int K>
__global__ void __launch_bounds__(256) token_grad_kernel(
    const float4* __restrict__ dX, const int32_t* __restrict__ perm_dst,
    const int32_t* __restrict__ topk_idx, const float* __restrict__ gates,
    const float* __restrict__ dg, const float4* __restrict__ WgT, int T, int h8, int E,
    float* __restrict__ dl, uint4* __restrict__ dx, int* __restrict__ status) {
  constexpr int U = K <= 2 ? 2 : 1;
  constexpr bool SPLIT = K <= 2;   // items are row pieces of NSTEP steps
  constexpr int NSTEP = 2;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const long long R = static_cast<long long>(T) * K;
  // items per token
  const int per = SPLIT ? (h8 + 32 * U * NSTEP - 1) / (32 * U * NSTEP) : 1;
  using Item = typename std::conditional<SPLIT, long long, int>::type;
  const Item items = static_cast<Item>(T) * per;
  for (Item item = gw; item < items; item += nw) {
    const int t = static_cast<int>(SPLIT ? item / per : item);
    const int cb = SPLIT ? static_cast<int>(item - static_cast<Item>(t) * per) : 0;
    long long rows[K];
    int ex[K];
    bool kept[K];
    float g[K], d[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      const size_t a = static_cast<size_t>(t) * K + j;
      const long long r = __ldg(perm_dst + a);
      const int e = __ldg(topk_idx + a);
      // out-of-range entries are recorded; such a slot adds nothing
      if ((r >= R || e < 0 || e >= E) && lane == 0 && cb == 0) report_bad_index(status);
      kept[j] = r >= 0 && r < R;  // a dropped slot has no expert output: dg = 0, no dX
      rows[j] = kept[j] ? r : 0;
      ex[j] = (e < 0 || e >= E) ? -1 : e;
      g[j] = ex[j] < 0 ? 0.f : __ldg(gates + a);
      d[j] = kept[j] ? __ldg(dg + a) : 0.f;
    }
    // dl_j = g_j (dg_j - sum_i g_i dg_i), evaluated as g_j sum_i g_i (dg_j - dg_i)
    // (sum_i g_i = 1): no cancellation when one gate is close to 1, and
    // exactly 0 for k = 1.
    float dlj[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < K; ++i)
        if (i != j) acc = fmaf(g[i], d[j] - d[i], acc);
      dlj[j] = g[j] * acc;
    }
    if (cb == 0) {
      for (int e = lane; e < E; e += 32) {
        float v = 0.f;
#pragma unroll
        for (int j = 0; j < K; ++j)
          if (ex[j] == e) v = dlj[j];
        dl[static_cast<size_t>(t) * E + e] = v;
      }
    }
    const int cend = SPLIT ? min(h8, (cb + 1) * 32 * U * NSTEP) : h8;
    for (int c0 = cb * 32 * U * NSTEP + lane; c0 < cend; c0 += 32 * U) {
      float4 q[U][K][2];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
#pragma unroll
        for (int j = 0; j < K; ++j) {
          if (c < h8 && kept[j]) {
            q[u][j][0] = __ldg(dX + (rows[j] * h8 + c) * 2);
            q[u][j][1] = __ldg(dX + (rows[j] * h8 + c) * 2 + 1);
          } else {
            q[u][j][0] = make_float4(0.f, 0.f, 0.f, 0.f);
            q[u][j][1] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        if (c >= h8) break;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < K; ++j) {
          acc[0] += q[u][j][0].x; acc[1] += q[u][j][0].y; acc[2] += q[u][j][0].z; acc[3] += q[u][j][0].w;
          acc[4] += q[u][j][1].x; acc[5] += q[u][j][1].y; acc[6] += q[u][j][1].z; acc[7] += q[u][j][1].w;
        }
#pragma unroll
        for (int j = 0; j < K; ++j) {
          if (ex[j] < 0) continue;
          const size_t wo = (static_cast<size_t>(ex[j]) * h8 + c) * 2;
          const float4 w0 = __ldg(WgT + wo);
          const float4 w1 = __ldg(WgT + wo + 1);
          acc[0] = fmaf(dlj[j], w0.x, acc[0]); acc[1] = fmaf(dlj[j], w0.y, acc[1]);
          acc[2] = fmaf(dlj[j], w0.z, acc[2]); acc[3] = fmaf(dlj[j], w0.w, acc[3]);
          acc[4] = fmaf(dlj[j], w1.x, acc[4]); acc[5] = fmaf(dlj[j], w1.y, acc[5]);
          acc[6] = fmaf(dlj[j], w1.z, acc[6]); acc[7] = fmaf(dlj[j], w1.w, acc[7]);
        }
        dx[static_cast<size_t>(t) * h8 + c] = pack8(acc);
      }
    }
  }
}

// dWg = x^T dl as a register-blocked fp32 GEMM on the CUDA cores (M = h
// columns of x, N = EP experts, K = T tokens), split over token chunks.  A
// block computes BM columns x EP experts over one chunk; each thread 8
// consecutive columns x 8 experts.  Tokens run in steps of BK = 16 through a
// 2-stage cp.async ring holding the x tile [BK][BM] bf16 (rows of x as they
// lie in memory) and the dl tile [BK][EP] fp32.  Per token a thread reads its
// 8 columns of x as one 16-byte load and its 8 experts of dl as two: 3 loads
// feed 64 FMAs.  Each (column, expert) sum runs over the chunk's tokens in
// order; router_wgrad_reduce_kernel adds the chunks in order.
template <int EP>
struct WgradC {
  static constexpr int TN = EP / 8;
  static constexpr int THREADS = EP <= 16 ? 128 : 256;
  static constexpr int TMT = THREADS / TN;
  static constexpr int BM = TMT * 8;                 // columns per block
  static constexpr int BK = 16;                      // tokens per step
  static constexpr int XSTAGE = BK * BM;             // bf16
  static constexpr int DSTAGE = BK * EP;             // fp32
  static constexpr int SMEM = 2 * (XSTAGE * 2 + DSTAGE * 4);
};

template <int EP>
__global__ void __launch_bounds__(WgradC<EP>::THREADS, 2) router_wgrad_c_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ dl, int T, int h, int E, int nch,
    float* __restrict__ partial) {
  using S = WgradC<EP>;
  constexpr int BM = S::BM, BK = S::BK, NT = S::THREADS;
  extern __shared__ float wc[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(wc);   // [2][BK][BM]
  float* ds = wc + S::XSTAGE;                        // [2][BK][EP] after the two x stages
  const int tid = threadIdx.x;
  const int tn = tid % S::TN;
  const int tm = tid / S::TN;
  const int c = blockIdx.x % nch;
  const int i0 = (blockIdx.x / nch) * BM;
  const int S_all = (T + BK - 1) / BK;
  const int s0 = static_cast<int>(static_cast<long long>(c) * S_all / nch);
  const int s1 = static_cast<int>(static_cast<long long>(c + 1) * S_all / nch);
  const int nsteps = s1 - s0;

  auto issue = [&](int st) {
    if (st < nsteps) {
      const int tb = (s0 + st) * BK;
      const int slot = st & 1;
      const uint32_t xb = smem_addr(xs + slot * S::XSTAGE);
      for (int q = tid; q < BK * (BM / 8); q += NT) {
        const int r = q / (BM / 8), p8 = q % (BM / 8);
        const int t = tb + r, col = i0 + 8 * p8;
        const bool ok = t < T && col < h;
        const uint16_t* src = ok ? x + static_cast<size_t>(t) * h + col : x;
        cp_async16(xb + (r * BM + 8 * p8) * 2, src, ok);
      }
      if (E % 4 == 0) {
        const uint32_t db = smem_addr(ds + slot * S::DSTAGE);
        for (int q = tid; q < BK * (EP / 4); q += NT) {
          const int r = q / (EP / 4), e4 = q % (EP / 4);
          const int t = tb + r;
          const bool ok = t < T && 4 * e4 < E;
          const float* src = ok ? dl + static_cast<size_t>(t) * E + 4 * e4 : dl;
          cp_async16(db + (r * EP + 4 * e4) * 4, src, ok);
        }
      } else {
        float* dd = ds + slot * S::DSTAGE;
        for (int q = tid; q < BK * EP; q += NT) {
          const int r = q / EP, e = q % EP;
          const int t = tb + r;
          dd[q] = (t < T && e < E) ? __ldg(dl + static_cast<size_t>(t) * E + e) : 0.f;
        }
      }
    }
    cp_async_commit();
  };

  float acc[8][8];
#pragma unroll
  for (int u = 0; u < 8; ++u)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[u][j] = 0.f;

  issue(0);
  for (int st = 0; st < nsteps; ++st) {
    issue(st + 1);
    cp_async_wait<1>();
    __syncthreads();
    const uint16_t* xt = xs + (st & 1) * S::XSTAGE + 8 * tm;
    const float* dt = ds + (st & 1) * S::DSTAGE + 8 * tn;
#pragma unroll 4
    for (int r = 0; r < BK; ++r) {
      const uint4 xq = *reinterpret_cast<const uint4*>(xt + r * BM);
      const float4 d0 = *reinterpret_cast<const float4*>(dt + r * EP);
      const float4 d1 = *reinterpret_cast<const float4*>(dt + r * EP + 4);
      float xv[8];
      unpack8(xq, xv);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc[u][0] = fmaf(xv[u], d0.x, acc[u][0]);
        acc[u][1] = fmaf(xv[u], d0.y, acc[u][1]);
        acc[u][2] = fmaf(xv[u], d0.z, acc[u][2]);
        acc[u][3] = fmaf(xv[u], d0.w, acc[u][3]);
        acc[u][4] = fmaf(xv[u], d1.x, acc[u][4]);
        acc[u][5] = fmaf(xv[u], d1.y, acc[u][5]);
        acc[u][6] = fmaf(xv[u], d1.z, acc[u][6]);
        acc[u][7] = fmaf(xv[u], d1.w, acc[u][7]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int col = i0 + 8 * tm + u;
    if (col >= h) break;
    float* dst = partial + (static_cast<size_t>(c) * h + col) * E + 8 * tn;
    if (E % 4 == 0 && 8 * tn + 8 <= E) {
      reinterpret_cast<float4*>(dst)[0] = make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(acc[u][4], acc[u][5], acc[u][6], acc[u][7]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (8 * tn + j < E) dst[j] = acc[u][j];
    }
  }
}

__global__ void router_wgrad_reduce_kernel(const float* __restrict__ partial, int nchunks, int h,
                                           int E, float* __restrict__ dWg) {
  const long long n = static_cast<long long>(h) * E;
  for (long long q = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; q < n;
       q += static_cast<long long>(gridDim.x) * blockDim.x) {
    float s = 0.f;
    for (int c = 0; c < nchunks; ++c) s += partial[static_cast<size_t>(c) * n + q];
    dWg[q] = s;
  }
}

}  // namespace

size_t router_partial_bytes(int T, int h, int E) {
  const int nch = router_chunks(T, h, E);
  if (router_padded_e(E) == 8 && nch == 1) return 0;
  return static_cast<size_t>(nch) * T * router_padded_e(E) * sizeof(float);
}

cudaError_t launch_router(const uint16_t* x, const float* Wg, const float* b, int T, int h, int E,
                          int k, int32_t* idx, float* gates, float* partial, int num_sms,
                          cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int ep = router_padded_e(E);
  const int nch = router_chunks(T, h, E);
  cudaError_t err;
  if (ep == 8 && nch == 1) return router_a1_dispatch(x, Wg, b, T, h, E, k, idx, gates, num_sms, s);
  if (ep == 8) {
    err = set_smem_once(reinterpret_cast<const void*>(router_a_kernel), kRouterASmem);
    if (err != cudaSuccess) return err;
    const int tiles = (T + kRouterATile - 1) / kRouterATile;
    int bpc = num_sms / nch;
    if (bpc < 1) bpc = 1;
    if (bpc > tiles) bpc = tiles;
    router_a_kernel<<<nch * bpc, kRouterAThreads, kRouterASmem, s>>>(x, Wg, b, T, h, E, k, nch, idx, gates,
                                                        partial);
    err = launched();
    if (err != cudaSuccess || nch == 1) return err;
    return router_select_launch<8>(partial, nch, b, T, E, k, idx, gates, num_sms, s);
  }
  if (ep == 16) err = router_c_launch<16>(x, Wg, T, h, E, nch, partial, s);
  else if (ep == 32) err = router_c_launch<32>(x, Wg, T, h, E, nch, partial, s);
  else err = router_c_launch<64>(x, Wg, T, h, E, nch, partial, s);
  if (err != cudaSuccess) return err;
  if (ep == 16) return router_select_launch<16>(partial, nch, b, T, E, k, idx, gates, num_sms, s);
  if (ep == 32) return router_select_launch<32>(partial, nch, b, T, E, k, idx, gates, num_sms, s);
  return router_select_launch<64>(partial, nch, b, T, E, k, idx, gates, num_sms, s);
}


cudaError_t launch_dispatch_hist(const int32_t* topk_idx, long long n, int E,
                                 const DispatchSel& sel, int32_t* blk_counts, cudaStream_t s,
                                 int* status) {
  const int nblk = dispatch_blocks(n);
  if (nblk == 0) return cudaSuccess;
  dispatch_kernel<false><<<nblk, kDispThreads, 0, s>>>(topk_idx, n, E, sel.e_lo, sel.count,
                                                        sel.capacity, blk_counts, nullptr, nullptr,
                                                        nullptr, nullptr, status);
  return launched();
}

cudaError_t launch_dispatch_scan(const int32_t* blk_counts, int nblk, const DispatchSel& sel,
                                 int32_t* counts, int32_t* offsets, int32_t* bases,
                                 cudaStream_t s) {
  dispatch_scan_kernel<<<1, 256, 0, s>>>(blk_counts, nblk, sel.count, sel.capacity, counts,
                                         offsets, bases);
  return launched();
}

cudaError_t launch_dispatch_scatter(const int32_t* topk_idx, long long n, int E,
                                    const DispatchSel& sel, const int32_t* bases,
                                    const int32_t* offsets, int32_t* perm_src, int32_t* perm_dst,
                                    cudaStream_t s, int* status) {
  const int nblk = dispatch_blocks(n);
  if (nblk == 0) return cudaSuccess;
  dispatch_kernel<true><<<nblk, kDispThreads, 0, s>>>(topk_idx, n, E, sel.e_lo, sel.count,
                                                       sel.capacity, nullptr, bases, offsets,
                                                       perm_src, perm_dst, status);
  return launched();
}

cudaError_t launch_gather_rows(const uint16_t* in, const int32_t* idx, int div, long long rows,
                               long long src_rows, int h, uint16_t* out, int num_sms,
                               cudaStream_t s, const int32_t* nvalid, const float* gsrc,
                               float* gdst, int* status) {
  if (rows == 0) return cudaSuccess;
  const int grid = grid_for(rows, num_sms, 8, 16);
  gather_rows_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(in), idx, div, rows,
                                          src_rows, nvalid, h / 8, reinterpret_cast<uint4*>(out),
                                          gsrc, gdst, status);
  return launched();
}

cudaError_t launch_combine(const uint16_t* O, const float* gates, const int32_t* perm_dst, int T,
                           int k, int h, uint16_t* y, int num_sms, cudaStream_t s, int* status) {
  if (T == 0) return cudaSuccess;
  const int grid = grid_for(T, num_sms, 8, 16);
  const uint4* o = reinterpret_cast<const uint4*>(O);
  uint4* yy = reinterpret_cast<uint4*>(y);
  switch (k) {
    case 1: combine_kernel<1><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy, status); break;
    case 2: combine_kernel<2><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy, status); break;
    case 3: combine_kernel<3><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy, status); break;
    case 4: combine_kernel<4><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy, status); break;
    case 5: combine_kernel<5><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy, status); break;
    case 6: combine_kernel<6><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy, status); break;
    case 7: combine_kernel<7><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy, status); break;
    default: combine_kernel<8><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy, status); break;
  }
  return launched();
}

// The bounded-wait path on its own: one thread waits on an mbarrier that
// nothing will ever complete; the wait gives up after limit_ns and records
// MOE_ERR_DEVICE_TIMEOUT (5) in *status, as a stalled matmul pipeline would.
__global__ void wait_timeout_probe_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, status, 5, limit_ns);
}

cudaError_t launch_wait_timeout_probe(int* status, unsigned long long limit_ns, cudaStream_t s) {
  wait_timeout_probe_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return launched();
}

cudaError_t launch_dg_reduce(const float* part, int nt, const int32_t* perm_src, long long rows,
                             const int32_t* nvalid, float* dg, int num_sms, cudaStream_t s,
                             int* status) {
  if (rows == 0) return cudaSuccess;
  long long blocks = (rows + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 8;
  dg_reduce_kernel<<<static_cast<int>(blocks < cap ? blocks : cap), 256, 0, s>>>(part, nt, perm_src,
                                                                                 rows, nvalid, dg,
                                                                                 status);
  return launched();
}

cudaError_t launch_bwd_prep(const uint16_t* dy, const uint16_t* O, const float* gates,
                            const int32_t* perm_src, long long rows, int k, int h, uint16_t* dO,
                            float* dg, int num_sms, cudaStream_t s, const int32_t* nvalid,
                            int* status) {
  if (rows == 0) return cudaSuccess;
  const int grid = grid_for(rows, num_sms, 8, 16);
  bwd_prep_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(dy),
                                       reinterpret_cast<const uint4*>(O), gates, perm_src, rows,
                                       nvalid, k, h / 8, reinterpret_cast<uint4*>(dO), dg, status);
  return launched();
}

cudaError_t launch_transpose_wg(const float* Wg, int h, int E, float* WgT, cudaStream_t s) {
  const long long n = static_cast<long long>(h) * E;
  int grid = static_cast<int>((n + 255) / 256);
  if (grid > 1024) grid = 1024;
  transpose_wg_kernel<<<grid, 256, 0, s>>>(Wg, h, E, WgT);
  return launched();
}

cudaError_t launch_token_grad(const float* dX_perm, const int32_t* perm_dst,
                              const int32_t* topk_idx, const float* gates, const float* dg,
                              const float* WgT, int T, int k, int h, int E, float* dl,
                              uint16_t* dx, int num_sms, cudaStream_t s, int* status) {
  if (T == 0) return cudaSuccess;
  const float4* d4 = reinterpret_cast<const float4*>(dX_perm);
  const float4* w4 = reinterpret_cast<const float4*>(WgT);
  uint4* o = reinterpret_cast<uint4*>(dx);
  const int h8 = h / 8;
  // k <= 2: one wave of resident blocks whose warps stride over the row
  // pieces (a grid of T / 8 blocks left a partial second wave); k >= 3: a
  // block per 8 tokens, up to 16 blocks per SM
  auto go = [&](auto kern) {
    const int per_sm = k <= 2 ? resident_blocks(reinterpret_cast<const void*>(kern), 256) : 16;
    const int grid = grid_for(T, num_sms, 8, per_sm);
    kern<<<grid, 256, 0, s>>>(d4, perm_dst, topk_idx, gates, dg, w4, T, h8, E, dl, o, status);
  };
  switch (k) {
    case 1: go(token_grad_kernel<1>); break;
    case 2: go(token_grad_kernel<2>); break;
    case 3: go(token_grad_kernel<3>); break;
    case 4: go(token_grad_kernel<4>); break;
    case 5: go(token_grad_kernel<5>); break;
    case 6: go(token_grad_kernel<6>); break;
    case 7: go(token_grad_kernel<7>); break;
    default: go(token_grad_kernel<8>); break;
  }
  return launched();
}

template <int EP>
int wgrad_c_nch(int T, int h) {
  const long long tiles = (h + WgradC<EP>::BM - 1) / WgradC<EP>::BM;
  return split_k_chunks(tiles, (T + WgradC<EP>::BK - 1) / WgradC<EP>::BK, 128);
}

int wgrad_c_chunks(int T, int h, int E) {
  const int ep = router_padded_e(E);
  return ep == 8 ? wgrad_c_nch<8>(T, h)
                 : ep == 16 ? wgrad_c_nch<16>(T, h)
                            : ep == 32 ? wgrad_c_nch<32>(T, h) : wgrad_c_nch<64>(T, h);
}

template <int EP>
cudaError_t router_wgrad_c_launch(const uint16_t* x, const float* dl, int T, int h, int E,
                                  int nch, float* partial, cudaStream_t s) {
  using S = WgradC<EP>;
  const cudaError_t e =
      set_smem_once(reinterpret_cast<const void*>(router_wgrad_c_kernel<EP>), S::SMEM);
  if (e != cudaSuccess) return e;
  const long long tiles = (h + S::BM - 1) / S::BM;
  router_wgrad_c_kernel<EP><<<static_cast<int>(tiles * nch), S::THREADS, S::SMEM, s>>>(
      x, dl, T, h, E, nch, partial);
  return launched();
}

int wgrad_router_chunks(int T, int h, int E) { return T > 0 ? wgrad_c_chunks(T, h, E) : 0; }

namespace {
__global__ void check_offsets_kernel(const int32_t* __restrict__ offsets, int E, long long rows,
                                     int* __restrict__ status) {
  bool ok = true;
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    const long long o = __ldg(offsets + e);
    if (o < 0 || o > rows || (e == 0 && o != 0) || (e > 0 && o < __ldg(offsets + e - 1)))
      ok = false;
  }
  if (!ok) report_bad_index(status);
}

// the status word of the calls without a workspace, one per device
__device__ int g_nows_status = 0;
std::mutex g_nows_mu;
int* g_nows_addr[64] = {nullptr};
}  // namespace

cudaError_t launch_check_offsets(const int32_t* offsets, int E, long long rows, int* status,
                                 cudaStream_t s) {
  check_offsets_kernel<<<1, 256, 0, s>>>(offsets, E, rows, status);
  return launched();
}

cudaError_t set_smem_once(const void* kern, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> done;  // (kernel, device) -> bytes set
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorNoDevice;
  std::lock_guard<std::mutex> lock(mu);
  int& have = done[{kern, dev}];
  if (have >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

int* nows_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_nows_mu);
  if (!g_nows_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_nows_status) != cudaSuccess) return nullptr;
    g_nows_addr[dev] = static_cast<int*>(p);
  }
  return g_nows_addr[dev];
}

cudaError_t launch_router_wgrad(const uint16_t* x, const float* dl, int T, int h, int E,
                                float* partial, float* dWg, cudaStream_t s) {
  const int nchunks = wgrad_router_chunks(T, h, E);
  if (nchunks > 0) {
    const int ep = router_padded_e(E);
    cudaError_t e;
    if (ep == 8) e = router_wgrad_c_launch<8>(x, dl, T, h, E, nchunks, partial, s);
    else if (ep == 16) e = router_wgrad_c_launch<16>(x, dl, T, h, E, nchunks, partial, s);
    else if (ep == 32) e = router_wgrad_c_launch<32>(x, dl, T, h, E, nchunks, partial, s);
    else e = router_wgrad_c_launch<64>(x, dl, T, h, E, nchunks, partial, s);
    if (e != cudaSuccess) return e;
  }
  const long long n = static_cast<long long>(h) * E;
  int grid2 = static_cast<int>((n + 255) / 256);
  if (grid2 > 2048) grid2 = 2048;
  router_wgrad_reduce_kernel<<<grid2, 256, 0, s>>>(partial, nchunks, h, E, dWg);
  return launched();
}

}  // namespace moe
