// kernels.cu -- router, dispatch, row-move, combine and router-backward kernels.
//
// Everything here is HBM- or FP32-bound; none of it uses tensor cores.  Every
// reduction has a fixed order and no kernel uses atomics, so results are
// bitwise reproducible run to run.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {

namespace {
thread_local long long g_launches = 0;
}  // namespace

long long kernel_launches() { return g_launches; }

cudaError_t launched() {
  ++g_launches;
  return cudaGetLastError();
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

int grid_for(long long warps_needed, int num_sms, int warps_per_block, int blocks_per_sm) {
  long long blocks = (warps_needed + warps_per_block - 1) / warps_per_block;
  long long cap = static_cast<long long>(num_sms) * blocks_per_sm;
  if (blocks > cap) blocks = cap;
  return blocks < 1 ? 1 : static_cast<int>(blocks);
}

// ------------------------------------------------------------------ router
// The hidden dimension is cut into chunks of CH columns; each block stages one
// chunk of the router weights in shared memory once and then streams every
// token tile of its share through it.  With one chunk (E <= 8, h <= 4096) the
// kernel finishes the routing itself; otherwise it writes fp32 partial logits
// [chunk][T][EP] and router_select_kernel adds them in chunk order.

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
constexpr int kRouterA1Threads = 256;
constexpr int kRouterA1Warps = kRouterA1Threads / 32;
constexpr int kRouterA1Step = 256;  // columns per stage
constexpr int kRouterA1NStage = 3;
constexpr int kRouterA1MaxH = 4096;
constexpr size_t router_a1_smem(int h, int tok) {
  return static_cast<size_t>((h + 7) / 8) * kRouterASlice * 4 +
         static_cast<size_t>(kRouterA1Warps) * kRouterA1NStage * tok * kRouterA1Step * 2 +
         static_cast<size_t>(kRouterA1Warps) * 64 * 4;
}

template <int TOK>
__global__ void __launch_bounds__(kRouterA1Threads, 1) router_a1_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ Wg, const float* __restrict__ b,
    int T, int h, int E, int k, int32_t* __restrict__ topk_idx, float* __restrict__ gates) {
  constexpr int EP = 8, SLICE = kRouterASlice, NST = kRouterA1NStage, SC = kRouterA1Step;
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

// ---- E > 8: lanes own experts.  A group of GL = EP / 4 lanes handles TOK
// tokens; lane i of a group owns the four consecutive experts 4i .. 4i + 3,
// whose weights for one column are one conflict-free 16-byte shared-memory
// load, so every unpacked x value feeds four FMAs.  Each warp stages its
// tokens' x slice (XS columns) in shared memory and reads it as broadcasts;
// the slice is stored token-interleaved (token u of group g at row u NG + g),
// so the NG groups of a warp read adjacent rows, which the padded pitch puts
// in different banks.  Every weight value a lane loads then feeds TOK tokens.
// No cross-lane reduction.
constexpr int kRouterBXs = 64;
constexpr int kRouterBXsp = kRouterBXs + 8;  // padded row (bf16) of a staged x slice

template <int EP>
struct RouterB {
  static constexpr int EPL = 4;                  // experts per lane
  static constexpr int GL = EP / EPL;            // lanes per token group
  static constexpr int NG = 32 / GL;             // token groups per warp
  static constexpr int TOK = 8;                  // tokens per group
  static constexpr int CH = 32768 / EP;          // columns per chunk (128 KiB of weights)
  static constexpr int XROWS = NG * TOK;         // staged token rows per warp
  static constexpr int SMEM = CH * EP * 4 + 8 * XROWS * kRouterBXsp * 2;
};

template <int EP>
__global__ void __launch_bounds__(256, 1) router_b_kernel(const uint16_t* __restrict__ x,
                                                          const float* __restrict__ Wg, int T,
                                                          int h, int E, int nch,
                                                          float* __restrict__ partial) {
  using S = RouterB<EP>;
  constexpr int TOK = S::TOK, EPL = S::EPL, XS = kRouterBXs, XSP = kRouterBXsp;
  extern __shared__ float sw[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(sw + S::CH * EP);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int g = lane / S::GL;
  const int el = lane % S::GL;
  const int c = blockIdx.x % nch;
  const int sub = blockIdx.x / nch;
  const int bpc = gridDim.x / nch;
  const int c0 = c * S::CH;
  const int rows = min(S::CH, h - c0);
  for (int q = threadIdx.x; q < rows * EP; q += 256) {
    const int lr = q / EP;
    const int e = q - lr * EP;
    sw[q] = (e < E) ? __ldg(Wg + static_cast<size_t>(c0 + lr) * E + e) : 0.f;
  }
  __syncthreads();
  uint16_t* xw = xs + warp * S::XROWS * XSP;
  const int btile = 8 * S::XROWS;
  for (int t0 = sub * btile; t0 < T; t0 += bpc * btile) {
    const int tw = t0 + warp * S::XROWS;  // this warp's first token
    float acc[TOK][EPL];
#pragma unroll
    for (int u = 0; u < TOK; ++u)
#pragma unroll
      for (int i = 0; i < EPL; ++i) acc[u][i] = 0.f;
    for (int cs = 0; cs < rows; cs += XS) {
      // stage x[tw .. tw + XROWS)[c0 + cs .. + XS) (rows of 128 bytes)
#pragma unroll
      for (int r = 0; r < S::XROWS * (XS / 8) / 32; ++r) {
        const int id = r * 32 + lane;
        const int row = id / (XS / 8);
        const int c8 = id % (XS / 8);
        const int t = tw + row;
        const bool ok = t < T && cs + 8 * c8 < rows;
        const uint4 v = ok ? __ldg(reinterpret_cast<const uint4*>(
                                 x + static_cast<size_t>(t) * h + c0 + cs + 8 * c8))
                           : make_uint4(0, 0, 0, 0);
        const int srow = (row % TOK) * S::NG + row / TOK;  // token-interleaved
        *reinterpret_cast<uint4*>(xw + srow * XSP + 8 * c8) = v;
      }
      __syncwarp();
#pragma unroll 1
      for (int c8 = 0; c8 < XS / 8; ++c8) {
        uint4 xq[TOK];
#pragma unroll
        for (int u = 0; u < TOK; ++u)
          xq[u] = *reinterpret_cast<const uint4*>(xw + (u * S::NG + g) * XSP + 8 * c8);
        const float4* wr = reinterpret_cast<const float4*>(sw + (cs + 8 * c8) * EP) + el;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 w = wr[j * (EP / 4)];
#pragma unroll
          for (int u = 0; u < TOK; ++u) {
            const uint32_t q = j < 2 ? xq[u].x : j < 4 ? xq[u].y : j < 6 ? xq[u].z : xq[u].w;
            const float xv = (j & 1) ? bf16_hi(q) : bf16_lo(q);
            acc[u][0] = fmaf(xv, w.x, acc[u][0]);
            acc[u][1] = fmaf(xv, w.y, acc[u][1]);
            acc[u][2] = fmaf(xv, w.z, acc[u][2]);
            acc[u][3] = fmaf(xv, w.w, acc[u][3]);
          }
        }
      }
      __syncwarp();
    }
#pragma unroll
    for (int u = 0; u < TOK; ++u) {
      const int t = tw + g * TOK + u;
      if (t >= T) continue;
      *reinterpret_cast<float4*>(partial + (static_cast<size_t>(c) * T + t) * EP + EPL * el) =
          make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
    }
  }
}

// Thread per token: logits = sum of the chunks' partials (in chunk order) + b.
template <int EP>
__global__ void __launch_bounds__(128) router_select_kernel(const float* __restrict__ partial,
                                                            int nch, const float* __restrict__ b,
                                                            int T, int E, int k,
                                                            int32_t* __restrict__ topk_idx,
                                                            float* __restrict__ gates) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    float l[EP];
#pragma unroll
    for (int e = 0; e < EP; ++e) l[e] = 0.f;
    for (int c = 0; c < nch; ++c) {
      const float4* src =
          reinterpret_cast<const float4*>(partial + (static_cast<size_t>(c) * T + t) * EP);
#pragma unroll
      for (int e4 = 0; e4 < EP / 4; ++e4) {
        const float4 v = __ldg(src + e4);
        l[4 * e4 + 0] += v.x;
        l[4 * e4 + 1] += v.y;
        l[4 * e4 + 2] += v.z;
        l[4 * e4 + 3] += v.w;
      }
    }
#pragma unroll
    for (int e = 0; e < EP; ++e)
      if (e < E && b) l[e] += __ldg(b + e);
    select_topk<EP>(l, E, k, topk_idx + static_cast<size_t>(t) * k,
                    gates + static_cast<size_t>(t) * k);
  }
}

int router_padded_e(int E) { return E <= 8 ? 8 : E <= 16 ? 16 : E <= 32 ? 32 : 64; }

int router_chunks(int h, int E) {
  const int ep = router_padded_e(E);
  if (ep == 8 && h <= kRouterA1MaxH) return 1;  // router_a1_kernel holds all of Wg
  const int ch = ep == 8 ? kRouterACh : 32768 / ep;
  return (h + ch - 1) / ch;
}

// router_a1_kernel<TOK>: the TOK whose items spread most evenly over the
// grid's warps (fewest token slots on the busiest warp; ties to the larger
// TOK), within the shared-memory limit.
template <int TOK>
cudaError_t router_a1_launch(const uint16_t* x, const float* Wg, const float* b, int T, int h,
                             int E, int k, int32_t* idx, float* gates, int blocks,
                             cudaStream_t s) {
  const size_t smem = router_a1_smem(h, TOK);
  static int attr_smem = 0;
  if (attr_smem < static_cast<int>(smem)) {
    const cudaError_t e = cudaFuncSetAttribute(
        router_a1_kernel<TOK>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_smem = static_cast<int>(smem);
  }
  router_a1_kernel<TOK><<<blocks, kRouterA1Threads, smem, s>>>(x, Wg, b, T, h, E, k, idx, gates);
  return launched();
}

cudaError_t router_a1_dispatch(const uint16_t* x, const float* Wg, const float* b, int T, int h,
                               int E, int k, int32_t* idx, float* gates, int num_sms,
                               cudaStream_t s) {
  const long long nw = static_cast<long long>(num_sms) * kRouterA1Warps;
  int best = 4;
  long long best_slots = -1;
  for (int tok = 4; tok <= 7; ++tok) {
    if (router_a1_smem(h, tok) > 232448) continue;
    const long long items = (T + tok - 1) / tok;
    const long long slots = (items + nw - 1) / nw * tok;
    if (best_slots < 0 || slots <= best_slots) {
      best = tok;
      best_slots = slots;
    }
  }
  // blocks: enough warps for the items, at most one block per SM
  const long long items = (T + best - 1) / best;
  int blocks = static_cast<int>((items + kRouterA1Warps - 1) / kRouterA1Warps);
  if (blocks > num_sms) blocks = num_sms;
  switch (best) {
    case 4: return router_a1_launch<4>(x, Wg, b, T, h, E, k, idx, gates, blocks, s);
    case 5: return router_a1_launch<5>(x, Wg, b, T, h, E, k, idx, gates, blocks, s);
    case 6: return router_a1_launch<6>(x, Wg, b, T, h, E, k, idx, gates, blocks, s);
    default: return router_a1_launch<7>(x, Wg, b, T, h, E, k, idx, gates, blocks, s);
  }
}

template <int EP>
cudaError_t router_b_launch(const uint16_t* x, const float* Wg, int T, int h, int E, int nch,
                            float* partial, int num_sms, cudaStream_t s) {
  using S = RouterB<EP>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(router_b_kernel<EP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int tiles = (T + 8 * S::XROWS - 1) / (8 * S::XROWS);
  int bpc = num_sms / nch;
  if (bpc < 1) bpc = 1;
  if (bpc > tiles) bpc = tiles;
  router_b_kernel<EP><<<nch * bpc, 256, S::SMEM, s>>>(x, Wg, T, h, E, nch, partial);
  return launched();
}

template <int EP>
cudaError_t router_select_launch(const float* partial, int nch, const float* b, int T, int E,
                                 int k, int32_t* idx, float* gates, int num_sms, cudaStream_t s) {
  long long blocks = (T + 127) / 128;
  if (blocks > num_sms * 8) blocks = num_sms * 8;
  router_select_kernel<EP><<<static_cast<int>(blocks), 128, 0, s>>>(partial, nch, b, T, E, k, idx,
                                                                   gates);
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
// offsets[e] + rank, the others get perm_dst = -1.
constexpr int kDispThreads = 256;
constexpr int kDispWarps = kDispThreads / 32;
constexpr int kDispMaxE = 256;

template <bool WRITE>
__global__ void __launch_bounds__(kDispThreads) dispatch_kernel(
    const int32_t* __restrict__ topk_idx, long long n, int E, int e_lo, int EL, int cap,
    int32_t* __restrict__ blk_counts, const int32_t* __restrict__ bases,
    const int32_t* __restrict__ offsets, int32_t* __restrict__ perm_src,
    int32_t* __restrict__ perm_dst) {
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
      int e = __ldg(topk_idx + a);
      e = e < 0 ? 0 : (e >= E ? E - 1 : e);  // keep every index in range
      le = (e >= e_lo && e < e_lo + EL) ? e - e_lo : -1;
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
// zero row.  With gsrc/gdst, also gdst[p] = gsrc[idx[p]] (a value per row).
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ in,
                                                          const int32_t* __restrict__ idx, int div,
                                                          long long rows, long long src_rows,
                                                          const int32_t* __restrict__ nvalid,
                                                          int h8, uint4* __restrict__ out,
                                                          const float* __restrict__ gsrc,
                                                          float* __restrict__ gdst) {
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
    if (gdst && lane == 0) gdst[p] = i < 0 ? 0.f : __ldg(gsrc + i);
    if (i < 0) {
      for (int c = lane; c < h8; c += 32) d[c] = make_uint4(0, 0, 0, 0);
      continue;
    }
    long long src = i / div;
    src = src >= src_rows ? src_rows - 1 : src;  // stay inside `in`
    const uint4* s = in + src * h8;
#pragma unroll 4
    for (int c = lane; c < h8; c += 32) d[c] = __ldg(s + c);
  }
}

// y[t] = sum_j g[t,j] * O[perm_dst[t*k+j]], fp32 in slot order.  K = k.
template <int K>
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ O,
                                                      const float* __restrict__ gates,
                                                      const int32_t* __restrict__ perm_dst, int T,
                                                      int h8, uint4* __restrict__ y) {
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
        // a dropped slot (r < 0) adds nothing and reads no row
        kept[j] = r >= 0;
        rows[j] = r < 0 ? 0 : (r >= static_cast<long long>(T) * k ? static_cast<long long>(T) * k - 1 : r);
        g[j] = r < 0 ? 0.f : __ldg(gates + static_cast<size_t>(t) * k + j);
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

// dO[p] = bf16(g[a] * dy[t]); dg[a] = <dy[t], O[p]>.
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint4* __restrict__ dy,
                                                       const uint4* __restrict__ O,
                                                       const float* __restrict__ gates,
                                                       const int32_t* __restrict__ perm_src,
                                                       long long rows,
                                                       const int32_t* __restrict__ nvalid, int k,
                                                       int h8, uint4* __restrict__ dO,
                                                       float* __restrict__ dg) {
  const int lane = threadIdx.x & 31;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const long long total = rows;
  if (nvalid) {
    const long long nv = __ldg(nvalid);
    rows = nv < rows ? (nv < 0 ? 0 : nv) : rows;
  }
  for (long long p = gw; p < rows; p += nw) {
    int a = __ldg(perm_src + p);
    a = a < 0 ? 0 : (a >= total ? static_cast<int>(total - 1) : a);
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
                                                        float* __restrict__ dg) {
  const long long nv = __ldg(nvalid);
  const long long n = nv < rows ? (nv < 0 ? 0 : nv) : rows;
  for (long long p = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; p < n;
       p += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float* q = part + p * nt;
    float s = 0.f;
    for (int i = 0; i < nt; ++i) s += __ldg(q + i);
    long long a = __ldg(perm_src + p);
    a = a < 0 ? 0 : (a >= rows ? rows - 1 : a);
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

// Router backward per token + dx, warp per token (K = k).  U 16-byte pieces of
// the row per lane per step keep 2 * U * K fp32 loads of dX_perm in flight.
template <int K>
__global__ void __launch_bounds__(256) token_grad_kernel(
    const float4* __restrict__ dX, const int32_t* __restrict__ perm_dst,
    const int32_t* __restrict__ topk_idx, const float* __restrict__ gates,
    const float* __restrict__ dg, const float4* __restrict__ WgT, int T, int h8, int E,
    float* __restrict__ dl, uint4* __restrict__ dx) {
  constexpr int U = K <= 2 ? 2 : 1;
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const long long R = static_cast<long long>(T) * K;
  for (int t = gw; t < T; t += nw) {
    long long rows[K];
    int ex[K];
    bool kept[K];
    float g[K], d[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      const size_t a = static_cast<size_t>(t) * K + j;
      const long long r = __ldg(perm_dst + a);
      kept[j] = r >= 0;  // a dropped slot has no expert output: dg = 0, no dX
      rows[j] = r < 0 ? 0 : (r >= R ? R - 1 : r);
      const int e = __ldg(topk_idx + a);
      ex[j] = e < 0 ? 0 : (e >= E ? E - 1 : e);
      g[j] = __ldg(gates + a);
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
    for (int e = lane; e < E; e += 32) {
      float v = 0.f;
#pragma unroll
      for (int j = 0; j < K; ++j)
        if (ex[j] == e) v = dlj[j];
      dl[static_cast<size_t>(t) * E + e] = v;
    }
    for (int c0 = lane; c0 < h8; c0 += 32 * U) {
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

// dWg partials: block = (column tile, token chunk of kWgChunk); thread owns
// CPT consecutive columns (2 for E <= 8, so a warp's x loads are whole
// 128-byte lines) and EP experts; dl rows of the chunk are staged in shared
// memory.
constexpr int kWgChunk = 256;
constexpr int kWgStage = 32;

template <int EP>
struct WgShape {
  static constexpr int CPT = EP <= 8 ? 2 : 16 / EP >= 1 ? 16 / EP : 1;  // columns per thread
  static constexpr int COLS = 256 * CPT;             // columns per block
};

template <int EP>
__global__ void __launch_bounds__(256) router_wgrad_kernel(const uint16_t* __restrict__ x,
                                                           const float* __restrict__ dl, int T,
                                                           int h, int E,
                                                           float* __restrict__ partial) {
  constexpr int CPT = WgShape<EP>::CPT;
  __shared__ float sdl[kWgStage][EP];
  const int i0 = blockIdx.x * WgShape<EP>::COLS + threadIdx.x * CPT;  // first column
  const int chunk = blockIdx.y;
  const int t0 = chunk * kWgChunk;
  const int t1 = min(T, t0 + kWgChunk);
  float acc[CPT][EP];
#pragma unroll
  for (int c = 0; c < CPT; ++c)
#pragma unroll
    for (int e = 0; e < EP; ++e) acc[c][e] = 0.f;
  for (int ts = t0; ts < t1; ts += kWgStage) {
    __syncthreads();
    for (int q = threadIdx.x; q < kWgStage * EP; q += 256) {
      const int tt = ts + q / EP;
      const int e = q % EP;
      sdl[q / EP][e] = (tt < t1 && e < E) ? dl[static_cast<size_t>(tt) * E + e] : 0.f;
    }
    __syncthreads();
    if (i0 < h) {
      const int n = min(kWgStage, t1 - ts);
      for (int u = 0; u < n; ++u) {
        const uint16_t* xr = x + static_cast<size_t>(ts + u) * h + i0;
        float xv[CPT];
        if constexpr (CPT == 8) {
          unpack8(__ldg(reinterpret_cast<const uint4*>(xr)), xv);
        } else if constexpr (CPT == 4) {
          const uint2 q = __ldg(reinterpret_cast<const uint2*>(xr));
          xv[0] = bf16_lo(q.x);
          xv[1] = bf16_hi(q.x);
          xv[2] = bf16_lo(q.y);
          xv[3] = bf16_hi(q.y);
        } else if constexpr (CPT == 2) {
          const uint32_t q = __ldg(reinterpret_cast<const uint32_t*>(xr));
          xv[0] = bf16_lo(q);
          xv[1] = bf16_hi(q);
        } else {
          xv[0] = __uint_as_float(static_cast<uint32_t>(__ldg(xr)) << 16);
        }
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
          for (int e = 0; e < EP; ++e) acc[c][e] = fmaf(xv[c], sdl[u][e], acc[c][e]);
      }
    }
  }
  if (i0 < h) {
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      float* dst = partial + (static_cast<size_t>(chunk) * h + i0 + c) * E;
#pragma unroll
      for (int e = 0; e < EP; ++e)
        if (e < E) dst[e] = acc[c][e];
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
  const int nch = router_chunks(h, E);
  if (router_padded_e(E) == 8 && nch == 1) return 0;
  return static_cast<size_t>(nch) * T * router_padded_e(E) * sizeof(float);
}

cudaError_t launch_router(const uint16_t* x, const float* Wg, const float* b, int T, int h, int E,
                          int k, int32_t* idx, float* gates, float* partial, int num_sms,
                          cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int ep = router_padded_e(E);
  const int nch = router_chunks(h, E);
  cudaError_t err;
  if (ep == 8 && nch == 1) return router_a1_dispatch(x, Wg, b, T, h, E, k, idx, gates, num_sms, s);
  if (ep == 8) {
    static bool attr = false;
    if (!attr) {
      err = cudaFuncSetAttribute(router_a_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kRouterASmem);
      if (err != cudaSuccess) return err;
      attr = true;
    }
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
  if (ep == 16) err = router_b_launch<16>(x, Wg, T, h, E, nch, partial, num_sms, s);
  else if (ep == 32) err = router_b_launch<32>(x, Wg, T, h, E, nch, partial, num_sms, s);
  else err = router_b_launch<64>(x, Wg, T, h, E, nch, partial, num_sms, s);
  if (err != cudaSuccess) return err;
  if (ep == 16) return router_select_launch<16>(partial, nch, b, T, E, k, idx, gates, num_sms, s);
  if (ep == 32) return router_select_launch<32>(partial, nch, b, T, E, k, idx, gates, num_sms, s);
  return router_select_launch<64>(partial, nch, b, T, E, k, idx, gates, num_sms, s);
}


cudaError_t launch_dispatch_hist(const int32_t* topk_idx, long long n, int E,
                                 const DispatchSel& sel, int32_t* blk_counts, cudaStream_t s) {
  const int nblk = dispatch_blocks(n);
  if (nblk == 0) return cudaSuccess;
  dispatch_kernel<false><<<nblk, kDispThreads, 0, s>>>(topk_idx, n, E, sel.e_lo, sel.count,
                                                        sel.capacity, blk_counts, nullptr, nullptr,
                                                        nullptr, nullptr);
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
                                    cudaStream_t s) {
  const int nblk = dispatch_blocks(n);
  if (nblk == 0) return cudaSuccess;
  dispatch_kernel<true><<<nblk, kDispThreads, 0, s>>>(topk_idx, n, E, sel.e_lo, sel.count,
                                                       sel.capacity, nullptr, bases, offsets,
                                                       perm_src, perm_dst);
  return launched();
}

cudaError_t launch_gather_rows(const uint16_t* in, const int32_t* idx, int div, long long rows,
                               long long src_rows, int h, uint16_t* out, int num_sms,
                               cudaStream_t s, const int32_t* nvalid, const float* gsrc,
                               float* gdst) {
  if (rows == 0 || src_rows == 0) return cudaSuccess;
  const int grid = grid_for(rows, num_sms, 8, 16);
  gather_rows_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(in), idx, div, rows,
                                          src_rows, nvalid, h / 8, reinterpret_cast<uint4*>(out),
                                          gsrc, gdst);
  return launched();
}

cudaError_t launch_combine(const uint16_t* O, const float* gates, const int32_t* perm_dst, int T,
                           int k, int h, uint16_t* y, int num_sms, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int grid = grid_for(T, num_sms, 8, 16);
  const uint4* o = reinterpret_cast<const uint4*>(O);
  uint4* yy = reinterpret_cast<uint4*>(y);
  switch (k) {
    case 1: combine_kernel<1><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy); break;
    case 2: combine_kernel<2><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy); break;
    case 3: combine_kernel<3><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy); break;
    case 4: combine_kernel<4><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy); break;
    case 5: combine_kernel<5><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy); break;
    case 6: combine_kernel<6><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy); break;
    case 7: combine_kernel<7><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy); break;
    default: combine_kernel<8><<<grid, 256, 0, s>>>(o, gates, perm_dst, T, h / 8, yy); break;
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
                             const int32_t* nvalid, float* dg, int num_sms, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  long long blocks = (rows + 255) / 256;
  const long long cap = static_cast<long long>(num_sms) * 8;
  dg_reduce_kernel<<<static_cast<int>(blocks < cap ? blocks : cap), 256, 0, s>>>(part, nt, perm_src,
                                                                                 rows, nvalid, dg);
  return launched();
}

cudaError_t launch_bwd_prep(const uint16_t* dy, const uint16_t* O, const float* gates,
                            const int32_t* perm_src, long long rows, int k, int h, uint16_t* dO,
                            float* dg, int num_sms, cudaStream_t s, const int32_t* nvalid) {
  if (rows == 0) return cudaSuccess;
  const int grid = grid_for(rows, num_sms, 8, 16);
  bwd_prep_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const uint4*>(dy),
                                       reinterpret_cast<const uint4*>(O), gates, perm_src, rows,
                                       nvalid, k, h / 8, reinterpret_cast<uint4*>(dO), dg);
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
                              uint16_t* dx, int num_sms, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int grid = grid_for(T, num_sms, 8, 16);
  const float4* d4 = reinterpret_cast<const float4*>(dX_perm);
  const float4* w4 = reinterpret_cast<const float4*>(WgT);
  uint4* o = reinterpret_cast<uint4*>(dx);
  const int h8 = h / 8;
  switch (k) {
    case 1: token_grad_kernel<1><<<grid, 256, 0, s>>>(d4, perm_dst, topk_idx, gates, dg, w4, T, h8, E, dl, o); break;
    case 2: token_grad_kernel<2><<<grid, 256, 0, s>>>(d4, perm_dst, topk_idx, gates, dg, w4, T, h8, E, dl, o); break;
    case 3: token_grad_kernel<3><<<grid, 256, 0, s>>>(d4, perm_dst, topk_idx, gates, dg, w4, T, h8, E, dl, o); break;
    case 4: token_grad_kernel<4><<<grid, 256, 0, s>>>(d4, perm_dst, topk_idx, gates, dg, w4, T, h8, E, dl, o); break;
    case 5: token_grad_kernel<5><<<grid, 256, 0, s>>>(d4, perm_dst, topk_idx, gates, dg, w4, T, h8, E, dl, o); break;
    case 6: token_grad_kernel<6><<<grid, 256, 0, s>>>(d4, perm_dst, topk_idx, gates, dg, w4, T, h8, E, dl, o); break;
    case 7: token_grad_kernel<7><<<grid, 256, 0, s>>>(d4, perm_dst, topk_idx, gates, dg, w4, T, h8, E, dl, o); break;
    default: token_grad_kernel<8><<<grid, 256, 0, s>>>(d4, perm_dst, topk_idx, gates, dg, w4, T, h8, E, dl, o); break;
  }
  return launched();
}

int wgrad_router_chunks(int T) { return (T + kWgChunk - 1) / kWgChunk; }

cudaError_t launch_router_wgrad(const uint16_t* x, const float* dl, int T, int h, int E,
                                float* partial, float* dWg, cudaStream_t s) {
  const int nchunks = wgrad_router_chunks(T);
  if (nchunks > 0) {
    auto cols = [&](int c) { return dim3((h + c - 1) / c, nchunks); };
    if (E <= 8)
      router_wgrad_kernel<8><<<cols(WgShape<8>::COLS), 256, 0, s>>>(x, dl, T, h, E, partial);
    else if (E <= 16)
      router_wgrad_kernel<16><<<cols(WgShape<16>::COLS), 256, 0, s>>>(x, dl, T, h, E, partial);
    else if (E <= 32)
      router_wgrad_kernel<32><<<cols(WgShape<32>::COLS), 256, 0, s>>>(x, dl, T, h, E, partial);
    else
      router_wgrad_kernel<64><<<cols(WgShape<64>::COLS), 256, 0, s>>>(x, dl, T, h, E, partial);
    cudaError_t e = launched();
    if (e != cudaSuccess) return e;
  }
  const long long n = static_cast<long long>(h) * E;
  int grid2 = static_cast<int>((n + 255) / 256);
  if (grid2 > 2048) grid2 = 2048;
  router_wgrad_reduce_kernel<<<grid2, 256, 0, s>>>(partial, nchunks, h, E, dWg);
  return launched();
}

}  // namespace moe
