// grouped_gemm.cu -- persistent tcgen05/TMEM GroupedGEMM for the SwiGLU experts.
//
// One kernel template serves all six expert matmuls of the layer (forward FC1
// and FC2, the two dgrads and the two ragged-K wgrads).  Design (sm_103a):
//   * persistent grid, one CTA per SM, 192 threads in three roles:
//       warp 0     TMA producer: 128B-swizzled tiles into a 4-stage smem ring
//       warp 1     tensor-memory allocator and MMA issuer (tcgen05.mma,
//                  128 x 256 x 16 per instruction, fp32 accumulator in TMEM)
//       warps 2-5  epilogue: tcgen05.ld of the accumulator, fused elementwise
//                  work (SwiGLU, SwiGLU backward), stores to global memory
//   * two 256-column TMEM accumulators, so the epilogue of tile i overlaps the
//     main loop of tile i+1;
//   * groups come from the device-resident expert offsets: M-grouped matmuls
//     (forward, dgrad) tile each expert's row range; K-grouped ones (wgrad)
//     reduce over it, zeroing the k-rows of the last block that belong to the
//     next expert before they reach the tensor core.
// Shapes: M tile 128, K block 64 (one 128-byte swizzle row of bf16), N tile
// 256 accumulator columns (one B operand of 256, or two of 128 sharing A).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "grouped_gemm.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace moe {


const char* const kGemmNames[6] = {"gg_fc1_fwd_swiglu", "gg_fc2_fwd",
                                   "gg_fc2_dgrad_swiglu_bwd", "gg_fc1_dgrad",
                                   "gg_fc2_wgrad", "gg_fc1_wgrad"};
const char* const kGemmSarDgradName = "gg_fc2_dgrad_swiglu_bwd_sar";

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int BN = 256;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KiB
constexpr int B_BYTES = BN * BK * 2;            // 32 KiB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KiB
constexpr int CHUNK_BYTES = 64 * BK * 2;        // one 64 x 64 MN-major box: 8 KiB
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr int MAX_E = 64;   // the C ABI limits E to 64
constexpr int kTimeoutCode = 5;  // MOE_ERR_DEVICE_TIMEOUT

// Shared memory after the stage ring.
struct alignas(8) Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int off[MAX_E + 1];   // expert offsets
  int cum[MAX_E + 1];   // M-grouped: prefix of m-tiles per expert
};
// Each epilogue warp owns two 4 KiB staging blocks between the stage ring and
// the control words: 32 x 32 fp32 tiles on their way to global memory (see
// store_f32_block).
constexpr int EPI_STAGE_BYTES = 32 * 32 * 4;
constexpr int EPI_SMEM_BYTES = 4 * 2 * EPI_STAGE_BYTES;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_SMEM_BYTES + static_cast<int>(sizeof(Ctrl));

enum Epi {
  EPI_SWIGLU = 0,
  EPI_BF16 = 1,
  EPI_SWIGLU_BWD = 2,
  EPI_F32 = 3,
  EPI_WGRAD = 4,
  EPI_SWIGLU_BWD_SAR = 5,  // SwiGLU backward that rebuilds H from A, B (no saved H or O)
  EPI_SWIGLU_F8 = 6,       // EPI_SWIGLU on e4m3 operands: sums rescaled by row x column scales
  EPI_BF16_F8 = 7,         // EPI_BF16 on e4m3 operands, likewise
  EPI_F32_F8 = 8           // EPI_F32 on e4m3 operands
};
__host__ __device__ constexpr bool is_f8(int epi) {
  return epi == EPI_SWIGLU_F8 || epi == EPI_BF16_F8 || epi == EPI_F32_F8;
}
// The epilogue an FP8 matmul runs after rescaling its sums.
__host__ __device__ constexpr int base_epi(int epi) {
  return epi == EPI_SWIGLU_F8 ? EPI_SWIGLU
         : epi == EPI_BF16_F8 ? EPI_BF16
         : epi == EPI_F32_F8  ? EPI_F32
                              : epi;
}

struct Params {
  int E;
  const int32_t* offsets;
  int rows;          // permuted rows; offsets are clamped into [0, rows]
  int M;             // K-grouped: output rows per expert
  int N;             // output columns per B operand
  int kblocks;       // M-grouped: K blocks per operand pair
  int kconcat;       // M-grouped: 2 = after kblocks, continue with (a1, b1)
  int b_rows;        // rows per expert of the weight tensor viewed 2-D
  void* out0;
  void* out1;
  void* out2;
  const void* in0;
  const void* in1;
  const float* in2;  // EPI_SWIGLU_BWD_SAR: gate of each permuted row
  float* part;       // EPI_SWIGLU_BWD_SAR: per-(row, n-tile) partial sums of <H, dY W2^T>;
                     // EPI_SWIGLU_F8: per-(row, n-tile) amax of H;
                     // EPI_SWIGLU_BWD (optional): per-(row, n-tile) amax of dA and dB
  int part_ld;       // n-tiles per row of `part`
  const float* row_scale;   // FP8: scale of each A row (permuted row)
  const float* col_scale0;  // FP8: [E, N] scales of the B columns (first operand)
  const float* col_scale1;  // FP8: [E, N] scales of the second operand's columns
  int ldo;           // row stride (elements) of M-grouped outputs and inputs
  int* status;
  int ktiles;        // K-grouped: tiles in total
  int raster_n;      // tile order: 0 = groups of m-tiles, 1 = groups of n-tiles
  int group;         // tiles per group along that dimension
};

struct Maps {
  CUtensorMap a0, a1, b0, b1;
  // Outputs written by TMA from the epilogue's staging blocks (32 x 32 boxes):
  // fp32 (EPI_WGRAD, EPI_F32; 128B swizzle) or bf16 (the rest; 64B swizzle).
  CUtensorMap o0, o1, o2;
  // EPI_SWIGLU_BWD(_SAR): A and B [rows, f] bf16, 256 x 32 boxes, for the L2
  // prefetch of the next tile's rows
  CUtensorMap i0, i1;
  // EPI_SWIGLU_BWD on the CTA pair: A and B again, 32 x 32 boxes with 64B
  // swizzle (the layout of the dA / dB staging blocks), loaded by TMA into the
  // epilogue's staging sets
  CUtensorMap l0, l1;
};

struct Tile {
  int e, mb, nb;
  int row0;     // M-grouped: first permuted row; K-grouped: first K row
  int row_end;  // end of the expert's rows
  int nkb;      // K blocks
};

// Tile order inside one expert's MT x NT tile grid.  raster_n = 0: groups of
// `group` m-tiles, and within a group n-major, m fastest; raster_n = 1: the
// same with the roles of m and n swapped.  The ~152 tiles in flight at once
// then share the slabs of the grouped operand, which stay in L2 while the
// group sweeps the other operand once.  The host picks the orientation and the
// group so that, where one operand of an expert fits in L2, that operand stays
// resident and the other streams from DRAM exactly once.
__device__ __forceinline__ void raster(const Params& p, int local, int MT, int NT, int& mb,
                                       int& nb) {
  const int G = p.group;
  if (!p.raster_n) {
    const int g = local / (G * NT);
    const int base = g * G;
    const int gsz = min(G, MT - base);
    const int r = local - g * G * NT;
    nb = r / gsz;
    mb = base + r % gsz;
  } else {
    const int g = local / (G * MT);
    const int base = g * G;
    const int gsz = min(G, NT - base);
    const int r = local - g * G * MT;
    mb = r / gsz;
    nb = base + r % gsz;
  }
}

// Tile t of the launch -> expert, m-tile, n-tile and K range.  TM = rows per
// tile (128 for one CTA, 256 for a CTA pair); off = clamped expert offsets;
// cum = M-grouped prefix of m-tiles per expert.
template <int TM, bool GROUP_K, int NUM_B>
__device__ __forceinline__ bool decode(const Params& p, const int* off, const int* cum, int t,
                                       Tile& tl) {
  const int NT = (p.N + (BN / NUM_B) - 1) / (BN / NUM_B);
  if (!GROUP_K) {
    const int total = NT * cum[p.E];
    if (t >= total) return false;
    // the expert whose tiles hold t: the last e with NT cum[e] <= t, which has
    // rows (cum is non-decreasing and t < NT cum[E]).  A binary search: every
    // warp role decodes each of its tiles, and a scan over 64 experts in
    // shared memory cost up to a couple of thousand cycles per tile.
    int e = 0, hi = p.E - 1;
    while (e < hi) {
      const int mid = (e + hi + 1) >> 1;
      if (NT * cum[mid] <= t)
        e = mid;
      else
        hi = mid - 1;
    }
    const int local = t - NT * cum[e];
    const int mt = cum[e + 1] - cum[e];
    tl.e = e;
    raster(p, local, mt, NT, tl.mb, tl.nb);
    tl.row0 = off[e] + tl.mb * TM;
    tl.row_end = off[e + 1];
    tl.nkb = p.kblocks * p.kconcat;
  } else {
    if (t >= p.ktiles) return false;
    const int MT = (p.M + TM - 1) / TM;
    const int per = MT * NT;
    const int e = t / per;
    tl.e = e;
    raster(p, t - e * per, MT, NT, tl.mb, tl.nb);
    tl.row0 = off[e];
    tl.row_end = off[e + 1];
    tl.nkb = (tl.row_end - tl.row0 + BK - 1) / BK;
  }
  return true;
}

// sigmoid and silu for the SwiGLU epilogues, with CUDA's fast exponential and
// division intrinsics: their few-ulp error in fp32 is far below the bf16
// rounding of every value these epilogues store.  (For a < -88, __expf(-a)
// overflows to inf and both give 0, the limit.)
__device__ __forceinline__ float sigmoid_f(float a) { return __fdividef(1.0f, 1.0f + __expf(-a)); }
__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void store_bf16x32(void* dst, const float* v) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    d[i] = make_uint4(pack_bf16(v[8 * i + 0], v[8 * i + 1]), pack_bf16(v[8 * i + 2], v[8 * i + 3]),
                      pack_bf16(v[8 * i + 4], v[8 * i + 5]), pack_bf16(v[8 * i + 6], v[8 * i + 7]));
}

__device__ __forceinline__ void store_f32x32(void* dst, const float* v) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

// A warp's 32 consecutive rows x 32 fp32 columns (lane i holds row i in v) to
// global memory.  Written straight from the registers, every store
// instruction would touch 32 rows with 16 bytes each; instead the block goes
// to shared memory in the 128-byte-swizzled layout (16-byte piece j of row i
// in slot j ^ (i & 7), which also keeps the writes free of bank conflicts),
// and one TMA copy (map, box origin x, y) writes it out as whole rows while
// the warp goes on.  Two staging blocks alternate: before one is refilled,
// the copy that last read it must be done reading.  A block with rows that
// must stay untouched (bit clear in `ok`: past the expert's rows) is written
// by the warp itself instead, row i at dst0 + i * ld, four whole rows per
// instruction.
__device__ __forceinline__ void store_f32_block(float4* stage, int& nblk, const float* v,
                                                const CUtensorMap* map, int x, int y, float* dst0,
                                                size_t ld, unsigned ok, int lane) {
  float4* buf = stage + (nblk & 1) * (EPI_STAGE_BYTES / 16);
  ++nblk;
  if (lane == 0) bulk_wait_read_1();
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 8; ++j)
    buf[lane * 8 + (j ^ (lane & 7))] =
        make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  if (ok == 0xffffffffu) {
    fence_proxy_async_smem();  // the generic-proxy writes, seen by the copy
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map, smem_u32(buf), x, y);
      bulk_commit();
    }
    return;
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = i * 4 + (lane >> 3);
    const int c = lane & 7;
    const float4 q = buf[r * 8 + (c ^ (r & 7))];
    if ((ok >> r) & 1u) reinterpret_cast<float4*>(dst0 + static_cast<size_t>(r) * ld)[c] = q;
  }
  __syncwarp();
}

// Lane i's 32 values as bf16 into row i of a 32 x 32 block (2 KiB) in the
// layout of a TMA box {32, 32} with 64-byte swizzle: 16-byte piece j of row i
// in slot j ^ ((i >> 1) & 3), which also keeps the writes free of bank
// conflicts.
__device__ __forceinline__ void stage_bf16(uint4* buf, const float* v, int lane) {
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    buf[lane * 4 + (j ^ sw)] =
        make_uint4(pack_bf16(v[8 * j + 0], v[8 * j + 1]), pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                   pack_bf16(v[8 * j + 4], v[8 * j + 5]), pack_bf16(v[8 * j + 6], v[8 * j + 7]));
}

// NOUT bf16 outputs (x0 -> out0 / o0, x1 -> out1 / o1, x2 -> out2 / o2) of one
// 32-column chunk of a warp's 32 rows, lane i holding row grow0 + i.  With all
// 32 rows in range the blocks go through the warp's staging area and one TMA
// copy per output writes each (a store instruction from the registers would
// touch 32 rows with 16 bytes each); the warp does not wait for the copies,
// only, before it refills a staging set, for the copies that last read it.
// Otherwise (rows past the expert's end, which belong to the next expert)
// each lane in range stores its own row.
template <int NOUT>
__device__ __forceinline__ void store_bf16_chunk(const Params& p, const Maps& maps, uint4* stage,
                                                 int& nblk, int grow0, int col, bool row_ok,
                                                 const float* x0, const float* x1,
                                                 const float* x2, int lane) {
  const unsigned ok = __ballot_sync(0xffffffffu, row_ok);
  if (ok == 0xffffffffu) {
    constexpr int NSETS = NOUT <= 2 ? 2 : 1;  // staging sets in the warp's 8 KiB
    uint4* buf = stage + (nblk % NSETS) * (NOUT * 128);
    ++nblk;
    if (lane == 0) {
      if (NSETS == 2)
        bulk_wait_read_1();
      else
        bulk_wait_read_0();
    }
    __syncwarp();
    stage_bf16(buf, x0, lane);
    if (NOUT > 1) stage_bf16(buf + 128, x1, lane);
    if (NOUT > 2) stage_bf16(buf + 256, x2, lane);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&maps.o0, smem_u32(buf), col, grow0);
      if (NOUT > 1) tma_store_2d(&maps.o1, smem_u32(buf + 128), col, grow0);
      if (NOUT > 2) tma_store_2d(&maps.o2, smem_u32(buf + 256), col, grow0);
      bulk_commit();
    }
  } else if (row_ok) {
    const size_t o = static_cast<size_t>(grow0 + lane) * p.ldo + col;
    store_bf16x32(static_cast<__nv_bfloat16*>(p.out0) + o, x0);
    if (NOUT > 1) store_bf16x32(static_cast<__nv_bfloat16*>(p.out1) + o, x1);
    if (NOUT > 2) store_bf16x32(static_cast<__nv_bfloat16*>(p.out2) + o, x2);
  }
}

// The bf16-output forward epilogues (EPI_SWIGLU, EPI_BF16 and their FP8
// forms) on one 32-column chunk of a warp's 32 rows; v0 (and v1 for two B
// operands) are lane i's fp32 accumulator values for row grow0 + i.
template <int NUM_B, int EPI_>
__device__ __forceinline__ void bf16_chunk(const Params& p, const Maps& maps, uint4* stage,
                                           int& nblk, int grow0, int col, bool row_ok,
                                           const float* v0, const float* v1, float& acc,
                                           int lane) {
  constexpr int EPI = base_epi(EPI_);
  if constexpr (EPI == EPI_SWIGLU) {
    float hv[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) hv[i] = silu_f(v0[i]) * v1[i];
    if (EPI_ == EPI_SWIGLU_F8) {  // amax of H for its per-row e4m3 scale
#pragma unroll
      for (int i = 0; i < 32; ++i) acc = fmaxf(acc, fabsf(hv[i]));
    }
    store_bf16_chunk<3>(p, maps, stage, nblk, grow0, col, row_ok, v0, v1, hv, lane);
  } else {
    static_assert(EPI == EPI_BF16, "bf16_chunk serves the forward epilogues only");
    store_bf16_chunk<1>(p, maps, stage, nblk, grow0, col, row_ok, v0, v0, v0, lane);
  }
}

// Eight bf16 pairs (two 16-byte pieces x 4) -> 32 floats.
__device__ __forceinline__ void unpack_bf16x32(const uint4 (&q)[4], float* v) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
      v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
}

// dA = dH * B * s (1 + A (1 - s)), dB = dH * silu(A), s = sigmoid(A), on one
// lane's 32 values; with p.part, acc = the amax of the row's dA and dB.
__device__ __forceinline__ void swiglu_bwd_math(const Params& p, const float* v0, const float* av,
                                                const float* bv, float* da, float* db,
                                                float& acc) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float a = av[i];
    const float sg = sigmoid_f(a);
    const float dh = v0[i];
    da[i] = dh * bv[i] * sg * (1.0f + a * (1.0f - sg));
    db[i] = dh * a * sg;
  }
  if (p.part) {
#pragma unroll
    for (int i = 0; i < 32; ++i) acc = fmaxf(acc, fmaxf(fabsf(da[i]), fabsf(db[i])));
  }
}

// The SwiGLU-backward epilogues on a 32-column chunk of a warp's 32 rows (lane
// i: row grow0 + i) whose A and B values were loaded ahead (raw bf16).
//   EPI_SWIGLU_BWD: v0 = dH;  dA = dH * B * s (1 + A (1 - s)), dB = dH * silu(A)
//   with s = sigmoid(A); with p.part, acc = the amax of the row's dA and dB.
//   EPI_SWIGLU_BWD_SAR: v0 = u = dy_perm W2^T without the gate.  With the
//   row's gate g and H = silu(A) * B rebuilt from the kept A, B: dH = g u;
//   dA, dB as above; gH = g H (FC2 wgrad's operand, since dW2 = H^T (g dy) =
//   (g H)^T dy); acc += <H, u> (= <dy, O>).
template <int EPI>
__device__ __forceinline__ void swiglu_bwd_chunk(const Params& p, const Maps& maps, uint4* stage,
                                                 int& nblk, int grow0, int col, bool row_ok,
                                                 const float* v0, const uint4 (&ra)[4],
                                                 const uint4 (&rb)[4], float& acc, int lane) {
  float av[32], bv[32];
  unpack_bf16x32(ra, av);
  unpack_bf16x32(rb, bv);
  float da[32], db[32];
  if (EPI == EPI_SWIGLU_BWD) {
    swiglu_bwd_math(p, v0, av, bv, da, db, acc);
    store_bf16_chunk<2>(p, maps, stage, nblk, grow0, col, row_ok, da, db, db, lane);
  } else {
    const float g = row_ok ? __ldg(p.in2 + grow0 + lane) : 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float a = av[i];
      const float sg = sigmoid_f(a);
      const float sl = a * sg;
      const float hh = sl * bv[i];
      const float dh = g * v0[i];
      acc = fmaf(hh, v0[i], acc);
      da[i] = dh * bv[i] * sg * (1.0f + a * (1.0f - sg));
      db[i] = dh * sl;
      av[i] = g * hh;  // gH
    }
    store_bf16_chunk<3>(p, maps, stage, nblk, grow0, col, row_ok, da, db, av, lane);
  }
}

// EPI_SWIGLU_BWD on the CTA pair.  A TMA load put the chunk's A and B blocks
// (32 rows x 32 columns of bf16, 64B-swizzled) in the staging set `buf`: A at
// buf, B at buf + 128.  Lane i reads row i of both, and dA and dB are written
// over them (the same row, the same places, so no lane touches another's
// data) and stored from there by TMA.  Rows past the expert's end are stored
// by their lanes instead, and the set is then free at once.
__device__ __forceinline__ void swiglu_bwd_chunk_staged(const Params& p, const Maps& maps,
                                                        uint4* buf, int grow0, int col,
                                                        bool row_ok, const float* v0, float& acc,
                                                        int lane) {
  const int sw = (lane >> 1) & 3;
  uint4 ra[4], rb[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    ra[j] = buf[lane * 4 + (j ^ sw)];
    rb[j] = buf[128 + lane * 4 + (j ^ sw)];
  }
  float av[32], bv[32], da[32], db[32];
  unpack_bf16x32(ra, av);
  unpack_bf16x32(rb, bv);
  swiglu_bwd_math(p, v0, av, bv, da, db, acc);
  const unsigned ok = __ballot_sync(0xffffffffu, row_ok);
  if (ok == 0xffffffffu) {
    stage_bf16(buf, da, lane);
    stage_bf16(buf + 128, db, lane);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(&maps.o0, smem_u32(buf), col, grow0);
      tma_store_2d(&maps.o1, smem_u32(buf + 128), col, grow0);
      bulk_commit();
    }
  } else if (row_ok) {
    const size_t o = static_cast<size_t>(grow0 + lane) * p.ldo + col;
    store_bf16x32(static_cast<__nv_bfloat16*>(p.out0) + o, da);
    store_bf16x32(static_cast<__nv_bfloat16*>(p.out1) + o, db);
  }
}

// The SwiGLU-backward epilogue reads A and B of its tile's rows straight from
// DRAM one chunk ahead, which does not cover DRAM latency; so while tile t is
// in its epilogue, each warp asks the TMA unit to bring its 32 rows of the
// CTA's next tile into L2 (the main loop of that tile gives them time to land).
template <int BNB>
__device__ __forceinline__ void prefetch_ab_rows(const Maps& maps, const Tile& tn, int row_off) {
  tma_prefetch_l2_2d(&maps.i0, tn.nb * BNB, tn.row0 + row_off);
  tma_prefetch_l2_2d(&maps.i1, tn.nb * BNB, tn.row0 + row_off);
}

// The next chunk's A and B pieces (nothing for rows or columns out of range).
__device__ __forceinline__ void load_ab_chunk(const Params& p, bool ok, size_t o, uint4 (&ra)[4],
                                              uint4 (&rb)[4]) {
  if (!ok) return;
  const uint4* a = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.in0) + o);
  const uint4* b = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.in1) + o);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ra[i] = __ldg(a + i);
    rb[i] = __ldg(b + i);
  }
}

// FP8: the sums of e4m3 products times the row's and the columns' scales.
template <int NUM_B>
__device__ __forceinline__ void rescale_f8(const Params& p, const Tile& tl, int grow, int col,
                                           float* v0, float* v1) {
  const float sr = __ldg(p.row_scale + grow);
  const float* c0 = p.col_scale0 + static_cast<size_t>(tl.e) * p.N + col;
#pragma unroll
  for (int i = 0; i < 32; ++i) v0[i] *= sr * __ldg(c0 + i);
  if (NUM_B == 2) {
    const float* c1 = p.col_scale1 + static_cast<size_t>(tl.e) * p.N + col;
#pragma unroll
    for (int i = 0; i < 32; ++i) v1[i] *= sr * __ldg(c1 + i);
  }
}

// Weight gradient of an expert without tokens: zeros for this row's columns.
template <int NUM_B>
__device__ __forceinline__ void zero_wgrad_row(const Params& p, const Tile& tl, int orow) {
  constexpr int BNB = BN / NUM_B;
  if (orow >= p.M) return;
  float z[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) z[i] = 0.f;
  for (int ch = 0; ch < BNB / 32; ++ch) {
    const int col = tl.nb * BNB + ch * 32;
    if (col >= p.N) break;
    const size_t o = (static_cast<size_t>(tl.e) * p.M + orow) * p.N + col;
    store_f32x32(static_cast<float*>(p.out0) + o, z);
    if (NUM_B == 2) store_f32x32(static_cast<float*>(p.out1) + o, z);
  }
}

// Zero k-rows kv..63 of an MN-major 128-wide A tile (two 64-column chunks):
// they hold the next expert's rows (or the zero fill) and must add nothing.
// The rows past kv are contiguous in each chunk, so a lane clears 16-byte
// words i and i + 32 ... of both chunks with no index arithmetic beyond the
// stride (an earlier form divided by the chunk length per word, which put
// about a thousand cycles per ragged tile on the path to the MMA).
__device__ __forceinline__ void zero_a_tail(uint8_t* a_tile, int kv, int lane) {
  const int n = (BK - kv) * 8;  // 16-byte words per chunk
  uint4* c0 = reinterpret_cast<uint4*>(a_tile + kv * 128);
  uint4* c1 = reinterpret_cast<uint4*>(a_tile + CHUNK_BYTES + kv * 128);
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int i = lane; i < n; i += 32) {
    c0[i] = z;
    c1[i] = z;
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// The fp32 epilogues (EPI_WGRAD, EPI_F32) on one 32-column chunk of a warp's
// 32 rows.  grow0 / orow0: the M-grouped / K-grouped output row of lane 0.
// The output maps view dW as [E * M, N] and dX as [rows, ldo].
template <int NUM_B, int EPI>
__device__ __forceinline__ void fp32_rows_chunk(const Params& p, const Maps& maps, const Tile& tl,
                                                float4* stage, int& nblk, int grow0, int orow0,
                                                int col, bool row_ok, const float* v0,
                                                const float* v1, int lane) {
  const unsigned ok = __ballot_sync(0xffffffffu, row_ok);
  if (ok == 0u) return;
  if (EPI == EPI_WGRAD) {
    const int y = tl.e * p.M + orow0;
    const size_t o = static_cast<size_t>(y) * p.N + col;
    store_f32_block(stage, nblk, v0, &maps.o0, col, y, static_cast<float*>(p.out0) + o, p.N, ok,
                    lane);
    if (NUM_B == 2)
      store_f32_block(stage, nblk, v1, &maps.o1, col, y, static_cast<float*>(p.out1) + o, p.N,
                      ok, lane);
  } else {
    const size_t o = static_cast<size_t>(grow0) * p.ldo + col;
    store_f32_block(stage, nblk, v0, &maps.o0, col, grow0, static_cast<float*>(p.out0) + o,
                    p.ldo, ok, lane);
  }
}

template <bool A_MN, bool B_MN, int NUM_B, int EPI, bool GROUP_K>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gg_kernel(const __grid_constant__ Params p, const __grid_constant__ Maps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctrl& c = *reinterpret_cast<Ctrl*>(smem + STAGES * STAGE_BYTES + EPI_SMEM_BYTES);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int BNB = BN / NUM_B;  // accumulator columns per B operand
  constexpr bool F8 = is_f8(EPI);  // e4m3 operands (K-major only): 128 per 128-byte row
  constexpr int BKE = F8 ? 2 * BK : BK;  // K elements per stage
  static_assert(!F8 || (!A_MN && !B_MN && !GROUP_K), "FP8 matmuls take K-major operands");

  // ------------------------------------------------------------ set-up
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&c.full[s]), 1);
      mbar_init(smem_u32(&c.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&c.tfull[b]), 1);
      mbar_init(smem_u32(&c.tempty[b]), 128);
    }
    mbar_init(smem_u32(&c.drain), 1);
    c.abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&maps.a0);
    tma_prefetch_desc(&maps.b0);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&c.tmem_base), TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  if (warp >= 2) {
    for (int e = threadIdx.x - 64; e <= p.E; e += 128) {
      const int o = __ldg(p.offsets + e);
      c.off[e] = o < 0 ? 0 : (o > p.rows ? p.rows : o);
    }
  }
  __syncthreads();
  if (threadIdx.x == 64) {
    // ranges must not run backwards; this keeps every store inside its buffer
    for (int e = 1; e <= p.E; ++e) c.off[e] = max(c.off[e], c.off[e - 1]);
  }
  __syncthreads();
  if (!GROUP_K && threadIdx.x == 64) {
    c.cum[0] = 0;
    for (int e = 0; e < p.E; ++e) c.cum[e + 1] = c.cum[e] + (c.off[e + 1] - c.off[e] + BM - 1) / BM;
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  volatile int* abort_flag = &c.abort;

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      int q = 0;
      bool ok = true;
      Tile tl;
      for (int t = blockIdx.x; ok && decode<BM, GROUP_K, NUM_B>(p, c.off, c.cum, t, tl); t += gridDim.x) {
        for (int kb = 0; kb < tl.nkb; ++kb, ++q) {
          const int s = q % STAGES;
          const uint32_t ph = (q / STAGES) & 1;
          if (*abort_flag || !mbar_wait(smem_u32(&c.empty[s]), ph ^ 1, p.status, kTimeoutCode)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          const uint32_t full = smem_u32(&c.full[s]);
          mbar_expect_tx(full, STAGE_BYTES);
          const uint32_t a_dst = smem_u32(smem + s * STAGE_BYTES);
          const uint32_t b_dst = a_dst + A_BYTES;
          if (!GROUP_K) {
            const bool second = p.kconcat == 2 && kb >= p.kblocks;
            const int kx = (second ? kb - p.kblocks : kb) * BKE;
            tma_load_2d(a_dst, second ? &maps.a1 : &maps.a0, kx, tl.row0, full);
            if (!B_MN) {
              // FP8 FC1: one 256-row tile of the interleaved W1/W3 operand
              tma_load_2d(b_dst, second ? &maps.b1 : &maps.b0, kx,
                          tl.e * p.b_rows + tl.nb * (F8 ? BN : BNB), full);
            } else {
              // MN-major: one 3-D copy fills the BNB / 64 column chunks of an operand
#pragma unroll
              for (int i = 0; i < NUM_B; ++i)
                tma_load_3d(b_dst + i * (B_BYTES / NUM_B), i ? &maps.b1 : &maps.b0, 0,
                            tl.e * p.b_rows + kx, tl.nb * (BNB / 64), full);
            }
          } else {
            const int ky = tl.row0 + kb * BK;
            tma_load_3d(a_dst, &maps.a0, 0, ky, tl.mb * (BM / 64), full);
#pragma unroll
            for (int i = 0; i < NUM_B; ++i)
              tma_load_3d(b_dst + i * (B_BYTES / NUM_B), i ? &maps.b1 : &maps.b0, 0, ky,
                          tl.nb * (BNB / 64), full);
          }
        }
      }
      if (!ok) {
        // let every load already issued land before the CTA can exit
        const int first = q > STAGES ? q - STAGES : 0;
        for (int r = first; r < q; ++r)
          mbar_wait(smem_u32(&c.full[r % STAGES]), (r / STAGES) & 1, p.status, kTimeoutCode);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    // MN-major B tiles are stored as 64-column chunks 8 KiB apart, so the two
    // 128-column operands of NUM_B = 2 form one 256-column operand: a single
    // N = 256 MMA fills both accumulators and reads the A tile once per K step.
    constexpr bool B_FUSED = B_MN || NUM_B == 1 || F8;
    constexpr uint32_t IDESC =
        F8 ? idesc_e4m3(BM, BN) : idesc_bf16(BM, B_FUSED ? BN : BNB, A_MN, B_MN);
    constexpr uint32_t A_LBO = A_MN ? CHUNK_BYTES : 16;
    constexpr uint32_t B_LBO = B_MN ? CHUNK_BYTES : 16;
    constexpr uint32_t A_KSTEP = A_MN ? 2048 : 32;  // bytes per 16-deep K step
    constexpr uint32_t B_KSTEP = B_MN ? 2048 : 32;
    int q = 0, it = 0;
    bool ok = true;
    Tile tl;
    for (int t = blockIdx.x; ok && decode<BM, GROUP_K, NUM_B>(p, c.off, c.cum, t, tl); t += gridDim.x) {
      if (tl.nkb == 0) continue;
      const int buf = it & 1;
      const uint32_t u = (it >> 1) & 1;
      ++it;
      if (*abort_flag || !mbar_wait(smem_u32(&c.tempty[buf]), u ^ 1, p.status, kTimeoutCode)) {
        *abort_flag = 1;
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem_base + buf * BN;
      for (int kb = 0; kb < tl.nkb; ++kb, ++q) {
        const int s = q % STAGES;
        const uint32_t ph = (q / STAGES) & 1;
        if (*abort_flag || !mbar_wait(smem_u32(&c.full[s]), ph, p.status, kTimeoutCode)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        uint8_t* a_tile = smem + s * STAGE_BYTES;
        if (GROUP_K) {
          const int kv = tl.row_end - (tl.row0 + kb * BK);
          if (kv < BK) zero_a_tail(a_tile, kv, lane);
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t a_base = smem_u32(a_tile);
          const uint32_t b_base = a_base + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = smem_desc(a_base + kk * A_KSTEP, A_LBO, 1024);
            if (F8) {
              umma_e4m3(acc, ad, smem_desc(b_base + kk * B_KSTEP, B_LBO, 1024), IDESC,
                        (kb | kk) != 0);
            } else if (B_FUSED) {
              umma_bf16(acc, ad, smem_desc(b_base + kk * B_KSTEP, B_LBO, 1024), IDESC,
                        (kb | kk) != 0);
            } else {
#pragma unroll
              for (int i = 0; i < NUM_B; ++i) {
                const uint64_t bd =
                    smem_desc(b_base + i * (B_BYTES / NUM_B) + kk * B_KSTEP, B_LBO, 1024);
                umma_bf16(acc + i * BNB, ad, bd, IDESC, (kb | kk) != 0);
              }
            }
          }
          umma_commit(smem_u32(&c.empty[s]));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) umma_commit(smem_u32(&c.tfull[buf]));
      __syncwarp();
    }
    // every MMA this thread issued must finish before tensor memory is freed
    if (lane == 0) {
      umma_commit(smem_u32(&c.drain));
      mbar_wait(smem_u32(&c.drain), 0, p.status, kTimeoutCode);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    const int r = quarter * 32 + lane;
    float4* stage =
        reinterpret_cast<float4*>(smem + STAGES * STAGE_BYTES + (warp - 2) * 2 * EPI_STAGE_BYTES);
    int nblk = 0;  // fp32 blocks this warp has staged
    int it = 0;
    Tile tl;
    if constexpr (EPI == EPI_SWIGLU_BWD || EPI == EPI_SWIGLU_BWD_SAR) {
      Tile tn;
      if (lane == 0 && decode<BM, GROUP_K, NUM_B>(p, c.off, c.cum, blockIdx.x, tn))
        prefetch_ab_rows<BNB>(maps, tn, quarter * 32);
    }
    for (int t = blockIdx.x; decode<BM, GROUP_K, NUM_B>(p, c.off, c.cum, t, tl); t += gridDim.x) {
      // every decision to stop is taken by the whole warp: the TMEM loads and
      // the staged stores below are warp-collective
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      if constexpr (EPI == EPI_SWIGLU_BWD || EPI == EPI_SWIGLU_BWD_SAR) {
        Tile tn;
        if (lane == 0 && decode<BM, GROUP_K, NUM_B>(p, c.off, c.cum, t + gridDim.x, tn))
          prefetch_ab_rows<BNB>(maps, tn, quarter * 32);
      }
      if (GROUP_K && tl.nkb == 0) {  // expert without tokens: zero weight gradient
        zero_wgrad_row<NUM_B>(p, tl, tl.mb * BM + r);
        continue;
      }
      const int buf = it & 1;
      const uint32_t u = (it >> 1) & 1;
      ++it;
      const bool filled = mbar_wait(smem_u32(&c.tfull[buf]), u, p.status, kTimeoutCode);
      if (!__all_sync(0xffffffffu, filled)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + buf * BN + (static_cast<uint32_t>(quarter * 32) << 16);
      const int grow = tl.row0 + r;                        // M-grouped row
      const bool row_ok = GROUP_K ? (tl.mb * BM + r < p.M) : (grow < tl.row_end);
      float acc = 0.f;
      if constexpr (EPI == EPI_SWIGLU_BWD || EPI == EPI_SWIGLU_BWD_SAR) {
        // A and B of chunk ch + 1 are in flight while chunk ch is computed
        const size_t o0 = static_cast<size_t>(grow) * p.ldo + tl.nb * BNB;
        uint4 ra[4], rb[4];
        load_ab_chunk(p, row_ok && tl.nb * BNB < p.N, o0, ra, rb);
#pragma unroll 1
        for (int ch = 0; ch < BNB / 32; ++ch) {
          uint4 ca[4], cb[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            ca[i] = ra[i];
            cb[i] = rb[i];
          }
          const int col = tl.nb * BNB + ch * 32;
          if (ch + 1 < BNB / 32)
            load_ab_chunk(p, row_ok && col + 32 < p.N, o0 + (ch + 1) * 32, ra, rb);
          float v0[32];
          tmem_ld32(tbase + ch * 32, v0);
          if (col >= p.N) continue;  // the same for the whole warp
          swiglu_bwd_chunk<EPI>(p, maps, reinterpret_cast<uint4*>(stage), nblk, grow - lane, col,
                                row_ok, v0, ca, cb, acc, lane);
        }
      } else {
#pragma unroll 1
        for (int ch = 0; ch < BNB / 32; ++ch) {
          float v0[32];
          float v1[32];
          tmem_ld32(tbase + ch * 32, v0);
          if (NUM_B == 2) tmem_ld32(tbase + BNB + ch * 32, v1);
          const int col = tl.nb * BNB + ch * 32;
          if constexpr (EPI == EPI_WGRAD || base_epi(EPI) == EPI_F32) {
            if (col >= p.N) continue;  // the same for the whole warp
            if (is_f8(EPI) && row_ok) rescale_f8<NUM_B>(p, tl, grow, col, v0, v1);
            fp32_rows_chunk<NUM_B, EPI>(p, maps, tl, stage, nblk, grow - lane,
                                        tl.mb * BM + quarter * 32, col, row_ok, v0, v1, lane);
          } else {
            if (col >= p.N) continue;  // the same for the whole warp
            if (is_f8(EPI) && row_ok) rescale_f8<NUM_B>(p, tl, grow, col, v0, v1);
            bf16_chunk<NUM_B, EPI>(p, maps, reinterpret_cast<uint4*>(stage), nblk, grow - lane,
                                   col, row_ok, v0, v1, acc, lane);
          }
        }
      }
      if ((EPI == EPI_SWIGLU_BWD_SAR || EPI == EPI_SWIGLU_F8 ||
           (EPI == EPI_SWIGLU_BWD && p.part)) && row_ok)
        p.part[static_cast<size_t>(grow) * p.part_ld + tl.nb] = acc;
      tc_fence_before();
      mbar_arrive(smem_u32(&c.tempty[buf]));
    }
    if (lane == 0) bulk_wait_all();  // staged fp32 blocks written out before the CTA ends
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ========================================================= CTA-pair kernel
// Two CTAs of a cluster compute one 256 x 256 tile with tcgen05.mma.cta_group::2:
// CTA r stages rows [128 r, 128 r + 128) of the A tile and B columns
// [128 r, 128 r + 128) in its own shared memory; the even CTA's single issuer
// thread runs the MMAs for both, and each CTA's TMEM holds its 128 rows of the
// 256-column accumulator.  Per SM this halves the B bytes staged and read per
// MAC (a 32 KiB stage feeds 128 x 256 x 64 MACs instead of 48 KiB), so the
// same ring of stages covers more MMA time.  Measured on GB300, the pair is
// 1-3.5% faster than the one-CTA kernel on every matmul but FC1 forward (see
// pair_for below).
// Synchronisation: the even CTA's `full` barrier counts both CTAs' bytes: its
// own loads signal it directly, and the odd CTA's loads signal it across the
// pair (TMA .cta_group::2).  The exception is the last K block of a wgrad tile
// whose rows run into the next expert: each CTA then loads it against its own
// `tailbar`, and its relay warp (warp 6) waits for the bytes, clears the
// stale k-rows and arrives on the even CTA's `full` (count 2: the even
// producer's two arrivals for a plain block, the two relays for such a
// block).  Clearing there, rather than in the issuer, keeps the issuer's
// stream of MMAs free of stores and proxy fences: measured on GB300, the
// issuer-side clearing cost the wgrads about 5%.  The issuer's commits are
// multicast to the `empty` and `tfull` barriers of both CTAs; all eight
// epilogue warps arrive on the even CTA's `tempty` barrier.
constexpr int PM = 256;                           // rows of a pair tile
constexpr int STAGES2 = 6;
constexpr int A2_BYTES = 128 * BK * 2;            // this CTA's 128 rows: 16 KiB
constexpr int B2_BYTES = 128 * BK * 2;            // this CTA's 128 columns: 16 KiB
constexpr int STAGE2_BYTES = A2_BYTES + B2_BYTES;  // 32 KiB
constexpr int NUM_THREADS2 = NUM_THREADS + 32;     // the one-CTA roles plus the relay warp

struct alignas(8) Ctrl2 {
  uint64_t full[STAGES2];
  uint64_t empty[STAGES2];
  uint64_t tailbar[STAGES2];  // wgrad K blocks that run past the expert (see above)
  uint64_t abar[4][2];        // EPI_SWIGLU_BWD: A/B block loads into each epilogue warp's sets
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int off[MAX_E + 1];
  int cum[MAX_E + 1];
};
constexpr int SMEM2_BYTES =
    1024 + STAGES2 * STAGE2_BYTES + EPI_SMEM_BYTES + static_cast<int>(sizeof(Ctrl2));
static_assert(SMEM2_BYTES <= 232448, "pair kernel exceeds the 227 KiB shared-memory limit");
static_assert(SMEM_BYTES <= 232448, "one-CTA kernel exceeds the 227 KiB shared-memory limit");

template <bool A_MN, bool B_MN, int NUM_B, int EPI, bool GROUP_K>
__global__ void __launch_bounds__(NUM_THREADS2, 1)
    gg2_kernel(const __grid_constant__ Params p, const __grid_constant__ Maps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctrl2& c = *reinterpret_cast<Ctrl2*>(smem + STAGES2 * STAGE2_BYTES + EPI_SMEM_BYTES);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();     // 0: issues the MMAs of the pair
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(cluster_count_x());
  constexpr int BNB = BN / NUM_B;
  constexpr bool F8 = is_f8(EPI);  // e4m3 operands (K-major only): 128 per 128-byte row
  constexpr int BKE = F8 ? 2 * BK : BK;  // K elements per stage
  static_assert(!F8 || (!A_MN && !B_MN && !GROUP_K), "FP8 matmuls take K-major operands");

  // ------------------------------------------------------------ set-up
  if (warp == 0 && lane == 0) {
    for (int s = 0; s < STAGES2; ++s) {
      mbar_init(smem_u32(&c.full[s]), rank == 0 ? 2 : 1);
      mbar_init(smem_u32(&c.empty[s]), 1);
      mbar_init(smem_u32(&c.tailbar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&c.tfull[b]), 1);
      mbar_init(smem_u32(&c.tempty[b]), 8);
    }
    for (int w = 0; w < 4; ++w) {
      mbar_init(smem_u32(&c.abar[w][0]), 1);
      mbar_init(smem_u32(&c.abar[w][1]), 1);
    }
    mbar_init(smem_u32(&c.drain), 1);
    c.abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&maps.a0);
    tma_prefetch_desc(&maps.b0);
  }
  if (warp == 1) {
    tmem_alloc2(smem_u32(&c.tmem_base), TMEM_COLS);
    tmem_relinquish2();
    tc_fence_before();
  }
  if (warp >= 2 && warp < 6) {
    for (int e = threadIdx.x - 64; e <= p.E; e += 128) {
      const int o = __ldg(p.offsets + e);
      c.off[e] = o < 0 ? 0 : (o > p.rows ? p.rows : o);
    }
  }
  __syncthreads();
  if (threadIdx.x == 64) {
    for (int e = 1; e <= p.E; ++e) c.off[e] = max(c.off[e], c.off[e - 1]);
    if (!GROUP_K) {
      c.cum[0] = 0;
      for (int e = 0; e < p.E; ++e) c.cum[e + 1] = c.cum[e] + (c.off[e + 1] - c.off[e] + PM - 1) / PM;
    }
  }
  cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA arrive
  tc_fence_after();
  const uint32_t tmem_base = c.tmem_base;
  volatile int* abort_flag = &c.abort;
  const uint32_t peer_abort = mapa_shared(smem_u32(&c.abort), rank ^ 1u);
  auto give_up = [&]() {
    *abort_flag = 1;
    st_cluster_u32(peer_abort, 1);
  };

  if (warp == 0) {
    // ------------------------------------------------------- TMA producer
    if (lane == 0) {
      int q = 0;
      bool ok = true;
      Tile tl;
      for (int t = cid; ok && decode<PM, GROUP_K, NUM_B>(p, c.off, c.cum, t, tl); t += ncl) {
        for (int kb = 0; kb < tl.nkb; ++kb, ++q) {
          const int s = q % STAGES2;
          const uint32_t ph = (q / STAGES2) & 1;
          if (*abort_flag || !mbar_wait(smem_u32(&c.empty[s]), ph ^ 1, p.status, kTimeoutCode)) {
            give_up();
            ok = false;
            break;
          }
          // a wgrad K block whose rows run past the expert needs its stale
          // rows cleared in both CTAs before the MMA (see the relay below)
          const bool tail = GROUP_K && tl.row_end - (tl.row0 + kb * BK) < BK;
          const uint32_t own_full = smem_u32(&c.full[s]);
          uint32_t bar;  // where this CTA's loads complete
          if (tail) {
            bar = smem_u32(&c.tailbar[s]);  // the relay warp takes it from here
            mbar_expect_tx(bar, STAGE2_BYTES);
          } else if (rank == 0) {
            bar = own_full;
            mbar_expect_tx(own_full, 2 * STAGE2_BYTES);  // both CTAs' bytes
            mbar_arrive(own_full);
          } else {
            bar = mapa_shared(own_full, 0);
          }
          const bool cross = rank != 0 && !tail;
          auto load = [&](uint32_t dst, const CUtensorMap* m, int x, int y) {
            if (cross)
              tma_load_2d_pair(dst, m, x, y, bar);
            else
              tma_load_2d(dst, m, x, y, bar);
          };
          // MN-major operands: one 3-D copy of two 64-column chunks
          auto load_mn = [&](uint32_t dst, const CUtensorMap* m, int y, int chunk) {
            if (cross)
              tma_load_3d_pair(dst, m, 0, y, chunk, bar);
            else
              tma_load_3d(dst, m, 0, y, chunk, bar);
          };
          const uint32_t a_dst = smem_u32(smem + s * STAGE2_BYTES);
          const uint32_t b_dst = a_dst + A2_BYTES;
          // B columns of this CTA: the second operand for NUM_B = 2 (W3 / dB),
          // else the upper 128 of the 256
          const CUtensorMap* bmap = (NUM_B == 2 && rank) ? &maps.b1 : &maps.b0;
          const int bcol = NUM_B == 2 ? tl.nb * BNB : tl.nb * BN + 128 * static_cast<int>(rank);
          if (!GROUP_K) {
            const bool second = p.kconcat == 2 && kb >= p.kblocks;
            const int kx = (second ? kb - p.kblocks : kb) * BKE;
            load(a_dst, second ? &maps.a1 : &maps.a0, kx, tl.row0 + 128 * static_cast<int>(rank));
            if (!B_MN) {
              load(b_dst, second ? &maps.b1 : &maps.b0, kx,
                   tl.e * p.b_rows + tl.nb * BN + 128 * static_cast<int>(rank));
            } else {
              load_mn(b_dst, bmap, tl.e * p.b_rows + kx, bcol / 64);
            }
          } else {
            const int ky = tl.row0 + kb * BK;
            load_mn(a_dst, &maps.a0, ky, (tl.mb * PM + 128 * static_cast<int>(rank)) / 64);
            load_mn(b_dst, bmap, ky, bcol / 64);
          }
        }
      }
      if (!ok && rank == 0) {
        // let the loads already issued land before the CTA can exit
        const int first = q > STAGES2 ? q - STAGES2 : 0;
        for (int r = first; r < q; ++r)
          mbar_wait_cluster(smem_u32(&c.full[r % STAGES2]), (r / STAGES2) & 1, p.status,
                            kTimeoutCode);
      }
    }
  } else if (warp == 1) {
    if (rank == 0) {
      // ----------------------------------------------- MMA issuer (even CTA)
      constexpr uint32_t IDESC = F8 ? idesc_e4m3(PM, BN) : idesc_bf16(PM, BN, A_MN, B_MN);
      constexpr uint32_t A_LBO = A_MN ? CHUNK_BYTES : 16;
      constexpr uint32_t B_LBO = B_MN ? CHUNK_BYTES : 16;
      constexpr uint32_t A_KSTEP = A_MN ? 2048 : 32;
      constexpr uint32_t B_KSTEP = B_MN ? 2048 : 32;
      int q = 0, it = 0;
      bool ok = true;
      Tile tl;
      for (int t = cid; ok && decode<PM, GROUP_K, NUM_B>(p, c.off, c.cum, t, tl); t += ncl) {
        if (tl.nkb == 0) continue;
        const int buf = it & 1;
        const uint32_t u = (it >> 1) & 1;
        ++it;
        if (*abort_flag || !mbar_wait(smem_u32(&c.tempty[buf]), u ^ 1, p.status, kTimeoutCode)) {
          give_up();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem_base + buf * BN;
        for (int kb = 0; kb < tl.nkb; ++kb, ++q) {
          const int s = q % STAGES2;
          const uint32_t ph = (q / STAGES2) & 1;
          if (*abort_flag || !mbar_wait(smem_u32(&c.full[s]), ph, p.status, kTimeoutCode)) {
            give_up();
            ok = false;
            break;
          }
          uint8_t* a_tile = smem + s * STAGE2_BYTES;
          if (lane == 0) {
            tc_fence_after();
            const uint32_t a_base = smem_u32(a_tile);
            const uint32_t b_base = a_base + A2_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = smem_desc(a_base + kk * A_KSTEP, A_LBO, 1024);
              const uint64_t bd = smem_desc(b_base + kk * B_KSTEP, B_LBO, 1024);
              if (F8)
                umma2_e4m3(acc, ad, bd, IDESC, (kb | kk) != 0);
              else
                umma2_bf16(acc, ad, bd, IDESC, (kb | kk) != 0);
            }
            umma2_commit_mc(smem_u32(&c.empty[s]), 0x3);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) umma2_commit_mc(smem_u32(&c.tfull[buf]), 0x3);
        __syncwarp();
      }
      if (lane == 0) {
        umma2_commit(smem_u32(&c.drain));
        mbar_wait(smem_u32(&c.drain), 0, p.status, kTimeoutCode);
      }
      __syncwarp();
    }
  } else if (warp == 6) {
    // ----------------------------------------------- relay (both CTAs)
    // Only wgrad tiles whose last K block runs into the next expert need it:
    // that block was loaded against this CTA's `tailbar`.
    if (GROUP_K) {
      int q = 0;
      uint32_t phase_bits = 0;  // completed phases of each `tailbar`
      Tile tl;
      const uint32_t full0 = rank == 0 ? 0u : 1u;  // 0: arrive locally
      for (int t = cid; decode<PM, GROUP_K, NUM_B>(p, c.off, c.cum, t, tl); t += ncl) {
        if (tl.nkb == 0) continue;
        const int last = q + tl.nkb - 1;
        q += tl.nkb;
        const int kv = tl.row_end - (tl.row0 + (tl.nkb - 1) * BK);
        if (kv >= BK) continue;
        const int s = last % STAGES2;
        const uint32_t ph = (phase_bits >> s) & 1u;
        phase_bits ^= 1u << s;
        if (*abort_flag || !mbar_wait(smem_u32(&c.tailbar[s]), ph, p.status, kTimeoutCode)) {
          give_up();
          break;
        }
        zero_a_tail(smem + s * STAGE2_BYTES, kv, lane);
        if (lane == 0) {
          if (full0 == 0)
            mbar_arrive(smem_u32(&c.full[s]));
          else
            mbar_arrive_cluster(mapa_shared(smem_u32(&c.full[s]), 0));
        }
        __syncwarp();
      }
    }
  } else {
    // ------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;             // TMEM lane = row within this CTA's half
    const int half = 128 * static_cast<int>(rank);
    float4* stage = reinterpret_cast<float4*>(smem + STAGES2 * STAGE2_BYTES +
                                              (warp - 2) * 2 * EPI_STAGE_BYTES);
    int nblk = 0;
    int it = 0;
    Tile tl;
    // The L2 prefetch of the next tile's A / B rows serves the SAR form, whose
    // lanes load them one chunk ahead.  The TMA-loaded form runs faster without
    // it (measured on GB300: FC2 dgrad 2.67 against 2.75 ms).
    if constexpr (EPI == EPI_SWIGLU_BWD_SAR) {
      Tile tn;
      if (lane == 0 && decode<PM, GROUP_K, NUM_B>(p, c.off, c.cum, cid, tn))
        prefetch_ab_rows<BNB>(maps, tn, half + quarter * 32);
    }
    // EPI_SWIGLU_BWD: each chunk's A and B blocks come by TMA into one of the
    // warp's two 4 KiB staging sets, one chunk ahead (the last chunk of a tile
    // asks for the first of the CTA's next tile); see swiglu_bwd_chunk_staged.
    // Load n goes to set n & 1 and completes phase (n >> 1) & 1 of its barrier.
    constexpr bool kStagedAB = EPI == EPI_SWIGLU_BWD;
    uint4* sets = reinterpret_cast<uint4*>(stage);
    int lq = 0;  // A/B block loads issued
    int lw = 0;  // and waited for
    auto ab_bar = [&](int n) { return smem_u32(&c.abar[warp - 2][n & 1]); };
    auto issue_ab = [&](int col, int row) {
      fence_proxy_async_smem();  // the warp's reads of the set come before the refill
      __syncwarp();
      if (lane == 0) {
        bulk_wait_read_0();  // and so does the TMA store that last read it
        mbar_expect_tx(ab_bar(lq), 4096);
        tma_load_2d(smem_u32(sets + (lq & 1) * 256), &maps.l0, col, row, ab_bar(lq));
        tma_load_2d(smem_u32(sets + (lq & 1) * 256 + 128), &maps.l1, col, row, ab_bar(lq));
      }
      __syncwarp();
      ++lq;
    };
    if constexpr (kStagedAB) {
      Tile t0;
      if (decode<PM, GROUP_K, NUM_B>(p, c.off, c.cum, cid, t0))
        issue_ab(t0.nb * BNB, t0.row0 + half + quarter * 32);
    }
    for (int t = cid; decode<PM, GROUP_K, NUM_B>(p, c.off, c.cum, t, tl); t += ncl) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;  // warp-wide, as above
      if constexpr (EPI == EPI_SWIGLU_BWD_SAR) {
        Tile tn;
        if (lane == 0 && decode<PM, GROUP_K, NUM_B>(p, c.off, c.cum, t + ncl, tn))
          prefetch_ab_rows<BNB>(maps, tn, half + quarter * 32);
      }
      const int orow = tl.mb * PM + half + r;       // K-grouped output row
      if (GROUP_K && tl.nkb == 0) {
        zero_wgrad_row<NUM_B>(p, tl, orow);
        continue;
      }
      const int buf = it & 1;
      const uint32_t u = (it >> 1) & 1;
      ++it;
      const bool filled = mbar_wait(smem_u32(&c.tfull[buf]), u, p.status, kTimeoutCode);
      if (!__all_sync(0xffffffffu, filled)) {
        give_up();
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + buf * BN + (static_cast<uint32_t>(quarter * 32) << 16);
      const int grow = tl.row0 + half + r;           // M-grouped row
      const bool row_ok = GROUP_K ? (orow < p.M) : (grow < tl.row_end);
      float acc = 0.f;
      if constexpr (kStagedAB) {
        Tile tn;
        const bool has_next = decode<PM, GROUP_K, NUM_B>(p, c.off, c.cum, t + ncl, tn);
        bool lost = false;
#pragma unroll 1
        for (int ch = 0; ch < BNB / 32; ++ch) {
          const int col = tl.nb * BNB + ch * 32;
          const int n = lw++;
          const bool got = mbar_wait(ab_bar(n), (n >> 1) & 1, p.status, kTimeoutCode);
          if (!__all_sync(0xffffffffu, got)) {
            lost = true;
            break;
          }
          if (ch + 1 < BNB / 32)
            issue_ab(col + 32, grow - lane);
          else if (has_next)
            issue_ab(tn.nb * BNB, tn.row0 + half + quarter * 32);
          float v0[32];
          tmem_ld32(tbase + ch * 32, v0);
          if (col >= p.N) continue;  // the same for the whole warp
          swiglu_bwd_chunk_staged(p, maps, sets + (n & 1) * 256, grow - lane, col, row_ok, v0,
                                  acc, lane);
        }
        if (lost) {
          give_up();
          break;
        }
      } else if constexpr (EPI == EPI_SWIGLU_BWD_SAR) {
        // A and B of chunk ch + 1 are in flight while chunk ch is computed
        const size_t o0 = static_cast<size_t>(grow) * p.ldo + tl.nb * BNB;
        uint4 ra[4], rb[4];
        load_ab_chunk(p, row_ok && tl.nb * BNB < p.N, o0, ra, rb);
#pragma unroll 1
        for (int ch = 0; ch < BNB / 32; ++ch) {
          uint4 ca[4], cb[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            ca[i] = ra[i];
            cb[i] = rb[i];
          }
          const int col = tl.nb * BNB + ch * 32;
          if (ch + 1 < BNB / 32)
            load_ab_chunk(p, row_ok && col + 32 < p.N, o0 + (ch + 1) * 32, ra, rb);
          float v0[32];
          tmem_ld32(tbase + ch * 32, v0);
          if (col >= p.N) continue;  // the same for the whole warp
          swiglu_bwd_chunk<EPI>(p, maps, reinterpret_cast<uint4*>(stage), nblk, grow - lane, col,
                                row_ok, v0, ca, cb, acc, lane);
        }
      } else {
#pragma unroll 1
        for (int ch = 0; ch < BNB / 32; ++ch) {
          float v0[32];
          float v1[32];
          tmem_ld32(tbase + ch * 32, v0);
          if (NUM_B == 2) tmem_ld32(tbase + BNB + ch * 32, v1);
          const int col = tl.nb * BNB + ch * 32;
          if constexpr (EPI == EPI_WGRAD || base_epi(EPI) == EPI_F32) {
            if (col >= p.N) continue;  // the same for the whole warp
            if (is_f8(EPI) && row_ok) rescale_f8<NUM_B>(p, tl, grow, col, v0, v1);
            fp32_rows_chunk<NUM_B, EPI>(p, maps, tl, stage, nblk, grow - lane, orow - lane, col,
                                        row_ok, v0, v1, lane);
          } else {
            if (col >= p.N) continue;  // the same for the whole warp
            if (is_f8(EPI) && row_ok) rescale_f8<NUM_B>(p, tl, grow, col, v0, v1);
            bf16_chunk<NUM_B, EPI>(p, maps, reinterpret_cast<uint4*>(stage), nblk, grow - lane,
                                   col, row_ok, v0, v1, acc, lane);
          }
        }
      }
      if ((EPI == EPI_SWIGLU_BWD_SAR || EPI == EPI_SWIGLU_F8 ||
           (EPI == EPI_SWIGLU_BWD && p.part)) && row_ok)
        p.part[static_cast<size_t>(grow) * p.part_ld + tl.nb] = acc;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&c.tempty[buf]), 0));
    }
    if constexpr (kStagedAB) {  // an A/B load still in flight (after an abort)
      while (lw < lq && mbar_wait(ab_bar(lw), (lw >> 1) & 1, p.status, kTimeoutCode)) ++lw;
    }
    if (lane == 0) bulk_wait_all();  // staged fp32 blocks written out before the CTA ends
  }

  // ------------------------------------------------------------ teardown
  __syncthreads();
  cluster_sync_all();  // the pair's MMAs and TMEM reads are finished
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc2(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<EncodeTiledFn>(ptr);
  }();
  return fn;
}

// bf16 matrix [outer, inner] (row-major), box {box_inner, box_outer}, 128B swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
              uint32_t box_inner, uint32_t box_outer, bool bytes = false) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * (bytes ? 1 : 2)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MN-major operand: bf16 matrix [outer, inner] (row-major, inner a multiple of
// 64) viewed as {64, outer, inner / 64}, so that one box of {64, box_outer,
// chunks} copies `chunks` 64-column chunks of box_outer rows, 128B swizzle.
bool make_map_mn(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                 uint32_t box_outer, uint32_t chunks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || inner % 64 != 0) return false;
  cuuint64_t dims[3] = {64, outer, inner / 64};
  cuuint64_t strides[2] = {inner * 2, 128};
  cuuint32_t box[3] = {64, box_outer, chunks};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 output [outer, inner] (row-major) for the epilogue's TMA stores: 32 x 32
// boxes, 128B swizzle (one 128-byte row of 32 floats per box row).
bool make_map_out(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [outer, inner] (row-major) in 32 x 32 boxes, 64B swizzle (one 64-byte
// row of 32 values per box row): the epilogue's TMA stores, and the A / B block
// loads of the pair's SwiGLU-backward epilogue.
bool make_map_out_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [outer, inner] for L2 prefetches of 256 x 32 boxes.
bool make_map_prefetch(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(inner < 256 ? inner : 256), 32};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Which kernel runs each matmul.  Measured on GB300 (Mixtral-8x7B-shaped
// layer): the CTA pair is as fast or faster for every matmul but FC1 forward
// (bf16: wgrads 2-3%, FC2 forward 1%; e4m3: FC1 dgrad 3.5%, FC2 forward 2%).
// FC1 forward runs 2-3% faster on the one-CTA kernel, in bf16 and e4m3: its
// 256-row pair tiles waste more rows at each expert's end.  MOE_GEMM_CTAS=1
// or =2 forces one kind for every matmul (for measurement).
int forced_ctas() {
  static const int v = [] {
    const char* e = getenv("MOE_GEMM_CTAS");
    return (e && (e[0] == '1' || e[0] == '2')) ? e[0] - '0' : 0;
  }();
  return v;
}
bool pair_for(int epi) {
  if (forced_ctas()) return forced_ctas() == 2;
  return epi != EPI_SWIGLU && epi != EPI_SWIGLU_F8;
}

// Co-resident clusters of CTA pairs for a pair kernel on the current device,
// computed once per (kernel, device); safe from several host threads.
int coresident_pairs(const void* kern, cudaLaunchConfig_t cfg, int num_sms) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return num_sms / 2;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find({kern, dev});
  if (it != cache.end()) return it->second;
  cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) n = num_sms / 2;
  cache[{kern, dev}] = n;
  return n;
}

template <bool A_MN, bool B_MN, int NUM_B, int EPI, bool GROUP_K>
cudaError_t launch(const Params& prm, const Maps& maps, long long tiles, int num_sms,
                   cudaStream_t s) {
  if (tiles <= 0) return cudaSuccess;
  if (!pair_for(EPI)) {
    auto kern = gg_kernel<A_MN, B_MN, NUM_B, EPI, GROUP_K>;
    const cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
    kern<<<grid, NUM_THREADS, SMEM_BYTES, s>>>(prm, maps);
    return launched();
  }
  {
    auto kern = gg2_kernel<A_MN, B_MN, NUM_B, EPI, GROUP_K>;
    const cudaError_t ea = set_smem_once(reinterpret_cast<const void*>(kern), SMEM2_BYTES);
    if (ea != cudaSuccess) return ea;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NUM_THREADS2, 1, 1);
    cfg.dynamicSmemBytes = SMEM2_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // A persistent grid must fit on the GPU at once: SMs that cannot pair up
    // inside their GPC host no cluster, so size the grid by what is co-resident
    // (looked up once per kernel and device).
    const int max_clusters = coresident_pairs(reinterpret_cast<const void*>(kern), cfg, num_sms);
    const int clusters = static_cast<int>(tiles < max_clusters ? tiles : max_clusters);
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, prm, maps);
    return e == cudaSuccess ? launched() : e;
  }
}

Params base_params(const GemmProblem& g) {
  Params p;
  memset(&p, 0, sizeof(p));
  p.E = g.E;
  p.offsets = g.offsets;
  p.rows = g.rows;
  p.status = g.status;
  p.kconcat = 1;
  p.raster_n = 0;
  p.group = 16;
  return p;
}

int tile_rows(int epi) { return pair_for(epi) ? PM : BM; }

// Tile order of one launch (see raster).  Per expert, operand A (the tiled-M
// side) holds a_bytes and operand B (the tiled-N side) b_bytes; one m-tile
// reads slab_a bytes of A over the whole K loop, one n-tile slab_b of B.  When
// the smaller operand fits the L2 budget, its tiles form one group, so it is
// read from DRAM once and the larger one streams past it once.  Otherwise both
// stream, in groups of 16 m-tiles.
// MOE_GEMM_RASTER=m<G> or n<G> forces one order and group size on every
// matmul (for tests and measurement).
constexpr long long kL2ResidentBytes = 48ll << 20;
void set_raster(Params& p, long long a_bytes, long long b_bytes, long long slab_a,
                long long slab_b) {
  static const int forced = [] {
    const char* e = getenv("MOE_GEMM_RASTER");
    if (!e || (e[0] != 'm' && e[0] != 'n')) return 0;
    const int g = atoi(e + 1);
    return (g >= 1 && g <= 4096) ? (e[0] == 'n' ? -g : g) : 0;
  }();
  if (forced) {
    p.raster_n = forced < 0;
    p.group = forced < 0 ? -forced : forced;
    return;
  }
  auto group_of = [](long long slab) {
    const long long g = slab > 0 ? kL2ResidentBytes / slab : 1;
    return static_cast<int>(g < 1 ? 1 : (g > 4096 ? 4096 : g));
  };
  if (a_bytes <= kL2ResidentBytes && a_bytes <= b_bytes) {
    p.raster_n = 0;
    p.group = group_of(slab_a);
  } else if (b_bytes <= kL2ResidentBytes) {
    p.raster_n = 1;
    p.group = group_of(slab_b);
  } else {
    p.raster_n = 0;
    p.group = 16;
  }
}

// Average rows per expert (the K extent of a wgrad, the M extent of the rest).
long long rows_per_expert(const GemmProblem& g) { return (g.rows + g.E - 1) / g.E; }

// Upper bound of an M-grouped tile count without reading the offsets.
long long mgrouped_tiles(const GemmProblem& g, int epi, int N, int bnb) {
  const long long nt = (N + bnb - 1) / bnb;
  const long long tm = tile_rows(epi);
  return nt * ((g.rows + tm - 1) / tm + g.E);
}

long long kgrouped_tiles(const GemmProblem& g, int epi, int M, int N, int bnb) {
  const long long tm = tile_rows(epi);
  return static_cast<long long>(g.E) * ((M + tm - 1) / tm) * ((N + bnb - 1) / bnb);
}

// Rows of a K-major B box: the whole 256-column tile (one CTA) or this CTA's
// half of it (pair).
uint32_t kmajor_b_rows(int epi) { return pair_for(epi) ? 128 : BN; }

// 64-column chunks per MN-major B copy: an operand's columns of one tile (one
// CTA), or this CTA's 128 of them (pair).  An MN-major A copy is this CTA's
// 128 rows of the tile in both kernels: BM / 64 chunks.
uint32_t mn_chunks(int epi, int num_b) { return pair_for(epi) ? 2 : BN / num_b / 64; }

}  // namespace

cudaError_t gemm_fc1_fwd(const GemmProblem& g, const void* x_perm, const void* W1,
                         const void* W3, void* A, void* B, void* H, cudaStream_t s) {
  Maps m;
  memset(&m, 0, sizeof(m));
  if (!make_map(&m.a0, x_perm, g.h, g.rows, BK, BM) ||
      !make_map_mn(&m.b0, W1, g.f, static_cast<uint64_t>(g.E) * g.h, BK, mn_chunks(EPI_SWIGLU, 2)) ||
      !make_map_mn(&m.b1, W3, g.f, static_cast<uint64_t>(g.E) * g.h, BK, mn_chunks(EPI_SWIGLU, 2)))
    return cudaErrorInvalidValue;
  m.a1 = m.a0;
  Params p = base_params(g);
  p.N = g.f;
  p.kblocks = g.h / BK;
  p.b_rows = g.h;
  p.out0 = A;
  p.out1 = B;
  p.out2 = H;
  p.ldo = g.f;
  if (!make_map_out_bf16(&m.o0, A, g.f, g.rows) || !make_map_out_bf16(&m.o1, B, g.f, g.rows) ||
      !make_map_out_bf16(&m.o2, H, g.f, g.rows))
    return cudaErrorInvalidValue;
  const long long R = rows_per_expert(g);
  set_raster(p, R * g.h * 2, 2ll * g.h * 2 * g.f, 1ll * tile_rows(EPI_SWIGLU) * g.h * 2, 1ll * BN * g.h * 2);
  return launch<false, true, 2, EPI_SWIGLU, false>(p, m, mgrouped_tiles(g, EPI_SWIGLU, g.f, BN / 2),
                                                    g.num_sms, s);
}

cudaError_t gemm_fc2_fwd(const GemmProblem& g, const void* H, const void* W2, void* O,
                         cudaStream_t s) {
  Maps m;
  memset(&m, 0, sizeof(m));
  if (!make_map(&m.a0, H, g.f, g.rows, BK, BM) ||
      !make_map_mn(&m.b0, W2, g.h, static_cast<uint64_t>(g.E) * g.f, BK, mn_chunks(EPI_BF16, 1)))
    return cudaErrorInvalidValue;
  m.a1 = m.a0;
  m.b1 = m.b0;
  Params p = base_params(g);
  p.N = g.h;
  p.kblocks = g.f / BK;
  p.b_rows = g.f;
  p.out0 = O;
  p.ldo = g.h;
  if (!make_map_out_bf16(&m.o0, O, g.h, g.rows)) return cudaErrorInvalidValue;
  const long long R = rows_per_expert(g);
  set_raster(p, R * g.f * 2, 2ll * g.f * g.h, 1ll * tile_rows(EPI_BF16) * g.f * 2, 1ll * BN * g.f * 2);
  return launch<false, true, 1, EPI_BF16, false>(p, m, mgrouped_tiles(g, EPI_BF16, g.h, BN),
                                                g.num_sms, s);
}

cudaError_t gemm_fc2_dgrad(const GemmProblem& g, const void* dO, const void* W2, const void* A,
                           const void* B, void* dA, void* dB, cudaStream_t s, float* ab_amax) {
  Maps m;
  memset(&m, 0, sizeof(m));
  // B operand: W2[e] viewed as [f rows (N), h (K)] -- K-major
  if (!make_map(&m.a0, dO, g.h, g.rows, BK, BM) ||
      !make_map(&m.b0, W2, g.h, static_cast<uint64_t>(g.E) * g.f, BK, kmajor_b_rows(EPI_SWIGLU_BWD)))
    return cudaErrorInvalidValue;
  m.a1 = m.a0;
  m.b1 = m.b0;
  Params p = base_params(g);
  p.N = g.f;
  p.kblocks = g.h / BK;
  p.b_rows = g.f;
  p.in0 = A;
  p.in1 = B;
  if (!make_map_prefetch(&m.i0, A, g.f, g.rows) || !make_map_prefetch(&m.i1, B, g.f, g.rows) ||
      !make_map_out_bf16(&m.l0, A, g.f, g.rows) || !make_map_out_bf16(&m.l1, B, g.f, g.rows))
    return cudaErrorInvalidValue;
  p.out0 = dA;
  p.out1 = dB;
  p.ldo = g.f;
  if (!make_map_out_bf16(&m.o0, dA, g.f, g.rows) || !make_map_out_bf16(&m.o1, dB, g.f, g.rows))
    return cudaErrorInvalidValue;
  p.part = ab_amax;
  p.part_ld = gemm_col_tiles(g.f);
  const long long R = rows_per_expert(g);
  set_raster(p, R * g.h * 2, 2ll * g.h * g.f, 1ll * tile_rows(EPI_SWIGLU_BWD) * g.h * 2, 1ll * BN * g.h * 2);
  return launch<false, false, 1, EPI_SWIGLU_BWD, false>(p, m, mgrouped_tiles(g, EPI_SWIGLU_BWD, g.f, BN),
                                                         g.num_sms, s);
}

int gemm_col_tiles(int n) { return (n + BN - 1) / BN; }
int gemm_fc1_col_tiles(int f) { return (f + BN / 2 - 1) / (BN / 2); }

// FP8 data gradients (one-CTA kernel, e4m3 K-major operands).
cudaError_t gemm_fc1_dgrad_fp8(const GemmProblem& g, const void* dAq, const void* dBq,
                               const float* sab, const void* W1r, const void* W3r,
                               const float* s13r, float* dX, cudaStream_t s) {
  Maps m;
  memset(&m, 0, sizeof(m));
  // A: dAq then dBq [rows, f] (K concatenated);  B: W1r then W3r [E * h rows (N), f (K)]
  if (!make_map(&m.a0, dAq, g.f, g.rows, 2 * BK, BM, true) ||
      !make_map(&m.a1, dBq, g.f, g.rows, 2 * BK, BM, true) ||
      !make_map(&m.b0, W1r, g.f, static_cast<uint64_t>(g.E) * g.h, 2 * BK, kmajor_b_rows(EPI_F32_F8), true) ||
      !make_map(&m.b1, W3r, g.f, static_cast<uint64_t>(g.E) * g.h, 2 * BK, kmajor_b_rows(EPI_F32_F8), true))
    return cudaErrorInvalidValue;
  Params p = base_params(g);
  p.N = g.h;
  p.kblocks = g.f / (2 * BK);
  p.kconcat = 2;
  p.b_rows = g.h;
  p.row_scale = sab;
  p.col_scale0 = s13r;
  p.out0 = dX;
  p.ldo = g.h;
  if (!make_map_out(&m.o0, dX, g.h, g.rows)) return cudaErrorInvalidValue;
  const long long R = rows_per_expert(g);
  set_raster(p, R * 2 * g.f, 2ll * g.f * g.h, 1ll * BM * 2 * g.f, 1ll * BN * 2 * g.f);
  return launch<false, false, 1, EPI_F32_F8, false>(p, m, mgrouped_tiles(g, EPI_F32_F8, g.h, BN),
                                                    g.num_sms, s);
}

// FP8 forward.  Operands are e4m3 codes, K-major, one byte each: a K block is
// 128 codes (one 128-byte swizzled row), and the MMA is kind::f8f6f4.
cudaError_t gemm_fc1_fwd_fp8(const GemmProblem& g, const void* Xq, const float* sx,
                             const void* W13q, const float* s1, const float* s3, void* A, void* B,
                             void* H, float* h_amax, cudaStream_t s) {
  Maps m;
  memset(&m, 0, sizeof(m));
  // A: Xq [rows, h];  B: W13q viewed as [E * 2f rows (N), h (K)], 256-row tiles
  if (!make_map(&m.a0, Xq, g.h, g.rows, 2 * BK, BM, true) ||
      !make_map(&m.b0, W13q, g.h, static_cast<uint64_t>(g.E) * 2 * g.f, 2 * BK, kmajor_b_rows(EPI_SWIGLU_F8), true))
    return cudaErrorInvalidValue;
  m.a1 = m.a0;
  m.b1 = m.b0;
  Params p = base_params(g);
  p.N = g.f;
  p.kblocks = g.h / (2 * BK);
  p.b_rows = 2 * g.f;
  p.row_scale = sx;
  p.col_scale0 = s1;
  p.col_scale1 = s3;
  p.part = h_amax;
  p.part_ld = g.f / (BN / 2);
  p.out0 = A;
  p.out1 = B;
  p.out2 = H;
  p.ldo = g.f;
  if (!make_map_out_bf16(&m.o0, A, g.f, g.rows) || !make_map_out_bf16(&m.o1, B, g.f, g.rows) ||
      !make_map_out_bf16(&m.o2, H, g.f, g.rows))
    return cudaErrorInvalidValue;
  const long long R = rows_per_expert(g);
  set_raster(p, R * g.h, 2ll * g.h * g.f, 1ll * BM * g.h, 1ll * BN * g.h);
  return launch<false, false, 2, EPI_SWIGLU_F8, false>(
      p, m, mgrouped_tiles(g, EPI_SWIGLU_F8, g.f, BN / 2), g.num_sms, s);
}

cudaError_t gemm_fc2_fwd_fp8(const GemmProblem& g, const void* Hq, const float* sh,
                             const void* W2q, const float* s2, void* O, cudaStream_t s) {
  Maps m;
  memset(&m, 0, sizeof(m));
  // A: Hq [rows, f];  B: W2q viewed as [E * h rows (N), f (K)]
  if (!make_map(&m.a0, Hq, g.f, g.rows, 2 * BK, BM, true) ||
      !make_map(&m.b0, W2q, g.f, static_cast<uint64_t>(g.E) * g.h, 2 * BK, kmajor_b_rows(EPI_BF16_F8), true))
    return cudaErrorInvalidValue;
  m.a1 = m.a0;
  m.b1 = m.b0;
  Params p = base_params(g);
  p.N = g.h;
  p.kblocks = g.f / (2 * BK);
  p.b_rows = g.h;
  p.row_scale = sh;
  p.col_scale0 = s2;
  p.out0 = O;
  p.ldo = g.h;
  if (!make_map_out_bf16(&m.o0, O, g.h, g.rows)) return cudaErrorInvalidValue;
  const long long R = rows_per_expert(g);
  set_raster(p, R * g.f, 1ll * g.f * g.h, 1ll * BM * g.f, 1ll * BN * g.f);
  return launch<false, false, 1, EPI_BF16_F8, false>(p, m, mgrouped_tiles(g, EPI_BF16_F8, g.h, BN),
                                                     g.num_sms, s);
}

cudaError_t gemm_fc2_dgrad_sar(const GemmProblem& g, const void* dy_perm, const void* W2,
                               const void* A, const void* B, const float* gate_rows, void* dA,
                               void* dB, void* gH, float* dg_part, cudaStream_t s) {
  Maps m;
  memset(&m, 0, sizeof(m));
  if (!make_map(&m.a0, dy_perm, g.h, g.rows, BK, BM) ||
      !make_map(&m.b0, W2, g.h, static_cast<uint64_t>(g.E) * g.f, BK,
                kmajor_b_rows(EPI_SWIGLU_BWD_SAR)))
    return cudaErrorInvalidValue;
  m.a1 = m.a0;
  m.b1 = m.b0;
  Params p = base_params(g);
  p.N = g.f;
  p.kblocks = g.h / BK;
  p.b_rows = g.f;
  p.in0 = A;
  p.in1 = B;
  if (!make_map_prefetch(&m.i0, A, g.f, g.rows) || !make_map_prefetch(&m.i1, B, g.f, g.rows))
    return cudaErrorInvalidValue;
  p.in2 = gate_rows;
  p.part = dg_part;
  p.part_ld = gemm_col_tiles(g.f);
  p.out0 = dA;
  p.out1 = dB;
  p.out2 = gH;
  p.ldo = g.f;
  if (!make_map_out_bf16(&m.o0, dA, g.f, g.rows) || !make_map_out_bf16(&m.o1, dB, g.f, g.rows) ||
      !make_map_out_bf16(&m.o2, gH, g.f, g.rows))
    return cudaErrorInvalidValue;
  const long long R = rows_per_expert(g);
  set_raster(p, R * g.h * 2, 2ll * g.h * g.f, 1ll * tile_rows(EPI_SWIGLU_BWD_SAR) * g.h * 2, 1ll * BN * g.h * 2);
  return launch<false, false, 1, EPI_SWIGLU_BWD_SAR, false>(
      p, m, mgrouped_tiles(g, EPI_SWIGLU_BWD_SAR, g.f, BN), g.num_sms, s);
}

cudaError_t gemm_fc1_dgrad(const GemmProblem& g, const void* dA, const void* dB, const void* W1,
                           const void* W3, float* dX, cudaStream_t s) {
  Maps m;
  memset(&m, 0, sizeof(m));
  // B operands: W1[e], W3[e] viewed as [h rows (N), f (K)] -- K-major
  if (!make_map(&m.a0, dA, g.f, g.rows, BK, BM) || !make_map(&m.a1, dB, g.f, g.rows, BK, BM) ||
      !make_map(&m.b0, W1, g.f, static_cast<uint64_t>(g.E) * g.h, BK, kmajor_b_rows(EPI_F32)) ||
      !make_map(&m.b1, W3, g.f, static_cast<uint64_t>(g.E) * g.h, BK, kmajor_b_rows(EPI_F32)))
    return cudaErrorInvalidValue;
  Params p = base_params(g);
  p.N = g.h;
  p.kblocks = g.f / BK;
  p.kconcat = 2;
  p.b_rows = g.h;
  p.out0 = dX;
  p.ldo = g.h;
  if (!make_map_out(&m.o0, dX, g.h, g.rows)) return cudaErrorInvalidValue;
  const long long R = rows_per_expert(g);
  set_raster(p, R * 2 * g.f * 2, 4ll * g.f * g.h, 1ll * tile_rows(EPI_F32) * 2 * g.f * 2, 1ll * BN * 2 * g.f * 2);
  return launch<false, false, 1, EPI_F32, false>(p, m, mgrouped_tiles(g, EPI_F32, g.h, BN),
                                                 g.num_sms, s);
}

cudaError_t gemm_fc2_wgrad(const GemmProblem& g, const void* H, const void* dO, float* dW2,
                           cudaStream_t s) {
  Maps m;
  memset(&m, 0, sizeof(m));
  if (!make_map_mn(&m.a0, H, g.f, g.rows, BK, BM / 64) ||
      !make_map_mn(&m.b0, dO, g.h, g.rows, BK, mn_chunks(EPI_WGRAD, 1)))
    return cudaErrorInvalidValue;
  m.a1 = m.a0;
  m.b1 = m.b0;
  Params p = base_params(g);
  p.M = g.f;
  p.N = g.h;
  p.out0 = dW2;
  if (!make_map_out(&m.o0, dW2, g.h, static_cast<uint64_t>(g.E) * g.f)) return cudaErrorInvalidValue;
  p.ktiles = static_cast<int>(kgrouped_tiles(g, EPI_WGRAD, g.f, g.h, BN));
  const long long R = rows_per_expert(g);
  set_raster(p, R * g.f * 2, R * g.h * 2, tile_rows(EPI_WGRAD) * R * 2, BN * R * 2);
  return launch<true, true, 1, EPI_WGRAD, true>(p, m, p.ktiles, g.num_sms, s);
}

cudaError_t gemm_fc1_wgrad(const GemmProblem& g, const void* x_perm, const void* dA,
                           const void* dB, float* dW1, float* dW3, cudaStream_t s) {
  Maps m;
  memset(&m, 0, sizeof(m));
  if (!make_map_mn(&m.a0, x_perm, g.h, g.rows, BK, BM / 64) ||
      !make_map_mn(&m.b0, dA, g.f, g.rows, BK, mn_chunks(EPI_WGRAD, 2)) ||
      !make_map_mn(&m.b1, dB, g.f, g.rows, BK, mn_chunks(EPI_WGRAD, 2)))
    return cudaErrorInvalidValue;
  m.a1 = m.a0;
  Params p = base_params(g);
  p.M = g.h;
  p.N = g.f;
  p.out0 = dW1;
  p.out1 = dW3;
  if (!make_map_out(&m.o0, dW1, g.f, static_cast<uint64_t>(g.E) * g.h) ||
      !make_map_out(&m.o1, dW3, g.f, static_cast<uint64_t>(g.E) * g.h))
    return cudaErrorInvalidValue;
  p.ktiles = static_cast<int>(kgrouped_tiles(g, EPI_WGRAD, g.h, g.f, BN / 2));
  const long long R = rows_per_expert(g);
  set_raster(p, R * g.h * 2, R * 2 * g.f * 2, tile_rows(EPI_WGRAD) * R * 2, BN * R * 2);
  return launch<true, true, 2, EPI_WGRAD, true>(p, m, p.ktiles, g.num_sms, s);
}

}  // namespace moe
