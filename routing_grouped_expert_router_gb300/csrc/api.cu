// api.cu -- the C ABI of libmoe_gb300 (declared in include/moe.h).
//
// Host-side only: validates arguments before any launch, carves the caller's
// workspace and context buffers, and enqueues the kernels of each operation on
// the caller's stream.  No device memory is allocated here and no call
// synchronises except moe_read_device_status.
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/moe.h"
#include "api_internal.h"
#include "grouped_gemm.cuh"
#include "kernels.cuh"

namespace {

using moe::GemmProblem;

constexpr size_t kAlign = 256;
constexpr size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// ------------------------------------------------------- measurement hook
struct ProfileState {
  cudaEvent_t* events = nullptr;
  int capacity = 0;
  int count = 0;
  const char* names[4096];
};
thread_local ProfileState g_prof;

bool note(cudaStream_t s, const char* name) {
  if (!g_prof.events) return true;
  if (g_prof.count >= g_prof.capacity) return true;
  if (g_prof.count < 4096) g_prof.names[g_prof.count] = name;
  return cudaEventRecord(g_prof.events[g_prof.count++], s) == cudaSuccess;
}

// ----------------------------------------------------------- validation
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool ptr_ok(const void* p) { return p != nullptr && aligned(p, 16); }
// A buffer of `bytes` bytes: may be NULL only when it is empty.
bool buf_ok(const void* p, size_t bytes) {
  return bytes == 0 ? (p == nullptr || aligned(p, 16)) : ptr_ok(p);
}

// `routed`: the call selects k distinct experts per token, so k <= E.  Calls
// that only move or transform already-routed rows also take a subset of the
// experts (E = the local experts of moe_permute_local), where k may exceed E.
moe_status check_dims(const moe_dims* d, bool routed) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->h <= 0 || d->f <= 0 || d->E <= 0 || d->k <= 0) return MOE_ERR_INVALID_ARG;
  if ((routed && d->k > d->E) || d->capacity < 0) return MOE_ERR_INVALID_ARG;
  if (d->sar != 0 && d->sar != 1) return MOE_ERR_INVALID_ARG;
  if (d->k > 8 || d->E > moe::kRouterMaxE) return MOE_ERR_UNSUPPORTED;
  if (d->h % 64 != 0 || d->f % 64 != 0) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->T) * d->k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

bool routed_op(int op) {
  return op == MOE_OP_ROUTE || op == MOE_OP_LAYER_FWD || op == MOE_OP_LAYER_BWD ||
         op == MOE_OP_LAYER_FWD_FP8 || op == MOE_OP_LAYER_BWD_FP8;
}



int num_sms() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// ------------------------------------------------------------- layouts
struct Carve {
  size_t off = 0;
  size_t take(size_t bytes) {
    size_t o = off;
    off += align_up(bytes);
    return o;
  }
};

// ------------------------------------------------------ fp8 weights
// The caller's quantised-weight buffer: codes K-major, then the scales.
struct Fp8WeightLayout {
  size_t W13q, W2q, s1, s3, s2, total;
};
Fp8WeightLayout fp8_weight_layout(const moe_dims& d) {
  const size_t E = d.E, h = d.h, f = d.f;
  Carve c;
  Fp8WeightLayout L;
  L.W13q = c.take(E * 2 * f * h);
  L.W2q = c.take(E * h * f);
  L.s1 = c.take(E * f * 4);
  L.s3 = c.take(E * f * 4);
  L.s2 = c.take(E * h * 4);
  L.total = c.off;
  return L;
}
bool fp8_shape_ok(const moe_dims& d) { return d.h % 128 == 0 && d.f % 128 == 0; }

// The backward's quantised weights: FC1 dgrad's B operand, per output row h
// of W1[e] and W3[e] with one shared scale.
struct Fp8BwdWeightLayout {
  size_t W1r, W3r, s13r, total;
};
Fp8BwdWeightLayout fp8_bwd_weight_layout(const moe_dims& d) {
  const size_t E = d.E, h = d.h, f = d.f;
  Carve c;
  Fp8BwdWeightLayout L;
  L.W1r = c.take(E * h * f);
  L.W3r = c.take(E * h * f);
  L.s13r = c.take(E * h * 4);
  L.total = c.off;
  return L;
}

size_t rows_of(const moe_dims& d) { return static_cast<size_t>(d.T) * d.k; }

struct SavedLayout {
  size_t topk_idx, gates, counts, offsets, perm_src, perm_dst, x_perm, A, B, H, O, total;
};
constexpr size_t kAbsent = ~size_t(0);  // a tensor this mode does not keep

// The forward->backward context.  Default: the routing, the dispatch maps and
// every expert activation (x_perm, A, B, H, O).  Selective activation
// rematerialisation (dims.sar = 1): A and B only of the activations; x_perm is
// gathered again, H rebuilt from A and B, and O is not needed because
// <dy, O> = <H, dy W2^T> comes out of the FC2 dgrad.
SavedLayout saved_layout(const moe_dims& d) {
  const size_t R = rows_of(d);
  Carve c;
  SavedLayout L;
  L.topk_idx = c.take(R * 4);
  L.gates = c.take(R * 4);
  L.counts = c.take(static_cast<size_t>(d.E) * 4);
  L.offsets = c.take(static_cast<size_t>(d.E + 1) * 4);
  L.perm_src = c.take(R * 4);
  L.perm_dst = c.take(R * 4);
  L.x_perm = d.sar ? kAbsent : c.take(R * d.h * 2);
  L.A = c.take(R * d.f * 2);
  L.B = c.take(R * d.f * 2);
  L.H = d.sar ? kAbsent : c.take(R * d.f * 2);
  L.O = d.sar ? kAbsent : c.take(R * d.h * 2);
  L.total = c.off;
  return L;
}

struct WsLayout {
  size_t status = 0;
  size_t blk_counts = 0, bases = 0;          // dispatch
  size_t x_perm = 0, dO = 0, dA = 0, dB = 0;  // expert backward
  size_t dX = 0, dg = 0;                     // layer backward
  size_t dl = 0, WgT = 0, partial = 0;       // router backward
  size_t logits = 0;                         // router partial logits
  size_t H = 0, O = 0;                       // sar forward: activations not kept
  size_t gH = 0, gate_rows = 0, dg_part = 0;  // sar backward
  size_t Xq = 0, sx = 0, Hq = 0, sh = 0;     // fp8 forward
  size_t h_amax = 0;                         // fp8 forward: per-tile amax of H
  size_t dAq = 0, dBq = 0, sab = 0, ab_amax = 0;  // fp8 backward
  size_t total = 0;
};
WsLayout ws_layout(const moe_dims& d, int op) {
  const size_t R = rows_of(d);
  const size_t nblk = static_cast<size_t>(moe::dispatch_blocks(static_cast<long long>(R)));
  Carve c;
  WsLayout L;
  L.status = c.take(kAlign);
  auto route = [&] { L.logits = c.take(moe::router_partial_bytes(d.T, d.h, d.E)); };
  auto dispatch = [&] {
    L.blk_counts = c.take(nblk * d.E * 4);
    L.bases = c.take(nblk * d.E * 4);
  };
  auto router_bwd = [&] {
    L.dl = c.take(static_cast<size_t>(d.T) * d.E * 4);
    L.WgT = c.take(static_cast<size_t>(d.E) * d.h * 4);
    L.partial = c.take(static_cast<size_t>(moe::wgrad_router_chunks(d.T, d.h, d.E)) * d.h * d.E * 4);
  };
  auto expert_bwd = [&](bool with_x) {
    if (with_x) L.x_perm = c.take(R * d.h * 2);
    L.dO = c.take(R * d.h * 2);
    L.dA = c.take(R * d.f * 2);
    L.dB = c.take(R * d.f * 2);
  };
  switch (op) {
    case MOE_OP_ROUTE: route(); break;
    case MOE_OP_PERMUTE: dispatch(); break;
    case MOE_OP_EXPERT_FFN_FWD: L.x_perm = c.take(R * d.h * 2); break;
    case MOE_OP_EXPERT_FFN_BWD: expert_bwd(true); break;
    case MOE_OP_ROUTER_BWD: router_bwd(); break;
    case MOE_OP_LAYER_FWD:
    case MOE_OP_LAYER_FWD_FP8:
      route();
      dispatch();
      if (op == MOE_OP_LAYER_FWD_FP8) {
        L.Xq = c.take(R * d.h);
        L.sx = c.take(R * 4);
        L.Hq = c.take(R * d.f);
        L.sh = c.take(R * 4);
        L.h_amax = c.take(R * static_cast<size_t>(moe::gemm_fc1_col_tiles(d.f)) * 4);
      }
      if (d.sar) {
        L.x_perm = c.take(R * d.h * 2);
        L.H = c.take(R * d.f * 2);
        L.O = c.take(R * d.h * 2);
      }
      break;
    case MOE_OP_LAYER_BWD:
    case MOE_OP_LAYER_BWD_FP8:
      if (op == MOE_OP_LAYER_BWD_FP8) {
        L.dAq = c.take(R * d.f);
        L.dBq = c.take(R * d.f);
        L.sab = c.take(R * 4);
        L.ab_amax = c.take(R * static_cast<size_t>(moe::gemm_col_tiles(d.f)) * 4);
      }
      expert_bwd(d.sar != 0);
      L.dX = c.take(R * d.h * 4);
      L.dg = c.take(R * 4);
      router_bwd();
      if (d.sar) {
        L.gH = c.take(R * d.f * 2);
        L.gate_rows = c.take(R * 4);
        L.dg_part = c.take(R * static_cast<size_t>(moe::gemm_col_tiles(d.f)) * 4);
      }
      break;
    default: return WsLayout{};
  }
  L.total = c.off;
  return L;
}

template <class T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(base) + off);
}
template <class T>
const T* at(const void* base, size_t off) {
  return reinterpret_cast<const T*>(static_cast<const uint8_t*>(base) + off);
}

moe_status ws_check(const moe_dims& d, int op, const void* ws, size_t ws_bytes) {
  if (!ws || !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_layout(d, op).total) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

#define MOE_CU(expr)                                   \
  do {                                                 \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA;    \
  } while (0)
#define MOE_RUN(expr, name)                            \
  do {                                                 \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA;    \
    if (!note(stream, name)) return MOE_ERR_CUDA;      \
  } while (0)

GemmProblem problem(const moe_dims& d, const int32_t* offsets, void* ws) {
  GemmProblem p;
  p.E = d.E;
  p.offsets = offsets;
  p.rows = static_cast<int>(rows_of(d));
  p.h = d.h;
  p.f = d.f;
  p.status = at<int>(ws, 0);
  p.num_sms = num_sms();
  return p;
}

}  // namespace

namespace moe_api {
moe_status check_dims(const moe_dims* d, bool routed) { return ::check_dims(d, routed); }
int num_sms() { return ::num_sms(); }
bool note(cudaStream_t s, const char* name) { return ::note(s, name); }
}  // namespace moe_api

namespace {

// --------------------------------------------------------- the steps
moe_status do_route(const moe_dims& d, const uint16_t* x, const float* Wg, const float* b,
                    int32_t* idx, float* gates, void* ws, const WsLayout& L, cudaStream_t stream) {
  MOE_RUN(moe::launch_router(x, Wg, d.has_bias ? b : nullptr, d.T, d.h, d.E, d.k, idx, gates,
                             at<float>(ws, L.logits), num_sms(), stream),
          "router_topk");
  return MOE_OK;
}

// Experts [e_lo, e_hi) of the layer, each taking at most d.capacity
// assignments (all of them when capacity is 0).
moe::DispatchSel selection(const moe_dims& d, int e_lo, int e_hi) {
  return moe::DispatchSel{e_lo, e_hi - e_lo, d.capacity > 0 ? d.capacity : INT_MAX};
}

moe_status do_dispatch(const moe_dims& d, const moe::DispatchSel& sel, const int32_t* idx,
                       int32_t* counts, int32_t* offsets, int32_t* psrc, int32_t* pdst, void* ws,
                       const WsLayout& L, cudaStream_t stream) {
  const long long R = static_cast<long long>(rows_of(d));
  const int nblk = moe::dispatch_blocks(R);
  int32_t* blk = at<int32_t>(ws, L.blk_counts);
  int32_t* bases = at<int32_t>(ws, L.bases);
  int* status = at<int>(ws, 0);
  MOE_RUN(moe::launch_dispatch_hist(idx, R, d.E, sel, blk, stream, status), "dispatch_hist");
  MOE_RUN(moe::launch_dispatch_scan(blk, nblk, sel, counts, offsets, bases, stream),
          "dispatch_scan");
  MOE_RUN(moe::launch_dispatch_scatter(idx, R, d.E, sel, bases, offsets, psrc, pdst, stream,
                                       status),
          "dispatch_scatter");
  return MOE_OK;
}

moe_status do_ffn_fwd(const moe_dims& d, const uint16_t* x_perm, const int32_t* offsets,
                      const uint16_t* W1, const uint16_t* W3, const uint16_t* W2, uint16_t* A,
                      uint16_t* B, uint16_t* H, uint16_t* O, void* ws, cudaStream_t stream) {
  if (rows_of(d) == 0) return MOE_OK;
  const GemmProblem g = problem(d, offsets, ws);
  MOE_RUN(moe::gemm_fc1_fwd(g, x_perm, W1, W3, A, B, H, stream), moe::kGemmNames[0]);
  MOE_RUN(moe::gemm_fc2_fwd(g, H, W2, O, stream), moe::kGemmNames[1]);
  return MOE_OK;
}

moe_status do_ffn_bwd(const moe_dims& d, const uint16_t* x_perm, const uint16_t* dO,
                      const int32_t* offsets, const uint16_t* W1, const uint16_t* W3,
                      const uint16_t* W2, const uint16_t* A, const uint16_t* B, const uint16_t* H,
                      uint16_t* dA, uint16_t* dB, float* dX, float* dW1, float* dW3, float* dW2,
                      void* ws, cudaStream_t stream) {
  if (rows_of(d) == 0) {
    const size_t wbytes = static_cast<size_t>(d.E) * d.h * d.f * 4;
    MOE_RUN(cudaMemsetAsync(dW1, 0, wbytes, stream), "zero_dW1");
    MOE_RUN(cudaMemsetAsync(dW3, 0, wbytes, stream), "zero_dW3");
    MOE_RUN(cudaMemsetAsync(dW2, 0, wbytes, stream), "zero_dW2");
    return MOE_OK;
  }
  const GemmProblem g = problem(d, offsets, ws);
  MOE_RUN(moe::gemm_fc2_dgrad(g, dO, W2, A, B, dA, dB, stream), moe::kGemmNames[2]);
  MOE_RUN(moe::gemm_fc2_wgrad(g, H, dO, dW2, stream), moe::kGemmNames[4]);
  MOE_RUN(moe::gemm_fc1_dgrad(g, dA, dB, W1, W3, dX, stream), moe::kGemmNames[3]);
  MOE_RUN(moe::gemm_fc1_wgrad(g, x_perm, dA, dB, dW1, dW3, stream), moe::kGemmNames[5]);
  return MOE_OK;
}

// Expert backward from a sar context (A, B kept): gathers x_perm and the
// ungated dy rows again, rebuilds H inside the FC2 dgrad, and reduces the gate
// gradients from the dgrad's per-tile partial sums.
moe_status do_ffn_bwd_sar(const moe_dims& d, const uint16_t* x, const uint16_t* dy,
                          const float* gates, const int32_t* psrc, const int32_t* offsets,
                          const uint16_t* W1, const uint16_t* W3, const uint16_t* W2,
                          const uint16_t* A, const uint16_t* B, float* dX, float* dg, float* dW1,
                          float* dW3, float* dW2, void* ws, const WsLayout& L,
                          cudaStream_t stream) {
  const long long R = static_cast<long long>(rows_of(d));
  uint16_t* xp = at<uint16_t>(ws, L.x_perm);
  uint16_t* dyp = at<uint16_t>(ws, L.dO);
  uint16_t* dA = at<uint16_t>(ws, L.dA);
  uint16_t* dB = at<uint16_t>(ws, L.dB);
  uint16_t* gH = at<uint16_t>(ws, L.gH);
  float* grow = at<float>(ws, L.gate_rows);
  float* part = at<float>(ws, L.dg_part);
  const int32_t* nvalid = offsets + d.E;
  int* status = at<int>(ws, 0);
  MOE_RUN(moe::launch_gather_rows(x, psrc, d.k, R, d.T, d.h, xp, num_sms(), stream, nvalid,
                                  nullptr, nullptr, status),
          "permute_rows");
  MOE_RUN(moe::launch_gather_rows(dy, psrc, d.k, R, d.T, d.h, dyp, num_sms(), stream, nvalid,
                                  gates, grow, status),
          "permute_dy");
  if (R == 0) {
    const size_t wbytes = static_cast<size_t>(d.E) * d.h * d.f * 4;
    MOE_RUN(cudaMemsetAsync(dW1, 0, wbytes, stream), "zero_dW1");
    MOE_RUN(cudaMemsetAsync(dW3, 0, wbytes, stream), "zero_dW3");
    MOE_RUN(cudaMemsetAsync(dW2, 0, wbytes, stream), "zero_dW2");
    return MOE_OK;
  }
  const GemmProblem g = problem(d, offsets, ws);
  MOE_RUN(moe::gemm_fc2_dgrad_sar(g, dyp, W2, A, B, grow, dA, dB, gH, part, stream),
          moe::kGemmSarDgradName);
  MOE_RUN(moe::gemm_fc2_wgrad(g, gH, dyp, dW2, stream), moe::kGemmNames[4]);
  MOE_RUN(moe::gemm_fc1_dgrad(g, dA, dB, W1, W3, dX, stream), moe::kGemmNames[3]);
  MOE_RUN(moe::gemm_fc1_wgrad(g, xp, dA, dB, dW1, dW3, stream), moe::kGemmNames[5]);
  MOE_RUN(moe::launch_dg_reduce(part, moe::gemm_col_tiles(d.f), psrc, R, nvalid, dg, num_sms(),
                                stream, status),
          "dg_reduce");
  return MOE_OK;
}

moe_status do_router_bwd(const moe_dims& d, const uint16_t* x, const float* Wg,
                         const int32_t* idx, const float* gates, const float* dg,
                         const float* dX, const int32_t* pdst, uint16_t* dx, float* dWg, void* ws,
                         const WsLayout& L, cudaStream_t stream) {
  float* WgT = at<float>(ws, L.WgT);
  float* dl = at<float>(ws, L.dl);
  float* partial = at<float>(ws, L.partial);
  MOE_RUN(moe::launch_transpose_wg(Wg, d.h, d.E, WgT, stream), "transpose_wg");
  MOE_RUN(moe::launch_token_grad(dX, pdst, idx, gates, dg, WgT, d.T, d.k, d.h, d.E, dl, dx,
                                 num_sms(), stream, at<int>(ws, 0)),
          "token_grad");
  MOE_RUN(moe::launch_router_wgrad(x, dl, d.T, d.h, d.E, partial, dWg, stream), "router_wgrad");
  return MOE_OK;
}

}  // namespace

// =================================================================== C ABI
extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: null, misaligned or inconsistent argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape outside the supported set";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace smaller than required";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a kernel's bounded wait ran out";
    case MOE_ERR_DEVICE_INDEX:
      return "MOE_ERR_DEVICE_INDEX: an expert id, permutation entry or offset read on the device "
             "was out of range (the element was skipped)";
  }
  return "unknown moe_status";
}

int32_t moe_capacity_for(int32_t T, int32_t k, int32_t E, double factor) {
  if (T < 0 || k < 1 || E < 1 || !(factor > 0.0)) return -1;
  const double c = std::ceil(factor * static_cast<double>(T) * k / E);
  if (!(c < 2147483647.0)) return -1;
  return static_cast<int32_t>(c);
}

const char* moe_version(void) { return "libmoe_gb300 0.1 (sm_103a, tcgen05 GroupedGEMM)"; }

size_t moe_workspace_bytes(const moe_dims* dims, int op) {
  if (check_dims(dims, routed_op(op)) != MOE_OK) return 0;
  return ws_layout(*dims, op).total;
}

size_t moe_saved_bytes(const moe_dims* dims) {
  if (check_dims(dims, true) != MOE_OK) return 0;
  return saved_layout(*dims).total;
}

void* moe_saved_view(const moe_dims* dims, void* saved, const char* name) {
  if (check_dims(dims, true) != MOE_OK || !saved || !name) return nullptr;
  const SavedLayout L = saved_layout(*dims);
  struct {
    const char* n;
    size_t off;
  } tab[] = {{"topk_idx", L.topk_idx}, {"gates", L.gates},       {"counts", L.counts},
             {"offsets", L.offsets},   {"perm_src", L.perm_src}, {"perm_dst", L.perm_dst},
             {"x_perm", L.x_perm},     {"A", L.A},               {"B", L.B},
             {"H", L.H},               {"O", L.O}};
  for (auto& e : tab)
    if (strcmp(e.n, name) == 0) return e.off == kAbsent ? nullptr : at<uint8_t>(saved, e.off);
  return nullptr;
}

int moe_profile_events(moe_event_t* events, int capacity) {
  const int n = g_prof.count;
  g_prof.events = reinterpret_cast<cudaEvent_t*>(events);
  g_prof.capacity = events ? capacity : 0;
  g_prof.count = 0;
  return n;
}

int64_t moe_kernel_launches(void) { return moe::kernel_launches(); }

void moe_test_fail_launch_after(int n) { moe::fail_launch_after(n); }

const char* moe_profile_kernel_name(int i) {
  if (i < 0 || i >= 4096) return "";
  return g_prof.names[i] ? g_prof.names[i] : "";
}

moe_status moe_read_device_status(void* ws, moe_stream_t stream) {
  if (ws && !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  int* word = ws ? static_cast<int*>(ws) : moe::nows_status_word();
  if (!word) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  MOE_CU(cudaStreamSynchronize(s));
  MOE_CU(cudaMemcpy(&v, word, sizeof(int), cudaMemcpyDeviceToHost));
  MOE_CU(cudaMemset(word, 0, sizeof(int)));
  return static_cast<moe_status>(v);
}

moe_status moe_selftest_wait_timeout(void* ws, uint32_t limit_us, moe_stream_t stream_) {
  if (!ws || !aligned(ws, kAlign) || limit_us == 0 || limit_us > 1000000u) return MOE_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  MOE_RUN(moe::launch_wait_timeout_probe(at<int>(ws, 0), 1000ull * limit_us, stream),
          "wait_timeout_probe");
  return MOE_OK;
}

moe_status moe_clear_device_status(void* ws, moe_stream_t stream) {
  if (ws && !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  int* word = ws ? static_cast<int*>(ws) : moe::nows_status_word();
  if (!word) return MOE_ERR_CUDA;
  MOE_CU(cudaMemsetAsync(word, 0, sizeof(int), reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

moe_status moe_route(const moe_dims* dims, const moe_bf16* x, const float* Wg, const float* b,
                     int32_t* topk_idx, float* gates, void* ws, size_t ws_bytes,
                     moe_stream_t stream_) {
  moe_status st = check_dims(dims, true);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  const size_t T = d.T, R = rows_of(d);
  if (!buf_ok(x, T * d.h) || !ptr_ok(Wg) || !buf_ok(topk_idx, R) || !buf_ok(gates, R) ||
      (d.has_bias && !ptr_ok(b)))
    return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(d, MOE_OP_ROUTE, ws, ws_bytes)) != MOE_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  return do_route(d, x, Wg, b, topk_idx, gates, ws, ws_layout(d, MOE_OP_ROUTE), stream);
}

moe_status moe_permute(const moe_dims* dims, const int32_t* topk_idx, const moe_bf16* x,
                       int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* perm_dst,
                       moe_bf16* x_perm, void* ws, size_t ws_bytes, moe_stream_t stream_) {
  moe_status st = check_dims(dims, false);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  const size_t R = rows_of(d);
  if (!buf_ok(topk_idx, R) || !ptr_ok(counts) || !ptr_ok(offsets) || !buf_ok(perm_src, R) ||
      !buf_ok(perm_dst, R))
    return MOE_ERR_INVALID_ARG;
  if ((x && !aligned(x, 16)) || (x_perm && !aligned(x_perm, 16))) return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(d, MOE_OP_PERMUTE, ws, ws_bytes)) != MOE_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const WsLayout L = ws_layout(d, MOE_OP_PERMUTE);
  if ((st = do_dispatch(d, selection(d, 0, d.E), topk_idx, counts, offsets, perm_src, perm_dst,
                        ws, L, stream)) != MOE_OK)
    return st;
  if (x && x_perm)
    MOE_RUN(moe::launch_gather_rows(x, perm_src, d.k, static_cast<long long>(rows_of(d)), d.T,
                                    d.h, x_perm, num_sms(), stream, offsets + d.E, nullptr,
                                    nullptr, at<int>(ws, 0)),
            "permute_rows");
  return MOE_OK;
}

moe_status moe_permute_local(const moe_dims* dims, const int32_t* topk_idx, int32_t e_lo,
                             int32_t e_hi, const moe_bf16* x, int32_t* counts, int32_t* offsets,
                             int32_t* perm_src, int32_t* perm_dst, moe_bf16* x_perm, void* ws,
                             size_t ws_bytes, moe_stream_t stream_) {
  moe_status st = check_dims(dims, false);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (e_lo < 0 || e_hi <= e_lo || e_hi > d.E) return MOE_ERR_INVALID_ARG;
  const size_t R = rows_of(d);
  if (!buf_ok(topk_idx, R) || !ptr_ok(counts) || !ptr_ok(offsets) || !buf_ok(perm_src, R) ||
      !buf_ok(perm_dst, R))
    return MOE_ERR_INVALID_ARG;
  if ((x && !aligned(x, 16)) || (x_perm && !aligned(x_perm, 16))) return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(d, MOE_OP_PERMUTE, ws, ws_bytes)) != MOE_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const WsLayout L = ws_layout(d, MOE_OP_PERMUTE);
  if ((st = do_dispatch(d, selection(d, e_lo, e_hi), topk_idx, counts, offsets, perm_src,
                        perm_dst, ws, L, stream)) != MOE_OK)
    return st;
  if (x && x_perm)
    MOE_RUN(moe::launch_gather_rows(x, perm_src, d.k, static_cast<long long>(R), d.T, d.h, x_perm,
                                    num_sms(), stream, offsets + (e_hi - e_lo), nullptr, nullptr,
                                    at<int>(ws, 0)),
            "permute_rows");
  return MOE_OK;
}

moe_status moe_unpermute(const moe_dims* dims, const int32_t* perm_dst, const moe_bf16* rows_perm,
                         moe_bf16* rows_assign, moe_stream_t stream_) {
  moe_status st = check_dims(dims, false);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  const size_t R = rows_of(d);
  if (!buf_ok(perm_dst, R) || !buf_ok(rows_perm, R) || !buf_ok(rows_assign, R))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int* status = moe::nows_status_word();
  if (!status) return MOE_ERR_CUDA;
  MOE_RUN(moe::launch_gather_rows(rows_perm, perm_dst, 1, static_cast<long long>(rows_of(d)),
                                  static_cast<long long>(rows_of(d)), d.h, rows_assign, num_sms(),
                                  stream, nullptr, nullptr, nullptr, status),
          "unpermute_rows");
  return MOE_OK;
}

moe_status moe_expert_ffn_fwd(const moe_dims* dims, const moe_bf16* x, const int32_t* perm_src,
                              const int32_t* offsets, const moe_bf16* W1, const moe_bf16* W3,
                              const moe_bf16* W2, moe_bf16* A, moe_bf16* B, moe_bf16* H,
                              moe_bf16* O, void* ws, size_t ws_bytes, moe_stream_t stream_) {
  moe_status st = check_dims(dims, false);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  const size_t T = d.T, R = rows_of(d);
  if (!buf_ok(x, T) || !buf_ok(perm_src, R) || !ptr_ok(offsets) || !ptr_ok(W1) || !ptr_ok(W3) ||
      !ptr_ok(W2) || !buf_ok(A, R) || !buf_ok(B, R) || !buf_ok(H, R) || !buf_ok(O, R))
    return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(d, MOE_OP_EXPERT_FFN_FWD, ws, ws_bytes)) != MOE_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const WsLayout L = ws_layout(d, MOE_OP_EXPERT_FFN_FWD);
  uint16_t* xp = at<uint16_t>(ws, L.x_perm);
  int* status = at<int>(ws, 0);
  MOE_RUN(moe::launch_check_offsets(offsets, d.E, static_cast<long long>(R), status, stream),
          "check_offsets");
  MOE_RUN(moe::launch_gather_rows(x, perm_src, d.k, static_cast<long long>(rows_of(d)), d.T, d.h,
                                  xp, num_sms(), stream, offsets + d.E, nullptr, nullptr, status),
          "permute_rows");
  return do_ffn_fwd(d, xp, offsets, W1, W3, W2, A, B, H, O, ws, stream);
}

moe_status moe_combine(const moe_dims* dims, const moe_bf16* O, const float* gates,
                       const int32_t* perm_dst, moe_bf16* y, moe_stream_t stream_) {
  moe_status st = check_dims(dims, false);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  const size_t T = d.T, R = rows_of(d);
  if (!buf_ok(O, R) || !buf_ok(gates, R) || !buf_ok(perm_dst, R) || !buf_ok(y, T))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int* status = moe::nows_status_word();
  if (!status) return MOE_ERR_CUDA;
  MOE_RUN(moe::launch_combine(O, gates, perm_dst, d.T, d.k, d.h, y, num_sms(), stream, status),
          "combine");
  return MOE_OK;
}

moe_status moe_expert_ffn_bwd(const moe_dims* dims, const moe_bf16* x, const moe_bf16* dy,
                              const float* gates, const int32_t* perm_src, const int32_t* offsets,
                              const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2,
                              const moe_bf16* A, const moe_bf16* B, const moe_bf16* H,
                              const moe_bf16* O, float* dX_perm, float* dg, float* dW1,
                              float* dW3, float* dW2, void* ws, size_t ws_bytes,
                              moe_stream_t stream_) {
  moe_status st = check_dims(dims, false);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  const size_t T = d.T, R = rows_of(d);
  if (!buf_ok(x, T) || !buf_ok(dy, T) || !buf_ok(gates, R) || !buf_ok(perm_src, R) ||
      !ptr_ok(offsets) || !ptr_ok(W1) || !ptr_ok(W3) || !ptr_ok(W2) || !buf_ok(A, R) ||
      !buf_ok(B, R) || !buf_ok(H, R) || !buf_ok(O, R) || !buf_ok(dX_perm, R) || !buf_ok(dg, R) ||
      !ptr_ok(dW1) || !ptr_ok(dW3) || !ptr_ok(dW2))
    return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(d, MOE_OP_EXPERT_FFN_BWD, ws, ws_bytes)) != MOE_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const WsLayout L = ws_layout(d, MOE_OP_EXPERT_FFN_BWD);
  uint16_t* xp = at<uint16_t>(ws, L.x_perm);
  uint16_t* dO = at<uint16_t>(ws, L.dO);
  const long long nrows = static_cast<long long>(R);
  int* status = at<int>(ws, 0);
  MOE_RUN(moe::launch_check_offsets(offsets, d.E, nrows, status, stream), "check_offsets");
  MOE_RUN(moe::launch_gather_rows(x, perm_src, d.k, nrows, d.T, d.h, xp, num_sms(), stream,
                                  offsets + d.E, nullptr, nullptr, status),
          "permute_rows");
  MOE_RUN(moe::launch_bwd_prep(dy, O, gates, perm_src, nrows, d.k, d.h, dO, dg, num_sms(), stream,
                               offsets + d.E, status),
          "bwd_prep");
  return do_ffn_bwd(d, xp, dO, offsets, W1, W3, W2, A, B, H, at<uint16_t>(ws, L.dA),
                    at<uint16_t>(ws, L.dB), dX_perm, dW1, dW3, dW2, ws, stream);
}

moe_status moe_router_bwd(const moe_dims* dims, const moe_bf16* x, const float* Wg,
                          const int32_t* topk_idx, const float* gates, const float* dg,
                          const float* dX_perm, const int32_t* perm_src, const int32_t* perm_dst,
                          const int32_t* offsets, moe_bf16* dx, float* dWg, void* ws,
                          size_t ws_bytes, moe_stream_t stream_) {
  moe_status st = check_dims(dims, false);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  const size_t T = d.T, R = rows_of(d);
  if (!buf_ok(x, T) || !ptr_ok(Wg) || !buf_ok(topk_idx, R) || !buf_ok(gates, R) ||
      !buf_ok(dg, R) || !buf_ok(dX_perm, R) || !buf_ok(perm_src, R) || !buf_ok(perm_dst, R) ||
      !ptr_ok(offsets) || !buf_ok(dx, T) || !ptr_ok(dWg))
    return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(d, MOE_OP_ROUTER_BWD, ws, ws_bytes)) != MOE_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const WsLayout L = ws_layout(d, MOE_OP_ROUTER_BWD);
  return do_router_bwd(d, x, Wg, topk_idx, gates, dg, dX_perm, perm_dst, dx, dWg, ws, L, stream);
}

moe_status moe_layer_fwd(const moe_dims* dims, const moe_bf16* x, const float* Wg, const float* b,
                         const moe_bf16* W1, const moe_bf16* W3, const moe_bf16* W2, moe_bf16* y,
                         void* saved, void* ws, size_t ws_bytes, moe_stream_t stream_) {
  moe_status st = check_dims(dims, true);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  const size_t T = d.T;
  if (!buf_ok(x, T) || !ptr_ok(Wg) || !ptr_ok(W1) || !ptr_ok(W3) || !ptr_ok(W2) || !buf_ok(y, T) ||
      (d.has_bias && !ptr_ok(b)) || !saved || !aligned(saved, kAlign))
    return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(d, MOE_OP_LAYER_FWD, ws, ws_bytes)) != MOE_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const WsLayout L = ws_layout(d, MOE_OP_LAYER_FWD);
  const SavedLayout S = saved_layout(d);
  int32_t* idx = at<int32_t>(saved, S.topk_idx);
  float* gates = at<float>(saved, S.gates);
  int32_t* offsets = at<int32_t>(saved, S.offsets);
  int32_t* psrc = at<int32_t>(saved, S.perm_src);
  int32_t* pdst = at<int32_t>(saved, S.perm_dst);
  // activations that sar does not keep live in the workspace
  uint16_t* xp = d.sar ? at<uint16_t>(ws, L.x_perm) : at<uint16_t>(saved, S.x_perm);
  uint16_t* H = d.sar ? at<uint16_t>(ws, L.H) : at<uint16_t>(saved, S.H);
  uint16_t* O = d.sar ? at<uint16_t>(ws, L.O) : at<uint16_t>(saved, S.O);
  if ((st = do_route(d, x, Wg, b, idx, gates, ws, L, stream)) != MOE_OK) return st;
  if ((st = do_dispatch(d, selection(d, 0, d.E), idx, at<int32_t>(saved, S.counts), offsets, psrc,
                        pdst, ws, L, stream)) != MOE_OK)
    return st;
  MOE_RUN(moe::launch_gather_rows(x, psrc, d.k, static_cast<long long>(rows_of(d)), d.T, d.h, xp,
                                  num_sms(), stream, offsets + d.E, nullptr, nullptr,
                                  at<int>(ws, 0)),
          "permute_rows");
  if ((st = do_ffn_fwd(d, xp, offsets, W1, W3, W2, at<uint16_t>(saved, S.A),
                       at<uint16_t>(saved, S.B), H, O, ws, stream)) != MOE_OK)
    return st;
  MOE_RUN(moe::launch_combine(O, gates, pdst, d.T, d.k, d.h, y, num_sms(), stream,
                              at<int>(ws, 0)),
          "combine");
  return MOE_OK;
}

size_t moe_fp8_weight_bytes(const moe_dims* dims) {
  if (check_dims(dims, false) != MOE_OK || !fp8_shape_ok(*dims)) return 0;
  return fp8_weight_layout(*dims).total;
}

void* moe_fp8_weight_view(const moe_dims* dims, void* qw, const char* name) {
  if (check_dims(dims, false) != MOE_OK || !fp8_shape_ok(*dims) || !qw || !name) return nullptr;
  const Fp8WeightLayout L = fp8_weight_layout(*dims);
  struct {
    const char* n;
    size_t off;
  } tab[] = {{"W13q", L.W13q}, {"W2q", L.W2q}, {"s1", L.s1}, {"s3", L.s3}, {"s2", L.s2}};
  for (auto& e : tab)
    if (strcmp(e.n, name) == 0) return at<uint8_t>(qw, e.off);
  return nullptr;
}

moe_status moe_quantize_weights_fp8(const moe_dims* dims, const moe_bf16* W1, const moe_bf16* W3,
                                    const moe_bf16* W2, void* qw, moe_stream_t stream_) {
  moe_status st = check_dims(dims, false);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!fp8_shape_ok(d)) return MOE_ERR_UNSUPPORTED;
  if (!ptr_ok(W1) || !ptr_ok(W3) || !ptr_ok(W2) || !qw || !aligned(qw, kAlign))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const Fp8WeightLayout L = fp8_weight_layout(d);
  uint8_t* W13q = at<uint8_t>(qw, L.W13q);
  // W1, W3 [E, h, f] -> interleaved 128-row groups of W13q [E, 2f, h]
  MOE_RUN(moe::launch_quant_cols(W1, d.E, d.h, d.f, 2 * d.f, 256, 0, W13q, at<float>(qw, L.s1),
                                 num_sms(), stream),
          "quant_w1");
  MOE_RUN(moe::launch_quant_cols(W3, d.E, d.h, d.f, 2 * d.f, 256, 1, W13q, at<float>(qw, L.s3),
                                 num_sms(), stream),
          "quant_w3");
  // W2 [E, f, h] -> W2q [E, h, f]
  MOE_RUN(moe::launch_quant_cols(W2, d.E, d.f, d.h, d.h, 128, 0, at<uint8_t>(qw, L.W2q),
                                 at<float>(qw, L.s2), num_sms(), stream),
          "quant_w2");
  return MOE_OK;
}

moe_status moe_quantize_rows_fp8(const moe_bf16* in, int64_t rows, int32_t n, const int32_t* idx,
                                 int32_t div, int64_t src_rows, uint8_t* q, float* scale,
                                 moe_stream_t stream_) {
  if (rows < 0 || src_rows < 0 || n <= 0 || n % 16 != 0 || (idx && div <= 0))
    return MOE_ERR_INVALID_ARG;
  if (rows > 0 && (!ptr_ok(in) || !ptr_ok(q) || !ptr_ok(scale) || (idx && !ptr_ok(idx))))
    return MOE_ERR_INVALID_ARG;
  if (rows > 0 && !idx && src_rows < rows) return MOE_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int* status = moe::nows_status_word();
  if (!status) return MOE_ERR_CUDA;
  MOE_RUN(moe::launch_quant_rows(in, idx, idx ? div : 1, rows, src_rows, n, q, scale, num_sms(),
                                 stream, nullptr, nullptr, 0, nullptr, nullptr, nullptr, status),
          "quant_rows");
  return MOE_OK;
}

moe_status moe_layer_fwd_fp8(const moe_dims* dims, const moe_bf16* x, const float* Wg,
                             const float* b, const void* qw, moe_bf16* y, void* saved, void* ws,
                             size_t ws_bytes, moe_stream_t stream_) {
  moe_status st = check_dims(dims, true);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!fp8_shape_ok(d)) return MOE_ERR_UNSUPPORTED;
  // The sar backward takes <dy, O> as <H, dy W2^T>, which needs O = H W2
  // exactly; here O comes from the e4m3 codes of H and W2.
  if (d.sar) return MOE_ERR_UNSUPPORTED;
  const size_t T = d.T;
  if (!buf_ok(x, T) || !ptr_ok(Wg) || !qw || !aligned(qw, kAlign) || !buf_ok(y, T) ||
      (d.has_bias && !ptr_ok(b)) || !saved || !aligned(saved, kAlign))
    return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(d, MOE_OP_LAYER_FWD_FP8, ws, ws_bytes)) != MOE_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const WsLayout L = ws_layout(d, MOE_OP_LAYER_FWD_FP8);
  const SavedLayout S = saved_layout(d);
  const Fp8WeightLayout Q = fp8_weight_layout(d);
  int32_t* idx = at<int32_t>(saved, S.topk_idx);
  float* gates = at<float>(saved, S.gates);
  int32_t* offsets = at<int32_t>(saved, S.offsets);
  int32_t* psrc = at<int32_t>(saved, S.perm_src);
  int32_t* pdst = at<int32_t>(saved, S.perm_dst);
  uint16_t* H = at<uint16_t>(saved, S.H);
  uint16_t* O = at<uint16_t>(saved, S.O);
  uint8_t* Xq = at<uint8_t>(ws, L.Xq);
  uint8_t* Hq = at<uint8_t>(ws, L.Hq);
  float* sx = at<float>(ws, L.sx);
  float* sh = at<float>(ws, L.sh);
  const long long R = static_cast<long long>(rows_of(d));
  const int32_t* nvalid = offsets + d.E;
  if ((st = do_route(d, x, Wg, b, idx, gates, ws, L, stream)) != MOE_OK) return st;
  if ((st = do_dispatch(d, selection(d, 0, d.E), idx, at<int32_t>(saved, S.counts), offsets, psrc,
                        pdst, ws, L, stream)) != MOE_OK)
    return st;
  // e4m3 rows for FC1 and, in the same pass, the bf16 rows the backward's FC1
  // weight gradient takes
  MOE_RUN(moe::launch_quant_rows(x, psrc, d.k, R, d.T, d.h, Xq, sx, num_sms(), stream, nvalid,
                                 nullptr, 0, at<uint16_t>(saved, S.x_perm), nullptr, nullptr,
                                 at<int>(ws, 0)),
          "permute_quant_x");
  if (R > 0) {
    const GemmProblem g = problem(d, offsets, ws);
    MOE_RUN(moe::gemm_fc1_fwd_fp8(g, Xq, sx, at<uint8_t>(qw, Q.W13q), at<float>(qw, Q.s1),
                                  at<float>(qw, Q.s3), at<uint16_t>(saved, S.A),
                                  at<uint16_t>(saved, S.B), H, at<float>(ws, L.h_amax), stream),
            "gg_fc1_fwd_swiglu_fp8");
    MOE_RUN(moe::launch_quant_rows(H, nullptr, 1, R, R, d.f, Hq, sh, num_sms(), stream, nvalid,
                                   at<float>(ws, L.h_amax), moe::gemm_fc1_col_tiles(d.f)),
            "quant_h");
    MOE_RUN(moe::gemm_fc2_fwd_fp8(g, Hq, sh, at<uint8_t>(qw, Q.W2q), at<float>(qw, Q.s2), O,
                                  stream),
            "gg_fc2_fwd_fp8");
  }
  MOE_RUN(moe::launch_combine(O, gates, pdst, d.T, d.k, d.h, y, num_sms(), stream,
                              at<int>(ws, 0)),
          "combine");
  return MOE_OK;
}

size_t moe_fp8_bwd_weight_bytes(const moe_dims* dims) {
  if (check_dims(dims, false) != MOE_OK || !fp8_shape_ok(*dims)) return 0;
  return fp8_bwd_weight_layout(*dims).total;
}

void* moe_fp8_bwd_weight_view(const moe_dims* dims, void* qwb, const char* name) {
  if (check_dims(dims, false) != MOE_OK || !fp8_shape_ok(*dims) || !qwb || !name) return nullptr;
  const Fp8BwdWeightLayout L = fp8_bwd_weight_layout(*dims);
  struct {
    const char* n;
    size_t off;
  } tab[] = {{"W1r", L.W1r}, {"W3r", L.W3r}, {"s13r", L.s13r}};
  for (auto& e : tab)
    if (strcmp(e.n, name) == 0) return at<uint8_t>(qwb, e.off);
  return nullptr;
}

moe_status moe_quantize_weights_fp8_bwd(const moe_dims* dims, const moe_bf16* W1,
                                        const moe_bf16* W3, void* qwb, moe_stream_t stream_) {
  moe_status st = check_dims(dims, false);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!fp8_shape_ok(d)) return MOE_ERR_UNSUPPORTED;
  if (!ptr_ok(W1) || !ptr_ok(W3) || !qwb || !aligned(qwb, kAlign)) return MOE_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const Fp8BwdWeightLayout L = fp8_bwd_weight_layout(d);
  const long long Eh = static_cast<long long>(d.E) * d.h;
  // W1, W3 [E, h, f]: rows h, one scale over both matrices' rows
  MOE_RUN(moe::launch_quant_rows(W1, nullptr, 1, Eh, Eh, d.f, at<uint8_t>(qwb, L.W1r),
                                 at<float>(qwb, L.s13r), num_sms(), stream, nullptr, nullptr, 0,
                                 nullptr, W3, at<uint8_t>(qwb, L.W3r)),
          "quant_w13_rows");
  return MOE_OK;
}

moe_status moe_layer_bwd_fp8(const moe_dims* dims, const moe_bf16* x, const moe_bf16* dy,
                             const float* Wg, const moe_bf16* W2, const void* qwb,
                             const void* saved, moe_bf16* dx,
                             float* dWg, float* dW1, float* dW3, float* dW2, void* ws,
                             size_t ws_bytes, moe_stream_t stream_) {
  moe_status st = check_dims(dims, true);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  if (!fp8_shape_ok(d) || d.sar) return MOE_ERR_UNSUPPORTED;
  const size_t T = d.T;
  if (!buf_ok(x, T) || !buf_ok(dy, T) || !ptr_ok(Wg) || !ptr_ok(W2) || !qwb ||
      !aligned(qwb, kAlign) ||
      !saved || !aligned(saved, kAlign) || !buf_ok(dx, T) || !ptr_ok(dWg) || !ptr_ok(dW1) ||
      !ptr_ok(dW3) || !ptr_ok(dW2))
    return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(d, MOE_OP_LAYER_BWD_FP8, ws, ws_bytes)) != MOE_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const WsLayout L = ws_layout(d, MOE_OP_LAYER_BWD_FP8);
  const SavedLayout S = saved_layout(d);
  const Fp8BwdWeightLayout Q = fp8_bwd_weight_layout(d);
  const int32_t* idx = at<int32_t>(saved, S.topk_idx);
  const float* gates = at<float>(saved, S.gates);
  const int32_t* offsets = at<int32_t>(saved, S.offsets);
  const int32_t* psrc = at<int32_t>(saved, S.perm_src);
  const int32_t* pdst = at<int32_t>(saved, S.perm_dst);
  uint16_t* dO = at<uint16_t>(ws, L.dO);
  uint16_t* dA = at<uint16_t>(ws, L.dA);
  uint16_t* dB = at<uint16_t>(ws, L.dB);
  float* dX = at<float>(ws, L.dX);
  float* dg = at<float>(ws, L.dg);
  const long long R = static_cast<long long>(rows_of(d));
  const int32_t* nvalid = offsets + d.E;
  MOE_RUN(moe::launch_bwd_prep(dy, at<uint16_t>(saved, S.O), gates, psrc, R, d.k, d.h, dO, dg,
                               num_sms(), stream, nvalid, at<int>(ws, 0)),
          "bwd_prep");
  if (R == 0) {
    const size_t wbytes = static_cast<size_t>(d.E) * d.h * d.f * 4;
    MOE_RUN(cudaMemsetAsync(dW1, 0, wbytes, stream), "zero_dW1");
    MOE_RUN(cudaMemsetAsync(dW3, 0, wbytes, stream), "zero_dW3");
    MOE_RUN(cudaMemsetAsync(dW2, 0, wbytes, stream), "zero_dW2");
  } else {
    const GemmProblem g = problem(d, offsets, ws);
    // FC2 dgrad stays bf16 (its cost is the fused SwiGLU-backward epilogue);
    // it also records the per-tile amax of dA and dB for their e4m3 scale
    MOE_RUN(moe::gemm_fc2_dgrad(g, dO, W2, at<uint16_t>(saved, S.A), at<uint16_t>(saved, S.B), dA,
                                dB, stream, at<float>(ws, L.ab_amax)),
            moe::kGemmNames[2]);
    MOE_RUN(moe::launch_quant_rows(dA, nullptr, 1, R, R, d.f, at<uint8_t>(ws, L.dAq),
                                   at<float>(ws, L.sab), num_sms(), stream, nvalid,
                                   at<float>(ws, L.ab_amax), moe::gemm_col_tiles(d.f), nullptr,
                                   dB, at<uint8_t>(ws, L.dBq)),
            "quant_dAdB");
    MOE_RUN(moe::gemm_fc2_wgrad(g, at<uint16_t>(saved, S.H), dO, dW2, stream),
            moe::kGemmNames[4]);
    MOE_RUN(moe::gemm_fc1_dgrad_fp8(g, at<uint8_t>(ws, L.dAq), at<uint8_t>(ws, L.dBq),
                                    at<float>(ws, L.sab), at<uint8_t>(qwb, Q.W1r),
                                    at<uint8_t>(qwb, Q.W3r), at<float>(qwb, Q.s13r), dX, stream),
            "gg_fc1_dgrad_fp8");
    MOE_RUN(moe::gemm_fc1_wgrad(g, at<uint16_t>(saved, S.x_perm), dA, dB, dW1, dW3, stream),
            moe::kGemmNames[5]);
  }
  return do_router_bwd(d, x, Wg, idx, gates, dg, dX, pdst, dx, dWg, ws, L, stream);
}

moe_status moe_layer_bwd(const moe_dims* dims, const moe_bf16* x, const moe_bf16* dy,
                         const float* Wg, const moe_bf16* W1, const moe_bf16* W3,
                         const moe_bf16* W2, const void* saved, moe_bf16* dx, float* dWg,
                         float* dW1, float* dW3, float* dW2, void* ws, size_t ws_bytes,
                         moe_stream_t stream_) {
  moe_status st = check_dims(dims, true);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  const size_t T = d.T;
  if (!buf_ok(x, T) || !buf_ok(dy, T) || !ptr_ok(Wg) || !ptr_ok(W1) || !ptr_ok(W3) ||
      !ptr_ok(W2) || !saved || !aligned(saved, kAlign) || !buf_ok(dx, T) || !ptr_ok(dWg) ||
      !ptr_ok(dW1) || !ptr_ok(dW3) || !ptr_ok(dW2))
    return MOE_ERR_INVALID_ARG;
  if ((st = ws_check(d, MOE_OP_LAYER_BWD, ws, ws_bytes)) != MOE_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const WsLayout L = ws_layout(d, MOE_OP_LAYER_BWD);
  const SavedLayout S = saved_layout(d);
  const int32_t* idx = at<int32_t>(saved, S.topk_idx);
  const float* gates = at<float>(saved, S.gates);
  const int32_t* offsets = at<int32_t>(saved, S.offsets);
  const int32_t* psrc = at<int32_t>(saved, S.perm_src);
  const int32_t* pdst = at<int32_t>(saved, S.perm_dst);
  uint16_t* dO = at<uint16_t>(ws, L.dO);
  float* dX = at<float>(ws, L.dX);
  float* dg = at<float>(ws, L.dg);
  const long long R = static_cast<long long>(rows_of(d));
  if (d.sar) {
    if ((st = do_ffn_bwd_sar(d, x, dy, gates, psrc, offsets, W1, W3, W2, at<uint16_t>(saved, S.A),
                             at<uint16_t>(saved, S.B), dX, dg, dW1, dW3, dW2, ws, L, stream)) !=
        MOE_OK)
      return st;
    return do_router_bwd(d, x, Wg, idx, gates, dg, dX, pdst, dx, dWg, ws, L, stream);
  }
  MOE_RUN(moe::launch_bwd_prep(dy, at<uint16_t>(saved, S.O), gates, psrc, R, d.k, d.h, dO, dg,
                               num_sms(), stream, offsets + d.E, at<int>(ws, 0)),
          "bwd_prep");
  if ((st = do_ffn_bwd(d, at<uint16_t>(saved, S.x_perm), dO, offsets, W1, W3, W2,
                       at<uint16_t>(saved, S.A), at<uint16_t>(saved, S.B),
                       at<uint16_t>(saved, S.H), at<uint16_t>(ws, L.dA), at<uint16_t>(ws, L.dB),
                       dX, dW1, dW3, dW2, ws, stream)) != MOE_OK)
    return st;
  return do_router_bwd(d, x, Wg, idx, gates, dg, dX, pdst, dx, dWg, ws, L, stream);
}

}  // extern "C"
