// noalloc.cu -- moe_permute_noalloc: the dispatch step without a workspace.
//
// Some callers cannot call cudaMalloc at the point where they dispatch
// tokens, such as a host runtime or plugin that owns a fixed device-memory
// budget and hands its kernels only their inputs and outputs.  For them this
// entry point keeps its scratch memory --
// the per-block expert counts and the per-block base offsets of the stable
// scatter -- in one fixed-size array that lives in the library's own device
// memory.  Every GPU that loads the library holds that array until the
// process exits.
//
// The array is a host-side stand-in in host code, not a device address; the
// address kernels need is looked up with cudaGetSymbolAddress, once per
// device, on the first call made with that device current.
//
// All calls share the one array and it keeps whatever the last call left in
// it.  Nothing in it has to start at zero: each call writes every entry it
// later reads.  Calls whose kernels overlap on the GPU (different streams,
// no ordering between them) race on the array and produce wrong maps.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "../../include/moe.h"
#include "api_internal.h"
#include "kernels.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(1) << 20;  // 1 MiB
constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Device address of the scratch array on the current device.
moe_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// a launcher's result, reported to the measurement hook like every other entry point's
bool ran(cudaError_t e, cudaStream_t s, const char* name) {
  return e == cudaSuccess && moe_api::note(s, name);
}
bool buf_ok(const void* p, size_t n) { return n == 0 ? (p == nullptr || aligned16(p)) : (p && aligned16(p)); }

}  // namespace

extern "C" moe_status moe_permute_noalloc(const moe_dims* dims, const int32_t* topk_idx,
                                          const moe_bf16* x, int32_t* counts, int32_t* offsets,
                                          int32_t* perm_src, int32_t* perm_dst, moe_bf16* x_perm,
                                          moe_stream_t stream_) {
  // the same checks as moe_permute
  moe_status st = moe_api::check_dims(dims, false);
  if (st != MOE_OK) return st;
  const moe_dims& d = *dims;
  const long long R = static_cast<long long>(d.T) * d.k;
  if (!buf_ok(topk_idx, R) || !buf_ok(counts, 1) || !buf_ok(offsets, 1) ||
      !buf_ok(perm_src, R) || !buf_ok(perm_dst, R))
    return MOE_ERR_INVALID_ARG;
  if ((x && !aligned16(x)) || (x_perm && !aligned16(x_perm))) return MOE_ERR_INVALID_ARG;

  // scratch: per-block counts [nblk, E] and bases [nblk, E], int32 each
  const int nblk = moe::dispatch_blocks(R);
  const size_t part = align_up(static_cast<size_t>(nblk) * d.E * sizeof(int32_t));
  if (2 * part > kScratchBytes) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch

  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != MOE_OK) return st;
  // index errors go to the per-device status word of the calls without a workspace
  int* status = moe::nows_status_word();
  if (!status) return MOE_ERR_CUDA;
  int32_t* blk_counts = static_cast<int32_t*>(scratch);
  int32_t* bases = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(scratch) + part);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream_);
  const moe::DispatchSel sel{0, d.E, d.capacity > 0 ? d.capacity : INT_MAX};
  if (!ran(moe::launch_dispatch_hist(topk_idx, R, d.E, sel, blk_counts, s, status), s,
           "dispatch_hist") ||
      !ran(moe::launch_dispatch_scan(blk_counts, nblk, sel, counts, offsets, bases, s), s,
           "dispatch_scan") ||
      !ran(moe::launch_dispatch_scatter(topk_idx, R, d.E, sel, bases, offsets, perm_src, perm_dst,
                                        s, status),
           s, "dispatch_scatter"))
    return MOE_ERR_CUDA;
  if (x && x_perm &&
      !ran(moe::launch_gather_rows(x, perm_src, d.k, R, d.T, d.h, x_perm, moe_api::num_sms(), s,
                                   offsets + d.E, nullptr, nullptr, status),
           s, "permute_rows"))
    return MOE_ERR_CUDA;
  return MOE_OK;
}
