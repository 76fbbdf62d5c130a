// moe_router_topk_noalloc: the router + capacity slotting for callers that
// cannot allocate device memory (a plugin whose host program owns every
// allocation, a fixed start-up memory budget, or a latency-critical loop that
// cannot pay for cudaMalloc's implicit device synchronisation).
//
// It runs the same kernels as moe_router_topk for the same layer (the
// tensor-core router for bf16 layers of at least 128 tokens, the SIMT router
// otherwise), so its results are bit for bit those of moe_router_topk.  The
// routing histograms, their scan, the last-block ticket and, for the
// tensor-core router, the three bf16 parts of W_r live in a file-scope device
// array owned by this library.  Host code cannot use the array's name as a
// device address, so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current and keeps it.  Nothing
// here calls cudaMalloc, cudaFree or an allocating library routine.  Every
// call on a device shares the array and sees the previous call's contents:
// the router kernel clears the ticket itself and every other word is
// rewritten before it is read, but calls that overlap on the GPU race.
#include <mutex>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kAlign = 256;
inline size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

std::mutex g_mu;
void* g_scratch_addr[64] = {nullptr};

// Device address of the scratch array on the current device (looked up once per device).
moe_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

inline moe_status check_ptr(const void* p, size_t a) {
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  return (reinterpret_cast<uintptr_t>(p) % a) == 0 ? MOE_OK : MOE_ERR_ALIGNMENT;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_router_topk_noalloc(const moe_config* cfg, const void* x, const float* W_r,
                                              const float* bias, int32_t* ids, float* gates, float* probs,
                                              int32_t* slot, int32_t* row_of, int32_t* src_token, int32_t* counts,
                                              int32_t* offsets, moe_stream_t stream) {
  using namespace moe;
  Shape s;
  moe_status st = static_cast<moe_status>(validate_config(cfg, &s));
  if (st != MOE_OK) return st;
  const void* p16[] = {x};
  const void* p4[] = {W_r, ids, gates, slot, row_of, src_token, counts, offsets};
  for (const void* p : p16)
    if ((st = check_ptr(p, 16)) != MOE_OK) return st;
  for (const void* p : p4)
    if ((st = check_ptr(p, 4)) != MOE_OK) return st;
  if (bias != nullptr && (st = check_ptr(bias, 4)) != MOE_OK) return st;
  if (probs != nullptr && (st = check_ptr(probs, 4)) != MOE_OK) return st;

  // scratch layout: hist | base (E*k*blocks ints each) | totals (E ints) | ticket | W_r parts (tensor-core router)
  const size_t n = (size_t)s.E * s.k * router_blocks(s.T);
  const bool tc = router_tc_supported(s);
  const size_t o_scan = round_up(n * 4), o_totals = 2 * round_up(n * 4);
  const size_t o_ticket = o_totals + round_up((size_t)s.E * 4), o_wsplit = o_ticket + round_up(4);
  const size_t bytes = o_wsplit + (tc ? round_up(router_wsplit_bytes(s)) : 0);
  if (bytes > MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;

  uint32_t* err = nullptr;
  if ((st = static_cast<moe_status>(current_error_word(&err))) != MOE_OK) return st;
  void* base = nullptr;
  if ((st = scratch_address(&base)) != MOE_OK) return st;
  char* b = static_cast<char*>(base);
  int32_t* hist = reinterpret_cast<int32_t*>(b);
  int32_t* scan = reinterpret_cast<int32_t*>(b + o_scan);
  int32_t* totals = reinterpret_cast<int32_t*>(b + o_totals);
  int32_t* ticket = reinterpret_cast<int32_t*>(b + o_ticket);

  if (s.T == 0) {
    if (cudaMemsetAsync(counts, 0, (size_t)s.E * 4, stream) != cudaSuccess ||
        cudaMemsetAsync(offsets, 0, (size_t)(s.E + 1) * 4, stream) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const cudaError_t e = tc ? launch_router_tc(s, x, W_r, bias, b + o_wsplit, ids, gates, probs, hist, ticket, err,
                                              stream)
                           : launch_router(s, x, W_r, bias, ids, gates, probs, hist, ticket, stream);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_slot_scan(s, hist, scan, totals, ticket, counts, offsets, err, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_slot_assign(s, ids, scan, counts, offsets, slot, row_of, src_token, err, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
