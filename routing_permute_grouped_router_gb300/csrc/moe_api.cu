// C ABI of the mixture-of-experts layer step: argument validation, workspace
// carving, the per-device error word, launch accounting, the optional event
// profiler, and the sequencing of the kernels in routing.cu, rows.cu,
// gemm_tc.cu and gemm_simt.cu.  Declarations and contracts are in moe.h.
#include <atomic>
#include <climits>
#include <cmath>
#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {

// ------------------------------ error word -------------------------------- //
__device__ uint32_t g_device_error[2];

namespace {

struct DeviceState {
  bool init = false;
  bool supported = false;
  uint32_t* err = nullptr;
};
std::mutex g_dev_mu;
DeviceState g_dev[64];

moe_status device_ready(uint32_t** err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceState& ds = g_dev[dev];
  if (!ds.init) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    ds.supported = (major == 10 && minor == 3);
    if (ds.supported) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return MOE_ERR_CUDA;
      ds.err = static_cast<uint32_t*>(p);
    }
    ds.init = true;
  }
  if (!ds.supported) return MOE_ERR_UNSUPPORTED;
  *err = ds.err;
  return MOE_OK;
}

// ------------------------------ accounting -------------------------------- //
std::atomic<uint64_t> g_launches{0};

struct ProfRec {
  int kind;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
int g_prof_filter = -1;
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_event_pool;
thread_local int t_open_rec = -1;
// NVTX ranges around every launch and layer call, for nsys/ncu timelines
std::atomic<bool> g_nvtx{false};
thread_local bool t_nvtx_open = false;

cudaEvent_t pool_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

const char* const kKernelNames[KK_COUNT] = {
    "router_topk",  "slot_scan",  "slot_assign",     "permute",      "gemm_up_swiglu", "gemm_down",
    "unpermute_combine", "combine_bwd", "gemm_dgrad_h_swiglu_bwd", "gemm_wgrad", "gemm_dgrad_x",
    "transpose_wr", "dx_router",  "dwr",     "dwr_reduce",   "zero", "split_wr", "selftest_bounded_wait",
    "split_dl", "aux_loss", "aux_grad", "router_logit_grad"};

}  // namespace

void launch_begin(int kind, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  t_nvtx_open = g_nvtx.load(std::memory_order_relaxed);
  if (t_nvtx_open) nvtxRangePushA(kKernelNames[kind]);
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_on || (g_prof_filter >= 0 && g_prof_filter != kind)) {
    t_open_rec = -1;
    return;
  }
  ProfRec r{kind, pool_event(), pool_event()};
  cudaEventRecord(r.a, s);
  g_prof_recs.push_back(r);
  t_open_rec = (int)g_prof_recs.size() - 1;
}

void launch_end(int kind, cudaStream_t s) {
  (void)kind;
  if (t_nvtx_open) nvtxRangePop();
  t_nvtx_open = false;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (t_open_rec >= 0 && t_open_rec < (int)g_prof_recs.size()) cudaEventRecord(g_prof_recs[t_open_rec].b, s);
  t_open_rec = -1;
}

namespace {

// An NVTX range over a whole layer call while NVTX ranges are on.
struct NvtxScope {
  bool on;
  explicit NvtxScope(const char* name) : on(g_nvtx.load(std::memory_order_relaxed)) {
    if (on) nvtxRangePushA(name);
  }
  ~NvtxScope() {
    if (on) nvtxRangePop();
  }
};

// ------------------------------ validation -------------------------------- //
constexpr size_t ALIGN = 256;
inline size_t up(size_t x, size_t a = ALIGN) { return (x + a - 1) / a * a; }

moe_status make_shape(const moe_config* c, Shape* s) {
  if (c == nullptr || s == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_DTYPE;
  if (c->T < 0 || c->d_model <= 0 || c->d_ff <= 0 || c->E < 1 || c->E > 128 || c->k < 1 || c->k > 8 ||
      c->k > c->E)
    return MOE_ERR_SHAPE;
  const bool bf16 = c->dtype == MOE_BF16;
  if (bf16 && (c->d_model % 256 != 0 || c->d_ff % 256 != 0)) return MOE_ERR_SHAPE;
  if (!bf16 && (c->d_model % 4 != 0 || c->d_ff % 4 != 0)) return MOE_ERR_SHAPE;
  if (c->d_model > (1 << 16) || c->d_ff > (1 << 16)) return MOE_ERR_SHAPE;
  const int64_t Tk = (int64_t)c->T * c->k;
  if (Tk > (int64_t)1 << 28) return MOE_ERR_SHAPE;
  int64_t cap = INT_MAX;
  if (c->capacity >= 0) {
    cap = c->capacity;
  } else if (c->capacity_factor > 0.f) {
    if (!std::isfinite(c->capacity_factor)) return MOE_ERR_SHAPE;
    const double v = std::ceil((double)c->capacity_factor * (double)c->T * (double)c->k / (double)c->E);
    if (v > (double)INT_MAX) return MOE_ERR_SHAPE;
    cap = (int64_t)v;
  }
  int64_t rows = Tk + 127 * (int64_t)c->E;
  if (cap != INT_MAX) {
    const int64_t rc = (int64_t)c->E * ((cap + 127) / 128 * 128);
    if (rc < rows) rows = rc;
  }
  rows = (rows + 127) / 128 * 128;
  if (rows > (int64_t)INT_MAX - 128) return MOE_ERR_SHAPE;
  if (!std::isfinite(c->aux_loss_coeff) || c->aux_loss_coeff < 0.f) return MOE_ERR_INVALID_ARG;
  s->T = c->T;
  s->d = c->d_model;
  s->f = c->d_ff;
  s->E = c->E;
  s->k = c->k;
  s->cap = (int)cap;
  s->bf16 = bf16 ? 1 : 0;
  s->max_rows = rows;
  s->aux = c->aux_loss_coeff;
  return MOE_OK;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
// The recompute variant: the caller keeps none of a, b, h (all three null).
inline bool recompute_mode(const moe_saved* sv) { return sv->a == nullptr && sv->b == nullptr && sv->h == nullptr; }
inline moe_status need(const void* p, size_t a = 16) {
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  return aligned(p, a) ? MOE_OK : MOE_ERR_ALIGNMENT;
}
#define MOE_TRY(expr)                 \
  do {                                \
    const moe_status st_ = (expr);    \
    if (st_ != MOE_OK) return st_;    \
  } while (0)
#define CUDA_TRY(expr)                             \
  do {                                             \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

// ------------------------------ workspace --------------------------------- //
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  void* take(size_t bytes) {
    void* p = base ? base + off : nullptr;
    off += up(bytes);
    return p;
  }
};

struct RoutingScratch {
  int32_t* hist;
  int32_t* base;
  int32_t* totals;
  int32_t* ticket;
  void* wsplit;  // bf16 parts of W_r for the tensor-core router
};
struct FwdScratch {
  int32_t *ids, *slot, *row_of, *src_token, *counts, *offsets;
  float* gates;
  void *x_perm, *h, *y_perm;
  float* row_gate;  // gate of each row (inference forward with the combine in the down product)
};
// The layer backward takes dg from the dgrad h product (and skips reading Y_perm
// back in the combine backward) when the Y_perm bytes saved, up to T k d of
// bf16, are at least 256 MB; below that the extra launch costs about as much
// as the read it saves or more (top-2 E=8 layer: +6 us a step; 4-micro-batch
// E=16 and Zipf E=64: within 0.2 %; dropless E=32: -170 us).
bool fused_dg_pays(const Shape& s) { return s.bf16 && (int64_t)s.T * s.k * s.d * 2 >= ((int64_t)256 << 20); }

struct BwdScratch {
  void *dy_perm, *da, *db, *dx_perm;
  float *dg, *dl, *W_rT, *partial;
  float* sdot;    // bf16: per row and 256-column tile, sum of dH * h (the layer backward's dg * g)
  int* round_ctr;  // bf16: wgrad's round counters
  void* dlsplit;  // bf16 parts of dl for the tensor-core router-weight gradient
  void* aux;      // auxiliary-loss partial sums
};

RoutingScratch carve_routing(Carver& c, const Shape& s) {
  const size_t n = (size_t)s.E * s.k * router_blocks(s.T);
  RoutingScratch r;
  r.hist = static_cast<int32_t*>(c.take(n * 4));
  r.base = static_cast<int32_t*>(c.take(n * 4));
  r.totals = static_cast<int32_t*>(c.take((size_t)s.E * 4));
  r.ticket = static_cast<int32_t*>(c.take(4));
  r.wsplit = c.take(router_wsplit_bytes(s));
  return r;
}
FwdScratch carve_fwd(Carver& c, const Shape& s) {
  const size_t Tk = (size_t)s.T * s.k, R = (size_t)s.max_rows, es = s.bf16 ? 2 : 4;
  FwdScratch f;
  f.ids = static_cast<int32_t*>(c.take(Tk * 4));
  f.slot = static_cast<int32_t*>(c.take(Tk * 4));
  f.row_of = static_cast<int32_t*>(c.take(Tk * 4));
  f.gates = static_cast<float*>(c.take(Tk * 4));
  f.counts = static_cast<int32_t*>(c.take((size_t)s.E * 4));
  f.offsets = static_cast<int32_t*>(c.take((size_t)(s.E + 1) * 4));
  f.src_token = static_cast<int32_t*>(c.take(R * 4));
  f.x_perm = c.take(R * s.d * es);
  f.h = c.take(R * s.f * es);
  f.y_perm = c.take(R * s.d * es);
  f.row_gate = static_cast<float*>(c.take(R * 4));
  return f;
}
BwdScratch carve_bwd(Carver& c, const Shape& s) {
  const size_t R = (size_t)s.max_rows, es = s.bf16 ? 2 : 4;
  BwdScratch b;
  b.dy_perm = c.take(R * s.d * es);
  b.da = c.take(R * s.f * es);
  b.db = c.take(R * s.f * es);
  b.dx_perm = c.take(R * s.d * es);
  b.dg = static_cast<float*>(c.take((size_t)s.T * s.k * 4));
  b.dl = static_cast<float*>(c.take((size_t)s.T * s.E * 4));
  b.W_rT = static_cast<float*>(c.take((size_t)s.E * s.d * 4));
  const bool tc = dwr_tc_supported(s);
  b.partial = static_cast<float*>(c.take((size_t)(tc ? dwr_tc_ranges(s) : dwr_splits(s)) * s.d * s.E * 4));
  b.dlsplit = c.take(tc ? dwr_tc_split_bytes(s) : 0);
  b.aux = c.take(aux_scratch_bytes(s));
  b.sdot = static_cast<float*>(c.take(fused_dg_pays(s) ? R * (size_t)(s.f / 256) * 4 : 0));
  b.round_ctr = static_cast<int*>(c.take(s.bf16 ? sizeof(int) * WG_ROUNDS : 0));
  return b;
}
// a, b, h of the expert FFN when the forward does not keep them (the
// recompute variant): the forward writes h here for the down product, the
// backward recomputes all three here before the dgrad.
struct RecomputeScratch {
  void *a, *b, *h;
};
RecomputeScratch carve_recompute(Carver& c, const Shape& s) {
  const size_t n = (size_t)s.max_rows * s.f * (s.bf16 ? 2 : 4);
  RecomputeScratch r;
  r.a = c.take(n);
  r.b = c.take(n);
  r.h = c.take(n);
  return r;
}
// training: 0 inference, 1 training, 2 training with the activations recomputed
size_t ws_bytes_for(const Shape& s, int training) {
  Carver c(nullptr);
  carve_routing(c, s);
  if (training) carve_bwd(c, s);
  else carve_fwd(c, s);
  if (training == 2) carve_recompute(c, s);
  return c.off + ALIGN;  // room to align an unaligned base
}
void* align_ws(void* ws) {
  return reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(ws) + ALIGN - 1) / ALIGN * ALIGN);
}

// ------------------------------ steps ------------------------------------- //
moe_status do_router(const Shape& s, const void* x, const float* W_r, const float* bias, int32_t* ids, float* gates,
                     float* probs, int32_t* slot, int32_t* row_of, int32_t* src_token, int32_t* counts,
                     int32_t* offsets, const RoutingScratch& rs, uint32_t* err, cudaStream_t st) {
  if (s.T == 0) {
    CUDA_TRY(cudaMemsetAsync(counts, 0, (size_t)s.E * 4, st));
    CUDA_TRY(cudaMemsetAsync(offsets, 0, (size_t)(s.E + 1) * 4, st));
    return MOE_OK;
  }
  if (router_tc_supported(s))
    CUDA_TRY(launch_router_tc(s, x, W_r, bias, rs.wsplit, ids, gates, probs, rs.hist, rs.ticket, err, st));
  else
    CUDA_TRY(launch_router(s, x, W_r, bias, ids, gates, probs, rs.hist, rs.ticket, st));
  CUDA_TRY(launch_slot_scan(s, rs.hist, rs.base, rs.totals, rs.ticket, counts, offsets, err, st));
  CUDA_TRY(launch_slot_assign(s, ids, rs.base, counts, offsets, slot, row_of, src_token, err, st));
  return MOE_OK;
}

moe_status do_ffn_fwd(const Shape& s, const FfnFwdArgs& f, uint32_t* err, cudaStream_t st) {
  if (s.max_rows == 0 || s.T == 0) return MOE_OK;
  cudaError_t e = s.bf16 ? tc_ffn_fwd(s, f, err, st) : simt_ffn_fwd(s, f, err, st);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status do_ffn_bwd(const Shape& s, const FfnBwdArgs& b, uint32_t* err, cudaStream_t st) {
  if (s.max_rows == 0 || s.T == 0) {
    if (b.accumulate || b.part == 1) return MOE_OK;
    const size_t n = (size_t)s.E * s.d * s.f * 4;
    CUDA_TRY(cudaMemsetAsync(b.dW1, 0, n, st));
    CUDA_TRY(cudaMemsetAsync(b.dW3, 0, n, st));
    CUDA_TRY(cudaMemsetAsync(b.dW2, 0, n, st));
    return MOE_OK;
  }
  cudaError_t e = s.bf16 ? tc_ffn_bwd(s, b, err, st) : simt_ffn_bwd(s, b, err, st);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status do_dx_router(const Shape& s, const void* x, const void* dx_perm, const int32_t* row_of, const float* dl,
                        const float* W_r, void* dx, float* dW_r, int accumulate, const BwdScratch& bs, uint32_t* err,
                        cudaStream_t st, const int32_t* kept_ids = nullptr) {
  if (s.T == 0) {
    if (!accumulate) CUDA_TRY(cudaMemsetAsync(dW_r, 0, (size_t)s.d * s.E * 4, st));
    return MOE_OK;
  }
  CUDA_TRY(launch_dx_router(s, dx_perm, row_of, dl, W_r, bs.W_rT, dx, err, st, kept_ids));
  if (dwr_tc_supported(s)) {
    CUDA_TRY(launch_dwr_tc(s, x, dl, bs.dlsplit, bs.partial, err, st));
    CUDA_TRY(launch_dwr_reduce(bs.partial, dW_r, dwr_tc_ranges(s), (int64_t)s.d * s.E, accumulate, st));
  } else {
    CUDA_TRY(launch_dwr(s, x, dl, bs.partial, dW_r, accumulate, st));
  }
  return MOE_OK;
}

}  // namespace

int validate_config(const void* cfg, Shape* s) { return make_shape(static_cast<const moe_config*>(cfg), s); }
int current_error_word(uint32_t** err) { return device_ready(err); }

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_SHAPE: return "MOE_ERR_SHAPE";
    case MOE_ERR_DTYPE: return "MOE_ERR_DTYPE";
    case MOE_ERR_ALIGNMENT: return "MOE_ERR_ALIGNMENT";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_CHECK: return "MOE_ERR_DEVICE_CHECK";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status moe_capacity(const moe_config* cfg, int32_t* C) {
  Shape s;
  MOE_TRY(make_shape(cfg, &s));
  if (C == nullptr) return MOE_ERR_INVALID_ARG;
  *C = s.cap == INT_MAX ? -1 : s.cap;
  return MOE_OK;
}

moe_status moe_max_rows(const moe_config* cfg, int64_t* rows) {
  Shape s;
  MOE_TRY(make_shape(cfg, &s));
  if (rows == nullptr) return MOE_ERR_INVALID_ARG;
  *rows = s.max_rows;
  return MOE_OK;
}

moe_status moe_workspace_size(const moe_config* cfg, int training, size_t* bytes) {
  Shape s;
  MOE_TRY(make_shape(cfg, &s));
  if (bytes == nullptr || training < 0 || training > 2) return MOE_ERR_INVALID_ARG;
  *bytes = ws_bytes_for(s, training);
  return MOE_OK;
}

moe_status moe_router_topk(const moe_config* cfg, const void* x, const float* W_r, const float* bias, int32_t* ids,
                           float* gates, float* probs, int32_t* slot, int32_t* row_of, int32_t* src_token,
                           int32_t* counts, int32_t* offsets, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Shape s;
  MOE_TRY(make_shape(cfg, &s));
  MOE_TRY(need(x));
  MOE_TRY(need(W_r, 4));
  if (bias != nullptr) MOE_TRY(need(bias, 4));
  if (probs != nullptr) MOE_TRY(need(probs, 4));
  MOE_TRY(need(ids, 4));
  MOE_TRY(need(gates, 4));
  MOE_TRY(need(slot, 4));
  MOE_TRY(need(row_of, 4));
  MOE_TRY(need(src_token, 4));
  MOE_TRY(need(counts, 4));
  MOE_TRY(need(offsets, 4));
  if (ws == nullptr || ws_bytes < ws_bytes_for(s, 0)) return MOE_ERR_WORKSPACE;
  uint32_t* err = nullptr;
  MOE_TRY(device_ready(&err));
  Carver c(align_ws(ws));
  RoutingScratch rs = carve_routing(c, s);
  return do_router(s, x, W_r, bias, ids, gates, probs, slot, row_of, src_token, counts, offsets, rs, err, stream);
}

moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* row_of, const int32_t* counts,
                       const int32_t* offsets, void* x_perm, moe_stream_t stream) {
  Shape s;
  MOE_TRY(make_shape(cfg, &s));
  MOE_TRY(need(x));
  MOE_TRY(need(row_of, 4));
  MOE_TRY(need(counts, 4));
  MOE_TRY(need(offsets, 4));
  MOE_TRY(need(x_perm));
  uint32_t* err = nullptr;
  MOE_TRY(device_ready(&err));
  if (s.T == 0) return MOE_OK;
  CUDA_TRY(launch_permute(s, x, row_of, counts, offsets, x_perm, err, stream));
  return MOE_OK;
}

moe_status moe_grouped_ffn(const moe_config* cfg, const void* x_perm, const int32_t* counts, const int32_t* offsets,
                           const void* W1, const void* W3, const void* W2, void* h, void* y_perm, void* a, void* b,
                           moe_stream_t stream) {
  Shape s;
  MOE_TRY(make_shape(cfg, &s));
  MOE_TRY(need(x_perm));
  MOE_TRY(need(counts, 4));
  MOE_TRY(need(offsets, 4));
  MOE_TRY(need(W1));
  MOE_TRY(need(W3));
  MOE_TRY(need(W2));
  MOE_TRY(need(h));
  MOE_TRY(need(y_perm));
  if (a != nullptr) MOE_TRY(need(a));
  if (b != nullptr) MOE_TRY(need(b));
  uint32_t* err = nullptr;
  MOE_TRY(device_ready(&err));
  FfnFwdArgs f{x_perm, counts, offsets, W1, W3, W2, h, y_perm, a, b};
  return do_ffn_fwd(s, f, err, stream);
}

moe_status moe_unpermute_combine(const moe_config* cfg, const void* y_perm, const int32_t* row_of, const float* gates,
                                 void* y, moe_stream_t stream) {
  Shape s;
  MOE_TRY(make_shape(cfg, &s));
  MOE_TRY(need(y_perm));
  MOE_TRY(need(row_of, 4));
  MOE_TRY(need(gates, 4));
  MOE_TRY(need(y));
  uint32_t* err = nullptr;
  MOE_TRY(device_ready(&err));
  CUDA_TRY(launch_combine(s, y_perm, row_of, gates, y, err, stream));
  return MOE_OK;
}

moe_status moe_layer_fwd(const moe_config* cfg, const moe_weights* w, const void* x, void* y, const moe_saved* saved,
                         void* ws, size_t ws_bytes, moe_stream_t stream) {
  Shape s;
  MOE_TRY(make_shape(cfg, &s));
  if (w == nullptr) return MOE_ERR_INVALID_ARG;
  MOE_TRY(need(x));
  MOE_TRY(need(y));
  MOE_TRY(need(w->W_r, 4));
  if (w->bias != nullptr) MOE_TRY(need(w->bias, 4));
  MOE_TRY(need(w->W1));
  MOE_TRY(need(w->W3));
  MOE_TRY(need(w->W2));
  if (saved != nullptr) {
    MOE_TRY(need(saved->ids, 4));
    MOE_TRY(need(saved->gates, 4));
    MOE_TRY(need(saved->slot, 4));
    MOE_TRY(need(saved->row_of, 4));
    MOE_TRY(need(saved->src_token, 4));
    MOE_TRY(need(saved->counts, 4));
    MOE_TRY(need(saved->offsets, 4));
    MOE_TRY(need(saved->probs, 4));
    MOE_TRY(need(saved->x_perm));
    MOE_TRY(need(saved->y_perm));
    if (!recompute_mode(saved)) {
      MOE_TRY(need(saved->a));
      MOE_TRY(need(saved->b));
      MOE_TRY(need(saved->h));
    }
  }
  Carver probe(nullptr);
  carve_routing(probe, s);
  const size_t need_ws = saved == nullptr ? ws_bytes_for(s, 0)
                         : recompute_mode(saved) ? ws_bytes_for(s, 2) : probe.off + ALIGN;
  if (ws == nullptr || ws_bytes < need_ws) return MOE_ERR_WORKSPACE;
  uint32_t* err = nullptr;
  MOE_TRY(device_ready(&err));
  NvtxScope range("moe_layer_fwd");
  Carver c(align_ws(ws));
  RoutingScratch rs = carve_routing(c, s);
  FwdScratch f;
  void *a = nullptr, *b = nullptr;
  float* probs = nullptr;
  if (saved != nullptr) {
    f.ids = saved->ids;
    f.slot = saved->slot;
    f.row_of = saved->row_of;
    f.gates = saved->gates;
    f.counts = saved->counts;
    f.offsets = saved->offsets;
    f.src_token = saved->src_token;
    f.x_perm = saved->x_perm;
    f.h = saved->h;
    f.y_perm = saved->y_perm;
    f.row_gate = nullptr;
    a = saved->a;
    b = saved->b;
    probs = saved->probs;
    if (recompute_mode(saved)) {  // h lives in the workspace; a and b are not kept
      carve_bwd(c, s);
      f.h = carve_recompute(c, s).h;
    }
  } else {
    f = carve_fwd(c, s);
  }
  MOE_TRY(do_router(s, x, w->W_r, w->bias, f.ids, f.gates, probs, f.slot, f.row_of, f.src_token, f.counts, f.offsets,
                    rs, err, stream));
  if (s.T == 0) return MOE_OK;
  // Inference forward of a bf16 layer with k <= 2: the combine runs in the down
  // product's epilogue (y zeroed by the permute, each row added in once with
  // its gate), so y_perm is neither written nor read back.
  const bool fused = saved == nullptr && s.bf16 && s.k <= 2;
  CUDA_TRY(launch_permute(s, x, f.row_of, f.counts, f.offsets, f.x_perm, err, stream, fused ? f.gates : nullptr,
                          fused ? f.row_gate : nullptr, fused ? y : nullptr));
  FfnFwdArgs fa{f.x_perm, f.counts, f.offsets, w->W1, w->W3, w->W2, f.h, f.y_perm, a, b};
  if (fused) {
    fa.src_token = f.src_token;
    fa.row_gate = f.row_gate;
    fa.y_comb = y;
  }
  MOE_TRY(do_ffn_fwd(s, fa, err, stream));
  if (!fused) CUDA_TRY(launch_combine(s, f.y_perm, f.row_of, f.gates, y, err, stream));
  return MOE_OK;
}

moe_status moe_combine_bwd(const moe_config* cfg, const void* dy, const void* y_perm, const int32_t* ids,
                           const int32_t* row_of, const float* gates, const float* probs, const int32_t* counts,
                           const int32_t* offsets, void* dy_perm, float* dg, float* dl, moe_stream_t stream) {
  Shape s;
  MOE_TRY(make_shape(cfg, &s));
  MOE_TRY(need(dy));
  MOE_TRY(need(y_perm));
  MOE_TRY(need(ids, 4));
  MOE_TRY(need(row_of, 4));
  MOE_TRY(need(gates, 4));
  if (s.k == 1) MOE_TRY(need(probs, 4));
  MOE_TRY(need(counts, 4));
  MOE_TRY(need(offsets, 4));
  MOE_TRY(need(dy_perm));
  MOE_TRY(need(dg, 4));
  MOE_TRY(need(dl, 4));
  uint32_t* err = nullptr;
  MOE_TRY(device_ready(&err));
  if (s.T == 0) return MOE_OK;
  CUDA_TRY(launch_combine_bwd(s, dy, y_perm, ids, row_of, gates, probs, counts, offsets, dy_perm, dg, dl, err,
                              stream));
  return MOE_OK;
}

moe_status moe_grouped_ffn_bwd(const moe_config* cfg, const void* x_perm, const void* a, const void* b, const void* h,
                               const void* dy_perm, const int32_t* counts, const int32_t* offsets, const void* W1,
                               const void* W3, const void* W2, void* da, void* db, void* dx_perm, float* dW1,
                               float* dW3, float* dW2, int accumulate, moe_stream_t stream) {
  Shape s;
  MOE_TRY(make_shape(cfg, &s));
  if (accumulate != 0 && accumulate != 1) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x_perm, a, b, h, dy_perm, W1, W3, W2, da, db, dx_perm, dW1, dW3, dW2};
  for (const void* p : ptrs) MOE_TRY(need(p));
  MOE_TRY(need(counts, 4));
  MOE_TRY(need(offsets, 4));
  uint32_t* err = nullptr;
  MOE_TRY(device_ready(&err));
  FfnBwdArgs fb{x_perm, a, b, h, dy_perm, counts, offsets, W1, W3, W2, da, db, dx_perm, dW1, dW3, dW2, accumulate};
  return do_ffn_bwd(s, fb, err, stream);
}

moe_status moe_aux_loss(const moe_config* cfg, const float* probs, const int32_t* ids, float* loss, float* dl,
                        void* ws, size_t ws_bytes, moe_stream_t stream) {
  Shape s;
  MOE_TRY(make_shape(cfg, &s));
  MOE_TRY(need(probs, 4));
  MOE_TRY(need(ids, 4));
  MOE_TRY(need(dl, 4));
  if (loss != nullptr) MOE_TRY(need(loss, 4));
  if (ws == nullptr || ws_bytes < ws_bytes_for(s, 1)) return MOE_ERR_WORKSPACE;
  uint32_t* err = nullptr;
  MOE_TRY(device_ready(&err));
  Carver c(align_ws(ws));
  carve_routing(c, s);
  BwdScratch bs = carve_bwd(c, s);
  CUDA_TRY(launch_aux_loss(s, s.aux, probs, ids, loss, dl, bs.aux, err, stream));
  return MOE_OK;
}

moe_status moe_unpermute_dx_router_bwd(const moe_config* cfg, const void* x, const void* dx_perm,
                                       const int32_t* row_of, const float* dl, const float* W_r, void* dx,
                                       float* dW_r, int accumulate, void* ws, size_t ws_bytes, moe_stream_t stream) {
  Shape s;
  MOE_TRY(make_shape(cfg, &s));
  if (accumulate != 0 && accumulate != 1) return MOE_ERR_INVALID_ARG;
  MOE_TRY(need(x));
  MOE_TRY(need(dx_perm));
  MOE_TRY(need(row_of, 4));
  MOE_TRY(need(dl, 4));
  MOE_TRY(need(W_r, 4));
  MOE_TRY(need(dx));
  MOE_TRY(need(dW_r, 4));
  if (ws == nullptr || ws_bytes < ws_bytes_for(s, 1)) return MOE_ERR_WORKSPACE;
  uint32_t* err = nullptr;
  MOE_TRY(device_ready(&err));
  Carver c(align_ws(ws));
  carve_routing(c, s);
  BwdScratch bs = carve_bwd(c, s);
  return do_dx_router(s, x, dx_perm, row_of, dl, W_r, dx, dW_r, accumulate, bs, err, stream);
}

moe_status moe_layer_bwd(const moe_config* cfg, const moe_weights* w, const void* x, const void* dy,
                         const moe_saved* saved, void* dx, const moe_grads* grads, int accumulate, void* ws,
                         size_t ws_bytes, moe_stream_t stream) {
  Shape s;
  MOE_TRY(make_shape(cfg, &s));
  if (w == nullptr || saved == nullptr || grads == nullptr) return MOE_ERR_INVALID_ARG;
  if (accumulate != 0 && accumulate != 1) return MOE_ERR_INVALID_ARG;
  MOE_TRY(need(x));
  MOE_TRY(need(dy));
  MOE_TRY(need(dx));
  MOE_TRY(need(w->W_r, 4));
  MOE_TRY(need(w->W1));
  MOE_TRY(need(w->W3));
  MOE_TRY(need(w->W2));
  const bool recompute = recompute_mode(saved);
  MOE_TRY(need(saved->x_perm));
  MOE_TRY(need(saved->y_perm));
  if (!recompute) {
    MOE_TRY(need(saved->a));
    MOE_TRY(need(saved->b));
    MOE_TRY(need(saved->h));
  }
  const void* sp4[] = {saved->ids, saved->gates, saved->row_of, saved->src_token, saved->counts, saved->offsets};
  for (const void* p : sp4) MOE_TRY(need(p, 4));
  if (s.k == 1 || s.aux > 0.f) MOE_TRY(need(saved->probs, 4));
  if (grads->aux_loss != nullptr) MOE_TRY(need(grads->aux_loss, 4));
  MOE_TRY(need(grads->dW_r, 4));
  MOE_TRY(need(grads->dW1));
  MOE_TRY(need(grads->dW3));
  MOE_TRY(need(grads->dW2));
  if (ws == nullptr || ws_bytes < ws_bytes_for(s, recompute ? 2 : 1)) return MOE_ERR_WORKSPACE;
  uint32_t* err = nullptr;
  MOE_TRY(device_ready(&err));
  NvtxScope range("moe_layer_bwd");
  Carver c(align_ws(ws));
  carve_routing(c, s);
  BwdScratch bs = carve_bwd(c, s);
  const void *act_a = saved->a, *act_b = saved->b, *act_h = saved->h;
  if (recompute && s.T > 0) {
    // the up product again from the kept x_perm: a, b and h, bit for bit the
    // forward's (same kernel, same inputs); no down product
    const RecomputeScratch rc = carve_recompute(c, s);
    FfnFwdArgs up{saved->x_perm, saved->counts, saved->offsets, w->W1, w->W3, w->W2, rc.h, nullptr, rc.a, rc.b};
    MOE_TRY(do_ffn_fwd(s, up, err, stream));
    act_a = rc.a;
    act_b = rc.b;
    act_h = rc.h;
  }
  // bf16 layers: the router term of each kept row, dl[t, e] W_r[:, e], is added
  // in the dgrad x epilogue (its expert is the tile's), so the dx gather adds
  // only the terms of the experts a token does not keep a row for.  Large bf16
  // layers also take each kept row's g * dg = <g dY W2^T, h> = <dH, h> from the
  // dgrad h epilogue, so the combine backward only scatters g * dY (Y_perm is not
  // read back) and the logit gradient dl follows the dgrad h product.
  const bool fuse_router = s.bf16 != 0;
  const bool fuse_dg = fuse_router && fused_dg_pays(s);
  if (s.T > 0)
    CUDA_TRY(launch_combine_bwd(s, dy, saved->y_perm, saved->ids, saved->row_of, saved->gates, saved->probs,
                                saved->counts, saved->offsets, bs.dy_perm, fuse_dg ? nullptr : bs.dg,
                                fuse_dg ? nullptr : bs.dl, err, stream));
  FfnBwdArgs fb{saved->x_perm, act_a, act_b, act_h, bs.dy_perm, saved->counts, saved->offsets,
                w->W1, w->W3, w->W2, bs.da, bs.db, bs.dx_perm, grads->dW1, grads->dW3, grads->dW2, accumulate};
  fb.round_ctr = bs.round_ctr;
  if (fuse_router) {
    fb.rdl = bs.dl;
    fb.rwr = w->W_r;
    fb.src_token = saved->src_token;
  }
  if (fuse_dg) {
    fb.sdot = bs.sdot;
    fb.part = 1;  // dgrad h
    MOE_TRY(do_ffn_bwd(s, fb, err, stream));
    CUDA_TRY(launch_dl_from_dots(s, bs.sdot, s.f / 256, saved->row_of, saved->ids, saved->gates, saved->probs,
                                 bs.dl, err, stream));
    fb.sdot = nullptr;
    fb.part = 2;  // wgrad and dgrad x
  }
  CUDA_TRY(launch_aux_loss(s, s.aux, saved->probs, saved->ids, grads->aux_loss, bs.dl, bs.aux, err, stream));
  MOE_TRY(do_ffn_bwd(s, fb, err, stream));
  return do_dx_router(s, x, bs.dx_perm, saved->row_of, bs.dl, w->W_r, dx, grads->dW_r, accumulate, bs, err, stream,
                      fuse_router ? saved->ids : nullptr);
}

moe_status moe_get_device_error(int32_t* code, int32_t* detail, int clear) {
  uint32_t* err = nullptr;
  MOE_TRY(device_ready(&err));
  CUDA_TRY(cudaDeviceSynchronize());
  uint32_t h[2] = {0, 0};
  CUDA_TRY(cudaMemcpyFromSymbol(h, g_device_error, sizeof(h)));
  if (clear) {
    const uint32_t z[2] = {0, 0};
    CUDA_TRY(cudaMemcpyToSymbol(g_device_error, z, sizeof(z)));
  }
  int32_t c = MOE_OK;
  if (h[0] == DEV_TIMEOUT) c = MOE_ERR_TIMEOUT;
  else if (h[0] != 0) c = MOE_ERR_DEVICE_CHECK;
  if (code) *code = c;
  if (detail) *detail = (int32_t)(h[0] == 0 ? 0 : (h[0] << 24) | (h[1] & 0xFFFFFFu));
  return MOE_OK;
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

moe_status moe_profiler_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (on) {
    for (auto& r : g_prof_recs) {
      g_event_pool.push_back(r.a);
      g_event_pool.push_back(r.b);
    }
    g_prof_recs.clear();
  }
  g_prof_on = on != 0;
  return MOE_OK;
}

moe_status moe_nvtx_enable(int on) {
  g_nvtx.store(on != 0, std::memory_order_relaxed);
  return MOE_OK;
}

int32_t moe_kernel_kinds(void) { return KK_COUNT; }

moe_status moe_profiler_filter(int32_t id) {
  if (id >= KK_COUNT) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_filter = id < 0 ? -1 : id;
  return MOE_OK;
}

const char* moe_kernel_name(int32_t id) {
  if (id < 0 || id >= KK_COUNT) return nullptr;
  return kKernelNames[id];
}

moe_status moe_profiler_read(int32_t id, int64_t* launches, double* total_ms) {
  if (id < 0 || id >= KK_COUNT) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  int64_t n = 0;
  double ms = 0.0;
  for (auto& r : g_prof_recs) {
    if (r.kind != id) continue;
    if (cudaEventSynchronize(r.b) != cudaSuccess) return MOE_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return MOE_ERR_CUDA;
    ++n;
    ms += t;
  }
  if (launches) *launches = n;
  if (total_ms) *total_ms = ms;
  return MOE_OK;
}

}  // extern "C"
