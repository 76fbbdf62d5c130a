// Internal declarations shared by the library's translation units: kernel
// kinds for launch accounting, the device error word codes, and the launchers
// that the C ABI layer (moe_api.cu) sequences.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

enum KernelKind : int {
  KK_ROUTER = 0,
  KK_SLOT_SCAN,
  KK_SLOT_ASSIGN,
  KK_PERMUTE,
  KK_GEMM_UP,
  KK_GEMM_DOWN,
  KK_COMBINE,
  KK_COMBINE_BWD,
  KK_GEMM_DGRAD_H,
  KK_GEMM_WGRAD,
  KK_GEMM_DGRAD_X,
  KK_TRANSPOSE_WR,
  KK_DX_ROUTER,
  KK_DWR,
  KK_DWR_REDUCE,
  KK_ZERO,
  KK_SPLIT_WR,
  KK_SELFTEST,
  KK_SPLIT_DL,
  KK_AUX_LOSS,
  KK_AUX_GRAD,
  KK_LOGIT_GRAD,
  KK_COUNT
};

// Device error word: err[0] = first code (0 = none), err[1] = detail of that code.
enum DevErr : uint32_t {
  DEV_OK = 0,
  DEV_BAD_ROW = 1,      // a row index outside [0, max_rows)
  DEV_BAD_EXPERT = 2,   // an expert id outside [0, E)
  DEV_BAD_OFFSETS = 3,  // offsets not monotone / not 128-aligned / beyond max_rows
  DEV_TIMEOUT = 4,      // a pipeline wait ran out of time
  DEV_BAD_COUNT = 5     // counts[e] larger than its segment
};

// Launch accounting (defined in moe_api.cu): every kernel launch is bracketed
// by launch_begin/launch_end so the library can count launches and, when the
// profiler is on, record CUDA events around it on the launch stream.
void launch_begin(int kind, cudaStream_t s);
void launch_end(int kind, cudaStream_t s);

struct LaunchScope {
  int kind;
  cudaStream_t s;
  LaunchScope(int k, cudaStream_t st) : kind(k), s(st) { launch_begin(kind, s); }
  ~LaunchScope() { launch_end(kind, s); }
};

struct Shape {
  int T, d, f, E, k;
  int cap;           // INT32_MAX when dropless
  int bf16;          // 1 = bf16 activations/weights, 0 = fp32
  int64_t max_rows;  // bound on offsets[E]
  float aux;         // auxiliary load-balancing loss coefficient (0: off)
};

// ---- routing.cu ----
// Router GEMV/top-k, then the per-expert scan, then slot assignment.
cudaError_t launch_router(const Shape& s, const void* x, const float* W_r, const float* bias, int32_t* ids,
                          float* gates, float* probs, int32_t* hist, int32_t* ticket, cudaStream_t st);
cudaError_t launch_slot_scan(const Shape& s, const int32_t* hist, int32_t* base, int32_t* totals,
                             int32_t* ticket, int32_t* counts, int32_t* offsets, uint32_t* err, cudaStream_t st);
cudaError_t launch_slot_assign(const Shape& s, const int32_t* ids, const int32_t* base, const int32_t* counts,
                               const int32_t* offsets, int32_t* slot, int32_t* row_of, int32_t* src_token,
                               uint32_t* err, cudaStream_t st);
int router_blocks(int T);  // tokens per router block is fixed; this is the block count

// ---- router_tc.cu: tensor-core router for bf16 layers with T >= 128 ----
bool router_tc_supported(const Shape& s);
size_t router_wsplit_bytes(const Shape& s);  // scratch for the three bf16 parts of W_r
cudaError_t launch_router_tc(const Shape& s, const void* x, const float* W_r, const float* bias, void* wsplit,
                             int32_t* ids, float* gates, float* probs, int32_t* hist, int32_t* ticket,
                             uint32_t* err, cudaStream_t st);

// ---- rows.cu ----
// With y_zero and row_gate given it also zeroes y_zero[t] and writes
// row_gate[row_of[t,j]] = gates[t,j] (the combine fused into the down product).
cudaError_t launch_permute(const Shape& s, const void* x, const int32_t* row_of, const int32_t* counts,
                           const int32_t* offsets, void* x_perm, uint32_t* err, cudaStream_t st,
                           const float* gates = nullptr, float* row_gate = nullptr, void* y_zero = nullptr);
cudaError_t launch_combine(const Shape& s, const void* y_perm, const int32_t* row_of, const float* gates, void* y,
                           uint32_t* err, cudaStream_t st);
cudaError_t launch_combine_bwd(const Shape& s, const void* dy, const void* y_perm, const int32_t* ids,
                               const int32_t* row_of, const float* gates, const float* probs,
                               const int32_t* counts, const int32_t* offsets, void* dy_perm, float* dg, float* dl,
                               uint32_t* err, cudaStream_t st);
// dg and dl may be null: then only dy_perm = g * dy is written (y_perm unread)
// dl [T, E] from the dgrad h product's per-row, per-256-column-tile sums of
// dH * h (sdot [max_rows, nt]); overwrites dl
cudaError_t launch_dl_from_dots(const Shape& s, const float* sdot, int nt, const int32_t* row_of,
                                const int32_t* ids, const float* gates, const float* probs, float* dl, uint32_t* err,
                                cudaStream_t st);
// With ids given (skip_kept), the router terms of the token's kept experts are
// taken to be in dx_perm already and only the other experts' terms are added.
cudaError_t launch_dx_router(const Shape& s, const void* dx_perm, const int32_t* row_of, const float* dl,
                             const float* W_r, float* W_rT, void* dx, uint32_t* err, cudaStream_t st,
                             const int32_t* ids = nullptr);
cudaError_t launch_dwr(const Shape& s, const void* x, const float* dl, float* partial, float* dW_r, int accumulate,
                       cudaStream_t st);
int dwr_splits(const Shape& s);  // token slices of the router-weight gradient (partial buffer [splits][d][E])
// Adds the token-slice partials [splits][d][E] in slice order into dW_r (n = d * E).
cudaError_t launch_dwr_reduce(const float* partial, float* dW_r, int splits, int64_t n, int accumulate,
                              cudaStream_t st);

// ---- aux_loss.cu: auxiliary load-balancing loss (adds its logit gradient into dl) ----
size_t aux_scratch_bytes(const Shape& s);
cudaError_t launch_aux_loss(const Shape& s, float coeff, const float* probs, const int32_t* ids, float* loss,
                            float* dl, void* scratch, uint32_t* err, cudaStream_t st);

// ---- dwr_tc.cu: the router-weight gradient on the tensor cores (bf16 layers) ----
bool dwr_tc_supported(const Shape& s);
int dwr_tc_ranges(const Shape& s);           // token ranges (partial buffer [ranges][d][E])
size_t dwr_tc_split_bytes(const Shape& s);   // the bf16 parts of dl
// partial[r] = x^T dl over token range r; dW_r is then formed by launch_dwr_reduce.
cudaError_t launch_dwr_tc(const Shape& s, const void* x, const float* dl, void* dlsplit, float* partial,
                          uint32_t* err, cudaStream_t st);
cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t st);

// ---- gemm_tc.cu (bf16, tcgen05) and gemm_simt.cu (fp32) ----
struct FfnFwdArgs {
  const void* x_perm; const int32_t* counts; const int32_t* offsets;
  const void* W1; const void* W3; const void* W2;
  void* h; void* y_perm; void* a; void* b;  // y_perm null: the up product only
  // bf16 only: with y_comb set the down product adds row_gate[row] * its row into
  // y_comb[src_token[row]] (zeroed beforehand) instead of writing y_perm
  const int32_t* src_token = nullptr; const float* row_gate = nullptr; void* y_comb = nullptr;
};
struct FfnBwdArgs {
  const void* x_perm; const void* a; const void* b; const void* h; const void* dy_perm;
  const int32_t* counts; const int32_t* offsets;
  const void* W1; const void* W3; const void* W2;
  void* da; void* db; void* dx_perm;
  float* dW1; float* dW3; float* dW2; int accumulate;
  // bf16 only, optional: with rdl (dl [T, E]), rwr (W_r [d, E]) and src_token
  // set, dx_perm[row] also holds the row's router term dl[token, e] * W_r[:, e]
  const float* rdl = nullptr; const float* rwr = nullptr; const int32_t* src_token = nullptr;
  // bf16 only, optional: per row and 256-column tile of dH, the sum of dH * h
  // ([max_rows, f / 256] fp32), written by the dgrad h product
  float* sdot = nullptr;
  // bf16 only: 0 runs dgrad h, wgrad and dgrad x; 1 dgrad h alone; 2 wgrad and dgrad x
  int part = 0;
  // bf16 only, optional: WG_ROUNDS ints of scratch (zeroed by the call) with which
  // wgrad keeps its rounds of host and guest tiles in step
  int* round_ctr = nullptr;
};
constexpr int WG_ROUNDS = 4096;  // rounds of host and guest tiles kept in step (later ones run free)
cudaError_t tc_ffn_fwd(const Shape& s, const FfnFwdArgs& a, uint32_t* err, cudaStream_t st);
cudaError_t tc_ffn_bwd(const Shape& s, const FfnBwdArgs& a, uint32_t* err, cudaStream_t st);
cudaError_t simt_ffn_fwd(const Shape& s, const FfnFwdArgs& a, uint32_t* err, cudaStream_t st);
cudaError_t simt_ffn_bwd(const Shape& s, const FfnBwdArgs& a, uint32_t* err, cudaStream_t st);
bool tc_driver_ready();  // tensor-map encoder resolved from the driver

// ---- moe_api.cu: shared with the allocation-free router entry point ----
// Validates a moe_config and derives its Shape; returns a moe_status value.
int validate_config(const void* cfg, Shape* s);
// Device error word of the current device (checks the device is sm_103);
// returns a moe_status value.
int current_error_word(uint32_t** err);

}  // namespace moe
