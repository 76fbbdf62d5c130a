// Router scoring, top-k and capacity slotting.
//
// Three kernels, all deterministic:
//   1. router_topk: each block takes 64 tokens, computes their logits
//      l = x W_r + b in fp32 (W_r staged through shared memory in 32-row
//      chunks), then one warp per token takes the fp32 softmax and the top-k
//      (value descending, lower expert index on ties), writes ids/gates/probs
//      and a per-(expert, choice) histogram of the block;
//   2. slot_scan: one block per expert turns that expert's histogram row,
//      ordered (choice, token block), into exclusive prefix sums; the last
//      block to finish derives counts[e] = min(total, C) and the 128-aligned
//      offsets;
//   3. slot_assign: one block per token block and choice ranks tokens of the
//      same expert inside the block with __match_any_sync, adds the prefix
//      from (2), and writes slot, row_of and src_token.
//
// Slot order is choice-major then token order: the first choices of all
// tokens are served before any second choice (the top-2 layer configuration);
// the capacity cut-off is the capacity-factor passage of the Expert
// Parallelism section of the distributed-training tutorial.
#include <float.h>
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int RT_TOK = 64;
constexpr int RT_DC = 32;
constexpr int RT_THREADS = 256;
constexpr int MAX_K = 8;

struct RouterArgs {
  const void* x;
  const float* W_r;
  const float* bias;
  int32_t* ids;
  float* gates;
  float* probs;
  int32_t* hist;
  int32_t* ticket;
  int T, d, E, k, nb;
};

template <int EP, typename Tx>
__global__ void __launch_bounds__(RT_THREADS) router_topk_kernel(RouterArgs a) {
  pdl_enter();  // see pdl_wait: no global access before this
  constexpr int NT_E = EP < 32 ? EP : 32;   // threads along experts
  constexpr int TN = EP / NT_E;             // experts per thread
  constexpr int NT_T = RT_THREADS / NT_E;   // threads along tokens
  constexpr int TM = RT_TOK / NT_T;         // tokens per thread
  constexpr int EPL = (EP + 31) / 32;       // logits per lane in the top-k stage
  constexpr int GEMM_FLOATS = RT_DC * (RT_TOK + 1) + RT_DC * EP;
  constexpr int LG_FLOATS = RT_TOK * (EP + 1);
  constexpr int POOL = GEMM_FLOATS > LG_FLOATS ? GEMM_FLOATS : LG_FLOATS;
  __shared__ float pool[POOL];
  __shared__ int hist_s[MAX_K][EP];
  float (*xs)[RT_TOK + 1] = reinterpret_cast<float (*)[RT_TOK + 1]>(pool);
  float (*wsm)[EP] = reinterpret_cast<float (*)[EP]>(pool + RT_DC * (RT_TOK + 1));
  float (*lg)[EP + 1] = reinterpret_cast<float (*)[EP + 1]>(pool);

  const Tx* x = static_cast<const Tx*>(a.x);
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * RT_TOK;
  if (blockIdx.x == 0 && tid == 0) *a.ticket = 0;  // for the last-block election of slot_scan
  for (int i = tid; i < MAX_K * EP; i += RT_THREADS) (&hist_s[0][0])[i] = 0;

  const int te = tid % NT_E, tt = tid / NT_E;
  float acc[TM][TN];
#pragma unroll
  for (int m = 0; m < TM; ++m)
#pragma unroll
    for (int n = 0; n < TN; ++n) acc[m][n] = 0.f;

  for (int i0 = 0; i0 < a.d; i0 += RT_DC) {
    for (int idx = tid; idx < RT_TOK * RT_DC; idx += RT_THREADS) {
      const int r = idx / RT_DC, c = idx % RT_DC;
      const int t = t0 + r, i = i0 + c;
      xs[c][r] = (t < a.T && i < a.d) ? to_f32(x[(size_t)t * a.d + i]) : 0.f;
    }
    for (int idx = tid; idx < RT_DC * EP; idx += RT_THREADS) {
      const int r = idx / EP, c = idx % EP;
      const int i = i0 + r;
      wsm[r][c] = (i < a.d && c < a.E) ? a.W_r[(size_t)i * a.E + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int i = 0; i < RT_DC; ++i) {
      float xv[TM], wv[TN];
#pragma unroll
      for (int m = 0; m < TM; ++m) xv[m] = xs[i][tt * TM + m];
#pragma unroll
      for (int n = 0; n < TN; ++n) wv[n] = wsm[i][te + n * NT_E];
#pragma unroll
      for (int m = 0; m < TM; ++m)
#pragma unroll
        for (int n = 0; n < TN; ++n) acc[m][n] = fmaf(xv[m], wv[n], acc[m][n]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int m = 0; m < TM; ++m)
#pragma unroll
    for (int n = 0; n < TN; ++n) {
      const int e = te + n * NT_E;
      const float b = (a.bias != nullptr && e < a.E) ? a.bias[e] : 0.f;
      lg[tt * TM + m][e] = acc[m][n] + b;
    }
  __syncthreads();

  const int warp = tid / 32, lane = tid % 32;
  for (int q = warp; q < RT_TOK; q += RT_THREADS / 32) {
    const int t = t0 + q;
    if (t >= a.T) break;
    float v[EPL];
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < EPL; ++c) {
      const int e = lane + 32 * c;
      float val = (e < a.E) ? lg[q][e] : -INFINITY;
      if (isnan(val)) val = -INFINITY;
      v[c] = val;
      mx = fmaxf(mx, val);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float se = 0.f;
#pragma unroll
    for (int c = 0; c < EPL; ++c)
      if (lane + 32 * c < a.E) se += expf(v[c] - mx);
    se = warp_sum(se);

    uint32_t taken = 0;
    float lj[MAX_K];
    int ej[MAX_K];
#pragma unroll
    for (int j = 0; j < MAX_K; ++j) {
      lj[j] = 0.f;
      ej[j] = 0;
      if (j < a.k) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int c = 0; c < EPL; ++c) {
          const int e = lane + 32 * c;
          if (e < a.E && !((taken >> c) & 1u) && (v[c] > bv || (v[c] == bv && e < be))) {
            bv = v[c];
            be = e;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oe = __shfl_xor_sync(0xffffffffu, be, o);
          if (ov > bv || (ov == bv && oe < be)) {
            bv = ov;
            be = oe;
          }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        lj[j] = bv;
        ej[j] = be;
      }
    }
    if (lane == 0) {
      float g[MAX_K];
      if (a.k == 1) {
        g[0] = expf(lj[0] - mx) / se;
      } else {
        float den = 0.f;
#pragma unroll
        for (int j = 0; j < MAX_K; ++j)
          if (j < a.k) {
            g[j] = expf(lj[j] - lj[0]);
            den += g[j];
          }
#pragma unroll
        for (int j = 0; j < MAX_K; ++j)
          if (j < a.k) g[j] = g[j] / den;
      }
#pragma unroll
      for (int j = 0; j < MAX_K; ++j)
        if (j < a.k) {
          a.ids[(size_t)t * a.k + j] = ej[j];
          a.gates[(size_t)t * a.k + j] = g[j];
          atomicAdd(&hist_s[j][ej[j]], 1);
        }
    }
    if (a.probs != nullptr) {
#pragma unroll
      for (int c = 0; c < EPL; ++c) {
        const int e = lane + 32 * c;
        if (e < a.E) a.probs[(size_t)t * a.E + e] = expf(v[c] - mx) / se;
      }
    }
  }
  __syncthreads();
  for (int idx = tid; idx < a.k * EP; idx += RT_THREADS) {
    const int j = idx / EP, e = idx % EP;
    if (e < a.E) a.hist[((size_t)e * a.k + j) * a.nb + blockIdx.x] = hist_s[j][e];
  }
}

struct ScanArgs {
  const int32_t* hist;
  int32_t* base;
  int32_t* totals;
  int32_t* ticket;
  int32_t* counts;
  int32_t* offsets;
  uint32_t* err;
  int E, L, cap;
  int64_t max_rows;
};

__global__ void __launch_bounds__(256) slot_scan_kernel(ScanArgs a) {
  pdl_enter();  // see pdl_wait: no global access before this
  __shared__ int warp_sums[8];
  __shared__ int is_last;
  const int e = blockIdx.x, tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int32_t* h = a.hist + (size_t)e * a.L;
  int32_t* bse = a.base + (size_t)e * a.L;
  const int per = (a.L + 255) / 256;
  const int beg = min(a.L, tid * per), end = min(a.L, beg + per);
  int s = 0;
  for (int i = beg; i < end; ++i) s += h[i];
  // block-wide exclusive scan of the per-thread sums
  int incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  int wpre = 0, total = 0;
  for (int w = 0; w < 8; ++w) {
    if (w < warp) wpre += warp_sums[w];
    total += warp_sums[w];
  }
  int run = wpre + incl - s;
  for (int i = beg; i < end; ++i) {
    bse[i] = run;
    run += h[i];
  }
  if (tid == 0) a.totals[e] = total;
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = (atomicAdd(a.ticket, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (is_last) {
    // counts[e] = min(total, C) and the 128-aligned offsets: one expert per
    // thread (E <= 128), an exclusive scan of the padded counts over the block
    __shared__ int64_t pad_sums[8];
    __threadfence();
    int c = 0;
    int64_t padded = 0;
    if (tid < a.E) {
      const int tot = __ldcg(a.totals + tid);
      c = tot < a.cap ? tot : a.cap;
      padded = ((int64_t)c + 127) / 128 * 128;
    }
    int64_t pincl = padded;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t n = __shfl_up_sync(0xffffffffu, pincl, o);
      if (lane >= o) pincl += n;
    }
    if (lane == 31) pad_sums[warp] = pincl;
    __syncthreads();
    int64_t off = pincl - padded;
    for (int w = 0; w < warp; ++w) off += pad_sums[w];
    if (tid < a.E) {
      a.counts[tid] = c;
      a.offsets[tid] = (int32_t)off;
    }
    if (tid == a.E - 1) {
      const int64_t end = off + padded;
      if (end > a.max_rows) report_error(a.err, DEV_BAD_OFFSETS, 1);
      a.offsets[a.E] = (int32_t)(end > a.max_rows ? a.max_rows : end);
    }
  }
}

struct AssignArgs {
  const int32_t* ids;
  const int32_t* base;
  const int32_t* counts;
  const int32_t* offsets;
  int32_t* slot;
  int32_t* row_of;
  int32_t* src_token;
  uint32_t* err;
  int T, E, k, nb, cap;
  int64_t max_rows;
};

__global__ void __launch_bounds__(RT_TOK) slot_assign_kernel(AssignArgs a) {
  pdl_enter();  // see pdl_wait: no global access before this
  __shared__ int cnt0[128];
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int b = blockIdx.x;
  if (b >= a.nb) {
    // pad rows of one expert: src_token = -1
    const int e = b - a.nb;
    const int64_t beg = (int64_t)a.offsets[e] + a.counts[e], end = a.offsets[e + 1];
    if (end > a.max_rows || beg > end) {
      if (tid == 0) report_error(a.err, DEV_BAD_OFFSETS, 2);
      return;
    }
    for (int64_t r = beg + tid; r < end; r += RT_TOK) a.src_token[r] = -1;
    return;
  }
  const int t = b * RT_TOK + tid;
  const bool valid = t < a.T;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int j = 0; j < a.k; ++j) {
    for (int i = tid; i < 128; i += RT_TOK) cnt0[i] = 0;
    __syncthreads();
    int e = valid ? a.ids[(size_t)t * a.k + j] : -1;
    if (valid && (e < 0 || e >= a.E)) {
      report_error(a.err, DEV_BAD_EXPERT, (uint32_t)t);
      e = -1;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    int rank = __popc(peers & lt_mask);
    if (warp == 0 && e >= 0 && (31 - __clz(peers)) == lane) cnt0[e] = __popc(peers);
    __syncthreads();
    if (warp == 1 && e >= 0) rank += cnt0[e];
    if (e >= 0) {
      const int s = a.base[((size_t)e * a.k + j) * a.nb + b] + rank;
      int sl = -1, row = -1;
      if (s < a.cap) {
        const int64_t r = (int64_t)a.offsets[e] + s;
        if (s >= a.counts[e] || r >= a.offsets[e + 1] || r >= a.max_rows) {
          report_error(a.err, DEV_BAD_ROW, (uint32_t)t);
        } else {
          sl = s;
          row = (int)r;
          a.src_token[r] = t;
        }
      }
      a.slot[(size_t)t * a.k + j] = sl;
      a.row_of[(size_t)t * a.k + j] = row;
    }
    __syncthreads();
  }
}

template <int EP>
cudaError_t launch_router_ep(const Shape& s, const RouterArgs& ra, cudaStream_t st) {
  LaunchScope ls(KK_ROUTER, st);
  if (s.bf16) return launch_pdl(router_topk_kernel<EP, __nv_bfloat16>, dim3(ra.nb), dim3(RT_THREADS), 0, st, ra);
  return launch_pdl(router_topk_kernel<EP, float>, dim3(ra.nb), dim3(RT_THREADS), 0, st, ra);
}

}  // namespace

int router_blocks(int T) { return (T + RT_TOK - 1) / RT_TOK; }

cudaError_t launch_router(const Shape& s, const void* x, const float* W_r, const float* bias, int32_t* ids,
                          float* gates, float* probs, int32_t* hist, int32_t* ticket, cudaStream_t st) {
  RouterArgs ra{x, W_r, bias, ids, gates, probs, hist, ticket, s.T, s.d, s.E, s.k, router_blocks(s.T)};
  if (ra.nb == 0) return cudaSuccess;
  if (s.E <= 8) return launch_router_ep<8>(s, ra, st);
  if (s.E <= 16) return launch_router_ep<16>(s, ra, st);
  if (s.E <= 32) return launch_router_ep<32>(s, ra, st);
  if (s.E <= 64) return launch_router_ep<64>(s, ra, st);
  return launch_router_ep<128>(s, ra, st);
}

cudaError_t launch_slot_scan(const Shape& s, const int32_t* hist, int32_t* base, int32_t* totals,
                             int32_t* ticket, int32_t* counts, int32_t* offsets, uint32_t* err, cudaStream_t st) {
  ScanArgs a{hist, base, totals, ticket, counts, offsets, err, s.E, s.k * router_blocks(s.T), s.cap, s.max_rows};
  LaunchScope ls(KK_SLOT_SCAN, st);
  return launch_pdl(slot_scan_kernel, dim3(s.E), dim3(256), 0, st, a);
}

cudaError_t launch_slot_assign(const Shape& s, const int32_t* ids, const int32_t* base, const int32_t* counts,
                               const int32_t* offsets, int32_t* slot, int32_t* row_of, int32_t* src_token,
                               uint32_t* err, cudaStream_t st) {
  AssignArgs a{ids, base, counts, offsets, slot, row_of, src_token, err, s.T, s.E, s.k,
               router_blocks(s.T), s.cap, s.max_rows};
  LaunchScope ls(KK_SLOT_ASSIGN, st);
  return launch_pdl(slot_assign_kernel, dim3(a.nb + s.E), dim3(RT_TOK), 0, st, a);
}

}  // namespace moe
