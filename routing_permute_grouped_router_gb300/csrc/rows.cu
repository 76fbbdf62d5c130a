// Row-moving kernels of the layer step: the permute into per-expert buffers,
// the gate-weighted unpermute + combine, their backward (token-gradient
// routing), the dx gather with the router's input gradient, and the router
// weight gradient.
//
// All of them are HBM-bound row copies.  One warp owns one token row and moves
// it in 16-byte vectors (8 bf16 or 4 fp32 per lane), so every warp access is a
// contiguous 512-byte segment.  The kernels are templated on k so that each
// lane issues all of a chunk's loads (8 vectors over the k rows) before it
// uses any of them: one memory round trip per chunk instead of one per vector.
// Sums run in fp32 in a fixed order (choice j ascending), so results are
// deterministic and use no atomics.
#include <float.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int RW_WARPS = 8;  // warps (= token rows) per block
constexpr int INFLIGHT = 8;  // 16-byte loads each lane keeps in flight

__device__ __forceinline__ bool row_ok(int64_t r, int64_t max_rows) { return r >= 0 && r < max_rows; }

// Row indices of token t's k assignments; out-of-range rows are reported and
// treated as dropped.
template <int K>
__device__ __forceinline__ void load_rows(const int32_t* __restrict__ row_of, int t, int64_t max_rows, uint32_t* err,
                                          int lane, uint32_t detail, int64_t (&rows)[K]) {
#pragma unroll
  for (int j = 0; j < K; ++j) {
    const int64_t r = row_of[(size_t)t * K + j];
    rows[j] = -1;
    if (r >= 0 && !row_ok(r, max_rows)) {
      if (lane == 0) report_error(err, DEV_BAD_ROW, detail);
    } else {
      rows[j] = r;
    }
  }
}

__device__ __forceinline__ void zero_pad_rows(const int32_t* counts, const int32_t* offsets, int e, char* buf,
                                              int nvec, int64_t max_rows, uint32_t* err, int warp, int lane,
                                              uint32_t detail) {
  const int64_t beg = (int64_t)offsets[e] + counts[e], end = offsets[e + 1];
  if (end > max_rows || beg > end) {
    if (warp == 0 && lane == 0) report_error(err, DEV_BAD_OFFSETS, detail);
    return;
  }
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int64_t r = beg + warp; r < end; r += RW_WARPS)
    for (int v = lane; v < nvec; v += 32) stg16(buf + (r * nvec + v) * 16, z);
}

// -------------------------------------------------------------------------- //
// Permute (scatter form: each token row is read once and written to each of
// its kept rows); blocks past the token range zero the pad rows of one expert.
// When the combine is fused into the down product it also zeroes the token's
// row of y and records the gate of each kept row.
// -------------------------------------------------------------------------- //
struct PermArgs {
  const char* x;
  const int32_t* row_of;
  const int32_t* counts;
  const int32_t* offsets;
  char* x_perm;
  const float* gates;  // with row_gate and y_zero: the fused combine's inputs
  float* row_gate;
  char* y_zero;
  uint32_t* err;
  int T, E, nvec;  // nvec = 16-byte vectors per row
  int64_t max_rows;
  int token_blocks;
};

template <int K>
__global__ void __launch_bounds__(RW_WARPS * 32) permute_kernel(PermArgs a) {
  pdl_enter();  // see pdl_wait: no global access before this
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if ((int)blockIdx.x >= a.token_blocks) {
    zero_pad_rows(a.counts, a.offsets, blockIdx.x - a.token_blocks, a.x_perm, a.nvec, a.max_rows, a.err, warp,
                  lane, 10);
    return;
  }
  const int t = blockIdx.x * RW_WARPS + warp;
  if (t >= a.T) return;
  int64_t rows[K];
  load_rows<K>(a.row_of, t, a.max_rows, a.err, lane, 10, rows);
  if (a.row_gate != nullptr) {
    if (lane < K) {
#pragma unroll
      for (int j = 0; j < K; ++j)
        if (lane == j && rows[j] >= 0) a.row_gate[rows[j]] = a.gates[(size_t)t * K + j];
    }
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (int v = lane; v < a.nvec; v += 32) stg16(a.y_zero + ((int64_t)t * a.nvec + v) * 16, z);
  }
  const char* __restrict__ src = a.x + (int64_t)t * a.nvec * 16;
  char* __restrict__ dst = a.x_perm;
  for (int v0 = 0; v0 < a.nvec; v0 += 32 * INFLIGHT) {
    uint4 val[INFLIGHT];
#pragma unroll
    for (int u = 0; u < INFLIGHT; ++u) {
      const int v = v0 + lane + 32 * u;
      if (v < a.nvec) val[u] = ldg16(src + v * 16);
    }
#pragma unroll
    for (int j = 0; j < K; ++j) {
      if (rows[j] < 0) continue;
#pragma unroll
      for (int u = 0; u < INFLIGHT; ++u) {
        const int v = v0 + lane + 32 * u;
        if (v < a.nvec) stg16(dst + (rows[j] * a.nvec + v) * 16, val[u]);
      }
    }
  }
}

// -------------------------------------------------------------------------- //
// Unpermute + combine: y[t] = sum_j g[t,j] * Y[row_of[t,j]] (fp32, j order).
// -------------------------------------------------------------------------- //
struct CombArgs {
  const char* y_perm;
  const int32_t* row_of;
  const float* gates;
  char* y;
  uint32_t* err;
  int T, nvec;
  int64_t max_rows;
};

template <typename Tx, int K>
__global__ void __launch_bounds__(RW_WARPS * 32) combine_kernel(CombArgs a) {
  pdl_enter();  // see pdl_wait: no global access before this
  constexpr int VN = Vec<Tx>::N;
  constexpr int U = INFLIGHT / K > 0 ? INFLIGHT / K : 1;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t = blockIdx.x * RW_WARPS + warp;
  if (t >= a.T) return;
  int64_t rows[K];
  load_rows<K>(a.row_of, t, a.max_rows, a.err, lane, 11, rows);
  float g[K];
#pragma unroll
  for (int j = 0; j < K; ++j) g[j] = rows[j] >= 0 ? a.gates[(size_t)t * K + j] : 0.f;
  const char* __restrict__ yp = a.y_perm;
  char* __restrict__ dst = a.y + (int64_t)t * a.nvec * 16;
  for (int v0 = 0; v0 < a.nvec; v0 += 32 * U) {
    uint4 buf[K][U];
#pragma unroll
    for (int j = 0; j < K; ++j)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + lane + 32 * u;
        buf[j][u] = (rows[j] >= 0 && v < a.nvec) ? ldg16(yp + (rows[j] * a.nvec + v) * 16) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + lane + 32 * u;
      if (v >= a.nvec) continue;
      float acc[VN];
#pragma unroll
      for (int i = 0; i < VN; ++i) acc[i] = 0.f;
#pragma unroll
      for (int j = 0; j < K; ++j) {
        if (rows[j] < 0) continue;
        float val[VN];
        unpack(buf[j][u], val);
#pragma unroll
        for (int i = 0; i < VN; ++i) acc[i] = fmaf(g[j], val[i], acc[i]);
      }
      stg16(dst + v * 16, pack(acc));
    }
  }
}

// -------------------------------------------------------------------------- //
// Combine backward: dy_perm[row] = g * dy[t]; dg[t,j] = <dy[t], Y[row]>;
// then the logit gradient dl[t, :] of the gates.
// -------------------------------------------------------------------------- //
struct CombBwdArgs {
  const char* dy;
  const char* y_perm;
  const int32_t* ids;
  const int32_t* row_of;
  const float* gates;
  const float* probs;
  const int32_t* counts;
  const int32_t* offsets;
  char* dy_perm;
  float* dg;
  float* dl;
  uint32_t* err;
  int T, E, nvec;
  int64_t max_rows;
  int token_blocks;
};

// DG: also dg = <dY[t], Y_perm[row]> and dl from it; without DG only the
// scatter dY_perm = g * dY (the layer backward of bf16 layers takes dg * g
// from the dgrad h product instead, see dl_from_dots_kernel)
template <typename Tx, int K, bool DG>
__global__ void __launch_bounds__(RW_WARPS * 32) combine_bwd_kernel(CombBwdArgs a) {
  pdl_enter();  // see pdl_wait: no global access before this
  constexpr int VN = Vec<Tx>::N;
  constexpr int U = !DG ? INFLIGHT : (INFLIGHT / (K + 1) > 0 ? INFLIGHT / (K + 1) : 1);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if ((int)blockIdx.x >= a.token_blocks) {
    zero_pad_rows(a.counts, a.offsets, blockIdx.x - a.token_blocks, a.dy_perm, a.nvec, a.max_rows, a.err, warp,
                  lane, 12);
    return;
  }
  const int t = blockIdx.x * RW_WARPS + warp;
  if (t >= a.T) return;
  int64_t rows[K];
  load_rows<K>(a.row_of, t, a.max_rows, a.err, lane, 12, rows);
  float g[K], part[K];
#pragma unroll
  for (int j = 0; j < K; ++j) {
    g[j] = a.gates[(size_t)t * K + j];
    part[j] = 0.f;
  }
  const char* __restrict__ src = a.dy + (int64_t)t * a.nvec * 16;
  const char* __restrict__ yp = a.y_perm;
  char* __restrict__ out = a.dy_perm;
  for (int v0 = 0; v0 < a.nvec; v0 += 32 * U) {
    uint4 dyb[U], yb[K][U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + lane + 32 * u;
      dyb[u] = v < a.nvec ? ldg16(src + v * 16) : make_uint4(0, 0, 0, 0);
    }
    if constexpr (DG) {
#pragma unroll
      for (int j = 0; j < K; ++j)
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + lane + 32 * u;
          yb[j][u] = (rows[j] >= 0 && v < a.nvec) ? ldg16(yp + (rows[j] * a.nvec + v) * 16) : make_uint4(0, 0, 0, 0);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + lane + 32 * u;
      if (v >= a.nvec) continue;
      float dyv[VN];
      unpack(dyb[u], dyv);
#pragma unroll
      for (int j = 0; j < K; ++j) {
        if (rows[j] < 0) continue;
        float o[VN];
        if constexpr (DG) {
          float yv[VN];
          unpack(yb[j][u], yv);
#pragma unroll
          for (int i = 0; i < VN; ++i) part[j] = fmaf(dyv[i], yv[i], part[j]);
        }
#pragma unroll
        for (int i = 0; i < VN; ++i) o[i] = g[j] * dyv[i];
        stg16(out + (rows[j] * a.nvec + v) * 16, pack(o));
      }
    }
  }
  if constexpr (!DG) return;
  float dg[K];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < K; ++j) {
    dg[j] = warp_sum(part[j]);
    s = fmaf(g[j], dg[j], s);
  }
  if (lane < K) {
    float mine = 0.f;
#pragma unroll
    for (int j = 0; j < K; ++j)
      if (lane == j) mine = dg[j];
    a.dg[(size_t)t * K + lane] = mine;
  }
  if (K == 1) {
    const int e1 = a.ids[(size_t)t];
    const float gd = g[0] * dg[0];
    for (int e = lane; e < a.E; e += 32) {
      const float p = a.probs[(size_t)t * a.E + e];
      a.dl[(size_t)t * a.E + e] = gd * ((e == e1 ? 1.f : 0.f) - p);
    }
  } else {
    int ids[K];
#pragma unroll
    for (int j = 0; j < K; ++j) ids[j] = a.ids[(size_t)t * K + j];
    for (int e = lane; e < a.E; e += 32) {
      float v = 0.f;
#pragma unroll
      for (int j = 0; j < K; ++j)
        if (ids[j] == e) v += g[j] * (dg[j] - s);
      a.dl[(size_t)t * a.E + e] = v;
    }
  }
}

// -------------------------------------------------------------------------- //
// W_r^T (E x d) so the router's input gradient reads contiguous rows.
// -------------------------------------------------------------------------- //
__global__ void transpose_wr_kernel(const float* W_r, float* W_rT, int d, int E) {
  pdl_enter();  // see pdl_wait: no global access before this
  __shared__ float tile[32][33];
  const int i0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int i = i0 + r, e = e0 + threadIdx.x;
    tile[r][threadIdx.x] = (i < d && e < E) ? W_r[(size_t)i * E + e] : 0.f;
  }
  __syncthreads();
  for (int r = threadIdx.y; r < 32; r += 8) {
    const int e = e0 + r, i = i0 + threadIdx.x;
    if (e < E && i < d) W_rT[(size_t)e * d + i] = tile[threadIdx.x][r];
  }
}

// -------------------------------------------------------------------------- //
// Router logit gradient from the dgrad h product's row sums.  For a kept row,
// g * dg = g <dY[t], Y_perm[row]> = <g dY[t] W2^T, h[row]> = <dH[row], h[row]>,
// which the dgrad h epilogue has summed per 256-column tile (sdot); with
// s_j = g_j dg_j (0 for a dropped pick) the softmax-over-picks Jacobian gives
// dl[t, e_j] = s_j - g_j sum_i s_i for k > 1 and dl[t, e] = s (onehot - p[e])
// for k = 1 ("The step timeline", gpu_expert_parallel page: the backward walks
// the path in reverse; the router's logits are the gates' parameters).
// -------------------------------------------------------------------------- //
struct DotArgs {
  const float* sdot;  // [max_rows, nt]
  const int32_t* row_of;
  const int32_t* ids;
  const float* gates;
  const float* probs;  // [T, E], k = 1
  float* dl;           // [T, E]
  uint32_t* err;
  int T, E, nt;
  int64_t max_rows;
};

// Eight lanes a token, four tokens a warp (the per-token work is small: k row
// sums of f / 256 values and E outputs).
template <int K>
__global__ void __launch_bounds__(RW_WARPS * 32) dl_from_dots_kernel(DotArgs a) {
  pdl_enter();  // see pdl_wait: no global access before this
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int u = lane & 7;  // lane within the token's group of eight
  const int t = (blockIdx.x * RW_WARPS + warp) * 4 + (lane >> 3);
  const bool live = t < a.T;  // every lane takes part in the shuffles below
  float sj[K], g[K];
  int ids[K];
#pragma unroll
  for (int j = 0; j < K; ++j) {
    sj[j] = 0.f;
    g[j] = 0.f;
    ids[j] = -1;
    if (!live) continue;
    const int64_t r = a.row_of[(size_t)t * K + j];
    g[j] = a.gates[(size_t)t * K + j];
    ids[j] = a.ids[(size_t)t * K + j];
    if (r >= 0 && !row_ok(r, a.max_rows)) {
      if (u == 0) report_error(a.err, DEV_BAD_ROW, 15);
    } else if (r >= 0) {
      for (int n = u; n < a.nt; n += 8) sj[j] += a.sdot[r * a.nt + n];
    }
  }
  // the group's eight partial sums of each pick, by a fixed butterfly (the same
  // bits every run)
#pragma unroll
  for (int o = 4; o > 0; o >>= 1)
#pragma unroll
    for (int j = 0; j < K; ++j) sj[j] += __shfl_xor_sync(0xffffffffu, sj[j], o);
  if (!live) return;
  float S = 0.f;
#pragma unroll
  for (int j = 0; j < K; ++j) S += sj[j];
  if (K == 1) {
    for (int e = u; e < a.E; e += 8) {
      const float p = a.probs[(size_t)t * a.E + e];
      a.dl[(size_t)t * a.E + e] = sj[0] * ((e == ids[0] ? 1.f : 0.f) - p);
    }
  } else {
    for (int e = u; e < a.E; e += 8) {
      float v = 0.f;
#pragma unroll
      for (int j = 0; j < K; ++j)
        if (ids[j] == e) v += sj[j] - g[j] * S;
      a.dl[(size_t)t * a.E + e] = v;
    }
  }
}

// -------------------------------------------------------------------------- //
// dx[t] = sum_j dX_perm[row_of[t,j]] + sum_{e: dl[t,e] != 0} dl[t,e] W_r[:, e]
// -------------------------------------------------------------------------- //
struct DxArgs {
  const char* dx_perm;
  const int32_t* row_of;
  const int32_t* ids;  // non-null: the kept experts' router terms are already in dx_perm
  const float* dl;
  const float* W_rT;
  char* dx;
  uint32_t* err;
  int T, E, d, nvec;
  int64_t max_rows;
};

template <typename Tx, int K>
__global__ void __launch_bounds__(RW_WARPS * 32) dx_router_kernel(DxArgs a) {
  pdl_enter();  // see pdl_wait: no global access before this
  constexpr int VN = Vec<Tx>::N;
  constexpr int U = INFLIGHT / K > 0 ? INFLIGHT / K : 1;
  constexpr int US = U;  // sparse path: the W_r^T vectors load alongside the rows' (no spills up to k = 8)
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t = blockIdx.x * RW_WARPS + warp;
  if (t >= a.T) return;
  int64_t rows[K];
  load_rows<K>(a.row_of, t, a.max_rows, a.err, lane, 13, rows);
  // Experts with a nonzero logit gradient, found with all lanes active before
  // the row loop.
  const float* dlt = a.dl + (size_t)t * a.E;
  int kept[K];  // experts whose router term dx_perm already holds (or -1)
#pragma unroll
  for (int j = 0; j < K; ++j) kept[j] = (a.ids != nullptr && rows[j] >= 0) ? a.ids[(size_t)t * K + j] : -1;
  unsigned nzmask[4];
  float dlv[4];
  int nnz = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int e = 32 * c + lane;
    dlv[c] = (e < a.E) ? dlt[e] : 0.f;
#pragma unroll
    for (int j = 0; j < K; ++j)
      if (e == kept[j]) dlv[c] = 0.f;
    nzmask[c] = __ballot_sync(0xffffffffu, dlv[c] != 0.f);
    nnz += __popc(nzmask[c]);
  }
  const char* __restrict__ xp = a.dx_perm;
  char* __restrict__ dst = a.dx + (int64_t)t * a.nvec * 16;
  if (nnz == 0) {
    // no router term left to add (all in dx_perm already, or dl zero): the k
    // rows' sum alone, with U vectors of every row in flight
    for (int v0 = 0; v0 < a.nvec; v0 += 32 * U) {
      uint4 buf[K][U];
#pragma unroll
      for (int j = 0; j < K; ++j)
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + lane + 32 * u;
          buf[j][u] = (rows[j] >= 0 && v < a.nvec) ? ldg16(xp + (rows[j] * a.nvec + v) * 16) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + lane + 32 * u;
        if (v >= a.nvec) continue;
        float acc[VN];
#pragma unroll
        for (int i = 0; i < VN; ++i) acc[i] = 0.f;
#pragma unroll
        for (int j = 0; j < K; ++j) {
          if (rows[j] < 0) continue;
          float val[VN];
          unpack(buf[j][u], val);
#pragma unroll
          for (int i = 0; i < VN; ++i) acc[i] += val[i];
        }
        stg16(dst + v * 16, pack(acc));
      }
    }
    return;
  }
  if (nnz <= K) {
    // Sparse logit gradient (at most k nonzero experts: k > 1 without an extra
    // term): the experts and their dl values in expert order, so that their
    // W_r^T rows are loaded together with the dx_perm rows.
    int ez[K];
    float wz[K];
    unsigned m0 = nzmask[0], m1 = nzmask[1], m2 = nzmask[2], m3 = nzmask[3];
#pragma unroll
    for (int n = 0; n < K; ++n) {
      unsigned mm = m0;
      int cb = 0;
      float sv = dlv[0];
      if (m0 == 0u) {
        mm = m1; cb = 32; sv = dlv[1];
        if (m1 == 0u) {
          mm = m2; cb = 64; sv = dlv[2];
          if (m2 == 0u) { mm = m3; cb = 96; sv = dlv[3]; }
        }
      }
      const int src = mm ? __ffs(mm) - 1 : 0;
      const float w = __shfl_sync(0xffffffffu, sv, src);
      ez[n] = mm ? cb + src : -1;
      wz[n] = mm ? w : 0.f;
      if (m0) m0 &= m0 - 1;
      else if (m1) m1 &= m1 - 1;
      else if (m2) m2 &= m2 - 1;
      else if (m3) m3 &= m3 - 1;
    }
    for (int v0 = 0; v0 < a.nvec; v0 += 32 * US) {
      uint4 buf[K][US];
      float4 wv[K][US][VN / 4];
#pragma unroll
      for (int j = 0; j < K; ++j)
#pragma unroll
        for (int u = 0; u < US; ++u) {
          const int v = v0 + lane + 32 * u;
          buf[j][u] = (rows[j] >= 0 && v < a.nvec) ? ldg16(xp + (rows[j] * a.nvec + v) * 16) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
      for (int n = 0; n < K; ++n)
#pragma unroll
        for (int u = 0; u < US; ++u) {
          const int v = v0 + lane + 32 * u;
          const float4* wr = reinterpret_cast<const float4*>(a.W_rT + (size_t)(ez[n] >= 0 ? ez[n] : 0) * a.d +
                                                             (size_t)v * VN);
#pragma unroll
          for (int qq = 0; qq < VN / 4; ++qq)
            wv[n][u][qq] = (ez[n] >= 0 && v < a.nvec) ? __ldg(wr + qq) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int u = 0; u < US; ++u) {
        const int v = v0 + lane + 32 * u;
        if (v >= a.nvec) continue;
        float acc[VN];
#pragma unroll
        for (int i = 0; i < VN; ++i) acc[i] = 0.f;
#pragma unroll
        for (int j = 0; j < K; ++j) {
          if (rows[j] < 0) continue;
          float val[VN];
          unpack(buf[j][u], val);
#pragma unroll
          for (int i = 0; i < VN; ++i) acc[i] += val[i];
        }
#pragma unroll
        for (int n = 0; n < K; ++n) {
          const float w = wz[n];  // 0 for missing experts: adds exact zeros, as the loop below skips them
          if (ez[n] < 0) continue;
#pragma unroll
          for (int qq = 0; qq < VN / 4; ++qq) {
            acc[4 * qq + 0] = fmaf(w, wv[n][u][qq].x, acc[4 * qq + 0]);
            acc[4 * qq + 1] = fmaf(w, wv[n][u][qq].y, acc[4 * qq + 1]);
            acc[4 * qq + 2] = fmaf(w, wv[n][u][qq].z, acc[4 * qq + 2]);
            acc[4 * qq + 3] = fmaf(w, wv[n][u][qq].w, acc[4 * qq + 3]);
          }
        }
        stg16(dst + v * 16, pack(acc));
      }
    }
    return;
  }
  // dense logit gradient (k = 1, or an added term): every nonzero expert in turn
  for (int v0 = 0; v0 < a.nvec; v0 += 32 * U) {
    uint4 buf[K][U];
#pragma unroll
    for (int j = 0; j < K; ++j)
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + lane + 32 * u;
        buf[j][u] = (rows[j] >= 0 && v < a.nvec) ? ldg16(xp + (rows[j] * a.nvec + v) * 16) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + lane + 32 * u;
      if (v >= a.nvec) continue;
      float acc[VN];
#pragma unroll
      for (int i = 0; i < VN; ++i) acc[i] = 0.f;
#pragma unroll
      for (int j = 0; j < K; ++j) {
        if (rows[j] < 0) continue;
        float val[VN];
        unpack(buf[j][u], val);
#pragma unroll
        for (int i = 0; i < VN; ++i) acc[i] += val[i];
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        unsigned nz = nzmask[c];
        while (nz) {
          const int e = 32 * c + __ffs(nz) - 1;
          nz &= nz - 1;
          const float w = dlt[e];  // e is not a kept expert here (those were masked before the ballot)
          const float4* wr = reinterpret_cast<const float4*>(a.W_rT + (size_t)e * a.d + (size_t)v * VN);
#pragma unroll
          for (int qq = 0; qq < VN / 4; ++qq) {
            const float4 w4 = wr[qq];
            acc[4 * qq + 0] = fmaf(w, w4.x, acc[4 * qq + 0]);
            acc[4 * qq + 1] = fmaf(w, w4.y, acc[4 * qq + 1]);
            acc[4 * qq + 2] = fmaf(w, w4.z, acc[4 * qq + 2]);
            acc[4 * qq + 3] = fmaf(w, w4.w, acc[4 * qq + 3]);
          }
        }
      }
      stg16(dst + v * 16, pack(acc));
    }
  }
}

// -------------------------------------------------------------------------- //
// dW_r (+)= x^T dl in two passes, deterministic and without atomics.  dl has at
// most k nonzero experts per token when k > 1, so the product is taken
// sparsely.  Pass 1: a block owns 64 columns of x and one slice of the tokens;
// each warp takes a sub-slice in token order, lane l owning columns 2l, 2l+1,
// and adds dl[t,e] * x[t, cols] into its private shared-memory accumulator row
// e for every e with dl[t,e] != 0 (found with a ballot).  The block then sums
// its warps in index order and writes the slice's partial.  Pass 2 adds the
// slices in slice order.
// -------------------------------------------------------------------------- //
constexpr int DW_COLS = 64;
constexpr int DW_STRIDE = DW_COLS + 2;  // accumulator row pitch: float2 adds stay aligned, column reads spread over banks
constexpr int DW_BATCH = 8;             // tokens whose loads a warp issues together

struct DwArgs {
  const void* x;
  const float* dl;
  float* partial;  // [splits][d][E]
  int T, d, E, tok_per_split, warps;
};

__device__ __forceinline__ float2 load_pair(const float* p) { return *reinterpret_cast<const float2*>(p); }
__device__ __forceinline__ float2 load_pair(const __nv_bfloat16* p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}

template <typename Tx>
__global__ void __launch_bounds__(256) dwr_partial_kernel(DwArgs a) {
  pdl_enter();  // see pdl_wait: no global access before this
  extern __shared__ float dw_acc[];  // [warps][E][DW_STRIDE]
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int i0 = blockIdx.x * DW_COLS, s = blockIdx.y;
  const int col = i0 + 2 * lane;
  const bool has_col = col < a.d;  // d is even for both dtypes
  const int chunks = (a.E + 31) / 32;
  float* acc = dw_acc + (size_t)warp * a.E * DW_STRIDE;
  for (int i = lane; i < a.E * DW_STRIDE; i += 32) acc[i] = 0.f;
  __syncwarp();
  const int sb = s * a.tok_per_split, se = min(a.T, sb + a.tok_per_split);
  const int per = (se - sb + a.warps - 1) / a.warps;
  const int tb = sb + warp * per, te = min(se, tb + per);
  const Tx* x = static_cast<const Tx*>(a.x);
  for (int t0 = tb; t0 < te; t0 += DW_BATCH) {
    float2 xv[DW_BATCH];
    float lv[DW_BATCH][4];
#pragma unroll
    for (int b = 0; b < DW_BATCH; ++b) {
      const int t = t0 + b;
      const bool ok = t < te;
      xv[b] = (ok && has_col) ? load_pair(x + (size_t)t * a.d + col) : make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int e = 32 * c + lane;
        lv[b][c] = (ok && c < chunks && e < a.E) ? a.dl[(size_t)t * a.E + e] : 0.f;
      }
    }
#pragma unroll
    for (int b = 0; b < DW_BATCH; ++b) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        if (c >= chunks) break;  // warp-uniform
        unsigned nz = __ballot_sync(0xffffffffu, lv[b][c] != 0.f);
        while (nz) {  // the experts of this token with a nonzero logit gradient, in expert order
          const int src = __ffs(nz) - 1;
          nz &= nz - 1;
          const float w = __shfl_sync(0xffffffffu, lv[b][c], src);
          float2* r = reinterpret_cast<float2*>(acc + (size_t)(32 * c + src) * DW_STRIDE + 2 * lane);
          float2 v = *r;
          v.x = fmaf(w, xv[b].x, v.x);
          v.y = fmaf(w, xv[b].y, v.y);
          *r = v;
        }
      }
    }
  }
  __syncthreads();
  // sum the warps in index order; write this slice's partial [d][E]
  for (int idx = tid; idx < a.E * DW_COLS; idx += blockDim.x) {
    const int c = idx / a.E, e = idx % a.E;  // consecutive threads: consecutive experts of one column
    float v = 0.f;
    for (int w = 0; w < a.warps; ++w) v += dw_acc[((size_t)w * a.E + e) * DW_STRIDE + c];
    if (i0 + c < a.d) a.partial[((size_t)s * a.d + i0 + c) * a.E + e] = v;
  }
}

__global__ void dwr_reduce_kernel(const float* partial, float* dW_r, int splits, int64_t n, int accumulate) {
  pdl_enter();  // see pdl_wait: no global access before this
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float p = 0.f;
#pragma unroll 8
  for (int q = 0; q < splits; ++q) p += partial[(size_t)q * n + i];
  dW_r[i] = accumulate ? dW_r[i] + p : p;
}

int row_vecs(const Shape& s) { return s.d * (s.bf16 ? 2 : 4) / 16; }

// Dispatch a (dtype, k) templated row kernel; k ranges over 1..8.
template <template <typename, int> class Kern, typename Args>
cudaError_t launch_typed_k(const Shape& s, const Args& a, int grid, cudaStream_t st) {
#define MOE_ROWS_CASE(KK)                                           \
  case KK:                                                          \
    if (s.bf16) return Kern<__nv_bfloat16, KK>::launch(a, grid, st); \
    return Kern<float, KK>::launch(a, grid, st);
  switch (s.k) {
    MOE_ROWS_CASE(1)
    MOE_ROWS_CASE(2)
    MOE_ROWS_CASE(3)
    MOE_ROWS_CASE(4)
    MOE_ROWS_CASE(5)
    MOE_ROWS_CASE(6)
    MOE_ROWS_CASE(7)
    MOE_ROWS_CASE(8)
    default: return cudaErrorInvalidValue;
  }
#undef MOE_ROWS_CASE
}

template <typename Tx, int K>
struct CombineL {
  static cudaError_t launch(const CombArgs& a, int grid, cudaStream_t st) {
    return launch_pdl(combine_kernel<Tx, K>, dim3(grid), dim3(RW_WARPS * 32), 0, st, a);
  }
};
template <typename Tx, int K>
struct CombineBwdL {
  static cudaError_t launch(const CombBwdArgs& a, int grid, cudaStream_t st) {
    if (a.dg == nullptr) return launch_pdl(combine_bwd_kernel<Tx, K, false>, dim3(grid), dim3(RW_WARPS * 32), 0, st, a);
    return launch_pdl(combine_bwd_kernel<Tx, K, true>, dim3(grid), dim3(RW_WARPS * 32), 0, st, a);
  }
};
template <typename Tx, int K>
struct DotL {  // no activation data: the element type does not matter
  static cudaError_t launch(const DotArgs& a, int grid, cudaStream_t st) {
    return launch_pdl(dl_from_dots_kernel<K>, dim3(grid), dim3(RW_WARPS * 32), 0, st, a);
  }
};
template <typename Tx, int K>
struct DxL {
  static cudaError_t launch(const DxArgs& a, int grid, cudaStream_t st) {
    return launch_pdl(dx_router_kernel<Tx, K>, dim3(grid), dim3(RW_WARPS * 32), 0, st, a);
  }
};
template <typename Tx, int K>
struct PermuteL {  // byte copies: the element type does not matter
  static cudaError_t launch(const PermArgs& a, int grid, cudaStream_t st) {
    return launch_pdl(permute_kernel<K>, dim3(grid), dim3(RW_WARPS * 32), 0, st, a);
  }
};

}  // namespace

cudaError_t launch_permute(const Shape& s, const void* x, const int32_t* row_of, const int32_t* counts,
                           const int32_t* offsets, void* x_perm, uint32_t* err, cudaStream_t st, const float* gates,
                           float* row_gate, void* y_zero) {
  PermArgs a{static_cast<const char*>(x), row_of, counts, offsets, static_cast<char*>(x_perm), gates, row_gate,
             static_cast<char*>(y_zero), err, s.T, s.E, row_vecs(s), s.max_rows, (s.T + RW_WARPS - 1) / RW_WARPS};
  LaunchScope ls(KK_PERMUTE, st);
  return launch_typed_k<PermuteL>(s, a, a.token_blocks + s.E, st);
}

cudaError_t launch_combine(const Shape& s, const void* y_perm, const int32_t* row_of, const float* gates, void* y,
                           uint32_t* err, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  CombArgs a{static_cast<const char*>(y_perm), row_of, gates, static_cast<char*>(y), err, s.T, row_vecs(s),
             s.max_rows};
  LaunchScope ls(KK_COMBINE, st);
  return launch_typed_k<CombineL>(s, a, (s.T + RW_WARPS - 1) / RW_WARPS, st);
}

cudaError_t launch_combine_bwd(const Shape& s, const void* dy, const void* y_perm, const int32_t* ids,
                               const int32_t* row_of, const float* gates, const float* probs,
                               const int32_t* counts, const int32_t* offsets, void* dy_perm, float* dg, float* dl,
                               uint32_t* err, cudaStream_t st) {
  CombBwdArgs a{static_cast<const char*>(dy), static_cast<const char*>(y_perm), ids, row_of, gates, probs,
                counts, offsets, static_cast<char*>(dy_perm), dg, dl, err, s.T, s.E, row_vecs(s), s.max_rows,
                (s.T + RW_WARPS - 1) / RW_WARPS};
  LaunchScope ls(KK_COMBINE_BWD, st);
  return launch_typed_k<CombineBwdL>(s, a, a.token_blocks + s.E, st);
}

cudaError_t launch_dl_from_dots(const Shape& s, const float* sdot, int nt, const int32_t* row_of,
                                const int32_t* ids, const float* gates, const float* probs, float* dl, uint32_t* err,
                                cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  DotArgs a{sdot, row_of, ids, gates, probs, dl, err, s.T, s.E, nt, s.max_rows};
  LaunchScope ls(KK_LOGIT_GRAD, st);
  return launch_typed_k<DotL>(s, a, (s.T + 4 * RW_WARPS - 1) / (4 * RW_WARPS), st);
}

cudaError_t launch_dx_router(const Shape& s, const void* dx_perm, const int32_t* row_of, const float* dl,
                             const float* W_r, float* W_rT, void* dx, uint32_t* err, cudaStream_t st,
                             const int32_t* ids) {
  if (s.T == 0) return cudaSuccess;
  {
    dim3 grid((s.d + 31) / 32, (s.E + 31) / 32);
    LaunchScope ls(KK_TRANSPOSE_WR, st);
    cudaError_t e = launch_pdl(transpose_wr_kernel, grid, dim3(32, 8), 0, st, W_r, W_rT, s.d, s.E);
    if (e != cudaSuccess) return e;
  }
  DxArgs a{static_cast<const char*>(dx_perm), row_of, ids, dl, W_rT, static_cast<char*>(dx), err, s.T, s.E, s.d,
           row_vecs(s), s.max_rows};
  LaunchScope ls(KK_DX_ROUTER, st);
  return launch_typed_k<DxL>(s, a, (s.T + RW_WARPS - 1) / RW_WARPS, st);
}

// Warps per block: the private accumulators stay near 66 KB so that three
// blocks fit on an SM.
int dwr_warps(const Shape& s) { return s.E <= 32 ? 8 : (s.E <= 64 ? 4 : 2); }

int dwr_splits(const Shape& s) {
  const int warps = dwr_warps(s), col_blocks = (s.d + DW_COLS - 1) / DW_COLS;
  int splits = (s.T + 64 * warps - 1) / (64 * warps);  // 64 tokens a warp
  const int want = (4 * 152 + col_blocks - 1) / col_blocks;  // about four blocks an SM
  if (splits < want) splits = std::min(want, (s.T + 16 * warps - 1) / (16 * warps));  // at least 16 tokens a warp
  const int64_t cap = ((int64_t)64 << 20) / ((int64_t)s.d * s.E * 4);  // partials within 64 MB
  if (splits > cap) splits = (int)std::max<int64_t>(cap, 1);
  if (splits > 65535) splits = 65535;  // grid y limit
  return splits < 1 ? 1 : splits;
}

cudaError_t launch_dwr(const Shape& s, const void* x, const float* dl, float* partial, float* dW_r, int accumulate,
                       cudaStream_t st) {
  const int splits = dwr_splits(s), warps = dwr_warps(s);
  DwArgs a{x, dl, partial, s.T, s.d, s.E, (s.T + splits - 1) / splits, warps};
  const size_t smem = (size_t)warps * s.E * DW_STRIDE * 4;
  {
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (!attr_done[dev]) {
      cudaError_t e1 = cudaFuncSetAttribute(dwr_partial_kernel<__nv_bfloat16>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
      cudaError_t e2 = cudaFuncSetAttribute(dwr_partial_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            96 * 1024);
      if (e1 != cudaSuccess || e2 != cudaSuccess) return e1 != cudaSuccess ? e1 : e2;
      attr_done[dev] = true;
    }
    dim3 grid((s.d + DW_COLS - 1) / DW_COLS, splits);
    LaunchScope ls(KK_DWR, st);
    cudaError_t e = s.bf16 ? launch_pdl(dwr_partial_kernel<__nv_bfloat16>, grid, dim3(warps * 32), smem, st, a)
                           : launch_pdl(dwr_partial_kernel<float>, grid, dim3(warps * 32), smem, st, a);
    if (e != cudaSuccess) return e;
  }
  return launch_dwr_reduce(partial, dW_r, splits, (int64_t)s.d * s.E, accumulate, st);
}

cudaError_t launch_dwr_reduce(const float* partial, float* dW_r, int splits, int64_t n, int accumulate,
                              cudaStream_t st) {
  LaunchScope ls(KK_DWR_REDUCE, st);
  return launch_pdl(dwr_reduce_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, partial, dW_r, splits,
                    n, accumulate);
}

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t st) {
  if (bytes == 0) return cudaSuccess;
  return cudaMemsetAsync(p, 0, bytes, st);
}

}  // namespace moe
