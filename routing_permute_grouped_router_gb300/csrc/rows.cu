// Row-moving kernels of the layer step: the permute into per-expert buffers,
// the gate-weighted unpermute + combine, their backward (token-gradient
// routing), the dx gather with the router's input gradient, and the router
// weight gradient.
//
// All of them are HBM-bound row copies.  One warp owns one token row and moves
// it in 16-byte vectors (8 bf16 or 4 fp32 per lane), so every warp access is a
// contiguous 512-byte segment.  Sums run in fp32 in a fixed order (choice j
// ascending), so results are deterministic and use no atomics.
#include <float.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int RW_WARPS = 8;  // warps (= token rows) per block
constexpr int MAXK = 8;

__device__ __forceinline__ bool row_ok(int64_t r, int64_t max_rows) { return r >= 0 && r < max_rows; }

// -------------------------------------------------------------------------- //
// Permute (scatter form: each token row is read once and written to each of
// its kept rows); blocks past the token range zero the pad rows of one expert.
// -------------------------------------------------------------------------- //
struct PermArgs {
  const char* x;
  const int32_t* row_of;
  const int32_t* counts;
  const int32_t* offsets;
  char* x_perm;
  uint32_t* err;
  int T, k, E, nvec;  // nvec = 16-byte vectors per row
  int64_t max_rows;
  int token_blocks;
};

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

__global__ void __launch_bounds__(RW_WARPS * 32) permute_kernel(PermArgs a) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if ((int)blockIdx.x >= a.token_blocks) {
    zero_pad_rows(a.counts, a.offsets, blockIdx.x - a.token_blocks, a.x_perm, a.nvec, a.max_rows, a.err, warp,
                  lane, 10);
    return;
  }
  const int t = blockIdx.x * RW_WARPS + warp;
  if (t >= a.T) return;
  int64_t rows[MAXK];
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    rows[j] = -1;
    if (j < a.k) {
      const int64_t r = a.row_of[(size_t)t * a.k + j];
      if (r >= 0 && !row_ok(r, a.max_rows)) {
        if (lane == 0) report_error(a.err, DEV_BAD_ROW, 10);
      } else {
        rows[j] = r;
      }
    }
  }
  const char* src = a.x + (int64_t)t * a.nvec * 16;
  constexpr int U = 4;
  for (int v0 = lane; v0 < a.nvec; v0 += 32 * U) {
    uint4 val[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v < a.nvec) val[u] = ldg16(src + v * 16);
    }
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      if (rows[j] < 0) continue;
      char* dst = a.x_perm + rows[j] * a.nvec * 16;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = v0 + 32 * u;
        if (v < a.nvec) stg16(dst + v * 16, val[u]);
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
  int T, k, nvec;
  int64_t max_rows;
};

template <typename Tx>
__global__ void __launch_bounds__(RW_WARPS * 32) combine_kernel(CombArgs a) {
  constexpr int VN = Vec<Tx>::N;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t = blockIdx.x * RW_WARPS + warp;
  if (t >= a.T) return;
  int64_t rows[MAXK];
  float g[MAXK];
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    rows[j] = -1;
    g[j] = 0.f;
    if (j < a.k) {
      const int64_t r = a.row_of[(size_t)t * a.k + j];
      if (r >= 0 && !row_ok(r, a.max_rows)) {
        if (lane == 0) report_error(a.err, DEV_BAD_ROW, 11);
      } else if (r >= 0) {
        rows[j] = r;
        g[j] = a.gates[(size_t)t * a.k + j];
      }
    }
  }
  char* dst = a.y + (int64_t)t * a.nvec * 16;
  for (int v = lane; v < a.nvec; v += 32) {
    float acc[VN];
#pragma unroll
    for (int i = 0; i < VN; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      if (rows[j] < 0) continue;
      float val[VN];
      unpack(ldg16(a.y_perm + (rows[j] * a.nvec + v) * 16), val);
#pragma unroll
      for (int i = 0; i < VN; ++i) acc[i] = fmaf(g[j], val[i], acc[i]);
    }
    stg16(dst + v * 16, pack(acc));
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
  int T, k, E, nvec;
  int64_t max_rows;
  int token_blocks;
};

template <typename Tx>
__global__ void __launch_bounds__(RW_WARPS * 32) combine_bwd_kernel(CombBwdArgs a) {
  constexpr int VN = Vec<Tx>::N;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if ((int)blockIdx.x >= a.token_blocks) {
    zero_pad_rows(a.counts, a.offsets, blockIdx.x - a.token_blocks, a.dy_perm, a.nvec, a.max_rows, a.err, warp,
                  lane, 12);
    return;
  }
  const int t = blockIdx.x * RW_WARPS + warp;
  if (t >= a.T) return;
  int64_t rows[MAXK];
  float g[MAXK], part[MAXK];
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    rows[j] = -1;
    g[j] = 0.f;
    part[j] = 0.f;
    if (j < a.k) {
      g[j] = a.gates[(size_t)t * a.k + j];
      const int64_t r = a.row_of[(size_t)t * a.k + j];
      if (r >= 0 && !row_ok(r, a.max_rows)) {
        if (lane == 0) report_error(a.err, DEV_BAD_ROW, 12);
      } else {
        rows[j] = r;
      }
    }
  }
  const char* src = a.dy + (int64_t)t * a.nvec * 16;
  for (int v = lane; v < a.nvec; v += 32) {
    float dyv[VN];
    unpack(ldg16(src + v * 16), dyv);
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      if (rows[j] < 0) continue;
      float yv[VN], o[VN];
      unpack(ldg16(a.y_perm + (rows[j] * a.nvec + v) * 16), yv);
#pragma unroll
      for (int i = 0; i < VN; ++i) {
        part[j] = fmaf(dyv[i], yv[i], part[j]);
        o[i] = g[j] * dyv[i];
      }
      stg16(a.dy_perm + (rows[j] * a.nvec + v) * 16, pack(o));
    }
  }
  float dg[MAXK];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    dg[j] = (j < a.k) ? warp_sum(part[j]) : 0.f;
    s = fmaf(g[j], dg[j], s);
  }
  if (lane == 0) {
#pragma unroll
    for (int j = 0; j < MAXK; ++j)
      if (j < a.k) a.dg[(size_t)t * a.k + j] = dg[j];
  }
  if (a.k == 1) {
    const int e1 = a.ids[(size_t)t];
    const float gd = g[0] * dg[0];
    for (int e = lane; e < a.E; e += 32) {
      const float p = a.probs[(size_t)t * a.E + e];
      a.dl[(size_t)t * a.E + e] = gd * ((e == e1 ? 1.f : 0.f) - p);
    }
  } else {
    for (int e = lane; e < a.E; e += 32) {
      float v = 0.f;
#pragma unroll
      for (int j = 0; j < MAXK; ++j)
        if (j < a.k && a.ids[(size_t)t * a.k + j] == e) v += g[j] * (dg[j] - s);
      a.dl[(size_t)t * a.E + e] = v;
    }
  }
}

// -------------------------------------------------------------------------- //
// W_r^T (E x d) so the router's input gradient reads contiguous rows.
// -------------------------------------------------------------------------- //
__global__ void transpose_wr_kernel(const float* W_r, float* W_rT, int d, int E) {
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
// dx[t] = sum_j dX_perm[row_of[t,j]] + sum_{e: dl[t,e] != 0} dl[t,e] W_r[:, e]
// -------------------------------------------------------------------------- //
struct DxArgs {
  const char* dx_perm;
  const int32_t* row_of;
  const float* dl;
  const float* W_rT;
  char* dx;
  uint32_t* err;
  int T, k, E, d, nvec;
  int64_t max_rows;
};

template <typename Tx>
__global__ void __launch_bounds__(RW_WARPS * 32) dx_router_kernel(DxArgs a) {
  constexpr int VN = Vec<Tx>::N;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t = blockIdx.x * RW_WARPS + warp;
  if (t >= a.T) return;
  int64_t rows[MAXK];
#pragma unroll
  for (int j = 0; j < MAXK; ++j) {
    rows[j] = -1;
    if (j < a.k) {
      const int64_t r = a.row_of[(size_t)t * a.k + j];
      if (r >= 0 && !row_ok(r, a.max_rows)) {
        if (lane == 0) report_error(a.err, DEV_BAD_ROW, 13);
      } else {
        rows[j] = r;
      }
    }
  }
  // Experts with a nonzero logit gradient (at most k of them when k > 1),
  // found with all lanes active before the row loop.
  const float* dlt = a.dl + (size_t)t * a.E;
  unsigned nzmask[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int e = 32 * c + lane;
    const float mine = (e < a.E) ? dlt[e] : 0.f;
    nzmask[c] = __ballot_sync(0xffffffffu, mine != 0.f);
  }
  for (int v = lane; v < a.nvec; v += 32) {
    float acc[VN];
#pragma unroll
    for (int i = 0; i < VN; ++i) acc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < MAXK; ++j) {
      if (rows[j] < 0) continue;
      float val[VN];
      unpack(ldg16(a.dx_perm + (rows[j] * a.nvec + v) * 16), val);
#pragma unroll
      for (int i = 0; i < VN; ++i) acc[i] += val[i];
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      unsigned nz = nzmask[c];
      while (nz) {
        const int e = 32 * c + __ffs(nz) - 1;
        nz &= nz - 1;
        const float w = dlt[e];
        const float4* wr = reinterpret_cast<const float4*>(a.W_rT + (size_t)e * a.d + (size_t)v * VN);
#pragma unroll
        for (int q = 0; q < VN / 4; ++q) {
          const float4 w4 = wr[q];
          acc[4 * q + 0] = fmaf(w, w4.x, acc[4 * q + 0]);
          acc[4 * q + 1] = fmaf(w, w4.y, acc[4 * q + 1]);
          acc[4 * q + 2] = fmaf(w, w4.z, acc[4 * q + 2]);
          acc[4 * q + 3] = fmaf(w, w4.w, acc[4 * q + 3]);
        }
      }
    }
    stg16(a.dx + ((int64_t)t * a.nvec + v) * 16, pack(acc));
  }
}

// -------------------------------------------------------------------------- //
// dW_r = x^T dl: partial sums over token splits, then a fixed-order reduction.
// -------------------------------------------------------------------------- //
constexpr int DW_COLS = 64;
constexpr int DW_TOK = 32;

struct DwArgs {
  const void* x;
  const float* dl;
  float* partial;  // [splits, d, E]
  int T, d, E, tok_per_split;
};

template <int EP, typename Tx>
__global__ void __launch_bounds__(256) dwr_partial_kernel(DwArgs a) {
  constexpr int EQ = EP / 4;  // experts per thread
  __shared__ float dls[DW_TOK][EP];
  __shared__ float xs[DW_TOK][DW_COLS + 1];
  const Tx* x = static_cast<const Tx*>(a.x);
  const int tid = threadIdx.x, col = tid % DW_COLS, eg = tid / DW_COLS;
  const int i0 = blockIdx.x * DW_COLS, s = blockIdx.y;
  const int tb = s * a.tok_per_split, te = min(a.T, tb + a.tok_per_split);
  float acc[EQ];
#pragma unroll
  for (int q = 0; q < EQ; ++q) acc[q] = 0.f;
  for (int t0 = tb; t0 < te; t0 += DW_TOK) {
    for (int idx = tid; idx < DW_TOK * EP; idx += 256) {
      const int r = idx / EP, e = idx % EP, t = t0 + r;
      dls[r][e] = (t < te && e < a.E) ? a.dl[(size_t)t * a.E + e] : 0.f;
    }
    for (int idx = tid; idx < DW_TOK * DW_COLS; idx += 256) {
      const int r = idx / DW_COLS, c = idx % DW_COLS, t = t0 + r, i = i0 + c;
      xs[r][c] = (t < te && i < a.d) ? to_f32(x[(size_t)t * a.d + i]) : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int r = 0; r < DW_TOK; ++r) {
      const float xv = xs[r][col];
#pragma unroll
      for (int q = 0; q < EQ; ++q) acc[q] = fmaf(xv, dls[r][eg + 4 * q], acc[q]);
    }
    __syncthreads();
  }
  const int i = i0 + col;
  if (i < a.d) {
#pragma unroll
    for (int q = 0; q < EQ; ++q) {
      const int e = eg + 4 * q;
      if (e < a.E) a.partial[((size_t)s * a.d + i) * a.E + e] = acc[q];
    }
  }
}

__global__ void dwr_reduce_kernel(const float* partial, float* dW_r, int splits, int64_t n, int accumulate) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float s = accumulate ? dW_r[i] : 0.f;
  float p = 0.f;
  for (int q = 0; q < splits; ++q) p += partial[(size_t)q * n + i];
  dW_r[i] = s + p;
}

template <int EP>
cudaError_t launch_dwr_ep(const Shape& s, const DwArgs& a, int splits, cudaStream_t st) {
  dim3 grid((s.d + DW_COLS - 1) / DW_COLS, splits);
  LaunchScope ls(KK_DWR_PARTIAL, st);
  if (s.bf16)
    dwr_partial_kernel<EP, __nv_bfloat16><<<grid, 256, 0, st>>>(a);
  else
    dwr_partial_kernel<EP, float><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

int row_vecs(const Shape& s) { return s.d * (s.bf16 ? 2 : 4) / 16; }

}  // namespace

cudaError_t launch_permute(const Shape& s, const void* x, const int32_t* row_of, const int32_t* counts,
                           const int32_t* offsets, void* x_perm, uint32_t* err, cudaStream_t st) {
  PermArgs a{static_cast<const char*>(x), row_of, counts, offsets, static_cast<char*>(x_perm), err,
             s.T, s.k, s.E, row_vecs(s), s.max_rows, (s.T + RW_WARPS - 1) / RW_WARPS};
  const int grid = a.token_blocks + s.E;
  LaunchScope ls(KK_PERMUTE, st);
  permute_kernel<<<grid, RW_WARPS * 32, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_combine(const Shape& s, const void* y_perm, const int32_t* row_of, const float* gates, void* y,
                           uint32_t* err, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  CombArgs a{static_cast<const char*>(y_perm), row_of, gates, static_cast<char*>(y), err, s.T, s.k, row_vecs(s),
             s.max_rows};
  const int grid = (s.T + RW_WARPS - 1) / RW_WARPS;
  LaunchScope ls(KK_COMBINE, st);
  if (s.bf16)
    combine_kernel<__nv_bfloat16><<<grid, RW_WARPS * 32, 0, st>>>(a);
  else
    combine_kernel<float><<<grid, RW_WARPS * 32, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const Shape& s, const void* dy, const void* y_perm, const int32_t* ids,
                               const int32_t* row_of, const float* gates, const float* probs,
                               const int32_t* counts, const int32_t* offsets, void* dy_perm, float* dg, float* dl,
                               uint32_t* err, cudaStream_t st) {
  CombBwdArgs a{static_cast<const char*>(dy), static_cast<const char*>(y_perm), ids, row_of, gates, probs,
                counts, offsets, static_cast<char*>(dy_perm), dg, dl, err, s.T, s.k, s.E, row_vecs(s), s.max_rows,
                (s.T + RW_WARPS - 1) / RW_WARPS};
  const int grid = a.token_blocks + s.E;
  LaunchScope ls(KK_COMBINE_BWD, st);
  if (s.bf16)
    combine_bwd_kernel<__nv_bfloat16><<<grid, RW_WARPS * 32, 0, st>>>(a);
  else
    combine_bwd_kernel<float><<<grid, RW_WARPS * 32, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dx_router(const Shape& s, const void* dx_perm, const int32_t* row_of, const float* dl,
                             const float* W_r, float* W_rT, void* dx, uint32_t* err, cudaStream_t st) {
  if (s.T == 0) return cudaSuccess;
  {
    dim3 grid((s.d + 31) / 32, (s.E + 31) / 32);
    LaunchScope ls(KK_TRANSPOSE_WR, st);
    transpose_wr_kernel<<<grid, dim3(32, 8), 0, st>>>(W_r, W_rT, s.d, s.E);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  DxArgs a{static_cast<const char*>(dx_perm), row_of, dl, W_rT, static_cast<char*>(dx), err, s.T, s.k, s.E, s.d,
           row_vecs(s), s.max_rows};
  const int grid = (s.T + RW_WARPS - 1) / RW_WARPS;
  LaunchScope ls(KK_DX_ROUTER, st);
  if (s.bf16)
    dx_router_kernel<__nv_bfloat16><<<grid, RW_WARPS * 32, 0, st>>>(a);
  else
    dx_router_kernel<float><<<grid, RW_WARPS * 32, 0, st>>>(a);
  return cudaGetLastError();
}

int dwr_splits(const Shape& s) {
  const int col_blocks = (s.d + DW_COLS - 1) / DW_COLS;
  int splits = (2 * 152 + col_blocks - 1) / col_blocks;
  const int max_splits = (s.T + DW_TOK - 1) / DW_TOK;
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  return splits;
}

cudaError_t launch_dwr(const Shape& s, const void* x, const float* dl, float* partial, int splits, float* dW_r,
                       int accumulate, cudaStream_t st) {
  int tps = (s.T + splits - 1) / splits;
  tps = (tps + DW_TOK - 1) / DW_TOK * DW_TOK;
  DwArgs a{x, dl, partial, s.T, s.d, s.E, tps};
  cudaError_t e;
  if (s.E <= 8) e = launch_dwr_ep<8>(s, a, splits, st);
  else if (s.E <= 16) e = launch_dwr_ep<16>(s, a, splits, st);
  else if (s.E <= 32) e = launch_dwr_ep<32>(s, a, splits, st);
  else if (s.E <= 64) e = launch_dwr_ep<64>(s, a, splits, st);
  else e = launch_dwr_ep<128>(s, a, splits, st);
  if (e != cudaSuccess) return e;
  const int64_t n = (int64_t)s.d * s.E;
  LaunchScope ls(KK_DWR_REDUCE, st);
  dwr_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(partial, dW_r, splits, n, accumulate);
  return cudaGetLastError();
}

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t st) {
  if (bytes == 0) return cudaSuccess;
  return cudaMemsetAsync(p, 0, bytes, st);
}

}  // namespace moe
