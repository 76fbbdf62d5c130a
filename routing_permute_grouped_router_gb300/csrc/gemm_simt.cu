// fp32 grouped GEMMs on the CUDA cores, for fp32 layers.
//
// Same five products as the tensor-core path (gemm_tc.cu):
//   UP      a = X_e W1_e, b = X_e W3_e, h = silu(a) * b          (rows ragged)
//   DOWN    y_perm = H_e W2_e                                      (rows ragged)
//   DGRAD_H dH = dY_e W2_e^T; SwiGLU backward -> da, db            (rows ragged)
//   DGRAD_X dx_perm = da W1_e^T + db W3_e^T                        (rows ragged)
//   WGRAD   dW1_e = X_e^T da, dW3_e = X_e^T db, dW2_e = H_e^T dY_e (K ragged)
// fp32 FMA keeps the fp32 layer inside a 1e-4 relative tolerance, which the
// tf32 tensor-core kinds would not.  64x64 output tiles, K steps of 16,
// 256 threads with 4x4 outputs each.  Rows of one expert start at multiples of
// 128, so a 64-row tile never spans two experts.
#include "common.cuh"

namespace moe {
namespace {

enum SimtMode { S_UP = 0, S_DOWN, S_DGRAD_H, S_DGRAD_X, S_WGRAD };

struct SimtArgs {
  const float* x_perm;
  const float* a_in;
  const float* b_in;
  const float* h_in;
  const float* dy_perm;
  const float* da_in;
  const float* db_in;
  const float* W1;
  const float* W3;
  const float* W2;
  const int32_t* counts;
  const int32_t* offsets;
  float* o0;
  float* o1;
  float* o2;
  float* dW1;
  float* dW3;
  float* dW2;
  int accumulate;
  int E, d, f;
  int64_t max_rows;
  uint32_t* err;
};

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + expf(-z)); }

__device__ int expert_of_row(const int32_t* offsets, int E, int64_t row) {
  int lo = 0, hi = E - 1;  // largest e with offsets[e] <= row
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if (offsets[mid] <= row) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <int MODE>
__global__ void __launch_bounds__(256) simt_gemm_kernel(SimtArgs p) {
  pdl_enter();  // see pdl_wait: no global access before this
  constexpr bool DUAL = MODE == S_UP;
  __shared__ float As[16][64 + 4];
  __shared__ float Bs[16][64 + 4];
  __shared__ float B2s[DUAL ? 16 : 1][64 + 4];
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;

  int e = 0, M = 0, N = 0, K = 0, sub = 0;
  int64_t row0 = 0, krow0 = 0;
  int m0 = 0, n0 = 0;
  if (MODE == S_WGRAD) {
    sub = blockIdx.z % 3;
    e = blockIdx.z / 3;
    M = sub == 2 ? p.f : p.d;
    N = sub == 2 ? p.d : p.f;
    m0 = blockIdx.x * 64;
    n0 = blockIdx.y * 64;
    if (m0 >= M || n0 >= N) return;
    krow0 = p.offsets[e];
    K = p.counts[e];
  } else {
    row0 = (int64_t)blockIdx.x * 64;
    const int64_t total = p.offsets[p.E];
    if (total > p.max_rows) {
      if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) report_error(p.err, DEV_BAD_OFFSETS, 20 + MODE);
      return;
    }
    if (row0 >= total) return;
    e = expert_of_row(p.offsets, p.E, row0);
    N = (MODE == S_UP || MODE == S_DGRAD_H) ? p.f : p.d;
    K = (MODE == S_UP || MODE == S_DGRAD_H) ? p.d : (MODE == S_DOWN ? p.f : 2 * p.f);
    n0 = blockIdx.y * 64;
    if (n0 >= N) return;
  }

  float acc[4][4], acc2[DUAL ? 4 : 1][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[i][j] = 0.f;
      if (DUAL) acc2[DUAL ? i : 0][j] = 0.f;
    }

  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int idx = tid; idx < 16 * 64; idx += 256) {
      const int kk = idx / 64, mm = idx % 64;
      const int k = k0 + kk;
      float av = 0.f, bv = 0.f, b2 = 0.f;
      if (k < K) {
        const int64_t row = row0 + mm;
        const int n = n0 + mm;
        if (MODE == S_UP) {
          av = p.x_perm[row * p.d + k];
          if (n < N) {
            bv = p.W1[((int64_t)e * p.d + k) * p.f + n];
            b2 = p.W3[((int64_t)e * p.d + k) * p.f + n];
          }
        } else if (MODE == S_DOWN) {
          av = p.h_in[row * p.f + k];
          if (n < N) bv = p.W2[((int64_t)e * p.f + k) * p.d + n];
        } else if (MODE == S_DGRAD_H) {
          av = p.dy_perm[row * p.d + k];
          if (n < N) bv = p.W2[((int64_t)e * p.f + n) * p.d + k];
        } else if (MODE == S_DGRAD_X) {
          if (k < p.f) {
            av = p.da_in[row * p.f + k];
            if (n < N) bv = p.W1[((int64_t)e * p.d + n) * p.f + k];
          } else {
            av = p.db_in[row * p.f + (k - p.f)];
            if (n < N) bv = p.W3[((int64_t)e * p.d + n) * p.f + (k - p.f)];
          }
        } else {  // WGRAD: A(m,k) = src[(krow0 + k) * M + m], B(n,k) = src[(krow0 + k) * N + n]
          const int64_t r = krow0 + k;
          const int m = m0 + mm;
          const float* asrc = sub == 2 ? p.h_in : p.x_perm;
          const float* bsrc = sub == 0 ? p.da_in : (sub == 1 ? p.db_in : p.dy_perm);
          if (m < M) av = asrc[r * M + m];
          if (n < N) bv = bsrc[r * N + n];
        }
      }
      As[kk][mm] = av;
      Bs[kk][mm] = bv;
      if (DUAL) B2s[DUAL ? kk : 0][mm] = b2;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float av[4], bv[4], b2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        av[i] = As[kk][ty * 4 + i];
        bv[i] = Bs[kk][tx * 4 + i];
        if (DUAL) b2[i] = B2s[DUAL ? kk : 0][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
          if (DUAL) acc2[DUAL ? i : 0][j] = fmaf(av[i], b2[j], acc2[DUAL ? i : 0][j]);
        }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      if (MODE == S_WGRAD) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
        float* out = sub == 0 ? p.dW1 : (sub == 1 ? p.dW3 : p.dW2);
        float* o = out + ((int64_t)e * M + m) * N + n;
        *o = p.accumulate ? *o + acc[i][j] : acc[i][j];
        continue;
      }
      const int64_t row = row0 + ty * 4 + i;
      if (MODE == S_UP) {
        const float av = acc[i][j], bv = acc2[DUAL ? i : 0][j];
        p.o0[row * p.f + n] = silu_f(av) * bv;
        if (p.o1) p.o1[row * p.f + n] = av;
        if (p.o2) p.o2[row * p.f + n] = bv;
      } else if (MODE == S_DOWN || MODE == S_DGRAD_X) {
        p.o0[row * p.d + n] = acc[i][j];
      } else {  // DGRAD_H
        const float dh = acc[i][j];
        const float av = p.a_in[row * p.f + n], bv = p.b_in[row * p.f + n];
        const float s = 1.f / (1.f + expf(-av));
        p.o0[row * p.f + n] = dh * bv * s * (1.f + av * (1.f - s));
        p.o1[row * p.f + n] = dh * av * s;
      }
    }
}

template <int MODE>
cudaError_t launch_simt(const SimtArgs& a, dim3 grid, int kind, cudaStream_t st) {
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  LaunchScope ls(kind, st);
  return launch_pdl(simt_gemm_kernel<MODE>, grid, dim3(256), 0, st, a);
}

}  // namespace

cudaError_t simt_ffn_fwd(const Shape& s, const FfnFwdArgs& f, uint32_t* err, cudaStream_t st) {
  SimtArgs a{};
  a.x_perm = static_cast<const float*>(f.x_perm);
  a.W1 = static_cast<const float*>(f.W1);
  a.W3 = static_cast<const float*>(f.W3);
  a.W2 = static_cast<const float*>(f.W2);
  a.counts = f.counts;
  a.offsets = f.offsets;
  a.E = s.E;
  a.d = s.d;
  a.f = s.f;
  a.max_rows = s.max_rows;
  a.err = err;
  const unsigned mt = (unsigned)(s.max_rows / 64);
  a.o0 = static_cast<float*>(f.h);
  a.o1 = static_cast<float*>(f.a);
  a.o2 = static_cast<float*>(f.b);
  cudaError_t e = launch_simt<S_UP>(a, dim3(mt, (s.f + 63) / 64), KK_GEMM_UP, st);
  if (e != cudaSuccess || f.y_perm == nullptr) return e;  // null: the up product alone
  a.h_in = static_cast<const float*>(f.h);
  a.o0 = static_cast<float*>(f.y_perm);
  a.o1 = a.o2 = nullptr;
  return launch_simt<S_DOWN>(a, dim3(mt, (s.d + 63) / 64), KK_GEMM_DOWN, st);
}

cudaError_t simt_ffn_bwd(const Shape& s, const FfnBwdArgs& b, uint32_t* err, cudaStream_t st) {
  if (b.part != 0 || b.sdot != nullptr) return cudaErrorInvalidValue;  // the staged backward is bf16 only
  SimtArgs a{};
  a.x_perm = static_cast<const float*>(b.x_perm);
  a.a_in = static_cast<const float*>(b.a);
  a.b_in = static_cast<const float*>(b.b);
  a.h_in = static_cast<const float*>(b.h);
  a.dy_perm = static_cast<const float*>(b.dy_perm);
  a.da_in = static_cast<const float*>(b.da);
  a.db_in = static_cast<const float*>(b.db);
  a.W1 = static_cast<const float*>(b.W1);
  a.W3 = static_cast<const float*>(b.W3);
  a.W2 = static_cast<const float*>(b.W2);
  a.counts = b.counts;
  a.offsets = b.offsets;
  a.E = s.E;
  a.d = s.d;
  a.f = s.f;
  a.max_rows = s.max_rows;
  a.err = err;
  a.dW1 = b.dW1;
  a.dW3 = b.dW3;
  a.dW2 = b.dW2;
  a.accumulate = b.accumulate;
  const unsigned mt = (unsigned)(s.max_rows / 64);
  a.o0 = static_cast<float*>(b.da);
  a.o1 = static_cast<float*>(b.db);
  cudaError_t e = launch_simt<S_DGRAD_H>(a, dim3(mt, (s.f + 63) / 64), KK_GEMM_DGRAD_H, st);
  if (e != cudaSuccess) return e;
  const int mx = s.d > s.f ? s.d : s.f;
  e = launch_simt<S_WGRAD>(a, dim3((mx + 63) / 64, (mx + 63) / 64, 3 * s.E), KK_GEMM_WGRAD, st);
  if (e != cudaSuccess) return e;
  a.o0 = static_cast<float*>(b.dx_perm);
  a.o1 = nullptr;
  return launch_simt<S_DGRAD_X>(a, dim3(mt, (s.d + 63) / 64), KK_GEMM_DGRAD_X, st);
}

}  // namespace moe
