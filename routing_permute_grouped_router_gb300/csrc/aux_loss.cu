// Auxiliary load-balancing loss of the router and its logit gradient.
//
// The distributed-training tutorial's MoE configuration example ("The
// Conflict Between EP and TP") names an aux_loss coefficient but no formula;
// the usual expert-balance form is taken:
//
//   f_e = #{(t, j): ids[t, j] = e} / (T k)      assignment share before the drop
//   P_e = (1/T) sum_t p[t, e]                   mean router probability
//   L   = c E sum_e f_e P_e
//   dL/dl[t, e'] = c E / T p[t, e'] (f_e' - sum_e f_e p[t, e])
//
// (f is a count: no gradient flows through it).  Three small kernels, every
// sum in a fixed order so the result is bitwise reproducible:
//   aux_partial_kernel  per 256-token block: column sums of p and counts of ids;
//   aux_reduce_kernel   one block: adds the blocks in block order -> f, L;
//   aux_grad_kernel     a warp per token: dl[t, :] += ... in place.
#include "common.cuh"

namespace moe {
namespace {

constexpr int AUX_TOK = 256;  // tokens per partial block

__global__ void __launch_bounds__(AUX_TOK) aux_partial_kernel(const float* probs, const int32_t* ids, int T, int E,
                                                              int k, float* part_p, int32_t* part_c, uint32_t* err) {
  pdl_enter();  // see pdl_wait: no global access before this
  __shared__ int cnt[128];
  __shared__ float colsum[AUX_TOK];
  const int t0 = blockIdx.x * AUX_TOK;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int t = t0 + threadIdx.x;
  if (t < T)
    for (int j = 0; j < k; ++j) {
      const int e = ids[(size_t)t * k + j];
      if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);  // integer: the order does not matter
      else report_error(err, DEV_BAD_EXPERT, 40);
    }
  // column sums of p over the block's tokens: thread (g, e) adds tokens g, g + G,
  // ... in order, then thread e adds the G group sums in group order
  const int tn = min(AUX_TOK, T - t0);
  const int G = AUX_TOK / E;  // E <= 128, so G >= 2
  const int g = threadIdx.x / E, e = threadIdx.x % E;
  if (g < G) {
    float s = 0.f;
    for (int r = g; r < tn; r += G) s += probs[(size_t)(t0 + r) * E + e];
    colsum[g * E + e] = s;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < E; c += blockDim.x) {
    float s = 0.f;
    for (int q = 0; q < G; ++q) s += colsum[q * E + c];
    part_p[(size_t)blockIdx.x * E + c] = s;
    part_c[(size_t)blockIdx.x * E + c] = cnt[c];
  }
}

__global__ void __launch_bounds__(128) aux_reduce_kernel(const float* part_p, const int32_t* part_c, int nb, int T,
                                                         int E, int k, float coeff, float* f_out, float* loss) {
  pdl_enter();  // see pdl_wait: no global access before this
  __shared__ float term[128];
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float P = 0.f;
    int64_t c = 0;
    for (int b = 0; b < nb; ++b) {  // block order
      P += part_p[(size_t)b * E + e];
      c += part_c[(size_t)b * E + e];
    }
    const float f = (float)((double)c / ((double)T * (double)k));
    f_out[e] = f;
    term[e] = f * (P / (float)T);
  }
  __syncthreads();
  if (threadIdx.x == 0 && loss != nullptr) {
    float s = 0.f;
    for (int e = 0; e < E; ++e) s += term[e];  // expert order
    *loss = coeff * (float)E * s;
  }
}

__global__ void __launch_bounds__(256) aux_grad_kernel(const float* probs, const float* f, int T, int E, float scale,
                                                       float* dl) {
  pdl_enter();  // see pdl_wait: no global access before this
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const float* pt = probs + (size_t)t * E;
  float p[4], fe[4];
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int e = 32 * c + lane;
    p[c] = e < E ? pt[e] : 0.f;
    fe[c] = e < E ? f[e] : 0.f;
    s = fmaf(fe[c], p[c], s);
  }
  s = warp_sum(s);  // the same butterfly in every warp
  float* dt = dl + (size_t)t * E;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int e = 32 * c + lane;
    if (e < E) dt[e] += scale * p[c] * (fe[c] - s);
  }
}

}  // namespace

int aux_blocks(const Shape& s) { return (s.T + AUX_TOK - 1) / AUX_TOK; }

size_t aux_scratch_bytes(const Shape& s) {
  return (size_t)aux_blocks(s) * s.E * 8 + (size_t)s.E * 4 + 64;  // partial sums and counts, f
}

cudaError_t launch_aux_loss(const Shape& s, float coeff, const float* probs, const int32_t* ids, float* loss,
                            float* dl, void* scratch, uint32_t* err, cudaStream_t st) {
  if (s.T == 0 || coeff <= 0.f) {
    // no loss term: a caller that reads the scalar every step sees 0, not a stale value
    return loss != nullptr ? cudaMemsetAsync(loss, 0, sizeof(float), st) : cudaSuccess;
  }
  const int nb = aux_blocks(s);
  float* part_p = static_cast<float*>(scratch);
  int32_t* part_c = reinterpret_cast<int32_t*>(part_p + (size_t)nb * s.E);
  float* f = reinterpret_cast<float*>(part_c + (size_t)nb * s.E);
  {
    LaunchScope ls(KK_AUX_LOSS, st);
    cudaError_t e = launch_pdl(aux_partial_kernel, dim3(nb), dim3(AUX_TOK), 0, st, probs, ids, s.T, s.E, s.k, part_p,
                               part_c, err);
    if (e != cudaSuccess) return e;
    e = launch_pdl(aux_reduce_kernel, dim3(1), dim3(128), 0, st, static_cast<const float*>(part_p),
                   static_cast<const int32_t*>(part_c), nb, s.T, s.E, s.k, coeff, f, loss);
    if (e != cudaSuccess) return e;
  }
  LaunchScope ls(KK_AUX_GRAD, st);
  return launch_pdl(aux_grad_kernel, dim3((unsigned)((s.T + 7) / 8)), dim3(256), 0, st, probs,
                    static_cast<const float*>(f), s.T, s.E, coeff * (float)s.E / (float)s.T, dl);
}

}  // namespace moe
