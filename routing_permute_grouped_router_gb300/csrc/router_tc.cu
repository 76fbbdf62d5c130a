// Router scoring on the tensor cores: logits = x W_r + b, then fp32 softmax,
// top-k and the per-block expert histogram, for bf16 layers.
//
// "The router scores every token" (gpu_expert_parallel page, step timeline)
// is a skinny product, T x d by d x E, that must come out in fp32 precision
// (the layer configurations fix an fp32 router).  x is exact in bf16; W_r is
// split into three bf16 parts, hi + mid + lo, which together carry its 24
// significand bits (the bf16x3 technique of Henry, Tang and Heinecke,
// "Leveraging the bfloat16 AI datatype for higher-precision computations",
// 2019).  Each product x * part is exact in the fp32 accumulator, so three
// MMAs per K step give fp32-accurate logits while reading x from HBM once at
// TMA speed.
//
// One cluster of cs CTAs per 128-token tile, CTA r of the cluster taking the
// r-th of cs equal K ranges (cs = 1, 2, 4 or 8, the largest that keeps tiles x
// cs within the SM count, so that few tokens still spread over the GPU): warp
// 0 lane 0 loads 128x64 x tiles and the three E_pad x 64 weight tiles with
// TMA (the parts land as consecutive E_pad-row blocks: one K-major operand of
// 3 * E_pad rows), warp 1 lane 0 issues one tcgen05.mma (M=128, N=3*E_pad,
// K=16; 256 + 128 columns when E_pad = 128) per K step into an fp32 TMEM
// accumulator of three column groups (x hi, x mid, x lo), and warps 2-5 read
// one token row per thread from TMEM, adding each logit's three groups, lo +
// mid first.
// CTAs r > 0 park their partial logits in their shared memory; the first CTA
// adds them over distributed shared memory in rank order (so the sum does not
// depend on timing) and does softmax and top-k in registers (value
// descending, lower expert index on ties).  The histogram is written per
// 64-token block, the layout the slot scan reads.
#include <cudaTypedefs.h>
#include <float.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int RT = 128;  // tokens per tile
constexpr int RK = 64;   // columns of one box (128-byte rows)
constexpr int HIST_TOK = 64;
constexpr int R_THREADS = 192;
constexpr int R_MAXK = 8;
constexpr int MAX_CS = 8;  // K ranges (cluster size) per token tile

template <int N>
struct RCfg {
  // up to N = 32 two CTAs fit on an SM (shared memory and registers), so a
  // large T runs in one wave; the stages fill what is left of the CTA's share
  static constexpr int MIN_BLOCKS = N <= 32 ? 2 : 1;
  // boxes per stage: a stage reads RB * 128 contiguous bytes of each token row
  static constexpr int RB = 1;
  static constexpr int A_BYTES = RB * RT * RK * 2;
  static constexpr int B_BYTES = RB * 3 * N * RK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STATIC_SMEM = 2 * R_MAXK * N * 4 + N * 4;
  static constexpr int BUDGET = (MIN_BLOCKS == 2 ? 115712 : 232448) - STATIC_SMEM - 256 - 1024;
  static constexpr int NST = BUDGET / STAGE > 8 ? 8 : BUDGET / STAGE;
  static constexpr int CTRL_OFF = NST * STAGE;
  static constexpr int SMEM = CTRL_OFF + 256 + 1024;
  // accumulator columns: the three parts side by side
  static constexpr int NS = 3 * N;
  static constexpr uint32_t TCOLS = NS <= 64 ? 64 : (NS <= 128 ? 128 : (NS <= 256 ? 256 : 512));
  static_assert(NST >= 2, "at least two stages");
  static_assert(RT * (N + 4) * 4 <= NST * STAGE, "partial logits fit in the stage buffers");
  // MMA widths: one of 3 * E_pad columns, or 256 + 128 for E_pad = 128
  static constexpr int N0 = NS <= 256 ? NS : 256;
  static constexpr int N1 = NS - N0;
  // fp32 D, bf16 A and B, both K-major, M = 128, N = N0 or N1
  static constexpr uint32_t IDESC0 = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N0 >> 3) << 17) |
                                     ((uint32_t)(RT >> 4) << 24);
  static constexpr uint32_t IDESC1 = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)((N1 > 0 ? N1 : 16) >> 3) << 17) |
                                     ((uint32_t)(RT >> 4) << 24);
};

struct RouterTcArgs {
  const float* bias;
  int32_t* ids;
  float* gates;
  float* probs;
  int32_t* hist;
  int32_t* ticket;
  uint32_t* err;
  int T, d, E, k, nb;
};

// W_r [d, E] fp32 -> wsplit [3][N][d] bf16 (hi, mid, lo; rows e >= E are zero).
__global__ void split_wr_kernel(const float* W_r, __nv_bfloat16* wsplit, int d, int E, int N) {
  pdl_enter();  // see pdl_wait: no global access before this
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)N * d) return;
  const int e = (int)(i / d), c = (int)(i % d);
  const float w = e < E ? W_r[(size_t)c * E + e] : 0.f;
  const __nv_bfloat16 hi = __float2bfloat16_rn(w);
  const float r1 = w - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(mid);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
  const size_t plane = (size_t)N * d;
  wsplit[i] = hi;
  wsplit[plane + i] = mid;
  wsplit[2 * plane + i] = lo;
}

// One token's logits v (no bias yet) -> bias (bias_s: the bias in shared
// memory, zero without one), top-k (value descending, lower expert index on
// ties; taken first, so the maximum is the first pick), fp32 softmax
// (probabilities written to the token's row prow of [T, E] unless it is null),
// gates and ids; the picks are returned in ej for the caller's histogram.
template <int N>
__device__ __forceinline__ void token_epilogue(const RouterTcArgs& a, float (&v)[N], int t, const float* bias_s,
                                               float* prow, int (&ej)[R_MAXK]) {
#pragma unroll
  for (int e = 0; e < N; ++e) {
    float l = -INFINITY;
    if (e < a.E) {
      l = v[e] + bias_s[e];
      if (isnan(l)) l = -INFINITY;
    }
    v[e] = l;
  }
  // if every untaken logit is -inf the lowest untaken index is picked; the
  // padding experts e >= E hold -inf and come after every real one, so they
  // never win (k <= E)
  constexpr int NW = (N + 31) / 32;
  uint32_t taken[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) taken[w] = 0u;
  float lj[R_MAXK];
#pragma unroll
  for (int j = 0; j < R_MAXK; ++j) {
    lj[j] = 0.f;
    ej[j] = 0;
  }
  // one pick per pass, the passes not unrolled: eight unrolled copies of the
  // scan made the kernel's code several times larger, and with E = 64 the
  // epilogue took 8 us longer
#pragma unroll 1
  for (int j = 0; j < a.k; ++j) {
    float bv = -INFINITY;
    int be = -1;
#pragma unroll
    for (int e = 0; e < N; ++e)
      if (!((taken[e >> 5] >> (e & 31)) & 1u) && (be < 0 || v[e] > bv)) {  // strict: lower index on ties
        bv = v[e];
        be = e;
      }
#pragma unroll
    for (int w = 0; w < NW; ++w)
      if ((be >> 5) == w) taken[w] |= 1u << (be & 31);
    lj[j] = bv;
    ej[j] = be;
  }
  const float mx = lj[0];
  // the exponentials first (independent, so they overlap), then their sum in
  // expert order
#pragma unroll
  for (int e = 0; e < N; ++e) v[e] = e < a.E ? expf(v[e] - mx) : 0.f;
  float se = 0.f;
#pragma unroll
  for (int e = 0; e < N; ++e)
    if (e < a.E) se += v[e];
  if (prow != nullptr) {
    const float inv = 1.f / se;  // one division; each probability within an ulp of exp / sum
    if ((a.E & 3) == 0) {  // the row starts on 16 bytes: whole float4 pieces
#pragma unroll
      for (int c = 0; c < N / 4; ++c)
        if (4 * c < a.E)
          reinterpret_cast<float4*>(prow)[c] =
              make_float4(v[4 * c] * inv, v[4 * c + 1] * inv, v[4 * c + 2] * inv, v[4 * c + 3] * inv);
    } else {
#pragma unroll
      for (int e = 0; e < N; ++e)
        if (e < a.E) prow[e] = v[e] * inv;
    }
  }
  float g[R_MAXK];
  if (a.k == 1) {
    g[0] = expf(lj[0] - mx) / se;
  } else {
    float den = 0.f;
#pragma unroll
    for (int j = 0; j < R_MAXK; ++j)
      if (j < a.k) {
        g[j] = expf(lj[j] - lj[0]);
        den += g[j];
      }
#pragma unroll
    for (int j = 0; j < R_MAXK; ++j)
      if (j < a.k) g[j] = g[j] / den;
  }
#pragma unroll
  for (int j = 0; j < R_MAXK; ++j)
    if (j < a.k) {
      a.ids[(size_t)t * a.k + j] = ej[j];
      a.gates[(size_t)t * a.k + j] = g[j];
    }
}

template <int N>
__global__ void __launch_bounds__(R_THREADS, RCfg<N>::MIN_BLOCKS) router_tc_kernel(const __grid_constant__ CUtensorMap map_x,
                                                                 const __grid_constant__ CUtensorMap map_w,
                                                                 const __grid_constant__ RouterTcArgs a) {
  using C = RCfg<N>;
  constexpr int PSTRIDE = N + 4;  // floats per parked row (16-byte rows, no bank conflicts)
  extern __shared__ uint8_t smem_raw[];
  __shared__ int hist_s[2][R_MAXK][N];
  __shared__ float bias_s[N];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::CTRL_OFF);
  uint64_t* empty_bar = full_bar + 8;
  uint64_t* tfull_bar = empty_bar + 8;
  uint64_t* drain_bar = tfull_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t cs = cluster_nctarank(), rank = cluster_ctarank();
  const int tile = blockIdx.x / (int)cs;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(smem_addr(&full_bar[i]), 1);
      mbar_init(smem_addr(&empty_bar[i]), 1);
    }
    mbar_init(smem_addr(tfull_bar), 1);
    mbar_init(smem_addr(drain_bar), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = threadIdx.x; i < 2 * R_MAXK * N; i += R_THREADS) (&hist_s[0][0][0])[i] = 0;
  pdl_enter();  // no global memory or TMEM access above this line
  for (int e = threadIdx.x; e < N; e += R_THREADS) bias_s[e] = (a.bias != nullptr && e < a.E) ? a.bias[e] : 0.f;
  if (threadIdx.x == 0 && tile == 0 && rank == 0) *a.ticket = 0;  // for the last-block election of the slot scan
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C::TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t smem_base = smem_addr(smem);
  const int kall = a.d / (RK * C::RB);
  const int kb0 = (int)rank * kall / (int)cs, kb1 = ((int)rank + 1) * kall / (int)cs;
  const int kblocks = kb1 - kb0;
  // Tiles start their K loop at different k-blocks, so CTAs running together
  // read different parts of W_r instead of all loading the same boxes from the
  // same L2 lines.  The order is fixed per tile, so the sums do not depend on
  // timing.
  const int rot = kblocks > 0 ? (int)(((unsigned)tile * 7u) % (unsigned)kblocks) : 0;
  float v[N];  // this thread's token row of logits (epilogue warps)
  bool have = false;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_map(&map_x);
      prefetch_map(&map_w);
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool alive = true;
      for (int i = 0; i < kblocks; ++i) {
        const int kb = (i + rot) % kblocks;
        if (!mbar_wait(smem_addr(&empty_bar[stage]), phase ^ 1u, abort_flag, a.err, 600)) {
          alive = false;
          break;
        }
        const uint32_t fb = smem_addr(&full_bar[stage]);
        mbar_expect_tx(fb, C::STAGE);
        const uint32_t sA = smem_base + stage * C::STAGE;
#pragma unroll
        for (int b = 0; b < C::RB; ++b) {
          const int col = ((kb0 + kb) * C::RB + b) * RK;
          tma_load_2d(sA + b * RT * 128, &map_x, fb, col, tile * RT);
#pragma unroll
          for (int s = 0; s < 3; ++s) tma_load_2d(sA + C::A_BYTES + (b * 3 + s) * N * 128, &map_w, fb, col, s * N);
        }
        ++issued;
        if (++stage == C::NST) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!alive) {
        const int n = issued < C::NST ? issued : C::NST;
        int s = stage;
        uint32_t ph = phase;
        for (int i = 0; i < n; ++i) {
          if (--s < 0) {
            s = C::NST - 1;
            ph ^= 1u;
          }
          for (uint32_t it = 0; it < (1u << 24) && !mbar_try_wait(smem_addr(&full_bar[s]), ph); ++it) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool alive = true;
      for (int i = 0; i < kblocks; ++i) {
        if (!mbar_wait(smem_addr(&full_bar[stage]), phase, abort_flag, a.err, 601)) {
          alive = false;
          break;
        }
        tc_fence_after();
        const uint32_t sA = smem_base + stage * C::STAGE;
        const uint32_t sB = sA + C::A_BYTES;
#pragma unroll
        for (int b = 0; b < C::RB; ++b)
#pragma unroll
          for (int k16 = 0; k16 < RK / 16; ++k16) {
            const uint64_t ad = sdesc(sA + b * RT * 128 + k16 * 32, 16, 1024);
            const uint32_t acc = (i | b | k16) != 0 ? 1u : 0u;
            const uint32_t sBb = sB + b * 3 * N * 128;
            umma_bf16(tmem_base, ad, sdesc(sBb + k16 * 32, 16, 1024), C::IDESC0, acc);
            if (C::N1 > 0)
              umma_bf16(tmem_base + C::N0, ad, sdesc(sBb + C::N0 * 128 + k16 * 32, 16, 1024), C::IDESC1, acc);
          }
        umma_commit(smem_addr(&empty_bar[stage]));
        if (++stage == C::NST) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (alive) umma_commit(smem_addr(tfull_bar));
      umma_commit(smem_addr(drain_bar));
      for (uint32_t it = 0; it < (1u << 26) && !mbar_try_wait(smem_addr(drain_bar), 0); ++it) {
      }
    }
  } else {
    // ---- epilogue: one token row per thread ----
    const int q = warp & 3;
    if (mbar_wait(smem_addr(tfull_bar), 0, abort_flag, a.err, 602)) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < N / 16; ++c) {
        uint32_t hi[16], mid[16], lo[16];
        const uint32_t col = tmem_base + ((uint32_t)(q * 32) << 16) + c * 16;
        tmem_ld16(col, hi);
        tmem_ld16(col + N, mid);
        tmem_ld16(col + 2 * N, lo);
        tmem_ld_wait16(hi);
        tmem_reg_fence16(mid);
        tmem_reg_fence16(lo);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          v[c * 16 + i] = (__uint_as_float(lo[i]) + __uint_as_float(mid[i])) + __uint_as_float(hi[i]);
      }
      have = true;
      if (rank != 0) {
        // the stage buffers are free once every MMA has completed
        float4* prow = reinterpret_cast<float4*>(smem + (size_t)(q * 32 + lane) * PSTRIDE * 4);
#pragma unroll
        for (int c = 0; c < N / 4; ++c) prow[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (cs > 1) cluster_sync();  // every partial of the tile is in place
  if (warp >= 2 && rank == 0) {
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int t = tile * RT + row;
    if (cs > 1) {
      // add the other ranks' partial logits, in rank order
      const uint32_t off = smem_addr(smem) + (uint32_t)row * PSTRIDE * 4;
      for (uint32_t r = 1; r < cs; ++r) {
        const uint32_t src = mapa_shared(off, r);
        // up to eight loads in flight before their first use
        constexpr int B = N / 4 < 8 ? N / 4 : 8;
#pragma unroll
        for (int c0 = 0; c0 < N / 4; c0 += B) {
          float4 pv[B];
#pragma unroll
          for (int c = 0; c < B; ++c) pv[c] = ld_shared_cluster_f4(src + 16 * (c0 + c));
#pragma unroll
          for (int c = 0; c < B; ++c) {
            v[4 * (c0 + c)] += pv[c].x;
            v[4 * (c0 + c) + 1] += pv[c].y;
            v[4 * (c0 + c) + 2] += pv[c].z;
            v[4 * (c0 + c) + 3] += pv[c].w;
          }
        }
      }
    }
    if (have && t < a.T) {
      int ej[R_MAXK];
      // rank 0's stage buffers are free once its MMAs are done: probabilities go there
      token_epilogue<N>(a, v, t, bias_s, a.probs != nullptr ? a.probs + (size_t)t * a.E : nullptr, ej);
#pragma unroll
      for (int j = 0; j < R_MAXK; ++j)
        if (j < a.k) atomicAdd(&hist_s[row / HIST_TOK][j][ej[j]], 1);
    }
  }
  if (cs > 1) cluster_sync();  // the first CTA has read every partial
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // histogram of the two 64-token blocks of this tile, laid out [e][j][block]
  for (int i = threadIdx.x; i < 2 * a.k * a.E && rank == 0; i += R_THREADS) {
    const int half = i / (a.k * a.E), r = i % (a.k * a.E), j = r / a.E, e = r % a.E;
    const int b = tile * 2 + half;
    if (b < a.nb) a.hist[((size_t)e * a.k + j) * a.nb + b] = hist_s[half][j][e];
  }
  if (warp == 1) tmem_dealloc(tmem_base, C::TCOLS);
}

PFN_cuTensorMapEncodeTiled_v12000 r_encode = nullptr;

bool router_encode_ready() {
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      r_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return r_encode != nullptr;
}

bool make_map_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                   uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return r_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int padded_experts(int E) { return E <= 16 ? 16 : (E <= 32 ? 32 : (E <= 64 ? 64 : 128)); }

template <int N>
cudaError_t launch_n(const CUtensorMap& mx, const CUtensorMap& mw, const RouterTcArgs& args, int tiles, int cs,
                     cudaStream_t st) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!attr_done[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(router_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, RCfg<N>::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(tiles * cs));
  cfg.blockDim = dim3(R_THREADS);
  cfg.dynamicSmemBytes = RCfg<N>::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  LaunchScope ls(KK_ROUTER, st);
  return cudaLaunchKernelEx(&cfg, router_tc_kernel<N>, mx, mw, args);
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 1;
  }
  return cached[dev];
}

}  // namespace

bool router_tc_supported(const Shape& s) { return s.bf16 && s.T >= RT && s.d % 256 == 0 && s.E <= 128; }

size_t router_wsplit_bytes(const Shape& s) { return (size_t)3 * padded_experts(s.E) * s.d * 2; }

cudaError_t launch_router_tc(const Shape& s, const void* x, const float* W_r, const float* bias, void* wsplit,
                             int32_t* ids, float* gates, float* probs, int32_t* hist, int32_t* ticket,
                             uint32_t* err, cudaStream_t st) {
  if (!router_encode_ready()) return cudaErrorNotSupported;
  const int N = padded_experts(s.E);
  {
    const int64_t n = (int64_t)N * s.d;
    LaunchScope ls(KK_SPLIT_WR, st);
    cudaError_t e = launch_pdl(split_wr_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, W_r,
                               static_cast<__nv_bfloat16*>(wsplit), s.d, s.E, N);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mx, mw;
  if (!make_map_bf16(&mx, x, (uint64_t)s.T, (uint64_t)s.d, RK, RT) ||
      !make_map_bf16(&mw, wsplit, (uint64_t)3 * N, (uint64_t)s.d, RK, (uint32_t)N))
    return cudaErrorInvalidValue;
  RouterTcArgs a{bias, ids, gates, probs, hist, ticket, err, s.T, s.d, s.E, s.k, router_blocks(s.T)};
  const int tiles = (s.T + RT - 1) / RT;
  // K ranges per tile: the most (up to 8) that keep one CTA per SM and at
  // least two k-blocks per range
  int cs = 1;
  const int rb = N == 16 ? RCfg<16>::RB : (N == 32 ? RCfg<32>::RB : (N == 64 ? RCfg<64>::RB : RCfg<128>::RB));
  while (cs < MAX_CS && tiles * cs * 2 <= sm_count() && s.d / (RK * rb) >= 4 * cs) cs *= 2;
  switch (N) {
    case 16: return launch_n<16>(mx, mw, a, tiles, cs, st);
    case 32: return launch_n<32>(mx, mw, a, tiles, cs, st);
    case 64: return launch_n<64>(mx, mw, a, tiles, cs, st);
    default: return launch_n<128>(mx, mw, a, tiles, cs, st);
  }
}

}  // namespace moe
