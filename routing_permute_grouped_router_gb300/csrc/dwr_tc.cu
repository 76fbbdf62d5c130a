// Router-weight gradient on the tensor cores, for bf16 layers:
//
//   dW_r (+)= x^T dl        [d x E] = [d x T] [T x E]
//
// (the router weight is a shared parameter whose gradient "behaves like any
// other", gpu_expert_parallel page).  The product is skinny (E <= 128) with a
// long K = T, so it is bound by reading x once.  x is exact in bf16; dl is
// fp32 and is split into three bf16 parts hi + mid + lo that together carry
// its 24 significand bits (the bf16x3 technique of Henry, Tang and Heinecke,
// 2019, also used for the router logits), so three MMAs per K step give an
// fp32-accurate product.
//
// split_dl_kernel writes the parts transposed, [3][E_pad][T_pitch] bf16, so
// that each part is a K-major MMA operand with 128-byte rows.  dwr_tc_kernel
// takes MT consecutive 128-row blocks of d (M; MT = 2 up to 64 experts) and one
// of S contiguous ranges of T (K): warp 0 lane 0 loads x^T (MN-major, two
// 64 x 64 boxes per block, so each token row is read in MT * 256-byte runs)
// and the three dl parts once per stage with TMA; the parts land as
// consecutive E_pad-row blocks, so together they are one K-major operand of
// 3 * E_pad rows, and warp 1 lane 0 issues one tcgen05.mma (M=128,
// N=3*E_pad, K=16; two MMAs of 256 and 128 columns when E_pad = 128) per block
// and K step against them into MT fp32 TMEM accumulators of three column
// groups (x^T hi, x^T mid, x^T lo); warps 2-5 add each row's three groups,
// lo + mid first, and write the (MT * 128) x E partial to partial[range][d][E].  The grid is one wave (at
// most one CTA per SM).  The ranges are then added in range order
// (dwr_reduce_kernel), so the result does not depend on timing.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int DM = 128;  // rows of d per MMA block
constexpr int DK = 64;   // tokens per stage (128-byte rows)
constexpr int D_THREADS = 192;
constexpr int D_SMEM_MAX = 232448;  // 227 KB per CTA

// MT 128-row blocks of d per CTA: two while the staged dl parts are small, so a
// stage's dl parts serve twice the MMA work and x is read in 512-byte runs.
template <int N>
struct DCfg {
  static constexpr int MT = N <= 64 ? 2 : 1;
  static constexpr int A_BYTES = MT * DM * DK * 2;  // x^T: two 64 x 64 boxes per block
  static constexpr int B_BYTES = 3 * N * DK * 2;    // the three dl parts
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int NST0 = (D_SMEM_MAX - 256 - 1024) / STAGE;
  static constexpr int NST = NST0 > 6 ? 6 : NST0;
  static constexpr int CTRL_OFF = NST * STAGE;
  static constexpr int SMEM = CTRL_OFF + 256 + 1024;
  // accumulator columns per block: the three parts side by side
  static constexpr int NS = 3 * N;
  static constexpr uint32_t TCOLS = MT * NS <= 32 ? 32 : (MT * NS <= 64 ? 64 : (MT * NS <= 128 ? 128 : (MT * NS <= 256 ? 256 : 512)));
  static_assert(MT * NS <= 512, "TMEM columns");
  static_assert(NST >= 2 && SMEM <= D_SMEM_MAX, "shared memory budget");
  // MMA widths: one of 3 * E_pad columns, or 256 + 128 for E_pad = 128
  static constexpr int N0 = NS <= 256 ? NS : 256;
  static constexpr int N1 = NS - N0;
  // fp32 D, bf16 A (MN-major) and B (K-major), M = 128, N = n
  static constexpr uint32_t IDESC0 =
      (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | ((uint32_t)(N0 >> 3) << 17) | ((uint32_t)(DM >> 4) << 24);
  static constexpr uint32_t IDESC1 = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) |
                                     ((uint32_t)((N1 > 0 ? N1 : 16) >> 3) << 17) | ((uint32_t)(DM >> 4) << 24);
};

// dl [T, E] fp32 -> parts [3][N][tp] bf16 (rows e >= E and columns t >= T are
// zero).  Block: 64 tokens; the tile goes through shared memory so both the
// reads (rows of E) and the writes (64 tokens of one expert) are contiguous.
__global__ void __launch_bounds__(256) split_dl_kernel(const float* dl, __nv_bfloat16* parts, int T, int E, int N,
                                                       int tp) {
  pdl_enter();  // see pdl_wait: no global access before this
  __shared__ float tile[64][129];
  const int t0 = blockIdx.x * 64;
  for (int i = threadIdx.x; i < 64 * E; i += blockDim.x) {
    const int r = i / E, e = i % E;
    tile[r][e] = t0 + r < T ? dl[(size_t)(t0 + r) * E + e] : 0.f;
  }
  __syncthreads();
  const size_t plane = (size_t)N * tp;
  for (int i = threadIdx.x; i < 64 * N; i += blockDim.x) {
    const int e = i / 64, r = i % 64, t = t0 + r;
    if (t >= tp) continue;
    const float w = (e < E && t < T) ? tile[r][e] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    const size_t o = (size_t)e * tp + t;
    parts[o] = hi;
    parts[plane + o] = mid;
    parts[2 * plane + o] = lo;
  }
}

struct DwrTcArgs {
  float* partial;  // [S][d][E]
  uint32_t* err;
  int T, d, E, S, kall;
};

template <int N>
__global__ void __launch_bounds__(D_THREADS, 1) dwr_tc_kernel(const __grid_constant__ CUtensorMap map_x,
                                                              const __grid_constant__ CUtensorMap map_l,
                                                              const __grid_constant__ DwrTcArgs a) {
  using C = DCfg<N>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::CTRL_OFF);
  uint64_t* empty_bar = full_bar + 8;
  uint64_t* tfull_bar = empty_bar + 8;
  uint64_t* drain_bar = tfull_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int m0 = blockIdx.x * (C::MT * DM), range = blockIdx.y;
  const int kb0 = range * a.kall / a.S, kb1 = (range + 1) * a.kall / a.S;
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
  pdl_enter();  // no global memory or TMEM access above this line
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C::TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t smem_base = smem_addr(smem);

  if (warp == 0) {
    if (lane == 0) {
      prefetch_map(&map_x);
      prefetch_map(&map_l);
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool alive = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(smem_addr(&empty_bar[stage]), phase ^ 1u, abort_flag, a.err, 650)) {
          alive = false;
          break;
        }
        const uint32_t fb = smem_addr(&full_bar[stage]);
        mbar_expect_tx(fb, C::STAGE);
        const uint32_t sA = smem_base + stage * C::STAGE;
#pragma unroll
        for (int b = 0; b < 2 * C::MT; ++b) tma_load_2d(sA + b * 8192, &map_x, fb, m0 + 64 * b, kb * DK);
#pragma unroll
        for (int p = 0; p < 3; ++p) tma_load_2d(sA + C::A_BYTES + p * N * 128, &map_l, fb, kb * DK, p * N);
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
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(smem_addr(&full_bar[stage]), phase, abort_flag, a.err, 651)) {
          alive = false;
          break;
        }
        tc_fence_after();
        const uint32_t sA = smem_base + stage * C::STAGE;
        const uint32_t sB = sA + C::A_BYTES;
#pragma unroll
        for (int k16 = 0; k16 < DK / 16; ++k16) {
          const uint32_t acc = (kb != kb0 || k16 != 0) ? 1u : 0u;
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) {
            const uint64_t ad = sdesc(sA + mt * (DM * DK * 2) + k16 * 2048, 8192, 1024);
            umma_bf16(tmem_base + mt * C::NS, ad, sdesc(sB + k16 * 32, 16, 1024), C::IDESC0, acc);
            if (C::N1 > 0)
              umma_bf16(tmem_base + mt * C::NS + C::N0, ad, sdesc(sB + C::N0 * 128 + k16 * 32, 16, 1024),
                        C::IDESC1, acc);
          }
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
    // ---- epilogue: one row of d per thread and block ----
    const int q = warp & 3;
    if (mbar_wait(smem_addr(tfull_bar), 0, abort_flag, a.err, 652)) {
      tc_fence_after();
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt) {
        const int row = m0 + mt * DM + q * 32 + lane;
        float* dst = a.partial + ((size_t)range * a.d + row) * a.E;
#pragma unroll
        for (int c = 0; c < N / 16; ++c) {
          uint32_t hi[16], mid[16], lo[16];
          const uint32_t col = tmem_base + ((uint32_t)(q * 32) << 16) + mt * C::NS + c * 16;
          tmem_ld16(col, hi);
          tmem_ld16(col + N, mid);
          tmem_ld16(col + 2 * N, lo);
          tmem_ld_wait16(hi);
          tmem_reg_fence16(mid);
          tmem_reg_fence16(lo);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (c * 16 + i < a.E)
              dst[c * 16 + i] = (__uint_as_float(lo[i]) + __uint_as_float(mid[i])) + __uint_as_float(hi[i]);
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::TCOLS);
}

PFN_cuTensorMapEncodeTiled_v12000 d_encode = nullptr;

bool dwr_encode_ready() {
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      d_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return d_encode != nullptr;
}

// 2-D bf16 tensor map: rows x cols with the given row pitch (elements), 128-byte swizzle.
bool map_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t pitch, uint32_t box_cols,
              uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return d_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int pad_experts(int E) { return E <= 16 ? 16 : (E <= 32 ? 32 : (E <= 64 ? 64 : 128)); }
int dl_pitch(int T) { return (T + 7) / 8 * 8; }  // 16-byte rows for the tensor map

int sms() {
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

template <int N>
cudaError_t launch_dwr_n(const CUtensorMap& mx, const CUtensorMap& ml, const DwrTcArgs& args, cudaStream_t st) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(dwr_tc_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, DCfg<N>::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  LaunchScope ls(KK_DWR, st);
  return launch_pdl(dwr_tc_kernel<N>, dim3(args.d / (DCfg<N>::MT * DM), args.S), dim3(D_THREADS),
                    (size_t)DCfg<N>::SMEM, st, mx, ml, args);
}

}  // namespace

int dwr_mt(const Shape& s) { return pad_experts(s.E) <= 64 ? 2 : 1; }

bool dwr_tc_supported(const Shape& s) { return s.bf16 && s.d % (dwr_mt(s) * DM) == 0 && s.E <= 128 && s.T > 0; }

// Ranges of T: as many as keep the grid within one wave (one CTA per SM over
// the blocks of d), each range at least two k-blocks of 64 tokens.
int dwr_tc_ranges(const Shape& s) {
  const int mt = s.d / (dwr_mt(s) * DM), kall = (s.T + DK - 1) / DK;
  int S = sms() / (mt > 0 ? mt : 1);
  const int most = (kall + 1) / 2;
  if (S > most) S = most;
  return S < 1 ? 1 : S;
}

size_t dwr_tc_split_bytes(const Shape& s) { return (size_t)3 * pad_experts(s.E) * dl_pitch(s.T) * 2; }

cudaError_t launch_dwr_tc(const Shape& s, const void* x, const float* dl, void* dlsplit, float* partial,
                          uint32_t* err, cudaStream_t st) {
  if (!dwr_encode_ready()) return cudaErrorNotSupported;
  const int N = pad_experts(s.E), tp = dl_pitch(s.T);
  {
    LaunchScope ls(KK_SPLIT_DL, st);
    cudaError_t e = launch_pdl(split_dl_kernel, dim3((unsigned)((tp + 63) / 64)), dim3(256), 0, st, dl,
                               static_cast<__nv_bfloat16*>(dlsplit), s.T, s.E, N, tp);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mx, ml;
  if (!map_bf16(&mx, x, (uint64_t)s.T, (uint64_t)s.d, (uint64_t)s.d, 64, DK) ||
      !map_bf16(&ml, dlsplit, (uint64_t)3 * N, (uint64_t)s.T, (uint64_t)tp, DK, (uint32_t)N))
    return cudaErrorInvalidValue;
  DwrTcArgs a{partial, err, s.T, s.d, s.E, dwr_tc_ranges(s), (s.T + DK - 1) / DK};
  switch (N) {
    case 16: return launch_dwr_n<16>(mx, ml, a, st);
    case 32: return launch_dwr_n<32>(mx, ml, a, st);
    case 64: return launch_dwr_n<64>(mx, ml, a, st);
    default: return launch_dwr_n<128>(mx, ml, a, st);
  }
}

}  // namespace moe
