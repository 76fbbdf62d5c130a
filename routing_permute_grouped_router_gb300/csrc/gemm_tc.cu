// bf16 grouped GEMMs of the expert FFN on the 5th-generation tensor cores.
//
// The permute makes each expert's tokens one contiguous row segment, so the
// expert computation is one grouped matrix multiply over ragged segments
// ("The permutation step matters more than it looks", gpu_expert_parallel
// page).  Five products share one persistent kernel:
//
//   UP      [a | b] = X_e [W1_e | W3_e]   -> h = silu(a) * b (and a, b)   A K-major, B MN-major
//   DOWN    y_perm  = H_e W2_e                                            A K-major, B MN-major
//   DOWN_COMBINE  y[t] += g * (H_e W2_e)[row] for the token t of each row (the
//           inference forward at k <= 2: the combine in the epilogue)      A K-major, B MN-major
//   DGRAD_H dH = dY_e W2_e^T -> da, db (SwiGLU backward in the epilogue)  A K-major, B K-major
//   DGRAD_X dx_perm = [da | db] [W1_e | W3_e]^T (K concatenated)          A K-major, B K-major
//   WGRAD   dW1_e = X_e^T da, dW3_e = X_e^T db, dW2_e = H_e^T dY_e (fp32)  A MN-major, B MN-major
//
// Structure: CTA pairs (clusters of two, one CTA per SM, 192 threads each).
// A pair computes a 256 x 256 tile with the 2-SM tcgen05 MMA: each CTA stages
// its own 128 rows of A and one half (128 columns) of B, and its TMEM receives
// its 128 rows of the fp32 accumulator.  Per 256 x 256 x 64 step an SM thus
// reads 32 KB of operands instead of the 48 KB a single-SM 128 x 256 tile
// needs for half the work.  Up, down and dgrad x run three 64 KB stages of two
// such steps behind one pair of barriers; dgrad h and wgrad, whose epilogues
// stage inputs, run five 32 KB stages of one step when K is short and three
// 64 KB stages of two steps when it is long (the _L modes).
//   warp 0, one lane: TMA producer of this CTA's halves into the stage ring;
//     the byte count of both CTAs lands on the first CTA's barrier;
//   warp 1: allocates TMEM with its peer; in the first CTA one lane issues
//     tcgen05.mma.cta_group::2 (M=256, N=256, K=16) and commits stage
//     releases and accumulator-ready events to the barriers of both CTAs;
//   warps 2-5 of both CTAs: epilogue of their own rows; tcgen05.ld moves a
//     32-row x 32-column slice per warp into registers, the fused math runs
//     there, results go to HBM by TMA; they release the accumulator on the
//     first CTA's barrier.
// Tiles are dealt to the pairs from a list the kernel derives on the device
// from offsets/counts, so the host never reads the routing outcome: round-robin,
// or for wgrad over experts of very different sizes in host and guest groups
// (see next_group).
// Expert segments are 128-row aligned, so the second half of an expert's last
// pair tile may lie outside the expert: it is computed and not stored.  Every
// mbarrier wait is bounded (2 s); on expiry the kernel records DEV_TIMEOUT in
// the error word, drains its own copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;  // BM: rows per CTA (the pair covers 2 * BM)
constexpr int BNH = BN / 2;                 // B columns staged by each CTA of the pair
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int B_BYTES = BNH * BK * 2;       // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int PAIR_STAGE_BYTES = 2 * STAGE_BYTES;  // bytes both CTAs land on the first CTA's full barrier
constexpr int CTRL_BYTES = 2048;
constexpr int THREADS = 192;
constexpr int EPI_WARPS = 4;
constexpr int BOX_BYTES = 4096;  // one staged output box: 32 rows x 128 bytes
constexpr int ACC_BUFS = 2;      // TMEM accumulators (256 columns each)
constexpr uint64_t ROUND_WAIT_NS = 20000000ull;  // a wgrad producer waits at most 20 ms for a round's others
constexpr uint32_t TMEM_COLS = 256 * ACC_BUFS;
constexpr int MAX_E = 128;
constexpr int MAX_SMEM = 232448;  // 227 KB per CTA
constexpr int MAX_ST = 6;

enum Mode { M_UP = 0, M_DOWN = 1, M_DGRAD_H = 2, M_DGRAD_X = 3, M_WGRAD = 4, M_DOWN_COMB = 5, M_WGRAD_L = 6,
            M_DGRAD_H_L = 7 };
// wgrad comes in two shapes, chosen on the host from the expert capacity:
// M_WGRAD for short K per tile (capacity-limited layers: the fp32 gradient
// read-modify-write dominates, so four staged gradient boxes a warp with two
// in flight, and five 32 KB stages) and M_WGRAD_L for long K (dropless
// layers: three 64 KB stages of two k-blocks, two gradient boxes a warp).
__host__ __device__ constexpr bool is_wgrad(int m) { return m == M_WGRAD || m == M_WGRAD_L; }
// dgrad h likewise: M_DGRAD_H (five 32 KB stages, its a|b boxes double-buffered)
// for short K, M_DGRAD_H_L for d >= 2048 (three 64 KB stages of two k-blocks,
// one a|b buffer a warp: a chunk's a and b are requested once the previous
// chunk's da and db have left the buffer, behind a long mainloop).
__host__ __device__ constexpr bool is_dgrad_h(int m) { return m == M_DGRAD_H || m == M_DGRAD_H_L; }

// Pipeline depth and epilogue staging per product.  Each epilogue warp owns two
// output boxes (double buffering of its TMA stores).  dgrad h also stages its a
// and b inputs, and wgrad the old fp32 gradient it adds to; both give up one
// mainloop stage for four boxes per warp.  The products with light epilogues
// take two 64-wide k-blocks per stage: half the barrier round trips and
// commits per FLOP (measured 7-8 % faster on the dropless E=32 layer).
static_assert(MAX_ST >= 6, "barrier arrays");
// control block: 33 mbarriers and 4 words below byte 320, then offsets, counts and pair prefixes
static_assert((2 * MAX_ST + 5 + 4 * 4) * 8 + 16 <= 320, "control block");
static_assert(320 + (3 * 128 + 2) * 4 <= 2048, "control block");
constexpr int KB_NARROW = 2;  // 64-wide k-blocks per stage of the products with light epilogues
template <int MODE>
struct ModeCfg {
  // k-blocks of 64 behind one pair of barriers
  static constexpr int KB = (MODE == M_DGRAD_H || MODE == M_WGRAD) ? 1 : KB_NARROW;
  // wgrad: staged fp32 gradient boxes per epilogue warp, and old-gradient boxes
  // requested ahead of the one being added
  static constexpr int WBUFS = MODE == M_WGRAD ? 4 : 2;
  static constexpr int WAHEAD = MODE == M_WGRAD ? 2 : 1;
  // wgrad with interleaved tiles: stages of the long (host) tile issued
  // between two short (guest) tiles, about 8 us of MMA work, longer than one
  // guest's epilogue; and the most stages a guest may have
  static constexpr int GUEST_GAP = KB == 2 ? 12 : 24;
  static constexpr int GUEST_MAX = KB == 2 ? 12 : 24;
  static constexpr int STAGE = KB * STAGE_BYTES;
  static constexpr int ABUFS = MODE == M_DGRAD_H ? 2 : 1;  // dgrad h: [a | b] box pairs per warp
  static constexpr int EPI_WARP_BYTES =
      (is_dgrad_h(MODE) ? 2 * ABUFS : (is_wgrad(MODE) ? WBUFS : 2)) * BOX_BYTES;
  // as many stages as fit next to the epilogue staging, at most MAX_ST
  static constexpr int NST0 = (MAX_SMEM - CTRL_BYTES - 1024 - EPI_WARPS * EPI_WARP_BYTES) / STAGE;
  static constexpr int NST = NST0 > MAX_ST ? MAX_ST : NST0;
  static constexpr int EPI_OFF = NST * STAGE;
  static constexpr int CTRL_OFF = EPI_OFF + EPI_WARPS * EPI_WARP_BYTES;
  static constexpr int SMEM = CTRL_OFF + CTRL_BYTES + 1024;  // + alignment slack
};
static_assert(ModeCfg<M_UP>::SMEM <= MAX_SMEM, "shared memory budget");
static_assert(ModeCfg<M_DGRAD_H>::SMEM <= MAX_SMEM, "shared memory budget");
static_assert(ModeCfg<M_DGRAD_H_L>::SMEM <= MAX_SMEM && ModeCfg<M_DGRAD_H_L>::NST >= 3, "shared memory budget");
static_assert(ModeCfg<M_WGRAD>::SMEM <= MAX_SMEM, "shared memory budget");
static_assert(ModeCfg<M_WGRAD_L>::SMEM <= MAX_SMEM && ModeCfg<M_WGRAD_L>::NST >= 3, "shared memory budget");

// Tensor maps per product (loads of the mainloop first, then epilogue maps):
//   UP      0 x_perm, 1 W1, 2 W3, 3 h (store), 4 a (store), 5 b (store)
//   DOWN    0 h, 1 W2, 2 y_perm (store)
//   DGRAD_H 0 dy_perm, 1 W2, 2 a (load), 3 b (load), 4 da (store), 5 db (store)
//   DGRAD_X 0 da, 1 db, 2 W1, 3 W3, 4 dx_perm (store)
//   WGRAD   0 x_perm, 1 h, 2 da, 3 db, 4 dy_perm, 5 dW1, 6 dW3, 7 dW2 (fp32 store / reduce-add)
struct TcMaps {
  CUtensorMap m[8];
};

struct TcArgs {
  const int32_t* counts;
  const int32_t* offsets;
  int E, d, f;
  int64_t max_rows;
  __nv_bfloat16* o0;  // UP: h      DOWN: y_perm   DGRAD_H: da   DGRAD_X: dx_perm
  __nv_bfloat16* o1;  // UP: a (or null)           DGRAD_H: db
  __nv_bfloat16* o2;  // UP: b (or null)
  const __nv_bfloat16* i0;  // DGRAD_H: a
  const __nv_bfloat16* i1;  // DGRAD_H: b
  float* w0;  // WGRAD: dW1
  float* w1;  // WGRAD: dW3
  float* w2;  // WGRAD: dW2
  const int32_t* src_token;  // DOWN_COMBINE: token of each row (-1: pad row)
  const float* row_gate;     // DOWN_COMBINE: gate of each row
  __nv_bfloat16* y;          // DOWN_COMBINE: [T, d] output, zeroed beforehand
  const float* rdl;          // DGRAD_X, optional: logit gradient dl [T, E]; with it the row's
  const float* rwr;          //   router term dl[token, e] * W_r[:, e] is added (W_r [d, E])
  int rE;
  float* sdot;  // DGRAD_H, optional: per row and column tile, sum over the tile's
                // columns of dH * h ([max_rows, f / 256], h = silu(a) * b)
  int* round_ctr;  // WGRAD, optional: zeroed counters, one a round of host and guest
                   // tiles, that keep the pairs' rounds in step (WG_ROUNDS of them)
  int accumulate;
  uint32_t* err;
};

// Instruction descriptor of kind::f16: fp32 D, bf16 A and B, M = 256 (the
// pair), N = 256.
__host__ __device__ constexpr uint32_t idesc_bf16(bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((2 * BM) >> 4) << 24);
}

// silu and sigmoid with the fast intrinsic divide (about 2 ulp; the results
// are rounded to bf16).  For z -> -inf the divisor overflows to inf and the
// intrinsic returns 0, the right limit.
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.f + __expf(-z)); }
__device__ __forceinline__ float sigmoid_f(float z) { return __fdividef(1.f, 1.f + __expf(-z)); }

// A staged output box is 32 rows x 128 bytes (64 bf16 or 32 fp32 per row) in
// the 128-byte swizzle the TMA expects: 16-byte chunk j of row r sits at chunk
// j ^ (r % 8).  Boxes start on 1024-byte boundaries.  Row r belongs to lane r.
__device__ __forceinline__ uint32_t box_chunk(uint32_t box, int lane, int j) {
  return box + lane * 128 + (((uint32_t)j ^ (uint32_t)(lane & 7)) << 4);
}
__device__ __forceinline__ void box_put_bf16x32(uint32_t box, int lane, int j0, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = v[8 * q + i];
    sts128(box_chunk(box, lane, j0 + q), pack(w));
  }
}
__device__ __forceinline__ void box_get_bf16x32(uint32_t box, int lane, int j0, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float w[8];
    unpack(lds128(box_chunk(box, lane, j0 + q)), w);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[8 * q + i] = w[i];
  }
}
__device__ __forceinline__ void box_put_f32x32(uint32_t box, int lane, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    sts128(box_chunk(box, lane, q), make_uint4(__float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]),
                                               __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3])));
}
__device__ __forceinline__ void box_get_f32x32(uint32_t box, int lane, float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint4 u = lds128(box_chunk(box, lane, q));
    v[4 * q] = __uint_as_float(u.x);
    v[4 * q + 1] = __uint_as_float(u.y);
    v[4 * q + 2] = __uint_as_float(u.z);
    v[4 * q + 3] = __uint_as_float(u.w);
  }
}
__device__ __forceinline__ void regs_to_f32(const uint32_t (&r)[32], float (&v)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------ tile schedule ------------------------------ //
// A pair tile is 256 rows (this CTA: the half `rank`) by 256 columns.
struct Tile {
  int e;
  int64_t row0;  // ragged-M modes: this CTA's first row; WGRAD: first K row
  int m0, n0;    // WGRAD: this CTA's output rows m0.. and the tile's columns n0..; others: n0
  int sub;       // WGRAD product: 0 = dW1, 1 = dW3, 2 = dW2
  int kblocks;
  bool valid;    // this CTA's rows belong to the tile's expert
};

template <int MODE>
__device__ __forceinline__ int n_tiles_of(const TcArgs& a) {
  if (MODE == M_UP) return a.f / 128;
  if (MODE == M_DOWN || MODE == M_DOWN_COMB || MODE == M_DGRAD_X) return a.d / BN;
  return a.f / BN;  // DGRAD_H, DGRAD_H_L
}

// Work is dealt to the pairs in groups: one host tile and g >= 0 guest tiles.
// Without interleaving every group is one tile, dealt round-robin (group j of
// pair p is tile p + j * npairs) into the two TMEM accumulators in turn.
//
// When WGRAD's experts differ widely in rows (`interleave`), its tiles are
// listed by expert from the most rows to the fewest (s_pair holds that expert
// order).  A tile's fp32 gradient read-modify-write (its epilogue) takes about
// as long whatever its K, so a short tile finishes its MMAs well before the
// epilogue of the tile before it is done, and with two accumulators the next
// MMA would wait for that epilogue.  So each round gives every pair one host
// from the front of the list and, when the host is long, g guests from the
// back: the pair issues GUEST_GAP stages of the host, one whole guest, the
// next GUEST_GAP stages, the next guest, ... and the rest of the host.  The
// host holds one accumulator for its whole K loop while the guests take turns
// in the other, each guest's epilogue running under the next host stages.
// Commits, and so epilogues, come in the order guest 0 .. guest g-1, host.
// Group k puts its host in accumulator k & 1 and its guests in the other:
// the next host then takes the accumulator the last guest used (its epilogue
// comes before this host's), and the next guests the one this host used.
// g is the same for all pairs of a round (from the round's last, shortest
// host: one guest per GUEST_GAP stages, with at least GUEST_GAP stages of the
// host after the last guest), and guests have at most GUEST_MAX stages.
struct Group {
  int members;  // pairs with a group in this round (interleaving)
  int host;   // tile index of the host
  int g;      // guests
  int gbase;  // guest i is tile gbase - i
};
struct GroupIter {
  int F, B;  // interleaving: the tiles not yet dealt are [F, B)
  int j;     // round-robin: the next group
};

// stages (of KB k-blocks) of WGRAD tile `tile`: its expert's rows over BK * KB
template <int MODE>
__device__ __forceinline__ int wg_stages(int tile, const TcArgs& a, const int* s_cnt, const int* s_pair) {
  const int P = (a.d / (2 * BM)) * (a.f / BN);
  const int c = s_cnt[s_pair[tile / (3 * P)]];
  return (c + BK * ModeCfg<MODE>::KB - 1) / (BK * ModeCfg<MODE>::KB);
}

// The next group of pair `pair`; false past the last one.  Every role of
// every CTA walks the same sequence of rounds, so they agree on the groups.
template <int MODE>
__device__ __forceinline__ bool next_group(GroupIter& it, Group& gr, int pair, int npairs, int total,
                                           bool interleave, const TcArgs& a, const int* s_cnt,
                                           const int* s_pair) {
  gr.g = 0;
  gr.gbase = 0;
  if (!is_wgrad(MODE) || !interleave) {
    gr.host = pair + it.j * npairs;
    ++it.j;
    return gr.host < total;
  }
  if (it.F >= it.B) return false;
  const int left = it.B - it.F;
  int g = 0;
  if (left > npairs) {
    // the round's last host is its shortest
    g = wg_stages<MODE>(it.F + npairs - 1, a, s_cnt, s_pair) / ModeCfg<MODE>::GUEST_GAP - 1;
    const int room = (left - npairs) / npairs;
    if (g > room) g = room;
    while (g > 0 && wg_stages<MODE>(it.B - g * npairs, a, s_cnt, s_pair) > ModeCfg<MODE>::GUEST_MAX) --g;
    if (g < 0) g = 0;
  }
  const int F0 = it.F, B0 = it.B;
  gr.members = left < npairs ? left : npairs;
  it.F += npairs;
  it.B -= g * npairs;
  if (pair >= (left < npairs ? left : npairs)) return false;
  gr.host = F0 + pair;
  gr.g = g;
  gr.gbase = B0 - 1 - pair * g;
  return true;
}

// s_pair[e]: pair tiles (of 2 x 128 rows) before expert e in the ragged-M modes;
// WGRAD: s_pair[r] is the r-th expert of the tile list (the expert with the
// r-th most rows, ties to the lower index, when interleaving; else r).
template <int MODE>
__device__ __forceinline__ Tile decode(int tile, uint32_t rank, const TcArgs& a, const int* s_off, const int* s_cnt,
                                       const int* s_pair) {
  Tile t{};
  t.valid = true;
  if (is_wgrad(MODE)) {
    const int P = (a.d / (2 * BM)) * (a.f / BN);  // pair tiles of one product of one expert
    t.e = s_pair[tile / (3 * P)];
    const int q = tile % (3 * P);
    int r, nt;
    if (q < 2 * P) {
      t.sub = q & 1;
      r = q >> 1;
      nt = a.f / BN;
    } else {
      t.sub = 2;
      r = q - 2 * P;
      nt = a.d / BN;
    }
    t.m0 = (r / nt) * 2 * BM + (int)rank * BM;
    t.n0 = (r % nt) * BN;
    t.row0 = s_off[t.e];
    // stages of KB k-blocks; the segment is 128-row aligned and zero past its
    // rows, so a last stage reaching past the rows reads zeros of the segment
    t.kblocks = (s_cnt[t.e] + BK * ModeCfg<MODE>::KB - 1) / (BK * ModeCfg<MODE>::KB);
  } else {
    // expert e owns tiles [s_pair[e] * nt, s_pair[e + 1] * nt); inside it the
    // column blocks run fastest, so the CTAs working at one time share a few
    // row pairs of A (read from DRAM once) and the expert's whole weight panel,
    // which stays in L2 while the row pairs advance.  (With row pairs fastest,
    // an expert of tens of thousands of rows spreads the concurrent tiles over
    // more A rows than L2 holds, and A is read again for every column block.)
    const int nt = n_tiles_of<MODE>(a);
    const int q = tile / nt;
    int lo = 0, hi = a.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pair[mid] <= q) lo = mid;
      else hi = mid - 1;
    }
    t.e = lo;
    const int l = tile - s_pair[t.e] * nt;
    t.n0 = (l % nt) * (MODE == M_UP ? 128 : BN);
    const int local = 2 * (l / nt) + (int)rank;
    t.valid = local < (s_off[t.e + 1] - s_off[t.e]) / BM;
    t.row0 = (int64_t)s_off[t.e] + (int64_t)local * BM;
    const int K = (MODE == M_UP || is_dgrad_h(MODE)) ? a.d : ((MODE == M_DOWN || MODE == M_DOWN_COMB) ? a.f : 2 * a.f);
    t.kblocks = K / (BK * ModeCfg<MODE>::KB);
  }
  return t;
}

// This CTA's half of one stage: its 128 rows of A and its 128 columns of B.
// bar is the first CTA's full barrier (a shared::cluster address in the second).
template <int MODE>
__device__ __forceinline__ void issue_stage(const TcMaps& maps, const TcArgs& a, const Tile& t, int kb, uint32_t sA,
                                            uint32_t sB, uint32_t bar, uint32_t rank) {
  auto ld = [&](uint32_t dst, const CUtensorMap* m, int c0, int c1) {
    if (rank == 0) tma_load_2d(dst, m, bar, c0, c1);
    else tma_load_2d_pair(dst, m, bar, c0, c1);
  };
  const int r0 = static_cast<int>(t.row0);
  const int nh = (int)rank * BNH;  // this CTA's B columns start here
  if (MODE == M_UP) {
    // B = [W1 columns n0.. | W3 columns n0..]: the first CTA stages the W1 half
    ld(sA, &maps.m[0], kb * BK, r0);
    const CUtensorMap* bm = rank == 0 ? &maps.m[1] : &maps.m[2];
    const int wr = t.e * a.d + kb * BK;
    ld(sB, bm, t.n0, wr);
    ld(sB + 8192, bm, t.n0 + 64, wr);
  } else if (MODE == M_DOWN || MODE == M_DOWN_COMB) {
    ld(sA, &maps.m[0], kb * BK, r0);
    const int wr = t.e * a.f + kb * BK;
    ld(sB, &maps.m[1], t.n0 + nh, wr);
    ld(sB + 8192, &maps.m[1], t.n0 + nh + 64, wr);
  } else if (is_dgrad_h(MODE)) {
    ld(sA, &maps.m[0], kb * BK, r0);
    ld(sB, &maps.m[1], kb * BK, t.e * a.f + t.n0 + nh);
  } else if (MODE == M_DGRAD_X) {
    const int kf = a.f / BK;
    if (kb < kf) {
      ld(sA, &maps.m[0], kb * BK, r0);
      ld(sB, &maps.m[2], kb * BK, t.e * a.d + t.n0 + nh);
    } else {
      ld(sA, &maps.m[1], (kb - kf) * BK, r0);
      ld(sB, &maps.m[3], (kb - kf) * BK, t.e * a.d + t.n0 + nh);
    }
  } else {  // WGRAD
    const CUtensorMap* am = t.sub == 2 ? &maps.m[1] : &maps.m[0];
    const CUtensorMap* bm = t.sub == 0 ? &maps.m[2] : (t.sub == 1 ? &maps.m[3] : &maps.m[4]);
    const int kr = r0 + kb * BK;
    ld(sA, am, t.m0, kr);
    ld(sA + 8192, am, t.m0 + 64, kr);
    ld(sB, bm, t.n0 + nh, kr);
    ld(sB + 8192, bm, t.n0 + nh + 64, kr);
  }
}

// ------------------------------ epilogues --------------------------------- //
// Each epilogue warp owns TMEM lanes q*32 .. q*32+31 (rows of the tile) and a
// private staging area in shared memory.  It moves 32-column slices out of
// TMEM with tcgen05.ld, applies the fused math, writes the result into a
// swizzled box and lets the TMA store it (or add it, for accumulated fp32
// gradients); two boxes alternate so the next box is filled while the
// previous one drains.
struct EpiState {
  uint32_t nbox;     // boxes this warp has staged so far (selects the buffer)
  uint32_t uses[4];  // completed waits on the input barriers of the four buffers
  bool pending[4];   // an input load is in flight into buffer h
};

// Stage and store one bf16 output box of 64 columns taken from 2 TMEM slices.
__device__ __forceinline__ void stage_wait(int lane) {
  if (lane == 0) bulk_wait_read1();
  __syncwarp();
}
// bf16 results go out with an L2 evict-first policy (they are read back only by
// a later kernel, after far more data has passed through L2), which keeps the
// operand panels and weights in L2 a little longer (4-micro-batch E=16 step
// -0.4 %, 0.3 GB less DRAM traffic a dropless E=32 step); wgrad's fp32 gradient
// boxes use the default policy (evict-first there was slower)
__device__ __forceinline__ void box_issue_store(const CUtensorMap* map, uint32_t buf, int c0, int c1, int lane,
                                                bool first = true) {
  fence_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (first) tma_store_2d_hint(map, buf, c0, c1, l2_evict_first_policy());
    else tma_store_2d(map, buf, c0, c1);
    bulk_commit();
  }
}

template <int MODE>
__device__ __forceinline__ bool epilogue_tile(const TcMaps& maps, const TcArgs& a, const Tile& t, uint32_t tacc,
                                              int q, int lane, uint32_t ebuf, uint32_t lbar, EpiState& es,
                                              uint32_t tfull, uint32_t tfull_parity, volatile int* abort_flag) {
  if (!t.valid) {  // rows outside the expert: nothing to store
    if (!mbar_wait(tfull, tfull_parity, abort_flag, a.err, 400 + MODE)) return false;
    tc_fence_after();
    return true;
  }
  const int row0 = static_cast<int>(t.row0) + q * 32;
  if (is_dgrad_h(MODE)) {
    // fetch the first a/b boxes of the tile while its mainloop still runs
    const uint32_t h = ModeCfg<MODE>::ABUFS == 2 ? (es.nbox & 1) : 0;
    if (lane == 0) {
      bulk_wait_read0();
      const uint32_t bar = lbar + 8 * h;
      mbar_expect_tx(bar, 2 * BOX_BYTES);
      tma_load_2d(ebuf + h * 2 * BOX_BYTES, &maps.m[2], bar, t.n0, row0);
      tma_load_2d(ebuf + h * 2 * BOX_BYTES + BOX_BYTES, &maps.m[3], bar, t.n0, row0);
    }
    es.pending[h] = true;
    __syncwarp();
  }
  // wgrad accumulating into the fp32 gradient: fetch the first box of old
  // values while the mainloop still runs (read, add and store back below)
  constexpr int WG_BUFS = ModeCfg<MODE>::WBUFS, WG_AHEAD = ModeCfg<MODE>::WAHEAD;
  const bool wg_add = is_wgrad(MODE) && a.accumulate && t.kblocks > 0;
  const int wg_rows = is_wgrad(MODE) ? (t.sub == 2 ? a.f : a.d) : 0;
  const CUtensorMap* wg_map = &maps.m[is_wgrad(MODE) ? 5 + t.sub : 0];
  const int wg_orow = t.e * wg_rows + t.m0 + q * 32;
  if (wg_add) {
    // boxes 0 and 1 of the tile: their buffers were last read by the stores of
    // boxes nbox-4 and nbox-3, older than the two latest stores
    // their buffers were last read by the stores of boxes nbox + c - WG_BUFS,
    // older than the WG_BUFS - WG_AHEAD latest stores
    if (lane == 0) {
      if (WG_BUFS - WG_AHEAD >= 2) bulk_wait_read2();
      else bulk_wait_read1();
    }
#pragma unroll
    for (int c = 0; c < WG_AHEAD; ++c) {
      const uint32_t h = (es.nbox + c) % WG_BUFS;
      if (lane == 0) {
        const uint32_t bar = lbar + 8 * h;
        mbar_expect_tx(bar, BOX_BYTES);
        tma_load_2d(ebuf + h * BOX_BYTES, wg_map, bar, t.n0 + c * 32, wg_orow);
      }
      es.pending[h] = true;
    }
    __syncwarp();
  }
  // dgrad x with the router term of the kept rows: each lane's row gets
  // dl[token, e] * W_r[columns, e] added before rounding (e = the tile's expert);
  // the token's dl and the tile's W_r values are fetched while the mainloop runs
  const bool rfuse = MODE == M_DGRAD_X && a.rdl != nullptr;
  float rg = 0.f;
  float rw[8];
#pragma unroll
  for (int sl = 0; sl < 8; ++sl) rw[sl] = 0.f;
  if (rfuse) {
    const int tok = a.src_token[(int64_t)row0 + lane];
    rg = tok >= 0 ? a.rdl[(int64_t)tok * a.rE + t.e] : 0.f;
#pragma unroll
    for (int sl = 0; sl < 8; ++sl) rw[sl] = a.rwr[(int64_t)(t.n0 + sl * 32 + lane) * a.rE + t.e];
  }
  if (!mbar_wait(tfull, tfull_parity, abort_flag, a.err, 400 + MODE)) return false;
  tc_fence_after();

  if (MODE == M_UP) {
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {  // h = silu(a) * b, 64 columns per box
      const uint32_t buf = ebuf + (es.nbox & 1) * BOX_BYTES;
      stage_wait(lane);
#pragma unroll 1
      for (int s = 0; s < 2; ++s) {
        uint32_t ra[32], rb[32];
        tmem_ld32(tacc + c * 64 + s * 32, ra);
        tmem_ld32(tacc + 128 + c * 64 + s * 32, rb);
        tmem_ld_wait(ra);
        reg_fence(rb);
        float hv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) hv[i] = silu_f(__uint_as_float(ra[i])) * __uint_as_float(rb[i]);
        box_put_bf16x32(buf, lane, 4 * s, hv);
      }
      box_issue_store(&maps.m[3], buf, t.n0 + c * 64, row0, lane);
      ++es.nbox;
    }
#pragma unroll 1
    for (int which = 0; which < 2; ++which) {  // a and b themselves, kept for the backward
      if ((which == 0 ? a.o1 : a.o2) == nullptr) continue;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        const uint32_t buf = ebuf + (es.nbox & 1) * BOX_BYTES;
        stage_wait(lane);
#pragma unroll 1
        for (int s = 0; s < 2; ++s) {
          uint32_t r[32];
          tmem_ld32(tacc + which * 128 + c * 64 + s * 32, r);
          tmem_ld_wait(r);
          float v[32];
          regs_to_f32(r, v);
          box_put_bf16x32(buf, lane, 4 * s, v);
        }
        box_issue_store(&maps.m[4 + which], buf, t.n0 + c * 64, row0, lane);
        ++es.nbox;
      }
    }
  } else if (MODE == M_DOWN_COMB) {
    // each lane owns one row: scale it by its gate and add it into its token's
    // row of y, 16 bytes (eight bf16) per reduction.  A token has at most two
    // kept rows, and two additions onto a zero commute, so y does not depend
    // on which of its rows lands first.
    const int64_t row = (int64_t)row0 + lane;
    const int tok = row < a.max_rows ? a.src_token[row] : -1;
    const float g = tok >= 0 ? a.row_gate[row] : 0.f;
    __nv_bfloat16* yrow = a.y + (int64_t)(tok >= 0 ? tok : 0) * a.d + t.n0;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      uint32_t r[32];
      tmem_ld32(tacc + c * 32, r);
      tmem_ld_wait(r);
      if (tok >= 0) {
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          float w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) w[i] = g * __uint_as_float(r[8 * q8 + i]);
          const uint4 v = pack(w);
          asm volatile("red.global.add.noftz.v4.bf16x2 [%0], {%1, %2, %3, %4};" ::"l"(yrow + c * 32 + q8 * 8),
                       "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                       : "memory");
        }
      }
    }
  } else if (MODE == M_DOWN || MODE == M_DGRAD_X) {
    const CUtensorMap* om = MODE == M_DOWN ? &maps.m[2] : &maps.m[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t buf = ebuf + (es.nbox & 1) * BOX_BYTES;
      stage_wait(lane);
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        uint32_t r[32];
        tmem_ld32(tacc + c * 64 + s * 32, r);
        tmem_ld_wait(r);
        float v[32];
        regs_to_f32(r, v);
        if (rfuse) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = fmaf(rg, __shfl_sync(0xffffffffu, rw[c * 2 + s], i), v[i]);
        }
        box_put_bf16x32(buf, lane, 4 * s, v);
      }
      box_issue_store(om, buf, t.n0 + c * 64, row0, lane);
      ++es.nbox;
    }
  } else if (is_dgrad_h(MODE)) {
    constexpr bool DOUBLE = ModeCfg<MODE>::ABUFS == 2;
    float dot = 0.f;  // this lane's row: sum of dH * h over the tile's columns
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const uint32_t h = DOUBLE ? ((es.nbox + c) & 1) : 0u;
      const uint32_t buf = ebuf + h * 2 * BOX_BYTES;  // [a box | b box], overwritten with [da | db]
      if (DOUBLE && c + 1 < 4) {
        const uint32_t hn = h ^ 1u;
        if (lane == 0) {
          bulk_wait_read0();  // the stores that last used buffer hn have read it
          const uint32_t bar = lbar + 8 * hn;
          mbar_expect_tx(bar, 2 * BOX_BYTES);
          tma_load_2d(ebuf + hn * 2 * BOX_BYTES, &maps.m[2], bar, t.n0 + (c + 1) * 64, row0);
          tma_load_2d(ebuf + hn * 2 * BOX_BYTES + BOX_BYTES, &maps.m[3], bar, t.n0 + (c + 1) * 64, row0);
        }
        es.pending[hn] = true;
      }
      if (!mbar_wait(lbar + 8 * h, es.uses[h] & 1u, abort_flag, a.err, 500)) return false;
      ++es.uses[h];
      es.pending[h] = false;
      uint32_t r0[32], r1[32];
      tmem_ld32(tacc + c * 64, r0);
      tmem_ld32(tacc + c * 64 + 32, r1);
      tmem_ld_wait(r0);
      reg_fence(r1);
#pragma unroll 1
      for (int s = 0; s < 2; ++s) {
        float av[32], bv[32], dav[32], dbv[32];
        box_get_bf16x32(buf, lane, 4 * s, av);
        box_get_bf16x32(buf + BOX_BYTES, lane, 4 * s, bv);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float dh = __uint_as_float(s == 0 ? r0[i] : r1[i]);
          const float sg = sigmoid_f(av[i]);
          dav[i] = dh * bv[i] * sg * (1.f + av[i] * (1.f - sg));
          dbv[i] = dh * av[i] * sg;
        }
        if (a.sdot != nullptr) {
#pragma unroll
          for (int i = 0; i < 32; ++i) dot = fmaf(dbv[i], bv[i], dot);  // dH * silu(a) * b
        }
        box_put_bf16x32(buf, lane, 4 * s, dav);
        box_put_bf16x32(buf + BOX_BYTES, lane, 4 * s, dbv);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d_hint(&maps.m[4], buf, t.n0 + c * 64, row0, l2_evict_first_policy());
        tma_store_2d_hint(&maps.m[5], buf + BOX_BYTES, t.n0 + c * 64, row0, l2_evict_first_policy());
        bulk_commit();
      }
      if (!DOUBLE && c + 1 < 4) {
        // one buffer: the next chunk's a and b once da and db have been read out
        if (lane == 0) {
          bulk_wait_read0();
          mbar_expect_tx(lbar, 2 * BOX_BYTES);
          tma_load_2d(buf, &maps.m[2], lbar, t.n0 + (c + 1) * 64, row0);
          tma_load_2d(buf + BOX_BYTES, &maps.m[3], lbar, t.n0 + (c + 1) * 64, row0);
        }
        es.pending[0] = true;
        __syncwarp();
      }
    }
    es.nbox += 4;
    if (a.sdot != nullptr) a.sdot[(int64_t)(row0 + lane) * (a.f / BN) + t.n0 / BN] = dot;
  } else if (wg_add) {  // WGRAD, accumulate: dW += acc via TMA load, add, TMA store
    // WG_BUFS buffers per warp; the old values of box c + WG_AHEAD are
    // requested while box c is added, so WG_AHEAD loads are in flight behind
    // the one being used
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      const uint32_t g = es.nbox + c;
      const uint32_t h = g % WG_BUFS;
      if (c + WG_AHEAD < 8) {
        const uint32_t hn = (g + WG_AHEAD) % WG_BUFS;
        if (lane == 0) {
          // buffer hn was last read by the store of box c + WG_AHEAD - WG_BUFS:
          // at most WG_BUFS - WG_AHEAD - 1 newer stores may still be reading
          if (WG_BUFS - WG_AHEAD - 1 >= 1) bulk_wait_read1();
          else bulk_wait_read0();
          const uint32_t bar = lbar + 8 * hn;
          mbar_expect_tx(bar, BOX_BYTES);
          tma_load_2d(ebuf + hn * BOX_BYTES, wg_map, bar, t.n0 + (c + WG_AHEAD) * 32, wg_orow);
        }
        es.pending[hn] = true;
      }
      uint32_t r[32];
      tmem_ld32(tacc + c * 32, r);
      tmem_ld_wait(r);
      if (!mbar_wait(lbar + 8 * h, es.uses[h] & 1u, abort_flag, a.err, 501)) return false;
      ++es.uses[h];
      es.pending[h] = false;
      const uint32_t buf = ebuf + h * BOX_BYTES;
      float old[32], v[32];
      box_get_f32x32(buf, lane, old);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = old[i] + __uint_as_float(r[i]);
      box_put_f32x32(buf, lane, v);
      box_issue_store(wg_map, buf, t.n0 + c * 32, wg_orow, lane, false);
    }
    es.nbox += 8;
  } else {  // WGRAD, overwrite (or an expert with no rows and accumulate = 0)
    if (t.kblocks == 0 && a.accumulate) return true;
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      const uint32_t buf = ebuf + (es.nbox & 1) * BOX_BYTES;
      stage_wait(lane);
      float v[32];
      if (t.kblocks > 0) {
        uint32_t r[32];
        tmem_ld32(tacc + c * 32, r);
        tmem_ld_wait(r);
        regs_to_f32(r, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
      }
      box_put_f32x32(buf, lane, v);
      box_issue_store(wg_map, buf, t.n0 + c * 32, wg_orow, lane, false);
      ++es.nbox;
    }
  }
  return true;
}

// ------------------------------ the kernel -------------------------------- //
template <int MODE>
__global__ void __launch_bounds__(THREADS, 1) tc_gemm_kernel(const __grid_constant__ TcMaps maps,
                                                             const __grid_constant__ TcArgs a) {
  using Cfg = ModeCfg<MODE>;
  constexpr int NST = Cfg::NST;
  extern __shared__ uint8_t smem_raw[];
  // the same offsets in both CTAs of the pair: the MMA reads both at these addresses
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ctrl = smem + Cfg::CTRL_OFF;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(ctrl);  // [MAX_ST] (used in the first CTA)
  uint64_t* empty_bar = full_bar + MAX_ST;                  // [MAX_ST]
  uint64_t* tfull_bar = empty_bar + MAX_ST;                 // [2]
  uint64_t* tempty_bar = tfull_bar + 2;                     // [2] (used in the first CTA)
  uint64_t* drain_bar = tempty_bar + 2;                     // [1]
  uint64_t* load_bar = drain_bar + 1;                       // [EPI_WARPS][4] (dgrad h, wgrad inputs)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(load_bar + 4 * EPI_WARPS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_total = reinterpret_cast<int*>(tmem_slot + 2);
  int* s_interleave = reinterpret_cast<int*>(tmem_slot + 3);
  int* s_off = reinterpret_cast<int*>(ctrl + 320);  // E + 1 ints
  int* s_cnt = s_off + MAX_E + 1;                   // E ints
  int* s_pair = s_cnt + MAX_E;                      // E + 1 ints

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs of the pair
  const int pair = blockIdx.x / 2, npairs = gridDim.x / 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(smem_addr(&full_bar[i]), 1);
      mbar_init(smem_addr(&empty_bar[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&tfull_bar[i]), 1);
      mbar_init(smem_addr(&tempty_bar[i]), 2 * EPI_WARPS);
    }
    mbar_init(smem_addr(drain_bar), 1);
    for (int i = 0; i < 4 * EPI_WARPS; ++i) mbar_init(smem_addr(&load_bar[i]), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_enter();  // no global memory or TMEM access above this line
  for (int i = threadIdx.x; i <= a.E; i += THREADS) s_off[i] = a.offsets[i];
  for (int i = threadIdx.x; i < a.E; i += THREADS) s_cnt[i] = a.counts[i];
  __syncthreads();
  if (is_wgrad(MODE)) {
    // experts ordered by rows, most first (the rank of each expert, computed in parallel)
    for (int e = threadIdx.x; e < a.E; e += THREADS) {
      int r = 0;
      for (int o = 0; o < a.E; ++o) r += (s_cnt[o] > s_cnt[e]) || (s_cnt[o] == s_cnt[e] && o < e);
      s_pair[r] = e;
    }
    __syncthreads();
  }
  cluster_sync();  // the peer's barriers exist before any arrival crosses the pair
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both TMEM bases written
  tc_fence_after();
  if (threadIdx.x == 0) {
    // both CTAs must see one TMEM base: the MMA writes the same columns in both
    const uint32_t other = ld_shared_cluster_u32(mapa_shared(smem_addr(tmem_slot), rank ^ 1u));
    const bool same_tmem = other == *tmem_slot;
    if (!same_tmem) report_error(a.err, DEV_BAD_OFFSETS, 60 + MODE);
    // validate the routing state before trusting it for addresses
    bool ok = s_off[0] == 0 && (int64_t)s_off[a.E] <= a.max_rows && (s_off[a.E] & (BM - 1)) == 0;
    for (int e = 0; e < a.E && ok; ++e) {
      const int len = s_off[e + 1] - s_off[e];
      ok = len >= 0 && (s_off[e] & (BM - 1)) == 0 && s_cnt[e] >= 0 && s_cnt[e] <= len;
    }
    int total = 0;
    *s_interleave = 0;
    if (ok && same_tmem) {
      if (is_wgrad(MODE)) {
        total = a.E * 3 * (a.d / (2 * BM)) * (a.f / BN);
        // interleave long and short tiles only when some tiles are long (at least
        // 64 k-blocks) and the experts' rows differ at least eightfold
        const int kb_most = (s_cnt[s_pair[0]] + BK - 1) / BK, kb_least = (s_cnt[s_pair[a.E - 1]] + BK - 1) / BK;
        const bool il = kb_most >= 64 && kb_most >= 8 * (kb_least > 0 ? kb_least : 1);
        *s_interleave = il ? 1 : 0;
        if (!il)
          for (int r = 0; r < a.E; ++r) s_pair[r] = r;
      } else {
        s_pair[0] = 0;
        for (int e = 0; e < a.E; ++e) s_pair[e + 1] = s_pair[e] + ((s_off[e + 1] - s_off[e]) / BM + 1) / 2;
        total = s_pair[a.E] * n_tiles_of<MODE>(a);
      }
    } else if (!ok && blockIdx.x == 0) {
      report_error(a.err, DEV_BAD_OFFSETS, 30 + MODE);
    }
    *s_total = total;
  }
  __syncthreads();
  const int total = *s_total;
  const bool interleave = *s_interleave != 0;
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t smem_base = smem_addr(smem);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      constexpr int NLOAD = MODE == M_UP ? 3 : (MODE == M_DGRAD_X ? 4 : (is_wgrad(MODE) ? 5 : 2));
      for (int i = 0; i < NLOAD; ++i) prefetch_map(&maps.m[i]);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool alive = true;
      // one stage of tile t: its k-blocks kb * KB .. kb * KB + KB - 1
      auto load_stage = [&](const Tile& t, int kb) -> bool {
        if (!mbar_wait(smem_addr(&empty_bar[stage]), phase ^ 1u, abort_flag, a.err, 100 + MODE)) return false;
        const uint32_t fb_local = smem_addr(&full_bar[stage]);
        if (rank == 0) mbar_expect_tx(fb_local, Cfg::KB * PAIR_STAGE_BYTES);
        const uint32_t fb = rank == 0 ? fb_local : mapa_shared(fb_local, 0);
#pragma unroll
        for (int kk = 0; kk < Cfg::KB; ++kk) {
          const uint32_t sA = smem_base + stage * Cfg::STAGE + kk * STAGE_BYTES;
          issue_stage<MODE>(maps, a, t, kb * Cfg::KB + kk, sA, sA + A_BYTES, fb, rank);
        }
        ++issued;
        if (++stage == NST) {
          stage = 0;
          phase ^= 1u;
        }
        return true;
      };
      GroupIter it{0, total, 0};
      Group gr;
      int rnd = 0;
      bool in_step = is_wgrad(MODE) && interleave && a.round_ctr != nullptr;
      while (alive && next_group<MODE>(it, gr, pair, npairs, total, interleave, a, s_cnt, s_pair)) {
        // Keep the rounds of host and guest tiles in step: the tiles running
        // together share operand panels through L2 only while they walk K
        // together, and after a round that straddles experts of different sizes
        // the pairs would otherwise drift apart for the rest of the launch.
        // Every producer of the round arrives on the round's counter and waits
        // for the others.  The CTAs are normally all resident, one an SM; if a
        // wait exceeds ROUND_WAIT_NS (fewer SMs than CTAs, say) this CTA stops
        // keeping step for the rest of the launch: the barrier only orders the
        // loads, so the results do not depend on it.
        if (in_step && rnd > 0 && rnd < WG_ROUNDS) {
          atomicAdd(&a.round_ctr[rnd], 1);
          const int need = 2 * gr.members;
          const uint64_t t0 = globaltimer();
          while (*reinterpret_cast<volatile int*>(&a.round_ctr[rnd]) < need) {
            if (globaltimer() - t0 > ROUND_WAIT_NS) {
              in_step = false;
              break;
            }
            __nanosleep(128);
          }
        }
        ++rnd;
        const Tile th = decode<MODE>(gr.host, rank, a, s_off, s_cnt, s_pair);
        int hk = 0;
        for (int i = 0; i <= gr.g && alive; ++i) {
          const int hend = i < gr.g && (i + 1) * Cfg::GUEST_GAP < th.kblocks ? (i + 1) * Cfg::GUEST_GAP : th.kblocks;
          for (; hk < hend && alive; ++hk) alive = load_stage(th, hk);
          if (i < gr.g && alive) {
            const Tile tg = decode<MODE>(gr.gbase - i, rank, a, s_off, s_cnt, s_pair);
            for (int kb = 0; kb < tg.kblocks && alive; ++kb) alive = load_stage(tg, kb);
          }
        }
      }
      if (!alive) {
        // drain the copies still in flight before the CTA may exit: the first
        // CTA watches its full barriers; the second, whose copies complete on
        // the first CTA's barriers, gives its copies a bounded 20 ms
        if (rank == 0) {
          const int n = issued < NST ? issued : NST;
          int s = stage;
          uint32_t ph = phase;
          for (int i = 0; i < n; ++i) {
            if (--s < 0) {
              s = NST - 1;
              ph ^= 1u;
            }
            const uint32_t fb = smem_addr(&full_bar[s]);
            for (uint32_t it = 0; it < (1u << 24) && !mbar_try_wait(fb, ph); ++it) {
            }
          }
        } else if (issued > 0) {
          const uint64_t t0 = globaltimer();
          while (globaltimer() - t0 < 20000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (first CTA of the pair) ----------------
      constexpr bool A_MN = is_wgrad(MODE);
      constexpr bool B_MN = MODE == M_UP || MODE == M_DOWN || MODE == M_DOWN_COMB || is_wgrad(MODE);
      constexpr uint32_t IDESC = idesc_bf16(A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t par = 0u;  // bit acc: parity of the completed uses of accumulator acc
      bool alive = true;
      // wait until the epilogue has emptied accumulator acc
      auto acquire = [&](int acc) -> bool {
        if (!mbar_wait(smem_addr(&tempty_bar[acc]), ((par >> acc) & 1u) ^ 1u, abort_flag, a.err, 200 + MODE))
          return false;
        tc_fence_after();
        return true;
      };
      // the MMAs of stages kb0 .. kb1 - 1 of tile t into accumulator acc
      auto mma_stages = [&](const Tile& t, int acc, int kb0, int kb1) -> bool {
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(smem_addr(&full_bar[stage]), phase, abort_flag, a.err, 300 + MODE)) return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < Cfg::KB; ++kk) {
            const uint32_t sA = smem_base + stage * Cfg::STAGE + kk * STAGE_BYTES;
            const uint32_t sB = sA + A_BYTES;
#pragma unroll
            for (int k16 = 0; k16 < BK / 16; ++k16) {
              const uint64_t ad = A_MN ? sdesc(sA + k16 * 2048, 8192, 1024) : sdesc(sA + k16 * 32, 16, 1024);
              const uint64_t bd = B_MN ? sdesc(sB + k16 * 2048, 8192, 1024) : sdesc(sB + k16 * 32, 16, 1024);
              umma_bf16_pair(d_tmem, ad, bd, IDESC, (kb | kk | k16) != 0 ? 1u : 0u);
            }
          }
          umma_commit_pair(smem_addr(&empty_bar[stage]), 0x3);
          if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
          }
        }
        return true;
      };
      GroupIter it{0, total, 0};
      Group gr;
      for (int k = 0; alive && next_group<MODE>(it, gr, pair, npairs, total, interleave, a, s_cnt, s_pair); ++k) {
        const int ha = k & 1, ga = ha ^ 1;
        const Tile th = decode<MODE>(gr.host, rank, a, s_off, s_cnt, s_pair);
        if (!acquire(ha)) break;
        int hk = 0;
        for (int i = 0; i <= gr.g && alive; ++i) {
          const int hend = i < gr.g && (i + 1) * Cfg::GUEST_GAP < th.kblocks ? (i + 1) * Cfg::GUEST_GAP : th.kblocks;
          alive = mma_stages(th, ha, hk, hend);
          hk = hend;
          if (i < gr.g && alive) {
            const Tile tg = decode<MODE>(gr.gbase - i, rank, a, s_off, s_cnt, s_pair);
            alive = acquire(ga) && mma_stages(tg, ga, 0, tg.kblocks);
            if (alive) {
              umma_commit_pair(smem_addr(&tfull_bar[ga]), 0x3);
              par ^= 1u << ga;
            }
          }
        }
        if (!alive) break;
        umma_commit_pair(smem_addr(&tfull_bar[ha]), 0x3);
        par ^= 1u << ha;
      }
      // all MMAs of the pair complete (in both CTAs' TMEM) before TMEM is released
      if (total > 0) umma_commit_pair(smem_addr(drain_bar), 0x3);
    }
    if (lane == 0 && total > 0) {
      for (uint32_t it = 0; it < (1u << 26) && !mbar_try_wait(smem_addr(drain_bar), 0); ++it) {
      }
    }
  } else {
    // ---------------- epilogue warps 2..5 (both CTAs) ----------------
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int ew = warp - 2;
    const uint32_t ebuf = smem_base + Cfg::EPI_OFF + ew * Cfg::EPI_WARP_BYTES;
    const uint32_t lbar = smem_addr(&load_bar[4 * ew]);
    EpiState es{0u, {0u, 0u, 0u, 0u}, {false, false, false, false}};
    uint32_t par = 0u;  // bit acc: parity of the completed uses of accumulator acc
    // the epilogue of tile t from accumulator acc, which is then released to the MMA
    auto drain = [&](const Tile& t, int acc) -> bool {
      const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      if (!epilogue_tile<MODE>(maps, a, t, tacc, q, lane, ebuf, lbar, es, smem_addr(&tfull_bar[acc]),
                               (par >> acc) & 1u, abort_flag))
        return false;
      par ^= 1u << acc;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const uint32_t te = smem_addr(&tempty_bar[acc]);
        if (rank == 0) mbar_arrive(te);
        else mbar_arrive_cluster(mapa_shared(te, 0));
      }
      return true;
    };
    GroupIter it{0, total, 0};
    Group gr;
    bool ok = true;
    for (int k = 0; ok && next_group<MODE>(it, gr, pair, npairs, total, interleave, a, s_cnt, s_pair); ++k) {
      const int ha = k & 1, ga = ha ^ 1;
      for (int i = 0; i < gr.g && ok; ++i) ok = drain(decode<MODE>(gr.gbase - i, rank, a, s_off, s_cnt, s_pair), ga);
      if (ok) ok = drain(decode<MODE>(gr.host, rank, a, s_off, s_cnt, s_pair), ha);
    }
    // input loads still in flight (only after an abort), then every store
    for (int h = 0; h < 4; ++h)
      if (es.pending[h])
        for (uint32_t it = 0; it < (1u << 24) && !mbar_try_wait(lbar + 8 * h, es.uses[h] & 1u); ++it) {
        }
    if (lane == 0) bulk_wait_all();
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still touch its barriers, operands or TMEM
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// ------------------------------ host side --------------------------------- //
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_tried = false;

bool resolve_encode() {
  if (!g_encode_tried) {
    g_encode_tried = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode != nullptr;
}

// 2-D tensor map over a row-major [rows, cols] matrix, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows,
              bool fp32 = false) {
  const uint64_t es = fp32 ? 4 : 2;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * es};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
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

// Clusters of two resident at once for this kernel (one CTA per SM).
template <int MODE>
int max_pairs(cudaLaunchConfig_t cfg) {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<MODE>, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = num_sms() / 2;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

template <int MODE>
cudaError_t launch_mode(const TcMaps& maps, const TcArgs& args, int64_t pair_bound, int kind, cudaStream_t st) {
  static bool attr_done[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         ModeCfg<MODE>::SMEM);
    if (e != cudaSuccess) return e;
    attr_done[dev] = true;
  }
  if (pair_bound <= 0) return cudaSuccess;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = ModeCfg<MODE>::SMEM;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2);
  const int64_t pairs = std::min<int64_t>(pair_bound, max_pairs<MODE>(cfg));
  cfg.gridDim = dim3((unsigned)(2 * pairs));
  cfg.numAttrs = 2;
  LaunchScope ls(kind, st);
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<MODE>, maps, args);
}

}  // namespace

bool tc_driver_ready() { return resolve_encode(); }

cudaError_t tc_ffn_fwd(const Shape& s, const FfnFwdArgs& f, uint32_t* err, cudaStream_t st) {
  if (!resolve_encode()) return cudaErrorNotSupported;
  if (s.max_rows == 0) return cudaSuccess;
  const uint64_t R = (uint64_t)s.max_rows, E = (uint64_t)s.E, d = (uint64_t)s.d, ff = (uint64_t)s.f;
  TcArgs a{};
  a.counts = f.counts;
  a.offsets = f.offsets;
  a.E = s.E;
  a.d = s.d;
  a.f = s.f;
  a.max_rows = s.max_rows;
  a.err = err;
  TcMaps up{}, down{};
  bool ok = make_map(&up.m[0], f.x_perm, R, d, 64, BM) && make_map(&up.m[1], f.W1, E * d, ff, 64, 64) &&
            make_map(&up.m[2], f.W3, E * d, ff, 64, 64) && make_map(&up.m[3], f.h, R, ff, 64, 32);
  if (f.a != nullptr) ok = ok && make_map(&up.m[4], f.a, R, ff, 64, 32);
  if (f.b != nullptr) ok = ok && make_map(&up.m[5], f.b, R, ff, 64, 32);
  if (f.y_comb != nullptr)  // the down product adds into y (inference forward, k <= 2)
    ok = ok && make_map(&down.m[0], f.h, R, ff, 64, BM) && make_map(&down.m[1], f.W2, E * ff, d, 64, 64);
  else if (f.y_perm != nullptr)  // null: the up product alone (the backward's recompute)
    ok = ok && make_map(&down.m[0], f.h, R, ff, 64, BM) && make_map(&down.m[1], f.W2, E * ff, d, 64, 64) &&
         make_map(&down.m[2], f.y_perm, R, d, 64, 32);
  if (!ok) return cudaErrorInvalidValue;
  const int64_t mp = (s.max_rows / BM + s.E + 1) / 2;  // bound on pair tiles of 2 x 128 rows
  a.o0 = static_cast<__nv_bfloat16*>(f.h);
  a.o1 = static_cast<__nv_bfloat16*>(f.a);
  a.o2 = static_cast<__nv_bfloat16*>(f.b);
  cudaError_t e = launch_mode<M_UP>(up, a, mp * (s.f / 128), KK_GEMM_UP, st);
  if (e != cudaSuccess) return e;
  if (f.y_comb != nullptr) {
    a.o1 = a.o2 = nullptr;
    a.src_token = f.src_token;
    a.row_gate = f.row_gate;
    a.y = static_cast<__nv_bfloat16*>(f.y_comb);
    return launch_mode<M_DOWN_COMB>(down, a, mp * (s.d / BN), KK_GEMM_DOWN, st);
  }
  if (f.y_perm == nullptr) return e;
  a.o0 = static_cast<__nv_bfloat16*>(f.y_perm);
  a.o1 = a.o2 = nullptr;
  return launch_mode<M_DOWN>(down, a, mp * (s.d / BN), KK_GEMM_DOWN, st);
}

cudaError_t tc_ffn_bwd(const Shape& s, const FfnBwdArgs& b, uint32_t* err, cudaStream_t st) {
  if (!resolve_encode()) return cudaErrorNotSupported;
  const uint64_t E = (uint64_t)s.E, d = (uint64_t)s.d, ff = (uint64_t)s.f;
  if (s.max_rows == 0) {
    if (b.accumulate || b.part == 1) return cudaSuccess;
    cudaError_t e = cudaMemsetAsync(b.dW1, 0, E * d * ff * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(b.dW3, 0, E * d * ff * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(b.dW2, 0, E * d * ff * 4, st);
    return e;
  }
  const uint64_t R = (uint64_t)s.max_rows;
  TcArgs a{};
  a.counts = b.counts;
  a.offsets = b.offsets;
  a.E = s.E;
  a.d = s.d;
  a.f = s.f;
  a.max_rows = s.max_rows;
  a.err = err;
  a.accumulate = b.accumulate;
  TcMaps mh{}, mw{}, mx{};
  bool ok = make_map(&mh.m[0], b.dy_perm, R, d, 64, BM) && make_map(&mh.m[1], b.W2, E * ff, d, 64, BNH) &&
            make_map(&mh.m[2], b.a, R, ff, 64, 32) && make_map(&mh.m[3], b.b, R, ff, 64, 32) &&
            make_map(&mh.m[4], b.da, R, ff, 64, 32) && make_map(&mh.m[5], b.db, R, ff, 64, 32);
  ok = ok && make_map(&mw.m[0], b.x_perm, R, d, 64, 64) && make_map(&mw.m[1], b.h, R, ff, 64, 64) &&
       make_map(&mw.m[2], b.da, R, ff, 64, 64) && make_map(&mw.m[3], b.db, R, ff, 64, 64) &&
       make_map(&mw.m[4], b.dy_perm, R, d, 64, 64) && make_map(&mw.m[5], b.dW1, E * d, ff, 32, 32, true) &&
       make_map(&mw.m[6], b.dW3, E * d, ff, 32, 32, true) && make_map(&mw.m[7], b.dW2, E * ff, d, 32, 32, true);
  ok = ok && make_map(&mx.m[0], b.da, R, ff, 64, BM) && make_map(&mx.m[1], b.db, R, ff, 64, BM) &&
       make_map(&mx.m[2], b.W1, E * d, ff, 64, BNH) && make_map(&mx.m[3], b.W3, E * d, ff, 64, BNH) &&
       make_map(&mx.m[4], b.dx_perm, R, d, 64, 32);
  if (!ok) return cudaErrorInvalidValue;
  const int64_t mp = (s.max_rows / BM + s.E + 1) / 2;
  a.o0 = static_cast<__nv_bfloat16*>(b.da);
  a.o1 = static_cast<__nv_bfloat16*>(b.db);
  a.i0 = static_cast<const __nv_bfloat16*>(b.a);
  a.i1 = static_cast<const __nv_bfloat16*>(b.b);
  a.sdot = b.sdot;
  cudaError_t e = cudaSuccess;
  if (b.part != 2) {
    // long K (d >= 2048, at least 32 k-blocks a tile): the wide-stage shape
    e = s.d >= 2048 ? launch_mode<M_DGRAD_H_L>(mh, a, mp * (s.f / BN), KK_GEMM_DGRAD_H, st)
                    : launch_mode<M_DGRAD_H>(mh, a, mp * (s.f / BN), KK_GEMM_DGRAD_H, st);
    if (e != cudaSuccess || b.part == 1) return e;
  }
  a.sdot = nullptr;
  a.w0 = b.dW1;
  a.w1 = b.dW3;
  a.w2 = b.dW2;
  // long K per tile (dropless, or a capacity above 2048 rows): the wide-stage shape
  const int64_t wg_tiles = (int64_t)s.E * 3 * (s.d / (2 * BM)) * (s.f / BN);
  if (s.cap > 2048) {
    if (b.round_ctr != nullptr) {
      e = cudaMemsetAsync(b.round_ctr, 0, sizeof(int) * WG_ROUNDS, st);
      if (e != cudaSuccess) return e;
      a.round_ctr = b.round_ctr;
    }
    e = launch_mode<M_WGRAD_L>(mw, a, wg_tiles, KK_GEMM_WGRAD, st);
    a.round_ctr = nullptr;
  }
  else
    e = launch_mode<M_WGRAD>(mw, a, wg_tiles, KK_GEMM_WGRAD, st);
  if (e != cudaSuccess) return e;
  a.o0 = static_cast<__nv_bfloat16*>(b.dx_perm);
  a.o1 = nullptr;
  a.rdl = b.rdl;
  a.rwr = b.rwr;
  a.rE = s.E;
  a.src_token = b.src_token;
  return launch_mode<M_DGRAD_X>(mx, a, mp * (s.d / BN), KK_GEMM_DGRAD_X, st);
}

}  // namespace moe
