// bf16 grouped GEMMs of the expert MLP on tcgen05 tensor cores (sm_103a).
//
// The per-expert loop of the expert MLP, replaced by one grouped matmul per
// projection with SwiGLU fused in (twinkle PR "NPU EP experts forward uses
// NPU grouped matmul"), written for Blackwell:
//
//   * one persistent CTA per SM walks a static round-robin list of
//     (expert, m-tile, n-tile) tiles computed on the device from the expert
//     row offsets (no host sync, empty experts have no tiles);
//   * warp 0 issues TMA loads of 128x64 A and 256x64 B bf16 tiles (128-byte
//     swizzle) into a 4-stage shared-memory ring (the down dgrad, whose
//     epilogue stages two units per piece, has 4 stages only with its
//     control block sized for at most 192 experts, else 3);
//   * warp 1 allocates 512 tensor-memory columns (two 128x256 fp32
//     accumulators) and one thread issues tcgen05.mma (M=128, N=256, K=16);
//   * warps 2-9 (two per TMEM lane quarter, each taking half of the
//     columns) drain an accumulator with tcgen05.ld while the next tile
//     accumulates into the other one, apply the epilogue, stage bf16 in
//     shared memory and write it with TMA stores;
//   * the wgrads reduce over each expert's own rows: the last, partial k
//     block of an expert is loaded through a tensor map that zero-fills the
//     rows past the expert's end (see the wgrad tail below);
//   * gate/up, down and the gate/up dgrad also come as CTA pairs (tcgen05
//     cta_group::2, a 2-CTA cluster on one TPC, M=256 per MMA, half of the
//     B tile per CTA, 6-stage ring; an expert's last <= 128 rows as an M=128
//     half tile), chosen per call and kind from the rows per expert; the two
//     wgrads always run as pairs (their tiles cover the weight dimensions,
//     so every pair tile is full);
//   * the forward gate/up and its wgrad can also read the token matrix
//     through sorted_indices themselves (the producer warp gathers rows with
//     cp.async) instead of the permuted copy.
//
// Six kinds (KIND; + kPaired for the CTA-pair form) share the machinery:
//   FwdGateUp   act = silu(X Wg^T) * (X Wu^T)       B tile = 128 rows of Wg
//                                                   + 128 rows of Wu
//   FwdDown     expanded = act Wd^T
//   DgradDown   dA = dY Wd, then the SwiGLU backward -> dgu = (dg, du)
//   DgradGateUp dX = dg Wg + du Wu  (one K loop over [dg | du] x [Wg ; Wu])
//   WgradDown   dWd[e] = dY_e^T act_e               (K = the expert's rows)
//   WgradGateUp [dWg; dWu][e] = dgu_e^T X_e
// Forward operands are K-major.  In the backward the weight operand of the
// dgrads and both operands of the wgrads are MN-major (contiguous along the
// output dimension), which UMMA reads directly from 64-element-wide
// swizzled TMA boxes, so no transposed copy of any tensor is made.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "sched.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128, UK = 16;
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, each half of the columns
constexpr uint32_t TMEM_COLS = 512;
// Epilogue staging: each epilogue warp owns a ring of NBUF units of 32 rows x
// 32 bf16 (2 KB, 64-byte swizzle) that TMA stores copy to global memory.
constexpr uint32_t UNIT_BYTES = 32 * 64;
constexpr int kMaxStages = 8;
// control block: 4 * stages + 5 mbarriers, then the TMEM address, the abort
// flag, the tile prefix, the staged expert offsets and the scan scratch
constexpr uint32_t kHolderOff = 8 * (4 * kMaxStages + 5);
constexpr uint32_t kPrefixOff = kHolderOff + 24;
constexpr uint32_t ctrl_bytes(int max_experts) {
  return kPrefixOff + 2 * (uint32_t)(max_experts + 1) * 4 + 32 * 4;
}
// Experts a control block sized for few experts holds (kFewExperts below).
constexpr int kFewMaxExperts = 192;

enum Kind : int {
  kFwdGateUp = 0,
  kFwdDown = 1,
  kDgradDown = 2,
  kDgradGateUp = 3,
  kWgradDown = 4,
  kWgradGateUp = 5,
};
// A kernel variant is a Kind, plus kPaired for the CTA-pair form and
// kFewExperts for a control block sized for at most kFewMaxExperts experts
// (the shared memory it frees holds another pipeline stage).
constexpr int kPaired = 8;
constexpr int kFewExperts = 16;
constexpr int kind_of(int variant) { return variant & 7; }

template <int KIND>
struct Traits {
  static constexpr bool a_mn = (kind_of(KIND) == kWgradDown || kind_of(KIND) == kWgradGateUp);
  static constexpr bool b_mn = (kind_of(KIND) >= kDgradDown);
  static constexpr bool wgrad = (kind_of(KIND) == kWgradDown || kind_of(KIND) == kWgradGateUp);
  // TMA producer, MMA issuer, epilogue warps.
  static constexpr int threads = 64 + 32 * kEpiWarps;
  // UMMA N (256 for every kind; a 192-wide down-dgrad tile, which evens out
  // its waves at I = 768, measured slower because that kernel is bound by
  // its epilogue, not by idle SMs).
  static constexpr int bn = 256;
  static constexpr int pieces = bn / 32;  // 32-column epilogue pieces per tile
  static constexpr int n_per_tile = (kind_of(KIND) == kFwdGateUp) ? bn / 2 : bn;  // output columns
  // CTA pairs (cta_group::2): the two CTAs of a cluster take vertically
  // adjacent 128-row tiles of one expert and n tile and hold half of the
  // B tile each, so per SM the MMA reads and the TMA writes 32 KB of shared
  // memory per k block instead of 48 KB, which leaves room for a 6-stage
  // ring.  When at most 128 of an expert's rows are left, the pair takes
  // them as a half tile (M=128 over the pair, 64 rows per CTA), so pairs
  // cover the same rows as single CTAs.  Whether a call runs paired
  // is decided per call and kind from the rows per expert (use_pairs).
  static constexpr bool pair = (KIND & kPaired) != 0;
  static constexpr int cs = pair ? 2 : 1;  // CTAs per cluster
  static constexpr int b_rows = pair ? bn / 2 : bn;  // B rows (N) this CTA holds
  static constexpr uint32_t idesc = idesc_bf16_f32(BM * cs, bn, a_mn, b_mn);
  // a pair's half tile: M=128 over the pair, 64 A rows per CTA
  static constexpr uint32_t idesc_half = idesc_bf16_f32(BM, bn, a_mn, b_mn);
  // k-block depth and ring depth: 64-deep blocks (one 128-byte swizzle row);
  // single CTAs hold 4 stages of 48 KB (3 for the down dgrad, below), pairs
  // 6 of 32 KB.  Measured on GB300: a fourth stage beats a second staging
  // unit per epilogue warp, and for the wgrads 32-deep blocks in 8 stages (a
  // ring holding two tiles) lose more to the smaller TMA boxes than they
  // gain from overlap.
  static constexpr int bk = 64;
  // The SwiGLU-backward epilogue stages two units (dg, du) per piece: its
  // two-unit ring costs a stage unless the control block is sized for few
  // experts (4 stages and the two-unit ring then fit; measured 133.0 against
  // 143.9 us with 3 stages at T=4096 K=8 E=128 H=2048 I=768).
  static constexpr int nbuf = kind_of(KIND) == kDgradDown ? 2 : 1;
  static constexpr int max_e = (KIND & kFewExperts) ? kFewMaxExperts : kMaxExperts;
  static constexpr int stages =
      pair ? 6 : (kind_of(KIND) == kDgradDown && max_e == kMaxExperts ? 3 : 4);
  static_assert(!(pair && kind_of(KIND) == kDgradDown), "the down dgrad runs single-CTA");
  static constexpr uint32_t a_bytes = BM * bk * 2;
  static constexpr uint32_t b_bytes = b_rows * bk * 2;
  static constexpr uint32_t stage_bytes = a_bytes + b_bytes;
  static constexpr uint32_t mn_box = 64 * bk * 2;  // one 64 (M/N) x bk (K) MN-major box
  static_assert(stages <= kMaxStages, "more stages than the control block holds");
  static constexpr uint32_t staging_bytes = kEpiWarps * nbuf * UNIT_BYTES;
  static constexpr uint32_t smem_bytes = stages * stage_bytes + staging_bytes + ctrl_bytes(max_e) + 1024;
  static_assert(smem_bytes <= 232448, "more shared memory than one CTA may use");
};

struct Params {
  const int32_t* off;  // expert row offsets [E+1]; nullptr: one expert owning all N rows
  int N;        // row capacity of the token-major buffers
  int E;
  int Kd;       // reduction length of the row-tiled kinds
  int I;        // expert intermediate size
  int Nout;     // output columns
  int Mout;     // output rows per expert (wgrad)
  int n_tiles;  // tiles along the output columns
  int m_tiles;  // tiles along the output rows per expert (wgrad)
  __nv_bfloat16* out;
  __nv_bfloat16* out2;
  __nv_bfloat16* save;
  const __nv_bfloat16* aux;
  int32_t* status;
  // Permute fused into the load (forward gate/up A rows, gate/up wgrad X
  // rows): row i of the expert-major operand is row gather[i] / gk of the
  // [g_rows, g_cols] bf16 token matrix at gsrc.  nullptr: the operand is the
  // permuted buffer.
  const int32_t* gather;
  int gk;
  int g_rows;
  int g_cols;
  const uint8_t* gsrc;
};

// Stage barriers of a gathering producer: lane 0's arrival (with the byte
// count of the TMA-loaded operand) and one cp.async arrival per lane.
constexpr uint32_t kGatherArrivals = 33;

// Token row behind expert-major row i, or row 0 for rows that are never
// stored or are zeroed (past the expert's end); clamped so that a corrupt
// index cannot leave the token matrix.
__device__ __forceinline__ int gather_row(const Params& p, int i, int hi) {
  if (i >= hi) return 0;
  const int t = __ldg(p.gather + i) / p.gk;
  return (t >= 0 && t < p.g_rows) ? t : 0;
}

struct Tile {
  int e, lo, hi;  // expert and its row range
  int m0, n0;     // first output row / column of the tile
  int kblocks;    // 64-deep k blocks
  int rows;       // A rows this CTA owns: 128, or 64 in a pair's half tile
  int nw;         // UMMA N of the tile: 256, or 128 / 64 for a split last-wave tile
};

// Last-wave split (single-CTA down projection and dgrads): when the
// tiles leave a last wave that fills at most half of the persistent grid,
// each of its tiles is split along N into `split` narrower tiles (N = 128 or
// 64), so that 2x or 4x as many SMs share it.  Tile slots [0, tail0) are
// whole tiles; slot tail0 + u is part u % split of whole tile
// tail0 + u / split.
struct Waves {
  int tail0, split, slots;
};

template <int KIND>
__device__ __forceinline__ Waves plan_waves(int total, int grid) {
  Waves w{total, 1, total};
  if constexpr (kind_of(KIND) == kDgradDown || KIND == kFwdDown || KIND == kDgradGateUp) {
    const int left = total % grid;
    if (left > 0 && 2 * left <= grid) {
      w.split = 4 * left <= grid ? 4 : 2;
      w.tail0 = total - left;
      w.slots = w.tail0 + left * w.split;
    }
  }
  return w;
}

// Wgrad tail.  The wgrads reduce over an expert's token rows (k), and the
// rows after the expert's end belong to the next expert: the last, partial
// k block of an expert must read them as zero.  Both operands are loaded
// through 3-D tensor maps whose dimensions 1 and 2 both step one row
// (element (c, i, j) is row i + j, dimension 1 of extent bk): a k block at
// row r0 = lo + kb * bk with rem = hi - r0 < bk valid rows is loaded at
// (c, rem - bk, r0), so that box row q holds row r0 + q - (bk - rem), and
// its first bk - rem rows, whose dimension-1 coordinates are negative, are
// zero-filled by the TMA unit.  A and B are shifted alike, so the k sum is
// that of the expert's rows alone; the MMAs skip the leading groups of 16
// rows that are all zero.  Full blocks load at (c, 0, r0).
template <int KIND>
__device__ __forceinline__ int k_shift(const Tile& x, int kb) {
  constexpr int BK = Traits<KIND>::bk;
  const int rem = x.hi - (x.lo + kb * BK);
  return rem < BK ? BK - rem : 0;
}

// Tile t: a group of CS (1, or 2 for a pair) vertically adjacent 128-row tiles of one
// expert and one n tile; this CTA (cluster rank `rank`) takes the rank-th.
// When at most 128 rows of the expert are left, a pair takes them as a half
// tile (M=128 over the pair, 64 rows per CTA), so that pairs cover exactly
// the rows single CTAs would.  Rows past the expert's end are computed and
// never stored (their loads read the next expert's rows, or zeros past the
// buffer).
template <int KIND>
__device__ __forceinline__ Tile decode_tile(int t, const Params& p, const int32_t* prefix,
                                            const int32_t* offs, int rank) {
  constexpr int CS = Traits<KIND>::cs;
  Tile x;
  if constexpr (!Traits<KIND>::wgrad) {
    const int mg = t / p.n_tiles, nt = t - mg * p.n_tiles;
    const int e = find_expert(prefix, p.E, mg);
    const ExpertRows r = expert_rows(offs, e, p.N);
    x.e = e;
    x.lo = r.lo;
    x.hi = r.hi;
    const int g0 = r.lo + (mg - prefix[e]) * (BM * CS);  // first row of the (pair) tile
    x.rows = (CS == 2 && g0 + BM >= r.hi) ? BM / 2 : BM;
    x.m0 = g0 + rank * x.rows;
    x.n0 = nt * Traits<KIND>::n_per_tile;
    x.kblocks = p.Kd / Traits<KIND>::bk;
    x.nw = Traits<KIND>::bn;
  } else {
    const int m_groups = (p.m_tiles + CS - 1) / CS;
    const int per = m_groups * p.n_tiles;
    const int e = t / per, rem = t - e * per;
    const int mg = rem / p.n_tiles, nt = rem - mg * p.n_tiles;
    const ExpertRows r = expert_rows(offs, e, p.N);
    x.e = e;
    x.lo = r.lo;
    x.hi = r.hi;
    x.m0 = (mg * CS + rank) * BM;
    x.rows = BM;
    x.n0 = nt * Traits<KIND>::bn;
    x.kblocks = (r.hi - r.lo + Traits<KIND>::bk - 1) / Traits<KIND>::bk;
    x.nw = Traits<KIND>::bn;
  }
  return x;
}

// Tile slot t of the plan w (see Waves).
template <int KIND>
__device__ __forceinline__ Tile decode_slot(int t, const Waves& w, const Params& p,
                                            const int32_t* prefix, const int32_t* offs, int rank) {
  if (t < w.tail0) return decode_tile<KIND>(t, p, prefix, offs, rank);
  const int u = t - w.tail0;
  Tile x = decode_tile<KIND>(w.tail0 + u / w.split, p, prefix, offs, rank);
  x.nw = Traits<KIND>::bn / w.split;
  x.n0 += (u % w.split) * x.nw;
  return x;
}

// TMA loads of k block kb of tile x into one stage: this CTA's own 128 rows
// of A (64 in a pair's half tile) and its part of B: all of it for a single
// CTA, the rank-th half (128 of the 256 N rows) in a pair.  `bar` receives
// the bytes: this CTA's full barrier, or the leader's in a pair.
template <int KIND>
__device__ __forceinline__ void load_stage(const Tile& x, int kb, const Params& p, uint32_t sa,
                                           uint32_t sb, uint32_t bar, const CUtensorMap* mA,
                                           const CUtensorMap* mA64, const CUtensorMap* mB0,
                                           const CUtensorMap* mB1, int rank) {
  constexpr bool PAIR = Traits<KIND>::pair;
  constexpr int B_ROWS = Traits<KIND>::b_rows;
  constexpr uint32_t MN_BOX_BYTES = Traits<KIND>::mn_box;
  const int k0 = kb * Traits<KIND>::bk;
  auto l2 = [&](uint32_t dst, const CUtensorMap* m, int bx, int by) {
    if constexpr (PAIR) tma_load_2d_pair(dst, m, bar, bx, by);
    else tma_load_2d(dst, m, bar, bx, by);
  };
  auto l3 = [&](uint32_t dst, const CUtensorMap* m, int bx, int by, int bz) {
    if constexpr (PAIR) tma_load_3d_pair(dst, m, bar, bx, by, bz);
    else tma_load_3d(dst, m, bar, bx, by, bz);
  };
  const int nb = x.n0 + (PAIR ? rank * B_ROWS : 0);  // first B row (N) of this CTA's part
  // a pair's half tile needs only its 64 A rows
  const CUtensorMap* mAr = (PAIR && x.rows < BM) ? mA64 : mA;
  if constexpr (kind_of(KIND) == kFwdGateUp) {
    // B tile = 128 rows of W_gate, then the same 128 rows of W_up; in a pair
    // each CTA holds 64 gate rows then the same 64 up rows (its N half), so
    // that gate and up of one output column meet in one thread
    l2(sa, mAr, k0, x.m0);
    if constexpr (PAIR) {
      l3(sb, mB0, k0, x.n0 + 64 * rank, x.e);
      l3(sb + Traits<KIND>::b_bytes / 2, mB1, k0, x.n0 + 64 * rank, x.e);
    } else {
      l3(sb, mB0, k0, x.n0, x.e);
      l3(sb + Traits<KIND>::b_bytes / 2, mB1, k0, x.n0, x.e);
    }
  } else if constexpr (kind_of(KIND) == kFwdDown) {
    l2(sa, mAr, k0, x.m0);
    if (PAIR || x.nw == Traits<KIND>::bn) {
      l3(sb, mB0, k0, nb, x.e);  // B_ROWS rows of the W_down panel in one box
    } else {
      // a split tile: its rows in 64-row boxes (mB1), which stack into the
      // same swizzled layout as the whole box
#pragma unroll
      for (int j = 0; j < B_ROWS / 64; ++j)
        if (j * 64 < x.nw) l3(sb + j * 8192u, mB1, k0, nb + j * 64, x.e);
    }
  } else if constexpr (kind_of(KIND) == kDgradDown) {
    l2(sa, mAr, k0, x.m0);
#pragma unroll
    for (int j = 0; j < B_ROWS / 64; ++j)
      if (j * 64 < x.nw) l3(sb + j * MN_BOX_BYTES, mB0, nb + j * 64, k0, x.e);
  } else if constexpr (kind_of(KIND) == kDgradGateUp) {
    l2(sa, mAr, k0, x.m0);
    const bool up = k0 >= p.I;
    const int kk = up ? k0 - p.I : k0;
#pragma unroll
    for (int j = 0; j < B_ROWS / 64; ++j)
      if (j * 64 < x.nw) l3(sb + j * MN_BOX_BYTES, up ? mB1 : mB0, nb + j * 64, kk, x.e);
  } else {  // wgrad: both operands MN-major, k = token rows of the expert
    const int row = x.lo + k0;
    const int sh = k_shift<KIND>(x, kb);  // leading rows zero-filled (wgrad tail)
#pragma unroll
    for (int j = 0; j < 2; ++j) l3(sa + j * MN_BOX_BYTES, mA, x.m0 + j * 64, -sh, row);
#pragma unroll
    for (int j = 0; j < B_ROWS / 64; ++j) l3(sb + j * MN_BOX_BYTES, mB0, nb + j * 64, -sh, row);
  }
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void load_row32(const __nv_bfloat16* src, float (&f)[32]) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 v = s[q];
    f[8 * q + 0] = bf_lo(v.x);
    f[8 * q + 1] = bf_hi(v.x);
    f[8 * q + 2] = bf_lo(v.y);
    f[8 * q + 3] = bf_hi(v.y);
    f[8 * q + 4] = bf_lo(v.z);
    f[8 * q + 5] = bf_hi(v.z);
    f[8 * q + 6] = bf_lo(v.w);
    f[8 * q + 7] = bf_hi(v.w);
  }
}

// ---- epilogue ---------------------------------------------------------------
//
// Each epilogue warp owns 32 accumulator rows (its TMEM lane quarter).  It
// converts 32-column pieces to bf16 into its staging ring (lane i writes row
// i, 64-byte swizzle, so the warp's 16-byte stores hit distinct banks) and
// one lane hands each 32 x 32 unit to a TMA store, which writes whole 64-byte
// row segments.  Units that would cross the end of an expert's rows (the next
// expert's rows follow) are copied out by the lanes whose rows are valid
// instead.  Every unit commits one bulk group (an empty one for the copied
// units), so the ring is recycled by counting groups.

template <int NBUF>
struct Ring {
  uint32_t base;  // this warp's NBUF units
  int slot;       // next unit to fill
  // Next unit, once the store that last used it has read it.
  __device__ __forceinline__ uint32_t next(int lane) {
    if (lane == 0) bulk_wait_group_read<NBUF - 1>();
    __syncwarp();
    const uint32_t b = base + (uint32_t)(slot % NBUF) * UNIT_BYTES;
    ++slot;
    return b;
  }
};

__device__ __forceinline__ void pack32(const uint32_t (&v)[32], uint32_t (&w)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
}

// 64-byte swizzle: 16-byte chunk c of row r sits at chunk c ^ ((r >> 1) & 3).
__device__ __forceinline__ uint32_t unit_chunk(uint32_t buf, int r, int c) {
  return buf + (uint32_t)r * 64u + ((uint32_t)(c ^ ((r >> 1) & 3)) << 4);
}

__device__ __forceinline__ void stage_row(uint32_t buf, int lane, const uint32_t (&w)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    st_shared_v4(unit_chunk(buf, lane, j), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
}

// Hand a staged unit to TMA (all 32 rows valid) or copy this lane's row to
// `row_dst` (nullptr: row not written); then close the unit's bulk group.
template <bool k3D>
__device__ __forceinline__ void flush_unit(uint32_t buf, int lane, bool tma, const CUtensorMap* map,
                                           int x, int y, int z, __nv_bfloat16* row_dst) {
  if (tma) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if constexpr (k3D) tma_store_3d(map, buf, x, y, z);
      else tma_store_2d(map, buf, x, y);
    }
  } else {
    if (row_dst != nullptr) {
      uint4* d = reinterpret_cast<uint4*>(row_dst);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint4 v;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(unit_chunk(buf, lane, j)));
        d[j] = v;
      }
    }
    __syncwarp();
  }
  if (lane == 0) bulk_commit_group();
}

// Epilogue of one tile for one epilogue warp.  tacc: TMEM address of the
// warp's lane quarter of the accumulator; quarter: that lane quarter; half:
// which of the quarter's two warps.
template <int KIND>
__device__ __forceinline__ void epilogue(const Tile& x, const Params& p, uint32_t tacc, int quarter,
                                         int half, int lane, Ring<Traits<KIND>::nbuf>& ring,
                                         const CUtensorMap* mC0,
                                         const CUtensorMap* mC1) {
  if constexpr (!Traits<KIND>::wgrad) {
    // The 32 x 32 pieces this warp drains: piece i covers accumulator rows
    // r0.. (the warp's TMEM lane quarter), TMEM columns tc0 + 32i and output
    // columns col0 + 32i.  Single CTAs and full pair tiles hold rows 32q in
    // lane quarter q with all N columns in TMEM columns 0..N-1; a pair's half
    // tile holds the CTA's 64 rows in lanes 0-63 for the first N/2 columns
    // and again in lanes 64-127 for the last N/2, in TMEM columns 0..N/2-1.
    // Gate/up accumulators hold [gate 128 | up 128] in a single CTA and, in
    // a pair, [gate 64 | up 64] per CTA half of N (the pair's B halves
    // interleave gate and up rows), so the up column is tc + uoff.
    constexpr bool PAIR = Traits<KIND>::pair;
    const bool halft = PAIR && x.rows < BM;
    const int r0 = x.m0 + (halft ? 32 * (quarter & 1) : 32 * quarter);
    const int blk = halft ? (quarter >> 1) : 0;  // which half of N (half tiles)
    int np, tc0, col0, uoff = 0;
    if constexpr (kind_of(KIND) == kFwdGateUp) {
      if (!PAIR) {
        np = 2, tc0 = 64 * half, uoff = 128, col0 = x.n0 + 64 * half;
      } else if (!halft) {
        np = 2, tc0 = 128 * half, uoff = 64, col0 = x.n0 + 64 * half;
      } else {
        np = 1, tc0 = 32 * half, uoff = 64, col0 = x.n0 + 64 * blk + 32 * half;
      }
    } else {
      if (!halft) np = x.nw / 64, tc0 = (x.nw / 2) * half, col0 = x.n0 + (x.nw / 2) * half;
      else np = 2, tc0 = 64 * half, col0 = x.n0 + 128 * blk + 64 * half;
    }
    if (r0 >= x.hi) return;  // warp-uniform: no row of this warp is valid
    const bool full = r0 + 32 <= x.hi;
    const int row = r0 + lane;
    const bool rv = row < x.hi;
    if constexpr (kind_of(KIND) == kFwdGateUp) {
      const int I = p.Nout;
#pragma unroll 1
      for (int i = 0; i < np; ++i) {
        const int col = col0 + 32 * i, tc = tc0 + 32 * i;
        if (col >= I) break;
        uint32_t g[32], u[32], w[16];
        tmem_ld_32x32b_x32(tacc + tc, g);
        tmem_ld_32x32b_x32(tacc + tc + uoff, u);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float g0 = __uint_as_float(g[2 * j]), g1 = __uint_as_float(g[2 * j + 1]);
          const float u0 = __uint_as_float(u[2 * j]), u1 = __uint_as_float(u[2 * j + 1]);
          w[j] = pack_bf16x2(__fdividef(g0, 1.f + __expf(-g0)) * u0,
                             __fdividef(g1, 1.f + __expf(-g1)) * u1);
        }
        uint32_t b = ring.next(lane);
        stage_row(b, lane, w);
        flush_unit<false>(b, lane, full, mC0, col, r0, 0,
                          (!full && rv) ? p.out + (size_t)row * I + col : nullptr);
        if (p.save != nullptr) {
          pack32(g, w);
          b = ring.next(lane);
          stage_row(b, lane, w);
          flush_unit<false>(b, lane, full, mC1, col, r0, 0,
                            (!full && rv) ? p.save + (size_t)row * 2 * I + col : nullptr);
          pack32(u, w);
          b = ring.next(lane);
          stage_row(b, lane, w);
          flush_unit<false>(b, lane, full, mC1, I + col, r0, 0,
                            (!full && rv) ? p.save + (size_t)row * 2 * I + I + col : nullptr);
        }
      }
    } else if constexpr (kind_of(KIND) == kFwdDown || kind_of(KIND) == kDgradGateUp) {
#pragma unroll 1
      for (int i = 0; i < np; ++i) {
        const int col = col0 + 32 * i, tc = tc0 + 32 * i;
        if (col >= p.Nout) break;
        uint32_t v[32], w[16];
        tmem_ld_32x32b_x32(tacc + tc, v);
        tmem_ld_wait();
        pack32(v, w);
        const uint32_t b = ring.next(lane);
        stage_row(b, lane, w);
        flush_unit<false>(b, lane, full, mC0, col, r0, 0,
                          (!full && rv) ? p.out + (size_t)row * p.Nout + col : nullptr);
      }
    } else {  // kDgradDown
      // dA -> SwiGLU backward with the saved pre-activations (g, u):
      //   dg = dA * u * s * (1 + g (1 - s)),  du = dA * g * s,  s = sigmoid(g)
      const int I = p.I;
      const __nv_bfloat16* gu_row = p.aux + (size_t)row * 2 * I;
      // raw bf16 (g, u) of the current piece; the next piece's are loaded
      // before the current one is processed
      uint4 rg[4], ru[4];
      auto fetch = [&](int col, uint4(&a)[4], uint4(&b)[4]) {
        if (rv && col < I) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            a[q] = ld_v4(gu_row + col + 8 * q);
            b[q] = ld_v4(gu_row + I + col + 8 * q);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) a[q] = b[q] = make_uint4(0u, 0u, 0u, 0u);
        }
      };
      fetch(col0, rg, ru);
#pragma unroll 1
      for (int i = 0; i < np; ++i) {
        const int col = col0 + 32 * i, tc = tc0 + 32 * i;
        if (col >= I) break;
        uint4 ng[4], nu[4];
        fetch(i + 1 < np ? col + 32 : I, ng, nu);
        uint32_t v[32];
        tmem_ld_32x32b_x32(tacc + tc, v);
        tmem_ld_wait();
        float g[32], u[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t gw[4] = {rg[q].x, rg[q].y, rg[q].z, rg[q].w};
          const uint32_t uw[4] = {ru[q].x, ru[q].y, ru[q].z, ru[q].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            g[8 * q + 2 * k] = bf_lo(gw[k]);
            g[8 * q + 2 * k + 1] = bf_hi(gw[k]);
            u[8 * q + 2 * k] = bf_lo(uw[k]);
            u[8 * q + 2 * k + 1] = bf_hi(uw[k]);
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          rg[q] = ng[q];
          ru[q] = nu[q];
        }
        uint32_t wg[16], wu[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float dg2[2], du2[2];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int k = 2 * j + q;
            const float da = __uint_as_float(v[k]);
            const float sg = __fdividef(1.f, 1.f + __expf(-g[k]));
            dg2[q] = da * u[k] * sg * (1.f + g[k] * (1.f - sg));
            du2[q] = da * g[k] * sg;
          }
          wg[j] = pack_bf16x2(dg2[0], dg2[1]);
          wu[j] = pack_bf16x2(du2[0], du2[1]);
        }
        uint32_t b = ring.next(lane);
        stage_row(b, lane, wg);
        flush_unit<false>(b, lane, full, mC0, col, r0, 0,
                          (!full && rv) ? p.out + (size_t)row * 2 * I + col : nullptr);
        b = ring.next(lane);
        stage_row(b, lane, wu);
        flush_unit<false>(b, lane, full, mC0, I + col, r0, 0,
                          (!full && rv) ? p.out + (size_t)row * 2 * I + I + col : nullptr);
      }
    }
  } else {  // wgrad: output rows m of expert e; Mout and I are multiples of 32
    const int r0 = x.m0 + quarter * 32;
    if (r0 >= p.Mout) return;
    const CUtensorMap* map = mC0;
    int y = r0;
    if constexpr (kind_of(KIND) == kWgradGateUp) {
      if (r0 >= p.I) {
        map = mC1;
        y = r0 - p.I;
      }
    }
    const bool empty = x.kblocks == 0;  // uniform over the tile
    constexpr int HP = Traits<KIND>::pieces / 2;
#pragma unroll 1
    for (int c = HP * half; c < HP * half + HP; ++c) {
      const int col = x.n0 + c * 32;
      if (col >= p.Nout) break;
      uint32_t w[16];
      if (empty) {
#pragma unroll
        for (int j = 0; j < 16; ++j) w[j] = 0u;
      } else {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tacc + c * 32, v);
        tmem_ld_wait();
        pack32(v, w);
      }
      const uint32_t b = ring.next(lane);
      stage_row(b, lane, w);
      flush_unit<true>(b, lane, true, map, col, y, x.e, nullptr);
    }
  }
}

// Producer warp when the operand rows are gathered from the token matrix:
// all 32 lanes copy the gathered operand with 16-byte cp.async copies into
// the 128-byte-swizzled layout the TMA box loads produce (eight lanes per
// 128-byte row segment, so the reads are coalesced; chunk c of row r lands in
// chunk c ^ (r & 7)), then arrive on the stage's full barrier when their
// copies have landed; lane 0 arms the barrier with the byte count of the
// other operand and loads it with TMA.  Forward gate/up: the 128 A rows of a
// tile (row indices read once per tile).  Gate/up wgrad: the 64 X rows (k)
// of a k block in each of the four 64-column B boxes (the next block's row
// indices read before waiting for its stage), shifted like the TMA-loaded
// dgu rows of an expert's last block (the wgrad tail above), the leading
// rows zero-filled.  Single-CTA kinds only.  (A
// tile::gather4 TMA form of the same loads was correct but measured 2.4x
// slower for the forward and 5x for the wgrad on GB300: it moves 512 bytes
// per instruction and the TMA unit takes ~40 ns per gather.)
template <int KIND>
__device__ __forceinline__ void produce_gathered(const Params& p, const int32_t* prefix,
                                                 const int32_t* offs, int total, int t_first,
                                                 int t_step, int lane, uint32_t sA, uint32_t sB,
                                                 uint32_t ctrl, volatile int* abort_flag,
                                                 const CUtensorMap* mA, const CUtensorMap* mB0,
                                                 const CUtensorMap* mB1) {
  constexpr int STAGES = Traits<KIND>::stages;
  constexpr uint32_t A_BYTES = Traits<KIND>::a_bytes;
  constexpr uint32_t B_BYTES = Traits<KIND>::b_bytes;
  constexpr uint32_t MN_BOX_BYTES = Traits<KIND>::mn_box;
  constexpr int BK = Traits<KIND>::bk;
  static_assert(!Traits<KIND>::pair, "gathered operands are single-CTA");
  auto full_bar = [&](int s) { return ctrl + 8u * s; };
  auto empty_bar = [&](int s) { return ctrl + 8u * (STAGES + s); };
  const int c = lane & 7, r0 = lane >> 3;  // 16-byte chunk and first row of this lane
  const size_t ld = (size_t)p.g_cols * 2;  // token row bytes
  auto swz = [&](int row) { return (uint32_t)row * 128u + ((uint32_t)(c ^ (row & 7)) << 4); };
  int issued[kMaxStages];
#pragma unroll
  for (int s = 0; s < STAGES; ++s) issued[s] = -1;
  int g = 0;
  bool run = true;
  if constexpr (kind_of(KIND) == kFwdGateUp) {
    for (int t = t_first; run && t < total; t += t_step) {
      const Tile x = decode_tile<KIND>(t, p, prefix, offs, 0);
      int tok[BM / 4];  // token rows of tile rows r0 + 4j
#pragma unroll
      for (int j = 0; j < BM / 4; ++j) tok[j] = gather_row(p, x.m0 + r0 + 4 * j, x.hi);
      for (int kb = 0; kb < x.kblocks; ++kb, ++g) {
        const int s = g % STAGES;
        const uint32_t ph = (g / STAGES) & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, p.status))) {
          run = false;
          break;
        }
        const int k0 = kb * BK;
        const uint32_t sa = sA + s * A_BYTES, sb = sB + s * B_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(full_bar(s), B_BYTES);
          tma_load_3d(sb, mB0, full_bar(s), k0, x.n0, x.e);
          tma_load_3d(sb + B_BYTES / 2, mB1, full_bar(s), k0, x.n0, x.e);
          issued[s] = (int)ph;
        }
        const uint8_t* col = p.gsrc + (size_t)k0 * 2 + (size_t)c * 16;
#pragma unroll
        for (int j = 0; j < BM / 4; ++j) cp_async_16(sa + swz(r0 + 4 * j), col + (size_t)tok[j] * ld, 16);
        cp_async_arrive(full_bar(s));
      }
    }
  } else {
    static_assert(kind_of(KIND) == kWgradGateUp, "gathers serve the gate/up GEMMs");
    // the (tile, k block) position the producer fills next, skipping tiles
    // without rows (they have no k blocks)
    int t = t_first, kb = 0;
    Tile x{};
    auto next_tile = [&]() {
      for (; t < total; t += t_step) {
        x = decode_tile<KIND>(t, p, prefix, offs, 0);
        if (x.kblocks > 0) return true;
      }
      return false;
    };
    bool have = next_tile();
    int tok[BK / 4];  // token rows of box rows r0 + 4j of the block (-1: zero row)
    auto load_rows = [&]() {
      const int sh = k_shift<KIND>(x, kb);
      const int base = x.lo + kb * BK + r0 - sh;
#pragma unroll
      for (int j = 0; j < BK / 4; ++j)
        tok[j] = r0 + 4 * j < sh ? -1 : gather_row(p, base + 4 * j, x.hi);
    };
    if (have) load_rows();
    while (have) {
      const int s = g % STAGES;
      const uint32_t ph = (g / STAGES) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, p.status))) break;
      const uint32_t sa = sA + s * A_BYTES, sb = sB + s * B_BYTES;
      const int row = x.lo + kb * BK;
      if (lane == 0) {
        mbar_arrive_expect_tx(full_bar(s), A_BYTES);
        const int sh = k_shift<KIND>(x, kb);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tma_load_3d(sa + j * MN_BOX_BYTES, mA, full_bar(s), x.m0 + j * 64, -sh, row);
        issued[s] = (int)ph;
      }
#pragma unroll
      for (int box = 0; box < Traits<KIND>::b_rows / 64; ++box) {
        const int colx = x.n0 + box * 64 + c * 8;  // columns past H are zero-filled
        const bool in_cols = colx < p.g_cols;
#pragma unroll
        for (int j = 0; j < BK / 4; ++j) {
          const uint32_t bytes = (in_cols && tok[j] >= 0) ? 16u : 0u;
          const uint8_t* src = bytes ? p.gsrc + (size_t)colx * 2 + (size_t)tok[j] * ld : p.gsrc;
          cp_async_16(sb + box * MN_BOX_BYTES + swz(r0 + 4 * j), src, bytes);
        }
      }
      cp_async_arrive(full_bar(s));
      ++g;
      if (++kb == x.kblocks) {
        kb = 0;
        t += t_step;
        have = next_tile();
      }
      if (have) load_rows();  // in flight while the next stage is awaited
    }
  }
  // wait for every copy issued before the CTA may exit (the full barriers
  // count the lanes' cp.async arrivals too)
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s)
      if (issued[s] >= 0) mbar_wait(full_bar(s), (uint32_t)issued[s], abort_flag, p.status, false);
  }
  __syncwarp();
  (void)mA;
}

template <int KIND>
__global__ void __launch_bounds__(Traits<KIND>::threads, 1)
gmm_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapA64,
              const __grid_constant__ CUtensorMap mapB0,
              const __grid_constant__ CUtensorMap mapB1, const __grid_constant__ CUtensorMap mapC0,
              const __grid_constant__ CUtensorMap mapC1, const Params p) {
  constexpr int STAGES = Traits<KIND>::stages;
  constexpr int NBUF = Traits<KIND>::nbuf;
  constexpr int CS = Traits<KIND>::cs;
  constexpr bool PAIR = Traits<KIND>::pair;
  constexpr int BK = Traits<KIND>::bk;
  constexpr uint32_t A_BYTES = Traits<KIND>::a_bytes;
  constexpr uint32_t B_BYTES = Traits<KIND>::b_bytes;
  constexpr uint32_t STAGE_BYTES = Traits<KIND>::stage_bytes;
  constexpr uint32_t MN_BOX_BYTES = Traits<KIND>::mn_box;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + STAGES * A_BYTES;
  const uint32_t staging = base + STAGES * STAGE_BYTES;
  const uint32_t ctrl = staging + Traits<KIND>::staging_bytes;
  uint8_t* gctrl = gbase + STAGES * STAGE_BYTES + Traits<KIND>::staging_bytes;
  auto full_bar = [&](int s) { return ctrl + 8u * s; };
  auto empty_bar = [&](int s) { return ctrl + 8u * (STAGES + s); };
  auto tfull_bar = [&](int a) { return ctrl + 8u * (2 * STAGES + a); };
  auto tempty_bar = [&](int a) { return ctrl + 8u * (2 * STAGES + 2 + a); };
  const uint32_t drain_bar = ctrl + 8u * (2 * STAGES + 4);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(gctrl + kHolderOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gctrl + kHolderOff + 4);
  int32_t* prefix = reinterpret_cast<int32_t*>(gctrl + kPrefixOff);
  int32_t* offs = prefix + (Traits<KIND>::max_e + 1);  // expert offsets, staged once per CTA
  int32_t* scratch = offs + (Traits<KIND>::max_e + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // operand rows gathered from the token matrix by the producer's cp.async
  bool gathered = false;
  if constexpr ((kind_of(KIND) == kFwdGateUp || kind_of(KIND) == kWgradGateUp) && !PAIR)
    gathered = p.gather != nullptr;
  if (threadIdx.x == 0) {
    // In a pair the leader's full barriers count both CTAs' bytes, the
    // leader's MMA commits release the stages and accumulators of both CTAs,
    // and the leader's tempty barriers take one arrival per epilogue warp of
    // both CTAs.
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), gathered ? kGatherArrivals : 1u);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), PAIR ? 2 * kEpiWarps : kEpiWarps * 32);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    if constexpr (PAIR) tma_prefetch_desc(&mapA64);
    tma_prefetch_desc(&mapB0);
    tma_prefetch_desc(&mapB1);
    tma_prefetch_desc(&mapC0);
    tma_prefetch_desc(&mapC1);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_holder), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
      tmem_relinquish();
    }
  }
  // Every role decodes every tile; the offsets are read from global memory
  // once here (sanitised) instead of once per tile and role.
  stage_offsets(p.off, p.E, p.N, offs, scratch);
  int total;
  if constexpr (Traits<KIND>::wgrad) {
    total = p.E * ((p.m_tiles + CS - 1) / CS) * p.n_tiles;
  } else {
    build_tile_prefix(offs, p.E, p.N, BM * CS, prefix, scratch);  // ends with __syncthreads
    total = prefix[p.E] * p.n_tiles;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // The peer's loads, commits and arrivals target this CTA's barriers: they
  // must all be initialised cluster-wide first.
  if constexpr (CS > 1) cluster_sync_all();
  const int rank = CS > 1 ? (int)cluster_ctarank() : 0;
  const int t_first = CS > 1 ? (int)cluster_id_x() : (int)blockIdx.x;
  const int t_step = CS > 1 ? (int)cluster_count_x() : (int)gridDim.x;
  const Waves wv = plan_waves<KIND>(total, t_step);

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if constexpr ((kind_of(KIND) == kFwdGateUp || kind_of(KIND) == kWgradGateUp) && !PAIR) {
      if (gathered)
        produce_gathered<KIND>(p, prefix, offs, total, t_first, t_step, lane, sA, sB, ctrl,
                               abort_flag, &mapA, &mapB0, &mapB1);
    }
    if (!gathered && lane == 0) {
      int g = 0, s = 0;  // k blocks issued; stage and phase of the next
      uint32_t ph = 0;
      bool run = true;
      for (int t = t_first; run && t < wv.slots; t += t_step) {
        const Tile x = decode_slot<KIND>(t, wv, p, prefix, offs, rank);
        // Each CTA loads its A rows (64 in a half tile) and its half of B;
        // the leader's barrier counts both CTAs.  A split tile loads only
        // the B boxes of its columns.
        const uint32_t tx =
            PAIR ? 2 * (B_BYTES + (x.rows < BM ? A_BYTES / 2 : A_BYTES))
                 : A_BYTES + B_BYTES / Traits<KIND>::bn * (uint32_t)x.nw;
        for (int kb = 0; kb < x.kblocks; ++kb) {
          if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, p.status)) {
            run = false;
            break;
          }
          uint32_t fb = full_bar(s);
          if constexpr (PAIR) {
            fb = mapa_shared(full_bar(s), 0);  // the leader's barrier counts both CTAs' bytes
            if (rank == 0) mbar_arrive_expect_tx(full_bar(s), tx);
          } else {
            mbar_arrive_expect_tx(full_bar(s), tx);
          }
          load_stage<KIND>(x, kb, p, sA + s * A_BYTES, sB + s * B_BYTES, fb, &mapA, &mapA64, &mapB0, &mapB1,
                           rank);
          ++g;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // Wait for every copy issued before the CTA may exit: the last use of
      // stage st was k block st + S * floor((g - 1 - st) / S).  In a pair the
      // leader's full barriers also count the peer's copies (the peer stays
      // until the closing cluster barrier, which the leader reaches after
      // this wait).
      if (!PAIR || rank == 0) {
        for (int st = 0; st < STAGES && st < g; ++st) {
          const int last = st + (g - 1 - st) / STAGES * STAGES;
          mbar_wait(full_bar(st), (uint32_t)(last / STAGES) & 1u, abort_flag, p.status, false);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: one thread (the leader's, in a pair) ----------------
    // The tensor pipe is kept fed only if consecutive MMAs are issued with
    // few instructions between them, so one thread runs this loop alone (no
    // per-block vote or warp synchronisation), steps the stage and phase
    // instead of dividing, and forms each MMA's shared-memory descriptors
    // from per-stage bases and a constant step (the 14-bit address field
    // cannot carry: shared-memory addresses stay below 2^18 bytes).
    if ((!PAIR || rank == 0) && lane == 0) {
      constexpr uint32_t kAStep = Traits<KIND>::a_mn ? (UK * 128) >> 4 : (UK * 2) >> 4;
      constexpr uint32_t kBStep = Traits<KIND>::b_mn ? (UK * 128) >> 4 : (UK * 2) >> 4;
      const uint64_t a_desc0 = Traits<KIND>::a_mn ? desc_sw128(sA, MN_BOX_BYTES, 1024) : desc_sw128(sA, 16, 1024);
      const uint64_t b_desc0 = Traits<KIND>::b_mn ? desc_sw128(sB, MN_BOX_BYTES, 1024) : desc_sw128(sB, 16, 1024);
      int s = 0, it = 0;
      uint32_t ph = 0;
      bool run = true;
      for (int t = t_first; run && t < wv.slots; t += t_step, ++it) {
        const Tile x = decode_slot<KIND>(t, wv, p, prefix, offs, rank);
        uint32_t idesc;
        if constexpr (PAIR) idesc = x.rows < BM ? Traits<KIND>::idesc_half : Traits<KIND>::idesc;
        else idesc = x.nw == Traits<KIND>::bn ? Traits<KIND>::idesc
                                              : idesc_bf16_f32(BM, x.nw, Traits<KIND>::a_mn, Traits<KIND>::b_mn);
        const int acc = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait<PAIR>(tempty_bar(acc), aph ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t tacc = tmem_base + acc * Traits<KIND>::bn;
        uint32_t accum = 0u;  // the tile's first MMA overwrites the accumulator
        for (int kb = 0; kb < x.kblocks; ++kb) {
          if (!mbar_wait(full_bar(s), ph, abort_flag, p.status)) {
            run = false;
            break;
          }
          tc_fence_after();
          // operand rows written by the producer's cp.async (generic proxy),
          // made visible to the MMA's reads
          if (gathered) fence_proxy_async_smem();
          // the last k block of an expert in a wgrad: its leading groups of
          // 16 rows are zero-filled (see the wgrad tail) and skipped
          int kk0 = 0;
          if constexpr (Traits<KIND>::wgrad) kk0 = k_shift<KIND>(x, kb) / UK;
          const uint64_t ad = a_desc0 + (uint64_t)s * (A_BYTES >> 4);
          const uint64_t bd = b_desc0 + (uint64_t)s * (B_BYTES >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk) {
            if (kk < kk0) continue;
            if constexpr (PAIR) umma_f16_pair(tacc, ad + kk * kAStep, bd + kk * kBStep, idesc, accum);
            else umma_f16(tacc, ad + kk * kAStep, bd + kk * kBStep, idesc, accum);
            accum = 1u;
          }
          // the stage is free in both CTAs once these MMAs have read it
          if constexpr (PAIR) umma_commit_pair(empty_bar(s), 3);
          else umma_commit(empty_bar(s));
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!run) break;
        if constexpr (PAIR) umma_commit_pair(tfull_bar(acc), 3);
        else umma_commit(tfull_bar(acc));
      }
      if constexpr (PAIR) umma_commit_pair(drain_bar, 1);
      else umma_commit(drain_bar);
      mbar_wait(drain_bar, 0, abort_flag, p.status, false);
    }
  } else if (warp < 2 + kEpiWarps) {
    // ---------------- epilogue warps 2..9 ----------------
    const int quarter = warp & 3;        // TMEM lanes [32*quarter, 32*quarter + 32)
    const int half = (warp - 2) >> 2;    // which half of the tile's columns
    Ring<NBUF> ring{staging + (uint32_t)(warp - 2) * NBUF * UNIT_BYTES, 0};
    int it = 0;
    for (int t = t_first; t < wv.slots; t += t_step, ++it) {
      const Tile x = decode_slot<KIND>(t, wv, p, prefix, offs, rank);
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar(acc), aph, abort_flag, p.status))) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + acc * Traits<KIND>::bn + ((uint32_t)(quarter * 32) << 16);
      epilogue<KIND>(x, p, tacc, quarter, half, lane, ring, &mapC0, &mapC1);
      tc_fence_before();
      if constexpr (PAIR) {
        // one arrival per warp on the leader's barrier
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
      } else {
        mbar_arrive(tempty_bar(acc));
      }
    }
    // the CTA's stores must be complete before it exits
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  // No CTA leaves while its peer may still signal its barriers.
  if constexpr (CS > 1) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// A bounded wait that runs out: nothing arrives on the barrier.
__global__ void wait_selftest_kernel(int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(smem_u32(&bar), 0, &abort_flag, status);
}

// ---- host side -----------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// bf16 tensor map, 128-byte swizzle; dims innermost first, strides in bytes.
bool make_map(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims, const uint32_t* box,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gdim[3], gstride[2];
  cuuint32_t bdim[3], estr[3] = {1, 1, 1};
  uint64_t stride = 2;
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    if (i > 0) gstride[i - 1] = stride;
    stride *= dims[i];
  }
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), gdim,
                        gstride, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D view of a row-major [rows, cols] bf16 matrix whose dimensions 1 and 2
// both step one row: element (c, i, j) is row i + j, dimension 1 of extent
// bk.  The wgrad operands are loaded through it in 64 x bk boxes (128-byte
// swizzle); a box at (c, i0, j) with i0 < 0 zero-fills its first -i0 rows
// (see the wgrad tail).  The coordinates used keep every element read
// inside rows [0, rows).
bool k_rows_map(CUtensorMap* m, const void* ptr, int cols, int rows, int bk) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t row_bytes = (cuuint64_t)cols * 2;
  cuuint64_t gdim[3] = {(cuuint64_t)cols, (cuuint64_t)bk, (cuuint64_t)rows};
  cuuint64_t gstride[2] = {row_bytes, row_bytes};
  cuuint32_t bdim[3] = {64, (cuuint32_t)bk, 1}, estr[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), gdim,
                        gstride, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int KIND>
int launch(const CUtensorMap& a, const CUtensorMap& a64, const CUtensorMap& b0, const CUtensorMap& b1,
           const CUtensorMap& c0, const CUtensorMap& c1, const Params& p, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(gmm_tc_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Traits<KIND>::smem_bytes);
  });
  if (attr != cudaSuccess) return MOE_ERR_CUDA;
  constexpr int CS = Traits<KIND>::cs;
  if constexpr (CS == 1) {
    // One persistent CTA per SM.  A plain launch: the same kernel launched
    // through the cluster-attribute path (cluster size 1) measured ~20 % slower.
    gmm_tc_kernel<KIND><<<sm_count(), Traits<KIND>::threads, Traits<KIND>::smem_bytes, s>>>(a, a64, b0, b1, c0, c1, p);
    count_launches(1);
    MOE_LAUNCH_CHECK();
    return MOE_OK;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = CS;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(Traits<KIND>::threads, 1, 1);
  cfg.dynamicSmemBytes = Traits<KIND>::smem_bytes;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  // one persistent CTA per SM, as many whole clusters as can be resident
  int clusters = sm_count() / CS;
  static int resident = -1;
  if (resident < 0) {
    cfg.gridDim = dim3(clusters * CS, 1, 1);
    int n = 0;
    resident = (cudaOccupancyMaxActiveClusters(&n, gmm_tc_kernel<KIND>, &cfg) == cudaSuccess && n > 0)
                   ? n
                   : 0;
    (void)cudaGetLastError();
  }
  if (resident > 0 && resident < clusters) clusters = resident;
  cfg.gridDim = dim3(clusters * CS, 1, 1);
  if (cudaLaunchKernelEx(&cfg, gmm_tc_kernel<KIND>, a, a64, b0, b1, c0, c1, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  count_launches(1);
  return MOE_OK;
}

int device_ok() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return (major == 10 && minor == 3) ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

// Whether a GEMM runs as CTA pairs, from the rows per expert (the routing's
// skew is not known on the host without a sync).  With half tiles a pair
// covers the same rows as single CTAs; what remains is how well each kind
// uses a pair.  GB300, H=2048, bf16, us, pair / single, with the one-thread
// MMA issue and the CTA-scope accumulator release:
//   routing     rows/    gate/up            gate/up      down         gate/up
//               expert   saving (g, u)      not saving                dgrad
//   uniform       256    190.7 / 208.8      180.2 / 194.4  105.3 / 108.6  183.3 / 194.7
//   Zipf(1.2)     256    276.7 / 282.5      264.1 / 262.0  166.0 / 158.6  280.4 / 281.3
// (gate/up and its dgrad I=768 uniform, I=512 Zipf; the Zipf routing has
// experts of 22 to 7636 rows, median 72.)  Earlier measurements of the same
// kinds at 512 and 1024 rows per expert favoured pairs more strongly (for
// the down projection from 2048 rows, 531 / 569 us); the down projection
// stays single below that because at 256 rows per expert the skewed routing
// loses more (+4 %) than the uniform one gains (-3 %).  The down dgrad,
// whose SwiGLU-backward epilogue dominates, measured slower paired
// everywhere; the wgrads always run paired.
constexpr long long kPairMinRowsGateUpSave = 256;
constexpr long long kPairMinRowsGateUp = 256;
constexpr long long kPairMinRowsDown = 2048;
constexpr long long kPairMinRowsDgradGateUp = 256;
constexpr long long kPairMinRowsWgrad = 0;
inline bool use_pairs(long long min_rows, int N, int E) { return (long long)N >= min_rows * E; }

Params base_params(const int32_t* off, int N, int E, int32_t* status) {
  Params p{};
  p.off = off;
  p.N = N;
  p.E = E;
  p.status = status;
  return p;
}

}  // namespace tc

using namespace tc;

// Store maps: units of 32 columns x 32 rows (one epilogue warp's rows),
// 64-byte swizzle to match the staging layout.
bool store_map_2d(CUtensorMap* m, const void* ptr, int cols, int rows) {
  const uint64_t d[2] = {(uint64_t)cols, (uint64_t)rows};
  const uint32_t b[2] = {32, 32};
  return make_map(m, ptr, 2, d, b, CU_TENSOR_MAP_SWIZZLE_64B);
}

bool store_map_3d(CUtensorMap* m, const void* ptr, int cols, int rows, int E) {
  const uint64_t d[3] = {(uint64_t)cols, (uint64_t)rows, (uint64_t)E};
  const uint32_t b[3] = {32, 32, 1};
  return make_map(m, ptr, 3, d, b, CU_TENSOR_MAP_SWIZZLE_64B);
}

// Forward gate/up.  gather == nullptr: A is the permuted [N, H] buffer;
// otherwise A row i is row gather[i] / K of the token matrix A [T, H].
static int gate_up_bf16(const void* A, int T, const int32_t* gather, int K, const void* Wg,
                        const void* Wu, const int32_t* off, int N, int H, int I, int E, void* act,
                        void* save, int32_t* status, cudaStream_t s) {
  if (int rc = device_ok()) return rc;
  CUtensorMap ma, mg, mu;
  const uint64_t da[2] = {(uint64_t)H, (uint64_t)(gather ? T : N)};
  const uint32_t ba[2] = {64, gather ? 1u : 128u};  // (not read when gathering)
  // gathered A rows are loaded by the single-CTA producer only
  const bool paired =
      gather == nullptr &&
      use_pairs(save != nullptr ? kPairMinRowsGateUpSave : kPairMinRowsGateUp, N, E);
  const uint64_t dw[3] = {(uint64_t)H, (uint64_t)I, (uint64_t)E};
  const uint32_t bw[3] = {64, paired ? 64u : 128u, 1};  // a pair CTA: 64 gate + 64 up rows
  if (!make_map(&ma, A, 2, da, ba) || !make_map(&mg, Wg, 3, dw, bw) || !make_map(&mu, Wu, 3, dw, bw))
    return MOE_ERR_CUDA;
  Params p = base_params(off, N, E, status);
  p.Kd = H;
  p.I = I;
  p.Nout = I;
  p.n_tiles = (I + 127) / 128;
  p.out = static_cast<__nv_bfloat16*>(act);
  p.save = static_cast<__nv_bfloat16*>(save);
  p.gather = gather;
  p.gk = K;
  p.g_rows = T;
  p.g_cols = H;
  p.gsrc = static_cast<const uint8_t*>(A);
  CUtensorMap c_act, c_save;
  if (!store_map_2d(&c_act, act, I, N) || !store_map_2d(&c_save, save ? save : act, save ? 2 * I : I, N))
    return MOE_ERR_CUDA;
  CUtensorMap ma64 = ma;  // 64-row A boxes for a pair's half tiles
  if (paired) {
    const uint32_t b64[2] = {64, 64};
    if (!make_map(&ma64, A, 2, da, b64)) return MOE_ERR_CUDA;
  }
  return paired ? launch<kFwdGateUp | kPaired>(ma, ma64, mg, mu, c_act, c_save, p, s)
                : launch<kFwdGateUp>(ma, ma, mg, mu, c_act, c_save, p, s);
}

int launch_gmm_bf16_gate_up(const void* A, const void* Wg, const void* Wu, const int32_t* off,
                            int N, int H, int I, int E, void* act, void* save, int32_t* status,
                            cudaStream_t s) {
  return gate_up_bf16(A, N, nullptr, 1, Wg, Wu, off, N, H, I, E, act, save, status, s);
}

int launch_gmm_bf16_gate_up_gather(const void* tokens, int T, const int32_t* sorted_indices, int K,
                                   const void* Wg, const void* Wu, const int32_t* off, int N, int H,
                                   int I, int E, void* act, void* save, int32_t* status,
                                   cudaStream_t s) {
  return gate_up_bf16(tokens, T, sorted_indices, K, Wg, Wu, off, N, H, I, E, act, save, status, s);
}

int launch_gmm_bf16_down(const void* A, const void* Wd, const int32_t* off, int N, int H, int I,
                         int E, void* out, int32_t* status, cudaStream_t s) {
  if (int rc = device_ok()) return rc;
  CUtensorMap ma, md;
  const uint64_t da[2] = {(uint64_t)I, (uint64_t)N};
  const uint32_t ba[2] = {64, 128};
  const uint64_t dw[3] = {(uint64_t)I, (uint64_t)H, (uint64_t)E};
  const bool paired = use_pairs(kPairMinRowsDown, N, E);
  const uint32_t bw[3] = {64, (uint32_t)(paired ? Traits<kFwdDown | kPaired>::b_rows
                                                : Traits<kFwdDown>::b_rows), 1};
  if (!make_map(&ma, A, 2, da, ba) || !make_map(&md, Wd, 3, dw, bw)) return MOE_ERR_CUDA;
  Params p = base_params(off, N, E, status);
  p.Kd = I;
  p.I = I;
  p.Nout = H;
  p.n_tiles = (H + 255) / 256;
  p.out = static_cast<__nv_bfloat16*>(out);
  CUtensorMap c_out;
  if (!store_map_2d(&c_out, out, H, N)) return MOE_ERR_CUDA;
  CUtensorMap ma64 = ma;
  if (paired) {
    const uint32_t b64[2] = {64, 64};
    if (!make_map(&ma64, A, 2, da, b64)) return MOE_ERR_CUDA;
    return launch<kFwdDown | kPaired>(ma, ma64, md, md, c_out, c_out, p, s);
  }
  // 64-row boxes of W_down for the split tiles of a short last wave
  CUtensorMap md64;
  const uint32_t bw64[3] = {64, 64, 1};
  if (!make_map(&md64, Wd, 3, dw, bw64)) return MOE_ERR_CUDA;
  return launch<kFwdDown>(ma, ma, md, md64, c_out, c_out, p, s);
}

int launch_down_dgrad_bf16(const void* dY, const void* gate_up, const int32_t* off, int N, int H,
                           int I, int E, const void* Wd, void* dgu, int32_t* status,
                           cudaStream_t s) {
  if (int rc = device_ok()) return rc;
  if (N == 0) return MOE_OK;
  const uint32_t box_k[2] = {64, 128};
  const uint32_t box_mn3[3] = {64, 64, 1};
  CUtensorMap m_dy, m_wd;
  const uint64_t d_dy[2] = {(uint64_t)H, (uint64_t)N};
  const uint64_t d_wd[3] = {(uint64_t)I, (uint64_t)H, (uint64_t)E};
  if (!make_map(&m_dy, dY, 2, d_dy, box_k) || !make_map(&m_wd, Wd, 3, d_wd, box_mn3))
    return MOE_ERR_CUDA;
  Params p = base_params(off, N, E, status);
  p.Kd = H;
  p.I = I;
  p.Nout = I;
  p.n_tiles = (I + Traits<kDgradDown>::bn - 1) / Traits<kDgradDown>::bn;
  p.out = static_cast<__nv_bfloat16*>(dgu);
  p.aux = static_cast<const __nv_bfloat16*>(gate_up);
  CUtensorMap c_dgu;
  if (!store_map_2d(&c_dgu, dgu, 2 * I, N)) return MOE_ERR_CUDA;
  return E <= kFewMaxExperts ? launch<kDgradDown | kFewExperts>(m_dy, m_dy, m_wd, m_wd, c_dgu, c_dgu, p, s)
                             : launch<kDgradDown>(m_dy, m_dy, m_wd, m_wd, c_dgu, c_dgu, p, s);
}

int launch_gate_up_dgrad_bf16(const void* dgu, const int32_t* off, int N, int H, int I, int E,
                              const void* Wg, const void* Wu, void* dX, int32_t* status,
                              cudaStream_t s) {
  if (int rc = device_ok()) return rc;
  if (N == 0) return MOE_OK;
  const uint32_t box_k[2] = {64, 128};
  const uint32_t box_mn3[3] = {64, 64, 1};
  CUtensorMap m_dgu, m_wg, m_wu;
  const uint64_t d_dgu[2] = {(uint64_t)2 * I, (uint64_t)N};
  const uint64_t d_w[3] = {(uint64_t)H, (uint64_t)I, (uint64_t)E};
  if (!make_map(&m_dgu, dgu, 2, d_dgu, box_k) || !make_map(&m_wg, Wg, 3, d_w, box_mn3) ||
      !make_map(&m_wu, Wu, 3, d_w, box_mn3))
    return MOE_ERR_CUDA;
  Params q = base_params(off, N, E, status);
  q.Kd = 2 * I;
  q.I = I;
  q.Nout = H;
  q.n_tiles = (H + 255) / 256;
  q.out = static_cast<__nv_bfloat16*>(dX);
  CUtensorMap c_dx;
  if (!store_map_2d(&c_dx, dX, H, N)) return MOE_ERR_CUDA;
  const bool paired = use_pairs(kPairMinRowsDgradGateUp, N, E);
  CUtensorMap m_dgu64 = m_dgu;  // 64-row A boxes for a pair's half tiles
  if (paired) {
    const uint32_t b64[2] = {64, 64};
    if (!make_map(&m_dgu64, dgu, 2, d_dgu, b64)) return MOE_ERR_CUDA;
  }
  return paired
             ? launch<kDgradGateUp | kPaired>(m_dgu, m_dgu64, m_wg, m_wu, c_dx, c_dx, q, s)
             : launch<kDgradGateUp>(m_dgu, m_dgu, m_wg, m_wu, c_dx, c_dx, q, s);
}

// With no rows at all the operand maps are never read (every tile has zero
// k blocks); they point at the output so that they are well formed.
int launch_down_wgrad_bf16(const void* dY, const void* act, const int32_t* off, int N, int H,
                           int I, int E, void* dWd, int32_t* status, cudaStream_t s) {
  if (int rc = device_ok()) return rc;
  constexpr int BK = Traits<kWgradDown>::bk;
  CUtensorMap m_a, m_b;
  const int rows = N > 0 ? N : 1;
  if (!k_rows_map(&m_a, N > 0 ? dY : dWd, H, rows, BK) ||
      !k_rows_map(&m_b, N > 0 ? act : dWd, I, rows, BK))
    return MOE_ERR_CUDA;
  Params p = base_params(off, N, E, status);
  p.I = I;
  p.Mout = H;
  p.Nout = I;
  p.m_tiles = (H + 127) / 128;
  p.n_tiles = (I + 255) / 256;
  p.out = static_cast<__nv_bfloat16*>(dWd);
  CUtensorMap c_dwd;
  if (!store_map_3d(&c_dwd, dWd, I, H, E)) return MOE_ERR_CUDA;
  return use_pairs(kPairMinRowsWgrad, N, E)
             ? launch<kWgradDown | kPaired>(m_a, m_a, m_b, m_b, c_dwd, c_dwd, p, s)
             : launch<kWgradDown>(m_a, m_a, m_b, m_b, c_dwd, c_dwd, p, s);
}

// Gate/up wgrad.  gather == nullptr: X is the permuted [N, H] buffer;
// otherwise X row i is row gather[i] / K of the token matrix X [T, H].
static int gate_up_wgrad_bf16(const void* dgu, const void* X, int T, const int32_t* gather, int K,
                              const int32_t* off, int N, int H, int I, int E, void* dWg,
                              void* dWu, int32_t* status, cudaStream_t s) {
  if (int rc = device_ok()) return rc;
  constexpr int BK = Traits<kWgradGateUp>::bk;
  CUtensorMap m_a, m_b;
  const int rows = N > 0 ? N : 1;
  const bool any = N > 0 && (gather == nullptr || T > 0);
  // (B is not read through a map when gathering)
  if (!k_rows_map(&m_a, any ? dgu : dWg, 2 * I, rows, BK) ||
      !k_rows_map(&m_b, any ? X : dWg, H, gather ? (T > 0 ? T : 1) : rows, BK))
    return MOE_ERR_CUDA;
  Params p = base_params(off, N, E, status);
  p.I = I;
  p.Mout = 2 * I;
  p.Nout = H;
  p.m_tiles = (2 * I + 127) / 128;
  p.n_tiles = (H + 255) / 256;
  p.out = static_cast<__nv_bfloat16*>(dWg);
  p.out2 = static_cast<__nv_bfloat16*>(dWu);
  p.gather = gather;
  p.gk = K;
  p.g_rows = T;
  p.g_cols = H;
  p.gsrc = static_cast<const uint8_t*>(X);
  CUtensorMap c_dwg, c_dwu;
  if (!store_map_3d(&c_dwg, dWg, H, I, E) || !store_map_3d(&c_dwu, dWu, H, I, E))
    return MOE_ERR_CUDA;
  // gathered X rows are loaded by the single-CTA producer only
  return (gather == nullptr && use_pairs(kPairMinRowsWgrad, N, E))
             ? launch<kWgradGateUp | kPaired>(m_a, m_a, m_b, m_b, c_dwg, c_dwu, p, s)
             : launch<kWgradGateUp>(m_a, m_a, m_b, m_b, c_dwg, c_dwu, p, s);
}

int launch_gate_up_wgrad_bf16(const void* dgu, const void* X, const int32_t* off, int N, int H,
                              int I, int E, void* dWg, void* dWu, int32_t* status,
                              cudaStream_t s) {
  return gate_up_wgrad_bf16(dgu, X, N, nullptr, 1, off, N, H, I, E, dWg, dWu, status, s);
}

int launch_wait_selftest(int32_t* status, cudaStream_t s) {
  tc::wait_selftest_kernel<<<1, 32, 0, s>>>(status);
  count_launches(1);
  return cudaPeekAtLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_gate_up_wgrad_bf16_gather(const void* dgu, const void* tokens, int T,
                                     const int32_t* sorted_indices, int K, const int32_t* off,
                                     int N, int H, int I, int E, void* dWg, void* dWu,
                                     int32_t* status, cudaStream_t s) {
  return gate_up_wgrad_bf16(dgu, tokens, T, sorted_indices, K, off, N, H, I, E, dWg, dWu, status,
                            s);
}

}  // namespace moe
