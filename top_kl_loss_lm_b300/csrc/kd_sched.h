// kd_sched.h — static work schedule of the persistent GEMM kernels (host + device).
//
// A "unit" is what one CTA does without handing off: a run of output tiles in
// one row block (forward / dZ recompute), or one output tile over a range of
// k-blocks (dH, dW). Units are numbered so that units that run at the same time
// (consecutive numbers, dealt round-robin to the CTAs) share operand tiles in L2.
#pragma once

#include <cstdint>

#ifndef __CUDACC__
#define KD_HD
#else
#define KD_HD __host__ __device__
#endif

namespace kd {

constexpr int kBM = 128;        // tile rows (MMA M)
constexpr int kBK = 64;         // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int kBNMax = 256;     // widest tile (MMA N)
constexpr int kPanelRows = 16;  // row blocks per panel (and per forward launch)
constexpr int kMaxSlots = 64;   // max vocabulary splits per row (LSE partial slots)
constexpr int kMaxKSplits = 8;  // max split of the dH contraction

enum SchedMode : int { kSchedPanel = 0, kSchedTiles = 1 };

struct Sched {
  int mode;
  int MB, NB, KB;      // row blocks, column tiles, k-blocks
  int G0, S0;          // full panel: row blocks, vocabulary splits
  int Gl, Sl;          // last panel
  int P;               // panels
  int KS;              // k-splits (tiles mode)
  int64_t upp;         // units per full panel
  int64_t total;       // units
};

struct Unit {
  int m_blk, n_begin, n_end, kb_begin, kb_end, slot;
};

KD_HD inline Unit sched_unit(const Sched& s, int64_t u) {
  Unit d;
  if (s.mode == kSchedPanel) {
    int p = static_cast<int>(u / s.upp);
    if (p > s.P - 1) p = s.P - 1;
    const int64_t ul = u - static_cast<int64_t>(p) * s.upp;
    const bool last = (p == s.P - 1);
    const int G = last ? s.Gl : s.G0;
    const int S = last ? s.Sl : s.S0;
    const int sp = static_cast<int>(ul / G);
    const int mi = static_cast<int>(ul % G);
    d.m_blk = p * s.G0 + mi;
    d.n_begin = static_cast<int>(static_cast<int64_t>(sp) * s.NB / S);
    d.n_end = static_cast<int>(static_cast<int64_t>(sp + 1) * s.NB / S);
    d.kb_begin = 0;
    d.kb_end = s.KB;
    d.slot = sp;
  } else {
    const int64_t per = static_cast<int64_t>(s.MB) * s.NB;
    const int ks = static_cast<int>(u / per);
    const int64_t r = u - static_cast<int64_t>(ks) * per;
    d.m_blk = static_cast<int>(r / s.NB);
    d.n_begin = static_cast<int>(r % s.NB);
    d.n_end = d.n_begin + 1;
    d.kb_begin = static_cast<int>(static_cast<int64_t>(ks) * s.KB / s.KS);
    d.kb_end = static_cast<int>(static_cast<int64_t>(ks + 1) * s.KB / s.KS);
    d.slot = ks;
  }
  return d;
}

KD_HD inline int kd_gcd(int a, int b) {
  while (b) {
    const int t = a % b;
    a = b;
    b = t;
  }
  return a;
}

// Panel schedule over MB row blocks x NB vocabulary tiles. Each panel of G row
// blocks is cut into S vocabulary splits with S = grid / gcd(G, grid) when that
// fits, so that G * S is a multiple of the grid and every CTA gets the same
// number of equal-sized units.
inline Sched make_panel_sched(int MB, int NB, int KB, int grid) {
  Sched s{};
  s.mode = kSchedPanel;
  s.MB = MB;
  s.NB = NB;
  s.KB = KB;
  s.KS = 1;
  s.G0 = MB < kPanelRows ? MB : kPanelRows;
  s.P = (MB + s.G0 - 1) / s.G0;
  s.Gl = MB - (s.P - 1) * s.G0;
  auto splits = [&](int G) {
    int S = grid / kd_gcd(G, grid);
    if (S > kMaxSlots) S = kMaxSlots;
    if (S > NB) S = NB;
    if (S < 1) S = 1;
    return S;
  };
  s.S0 = splits(s.G0);
  s.Sl = splits(s.Gl);
  s.upp = static_cast<int64_t>(s.G0) * s.S0;
  s.total = static_cast<int64_t>(s.P - 1) * s.upp + static_cast<int64_t>(s.Gl) * s.Sl;
  return s;
}

// One tile per unit, optionally split over k (order: split, row block, column tile).
inline Sched make_tile_sched(int MB, int NB, int KB, int KS) {
  Sched s{};
  s.mode = kSchedTiles;
  s.MB = MB;
  s.NB = NB;
  s.KB = KB;
  s.KS = KS < 1 ? 1 : (KS > KB ? KB : KS);
  s.G0 = MB;
  s.S0 = 1;
  s.Gl = MB;
  s.Sl = 1;
  s.P = 1;
  s.upp = static_cast<int64_t>(MB) * NB;
  s.total = s.upp * s.KS;
  return s;
}

// k-split for a tile grid: the split in [1, kMaxKSplits] whose last wave is fullest.
inline int choose_ksplit(int64_t tiles, int KB, int grid) {
  int best = 1;
  double best_eff = 0.0;
  for (int ks = 1; ks <= kMaxKSplits && ks <= KB; ++ks) {
    const int64_t units = tiles * ks;
    const int64_t waves = (units + grid - 1) / grid;
    const double eff = static_cast<double>(units) / static_cast<double>(waves * grid);
    if (eff > best_eff + 0.02) {
      best_eff = eff;
      best = ks;
    }
  }
  return best;
}

// Column tile width over the hidden size D for a K-major B operand (dW, whose B
// is the token group's H transposed): D is split evenly into ceil(D / 256)
// tiles, each rounded up to a multiple of 16, e.g. 12 x 240 for D = 2,880
// instead of 12 x 256 with 192 zero-filled columns. Each CTA of a pair then
// holds 120 rows of B, a multiple of the 8-row core matrix.
inline int hidden_tile_width(int D) {
  const int nt = (D + kBNMax - 1) / kBNMax;
  const int w = (D + nt - 1) / nt;
  return (w + 15) / 16 * 16;
}

// Column tile width for an MN-major B operand (dH, whose B is W [V x D]): 256
// above 256 columns, so every 64-column slab a CTA loads starts on a 128-byte
// line (an even split such as 240 would start every other slab mid-line and
// measured about 9% slower per useful FLOP); a single tile is N rounded up to a
// multiple of 16.
inline int mn_major_tile_width(int N) {
  if (N > kBNMax) return kBNMax;
  return (N + 15) / 16 * 16;
}

}  // namespace kd
