// Tile schedule of the persistent grouped GEMM, shared by the kernel (device) and the
// diagnostics entry point (host) so that the host can check the exact index arithmetic the
// kernel uses.
#pragma once
#include "moe_internal.h"

#if defined(__CUDACC__)
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif

namespace moe {

// Whether every tile of a grouped operand set is tall: the n-tile cap is the tall-tile limit,
// so a segment of n rows runs as ceil(n / tall_rows) tall n-tiles.
MOE_HD bool all_tall(int bn, int tall_rows) { return tall_rows > 0 && bn <= tall_rows; }

// Tile units of a segment of n rows with n-tile cap bn: when every tile is tall, one unit per
// tall n-tile; otherwise a segment of 1..tall_rows rows is one unit (a tall tile per two
// scheduled m-tiles) and each of the ceil(n / bn) n-tiles of a longer segment is one unit per
// scheduled m-tile, counted twice when tall tiles exist so that a unit is always worth
// (m_tiles / 2) tiles.
MOE_HD int seg_units(int n, int bn, int tall_rows) {
  if (n <= 0) return 0;
  if (all_tall(bn, tall_rows)) return (n + tall_rows - 1) / tall_rows;
  if (tall_rows > 0 && n <= tall_rows) return 1;
  return (tall_rows > 0 ? 2 : 1) * ((n + bn - 1) / bn);
}

// Tiles per unit of a grouped operand set.
MOE_HD int tiles_per_unit(const TcProblem& P) {
  return P.tall_rows > 0 ? P.m_tiles / 2 : P.m_tiles;
}

struct Tile {
  int prob;   // 0 = first operand set (grouped or single), 1 = second (single)
  int seg;    // segment (expert) within the operand set
  int m;      // scheduled m-tile within the segment (a pair's tiles are 2m and 2m + 1); for a
              // tall tile, the pair of scheduled m-tiles 2m and 2m + 1
  int tall;   // 1: a tall tile (two scheduled m-tiles over the whole segment, one per issuer)
  int row0;   // first B row of the tile
  int ncols;  // MMA N: multiple of 16, at most the n-tile cap
  int valid;  // B rows of the tile that belong to the segment (<= ncols)
  int nt;     // n-tiles of the segment (> 1: the weight tile is read again by a neighbour)
};

// Tile t of the schedule.  Operand set 0 comes first (tiles0 tiles), then set 1.  Within a
// segment tiles run in (m-group, m, n-tile) order: the n-tiles that share a weight tile are
// neighbours in the schedule (and so run at the same time on neighbouring CTAs, sharing the
// weight tile through L2), and a group of m-tiles shares each token tile.  A segment of n
// rows is cut into nt n-tiles of whole 16-row units, as even as possible.  A segment of at
// most tall_rows rows instead runs as m_tiles / 2 tall tiles over all its rows.  `seg_off` /
// `ntp` are the segment row offsets and the unit prefix of set 0 when it is grouped.
MOE_HD void decode_tile(const TcParams& p, const int* seg_off, const int* ntp, int tiles0, int t,
                        Tile& tl) {
  int prob = 0, local = t;
  if (t >= tiles0) {
    prob = 1;
    local = t - tiles0;
  }
  const TcProblem& P = p.prob[prob];
  int seg = 0, nt, seg_row0 = 0, seg_rows;
  tl.tall = 0;
  if (prob == 0 && P.seg_off != nullptr) {
    const int tpu = tiles_per_unit(P);
    const int q = local / tpu;
    int lo = 0, hi = P.n_seg;  // largest lo with ntp[lo] <= q
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (ntp[mid] <= q) lo = mid;
      else hi = mid;
    }
    seg = lo;
    const int units = ntp[seg + 1] - ntp[seg];
    local -= ntp[seg] * tpu;
    seg_row0 = seg_off[seg];
    seg_rows = seg_off[seg + 1] - seg_row0;
    if (all_tall(p.bn, P.tall_rows)) {
      // tall n-tiles: order (group of m-tile pairs, m-tile pair, n-tile), rows split evenly
      const int pairs = P.m_tiles >> 1;
      const int G2 = (P.group >> 1) > 0 && pairs % (P.group >> 1) == 0 ? (P.group >> 1) : 1;
      const int ntt = units;
      const int mg = local / (G2 * ntt);
      const int r = local - mg * G2 * ntt;
      const int mi = r / ntt;
      const int j = r - mi * ntt;
      tl.prob = prob;
      tl.seg = seg;
      tl.m = mg * G2 + mi;
      tl.tall = 1;
      tl.nt = ntt;
      const int u16 = (seg_rows + 15) >> 4;
      const int q16 = u16 / ntt, rem = u16 - q16 * ntt;
      const int u0 = j * q16 + (j < rem ? j : rem);
      const int nu = q16 + (j < rem ? 1 : 0);
      tl.row0 = seg_row0 + u0 * 16;
      tl.ncols = nu * 16;
      const int left = seg_rows - u0 * 16;
      tl.valid = left < tl.ncols ? left : tl.ncols;
      return;
    }
    if (P.tall_rows > 0 && units == 1) {
      tl.prob = prob;
      tl.seg = seg;
      tl.m = local;
      tl.tall = 1;
      tl.nt = 1;
      tl.row0 = seg_row0;
      tl.ncols = ((seg_rows + 15) >> 4) << 4;
      tl.valid = seg_rows;
      return;
    }
    nt = P.tall_rows > 0 ? units >> 1 : units;
  } else {
    nt = P.nt;
    seg_rows = P.rows;
  }
  const int G = P.group;
  const int mg = local / (G * nt);
  const int r = local - mg * G * nt;
  const int mi = r / nt;
  const int j = r - mi * nt;
  tl.prob = prob;
  tl.seg = seg;
  tl.m = mg * G + mi;
  tl.nt = nt;
  const int units = (seg_rows + 15) >> 4;
  const int q16 = units / nt, rem = units - q16 * nt;
  const int u0 = j * q16 + (j < rem ? j : rem);
  const int nu = q16 + (j < rem ? 1 : 0);
  tl.row0 = seg_row0 + u0 * 16;
  tl.ncols = nu * 16;
  const int left = seg_rows - u0 * 16;
  tl.valid = left < tl.ncols ? left : tl.ncols;
}

// Whether the CTA that owns 128-row weight tile `m` loads the second 64-row weight box.
MOE_HD bool a_has_box1(const TcProblem& P, int m) {
  return P.a_box_rows == 64 && (m * P.a_m_stride + P.a_box1_off) < P.a_valid_rows;
}

// Weight bytes the CTA that owns weight tile `m` loads per 64-deep k-block.
MOE_HD unsigned a_block_bytes(const TcProblem& P, int m) {
  return static_cast<unsigned>((a_has_box1(P, m) ? 2 : 1) * P.a_box_rows * 128);
}

}  // namespace moe
