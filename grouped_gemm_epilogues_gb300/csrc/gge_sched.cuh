// FastDivmod and the persistent tile schedule (host + device).
//
// FastDivmod follows quack/fast_math.py (quack-kernels 0.2.0): for a divisor
// d, p = 31 + ceil(log2 d), multiplier = ceil(2^p / d), shift = p - 32, and
// n / d = umulhi(n, multiplier) >> shift for 0 <= n < 2^31 (d == 1 is passed
// through, since its shift would be -1).  It is exact on that domain
// (Granlund & Montgomery 1994: m*d - 2^p lies in [0, d), so the error term
// n*(m*d - 2^p) < 2^31 * 2^ceil(log2 d) = 2^p never reaches the next integer).
//
// The plain schedule maps a linear tile index to (batch, m-tile, n-tile):
// batches outermost, then bands of `band` m-tiles; inside a band the m-tile
// varies fastest, so CTAs that run at the same time share B tiles and a
// band's A rows, which keeps the working set of one wave inside L2.  With
// `along_n` the roles swap: bands of n-tiles, the n-tile varying fastest.
// This plays the role of the pages' raster order / max_swizzle_size
// (quack/dense_gemm_sm90.py, GemmSm90 tile scheduler arguments).
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define GGE_HD __host__ __device__ __forceinline__
#else
#define GGE_HD inline
#endif

namespace gge {

struct FastDivmod {
  int32_t divisor;
  uint32_t multiplier;
  uint32_t shift;

  static inline FastDivmod create(int32_t d) {
    FastDivmod f;
    f.divisor = d;
    // ceil(log2 d): floor(log2 d) plus one unless d is a power of two
    int lg = 0;
    while ((1u << lg) < static_cast<uint32_t>(d) && lg < 31) ++lg;
    const uint32_t p = 31u + static_cast<uint32_t>(lg);
    const uint64_t num = (uint64_t(1) << p) + static_cast<uint64_t>(d) - 1u;
    f.multiplier = static_cast<uint32_t>(num / static_cast<uint64_t>(d));
    f.shift = p - 32u;  // wraps to 0xffffffff for d == 1, never used then
    return f;
  }

  GGE_HD int32_t div(int32_t n) const {
    if (divisor == 1) return n;
#if defined(__CUDA_ARCH__)
    uint32_t hi;
    asm("mul.hi.u32 %0, %1, %2;" : "=r"(hi) : "r"(static_cast<uint32_t>(n)), "r"(multiplier));
#else
    const uint32_t hi = static_cast<uint32_t>(
        (static_cast<uint64_t>(static_cast<uint32_t>(n)) * multiplier) >> 32);
#endif
    return static_cast<int32_t>(hi >> shift);
  }

  GGE_HD void divmod(int32_t n, int32_t& q, int32_t& r) const {
    q = div(n);
    r = n - q * divisor;
  }
};

struct PlainSchedule {
  int32_t tiles_m, tiles_n, batches;
  int32_t band;          // tiles of the banded dimension per raster band
  int32_t along_n;       // 1: bands of n-tiles (n varies fastest); 0: bands of m-tiles
  int32_t full_bands;    // banded tiles / band
  int32_t num_tiles;     // tiles_m * tiles_n * batches
  FastDivmod per_batch;  // tiles_m * tiles_n
  FastDivmod band_tiles; // band * (tiles of the other dimension)
  FastDivmod band_rows;  // band
  FastDivmod tail_rows;  // banded tiles % band (1 when the bands divide evenly)

  static inline PlainSchedule create(int32_t tiles_m, int32_t tiles_n, int32_t batches,
                                     int32_t band, bool along_n = false) {
    PlainSchedule s;
    const int32_t banded = along_n ? tiles_n : tiles_m;
    const int32_t other = along_n ? tiles_m : tiles_n;
    if (band < 1) band = 1;
    if (band > banded) band = banded > 0 ? banded : 1;
    s.tiles_m = tiles_m;
    s.tiles_n = tiles_n;
    s.batches = batches;
    s.band = band;
    s.along_n = along_n ? 1 : 0;
    s.full_bands = banded / band;
    s.num_tiles = tiles_m * tiles_n * batches;
    s.per_batch = FastDivmod::create(tiles_m * tiles_n > 0 ? tiles_m * tiles_n : 1);
    s.band_tiles = FastDivmod::create(band * (other > 0 ? other : 1));
    s.band_rows = FastDivmod::create(band);
    const int32_t tail = banded % band;
    s.tail_rows = FastDivmod::create(tail > 0 ? tail : 1);
    return s;
  }

  // t in [0, num_tiles)  ->  (batch, m-tile, n-tile)
  GGE_HD void map(int32_t t, int32_t& l, int32_t& mb, int32_t& nb) const {
    int32_t r, b, w, i, o;
    per_batch.divmod(t, l, r);
    band_tiles.divmod(r, b, w);
    const FastDivmod& rows = (b < full_bands) ? band_rows : tail_rows;
    rows.divmod(w, o, i);
    if (along_n) {
      nb = b * band + i;
      mb = o;
    } else {
      mb = b * band + i;
      nb = o;
    }
  }
};

// Raster band width that keeps one wave's operand footprint smallest: a wave
// of `units` tiles spread over `band` rows of tile_m and units / band columns
// of tile_n reads band * tile_m + (units / band) * tile_n rows of K, least at
// band = sqrt(units * tile_n / tile_m) (m-tiles per band; along N the ratio
// inverts).  At least 1, at most 32.
inline int32_t auto_band(int32_t units, int32_t tile_m, int32_t tile_n, bool along_n) {
  if (units < 1 || tile_m < 1 || tile_n < 1) return 8;
  const double ratio = along_n ? static_cast<double>(tile_m) / tile_n
                               : static_cast<double>(tile_n) / tile_m;
  double b = 1.0;
  while ((b + 1.0) * (b + 1.0) <= units * ratio) b += 1.0;
  // b = floor(sqrt(units * ratio)); take b + 1 when it is nearer
  const double x = units * ratio;
  if ((b + 1.0) * (b + 1.0) - x < x - b * b) b += 1.0;
  return static_cast<int32_t>(b < 1.0 ? 1.0 : (b > 32.0 ? 32.0 : b));
}

// Split of the last, partly filled wave along K.  T tiles run on U units (CTAs
// or CTA pairs) of a persistent grid: W = T / U full waves, then R = T - W U
// tiles.  When R <= U / 2 each of those R tiles is cut into S K-slices (S <=
// U / R, so the slices still form one wave; at most 8; at least 8 k-tiles a
// slice), which S different units compute; whichever unit finishes a tile's
// slices last adds their fp32 partial accumulators before the epilogue.  Work
// item v < W U is tile v; item W U + q is slice q % S of tile W U + q / S, so
// the S slices of a tile run side by side on units q - q % S ...  The unit
// stride of the persistent schedule (unit u takes items u, u + U, ...) is
// unchanged.  (Cutting a last wave that the tiles fill exactly into two
// slices a tile as well, so that half the final epilogues overlap the second
// half of the MMAs, measured 18 % slower on 4096^3: the partial sums' traffic
// costs more than the hidden epilogues.)
struct TailSplit {
  int32_t full;    // W * U: items that are whole tiles
  int32_t tail;    // R: tiles split (0: no split)
  int32_t splits;  // S
};

GGE_HD TailSplit plan_tail_split(int64_t tiles, int32_t units, int32_t k_tiles) {
  TailSplit s;
  s.full = static_cast<int32_t>(tiles);
  s.tail = 0;
  s.splits = 1;
  if (units < 2 || tiles <= 0) return s;
  const int64_t waves = tiles / units;
  const int64_t r = tiles - waves * units;
  if (r == 0) return s;
  int64_t splits = units / r;
  if (splits > 8) splits = 8;
  if (splits > k_tiles / 8) splits = k_tiles / 8;
  if (splits < 2) return s;
  s.full = static_cast<int32_t>(waves * units);
  s.tail = static_cast<int32_t>(r);
  s.splits = static_cast<int32_t>(splits);
  return s;
}

}  // namespace gge
