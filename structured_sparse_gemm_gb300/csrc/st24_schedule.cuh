// st24_schedule.cuh -- the persistent-grid work schedule shared by the SpMM
// kernels: data-parallel waves of whole output tiles followed by a stream-K
// tail.
//
// Output tiles are numbered in the raster of tile_coords.  The first
// dp_tiles tiles go round-robin to the G CTAs (tile c, c + G, c + 2G, ... for
// CTA c), so at any moment the grid works on G consecutive tiles, which keeps
// the B panel and a few A rows hot in L2.  The remaining sk_tiles tiles are
// flattened into (tile, k-block) iterations and CTA c takes the contiguous run
// [c*I/G, (c+1)*I/G) of the I = sk_tiles * k_iters iterations, so the last
// wave is balanced to one k-block.  A tile whose k-blocks are spread over
// several CTAs ("segments", consecutive CTAs in k order) is finished through
// the workspace by whichever contributor arrives last.
#pragma once

#include <cstdint>

namespace st24 {

// a / b for a >= 0 and b > 0, in 32-bit arithmetic when both fit (64-bit
// integer division is a long software sequence on the GPU, and this math runs
// on the producer's critical path at every tile).
__device__ __forceinline__ int64_t div_nn(int64_t a, int64_t b) {
  if (((a | b) >> 31) == 0) return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
  return a / b;
}

struct Segment {
  int64_t tile;
  int64_t kb0, kb1;   // k-blocks [kb0, kb1) of the tile
};

// Output tile index -> (m-tile, n-tile): groups of group_m m-tiles, n-tile
// outer inside a group (group_m = 1 is row-major, group_m = tiles_m is
// column-major).
__device__ __forceinline__ void tile_coords(int64_t tile, int64_t tiles_m, int64_t tiles_n, int64_t group_m,
                                            int64_t& mt, int64_t& nt) {
  const int64_t per_group = group_m * tiles_n;
  const int64_t g = div_nn(tile, per_group);
  const int64_t first = g * group_m;
  const int64_t rows = (tiles_m - first) < group_m ? (tiles_m - first) : group_m;
  const int64_t i = tile - g * per_group;
  nt = div_nn(i, rows);
  mt = first + (i - nt * rows);
}

struct Schedule {
  int64_t k_iters, dp_tiles, sk_iters, G, cta;
  int64_t dp_next, sk_it, sk_end;

  __device__ __forceinline__ Schedule(int64_t k_iters_, int64_t dp_tiles_, int64_t sk_tiles, int64_t G_,
                                      int64_t cta_)
      : k_iters(k_iters_), dp_tiles(dp_tiles_), sk_iters(sk_tiles * k_iters_), G(G_), cta(cta_) {
    dp_next = cta;
    sk_it = run_begin(cta);
    sk_end = run_begin(cta + 1);
  }

  __device__ __forceinline__ int64_t run_begin(int64_t c) const { return div_nn(c * sk_iters, G); }

  // Next piece of work of this CTA; false when there is none.
  __device__ __forceinline__ bool next(Segment& s) {
    if (dp_next < dp_tiles) {
      s.tile = dp_next;
      s.kb0 = 0;
      s.kb1 = k_iters;
      dp_next += G;
      return true;
    }
    if (sk_it < sk_end) {
      const int64_t local = div_nn(sk_it, k_iters);
      s.tile = dp_tiles + local;
      s.kb0 = sk_it - local * k_iters;
      s.kb1 = s.kb0 + (sk_end - sk_it) < k_iters ? s.kb0 + (sk_end - sk_it) : k_iters;
      sk_it += s.kb1 - s.kb0;
      return true;
    }
    return false;
  }

  // The CTA whose stream-K run contains iteration u of the tail.
  __device__ __forceinline__ int64_t owner(int64_t u) const { return div_nn((u + 1) * G - 1, sk_iters); }
  // First and last CTA contributing to stream-K tile `tile`.
  __device__ __forceinline__ int64_t first_cta(int64_t tile) const { return owner((tile - dp_tiles) * k_iters); }
  __device__ __forceinline__ int64_t last_cta(int64_t tile) const {
    return owner((tile - dp_tiles) * k_iters + k_iters - 1);
  }
  // Workspace slot of CTA c's partial of `tile`: 2c for the first tile of its
  // run, 2c + 1 for the last (a run has at most these two partial tiles).
  __device__ __forceinline__ int64_t slot(int64_t c, int64_t tile) const {
    return 2 * c + ((dp_tiles + div_nn(run_begin(c), k_iters)) == tile ? 0 : 1);
  }
};

}  // namespace st24
