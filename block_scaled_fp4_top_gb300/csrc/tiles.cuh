// Tile order of the persistent grouped GEMMs (gemm.cu, mxgemm.cu).
#pragma once

#include "common.cuh"

namespace fp4moe {

struct Tile {
  int e, nt, mt, me;  // expert, n-tile, m-tile, m-tiles of the expert
  bool last;          // the expert's last m-tile: the only one that can hold padding rows
};

// Position in the tile order. Expert e owns tiles [NT pm(e-1), NT pm(e)) with pm(e) = min(padded_offsets[e],
// R) / 128, so the expert of tile tau is the first e with NT pm(e) > tau: the searchsorted(right=True) rule on
// padded offsets. Inside the expert, local index L gives n-tile L / M_e and m-tile pm(e-1) + L % M_e. A
// cursor finds its first tile with one binary search and then steps in O(1), because the MMA issuer, which
// bounds the kernel's throughput, walks it once per tile. `poff` is the CTA's shared-memory copy of the
// padded offsets; r128 = R / 128 keeps every tile inside the R rows that exist.
struct TileCursor {
  int e, nt, ml, me, pm0;  // expert, n-tile, m-tile inside the expert, m-tiles of the expert, its first m-tile

  __device__ __forceinline__ void seek(int tau, const int* poff, int E, int NT, int r128) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (NT * min(poff[mid] >> 7, r128) > tau) hi = mid;
      else lo = mid + 1;
    }
    e = lo;
    pm0 = lo > 0 ? min(poff[lo - 1] >> 7, r128) : 0;
    me = min(poff[lo] >> 7, r128) - pm0;
    const int L = tau - NT * pm0;
    nt = L / me;
    ml = L - nt * me;
  }
  // the next tile; only called while one exists
  __device__ __forceinline__ void step(const int* poff, int E, int NT, int r128) {
    if (++ml < me) return;
    ml = 0;
    if (++nt < NT) return;
    nt = 0;
    pm0 += me;
    do {
      ++e;
      me = min(poff[e] >> 7, r128) - pm0;
    } while (me == 0 && e < E - 1);
  }
  __device__ __forceinline__ Tile tile() const { return Tile{e, nt, pm0 + ml, me, ml == me - 1}; }
};

}  // namespace fp4moe
