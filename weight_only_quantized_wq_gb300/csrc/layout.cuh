// layout.cuh -- geometry of the packed weight layout written by wq_pack.
//
// Input (BitDistiller quant_matmul_kernel docstring and K loop): qw (K/V, N)
// int32, V = 32 / W values per word, code of (k, n) in field k % V of word
// [k / V][n], least significant field first.  int8 (W = 8) input is q (N, K)
// (tiny-llm int8_matmul docstring).
//
// Output: chunk rows of KC = 8 V values along K.  Chunk row kc holds N/16
// tiles of 16 output channels (n) x KC; one tile is 512 bytes = 32 lanes x 4
// words.  Lane l = 4 g + t (g = l / 4, t = l % 4) of a warp owns rows g and
// g + 8 of the tile and, in each k-step of 16 values, the four k positions
// 4t, 4t+1, 4t+2, 4t+3.  Its word wi = 2 h + r (r = 0: row g, r = 1: row g+8)
// holds V values of one row spanning WK = V/4 k-steps (h selects which half
// of the chunk's k-steps).
//
// Field order inside a word (W = 2, 4), chosen so that one shift and one
// LOP3 yield the pair of codes a tensor-core A register needs: with H = V/2,
//   field f <  H : k-step j = f / 2,       position c = 2 (f % 2)
//   field f >= H : k-step j = (f - H) / 2, position c = 2 ((f - H) % 2) + 1
// so (word >> (W i)) masked to the low field of each 16-bit half gives the
// codes at positions (c, c+1) = (0, 1) (i even) or (2, 3) (i odd) of k-step i/2.
// For W = 8 byte c is position c (natural order), the value the signed int8.
#pragma once

namespace wq {

template <int W>
struct Geo {
  static constexpr int V = 32 / W;        // values per 32-bit word
  static constexpr int KC = 8 * V;        // values along K per chunk row
  static constexpr int KS = KC / 16;      // k-steps (of 16) per chunk row
  static constexpr int WK = (W == 8) ? 1 : V / 4;  // k-steps per word
  static constexpr int H = V / 2;
};

// k offset inside a chunk row and tile row of field f of word wi of lane `lane`.
template <int W>
__host__ __device__ inline void field_coords(int lane, int wi, int f, int &kk, int &nn) {
  const int g = lane >> 2, t = lane & 3, h = wi >> 1, r = wi & 1;
  int j, c;
  if (W == 8) {
    j = 0;
    c = f;
  } else if (f < Geo<W>::H) {
    j = f >> 1;
    c = 2 * (f & 1);
  } else {
    j = (f - Geo<W>::H) >> 1;
    c = 2 * ((f - Geo<W>::H) & 1) + 1;
  }
  kk = 16 * (h * Geo<W>::WK + j) + 4 * t + c;
  nn = g + 8 * r;
}

}  // namespace wq
