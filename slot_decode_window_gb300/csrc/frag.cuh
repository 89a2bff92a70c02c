// Where each element of an activation vector lands in the B-operand fragment
// records, and the power-of-two factor it carries (the inverse of the factor
// the packed A codes carry for the same k-slot).
#pragma once
#include "common.cuh"

namespace strata {

// Offset (in halves, within one part: hi or lo) of element i of a vector
// whose matrix is BITS-bit, and the factor applied before the hi/lo split.
template <int BITS>
__host__ __device__ inline void frag_main_pos(int i, int& off, float& factor);

template <>
__host__ __device__ inline void frag_main_pos<4>(int i, int& off, float& factor) {
  // lane c covers elements 8c..8c+7 of a 32-element block; per block the
  // record is [mma0 b0b1: e0 e1 | mma0 b2b3: e4 e5 | mma1 b0b1: e2 e3 | mma1 b2b3: e6 e7]
  const int blk = i >> 5, e = i & 31, c = e >> 3, u = e & 7;
  const int ks = blk >> 1, bpar = blk & 1;
  const int slot = (u & 2) ? (4 + ((u >> 2) << 1) + (u & 1)) : (((u >> 2) << 1) + (u & 1));
  factor = (u & 2) ? (1.0f / 16.0f) : 1.0f;
  off = ((ks * 4 + c) * 16) + bpar * 8 + slot;
}

template <>
__host__ __device__ inline void frag_main_pos<2>(int i, int& off, float& factor) {
  // lane c covers elements 4c..4c+3 of a 16-element block; per block the
  // record is [b0b1: e0 e1 | b2b3: e2 e3]; blocks pair up inside a code word
  // and the odd block of a pair carries factors 16 and 64.
  const int blk = i >> 4, e = i & 15, c = e >> 2, u = e & 3;
  const int ks = blk >> 3, bi = blk & 7;
  factor = (bi & 1) ? ((u >> 1) ? 1.0f / 64.0f : 1.0f / 16.0f) : ((u >> 1) ? 0.25f : 1.0f);
  off = ((ks * 4 + c) * 32) + bi * 4 + u;
}

// Offset (halves, within one part) of block beta's sum in the sums region.
__host__ __device__ inline int frag_sum_pos(int beta) {
  const int mk = beta >> 4, w = beta & 15;
  const int c = (w & 7) >> 1;
  const int slot = ((w >> 3) << 1) + (w & 1);
  return (mk * 4 + c) * 4 + slot;
}

// Block index held by (mk, c, slot) of the sums region.
__host__ __device__ inline int frag_sum_block(int mk, int c, int slot) {
  return mk * 16 + 2 * c + ((slot >> 1) << 3) + (slot & 1);
}

}  // namespace strata
