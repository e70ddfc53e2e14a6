// Interleaved, rotated storage of PQ codes inside a block of 32 vector slots
// (see ivfpq_index.cu for the rationale). Used by the writer (ivfpq_add) and
// the readers (list scan); the Python tests restate it to check invariants.
#pragma once

#include <stdint.h>

namespace ivfpq {

// Sub-quantizers are handled in groups of up to 32: group g covers
// [32g, 32g + group_size(g, m)).
__host__ __device__ __forceinline__ int group_size(int g, int m) {
  const int r = m - 32 * g;
  return r < 32 ? r : 32;
}

// Code byte (sub-quantizer index) kept at stored position s of the vector in
// slot `lane`: inside each group the bytes are rotated left by the slot index.
__host__ __device__ __forceinline__ int stored_source_byte(int lane, int s, int m) {
  const int g0 = s & ~31;
  const int gs = group_size(s >> 5, m);
  return g0 + (lane + (s - g0)) % gs;
}

// Byte offset, inside the 32*m-byte block, of stored position s of slot `lane`:
// full 16-byte chunks are [chunk][slot][16], the remainder is [slot][m % 16].
__host__ __device__ __forceinline__ int stored_byte_offset(int lane, int s, int m) {
  const int nfull = m >> 4;
  const int c = s >> 4;
  if (c < nfull) return c * 512 + lane * 16 + (s & 15);
  const int r = m & 15;
  return nfull * 512 + lane * r + (s - (nfull << 4));
}

}  // namespace ivfpq
