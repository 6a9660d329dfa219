// Copy of a contiguous run of 2-byte output (or source) elements between
// global memory and a shared-memory stage with 16-byte accesses: used by the
// epilogues whose rows are not 16-byte multiples (few output channels).
#pragma once

#include <cstdint>

namespace convgb300 {

// Copies `bytes` bytes between global address g and shared stage st, where
// st + phase16 holds the first byte and phase16 = g mod 16: every 16-byte
// aligned word of the range moves as one 16-byte access (thread i of n takes
// words i, i + n, ...); the bytes before the first and after the last
// aligned word move as 2-byte elements.  kIn: global -> shared, else
// shared -> global.  Element sizes are 2 bytes, so bytes and phase16 are even.
template <bool kIn>
__device__ __forceinline__ void copy_segment16(const uint8_t* g_const, uint8_t* st, int phase16,
                                                int bytes, int i, int n) {
  uint8_t* g = const_cast<uint8_t*>(g_const);
  const int head = phase16 == 0 ? 0 : min(16 - phase16, bytes);  // bytes before the first aligned word
  const int words = (bytes - head) >> 4;
  const int tail_start = head + (words << 4);
  // aligned words: global g + head + 16 w  <->  shared st + phase16 + head + 16 w
  for (int w = i; w < words; w += n) {
    uint4* gw = reinterpret_cast<uint4*>(g + head + 16 * w);
    uint4* sw = reinterpret_cast<uint4*>(st + phase16 + head + 16 * w);
    if (kIn)
      *sw = __ldg(gw);
    else
      *gw = *sw;
  }
  // head and tail elements (at most 7 each)
  const int nhead = head >> 1, ntail = (bytes - tail_start) >> 1;
  if (i < nhead + ntail) {
    const int off = i < nhead ? 2 * i : tail_start + 2 * (i - nhead);
    uint16_t* ge = reinterpret_cast<uint16_t*>(g + off);
    uint16_t* se = reinterpret_cast<uint16_t*>(st + phase16 + off);
    if (kIn)
      *se = *ge;
    else
      *ge = *se;
  }
}

}  // namespace convgb300
