// host_cast.h -- exact 16-bit <-> binary32 conversions on the host, shared by
// the offloaded host step and the shard files of 16-bit master weights.
#pragma once

#include <cstdint>
#include <cstring>

namespace zo {
namespace hc {

// IEEE binary16 to binary32 for all 65536 patterns (exact; NaN payloads kept).
struct HalfTable {
  float v[65536];
  HalfTable() {
    for (uint32_t h = 0; h < 65536; ++h) {
      const uint32_t sign = (h & 0x8000u) << 16;
      const uint32_t e = (h >> 10) & 0x1fu, f = h & 0x3ffu;
      float x;
      if (e == 0) {
        x = (float)f * 0x1p-24f;  // zero or subnormal: f * 2^-24, exact
        uint32_t b;
        std::memcpy(&b, &x, 4);
        b |= sign;
        std::memcpy(&x, &b, 4);
      } else {
        const uint32_t b = sign | (e == 31 ? (0xffu << 23) | (f << 13)
                                           : ((e + 112u) << 23) | (f << 13));
        std::memcpy(&x, &b, 4);
      }
      v[h] = x;
    }
  }
};
inline const HalfTable& half_table() {
  static const HalfTable* t = new HalfTable();
  return *t;
}

inline float bf16_to_f32(uint16_t h) {
  const uint32_t b = (uint32_t)h << 16;
  float x;
  std::memcpy(&x, &b, 4);
  return x;
}

// The two casts below are written without branches (every case computed,
// then selected) so that the compiler can vectorise the loops that use them.

inline uint32_t bits_of(float x) {
  uint32_t b;
  std::memcpy(&b, &x, 4);
  return b;
}
inline float float_of(uint32_t b) {
  float x;
  std::memcpy(&x, &b, 4);
  return x;
}

// binary32 to bfloat16, round to nearest even; NaN stays a (quiet) NaN.
inline uint16_t f32_to_bf16(float x) {
  const uint32_t b = bits_of(x);
  const uint32_t rounded = (b + 0x7fffu + ((b >> 16) & 1u)) >> 16;
  const uint32_t quiet = (b >> 16) | 0x40u;
  return (uint16_t)((b & 0x7fffffffu) > 0x7f800000u ? quiet : rounded);
}

// binary32 to binary16, round to nearest even, overflow to infinity, NaN to
// the quiet NaN 0x7e00 (with the sign).
inline uint16_t f32_to_f16(float x) {
  const uint32_t b = bits_of(x);
  const uint32_t sign = (b >> 16) & 0x8000u;
  const uint32_t a = b & 0x7fffffffu;
  // normal results: round the 23-bit fraction at bit 13, rebias 127 -> 15
  const uint32_t normal = (a + 0xfffu + ((a >> 13) & 1u) - (112u << 23)) >> 13;
  // below 2^-14 the result is a multiple of 2^-24: |x| * 2^24 < 1024 is
  // exact, and adding then removing 2^23 rounds it to an integer (RNE)
  const float f = float_of(a < 0x38800000u ? a : 0x38800000u);
  const uint32_t sub = (uint32_t)(int32_t)((f * 0x1p24f + 0x1p23f) - 0x1p23f);
  uint32_t r = a < 0x38800000u ? sub : normal;
  r = a >= 0x477ff000u ? 0x7c00u : r;  // >= 65520 rounds to infinity (and inf)
  r = a > 0x7f800000u ? 0x7e00u : r;   // NaN
  return (uint16_t)(sign | r);
}

// The 16-bit pattern whose binary32 widening is x, when there is one, so that
// a widened 16-bit value comes back bit for bit (NaN payloads included);
// otherwise x rounded to nearest even.  fp16 selects binary16, else bfloat16.
inline uint16_t narrow16(float x, bool fp16) {
  const uint32_t b = bits_of(x);
  if (!fp16) return (b & 0xffffu) == 0 ? (uint16_t)(b >> 16) : f32_to_bf16(x);
  const uint16_t r = f32_to_f16(x);
  if (bits_of(half_table().v[r]) == b) return r;
  const uint32_t a = b & 0x7fffffffu;
  if (a > 0x7f800000u && (a & 0x1fffu) == 0)  // a NaN whose payload fits 10 bits
    return (uint16_t)(((b >> 16) & 0x8000u) | 0x7c00u | ((a >> 13) & 0x3ffu));
  return r;
}

// binary32 widening of a 16-bit pattern (exact).
inline float widen16(uint16_t h, bool fp16) { return fp16 ? half_table().v[h] : bf16_to_f32(h); }

}  // namespace hc
}  // namespace zo
