// common.cuh -- device helpers shared by the apply and sample kernels of liblp.so:
// element-type traits for 16-byte vectors, the bitmask bit window of a vector, an
// order-preserving integer key for float logits, Philox4x32-10 and Gumbel noise.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lp.h"

namespace lp {

constexpr uint32_t kFullWarp = 0xffffffffu;

// ------------------------------------------------------------------ elements

// A 16-byte vector holds 4 float32 or 8 half/bfloat16 elements.
template <int DT>
struct Elt;

template <>
struct Elt<LP_F32> {
  static constexpr int kBytes = 4;
  static constexpr int kPerVec = 4;
  static constexpr uint32_t kLowKeyBit = 0;  // lowest key bit that can differ
  __device__ static __forceinline__ float get(const uint4& v, int e) {
    const uint32_t w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    return __uint_as_float(w);
  }
  __device__ static __forceinline__ float load1(const char* p) {
    return __uint_as_float(*reinterpret_cast<const uint32_t*>(p));
  }
  __device__ static __forceinline__ void store1(char* p, uint32_t bits) {
    *reinterpret_cast<uint32_t*>(p) = bits;
  }
  __device__ static __forceinline__ uint32_t bits1(const char* p) {
    return *reinterpret_cast<const uint32_t*>(p);
  }
  // keep element e of v where bit e of keep is set, else the fill pattern
  __device__ static __forceinline__ uint4 blend(const uint4& v, uint32_t keep, uint32_t fill) {
    uint4 r;
    r.x = (keep & 1u) ? v.x : fill;
    r.y = (keep & 2u) ? v.y : fill;
    r.z = (keep & 4u) ? v.z : fill;
    r.w = (keep & 8u) ? v.w : fill;
    return r;
  }
  __device__ static __forceinline__ uint32_t fill_word(uint32_t fill) { return fill; }
};

// 16-bit element helpers: element e of a vector is half (e & 1) of word e >> 1.
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint32_t keep_mask16(uint32_t keep, int i) {
  return ((keep >> (2 * i)) & 1u ? 0x0000ffffu : 0u) |
         ((keep >> (2 * i + 1)) & 1u ? 0xffff0000u : 0u);
}

__device__ __forceinline__ uint4 blend16(const uint4& v, uint32_t keep, uint32_t fill2) {
  uint4 r;
  uint32_t m;
  m = keep_mask16(keep, 0); r.x = (v.x & m) | (fill2 & ~m);
  m = keep_mask16(keep, 1); r.y = (v.y & m) | (fill2 & ~m);
  m = keep_mask16(keep, 2); r.z = (v.z & m) | (fill2 & ~m);
  m = keep_mask16(keep, 3); r.w = (v.w & m) | (fill2 & ~m);
  return r;
}

template <>
struct Elt<LP_BF16> {
  static constexpr int kBytes = 2;
  static constexpr int kPerVec = 8;
  static constexpr uint32_t kLowKeyBit = 16;
  __device__ static __forceinline__ float get(const uint4& v, int e) {
    const uint32_t w = word_of(v, e >> 1);
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
  }
  __device__ static __forceinline__ float load1(const char* p) {
    return __uint_as_float(uint32_t(*reinterpret_cast<const uint16_t*>(p)) << 16);
  }
  __device__ static __forceinline__ void store1(char* p, uint32_t bits) {
    *reinterpret_cast<uint16_t*>(p) = uint16_t(bits);
  }
  __device__ static __forceinline__ uint32_t bits1(const char* p) {
    return *reinterpret_cast<const uint16_t*>(p);
  }
  __device__ static __forceinline__ uint4 blend(const uint4& v, uint32_t keep, uint32_t fill) {
    return blend16(v, keep, fill_word(fill));
  }
  __device__ static __forceinline__ uint32_t fill_word(uint32_t fill) {
    return (fill & 0xffffu) | (fill << 16);
  }
};

template <>
struct Elt<LP_F16> {
  static constexpr int kBytes = 2;
  static constexpr int kPerVec = 8;
  static constexpr uint32_t kLowKeyBit = 13;
  __device__ static __forceinline__ float half_bits_to_float(uint32_t h) {
    float f;
    asm("{ .reg .f16 t; mov.b16 t, %1; cvt.f32.f16 %0, t; }" : "=f"(f) : "h"(uint16_t(h)));
    return f;
  }
  __device__ static __forceinline__ float get(const uint4& v, int e) {
    const uint32_t w = word_of(v, e >> 1);
    return half_bits_to_float((e & 1) ? (w >> 16) : (w & 0xffffu));
  }
  __device__ static __forceinline__ float load1(const char* p) {
    return half_bits_to_float(*reinterpret_cast<const uint16_t*>(p));
  }
  __device__ static __forceinline__ void store1(char* p, uint32_t bits) {
    *reinterpret_cast<uint16_t*>(p) = uint16_t(bits);
  }
  __device__ static __forceinline__ uint32_t bits1(const char* p) {
    return *reinterpret_cast<const uint16_t*>(p);
  }
  __device__ static __forceinline__ uint4 blend(const uint4& v, uint32_t keep, uint32_t fill) {
    return blend16(v, keep, fill_word(fill));
  }
  __device__ static __forceinline__ uint32_t fill_word(uint32_t fill) {
    return (fill & 0xffffu) | (fill << 16);
  }
};

// ------------------------------------------------------------ vector max

// Max over the elements e of a vector with bit e of `keep` set (-inf if none).
// 16-bit types take the max of the element pairs with one packed instruction
// per pair of words; masked elements are first replaced by -inf.
template <int DT>
struct VecMax;

template <>
struct VecMax<LP_F32> {
  __device__ static __forceinline__ float run(const uint4& v, uint32_t keep) {
    const float x0 = (keep & 1u) ? __uint_as_float(v.x) : -INFINITY;
    const float x1 = (keep & 2u) ? __uint_as_float(v.y) : -INFINITY;
    const float x2 = (keep & 4u) ? __uint_as_float(v.z) : -INFINITY;
    const float x3 = (keep & 8u) ? __uint_as_float(v.w) : -INFINITY;
    return fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
  }
};

template <>
struct VecMax<LP_BF16> {
  static constexpr uint32_t kNegInf2 = 0xff80ff80u;
  __device__ static __forceinline__ uint32_t mx(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
  }
  __device__ static __forceinline__ float run(const uint4& v, uint32_t keep) {
    uint32_t w0 = v.x, w1 = v.y, w2 = v.z, w3 = v.w;
    if (keep != 0xffu) {
      uint32_t m;
      m = keep_mask16(keep, 0); w0 = (w0 & m) | (kNegInf2 & ~m);
      m = keep_mask16(keep, 1); w1 = (w1 & m) | (kNegInf2 & ~m);
      m = keep_mask16(keep, 2); w2 = (w2 & m) | (kNegInf2 & ~m);
      m = keep_mask16(keep, 3); w3 = (w3 & m) | (kNegInf2 & ~m);
    }
    const uint32_t t = mx(mx(w0, w1), mx(w2, w3));
    return fmaxf(__uint_as_float(t << 16), __uint_as_float(t & 0xffff0000u));
  }
};

template <>
struct VecMax<LP_F16> {
  static constexpr uint32_t kNegInf2 = 0xfc00fc00u;
  __device__ static __forceinline__ uint32_t mx(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
  }
  __device__ static __forceinline__ float run(const uint4& v, uint32_t keep) {
    uint32_t w0 = v.x, w1 = v.y, w2 = v.z, w3 = v.w;
    if (keep != 0xffu) {
      uint32_t m;
      m = keep_mask16(keep, 0); w0 = (w0 & m) | (kNegInf2 & ~m);
      m = keep_mask16(keep, 1); w1 = (w1 & m) | (kNegInf2 & ~m);
      m = keep_mask16(keep, 2); w2 = (w2 & m) | (kNegInf2 & ~m);
      m = keep_mask16(keep, 3); w3 = (w3 & m) | (kNegInf2 & ~m);
    }
    const uint32_t t = mx(mx(w0, w1), mx(w2, w3));
    return fmaxf(Elt<LP_F16>::half_bits_to_float(t & 0xffffu),
                 Elt<LP_F16>::half_bits_to_float(t >> 16));
  }
};

// ------------------------------------------------------------- bitmask bits

// Bits [0, n) of the result are the bitmask bits of tokens j .. j+n-1 of one
// bitmask row (n <= 8, j >= 0).  Only words that hold a token < limit are read;
// bits of tokens >= limit come back SET (keep), so they never mask anything.
__device__ __forceinline__ uint32_t mask_bits(const uint32_t* __restrict__ row, int64_t j, int n,
                                              int64_t limit) {
  const uint32_t all = (1u << n) - 1u;
  if (j >= limit) return all;
  const int64_t w = j >> 5;
  const int sh = int(j & 31);
  uint64_t two = __ldg(row + w);
  if (sh + n > 32 && (w + 1) * 32 < limit) two |= uint64_t(__ldg(row + w + 1)) << 32;
  uint32_t bits = uint32_t(two >> sh) & all;
  const int64_t valid = limit - j;
  if (valid < n) bits |= all & ~((1u << valid) - 1u);
  return bits;
}

// ----------------------------------------------------------- ordering keys

// Order-preserving map from float to uint32: a < b (as floats) iff key(a) <
// key(b).  -0 is folded onto +0, so equal values share one key.
__device__ __forceinline__ uint32_t fkey(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// ------------------------------------------------------------------- Philox

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two 32x32->64
// multiplies by the round constants, the high halves XORed with the other two
// counter words and the round key; the key takes a Weyl step between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k.x += 0x9E3779B9u;
      k.y += 0xBB67AE85u;
    }
    const uint32_t lo0 = c.x * 0xD2511F53u, hi0 = __umulhi(c.x, 0xD2511F53u);
    const uint32_t lo1 = c.z * 0xCD9E8D57u, hi1 = __umulhi(c.z, 0xCD9E8D57u);
    c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
  }
  return c;
}

// Gumbel noise from one 32-bit word: u = ((x >> 9) + 0.5) * 2^-23 lies in
// [2^-24, 1 - 2^-24] and is exact in float; g = -log(-log u).
__device__ __forceinline__ float gumbel_from_word(uint32_t x) {
  const float u = (float(x >> 9) + 0.5f) * 1.1920928955078125e-07f;
  return -logf(-logf(u));
}

// 2^x by the hardware approximation (one MUFU op, relative error below 2^-22);
// used for softmax sums and masses, never for the Gumbel noise.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Upper bound of gumbel_from_word over all words (u = 1 - 2^-24 gives 16.6355;
// the margin absorbs float rounding in the two logarithms).
constexpr float kGumbelMax = 16.64f;
// Lower bound (u = 2^-24 gives -2.8116), with margin.
constexpr float kGumbelMin = -2.82f;

}  // namespace lp
