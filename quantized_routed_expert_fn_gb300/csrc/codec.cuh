// codec.cuh -- b-bit affine codes -> exact bf16 integers for tensor-core fragments.
//
// Record format (gpu.rs source page, `struct Q`): codes are uint32 words,
// each weight row one little-endian bitstream, code i in bits [i*b, i*b+b).
// Groups of 64 codes share one bf16 scale and one bf16 bias (the "64-code
// quantization group" of the load.rs checks); weight = scale * code + bias.
//
// The matvec kernels feed the raw code q (an exact small integer) to a bf16
// tensor-core MMA and apply scale and bias per group in fp32 afterwards:
//   sum_i (s*q_i + beta) x_i = s * sum_i q_i x_i + beta * sum_i x_i.
//
// Work split: within a block of 128 input positions, lane quad position t
// (0..3) owns the 32 codes at positions 32t..32t+31, i.e. 4*b bytes of a row
// (codes of group t/2 of the block).  Those 32 codes are consumed as 16
// pairs; pair p supplies one bf16x2 B-fragment register (first code in the
// low half).  MMA step m (0..7) of the block uses pairs 2m and 2m+1 as the
// k-slots (2t, 2t+1) and (2t+8, 2t+9).  Which code goes to which pair is a
// free permutation (the dot product does not care) chosen so that one mask
// places both codes of a pair in the mantissas of 128.0 (bf16 0x4300):
// the B value is 128 + q*2^s, exact for q*2^s < 128.  Neither the 2^s nor
// the 128 is removed here: the activation at that k-slot is pre-scaled by
// 2^-s (exact), so the product is q*x + 128*2^-s*x, and the MMA accumulator
// starts at -128 * sum(2^-s * x) over the group, which cancels the offset.
// Unpacking is therefore only shifts and one mask-or per pair.  The
// activation fragments use the same permutation and exponents.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace moe {

constexpr uint32_t kMagic = 0x43004300u;  // bf16x2 (128, 128)

// 2^-s as a float (s = 0..7)
__host__ __device__ constexpr float pow2neg(int s) { return 1.0f / (float)(1 << s); }

template <int BITS>
struct Codec;

// 4-bit: 4 words; pair 4w+j = nibbles (j, j+4) of word w, both at shift 4j.
template <>
struct Codec<4> {
  static constexpr int kWords = 4;
  __host__ __device__ static constexpr int lo(int p) { return 8 * (p / 4) + p % 4; }
  __host__ __device__ static constexpr int hi(int p) { return lo(p) + 4; }
  __host__ __device__ static constexpr int slo(int) { return 0; }
  __host__ __device__ static constexpr int shi(int) { return 0; }
  __device__ static __forceinline__ void unpack(const uint32_t (&w)[kWords], uint32_t (&bf)[16]) {
#pragma unroll
    for (int p = 0; p < 4; p++) {
#pragma unroll
      for (int j = 0; j < 4; j++) bf[4 * p + j] = ((w[p] >> (4 * j)) & 0x000f000fu) | kMagic;
    }
  }
};

// 2-bit: 2 words; pair 8w+j = codes (j, j+8) of word w (bits 2j and 16+2j),
// read from w, w>>6 or w>>12 so that both sit at shift s <= 4.
template <>
struct Codec<2> {
  static constexpr int kWords = 2;
  __host__ __device__ static constexpr int lo(int p) { return 16 * (p / 8) + p % 8; }
  __host__ __device__ static constexpr int hi(int p) { return lo(p) + 8; }
  // pair j of a word is read from w >> 6k, k = j / 3, at shift s = 2 (j - 3k)
  __host__ __device__ static constexpr int slo(int p) { return 2 * (p % 8 - 3 * ((p % 8) / 3)); }
  __host__ __device__ static constexpr int shi(int p) { return slo(p); }
  __device__ static __forceinline__ void unpack(const uint32_t (&w)[kWords], uint32_t (&bf)[16]) {
#pragma unroll
    for (int p = 0; p < 2; p++) {
      const uint32_t src[3] = {w[p], w[p] >> 6, w[p] >> 12};
#pragma unroll
      for (int j = 0; j < 8; j++) {
        const int s = slo(j);
        const uint32_t mask = (3u << s) | (3u << (16 + s));
        bf[8 * p + j] = (src[j / 3] & mask) | kMagic;
      }
    }
  }
};

// 3-bit: 3 words = one 96-bit stream of 32 codes (codes straddle words).
// Each pair is read from a 32-bit window of the stream starting at bit o;
// the low code sits at window bit s_lo <= 4, the high code at 16 + s_hi.
// Ten windows cover all 32 codes (found by a small integer program over
// window offsets; any exact cover works).
struct Pair3 {
  int o, lo, hi, slo, shi;
};
__host__ __device__ constexpr Pair3 pair3(int p) {
  constexpr Pair3 t[16] = {{-1, 0, 5, 1, 0},   {-1, 1, 6, 4, 3},   {5, 2, 8, 1, 3},
                           {5, 3, 7, 4, 0},    {11, 4, 10, 1, 3},  {23, 9, 13, 4, 0},
                           {32, 11, 16, 1, 0}, {32, 12, 17, 4, 3}, {41, 14, 20, 1, 3},
                           {41, 15, 19, 4, 0}, {50, 18, 22, 4, 0}, {61, 21, 27, 2, 4},
                           {68, 23, 29, 1, 3}, {68, 24, 28, 4, 0}, {74, 25, 30, 1, 0},
                           {74, 26, 31, 4, 3}};
  return t[p];
}

template <>
struct Codec<3> {
  static constexpr int kWords = 3;
  __host__ __device__ static constexpr int lo(int p) { return pair3(p).lo; }
  __host__ __device__ static constexpr int hi(int p) { return pair3(p).hi; }
  __host__ __device__ static constexpr int slo(int p) { return pair3(p).slo; }
  __host__ __device__ static constexpr int shi(int p) { return pair3(p).shi; }
  __device__ static __forceinline__ uint32_t window(const uint32_t (&w)[kWords], int o) {
    if (o < 0) return w[0] << (-o);
    if (o == 0) return w[0];
    if (o < 32) return __funnelshift_r(w[0], w[1], o);
    if (o == 32) return w[1];
    if (o < 64) return __funnelshift_r(w[1], w[2], o - 32);
    if (o == 64) return w[2];
    return w[2] >> (o - 64);
  }
  __device__ static __forceinline__ void unpack(const uint32_t (&w)[kWords], uint32_t (&bf)[16]) {
#pragma unroll
    for (int p = 0; p < 16; p++) {
      const Pair3 q = pair3(p);
      const uint32_t win = window(w, q.o);
      const uint32_t mask = (7u << q.slo) | (7u << (16 + q.shi));
      bf[p] = (win & mask) | kMagic;
    }
  }
};

// The same codes in the pair order of the 4-bit codec (lo, hi and shifts of
// Codec<4>), so that records of every width can share one set of
// activation fragments: the codec a union mixing widths uses.  Pair p holds
// codes 8(p/4) + p%4 and 8(p/4) + p%4 + 4 of the lane's 32, both at shift 0.
template <int BITS>
struct CodecO4;

template <>
struct CodecO4<4> : Codec<4> {};

// 2-bit: the codes 8h..8h+7 of word w are bytes 2h (codes 8h..8h+3) and
// 2h+1 (8h+4..8h+7); a byte permute puts them at bits 0 and 16, so pair j of
// the group is one shift and one mask-or away.
template <>
struct CodecO4<2> {
  static constexpr int kWords = 2;
  __device__ static __forceinline__ void unpack(const uint32_t (&w)[kWords], uint32_t (&bf)[16]) {
#pragma unroll
    for (int g = 0; g < 4; g++) {
      const int h = g & 1;
      // result bytes: w.byte(2h), 0, w.byte(2h+1), 0 (selector 4 = the zero operand's byte 0)
      const uint32_t v = __byte_perm(w[g >> 1], 0u, (2 * h) | (4 << 4) | ((2 * h + 1) << 8) | (4 << 12));
#pragma unroll
      for (int j = 0; j < 4; j++) bf[4 * g + j] = ((v >> (2 * j)) & 0x00030003u) | kMagic;
    }
  }
};

// 3-bit: the codes 8g..8g+7 are the 24 bits of the 96-bit stream from bit
// 24g; codes 4..7 of that window move up by 4 bits (to bit 16 + 3j) with
// one shift and one bit select, then pair j is one shift and one mask-or.
template <>
struct CodecO4<3> {
  static constexpr int kWords = 3;
  __device__ static __forceinline__ void unpack(const uint32_t (&w)[kWords], uint32_t (&bf)[16]) {
    const uint32_t win[4] = {w[0], __funnelshift_r(w[0], w[1], 24), __funnelshift_r(w[1], w[2], 16), w[2] >> 8};
#pragma unroll
    for (int g = 0; g < 4; g++) {
      const uint32_t v = win[g];
      const uint32_t u = (v & 0x0000ffffu) | ((v << 4) & 0xffff0000u);
#pragma unroll
      for (int j = 0; j < 4; j++) bf[4 * g + j] = ((u >> (3 * j)) & 0x00070007u) | kMagic;
    }
  }
};

}  // namespace moe
