// kv8_decode.cuh -- exact decoding of 8-bit latent KV codes (OCP e4m3fn or two's-complement
// int8) into f16, 16 bytes at a time, stored into 128-byte-swizzled shared-memory rows.
// Shared by the decode kernels that read 8-bit pools.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "sm103a_ptx.cuh"

namespace mla {

// Four e4m3 codes (bytes of w) -> four f16 holding the codes' values times 2^-8, exactly,
// with integer ops only.  An e4m3 code s.eeee.mmm moved to f16 bit positions s.0eeee.mmm0000000
// reads as the same significand with exponent bias 15 instead of 7, i.e. the value times
// 2^-8; e4m3 subnormals land on f16 subnormals with the same factor.  (The finite e4m3 range,
// |v| <= 448, becomes |v| <= 1.75.)  The kernel folds 2^8 back into the softmax and output
// scales.
__device__ __forceinline__ void e4m3x4_to_f16x4_scaled(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t h0 = __byte_perm(w, 0u, 0x1404);  // code 0 in bits 8-15, code 1 in bits 24-31
  const uint32_t h1 = __byte_perm(w, 0u, 0x3424);  // codes 2 and 3
  lo = (h0 & 0x80008000u) | ((h0 >> 1) & 0x3F803F80u);
  hi = (h1 & 0x80008000u) | ((h1 >> 1) & 0x3F803F80u);
}

// The same four codes through the conversion unit (cvt e4m3x2 -> f16x2, exact), scaled by
// 2^-8 on the FMA pipe (exact: a power of two, and every result stays an f16 value).  The
// dequant warps decode half of each chunk this way and half with the integer ops above, so
// that the conversion and integer pipes share the work.
__device__ __forceinline__ void e4m3x4_to_f16x4_scaled_cvt(uint32_t w, uint32_t& lo, uint32_t& hi) {
  uint32_t a, b;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(a), "=r"(b)
      : "r"(w));
  const __half2 k = __half2half2(__ushort_as_half(0x1C00));  // 2^-8
  const __half2 ra = __hmul2(*reinterpret_cast<const __half2*>(&a), k);
  const __half2 rb = __hmul2(*reinterpret_cast<const __half2*>(&b), k);
  lo = *reinterpret_cast<const uint32_t*>(&ra);
  hi = *reinterpret_cast<const uint32_t*>(&rb);
}

// Two bf16 -> two f16, round to nearest (exact for magnitudes in f16's normal range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// Decode 16 e4m3 codes (one 16-byte chunk of a row: 16 consecutive columns) into two 16-byte
// f16 chunks (values times 2^-8) of a 128-byte-swizzled row.  rbase: shared address of the
// row's 128-byte line plus 32 bytes per chunk index (chunk pair 2m, 2m+1 of the row);
// sw: the row's swizzle (row mod 8, times 16).  Half of the codes go through the conversion
// unit, half through the integer path, so that both pipes share the work.
__device__ __forceinline__ void store_f16_chunk(uint32_t rbase, int sw, uint4 w) {
  uint32_t o[8];
  e4m3x4_to_f16x4_scaled_cvt(w.x, o[0], o[1]);
  e4m3x4_to_f16x4_scaled_cvt(w.y, o[2], o[3]);
  e4m3x4_to_f16x4_scaled(w.z, o[4], o[5]);
  e4m3x4_to_f16x4_scaled(w.w, o[6], o[7]);
  // the chunk pair sits at byte offsets 32m and 32m + 16 of the unswizzled row; rbase
  // already holds row base + 32m
  const uint32_t row0 = rbase & ~127u;
  const uint32_t c0 = (rbase & 127u);
  st_shared_v4(row0 + (c0 ^ sw), o[0], o[1], o[2], o[3]);
  st_shared_v4(row0 + ((c0 + 16) ^ sw), o[4], o[5], o[6], o[7]);
}

// Four int8 codes (bytes of w) -> four f16 holding the codes' values exactly: the top bit
// of each byte is flipped (code + 128 as an unsigned byte u), u is placed under the f16
// pattern 0x64 (the value 1024 + u, exact since u < 1024) by two byte permutes, and 1152
// is subtracted in f16 (exact: the result is a small integer).
__device__ __forceinline__ void int8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(a) : "r"(x), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(b) : "r"(x), "r"(0x64646464u));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
  asm("sub.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

// Sixteen int8 codes -> sixteen f16 stored like store_f16_chunk.
__device__ __forceinline__ void store_f16_chunk_int8(uint32_t rbase, int sw, uint4 w) {
  uint32_t o[8];
  int8x4_to_f16x4(w.x, o[0], o[1]);
  int8x4_to_f16x4(w.y, o[2], o[3]);
  int8x4_to_f16x4(w.z, o[4], o[5]);
  int8x4_to_f16x4(w.w, o[6], o[7]);
  const uint32_t row0 = rbase & ~127u;
  const uint32_t c0 = (rbase & 127u);
  st_shared_v4(row0 + (c0 ^ sw), o[0], o[1], o[2], o[3]);
  st_shared_v4(row0 + ((c0 + 16) ^ sw), o[4], o[5], o[6], o[7]);
}

}  // namespace mla
