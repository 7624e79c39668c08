// kv8_decode.cuh -- exact decoding of int8 latent KV codes (two's complement) into f16, 16
// bytes at a time, stored into 128-byte-swizzled shared-memory rows, for the int8 decode
// kernel (an e4m3 pool needs no decode: its kernel multiplies the codes as they are).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "sm103a_ptx.cuh"

namespace mla {

// Two bf16 -> two f16, round to nearest (exact for magnitudes in f16's normal range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
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

// Sixteen int8 codes (one 16-byte chunk of a row: 16 consecutive columns) -> two 16-byte
// f16 chunks of a 128-byte-swizzled row.  rbase: shared address of the row's 128-byte line
// plus 32 bytes per chunk index (chunk pair 2m, 2m+1 of the row); sw: the row's swizzle
// (row mod 8, times 16).
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
