// epilogue.cuh -- moving a tcgen05 accumulator block out of TMEM.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace hmm {

// The row-mode GEMMs keep the weights on the MMA's M side, so a tcgen05.ld
// (32x32b) hands each thread of a warp one output column (its TMEM lane) over
// 32 output rows (TMEM columns).  Written out in that form every 16-byte
// store of the warp would land in 32 different rows.  Instead each warp
// passes its 32x32 fp32 block through a padded shared-memory buffer and
// continues with lane l owning the eight columns 8*(l & 3) .. +7 of the rows
// (l >> 2) + 8k, k = 0..3: a warp-wide 16-byte access then covers 8 rows x 64
// contiguous bytes.  (The weight-gradient kernel uses the same per-warp
// buffer to stage bf16 chunks for TMA stores.)
//
// Buffer: 32 rows with a stride of XS floats (16-byte aligned rows; both the
// column-wise writes and the row-group reads below are free of bank
// conflicts).
constexpr int XS = 36;
constexpr int XBUF_BYTES = 32 * XS * 4;  // per epilogue warp

// Thread t writes its 32 values, rows 0..31 of column t, down column t of the
// buffer (conflict-free: row i of the 32 threads spans all banks), so the
// buffer holds the block row-major ...
__device__ __forceinline__ void xwrite_t(float* buf, int lane, const uint32_t (&r)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) buf[i * XS + lane] = __uint_as_float(r[i]);
}
// ... and, after a __syncwarp (or a barrier with the writing warp), lane l
// reads the eight columns 8*(l & 3) .. +7 of the rows (l >> 2) + 8k.
__device__ __forceinline__ void xread(const float* buf, int lane, float (&o)[4][8]) {
  const float* s = buf + (lane >> 2) * XS + (lane & 3) * 8;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4 a = *reinterpret_cast<const float4*>(s + k * 8 * XS);
    const float4 b = *reinterpret_cast<const float4*>(s + k * 8 * XS + 4);
    o[k][0] = a.x; o[k][1] = a.y; o[k][2] = a.z; o[k][3] = a.w;
    o[k][4] = b.x; o[k][5] = b.y; o[k][6] = b.z; o[k][7] = b.w;
  }
}

// Half blocks (16 rows x 32 columns) for two warps per TMEM lane quarter:
// thread t writes its 16 values down column t of a 16-row buffer (XBUF_HALF
// bytes per warp), then lane l reads the eight columns 8*(l & 3) .. +7 of
// the rows (l >> 2) + 8k, k = 0, 1.
constexpr int XBUF_HALF = 16 * XS * 4;
__device__ __forceinline__ void xwrite_t16(float* buf, int lane, const uint32_t (&r)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) buf[i * XS + lane] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void xread16(const float* buf, int lane, float (&o)[2][8]) {
  const float* s = buf + (lane >> 2) * XS + (lane & 3) * 8;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float4 a = *reinterpret_cast<const float4*>(s + k * 8 * XS);
    const float4 b = *reinterpret_cast<const float4*>(s + k * 8 * XS + 4);
    o[k][0] = a.x; o[k][1] = a.y; o[k][2] = a.z; o[k][3] = a.w;
    o[k][4] = b.x; o[k][5] = b.y; o[k][6] = b.z; o[k][7] = b.w;
  }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float* v) {
  uint4 u;
  u.x = pack_bf16(v[0], v[1]);
  u.y = pack_bf16(v[2], v[3]);
  u.z = pack_bf16(v[4], v[5]);
  u.w = pack_bf16(v[6], v[7]);
  return u;
}

}  // namespace hmm
