// Online tile quantizers: 1x128 (row tiles), 128x1 (column tiles, emitted
// transposed), 128x128 blocks (weights, emitted transposed) and the 1x128 ->
// 128x1 re-tiling of cached FP8 activations.
//
// "why-be.co.kr" board post 61844: the max-abs is computed online for every
// 1x128 activation tile and 128x128 weight block, a scale is derived from it
// and the tensor is quantized to E4M3; activations cached in FP8 are re-tiled
// from 1x128 to 128x1 for the backward pass, some with power-of-2 scales.
// "OMG! The most effective Deepseek Ever!": the max-abs is mapped to the FP8
// maximum (448 for E4M3).
//
// All kernels are HBM-bound streaming kernels: 16-byte vector loads/stores,
// the amax reduced with warp shuffles (row tiles) or through shared memory
// (column tiles and blocks), IEEE float32 division for the quotient (a
// multiplication by 2^-p, which rounds identically, for power-of-2 scales),
// and cvt.rn.satfinite for the E4M3 encoding.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace fp8q {

constexpr float kE4M3Max = 448.0f;
constexpr float kMinScale = 1.17549435082228750797e-38f;  // 2^-126

// two float32 -> two E4M3 codes (round to nearest even, saturate to +-448);
// `lo` lands in the low byte.
__device__ __forceinline__ uint32_t enc2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t enc4(float a, float b, float c, float d) {
  return enc2(a, b) | (enc2(c, d) << 16);
}
// two E4M3 codes (low byte first) -> exact float32 values
__device__ __forceinline__ float2 dec2(uint32_t two_codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(two_codes)));
  float lo, hi;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
  return make_float2(lo, hi);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// p = least integer >= -126 with amax <= 448 * 2^p. With amax = 1.m * 2^(E-127),
// 448 = 1.75 * 2^8: p = E - 135, plus one when 1.m > 1.75 (mantissa > 0x600000).
__device__ __forceinline__ int pow2_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int E = static_cast<int>(b >> 23);
  if (E == 0) return -126;  // zero or subnormal max-abs
  const int p = E - 135 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return p < -126 ? -126 : p;
}
__device__ __forceinline__ float exp2i(int p) {  // 2^p for -126 <= p <= 127
  return __uint_as_float(static_cast<uint32_t>(p + 127) << 23);
}

// Scale of one tile and the quotient x / s.
template <bool kPow2>
struct TileScale {
  float s;    // dequantization scale (what is stored)
  float inv;  // 2^-p for power-of-2 scales
  TileScale() = default;
  __device__ __forceinline__ TileScale(float s_, float inv_) : s(s_), inv(inv_) {}
  __device__ __forceinline__ explicit TileScale(float amax) {
    if (kPow2) {
      const int p = pow2_exponent(amax);
      s = exp2i(p);
      inv = exp2i(-p);
    } else {
      s = fmaxf(__fdiv_rn(amax, kE4M3Max), kMinScale);
      inv = 0.0f;
    }
  }
  __device__ __forceinline__ float quot(float x) const {
    return kPow2 ? __fmul_rn(x, inv) : __fdiv_rn(x, s);
  }
};

// -------------------------------------------------------------------------
// 1x128 row tiles. CTA = 256 threads = 16 half-warps; a half-warp owns one
// 128-element row tile (16 lanes x 8 bf16) and a CTA covers 64 rows of one
// K-block, each thread keeping 4 independent 16-byte loads in flight.
// -------------------------------------------------------------------------
constexpr int kRowQuantRows = 64;

template <bool kPow2>
__global__ void __launch_bounds__(256) quant_rows_1x128_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t M, int64_t ldx, uint8_t* __restrict__ q,
    int64_t ldq, float* __restrict__ sa) {
  const int kb = blockIdx.y;
  const int64_t row0 = static_cast<int64_t>(blockIdx.x) * kRowQuantRows;
  const int hw = threadIdx.x >> 4;
  const int l = threadIdx.x & 15;
  const int64_t col = static_cast<int64_t>(kb) * 128 + l * 8;
  uint4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t r = row0 + hw + 16 * i;
    v[i] = make_uint4(0u, 0u, 0u, 0u);
    if (r < M) v[i] = __ldcs(reinterpret_cast<const uint4*>(x + r * ldx + col));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t r = row0 + hw + 16 * i;
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      f[2 * j] = bf16_lo(w[j]);
      f[2 * j + 1] = bf16_hi(w[j]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    // reduce over the 16 lanes of this half-warp
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const TileScale<kPow2> ts(amax);
    uint2 out;
    out.x = enc4(ts.quot(f[0]), ts.quot(f[1]), ts.quot(f[2]), ts.quot(f[3]));
    out.y = enc4(ts.quot(f[4]), ts.quot(f[5]), ts.quot(f[6]), ts.quot(f[7]));
    if (r < M) {
      *reinterpret_cast<uint2*>(q + r * ldq + col) = out;
      if (l == 0) sa[static_cast<int64_t>(kb) * M + r] = ts.s;
    }
  }
}

// -------------------------------------------------------------------------
// Column tiles (128x1, one scale per column of a 128-row slab) or 128x128
// blocks over an input In[R][Cc]; the codes are emitted transposed:
// Out[c][r] (row stride ldo bytes). One CTA per 128x128 tile, staged in
// shared memory so that both the reads (along c) and the writes (along r)
// are contiguous.
//   kIn == 0: In is bf16 [R][ldin];
//   kIn == 1: In is E4M3 codes [R][ldin] with 1x128 row scales
//             s_in[c/128][r] (R entries per row): x = RN32(dec(q) * s_row).
// Scales: per column s_out[rb*Cc + c]; per block s_out[rb*(Cc/128) + cb].
// R % 128 == 0. Cc may be ragged only for kIn == 0 without kBlock.
// -------------------------------------------------------------------------
template <int kIn, bool kBlock, bool kPow2>
__global__ void __launch_bounds__(256) quant_cols_kernel(
    const void* __restrict__ in, int64_t R, int64_t Cc, int64_t ldin,
    const float* __restrict__ s_in, uint8_t* __restrict__ out, int64_t ldo,
    float* __restrict__ s_out) {
  constexpr int kPadBf16 = 136;  // bf16 per staged row (272 B: conflict-free columns)
  constexpr int kPadU8 = 144;    // bytes per staged row of codes
  __shared__ __align__(16) uint8_t tile_raw[kIn == 0 ? 128 * kPadBf16 * 2 : 128 * kPadU8];
  __shared__ float red[8][128];
  __shared__ float srow[128];
  __shared__ float scol[128];
  __shared__ float sinv[128];
  __shared__ float bred[4];

  const int t = threadIdx.x;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128;

  // ---- stage the tile
  if (kIn == 0) {
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(in);
    __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(tile_raw);
    const int j = t & 15;
    const bool full = c0 + 128 <= Cc;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = (t >> 4) + 16 * i;
      const __nv_bfloat16* p = src + (r0 + r) * ldin + c0 + 8 * j;
      uint4 v;
      if (full) {
        v = __ldcs(reinterpret_cast<const uint4*>(p));
      } else {
        uint16_t e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          e[k] = (c0 + 8 * j + k < Cc) ? __bfloat16_as_ushort(p[k]) : static_cast<uint16_t>(0);
        }
        v.x = e[0] | (static_cast<uint32_t>(e[1]) << 16);
        v.y = e[2] | (static_cast<uint32_t>(e[3]) << 16);
        v.z = e[4] | (static_cast<uint32_t>(e[5]) << 16);
        v.w = e[6] | (static_cast<uint32_t>(e[7]) << 16);
      }
      *reinterpret_cast<uint4*>(tile + r * kPadBf16 + 8 * j) = v;
    }
  } else {
    const uint8_t* src = static_cast<const uint8_t*>(in);
    const int j = t & 7;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = (t >> 3) + 32 * i;
      const uint4 v = __ldcs(reinterpret_cast<const uint4*>(src + (r0 + r) * ldin + c0 + 16 * j));
      *reinterpret_cast<uint4*>(tile_raw + r * kPadU8 + 16 * j) = v;
    }
    if (t < 128) srow[t] = s_in[(c0 / 128) * R + r0 + t];
  }
  __syncthreads();

  // ---- pass 1: column max-abs
  if (kIn == 0) {
    const __nv_bfloat16* tile = reinterpret_cast<const __nv_bfloat16*>(tile_raw);
    const int cp = t & 63, rg = t >> 6;  // column pair, 32-row group
    float a0 = 0.0f, a1 = 0.0f;
#pragma unroll 8
    for (int rr = 0; rr < 32; ++rr) {
      const uint32_t w =
          *reinterpret_cast<const uint32_t*>(tile + (rg * 32 + rr) * kPadBf16 + 2 * cp);
      a0 = fmaxf(a0, fabsf(bf16_lo(w)));
      a1 = fmaxf(a1, fabsf(bf16_hi(w)));
    }
    red[rg][2 * cp] = a0;
    red[rg][2 * cp + 1] = a1;
  } else {
    const int cq = t & 31, rg = t >> 5;  // column quad, 16-row group
    float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
    for (int rr = 0; rr < 16; ++rr) {
      const int r = rg * 16 + rr;
      const uint32_t w = *reinterpret_cast<const uint32_t*>(tile_raw + r * kPadU8 + 4 * cq);
      const float2 lo = dec2(w & 0xFFFFu), hi = dec2(w >> 16);
      const float s = srow[r];
      a[0] = fmaxf(a[0], fabsf(__fmul_rn(lo.x, s)));
      a[1] = fmaxf(a[1], fabsf(__fmul_rn(lo.y, s)));
      a[2] = fmaxf(a[2], fabsf(__fmul_rn(hi.x, s)));
      a[3] = fmaxf(a[3], fabsf(__fmul_rn(hi.y, s)));
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) red[rg][4 * cq + k] = a[k];
  }
  __syncthreads();

  constexpr int kGroups = kIn == 0 ? 4 : 8;
  if (t < 128) {
    float a = red[0][t];
#pragma unroll
    for (int g = 1; g < kGroups; ++g) a = fmaxf(a, red[g][t]);
    if (kBlock) {
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
      if ((t & 31) == 0) bred[t >> 5] = a;
    } else {
      const TileScale<kPow2> ts(a);
      scol[t] = ts.s;
      sinv[t] = ts.inv;
      if (c0 + t < Cc) s_out[blockIdx.y * Cc + c0 + t] = ts.s;
    }
  }
  if (kBlock) {
    __syncthreads();
    if (t < 128) {
      const float a = fmaxf(fmaxf(bred[0], bred[1]), fmaxf(bred[2], bred[3]));
      const TileScale<kPow2> ts(a);
      scol[t] = ts.s;
      sinv[t] = ts.inv;
      if (t == 0) s_out[blockIdx.y * (Cc / 128) + blockIdx.x] = ts.s;
    }
  }
  __syncthreads();

  // ---- pass 2: quantize and store transposed
  if (kIn == 0) {
    const __nv_bfloat16* tile = reinterpret_cast<const __nv_bfloat16*>(tile_raw);
    const int cp = t & 63, rg = t >> 6;
    const TileScale<kPow2> ts0(scol[2 * cp], sinv[2 * cp]);
    const TileScale<kPow2> ts1(scol[2 * cp + 1], sinv[2 * cp + 1]);
    uint32_t o0[8], o1[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      float x0[4], x1[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(
            tile + (rg * 32 + 4 * k + u) * kPadBf16 + 2 * cp);
        x0[u] = ts0.quot(bf16_lo(w));
        x1[u] = ts1.quot(bf16_hi(w));
      }
      o0[k] = enc4(x0[0], x0[1], x0[2], x0[3]);
      o1[k] = enc4(x1[0], x1[1], x1[2], x1[3]);
    }
    const int64_t ca = c0 + 2 * cp;
    if (ca < Cc) {
      uint4* d = reinterpret_cast<uint4*>(out + ca * ldo + r0 + rg * 32);
      d[0] = make_uint4(o0[0], o0[1], o0[2], o0[3]);
      d[1] = make_uint4(o0[4], o0[5], o0[6], o0[7]);
    }
    if (ca + 1 < Cc) {
      uint4* d = reinterpret_cast<uint4*>(out + (ca + 1) * ldo + r0 + rg * 32);
      d[0] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
      d[1] = make_uint4(o1[4], o1[5], o1[6], o1[7]);
    }
  } else {
    const int cq = t & 31, rg = t >> 5;
    TileScale<kPow2> ts[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) ts[k] = TileScale<kPow2>(scol[4 * cq + k], sinv[4 * cq + k]);
    uint32_t o[4][4];
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {  // 4 rows at a time -> one word per column
      float x[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = rg * 16 + 4 * k4 + u;
        const uint32_t w = *reinterpret_cast<const uint32_t*>(tile_raw + r * kPadU8 + 4 * cq);
        const float2 lo = dec2(w & 0xFFFFu), hi = dec2(w >> 16);
        const float s = srow[r];
        x[0][u] = ts[0].quot(__fmul_rn(lo.x, s));
        x[1][u] = ts[1].quot(__fmul_rn(lo.y, s));
        x[2][u] = ts[2].quot(__fmul_rn(hi.x, s));
        x[3][u] = ts[3].quot(__fmul_rn(hi.y, s));
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) o[k][k4] = enc4(x[k][0], x[k][1], x[k][2], x[k][3]);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      *reinterpret_cast<uint4*>(out + (c0 + 4 * cq + k) * ldo + r0 + rg * 16) =
          make_uint4(o[k][0], o[k][1], o[k][2], o[k][3]);
    }
  }
}

}  // namespace fp8q
