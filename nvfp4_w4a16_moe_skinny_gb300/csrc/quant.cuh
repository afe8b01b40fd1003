// Offline NVFP4 quantizer and repack kernels.
//
// Quantizer: formula (1) of nvfp4_skinny.h in reverse (E2M1 weights, E4M3
// group-16 scales, fp32 global scale -- gemma-cuda-hybrid README, "Everything
// it has / Inference engine").  The codes are the round-to-nearest-even codes
// of the exact quotients bmax / (6 g) and w / (e4m3(s) g): each quotient is one
// float64 division by an exact divisor, narrowed to fp32 with round-to-odd and
// handed to the hardware round-to-nearest-even saturating converter.  The
// grids' midpoints have at most 5 significant bits and a quotient of fp32
// values that is not a midpoint lies at least 2^-32 (relative) from every
// midpoint, so one float64 rounding cannot move it across one; round-to-odd to
// 24 bits followed by rounding to at most 5 bits is the correctly rounded result.
//
// Repack: canonical bytes -> the tiled layout documented in nvfp4_skinny.h
// ("offline weight repack into mma-fragment order" -- gemma-cuda-hybrid README,
// "NVFP4-specific").
#pragma once

#include "common.cuh"

namespace nvfp4 {

// An input element as fp32: fp32 weights, or bf16 activations (exact).
__device__ __forceinline__ float in_value(float v) { return v; }
__device__ __forceinline__ float in_value(uint16_t v) { return __uint_as_float(static_cast<uint32_t>(v) << 16); }

// 16 consecutive input elements (16-element aligned) as fp32.
__device__ __forceinline__ void load16(const float* __restrict__ p, float (&v)[16]) {
  const float4* src = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = src[i];
    v[4 * i] = f.x, v[4 * i + 1] = f.y, v[4 * i + 2] = f.z, v[4 * i + 3] = f.w;
  }
}
__device__ __forceinline__ void load16(const uint16_t* __restrict__ p, float (&v)[16]) {
  const uint4* src = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 u = src[i];
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * i + 2 * j] = __uint_as_float(w4[j] << 16);
      v[8 * i + 2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
    }
  }
}

// Per-matrix amax of |w| as the bit pattern of a non-negative float: for such
// floats unsigned integer order equals numeric order, so atomicMax is exact and
// order-independent.  T: float (weights) or uint16_t (bf16 activations, one
// "matrix" per token row).
template <typename T>
__global__ void quant_amax_kernel(const T* __restrict__ w, size_t per_matrix, unsigned* __restrict__ amax_bits) {
  const int e = blockIdx.y;
  const T* src = w + static_cast<size_t>(e) * per_matrix;
  unsigned best = 0;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < per_matrix;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const unsigned b = __float_as_uint(fabsf(in_value(src[i])));
    best = b > best ? b : best;
  }
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned o = __shfl_xor_sync(0xffffffffu, best, off);
    best = o > best ? o : best;
  }
  __shared__ unsigned warp_best[32];
  if ((threadIdx.x & 31) == 0) warp_best[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned b = 0;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) b = warp_best[i] > b ? warp_best[i] : b;
    atomicMax(&amax_bits[e], b);
  }
}

__device__ __forceinline__ uint32_t e4m3_code_rne(float t) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(t));  // t -> low byte
  return r & 0xFF;
}

// (hi, lo) -> one byte of two E2M1 codes: lo in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2_code_rne(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  // keep the sign of values that round to zero (-tiny -> code 8)
  r &= 0x77u;
  r |= (__float_as_uint(lo) >> 31) << 3;
  r |= (__float_as_uint(hi) >> 31) << 7;
  return r;
}

// double -> float, round to odd: truncate, and set the lowest significand bit
// when the truncation was inexact.  A later round-to-nearest-even to 22 or fewer
// significant bits then equals rounding the double directly.
__device__ __forceinline__ float f64_to_f32_round_odd(double x) {
  const float f = __double2float_rz(x);
  return static_cast<double>(f) == x ? f : __uint_as_float(__float_as_uint(f) | 1u);
}

__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 0xF, m = c & 7;
  const float mag = e == 0 ? static_cast<float>(m) * 0.001953125f  // m/8 * 2^-6
                           : __uint_as_float(((e + 120u) << 23) | (m << 20));  // (1+m/8) * 2^(e-7)
  return (c & 0x80) ? -mag : mag;
}

// One 16-element group under global scale g: its E4M3 scale code and its eight
// code bytes (two words, column 2i in the low nibble of byte i).
//
// The scale code comes from one float64 division (the exact quotient's
// decision, as above).  An element's code is the E2M1 rounding of the exact
// quotient w / d, d = e4m3(s) * g; it is taken in fp32 where that is provably the
// same: q = |w| * fp32(1/d) is within 2^-23 (relative) of the exact quotient, so
// the exact quotient lies in [q (1 - 2^-20), q (1 + 2^-20)] (both products
// rounded in fp32, still enclosing it); rounding is monotonic, so when both ends
// round to the same code that code is the exact quotient's.  Otherwise (a
// quotient within 2^-20 of a rounding midpoint) the element takes the float64
// division.
__device__ __forceinline__ void quantize_group16(const float (&v)[16], float g, uint32_t& s_code,
                                                 uint32_t (&packed)[2]) {
  float bmax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
  s_code = 0;
  double denom = 0.0;
  if (g > 0.f) {
    const double t = static_cast<double>(bmax) / (6.0 * static_cast<double>(g));  // exact divisor
    s_code = e4m3_code_rne(f64_to_f32_round_odd(t));
    denom = static_cast<double>(e4m3_value(s_code)) * static_cast<double>(g);      // exact product
  }
  packed[0] = packed[1] = 0u;
  if (!(denom > 0.0)) return;
  const float inv = static_cast<float>(1.0 / denom);
  const bool fast = inv < 1e30f;  // (an fp32 1/d far from overflow)
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float lo = v[2 * i], hi = v[2 * i + 1];
    uint32_t code = 0;
    bool exact = !fast;
    if (fast) {
      const float ql = fabsf(lo) * inv, qh = fabsf(hi) * inv;
      const uint32_t c_dn = e2m1x2_code_rne(ql * 0.99999904632568359375f, qh * 0.99999904632568359375f);
      const uint32_t c_up = e2m1x2_code_rne(ql * 1.00000095367431640625f, qh * 1.00000095367431640625f);
      exact = c_dn != c_up;
      code = c_dn;
    }
    if (exact) {
      const float ql = f64_to_f32_round_odd(fabs(static_cast<double>(lo)) / denom);
      const float qh = f64_to_f32_round_odd(fabs(static_cast<double>(hi)) / denom);
      code = e2m1x2_code_rne(ql, qh);
    }
    // the signs of w (kept for codes that round to zero)
    code |= ((__float_as_uint(lo) >> 31) << 3) | ((__float_as_uint(hi) >> 31) << 7);
    packed[i >> 2] |= code << (8 * (i & 3));
  }
}

// One thread per 16-element group.
template <typename T>
__global__ void quant_groups_kernel(const T* __restrict__ w, int n, int k, const unsigned* __restrict__ amax_bits,
                                    uint8_t* __restrict__ nibbles, uint8_t* __restrict__ scales,
                                    float* __restrict__ global_scale) {
  const int e = blockIdx.y;
  const int groups_per_row = k / 16;
  const size_t groups = static_cast<size_t>(n) * groups_per_row;
  const float amax = __uint_as_float(amax_bits[e]);
  const float g = __fdiv_rn(amax, 2688.0f);
  if (blockIdx.x == 0 && threadIdx.x == 0) global_scale[e] = g;
  for (size_t gi = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; gi < groups;
       gi += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float v[16];
    load16(w + (static_cast<size_t>(e) * n * k) + gi * 16, v);
    uint32_t s_code, packed[2];
    quantize_group16(v, g, s_code, packed);
    uint2* dst = reinterpret_cast<uint2*>(nibbles + (static_cast<size_t>(e) * n * k) / 2 + gi * 8);
    *dst = make_uint2(packed[0], packed[1]);
    scales[static_cast<size_t>(e) * groups + gi] = static_cast<uint8_t>(s_code);
  }
}

// Activation rows (bf16 [m, k]) to NVFP4 with one global scale per row, in one
// grid: CTA r reduces row r's amax, then quantizes its 16-element groups.  The
// rows may come from the previous grid (programmatic dependent launch).
constexpr int kActQuantThreads = 256;
__global__ void __launch_bounds__(kActQuantThreads) quant_act_rows_kernel(
    const uint16_t* __restrict__ x, int k, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
    float* __restrict__ global_scale) {
  pdl_wait();
  pdl_launch_dependents();
  const int r = blockIdx.x;
  const uint16_t* row = x + static_cast<size_t>(r) * k;
  const int groups = k / 16;
  // the row's amax, 16 elements (two 16-byte loads) per thread and step
  unsigned best = 0;  // as in quant_amax_kernel: the largest |x| bit pattern
  for (int gi = threadIdx.x; gi < groups; gi += blockDim.x) {
    float v[16];
    load16(row + gi * 16, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) best = max(best, __float_as_uint(fabsf(v[i])));
  }
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned o = __shfl_xor_sync(0xffffffffu, best, off);
    best = o > best ? o : best;
  }
  __shared__ unsigned warp_best[kActQuantThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_best[threadIdx.x >> 5] = best;
  __syncthreads();
  unsigned amax = 0;
#pragma unroll
  for (int i = 0; i < kActQuantThreads / 32; ++i) amax = warp_best[i] > amax ? warp_best[i] : amax;
  const float g = __fdiv_rn(__uint_as_float(amax), 2688.0f);
  if (threadIdx.x == 0) global_scale[r] = g;
  for (int gi = threadIdx.x; gi < groups; gi += blockDim.x) {
    float v[16];
    load16(row + gi * 16, v);
    uint32_t s_code, packed[2];
    quantize_group16(v, g, s_code, packed);
    *reinterpret_cast<uint2*>(codes + static_cast<size_t>(r) * (k / 2) + gi * 8) = make_uint2(packed[0], packed[1]);
    scales[static_cast<size_t>(r) * groups + gi] = static_cast<uint8_t>(s_code);
  }
}

// The 16-byte output chunk c (36 chunks per 576-byte tile) of a repacked stack.
// Tile t of a matrix is (group G, 64-column chunk kc, 16-row block r) with
// t = (G * kc_count + kc) * 4 + r (layout version 2: the four tiles of a 64-row
// group and one chunk are contiguous).  Chunks 0..31 are the A-fragment bytes
// (lane 4g + t of the m16n8k16 A operand, four 16-column k-steps), 32..35 the
// tile's 64 scale bytes.  A negative scale is folded into the signs of its 16
// codes.  The device repack and the host repack both call this.
__host__ __device__ inline void repack_chunk(const uint8_t* __restrict__ nib, const uint8_t* __restrict__ sc, int n,
                                             int k, int ng, int kc_count, bool gated, size_t c, uint32_t words[4]) {
  const int kh = k / 2, kg = k / 16, inter = n / 2;
  const size_t tiles_per_matrix = static_cast<size_t>(ng) * kc_count * 4;
  const size_t tile = c / 36;
  const int part = static_cast<int>(c % 36);
  const int e = static_cast<int>(tile / tiles_per_matrix);
  const size_t tm = tile % tiles_per_matrix;
  const int r = static_cast<int>(tm & 3);
  const int grp = static_cast<int>((tm >> 2) / kc_count), kc = static_cast<int>((tm >> 2) % kc_count);
  const int rb = grp * 4 + r;
  const uint8_t* nib_e = nib + static_cast<size_t>(e) * n * kh;
  const uint8_t* sc_e = sc + static_cast<size_t>(e) * n * kg;
  // source row of destination row `dr`, or -1 for padding
  auto src_row = [&](int dr) -> int {
    if (gated) {
      const int blk = dr >> 4, j = dr & 15;
      return (j < 8) ? (8 * blk + j) : (inter + 8 * blk + (j - 8));
    }
    return dr < n ? dr : -1;
  };
  if (part < 32) {
    const int g = part >> 2, t = part & 3;
    for (int kt = 0; kt < 4; ++kt) {
      uint32_t wv = 0;
      for (int rr = 0; rr < 4; ++rr) {
        const int dr = rb * 16 + g + 8 * (rr & 1);
        const int col = kc * 64 + kt * 16 + 2 * t + 8 * (rr >> 1);
        const int sr = src_row(dr);
        uint32_t byte = 0;
        if (sr >= 0 && col < k) {
          byte = nib_e[static_cast<size_t>(sr) * kh + col / 2];
          if (sc_e[static_cast<size_t>(sr) * kg + col / 16] & 0x80) byte ^= 0x88u;  // fold a negative scale
        }
        wv |= byte << (8 * rr);
      }
      words[kt] = wv;
    }
  } else {
    // scale bytes 16*(part-32) .. +15 of the 64-byte scale block: byte j -> g = j/8, kt = (j%8)/2, h = j%2
    for (int wi = 0; wi < 4; ++wi) {
      uint32_t wv = 0;
      for (int bi = 0; bi < 4; ++bi) {
        const int j = 16 * (part - 32) + 4 * wi + bi;
        const int g = j >> 3, kt = (j & 7) >> 1, h = j & 1;
        const int dr = rb * 16 + g + 8 * h;
        const int grp16 = kc * 4 + kt;
        const int sr = src_row(dr);
        uint32_t byte = 0;
        if (sr >= 0 && grp16 < kg) byte = sc_e[static_cast<size_t>(sr) * kg + grp16] & 0x7Fu;
        wv |= byte << (8 * bi);
      }
      words[wi] = wv;
    }
  }
}

// One thread per 16-byte output chunk.
__global__ void repack_kernel(const uint8_t* __restrict__ nib, const uint8_t* __restrict__ sc, int n, int k, int ng,
                              int kc_count, bool gated, size_t tiles_total, uint8_t* __restrict__ out) {
  const size_t chunks = tiles_total * 36;
  for (size_t c = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; c < chunks;
       c += static_cast<size_t>(gridDim.x) * blockDim.x) {
    uint32_t words[4];
    repack_chunk(nib, sc, n, k, ng, kc_count, gated, c, words);
    reinterpret_cast<uint4*>(out)[c] = make_uint4(words[0], words[1], words[2], words[3]);
  }
}

}  // namespace nvfp4
