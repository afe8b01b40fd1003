// Device helpers shared by the NVFP4 skinny kernels (sm_103a only).
//
// Inline PTX for: mbarriers with bounded waits, 1-D bulk copies (TMA engine)
// global -> shared with an L2 evict-first hint, the hardware E2M1/E4M3
// converters, and the m16n8k16 f16 tensor-core MMA.
#pragma once

#include <cstdint>
#include <cuda.h>  // CUtensorMap (the type only; the library does not link the driver API)
#include <cuda_runtime.h>

#include "nvfp4_skinny.h"

namespace nvfp4 {

constexpr int kTileRows = 16;       // rows per repacked tile
constexpr int kGroupRows = 64;      // rows per group of four tiles (the streaming unit)
constexpr int kTileK = 64;          // K columns per repacked tile
constexpr int kTileBytes = 576;     // 512 B of nibbles + 64 B of scales
constexpr int kTileNibBytes = 512;

// Device error word of the kernels of one translation unit (each unit of the
// library has its own copy; nvfp4_device_error() reads them all).  Bit 0: an
// mbarrier wait ran out of time.
static __device__ unsigned int g_device_error = 0;

constexpr unsigned kErrWaitTimeout = 1u;
// ~1 s at 2 GHz: far above any legitimate wait for a bulk copy.
constexpr long long kWaitCycles = 2000000000ll;

// Word 0 of the counter-based generator Philox4x32-10 (Salmon, Moraes, Dror,
// Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011) for the counter
// (c0, c1, 0, 0) and key (k0, k1): ten rounds, each two 32x32 -> 64-bit products
// by the generator's multipliers, the high halves crossed and XORed with the
// other words and the round key, the key bumped by the Weyl increments between
// rounds.
__device__ __forceinline__ uint32_t philox4x32_10_word0(uint32_t c0, uint32_t c1, uint32_t k0, uint32_t k1) {
  uint32_t c2 = 0, c3 = 0;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) k0 += 0x9E3779B9u, k1 += 0xBB67AE85u;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0, c1 = lo1, c2 = n2, c3 = lo0;
  }
  return c0;
}

// Standard Gumbel noise -log(-log u) from a 32-bit draw, u = ((w >> 9) + 0.5) / 2^23:
// (w >> 9) + 0.5 needs 24 significant bits, so u is exact in fp32 and lies
// strictly inside (0, 1).
__device__ __forceinline__ float gumbel_from_bits(uint32_t w) {
  const float u = (static_cast<float>(w >> 9) + 0.5f) * (1.0f / 8388608.0f);
  return -logf(-logf(u));
}

// Bytes of dynamic shared memory this launch was given.
__device__ __forceinline__ uint32_t dynamic_smem_bytes() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: a thread whose phase is not complete sleeps
// in hardware until the phase completes or about `ns` nanoseconds pass.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Bounded warp-collective wait (all 32 lanes call it) for the phase with the
// given parity to complete.  Every lane observes the completion itself (so the
// bulk-copied bytes are visible to it) and all lanes return the same answer:
// false, with kErrWaitTimeout recorded, if the phase did not complete within
// `limit` SM clock cycles (the kernels: kWaitCycles).  The first probe does not
// suspend: a stage is usually full already.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, long long limit = kWaitCycles) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  const long long t0 = clock64();
  while (true) {
    if (__all_sync(0xffffffffu, mbar_try_wait_sleep(bar, parity, 1u << 20))) return true;
    if (__any_sync(0xffffffffu, clock64() - t0 > limit)) {
      if ((threadIdx.x & 31) == 0) atomicOr(&g_device_error, kErrWaitTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// The same three operations on shared-space addresses (no address conversion).
__device__ __forceinline__ void mbar_arrive_expect_tx_s(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_g2s_s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d_s(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "l"(policy)
      : "memory");
}

// 1-D bulk copy global -> shared (TMA engine); completion is counted on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 4-D tiled tensor copy global -> shared (TMA engine) of the box at
// coordinates (c0, c1, c2, c3) of `map`; completion is counted on `bar`.  The
// destination is 128-byte aligned; c0 (the innermost coordinate) is 0 for every
// copy of this library, so the 16-byte rule on it always holds.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Four E2M1 pairs (the four bytes of w) -> four f16x2 (low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Scale byte j of `w` (an E4M3 code with its sign bit clear) as an f16x2 with
// the value in both halves, times 2^-8: the code's 7 magnitude bits moved to
// f16 bits 7..13 read as an f16 equal e4m3 * 2^-8 for normals and subnormals
// alike.  PRMT + shift on the integer pipe keeps the conversion pipe free.
template <int J>
__device__ __forceinline__ uint32_t scale_pair_x2(uint32_t w) {
  constexpr uint32_t sel = (J << 12) | (4 << 8) | (J << 4) | 4;  // bytes [0, sJ, 0, sJ]
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(w), "n"(sel));
  return r >> 1;
}

// Scale bytes 0 and 1 of the low half of `w` as f16x2 (s0 -> low, s1 -> high), times 2^-8.
__device__ __forceinline__ uint32_t scale_lohi_x2(uint32_t w) {
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(w), "n"(0x1404));  // bytes [0, s0, 0, s1]
  return r >> 1;
}

// Scale bytes J0 and J1 of `w` as an f16x2 (byte J0 -> low half, J1 -> high),
// times 2^-8: PRMT places the two codes in bytes 1 and 3 of zeroed halves, then
// a multiply by 128 (an integer multiply, off the ALU pipe) moves them to bits
// 7..13 of each half.
template <int J0, int J1>
__device__ __forceinline__ uint32_t scale_pair_lohi(uint32_t w) {
  constexpr uint32_t sel = (4 << 12) | (J1 << 8) | (4 << 4) | J0;  // bytes [sJ0, 0, sJ1, 0]
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(w), "n"(sel));
  uint32_t d;
  asm("mul.lo.u32 %0, %1, 128;" : "=r"(d) : "r"(r));
  return d;
}

// (a * [s.lo, s.lo], b * [s.hi, s.hi]): each half of `s` scales a whole f16x2.
__device__ __forceinline__ void hmul2_bcast(uint32_t a, uint32_t b, uint32_t s, uint32_t& ra, uint32_t& rb) {
  asm("{\n\t.reg .b16 l, h;\n\t.reg .b32 ll, hh;\n\t"
      "mov.b32 {l, h}, %2;\n\tmov.b32 ll, {l, l};\n\tmov.b32 hh, {h, h};\n\t"
      "mul.rn.f16x2 %0, %3, ll;\n\tmul.rn.f16x2 %1, %4, hh;\n\t}"
      : "=r"(ra), "=r"(rb)
      : "r"(s), "r"(a), "r"(b));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// f32 += f16 * f16 (mixed-precision fma; the products of an E2M1 value and an
// 8-significant-bit activation are exact in f32).
__device__ __forceinline__ float fma_f16lo(uint32_t a2, uint32_t b2, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %3;\n\t}"
      : "=f"(d)
      : "r"(a2), "r"(b2), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_f16hi(uint32_t a2, uint32_t b2, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, ah, bh, %3;\n\t}"
      : "=f"(d)
      : "r"(a2), "r"(b2), "f"(c));
  return d;
}

__device__ __forceinline__ float f16lo_to_f32(uint32_t h2) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}
__device__ __forceinline__ float f16hi_to_f32(uint32_t h2) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}

// D += A * B, m16n8k16, f16 operands, f32 accumulate.
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

// Programmatic dependent launch.  wait: block until the grids this one depends
// on have completed and their memory is visible (a no-op for a normal launch).
// launch_dependents: let the next grid in the stream start its prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_addr(p)));
  return v;
}
__device__ __forceinline__ uint2 lds64(const void* p) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(smem_addr(p)));
  return v;
}
__device__ __forceinline__ uint32_t lds32(const void* p) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)));
  return v;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// float -> bf16 bits, round to nearest even (finite inputs).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

// Two floats to an f16x2 (lo in the low half), each rounded to nearest even, in
// one conversion.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Power-of-two activation rescale: the exponent s with amax * 2^s in [2^14, 2^15),
// so every bf16 value of the row lands in f16's normal range, or is still exact
// in f16's subnormal range down to 2^-31 of the row maximum.  0 for an all-zero
// row; clamped to [-100, 100] so 2^s and the epilogue's 2^(8-s) stay normal fp32.
__device__ __forceinline__ int pow2_rescale_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF);  // biased exponent
  const int s = 141 - e;  // amax in [2^(e-127), 2^(e-126)) -> times 2^(141-e) in [2^14, 2^15)
  return s > 100 ? 100 : (s < -100 ? -100 : s);
}

__device__ __forceinline__ float exp2i(int e) {
  // 2^e for e in [-126, 127]; callers keep e in range.
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

}  // namespace nvfp4
