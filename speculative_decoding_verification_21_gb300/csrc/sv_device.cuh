// sv_device.cuh -- device-side building blocks of libspecverify (sm_103a).
//
// Philox4x32-10 and the uniform/Gumbel mapping, logit loads, and the small
// reductions every kernel uses.  Written for the GPU path only; the CPU oracle
// has its own independent implementations.
#pragma once

#include <cstdint>
#include <limits>

#include <cuda_runtime.h>

#include "specverify.h"

namespace sv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kInf = std::numeric_limits<float>::infinity();

// --------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11): per round, two 32x32->64-bit products of counter words
// 0 and 2 with the round multipliers; the high halves are xored with counter
// words 1 and 3 and the round key; the key advances by the Weyl constants.
// --------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Counter for tag/position/batch row/round; c0 selects the vocabulary block.
__device__ __forceinline__ uint4 sv_counter(uint32_t c0, uint32_t tag, uint32_t pos, uint32_t b,
                                            uint64_t round) {
  return make_uint4(c0, (tag << 24) | (pos & 0xFFFFFFu), b, (uint32_t)round);
}

// 23 random bits -> odd multiple of 2^-24, strictly inside (0,1); exact in fp32.
__device__ __forceinline__ float sv_u01(uint32_t x) {
  return __uint2float_rn(2u * (x >> 9) + 1u) * 0x1p-24f;
}

// E = -ln(u) for u = sv_u01(x) in double, where a decision is refined.
__device__ __forceinline__ double sv_neglog_u_f64(uint32_t x) {
  const double u = (2.0 * (double)(x >> 9) + 1.0) * 0x1p-24;
  return -log(u);
}

// --------------------------------------------------------------------------
// Fast exp2 (MUFU.EX2, flush-to-zero below 2^-126).
// --------------------------------------------------------------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// --------------------------------------------------------------------------
// Logit access.  bf16 values are carried as raw bits; widening to fp32 is a
// shift (low half) or a mask (high half).
// --------------------------------------------------------------------------
// Packed pairs of fp32 (one 64-bit register pair) and the paired IEEE
// operations of sm_100+: two FMAs / two adds per instruction, each rounded as
// its scalar form.
__device__ __forceinline__ uint64_t pack2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int DT>
__device__ __forceinline__ float load_logit(const void* base, int64_t idx);
template <>
__device__ __forceinline__ float load_logit<SV_F32>(const void* base, int64_t idx) {
  return __ldg(reinterpret_cast<const float*>(base) + idx);
}
template <>
__device__ __forceinline__ float load_logit<SV_BF16>(const void* base, int64_t idx) {
  const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(base) + idx);
  return __uint_as_float((uint32_t)h << 16);
}

// Streaming 16-byte load that does not allocate in L1 (data is read once per SM).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Elements per 16-byte vector.
template <int DT>
struct VecInfo;
template <>
struct VecInfo<SV_F32> {
  static constexpr int kElems = 4;
};
template <>
struct VecInfo<SV_BF16> {
  static constexpr int kElems = 8;
};

// Unpack a 16-byte vector into fp32 values.
template <int DT>
__device__ __forceinline__ void unpack(const uint4& v, float* f);
template <>
__device__ __forceinline__ void unpack<SV_F32>(const uint4& v, float* f) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}
template <>
__device__ __forceinline__ void unpack<SV_BF16>(const uint4& v, float* f) {
  f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
  f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
  f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

// Max over a vector, NaN ignored (fmaxf semantics).
template <int DT>
__device__ __forceinline__ float vmax(const uint4& v);
template <>
__device__ __forceinline__ float vmax<SV_F32>(const uint4& v) {
  return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
               fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}
template <>
__device__ __forceinline__ float vmax<SV_BF16>(const uint4& v) {
  // packed bf16x2 max (NaN-ignoring), then the two halves
  uint32_t a, b, c;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(v.x), "r"(v.y));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(v.z), "r"(v.w));
  asm("max.bf16x2 %0, %1, %2;" : "=r"(c) : "r"(a), "r"(b));
  return fmaxf(bf16lo(c), bf16hi(c));
}

// --------------------------------------------------------------------------
// (max, sum) pairs of the online softmax: S is a sum of 2^(y - m).
// --------------------------------------------------------------------------
struct MS {
  float m;
  float s;
};

__device__ __forceinline__ MS ms_combine(MS a, MS b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -kInf) return MS{-kInf, 0.0f};
  const float sa = (a.m == -kInf) ? 0.0f : a.s * ex2(a.m - m);
  const float sb = (b.m == -kInf) ? 0.0f : b.s * ex2(b.m - m);
  return MS{m, sa + sb};
}

__device__ __forceinline__ MS warp_reduce_ms(MS v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    MS w{__shfl_xor_sync(0xffffffffu, v.m, o), __shfl_xor_sync(0xffffffffu, v.s, o)};
    v = ms_combine(v, w);
  }
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// (key, index) with "larger key wins, lower index wins ties".
struct KI {
  float k;
  int i;
};

__device__ __forceinline__ bool ki_better(KI a, KI b) {
  return (a.k > b.k) || (a.k == b.k && (unsigned)a.i < (unsigned)b.i);
}

__device__ __forceinline__ KI warp_reduce_ki(KI t) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    KI w{__shfl_xor_sync(0xffffffffu, t.k, o), __shfl_xor_sync(0xffffffffu, t.i, o)};
    if (ki_better(w, t)) t = w;
  }
  return t;
}

// -log2(u) for u = sv_u01(x): the exponential variate E of the race, in log2
// units (a common scale factor of all keys, so the argmax is unchanged).  Near
// u = 1 it comes from w = 1 - u (exact) and -log2(1-w) = (w + w^2/2 + ...)/ln 2,
// truncated after w^2 (relative error < w^2/3 < 2^-17.5 for w < 2^-8).
__device__ __forceinline__ float neglog2_u(uint32_t x) {
  const float u = __uint_as_float(0x3f800000u | (x >> 9)) - 0x1.fffffep-1f;
  const float w = 1.0f - u;
  const float series = w * fmaf(w, 0.5f * kLog2e, kLog2e);
  return (w < 0x1p-8f) ? series : -__log2f(u);
}

// Philox4x32-10 with the ten round keys precomputed (the key schedule depends
// only on the seed).
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
};
__device__ __forceinline__ PhiloxKeys philox_keys(uint64_t seed) {
  PhiloxKeys k;
  uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    k.k0[r] = a;
    k.k1[r] = b;
    a += 0x9E3779B9u;
    b += 0xBB67AE85u;
  }
  return k;
}
__device__ __forceinline__ uint4 philox_rk(uint4 c, const PhiloxKeys& k) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    // one 32x32 -> 64-bit multiply gives both halves of each product
    uint64_t p0, p1;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c.x), "r"(0xD2511F53u));
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(c.z), "r"(0xCD9E8D57u));
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k.k0[r], (uint32_t)p1,
                   (uint32_t)(p0 >> 32) ^ c.w ^ k.k1[r], (uint32_t)p0);
  }
  return c;
}

}  // namespace sv
