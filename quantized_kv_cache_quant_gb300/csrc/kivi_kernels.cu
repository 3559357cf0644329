// KIVI 2/4-bit KV cache kernels for sm_103a: group quantize + pack (prefill and
// residual flush), token copies (window fill, append), split-K decode attention
// over the packed codes with in-register dequantization, and the log-sum-exp
// merge of the split partials.
//
// Method: "4.4 KV Cache 量化：KIVI 2-bit 与 FP8 KV Cache" (aiinfraguide), section 3
// (keys per channel, values per token, groups of 32 tokens, fp16 residual
// window flushed when full); affine form of "大模型量化从0到1（十三）：KV Cache 量化"
// (CSDN), section 10; attention softmax(q K^T / sqrt(d)) V of the same page,
// section 2, with grouped-query sharing (section 5).
#include <cfloat>
#include <cmath>
#include <type_traits>

#include "kvq_device.cuh"
#include "kvq_internal.h"

// Resident decode blocks per SM the register budget is sized for: 3 at D = 128
// (168 registers; a 128-register bound spills 112-204 bytes), 4 at D = 64
// (118-128 registers, no spills; 5 blocks spill). D = 64 against 3 blocks,
// GB300: GQA-8 8K 2-bit 97.0 -> 95.7 us, 4-bit 103.1 -> 100.7 us, paged
// 512-16384 tokens 62.1 -> 59.3 us.
template <int D>
struct DecodeMinBlocks {
  static constexpr int value = (D == 64) ? 4 : 3;
};
namespace kvq {
namespace {

template <int D, int KB, int VB>
struct Kivi {
  static constexpr int KS = D / 16;                     // k-steps of q . k^T
  static constexpr int NTV = D / 8;                     // n-tiles of p . V
  static constexpr int NQ = D / 32;                     // value code words per (k-step[, r])
  static constexpr int KW = (KB == 2) ? D / 16 : D / 8;  // key code words per lane
  static constexpr int VW = (VB == 2) ? D / 16 : D / 8;  // value code words per lane
  static constexpr int KC = 32 * D * KB / 8;            // bytes of one group's records
  static constexpr int KM = 4 * D;
  static constexpr int VC = 32 * D * VB / 8;
  static constexpr int VM = 128;
  static constexpr int STAGE = KC + KM + VC + VM;
  static_assert(STAGE % 16 == 0, "bulk copies need 16-byte multiples");
};

// Masks that keep the code field of each fp16 half after the shift: bits 6-7
// or 8-9 for 2-bit codes, bits 6-9 for 4-bit codes. The field then reads as
// the fp16 subnormal code * 2^(P-24), P = 6 or 8; the top mantissa bits keep
// the tensor-core products at full fp32-accumulation accuracy. A 2-bit word
// holds 8 fields per half; the word itself, its shifts by 4 either way and its
// per-half byte swap bring two fields each to bits 6-7 and 8-9 (field order
// f = (4r + nt + 1) mod 8 of the packed layout): three operations and eight
// masks for 16 codes.
constexpr uint32_t kMaskP6 = 0x00C000C0u;
constexpr uint32_t kMaskP8 = 0x03000300u;
constexpr uint32_t kMask4 = 0x03C003C0u;
constexpr float kInvP6 = 262144.0f;  // 2^18 = 2^(24-6)
constexpr float kInvP8 = 65536.0f;   // 2^16 = 2^(24-8)

// ---------------------------------------------------------------------------
// Group quantization (one thread block per (group, kv head, batch row))
// ---------------------------------------------------------------------------

// The group formula in IEEE fp32 with round-to-nearest-even everywhere.
__device__ __forceinline__ void group_scale_zero(float mn, float mx, float levels, __half& s16, __half& z16) {
  s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), levels));
  z16 = __float2half_rn(__fadd_rn(mn, 0.0f));  // exact; -0 becomes +0
}

// fl32(x - z) of both halves of the fp16 pair x (nz = -z): one mixed-precision
// fused multiply-add x * 1 + nz per element, the widening to fp32 included
// (the product is exact, the sum rounds once).
__device__ __forceinline__ float2 sub_f16_f32(uint32_t x, float2 nz) {
  float2 d;
  asm("{\n\t.reg .b16 xl, xh, one;\n\t"
      "mov.b32 {xl, xh}, %2;\n\t"
      "mov.b16 one, 0x3C00;\n\t"
      "fma.rn.f32.f16 %0, xl, one, %3;\n\t"
      "fma.rn.f32.f16 %1, xh, one, %4;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "r"(x), "f"(nz.x), "f"(nz.y));
  return d;
}

// The group formula's codes clamp(rint(fl32((x - z) / s)), 0, levels) of two
// fp16 values x (one group each: nz = -z, and sr = {-s, -s', rcp, rcp'} with
// rcp = RN(1/s)) in packed fp32 operations, as {code0, code1} in the two
// 16-bit halves. The quotient comes from rcp and one correction step (q0 =
// d rcp, r = d - q0 s by fused multiply-add, q = q0 + r rcp), bit-identical
// to the IEEE division here (x, z and s are fp16 values, so nothing under- or
// overflows; s = 0 has rcp = 0 and gives code 0 as the formula does). x >= z
// leaves no negative quotient, so q + 2^23 rounds q to an integer to nearest
// even in its low bits (q < 2^22); the two low halves are merged and clamped
// to the top code with one 16-bit SIMD min.
__device__ __forceinline__ uint32_t group_code_pair(uint32_t x, float2 nz, float4 sr, uint32_t levels) {
  const float2 d = sub_f16_f32(x, nz);
  const float2 rcp = make_float2(sr.z, sr.w);
  const float2 q0 = __fmul2_rn(d, rcp);
  const float2 r = __ffma2_rn(q0, make_float2(sr.x, sr.y), d);
  const float2 q = __ffma2_rn(r, rcp, q0);
  const float2 t = __fadd2_rn(q, make_float2(0x1p23f, 0x1p23f));
  const uint32_t pair = __byte_perm(__float_as_uint(t.x), __float_as_uint(t.y), 0x5410);
  return __vminu2(pair, levels * 0x00010001u);
}

// ---- 2-bit codes by thresholds -------------------------------------------
// The group formula's code is a non-decreasing function of x (every step of it
// is monotone), so for 2-bit codes code(x) = #{k = 1..3 : x >= theta_k} with
// theta_k the smallest fp16 value whose code is at least k. The thresholds are
// exact, from the rounding rules of the formula's two fp32 steps:
//  * rint(q) >= k  <=>  q >= k - 1/2 (even k: the tie rounds to k) or
//    q > k - 1/2 (odd k); q = fl32(d / s) reaches m = k - 1/2 from the
//    midpoint between m and its fp32 neighbour (m's significand is even, so a
//    tie there rounds to m). Hence code >= k  <=>  d >= D_k with the fp32
//    threshold D_k = RU(s (1.5 - 2^-24)) for k = 2, and for k = 1, 3 the
//    smallest fp32 above s (m + h), h = 2^-25, 2^-23 (one fused multiply-add
//    rounded up, and one rounded down to see whether it was exact);
//  * d = fl32(x - z) is monotone in x, so theta_k is the smallest fp16 x with
//    fl32(x - z) >= D_k: RU16(z + D_k) when the subtraction is exact near it
//    (checked at that value and the fp16 value below it), else found by a
//    bisection over the fp16 order keys (x close to 0 while |z| is large).
// Every element then costs three fp16 comparisons and no division.

// Order keys of fp16 bit patterns: a pattern maps to an int in the order of
// the values (both zeros to 0, +inf to 0x7C00), and back.
__device__ __forceinline__ int f16_key(uint32_t b) {
  return (b & 0x8000u) ? -static_cast<int>(b & 0x7FFFu) : static_cast<int>(b & 0x7FFFu);
}
__device__ __forceinline__ uint32_t f16_from_key(int key) {
  return key >= 0 ? static_cast<uint32_t>(key) : (0x8000u | static_cast<uint32_t>(-key));
}

// D_k above (s > 0, k = 1, 2, 3).
__device__ __forceinline__ float code_step(float s, int k) {
  if (k == 2) return __fmaf_ru(-0x1p-24f, s, __fmul_rn(1.5f, s));
  const float ms = __fmul_rn(k == 1 ? 0.5f : 2.5f, s);  // exact
  const float h = (k == 1) ? 0x1p-25f : 0x1p-23f;
  const float up = __fmaf_ru(h, s, ms), dn = __fmaf_rd(h, s, ms);
  return (up == dn) ? __uint_as_float(__float_as_uint(up) + 1u) : up;  // exact: the next fp32 above
}

// fl32(x - z) >= d for the fp16 value with bits xb.
__device__ __forceinline__ bool reaches(uint32_t xb, float zf, float d) {
  return __fsub_rn(__half2float(__ushort_as_half(static_cast<unsigned short>(xb))), zf) >= d;
}

// theta_k as fp16 bits (+inf, 0x7C00, when no fp16 value reaches code k;
// every code is 0 when s = 0).
__device__ __forceinline__ uint32_t code_threshold(uint32_t zb, float zf, float sf, int k) {
  if (sf == 0.0f) return 0x7C00u;
  const float d = code_step(sf, k);
  const uint32_t x0 = __half_as_ushort(__float2half_ru(__fadd_ru(zf, d)));
  const int k0 = f16_key(x0), kz = f16_key(zb);
  const bool r0 = reaches(x0, zf, d);
  const bool r1 = (k0 - 1 > kz) && reaches(f16_from_key(k0 - 1), zf, d);
  if (r0 && !r1) return x0;
  // rare: bisection with reaches(lo) false and reaches(hi) true (z never reaches d > 0; +inf always does)
  int lo = r0 ? kz : k0, hi = r0 ? k0 - 1 : 0x7C00;
  for (int it = 0; it < 17 && hi - lo > 1; ++it) {
    const int mid = lo + (hi - lo) / 2;
    if (reaches(f16_from_key(mid), zf, d))
      hi = mid;
    else
      lo = mid;
  }
  return f16_from_key(hi);
}

// One 2-bit code pair from thresholds (t1 <= t2 <= t3), per fp16 half: the
// high code bit is [x >= t2] (as a mask m); the low bit compares x with t3 or
// t1 as m selects, read as 1024 + bit (exact) whose bits are 0x6400 + bit; m
// adds the high bit. A word adds eight such pairs, each shifted to its field;
// the 0x6400 parts sum to a constant (kThresholdBase) that is subtracted once
// per word.
__device__ __forceinline__ uint32_t threshold_pair(__half2 x, uint32_t t1, uint32_t t2, uint32_t t3) {
  const uint32_t m = __hge2_mask(x, bits_h2(t2));
  const uint32_t tl = (m & t3) | (~m & t1);
  const uint32_t lo = h2_bits(__hadd2(__hge2(x, bits_h2(tl)), __float2half2_rn(1024.0f)));
  return lo | (m & 0x00020002u);
}
constexpr uint32_t threshold_base() {
  uint32_t s = 0;
  for (int f = 0; f < 8; ++f) s += 0x64006400u << (2 * f);
  return s;
}
constexpr uint32_t kThresholdBase = threshold_base();

// One packed code word of a group (storage word u of lane l = 4 gg + tg),
// from the row-major tiles xk and xv (RS halves per token). The elements a
// word packs come as fp16 pairs from one ldmatrix of four 8 x 8 tiles: keys
// {x[8 nt + gg][d0], x[8 nt + gg][d0 + 1]} (tiles nt = 0..3 of tokens 8 nt ..,
// channels d0 - 2 tg ..), values {x[t0][ch], x[t0 + 1][ch]} (the transposed
// tiles of tokens t0 - 2 tg .., channels ch - gg ..).
template <int D, int KB>
__device__ __forceinline__ uint32_t key_word(const __half* xk, int RS, const float4* srk, const float2* nzk,
                                             const uint4* thk, int u, int lane) {
  constexpr uint32_t KL = (1u << KB) - 1u;
  const int tg = lane & 3;
  uint32_t w = 0;
#pragma unroll
  for (int rr = 0; rr < (KB == 2 ? 2 : 1); ++rr) {
    const int ks = (KB == 2) ? u : (u >> 1);
    const int r = (KB == 2) ? rr : (u & 1);
    const int d0 = 16 * ks + 8 * r + 2 * tg;
    uint32_t xr[4];
    ldsm_x4(xr, xk + lane * RS + 16 * ks + 8 * r);  // lane l addresses row l of tile l / 8
    if constexpr (KB == 2) {
      const uint4 th = thk[d0 / 2];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int f = (4 * r + nt + 1) & 7;
        w += threshold_pair(bits_h2(xr[nt]), th.x, th.y, th.z) << (2 * f);
      }
    } else {
      const float4 sr = srk[d0 / 2];
      const float2 nz = nzk[d0 / 2];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)  // fields never overlap: adding the shifted pair sets the same bits as or-ing
        w += group_code_pair(xr[nt], nz, sr, KL) << (KB * nt);
    }
  }
  return (KB == 2) ? w - kThresholdBase : w;
}

template <int D, int VB>
__device__ __forceinline__ uint32_t value_word(const __half* xv, int RS, const float4* srv, const float2* nzv,
                                               const uint4* thv, int u, int lane) {
  constexpr uint32_t VL = (1u << VB) - 1u;
  constexpr int NQ = D / 32;
  const int tg = lane & 3;
  uint32_t w = 0;
#pragma unroll
  for (int rr = 0; rr < (VB == 2 ? 2 : 1); ++rr) {
    const int ks = (VB == 2) ? u / NQ : u / (2 * NQ);
    const int r = (VB == 2) ? rr : (u / NQ) % 2;
    const int q = u % NQ;
    const int t0 = 16 * ks + 8 * r + 2 * tg;  // tokens t0, t0 + 1
    uint32_t xr[4];
    ldsm_x4_trans(xr, xv + (16 * ks + 8 * r + (lane & 7)) * RS + 8 * (4 * q + (lane >> 3)));
    if constexpr (VB == 2) {
      const uint4 th = thv[t0 / 2];
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const int f = (4 * r + n + 1) & 7;
        w += threshold_pair(bits_h2(xr[n]), th.x, th.y, th.z) << (2 * f);
      }
    } else {
      const float4 sr = srv[t0 / 2];
      const float2 nz = nzv[t0 / 2];
#pragma unroll
      for (int n = 0; n < 4; ++n) w += group_code_pair(xr[n], nz, sr, VL) << (VB * n);
    }
  }
  return (VB == 2) ? w - kThresholdBase : w;
}

// Row stride of a staged 32-token tile (halves): the 8 rows of an ldmatrix
// tile hit distinct banks.
template <int D>
struct Tile {
  static constexpr int RS = D + 8;
};

// Start the 16-byte asynchronous copies of one group's fp16 rows k_src[0 ..
// 32*D) and v_src[...] (32 consecutive tokens of D channels) into the tiles xk
// and xv; the caller commits and waits. Run by a whole block of 128 threads.
template <int D>
__device__ __forceinline__ void load_group_async(const uint16_t* k_src, const uint16_t* v_src, __half* xk, __half* xv) {
  constexpr int RS = Tile<D>::RS;
  const uint4* srck = reinterpret_cast<const uint4*>(k_src);
  const uint4* srcv = reinterpret_cast<const uint4*>(v_src);
#pragma unroll
  for (int i = threadIdx.x; i < 32 * D / 8; i += 128) {
    const int row = i / (D / 8), c8 = i % (D / 8);
    cp_async16(xk + row * RS + 8 * c8, srck + i);
    cp_async16(xv + row * RS + 8 * c8, srcv + i);
  }
}

// Quantize and pack one staged group of 32 tokens of one (batch row, kv head)
// into the four records at kc, km, vc and vm (nothing is written when write is
// false; the block still takes part in every barrier). Run by a whole block of
// 128 threads after a barrier that makes the tiles visible; it leaves the
// tiles unread behind a final barrier of its own.
template <int D, int KB, int VB>
__device__ __forceinline__ void quantize_tiles(const __half* xk, const __half* xv, uint8_t* kc, uint8_t* km,
                                               uint8_t* vc, uint8_t* vm, bool write) {
  using P = Kivi<D, KB, VB>;
  constexpr int RS = Tile<D>::RS;
  // 4-bit codes: per pair of key channels (value tokens) {-s, -s', RN(1/s), RN(1/s')} and {-z, -z'}
  __shared__ float4 srk[D / 2];
  __shared__ float2 nzk[D / 2];
  __shared__ float4 srv[16];
  __shared__ float2 nzv[16];
  __shared__ uint16_t skb[D], zkb[D], svb[32], zvb[32];  // fp16 bits of scale and zero
  // 2-bit thresholds: entry j = {t1, t2, t3} of channels (keys) or tokens (values) 2j and 2j + 1
  __shared__ __align__(16) uint4 thk[D / 2];
  __shared__ __align__(16) uint4 thv[16];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;

  constexpr float KL = static_cast<float>((1 << KB) - 1);
  constexpr float VL = static_cast<float>((1 << VB) - 1);

  if (tid < D / 2) {
    // keys: one pair of channels per thread, exact fp16 min/max over the 32 tokens
    const __half2* col = reinterpret_cast<const __half2*>(xk) + tid;
    __half2 mn = col[0], mx = col[0];
#pragma unroll 8
    for (int t = 1; t < 32; ++t) {
      const __half2 v = col[t * (RS / 2)];
      mn = __hmin2(mn, v);
      mx = __hmax2(mx, v);
    }
    const float2 mnf = __half22float2(mn), mxf = __half22float2(mx);
    uint32_t th[3] = {0u, 0u, 0u};  // KB == 2: thresholds of channels 2 tid (low half) and 2 tid + 1
    float sr[4], nz[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      __half s16, z16;
      group_scale_zero(e ? mnf.y : mnf.x, e ? mxf.y : mxf.x, KL, s16, z16);
      const int c = 2 * tid + e;
      sr[e] = -__half2float(s16);
      sr[2 + e] = (__half2float(s16) == 0.0f) ? 0.0f : __frcp_rn(__half2float(s16));
      nz[e] = -__half2float(z16);
      skb[c] = __half_as_ushort(s16);
      zkb[c] = __half_as_ushort(z16);
      if constexpr (KB == 2) {
#pragma unroll
        for (int k = 1; k <= 3; ++k)
          th[k - 1] |= code_threshold(__half_as_ushort(z16), __half2float(z16), __half2float(s16), k) << (16 * e);
      }
    }
    if constexpr (KB == 2) {
      thk[tid] = make_uint4(th[0], th[1], th[2], 0u);
    } else {
      srk[tid] = make_float4(sr[0], sr[1], sr[2], sr[3]);
      nzk[tid] = make_float2(nz[0], nz[1]);
    }
  } else if (warp >= 2) {
    // values: warps 2 and 3, two lanes per token, each over half of the row
    // with fp16 pair min/max; lane L reads its words in the order (c + L) mod
    // (D / 4), which keeps every shared-memory read conflict-free at D = 128
    constexpr int W2 = D / 4;                 // half2 words per lane
    const int t = 16 * (warp - 2) + (lane & 15), hh = lane >> 4;
    const __half2* row = reinterpret_cast<const __half2*>(xv) + t * (RS / 2) + hh * W2;
    __half2 mn = row[lane & (W2 - 1)], mx = mn;
#pragma unroll 8
    for (int c = 1; c < W2; ++c) {
      const __half2 v = row[(c + lane) & (W2 - 1)];
      mn = __hmin2(mn, v);
      mx = __hmax2(mx, v);
    }
    const float2 mnf2 = __half22float2(mn), mxf2 = __half22float2(mx);
    float mnf = fminf(mnf2.x, mnf2.y), mxf = fmaxf(mxf2.x, mxf2.y);
    mnf = fminf(mnf, __shfl_xor_sync(0xffffffffu, mnf, 16));
    mxf = fmaxf(mxf, __shfl_xor_sync(0xffffffffu, mxf, 16));
    __half s16, z16;
    group_scale_zero(mnf, mxf, VL, s16, z16);
    if (hh == 0) {
      if constexpr (VB != 2) {
        float* sr = reinterpret_cast<float*>(srv + (t >> 1));
        sr[t & 1] = -__half2float(s16);
        sr[2 + (t & 1)] = (__half2float(s16) == 0.0f) ? 0.0f : __frcp_rn(__half2float(s16));
        reinterpret_cast<float*>(nzv + (t >> 1))[t & 1] = -__half2float(z16);
      }
      svb[t] = __half_as_ushort(s16);
      zvb[t] = __half_as_ushort(z16);
    }
    if constexpr (VB == 2) {
      // both lanes of the token share its three thresholds: t1 on lane hh = 0, t2 and t3 on hh = 1
      uint16_t* th16 = reinterpret_cast<uint16_t*>(thv + (t >> 1)) + (t & 1);
#pragma unroll
      for (int k = 1; k <= 2; ++k) {
        const int kk = hh ? k + 1 : 1;
        if (hh || k == 1)
          th16[2 * (kk - 1)] = static_cast<uint16_t>(
              code_threshold(__half_as_ushort(z16), __half2float(z16), __half2float(s16), kk));
      }
    }
  }
  __syncthreads();

  // Code words, computed straight from the staged tiles: warps 0-1 the key
  // words, warps 2-3 the value words. Storage words 4*ug .. 4*ug + 3 of
  // fragment lane L are one 16-byte chunk (uint4 ug*32 + L); lane L of a warp
  // computes that chunk (its elements from conflict-free ldmatrix loads), and
  // each store of the warp writes 512 contiguous bytes.
  if (!write) {
    // a skipped pool block: nothing to compute or store
  } else if (warp < 2) {
    uint4* kdst = reinterpret_cast<uint4*>(kc);
    for (int ug = warp; ug < P::KW / 4; ug += 2) {
      uint4 w;
      w.x = key_word<D, KB>(xk, RS, srk, nzk, thk, 4 * ug, lane);
      w.y = key_word<D, KB>(xk, RS, srk, nzk, thk, 4 * ug + 1, lane);
      w.z = key_word<D, KB>(xk, RS, srk, nzk, thk, 4 * ug + 2, lane);
      w.w = key_word<D, KB>(xk, RS, srk, nzk, thk, 4 * ug + 3, lane);
      kdst[ug * 32 + lane] = w;
    }
  } else {
    uint4* vdst = reinterpret_cast<uint4*>(vc);
    for (int ug = warp - 2; ug < P::VW / 4; ug += 2) {
      uint4 w;
      w.x = value_word<D, VB>(xv, RS, srv, nzv, thv, 4 * ug, lane);
      w.y = value_word<D, VB>(xv, RS, srv, nzv, thv, 4 * ug + 1, lane);
      w.z = value_word<D, VB>(xv, RS, srv, nzv, thv, 4 * ug + 2, lane);
      w.w = value_word<D, VB>(xv, RS, srv, nzv, thv, 4 * ug + 3, lane);
      vdst[ug * 32 + lane] = w;
    }
  }

  // Key meta: record ks*4 + tig = {s[d0], s[d0+1], s[d0+8], s[d0+9], z[...]}.
  if (!write) {
  } else if (tid < D / 4) {
    const int ks = tid >> 2, tg = tid & 3, d0 = 16 * ks + 2 * tg;
    uint4 rec;
    rec.x = skb[d0] | (static_cast<uint32_t>(skb[d0 + 1]) << 16);
    rec.y = skb[d0 + 8] | (static_cast<uint32_t>(skb[d0 + 9]) << 16);
    rec.z = zkb[d0] | (static_cast<uint32_t>(zkb[d0 + 1]) << 16);
    rec.w = zkb[d0 + 8] | (static_cast<uint32_t>(zkb[d0 + 9]) << 16);
    reinterpret_cast<uint4*>(km)[tid] = rec;
  } else if (tid >= 64 && tid < 72) {
    // Value meta: 4 records of scales, then 4 of zero points.
    const int i = tid - 64, tg = i & 3;
    const uint16_t* src = (i < 4) ? svb : zvb;
    uint4 rec;
    rec.x = src[2 * tg] | (static_cast<uint32_t>(src[2 * tg + 1]) << 16);
    rec.y = src[8 + 2 * tg] | (static_cast<uint32_t>(src[9 + 2 * tg]) << 16);
    rec.z = src[16 + 2 * tg] | (static_cast<uint32_t>(src[17 + 2 * tg]) << 16);
    rec.w = src[24 + 2 * tg] | (static_cast<uint32_t>(src[25 + 2 * tg]) << 16);
    reinterpret_cast<uint4*>(vm)[i] = rec;
  }
  __syncthreads();  // the tiles and the block's statistics are free again
}

// The 16-byte vectors first, first + stride, ... of a token copy (vector i: (b, h)
// row i / (n_tokens * D/8), token and vector within it), K and V together.
__device__ __forceinline__ void copy_token_vectors(const CopyTokensArgs& a, long long first, long long stride) {
  const int vec_per_tok = a.head_dim / 8;
  const long long per_bh = static_cast<long long>(a.n_tokens) * vec_per_tok;
  const long long total = per_bh * a.bh;
  for (long long i = first; i < total; i += stride) {
    const long long bh = i / per_bh;
    const long long rem = i % per_bh;
    const long long tok = rem / vec_per_tok, v = rem % vec_per_tok;
    const long long s = (bh * a.src_bh_stride + (a.src_tok0 + tok) * a.head_dim) / 8 + v;
    const long long d = (bh * a.dst_bh_stride + (a.dst_tok0 + tok) * a.head_dim) / 8 + v;
    reinterpret_cast<uint4*>(a.k_dst)[d] = reinterpret_cast<const uint4*>(a.k_src)[s];
    reinterpret_cast<uint4*>(a.v_dst)[d] = reinterpret_cast<const uint4*>(a.v_src)[s];
  }
}

// Persistent blocks over the items (group, kv head, batch row), group index
// fastest: item i goes to group dst_group0 + grp of the contiguous grouped
// region, read from source token src_tok0 + 32 * grp. Each block stages the
// next item's tiles with asynchronous copies into its second buffer while it
// quantizes the current one. Then the grid copies the fp16 tokens of w (a
// prefill's window fill; n_tokens = 0: none) in a grid-stride loop, so that
// blocks that run out of groups early copy while the others finish.
template <int D, int KB, int VB>
__global__ void __launch_bounds__(128) kivi_quantize_kernel(QuantGroupsArgs a, CopyTokensArgs w) {
  using P = Kivi<D, KB, VB>;
  constexpr int TILE = 32 * Tile<D>::RS;
  __shared__ __align__(16) __half tiles[2][2][TILE];  // [buffer][keys, values]
  const int n_bh = a.kv_heads * a.batch;
  // item = bh * n_groups + grp, advanced by gridDim.x = step_bh * n_groups + step_grp per turn
  const int step_bh = static_cast<int>(gridDim.x) / a.n_groups, step_grp = static_cast<int>(gridDim.x) % a.n_groups;
  int bh = static_cast<int>(blockIdx.x) / a.n_groups, grp = static_cast<int>(blockIdx.x) % a.n_groups;
  auto src_off = [&](int pbh, int pgrp) {
    return static_cast<long long>(pbh) * a.src_bh_stride + static_cast<long long>(a.src_tok0 + 32 * pgrp) * D;
  };
  if (bh < n_bh) {
    const long long off = src_off(bh, grp);
    load_group_async<D>(a.k_src + off, a.v_src + off, tiles[0][0], tiles[0][1]);
  }
  cp_async_commit();
  for (int buf = 0; bh < n_bh; buf ^= 1) {
    int nbh = bh + step_bh, ngrp = grp + step_grp;
    if (ngrp >= a.n_groups) ngrp -= a.n_groups, ++nbh;
    if (nbh < n_bh) {
      const long long off = src_off(nbh, ngrp);
      load_group_async<D>(a.k_src + off, a.v_src + off, tiles[buf ^ 1][0], tiles[buf ^ 1][1]);
    }
    cp_async_commit();
    cp_async_wait_all_but_newest();  // this item's copies have landed
    __syncthreads();
    const long long gi = static_cast<long long>(bh) * a.groups_cap + a.dst_group0 + grp;
    quantize_tiles<D, KB, VB>(tiles[buf][0], tiles[buf][1], a.k_codes + gi * P::KC, a.k_meta + gi * P::KM,
                              a.v_codes + gi * P::VC, a.v_meta + gi * P::VM, true);
    bh = nbh;
    grp = ngrp;
  }
  if (w.n_tokens > 0)
    copy_token_vectors(w, blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x,
                       static_cast<long long>(gridDim.x) * blockDim.x);
}

// The sequence that owns item x of a batched launch: the b < n with
// begin[b] <= x < begin[b + 1] (begin is non-decreasing, begin[0] = 0 <= x <
// begin[n]). Binary search over the parameter array.
__device__ __forceinline__ int seq_of(const int* begin, int n, long long x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (begin[mid] <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Persistent blocks over the items (x, kv head h), x fastest: x is group
// x - begin[b] of sequence b's range, read from source token src0[b] + 32 *
// (x - begin[b]) and written to the pool block of logical group dst0[b] + (x -
// begin[b]), its four records back to back in the block's entry for kv head
// h. A block-table entry outside [0, num_blocks) is skipped: nothing is
// written for it. The next item's tiles are staged while this one is
// quantized, as in the contiguous kernel.
template <int D, int KB, int VB>
__global__ void __launch_bounds__(128) kivi_quantize_paged_kernel(PagedQuantArgs a) {
  using P = Kivi<D, KB, VB>;
  constexpr int TILE = 32 * Tile<D>::RS;
  __shared__ __align__(16) __half tiles[2][2][TILE];
  const int total_x = a.r.begin[a.n_seqs];
  // item = h * total_x + x, advanced by gridDim.x = step_h * total_x + step_x per turn; the
  // sequence b of x only moves forward while h stays, and restarts its search when h moves
  const int step_h = static_cast<int>(gridDim.x) / total_x, step_x = static_cast<int>(gridDim.x) % total_x;
  int h = static_cast<int>(blockIdx.x) / total_x, x = static_cast<int>(blockIdx.x) % total_x;
  if (h >= a.q.kv_heads) return;
  int b = seq_of(a.r.begin, a.n_seqs, x);
  auto src_off = [&](int pb, int px, int ph) {
    const long long bh = static_cast<long long>(pb) * a.q.kv_heads + ph;
    return bh * a.q.src_bh_stride + static_cast<long long>(a.r.src0[pb] + 32 * (px - a.r.begin[pb])) * D;
  };
  // the pool block of item x of sequence pb (its block-table entry), loaded one item ahead
  // together with that item's tiles, so that the load is not waited for
  auto table_entry = [&](int pb, int px) {
    return __ldg(a.pools.block_table + static_cast<long long>(pb) * a.pools.groups_cap + a.r.dst0[pb] +
                 (px - a.r.begin[pb]));
  };
  int blk = table_entry(b, x);
  {
    const long long off = src_off(b, x, h);
    load_group_async<D>(a.q.k_src + off, a.q.v_src + off, tiles[0][0], tiles[0][1]);
  }
  cp_async_commit();
  for (int buf = 0; h < a.q.kv_heads; buf ^= 1) {
    int nh = h + step_h, nx = x + step_x, nb = b;
    if (nx >= total_x) nx -= total_x, ++nh;
    if (nh != h || nx < x) {
      nb = seq_of(a.r.begin, a.n_seqs, nx);
    } else {
      while (a.r.begin[nb + 1] <= nx) ++nb;  // nb < n_seqs: nx < total_x = begin[n_seqs]
    }
    int nblk = -1;
    if (nh < a.q.kv_heads) {
      nblk = table_entry(nb, nx);
      const long long off = src_off(nb, nx, nh);
      load_group_async<D>(a.q.k_src + off, a.q.v_src + off, tiles[buf ^ 1][0], tiles[buf ^ 1][1]);
    }
    cp_async_commit();
    cp_async_wait_all_but_newest();
    __syncthreads();
    const bool ok = blk >= 0 && blk < a.pools.num_blocks;
    uint8_t* e = a.q.k_codes + (static_cast<long long>(ok ? blk : 0) * a.q.kv_heads + h) * P::STAGE;
    quantize_tiles<D, KB, VB>(tiles[buf][0], tiles[buf][1], e, e + P::KC, e + P::KC + P::KM,
                              e + P::KC + P::KM + P::VC, ok);
    h = nh;
    x = nx;
    b = nb;
    blk = nblk;
  }
}

// ---------------------------------------------------------------------------
// Token copies (fill the fp16 window, append a decode token, move a remainder)
// ---------------------------------------------------------------------------
__global__ void copy_tokens_kernel(CopyTokensArgs a) {
  // A decode launched right after this copy may start now: it reads what this
  // kernel writes (the fp16 window) only after its griddepcontrol.wait.
  asm volatile("griddepcontrol.launch_dependents;");
  copy_token_vectors(a, blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x,
                     static_cast<long long>(gridDim.x) * blockDim.x);
}

// Batched copies of a paged cache: token x of the launch (x < begin[n]) is
// token x - begin[b] of sequence b's range; for each kv head h its D channels
// go from source row src0[b] + (x - begin[b]) of (b, h) to window row
// dst0[b] + (x - begin[b]). Sources and destinations of one launch do not
// overlap.
__global__ void copy_tokens_paged_kernel(PagedCopyArgs a) {
  asm volatile("griddepcontrol.launch_dependents;");
  const int vec_per_tok = a.c.head_dim / 8;
  const long long per_tok = static_cast<long long>(a.kv_heads) * vec_per_tok;
  const long long total = static_cast<long long>(a.r.begin[a.n_seqs]) * per_tok;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long x = i / per_tok, rem = i % per_tok;
    const int h = static_cast<int>(rem / vec_per_tok), v = static_cast<int>(rem % vec_per_tok);
    const int b = seq_of(a.r.begin, a.n_seqs, x);
    const long long tok = x - a.r.begin[b];
    const long long bh = static_cast<long long>(b) * a.kv_heads + h;
    const long long s = (bh * a.c.src_bh_stride + (a.r.src0[b] + tok) * a.c.head_dim) / 8 + v;
    const long long d = (bh * a.c.dst_bh_stride + (a.r.dst0[b] + tok) * a.c.head_dim) / 8 + v;
    reinterpret_cast<uint4*>(a.c.k_dst)[d] = reinterpret_cast<const uint4*>(a.c.k_src)[s];
    reinterpret_cast<uint4*>(a.c.v_dst)[d] = reinterpret_cast<const uint4*>(a.c.v_src)[s];
  }
}

// ---------------------------------------------------------------------------
// Split-K decode attention
// ---------------------------------------------------------------------------
// Grid (splits, H_kv, B), 4 warps. The work of one (batch row, kv head) is a
// range of units: its groups, then its fp16 window cut into 32-token chunks
// worth kChunkUnits units each; split x takes units [x * U, (x + 1) * U).
// Warp w of a block takes the block's groups begin + w, begin + w + 4, ...
// through its own ring of STAGES shared-memory stages filled by bulk copies
// (one mbarrier per stage), then its window chunks. Each block writes
// unnormalized (m, l, o) partials per query head; m and the scores are in
// log2 units.
//
// Tensor-core mapping per group (m16n8k16, M = 16 rows = 8 query heads x
// {hi, lo} fp16 parts):
//   q.k^T : A = q'_{h,d} = q_{h,d} * s_{g,d} split exactly into fp16 hi + lo
//           (hi = fp16(q*s), lo = fma(q, s, -hi)); B = key codes (fields as
//           fp16 subnormals); plus q . z_g on CUDA cores.
//   p.V   : A = p_t * s_t split into fp16 hi + lo (lo carried times
//           kLoGain); B = value codes; plus sum_t p_t z_t on CUDA cores.
// Per window chunk the same tiles take fp16 operands straight from shared
// memory (ldmatrix): A = q for q.k^T, A = p split into hi + lo, B = values.
template <int D>
struct CombineSmem {
  static constexpr int O_FLOATS = 4 * 8 * D;
  static constexpr int BYTES = (O_FLOATS + 64) * 4;
};

template <int D, int KB, int VB, int STAGES>
struct DecodeSmem {
  static constexpr int BAR_BYTES = 256;
  static constexpr int STAGE_BYTES = 4 * STAGES * Kivi<D, KB, VB>::STAGE;
  static constexpr int WIN_ROW = 2 * D + 16;  // one fp16 window row, padded: ldmatrix rows hit distinct banks
  static constexpr int AREA = (STAGE_BYTES > CombineSmem<D>::BYTES) ? STAGE_BYTES : CombineSmem<D>::BYTES;
  static constexpr int BYTES = BAR_BYTES + AREA;
  static_assert((4 * STAGES + 4) * 8 <= BAR_BYTES, "barrier area");
  static_assert(STAGES * Kivi<D, KB, VB>::STAGE >= 32 * WIN_ROW, "a warp's stages hold one window chunk");
};

// Online softmax over the 32 scores of one group or chunk (log2 domain): this
// thread's 8 scores sc of row g give the weights p = 2^(sc - m_run). The
// reference m_run moves only when a score exceeds it by more than 0.5, so
// weights stay <= 2^0.5 and p * s_t still fits fp16 for any scale
// (2^0.5 * 43669 < 65504); the rescale of the accumulators then runs rarely
// instead of whenever some head's max grows.
template <int NTV>
__device__ __forceinline__ void online_softmax(const float (&sc)[8], float (&p)[8], float (&o_acc)[NTV][4], float& m_run,
                                               float& l_run, float& vz_run) {
  float mx = sc[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) mx = fmaxf(mx, sc[i]);
  mx = quad_max(mx);
  if (mx > m_run + 0.5f) {
    const float alpha = fast_exp2(m_run - mx);
    l_run *= alpha;
    vz_run *= alpha;
#pragma unroll
    for (int i = 0; i < NTV; ++i) {
      o_acc[i][0] *= alpha;
      o_acc[i][1] *= alpha;
      o_acc[i][2] *= alpha;
      o_acc[i][3] *= alpha;
    }
    m_run = mx;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) p[i] = fast_exp2(sc[i] - m_run);
}

// The fp16 window chunks c_first, c_first + 4, ... < c_end of one warp, after
// its groups. The warp's stages are free by then and hold one chunk at a time
// (rows padded to win_row bytes, one bulk copy per row, keys first, then the
// values into the same rows). o_acc is first brought from code units to real
// units so that p . V of the fp16 values adds straight into it. Kept out of
// line: the main loop then keeps its own register allocation. Returns false
// when a copy wait timed out (that copy may still be in flight on phase
// `wphase` of `wbar`).
template <int D, int VB>
__device__ __noinline__ bool window_chunks(const uint16_t* k_res, const uint16_t* v_res, long long row_base,
                                           int n_resid, int c_first, int c_end, uint8_t* buf, int win_row,
                                           uint64_t* wbar, uint32_t& wphase, const uint32_t (&qs)[D / 16][2],
                                           float p2e, float (&o_io)[D / 8][4], float& m_run, float& l_run,
                                           float& vz_run) {
  constexpr int KS = D / 16, NTV = D / 8;
  const int lane = threadIdx.x & 31, tig = lane & 3;
  const int mat = lane >> 3, mrow = lane & 7;  // ldmatrix row of this lane inside four 8x8 tiles
  float o_acc[NTV][4];
#pragma unroll
  for (int nt = 0; nt < NTV; ++nt) {
    const float om = (VB == 2 && (nt & 1)) ? kInvP8 : kInvP6;
#pragma unroll
    for (int i = 0; i < 4; ++i) o_acc[nt][i] = o_io[nt][i] * om;
  }
  uint32_t q[KS][2];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) q[ks][0] = qs[ks][0], q[ks][1] = qs[ks][1];
  bool ok = true;
  for (int c = c_first; c < c_end; c += 4) {
    const int t0 = c * kGroup;
    const int nv = min(kGroup, n_resid - t0);
    const long long row0 = row_base + t0;
    // keys of the chunk
    __syncwarp();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (lane == 0) mbar_arrive_expect_tx(wbar, nv * D * 2);
    __syncwarp();
    if (lane < nv) bulk_g2s(buf + lane * win_row, k_res + (row0 + lane) * D, D * 2, wbar);
    if (!mbar_wait_bounded(wbar, wphase)) {
      ok = false;
      break;
    }
    wphase ^= 1u;
    float sacc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.0f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t kb[4];  // {b0, b1} of n-tiles 2np and 2np + 1
        ldsm_x4(kb, buf + (16 * np + 8 * (mat >> 1) + mrow) * win_row + (16 * ks + 8 * (mat & 1)) * 2);
        mma16816(sacc[2 * np], q[ks][0], 0u, q[ks][1], 0u, kb[0], kb[1]);
        mma16816(sacc[2 * np + 1], q[ks][0], 0u, q[ks][1], 0u, kb[2], kb[3]);
      }
    // values of the chunk into the same rows; the rows past the window are zeroed
    __syncwarp();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (lane == 0) mbar_arrive_expect_tx(wbar, nv * D * 2);
    __syncwarp();
    if (lane < nv) {
      bulk_g2s(buf + lane * win_row, v_res + (row0 + lane) * D, D * 2, wbar);
    } else {
      uint4* zr = reinterpret_cast<uint4*>(buf + lane * win_row);
#pragma unroll
      for (int i = 0; i < D / 8; ++i) zr[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    float sc[8], p[8];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int i = 0; i < 2; ++i) sc[2 * nt + i] = (8 * nt + 2 * tig + i < nv) ? sacc[nt][i] * p2e : -INFINITY;
    online_softmax<NTV>(sc, p, o_acc, m_run, l_run, vz_run);
    uint32_t phi[4], plo[4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const __half2 hh = __floats2half2_rn(p[2 * nt], p[2 * nt + 1]);
      const float2 hf = __half22float2(hh);
      phi[nt] = h2_bits(hh);
      plo[nt] = pack_rn_f16x2((p[2 * nt] - hf.x) * kLoGain, (p[2 * nt + 1] - hf.y) * kLoGain);
      l_run += p[2 * nt] + p[2 * nt + 1];
    }
    if (!mbar_wait_bounded(wbar, wphase)) {
      ok = false;
      break;
    }
    wphase ^= 1u;
    __syncwarp();  // the zeroed rows of the other lanes
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      const uint32_t A0 = phi[2 * ks], A1 = plo[2 * ks], A2 = phi[2 * ks + 1], A3 = plo[2 * ks + 1];
#pragma unroll
      for (int np = 0; np < NTV / 2; ++np) {
        uint32_t vb[4];  // {b0, b1} of channel tiles 2np and 2np + 1
        ldsm_x4_trans(vb, buf + (16 * ks + 8 * (mat & 1) + mrow) * win_row + (16 * np + 8 * (mat >> 1)) * 2);
        mma16816(o_acc[2 * np], A0, A1, A2, A3, vb[0], vb[1]);
        mma16816(o_acc[2 * np + 1], A0, A1, A2, A3, vb[2], vb[3]);
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < NTV; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) o_io[nt][i] = o_acc[nt][i];
  return ok;
}

// Sequence state of the contiguous cache: every pair has a.n_groups groups and
// a.n_resid window tokens, at unit p * pair_stride.
struct NoSeqs {};

// Block-table entries a warp of the paged decode keeps in its lanes (nothing
// for the contiguous cache).
template <bool kPaged>
struct TableLanes {
  int tbase = 0, tblk = 0;
};
template <>
struct TableLanes<false> {};

template <int D, int KB, int VB, int STAGES, class SeqT>
__global__ void __launch_bounds__(128, DecodeMinBlocks<D>::value) kivi_decode_kernel(KiviDecodeArgs a, SeqT seqs) {
  using P = Kivi<D, KB, VB>;
  constexpr bool kPaged = !std::is_same<SeqT, NoSeqs>::value;
  using S = DecodeSmem<D, KB, VB, STAGES>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* area = smem + S::BAR_BYTES;
  float* o_s = reinterpret_cast<float*>(area);  // [4 warps][8 rows][D]  (after a segment's loop)
  float* m_s = o_s + CombineSmem<D>::O_FLOATS;  // [4][8]
  float* l_s = m_s + 32;                        // [4][8]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
  const int gq = a.q_heads / a.kv_heads;
  // The warp's ring: NS slots of GPS consecutive groups each, one bulk copy
  // per record type and slot (records of consecutive groups are contiguous).
  constexpr int GPS = 2, NS = STAGES / GPS;
  static_assert(STAGES % GPS == 0, "whole slots");
  constexpr int SLOT = GPS * P::STAGE;
  uint64_t* bar = bars + warp * STAGES;
  uint64_t* wbar = bars + 4 * STAGES + warp;  // window chunk copies
  uint8_t* ring = area + warp * STAGES * P::STAGE;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
    mbar_init(wbar, 1);
    fence_mbar_init();
  }
  __syncwarp();

  // This block's slice [u0, u1) of all units, pair after pair; one segment
  // (and one partial) per (batch row, kv head) it touches.
  long long all_units = static_cast<long long>(a.n_pairs) * a.pair_stride;
  if constexpr (kPaged) all_units = seqs.unit0[seqs.n_seqs];
  const long long u0 = static_cast<long long>(blockIdx.x) * a.units_per_block;
  const long long u1 = min(all_units, u0 + a.units_per_block);
  int jg = 0;               // slots this warp has filled so far: ring position and phase of the next
  uint32_t wphase = 0;      // phase of the window barrier
  bool timed_out = false;   // sticky: after a wait gives up the warp starts no more copies
  for (long long u = u0; u < u1;) {
    int pair, upp, n_grp, n_res;  // the pair, its units, groups and window tokens
    long long pbase;              // its first unit
    if constexpr (kPaged) {
      const int sb = seq_of(seqs.unit0, seqs.n_seqs, u);
      n_grp = seqs.n_groups[sb];
      n_res = seqs.n_resid[sb];
      upp = n_grp + kChunkUnits * ((n_res + kGroup - 1) / kGroup);
      // each pair's range opens with pair_lead units of no work (the cost of
      // one more segment); pbase is its first unit of work
      const int span = upp + seqs.pair_lead;
      const int hh = static_cast<int>((u - seqs.unit0[sb]) / span);
      pair = sb * a.kv_heads + hh;
      const long long vbase = seqs.unit0[sb] + static_cast<long long>(hh) * span;
      pbase = vbase + seqs.pair_lead;
      u = vbase + span;
    } else {
      pair = static_cast<int>(u / a.pair_stride);
      pbase = static_cast<long long>(pair) * a.pair_stride;
      upp = a.units_per_pair;
      n_grp = a.n_groups;
      n_res = a.n_resid;
      u = pbase + a.pair_stride;
    }
    const int lo = static_cast<int>(u0 > pbase ? u0 - pbase : 0LL);
    const int hi = static_cast<int>(min(static_cast<long long>(upp), u1 - pbase));
    if (lo >= upp) continue;  // padding after the pair's units (the same for the whole block)
    if constexpr (kPaged) {
      if (hi <= 0) continue;  // the slice ends inside the pair's lead-in: no work here
    }
    const int b = pair / a.kv_heads, h = pair % a.kv_heads;
    const long long bh = pair;
    const int first_block = static_cast<int>(pbase / a.units_per_block);
    const int split = static_cast<int>(blockIdx.x) - first_block;
    const int n_splits = static_cast<int>((pbase + upp - 1) / a.units_per_block) - first_block + 1;
    // the stages and the combine area of the previous segment are reused
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();

    // groups [g_begin, g_end) and window chunks [c_begin, c_end) of the segment
    const int n_chunks = (n_res + kGroup - 1) / kGroup;
    const int g_begin = min(n_grp, lo);
    const int g_end = min(n_grp, hi);
    const int c_begin = min(n_chunks, max(0, lo - n_grp + kChunkUnits - 1) / kChunkUnits);
    const int c_end = min(n_chunks, max(0, hi - n_grp + kChunkUnits - 1) / kChunkUnits);

    float m_run = -INFINITY, l_run = 0.0f, vz_run = 0.0f;
    float o_acc[P::NTV][4];
#pragma unroll
    for (int i = 0; i < P::NTV; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.0f;
    // ------------------------------- grouped region -------------------------------
    // this warp's groups: pairs g_begin + GPS * (warp + 4 * k) + {0, .., GPS - 1}
    const int n_here = g_end - g_begin;
    int n_mine = 0;
    if (!timed_out && n_here > GPS * warp) {
      const int np = (n_here - GPS * warp + 4 * GPS - 1) / (4 * GPS);
      n_mine = GPS * (np - 1) + min(GPS, n_here - GPS * (warp + 4 * (np - 1)));
    }
    const int n_slots = (n_mine + GPS - 1) / GPS;
    // contiguous: the pair's records, groups one after the other
    const long long rec0 = bh * a.groups_cap;
    const uint8_t* kc_g = a.k_codes + rec0 * P::KC;
    const uint8_t* km_g = a.k_meta + rec0 * P::KM;
    const uint8_t* vc_g = a.v_codes + rec0 * P::VC;
    const uint8_t* vm_g = a.v_meta + rec0 * P::VM;
    // paged: group j's pool blocks come from the block table through the
    // lanes (lane l holds the entry of the warp's group tbase + l)
    TableLanes<kPaged> tl;
    auto load_table = [&](int base) {  // warp-wide
      if constexpr (kPaged) {
        tl.tbase = base;
        const int jl = base + lane;
        if (jl < n_mine) {
          const int grp = g_begin + GPS * (warp + 4 * (jl / GPS)) + jl % GPS;
          tl.tblk = min(max(__ldg(seqs.pools.block_table + static_cast<long long>(b) * a.groups_cap + grp), 0),
                        seqs.pools.num_blocks - 1);
        }
      }
    };
    // the pool blocks of slot k's groups (warp-wide)
    auto slot_blocks = [&](int k, int& b0, int& b1) {
      if constexpr (kPaged) {
        if (GPS * k + GPS > tl.tbase + 32) load_table(GPS * k);
        b0 = __shfl_sync(0xffffffffu, tl.tblk, GPS * k - tl.tbase);
        b1 = __shfl_sync(0xffffffffu, tl.tblk, GPS * k + 1 - tl.tbase);
      }
    };

    // slot k of this segment (groups GPS*k .. of the warp) goes through ring
    // position (jg + k) % NS as [key codes x GPS | key meta x GPS | value codes
    // x GPS | value meta x GPS]
    auto issue = [&](int k, int b0 = 0, int b1 = 0) {
      const int grp = g_begin + GPS * (warp + 4 * k);
      const uint32_t cnt = static_cast<uint32_t>(min(GPS, g_end - grp));
      uint8_t* dst = ring + ((jg + k) % NS) * SLOT;
      uint64_t* bb = &bar[(jg + k) % NS];
      mbar_arrive_expect_tx(bb, cnt * P::STAGE);
      if constexpr (kPaged) {
        // one copy per group: kv head h's entry of its pool block (the pool is
        // a.k_codes; table entries outside [0, num_blocks) were clamped)
        static_assert(GPS == 2, "two blocks per slot");
        const uint8_t* pool_h = a.k_codes + static_cast<long long>(h) * P::STAGE;
        bulk_g2s(dst, pool_h + static_cast<long long>(b0) * a.kv_heads * P::STAGE, P::STAGE, bb);
        if (cnt > 1) bulk_g2s(dst + P::STAGE, pool_h + static_cast<long long>(b1) * a.kv_heads * P::STAGE, P::STAGE, bb);
      } else {
        bulk_g2s(dst, kc_g + grp * static_cast<long long>(P::KC), cnt * P::KC, bb);
        bulk_g2s(dst + GPS * P::KC, km_g + grp * static_cast<long long>(P::KM), cnt * P::KM, bb);
        bulk_g2s(dst + GPS * (P::KC + P::KM), vc_g + grp * static_cast<long long>(P::VC), cnt * P::VC, bb);
        bulk_g2s(dst + GPS * (P::KC + P::KM + P::VC), vm_g + grp * static_cast<long long>(P::VM), cnt * P::VM, bb);
      }
    };
    auto wait_slot = [&](int k) { return mbar_wait_bounded(&bar[(jg + k) % NS], ((jg + k) / NS) & 1); };
    // the records of group j of the warp (paged: each group's four records
    // back to back; contiguous: the GPS groups' records of one kind together)
    auto slot_base = [&](int j) { return ring + ((jg + j / GPS) % NS) * SLOT; };
    auto kc_of = [&](int j) {
      if constexpr (kPaged) return slot_base(j) + (j % GPS) * P::STAGE;
      else return slot_base(j) + (j % GPS) * P::KC;
    };
    auto km_of = [&](int j) {
      if constexpr (kPaged) return slot_base(j) + (j % GPS) * P::STAGE + P::KC;
      else return slot_base(j) + GPS * P::KC + (j % GPS) * P::KM;
    };
    auto vc_of = [&](int j) {
      if constexpr (kPaged) return slot_base(j) + (j % GPS) * P::STAGE + P::KC + P::KM;
      else return slot_base(j) + GPS * (P::KC + P::KM) + (j % GPS) * P::VC;
    };
    auto vm_of = [&](int j) {
      if constexpr (kPaged) return slot_base(j) + (j % GPS) * P::STAGE + P::KC + P::KM + P::VC;
      else return slot_base(j) + GPS * (P::KC + P::KM + P::VC) + (j % GPS) * P::VM;
    };
    if constexpr (kPaged) {
      if (n_mine > 0) load_table(0);
      for (int k = 0; k < NS && k < n_slots; ++k) {
        int b0, b1;
        slot_blocks(k, b0, b1);
        if (lane == 0) issue(k, b0, b1);
      }
    } else {
      if (lane == 0) {
        for (int k = 0; k < NS && k < n_slots; ++k) issue(k);
      }
    }

    // Query fragments of row g (query head h*gq + g), scaled by 2^-e so that
    // |q| < 1 and q * s stays inside the fp16 range.
    const bool row_ok = g < gq;
    const __half* qrow = reinterpret_cast<const __half*>(a.q) +
                         (static_cast<long long>(b) * a.q_heads + h * gq + (row_ok ? g : 0)) * D;
    float2 qv[P::KS][2];
    float qmax = 0.0f;
#pragma unroll
    for (int ks = 0; ks < P::KS; ++ks)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const __half2 v = row_ok ? *reinterpret_cast<const __half2*>(qrow + 16 * ks + 8 * j + 2 * tig)
                                 : __float2half2_rn(0.0f);
        qv[ks][j] = __half22float2(v);
        qmax = fmaxf(qmax, fmaxf(fabsf(qv[ks][j].x), fabsf(qv[ks][j].y)));
      }
    qmax = quad_max(qmax);
    int e = 0;
    if (qmax > 0.0f) frexpf(qmax, &e);
    const float qscale = ldexpf(1.0f, -e);
    uint32_t qs[P::KS][2];
#pragma unroll
    for (int ks = 0; ks < P::KS; ++ks)
#pragma unroll
      for (int j = 0; j < 2; ++j) qs[ks][j] = pack_rn_f16x2(qv[ks][j].x * qscale, qv[ks][j].y * qscale);
    const float p2e = ldexpf(1.0f, e) * a.scale_log2;
    const float mult6 = kInvP6 * p2e, mult8 = kInvP8 * p2e;

    // q . k_hat of the 32 tokens of group j of the warp: 8 scores (log2
    // units) of this thread's row, tokens 8*nt + 2*tig + {0, 1}.
    auto qk_scores = [&](int jj, float (&sc)[8]) {
      const uint4* kcw = reinterpret_cast<const uint4*>(kc_of(jj));
      const uint4* kmr = reinterpret_cast<const uint4*>(km_of(jj));
      uint32_t kw[P::KW];
#pragma unroll
      for (int c = 0; c < P::KW / 4; ++c) {
        const uint4 x = kcw[c * 32 + lane];
        kw[4 * c] = x.x;
        kw[4 * c + 1] = x.y;
        kw[4 * c + 2] = x.z;
        kw[4 * c + 3] = x.w;
      }
      float sacc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.0f;
      // q . z: this lane's four channels of head g on the FMA pipe (the tensor pipe is the
      // busier one here); a quad sum after the loop completes the dot product.
      float bsum = 0.0f;
#pragma unroll
      for (int ks = 0; ks < P::KS; ++ks) {
        const uint4 md = kmr[ks * 4 + tig];  // {s(d0,d0+1), s(d0+8,d0+9), z(d0,d0+1), z(d0+8,d0+9)}
        const __half2 q0 = bits_h2(qs[ks][0]), q1 = bits_h2(qs[ks][1]);
        const __half2 hi0 = __hmul2(q0, bits_h2(md.x));
        const __half2 lo0 = __hfma2(q0, bits_h2(md.x), __hneg2(hi0));
        const __half2 hi1 = __hmul2(q1, bits_h2(md.y));
        const __half2 lo1 = __hfma2(q1, bits_h2(md.y), __hneg2(hi1));
        const uint32_t A0 = h2_bits(hi0), A1 = h2_bits(lo0), A2 = h2_bits(hi1), A3 = h2_bits(lo1);
        bsum = dot2_f16_f32(qs[ks][0], md.z, dot2_f16_f32(qs[ks][1], md.w, bsum));
        if constexpr (KB == 2) {
          const uint32_t w = kw[ks];
          const uint32_t l4 = w << 4, r4 = w >> 4, sw = __byte_perm(w, 0u, 0x2301u);
          mma16816(sacc[0], A0, A1, A2, A3, l4 & kMaskP6, r4 & kMaskP6);
          mma16816(sacc[1], A0, A1, A2, A3, l4 & kMaskP8, r4 & kMaskP8);
          mma16816(sacc[2], A0, A1, A2, A3, w & kMaskP6, sw & kMaskP6);
          mma16816(sacc[3], A0, A1, A2, A3, w & kMaskP8, sw & kMaskP8);
        } else {
          const uint32_t w0 = kw[2 * ks], w1 = kw[2 * ks + 1];
          mma16816(sacc[0], A0, A1, A2, A3, (w0 << 6) & kMask4, (w1 << 6) & kMask4);
          mma16816(sacc[1], A0, A1, A2, A3, (w0 << 2) & kMask4, (w1 << 2) & kMask4);
          mma16816(sacc[2], A0, A1, A2, A3, (w0 >> 2) & kMask4, (w1 >> 2) & kMask4);
          mma16816(sacc[3], A0, A1, A2, A3, (w0 >> 6) & kMask4, (w1 >> 6) & kMask4);
        }
      }
      const float bias = quad_sum(bsum) * p2e;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const float mult = (KB == 2 && (nt & 1)) ? mult8 : mult6;
        sc[2 * nt] = fmaf(sacc[nt][0] + sacc[nt][2], mult, bias);
        sc[2 * nt + 1] = fmaf(sacc[nt][1] + sacc[nt][3], mult, bias);
      }
    };

    // One group at a time: q . k^T, the softmax and p . V of group j. (Issuing
    // q . k^T of group j + 1 inside group j's p . V, a software pipeline, was
    // measured on GB300 against this: 2-bit D 128 equal, the other bit widths
    // and D 64 1.5-4.5 % slower, GQA-8 4-bit at 8K 95.0 against 90.8 us.)
    int j = 0;  // after the loop: the group a timed-out wait stopped at
    for (; !timed_out && j < n_mine; ++j) {
      if (j % GPS == 0 && !wait_slot(j / GPS)) {
        timed_out = true;
        break;
      }
      float sc[8];
      qk_scores(j, sc);
      const uint4* vcw = reinterpret_cast<const uint4*>(vc_of(j));
      const uint4* vmr = reinterpret_cast<const uint4*>(vm_of(j));

      float p[8];
      online_softmax<P::NTV>(sc, p, o_acc, m_run, l_run, vz_run);

      // ---- p' = p * s_t as fp16 hi + lo; the zero-point term on CUDA cores ----
      const uint4 vs = vmr[tig], vz = vmr[4 + tig];
      const uint32_t vsw[4] = {vs.x, vs.y, vs.z, vs.w};
      const uint32_t vzw[4] = {vz.x, vz.y, vz.z, vz.w};
      uint32_t phi[4], plo[4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const float2 sf = __half22float2(bits_h2(vsw[nt]));
        const float2 zf = __half22float2(bits_h2(vzw[nt]));
        const float pp0 = p[2 * nt] * sf.x, pp1 = p[2 * nt + 1] * sf.y;
        const __half2 hh = __floats2half2_rn(pp0, pp1);
        const float2 hf = __half22float2(hh);
        phi[nt] = h2_bits(hh);
        plo[nt] = pack_rn_f16x2((pp0 - hf.x) * kLoGain, (pp1 - hf.y) * kLoGain);
        l_run += p[2 * nt] + p[2 * nt + 1];
        vz_run = fmaf(p[2 * nt], zf.x, fmaf(p[2 * nt + 1], zf.y, vz_run));
      }

      // ---- o += p' . codes (group j) ----
      uint32_t vw[P::VW];
#pragma unroll
      for (int c = 0; c < P::VW / 4; ++c) {
        const uint4 x = vcw[c * 32 + lane];
        vw[4 * c] = x.x;
        vw[4 * c + 1] = x.y;
        vw[4 * c + 2] = x.z;
        vw[4 * c + 3] = x.w;
      }
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const uint32_t A0 = phi[2 * ks], A1 = plo[2 * ks], A2 = phi[2 * ks + 1], A3 = plo[2 * ks + 1];
#pragma unroll
        for (int q = 0; q < P::NQ; ++q) {
          if constexpr (VB == 2) {
            const uint32_t w = vw[ks * P::NQ + q];
            const uint32_t l4 = w << 4, r4 = w >> 4, sw = __byte_perm(w, 0u, 0x2301u);
            mma16816(o_acc[4 * q + 0], A0, A1, A2, A3, l4 & kMaskP6, r4 & kMaskP6);
            mma16816(o_acc[4 * q + 1], A0, A1, A2, A3, l4 & kMaskP8, r4 & kMaskP8);
            mma16816(o_acc[4 * q + 2], A0, A1, A2, A3, w & kMaskP6, sw & kMaskP6);
            mma16816(o_acc[4 * q + 3], A0, A1, A2, A3, w & kMaskP8, sw & kMaskP8);
          } else {
            const uint32_t w0 = vw[(2 * ks) * P::NQ + q], w1 = vw[(2 * ks + 1) * P::NQ + q];
            mma16816(o_acc[4 * q + 0], A0, A1, A2, A3, (w0 << 6) & kMask4, (w1 << 6) & kMask4);
            mma16816(o_acc[4 * q + 1], A0, A1, A2, A3, (w0 << 2) & kMask4, (w1 << 2) & kMask4);
            mma16816(o_acc[4 * q + 2], A0, A1, A2, A3, (w0 >> 2) & kMask4, (w1 >> 2) & kMask4);
            mma16816(o_acc[4 * q + 3], A0, A1, A2, A3, (w0 >> 6) & kMask4, (w1 >> 6) & kMask4);
          }
        }
      }

      // after the last group of its slot: release the slot and refill it NS slots ahead
      if (j % GPS == GPS - 1 || j + 1 == n_mine) {
        __syncwarp();
        if constexpr (kPaged) {
          const int kn = j / GPS + NS;
          if (kn < n_slots) {
            int b0, b1;
            slot_blocks(kn, b0, b1);
            if (lane == 0) {
              asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
              issue(kn, b0, b1);
            }
          }
        } else {
          if (lane == 0 && j / GPS + NS < n_slots) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(j / GPS + NS);
          }
        }
      }
    }

    // ------------------------ fp16 window, 32-token chunks ------------------------
    constexpr bool kTwoFields = (VB == 2);
    bool real_units = false, win_pending = false, seg_timeout = timed_out && n_mine > 0;
    if (!timed_out && c_begin + warp < c_end) {
      real_units = true;
      // the call takes copies: a variable whose address escapes would live in
      // local memory for the whole kernel, main loop included
      float o_io[P::NTV][4], st[3] = {m_run, l_run, vz_run};
      uint32_t q_io[P::KS][2];
#pragma unroll
      for (int i = 0; i < P::NTV; ++i)
        o_io[i][0] = o_acc[i][0], o_io[i][1] = o_acc[i][1], o_io[i][2] = o_acc[i][2], o_io[i][3] = o_acc[i][3];
#pragma unroll
      for (int ks = 0; ks < P::KS; ++ks) q_io[ks][0] = qs[ks][0], q_io[ks][1] = qs[ks][1];
      uint32_t ph = wphase;
      asm volatile("griddepcontrol.wait;" ::: "memory");  // the window is complete (see decode_dispatch)
      const bool ok = window_chunks<D, VB>(a.k_res, a.v_res, bh * a.res_cap, n_res, c_begin + warp, c_end, ring,
                                           S::WIN_ROW, wbar, ph, q_io, p2e, o_io, st[0], st[1], st[2]);
#pragma unroll
      for (int i = 0; i < P::NTV; ++i)
        o_acc[i][0] = o_io[i][0], o_acc[i][1] = o_io[i][1], o_acc[i][2] = o_io[i][2], o_acc[i][3] = o_io[i][3];
      m_run = st[0];
      l_run = st[1];
      vz_run = st[2];
      wphase = ph;
      if (!ok) {
        timed_out = true;
        seg_timeout = true;
        win_pending = true;
      }
    }

    if (seg_timeout) {
      if (lane == 0) report_timeout(a.status);
      // let the copies already in flight land before the stages are reused
      for (int k = j / GPS; k < n_slots && k < j / GPS + NS; ++k) (void)wait_slot(k);
      if (win_pending) (void)mbar_wait_bounded(wbar, wphase);
    }
    if (timed_out) {
      m_run = -INFINITY;
      l_run = 0.0f;
      vz_run = 0.0f;
#pragma unroll
      for (int i = 0; i < P::NTV; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.0f;
    }
    jg += n_slots;
    l_run = quad_sum(l_run);
    vz_run = quad_sum(vz_run);
    __syncthreads();  // every warp is done with its stages; the area is reused below
#pragma unroll
    for (int nt = 0; nt < P::NTV; ++nt) {
      const float om = real_units ? 1.0f : ((kTwoFields && (nt & 1)) ? kInvP8 : kInvP6);
      const int c = 8 * nt + 2 * tig;
      o_s[(warp * 8 + g) * D + c] = fmaf(fmaf(o_acc[nt][2], kLoGainInv, o_acc[nt][0]), om, vz_run);
      o_s[(warp * 8 + g) * D + c + 1] = fmaf(fmaf(o_acc[nt][3], kLoGainInv, o_acc[nt][1]), om, vz_run);
    }
    if (tig == 0) {
      m_s[warp * 8 + g] = m_run;
      l_s[warp * 8 + g] = l_run;
    }

    // the kernel before this one has finished before any workspace write (see decode_dispatch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();
    finish_split<D>(o_s, m_s, l_s, gq, static_cast<long long>(b) * a.q_heads + h * gq, split, n_splits,
                    a.part_stride, a.part_o, a.part_ml, a.counters + bh, a.out, a.out_fp32);
  }
}

constexpr int kDecodeStages = 4;

// Persistent quantize grid: every resident block slot of the GPU (occupancy
// queried once per kernel and device), at most one block per item.
template <class Kern>
int quantize_grid(Kern kern, long long items, int (&cached)[64]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (cached[dev] == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 128, 0) != cudaSuccess || per_sm < 1) per_sm = 1;
    cached[dev] = per_sm;
  }
  const long long slots = static_cast<long long>(cached[dev]) * device_sm_count();
  return static_cast<int>(items < slots ? items : slots);
}

template <int D, int KB, int VB>
cudaError_t quantize_dispatch(const QuantGroupsArgs& a, const CopyTokensArgs& w, cudaStream_t s) {
  const long long total = static_cast<long long>(a.n_groups) * a.kv_heads * a.batch;
  static int cached[64] = {0};
  const int blocks = quantize_grid(kivi_quantize_kernel<D, KB, VB>, total, cached);
  kivi_quantize_kernel<D, KB, VB><<<blocks, 128, 0, s>>>(a, w);
  return cudaGetLastError();
}

template <int D, int KB, int VB>
cudaError_t quantize_paged_dispatch(const PagedQuantArgs& a, cudaStream_t s) {
  const long long total = static_cast<long long>(a.r.begin[a.n_seqs]) * a.q.kv_heads;
  static int cached[64] = {0};
  const int blocks = quantize_grid(kivi_quantize_paged_kernel<D, KB, VB>, total, cached);
  kivi_quantize_paged_kernel<D, KB, VB><<<blocks, 128, 0, s>>>(a);
  return cudaGetLastError();
}

template <int D, int KB, int VB, class SeqT>
int decode_occupancy() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    constexpr int smem = DecodeSmem<D, KB, VB, kDecodeStages>::BYTES;
    auto kern = kivi_decode_kernel<D, KB, VB, kDecodeStages, SeqT>;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 128, smem) != cudaSuccess || n <= 0)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

// The decode is launched as a programmatic dependent of the kernel before it
// on the stream. Only the token copy of kv_append_token (and of the window
// fill) lets its dependent start early; every other kernel releases it at its
// end as usual. So the decode's grouped loop, which reads only group records
// and q (complete before that copy started), overlaps the copy, while the
// fp16 window and the workspace (partials, split counters, shared with the
// previous decode) are touched only after griddepcontrol.wait, i.e. after the
// preceding kernel has completed.
template <int D, int KB, int VB, class SeqT>
cudaError_t decode_dispatch(const KiviDecodeArgs& a, const SeqT& seqs, cudaStream_t s) {
  constexpr int smem = DecodeSmem<D, KB, VB, kDecodeStages>::BYTES;
  auto kern = kivi_decode_kernel<D, KB, VB, kDecodeStages, SeqT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.n_blocks));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, seqs);
}

}  // namespace

cudaError_t launch_kivi_quantize(const QuantGroupsArgs& a, cudaStream_t s, const CopyTokensArgs* window) {
  CopyTokensArgs w{};
  if (window != nullptr && window->n_tokens > 0) w = *window;
  if (a.n_groups <= 0) return launch_copy_tokens(w, s);  // nothing to quantize: the copy alone (if any)
  const int key = a.head_dim * 100 + a.k_bits * 10 + a.v_bits;
  switch (key) {
    case 6422: return quantize_dispatch<64, 2, 2>(a, w, s);
    case 6424: return quantize_dispatch<64, 2, 4>(a, w, s);
    case 6442: return quantize_dispatch<64, 4, 2>(a, w, s);
    case 6444: return quantize_dispatch<64, 4, 4>(a, w, s);
    case 12822: return quantize_dispatch<128, 2, 2>(a, w, s);
    case 12824: return quantize_dispatch<128, 2, 4>(a, w, s);
    case 12842: return quantize_dispatch<128, 4, 2>(a, w, s);
    case 12844: return quantize_dispatch<128, 4, 4>(a, w, s);
    default: return cudaErrorInvalidValue;
  }
}

namespace {

template <class SeqT>
cudaError_t decode_by_key(const KiviDecodeArgs& a, const SeqT& seqs, cudaStream_t s) {
  switch (a.head_dim * 100 + a.k_bits * 10 + a.v_bits) {
    case 6422: return decode_dispatch<64, 2, 2>(a, seqs, s);
    case 6424: return decode_dispatch<64, 2, 4>(a, seqs, s);
    case 6442: return decode_dispatch<64, 4, 2>(a, seqs, s);
    case 6444: return decode_dispatch<64, 4, 4>(a, seqs, s);
    case 12822: return decode_dispatch<128, 2, 2>(a, seqs, s);
    case 12824: return decode_dispatch<128, 2, 4>(a, seqs, s);
    case 12842: return decode_dispatch<128, 4, 2>(a, seqs, s);
    case 12844: return decode_dispatch<128, 4, 4>(a, seqs, s);
    default: return cudaErrorInvalidValue;
  }
}

template <class SeqT>
int occupancy_by_key(int head_dim, int k_bits, int v_bits) {
  switch (head_dim * 100 + k_bits * 10 + v_bits) {
    case 6422: return decode_occupancy<64, 2, 2, SeqT>();
    case 6424: return decode_occupancy<64, 2, 4, SeqT>();
    case 6442: return decode_occupancy<64, 4, 2, SeqT>();
    case 6444: return decode_occupancy<64, 4, 4, SeqT>();
    case 12822: return decode_occupancy<128, 2, 2, SeqT>();
    case 12824: return decode_occupancy<128, 2, 4, SeqT>();
    case 12842: return decode_occupancy<128, 4, 2, SeqT>();
    case 12844: return decode_occupancy<128, 4, 4, SeqT>();
    default: return 1;
  }
}

}  // namespace

cudaError_t launch_kivi_decode(const KiviDecodeArgs& a, cudaStream_t s) { return decode_by_key(a, NoSeqs{}, s); }

cudaError_t launch_kivi_decode_paged(const KiviDecodeArgs& a, const PagedSeqs& seqs, cudaStream_t s) {
  return decode_by_key(a, seqs, s);
}

int kivi_decode_blocks_per_sm(int head_dim, int k_bits, int v_bits) {
  return occupancy_by_key<NoSeqs>(head_dim, k_bits, v_bits);
}

int kivi_paged_decode_blocks_per_sm(int head_dim, int k_bits, int v_bits) {
  return occupancy_by_key<PagedSeqs>(head_dim, k_bits, v_bits);
}

cudaError_t launch_kivi_quantize_paged(const PagedQuantArgs& a, cudaStream_t s) {
  if (a.n_seqs <= 0 || a.r.begin[a.n_seqs] <= 0) return cudaSuccess;
  switch (a.q.head_dim * 100 + a.q.k_bits * 10 + a.q.v_bits) {
    case 6422: return quantize_paged_dispatch<64, 2, 2>(a, s);
    case 6424: return quantize_paged_dispatch<64, 2, 4>(a, s);
    case 6442: return quantize_paged_dispatch<64, 4, 2>(a, s);
    case 6444: return quantize_paged_dispatch<64, 4, 4>(a, s);
    case 12822: return quantize_paged_dispatch<128, 2, 2>(a, s);
    case 12824: return quantize_paged_dispatch<128, 2, 4>(a, s);
    case 12842: return quantize_paged_dispatch<128, 4, 2>(a, s);
    case 12844: return quantize_paged_dispatch<128, 4, 4>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_copy_tokens_paged(const PagedCopyArgs& a, cudaStream_t s) {
  if (a.n_seqs <= 0 || a.r.begin[a.n_seqs] <= 0) return cudaSuccess;
  const long long total = static_cast<long long>(a.r.begin[a.n_seqs]) * a.kv_heads * (a.c.head_dim / 8);
  const int blocks = static_cast<int>((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  copy_tokens_paged_kernel<<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_copy_tokens(const CopyTokensArgs& a, cudaStream_t s) {
  if (a.n_tokens <= 0) return cudaSuccess;
  const long long total = static_cast<long long>(a.n_tokens) * (a.head_dim / 8) * a.bh;
  const int blocks = static_cast<int>((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
  copy_tokens_kernel<<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

}  // namespace kvq
